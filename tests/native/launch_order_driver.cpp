// Command-line driver of qa::LaunchOrder for the CPU tests: one command per
// input line, one output line per `admit`.
//   admit <stream> <cache> <layer> <ctas> <tmax> <early 0|1> <resident_max>  -> guard
//   barrier <stream>
//   clear
//   fill <stream> <cache> <layer> <n>   (n admits of one block each, outputs nothing)
//   settled <stream> <cache> <layer> <resident_max>  -> 0 | 1
//   inflight <stream> <cache> <layer> <resident_max> -> 0 | 1 | 2
#include <cstdint>
#include <iostream>
#include <sstream>
#include <string>

#include "launch_order.h"

int main() {
    qa::LaunchOrder order;
    std::string line;
    while (std::getline(std::cin, line)) {
        std::istringstream in(line);
        std::string cmd;
        in >> cmd;
        if (cmd == "admit") {
            uintptr_t s, c;
            int layer, ctas, tmax, early;
            long long rmax;
            in >> s >> c >> layer >> ctas >> tmax >> early >> rmax;
            std::cout << order.admit(reinterpret_cast<const void *>(s), reinterpret_cast<const void *>(c),
                                     layer, ctas, tmax, early != 0, rmax)
                      << "\n";
        } else if (cmd == "barrier") {
            uintptr_t s;
            in >> s;
            order.barrier(reinterpret_cast<const void *>(s));
        } else if (cmd == "settled" || cmd == "inflight") {
            uintptr_t s, c;
            int layer;
            long long rmax;
            in >> s >> c >> layer >> rmax;
            const void *sp = reinterpret_cast<const void *>(s), *cp = reinterpret_cast<const void *>(c);
            std::cout << (cmd == "settled" ? int(order.layer_settled(sp, cp, layer, rmax))
                                           : order.in_flight(sp, cp, layer, rmax))
                      << "\n";
        } else if (cmd == "clear") {
            order.clear();
        } else if (cmd == "fill") {
            uintptr_t s, c;
            int layer;
            long long n;
            in >> s >> c >> layer >> n;
            for (long long i = 0; i < n; ++i)
                order.admit(reinterpret_cast<const void *>(s), reinterpret_cast<const void *>(c), layer, 1,
                            1, true, int64_t(1) << 40);
        }
    }
    return 0;
}
