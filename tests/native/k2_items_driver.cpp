// Command-line driver of the prefill attention's work items (csrc/k2_items.h)
// for the CPU tests.  One case per input line:
//   nseq Hkv G npairs hpi window len[0..7] start[0..7] cu[0..7] workers
// Output per case: for every worker c and each of its items in snake order,
//   c k idx b kvh qb h0 L qmin j0 nkv jmask row0 same
// where `same` is 1 when decoding index k + 1 ahead and then again (as the Q
// copy warp does) gave the same item; then a line "end".
#include <algorithm>
#include <iostream>
#include <sstream>
#include <string>

#include "k2_items.h"

struct Params {
    int nseq, Hkv, G, npairs, hpi, max_qblocks, nitems, window;
    int len[8], start[8], cu[8];
};

template <bool kWindow>
void run(const Params &p, int workers) {
    for (int c = 0; c < workers; ++c) {
        qa::K2Walk w, w2;
        qa::K2Item it, ahead;
        bool have_ahead = false;
        for (int k = 0;; ++k) {
            const int idx = qa::k2_snake_index(k, workers, c);
            if (!qa::k2_item_at<kWindow>(p, idx, w, it)) break;
            // the same walk used one index ahead and then again
            bool same = true;
            if (have_ahead)
                same = ahead.b == it.b && ahead.kvh == it.kvh && ahead.qb == it.qb && ahead.h0 == it.h0;
            qa::K2Item nx;
            have_ahead = qa::k2_item_at<kWindow>(p, qa::k2_snake_index(k + 1, workers, c), w2, nx);
            if (have_ahead) {
                ahead = nx;
                qa::K2Item again;
                qa::k2_item_at<kWindow>(p, qa::k2_snake_index(k + 1, workers, c), w2, again);
                same = same && again.b == nx.b && again.qb == nx.qb && again.h0 == nx.h0;
            }
            std::cout << c << ' ' << k << ' ' << idx << ' ' << it.b << ' ' << it.kvh << ' ' << it.qb << ' '
                      << it.h0 << ' ' << it.L << ' ' << it.qmin << ' ' << it.j0 << ' ' << it.nkv << ' '
                      << it.jmask << ' ' << it.row0 << ' ' << int(same) << '\n';
        }
    }
    std::cout << "end\n";
}

int main() {
    std::string line;
    while (std::getline(std::cin, line)) {
        std::istringstream in(line);
        Params p{};
        int workers = 1;
        in >> p.nseq >> p.Hkv >> p.G >> p.npairs >> p.hpi >> p.window;
        for (int &x : p.len) in >> x;
        for (int &x : p.start) in >> x;
        for (int &x : p.cu) in >> x;
        in >> workers;
        // as the host plans a launch: levels and items of the sequences' blocks
        int blocks = 0;
        p.max_qblocks = 0;
        for (int s = 0; s < p.nseq; ++s) {
            p.max_qblocks = std::max(p.max_qblocks, (p.len[s] + 127) / 128);
            blocks += (p.len[s] + 127) / 128;
        }
        p.nitems = blocks * p.Hkv * p.npairs;
        if (p.window > 0)
            run<true>(p, workers);
        else
            run<false>(p, workers);
    }
    return 0;
}
