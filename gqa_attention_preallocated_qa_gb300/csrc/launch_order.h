// launch_order.h -- host-side bookkeeping of programmatic dependent launch
// for the decode kernel family (host code only, no CUDA dependency).
//
// Decode-family launches with host positions (decode steps, short chunks)
// signal their dependents at kernel start, and every one of their thread
// blocks waits for the previous kernel on the stream before it exits, so a
// launch that has finished implies that its predecessor has.  When launch X
// starts, the launches that may still run are N, N-1, ..., N-k (N the one just
// before X) such that all thread blocks of N-k+1..N were resident together
// with one of N-k: none of them can have exited while N-k runs, and X starts
// only once every block of N has started.  The walk back from N therefore
// stops where the blocks counted so far plus one would exceed what the device
// holds at once, at a launch that signals only after its own wait (nothing
// before it still runs), or at a barrier: a kernel that never signals early
// (the prefill kernels, reset) or a synchronisation of the stream, after which
// nothing enqueued earlier still runs when the next launch starts.
//
// X must load only after its own wait the cache rows that those launches
// append to X's layer: at most the sum of their new tokens per sequence, just
// below X's first new slot (positions only grow between barriers).
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <deque>
#include <mutex>
#include <unordered_map>

namespace qa {

class LaunchOrder {
  public:
    // Guard value meaning "every cache row may still be written".
    static constexpr int kGuardAll = 1 << 30;

    // Records a launch of `ctas` thread blocks on `stream` that appends up to
    // `tmax` tokens per sequence to (cache, layer), and returns its guard: the
    // number of rows below its first new slot that launches possibly still
    // running append to the same (cache, layer).  early: the launch signals its
    // dependents before waiting for its predecessor.  resident_max: the most
    // thread blocks of this family the device holds at once.
    int admit(const void *stream, const void *cache, int layer, int ctas, int tmax, bool early,
              int64_t resident_max) {
        std::lock_guard<std::mutex> lock(mu_);
        Hist &h = hist_[stream];
        int64_t guard = 0, resident = 0;
        bool bounded = false;
        for (auto it = h.recs.rbegin(); it != h.recs.rend(); ++it) {
            if (it->cache == cache && it->layer == layer) guard += it->tmax;
            if (!it->early) {  // it waited before signalling: nothing before it still runs
                bounded = true;
                break;
            }
            resident += it->ctas;  // all of its blocks resident while anything before it runs
            if (resident + 1 > resident_max) {
                bounded = true;
                break;
            }
        }
        if (!bounded && h.truncated) guard = kGuardAll;  // the older launches are not known
        h.recs.push_back({cache, layer, std::max(ctas, 1), tmax, early});
        if (h.recs.size() > kCap) {
            h.recs.pop_front();
            h.truncated = true;
        }
        return static_cast<int>(std::min<int64_t>(guard, kGuardAll));
    }

    // True when no launch that may still run when the next launch on `stream`
    // starts appends to (cache, layer): the same walk as admit, nothing recorded.
    // A launch for which this holds may read that layer's device lengths
    // before its own wait.
    bool layer_settled(const void *stream, const void *cache, int layer, int64_t resident_max) {
        std::lock_guard<std::mutex> lock(mu_);
        auto found = hist_.find(stream);
        if (found == hist_.end()) return true;
        const Hist &h = found->second;
        int64_t resident = 0;
        for (auto it = h.recs.rbegin(); it != h.recs.rend(); ++it) {
            if (it->cache == cache && it->layer == layer) return false;
            if (!it->early) return true;
            resident += it->ctas;
            if (resident + 1 > resident_max) return true;
        }
        return !h.truncated;
    }

    // What the next launch on `stream` may run beside: 0 nothing (no launch
    // recorded since the last barrier), 1 launches of other layers only, 2 a
    // launch that appends to (cache, layer).
    int in_flight(const void *stream, const void *cache, int layer, int64_t resident_max) {
        {
            std::lock_guard<std::mutex> lock(mu_);
            auto found = hist_.find(stream);
            if (found == hist_.end() || found->second.recs.empty()) return 0;
        }
        return layer_settled(stream, cache, layer, resident_max) ? 1 : 2;
    }

    // A kernel that never signals early was enqueued on `stream`, or the
    // stream was synchronised.
    void barrier(const void *stream) {
        std::lock_guard<std::mutex> lock(mu_);
        hist_.erase(stream);
    }

    // The device was synchronised.
    void clear() {
        std::lock_guard<std::mutex> lock(mu_);
        hist_.clear();
    }

    // Launches kept per stream; the walk needs at most resident_max of them.
    static constexpr size_t kCap = size_t(1) << 14;

  private:
    struct Rec {
        const void *cache;
        int layer, ctas, tmax;
        bool early;
    };
    struct Hist {
        std::deque<Rec> recs;
        bool truncated = false;
    };
    std::mutex mu_;
    std::unordered_map<const void *, Hist> hist_;
};

}  // namespace qa
