// txl_sched.cu -- host-side static balance of the persistent attention kernel's work items.
//
// The work items of one launch fall into classes: every query tile qt of every (b, h) is one item
// of class qt, and all items of a class cost the same (its number of key tiles plus a fixed
// per-item overhead).  Items of a class are interchangeable, so a schedule is a matrix of counts:
// how many items of each class each CTA processes.  It is found by longest-processing-time-first
// list scheduling followed by a local search that moves or swaps single items between the most
// loaded CTA and the others while that lowers the maximum load.  (Plain serpentine order leaves
// the CTAs that receive one item more than the others with long items, e.g. 30 key tiles against
// an average of 25.3 for 768 items of 4, 5 and 6 tiles on 152 CTAs; this finds 26.)
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "txl_internal.h"

namespace txl {

namespace {

struct SchedKey {
    int G, n_cls, per_cls, len0;
    bool operator==(const SchedKey& o) const
    {
        return G == o.G && n_cls == o.n_cls && per_cls == o.per_cls && len0 == o.len0;
    }
};

std::mutex g_sched_mu;
SchedKey g_sched_key{0, 0, 0, 0};
std::vector<uint8_t> g_sched_counts;

// Class q costs len0 + q key tiles plus `tau` (tiles) of per-item overhead: an item transition of
// the persistent kernel (waiting for the item's last P.V, the epilogue, the ring reset) takes about
// 5 K cycles against about 2.6 K per key tile.
bool compute(int G, int n_cls, int per_cls, int len0, std::vector<uint8_t>& out)
{
    const float tau = 1.9f;
    std::vector<float> cost(n_cls);
    for (int q = 0; q < n_cls; ++q) cost[q] = static_cast<float>(len0 + q) + tau;
    std::vector<int> cnt(static_cast<size_t>(G) * n_cls, 0);
    std::vector<float> load(G, 0.f);
    // LPT: classes longest first, each item to the least loaded CTA
    using E = std::pair<float, int>;
    std::priority_queue<E, std::vector<E>, std::greater<E>> heap;
    for (int c = 0; c < G; ++c) heap.push({0.f, c});
    for (int q = n_cls - 1; q >= 0; --q)
        for (int k = 0; k < per_cls; ++k) {
            E e = heap.top();
            heap.pop();
            ++cnt[static_cast<size_t>(e.second) * n_cls + q];
            load[e.second] = e.first + cost[q];
            heap.push({load[e.second], e.second});
        }
    // local search on the most loaded CTA
    std::vector<int> order(G);
    const int max_iter = 20 * G + 1000;
    for (int it = 0; it < max_iter; ++it) {
        const int A = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
        const float la = load[A];
        for (int c = 0; c < G; ++c) order[c] = c;
        std::sort(order.begin(), order.end(), [&](int a, int b) { return load[a] < load[b]; });
        bool improved = false;
        for (int B : order) {
            if (B == A) continue;
            const float lb = load[B];
            for (int x = 0; x < n_cls && !improved; ++x) {
                int& ax = cnt[static_cast<size_t>(A) * n_cls + x];
                if (ax == 0) continue;
                if (lb + cost[x] < la - 1e-4f) {                      // move one item of class x
                    --ax;
                    ++cnt[static_cast<size_t>(B) * n_cls + x];
                    load[A] -= cost[x];
                    load[B] += cost[x];
                    improved = true;
                    break;
                }
                for (int y = 0; y < x; ++y) {                         // swap x (A) with a shorter y (B)
                    int& by = cnt[static_cast<size_t>(B) * n_cls + y];
                    if (by == 0) continue;
                    const float d = cost[x] - cost[y];
                    if (std::max(la - d, lb + d) < la - 1e-4f) {
                        --ax;
                        ++cnt[static_cast<size_t>(B) * n_cls + x];
                        --by;
                        ++cnt[static_cast<size_t>(A) * n_cls + y];
                        load[A] -= d;
                        load[B] += d;
                        improved = true;
                        break;
                    }
                }
            }
            if (improved) break;
        }
        if (!improved) break;
    }
    out.assign(cnt.size(), 0);
    for (size_t i = 0; i < cnt.size(); ++i) {
        if (cnt[i] > 255) return false;
        out[i] = static_cast<uint8_t>(cnt[i]);
    }
    return true;
}

}  // namespace

bool schedule_items(int G, int n_cls, int per_cls, int len0, uint8_t* counts, int capacity)
{
    if (G <= 0 || n_cls <= 0 || per_cls <= 0 || static_cast<int64_t>(G) * n_cls > capacity) return false;
    std::lock_guard<std::mutex> lock(g_sched_mu);
    const SchedKey key{G, n_cls, per_cls, len0};
    if (!(key == g_sched_key)) {
        std::vector<uint8_t> c;
        if (!compute(G, n_cls, per_cls, len0, c)) return false;
        g_sched_counts.swap(c);
        g_sched_key = key;
    }
    std::memcpy(counts, g_sched_counts.data(), g_sched_counts.size());
    return true;
}

}  // namespace txl
