// worklist.cpp -- host-side schedulers for the persistent attention kernels.
//
// DISTFLASHATTN (paperlayer.ai summary of arXiv 2310.03294), §3.2 and App. B:
// under causal attention a worker that owns later tokens has more key/value
// blocks to visit, so with one contiguous token range per worker roughly half
// the workers sit idle; the balanced schedule lets the early workers take
// over part of the late workers' work, which on one GPU becomes a work list
// for persistent CTAs.  §4.5 quotes the resulting ideal speedups for eight
// workers: 36 blocks in 8 steps (4.5x) unbalanced, in 5 steps (7.2x) balanced.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/dfa.h"

namespace {

// Split n units into `parts` contiguous ranges; range r is [lo(r), lo(r+1)).
inline int64_t range_lo(int64_t n, int64_t parts, int64_t r) { return (n * r) / parts; }

}  // namespace

extern "C" int64_t dfa_build_worklist(int n_rows, int n_units, int n_workers, dfa_sched sched,
                                      int32_t* offsets, int32_t* items) {
    if (n_rows < 0 || n_units < 0 || n_workers <= 0 || !offsets ||
        (n_rows > 0 && n_units > 0 && !items))
        return -1;
    if (sched != DFA_SCHED_BALANCED && sched != DFA_SCHED_UNBALANCED) return -1;
    if ((int64_t)n_rows * n_units > INT32_MAX) return -1;
    const int64_t W = n_workers;
    std::vector<std::vector<int32_t>> per(W);
    std::vector<int64_t> cost(W, 0);
    // Each worker walks the (batch, head) rows in the same order, so workers
    // run on the same head at about the same time and share its K/V in L2.
    if (sched == DFA_SCHED_UNBALANCED) {
        // One contiguous range of units per worker, the same for every row.
        for (int64_t row = 0; row < n_rows; ++row)
            for (int64_t w = 0; w < W; ++w)
                for (int64_t u = range_lo(n_units, W, w); u < range_lo(n_units, W, w + 1); ++u) {
                    per[w].push_back((int32_t)(row * n_units + u));
                    cost[w] += u + 1;
                }
    } else {
        // Mirror pairs (n-1-u, u) cost n+1 tiles each; pairs are dealt to the
        // workers cyclically across rows, so no worker holds more than one
        // pair above the average.  The heavier unit of a pair goes first.
        int64_t t = 0;
        for (int64_t row = 0; row < n_rows; ++row)
            for (int64_t u = 0; u < (n_units + 1) / 2; ++u, ++t) {
                const int64_t w = t % W, heavy = n_units - 1 - u;
                per[w].push_back((int32_t)(row * n_units + heavy));
                cost[w] += heavy + 1;
                if (heavy != u) {
                    per[w].push_back((int32_t)(row * n_units + u));
                    cost[w] += u + 1;
                }
            }
    }
    int64_t pos = 0, makespan = 0;
    for (int64_t w = 0; w < W; ++w) {
        offsets[w] = (int32_t)pos;
        for (int32_t it : per[w]) items[pos++] = it;
        makespan = std::max(makespan, cost[w]);
    }
    offsets[W] = (int32_t)pos;
    return makespan;
}

namespace {

// Key tiles a forward query block sees: [0, hi(u)).
inline int64_t block_hi(int64_t u, int64_t kv_tiles, int causal) {
    return causal ? std::min(2 * u + 2, kv_tiles) : kv_tiles;
}

}  // namespace

extern "C" int dfa_split_piece_tiles(int B, int H, int S, int causal, int n_sms) {
    if (B <= 0 || H <= 0 || S <= 0 || n_sms <= 0) return 0;
    const int64_t units = (S + 255) / 256, kv_tiles = (S + 127) / 128;
    const int64_t rows = (int64_t)B * H;
    if (rows * units >= n_sms) return 0;   // every SM already has a query block
    int64_t work = 0;                      // key tiles over all blocks
    for (int64_t u = 0; u < units; ++u) work += block_hi(u, kv_tiles, causal);
    work *= rows;
    // About two pieces per SM so the greedy deal can even out the causal
    // triangle; at least four tiles so a piece amortises its Q load and its
    // fp32 partial store.
    const int64_t piece = std::max<int64_t>(4, (work + 2 * n_sms - 1) / (2 * n_sms));
    if ((kv_tiles + piece - 1) / piece <= 1) return 0;
    return (int)piece;
}

extern "C" int64_t dfa_build_split_worklist(int n_rows, int n_units, int kv_tiles, int causal, int piece_tiles,
                                            int n_workers, int32_t* offsets, int32_t* items) {
    if (n_rows < 0 || n_units < 0 || kv_tiles < 0 || piece_tiles <= 0 || n_workers <= 0 || !offsets) return -1;
    const int64_t n_split = std::max<int64_t>(1, (kv_tiles + piece_tiles - 1) / piece_tiles);
    if ((int64_t)n_rows * n_units * n_split > INT32_MAX) return -1;
    struct Piece {
        int64_t cost;
        int32_t value;
    };
    std::vector<Piece> pieces;
    for (int64_t row = 0; row < n_rows; ++row)
        for (int64_t u = 0; u < n_units; ++u) {
            const int64_t hi = block_hi(u, kv_tiles, causal);
            for (int64_t s = 0; s * piece_tiles < hi; ++s) {
                const int64_t len = std::min<int64_t>(hi, (s + 1) * piece_tiles) - s * piece_tiles;
                pieces.push_back({2 * len, (int32_t)((row * n_units + u) * n_split + s)});
            }
        }
    if (!pieces.empty() && !items) return -1;
    std::stable_sort(pieces.begin(), pieces.end(), [](const Piece& x, const Piece& y) { return x.cost > y.cost; });
    const int64_t W = n_workers;
    std::vector<std::vector<int32_t>> per(W);
    using Load = std::pair<int64_t, int64_t>;   // (cost so far, worker): the smallest first
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int64_t w = 0; w < W; ++w) heap.push({0, w});
    int64_t makespan = 0;
    for (const Piece& pc : pieces) {
        Load l = heap.top();
        heap.pop();
        per[l.second].push_back(pc.value);
        l.first += pc.cost;
        makespan = std::max(makespan, l.first);
        heap.push(l);
    }
    int64_t pos = 0;
    for (int64_t w = 0; w < W; ++w) {
        offsets[w] = (int32_t)pos;
        for (int32_t it : per[w]) items[pos++] = it;
    }
    offsets[W] = (int32_t)pos;
    return makespan;
}

extern "C" int dfa_split_bwd_piece_tiles(int B, int H_kv, int S, int causal, int n_sms) {
    if (B <= 0 || H_kv <= 0 || S <= 0 || n_sms <= 0) return 0;
    const int64_t n = (S + 127) / 128, rows = (int64_t)B * H_kv;
    // Split only when the mirror pairs leave a quarter of the SMs or more idle:
    // measured on one GB300, 32 / 64 / 96 pairs on 152 SMs gain 2.3x / 1.76x /
    // 1.33x, 128 pairs nothing (the pieces' dK/dV reductions and casts eat it).
    if (4 * rows * ((n + 1) / 2) > 3 * (int64_t)n_sms) return 0;
    const int64_t work = rows * (causal ? n * (n + 1) / 2 : n * n);   // (key tile, query tile) pairs
    // About two pieces per SM; at least 16 query tiles so that a piece's K/V
    // load and its 128 KB of dK/dV reductions stay small against its MMAs.
    const int64_t piece = std::max<int64_t>(16, (work + 2 * n_sms - 1) / (2 * n_sms));
    if ((n + piece - 1) / piece <= 1) return 0;
    return (int)piece;
}

extern "C" int64_t dfa_build_bwd_split_worklist(int n_rows, int kv_tiles, int causal, int piece_tiles,
                                                int n_workers, int32_t* offsets, int32_t* items) {
    if (n_rows < 0 || kv_tiles < 0 || piece_tiles <= 0 || n_workers <= 0 || !offsets) return -1;
    const int64_t n = kv_tiles, n_split = std::max<int64_t>(1, (n + piece_tiles - 1) / piece_tiles);
    if ((int64_t)n_rows * n * n_split > INT32_MAX) return -1;
    struct Piece {
        int64_t cost;
        int32_t value;
    };
    std::vector<Piece> pieces;
    for (int64_t row = 0; row < n_rows; ++row)
        for (int64_t u = 0; u < n; ++u) {
            const int64_t t = n - 1 - u;                    // key tile of unit u
            const int64_t visible = causal ? n - t : n;     // query tiles [t, n) or [0, n)
            for (int64_t s = 0; s * piece_tiles < visible; ++s) {
                const int64_t len = std::min<int64_t>(visible, (s + 1) * piece_tiles) - s * piece_tiles;
                pieces.push_back({len, (int32_t)((row * n + u) * n_split + s)});
            }
        }
    if (!pieces.empty() && !items) return -1;
    std::stable_sort(pieces.begin(), pieces.end(), [](const Piece& x, const Piece& y) { return x.cost > y.cost; });
    const int64_t W = n_workers;
    std::vector<std::vector<int32_t>> per(W);
    using Load = std::pair<int64_t, int64_t>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int64_t w = 0; w < W; ++w) heap.push({0, w});
    int64_t makespan = 0;
    for (const Piece& pc : pieces) {
        Load l = heap.top();
        heap.pop();
        per[l.second].push_back(pc.value);
        l.first += pc.cost;
        makespan = std::max(makespan, l.first);
        heap.push(l);
    }
    int64_t pos = 0;
    for (int64_t w = 0; w < W; ++w) {
        offsets[w] = (int32_t)pos;
        for (int32_t it : per[w]) items[pos++] = it;
    }
    offsets[W] = (int32_t)pos;
    return makespan;
}

extern "C" int64_t dfa_build_varlen_worklist(int n_seq, const int32_t* seq_units, int heads, int n_units_max,
                                             int causal, int n_workers, int32_t* offsets, int32_t* items) {
    if (n_seq < 0 || heads <= 0 || n_units_max < 0 || n_workers <= 0 || !offsets || (n_seq > 0 && !seq_units))
        return -1;
    if ((int64_t)n_seq * heads * n_units_max > INT32_MAX) return -1;
    // Groups dealt as a whole: causal mirror pairs (heavy unit first) of equal
    // cost n_s + 1, or single units (the middle one, every non-causal unit).
    struct Group {
        int64_t cost;
        int32_t first, second;   // item values; second = -1 for a single unit
    };
    std::vector<Group> groups;
    for (int64_t s = 0; s < n_seq; ++s) {
        const int64_t n = seq_units[s];
        if (n < 0 || n > n_units_max) return -1;
        for (int64_t h = 0; h < heads; ++h) {
            const int64_t row = (s * heads + h) * n_units_max;
            if (!causal) {
                for (int64_t u = 0; u < n; ++u) groups.push_back({n, (int32_t)(row + u), -1});
                continue;
            }
            for (int64_t u = 0; u < (n + 1) / 2; ++u) {
                const int64_t heavy = n - 1 - u;
                if (heavy == u) groups.push_back({u + 1, (int32_t)(row + u), -1});
                else groups.push_back({n + 1, (int32_t)(row + heavy), (int32_t)(row + u)});
            }
        }
    }
    if (!groups.empty() && !items) return -1;
    std::stable_sort(groups.begin(), groups.end(), [](const Group& x, const Group& y) { return x.cost > y.cost; });
    const int64_t W = n_workers;
    std::vector<std::vector<int32_t>> per(W);
    using Load = std::pair<int64_t, int64_t>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int64_t w = 0; w < W; ++w) heap.push({0, w});
    int64_t makespan = 0;
    for (const Group& g : groups) {
        Load l = heap.top();
        heap.pop();
        per[l.second].push_back(g.first);
        if (g.second >= 0) per[l.second].push_back(g.second);
        l.first += g.cost;
        makespan = std::max(makespan, l.first);
        heap.push(l);
    }
    int64_t pos = 0;
    for (int64_t w = 0; w < W; ++w) {
        offsets[w] = (int32_t)pos;
        for (int32_t it : per[w]) items[pos++] = it;
    }
    offsets[W] = (int32_t)pos;
    return makespan;
}

extern "C" int dfa_chunk_schedule(int P, dfa_sched sched, int max_steps, int32_t* steps) {
    if (P <= 0 || max_steps <= 0 || !steps) return -1;
    if (sched != DFA_SCHED_BALANCED && sched != DFA_SCHED_UNBALANCED) return -1;
    // Per worker, the ordered list of (qchunk, kvchunk) blocks it computes.
    std::vector<std::vector<int32_t>> work(P);
    auto block = [&](int qc, int kc) { return (int32_t)(qc * P + kc); };
    if (sched == DFA_SCHED_UNBALANCED) {
        for (int p = 0; p < P; ++p)
            for (int t = 0; t <= p; ++t) work[p].push_back(block(p, t));
    } else {
        // Worker p >= P/2 owns p+1 blocks, its helper P-1-p owns P-p; together
        // P+1, shared so both finish within ceil((P+1)/2) steps.  The helper
        // computes its own blocks first, then the tail of the owner's blocks
        // and hands the partial output and lse back for merging.
        const int per_worker = (P + 2) / 2;   // ceil((P+1)/2)
        for (int p = P - 1; p >= 0; --p) {
            const int helper = P - 1 - p;
            if (helper > p) break;             // pairs done
            if (helper == p) {                 // odd P: the middle worker is alone
                for (int t = 0; t <= p; ++t) work[p].push_back(block(p, t));
                continue;
            }
            const int own = std::min(p + 1, per_worker);
            for (int t = 0; t < own; ++t) work[p].push_back(block(p, t));
            for (int t = 0; t <= helper; ++t) work[helper].push_back(block(helper, t));
            for (int t = own; t <= p; ++t) work[helper].push_back(block(p, t));
        }
    }
    int n_steps = 0;
    for (auto& w : work) n_steps = std::max(n_steps, (int)w.size());
    if (n_steps > max_steps) return -1;
    for (int s = 0; s < n_steps; ++s)
        for (int p = 0; p < P; ++p)
            steps[s * P + p] = s < (int)work[p].size() ? work[p][s] : -1;
    return n_steps;
}
