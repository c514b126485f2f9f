// fwd_tc.cu -- tcgen05 tensor-core causal attention forward for sm_103a.
//
// DISTFLASHATTN (paperlayer.ai summary of arXiv 2310.03294): each query chunk
// attends to the key/value chunks at or before it (§3.2), every chunk step
// updates the attention state and yields an output with its log-sum-exp
// (App. D), and states combine by the online-softmax rescale-and-merge rule.
// Here one CTA owns a block of 256 query rows (two 128-row tiles) and streams
// every visible 128-row key/value tile through shared memory; the running
// (max, sum, unnormalised output) of each row IS the merged state of all
// chunk steps so far, so partials of consecutive chunks merge on chip.
//
// Roles (384 threads, one CTA per SM, persistent over a host-built work list):
//   warp 0      TMA producer: Q tiles once per block, then K_j, V_j into a
//               ring of shared-memory slots (the single-GPU analogue of the
//               pages' key/value prefetch overlapping compute, §3.2).
//   warp 1      MMA issuer (one thread): S_w = Q_w K_j^T and O_w += P_w V_j
//               on the 5th-generation tensor cores, fp32 accumulators in TMEM.
//   warp 2      TMEM allocation.
//   warps 4-11  two softmax warpgroups, one query row per thread: row max,
//               exp2, row sum, P (bf16) written back into TMEM over S, lazy
//               rescale of O, and the epilogue O/l, lse.
// The two Q tiles ping-pong: while one warpgroup runs its softmax the tensor
// cores run the other tile's MMAs.
//
// TMEM columns: S_0 [0,128) S_1 [128,256) O_0 [256,256+D) O_1 [384,384+D);
// P_w (bf16 pairs) overwrites the first 64 columns of S_w.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dfa {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int BM = 128;            // query rows per tile (MMA M)
constexpr int BN = 128;            // key rows per tile
constexpr int kBlockRows = 2 * BM; // query rows per work unit
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O only when the max grows by > 2^8

template <int D>
struct Cfg {
    static constexpr int kTileBytes = BN * D * 2;              // one bf16 tile of 128 rows
    static constexpr int kSlots = D == 128 ? 4 : 6;            // K/V ring depth
    static constexpr int kQBytes = 2 * kTileBytes;
    static constexpr int kSmem = kQBytes + kSlots * kTileBytes + 1024 /*barriers*/ + 1024 /*align*/;
};

struct FwdArgs {
    int B, H, Hkv, Lq, Lkv;
    int64_t q_offset, kv_offset;
    int causal;
    int64_t win_c;         // local window: chunk length (tokens) ...
    int win_w;             // ... and chunks per window (0: no window)
    float scale_log2;      // scale * log2(e)
    void* O;               // dense [B, Lq, H, D], bf16 or fp32
    float* lse;            // [B, H, Lq]
    const int32_t* wl_offsets;
    const int32_t* wl_items;
    int n_units;
    // Split-kv helper items: item values carry a piece index s < n_split and
    // see key tiles [s * piece_tiles, (s + 1) * piece_tiles) only; piece s
    // writes its partial to O + s * o_piece_stride, lse + s * lse_piece_stride.
    int n_split, piece_tiles;
    int64_t o_piece_stride, lse_piece_stride;
    // Variable-length batch: tensors are packed [1, T, heads, D] (Lq = Lkv = T),
    // lse [1, H, T]; sequence b holds tokens [seq[b], seq[b + 1]).  nullptr: dense.
    const int32_t* seq;
    int* err;
    uint64_t* trace;              // optional per-CTA timeline (nullptr: off)
    int trace_cap;
};

struct Item {
    int b, h, g, q0, j0, n_kv;   // key/value tiles [j0, n_kv) can be visible to the block
    int s;                       // key/value piece (0 without split-kv items)
    int tb, base;                // tensor batch index and first token of the sequence
    int lq, lkv;                 // query and key/value rows of the sequence
};

// First key position a query at position qp may see under the local window.
__device__ __forceinline__ int64_t window_lo(const FwdArgs& a, int64_t qp) {
    return (qp / a.win_c - (a.win_w - 1)) * a.win_c;
}

__device__ __forceinline__ Item decode(const FwdArgs& a, int it, bool win) {
    Item x;
    x.s = 0;
    if (a.n_split > 1) {
        x.s = it % a.n_split;
        it /= a.n_split;
    }
    const int row = it / a.n_units, unit = it % a.n_units;
    x.b = row / a.H;
    x.h = row % a.H;
    x.g = x.h / (a.H / a.Hkv);
    x.q0 = unit * kBlockRows;
    if (a.seq) {
        x.tb = 0;
        x.base = a.seq[x.b];
        x.lq = x.lkv = a.seq[x.b + 1] - x.base;
    } else {
        x.tb = x.b;
        x.base = 0;
        x.lq = a.Lq;
        x.lkv = a.Lkv;
    }
    const int total = (x.lkv + BN - 1) / BN;
    if (x.q0 >= x.lq) {   // past the end of a short sequence: nothing to compute or store
        x.n_kv = 0;
    } else if (!a.causal) {
        x.n_kv = total;
    } else {
        const int64_t last_q = a.q_offset + min(x.q0 + kBlockRows, x.lq) - 1;
        const int64_t visible = last_q - a.kv_offset + 1;   // keys [0, visible) may be seen
        const int64_t tiles = (visible + BN - 1) / BN;
        x.n_kv = visible <= 0 ? 0 : (int)(tiles < total ? tiles : total);
    }
    x.j0 = 0;
    if (win) {   // the block's first row has the lowest window start
        const int64_t lo = window_lo(a, a.q_offset + x.q0) - a.kv_offset;
        x.j0 = lo <= 0 ? 0 : (int)(lo / BN < x.n_kv ? lo / BN : x.n_kv);
    }
    if (a.n_split > 1) {   // this piece's tiles only (an empty range does no MMA work)
        const int lo = x.s * a.piece_tiles, hi = lo + a.piece_tiles;
        x.j0 = max(x.j0, lo);
        x.n_kv = max(min(x.n_kv, hi), x.j0);
    }
    return x;
}

// Row max of this thread's 128 scores in TMEM (columns outside [lo, lim) masked when MASK).
// Four independent accumulators keep the dependent chain short; the chunk
// loop stays rolled to keep the kernel's code small (several roles run
// different code at once and share the instruction cache).
template <bool MASK>
__device__ __forceinline__ float row_max(uint32_t tS, int lo, int lim) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tS + c * 32, u);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(u[e]);
            m[e & 3] = fmaxf(m[e & 3], (!MASK || (c * 32 + e >= lo && c * 32 + e < lim)) ? x : -INFINITY);
        }
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// P = exp2(s * c2 - m) for this thread's row, written as bf16 pairs over the
// first 64 TMEM columns of S (behind the columns still to be read).  Returns
// the row sum of the fp32 P values.
template <bool MASK>
__device__ __forceinline__ float row_exp(uint32_t tS, int lo, int lim, float c2, float m) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(tS + c * 32, u);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int c0 = c * 32 + 2 * e;
            float p0 = ex2(fmaf(__uint_as_float(u[2 * e]), c2, -m));
            float p1 = ex2(fmaf(__uint_as_float(u[2 * e + 1]), c2, -m));
            if (MASK) {
                p0 = c0 >= lo && c0 < lim ? p0 : 0.f;
                p1 = c0 + 1 >= lo && c0 + 1 < lim ? p1 : 0.f;
            }
            acc[e & 3] += p0 + p1;
            pk[e] = pack_bf16(p0, p1);
        }
        tmem_st16(tS + c * 16, pk);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// WIN: local window (its range and mask code is compiled only into this variant).
template <int D, bool OUT_F32, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                                   // 2 tiles
    uint8_t* sKV = smem + C::kQBytes;                     // ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::kSlots * C::kTileBytes);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* s_full = bars + 2;          // [2]
    uint64_t* p_full = bars + 4;          // [2]
    uint64_t* o_full = bars + 6;          // [2]
    uint64_t* done = bars + 8;
    uint64_t* kv_full = bars + 16;        // [kSlots]
    uint64_t* kv_empty = bars + 16 + C::kSlots;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 33);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int it_begin, it_end;
    if (a.wl_items) {
        it_begin = a.wl_offsets[blockIdx.x];
        it_end = a.wl_offsets[blockIdx.x + 1];
    } else {
        it_begin = blockIdx.x;
        it_end = blockIdx.x + 1;
    }

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int w = 0; w < 2; ++w) {
            mbar_init(&s_full[w], 1);
            mbar_init(&p_full[w], BM);
            mbar_init(&o_full[w], 1);
        }
        mbar_init(done, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t t_start = globaltimer();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        uint32_t ld = 0, qi = 0, qi_issued = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode(a, a.wl_items ? a.wl_items[it] : it, WIN);
            if (x.n_kv <= x.j0) continue;
            ok = __all_sync(0xffffffffu, mbar_wait_acc(q_empty, (qi & 1) ^ 1, abort_flag, a.err, nullptr));
            if (!ok) break;
            ++qi_issued;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full, C::kQBytes);
                for (int w = 0; w < 2; ++w)
                    for (int blk = 0; blk < D / 64; ++blk)
                        tma_load_4d(sQ + w * C::kTileBytes + blk * 16384, &tmQ, q_full, blk * 64, x.h,
                                    x.base + x.q0 + w * BM, x.tb);
            }
            __syncwarp();
            for (int j = x.j0; j < x.n_kv && ok; ++j) {
                for (int which = 0; which < 2; ++which, ++ld) {
                    const int slot = ld % C::kSlots;
                    ok = __all_sync(0xffffffffu, mbar_wait_acc(&kv_empty[slot], ((ld / C::kSlots) & 1) ^ 1,
                                                               abort_flag, a.err, nullptr));
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&kv_full[slot], C::kTileBytes);
                        for (int blk = 0; blk < D / 64; ++blk)
                            tma_load_4d(sKV + slot * C::kTileBytes + blk * 16384, which ? &tmV : &tmK,
                                        &kv_full[slot], blk * 64, x.g, x.base + j * BN, x.tb);
                    }
                    __syncwarp();
                }
            }
            ++qi;
        }
        if (!ok && lane == 0) {
            // Aborted: let the copies already issued land before the CTA exits.
            // The newest load into each used slot is the only one possibly in flight.
            int dummy = 0;
            for (uint32_t s = 0; s < (uint32_t)C::kSlots && s < ld; ++s) {
                const uint32_t last = s + C::kSlots * ((ld - 1 - s) / C::kSlots);
                mbar_wait(&kv_full[s], (last / C::kSlots) & 1, &dummy, nullptr);
            }
            if (qi_issued > 0) mbar_wait(q_full, (qi_issued - 1) & 1, &dummy, nullptr);
        }
        if (lane == 0) trace_count(a.trace, a.trace_cap, 6, ld / 2);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // One thread: MMAs, commits, fences and mbarrier waits are per-thread, and a
        // lone thread keeps the gaps between MMA groups (idle tensor-pipe time) short.
        const uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
        const uint32_t idO = idesc_bf16_f32(BM, D, false, true);
        // Descriptors are built once and advanced by adding (byte offset / 16):
        // the start-address field is addr >> 4 and shared addresses stay below
        // 256 KB, so the addition never carries out of the field.  Keeping the
        // issue loop this short is what lets one thread feed the tensor core.
        const uint64_t dQk = sdesc_sw128(smem_u32(sQ), 16, 1024);          // Q, K-major
        const uint64_t dKk = sdesc_sw128(smem_u32(sKV), 16, 1024);         // K slots, K-major
        const uint64_t dVn = sdesc_sw128(smem_u32(sKV), 16384, 1024);      // V slots, N-major
        constexpr uint64_t kSlotStep = C::kTileBytes >> 4;
        uint32_t cons = 0, t = 0, qi = 0;
        bool ok = true;
        auto issue_S = [&](int w, uint32_t slot) {
            {
                const uint64_t a0 = dQk + w * kSlotStep, b0 = dKk + slot * kSlotStep;
                const uint32_t d = tmem + w * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                    mma_ss(d, a0 + off, b0 + off, idS, kk > 0);
                }
            }
        };
        auto issue_PV = [&](int w, uint32_t slot, bool acc) {
            {
                const uint64_t b0 = dVn + slot * kSlotStep;
                const uint32_t d = tmem + 256 + w * 128, a = tmem + w * 128;
                mma_ts(d, a, b0, idO, acc ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < BN / 16; ++kk) mma_ts(d, a + kk * 8, b0 + kk * (2048 >> 4), idO, 1u);
            }
        };
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            ok = ok && mbar_wait_issuer(bar, parity, abort_flag, a.err);
            if (ok) tc_fence_after();
            return ok;
        };
        auto commit = [&](uint64_t* bar) { mma_commit(bar); };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode(a, a.wl_items ? a.wl_items[it] : it, WIN);
            if (x.n_kv <= x.j0) continue;
            if (!wait(q_full, qi & 1)) break;
            uint32_t slotK = cons % C::kSlots;
            if (!wait(&kv_full[slotK], (cons / C::kSlots) & 1)) break;
            issue_S(0, slotK);
            commit(&s_full[0]);
            issue_S(1, slotK);
            commit(&s_full[1]);
            commit(&kv_empty[slotK]);
            ++cons;
            for (int j = x.j0; j < x.n_kv && ok; ++j, ++t) {
                const bool more = j + 1 < x.n_kv;
                const uint32_t slotV = cons % C::kSlots;
                if (!wait(&kv_full[slotV], (cons / C::kSlots) & 1)) break;
                if (!wait(&p_full[0], t & 1)) break;
                issue_PV(0, slotV, j > x.j0);
                if (!more) commit(&o_full[0]);
                uint32_t slotK1 = (cons + 1) % C::kSlots;
                if (more) {
                    if (!wait(&kv_full[slotK1], ((cons + 1) / C::kSlots) & 1)) break;
                    issue_S(0, slotK1);
                    commit(&s_full[0]);
                }
                if (!wait(&p_full[1], t & 1)) break;
                issue_PV(1, slotV, j > x.j0);
                commit(&kv_empty[slotV]);
                if (!more) commit(&o_full[1]);
                if (more) {
                    issue_S(1, slotK1);
                    commit(&s_full[1]);
                    commit(&kv_empty[slotK1]);
                }
                cons += more ? 2 : 1;
            }
            if (!ok) break;
            commit(q_empty);
            ++qi;
        }
        // Drain: every MMA this thread issued has finished before TMEM is freed.
        commit(done);
        int dummy = 0;
        mbar_wait(done, 0, &dummy, a.err);
        trace_count(a.trace, a.trace_cap, 4, t);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax warpgroups
        const int w = (warp - 4) / 4;                 // which query tile
        const int r = (warp % 4) * 32 + lane;         // row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + lane_base + w * 128;
        const uint32_t tO = tmem + lane_base + 256 + w * 128;
        const float c2 = a.scale_log2;
        uint32_t t = 0, qi = 0;
        bool ok = true;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode(a, a.wl_items ? a.wl_items[it] : it, WIN);
            const int row = x.q0 + w * BM + r;                 // row within the query chunk
            const int64_t qpos = a.q_offset + row;
            float m_run = -INFINITY, l = 0.f;
            // local window: this row's first visible key (relative to the chunk's keys),
            // and the highest such start among the tile's rows (decides the mask path)
            const int64_t lo_row = WIN ? window_lo(a, qpos) - a.kv_offset : INT64_MIN;
            const int64_t lo_tile = WIN ? window_lo(a, a.q_offset + x.q0 + w * BM + BM - 1) - a.kv_offset : INT64_MIN;
            for (int j = x.j0; j < x.n_kv; ++j, ++t) {
                ok = __all_sync(0xffffffffu, mbar_wait_acc(&s_full[w], t & 1, abort_flag, a.err, nullptr));
                if (!ok) break;
                tc_fence_after();
                // Pass 1: row max over the tile (S read from TMEM 32 columns at a time).
                const int kv0 = j * BN;
                const bool edge = kv0 + BN > x.lkv;
                const bool diag = a.causal && (a.kv_offset + kv0 + BN - 1 > a.q_offset + x.q0 + w * BM);
                const bool masked = edge || diag || (WIN && kv0 < lo_tile);
                // Column c of this tile is visible iff lo <= c < lim.
                int lo = 0, lim = BN;
                if (masked) {
                    if (WIN && lo_row > kv0) lo = lo_row - kv0 > BN ? BN : (int)(lo_row - kv0);
                    int64_t v = (int64_t)x.lkv - kv0;
                    if (a.causal) {
                        const int64_t vc = qpos - a.kv_offset - kv0 + 1;
                        v = vc < v ? vc : v;
                    }
                    lim = v < 0 ? 0 : (v > BN ? BN : (int)v);
                }
                const float mx = masked ? row_max<true>(tS, lo, lim) : row_max<false>(tS, lo, lim);
                const float mx2 = mx * c2;
                // Lazy rescale: move this row's reference max only when the tile
                // max exceeds it by more than 2^8.  The decision is per row, but
                // tcgen05.ld/st are warp-collective, so the O rescale runs for the
                // whole warp whenever any of its rows needs it (alpha = 1 elsewhere).
                float alpha = 1.f;
                bool resc = false;
                if (mx2 > m_run + kRescaleThreshold) {
                    if (m_run != -INFINITY) {
                        alpha = ex2(m_run - mx2);
                        l *= alpha;
                        resc = true;
                    }
                    m_run = mx2;
                }
                if (j > x.j0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t u[32];
                        tmem_ld32(tO + c * 32, u);
#pragma unroll
                        for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                        tmem_st32(tO + c * 32, u);
                    }
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                // Pass 2: P = exp2(s * c2 - m), row sum, bf16 P written over S.
                l += masked ? row_exp<true>(tS, lo, lim, c2, m_use) : row_exp<false>(tS, lo, lim, c2, m_use);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&p_full[w]);
            }
            if (!ok) break;
            // ---- epilogue: O = O_acc / l, lse = ln(sum exp(s))
            const bool valid_row = row < x.lq;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t orow = (((int64_t)x.tb * a.Lq + x.base + row) * a.H + x.h) * D + x.s * a.o_piece_stride;
            if (x.n_kv > x.j0) {
                ok = __all_sync(0xffffffffu, mbar_wait_acc(&o_full[w], qi & 1, abort_flag, a.err, nullptr));
                if (!ok) break;
                tc_fence_after();
                ++qi;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t u[32];
                    tmem_ld32(tO + c * 32, u);
                    if (valid_row) {
                        if (OUT_F32) {
                            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.O) + orow + c * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                dst[e] = make_float4(__uint_as_float(u[4 * e]) * inv, __uint_as_float(u[4 * e + 1]) * inv,
                                                     __uint_as_float(u[4 * e + 2]) * inv,
                                                     __uint_as_float(u[4 * e + 3]) * inv);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.O) + orow + c * 32);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                uint4 v;
                                v.x = pack_bf16(__uint_as_float(u[8 * e + 0]) * inv, __uint_as_float(u[8 * e + 1]) * inv);
                                v.y = pack_bf16(__uint_as_float(u[8 * e + 2]) * inv, __uint_as_float(u[8 * e + 3]) * inv);
                                v.z = pack_bf16(__uint_as_float(u[8 * e + 4]) * inv, __uint_as_float(u[8 * e + 5]) * inv);
                                v.w = pack_bf16(__uint_as_float(u[8 * e + 6]) * inv, __uint_as_float(u[8 * e + 7]) * inv);
                                dst[e] = v;
                            }
                        }
                    }
                }
                tc_fence_before();
            } else if (valid_row) {
                for (int c = 0; c < D; ++c) {
                    if (OUT_F32) static_cast<float*>(a.O)[orow + c] = 0.f;
                    else static_cast<__nv_bfloat16*>(a.O)[orow + c] = __float2bfloat16_rn(0.f);
                }
            }
            if (valid_row)
                a.lse[((int64_t)x.tb * a.H + x.h) * a.Lq + x.base + row + x.s * a.lse_piece_stride] = l > 0.f ? (m_run + __log2f(l)) * kLn2 : -INFINITY;
        }
        if (threadIdx.x == 128) trace_count(a.trace, a.trace_cap, 5, t);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) trace_cta(a.trace, a.trace_cap, t_start, it_end - it_begin);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// 4-D bf16 tensor map over [B, L, heads, D] (element strides sb, ss, sh; D
// contiguous) with a {64, 1, 128, 1} box and the 128-byte swizzle.
bool make_tmap_bshd(void* map, const void* base, int B, int L, int heads, int D, int64_t sb,
                    int64_t ss, int64_t sh) {
    CUtensorMap* m = static_cast<CUtensorMap*>(map);
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(L > 0 ? L : 1), (cuuint64_t)(B > 0 ? B : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)sh * 2, (cuuint64_t)ss * 2, (cuuint64_t)sb * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    // A stride of a size-1 dimension is never used; keep it valid for the encoder.
    if (heads == 1 && strides[0] == 0) strides[0] = 16;
    if (strides[0] == 0) strides[0] = 16;
    if (strides[1] == 0) strides[1] = 16;
    if (strides[2] == 0) strides[2] = 16;
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, bool OUT_F32>
static dfa_status launch(const AttnProblem& p, const void* q, const void* k, const void* v, void* O,
                         float* lse, const WorkList* wl, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    // With no keys nothing is loaded from K/V; any valid address serves the encoder.
    if (p.Lkv == 0) k = v = q;
    const int tB = p.seq ? 1 : p.B;   // a packed batch is one tensor row of T tokens
    if (!make_tmap_bshd(&mq, q, tB, p.Lq, p.H, D, p.q_sb, p.q_ss, p.q_sh) ||
        !make_tmap_bshd(&mk, k, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh) ||
        !make_tmap_bshd(&mv, v, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh))
        return fail(DFA_ERR_CUDA, "tensor map encoding failed");
    FwdArgs a{};
    a.seq = p.seq;
    a.B = p.B; a.H = p.H; a.Hkv = p.Hkv; a.Lq = p.Lq; a.Lkv = p.Lkv;
    a.q_offset = p.q_offset; a.kv_offset = p.kv_offset; a.causal = p.causal;
    a.win_c = p.win_c; a.win_w = p.causal ? p.win_w : 0;
    a.scale_log2 = p.scale * kLog2e;
    a.O = O; a.lse = lse;
    a.n_units = wl ? wl->n_units : (p.Lq + kBlockRows - 1) / kBlockRows;
    a.err = device_error_flag();
    a.trace = cta_trace(&a.trace_cap);
    int grid;
    a.n_split = 1;
    if (wl) {
        a.wl_offsets = wl->offsets;
        a.wl_items = wl->items;
        grid = wl->n_workers;
        if (wl->n_split > 1) {
            if (!OUT_F32 || wl->piece_tiles <= 0) return fail(DFA_ERR_INVALID_ARG, "split-kv pieces need fp32 partials");
            a.n_split = wl->n_split;
            a.piece_tiles = wl->piece_tiles;
            a.o_piece_stride = (int64_t)p.B * p.Lq * p.H * D;
            a.lse_piece_stride = (int64_t)p.B * p.H * p.Lq;
        }
    } else {
        a.wl_offsets = nullptr;
        a.wl_items = nullptr;
        grid = p.B * p.H * a.n_units;
    }
    auto kern = a.win_w > 0 ? fwd_tc_kernel<D, OUT_F32, true> : fwd_tc_kernel<D, OUT_F32, false>;
    const int smem = Cfg<D>::kSmem;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "fwd_tc: shared memory attribute");
    if (grid <= 0) return DFA_OK;
    kern<<<grid, kThreads, smem, s>>>(mq, mk, mv, a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "fwd_tc launch: %s", cudaGetErrorString(e));
}

dfa_status tc_fwd(const AttnProblem& p, const void* q, const void* k, const void* v, void* O,
                  bool O_is_f32, float* lse, const WorkList* wl, cudaStream_t s) {
    if (p.B == 0 || p.Lq == 0) return DFA_OK;
    if (p.D == 128) return O_is_f32 ? launch<128, true>(p, q, k, v, O, lse, wl, s) : launch<128, false>(p, q, k, v, O, lse, wl, s);
    return O_is_f32 ? launch<64, true>(p, q, k, v, O, lse, wl, s) : launch<64, false>(p, q, k, v, O, lse, wl, s);
}

}  // namespace dfa
