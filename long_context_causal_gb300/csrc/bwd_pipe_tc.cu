// bwd_pipe_tc.cu -- pipelined tcgen05 causal attention backward, head dim 128.
//
// Same mathematics and contract as bwd_tc.cu (DISTFLASHATTN §3.3, paperlayer.ai
// summary of arXiv 2310.03294: the backward reads the saved output and
// log-sum-exp and never re-runs the forward; P is recomputed from lse):
//   dV_j += P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - Delta_i),
//   dK_j += dS_ij q_i,  dQ_i += dS_ij k_j           (scale applied at the end).
//
// What differs from bwd_tc.cu is the schedule.  The softmax-gradient work of
// a (128-key x 128-query) tile is split into two phases:
//   phase 1  P^T = exp2(S^T c + nlse2)  -- needs S^T only; P^T goes to TMEM
//            (bf16, over S^T) for dV and stays in registers (bf16 pairs);
//   phase 2  dS^T = P^T (dP^T - Delta) -- needs dP^T; dS^T goes to swizzled
//            shared memory for dK and dQ.
// so the tensor cores can run dV(n) and S^T(n+1) as soon as phase 1 of tile n
// is done, and the exponentials of tile n+1 overlap dK/dQ of tile n:
//   MMA order per tile n:  [phase1(n)] dV(n), S^T(n+1)  [phase2(n)] dQ^T(n),
//                          dK(n)  [drain(n)] dP^T(n+1)
// (dQ^T before dK, so the drain reads dQ^T out of TMEM while dK runs).
//   P/dS warps per tile:   phase1(n), phase2(n), phase1(n+1), ...
// All MMAs are N = 128 or 128-row wide (few, large instructions: one thread
// issues them all).  Two warpgroups split the 128 query columns (two warps
// per SM sub-partition hide each other's latency); two more drain dQ.
//
// TMEM columns: dV [0,128) dK [128,256) S^T [256,384) (P^T of query half h at
// [256+64h, 256+64h+32)), dP^T / dQ^T [384,512).
// Roles (640 threads, one CTA per SM, persistent over the work list):
// warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM owner, warps 4-11
// P/dS (two warpgroups by query half) and the dK/dV epilogue, warps 12-19
// dQ drain (two warpgroups by query half: dQ^T out of TMEM, 16-byte fp32
// reductions; a warp instruction covers four full 128-byte dQ rows).
// dQ^T shares its TMEM columns with the next tile's dP^T, so the drain reads
// all of its 64 columns into registers and releases the columns before any
// reduction: the next dP^T then waits for two TMEM loads, not for 64 KB of
// reductions.  The registers for that come from a setmaxnreg split (the
// control warpgroup needs few).
// The MMA thread polls its barriers (bounded, loop out of line) and moves its
// shared-memory descriptors with 32-bit adds on their low word: it shares its
// sub-partition's issue slots with four busy warps, so every instruction it
// saves per MMA shortens the tensor pipe's idle gaps.
// Trace wait slots (cycles): 0 P/dS dP^T, 5 P/dS Q + S^T, 6 P/dS accumulators,
// 7 drain; slots 1-4 stay 0 (the MMA thread's waits carry no trace hook).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dfa {
namespace {

using namespace ptx;

constexpr int kThreads = 640;
constexpr int BT = 128;          // key rows per work item; query rows per tile
constexpr int D = 128;
constexpr int kTile = BT * D * 2;                  // 32 KB bf16 tile
constexpr int kSide = 1024;                        // nlse2[128] + Delta[128] per query tile
constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 4 * kTile, kOffDS = 6 * kTile;
constexpr int kOffSide = kOffDS + 32768;
constexpr int kOffBar = kOffSide + 2 * kSide;
constexpr int kSmem = kOffBar + 256;
static_assert(kSmem <= 232448, "shared memory");

constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;

// Register split (setmaxnreg).  The kernel launches with kLaunchRegs per
// thread (640 x 96 = 61440); the control warpgroup (TMA, MMA, TMEM owner, one
// idle warp) and the two dQ drain warpgroups give registers up, the two P/dS
// warpgroups take them: 128 x 64 + 256 x 128 + 256 x 80 = 61440.  A drain
// thread holds its 64 dQ^T values at once.
constexpr uint32_t kLaunchRegs = 96, kCtrlRegs = 64, kPdsRegs = 128, kDrainRegs = 80;
static_assert(kThreads * kLaunchRegs <= 65536, "launch register file");
static_assert(128 * kCtrlRegs + 256 * kPdsRegs + 256 * kDrainRegs <= kThreads * kLaunchRegs, "register split");

struct Args {
    int B, H, Hkv, Lq, Lkv, S_pad, causal;
    int rel;                      // kv_offset - q_offset (a multiple of 128)
    int64_t q_off, kv_off;        // absolute positions of the first query and key row
    int64_t win_c;                // local window: chunk length ...
    int win_w;                    // ... and chunks per window (0: none)
    int acc_f32;                  // dK/dV: fp32 accumulate (+=) instead of bf16 store
    float scale, c2;
    const float* nlse2;
    const float* delta;
    float* dq_acc;                // [B, H, acc_rows, D] fp32, zeroed by the caller
    int64_t acc_rows;             // Lq; for a packed batch the padded rows per head
    void* dK;                     // [B, Lkv, Hkv, D]
    void* dV;
    const int32_t* seq;           // packed batch: token starts [B+1], padded starts [B+1]; nullptr: dense
    const int32_t* wl_offsets;
    const int32_t* wl_items;
    int n_units;
    int n_split, piece_tiles;     // split-kv pieces of each key tile's query range (SPLIT)
    int* err;
    uint64_t* trace;
    int trace_cap;
};

// Query tiles of an item are swept upwards for key tiles in the lower half of
// the sequence and downwards for the upper half.  The balanced list gives a
// worker a key tile t and then its mirror n-1-t; sweeping both upwards would
// bring every worker's second item onto the same query tile at the same time
// (all of them end at the last tile), and their fp32 dQ reductions would then
// serialise on the same lines.  With the mirror swept downwards, workers stay
// on distinct tiles of a window of about 150 tiles.  Any order is correct:
// dK/dV accumulate and the dQ reductions commute.
struct Item {
    int b, g, t, i0, i1, n_q, ntiles;   // query tiles [i0, i1) per head; ntiles over the group's heads
    bool down;                      // sweep query tiles from the last one down
    // k-th tile of the item: head h of the group, query tile i
    __device__ __forceinline__ void tile(int k, int G, int& h, int& i) const {
        const int len = i1 - i0, r = k % len;
        h = g * G + k / len;
        i = down ? i1 - 1 - r : i0 + r;
    }
};

// VARLEN: a packed batch (a.seq set).  SPLIT: split-kv items, a piece of
// piece_tiles query tiles of a key tile's range (item value * n_split + piece);
// their dK/dV go to fp32 accumulators by reduction.  The dense kernel is a
// separate instantiation in which the sequence base is 0 and the lengths are
// the problem's, so it keeps its registers for the tile loop.
template <bool VARLEN, bool SPLIT>
__device__ __forceinline__ Item decode(const Args& a, int it) {
    Item x;
    int piece = 0;
    if constexpr (SPLIT) {
        piece = it % a.n_split;
        it /= a.n_split;
    }
    const int row = it / a.n_units, unit = it % a.n_units;
    x.b = row / a.Hkv;
    x.g = row % a.Hkv;
    int n_k = a.n_units;          // key tiles of the sequence
    if constexpr (VARLEN) {
        n_k = (a.seq[x.b + 1] - a.seq[x.b] + BT - 1) / BT;
    }
    x.t = n_k - 1 - unit;
    x.n_q = VARLEN ? n_k : (a.Lq + BT - 1) / BT;
    // first query tile that sees any key of tile t: q_offset + 128 i + 127 >= kv_offset + 128 t
    x.i0 = a.causal ? min(max(x.t + a.rel / BT, 0), x.n_q) : 0;
    x.i1 = x.n_q;
    if (a.win_w > 0) {   // local window: queries below q_hi of the tile's last key may see it
        const int64_t kp = a.kv_off + (int64_t)x.t * BT + BT - 1;
        const int64_t q_hi = (kp / a.win_c + a.win_w) * a.win_c - a.q_off;
        int64_t i1 = q_hi <= 0 ? 0 : (q_hi + BT - 1) / BT;
        if (i1 > x.n_q) i1 = x.n_q;
        x.i1 = i1 < x.i0 ? x.i0 : (int)i1;
    }
    if constexpr (SPLIT) {   // this piece's query tiles only
        const int lo = x.i0 + piece * a.piece_tiles;
        x.i1 = min(x.i1, lo + a.piece_tiles);
        x.i0 = min(lo, x.i1);
    }
    x.ntiles = (a.H / a.Hkv) * (x.i1 - x.i0);
    if (VARLEN && x.t < 0) x.ntiles = 0;   // unit past the end of a short sequence
    x.down = 2 * x.t >= n_k;
    return x;
}

// Sequence geometry of item x, selected at compile time: the dense kernel
// reads its lengths from the parameters; the packed-batch kernel re-reads the
// small, cache-resident sequence table where a value is used instead of
// holding it in registers across the tile loop (the warps here run at the
// register limit, and a few more live values cost about a tenth of the speed).
#define SEQ_LQ(x) (VARLEN ? a.seq[(x).b + 1] - a.seq[(x).b] : a.Lq)
#define SEQ_LKV(x) (VARLEN ? a.seq[(x).b + 1] - a.seq[(x).b] : a.Lkv)
#define SEQ_BASE(x) (VARLEN ? a.seq[(x).b] : 0)
#define SEQ_PBASE(x) (VARLEN ? a.seq[a.B + 1 + (x).b] : 0)
#define SEQ_TB(x) (VARLEN ? 0 : (x).b)

template <bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_pipe_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO, const Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0 && a.err) atomicExch(a.err, 2);
        return;
    }
    uint8_t* sK = smem + kOffK;
    uint8_t* sV = smem + kOffV;
    uint8_t* sQ = smem + kOffQ;
    uint8_t* sdO = smem + kOffDO;
    uint8_t* sdS = smem + kOffDS;
    uint8_t* sSide = smem + kOffSide;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* kv_full = bars + 0;
    uint64_t* kv_empty = bars + 1;
    uint64_t* q_full = bars + 2;      // [2] per tile slot
    uint64_t* q_empty = bars + 4;     // [2]
    uint64_t* do_full = bars + 6;     // [2]
    uint64_t* do_empty = bars + 8;    // [2]
    uint64_t* s_full = bars + 10;     // S^T of the tile ready
    uint64_t* dp_full = bars + 11;    // dP^T of the tile ready
    uint64_t* p_done = bars + 12;     // phase 1 done: P^T in TMEM, S^T columns read
    uint64_t* ds_done = bars + 13;    // phase 2 done: dS^T in smem, dP^T columns read
    uint64_t* dq_full = bars + 14;    // dQ^T ready
    uint64_t* dq_free = bars + 15;    // dQ^T read out
    uint64_t* kd_full = bars + 16;
    uint64_t* kd_empty = bars + 17;
    uint64_t* done = bars + 18;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 25);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int it_begin = a.wl_offsets[blockIdx.x], it_end = a.wl_offsets[blockIdx.x + 1];
    const int G = a.H / a.Hkv;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
            mbar_init(&do_full[s], 1);
            mbar_init(&do_empty[s], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_done, 2 * BT);
        mbar_init(ds_done, 2 * BT);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 2 * BT);
        mbar_init(kd_full, 1);
        mbar_init(kd_empty, 2 * BT);
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
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

    // Every warp of a warpgroup executes its warpgroup's setmaxnreg, and each
    // role's code sits inside the branch that set its budget (code reached
    // under two budgets cannot be shared, hence one barrier copy per branch).
    if (warp < 4) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        uint32_t n = 0, kvi = 0, kv_issued = 0, q_issued = 0, do_issued = 0;
        bool ok = true;
        uint64_t wt = 0;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            ok = ok && __all_sync(0xffffffffu, mbar_wait_acc(bar, parity, abort_flag, a.err, a.trace ? &wt : nullptr));
            return ok;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode<VARLEN, SPLIT>(a, a.wl_items[it]);
            if (x.ntiles == 0) continue;   // key tile entirely above the diagonal: nothing to do
            if (!wait(kv_empty, (kvi & 1) ^ 1)) break;
            ++kv_issued;
            if (lane == 0) {
                mbar_arrive_expect_tx(kv_full, 2 * kTile);
                for (int blk = 0; blk < 2; ++blk) {
                    tma_load_4d(sK + blk * 16384, &tmK, kv_full, blk * 64, x.g, SEQ_BASE(x) + x.t * BT, SEQ_TB(x));
                    tma_load_4d(sV + blk * 16384, &tmV, kv_full, blk * 64, x.g, SEQ_BASE(x) + x.t * BT, SEQ_TB(x));
                }
            }
            __syncwarp();
            for (int k = 0; k < x.ntiles && ok; ++k, ++n) {
                int h, i;
                x.tile(k, G, h, i);
                const size_t side_off = ((size_t)SEQ_TB(x) * a.H + h) * a.S_pad + SEQ_PBASE(x) + (size_t)i * BT;
                const uint32_t s = n & 1, ph = ((n >> 1) & 1) ^ 1;
                if (!wait(&q_empty[s], ph)) break;
                ++q_issued;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&q_full[s], kTile + kSide);
                    for (int blk = 0; blk < 2; ++blk)
                        tma_load_4d(sQ + s * kTile + blk * 16384, &tmQ, &q_full[s], blk * 64, h, SEQ_BASE(x) + i * BT,
                                    SEQ_TB(x));
                    bulk_load(sSide + s * kSide, a.nlse2 + side_off, 512, &q_full[s]);
                    bulk_load(sSide + s * kSide + 512, a.delta + side_off, 512, &q_full[s]);
                }
                __syncwarp();
                if (!wait(&do_empty[s], ph)) break;
                ++do_issued;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&do_full[s], kTile);
                    for (int blk = 0; blk < 2; ++blk)
                        tma_load_4d(sdO + s * kTile + blk * 16384, &tmdO, &do_full[s], blk * 64, h,
                                    SEQ_BASE(x) + i * BT, SEQ_TB(x));
                }
                __syncwarp();
            }
            ++kvi;
        }
        if (!ok && lane == 0) {
            int dummy = 0;
            if (kv_issued) mbar_wait(kv_full, (kv_issued - 1) & 1, &dummy, nullptr);
            for (uint32_t m = (q_issued >= 2 ? q_issued - 2 : 0); m < q_issued; ++m)
                mbar_wait(&q_full[m & 1], (m >> 1) & 1, &dummy, nullptr);
            for (uint32_t m = (do_issued >= 2 ? do_issued - 2 : 0); m < do_issued; ++m)
                mbar_wait(&do_full[m & 1], (m >> 1) & 1, &dummy, nullptr);
        }
        if (lane == 0) {
            trace_count(a.trace, a.trace_cap, 6, n);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // One thread: tcgen05.mma / commit / fence and mbarrier waits are all
        // per-thread, and a lone thread keeps the gaps between MMA groups short
        // (the tensor pipe queues little ahead, so every cycle between groups is idle).
        constexpr uint32_t idS = idesc_bf16_f32(BT, BT, false, false);   // S^T, dP^T
        constexpr uint32_t idKM = idesc_bf16_f32(BT, D, false, true);    // dV, dK: B N-major
        constexpr uint32_t idQ = idesc_bf16_f32(D, BT, true, true);      // dQ^T: M = head dim
        // Descriptors as SDesc words: moved by 32-bit adds on the low word.
        auto desc = [](const void* p, uint32_t lbo) { return sdesc_words(sdesc_sw128(smem_u32(p), lbo, 1024)); };
        const SDesc dKk = desc(sK, 16), dKn = desc(sK, 16384);
        const SDesc dVk = desc(sV, 16);
        const SDesc dQk = desc(sQ, 16), dQn = desc(sQ, 16384);
        const SDesc dOk = desc(sdO, 16), dOn = desc(sdO, 16384);
        const SDesc dSk = desc(sdS, 16), dSn = desc(sdS, 16384);
        constexpr uint32_t kSlot = kTile >> 4, kRows16 = 2048 >> 4;
        auto kmaj = [](int kk) -> uint32_t { return (uint32_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4); };
        uint32_t n = 0, kvi = 0;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t parity, int slot) {
            // Not profiled, even when tracing: any profiling hook in this
            // thread's waits (a pointer select, a traced branch) cost 1-2%.
            ok = ok && mbar_wait_spin(bar, parity, abort_flag, a.err);
            (void)slot;
            if (ok) tc_fence_after();
            return ok;
        };
        auto commit = [&](uint64_t* bar) { mma_commit(bar); };
        auto issue_S = [&](uint32_t m) {   // S^T(m) = K Q_m^T
            const uint32_t s = m & 1;
            if (!wait(&q_full[s], (m >> 1) & 1, 0)) return false;
            {
                const SDesc b0 = dQk + s * kSlot;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kColS, dKk + kmaj(kk), b0 + kmaj(kk), idS, kk > 0);
            }
            commit(s_full);
            return true;
        };
        auto issue_dP = [&](uint32_t m) {  // dP^T(m) = V dO_m^T, over the drained dQ^T(m-1)
            const uint32_t s = m & 1;
            if (!wait(&do_full[s], (m >> 1) & 1, 0)) return false;
            if (m > 0 && !wait(dq_free, (m - 1) & 1, 1)) return false;
            {
                const SDesc b0 = dOk + s * kSlot;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kColDP, dVk + kmaj(kk), b0 + kmaj(kk), idS, kk > 0);
            }
            commit(dp_full);
            return true;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode<VARLEN, SPLIT>(a, a.wl_items[it]);
            if (x.ntiles == 0) continue;   // key tile entirely above the diagonal: nothing to do
            if (!wait(kv_full, kvi & 1, 0)) break;
            if (!issue_S(n) || !issue_dP(n)) break;
            for (int k = 0; k < x.ntiles && ok; ++k, ++n) {
                const uint32_t s = n & 1;
                const bool more = k + 1 < x.ntiles;
                if (k == 0 && !wait(kd_empty, (kvi & 1) ^ 1, 0)) break;
                if (!wait(p_done, n & 1, 2)) break;
                const uint32_t acc0 = k > 0 ? 1u : 0u;
                {   // dV += P^T dO: P^T of query half h at S + 64h
                    const SDesc b0 = dOn + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        mma_ts(tmem + kColDV, tmem + kColS + kk * 8 + (kk >= 4 ? 32 : 0), b0 + kk * kRows16, idKM,
                               kk > 0 ? 1u : acc0);
                }
                commit(&do_empty[s]);
                if (more && !issue_S(n + 1)) break;       // S^T columns are free after phase 1
                if (!wait(ds_done, n & 1, 3)) break;
                {   // dQ^T = K^T dS^T into the dP^T columns; drained while dK runs
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        mma_ss(tmem + kColDP, dKn + kk * kRows16, dSn + kk * kRows16, idQ, kk > 0);
                }
                commit(dq_full);
                {   // dK += dS^T Q
                    const SDesc bq = dQn + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        mma_ss(tmem + kColDK, dSk + kmaj(kk), bq + kk * kRows16, idKM, kk > 0 ? 1u : acc0);
                }
                commit(&q_empty[s]);
                if (!more) {
                    commit(kd_full);
                    commit(kv_empty);
                } else if (!issue_dP(n + 1)) {
                    break;
                }
            }
            if (!ok) break;
            ++kvi;
        }
        commit(done);
        int dummy = 0;
        mbar_wait(done, 0, &dummy, a.err);
        {
            trace_count(a.trace, a.trace_cap, 4, n);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) trace_cta(a.trace, a.trace_cap, t_start, it_end - it_begin);
    } else if (warp < 12) {
        setmaxnreg_inc<kPdsRegs>();
        // ------------------------------------------------------------ P^T / dS^T, dK/dV epilogue
        const int half = (warp - 4) / 4;                   // query columns [64 half, 64 half + 64)
        const int r = (warp % 4) * 32 + lane;              // key row == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + lane_base + kColS + half * 64;
        const uint32_t tdP = tmem + lane_base + kColDP + half * 64;
        uint8_t* blk = sdS + half * 16384;
        uint32_t n = 0, kvi = 0;
        bool ok = true;
        uint64_t wt[3] = {0, 0, 0};   // Q/S^T, dK/dV accumulators, dP^T
        auto wait = [&](uint64_t* bar, uint32_t parity, int slot) {
            ok = ok && __all_sync(0xffffffffu,
                                  mbar_wait_acc<1>(bar, parity, abort_flag, a.err, a.trace ? &wt[slot] : nullptr));
            return ok;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode<VARLEN, SPLIT>(a, a.wl_items[it]);
            if (x.ntiles == 0) continue;   // key tile entirely above the diagonal: nothing to do
            const int kvg = x.t * BT + r;
            const bool row_ok = kvg < SEQ_LKV(x);
            // local window: this key is seen by queries below q_hi (chunk-relative);
            // q_hi_tile is the lowest such bound over the tile's keys
            const int64_t q_hi = a.win_w > 0 ? ((a.kv_off + kvg) / a.win_c + a.win_w) * a.win_c - a.q_off : INT64_MAX;
            const int64_t q_hi_tile =
                a.win_w > 0 ? ((a.kv_off + (int64_t)x.t * BT) / a.win_c + a.win_w) * a.win_c - a.q_off : INT64_MAX;
            for (int k = 0; k < x.ntiles; ++k, ++n) {
                int h, i;
                x.tile(k, G, h, i);
                (void)h;
                const uint32_t s = n & 1;
                const int q0 = i * BT + half * 64;
                if (!wait(&q_full[s], (n >> 1) & 1, 0) || !wait(s_full, n & 1, 0)) break;
                tc_fence_after();
                const float* nlse2 = reinterpret_cast<const float*>(sSide + s * kSide) + half * 64;
                const float* dl = nlse2 + BT;
                // Elements outside the causal triangle or the sequence only occur on
                // the diagonal tile and on ragged edges; elsewhere no mask is applied.
                const bool full = !(a.causal && i == x.t + a.rel / BT) && (i + 1) * BT <= SEQ_LQ(x) &&
                                  (int64_t)(i + 1) * BT <= q_hi_tile &&
                                  (x.t + 1) * BT <= SEQ_LKV(x);
                // ---- phase 1: P^T = exp2(S^T c + nlse2) -> TMEM (bf16) and registers
                uint32_t u[32], pk[32];
#pragma unroll
                for (int c = 0; c < 64; c += 32) {
                    tmem_ld32(tS + c, u);
                    if (!full) {   // masked scores become -inf, so exp2 gives exactly 0
#pragma unroll
                        for (int z = 0; z < 32; ++z) {
                            const int qg = q0 + c + z;
                            if (!(row_ok && qg < SEQ_LQ(x) && !(a.causal && kvg + a.rel > qg) && qg < q_hi))
                                u[z] = 0xff800000u;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c + e);
                        pk[(c + e) / 2] = exp2_pack_bf16(__uint_as_float(u[e]), __uint_as_float(u[e + 1]), a.c2,
                                                         l4.x, l4.y);
                        pk[(c + e) / 2 + 1] = exp2_pack_bf16(__uint_as_float(u[e + 2]), __uint_as_float(u[e + 3]),
                                                             a.c2, l4.z, l4.w);
                    }
                    tmem_st16(tS + c / 2, *reinterpret_cast<uint32_t(*)[16]>(&pk[c / 2]));
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_done);
                // ---- phase 2: dS^T = P^T (dP^T - Delta) -> swizzled smem (bf16)
                if (!wait(dp_full, n & 1, 2)) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 64; c += 32) {
                    tmem_ld32(tdP + c, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint32_t dk[4];
#pragma unroll
                        for (int w = 0; w < 8; w += 4) {
                            const float4 d4 = *reinterpret_cast<const float4*>(dl + c + e + w);
                            const float2 p01 =
                                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[(c + e + w) / 2]));
                            const float2 p23 =
                                __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[(c + e + w) / 2 + 1]));
                            dk[w / 2] = ds_pack_bf16(p01.x, p01.y, __uint_as_float(u[e + w]),
                                                     __uint_as_float(u[e + w + 1]), d4.x, d4.y);
                            dk[w / 2 + 1] = ds_pack_bf16(p23.x, p23.y, __uint_as_float(u[e + w + 2]),
                                                         __uint_as_float(u[e + w + 3]), d4.z, d4.w);
                        }
                        *reinterpret_cast<uint4*>(blk + sw128_offset(r, c + e)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(ds_done);
            }
            if (!ok) break;
            // ---- epilogue: dV = acc, dK = scale * acc into [B, Lkv, Hkv, D] (bf16 store,
            // or fp32 += for a chunk pair's partial gradients); this half's columns
            if (!wait(kd_full, kvi & 1, 1)) break;
            tc_fence_after();
            const int64_t orow = (((int64_t)SEQ_TB(x) * a.Lkv + SEQ_BASE(x) + kvg) * a.Hkv + x.g) * D;
#pragma unroll 1
            for (int c = half * 2; c < half * 2 + 2; ++c) {
                uint32_t uv[32], uk[32];
                tmem_ld32x2(tmem + lane_base + kColDV + c * 32, tmem + lane_base + kColDK + c * 32, uv, uk);
                if constexpr (SPLIT) {   // a piece's partial: fp32 reductions, other pieces add to the same rows
                    if (row_ok) {
                        float* pv = static_cast<float*>(a.dV) + orow + c * 32;
                        float* pkk = static_cast<float*>(a.dK) + orow + c * 32;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            red_add_v4(pv + 4 * e, __uint_as_float(uv[4 * e]), __uint_as_float(uv[4 * e + 1]),
                                       __uint_as_float(uv[4 * e + 2]), __uint_as_float(uv[4 * e + 3]));
                            red_add_v4(pkk + 4 * e, a.scale * __uint_as_float(uk[4 * e]),
                                       a.scale * __uint_as_float(uk[4 * e + 1]), a.scale * __uint_as_float(uk[4 * e + 2]),
                                       a.scale * __uint_as_float(uk[4 * e + 3]));
                        }
                    }
                } else if (row_ok && a.acc_f32) {
                    float4* pv = reinterpret_cast<float4*>(static_cast<float*>(a.dV) + orow + c * 32);
                    float4* pkk = reinterpret_cast<float4*>(static_cast<float*>(a.dK) + orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float4 v = pv[e], w = pkk[e];
                        v.x += __uint_as_float(uv[4 * e]);
                        v.y += __uint_as_float(uv[4 * e + 1]);
                        v.z += __uint_as_float(uv[4 * e + 2]);
                        v.w += __uint_as_float(uv[4 * e + 3]);
                        w.x += a.scale * __uint_as_float(uk[4 * e]);
                        w.y += a.scale * __uint_as_float(uk[4 * e + 1]);
                        w.z += a.scale * __uint_as_float(uk[4 * e + 2]);
                        w.w += a.scale * __uint_as_float(uk[4 * e + 3]);
                        pv[e] = v;
                        pkk[e] = w;
                    }
                } else if (row_ok) {
                    uint4* pv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dV) + orow + c * 32);
                    uint4* pkk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dK) + orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 v, w;
                        v.x = pack_bf16(__uint_as_float(uv[8 * e + 0]), __uint_as_float(uv[8 * e + 1]));
                        v.y = pack_bf16(__uint_as_float(uv[8 * e + 2]), __uint_as_float(uv[8 * e + 3]));
                        v.z = pack_bf16(__uint_as_float(uv[8 * e + 4]), __uint_as_float(uv[8 * e + 5]));
                        v.w = pack_bf16(__uint_as_float(uv[8 * e + 6]), __uint_as_float(uv[8 * e + 7]));
                        w.x = pack_bf16(a.scale * __uint_as_float(uk[8 * e + 0]), a.scale * __uint_as_float(uk[8 * e + 1]));
                        w.y = pack_bf16(a.scale * __uint_as_float(uk[8 * e + 2]), a.scale * __uint_as_float(uk[8 * e + 3]));
                        w.z = pack_bf16(a.scale * __uint_as_float(uk[8 * e + 4]), a.scale * __uint_as_float(uk[8 * e + 5]));
                        w.w = pack_bf16(a.scale * __uint_as_float(uk[8 * e + 6]), a.scale * __uint_as_float(uk[8 * e + 7]));
                        pv[e] = v;
                        pkk[e] = w;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(kd_empty);
            ++kvi;
        }
        if (threadIdx.x == 128) {
            trace_count(a.trace, a.trace_cap, 5, n);
            trace_wait(a.trace, a.trace_cap, 5, wt[0]);
            trace_wait(a.trace, a.trace_cap, 6, wt[1]);
            trace_wait(a.trace, a.trace_cap, 0, wt[2]);
        }
        tc_fence_before();
        __syncthreads();
    } else {
        setmaxnreg_dec<kDrainRegs>();
        // ------------------------------------------------------------ dQ drain
        // TMEM lane = head-dim element of dQ^T; column c = query row i*128 + c.
        // Two warpgroups: warpgroup dg drains query columns [64 dg, 64 dg + 64).
        const int dg = (warp - 12) / 4;
        const uint32_t tdQ = tmem + ((uint32_t)((warp % 4) * 32) << 16) + kColDP + dg * 64;
        uint32_t n = 0;
        bool ok = true;
        uint64_t wt = 0;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const Item x = decode<VARLEN, SPLIT>(a, a.wl_items[it]);
            if (x.ntiles == 0) continue;   // key tile entirely above the diagonal: nothing to do
            const int s_pbase = SEQ_PBASE(x), s_len = SEQ_LQ(x);   // once per item
            for (int k = 0; k < x.ntiles; ++k, ++n) {
                int h, i;
                x.tile(k, G, h, i);
                ok = __all_sync(0xffffffffu, mbar_wait_acc<2>(dq_full, n & 1, abort_flag, a.err, a.trace ? &wt : nullptr));
                if (!ok) break;
                tc_fence_after();
                // dQ accumulator is head-major [B, H, S, D]: the tile is one contiguous
                // 64 KB block.  Each group of four query columns is transposed inside
                // lane quads, so lane 4q+m adds head-dim elements 4q..4q+3 of query
                // column m with one 16-byte reduction and a warp instruction covers
                // four full 128-byte rows.
                const int m = lane & 3;
                float* base = a.dq_acc + (((int64_t)SEQ_TB(x) * a.H + h) * (VARLEN ? a.acc_rows : a.Lq) + s_pbase +
                                          (int64_t)i * BT + m) * D +
                              (warp % 4) * 32 + (lane >> 2) * 4;
                const int nq = min(BT, s_len - i * BT) - dg * 64;
                // This warpgroup's 64 query columns are read at once, then TMEM is
                // released (relaxed: the arrival must not wait for any reduction).
                uint32_t v[64];
                tmem_ld32x2(tdQ, tdQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[0]),
                            *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tc_fence_before();
                mbar_arrive_relaxed(dq_free);
#pragma unroll
                for (int g = 0; g < 16; ++g) {
                    float xq[4] = {__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                   __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])};
                    quad_transpose(xq, lane);
                    if (4 * g + m < nq)
                        red_add_v4(base + (dg * 64 + 4 * g) * D, xq[0], xq[1], xq[2], xq[3]);
                }
            }
        }
        if (threadIdx.x == 384) {
            trace_count(a.trace, a.trace_cap, 7, n);
            trace_wait(a.trace, a.trace_cap, 7, wt);
        }
        tc_fence_before();
        __syncthreads();
    }
}

#undef SEQ_LQ
#undef SEQ_LKV
#undef SEQ_BASE
#undef SEQ_PBASE
#undef SEQ_TB

}  // namespace

dfa_status tc_bwd_pipelined(const AttnProblem& p, const void* q, const void* k, const void* v, const void* dO,
                            const float* nlse2, const float* delta, int S_pad, float* dq_acc, void* dK, void* dV,
                            bool acc_f32, const WorkList* wl, cudaStream_t s) {
    if (p.D != D) return fail(DFA_ERR_UNSUPPORTED, "pipelined backward needs D = 128");
    const int64_t rel = p.kv_offset - p.q_offset;
    if (rel % BT != 0 || rel > (int64_t)1 << 30 || rel < -((int64_t)1 << 30))
        return fail(DFA_ERR_UNSUPPORTED, "tensor-core backward needs kv_offset - q_offset a multiple of 128");
    alignas(64) CUtensorMap mq, mk, mv, mdo;
    const int tB = p.seq ? 1 : p.B;   // a packed batch is one tensor row of T tokens
    if (!make_tmap_bshd(&mq, q, tB, p.Lq, p.H, D, p.q_sb, p.q_ss, p.q_sh) ||
        !make_tmap_bshd(&mdo, dO, tB, p.Lq, p.H, D, p.q_sb, p.q_ss, p.q_sh) ||
        !make_tmap_bshd(&mk, k, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh) ||
        !make_tmap_bshd(&mv, v, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh))
        return fail(DFA_ERR_CUDA, "tensor map encoding failed");
    Args a{};
    a.seq = p.seq;
    a.acc_rows = p.seq ? S_pad : p.Lq;
    a.B = p.B; a.H = p.H; a.Hkv = p.Hkv; a.Lq = p.Lq; a.Lkv = p.Lkv; a.S_pad = S_pad; a.causal = p.causal;
    a.rel = (int)rel; a.acc_f32 = acc_f32;
    a.q_off = p.q_offset; a.kv_off = p.kv_offset; a.win_c = p.win_c; a.win_w = p.causal ? p.win_w : 0;
    a.scale = p.scale; a.c2 = p.scale * 1.4426950408889634f;
    a.nlse2 = nlse2; a.delta = delta; a.dq_acc = dq_acc;
    a.dK = dK;
    a.dV = dV;
    a.wl_offsets = wl->offsets; a.wl_items = wl->items; a.n_units = wl->n_units;
    a.err = device_error_flag();
    a.trace = cta_trace(&a.trace_cap);
    const bool split = wl->n_split > 1;
    if (split && (!acc_f32 || p.seq || wl->piece_tiles <= 0))
        return fail(DFA_ERR_INVALID_ARG, "split-kv backward pieces need fp32 dK/dV accumulators");
    a.n_split = wl->n_split;
    a.piece_tiles = wl->piece_tiles;
    auto kern = p.seq ? bwd_pipe_kernel<true, false> : split ? bwd_pipe_kernel<false, true> : bwd_pipe_kernel<false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "bwd_pipe: shared memory attribute");
    // The setmaxnreg split assumes the launch register count; a different
    // count could leave a warpgroup's register increase waiting forever.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || fa.numRegs != (int)kLaunchRegs)
        return fail(DFA_ERR_CUDA, "bwd_pipe: built with %d registers per thread, the register split needs %u",
                    fa.numRegs, kLaunchRegs);
    kern<<<wl->n_workers, kThreads, kSmem, s>>>(mq, mk, mv, mdo, a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "bwd_pipe launch: %s", cudaGetErrorString(e));
}

}  // namespace dfa
