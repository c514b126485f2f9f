// bwd_tc.cu -- tcgen05 tensor-core causal attention backward for sm_103a.
//
// DISTFLASHATTN (paperlayer.ai summary of arXiv 2310.03294) §3.3: with
// rematerialization-aware checkpointing the attention forward runs once; the
// backward reads the SAVED output and log-sum-exp and never re-runs it.  Here
// P is recomputed tile by tile from the saved lse (P is never stored), and
//   dV_j += P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - Delta_i),
//   dK_j += dS_ij q_i,  dQ_i += dS_ij k_j         (scale applied at the end)
// with Delta_i = dO_i . O_i precomputed from the saved O.
//
// One CTA owns a 128-key tile of one key/value head (persistent over a
// host-built work list) and loops over every visible 128-row query tile of
// every query head of its GQA group, keeping dK and dV in TMEM for the whole
// loop; dQ partials leave through fp32 atomics into a workspace accumulator.
//
// Roles (384 threads, one CTA per SM):
//   warp 0      TMA producer: K, V once per work item; Q_i, dO_i (2-slot rings)
//               plus the query tile's lse and Delta (bulk copies).
//   warp 1      MMA issuer (one thread), per query tile:
//                 S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q,
//                 dQ = dS K (stored transposed, dQ^T = K^T dS^T, for D = 128).
//   warp 2      TMEM allocation.
//   warps 4-7   one key row per thread: P^T = exp2(S^T c + nlse2),
//               dS^T = P^T (dP^T - Delta); P^T (bf16) back into TMEM over S^T,
//               dS^T (bf16) into swizzled shared memory where it serves as the
//               K-major A operand of dK and the M-major A operand of dQ; at the
//               end of an item the dK/dV epilogue.
//   warps 8-11  dQ partial out of TMEM, then fp32 atomic adds into the
//               accumulator (D = 128: one head-dim element per thread, so a
//               warp's adds cover 128 contiguous bytes of one dQ row).
//
// TMEM columns: dV [0,128) dK [128,256) S^T/P^T [256,384) dP^T/dQ [384,512).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dfa {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int BT = 128;   // rows per query / key tile
constexpr int kSide = 1024;   // per query slot: nlse2[128] and Delta[128] (fp32)

template <int D>
struct BCfg {
    static constexpr int kTile = BT * D * 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kTile;
    static constexpr int kOffQ = 2 * kTile;            // 2 slots
    static constexpr int kOffDO = 4 * kTile;           // 2 slots
    static constexpr int kOffDS = 6 * kTile;           // 128 x 128 bf16 = 32 KB
    static constexpr int kOffSide = kOffDS + 32768;    // 2 x kSide
    static constexpr int kOffBar = kOffSide + 2 * kSide;
    static constexpr int kSmem = kOffBar + 256;
};
static_assert(BCfg<128>::kSmem <= 232448, "backward shared memory");

struct BwdArgs {
    int B, H, Hkv, S, S_pad, causal;
    int64_t win_c;                // local window: chunk length ...
    int win_w;                    // ... and chunks per window (0: none)
    float scale, c2;              // c2 = scale * log2(e)
    const float* nlse2;            // [B, H, S_pad]  -lse * log2(e)
    const float* delta;           // [B, H, S_pad]
    float* dq_acc;                // [B, H, acc_rows, D] fp32, zeroed by the caller
    int64_t acc_rows;             // S; for a packed batch the padded rows per head
    __nv_bfloat16* dK;            // [B, S, Hkv, D]
    __nv_bfloat16* dV;
    const int32_t* seq;           // packed batch: token starts [B+1], padded starts [B+1]; nullptr: dense
    const int32_t* wl_offsets;
    const int32_t* wl_items;
    int n_units;                  // key tiles per (batch, kv head)
    int* err;
    uint64_t* trace;              // optional per-CTA timeline (nullptr: off)
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
struct BItem {
    int b, g, t, i0, i1, n_q, ntiles;   // query tiles [i0, i1) per head
    bool down;                      // sweep query tiles from the last one down
    int base, pbase, len;           // packed batch: first token, first padded row, tokens of the sequence
    // k-th tile of the item: head hh of the group (0..G-1), query tile i
    __device__ __forceinline__ void tile(int k, int& hh, int& i) const {
        const int len = i1 - i0, r = k % len;
        hh = k / len;
        i = down ? i1 - 1 - r : i0 + r;
    }
};

// VARLEN: a packed batch (a.seq set), compiled as its own instantiation so
// the dense kernel reads its lengths straight from the parameters.
template <bool VARLEN>
__device__ __forceinline__ BItem bdecode(const BwdArgs& a, int it) {
    BItem x;
    const int row = it / a.n_units, unit = it % a.n_units;
    x.b = row / a.Hkv;
    x.g = row % a.Hkv;
    int n_k = a.n_units;                 // key tiles of the sequence
    if constexpr (VARLEN) {
        x.base = a.seq[x.b];
        x.pbase = a.seq[a.B + 1 + x.b];
        x.len = a.seq[x.b + 1] - x.base;
        n_k = (x.len + BT - 1) / BT;
    }
    x.t = n_k - 1 - unit;                // unit u costs u + 1 query tiles per head
    x.n_q = ((VARLEN ? x.len : a.S) + BT - 1) / BT;
    x.i0 = a.causal ? x.t : 0;
    x.i1 = x.n_q;
    if (a.win_w > 0) {   // local window: queries below q_hi of the tile's last key may see it
        const int64_t q_hi = (((int64_t)x.t * BT + BT - 1) / a.win_c + a.win_w) * a.win_c;
        int64_t i1 = (q_hi + BT - 1) / BT;
        if (i1 > x.n_q) i1 = x.n_q;
        x.i1 = i1 < x.i0 ? x.i0 : (int)i1;
    }
    x.ntiles = (a.H / a.Hkv) * (x.i1 - x.i0);
    if (VARLEN && x.t < 0) x.ntiles = 0;   // unit past the end of a short sequence
    x.down = 2 * x.t >= n_k;
    return x;
}

// Sequence geometry of item x (see bdecode).
#define SEQ_LEN(x) (VARLEN ? (x).len : a.S)
#define SEQ_BASE(x) (VARLEN ? (x).base : 0)
#define SEQ_PBASE(x) (VARLEN ? (x).pbase : 0)
#define SEQ_TB(x) (VARLEN ? 0 : (x).b)

template <int D, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const BwdArgs a) {
    using C = BCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {            // the swizzled layouts need a 1 KB aligned base
        if (threadIdx.x == 0 && a.err) atomicExch(a.err, 2);
        return;
    }
    uint8_t* sK = smem + C::kOffK;
    uint8_t* sV = smem + C::kOffV;
    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sdO = smem + C::kOffDO;
    uint8_t* sdS = smem + C::kOffDS;
    uint8_t* sSide = smem + C::kOffSide;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* kv_full = bars + 0;
    uint64_t* kv_empty = bars + 1;
    uint64_t* q_full = bars + 2;      // [2]
    uint64_t* q_empty = bars + 4;     // [2]
    uint64_t* do_full = bars + 6;     // [2]
    uint64_t* do_empty = bars + 8;    // [2]
    uint64_t* s_full = bars + 10;
    uint64_t* dp_full = bars + 11;
    uint64_t* pds_full = bars + 12;
    uint64_t* dq_full = bars + 13;
    uint64_t* dq_free = bars + 14;
    uint64_t* kd_full = bars + 15;
    uint64_t* kd_empty = bars + 16;
    uint64_t* done = bars + 17;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 21);

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
        mbar_init(pds_full, BT);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, BT);
        mbar_init(kd_full, 1);
        mbar_init(kd_empty, BT);
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
    constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 384;

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
            const BItem x = bdecode<VARLEN>(a, a.wl_items[it]);
            if (!wait(kv_empty, (kvi & 1) ^ 1)) break;
            ++kv_issued;
            if (lane == 0) {
                mbar_arrive_expect_tx(kv_full, 2 * C::kTile);
                for (int blk = 0; blk < D / 64; ++blk) {
                    tma_load_4d(sK + blk * 16384, &tmK, kv_full, blk * 64, x.g, SEQ_BASE(x) + x.t * BT, SEQ_TB(x));
                    tma_load_4d(sV + blk * 16384, &tmV, kv_full, blk * 64, x.g, SEQ_BASE(x) + x.t * BT, SEQ_TB(x));
                }
            }
            __syncwarp();
            for (int k = 0; k < x.ntiles && ok; ++k, ++n) {
                int hh, i;
                x.tile(k, hh, i);
                const int h = x.g * G + hh;
                const size_t side_off = ((size_t)SEQ_TB(x) * a.H + h) * a.S_pad + SEQ_PBASE(x);
                const uint32_t s = n & 1, ph = ((n >> 1) & 1) ^ 1;
                if (!wait(&q_empty[s], ph)) break;
                ++q_issued;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&q_full[s], C::kTile + kSide);
                    for (int blk = 0; blk < D / 64; ++blk)
                        tma_load_4d(sQ + s * C::kTile + blk * 16384, &tmQ, &q_full[s], blk * 64, h, SEQ_BASE(x) + i * BT,
                                    SEQ_TB(x));
                    bulk_load(sSide + s * kSide, a.nlse2 + side_off + i * BT, 512, &q_full[s]);
                    bulk_load(sSide + s * kSide + 512, a.delta + side_off + i * BT, 512, &q_full[s]);
                }
                __syncwarp();
                if (!wait(&do_empty[s], ph)) break;
                ++do_issued;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&do_full[s], C::kTile);
                    for (int blk = 0; blk < D / 64; ++blk)
                        tma_load_4d(sdO + s * C::kTile + blk * 16384, &tmdO, &do_full[s], blk * 64, h,
                                    SEQ_BASE(x) + i * BT, SEQ_TB(x));
                }
                __syncwarp();
            }
            ++kvi;
        }
        if (!ok && lane == 0) {
            // Aborted: wait (bounded) for the newest copy into each buffer to land.
            int dummy = 0;
            if (kv_issued) mbar_wait(kv_full, (kv_issued - 1) & 1, &dummy, nullptr);
            for (uint32_t m = (q_issued >= 2 ? q_issued - 2 : 0); m < q_issued; ++m)
                mbar_wait(&q_full[m & 1], (m >> 1) & 1, &dummy, nullptr);
            for (uint32_t m = (do_issued >= 2 ? do_issued - 2 : 0); m < do_issued; ++m)
                mbar_wait(&do_full[m & 1], (m >> 1) & 1, &dummy, nullptr);
        }
        if (lane == 0) {
            trace_count(a.trace, a.trace_cap, 6, n);
            trace_wait(a.trace, a.trace_cap, 0, wt);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idS = idesc_bf16_f32(BT, BT, false, false);     // S^T, dP^T
        const uint32_t idKM = idesc_bf16_f32(BT, D, false, true);      // dV, dK: A K-major, B N-major
        // dQ (D = 64): M = query rows; dQ^T (D = 128): M = head dim.  A, B both MN-major.
        const uint32_t idQ = D == 128 ? idesc_bf16_f32(D, BT, true, true) : idesc_bf16_f32(BT, D, true, true);
        // Descriptors are built once and advanced by adding (byte offset / 16)
        // (start-address field = addr >> 4, shared addresses < 256 KB): a short
        // issue loop is what lets one thread keep the tensor core busy.
        const uint64_t dKk = sdesc_sw128(smem_u32(sK), 16, 1024), dKn = sdesc_sw128(smem_u32(sK), 16384, 1024);
        const uint64_t dVk = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t dQk = sdesc_sw128(smem_u32(sQ), 16, 1024), dQn = sdesc_sw128(smem_u32(sQ), 16384, 1024);
        const uint64_t dOk = sdesc_sw128(smem_u32(sdO), 16, 1024), dOn = sdesc_sw128(smem_u32(sdO), 16384, 1024);
        const uint64_t dSk = sdesc_sw128(smem_u32(sdS), 16, 1024), dSn = sdesc_sw128(smem_u32(sdS), 16384, 1024);
        constexpr uint64_t kSlot = C::kTile >> 4, kRows16 = 2048 >> 4;
        auto kmaj = [](int kk) -> uint64_t { return (uint64_t)(((kk / 4) * 16384 + (kk % 4) * 32) >> 4); };
        uint32_t n = 0, kvi = 0;
        bool ok = true;
        uint64_t wt[4] = {0, 0, 0, 0};   // loads, dq_free, pds_full, kv_full + kd_empty
        auto wait = [&](uint64_t* bar, uint32_t parity, int slot) {
            ok = ok && __all_sync(0xffffffffu,
                                  mbar_wait_acc(bar, parity, abort_flag, a.err, a.trace ? &wt[slot] : nullptr));
            if (ok) tc_fence_after();
            return ok;
        };
        auto commit = [&](uint64_t* bar) {
            if (lane == 0) mma_commit(bar);
            __syncwarp();
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const BItem x = bdecode<VARLEN>(a, a.wl_items[it]);
            if (!wait(kv_full, kvi & 1, 3)) break;
            for (int k = 0; k < x.ntiles; ++k, ++n) {
                const uint32_t s = n & 1, ph = (n >> 1) & 1;
                if (!wait(&q_full[s], ph, 0)) break;
                if (lane == 0) {   // S^T = K Q^T
                    const uint64_t b0 = dQk + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kColS, dKk + kmaj(kk), b0 + kmaj(kk), idS, kk > 0);
                }
                commit(s_full);
                if (!wait(&do_full[s], ph, 0)) break;
                if (n > 0 && !wait(dq_free, (n - 1) & 1, 1)) break;
                if (lane == 0) {   // dP^T = V dO^T
                    const uint64_t b0 = dOk + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + kColDP, dVk + kmaj(kk), b0 + kmaj(kk), idS, kk > 0);
                }
                commit(dp_full);
                if (k == 0 && !wait(kd_empty, (kvi & 1) ^ 1, 3)) break;
                if (!wait(pds_full, n & 1, 2)) break;
                const uint32_t acc0 = k > 0 ? 1u : 0u;
                if (lane == 0) {   // dV += P^T dO
                    const uint64_t b0 = dOn + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        mma_ts(tmem + kColDV, tmem + kColS + kk * 8, b0 + kk * kRows16, idKM, kk > 0 ? 1u : acc0);
                }
                commit(&do_empty[s]);
                if (lane == 0) {   // dK += dS^T Q
                    const uint64_t b0 = dQn + s * kSlot;
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        mma_ss(tmem + kColDK, dSk + kmaj(kk), b0 + kk * kRows16, idKM, kk > 0 ? 1u : acc0);
                }
                commit(&q_empty[s]);
                if (lane == 0) {
                    if constexpr (D == 128) {
                        // dQ^T = K^T dS^T (M = head dim, N = query rows): the head
                        // dimension lands on TMEM lanes, so each warp of the drain
                        // warpgroup adds one contiguous 128-byte piece of a dQ row.
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)
                            mma_ss(tmem + kColDP, dKn + kk * kRows16, dSn + kk * kRows16, idQ, kk > 0);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk)   // dQ = dS K
                            mma_ss(tmem + kColDP, dSn + kk * kRows16, dKn + kk * kRows16, idQ, kk > 0);
                    }
                }
                commit(dq_full);
                if (k == x.ntiles - 1) {
                    commit(kd_full);
                    commit(kv_empty);
                }
            }
            if (!ok) break;
            ++kvi;
        }
        commit(done);
        int dummy = 0;
        mbar_wait(done, 0, &dummy, a.err);
        if (lane == 0) {
            trace_count(a.trace, a.trace_cap, 4, n);
            for (int z = 0; z < 4; ++z) trace_wait(a.trace, a.trace_cap, 1 + z, wt[z]);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ P^T / dS^T warpgroup
        const int r = (warp % 4) * 32 + lane;              // key row in the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t tS = tmem + lane_base + kColS, tP = tS;
        const uint32_t tdP = tmem + lane_base + kColDP;
        uint32_t n = 0, kvi = 0;
        bool ok = true;
        uint64_t wt[2] = {0, 0};   // tile inputs (q_full, s_full, dp_full), kd_full
        auto wait = [&](uint64_t* bar, uint32_t parity, int slot) {
            ok = ok && __all_sync(0xffffffffu,
                                  mbar_wait_acc(bar, parity, abort_flag, a.err, a.trace ? &wt[slot] : nullptr));
            return ok;
        };
        for (int it = it_begin; it < it_end && ok; ++it) {
            const BItem x = bdecode<VARLEN>(a, a.wl_items[it]);
            const int kvg = x.t * BT + r;                   // global key index of this thread's row
            const bool row_ok = kvg < SEQ_LEN(x);
            const int64_t q_hi = a.win_w > 0 ? ((int64_t)kvg / a.win_c + a.win_w) * a.win_c : INT64_MAX;
            for (int k = 0; k < x.ntiles; ++k, ++n) {
                int hh, i;
                x.tile(k, hh, i);
                const uint32_t s = n & 1, ph = (n >> 1) & 1;
                if (!wait(&q_full[s], ph, 0) || !wait(s_full, n & 1, 0) || !wait(dp_full, n & 1, 0)) break;
                tc_fence_after();
                const float* nlse2 = reinterpret_cast<const float*>(sSide + s * kSide);
                const float* dl = nlse2 + BT;
                const int q0 = i * BT;
#pragma unroll 1
                for (int c = 0; c < BT / 32; ++c) {
                    uint32_t us[32], ud[32];
                    tmem_ld32x2(tS + c * 32, tdP + c * 32, us, ud);   // one round trip for both
                    uint32_t pk[16], dk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c * 32 + e);
                        const float4 d4 = *reinterpret_cast<const float4*>(dl + c * 32 + e);
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
                        float pp[4], dd[4];
#pragma unroll
                        for (int z = 0; z < 4; ++z) {
                            const int qg = q0 + c * 32 + e + z;
                            const bool vis = row_ok && qg < SEQ_LEN(x) && !(a.causal && kvg > qg) && qg < q_hi;
                            const float p = vis ? ex2(fmaf(__uint_as_float(us[e + z]), a.c2, lv[z])) : 0.f;
                            pp[z] = p;
                            dd[z] = p * (__uint_as_float(ud[e + z]) - dv[z]);
                        }
                        pk[e / 2] = pack_bf16(pp[0], pp[1]);
                        pk[e / 2 + 1] = pack_bf16(pp[2], pp[3]);
                        dk[e / 2] = pack_bf16(dd[0], dd[1]);
                        dk[e / 2 + 1] = pack_bf16(dd[2], dd[3]);
                    }
                    tmem_st16(tP + c * 16, pk);
                    uint8_t* blk = sdS + (c / 2) * 16384;
#pragma unroll
                    for (int z = 0; z < 4; ++z)
                        *reinterpret_cast<uint4*>(blk + sw128_offset(r, (c % 2) * 32 + z * 8)) =
                            make_uint4(dk[4 * z], dk[4 * z + 1], dk[4 * z + 2], dk[4 * z + 3]);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(pds_full);
            }
            if (!ok) break;
            // ---- epilogue: dV = acc, dK = scale * acc, bf16, [B, S, Hkv, D]
            if (!wait(kd_full, kvi & 1, 1)) break;
            tc_fence_after();
            const int64_t orow = (((int64_t)SEQ_TB(x) * a.S + SEQ_BASE(x) + kvg) * a.Hkv + x.g) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t uv[32], uk[32];
                tmem_ld32(tmem + lane_base + kColDV + c * 32, uv);
                tmem_ld32(tmem + lane_base + kColDK + c * 32, uk);
                if (row_ok) {
                    uint4* pv = reinterpret_cast<uint4*>(a.dV + orow + c * 32);
                    uint4* pkk = reinterpret_cast<uint4*>(a.dK + orow + c * 32);
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
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ dQ drain warpgroup
        // TMEM lane r = head-dim element r of dQ^T (D = 128) or query row r of dQ (D = 64).
        const int r = (warp % 4) * 32 + lane;
        const uint32_t tdQ = tmem + ((uint32_t)((warp % 4) * 32) << 16) + kColDP;
        constexpr int kCols = D == 128 ? BT : D;
        uint32_t n = 0;
        bool ok = true;
        uint64_t wt = 0;
        for (int it = it_begin; it < it_end && ok; ++it) {
            const BItem x = bdecode<VARLEN>(a, a.wl_items[it]);
            for (int k = 0; k < x.ntiles; ++k, ++n) {
                int hh, i;
                x.tile(k, hh, i);
                const int h = x.g * G + hh;
                ok = __all_sync(0xffffffffu, mbar_wait_acc(dq_full, n & 1, abort_flag, a.err, a.trace ? &wt : nullptr));
                if (!ok) break;
                tc_fence_after();
                uint32_t u[kCols];
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) {
                    uint32_t t32[32];
                    tmem_ld32(tdQ + c * 32, t32);
#pragma unroll
                    for (int e = 0; e < 32; ++e) u[c * 32 + e] = t32[e];
                }
                tc_fence_before();
                mbar_arrive(dq_free);
                if constexpr (D == 128) {
                    // Column c is query row i*128 + c: the warp adds 32 consecutive floats of it.
                    float* base = a.dq_acc + (((int64_t)SEQ_TB(x) * a.H + h) * (VARLEN ? a.acc_rows : a.S) + SEQ_PBASE(x) +
                                                  (int64_t)i * BT) * D + r;
                    const int nq = min(BT, SEQ_LEN(x) - i * BT);
#pragma unroll
                    for (int c = 0; c < BT; ++c)
                        if (c < nq) atomicAdd(base + (int64_t)c * D, __uint_as_float(u[c]));
                } else {
                    const int qg = i * BT + r;
                    if (qg < SEQ_LEN(x)) {
                        float4* dst = reinterpret_cast<float4*>(
                            a.dq_acc + (((int64_t)SEQ_TB(x) * a.H + h) * (VARLEN ? a.acc_rows : a.S) + SEQ_PBASE(x) + qg) * D);
#pragma unroll
                        for (int e = 0; e < D / 4; ++e)
                            atomicAdd(dst + e, make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                                           __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3])));
                    }
                }
            }
        }
        if (threadIdx.x == 256) {
            trace_count(a.trace, a.trace_cap, 7, n);
            trace_wait(a.trace, a.trace_cap, 7, wt);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) trace_cta(a.trace, a.trace_cap, t_start, it_end - it_begin);
}

#undef SEQ_LEN
#undef SEQ_BASE
#undef SEQ_PBASE
#undef SEQ_TB

template <int D>
dfa_status launch(const AttnProblem& p, const void* q, const void* k, const void* v, const void* dO,
                  const float* nlse2, const float* delta, int S_pad, float* dq_acc, void* dK, void* dV,
                  const WorkList* wl, cudaStream_t s) {
    alignas(64) CUtensorMap mq, mk, mv, mdo;
    const int tB = p.seq ? 1 : p.B;   // a packed batch is one tensor row of T tokens
    if (!make_tmap_bshd(&mq, q, tB, p.Lq, p.H, D, p.q_sb, p.q_ss, p.q_sh) ||
        !make_tmap_bshd(&mdo, dO, tB, p.Lq, p.H, D, p.q_sb, p.q_ss, p.q_sh) ||
        !make_tmap_bshd(&mk, k, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh) ||
        !make_tmap_bshd(&mv, v, tB, p.Lkv, p.Hkv, D, p.kv_sb, p.kv_ss, p.kv_sh))
        return fail(DFA_ERR_CUDA, "tensor map encoding failed");
    BwdArgs a{};
    a.seq = p.seq;
    a.acc_rows = p.seq ? S_pad : p.Lq;
    a.B = p.B; a.H = p.H; a.Hkv = p.Hkv; a.S = p.Lq; a.S_pad = S_pad; a.causal = p.causal;
    a.win_c = p.win_c; a.win_w = p.causal ? p.win_w : 0;
    a.scale = p.scale; a.c2 = p.scale * 1.4426950408889634f;
    a.nlse2 = nlse2; a.delta = delta; a.dq_acc = dq_acc;
    a.dK = static_cast<__nv_bfloat16*>(dK);
    a.dV = static_cast<__nv_bfloat16*>(dV);
    a.wl_offsets = wl->offsets; a.wl_items = wl->items; a.n_units = wl->n_units;
    a.err = device_error_flag();
    a.trace = cta_trace(&a.trace_cap);
    auto kern = p.seq ? bwd_tc_kernel<D, true> : bwd_tc_kernel<D, false>;
    const int smem = BCfg<D>::kSmem;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "bwd_tc: shared memory attribute");
    kern<<<wl->n_workers, kThreads, smem, s>>>(mq, mk, mv, mdo, a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "bwd_tc launch: %s", cudaGetErrorString(e));
}

}  // namespace

dfa_status tc_bwd(const AttnProblem& p, const void* q, const void* k, const void* v, const void* dO,
                  const float* nlse2, const float* delta, int S_pad, float* dq_acc, void* dK, void* dV,
                  const WorkList* wl, cudaStream_t s) {
    if (p.B == 0 || p.Lq == 0) return DFA_OK;
    // Head dim 128 takes the two-stream pipelined kernel (bwd_pipe_tc.cu).
    if (p.D == 128) return tc_bwd_pipelined(p, q, k, v, dO, nlse2, delta, S_pad, dq_acc, dK, dV, false, wl, s);
    return launch<64>(p, q, k, v, dO, nlse2, delta, S_pad, dq_acc, dK, dV, wl, s);
}

}  // namespace dfa
