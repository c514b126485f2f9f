// simt_attn.cu -- fp32 CUDA-core attention kernels (the fp32-I/O path).
//
// Exact causal softmax attention as in DISTFLASHATTN §3.1/§3.2 (paperlayer.ai
// summary of arXiv 2310.03294), computed FlashAttention-style: key/value tiles
// stream through shared memory and each query row keeps a running maximum,
// running sum and unnormalised output that are rescaled as new tiles arrive
// (the online-normalizer rule the pages build on).  All arithmetic is fp32 on
// CUDA cores, so fp32 inputs keep fp32 accuracy (one-pass tf32 tensor-core
// MMAs would not).  The backward (§3.3) reads the saved lse and never
// recomputes the forward: two kernels, one producing dQ per query tile and
// one producing dK/dV per key/value tile (summing a GQA group's heads), both
// deterministic (no atomics).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace dfa {
namespace {

constexpr int BQ = 64;      // query rows per CTA
constexpr int BK = 64;      // key rows per tile
constexpr int NWARP = 8;
constexpr int RPW = BQ / NWARP;  // rows per warp
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st(T* p, float x);
template <> __device__ __forceinline__ void st<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}
// Key position kp lies outside the local window of query position qp.
__device__ __forceinline__ bool out_of_window(const AttnProblem& p, int64_t qp, int64_t kp) {
    return p.win_w > 0 && p.causal && kp / p.win_c < qp / p.win_c - (p.win_w - 1);
}
// Store, or add to the value already there (each output element has one writer).
template <typename T> __device__ __forceinline__ void put(T* p, float x, bool acc) { st(p, acc ? ld(p) + x : x); }

__device__ __forceinline__ int64_t mn64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t mx64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ float warp_max(float x) {
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Loads rows [r0, r0+64) of one head into a padded fp32 smem tile (zero past L).
template <typename T, int D>
__device__ void load_tile(float (*dst)[D + 1], const T* base, int64_t ss, int r0, int L,
                          float mul) {
    for (int x = threadIdx.x; x < BK * D; x += blockDim.x) {
        int r = x / D, d = x % D;
        dst[r][d] = (r0 + r < L) ? mul * ld(base + (int64_t)(r0 + r) * ss + d) : 0.f;
    }
}

// ---------------------------------------------------------------- forward
template <typename T, typename OT, int D>
__global__ void __launch_bounds__(NWARP * 32)
simt_fwd_kernel(AttnProblem p, const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, OT* __restrict__ O, float* __restrict__ lse) {
    extern __shared__ float smem[];
    float(*Qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem);
    float(*Ks)[D + 1] = Qs + BQ;
    float(*Vs)[D + 1] = Ks + BK;
    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * BQ;
    const int g = h / (p.H / p.Hkv);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const T* qb = q + b * p.q_sb + h * p.q_sh;
    const T* kb = k + b * p.kv_sb + g * p.kv_sh;
    const T* vb = v + b * p.kv_sb + g * p.kv_sh;
    // Scores are kept in the log2 domain: s2 = scale * log2(e) * <q, k>.
    load_tile<T, D>(Qs, qb, p.q_ss, q0, p.Lq, p.scale * LOG2E);

    float m[RPW], l[RPW], o[RPW][D / 32];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) o[r][c] = 0.f;
    }
    // Keys beyond jend are invisible to every row of this tile.
    int64_t jend = p.Lkv;
    if (p.causal) {
        int64_t last_q = p.q_offset + min(q0 + BQ, p.Lq) - 1;
        jend = mn64(p.Lkv, mx64(0, last_q - p.kv_offset + 1));
    }
    for (int kt = 0; kt < jend; kt += BK) {
        __syncthreads();
        load_tile<T, D>(Ks, kb, p.kv_ss, kt, p.Lkv, 1.f);
        load_tile<T, D>(Vs, vb, p.kv_ss, kt, p.Lkv, 1.f);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int row = warp * RPW + r;
            const int64_t qpos = p.q_offset + q0 + row;
            float sa = 0.f, sb = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                sa = fmaf(Qs[row][d], Ks[lane][d], sa);
                sb = fmaf(Qs[row][d], Ks[lane + 32][d], sb);
            }
            const int ja = kt + lane, jb = kt + lane + 32;
            if (ja >= p.Lkv || (p.causal && p.kv_offset + ja > qpos) || out_of_window(p, qpos, p.kv_offset + ja))
                sa = -INFINITY;
            if (jb >= p.Lkv || (p.causal && p.kv_offset + jb > qpos) || out_of_window(p, qpos, p.kv_offset + jb))
                sb = -INFINITY;
            const float mn = fmaxf(m[r], warp_max(fmaxf(sa, sb)));
            if (mn == -INFINITY) continue;          // nothing visible yet in this row
            const float alpha = exp2f(m[r] - mn);   // 0 when m was -inf
            const float pa = exp2f(sa - mn), pb = exp2f(sb - mn);
            l[r] = l[r] * alpha + warp_sum(pa + pb);
            m[r] = mn;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) o[r][c] *= alpha;
#pragma unroll 4
            for (int jj = 0; jj < 32; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, pa, jj);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) o[r][c] = fmaf(pj, Vs[jj][lane + 32 * c], o[r][c]);
            }
#pragma unroll 4
            for (int jj = 0; jj < 32; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, pb, jj);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) o[r][c] = fmaf(pj, Vs[jj + 32][lane + 32 * c], o[r][c]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int i = q0 + warp * RPW + r;
        if (i >= p.Lq) continue;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
        OT* orow = O + (((int64_t)b * p.Lq + i) * p.H + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) st(orow + lane + 32 * c, o[r][c] * inv);
        if (lane == 0)
            lse[((int64_t)b * p.H + h) * p.Lq + i] = l[r] > 0.f ? (m[r] + log2f(l[r])) * LN2 : -INFINITY;
    }
}

// ---------------------------------------------------------------- backward: dQ
template <typename T, typename OT, int D>
__global__ void __launch_bounds__(NWARP * 32)
simt_bwd_dq_kernel(AttnProblem p, const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, const T* __restrict__ dO, const float* __restrict__ lse,
                   const float* __restrict__ delta, OT* __restrict__ dQ) {
    extern __shared__ float smem[];
    float(*Qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem);
    float(*dOs)[D + 1] = Qs + BQ;
    float(*Ks)[D + 1] = dOs + BQ;
    float(*Vs)[D + 1] = Ks + BK;
    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * BQ;
    const int g = h / (p.H / p.Hkv);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const T* qb = q + b * p.q_sb + h * p.q_sh;
    const T* dob = dO + b * p.q_sb + h * p.q_sh;
    const T* kb = k + b * p.kv_sb + g * p.kv_sh;
    const T* vb = v + b * p.kv_sb + g * p.kv_sh;
    load_tile<T, D>(Qs, qb, p.q_ss, q0, p.Lq, p.scale * LOG2E);
    load_tile<T, D>(dOs, dob, p.q_ss, q0, p.Lq, 1.f);

    float lse2[RPW], dl[RPW], acc[RPW][D / 32];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int i = q0 + warp * RPW + r;
        const bool ok = i < p.Lq;
        lse2[r] = ok ? lse[((int64_t)b * p.H + h) * p.Lq + i] * LOG2E : -INFINITY;
        dl[r] = ok ? delta[((int64_t)b * p.H + h) * p.Lq + i] : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) acc[r][c] = 0.f;
    }
    int64_t jend = p.Lkv;
    if (p.causal) {
        int64_t last_q = p.q_offset + min(q0 + BQ, p.Lq) - 1;
        jend = mn64(p.Lkv, mx64(0, last_q - p.kv_offset + 1));
    }
    for (int kt = 0; kt < jend; kt += BK) {
        __syncthreads();
        load_tile<T, D>(Ks, kb, p.kv_ss, kt, p.Lkv, 1.f);
        load_tile<T, D>(Vs, vb, p.kv_ss, kt, p.Lkv, 1.f);
        __syncthreads();
#pragma unroll 1
        for (int r = 0; r < RPW; ++r) {
            if (lse2[r] == -INFINITY) continue;
            const int row = warp * RPW + r;
            const int64_t qpos = p.q_offset + q0 + row;
            float sa = 0.f, sb = 0.f, pa_ = 0.f, pb_ = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                sa = fmaf(Qs[row][d], Ks[lane][d], sa);
                sb = fmaf(Qs[row][d], Ks[lane + 32][d], sb);
                pa_ = fmaf(dOs[row][d], Vs[lane][d], pa_);
                pb_ = fmaf(dOs[row][d], Vs[lane + 32][d], pb_);
            }
            const int ja = kt + lane, jb = kt + lane + 32;
            const bool va = ja < p.Lkv && !(p.causal && p.kv_offset + ja > qpos) &&
                            !out_of_window(p, qpos, p.kv_offset + ja);
            const bool vb_ = jb < p.Lkv && !(p.causal && p.kv_offset + jb > qpos) &&
                             !out_of_window(p, qpos, p.kv_offset + jb);
            const float Pa = va ? exp2f(sa - lse2[r]) : 0.f;
            const float Pb = vb_ ? exp2f(sb - lse2[r]) : 0.f;
            const float dsa = Pa * (pa_ - dl[r]), dsb = Pb * (pb_ - dl[r]);
#pragma unroll 4
            for (int jj = 0; jj < 32; ++jj) {
                const float x = __shfl_sync(0xffffffffu, dsa, jj);
                const float y = __shfl_sync(0xffffffffu, dsb, jj);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    acc[r][c] = fmaf(x, Ks[jj][lane + 32 * c], acc[r][c]);
                    acc[r][c] = fmaf(y, Ks[jj + 32][lane + 32 * c], acc[r][c]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int i = q0 + warp * RPW + r;
        if (i >= p.Lq) continue;
        OT* row = dQ + (((int64_t)b * p.Lq + i) * p.H + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) put(row + lane + 32 * c, p.scale * acc[r][c], p.acc_out);
    }
}

// ---------------------------------------------------------------- backward: dK, dV
template <typename T, typename OT, int D>
__global__ void __launch_bounds__(NWARP * 32)
simt_bwd_dkv_kernel(AttnProblem p, const T* __restrict__ q, const T* __restrict__ k,
                    const T* __restrict__ v, const T* __restrict__ dO, const float* __restrict__ lse,
                    const float* __restrict__ delta, OT* __restrict__ dK, OT* __restrict__ dV) {
    extern __shared__ float smem[];
    float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem);
    float(*Vs)[D + 1] = Ks + BK;
    float(*Qs)[D + 1] = Vs + BK;
    float(*dOs)[D + 1] = Qs + BQ;
    float* lse2s = reinterpret_cast<float*>(dOs + BQ);
    float* dls = lse2s + BQ;
    const int b = blockIdx.z, g = blockIdx.y, j0 = blockIdx.x * BK;
    const int G = p.H / p.Hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float c2 = p.scale * LOG2E;
    load_tile<T, D>(Ks, k + b * p.kv_sb + g * p.kv_sh, p.kv_ss, j0, p.Lkv, 1.f);
    load_tile<T, D>(Vs, v + b * p.kv_sb + g * p.kv_sh, p.kv_ss, j0, p.Lkv, 1.f);

    float dk[RPW][D / 32], dv[RPW][D / 32];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) dk[r][c] = dv[r][c] = 0.f;

    // First query row that can see key j0: q_offset + i >= kv_offset + j0.
    int64_t ifirst = 0;
    if (p.causal) ifirst = mx64(0, p.kv_offset + j0 - p.q_offset);
    const int qstart = (int)mn64(p.Lq, (ifirst / BQ) * BQ);
    for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh;
        const T* qb = q + b * p.q_sb + h * p.q_sh;
        const T* dob = dO + b * p.q_sb + h * p.q_sh;
        for (int qt = qstart; qt < p.Lq; qt += BQ) {
            __syncthreads();
            load_tile<T, D>(Qs, qb, p.q_ss, qt, p.Lq, 1.f);
            load_tile<T, D>(dOs, dob, p.q_ss, qt, p.Lq, 1.f);
            for (int x = threadIdx.x; x < BQ; x += blockDim.x) {
                const int i = qt + x;
                const bool ok = i < p.Lq;
                lse2s[x] = ok ? lse[((int64_t)b * p.H + h) * p.Lq + i] * LOG2E : -INFINITY;
                dls[x] = ok ? delta[((int64_t)b * p.H + h) * p.Lq + i] : 0.f;
            }
            __syncthreads();
#pragma unroll 1
            for (int r = 0; r < RPW; ++r) {
                const int jr = warp * RPW + r;
                const int64_t kpos = p.kv_offset + j0 + jr;
                float Pv[2], dS[2];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int ir = lane + 32 * half;
                    float s = 0.f, dp = 0.f;
#pragma unroll 8
                    for (int d = 0; d < D; ++d) {
                        s = fmaf(Qs[ir][d], Ks[jr][d], s);
                        dp = fmaf(dOs[ir][d], Vs[jr][d], dp);
                    }
                    const bool vis = (j0 + jr < p.Lkv) && (qt + ir < p.Lq) && lse2s[ir] != -INFINITY &&
                                     !(p.causal && kpos > p.q_offset + qt + ir) &&
                                     !out_of_window(p, p.q_offset + qt + ir, kpos);
                    Pv[half] = vis ? exp2f(s * c2 - lse2s[ir]) : 0.f;
                    dS[half] = Pv[half] * (dp - dls[ir]);
                }
#pragma unroll 4
                for (int ii = 0; ii < 32; ++ii) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const float pp = __shfl_sync(0xffffffffu, Pv[half], ii);
                        const float ds = __shfl_sync(0xffffffffu, dS[half], ii);
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            dv[r][c] = fmaf(pp, dOs[ii + 32 * half][lane + 32 * c], dv[r][c]);
                            dk[r][c] = fmaf(ds, Qs[ii + 32 * half][lane + 32 * c], dk[r][c]);
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int j = j0 + warp * RPW + r;
        if (j >= p.Lkv) continue;
        OT* krow = dK + (((int64_t)b * p.Lkv + j) * p.Hkv + g) * D;
        OT* vrow = dV + (((int64_t)b * p.Lkv + j) * p.Hkv + g) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            put(krow + lane + 32 * c, p.scale * dk[r][c], p.acc_out);
            put(vrow + lane + 32 * c, dv[r][c], p.acc_out);
        }
    }
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <typename T, typename OT, int D>
dfa_status fwd_impl(const AttnProblem& p, const void* q, const void* k, const void* v, void* O,
                    float* lse, cudaStream_t s) {
    const size_t smem = sizeof(float) * (BQ + 2 * BK) * (D + 1);
    auto kern = simt_fwd_kernel<T, OT, D>;
    if (prep(kern, smem) != cudaSuccess) return fail(DFA_ERR_CUDA, "simt fwd: smem attribute");
    dim3 grid((p.Lq + BQ - 1) / BQ, p.H, p.B);
    kern<<<grid, NWARP * 32, smem, s>>>(p, (const T*)q, (const T*)k, (const T*)v, (OT*)O, lse);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "simt fwd launch: %s", cudaGetErrorString(e));
}

template <typename T, typename OT, int D>
dfa_status bwd_impl(const AttnProblem& p, const void* q, const void* k, const void* v,
                    const void* dO, const float* lse, const float* delta, void* dQ, void* dK,
                    void* dV, cudaStream_t s) {
    const size_t smem_q = sizeof(float) * (2 * BQ + 2 * BK) * (D + 1);
    const size_t smem_kv = sizeof(float) * ((2 * BQ + 2 * BK) * (D + 1) + 2 * BQ);
    auto kq = simt_bwd_dq_kernel<T, OT, D>;
    auto kkv = simt_bwd_dkv_kernel<T, OT, D>;
    if (prep(kq, smem_q) != cudaSuccess || prep(kkv, smem_kv) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "simt bwd: smem attribute");
    if (p.Lq > 0) {
        dim3 gq((p.Lq + BQ - 1) / BQ, p.H, p.B);
        kq<<<gq, NWARP * 32, smem_q, s>>>(p, (const T*)q, (const T*)k, (const T*)v, (const T*)dO,
                                          lse, delta, (OT*)dQ);
    }
    if (p.Lkv > 0) {
        dim3 gkv((p.Lkv + BK - 1) / BK, p.Hkv, p.B);
        kkv<<<gkv, NWARP * 32, smem_kv, s>>>(p, (const T*)q, (const T*)k, (const T*)v,
                                             (const T*)dO, lse, delta, (OT*)dK, (OT*)dV);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "simt bwd launch: %s", cudaGetErrorString(e));
}

}  // namespace

dfa_status simt_fwd(const AttnProblem& p, dfa_dtype dt, const void* q, const void* k,
                    const void* v, void* O, bool O_is_f32, float* lse, cudaStream_t s) {
    if (p.Lq == 0 || p.B == 0) return DFA_OK;
    using bf = __nv_bfloat16;
    if (dt == DFA_F32) {
        return p.D == 64 ? fwd_impl<float, float, 64>(p, q, k, v, O, lse, s)
                         : fwd_impl<float, float, 128>(p, q, k, v, O, lse, s);
    }
    if (O_is_f32)
        return p.D == 64 ? fwd_impl<bf, float, 64>(p, q, k, v, O, lse, s)
                         : fwd_impl<bf, float, 128>(p, q, k, v, O, lse, s);
    return p.D == 64 ? fwd_impl<bf, bf, 64>(p, q, k, v, O, lse, s)
                     : fwd_impl<bf, bf, 128>(p, q, k, v, O, lse, s);
}

dfa_status simt_bwd(const AttnProblem& p, dfa_dtype dt, const void* q, const void* k,
                    const void* v, const void* dO, const float* lse, const float* delta,
                    void* dQ, void* dK, void* dV, cudaStream_t s) {
    if (p.B == 0) return DFA_OK;
    using bf = __nv_bfloat16;
    if (dt == DFA_F32)
        return p.D == 64 ? bwd_impl<float, float, 64>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s)
                         : bwd_impl<float, float, 128>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s);
    if (p.acc_out)
        return p.D == 64 ? bwd_impl<bf, float, 64>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s)
                         : bwd_impl<bf, float, 128>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s);
    return p.D == 64 ? bwd_impl<bf, bf, 64>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s)
                     : bwd_impl<bf, bf, 128>(p, q, k, v, dO, lse, delta, dQ, dK, dV, s);
}

}  // namespace dfa
