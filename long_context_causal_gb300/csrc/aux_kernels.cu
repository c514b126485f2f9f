// aux_kernels.cu -- HBM-bound helper kernels of the attention path.
//
//  * merge:   the online-softmax rescale-and-merge of two partial results
//             (DISTFLASHATTN §3.2, paperlayer.ai summary of arXiv 2310.03294:
//             helpers return partial outputs plus softmax statistics that the
//             owner rescales before combining);
//  * merge_pieces: the same rule over the split-kv pieces of a forward, fp32
//             partials in, the output dtype out;
//  * delta:   Delta_i = <dO_i, O_i>, the per-row term of the softmax gradient,
//             read once from the SAVED output (§3.3: the backward reuses the
//             forward's output instead of recomputing it);
//  * convert: the head-major fp32 dQ accumulator [B, H, S, D] scaled, cast to the
//    output dtype and written as [B, S, H, D].
// Each is a streaming pass: one warp per row, 16-byte loads, no reuse.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace dfa {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__global__ void __launch_bounds__(kThreads)
merge_kernel(int B, int H, int L, int D, const float* Oa, const float* la, const float* Ob,
             const float* lb, float* O, float* l) {
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;  // (b, i, h)
    const int lane = threadIdx.x % 32;
    if (row >= (int64_t)B * L * H) return;
    const int h = row % H;
    const int64_t bi = row / H;
    const int i = bi % L, b = bi / L;
    const int64_t li = ((int64_t)b * H + h) * L + i;
    const float a = la[li], c = lb[li];
    const float m = fmaxf(a, c);
    float wa = 0.f, wc = 0.f, lse = -INFINITY;
    if (m != -INFINITY) {
        const float ea = expf(a - m), ec = expf(c - m);
        const float sum = ea + ec;
        lse = m + logf(sum);
        wa = ea / sum;
        wc = ec / sum;
    }
    const float4* pa = reinterpret_cast<const float4*>(Oa + row * D);
    const float4* pb = reinterpret_cast<const float4*>(Ob + row * D);
    float4* po = reinterpret_cast<float4*>(O + row * D);
    for (int x = lane; x < D / 4; x += 32) {
        const float4 u = pa[x], w = pb[x];
        po[x] = make_float4(wa * u.x + wc * w.x, wa * u.y + wc * w.y, wa * u.z + wc * w.z,
                            wa * u.w + wc * w.w);
    }
    __syncwarp();
    if (lane == 0) l[li] = lse;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* out);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* out) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const float2 f = __bfloat1622float2(h[x]);
        out[2 * x] = f.x;
        out[2 * x + 1] = f.y;
    }
}

// One warp per (b, i, h) row; D / 8 lanes each read 8 elements.
template <typename T>
__global__ void __launch_bounds__(kThreads)
delta_kernel(int B, int H, int S, int D, const T* __restrict__ O, const T* __restrict__ dO,
             float* __restrict__ delta) {
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= (int64_t)B * S * H) return;
    float acc = 0.f;
    for (int x = lane; x < D / 8; x += 32) {
        float a[8], c[8];
        load8<T>(O + row * D + 8 * x, a);
        load8<T>(dO + row * D + 8 * x, c);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(a[e], c[e], acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        const int h = row % H;
        const int64_t bi = row / H;
        const int i = bi % S, b = bi / S;
        delta[((int64_t)b * H + h) * S + i] = acc;
    }
}

// One warp per (b, i, h) row of the padded range i < S_pad.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_prep_kernel(int B, int H, int S, int S_pad, int D, const T* __restrict__ O, const T* __restrict__ dO,
                const float* __restrict__ lse, float* __restrict__ nlse2, float* __restrict__ delta) {
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= (int64_t)B * S_pad * H) return;
    const int h = row % H;
    const int64_t bi = row / H;
    const int i = bi % S_pad, b = bi / S_pad;
    const int64_t dst = ((int64_t)b * H + h) * S_pad + i;
    if (i >= S) {
        if (lane == 0) {
            nlse2[dst] = 0.f;
            delta[dst] = 0.f;
        }
        return;
    }
    const int64_t src = (((int64_t)b * S + i) * H + h) * D;
    float acc = 0.f;
    for (int x = lane; x < D / 8; x += 32) {
        float a[8], c[8];
        load8<T>(O + src + 8 * x, a);
        load8<T>(dO + src + 8 * x, c);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(a[e], c[e], acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        delta[dst] = acc;
        nlse2[dst] = lse[((int64_t)b * H + h) * S + i] * -1.4426950408889634f;   // -lse log2(e), exact negation
    }
}

// Eight consecutive head-dim elements per thread: output x*8 of [B, S, H, D]
// comes from the head-major accumulator [B, H, S, D].
__device__ __forceinline__ int64_t acc_index(int64_t o, int H, int S, int D) {
    const int d = (int)(o % D);
    const int64_t r = o / D;
    const int h = (int)(r % H);
    const int64_t bs = r / H;
    const int s = (int)(bs % S);
    const int64_t b = bs / S;
    return ((b * H + h) * S + s) * D + d;
}

__global__ void convert_bf16_kernel(int64_t n, int H, int S, int D, float scale, const float* __restrict__ in,
                                    __nv_bfloat16* __restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n / 8; x += stride) {
        const float4* src = reinterpret_cast<const float4*>(in + acc_index(8 * x, H, S, D));
        const float4 a = src[0], b = src[1];
        __nv_bfloat162 r[4] = {__floats2bfloat162_rn(scale * a.x, scale * a.y),
                               __floats2bfloat162_rn(scale * a.z, scale * a.w),
                               __floats2bfloat162_rn(scale * b.x, scale * b.y),
                               __floats2bfloat162_rn(scale * b.z, scale * b.w)};
        reinterpret_cast<uint4*>(out)[x] = *reinterpret_cast<uint4*>(r);
    }
}

__global__ void convert_f32_kernel(int64_t n, int H, int S, int D, float scale, const float* __restrict__ in,
                                   float* __restrict__ out, int accumulate) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n / 8; x += stride) {
        const float4* src = reinterpret_cast<const float4*>(in + acc_index(8 * x, H, S, D));
        const float4 a = src[0], b = src[1];
        float4* dst = reinterpret_cast<float4*>(out) + 2 * x;
        float4 o0 = make_float4(scale * a.x, scale * a.y, scale * a.z, scale * a.w);
        float4 o1 = make_float4(scale * b.x, scale * b.y, scale * b.z, scale * b.w);
        if (accumulate) {
            const float4 p0 = dst[0], p1 = dst[1];
            o0.x += p0.x; o0.y += p0.y; o0.z += p0.z; o0.w += p0.w;
            o1.x += p1.x; o1.y += p1.y; o1.z += p1.z; o1.w += p1.w;
        }
        dst[0] = o0;
        dst[1] = o1;
    }
}

// Sequence of a packed batch that holds position p, given the non-decreasing
// starts st[0..n] (st[n] is the end): the last s < n with st[s] <= p.
__device__ __forceinline__ int seq_of(const int32_t* st, int n, int64_t p) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (st[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Packed batch: one warp per (padded row p, head h) of the [H, P] arrays;
// seq = token starts [n+1] then padded starts [n+1].  Rows past a sequence's
// end are zero.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_prep_varlen_kernel(int n, int H, int64_t Ttok, int64_t P, int D, const int32_t* __restrict__ seq,
                       const T* __restrict__ O, const T* __restrict__ dO, const float* __restrict__ lse,
                       float* __restrict__ nlse2, float* __restrict__ delta) {
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= P * H) return;
    const int h = row % H;
    const int64_t p = row / H;
    const int s = seq_of(seq + n + 1, n, p);
    const int64_t rel = p - seq[n + 1 + s], tok = seq[s] + rel;
    const int64_t dst = (int64_t)h * P + p;
    if (rel >= seq[s + 1] - seq[s]) {
        if (lane == 0) {
            nlse2[dst] = 0.f;
            delta[dst] = 0.f;
        }
        return;
    }
    const int64_t src = (tok * H + h) * D;
    float acc = 0.f;
    for (int x = lane; x < D / 8; x += 32) {
        float a[8], c[8];
        load8<T>(O + src + 8 * x, a);
        load8<T>(dO + src + 8 * x, c);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(a[e], c[e], acc);
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        delta[dst] = acc;
        nlse2[dst] = lse[(int64_t)h * Ttok + tok] * -1.4426950408889634f;
    }
}

// Packed batch: dQ [T, H, D] (bf16) = scale * the head-major padded
// accumulator [H, P, D]; eight head-dim elements per thread.
__global__ void convert_varlen_bf16_kernel(int n, int H, int64_t Ttok, int64_t P, int D, float scale,
                                           const int32_t* __restrict__ seq, const float* __restrict__ in,
                                           __nv_bfloat16* __restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x, n8 = Ttok * H * D / 8;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n8; x += stride) {
        const int64_t o = 8 * x;
        const int d = (int)(o % D);
        const int64_t r = o / D;
        const int h = (int)(r % H);
        const int64_t tok = r / H;
        const int s = seq_of(seq, n, tok);
        const int64_t p = seq[n + 1 + s] + (tok - seq[s]);
        const float4* src = reinterpret_cast<const float4*>(in + ((int64_t)h * P + p) * D + d);
        const float4 a = src[0], b = src[1];
        __nv_bfloat162 v[4] = {__floats2bfloat162_rn(scale * a.x, scale * a.y),
                               __floats2bfloat162_rn(scale * a.z, scale * a.w),
                               __floats2bfloat162_rn(scale * b.x, scale * b.y),
                               __floats2bfloat162_rn(scale * b.z, scale * b.w)};
        reinterpret_cast<uint4*>(out)[x] = *reinterpret_cast<uint4*>(v);
    }
}

// fp32 -> bf16, eight elements per thread (n a multiple of 8).
__global__ void cast_bf16_kernel(int64_t n, const float* __restrict__ in, __nv_bfloat16* __restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n / 8; x += stride) {
        const float4 a = reinterpret_cast<const float4*>(in)[2 * x], b = reinterpret_cast<const float4*>(in)[2 * x + 1];
        __nv_bfloat162 r[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                               __floats2bfloat162_rn(b.x, b.y), __floats2bfloat162_rn(b.z, b.w)};
        reinterpret_cast<uint4*>(out)[x] = *reinterpret_cast<uint4*>(r);
    }
}

// Grid-stride copies for dfa_copy.  Either side may be pinned host memory:
// the SMs read and write it directly over the GPU's coherent host link.
__global__ void __launch_bounds__(512) copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
#pragma unroll 4
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}
__global__ void __launch_bounds__(512) copy1_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, size_t n) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

dfa_status launched(const char* what) {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
}

}  // namespace

// Split-kv merge (the owner's side of the pages' helper exchange, §3.2): one
// warp per (b, i, h) row combines the row's pieces with the rescale rule
//   lse = m + ln sum_s e^(lse_s - m),  O = sum_s e^(lse_s - lse) O_s,
// m = max_s lse_s; pieces with lse_s = -inf weigh 0.  Every row's piece 0
// holds key 0, so lse is finite for every row that sees a key.
template <typename T>
__global__ void __launch_bounds__(kThreads)
merge_pieces_kernel(int B, int H, int S, int D, int causal, int piece_tiles, int n_split, const float* O_part,
                    const float* lse_part, T* O, float* lse) {
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + threadIdx.x / 32;  // (b, i, h)
    const int lane = threadIdx.x % 32;
    if (row >= (int64_t)B * S * H) return;
    const int h = row % H;
    const int64_t bi = row / H;
    const int i = bi % S, b = bi / S;
    const int kv_tiles = (S + 127) / 128, u = i / 256;
    const int hi = causal ? min(2 * u + 2, kv_tiles) : kv_tiles;
    const int np = min((hi + piece_tiles - 1) / piece_tiles, n_split);
    const int64_t li = ((int64_t)b * H + h) * S + i, lstride = (int64_t)B * H * S;
    const int64_t ostride = (int64_t)B * S * H * D;
    float m = -INFINITY;
    for (int s = 0; s < np; ++s) m = fmaxf(m, lse_part[s * lstride + li]);
    float sum = 0.f;
    if (m != -INFINITY)
        for (int s = 0; s < np; ++s) sum += expf(lse_part[s * lstride + li] - m);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int x = lane; x < D / 4; x += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m != -INFINITY)
            for (int s = 0; s < np; ++s) {
                const float w = expf(lse_part[s * lstride + li] - m) * inv;
                const float4 o = reinterpret_cast<const float4*>(O_part + s * ostride + row * D)[x];
                acc.x += w * o.x;
                acc.y += w * o.y;
                acc.z += w * o.z;
                acc.w += w * o.w;
            }
        T* dst = O + row * D + 4 * x;
        dst[0] = from_f32<T>(acc.x);
        dst[1] = from_f32<T>(acc.y);
        dst[2] = from_f32<T>(acc.z);
        dst[3] = from_f32<T>(acc.w);
    }
    if (lane == 0) lse[li] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

dfa_status launch_merge(int B, int H, int L, int D, const float* Oa, const float* la,
                        const float* Ob, const float* lb, float* O, float* l, cudaStream_t s) {
    const int64_t rows = (int64_t)B * L * H;
    if (rows == 0) return DFA_OK;
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    merge_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(B, H, L, D, Oa, la, Ob, lb, O, l);
    return launched("merge");
}

dfa_status launch_merge_pieces(dfa_dtype dt, int B, int H, int S, int D, int causal, int piece_tiles,
                               int n_split, const float* O_part, const float* lse_part, void* O, float* lse,
                               cudaStream_t s) {
    const int64_t rows = (int64_t)B * S * H;
    if (rows == 0) return DFA_OK;
    if (piece_tiles <= 0 || n_split <= 0 || D % 4 != 0) return fail(DFA_ERR_INVALID_ARG, "bad split-kv merge sizes");
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    if (dt == DFA_F32)
        merge_pieces_kernel<float><<<(unsigned)blocks, kThreads, 0, s>>>(B, H, S, D, causal, piece_tiles, n_split,
                                                                         O_part, lse_part, (float*)O, lse);
    else
        merge_pieces_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(
            B, H, S, D, causal, piece_tiles, n_split, O_part, lse_part, (__nv_bfloat16*)O, lse);
    return launched("split-kv merge");
}

dfa_status launch_bwd_prep_varlen(int n_seq, int H, int64_t T, int64_t P, int D, const int32_t* seq,
                                  const void* O, const void* dO, const float* lse, float* nlse2, float* delta,
                                  cudaStream_t s) {
    const int64_t rows = P * H;
    if (rows == 0 || n_seq <= 0) return DFA_OK;
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    bwd_prep_varlen_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(
        n_seq, H, T, P, D, seq, (const __nv_bfloat16*)O, (const __nv_bfloat16*)dO, lse, nlse2, delta);
    return launched("varlen bwd prep");
}

dfa_status launch_convert_varlen(int n_seq, int H, int64_t T, int64_t P, int D, float scale, const int32_t* seq,
                                 const float* acc, void* out, cudaStream_t s) {
    const int64_t n8 = T * H * D / 8;
    if (n8 == 0 || n_seq <= 0) return DFA_OK;
    const int blocks = 8 * num_sms();
    convert_varlen_bf16_kernel<<<blocks, kThreads, 0, s>>>(n_seq, H, T, P, D, scale, seq, acc,
                                                                 (__nv_bfloat16*)out);
    return launched("varlen dQ convert");
}

// One block of 512 threads per SM: enough to hold the host link at its limit
// in either direction (measured 211 GB/s in, 193 out on a GB300).
dfa_status launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return DFA_OK;
    const int blocks = num_sms();
    const bool aligned = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
    const size_t n16 = aligned ? bytes / 16 : 0;
    if (n16) copy16_kernel<<<blocks, 512, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
    const size_t done = n16 * 16;
    if (done < bytes)
        copy1_kernel<<<aligned ? 1 : blocks, 512, 0, s>>>(static_cast<const uint8_t*>(src) + done,
                                                           static_cast<uint8_t*>(dst) + done, bytes - done);
    return launched("copy");
}

dfa_status launch_cast_bf16(int64_t n, const float* in, void* out, cudaStream_t s) {
    if (n == 0) return DFA_OK;
    if (n % 8 != 0) return fail(DFA_ERR_INVALID_ARG, "cast: element count not a multiple of 8");
    cast_bf16_kernel<<<8 * num_sms(), kThreads, 0, s>>>(n, in, static_cast<__nv_bfloat16*>(out));
    return launched("bf16 cast");
}

dfa_status launch_delta(dfa_dtype dt, int B, int H, int S, int D, const void* O,
                        const void* dO, float* delta, cudaStream_t s) {
    const int64_t rows = (int64_t)B * S * H;
    if (rows == 0) return DFA_OK;
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    if (dt == DFA_F32)
        delta_kernel<float><<<(unsigned)blocks, kThreads, 0, s>>>(B, H, S, D, (const float*)O,
                                                                  (const float*)dO, delta);
    else
        delta_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(
            B, H, S, D, (const __nv_bfloat16*)O, (const __nv_bfloat16*)dO, delta);
    return launched("delta");
}

dfa_status launch_bwd_prep(dfa_dtype dt, int B, int H, int S, int S_pad, int D, const void* O,
                           const void* dO, const float* lse, float* nlse2, float* delta, cudaStream_t s) {
    const int64_t rows = (int64_t)B * S_pad * H;
    if (rows == 0) return DFA_OK;
    const int64_t blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
    if (dt == DFA_F32)
        bwd_prep_kernel<float><<<(unsigned)blocks, kThreads, 0, s>>>(B, H, S, S_pad, D, (const float*)O,
                                                                     (const float*)dO, lse, nlse2, delta);
    else
        bwd_prep_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(
            B, H, S, S_pad, D, (const __nv_bfloat16*)O, (const __nv_bfloat16*)dO, lse, nlse2, delta);
    return launched("bwd prep");
}

dfa_status launch_convert(dfa_dtype dt, int B, int H, int S, int D, float scale, const float* acc, void* out,
                          bool accumulate, cudaStream_t s) {
    const int64_t n = (int64_t)B * S * H * D;
    if (n == 0) return DFA_OK;
    const int blocks = 8 * num_sms();
    if (dt == DFA_BF16 && !accumulate)
        convert_bf16_kernel<<<blocks, kThreads, 0, s>>>(n, H, S, D, scale, acc, (__nv_bfloat16*)out);
    else
        convert_f32_kernel<<<blocks, kThreads, 0, s>>>(n, H, S, D, scale, acc, (float*)out, accumulate);
    return launched("convert");
}

}  // namespace dfa
