// tc_selftest.cu -- bring-up hooks of include/dfa_debug.h: one 128x128x128
// tcgen05 product per operand form (exactly the descriptors, swizzle and TMEM
// layouts of the attention kernels, so each form can be checked on its own),
// and a kernel whose bounded waits run out, to test failure detection
// without faulting or hanging the GPU.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dfa_debug.h"
#include "internal.h"
#include "ptx.cuh"

namespace dfa {
namespace {

using namespace ptx;

constexpr int N = 128;
constexpr int kTile = N * N * 2;   // 32 KB: two 16 KB swizzle blocks of 64 columns

__global__ void __launch_bounds__(128, 1)
mma_selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int form,
                    const __nv_bfloat16* __restrict__ A, float* __restrict__ C, int* err) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kTile;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kTile);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 5);
    const int t = threadIdx.x, warp = t / 32;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    if (t == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;   // D at columns [0,128), A (form 1) at [128,192)

    if (form == 1) {
        // Row t of A into TMEM lane t as bf16 pairs.
        const uint32_t* row = reinterpret_cast<const uint32_t*>(A + (size_t)t * N);
        for (int c = 0; c < 2; ++c) {
            uint32_t u[32];
            for (int e = 0; e < 32; ++e) u[e] = row[c * 32 + e];
            tmem_st32(tmem + lane_base + 128 + c * 32, u);
        }
        tmem_st_wait();
    } else if (form == 2 || form == 3) {
        // Thread t writes row t of A (128 elements) into two 64-column swizzled blocks.
        for (int c = 0; c < N; c += 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(A + (size_t)t * N + c);
            *reinterpret_cast<uint4*>(sA + (c / 64) * 16384 + sw128_offset(t, c % 64)) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (t == 0) {
        const uint32_t bytes = (form == 0 ? 2 : 1) * kTile;
        mbar_arrive_expect_tx(&bars[0], bytes);
        for (int blk = 0; blk < 2; ++blk) {
            if (form == 0) tma_load_4d(sA + blk * 16384, &tmA, &bars[0], blk * 64, 0, 0, 0);
            tma_load_4d(sB + blk * 16384, &tmB, &bars[0], blk * 64, 0, 0, 0);
        }
    }
    bool ok = mbar_wait(&bars[0], 0, abort_flag, err);
    tc_fence_after();
    if (t == 0 && ok) {
        const uint32_t a = smem_u32(sA), b = smem_u32(sB);
        for (int kk = 0; kk < N / 16; ++kk) {
            const uint32_t kmaj = (kk / 4) * 16384 + (kk % 4) * 32;   // K-major step
            const uint32_t mnmaj = kk * 2048;                          // MN-major step (16 rows)
            if (form == 0) {
                mma_ss(tmem, sdesc_sw128(a + kmaj, 16, 1024), sdesc_sw128(b + kmaj, 16, 1024),
                       idesc_bf16_f32(128, 128, false, false), kk > 0);
            } else if (form == 1) {
                mma_ts(tmem, tmem + 128 + kk * 8, sdesc_sw128(b + mnmaj, 16384, 1024),
                       idesc_bf16_f32(128, 128, false, true), kk > 0);
            } else if (form == 2) {
                mma_ss(tmem, sdesc_sw128(a + mnmaj, 16384, 1024), sdesc_sw128(b + mnmaj, 16384, 1024),
                       idesc_bf16_f32(128, 128, true, true), kk > 0);
            } else {
                mma_ss(tmem, sdesc_sw128(a + kmaj, 16, 1024), sdesc_sw128(b + kmaj, 16, 1024),
                       idesc_bf16_f32(128, 128, false, false), kk > 0);
            }
        }
        mma_commit(&bars[1]);
    }
    __syncwarp();
    ok = mbar_wait(&bars[1], 0, abort_flag, err) && ok;
    tc_fence_after();
    for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + c * 32, u);
        for (int e = 0; e < 32; ++e) C[(size_t)t * N + c * 32 + e] = ok ? __uint_as_float(u[e]) : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// Two warps wait on mbarriers that nothing ever arrives on, through the same
// bounded wait as the attention kernels.  Warp 0 gives up after the limit and
// raises the CTA's abort flag and the device error flag; warp 1 (no error
// flag of its own) leaves on the abort flag or on its own limit, as the other
// roles of a CTA do.  out[w] = 1 if warp w's wait completed, 0 if it gave up.
__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(int* err, int* out) {
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x / 32;
    const bool ok = mbar_wait(&bars[warp], 0, &abort_flag, warp == 0 ? err : nullptr);
    if (out && (threadIdx.x & 31) == 0) out[warp] = ok ? 1 : 0;
}

}  // namespace
}  // namespace dfa

extern "C" dfa_status dfa_debug_wait_timeout(int* out, void* stream) {
    using namespace dfa;
    if (out && (reinterpret_cast<uintptr_t>(out) & 3u)) return fail(DFA_ERR_INVALID_ARG, "misaligned out");
    int* err = device_error_flag();
    if (!err) return fail(DFA_ERR_CUDA, "device error flag unavailable");
    wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(err, out);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "wait-timeout launch: %s", cudaGetErrorString(e));
}

extern "C" dfa_status dfa_debug_mma(int form, const void* A, const void* B, float* C, void* stream) {
    using namespace dfa;
    if (form < 0 || form > 3) return fail(DFA_ERR_INVALID_ARG, "unknown form %d", form);
    if (!A || !B || !C || ((uintptr_t)A | (uintptr_t)B | (uintptr_t)C) & 15u)
        return fail(DFA_ERR_INVALID_ARG, "null or misaligned pointer");
    CUtensorMap ma, mb;
    // A [128, 128] and B [128, 128] row-major bf16 seen as [B=1, L=128, heads=1, D=128].
    if (!make_tmap_bshd(&ma, A, 1, N, 1, N, (int64_t)N * N, N, N) ||
        !make_tmap_bshd(&mb, B, 1, N, 1, N, (int64_t)N * N, N, N))
        return fail(DFA_ERR_CUDA, "tensor map encoding failed");
    const int smem = 2 * kTile + 1024 + 1024;
    if (cudaFuncSetAttribute(mma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "selftest smem attribute");
    mma_selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        ma, mb, form, static_cast<const __nv_bfloat16*>(A), C, device_error_flag());
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
}
