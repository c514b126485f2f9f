// noalloc.cu -- dfa_attn_fwd_noalloc: the whole-sequence forward for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run attention: a framework plugin whose host owns every byte of
// device memory through its own pool, or a service that forbids allocation
// once it has started serving.  dfa_attn_fwd needs a caller workspace only for
// its per-CTA work list; this entry point keeps that list in a fixed
// file-scope device array instead, so the caller passes only inputs and
// outputs.
//
// The array is shared by every call in the process and keeps whatever the
// last call wrote; each call rewrites the part it uses before its kernel
// reads it.  Calls whose kernels overlap on the GPU (different streams, or
// several host threads) race on the array.
//
// The list is uploaded from a host array shared by all calls, with a pageable
// copy.  A captured copy would read that array when the graph is replayed,
// after later calls may have rewritten it for another shape, so a call on a
// capturing stream is refused (DFA_ERR_INVALID_ARG) before anything is
// enqueued.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "internal.h"

namespace dfa {
namespace {

// Capacity of the static work list, in int32 entries (4 MiB per device).
constexpr int64_t kNoAllocEntries = int64_t(1) << 20;
// Worst-case persistent grid used for the capacity check (device independent).
constexpr int64_t kNoAllocMaxWorkers = 1024;
constexpr int kUnitRows = 256;       // query rows per forward work unit

// Device scratch: offsets[workers + 1] followed by the item values.
static __device__ __align__(256) int32_t g_noalloc_list[kNoAllocEntries];

// Host staging copy of the list (static, so building it allocates nothing).
int32_t g_host_list[kNoAllocEntries];
std::mutex g_host_mu;

constexpr int kMaxDev = 64;
int32_t* g_dev_ptr[kMaxDev] = {};
std::mutex g_setup_mu;

// Device address of g_noalloc_list on the current device, looked up once per
// device with that device current.
dfa_status scratch_address(int32_t** out) {
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess || d < 0 || d >= kMaxDev)
        return fail(DFA_ERR_CUDA, "no current CUDA device (%s)", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_dev_ptr[d]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_list);
        if (e != cudaSuccess || !p)
            return fail(DFA_ERR_CUDA, "cudaGetSymbolAddress of the static work list failed: %s",
                        cudaGetErrorString(e));
        g_dev_ptr[d] = static_cast<int32_t*>(p);
    }
    *out = g_dev_ptr[d];
    return DFA_OK;
}

inline int64_t lo(int64_t n, int64_t parts, int64_t r) { return (n * r) / parts; }

// The same schedules as dfa_build_worklist, written straight into `buf`
// (offsets[W + 1], then items) without any allocation: a counting pass sizes
// every worker's range, a second pass fills it.
void build_list(int64_t rows, int64_t units, int64_t W, dfa_sched sched, int32_t* buf) {
    int32_t* off = buf;
    int32_t* items = buf + W + 1;
    for (int64_t w = 0; w <= W; ++w) off[w] = 0;
    const int64_t pairs = (units + 1) / 2;
    if (sched == DFA_SCHED_UNBALANCED) {
        for (int64_t w = 0; w < W; ++w) off[w + 1] = (int32_t)(rows * (lo(units, W, w + 1) - lo(units, W, w)));
    } else {
        for (int64_t t = 0; t < rows * pairs; ++t) {
            const int64_t u = t % pairs;
            off[t % W + 1] += (units - 1 - u != u) ? 2 : 1;
        }
    }
    for (int64_t w = 0; w < W; ++w) off[w + 1] += off[w];
    // Fill: off[w] is used as the running cursor, then restored.
    if (sched == DFA_SCHED_UNBALANCED) {
        for (int64_t w = 0; w < W; ++w) {
            int64_t pos = off[w];
            for (int64_t row = 0; row < rows; ++row)
                for (int64_t u = lo(units, W, w); u < lo(units, W, w + 1); ++u)
                    items[pos++] = (int32_t)(row * units + u);
        }
    } else {
        for (int64_t w = W; w > 0; --w) off[w] = off[w - 1];
        off[0] = 0;
        for (int64_t t = 0; t < rows * pairs; ++t) {
            const int64_t row = t / pairs, u = t % pairs, w = t % W, heavy = units - 1 - u;
            items[off[w + 1]++] = (int32_t)(row * units + heavy);
            if (heavy != u) items[off[w + 1]++] = (int32_t)(row * units + u);
        }
    }
}

}  // namespace
}  // namespace dfa

using namespace dfa;

extern "C" dfa_status dfa_attn_fwd_noalloc(const void* q, const void* k, const void* v, dfa_dtype dt,
                                           int B, int H, int H_kv, int S, int D, int n_chunks, int causal,
                                           float scale, dfa_sched sched, void* O, float* lse, void* stream) {
    if (dt != DFA_F32 && dt != DFA_BF16) return fail(DFA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    if (B < 0 || H <= 0 || H_kv <= 0 || S < 0) return fail(DFA_ERR_INVALID_ARG, "bad sizes");
    if (H % H_kv != 0) return fail(DFA_ERR_INVALID_ARG, "H (%d) must be a multiple of H_kv (%d)", H, H_kv);
    if (D != 64 && D != 128) return fail(DFA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DFA_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (!chunks_valid(S, n_chunks))
        return fail(DFA_ERR_INVALID_ARG, "S=%d does not split into n_chunks=%d non-empty chunks of ceil(S/n_chunks) tokens",
                    S, n_chunks);
    if (sched != DFA_SCHED_BALANCED && sched != DFA_SCHED_UNBALANCED && sched != DFA_SCHED_SPLIT_KV)
        return fail(DFA_ERR_INVALID_ARG, "unknown schedule %d", (int)sched);
    if (sched == DFA_SCHED_SPLIT_KV) sched = DFA_SCHED_BALANCED;   // no workspace for pieces
    if ((int64_t)B * S == 0) return DFA_OK;
    const int64_t rows = (int64_t)B * H, units = (S + kUnitRows - 1) / kUnitRows;
    if (kNoAllocMaxWorkers + 1 + rows * units > kNoAllocEntries)
        return fail(DFA_ERR_INVALID_ARG,
                    "B*H*ceil(S/256) = %lld work items exceed the static work list (at most %lld items)",
                    (long long)(rows * units), (long long)(kNoAllocEntries - kNoAllocMaxWorkers - 1));
    for (const void* p : {q, k, v, (const void*)O, (const void*)lse})
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15u))
            return fail(DFA_ERR_INVALID_ARG, "null or not 16-byte aligned pointer");
    AttnProblem p{};
    p.B = B; p.H = H; p.Hkv = H_kv; p.Lq = S; p.Lkv = S; p.D = D;
    p.q_sb = (int64_t)S * H * D; p.q_ss = (int64_t)H * D; p.q_sh = D;
    p.kv_sb = (int64_t)S * H_kv * D; p.kv_ss = (int64_t)H_kv * D; p.kv_sh = D;
    p.q_offset = 0; p.kv_offset = 0; p.causal = causal != 0; p.scale = scale;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(s, &cap);
    if (ce != cudaSuccess) return fail(DFA_ERR_CUDA, "cudaStreamIsCapturing: %s", cudaGetErrorString(ce));
    if (cap != cudaStreamCaptureStatusNone)
        return fail(DFA_ERR_INVALID_ARG,
                    "dfa_attn_fwd_noalloc cannot be captured in a CUDA graph: its work-list upload reads a "
                    "shared host array when it runs; use dfa_attn_fwd with a workspace under capture");
    dfa_status st;
    if (dt == DFA_F32) {
        st = simt_fwd(p, dt, q, k, v, O, true, lse, s);    // needs no scratch
    } else {
        int32_t* dev = nullptr;
        if ((st = scratch_address(&dev))) return st;
        const int workers = (int)std::min<int64_t>(num_sms(), rows * units);
        const size_t count = (size_t)workers + 1 + (size_t)(rows * units);
        {
            // The pageable copy has read the staging buffer when it returns,
            // so the lock only has to cover build + enqueue.
            std::lock_guard<std::mutex> lk(g_host_mu);
            build_list(rows, units, workers, sched, g_host_list);
            cudaError_t e = cudaMemcpyAsync(dev, g_host_list, count * sizeof(int32_t), cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "work-list upload: %s", cudaGetErrorString(e));
        }
        WorkList wl{dev, dev + workers + 1, workers, (int)units};
        st = tc_fwd(p, q, k, v, O, false, lse, &wl, s);
    }
    if (st == DFA_OK) count_launch(DFA_KERNEL_FWD);
    return st;
}
