// dfa_api.cu -- the C ABI (include/dfa.h): argument validation, workspace
// layout, work-list upload, dispatch to the kernels and error reporting.
// No exception crosses this boundary and no device memory is allocated here.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "internal.h"

namespace dfa {
namespace {

thread_local char g_msg[512] = "";
std::atomic<int64_t> g_launches[DFA_KERNEL_KINDS];

// Set by a kernel that gave up on a bounded wait; read by dfa_check_errors.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

constexpr int kMaxWorkers = 1024;    // upper bound on the persistent grid
constexpr int kFwdUnitRows = 256;    // query rows per forward work unit
constexpr int kBwdUnitRows = 128;    // key rows per backward work unit

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}

// Host-side cache of built work lists, kept in pinned memory so the upload is
// a plain async copy (also legal inside stream capture).
struct CachedList {
    int32_t* host = nullptr;  // offsets[W+1] followed by items[n]
    size_t count = 0;
    int workers = 0;
};
std::map<std::tuple<int, int, int, int>, CachedList> g_lists;

// Returns the pinned host copy of the list (nullptr on failure).
const CachedList* get_list(int rows, int units, int workers, dfa_sched sched) {
    if (sched == DFA_SCHED_SPLIT_KV) sched = DFA_SCHED_BALANCED;   // pieces are listed by get_split_list
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(rows, units, workers, (int)sched);
    auto it = g_lists.find(key);
    if (it != g_lists.end()) return &it->second;
    const size_t n = (size_t)rows * units;
    CachedList c;
    c.count = (size_t)workers + 1 + n;
    c.workers = workers;
    if (cudaHostAlloc((void**)&c.host, c.count * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess)
        return nullptr;
    if (dfa_build_worklist(rows, units, workers, sched, c.host, c.host + workers + 1) < 0) {
        cudaFreeHost(c.host);
        return nullptr;
    }
    return &(g_lists[key] = c);
}

// Split-kv pieces of a forward (dfa_build_split_worklist), cached like the
// plain lists; key (rows, units, kv_tiles, causal, piece_tiles, workers).
std::map<std::tuple<int, int, int, int, int, int>, CachedList> g_split_lists;

int64_t count_pieces(int rows, int units, int kv_tiles, int causal, int piece) {
    int64_t n = 0;
    for (int u = 0; u < units; ++u) {
        const int hi = causal ? std::min(2 * u + 2, kv_tiles) : kv_tiles;
        n += (hi + piece - 1) / piece;
    }
    return n * rows;
}

const CachedList* get_split_list(int rows, int units, int kv_tiles, int causal, int piece, int workers) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(rows, units, kv_tiles, causal, piece, workers);
    auto it = g_split_lists.find(key);
    if (it != g_split_lists.end()) return &it->second;
    const int64_t n = count_pieces(rows, units, kv_tiles, causal, piece);
    CachedList c;
    c.count = (size_t)workers + 1 + (size_t)n;
    c.workers = workers;
    if (cudaHostAlloc((void**)&c.host, c.count * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess)
        return nullptr;
    if (dfa_build_split_worklist(rows, units, kv_tiles, causal, piece, workers, c.host, c.host + workers + 1) < 0 ||
        c.host[workers] != n) {
        cudaFreeHost(c.host);
        return nullptr;
    }
    return &(g_split_lists[key] = c);
}

// Backward split-kv pieces (dfa_build_bwd_split_worklist); key (rows,
// kv_tiles, causal, piece_tiles, workers).
std::map<std::tuple<int, int, int, int, int>, CachedList> g_bwd_split_lists;

int64_t count_bwd_pieces(int rows, int kv_tiles, int causal, int piece) {
    int64_t n = 0;
    for (int t = 0; t < kv_tiles; ++t) n += ((causal ? kv_tiles - t : kv_tiles) + piece - 1) / piece;
    return n * rows;
}

const CachedList* get_bwd_split_list(int rows, int kv_tiles, int causal, int piece, int workers) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(rows, kv_tiles, causal, piece, workers);
    auto it = g_bwd_split_lists.find(key);
    if (it != g_bwd_split_lists.end()) return &it->second;
    const int64_t n = count_bwd_pieces(rows, kv_tiles, causal, piece);
    CachedList c;
    c.count = (size_t)workers + 1 + (size_t)n;
    c.workers = workers;
    if (cudaHostAlloc((void**)&c.host, c.count * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess)
        return nullptr;
    if (dfa_build_bwd_split_worklist(rows, kv_tiles, causal, piece, workers, c.host, c.host + workers + 1) < 0 ||
        c.host[workers] != n) {
        cudaFreeHost(c.host);
        return nullptr;
    }
    return &(g_bwd_split_lists[key] = c);
}

struct Layout {
    size_t delta = 0, nlse2 = 0, dq = 0, wl = 0, opart = 0, lpart = 0, dk = 0, dv = 0, total = 0;
    int S_pad = 0;
    int n_split = 1;   // split-kv pieces the workspace has room for
};

Layout layout(int B, int H, int Hkv, int S, int D, bool bwd) {
    Layout L;
    size_t off = 0;
    L.S_pad = (S + kBwdUnitRows - 1) / kBwdUnitRows * kBwdUnitRows;
    if (bwd) {
        L.delta = off;
        off = align_up(off + sizeof(float) * (size_t)B * H * L.S_pad);
        L.nlse2 = off;
        off = align_up(off + sizeof(float) * (size_t)B * H * L.S_pad);
        L.dq = off;
        off = align_up(off + sizeof(float) * (size_t)B * S * H * D);
    }
    L.wl = off;
    const size_t units = bwd ? (size_t)(S + kBwdUnitRows - 1) / kBwdUnitRows
                             : (size_t)(S + kFwdUnitRows - 1) / kFwdUnitRows;
    const size_t rows = bwd ? (size_t)B * Hkv : (size_t)B * H;
    // Room for SPLIT_KV pieces when the problem is small enough to be split;
    // the causal plan has the shortest pieces, so it bounds both masks.
    const int piece = bwd ? (D == 128 ? dfa_split_bwd_piece_tiles(B, Hkv, S, 1, num_sms()) : 0)
                          : dfa_split_piece_tiles(B, H, S, 1, num_sms());
    if (piece > 0) L.n_split = (int)(((S + 127) / 128 + piece - 1) / piece);
    off = align_up(off + sizeof(int32_t) * (kMaxWorkers + 1 + rows * units * (size_t)L.n_split));
    if (bwd && L.n_split > 1) {   // fp32 dK, dV accumulators [B, S, H_kv, D] the pieces add into
        L.dk = off;
        off = align_up(off + sizeof(float) * (size_t)B * S * Hkv * D);
        L.dv = off;
        off = align_up(off + sizeof(float) * (size_t)B * S * Hkv * D);
    }
    if (L.n_split > 1) {
        L.opart = off;
        off = align_up(off + sizeof(float) * (size_t)L.n_split * B * S * H * D);
        L.lpart = off;
        off = align_up(off + sizeof(float) * (size_t)L.n_split * B * H * S);
    }
    L.total = off;
    return L;
}

dfa_status check_common(int B, int H, int Hkv, int D, float scale) {
    if (B < 0 || H <= 0 || Hkv <= 0) return fail(DFA_ERR_INVALID_ARG, "B/H/H_kv must be >= 0/> 0/> 0");
    if (H % Hkv != 0) return fail(DFA_ERR_INVALID_ARG, "H (%d) must be a multiple of H_kv (%d)", H, Hkv);
    if (D != 64 && D != 128) return fail(DFA_ERR_UNSUPPORTED, "head dim D=%d (supported: 64, 128)", D);
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(DFA_ERR_INVALID_ARG, "scale must be finite and > 0");
    return DFA_OK;
}

dfa_status check_dtype(dfa_dtype dt) {
    if (dt != DFA_F32 && dt != DFA_BF16) return fail(DFA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
    return DFA_OK;
}

dfa_status check_ptrs(std::initializer_list<const void*> ps) {
    for (const void* p : ps) {
        if (!p) return fail(DFA_ERR_INVALID_ARG, "null pointer");
        if (!aligned16(p)) return fail(DFA_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", p);
    }
    return DFA_OK;
}

dfa_status upload_list(const CachedList* c, void* dst, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(dst, c->host, c->count * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    return e == cudaSuccess ? DFA_OK : fail(DFA_ERR_CUDA, "work-list upload: %s", cudaGetErrorString(e));
}

}  // namespace

dfa_status fail(dfa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

void count_launch(dfa_kernel_kind kind, int n) { g_launches[kind].fetch_add(n); }

namespace {
std::atomic<uint64_t*> g_trace{nullptr};
std::atomic<int> g_trace_cap{0};
}  // namespace

uint64_t* cta_trace(int* capacity) {
    *capacity = g_trace_cap.load();
    return g_trace.load();
}

int* device_error_flag() {
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[d] = static_cast<int*>(p);
    }
    return g_err_ptr[d];
}

int num_sms() {
    const int d = current_device();
    if (d < 0) return 1;
    if (!g_sms[d]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 1;
    }
    return g_sms[d];
}

}  // namespace dfa

using namespace dfa;


extern "C" const char* dfa_last_error(void) { return g_msg; }

extern "C" dfa_status dfa_debug_cta_trace(uint64_t* buf, int capacity) {
    if (buf && (capacity <= 0 || (reinterpret_cast<uintptr_t>(buf) & 7u)))
        return fail(DFA_ERR_INVALID_ARG, "trace buffer needs capacity > 0 and 8-byte alignment");
    g_trace_cap.store(buf ? capacity : 0);
    g_trace.store(buf);
    return DFA_OK;
}

extern "C" int64_t dfa_launch_count(dfa_kernel_kind kind) {
    if (kind < 0 || kind >= DFA_KERNEL_KINDS) return -1;
    return g_launches[kind].load();
}

// dfa_copy: both sides must be reachable by the SMs (device, managed or pinned
// host memory); pageable host memory is refused rather than guessed at.
static dfa_status check_copy_side(const void* p, const char* which) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return fail(DFA_ERR_INVALID_ARG, "dfa_copy: %s is not a CUDA-visible pointer", which);
    }
    if (at.type == cudaMemoryTypeUnregistered)
        return fail(DFA_ERR_INVALID_ARG, "dfa_copy: %s is pageable host memory (pin it first)", which);
    return DFA_OK;
}

extern "C" dfa_status dfa_copy(void* dst, const void* src, size_t bytes, void* stream) {
    g_msg[0] = 0;
    if (bytes == 0) return DFA_OK;
    if (!dst || !src) return fail(DFA_ERR_INVALID_ARG, "dfa_copy: null pointer");
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), r = reinterpret_cast<uintptr_t>(src);
    if (d < r + bytes && r < d + bytes) return fail(DFA_ERR_INVALID_ARG, "dfa_copy: source and destination overlap");
    dfa_status st;
    if ((st = check_copy_side(dst, "dst")) || (st = check_copy_side(src, "src"))) return st;
    st = launch_copy(dst, src, bytes, static_cast<cudaStream_t>(stream));
    if (st == DFA_OK) count_launch(DFA_KERNEL_COPY);
    return st;
}

extern "C" size_t dfa_attn_workspace_size(int B, int H, int H_kv, int S, int D, int n_chunks, int bwd) {
    if (B < 0 || H <= 0 || H_kv <= 0 || S < 0 || n_chunks <= 0 || (D != 64 && D != 128)) return 0;
    if (H % H_kv != 0 || !chunks_valid(S, n_chunks)) return 0;
    return layout(B, H, H_kv, S, D, bwd != 0).total;
}

extern "C" dfa_status dfa_chunk_attn_fwd(const void* q, const void* k, const void* v, dfa_dtype dt,
                                         int B, int H, int H_kv, int Lq, int Lkv, int D,
                                         const int64_t* q_strides, const int64_t* kv_strides,
                                         int64_t q_offset, int64_t kv_offset, int causal, float scale,
                                         float* O_partial, float* lse, void* stream) {
    g_msg[0] = 0;
    dfa_status st;
    if ((st = check_dtype(dt)) || (st = check_common(B, H, H_kv, D, scale))) return st;
    if (Lq < 0 || Lkv < 0) return fail(DFA_ERR_INVALID_ARG, "negative chunk length");
    if (q_offset < 0 || kv_offset < 0) return fail(DFA_ERR_INVALID_ARG, "negative chunk offset");
    if ((int64_t)B * Lq == 0) return DFA_OK;
    if ((st = check_ptrs({q, O_partial, lse}))) return st;
    if (Lkv > 0 && (st = check_ptrs({k, v}))) return st;
    AttnProblem p{};
    p.B = B; p.H = H; p.Hkv = H_kv; p.Lq = Lq; p.Lkv = Lkv; p.D = D;
    p.q_sb = q_strides ? q_strides[0] : (int64_t)Lq * H * D;
    p.q_ss = q_strides ? q_strides[1] : (int64_t)H * D;
    p.q_sh = q_strides ? q_strides[2] : D;
    p.kv_sb = kv_strides ? kv_strides[0] : (int64_t)Lkv * H_kv * D;
    p.kv_ss = kv_strides ? kv_strides[1] : (int64_t)H_kv * D;
    p.kv_sh = kv_strides ? kv_strides[2] : D;
    for (int64_t x : {p.q_sb, p.q_ss, p.q_sh, p.kv_sb, p.kv_ss, p.kv_sh})
        if (x < 0 || x % 8 != 0) return fail(DFA_ERR_INVALID_ARG, "strides must be non-negative multiples of 8 elements");
    p.q_offset = q_offset; p.kv_offset = kv_offset; p.causal = causal != 0; p.scale = scale;
    if (Lkv == 0) {
        // No keys: every row is empty (O = 0, lse = -inf) -- handled by the kernels'
        // empty-row path with an empty key loop.
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == DFA_F32) {
        st = simt_fwd(p, dt, q, k, v, O_partial, true, lse, s);
    } else {
        st = tc_fwd(p, q, k, v, O_partial, true, lse, nullptr, s);
    }
    if (st == DFA_OK) count_launch(DFA_KERNEL_FWD);
    return st;
}

extern "C" dfa_status dfa_merge_partials(int B, int H, int L, int D, const float* O_a, const float* lse_a,
                                         const float* O_b, const float* lse_b, float* O_out, float* lse_out,
                                         void* stream) {
    g_msg[0] = 0;
    if (B < 0 || H <= 0 || L < 0 || D <= 0 || D % 4 != 0)
        return fail(DFA_ERR_INVALID_ARG, "bad merge sizes (B=%d H=%d L=%d D=%d)", B, H, L, D);
    if ((int64_t)B * L == 0) return DFA_OK;
    dfa_status st;
    if ((st = check_ptrs({O_a, lse_a, O_b, lse_b, O_out, lse_out}))) return st;
    st = launch_merge(B, H, L, D, O_a, lse_a, O_b, lse_b, O_out, lse_out, static_cast<cudaStream_t>(stream));
    if (st == DFA_OK) count_launch(DFA_KERNEL_MERGE);
    return st;
}

static dfa_status check_whole(dfa_dtype dt, int B, int H, int H_kv, int S, int D, int n_chunks,
                              float scale, dfa_sched sched, void* workspace, size_t ws_bytes, bool bwd) {
    dfa_status st;
    if ((st = check_dtype(dt)) || (st = check_common(B, H, H_kv, D, scale))) return st;
    if (S < 0) return fail(DFA_ERR_INVALID_ARG, "negative sequence length");
    if (!chunks_valid(S, n_chunks))
        return fail(DFA_ERR_INVALID_ARG, "S=%d does not split into n_chunks=%d non-empty chunks of ceil(S/n_chunks) tokens",
                    S, n_chunks);
    if (sched != DFA_SCHED_BALANCED && sched != DFA_SCHED_UNBALANCED && sched != DFA_SCHED_SPLIT_KV)
        return fail(DFA_ERR_INVALID_ARG, "unknown schedule %d", (int)sched);
    if ((int64_t)B * S == 0) return DFA_OK;
    const size_t need = layout(B, H, H_kv, S, D, bwd).total;
    if (!workspace || ws_bytes < need)
        return fail(DFA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(workspace)) return fail(DFA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    return DFA_OK;
}

static AttnProblem whole_problem(int B, int H, int H_kv, int S, int D, int causal, float scale,
                                 int n_chunks = 1, int window = 0) {
    AttnProblem p{};
    if (window > 0) {
        p.win_c = chunk_tokens(S, n_chunks);   // the last chunk may be shorter
        p.win_w = window;
    }
    p.B = B; p.H = H; p.Hkv = H_kv; p.Lq = S; p.Lkv = S; p.D = D;
    p.q_sb = (int64_t)S * H * D; p.q_ss = (int64_t)H * D; p.q_sh = D;
    p.kv_sb = (int64_t)S * H_kv * D; p.kv_ss = (int64_t)H_kv * D; p.kv_sh = D;
    p.q_offset = 0; p.kv_offset = 0; p.causal = causal != 0; p.scale = scale;
    return p;
}

static dfa_status check_window(int causal, int window) {
    if (window < 1) return fail(DFA_ERR_INVALID_ARG, "window must be at least one chunk (got %d)", window);
    if (!causal) return fail(DFA_ERR_INVALID_ARG, "a local window needs causal attention");
    return DFA_OK;
}

static dfa_status attn_fwd_impl(const void* q, const void* k, const void* v, dfa_dtype dt, int B, int H,
                                int H_kv, int S, int D, int n_chunks, int causal, int window, float scale,
                                dfa_sched sched, void* O, float* lse, void* workspace, size_t ws_bytes,
                                void* stream) {
    g_msg[0] = 0;
    dfa_status st = check_whole(dt, B, H, H_kv, S, D, n_chunks, scale, sched, workspace, ws_bytes, false);
    if (st || (window && (st = check_window(causal, window))) || (int64_t)B * S == 0) return st;
    if ((st = check_ptrs({q, k, v, O, lse}))) return st;
    const AttnProblem p = whole_problem(B, H, H_kv, S, D, causal, scale, n_chunks, window);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == DFA_F32) {
        st = simt_fwd(p, dt, q, k, v, O, true, lse, s);
    } else {
        const Layout L = layout(B, H, H_kv, S, D, false);
        const int units = (S + kFwdUnitRows - 1) / kFwdUnitRows;
        const int piece = sched == DFA_SCHED_SPLIT_KV && !window ? dfa_split_piece_tiles(B, H, S, causal, num_sms()) : 0;
        if (piece > 0) {
            // Helper items: pieces of every block's key range, partials to the
            // workspace, then the rescale-and-merge of each row's pieces.
            const int kv_tiles = (S + 127) / 128, n_split = (kv_tiles + piece - 1) / piece;
            if (n_split > L.n_split) return fail(DFA_ERR_WORKSPACE, "split-kv plan exceeds the workspace layout");
            const int64_t n = count_pieces(B * H, units, kv_tiles, causal != 0, piece);
            const int workers = (int)std::min<int64_t>(num_sms(), n);
            const CachedList* c = get_split_list(B * H, units, kv_tiles, causal != 0, piece, workers);
            if (!c) return fail(DFA_ERR_CUDA, "could not build the split-kv work list");
            int32_t* dev = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.wl);
            if ((st = upload_list(c, dev, s))) return st;
            WorkList wl{dev, dev + workers + 1, workers, units};
            wl.n_split = n_split;
            wl.piece_tiles = piece;
            float* opart = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.opart);
            float* lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.lpart);
            if ((st = tc_fwd(p, q, k, v, opart, true, lpart, &wl, s))) return st;
            count_launch(DFA_KERNEL_FWD);
            st = launch_merge_pieces(dt, B, H, S, D, causal != 0, piece, n_split, opart, lpart, O, lse, s);
            if (st == DFA_OK) count_launch(DFA_KERNEL_MERGE);
            return st;
        }
        const int workers = std::min(num_sms(), B * H * units);
        const CachedList* c = get_list(B * H, units, workers, sched);
        if (!c) return fail(DFA_ERR_CUDA, "could not build the work list");
        int32_t* dev = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.wl);
        if ((st = upload_list(c, dev, s))) return st;
        WorkList wl{dev, dev + workers + 1, workers, units};
        st = tc_fwd(p, q, k, v, O, false, lse, &wl, s);
    }
    if (st == DFA_OK) count_launch(DFA_KERNEL_FWD);
    return st;
}

extern "C" dfa_status dfa_attn_fwd(const void* q, const void* k, const void* v, dfa_dtype dt, int B, int H,
                                   int H_kv, int S, int D, int n_chunks, int causal, float scale,
                                   dfa_sched sched, void* O, float* lse, void* workspace, size_t ws_bytes,
                                   void* stream) {
    return attn_fwd_impl(q, k, v, dt, B, H, H_kv, S, D, n_chunks, causal, 0, scale, sched, O, lse, workspace,
                         ws_bytes, stream);
}

extern "C" dfa_status dfa_attn_fwd_local(const void* q, const void* k, const void* v, dfa_dtype dt, int B,
                                         int H, int H_kv, int S, int D, int n_chunks, int window, float scale,
                                         dfa_sched sched, void* O, float* lse, void* workspace,
                                         size_t ws_bytes, void* stream) {
    g_msg[0] = 0;
    if (window < 1) return fail(DFA_ERR_INVALID_ARG, "window must be at least one chunk (got %d)", window);
    return attn_fwd_impl(q, k, v, dt, B, H, H_kv, S, D, n_chunks, 1, window, scale, sched, O, lse, workspace,
                         ws_bytes, stream);
}

static dfa_status attn_bwd_impl(const void* q, const void* k, const void* v, const void* O, const float* lse,
                                const void* dO, dfa_dtype dt, int B, int H, int H_kv, int S, int D,
                                int n_chunks, int causal, int window, float scale, dfa_sched sched, void* dQ,
                                void* dK, void* dV, void* workspace, size_t ws_bytes, void* stream) {
    g_msg[0] = 0;
    dfa_status st = check_whole(dt, B, H, H_kv, S, D, n_chunks, scale, sched, workspace, ws_bytes, true);
    if (st || (window && (st = check_window(causal, window))) || (int64_t)B * S == 0) return st;
    if ((st = check_ptrs({q, k, v, O, lse, dO, dQ, dK, dV}))) return st;
    const AttnProblem p = whole_problem(B, H, H_kv, S, D, causal, scale, n_chunks, window);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout L = layout(B, H, H_kv, S, D, true);
    char* ws = static_cast<char*>(workspace);
    float* delta = reinterpret_cast<float*>(ws + L.delta);
    if (dt == DFA_F32) {
        if ((st = launch_delta(dt, B, H, S, D, O, dO, delta, s))) return st;
        count_launch(DFA_KERNEL_DELTA);
        st = simt_bwd(p, dt, q, k, v, dO, lse, delta, dQ, dK, dV, s);
        if (st == DFA_OK) count_launch(DFA_KERNEL_BWD, 2);
        return st;
    }
    float* nlse2 = reinterpret_cast<float*>(ws + L.nlse2);
    if ((st = launch_bwd_prep(dt, B, H, S, L.S_pad, D, O, dO, lse, nlse2, delta, s))) return st;
    count_launch(DFA_KERNEL_DELTA);
    float* dq_acc = reinterpret_cast<float*>(ws + L.dq);
    cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)B * S * H * D, s);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "dQ accumulator clear: %s", cudaGetErrorString(e));
    const int units = (S + kBwdUnitRows - 1) / kBwdUnitRows;
    const int piece = sched == DFA_SCHED_SPLIT_KV && D == 128 && !window
                          ? dfa_split_bwd_piece_tiles(B, H_kv, S, causal, num_sms()) : 0;
    if (piece > 0) {
        // Helper items: pieces of every key tile's query range, each adding its
        // partial dK, dV to fp32 accumulators; then the bf16 casts.
        const int n_split = (units + piece - 1) / piece;
        if (n_split > L.n_split) return fail(DFA_ERR_WORKSPACE, "split-kv plan exceeds the workspace layout");
        const int64_t np = count_bwd_pieces(B * H_kv, units, causal != 0, piece);
        const int workers = (int)std::min<int64_t>(num_sms(), np);
        const CachedList* c = get_bwd_split_list(B * H_kv, units, causal != 0, piece, workers);
        if (!c) return fail(DFA_ERR_CUDA, "could not build the split-kv work list");
        int32_t* dev = reinterpret_cast<int32_t*>(ws + L.wl);
        if ((st = upload_list(c, dev, s))) return st;
        WorkList wl{dev, dev + workers + 1, workers, units};
        wl.n_split = n_split;
        wl.piece_tiles = piece;
        float* dk_acc = reinterpret_cast<float*>(ws + L.dk);
        float* dv_acc = reinterpret_cast<float*>(ws + L.dv);
        const size_t kv_elems = (size_t)B * S * H_kv * D;
        if ((e = cudaMemsetAsync(dk_acc, 0, sizeof(float) * kv_elems, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(dv_acc, 0, sizeof(float) * kv_elems, s)) != cudaSuccess)
            return fail(DFA_ERR_CUDA, "dK/dV accumulator clear: %s", cudaGetErrorString(e));
        if ((st = tc_bwd_pipelined(p, q, k, v, dO, nlse2, delta, L.S_pad, dq_acc, dk_acc, dv_acc, true, &wl, s)))
            return st;
        count_launch(DFA_KERNEL_BWD);
        if ((st = launch_convert(dt, B, H, S, D, scale, dq_acc, dQ, false, s)) ||
            (st = launch_cast_bf16((int64_t)kv_elems, dk_acc, dK, s)) ||
            (st = launch_cast_bf16((int64_t)kv_elems, dv_acc, dV, s)))
            return st;
        count_launch(DFA_KERNEL_CONVERT, 3);
        return DFA_OK;
    }
    const int workers = std::min(num_sms(), B * H_kv * units);
    const CachedList* c = get_list(B * H_kv, units, workers, sched);
    if (!c) return fail(DFA_ERR_CUDA, "could not build the work list");
    int32_t* dev = reinterpret_cast<int32_t*>(ws + L.wl);
    if ((st = upload_list(c, dev, s))) return st;
    WorkList wl{dev, dev + workers + 1, workers, units};
    if ((st = tc_bwd(p, q, k, v, dO, nlse2, delta, L.S_pad, dq_acc, dK, dV, &wl, s))) return st;
    count_launch(DFA_KERNEL_BWD);
    st = launch_convert(dt, B, H, S, D, scale, dq_acc, dQ, false, s);
    if (st == DFA_OK) count_launch(DFA_KERNEL_CONVERT);
    return st;
}

extern "C" dfa_status dfa_attn_bwd(const void* q, const void* k, const void* v, const void* O, const float* lse,
                                   const void* dO, dfa_dtype dt, int B, int H, int H_kv, int S, int D,
                                   int n_chunks, int causal, float scale, dfa_sched sched, void* dQ, void* dK,
                                   void* dV, void* workspace, size_t ws_bytes, void* stream) {
    return attn_bwd_impl(q, k, v, O, lse, dO, dt, B, H, H_kv, S, D, n_chunks, causal, 0, scale, sched, dQ, dK,
                         dV, workspace, ws_bytes, stream);
}

extern "C" dfa_status dfa_attn_bwd_local(const void* q, const void* k, const void* v, const void* O,
                                         const float* lse, const void* dO, dfa_dtype dt, int B, int H, int H_kv,
                                         int S, int D, int n_chunks, int window, float scale, dfa_sched sched,
                                         void* dQ, void* dK, void* dV, void* workspace, size_t ws_bytes,
                                         void* stream) {
    g_msg[0] = 0;
    if (window < 1) return fail(DFA_ERR_INVALID_ARG, "window must be at least one chunk (got %d)", window);
    return attn_bwd_impl(q, k, v, O, lse, dO, dt, B, H, H_kv, S, D, n_chunks, 1, window, scale, sched, dQ, dK,
                         dV, workspace, ws_bytes, stream);
}

// ---------------------------------------------------------------- chunk-pair backward
struct ChunkLayout {
    size_t delta = 0, nlse2 = 0, dq = 0, wl = 0, total = 0;
    int Lq_pad = 0;
};

ChunkLayout chunk_layout(int B, int H, int Hkv, int Lq, int Lkv, int D) {
    ChunkLayout L;
    size_t off = 0;
    L.Lq_pad = (Lq + kBwdUnitRows - 1) / kBwdUnitRows * kBwdUnitRows;
    L.delta = off;
    off = align_up(off + sizeof(float) * (size_t)B * H * L.Lq_pad);
    L.nlse2 = off;
    off = align_up(off + sizeof(float) * (size_t)B * H * L.Lq_pad);
    L.dq = off;
    off = align_up(off + sizeof(float) * (size_t)B * Lq * H * D);
    L.wl = off;
    const size_t units = (size_t)(Lkv + kBwdUnitRows - 1) / kBwdUnitRows;
    off = align_up(off + sizeof(int32_t) * (kMaxWorkers + 1 + (size_t)B * Hkv * units));
    L.total = off;
    return L;
}

extern "C" size_t dfa_chunk_bwd_workspace_size(int B, int H, int H_kv, int Lq, int Lkv, int D) {
    if (B < 0 || H <= 0 || H_kv <= 0 || Lq < 0 || Lkv < 0 || (D != 64 && D != 128) || H % H_kv != 0) return 0;
    return chunk_layout(B, H, H_kv, Lq, Lkv, D).total;
}

extern "C" dfa_status dfa_chunk_attn_bwd(const void* q, const void* k, const void* v, const void* O,
                                         const float* lse, const void* dO, dfa_dtype dt, int B, int H, int H_kv,
                                         int Lq, int Lkv, int D, int64_t q_offset, int64_t kv_offset, int causal,
                                         float scale, float* dQ_acc, float* dK_acc, float* dV_acc,
                                         void* workspace, size_t ws_bytes, void* stream) {
    g_msg[0] = 0;
    dfa_status st;
    if ((st = check_dtype(dt)) || (st = check_common(B, H, H_kv, D, scale))) return st;
    if (Lq < 0 || Lkv < 0) return fail(DFA_ERR_INVALID_ARG, "negative chunk length");
    if (q_offset < 0 || kv_offset < 0) return fail(DFA_ERR_INVALID_ARG, "negative chunk offset");
    if ((int64_t)B * Lq == 0 || Lkv == 0) return DFA_OK;   // nothing to add
    if ((st = check_ptrs({q, k, v, O, lse, dO, dQ_acc, dK_acc, dV_acc}))) return st;
    const ChunkLayout L = chunk_layout(B, H, H_kv, Lq, Lkv, D);
    if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(DFA_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned (got %zu)", L.total, ws_bytes);
    AttnProblem p{};
    p.B = B; p.H = H; p.Hkv = H_kv; p.Lq = Lq; p.Lkv = Lkv; p.D = D;
    p.q_sb = (int64_t)Lq * H * D; p.q_ss = (int64_t)H * D; p.q_sh = D;
    p.kv_sb = (int64_t)Lkv * H_kv * D; p.kv_ss = (int64_t)H_kv * D; p.kv_sh = D;
    p.q_offset = q_offset; p.kv_offset = kv_offset; p.causal = causal != 0; p.scale = scale;
    p.acc_out = 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* delta = reinterpret_cast<float*>(ws + L.delta);
    const bool tc = dt == DFA_BF16 && D == 128 && (kv_offset - q_offset) % kBwdUnitRows == 0;
    if (!tc) {
        if ((st = launch_delta(dt, B, H, Lq, D, O, dO, delta, s))) return st;
        count_launch(DFA_KERNEL_DELTA);
        st = simt_bwd(p, dt, q, k, v, dO, lse, delta, dQ_acc, dK_acc, dV_acc, s);
        if (st == DFA_OK) count_launch(DFA_KERNEL_BWD, 2);
        return st;
    }
    float* nlse2 = reinterpret_cast<float*>(ws + L.nlse2);
    if ((st = launch_bwd_prep(dt, B, H, Lq, L.Lq_pad, D, O, dO, lse, nlse2, delta, s))) return st;
    count_launch(DFA_KERNEL_DELTA);
    float* dq = reinterpret_cast<float*>(ws + L.dq);
    cudaError_t e = cudaMemsetAsync(dq, 0, sizeof(float) * (size_t)B * Lq * H * D, s);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "dQ accumulator clear: %s", cudaGetErrorString(e));
    const int units = (Lkv + kBwdUnitRows - 1) / kBwdUnitRows;
    const int workers = std::min(num_sms(), B * H_kv * units);
    const CachedList* c = get_list(B * H_kv, units, workers, DFA_SCHED_BALANCED);
    if (!c) return fail(DFA_ERR_CUDA, "could not build the work list");
    int32_t* dev = reinterpret_cast<int32_t*>(ws + L.wl);
    if ((st = upload_list(c, dev, s))) return st;
    WorkList wl{dev, dev + workers + 1, workers, units};
    if ((st = tc_bwd_pipelined(p, q, k, v, dO, nlse2, delta, L.Lq_pad, dq, dK_acc, dV_acc, true, &wl, s)))
        return st;
    count_launch(DFA_KERNEL_BWD);
    st = launch_convert(DFA_F32, B, H, Lq, D, scale, dq, dQ_acc, true, s);
    if (st == DFA_OK) count_launch(DFA_KERNEL_CONVERT);
    return st;
}

// ---------------------------------------------------------------- packed (variable-length) batches
namespace {

// Pinned host buffers for the per-call sequence table and work list of packed
// batches (these change with every batch, so they are not cached).  A ring of
// kStages buffers per device, each reused only after the copy that last read
// it has completed (an event recorded after the copy).
constexpr int kStages = 4;
struct Stage {
    int32_t* host = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    bool pending = false;
};
Stage g_stage[kMaxDevices][kStages];
int g_stage_next[kMaxDevices] = {};
std::mutex g_stage_mu;

struct VarlenLayout {
    size_t delta = 0, nlse2 = 0, dq = 0, seq = 0, wl = 0, total = 0;
    int64_t T = 0, P = 0;        // tokens; 128-row padded rows per head
    int units_max = 0;           // work units of the longest sequence
    int64_t items = 0;           // work items over all sequences and heads
};

// Validates the host offsets; returns false (with a message) on bad input.
bool varlen_sizes(const int32_t* cu, int n, int unit_rows, int heads, VarlenLayout* L) {
    if (n < 0) return fail(DFA_ERR_INVALID_ARG, "n_seq must be >= 0"), false;
    if (!cu) return fail(DFA_ERR_INVALID_ARG, "cu_seqlens is null"), false;
    if (cu[0] != 0) return fail(DFA_ERR_INVALID_ARG, "cu_seqlens[0] must be 0"), false;
    int64_t P = 0, items = 0;
    int umax = 0;
    for (int s = 0; s < n; ++s) {
        const int64_t len = (int64_t)cu[s + 1] - cu[s];
        if (len < 0) return fail(DFA_ERR_INVALID_ARG, "cu_seqlens decreases at %d", s + 1), false;
        P += (len + 127) / 128 * 128;
        const int u = (int)((len + unit_rows - 1) / unit_rows);
        umax = std::max(umax, u);
        items += (int64_t)u * heads;
    }
    if (P > INT32_MAX / 2 || items > INT32_MAX / 2 || (int64_t)n * heads * std::max(umax, 1) > INT32_MAX)
        return fail(DFA_ERR_INVALID_ARG, "packed batch too large"), false;
    L->T = cu[n];
    L->P = P;
    L->units_max = umax;
    L->items = items;
    return true;
}

bool varlen_layout(const int32_t* cu, int n, int H, int Hkv, int D, bool bwd, VarlenLayout* L) {
    if (!varlen_sizes(cu, n, bwd ? kBwdUnitRows : kFwdUnitRows, bwd ? Hkv : H, L)) return false;
    size_t off = 0;
    if (bwd) {
        L->delta = off;
        off = align_up(off + sizeof(float) * (size_t)H * L->P);
        L->nlse2 = off;
        off = align_up(off + sizeof(float) * (size_t)H * L->P);
        L->dq = off;
        off = align_up(off + sizeof(float) * (size_t)H * L->P * D);
    }
    // The sequence table and the work list are one contiguous int32 block (one copy).
    L->seq = off;
    L->wl = off + sizeof(int32_t) * 2 * ((size_t)n + 1);
    off = align_up(L->wl + sizeof(int32_t) * (kMaxWorkers + 1 + (size_t)L->items));
    L->total = off;
    return true;
}

// Builds [token starts | padded starts | offsets | items] in a staging buffer
// and copies it to the workspace on `s`; *workers receives the worker count.
dfa_status upload_varlen(const int32_t* cu, int n, int unit_rows, int heads, int causal, const VarlenLayout& L,
                         char* ws, cudaStream_t s, int* workers_out) {
    const int dev = current_device();
    if (dev < 0) return fail(DFA_ERR_CUDA, "no current device");
    const int workers = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), L.items));
    const size_t head = 2 * ((size_t)n + 1), count = head + workers + 1 + (size_t)L.items;
    std::vector<int32_t> units(n);
    for (int q = 0; q < n; ++q) units[q] = (cu[q + 1] - cu[q] + unit_rows - 1) / unit_rows;
    std::lock_guard<std::mutex> lk(g_stage_mu);
    Stage& st = g_stage[dev][g_stage_next[dev]++ % kStages];
    if (st.pending) {
        if (cudaEventSynchronize(st.ev) != cudaSuccess) return fail(DFA_ERR_CUDA, "staging event");
        st.pending = false;
    }
    if (!st.ev && cudaEventCreateWithFlags(&st.ev, cudaEventDisableTiming) != cudaSuccess)
        return fail(DFA_ERR_CUDA, "staging event");
    if (st.cap < count) {
        if (st.host) cudaFreeHost(st.host);
        st.host = nullptr;
        st.cap = 0;
        const size_t cap = std::max<size_t>(count, 4096);
        if (cudaHostAlloc((void**)&st.host, cap * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess)
            return fail(DFA_ERR_CUDA, "pinned staging buffer of %zu bytes", cap * sizeof(int32_t));
        st.cap = cap;
    }
    int32_t* h = st.host;
    int32_t pad = 0;
    for (int q = 0; q <= n; ++q) {
        h[q] = cu[q];
        h[n + 1 + q] = pad;
        if (q < n) pad += (cu[q + 1] - cu[q] + 127) / 128 * 128;
    }
    if (dfa_build_varlen_worklist(n, units.data(), heads, std::max(L.units_max, 1), causal, workers, h + head,
                                  h + head + workers + 1) < 0)
        return fail(DFA_ERR_INVALID_ARG, "could not build the packed-batch work list");
    cudaError_t e = cudaMemcpyAsync(ws + L.seq, h, count * sizeof(int32_t), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "packed-batch upload: %s", cudaGetErrorString(e));
    if (cudaEventRecord(st.ev, s) != cudaSuccess) return fail(DFA_ERR_CUDA, "staging event record");
    st.pending = true;
    *workers_out = workers;
    return DFA_OK;
}

AttnProblem varlen_problem(int n, int H, int Hkv, int64_t T, int D, int causal, float scale, const int32_t* seq) {
    AttnProblem p{};
    p.B = n; p.H = H; p.Hkv = Hkv; p.Lq = (int)T; p.Lkv = (int)T; p.D = D;
    p.q_sb = T * H * D; p.q_ss = (int64_t)H * D; p.q_sh = D;
    p.kv_sb = T * Hkv * D; p.kv_ss = (int64_t)Hkv * D; p.kv_sh = D;
    p.causal = causal != 0;
    p.scale = scale;
    p.seq = seq;
    return p;
}

dfa_status varlen_common(dfa_dtype dt, const int32_t* cu, int n, int H, int Hkv, int D, float scale, bool bwd,
                         void* workspace, size_t ws_bytes, VarlenLayout* L) {
    dfa_status st;
    if ((st = check_dtype(dt)) || (st = check_common(1, H, Hkv, D, scale))) return st;
    if (dt != DFA_BF16) return fail(DFA_ERR_UNSUPPORTED, "packed batches run on the bf16 tensor-core path only");
    if (!varlen_layout(cu, n, H, Hkv, D, bwd, L)) return DFA_ERR_INVALID_ARG;
    if (L->T == 0) return DFA_OK;
    if (!workspace || ws_bytes < L->total)
        return fail(DFA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L->total, ws_bytes);
    if (!aligned16(workspace)) return fail(DFA_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    return DFA_OK;
}

}  // namespace

extern "C" size_t dfa_attn_varlen_workspace_size(const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D,
                                                int bwd) {
    if (H <= 0 || H_kv <= 0 || H % H_kv != 0 || (D != 64 && D != 128)) return 0;
    VarlenLayout L;
    const std::string keep = g_msg;   // a size query does not change dfa_last_error()
    const bool ok = varlen_layout(cu_seqlens, n_seq, H, H_kv, D, bwd != 0, &L);
    snprintf(g_msg, sizeof(g_msg), "%s", keep.c_str());
    return ok ? L.total : 0;
}

extern "C" dfa_status dfa_attn_fwd_varlen(const void* q, const void* k, const void* v, dfa_dtype dt,
                                          const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D,
                                          int causal, float scale, void* O, float* lse, void* workspace,
                                          size_t ws_bytes, void* stream) {
    g_msg[0] = 0;
    VarlenLayout L;
    dfa_status st = varlen_common(dt, cu_seqlens, n_seq, H, H_kv, D, scale, false, workspace, ws_bytes, &L);
    if (st || L.T == 0) return st;
    if ((st = check_ptrs({q, k, v, O, lse}))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    int workers = 0;
    if ((st = upload_varlen(cu_seqlens, n_seq, kFwdUnitRows, H, causal, L, ws, s, &workers))) return st;
    const int32_t* seq = reinterpret_cast<const int32_t*>(ws + L.seq);
    const int32_t* wl_dev = reinterpret_cast<const int32_t*>(ws + L.wl);
    const AttnProblem p = varlen_problem(n_seq, H, H_kv, L.T, D, causal, scale, seq);
    WorkList wl{wl_dev, wl_dev + workers + 1, workers, std::max(L.units_max, 1)};
    st = tc_fwd(p, q, k, v, O, false, lse, &wl, s);
    if (st == DFA_OK) count_launch(DFA_KERNEL_FWD);
    return st;
}

extern "C" dfa_status dfa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* O,
                                          const float* lse, const void* dO, dfa_dtype dt,
                                          const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D,
                                          int causal, float scale, void* dQ, void* dK, void* dV, void* workspace,
                                          size_t ws_bytes, void* stream) {
    g_msg[0] = 0;
    VarlenLayout L;
    dfa_status st = varlen_common(dt, cu_seqlens, n_seq, H, H_kv, D, scale, true, workspace, ws_bytes, &L);
    if (st || L.T == 0) return st;
    if ((st = check_ptrs({q, k, v, O, lse, dO, dQ, dK, dV}))) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    int workers = 0;
    if ((st = upload_varlen(cu_seqlens, n_seq, kBwdUnitRows, H_kv, causal, L, ws, s, &workers))) return st;
    const int32_t* seq = reinterpret_cast<const int32_t*>(ws + L.seq);
    const int32_t* wl_dev = reinterpret_cast<const int32_t*>(ws + L.wl);
    float* delta = reinterpret_cast<float*>(ws + L.delta);
    float* nlse2 = reinterpret_cast<float*>(ws + L.nlse2);
    float* dq_acc = reinterpret_cast<float*>(ws + L.dq);
    if ((st = launch_bwd_prep_varlen(n_seq, H, L.T, L.P, D, seq, O, dO, lse, nlse2, delta, s))) return st;
    count_launch(DFA_KERNEL_DELTA);
    cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)H * L.P * D, s);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "dQ accumulator clear: %s", cudaGetErrorString(e));
    const AttnProblem p = varlen_problem(n_seq, H, H_kv, L.T, D, causal, scale, seq);
    WorkList wl{wl_dev, wl_dev + workers + 1, workers, std::max(L.units_max, 1)};
    if ((st = tc_bwd(p, q, k, v, dO, nlse2, delta, (int)L.P, dq_acc, dK, dV, &wl, s))) return st;
    count_launch(DFA_KERNEL_BWD);
    st = launch_convert_varlen(n_seq, H, L.T, L.P, D, scale, seq, dq_acc, dQ, s);
    if (st == DFA_OK) count_launch(DFA_KERNEL_CONVERT);
    return st;
}

extern "C" void dfa_shutdown(void) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto& kv : g_lists) cudaFreeHost(kv.second.host);
        for (auto& kv : g_split_lists) cudaFreeHost(kv.second.host);
        for (auto& kv : g_bwd_split_lists) cudaFreeHost(kv.second.host);
        g_lists.clear();
        g_split_lists.clear();
        g_bwd_split_lists.clear();
    }
    std::lock_guard<std::mutex> lk(g_stage_mu);
    for (auto& dev : g_stage)
        for (Stage& st : dev) {
            if (st.pending) cudaEventSynchronize(st.ev);
            if (st.host) cudaFreeHost(st.host);
            if (st.ev) cudaEventDestroy(st.ev);
            st = Stage{};
        }
}

extern "C" dfa_status dfa_check_errors(void* stream) {
    g_msg[0] = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
    int* flag = device_error_flag();
    if (!flag) return fail(DFA_ERR_CUDA, "device error flag unavailable");
    int v = 0;
    e = cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(DFA_ERR_CUDA, "reading the error flag: %s", cudaGetErrorString(e));
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
        return fail(DFA_ERR_TIMEOUT, "a kernel gave up on a bounded wait (code %d)", v);
    }
    return DFA_OK;
}
