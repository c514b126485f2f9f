/*
 * dfa.h -- C ABI of the GB300 (sm_103a) causal chunk-attention library.
 *
 * The operation is the hot path of DISTFLASHATTN ("DISTFLASHATTN: Distributed
 * Memory-efficient Attention for Long-context LLMs Training", paperlayer.ai
 * summary of arXiv 2310.03294): exact causal softmax attention over a
 * sequence split into P token chunks.  Each query chunk attends to the
 * key/value chunks at or before it (§3.2), each chunk step returns a partial
 * output with its log-sum-exp (App. D), partials combine with the
 * online-softmax rescale-and-merge rule (§3.2), and the backward reuses the
 * saved output and log-sum-exp so the forward is never recomputed (§3.3).
 *
 * Mathematical definition (natural-log lse, scale applied to the scores):
 *   s_ij = scale * <q_i, k_j>, visible iff !causal or kv_pos(j) <= q_pos(i)
 *   lse_i = ln sum_j exp(s_ij),  O_i = sum_j exp(s_ij - lse_i) v_j
 * A row with no visible key has O_i = 0 and lse_i = -inf.  Grouped-query
 * attention: query head h reads key/value head h / (H / H_kv).
 *
 * Conventions shared by every entry point
 *  - Layouts: Q, O, dO, dQ are [B, S, H, D]; K, V, dK, dV are [B, S, H_kv, D]
 *    (BSHD, D contiguous); lse and Delta are fp32 [B, H, S] contiguous.
 *  - Every pointer is a DEVICE pointer owned by the caller; the library never
 *    allocates device memory.  `stream` is a cudaStream_t (NULL = legacy default).
 *  - Calls are asynchronous on `stream`: DFA_OK means "validated and launched".
 *    A kernel that gives up on a bounded wait sets a device error flag that
 *    dfa_check_errors() reports as DFA_ERR_TIMEOUT.
 *  - No exception crosses this boundary.  On a non-OK status nothing was
 *    launched and dfa_last_error() holds a message (thread-local).
 *  - dtype: DFA_BF16 runs the tcgen05 tensor-core kernels (fp32 accumulation);
 *    DFA_F32 runs fp32 CUDA-core kernels (fp32 I/O needs more than one-pass
 *    tf32 accuracy).  O, dO, dQ, dK and dV share the input dtype.
 *  - Supported head dims: D in {64, 128}.  Pointers must be 16-byte aligned.
 */
#ifndef DFA_H
#define DFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DFA_OK = 0,
    DFA_ERR_INVALID_ARG = 1,   /* bad pointer, size, stride, alignment or scale   */
    DFA_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement   */
    DFA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed            */
    DFA_ERR_TIMEOUT = 4,       /* a kernel gave up on a bounded wait              */
    DFA_ERR_WORKSPACE = 5      /* workspace missing or smaller than required      */
} dfa_status;

typedef enum { DFA_F32 = 0, DFA_BF16 = 1 } dfa_dtype;

/* Work distribution over persistent CTAs (DISTFLASHATTN §3.2 and App. B).
 * UNBALANCED: the pages' baseline -- the sequence is cut into one contiguous
 *   token range per worker (CTA) and each worker computes its causal prefix,
 *   so late workers carry most of the triangle.
 * BALANCED: the token-level balanced schedule -- a worker that takes an
 *   early (cheap) query tile also takes its mirror image at the end of the
 *   sequence, and these equal-cost pairs are dealt to the workers in turn,
 *   so every worker gets the same amount of work to within one pair.
 * SPLIT_KV: BALANCED plus helper items (§3.2: idle workers compute part of a
 *   busy worker's attention and hand back a partial output with its
 *   log-sum-exp, which the owner merges).  When a bf16 whole-sequence forward
 *   has fewer 256-row query blocks than the GPU has SMs, every block's
 *   key/value range is cut into pieces of dfa_split_piece_tiles() 128-key
 *   tiles; each piece is an item of its own whose fp32 partial (O, lse) goes
 *   to the workspace, and a merge kernel combines each row's pieces with the
 *   rescale-and-merge rule.  In a bf16 head-dim-128 backward whose mirror
 *   pairs of key tiles number at most 3/4 of the SMs, every key tile's
 *   query range is cut into pieces of dfa_split_bwd_piece_tiles() query
 *   tiles (§3.3: a helper computes part of a worker's gradients), and each
 *   piece adds its partial dK, dV to fp32 accumulators in the workspace
 *   (vector reductions), cast to bf16 at the end.  Larger problems, the
 *   local window, fp32 I/O, head dim 64 (backward) and the no-alloc forward
 *   treat it as BALANCED. */
typedef enum { DFA_SCHED_BALANCED = 0, DFA_SCHED_UNBALANCED = 1, DFA_SCHED_SPLIT_KV = 2 } dfa_sched;

/* One chunk step (DISTFLASHATTN App. D: a worker's step advances its attention
 * state and hands back the output with its log-sum-exp): a query chunk of Lq rows at global
 * position q_offset against a key/value chunk of Lkv rows at kv_offset.
 *   q:        [B, Lq, H, D] with element strides q_strides = {batch, seq, head}
 *   k, v:     [B, Lkv, H_kv, D] with element strides kv_strides (shared by k, v)
 *             (either stride array may be NULL for the dense layout; strides
 *             must be multiples of 8 elements so rows stay 16-byte aligned)
 *   causal:   1 = mask kv_offset + j > q_offset + i; 0 = attend to the whole chunk
 *   O_partial: fp32 [B, Lq, H, D] dense, the normalised partial output
 *   lse:      fp32 [B, H, Lq] dense, natural-log log-sum-exp of the partial
 * Rows that see no key of this chunk get O_partial = 0 and lse = -inf. */
dfa_status dfa_chunk_attn_fwd(const void* q, const void* k, const void* v, dfa_dtype dt,
                              int B, int H, int H_kv, int Lq, int Lkv, int D,
                              const int64_t* q_strides, const int64_t* kv_strides,
                              int64_t q_offset, int64_t kv_offset, int causal, float scale,
                              float* O_partial, float* lse, void* stream);

/* Online-softmax rescale-and-merge of two partials over the same rows
 * (DISTFLASHATTN §3.2: helpers return partial outputs plus softmax statistics
 * that the owner rescales):
 *   lse = ln(e^lse_a + e^lse_b),  O = e^(lse_a - lse) O_a + e^(lse_b - lse) O_b.
 * A partial with lse = -inf has weight 0; both -inf gives O = 0, lse = -inf.
 *   O_a, O_b, O_out: fp32 [B, L, H, D];  lse_a, lse_b, lse_out: fp32 [B, H, L].
 * O_out may alias O_a or O_b, lse_out may alias lse_a or lse_b. */
dfa_status dfa_merge_partials(int B, int H, int L, int D,
                              const float* O_a, const float* lse_a,
                              const float* O_b, const float* lse_b,
                              float* O_out, float* lse_out, void* stream);

/* Backward step for one (query chunk, key chunk) pair -- the per-worker
 * backward of DISTFLASHATTN §3.3: the owner's saved output O and log-sum-exp
 * of its query rows (global, over the whole key sequence, as returned by the
 * forward and its merges) are reused, never recomputed.  With
 *   P_ij = exp(scale <q_i, k_j> - lse_i),  Delta_i = <dO_i, O_i>,
 *   dS_ij = P_ij (<dO_i, v_j> - Delta_i)   for the pair's visible (i, j)
 * it ADDS this pair's share to three fp32 accumulators:
 *   dQ_acc[i] += scale sum_j dS_ij k_j,  dK_acc[j] += scale sum_i dS_ij q_i,
 *   dV_acc[j] += sum_i P_ij dO_i
 * so that summing the pairs over all key chunks (dQ) and all query chunks
 * (dK, dV) gives the full gradients.
 *   q, O, dO: [B, Lq, H, D] dense in dt;  k, v: [B, Lkv, H_kv, D] dense in dt
 *   lse:      fp32 [B, H, Lq], natural log (the rows' final lse)
 *   causal:   1 = pairs with kv_offset + j > q_offset + i are skipped
 *   dQ_acc:   fp32 [B, Lq, H, D];  dK_acc, dV_acc: fp32 [B, Lkv, H_kv, D];
 *             all caller-owned, updated in place (+=), never cleared
 *   workspace: >= dfa_chunk_bwd_workspace_size(...) bytes, 256-byte aligned,
 *             caller-owned scratch (contents not preserved)
 * bf16 with D = 128 and kv_offset - q_offset a multiple of 128 runs on the
 * tensor cores; other cases on the CUDA-core kernels.  Errors: INVALID_ARG
 * for bad sizes, offsets, pointers or workspace; nothing is launched then.
 * Calls on one stream may share accumulators; concurrent calls must not. */
dfa_status dfa_chunk_attn_bwd(const void* q, const void* k, const void* v, const void* O,
                              const float* lse, const void* dO, dfa_dtype dt,
                              int B, int H, int H_kv, int Lq, int Lkv, int D,
                              int64_t q_offset, int64_t kv_offset, int causal, float scale,
                              float* dQ_acc, float* dK_acc, float* dV_acc,
                              void* workspace, size_t ws_bytes, void* stream);

/* Bytes of workspace dfa_chunk_attn_bwd needs (0 for invalid sizes). */
size_t dfa_chunk_bwd_workspace_size(int B, int H, int H_kv, int Lq, int Lkv, int D);

/* Bytes of workspace dfa_attn_fwd (bwd = 0) or dfa_attn_bwd (bwd = 1) needs,
 * for every schedule: on a problem small enough for SPLIT_KV it includes the
 * pieces' fp32 partials (forward) or dK/dV accumulators (backward), sized
 * for the current device's SM count.  Returns 0 for invalid sizes, including
 * an n_chunks that leaves the last chunk empty. */
size_t dfa_attn_workspace_size(int B, int H, int H_kv, int S, int D, int n_chunks, int bwd);

/* Whole-sequence causal forward over n_chunks token chunks (DISTFLASHATTN §3.1,
 * §3.2).  Chunk partials of one query tile are merged on chip with the
 * rescale-and-merge rule as the key/value chunks stream by, so the result
 * equals the monolithic softmax up to rounding.
 *   q: [B, S, H, D], k, v: [B, S, H_kv, D] dense;  O: [B, S, H, D] in dt;
 *   lse: fp32 [B, H, S] (saved for the backward).
 * Chunks: the first n_chunks - 1 hold C = ceil(S / n_chunks) tokens and the
 * last one the rest (a ragged last chunk), which must hold at least one
 * token, else INVALID_ARG (e.g. S = 9, n_chunks = 4).  n_chunks changes only
 * the decomposition, never the result. */
dfa_status dfa_attn_fwd(const void* q, const void* k, const void* v, dfa_dtype dt,
                        int B, int H, int H_kv, int S, int D, int n_chunks, int causal,
                        float scale, dfa_sched sched, void* O, float* lse,
                        void* workspace, size_t ws_bytes, void* stream);

/* Backward from the SAVED O and lse (DISTFLASHATTN §3.3, rematerialization-aware
 * checkpointing: the forward is computed once and never re-run here):
 *   Delta_i = <dO_i, O_i>,  P_ij = exp(s_ij - lse_i),  dS_ij = P_ij (dO_i.v_j - Delta_i)
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO  (dK, dV summed over a GQA group).
 * Same layouts as dfa_attn_fwd; dQ/dK/dV are written (not accumulated) in dt.
 * The workspace holds the fp32 dQ accumulator and Delta.
 * Reproducibility: O and lse of the forward, and dK, dV of the backward
 * under BALANCED and UNBALANCED, are the same bits on every call (one CTA
 * owns each output row).  dQ adds fp32 partials with atomics in no fixed
 * order, so it may differ in the last bits from call to call; so may dK and
 * dV when SPLIT_KV cuts the backward into pieces. */
dfa_status dfa_attn_bwd(const void* q, const void* k, const void* v, const void* O,
                        const float* lse, const void* dO, dfa_dtype dt,
                        int B, int H, int H_kv, int S, int D, int n_chunks, int causal,
                        float scale, dfa_sched sched, void* dQ, void* dK, void* dV,
                        void* workspace, size_t ws_bytes, void* stream);

/* Local sliding window (DISTFLASHATTN App. F: with a local window each worker
 * attends only to its own chunk and the neighbouring chunks before it, and
 * fetches only those key/value blocks).  Causal attention in which a query at
 * position qp sees key kp only if kp <= qp and kp / C >= qp / C - (window - 1),
 * C = ceil(S / n_chunks) the chunk length (the last chunk may be shorter);
 * window >= n_chunks is plain causal.
 * Arguments, layouts, workspace and errors as dfa_attn_fwd / dfa_attn_bwd
 * (causal implied); INVALID_ARG for window < 1.  Key/value tiles entirely
 * outside a query tile's window are not loaded or computed. */
dfa_status dfa_attn_fwd_local(const void* q, const void* k, const void* v, dfa_dtype dt,
                              int B, int H, int H_kv, int S, int D, int n_chunks, int window,
                              float scale, dfa_sched sched, void* O, float* lse,
                              void* workspace, size_t ws_bytes, void* stream);
dfa_status dfa_attn_bwd_local(const void* q, const void* k, const void* v, const void* O,
                              const float* lse, const void* dO, dfa_dtype dt,
                              int B, int H, int H_kv, int S, int D, int n_chunks, int window,
                              float scale, dfa_sched sched, void* dQ, void* dK, void* dV,
                              void* workspace, size_t ws_bytes, void* stream);

/* Variable-length batch: n_seq sequences of different lengths packed along
 * the token axis.  The pages (DISTFLASHATTN §3.1-§3.3) define the method for
 * one sequence per batch entry; a packed batch applies that definition to
 * every sequence on its own, so no token attends across a sequence boundary
 * (causal inside each sequence when causal = 1).  One launch covers all
 * sequences: the work list holds (sequence, head, block) items dealt to the
 * persistent CTAs, each sequence's causal blocks paired as in BALANCED.
 *   cu_seqlens: HOST array of n_seq + 1 int32, cu_seqlens[0] = 0, never
 *               decreasing; sequence s holds tokens [cu[s], cu[s+1]) and
 *               T = cu[n_seq] is the packed length (empty sequences allowed)
 *   q, O, dO, dQ: [T, H, D] dense;  k, v, dK, dV: [T, H_kv, D] dense
 *   lse:        fp32 [H, T] (natural log), saved by the forward for the backward
 *   workspace:  >= dfa_attn_varlen_workspace_size(...) bytes, 16-byte aligned
 * bf16 only (DFA_ERR_UNSUPPORTED for fp32), D in {64, 128}.  The work list
 * and the sequence table are copied from a small ring of pinned host buffers,
 * so these calls cannot be captured in a CUDA graph.  Backward as
 * dfa_attn_bwd: from the saved O and lse, never re-running the forward.
 * Errors: INVALID_ARG for bad offsets, sizes or pointers; WORKSPACE if the
 * workspace is too small; nothing is launched then. */
size_t dfa_attn_varlen_workspace_size(const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D, int bwd);
dfa_status dfa_attn_fwd_varlen(const void* q, const void* k, const void* v, dfa_dtype dt,
                               const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D, int causal,
                               float scale, void* O, float* lse, void* workspace, size_t ws_bytes,
                               void* stream);
dfa_status dfa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* O,
                               const float* lse, const void* dO, dfa_dtype dt,
                               const int32_t* cu_seqlens, int n_seq, int H, int H_kv, int D, int causal,
                               float scale, void* dQ, void* dK, void* dV, void* workspace,
                               size_t ws_bytes, void* stream);

/* dfa_attn_fwd for callers that cannot allocate device memory.  The paper
 * has no counterpart to this entry point.  Some callers cannot call
 * cudaMalloc where they run attention: a plugin whose host framework owns
 * every byte of device memory, or a service that forbids allocation once it
 * is serving.  This variant takes no workspace: the per-CTA work list lives
 * in a static device array of the library, 2^20 int32 entries (4 MiB) that
 * every GPU which loads the library holds until the process exits.  Same
 * arguments, layouts and results as dfa_attn_fwd without
 * `workspace`/`ws_bytes`; for the same schedule the outputs are bit-equal.
 *  - Limit: B*H*ceil(S/256) must not exceed 2^20 - 1025 work items; larger
 *    problems return DFA_ERR_INVALID_ARG without launching anything.
 *  - Set-up: the first bf16 call on a device looks up the array's device
 *    address, with that device current.
 *  - Not for CUDA graphs: the list is uploaded from a host array shared by
 *    all calls, so a call on a capturing stream returns DFA_ERR_INVALID_ARG
 *    and enqueues nothing (dfa_attn_fwd with a workspace can be captured).
 *  - The array is shared by all calls and keeps the last call's contents;
 *    each call rewrites what it uses.  Calls that overlap on the GPU (other
 *    streams or host threads) race on it: serialise them.
 *  - It allocates nothing: no cudaMalloc, cudaFree or other allocating call. */
dfa_status dfa_attn_fwd_noalloc(const void* q, const void* k, const void* v, dfa_dtype dt,
                                int B, int H, int H_kv, int S, int D, int n_chunks, int causal,
                                float scale, dfa_sched sched, void* O, float* lse, void* stream);

/* Releases what the library keeps between calls: the pinned host copies of
 * the work lists it has built (one per problem shape and schedule) and the
 * pinned staging buffers and events of the packed-batch calls.  Waits for the
 * last copy out of each staging buffer.  No device memory is held.  Call it
 * only when no call of this library is running on another host thread;
 * later calls rebuild what they need. */
void dfa_shutdown(void);

/* Synchronises `stream`, then reports and clears the device error flag:
 * DFA_ERR_TIMEOUT if a kernel gave up on a bounded wait, DFA_ERR_CUDA if the
 * stream holds a CUDA error, DFA_OK otherwise. */
dfa_status dfa_check_errors(void* stream);

/* Copy `bytes` bytes from src to dst through the SMs: a grid-stride kernel
 * (one 512-thread block per SM, 16-byte accesses when both pointers are
 * 16-byte aligned) reads and writes the two sides directly, so a pinned host
 * buffer is read or written over the GPU's coherent host link without the
 * DMA copy engines.  Not part of the pages' method: a staging helper for
 * callers that stream batches between host and device (the benchmark's
 * end-to-end leg uses it).  On a GB300 it moves 211 GB/s host to device and
 * 193 GB/s back, the same as the copy engines.  Right after heavy
 * multi-threaded CPU work on the host it kept 210 and 175 GB/s where the copy
 * engines fell to 114 GB/s in (one box) or 67 GB/s out (another).
 *   dst, src: device, managed or pinned (page-locked) host memory; must not
 *             overlap
 *   bytes:    any size
 * Asynchronous on stream (an ordinary kernel launch: it occupies SMs while it
 * runs).  Errors: INVALID_ARG for a null pointer (bytes > 0), overlapping
 * ranges, or a pointer that is pageable host memory or unknown to CUDA;
 * nothing is launched then. */
dfa_status dfa_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* dfa_last_error(void);

/* Kernel launches issued by this process, per kind (host-side counters,
 * incremented when a launch is enqueued).  Lets callers verify, for example,
 * that dfa_attn_bwd never launches a forward kernel. */
typedef enum {
    DFA_KERNEL_FWD = 0,       /* attention forward (tensor-core or fp32)   */
    DFA_KERNEL_BWD = 1,       /* attention backward main kernel(s)         */
    DFA_KERNEL_MERGE = 2,     /* partial rescale-and-merge                 */
    DFA_KERNEL_DELTA = 3,     /* Delta = rowsum(dO * O) preprocessing      */
    DFA_KERNEL_CONVERT = 4,   /* fp32 dQ accumulator -> output dtype       */
    DFA_KERNEL_COPY = 5,      /* dfa_copy                                  */
    DFA_KERNEL_KINDS = 6
} dfa_kernel_kind;
int64_t dfa_launch_count(dfa_kernel_kind kind);

/* ---- host-only scheduling helpers (no GPU needed; used by the tests) ---- */

/* Builds the persistent-CTA work list for `n_units` units of causal work per
 * (batch, head) row of `n_rows` rows, unit u costing (u + 1) key/value tiles.
 * Writes per-worker item ranges into offsets[n_workers + 1] and the unit
 * indices into items[n_rows * n_units] as (row * n_units + u), in the order
 * each worker processes them.  Returns the makespan in tiles (the largest
 * per-worker cost) or -1 on bad arguments. */
int64_t dfa_build_worklist(int n_rows, int n_units, int n_workers, dfa_sched sched,
                           int32_t* offsets, int32_t* items);

/* Piece length, in 128-key tiles, that SPLIT_KV uses for a whole-sequence
 * forward of B*H rows of S tokens on a GPU with n_sms SMs, or 0 when the
 * problem has at least n_sms 256-row query blocks (or is too short to gain)
 * and is not split.  Pieces hold at least 4 tiles and are sized so that the
 * pieces number about twice n_sms. */
int dfa_split_piece_tiles(int B, int H, int S, int causal, int n_sms);

/* Work list of SPLIT_KV items.  Query block u of a row covers query tiles
 * [2u, 2u + 2) and sees key tiles [0, hi(u)), hi(u) = min(2u + 2, kv_tiles)
 * when causal, kv_tiles otherwise; that range is cut into pieces
 * [s * piece_tiles, (s + 1) * piece_tiles) and only non-empty pieces become
 * items, with value (row * n_units + u) * n_split + s, n_split =
 * ceil(kv_tiles / piece_tiles).  Pieces are dealt longest first, each to the
 * least-loaded worker.  offsets[n_workers + 1] as for dfa_build_worklist;
 * items needs n_rows * n_units * n_split entries at most.  Returns the
 * makespan in (query tile x key tile) units, or -1 on bad arguments. */
int64_t dfa_build_split_worklist(int n_rows, int n_units, int kv_tiles, int causal, int piece_tiles,
                                 int n_workers, int32_t* offsets, int32_t* items);

/* Split-kv for the backward (SPLIT_KV): query-tile piece length for a bf16
 * head-dim-128 backward of B * H_kv key-tile rows of S tokens on n_sms SMs,
 * or 0 when the mirror pairs of key tiles number more than 3/4 of n_sms (or
 * nothing gains).  Pieces hold at least 16 query tiles and number about
 * twice n_sms. */
int dfa_split_bwd_piece_tiles(int B, int H_kv, int S, int causal, int n_sms);

/* Work list of backward split-kv items.  Unit u of a row is key tile
 * t = kv_tiles - 1 - u, which sees query tiles [t, kv_tiles) when causal and
 * all of them otherwise; that range is cut into pieces of piece_tiles tiles
 * [t + s * piece_tiles, ...) and every non-empty piece is an item with value
 * (row * kv_tiles + u) * n_split + s, n_split = ceil(kv_tiles / piece_tiles).
 * Each piece adds its partial dK, dV (fp32) to accumulators shared with the
 * other pieces of its key tile (DISTFLASHATTN §3.3: a helper computes part of
 * a worker's gradients and hands them back).  Dealt longest first to the
 * least-loaded worker.  Returns the makespan in query tiles, or -1. */
int64_t dfa_build_bwd_split_worklist(int n_rows, int kv_tiles, int causal, int piece_tiles, int n_workers,
                                     int32_t* offsets, int32_t* items);

/* Work list of a variable-length batch: sequence s has seq_units[s] units
 * (<= n_units_max) per head, unit u costing u + 1 tiles when causal (the
 * dfa_build_worklist cost) and seq_units[s] otherwise.  Causal units of one
 * (sequence, head) are paired with their mirror (cost n_s + 1); pairs and
 * single units are dealt longest first to the least-loaded worker.  Item
 * values are (s * heads + h) * n_units_max + u; items needs
 * n_seq * heads * n_units_max entries at most.  Returns the makespan or -1. */
int64_t dfa_build_varlen_worklist(int n_seq, const int32_t* seq_units, int heads, int n_units_max,
                                  int causal, int n_workers, int32_t* offsets, int32_t* items);

/* The pages' distributed schedule at chunk-step granularity (DISTFLASHATTN
 * App. B, Figs. 5-6, and §4.5): P workers own one chunk each, a step computes
 * one (query chunk, key/value chunk) block per worker.  Writes for each step s
 * and worker w the block it computes as (qchunk * P + kvchunk), or -1 if idle,
 * into steps[s * P + w] (capacity max_steps * P).  Returns the number of
 * steps (the makespan), or -1 on bad arguments / insufficient capacity. */
int dfa_chunk_schedule(int P, dfa_sched sched, int max_steps, int32_t* steps);

#ifdef __cplusplus
}
#endif

#endif /* DFA_H */
