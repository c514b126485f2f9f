// internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/dfa.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/dfa.h"

namespace dfa {

// Problem description handed from the C ABI to the kernel launchers.
// Element strides are for the (batch, seq, head) dimensions; D is contiguous.
struct AttnProblem {
    int B, H, Hkv, Lq, Lkv, D;
    int64_t q_sb, q_ss, q_sh;     // Q (and dO when used) strides
    int64_t kv_sb, kv_ss, kv_sh;  // K and V strides
    int64_t q_offset, kv_offset;  // global token positions of row 0
    int causal;
    float scale;
    int acc_out;                  // backward outputs are fp32 accumulators (+=)
    int64_t win_c;                // local window (causal only): chunk length in tokens ...
    int win_w;                    // ... and chunks per window; key kp is visible from query qp iff
                                  // kp <= qp and kp / win_c >= qp / win_c - (win_w - 1).  0: none
    // Variable-length batch (device, int32): seq[0..B] are the first tokens of
    // the B sequences in the packed [1, Lq, heads, D] tensors (Lq = Lkv = T
    // tokens), seq[B+1..2B+1] their first rows in the 128-row-padded per-head
    // arrays of the backward (nlse2, Delta, fp32 dQ accumulator).  nullptr: dense.
    const int32_t* seq = nullptr;
};

// Device error flag (set by bounded waits that gave up).  Returns the device
// address for the current device, or nullptr on failure.
int* device_error_flag();

// Records a message for dfa_last_error() and returns `st`.
dfa_status fail(dfa_status st, const char* fmt, ...);

// ---- fp32 CUDA-core kernels (simt_attn.cu) ----
// Forward: O (dense [B,Lq,H,D], float or the input type) and lse (fp32 [B,H,Lq]).
dfa_status simt_fwd(const AttnProblem& p, dfa_dtype dt, const void* q, const void* k,
                    const void* v, void* O, bool O_is_f32, float* lse, cudaStream_t s);
// Backward pieces: dQ (dense, dtype dt), dK/dV (dense, dtype dt).  Needs Delta.
// With p.acc_out set, dQ/dK/dV are fp32 and the results are added to them.
dfa_status simt_bwd(const AttnProblem& p, dfa_dtype dt, const void* q, const void* k,
                    const void* v, const void* dO, const float* lse, const float* delta,
                    void* dQ, void* dK, void* dV, cudaStream_t s);

// ---- small HBM-bound kernels (aux_kernels.cu) ----
dfa_status launch_merge(int B, int H, int L, int D, const float* Oa, const float* la,
                        const float* Ob, const float* lb, float* O, float* l, cudaStream_t s);
// Merge of the split-kv pieces of a whole-sequence forward: row i of query
// block u = i / 256 has pieces s < ceil(hi(u) / piece_tiles) (hi as in
// dfa_build_split_worklist) in O_part [n_split][B, S, H, D] fp32 and
// lse_part [n_split][B, H, S]; writes O [B, S, H, D] in dt and lse [B, H, S].
dfa_status launch_merge_pieces(dfa_dtype dt, int B, int H, int S, int D, int causal, int piece_tiles,
                               int n_split, const float* O_part, const float* lse_part, void* O, float* lse,
                               cudaStream_t s);
// Delta[b,h,i] = sum_d dO[b,i,h,d] * O[b,i,h,d]   (dense BSHD, fp32 out [B,H,S]).
dfa_status launch_delta(dfa_dtype dt, int B, int H, int S, int D, const void* O,
                        const void* dO, float* delta, cudaStream_t s);
// Backward preprocessing for the tensor-core path: nlse2 = -lse * log2(e) (negated so
// that a score's base-2 exponent is one fused multiply-add, s c2 + nlse2) and
// Delta = rowsum(dO * O), both written to [B, H, S_pad] with zero padding.
dfa_status launch_bwd_prep(dfa_dtype dt, int B, int H, int S, int S_pad, int D, const void* O,
                           const void* dO, const float* lse, float* nlse2, float* delta, cudaStream_t s);
// Packed batch of n_seq sequences, T tokens, bf16 (seq as in AttnProblem::seq,
// P = padded rows per head): nlse2 and Delta [H, P] (zero past each sequence's
// end) from O, dO [T, H, D] and lse [H, T]; and dQ [T, H, D] = scale * acc [H, P, D].
dfa_status launch_bwd_prep_varlen(int n_seq, int H, int64_t T, int64_t P, int D, const int32_t* seq,
                                  const void* O, const void* dO, const float* lse, float* nlse2, float* delta,
                                  cudaStream_t s);
dfa_status launch_convert_varlen(int n_seq, int H, int64_t T, int64_t P, int D, float scale, const int32_t* seq,
                                 const float* acc, void* out, cudaStream_t s);
// out[i] = bf16(in[i]) for n elements (n a multiple of 8; 16-byte aligned).
dfa_status launch_cast_bf16(int64_t n, const float* in, void* out, cudaStream_t s);
dfa_status launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s);
// out[b, s, h, :] = scale * acc[b, h, s, :] cast to dt (acc is the head-major
// fp32 dQ accumulator of the tensor-core backward; D a multiple of 8).
// With accumulate, out is fp32 and the scaled values are added to it.
dfa_status launch_convert(dfa_dtype dt, int B, int H, int S, int D, float scale, const float* acc, void* out,
                          bool accumulate, cudaStream_t s);

// ---- tcgen05 tensor-core kernels (fwd_tc.cu, bwd_tc.cu) ----
struct WorkList {
    const int32_t* offsets;  // [n_workers + 1], device
    const int32_t* items;    // [n_items], device: row * n_units + unit
    int n_workers;
    int n_units;
    // Split-kv items (dfa_build_split_worklist for the forward,
    // dfa_build_bwd_split_worklist for the backward): values are
    // (row * n_units + unit) * n_split + piece; 1 / 0 without pieces.
    int n_split = 1;
    int piece_tiles = 0;
};
// With split-kv items (wl->n_split > 1) O must be fp32: piece s of every row
// goes to O + s * B*Lq*H*D and lse + s * B*H*Lq.
dfa_status tc_fwd(const AttnProblem& p, const void* q, const void* k, const void* v, void* O,
                  bool O_is_f32, float* lse, const WorkList* wl, cudaStream_t s);
// nlse2 = -lse * log2(e) and delta are [B, H, S_pad] (S_pad = S rounded up to 128,
// zero in the padding); dq_acc is fp32 [B, S, H, D] and must be zero.
dfa_status tc_bwd(const AttnProblem& p, const void* q, const void* k, const void* v,
                  const void* dO, const float* nlse2, const float* delta, int S_pad, float* dq_acc,
                  void* dK, void* dV, const WorkList* wl, cudaStream_t s);

// Head-dim-128 backward with the softmax-gradient split into two phases so the
// tensor cores overlap it (bwd_pipe_tc.cu).
// Problems with Lq != Lkv and offsets (kv_offset - q_offset a multiple of 128)
// are the chunk-pair backward; acc_f32 makes dK/dV fp32 accumulators (+=).
dfa_status tc_bwd_pipelined(const AttnProblem& p, const void* q, const void* k, const void* v,
                            const void* dO, const float* nlse2, const float* delta, int S_pad,
                            float* dq_acc, void* dK, void* dV, bool acc_f32, const WorkList* wl,
                            cudaStream_t s);

int num_sms();

// A sequence of S tokens cut into n_chunks chunks (DISTFLASHATTN §3.1: one
// chunk per worker): every chunk but the last holds ceil(S / n_chunks)
// tokens and the last one the rest, which must be at least one token.  An
// empty sequence splits into any positive number of chunks.
inline int64_t chunk_tokens(int64_t S, int n_chunks) { return (S + n_chunks - 1) / n_chunks; }
inline bool chunks_valid(int64_t S, int n_chunks) {
    return n_chunks > 0 && (S == 0 || (int64_t)(n_chunks - 1) * chunk_tokens(S, n_chunks) < S);
}

// 4-D bf16 TMA descriptor over a [B, L, heads, D] tensor (element strides sb,
// ss, sh; D contiguous), box {64, 1, 128, 1}, 128-byte swizzle.  The map is
// written into `map` (a CUtensorMap, 128 bytes, 64-byte aligned).
bool make_tmap_bshd(void* map, const void* base, int B, int L, int heads, int D, int64_t sb,
                    int64_t ss, int64_t sh);

// Per-CTA trace buffer set by dfa_debug_cta_trace (nullptr when off).
uint64_t* cta_trace(int* capacity);

// Host-side launch counters behind dfa_launch_count().
void count_launch(dfa_kernel_kind kind, int n = 1);

}  // namespace dfa
