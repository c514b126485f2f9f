/*
 * dfa_debug.h -- bring-up hooks of the GB300 attention library.  Not part of
 * the attention API: they exercise the individual tensor-core operand forms
 * the attention kernels are built from, so a wrong descriptor shows up as a
 * wrong 128x128 product instead of a wrong attention output.
 */
#ifndef DFA_DEBUG_H
#define DFA_DEBUG_H

#include "dfa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One 128x128x128 bf16 product with fp32 accumulation on the tcgen05 tensor
 * cores, written to C (fp32 [128, 128] row-major, device).  A and B are device
 * bf16 [128, 128] row-major, 16-byte aligned.
 *   form 0: C = A  B^T   A, B loaded by TMA, both K-major       (S = Q K^T)
 *   form 1: C = A  B     A staged in tensor memory, B by TMA as
 *                        an N-major operand                    (O += P V)
 *   form 2: C = A^T B    A written to shared memory by threads
 *                        as an M-major operand, B by TMA N-major (dQ = dS K)
 *   form 3: C = A  B^T   A written to shared memory by threads
 *                        K-major, B by TMA K-major              (dK = dS^T Q ...)
 * Returns DFA_ERR_INVALID_ARG for an unknown form or bad pointers. */
dfa_status dfa_debug_mma(int form, const void* A, const void* B, float* C, void* stream);

/* Per-CTA timeline of the persistent attention kernels.  When `buf` is a
 * device buffer of 16 x `capacity` uint64, every later launch of the
 * forward or backward kernel writes, for each CTA b < capacity, a record
 *   buf[8b + 0] = SM id, [8b + 1] = start time (ns, %globaltimer),
 *   [8b + 2] = end time (ns), [8b + 3] = work items in its list,
 *   [8b + 4] = tiles its MMA thread processed, [8b + 5] = tiles its first
 *   softmax/compute thread processed, [8b + 6] = tiles its producer loaded,
 *   [8b + 7] = tiles its dQ drain warpgroup processed (backward; 0 forward),
 * and a wait profile at buf[8 capacity + 8b + slot]: SM clock cycles each
 * role spent blocked on barriers.  Backward slots: 0 P/dS warpgroup on dP^T,
 * 5 P/dS warpgroup on its tile inputs, 6 P/dS warpgroup on the dK/dV
 * accumulators, 7 dQ drain on the dQ MMA; slots 1-4 stay 0 (the MMA thread's
 * waits are not profiled: any hook in them slows the backward by 1-2%).
 * Forward: 0.
 * Pass NULL to stop tracing.  The setting is process-wide; the caller owns
 * the buffer and must keep it alive while tracing is on. */
dfa_status dfa_debug_cta_trace(uint64_t* buf, int capacity);

/* Failure detection without a GPU fault: launches one CTA of two warps that
 * wait on mbarriers nothing ever arrives on, through the same bounded wait
 * the attention kernels use (4 s).  The first warp gives up, raises the
 * CTA's abort flag and the device error flag; the second leaves on the abort
 * flag.  The kernel then returns normally, so the context stays usable, and
 * dfa_check_errors() reports DFA_ERR_TIMEOUT (and clears the flag).  If `out`
 * (device, 2 ints) is given, out[w] = 1 if warp w's wait completed, else 0. */
dfa_status dfa_debug_wait_timeout(int* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFA_DEBUG_H */
