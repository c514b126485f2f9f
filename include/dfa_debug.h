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

#ifdef __cplusplus
}
#endif

#endif /* DFA_DEBUG_H */
