// Temporary: routes the bf16 entry points to the CUDA-core kernels until the
// tcgen05 kernels land.
#include "internal.h"
namespace dfa {
dfa_status tc_fwd(const AttnProblem& p, const void* q, const void* k, const void* v, void* O,
                  bool O_is_f32, float* lse, const WorkList*, cudaStream_t s) {
    return simt_fwd(p, DFA_BF16, q, k, v, O, O_is_f32, lse, s);
}
dfa_status tc_bwd(const AttnProblem&, const void*, const void*, const void*, const void*,
                  const float*, const float*, float*, void*, void*, const WorkList*, cudaStream_t) {
    return fail(DFA_ERR_UNSUPPORTED, "tensor-core backward not built yet");
}
}  // namespace dfa
