// Temporary: the tensor-core backward is not built yet.
#include "internal.h"
namespace dfa {
dfa_status tc_bwd(const AttnProblem&, const void*, const void*, const void*, const void*,
                  const float*, const float*, float*, void*, void*, const WorkList*, cudaStream_t) {
    return fail(DFA_ERR_UNSUPPORTED, "tensor-core backward not built yet");
}
}  // namespace dfa
