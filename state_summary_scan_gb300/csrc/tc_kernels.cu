// tc_kernels.cu -- tensor-core (tcgen05) path; not enabled yet.
#include "internal.h"

namespace rmcp {

bool tc_supports(const Dims&, rm_dtype) { return false; }

rm_status launch_tc(Op, const Dims&, const Ptrs&, cudaStream_t) { return RM_ERR_UNSUPPORTED; }

}  // namespace rmcp
