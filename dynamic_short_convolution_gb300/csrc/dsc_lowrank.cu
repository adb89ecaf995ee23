// dsc_lowrank.cu -- low-rank fused dynamic short convolution (placeholder
// until the tensor-core kernels land).
#include "dsc_internal.h"

namespace dsc {

dsc_status lowrank_fwd(const LowrankArgs &) { return DSC_ERR_UNSUPPORTED; }
dsc_status lowrank_bwd(const LowrankArgs &) { return DSC_ERR_UNSUPPORTED; }
size_t lowrank_bwd_workspace(int, int, int, int, int) { return 0; }

}  // namespace dsc
