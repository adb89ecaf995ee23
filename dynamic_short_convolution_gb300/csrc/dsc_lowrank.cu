// dsc_lowrank.cu -- low-rank fused dynamic short convolution, backward pass
// (placeholder until the tensor-core kernel lands).
#include "dsc_internal.h"

namespace dsc {

dsc_status lowrank_bwd(const LowrankArgs &) { return DSC_ERR_UNSUPPORTED; }
size_t lowrank_bwd_workspace(int, int, int, int, int) { return 0; }

}  // namespace dsc
