// scan_fwd_inst_ff.cu -- explicit instantiations of the scan forward kernels.
#include "scan_fwd_kernels.cuh"

namespace ssm {
template cudaError_t dispatch_G<float, float, false>(const FwdArgs&, int, bool, bool, cudaStream_t);
template cudaError_t dispatch_G<float, __nv_bfloat16, false>(const FwdArgs&, int, bool, bool, cudaStream_t);
}  // namespace ssm
