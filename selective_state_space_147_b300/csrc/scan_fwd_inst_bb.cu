// scan_fwd_inst_bb.cu -- explicit instantiations of the scan forward kernels.
#include "scan_fwd_kernels.cuh"

namespace ssm {
template cudaError_t dispatch_G<__nv_bfloat16, __nv_bfloat16, true>(const FwdArgs&, int, bool, bool, cudaStream_t);
template cudaError_t dispatch_G<__nv_bfloat16, __nv_bfloat16, false>(const FwdArgs&, int, bool, bool, cudaStream_t);
}  // namespace ssm
