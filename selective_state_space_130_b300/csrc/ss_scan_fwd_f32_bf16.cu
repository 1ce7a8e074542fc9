// Scan-forward kernels for one input/output dtype pair (float in, __nv_bfloat16 out).
#include "ss_scan_fwd_kernel.cuh"

namespace ssk {
cudaError_t scan_launch_f32_bf16(const ScanParams& p, int sg, bool tma, cudaStream_t s) {
  return scan_detail::launch_io<float, __nv_bfloat16>(p, sg, tma, s);
}
}  // namespace ssk
