// Scan-forward kernels for one input/output dtype pair (__nv_bfloat16 in, float out).
#include "ss_scan_fwd_kernel.cuh"

namespace ssk {
cudaError_t scan_launch_bf16_f32(const ScanParams& p, int sg, bool tma, cudaStream_t s) {
  return scan_detail::launch_io<__nv_bfloat16, float>(p, sg, tma, s);
}
}  // namespace ssk
