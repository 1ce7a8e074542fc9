// Scan-forward host side: launch dispatch by dtype, shape queries used by the
// launch planner, and the library's own fault word. The kernel itself is in
// ss_scan_fwd_kernel.cuh.
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "ss_scan_fwd_kernel.cuh"

namespace ssk {

// Fault word used by calls that are given no workspace.
__device__ unsigned int g_fault_word = 0;

int scan_channels_per_block(int sg) {
  using scan_detail::Cfg;
  return sg == 1 ? Cfg<float, 1>::CC : Cfg<float, 2>::CC;
}
int scan_tile_len(ss_dtype in_dtype, int sg) {
  using scan_detail::Cfg;
  if (in_dtype == SS_BF16) return sg == 1 ? Cfg<__nv_bfloat16, 1>::TILE : Cfg<__nv_bfloat16, 2>::TILE;
  return sg == 1 ? Cfg<float, 1>::TILE : Cfg<float, 2>::TILE;
}
int scan_header_words() { return scan_detail::kHeaderWords; }
uint32_t scan_header_magic() { return scan_detail::kHeaderMagic; }

// The fault word's device address, resolved once per device (with that device
// current) and cached per device under a mutex: host threads that drive
// different GPUs each get their own device's address.
unsigned int* device_fault_word() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static unsigned int* cache[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fault_word) != cudaSuccess || !a) return nullptr;
    cache[dev] = static_cast<unsigned int*>(a);
  }
  return cache[dev];
}

cudaError_t launch_scan_fwd(const ScanParams& p, const ScanPlan& plan, ss_dtype in_dtype, ss_dtype out_dtype,
                            bool use_tma, cudaStream_t stream) {
  if (in_dtype == SS_BF16)
    return out_dtype == SS_BF16 ? scan_launch_bf16_bf16(p, plan.sg, use_tma, stream)
                                : scan_launch_bf16_f32(p, plan.sg, use_tma, stream);
  return out_dtype == SS_BF16 ? scan_launch_f32_bf16(p, plan.sg, use_tma, stream)
                              : scan_launch_f32_f32(p, plan.sg, use_tma, stream);
}

}  // namespace ssk
