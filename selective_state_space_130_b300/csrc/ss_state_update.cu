// Single-token selective-SSM decode step for sm_103a, state updated in place.
//
// The step is bound by the state bytes: every channel reads and writes its 16
// fp32 states (128 B) against 6-8 B of token inputs, so the kernel is a
// streaming pass over h. Two threads own one channel (8 states = two 16-byte
// vectors each); a warp covers 16 consecutive channels, i.e. 1 KiB of
// contiguous state, so every load and store is a full 128-byte line. The
// readout C.h is reduced across the thread pair with one shuffle. This is the
// per-token state update the inference page describes for decode ("AI 推理系列
// （十四）：Mamba 的 Selective State Space", sections on Selective Scan for
// Decode and on request state: allocate, write after prefill, update in place).
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kStepThreads = 256;

template <typename TIn, typename TOut, bool HAS_Z>
__global__ void __launch_bounds__(kStepThreads) state_update_kernel(const __grid_constant__ StepParams p) {
  const int64_t nch = p.batch * p.dim;
  const int64_t gid = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;
  const int64_t ch = gid >> 1;
  const int half = (int)(gid & 1);
  const bool valid = ch < nch;
  const int64_t cs = valid ? ch : 0;  // keep every lane in the shuffle
  const int64_t b = cs / p.dim, d = cs % p.dim;
  const int n0 = half * 8;

  float4* hp = reinterpret_cast<float4*>(p.h + cs * kDState + n0);
  float4 h0 = make_float4(0.f, 0.f, 0.f, 0.f), h1 = h0;
  if (valid) {
    h0 = __ldcs(hp);
    h1 = __ldcs(hp + 1);
  }
  const float4* ap = reinterpret_cast<const float4*>(p.A + d * kDState + n0);
  const float4 a0 = __ldg(ap), a1 = __ldg(ap + 1);

  const TIn* gu = static_cast<const TIn*>(p.u);
  const TIn* gdr = static_cast<const TIn*>(p.delta_raw);
  const float xu = to_f32(gu[cs]);
  const float dl = softplus(to_f32(gdr[cs]) + (p.delta_bias ? __ldg(p.delta_bias + d) : 0.f));
  const float du = dl * xu;

  float bb[8], cc[8];
  if constexpr (sizeof(TIn) == 2) {
    const uint4 vb = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.B) + b * kDState + n0));
    const uint4 vc = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.C) + b * kDState + n0));
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w}, wc[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
      bb[2 * k] = __uint_as_float(wb[k] << 16);
      bb[2 * k + 1] = __uint_as_float(wb[k] & 0xffff0000u);
      cc[2 * k] = __uint_as_float(wc[k] << 16);
      cc[2 * k + 1] = __uint_as_float(wc[k] & 0xffff0000u);
    }
  } else {
    const float4* fb = reinterpret_cast<const float4*>(static_cast<const float*>(p.B) + b * kDState + n0);
    const float4* fc = reinterpret_cast<const float4*>(static_cast<const float*>(p.C) + b * kDState + n0);
    const float4 b0 = __ldg(fb), b1 = __ldg(fb + 1), c0 = __ldg(fc), c1 = __ldg(fc + 1);
    bb[0] = b0.x; bb[1] = b0.y; bb[2] = b0.z; bb[3] = b0.w; bb[4] = b1.x; bb[5] = b1.y; bb[6] = b1.z; bb[7] = b1.w;
    cc[0] = c0.x; cc[1] = c0.y; cc[2] = c0.z; cc[3] = c0.w; cc[4] = c1.x; cc[5] = c1.y; cc[6] = c1.z; cc[7] = c1.w;
  }

  float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int n = 0; n < 8; n++) {
    const float abar = ex2(dl * (av[n] * kLog2e));
    hv[n] = fmaf(abar, hv[n], du * bb[n]);
    if (n & 1) acc1 = fmaf(cc[n], hv[n], acc1);
    else acc0 = fmaf(cc[n], hv[n], acc0);
  }
  float part = acc0 + acc1;
  part += __shfl_xor_sync(0xffffffffu, part, 1);

  if (valid) {
    __stcs(hp, make_float4(hv[0], hv[1], hv[2], hv[3]));
    __stcs(hp + 1, make_float4(hv[4], hv[5], hv[6], hv[7]));
    if (half == 0) {
      float yv = part + (p.D ? __ldg(p.D + d) : 0.f) * xu;
      if (HAS_Z) yv *= silu(to_f32(static_cast<const TIn*>(p.z)[cs]));
      static_cast<TOut*>(p.y)[cs] = from_f32<TOut>(yv);
    }
  }
}

template <typename TIn, typename TOut>
cudaError_t launch_io(const StepParams& p, cudaStream_t stream) {
  const int64_t threads = p.batch * p.dim * 2;
  const int64_t blocks = (threads + kStepThreads - 1) / kStepThreads;
  if (p.z) state_update_kernel<TIn, TOut, true><<<(unsigned)blocks, kStepThreads, 0, stream>>>(p);
  else state_update_kernel<TIn, TOut, false><<<(unsigned)blocks, kStepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_update(const StepParams& p, ss_dtype in_dtype, ss_dtype out_dtype, cudaStream_t stream) {
  if (in_dtype == SS_BF16)
    return out_dtype == SS_BF16 ? launch_io<__nv_bfloat16, __nv_bfloat16>(p, stream)
                                : launch_io<__nv_bfloat16, float>(p, stream);
  return out_dtype == SS_BF16 ? launch_io<float, __nv_bfloat16>(p, stream) : launch_io<float, float>(p, stream);
}

}  // namespace ssk
