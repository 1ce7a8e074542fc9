// Single-token selective-SSM decode step for sm_103a, state updated in place.
//
// The step is bound by the state bytes: every channel reads and writes its 16
// fp32 states (128 B) against 6-8 B of token inputs, so the kernel is a
// streaming pass over h. A quad of lanes owns one channel, four states (one
// 16-byte vector) each, so a warp-wide load or store covers 8 channels = 512
// contiguous bytes with every sector fully used. A warp takes 32 consecutive
// channels in four rounds and issues all four state loads before any
// arithmetic: 64 bytes in flight per thread. The readout C.h is reduced across
// the quad with two shuffles. The per-channel scalars (softplus, silu, the skip
// term) are computed once per channel: lane k of a quad owns the channel of
// round k, hands (delta, delta*u) and the channel's coordinates to its quad by
// shuffle, and stores that channel's y. This is the per-token state update the
// inference page describes for decode ("AI 推理系列（十四）：Mamba 的 Selective
// State Space", sections on Selective Scan for Decode and on request state:
// allocate, write after prefill, update in place).
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kStepWarps = 8;                // warps per block
constexpr int kRounds = 4;                   // 8-channel rounds per warp
constexpr int kChPerWarp = 8 * kRounds;      // channels per warp
constexpr int kStepThreads = 32 * kStepWarps;

template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                     __uint_as_float(v.y & 0xffff0000u));
}

template <typename TIn, typename TOut, bool HAS_Z>
__global__ void __launch_bounds__(kStepThreads) state_update_kernel(const __grid_constant__ StepParams p) {
  const int64_t nch = p.batch * p.dim;
  const int lane = threadIdx.x & 31;
  const int qd = lane & 3;   // which four states of the channel
  const int cl = lane >> 2;  // channel within a round
  const int64_t wbase = ((int64_t)blockIdx.x * kStepWarps + (threadIdx.x >> 5)) * kChPerWarp;

  // all state loads first
  float4 hv[kRounds];
  bool valid[kRounds];
#pragma unroll
  for (int k = 0; k < kRounds; k++) {
    const int64_t c = wbase + 8 * k + cl;
    valid[k] = c < nch;
    hv[k] = valid[k] ? __ldcs(reinterpret_cast<const float4*>(p.h + c * kDState) + qd)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // this lane's own channel (round qd of its quad): scalars computed once
  const TIn* gB = static_cast<const TIn*>(p.B);
  const TIn* gC = static_cast<const TIn*>(p.C);
  const int64_t c_own = wbase + 8 * qd + cl;
  const bool own_valid = c_own < nch;
  const int64_t co = own_valid ? c_own : 0;
  const int64_t b_own = co / p.dim;
  const int64_t d_own = co - b_own * p.dim;
  const float xu = to_f32(static_cast<const TIn*>(p.u)[co]);
  const float dl_own =
      softplus(to_f32(static_cast<const TIn*>(p.delta_raw)[co]) + (p.delta_bias ? __ldg(p.delta_bias + d_own) : 0.f));
  const float du_own = dl_own * xu;
  const float post = (p.D ? __ldg(p.D + d_own) : 0.f) * xu;
  const float gate = HAS_Z ? silu(to_f32(static_cast<const TIn*>(p.z)[co])) : 1.f;

#pragma unroll
  for (int k = 0; k < kRounds; k++) {
    const int src = (lane & ~3) | k;  // owner of this round's channel in the quad
    const float dl = __shfl_sync(0xffffffffu, dl_own, src);
    const float du = __shfl_sync(0xffffffffu, du_own, src);
    const int64_t d = __shfl_sync(0xffffffffu, (int)d_own, src);  // dim and batch are below 2^31
    const int64_t b = __shfl_sync(0xffffffffu, (int)b_own, src);
    const float4 a = __ldg(reinterpret_cast<const float4*>(p.A + d * kDState) + qd);
    const float4 bb = load4(gB + b * kDState + 4 * qd);
    const float4 cc = load4(gC + b * kDState + 4 * qd);
    float4 h = hv[k];
    h.x = fmaf(ex2(dl * (a.x * kLog2e)), h.x, du * bb.x);
    h.y = fmaf(ex2(dl * (a.y * kLog2e)), h.y, du * bb.y);
    h.z = fmaf(ex2(dl * (a.z * kLog2e)), h.z, du * bb.z);
    h.w = fmaf(ex2(dl * (a.w * kLog2e)), h.w, du * bb.w);
    float part = fmaf(cc.x, h.x, cc.y * h.y) + fmaf(cc.z, h.z, cc.w * h.w);
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    if (valid[k]) __stcs(reinterpret_cast<float4*>(p.h + (wbase + 8 * k + cl) * kDState) + qd, h);
    if (qd == k && own_valid) static_cast<TOut*>(p.y)[c_own] = from_f32<TOut>((part + post) * gate);
  }
}

template <typename TIn, typename TOut>
cudaError_t launch_io(const StepParams& p, cudaStream_t stream) {
  const int64_t nch = p.batch * p.dim;
  const int64_t per_block = (int64_t)kStepWarps * kChPerWarp;
  const int64_t blocks = (nch + per_block - 1) / per_block;
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
