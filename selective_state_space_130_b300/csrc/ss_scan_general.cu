// Generalised selective scan forward for sm_103a: state sizes 16 to 128, B and
// C shared within groups of channels, and the first-order or the zero-order-hold
// input matrix.
//
// Per channel d of group g = d / (dim / G), for t = 0 .. L-1:
//   delta = softplus(delta_raw + bias);  Abar_n = exp(delta A_n)
//   Bbar_n = delta B_n                  (first order)
//          = (Abar_n - 1) / A_n * B_n   (zero-order hold; delta B_n when A_n = 0)
//   h_n = Abar_n h_n + Bbar_n u;  y = (sum_n C_n h_n + D u) * silu(z)
// The state size may grow beyond 16 (mlqm.cn tutorial, section 3.1); the
// zero-order hold is the exact discretisation for an input held over the step
// ("外文文献精读：Mamba - 线性时间序列建模与结构化状态空间模型", section 1.2;
// tutorial section 3.2); groups generalise the one B and C the pages share by
// all channels.
//
// One warp owns CW = 32 / SG channels of one batch element; SG = N / 16 lanes
// share a channel, 16 fp32 states each (packed f32x2 pairs). Inputs stream
// through a two-buffer cp.async ring of 16-step sub-tiles: u, delta_raw, z rows
// of the warp's channels and the B and C rows of the groups those channels
// span (contiguous in [batch, L, G, N]). The readout is summed over the SG
// lanes of a channel by shuffle; the first lane of each channel stores y.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kGT = 16;  // timesteps per staged sub-tile

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// Copy kGT rows (rows `stride` elements apart in global memory, starting at
// element e0 of base) into shared rows of rowb bytes at dst. Rows at or past
// nrows and elements at or past nelem are zero. chunk: 16 or 4 = asynchronous
// copies of that many bytes (every piece wholly inside or outside the valid
// range, source pieces aligned), 0 = element-wise loads and stores.
template <typename T>
__device__ __forceinline__ void stage_rows(uint8_t* dst, int rowb, int chunk, const void* base, int64_t e0,
                                           int64_t stride, int nrows, int nelem, int lane) {
  constexpr int ES = (int)sizeof(T);
  if (chunk > 0) {
    const int epc = chunk / ES;
    const int cpr = rowb / chunk;
    const uint32_t d0 = smem_u32(dst);
    for (int c = lane; c < kGT * cpr; c += 32) {
      const int tt = c / cpr, k = c - tt * cpr;
      const bool ok = tt < nrows && k * epc < nelem;
      const T* src = static_cast<const T*>(base) + (ok ? e0 + tt * stride + (int64_t)k * epc : 0);
      if (chunk == 16) cp_async16(d0 + tt * rowb + k * 16, src, ok ? 16u : 0u);
      else cp_async4(d0 + tt * rowb + k * 4, src, ok ? 4u : 0u);
    }
  } else {
    const int epr = rowb / ES;
    for (int c = lane; c < kGT * epr; c += 32) {
      const int tt = c / epr, k = c - tt * epr;
      const bool ok = tt < nrows && k < nelem;
      reinterpret_cast<T*>(dst)[c] = ok ? static_cast<const T*>(base)[e0 + tt * stride + k] : from_f32<T>(0.f);
    }
  }
}

// 16 consecutive elements of a staged row (16-byte aligned) as 8 packed pairs
template <typename T>
__device__ __forceinline__ void row16_pairs(const uint8_t* p, f2 (&o)[8]) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const ulonglong2 v = reinterpret_cast<const ulonglong2*>(p)[q];
      o[2 * q] = v.x;
      o[2 * q + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[q];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; k++) o[4 * q + k] = pk(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    }
  }
}

template <typename T>
__device__ __forceinline__ float sm_elem(const uint8_t* row, int i) {
  return to_f32(reinterpret_cast<const T*>(row)[i]);
}

// e^x - 1 for a pair, given e = e^x from the MUFU exponential: below |x| =
// 1/32 the series x + x^2/2 + x^3/6 + x^4/24 (truncation under x^5/120, a
// relative 8e-9), above it e - 1 (the exponential's absolute error is then a
// relative one below 1e-5 of the result)
__device__ __forceinline__ f2 expm1_pair(f2 x, f2 e) {
  f2 p = fma2(x, pk(1.f / 24.f, 1.f / 24.f), pk(1.f / 6.f, 1.f / 6.f));
  p = fma2(x, p, pk(0.5f, 0.5f));
  p = fma2(x, p, pk(1.f, 1.f));
  const f2 ser = mul2(x, p);
  const f2 em = add2(e, pk(-1.f, -1.f));
  const float r0 = fabsf(f2lo(x)) < 0.03125f ? f2lo(ser) : f2lo(em);
  const float r1 = fabsf(f2hi(x)) < 0.03125f ? f2hi(ser) : f2hi(em);
  return pk(r0, r1);
}

template <typename TIn, typename TOut, int SG, bool ZOH>
__global__ void __launch_bounds__(32) scan_general_kernel(const __grid_constant__ GenParams p) {
  constexpr int CW = 32 / SG;        // channels per warp
  constexpr int NST = SG * 16;       // state size
  constexpr int IN_ROW = CW * (int)sizeof(TIn);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int lane = threadIdx.x;
  const int ch = lane / SG;
  const int soff = (lane % SG) * 16;
  const bool owner = (lane % SG) == 0;
  const int64_t blk = blockIdx.x;
  const int64_t b = blk / p.ncblk;
  const int64_t c0 = (blk % p.ncblk) * CW;
  const int64_t d = c0 + ch;
  const bool dv = d < p.dim;
  // lanes past the last channel stand in for the block's first channel, so
  // their group row below is the warp's first staged one (never outside it)
  const int64_t dc = dv ? d : c0;
  const int64_t L = p.seqlen, Dm = p.dim, G = p.ngroups;
  const int nch = (int)min((int64_t)CW, Dm - c0);
  // the groups this warp's channels span, and this lane's row among them
  const int64_t g_lo = c0 / p.cpg;
  const int ngw = (int)((c0 + nch - 1) / p.cpg - g_lo + 1);
  const int gi = (int)(dc / p.cpg - g_lo);
  const int bc_row = p.ngw_max * NST * (int)sizeof(TIn);  // bytes of one step's staged B (or C)
  const int off_dr = kGT * IN_ROW, off_z = 2 * kGT * IN_ROW, off_b = 3 * kGT * IN_ROW;
  const int off_c = off_b + kGT * bc_row;
  const int stage_bytes = off_c + kGT * bc_row;

  f2 A2[8], h[8];
  [[maybe_unused]] f2 An[8], invA[8], zm[8];
  {
    const int64_t arow = dc * NST + soff, hrow = (b * Dm + dc) * NST + soff;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const float a0 = dv ? __ldg(p.A + arow + 2 * j) : 0.f;
      const float a1 = dv ? __ldg(p.A + arow + 2 * j + 1) : 0.f;
      A2[j] = pk(a0 * kLog2e, a1 * kLog2e);
      h[j] = (dv && p.h0) ? pk(__ldg(p.h0 + hrow + 2 * j), __ldg(p.h0 + hrow + 2 * j + 1)) : pk(0.f, 0.f);
      if constexpr (ZOH) {
        An[j] = pk(a0, a1);
        invA[j] = pk(a0 != 0.f ? 1.f / a0 : 0.f, a1 != 0.f ? 1.f / a1 : 0.f);
        zm[j] = pk(a0 != 0.f ? 0.f : 1.f, a1 != 0.f ? 0.f : 1.f);  // A = 0: Bbar = delta B
      }
    }
  }
  const float bias_d = (dv && p.delta_bias) ? __ldg(p.delta_bias + dc) : 0.f;
  const float D_d = (dv && p.D) ? __ldg(p.D + dc) : 0.f;
  const bool has_z = p.z != nullptr;
  const int64_t nsub = (L + kGT - 1) / kGT;

  auto stage = [&](int64_t s) {
    uint8_t* buf = smem_raw + (s & 1) * stage_bytes;
    const int64_t t0 = s * kGT;
    const int nr = (int)min((int64_t)kGT, L - t0);
    const int64_t e0 = (b * L + t0) * Dm + c0;
    stage_rows<TIn>(buf, IN_ROW, p.chunk_in, p.u, e0, Dm, nr, nch, lane);
    stage_rows<TIn>(buf + off_dr, IN_ROW, p.chunk_in, p.delta_raw, e0, Dm, nr, nch, lane);
    if (has_z) stage_rows<TIn>(buf + off_z, IN_ROW, p.chunk_in, p.z, e0, Dm, nr, nch, lane);
    const int64_t eb = ((b * L + t0) * G + g_lo) * NST;
    stage_rows<TIn>(buf + off_b, bc_row, 16, p.B, eb, G * NST, nr, ngw * NST, lane);
    stage_rows<TIn>(buf + off_c, bc_row, 16, p.C, eb, G * NST, nr, ngw * NST, lane);
    cp_async_commit();
  };

  stage(0);
  for (int64_t s = 0; s < nsub; s++) {
    if (s + 1 < nsub) stage(s + 1);
    else cp_async_commit();
    cp_async_wait1();
    __syncwarp();
    const uint8_t* buf = smem_raw + (s & 1) * stage_bytes;
    const int64_t t0 = s * kGT;
    const int ns = (int)min((int64_t)kGT, L - t0);
#pragma unroll 2
    for (int tt = 0; tt < ns; tt++) {
      const float xu = sm_elem<TIn>(buf + tt * IN_ROW, ch);
      const float dl = softplus_fast(sm_elem<TIn>(buf + off_dr + tt * IN_ROW, ch) + bias_d);
      const f2 dl2 = pk(dl, dl);
      f2 Bv[8], Cv[8];
      row16_pairs<TIn>(buf + off_b + tt * bc_row + (gi * NST + soff) * (int)sizeof(TIn), Bv);
      row16_pairs<TIn>(buf + off_c + tt * bc_row + (gi * NST + soff) * (int)sizeof(TIn), Cv);
      f2 y0 = pk(0.f, 0.f), y1 = pk(0.f, 0.f);
      if constexpr (ZOH) {
        const f2 xu2 = pk(xu, xu), du2 = pk(dl * xu, dl * xu);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const f2 e2 = mul2(dl2, A2[j]);
          const f2 a = pk(ex2(f2lo(e2)), ex2(f2hi(e2)));
          const f2 em1 = expm1_pair(mul2(dl2, An[j]), a);
          // Bbar u = (Abar - 1) / A * u, or delta u where A = 0
          const f2 bu = fma2(zm[j], du2, mul2(em1, mul2(invA[j], xu2)));
          h[j] = fma2(a, h[j], mul2(bu, Bv[j]));
          if (j & 1) y1 = fma2(Cv[j], h[j], y1);
          else y0 = fma2(Cv[j], h[j], y0);
        }
      } else {
        const f2 du2 = pk(dl * xu, dl * xu);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          const f2 e2 = mul2(dl2, A2[j]);
          const f2 a = pk(ex2(f2lo(e2)), ex2(f2hi(e2)));
          h[j] = fma2(a, h[j], mul2(du2, Bv[j]));
          if (j & 1) y1 = fma2(Cv[j], h[j], y1);
          else y0 = fma2(Cv[j], h[j], y0);
        }
      }
      const f2 ys = add2(y0, y1);
      float yp = f2lo(ys) + f2hi(ys);
#pragma unroll
      for (int m = 1; m < SG; m <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, m);
      float yv = fmaf(D_d, xu, yp);
      if (has_z) yv *= silu(sm_elem<TIn>(buf + off_z + tt * IN_ROW, ch));
      st_out(static_cast<TOut*>(p.y) + (b * L + t0 + tt) * Dm + dc, yv, dv && owner);
    }
    __syncwarp();  // buffer s & 1 is refilled next iteration
  }
  if (dv && p.h_last) {
    float* hl = p.h_last + (b * Dm + d) * NST + soff;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      hl[2 * j] = f2lo(h[j]);
      hl[2 * j + 1] = f2hi(h[j]);
    }
  }
}

template <typename TIn, typename TOut, int SG>
cudaError_t launch_sg(const GenParams& p, int smem, cudaStream_t s) {
  const int64_t nblk = p.batch * (int64_t)p.ncblk;
  auto k = p.disc == 1 ? scan_general_kernel<TIn, TOut, SG, true> : scan_general_kernel<TIn, TOut, SG, false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<(unsigned)nblk, 32, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_io(const GenParams& p, int sg, int smem, cudaStream_t s) {
  switch (sg) {
    case 1: return launch_sg<TIn, TOut, 1>(p, smem, s);
    case 2: return launch_sg<TIn, TOut, 2>(p, smem, s);
    case 4: return launch_sg<TIn, TOut, 4>(p, smem, s);
    default: return launch_sg<TIn, TOut, 8>(p, smem, s);
  }
}

}  // namespace

int scan_general_stage_bytes(int64_t dstate, int ngw_max, ss_dtype in_dtype) {
  const int es = in_dtype == SS_BF16 ? 2 : 4;
  const int sg = (int)(dstate / 16);
  const int in_row = (32 / sg) * es;
  return kGT * (3 * in_row + 2 * ngw_max * (int)dstate * es);
}

cudaError_t launch_scan_general(const GenParams& p, int sg, ss_dtype in_dtype, ss_dtype out_dtype,
                                cudaStream_t stream) {
  const int smem = 2 * scan_general_stage_bytes(16 * sg, p.ngw_max, in_dtype);
  if (in_dtype == SS_BF16)
    return out_dtype == SS_BF16 ? launch_io<__nv_bfloat16, __nv_bfloat16>(p, sg, smem, stream)
                                : launch_io<__nv_bfloat16, float>(p, sg, smem, stream);
  return out_dtype == SS_BF16 ? launch_io<float, __nv_bfloat16>(p, sg, smem, stream)
                              : launch_io<float, float>(p, sg, smem, stream);
}

}  // namespace ssk
