// State-space-dual (Mamba-2) layer forward for sm_103a on the tensor cores.
//
// Per batch element and head h (scalar decay A_h, head channels p < P = 64,
// state n < N), with delta_t = softplus(dt_t + dt_bias_h):
//   H_t = exp(delta_t A_h) H_{t-1} + delta_t x_t B_t^T      ([P, N])
//   y_t = H_t C_t + D_h x_t
// Because the decay is one scalar per head, the map x -> y is multiplication by
// a semiseparable matrix M[t, s] = (C_t . B_s) delta_s exp(sum_{s<k<=t} delta_k
// A_h), shared by the head's P channels, and chunks of the sequence turn the
// scan into matrix products ("AI 推理系列（十四）：Mamba 的 Selective State
// Space", section on Mamba-2 reorganising the SSM as matrix computation;
// mlqm.cn tutorial, section 8). With cs_t the decay accumulated inside a chunk
// of Q = 64 steps and H_in the state entering it:
//   S = C B^T;  M = S o decay mask o delta;  Y = M X + exp(cs) o (C H_in) + D X
//   H_out = exp(cs_end) H_in + (B o exp(cs_end - cs) delta)^T X
// One CTA (4 warps) owns one (batch, head) and walks its chunks in order; the
// state lives in mma accumulators ([N, P] over the 4 warps). All products run
// on mma.sync m16n8k16 (bf16 in, fp32 accumulate). x, B and C enter as the
// bf16 values stored; the operands computed on chip (M, the weighted B, the
// state) are split into a bf16 high part and a bf16 remainder, two products
// each, so they carry about 16 significant bits. Tiles are staged by cp.async
// into XOR-swizzled shared memory (conflict-free fragment loads); the next
// chunk's tiles load while the state update runs.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kQ = 64;        // chunk length
constexpr int kP = 64;        // head channels
constexpr int kThreads = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Byte offset of element (r, c) of a bf16 tile with ROWB bytes per row (a
// multiple of 128): 16-byte pieces of row r are permuted by r mod 8, so the
// eight rows a fragment load touches fall in different banks.
template <int ROWB>
__device__ __forceinline__ int swz(int r, int c) {
  return r * ROWB + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1);
}
template <int ROWB>
__device__ __forceinline__ uint32_t ld32(const uint8_t* t, int r, int c) {
  return *reinterpret_cast<const uint32_t*>(t + swz<ROWB>(r, c));
}
template <int ROWB>
__device__ __forceinline__ void st16(uint8_t* t, int r, int c, __nv_bfloat16 v) {
  *reinterpret_cast<__nv_bfloat16*>(t + swz<ROWB>(r, c)) = v;
}
template <int ROWB>
__device__ __forceinline__ __nv_bfloat16 ld16(const uint8_t* t, int r, int c) {
  return *reinterpret_cast<const __nv_bfloat16*>(t + swz<ROWB>(r, c));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
// v = hi + lo with hi = bf16(v), lo = bf16(v - hi); returns packed pairs for two values
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
  hi = pack_bf16(h0, h1);
  lo = pack_bf16(__float2bfloat16_rn(v0 - __bfloat162float(h0)), __float2bfloat16_rn(v1 - __bfloat162float(h1)));
}

template <int N>
struct SsdSmem {
  static constexpr int XR = kP * 2;  // bytes per row of x [s][p]
  static constexpr int TR = kQ * 2;  // bytes per row of the transposed tiles [.][s]
  static constexpr int BR = N * 2;   // bytes per row of B, C [s][n] and of the state [p][n]
  static constexpr int X = 0;
  static constexpr int XT = X + kQ * XR;           // x^T [p][s]
  static constexpr int B = XT + kP * TR;           // B [s][n]
  static constexpr int C = B + kQ * BR;            // C [s][n]
  static constexpr int BT_HI = C + kQ * BR;        // weighted B^T [n][s], high part
  static constexpr int BT_LO = BT_HI + N * TR;     // remainder
  static constexpr int HT_HI = BT_LO + N * TR;     // state^T [p][n], high part
  static constexpr int HT_LO = HT_HI + kP * BR;
  static constexpr int DELTA = HT_LO + kP * BR;    // delta_t [Q] (float)
  static constexpr int CS = DELTA + kQ * 4;        // log2 of the decay accumulated to t [Q] (float)
  static constexpr int BYTES = CS + kQ * 4;
};

template <int N, typename TOut>
__global__ void __launch_bounds__(kThreads) ssd_fwd_kernel(const __grid_constant__ SsdParams p) {
  using SM = SsdSmem<N>;
  constexpr int NW = N / 4;      // state rows per warp in the state update
  constexpr int MT = NW / 16;    // m-tiles per warp there
  extern __shared__ __align__(128) uint8_t sm[];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / p.nheads, h = bh % p.nheads;
  const int64_t L = p.seqlen, H = p.nheads, G = p.ngroups;
  const int64_t grp = h / (H / G);
  const float a2 = __ldg(p.A + h) * kLog2e;  // decay exponent per unit delta, base 2
  const float dtb = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
  const float Dh = p.D ? __ldg(p.D + h) : 0.f;
  const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(p.x);
  const __nv_bfloat16* DT = static_cast<const __nv_bfloat16*>(p.dt);
  const __nv_bfloat16* Bg = static_cast<const __nv_bfloat16*>(p.B);
  const __nv_bfloat16* Cg = static_cast<const __nv_bfloat16*>(p.C);
  const int64_t nchunk = (L + kQ - 1) / kQ;

  auto stage = [&](int64_t c) {
    const int64_t t0 = c * kQ;
    const uint32_t s0 = smem_u32(sm);
    // x rows: 64 rows x 8 pieces
    for (int i = tid; i < kQ * (SM::XR / 16); i += kThreads) {
      const int r = i / (SM::XR / 16), k = i % (SM::XR / 16);
      const bool ok = t0 + r < L;
      const __nv_bfloat16* src = X + (ok ? ((b * L + t0 + r) * H + h) * kP + k * 8 : 0);
      cp_async16(s0 + SM::X + r * SM::XR + ((k ^ (r & 7)) << 4), src, ok ? 16u : 0u);
    }
    for (int i = tid; i < kQ * (SM::BR / 16); i += kThreads) {
      const int r = i / (SM::BR / 16), k = i % (SM::BR / 16);
      const bool ok = t0 + r < L;
      const int64_t e = ok ? ((b * L + t0 + r) * G + grp) * N + k * 8 : 0;
      const int off = r * SM::BR + ((k ^ (r & 7)) << 4);
      cp_async16(s0 + SM::B + off, Bg + e, ok ? 16u : 0u);
      cp_async16(s0 + SM::C + off, Cg + e, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  // the state: warp w holds rows n in [w NW, (w+1) NW) x all 64 head channels
  float Hacc[MT][8][4];
  {
    const float* h0 = p.h0 ? p.h0 + (b * H + h) * kP * N : nullptr;
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int n = w * NW + mt * 16 + g + (e >> 1) * 8, pc = q * 8 + 2 * t4 + (e & 1);
          Hacc[mt][q][e] = h0 ? __ldg(h0 + pc * N + n) : 0.f;
        }
  }
  // the state's transpose [p][n] in shared memory, split into two bf16 parts
  auto write_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int n = w * NW + mt * 16 + g + (e >> 1) * 8, pc = q * 8 + 2 * t4 + (e & 1);
          const float v = Hacc[mt][q][e];
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          st16<SM::BR>(sm + SM::HT_HI, pc, n, hi);
          st16<SM::BR>(sm + SM::HT_LO, pc, n, __float2bfloat16_rn(v - __bfloat162float(hi)));
        }
  };
  write_state();
  bool state_nonzero = p.h0 != nullptr;

  stage(0);
  for (int64_t c = 0; c < nchunk; c++) {
    const int64_t t0 = c * kQ;
    cp_async_wait0();
    __syncthreads();  // tiles of chunk c and the state are in shared memory
    // delta and the accumulated decay (warp 0); x^T (the others)
    if (w == 0) {
      float dl[2], da[2];
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const int r = 2 * lane + k;
        const bool ok = t0 + r < L;
        dl[k] = ok ? softplus_fast(__bfloat162float(DT[(b * L + t0 + r) * H + h]) + dtb) : 0.f;
        da[k] = dl[k] * a2;
      }
      // inclusive prefix sum over the 64 steps (two per lane)
      float s = da[0] + da[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
      }
      const float excl = s - (da[0] + da[1]);
      float* dls = reinterpret_cast<float*>(sm + SM::DELTA);
      float* css = reinterpret_cast<float*>(sm + SM::CS);
      dls[2 * lane] = dl[0];
      dls[2 * lane + 1] = dl[1];
      css[2 * lane] = excl + da[0];
      css[2 * lane + 1] = s;
    } else {
      for (int i = tid - 32; i < kQ * kP; i += kThreads - 32) {
        const int s = i / kP, pc = i % kP;
        st16<SM::TR>(sm + SM::XT, pc, s, ld16<SM::XR>(sm + SM::X, s, pc));
      }
    }
    __syncthreads();
    const float* dls = reinterpret_cast<const float*>(sm + SM::DELTA);
    const float* css = reinterpret_cast<const float*>(sm + SM::CS);
    const float cs_end = css[kQ - 1];

    // ---- outputs of rows t in [16 w, 16 w + 16)
    {
      const int r0 = 16 * w;
      float S[8][4];
#pragma unroll
      for (int j = 0; j < 8; j++)
#pragma unroll
        for (int e = 0; e < 4; e++) S[j][e] = 0.f;
      // S = C B^T on the causal tiles (s < 16 (w + 1))
#pragma unroll
      for (int k0 = 0; k0 < N; k0 += 16) {
        uint32_t a[4];
        a[0] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4);
        a[1] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4);
        a[2] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4 + 8);
        a[3] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4 + 8);
#pragma unroll
        for (int j = 0; j < 8; j++) {
          if (j <= 2 * w + 1) {
            const uint32_t b0 = ld32<SM::BR>(sm + SM::B, 8 * j + g, k0 + 2 * t4);
            const uint32_t b1 = ld32<SM::BR>(sm + SM::B, 8 * j + g, k0 + 2 * t4 + 8);
            mma16816(S[j], a, b0, b1);
          }
        }
      }
      // M = S o exp(cs_t - cs_s) o delta_s for s <= t, else 0
#pragma unroll
      for (int j = 0; j < 8; j++) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int t = r0 + g + (e >> 1) * 8, s = 8 * j + 2 * t4 + (e & 1);
          S[j][e] = (j <= 2 * w + 1 && s <= t) ? S[j][e] * ex2(css[t] - css[s]) * dls[s] : 0.f;
        }
      }
      float Y[8][4];
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int e = 0; e < 4; e++) Y[q][e] = 0.f;
      // Y = M X (k over s < 16 (w + 1))
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        if (kk <= w) {
          uint32_t ah[4], al[4];
          split2(S[2 * kk][0], S[2 * kk][1], ah[0], al[0]);
          split2(S[2 * kk][2], S[2 * kk][3], ah[1], al[1]);
          split2(S[2 * kk + 1][0], S[2 * kk + 1][1], ah[2], al[2]);
          split2(S[2 * kk + 1][2], S[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
          for (int q = 0; q < 8; q++) {
            const uint32_t b0 = ld32<SM::TR>(sm + SM::XT, 8 * q + g, 16 * kk + 2 * t4);
            const uint32_t b1 = ld32<SM::TR>(sm + SM::XT, 8 * q + g, 16 * kk + 2 * t4 + 8);
            mma16816(Y[q], ah, b0, b1);
            mma16816(Y[q], al, b0, b1);
          }
        }
      }
      // + exp(cs_t) C_t H_in
      if (state_nonzero) {
        float Yo[8][4];
#pragma unroll
        for (int q = 0; q < 8; q++)
#pragma unroll
          for (int e = 0; e < 4; e++) Yo[q][e] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
          uint32_t a[4];
          a[0] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4);
          a[1] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4);
          a[2] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4 + 8);
          a[3] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4 + 8);
#pragma unroll
          for (int q = 0; q < 8; q++) {
            mma16816(Yo[q], a, ld32<SM::BR>(sm + SM::HT_HI, 8 * q + g, k0 + 2 * t4),
                     ld32<SM::BR>(sm + SM::HT_HI, 8 * q + g, k0 + 2 * t4 + 8));
            mma16816(Yo[q], a, ld32<SM::BR>(sm + SM::HT_LO, 8 * q + g, k0 + 2 * t4),
                     ld32<SM::BR>(sm + SM::HT_LO, 8 * q + g, k0 + 2 * t4 + 8));
          }
        }
        const float d0 = ex2(css[r0 + g]), d1 = ex2(css[r0 + g + 8]);
#pragma unroll
        for (int q = 0; q < 8; q++) {
          Y[q][0] = fmaf(d0, Yo[q][0], Y[q][0]);
          Y[q][1] = fmaf(d0, Yo[q][1], Y[q][1]);
          Y[q][2] = fmaf(d1, Yo[q][2], Y[q][2]);
          Y[q][3] = fmaf(d1, Yo[q][3], Y[q][3]);
        }
      }
      // + D x, store
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int t = r0 + g + 8 * half;
        if (t0 + t < L) {
          TOut* yrow = static_cast<TOut*>(p.y) + ((b * L + t0 + t) * H + h) * kP;
#pragma unroll
          for (int q = 0; q < 8; q++) {
            const int pc = 8 * q + 2 * t4;
            const float x0 = __bfloat162float(ld16<SM::XR>(sm + SM::X, t, pc));
            const float x1 = __bfloat162float(ld16<SM::XR>(sm + SM::X, t, pc + 1));
            const float v0 = fmaf(Dh, x0, Y[q][2 * half]), v1 = fmaf(Dh, x1, Y[q][2 * half + 1]);
            if constexpr (sizeof(TOut) == 4) {
              *reinterpret_cast<float2*>(yrow + pc) = make_float2(v0, v1);
            } else {
              *reinterpret_cast<uint32_t*>(yrow + pc) = pack_bf16(__float2bfloat16_rn(v0), __float2bfloat16_rn(v1));
            }
          }
        }
      }
    }

    // ---- weighted B^T [n][s] = B[s][n] exp(cs_end - cs_s) delta_s (two bf16 parts)
    for (int i = tid; i < kQ * N; i += kThreads) {
      const int s = i / N, n = i % N;
      const float v = __bfloat162float(ld16<SM::BR>(sm + SM::B, s, n)) * ex2(cs_end - css[s]) * dls[s];
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      st16<SM::TR>(sm + SM::BT_HI, n, s, hi);
      st16<SM::TR>(sm + SM::BT_LO, n, s, __float2bfloat16_rn(v - __bfloat162float(hi)));
    }
    __syncthreads();  // every warp is past its reads of x, B, C and the state
    if (c + 1 < nchunk) stage(c + 1);

    // ---- H = exp(cs_end) H + Bw^T X
    {
      const float dec = ex2(cs_end);
#pragma unroll
      for (int mt = 0; mt < MT; mt++)
#pragma unroll
        for (int q = 0; q < 8; q++)
#pragma unroll
          for (int e = 0; e < 4; e++) Hacc[mt][q][e] *= dec;
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
          const int m0 = w * NW + mt * 16;
          uint32_t ah[4], al[4];
          ah[0] = ld32<SM::TR>(sm + SM::BT_HI, m0 + g, 16 * kk + 2 * t4);
          ah[1] = ld32<SM::TR>(sm + SM::BT_HI, m0 + g + 8, 16 * kk + 2 * t4);
          ah[2] = ld32<SM::TR>(sm + SM::BT_HI, m0 + g, 16 * kk + 2 * t4 + 8);
          ah[3] = ld32<SM::TR>(sm + SM::BT_HI, m0 + g + 8, 16 * kk + 2 * t4 + 8);
          al[0] = ld32<SM::TR>(sm + SM::BT_LO, m0 + g, 16 * kk + 2 * t4);
          al[1] = ld32<SM::TR>(sm + SM::BT_LO, m0 + g + 8, 16 * kk + 2 * t4);
          al[2] = ld32<SM::TR>(sm + SM::BT_LO, m0 + g, 16 * kk + 2 * t4 + 8);
          al[3] = ld32<SM::TR>(sm + SM::BT_LO, m0 + g + 8, 16 * kk + 2 * t4 + 8);
#pragma unroll
          for (int q = 0; q < 8; q++) {
            const uint32_t b0 = ld32<SM::TR>(sm + SM::XT, 8 * q + g, 16 * kk + 2 * t4);
            const uint32_t b1 = ld32<SM::TR>(sm + SM::XT, 8 * q + g, 16 * kk + 2 * t4 + 8);
            mma16816(Hacc[mt][q], ah, b0, b1);
            mma16816(Hacc[mt][q], al, b0, b1);
          }
        }
      }
    }
    write_state();
    state_nonzero = true;
  }

  if (p.h_last) {
    float* hl = p.h_last + (b * H + h) * kP * N;
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const int n = w * NW + mt * 16 + g + (e >> 1) * 8, pc = q * 8 + 2 * t4 + (e & 1);
          hl[pc * N + n] = Hacc[mt][q][e];
        }
  }
}

template <int N, typename TOut>
cudaError_t launch_n(const SsdParams& p, cudaStream_t s) {
  const int smem = SsdSmem<N>::BYTES;
  auto k = ssd_fwd_kernel<N, TOut>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<(unsigned)(p.batch * p.nheads), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_fwd(const SsdParams& p, int dstate, ss_dtype out_dtype, cudaStream_t stream) {
  if (dstate == 64)
    return out_dtype == SS_BF16 ? launch_n<64, __nv_bfloat16>(p, stream) : launch_n<64, float>(p, stream);
  return out_dtype == SS_BF16 ? launch_n<128, __nv_bfloat16>(p, stream) : launch_n<128, float>(p, stream);
}

}  // namespace ssk
