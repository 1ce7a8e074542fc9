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
// into XOR-swizzled shared memory; fragments that run along a stored tile's
// rows (x, the state, B^T) come by ldmatrix.trans, so nothing is transposed
// through shared memory. The next chunk's C tile loads during the state update,
// its x and B tiles after it. 72.5 KB of shared memory per CTA keeps three
// CTAs on an SM.
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

// ldmatrix .x4 .trans: four 8x8 bf16 blocks whose rows (16 bytes each) the
// lanes address (lanes 8j..8j+7 give the rows of block j); lane l receives, per
// block, the elements (rows 2(l%4), 2(l%4)+1; column l/4): the pair that an
// mma fragment needs along the stored row dimension.
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <int N>
struct SsdSmem {
  static constexpr int XR = kP * 2;  // bytes per row of x [s][p] and of the state [n][p]
  static constexpr int BR = N * 2;   // bytes per row of B, C [s][n]
  static constexpr int X = 0;
  static constexpr int B = X + kQ * XR;            // B [s][n]
  static constexpr int C = B + kQ * BR;            // C [s][n]
  static constexpr int H_HI = C + kQ * BR;         // state [n][p], high part
  static constexpr int H_LO = H_HI + N * XR;       // remainder
  static constexpr int DELTA = H_LO + N * XR;      // delta_t [Q] (float)
  static constexpr int CS = DELTA + kQ * 4;        // log2 of the decay accumulated to t [Q] (float)
  static constexpr int W = CS + kQ * 4;            // weight of step s in the chunk's state: exp(cs_end - cs_s) delta_s
  static constexpr int BYTES = W + kQ * 4;
};

template <int N, typename TOut>
__global__ void __launch_bounds__(kThreads, 3) ssd_fwd_kernel(const __grid_constant__ SsdParams p) {
  using SM = SsdSmem<N>;
  constexpr int NW = N / 4;      // state rows per warp in the state update
  constexpr int MT = NW / 16;    // m-tiles per warp there
  extern __shared__ __align__(128) uint8_t sm[];
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int lj = lane >> 3, lr = lane & 7;  // ldmatrix block and row this lane addresses
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
  const uint32_t s0 = smem_u32(sm);

  // cp.async of chunk c's x and B tiles, or of its C tile
  auto stage_xb = [&](int64_t c) {
    const int64_t t0 = c * kQ;
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
      cp_async16(s0 + SM::B + r * SM::BR + ((k ^ (r & 7)) << 4), Bg + e, ok ? 16u : 0u);
    }
  };
  auto stage_c = [&](int64_t c) {
    const int64_t t0 = c * kQ;
    for (int i = tid; i < kQ * (SM::BR / 16); i += kThreads) {
      const int r = i / (SM::BR / 16), k = i % (SM::BR / 16);
      const bool ok = t0 + r < L;
      const int64_t e = ok ? ((b * L + t0 + r) * G + grp) * N + k * 8 : 0;
      cp_async16(s0 + SM::C + r * SM::BR + ((k ^ (r & 7)) << 4), Cg + e, ok ? 16u : 0u);
    }
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
  // the state [n][p] in shared memory as two bf16 parts (32-bit stores of pairs)
  auto write_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < MT; mt++)
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int hf = 0; hf < 2; hf++) {
          const int n = w * NW + mt * 16 + g + hf * 8, pc = q * 8 + 2 * t4;
          uint32_t hi, lo;
          split2(Hacc[mt][q][2 * hf], Hacc[mt][q][2 * hf + 1], hi, lo);
          *reinterpret_cast<uint32_t*>(sm + SM::H_HI + swz<SM::XR>(n, pc)) = hi;
          *reinterpret_cast<uint32_t*>(sm + SM::H_LO + swz<SM::XR>(n, pc)) = lo;
        }
  };
  write_state();
  bool state_nonzero = p.h0 != nullptr;

  stage_xb(0);
  stage_c(0);
  cp_async_commit();
  for (int64_t c = 0; c < nchunk; c++) {
    const int64_t t0 = c * kQ;
    cp_async_wait0();
    __syncthreads();  // tiles of chunk c and the state are in shared memory
    // delta, the accumulated decay and the state weights (warp 0)
    if (w == 0) {
      float dl[2], da[2];
#pragma unroll
      for (int k = 0; k < 2; k++) {
        const int r = 2 * lane + k;
        const bool ok = t0 + r < L;
        dl[k] = ok ? softplus_fast(__bfloat162float(DT[(b * L + t0 + r) * H + h]) + dtb) : 0.f;
        da[k] = dl[k] * a2;
      }
      float s = da[0] + da[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += v;
      }
      const float c0v = s - da[1];  // inclusive through step 2 lane
      const float cend = __shfl_sync(0xffffffffu, s, 31);
      float* dls = reinterpret_cast<float*>(sm + SM::DELTA);
      float* css = reinterpret_cast<float*>(sm + SM::CS);
      float* wts = reinterpret_cast<float*>(sm + SM::W);
      dls[2 * lane] = dl[0];
      dls[2 * lane + 1] = dl[1];
      css[2 * lane] = c0v;
      css[2 * lane + 1] = s;
      wts[2 * lane] = ex2(cend - c0v) * dl[0];
      wts[2 * lane + 1] = ex2(cend - s) * dl[1];
    }
    __syncthreads();
    const float* dls = reinterpret_cast<const float*>(sm + SM::DELTA);
    const float* css = reinterpret_cast<const float*>(sm + SM::CS);
    const float* wts = reinterpret_cast<const float*>(sm + SM::W);
    const float cs_end = css[kQ - 1];

    // ---- outputs of rows t in [16 w, 16 w + 16)
    {
      const int r0 = 16 * w;
      float Y[8][4];
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int e = 0; e < 4; e++) Y[q][e] = 0.f;
      // exp(cs_t) C_t H_in first, scaled in place
      if (state_nonzero) {
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
          uint32_t a[4];
          a[0] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4);
          a[1] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4);
          a[2] = ld32<SM::BR>(sm + SM::C, r0 + g, k0 + 2 * t4 + 8);
          a[3] = ld32<SM::BR>(sm + SM::C, r0 + g + 8, k0 + 2 * t4 + 8);
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            const int row = k0 + (lj & 1) * 8 + lr, col = 8 * (q + (lj >> 1));
            uint32_t bh4[4], bl4[4];
            ldsm_x4_t(bh4, s0 + SM::H_HI + swz<SM::XR>(row, col));
            ldsm_x4_t(bl4, s0 + SM::H_LO + swz<SM::XR>(row, col));
            mma16816(Y[q], a, bh4[0], bh4[1]);
            mma16816(Y[q], a, bl4[0], bl4[1]);
            mma16816(Y[q + 1], a, bh4[2], bh4[3]);
            mma16816(Y[q + 1], a, bl4[2], bl4[3]);
          }
        }
        const float d0 = ex2(css[r0 + g]), d1 = ex2(css[r0 + g + 8]);
#pragma unroll
        for (int q = 0; q < 8; q++) {
          Y[q][0] *= d0;
          Y[q][1] *= d0;
          Y[q][2] *= d1;
          Y[q][3] *= d1;
        }
      }
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
      // Y += M X (k over s < 16 (w + 1)); X fragments by ldmatrix.trans
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        if (kk <= w) {
          uint32_t ah[4], al[4];
          split2(S[2 * kk][0], S[2 * kk][1], ah[0], al[0]);
          split2(S[2 * kk][2], S[2 * kk][3], ah[1], al[1]);
          split2(S[2 * kk + 1][0], S[2 * kk + 1][1], ah[2], al[2]);
          split2(S[2 * kk + 1][2], S[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            uint32_t bx[4];
            ldsm_x4_t(bx, s0 + SM::X + swz<SM::XR>(16 * kk + (lj & 1) * 8 + lr, 8 * (q + (lj >> 1))));
            mma16816(Y[q], ah, bx[0], bx[1]);
            mma16816(Y[q], al, bx[0], bx[1]);
            mma16816(Y[q + 1], ah, bx[2], bx[3]);
            mma16816(Y[q + 1], al, bx[2], bx[3]);
          }
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
            const uint32_t xw = ld32<SM::XR>(sm + SM::X, t, pc);
            const float x0 = __uint_as_float(xw << 16), x1 = __uint_as_float(xw & 0xffff0000u);
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
    __syncthreads();  // every warp is past its reads of C and of the state
    if (c + 1 < nchunk) stage_c(c + 1);

    // ---- H = exp(cs_end) H + (w o B)^T X: A fragments of B^T by ldmatrix.trans, weighted and split
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
        const int s0k = 16 * kk + 2 * t4;
        const float w0 = wts[s0k], w1 = wts[s0k + 1], w8 = wts[s0k + 8], w9 = wts[s0k + 9];
#pragma unroll
        for (int mt = 0; mt < MT; mt++) {
          const int m0 = w * NW + mt * 16;
          uint32_t raw[4];
          ldsm_x4_t(raw, s0 + SM::B + swz<SM::BR>(16 * kk + (lj >> 1) * 8 + lr, m0 + (lj & 1) * 8));
          uint32_t ah[4], al[4];
#pragma unroll
          for (int r = 0; r < 4; r++) {
            const float wl = r < 2 ? w0 : w8, wh = r < 2 ? w1 : w9;
            split2(__uint_as_float(raw[r] << 16) * wl, __uint_as_float(raw[r] & 0xffff0000u) * wh, ah[r], al[r]);
          }
#pragma unroll
          for (int q = 0; q < 8; q += 2) {
            uint32_t bx[4];
            ldsm_x4_t(bx, s0 + SM::X + swz<SM::XR>(16 * kk + (lj & 1) * 8 + lr, 8 * (q + (lj >> 1))));
            mma16816(Hacc[mt][q], ah, bx[0], bx[1]);
            mma16816(Hacc[mt][q], al, bx[0], bx[1]);
            mma16816(Hacc[mt][q + 1], ah, bx[2], bx[3]);
            mma16816(Hacc[mt][q + 1], al, bx[2], bx[3]);
          }
        }
      }
    }
    write_state();
    state_nonzero = true;
    __syncthreads();  // every warp is past its reads of x and B
    if (c + 1 < nchunk) stage_xb(c + 1);
    cp_async_commit();
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
  if (dstate == 128) return launch_ssd_fwd_tc(p, out_dtype, stream);
  return out_dtype == SS_BF16 ? launch_n<64, __nv_bfloat16>(p, stream) : launch_n<64, float>(p, stream);
}

}  // namespace ssk
