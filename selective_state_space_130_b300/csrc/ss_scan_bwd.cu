// Gradients of the selective scan (the backward pass) for sm_103a, with the
// forward states recomputed instead of stored.
//
// The pages train Mamba end to end and say the backward pass recomputes the
// intermediate states rather than reading them back from HBM ("Mamba:
// Linear-Time Sequence Modeling with Selective State Spaces" review page,
// method step 2 (3)). For each channel the gradients follow from the reverse
// sweep of the adjoint state lambda_t = dL/dh_t:
//   lambda_t = C_t dyv_t + Abar_{t+1} lambda_{t+1},  dyv_t = dy_t silu(z_t)
// with dB, dC summed over channels and dA, dD, dbias summed over batch and
// time (the per-term formulas are in the C header, ss_scan_bwd).
//
// One warp owns 32 channels of one batch element (lane = channel, 16 fp32
// states in registers). Phase 1 runs the recurrence forward and writes the
// state every kSub steps to a checkpoint buffer in the workspace. Phase 2
// walks the sub-tiles backwards: it recomputes the kSub states of a sub-tile
// from its checkpoint into shared memory, then runs the adjoint backwards
// through them. dB and dC, shared by all channels, are summed over the warp by
// a shuffle butterfly (lane l ends with element l of the 32 per-token values)
// and added to global memory with one atomic per lane per token.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kSub = 16;  // timesteps per recomputed sub-tile

__device__ __forceinline__ float sigmoidf_fast(float x) { return rcp(1.f + ex2(-x * kLog2e)); }

// Shared memory of one warp: the recomputed states of a sub-tile and two
// staging buffers of raw inputs (one being read, one being filled). SG lanes
// share a channel, each holding NS = 16 / SG of its states; a warp covers
// CW = 32 / SG channels.
template <typename TIn, typename TDy, int SG>
struct BwdLayout {
  static constexpr int CW = 32 / SG;
  static constexpr int NS = kDState / SG;
  static constexpr int NQ = NS / 4;  // 16-byte entries per lane per saved state
  static constexpr int IN_ROW = CW * (int)sizeof(TIn);  // one step of u, delta_raw or z
  static constexpr int DY_ROW = CW * (int)sizeof(TDy);
  static constexpr int BC_ROW = kDState * (int)sizeof(TIn);  // one step of B (or C)
  static constexpr int OFF_U = 0;
  static constexpr int OFF_DR = OFF_U + kSub * IN_ROW;
  static constexpr int OFF_Z = OFF_DR + kSub * IN_ROW;
  static constexpr int OFF_DY = OFF_Z + kSub * IN_ROW;
  static constexpr int OFF_B = OFF_DY + kSub * DY_ROW;
  static constexpr int OFF_C = OFF_B + kSub * BC_ROW;
  static constexpr int STAGE = OFF_C + kSub * BC_ROW;
  static constexpr int HIST = (kSub + 1) * NQ * 32 * 16;  // one 16-byte entry per (slot, quad, lane)
  // the current sub-tile's B and C widened to fp32 (bf16 inputs; fp32 ones are
  // read from the stage), and its delta = softplus(delta_raw + bias) per step
  // and channel, each computed once per sub-tile
  static constexpr bool WIDEN = sizeof(TIn) == 2;
  static constexpr int OFF_WB = HIST + 2 * STAGE;
  static constexpr int OFF_WC = OFF_WB + (WIDEN ? kSub * kDState * 4 : 0);
  static constexpr int OFF_DL = OFF_WC + (WIDEN ? kSub * kDState * 4 : 0);
  static constexpr int SMEM = OFF_DL + kSub * CW * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

template <typename T>
__device__ __forceinline__ float sm_elem(const uint8_t* row, int i) {
  return to_f32(reinterpret_cast<const T*>(row)[i]);
}

// Copy kSub rows of `rowb` bytes (rows `stride` elements apart, starting at
// element `e0` of `base`) into shared memory at `dst`. Rows at or past
// `nrows` and elements at or past `nelem` within a row are filled with zeros.
// VEC: 16-byte asynchronous copies (every 16-byte piece lies wholly inside or
// wholly outside the valid range); otherwise element-wise loads and stores.
template <typename T, int ROWB, bool VEC>
__device__ __forceinline__ void stage_rows(uint8_t* dst, const void* base, int64_t e0, int64_t stride, int nrows,
                                           int nelem, int lane) {
  constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte piece
  constexpr int CPR = ROWB / 16;            // pieces per row
  if constexpr (VEC) {
    const uint32_t d0 = (uint32_t)__cvta_generic_to_shared(dst);
#pragma unroll
    for (int c = lane; c < kSub * CPR; c += 32) {
      const int tt = c / CPR, k = c % CPR;
      const bool ok = tt < nrows && k * EPC < nelem;
      const T* src = static_cast<const T*>(base) + (ok ? e0 + tt * stride + k * EPC : 0);
      cp_async16(d0 + tt * ROWB + k * 16, src, ok ? 16u : 0u);
    }
  } else {
    constexpr int EPR = ROWB / (int)sizeof(T);  // elements per row
#pragma unroll 4
    for (int c = lane; c < kSub * EPR; c += 32) {
      const int tt = c / EPR, k = c % EPR;
      const bool ok = tt < nrows && k < nelem;
      reinterpret_cast<T*>(dst)[c] = ok ? static_cast<const T*>(base)[e0 + tt * stride + k] : from_f32<T>(0.f);
    }
  }
}

// Abar for a pair of states: 2^(delta * A2)
__device__ __forceinline__ f2 abar2(f2 dl2, f2 a2) {
  const f2 e = mul2(dl2, a2);
  return pk(ex2(f2lo(e)), ex2(f2hi(e)));
}

constexpr int kBwdWarps = 4;  // warps per CTA, one per SM sub-partition; each runs its own share

template <typename TIn, typename TDy, int SG, bool HAS_Z, bool VEC>
__global__ void __launch_bounds__(32 * kBwdWarps) scan_bwd_kernel(const __grid_constant__ BwdParams p) {
  using LY = BwdLayout<TIn, TDy, SG>;
  constexpr int CW = LY::CW, NS = LY::NS, NQ = LY::NQ, NP = NS / 2;
  extern __shared__ __align__(16) uint8_t smem_all[];
  const int wib = threadIdx.x >> 5;  // warp within the CTA: its own slice of shared memory
  uint8_t* smem_raw = smem_all + wib * LY::SMEM;
  ulonglong2* hist = reinterpret_cast<ulonglong2*>(smem_raw);  // [slot][quad][lane], two f2 per entry
  uint8_t* stage_buf = smem_raw + LY::HIST;
  const int lane = threadIdx.x & 31;
  const int64_t share = (int64_t)blockIdx.x * kBwdWarps + wib;
  if (share >= p.nshares) return;  // (warps past the last block when each warp runs one)
  const int ch = lane / SG;           // channel within the block
  const int soff = (lane % SG) * NS;  // first state of this lane
  const bool owner = (lane % SG) == 0;
  // The lane's state pairs in a lane-dependent order: position j holds pair
  // j ^ gp. gp is made of the lane bits over which the first stages of the
  // dB/dC reduction below run (16 and 8, and 4 with one lane per channel), so
  // that in those stages two partners hold the same element at positions e
  // and e + w, and every lane keeps its lower half without a select.
  constexpr int kPairBits = NP == 8 ? 3 : 2;
  static_assert(NP == 8 || NP == 4, "one or two lanes per channel");
  int gp = 0;
#pragma unroll
  for (int i = 0; i < kPairBits; i++) gp |= ((lane >> (4 - i)) & 1) << (kPairBits - 1 - i);
  // first state of the pair at position j
  auto sidx = [&](int j) { return soff + 2 * (j ^ gp); };
  const int64_t L = p.seqlen, Dm = p.dim, nsub = p.nsub;
  const uint64_t wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;

  // The share: items [g0, g1) of the blocks' sub-tiles, block-major. It covers
  // the tail of one block, whole blocks and the head of another (the job
  // order is below).
  const int64_t T = p.batch * (int64_t)p.ncblk * nsub;
  const int64_t qn = T / p.nshares, rm = T % p.nshares;
  const int64_t g0 = share * qn + (share < rm ? share : rm), g1 = g0 + qn + (share < rm ? 1 : 0);
  const int64_t u0 = g0 / nsub, u1 = (g1 - 1) / nsub;
  const int nseg = g1 > g0 ? (int)(u1 - u0 + 1) : 0;
  struct Seg {
    int64_t u, sb, se;  // block and its sub-tiles [sb, se)
  };
  auto segment = [&](int sgi) -> Seg {
    if (nseg == 1) return {u0, g0 - u0 * nsub, g1 - u0 * nsub};
    if (sgi == 0) return {u1, 0, g1 - u1 * nsub};
    if (sgi == nseg - 1) return {u0, g0 - u0 * nsub, nsub};
    return {u0 + sgi, 0, nsub};
  };
  const bool withhold = share == p.withhold_share;
  bool aborted = false;  // a hand-over wait gave up (the same on every lane)
  // bounded wait until *flag >= v (lane 0 polls; the result is the warp's)
  auto wait_flag = [&](const unsigned int* flag, uint32_t v) -> bool {
    bool got = true;
    if (lane == 0) {
      got = ld_acquire_gpu(flag) >= v;
      const uint64_t t_start = globaltimer();
      while (!got && globaltimer() - t_start <= wait_ns) got = ld_acquire_gpu(flag) >= v;
    }
    return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
  };
  auto publish = [&](unsigned int* flag, uint32_t v) {
    __syncwarp();
    if (lane == 0 && !withhold) {
      __threadfence();
      st_release_gpu(flag, v);
    }
  };

  // per-block quantities, set at the start of each job
  int64_t b = 0, c0 = 0, d = 0, dc = 0;
  bool dv = false;
  int nch = 0;
  f2 A2[NP];
  float bias_d = 0.f, D_d = 0.f;
  float bias_p = 0.f;  // bias of channel lane % CW, whose deltas this lane computes in prep
  auto set_block = [&](int64_t u) {
    b = u / p.ncblk;
    c0 = (u % p.ncblk) * CW;
    d = c0 + ch;
    dv = d < Dm;
    dc = dv ? d : 0;
    nch = (int)min((int64_t)CW, Dm - c0);
#pragma unroll
    for (int j = 0; j < NP; j++) {
      const float a0 = dv ? __ldg(p.A + dc * kDState + sidx(j)) : 0.f;
      const float a1 = dv ? __ldg(p.A + dc * kDState + sidx(j) + 1) : 0.f;
      A2[j] = pk(a0 * kLog2e, a1 * kLog2e);
    }
    bias_d = (dv && p.delta_bias) ? __ldg(p.delta_bias + dc) : 0.f;
    D_d = (dv && p.D) ? __ldg(p.D + dc) : 0.f;
    const int64_t dp = c0 + lane % CW;
    bias_p = (dp < Dm && p.delta_bias) ? __ldg(p.delta_bias + dp) : 0.f;
  };
  // stage sub-tile s of the current block into buffer s & 1: the forward sweep
  // needs u, delta_raw, B; the reverse sweep everything
  auto stage = [&](int64_t s, bool all) {
    uint8_t* buf = stage_buf + (s & 1) * LY::STAGE;
    const int64_t t0 = s * kSub;
    const int nr = (int)min((int64_t)kSub, L - t0);
    const int64_t e0 = (b * L + t0) * Dm + c0;
    stage_rows<TIn, LY::IN_ROW, VEC>(buf + LY::OFF_U, p.u, e0, Dm, nr, nch, lane);
    stage_rows<TIn, LY::IN_ROW, VEC>(buf + LY::OFF_DR, p.delta_raw, e0, Dm, nr, nch, lane);
    stage_rows<TIn, LY::BC_ROW, VEC>(buf + LY::OFF_B, p.B, (b * L + t0) * kDState, kDState, nr, kDState, lane);
    if (all) {
      if constexpr (HAS_Z) stage_rows<TIn, LY::IN_ROW, VEC>(buf + LY::OFF_Z, p.z, e0, Dm, nr, nch, lane);
      stage_rows<TDy, LY::DY_ROW, VEC>(buf + LY::OFF_DY, p.dy, e0, Dm, nr, nch, lane);
      stage_rows<TIn, LY::BC_ROW, VEC>(buf + LY::OFF_C, p.C, (b * L + t0) * kDState, kDState, nr, kDState, lane);
    }
    cp_async_commit();
  };
  // sum over the SG lanes of a channel
  auto chan_sum = [&](float x) {
    if constexpr (SG == 2) x += __shfl_xor_sync(0xffffffffu, x, 1);
    return x;
  };
  // this lane's B or C pairs of step tt of a staged buffer
  auto row_pairs = [&](const uint8_t* buf, int off, int tt, f2 (&o)[NP]) {
    if constexpr (sizeof(TIn) == 4) {  // (bf16 rows are read widened, from wB and wC)
      const float* r = reinterpret_cast<const float*>(buf + off + tt * LY::BC_ROW);
#pragma unroll
      for (int j = 0; j < NP; j++) {
        const float2 v = *reinterpret_cast<const float2*>(r + sidx(j));
        o[j] = pk(v.x, v.y);
      }
    }
  };
  float* wB = reinterpret_cast<float*>(smem_raw + LY::OFF_WB);
  float* wC = reinterpret_cast<float*>(smem_raw + LY::OFF_WC);
  float* dlt = reinterpret_cast<float*>(smem_raw + LY::OFF_DL);  // [kSub][CW]
  // Once sub-tile data has landed in `buf`: its B (and C) widened to fp32, and
  // delta for every (step, channel), lane l taking channel l % CW. Read after
  // the next __syncwarp.
  auto prep = [&](const uint8_t* buf, int ns, bool with_c) {
    if constexpr (LY::WIDEN) {  // kSub x 16 bf16 = 512 bytes: one 16-byte piece per lane
#pragma unroll
      for (int which = 0; which < 2; which++) {
        if (which == 1 && !with_c) break;
        const uint4 w = reinterpret_cast<const uint4*>(buf + (which ? LY::OFF_C : LY::OFF_B))[lane];
        float4* o = reinterpret_cast<float4*>((which ? wC : wB) + 8 * lane);
        o[0] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        o[1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                           __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
      }
    }
    const int cp = lane % CW;
#pragma unroll
    for (int tt = lane / CW; tt < kSub; tt += 32 / CW)
      if (tt < ns) dlt[tt * CW + cp] = softplus_fast(sm_elem<TIn>(buf + LY::OFF_DR + tt * LY::IN_ROW, cp) + bias_p);
  };
  // this lane's B or C pairs of step tt of the current sub-tile
  auto rowB = [&](const uint8_t* buf, int tt, f2 (&o)[NP]) {
    if constexpr (LY::WIDEN) {
#pragma unroll
      for (int j = 0; j < NP; j++) {
        const float2 v = *reinterpret_cast<const float2*>(wB + tt * kDState + sidx(j));
        o[j] = pk(v.x, v.y);
      }
    } else {
      row_pairs(buf, LY::OFF_B, tt, o);
    }
  };
  auto rowC = [&](const uint8_t* buf, int tt, f2 (&o)[NP]) {
    if constexpr (LY::WIDEN) {
#pragma unroll
      for (int j = 0; j < NP; j++) {
        const float2 v = *reinterpret_cast<const float2*>(wC + tt * kDState + sidx(j));
        o[j] = pk(v.x, v.y);
      }
    } else {
      row_pairs(buf, LY::OFF_C, tt, o);
    }
  };
  // this lane's 2 NP floats of a hand-over slot ([block][32 lanes][16])
  auto slot = [&](float* base, int64_t u) { return base + (u * 32 + lane) * kDState; };

  // ---- forward sweep of segment q: the recurrence, its state saved at the
  // start of every sub-tile; the state leaving a head goes to the next share
  auto fwd_job = [&](const Seg& q) {
    f2 h[NP];
    const int64_t hrow = (b * Dm + dc) * kDState;
    if (q.sb > 0) {
      if (!wait_flag(p.flags_h + q.u, (uint32_t)q.sb)) {
        aborted = true;
        return;
      }
      const float* src = slot(p.ws_h, q.u);
#pragma unroll
      for (int j = 0; j < NP; j++) h[j] = pk(src[2 * j], src[2 * j + 1]);
    } else {
#pragma unroll
      for (int j = 0; j < NP; j++)
        h[j] = (dv && p.h0) ? pk(__ldg(p.h0 + hrow + sidx(j)), __ldg(p.h0 + hrow + sidx(j) + 1)) : pk(0.f, 0.f);
    }
    ulonglong2* ck = reinterpret_cast<ulonglong2*>(p.ckpt) + (size_t)q.u * nsub * NQ * 32;
    stage(q.sb, false);
    for (int64_t s = q.sb; s < q.se; s++) {
      if (s + 1 < q.se) stage(s + 1, false);
      else cp_async_commit();
      cp_async_wait1();
      __syncwarp();
      const uint8_t* buf = stage_buf + (s & 1) * LY::STAGE;
      const int ns = (int)min((int64_t)kSub, L - s * kSub);
      prep(buf, ns, false);
      {
        ulonglong2* dst = ck + (size_t)s * NQ * 32;
#pragma unroll
        for (int qq = 0; qq < NQ; qq++) dst[qq * 32 + lane] = make_ulonglong2(h[2 * qq], h[2 * qq + 1]);
      }
      __syncwarp();
#pragma unroll 2
      for (int tt = 0; tt < ns; tt++) {
        const float xu = sm_elem<TIn>(buf + LY::OFF_U + tt * LY::IN_ROW, ch);
        const float dl = dlt[tt * CW + ch];
        const f2 dl2 = pk(dl, dl), du2 = pk(dl * xu, dl * xu);
        f2 Bv[NP];
        rowB(buf, tt, Bv);
#pragma unroll
        for (int j = 0; j < NP; j++) h[j] = fma2(abar2(dl2, A2[j]), h[j], mul2(du2, Bv[j]));
      }
      __syncwarp();  // buffer s & 1 is refilled next iteration
    }
    if (q.se < nsub) {  // a head: its state goes on to the share that holds the rest of the block
      float* dst = slot(p.ws_h, q.u);
#pragma unroll
      for (int j = 0; j < NP; j++) {
        dst[2 * j] = f2lo(h[j]);
        dst[2 * j + 1] = f2hi(h[j]);
      }
      publish(p.flags_h + q.u, (uint32_t)q.se);
    }
  };

  // ---- reverse sweep of segment q, sub-tiles in reverse order: recompute the
  // sub-tile's states from its checkpoint, then run the adjoint through them.
  // The adjoint entering a tail comes from dh_last; a head's comes from the
  // share that holds the rest of the block, and the adjoint leaving a tail
  // goes back to the share that holds the block's start.
  auto rev_job = [&](const Seg& q) {
    f2 lam[NP], dAacc[NP];
    const int64_t hrow = (b * Dm + dc) * kDState;
    if (q.se < nsub) {
      if (!wait_flag(p.flags_lam + q.u, (uint32_t)(nsub - q.se))) {
        aborted = true;
        return;
      }
      const float* src = slot(p.ws_lam, q.u);
#pragma unroll
      for (int j = 0; j < NP; j++) lam[j] = pk(src[2 * j], src[2 * j + 1]);
    } else {
#pragma unroll
      for (int j = 0; j < NP; j++)
        lam[j] = (dv && p.dh_last) ? pk(__ldg(p.dh_last + hrow + sidx(j)), __ldg(p.dh_last + hrow + sidx(j) + 1))
                                   : pk(0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < NP; j++) dAacc[j] = pk(0.f, 0.f);
    float dDacc = 0.f, dbacc = 0.f;
    const ulonglong2* ck = reinterpret_cast<const ulonglong2*>(p.ckpt) + (size_t)q.u * nsub * NQ * 32;
    stage(q.se - 1, true);
    ulonglong2 ck_next[NQ];
#pragma unroll
    for (int qq = 0; qq < NQ; qq++) ck_next[qq] = ck[(size_t)(q.se - 1) * NQ * 32 + qq * 32 + lane];
    for (int64_t s = q.se - 1; s >= q.sb; s--) {
      const int64_t t0 = s * kSub;
      const int ns = (int)min((int64_t)kSub, L - t0);
      f2 hh[NP];
#pragma unroll
      for (int qq = 0; qq < NQ; qq++) {
        hist[qq * 32 + lane] = ck_next[qq];
        hh[2 * qq] = ck_next[qq].x;
        hh[2 * qq + 1] = ck_next[qq].y;
      }
      if (s > q.sb) {
        stage(s - 1, true);
#pragma unroll
        for (int qq = 0; qq < NQ; qq++) ck_next[qq] = ck[(size_t)(s - 1) * NQ * 32 + qq * 32 + lane];
      } else {
        cp_async_commit();
      }
      cp_async_wait1();
      __syncwarp();
      const uint8_t* buf = stage_buf + (s & 1) * LY::STAGE;
      prep(buf, ns, true);
      __syncwarp();
      // recompute the sub-tile's states into shared memory (lane-private slots); dz
#pragma unroll 2
      for (int tt = 0; tt < ns; tt++) {
        const int64_t i = (b * L + t0 + tt) * Dm + dc;
        const float xu = sm_elem<TIn>(buf + LY::OFF_U + tt * LY::IN_ROW, ch);
        const float dl = dlt[tt * CW + ch];
        const f2 dl2 = pk(dl, dl), du2 = pk(dl * xu, dl * xu);
        f2 Bv[NP], Cv[NP];
        rowB(buf, tt, Bv);
        rowC(buf, tt, Cv);
        f2 y0 = pk(0.f, 0.f), y1 = pk(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NP; j++) {
          hh[j] = fma2(abar2(dl2, A2[j]), hh[j], mul2(du2, Bv[j]));
          if (j & 1) y1 = fma2(Cv[j], hh[j], y1);
          else y0 = fma2(Cv[j], hh[j], y0);
        }
        ulonglong2* hs = hist + (tt + 1) * NQ * 32 + lane;
#pragma unroll
        for (int qq = 0; qq < NQ; qq++) hs[qq * 32] = make_ulonglong2(hh[2 * qq], hh[2 * qq + 1]);
        if constexpr (HAS_Z) {
          const f2 ys = add2(y0, y1);
          const float yv = fmaf(D_d, xu, chan_sum(f2lo(ys) + f2hi(ys)));
          const float dyt = sm_elem<TDy>(buf + LY::OFF_DY + tt * LY::DY_ROW, ch);
          const float zz = sm_elem<TIn>(buf + LY::OFF_Z + tt * LY::IN_ROW, ch);
          const float sg = sigmoidf_fast(zz);
          st_out(static_cast<TIn*>(p.dz) + i, dyt * yv * sg * fmaf(zz, 1.f - sg, 1.f), dv && owner);
        }
      }
      // the adjoint backwards through the sub-tile
#pragma unroll 2
      for (int tt = ns - 1; tt >= 0; tt--) {
        const int64_t t = t0 + tt;
        const float xu = sm_elem<TIn>(buf + LY::OFF_U + tt * LY::IN_ROW, ch);
        const float xr = sm_elem<TIn>(buf + LY::OFF_DR + tt * LY::IN_ROW, ch) + bias_d;
        const float dl = dlt[tt * CW + ch];
        float dyv = sm_elem<TDy>(buf + LY::OFF_DY + tt * LY::DY_ROW, ch);
        if constexpr (HAS_Z) dyv *= silu(sm_elem<TIn>(buf + LY::OFF_Z + tt * LY::IN_ROW, ch));
        const f2 dl2 = pk(dl, dl), dyv2 = pk(dyv, dyv), dlu2 = pk(dl * xu, dl * xu);
        f2 Bv[NP], Cv[NP];
        rowB(buf, tt, Bv);
        rowC(buf, tt, Cv);
        f2 vB[NP], vC[NP];  // this lane's terms of dB and dC for its states
        f2 dub0 = pk(0.f, 0.f), dub1 = pk(0.f, 0.f), dda0 = pk(0.f, 0.f), dda1 = pk(0.f, 0.f);
        const ulonglong2* hc = hist + (tt + 1) * NQ * 32 + lane;
        const ulonglong2* hq = hist + tt * NQ * 32 + lane;
#pragma unroll
        for (int qq = 0; qq < NQ; qq++) {
          const ulonglong2 c4 = hc[qq * 32];
          const ulonglong2 p4 = hq[qq * 32];
          const f2 ht[2] = {c4.x, c4.y};
          const f2 hp[2] = {p4.x, p4.y};
#pragma unroll
          for (int k = 0; k < 2; k++) {
            const int j = 2 * qq + k;
            const f2 a = abar2(dl2, A2[j]);
            lam[j] = fma2(Cv[j], dyv2, lam[j]);
            vC[j] = mul2(dyv2, ht[k]);
            vB[j] = mul2(lam[j], dlu2);
            const f2 lpa = mul2(lam[j], mul2(hp[k], a));
            if (k) {
              dub1 = fma2(lam[j], Bv[j], dub1);
              dda1 = fma2(lpa, A2[j], dda1);
            } else {
              dub0 = fma2(lam[j], Bv[j], dub0);
              dda0 = fma2(lpa, A2[j], dda0);
            }
            dAacc[j] = fma2(lpa, dl2, dAacc[j]);
            lam[j] = mul2(lam[j], a);
          }
        }
        const f2 dubs = add2(dub0, dub1), ddas = add2(dda0, dda1);
        const float dub = chan_sum(f2lo(dubs) + f2hi(dubs));
        const float dda = chan_sum(f2lo(ddas) + f2hi(ddas));
        // dL/d delta = sum_n lambda (h_prev Abar A + B u) = ln2 * dda + u * dub
        const float ddel = fmaf(kLn2, dda, xu * dub);
        const float dxr = ddel * sigmoidf_fast(xr);
        dbacc += dxr;
        dDacc = fmaf(dyv, xu, dDacc);
        const int64_t i = (b * L + t) * Dm + dc;
        st_out(static_cast<TIn*>(p.du) + i, fmaf(dyv, D_d, dl * dub), dv && owner);
        st_out(static_cast<TIn*>(p.ddelta_raw) + i, dxr, dv && owner);
        // Sum over the warp's channels (lanes with the same lane % SG). Element
        // 4 j + 2 k + c is the dB (c = 0) or dC (c = 1) term of state 2 j + k
        // of the lane's pair j; position 4 j + 2 k + c of v holds the element
        // of pair j ^ gp. At each stage (mask m, width w) a lane keeps w values
        // and adds its partner's other w. In the stages over the pair bits the
        // partners' orders differ exactly by w, so every lane keeps the lower
        // half; the last two stages (the bits of k and c) select. After them
        // lane l holds element l / SG.
        float v[2 * NS];
#pragma unroll
        for (int j = 0; j < NP; j++) {
          v[4 * j] = f2lo(vB[j]);
          v[4 * j + 1] = f2lo(vC[j]);
          v[4 * j + 2] = f2hi(vB[j]);
          v[4 * j + 3] = f2hi(vC[j]);
        }
#pragma unroll
        for (int m = 16, w = NS; w >= 4; m >>= 1, w >>= 1) {
#pragma unroll
          for (int e = 0; e < w; e++) v[e] += __shfl_xor_sync(0xffffffffu, v[e + w], m);
        }
#pragma unroll
        for (int m = 2 * SG, w = 2; m >= SG; m >>= 1, w >>= 1) {
          const bool up = (lane & m) != 0;
#pragma unroll
          for (int e = 0; e < w; e++) {
            const float keep = up ? v[e + w] : v[e];
            const float send = up ? v[e] : v[e + w];
            v[e] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
        }
        const int e = ch;  // 0 .. 2NS-1
        float* row = ((e & 1) ? p.dC : p.dB) + (b * L + t) * kDState + soff;
        atomicAdd(row + (e >> 1), v[0]);
      }
      __syncwarp();  // buffer s & 1 is refilled next iteration
    }
    // the adjoint leaving the segment: dh0 at the block's start, else back to
    // the share that holds the block's earlier sub-tiles
    if (q.sb == 0) {
      if (dv && p.dh0) {
#pragma unroll
        for (int j = 0; j < NP; j++) {
          p.dh0[(b * Dm + d) * kDState + sidx(j)] = f2lo(lam[j]);
          p.dh0[(b * Dm + d) * kDState + sidx(j) + 1] = f2hi(lam[j]);
        }
      }
    } else {
      float* dst = slot(p.ws_lam, q.u);
#pragma unroll
      for (int j = 0; j < NP; j++) {
        dst[2 * j] = f2lo(lam[j]);
        dst[2 * j + 1] = f2hi(lam[j]);
      }
      publish(p.flags_lam + q.u, (uint32_t)(nsub - q.sb));
    }
    // this segment's part of the sums over time (the other part, if the
    // block is cut, comes from the other share)
    if (dv) {
#pragma unroll
      for (int j = 0; j < NP; j++) {
        atomicAdd(p.dA + d * kDState + sidx(j), f2lo(dAacc[j]));
        atomicAdd(p.dA + d * kDState + sidx(j) + 1, f2hi(dAacc[j]));
      }
      if (owner) {
        if (p.dD) atomicAdd(p.dD + d, dDacc);
        if (p.dbias) atomicAdd(p.dbias + d, dbacc);
      }
    }
  };

  // ---- the jobs. A share of one segment runs its forward then its reverse
  // sweep. Otherwise, with n segments: the head's forward sweep (its state
  // goes to the next share), the whole blocks' forward sweeps (while the
  // previous share sweeps the block whose tail this share holds), the tail's
  // forward and reverse sweeps (its adjoint goes back to the previous share,
  // which waits for it), the whole blocks' reverse sweeps, and the head's
  // reverse sweep last (it waits for the next share's tail).
  for (int jb = 0; jb < 2 * nseg && !aborted; jb++) {
    int sgi, rev;
    if (nseg == 1) {
      sgi = 0, rev = jb;
    } else if (jb < nseg) {  // forward: head, whole blocks, tail
      sgi = jb, rev = 0;
    } else if (jb == nseg) {  // the tail's reverse sweep
      sgi = nseg - 1, rev = 1;
    } else if (jb < 2 * nseg - 1) {  // the whole blocks' reverse sweeps
      sgi = jb - nseg, rev = 1;
    } else {  // the head's reverse sweep
      sgi = 0, rev = 1;
    }
    const Seg q = segment(sgi);
    set_block(q.u);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();  // the previous job's staging is complete and read
    if (rev)
      rev_job(q);
    else
      fwd_job(q);
  }
  if (aborted && lane == 0) atomicOr(p.fault, kFaultTileWait);
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename TIn, typename TDy, int SG, bool HAS_Z, bool VEC>
cudaError_t launch_bwd_k(const BwdParams& p, cudaStream_t s) {
  const int smem = kBwdWarps * BwdLayout<TIn, TDy, SG>::SMEM;
  auto k = scan_bwd_kernel<TIn, TDy, SG, HAS_Z, VEC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = p.batch * (int64_t)p.ncblk;
  BwdParams q = p;
  q.nshares = blocks;
  if (p.flags_h) {
    // More blocks than warp slots: one CTA per slot, every warp an equal
    // share of all blocks' sub-tiles. A head's reverse sweep waits for a
    // later share, so all CTAs must be resident at once: a cooperative
    // launch, which fails rather than leaving a CTA unscheduled.
    int occ = 0, dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int coop = 0;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, 32 * kBwdWarps, smem)) != cudaSuccess) return e;
    const int64_t grid = (int64_t)occ * device_sm_count();
    const int64_t R = p.force_shares > 0 ? p.force_shares : grid * kBwdWarps;
    if (coop && occ > 0 && R < blocks * p.nsub && (p.force_shares > 0 || blocks > R) &&
        (R + kBwdWarps - 1) / kBwdWarps <= grid) {
      q.nshares = R;
      if ((e = cudaMemsetAsync(p.flags_h, 0, (size_t)blocks * 4, s)) != cudaSuccess) return e;
      if ((e = cudaMemsetAsync(p.flags_lam, 0, (size_t)blocks * 4, s)) != cudaSuccess) return e;
      void* args[] = {&q};
      e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k), dim3((unsigned)((R + kBwdWarps - 1) / kBwdWarps)),
                                      dim3(32 * kBwdWarps), args, (size_t)smem, s);
      if (e == cudaSuccess) return cudaSuccess;
      (void)cudaGetLastError();  // a cooperative launch that is refused: one warp per block instead
      q.nshares = blocks;
    }
  }
  k<<<(unsigned)((blocks + kBwdWarps - 1) / kBwdWarps), 32 * kBwdWarps, smem, s>>>(q);
  return cudaGetLastError();
}

template <typename TIn, typename TDy, int SG>
cudaError_t launch_bwd_sg(const BwdParams& p, cudaStream_t s) {
  // 16-byte copies need every staged row to start on a 16-byte boundary
  const bool vec = (p.dim * (int64_t)sizeof(TIn)) % 16 == 0 && (p.dim * (int64_t)sizeof(TDy)) % 16 == 0;
  if (p.z) return vec ? launch_bwd_k<TIn, TDy, SG, true, true>(p, s) : launch_bwd_k<TIn, TDy, SG, true, false>(p, s);
  return vec ? launch_bwd_k<TIn, TDy, SG, false, true>(p, s) : launch_bwd_k<TIn, TDy, SG, false, false>(p, s);
}

template <typename TIn, typename TDy>
cudaError_t launch_bwd_t(const BwdParams& p, int sg, cudaStream_t s) {
  return sg == 2 ? launch_bwd_sg<TIn, TDy, 2>(p, s) : launch_bwd_sg<TIn, TDy, 1>(p, s);
}

}  // namespace

size_t scan_bwd_checkpoint_bytes(int64_t batch, int64_t seqlen, int64_t dim, int sg) {
  const int64_t cw = 32 / sg;
  const int64_t nblk = batch * ((dim + cw - 1) / cw);
  const int64_t nsub = (seqlen + kSub - 1) / kSub;
  return (size_t)nblk * (size_t)nsub * 32 * (kDState / sg) * sizeof(float);
}

int64_t scan_bwd_subtiles(int64_t seqlen) { return (seqlen + kSub - 1) / kSub; }

// The hand-over area after the checkpoints: two flags per block (each array
// padded to 256 bytes), then two [blocks, 32 lanes, 16] fp32 slots.
size_t scan_bwd_handover_bytes(int64_t batch, int64_t dim, int sg) {
  const int64_t cw = 32 / sg;
  const int64_t nblk = batch * ((dim + cw - 1) / cw);
  return 2 * (size_t)((nblk * 4 + 255) / 256 * 256) + 2 * (size_t)nblk * 32 * kDState * sizeof(float);
}

cudaError_t launch_scan_bwd(const BwdParams& p, int sg, ss_dtype in_dtype, ss_dtype dy_dtype, cudaStream_t stream) {
  if (in_dtype == SS_BF16)
    return dy_dtype == SS_BF16 ? launch_bwd_t<__nv_bfloat16, __nv_bfloat16>(p, sg, stream)
                               : launch_bwd_t<__nv_bfloat16, float>(p, sg, stream);
  return dy_dtype == SS_BF16 ? launch_bwd_t<float, __nv_bfloat16>(p, sg, stream)
                             : launch_bwd_t<float, float>(p, sg, stream);
}

}  // namespace ssk
