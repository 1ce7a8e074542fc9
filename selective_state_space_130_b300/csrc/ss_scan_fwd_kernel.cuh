// Selective-scan (S6) forward kernel for sm_103a (template; instantiated per
// input/output dtype pair in ss_scan_fwd_<in>_<out>.cu).
//
// Work decomposition. A thread block is ONE warp that owns DC = 32/SG
// consecutive channels of one batch element over one chunk of the sequence.
// Each channel's 16-element fp32 state lives in registers of SG lanes (16/SG
// states each). Small one-warp blocks let the ~20k channels of a layer spread
// evenly over the 148 SMs in a single wave (about nine warps per SM).
//
// Data path per block. Tiles of kTile timesteps flow through a kStages-deep
// shared-memory ring: u, delta_raw, z ([kTile, DC] boxes) and the tile's B and
// C rows ([kTile, 16] boxes) arrive by TMA (cp.async.bulk.tensor), completion
// counted on one mbarrier per stage; the warp issues tile k+kStages-1 before it
// waits for tile k. bf16 B/C rows are converted once per tile into an fp32
// buffer that every channel of the block reads by broadcast. The warp then
// walks the tile token by token: delta = softplus(delta_raw + bias),
// Abar = 2^(delta * A * log2 e), h = Abar*h + (delta*u)*B, y = C.h + D*u,
// y *= silu(z). With SG > 1 the SG lanes of a channel take turns computing the
// per-token scalars (one token each) and exchange them by shuffle; the readout
// is reduce-scattered so each lane stores one token. Only y and the final
// state leave the chip: the fused, SRAM-resident scan of the Mamba pages
// (review page, method step 2; "Transformer时代终结？" section 二.3), laid out
// for B300 rather than translated.
//
// Long sequences are split into chunks so that enough warps run. A chunk's
// carry pair (P = prod Abar = exp(A * sum delta), S = state reached from a zero
// start) composes as (P1,S1) o (P2,S2) = (P1 P2, P2 S1 + S2) ("外文文献精读"
// section 2.2 block combination; mlqm.cn tutorial section 6 associativity).
// Chunks publish their pair to a workspace and resolve their incoming state by
// decoupled look-back over predecessors (a single-pass chained scan; tickets
// taken in launch order make every awaited predecessor a started block). A
// chunk that started from zero then recomputes its head from the true
// incoming state and stops once, for every state n, the carried-in part
// P_t,n * h_in,n is at most 2^-24 of the true state (for A <= 0 it only decays
// further), so the outputs equal the sequential recurrence up to fp32
// rounding.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace scan_detail {

constexpr int kTile = 32;    // timesteps per pipeline stage
constexpr int kStages = 3;   // TMA ring depth
constexpr float kStopRel = 5.9604645e-8f;  // 2^-24

constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagInclusive = 2u;
constexpr int kHeaderWords = 64;
constexpr uint32_t kHeaderMagic = 0x53535753u;  // header word 2: "this call used the workspace"

template <typename TIn, int SG>
struct Cfg {
  static constexpr int NS = kDState / SG;  // states per lane
  static constexpr int DC = 32 / SG;       // channels per block (one warp)
  static constexpr bool BF = sizeof(TIn) == 2;
  static constexpr int XB = kTile * DC * (int)sizeof(TIn);        // one u / delta_raw / z tile
  static constexpr int RB = kTile * kDState * (int)sizeof(TIn);   // one raw B or C tile
  static constexpr int OFF_U = 0, OFF_DR = XB, OFF_Z = 2 * XB, OFF_B = 3 * XB, OFF_C = 3 * XB + RB;
  static constexpr int STAGE = (3 * XB + 2 * RB + 127) & ~127;
  static constexpr int OFF_BCF = kStages * STAGE;                  // fp32 B|C of the current tile (bf16 only)
  static constexpr int BCF = BF ? 2 * kTile * kDState * 4 : 0;
  static constexpr int OFF_BAR = OFF_BCF + BCF;
  static constexpr int SMEM = OFF_BAR + kStages * 8 + 32 + 128;    // + alignment slack
};

// softplus(x) = log(1 + e^x), from w = e^x:
//   x > 20    : x (the correction log1p(e^-x) < 2.1e-9 is below half an ulp of x)
//   w < 1/16  : series w - w^2/2 + w^3/3 - w^4/4 + w^5/5 - w^6/6 (truncation < w^7/7)
//   otherwise : ln2 * log2(1 + w); 1 + w >= 1.0625 keeps the MUFU log2's absolute
//               error a small relative one
__device__ __forceinline__ float softplus_fast(float x) {
  const float w = ex2(x * kLog2e);
  float p = fmaf(w, -1.f / 6.f, 0.2f);
  p = fmaf(w, p, -0.25f);
  p = fmaf(w, p, 1.f / 3.f);
  p = fmaf(w, p, -0.5f);
  p = fmaf(w, p, 1.f);
  const float series = w * p;
  float lg;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(1.f + w));
  const float r = w < 0.0625f ? series : lg * kLn2;
  return x > 20.f ? x : r;
}

struct TokenScalars {
  float dl, du, post, gate;
};

template <int SG>
__device__ __forceinline__ float reduce_scatter(const float (&part)[SG], int s) {
  if constexpr (SG == 1) {
    return part[0];
  } else if constexpr (SG == 2) {
    const float keep = s ? part[1] : part[0];
    const float send = s ? part[0] : part[1];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
  } else {
    const bool hi = (s & 2) != 0;
    const float k0 = hi ? part[2] : part[0], k1 = hi ? part[3] : part[1];
    const float o0 = hi ? part[0] : part[2], o1 = hi ? part[1] : part[3];
    const float q0 = k0 + __shfl_xor_sync(0xffffffffu, o0, 2);
    const float q1 = k1 + __shfl_xor_sync(0xffffffffu, o1, 2);
    const bool lo = (s & 1) != 0;
    return (lo ? q1 : q0) + __shfl_xor_sync(0xffffffffu, lo ? q0 : q1, 1);
  }
}

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, bool CHUNKED>
__global__ void __launch_bounds__(32) scan_fwd_kernel(const __grid_constant__ ScanParams p,
                                                      const __grid_constant__ CUtensorMap tm_u,
                                                      const __grid_constant__ CUtensorMap tm_dr,
                                                      const __grid_constant__ CUtensorMap tm_z,
                                                      const __grid_constant__ CUtensorMap tm_b,
                                                      const __grid_constant__ CUtensorMap tm_c) {
  using K = Cfg<TIn, SG>;
  constexpr int NS = K::NS, DC = K::DC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
  const int lane = threadIdx.x;
  const int s = lane % SG;
  const int cw = lane / SG;  // channel within the block
  const int n0 = s * NS;

  // ---- which (batch, channel block, chunk) this block owns
  int vb = blockIdx.x;
  if constexpr (CHUNKED) {
    if (lane == 0) vb = (int)atomicAdd(p.ws_header, 1u);  // launch-order ticket
    vb = __shfl_sync(0xffffffffu, vb, 0);
  }
  if (lane == 0) {
    for (int i = 0; i < kStages; i++) mbar_init(&full[i], 1);
    fence_mbar_init();
    if (p.ws_header && vb == 0) p.ws_header[2] = kHeaderMagic;
  }
  __syncwarp();
  const int per_chunk = (int)p.batch * p.ncblk;
  const int chunk = CHUNKED ? vb / per_chunk : 0;
  const int rem = CHUNKED ? vb % per_chunk : vb;
  const int b = rem / p.ncblk, cb = rem % p.ncblk;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = CHUNKED ? min(L, t_begin + p.chunk_len) : L;
  const int n_tiles = (int)((t_end - t_begin + kTile - 1) / kTile);
  const int64_t d = (int64_t)cb * DC + cw;
  const bool dvalid = d < Dm;
  const int x0 = cb * DC;

  // ---- per-channel constants and the state
  float A2[NS], h[NS];
#pragma unroll
  for (int n = 0; n < NS; n++) {
    A2[n] = dvalid ? __ldg(p.A + d * kDState + n0 + n) * kLog2e : 0.f;
    h[n] = (dvalid && p.h0 && chunk == 0) ? __ldg(p.h0 + ((int64_t)b * Dm + d) * kDState + n0 + n) : 0.f;
  }
  const float bias_d = (dvalid && p.delta_bias) ? __ldg(p.delta_bias + d) : 0.f;
  const float D_d = (dvalid && p.D) ? __ldg(p.D + d) : 0.f;
  TOut* const yout = static_cast<TOut*>(p.y);

  if (TMA && lane == 0) {
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_dr);
    if (HAS_Z) tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
  }

  int g_issued = 0, g_done = 0;  // tiles issued / consumed (mbarrier phase bookkeeping)
  bool abort = false;

  // Issue the loads of the tile starting at t0 into the next ring slot.
  auto issue = [&](int64_t t0) {
    const int st = g_issued % kStages;
    uint8_t* base = smem + st * K::STAGE;
    if constexpr (TMA) {
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(&full[st], (HAS_Z ? 3 : 2) * K::XB + 2 * K::RB);
        tma_load_3d(base + K::OFF_U, &tm_u, x0, (int)t0, b, &full[st]);
        tma_load_3d(base + K::OFF_DR, &tm_dr, x0, (int)t0, b, &full[st]);
        if (HAS_Z) tma_load_3d(base + K::OFF_Z, &tm_z, x0, (int)t0, b, &full[st]);
        tma_load_3d(base + K::OFF_B, &tm_b, 0, (int)t0, b, &full[st]);
        tma_load_3d(base + K::OFF_C, &tm_c, 0, (int)t0, b, &full[st]);
        mbar_arrive(&full[st]);
      }
    } else {
      // plain loads with bounds checks (shapes no TMA descriptor can cover)
      const TIn* gu = static_cast<const TIn*>(p.u);
      const TIn* gdr = static_cast<const TIn*>(p.delta_raw);
      const TIn* gz = static_cast<const TIn*>(p.z);
      TIn* su = reinterpret_cast<TIn*>(base + K::OFF_U);
      TIn* sdr = reinterpret_cast<TIn*>(base + K::OFF_DR);
      TIn* sz = reinterpret_cast<TIn*>(base + K::OFF_Z);
      for (int i = lane; i < kTile * DC; i += 32) {
        const int tt = i / DC, c = i % DC;
        const int64_t t = t0 + tt, dd = (int64_t)x0 + c;
        TIn vu = from_f32<TIn>(0.f), vr = vu, vz = vu;
        if (t < L && dd < Dm) {
          const int64_t gi = ((int64_t)b * L + t) * Dm + dd;
          vu = gu[gi];
          vr = gdr[gi];
          if (HAS_Z) vz = gz[gi];
        }
        su[i] = vu;
        sdr[i] = vr;
        if (HAS_Z) sz[i] = vz;
      }
      const TIn* gB = static_cast<const TIn*>(p.B);
      const TIn* gC = static_cast<const TIn*>(p.C);
      TIn* sB = reinterpret_cast<TIn*>(base + K::OFF_B);
      TIn* sC = reinterpret_cast<TIn*>(base + K::OFF_C);
      for (int i = lane; i < kTile * kDState; i += 32) {
        const int64_t t = t0 + i / kDState;
        const bool ok = t < L;
        const int64_t gi = ((int64_t)b * L + (ok ? t : 0)) * kDState + i % kDState;
        sB[i] = ok ? gB[gi] : from_f32<TIn>(0.f);
        sC[i] = ok ? gC[gi] : from_f32<TIn>(0.f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
    }
    g_issued++;
  };

  // Wait for the next ring slot; returns the fp32 B|C base of the tile
  // (converted once here when the inputs are bf16).
  auto acquire = [&]() -> const float* {
    const int st = g_done % kStages;
    if (!abort && !mbar_wait(&full[st], (g_done / kStages) & 1)) {
      abort = true;
      atomicOr(p.fault, kFaultTileWait);
    }
    __syncwarp();
    const uint8_t* base = smem + st * K::STAGE;
    if constexpr (K::BF) {
      // lane r converts row r of B and of C
      const uint4* rb = reinterpret_cast<const uint4*>(base + K::OFF_B) + lane * 2;
      const uint4* rc = reinterpret_cast<const uint4*>(base + K::OFF_C) + lane * 2;
      float4* fb = reinterpret_cast<float4*>(smem + K::OFF_BCF) + lane * 4;
      float4* fc = reinterpret_cast<float4*>(smem + K::OFF_BCF + kTile * kDState * 4) + lane * 4;
#pragma unroll
      for (int q = 0; q < 2; q++) {
        const uint4 vb4 = rb[q], vc4 = rc[q];
        fb[2 * q] = make_float4(__uint_as_float(vb4.x << 16), __uint_as_float(vb4.x & 0xffff0000u),
                                __uint_as_float(vb4.y << 16), __uint_as_float(vb4.y & 0xffff0000u));
        fb[2 * q + 1] = make_float4(__uint_as_float(vb4.z << 16), __uint_as_float(vb4.z & 0xffff0000u),
                                    __uint_as_float(vb4.w << 16), __uint_as_float(vb4.w & 0xffff0000u));
        fc[2 * q] = make_float4(__uint_as_float(vc4.x << 16), __uint_as_float(vc4.x & 0xffff0000u),
                                __uint_as_float(vc4.y << 16), __uint_as_float(vc4.y & 0xffff0000u));
        fc[2 * q + 1] = make_float4(__uint_as_float(vc4.z << 16), __uint_as_float(vc4.z & 0xffff0000u),
                                    __uint_as_float(vc4.w << 16), __uint_as_float(vc4.w & 0xffff0000u));
      }
      __syncwarp();
      return reinterpret_cast<const float*>(smem + K::OFF_BCF);
    } else {
      return reinterpret_cast<const float*>(base + K::OFF_B);  // fp32 B then C, contiguous
    }
  };

  // Per-token scalars of token tt of the current tile (this lane's channel).
  auto scalars = [&](const uint8_t* base, int tt) -> TokenScalars {
    const TIn* su = reinterpret_cast<const TIn*>(base + K::OFF_U);
    const TIn* sdr = reinterpret_cast<const TIn*>(base + K::OFF_DR);
    const TIn* sz = reinterpret_cast<const TIn*>(base + K::OFF_Z);
    const float xu = to_f32(su[tt * DC + cw]);
    TokenScalars r;
    r.dl = softplus_fast(to_f32(sdr[tt * DC + cw]) + bias_d);
    r.du = r.dl * xu;
    r.post = D_d * xu;
    r.gate = HAS_Z ? silu(to_f32(sz[tt * DC + cw])) : 1.f;
    return r;
  };

  float ssum = 0.f;  // sum of delta over the tokens consumed in the current pass

  // One group of SG tokens starting at token tg of the tile; the first
  // `nvalid` tokens of the group are real (SG for full tiles).
  auto group = [&](const float* bcf, int tg, const TokenScalars& sc, int nvalid, TOut* yrow) {
    float dlv[SG], duv[SG];
#pragma unroll
    for (int j = 0; j < SG; j++) {
      if constexpr (SG == 1) {
        dlv[j] = sc.dl;
        duv[j] = sc.du;
      } else {
        const int src = (lane & ~(SG - 1)) | j;
        dlv[j] = __shfl_sync(0xffffffffu, sc.dl, src);
        duv[j] = __shfl_sync(0xffffffffu, sc.du, src);
      }
    }
    float part[SG];
#pragma unroll
    for (int j = 0; j < SG; j++) {
      part[j] = 0.f;
      if (j < nvalid) {
        const float4* bq = reinterpret_cast<const float4*>(bcf + (tg + j) * kDState + n0);
        const float4* cq = reinterpret_cast<const float4*>(bcf + kTile * kDState + (tg + j) * kDState + n0);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int q = 0; q < NS / 4; q++) {
          const float4 bv = bq[q], cv = cq[q];
          const float bb[4] = {bv.x, bv.y, bv.z, bv.w}, cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
          for (int k = 0; k < 4; k++) {
            const int n = 4 * q + k;
            const float a = ex2(dlv[j] * A2[n]);
            h[n] = fmaf(a, h[n], duv[j] * bb[k]);
            if (k & 1) acc1 = fmaf(cc[k], h[n], acc1);
            else acc0 = fmaf(cc[k], h[n], acc0);
          }
        }
        part[j] = acc0 + acc1;
        if constexpr (CHUNKED) ssum += dlv[j];
      }
    }
    const float yv = reduce_scatter<SG>(part, s);
    if (s < nvalid && dvalid) *yrow = from_f32<TOut>((yv + sc.post) * sc.gate);
  };

  // Process the acquired tile of `tlen` tokens starting at timestep t0.
  auto tile = [&](const float* bcf, int64_t t0, int tlen) {
    const uint8_t* base = smem + (g_done % kStages) * K::STAGE;
    TOut* yrow = yout + ((int64_t)b * L + t0 + s) * Dm + d;
    const int64_t ystep = (int64_t)SG * Dm;
    if (tlen == kTile) {
      TokenScalars sc = scalars(base, s);
#pragma unroll
      for (int tg = 0; tg < kTile; tg += SG) {
        TokenScalars nx = sc;
        if (tg + SG < kTile) nx = scalars(base, tg + SG + s);  // next group's scalars, ahead of time
        group(bcf, tg, sc, SG, yrow);
        yrow += ystep;
        sc = nx;
      }
    } else {
      for (int tg = 0; tg < tlen; tg += SG) {
        const int tt = tg + s;
        TokenScalars sc{0.f, 0.f, 0.f, 1.f};
        if (tt < tlen) sc = scalars(base, tt);
        group(bcf, tg, sc, min(SG, tlen - tg), yrow);
        yrow += ystep;
      }
    }
  };

  // Stream tiles [0, ntiles) of the chunk; with `stop_check`, stop after the
  // first tile at whose end the carried-in part is negligible. Loads issued
  // past the stop point are drained before returning.
  auto pass = [&](int ntiles, bool stop_check, const float* hin) {
    const int pre = min(kStages - 1, ntiles);
    for (int i = 0; i < pre; i++) issue(t_begin + (int64_t)i * kTile);
    for (int k = 0; k < ntiles; k++) {
      if (k + kStages - 1 < ntiles) issue(t_begin + (int64_t)(k + kStages - 1) * kTile);
      const float* bcf = acquire();
      const int64_t t0 = t_begin + (int64_t)k * kTile;
      tile(bcf, t0, (int)min((int64_t)kTile, t_end - t0));
      g_done++;
      if (stop_check && k + 1 < ntiles) {
        bool done = true;
#pragma unroll
        for (int n = 0; n < NS; n++) {
          const float carried = fabsf(ex2(A2[n] * ssum) * hin[n]);
          done = done && (A2[n] <= 0.f) && (carried <= kStopRel * fabsf(h[n]));
        }
        if (__all_sync(0xffffffffu, done || !dvalid) || abort) break;
      }
    }
    while (g_done < g_issued) {
      const int st = g_done % kStages;
      if (!abort && !mbar_wait(&full[st], (g_done / kStages) & 1)) {
        abort = true;
        atomicOr(p.fault, kFaultTileWait);
      }
      g_done++;
    }
  };

  pass(n_tiles, false, nullptr);

  float* hl_out = (dvalid && p.h_last) ? p.h_last + ((int64_t)b * Dm + d) * kDState + n0 : nullptr;
  if constexpr (!CHUNKED) {
    if (hl_out) {
#pragma unroll
      for (int n = 0; n < NS; n++) hl_out[n] = h[n];
    }
  } else {
    // ---- chunk carries: publish the local pair, look back, publish inclusive
    const int64_t tile_id = ((int64_t)b * p.ncblk + cb) * p.nchunks + chunk;
    uint32_t* flags = p.ws_header + kHeaderWords;
    float* carry_me = p.ws_carry + ((size_t)tile_id * DC + cw) * 48 + n0;
    if (chunk == 0) {
#pragma unroll
      for (int n = 0; n < NS; n++) carry_me[32 + n] = h[n];
    } else {
#pragma unroll
      for (int n = 0; n < NS; n++) {
        carry_me[n] = ex2(A2[n] * ssum);  // P = exp(A * sum delta)
        carry_me[16 + n] = h[n];          // S = state from a zero start
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_gpu(&flags[tile_id], chunk == 0 ? kFlagInclusive : kFlagAggregate);
    if (chunk == 0) return;

    float Pa[NS], Sa[NS];
#pragma unroll
    for (int n = 0; n < NS; n++) {
      Pa[n] = 1.f;
      Sa[n] = 0.f;
    }
    for (int j = chunk - 1; j >= 0; j--) {
      const int64_t pid = tile_id - (chunk - j);
      uint32_t f = 0;
      if (lane == 0) {
        f = ld_acquire_gpu(&flags[pid]);
        if (f == 0 && !abort) {
          const uint64_t tw = globaltimer();
          while ((f = ld_acquire_gpu(&flags[pid])) == 0) {
            if (globaltimer() - tw > kWaitNs) {
              atomicOr(p.fault, kFaultLookback);
              f = kFlagInclusive;  // give up: treat as resolved
              break;
            }
          }
        }
      }
      f = __shfl_sync(0xffffffffu, f, 0);
      const float* cp = p.ws_carry + ((size_t)pid * DC + cw) * 48 + n0;
      if (f == kFlagInclusive) {
#pragma unroll
        for (int n = 0; n < NS; n++) Sa[n] = fmaf(Pa[n], __ldcg(cp + 32 + n), Sa[n]);
        break;
      }
#pragma unroll
      for (int n = 0; n < NS; n++) {
        Sa[n] = fmaf(Pa[n], __ldcg(cp + 16 + n), Sa[n]);
        Pa[n] *= __ldcg(cp + n);
      }
    }
    // Sa is the true state entering this chunk
#pragma unroll
    for (int n = 0; n < NS; n++) {
      const float incl = fmaf(carry_me[n], Sa[n], h[n]);  // P_end * h_in + S_local
      carry_me[32 + n] = incl;
      if (hl_out && chunk == p.nchunks - 1) hl_out[n] = incl;
      h[n] = Sa[n];  // restart the head from the true incoming state
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_gpu(&flags[tile_id], kFlagInclusive);

    ssum = 0.f;
    pass(n_tiles, true, Sa);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  }
  return fn;
}

// 3-D map over a [batch, L, inner] row-major tensor with a [1, kTile, box_inner] box.
inline bool make_map(CUtensorMap* m, const void* ptr, size_t es, int64_t batch, int64_t L, int64_t inner,
                     int box_inner) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)inner * es, (cuuint64_t)L * inner * es};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, bool CHUNKED>
cudaError_t launch_t(const ScanParams& p, cudaStream_t stream) {
  using K = Cfg<TIn, SG>;
  auto kern = scan_fwd_kernel<TIn, TOut, SG, TMA, HAS_Z, CHUNKED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mu{}, mdr{}, mz{}, mb{}, mc{};
  if (TMA) {
    const size_t es = sizeof(TIn);
    if (!make_map(&mu, p.u, es, p.batch, p.seqlen, p.dim, K::DC) ||
        !make_map(&mdr, p.delta_raw, es, p.batch, p.seqlen, p.dim, K::DC) ||
        (HAS_Z && !make_map(&mz, p.z, es, p.batch, p.seqlen, p.dim, K::DC)) ||
        !make_map(&mb, p.B, es, p.batch, p.seqlen, kDState, kDState) ||
        !make_map(&mc, p.C, es, p.batch, p.seqlen, kDState, kDState))
      return cudaErrorInvalidValue;
  }
  const int64_t nblk = p.batch * (int64_t)p.ncblk * p.nchunks;
  kern<<<(unsigned)nblk, 32, K::SMEM, stream>>>(p, mu, mdr, mz, mb, mc);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int SG, bool TMA>
cudaError_t launch_z(const ScanParams& p, cudaStream_t stream) {
  const bool hz = p.z != nullptr, ch = p.nchunks > 1;
  if (hz)
    return ch ? launch_t<TIn, TOut, SG, TMA, true, true>(p, stream)
              : launch_t<TIn, TOut, SG, TMA, true, false>(p, stream);
  return ch ? launch_t<TIn, TOut, SG, TMA, false, true>(p, stream)
            : launch_t<TIn, TOut, SG, TMA, false, false>(p, stream);
}

template <typename TIn, typename TOut, int SG>
cudaError_t launch_sg(const ScanParams& p, bool tma, cudaStream_t stream) {
  return tma ? launch_z<TIn, TOut, SG, true>(p, stream) : launch_z<TIn, TOut, SG, false>(p, stream);
}

template <typename TIn, typename TOut>
cudaError_t launch_io(const ScanParams& p, int sg, bool tma, cudaStream_t stream) {
  switch (sg) {
    case 1: return launch_sg<TIn, TOut, 1>(p, tma, stream);
    case 2: return launch_sg<TIn, TOut, 2>(p, tma, stream);
    case 4: return launch_sg<TIn, TOut, 4>(p, tma, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace scan_detail

// One instantiation per (input, output) dtype pair, each in its own
// translation unit so the build compiles them in parallel.
cudaError_t scan_launch_bf16_bf16(const ScanParams& p, int sg, bool tma, cudaStream_t s);
cudaError_t scan_launch_bf16_f32(const ScanParams& p, int sg, bool tma, cudaStream_t s);
cudaError_t scan_launch_f32_bf16(const ScanParams& p, int sg, bool tma, cudaStream_t s);
cudaError_t scan_launch_f32_f32(const ScanParams& p, int sg, bool tma, cudaStream_t s);

}  // namespace ssk
