// Selective-scan (S6) forward kernel for sm_103a.
//
// Work decomposition. One thread block owns DC consecutive channels of one
// batch element over one chunk of the sequence. Each channel's 16-element
// fp32 state lives in registers of SG threads (16/SG states each). A producer
// warp streams tiles of kTile timesteps through a kStages-deep shared-memory
// ring: u, delta_raw, z tiles arrive by TMA (cp.async.bulk.tensor, completion
// counted on an mbarrier), and the B and C rows of the tile (shared by every
// channel) are converted once to fp32 by the producer. Consumer warps walk the
// tile token by token: delta = softplus(delta_raw + bias), Abar = 2^(delta*A*log2e),
// h = Abar*h + (delta*u)*B, y = C.h + D*u, y *= silu(z). Only y and the final
// state leave the chip. This is the hardware-aware, SRAM-resident scan the
// Mamba pages describe (review page, method step 2; "Transformer时代终结？"
// section 二.3 kernel fusion), laid out for B300 rather than translated.
//
// Long sequences are split into chunks so that enough warps run. A chunk's
// carry pair (P = prod Abar = exp(A * sum delta), S = state reached from a zero
// start) composes as (P1,S1) o (P2,S2) = (P1 P2, P2 S1 + S2) ("外文文献精读"
// section 2.2 block combination; tutorial section 6 associativity). Chunks
// publish their pair to a workspace and resolve their incoming state by
// decoupled look-back over predecessors (a single-pass chained scan). A chunk
// that started from zero then recomputes its head from the true incoming state
// and stops once, for every state n, the carried-in part P_t,n * h_in,n has
// fallen below 2^-24 of the true state (it only decays further for A <= 0), so
// the outputs equal the sequential recurrence up to fp32 rounding.
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {

__device__ unsigned int g_fault_word = 0;

namespace {

constexpr int kCW = 4;                    // consumer warps per block
constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kTile = 32;                 // timesteps per pipeline stage
constexpr int kStages = 4;
constexpr float kStopRel = 5.9604645e-8f;  // 2^-24

constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagInclusive = 2u;
constexpr int kHeaderWords = 64;

template <typename TIn, int SG>
struct Cfg {
  static constexpr int NS = kDState / SG;    // states per thread
  static constexpr int CPW = 32 / SG;        // channels per consumer warp
  static constexpr int DC = kCW * CPW;       // channels per block
  static constexpr int XB = kTile * DC * (int)sizeof(TIn);
  static constexpr int XB_AL = (XB + 1023) & ~1023;
  static constexpr int BCB = kTile * kDState * 4;
  static constexpr int STAGE = 3 * XB_AL + 2 * BCB;
  static constexpr int OFF_BAR = kStages * STAGE;
  static constexpr int SMEM = OFF_BAR + 2 * kStages * 8 + 64 + 1024;
};

struct Shared {  // small control block after the barriers
  int b, cb, chunk;
  volatile int approved;  // recompute tiles the producer may issue
  volatile int rec_stop;  // consumers are done recomputing
  volatile int abort;     // a bounded wait gave up
  uint32_t flag_seen;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory"); }
__device__ __forceinline__ bool consumer_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.and.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kCW * 32)
      : "memory");
  return r != 0;
}

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

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z>
__global__ void __launch_bounds__(kThreads, SG == 1 ? 2 : 3) scan_fwd_kernel(const __grid_constant__ ScanParams p,
                                                            const __grid_constant__ CUtensorMap tm_u,
                                                            const __grid_constant__ CUtensorMap tm_dr,
                                                            const __grid_constant__ CUtensorMap tm_z) {
  using K = Cfg<TIn, SG>;
  constexpr int NS = K::NS, DC = K::DC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
  uint64_t* empty = full + kStages;
  Shared* sh = reinterpret_cast<Shared*>(empty + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool chunked = p.nchunks > 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; i++) {
      mbar_init(&full[i], 32);   // 32 producer-lane arrivals (+ TMA bytes)
      mbar_init(&empty[i], kCW); // one arrival per consumer warp
    }
    fence_mbar_init();
    int vb = blockIdx.x;
    if (chunked) vb = (int)atomicAdd(p.ws_header, 1u);  // launch-order ticket
    const int per_chunk = (int)p.batch * p.ncblk;
    sh->chunk = vb / per_chunk;
    const int r = vb % per_chunk;
    sh->b = r / p.ncblk;
    sh->cb = r % p.ncblk;
    sh->approved = 0;
    sh->rec_stop = 0;
    sh->abort = 0;
  }
  __syncthreads();

  const int b = sh->b, cb = sh->cb, chunk = sh->chunk;
  const int64_t L = p.seqlen, Dm = p.dim;
  const int64_t t_begin = (int64_t)chunk * p.chunk_len;
  const int64_t t_end = min(L, t_begin + p.chunk_len);
  const int n_main = (int)((t_end - t_begin + kTile - 1) / kTile);
  const bool recompute = chunk > 0;
  const int64_t tile_id = ((int64_t)b * p.ncblk + cb) * p.nchunks + chunk;

  auto stage_ptr = [&](int st) { return smem + (size_t)st * K::STAGE; };

  // ======================================================== producer warp
  if (warp == kCW) {
    if (TMA && lane == 0) {
      tma_prefetch_desc(&tm_u);
      tma_prefetch_desc(&tm_dr);
      if (HAS_Z) tma_prefetch_desc(&tm_z);
    }
    auto produce = [&](int g, int64_t t0) {
      const int st = g % kStages;
      if (g >= kStages) {
        if (!sh->abort && !mbar_wait(&empty[st], ((g / kStages) - 1) & 1)) {
          sh->abort = 1;
          atomicOr(p.fault, kFaultTileWait);
        }
      }
      uint8_t* base = stage_ptr(st);
      TIn* xs_u = reinterpret_cast<TIn*>(base);
      TIn* xs_dr = reinterpret_cast<TIn*>(base + K::XB_AL);
      TIn* xs_z = reinterpret_cast<TIn*>(base + 2 * K::XB_AL);
      float* bs = reinterpret_cast<float*>(base + 3 * K::XB_AL);
      float* cs = bs + kTile * kDState;
      const int x0 = cb * DC;
      if constexpr (TMA) {
        if (lane == 0 && !sh->abort) {
          mbar_expect_tx(&full[st], (uint32_t)((HAS_Z ? 3 : 2) * K::XB));
          tma_load_3d(xs_u, &tm_u, x0, (int)t0, b, &full[st]);
          tma_load_3d(xs_dr, &tm_dr, x0, (int)t0, b, &full[st]);
          if (HAS_Z) tma_load_3d(xs_z, &tm_z, x0, (int)t0, b, &full[st]);
        }
      } else {
        // plain loads with bounds checks (shapes a TMA descriptor cannot cover)
        const TIn* gu = static_cast<const TIn*>(p.u);
        const TIn* gdr = static_cast<const TIn*>(p.delta_raw);
        const TIn* gz = static_cast<const TIn*>(p.z);
        for (int i = lane; i < kTile * DC; i += 32) {
          const int tt = i / DC, c = i % DC;
          const int64_t t = t0 + tt, d = (int64_t)x0 + c;
          TIn vu = from_f32<TIn>(0.f), vr = vu, vz = vu;
          if (t < L && d < Dm) {
            const int64_t gi = ((int64_t)b * L + t) * Dm + d;
            vu = gu[gi];
            vr = gdr[gi];
            if (HAS_Z) vz = gz[gi];
          }
          xs_u[i] = vu;
          xs_dr[i] = vr;
          if (HAS_Z) xs_z[i] = vz;
        }
      }
      // B and C rows of this tile, converted once to fp32
      for (int r = lane; r < kTile; r += 32) {
        const int64_t t = t0 + r;
        float4* bo = reinterpret_cast<float4*>(bs + r * kDState);
        float4* co = reinterpret_cast<float4*>(cs + r * kDState);
        if (t < L) {
          const int64_t row = ((int64_t)b * L + t) * kDState;
          if constexpr (sizeof(TIn) == 2) {
            const uint4* gb = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.B) + row);
            const uint4* gc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.C) + row);
#pragma unroll
            for (int q = 0; q < 2; q++) {
              const uint4 vb = __ldg(gb + q), vc = __ldg(gc + q);
              const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w}, wc[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
              for (int k = 0; k < 2; k++) {
                bo[q * 2 + k] = make_float4(__uint_as_float(wb[2 * k] << 16), __uint_as_float(wb[2 * k] & 0xffff0000u),
                                            __uint_as_float(wb[2 * k + 1] << 16),
                                            __uint_as_float(wb[2 * k + 1] & 0xffff0000u));
                co[q * 2 + k] = make_float4(__uint_as_float(wc[2 * k] << 16), __uint_as_float(wc[2 * k] & 0xffff0000u),
                                            __uint_as_float(wc[2 * k + 1] << 16),
                                            __uint_as_float(wc[2 * k + 1] & 0xffff0000u));
              }
            }
          } else {
            const float4* gb = reinterpret_cast<const float4*>(static_cast<const float*>(p.B) + row);
            const float4* gc = reinterpret_cast<const float4*>(static_cast<const float*>(p.C) + row);
#pragma unroll
            for (int q = 0; q < 4; q++) {
              bo[q] = __ldg(gb + q);
              co[q] = __ldg(gc + q);
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; q++) bo[q] = co[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      mbar_arrive(&full[st]);
    };

    int g = 0;
    for (int k = 0; k < n_main; k++, g++) produce(g, t_begin + (int64_t)k * kTile);
    if (recompute) {
      const uint64_t tw = globaltimer();
      for (int j = 0; j < n_main;) {
        const int stop = sh->rec_stop;
        __threadfence_block();
        const int appr = sh->approved;
        if (j < appr) {
          produce(g, t_begin + (int64_t)j * kTile);
          g++;
          j++;
        } else if (stop || sh->abort) {
          break;
        } else if (globaltimer() - tw > kWaitNs) {
          sh->abort = 1;
          atomicOr(p.fault, kFaultTileWait);
          break;
        }
      }
    }
    return;
  }

  // ======================================================== consumer warps
  constexpr int CPW = K::CPW;
  const int s = lane % SG;
  const int cw = warp * CPW + lane / SG;  // channel within block
  const int64_t d = (int64_t)cb * DC + cw;
  const bool dvalid = d < Dm;
  const int n0 = s * NS;

  float A2[NS], h[NS];
#pragma unroll
  for (int n = 0; n < NS; n++) {
    A2[n] = dvalid ? p.A[d * kDState + n0 + n] * kLog2e : 0.f;
    h[n] = (dvalid && p.h0 && chunk == 0) ? p.h0[((int64_t)b * Dm + d) * kDState + n0 + n] : 0.f;
  }
  const float bias_d = (dvalid && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const float D_d = (dvalid && p.D) ? p.D[d] : 0.f;
  TOut* yout = static_cast<TOut*>(p.y);

  int g = 0;  // global tile counter (matches the producer's)
  float ssum = 0.f;  // sum of delta over the timesteps consumed in this pass

  // Consume one tile starting at timestep t0 with tlen valid timesteps.
  auto consume = [&](int gg, int64_t t0, int tlen, bool store) {
    const int st = gg % kStages;
    if (!sh->abort && !mbar_wait(&full[st], (gg / kStages) & 1)) {
      sh->abort = 1;
      atomicOr(p.fault, kFaultTileWait);
    }
    const uint8_t* base = stage_ptr(st);
    const TIn* xs_u = reinterpret_cast<const TIn*>(base);
    const TIn* xs_dr = reinterpret_cast<const TIn*>(base + K::XB_AL);
    const TIn* xs_z = reinterpret_cast<const TIn*>(base + 2 * K::XB_AL);
    const float* bs = reinterpret_cast<const float*>(base + 3 * K::XB_AL);
    const float* cs = bs + kTile * kDState;
    const int64_t row0 = (int64_t)b * L + t0;
#pragma unroll 2
    for (int tg = 0; tg < tlen; tg += SG) {
      const int tt = tg + s;
      float dl = 0.f, du = 0.f, post = 0.f, gate = 1.f;
      if (tt < tlen) {
        const float xu = to_f32(xs_u[tt * DC + cw]);
        dl = softplus(to_f32(xs_dr[tt * DC + cw]) + bias_d);
        du = dl * xu;
        post = D_d * xu;
        if (HAS_Z) gate = silu(to_f32(xs_z[tt * DC + cw]));
      }
      float dlv[SG], duv[SG];
#pragma unroll
      for (int j = 0; j < SG; j++) {
        if constexpr (SG == 1) {
          dlv[j] = dl;
          duv[j] = du;
        } else {
          const int src = (lane & ~(SG - 1)) | j;
          dlv[j] = __shfl_sync(0xffffffffu, dl, src);
          duv[j] = __shfl_sync(0xffffffffu, du, src);
        }
      }
      float part[SG];
#pragma unroll
      for (int j = 0; j < SG; j++) {
        part[j] = 0.f;
        if (tg + j < tlen) {
          const float4* bq = reinterpret_cast<const float4*>(bs + (tg + j) * kDState + n0);
          const float4* cq = reinterpret_cast<const float4*>(cs + (tg + j) * kDState + n0);
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
          ssum += dlv[j];
        }
      }
      const float yv = reduce_scatter<SG>(part, s);
      if (store && tt < tlen && dvalid) yout[(row0 + tt) * Dm + d] = from_f32<TOut>((yv + post) * gate);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  };

  // ---- main pass over the chunk
  for (int k = 0; k < n_main; k++, g++) {
    const int64_t t0 = t_begin + (int64_t)k * kTile;
    consume(g, t0, (int)(t_end - t0 < kTile ? t_end - t0 : kTile), true);
  }

  float* hl_out = (dvalid && p.h_last) ? p.h_last + ((int64_t)b * Dm + d) * kDState + n0 : nullptr;
  if (!chunked) {
    if (hl_out) {
#pragma unroll
      for (int n = 0; n < NS; n++) hl_out[n] = h[n];
    }
    return;
  }

  // ---- chunk carries: publish, look back, publish inclusive
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
  consumer_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release_gpu(&flags[tile_id], chunk == 0 ? kFlagInclusive : kFlagAggregate);
  }
  if (chunk == 0) {
    if (hl_out && p.nchunks == 1) {
#pragma unroll
      for (int n = 0; n < NS; n++) hl_out[n] = h[n];
    }
    return;
  }

  float Pa[NS], Sa[NS];
#pragma unroll
  for (int n = 0; n < NS; n++) {
    Pa[n] = 1.f;
    Sa[n] = 0.f;
  }
  for (int j = chunk - 1; j >= 0; j--) {
    const int64_t pid = tile_id - (chunk - j);
    if (threadIdx.x == 0) {
      uint32_t f = ld_acquire_gpu(&flags[pid]);
      if (f == 0 && !sh->abort) {
        const uint64_t tw = globaltimer();
        while ((f = ld_acquire_gpu(&flags[pid])) == 0) {
          if (globaltimer() - tw > kWaitNs) {
            sh->abort = 1;
            atomicOr(p.fault, kFaultLookback);
            f = kFlagInclusive;  // give up: treat as resolved
            break;
          }
        }
      }
      sh->flag_seen = f;
    }
    consumer_sync();
    const uint32_t f = sh->flag_seen;
    const float* cp = p.ws_carry + ((size_t)pid * DC + cw) * 48 + n0;
    if (f == kFlagInclusive) {
#pragma unroll
      for (int n = 0; n < NS; n++) Sa[n] = fmaf(Pa[n], __ldcg(cp + 32 + n), Sa[n]);
      consumer_sync();
      break;
    }
#pragma unroll
    for (int n = 0; n < NS; n++) {
      Sa[n] = fmaf(Pa[n], __ldcg(cp + 16 + n), Sa[n]);
      Pa[n] *= __ldcg(cp + n);
    }
    consumer_sync();
  }
  // Sa is now the true state entering this chunk
  float hin[NS];
#pragma unroll
  for (int n = 0; n < NS; n++) {
    hin[n] = Sa[n];
    const float incl = fmaf(carry_me[n], hin[n], h[n]);  // P_end * h_in + S_local
    carry_me[32 + n] = incl;
    if (hl_out && chunk == p.nchunks - 1) hl_out[n] = incl;
  }
  __threadfence();
  consumer_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release_gpu(&flags[tile_id], kFlagInclusive);
    sh->approved = min(kStages, n_main);
    __threadfence_block();
  }

  // ---- head recompute from the true incoming state
  bool can_stop = true;
#pragma unroll
  for (int n = 0; n < NS; n++) {
    h[n] = hin[n];
    if (A2[n] > 0.f) can_stop = false;  // growing modes: never truncate
  }
  ssum = 0.f;
  int j = 0;
  for (; j < n_main; j++, g++) {
    const int64_t t0 = t_begin + (int64_t)j * kTile;
    consume(g, t0, (int)(t_end - t0 < kTile ? t_end - t0 : kTile), true);
    bool done = can_stop;
    if (done) {
#pragma unroll
      for (int n = 0; n < NS; n++) {
        const float carried = fabsf(ex2(A2[n] * ssum) * hin[n]);
        done = done && (carried <= kStopRel * fabsf(h[n]));
      }
    }
    if (!dvalid) done = true;
    done = consumer_and(done) || sh->abort;
    if (done || j + 1 == n_main) {
      j++;
      g++;
      break;
    }
    if (threadIdx.x == 0) {
      sh->approved = min(j + 1 + kStages, n_main);
      __threadfence_block();
    }
  }
  // stop the producer, then drain the tiles it already issued
  if (threadIdx.x == 0) {
    __threadfence_block();
    sh->rec_stop = 1;
  }
  consumer_sync();
  const int issued = sh->approved;
  for (; j < issued; j++, g++) {
    const int st = g % kStages;
    if (!sh->abort && !mbar_wait(&full[st], (g / kStages) & 1)) {
      sh->abort = 1;
      atomicOr(p.fault, kFaultTileWait);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

template <typename TIn>
bool make_map(CUtensorMap* m, const void* ptr, int64_t batch, int64_t L, int64_t D, int box_c);

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
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

template <typename TIn>
bool make_map(CUtensorMap* m, const void* ptr, int64_t batch, int64_t L, int64_t D, int box_c) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = sizeof(TIn);
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)L * D * es};
  cuuint32_t box[3] = {(cuuint32_t)box_c, (cuuint32_t)kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      sizeof(TIn) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z>
cudaError_t launch_t(const ScanParams& p, cudaStream_t stream) {
  using K = Cfg<TIn, SG>;
  auto kern = scan_fwd_kernel<TIn, TOut, SG, TMA, HAS_Z>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mu{}, mdr{}, mz{};
  if (TMA) {
    if (!make_map<TIn>(&mu, p.u, p.batch, p.seqlen, p.dim, K::DC) ||
        !make_map<TIn>(&mdr, p.delta_raw, p.batch, p.seqlen, p.dim, K::DC) ||
        (HAS_Z && !make_map<TIn>(&mz, p.z, p.batch, p.seqlen, p.dim, K::DC)))
      return cudaErrorInvalidValue;
  }
  const int64_t nblk = p.batch * (int64_t)p.ncblk * p.nchunks;
  kern<<<(unsigned)nblk, kThreads, K::SMEM, stream>>>(p, mu, mdr, mz);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int SG>
cudaError_t launch_sg(const ScanParams& p, bool tma, cudaStream_t stream) {
  const bool hz = p.z != nullptr;
  if (tma) return hz ? launch_t<TIn, TOut, SG, true, true>(p, stream) : launch_t<TIn, TOut, SG, true, false>(p, stream);
  return hz ? launch_t<TIn, TOut, SG, false, true>(p, stream) : launch_t<TIn, TOut, SG, false, false>(p, stream);
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

}  // namespace

int scan_channels_per_block(int sg) { return kCW * (32 / sg); }
int scan_tile_len() { return kTile; }
int scan_header_words() { return kHeaderWords; }

unsigned int* device_fault_word() {
  static unsigned int* ptr = nullptr;
  static int dev_cached = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (!ptr || dev != dev_cached) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fault_word) != cudaSuccess) return nullptr;
    ptr = static_cast<unsigned int*>(a);
    dev_cached = dev;
  }
  return ptr;
}

cudaError_t launch_scan_fwd(const ScanParams& p, const ScanPlan& plan, ss_dtype in_dtype, ss_dtype out_dtype,
                            bool use_tma, cudaStream_t stream) {
  if (in_dtype == SS_BF16) {
    return out_dtype == SS_BF16 ? launch_io<__nv_bfloat16, __nv_bfloat16>(p, plan.sg, use_tma, stream)
                                : launch_io<__nv_bfloat16, float>(p, plan.sg, use_tma, stream);
  }
  return out_dtype == SS_BF16 ? launch_io<float, __nv_bfloat16>(p, plan.sg, use_tma, stream)
                              : launch_io<float, float>(p, plan.sg, use_tma, stream);
}

}  // namespace ssk
