// Selective-scan (S6) forward kernel for sm_103a (template; instantiated per
// input/output dtype pair in ss_scan_fwd_<in>_<out>.cu).
//
// What a thread computes. A CTA of kWarps warps owns CC consecutive channels
// of one batch element (a "channel block"); each warp owns DC = 32/SG of them.
// With SG = 1 each lane owns one channel and all 16 of its fp32 states; with
// SG = 2 two lanes share a channel, 8 states each. Per token a channel's
// delta = softplus(delta_raw + bias), Abar = 2^(delta * A * log2 e),
// h = Abar*h + (delta*u)*B, y = C.h + D*u and y *= silu(z): the fused,
// SRAM-resident scan the Mamba pages describe (review page, method step 2;
// "Transformer时代终结？" section 二.3), laid out for B300. The state update runs
// on packed f32x2 FMUL2/FFMA2 (two states per instruction); the exponentials
// run on the MUFU pipe. On B300 these two pipes, not HBM, bound the exact fp32
// recurrence.
//
// Data path. The CTA streams tiles of TILE timesteps through a two-stage ring
// in shared memory: u, delta_raw, z ([TILE, CC] boxes) and the tile's B and C
// rows ([TILE, 16]) arrive by TMA (cp.async.bulk.tensor), issued a tile ahead
// by a fifth warp that computes nothing (issuing five bulk loads takes several
// hundred cycles, which a compute warp would make its CTA wait for at the next
// barrier), with completion counted on one mbarrier per stage. bf16 B/C rows
// are widened once per tile into fp32 (each compute warp a quarter) and read by
// broadcast. One CTA-wide barrier per tile orders the widening and frees the
// stage the next load overwrites. Only y and the final state leave the chip.
//
// Work split (ScanMode), in units of (channel block, tile):
//  - static: one CTA per channel block, the whole sequence.
//  - stream-K: the (channel block, tile) space, block-major, is cut into
//    nworkers equal contiguous ranges, at least one block long each, so a range
//    holds at most one partial block at either end. A CTA first runs the head
//    of the block its range ends in (from that block's initial state) and hands
//    the state at its range end to the next CTA, then runs the rest of its
//    range in order; the first segment, when it starts inside a block, waits
//    for the state the previous CTA handed over (almost always already there).
//  - chunked (long sequences, few channel blocks): each block's sequence is
//    cut into chunks run by different CTAs. A chunk's carry pair
//    (P = prod Abar = exp(A * sum delta), S = state reached from zero) composes
//    as (P1,S1) o (P2,S2) = (P1 P2, P2 S1 + S2) ("外文文献精读" section 2.2;
//    mlqm.cn tutorial section 6). Chunks publish their pair and resolve their
//    incoming state by decoupled look-back, then recompute their head from the
//    true state until, for every state of every channel of the block, the
//    carried-in part P_t,n * h_in,n is at most 2^-24 of h_t,n (for A <= 0 it only
//    decays further): the outputs equal the sequential recurrence up to fp32
//    rounding.
// CTAs take their worker index from a ticket counter in launch order, so a CTA
// only ever waits for CTAs that have already started; every wait is bounded
// (p.wait_ns) and reports a timeout through the fault word.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace scan_detail {

constexpr int kWarps = 4;    // compute warps per CTA (one per SM sub-partition)
constexpr int kThreads = 32 * (kWarps + 1);  // plus one warp that issues the tile loads
constexpr int kStages = 2;   // TMA ring depth (the next tile loads while one is computed)
constexpr float kStopRel = 5.9604645e-8f;  // 2^-24

constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagInclusive = 2u;
constexpr uint32_t kFlagHanded = 1u;
constexpr int kHeaderWords = 64;
constexpr uint32_t kHeaderMagic = 0x53535753u;  // header word 2: "this call used the workspace"

template <typename TIn, int SG>
struct Cfg {
  static constexpr int NS = kDState / SG;  // states per lane
  static constexpr int NP = NS / 2;        // packed state pairs per lane
  static constexpr int DC = 32 / SG;       // channels per warp
  static constexpr int CC = kWarps * DC;   // channels per CTA (channel block)
  static constexpr bool BF = sizeof(TIn) == 2;
  static constexpr int TILE = BF ? 64 : 32;                          // timesteps per tile
  static constexpr int XB = TILE * CC * (int)sizeof(TIn);           // one u / delta_raw / z tile
  static constexpr int RB = TILE * kDState * (int)sizeof(TIn);      // one raw B or C tile
  static constexpr int OFF_U = 0, OFF_DR = XB, OFF_Z = 2 * XB, OFF_B = 3 * XB, OFF_C = 3 * XB + RB;
  static constexpr int STAGE = (3 * XB + 2 * RB + 127) & ~127;
  // fp32 B|C per stage (bf16 inputs): row t holds B[t][16] then C[t][16]
  static constexpr int BCF = BF ? TILE * 2 * kDState * 4 : 0;
  static constexpr int OFF_BCF = kStages * STAGE;
  static constexpr int OFF_BAR = OFF_BCF + kStages * BCF;
  static constexpr int SMEM = OFF_BAR + kStages * 8 + 128;           // + base alignment slack
};

// Widen this thread's share of a bf16 B and C tile ([TILE][16] each,
// contiguous) into the fp32 [TILE][B 16 | C 16] layout.
template <int TILE>
__device__ __forceinline__ void widen_bc(const uint8_t* raw_b, float* bcf, int tid) {
  // one item = 4 consecutive bf16 of B or C (8 bytes) -> 16 bytes of fp32
  constexpr int ITEMS = 2 * TILE * kDState / 4;
  constexpr int PER = ITEMS / (32 * kWarps);
  static_assert(ITEMS % (32 * kWarps) == 0, "widening share");
  const uint2* src = reinterpret_cast<const uint2*>(raw_b);
#pragma unroll
  for (int k = 0; k < PER; k++) {
    const int i = k * 32 * kWarps + tid;  // item i: tensor i / (TILE*4), row (i / 4) % TILE, quarter i % 4
    const int which = i / (TILE * 4);
    const int rem = i - which * TILE * 4;
    const int row = rem >> 2, qtr = rem & 3;
    const uint2 v = src[i];
    reinterpret_cast<float4*>(bcf + row * 32 + which * 16)[qtr] =
        make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                    __uint_as_float(v.y & 0xffff0000u));
  }
}

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, int MODE>
__global__ void __launch_bounds__(kThreads, 1) scan_fwd_kernel(const __grid_constant__ ScanParams p,
                                                                  const __grid_constant__ CUtensorMap tm_u,
                                                                  const __grid_constant__ CUtensorMap tm_dr,
                                                                  const __grid_constant__ CUtensorMap tm_z,
                                                                  const __grid_constant__ CUtensorMap tm_b,
                                                                  const __grid_constant__ CUtensorMap tm_c) {
  using K = Cfg<TIn, SG>;
  constexpr int NS = K::NS, NP = K::NP, DC = K::DC, CC = K::CC, TILE = K::TILE;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // 128-byte aligned base, derived from the shared array by pointer arithmetic
  // only (a round trip through an integer would hide from the compiler that
  // every tile access is a shared-memory access)
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
  __shared__ uint32_t s_wid;
  __shared__ uint32_t s_flag;
  const bool producer = warp == kWarps;  // the load-issuing warp
  const int s = lane % SG;                // which part of the channel's states this lane holds
  const int cw = lane / SG;               // channel within the warp
  const int cb = producer ? 0 : warp * DC + cw;  // channel within the CTA's block
  const int n0 = s * NS;
  const int tid_issue = kWarps * 32;      // the thread that issues the tile loads

  // ---- worker index (launch-order ticket in the split modes)
  if (tid == 0) {
    s_wid = MODE == kModeStatic ? blockIdx.x : atomicAdd(p.ws_header, 1u);
    for (int i = 0; i < kStages; i++) mbar_init(&full[i], 1);
    fence_mbar_init();
    if (TMA) {
      tma_prefetch_desc(&tm_u);
      tma_prefetch_desc(&tm_dr);
      if (HAS_Z) tma_prefetch_desc(&tm_z);
      tma_prefetch_desc(&tm_b);
      tma_prefetch_desc(&tm_c);
    }
  }
  __syncthreads();
  const int64_t wid = s_wid;
  if (wid >= p.nworkers) return;  // CTA-uniform
  if (tid == 0 && p.ws_header && wid == 0) p.ws_header[2] = kHeaderMagic;

  const int64_t T = p.tiles_per_blk, L = p.seqlen, Dm = p.dim;
  const int ncblk = p.ncblk;
  const uint64_t wait_ns = p.wait_ns;

  // ---- the worker's steps: step q runs tile j of channel block blk
  int64_t r0 = 0, zs = 0, zlen = 0, af = 0, nfull = 0, nsteps = 0;  // stream-K
  int64_t cblk = 0, c = 0, j0 = 0, nk = 0;                          // chunked
  if constexpr (MODE == kModeStatic) {
    nsteps = T;
  } else if constexpr (MODE == kModeStreamK) {
    const int64_t total = p.nblk * T;
    r0 = wid * total / p.nworkers;
    const int64_t r1 = (wid + 1) * total / p.nworkers;
    const int64_t tail = r1 % T;  // tiles of the last block inside the range
    if (tail != 0) {
      zs = r1 - tail;
      zlen = tail;
    } else {
      zs = r1;
    }
    const int64_t head = r0 % T;
    af = head != 0 ? r0 - head + T : r0;  // first block start at or after r0
    nfull = zs - af;                     // tiles of whole blocks
    nsteps = r1 - r0;
  } else {
    c = wid / p.nblk;
    cblk = wid % p.nblk;
    j0 = c * p.chunk_tiles;
    nk = min(T, j0 + p.chunk_tiles) - j0;
    nsteps = c == 0 ? nk : 2 * nk;  // chunks after the first recompute their head
  }
  // Step cursor: step q runs tile j of channel block blk from ring slot st
  // (mbarrier phase ph). Advancing costs a compare and an add; the divisions
  // that place a cursor happen only where a new segment or block begins.
  struct Cursor {
    int64_t q, blk, j;
    int b, x0, st;
    uint32_t ph;
  };
  auto place = [&](Cursor& cu) {  // (blk, j) and the block's coordinates for step cu.q
    if constexpr (MODE == kModeStatic) {
      cu.blk = wid;
      cu.j = cu.q;
    } else if constexpr (MODE == kModeStreamK) {
      // the head of the last block (handed over to the next CTA), then the
      // whole blocks, then the first segment, which waits for the previous
      // CTA's hand-over: with ranges of at least one block that hand-over is
      // already done by the time this CTA gets there
      const int64_t q = cu.q;
      const int64_t g = q < zlen ? zs + q : (q < zlen + nfull ? af + (q - zlen) : r0 + (q - zlen - nfull));
      cu.blk = g / T;
      cu.j = g - cu.blk * T;
    } else {
      cu.blk = cblk;
      cu.j = j0 + (cu.q < nk ? cu.q : cu.q - nk);
    }
    cu.b = (int)(cu.blk / ncblk);
    cu.x0 = (int)(cu.blk - (int64_t)cu.b * ncblk) * CC;
  };
  auto advance = [&](Cursor& cu) {
    cu.q++;
    if (++cu.st == kStages) {
      cu.st = 0;
      cu.ph ^= 1u;
    }
    bool jump = false;
    if constexpr (MODE == kModeStreamK) jump = cu.q == zlen || cu.q == zlen + nfull;
    if constexpr (MODE == kModeChunked) jump = cu.q == nk;
    if (jump) {
      place(cu);
    } else if (++cu.j == T) {
      cu.j = 0;
      cu.blk++;
      cu.x0 += CC;
      if (cu.x0 >= ncblk * CC) {
        cu.x0 = 0;
        cu.b++;
      }
    }
  };
  Cursor cc{0, 0, 0, 0, 0, 0, 0u};  // the step being run
  place(cc);

  // ---- tile loads
  // TMA: one thread issues the five boxes of a step into its ring slot
  auto issue_tma = [&](const Cursor& cu) {
    uint8_t* base = smem + cu.st * K::STAGE;
    const int y0 = (int)(cu.j * TILE);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(&full[cu.st], (HAS_Z ? 3 : 2) * K::XB + 2 * K::RB);
    tma_load_3d(base + K::OFF_U, &tm_u, cu.x0, y0, cu.b, &full[cu.st]);
    tma_load_3d(base + K::OFF_DR, &tm_dr, cu.x0, y0, cu.b, &full[cu.st]);
    if (HAS_Z) tma_load_3d(base + K::OFF_Z, &tm_z, cu.x0, y0, cu.b, &full[cu.st]);
    tma_load_3d(base + K::OFF_B, &tm_b, 0, y0, cu.b, &full[cu.st]);
    tma_load_3d(base + K::OFF_C, &tm_c, 0, y0, cu.b, &full[cu.st]);
    mbar_arrive(&full[cu.st]);
  };
  // plain loads with bounds checks (shapes no TMA descriptor can cover): the
  // whole CTA stages the step's tile synchronously
  auto load_plain = [&](const Cursor& cu) {
    uint8_t* base = smem + cu.st * K::STAGE;
    const int64_t y0 = cu.j * TILE;
    const TIn* gu = static_cast<const TIn*>(p.u);
    const TIn* gdr = static_cast<const TIn*>(p.delta_raw);
    const TIn* gz = static_cast<const TIn*>(p.z);
    TIn* su = reinterpret_cast<TIn*>(base + K::OFF_U);
    TIn* sdr = reinterpret_cast<TIn*>(base + K::OFF_DR);
    TIn* sz = reinterpret_cast<TIn*>(base + K::OFF_Z);
    for (int i = tid; i < TILE * CC; i += kThreads) {
      const int tt = i / CC, ch = i % CC;
      const int64_t t = y0 + tt, dd = (int64_t)cu.x0 + ch;
      TIn vu = from_f32<TIn>(0.f), vr = vu, vz = vu;
      if (t < L && dd < Dm) {
        const int64_t gi = ((int64_t)cu.b * L + t) * Dm + dd;
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
    for (int i = tid; i < TILE * kDState; i += kThreads) {
      const int64_t t = y0 + i / kDState;
      const bool ok = t < L;
      const int64_t gi = ((int64_t)cu.b * L + (ok ? t : 0)) * kDState + i % kDState;
      sB[i] = ok ? gB[gi] : from_f32<TIn>(0.f);
      sC[i] = ok ? gC[gi] : from_f32<TIn>(0.f);
    }
  };

  bool abort = false;  // CTA-uniform: set only from CTA-wide votes and broadcasts
  // Wait for the current step's tile, widen B/C, and synchronise the CTA.
  // After this barrier every thread has finished the previous step, so the
  // slot that the next step loads into is free. Returns the fp32 B|C rows.
  auto acquire = [&](const Cursor& cu) -> const float* {
    const uint8_t* base = smem + cu.st * K::STAGE;
    bool timed_out = false;
    if constexpr (TMA) {
      if (!producer) timed_out = !mbar_wait(&full[cu.st], cu.ph, wait_ns);
    } else {
      __syncthreads();  // every thread is done with the slot before it is restaged
      load_plain(cu);
      __syncthreads();
    }
    float* bcf = nullptr;
    if constexpr (K::BF) {
      bcf = reinterpret_cast<float*>(smem + K::OFF_BCF + cu.st * K::BCF);
      if (!timed_out && !producer) widen_bc<TILE>(base + K::OFF_B, bcf, tid);
    }
    if (__syncthreads_or(timed_out ? 1 : 0)) {
      if (tid == 0) atomicOr(p.fault, kFaultTileWait);
      abort = true;
    }
    if constexpr (K::BF) return bcf;
    else return reinterpret_cast<const float*>(base + K::OFF_B);  // fp32 B then C: [TILE][16] each
  };

  // ---- per-channel constants of the current block and the state
  f2 A2p[NP], hp[NP];
  float bias_d = 0.f, D_d = 0.f;
  int64_t d = 0;
  bool dvalid = false;
  TOut* ycol = nullptr;  // y[b, 0, d]
  int64_t hoff = 0;      // element offset of this lane's states in h0 / h_last
  auto load_block = [&](int64_t blk) {
    const int64_t b = blk / ncblk;
    d = (blk % ncblk) * CC + cb;
    dvalid = !producer && d < Dm;
    const int64_t dc = dvalid ? d : 0;
#pragma unroll
    for (int i = 0; i < NP; i++) {
      const float2 a = dvalid ? __ldg(reinterpret_cast<const float2*>(p.A + dc * kDState + n0) + i)
                              : make_float2(0.f, 0.f);
      A2p[i] = pk(a.x * kLog2e, a.y * kLog2e);
    }
    bias_d = (dvalid && p.delta_bias) ? __ldg(p.delta_bias + dc) : 0.f;
    D_d = (dvalid && p.D) ? __ldg(p.D + dc) : 0.f;
    ycol = static_cast<TOut*>(p.y) + (b * L) * Dm + dc;
    hoff = (b * Dm + dc) * kDState + n0;
  };
  auto set_state_initial = [&]() {
#pragma unroll
    for (int i = 0; i < NP; i++) {
      float2 v = make_float2(0.f, 0.f);
      if (dvalid && p.h0) v = __ldg(reinterpret_cast<const float2*>(p.h0 + hoff) + i);
      hp[i] = pk(v.x, v.y);
    }
  };

  // One state update of this lane's NS states for one token; returns the
  // lane's part of C.h. brow / crow: the token's fp32 B and C rows.
  auto update = [&](float dl, float du, const float* brow, const float* crow) -> float {
    const f2 dl2 = pk(dl, dl), du2 = pk(du, du);
    const ulonglong2* bq = reinterpret_cast<const ulonglong2*>(brow + n0);
    const ulonglong2* cq = reinterpret_cast<const ulonglong2*>(crow + n0);
    f2 acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int i = 0; i < NP / 2; i++) {
      const ulonglong2 bv = bq[i], cv = cq[i];
      {
        const f2 x = mul2(dl2, A2p[2 * i]);
        const f2 a = pk(ex2(f2lo(x)), ex2(f2hi(x)));
        hp[2 * i] = fma2(a, hp[2 * i], mul2(du2, bv.x));
        acc0 = fma2(cv.x, hp[2 * i], acc0);
      }
      {
        const f2 x = mul2(dl2, A2p[2 * i + 1]);
        const f2 a = pk(ex2(f2lo(x)), ex2(f2hi(x)));
        hp[2 * i + 1] = fma2(a, hp[2 * i + 1], mul2(du2, bv.y));
        acc1 = fma2(cv.y, hp[2 * i + 1], acc1);
      }
    }
    const f2 a = add2(acc0, acc1);
    return f2lo(a) + f2hi(a);
  };

  float ssum = 0.f;  // sum of delta over the tokens of the current pass (chunked mode)

  // Run `tlen` tokens of the acquired tile (ring slot st) starting at timestep t0.
  auto run_tile = [&](int st, const float* bcf, int64_t t0, int tlen) {
    const uint8_t* base = smem + st * K::STAGE;
    const TIn* su = reinterpret_cast<const TIn*>(base + K::OFF_U) + cb;
    const TIn* sdr = reinterpret_cast<const TIn*>(base + K::OFF_DR) + cb;
    const TIn* sz = reinterpret_cast<const TIn*>(base + K::OFF_Z) + cb;
    // token tt's fp32 B and C rows
    constexpr int BSTR = K::BF ? 2 * kDState : kDState;  // floats between rows
    constexpr int COFF = K::BF ? kDState : TILE * kDState;
    auto brow = [&](int tt) { return bcf + tt * BSTR; };
    auto crow = [&](int tt) { return bcf + COFF + tt * BSTR; };
    const f2 bias2 = pk(bias_d, bias_d), D2 = pk(D_d, D_d);
    // scalars of tokens (tt, tt+1) of this lane's channel, as packed pairs
    struct PairScalars {
      f2 dl, du, post, g;
    };
    auto scalars_pair = [&](int tt) -> PairScalars {
      PairScalars r;
      const f2 xu = pk(to_f32(su[tt * CC]), to_f32(su[(tt + 1) * CC]));
      r.dl = softplus_fast2(add2(pk(to_f32(sdr[tt * CC]), to_f32(sdr[(tt + 1) * CC])), bias2));
      r.du = mul2(r.dl, xu);
      r.post = mul2(D2, xu);
      r.g = HAS_Z ? silu2(pk(to_f32(sz[tt * CC]), to_f32(sz[(tt + 1) * CC]))) : pk(1.f, 1.f);
      return r;
    };
    if constexpr (SG == 1) {
      TOut* yp = ycol + t0 * Dm;
      auto token = [&](int tt) {
        const float xu = to_f32(su[tt * CC]);
        const float dl = softplus_fast(to_f32(sdr[tt * CC]) + bias_d);
        const float g = HAS_Z ? silu(to_f32(sz[tt * CC])) : 1.f;
        const float yv = update(dl, dl * xu, brow(tt), crow(tt));
        st_out(yp + tt * Dm, fmaf(D_d, xu, yv) * g, dvalid);
        if constexpr (MODE == kModeChunked) ssum += dl;
      };
      auto update_pair = [&](int tt, const PairScalars& r) {
        const float y0 = update(f2lo(r.dl), f2lo(r.du), brow(tt), crow(tt));
        const float y1 = update(f2hi(r.dl), f2hi(r.du), brow(tt + 1), crow(tt + 1));
        const f2 yv = mul2(add2(pk(y0, y1), r.post), r.g);
        st_out(yp + tt * Dm, f2lo(yv), dvalid);
        st_out(yp + (tt + 1) * Dm, f2hi(yv), dvalid);
        if constexpr (MODE == kModeChunked) ssum += f2lo(r.dl) + f2hi(r.dl);
      };
      if (tlen == TILE) {
        // software-pipelined groups of eight tokens: the loop body computes
        // the next group's scalars (a long softplus -> ex2 chain) next to the
        // current group's state updates, so the two overlap in one basic
        // block; the last group, with no next group in the tile, runs after
        // the loop on its own
        PairScalars cur0 = scalars_pair(0), cur1 = scalars_pair(2), cur2 = scalars_pair(4), cur3 = scalars_pair(6);
#pragma unroll 1
        for (int tt = 0; tt < TILE - 8; tt += 8) {
          const PairScalars nx0 = scalars_pair(tt + 8), nx1 = scalars_pair(tt + 10), nx2 = scalars_pair(tt + 12),
                            nx3 = scalars_pair(tt + 14);
          update_pair(tt, cur0);
          update_pair(tt + 2, cur1);
          update_pair(tt + 4, cur2);
          update_pair(tt + 6, cur3);
          cur0 = nx0;
          cur1 = nx1;
          cur2 = nx2;
          cur3 = nx3;
        }
        update_pair(TILE - 8, cur0);
        update_pair(TILE - 6, cur1);
        update_pair(TILE - 4, cur2);
        update_pair(TILE - 2, cur3);
      } else {
#pragma unroll 1
        for (int tt = 0; tt < tlen; tt++) token(tt);
      }
    } else {
      // Two lanes per channel. Per group of four tokens lane s computes the
      // scalars of tokens tt+2s and tt+2s+1 as a packed pair; the lane pair
      // swaps them, each lane updates its 8 states for all four tokens, and
      // lane s finishes y of its own two tokens from both halves of C.h.
      auto shfl2 = [&](f2 v) -> f2 {
        return pk(__shfl_xor_sync(FULL, f2lo(v), 1), __shfl_xor_sync(FULL, f2hi(v), 1));
      };
      auto group = [&](int tt, const PairScalars& r) {
        const f2 odl = shfl2(r.dl), odu = shfl2(r.du);
        const f2 dlA = s ? odl : r.dl, duA = s ? odu : r.du;  // tokens tt, tt+1
        const f2 dlB = s ? r.dl : odl, duB = s ? r.du : odu;  // tokens tt+2, tt+3
        const float p0 = update(f2lo(dlA), f2lo(duA), brow(tt), crow(tt));
        const float p1 = update(f2hi(dlA), f2hi(duA), brow(tt + 1), crow(tt + 1));
        const float p2 = update(f2lo(dlB), f2lo(duB), brow(tt + 2), crow(tt + 2));
        const float p3 = update(f2hi(dlB), f2hi(duB), brow(tt + 3), crow(tt + 3));
        const f2 mine = s ? pk(p2, p3) : pk(p0, p1), theirs = s ? pk(p0, p1) : pk(p2, p3);
        const f2 yv = mul2(add2(add2(mine, shfl2(theirs)), r.post), r.g);
        TOut* yp = ycol + (t0 + tt + 2 * s) * Dm;
        st_out(yp, f2lo(yv), dvalid);
        st_out(yp + Dm, f2hi(yv), dvalid);
        if constexpr (MODE == kModeChunked) ssum += (f2lo(dlA) + f2hi(dlA)) + (f2lo(dlB) + f2hi(dlB));
      };
      // a single token (the ragged tail): both lanes compute its scalars
      auto token = [&](int tt) {
        const float xu = to_f32(su[tt * CC]);
        const float dl = softplus_fast(to_f32(sdr[tt * CC]) + bias_d);
        const float g = HAS_Z ? silu(to_f32(sz[tt * CC])) : 1.f;
        const float part = update(dl, dl * xu, brow(tt), crow(tt));
        const float yv = part + __shfl_xor_sync(FULL, part, 1);
        st_out(ycol + (t0 + tt) * Dm, fmaf(D_d, xu, yv) * g, dvalid && s == 0);
        if constexpr (MODE == kModeChunked) ssum += dl;
      };
      if (tlen == TILE) {
        // as with one lane per channel: the tile's last eight tokens run after
        // the pipelined loop, which computes scalars only for a group that follows
        PairScalars cur0 = scalars_pair(2 * s), cur1 = scalars_pair(4 + 2 * s);
#pragma unroll 1
        for (int tt = 0; tt < TILE - 8; tt += 8) {
          const PairScalars nx0 = scalars_pair(tt + 8 + 2 * s), nx1 = scalars_pair(tt + 12 + 2 * s);
          group(tt, cur0);
          group(tt + 4, cur1);
          cur0 = nx0;
          cur1 = nx1;
        }
        group(TILE - 8, cur0);
        group(TILE - 4, cur1);
      } else {
#pragma unroll 1
        for (int tt = 0; tt < tlen; tt++) token(tt);
      }
    }
  };

  auto store_h = [&](float* dst) {
#pragma unroll
    for (int i = 0; i < NP; i++) reinterpret_cast<float2*>(dst)[i] = make_float2(f2lo(hp[i]), f2hi(hp[i]));
  };
  // Bounded wait (thread 0) for a flag to become nonzero, broadcast to the
  // CTA; every thread then acquires the flag itself (orders its later reads of
  // the published record). Returns the flag value; a timeout sets `abort`
  // CTA-wide and returns kFlagInclusive.
  auto wait_flag = [&](uint32_t* f) -> uint32_t {
    if (tid == 0) {
      uint32_t v = ld_acquire_gpu(f);
      if (v == 0) {
        const uint64_t tw = globaltimer();
        while ((v = ld_acquire_gpu(f)) == 0) {
          if (globaltimer() - tw > wait_ns) {
            atomicOr(p.fault, kFaultLookback);
            break;
          }
        }
      }
      s_flag = v;
    }
    __syncthreads();
    // thread 0's observation decides for the whole CTA (the flag may move on
    // from aggregate to inclusive meanwhile: per-thread values could split the
    // CTA); each thread's own acquire load only orders its later reads of the
    // published record, which any value at or above thread 0's covers
    const uint32_t v = s_flag;
    __syncthreads();  // s_flag is free for the next wait
    if (v == 0) {
      abort = true;
      return kFlagInclusive;
    }
    for (int i = 0; i < (1 << 20) && ld_acquire_gpu(f) < v; i++) {
    }
    return v;
  };
  // publish: every thread's stores are done (CTA barrier), then thread 0
  // releases the flag at gpu scope (unless the test knob withholds it)
  auto publish = [&](uint32_t* f, uint32_t v, bool withhold) {
    __threadfence();
    __syncthreads();
    if (tid == 0 && !withhold) st_release_gpu(f, v);
  };

  float hin[MODE == kModeChunked ? NS : 1];  // chunked: the true state entering the chunk
  hin[0] = 0.f;

  // ---- main loop over the worker's steps
  if (TMA && tid == tid_issue && nsteps > 0) issue_tma(cc);
  int64_t q = 0;
  bool next_issued = nsteps > 0;  // whether step q's load was issued (TMA)
  for (; q < nsteps; q++, advance(cc)) {
    const int64_t blk = cc.blk, j = cc.j;

    // segment start: per-channel constants and the incoming state
    if constexpr (MODE == kModeStatic) {
      if (q == 0) {
        load_block(blk);
        set_state_initial();
      }
    } else if constexpr (MODE == kModeStreamK) {
      if (q == 0 || q == zlen || q == zlen + nfull || j == 0) {
        load_block(blk);
        if (j == 0) {
          set_state_initial();
        } else {
          // the first segment starts inside a block: take the state the
          // previous CTA handed over at this range boundary
          wait_flag(p.flags + wid);
          const float* src = p.ws_carry + ((size_t)wid * CC + cb) * kDState + n0;
#pragma unroll
          for (int i = 0; i < NP; i++) {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(src) + i);
            hp[i] = pk(v.x, v.y);
          }
        }
      }
    } else {
      if (q == 0) {
        load_block(blk);
        if (c == 0) set_state_initial();
        else
          for (int i = 0; i < NP; i++) hp[i] = 0ull;
        ssum = 0.f;
      }
    }

    const float* bcf = acquire(cc);
    next_issued = false;
    if (abort) break;
    // the slot of the previous step is free: load the next step into it
    if (TMA && q + 1 < nsteps) {
      if (tid == tid_issue) {
        Cursor cn = cc;
        advance(cn);
        issue_tma(cn);
      }
      next_issued = true;
    }
    const int64_t t0 = j * TILE;
    if (!producer) run_tile(cc.st, bcf, t0, (int)min((int64_t)TILE, L - t0));

    // segment end: final state or hand-over
    if constexpr (MODE == kModeStatic) {
      if (j == T - 1 && dvalid && p.h_last) store_h(p.h_last + hoff);
    } else if constexpr (MODE == kModeStreamK) {
      if (j == T - 1) {
        if (dvalid && p.h_last) store_h(p.h_last + hoff);
      } else if (q + 1 == zlen) {
        if (!producer) store_h(p.ws_carry + ((size_t)(wid + 1) * CC + cb) * kDState + n0);
        publish(p.flags + wid + 1, kFlagHanded, wid + 1 == p.withhold_item);
      }
      if (abort) break;
    } else {
      if (q == nk - 1) {
        // ---- end of the first pass: publish the chunk's carry, look back
        const int64_t tile_id = cblk * p.nchunks + c;
        float* carry_me = p.ws_carry + ((size_t)tile_id * CC + cb) * 48 + n0;
        float hl[NS], A2[NS];
#pragma unroll
        for (int i = 0; i < NP; i++) {
          hl[2 * i] = f2lo(hp[i]);
          hl[2 * i + 1] = f2hi(hp[i]);
          A2[2 * i] = f2lo(A2p[i]);
          A2[2 * i + 1] = f2hi(A2p[i]);
        }
        const bool withhold = tile_id == p.withhold_item;
        if (producer) {
        } else if (c == 0) {
#pragma unroll
          for (int n = 0; n < NS; n++) carry_me[32 + n] = hl[n];
        } else {
#pragma unroll
          for (int n = 0; n < NS; n++) {
            carry_me[n] = ex2(A2[n] * ssum);  // P = exp(A * sum delta)
            carry_me[16 + n] = hl[n];         // S = state from a zero start
          }
        }
        publish(p.flags + tile_id, c == 0 ? kFlagInclusive : kFlagAggregate, withhold);
        if (c > 0) {
          float Pa[NS], Sa[NS];
#pragma unroll
          for (int n = 0; n < NS; n++) {
            Pa[n] = 1.f;
            Sa[n] = 0.f;
          }
          for (int64_t jj = c - 1; jj >= 0; jj--) {
            const int64_t pid = tile_id - (c - jj);
            const uint32_t f = wait_flag(p.flags + pid);
            if (abort) break;
            const float* cp = p.ws_carry + ((size_t)pid * CC + cb) * 48 + n0;
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
          if (abort) break;
          // Sa is the true state entering this chunk
          if (!producer) {
#pragma unroll
            for (int n = 0; n < NS; n++) {
              const float incl = fmaf(carry_me[n], Sa[n], hl[n]);  // P_end * h_in + S_local
              carry_me[32 + n] = incl;
              hl[n] = incl;
            }
          }
          publish(p.flags + tile_id, kFlagInclusive, withhold);
          if (c == p.nchunks - 1 && dvalid && p.h_last) {
#pragma unroll
            for (int n = 0; n < NS; n++) p.h_last[hoff + n] = hl[n];
          }
          // second pass: recompute the head from the true incoming state
#pragma unroll
          for (int i = 0; i < NP; i++) hp[i] = pk(Sa[2 * i], Sa[2 * i + 1]);
#pragma unroll
          for (int n = 0; n < NS; n++) hin[n] = Sa[n];
          ssum = 0.f;
        } else if (p.nchunks == 1 && dvalid && p.h_last) {
          store_h(p.h_last + hoff);
        }
      } else if (q >= nk && q + 1 < nsteps) {
        // second pass: stop once the carried-in part is negligible everywhere
        bool done = true;
#pragma unroll
        for (int i = 0; i < NP; i++) {
          const float a0 = f2lo(A2p[i]), a1 = f2hi(A2p[i]);
          const float c0 = fabsf(ex2(a0 * ssum) * hin[2 * i]);
          const float c1 = fabsf(ex2(a1 * ssum) * hin[2 * i + 1]);
          done = done && a0 <= 0.f && a1 <= 0.f && c0 <= kStopRel * fabsf(f2lo(hp[i])) &&
                 c1 <= kStopRel * fabsf(f2hi(hp[i]));
        }
        if (__syncthreads_and((done || !dvalid) ? 1 : 0)) break;
      }
    }
  }
  // a load issued for a step that was not run must land before the CTA ends
  // (bounded wait on that slot's phase)
  if (TMA && tid == tid_issue && next_issued) {
    Cursor cn = cc;
    advance(cn);
    if (!mbar_wait(&full[cn.st], cn.ph, wait_ns)) atomicOr(p.fault, kFaultTileWait);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised exactly once even when several host threads arrive together).
inline EncodeFn encode_fn() {
  static const EncodeFn fn = []() -> EncodeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeFn>(f);
    return nullptr;
  }();
  return fn;
}

// 3-D map over a [batch, L, inner] row-major tensor with a [1, box_t, box_inner] box.
inline bool make_map(CUtensorMap* m, const void* ptr, size_t es, int64_t batch, int64_t L, int64_t inner,
                     int box_inner, int box_t) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)inner * es, (cuuint64_t)L * inner * es};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_t, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Dynamic shared memory of every launch is at least this much, so that two
// CTAs never share an SM (the split modes size their work for one CTA per SM).
constexpr int kSmemOneCtaPerSm = 116 * 1024;

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, int MODE>
cudaError_t launch_t(const ScanParams& p, cudaStream_t stream) {
  using K = Cfg<TIn, SG>;
  auto kern = scan_fwd_kernel<TIn, TOut, SG, TMA, HAS_Z, MODE>;
  constexpr int smem = K::SMEM > kSmemOneCtaPerSm ? K::SMEM : kSmemOneCtaPerSm;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  CUtensorMap mu{}, mdr{}, mz{}, mb{}, mc{};
  if (TMA) {
    const size_t es = sizeof(TIn);
    if (!make_map(&mu, p.u, es, p.batch, p.seqlen, p.dim, K::CC, K::TILE) ||
        !make_map(&mdr, p.delta_raw, es, p.batch, p.seqlen, p.dim, K::CC, K::TILE) ||
        (HAS_Z && !make_map(&mz, p.z, es, p.batch, p.seqlen, p.dim, K::CC, K::TILE)) ||
        !make_map(&mb, p.B, es, p.batch, p.seqlen, kDState, kDState, K::TILE) ||
        !make_map(&mc, p.C, es, p.batch, p.seqlen, kDState, kDState, K::TILE))
      return cudaErrorInvalidValue;
  }
  kern<<<(unsigned)p.nworkers, kThreads, smem, stream>>>(p, mu, mdr, mz, mb, mc);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z>
cudaError_t launch_m(const ScanParams& p, cudaStream_t stream) {
  switch (p.mode) {
    case kModeStatic: return launch_t<TIn, TOut, SG, TMA, HAS_Z, kModeStatic>(p, stream);
    case kModeStreamK: return launch_t<TIn, TOut, SG, TMA, HAS_Z, kModeStreamK>(p, stream);
    case kModeChunked: return launch_t<TIn, TOut, SG, TMA, HAS_Z, kModeChunked>(p, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TIn, typename TOut, int SG, bool TMA>
cudaError_t launch_z(const ScanParams& p, cudaStream_t stream) {
  return p.z ? launch_m<TIn, TOut, SG, TMA, true>(p, stream) : launch_m<TIn, TOut, SG, TMA, false>(p, stream);
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
