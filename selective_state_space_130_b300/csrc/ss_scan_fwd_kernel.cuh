// Selective-scan (S6) forward kernel for sm_103a (template; instantiated per
// input/output dtype pair in ss_scan_fwd_<in>_<out>.cu).
//
// What one warp computes. A warp owns DC = 32/SG consecutive channels of one
// batch element (a "channel block"). With SG = 1 each lane owns one channel and
// all 16 of its fp32 states; with SG = 2 two lanes share a channel, 8 states
// each. Per token the lane computes delta = softplus(delta_raw + bias),
// Abar = 2^(delta * A * log2 e), h = Abar*h + (delta*u)*B, y = C.h + D*u and
// y *= silu(z): the fused, SRAM-resident scan the Mamba pages describe (review
// page, method step 2; "Transformer时代终结？" section 二.3), laid out for B300.
// The state update runs on packed f32x2 FMUL2/FFMA2 (two states per issue
// slot); the exponentials run on the MUFU pipe. On B300 that pair of pipes,
// not HBM, bounds the exact fp32 recurrence: about 30 state updates per clock
// per SM at best against 4 bytes of HBM traffic per 16 updates.
//
// Data path. Tiles of TILE timesteps stream through a kStages-deep ring in
// the warp's shared memory: u, delta_raw, z ([TILE, DC] boxes) and the tile's
// B and C rows ([TILE, 16]) arrive by TMA (cp.async.bulk.tensor) with
// completion counted on one mbarrier per stage, issued by the warp itself
// kStages-1 tiles ahead. bf16 B/C rows are widened once per tile into an fp32
// buffer read by broadcast. Only y and the final state leave the chip. A
// block holds kWarps independent warps (one per SM sub-partition).
//
// Work split (ScanMode).
//  - static: one warp per channel block, the whole sequence.
//  - stream-K: the (channel block, tile) space, block-major, is cut into
//    nworkers equal contiguous ranges, at least one block long each, so a range
//    crosses at most one block start in its interior... and holds at most one
//    partial block at either end. A warp first runs the head of the block its
//    range ends in (from that block's initial state) and hands the state at
//    its range end to the next warp, then runs the rest of its range in order;
//    the first segment, when it starts inside a block, waits for the state the
//    previous warp handed over (almost always already there). Equal ranges keep
//    every SM sub-partition equally busy whatever the channel count.
//  - chunked (long sequences, few channel blocks): each block's sequence is
//    cut into chunks run by different warps. A chunk's carry pair
//    (P = prod Abar = exp(A * sum delta), S = state reached from zero) composes
//    as (P1,S1) o (P2,S2) = (P1 P2, P2 S1 + S2) ("外文文献精读" section 2.2;
//    mlqm.cn tutorial section 6). Chunks publish their pair and resolve their
//    incoming state by decoupled look-back, then recompute their head from the
//    true state until, for every state n, the carried-in part P_t,n * h_in,n is
//    at most 2^-24 of h_t,n (for A <= 0 it only decays further): the outputs
//    equal the sequential recurrence up to fp32 rounding.
// Warps take their worker index from a ticket counter in launch order, so a
// warp only ever waits for warps that have already started; every wait is
// bounded and reports a timeout through the fault word.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace scan_detail {

constexpr int kTile = 32;    // timesteps per pipeline stage (64 for bf16 one-lane channels)
constexpr int kStages = 3;   // TMA ring depth
constexpr int kWarps = 4;    // warps (independent workers) per block
constexpr int kUnroll = 8;   // tokens per step of the token loop (written out by hand below)
constexpr float kStopRel = 5.9604645e-8f;  // 2^-24

constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagInclusive = 2u;
constexpr uint32_t kFlagHanded = 1u;
constexpr int kHeaderWords = 64;
constexpr uint32_t kHeaderMagic = 0x53535753u;  // header word 2: "this call used the workspace"
constexpr int kSmemPerSM = 233472;              // 228 KiB per SM, 1 KiB of it reserved per block

template <typename TIn, int SG>
struct Cfg {
  static constexpr int NS = kDState / SG;  // states per lane
  static constexpr int NP = NS / 2;        // packed state pairs per lane
  static constexpr int DC = 32 / SG;       // channels per warp
  static constexpr bool BF = sizeof(TIn) == 2;
  // timesteps per tile: the bf16 one-lane-per-channel layout fits 64 in the
  // shared memory of four warps per SM, halving the per-tile ring overhead
  static constexpr int TILE = (BF && SG == 1) ? 2 * kTile : kTile;
  static constexpr int XB = TILE * DC * (int)sizeof(TIn);         // one u / delta_raw / z tile
  static constexpr int RB = TILE * kDState * (int)sizeof(TIn);    // one raw B or C tile
  static constexpr int OFF_U = 0, OFF_DR = XB, OFF_Z = 2 * XB, OFF_B = 3 * XB, OFF_C = 3 * XB + RB;
  static constexpr int STAGE = (3 * XB + 2 * RB + 127) & ~127;
  static constexpr int OFF_BCF = kStages * STAGE;                  // fp32 B|C of the current tile (bf16 only)
  static constexpr int BCF = BF ? 2 * TILE * kDState * 4 : 0;
  static constexpr int OFF_BAR = OFF_BCF + BCF;
  static constexpr int WARP_SMEM = (OFF_BAR + kStages * 8 + 127) & ~127;
  static constexpr int SMEM = kWarps * WARP_SMEM + 128;            // + base alignment slack
  static constexpr int BLOCKS_PER_SM = kSmemPerSM / (SMEM + 1024);
};

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, int MODE>
__global__ void __launch_bounds__(32 * kWarps, 1) scan_fwd_kernel(const __grid_constant__ ScanParams p,
                                                                  const __grid_constant__ CUtensorMap tm_u,
                                                                  const __grid_constant__ CUtensorMap tm_dr,
                                                                  const __grid_constant__ CUtensorMap tm_z,
                                                                  const __grid_constant__ CUtensorMap tm_b,
                                                                  const __grid_constant__ CUtensorMap tm_c) {
  using K = Cfg<TIn, SG>;
  constexpr int NS = K::NS, NP = K::NP, DC = K::DC, TILE = K::TILE;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 128-byte aligned base, derived from the shared array by pointer arithmetic
  // only (a round trip through an integer would hide from the compiler that
  // every tile access is a shared-memory access)
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad + warp * K::WARP_SMEM;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
  const int s = lane % SG;   // which part of the channel's states this lane holds
  const int cw = lane / SG;  // channel within the warp's block
  const int n0 = s * NS;

  // ---- worker index
  int64_t wid;
  if constexpr (MODE == kModeStatic) {
    wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  } else {
    uint32_t t = 0;
    if (lane == 0) t = atomicAdd(p.ws_header, 1u);  // launch-order ticket
    wid = __shfl_sync(FULL, t, 0);
  }
  if (wid >= p.nworkers) return;
  if (lane == 0) {
    for (int i = 0; i < kStages; i++) mbar_init(&full[i], 1);
    fence_mbar_init();
    if (p.ws_header && wid == 0) p.ws_header[2] = kHeaderMagic;
  }
  __syncwarp();
  if (TMA && lane == 0) {
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_dr);
    if (HAS_Z) tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
  }

  const int64_t T = p.tiles_per_blk, L = p.seqlen, Dm = p.dim;
  const int ncblk = p.ncblk;

  // ---- the worker's steps: step q runs tile j of channel block blk
  int64_t r0 = 0, zs = 0, zlen = 0, af = 0, nfull = 0, nsteps = 0;  // stream-K
  int64_t cblk = 0, c = 0, j0 = 0, nk = 0;        // chunked
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
  auto place = [&](Cursor& c) {  // (blk, j) and the block's coordinates for step c.q
    if constexpr (MODE == kModeStatic) {
      c.blk = wid;
      c.j = c.q;
    } else if constexpr (MODE == kModeStreamK) {
      // the head of the last block (handed over to the next warp), then the
      // whole blocks, then the first segment, which waits for the previous
      // warp's hand-over: with ranges of at least one block that hand-over is
      // already done by the time this warp gets there
      const int64_t q = c.q;
      const int64_t g = q < zlen ? zs + q : (q < zlen + nfull ? af + (q - zlen) : r0 + (q - zlen - nfull));
      c.blk = g / T;
      c.j = g - c.blk * T;
    } else {
      c.blk = cblk;
      c.j = j0 + (c.q < nk ? c.q : c.q - nk);
    }
    c.b = (int)(c.blk / ncblk);
    c.x0 = (int)(c.blk - (int64_t)c.b * ncblk) * DC;
  };
  auto advance = [&](Cursor& c) {
    c.q++;
    if (++c.st == kStages) {
      c.st = 0;
      c.ph ^= 1u;
    }
    bool jump = false;
    if constexpr (MODE == kModeStreamK) jump = c.q == zlen || c.q == zlen + nfull;
    if constexpr (MODE == kModeChunked) jump = c.q == nk;
    if (jump) {
      place(c);
    } else if (++c.j == T) {
      c.j = 0;
      c.blk++;
      c.x0 += DC;
      if (c.x0 >= ncblk * DC) {
        c.x0 = 0;
        c.b++;
      }
    }
  };
  Cursor ci{0, 0, 0, 0, 0, 0, 0u};  // next step to issue
  place(ci);
  Cursor cc = ci;                   // next step to consume

  // ---- TMA ring
  bool abort = false;
  auto issue = [&](const Cursor& c) {
    const int st = c.st;
    uint8_t* base = smem + st * K::STAGE;
    const int b = c.b;
    const int x0 = c.x0;
    const int y0 = (int)(c.j * TILE);
    if constexpr (TMA) {
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(&full[st], (HAS_Z ? 3 : 2) * K::XB + 2 * K::RB);
        tma_load_3d(base + K::OFF_U, &tm_u, x0, y0, b, &full[st]);
        tma_load_3d(base + K::OFF_DR, &tm_dr, x0, y0, b, &full[st]);
        if (HAS_Z) tma_load_3d(base + K::OFF_Z, &tm_z, x0, y0, b, &full[st]);
        tma_load_3d(base + K::OFF_B, &tm_b, 0, y0, b, &full[st]);
        tma_load_3d(base + K::OFF_C, &tm_c, 0, y0, b, &full[st]);
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
      for (int i = lane; i < TILE * DC; i += 32) {
        const int tt = i / DC, cc = i % DC;
        const int64_t t = (int64_t)y0 + tt, dd = (int64_t)x0 + cc;
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
      for (int i = lane; i < TILE * kDState; i += 32) {
        const int64_t t = (int64_t)y0 + i / kDState;
        const bool ok = t < L;
        const int64_t gi = ((int64_t)b * L + (ok ? t : 0)) * kDState + i % kDState;
        sB[i] = ok ? gB[gi] : from_f32<TIn>(0.f);
        sC[i] = ok ? gC[gi] : from_f32<TIn>(0.f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
    }
  };
  // issue every step below qmax not yet issued; the caller has synchronised
  // the warp, so the ring slot being refilled is no longer read
  auto issue_upto = [&](int64_t qmax) {
    const int64_t lim = min(qmax, nsteps);
    while (ci.q < lim) {
      issue(ci);
      advance(ci);
    }
  };
  // wait for step q's tile; returns the fp32 B|C rows of the tile
  auto acquire = [&](const Cursor& c) -> const float* {
    const int st = c.st;
    const bool timed_out = !abort && !mbar_wait(&full[st], c.ph);
    if (__any_sync(FULL, timed_out)) {  // keep `abort` warp-uniform
      abort = true;
      if (lane == 0) atomicOr(p.fault, kFaultTileWait);
    }
    const uint8_t* base = smem + st * K::STAGE;
    if constexpr (K::BF) {
      // B then C (2 x TILE x 16 bf16, contiguous in the stage) widened to
      // fp32: per pass each lane takes four consecutive values, so both the
      // 8-byte loads and the 16-byte stores are contiguous across the warp
      const uint2* src = reinterpret_cast<const uint2*>(base + K::OFF_B);
      float4* dst = reinterpret_cast<float4*>(smem + K::OFF_BCF);
#pragma unroll
      for (int i = 0; i < (2 * TILE * kDState) / (4 * 32); i++) {
        const uint2 v = src[i * 32 + lane];
        dst[i * 32 + lane] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                         __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
      }
      __syncwarp();
      return reinterpret_cast<const float*>(smem + K::OFF_BCF);
    } else {
      return reinterpret_cast<const float*>(base + K::OFF_B);  // fp32 B then C, contiguous
    }
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
    d = (blk % ncblk) * DC + cw;
    dvalid = d < Dm;
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
  // lane's part of C.h.
  auto update = [&](float dl, float du, const float* brow, const float* crow) -> float {
    const f2 dl2 = pk(dl, dl), du2 = pk(du, du);
    const ulonglong2* bq = reinterpret_cast<const ulonglong2*>(brow);
    const ulonglong2* cq = reinterpret_cast<const ulonglong2*>(crow);
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

  // Run `tlen` tokens of the acquired tile (slot `st`) starting at timestep t0.
  auto run_tile = [&](int st, const float* bcf, int64_t t0, int tlen) {
    const uint8_t* base = smem + st * K::STAGE;
    const TIn* su = reinterpret_cast<const TIn*>(base + K::OFF_U) + cw;
    const TIn* sdr = reinterpret_cast<const TIn*>(base + K::OFF_DR) + cw;
    const TIn* sz = reinterpret_cast<const TIn*>(base + K::OFF_Z) + cw;
    const float* brow = bcf + n0;
    const float* crow = bcf + TILE * kDState + n0;
    if constexpr (SG == 1) {
      TOut* yp = ycol + t0 * Dm;
      auto token = [&](int tt) {
        const float xu = to_f32(su[tt * DC]);
        const float dl = softplus_fast(to_f32(sdr[tt * DC]) + bias_d);
        const float g = HAS_Z ? silu(to_f32(sz[tt * DC])) : 1.f;
        const float yv = update(dl, dl * xu, brow + tt * kDState, crow + tt * kDState);
        st_out(yp + tt * Dm, fmaf(D_d, xu, yv) * g, dvalid);
        if constexpr (MODE == kModeChunked) ssum += dl;
      };
      // two tokens whose per-token scalars are computed as packed pairs
      const f2 bias2 = pk(bias_d, bias_d), D2 = pk(D_d, D_d);
      struct PairScalars {
        f2 dl, du, post, g;
      };
      auto scalars_pair = [&](int tt) -> PairScalars {
        PairScalars r;
        const f2 xu = pk(to_f32(su[tt * DC]), to_f32(su[(tt + 1) * DC]));
        r.dl = softplus_fast2(add2(pk(to_f32(sdr[tt * DC]), to_f32(sdr[(tt + 1) * DC])), bias2));
        r.du = mul2(r.dl, xu);
        r.post = mul2(D2, xu);
        r.g = HAS_Z ? silu2(pk(to_f32(sz[tt * DC]), to_f32(sz[(tt + 1) * DC]))) : pk(1.f, 1.f);
        return r;
      };
      auto update_pair = [&](int tt, const PairScalars& r) {
        const float y0 = update(f2lo(r.dl), f2lo(r.du), brow + tt * kDState, crow + tt * kDState);
        const float y1 = update(f2hi(r.dl), f2hi(r.du), brow + (tt + 1) * kDState, crow + (tt + 1) * kDState);
        const f2 yv = mul2(add2(pk(y0, y1), r.post), r.g);
        st_out(yp + tt * Dm, f2lo(yv), dvalid);
        st_out(yp + (tt + 1) * Dm, f2hi(yv), dvalid);
        if constexpr (MODE == kModeChunked) ssum += f2lo(r.dl) + f2hi(r.dl);
      };
      if (tlen == TILE) {
        // software-pipelined groups of eight tokens: the loop body computes
        // the next group's scalars (a long softplus -> ex2 chain) next to the
        // current group's state updates, so the two overlap in one basic
        // block; the last group recomputes its own scalars instead of reading
        // past the tile
        PairScalars cur0 = scalars_pair(0), cur1 = scalars_pair(2), cur2 = scalars_pair(4), cur3 = scalars_pair(6);
#pragma unroll 1
        for (int tt = 0; tt < TILE; tt += kUnroll) {
          const int tn = min(tt + kUnroll, TILE - kUnroll);
          const PairScalars nx0 = scalars_pair(tn), nx1 = scalars_pair(tn + 2), nx2 = scalars_pair(tn + 4),
                            nx3 = scalars_pair(tn + 6);
          update_pair(tt, cur0);
          update_pair(tt + 2, cur1);
          update_pair(tt + 4, cur2);
          update_pair(tt + 6, cur3);
          cur0 = nx0;
          cur1 = nx1;
          cur2 = nx2;
          cur3 = nx3;
        }
      } else {
#pragma unroll 1
        for (int tt = 0; tt < tlen; tt++) token(tt);
      }
    } else {
      // token pair (tt, tt+1): lane s computes the scalars of token tt+s and
      // stores its y; the pair exchanges (delta, delta*u) and the halves of C.h
      TOut* yp = ycol + (t0 + s) * Dm;
      auto pair = [&](int tt, bool two) {
        const int tm = tt + s;  // may be tlen for an odd tail: a row of the tile buffer, unused
        const float xu = to_f32(su[tm * DC]);
        const float dl = softplus_fast(to_f32(sdr[tm * DC]) + bias_d);
        const float g = HAS_Z ? silu(to_f32(sz[tm * DC])) : 1.f;
        const float du = dl * xu;
        const float dlo = __shfl_xor_sync(FULL, dl, 1), duo = __shfl_xor_sync(FULL, du, 1);
        const float pa = update(s ? dlo : dl, s ? duo : du, brow + tt * kDState, crow + tt * kDState);
        float pb = 0.f;
        if (two) pb = update(s ? dl : dlo, s ? du : duo, brow + (tt + 1) * kDState, crow + (tt + 1) * kDState);
        const float keep = s ? pb : pa, send = s ? pa : pb;
        const float yv = keep + __shfl_xor_sync(FULL, send, 1);
        st_out(yp + tt * Dm, fmaf(D_d, xu, yv) * g, dvalid && (two || s == 0));
        if constexpr (MODE == kModeChunked) ssum += (s ? dlo : dl) + (two ? (s ? dl : dlo) : 0.f);
      };
      if (tlen == TILE) {
#pragma unroll 1
        for (int tt = 0; tt < TILE; tt += kUnroll) {
          pair(tt, true);
          pair(tt + 2, true);
          pair(tt + 4, true);
          pair(tt + 6, true);
        }
      } else {
#pragma unroll 1
        for (int tt = 0; tt < tlen; tt += 2) pair(tt, tt + 1 < tlen);
      }
    }
  };

  auto store_h = [&](float* dst) {
#pragma unroll
    for (int i = 0; i < NP; i++) reinterpret_cast<float2*>(dst)[i] = make_float2(f2lo(hp[i]), f2hi(hp[i]));
  };
  // bounded wait (lane 0) for a flag to become nonzero; every lane then
  // acquires it itself. Returns the flag value (forced nonzero on timeout).
  auto wait_flag = [&](uint32_t* f) -> uint32_t {
    uint32_t v = 0;
    if (lane == 0) {
      v = ld_acquire_gpu(f);
      if (v == 0 && !abort) {
        const uint64_t tw = globaltimer();
        while ((v = ld_acquire_gpu(f)) == 0) {
          if (globaltimer() - tw > kWaitNs) {
            atomicOr(p.fault, kFaultLookback);
            abort = true;
            break;
          }
        }
      }
    }
    // lane 0's observation decides for the whole warp (the flag may move on
    // from aggregate to inclusive meanwhile: a per-lane value could split the
    // warp); each lane's own acquire load only orders its later reads of the
    // published record, which any value at or above lane 0's covers
    v = __shfl_sync(FULL, v, 0);
    abort = __shfl_sync(FULL, abort ? 1 : 0, 0) != 0;
    if (v != 0)
      for (int i = 0; i < (1 << 20) && ld_acquire_gpu(f) < v; i++) {
      }
    return v == 0 ? kFlagInclusive : v;
  };

  float hin[MODE == kModeChunked ? NS : 1];  // chunked: the true state entering the chunk
  hin[0] = 0.f;

  // ---- main loop over the worker's steps
  issue_upto(kStages - 1);
  int64_t q = 0;
  for (; q < nsteps; q++, advance(cc)) {
    __syncwarp();
    issue_upto(q + kStages);
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
          // previous worker handed over at this range boundary
          wait_flag(p.flags + wid);
          const float* src = p.ws_carry + (size_t)wid * DC * kDState + cw * kDState + n0;
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
    const int64_t t0 = j * TILE;
    run_tile(cc.st, bcf, t0, (int)min((int64_t)TILE, L - t0));

    // segment end: final state or hand-over
    if constexpr (MODE == kModeStatic) {
      if (j == T - 1 && dvalid && p.h_last) store_h(p.h_last + hoff);
    } else if constexpr (MODE == kModeStreamK) {
      if (j == T - 1) {
        if (dvalid && p.h_last) store_h(p.h_last + hoff);
      } else if (q + 1 == zlen) {
        float* dst = p.ws_carry + (size_t)(wid + 1) * DC * kDState + cw * kDState + n0;
        store_h(dst);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.flags + wid + 1, kFlagHanded);
      }
    } else {
      if (q == nk - 1) {
        // ---- end of the first pass: publish the chunk's carry, look back
        const int64_t tile_id = cblk * p.nchunks + c;
        float* carry_me = p.ws_carry + ((size_t)tile_id * DC + cw) * 48 + n0;
        float hl[NS];
#pragma unroll
        for (int i = 0; i < NP; i++) {
          hl[2 * i] = f2lo(hp[i]);
          hl[2 * i + 1] = f2hi(hp[i]);
        }
        float A2[NS];
#pragma unroll
        for (int i = 0; i < NP; i++) {
          A2[2 * i] = f2lo(A2p[i]);
          A2[2 * i + 1] = f2hi(A2p[i]);
        }
        if (c == 0) {
#pragma unroll
          for (int n = 0; n < NS; n++) carry_me[32 + n] = hl[n];
        } else {
#pragma unroll
          for (int n = 0; n < NS; n++) {
            carry_me[n] = ex2(A2[n] * ssum);  // P = exp(A * sum delta)
            carry_me[16 + n] = hl[n];         // S = state from a zero start
          }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.flags + tile_id, c == 0 ? kFlagInclusive : kFlagAggregate);
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
          float Pend[NS];
#pragma unroll
          for (int n = 0; n < NS; n++) Pend[n] = carry_me[n];
#pragma unroll
          for (int n = 0; n < NS; n++) {
            const float incl = fmaf(Pend[n], Sa[n], hl[n]);  // P_end * h_in + S_local
            carry_me[32 + n] = incl;
            hl[n] = incl;
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) st_release_gpu(p.flags + tile_id, kFlagInclusive);
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
        if (__all_sync(FULL, done || !dvalid)) {
          q++;
          break;
        }
      }
    }
    if (abort) {
      q++;
      break;
    }
  }
  // drain loads issued past the last consumed step (bounded waits)
  __syncwarp();
  if (q < nsteps) {
    if (cc.q != q) {  // left the loop by break: cc still names step q-1
      cc.q = q - 1;
      advance(cc);
    }
    for (; cc.q < ci.q; advance(cc))
      if (!mbar_wait(&full[cc.st], cc.ph)) atomicOr(p.fault, kFaultTileWait);
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

template <typename TIn, typename TOut, int SG, bool TMA, bool HAS_Z, int MODE>
cudaError_t launch_t(const ScanParams& p, cudaStream_t stream) {
  using K = Cfg<TIn, SG>;
  auto kern = scan_fwd_kernel<TIn, TOut, SG, TMA, HAS_Z, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, K::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mu{}, mdr{}, mz{}, mb{}, mc{};
  if (TMA) {
    const size_t es = sizeof(TIn);
    if (!make_map(&mu, p.u, es, p.batch, p.seqlen, p.dim, K::DC, K::TILE) ||
        !make_map(&mdr, p.delta_raw, es, p.batch, p.seqlen, p.dim, K::DC, K::TILE) ||
        (HAS_Z && !make_map(&mz, p.z, es, p.batch, p.seqlen, p.dim, K::DC, K::TILE)) ||
        !make_map(&mb, p.B, es, p.batch, p.seqlen, kDState, kDState, K::TILE) ||
        !make_map(&mc, p.C, es, p.batch, p.seqlen, kDState, kDState, K::TILE))
      return cudaErrorInvalidValue;
  }
  // the split modes place kWarps workers per block, one per SM sub-partition;
  // one-warp blocks spread the few warps of the static mode over all SMs
  const int wpb = MODE == kModeStatic ? 1 : kWarps;
  const int64_t nblocks = (p.nworkers + wpb - 1) / wpb;
  const int smem = wpb * K::WARP_SMEM + 128;
  kern<<<(unsigned)nblocks, 32 * wpb, smem, stream>>>(p, mu, mdr, mz, mb, mc);
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
