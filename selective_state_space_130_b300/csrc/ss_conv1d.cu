// Causal depthwise convolution front-end of the Mamba block (width K <= 4,
// optional SiLU) and its single-token decode step, for sm_103a.
//
// The block feeds the expanded input through a short causal convolution along
// the sequence and a SiLU before the selective SSM ("Mamba: Linear-Time
// Sequence Modeling with Selective State Spaces" review page, method step 3;
// mlqm.cn tutorial section 7.1). Decoding keeps per request only the last K-1
// inputs that convolution needs ("AI 推理系列（十四）：Mamba 的 Selective State
// Space", the decode-state table and the request-state sections). Tap k
// multiplies x[t-(K-1)+k]; the state holds the K-1 inputs before t = 0,
// oldest first.
//
// Both kernels are HBM-bound streams: the forward reads x once and writes y
// once (plus a halo of K-1 rows per tile, served by L2).
//  - Rows of 16-byte-aligned width stream through shared memory: persistent
//    CTAs (three per SM) take ranges of tiles of [64 timesteps + halo, 256 bytes
//    of channels]; a producer warp keeps a four-stage ring of TMA
//    (cp.async.bulk.tensor) loads in flight, so the HBM requests never pause
//    while a tile is computed, and four compute warps run the taps, bias and
//    SiLU on channel pairs as packed f32x2 arithmetic. y of x's type goes back
//    into the stage and leaves by one bulk-tensor store per tile.
//  - Other rows: a thread owns one channel over kConvTT timesteps and issues
//    every load of its window before any arithmetic.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTT = 8;   // timesteps per thread

// V consecutive elements of a row, loaded as one vector (or one element)
template <typename T, int V>
struct Row {
  static constexpr int kWords = (int)(V * sizeof(T) / 4);  // 32-bit words (0 for a lone bf16)
  static constexpr int kN = kWords > 0 ? kWords : 1;        // storage words
  uint32_t w[kN];
};

template <typename T, int V>
__device__ __forceinline__ Row<T, V> load_row(const T* p) {
  Row<T, V> r;
  if constexpr (V * sizeof(T) == 16) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
    r.w[0] = v.x;
    r.w[1] = v.y;
    r.w[2] = v.z;
    r.w[3] = v.w;
  } else if constexpr (sizeof(T) == 4) {
    r.w[0] = __float_as_uint(__ldcs(reinterpret_cast<const float*>(p)));
  } else {
    r.w[0] = (uint32_t)__bfloat16_as_ushort(p[0]);
  }
  return r;
}

template <typename T, int V>
__device__ __forceinline__ float row_get(const Row<T, V>& r, int v) {
  if constexpr (sizeof(T) == 4) {
    return __uint_as_float(r.w[v]);
  } else if constexpr (V == 1) {
    return __uint_as_float(r.w[0] << 16);
  } else {
    const uint32_t w = r.w[v >> 1];
    return __uint_as_float((v & 1) ? (w & 0xffff0000u) : (w << 16));
  }
}

template <typename T>
__device__ __forceinline__ T raw_elem(uint32_t bits);
template <>
__device__ __forceinline__ float raw_elem<float>(uint32_t bits) {
  return __uint_as_float(bits);
}
template <>
__device__ __forceinline__ __nv_bfloat16 raw_elem<__nv_bfloat16>(uint32_t bits) {
  return __ushort_as_bfloat16((unsigned short)bits);
}

// the raw stored bits of element v (exact copy for the carried state)
template <typename T, int V>
__device__ __forceinline__ T row_raw(const Row<T, V>& r, int v) {
  if constexpr (sizeof(T) == 4) {
    return raw_elem<T>(r.w[v]);
  } else if constexpr (V == 1) {
    return raw_elem<T>(r.w[0]);
  } else {
    const uint32_t w = r.w[v >> 1];
    return raw_elem<T>((v & 1) ? (w >> 16) : (w & 0xffffu));
  }
}

template <typename TOut, int V>
__device__ __forceinline__ void store_out(TOut* p, const float (&o)[V]) {
  if constexpr (sizeof(TOut) == 2 && V == 8) {
    uint4 v;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < 4; i++)
      w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i])) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i + 1])) << 16);
    __stcs(reinterpret_cast<uint4*>(p), v);
  } else if constexpr (sizeof(TOut) == 4 && V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V / 4; i++)
      __stcs(reinterpret_cast<float4*>(p) + i, make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < V; i++) p[i] = from_f32<TOut>(o[i]);
  }
}

template <typename TIn, typename TOut, int K, int V, bool SILU>
__global__ void __launch_bounds__(kConvThreads, 2) conv1d_fwd_kernel(const __grid_constant__ ConvParams p) {
  constexpr int H = K - 1;
  constexpr int W = kConvTT + H;  // window rows
  const int64_t L = p.seqlen, Dm = p.dim;
  const int64_t nvec = Dm / V;
  const int64_t nt = (L + kConvTT - 1) / kConvTT;
  const int64_t gid = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
  if (gid >= p.batch * nt * nvec) return;
  const int64_t vec = gid % nvec, rest = gid / nvec;
  const int64_t tc = rest % nt, b = rest / nt;
  const int64_t d0 = vec * V, t0 = tc * kConvTT;
  const TIn* gx = static_cast<const TIn*>(p.x);
  const TIn* gs = static_cast<const TIn*>(p.state_in);

  // the window: rows t0-H .. t0+kConvTT-1, all loads first
  Row<TIn, V> win[W];
#pragma unroll
  for (int r = 0; r < W; r++) {
    const int64_t t = t0 - H + r;
    if (t >= 0 && t < L) {
      win[r] = load_row<TIn, V>(gx + (b * L + t) * Dm + d0);
    } else if (t < 0 && gs) {
      // the carried inputs before t = 0: state[b, d, t + H] per channel
#pragma unroll
      for (int i = 0; i < Row<TIn, V>::kN; i++) win[r].w[i] = 0u;
      if constexpr (sizeof(TIn) == 4) {
#pragma unroll
        for (int v = 0; v < V; v++)
          win[r].w[v] = __float_as_uint(reinterpret_cast<const float*>(gs)[(b * Dm + d0 + v) * H + t + H]);
      } else if constexpr (V == 1) {
        win[r].w[0] = (uint32_t)__bfloat16_as_ushort(gs[(b * Dm + d0) * H + t + H]);
      } else {
#pragma unroll
        for (int v = 0; v < V; v++) {
          const uint32_t bits = (uint32_t)__bfloat16_as_ushort(gs[(b * Dm + d0 + v) * H + t + H]);
          win[r].w[v >> 1] |= (v & 1) ? (bits << 16) : bits;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < Row<TIn, V>::kN; i++) win[r].w[i] = 0u;
    }
  }

  // taps and biases of the thread's V channels: contiguous, loaded as 16-byte
  // vectors when the thread owns a vector of channels
  float w[V * K], bias[V];
  if constexpr (V > 1) {
#pragma unroll
    for (int i = 0; i < V * K / 4; i++) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.w + d0 * K) + i);
      w[4 * i] = q.x;
      w[4 * i + 1] = q.y;
      w[4 * i + 2] = q.z;
      w[4 * i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < V / 4; i++) {
      const float4 q = p.bias ? __ldg(reinterpret_cast<const float4*>(p.bias + d0) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      bias[4 * i] = q.x;
      bias[4 * i + 1] = q.y;
      bias[4 * i + 2] = q.z;
      bias[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < K; k++) w[k] = __ldg(p.w + d0 * K + k);
    bias[0] = p.bias ? __ldg(p.bias + d0) : 0.f;
  }

  // each input row is widened once and scattered into the K outputs that use
  // it; output j is complete after row j + H and is stored then (a ring of K
  // partial sums per channel, indexed at compile time)
  TOut* gy = static_cast<TOut*>(p.y) + (b * L + t0) * Dm + d0;
  float acc[K][V];
#pragma unroll
  for (int r = 0; r < W; r++) {
    float xr[V];
#pragma unroll
    for (int v = 0; v < V; v++) xr[v] = row_get<TIn, V>(win[r], v);
    // row r is tap k of output j = r - k
#pragma unroll
    for (int k = 0; k < K; k++) {
      const int j = r - k;
      if (j >= 0 && j < kConvTT) {
        float (&a)[V] = acc[j % K];
#pragma unroll
        for (int v = 0; v < V; v++) a[v] = fmaf(w[v * K + k], xr[v], k == 0 ? bias[v] : a[v]);
      }
    }
    const int jd = r - H;  // the output completed by this row
    if (jd >= 0 && t0 + jd < L) {
      float o[V];
#pragma unroll
      for (int v = 0; v < V; v++) o[v] = SILU ? silu(acc[jd % K][v]) : acc[jd % K][v];
      store_out<TOut, V>(gy + jd * Dm, o);
    }
  }

  // the chunk holding the last timestep hands on the last H inputs
  if (p.state_out && t0 + kConvTT >= L) {
    TIn* so = static_cast<TIn*>(p.state_out);
    // rows at positions L-H .. L-1 (compile-time row indices keep the window
    // in registers)
#pragma unroll
    for (int r = 0; r < W; r++) {
      const int64_t k = t0 - H + r - (L - H);  // state slot of window row r
      if (k >= 0 && k < H) {
#pragma unroll
        for (int v = 0; v < V; v++) so[(b * Dm + d0 + v) * H + k] = row_raw<TIn, V>(win[r], v);
      }
    }
  }
}

// element i of a packed array of T held in 32-bit words (i known at compile time)
template <typename T>
__device__ __forceinline__ uint32_t word_elem(const uint32_t* wd, int i) {
  if constexpr (sizeof(T) == 4) return wd[i];
  else return (i & 1) ? (wd[i >> 1] >> 16) : (wd[i >> 1] & 0xffffu);
}
template <typename T>
__device__ __forceinline__ void set_word_elem(uint32_t* wd, int i, uint32_t bits) {
  if constexpr (sizeof(T) == 4) wd[i] = bits;
  else wd[i >> 1] = (i & 1) ? ((wd[i >> 1] & 0xffffu) | (bits << 16)) : ((wd[i >> 1] & 0xffff0000u) | bits);
}
template <typename T>
__device__ __forceinline__ float bits_f32(uint32_t bits) {
  return sizeof(T) == 4 ? __uint_as_float(bits) : __uint_as_float(bits << 16);
}

template <typename TIn, typename TOut, int K, int V, bool SILU, int BS>
__global__ void __launch_bounds__(kConvThreads) conv1d_update_kernel(const __grid_constant__ ConvParams p) {
  // V consecutive channels of BS consecutive streams per thread: the V
  // channels' states (V x H elements) are contiguous, so state, x and y move
  // as whole 16-byte vectors when V > 1; the taps and biases, loaded once, serve
  // all BS streams. (With V > 1, dim is a multiple of V.)
  constexpr int H = K - 1;
  const int64_t g = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;
  const int64_t ncg = (p.dim + V - 1) / V;  // channel groups per stream
  const int64_t d0 = (g % ncg) * V;          // first channel of the group
  const int64_t b0 = (g / ncg) * BS;         // first stream
  if (b0 >= p.batch) return;
  // taps and biases of the V channels: contiguous, 16-byte vectors when V > 1
  float w[V * K], bias[V];
  if constexpr (V > 1) {
#pragma unroll
    for (int i = 0; i < V * K / 4; i++) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p.w + d0 * K) + i);
      w[4 * i] = q.x;
      w[4 * i + 1] = q.y;
      w[4 * i + 2] = q.z;
      w[4 * i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < V / 4; i++) {
      const float4 q = p.bias ? __ldg(reinterpret_cast<const float4*>(p.bias + d0) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      bias[4 * i] = q.x;
      bias[4 * i + 1] = q.y;
      bias[4 * i + 2] = q.z;
      bias[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < K; k++) w[k] = __ldg(p.w + d0 * K + k);
    bias[0] = p.bias ? __ldg(p.bias + d0) : 0.f;
  }
  constexpr int SW = (int)((V * H * sizeof(TIn) + 3) / 4), XW = (int)((V * sizeof(TIn) + 3) / 4);
#pragma unroll
  for (int bs = 0; bs < BS; bs++) {
    if (b0 + bs >= p.batch) break;
    const int64_t c0 = (b0 + bs) * p.dim + d0;  // first channel, flattened over batch x dim
    TIn* st = static_cast<TIn*>(p.state_out) + c0 * H;
    const TIn* gx = static_cast<const TIn*>(p.x) + c0;
    uint32_t sw[SW], xw[XW];
    if constexpr (V > 1) {
#pragma unroll
      for (int i = 0; i < SW / 4; i++) {
        const uint4 q = reinterpret_cast<const uint4*>(st)[i];
        sw[4 * i] = q.x;
        sw[4 * i + 1] = q.y;
        sw[4 * i + 2] = q.z;
        sw[4 * i + 3] = q.w;
      }
#pragma unroll
      for (int i = 0; i < XW / 4; i++) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(gx) + i);
        xw[4 * i] = q.x;
        xw[4 * i + 1] = q.y;
        xw[4 * i + 2] = q.z;
        xw[4 * i + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < SW; i++) sw[i] = 0u;
      xw[0] = 0u;
#pragma unroll
      for (int k = 0; k < H; k++) set_word_elem<TIn>(sw, k, sizeof(TIn) == 4 ? __float_as_uint(to_f32(st[k])) : (uint32_t)__bfloat16_as_ushort(*reinterpret_cast<const __nv_bfloat16*>(st + k)));
      set_word_elem<TIn>(xw, 0, sizeof(TIn) == 4 ? __float_as_uint(to_f32(gx[0])) : (uint32_t)__bfloat16_as_ushort(*reinterpret_cast<const __nv_bfloat16*>(gx)));
    }
    float o[V];
#pragma unroll
    for (int v = 0; v < V; v++) {
      float acc = bias[v];
#pragma unroll
      for (int k = 0; k < H; k++) acc = fmaf(w[v * K + k], bits_f32<TIn>(word_elem<TIn>(sw, v * H + k)), acc);
      acc = fmaf(w[v * K + H], bits_f32<TIn>(word_elem<TIn>(xw, v)), acc);
      o[v] = SILU ? silu(acc) : acc;
    }
    store_out<TOut, V>(static_cast<TOut*>(p.y) + c0, o);
    // drop each channel's oldest input, append the new one
    uint32_t nw[SW];
#pragma unroll
    for (int i = 0; i < SW; i++) nw[i] = 0u;
#pragma unroll
    for (int v = 0; v < V; v++) {
#pragma unroll
      for (int k = 0; k + 1 < H; k++) set_word_elem<TIn>(nw, v * H + k, word_elem<TIn>(sw, v * H + k + 1));
      set_word_elem<TIn>(nw, v * H + H - 1, word_elem<TIn>(xw, v));
    }
    if constexpr (V > 1) {
#pragma unroll
      for (int i = 0; i < SW / 4; i++) reinterpret_cast<uint4*>(st)[i] = make_uint4(nw[4 * i], nw[4 * i + 1], nw[4 * i + 2], nw[4 * i + 3]);
    } else {
#pragma unroll
      for (int k = 0; k < H; k++) {
        const uint32_t bits = word_elem<TIn>(nw, k);
        if constexpr (sizeof(TIn) == 4) reinterpret_cast<float*>(st)[k] = __uint_as_float(bits);
        else reinterpret_cast<__nv_bfloat16*>(st)[k] = __ushort_as_bfloat16((unsigned short)bits);
      }
    }
  }
}


// ---------------------------------------------------------------- TMA-streamed forward pass
constexpr int kTT = 64;         // timesteps per tile
constexpr int kRing = 4;        // ring stages
constexpr int kCompute = 4;     // compute warps (plus one producer warp)
constexpr int kConvBar = 1;     // named barrier of the compute warps (0 is __syncthreads)

template <typename TIn, int K>
struct ConvTile {
  static constexpr int H = K - 1;
  static constexpr int CB = 256 / (int)sizeof(TIn);  // channels per tile (256-byte rows)
  static constexpr int ROWS = kTT + H;                // box height: the tile and its halo
  static constexpr int STAGE = ROWS * 256;            // bytes per ring stage (a multiple of 128)
  static constexpr int NPAIR = CB / 2;
  static constexpr int SPLIT = 32 * kCompute / NPAIR; // threads per channel pair (row ranges)
  static constexpr int RPT = kTT / SPLIT;             // output rows per thread
  static constexpr int OFF_BAR = kRing * STAGE;
  static constexpr int SMEM = OFF_BAR + 2 * kRing * 8 + 128;
};

// bulk-tensor store of a box of shared memory to global memory; the copy
// drops the box's elements that fall outside the tensor
__device__ __forceinline__ void conv_tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void conv_bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed store but the newest has finished reading shared memory
__device__ __forceinline__ void conv_bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void conv_bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void conv_bar_compute() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConvBar), "n"(32 * kCompute) : "memory");
}
// barrier of the compute warps that also ORs a flag over them
__device__ __forceinline__ bool conv_bar_or_compute(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConvBar), "n"(32 * kCompute)
      : "memory");
  return r != 0;
}

// Units of work are (channel block, batch element, tile), the tile varying
// fastest. CTA i takes the contiguous range [i n / G, (i + 1) n / G) of the n
// units, so its taps change only where the range crosses a channel block.
//
// When x and y have one type (kStage), y goes back into the stage it was
// computed from: stage row r + H holds timestep t0 + r of both. A thread
// overwrites a row only after its own last read of it, and the first H rows of
// a thread's range, which the range before it also writes, are read before the
// tile's first barrier. One bulk-tensor store per tile then writes the 64 rows;
// rows past the sequence end and channels past dim are dropped by the copy. The
// stage returns to the producer once that store has read it. Mixed types store
// y from registers.
template <typename TIn, typename TOut, int K, bool SILU>
__global__ void __launch_bounds__(32 * (kCompute + 1), 3) conv1d_fwd_tma_kernel(const __grid_constant__ ConvParams p,
                                                                            const __grid_constant__ CUtensorMap tm_x,
                                                                            const __grid_constant__ CUtensorMap tm_y) {
  using CT = ConvTile<TIn, K>;
  constexpr int H = CT::H, CB = CT::CB, NPAIR = CT::NPAIR, RPT = CT::RPT;
  constexpr bool kStage = std::is_same<TIn, TOut>::value;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + CT::OFF_BAR);
  uint64_t* empty = full + kRing;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kRing; i++) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kStage ? 1 : kCompute);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t L = p.seqlen, Dm = p.dim;
  const int64_t ntile = (L + kTT - 1) / kTT, ncb = (Dm + CB - 1) / CB;
  const int64_t nunits = p.batch * ntile * ncb;
  const int64_t G = gridDim.x;
  const int64_t u_begin = (int64_t)blockIdx.x * nunits / G, u_end = ((int64_t)blockIdx.x + 1) * nunits / G;
  // unit u: tile u % ntile, batch element (u / ntile) % batch, channel block u / (ntile * batch)

  if (warp == kCompute) {
    // ---- producer: one thread keeps the ring full
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      if (kStage) tma_prefetch_desc(&tm_y);
      int64_t k = 0;
      for (int64_t u = u_begin; u < u_end; u++, k++) {
        const int s = (int)(k % kRing);
        if (k >= kRing && !mbar_wait(&empty[s], (uint32_t)(((k / kRing) - 1) & 1))) {
          atomicOr(p.fault, kFaultTileWait);
          break;
        }
        const int64_t j = u % ntile, rest = u / ntile;
        const int64_t b = rest % p.batch, cbk = rest / p.batch;
        fence_proxy_async_smem();
        mbar_expect_tx(&full[s], CT::STAGE);
        tma_load_3d(smem + s * CT::STAGE, &tm_x, (int)(cbk * CB), (int)(j * kTT - H), (int)b, &full[s]);
        mbar_arrive(&full[s]);
      }
    }
    return;
  }

  // ---- compute warps: thread = (channel pair q, row range rr)
  const int q = tid % NPAIR, rr = tid / NPAIR;
  const int r0 = rr * RPT;  // first output row of the range in the tile
  const TIn* gs = static_cast<const TIn*>(p.state_in);
  f2 w2[K], bias2 = pk(0.f, 0.f);  // taps and bias of the pair: w2[k] = (w[d][k], w[d+1][k])
  int64_t wcb = -1;                // channel block the taps belong to
  int64_t k = 0;
  for (int64_t u = u_begin; u < u_end; u++, k++) {
    const int s = (int)(k % kRing);
    const int64_t j = u % ntile, rest = u / ntile;
    const int64_t b = rest % p.batch, cbk = rest / p.batch;
    const int64_t t0 = j * kTT, d = cbk * CB + 2 * q;  // first timestep of the tile, first channel of the pair
    const bool dv = d < Dm;                           // Dm is even here: the pair is whole or absent
    if (cbk != wcb) {  // CTA-uniform; the loads overlap the wait below
      wcb = cbk;
      if (dv) {
        float wf[2 * K];
#pragma unroll
        for (int i = 0; i < K; i++) {  // 2K contiguous floats, 8-byte aligned (d even)
          const float2 v = __ldg(reinterpret_cast<const float2*>(p.w + d * K) + i);
          wf[2 * i] = v.x;
          wf[2 * i + 1] = v.y;
        }
#pragma unroll
        for (int i = 0; i < K; i++) w2[i] = pk(wf[i], wf[K + i]);
        bias2 = pk(0.f, 0.f);
        if (p.bias) {
          const float2 bv = __ldg(reinterpret_cast<const float2*>(p.bias + d));
          bias2 = pk(bv.x, bv.y);
        }
      } else {
#pragma unroll
        for (int i = 0; i < K; i++) w2[i] = pk(0.f, 0.f);
        bias2 = pk(0.f, 0.f);
      }
    }
    const bool ok = mbar_wait(&full[s], (uint32_t)((k / kRing) & 1));
    if constexpr (!kStage) {
      if (__any_sync(0xffffffffu, !ok)) {  // warp-uniform
        if (lane == 0) atomicOr(p.fault, kFaultTileWait);
        break;
      }
    }
    TIn* tile = reinterpret_cast<TIn*>(smem + s * CT::STAGE);  // row i = timestep t0 - H + i
    // rows before t = 0 (zero-filled by the load) come from the carried state;
    // only the thread range that reads them patches its own pair's columns
    const bool patch = ok && j == 0 && gs && rr == 0 && dv;
    if (patch) {
#pragma unroll
      for (int i = 0; i < H; i++) {
        tile[i * CB + 2 * q] = gs[(b * Dm + d) * H + i];
        tile[i * CB + 2 * q + 1] = gs[(b * Dm + d + 1) * H + i];
      }
    }
    // the tile holding the last timestep hands on the last H inputs (raw bits),
    // read before any y overwrites them
    const bool hand_on = ok && p.state_out && j == ntile - 1 && rr == 0 && dv;
    auto hand_on_state = [&]() {
      TIn* so = static_cast<TIn*>(p.state_out);
#pragma unroll
      for (int i = 0; i < H; i++) {
        const int64_t row = (L - H + i) - (t0 - H);  // tile row of timestep L-H+i (>= 0: t0 <= L-1)
        so[(b * Dm + d) * H + i] = tile[row * CB + 2 * q];
        so[(b * Dm + d + 1) * H + i] = tile[row * CB + 2 * q + 1];
      }
    };
    if (kStage && hand_on) hand_on_state();
    auto ld_pair = [&](int row) -> f2 {  // widened (channel d, channel d+1) of tile row `row`
      if constexpr (sizeof(TIn) == 4) {
        const float2 v = *reinterpret_cast<const float2*>(tile + row * CB + 2 * q);
        return pk(v.x, v.y);
      } else {
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(tile + row * CB + 2 * q);
        return pk(__uint_as_float(wd << 16), __uint_as_float(wd & 0xffff0000u));
      }
    };
    // sliding window over the tile rows r .. r+H for output row r
    f2 win[K];
#pragma unroll
    for (int i = 0; i < H; i++) win[i] = ld_pair(r0 + i);
    if constexpr (kStage) {
      if (conv_bar_or_compute(!ok)) {  // CTA-uniform
        if (tid == 0) atomicOr(p.fault, kFaultTileWait);
        break;
      }
#pragma unroll
      for (int r = 0; r < RPT; r++) {
        win[H] = ld_pair(r0 + r + H);
        f2 a = bias2;
#pragma unroll
        for (int i = 0; i < K; i++) a = fma2(w2[i], win[i], a);
        if (SILU) a = silu2(a);
        TIn* dst = tile + (r0 + r + H) * CB + 2 * q;
        if constexpr (sizeof(TIn) == 2) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(f2lo(a), f2hi(a));
          *reinterpret_cast<__nv_bfloat162*>(dst) = h2;
        } else {
          *reinterpret_cast<float2*>(dst) = make_float2(f2lo(a), f2hi(a));
        }
#pragma unroll
        for (int i = 0; i < H; i++) win[i] = win[i + 1];
      }
      // order this thread's y writes before the bulk store's reads
      fence_proxy_async_smem();
      conv_bar_compute();
      if (tid == 0) {
        conv_tma_store_3d(&tm_y, smem + s * CT::STAGE + H * 256, (int)(cbk * CB), (int)t0, (int)b);
        conv_bulk_commit();
        // the previous tile's store has read its stage: hand that stage back
        conv_bulk_wait_read1();
        if (k > 0) mbar_arrive(&empty[(int)((k - 1) % kRing)]);
      }
    } else {
      TOut* yrow = static_cast<TOut*>(p.y) + (b * L + t0 + r0) * Dm + d;
#pragma unroll 8
      for (int r = 0; r < RPT; r++) {
        win[H] = ld_pair(r0 + r + H);
        f2 a = bias2;
#pragma unroll
        for (int i = 0; i < K; i++) a = fma2(w2[i], win[i], a);
        if (SILU) a = silu2(a);
        if (dv && t0 + r0 + r < L) {
          if constexpr (sizeof(TOut) == 2) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(f2lo(a), f2hi(a));
            __stcs(reinterpret_cast<unsigned int*>(yrow), *reinterpret_cast<const unsigned int*>(&h2));
          } else {
            __stcs(reinterpret_cast<float2*>(yrow), make_float2(f2lo(a), f2hi(a)));
          }
        }
        yrow += Dm;
#pragma unroll
        for (int i = 0; i < H; i++) win[i] = win[i + 1];
      }
      if (hand_on) hand_on_state();
      // the stage may be refilled by the next load: order this thread's
      // shared-memory writes before that async-proxy write
      if (patch) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  // shared memory must outlive the reads of the stores in flight
  if (kStage && tid == 0) conv_bulk_wait_all();
}

using ConvEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline ConvEncodeFn conv_encode_fn() {
  static const ConvEncodeFn fn = []() -> ConvEncodeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<ConvEncodeFn>(f);
    return nullptr;
  }();
  return fn;
}

template <typename TIn, typename TOut, int K>
cudaError_t launch_fwd_tma(const ConvParams& p, cudaStream_t s) {
  using CT = ConvTile<TIn, K>;
  constexpr bool kStage = std::is_same<TIn, TOut>::value;
  ConvEncodeFn fn = conv_encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  CUtensorMap mx{}, my{};
  const size_t es = sizeof(TIn);
  cuuint64_t dims[3] = {(cuuint64_t)p.dim, (cuuint64_t)p.seqlen, (cuuint64_t)p.batch};
  cuuint64_t strides[2] = {(cuuint64_t)p.dim * es, (cuuint64_t)p.seqlen * p.dim * es};
  cuuint32_t box[3] = {(cuuint32_t)CT::CB, (cuuint32_t)CT::ROWS, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (fn(&mx, dt, 3, const_cast<void*>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (kStage) {  // y: the same shape and type as x, stored 64 rows at a time
    cuuint32_t ybox[3] = {(cuuint32_t)CT::CB, (cuuint32_t)kTT, 1};
    if (fn(&my, dt, 3, p.y, dims, strides, ybox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    my = mx;  // unused
  }
  const int64_t ntile = (p.seqlen + kTT - 1) / kTT, ncb = (p.dim + CT::CB - 1) / CT::CB;
  const int64_t nunits = p.batch * ntile * ncb;
  const int sms = device_sm_count();
  const int64_t grid = std::min<int64_t>(nunits, 3 * (int64_t)sms);  // three CTAs per SM
  auto kern = p.silu ? conv1d_fwd_tma_kernel<TIn, TOut, K, true> : conv1d_fwd_tma_kernel<TIn, TOut, K, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CT::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, 32 * (kCompute + 1), CT::SMEM, s>>>(p, mx, my);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int K, int V>
cudaError_t launch_fwd_kv(const ConvParams& p, cudaStream_t s) {
  const int64_t nt = (p.seqlen + kConvTT - 1) / kConvTT;
  const int64_t n = p.batch * nt * (p.dim / V);
  const int64_t blocks = (n + kConvThreads - 1) / kConvThreads;
  if (p.silu) conv1d_fwd_kernel<TIn, TOut, K, V, true><<<(unsigned)blocks, kConvThreads, 0, s>>>(p);
  else conv1d_fwd_kernel<TIn, TOut, K, V, false><<<(unsigned)blocks, kConvThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename TIn, typename TOut, int K>
cudaError_t launch_fwd_k(const ConvParams& p, bool vec, cudaStream_t s) {
  // 16-byte-aligned rows stream through shared memory by TMA; others take the
  // per-thread window kernel, one channel per thread
  return vec ? launch_fwd_tma<TIn, TOut, K>(p, s) : launch_fwd_kv<TIn, TOut, K, 1>(p, s);
}

template <typename TIn, typename TOut>
cudaError_t launch_fwd_io(const ConvParams& p, bool vec, cudaStream_t s) {
  switch (p.width) {
    case 2: return launch_fwd_k<TIn, TOut, 2>(p, vec, s);
    case 3: return launch_fwd_k<TIn, TOut, 3>(p, vec, s);
    case 4: return launch_fwd_k<TIn, TOut, 4>(p, vec, s);
  }
  return cudaErrorInvalidValue;
}

template <typename TIn, typename TOut, int K, int V>
cudaError_t launch_upd_kv(const ConvParams& p, cudaStream_t s) {
  constexpr int BS = V > 1 ? 4 : 1;  // streams per thread, sharing the loaded taps
  const int64_t threads = (p.batch + BS - 1) / BS * ((p.dim + V - 1) / V);
  const int64_t blocks = (threads + kConvThreads - 1) / kConvThreads;
  if (p.silu) conv1d_update_kernel<TIn, TOut, K, V, true, BS><<<(unsigned)blocks, kConvThreads, 0, s>>>(p);
  else conv1d_update_kernel<TIn, TOut, K, V, false, BS><<<(unsigned)blocks, kConvThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_upd_io(const ConvParams& p, bool vec, cudaStream_t s) {
  constexpr int VV = 16 / (int)sizeof(TIn);
  switch (p.width) {
    case 2: return vec ? launch_upd_kv<TIn, TOut, 2, VV>(p, s) : launch_upd_kv<TIn, TOut, 2, 1>(p, s);
    case 3: return vec ? launch_upd_kv<TIn, TOut, 3, VV>(p, s) : launch_upd_kv<TIn, TOut, 3, 1>(p, s);
    case 4: return vec ? launch_upd_kv<TIn, TOut, 4, VV>(p, s) : launch_upd_kv<TIn, TOut, 4, 1>(p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_conv1d_fwd(const ConvParams& p, ss_dtype in_dtype, ss_dtype out_dtype, bool vec,
                              cudaStream_t stream) {
  if (in_dtype == SS_BF16)
    return out_dtype == SS_BF16 ? launch_fwd_io<__nv_bfloat16, __nv_bfloat16>(p, vec, stream)
                                : launch_fwd_io<__nv_bfloat16, float>(p, vec, stream);
  return out_dtype == SS_BF16 ? launch_fwd_io<float, __nv_bfloat16>(p, vec, stream)
                              : launch_fwd_io<float, float>(p, vec, stream);
}

cudaError_t launch_conv1d_update(const ConvParams& p, ss_dtype in_dtype, ss_dtype out_dtype, bool vec,
                                 cudaStream_t stream) {
  if (in_dtype == SS_BF16)
    return out_dtype == SS_BF16 ? launch_upd_io<__nv_bfloat16, __nv_bfloat16>(p, vec, stream)
                                : launch_upd_io<__nv_bfloat16, float>(p, vec, stream);
  return out_dtype == SS_BF16 ? launch_upd_io<float, __nv_bfloat16>(p, vec, stream)
                              : launch_upd_io<float, float>(p, vec, stream);
}

}  // namespace ssk
