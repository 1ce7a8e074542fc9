// State-space-dual (Mamba-2) layer forward on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA), for
// d_state 128.
//
// Per batch element and head h (scalar decay A_h, head channels p < 64,
// state n < 128), with delta_t = softplus(dt_t + dt_bias_h):
//   H_t = exp(delta_t A_h) H_{t-1} + delta_t x_t B_t^T      ([P, N])
//   y_t = H_t C_t + D_h x_t
// The decay being one scalar per head, the sequence splits into chunks whose
// outputs are matrix products ("AI 推理系列（十四）：Mamba 的 Selective State
// Space", section on Mamba-2 reorganising the SSM as matrix computation;
// mlqm.cn tutorial, section 8). For a chunk of Q = 128 steps, with cs_t the
// decay (base 2) accumulated inside the chunk and H_in the state entering it:
//   S = C B^T                                  [t, s]  (K = n)
//   M = S o 2^(cs_t - cs_s) o delta_s, s <= t  (else 0)
//   Y = M X + 2^cs_t o (C H_in^T) + D X        [t, p]  (K = s, K = n)
//   H_out^T = 2^cs_end H_in^T + W^T X,  W = B o 2^(cs_end - cs_s) delta_s   [n, p]  (K = s)
//
// One CTA of four warps owns one (batch, head) and walks its chunks in order;
// the state stays in registers (thread n holds row n of H^T). Per chunk:
//  - one thread loads the chunk's C and B (two 64-column boxes each) and x by
//    TMA with 128-byte swizzling, the layout the tensor core reads;
//  - S = C B^T runs as eight K=16 steps of tcgen05.mma (M = 128 rows t, N =
//    128 columns s) into tensor memory;
//  - thread t reads row t of S from tensor memory (tcgen05.ld) and writes row t
//    of M; thread s turns row s of B into row s of W in place (B is read only
//    by S); M, W and the state are computed in fp32 and enter the products as
//    a bf16 high part and a bf16 remainder (two products each, about 16
//    significant bits); x, B and C enter as the stored bf16 values;
//  - Y1 = M X, Y2 = C H_in^T and H_l^T = W^T X run on the tensor core
//    (operands in shared memory, K-major or MN-major descriptors);
//  - thread t writes y_t = Y1_t + 2^cs_t Y2_t + D x_t; thread n updates row n of
//    the state, H^T = 2^cs_end H^T + H_l^T, and writes its two parts for the
//    next chunk's Y2.
// Every wait is bounded and reports a timeout through the library fault word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ss_device.cuh"
#include "ss_internal.h"

namespace ssk {
namespace {

constexpr int kQ = 128;  // chunk length (the rows of every product)
constexpr int kP = 64;   // head channels
constexpr int kN = 128;  // state size
constexpr int kThreads = 256;  // two threads per row of a product, each taking half its columns
constexpr uint32_t kTmemCols = 512;  // S [0,128), Y1 [128,192), Y2 [192,256), H_l [256,320)
constexpr uint32_t kColS = 0, kColY1 = 128, kColY2 = 192, kColH = 256;

// Shared-memory layout (offsets from a 1024-byte aligned base). A "tile" is
// 128 rows of 128 bytes (64 bf16) in the 128-byte swizzle: the 16-byte piece c
// of row r sits at piece c ^ (r % 8).
struct TcSmem {
  static constexpr int TILE = 128 * 128;      // 16 KB
  static constexpr int C0 = 0;                // C [t][n 0..63], C1 = n 64..127
  static constexpr int C1 = C0 + TILE;
  static constexpr int B0 = C1 + TILE;        // B [s][n 0..63] (then W's high part), B1 = n 64..127
  static constexpr int B1 = B0 + TILE;
  static constexpr int WL0 = B1 + TILE;       // W's remainder [s][n 0..63], WL1 = n 64..127
  static constexpr int WL1 = WL0 + TILE;
  static constexpr int X = WL1 + TILE;        // x [s][p]
  static constexpr int MH0 = X + TILE;        // M high [t][s 0..63], MH1 = s 64..127
  static constexpr int MH1 = MH0 + TILE;
  static constexpr int ML0 = MH1 + TILE;      // M remainder
  static constexpr int ML1 = ML0 + TILE;
  static constexpr int HH = ML1 + TILE;       // H^T high [n][p]
  static constexpr int HL = HH + TILE;        // H^T remainder
  static constexpr int DL = HL + TILE;        // delta_t [128] f32
  static constexpr int CS = DL + 512;         // cs_t [128] f32
  static constexpr int WSUM = CS + 512;       // warp sums of the prefix scan [4] f32
  static constexpr int BAR = WSUM + 64;       // mbarriers: tma_cb, tma_x, mma_s, mma_rest
  static constexpr int TSLOT = BAR + 64;      // tensor-memory base address
  static constexpr int BYTES = TSLOT + 64;
  static constexpr int ALLOC = BYTES + 1024;  // + alignment slack
};

__device__ __forceinline__ int sw128(int r, int c) {  // byte offset of bf16 (r, c) in a tile
  return r * 128 + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1);
}

// Shared-memory matrix descriptor: 128-byte swizzle, the given leading and
// stride byte offsets (the sm_100 descriptor format: start address, LBO, SBO
// in 16-byte units; version 1; layout type 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}
// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, A/B major
// (0 = K-major, 1 = MN-major), N >> 3, M >> 4
__device__ __forceinline__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"(accumulate ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's tensor-memory lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}
// 4-D tiled TMA load (coordinates innermost first)
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
// eight floats -> eight bf16 (16 bytes), high part and remainder
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const __nv_bfloat162 hh = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const float2 hf = __bfloat1622float2(hh);
    const __nv_bfloat162 ll = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    h[i] = *reinterpret_cast<const uint32_t*>(&hh);
    l[i] = *reinterpret_cast<const uint32_t*>(&ll);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void widen8(uint4 w, float (&v)[8]) {
  const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    v[2 * i] = __uint_as_float(a[i] << 16);
    v[2 * i + 1] = __uint_as_float(a[i] & 0xffff0000u);
  }
}

template <typename TOut>
__global__ void __launch_bounds__(kThreads, 1) ssd_tc_kernel(const __grid_constant__ SsdParams p,
                                                            const __grid_constant__ CUtensorMap tm_x,
                                                            const __grid_constant__ CUtensorMap tm_b,
                                                            const __grid_constant__ CUtensorMap tm_c) {
  using SM = TcSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(sm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SM::BAR);  // 0 C and B, 1 x, 2 S product, 3 the other products
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM::TSLOT);
  float* dls = reinterpret_cast<float*>(sm + SM::DL);
  float* css = reinterpret_cast<float*>(sm + SM::CS);
  float* wsum = reinterpret_cast<float*>(sm + SM::WSUM);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kQ - 1);  // row of the products this thread reads and writes
  const int hf = tid >> 7;         // which half of the columns
  const int wq = warp & 3;         // the warp's tensor-memory lane quarter: rows 32wq .. 32wq+31
  const int64_t bh = blockIdx.x;
  const int64_t b = bh / p.nheads, h = bh % p.nheads;
  const int64_t L = p.seqlen, H = p.nheads, G = p.ngroups;
  const int grp = (int)(h / (H / G));
  const float a2 = __ldg(p.A + h) * kLog2e;  // decay exponent per unit delta, base 2
  const float dtb = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
  const float Dh = p.D ? __ldg(p.D + h) : 0.f;
  const __nv_bfloat16* DT = static_cast<const __nv_bfloat16*>(p.dt);
  const int64_t nchunk = (L + kQ - 1) / kQ;
  const uint64_t wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;

  if (tid == 0) {
    for (int i = 0; i < 4; i++) mbar_init(&bar[i], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tlane = tmem + ((uint32_t)(wq * 32) << 16);  // this warp's tensor-memory lanes

  // what thread 0 has issued and nobody has waited for yet (for the drain
  // after a timed-out wait), and the phase each barrier is at
  bool pend[4] = {false, false, false, false};
  uint32_t ph[4] = {0, 0, 0, 0};
  auto issue_cb = [&](int64_t c) {
    const int t0 = (int)(c * kQ);
    mbar_expect_tx(&bar[0], 4 * SM::TILE);
    tma_load_4d(sm + SM::C0, &tm_c, 0, grp, t0, (int)b, &bar[0]);
    tma_load_4d(sm + SM::C1, &tm_c, 64, grp, t0, (int)b, &bar[0]);
    tma_load_4d(sm + SM::B0, &tm_b, 0, grp, t0, (int)b, &bar[0]);
    tma_load_4d(sm + SM::B1, &tm_b, 64, grp, t0, (int)b, &bar[0]);
    mbar_arrive(&bar[0]);
    pend[0] = true;
  };
  auto issue_x = [&](int64_t c) {
    mbar_expect_tx(&bar[1], SM::TILE);
    tma_load_4d(sm + SM::X, &tm_x, 0, (int)h, (int)(c * kQ), (int)b, &bar[1]);
    mbar_arrive(&bar[1]);
    pend[1] = true;
  };
  // every thread waits for barrier i; false (for the whole CTA) if any gave up
  auto wait_all = [&](int i) -> bool {
    const bool mine = mbar_wait(&bar[i], ph[i], wait_ns);
    if (__syncthreads_or(mine ? 0 : 1)) {
      if (tid == 0) atomicOr(p.fault, kFaultTileWait);
      return false;
    }
    ph[i] ^= 1u;
    pend[i] = false;
    return true;
  };

  // the state: thread (row n, half hf) holds H^T[n][32 hf .. 32 hf + 31]
  float hst[32];
  {
    const float* h0 = p.h0 ? p.h0 + (b * H + h) * kP * kN : nullptr;
#pragma unroll
    for (int q = 0; q < 32; q++) hst[q] = h0 ? __ldg(h0 + (32 * hf + q) * kN + row) : 0.f;
  }
  // the state's two bf16 parts, row n of H^T, for the next chunk's C H^T
  auto write_state = [&]() {
#pragma unroll
    for (int c8 = 0; c8 < 4; c8++) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; i++) v[i] = hst[8 * c8 + i];
      uint4 hi, lo;
      split8(v, hi, lo);
      *reinterpret_cast<uint4*>(sm + SM::HH + sw128(row, 32 * hf + 8 * c8)) = hi;
      *reinterpret_cast<uint4*>(sm + SM::HL + sw128(row, 32 * hf + 8 * c8)) = lo;
    }
  };
  bool state_nonzero = p.h0 != nullptr;
  if (state_nonzero) write_state();

  if (tid == 0 && nchunk > 0) {
    issue_cb(0);
    issue_x(0);
  }
  bool ok = true;  // CTA-uniform: no wait has timed out
  for (int64_t c = 0; c < nchunk; c++) {
    const int64_t t0 = c * kQ;
    // ---- delta and the decay (base 2) accumulated inside the chunk, inclusive
    {
      float dl = 0.f, sc = 0.f;
      if (hf == 0) {
        dl = t0 + row < L ? softplus_fast(__bfloat162float(DT[(b * L + t0 + row) * H + h]) + dtb) : 0.f;
        sc = dl * a2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += v;
        }
        if (lane == 31) wsum[warp] = sc;
      }
      __syncthreads();
      if (hf == 0) {
        for (int w = 0; w < warp; w++) sc += wsum[w];
        dls[row] = dl;
        css[row] = sc;
      }
      __syncthreads();
    }
    // ---- S = C B^T
    if (!(ok = wait_all(0))) break;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc(kQ, kQ, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        const uint32_t off = (kk & 3) * 32;
        const uint64_t ad = sdesc(s0 + (kk < 4 ? SM::C0 : SM::C1) + off, 16, 1024);
        const uint64_t bd = sdesc(s0 + (kk < 4 ? SM::B0 : SM::B1) + off, 16, 1024);
        mma(tmem + kColS, ad, bd, id, kk > 0);
      }
      mma_commit(&bar[2]);
      pend[2] = true;
    }
    if (!(ok = wait_all(2))) break;
    tc_fence_after();
    // ---- M (row t, columns s in half hf) from S; W (row s, columns n in half hf) in place of B
    {
      const float cst = css[row];
#pragma unroll 1
      for (int j = 0; j < 2; j++) {
        const int sb = 64 * hf + 32 * j;  // first column s of this block of 32
        float sv[32];
        const bool any = sb <= 32 * wq + 31;  // warp-uniform: some row of the warp reaches column sb
        if (any) tmem_ld32(tlane + kColS + sb, sv);
#pragma unroll
        for (int c8 = 0; c8 < 4; c8++) {
          float v[8];
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const int s = sb + c8 * 8 + i;
            v[i] = (any && s <= row) ? sv[c8 * 8 + i] * ex2(cst - css[s]) * dls[s] : 0.f;
          }
          uint4 hi, lo;
          split8(v, hi, lo);
          const int col = 32 * j + 8 * c8;
          *reinterpret_cast<uint4*>(sm + (hf ? SM::MH1 : SM::MH0) + sw128(row, col)) = hi;
          *reinterpret_cast<uint4*>(sm + (hf ? SM::ML1 : SM::ML0) + sw128(row, col)) = lo;
        }
      }
      const float ws = ex2(css[kQ - 1] - css[row]) * dls[row];  // 2^(cs_end - cs_s) delta_s, s = row
#pragma unroll
      for (int c8 = 0; c8 < 8; c8++) {
        uint8_t* pb = sm + (hf ? SM::B1 : SM::B0) + sw128(row, 8 * c8);
        float v[8];
        widen8(*reinterpret_cast<const uint4*>(pb), v);
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] *= ws;
        uint4 hi, lo;
        split8(v, hi, lo);
        *reinterpret_cast<uint4*>(pb) = hi;
        *reinterpret_cast<uint4*>(sm + (hf ? SM::WL1 : SM::WL0) + sw128(row, 8 * c8)) = lo;
      }
    }
    fence_proxy_async_smem();  // M, W and the state are read by the tensor core next
    if (!(ok = wait_all(1))) break;  // x of the chunk; also orders the writes above before the issue
    // ---- Y1 = M X, H_l^T = W^T X, Y2 = C H_in^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idy = idesc(kQ, kP, 0, 1);  // A K-major (M or C), B MN-major (x or H^T)
      const uint32_t idh = idesc(kN, kP, 1, 1);  // A MN-major (W), B MN-major (x)
#pragma unroll
      for (int part = 0; part < 2; part++) {
        const int mb0 = part ? SM::ML0 : SM::MH0, mb1 = part ? SM::ML1 : SM::MH1;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint64_t ad = sdesc(s0 + (kk < 4 ? mb0 : mb1) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc(s0 + SM::X + kk * 2048, 16, 1024);
          mma(tmem + kColY1, ad, bd, idy, part > 0 || kk > 0);
        }
      }
#pragma unroll
      for (int part = 0; part < 2; part++) {
        // the two 64-column halves (n < 64, n >= 64) of W are one tile apart
        const int wb = part ? SM::WL0 : SM::B0;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint64_t ad = sdesc(s0 + wb + kk * 2048, SM::TILE, 1024);
          const uint64_t bd = sdesc(s0 + SM::X + kk * 2048, 16, 1024);
          mma(tmem + kColH, ad, bd, idh, part > 0 || kk > 0);
        }
      }
      if (state_nonzero) {
#pragma unroll
        for (int part = 0; part < 2; part++) {
          const int hb = part ? SM::HL : SM::HH;
#pragma unroll
          for (int kk = 0; kk < 8; kk++) {
            const uint64_t ad = sdesc(s0 + (kk < 4 ? SM::C0 : SM::C1) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc(s0 + hb + kk * 2048, 16, 1024);
            mma(tmem + kColY2, ad, bd, idy, part > 0 || kk > 0);
          }
        }
      }
      mma_commit(&bar[3]);
      pend[3] = true;
    }
    if (!(ok = wait_all(3))) break;
    tc_fence_after();
    // C, B (now W) and M are no longer read: load the next chunk's C and B
    if (tid == 0 && c + 1 < nchunk) issue_cb(c + 1);
    // ---- y of row t, columns p in half hf: Y1 + 2^cs_t Y2 + D x
    {
      const float et = ex2(css[row]);
      const int pb = 32 * hf;
      float y1[32], y2[32];
      tmem_ld32(tlane + kColY1 + pb, y1);
      if (state_nonzero) tmem_ld32(tlane + kColY2 + pb, y2);
      if (t0 + row < L) {
        TOut* yrow = static_cast<TOut*>(p.y) + ((b * L + t0 + row) * H + h) * kP + pb;
#pragma unroll
        for (int c8 = 0; c8 < 4; c8++) {
          float xv[8], o[8];
          widen8(*reinterpret_cast<const uint4*>(sm + SM::X + sw128(row, pb + c8 * 8)), xv);
#pragma unroll
          for (int i = 0; i < 8; i++) {
            const float yy = state_nonzero ? fmaf(et, y2[c8 * 8 + i], y1[c8 * 8 + i]) : y1[c8 * 8 + i];
            o[i] = fmaf(Dh, xv[i], yy);
          }
          if constexpr (sizeof(TOut) == 2) {
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
              w4[i] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            *reinterpret_cast<uint4*>(yrow + c8 * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          } else {
            *reinterpret_cast<float4*>(yrow + c8 * 8) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(yrow + c8 * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
    // ---- the state, row n of H^T: 2^cs_end H^T + H_l^T
    {
      const float dec = ex2(css[kQ - 1]);
      float hl[32];
      tmem_ld32(tlane + kColH + 32 * hf, hl);
#pragma unroll
      for (int i = 0; i < 32; i++) hst[i] = fmaf(dec, hst[i], hl[i]);
      write_state();
      state_nonzero = true;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // x is no longer read; the state is written for the next chunk
    if (tid == 0 && c + 1 < nchunk) issue_x(c + 1);
  }

  if (ok) {
    if (p.h_last) {
      float* hl = p.h_last + (b * H + h) * kP * kN;
#pragma unroll
      for (int q = 0; q < 32; q++) hl[(32 * hf + q) * kN + row] = hst[q];
    }
  } else if (tid == 0) {
    // a wait gave up: wait (bounded) for what this CTA still has in flight
    // before its shared and tensor memory are released
    for (int i = 0; i < 4; i++)
      if (pend[i]) mbar_wait(&bar[i], ph[i], wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

using TcEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TcEncodeFn tc_encode_fn() {
  static const TcEncodeFn fn = []() -> TcEncodeFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<TcEncodeFn>(f);
    return nullptr;
  }();
  return fn;
}

// 4-D bf16 map over a row-major [d3, d2, d1, d0] tensor with a [1, 128, 1, 64]
// box (64 innermost elements = 128 bytes, 128 rows of d2) in the 128-byte swizzle
bool make_map_4d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3) {
  TcEncodeFn fn = tc_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)kQ, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TOut>
cudaError_t launch_tc(const SsdParams& p, cudaStream_t s) {
  CUtensorMap mx{}, mb{}, mc{};
  // x [batch, L, H, 64]; B, C [batch, L, G, 128]
  if (!make_map_4d(&mx, p.x, kP, (uint64_t)p.nheads, (uint64_t)p.seqlen, (uint64_t)p.batch) ||
      !make_map_4d(&mb, p.B, kN, (uint64_t)p.ngroups, (uint64_t)p.seqlen, (uint64_t)p.batch) ||
      !make_map_4d(&mc, p.C, kN, (uint64_t)p.ngroups, (uint64_t)p.seqlen, (uint64_t)p.batch))
    return cudaErrorInvalidValue;
  auto k = ssd_tc_kernel<TOut>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::ALLOC);
  if (e != cudaSuccess) return e;
  k<<<(unsigned)(p.batch * p.nheads), kThreads, TcSmem::ALLOC, s>>>(p, mx, mb, mc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_fwd_tc(const SsdParams& p, ss_dtype out_dtype, cudaStream_t stream) {
  return out_dtype == SS_BF16 ? launch_tc<__nv_bfloat16>(p, stream) : launch_tc<float>(p, stream);
}

}  // namespace ssk
