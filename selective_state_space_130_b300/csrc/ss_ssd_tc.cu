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
//   S = C B^T                                              [t, s]  (K = n)
//   M = S o 2^(cs_t - cs_s) o delta_s for s <= t, else 0; plus D_h on the diagonal
//   Y = M X + 2^cs_t o (C H_in^T)                           [t, p]  (K = s, K = n)
//   H_out^T = 2^cs_end H_in^T + B^T X',  X' = diag(2^(cs_end - cs_s) delta_s) X   [n, p]  (K = s)
//
// One CTA owns one (batch, head) and walks its chunks in order. One thread of
// a ninth warp issues every TMA copy and tensor-core product; eight compute
// warps (two threads per row of a product, each taking half its columns) do
// the element-wise work and signal the issuer through mbarriers, so no
// compute thread ever waits for an issue. Per chunk:
//  - C and B (two 64-column boxes each) and x arrive by TMA in the 128-byte
//    swizzle, the layout the tensor core reads; each load is issued as soon as
//    the previous chunk's products have released its buffer;
//  - S = C B^T and Y2 = C H_in^T go to the tensor core first (Y2 needs only the
//    state entering the chunk); the compute threads meanwhile take delta and
//    the decay sums (dt was fetched a chunk ahead by cp.async);
//  - they scale row s of x by its state weight into X' (then B^T X' runs), and
//    turn row t of S, read from tensor memory, into row t of M, written back
//    over S (then M X runs with A read from tensor memory);
//  - the state H^T = 2^cs_end H^T + B^T X', kept in tensor memory, is updated
//    and its two parts written to shared memory for the next chunk's Y2; y_t =
//    Y1_t + 2^cs_t Y2_t is staged in shared memory and written by TMA.
// M, X' and the state are computed in fp32 and enter the products as a bf16
// high part and a bf16 remainder (about 16 significant bits; the two parts sit
// side by side along N where they are the B operand, so one N = 128 product
// covers both); x, B and C enter as the stored bf16 values.
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
constexpr int kComputeWarps = 8;  // two threads per row of a product, each taking half its columns
constexpr int kCompute = 32 * kComputeWarps;
// + three warps whose first lanes issue the copies and products: a single
// thread issues about one tcgen05.mma per hundred-odd cycles whatever its N,
// and several issuing warps overlap, so independent products go to different
// issuers
constexpr int kIssuers = 3;
constexpr int kThreads = kCompute + 32 * kIssuers;
// The compute thread that issues the y stores: one outside warps 0-3, which
// compute the chunk's scalars (its waits on the stores stay off their path).
constexpr int kStoreTid = 128;
// Tensor-memory columns: S (then M) [0,128); Y1 as two accumulators, over s
// < 64 [128,192) and over s >= 64 [192,256); Y2 [256,320) (the products with
// the state's high part and with its remainder, summed); H_l [320,448) (with
// X''s high part, then its remainder, side by side); the state [448,512)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColY1a = 128, kColY1b = 192, kColY2 = 256, kColH = 320, kColState = 448;

// Shared-memory layout (offsets from a 1024-byte aligned base). A "tile" is
// 128 rows of 128 bytes (64 bf16) in the 128-byte swizzle: the 16-byte piece c
// of row r sits at piece c ^ (r % 8).
struct TcSmem {
  static constexpr int TILE = 128 * 128;      // 16 KB
  static constexpr int C0 = 0;                // C [t][n 0..63], C1 = n 64..127
  static constexpr int C1 = C0 + TILE;
  static constexpr int B0 = C1 + TILE;        // B [s][n 0..63], B1 = n 64..127
  static constexpr int B1 = B0 + TILE;
  static constexpr int XH = B1 + TILE;        // X' high [s][p]
  static constexpr int XL = XH + TILE;        // X' remainder
  static constexpr int X0 = XL + TILE;        // x [s][p] of even chunks, X1 of odd ones
  static constexpr int X1 = X0 + TILE;
  static constexpr int YS0 = X1 + TILE;       // y staged for its TMA store [t][p] (bf16: one tile; fp32: two)
  static constexpr int YS1 = YS0 + TILE;
  static constexpr int HH = YS1 + TILE;       // H^T high [n][p]
  static constexpr int HL = HH + TILE;        // H^T remainder
  static constexpr int DL = HL + TILE;        // delta_t of two chunks [2][128] f32
  static constexpr int CS = DL + 1024;        // cs_t of two chunks [2][128] f32
  static constexpr int WSUM = CS + 1024;      // warp sums of the prefix scans [2][4] f32
  static constexpr int QS = WSUM + 64;        // q_s of two chunks [2][128] f32 (see the kernel)
  static constexpr int DTB = QS + 1024;       // dt words of two chunks [2][128] u32 (see the kernel)
  static constexpr int BAR = DTB + 1024;      // mbarriers, see the kernel (at most 16)
  static constexpr int TSLOT = BAR + 128;     // tensor-memory base address, the CTA's ticket, then its range (RangeDesc)
  static constexpr int BYTES = TSLOT + 64;
  static constexpr int ALLOC = BYTES + 1024;  // + alignment slack
};

// A CTA's range of chunks as the segments it runs, in shared memory: read at
// each segment's start, not held in registers through the chunk loops.
struct RangeDesc {
  int64_t u0;    // the range's first sequence
  int nseg;      // sequences it touches
  int cb_first;  // its first chunk in sequence u0
  int ce_last;   // one past its last chunk in sequence u0 + nseg - 1
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
// the same with A read from tensor memory (row i in lane i, two bf16 of
// consecutive K per 32-bit column, the even one in the low half)
__device__ __forceinline__ void mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t id, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(id), "r"(accumulate ? 1u : 0u)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's tensor-memory lane, without
// waiting: the registers are valid after tmem_wait_ld
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// wait for this thread's tensor-memory loads; r is passed through so that no
// use of it is scheduled before the wait
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// store 32 consecutive fp32 columns of this thread's tensor-memory lane and
// wait for the store
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 4-D tiled TMA store from shared memory (coordinates innermost first; the
// parts of the box outside the tensor are not written)
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// One product over K = 128 as eight K = 16 steps. Operands are tiles of 128
// rows x 128 bytes in the 128-byte swizzle at shared addresses a and b. A
// K-major operand holds K in two 64-column tiles one tile apart (a step is 32
// bytes along the row, the second four steps in the next tile); an MN-major
// operand holds K along its rows (a step is 16 rows, 2048 bytes). a_lbo,
// b_lbo: the leading byte offsets (for an MN-major operand 128 wide, the
// distance between its two 64-wide halves). The step is added to the
// descriptor's address field (bytes / 16).
__device__ __forceinline__ void mma_k128(uint32_t d, uint32_t a, bool a_kmajor, uint32_t b, bool b_kmajor,
                                         uint32_t a_lbo, uint32_t b_lbo, uint32_t id, bool accumulate = false) {
  const uint64_t ad = sdesc(a, a_lbo, 1024), bd = sdesc(b, b_lbo, 1024);
#pragma unroll 1
  for (int kk = 0; kk < 8; kk++) {
    const uint32_t kstep = (uint32_t)((kk & 3) * 2 + (kk >> 2) * (128 * 128 / 16));  // K-major
    const uint32_t mstep = (uint32_t)(kk * 128);                                      // MN-major
    mma(d, ad + (a_kmajor ? kstep : mstep), bd + (b_kmajor ? kstep : mstep), id, accumulate || kk > 0);
  }
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
__device__ __forceinline__ f2 splat2(float a) { return pk(a, a); }
// pair i (words 2i, 2i + 1) of a word array as packed floats
__device__ __forceinline__ f2 get2(const uint32_t* w, int i) {
  return pk(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}
__device__ __forceinline__ void set2(uint32_t* w, int i, f2 v) {
  w[2 * i] = __float_as_uint(f2lo(v));
  w[2 * i + 1] = __float_as_uint(f2hi(v));
}
// a pair of floats -> its bf16 high parts (one word, the first value in the
// low half) and the bf16 remainders
__device__ __forceinline__ void split2(f2 v, uint32_t& hi, uint32_t& lo) {
  uint32_t h, l;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(f2hi(v)), "f"(f2lo(v)));
  const f2 hv = pk(__uint_as_float(h << 16), __uint_as_float(h & 0xffff0000u));
  const f2 r = fma2(hv, splat2(-1.f), v);  // exact: v minus its rounded high part
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(f2hi(r)), "f"(f2lo(r)));
  hi = h;
  lo = l;
}

__device__ __forceinline__ void bar_sync_compute() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// barrier over the 256 compute threads that returns the OR of v over them
__device__ __forceinline__ bool bar_or_compute(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

template <typename TOut>
__global__ void __launch_bounds__(kThreads, 1) ssd_tc_kernel(const __grid_constant__ SsdParams p,
                                                            const __grid_constant__ CUtensorMap tm_x,
                                                            const __grid_constant__ CUtensorMap tm_b,
                                                            const __grid_constant__ CUtensorMap tm_c,
                                                            const __grid_constant__ CUtensorMap tm_y) {
  using SM = TcSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(sm);
  // Barriers. Completed by the copy engine or the tensor core: C and B
  // loaded, x of an even / odd chunk loaded, S done, the two halves of Y1
  // done, Y2 done, B^T X' done. Completed by the 256 compute threads: X'
  // written, M's column blocks 0 and 2 written, M's blocks 1 and 3 written (S
  // read), the state entering the next chunk written (B^T X' read), Y1 and Y2
  // read. By one compute thread: the y staging tiles are free again.
  enum {
    kBarCB = 0, kBarX0, kBarX1, kBarS, kBarY1a, kBarY1b, kBarY2, kBarH,
    kRdyX, kRdyM0, kRdyM1, kRdyH, kRdyY, kStg, kNumBars
  };
  static_assert(kNumBars * 8 <= SM::TSLOT - SM::BAR, "the barriers overlap the tensor-memory slot");
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + SM::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM::TSLOT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t L = p.seqlen, H = p.nheads, G = p.ngroups;
  const int64_t nchunk = (L + kQ - 1) / kQ;
  const uint64_t wait_ns = p.wait_ns ? p.wait_ns : kWaitNs;
  uint32_t* tk_slot = tslot + 1;

  // The chunks of all sequences in (batch, head)-major order are cut into
  // p.ranges contiguous ranges, one per CTA. A range covers the tail of one
  // sequence, whole sequences and the head of another; it runs the head first
  // (its state goes to the CTA with the next range), then the whole ones, then
  // the tail, whose entering state the CTA with the previous range published
  // when it ran its own head first. A range inside one sequence is a single
  // segment that waits for its predecessor.
  volatile RangeDesc* rd = reinterpret_cast<volatile RangeDesc*>(tslot + 2);
  if (tid == 0) {
    for (int i = 0; i < kNumBars; i++) mbar_init(&bar[i], (i < kRdyX || i == kStg) ? 1 : kCompute);
    fence_mbar_init();
    // the range this CTA runs: tickets in launch order, so the CTA that hands
    // a state on to this one has always started earlier
    const int64_t ticket = p.ws_ticket ? atomicAdd(p.ws_ticket, 1u) : blockIdx.x;
    *tk_slot = (uint32_t)ticket;
    const int64_t T = p.batch * H * nchunk;
    // ranges of T / ranges chunks, the first T % ranges one longer
    const int64_t q = T / p.ranges, r = T % p.ranges;
    const int64_t g0 = ticket * q + (ticket < r ? ticket : r), g1 = g0 + q + (ticket < r ? 1 : 0);
    const int64_t u0 = g0 / nchunk, u1 = (g1 - 1) / nchunk;
    rd->u0 = u0;
    rd->nseg = g1 > g0 ? (int)(u1 - u0 + 1) : 0;
    rd->cb_first = (int)(g0 - u0 * nchunk);
    rd->ce_last = (int)(g1 - u1 * nchunk);
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
  const int64_t ticket = *tk_slot;
  struct Seg {
    int64_t u;   // sequence (batch * nheads + head; below 2^31)
    int b, h;    // its batch element and head
    int cb, ce;  // its chunks [cb, ce)
  };
  auto nsegs = [&]() -> int { return rd->nseg; };
  auto segment = [&](int s) -> Seg {  // the s-th segment the CTA runs
    const int n = rd->nseg;
    const int64_t u0 = rd->u0;
    int64_t u;
    int cb, ce;
    if (n == 1) {
      u = u0, cb = rd->cb_first, ce = rd->ce_last;
    } else if (s == 0) {
      u = u0 + n - 1, cb = 0, ce = rd->ce_last;
    } else if (s == n - 1) {
      u = u0, cb = rd->cb_first, ce = (int)nchunk;
    } else {
      u = u0 + s, cb = 0, ce = (int)nchunk;
    }
    const uint32_t u32 = (uint32_t)u, H32 = (uint32_t)H;
    return {u, (int)(u32 / H32), (int)(u32 % H32), cb, ce};
  };
  uint32_t ph = 0;    // bit i: the phase of barrier i this thread waits for next
  bool fail = false;  // this thread gave up on a wait
  // wait for the next phase of barrier i; after a timeout the phase stays
  // (it is the one still in flight)
  auto wait = [&](int i) {
    if (mbar_wait(&bar[i], (ph >> i) & 1u, wait_ns)) {
      ph ^= 1u << i;
      return true;
    }
    fail = true;
    return false;
  };

  if (warp >= kComputeWarps) {
    // ============ the issuing warps: lane 0 of each issues. Issuer 0: the
    // tile loads, S and H_l; issuer 1: Y2, then Y1 over M's blocks 0 and 1;
    // issuer 2: Y1 over M's blocks 2 and 3. Buffers and barriers of a chunk
    // follow the parity of its place k in the CTA's run.
    const int role = warp - kComputeWarps;
    if (lane == 0) {
      uint32_t nissue[kRdyX] = {};  // copies or commits issued per barrier (for the drain after a timeout)
      auto commit = [&](int i) {
        mma_commit(&bar[i]);
        nissue[i]++;
      };
      // Y1 over M's S block blk (s in [32 blk, 32 blk + 32): K steps 2 blk and
      // 2 blk + 1, the high parts and the remainders) into accumulator d
      auto y1_block = [&](uint32_t d, uint32_t xs, int blk, bool first) {
        const uint64_t bd = sdesc(xs, 16, 1024);
#pragma unroll 1
        for (int i = 0; i < 4; i++) {
          const int e = i & 1, part = i >> 1, k = 2 * blk + e;
          const uint32_t ta = tmem + kColS + 32 * blk + 8 * e + 16 * part;
          mma_ta(tmem + d, ta, bd + (uint32_t)(k * 128), idesc(kQ, kP, 0, 1), !first || i > 0);
        }
      };
      int k = 0;  // chunks this CTA has begun
      if (role == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_b);
        tma_prefetch_desc(&tm_c);
        const int hpg = (int)(H / G);  // heads per group
        // the copies of chunk c of segment q (the kc-th chunk of the run)
        auto issue_cb = [&](const Seg& q, int c) {
          const int b = q.b, grp = q.h / hpg, t0 = c * kQ;
          mbar_expect_tx(&bar[kBarCB], 4 * SM::TILE);
          tma_load_4d(sm + SM::C0, &tm_c, 0, grp, t0, b, &bar[kBarCB]);
          tma_load_4d(sm + SM::C1, &tm_c, 64, grp, t0, b, &bar[kBarCB]);
          tma_load_4d(sm + SM::B0, &tm_b, 0, grp, t0, b, &bar[kBarCB]);
          tma_load_4d(sm + SM::B1, &tm_b, 64, grp, t0, b, &bar[kBarCB]);
          mbar_arrive(&bar[kBarCB]);
          nissue[kBarCB]++;
        };
        auto issue_x = [&](const Seg& q, int c, int kc) {  // into buffer kc & 1
          const int xb = kBarX0 + (kc & 1);
          mbar_expect_tx(&bar[xb], SM::TILE);
          tma_load_4d(sm + ((kc & 1) ? SM::X1 : SM::X0), &tm_x, 0, q.h, c * kQ, q.b, &bar[xb]);
          mbar_arrive(&bar[xb]);
          nissue[xb]++;
        };
        for (int sg = 0; sg < nsegs() && !fail; sg++) {
          const Seg sq = segment(sg);
          const bool has_h0 = sq.cb > 0 || p.h0 != nullptr;  // a state enters the segment
          if (sg == 0) {  // later segments' first copies were issued during the segment before
            issue_cb(sq, sq.cb);
            issue_x(sq, sq.cb, k);
          }
          for (int c = sq.cb; c < sq.ce; c++, k++) {
            // the chunk after this one in the run: the next of the segment, or
            // the first of the next segment (u < 0: none)
            Seg nx = sq;
            nx.cb = c + 1;
            if (c + 1 == sq.ce) {
              if (sg + 1 < nsegs())
                nx = segment(sg + 1);
              else
                nx.u = -1;
            }
            // S = C B^T (S's columns were read by the previous chunk's Y1)
            if (!wait(kBarCB)) break;
            tc_fence_after();
            mma_k128(tmem + kColS, s0 + SM::C0, true, s0 + SM::B0, true, 16, 16, idesc(kQ, kQ, 0, 0));
            commit(kBarS);
            // x of the next chunk, into the buffer of the chunk before this one
            // (its Y1 is done, its X' written)
            if (nx.u >= 0) issue_x(nx, nx.cb, k + 1);
            // H_l^T = B^T X' (A = B read MN-major: its two n halves are one tile
            // apart; B: X''s high part and remainder side by side, N = 128)
            if (!wait(kRdyX)) break;
            tc_fence_after();
            mma_k128(tmem + kColH, s0 + SM::B0, false, s0 + SM::XH, false, SM::TILE, SM::TILE, idesc(kN, 2 * kP, 1, 1));
            commit(kBarH);
            // C and B are free once S, H_l (in issue order) and Y2 are done;
            // S's columns and this x once both halves of Y1 are. (Issuer 1
            // has seen this copy's phase before Y2, or does not wait for it.)
            if (!wait(kBarH) || ((c > sq.cb || has_h0) && !wait(kBarY2))) break;
            if (nx.u >= 0) issue_cb(nx, nx.cb);
            if (!wait(kBarY1a) || !wait(kBarY1b)) break;
          }
        }
      } else if (role == 1) {
        for (int sg = 0; sg < nsegs() && !fail; sg++) {
          const Seg sq = segment(sg);
          const bool has_h0 = sq.cb > 0 || p.h0 != nullptr;
          for (int c = sq.cb; c < sq.ce; c++, k++) {
            const uint32_t xs = s0 + ((k & 1) ? SM::X1 : SM::X0);
            const bool y2 = c > sq.cb || has_h0;
            // C of the chunk, for Y2. Without Y2 the phase is passed over
            // unwaited: issuer 0 copies the next C only after this chunk's H_l
            // and Y2 are done (so it cannot run two phases ahead of this
            // thread's next wait), and this chunk's copy has landed before
            // this thread's next wait (M, waited for below, follows S, which
            // follows the copy)
            if (y2) {
              if (!wait(kBarCB)) break;
            } else {
              ph ^= 1u << kBarCB;
            }
            if (k > 0 && !wait(kRdyY)) break;  // the previous chunk's y has read Y1a and Y2
            // Y2 = C H_in^T: A K-major (C), B MN-major (H^T), the high part and
            // then the remainder into one accumulator
            if (y2) {
              if (!wait(kRdyH)) break;  // the state entering the chunk is written
              tc_fence_after();
              mma_k128(tmem + kColY2, s0 + SM::C0, true, s0 + SM::HH, false, 16, 16, idesc(kQ, kP, 0, 1));
              mma_k128(tmem + kColY2, s0 + SM::C0, true, s0 + SM::HL, false, 16, 16, idesc(kQ, kP, 0, 1), true);
              commit(kBarY2);
            }
            if (!wait(kRdyM0)) break;
            tc_fence_after();
            y1_block(kColY1a, xs, 0, true);
            if (!wait(kRdyM1)) break;
            tc_fence_after();
            y1_block(kColY1a, xs, 1, false);
            commit(kBarY1a);
          }
        }
      } else {
        for (int sg = 0; sg < nsegs() && !fail; sg++) {
          const Seg sq = segment(sg);
          for (int c = sq.cb; c < sq.ce; c++, k++) {
            const uint32_t xs = s0 + ((k & 1) ? SM::X1 : SM::X0);
            if (k > 0 && !wait(kRdyY)) break;  // the previous chunk's y has read Y1b
            if (!wait(kRdyM0)) break;
            tc_fence_after();
            y1_block(kColY1b, xs, 2, true);
            if (!wait(kRdyM1)) break;
            tc_fence_after();
            y1_block(kColY1b, xs, 3, false);
            commit(kBarY1b);
          }
        }
      }
      if (fail) {
        // a wait gave up: record it, and wait (bounded) for the last copy and
        // product this thread issued on each barrier (the k-th completion of a
        // barrier ends phase k, of parity k & 1) before shared and tensor
        // memory are released
        atomicOr(p.fault, kFaultTileWait);
#pragma unroll
        for (int i = 0; i < kRdyX; i++)
          if (nissue[i]) mbar_wait(&bar[i], (nissue[i] - 1) & 1u, wait_ns);
      }
    }
  } else {
    // ============ 256 compute threads: two per row of the products
    const int row = tid & (kQ - 1);  // row of the products this thread reads and writes
    const int hf = tid >> 7;         // which half of the columns
    const int wq = warp & 3;         // the warp's tensor-memory lane quarter: rows 32wq .. 32wq+31
    const uint32_t tlane = tmem + ((uint32_t)(wq * 32) << 16);
    float* const dls2 = reinterpret_cast<float*>(sm + SM::DL);   // [2][128]: the k-th chunk in half k & 1
    float* const css2 = reinterpret_cast<float*>(sm + SM::CS);   // [2][128]
    float* const wsum2 = reinterpret_cast<float*>(sm + SM::WSUM);  // [2][4]
    float* const qs2 = reinterpret_cast<float*>(sm + SM::QS);      // [2][128]
    const __nv_bfloat16* dt_all = static_cast<const __nv_bfloat16*>(p.dt);
    const int64_t dt_last = p.batch * L * H - 1;  // index of dt's last element
    uint32_t* dtb = reinterpret_cast<uint32_t*>(sm + SM::DTB);
    // the state lives in tensor memory: thread (row n, half hf) owns
    // H^T[n][32 hf .. 32 hf + 31], columns kColState + 32 hf of lane n
    const uint32_t tstate = tlane + kColState + 32 * hf;
    // the state's two bf16 parts, row n of H^T, for the next chunk's C H^T
    auto write_state = [&](const uint32_t (&hv)[32]) {
#pragma unroll
      for (int c8 = 0; c8 < 4; c8++) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; i++)
          split2(pk(__uint_as_float(hv[8 * c8 + 2 * i]), __uint_as_float(hv[8 * c8 + 2 * i + 1])), hi[i], lo[i]);
        *reinterpret_cast<uint4*>(sm + SM::HH + sw128(row, 32 * hf + 8 * c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + SM::HL + sw128(row, 32 * hf + 8 * c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    };
    // Row t of chunk c of sequence u needs dt[b, t, h]. It is fetched a chunk
    // ahead by an asynchronous 4-byte copy of the aligned pair of bf16 that
    // holds it (a plain load would be waited for by this thread's next release
    // fence), or, for dt's very last element when it starts a pair, by a plain
    // load; the kc-th chunk of the run goes to half kc & 1.
    auto dt_index = [&](const Seg& q, int c) { return ((int64_t)q.b * L + (int64_t)c * kQ + row) * H + q.h; };
    auto fetch_dt = [&](const Seg& q, int c, int kc) {
      uint32_t* dst = dtb + (kc & 1) * kQ + row;
      if ((int64_t)c * kQ + row >= L) return;
      const int64_t i = dt_index(q, c);
      if ((i & 1) == 0 && i == dt_last) {
        *dst = (uint32_t)__bfloat16_as_ushort(dt_all[i]);
      } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(dt_all + (i & ~(int64_t)1))
                     : "memory");
      }
    };
    // delta and the decay (base 2) accumulated inside chunk cc of segment sg
    // (the kc-th chunk of the run), inclusive, into half kc & 1 of dls2 /
    // css2, and q_s = 2^(cs_e - cs_s) delta_s with e the last step of s's
    // block of 32 (threads of the first column half, warp w holding block w;
    // all compute threads take part in its barrier). Visible to the others
    // after the next barrier. Also fetches the dt of the chunk after cc in the
    // run: the next of the segment or the first of the next segment.
    auto scalars = [&](const Seg& sq, int sg, int cc, int kc) {  // (sq: segment sg)
      float dl = 0.f, sc = 0.f;
      float* ws = wsum2 + (kc & 1) * 4;
      if (hf == 0) {
        const float a2 = __ldg(p.A + sq.h) * kLog2e;  // decay exponent per unit delta, base 2
        const float dtbias = p.dt_bias ? __ldg(p.dt_bias + sq.h) : 0.f;
        asm volatile("cp.async.wait_all;" ::: "memory");  // this row's dt of chunk cc
        if ((int64_t)cc * kQ + row < L) {
          const int64_t i = dt_index(sq, cc);
          const uint32_t w = dtb[(kc & 1) * kQ + row];
          dl = softplus_fast(__uint_as_float(((i & 1) ? (w >> 16) : (w & 0xffffu)) << 16) + dtbias);
        }
        if (cc + 1 < sq.ce) {
          fetch_dt(sq, cc + 1, kc + 1);
        } else if (sg + 1 < nsegs()) {
          const Seg nq = segment(sg + 1);
          fetch_dt(nq, nq.cb, kc + 1);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        sc = dl * a2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, sc, o);
          if (lane >= o) sc += v;
        }
        if (lane == 31) ws[warp] = sc;
      }
      bar_sync_compute();
      if (hf == 0) {
        for (int w = 0; w < warp; w++) sc += ws[w];
        dls2[(kc & 1) * kQ + row] = dl;
        css2[(kc & 1) * kQ + row] = sc;
        qs2[(kc & 1) * kQ + row] = ex2(__shfl_sync(0xffffffffu, sc, 31) - sc) * dl;
      }
    };
    bool aborted = false;  // a wait timed out; the same for every compute thread
    int k = 0;             // chunks this CTA has begun
    for (int sg = 0; sg < nsegs() && !aborted; sg++) {
      const Seg sq = segment(sg);
      const int b = sq.b, h = sq.h;
      const bool has_h0 = sq.cb > 0 || p.h0 != nullptr;  // a state enters the segment
      const float Dh = p.D ? __ldg(p.D + h) : 0.f;
      // the state entering the segment: h0 (or zeros) at a sequence's start,
      // else the one the CTA with the previous range published (a bounded wait)
      if (sq.cb > 0) {
        bool got = true;
        if (tid == 0) {
          const uint32_t* flag = p.ws_flags + sq.u;
          got = ld_acquire_gpu(flag) >= (uint32_t)sq.cb;
          const uint64_t t_start = globaltimer();
          while (!got && globaltimer() - t_start <= wait_ns) got = ld_acquire_gpu(flag) >= (uint32_t)sq.cb;
        }
        aborted = bar_or_compute(!got);
      }
      {
        uint32_t hv[32];
        // (h0 is [64, dstate]; the hand-over slot [64, 128]; state rows past
        // dstate are zero and stay zero, B's padded columns being zero)
        const int64_t sstride = sq.cb > 0 ? kN : p.dstate;
        const float* h0 =
            sq.cb > 0 ? p.ws_state + sq.u * kP * kN : (p.h0 ? p.h0 + sq.u * kP * p.dstate : nullptr);
        const bool rin = h0 && !aborted && row < sstride;
#pragma unroll
        for (int q = 0; q < 32; q++) hv[q] = __float_as_uint(rin ? h0[(32 * hf + q) * sstride + row] : 0.f);
        tmem_st32(tstate, hv);
        // (the previous segment's last C H_in^T has read the two parts: its
        // completion was waited for before that chunk's state update)
        if (has_h0) {
          write_state(hv);
          fence_proxy_async_smem();  // read by the tensor core
        }
        tc_fence_before();
        if (has_h0) mbar_arrive(&bar[kRdyH]);
      }
      if (aborted) break;
      if (sg == 0) {  // later segments' first scalars were computed during the segment before
        if (hf == 0) {
          fetch_dt(sq, sq.cb, k);
          asm volatile("cp.async.commit_group;" ::: "memory");
        }
        scalars(sq, sg, sq.cb, k);
        bar_sync_compute();
      }
      for (int c = sq.cb; c < sq.ce && !aborted; c++, k++) {
        const int64_t t0 = (int64_t)c * kQ;
        const float* dls = dls2 + (k & 1) * kQ;
        const float* css = css2 + (k & 1) * kQ;
        const float* qsv = qs2 + (k & 1) * kQ;
        const uint8_t* xs = sm + ((k & 1) ? SM::X1 : SM::X0);
        const bool y2 = c > sq.cb || has_h0;  // a state enters the chunk: C H_in^T runs
        // ---- X' (row s, columns p in half hf) = 2^(cs_end - cs_s) delta_s x_s
        wait(kBarX0 + (int)(k & 1));
        {
          const f2 ws = splat2(ex2(css[kQ - 1] - css[row]) * dls[row]);
#pragma unroll
          for (int c8 = 0; c8 < 4; c8++) {
            const int off = sw128(row, 32 * hf + 8 * c8);
            const uint4 xw = *reinterpret_cast<const uint4*>(xs + off);
            const uint32_t w[4] = {xw.x, xw.y, xw.z, xw.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; i++)
              split2(mul2(pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u)), ws), hi[i], lo[i]);
            *reinterpret_cast<uint4*>(sm + SM::XH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + SM::XL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[kRdyX]);
        if (tid == kStoreTid) {  // the previous chunk's y store has read its staging tiles
          bulk_wait_read();
          mbar_arrive(&bar[kStg]);
        }
        // ---- M (row t, columns s in half hf) from S, D_h on the diagonal,
        // written over S in tensor memory, where Y1 = M X reads it as its A
        // operand: the 32 columns of S block k (s in [32k, 32k + 32)) take the
        // block's high parts (16 columns, two bf16 each, the even s in the low
        // half) and then its remainders. This thread's blocks are kb0 and kb0 +
        // 1; the issuer starts Y1 on blocks 0 and 2 once every thread has
        // written its first one. Block k holds nonzeros for the warp's rows only
        // if k <= wq (warp-uniform).
        wait(kBarS);
        tc_fence_after();
        {
          const float cst = css[row];
          const int kb0 = 2 * hf;
#pragma unroll 1
          for (int j = 0; j < 2; j++) {
            const int kb = kb0 + j;
            uint32_t sr[32];  // S block kb, then M's words: [0, 16) the high parts, [16, 32) the remainders
            if (kb < wq) {
              // below the diagonal block: 2^(cs_t - cs_s) = 2^(cs_t - cs_e) 2^(cs_e - cs_s),
              // e the block's last step; both factors are at most 1
              tmem_ld32_async(tlane + kColS + 32 * kb, sr);
              const f2 rt = splat2(ex2(cst - css[32 * kb + 31]));
              tmem_wait_ld(sr);
              uint32_t lo[16];
#pragma unroll
              for (int i = 0; i < 16; i++) {  // (pair i reads S words 2i, 2i + 1 >= i: writing word i is safe)
                const float2 q = *reinterpret_cast<const float2*>(qsv + 32 * kb + 2 * i);
                const f2 v = mul2(mul2(get2(sr, i), pk(q.x, q.y)), rt);
                split2(v, sr[i], lo[i]);
              }
#pragma unroll
              for (int i = 0; i < 16; i++) sr[16 + i] = lo[i];
            } else if (kb == wq) {  // the block that holds the diagonal: causal mask, D_h on it
              tmem_ld32_async(tlane + kColS + 32 * kb, sr);
              tmem_wait_ld(sr);
              uint32_t lo[16];
              const int dr = row - 32 * kb;  // the diagonal's position in the block
#pragma unroll
              for (int i = 0; i < 16; i++) {  // (pair i reads S words 2i, 2i + 1 >= i: writing word i is safe)
                const float2 cs = *reinterpret_cast<const float2*>(css + 32 * kb + 2 * i);
                const float2 dl = *reinterpret_cast<const float2*>(dls + 32 * kb + 2 * i);
                f2 m = mul2(mul2(get2(sr, i), pk(ex2(cst - cs.x), ex2(cst - cs.y))), pk(dl.x, dl.y));
                float m0 = f2lo(m), m1 = f2hi(m);
                m0 = 2 * i < dr ? m0 : (2 * i == dr ? m0 + Dh : 0.f);
                m1 = 2 * i + 1 < dr ? m1 : (2 * i + 1 == dr ? m1 + Dh : 0.f);
                split2(pk(m0, m1), sr[i], lo[i]);
              }
#pragma unroll
              for (int i = 0; i < 16; i++) sr[16 + i] = lo[i];
            } else {
#pragma unroll
              for (int i = 0; i < 32; i++) sr[i] = 0u;
            }
            tmem_st32(tlane + kColS + 32 * kb, sr);
            tc_fence_before();
            mbar_arrive(&bar[j == 0 ? kRdyM0 : kRdyM1]);
          }
        }
        // ---- the state, row n of H^T: 2^cs_end H^T + H_l^T. Its two parts
        // are rewritten only after this chunk's C H_in^T has read them (that
        // product's own completion: it comes from another issuing thread than
        // B^T X'); a segment's last chunk writes them for no further product.
        wait(kBarH);
        if (y2) wait(kBarY2);
        tc_fence_after();
        {
          const float dec = ex2(css[kQ - 1]);
          uint32_t hl[32], hv[32];
          {
            uint32_t hl2[32];
            tmem_ld32_async(tlane + kColH + 32 * hf, hl);
            tmem_ld32_async(tlane + kColH + kP + 32 * hf, hl2);
            tmem_wait_ld(hl);
            tmem_wait_ld(hl2);
#pragma unroll
            for (int i = 0; i < 16; i++) set2(hl, i, add2(get2(hl, i), get2(hl2, i)));
          }
          tmem_ld32_async(tstate, hv);
          tmem_wait_ld(hv);
          const f2 dec2 = splat2(dec);
#pragma unroll
          for (int i = 0; i < 16; i++) set2(hv, i, fma2(dec2, get2(hv, i), get2(hl, i)));
          tmem_st32(tstate, hv);
          if (c + 1 < sq.ce) {
            write_state(hv);
            fence_proxy_async_smem();
          }
        }
        tc_fence_before();
        if (c + 1 < sq.ce) mbar_arrive(&bar[kRdyH]);
        // ---- the next chunk's delta and decay sums, while Y1 runs (the
        // next segment's first chunk after a segment's last)
        if (c + 1 < sq.ce) {
          scalars(sq, sg, c + 1, k + 1);
        } else if (sg + 1 < nsegs()) {
          const Seg nq = segment(sg + 1);
          scalars(nq, sg + 1, nq.cb, k + 1);
        }
        // ---- y of row t, columns p in half hf: Y1 + 2^cs_t Y2, staged in
        // shared memory and stored by TMA
        wait(kBarY1a);
        wait(kBarY1b);
        tc_fence_after();
        bool abort;
        {
          const int pb = 32 * hf;
          uint32_t r1[32], r2[32];
          {  // Y1 = the half over s < 64 + the half over s >= 64
            uint32_t r3[32];
            tmem_ld32_async(tlane + kColY1a + pb, r1);
            tmem_ld32_async(tlane + kColY1b + pb, r3);
            tmem_wait_ld(r1);
            tmem_wait_ld(r3);
#pragma unroll
            for (int i = 0; i < 16; i++) set2(r1, i, add2(get2(r1, i), get2(r3, i)));
          }
          if (y2) {
            tmem_ld32_async(tlane + kColY2 + pb, r2);
            tmem_wait_ld(r2);
          }
          tc_fence_before();
          mbar_arrive(&bar[kRdyY]);  // Y1 and Y2 are read
          if (y2) {
            const f2 et = splat2(ex2(css[row]));
#pragma unroll
            for (int i = 0; i < 16; i++) set2(r1, i, fma2(et, get2(r2, i), get2(r1, i)));
          }
          const float* o = reinterpret_cast<const float*>(r1);
          wait(kStg);  // the previous chunk's y store has read the staging tiles
          if constexpr (sizeof(TOut) == 2) {
#pragma unroll
            for (int c8 = 0; c8 < 4; c8++) {
              uint32_t w4[4];
#pragma unroll
              for (int i = 0; i < 4; i++) {
                const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[8 * c8 + 2 * i], o[8 * c8 + 2 * i + 1]);
                w4[i] = *reinterpret_cast<const uint32_t*>(&v2);
              }
              *reinterpret_cast<uint4*>(sm + SM::YS0 + sw128(row, pb + 8 * c8)) =
                  make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          } else {  // fp32: tile hf holds columns 32 hf .. 32 hf + 31, 128 bytes a row
#pragma unroll
            for (int c4 = 0; c4 < 8; c4++)
              *reinterpret_cast<float4*>(sm + (hf ? SM::YS1 : SM::YS0) + row * 128 + ((c4 ^ (row & 7)) << 4)) =
                  make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
          }
          fence_proxy_async_smem();
          // every row is staged and the next chunk's scalars are written; a
          // timeout anywhere ends the run for every compute thread
          abort = bar_or_compute(fail);
          aborted = abort;
          if (!abort && tid == kStoreTid) {
            tma_store_4d(&tm_y, sm + SM::YS0, 0, (int)h, (int)t0, (int)b);
            if constexpr (sizeof(TOut) == 4) tma_store_4d(&tm_y, sm + SM::YS1, 32, (int)h, (int)t0, (int)b);
          }
        }
        if (abort) break;
      }
      if (aborted) break;
      // the state leaving the segment: h_last at the sequence's end, else the
      // hand-over slot, published for the CTA with the next range
      const bool seq_end = sq.ce == nchunk;
      const int64_t ostride = seq_end ? p.dstate : kN;  // h_last [64, dstate]; the slot [64, 128]
      float* hout = seq_end ? (p.h_last ? p.h_last + sq.u * kP * p.dstate : nullptr) : p.ws_state + sq.u * kP * kN;
      if (hout && row < ostride) {  // (the same for every thread of a warp)
        uint32_t hv[32];
        tmem_ld32_async(tstate, hv);
        tmem_wait_ld(hv);
#pragma unroll
        for (int q = 0; q < 32; q++) hout[(32 * hf + q) * ostride + row] = __uint_as_float(hv[q]);
      }
      if (!seq_end) {
        bar_sync_compute();  // every thread's part of the state is written
        if (tid == 0 && ticket != p.withhold_range) {
          __threadfence();
          st_release_gpu(p.ws_flags + sq.u, (uint32_t)sq.ce);
        }
      }
    }
    if (tid == kStoreTid) bulk_wait_all();  // the y stores are complete
    if (aborted && tid == 0) atomicOr(p.fault, kFaultTileWait);
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

// 4-D map over a row-major [d3, d2, d1, d0] tensor of 2- or 4-byte elements
// with a [1, 128, 1, 128 bytes] box (128 rows of d2) in the 128-byte swizzle
bool make_map_4d(CUtensorMap* m, const void* ptr, int esize, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3) {
  TcEncodeFn fn = tc_encode_fn();
  if (!fn) return false;
  const uint64_t e = (uint64_t)esize;
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {d0 * e, d0 * d1 * e, d0 * d1 * d2 * e};
  cuuint32_t box[4] = {(cuuint32_t)(128 / esize), 1, (cuuint32_t)kQ, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TOut>
cudaError_t launch_tc(const SsdParams& p, cudaStream_t s) {
  CUtensorMap mx{}, mb{}, mc{}, my{};
  // x, y [batch, L, H, 64]; B, C [batch, L, G, 128]
  const uint64_t L = (uint64_t)p.seqlen, Bt = (uint64_t)p.batch, H = (uint64_t)p.nheads, G = (uint64_t)p.ngroups;
  // B and C [.., dstate]: with dstate 64 the box at column 64 lies wholly
  // outside the tensor and is zero-filled, padding both to 128 columns
  const uint64_t N = (uint64_t)p.dstate;
  if (!make_map_4d(&mx, p.x, 2, kP, H, L, Bt) || !make_map_4d(&mb, p.B, 2, N, G, L, Bt) ||
      !make_map_4d(&mc, p.C, 2, N, G, L, Bt) || !make_map_4d(&my, p.y, (int)sizeof(TOut), kP, H, L, Bt))
    return cudaErrorInvalidValue;
  auto k = ssd_tc_kernel<TOut>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::ALLOC);
  if (e != cudaSuccess) return e;
  k<<<(unsigned)p.ranges, kThreads, TcSmem::ALLOC, s>>>(p, mx, mb, mc, my);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_fwd_tc(const SsdParams& p, ss_dtype out_dtype, cudaStream_t stream) {
  return out_dtype == SS_BF16 ? launch_tc<__nv_bfloat16>(p, stream) : launch_tc<float>(p, stream);
}

}  // namespace ssk
