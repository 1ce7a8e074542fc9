// Device helpers for the sm_103a selective-scan kernels: fast transcendental
// wrappers, dtype conversion, mbarrier and TMA (cp.async.bulk.tensor) PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// Default limit of a device-side wait (nanoseconds of %globaltimer); the scan
// takes its limit per call (ScanParams::wait_ns).
constexpr uint64_t kWaitNs = 2000000000ull;

// Fault codes written to the fault word.
constexpr unsigned kFaultTileWait = 1u;   // a pipeline stage never became ready
constexpr unsigned kFaultLookback = 2u;   // a predecessor chunk never published

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = log(1 + e^x). Above 20 the correction log1p(e^-x) < 2.1e-9
// is below half an fp32 ulp of x and x is returned.
__device__ __forceinline__ float softplus(float x) {
  if (x > 20.f) return x;
  return log1pf(ex2(x * kLog2e));
}

// silu(z) = z / (1 + e^-z); e^-z overflows to +inf for z < -88, giving -0.
__device__ __forceinline__ float silu(float z) { return z * rcp(1.f + ex2(-z * kLog2e)); }

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- packed fp32x2
// A pair of fp32 values in one 64-bit register pair, for the sm_100+ packed
// FFMA2 / FMUL2 / FADD2 instructions (one issue slot for two lanes of work).
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
// The unpack is a register-pair view (no instruction); the half that is not
// returned is an unused asm output.
#pragma nv_diagnostic push
#pragma nv_diag_suppress 550
__device__ __forceinline__ float f2lo(f2 r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return a;
}
__device__ __forceinline__ float f2hi(f2 r) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
  return b;
}
#pragma nv_diagnostic pop
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------- fast activations
// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(v) with v = e^-|x| in (0, 1].
// log1p(v) = v * q(v), where q is a degree-7 polynomial fitted (relative-error
// least squares with reweighting, coefficients rounded to fp32) to
// log1p(v) / v on [0, 1]; evaluated by Horner in fp32 its relative error is
// below 3.3e-7 over the whole interval (fit_softplus.py beside this file
// regenerates the coefficients and the bound). One MUFU ex2 and nine FMA-pipe
// operations, against ex2 + lg2 on the MUFU pipe for the direct form. Large x
// gives v -> 0 and exactly x; x below about -87 gives v = 0 (flushed) and 0.
constexpr float kSp0 = 0.9999998211860657f, kSp1 = -0.4999740421772003f, kSp2 = 0.3327547609806061f,
                kSp3 = -0.244954451918602f, kSp4 = 0.17745192348957062f, kSp5 = -0.10768099874258041f,
                kSp6 = 0.04408911243081093f, kSp7 = -0.00853906013071537f;

__device__ __forceinline__ float softplus_fast(float x) {
  const float v = ex2(-fabsf(x) * kLog2e);
  float q = fmaf(v, kSp7, kSp6);
  q = fmaf(v, q, kSp5);
  q = fmaf(v, q, kSp4);
  q = fmaf(v, q, kSp3);
  q = fmaf(v, q, kSp2);
  q = fmaf(v, q, kSp1);
  q = fmaf(v, q, kSp0);
  return fmaf(v, q, fmaxf(x, 0.f));
}

// softplus_fast for two values at once: the polynomial runs as packed f32x2
// operations; the exponentials and the max stay per value.
__device__ __forceinline__ f2 softplus_fast2(f2 x) {
  const f2 xl = mul2(x, pk(kLog2e, kLog2e));
  const f2 v = pk(ex2(-fabsf(f2lo(xl))), ex2(-fabsf(f2hi(xl))));
  f2 q = fma2(v, pk(kSp7, kSp7), pk(kSp6, kSp6));
  q = fma2(v, q, pk(kSp5, kSp5));
  q = fma2(v, q, pk(kSp4, kSp4));
  q = fma2(v, q, pk(kSp3, kSp3));
  q = fma2(v, q, pk(kSp2, kSp2));
  q = fma2(v, q, pk(kSp1, kSp1));
  q = fma2(v, q, pk(kSp0, kSp0));
  return fma2(v, q, pk(fmaxf(f2lo(x), 0.f), fmaxf(f2hi(x), 0.f)));
}

// silu for two values: z / (1 + e^-z), the scalings and additions packed
__device__ __forceinline__ f2 silu2(f2 z) {
  const f2 e = mul2(z, pk(-kLog2e, -kLog2e));
  const f2 d = add2(pk(ex2(f2lo(e)), ex2(f2hi(e))), pk(1.f, 1.f));
  return mul2(z, pk(rcp(f2lo(d)), rcp(f2hi(d))));
}

// ---------------------------------------------------------------- global stores
// Output stores written as explicit, predicated st.global. The compiler then
// knows they cannot alias shared memory (later shared-memory loads stay free to
// move above them), and the guard is a predicate rather than a branch, so an
// unrolled token loop stays one basic block that the scheduler can interleave.
__device__ __forceinline__ void st_out(float* p, float v, bool on) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.f32 [%0], %1;\n\t}" ::"l"(p), "f"(v),
               "r"((unsigned)on));
}
__device__ __forceinline__ void st_out(__nv_bfloat16* p, float v, bool on) {
  const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.b16 [%0], %1;\n\t}" ::"l"(p), "h"(b),
               "r"((unsigned)on));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar`; false if it did not complete
// within limit_ns nanoseconds of %globaltimer.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- TMA
// 3-D tiled bulk-tensor load into shared memory, completion counted on `bar`.
// Coordinates are (x = innermost, y, z) in elements; x * elemsize must be a
// multiple of 16 bytes (the callers pass channel-block starts that are).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// order this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses of the same memory
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- global acquire/release
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

}  // namespace ssk
