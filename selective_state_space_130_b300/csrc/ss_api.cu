// C ABI of libssscan.so: argument checks, launch planning, dispatch.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "ss_internal.h"

namespace ssk {
int scan_channels_per_block(int sg);
int scan_tile_len();
int scan_header_words();
uint32_t scan_header_magic();
}  // namespace ssk

namespace {

thread_local std::string g_err;
thread_local int g_tune_sg = 0;           // 0 = automatic
thread_local int64_t g_tune_chunk = 0;    // 0 = automatic

constexpr int kVersion = 10000;  // 1.0.0
constexpr int kSMs = 148;

ss_status fail(ss_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ss_status fail(ss_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

ss_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernels are compiled for sm_103a only.
ss_status check_device() {
  static thread_local int cached_dev = -1;
  static thread_local bool cached_ok = false;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != cached_dev) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    cached_dev = dev;
    cached_ok = (major == 10 && minor == 3);
    if (!cached_ok)
      return fail(SS_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; libssscan is built for sm_103a", dev,
                  major, minor);
  }
  if (!cached_ok) return fail(SS_ERR_UNSUPPORTED, "current device is not compute capability 10.3");
  return SS_OK;
}

bool valid_dtype(int t) { return t == SS_F32 || t == SS_BF16; }
size_t dsize(ss_dtype t) { return t == SS_BF16 ? 2 : 4; }

}  // namespace

namespace ssk {

ScanPlan plan_scan(int64_t batch, int64_t seqlen, int64_t dim) {
  ScanPlan pl{};
  int sg = g_tune_sg;
  if (sg != 1 && sg != 2 && sg != 4) sg = 2;
  pl.sg = sg;
  pl.cblk = scan_channels_per_block(sg);
  const int tile = scan_tile_len();
  // Blocks are single warps; split the sequence only when the channel blocks
  // alone would leave SMs short of warps (target about eight per SM).
  const int64_t base_warps = batch * ((dim + pl.cblk - 1) / pl.cblk);
  const int64_t target = (int64_t)kSMs * 8;
  const int64_t min_chunk = 8192;
  int64_t chunk = seqlen;
  if (g_tune_chunk > 0) {
    chunk = g_tune_chunk;
  } else if (base_warps < target / 2 && seqlen >= 2 * min_chunk) {
    int64_t k = (target + base_warps - 1) / base_warps;
    k = std::min<int64_t>(k, seqlen / min_chunk);
    chunk = (seqlen + k - 1) / k;
  }
  chunk = std::max<int64_t>(tile, ((chunk + tile - 1) / tile) * tile);
  pl.chunk_len = chunk;
  pl.nchunks = seqlen > 0 ? (int)((seqlen + chunk - 1) / chunk) : 1;
  pl.workspace = 0;
  if (pl.nchunks > 1) {
    const int64_t ncblk = (dim + pl.cblk - 1) / pl.cblk;
    const int64_t tiles = batch * ncblk * pl.nchunks;
    const size_t head = (size_t)scan_header_words() * 4 + (((size_t)tiles * 4 + 255) & ~size_t(255));
    pl.workspace = head + (size_t)tiles * pl.cblk * 48 * sizeof(float);
  }
  return pl;
}

}  // namespace ssk

extern "C" {

int ss_version(void) { return kVersion; }

const char* ss_last_error(void) { return g_err.c_str(); }

void ss_scan_set_tuning(int threads_per_channel, int64_t chunk_len) {
  g_tune_sg = threads_per_channel;
  g_tune_chunk = chunk_len;
}

size_t ss_scan_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate) {
  if (batch <= 0 || seqlen <= 0 || dim <= 0 || dstate != ssk::kDState) return 0;
  return ssk::plan_scan(batch, seqlen, dim).workspace;
}

ss_status ss_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, ss_dtype in_dtype,
                      ss_dtype out_dtype, const void* u, const void* delta_raw, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias, const float* h0,
                      void* y, float* h_last, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (dstate != ssk::kDState) return fail(SS_ERR_UNSUPPORTED, "dstate must be 16 (got %lld)", (long long)dstate);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0)
    return fail(SS_ERR_INVALID_ARG, "negative size (batch %lld, seqlen %lld, dim %lld)", (long long)batch,
                (long long)seqlen, (long long)dim);
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (batch == 0 || dim == 0) return SS_OK;
  if ((double)batch * (double)seqlen * (double)dim > 4.0e18) return fail(SS_ERR_INVALID_ARG, "problem too large");
  const void* need[] = {u, delta_raw, A, B, C, y};
  const char* names[] = {"u", "delta_raw", "A", "B", "C", "y"};
  if (seqlen > 0) {
    for (int i = 0; i < 6; i++)
      if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  }
  const void* all[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, y, h_last, workspace};
  const char* all_names[] = {"u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "h0", "y", "h_last", "workspace"};
  for (int i = 0; i < 12; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t hbytes = (size_t)batch * dim * ssk::kDState * sizeof(float);
  if (seqlen == 0) {
    if (!h_last) return SS_OK;
    cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, hbytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h_last, 0, hbytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state copy");
  }

  const ssk::ScanPlan plan = ssk::plan_scan(batch, seqlen, dim);
  if (plan.workspace > 0 && (!workspace || workspace_bytes < plan.workspace))
    return fail(SS_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu%s)", plan.workspace, workspace_bytes,
                workspace ? "" : ", NULL");

  ssk::ScanParams p{};
  p.u = u;
  p.delta_raw = delta_raw;
  p.z = z;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.delta_bias = delta_bias;
  p.h0 = h0;
  p.y = y;
  p.h_last = h_last;
  p.batch = batch;
  p.seqlen = seqlen;
  p.dim = dim;
  p.chunk_len = plan.chunk_len;
  p.nchunks = plan.nchunks;
  p.ncblk = (int)((dim + plan.cblk - 1) / plan.cblk);
  if ((double)batch * p.ncblk * p.nchunks > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  // The fault word lives in the workspace header when a workspace is given
  // (so ss_scan_status(workspace) reads what this call wrote), else in the
  // library's own device word. The header is cleared on the stream first.
  const size_t hdr = (size_t)ssk::scan_header_words() * 4;
  if (workspace && workspace_bytes >= hdr) {
    p.ws_header = static_cast<uint32_t*>(workspace);
    p.fault = p.ws_header + 1;
    size_t clear = hdr;
    if (plan.nchunks > 1) {
      const int64_t tiles = batch * (int64_t)p.ncblk * plan.nchunks;
      clear = hdr + (((size_t)tiles * 4 + 255) & ~size_t(255));
      p.ws_carry = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + clear);
    }
    cudaError_t e = cudaMemsetAsync(workspace, 0, clear, s);
    if (e != cudaSuccess) return cuda_fail(e, "workspace initialisation");
  } else {
    p.fault = ssk::device_fault_word();
    if (!p.fault) return fail(SS_ERR_CUDA, "cannot resolve the library fault word");
  }
  const bool tma = ((size_t)dim * dsize(in_dtype)) % 16 == 0;
  cudaError_t e = ssk::launch_scan_fwd(p, plan, in_dtype, out_dtype, tma, s);
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  return SS_OK;
}

ss_status ss_state_update(int64_t batch, int64_t dim, int64_t dstate, ss_dtype in_dtype, ss_dtype out_dtype,
                          float* h, const void* u, const void* delta_raw, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias, void* y,
                          void* stream) {
  g_err.clear();
  if (dstate != ssk::kDState) return fail(SS_ERR_UNSUPPORTED, "dstate must be 16 (got %lld)", (long long)dstate);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || dim < 0) return fail(SS_ERR_INVALID_ARG, "negative size");
  if (batch == 0 || dim == 0) return SS_OK;
  if ((double)batch * (double)dim * 2 > 4.0e12) return fail(SS_ERR_INVALID_ARG, "problem too large");
  const void* need[] = {h, u, delta_raw, A, B, C, y};
  const char* names[] = {"h", "u", "delta_raw", "A", "B", "C", "y"};
  for (int i = 0; i < 7; i++)
    if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  const void* all[] = {h, u, delta_raw, A, B, C, D, z, delta_bias, y};
  const char* all_names[] = {"h", "u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "y"};
  for (int i = 0; i < 10; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  ssk::StepParams p{h, u, delta_raw, z, B, C, A, D, delta_bias, y, batch, dim};
  cudaError_t e = ssk::launch_state_update(p, in_dtype, out_dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "state update launch");
  return SS_OK;
}

ss_status ss_scan_status(void* workspace, void* stream) {
  g_err.clear();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int fault = 0, f2 = 0;
  unsigned int* own = ssk::device_fault_word();
  if (own) {
    if ((e = cudaMemcpy(&fault, own, sizeof fault, cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(e, "fault word read");
    if (fault && (e = cudaMemset(own, 0, sizeof fault)) != cudaSuccess) return cuda_fail(e, "fault word clear");
  }
  if (workspace) {
    // words 1 (fault) and 2 (magic written by a scan that used this buffer)
    uint32_t w[2] = {0, 0};
    uint32_t* dw = static_cast<uint32_t*>(workspace) + 1;
    if ((e = cudaMemcpy(w, dw, sizeof w, cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(e, "workspace fault word read");
    if (w[1] == ssk::scan_header_magic()) {
      f2 = w[0];
      if ((e = cudaMemset(dw, 0, sizeof w)) != cudaSuccess) return cuda_fail(e, "workspace fault clear");
    }
  }
  fault |= f2;
  if (fault)
    return fail(SS_ERR_TIMEOUT, "a device-side wait gave up (fault bits 0x%x: %s%s)", fault,
                (fault & 1u) ? "pipeline stage " : "", (fault & 2u) ? "chunk look-back" : "");
  return SS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scan forward with library-owned scratch, for callers that cannot allocate.
//
// Some callers have no device allocator to hand: code that runs inside another
// runtime's memory pool, a plugin handed only its input and output buffers, or
// a program that must not call cudaMalloc once it is serving. For them this
// entry point takes the cross-block carry scratch from a fixed array that the
// library itself declares in device memory. Every GPU that loads the library
// holds SS_SCAN_NOALLOC_SCRATCH_BYTES of it until the process exits.
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SS_SCAN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on device `dev` (the current device).
// The name g_noalloc_scratch in host code is only a host-side handle, so the
// address is resolved once per device with that device current.
ss_status noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(SS_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "scratch address lookup");
    if (!p) return fail(SS_ERR_CUDA, "scratch address lookup returned NULL");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SS_OK;
}

}  // namespace

extern "C" ss_status ss_scan_fwd_noalloc(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                         ss_dtype in_dtype, ss_dtype out_dtype, const void* u,
                                         const void* delta_raw, const float* A, const void* B, const void* C,
                                         const float* D, const void* z, const float* delta_bias, const float* h0,
                                         void* y, float* h_last, void* stream) {
  g_err.clear();
  if (dstate != ssk::kDState) return fail(SS_ERR_UNSUPPORTED, "dstate must be 16 (got %lld)", (long long)dstate);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0)
    return fail(SS_ERR_INVALID_ARG, "negative size (batch %lld, seqlen %lld, dim %lld)", (long long)batch,
                (long long)seqlen, (long long)dim);
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (batch == 0 || dim == 0) return SS_OK;
  if ((double)batch * (double)seqlen * (double)dim > 4.0e18) return fail(SS_ERR_INVALID_ARG, "problem too large");
  const void* need[] = {u, delta_raw, A, B, C, y};
  const char* names[] = {"u", "delta_raw", "A", "B", "C", "y"};
  if (seqlen > 0) {
    for (int i = 0; i < 6; i++)
      if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  }
  const void* all[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, y, h_last};
  const char* all_names[] = {"u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "h0", "y", "h_last"};
  for (int i = 0; i < 11; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);

  const ssk::ScanPlan plan = ssk::plan_scan(batch, seqlen > 0 ? seqlen : 1, dim);
  if (seqlen > 0 && plan.workspace > (size_t)SS_SCAN_NOALLOC_SCRATCH_BYTES)
    return fail(SS_ERR_INVALID_ARG,
                "this problem needs %zu bytes of scratch; the no-allocation scan holds at most %zu (use ss_scan_fwd "
                "with a caller-provided workspace)",
                plan.workspace, (size_t)SS_SCAN_NOALLOC_SCRATCH_BYTES);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  void* scratch = nullptr;
  if ((st = noalloc_scratch(dev, &scratch)) != SS_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (seqlen == 0) {
    if (!h_last) return SS_OK;
    const size_t hbytes = (size_t)batch * dim * ssk::kDState * sizeof(float);
    e = h0 ? cudaMemcpyAsync(h_last, h0, hbytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(h_last, 0, hbytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state copy");
  }

  ssk::ScanParams p{};
  p.u = u;
  p.delta_raw = delta_raw;
  p.z = z;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.delta_bias = delta_bias;
  p.h0 = h0;
  p.y = y;
  p.h_last = h_last;
  p.batch = batch;
  p.seqlen = seqlen;
  p.dim = dim;
  p.chunk_len = plan.chunk_len;
  p.nchunks = plan.nchunks;
  p.ncblk = (int)((dim + plan.cblk - 1) / plan.cblk);
  if ((double)batch * p.ncblk * p.nchunks > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  // Device-side waits that give up are recorded in the library's own fault
  // word, which ss_scan_status(NULL, stream) reads and clears.
  p.fault = ssk::device_fault_word();
  if (!p.fault) return fail(SS_ERR_CUDA, "cannot resolve the library fault word");
  if (plan.nchunks > 1) {
    // The scratch keeps the previous call's contents: the ticket counter and
    // the per-chunk flags must start at zero, so clear them on the stream.
    const int64_t tiles = batch * (int64_t)p.ncblk * plan.nchunks;
    const size_t clear = (size_t)ssk::scan_header_words() * 4 + (((size_t)tiles * 4 + 255) & ~size_t(255));
    p.ws_header = static_cast<uint32_t*>(scratch);
    p.ws_carry = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + clear);
    e = cudaMemsetAsync(scratch, 0, clear, s);
    if (e != cudaSuccess) return cuda_fail(e, "scratch initialisation");
  }
  const bool tma = ((size_t)dim * dsize(in_dtype)) % 16 == 0;
  e = ssk::launch_scan_fwd(p, plan, in_dtype, out_dtype, tma, s);
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  return SS_OK;
}
