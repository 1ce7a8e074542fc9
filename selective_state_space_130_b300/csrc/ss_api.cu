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

namespace {

thread_local std::string g_err;
thread_local int g_tune_sg = 0;           // 0 = automatic
thread_local int64_t g_tune_chunk = 0;    // 0 = automatic
thread_local int g_tune_workers = 0;      // cap on the CTAs a split uses; 0 = one per SM
thread_local uint64_t g_wait_ns = 2000000000ull;  // limit of the scan's device-side waits
thread_local int64_t g_withhold = -1;     // test knob: hand-over or chunk flag never published

constexpr int kVersion = 10200;  // 1.2.0
constexpr int kDefaultSMs = 148;  // B300, when the device cannot be queried
constexpr int64_t kMinChunk = 8192;  // shortest sequence chunk of the chunked mode

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

// Lanes per channel of the backward kernel. Two lanes per channel double the
// warps (one per 16 channels), which spreads the work more evenly over the
// SM sub-partitions and gives each of them more than one warp to switch
// between; one lane per channel needs fewer instructions per state and wins
// once there are several warps per sub-partition anyway.
int bwd_lanes_per_channel(int64_t batch, int64_t dim) {
  if (g_tune_sg == 1 || g_tune_sg == 2) return g_tune_sg;
  return batch * ((dim + 31) / 32) >= 3 * 4 * (int64_t)ssk::device_sm_count() ? 1 : 2;
}
size_t dsize(ss_dtype t) { return t == SS_BF16 ? 2 : 4; }

}  // namespace

namespace ssk {

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cache[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kDefaultSMs;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return kDefaultSMs;
    cache[dev] = n;
  }
  return cache[dev];
}

// Relative cost of one token of one channel block (CTA cycles per token, from
// the measured token loops on B300): one lane per channel runs 128 channels in
// about 148 cycles, two lanes per channel 64 channels in about 87.
static double block_token_cost(int sg) { return sg == 1 ? 148.0 : 87.0; }

ScanPlan plan_scan(int64_t batch, int64_t seqlen, int64_t dim, ss_dtype in_dtype, int sms, bool with_workspace) {
  ScanPlan pl{};
  const int64_t W = g_tune_workers > 0 ? std::min<int64_t>(sms, g_tune_workers) : sms;  // CTA slots (one per SM)
  const bool chunkable = seqlen >= 2 * kMinChunk;
  int sg = g_tune_sg;
  if (sg != 1 && sg != 2) {
    // the layout with the smaller estimated makespan: one lane per channel
    // needs fewer instructions per state update; two lanes per channel give
    // twice the channel blocks, which pays when one-lane blocks cannot fill
    // every SM and the sequence is too short to be split into chunks
    double best = 0.0;
    for (int cand = 1; cand <= 2; cand++) {
      const int64_t nb = batch * ((dim + scan_channels_per_block(cand) - 1) / scan_channels_per_block(cand));
      const double waves = (nb >= W || chunkable) ? (double)nb / (double)W : 1.0;
      const double est = waves * block_token_cost(cand);
      if (cand == 1 || est < best) {
        best = est;
        sg = cand;
      }
    }
  }
  pl.sg = sg;
  pl.cblk = scan_channels_per_block(sg);
  const int tile = scan_tile_len(in_dtype, sg);
  pl.tile = tile;
  const int64_t ncblk = (dim + pl.cblk - 1) / pl.cblk;
  const int64_t nblk = batch * ncblk;
  const int64_t T = seqlen > 0 ? (seqlen + tile - 1) / tile : 1;
  pl.mode = kModeStatic;
  pl.nworkers = nblk;
  pl.chunk_tiles = T;
  pl.nchunks = 1;
  if (!with_workspace) {
    // static: every block runs its whole sequence
  } else if (g_tune_chunk > 0) {
    pl.chunk_tiles = std::max<int64_t>(1, (g_tune_chunk + tile - 1) / tile);
  } else if (nblk > W) {
    // equal ranges, one per CTA slot; at least one block per range keeps every
    // hand-over one level deep
    pl.mode = kModeStreamK;
    pl.nworkers = W;
  } else if (chunkable) {
    // as many chunks as keep every CTA resident at once (a chunk waits only
    // for earlier chunks, but a second wave would double the makespan)
    int64_t k = std::max<int64_t>(1, W / nblk);
    k = std::min<int64_t>(k, seqlen / kMinChunk);
    pl.chunk_tiles = (T + k - 1) / k;
  }
  if (pl.chunk_tiles < T) {
    pl.nchunks = (int)((T + pl.chunk_tiles - 1) / pl.chunk_tiles);
    if (pl.nchunks > 1) {
      pl.mode = kModeChunked;
      pl.nworkers = nblk * pl.nchunks;
    }
  }
  const size_t hdr = (size_t)scan_header_words() * 4;
  pl.workspace = 0;
  if (pl.mode == kModeStreamK) {
    pl.workspace = hdr + (((size_t)pl.nworkers * 4 + 255) & ~size_t(255)) +
                   (size_t)pl.nworkers * pl.cblk * kDState * sizeof(float);
  } else if (pl.mode == kModeChunked) {
    const int64_t items = nblk * pl.nchunks;
    pl.workspace = hdr + (((size_t)items * 4 + 255) & ~size_t(255)) + (size_t)items * pl.cblk * 48 * sizeof(float);
  }
  return pl;
}

size_t scan_bind_workspace(ScanParams& p, const ScanPlan& plan, void* workspace) {
  const int64_t ncblk = (p.dim + plan.cblk - 1) / plan.cblk;
  p.ncblk = (int)ncblk;
  p.nblk = p.batch * ncblk;
  p.tiles_per_blk = p.seqlen > 0 ? (p.seqlen + plan.tile - 1) / plan.tile : 1;
  p.mode = plan.mode;
  p.nworkers = plan.nworkers;
  p.chunk_tiles = plan.chunk_tiles;
  p.nchunks = plan.nchunks;
  p.ws_header = nullptr;
  p.flags = nullptr;
  p.ws_carry = nullptr;
  if (plan.mode == kModeStatic || !workspace) return 0;
  const int64_t nflags = plan.mode == kModeStreamK ? plan.nworkers : p.nblk * plan.nchunks;
  const size_t hdr = (size_t)scan_header_words() * 4;
  const size_t clear = hdr + (((size_t)nflags * 4 + 255) & ~size_t(255));
  p.ws_header = static_cast<uint32_t*>(workspace);
  p.flags = p.ws_header + scan_header_words();
  p.ws_carry = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + clear);
  return clear;
}

}  // namespace ssk

namespace {

// Checks of the scan's arguments that need no device (sizes, dtypes, NULL
// and misaligned pointers), shared by ss_scan_fwd and ss_scan_fwd_noalloc.
// Sets *empty when the problem has no channel (nothing to do).
ss_status scan_check_args(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, ss_dtype in_dtype,
                          ss_dtype out_dtype, const void* u, const void* delta_raw, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias, const float* h0,
                          const void* y, const float* h_last, const void* workspace, bool* empty) {
  *empty = false;
  if (dstate != ssk::kDState) return fail(SS_ERR_UNSUPPORTED, "dstate must be 16 (got %lld)", (long long)dstate);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0)
    return fail(SS_ERR_INVALID_ARG, "negative size (batch %lld, seqlen %lld, dim %lld)", (long long)batch,
                (long long)seqlen, (long long)dim);
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (batch == 0 || dim == 0) {
    *empty = true;
    return SS_OK;
  }
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
  return SS_OK;
}

// Argument checks, planning and launch shared by ss_scan_fwd and
// ss_scan_fwd_noalloc. `workspace` is the caller's buffer or the library's
// scratch; `noalloc` routes device-side timeouts to the library's fault word
// instead of the workspace header.
ss_status scan_common(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, ss_dtype in_dtype,
                      ss_dtype out_dtype, const void* u, const void* delta_raw, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias, const float* h0,
                      void* y, float* h_last, void* workspace, size_t workspace_bytes, bool noalloc,
                      void* stream, bool static_only = false) {
  bool empty = false;
  ss_status st0 = scan_check_args(batch, seqlen, dim, dstate, in_dtype, out_dtype, u, delta_raw, A, B, C, D, z,
                                  delta_bias, h0, y, h_last, workspace, &empty);
  if (st0 != SS_OK || empty) return st0;
  const ssk::ScanPlan plan =
      ssk::plan_scan(batch, seqlen > 0 ? seqlen : 1, dim, in_dtype, ssk::device_sm_count(), !static_only);
  if (seqlen > 0 && plan.workspace > 0 && (!workspace || workspace_bytes < plan.workspace)) {
    if (noalloc)
      return fail(SS_ERR_INVALID_ARG,
                  "this problem needs %zu bytes of scratch; the no-allocation scan holds at most %zu (use ss_scan_fwd "
                  "with a caller-provided workspace)",
                  plan.workspace, workspace_bytes);
    return fail(SS_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu%s)", plan.workspace, workspace_bytes,
                workspace ? "" : ", NULL");
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (seqlen == 0) {
    if (!h_last) return SS_OK;
    const size_t hbytes = (size_t)batch * dim * ssk::kDState * sizeof(float);
    cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, hbytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h_last, 0, hbytes, s);
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
  p.wait_ns = g_wait_ns;
  p.withhold_item = g_withhold;
  if ((double)plan.nworkers > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  size_t clear = ssk::scan_bind_workspace(p, plan, plan.workspace > 0 ? workspace : nullptr);
  // The fault word: the workspace header when the caller gave a workspace (so
  // ss_scan_status(workspace) reads what this call wrote), else the library's
  // own device word (ss_scan_status(NULL)).
  const size_t hdr = (size_t)ssk::scan_header_words() * 4;
  if (!noalloc && workspace && workspace_bytes >= hdr) {
    if (!p.ws_header) {
      p.ws_header = static_cast<uint32_t*>(workspace);
      clear = hdr;
    }
    p.fault = p.ws_header + 1;
  } else {
    p.fault = ssk::device_fault_word();
    if (!p.fault) return fail(SS_ERR_CUDA, "cannot resolve the library fault word");
  }
  cudaError_t e;
  if (clear > 0) {
    // ticket counter, fault word and hand-over flags start at zero; a reused
    // buffer keeps the previous call's values, so clear them on the stream
    e = cudaMemsetAsync(p.ws_header, 0, clear, s);
    if (e != cudaSuccess) return cuda_fail(e, "workspace initialisation");
  }
  const bool tma = ((size_t)dim * dsize(in_dtype)) % 16 == 0;
  e = ssk::launch_scan_fwd(p, plan, in_dtype, out_dtype, tma, s);
  if (e != cudaSuccess) return cuda_fail(e, "scan launch");
  return SS_OK;
}

}  // namespace

// The backward's workspace with `sg` lanes per channel: the checkpoints, then
// (from a 256-byte boundary) the hand-over area of a split over warps.
static size_t bwd_checkpoint_span(int64_t batch, int64_t seqlen, int64_t dim, int sg) {
  return (ssk::scan_bwd_checkpoint_bytes(batch, seqlen, dim, sg) + 255) / 256 * 256;
}
static size_t bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int sg) {
  return bwd_checkpoint_span(batch, seqlen, dim, sg) + ssk::scan_bwd_handover_bytes(batch, dim, sg);
}

namespace ssk {
// CTAs (contiguous ranges of the sequences' chunks) for the tcgen05 kernel
// with a workspace. A CTA fills an SM (its shared and tensor memory), so CTAs
// run one per SM. With at most one sequence per SM, one CTA per sequence is
// best: a split cannot shorten a sequence, whose state runs through its chunks
// in order. With more sequences than SMs, one CTA per SM takes an equal share
// of all the chunks, so that no SM idles while others run a last partial round
// of sequences. force_steps > 0 sets the range length instead (rounded up to
// whole 128-step chunks), which makes hand-overs on small problems.
int64_t plan_ssd_ranges(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate, int sms,
                        int64_t force_steps) {
  const int64_t nchunk = (seqlen + 127) / 128, units = batch * nheads;
  if ((dstate != 64 && dstate != 128) || nchunk <= 1 || units <= 0) return units;
  if (force_steps > 0) {
    const int64_t rc = std::max<int64_t>(1, (force_steps + 127) / 128);
    return (units * nchunk + rc - 1) / rc;
  }
  return units <= sms ? units : (int64_t)sms;
}
// The split's workspace: a ticket counter (256 bytes), one flag per sequence
// (padded to 256 bytes), then one fp32 state per sequence.
size_t ssd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate) {
  const int64_t nchunk = (seqlen + 127) / 128, units = batch * nheads;
  if ((dstate != 64 && dstate != 128) || nchunk <= 1 || units <= 0) return 0;
  return 256 + (size_t)((units * 4 + 255) / 256 * 256) + (size_t)units * 64 * 128 * sizeof(float);
}
}  // namespace ssk

extern "C" {

int ss_version(void) { return kVersion; }

const char* ss_last_error(void) { return g_err.c_str(); }

void ss_scan_set_tuning(int threads_per_channel, int64_t chunk_len, int max_workers) {
  g_tune_sg = threads_per_channel;
  g_tune_chunk = chunk_len;
  g_tune_workers = max_workers;
}

void ss_scan_set_wait_limit(uint64_t wait_ns, int64_t withhold_item) {
  g_wait_ns = wait_ns > 0 ? wait_ns : 2000000000ull;
  g_withhold = withhold_item;
}

size_t ss_scan_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate) {
  if (batch <= 0 || seqlen <= 0 || dim <= 0 || dstate != ssk::kDState) return 0;
  const int sms = ssk::device_sm_count();
  return std::max(ssk::plan_scan(batch, seqlen, dim, SS_F32, sms).workspace,
                  ssk::plan_scan(batch, seqlen, dim, SS_BF16, sms).workspace);
}

ss_status ss_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, ss_dtype in_dtype,
                      ss_dtype out_dtype, const void* u, const void* delta_raw, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias, const float* h0,
                      void* y, float* h_last, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  return scan_common(batch, seqlen, dim, dstate, in_dtype, out_dtype, u, delta_raw, A, B, C, D, z, delta_bias, h0, y,
                     h_last, workspace, workspace_bytes, false, stream);
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

ss_status ss_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, ss_dtype in_dtype,
                        ss_dtype out_dtype, const void* x, const float* weight, const float* bias,
                        const void* state_in, int silu_on, void* y, void* state_out, void* stream) {
  g_err.clear();
  if (width < 2 || width > 4) return fail(SS_ERR_UNSUPPORTED, "width must be 2, 3 or 4 (got %lld)", (long long)width);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0) return fail(SS_ERR_INVALID_ARG, "negative size");
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (batch == 0 || dim == 0) return SS_OK;
  if (!weight) return fail(SS_ERR_INVALID_ARG, "weight must not be NULL");
  if (seqlen > 0 && (!x || !y)) return fail(SS_ERR_INVALID_ARG, "x and y must not be NULL");
  const void* all[] = {x, weight, bias, state_in, y, state_out};
  const char* names[] = {"x", "weight", "bias", "state_in", "y", "state_out"};
  for (int i = 0; i < 6; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
  if (state_in && state_in == state_out)
    return fail(SS_ERR_INVALID_ARG, "state_out must not be the buffer state_in (use a second buffer)");
  if (seqlen > 0) {
    // byte spans, saturated; [x0, x0 + nx) and [y0, y0 + ny) overlap when the
    // later start lies inside the earlier span
    uint64_t n = 0, nx = UINT64_MAX, ny = UINT64_MAX;
    if (!__builtin_mul_overflow((uint64_t)batch, (uint64_t)seqlen, &n) &&
        !__builtin_mul_overflow(n, (uint64_t)dim, &n)) {
      if (__builtin_mul_overflow(n, (uint64_t)dsize(in_dtype), &nx)) nx = UINT64_MAX;
      if (__builtin_mul_overflow(n, (uint64_t)dsize(out_dtype), &ny)) ny = UINT64_MAX;
    }
    const uint64_t x0 = (uint64_t)(uintptr_t)x, y0 = (uint64_t)(uintptr_t)y;
    if (x0 >= y0 ? x0 - y0 < ny : y0 - x0 < nx) return fail(SS_ERR_INVALID_ARG, "y must not overlap x");
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (seqlen == 0) {
    if (!state_out) return SS_OK;
    const size_t bytes = (size_t)batch * dim * (width - 1) * dsize(in_dtype);
    cudaError_t e = state_in ? cudaMemcpyAsync(state_out, state_in, bytes, cudaMemcpyDeviceToDevice, s)
                             : cudaMemsetAsync(state_out, 0, bytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state copy");
  }
  ssk::ConvParams p{x, weight, bias, state_in, y, state_out, batch, seqlen, dim, (int)width, silu_on ? 1 : 0,
                    ssk::device_fault_word()};
  if (!p.fault) return fail(SS_ERR_CUDA, "cannot resolve the library fault word");
  const bool vec = ((size_t)dim * dsize(in_dtype)) % 16 == 0;
  cudaError_t e = ssk::launch_conv1d_fwd(p, in_dtype, out_dtype, vec, s);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d launch");
  return SS_OK;
}

ss_status ss_conv1d_update(int64_t batch, int64_t dim, int64_t width, ss_dtype in_dtype, ss_dtype out_dtype,
                           void* state, const void* x, const float* weight, const float* bias, int silu_on, void* y,
                           void* stream) {
  g_err.clear();
  if (width < 2 || width > 4) return fail(SS_ERR_UNSUPPORTED, "width must be 2, 3 or 4 (got %lld)", (long long)width);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || dim < 0) return fail(SS_ERR_INVALID_ARG, "negative size");
  if (batch == 0 || dim == 0) return SS_OK;
  const void* need[] = {state, x, weight, y};
  const char* names[] = {"state", "x", "weight", "y"};
  for (int i = 0; i < 4; i++)
    if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  const void* all[] = {state, x, weight, bias, y};
  const char* all_names[] = {"state", "x", "weight", "bias", "y"};
  for (int i = 0; i < 5; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  ssk::ConvParams p{x, weight, bias, nullptr, y, state, batch, 1, dim, (int)width, silu_on ? 1 : 0, nullptr};
  // whole 16-byte vectors of channels per thread when a vector never straddles two batch rows
  const bool vec = ((size_t)dim * dsize(in_dtype)) % 16 == 0;
  cudaError_t e = ssk::launch_conv1d_update(p, in_dtype, out_dtype, vec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "conv1d update launch");
  return SS_OK;
}

size_t ss_scan_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate) {
  if (batch <= 0 || seqlen <= 0 || dim <= 0 || dstate != ssk::kDState) return 0;
  return std::max(bwd_workspace_bytes(batch, seqlen, dim, 1), bwd_workspace_bytes(batch, seqlen, dim, 2));
}

ss_status ss_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, ss_dtype in_dtype,
                      ss_dtype dy_dtype, const void* u, const void* delta_raw, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* delta_bias, const float* h0,
                      const void* dy, const float* dh_last, void* du, void* ddelta_raw, void* dz, float* dA,
                      float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0, void* workspace,
                      size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (dstate != ssk::kDState) return fail(SS_ERR_UNSUPPORTED, "dstate must be 16 (got %lld)", (long long)dstate);
  if (!valid_dtype(in_dtype) || !valid_dtype(dy_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, dy %d)", (int)in_dtype, (int)dy_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0) return fail(SS_ERR_INVALID_ARG, "negative size");
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (batch == 0 || dim == 0) return SS_OK;
  if ((double)batch * (double)seqlen * (double)dim > 4.0e18) return fail(SS_ERR_INVALID_ARG, "problem too large");
  if (!A || !dA) return fail(SS_ERR_INVALID_ARG, "A and dA must not be NULL");
  if (seqlen > 0) {
    const void* need[] = {u, delta_raw, B, C, dy, du, ddelta_raw, dB, dC};
    const char* names[] = {"u", "delta_raw", "B", "C", "dy", "du", "ddelta_raw", "dB", "dC"};
    for (int i = 0; i < 9; i++)
      if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
    if (z && !dz) return fail(SS_ERR_INVALID_ARG, "dz must not be NULL when z is given");
  }
  const void* all[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, dy, dh_last, du, ddelta_raw, dz,
                       dA, dB, dC, dD, ddelta_bias, dh0, workspace};
  const char* all_names[] = {"u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "h0", "dy", "dh_last",
                             "du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0", "workspace"};
  for (int i = 0; i < 21; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  const int sg = bwd_lanes_per_channel(batch, dim);
  const size_t need_ws = seqlen > 0 ? bwd_workspace_bytes(batch, seqlen, dim, sg) : 0;
  if (need_ws > 0 && (!workspace || workspace_bytes < need_ws))
    return fail(SS_ERR_INVALID_ARG, "workspace of %zu bytes needed (got %zu%s)", need_ws, workspace_bytes,
                workspace ? "" : ", NULL");
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the summed gradients start at zero
  cudaError_t e = cudaMemsetAsync(dA, 0, (size_t)dim * ssk::kDState * sizeof(float), s);
  if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, (size_t)dim * sizeof(float), s);
  if (e == cudaSuccess && ddelta_bias) e = cudaMemsetAsync(ddelta_bias, 0, (size_t)dim * sizeof(float), s);
  if (e == cudaSuccess && seqlen > 0) e = cudaMemsetAsync(dB, 0, (size_t)batch * seqlen * ssk::kDState * sizeof(float), s);
  if (e == cudaSuccess && seqlen > 0) e = cudaMemsetAsync(dC, 0, (size_t)batch * seqlen * ssk::kDState * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "gradient initialisation");
  if (seqlen == 0) {
    // no step: the state gradient passes through unchanged
    if (!dh0) return SS_OK;
    const size_t hbytes = (size_t)batch * dim * ssk::kDState * sizeof(float);
    e = dh_last ? cudaMemcpyAsync(dh0, dh_last, hbytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dh0, 0, hbytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state gradient copy");
  }
  ssk::BwdParams p{};
  p.u = u;
  p.delta_raw = delta_raw;
  p.z = z;
  p.B = B;
  p.C = C;
  p.A = A;
  p.D = D;
  p.delta_bias = delta_bias;
  p.h0 = h0;
  p.dy = dy;
  p.dh_last = dh_last;
  p.du = du;
  p.ddelta_raw = ddelta_raw;
  p.dz = z ? dz : nullptr;
  p.dA = dA;
  p.dB = dB;
  p.dC = dC;
  p.dD = dD;
  p.dbias = ddelta_bias;
  p.dh0 = dh0;
  p.ckpt = static_cast<float*>(workspace);
  p.batch = batch;
  p.seqlen = seqlen;
  p.dim = dim;
  p.ncblk = (int)((dim + 32 / sg - 1) / (32 / sg));
  p.nsub = ssk::scan_bwd_subtiles(seqlen);
  if ((double)batch * p.ncblk > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  {
    const int64_t blocks = batch * (int64_t)p.ncblk;
    uint8_t* w = static_cast<uint8_t*>(workspace) + bwd_checkpoint_span(batch, seqlen, dim, sg);
    const size_t fb = (size_t)((blocks * 4 + 255) / 256 * 256);
    p.flags_h = reinterpret_cast<unsigned int*>(w);
    p.flags_lam = reinterpret_cast<unsigned int*>(w + fb);
    p.ws_h = reinterpret_cast<float*>(w + 2 * fb);
    p.ws_lam = p.ws_h + blocks * 32 * ssk::kDState;
    p.fault = ssk::device_fault_word();
    p.wait_ns = g_wait_ns;
    p.withhold_share = g_withhold;
    // chunk_len > 0: shares of that many steps (whole 16-step sub-tiles)
    const int64_t rt = g_tune_chunk > 0 ? std::max<int64_t>(1, (g_tune_chunk + 15) / 16) : 0;
    p.force_shares = rt > 0 ? (blocks * p.nsub + rt - 1) / rt : 0;
    if (!p.fault) return fail(SS_ERR_CUDA, "cannot resolve the library fault word");
  }
  e = ssk::launch_scan_bwd(p, sg, in_dtype, dy_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "scan backward launch");
  return SS_OK;
}

size_t ss_scan_fwd_general_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                          int64_t ngroups, ss_disc disc, ss_dtype in_dtype) {
  // the CTA kernel splits units; d_state 16 in one group with the first-order
  // rule runs on the scan kernel's static split, and other shapes on the
  // one-warp kernel, neither of which uses one
  if (batch <= 0 || seqlen <= 0 || dim <= 0 || ngroups < 1 || dim % ngroups != 0 || !valid_dtype(in_dtype))
    return 0;
  if (dstate == 16 || !ssk::scan_general_cta_shape_ok(dim, dstate, dim / ngroups, in_dtype)) return 0;
  (void)disc;
  return ssk::scan_general_cta_workspace_bytes(batch, seqlen, dim, dstate);
}

ss_status ss_scan_fwd_general(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t ngroups,
                              ss_disc disc, ss_dtype in_dtype, ss_dtype out_dtype, const void* u,
                              const void* delta_raw, const float* A, const void* B, const void* C, const float* D,
                              const void* z, const float* delta_bias, const float* h0, void* y, float* h_last,
                              void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (dstate != 16 && dstate != 32 && dstate != 64 && dstate != 128)
    return fail(SS_ERR_UNSUPPORTED, "dstate must be 16, 32, 64 or 128 (got %lld)", (long long)dstate);
  if (disc != SS_DISC_FIRST_ORDER && disc != SS_DISC_ZOH)
    return fail(SS_ERR_UNSUPPORTED, "unknown discretisation %d", (int)disc);
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
    return fail(SS_ERR_UNSUPPORTED, "unknown dtype (in %d, out %d)", (int)in_dtype, (int)out_dtype);
  if (batch < 0 || seqlen < 0 || dim < 0 || ngroups < 1)
    return fail(SS_ERR_INVALID_ARG, "negative size or ngroups < 1");
  if (batch > INT32_MAX || seqlen > INT32_MAX || dim > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (dim > 0 && dim % ngroups != 0)
    return fail(SS_ERR_INVALID_ARG, "dim (%lld) is not a multiple of ngroups (%lld)", (long long)dim,
                (long long)ngroups);
  if (batch == 0 || dim == 0) return SS_OK;
  if ((double)batch * (double)seqlen * (double)dim * (double)dstate > 4.0e18)
    return fail(SS_ERR_INVALID_ARG, "problem too large");
  // d_state 16, one group, first order is exactly the selective scan of
  // ss_scan_fwd (B and C [batch, seqlen, 1, 16] are [batch, seqlen, 16]): run it
  // on that kernel, in its static split, which needs no workspace
  if (dstate == 16 && ngroups == 1 && disc == SS_DISC_FIRST_ORDER)
    return scan_common(batch, seqlen, dim, dstate, in_dtype, out_dtype, u, delta_raw, A, B, C, D, z, delta_bias, h0,
                       y, h_last, nullptr, 0, false, stream, true);
  const void* need[] = {u, delta_raw, A, B, C, y};
  const char* names[] = {"u", "delta_raw", "A", "B", "C", "y"};
  if (seqlen > 0) {
    for (int i = 0; i < 6; i++)
      if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  }
  const void* all[] = {u, delta_raw, A, B, C, D, z, delta_bias, h0, y, h_last, workspace};
  const char* all_names[] = {"u", "delta_raw", "A", "B", "C", "D", "z", "delta_bias", "h0", "y", "h_last",
                             "workspace"};
  for (int i = 0; i < 12; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  const size_t ws_need = ss_scan_fwd_general_workspace_size(batch, seqlen, dim, dstate, ngroups, disc, in_dtype);
  if (workspace && ws_need > 0 && workspace_bytes < ws_need)
    return fail(SS_ERR_INVALID_ARG, "workspace too small (%zu bytes, need %zu)", workspace_bytes, ws_need);
  if (ws_need > 0 && (double)batch * (double)dim > 2.0e9)
    return fail(SS_ERR_INVALID_ARG, "problem too large");
  const int sg = (int)(dstate / 16);
  const int64_t cw = 32 / sg;
  const int64_t ncblk = (dim + cw - 1) / cw;
  const int64_t cpg = dim / ngroups;
  int ngw_max = 1;
  for (int64_t k = 0; k < ncblk; k++) {
    const int64_t c0 = k * cw, c1 = std::min(c0 + cw, dim) - 1;
    ngw_max = std::max(ngw_max, (int)(c1 / cpg - c0 / cpg + 1));
  }
  const int smem = 2 * ssk::scan_general_stage_bytes(dstate, ngw_max, in_dtype);
  if (smem > 227 * 1024)
    return fail(SS_ERR_UNSUPPORTED, "staging of %d groups per warp needs %d bytes of shared memory", ngw_max, smem);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (seqlen == 0) {
    if (!h_last) return SS_OK;
    const size_t hbytes = (size_t)batch * dim * dstate * sizeof(float);
    cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, hbytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h_last, 0, hbytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state copy");
  }
  const size_t es = dsize(in_dtype);
  const size_t in_row = (size_t)cw * es;
  int chunk = 0;
  if (((size_t)dim * es) % 16 == 0 && in_row % 16 == 0) chunk = 16;
  else if (((size_t)dim * es) % 4 == 0 && in_row % 4 == 0) chunk = 4;
  ssk::GenParams p{u, delta_raw, z, B, C, A, D, delta_bias, h0, y, h_last, batch, seqlen, dim, ngroups, cpg,
                   (int)ncblk, ngw_max, chunk, (int)disc, ssk::device_fault_word(), g_wait_ns};
  p.workspace = ws_need > 0 ? workspace : nullptr;
  p.force_steps = g_tune_chunk;
  p.withhold_range = g_withhold;
  if ((double)batch * ncblk > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  cudaError_t e = ssk::scan_general_cta_supported(dim, dstate, cpg, in_dtype)
                      ? ssk::launch_scan_general_cta(p, dstate, in_dtype, out_dtype, s)
                      : ssk::launch_scan_general(p, sg, in_dtype, out_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "generalised scan launch");
  return SS_OK;
}


size_t ss_ssd_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate) {
  if (batch < 0 || seqlen < 0 || nheads < 0) return 0;
  if ((double)batch * (double)nheads * (double)seqlen > 4.0e18) return 0;
  return ssk::ssd_workspace_bytes(batch, seqlen, nheads, dstate);
}

ss_status ss_ssd_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                     int64_t ngroups, ss_dtype in_dtype, ss_dtype out_dtype, const void* x, const void* dt,
                     const float* A, const void* B, const void* C, const float* D, const float* dt_bias,
                     const float* h0, void* y, float* h_last, void* workspace, size_t workspace_bytes,
                     void* stream) {
  g_err.clear();
  if (in_dtype != SS_BF16) return fail(SS_ERR_UNSUPPORTED, "the state-space-dual layer takes bf16 inputs");
  if (!valid_dtype(out_dtype)) return fail(SS_ERR_UNSUPPORTED, "unknown output dtype %d", (int)out_dtype);
  if (headdim != 64) return fail(SS_ERR_UNSUPPORTED, "headdim must be 64 (got %lld)", (long long)headdim);
  if (dstate != 64 && dstate != 128)
    return fail(SS_ERR_UNSUPPORTED, "dstate must be 64 or 128 (got %lld)", (long long)dstate);
  if (batch < 0 || seqlen < 0 || nheads < 0 || ngroups < 1)
    return fail(SS_ERR_INVALID_ARG, "negative size or ngroups < 1");
  if (batch > INT32_MAX || seqlen > INT32_MAX || nheads > INT32_MAX)
    return fail(SS_ERR_INVALID_ARG, "a size exceeds 2^31-1");
  if (nheads > 0 && nheads % ngroups != 0)
    return fail(SS_ERR_INVALID_ARG, "nheads (%lld) is not a multiple of ngroups (%lld)", (long long)nheads,
                (long long)ngroups);
  if (batch == 0 || nheads == 0) return SS_OK;
  if ((double)batch * (double)seqlen * (double)nheads * 64.0 > 4.0e18)
    return fail(SS_ERR_INVALID_ARG, "problem too large");
  if (!A) return fail(SS_ERR_INVALID_ARG, "A must not be NULL");
  if (seqlen > 0) {
    const void* need[] = {x, dt, B, C, y};
    const char* names[] = {"x", "dt", "B", "C", "y"};
    for (int i = 0; i < 5; i++)
      if (!need[i]) return fail(SS_ERR_INVALID_ARG, "%s must not be NULL", names[i]);
  }
  const void* all[] = {x, dt, A, B, C, D, dt_bias, h0, y, h_last, workspace};
  const char* all_names[] = {"x", "dt", "A", "B", "C", "D", "dt_bias", "h0", "y", "h_last", "workspace"};
  for (int i = 0; i < 11; i++)
    if (all[i] && !aligned16(all[i])) return fail(SS_ERR_INVALID_ARG, "%s is not 16-byte aligned", all_names[i]);
  const size_t need = ssk::ssd_workspace_bytes(batch, seqlen, nheads, dstate);
  if (workspace && need > 0 && workspace_bytes < need)
    return fail(SS_ERR_INVALID_ARG, "workspace too small (%zu bytes, need %zu)", workspace_bytes, need);
  ss_status st = check_device();
  if (st != SS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (seqlen == 0) {
    if (!h_last) return SS_OK;
    const size_t hbytes = (size_t)batch * nheads * 64 * dstate * sizeof(float);
    cudaError_t e = h0 ? cudaMemcpyAsync(h_last, h0, hbytes, cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(h_last, 0, hbytes, s);
    return e == cudaSuccess ? SS_OK : cuda_fail(e, "empty-sequence state copy");
  }
  if ((double)batch * nheads > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
  ssk::SsdParams p{x, dt, A, B, C, D, dt_bias, h0, y, h_last, batch, seqlen, nheads, ngroups,
                   ssk::device_fault_word(), g_wait_ns, dstate};
  p.ranges = batch * nheads;  // one CTA per sequence
  p.ws_ticket = nullptr;
  p.ws_flags = nullptr;
  p.ws_state = nullptr;
  p.withhold_range = g_withhold;
  cudaError_t e = cudaSuccess;
  if (workspace && need > 0) {
    const int64_t R = ssk::plan_ssd_ranges(batch, seqlen, nheads, dstate, ssk::device_sm_count(), g_tune_chunk);
    if (R != p.ranges) {  // ranges that cut sequences: hand-overs through the workspace
      if ((double)R > 2.0e9) return fail(SS_ERR_INVALID_ARG, "grid too large");
      uint8_t* w = static_cast<uint8_t*>(workspace);
      const size_t flags_bytes = (size_t)((batch * nheads * 4 + 255) / 256 * 256);
      p.ranges = R;
      p.ws_ticket = reinterpret_cast<unsigned int*>(w);
      p.ws_flags = reinterpret_cast<unsigned int*>(w + 256);
      p.ws_state = reinterpret_cast<float*>(w + 256 + flags_bytes);
      if ((e = cudaMemsetAsync(w, 0, 256 + flags_bytes, s)) != cudaSuccess)
        return cuda_fail(e, "state-space-dual workspace reset");
    }
  }
  e = ssk::launch_ssd_fwd_tc(p, out_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "state-space-dual launch");
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
  // argument checks, then sizes beyond the fixed scratch, before any device call
  bool empty = false;
  ss_status st0 = scan_check_args(batch, seqlen, dim, dstate, in_dtype, out_dtype, u, delta_raw, A, B, C, D, z,
                                  delta_bias, h0, y, h_last, nullptr, &empty);
  if (st0 != SS_OK || empty) return st0;
  if (seqlen > 0) {
    const size_t need = ssk::plan_scan(batch, seqlen, dim, in_dtype, ssk::device_sm_count()).workspace;
    if (need > (size_t)SS_SCAN_NOALLOC_SCRATCH_BYTES)
      return fail(SS_ERR_INVALID_ARG,
                  "this problem needs %zu bytes of scratch; the no-allocation scan holds at most %zu (use ss_scan_fwd "
                  "with a caller-provided workspace)",
                  need, (size_t)SS_SCAN_NOALLOC_SCRATCH_BYTES);
  }
  void* scratch = nullptr;
  if (batch > 0 && dim > 0 && seqlen > 0) {
    ss_status st = check_device();
    if (st != SS_OK) return st;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if ((st = noalloc_scratch(dev, &scratch)) != SS_OK) return st;
  }
  return scan_common(batch, seqlen, dim, dstate, in_dtype, out_dtype, u, delta_raw, A, B, C, D, z, delta_bias, h0, y,
                     h_last, scratch, SS_SCAN_NOALLOC_SCRATCH_BYTES, true, stream);
}
