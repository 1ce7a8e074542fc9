// Internal host/device interface between the C ABI (ss_api.cu) and the
// kernels (ss_scan_fwd.cu, ss_state_update.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ss_scan.h"

namespace ssk {

constexpr int kDState = 16;

// How the (channel block, tile) work of one scan is split among CTAs.
enum ScanMode : int {
  kModeStatic = 0,   // one CTA per channel block, whole sequence; no workspace
  kModeStreamK = 1,  // contiguous equal ranges of the tile space per CTA; states
                     // handed over at block-interior range boundaries
  kModeChunked = 2   // sequence chunks per block, carries combined by look-back
};

// Parameters of one scan launch (device pointers, sizes, schedule).
struct ScanParams {
  const void* u;
  const void* delta_raw;
  const void* z;            // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;           // may be null
  const float* delta_bias;  // may be null
  const float* h0;          // may be null
  void* y;
  float* h_last;            // may be null
  // workspace (stream-K and chunked modes)
  uint32_t* ws_header;      // [0] ticket counter, [1] fault word, [2] magic; may be null (static mode)
  uint32_t* flags;          // stream-K: one per worker; chunked: one per (block, chunk)
  float* ws_carry;          // stream-K: handed-over states [worker][channel][16];
                            // chunked: per (block, chunk, channel) P[16], S_local[16], S_incl[16]
  unsigned int* fault;      // fault word (workspace header or the library's own)
  uint64_t wait_ns;         // limit of every device-side wait
  int64_t withhold_item;    // test knob: the hand-over (stream-K worker) or chunk whose
                            // flag is never published (-1: none)
  int64_t batch, seqlen, dim;
  int mode;                 // ScanMode
  int ncblk;                // channel blocks per batch element
  int64_t nblk;             // batch * ncblk
  int64_t tiles_per_blk;    // ceil(seqlen / tile)
  int64_t nworkers;         // CTAs (static: nblk; stream-K: ranges; chunked: nblk * nchunks)
  int64_t chunk_tiles;      // chunked: tiles per chunk
  int nchunks;              // chunked: chunks per block
};

// Parameters of one decode step.
struct StepParams {
  float* h;
  const void* u;
  const void* delta_raw;
  const void* z;
  const void* B;
  const void* C;
  const float* A;
  const float* D;
  const float* delta_bias;
  void* y;
  int64_t batch, dim;
};

// Parameters of the convolution front-end (forward: x [batch, seqlen, dim],
// state_in/state_out [batch, dim, width-1]; decode: x [batch, dim], state_out
// is the state updated in place).
struct ConvParams {
  const void* x;
  const float* w;        // [dim, width]
  const float* bias;     // [dim] or null
  const void* state_in;  // may be null (zeros before t = 0)
  void* y;
  void* state_out;       // may be null (forward)
  int64_t batch, seqlen, dim;
  int width;
  int silu;
  unsigned int* fault;   // the library's fault word (bounded waits of the forward pass)
};

// Parameters of the scan's backward pass (inputs of the forward, the output
// gradient, and the gradients written; see ss_scan_bwd).
struct BwdParams {
  const void* u;
  const void* delta_raw;
  const void* z;            // may be null
  const void* B;
  const void* C;
  const float* A;
  const float* D;           // may be null
  const float* delta_bias;  // may be null
  const float* h0;          // may be null
  const void* dy;
  const float* dh_last;     // may be null
  void* du;
  void* ddelta_raw;
  void* dz;                 // null when z is null
  float* dA;                // accumulated: zero before the launch
  float* dB;                // accumulated
  float* dC;                // accumulated
  float* dD;                // accumulated; may be null
  float* dbias;             // accumulated; may be null
  float* dh0;               // may be null
  float* ckpt;              // workspace: states saved every few steps
  int64_t batch, seqlen, dim;
  int ncblk;                // channel blocks (32 / sg channels) per batch element
  int64_t nsub;             // recomputed sub-tiles per block
  // Work split: the (block, sub-tile) items of all blocks, block-major, cut
  // into `nshares` contiguous shares, one per warp. Where a share starts
  // inside a block, the state entering it comes from the share before (through
  // ws_h / flags_h = the sub-tile of the cut), and the adjoint leaving it goes
  // back (through ws_lam / flags_lam = nsub - that sub-tile). nshares equal to
  // the number of blocks: one warp per block, no hand-over.
  int64_t nshares;
  unsigned int* flags_h;    // [blocks], zeroed before the launch
  unsigned int* flags_lam;  // [blocks], zeroed before the launch
  float* ws_h;              // [blocks, 512]
  float* ws_lam;            // [blocks, 512]
  unsigned int* fault;      // the library's fault word (timed-out waits)
  uint64_t wait_ns;         // limit of a device-side wait; 0 = the default
  int64_t withhold_share;   // test knob: this share publishes no hand-over (-1: none)
  int64_t force_shares;     // > 0: this many shares instead of the automatic plan (needs the slots)
};

// Parameters of the generalised scan (state size 16-128, grouped B/C, ZOH).
struct GenParams {
  const void* u;
  const void* delta_raw;
  const void* z;            // may be null
  const void* B;            // [batch, seqlen, ngroups, dstate]
  const void* C;
  const float* A;           // [dim, dstate]
  const float* D;           // may be null
  const float* delta_bias;  // may be null
  const float* h0;          // may be null
  void* y;
  float* h_last;            // may be null
  int64_t batch, seqlen, dim, ngroups;
  int64_t cpg;              // channels per group (dim / ngroups)
  int ncblk;                // channel blocks (32 / sg channels) per batch element
  int ngw_max;              // most groups one channel block spans
  int chunk_in;             // staging of u, delta_raw, z rows: 16- or 4-byte copies, or 0 (element-wise)
  int disc;                 // 0 first order, 1 zero-order hold
  unsigned int* fault;      // the library's fault word (timed-out waits)
  uint64_t wait_ns;         // limit of a device-side wait; 0 = the default
  // Work split of the CTA kernel. Its (unit, tile) items (a unit is one
  // channel block of one batch element), unit-major, are cut into `ranges`
  // contiguous shares, one per CTA. With a workspace the CTAs take shares by
  // ticket, and a share that starts inside a unit starts from the state the
  // share before it left in ws_state[unit], published through ws_flags[unit]
  // = the tile where the hand-over happens. The launch plans the shares from
  // `workspace` (null: one CTA per unit) and `force_steps`.
  void* workspace;          // the caller's workspace, or null
  int64_t force_steps;      // > 0: share length in steps instead of the automatic plan
  int64_t withhold_range;   // test knob: this share does not publish its state (-1: none)
  int64_t ranges;           // set by the launch
  unsigned int* ws_ticket;  //   ticket counter (or null: shares by block index)
  unsigned int* ws_flags;   //   [units]
  float* ws_state;          //   [units, 2048]
};

// Parameters of the state-space-dual (Mamba-2) layer forward.
struct SsdParams {
  const void* x;            // [batch, seqlen, nheads, 64] bf16
  const void* dt;           // [batch, seqlen, nheads] bf16
  const float* A;           // [nheads]
  const void* B;            // [batch, seqlen, ngroups, dstate] bf16
  const void* C;
  const float* D;           // [nheads] or null
  const float* dt_bias;     // [nheads] or null
  const float* h0;          // [batch, nheads, 64, dstate] or null
  void* y;                  // [batch, seqlen, nheads, 64]
  float* h_last;            // [batch, nheads, 64, dstate] or null
  int64_t batch, seqlen, nheads, ngroups;
  unsigned int* fault;      // the library's fault word (timed-out waits)
  uint64_t wait_ns;         // limit of a device-side wait; 0 = the default
  int64_t dstate;           // 64 or 128 (64: B and C run zero-padded to 128 columns)
  // Work split: the chunks of all (batch, head) sequences, sequence-major,
  // cut into `ranges` contiguous ranges, one per CTA. With a workspace the
  // CTAs take ranges in the order of a ticket counter, and a range that starts
  // inside a sequence starts from the state the range before it left in
  // ws_state[(batch, head)], published through ws_flags[(batch, head)] = the
  // chunk where the hand-over happens. Without one (ws_ticket null) there is
  // one range per sequence, taken by block index.
  int64_t ranges;
  unsigned int* ws_ticket;  // zeroed before the launch, or null
  unsigned int* ws_flags;   // [batch * nheads], zeroed before the launch
  float* ws_state;          // [batch * nheads, 64, 128]
  int64_t withhold_range;   // test knob: this ticket does not publish its state (-1: none)
};
// SSD split plan: CTAs (ranges of the sequences' chunks) for `sms` SMs, and
// the workspace bytes a split needs (0 when it cannot help).
int64_t plan_ssd_ranges(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate, int sms, int64_t force_steps);
size_t ssd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate);

// Launch plan for a scan problem.
struct ScanPlan {
  int sg;               // threads per channel (1 or 2); each owns 16/sg states
  int tile;             // timesteps per tile
  int cblk;             // channels per CTA (channel block)
  int mode;             // ScanMode
  int64_t nworkers;     // CTAs with work
  int64_t chunk_tiles;  // chunked mode: tiles per chunk
  int nchunks;          // chunked mode: chunks per block
  size_t workspace;     // bytes of workspace needed
};

// Plan for `sms` streaming multiprocessors (one CTA per SM at a time).
// with_workspace false: the static plan only (one CTA per channel block, no
// cross-CTA hand-over, no workspace).
ScanPlan plan_scan(int64_t batch, int64_t seqlen, int64_t dim, ss_dtype in_dtype, int sms,
                   bool with_workspace = true);
// SM count of the current device (cached per device), or a default when it
// cannot be queried.
int device_sm_count();

// Fill the schedule fields of `p` from `plan` and carve `workspace` (at least
// plan.workspace bytes, may be null when that is 0). Returns the number of
// leading workspace bytes that must be zero before the launch.
size_t scan_bind_workspace(ScanParams& p, const ScanPlan& plan, void* workspace);

// Launchers; return cudaSuccess or the launch error.
cudaError_t launch_scan_fwd(const ScanParams& p, const ScanPlan& plan, ss_dtype in_dtype, ss_dtype out_dtype,
                            bool use_tma, cudaStream_t stream);

// Shape constants of the scan kernels.
int scan_channels_per_block(int sg);           // channels per CTA
int scan_tile_len(ss_dtype in_dtype, int sg);  // timesteps per tile
int scan_header_words();
uint32_t scan_header_magic();
cudaError_t launch_state_update(const StepParams& p, ss_dtype in_dtype, ss_dtype out_dtype, cudaStream_t stream);
cudaError_t launch_conv1d_fwd(const ConvParams& p, ss_dtype in_dtype, ss_dtype out_dtype, bool vec,
                              cudaStream_t stream);
cudaError_t launch_conv1d_update(const ConvParams& p, ss_dtype in_dtype, ss_dtype out_dtype, bool vec,
                                 cudaStream_t stream);

// sg: lanes per channel (1 or 2); p.ncblk counts blocks of 32 / sg channels
cudaError_t launch_scan_bwd(const BwdParams& p, int sg, ss_dtype in_dtype, ss_dtype dy_dtype, cudaStream_t stream);
size_t scan_bwd_checkpoint_bytes(int64_t batch, int64_t seqlen, int64_t dim, int sg);
int64_t scan_bwd_subtiles(int64_t seqlen);
size_t scan_bwd_handover_bytes(int64_t batch, int64_t dim, int sg);

// sg = dstate / 16 lanes per channel; bytes of one staged 16-step sub-tile
cudaError_t launch_scan_general(const GenParams& p, int sg, ss_dtype in_dtype, ss_dtype out_dtype,
                                cudaStream_t stream);
int scan_general_stage_bytes(int64_t dstate, int ngw_max, ss_dtype in_dtype);
// CTA-cooperative generalised scan (ss_scan_general_cta.cu): d_state 32, 64 or
// 128 with every CTA's channels in one group and 16-byte rows.
bool scan_general_cta_supported(int64_t dim, int64_t dstate, int64_t cpg, ss_dtype in_dtype);
// the shape conditions alone (no driver query)
bool scan_general_cta_shape_ok(int64_t dim, int64_t dstate, int64_t cpg, ss_dtype in_dtype);
// Workspace bytes the CTA kernel can use to split units across CTAs (0: none).
size_t scan_general_cta_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate);
cudaError_t launch_scan_general_cta(const GenParams& p, int64_t dstate, ss_dtype in_dtype, ss_dtype out_dtype,
                                    cudaStream_t stream);

// the state-space-dual layer on the tcgen05 tensor cores (ss_ssd_tc.cu)
cudaError_t launch_ssd_fwd_tc(const SsdParams& p, ss_dtype out_dtype, cudaStream_t stream);

// The library's own fault word (device symbol), used when no workspace is given.
unsigned int* device_fault_word();

}  // namespace ssk
