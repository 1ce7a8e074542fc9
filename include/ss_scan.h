/*
 * ss_scan.h — C ABI of the B300 (sm_103a) selective state-space scan library
 * (libssscan.so).
 *
 * What it computes (the S6 layer's scan; its gradients are in ss_scan_bwd). For every batch
 * element b and channel d, with state h[n] (n < dstate) starting at h0[b,d,:]
 * (zeros when h0 is NULL), for t = 0 .. seqlen-1:
 *
 *   delta   = softplus(delta_raw[b,t,d] + delta_bias[d])
 *   h[n]    = exp(delta * A[d,n]) * h[n] + delta * B[b,t,n] * u[b,t,d]
 *   yv      = sum_n C[b,t,n] * h[n] + D[d] * u[b,t,d]
 *   y[b,t,d]= yv * silu(z[b,t,d])                 (yv itself when z is NULL)
 *
 * and h_last[b,d,:] = h after the last step. Passages:
 *  - recurrence h_t = Abar h_{t-1} + Bbar x_t, y_t = C h_t + D x_t:
 *    "Transformer时代终结？Mamba的状态空间革命重塑AI底层架构", section 二.1;
 *  - Abar = exp(delta*A) and the first-order Bbar = delta*B, with delta, B, C
 *    produced per token and B, C shared by all channels: the mlqm.cn SSM
 *    tutorial, sections 3.2, 5.2 and the 9.2 step sketch;
 *  - A = -exp(A_log) keeps |Abar| < 1: "外文文献精读：Mamba - 线性时间序列建模
 *    与结构化状态空间模型", section 4.1 (A is passed already exponentiated);
 *  - SiLU gate on the SSM output: "Mamba: Linear-Time Sequence Modeling with
 *    Selective State Spaces" (review page), method step 3; tutorial section 7.1;
 *  - softplus for delta is not printed on the pages; it is the standard
 *    softplus(x) = log(1 + e^x).
 * The decode entry point is the same step with seqlen = 1 and h updated in
 * place ("AI 推理系列（十四）：Mamba 的 Selective State Space", section on
 * Selective Scan for training and Decode: prefill by scan, then per-token
 * in-place state updates).
 *
 * Conventions shared by all entry points:
 *  - Every data pointer is a DEVICE pointer owned by the caller, 16-byte
 *    aligned, to a dense row-major (C-contiguous) array. The library never
 *    allocates device memory and keeps no pointer after a call returns.
 *  - u, delta_raw, z, B, C share `in_dtype` (SS_F32 or SS_BF16). A, D,
 *    delta_bias, h0, h_last and the decode state h are float32. y has
 *    `out_dtype`.
 *  - dstate must be 16 (SS_ERR_UNSUPPORTED otherwise).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on that stream; the return code covers argument checks and
 *    launch errors only. A device-side wait that gave up is reported later by
 *    ss_scan_status().
 *  - Empty problems (batch == 0 or dim == 0) launch nothing and return SS_OK.
 *  - On any error the call launches nothing (or stops at the failing launch)
 *    and ss_last_error() returns a message for the calling host thread.
 *  - The library runs on compute capability 10.3 devices (B300) only.
 */
#ifndef SS_SCAN_H
#define SS_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SS_OK = 0,
  SS_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, too-small workspace */
  SS_ERR_UNSUPPORTED = 2, /* dstate != 16, unknown dtype, wrong device */
  SS_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  SS_ERR_TIMEOUT = 4      /* a device-side bounded wait gave up (see ss_scan_status) */
} ss_status;

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int ss_version(void);

/* Message describing the last error on this host thread ("" if none). The
 * pointer stays valid until the next call on the same thread. */
const char *ss_last_error(void);

/*
 * Bytes of device workspace that ss_scan_fwd needs for this problem size (for
 * either input dtype). When the work is split along the sequence, states and
 * chunk carries (prod Abar, state) pass between warps through this workspace,
 * together with a ticket counter and per-boundary flags; problems run as one
 * warp per channel block need none (0 is returned). Depends only on the sizes
 * and the calling thread's tuning settings.
 */
size_t ss_scan_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate);

/*
 * Selective scan forward.
 *  u, delta_raw, z : [batch, seqlen, dim]   in_dtype; z may be NULL (no gate)
 *  A               : [dim, dstate]          float32 (the negative real diagonal)
 *  B, C            : [batch, seqlen, dstate] in_dtype, shared by all channels
 *  D               : [dim] float32 or NULL (no skip term)
 *  delta_bias      : [dim] float32 or NULL (zero)
 *  h0              : [batch, dim, dstate] float32 or NULL (zero initial state)
 *  y               : [batch, seqlen, dim]   out_dtype (output)
 *  h_last          : [batch, dim, dstate] float32 or NULL (final state, output)
 *  workspace       : device buffer of at least ss_scan_fwd_workspace_size()
 *                    bytes (may be NULL when that size is 0). When a buffer of
 *                    at least 256 bytes is given, the call also keeps its
 *                    fault record there (read by ss_scan_status(workspace)),
 *                    and clears what it uses on `stream` before the kernel.
 *                    The buffer must not be shared by calls that overlap on
 *                    the GPU.
 * seqlen == 0 writes h_last = h0 (or zeros) and nothing else.
 */
ss_status ss_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                      ss_dtype in_dtype, ss_dtype out_dtype,
                      const void *u, const void *delta_raw, const float *A,
                      const void *B, const void *C, const float *D, const void *z,
                      const float *delta_bias, const float *h0,
                      void *y, float *h_last,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Single-token decode step, state updated in place.
 *  h               : [batch, dim, dstate] float32, read and overwritten
 *  u, delta_raw, z : [batch, dim] in_dtype; z may be NULL
 *  B, C            : [batch, dstate] in_dtype
 *  A               : [dim, dstate] float32; D, delta_bias: [dim] float32 or NULL
 *  y               : [batch, dim] out_dtype (output)
 */
ss_status ss_state_update(int64_t batch, int64_t dim, int64_t dstate,
                          ss_dtype in_dtype, ss_dtype out_dtype,
                          float *h, const void *u, const void *delta_raw,
                          const float *A, const void *B, const void *C, const float *D,
                          const void *z, const float *delta_bias, void *y, void *stream);

/*
 * Causal depthwise convolution front-end of the Mamba block, with SiLU.
 *
 * The block passes the expanded input through a short causal convolution
 * along the sequence and a SiLU before the selective SSM ("Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces" review page, method step 3;
 * mlqm.cn tutorial section 7.1, the block diagram). The pages give no width,
 * tap order or bias; this library reads it as, for each b, d and width K:
 *
 *   e[p]       = x[b,p,d] for p >= 0; state_in[b,d,p+K-1] for -(K-1) <= p < 0
 *                (0 when state_in is NULL)
 *   pre        = bias[d] + sum_{k<K} weight[d,k] * e[t-(K-1)+k]
 *   y[b,t,d]   = silu(pre) when silu != 0, else pre
 *   state_out[b,d,k] = e[seqlen-(K-1)+k], k < K-1   (the last K-1 inputs)
 *
 *  x, y      : [batch, seqlen, dim] in_dtype / out_dtype; y must not overlap
 *              x (a tile's first K-1 rows are read from x after the tile
 *              before it may have been written), else SS_ERR_INVALID_ARG
 *  weight    : [dim, width] float32; bias: [dim] float32 or NULL
 *  state_in  : [batch, dim, width-1] in_dtype or NULL; state_out: same shape,
 *              in_dtype, or NULL; the two must be different buffers
 *  width     : 2, 3 or 4 (SS_ERR_UNSUPPORTED otherwise)
 * seqlen == 0 copies state_in (or zeros) to state_out and writes no y.
 */
ss_status ss_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width,
                        ss_dtype in_dtype, ss_dtype out_dtype,
                        const void *x, const float *weight, const float *bias,
                        const void *state_in, int silu, void *y, void *state_out, void *stream);

/*
 * One decode step of the convolution: the request's conv state (the inputs
 * the convolution still needs) is read and updated in place ("AI 推理系列（十
 * 四）：Mamba 的 Selective State Space", the decode-state table: per-layer SSM
 * state and conv state updated each token).
 *  state : [batch, dim, width-1] in_dtype, oldest input first; on return it
 *          holds the last width-1 inputs including x
 *  x     : [batch, dim] in_dtype;  y: [batch, dim] out_dtype
 *  y = silu(bias + sum_{k<K-1} weight[d,k] state[k] + weight[d,K-1] x)
 */
ss_status ss_conv1d_update(int64_t batch, int64_t dim, int64_t width,
                           ss_dtype in_dtype, ss_dtype out_dtype,
                           void *state, const void *x, const float *weight, const float *bias,
                           int silu, void *y, void *stream);

/*
 * Gradients of the selective scan (backward pass).
 *
 * The pages train the model end to end and say the backward pass recomputes
 * the scan's intermediate states instead of keeping them in HBM ("Mamba:
 * Linear-Time Sequence Modeling with Selective State Spaces" review page,
 * method step 2 (3); "AI 推理系列（十四）：Mamba 的 Selective State Space",
 * training section). They print no gradient formulas; these are the
 * derivatives of the forward defined above. Per channel (b, d), with
 * dyv_t = dy[b,t,d] * silu(z[b,t,d]) (dy itself when z is NULL),
 * yv_t the ungated output, Abar_t,n = exp(delta_t A[d,n]) and the adjoint
 * lambda_t,n = dL/dh_t,n:
 *
 *   lambda_{L-1} = C_{L-1} dyv_{L-1} + dh_last;  lambda_t = C_t dyv_t + Abar_{t+1} lambda_{t+1}
 *   du[b,t,d]          = dyv_t D[d] + delta_t sum_n lambda_t,n B[b,t,n]
 *   ddelta_raw[b,t,d]  = sigmoid(delta_raw + delta_bias[d])
 *                        * sum_n lambda_t,n (h_{t-1},n Abar_t,n A[d,n] + B[b,t,n] u[b,t,d])
 *   dz[b,t,d]          = dy yv_t silu'(z),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   dA[d,n]           = sum_{b,t} lambda_t,n h_{t-1},n Abar_t,n delta_t
 *   dB[b,t,n]         = sum_d lambda_t,n delta_t u[b,t,d]
 *   dC[b,t,n]         = sum_d dyv_t h_t,n
 *   dD[d]             = sum_{b,t} dyv_t u[b,t,d]
 *   ddelta_bias[d]    = sum_{b,t} ddelta_raw[b,t,d]
 *   dh0[b,d,n]        = Abar_0,n lambda_0,n
 *
 * Inputs are the forward's (same shapes, dtypes and NULL rules as
 * ss_scan_fwd) plus
 *  dy        : [batch, seqlen, dim] dy_dtype (SS_F32 or SS_BF16)
 *  dh_last   : [batch, dim, dstate] float32 or NULL (zero): gradient of h_last
 * Outputs (all overwritten):
 *  du, ddelta_raw : [batch, seqlen, dim] in_dtype
 *  dz             : [batch, seqlen, dim] in_dtype; required when z is given, ignored otherwise
 *  dA             : [dim, dstate] float32
 *  dB, dC         : [batch, seqlen, dstate] float32
 *  dD, ddelta_bias: [dim] float32 or NULL (not computed)
 *  dh0            : [batch, dim, dstate] float32 or NULL (not computed)
 *  workspace      : device buffer of at least ss_scan_bwd_workspace_size() bytes
 *                   (the states saved every 16 steps, then the hand-over area
 *                   of a split); must not be shared by calls that overlap on
 *                   the GPU.
 * Work split. One warp runs one block of 32 / (lanes per channel) channels
 * over the whole sequence. With more blocks than resident warps, every warp
 * takes an equal contiguous share of all blocks' 16-step sub-tiles instead:
 * where a share cuts a block, the forward state is handed on and the adjoint
 * handed back through the workspace. Those hand-overs need every warp resident
 * at once, so that launch is cooperative; where the device refuses it, the
 * call falls back to one warp per block. A hand-over that does not arrive
 * within the wait limit (ss_scan_set_wait_limit) ends the waiting warps and
 * is reported by ss_scan_status(NULL, stream) as SS_ERR_TIMEOUT; the outputs
 * are then undefined.
 * The sums over channels and time are accumulated with float32 atomic adds,
 * so dA, dB, dC, dD and ddelta_bias can differ in the last bits from run to
 * run; the other outputs are deterministic. seqlen == 0 writes dh0 = dh_last
 * (or zeros) and zero dA, dD, ddelta_bias.
 */
size_t ss_scan_bwd_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate);

ss_status ss_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                      ss_dtype in_dtype, ss_dtype dy_dtype,
                      const void *u, const void *delta_raw, const float *A,
                      const void *B, const void *C, const float *D, const void *z,
                      const float *delta_bias, const float *h0,
                      const void *dy, const float *dh_last,
                      void *du, void *ddelta_raw, void *dz, float *dA, float *dB, float *dC,
                      float *dD, float *ddelta_bias, float *dh0,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Generalised selective scan forward: larger states, B and C shared within
 * groups of channels, and a choice of the input matrix's discretisation.
 *
 *  - dstate: 16, 32, 64 or 128. The pages' tutorial lets the state size grow
 *    beyond the 16 of the language models (mlqm.cn tutorial, section 3.1).
 *  - ngroups G: B and C are [batch, seqlen, G, dstate]; channel d reads group
 *    d / (dim / G). G = 1 is the pages' one B and C shared by all channels;
 *    G = dim gives every channel its own. dim must be a multiple of G.
 *  - disc: SS_DISC_FIRST_ORDER uses Bbar = delta B, as ss_scan_fwd.
 *    SS_DISC_ZOH uses the zero-order hold, the exact discretisation of
 *    h' = A h + B x for an input held over the step: Bbar = (exp(delta A) - 1)
 *    / A * B, which is delta B where A = 0 ("外文文献精读：Mamba - 线性时间序列
 *    建模与结构化状态空间模型", section 1.2; mlqm.cn tutorial, section 3.2).
 *    Abar = exp(delta A) in both.
 *
 * Other arguments, layouts, dtypes and conventions are those of ss_scan_fwd
 * with 16 replaced by dstate (A [dim, dstate]; h0, h_last [batch, dim,
 * dstate]).
 *
 * Kernels. d_state 16 in one group with SS_DISC_FIRST_ORDER runs on the
 * ss_scan_fwd kernel. d_state 32, 64 or 128, when each group's channels are a
 * multiple of the CTA's block of 4 * 32 / (dstate / 16) channels and rows are
 * 16-byte aligned, runs on a CTA-cooperative kernel. Other shapes run one warp
 * per block of 32 / (dstate / 16) channels over the whole sequence.
 *
 * workspace (optional, device, 16-byte aligned, caller-owned, at least
 * ss_scan_fwd_general_workspace_size bytes when given): with it, and more
 * channel blocks (batch elements x blocks) than resident CTAs, the CTA kernel
 * runs one CTA per slot, each taking an equal contiguous share of all blocks'
 * 32-step tiles. Where a share starts inside a block's sequence, the state is
 * handed on through the workspace from the CTA with the share before. Its
 * first few KB are reset by the call (on `stream`), and it must not be shared
 * by calls that can run at the same time. NULL runs one CTA per block. A
 * workspace smaller than needed is SS_ERR_INVALID_ARG. A hand-over that does
 * not arrive within the wait limit (ss_scan_set_wait_limit) ends the waiting
 * CTAs and is reported by ss_scan_status(NULL, stream) as SS_ERR_TIMEOUT; the
 * outputs are then undefined.
 *
 * SS_ERR_UNSUPPORTED for another dstate or discretisation, or when the B and C
 * rows of the groups one channel block spans do not fit in shared memory.
 */
typedef enum { SS_DISC_FIRST_ORDER = 0, SS_DISC_ZOH = 1 } ss_disc;

ss_status ss_scan_fwd_general(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t ngroups,
                              ss_disc disc, ss_dtype in_dtype, ss_dtype out_dtype,
                              const void *u, const void *delta_raw, const float *A,
                              const void *B, const void *C, const float *D, const void *z,
                              const float *delta_bias, const float *h0,
                              void *y, float *h_last, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * Bytes of workspace ss_scan_fwd_general can use for this problem (0: it never
 * splits such a problem). Pure host computation: no device call, no error
 * state.
 */
size_t ss_scan_fwd_general_workspace_size(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                                          int64_t ngroups, ss_disc disc, ss_dtype in_dtype);

/*
 * State-space-dual (Mamba-2) layer forward on the tensor cores.
 *
 * The pages say Mamba-2 shows the selective scan to be dual to a structured
 * (semiseparable) matrix multiplication and re-blocks the state computation so
 * that more of it runs as matrix products ("AI 推理系列（十四）：Mamba 的
 * Selective State Space", section on Mamba-2; mlqm.cn tutorial, section 8).
 * They print no formulas; this library reads the layer as the selective scan
 * with one scalar decay per head, which is what makes the matrix shared by a
 * head's channels. Per batch element b and head h, with delta_t =
 * softplus(dt[b,t,h] + dt_bias[h]) and g = h / (nheads / ngroups):
 *
 *   H[p,n]  = exp(delta_t A[h]) H[p,n] + delta_t x[b,t,h,p] B[b,t,g,n]
 *   y[b,t,h,p] = sum_n H[p,n] C[b,t,g,n] + D[h] x[b,t,h,p]
 *
 * from H = h0[b,h] (zeros when NULL); h_last[b,h] = H after the last step.
 * Equivalently y = M x per (b, h) with M[t,s] = (C_t . B_s) delta_s
 * exp(A[h] sum_{s<k<=t} delta_k) for s <= t.
 *
 *  x            : [batch, seqlen, nheads, headdim] bf16 (in_dtype must be SS_BF16)
 *  dt           : [batch, seqlen, nheads] bf16
 *  A            : [nheads] float32 (negative)
 *  B, C         : [batch, seqlen, ngroups, dstate] bf16
 *  D, dt_bias   : [nheads] float32 or NULL
 *  h0, h_last   : [batch, nheads, headdim, dstate] float32 or NULL
 *  y            : [batch, seqlen, nheads, headdim] out_dtype
 * headdim must be 64 and dstate 64 or 128 (SS_ERR_UNSUPPORTED otherwise);
 * nheads must be a multiple of ngroups. Computed in chunks of 128 steps on the
 * tcgen05 tensor cores, products accumulated in float32 in tensor memory
 * (dstate 64 runs as 128 with B and C zero-padded); the operands computed on
 * chip (the masked C.B^T, the weighted x, the carried state) enter the
 * products as two bf16 parts (about 16 significant bits).
 *
 * workspace (optional, device, 16-byte aligned, caller-owned, at least
 * ss_ssd_fwd_workspace_size bytes when given): with it and more (batch, head)
 * sequences than SMs, a call runs one CTA per SM, each taking an equal
 * contiguous share of all the sequences' chunks; where a share starts inside a
 * sequence, the state is handed on through the workspace from the CTA with
 * the share before. Its first few KB are reset by the call (on `stream`) and
 * it must not be shared by calls that can run at the same time. NULL runs one
 * CTA per sequence. A workspace smaller than needed is SS_ERR_INVALID_ARG. A
 * hand-over that does not arrive within the wait limit (see
 * ss_scan_set_wait_limit) ends the waiting CTAs and is reported by
 * ss_scan_status(NULL, stream) as SS_ERR_TIMEOUT; the outputs are then
 * undefined.
 */
ss_status ss_ssd_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                     int64_t ngroups, ss_dtype in_dtype, ss_dtype out_dtype,
                     const void *x, const void *dt, const float *A, const void *B, const void *C,
                     const float *D, const float *dt_bias, const float *h0,
                     void *y, float *h_last, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace ss_ssd_fwd can use for this problem (0: it never splits
 * such a problem). Pure host computation: no device call, no error state.
 */
size_t ss_ssd_fwd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate);

/*
 * Launch-shape controls for the calling host thread (0 = automatic, the
 * default, for each). threads_per_channel in {1, 2} sets how many threads share
 * one channel's 16 states (a CTA then covers 128 or 64 channels). chunk_len > 0
 * forces the sequence to be split into chunks of that many timesteps (rounded
 * up to the tile: 64 steps for bf16 inputs, 32 for float32), which engages the
 * cross-CTA carry path. max_workers > 0 caps the number of CTAs a split of the
 * work uses (default: one per SM), which makes range boundaries and hand-overs
 * more frequent. Results do not depend on these settings beyond fp32 rounding;
 * ss_scan_fwd_workspace_size() follows them. For ss_ssd_fwd, ss_scan_fwd_general
 * (with a workspace) and ss_scan_bwd, chunk_len > 0 sets the length of the
 * shares (rounded up to 128 steps for ss_ssd_fwd, 32 for the generalised
 * scan's CTA kernel, 16 for the backward) instead of the automatic plan, so
 * that shares start inside sequences even on small problems; threads_per_channel
 * also sets the backward's lanes per channel.
 */
void ss_scan_set_tuning(int threads_per_channel, int64_t chunk_len, int max_workers);

/*
 * Fault-path controls of ss_scan_fwd for the calling host thread (no
 * counterpart on the pages; they exist to test the bounded device-side waits).
 * wait_ns is the limit of every device-side wait of later scans (0 restores
 * the default of 2 s). withhold_item >= 0 makes the scan never publish one
 * cross-CTA flag: the hand-over into stream-K worker `withhold_item`, or the
 * carry of chunk item `withhold_item` (block * nchunks + chunk) in the chunked
 * split; -1 (the default) publishes all. A withheld flag makes the CTAs that
 * need it give up after wait_ns, set the fault word and return, so the call
 * finishes and ss_scan_status() reports SS_ERR_TIMEOUT; its outputs are then
 * undefined. No wait in the library is unbounded. They apply to ss_ssd_fwd,
 * ss_scan_fwd_general and ss_scan_bwd too: there withhold_item is the share
 * (the shares in sequence order, numbered from 0) that hands nothing on.
 */
void ss_scan_set_wait_limit(uint64_t wait_ns, int64_t withhold_item);

/*
 * Selective scan forward that allocates nothing (no counterpart on the pages:
 * it is a deployment variant of ss_scan_fwd, not part of the method).
 *
 * For callers that cannot allocate device memory: code running inside another
 * runtime's memory pool or a graph-building framework that hands a plugin only
 * its input and output buffers, or a serving loop that must not call
 * cudaMalloc (which can synchronise the device) once it is running. Such a
 * caller cannot provide the workspace that long sequences need. This entry
 * point takes that scratch from a fixed array the library declares in device
 * memory: SS_SCAN_NOALLOC_SCRATCH_BYTES on every GPU that loads the library,
 * held until the process exits. It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * Arguments, layouts and results are those of ss_scan_fwd, without the
 * workspace arguments. Behaviour:
 *  - A problem whose scratch need (ss_scan_fwd_workspace_size) exceeds
 *    SS_SCAN_NOALLOC_SCRATCH_BYTES is rejected with SS_ERR_INVALID_ARG before
 *    anything is launched; use ss_scan_fwd with a workspace for it.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and keeps it; make that first call before any CUDA
 *    stream capture begins. The address belongs to the device's primary
 *    context (the one the CUDA runtime uses): calls must come from that
 *    context, and none may follow a cudaDeviceReset() of the device in the
 *    same process (the kept address would then be stale).
 *  - Argument errors (sizes, dtypes, NULL or misaligned pointers) are reported
 *    before any device call, as by ss_scan_fwd.
 *  - All calls on a device share the one array. Each call clears, on its
 *    stream, the part that must start at zero. Calls that overlap on the GPU
 *    (different streams, or different host threads without ordering) race on
 *    the array and give wrong results: serialise them.
 *  - A device-side wait that gives up is recorded in the library's own fault
 *    word: ss_scan_status(NULL, stream) reports it.
 */
#define SS_SCAN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

ss_status ss_scan_fwd_noalloc(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                              ss_dtype in_dtype, ss_dtype out_dtype,
                              const void *u, const void *delta_raw, const float *A,
                              const void *B, const void *C, const float *D, const void *z,
                              const float *delta_bias, const float *h0,
                              void *y, float *h_last, void *stream);

/*
 * Synchronises `stream`, then reports whether a device-side bounded wait of an
 * earlier ss_scan_fwd call on it gave up (SS_ERR_TIMEOUT) and clears that
 * record. `workspace` is the buffer that call was given (NULL if none).
 * Returns SS_ERR_CUDA if the stream reports an error.
 */
ss_status ss_scan_status(void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SS_SCAN_H */
