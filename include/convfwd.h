/*
 * convfwd.h -- C ABI of the GB300 (sm_103a) forward-convolution library.
 *
 * The operations follow three POPCORNBENCH reasoning-trace pages:
 *   - "Kimi-K2.6 l1_p60": nn.Conv3d with an asymmetric (3,5,7) kernel,
 *     turn 1 (the forward sum, the per-dimension output size, zero padding).
 *   - "Kimi-K2.6 l1_p76": nn.Conv1d with stride 3 and dilation 4, turns 1-2
 *     (tap positions j*stride + k*dilation, output length 174758).
 *   - "Kimi-K2.6 l2_p24": Conv3d -> torch.min(dim=2) -> torch.softmax(dim=1),
 *     turns 1-2 (min over output depth, then a max-subtracted channel softmax).
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, contiguous, row-major fp32 (PyTorch's default NC[D][H]W).
 *   - Pointers named x, w, bias, y are DEVICE pointers.  Dimension/hyper-
 *     parameter arrays (in_dims, k_dims, stride, pad, dilation, out_dims) and
 *     the descriptor structs are HOST memory, read during the call only.
 *   - The caller owns every buffer and the library keeps no pointer to one after
 *     the call returns.  y must not overlap x, w or bias.  Some calls take one
 *     stream-ordered block of device memory: conv_fwd_nd, conv_fwd_nd_ex,
 *     conv_fwd_nd_grouped, conv_fwd_nd_channels_last, conv_fwd_nd_bf16,
 *     conv_fwd_nd_f16 and conv_fwd_nd_host for a tensor-core layer whose
 *     weights exceed shared memory
 *     (conv_workspace_bytes > 0: the split weights), and
 *     conv3d_min_softmax(_ex) in the same case on its
 *     tensor-core kernel, or for a min over width on its FFMA kernels
 *     (transposed copies of x and w).  The block comes from a memory pool of
 *     the library's (from the device's default pool while `stream` is being
 *     captured into a graph), is allocated and freed on `stream`; if it
 *     cannot be had, the call runs without it where it can (reduction passes,
 *     the generic fused kernel) and returns CONV_ERR_CUDA otherwise.  conv_fwd_nd_ws, conv_fwd_nd_ws_noalloc and every other
 *     call allocate nothing.  Things held by the library itself: a 16 MiB
 *     file-scope device array (the scratch of conv_fwd_nd_ws_noalloc), which
 *     every device that loads the library holds until the process exits; from
 *     the first allocating call on a device, that memory pool, which keeps up
 *     to 64 MiB reserved between calls; and, from the first conv_fwd_nd_host
 *     call on a device, two copy streams and six events on that device, kept
 *     until exit.
 *   - All device work is enqueued on `stream` (NULL = legacy default stream);
 *     calls return without synchronising.  Errors from kernels that already
 *     ran surface at the caller's next synchronisation (cudaStreamSynchronize).
 *   - Every argument is validated on the host before anything is launched; a
 *     non-zero status means nothing was written to y.  conv_last_error()
 *     returns a human-readable reason for the most recent failure on the
 *     calling thread.
 *   - Kernels never trap or assert.  Waits inside kernels are bounded; if one
 *     gives up, the kernel records it in a device-side status word that
 *     conv_device_status() reads.
 *   - With CONVFWD_LOG=1 in the environment (read once per process), every
 *     call that launches kernels writes one line to stderr: the entry point,
 *     the problem, the kernel family and, for the tensor-core family, the plan
 *     (tiles, reduction length and padding, column order, slots, passes,
 *     channel blocks, resident or streamed weights, shared memory).
 *   - With CONVFWD_FORCE_ALGO=direct_ffma or =igemm_3xtf32 in the environment
 *     (read once per process), fp32 calls made with CONV_ALGO_AUTO -- the
 *     plain and grouped convolutions, conv3d_min_softmax and the two
 *     select_algo queries -- take that kernel family wherever it can run the
 *     problem, and the
 *     planner's choice elsewhere.  Other values are ignored (one line on
 *     stderr).  An explicit algo argument always wins.
 */
#ifndef CONVFWD_H
#define CONVFWD_H

#include <stdint.h>

#if defined(__GNUC__)
#define CONVFWD_API __attribute__((visibility("default")))
#else
#define CONVFWD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t / the driver's CUstream. */
struct CUstream_st;
typedef struct CUstream_st *conv_stream_t;

typedef enum {
  CONV_OK = 0,
  CONV_ERR_NULL = 1,        /* a required pointer is NULL */
  CONV_ERR_ARG = 2,         /* a size/hyper-parameter is out of range, or a pointer is misaligned */
  CONV_ERR_SHAPE = 3,       /* an output size is <= 0, or descriptor shapes disagree */
  CONV_ERR_UNSUPPORTED = 4, /* valid request that this library does not implement */
  CONV_ERR_CUDA = 5,        /* a CUDA runtime call failed (see conv_last_error) */
  CONV_ERR_INTERNAL = 6     /* debug build only: a launch plan failed one of its assertions (a library bug) */
} conv_status_t;

/* Kernel families.  AUTO lets the planner choose. */
typedef enum {
  CONV_ALGO_AUTO = 0,
  CONV_ALGO_DIRECT_FFMA = 1,  /* FP32 FFMA direct convolution (CUDA cores) */
  CONV_ALGO_IGEMM_3XTF32 = 2  /* implicit GEMM on tcgen05 tensor cores, 3xTF32 split, fp32 accumulation in TMEM */
} conv_algo_t;

/* Shape descriptors for the fused entry point (host structs, device data). */
typedef struct {
  const float *data; /* device pointer */
  int64_t dims[5];   /* x: [N, C_in, D, H, W];  w: [C_out, C_in, KD, KH, KW] */
} conv_tensor5_t;

typedef struct {
  float *data;     /* device pointer */
  int64_t dims[4]; /* y: [N, C_out, H_out, W_out] */
} conv_tensor4_t;

/*
 * Output size per spatial dimension (l1_p60 page turn 1 host code; l1_p76 page
 * turns 1-2):   out[i] = floor((in[i] + 2*pad[i] - dilation[i]*(k[i]-1) - 1) / stride[i]) + 1
 * ndim in {1,2,3}; in, k, stride, dilation >= 1; pad >= 0.  Writes out_dims
 * (host, ndim entries) and returns CONV_OK, or CONV_ERR_SHAPE when some size is
 * <= 0 (out_dims still written), CONV_ERR_ARG / CONV_ERR_NULL otherwise.
 */
CONVFWD_API int conv_out_dims(int ndim, const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                  const int64_t *pad, const int64_t *dilation, int64_t *out_dims);

/*
 * Forward N-D convolution, ndim in {1,2,3} (l1_p60 page turn 1; l1_p76 page turns 1-2):
 *   y[n,o,p] = bias[o] + sum_{c<C_in} sum_{k} w[o,c,k] * x[n,c, p*stride + k*dilation - pad]
 * with taps outside the input reading zero (symmetric zero padding, groups = 1).
 *   x    [N, C_in, in_dims...]          device, fp32
 *   w    [C_out, C_in, k_dims...]       device, fp32
 *   bias [C_out] or NULL (no bias)      device, fp32
 *   y    [N, C_out, out_dims...]        device, fp32, out_dims as conv_out_dims
 *   in_dims, k_dims, stride, pad, dilation: host arrays of ndim int64
 * N = 0 is a valid empty batch (nothing is launched).
 * Accuracy: |y - exact| <= 1e-4 * (1 + |exact|) elementwise for inputs of the
 * magnitudes used in the tests (accumulation in fp32; the tensor-core path
 * splits each operand into two TF32 halves and sums three products).
 * Returns CONV_OK or an error status; nothing is launched on error.
 */
CONVFWD_API int conv_fwd_nd(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                int64_t C_in, int64_t C_out, const int64_t *in_dims, const int64_t *k_dims,
                const int64_t *stride, const int64_t *pad, const int64_t *dilation, conv_stream_t stream);

/* conv_fwd_nd with an explicit kernel family (conv_algo_t).  CONV_ALGO_AUTO is
 * what conv_fwd_nd uses.  Returns CONV_ERR_UNSUPPORTED when the requested
 * family cannot run this shape (e.g. the tensor-core path's weight tile does
 * not fit in shared memory). */
CONVFWD_API int conv_fwd_nd_ex(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                   int64_t C_in, int64_t C_out, const int64_t *in_dims, const int64_t *k_dims,
                   const int64_t *stride, const int64_t *pad, const int64_t *dilation, int algo,
                   conv_stream_t stream);

/*
 * Grouped convolution (the pages' modules take a groups argument, left at 1
 * there): C_in and C_out split into `groups` equal groups; output channel
 * o = grp*(C_out/groups) + j sums over input channels grp*(C_in/groups) ...
 * (grp+1)*(C_in/groups) - 1 only:
 *   y[n,o,p] = bias[o] + sum_{c<C_in/groups} sum_k w[o,c,k] * x[n, grp*C_in/groups + c, p*stride + k*dilation - pad]
 *   w [C_out, C_in/groups, k_dims...]   device, fp32; x, bias, y as for conv_fwd_nd.
 * groups = 1 is conv_fwd_nd_ex.  groups must be >= 1 and divide C_in and C_out
 * (CONV_ERR_ARG otherwise).  `algo` as for conv_fwd_nd_ex; the planner judges
 * one group's problem (C_in/groups input and C_out/groups output channels).
 * The direct family runs all groups in one launch; the tensor-core family
 * launches once per group on the stream.
 */
CONVFWD_API int conv_fwd_nd_grouped(const float *x, const float *w, const float *bias, float *y, int ndim,
                                    int64_t N, int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                                    const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                    const int64_t *dilation, int algo, conv_stream_t stream);

/*
 * Channels-last layout: the same convolution (groups included) on tensors
 * stored N (D) (H) W C, i.e. PyTorch's channels_last / channels_last_3d memory
 * format; dims are still passed in the logical N, C, spatial order.
 *   x [N, in_dims..., C_in]   w [C_out, k_dims..., C_in/groups]   y [N, out_dims..., C_out]
 *   bias [C_out] or NULL.  Everything else as conv_fwd_nd_grouped.
 * The reduction runs tap by tap with the channels innermost, so with
 * C_in/groups % 8 == 0 and 32-byte aligned x each gather is one 32-byte load
 * of 8 channels (with % 4 and 16-byte alignment, one 16-byte load of 4;
 * otherwise one load per value), and each output position's channels are
 * written as one contiguous run.  Only the tensor-core family runs this layout: algo must be
 * CONV_ALGO_AUTO or CONV_ALGO_IGEMM_3XTF32; CONV_ALGO_DIRECT_FFMA and shapes
 * the tensor-core path does not take return CONV_ERR_UNSUPPORTED.  The weights
 * always stream through the kernel from a stream-ordered block of the call
 * (released on `stream`), which leaves the shared memory they would occupy to
 * the L1 that the gather re-reads; if that block cannot be had, they are held
 * in shared memory as in the other calls.
 */
CONVFWD_API int conv_fwd_nd_channels_last(const float *x, const float *w, const float *bias, float *y, int ndim,
                                          int64_t N, int64_t C_in, int64_t C_out, int64_t groups,
                                          const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                                          const int64_t *pad, const int64_t *dilation, int algo,
                                          conv_stream_t stream);

/*
 * BFloat16 tensors (the pages discuss BF16 tensor cores and keep fp32 for the
 * 1e-4 tolerance; this is the lower-precision option):
 *   x, w, bias, y hold bfloat16 bit patterns (uint16_t), same shapes and
 *   layout as conv_fwd_nd_grouped (contiguous N C spatial).
 * The products and their sum are formed in fp32 on the tensor cores (one
 * kind::f16 MMA per 16 reduction columns, no operand split); the bias is
 * added in fp32 and y is rounded once to bfloat16 (nearest even).  Hence
 * |y - exact| <= 2^-9 |exact| + (fp32 accumulation error) for every element.
 * Runs on the tensor-core family only: wider layers than 128 output channels
 * per group in channel blocks of 128, weights that exceed shared memory
 * streamed chunk by chunk from a stream-ordered block; kernel extents above 32
 * are CONV_ERR_UNSUPPORTED.  All pointers 2-byte aligned.
 */
CONVFWD_API int conv_fwd_nd_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, int ndim,
                                 int64_t N, int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                                 const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                 const int64_t *dilation, conv_stream_t stream);

/* The same for IEEE float16 tensors (x, w, bias, y hold float16 bit
 * patterns): one rounding of the fp32 sum to float16 at the store, so
 * |y - exact| <= 2^-11 |exact| + (fp32 accumulation error) while the result
 * stays inside the float16 range. */
CONVFWD_API int conv_fwd_nd_f16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, int ndim,
                                int64_t N, int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                                const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                const int64_t *dilation, conv_stream_t stream);

/*
 * Workspace for streamed weights.  The tensor-core family keeps one group's
 * weights (split into TF32 hi and lo) in shared memory; when they do not fit,
 * the weights are split once into a workspace, in the order the tensor cores
 * read them, and brought into shared memory chunk by chunk with bulk copies,
 * so the whole reduction runs in one pass.  The workspace is the caller's
 * (conv_fwd_nd_ws) or a stream-ordered allocation of the call (conv_fwd_nd and
 * the other allocating calls); without one the reduction runs in several
 * passes, each re-reading x and adding into y.
 * conv_workspace_bytes writes the bytes conv_fwd_nd_ws can use for the problem
 * (0 when its weights fit in shared memory, or a group has more than 128
 * output channels, or the column tables of the reduction exceed shared memory).
 */
CONVFWD_API int conv_workspace_bytes(int ndim, int64_t N, int64_t C_in, int64_t C_out, int64_t groups,
                                     const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                                     const int64_t *pad, const int64_t *dilation, size_t *bytes);

/* conv_fwd_nd_grouped (AUTO) with a device workspace of at least
 * conv_workspace_bytes bytes, 256-byte aligned, not overlapping x, w, bias or
 * y; the library writes it before reading it on `stream`, so calls that share
 * a workspace must be ordered (the same stream does that).  With a problem that
 * needs none it is conv_fwd_nd_grouped; with workspace NULL it is
 * conv_fwd_nd_grouped without its allocation (a layer whose weights exceed
 * shared memory then runs in several passes); a workspace smaller than needed
 * is CONV_ERR_ARG. */
CONVFWD_API int conv_fwd_nd_ws(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                               int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                               const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                               const int64_t *dilation, void *workspace, size_t workspace_bytes,
                               conv_stream_t stream);

/*
 * conv_fwd_nd_ws without a caller workspace and without allocating: the
 * streamed weights go to a 16 MiB scratch array that the library holds in
 * device memory from load time (a file-scope device array; its address is
 * looked up once per device).  The paper has no counterpart of this entry
 * point; it exists for callers that cannot allocate device memory.
 * Problems that need more scratch than the array holds return
 * CONV_ERR_UNSUPPORTED; problems that need none are conv_fwd_nd_grouped.  The
 * scratch is shared by every call on the device, so calls that use it must be
 * ordered (issue them on one stream).
 */
CONVFWD_API int conv_fwd_nd_ws_noalloc(const float *x, const float *w, const float *bias, float *y, int ndim,
                                       int64_t N, int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                                       const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                       const int64_t *dilation, conv_stream_t stream);

/*
 * Host buffers in, host buffer out.  x, w, bias and y are HOST pointers with the
 * layouts of conv_fwd_nd_grouped.  The call copies w and bias to the device,
 * then runs the batch through the device in chunks of `chunk` images (chunk <= 0
 * or > N: one chunk).  The host-to-device copy of chunk i+1 and the
 * device-to-host copy of chunk i-1 run on two library streams while chunk i is
 * convolved on `stream` (conv_fwd_nd_grouped, AUTO), so the copies overlap the
 * compute.  The forward convolution itself is the one of the pages' modules
 * (l1_p60 and l1_p76 pages); the chunked host interface has no counterpart
 * there.
 *
 * workspace: device memory of at least conv_host_workspace_bytes bytes (for the
 * same arguments and chunk), 256-byte aligned; it holds w, bias and two chunks
 * each of x and y.  The copies overlap only when x and y are page-locked
 * (cudaHostAlloc, cudaHostRegister or a pinned torch tensor); pageable memory
 * works but serialises.  All work is enqueued and the call returns without
 * synchronising: y is complete once `stream` has completed (the stream waits
 * for the last device-to-host copy).  The library's two copy streams and their
 * events are created on the first call on each device and kept; calls that
 * share a workspace must be ordered on one stream.  Calls from several host
 * threads are safe: each call enqueues its work under a per-device lock.
 *
 * Errors: CONV_ERR_NULL (x, w or y NULL with N > 0, workspace NULL),
 * CONV_ERR_ARG (bad sizes, a workspace too small or misaligned, y overlapping
 * an input), the statuses of conv_fwd_nd_grouped for the chunks, CONV_ERR_CUDA
 * for a failed copy, event or stream call.  Argument errors are found before
 * anything is enqueued; a CUDA error on a later chunk can leave the chunks
 * before it already copied into y.
 */
CONVFWD_API int conv_host_workspace_bytes(int ndim, int64_t N, int64_t C_in, int64_t C_out, int64_t groups,
                                          const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                                          const int64_t *pad, const int64_t *dilation, int64_t chunk,
                                          size_t *bytes);
CONVFWD_API int conv_fwd_nd_host(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                                 int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                                 const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                 const int64_t *dilation, int64_t chunk, void *workspace, size_t workspace_bytes,
                                 conv_stream_t stream);

/* The kernel family conv_fwd_nd would use for this problem (host only, no
 * device access).  Writes *algo_out and returns CONV_OK, or an error status
 * for an invalid problem.  (A call that cannot stream weights, conv_fwd_nd_ws
 * without a workspace, may take the direct family instead for a layer whose
 * weights exceed shared memory.) */
CONVFWD_API int conv_select_algo(int ndim, int64_t N, int64_t C_in, int64_t C_out, const int64_t *in_dims,
                     const int64_t *k_dims, const int64_t *stride, const int64_t *pad, const int64_t *dilation,
                     int *algo_out);

/* CONV_OK when kernel family `algo` can run this problem, CONV_ERR_UNSUPPORTED
 * when it cannot (reason in conv_last_error), or the validation status of an
 * invalid problem.  Host only, no device access. */
CONVFWD_API int conv_algo_supported(int ndim, int64_t N, int64_t C_in, int64_t C_out, const int64_t *in_dims,
                                    const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                                    const int64_t *dilation, int algo);

/*
 * Fused Conv3d -> min over one spatial dim of the conv output -> softmax over
 * channels (l2_p24 page, turns 1-2):
 *   z[n,o,d,h,w] = bias[o] + sum_{c,kd,kh,kw} w[o,c,kd,kh,kw] * x[n,c,d+kd,h+kh,w+kw]
 *   m[n,o,h,w]   = min_d z[n,o,d,h,w]                     (min_dim = 2, depth; the page's case)
 *   y[n,o,h,w]   = exp(m - max_o m) / sum_o exp(m - max_o m)
 * The page's module takes the min dimension as a constructor argument; min_dim
 * 3 reduces over height (m[n,o,d,w] = min_h z) and 4 over width (m[n,o,d,h]).
 * Conv hyper-parameters are fixed to stride 1, padding 0, dilation 1, groups 1.
 * The 5-D intermediate z is never written to memory.
 *   x->dims = [N, C_in, D, H, W], w->dims = [C_out, C_in, KD, KH, KW],
 *   bias: [C_out] device or NULL, y->dims = [N, C_out] followed by the conv's
 *   spatial output dims (D-KD+1, H-KH+1, W-KW+1) without the reduced one:
 *   [N, C_out, OH, OW] for min_dim 2, [N, C_out, OD, OW] for 3, [N, C_out, OD, OH] for 4.
 * min_dim outside {2, 3, 4}: CONV_ERR_ARG.  Two kernel families: the FFMA
 * kernels (C_out up to 96, a kernel extent along y's last axis up to 7) and a
 * tensor-core kernel (any C_out, kernel extents up to 32; a 3xTF32 implicit
 * GEMM whose epilogue keeps each position's running minimum over the reduced
 * dim in registers, 32 channels per launch: wider layers run block by block,
 * then one channel-softmax pass over y; when one input plane's receptive-field
 * columns along the other two axes number at most 32, each plane is gathered
 * once and shared by the tiles that read it; weights that exceed shared
 * memory stream through a stream-ordered block of the call, as for
 * conv_fwd_nd).  The min over width runs, in both
 * families where they can, as the min over height of x and w transposed in
 * their last two dims (a stream-ordered block).  Where both families run, the
 * planner takes the tensor-core kernel, measured faster on every shape class
 * tried (conv3d_min_softmax_select_algo reports the choice).  Shapes neither
 * family runs are CONV_ERR_UNSUPPORTED.
 */
CONVFWD_API int conv3d_min_softmax(const conv_tensor5_t *x, const conv_tensor5_t *w, const float *bias, conv_tensor4_t *y,
                       int min_dim, conv_stream_t stream);

/* conv3d_min_softmax with an explicit kernel family: CONV_ALGO_AUTO (the
 * planner), CONV_ALGO_DIRECT_FFMA (the FFMA kernels) or CONV_ALGO_IGEMM_3XTF32
 * (the tensor-core kernel); a family that cannot run the shape returns
 * CONV_ERR_UNSUPPORTED, an unknown value CONV_ERR_ARG. */
CONVFWD_API int conv3d_min_softmax_ex(const conv_tensor5_t *x, const conv_tensor5_t *w, const float *bias,
                                      conv_tensor4_t *y, int min_dim, int algo, conv_stream_t stream);

/* The kernel family conv3d_min_softmax would take for these shapes (only
 * x->dims and w->dims are read; host only, no device access): writes
 * CONV_ALGO_DIRECT_FFMA or CONV_ALGO_IGEMM_3XTF32 to *algo_out and returns
 * CONV_OK; CONV_ERR_UNSUPPORTED when neither family runs the shape; the
 * validation statuses of conv3d_min_softmax otherwise. */
CONVFWD_API int conv3d_min_softmax_select_algo(const conv_tensor5_t *x, const conv_tensor5_t *w, int min_dim,
                                               int *algo_out);

/*
 * Peak-rate microbenchmarks (diagnostics; not part of the convolution).  The
 * pages reason about their kernels against the FP32 and tensor-core peaks of
 * the GPU they name (l1_p60 page turn 1; l1_p76 page turn 2); these measure
 * the corresponding peaks of the GPU at hand, at the clock it runs, so that
 * roofline fractions rest on measured denominators.
 *
 * conv_peak_mma: one persistent CTA per SM; `issuers` (1-4) warps each issue
 * `iters` (1-262144) back-to-back tcgen05.mma of shape M = 128 x N = n
 * (16-256, a multiple of 16) x one K step, from one elected thread, on
 * operands resident on chip: kind 0 = kind::tf32 (K = 8), kind 1 = kind::f16
 * with BF16 operands (K = 16); A from tensor memory (a_in_tmem != 0) or shared
 * memory, B from shared memory; fp32 accumulation in tensor memory.
 * conv_peak_ffma: every resident thread runs 16 independent fp32 multiply-add
 * chains, scalar fma.rn.f32 (packed == 0) or fma.rn.f32x2 on pairs (packed != 0),
 * `iters` (1-1048576) rounds of 64 multiply-adds each.
 * Both launch the kernel once untimed and once timed, synchronise `stream`
 * before returning, and fill *out.  They allocate no device memory (their
 * per-CTA stamps live in file-scope device arrays, so concurrent calls on one
 * device race).  Errors: CONV_ERR_NULL, CONV_ERR_ARG for out-of-range
 * arguments, CONV_ERR_CUDA (also when a bounded wait inside the MMA kernel gave up).
 */
typedef struct {
  double flops;         /* operations of the timed launch (2 per multiply-add) */
  double seconds;       /* earliest CTA start to latest CTA end, device global timer */
  double event_ms;      /* the timed launch by CUDA events on `stream` */
  double sm_mhz;        /* median over CTAs of SM clock cycles / global-timer ns during each CTA's run */
  double cycles_per_op; /* MMA: SM cycles per MMA instruction on one SM; FFMA: SM cycles per warp-wide FMA
                           instruction on one SM */
  int ctas;             /* CTAs launched */
} conv_peak_result_t;

CONVFWD_API int conv_peak_mma(int kind, int n, int issuers, int a_in_tmem, int iters, conv_peak_result_t *out,
                              conv_stream_t stream);
CONVFWD_API int conv_peak_ffma(int packed, int iters, conv_peak_result_t *out, conv_stream_t stream);

/* Static description of a status code. */
CONVFWD_API const char *conv_status_string(int status);

/* Reason for the most recent non-OK return on the calling thread ("" if none). */
CONVFWD_API const char *conv_last_error(void);

/*
 * Test hook for the bounded waits (the paper has no counterpart): sets, for
 * every tensor-core launch made after the call in this process, the number
 * of SM clock cycles after which a pipeline wait inside the kernel gives up
 * (cycles <= 0 restores the default, about two seconds; 1-63 is CONV_ERR_ARG).
 * A kernel whose wait gives up stops its work, lets every role fall through,
 * waits for its own MMAs and copies with the full default limit, frees its
 * tensor memory, sets bit 0 of the device status word and returns: its output
 * is incomplete, and conv_device_status() reports it.  A limit of a few
 * hundred cycles makes the waits run out on purpose, so that tests can check
 * that this path leaves the device usable.  Process-wide; set it only while
 * no other thread launches convolutions.
 */
CONVFWD_API int conv_debug_set_wait_limit(long long cycles);

/* Synchronises the current device, then returns and clears the device-side
 * status word: 0 when no kernel gave up on a bounded wait since the last call,
 * else bit 0 (a tensor-core kernel gave up) plus, per CTA that gave up, the
 * wait that ran out first: bit 8 producers waiting for an A stage to drain,
 * bit 9 the MMA issuer waiting for an A stage to fill, bit 10 the issuer
 * waiting for streamed weights, bit 11 the epilogue waiting for an
 * accumulator, bit 12 the issuer waiting for an accumulator to drain.  In a
 * debug build (below) also the bounds checks since the last call: bit 1 an
 * index outside x, bit 2 outside w or bias, bit 3 outside y, bit 4 outside a
 * workspace, bit 5 outside a kernel's shared-memory staging buffer.  Writes
 * the word to *flags and returns CONV_OK, or CONV_ERR_CUDA. */
CONVFWD_API int conv_device_status(unsigned int *flags);

/*
 * Debug build (the library compiled with -DCONVFWD_DEBUG, libconvfwd_debug.so
 * beside libconvfwd.so; the Python binding loads it when CONVFWD_DEBUG=1 is in
 * the environment).  The stand-in for a memory checker: same entry points,
 * same results on correct inputs, slower.
 *   - Host: every launcher asserts its plan before launching (shared memory
 *     and tensor-memory budgets, chunk and stage sizes, alignment of the
 *     addresses bulk copies and 16-byte accesses use, the tiles covering the
 *     output); a failed assertion returns CONV_ERR_INTERNAL with the
 *     condition in conv_last_error(), and nothing is launched.
 *   - Device: every global index a kernel forms for x, w, bias, y or a
 *     workspace (and the shared-memory index of the staged copies) is tested
 *     against the extent of that tensor as the launch sees it.  An index
 *     outside it sets a bit of the status word (above), the first such index
 *     is kept, and the access is skipped (a load yields 0, a store or copy is
 *     dropped): no kernel traps, and nothing outside a tensor is touched.
 */
#define CONV_BUILD_DEBUG 1
/* CONV_BUILD_DEBUG when this library is the debug build, else 0. */
CONVFWD_API int conv_build_flags(void);
/* Debug build: the element index that the most recent conv_device_status()
 * call found first out of range (-1: none).  CONV_ERR_UNSUPPORTED (and -1) in
 * the release build; CONV_ERR_NULL when index is NULL. */
CONVFWD_API int conv_debug_first_bad_index(long long *index);
/* Debug-build test hook (the paper has no counterpart): the extent of x that
 * the device checks allow is reduced by `elems` elements for launches made
 * after the call (0 restores it), so that reads of the last elements of x --
 * which exist -- register as out of range and are skipped.  A test of the
 * checks that never touches memory outside a tensor.  Process-wide; set it
 * only while no other thread launches convolutions.  CONV_ERR_ARG for elems <
 * 0; CONV_ERR_UNSUPPORTED in the release build. */
CONVFWD_API int conv_debug_shrink_bounds(long long elems);

#ifdef __cplusplus
}
#endif

#endif /* CONVFWD_H */
