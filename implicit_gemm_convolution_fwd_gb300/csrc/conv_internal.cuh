// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace convfwd {

// A convolution problem in a uniform 3-D view: 1-D and 2-D problems are
// embedded with leading singleton dims (size 1, kernel 1, stride 1, pad 0,
// dilation 1), which leaves the sum in the l1_p60 / l1_p76 pages unchanged.
// With G > 1 groups, C and K count the channels of one group: x has G*C
// channels, y and w have G*K, and output channel grp*K + o reads input
// channels [grp*C, grp*C + C).
struct Geom {
  int64_t N, C, K;             // batch, input channels per group, output channels per group
  int64_t G;                   // groups (1: a plain convolution)
  int cl;                      // memory layout: 0 = N C D H W (PyTorch default), 1 = N D H W C (channels last)
  int D, H, W;                 // input spatial dims
  int OD, OH, OW;              // output spatial dims
  int KD, KH, KW;              // kernel dims
  int SD, SH, SW;              // stride
  int PD, PH, PW;              // zero padding (symmetric)
  int DD, DH, DW;              // dilation
  __host__ __device__ int64_t x_batch_stride() const { return G * C * (int64_t)D * H * W; }  // elements between images of x
  __host__ __device__ int64_t y_batch_stride() const { return G * K * (int64_t)OD * OH * OW; }
  __host__ __device__ int64_t in_spatial() const { return (int64_t)D * H * W; }
  __host__ __device__ int64_t out_spatial() const { return (int64_t)OD * OH * OW; }
  __host__ __device__ int taps() const { return KD * KH * KW; }
};

// Device-side status word written by kernels whose bounded waits gave up.
enum : unsigned {
  kStatusIgemmWatchdog = 1u,
  // beside bit 0, the wait that gave up first in a CTA
  kWaitSiteAEmpty = 1u << 8,   // producers: an A stage to drain
  kWaitSiteAFull = 1u << 9,    // MMA issuer: an A stage to fill
  kWaitSiteBFull = 1u << 10,   // MMA issuer: streamed weights to land
  kWaitSiteDFull = 1u << 11,   // epilogue: an accumulator to complete
  kWaitSiteDEmpty = 1u << 12,  // MMA issuer: an accumulator to drain
};

// Launchers (return cudaSuccess or the launch error).  All validation happens
// before these are called.
bool direct_supported(const Geom &g, const char **why);
cudaError_t launch_direct_ffma(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                               cudaStream_t stream);

// Fused conv3d -> min over tensor dim min_dim (2 = depth, 3 = height,
// 4 = width) -> channel softmax.
// ws: a device workspace of fused_transpose_bytes(g, min_dim) bytes, or
// nullptr.  With it, the min over width runs as the min over height of x and
// w transposed in their last two dims (the staged kernel); without it, on the
// generic kernel.
cudaError_t launch_fused_min_softmax(const float *x, const float *w, const float *bias, float *y,
                                     const Geom &g, int min_dim, cudaStream_t stream, float *ws = nullptr);
size_t fused_transpose_bytes(const Geom &g, int min_dim);
// The problem with H and W exchanged, and x and w transposed in their last
// two dims into ws (x at ws, w at ws + transposed_x_bytes(g) / 4 floats;
// transposed_hw_bytes(g) bytes in all, 256-byte sections).
Geom swap_hw_geom(const Geom &g);
size_t transposed_x_bytes(const Geom &g);
size_t transposed_hw_bytes(const Geom &g);
cudaError_t transpose_hw(const float *x, const float *w, float *ws, const Geom &g, cudaStream_t stream);
// True when launch_fused_min_softmax supports this geometry (channel count,
// kernel extent along the output's last axis, shared-memory footprint).
bool fused_supported(const Geom &g, int min_dim, const char **why);

// The same fused op on the tensor cores (3xTF32): min over depth, height or
// width (min_dim 2, 3, 4), weights resident in shared memory or streamed from
// ws (a device workspace of igemm_fused_stream_bytes(g) bytes; 0 = resident).
// One launch takes C_out <= 32; wider layers run as blocks of 32 channels with
// min_only (min + bias into y, whose images are y_chans channels apart) and
// then launch_channel_softmax over all of them.
bool igemm_fused_supported(const Geom &g, int min_dim, const char **why);
size_t igemm_fused_stream_bytes(const Geom &g);
cudaError_t launch_igemm_fused_min_softmax(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                                           int min_dim, cudaStream_t stream, float *ws = nullptr,
                                           bool min_only = false, int64_t y_chans = 0);
// In place over y [N][C][plane]: y[n, :, p] = softmax over the C channels
// (maximum subtracted).
cudaError_t launch_channel_softmax(float *y, int64_t N, int64_t C, int64_t plane, cudaStream_t stream);

// Tensor-core implicit GEMM on 16-bit tensors (bfloat16, or float16 when fp16; bit patterns),
// fp32 accumulation, output in the input type.
// Layers with more than 128 output channels per group run in channel blocks
// of 128; weights that exceed shared memory stream from ws, a device
// workspace of igemm_bf16_stream_bytes(g) bytes (0: resident weights).
bool igemm_bf16_supported(const Geom &g, const char **why);
size_t igemm_bf16_stream_bytes(const Geom &g);
cudaError_t launch_igemm_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, const Geom &g,
                              bool fp16, cudaStream_t stream, uint16_t *ws = nullptr);

// Tensor-core implicit GEMM (tcgen05, 3xTF32).  igemm_launches: kernel launches
// one group takes (channel blocks x reduction passes), 0 when unsupported.
bool igemm_supported(const Geom &g, const char **why);
int igemm_launches(const Geom &g);
// Streamed weights: workspace bytes one group needs (0: the layer does not use them).
size_t igemm_stream_bytes_one_group(const Geom &g);
// ws: device workspace of igemm_stream_bytes_one_group(g) bytes for streamed
// weights, or nullptr (then layers whose weights exceed shared memory run in
// reduction passes).
cudaError_t launch_igemm_3xtf32(const float *x, const float *w, const float *bias, float *y, const Geom &g,
                                cudaStream_t stream, float *ws = nullptr);
// One line of plan details for CONVFWD_LOG (tiles, reduction padding, slots,
// passes, whether the weights stream).
void describe_igemm_plan(const Geom &g, bool streamed, char *buf, size_t n);
cudaError_t read_and_clear_device_status(unsigned *flags);
// Clock cycles after which the tensor-core kernels' pipeline waits give up,
// for launches from now on (cycles <= 0: the default, about two seconds).
void set_wait_limit(long long cycles);

// Sets the calling thread's conv_last_error() text (printf format) and returns
// `status`; CONV_OK with an empty message clears it.
int report_error(int status, const char *fmt, ...);

}  // namespace convfwd
