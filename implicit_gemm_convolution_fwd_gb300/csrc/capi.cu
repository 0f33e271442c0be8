// C ABI entry points: argument validation, output-size arithmetic, kernel
// family selection and dispatch.  Nothing here touches tensor data on the host.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/convfwd.h"
#include "conv_internal.cuh"
#include "debug_check.cuh"

using convfwd::Geom;

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, const char *detail = nullptr, long long a = 0, long long b = 0) {
  snprintf(g_last_error, sizeof(g_last_error), fmt, detail ? detail : "", a, b);
  return status;
}

int fail_cuda(cudaError_t e, const char *where) {
  const char *plan = nullptr;
  if (convfwd::take_plan_failure(&plan)) {
    // a launcher's plan assertion (debug build) rather than a CUDA error
    snprintf(g_last_error, sizeof(g_last_error), "%s: plan assertion failed: %s", where, plan);
    return CONV_ERR_INTERNAL;
  }
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return CONV_ERR_CUDA;
}

// Debug build: the translation units' device debug words (registered at
// load time), the test hook's shrink of the checked input extent, and the
// first out-of-range index that conv_device_status last collected.
std::vector<convfwd::DebugReader> &debug_readers() {
  static std::vector<convfwd::DebugReader> r;
  return r;
}
std::atomic<long long> g_debug_x_shrink{0};
std::atomic<long long> g_debug_first_bad{-1};
thread_local char g_plan_failure[384] = "";
thread_local bool g_plan_failed = false;

// CONVFWD_LOG=1 in the environment: one line per launching call on stderr
// with the problem and the plan (kernel family, tiles, reduction padding,
// slots, passes, whether the weights stream).  Read once per process.
bool log_enabled() {
  static const bool on = [] {
    const char *e = getenv("CONVFWD_LOG");
    return e && *e && strcmp(e, "0") != 0;
  }();
  return on;
}

void log_plan(const char *entry, const Geom &g, const char *family, bool streamed) {
  if (!log_enabled()) return;
  char detail[256] = "";
  if (strncmp(family, "igemm_3xtf32", 12) == 0) convfwd::describe_igemm_plan(g, streamed, detail, sizeof(detail));
  fprintf(stderr,
          "convfwd: %s N=%lld C_in=%lld C_out=%lld groups=%lld in=%dx%dx%d k=%dx%dx%d s=%dx%dx%d p=%dx%dx%d "
          "d=%dx%dx%d out=%dx%dx%d%s -> %s %s\n",
          entry, (long long)g.N, (long long)(g.G * g.C), (long long)(g.G * g.K), (long long)g.G, g.D, g.H, g.W, g.KD,
          g.KH, g.KW, g.SD, g.SH, g.SW, g.PD, g.PH, g.PW, g.DD, g.DH, g.DW, g.OD, g.OH, g.OW,
          g.cl ? " channels-last" : "", family, detail);
}

constexpr int64_t kMaxDim = 0x7fffffff;  // every size must fit a signed 32-bit int
constexpr int64_t kMaxHyper = 1 << 20;   // kernel size, stride, pad, dilation cap

// floor(a / b) for b > 0.
int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) q -= 1;
  return q;
}

// a * b with overflow detection against `limit`.
bool mul_ok(int64_t a, int64_t b, int64_t limit, int64_t *out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > limit / a) return false;
  *out = a * b;
  return true;
}

bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes) {
  if (!a || !b) return false;
  uintptr_t a0 = (uintptr_t)a, a1 = a0 + (uintptr_t)abytes;
  uintptr_t b0 = (uintptr_t)b, b1 = b0 + (uintptr_t)bbytes;
  return a0 < b1 && b0 < a1;
}

// Hyper-parameter checks and output sizes (shared by every entry point).
int compute_out_dims(int ndim, const int64_t *in, const int64_t *k, const int64_t *s, const int64_t *p,
                     const int64_t *d, int64_t *out) {
  if (!in || !k || !s || !p || !d || !out) return fail(CONV_ERR_NULL, "conv: NULL dimension array%s");
  if (ndim < 1 || ndim > 3) return fail(CONV_ERR_ARG, "conv: ndim must be 1, 2 or 3%s");
  bool nonpos = false;
  for (int i = 0; i < ndim; ++i) {
    if (in[i] < 1 || in[i] > kMaxDim) return fail(CONV_ERR_ARG, "conv: in_dims[%s%lld] out of range", "", i);
    if (k[i] < 1 || k[i] > kMaxHyper) return fail(CONV_ERR_ARG, "conv: k_dims[%s%lld] out of range", "", i);
    if (s[i] < 1 || s[i] > kMaxHyper) return fail(CONV_ERR_ARG, "conv: stride[%s%lld] out of range", "", i);
    if (d[i] < 1 || d[i] > kMaxHyper) return fail(CONV_ERR_ARG, "conv: dilation[%s%lld] out of range", "", i);
    if (p[i] < 0 || p[i] > kMaxHyper) return fail(CONV_ERR_ARG, "conv: pad[%s%lld] out of range", "", i);
    // all terms are bounded well inside int64 by the caps above
    out[i] = floor_div(in[i] + 2 * p[i] - d[i] * (k[i] - 1) - 1, s[i]) + 1;
    if (out[i] < 1) nonpos = true;
  }
  if (nonpos) return fail(CONV_ERR_SHAPE, "conv: an output size is <= 0 (kernel extent exceeds padded input)%s");
  return CONV_OK;
}

// Shape validation of a conv problem; fills the 3-D geometry and the element
// counts of x, w and y.
int make_geom(int ndim, int64_t N, int64_t C_in, int64_t C_out, const int64_t *in, const int64_t *k,
              const int64_t *s, const int64_t *p, const int64_t *d, Geom *g, int64_t *xe, int64_t *we,
              int64_t *ye, int64_t groups = 1) {
  int64_t out[3];
  int st = compute_out_dims(ndim, in, k, s, p, d, out);
  if (st != CONV_OK) return st;
  if (N < 0 || N > kMaxDim || C_in < 1 || C_in > kMaxDim || C_out < 1 || C_out > kMaxDim)
    return fail(CONV_ERR_ARG, "conv: N must be in [0, 2^31), C_in and C_out in [1, 2^31)%s");
  if (groups < 1 || groups > kMaxDim || C_in % groups != 0 || C_out % groups != 0)
    return fail(CONV_ERR_ARG, "conv: groups must be >= 1 and divide C_in and C_out%s");
  const int64_t Cg = C_in / groups;  // input channels per group (w's second dim)
  const int64_t lim = INT64_MAX / 8;
  int64_t in_sp = 1, out_sp = 1, k_sp = 1, t;
  for (int i = 0; i < ndim; ++i) {
    if (!mul_ok(in_sp, in[i], lim, &in_sp) || !mul_ok(out_sp, out[i], lim, &out_sp) ||
        !mul_ok(k_sp, k[i], lim, &k_sp))
      return fail(CONV_ERR_ARG, "conv: tensor size overflows int64%s");
  }
  if (!mul_ok(N, C_in, lim, &t) || !mul_ok(t, in_sp, lim, xe) || !mul_ok(C_out, Cg, lim, &t) ||
      !mul_ok(t, k_sp, lim, we) || !mul_ok(N, C_out, lim, &t) || !mul_ok(t, out_sp, lim, ye))
    return fail(CONV_ERR_ARG, "conv: tensor size overflows int64%s");
  if (k_sp > kMaxDim || Cg * k_sp > kMaxDim)
    return fail(CONV_ERR_ARG, "conv: reduction length (C_in/groups)*prod(k) must fit in int32%s");
  // Embed into 3-D with leading singleton dims.
  const int off = 3 - ndim;
  int gi[3] = {1, 1, 1}, go[3] = {1, 1, 1}, gk[3] = {1, 1, 1}, gs[3] = {1, 1, 1}, gp[3] = {0, 0, 0},
      gd[3] = {1, 1, 1};
  for (int i = 0; i < ndim; ++i) {
    gi[off + i] = (int)in[i];
    go[off + i] = (int)out[i];
    gk[off + i] = (int)k[i];
    gs[off + i] = (int)s[i];
    gp[off + i] = (int)p[i];
    gd[off + i] = (int)d[i];
  }
  g->N = N;
  g->C = Cg;
  g->K = C_out / groups;
  g->G = groups;
  g->cl = 0;
  g->D = gi[0], g->H = gi[1], g->W = gi[2];
  g->OD = go[0], g->OH = go[1], g->OW = go[2];
  g->KD = gk[0], g->KH = gk[1], g->KW = gk[2];
  g->SD = gs[0], g->SH = gs[1], g->SW = gs[2];
  g->PD = gp[0], g->PH = gp[1], g->PW = gp[2];
  g->DD = gd[0], g->DH = gd[1], g->DW = gd[2];
  return CONV_OK;
}

// Full validation of a conv_fwd_nd call: shapes, then pointers.
// y_elems_override >= 0 replaces the conv output size in the overlap check
// (the fused entry point writes a reduced 4-D output).
int validate_conv(const float *x, const float *w, const float *bias, const float *y, int ndim, int64_t N,
                  int64_t C_in, int64_t C_out, const int64_t *in, const int64_t *k, const int64_t *s,
                  const int64_t *p, const int64_t *d, Geom *g, int64_t y_elems_override = -1,
                  int64_t groups = 1, int esize = 4) {
  int64_t xe, we, ye;
  int st = make_geom(ndim, N, C_in, C_out, in, k, s, p, d, g, &xe, &we, &ye, groups);
  if (st != CONV_OK) return st;
  // an empty batch has empty x and y, which may be NULL
  if (!w || (N > 0 && (!x || !y))) return fail(CONV_ERR_NULL, "conv: x, w and y must be non-NULL%s");
  if (y_elems_override >= 0) ye = y_elems_override;
  if (((uintptr_t)x | (uintptr_t)w | (uintptr_t)y | (uintptr_t)bias) & (uintptr_t)(esize - 1))
    return fail(CONV_ERR_ARG, "conv: x, w, bias, y must be aligned to their element size%s");
  if (ranges_overlap(y, ye * esize, x, xe * esize) || ranges_overlap(y, ye * esize, w, we * esize) ||
      ranges_overlap(y, ye * esize, bias, C_out * esize))
    return fail(CONV_ERR_ARG, "conv: y overlaps an input buffer%s");
  return CONV_OK;
}

// Planner: the tensor-core path where the reduction is a real dense
// contraction (K = C_in*taps and C_out large enough to fill an MMA tile), the
// FFMA direct path otherwise.  A call that can stream weights exceeding
// shared memory runs such a layer in one pass on the tensor cores (0.21 ms
// against 2.77 ms on the direct path for 64 -> 128 channels, 3x3x3, over
// [4, 64, 32, 32, 32]).  Without streaming, layers that need many tensor-core
// launches (channel blocks x reduction passes, each re-gathering x) measured
// no faster than the direct path beyond about six, so they take the direct
// path.
// can_stream: the call can stream weights that exceed shared memory (it has
// or may allocate a workspace), so such a layer runs in one pass.
// CONVFWD_FORCE_ALGO=direct_ffma | igemm_3xtf32 in the environment (read once
// per process): the family that fp32 calls with CONV_ALGO_AUTO (the plain and
// fused convolutions, and conv_select_algo) take wherever it can run the
// problem; elsewhere the planner decides.  Any other value is ignored, with
// one line on stderr.
int forced_algo() {
  static const int f = [] {
    const char *e = getenv("CONVFWD_FORCE_ALGO");
    if (!e || !*e) return -1;
    if (strcmp(e, "direct_ffma") == 0) return (int)CONV_ALGO_DIRECT_FFMA;
    if (strcmp(e, "igemm_3xtf32") == 0) return (int)CONV_ALGO_IGEMM_3XTF32;
    fprintf(stderr, "convfwd: CONVFWD_FORCE_ALGO=%s ignored (direct_ffma or igemm_3xtf32)\n", e);
    return -1;
  }();
  return f;
}


// The fused op's family for CONV_ALGO_AUTO: CONVFWD_FORCE_ALGO where that
// family runs the shape, else the tensor-core kernel wherever it runs, else the
// FFMA kernels.  Measured on GB300 against the FFMA kernels (device time, L2
// flushed) on [N, C_in, 24, 32, 32] inputs with N * C_in held near 384, 3x3x3
// kernels, C_out 8 .. 64, C_in 1 .. 8, min over depth, height and width: the
// tensor cores took every point, from 0.87x the FFMA time (C_in 1, up to 24
// channels) to 0.07x (C_in 8, 64 channels); over depth, FFMA / tensor cores
// in ms: C_out 24 at C_in 1 0.283 / 0.248, C_in 3 (the page's shape) 0.200 /
// 0.107, C_in 8 0.320 / 0.179; C_out 48 at C_in 1 0.593 / 0.495.
int fused_family(const Geom &g, int min_dim, bool ffma_ok, bool tc_ok) {
  (void)g;
  (void)min_dim;
  const int forced = forced_algo();
  if ((forced == CONV_ALGO_DIRECT_FFMA && ffma_ok) || (forced == CONV_ALGO_IGEMM_3XTF32 && tc_ok)) return forced;
  return tc_ok ? CONV_ALGO_IGEMM_3XTF32 : CONV_ALGO_DIRECT_FFMA;
}

int choose_algo(const Geom &g, bool can_stream) {
  const char *why = nullptr;
  const int forced = forced_algo();
  if (forced == CONV_ALGO_DIRECT_FFMA && convfwd::direct_supported(g, &why)) return forced;
  if (forced == CONV_ALGO_IGEMM_3XTF32 && convfwd::igemm_supported(g, &why)) return forced;
  const int64_t red = g.C * (int64_t)g.taps();
  if (red < 64 || g.K < 16 || !convfwd::igemm_supported(g, &why)) return CONV_ALGO_DIRECT_FFMA;
  if (can_stream && convfwd::igemm_stream_bytes_one_group(g) > 0) return CONV_ALGO_IGEMM_3XTF32;
  return convfwd::igemm_launches(g) <= 6 ? CONV_ALGO_IGEMM_3XTF32 : CONV_ALGO_DIRECT_FFMA;
}

// CONV_OK when kernel family `algo` can run geometry g, else the status to return.
int check_algo(const Geom &g, int algo) {
  const char *why = "";
  switch (algo) {
    case CONV_ALGO_DIRECT_FFMA:
      if (!convfwd::direct_supported(g, &why)) return fail(CONV_ERR_UNSUPPORTED, "conv: %s", why);
      return CONV_OK;
    case CONV_ALGO_IGEMM_3XTF32:
      if (!convfwd::igemm_supported(g, &why))
        return fail(CONV_ERR_UNSUPPORTED, "conv: tensor-core path cannot run this shape: %s", why);
      return CONV_OK;
    default:
      return fail(CONV_ERR_ARG, "conv: unknown algo %s%lld", "", algo);
  }
}

// Scratch of conv_fwd_nd_ws_noalloc: a file-scope device array (no allocation
// at call time), its address looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_ws[16u << 20];
void *g_noalloc_ws_ptr[64] = {nullptr};

int noalloc_ws_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_ws_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(CONV_ERR_UNSUPPORTED, "conv_fwd_nd_ws_noalloc: device index above 63%s");
  if (!g_noalloc_ws_ptr[dev]) {
    e = cudaGetSymbolAddress(&g_noalloc_ws_ptr[dev], g_noalloc_ws);
    if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_ws_noalloc: cudaGetSymbolAddress");
  }
  *out = g_noalloc_ws_ptr[dev];
  return CONV_OK;
}

// ---- host-buffer entry point: two copy streams and the events that order
// them against the compute, created on a device's first call and kept.
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t x_ready[2] = {}, comp_done[2] = {}, y_drained[2] = {};
  std::mutex enqueue;  // one call at a time records and waits on the events
};
HostPipe g_host_pipe[64];
std::mutex g_host_pipe_mutex;

int host_pipe(HostPipe **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(CONV_ERR_UNSUPPORTED, "conv_fwd_nd_host: device index above 63%s");
  std::lock_guard<std::mutex> lock(g_host_pipe_mutex);
  HostPipe &hp = g_host_pipe[dev];
  if (!hp.ready) {
    e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&hp.x_ready[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.comp_done[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.y_drained[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: creating its streams and events");
    hp.ready = true;
  }
  *out = &hp;
  return CONV_OK;
}

// Workspace of conv_fwd_nd_host: w, bias, two x chunks, two y chunks, each
// section 256-byte aligned.
struct HostLayout {
  size_t w_off, b_off, x_off[2], y_off[2], total;
  int64_t x_per, y_per;  // elements of one image of x and of y
};

HostLayout host_layout(const Geom &g, int64_t chunk) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  HostLayout L;
  L.x_per = g.G * g.C * g.in_spatial();
  L.y_per = g.G * g.K * g.out_spatial();
  size_t off = 0;
  L.w_off = off;
  off += up((size_t)(g.G * g.K * g.C * g.taps()) * 4);
  L.b_off = off;
  off += up((size_t)(g.G * g.K) * 4);
  for (int i = 0; i < 2; ++i) {
    L.x_off[i] = off;
    off += up((size_t)(chunk * L.x_per) * 4);
  }
  for (int i = 0; i < 2; ++i) {
    L.y_off[i] = off;
    off += up((size_t)(chunk * L.y_per) * 4);
  }
  L.total = off;
  return L;
}

int64_t host_chunk(int64_t N, int64_t chunk) { return (chunk <= 0 || chunk > N) ? (N > 0 ? N : 1) : chunk; }

}  // namespace

void convfwd::register_debug_reader(DebugReader r) { debug_readers().push_back(r); }

cudaError_t convfwd::plan_check_failed(const char *cond, const char *file, int line) {
  const char *base = strrchr(file, '/');
  snprintf(g_plan_failure, sizeof(g_plan_failure), "%s (%s:%d)", cond, base ? base + 1 : file, line);
  g_plan_failed = true;
  return cudaErrorInvalidConfiguration;
}

bool convfwd::take_plan_failure(const char **text) {
  if (!g_plan_failed) return false;
  g_plan_failed = false;
  *text = g_plan_failure;
  return true;
}

long long convfwd::debug_x_shrink() { return g_debug_x_shrink.load(); }

int convfwd::report_error(int status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

extern "C" {

const char *conv_status_string(int status) {
  switch (status) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_NULL: return "CONV_ERR_NULL: a required pointer is NULL";
    case CONV_ERR_ARG: return "CONV_ERR_ARG: argument out of range or misaligned";
    case CONV_ERR_SHAPE: return "CONV_ERR_SHAPE: non-positive output size or inconsistent shapes";
    case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED: valid request not implemented by this library";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA: CUDA runtime error";
    case CONV_ERR_INTERNAL: return "CONV_ERR_INTERNAL: a plan assertion of the debug build failed";
    default: return "unknown conv status";
  }
}

const char *conv_last_error(void) { return g_last_error; }

int conv_out_dims(int ndim, const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                  const int64_t *pad, const int64_t *dilation, int64_t *out_dims) {
  g_last_error[0] = 0;
  return compute_out_dims(ndim, in_dims, k_dims, stride, pad, dilation, out_dims);
}

int conv_select_algo(int ndim, int64_t N, int64_t C_in, int64_t C_out, const int64_t *in_dims,
                     const int64_t *k_dims, const int64_t *stride, const int64_t *pad, const int64_t *dilation,
                     int *algo_out) {
  g_last_error[0] = 0;
  if (!algo_out) return fail(CONV_ERR_NULL, "conv_select_algo: algo_out is NULL%s");
  Geom g;
  int64_t xe, we, ye;
  int st = make_geom(ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, &xe, &we, &ye);
  if (st != CONV_OK) return st;
  *algo_out = choose_algo(g, true);
  return CONV_OK;
}

// Stream-ordered blocks for streamed weights come from a pool of the
// library's, one per device, that keeps up to 64 MiB reserved between calls
// (the device's default pool returns its memory at every synchronisation, and
// mapping it again cost about 0.1 ms per call).  During stream capture the
// default pool serves instead, which graphs support.
cudaMemPool_t g_ws_pool[64] = {};
std::mutex g_ws_pool_mutex;

cudaError_t alloc_stream_ws(void **p, size_t bytes, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  if (cap != cudaStreamCaptureStatusNone) return cudaMallocAsync(p, bytes, s);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(g_ws_pool_mutex);
    if (!g_ws_pool[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t pool = nullptr;
      e = cudaMemPoolCreate(&pool, &props);
      if (e != cudaSuccess) return e;
      uint64_t keep = 64ull << 20;
      e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      if (e != cudaSuccess) {
        cudaMemPoolDestroy(pool);
        return e;
      }
      g_ws_pool[dev] = pool;
    }
  }
  return cudaMallocFromPoolAsync(p, bytes, g_ws_pool[dev], s);
}

// conv_fwd_nd_grouped; may_alloc: a layer whose weights exceed shared memory
// may take a stream-ordered workspace for streamed weights (else: passes).
static int conv_grouped_impl(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                             int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                             const int64_t *stride, const int64_t *pad, const int64_t *dilation, int algo,
                             conv_stream_t stream, bool may_alloc) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, -1,
                         groups);
  if (st != CONV_OK) return st;
  if (algo == CONV_ALGO_AUTO) algo = choose_algo(g, may_alloc);
  st = check_algo(g, algo);
  if (st != CONV_OK) return st;
  if (g.N == 0) return CONV_OK;  // empty batch: nothing to compute
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  if (algo == CONV_ALGO_DIRECT_FFMA) {
    log_plan("conv_fwd_nd", g, "direct_ffma", false);
    e = convfwd::launch_direct_ffma(x, w, bias, y, g, s);  // all groups in one grid
  } else {
    // A layer whose weights exceed shared memory streams them, split once per
    // call, through the kernel in one pass; the split copy lives in a
    // stream-ordered allocation of this call, released on `stream` after the
    // last launch.  Without it the kernel runs one pass per shared-memory load
    // of weights (measured 2.77 against 0.21 ms on a 64 -> 128 channel 3x3x3
    // layer over [4, 64, 32, 32, 32]).  If the allocation fails, the passes.
    const size_t sb = may_alloc ? convfwd::igemm_stream_bytes_one_group(g) : 0;
    float *wsp = nullptr;
    if (sb > 0 && alloc_stream_ws(reinterpret_cast<void **>(&wsp), sb, s) != cudaSuccess) {
      wsp = nullptr;
      (void)cudaGetLastError();
    }
    log_plan("conv_fwd_nd", g, "igemm_3xtf32", wsp != nullptr);
    // one persistent launch per group on views of x, w, bias and y (the
    // kernel's batch strides span all groups' channels); the groups reuse wsp
    // in stream order
    const int64_t xg = g.C * g.in_spatial(), wg = g.K * g.C * g.taps(), yg = g.K * g.out_spatial();
    for (int64_t grp = 0; grp < g.G && e == cudaSuccess; ++grp)
      e = convfwd::launch_igemm_3xtf32(x + grp * xg, w + grp * wg, bias ? bias + grp * g.K : nullptr, y + grp * yg,
                                       g, s, wsp);
    if (wsp) {
      const cudaError_t ef = cudaFreeAsync(wsp, s);
      if (e == cudaSuccess) e = ef;
    }
  }
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd: kernel launch");
  return CONV_OK;
}

int conv_fwd_nd_grouped(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                        int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                        const int64_t *stride, const int64_t *pad, const int64_t *dilation, int algo,
                        conv_stream_t stream) {
  return conv_grouped_impl(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation, algo,
                           stream, true);
}

int conv_fwd_nd_channels_last(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                              int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                              const int64_t *k_dims, const int64_t *stride, const int64_t *pad,
                              const int64_t *dilation, int algo, conv_stream_t stream) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, -1,
                         groups);
  if (st != CONV_OK) return st;
  g.cl = 1;
  if (algo == CONV_ALGO_DIRECT_FFMA)
    return fail(CONV_ERR_UNSUPPORTED, "conv: channels-last tensors run on the tensor-core family only%s");
  const char *why = "";
  if (!convfwd::igemm_supported(g, &why))
    return fail(CONV_ERR_UNSUPPORTED, "conv: tensor-core path cannot run this channels-last shape: %s", why);
  if (algo != CONV_ALGO_AUTO && algo != CONV_ALGO_IGEMM_3XTF32)
    return fail(CONV_ERR_ARG, "conv: unknown algo %s%lld", "", algo);
  if (g.N == 0) return CONV_OK;
  // weights beyond shared memory stream from a stream-ordered block, as in
  // conv_fwd_nd (one pass instead of one per shared-memory load of weights)
  cudaStream_t s = (cudaStream_t)stream;
  const size_t sb = convfwd::igemm_stream_bytes_one_group(g);
  float *wsp = nullptr;
  if (sb > 0 && alloc_stream_ws(reinterpret_cast<void **>(&wsp), sb, s) != cudaSuccess) {
    wsp = nullptr;
    (void)cudaGetLastError();
  }
  log_plan("conv_fwd_nd_channels_last", g, "igemm_3xtf32", wsp != nullptr);
  // one launch per group on channel offsets of x, w, bias and y (the groups reuse wsp in stream order)
  cudaError_t e = cudaSuccess;
  for (int64_t grp = 0; grp < g.G && e == cudaSuccess; ++grp)
    e = convfwd::launch_igemm_3xtf32(x + grp * g.C, w + grp * g.K * g.C * g.taps(), bias ? bias + grp * g.K : nullptr,
                                     y + grp * g.K, g, s, wsp);
  if (wsp) {
    const cudaError_t ef = cudaFreeAsync(wsp, s);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_channels_last: kernel launch");
  return CONV_OK;
}

// 16-bit tensors (bfloat16 or float16 bit patterns) on the tensor cores.
static int conv_fwd_16bit(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, int ndim, int64_t N,
                          int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                          const int64_t *stride, const int64_t *pad, const int64_t *dilation, bool fp16,
                          conv_stream_t stream, const char *name) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv((const float *)x, (const float *)w, (const float *)bias, (const float *)y, ndim, N, C_in,
                         C_out, in_dims, k_dims, stride, pad, dilation, &g, -1, groups, 2);
  if (st != CONV_OK) return st;
  const char *why = "";
  if (!convfwd::igemm_bf16_supported(g, &why))
    return fail(CONV_ERR_UNSUPPORTED, fp16 ? "conv_fwd_nd_f16: the tensor-core path cannot run this shape: %s"
                                           : "conv_fwd_nd_bf16: the tensor-core path cannot run this shape: %s",
                why);
  if (g.N == 0) return CONV_OK;
  // weights beyond shared memory stream from a stream-ordered block (reused
  // by every channel block and group in stream order)
  cudaStream_t s = (cudaStream_t)stream;
  const size_t sb = convfwd::igemm_bf16_stream_bytes(g);
  uint16_t *wsp = nullptr;
  if (sb > 0) {
    const cudaError_t ea = alloc_stream_ws(reinterpret_cast<void **>(&wsp), sb, s);
    if (ea != cudaSuccess) return fail_cuda(ea, name);
  }
  log_plan(name, g, fp16 ? "igemm_f16" : "igemm_bf16", wsp != nullptr);
  const int64_t xg = g.C * g.in_spatial(), wg = g.K * g.C * g.taps(), yg = g.K * g.out_spatial();
  cudaError_t e = cudaSuccess;
  for (int64_t grp = 0; grp < g.G && e == cudaSuccess; ++grp)
    e = convfwd::launch_igemm_bf16(x + grp * xg, w + grp * wg, bias ? bias + grp * g.K : nullptr, y + grp * yg, g,
                                   fp16, s, wsp);
  if (wsp) {
    const cudaError_t ef = cudaFreeAsync(wsp, s);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return fail_cuda(e, name);
  return CONV_OK;
}

int conv_fwd_nd_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, int ndim, int64_t N,
                     int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                     const int64_t *stride, const int64_t *pad, const int64_t *dilation, conv_stream_t stream) {
  return conv_fwd_16bit(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation, false,
                        stream, "conv_fwd_nd_bf16");
}

int conv_fwd_nd_f16(const uint16_t *x, const uint16_t *w, const uint16_t *bias, uint16_t *y, int ndim, int64_t N,
                    int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                    const int64_t *stride, const int64_t *pad, const int64_t *dilation, conv_stream_t stream) {
  return conv_fwd_16bit(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation, true,
                        stream, "conv_fwd_nd_f16");
}

int conv_workspace_bytes(int ndim, int64_t N, int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims,
                         const int64_t *k_dims, const int64_t *stride, const int64_t *pad, const int64_t *dilation,
                         size_t *bytes) {
  g_last_error[0] = 0;
  if (!bytes) return fail(CONV_ERR_NULL, "conv_workspace_bytes: bytes is NULL%s");
  Geom g;
  int64_t xe, we, ye;
  int st = make_geom(ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, &xe, &we, &ye, groups);
  if (st != CONV_OK) return st;
  *bytes = convfwd::igemm_stream_bytes_one_group(g) * (size_t)g.G;
  return CONV_OK;
}

int conv_fwd_nd_ws(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N, int64_t C_in,
                   int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                   const int64_t *pad, const int64_t *dilation, void *workspace, size_t workspace_bytes,
                   conv_stream_t stream) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, -1,
                         groups);
  if (st != CONV_OK) return st;
  const size_t one = convfwd::igemm_stream_bytes_one_group(g);
  if (one == 0 || !workspace)  // nothing to stream, or no workspace: the call without allocations
    return conv_grouped_impl(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation,
                             CONV_ALGO_AUTO, stream, false);
  if (workspace_bytes < one * (size_t)g.G)
    return fail(CONV_ERR_ARG, "conv_fwd_nd_ws: workspace smaller than conv_workspace_bytes%s");
  if ((uintptr_t)workspace & 255u) return fail(CONV_ERR_ARG, "conv_fwd_nd_ws: workspace must be 256-byte aligned%s");
  const int64_t ye = g.N * g.G * g.K * g.out_spatial(), xe = g.N * g.G * g.C * g.in_spatial();
  const int64_t we = g.G * g.K * g.C * g.taps();
  const int64_t wsb = (int64_t)(one * (size_t)g.G);
  if (ranges_overlap(workspace, wsb, x, xe * 4) || ranges_overlap(workspace, wsb, w, we * 4) ||
      ranges_overlap(workspace, wsb, y, ye * 4) || ranges_overlap(workspace, wsb, bias, g.G * g.K * 4))
    return fail(CONV_ERR_ARG, "conv_fwd_nd_ws: workspace overlaps a tensor%s");
  if (g.N == 0) return CONV_OK;
  log_plan("conv_fwd_nd_ws", g, "igemm_3xtf32", true);
  const int64_t xg = g.C * g.in_spatial(), wg = g.K * g.C * g.taps(), yg = g.K * g.out_spatial();
  float *wsf = static_cast<float *>(workspace);
  cudaError_t e = cudaSuccess;
  for (int64_t grp = 0; grp < g.G && e == cudaSuccess; ++grp)
    e = convfwd::launch_igemm_3xtf32(x + grp * xg, w + grp * wg, bias ? bias + grp * g.K : nullptr, y + grp * yg, g,
                                     (cudaStream_t)stream, wsf + grp * (int64_t)(one / 4));
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_ws: kernel launch");
  return CONV_OK;
}

int conv_fwd_nd_ws_noalloc(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                           int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                           const int64_t *stride, const int64_t *pad, const int64_t *dilation, conv_stream_t stream) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, -1,
                         groups);
  if (st != CONV_OK) return st;
  const size_t need = convfwd::igemm_stream_bytes_one_group(g) * (size_t)g.G;
  if (need == 0)
    return conv_grouped_impl(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation,
                             CONV_ALGO_AUTO, stream, false);
  if (need > sizeof(g_noalloc_ws))
    return fail(CONV_ERR_UNSUPPORTED, "conv_fwd_nd_ws_noalloc: needs %s%lld bytes of scratch, the static buffer holds %lld",
                "", (long long)need, (long long)sizeof(g_noalloc_ws));
  void *ws = nullptr;
  st = noalloc_ws_address(&ws);
  if (st != CONV_OK) return st;
  return conv_fwd_nd_ws(x, w, bias, y, ndim, N, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation, ws,
                        sizeof(g_noalloc_ws), stream);
}

int conv_host_workspace_bytes(int ndim, int64_t N, int64_t C_in, int64_t C_out, int64_t groups,
                              const int64_t *in_dims, const int64_t *k_dims, const int64_t *stride,
                              const int64_t *pad, const int64_t *dilation, int64_t chunk, size_t *bytes) {
  g_last_error[0] = 0;
  if (!bytes) return fail(CONV_ERR_NULL, "conv_host_workspace_bytes: bytes is NULL%s");
  Geom g;
  int64_t xe, we, ye;
  int st = make_geom(ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, &xe, &we, &ye, groups);
  if (st != CONV_OK) return st;
  *bytes = host_layout(g, host_chunk(N, chunk)).total;
  return CONV_OK;
}

int conv_fwd_nd_host(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                     int64_t C_in, int64_t C_out, int64_t groups, const int64_t *in_dims, const int64_t *k_dims,
                     const int64_t *stride, const int64_t *pad, const int64_t *dilation, int64_t chunk,
                     void *workspace, size_t workspace_bytes, conv_stream_t stream) {
  g_last_error[0] = 0;
  Geom g;
  int st = validate_conv(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, -1,
                         groups);
  if (st != CONV_OK) return st;
  if (!workspace) return fail(CONV_ERR_NULL, "conv_fwd_nd_host: workspace is NULL%s");
  if (g.N == 0) return CONV_OK;  // empty batch: nothing to copy or compute
  if ((uintptr_t)workspace & 255u) return fail(CONV_ERR_ARG, "conv_fwd_nd_host: workspace must be 256-byte aligned%s");
  chunk = host_chunk(N, chunk);
  const HostLayout L = host_layout(g, chunk);
  if (workspace_bytes < L.total)
    return fail(CONV_ERR_ARG, "conv_fwd_nd_host: workspace smaller than conv_host_workspace_bytes%s");
  HostPipe *hp = nullptr;
  st = host_pipe(&hp);
  if (st != CONV_OK) return st;
  // the events are shared by every call on the device: enqueue one call at a time
  std::lock_guard<std::mutex> lock(hp->enqueue);
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *wd = reinterpret_cast<float *>(ws + L.w_off);
  float *bd = bias ? reinterpret_cast<float *>(ws + L.b_off) : nullptr;
  const int64_t we = g.G * g.K * g.C * g.taps();
  // weights and bias travel on the compute stream, ahead of the first chunk
  cudaError_t e = cudaMemcpyAsync(wd, w, (size_t)we * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && bias) e = cudaMemcpyAsync(bd, bias, (size_t)(g.G * g.K) * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: weight copy");
  for (int64_t n0 = 0, i = 0; n0 < N; n0 += chunk, ++i) {
    const int slot = (int)(i & 1);
    const int64_t nb = N - n0 < chunk ? N - n0 : chunk;
    float *xd = reinterpret_cast<float *>(ws + L.x_off[slot]);
    float *yd = reinterpret_cast<float *>(ws + L.y_off[slot]);
    // x chunk into its slot once the conv that last read the slot is done
    e = cudaStreamWaitEvent(hp->h2d, hp->comp_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(xd, x + n0 * L.x_per, (size_t)(nb * L.x_per) * 4, cudaMemcpyHostToDevice, hp->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(hp->x_ready[slot], hp->h2d);
    // the conv waits for its input and for the slot's previous output to leave
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->x_ready[slot], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->y_drained[slot], 0);
    if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: input copy");
    st = conv_fwd_nd_grouped(xd, wd, bd, yd, ndim, nb, C_in, C_out, groups, in_dims, k_dims, stride, pad, dilation,
                             CONV_ALGO_AUTO, stream);
    if (st != CONV_OK) return st;
    e = cudaEventRecord(hp->comp_done[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->comp_done[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(y + n0 * L.y_per, yd, (size_t)(nb * L.y_per) * 4, cudaMemcpyDeviceToHost, hp->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(hp->y_drained[slot], hp->d2h);
    if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: output copy");
  }
  // `stream` completes after the last output copies
  e = cudaStreamWaitEvent(s, hp->y_drained[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->y_drained[1], 0);
  if (e != cudaSuccess) return fail_cuda(e, "conv_fwd_nd_host: final wait");
  return CONV_OK;
}

int conv_fwd_nd_ex(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                   int64_t C_in, int64_t C_out, const int64_t *in_dims, const int64_t *k_dims,
                   const int64_t *stride, const int64_t *pad, const int64_t *dilation, int algo,
                   conv_stream_t stream) {
  return conv_fwd_nd_grouped(x, w, bias, y, ndim, N, C_in, C_out, 1, in_dims, k_dims, stride, pad, dilation, algo,
                             stream);
}

int conv_algo_supported(int ndim, int64_t N, int64_t C_in, int64_t C_out, const int64_t *in_dims,
                        const int64_t *k_dims, const int64_t *stride, const int64_t *pad, const int64_t *dilation,
                        int algo) {
  g_last_error[0] = 0;
  Geom g;
  int64_t xe, we, ye;
  int st = make_geom(ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation, &g, &xe, &we, &ye);
  if (st != CONV_OK) return st;
  if (algo == CONV_ALGO_AUTO) return CONV_OK;
  return check_algo(g, algo);
}

int conv_fwd_nd(const float *x, const float *w, const float *bias, float *y, int ndim, int64_t N,
                int64_t C_in, int64_t C_out, const int64_t *in_dims, const int64_t *k_dims,
                const int64_t *stride, const int64_t *pad, const int64_t *dilation, conv_stream_t stream) {
  return conv_fwd_nd_ex(x, w, bias, y, ndim, N, C_in, C_out, in_dims, k_dims, stride, pad, dilation,
                        CONV_ALGO_AUTO, stream);
}

int conv3d_min_softmax(const conv_tensor5_t *x, const conv_tensor5_t *w, const float *bias, conv_tensor4_t *y,
                       int min_dim, conv_stream_t stream) {
  return conv3d_min_softmax_ex(x, w, bias, y, min_dim, CONV_ALGO_AUTO, stream);
}

int conv3d_min_softmax_ex(const conv_tensor5_t *x, const conv_tensor5_t *w, const float *bias, conv_tensor4_t *y,
                          int min_dim, int algo, conv_stream_t stream) {
  g_last_error[0] = 0;
  if (!x || !w || !y) return fail(CONV_ERR_NULL, "conv3d_min_softmax: descriptor pointer is NULL%s");
  if (!w->data || (x->dims[0] != 0 && (!x->data || !y->data)))
    return fail(CONV_ERR_NULL, "conv3d_min_softmax: tensor data is NULL%s");
  if (min_dim < 2 || min_dim > 4) return fail(CONV_ERR_ARG, "conv3d_min_softmax: min_dim must be 2, 3 or 4%s");
  for (int i = 0; i < 5; ++i) {
    if (x->dims[i] < (i == 0 ? 0 : 1) || x->dims[i] > kMaxDim)
      return fail(CONV_ERR_ARG, "conv3d_min_softmax: bad x dim%s");
    if (w->dims[i] < 1 || w->dims[i] > kMaxDim) return fail(CONV_ERR_ARG, "conv3d_min_softmax: bad w dim%s");
  }
  if (w->dims[1] != x->dims[1])
    return fail(CONV_ERR_SHAPE, "conv3d_min_softmax: w C_in %s%lld != x C_in %lld", "", w->dims[1], x->dims[1]);
  const int64_t ins[3] = {x->dims[2], x->dims[3], x->dims[4]};
  const int64_t ks[3] = {w->dims[2], w->dims[3], w->dims[4]};
  const int64_t one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
  Geom g;
  float *yd = y->data;
  int64_t y4 = 1;
  for (int i = 0; i < 4; ++i) {
    if (y->dims[i] < 0 || y->dims[i] > kMaxDim) return fail(CONV_ERR_SHAPE, "conv3d_min_softmax: bad y dim%s");
    y4 *= y->dims[i];  // each factor < 2^31, product checked against x/w sizes below
  }
  int st = validate_conv(x->data, w->data, bias, yd, 3, x->dims[0], x->dims[1], w->dims[0], ins, ks, one, zero,
                         one, &g, y4);
  if (st != CONV_OK) return st;
  // the output keeps the two spatial axes other than min_dim, in order
  const int64_t ya = (min_dim == 2) ? g.OH : g.OD, yb = (min_dim == 4) ? g.OH : g.OW;
  if (y->dims[0] != g.N || y->dims[1] != g.K || y->dims[2] != ya || y->dims[3] != yb)
    return fail(CONV_ERR_SHAPE,
                "conv3d_min_softmax: y dims must be [N, C_out] + the conv's spatial output dims without dim "
                "min_dim%s");
  const char *why = "", *why_tc = "";
  const bool ffma_ok = convfwd::fused_supported(g, min_dim, &why);
  const bool tc_ok = convfwd::igemm_fused_supported(g, min_dim, &why_tc);
  if (algo == CONV_ALGO_AUTO) algo = fused_family(g, min_dim, ffma_ok, tc_ok);
  if (algo == CONV_ALGO_DIRECT_FFMA) {
    if (!ffma_ok) return fail(CONV_ERR_UNSUPPORTED, "conv3d_min_softmax: %s", why);
  } else if (algo == CONV_ALGO_IGEMM_3XTF32) {
    if (!tc_ok) return fail(CONV_ERR_UNSUPPORTED, "conv3d_min_softmax: %s", why_tc);
  } else {
    return fail(CONV_ERR_ARG, "conv3d_min_softmax: unknown algo %s%lld", "", algo);
  }
  if (g.N == 0) return CONV_OK;  // empty batch
  log_plan(min_dim == 2 ? "conv3d_min_softmax(min over depth)" : min_dim == 3 ? "conv3d_min_softmax(min over height)"
                                                                             : "conv3d_min_softmax(min over width)",
           g, algo == CONV_ALGO_IGEMM_3XTF32 ? "fused igemm_3xtf32" : "fused ffma", false);
  cudaError_t e = cudaSuccess;
  if (algo == CONV_ALGO_IGEMM_3XTF32) {
    // The min over width runs as the min over height of x and w transposed in
    // their last two dims (its tiles then read rows of x, not columns); weights
    // beyond shared memory stream, as in conv_fwd_nd.  Both live in one
    // stream-ordered block (transposed copies first).
    cudaStream_t s = (cudaStream_t)stream;
    const Geom gt = min_dim == 4 ? convfwd::swap_hw_geom(g) : g;
    size_t tb = min_dim == 4 ? convfwd::transposed_hw_bytes(g) : 0;
    size_t sb = convfwd::igemm_fused_stream_bytes(gt);
    float *wsp = nullptr;
    if (tb + sb > 0 && alloc_stream_ws(reinterpret_cast<void **>(&wsp), tb + sb, s) != cudaSuccess) {
      (void)cudaGetLastError();
      wsp = nullptr;
      // without the transposed copies the min over width reads columns of x directly
      tb = 0;
      sb = convfwd::igemm_fused_stream_bytes(g);
      if (sb > 0) {
        e = alloc_stream_ws(reinterpret_cast<void **>(&wsp), sb, s);
        if (e != cudaSuccess) return fail_cuda(e, "conv3d_min_softmax: weight workspace");
      }
    }
    const float *xk = x->data, *wk = w->data;
    Geom gk = g;
    int mk = min_dim;
    if (tb > 0) {
      e = convfwd::transpose_hw(x->data, w->data, wsp, g, s);
      xk = wsp;
      wk = wsp + convfwd::transposed_x_bytes(g) / 4;
      gk = gt;
      mk = 3;
    }
    // at most 32 channels per launch: a wider layer runs block by block (min +
    // bias into y), then one softmax pass over all channels
    const int64_t plane = (int64_t)g.OD * g.OH * g.OW / (min_dim == 2 ? g.OD : min_dim == 3 ? g.OH : g.OW);
    const bool blocks = g.K > 32;
    for (int64_t c0 = 0; c0 < g.K && e == cudaSuccess; c0 += 32) {
      Geom gb = gk;
      gb.K = g.K - c0 < 32 ? g.K - c0 : 32;
      e = convfwd::launch_igemm_fused_min_softmax(xk, wk + c0 * g.C * g.taps(), bias ? bias + c0 : nullptr,
                                                  yd + c0 * plane, gb, mk, s, sb > 0 ? wsp + tb / 4 : nullptr,
                                                  blocks, g.K);
    }
    if (blocks && e == cudaSuccess) e = convfwd::launch_channel_softmax(yd, g.N, g.K, plane, s);
    if (wsp) {
      const cudaError_t ef = cudaFreeAsync(wsp, s);
      if (e == cudaSuccess) e = ef;
    }
  } else {
    // the min over width runs faster as a min over height of transposed copies of x and w
    // (a stream-ordered block); without the block, on the generic kernel
    const size_t tb = convfwd::fused_transpose_bytes(g, min_dim);
    float *wsp = nullptr;
    if (tb > 0 && alloc_stream_ws(reinterpret_cast<void **>(&wsp), tb, (cudaStream_t)stream) != cudaSuccess) {
      wsp = nullptr;
      (void)cudaGetLastError();
    }
    e = convfwd::launch_fused_min_softmax(x->data, w->data, bias, yd, g, min_dim, (cudaStream_t)stream, wsp);
    if (wsp) {
      const cudaError_t ef = cudaFreeAsync(wsp, (cudaStream_t)stream);
      if (e == cudaSuccess) e = ef;
    }
  }
  if (e != cudaSuccess) return fail_cuda(e, "conv3d_min_softmax: kernel launch");
  return CONV_OK;
}

int conv3d_min_softmax_select_algo(const conv_tensor5_t *x, const conv_tensor5_t *w, int min_dim, int *algo_out) {
  g_last_error[0] = 0;
  if (!x || !w || !algo_out) return fail(CONV_ERR_NULL, "conv3d_min_softmax_select_algo: a pointer is NULL%s");
  if (min_dim < 2 || min_dim > 4)
    return fail(CONV_ERR_ARG, "conv3d_min_softmax_select_algo: min_dim must be 2, 3 or 4%s");
  for (int i = 0; i < 5; ++i) {
    if (x->dims[i] < (i == 0 ? 0 : 1) || x->dims[i] > kMaxDim)
      return fail(CONV_ERR_ARG, "conv3d_min_softmax_select_algo: bad x dim%s");
    if (w->dims[i] < 1 || w->dims[i] > kMaxDim)
      return fail(CONV_ERR_ARG, "conv3d_min_softmax_select_algo: bad w dim%s");
  }
  if (w->dims[1] != x->dims[1])
    return fail(CONV_ERR_SHAPE, "conv3d_min_softmax_select_algo: w C_in %s%lld != x C_in %lld", "", w->dims[1],
                x->dims[1]);
  const int64_t ins[3] = {x->dims[2], x->dims[3], x->dims[4]};
  const int64_t ks[3] = {w->dims[2], w->dims[3], w->dims[4]};
  const int64_t one[3] = {1, 1, 1}, zero[3] = {0, 0, 0};
  Geom g;
  int64_t xe, we, ye;
  int st = make_geom(3, x->dims[0], x->dims[1], w->dims[0], ins, ks, one, zero, one, &g, &xe, &we, &ye);
  if (st != CONV_OK) return st;
  const char *why = "", *why_tc = "";
  const bool ffma_ok = convfwd::fused_supported(g, min_dim, &why);
  const bool tc_ok = convfwd::igemm_fused_supported(g, min_dim, &why_tc);
  if (!ffma_ok && !tc_ok) return fail(CONV_ERR_UNSUPPORTED, "conv3d_min_softmax_select_algo: %s", why_tc);
  *algo_out = fused_family(g, min_dim, ffma_ok, tc_ok);
  return CONV_OK;
}

int conv_debug_set_wait_limit(long long cycles) {
  g_last_error[0] = 0;
  if (cycles > 0 && cycles < 64) return fail(CONV_ERR_ARG, "conv_debug_set_wait_limit: at least 64 cycles%s");
  convfwd::set_wait_limit(cycles);
  return CONV_OK;
}

int conv_device_status(unsigned int *flags) {
  g_last_error[0] = 0;
  if (!flags) return fail(CONV_ERR_NULL, "conv_device_status: flags is NULL%s");
  cudaError_t e = convfwd::read_and_clear_device_status(flags);
  if (e != cudaSuccess) return fail_cuda(e, "conv_device_status");
  long long first = -1;
  for (convfwd::DebugReader r : debug_readers()) {
    unsigned b = 0;
    long long f = -1;
    e = r(&b, &f);
    if (e != cudaSuccess) return fail_cuda(e, "conv_device_status: debug words");
    *flags |= b;
    if (first < 0 && f >= 0) first = f;
  }
  if (!debug_readers().empty()) g_debug_first_bad.store(first);
  return CONV_OK;
}

int conv_build_flags(void) {
#ifdef CONVFWD_DEBUG
  return CONV_BUILD_DEBUG;
#else
  return 0;
#endif
}

int conv_debug_shrink_bounds(long long elems) {
  g_last_error[0] = 0;
#ifdef CONVFWD_DEBUG
  if (elems < 0) return fail(CONV_ERR_ARG, "conv_debug_shrink_bounds: elems = %s%lld is negative", nullptr, elems);
  g_debug_x_shrink.store(elems);
  return CONV_OK;
#else
  (void)elems;
  return fail(CONV_ERR_UNSUPPORTED, "conv_debug_shrink_bounds: this library was built without CONVFWD_DEBUG%s");
#endif
}

int conv_debug_first_bad_index(long long *index) {
  g_last_error[0] = 0;
  if (!index) return fail(CONV_ERR_NULL, "conv_debug_first_bad_index: index is NULL%s");
#ifdef CONVFWD_DEBUG
  *index = g_debug_first_bad.load();
  return CONV_OK;
#else
  *index = -1;
  return fail(CONV_ERR_UNSUPPORTED, "conv_debug_first_bad_index: this library was built without CONVFWD_DEBUG%s");
#endif
}

}  // extern "C"
