// Checks compiled into the debug build of the library (-DCONVFWD_DEBUG) and
// compiled away otherwise.
//
// Device side: every global index a kernel forms for x, w, y or a workspace is
// tested against the extent of that tensor as seen from the launch's pointer.
// An index outside it sets a bit of the translation unit's debug word,
// records the first such index, and the access is skipped (a load yields 0, a
// store or copy is dropped), so a wrong index never reaches memory and never
// traps.  conv_device_status() ORs the debug words of all translation units
// into the status word; conv_debug_first_bad_index() returns the index.
//
// Host side: CONV_PLAN_CHECK(cond) in a launcher returns, when cond is false,
// an error that the C API reports as CONV_ERR_INTERNAL with the condition's
// text, before anything is launched.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace convfwd {

enum : unsigned {
  kStatusBoundsX = 1u << 1,   // an input (x) index outside x
  kStatusBoundsW = 1u << 2,   // a weight or bias index outside w / bias
  kStatusBoundsY = 1u << 3,   // an output index outside y
  kStatusBoundsWs = 1u << 4,  // a workspace index outside the workspace
  kStatusBoundsShared = 1u << 5,  // a shared-memory staging index outside its buffer
};

// One reader per translation unit: returns and clears its debug word and the
// first recorded index (-1: none).
using DebugReader = cudaError_t (*)(unsigned *bits, long long *first);
void register_debug_reader(DebugReader r);
// Records a failed plan assertion (thread-local text for conv_last_error) and
// returns the cudaError_t the launcher passes up.
cudaError_t plan_check_failed(const char *cond, const char *file, int line);
// True (and clears the flag) when the last launcher error on this thread came
// from a plan assertion.
bool take_plan_failure(const char **text);
// Test hook of the debug build: the extent of x that the device checks use is
// reduced by this many elements (0: the true extent).
long long debug_x_shrink();

}  // namespace convfwd

#ifdef CONVFWD_DEBUG

namespace convfwd {
namespace {  // one copy per translation unit (no relocatable device code)

__device__ unsigned int dbg_bits = 0;
__device__ int dbg_have = 0;
__device__ long long dbg_first = -1;

__device__ __noinline__ void dbg_record(long long i, unsigned bit) {
  atomicOr(&dbg_bits, bit);
  if (atomicCAS(&dbg_have, 0, 1) == 0) *(volatile long long *)&dbg_first = i;
}

__device__ __forceinline__ bool dbg_ok(long long i, long long n, unsigned bit) {
  if ((unsigned long long)i < (unsigned long long)n) return true;
  dbg_record(i, bit);
  return false;
}

cudaError_t dbg_read(unsigned *bits, long long *first) {
  unsigned b = 0;
  long long f = -1;
  cudaError_t e = cudaMemcpyFromSymbol(&b, dbg_bits, sizeof(b));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&f, dbg_first, sizeof(f));
  const unsigned zb = 0;
  const int zh = 0;
  const long long none = -1;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dbg_bits, &zb, sizeof(zb));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dbg_have, &zh, sizeof(zh));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dbg_first, &none, sizeof(none));
  *bits = b;
  *first = b ? f : -1;
  return e;
}

struct DbgRegistrar {
  DbgRegistrar() { register_debug_reader(&dbg_read); }
};
DbgRegistrar dbg_registrar;

}  // namespace
}  // namespace convfwd

#define CONV_DBG_OK(i, n, bit) ::convfwd::dbg_ok((long long)(i), (long long)(n), (bit))
#define CONV_PLAN_CHECK(cond)                                                   \
  do {                                                                          \
    if (!(cond)) return ::convfwd::plan_check_failed(#cond, __FILE__, __LINE__); \
  } while (0)

#else

#define CONV_DBG_OK(i, n, bit) true
#define CONV_PLAN_CHECK(cond) \
  do {                        \
  } while (0)

#endif
