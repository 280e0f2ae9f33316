// Device-side index checks of the debug build (compiled with WKV7_DEBUG_CHECKS: build.py --debug makes
// libwkv7_debug.so).  A failed check sets its kernel's bit in a status word of the source file and the
// access is skipped or pointed at a safe address instead: nothing traps, nothing returns early (so no
// barrier is left waiting).  wkv7_debug_status() in wkv7_api.cu reads and clears every file's word.
// In release builds WKV7_IN(...) is the constant true and the readers report 0.
#pragma once

#include <cuda_runtime.h>

namespace wkv7 {
namespace dbg {
enum : unsigned {
  kOperand = 1u << 0,   // a shared-memory operand helper (row or column outside the array)
  kXopPrep = 1u << 1,   // chunk-operator prep
  kXopChain = 1u << 2,  // chunk-operator chain
  kColmat = 1u << 3,    // matrix column gradients
  kColfb = 1u << 4,     // token-by-token column gradients
  kOther = 1u << 5,     // any other kernel
};
}  // namespace dbg
}  // namespace wkv7

#ifdef WKV7_DEBUG_CHECKS
static __device__ unsigned int wkv7_dbg_word;
__device__ __forceinline__ bool wkv7_in_range(long long idx, long long lim, unsigned code) {
  if (idx >= 0 && idx < lim) return true;
  atomicOr(&wkv7_dbg_word, code);
  return false;
}
#define WKV7_IN(idx, lim, code) wkv7_in_range((long long)(idx), (long long)(lim), (code))
// host: read and clear this file's word
#define WKV7_DEBUG_READER(name)                                                          \
  int name(unsigned* out) {                                                              \
    unsigned v = 0, z = 0;                                                               \
    cudaError_t e = cudaMemcpyFromSymbol(&v, wkv7_dbg_word, sizeof(v));                  \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(wkv7_dbg_word, &z, sizeof(z));          \
    *out = v;                                                                            \
    return (int)e;                                                                       \
  }
#else
#define WKV7_IN(idx, lim, code) true
#define WKV7_DEBUG_READER(name) \
  int name(unsigned* out) {     \
    *out = 0;                   \
    return 0;                   \
  }
#endif
