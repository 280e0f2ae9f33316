// wkv7_backward_noalloc: the two-phase backward with its scratch in a fixed array that
// the library itself owns, for callers that cannot hand the library device memory.
//
// The scratch is one file-scope __device__ array.  The CUDA runtime reserves it on a device when this
// file's device code is loaded there (at the library's first use on that device under lazy module loading,
// the default; when the library loads under eager loading) and keeps it until the process exits.  In host
// code the array's name is only a host-side stand-in for the device symbol, never a device address, so its
// device address is looked up with cudaGetSymbolAddress on every call, on the current device: a device that
// was reset (cudaDeviceReset) gets the address of the array reloaded there, never a stale one.
#include <stdint.h>

#include "wkv7.h"
#include "wkv7_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_backward_scratch[WKV7_NOALLOC_SCRATCH_BYTES];

// device address of g_backward_scratch on the current device
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_backward_scratch);
  if (err != cudaSuccess) return wkv7::record_cuda_status(err);
  if (p == nullptr) return WKV7_ERR_CUDA;
  *out = p;
  return WKV7_OK;
}

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int wkv7_backward_noalloc(int B, int T, int H, int D, int chunk, int in_dtype, const void* r,
                                     const void* w, const void* k, const void* v, const void* a, const void* b,
                                     const float* h0, const float* h_ckpt, const float* sa, const float* dy,
                                     const float* dhT, float* dr, float* dw, float* dk, float* dv, float* da,
                                     float* db, float* dh0, void* stream) {
  size_t need = 0;
  int st = wkv7_backward_workspace_size(B, T, H, D, chunk, &need);  // the same size checks as wkv7_backward
  if (st) return st;
  if (in_dtype != WKV7_F32 && in_dtype != WKV7_BF16) return WKV7_ERR_DTYPE;
  if (T > 0) {
    const void* required[] = {r, w, k, v, a, b, h_ckpt, dy, dr, dw, dk, dv, da, db};
    for (const void* p : required)
      if (p == nullptr) return WKV7_ERR_ARG;
    for (const void* p : required)
      if (misaligned16(p)) return WKV7_ERR_ALIGN;
    if (chunk != 32 && sa == nullptr) return WKV7_ERR_ARG;  // the two-phase backward off 32-token chunks reads it
  }
  for (const void* p : {static_cast<const void*>(h0), static_cast<const void*>(dhT), static_cast<const void*>(dh0),
                        static_cast<const void*>(sa)})
    if (p != nullptr && misaligned16(p)) return WKV7_ERR_ALIGN;
  if (need > (size_t)WKV7_NOALLOC_SCRATCH_BYTES) return WKV7_ERR_SCRATCH_LIMIT;

  void* scratch = nullptr;
  if ((st = scratch_address(&scratch))) return st;

  wkv7::BwdArgs p;
  p.B = B; p.T = T; p.H = H; p.chunk = chunk; p.nchunks = wkv7_num_chunks(T, chunk);
  p.bf16 = in_dtype == WKV7_BF16;
  p.in = {r, w, k, v, a, b};
  p.h0 = h0; p.h_ckpt = h_ckpt; p.sa = T > 0 ? sa : nullptr; p.dy = dy; p.dhT = dhT;
  p.dr = dr; p.dw = dw; p.dk = dk; p.dv = dv; p.da = da; p.db = db; p.dh0 = dh0;
  // the same dispatch as wkv7_backward with a workspace.  Every scratch element the kernels read is
  // written earlier in the same call (the walk writes each chunk-end state gradient, and each dsa when
  // the column pass reads them, before the column pass runs): nothing to clear
  const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  return wkv7::record_cuda_status(p.sa == nullptr ? wkv7::launch_backward_transition(p, scratch, false, st_)
                                                  : wkv7::launch_backward_two_phase(p, scratch, st_));
}
