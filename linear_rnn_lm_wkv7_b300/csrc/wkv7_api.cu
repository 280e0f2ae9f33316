// extern "C" entry points of libwkv7: argument checks on the host, then one launch on
// the caller's stream.  Declared (with layouts, ownership and errors) in include/wkv7.h.
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <climits>
#include <initializer_list>

#include "wkv7.h"
#include "wkv7_launch.h"

namespace {

thread_local char g_last_cuda_error[256] = "";

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxChunk = 32;
constexpr int kHeadSize = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int record_cuda(cudaError_t err) {
  if (err == cudaSuccess) return WKV7_OK;
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(err),
           cudaGetErrorString(err));
  return WKV7_ERR_CUDA;
}

int check_dtype(int in_dtype) {
  return (in_dtype == WKV7_F32 || in_dtype == WKV7_BF16) ? WKV7_OK : WKV7_ERR_DTYPE;
}

// sizes shared by forward and backward; element counts must stay inside the index range
int check_sizes(int B, int T, int H, int D, int chunk) {
  if (B < 1 || H < 1 || T < 0) return WKV7_ERR_ARG;
  if (D != kHeadSize) return WKV7_ERR_SHAPE;
  if (chunk < 1 || chunk > kMaxChunk) return WKV7_ERR_SHAPE;
  const unsigned long long bh = (unsigned long long)B * (unsigned long long)H;
  if (bh * 4ull > (unsigned long long)INT_MAX) return WKV7_ERR_SHAPE;
  const unsigned long long elems = bh * (unsigned long long)(T > 0 ? T : 1) * 64ull;
  if (elems > (1ull << 40)) return WKV7_ERR_SHAPE;
  return WKV7_OK;
}

int check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
  for (const void* p : required)
    if (p == nullptr) return WKV7_ERR_ARG;
  for (const void* p : required)
    if (!aligned16(p)) return WKV7_ERR_ALIGN;
  for (const void* p : optional)
    if (p != nullptr && !aligned16(p)) return WKV7_ERR_ALIGN;
  return WKV7_OK;
}

}  // namespace

namespace wkv7 {

int record_cuda_status(cudaError_t err) { return record_cuda(err); }

int num_sms() {
  static thread_local int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace wkv7

extern "C" {

int wkv7_version(void) { return kVersion; }

int wkv7_num_chunks(int T, int chunk) {
  if (T <= 0 || chunk <= 0) return 0;
  return (T + chunk - 1) / chunk;
}

const char* wkv7_strerror(int status) {
  switch (status) {
    case WKV7_OK: return "ok";
    case WKV7_ERR_ARG: return "invalid argument: a required pointer is NULL or a size is out of range";
    case WKV7_ERR_SHAPE: return "unsupported shape: D must be 64, chunk in [1, 32], sizes within the index range";
    case WKV7_ERR_ALIGN: return "misaligned pointer: every buffer must be 16-byte aligned";
    case WKV7_ERR_DTYPE: return "unsupported input dtype: use WKV7_F32 or WKV7_BF16";
    case WKV7_ERR_CUDA: return "CUDA error at launch (see wkv7_last_cuda_error)";
    case WKV7_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case WKV7_ERR_WORKSPACE: return "workspace smaller than wkv7_backward_workspace_size()";
    case WKV7_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the library's fixed WKV7_NOALLOC_SCRATCH_BYTES: use wkv7_backward "
             "with a workspace";
    default: return "unknown wkv7 status";
  }
}

const char* wkv7_last_cuda_error(void) { return g_last_cuda_error; }

namespace {
int forward_impl(bool sequential, int B, int T, int H, int D, int chunk, int in_dtype, const void* r,
                 const void* w, const void* k, const void* v, const void* a, const void* b, const float* h0,
                 float* y, float* h_ckpt, float* hT, float* sa, void* workspace, size_t workspace_bytes,
                 void* stream) {
  int st = check_sizes(B, T, H, D, chunk);
  if (st) return st;
  if ((st = check_dtype(in_dtype))) return st;
  if (T > 0) {
    if ((st = check_ptrs({r, w, k, v, a, b, y}, {h0, h_ckpt, hT, sa}))) return st;
  } else if ((st = check_ptrs({}, {h0, hT}))) {
    return st;
  }
  wkv7::FwdArgs p;
  p.B = B; p.T = T; p.H = H; p.chunk = chunk; p.nchunks = wkv7_num_chunks(T, chunk);
  p.bf16 = in_dtype == WKV7_BF16;
  p.in = {r, w, k, v, a, b};
  p.h0 = h0; p.y = y; p.h_ckpt = h_ckpt; p.hT = hT; p.sa = T > 0 ? sa : nullptr;
  const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  if (sequential) return record_cuda(wkv7::launch_forward_sequential(p, st_));
  if (workspace != nullptr && chunk == 32 && p.sa == nullptr && T > 0) {
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return WKV7_ERR_ALIGN;
    if (workspace_bytes < wkv7::forward_workspace_bytes(B, T, H, chunk)) return WKV7_ERR_WORKSPACE;
    return record_cuda(wkv7::launch_xop_forward(p, workspace, 0, st_));
  }
  return record_cuda(wkv7::launch_forward(p, st_));
}
}  // namespace

int wkv7_forward(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w,
                 const void* k, const void* v, const void* a, const void* b, const float* h0, float* y,
                 float* h_ckpt, float* hT, float* sa, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(false, B, T, H, D, chunk, in_dtype, r, w, k, v, a, b, h0, y, h_ckpt, hT, sa, workspace,
                      workspace_bytes, stream);
}

int wkv7_forward_sequential(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w,
                            const void* k, const void* v, const void* a, const void* b, const float* h0, float* y,
                            float* h_ckpt, float* hT, float* sa, void* stream) {
  return forward_impl(true, B, T, H, D, chunk, in_dtype, r, w, k, v, a, b, h0, y, h_ckpt, hT, sa, nullptr, 0,
                      stream);
}

int wkv7_forward_bf16_y(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w,
                        const void* k, const void* v, const void* a, const void* b, const float* h0, void* y,
                        float* h_ckpt, float* hT, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_sizes(B, T, H, D, chunk);
  if (st) return st;
  if ((st = check_dtype(in_dtype))) return st;
  if (T > 0) {
    if ((st = check_ptrs({r, w, k, v, a, b, y}, {h0, h_ckpt, hT}))) return st;
  } else if ((st = check_ptrs({}, {h0, hT}))) {
    return st;
  }
  if (chunk != 32) return WKV7_ERR_SHAPE;
  if (workspace == nullptr) return WKV7_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return WKV7_ERR_ALIGN;
  if (workspace_bytes < wkv7::forward_workspace_bytes(B, T, H, chunk)) return WKV7_ERR_WORKSPACE;
  wkv7::FwdArgs p;
  p.B = B; p.T = T; p.H = H; p.chunk = chunk; p.nchunks = wkv7_num_chunks(T, chunk);
  p.bf16 = in_dtype == WKV7_BF16;
  p.in = {r, w, k, v, a, b};
  p.h0 = h0; p.y = static_cast<float*>(y); p.h_ckpt = h_ckpt; p.hT = hT; p.sa = nullptr; p.y_bf16 = true;
  const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  if (T == 0) return record_cuda(wkv7::launch_forward(p, st_));  // hT = h0 (or zeros); y is empty
  return record_cuda(wkv7::launch_xop_forward(p, workspace, 0, st_));
}

int wkv7_forward_workspace_size(int B, int T, int H, int D, int chunk, size_t* bytes) {
  int st = check_sizes(B, T, H, D, chunk);
  if (st) return st;
  if (bytes == nullptr) return WKV7_ERR_ARG;
  *bytes = wkv7::forward_workspace_bytes(B, T, H, chunk);
  return WKV7_OK;
}

namespace {
// the argument checks and BwdArgs shared by wkv7_backward and wkv7_backward_from_forward
int backward_args(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w, const void* k,
                  const void* v, const void* a, const void* b, const float* h0, const float* h_ckpt,
                  const float* sa, const float* dy, const float* dhT, float* dr, float* dw, float* dk, float* dv,
                  float* da, float* db, float* dh0, wkv7::BwdArgs* p) {
  int st = check_sizes(B, T, H, D, chunk);
  if (st) return st;
  if ((st = check_dtype(in_dtype))) return st;
  if (T > 0) {
    if ((st = check_ptrs({r, w, k, v, a, b, h_ckpt, dy, dr, dw, dk, dv, da, db}, {h0, sa, dhT, dh0}))) return st;
  } else if ((st = check_ptrs({}, {h0, dhT, dh0}))) {
    return st;
  }
  p->B = B; p->T = T; p->H = H; p->chunk = chunk; p->nchunks = wkv7_num_chunks(T, chunk);
  p->bf16 = in_dtype == WKV7_BF16;
  p->in = {r, w, k, v, a, b};
  p->h0 = h0; p->h_ckpt = h_ckpt; p->sa = T > 0 ? sa : nullptr; p->dy = dy; p->dhT = dhT;
  p->dr = dr; p->dw = dw; p->dk = dk; p->dv = dv; p->da = da; p->db = db; p->dh0 = dh0;
  return WKV7_OK;
}
}  // namespace

int wkv7_backward(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w,
                  const void* k, const void* v, const void* a, const void* b, const float* h0,
                  const float* h_ckpt, const float* sa, const float* dy, const float* dhT, float* dr, float* dw, float* dk,
                  float* dv, float* da, float* db, float* dh0, void* workspace, size_t workspace_bytes,
                  void* stream) {
  wkv7::BwdArgs p;
  const int st = backward_args(B, T, H, D, chunk, in_dtype, r, w, k, v, a, b, h0, h_ckpt, sa, dy, dhT, dr, dw, dk,
                               dv, da, db, dh0, &p);
  if (st) return st;
  if (workspace != nullptr && (chunk == 32 || p.sa != nullptr)) {
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return WKV7_ERR_ALIGN;
    if (workspace_bytes < wkv7::backward_workspace_bytes(B, T, H, chunk)) return WKV7_ERR_WORKSPACE;
    const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
    return record_cuda(p.sa == nullptr ? wkv7::launch_backward_transition(p, workspace, false, st_)
                                       : wkv7::launch_backward_two_phase(p, workspace, st_));
  }
  return record_cuda(wkv7::launch_backward(p, static_cast<cudaStream_t>(stream)));
}

int wkv7_backward_from_forward(int B, int T, int H, int D, int chunk, int in_dtype, const void* r, const void* w,
                               const void* k, const void* v, const void* a, const void* b, const float* h0,
                               const float* h_ckpt, const float* dy, const float* dhT, float* dr, float* dw,
                               float* dk, float* dv, float* da, float* db, float* dh0, void* fwd_workspace,
                               size_t fwd_workspace_bytes, void* stream) {
  wkv7::BwdArgs p;
  const int st = backward_args(B, T, H, D, chunk, in_dtype, r, w, k, v, a, b, h0, h_ckpt, nullptr, dy, dhT, dr, dw,
                               dk, dv, da, db, dh0, &p);
  if (st) return st;
  if (chunk != 32) return WKV7_ERR_SHAPE;
  if (fwd_workspace == nullptr) return WKV7_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(fwd_workspace) & 255u) return WKV7_ERR_ALIGN;
  if (fwd_workspace_bytes < wkv7::forward_workspace_bytes(B, T, H, chunk)) return WKV7_ERR_WORKSPACE;
  return record_cuda(wkv7::launch_backward_transition(p, fwd_workspace, true, static_cast<cudaStream_t>(stream)));
}

int wkv7_backward_workspace_size(int B, int T, int H, int D, int chunk, size_t* bytes) {
  int st = check_sizes(B, T, H, D, chunk);
  if (st) return st;
  if (bytes == nullptr) return WKV7_ERR_ARG;
  *bytes = wkv7::backward_workspace_bytes(B, T, H, chunk);
  return WKV7_OK;
}

int wkv7_debug_status(unsigned* word) {
  if (word == nullptr) return WKV7_ERR_ARG;
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return record_cuda(err);
  int (*const readers[])(unsigned*) = {wkv7::debug_word_xop,   wkv7::debug_word_colmat, wkv7::debug_word_fwd,
                                       wkv7::debug_word_fwdc,  wkv7::debug_word_chain,  wkv7::debug_word_bwd,
                                       wkv7::debug_word_bwd2,  wkv7::debug_word_decode};
  unsigned all = 0;
  for (auto rd : readers) {
    unsigned v = 0;
    const int e = rd(&v);
    if (e != 0) return record_cuda(static_cast<cudaError_t>(e));
    all |= v;
  }
  *word = all;
  return WKV7_OK;
}

int wkv7_debug_enabled(void) {
#ifdef WKV7_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

int wkv7_decode(int B, int H, int D, int in_dtype, float* state, const void* r, const void* w, const void* k,
                const void* v, const void* a, const void* b, float* y, void* stream) {
  int st = check_sizes(B, 1, H, D, 1);
  if (st) return st;
  if ((st = check_dtype(in_dtype))) return st;
  if ((st = check_ptrs({state, r, w, k, v, a, b, y}, {}))) return st;
  wkv7::DecodeArgs p;
  p.B = B; p.H = H;
  p.bf16 = in_dtype == WKV7_BF16;
  p.in = {r, w, k, v, a, b};
  p.state = state; p.y = y;
  return record_cuda(wkv7::launch_decode(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
