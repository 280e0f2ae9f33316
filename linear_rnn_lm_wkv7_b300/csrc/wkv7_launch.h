// Internal launchers of the WKV7 kernels (host side).  The extern "C" entry points in
// wkv7_api.cu validate arguments and call these; nothing here checks arguments again.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace wkv7 {

struct TokenInputs {
  const void* r;
  const void* w;
  const void* k;
  const void* v;
  const void* a;
  const void* b;
};

struct FwdArgs {
  int B, T, H, chunk, nchunks;
  bool bf16;
  TokenInputs in;
  const float* h0;
  float* y;
  float* h_ckpt;
  float* hT;
  float* sa;  // (B,T,H,D) fp32 sa_t per row, or null
  bool y_bf16 = false;  // y holds bf16 values (the chunk-operator forward only)
};

struct BwdArgs {
  int B, T, H, chunk, nchunks;
  bool bf16;
  TokenInputs in;
  const float* h0;
  const float* h_ckpt;
  const float* sa;  // saved by the forward, or null (then recomputed per chunk)
  const float* dy;
  const float* dhT;
  float *dr, *dw, *dk, *dv, *da, *db;
  float* dh0;
};

struct DecodeArgs {
  int B, H;
  bool bf16;
  TokenInputs in;
  float* state;
  float* y;
};

// multiprocessor count of the current device (cached per device)
int num_sms();

// WKV7_OK for cudaSuccess; otherwise records the CUDA error text for wkv7_last_cuda_error()
// and returns WKV7_ERR_CUDA
int record_cuda_status(cudaError_t err);

// the forward: sub-chunks of 16 tokens on tensor cores when chunk is a multiple of 16, else token by token
cudaError_t launch_forward(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_forward_sequential(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_forward_chunked(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_backward(const BwdArgs& a, cudaStream_t stream);

// two-phase backward (needs the saved sa): workspace of backward_workspace_bytes() bytes,
// 256-byte aligned, holding dsa (B,T,H,D) and the state gradient at every chunk end (B,H,C,D,D)
size_t backward_workspace_bytes(int B, int T, int H, int chunk);
cudaError_t launch_backward_two_phase(const BwdArgs& a, void* workspace, cudaStream_t stream);
// phase 1 of the two-phase backward (the state-gradient walk writing dv, dsa, X at the chunk ends and
// dh0) by the 16-step sub-chunk kernel: chunk % 16 == 0, T >= 1
cudaError_t launch_gwalk_chunked(const BwdArgs& a, float* dsa_ws, float* xck_ws, cudaStream_t stream);
// the forward as a chain of 32-token transition products (chunk == 32; no saved sa), and the backward's
// state-gradient walk on the same kernel: dv, the state gradient X at every chunk end into xck_ws
// (B,H,C,D,D), dh0
cudaError_t launch_forward_transition(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_gwalk_transition(const BwdArgs& a, float* xck_ws, cudaStream_t stream);
// the chunk operators (wkv7_xop.cu): a workspace of xop_workspace_bytes() bytes, 256-byte aligned (a status
// word, then one operator block per (head, chunk): 68 KB in the forward's, 40 KB in a backward's own).
// The forward: operators, then the chain writing y, h_ckpt and hT.  The walk: operators (on the forward's
// workspace only E_c, by its own kernel, or, with whole-head chain CTAs, inside the chain from Q_c and dy),
// then the chain writing G (the gradient w.r.t. the state after each chunk from every later token) over
// the blocks (returned in ChunkEnds) and dh0.  rows = state rows per chain CTA (16, 32 or 64; 0 picks by
// the head count).
size_t xop_workspace_bytes(int B, int T, int H, bool forward);
cudaError_t launch_xop_forward(const FwdArgs& a, void* workspace, int rows, cudaStream_t stream);
// what the walk leaves per chunk c of head bh (at (bh * C + c) * stride floats from each pointer): G, one
// int of scratch for the column kernels, and (a walk on the forward's workspace; else null) the forward's
// M_ak, M_rb, M_rk and T (bf16 hi rows then lo rows of 40 elements, 5 KB each)
struct ChunkEnds {
  const float* g;
  int* flags;
  size_t stride;
  const unsigned char* mats;
};
// from_forward: the blocks already hold the forward's A_c and Q_c (the same inputs); only E_c is formed
cudaError_t launch_xop_walk(const BwdArgs& a, void* workspace, bool from_forward, int rows, ChunkEnds* ends,
                            cudaStream_t stream);
// the column gradients dr, dw, dk, dv, da, db of every 32-token chunk in matrix form, from G at the chunk
// ends, the checkpoints and the inputs (no saved sa); chunks with tiny decays token by token
cudaError_t launch_colgrad_matrix(const BwdArgs& a, const ChunkEnds& ends, cudaStream_t stream);
// the backward without a saved sa at chunk 32: operators (or, from_forward, only E_c), walk, matrix column
// gradients
cudaError_t launch_backward_transition(const BwdArgs& a, void* workspace, bool from_forward, cudaStream_t stream);
// bytes of the forward's workspace (the transition operands)
size_t forward_workspace_bytes(int B, int T, int H, int chunk);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// debug builds: each source file's device status word, read and cleared (release builds: 0)
int debug_word_xop(unsigned* out);
int debug_word_colmat(unsigned* out);
int debug_word_fwd(unsigned* out);
int debug_word_fwdc(unsigned* out);
int debug_word_chain(unsigned* out);
int debug_word_bwd(unsigned* out);
int debug_word_bwd2(unsigned* out);
int debug_word_decode(unsigned* out);

}  // namespace wkv7
