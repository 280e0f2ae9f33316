// WKV7 single-token decode on sm_103a: the state of every (sequence, head) is read,
// advanced by one token and written back in place.
//
// The update is the forward recurrence with T = 1 ("RWKV-7 Pretraining on Apple Silicon
// (MLX)", section "Metal kernel architecture", Forward listing).  The workload it serves
// is the 7B model's per-token step: 32 layers x 64 heads of 64 x 64 fp32 state values
// per sequence ("RWKV-7 最新、最全的动态"), i.e. a pure stream over the state, ~1 FLOP
// per byte, bound by HBM bandwidth.
//
// Mapping: one CTA of 256 threads per (sequence, head).  Thread = 4 consecutive columns
// (one float4) of 4 rows (rows rs, rs+16, rs+32, rs+48); the 16 lanes sharing a row are
// one half-warp, so sa and y are 16-lane butterflies.  All four state float4s are loaded
// before any arithmetic (memory-level parallelism); loads and stores use the streaming
// cache hints because every state byte is touched exactly once.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

template <typename Tin>
__global__ void __launch_bounds__(256)
decode_kernel(float* __restrict__ state, const Tin* __restrict__ r, const Tin* __restrict__ w,
              const Tin* __restrict__ k, const Tin* __restrict__ v, const Tin* __restrict__ a,
              const Tin* __restrict__ b, float* __restrict__ y) {
  const size_t bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int cg = tid & 15;
  const int rs = tid >> 4;
  const int j0 = cg * 4;
  const size_t vb = bh * kD;
  float4* st = reinterpret_cast<float4*>(state + bh * kD * kD);

  float4 S[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) S[m] = __ldcs(st + (rs + 16 * m) * (kD / 4) + cg);
  const float4 wv = load4(w + vb + j0);
  const float4 kv = load4(k + vb + j0);
  const float4 av = load4(a + vb + j0);
  const float4 bv = load4(b + vb + j0);
  const float4 rv = load4(r + vb + j0);
  float vi[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) vi[m] = to_f32(v[vb + rs + 16 * m]);

  float sa[4];
#pragma unroll
  for (int m = 0; m < 4; ++m)
    sa[m] = fmaf(S[m].x, av.x, S[m].y * av.y) + fmaf(S[m].z, av.z, S[m].w * av.w);
#pragma unroll
  for (int s = 1; s < 16; s <<= 1)
#pragma unroll
    for (int m = 0; m < 4; ++m) sa[m] += __shfl_xor_sync(0xffffffffu, sa[m], s);

  float yp[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    S[m].x = fmaf(S[m].x, wv.x, fmaf(vi[m], kv.x, sa[m] * bv.x));
    S[m].y = fmaf(S[m].y, wv.y, fmaf(vi[m], kv.y, sa[m] * bv.y));
    S[m].z = fmaf(S[m].z, wv.z, fmaf(vi[m], kv.z, sa[m] * bv.z));
    S[m].w = fmaf(S[m].w, wv.w, fmaf(vi[m], kv.w, sa[m] * bv.w));
    __stcs(st + (rs + 16 * m) * (kD / 4) + cg, S[m]);
    yp[m] = fmaf(S[m].x, rv.x, S[m].y * rv.y) + fmaf(S[m].z, rv.z, S[m].w * rv.w);
  }
#pragma unroll
  for (int s = 1; s < 16; s <<= 1)
#pragma unroll
    for (int m = 0; m < 4; ++m) yp[m] += __shfl_xor_sync(0xffffffffu, yp[m], s);
  if (cg == 0) {
#pragma unroll
    for (int m = 0; m < 4; ++m) y[vb + rs + 16 * m] = yp[m];
  }
}

template <typename Tin>
cudaError_t launch_decode_t(const DecodeArgs& p, cudaStream_t stream) {
  const unsigned grid = (unsigned)p.B * p.H;
  decode_kernel<Tin><<<grid, 256, 0, stream>>>(p.state, (const Tin*)p.in.r, (const Tin*)p.in.w,
                                              (const Tin*)p.in.k, (const Tin*)p.in.v, (const Tin*)p.in.a,
                                              (const Tin*)p.in.b, p.y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& p, cudaStream_t stream) {
  return p.bf16 ? launch_decode_t<__nv_bfloat16>(p, stream) : launch_decode_t<float>(p, stream);
}

WKV7_DEBUG_READER(debug_word_decode)

}  // namespace wkv7
