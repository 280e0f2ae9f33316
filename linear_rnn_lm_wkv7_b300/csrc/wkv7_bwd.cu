// WKV7 checkpointed backward on sm_103a.
//
// Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Backward listing: chunks are walked in reverse starting from the
// exact checkpoints; inside a chunk the tokens are walked in reverse, the VJP gives
// dr, dw, dk, dv, da, db, and the previous state is rebuilt as (h - v k - sa b) / w.
// The listing does not say where sa comes from; here each chunk is first run forward
// from its start checkpoint (h0 for the first chunk), which yields every sa_t of the
// chunk and the chunk-end state, then walked in reverse.  Per token, in reverse, with
// G the gradient w.r.t. the state after the token:
//     G += dy r^T
//     dr = S'^T dy            (S' = state after the token)
//     S  = (S' - v k^T - sa b^T) diag(1/w)
//     dw_j = sum_i G_ij S_ij;  dk = G^T v;  db = G^T sa;  dv = G k;  dsa = G b
//     da = S^T dsa;  G <- G diag(w) + dsa a^T
//
// Mapping: one CTA per head (B*H CTAs); thread = RPT rows x 4 columns of the state
// and of G, in registers.  A warp holds 2 row groups x 16 column groups, so row sums
// (sa, dv, dsa) are 16-lane butterflies inside the warp.  Column sums (dr, dw, dk, db,
// da) are summed over the thread's rows in registers, over the two row groups of the
// warp by one shuffle, and over warps by shared-memory float atomics into the chunk's
// gradient tile, which is written to HBM as float4 runs when the chunk is done.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kMaxChunk = 32;

// shared-memory layout (floats)
constexpr int kColVecs = 6;  // w, 1/w, k, a, b, r
constexpr int kRowVecs = 2;  // v, dy
constexpr int kColGrads = 5; // dr, dw, dk, db, da
constexpr int kOffCol = 0;
constexpr int kOffRow = kOffCol + kColVecs * kMaxChunk * kD;
constexpr int kOffSa = kOffRow + kRowVecs * kMaxChunk * kD;
constexpr int kOffGcol = kOffSa + kMaxChunk * kD;
constexpr int kOffDv = kOffGcol + kColGrads * kMaxChunk * kD;
constexpr int kSmemFloats = kOffDv + kMaxChunk * kD;
constexpr size_t kBwdSmemBytes = sizeof(float) * kSmemFloats;

enum { CW = 0, CWINV = 1, CK = 2, CA = 3, CB = 4, CR = 5 };

template <typename Tin, int RPT>
__global__ void __launch_bounds__(16 * (kD / RPT))
bwd_kernel(int T, int H, int chunk, int nchunks,
           const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
           const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
           const float* __restrict__ h0, const float* __restrict__ h_ckpt,
           const float* __restrict__ dy, const float* __restrict__ dhT,
           float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
           float* __restrict__ dv, float* __restrict__ da, float* __restrict__ db,
           float* __restrict__ dh0) {
  constexpr int NRG = kD / RPT;  // row groups
  constexpr int NT = 16 * NRG;   // threads
  extern __shared__ float4 smem4[];
  float* sm = reinterpret_cast<float*>(smem4);
  float* s_col = sm + kOffCol;   // [6][kMaxChunk][kD]
  float* s_row = sm + kOffRow;   // [2][kMaxChunk][kD]: v, dy
  float* s_sa = sm + kOffSa;     // [kMaxChunk][kD]
  float* s_gcol = sm + kOffGcol; // [5][kMaxChunk][kD]
  float* s_dv = sm + kOffDv;     // [kMaxChunk][kD]

  const int bh = blockIdx.x;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int cg = lane & 15;
  const int rg = (tid >> 5) * 2 + (lane >> 4);
  const int i0 = rg * RPT;
  const int j0 = cg * 4;
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;

  float h[RPT][4], G[RPT][4];
  if (dhT != nullptr) {
#pragma unroll
    for (int ri = 0; ri < RPT; ++ri) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(dhT + sbase + (size_t)(i0 + ri) * kD + j0));
      G[ri][0] = x.x; G[ri][1] = x.y; G[ri][2] = x.z; G[ri][3] = x.w;
    }
  } else {
#pragma unroll
    for (int ri = 0; ri < RPT; ++ri)
#pragma unroll
      for (int c = 0; c < 4; ++c) G[ri][c] = 0.f;
  }

  for (int ci = nchunks - 1; ci >= 0; --ci) {
    const int t0 = ci * chunk;
    const int n = min(chunk, T - t0);
    __syncthreads();  // the previous chunk's tiles have been written out

    // ---- stage the chunk's inputs (fp32) and clear the column-gradient tile
    for (int e = tid; e < 5 * n * 8; e += NT) {
      const int q = e / (n * 8);
      const int rem = e - q * n * 8;
      const int tt = rem >> 3;
      const int c8 = rem & 7;
      const size_t off = base + (size_t)(t0 + tt) * tstride + c8 * 8;
      float o[8];
      if (q == 0) {
        load8(w + off, o);
        store8(s_col + (CW * kMaxChunk + tt) * kD + c8 * 8, o);
#pragma unroll
        for (int u = 0; u < 8; ++u) o[u] = 1.0f / o[u];
        store8(s_col + (CWINV * kMaxChunk + tt) * kD + c8 * 8, o);
      } else {
        const Tin* src = q == 1 ? k : q == 2 ? a : q == 3 ? b : r;
        const int slot = q == 1 ? CK : q == 2 ? CA : q == 3 ? CB : CR;
        load8(src + off, o);
        store8(s_col + (slot * kMaxChunk + tt) * kD + c8 * 8, o);
      }
    }
    for (int e = tid; e < 2 * n * 8; e += NT) {
      const int q = e / (n * 8);
      const int rem = e - q * n * 8;
      const int tt = rem >> 3;
      const int c8 = rem & 7;
      const size_t off = base + (size_t)(t0 + tt) * tstride + c8 * 8;
      float o[8];
      if (q == 0) load8(v + off, o);
      else load8(dy + off, o);
      store8(s_row + (q * kMaxChunk + tt) * kD + c8 * 8, o);
    }
    for (int e = tid; e < kColGrads * kMaxChunk * kD / 4; e += NT)
      reinterpret_cast<float4*>(s_gcol)[e] = make_float4(0.f, 0.f, 0.f, 0.f);

    // ---- chunk-start state
    const float* src = ci == 0 ? (h0 != nullptr ? h0 + sbase : nullptr)
                                : h_ckpt + ((size_t)bh * nchunks + (ci - 1)) * kD * kD;
    if (src != nullptr) {
#pragma unroll
      for (int ri = 0; ri < RPT; ++ri) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src + (size_t)(i0 + ri) * kD + j0));
        h[ri][0] = x.x; h[ri][1] = x.y; h[ri][2] = x.z; h[ri][3] = x.w;
      }
    } else {
#pragma unroll
      for (int ri = 0; ri < RPT; ++ri)
#pragma unroll
        for (int c = 0; c < 4; ++c) h[ri][c] = 0.f;
    }
    __syncthreads();

    // ---- recompute the chunk forward, recording sa_t
    for (int tt = 0; tt < n; ++tt) {
      const float4 av = *reinterpret_cast<const float4*>(s_col + (CA * kMaxChunk + tt) * kD + j0);
      const float4 wv = *reinterpret_cast<const float4*>(s_col + (CW * kMaxChunk + tt) * kD + j0);
      const float4 kv = *reinterpret_cast<const float4*>(s_col + (CK * kMaxChunk + tt) * kD + j0);
      const float4 bv = *reinterpret_cast<const float4*>(s_col + (CB * kMaxChunk + tt) * kD + j0);
      float sa[RPT];
#pragma unroll
      for (int ri = 0; ri < RPT; ++ri)
        sa[ri] = fmaf(h[ri][0], av.x, h[ri][1] * av.y) + fmaf(h[ri][2], av.z, h[ri][3] * av.w);
#pragma unroll
      for (int m = 1; m < 16; m <<= 1)
#pragma unroll
        for (int ri = 0; ri < RPT; ++ri) sa[ri] += __shfl_xor_sync(0xffffffffu, sa[ri], m);
      if (cg == 0) {
#pragma unroll
        for (int ri = 0; ri < RPT; ++ri) s_sa[tt * kD + i0 + ri] = sa[ri];
      }
#pragma unroll
      for (int ri = 0; ri < RPT; ++ri) {
        const float vi = s_row[tt * kD + i0 + ri];
        h[ri][0] = fmaf(h[ri][0], wv.x, fmaf(vi, kv.x, sa[ri] * bv.x));
        h[ri][1] = fmaf(h[ri][1], wv.y, fmaf(vi, kv.y, sa[ri] * bv.y));
        h[ri][2] = fmaf(h[ri][2], wv.z, fmaf(vi, kv.z, sa[ri] * bv.z));
        h[ri][3] = fmaf(h[ri][3], wv.w, fmaf(vi, kv.w, sa[ri] * bv.w));
      }
    }
    __syncwarp();  // s_sa rows of this warp are written by this warp

    // ---- reverse walk
    for (int tt = n - 1; tt >= 0; --tt) {
      const float4 rv = *reinterpret_cast<const float4*>(s_col + (CR * kMaxChunk + tt) * kD + j0);
      const float4 wv = *reinterpret_cast<const float4*>(s_col + (CW * kMaxChunk + tt) * kD + j0);
      const float4 wi = *reinterpret_cast<const float4*>(s_col + (CWINV * kMaxChunk + tt) * kD + j0);
      const float4 kv = *reinterpret_cast<const float4*>(s_col + (CK * kMaxChunk + tt) * kD + j0);
      const float4 av = *reinterpret_cast<const float4*>(s_col + (CA * kMaxChunk + tt) * kD + j0);
      const float4 bv = *reinterpret_cast<const float4*>(s_col + (CB * kMaxChunk + tt) * kD + j0);
      const float rr[4] = {rv.x, rv.y, rv.z, rv.w};
      const float ww[4] = {wv.x, wv.y, wv.z, wv.w};
      const float wiv[4] = {wi.x, wi.y, wi.z, wi.w};
      const float kk[4] = {kv.x, kv.y, kv.z, kv.w};
      const float aa[4] = {av.x, av.y, av.z, av.w};
      const float bb[4] = {bv.x, bv.y, bv.z, bv.w};

      float p_dr[4], p_dw[4], p_dk[4], p_db[4], p_da[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) p_dr[c] = p_dw[c] = p_dk[c] = p_db[c] = p_da[c] = 0.f;
      float p_dv[RPT], p_dsa[RPT];

#pragma unroll
      for (int ri = 0; ri < RPT; ++ri) {
        const float vi = s_row[tt * kD + i0 + ri];
        const float dyi = s_row[(kMaxChunk + tt) * kD + i0 + ri];
        const float sai = s_sa[tt * kD + i0 + ri];
        float dv_acc = 0.f, dsa_acc = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float g = fmaf(dyi, rr[c], G[ri][c]);
          G[ri][c] = g;
          p_dr[c] = fmaf(dyi, h[ri][c], p_dr[c]);
          const float s = fmaf(-sai, bb[c], fmaf(-vi, kk[c], h[ri][c])) * wiv[c];
          h[ri][c] = s;
          p_dw[c] = fmaf(g, s, p_dw[c]);
          p_dk[c] = fmaf(g, vi, p_dk[c]);
          p_db[c] = fmaf(g, sai, p_db[c]);
          dv_acc = fmaf(g, kk[c], dv_acc);
          dsa_acc = fmaf(g, bb[c], dsa_acc);
        }
        p_dv[ri] = dv_acc;
        p_dsa[ri] = dsa_acc;
      }
#pragma unroll
      for (int m = 1; m < 16; m <<= 1)
#pragma unroll
        for (int ri = 0; ri < RPT; ++ri) {
          p_dsa[ri] += __shfl_xor_sync(0xffffffffu, p_dsa[ri], m);
          p_dv[ri] += __shfl_xor_sync(0xffffffffu, p_dv[ri], m);
        }
#pragma unroll
      for (int ri = 0; ri < RPT; ++ri) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          p_da[c] = fmaf(p_dsa[ri], h[ri][c], p_da[c]);
          G[ri][c] = fmaf(G[ri][c], ww[c], p_dsa[ri] * aa[c]);
        }
      }
      if (cg == 0) {
#pragma unroll
        for (int ri = 0; ri < RPT; ++ri) s_dv[tt * kD + i0 + ri] = p_dv[ri];
      }
      // column sums: the two row groups of this warp, then all warps through shared atomics
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        p_dr[c] += __shfl_xor_sync(0xffffffffu, p_dr[c], 16);
        p_dw[c] += __shfl_xor_sync(0xffffffffu, p_dw[c], 16);
        p_dk[c] += __shfl_xor_sync(0xffffffffu, p_dk[c], 16);
        p_db[c] += __shfl_xor_sync(0xffffffffu, p_db[c], 16);
        p_da[c] += __shfl_xor_sync(0xffffffffu, p_da[c], 16);
      }
      float* gt = s_gcol + tt * kD + j0;
      constexpr int GS = kMaxChunk * kD;  // stride between gradient kinds
      if ((lane >> 4) == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          atomicAdd(gt + 0 * GS + c, p_dr[c]);
          atomicAdd(gt + 1 * GS + c, p_dw[c]);
        }
        atomicAdd(gt + 2 * GS + 0, p_dk[0]);
        atomicAdd(gt + 2 * GS + 1, p_dk[1]);
      } else {
        atomicAdd(gt + 2 * GS + 2, p_dk[2]);
        atomicAdd(gt + 2 * GS + 3, p_dk[3]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          atomicAdd(gt + 3 * GS + c, p_db[c]);
          atomicAdd(gt + 4 * GS + c, p_da[c]);
        }
      }
    }
    __syncthreads();

    // ---- write the chunk's gradients (dr, dw, dk, db, da from the tile; dv)
    for (int e = tid; e < 6 * n * (kD / 4); e += NT) {
      const int q = e / (n * (kD / 4));
      const int rem = e - q * n * (kD / 4);
      const int tt = rem / (kD / 4);
      const int c4 = rem - tt * (kD / 4);
      const float* srcp = q < 5 ? s_gcol + (q * kMaxChunk + tt) * kD : s_dv + tt * kD;
      float* dst = q == 0 ? dr : q == 1 ? dw : q == 2 ? dk : q == 3 ? db : q == 4 ? da : dv;
      reinterpret_cast<float4*>(dst + base + (size_t)(t0 + tt) * tstride)[c4] =
          reinterpret_cast<const float4*>(srcp)[c4];
    }
  }

  if (dh0 != nullptr) {
#pragma unroll
    for (int ri = 0; ri < RPT; ++ri)
      *reinterpret_cast<float4*>(dh0 + sbase + (size_t)(i0 + ri) * kD + j0) =
          make_float4(G[ri][0], G[ri][1], G[ri][2], G[ri][3]);
  }
}

template <typename Tin>
cudaError_t launch_bwd_t(const BwdArgs& p, cudaStream_t stream) {
  constexpr int RPT = 4;
  constexpr int NT = 16 * (kD / RPT);
  auto kern = bwd_kernel<Tin, RPT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdSmemBytes);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * p.H;
  kern<<<grid, NT, kBwdSmemBytes, stream>>>(p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r,
                                            (const Tin*)p.in.w, (const Tin*)p.in.k, (const Tin*)p.in.v,
                                            (const Tin*)p.in.a, (const Tin*)p.in.b, p.h0, p.h_ckpt, p.dy,
                                            p.dhT, p.dr, p.dw, p.dk, p.dv, p.da, p.db, p.dh0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdArgs& p, cudaStream_t stream) {
  return p.bf16 ? launch_bwd_t<__nv_bfloat16>(p, stream) : launch_bwd_t<float>(p, stream);
}

}  // namespace wkv7
