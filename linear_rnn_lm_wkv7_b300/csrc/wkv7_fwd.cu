// WKV7 forward on sm_103a: the per-token state recurrence with chunk checkpoints.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Forward listing), per head, row i of the fp32 state S:
//     sa_i = sum_j S_ij a_j;   S_ij <- S_ij w_j + v_i k_j + sa_i b_j;   y_i = sum_j S_ij r_j
// with a copy of S written after every `chunk` tokens.
//
// Mapping.  Rows of a head never interact in the forward, so a head is split into
// 64/ROWS row blocks, one CTA each (grid = B*H*64/ROWS).  Inside a CTA a row is held
// by L = 64/COLS consecutive lanes, COLS fp32 state values each, in registers for the
// whole sequence.  The two row sums per token (sa and y) are L-lane butterflies.
// The per-token column vectors w, k, a, b, r are shared by every row of the head: a
// tile of 32 tokens is staged into shared memory as fp32 (bf16 widened once per CTA),
// read back as broadcast float4s.  y goes through shared memory so it leaves as
// ROWS-float runs; checkpoints and hT leave straight from registers as float4s.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kTile = 32;  // tokens staged per shared-memory tile

template <int ROWS>
constexpr size_t fwd_smem_bytes() {
  return sizeof(float) * (5 * kTile * kD + 2 * kTile * ROWS);
}

template <typename Tin, int COLS, int ROWS>
__global__ void __launch_bounds__(ROWS*(kD / COLS))
fwd_kernel(int T, int H, int chunk, int nchunks,
           const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
           const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
           const float* __restrict__ h0, float* __restrict__ y, float* __restrict__ h_ckpt,
           float* __restrict__ hT) {
  constexpr int L = kD / COLS;   // lanes per row
  constexpr int NT = ROWS * L;   // threads per CTA
  constexpr int NRB = kD / ROWS; // row blocks per head
  static_assert(NT % 32 == 0 && 32 % L == 0, "a row group must sit inside one warp");

  extern __shared__ float4 smem4[];
  float* s_vec = reinterpret_cast<float*>(smem4);  // [5][kTile][kD]: w, k, a, b, r
  float* s_v = s_vec + 5 * kTile * kD;              // [kTile][ROWS]
  float* s_y = s_v + kTile * ROWS;                  // [kTile][ROWS]

  const int bh = blockIdx.x / NRB;
  const int rb = blockIdx.x - bh * NRB;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int g = tid % L;
  const int rl = tid / L;
  const int row = rb * ROWS + rl;
  const int c0 = g * COLS;
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;

  float S[COLS];
  if (h0 != nullptr) {
    const float4* p = reinterpret_cast<const float4*>(h0 + sbase + (size_t)row * kD + c0);
#pragma unroll
    for (int q = 0; q < COLS / 4; ++q) {
      const float4 x = __ldg(p + q);
      S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < COLS; ++c) S[c] = 0.f;
  }

  int to_ckpt = chunk;  // tokens left until the next checkpoint
  for (int t0 = 0; t0 < T; t0 += kTile) {
    const int nt = min(kTile, T - t0);
    __syncthreads();  // the previous tile's shared data is no longer read
    for (int e = tid; e < 5 * nt * 8; e += NT) {
      const int q = e / (nt * 8);
      const int rem = e - q * nt * 8;
      const int tt = rem >> 3;
      const int c8 = rem & 7;
      const Tin* src = q == 0 ? w : q == 1 ? k : q == 2 ? a : q == 3 ? b : r;
      float o[8];
      load8(src + base + (size_t)(t0 + tt) * tstride + c8 * 8, o);
      store8(s_vec + (q * kTile + tt) * kD + c8 * 8, o);
    }
    for (int e = tid; e < nt * ROWS; e += NT) {
      const int tt = e / ROWS;
      const int rr = e - tt * ROWS;
      s_v[tt * ROWS + rr] = to_f32(v[base + (size_t)(t0 + tt) * tstride + rb * ROWS + rr]);
    }
    __syncthreads();

    for (int tt = 0; tt < nt; ++tt) {
      const float4* pw = reinterpret_cast<const float4*>(s_vec + (0 * kTile + tt) * kD + c0);
      const float4* pk = reinterpret_cast<const float4*>(s_vec + (1 * kTile + tt) * kD + c0);
      const float4* pa = reinterpret_cast<const float4*>(s_vec + (2 * kTile + tt) * kD + c0);
      const float4* pb = reinterpret_cast<const float4*>(s_vec + (3 * kTile + tt) * kD + c0);
      const float4* pr = reinterpret_cast<const float4*>(s_vec + (4 * kTile + tt) * kD + c0);

      // sa = S a (this thread's columns, then the L-lane butterfly)
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < COLS / 4; ++q) {
        const float4 av = pa[q];
        part[0] = fmaf(S[4 * q], av.x, part[0]);
        part[1] = fmaf(S[4 * q + 1], av.y, part[1]);
        part[2] = fmaf(S[4 * q + 2], av.z, part[2]);
        part[3] = fmaf(S[4 * q + 3], av.w, part[3]);
      }
      float sa = (part[0] + part[1]) + (part[2] + part[3]);
#pragma unroll
      for (int m = 1; m < L; m <<= 1) sa += __shfl_xor_sync(0xffffffffu, sa, m);

      const float vi = s_v[tt * ROWS + rl];
      float yp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < COLS / 4; ++q) {
        const float4 wv = pw[q], kv = pk[q], bv = pb[q], rv = pr[q];
        S[4 * q] = fmaf(S[4 * q], wv.x, fmaf(vi, kv.x, sa * bv.x));
        S[4 * q + 1] = fmaf(S[4 * q + 1], wv.y, fmaf(vi, kv.y, sa * bv.y));
        S[4 * q + 2] = fmaf(S[4 * q + 2], wv.z, fmaf(vi, kv.z, sa * bv.z));
        S[4 * q + 3] = fmaf(S[4 * q + 3], wv.w, fmaf(vi, kv.w, sa * bv.w));
        yp[0] = fmaf(S[4 * q], rv.x, yp[0]);
        yp[1] = fmaf(S[4 * q + 1], rv.y, yp[1]);
        yp[2] = fmaf(S[4 * q + 2], rv.z, yp[2]);
        yp[3] = fmaf(S[4 * q + 3], rv.w, yp[3]);
      }
      float yi = (yp[0] + yp[1]) + (yp[2] + yp[3]);
#pragma unroll
      for (int m = 1; m < L; m <<= 1) yi += __shfl_xor_sync(0xffffffffu, yi, m);
      if (g == 0) s_y[tt * ROWS + rl] = yi;

      const int t = t0 + tt;
      if (--to_ckpt == 0 || t == T - 1) {
        to_ckpt = chunk;
        if (h_ckpt != nullptr) {
          float4* dst = reinterpret_cast<float4*>(
              h_ckpt + ((size_t)bh * nchunks + t / chunk) * kD * kD + (size_t)row * kD + c0);
#pragma unroll
          for (int q = 0; q < COLS / 4; ++q)
            dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < nt * ROWS; e += NT) {
      const int tt = e / ROWS;
      const int rr = e - tt * ROWS;
      y[base + (size_t)(t0 + tt) * tstride + rb * ROWS + rr] = s_y[tt * ROWS + rr];
    }
  }

  if (hT != nullptr) {
    float4* dst = reinterpret_cast<float4*>(hT + sbase + (size_t)row * kD + c0);
#pragma unroll
    for (int q = 0; q < COLS / 4; ++q)
      dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
  }
}

template <typename Tin>
cudaError_t launch_fwd_t(const FwdArgs& p, cudaStream_t stream) {
  constexpr int COLS = 16, ROWS = 16;
  constexpr int NT = ROWS * (kD / COLS);
  const size_t smem = fwd_smem_bytes<ROWS>();
  auto kern = fwd_kernel<Tin, COLS, ROWS>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * p.H * (kD / ROWS);
  kern<<<grid, NT, smem, stream>>>(p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r, (const Tin*)p.in.w,
                                   (const Tin*)p.in.k, (const Tin*)p.in.v, (const Tin*)p.in.a,
                                   (const Tin*)p.in.b, p.h0, p.y, p.h_ckpt, p.hT);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& p, cudaStream_t stream) {
  return p.bf16 ? launch_fwd_t<__nv_bfloat16>(p, stream) : launch_fwd_t<float>(p, stream);
}

}  // namespace wkv7
