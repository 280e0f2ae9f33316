// WKV7 forward on sm_103a: the per-token state recurrence with chunk checkpoints.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Forward listing), per head, row i of the fp32 state S:
//     sa_i = sum_j S_ij a_j;   S_ij <- S_ij w_j + v_i k_j + sa_i b_j;   y_i = sum_j S_ij r_j
// with a copy of S written after every `chunk` tokens.
//
// Mapping.  Rows of a head never interact in the forward, so a head is split into
// 64/ROWS row blocks, one CTA each.  Thread = RPT rows x 4 columns of the state, in
// registers for the whole sequence; the 16 lanes of a row group own column blocks 4g
// (g = lane % 16), so a half-warp reads one contiguous 256-byte row of each per-token
// vector without bank conflicts, and every value a lane loads feeds RPT rows.  (A
// 128-bit shared load whose lanes hit distinct addresses costs 4 wavefronts; loads
// feeding one row per lane made the shared-memory pipe the limit.)
//
// One-token lookahead.  The serial chain of the recurrence is sa_t -> S_t -> sa_{t+1}.
// Since S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T,
//     sa_{t+1} = S_{t-1} (w_t o a_{t+1}) + v_t (k_t . a_{t+1}) + sa_t (b_t . a_{t+1}),
// so the row sum that produces sa_{t+1} reads the state *before* token t and runs in
// parallel with token t's update.  c_t = w_t o a_{t+1} and the scalars k_t . a_{t+1},
// b_t . a_{t+1} do not depend on the state; they are formed once per CTA per tile.
// That row sum is a 4-level butterfly (shortest dependent chain); y, off the chain,
// uses the cheaper reduce-scatter.
//
// Staging.  Tiles of 32 tokens of w, k, a, b, r (+ one token of a ahead) and the CTA's
// slice of v are copied to shared memory with cp.async, double-buffered so the copy of
// tile i+1 overlaps the recurrence over tile i, then widened to fp32 once per CTA.  y
// leaves through shared memory as ROWS-float runs; checkpoints and hT leave from
// registers as float4s.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kTile = 32;          // tokens per staged tile
constexpr int kTileA = kTile + 1;  // rows of a per tile (one token of lookahead)

template <typename Tin, int ROWS>
struct FwdLayout {
  // raw (input dtype) buffer, double-buffered: W, K, B, R [kTile][64], A [kTileA][64], V [kTile][ROWS]
  static constexpr int kRawElems = 4 * kTile * kD + kTileA * kD + kTile * ROWS;
  static constexpr size_t kRawBytes = ((kRawElems * sizeof(Tin)) + 15) / 16 * 16;
  // fp32 tiles: W, K, B, R, C [kTile][64]; KA, BA [kTile]; V, Y, SA [kTile][ROWS]
  static constexpr int kF32 = 5 * kTile * kD + 2 * kTile + 3 * kTile * ROWS;
  static constexpr size_t kBytes = 2 * kRawBytes + sizeof(float) * kF32;
};

// Issue the cp.async copies of tile [t0, t0 + nt): W K B R rows, A rows t0 .. t0+na-1, V slice.
template <typename Tin, int ROWS, int NT>
__device__ __forceinline__ void issue_tile(Tin* raw, int t0, int nt, int na, size_t base, size_t tstride,
                                           int vcol, const Tin* __restrict__ w, const Tin* __restrict__ k,
                                           const Tin* __restrict__ b, const Tin* __restrict__ r,
                                           const Tin* __restrict__ a, const Tin* __restrict__ v) {
  constexpr int CPR = kD * (int)sizeof(Tin) / 16;  // 16-byte pieces per 64-wide row
  constexpr int EPC = 16 / (int)sizeof(Tin);       // elements per piece
  const Tin* srcs[4] = {w, k, b, r};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    Tin* dst = raw + q * kTile * kD;
    for (int e = threadIdx.x; e < nt * CPR; e += NT) {
      const int tt = e / CPR, pc = e % CPR;
      cp_async16(dst + tt * kD + pc * EPC, srcs[q] + base + (size_t)(t0 + tt) * tstride + pc * EPC);
    }
  }
  {
    Tin* dst = raw + 4 * kTile * kD;
    for (int e = threadIdx.x; e < na * CPR; e += NT) {
      const int tt = e / CPR, pc = e % CPR;
      cp_async16(dst + tt * kD + pc * EPC, a + base + (size_t)(t0 + tt) * tstride + pc * EPC);
    }
  }
  {
    constexpr int VPR = ROWS * (int)sizeof(Tin) / 16;  // pieces per token of the CTA's v slice
    Tin* dst = raw + 4 * kTile * kD + kTileA * kD;
    for (int e = threadIdx.x; e < nt * VPR; e += NT) {
      const int tt = e / VPR, pc = e % VPR;
      cp_async16(dst + tt * ROWS + pc * EPC, v + base + (size_t)(t0 + tt) * tstride + vcol + pc * EPC);
    }
  }
}

template <typename Tin, int ROWS, int RPT>
__global__ void __launch_bounds__(ROWS * 16 / RPT, 1)
fwd_kernel(int T, int H, int chunk, int nchunks,
           const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
           const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
           const float* __restrict__ h0, float* __restrict__ y, float* __restrict__ h_ckpt,
           float* __restrict__ hT, float* __restrict__ sa_out) {
  constexpr int NT = ROWS * 16 / RPT;
  constexpr int NW = NT / 32;
  constexpr int NRB = kD / ROWS;
  using Lay = FwdLayout<Tin, ROWS>;
  static_assert(RPT == 2 || RPT == 4, "2 or 4 rows per thread");
  static_assert(ROWS * (int)sizeof(Tin) % 16 == 0, "v slice must be whole 16-byte pieces");
  static_assert(ROWS % (2 * RPT) == 0, "a warp holds two row groups");

  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  Tin* raw0 = reinterpret_cast<Tin*>(sm);
  Tin* raw1 = reinterpret_cast<Tin*>(sm + Lay::kRawBytes);
  float* fW = reinterpret_cast<float*>(sm + 2 * Lay::kRawBytes);
  float* fK = fW + kTile * kD;
  float* fB = fK + kTile * kD;
  float* fR = fB + kTile * kD;
  float* fC = fR + kTile * kD;
  float* fKA = fC + kTile * kD;
  float* fBA = fKA + kTile;
  float* fV = fBA + kTile;
  float* fY = fV + kTile * ROWS;
  float* fSA = fY + kTile * ROWS;

  const int bh = blockIdx.x / NRB;
  const int rb = blockIdx.x - bh * NRB;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int l16 = tid & 15;
  const int rloc = RPT * (tid >> 4);  // first local row of this thread
  const int row0 = rb * ROWS + rloc;  // first row within the head
  const int j0 = 4 * l16;             // first column
  const int qrow = rs16_row<RPT>(l16);  // row whose y this lane ends up holding
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;
  const int ntiles = (T + kTile - 1) / kTile;

  // state: S[i] = row row0+i, columns j0..j0+3 as two float2
  float2 S[RPT][2];
  if (h0 != nullptr) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(h0 + sbase + (size_t)(row0 + i) * kD + j0));
      S[i][0] = lo2(x);
      S[i][1] = hi2(x);
    }
  } else {
#pragma unroll
    for (int i = 0; i < RPT; ++i) S[i][0] = S[i][1] = make_float2(0.f, 0.f);
  }

  if (ntiles > 0) {
    issue_tile<Tin, ROWS, NT>(raw0, 0, min(kTile, T), min(kTileA, T), base, tstride, rb * ROWS, w, k, b, r, a, v);
    cp_async_commit();
  }

  // sa for token 0 (the state before it is h0)
  float sa[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) sa[i] = 0.f;
  if (T > 0) {
    dot_rows<RPT>(S, load4(a + base + j0), sa);
    butterfly16<RPT>(sa);
  }

  int to_ckpt = chunk;
  for (int it = 0; it < ntiles; ++it) {
    const int t0 = it * kTile;
    const int nt = min(kTile, T - t0);
    Tin* raw = (it & 1) ? raw1 : raw0;
    if (it + 1 < ntiles) {
      const int t1 = t0 + kTile;
      issue_tile<Tin, ROWS, NT>((it & 1) ? raw0 : raw1, t1, min(kTile, T - t1), min(kTileA, T - t1), base,
                                tstride, rb * ROWS, w, k, b, r, a, v);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile `it` is in shared memory; the previous tile's fp32 data is consumed

    // ---- widen to fp32 and form the lookahead terms: 4 tokens per warp pass, 8 lanes per token
    {
      const Tin* rW = raw;
      const Tin* rK = raw + kTile * kD;
      const Tin* rB = raw + 2 * kTile * kD;
      const Tin* rR = raw + 3 * kTile * kD;
      const Tin* rA = raw + 4 * kTile * kD;
      for (int tg = warp * 4; tg < nt; tg += NW * 4) {
        const int tt = tg + (lane >> 3);
        const int c8 = (lane & 7) * 8;
        float ka = 0.f, ba = 0.f;
        if (tt < nt) {
          float ww[8], kk[8], bb[8], rr[8], an[8];
          raw8(rW + tt * kD + c8, ww);
          raw8(rK + tt * kD + c8, kk);
          raw8(rB + tt * kD + c8, bb);
          raw8(rR + tt * kD + c8, rr);
          if (t0 + tt + 1 < T) {
            raw8(rA + (tt + 1) * kD + c8, an);
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) an[u] = 0.f;
          }
          float cc[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            cc[u] = ww[u] * an[u];
            ka = fmaf(kk[u], an[u], ka);
            ba = fmaf(bb[u], an[u], ba);
          }
          store8(fW + tt * kD + c8, ww);
          store8(fK + tt * kD + c8, kk);
          store8(fB + tt * kD + c8, bb);
          store8(fR + tt * kD + c8, rr);
          store8(fC + tt * kD + c8, cc);
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
          ka += __shfl_xor_sync(0xffffffffu, ka, m);
          ba += __shfl_xor_sync(0xffffffffu, ba, m);
        }
        if (tt < nt && (lane & 7) == 0) {
          fKA[tt] = ka;
          fBA[tt] = ba;
        }
      }
      const Tin* rV = raw + 4 * kTile * kD + kTileA * kD;
      for (int e = tid; e < nt * ROWS; e += NT) fV[e] = to_f32(rV[e]);
    }
    __syncthreads();

    // ---- the recurrence over the tile (unrolled so consecutive tokens' shuffle chains overlap)
#pragma unroll 2
    for (int tt = 0; tt < nt; ++tt) {
      const float4 c4 = *reinterpret_cast<const float4*>(fC + tt * kD + j0);
      const float4 w4 = *reinterpret_cast<const float4*>(fW + tt * kD + j0);
      const float4 k4 = *reinterpret_cast<const float4*>(fK + tt * kD + j0);
      const float4 b4 = *reinterpret_cast<const float4*>(fB + tt * kD + j0);
      const float4 r4 = *reinterpret_cast<const float4*>(fR + tt * kD + j0);
      const float ka = fKA[tt], ba = fBA[tt];
      float vv[RPT];
      if constexpr (RPT == 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(fV + tt * ROWS + rloc);
        vv[0] = v4.x, vv[1] = v4.y, vv[2] = v4.z, vv[3] = v4.w;
        if (sa_out != nullptr && l16 == 0)
          *reinterpret_cast<float4*>(fSA + tt * ROWS + rloc) = make_float4(sa[0], sa[1], sa[2], sa[3]);
      } else {
        const float2 v2 = *reinterpret_cast<const float2*>(fV + tt * ROWS + rloc);
        vv[0] = v2.x, vv[1] = v2.y;
        if (sa_out != nullptr && l16 == 0) *reinterpret_cast<float2*>(fSA + tt * ROWS + rloc) = make_float2(sa[0], sa[1]);
      }

      // lookahead row sums on the state before this token
      float P[RPT];
      dot_rows<RPT>(S, c4, P);
      butterfly16<RPT>(P);

      // S <- S w + v k + sa b
#pragma unroll
      for (int i = 0; i < RPT; ++i) {
        const float2 s2 = make_float2(sa[i], sa[i]);
        const float2 v2 = make_float2(vv[i], vv[i]);
        const float2 u0 = __ffma2_rn(v2, lo2(k4), __fmul2_rn(s2, lo2(b4)));
        const float2 u1 = __ffma2_rn(v2, hi2(k4), __fmul2_rn(s2, hi2(b4)));
        S[i][0] = __ffma2_rn(S[i][0], lo2(w4), u0);
        S[i][1] = __ffma2_rn(S[i][1], hi2(w4), u1);
      }
      // y = S r
      float yp[RPT];
      dot_rows<RPT>(S, r4, yp);
      const float yq = rs16<RPT>(yp, l16);
      if ((l16 & (16 / RPT - 1)) == 0) fY[tt * ROWS + rloc + qrow] = yq;
#pragma unroll
      for (int i = 0; i < RPT; ++i) sa[i] = fmaf(sa[i], ba, fmaf(vv[i], ka, P[i]));

      const int t = t0 + tt;
      if (--to_ckpt == 0 || t == T - 1) {
        to_ckpt = chunk;
        if (h_ckpt != nullptr) {
          float* dst = h_ckpt + ((size_t)bh * nchunks + t / chunk) * kD * kD + (size_t)row0 * kD + j0;
#pragma unroll
          for (int i = 0; i < RPT; ++i)
            *reinterpret_cast<float4*>(dst + i * kD) = make_float4(S[i][0].x, S[i][0].y, S[i][1].x, S[i][1].y);
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < nt * ROWS; e += NT) {
      const int tt = e / ROWS;
      const int rr = e % ROWS;
      y[base + (size_t)(t0 + tt) * tstride + rb * ROWS + rr] = fY[e];
      if (sa_out != nullptr) sa_out[base + (size_t)(t0 + tt) * tstride + rb * ROWS + rr] = fSA[e];
    }
  }

  if (hT != nullptr) {
#pragma unroll
    for (int i = 0; i < RPT; ++i)
      *reinterpret_cast<float4*>(hT + sbase + (size_t)(row0 + i) * kD + j0) =
          make_float4(S[i][0].x, S[i][0].y, S[i][1].x, S[i][1].y);
  }
}

template <typename Tin, int ROWS, int RPT>
cudaError_t launch_fwd_cfg(const FwdArgs& p, cudaStream_t stream) {
  constexpr int NT = ROWS * 16 / RPT;
  const size_t smem = FwdLayout<Tin, ROWS>::kBytes;
  auto kern = fwd_kernel<Tin, ROWS, RPT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)p.B * p.H * (kD / ROWS);
  kern<<<grid, NT, smem, stream>>>(p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r, (const Tin*)p.in.w,
                                   (const Tin*)p.in.k, (const Tin*)p.in.v, (const Tin*)p.in.a,
                                   (const Tin*)p.in.b, p.h0, p.y, p.h_ckpt, p.hT, p.sa);
  return cudaGetLastError();
}

}  // namespace

template <typename Tin>
cudaError_t launch_fwd_t(const FwdArgs& p, cudaStream_t stream) {
  // Measured at 32 rows per CTA: when every row block has an SM of its own, 2 rows per thread (8 warps)
  // beat 4 rows per thread (4 warps) by 4-5%; past one wave the smaller per-thread tile loses (13%
  // slower at 256 row blocks), its extra shuffles and loads no longer hidden.
  if ((long long)p.B * p.H * (kD / 32) <= num_sms()) return launch_fwd_cfg<Tin, 32, 2>(p, stream);
  return launch_fwd_cfg<Tin, 32, 4>(p, stream);
}

cudaError_t launch_forward_sequential(const FwdArgs& p, cudaStream_t stream) {
  return p.bf16 ? launch_fwd_t<__nv_bfloat16>(p, stream) : launch_fwd_t<float>(p, stream);
}

cudaError_t launch_forward(const FwdArgs& p, cudaStream_t stream) {
  // 32-token chunks without a saved sa: the chain of transition products (one 64 x 64 product per chunk
  // on the serial path).  Otherwise the 16-token sub-chunk kernel writes the state every 16 tokens, so
  // checkpoints must fall on those; it holds one CTA per SM (183-205 KB of shared memory), so past one
  // wave of row blocks the token-by-token kernel (two CTAs per SM) is faster.
  if (p.chunk == 32 && p.sa == nullptr) return launch_forward_transition(p, stream);
  if (p.chunk % 16 == 0 && (long long)p.B * p.H * 2 <= num_sms()) return launch_forward_chunked(p, stream);
  return launch_forward_sequential(p, stream);
}

WKV7_DEBUG_READER(debug_word_fwd)

}  // namespace wkv7
