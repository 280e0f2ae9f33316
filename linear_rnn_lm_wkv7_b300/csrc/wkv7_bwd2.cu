// WKV7 checkpointed backward on sm_103a, in two phases.
//
// Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Backward listing: chunks walked in reverse from the exact checkpoints,
// the VJP giving dr, dw, dk, dv, da, db.  With X_t the gradient w.r.t. the state S_t after
// token t, including y_t's term:
//     X_t     = X'_t + dy_t r_t^T          (X'_t from later tokens; X'_{T-1} = dhT)
//     dsa_t   = X_t b_t,   dv_t = X_t k_t                     (row sums)
//     X'_{t-1} = X_t diag(w_t) + dsa_t a_t^T
//     dr_t = S_t^T dy_t,  dk_t = X_t^T v_t,  db_t = X_t^T sa_t (column sums)
//     dw_t = colsum(X_t o S_{t-1}),  da_t = S_{t-1}^T dsa_t    (column sums)
// The state-gradient recurrence needs only the row sums; the column sums need X_t and S_t
// but nothing serial once X at each chunk end and every dsa_t are known.  So:
//
// Phase 1 (one pass over the sequence, like the forward): X is walked in reverse with
// only its row sums -- dsa_t by a one-token lookahead
//     dsa_{t-1} = X_t (w_t o b_{t-1}) + dsa_t (a_t . b_{t-1}) + dy_{t-1} (r_{t-1} . b_{t-1})
// and dv_t -- writing dv, dsa (workspace), X at every chunk end (workspace) and dh0.
// Mapping as the forward: a head in two row blocks of 32 rows, thread = 4 rows x 4
// columns, 16-lane row sums, tiles of 32 tokens staged with cp.async (here in reverse).
// (With chunk % 16 == 0 the walk runs instead on the 16-token sub-chunk kernel.)
//
// Phase 2 (every chunk of every head at once): one CTA per (head, chunk), in two passes
// over the chunk, neither of which divides by w (the page's rebuild of S_{t-1} as
// (S_t - v k^T - sa b^T) / w amplifies the checkpoint's rounding by 1/w per token):
//   pass A walks X down from X at the chunk end -- dk_t, db_t;
//   pass B runs S up from the state before the chunk (h_ckpt[c-1], or h0) -- da_t, dr_t;
//   dw_t, the one sum that needs X_t and S_{t-1} together, comes from a column recurrence:
//   with Z'_t = colsum(X'_t o S_t),
//       w_t o dw_t = Z'_{t-1} - a_t o da_t,  Z'_t = w_t o dw_t + k_t o dk_t + b_t o db_t - r_t o dr_t
//   (both from the two recurrences above), started from Z'_{t0-1} summed at the chunk start.
//   Where w_t < 1/32 the division by w_t would cost digits, and dw_t is summed directly with
//   X_t rebuilt from the chunk end (exact, rare).
// Each pass keeps its matrix scaled by a running decay product per column (X_t = M o rho_t,
// S_t = M o gamma_t), so a token's update is two FMAs per element with coefficients
// a/rho, r/rho (k/gamma, b/gamma) computed once per column; where the product would fall
// below 2^-40 the step is taken unscaled (M <- M * product + ...), so any w >= 0 works.
// Thread = 16 rows x 4 columns of M (row pairs as fp32x2; blocks of 4 rows interleaved over
// the four row quarters); a column sum is the thread's rows plus a reduce-scatter over the
// four row-quarter lanes, which leaves each lane one finished column.
#include "wkv7_colpass.cuh"
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

// ============================================================================ phase 1

constexpr int kTile = 32;          // tokens per staged tile
constexpr int kRows1 = 32;         // state rows per CTA
constexpr int kNT1 = kRows1 * 4;   // 128 threads: 8 row groups x 16 lanes
constexpr int kNW1 = kNT1 / 32;

template <typename Tin>
struct P1Smem {
  // raw stage (x2), token row index u = t - (tlo - 1): w, a, k rows 1..nt; b, r rows 0..nt;
  // dy (fp32, this CTA's rows) rows 0..nt
  static constexpr int kRawCols = 5 * (kTile + 1) * kD;
  static constexpr size_t kRawT = ((kRawCols * sizeof(Tin)) + 15) / 16 * 16;
  static constexpr size_t kRawDy = (kTile + 1) * kRows1 * 4;
  static constexpr size_t kRaw = kRawT + kRawDy;
  // fp32 tiles indexed by tt = t - tlo: W, A, K, CB (w_t o b_{t-1}), R1 (r_{t-1}) [kTile][kD];
  // AB (a_t . b_{t-1}), RB (r_{t-1} . b_{t-1}) [kTile]; DY1 (dy_{t-1}) [kTile][kRows1];
  // outputs DSA, DV [kTile][kRows1]
  static constexpr size_t oTiles = 2 * kRaw;
  static constexpr int kF32 = 5 * kTile * kD + 2 * kTile + 3 * kTile * kRows1;
  static constexpr size_t kBytes = oTiles + (size_t)kF32 * 4;
};

// cp.async copies for the tile of tokens [tlo, thi): w, a, k of tokens tlo..thi-1 and b, r, dy
// of tokens tlo-1..thi-1 (token tlo-1 only when tlo > 0)
template <typename Tin>
__device__ __forceinline__ void p1_issue(unsigned char* raw, int tlo, int thi, size_t base, size_t tstride, int rcol,
                                         const Tin* __restrict__ w, const Tin* __restrict__ a,
                                         const Tin* __restrict__ k, const Tin* __restrict__ b,
                                         const Tin* __restrict__ r, const float* __restrict__ dy) {
  constexpr int CPR = kD * (int)sizeof(Tin) / 16;
  constexpr int EPC = 16 / (int)sizeof(Tin);
  Tin* cols = reinterpret_cast<Tin*>(raw);
  const int ulo = tlo > 0 ? 0 : 1;  // first valid row index u (u = t - tlo + 1)
  const int nu = thi - tlo + 1;      // rows 0 .. nu-1
  const Tin* srcs[5] = {w, a, k, b, r};
#pragma unroll
  for (int q = 0; q < 5; ++q) {
    const int u0 = q < 3 ? 1 : ulo;  // w, a, k only for the tile's own tokens
    for (int e = threadIdx.x; e < (nu - u0) * CPR; e += kNT1) {
      const int u = u0 + e / CPR, pc = e % CPR;
      cp_async16(cols + (q * (kTile + 1) + u) * kD + pc * EPC,
                 srcs[q] + base + (size_t)(tlo - 1 + u) * tstride + pc * EPC);
    }
  }
  float* dyr = reinterpret_cast<float*>(raw + P1Smem<Tin>::kRawT);
  constexpr int FPR = kRows1 / 4;
  for (int e = threadIdx.x; e < (nu - ulo) * FPR; e += kNT1) {
    const int u = ulo + e / FPR, pc = e % FPR;
    cp_async16(dyr + u * kRows1 + pc * 4, dy + base + (size_t)(tlo - 1 + u) * tstride + rcol + pc * 4);
  }
}

template <typename Tin>
__global__ void __launch_bounds__(kNT1, 1)
gwalk_kernel(int T, int H, int chunk, int nchunks,
             const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
             const Tin* __restrict__ a, const Tin* __restrict__ b,
             const float* __restrict__ dy, const float* __restrict__ dhT,
             float* __restrict__ dv, float* __restrict__ dh0,
             float* __restrict__ dsa_ws, float* __restrict__ xck_ws) {
  using L = P1Smem<Tin>;
  constexpr int NRB = kD / kRows1;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  float* fW = reinterpret_cast<float*>(sm + L::oTiles);
  float* fA = fW + kTile * kD;
  float* fK = fA + kTile * kD;
  float* fCB = fK + kTile * kD;
  float* fR1 = fCB + kTile * kD;
  float* fAB = fR1 + kTile * kD;
  float* fRB = fAB + kTile;
  float* fDY1 = fRB + kTile;
  float* fDSA = fDY1 + kTile * kRows1;
  float* fDV = fDSA + kTile * kRows1;

  const int bh = blockIdx.x / NRB;
  const int rb = blockIdx.x - bh * NRB;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int l16 = tid & 15;
  const int rloc = 4 * (tid >> 4);
  const int row0 = rb * kRows1 + rloc;
  const int j0 = 4 * l16;
  const int qrow = rs_row(l16);
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;
  const int ntiles = (T + kTile - 1) / kTile;

  // X: starts at dhT, then gains dy_{T-1} r_{T-1}^T
  float2 X[4][2];
  if (dhT != nullptr) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x4 = __ldg(reinterpret_cast<const float4*>(dhT + sbase + (size_t)(row0 + i) * kD + j0));
      X[i][0] = lo2(x4);
      X[i][1] = hi2(x4);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) X[i][0] = X[i][1] = make_float2(0.f, 0.f);
  }
  float dsa[4] = {0.f, 0.f, 0.f, 0.f};
  if (T > 0) {
    const size_t o = base + (size_t)(T - 1) * tstride;
    const float4 r4 = load4(r + o + j0);
    const float4 b4 = load4(b + o + j0);
    const float4 d4 = __ldg(reinterpret_cast<const float4*>(dy + o + row0));
    const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      X[i][0] = __ffma2_rn(bcast2(dd[i]), lo2(r4), X[i][0]);
      X[i][1] = __ffma2_rn(bcast2(dd[i]), hi2(r4), X[i][1]);
    }
    dot4x4(X, b4, dsa);
    butterfly4(dsa);
    p1_issue<Tin>(sm, max(0, T - kTile), T, base, tstride, rb * kRows1, w, a, k, b, r, dy);
    cp_async_commit();
  }

  // tokens until (and including) the next chunk end walking down: the chunk of token T-1 ends at T-1
  int to_end = 0;
  for (int it = 0; it < ntiles; ++it) {
    const int thi = T - it * kTile;
    const int tlo = max(0, thi - kTile);
    const int nt = thi - tlo;
    unsigned char* raw = sm + (size_t)(it & 1) * L::kRaw;
    if (it + 1 < ntiles) {
      p1_issue<Tin>(sm + (size_t)((it + 1) & 1) * L::kRaw, max(0, tlo - kTile), tlo, base, tstride, rb * kRows1, w, a,
                    k, b, r, dy);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // this tile's stage has landed; the previous tile's fp32 data is consumed

    // ---- widen (8 lanes per token): W A K, CB = w_t o b_{t-1}, R1 = r_{t-1}, AB, RB
    {
      const Tin* cols = reinterpret_cast<const Tin*>(raw);
      const Tin* rW = cols;
      const Tin* rA = cols + (kTile + 1) * kD;
      const Tin* rK = cols + 2 * (kTile + 1) * kD;
      const Tin* rB = cols + 3 * (kTile + 1) * kD;
      const Tin* rR = cols + 4 * (kTile + 1) * kD;
      for (int tg = warp * 4; tg < nt; tg += kNW1 * 4) {
        const int tt = tg + (lane >> 3);  // token tlo + tt, row u = tt + 1; previous token row tt
        const int c8 = (lane & 7) * 8;
        float ab = 0.f, rb1 = 0.f;
        if (tt < nt) {
          float ww[8], aa[8], kk[8], bp[8], rp[8], cb[8];
          raw8(rW + (tt + 1) * kD + c8, ww);
          raw8(rA + (tt + 1) * kD + c8, aa);
          raw8(rK + (tt + 1) * kD + c8, kk);
          if (tlo + tt > 0) {
            raw8(rB + tt * kD + c8, bp);
            raw8(rR + tt * kD + c8, rp);
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) bp[u] = rp[u] = 0.f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            cb[u] = ww[u] * bp[u];
            ab = fmaf(aa[u], bp[u], ab);
            rb1 = fmaf(rp[u], bp[u], rb1);
          }
          store8(fW + tt * kD + c8, ww);
          store8(fA + tt * kD + c8, aa);
          store8(fK + tt * kD + c8, kk);
          store8(fCB + tt * kD + c8, cb);
          store8(fR1 + tt * kD + c8, rp);
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
          ab += __shfl_xor_sync(0xffffffffu, ab, m);
          rb1 += __shfl_xor_sync(0xffffffffu, rb1, m);
        }
        if (tt < nt && (lane & 7) == 0) {
          fAB[tt] = ab;
          fRB[tt] = rb1;
        }
      }
      const float* dyr = reinterpret_cast<const float*>(raw + L::kRawT);
      for (int e = tid; e < nt * kRows1; e += kNT1) {
        const int tt = e / kRows1;
        fDY1[e] = (tlo + tt > 0) ? dyr[e] : 0.f;  // row tt of the stage = token tlo + tt - 1
      }
    }
    __syncthreads();

    // ---- the reverse walk over the tile
#pragma unroll 2
    for (int tt = nt - 1; tt >= 0; --tt) {
      const int t = tlo + tt;
      const float4 w4 = *reinterpret_cast<const float4*>(fW + tt * kD + j0);
      const float4 a4 = *reinterpret_cast<const float4*>(fA + tt * kD + j0);
      const float4 k4 = *reinterpret_cast<const float4*>(fK + tt * kD + j0);
      const float4 cb4 = *reinterpret_cast<const float4*>(fCB + tt * kD + j0);
      const float4 r14 = *reinterpret_cast<const float4*>(fR1 + tt * kD + j0);
      const float4 dp4 = *reinterpret_cast<const float4*>(fDY1 + tt * kRows1 + rloc);
      const float ab = fAB[tt], rb1 = fRB[tt];
      const float dp[4] = {dp4.x, dp4.y, dp4.z, dp4.w};
      if (l16 == 0) *reinterpret_cast<float4*>(fDSA + tt * kRows1 + rloc) = make_float4(dsa[0], dsa[1], dsa[2], dsa[3]);

      // X at this chunk's last token is the start of phase 2's walk over the chunk
      if (to_end == 0) {
        const int c = t / chunk;
        to_end = t - c * chunk;  // tokens below t in this chunk
        float* dst = xck_ws + ((size_t)bh * nchunks + c) * kD * kD + (size_t)row0 * kD + j0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float4*>(dst + i * kD) = make_float4(X[i][0].x, X[i][0].y, X[i][1].x, X[i][1].y);
      } else {
        --to_end;
      }
      // dv_t = X_t k_t, and the lookahead row sums X_t (w_t o b_{t-1})
      float pv[4], P[4];
      dot4x4(X, k4, pv);
      dot4x4(X, cb4, P);
      const float dvq = reduce_scatter4(pv, l16);
      if ((l16 & 3) == 0) fDV[tt * kRows1 + rloc + qrow] = dvq;
      butterfly4(P);
      // X <- X w + dsa a + dy_{t-1} r_{t-1}
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 q2 = bcast2(dsa[i]), e2 = bcast2(dp[i]);
        X[i][0] = __ffma2_rn(X[i][0], lo2(w4), __ffma2_rn(q2, lo2(a4), __fmul2_rn(e2, lo2(r14))));
        X[i][1] = __ffma2_rn(X[i][1], hi2(w4), __ffma2_rn(q2, hi2(a4), __fmul2_rn(e2, hi2(r14))));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) dsa[i] = fmaf(dsa[i], ab, fmaf(dp[i], rb1, P[i]));
    }
    __syncthreads();
    for (int e = tid; e < nt * kRows1; e += kNT1) {
      const int tt = e / kRows1;
      const int rr = e % kRows1;
      const size_t o = base + (size_t)(tlo + tt) * tstride + rb * kRows1 + rr;
      dv[o] = fDV[e];
      dsa_ws[o] = fDSA[e];
    }
  }

  if (dh0 != nullptr) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dh0 + sbase + (size_t)(row0 + i) * kD + j0) =
          make_float4(X[i][0].x, X[i][0].y, X[i][1].x, X[i][1].y);
  }
}

// ============================================================================ phase 2

constexpr int kNT2 = 64;  // 2 warps: warp q covers columns 32q .. 32q+31, all 64 rows

template <typename Tin>
struct P2Smem {
  // raw inputs of the chunk: w, k, a, b, r, v [kTile][kD] (input dtype); sa, dsa, dy fp32 [kTile][kD]
  static constexpr size_t oCols = 0;
  static constexpr size_t kColsBytes = ((6 * kTile * kD * sizeof(Tin)) + 15) / 16 * 16;
  static constexpr size_t oSa = oCols + kColsBytes;
  static constexpr size_t oDsa = oSa + kTile * kD * 4;
  static constexpr size_t oDy = oDsa + kTile * kD * 4;
  // widened: v fp32 [kTile][kD]
  static constexpr size_t oV = oDy + kTile * kD * 4;
  static constexpr size_t kBytes = oV + kTile * kD * 4;
};

template <typename Tin>
__global__ void __launch_bounds__(kNT2)
colgrad_kernel(int T, int H, int chunk, int nchunks,
               const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
               const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
               const float* __restrict__ h0, const float* __restrict__ h_ckpt, const float* __restrict__ sa,
               const float* __restrict__ dy, const float* __restrict__ dsa_ws, const float* __restrict__ xck_ws,
               float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
               float* __restrict__ da, float* __restrict__ db) {
  using L = P2Smem<Tin>;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  const Tin* cW = reinterpret_cast<const Tin*>(sm + L::oCols);
  const Tin* cK = cW + kTile * kD;
  const Tin* cA = cW + 2 * kTile * kD;
  const Tin* cB = cW + 3 * kTile * kD;
  const Tin* cR = cW + 4 * kTile * kD;
  const Tin* cV = cW + 5 * kTile * kD;
  const float* sSa = reinterpret_cast<const float*>(sm + L::oSa);
  const float* sDsa = reinterpret_cast<const float*>(sm + L::oDsa);
  const float* sDy = reinterpret_cast<const float*>(sm + L::oDy);
  float* sV = reinterpret_cast<float*>(sm + L::oV);

  const int ci = blockIdx.x % nchunks;
  const int bh = blockIdx.x / nchunks;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int c0 = 32 * (tid >> 5) + 4 * (lane & 7);  // columns c0 .. c0+3
  const int rq = lane >> 3;                         // rows 16 i + 4 rq .. 16 i + 4 rq + 3, i < 4
  const int r0 = 4 * rq;
  const int own = 2 * (rq & 1) + (rq >> 1);         // the column c0 + own this lane finishes
  const int t0 = ci * chunk;
  const int n = min(chunk, T - t0);
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const float* xend = xck_ws + ((size_t)bh * nchunks + ci) * kD * kD;
  const float* s0 = ci > 0 ? h_ckpt + ((size_t)bh * nchunks + ci - 1) * kD * kD
                           : (h0 != nullptr ? h0 + (size_t)bh * kD * kD : nullptr);

  // ---- stage the chunk's inputs
  {
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    Tin* cols = reinterpret_cast<Tin*>(sm + L::oCols);
    const Tin* srcs[6] = {w, k, a, b, r, v};
#pragma unroll
    for (int q = 0; q < 6; ++q)
      for (int e = tid; e < n * CPR; e += kNT2) {
        const int tt = e / CPR, pc = e % CPR;
        cp_async16(cols + (q * kTile + tt) * kD + pc * EPC, srcs[q] + base + (size_t)(t0 + tt) * tstride + pc * EPC);
      }
    const float* fsrc[3] = {sa, dsa_ws, dy};
    float* fdst[3] = {reinterpret_cast<float*>(sm + L::oSa), reinterpret_cast<float*>(sm + L::oDsa),
                      reinterpret_cast<float*>(sm + L::oDy)};
#pragma unroll
    for (int q = 0; q < 3; ++q)
      for (int e = tid; e < n * (kD / 4); e += kNT2) {
        const int tt = e / (kD / 4), pc = e % (kD / 4);
        cp_async16(fdst[q] + tt * kD + pc * 4, fsrc[q] + base + (size_t)(t0 + tt) * tstride + pc * 4);
      }
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();
  for (int e = tid; e < n * kD; e += kNT2) sV[e] = to_f32(cV[e]);
  __syncthreads();
  colpass::passes<Tin>(tid, n, t0, base, tstride, cW, sSa, sDsa, sDy, sV, xend, s0, dr, dw, dk, da, db);
}

template <typename Tin>
cudaError_t launch_bwd2_t(const BwdArgs& p, float* dsa_ws, float* xck_ws, cudaStream_t stream) {
  if (p.chunk % 16 == 0 && p.T > 0 && (long long)p.B * p.H * (kD / kRows1) <= num_sms()) {
    // the walk as the forward recurrence run backwards, in 16-step sub-chunks on tensor cores
    cudaError_t err = launch_gwalk_chunked(p, dsa_ws, xck_ws, stream);
    if (err != cudaSuccess) return err;
  } else {
    const size_t smem = P1Smem<Tin>::kBytes;
    static_assert(P1Smem<Tin>::kBytes <= 232448, "shared memory per CTA");
    auto kern = gwalk_kernel<Tin>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const unsigned grid = (unsigned)p.B * p.H * (kD / kRows1);
    kern<<<grid, kNT1, smem, stream>>>(p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r, (const Tin*)p.in.w,
                                       (const Tin*)p.in.k, (const Tin*)p.in.a, (const Tin*)p.in.b, p.dy, p.dhT,
                                       p.dv, p.dh0, dsa_ws, xck_ws);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (p.nchunks == 0) return cudaSuccess;
  {
    const size_t smem = P2Smem<Tin>::kBytes;
    static_assert(P2Smem<Tin>::kBytes <= 232448, "shared memory per CTA");
    auto kern = colgrad_kernel<Tin>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const unsigned grid = (unsigned)p.B * p.H * p.nchunks;
    kern<<<grid, kNT2, smem, stream>>>(p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r, (const Tin*)p.in.w,
                                       (const Tin*)p.in.k, (const Tin*)p.in.v, (const Tin*)p.in.a,
                                       (const Tin*)p.in.b, p.h0, p.h_ckpt, p.sa, p.dy, dsa_ws, xck_ws, p.dr, p.dw, p.dk,
                                       p.da, p.db);
    return cudaGetLastError();
  }
}

}  // namespace

namespace {
// the two-phase backward with a saved sa: dsa (B,T,H,D) then X at every chunk end (B,H,C,D,D)
size_t two_phase_bytes(int B, int T, int H, int chunk) {
  const size_t C = T > 0 ? (size_t)((T + chunk - 1) / chunk) : 0;
  const size_t dsa = (size_t)B * T * H * kD * 4;
  const size_t xck = (size_t)B * H * C * kD * kD * 4;
  return (dsa + 255) / 256 * 256 + xck;
}
}  // namespace

size_t backward_workspace_bytes(int B, int T, int H, int chunk) {
  const size_t a = two_phase_bytes(B, T, H, chunk);
  if (chunk != 32) return a;
  const size_t b = xop_workspace_bytes(B, T, H, false);
  return a > b ? a : b;
}

size_t forward_workspace_bytes(int B, int T, int H, int chunk) {
  return chunk == 32 ? xop_workspace_bytes(B, T, H, true) : 0;
}

cudaError_t launch_backward_transition(const BwdArgs& p, void* workspace, bool from_forward, cudaStream_t stream) {
  ChunkEnds ends;
  cudaError_t err = launch_xop_walk(p, workspace, from_forward, 0, &ends, stream);
  if (err != cudaSuccess) return err;
  return launch_colgrad_matrix(p, ends, stream);
}

cudaError_t launch_backward_two_phase(const BwdArgs& p, void* workspace, cudaStream_t stream) {
  float* dsa_ws = static_cast<float*>(workspace);
  const size_t dsa = (size_t)p.B * p.T * p.H * kD * 4;
  float* xck_ws = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + (dsa + 255) / 256 * 256);
  return p.bf16 ? launch_bwd2_t<__nv_bfloat16>(p, dsa_ws, xck_ws, stream)
                : launch_bwd2_t<float>(p, dsa_ws, xck_ws, stream);
}

WKV7_DEBUG_READER(debug_word_bwd2)

}  // namespace wkv7
