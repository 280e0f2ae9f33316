// The exact two-pass column gradients of one chunk on CUDA cores (used by the two-phase backward's
// column pass, and by the matrix-form column kernel for chunks whose decays are too strong for it).
//
// Over a chunk t0..te, with X_t the gradient w.r.t. the state after token t (including dy_t r_t^T):
//   pass A walks X down from X at the chunk end,
//       X_{t-1} = X_t diag(w_t) + dsa_t a_t^T + dy_{t-1} r_{t-1}^T,   dk_t = X_t^T v_t, db_t = X_t^T sa_t;
//   pass B runs the state up from the state before the chunk (h_ckpt[c-1], or h0),
//       S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T,   da_t = S_{t-1}^T dsa_t, dr_t = S_t^T dy_t;
//   dw_t = colsum(X_t o S_{t-1}) comes from the column recurrence of Z'_t = colsum(X'_t o S_t):
//       w_t o dw_t = Z'_{t-1} - a_t o da_t,  Z'_t = w_t o dw_t + k_t o dk_t + b_t o db_t - r_t o dr_t,
//   started from Z'_{t0-1} summed at the chunk start; where w_t < 1/32 dw_t is summed directly from
//   X_t (rebuilt from the chunk end) and S_{t-1}.  Neither pass divides a state by w.
// Each pass keeps its matrix scaled by a running decay product per column (X_t = M o rho_t,
// S_t = M o gamma_t), so a token's update is two FMAs per element; where the product would fall below
// 2^-40 the step is taken unscaled, so any w >= 0 works.  Thread = 16 rows x 4 columns of M (row pairs
// as fp32x2; blocks of 4 rows interleaved over the four row quarters); a column sum is the thread's
// rows plus a reduce-scatter over the four row-quarter lanes, leaving each lane one finished column.
// Source of the recurrence: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture" (Backward listing: chunks walked in reverse from the exact checkpoints).
#pragma once

#include "wkv7_device.cuh"

namespace wkv7 {
namespace colpass {

constexpr int kTile = 32;  // tokens per chunk at most
constexpr int kRP = 8;    // row pairs per thread (16 rows)
constexpr int kCT = 4;    // columns per thread
// a column's running decay product below 2^-40 is folded back into the state (keeps 1/product finite)
constexpr float kRenorm = 9.094947017729282e-13f;
// below this w_t, w_t dw_t (a difference of column sums) loses too many digits when divided by w_t:
// dw_t is then summed directly from X_t and S_{t-1}
constexpr float kWTiny = 0.03125f;


// four consecutive columns of a token row
template <typename Tin>
__device__ __forceinline__ void col4(const Tin* p, float (&o)[kCT]) {
  if constexpr (sizeof(Tin) == 2) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    o[0] = bf16_lo(u.x), o[1] = bf16_hi(u.x), o[2] = bf16_lo(u.y), o[3] = bf16_hi(u.y);
  } else {
    const float4 f = *reinterpret_cast<const float4*>(p);
    o[0] = f.x, o[1] = f.y, o[2] = f.z, o[3] = f.w;
  }
}

template <typename Tin>
__device__ __forceinline__ float col1(const Tin* p) {
  return to_f32(*p);
}

// A thread's rows: blocks of 4 rows, interleaved over the four row quarters (r0 = 4 rq) so that the
// quarters' reads of a token's row vector are 64 contiguous bytes.  Row pair p starts at prow(r0, p).
__device__ __forceinline__ int prow(int r0, int p) { return 16 * (p >> 1) + r0 + 2 * (p & 1); }

// the thread's row pairs (p < kRP) of columns c0 .. c0+3 of a row-major 64 x 64 fp32 matrix (global or shared)
__device__ __forceinline__ void load_block(const float* __restrict__ m, int r0, int c0, float2 (&o)[kRP][kCT]) {
#pragma unroll
  for (int p = 0; p < kRP; ++p) {
    const float4 e = *reinterpret_cast<const float4*>(m + (size_t)prow(r0, p) * kD + c0);
    const float4 f = *reinterpret_cast<const float4*>(m + (size_t)(prow(r0, p) + 1) * kD + c0);
    o[p][0] = make_float2(e.x, f.x);
    o[p][1] = make_float2(e.y, f.y);
    o[p][2] = make_float2(e.z, f.z);
    o[p][3] = make_float2(e.w, f.w);
  }
}

// The sums of x[c][j] over the four row-quarter lanes (lane bits 3 and 4), reduce-scattered: the lane
// with row quarter rq ends with both sums of column own(rq) = 2 (rq & 1) + (rq >> 1).
template <int NJ>
__device__ __forceinline__ void rs_cols(const float (&x)[kCT][NJ], int rq, float (&out)[NJ]) {
  const bool b0 = rq & 1, b1 = rq & 2;
  float k[2][NJ];
#pragma unroll
  for (int cc = 0; cc < 2; ++cc)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const float send = b0 ? x[cc][j] : x[2 + cc][j];
      const float keep = b0 ? x[2 + cc][j] : x[cc][j];
      k[cc][j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const float send = b1 ? k[0][j] : k[1][j];
    const float keep = b1 ? k[1][j] : k[0][j];
    out[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
}

// The running decay product of a column: next[c] = scale[c] * w[c].  Where it would drop below kRenorm
// the step is taken unscaled instead -- M[:, c] is multiplied by f[c] = scale[c] * w[c] in the update and
// next[c] = 1 -- so no coefficient is ever divided by a tiny product (any w >= 0 works).  Returns whether
// any lane of the warp takes such a step (then the sweep multiplies M by f).
__device__ __forceinline__ bool decay_step(const float (&scale)[kCT], const float (&wv)[kCT], float (&next)[kCT],
                                           float2 (&f)[kCT]) {
  bool any = false;
#pragma unroll
  for (int c = 0; c < kCT; ++c) {
    next[c] = scale[c] * wv[c];
    const bool fold = next[c] < kRenorm;
    f[c] = bcast2(fold ? next[c] : 1.f);
    if (fold) next[c] = 1.f;
    any |= fold;
  }
  return __any_sync(0xffffffffu, any);
}

// Pass A step at one token (M = X_t / rho_t): acc[0] += v_t o M, acc[1] += sa_t o M, then
// M <- M * f + dsa_t ca^T + dy_{t-1} cr^T
template <bool kFold>
__device__ __forceinline__ void sweep_a(float2 (&M)[kRP][kCT], const float* rv, const float* rs, const float* rq,
                                        const float* re, const float2 (&ca)[kCT], const float2 (&cr)[kCT],
                                        const float2 (&f)[kCT], float2 (&acc)[2][kCT][2]) {
#pragma unroll
  for (int p4 = 0; p4 < kRP / 2; ++p4) {
    const float4 v4 = *reinterpret_cast<const float4*>(rv + 16 * p4);
    const float4 s4 = *reinterpret_cast<const float4*>(rs + 16 * p4);
    const float4 q4 = *reinterpret_cast<const float4*>(rq + 16 * p4);
    const float4 e4 = *reinterpret_cast<const float4*>(re + 16 * p4);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int p = 2 * p4 + h;
      const float2 v2 = h ? hi2(v4) : lo2(v4), s2 = h ? hi2(s4) : lo2(s4);
      const float2 q2 = h ? hi2(q4) : lo2(q4), e2 = h ? hi2(e4) : lo2(e4);
#pragma unroll
      for (int c = 0; c < kCT; ++c) {
        acc[0][c][h] = p4 == 0 ? __fmul2_rn(v2, M[p][c]) : __ffma2_rn(v2, M[p][c], acc[0][c][h]);
        acc[1][c][h] = p4 == 0 ? __fmul2_rn(s2, M[p][c]) : __ffma2_rn(s2, M[p][c], acc[1][c][h]);
        const float2 m = kFold ? __fmul2_rn(M[p][c], f[c]) : M[p][c];
        M[p][c] = __ffma2_rn(q2, ca[c], __ffma2_rn(e2, cr[c], m));
      }
    }
  }
}

// Pass B step at one token (M = S_{t-1} / gamma_{t-1}): acc[0] += dsa_t o M, M <- M * f + v_t ck^T +
// sa_t cb^T, acc[1] += dy_t o M
template <bool kFold>
__device__ __forceinline__ void sweep_b(float2 (&M)[kRP][kCT], const float* rq, const float* rv, const float* rs,
                                        const float* rd, const float2 (&ck)[kCT], const float2 (&cb)[kCT],
                                        const float2 (&f)[kCT], float2 (&acc)[2][kCT][2]) {
#pragma unroll
  for (int p4 = 0; p4 < kRP / 2; ++p4) {
    const float4 q4 = *reinterpret_cast<const float4*>(rq + 16 * p4);
    const float4 v4 = *reinterpret_cast<const float4*>(rv + 16 * p4);
    const float4 s4 = *reinterpret_cast<const float4*>(rs + 16 * p4);
    const float4 d4 = *reinterpret_cast<const float4*>(rd + 16 * p4);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int p = 2 * p4 + h;
      const float2 q2 = h ? hi2(q4) : lo2(q4), v2 = h ? hi2(v4) : lo2(v4);
      const float2 s2 = h ? hi2(s4) : lo2(s4), d2 = h ? hi2(d4) : lo2(d4);
#pragma unroll
      for (int c = 0; c < kCT; ++c) {
        acc[0][c][h] = p4 == 0 ? __fmul2_rn(q2, M[p][c]) : __ffma2_rn(q2, M[p][c], acc[0][c][h]);
        const float2 m = kFold ? __fmul2_rn(M[p][c], f[c]) : M[p][c];
        M[p][c] = __ffma2_rn(v2, ck[c], __ffma2_rn(s2, cb[c], m));
        acc[1][c][h] = p4 == 0 ? __fmul2_rn(d2, M[p][c]) : __ffma2_rn(d2, M[p][c], acc[1][c][h]);
      }
    }
  }
}


// The two passes over one chunk of n tokens on 64 threads (tid < 64).  Shared memory holds the chunk's
// raw inputs cols (Tin [6][32][64]: w, k, a, b, r, v, rows 0..n-1) and fp32 [32][64] sa, dsa, dy and
// v widened; xend (X at the chunk's last token, row-major 64 x 64, global or shared memory) and s0 (the
// state before the chunk, global, or null for zeros).  Writes dr, dw, dk, da, db at tokens t0..t0+n-1 (element
// base + t*tstride + column).
template <typename Tin>
__device__ __forceinline__ void passes(int tid, int n, int t0, size_t base, size_t tstride, const Tin* cols,
                                       const float* sSa, const float* sDsa, const float* sDy, const float* sV,
                                       const float* __restrict__ xend, const float* __restrict__ s0,
                                       float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
                                       float* __restrict__ da, float* __restrict__ db) {
  const Tin* cW = cols;
  const Tin* cK = cW + kTile * kD;
  const Tin* cA = cW + 2 * kTile * kD;
  const Tin* cB = cW + 3 * kTile * kD;
  const Tin* cR = cW + 4 * kTile * kD;
  const int lane = tid & 31;
  const int c0 = 32 * (tid >> 5) + 4 * (lane & 7);  // columns c0 .. c0+3
  const int rq = lane >> 3;                         // rows 16 i + 4 rq .. 16 i + 4 rq + 3, i < 4
  const int r0 = 4 * rq;
  const int own = 2 * (rq & 1) + (rq >> 1);         // the column c0 + own this lane finishes

  // M = X at the chunk's last token (rho = 1): rows r0 .. r0+15, columns c0 .. c0+3, as row pairs
  float2 M[kRP][kCT];
  load_block(xend, r0, c0, M);

  // ---- pass A, tokens n-1 .. 0: X_t = M o rho_t (columns), X'_{t-1} = X_t diag(w_t) + dsa_t a_t^T,
  // X_{t-1} = X'_{t-1} + dy_{t-1} r_{t-1}^T; dk_t = X_t^T v_t, db_t = X_t^T sa_t
  float rho[kCT] = {1.f, 1.f, 1.f, 1.f};
  for (int tt = n - 1; tt >= 0; --tt) {
    const int tm = tt > 0 ? tt - 1 : 0;  // dy_{t-1}, r_{t-1}; token 0 of the chunk takes none
    float wv[kCT], av[kCT], rv[kCT];
    col4<Tin>(cW + tt * kD + c0, wv);
    col4<Tin>(cA + tt * kD + c0, av);
    col4<Tin>(cR + tm * kD + c0, rv);
    float rn[kCT];
    float2 f[kCT];
    const bool fold = decay_step(rho, wv, rn, f);
    float2 ca[kCT], cr[kCT];
#pragma unroll
    for (int c = 0; c < kCT; ++c) {
      const float ir = __fdividef(1.f, rn[c]);
      ca[c] = bcast2(av[c] * ir);
      cr[c] = bcast2(tt > 0 ? rv[c] * ir : 0.f);
    }
    const float* rvp = sV + tt * kD + r0;
    const float* rsp = sSa + tt * kD + r0;
    const float* rqp = sDsa + tt * kD + r0;
    const float* rep = sDy + tm * kD + r0;
    float2 acc[2][kCT][2];
    if (fold)
      sweep_a<true>(M, rvp, rsp, rqp, rep, ca, cr, f, acc);
    else
      sweep_a<false>(M, rvp, rsp, rqp, rep, ca, cr, f, acc);
    float x[kCT][2], g[2];
#pragma unroll
    for (int c = 0; c < kCT; ++c)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 s = __fadd2_rn(acc[j][c][0], acc[j][c][1]);
        x[c][j] = (s.x + s.y) * rho[c];
      }
    rs_cols<2>(x, rq, g);
    const size_t o = base + (size_t)(t0 + tt) * tstride + c0 + own;
    dk[o] = g[0];
    db[o] = g[1];
#pragma unroll
    for (int c = 0; c < kCT; ++c) rho[c] = rn[c];
  }

  // ---- M = S_{t0-1} (the state before the chunk; gamma = 1) and Z'_{t0-1} = colsum(X'_{t0-1} o S_{t0-1})
  float zq;
  {
    float2 S[kRP][kCT];
    if (s0 != nullptr) {
      load_block(s0, r0, c0, S);
    } else {
#pragma unroll
      for (int p = 0; p < kRP; ++p)
#pragma unroll
        for (int c = 0; c < kCT; ++c) S[p][c] = make_float2(0.f, 0.f);
    }
    float2 z[kCT];
#pragma unroll
    for (int c = 0; c < kCT; ++c) z[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int p = 0; p < kRP; ++p)
#pragma unroll
      for (int c = 0; c < kCT; ++c) {
        z[c] = __ffma2_rn(M[p][c], S[p][c], z[c]);
        M[p][c] = S[p][c];
      }
    float x[kCT][1], g[1];
#pragma unroll
    for (int c = 0; c < kCT; ++c) x[c][0] = (z[c].x + z[c].y) * rho[c];
    rs_cols<1>(x, rq, g);
    zq = g[0];
  }

  // ---- pass B, tokens 0 .. n-1: S_t = M o gamma_t; da_t = S_{t-1}^T dsa_t, dr_t = S_t^T dy_t and
  //   w_t o dw_t = Z'_{t-1} - a_t o da_t,  Z'_t = w_t o dw_t + k_t o dk_t + b_t o db_t - r_t o dr_t
  // with Z'_t = colsum(X'_t o S_t) (X'_t: X_t without dy_t r_t^T); this lane carries Z' of column c0 + own
  float gam[kCT] = {1.f, 1.f, 1.f, 1.f};
  for (int tt = 0; tt < n; ++tt) {
    float wv[kCT], kv[kCT], bv[kCT];
    col4<Tin>(cW + tt * kD + c0, wv);
    col4<Tin>(cK + tt * kD + c0, kv);
    col4<Tin>(cB + tt * kD + c0, bv);
    const size_t o = base + (size_t)(t0 + tt) * tstride + c0 + own;
    const float dko = dk[o], dbo = db[o];  // written by this thread in pass A
    const float wo = col1<Tin>(cW + tt * kD + c0 + own), ko = col1<Tin>(cK + tt * kD + c0 + own);
    const float bo = col1<Tin>(cB + tt * kD + c0 + own), ao = col1<Tin>(cA + tt * kD + c0 + own);
    const float ro = col1<Tin>(cR + tt * kD + c0 + own);

    // direct dw_t = colsum(X_t o S_{t-1}) where w_t is tiny: X_t rebuilt from the chunk end
    float dwd = 0.f;
    {
      bool tiny = false;
#pragma unroll
      for (int c = 0; c < kCT; ++c) tiny |= wv[c] < kWTiny;
      if (__any_sync(0xffffffffu, tiny)) {
        float x[kCT][1], g[1];
#pragma unroll
        for (int c = 0; c < kCT; ++c) x[c][0] = 0.f;
#pragma unroll
        for (int p = 0; p < kRP; ++p) {
          float2 X[kCT];
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const float4 e = *reinterpret_cast<const float4*>(xend + (size_t)(prow(r0, p) + hr) * kD + c0);
            const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
            for (int c = 0; c < kCT; ++c) (hr ? X[c].y : X[c].x) = ev[c];
          }
          for (int u = n - 1; u > tt; --u) {
            float wu[kCT], au[kCT], ru[kCT];
            col4<Tin>(cW + u * kD + c0, wu);
            col4<Tin>(cA + u * kD + c0, au);
            col4<Tin>(cR + (u - 1) * kD + c0, ru);
            const float2 q2 = *reinterpret_cast<const float2*>(sDsa + u * kD + prow(r0, p));
            const float2 e2 = *reinterpret_cast<const float2*>(sDy + (u - 1) * kD + prow(r0, p));
#pragma unroll
            for (int c = 0; c < kCT; ++c)
              X[c] = __ffma2_rn(X[c], bcast2(wu[c]), __ffma2_rn(q2, bcast2(au[c]), __fmul2_rn(e2, bcast2(ru[c]))));
          }
#pragma unroll
          for (int c = 0; c < kCT; ++c) {
            const float2 m = __fmul2_rn(X[c], M[p][c]);
            x[c][0] += (m.x + m.y) * gam[c];
          }
        }
        rs_cols<1>(x, rq, g);
        dwd = g[0];
      }
    }

    float gn[kCT];
    float2 f[kCT];
    const bool fold = decay_step(gam, wv, gn, f);
    float2 ck[kCT], cb[kCT];
#pragma unroll
    for (int c = 0; c < kCT; ++c) {
      const float ig = __fdividef(1.f, gn[c]);
      ck[c] = bcast2(kv[c] * ig);
      cb[c] = bcast2(bv[c] * ig);
    }
    const float* rqp = sDsa + tt * kD + r0;
    const float* rvp = sV + tt * kD + r0;
    const float* rsp = sSa + tt * kD + r0;
    const float* rdp = sDy + tt * kD + r0;
    float2 acc[2][kCT][2];
    if (fold)
      sweep_b<true>(M, rqp, rvp, rsp, rdp, ck, cb, f, acc);
    else
      sweep_b<false>(M, rqp, rvp, rsp, rdp, ck, cb, f, acc);
    float x[kCT][2], g[2];
#pragma unroll
    for (int c = 0; c < kCT; ++c) {
      const float2 sA = __fadd2_rn(acc[0][c][0], acc[0][c][1]);
      const float2 sR = __fadd2_rn(acc[1][c][0], acc[1][c][1]);
      x[c][0] = (sA.x + sA.y) * gam[c];  // gamma_{t-1}
      x[c][1] = (sR.x + sR.y) * gn[c];   // gamma_t
    }
    rs_cols<2>(x, rq, g);
    const float wdw = fmaf(-ao, g[0], zq);
    dw[o] = wo < kWTiny ? dwd : wdw * __fdividef(1.f, wo);
    da[o] = g[0];
    dr[o] = g[1];
    zq = fmaf(-ro, g[1], fmaf(bo, dbo, fmaf(ko, dko, wdw)));
#pragma unroll
    for (int c = 0; c < kCT; ++c) gam[c] = gn[c];
  }
}

}  // namespace colpass
}  // namespace wkv7
