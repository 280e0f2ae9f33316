// WKV7 checkpointed backward on sm_103a.
//
// Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Backward listing: chunks are walked in reverse starting from the
// exact checkpoints; inside a chunk the tokens are walked in reverse, the VJP gives
// dr, dw, dk, dv, da, db, and the previous state is rebuilt as (h - v k - sa b) / w.
// The listing does not say where sa comes from.  Either the forward saved it (one fp32
// per row and token, the `sa` buffer), or each chunk is first run forward from its start
// checkpoint (h0 for the first chunk) to recompute it.
//
// Per token t, in reverse, with Gh the gradient w.r.t. the state S' after token t
// including y_t's term (Gh = G + dy r^T) and S the state before it:
//     dr = S'^T dy
//     S  = (S' - v k^T - sa b^T) diag(1/w)
//     dw_j = sum_i Gh_ij S_ij;  dk = Gh^T v;  db = Gh^T sa;  dv = Gh k;  dsa = Gh b
//     da = S^T dsa;  G <- Gh diag(w) + dsa a^T
// Rows of S and G never interact (dsa and dv are row sums); the five column gradients
// are sums over all rows.
//
// Lookahead.  The serial chain is Gh_t -> dsa_t -> Gh_{t-1}.  Since
//     Gh_{t-1} = Gh_t diag(w_t) + dsa_t a_t^T + dy_{t-1} r_{t-1}^T,
//     dsa_{t-1} = Gh_t (w_t o b_{t-1}) + dsa_t (a_t . b_{t-1}) + dy_{t-1} (r_{t-1} . b_{t-1}),
// so the row sum that yields dsa_{t-1} reads Gh_t and runs beside token t's update.
// w_t o b_{t-1}, a_t . b_{t-1}, r_t . b_t and 1/w_t are formed once per chunk.
//
// Mapping.  A head is split into NCL row blocks of 64/NCL rows, one CTA each, the NCL
// CTAs of a head forming a thread-block cluster; every CTA has 8 warps (two per
// scheduler).  Thread = R consecutive rows x 2 columns of S and of G in registers, held
// as fp32x2 pairs along rows so that every update is a packed FMA; the 32 lanes of a
// warp cover the 64 columns and a warp owns R whole rows.  Row sums (dsa lookahead, dv)
// are 32-lane reduce-scatters; column sums need no exchange inside the warp: each lane
// sums its R rows and writes its 10 per-token partials (5 gradients x 2 columns) to the
// warp's slab in shared memory.  Every ST tokens the CTA sums the warps' slabs.  With
// NCL == 1 the sums go straight to HBM; with NCL == 2 each CTA owns half the columns:
// sums for its own columns stay in shared memory, the others are stored into the peer
// CTA's shared memory (distributed shared memory), and once per chunk, after a cluster
// barrier, each CTA adds the two halves and writes its columns.  Deterministic: every sum
// is taken in a fixed order, no atomics.
//
// Staging.  The chunk's r, w, k, a, b, the CTA's slices of v, dy and sa are copied to
// shared memory with cp.async one chunk ahead and widened to fp32 tiles (with 1/w,
// w_t o b_{t-1}, a_t . b_{t-1}, r_t . b_t) once per chunk; the checkpoint that starts the
// next chunk's walk is loaded into registers one chunk ahead.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kCT = 32;  // stage capacity in tokens (chunk <= 32)
constexpr int kNG = 5;   // column gradients in slab order: dr, dw, dk, db, da

#ifndef WKV7_BWD_NW2
#define WKV7_BWD_NW2 8  // warps per CTA with two CTAs per head
#endif
#ifndef WKV7_BWD_ST2
#define WKV7_BWD_ST2 4  // tokens per column-sum sub-tile with two CTAs per head
#endif

constexpr size_t al16(size_t x) { return (x + 15) / 16 * 16; }

template <typename Tin, int NCL, int NW, int ST>
struct BwdSmem {
  static constexpr int ROWS = kD / NCL;
  static constexpr int R = ROWS / NW;    // rows per thread
  static constexpr int CPC = kD / NCL;   // columns of the column gradients this CTA writes
  // raw stage (cp.async target): Tin [5][kCT][kD] (w k a b r), Tin [kCT][ROWS] (v), f32 [kCT][ROWS] (dy, sa)
  static constexpr size_t oCol = 0;
  static constexpr size_t oV = oCol + al16(5 * kCT * kD * sizeof(Tin));
  static constexpr size_t oDy = oV + al16(kCT * ROWS * sizeof(Tin));
  static constexpr size_t oSa = oDy + kCT * ROWS * 4;
  static constexpr size_t kStage = oSa + kCT * ROWS * 4;
  // fp32 tiles of the chunk being walked: [7][kCT][kD] (w, 1/w, k, a, b, r, w_t o b_{t-1}),
  // [3][kCT][ROWS] (v, dy, sa), [2][kCT] (a_t . b_{t-1}, r_t . b_t), dv [kCT][ROWS]
  static constexpr size_t oTile = kStage;
  static constexpr size_t oRowT = oTile + 7 * kCT * kD * 4;
  static constexpr size_t oScal = oRowT + 3 * kCT * ROWS * 4;
  static constexpr size_t oDv = oScal + 2 * kCT * 4;
  static constexpr size_t oSlab = oDv + kCT * ROWS * 4;                                 // f32 [NW][ST][kNG][kD]
  static constexpr size_t oPart = oSlab + (size_t)NW * ST * kNG * kD * 4;                // f32 [kNG][kCT][CPC]
  static constexpr size_t oRecv = oPart + (NCL > 1 ? (size_t)kNG * kCT * CPC * 4 : 0);  // f32 [2][kNG][kCT][CPC]
  static constexpr size_t kBytes = oRecv + (NCL > 1 ? (size_t)2 * kNG * kCT * CPC * 4 : 0);
};
enum { TW = 0, TWI = 1, TK = 2, TA = 3, TB = 4, TR = 5, TCB = 6 };

// cp.async copies of one chunk's inputs into the raw stage
template <typename Tin, int ROWS, int kNT, bool SAVED>
__device__ __forceinline__ void issue_stage(unsigned char* stg, size_t oV, size_t oDy, size_t oSa, int t0, int n,
                                            size_t base, size_t tstride, int rbase, const Tin* __restrict__ w,
                                            const Tin* __restrict__ k, const Tin* __restrict__ a,
                                            const Tin* __restrict__ b, const Tin* __restrict__ r,
                                            const Tin* __restrict__ v, const float* __restrict__ dy,
                                            const float* __restrict__ sa) {
  constexpr int CPR = kD * (int)sizeof(Tin) / 16;  // 16-byte pieces per 64-wide row
  constexpr int EPC = 16 / (int)sizeof(Tin);       // elements per piece
  Tin* col = reinterpret_cast<Tin*>(stg);
  const Tin* srcs[5] = {w, k, a, b, r};
#pragma unroll
  for (int q = 0; q < 5; ++q) {
    for (int e = threadIdx.x; e < n * CPR; e += kNT) {
      const int tt = e / CPR, pc = e % CPR;
      cp_async16(col + (q * kCT + tt) * kD + pc * EPC, srcs[q] + base + (size_t)(t0 + tt) * tstride + pc * EPC);
    }
  }
  {
    constexpr int VPR = ROWS * (int)sizeof(Tin) / 16;
    Tin* dst = reinterpret_cast<Tin*>(stg + oV);
    for (int e = threadIdx.x; e < n * VPR; e += kNT) {
      const int tt = e / VPR, pc = e % VPR;
      cp_async16(dst + tt * ROWS + pc * EPC, v + base + (size_t)(t0 + tt) * tstride + rbase + pc * EPC);
    }
  }
  {
    constexpr int FPR = ROWS / 4;
    float* ddy = reinterpret_cast<float*>(stg + oDy);
    float* dsa = reinterpret_cast<float*>(stg + oSa);
    for (int e = threadIdx.x; e < n * FPR; e += kNT) {
      const int tt = e / FPR, pc = e % FPR;
      const size_t off = base + (size_t)(t0 + tt) * tstride + rbase + pc * 4;
      cp_async16(ddy + tt * ROWS + pc * 4, dy + off);
      if (SAVED) cp_async16(dsa + tt * ROWS + pc * 4, sa + off);
    }
  }
}

__device__ __forceinline__ float* pick(int g, float* p0, float* p1, float* p2, float* p3, float* p4) {
  return g == 0 ? p0 : g == 1 ? p1 : g == 2 ? p2 : g == 3 ? p3 : p4;
}

// R consecutive fp32 values (R % 4 == 0) from shared memory
template <int R>
__device__ __forceinline__ void lds_rows(const float* p, float (&o)[R]) {
#pragma unroll
  for (int q = 0; q < R / 4; ++q) {
    const float4 x = reinterpret_cast<const float4*>(p)[q];
    o[4 * q] = x.x; o[4 * q + 1] = x.y; o[4 * q + 2] = x.z; o[4 * q + 3] = x.w;
  }
}

template <typename Tin, int NCL, int NW, int ST, bool SAVED>
__global__ void __launch_bounds__(32 * NW, 1)
bwd_kernel(int T, int H, int chunk, int nchunks,
           const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
           const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
           const float* __restrict__ h0, const float* __restrict__ h_ckpt, const float* __restrict__ sa_in,
           const float* __restrict__ dy, const float* __restrict__ dhT,
           float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
           float* __restrict__ dv, float* __restrict__ da, float* __restrict__ db,
           float* __restrict__ dh0) {
  using L = BwdSmem<Tin, NCL, NW, ST>;
  constexpr int ROWS = L::ROWS, R = L::R, RP = R / 2, CPC = L::CPC;
  constexpr int kNT = 32 * NW, kNW = NW;
  static_assert(NCL == 1 || NCL == 2, "one or two row blocks per head");
  static_assert(R == 4 || R == 8, "4 or 8 rows per thread");
  static_assert(kCT % ST == 0, "sub-tiles divide the stage");
  constexpr int NV = 2 * R;              // values per lane in the row reductions (lookahead + dv)
  constexpr int REP = 32 / NV;           // lanes holding each reduced value

  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  float* sT = reinterpret_cast<float*>(sm + L::oTile);     // [7][kCT][kD]
  float* sV = reinterpret_cast<float*>(sm + L::oRowT);     // [kCT][ROWS]
  float* sDy = sV + kCT * ROWS;
  float* sSa = sDy + kCT * ROWS;
  float* sAb = reinterpret_cast<float*>(sm + L::oScal);    // [kCT]
  float* sRb = sAb + kCT;
  float* sDv = reinterpret_cast<float*>(sm + L::oDv);
  float* sSlab = reinterpret_cast<float*>(sm + L::oSlab);
  float* sPart = reinterpret_cast<float*>(sm + L::oPart);
  float* sRecv = reinterpret_cast<float*>(sm + L::oRecv);

  const int q = NCL > 1 ? (int)cluster_rank() : 0;
  const int bh = blockIdx.x / NCL;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int c0 = 2 * lane;             // this lane's columns c0, c0 + 1
  const int rloc = R * warp;           // first row of this warp within the CTA
  const int rbase = q * ROWS;
  const int grow = rbase + rloc;       // first head row of this thread
  const int ridx = rs32_index<NV>(lane);
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;

  // R rows x 2 columns of a D x D fp32 matrix as row pairs: X[p][c] = (row 2p, row 2p+1) at column c0 + c
  auto load_rows = [&](const float* src, float2 (&X)[RP][2]) {
#pragma unroll
    for (int p = 0; p < RP; ++p) {
      const float2 e = __ldg(reinterpret_cast<const float2*>(src + (size_t)(grow + 2 * p) * kD + c0));
      const float2 o = __ldg(reinterpret_cast<const float2*>(src + (size_t)(grow + 2 * p + 1) * kD + c0));
      X[p][0] = make_float2(e.x, o.x);
      X[p][1] = make_float2(e.y, o.y);
    }
  };

  // G: gradient w.r.t. the state after the last processed token (starts at dhT)
  float2 G[RP][2];
  if (dhT != nullptr) {
    load_rows(dhT + sbase, G);
  } else {
#pragma unroll
    for (int p = 0; p < RP; ++p) G[p][0] = G[p][1] = make_float2(0.f, 0.f);
  }

  if (nchunks > 0) {
    const int t0 = (nchunks - 1) * chunk;
    issue_stage<Tin, ROWS, kNT, SAVED>(sm, L::oV, L::oDy, L::oSa, t0, T - t0, base, tstride, rbase, w, k, a, b, r, v, dy,
                                  sa_in);
    cp_async_commit();
  }
  if (NCL > 1) {  // peers' shared memory is live before the first remote store
    cluster_arrive();
    cluster_wait();
  }

  float2 Sn[RP][2];  // checkpoint that starts the next chunk's walk (prefetched one chunk ahead)
  if (nchunks > 0) load_rows(h_ckpt + ((size_t)bh * nchunks + (nchunks - 1)) * kD * kD, Sn);

  bool pending = false;  // NCL == 2: a chunk's column sums wait for the exchange
  int pend_t0 = 0, pend_n = 0, pend_buf = 0;

  // sum own-column partials with the peer's and write them (NCL == 2)
  auto exchange_sum = [&]() {
    const float* rb = sRecv + (size_t)pend_buf * kNG * kCT * CPC;
    for (int e = tid; e < pend_n * kNG * (CPC / 4); e += kNT) {
      const int c4 = e % (CPC / 4);
      const int g = (e / (CPC / 4)) % kNG;
      const int s = e / ((CPC / 4) * kNG);
      const int o = (g * kCT + s) * CPC + 4 * c4;
      const float4 x = add4(*reinterpret_cast<const float4*>(sPart + o), *reinterpret_cast<const float4*>(rb + o));
      float* dst = pick(g, dr, dw, dk, db, da);
      *reinterpret_cast<float4*>(dst + base + (size_t)(pend_t0 + s) * tstride + q * CPC + 4 * c4) = x;
    }
  };

  for (int ci = nchunks - 1, it = 0; ci >= 0; --ci, ++it) {
    const int t0 = ci * chunk;
    const int n = min(chunk, T - t0);

    cp_async_wait<0>();
    __syncthreads();  // this chunk's raw stage has landed; the previous chunk's tiles are no longer read

    // ---- widen to fp32 tiles: 8 lanes per token (8 columns each)
    for (int tg = 0; tg < kCT; tg += kNT / 8) {
      const Tin* col = reinterpret_cast<const Tin*>(sm);
      const int tt = tg + (tid >> 3);
      const int c8 = (tid & 7) * 8;
      float ab = 0.f, rb = 0.f;
      if (tt < n) {
        float ww[8], kk[8], aa[8], bb[8], rr[8], bp[8], tmp[8];
        raw8(col + (0 * kCT + tt) * kD + c8, ww);
        raw8(col + (1 * kCT + tt) * kD + c8, kk);
        raw8(col + (2 * kCT + tt) * kD + c8, aa);
        raw8(col + (3 * kCT + tt) * kD + c8, bb);
        raw8(col + (4 * kCT + tt) * kD + c8, rr);
        if (tt > 0) {
          raw8(col + (3 * kCT + tt - 1) * kD + c8, bp);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) bp[u] = 0.f;
        }
        store8(sT + (TW * kCT + tt) * kD + c8, ww);
        store8(sT + (TK * kCT + tt) * kD + c8, kk);
        store8(sT + (TA * kCT + tt) * kD + c8, aa);
        store8(sT + (TB * kCT + tt) * kD + c8, bb);
        store8(sT + (TR * kCT + tt) * kD + c8, rr);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          tmp[u] = 1.0f / ww[u];
          ab = fmaf(aa[u], bp[u], ab);
          rb = fmaf(rr[u], bb[u], rb);
        }
        store8(sT + (TWI * kCT + tt) * kD + c8, tmp);
#pragma unroll
        for (int u = 0; u < 8; ++u) tmp[u] = ww[u] * bp[u];
        store8(sT + (TCB * kCT + tt) * kD + c8, tmp);
      }
#pragma unroll
      for (int m = 1; m < 8; m <<= 1) {
        ab += __shfl_xor_sync(0xffffffffu, ab, m);
        rb += __shfl_xor_sync(0xffffffffu, rb, m);
      }
      if (tt < n && (tid & 7) == 0) {
        sAb[tt] = ab;
        sRb[tt] = rb;
      }
    }
    {
      const Tin* vr = reinterpret_cast<const Tin*>(sm + L::oV);
      const float* dyr = reinterpret_cast<const float*>(sm + L::oDy);
      const float* sar = reinterpret_cast<const float*>(sm + L::oSa);
      for (int e = tid; e < n * ROWS; e += kNT) {
        sV[e] = to_f32(vr[e]);
        sDy[e] = dyr[e];
        if (SAVED) sSa[e] = sar[e];
      }
    }
    __syncthreads();  // tiles complete; the raw stage is free
    if (ci > 0) {
      issue_stage<Tin, ROWS, kNT, SAVED>(sm, L::oV, L::oDy, L::oSa, (ci - 1) * chunk, chunk, base, tstride, rbase, w, k, a,
                                    b, r, v, dy, sa_in);
      cp_async_commit();
    }

    // ---- walk start: the exact checkpoint after this chunk; prefetch the one before it
    float2 S[RP][2];
#pragma unroll
    for (int p = 0; p < RP; ++p) {
      S[p][0] = Sn[p][0];
      S[p][1] = Sn[p][1];
    }
    if (ci > 0) load_rows(h_ckpt + ((size_t)bh * nchunks + (ci - 1)) * kD * kD, Sn);

    if (!SAVED) {
      // ---- recompute sa_t over the chunk from its start state (h_ckpt[ci-1], h0 or zeros)
      float2 Rs[RP][2];
      if (ci > 0) {
#pragma unroll
        for (int p = 0; p < RP; ++p) {
          Rs[p][0] = Sn[p][0];
          Rs[p][1] = Sn[p][1];
        }
      } else if (h0 != nullptr) {
        load_rows(h0 + sbase, Rs);
      } else {
#pragma unroll
        for (int p = 0; p < RP; ++p) Rs[p][0] = Rs[p][1] = make_float2(0.f, 0.f);
      }
      for (int tt = 0; tt < n; ++tt) {
        const float2 a2 = *reinterpret_cast<const float2*>(sT + (TA * kCT + tt) * kD + c0);
        const float2 w2 = *reinterpret_cast<const float2*>(sT + (TW * kCT + tt) * kD + c0);
        const float2 k2 = *reinterpret_cast<const float2*>(sT + (TK * kCT + tt) * kD + c0);
        const float2 b2 = *reinterpret_cast<const float2*>(sT + (TB * kCT + tt) * kD + c0);
        float vv[R];
        lds_rows<R>(sV + tt * ROWS + rloc, vv);
        float x[NV];
#pragma unroll
        for (int p = 0; p < RP; ++p) {
          const float2 d = __ffma2_rn(Rs[p][1], bcast2(a2.y), __fmul2_rn(Rs[p][0], bcast2(a2.x)));
          x[2 * p] = d.x;
          x[2 * p + 1] = d.y;
          x[R + 2 * p] = x[R + 2 * p + 1] = 0.f;
        }
        const float u = rs32<NV>(x, lane);
        if (ridx < R && (lane & (REP - 1)) == 0) sSa[tt * ROWS + rloc + ridx] = u;
        float s4[R];
        ag32_low<R>(u, lane, s4);
#pragma unroll
        for (int p = 0; p < RP; ++p) {
          const float2 sp = make_float2(s4[2 * p], s4[2 * p + 1]);
          const float2 vp = make_float2(vv[2 * p], vv[2 * p + 1]);
          Rs[p][0] = __ffma2_rn(Rs[p][0], bcast2(w2.x), __ffma2_rn(vp, bcast2(k2.x), __fmul2_rn(sp, bcast2(b2.x))));
          Rs[p][1] = __ffma2_rn(Rs[p][1], bcast2(w2.y), __ffma2_rn(vp, bcast2(k2.y), __fmul2_rn(sp, bcast2(b2.y))));
        }
      }
      __syncwarp();  // each warp reads back only the sa rows it wrote
      // walk back from the recomputed end state: it is the state these sa values belong to (the stored
      // checkpoint carries the forward's own rounding, which the division by w below would amplify)
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        S[p][0] = Rs[p][0];
        S[p][1] = Rs[p][1];
      }
    }

    // ---- reverse walk over the chunk
    int tt = n - 1;
    float dyt[R];
    lds_rows<R>(sDy + tt * ROWS + rloc, dyt);
    float dsa[R];
    {
      // Gh_t = G + dy_t r_t^T, dsa_t = Gh_t b_t (direct; later tokens use the lookahead)
      const float2 r2 = *reinterpret_cast<const float2*>(sT + (TR * kCT + tt) * kD + c0);
      const float2 b2 = *reinterpret_cast<const float2*>(sT + (TB * kCT + tt) * kD + c0);
      float x[NV];
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        const float2 d2 = make_float2(dyt[2 * p], dyt[2 * p + 1]);
        G[p][0] = __ffma2_rn(d2, bcast2(r2.x), G[p][0]);
        G[p][1] = __ffma2_rn(d2, bcast2(r2.y), G[p][1]);
        const float2 d = __ffma2_rn(G[p][1], bcast2(b2.y), __fmul2_rn(G[p][0], bcast2(b2.x)));
        x[2 * p] = d.x;
        x[2 * p + 1] = d.y;
        x[R + 2 * p] = x[R + 2 * p + 1] = 0.f;
      }
      ag32_low<R>(rs32<NV>(x, lane), lane, dsa);
    }

    for (; tt >= 0; --tt) {
      const float* trow = sT + tt * kD + c0;
      const float2 w2 = *reinterpret_cast<const float2*>(trow + TW * kCT * kD);
      const float2 wi2 = *reinterpret_cast<const float2*>(trow + TWI * kCT * kD);
      const float2 k2 = *reinterpret_cast<const float2*>(trow + TK * kCT * kD);
      const float2 a2 = *reinterpret_cast<const float2*>(trow + TA * kCT * kD);
      const float2 b2 = *reinterpret_cast<const float2*>(trow + TB * kCT * kD);
      float vv[R], ss[R], dp[R];
      lds_rows<R>(sV + tt * ROWS + rloc, vv);
      lds_rows<R>(sSa + tt * ROWS + rloc, ss);
      const bool more = tt > 0;
      float2 cb2 = make_float2(0.f, 0.f), rp2 = cb2;
      float ab = 0.f, rb = 0.f;
      if (more) {
        cb2 = *reinterpret_cast<const float2*>(trow + TCB * kCT * kD);
        rp2 = *reinterpret_cast<const float2*>(trow - kD + TR * kCT * kD);
        lds_rows<R>(sDy + (tt - 1) * ROWS + rloc, dp);
        ab = sAb[tt];
        rb = sRb[tt - 1];
      } else {
#pragma unroll
        for (int i = 0; i < R; ++i) dp[i] = 0.f;
      }
      const float2 wb[2] = {bcast2(w2.x), bcast2(w2.y)}, wib[2] = {bcast2(wi2.x), bcast2(wi2.y)};
      const float2 kb[2] = {bcast2(k2.x), bcast2(k2.y)}, nkb[2] = {bcast2(-k2.x), bcast2(-k2.y)};
      const float2 ab2[2] = {bcast2(a2.x), bcast2(a2.y)}, bb[2] = {bcast2(b2.x), bcast2(b2.y)};
      const float2 nbb[2] = {bcast2(-b2.x), bcast2(-b2.y)}, cbb[2] = {bcast2(cb2.x), bcast2(cb2.y)};
      const float2 rpb[2] = {bcast2(rp2.x), bcast2(rp2.y)};

      // per column c (pairs over rows): partial column sums, reconstruction, lookahead and dv row
      // sums from Gh_t, state-gradient update
      float2 cdr[2], cdw[2], cdk[2], cdb[2], cda[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) cdr[c] = cdw[c] = cdk[c] = cdb[c] = cda[c] = make_float2(0.f, 0.f);
      float2 P[RP], PV[RP];
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        const float2 v2 = make_float2(vv[2 * p], vv[2 * p + 1]);
        const float2 s2 = make_float2(ss[2 * p], ss[2 * p + 1]);
        const float2 d2 = make_float2(dyt[2 * p], dyt[2 * p + 1]);
        const float2 q2 = make_float2(dsa[2 * p], dsa[2 * p + 1]);
        const float2 e2 = make_float2(dp[2 * p], dp[2 * p + 1]);
        P[p] = __ffma2_rn(G[p][1], cbb[1], __fmul2_rn(G[p][0], cbb[0]));
        PV[p] = __ffma2_rn(G[p][1], kb[1], __fmul2_rn(G[p][0], kb[0]));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          cdr[c] = __ffma2_rn(d2, S[p][c], cdr[c]);
          const float2 sp = __fmul2_rn(__ffma2_rn(s2, nbb[c], __ffma2_rn(v2, nkb[c], S[p][c])), wib[c]);
          S[p][c] = sp;
          cdw[c] = __ffma2_rn(G[p][c], sp, cdw[c]);
          cdk[c] = __ffma2_rn(G[p][c], v2, cdk[c]);
          cdb[c] = __ffma2_rn(G[p][c], s2, cdb[c]);
          cda[c] = __ffma2_rn(q2, sp, cda[c]);
          G[p][c] = __ffma2_rn(G[p][c], wb[c], __ffma2_rn(q2, ab2[c], __fmul2_rn(e2, rpb[c])));
        }
      }
      float x[NV];
#pragma unroll
      for (int p = 0; p < RP; ++p) {
        x[2 * p] = P[p].x;
        x[2 * p + 1] = P[p].y;
        x[R + 2 * p] = PV[p].x;
        x[R + 2 * p + 1] = PV[p].y;
      }
      const float u = rs32<NV>(x, lane);
      if (ridx >= R && (lane & (REP - 1)) == 0) sDv[tt * ROWS + rloc + ridx - R] = u;
      if (more) {
        float pn[R];
        ag32_low<R>(u, lane, pn);
#pragma unroll
        for (int i = 0; i < R; ++i) dsa[i] = fmaf(dsa[i], ab, fmaf(dp[i], rb, pn[i]));
      }
#pragma unroll
      for (int i = 0; i < R; ++i) dyt[i] = dp[i];

      // column partials over this thread's R rows -> the warp's slab
      {
        float* sl = sSlab + (size_t)((warp * ST + (tt % ST)) * kNG) * kD + c0;
        *reinterpret_cast<float2*>(sl + 0 * kD) = make_float2(cdr[0].x + cdr[0].y, cdr[1].x + cdr[1].y);
        *reinterpret_cast<float2*>(sl + 1 * kD) = make_float2(cdw[0].x + cdw[0].y, cdw[1].x + cdw[1].y);
        *reinterpret_cast<float2*>(sl + 2 * kD) = make_float2(cdk[0].x + cdk[0].y, cdk[1].x + cdk[1].y);
        *reinterpret_cast<float2*>(sl + 3 * kD) = make_float2(cdb[0].x + cdb[0].y, cdb[1].x + cdb[1].y);
        *reinterpret_cast<float2*>(sl + 4 * kD) = make_float2(cda[0].x + cda[0].y, cda[1].x + cda[1].y);
      }

      if (tt % ST == 0) {
        // ---- sub-tile [tt, thi) complete: sum the warps' slabs
        const int thi = min(tt + ST, n);
        __syncthreads();
        if (NCL > 1 && pending) {
          cluster_wait();
          exchange_sum();
          pending = false;
          __syncthreads();  // partials read before this chunk's sums overwrite them
        }
        const int buf = it & 1;
        for (int e = tid; e < (thi - tt) * kNG * (kD / 4); e += kNT) {
          const int c4 = e % (kD / 4);
          const int g = (e / (kD / 4)) % kNG;
          const int s = tt + e / ((kD / 4) * kNG);
          float4 acc = *reinterpret_cast<const float4*>(sSlab + (size_t)(((s % ST) * kNG) + g) * kD + 4 * c4);
#pragma unroll
          for (int wv = 1; wv < kNW; ++wv)
            acc = add4(acc, *reinterpret_cast<const float4*>(sSlab + (size_t)(((wv * ST + (s % ST)) * kNG) + g) * kD +
                                                             4 * c4));
          if (NCL == 1) {
            float* dst = pick(g, dr, dw, dk, db, da);
            *reinterpret_cast<float4*>(dst + base + (size_t)(t0 + s) * tstride + 4 * c4) = acc;
          } else {
            const int owner = (4 * c4) / CPC;
            const int cc = 4 * c4 - owner * CPC;
            if (owner == q) {
              *reinterpret_cast<float4*>(sPart + (g * kCT + s) * CPC + cc) = acc;
            } else {
              float* rp = sRecv + ((size_t)(buf * kNG + g) * kCT + s) * CPC + cc;
              st_cluster(peer_smem(rp, (unsigned)owner), acc);
            }
          }
        }
        // dv for the sub-tile (row sums, local to this CTA)
        for (int e = tid; e < (thi - tt) * (ROWS / 4); e += kNT) {
          const int s = tt + e / (ROWS / 4);
          const int c4 = e % (ROWS / 4);
          *reinterpret_cast<float4*>(dv + base + (size_t)(t0 + s) * tstride + rbase + 4 * c4) =
              *reinterpret_cast<const float4*>(sDv + s * ROWS + 4 * c4);
        }
        __syncthreads();  // slabs consumed before the next sub-tile writes them
        if (NCL > 1 && tt == 0) {
          cluster_arrive();  // this chunk's partials (local and remote) are in place
          pending = true;
          pend_t0 = t0;
          pend_n = n;
          pend_buf = buf;
        }
      }
    }
  }
  if (NCL > 1 && pending) {
    cluster_wait();
    exchange_sum();
  }

  if (dh0 != nullptr) {
#pragma unroll
    for (int p = 0; p < RP; ++p) {
      *reinterpret_cast<float2*>(dh0 + sbase + (size_t)(grow + 2 * p) * kD + c0) = make_float2(G[p][0].x, G[p][1].x);
      *reinterpret_cast<float2*>(dh0 + sbase + (size_t)(grow + 2 * p + 1) * kD + c0) =
          make_float2(G[p][0].y, G[p][1].y);
    }
  }
}

template <typename Tin, int NCL, int NW, int ST, bool SAVED>
cudaError_t launch_bwd_cfg(const BwdArgs& p, cudaStream_t stream) {
  using L = BwdSmem<Tin, NCL, NW, ST>;
  static_assert(L::kBytes <= 232448, "shared memory per CTA");
  auto kern = bwd_kernel<Tin, NCL, NW, ST, SAVED>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B * p.H * NCL);
  cfg.blockDim = dim3(32 * NW);
  cfg.dynamicSmemBytes = L::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NCL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = NCL > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p.T, p.H, p.chunk, p.nchunks, (const Tin*)p.in.r, (const Tin*)p.in.w,
                            (const Tin*)p.in.k, (const Tin*)p.in.v, (const Tin*)p.in.a, (const Tin*)p.in.b, p.h0,
                            p.h_ckpt, p.sa, p.dy, p.dhT, p.dr, p.dw, p.dk, p.dv, p.da, p.db, p.dh0);
}

template <typename Tin, bool SAVED>
cudaError_t launch_bwd_t(const BwdArgs& p, cudaStream_t stream) {
  // two row blocks per head when that still fits the GPU in one wave
  if ((long long)p.B * p.H * 2 <= num_sms()) return launch_bwd_cfg<Tin, 2, WKV7_BWD_NW2, WKV7_BWD_ST2, SAVED>(p, stream);
  return launch_bwd_cfg<Tin, 1, 8, 4, SAVED>(p, stream);
}

}  // namespace

cudaError_t launch_backward(const BwdArgs& p, cudaStream_t stream) {
  if (p.sa != nullptr)
    return p.bf16 ? launch_bwd_t<__nv_bfloat16, true>(p, stream) : launch_bwd_t<float, true>(p, stream);
  return p.bf16 ? launch_bwd_t<__nv_bfloat16, false>(p, stream) : launch_bwd_t<float, false>(p, stream);
}

WKV7_DEBUG_READER(debug_word_bwd)

}  // namespace wkv7
