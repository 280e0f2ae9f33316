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
// CTAs of a head forming a thread-block cluster.  Thread = 4 rows x 4 columns of S and
// of G in registers; the 16 lanes of a row group own the 64 columns, so row sums are
// 16-lane shuffles.  Column sums: each thread sums its 4 rows, the two row groups of a
// warp split the 20 partials by one exchange (10 shuffles), and every warp writes its
// 320 per-token partials to a slab in shared memory.  Every ST tokens the CTA sums the
// warps' slabs.  With NCL == 1 the sums go straight to HBM; with NCL == 2 each CTA owns
// half the columns: sums for its own columns stay in shared memory, the others are
// stored into the peer CTA's shared memory (distributed shared memory), and once per
// chunk, after a cluster barrier, each CTA adds the two halves and writes its columns.
// Deterministic: every sum is taken in a fixed order, no atomics.
//
// Staging.  The chunk's r, w, k, a, b, the CTA's slices of v, dy and sa are copied to
// shared memory with cp.async one chunk ahead (double-buffered); the checkpoint that
// starts the next chunk's walk is loaded into registers one chunk ahead.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kCT = 32;  // stage capacity in tokens (chunk <= 32)
constexpr int kNG = 5;   // column gradients in slab order: dr, dw, dk, db, da

constexpr size_t al16(size_t x) { return (x + 15) / 16 * 16; }

template <typename Tin, int NCL, int ST>
struct BwdSmem {
  static constexpr int ROWS = kD / NCL;
  static constexpr int NT = 4 * ROWS;
  static constexpr int NW = NT / 32;
  static constexpr int CPC = kD / NCL;  // columns of the column gradients this CTA writes
  // one input stage: Tin [5][kCT][kD] (w k a b r), Tin [kCT][ROWS] (v), f32 [kCT][ROWS] (dy, sa)
  static constexpr size_t oCol = 0;
  static constexpr size_t oV = oCol + al16(5 * kCT * kD * sizeof(Tin));
  static constexpr size_t oDy = oV + al16(kCT * ROWS * sizeof(Tin));
  static constexpr size_t oSa = oDy + kCT * ROWS * 4;
  static constexpr size_t kStage = oSa + kCT * ROWS * 4;
  // per-chunk tiles after the two stages
  static constexpr size_t oWinv = 2 * kStage;                    // f32 [kCT][kD]   1/w_t
  static constexpr size_t oCb = oWinv + kCT * kD * 4;            // f32 [kCT][kD]   w_t o b_{t-1}
  static constexpr size_t oAb = oCb + kCT * kD * 4;              // f32 [kCT]       a_t . b_{t-1}
  static constexpr size_t oRb = oAb + kCT * 4;                   // f32 [kCT]       r_t . b_t
  static constexpr size_t oDv = oRb + kCT * 4;                   // f32 [kCT][ROWS] dv
  static constexpr size_t oSlab = oDv + kCT * ROWS * 4;          // f32 [NW][ST][kNG][kD]
  static constexpr size_t oPart = oSlab + (size_t)NW * ST * kNG * kD * 4;             // f32 [kNG][kCT][CPC]
  static constexpr size_t oRecv = oPart + (NCL > 1 ? (size_t)kNG * kCT * CPC * 4 : 0);  // f32 [2][kNG][kCT][CPC]
  static constexpr size_t kBytes = oRecv + (NCL > 1 ? (size_t)2 * kNG * kCT * CPC * 4 : 0);
};

// cp.async copies of one chunk's inputs into a stage
template <typename Tin, int ROWS, int NT, bool SAVED>
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
    for (int e = threadIdx.x; e < n * CPR; e += NT) {
      const int tt = e / CPR, pc = e % CPR;
      cp_async16(col + (q * kCT + tt) * kD + pc * EPC, srcs[q] + base + (size_t)(t0 + tt) * tstride + pc * EPC);
    }
  }
  {
    constexpr int VPR = ROWS * (int)sizeof(Tin) / 16;
    Tin* dst = reinterpret_cast<Tin*>(stg + oV);
    for (int e = threadIdx.x; e < n * VPR; e += NT) {
      const int tt = e / VPR, pc = e % VPR;
      cp_async16(dst + tt * ROWS + pc * EPC, v + base + (size_t)(t0 + tt) * tstride + rbase + pc * EPC);
    }
  }
  {
    constexpr int FPR = ROWS / 4;
    float* ddy = reinterpret_cast<float*>(stg + oDy);
    float* dsa = reinterpret_cast<float*>(stg + oSa);
    for (int e = threadIdx.x; e < n * FPR; e += NT) {
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

template <typename Tin, int NCL, int ST, bool SAVED>
__global__ void __launch_bounds__(4 * (kD / NCL), 1)
bwd_kernel(int T, int H, int chunk, int nchunks,
           const Tin* __restrict__ r, const Tin* __restrict__ w, const Tin* __restrict__ k,
           const Tin* __restrict__ v, const Tin* __restrict__ a, const Tin* __restrict__ b,
           const float* __restrict__ h0, const float* __restrict__ h_ckpt, const float* __restrict__ sa_in,
           const float* __restrict__ dy, const float* __restrict__ dhT,
           float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
           float* __restrict__ dv, float* __restrict__ da, float* __restrict__ db,
           float* __restrict__ dh0) {
  using L = BwdSmem<Tin, NCL, ST>;
  constexpr int ROWS = L::ROWS, NT = L::NT, NW = L::NW, CPC = L::CPC;
  static_assert(NCL == 1 || NCL == 2, "one or two row blocks per head");
  static_assert(kCT % ST == 0, "sub-tiles divide the stage");

  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  float* sWinv = reinterpret_cast<float*>(sm + L::oWinv);
  float* sCb = reinterpret_cast<float*>(sm + L::oCb);
  float* sAb = reinterpret_cast<float*>(sm + L::oAb);
  float* sRb = reinterpret_cast<float*>(sm + L::oRb);
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
  const int l16 = tid & 15;
  const int j0 = 4 * l16;
  const int rloc = 4 * (tid >> 4);
  const int half = (tid >> 4) & 1;
  const int qrow = rs_row(l16);
  const int rbase = q * ROWS;
  const int grow = rbase + rloc;  // first head row of this thread
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;

  // G: gradient w.r.t. the state after the last processed token (starts at dhT)
  float2 G[4][2];
  if (dhT != nullptr) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(dhT + sbase + (size_t)(grow + i) * kD + j0));
      G[i][0] = lo2(x);
      G[i][1] = hi2(x);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) G[i][0] = G[i][1] = make_float2(0.f, 0.f);
  }

  if (nchunks > 0) {
    const int t0 = (nchunks - 1) * chunk;
    issue_stage<Tin, ROWS, NT, SAVED>(sm, L::oV, L::oDy, L::oSa, t0, T - t0, base, tstride, rbase, w, k, a, b, r, v,
                                      dy, sa_in);
    cp_async_commit();
  }
  if (NCL > 1) {  // peers' shared memory is live before the first remote store
    cluster_arrive();
    cluster_wait();
  }

  float4 Sn[4];  // checkpoint that starts the next chunk's walk (prefetched one chunk ahead)
  if (nchunks > 0) {
    const float* src = h_ckpt + ((size_t)bh * nchunks + (nchunks - 1)) * kD * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) Sn[i] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(grow + i) * kD + j0));
  }

  bool pending = false;  // NCL == 2: a chunk's column sums wait for the exchange
  int pend_t0 = 0, pend_n = 0, pend_buf = 0;

  // sum own-column partials with the peer's and write them (NCL == 2)
  auto exchange_sum = [&]() {
    const float* rb = sRecv + (size_t)pend_buf * kNG * kCT * CPC;
    for (int e = tid; e < pend_n * kNG * (CPC / 4); e += NT) {
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
    unsigned char* stg = sm + (size_t)(it & 1) * L::kStage;
    const Tin* cW = reinterpret_cast<const Tin*>(stg);
    const Tin* cK = cW + kCT * kD;
    const Tin* cA = cW + 2 * kCT * kD;
    const Tin* cB = cW + 3 * kCT * kD;
    const Tin* cR = cW + 4 * kCT * kD;
    const Tin* sV = reinterpret_cast<const Tin*>(stg + L::oV);
    const float* sDy = reinterpret_cast<const float*>(stg + L::oDy);
    float* sSa = reinterpret_cast<float*>(stg + L::oSa);

    cp_async_wait<0>();
    __syncthreads();  // this chunk's stage has landed; the other stage and the chunk tiles are free
    if (ci > 0) {
      issue_stage<Tin, ROWS, NT, SAVED>(sm + (size_t)((it + 1) & 1) * L::kStage, L::oV, L::oDy, L::oSa,
                                        (ci - 1) * chunk, chunk, base, tstride, rbase, w, k, a, b, r, v, dy, sa_in);
      cp_async_commit();
    }

    // ---- per-token column tiles: 1/w, w_t o b_{t-1}, a_t . b_{t-1}, r_t . b_t (8 lanes per token)
    for (int tg = warp * 4; tg < n; tg += NW * 4) {
      const int tt = tg + (lane >> 3);
      const int c8 = (lane & 7) * 8;
      float ab = 0.f, rb = 0.f;
      if (tt < n) {
        float ww[8], bb[8], aa[8], rr[8], bp[8], wi[8], cb[8];
        raw8(cW + tt * kD + c8, ww);
        raw8(cB + tt * kD + c8, bb);
        raw8(cA + tt * kD + c8, aa);
        raw8(cR + tt * kD + c8, rr);
        if (tt > 0) {
          raw8(cB + (tt - 1) * kD + c8, bp);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) bp[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          wi[u] = 1.0f / ww[u];
          cb[u] = ww[u] * bp[u];
          ab = fmaf(aa[u], bp[u], ab);
          rb = fmaf(rr[u], bb[u], rb);
        }
        store8(sWinv + tt * kD + c8, wi);
        store8(sCb + tt * kD + c8, cb);
      }
#pragma unroll
      for (int m = 1; m < 8; m <<= 1) {
        ab += __shfl_xor_sync(0xffffffffu, ab, m);
        rb += __shfl_xor_sync(0xffffffffu, rb, m);
      }
      if (tt < n && (lane & 7) == 0) {
        sAb[tt] = ab;
        sRb[tt] = rb;
      }
    }

    // ---- walk start: the exact checkpoint after this chunk; prefetch the one before it
    float2 S[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      S[i][0] = lo2(Sn[i]);
      S[i][1] = hi2(Sn[i]);
    }
    if (ci > 0) {
      const float* src = h_ckpt + ((size_t)bh * nchunks + (ci - 1)) * kD * kD;
#pragma unroll
      for (int i = 0; i < 4; ++i) Sn[i] = __ldg(reinterpret_cast<const float4*>(src + (size_t)(grow + i) * kD + j0));
    }

    if (!SAVED) {
      // ---- recompute sa_t over the chunk from its start state (h_ckpt[ci-1], h0 or zeros)
      float2 R[4][2];
      if (ci > 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          R[i][0] = lo2(Sn[i]);
          R[i][1] = hi2(Sn[i]);
        }
      } else if (h0 != nullptr) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(h0 + sbase + (size_t)(grow + i) * kD + j0));
          R[i][0] = lo2(x);
          R[i][1] = hi2(x);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) R[i][0] = R[i][1] = make_float2(0.f, 0.f);
      }
      for (int tt = 0; tt < n; ++tt) {
        float p[4], s4[4];
        dot4x4(R, raw4(cA + tt * kD + j0), p);
        const float z = reduce_scatter4(p, l16);
        if ((l16 & 3) == 0) sSa[tt * ROWS + rloc + qrow] = z;
        all_gather4(z, l16, s4);
        const float4 w4 = raw4(cW + tt * kD + j0);
        const float4 k4 = raw4(cK + tt * kD + j0);
        const float4 b4 = raw4(cB + tt * kD + j0);
        const float4 v4 = raw4(sV + tt * ROWS + rloc);
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          R[i][0] = __ffma2_rn(R[i][0], lo2(w4), __ffma2_rn(bcast2(vv[i]), lo2(k4), __fmul2_rn(bcast2(s4[i]), lo2(b4))));
          R[i][1] = __ffma2_rn(R[i][1], hi2(w4), __ffma2_rn(bcast2(vv[i]), hi2(k4), __fmul2_rn(bcast2(s4[i]), hi2(b4))));
        }
      }
    }
    __syncthreads();  // chunk tiles (and recomputed sa) complete

    // ---- reverse walk over the chunk
    int tt = n - 1;
    float4 dyt = *reinterpret_cast<const float4*>(sDy + tt * ROWS + rloc);
    float dsa[4];
    {
      // Gh_t = G + dy_t r_t^T, dsa_t = Gh_t b_t (direct; later tokens use the lookahead)
      const float4 r4 = raw4(cR + tt * kD + j0);
      const float dd[4] = {dyt.x, dyt.y, dyt.z, dyt.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        G[i][0] = __ffma2_rn(bcast2(dd[i]), lo2(r4), G[i][0]);
        G[i][1] = __ffma2_rn(bcast2(dd[i]), hi2(r4), G[i][1]);
      }
      float p[4];
      dot4x4(G, raw4(cB + tt * kD + j0), p);
      all_gather4(reduce_scatter4(p, l16), l16, dsa);
    }

    for (; tt >= 0; --tt) {
      const float4 w4 = raw4(cW + tt * kD + j0);
      const float4 wi4 = *reinterpret_cast<const float4*>(sWinv + tt * kD + j0);
      const float4 k4 = raw4(cK + tt * kD + j0);
      const float4 a4 = raw4(cA + tt * kD + j0);
      const float4 b4 = raw4(cB + tt * kD + j0);
      const float4 v4 = raw4(sV + tt * ROWS + rloc);
      const float4 sa4 = *reinterpret_cast<const float4*>(sSa + tt * ROWS + rloc);
      const bool more = tt > 0;
      float4 cb4 = make_float4(0.f, 0.f, 0.f, 0.f), rp4 = cb4, dyp = cb4;
      float ab = 0.f, rb = 0.f;
      if (more) {
        cb4 = *reinterpret_cast<const float4*>(sCb + tt * kD + j0);
        rp4 = raw4(cR + (tt - 1) * kD + j0);
        dyp = *reinterpret_cast<const float4*>(sDy + (tt - 1) * ROWS + rloc);
        ab = sAb[tt];
        rb = sRb[tt - 1];
      }
      const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
      const float ss[4] = {sa4.x, sa4.y, sa4.z, sa4.w};
      const float dd[4] = {dyt.x, dyt.y, dyt.z, dyt.w};
      const float dp[4] = {dyp.x, dyp.y, dyp.z, dyp.w};

      // lookahead row sums (dsa_{t-1}) and dv_t, both from Gh_t
      float P[4], pv[4];
      dot4x4(G, cb4, P);
      dot4x4(G, k4, pv);
      const float Pz = reduce_scatter4(P, l16);
      const float dvz = reduce_scatter4(pv, l16);
      if ((l16 & 3) == 0) sDv[tt * ROWS + rloc + qrow] = dvz;

      // column partials over this thread's 4 rows; reconstruction; state-gradient update
      float2 cdr[2], cdw[2], cdk[2], cdb[2], cda[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) cdr[h] = cdw[h] = cdk[h] = cdb[h] = cda[h] = make_float2(0.f, 0.f);
      const float2 w2[2] = {lo2(w4), hi2(w4)}, wi2[2] = {lo2(wi4), hi2(wi4)}, k2[2] = {lo2(k4), hi2(k4)};
      const float2 a2[2] = {lo2(a4), hi2(a4)}, b2[2] = {lo2(b4), hi2(b4)}, rp2[2] = {lo2(rp4), hi2(rp4)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          cdr[h] = __ffma2_rn(bcast2(dd[i]), S[i][h], cdr[h]);
          const float2 sp =
              __fmul2_rn(__ffma2_rn(bcast2(-ss[i]), b2[h], __ffma2_rn(bcast2(-vv[i]), k2[h], S[i][h])), wi2[h]);
          S[i][h] = sp;
          cdw[h] = __ffma2_rn(G[i][h], sp, cdw[h]);
          cdk[h] = __ffma2_rn(G[i][h], bcast2(vv[i]), cdk[h]);
          cdb[h] = __ffma2_rn(G[i][h], bcast2(ss[i]), cdb[h]);
          cda[h] = __ffma2_rn(bcast2(dsa[i]), sp, cda[h]);
          G[i][h] = __ffma2_rn(G[i][h], w2[h], __ffma2_rn(bcast2(dsa[i]), a2[h], __fmul2_rn(bcast2(dp[i]), rp2[h])));
        }
      }
      if (more) {
        float pn[4];
        all_gather4(Pz, l16, pn);
#pragma unroll
        for (int i = 0; i < 4; ++i) dsa[i] = fmaf(dsa[i], ab, fmaf(dp[i], rb, pn[i]));
      }
      dyt = dyp;

      // split the 20 column partials between the two row groups of the warp, then slab
      {
        const float s0[10] = {cdr[0].x, cdr[0].y, cdr[1].x, cdr[1].y, cdw[0].x, cdw[0].y, cdw[1].x, cdw[1].y,
                              cdk[0].x, cdk[0].y};
        const float s1[10] = {cdk[1].x, cdk[1].y, cdb[0].x, cdb[0].y, cdb[1].x, cdb[1].y,
                              cda[0].x, cda[0].y, cda[1].x, cda[1].y};
        float kp[10];
#pragma unroll
        for (int u = 0; u < 10; ++u) {
          const float mine = half ? s1[u] : s0[u];
          const float other = half ? s0[u] : s1[u];
          kp[u] = mine + __shfl_xor_sync(0xffffffffu, other, 16);
        }
        float* sl = sSlab + (size_t)((warp * ST + (tt % ST)) * kNG) * kD;
        if (!half) {
          *reinterpret_cast<float4*>(sl + 0 * kD + j0) = make_float4(kp[0], kp[1], kp[2], kp[3]);
          *reinterpret_cast<float4*>(sl + 1 * kD + j0) = make_float4(kp[4], kp[5], kp[6], kp[7]);
          *reinterpret_cast<float2*>(sl + 2 * kD + j0) = make_float2(kp[8], kp[9]);
        } else {
          *reinterpret_cast<float2*>(sl + 2 * kD + j0 + 2) = make_float2(kp[0], kp[1]);
          *reinterpret_cast<float4*>(sl + 3 * kD + j0) = make_float4(kp[2], kp[3], kp[4], kp[5]);
          *reinterpret_cast<float4*>(sl + 4 * kD + j0) = make_float4(kp[6], kp[7], kp[8], kp[9]);
        }
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
        for (int e = tid; e < (thi - tt) * kNG * (kD / 4); e += NT) {
          const int c4 = e % (kD / 4);
          const int g = (e / (kD / 4)) % kNG;
          const int s = tt + e / ((kD / 4) * kNG);
          float4 acc = *reinterpret_cast<const float4*>(sSlab + (size_t)(((s % ST) * kNG) + g) * kD + 4 * c4);
#pragma unroll
          for (int wv = 1; wv < NW; ++wv)
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
        for (int e = tid; e < (thi - tt) * (ROWS / 4); e += NT) {
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
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(dh0 + sbase + (size_t)(grow + i) * kD + j0) =
          make_float4(G[i][0].x, G[i][0].y, G[i][1].x, G[i][1].y);
  }
}

template <typename Tin, int NCL, int ST, bool SAVED>
cudaError_t launch_bwd_cfg(const BwdArgs& p, cudaStream_t stream) {
  using L = BwdSmem<Tin, NCL, ST>;
  auto kern = bwd_kernel<Tin, NCL, ST, SAVED>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B * p.H * NCL);
  cfg.blockDim = dim3(L::NT);
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
  if ((long long)p.B * p.H * 2 <= num_sms()) {
    return launch_bwd_cfg<Tin, 2, 8, SAVED>(p, stream);
  }
  // (fp32 inputs double the stage: a shorter sub-tile keeps the CTA within shared memory)
  if constexpr (sizeof(Tin) == 2) {
    return launch_bwd_cfg<Tin, 1, 8, SAVED>(p, stream);
  } else {
    return launch_bwd_cfg<Tin, 1, 4, SAVED>(p, stream);
  }
}

}  // namespace

cudaError_t launch_backward(const BwdArgs& p, cudaStream_t stream) {
  if (p.sa != nullptr)
    return p.bf16 ? launch_bwd_t<__nv_bfloat16, true>(p, stream) : launch_bwd_t<float, true>(p, stream);
  return p.bf16 ? launch_bwd_t<__nv_bfloat16, false>(p, stream) : launch_bwd_t<float, false>(p, stream);
}

}  // namespace wkv7
