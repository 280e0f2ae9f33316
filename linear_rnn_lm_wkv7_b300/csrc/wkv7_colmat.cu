// WKV7 backward: the column gradients dr, dw, dk, da, db of every 32-token chunk at once, in matrix
// form on tensor cores.
//
// Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel architecture", Backward
// listing (chunks walked in reverse from the exact checkpoints; VJP for dr, dw, dk, dv, da, db).  With
// X_t the gradient w.r.t. the state after token t (including dy_t r_t^T) and S_t the state:
//     dr_t = S_t^T dy_t,  dk_t = X_t^T v_t,  db_t = X_t^T sa_t,  da_t = S_{t-1}^T dsa_t,
//     dw_t = colsum(X_t o S_{t-1}),  dsa_t = X_t b_t,  X_{t-1} = X_t diag(w_t) + dsa_t a_t^T + dy_{t-1} r_{t-1}^T.
// The walk over the chunks (wkv7_xop.cu) leaves G at every chunk end (the gradient w.r.t. the state
// after the chunk from every later token, X_e = G + dy_{n-1} r_{n-1}^T; 64 x 64 fp32 in mma accumulator
// order, acc_order in wkv7_mma.cuh) and dh0.
//
// Matrix form of one chunk of n tokens (t = 0..31, steps past n padded with w = 1 and zeros), from S0
// (the state before the chunk), G and S_e (the state after it), with gamma, A^, R^, K~, B~, M_ab, M_ak,
// M_rb, M_rk and T = (I - M_ab)^-1 as in the transition-chain kernels and Xb = G diag(gamma_{n-1}):
//     SA  = T U,    U = A^ S0^T + M_ak V                      (rows t: sa_t, recomputed)
//     DSA = T^T W,  W = B~ Xb^T + M_rb^T DY                   (rows t: dsa_t)
//     L1 = tril(DY V^T), L2 = tril(DY SA^T), L3 = tril(DSA V^T, -1), L4 = tril(DSA SA^T, -1)
//     DR = Gamma   o (DY  S0 + L1 K~ + L2 B~)
//     DA = Gamma_- o (DSA S0 + L3 K~ + L4 B~)                 (Gamma_- row t = gamma_{t-1})
//     DK = Gamma^-1 o (V  Xb + L3^T A^ + L1^T R^)
//     DB = Gamma^-1 o (SA Xb + L4^T A^ + L2^T R^)
//     DV = K~ Xb^T + M_ak^T DSA + M_rk^T DY                  (rows t: dv_t)
// (X_t diag(gamma_t) and S_t diag(1/gamma_t) unrolled over the chunk: every column sum above becomes a
// dot of the chunk's own vectors, masked to the tokens before or after t).  dw follows per column
// from Z_t = colsum(X_t o S_t): Z_{n-1} = colsum(G o S_e) + r_{n-1} o dr_{n-1}, w_t o dw_t = Z_t - k_t o dk_t - b_t o db_t,
// Z_{t-1} = w_t o dw_t + a_t o da_t + r_{t-1} o dr_{t-1}.  No state is divided by w.
//
// A chunk whose gamma_31 falls below 1e-20 in some column (or above 1e37, or is not finite), or that
// has some w_t below 1/32 (where dividing w_t o dw_t by w_t would cost digits), takes the exact
// token-by-token column passes instead (sa, dsa and dv by their own recurrences, then wkv7_colpass.cuh).
//
// Precision: products of fp32 operands as three bf16 products (hi hi + hi lo + lo hi, ~2^-17 each),
// fp32 accumulation; operands are stored once, row-major, split into bf16 hi and lo, and read with
// ldmatrix (.trans for the transposed uses).  Mapping: one CTA of 8 warps per SM (its shared memory),
// looping over the (head, chunk) jobs; the next chunk's loads are in flight during the current one's dw.
#include <type_traits>

#include "wkv7_colpass.cuh"
#include "wkv7_device.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace {

using namespace mma;

constexpr int kL = 32;
constexpr int kNT = 256;
constexpr int kNW = kNT / 32;
constexpr int kLD64 = 72;  // row stride (bf16 elements) of 64-wide operands
constexpr int kLD32 = 40;  // of 32-wide operands
constexpr float kMinGamma = 1e-20f;
constexpr float kMaxGamma = 1e37f;  // (1 / gamma by __fdividef, exact to a few ulp below 2^126)
constexpr float kWMin = 0.03125f;

__host__ __device__ constexpr int rm_bytes(int rows, int ld) { return 2 * rows * ld * 2; }  // hi + lo

template <typename Tin>
struct Lay {
  // ---- long-lived
  static constexpr int kGL = 64 + 8;                            // gamma row stride (floats): padded so that a
                                                                // warp's reads of eight rows hit distinct banks
  static constexpr int oG = 0;                                  // float [32][kGL] gamma
  static constexpr int oZP = oG + 32 * kGL * 4;                 // float [64] colsum(G o S_e)
  static constexpr int oBT = oZP + 64 * 4;                      // float [4][64] block totals of the scans
  static constexpr int oMeta = oBT + 4 * 64 * 4;                // int [8]
  static constexpr int oWc = oMeta + 256;                       // float [32][64] w (1 past n)
  static constexpr int oAh = oWc + 32 * 64 * 4;
  static constexpr int oBt = oAh + rm_bytes(32, kLD64);
  static constexpr int oKt = oBt + rm_bytes(32, kLD64);
  static constexpr int oRh = oKt + rm_bytes(32, kLD64);
  static constexpr int oS0 = oRh + rm_bytes(32, kLD64);
  static constexpr int oXb = oS0 + rm_bytes(64, kLD64);
  static constexpr int oV = oXb + rm_bytes(64, kLD64);
  static constexpr int oDY = oV + rm_bytes(32, kLD64);
  static constexpr int oSA = oDY + rm_bytes(32, kLD64);
  static constexpr int oDSA = oSA + rm_bytes(32, kLD64);
  static constexpr int oB = oDSA + rm_bytes(32, kLD64);
  // ---- phase scratch B: raw inputs first (w, k, a, b, r, v [32][64] Tin; dy fp32 [32][64]) ...
  static constexpr int oRaw = oB;
  static constexpr int kRawIn = 6 * kL * kD * (int)sizeof(Tin);
  static constexpr int oDyRaw = oRaw + kRawIn;
  static constexpr int kRawEnd = oDyRaw + kL * kD * 4;
  // ... then M_ak, M_rk, M_rb, T, U, W, M_ab (fp32), TI, E; then L1..L4 over U, W and M_ab
  static constexpr int oMak = oB;
  static constexpr int oMrk = oMak + rm_bytes(32, kLD32);
  static constexpr int oMrb = oMrk + rm_bytes(32, kLD32);
  static constexpr int oT = oMrb + rm_bytes(32, kLD32);
  static constexpr int oU = oT + rm_bytes(32, kLD32);
  static constexpr int oW = oU + rm_bytes(32, kLD64);
  static constexpr int kSM = 36;
  static constexpr int oMab = oW + rm_bytes(32, kLD64);         // float [32][36]
  static constexpr int oTI = oMab + 32 * kSM * 4;               // float [32][36]
  static constexpr int oE = oTI + 32 * kSM * 4;                 // float [16][16]
  static constexpr int kPhaseEnd = oE + 16 * 16 * 4;
  static constexpr int oL = oU;                                 // L1..L4 (32 x 32 each)
  static_assert(oL + 4 * rm_bytes(32, kLD32) <= oTI, "L1..L4 fit over U, W and M_ab");
  static constexpr int kMain = (kRawEnd > kPhaseEnd ? kRawEnd : kPhaseEnd);
  // ---- fp32 S0 and G [64][64] staged by cp.async (through P1b).  S_e [64][kSL] fp32 is staged over SA and
  // DSA (first written in P5).
  static constexpr int oS0f = (kMain + 127) / 128 * 128;
  static constexpr int oGf = oS0f + kD * kD * 4;
  static constexpr int oSef = oSA;
  static constexpr int kSL = kD + 8;  // S_e row stride (floats): padded so a warp's rows fall in distinct banks
  static_assert(oSef + kD * kSL * 4 <= oB, "S_e fits over SA and DSA");
  static constexpr int kBytes = oGf + kD * kD * 4;
  // ---- (matrices from the forward) M_ak, M_rb, M_rk, T, loaded with S0, G and S_e
  static constexpr int oM = kBytes;
  static constexpr int kBytesM = oM + 4 * rm_bytes(32, kLD32);
  // ---- r o dr, a o da, k o dk, b o db, fp32 [32][kTL] each, over A^ .. (after the last products); rows
  // padded so that the eight rows of a warp's stores fall in distinct banks
  static constexpr int kTL = kD + 8;
  static constexpr int oStage = oAh;
  static_assert(oStage + 4 * kL * kTL * 4 <= oV, "dw terms fit over A^ .. Xb");
};

// FM: M_ak, M_rb, M_rk and T come from the forward's operator blocks (`mats`, at the blocks' stride of
// xck_stride floats) instead of being formed here (no M_ab, no inverse).  The forward formed them in
// closed form for every chunk whose gamma_31 passes the same test as here (in [1e-20, 1e37]), a
// superset of the chunks this kernel takes in matrix form.
template <typename Tin, bool FM>
__global__ void __launch_bounds__(kNT, 1)
colmat_kernel(int T, int H, int nchunks, int total, const Tin* __restrict__ r, const Tin* __restrict__ w,
              const Tin* __restrict__ k, const Tin* __restrict__ v, const Tin* __restrict__ a,
              const Tin* __restrict__ b, const float* __restrict__ h0, const float* __restrict__ h_ckpt,
              const float* __restrict__ dy, const float* __restrict__ xck, int* __restrict__ flags, size_t xck_stride,
              const unsigned char* __restrict__ mats, float* __restrict__ dr,
              float* __restrict__ dw, float* __restrict__ dk, float* __restrict__ dv, float* __restrict__ da,
              float* __restrict__ db) {
  using LY = Lay<Tin>;
  constexpr bool kVExact = sizeof(Tin) == 2;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const size_t tstride = (size_t)H * kD;

  float* G = reinterpret_cast<float*>(sm + LY::oG);
  float* Wc = reinterpret_cast<float*>(sm + LY::oWc);
  float* ZP = reinterpret_cast<float*>(sm + LY::oZP);
  int* meta = reinterpret_cast<int*>(sm + LY::oMeta);
  Tin* raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  const Tin* rw = raw;
  const Tin* rk = raw + kL * kD;
  const Tin* ra = raw + 2 * kL * kD;
  const Tin* rbv = raw + 3 * kL * kD;
  const Tin* rr = raw + 4 * kL * kD;
  const Tin* rv = raw + 5 * kL * kD;
  float* dyr = reinterpret_cast<float*>(sm + LY::oDyRaw);
  auto bfp = [&](int off) { return reinterpret_cast<__nv_bfloat16*>(sm + off); };
  const RM Ah{bfp(LY::oAh), 32 * kLD64, kLD64}, Bt{bfp(LY::oBt), 32 * kLD64, kLD64};
  const RM Kt{bfp(LY::oKt), 32 * kLD64, kLD64}, Rh{bfp(LY::oRh), 32 * kLD64, kLD64};
  const RM S0{bfp(LY::oS0), 64 * kLD64, kLD64}, Xb{bfp(LY::oXb), 64 * kLD64, kLD64};
  const RM Vm{bfp(LY::oV), 32 * kLD64, kLD64}, DY{bfp(LY::oDY), 32 * kLD64, kLD64};
  const RM SA{bfp(LY::oSA), 32 * kLD64, kLD64}, DSA{bfp(LY::oDSA), 32 * kLD64, kLD64};
  const RM U{bfp(LY::oU), 32 * kLD64, kLD64}, W{bfp(LY::oW), 32 * kLD64, kLD64};
  constexpr int kRM32 = rm_bytes(32, kLD32);
  const RM Mak{bfp(FM ? LY::oM : LY::oMak), 32 * kLD32, kLD32};
  const RM Mrb{bfp(FM ? LY::oM + kRM32 : LY::oMrb), 32 * kLD32, kLD32};
  const RM Mrk{bfp(FM ? LY::oM + 2 * kRM32 : LY::oMrk), 32 * kLD32, kLD32};
  const RM Tm{bfp(FM ? LY::oM + 3 * kRM32 : LY::oT), 32 * kLD32, kLD32};
  const RM L1{bfp(LY::oL), 32 * kLD32, kLD32}, L2{bfp(LY::oL + rm_bytes(32, kLD32)), 32 * kLD32, kLD32};
  const RM L3{bfp(LY::oL + 2 * rm_bytes(32, kLD32)), 32 * kLD32, kLD32};
  const RM L4{bfp(LY::oL + 3 * rm_bytes(32, kLD32)), 32 * kLD32, kLD32};
  float* Mab = reinterpret_cast<float*>(sm + LY::oMab);
  float* TI = reinterpret_cast<float*>(sm + LY::oTI);
  float* E = reinterpret_cast<float*>(sm + LY::oE);
  constexpr int SM = LY::kSM;

  // ---- P0: a chunk's inputs (rows past n are not copied) in one cp.async group, S0, G and S_e in a second.
  // The CTA loops over chunks blockIdx.x, + gridDim.x, ...; the next chunk's groups are issued once the
  // current chunk's raw, staging and SA / DSA regions are dead (after its output products).
  auto issue = [&](int jb) {
    const int ci_ = jb % nchunks, bh_ = jb / nchunks;
    const int bi_ = bh_ / H, hi_ = bh_ - bi_ * H;
    const int t0_ = ci_ * kL, n_ = min(kL, T - t0_);
    const size_t base_ = ((size_t)bi_ * T * H + hi_) * kD;
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    const Tin* srcs[6] = {w, k, a, b, r, v};
#pragma unroll
    for (int s6 = 0; s6 < 6; ++s6)
      for (int e = tid; e < n_ * CPR; e += kNT) {
        const int tt = e / CPR, pc = e % CPR;
        cp_async16(raw + (s6 * kL + tt) * kD + pc * EPC, srcs[s6] + base_ + (size_t)(t0_ + tt) * tstride + pc * EPC);
      }
    for (int e = tid; e < n_ * (kD / 4); e += kNT) {
      const int tt = e / (kD / 4), pc = e % (kD / 4);
      cp_async16(dyr + tt * kD + pc * 4, dy + base_ + (size_t)(t0_ + tt) * tstride + pc * 4);
    }
    cp_async_commit();
    const float* gend_ = xck + ((size_t)bh_ * nchunks + ci_) * xck_stride;
    const float* send_ = h_ckpt + ((size_t)bh_ * nchunks + ci_) * kD * kD;
    const float* s0_ = ci_ > 0 ? h_ckpt + ((size_t)bh_ * nchunks + ci_ - 1) * kD * kD
                               : (h0 != nullptr ? h0 + (size_t)bh_ * kD * kD : nullptr);
    float* s0f = reinterpret_cast<float*>(sm + LY::oS0f);
    float* gf = reinterpret_cast<float*>(sm + LY::oGf);
    float* sef = reinterpret_cast<float*>(sm + LY::oSef);
    for (int e = tid; e < kD * kD / 4; e += kNT) {
      if (s0_ != nullptr) cp_async16(s0f + 4 * e, s0_ + 4 * e);
      cp_async16(gf + 4 * e, gend_ + 4 * e);
      cp_async16(sef + (e >> 4) * LY::kSL + 4 * (e & 15), send_ + 4 * e);
    }
    if (FM) {  // the four matrices in this kernel's operand layout (rows of kLD32 elements), as stored
      const unsigned char* msrc = mats + ((size_t)bh_ * nchunks + ci_) * xck_stride * 4;
      for (int e = tid; e < 4 * kRM32 / 16; e += kNT) cp_async16(sm + LY::oM + e * 16, msrc + e * 16);
    }
    cp_async_commit();
  };
  if (blockIdx.x < total) issue(blockIdx.x);

  for (int job = blockIdx.x; job < total; job += gridDim.x) {
  const int ci = job % nchunks;
  const int bh = job / nchunks;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int t0 = ci * kL;
  const int n = min(kL, T - t0);
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const float* s0 = ci > 0 ? h_ckpt + ((size_t)bh * nchunks + ci - 1) * kD * kD
                           : (h0 != nullptr ? h0 + (size_t)bh * kD * kD : nullptr);
  const int next = job + gridDim.x;
  cp_async_wait<1>();  // this chunk's inputs
  __syncthreads();

  // ---- P1a: gamma_t down each column as a scan (4 blocks of 8 tokens per column); the fallback flag
  float* BT = reinterpret_cast<float*>(sm + LY::oBT);
  {  // threads 0-255 (whole warps): column j, tokens 8 blk .. 8 blk + 7
    const int j = tid & 63, blk = tid >> 6;
    const bool act = tid < 256;
    float loc[8];
    float p = 1.f;
    bool bad = false;
    if (act) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = 8 * blk + u;
        const float wt = t < n ? to_f32(rw[t * kD + j]) : 1.f;
        bad |= !(wt >= kWMin);
        p *= wt;
        loc[u] = p;
        Wc[t * kD + j] = wt;
      }
      if (WKV7_IN(blk, 4, dbg::kColmat)) BT[blk * 64 + j] = p;
    }
    __syncthreads();
    if (act) {
      float pre = 1.f;
      for (int q2 = 0; q2 < blk; ++q2) pre *= BT[q2 * 64 + j];
#pragma unroll
      for (int u = 0; u < 8; ++u) G[(8 * blk + u) * LY::kGL + j] = pre * loc[u];
      if (blk == 3) {
        const float gm = pre * p;
        bad |= !(gm >= kMinGamma) || !(gm <= kMaxGamma);
      }
    }
    const unsigned any = __ballot_sync(0xffffffffu, bad);
    if (lane == 0 && warp < 8) meta[warp] = any != 0u;
  }
  __syncthreads();
  {  // chunks with tiny decays are left to colfb_kernel (token by token); the flag tells it which
    const bool flagged = (meta[0] | meta[1] | meta[2] | meta[3] | meta[4] | meta[5] | meta[6] | meta[7]) != 0;
    if (tid == 0 && WKV7_IN(ci, nchunks, dbg::kColmat)) flags[((size_t)bh * nchunks + ci) * xck_stride] = flagged ? 1 : 0;
    if (flagged) {
      cp_async_wait<0>();
      __syncthreads();  // every thread's copies have landed before the next chunk's land in the same places
      if (next < total) issue(next);
      continue;
    }
  }

  // ---- P1b: operands, one (token, 8 columns) block per thread: A^, R^, K~, B~, V, DY (steps past n zero)
  if (tid < 256) {
    const int t = tid >> 3, c0 = (tid & 7) * 8;
    const bool ok = t < n;
    float gt[8], gp[8], av[8], rv8[8], kv[8], bv[8], vv[8], dv8[8];
    raw8(G + t * LY::kGL + c0, gt);
    if (t > 0) {
      raw8(G + (t - 1) * LY::kGL + c0, gp);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) gp[u] = 1.f;
    }
    raw8(ra + t * kD + c0, av);
    raw8(rr + t * kD + c0, rv8);
    raw8(rk + t * kD + c0, kv);
    raw8(rbv + t * kD + c0, bv);
    raw8(rv + t * kD + c0, vv);
    raw8(dyr + t * kD + c0, dv8);
    float oa[8], orr[8], ok8[8], ob[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float ig = __fdividef(1.f, gt[u]);  // (the forward's operator kernel forms K~, B~ the same way)
      oa[u] = ok ? av[u] * gp[u] : 0.f;
      orr[u] = ok ? rv8[u] * gt[u] : 0.f;
      ok8[u] = ok ? kv[u] * ig : 0.f;
      ob[u] = ok ? bv[u] * ig : 0.f;
      vv[u] = ok ? vv[u] : 0.f;
      dv8[u] = ok ? dv8[u] : 0.f;
    }
    rm_store8(Ah, t, c0, oa);
    rm_store8(Rh, t, c0, orr);
    rm_store8(Kt, t, c0, ok8);
    rm_store8(Bt, t, c0, ob);
    if (kVExact) rm_store8_hi(Vm, t, c0, vv); else rm_store8(Vm, t, c0, vv);
    rm_store8(DY, t, c0, dv8);
  }
  cp_async_wait<0>();  // S0, G, S_e
  __syncthreads();
  // Xb = G diag(gamma_{n-1}) and colsum(G o S_e): warp w takes G's accumulator tiles (m-tile 0-3, n-tile w) in
  // their stored order, one float4 per lane -- (i, j), (i, j + 1), (i + 8, j), (i + 8, j + 1) -- and sums its
  // column pair over the rows by shuffles
  static_assert(kNW == 8, "one n-tile of G per warp");
  {
    const float4* gf4 = reinterpret_cast<const float4*>(sm + LY::oGf);
    const float* sef = reinterpret_cast<const float*>(sm + LY::oSef);
    const int j = warp * 8 + 2 * q;
    const float2 gl = *reinterpret_cast<const float2*>(G + (n - 1) * LY::kGL + j);
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int i = mt * 16 + g;
      const float4 x = gf4[(mt * 8 + warp) * 32 + lane];
      rm_store(Xb, i, j, x.x * gl.x, x.y * gl.y);
      rm_store(Xb, i + 8, j, x.z * gl.x, x.w * gl.y);
      const float2 e0 = *reinterpret_cast<const float2*>(sef + i * LY::kSL + j);
      const float2 e8 = *reinterpret_cast<const float2*>(sef + (i + 8) * LY::kSL + j);
      z0 = fmaf(x.x, e0.x, fmaf(x.z, e8.x, z0));
      z1 = fmaf(x.y, e0.y, fmaf(x.w, e8.y, z1));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      z0 += __shfl_xor_sync(0xffffffffu, z0, o);
      z1 += __shfl_xor_sync(0xffffffffu, z1, o);
    }
    if (g == 0 && WKV7_IN(j + 1, kD, dbg::kColmat)) {
      ZP[j] = z0;
      ZP[j + 1] = z1;
    }
  }
  {  // S0 (rows i, columns j)
    const float* s0f = reinterpret_cast<const float*>(sm + LY::oS0f);
#pragma unroll 4
    for (int e = tid; e < kD * (kD / 2); e += kNT) {
      const int i = e >> 5, j = 2 * (e & 31);
      const float2 s = s0 != nullptr ? *reinterpret_cast<const float2*>(s0f + i * kD + j) : make_float2(0.f, 0.f);
      rm_store(S0, i, j, s.x, s.y);
    }
  }
  __syncthreads();

  if constexpr (!FM) {  // (from the forward: loaded instead)
  // ---- P2: M_ab = tril(A^ B~^T, -1) (fp32), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T),
  // M_rk = tril(R^ K~^T); 16 jobs of (product, m-tile, pair of n-tiles), K = 64
  // warp w forms jobs w and w + 8 together: the same tile of (M_ab, M_rb) or (M_ak, M_rk), sharing B~ or K~
  static_assert(kNW == 8, "job pairing assumes 8 warps");
  {
    const int prodA = warp >> 2, mt = (warp >> 1) & 1, np = warp & 1;  // prodB = prodA + 2
    float acc[2][2][4] = {};
    if (!(mt == 0 && np == 1)) {  // rows 0-15 x columns 16-31: above the diagonal
      const RM& Y = (prodA & 1) ? Kt : Bt;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const FragA fa0 = rm_a(Ah, mt, kk, lane), fa1 = rm_a(Rh, mt, kk, lane);
        FragB fb[2];
        rm_b2(Y, 2 * np, kk, lane, fb[0], fb[1]);
        mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
      }
    }
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      const int prod = prodA + 2 * jb;
      const bool strict = prod < 2;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nj = 2 * np + h;
        const int tr = mt * 16 + g, sc = nj * 8 + 2 * q;
        float c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = tr + ((e >> 1) << 3), s2 = sc + (e & 1);
          c[e] = (strict ? s2 < t : s2 <= t) ? acc[jb][h][e] : 0.f;
        }
        if (prod == 0) {
          *reinterpret_cast<float2*>(Mab + tr * SM + sc) = make_float2(c[0], c[1]);
          *reinterpret_cast<float2*>(Mab + (tr + 8) * SM + sc) = make_float2(c[2], c[3]);
        } else {
          rm_store_acc(prod == 1 ? Mak : (prod == 2 ? Mrb : Mrk), mt, nj, lane, c);
        }
      }
    }
  }
  __syncthreads();
  }

  // ---- P3 || P4: warp 0 solves the diagonal blocks of T = (I - M_ab)^-1 (forward substitution, one column
  // per lane: lanes 0-15 T11, lanes 16-31 T22); the other warps form U = A^ S0^T + M_ak V and
  // W = B~ Xb^T + M_rb^T DY (rows t, columns i): 16 jobs of (product, m-tile, 4 n-tiles)
  // (from the forward: T is loaded, and all eight warps form U and W, each warp both m-tiles of one pair of
  // n-tiles so that the two share their right operands: warps 0-3 U, 4-7 W)
  if constexpr (FM) {
    const int pg = warp >> 2, nq = warp & 3;  // n-tiles 2nq, 2nq + 1
    float acc[2][2][4] = {};                 // [m-tile][n-tile]
    const RM& A1 = pg == 0 ? Ah : Bt;
    const RM& B1 = pg == 0 ? S0 : Xb;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      FragB fb[2];
      rm_b2(B1, 2 * nq, kk, lane, fb[0], fb[1]);
      const FragA fa0 = rm_a(A1, 0, kk, lane), fa1 = rm_a(A1, 1, kk, lane);
      mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
    }
    // U: M_ak V (V is B[k = u][n = i] = V[u][i]); W: M_rb^T DY.  Blocks above the diagonal are zero:
    // M_ak rows 0-15 at columns 16-31 (m-tile 0, k-tile 1), M_rb^T rows 16-31 at 0-15 (m-tile 1, k-tile 0)
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const bool on0 = pg == 0 ? kk == 0 : true, on1 = pg == 0 ? true : kk == 1;
      FragB fb[2];
      FragA fa0, fa1;
      if (pg == 0) {
        rm_bt2(Vm, 2 * nq, kk, lane, fb[0], fb[1], !kVExact);
        fa0 = rm_a(Mak, 0, kk, lane);
        fa1 = rm_a(Mak, 1, kk, lane);
      } else {
        rm_bt2(DY, 2 * nq, kk, lane, fb[0], fb[1]);
        fa0 = rm_at(Mrb, 0, kk, lane);
        fa1 = rm_at(Mrb, 1, kk, lane);
      }
      if (pg == 0 && kVExact) {
        if (on0) {
          mma2b(acc[0][0], fa0, fb[0]);
          mma2b(acc[0][1], fa0, fb[1]);
        }
        mma2b(acc[1][0], fa1, fb[0]);
        mma2b(acc[1][1], fa1, fb[1]);
      } else if (on0 && on1) {
        mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
      } else if (on0) {
        mma3n<2>(acc[0], fa0, fb);
      } else {
        mma3n<2>(acc[1], fa1, fb);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) rm_store_acc(pg == 0 ? U : W, mt, 2 * nq + h, lane, acc[mt][h]);
  } else if (warp == 0) {
    const int off = lane < 16 ? 0 : 16;
    const int c = lane & 15;
    float x[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float acc = t == c ? 1.f : 0.f;
#pragma unroll
      for (int u = 0; u < t; ++u) acc = fmaf(Mab[(off + t) * SM + off + u], x[u], acc);
      x[t] = acc;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) TI[(off + t) * SM + off + c] = x[t];
    __syncwarp();
    tri_inverse_t21(Mab, TI, SM, lane);  // T21 = T22 A21 T11 (A21 = M_ab[16..31][0..15])
  } else {
    for (int job = warp - 1; job < 16; job += kNW - 1) {
      const int prod = job >> 3, mt = (job >> 2) & 1, nq = job & 3;  // n-tiles 2nq, 2nq + 1
      float acc[2][4] = {};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const FragA fa = rm_a(prod == 0 ? Ah : Bt, mt, kk, lane);
        FragB f0, f1;
        rm_b2(prod == 0 ? S0 : Xb, 2 * nq, kk, lane, f0, f1);
        {
          const FragB fb2[2] = {f0, f1};
          mma3n<2>(acc, fa, fb2);
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (prod == 0) {  // M_ak V: V is B[k = u][n = i] = V[u][i]
          const FragA fa = rm_a(Mak, mt, kk, lane);
          FragB f0, f1;
          rm_bt2(Vm, 2 * nq, kk, lane, f0, f1, !kVExact);
          if (kVExact) {
            mma2b(acc[0], fa, f0);
            mma2b(acc[1], fa, f1);
          } else {
            {
              const FragB fb2[2] = {f0, f1};
              mma3n<2>(acc, fa, fb2);
            }
          }
        } else {  // M_rb^T DY
          const FragA fa = rm_at(Mrb, mt, kk, lane);
          FragB f0, f1;
          rm_bt2(DY, 2 * nq, kk, lane, f0, f1);
          {
            const FragB fb2[2] = {f0, f1};
            mma3n<2>(acc, fa, fb2);
          }
        }
      }
      rm_store_acc(prod == 0 ? U : W, mt, 2 * nq, lane, acc[0]);
      rm_store_acc(prod == 0 ? U : W, mt, 2 * nq + 1, lane, acc[1]);
    }
  }
  __syncthreads();
  if constexpr (!FM) {
    for (int e = tid; e < 32 * 16; e += kNT) {  // T (rows t, columns u), zero above the diagonal
      const int t = e >> 4, u = 2 * (e & 15);
      rm_store(Tm, t, u, u <= t ? TI[t * SM + u] : 0.f, u + 1 <= t ? TI[t * SM + u + 1] : 0.f);
    }
    __syncthreads();
  }

  // ---- P5: SA = T U, DSA = T^T W (rows t, columns i; K = 32); 16 jobs (product, m-tile, 4 n-tiles)
  {  // warp w: SA and DSA at the same tile (m-tile, 2 n-tiles)
    const int mt = (warp >> 2) & 1, nq = warp & 3;
    float acc[2][2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const bool on0 = !(mt == 0 && kk == 1), on1 = !(mt == 1 && kk == 0);  // T lower, T^T upper
      FragB fb0[2], fb1[2];
      rm_bt2(U, 2 * nq, kk, lane, fb0[0], fb0[1]);
      rm_bt2(W, 2 * nq, kk, lane, fb1[0], fb1[1]);
      const FragA fa0 = rm_a(Tm, mt, kk, lane), fa1 = rm_at(Tm, mt, kk, lane);
      if (on0 && on1)
        mma3n_two<2>(acc[0], fa0, fb0, acc[1], fa1, fb1);
      else if (on0)
        mma3n<2>(acc[0], fa0, fb0);
      else
        mma3n<2>(acc[1], fa1, fb1);
    }
    rm_store_acc(SA, mt, 2 * nq, lane, acc[0][0]);
    rm_store_acc(SA, mt, 2 * nq + 1, lane, acc[0][1]);
    rm_store_acc(DSA, mt, 2 * nq, lane, acc[1][0]);
    rm_store_acc(DSA, mt, 2 * nq + 1, lane, acc[1][1]);
  }
  __syncthreads();

  // ---- P6: L1 = tril(DY V^T), L2 = tril(DY SA^T), L3 = tril(DSA V^T, -1), L4 = tril(DSA SA^T, -1) (over U, W)
  {  // warp w: (L1, L3) or (L2, L4) at the same tile, sharing V or SA
    const int prodA = warp >> 2, mt = (warp >> 1) & 1, np = warp & 1;  // prodB = prodA + 2
    const bool exactB = kVExact && prodA == 0;
    float acc[2][2][4] = {};
    if (!(mt == 0 && np == 1)) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const FragA fa0 = rm_a(DY, mt, kk, lane), fa1 = rm_a(DSA, mt, kk, lane);
        FragB fb[2];
        rm_b2(prodA ? SA : Vm, 2 * np, kk, lane, fb[0], fb[1], !exactB);
        if (exactB)
          mma2b_two<2>(acc[0], fa0, acc[1], fa1, fb);
        else
          mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
      }
    }
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      const int prod = prodA + 2 * jb;
      const bool strict = prod >= 2;
      const RM& Lx = prod == 0 ? L1 : (prod == 1 ? L2 : (prod == 2 ? L3 : L4));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nj = 2 * np + h;
        float c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = mt * 16 + g + ((e >> 1) << 3), s2 = nj * 8 + 2 * q + (e & 1);
          c[e] = (strict ? s2 < t : s2 <= t) ? acc[jb][h][e] : 0.f;
        }
        rm_store_acc(Lx, mt, nj, lane, c);
      }
    }
  }
  __syncthreads();

  // ---- P7: DR, DA, DK, DB (rows t, columns j) at (m-tile, 4 n-tiles), in pairs that share their right
  // operands -- warps 0-3: DR and DA (S0, then [K~; B~]), warps 4-7: DK and DB (Xb, then [A^; R^]) -- each a
  // K = 64 product plus the masked products, the two accumulator sets pass-major; then DV (rows t, columns
  // i) at (m-tile, 2 n-tiles), one per warp, so that every warp forms the same number of products.  Each
  // gradient (dr, da, dk, db: the products scaled by Gamma, Gamma_-, 1 / Gamma) is written as soon as
  // formed, so that the stores drain during the warp's later products.  The dw terms r o dr, a o da, k o dk,
  // b o db are the unscaled products times R^, A^, K~, B~ (the same scalings), formed here and kept in
  // registers.
  static_assert(kNW == 8, "P7 job split assumes 8 warps");
  float res[2][4][4];  // the pair's products 2 pg and 2 pg + 1 (0 dr, 1 da, 2 dk, 3 db)
  const int pg = warp >> 2;
  {
    const int mt = (warp >> 1) & 1, nh = warp & 1;  // n-tiles 4nh .. 4nh + 3
#pragma unroll
    for (int rep = 0; rep < 2; ++rep)
#pragma unroll
      for (int x = 0; x < 4; ++x) res[rep][x][0] = res[rep][x][1] = res[rep][x][2] = res[rep][x][3] = 0.f;
    const RM& B1 = pg == 0 ? S0 : Xb;
    const RM& A0 = pg == 0 ? DY : Vm;   // DR: DY S0, DK: V Xb
    const RM& A1 = pg == 0 ? DSA : SA;  // DA: DSA S0, DB: SA Xb
    const bool exact0 = kVExact && pg == 1;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      FragB fb[4];
      rm_bt2(B1, 4 * nh, kk, lane, fb[0], fb[1]);
      rm_bt2(B1, 4 * nh + 2, kk, lane, fb[2], fb[3]);
      const FragA fa1 = rm_a(A1, mt, kk, lane);
      if (exact0) {
        const FragA fa0 = rm_a_hi(A0, mt, kk, lane);
        mma2n<4>(res[0], fa0, fb);
        mma3n<4>(res[1], fa1, fb);
      } else {
        const FragA fa0 = rm_a(A0, mt, kk, lane);
        mma3n_two<4>(res[0], fa0, fb, res[1], fa1, fb);
      }
    }
    // masked part: K = 64 over (block, s); DR: [L1 | L2] [K~; B~], DA: [L3 | L4] [K~; B~],
    // DK: [L3^T | L1^T] [A^; R^], DB: [L4^T | L2^T] [A^; R^]
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const int blk = kq >> 1, kk = kq & 1;
      if (pg == 0 ? (mt == 0 && kk == 1) : (mt == 1 && kk == 0)) continue;  // zero tiles
      const RM& BB = pg == 0 ? (blk ? Bt : Kt) : (blk ? Rh : Ah);
      FragB fb[4];
      rm_bt2(BB, 4 * nh, kk, lane, fb[0], fb[1]);
      rm_bt2(BB, 4 * nh + 2, kk, lane, fb[2], fb[3]);
      FragA fa0, fa1;
      if (pg == 0) {
        fa0 = rm_a(blk ? L2 : L1, mt, kk, lane);
        fa1 = rm_a(blk ? L4 : L3, mt, kk, lane);
      } else {
        fa0 = rm_at(blk ? L1 : L3, mt, kk, lane);
        fa1 = rm_at(blk ? L2 : L4, mt, kk, lane);
      }
      mma3n_two<4>(res[0], fa0, fb, res[1], fa1, fb);
    }
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int prod = 2 * pg + rep;
      float* outp = prod == 0 ? dr : (prod == 1 ? da : (prod == 2 ? dk : db));
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int j = (4 * nh + x) * 8 + 2 * q;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int t = mt * 16 + g + 8 * hr;
          float2 sc = make_float2(1.f, 1.f);
          if (prod == 0) {
            sc = *reinterpret_cast<const float2*>(G + t * LY::kGL + j);
          } else if (prod == 1) {
            if (t > 0) sc = *reinterpret_cast<const float2*>(G + (t - 1) * LY::kGL + j);
          } else {
            const float2 gt = *reinterpret_cast<const float2*>(G + t * LY::kGL + j);
            sc = make_float2(__fdividef(1.f, gt.x), __fdividef(1.f, gt.y));
          }
          const float2 sop = rm_get2(prod == 0 ? Rh : (prod == 1 ? Ah : (prod == 2 ? Kt : Bt)), t, j);
          const float u0 = res[rep][x][2 * hr], u1 = res[rep][x][2 * hr + 1];
          res[rep][x][2 * hr] = u0 * sop.x;  // the dw term (zero past the chunk: the operand rows are)
          res[rep][x][2 * hr + 1] = u1 * sop.y;
          if (t < n && WKV7_IN(t0 + t, T, dbg::kColmat) && WKV7_IN(j + 1, kD, dbg::kColmat))
            *reinterpret_cast<float2*>(outp + base + (size_t)(t0 + t) * tstride + j) = make_float2(u0 * sc.x, u1 * sc.y);
        }
      }
    }
  }
  {  // DV = K~ Xb^T + M_ak^T DSA + M_rk^T DY (rows t, columns i): m-tile w >> 2, n-tiles 2 (w & 3) + 0, 1
    const int mt = warp >> 2, nq = warp & 3;
    float acc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const FragA fa = rm_a(Kt, mt, kk, lane);
      FragB fb[2];
      rm_b2(Xb, 2 * nq, kk, lane, fb[0], fb[1]);
      mma3n<2>(acc, fa, fb);
    }
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const int blk = kq >> 1, kk = kq & 1;
      if (mt == 1 && kk == 0) continue;  // M_ak^T, M_rk^T upper triangular
      const FragA fa = rm_at(blk ? Mrk : Mak, mt, kk, lane);
      FragB fb[2];
      rm_bt2(blk ? DY : DSA, 2 * nq, kk, lane, fb[0], fb[1]);
      mma3n<2>(acc, fa, fb);
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int i = (2 * nq + x) * 8 + 2 * q;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int t = mt * 16 + g + 8 * hr;
        if (t < n && WKV7_IN(t0 + t, T, dbg::kColmat) && WKV7_IN(i + 1, kD, dbg::kColmat))
          *reinterpret_cast<float2*>(dv + base + (size_t)(t0 + t) * tstride + i) =
              make_float2(acc[x][2 * hr], acc[x][2 * hr + 1]);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // every operand has been read: stage over A^ .. Xb
  // ---- r o dr, a o da, k o dk, b o db into shared memory (over A^ ..) for dw
  float* terms = reinterpret_cast<float*>(sm + LY::oStage);
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int prod = 2 * pg + rep, mt = (warp >> 1) & 1, nh = warp & 1;
    float* sp = terms + prod * kL * LY::kTL;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int j = (4 * nh + x) * 8 + 2 * q;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int t = mt * 16 + g + 8 * hr;
        *reinterpret_cast<float2*>(sp + t * LY::kTL + j) = make_float2(res[rep][x][2 * hr], res[rep][x][2 * hr + 1]);
      }
    }
  }
  __syncthreads();

  if (next < total) issue(next);  // raw, staging and SA / DSA regions are dead from here on

  // ---- P8: dw per column from Z_t = colsum(X_t o S_t) (X_t: the gradient w.r.t. the state after token t):
  //   Z_{n-1} = colsum(G o S_e) + r_{n-1} o dr_{n-1},   w_t o dw_t = Z_t - k_t o dk_t - b_t o db_t,
  //   Z_{t-1} = w_t o dw_t + a_t o da_t + r_{t-1} o dr_{t-1} = Z_t + D_t,
  // so Z_t = Z_{n-1} + sum_{s = t+1}^{n-1} D_s, a suffix sum: 4 blocks of 8 tokens per column.
  {
    constexpr int TL = LY::kTL;
    const float* sRDR = terms;
    const float* sADA = terms + kL * TL;
    const float* sKDK = terms + 2 * kL * TL;
    const float* sBDB = terms + 3 * kL * TL;
    const int j = tid & 63, blk = tid >> 6;  // threads 0-255
    const bool act = tid < 256;
    float dsum[8];  // sum of D_s over this block's tokens s > t
    float tot = 0.f;
    if (act) {
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        const int t = 8 * blk + u;
        dsum[u] = tot;
        if (t >= 1 && t < n) tot += sADA[t * TL + j] + sRDR[(t - 1) * TL + j] - sKDK[t * TL + j] - sBDB[t * TL + j];
      }
      if (WKV7_IN(blk, 4, dbg::kColmat)) BT[blk * 64 + j] = tot;
    }
    __syncthreads();
    if (act) {
    float later = 0.f;
    for (int q2 = blk + 1; q2 < 4; ++q2) later += BT[q2 * 64 + j];
    const float zn = ZP[j] + sRDR[(n - 1) * TL + j];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = 8 * blk + u;
      if (t < n && WKV7_IN(t0 + t, T, dbg::kColmat)) {
        const float wdw = zn + later + dsum[u] - sKDK[t * TL + j] - sBDB[t * TL + j];
        dw[base + (size_t)(t0 + t) * tstride + j] = __fdividef(wdw, Wc[t * kD + j]);  // (w >= 1/32 here)
      }
    }
    }
  }
  }  // chunks
}

// The token-by-token column passes for the chunks colmat_kernel flagged (some w_t below 1/32, or gamma_31
// below 1e-20 or not finite): sa and dsa by their per-token recurrences, dv from X, then the exact column
// passes of wkv7_colpass.cuh.  A persistent grid reads every chunk's flag and skips the others.
template <typename Tin>
struct FbLay {
  static constexpr int oRaw = 0;  // w, k, a, b, r, v [32][64] Tin
  static constexpr int kRawIn = 6 * kL * kD * (int)sizeof(Tin);
  static constexpr int oDyRaw = oRaw + kRawIn;  // dy fp32 [32][64]
  static constexpr int oFSa = oDyRaw + kL * kD * 4;
  static constexpr int oFDsa = oFSa + kL * kD * 4;
  static constexpr int oFV = oFDsa + kL * kD * 4;
  static constexpr int oFXe = oFV + kL * kD * 4;  // X_e fp32 [64][64]
  static constexpr int kBytes = oFXe + kD * kD * 4;
};
constexpr int kNTF = 128;

template <typename Tin>
__global__ void __launch_bounds__(kNTF)
colfb_kernel(int T, int H, int nchunks, int total, const Tin* __restrict__ r, const Tin* __restrict__ w,
             const Tin* __restrict__ k, const Tin* __restrict__ v, const Tin* __restrict__ a,
             const Tin* __restrict__ b, const float* __restrict__ h0, const float* __restrict__ h_ckpt,
             const float* __restrict__ dy, const float* __restrict__ xck, const int* __restrict__ flags,
             size_t xck_stride, float* __restrict__ dr, float* __restrict__ dw, float* __restrict__ dk,
             float* __restrict__ dv, float* __restrict__ da, float* __restrict__ db) {
  using LY = FbLay<Tin>;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  const int tid = threadIdx.x;
  Tin* raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  const Tin* rw = raw;
  const Tin* rk = raw + kL * kD;
  const Tin* ra = raw + 2 * kL * kD;
  const Tin* rbv = raw + 3 * kL * kD;
  const Tin* rr = raw + 4 * kL * kD;
  const Tin* rv = raw + 5 * kL * kD;
  float* dyr = reinterpret_cast<float*>(sm + LY::oDyRaw);
  const size_t tstride = (size_t)H * kD;
  __shared__ int fl[kNTF];
  // this CTA's chunks are blockIdx.x + gridDim.x * m; their flags are read kNTF at a time, in parallel
  for (int m0 = 0; blockIdx.x + (size_t)gridDim.x * m0 < (size_t)total; m0 += kNTF) {
    {
      const size_t jt = blockIdx.x + (size_t)gridDim.x * (m0 + tid);
      fl[tid] = (jt < (size_t)total && flags[jt * xck_stride] != 0) ? 1 : 0;
    }
    if (__syncthreads_or(fl[tid]) == 0) continue;
    for (int m = 0; m < kNTF; ++m) {
      if (fl[m] == 0) continue;
      const int job = blockIdx.x + gridDim.x * (m0 + m);
      if (!WKV7_IN(job, total, dbg::kColfb)) continue;
      const int ci = job % nchunks;
      const int bh = job / nchunks;
      const int bi = bh / H;
      const int hi = bh - bi * H;
      const int t0 = ci * kL;
      const int n = min(kL, T - t0);
      const size_t base = ((size_t)bi * T * H + hi) * kD;
      const float* gend = xck + (size_t)job * xck_stride;
      const float* s0 = ci > 0 ? h_ckpt + ((size_t)bh * nchunks + ci - 1) * kD * kD
                               : (h0 != nullptr ? h0 + (size_t)bh * kD * kD : nullptr);
      {
        constexpr int CPR = kD * (int)sizeof(Tin) / 16;
        constexpr int EPC = 16 / (int)sizeof(Tin);
        const Tin* srcs[6] = {w, k, a, b, r, v};
  #pragma unroll
        for (int s6 = 0; s6 < 6; ++s6)
          for (int e = tid; e < n * CPR; e += kNTF) {
            const int tt = e / CPR, pc = e % CPR;
            cp_async16(raw + (s6 * kL + tt) * kD + pc * EPC, srcs[s6] + base + (size_t)(t0 + tt) * tstride + pc * EPC);
          }
        for (int e = tid; e < n * (kD / 4); e += kNTF) {
          const int tt = e / (kD / 4), pc = e % (kD / 4);
          cp_async16(dyr + tt * kD + pc * 4, dy + base + (size_t)(t0 + tt) * tstride + pc * 4);
        }
        cp_async_commit();
        cp_async_wait<0>();
      }
      __syncthreads();
      float* fsa = reinterpret_cast<float*>(sm + LY::oFSa);
      float* fdsa = reinterpret_cast<float*>(sm + LY::oFDsa);
      float* fv = reinterpret_cast<float*>(sm + LY::oFV);
      for (int e = tid; e < n * kD; e += kNTF) fv[e] = to_f32(rv[e]);
      if (tid < 64) {  // sa_t = S_{t-1} a_t, row tid, the state run up from S0
        const int i = tid;
        float Sr[64];
  #pragma unroll
        for (int j = 0; j < 64; ++j) Sr[j] = s0 != nullptr ? __ldg(s0 + i * kD + j) : 0.f;
        for (int t = 0; t < n; ++t) {
          float s = 0.f;
  #pragma unroll
          for (int j = 0; j < 64; ++j) s = fmaf(Sr[j], to_f32(ra[t * kD + j]), s);
          fsa[t * kD + i] = s;
          const float vi = to_f32(rv[t * kD + i]);
  #pragma unroll
          for (int j = 0; j < 64; ++j)
            Sr[j] = fmaf(Sr[j], to_f32(rw[t * kD + j]), fmaf(vi, to_f32(rk[t * kD + j]), s * to_f32(rbv[t * kD + j])));
        }
      } else if (tid < 128) {  // dsa_t = X_t b_t and dv_t = X_t k_t, row tid - 64, X walked down from X_e
        const int i = tid - 64;
        float* fxe = reinterpret_cast<float*>(sm + LY::oFXe);
        float Xr[64];
        const float dl = dyr[(n - 1) * kD + i];
  #pragma unroll
        for (int j = 0; j < 64; ++j) {
          Xr[j] = fmaf(dl, to_f32(rr[(n - 1) * kD + j]), __ldg(gend + acc_order(i, j)));
          fxe[i * kD + j] = Xr[j];
        }
        for (int t = n - 1; t >= 0; --t) {
          float s = 0.f, sv = 0.f;
  #pragma unroll
          for (int j = 0; j < 64; ++j) {
            s = fmaf(Xr[j], to_f32(rbv[t * kD + j]), s);
            sv = fmaf(Xr[j], to_f32(rk[t * kD + j]), sv);
          }
          fdsa[t * kD + i] = s;
          dv[base + (size_t)(t0 + t) * tstride + i] = sv;
          const float e = t > 0 ? dyr[(t - 1) * kD + i] : 0.f;
  #pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float rp = t > 0 ? to_f32(rr[(t - 1) * kD + j]) : 0.f;
            Xr[j] = fmaf(Xr[j], to_f32(rw[t * kD + j]), fmaf(s, to_f32(ra[t * kD + j]), e * rp));
          }
        }
      }
      __syncthreads();
      if (tid < 64)
        colpass::passes<Tin>(tid, n, t0, base, tstride, raw, fsa, fdsa, dyr, fv,
                             reinterpret_cast<const float*>(sm + LY::oFXe), s0, dr, dw, dk, da, db);
      __syncthreads();  // the next flagged chunk reuses the buffers
    }
    __syncthreads();  // fl is rewritten for the next kNTF chunks
  }
}

template <typename Tin>
cudaError_t launch_colmat_t(const BwdArgs& p, const ChunkEnds& ends, cudaStream_t stream) {
  using LY = Lay<Tin>;
  using FL = FbLay<Tin>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  // the forward's matrices are taken where their region fits beside the rest (bf16 inputs); fp32 inputs
  // (twice the raw staging) form them here
  constexpr bool kFits = LY::kBytesM <= 232448;
  const bool fm = kFits && ends.mats != nullptr;
  auto kern = colmat_kernel<Tin, false>;
  if constexpr (kFits)
    if (fm) kern = colmat_kernel<Tin, true>;
  const int smem = fm ? LY::kBytesM : LY::kBytes;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  const int total = p.B * p.H * p.nchunks;
  const int grid = min(total, num_sms());  // one CTA per SM (shared memory), each looping over its chunks
  kern<<<(unsigned)grid, kNT, smem, stream>>>(
      p.T, p.H, p.nchunks, total, (const Tin*)p.in.r, (const Tin*)p.in.w, (const Tin*)p.in.k, (const Tin*)p.in.v,
      (const Tin*)p.in.a, (const Tin*)p.in.b, p.h0, p.h_ckpt, p.dy, ends.g, ends.flags, ends.stride, ends.mats, p.dr,
      p.dw, p.dk, p.dv, p.da, p.db);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  auto fkern = colfb_kernel<Tin>;
  err = cudaFuncSetAttribute(fkern, cudaFuncAttributeMaxDynamicSharedMemorySize, FL::kBytes);
  if (err != cudaSuccess) return err;
  const int fgrid = min(total, 2 * num_sms());
  fkern<<<(unsigned)fgrid, kNTF, FL::kBytes, stream>>>(
      p.T, p.H, p.nchunks, total, (const Tin*)p.in.r, (const Tin*)p.in.w, (const Tin*)p.in.k, (const Tin*)p.in.v,
      (const Tin*)p.in.a, (const Tin*)p.in.b, p.h0, p.h_ckpt, p.dy, ends.g, ends.flags, ends.stride, p.dr, p.dw, p.dk,
      p.dv, p.da, p.db);
  return cudaGetLastError();
}

}  // namespace

WKV7_DEBUG_READER(debug_word_colmat)

cudaError_t launch_colgrad_matrix(const BwdArgs& p, const ChunkEnds& ends, cudaStream_t stream) {
  if (p.nchunks == 0) return cudaSuccess;
  return p.bf16 ? launch_colmat_t<__nv_bfloat16>(p, ends, stream) : launch_colmat_t<float>(p, ends, stream);
}

}  // namespace wkv7
