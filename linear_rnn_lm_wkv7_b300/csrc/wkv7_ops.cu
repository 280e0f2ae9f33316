// WKV7 on sm_103a in two steps per direction: the transition operands of every 32-token chunk at
// once, then the serial chain over the chunks reading them.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel architecture",
// Forward and Backward listings), per head, state S (rows i = value, columns j = key):
//     sa_t = S_{t-1} a_t;   S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T;   y_t = S_t r_t.
// Over a chunk of 32 tokens from state S0, with gamma_t = w_0 o .. o w_t per column and
//     A^_t = a_t o gamma_{t-1},  R^_t = r_t o gamma_t,  K~_t = k_t / gamma_t,  B~_t = b_t / gamma_t,
//     M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T),
//     T = (I - M_ab)^-1,  B' = (T^T B~) diag(gamma_31),  C = M_rb T,
//     K' = K~ diag(gamma_31) + M_ak^T B',  P = M_rk + C M_ak,
// (unrolled over the chunk, sa is coupled through the unit lower-triangular system I - M_ab;
// eliminating it gives one transition per chunk):
//   forward:  P1 = S0 A^^T;  S' = S0 diag(gamma_31) + P1 B' + V^T K';  Y^T = S0 R^^T + P1 C^T + V^T P^T
//   backward: with G the gradient w.r.t. the state after the chunk (from every later token),
//             G_prev = G diag(gamma_31) + (G B'^T + DY^T C) A^ + DY^T R^     (the transposed transition)
//
// ops_prep_kernel: one CTA per (head, chunk), all chunks at once; writes gamma_31, a flag, and B', K',
// C, P (bf16 hi and lo, row-major) per chunk.  A^ and R^ are rebuilt by the chains from the inputs.
// ops_chain_kernel: the forward chain, one CTA per (head, 32-row block): 2 chain warps (S as mma
// accumulators, P1, S', y), 2 v warps (V as an operand, N = V^T K'), 4 load warps (the next chunks'
// operands by cp.async, decays, A^ and R^).
// ops_walk_kernel: the backward's state-gradient walk over the same chunks, last to first, writing G
// at every chunk end (for the column gradients) and dh0.
// A chunk whose gamma_31 falls below 1e-20 (or is not finite) is taken token by token (exact fp32).
// Precision: three bf16 products per fp32 product (wkv7_mma.cuh), fp32 accumulation.
#include <type_traits>

#include "wkv7_device.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace {

using namespace mma;

constexpr int kL = 32;
constexpr int kR = 32;
constexpr int kLD64 = 72;
constexpr int kLD32 = 40;
constexpr float kMinGamma = 1e-20f;

template <int ID, int N>
__device__ __forceinline__ void bsync() { asm volatile("bar.sync %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }
template <int ID, int N>
__device__ __forceinline__ void barrive() { asm volatile("bar.arrive %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }

__host__ __device__ constexpr int rmb(int rows, int ld) { return 2 * rows * ld * 2; }

// ---- per-chunk operand block in global memory (bytes): gamma_31 fp32 [64], flag, then B', K'
// (32 x 64) and C, P (32 x 32) as bf16 hi then lo, rows unpadded
constexpr int kOpGL = 0;
constexpr int kOpMeta = 256;
constexpr int kOpBp = 512;
constexpr int kOpKp = kOpBp + 2 * 32 * 64 * 2;
constexpr int kOpC = kOpKp + 2 * 32 * 64 * 2;
constexpr int kOpP = kOpC + 2 * 32 * 32 * 2;
constexpr int kOpBytes = kOpP + 2 * 32 * 32 * 2;  // 25088

// copy an RM array (rows x cols bf16, hi and lo) between padded shared (ld) and unpadded global, by
// 16-byte pieces; `to_global` picks the direction; threads tid .. step
template <bool TO_GLOBAL>
__device__ __forceinline__ void copy_rm(const RM& x, int rows, int cols, unsigned char* g, int tid, int step) {
  const int ppr = cols / 8;  // 16-byte pieces per row
  for (int e = tid; e < 2 * rows * ppr; e += step) {
    const int half = e / (rows * ppr), rem = e - half * rows * ppr;
    const int rr = rem / ppr, pc = rem - rr * ppr;
    __nv_bfloat16* s = x.p + half * x.lo + rr * x.ld + pc * 8;
    unsigned char* gp = g + ((size_t)(half * rows + rr) * cols + pc * 8) * 2;
    if (TO_GLOBAL)
      *reinterpret_cast<uint4*>(gp) = *reinterpret_cast<const uint4*>(s);
    else
      cp_async16(s, gp);
  }
}

// ======================================================================================= prep

constexpr int kNTP = 256;

template <typename Tin>
struct PrepLay {
  static constexpr int oG = 0;                          // float [32][64]
  static constexpr int oAh = oG + 32 * 64 * 4;          // RM 32x64 A^ (then B')
  static constexpr int oRh = oAh + rmb(32, kLD64);      // R^ (then K')
  static constexpr int oKt = oRh + rmb(32, kLD64);
  static constexpr int oBt = oKt + rmb(32, kLD64);
  static constexpr int oMak = oBt + rmb(32, kLD64);     // RM 32x32
  static constexpr int oMrb = oMak + rmb(32, kLD32);
  static constexpr int oMrk = oMrb + rmb(32, kLD32);
  static constexpr int oT = oMrk + rmb(32, kLD32);
  static constexpr int oC = oT + rmb(32, kLD32);
  static constexpr int oP = oC + rmb(32, kLD32);
  static constexpr int oGL = oP + rmb(32, kLD32);       // float [64], then int [4]
  static constexpr int oRaw = oGL + 64 * 4 + 16 + 240;  // w, k, a, b, r [32][64]; then M_ab, T fp32, E
  static constexpr int kSM = 36;
  static constexpr int oMab = oRaw;
  static constexpr int oTI = oMab + 32 * kSM * 4;
  static constexpr int oE = oTI + 32 * kSM * 4;
  static constexpr int kRaw = 5 * kL * kD * (int)sizeof(Tin);
  static_assert(oE + 16 * 16 * 4 <= oRaw + kRaw, "M_ab, T and E fit over the raw inputs");
  static constexpr int kBytes = oRaw + kRaw;
};

template <typename Tin>
__global__ void __launch_bounds__(kNTP)
ops_prep_kernel(int T, int H, int nchunks, const Tin* __restrict__ r, const Tin* __restrict__ w,
                const Tin* __restrict__ k, const Tin* __restrict__ a, const Tin* __restrict__ b,
                unsigned char* __restrict__ ops) {
  using LY = PrepLay<Tin>;
  constexpr int SM = LY::kSM;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  const int ci = blockIdx.x % nchunks;
  const int bh = blockIdx.x / nchunks;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int pt = threadIdx.x;
  const int pw = pt >> 5;
  const int lane = pt & 31;
  const int g = lane >> 2, q = lane & 3;
  const int t0 = ci * kL;
  const int nm = min(kL, T - t0);
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  unsigned char* out = ops + ((size_t)bh * nchunks + ci) * kOpBytes;

  auto bfp = [&](int off) { return reinterpret_cast<__nv_bfloat16*>(sm + off); };
  const RM Ah{bfp(LY::oAh), 32 * kLD64, kLD64}, Rh{bfp(LY::oRh), 32 * kLD64, kLD64};
  const RM Kt{bfp(LY::oKt), 32 * kLD64, kLD64}, Bt{bfp(LY::oBt), 32 * kLD64, kLD64};
  const RM Bp = Ah, Kp = Rh;  // B' and K' over A^ and R^ (read for the last time by the coupling products)
  const RM Mak{bfp(LY::oMak), 32 * kLD32, kLD32}, Mrb{bfp(LY::oMrb), 32 * kLD32, kLD32};
  const RM Mrk{bfp(LY::oMrk), 32 * kLD32, kLD32}, Tm{bfp(LY::oT), 32 * kLD32, kLD32};
  const RM Cm{bfp(LY::oC), 32 * kLD32, kLD32}, Pm{bfp(LY::oP), 32 * kLD32, kLD32};
  float* G = reinterpret_cast<float*>(sm + LY::oG);
  float* GL = reinterpret_cast<float*>(sm + LY::oGL);
  int* meta = reinterpret_cast<int*>(sm + LY::oGL + 256);
  Tin* raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  float* Mab = reinterpret_cast<float*>(sm + LY::oMab);
  float* TI = reinterpret_cast<float*>(sm + LY::oTI);
  float* E = reinterpret_cast<float*>(sm + LY::oE);

  {  // the chunk's w, k, a, b, r (rows past the chunk are not copied)
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    const Tin* srcs[5] = {w, k, a, b, r};
#pragma unroll
    for (int s5 = 0; s5 < 5; ++s5)
      for (int e = pt; e < nm * CPR; e += kNTP) {
        const int t = e / CPR, pc = e % CPR;
        cp_async16(raw + (s5 * kL + t) * kD + pc * EPC, srcs[s5] + base + (size_t)(t0 + t) * tstride + pc * EPC);
      }
    cp_async_commit();
    cp_async_wait<0>();
  }
  __syncthreads();
  const Tin* rw = raw;
  const Tin* rk = raw + kL * kD;
  const Tin* ra = raw + 2 * kL * kD;
  const Tin* rbv = raw + 3 * kL * kD;
  const Tin* rr = raw + 4 * kL * kD;

  if (pt < kD) {  // gamma_t down each column; the token-by-token flag
    const int j = pt;
    float gm = 1.f;
#pragma unroll 8
    for (int t = 0; t < kL; ++t) {
      const float wt = t < nm ? to_f32(rw[t * kD + j]) : 1.f;
      gm *= wt;
      G[t * kD + j] = gm;
    }
    GL[j] = gm;
    const bool bad = !(gm >= kMinGamma) || !(gm <= 3.0e38f);
    const unsigned any = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) meta[pw] = any != 0u;
  }
  __syncthreads();
  const bool slow = (meta[0] | meta[1]) != 0;
  if (pt < 16) reinterpret_cast<float4*>(out + kOpGL)[pt] = reinterpret_cast<const float4*>(GL)[pt];
  if (pt == 0) *reinterpret_cast<int4*>(out + kOpMeta) = make_int4(slow ? 1 : 0, 0, 0, 0);
  if (slow) return;

  {  // one (token, 8 columns) block per thread: A^, R^, K~, B~
    const int t = pt >> 3, c0 = (pt & 7) * 8;
    const bool ok = t < nm;
    float gt[8], gp[8], av[8], rv[8], kv[8], bv[8];
    raw8(G + t * kD + c0, gt);
    if (t > 0) {
      raw8(G + (t - 1) * kD + c0, gp);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) gp[u] = 1.f;
    }
    raw8(ra + t * kD + c0, av);
    raw8(rr + t * kD + c0, rv);
    raw8(rk + t * kD + c0, kv);
    raw8(rbv + t * kD + c0, bv);
    float oa[8], orr[8], ok8[8], ob[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float ig = __fdividef(1.f, gt[u]);
      oa[u] = ok ? av[u] * gp[u] : 0.f;
      orr[u] = ok ? rv[u] * gt[u] : 0.f;
      ok8[u] = ok ? kv[u] * ig : 0.f;
      ob[u] = ok ? bv[u] * ig : 0.f;
    }
    rm_store8(Ah, t, c0, oa);
    rm_store8(Rh, t, c0, orr);
    rm_store8(Kt, t, c0, ok8);
    rm_store8(Bt, t, c0, ob);
  }
  __syncthreads();  // the raw inputs are consumed: M_ab, T and E reuse their space

  // M_ab = tril(A^ B~^T, -1) (fp32), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T)
  for (int job = pw; job < 16; job += 8) {
    const int prod = job >> 2, mt = (job >> 1) & 1, np = job & 1;
    const bool strict = prod < 2;
    float acc[2][4] = {};
    if (!(mt == 0 && np == 1)) {
      const RM& X = prod < 2 ? Ah : Rh;
      const RM& Y = (prod & 1) ? Kt : Bt;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const FragA fa = rm_a(X, mt, kk, lane);
        FragB f0, f1;
        rm_b2(Y, 2 * np, kk, lane, f0, f1);
        mma3(acc[0], fa, f0);
        mma3(acc[1], fa, f1);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int nj = 2 * np + h;
      const int tr = mt * 16 + g, sc = nj * 8 + 2 * q;
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tt = tr + ((e >> 1) << 3), s = sc + (e & 1);
        c[e] = (strict ? s < tt : s <= tt) ? acc[h][e] : 0.f;
      }
      if (prod == 0) {
        *reinterpret_cast<float2*>(Mab + tr * SM + sc) = make_float2(c[0], c[1]);
        *reinterpret_cast<float2*>(Mab + (tr + 8) * SM + sc) = make_float2(c[2], c[3]);
      } else {
        rm_store_acc(prod == 1 ? Mak : (prod == 2 ? Mrb : Mrk), mt, nj, lane, c);
      }
    }
  }
  __syncthreads();

  // T = (I - M_ab)^-1 by blocks of 16: diagonal blocks by forward substitution (one column per lane),
  // then T21 = T22 A21 T11
  if (pw == 0) {
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
  }
  __syncthreads();
  {
    const int t = pt >> 4, s = pt & 15;
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) acc = fmaf(Mab[(16 + t) * SM + u], TI[u * SM + s], acc);
    E[t * 16 + s] = acc;
  }
  __syncthreads();
  {
    const int t = pt >> 4, s = pt & 15;
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) acc = fmaf(TI[(16 + t) * SM + 16 + u], E[u * 16 + s], acc);
    TI[(16 + t) * SM + s] = acc;
  }
  __syncthreads();
  if (pt < 128) {
    const int t = pt >> 2, u0 = (pt & 3) * 8;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = u0 + e <= t ? TI[t * SM + u0 + e] : 0.f;
    rm_store8(Tm, t, u0, x);
  }
  __syncthreads();

  // B' = (T^T B~) diag(gamma_31) (over A^) and C = M_rb T
  for (int job = pw; job < 12; job += 8) {
    float acc[2][4] = {};
    if (job < 8) {
      const int mt = job >> 2, nq = job & 3;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (mt == 1 && kk == 0) continue;
        const FragA fa = rm_at(Tm, mt, kk, lane);
        FragB f0, f1;
        rm_bt2(Bt, 2 * nq, kk, lane, f0, f1);
        mma3(acc[0], fa, f0);
        mma3(acc[1], fa, f1);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 gl = *reinterpret_cast<const float2*>(GL + (2 * nq + h) * 8 + 2 * q);
        acc[h][0] *= gl.x; acc[h][1] *= gl.y; acc[h][2] *= gl.x; acc[h][3] *= gl.y;
      }
      rm_store_acc(Bp, mt, 2 * nq, lane, acc[0]);
      rm_store_acc(Bp, mt, 2 * nq + 1, lane, acc[1]);
    } else {
      const int mt = (job - 8) >> 1, np = (job - 8) & 1;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (mt == 0 && kk == 1) continue;
        const FragA fa = rm_a(Mrb, mt, kk, lane);
        FragB f0, f1;
        rm_bt2(Tm, 2 * np, kk, lane, f0, f1);
        mma3(acc[0], fa, f0);
        mma3(acc[1], fa, f1);
      }
      rm_store_acc(Cm, mt, 2 * np, lane, acc[0]);
      rm_store_acc(Cm, mt, 2 * np + 1, lane, acc[1]);
    }
  }
  __syncthreads();

  // K' = K~ diag(gamma_31) + M_ak^T B' (over R^) and P = M_rk + C M_ak
  for (int job = pw; job < 12; job += 8) {
    float acc[2][4] = {};
    if (job < 8) {
      const int mt = job >> 2, nq = job & 3;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (mt == 1 && kk == 0) continue;
        const FragA fa = rm_at(Mak, mt, kk, lane);
        FragB f0, f1;
        rm_bt2(Bp, 2 * nq, kk, lane, f0, f1);
        mma3(acc[0], fa, f0);
        mma3(acc[1], fa, f1);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = (2 * nq + h) * 8 + 2 * q;
        const int tr = mt * 16 + g;
        const float2 gl = *reinterpret_cast<const float2*>(GL + col);
        const float2 k0 = rm_get2(Kt, tr, col), k8 = rm_get2(Kt, tr + 8, col);
        acc[h][0] = fmaf(k0.x, gl.x, acc[h][0]);
        acc[h][1] = fmaf(k0.y, gl.y, acc[h][1]);
        acc[h][2] = fmaf(k8.x, gl.x, acc[h][2]);
        acc[h][3] = fmaf(k8.y, gl.y, acc[h][3]);
        rm_store_acc(Kp, mt, 2 * nq + h, lane, acc[h]);
      }
    } else {
      const int mt = (job - 8) >> 1, np = (job - 8) & 1;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (mt == 0 && kk == 1) continue;
        const FragA fa = rm_a(Cm, mt, kk, lane);
        FragB f0, f1;
        rm_bt2(Mak, 2 * np, kk, lane, f0, f1);
        mma3(acc[0], fa, f0);
        mma3(acc[1], fa, f1);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = (2 * np + h) * 8 + 2 * q;
        const int tr = mt * 16 + g;
        const float2 m0 = rm_get2(Mrk, tr, col), m8 = rm_get2(Mrk, tr + 8, col);
        acc[h][0] += m0.x; acc[h][1] += m0.y; acc[h][2] += m8.x; acc[h][3] += m8.y;
        rm_store_acc(Pm, mt, 2 * np + h, lane, acc[h]);
      }
    }
  }
  __syncthreads();
  copy_rm<true>(Bp, 32, 64, out + kOpBp, pt, kNTP);
  copy_rm<true>(Kp, 32, 64, out + kOpKp, pt, kNTP);
  copy_rm<true>(Cm, 32, 32, out + kOpC, pt, kNTP);
  copy_rm<true>(Pm, 32, 32, out + kOpP, pt, kNTP);
}

// =========================================================================== chains (shared parts)

constexpr int kNTC = 256;  // 8 warps: 2 chain, 2 v / dy, 4 load

// operand buffer of one chunk in shared memory: A^, R^, B', K' (RM 32x64), C, P (RM 32x32), gamma_31, flag
struct Buf {
  static constexpr int cAh = 0;
  static constexpr int cRh = cAh + rmb(32, kLD64);
  static constexpr int cBp = cRh + rmb(32, kLD64);
  static constexpr int cKp = cBp + rmb(32, kLD64);
  static constexpr int cC = cKp + rmb(32, kLD64);
  static constexpr int cP = cC + rmb(32, kLD32);
  static constexpr int cGL = cP + rmb(32, kLD32);
  static constexpr int cMeta = cGL + 64 * 4;
  static constexpr int kBytes = cMeta + 16;
};
constexpr int kNBuf = 3;  // operand buffers in flight: chunk n (chain), n + 1 (rebuilt), n + 2 (copying)

template <typename Tin, typename TV>
struct ChainLay {
  static constexpr int oBuf = 0;
  static constexpr int oRaw = oBuf + kNBuf * Buf::kBytes;     // w, a, r [32][64] of a chunk, x2
  static constexpr int kRaw = 3 * kL * kD * (int)sizeof(Tin);
  static constexpr int oG = oRaw + 2 * kRaw;                   // float [32][64]
  static constexpr int oVraw = oG + 32 * 64 * 4;              // v / dy of this CTA's rows [32 t][32 i], x2
  static constexpr int kVraw = kL * kR * (int)sizeof(TV);
  static constexpr int oVop = oVraw + 2 * kVraw;              // RM 32 t x 32 i
  static constexpr int oN = oVop + rmb(32, kLD32);             // float [2 mt][8 nj][32][4]
  static constexpr int oN2 = oN + 32 * 64 * 4;                 // float [2 mt][4 nj][32][4] (walk: DY^T C)
  static constexpr int kSY = 36;
  static constexpr int oY = oN2 + 32 * 32 * 4;                 // float [32 t][36]
  static constexpr int kSFS = 68;
  static constexpr int oFS = oN;                               // token-by-token path: float [32][68]
  static constexpr int kBytes = oY + kL * kSY * 4;
  static_assert(oFS + 32 * kSFS * 4 <= kBytes, "token-by-token state fits over N and y");
};

// The chunk schedule of the chains: chunk c covers tokens 32c .. min(T, 32c + 32) - 1.
// Forward: chunks 0, 1, ..; walk: C-1, .., 0 (period n works on chunk walk ? C-1-n : n).

// ========================================================================================== chain

template <typename Tin, bool WALK>
__global__ void __launch_bounds__(kNTC, 1)
ops_chain_kernel(int T, int H, int nchunks, const Tin* __restrict__ r, const Tin* __restrict__ w,
                 const Tin* __restrict__ k, const void* __restrict__ vin, const Tin* __restrict__ a,
                 const Tin* __restrict__ b, const unsigned char* __restrict__ ops, const float* __restrict__ s0,
                 float* __restrict__ y, float* __restrict__ ck, float* __restrict__ sT) {
  // forward: vin = v (Tin), s0 = h0, y, ck = h_ckpt, sT = hT.  walk: vin = dy (fp32), s0 = dhT,
  // y unused, ck = G at every chunk end, sT = dh0.
  using TV = typename std::conditional<WALK, float, Tin>::type;
  using LY = ChainLay<Tin, TV>;
  constexpr bool kVExact = sizeof(TV) == 2;
  const TV* __restrict__ v = static_cast<const TV*>(vin);
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);

  const int bh = blockIdx.x >> 1;
  const int rb = blockIdx.x & 1;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;
  const int nsub = nchunks;
  auto chunk_of = [&](int n) { return WALK ? nchunks - 1 - n : n; };
  auto clen = [&](int c) { return min(kL, T - c * kL); };

  auto buf = [&](int n) { return sm + LY::oBuf + (n % kNBuf) * Buf::kBytes; };
  auto bfp = [&](unsigned char* p, int off) { return reinterpret_cast<__nv_bfloat16*>(p + off); };
  auto rm64 = [&](unsigned char* cb, int off) { return RM{bfp(cb, off), 32 * kLD64, kLD64}; };
  auto rm32 = [&](unsigned char* cb, int off) { return RM{bfp(cb, off), 32 * kLD32, kLD32}; };
  auto slow_of = [&](const unsigned char* cb) { return *reinterpret_cast<const int*>(cb + Buf::cMeta) != 0; };
  auto vraw = [&](int n) { return reinterpret_cast<TV*>(sm + LY::oVraw + (n & 1) * LY::kVraw); };
  const RM Vop{bfp(sm, LY::oVop), 32 * kLD32, kLD32};
  float* const nb = reinterpret_cast<float*>(sm + LY::oN);
  float* const nb2 = reinterpret_cast<float*>(sm + LY::oN2);
  float* const ys = reinterpret_cast<float*>(sm + LY::oY);

  if (warp < 2) {
    // =============================================================== chain warps
    const int mt = warp;
    const int row = rb * kR + mt * 16 + g;
    float S[8][4];
#pragma unroll
    for (int nj = 0; nj < 8; ++nj) {
      if (s0 != nullptr) {
        const float2 x0 = __ldg(reinterpret_cast<const float2*>(s0 + sbase + (size_t)row * kD + nj * 8 + 2 * q));
        const float2 x8 = __ldg(reinterpret_cast<const float2*>(s0 + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q));
        S[nj][0] = x0.x; S[nj][1] = x0.y; S[nj][2] = x8.x; S[nj][3] = x8.y;
      } else {
        S[nj][0] = S[nj][1] = S[nj][2] = S[nj][3] = 0.f;
      }
    }
    __syncthreads();  // chunk 0's operands are in place

    for (int n = 0; n < nsub; ++n) {
      unsigned char* cb = buf(n);
      const int c = chunk_of(n);
      const int t0 = c * kL, nm = clen(c);
      if (WALK && ck != nullptr) {  // G at the end of chunk c (before this chunk's transition)
        float* dst = ck + ((size_t)bh * nchunks + c) * kD * kD;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(dst + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(dst + (size_t)(row + 8) * kD + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
      }
      if (!slow_of(cb)) {
        const RM Ah = rm64(cb, Buf::cAh), Rh = rm64(cb, Buf::cRh), Bp = rm64(cb, Buf::cBp);
        const RM Cm = rm32(cb, Buf::cC), Pm = rm32(cb, Buf::cP);
        const float* GL = reinterpret_cast<const float*>(cb + Buf::cGL);
        FragA fs[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) fs[kk] = frag_from_acc(S[2 * kk], S[2 * kk + 1]);
        if (!WALK) {
          // P1 = S A^^T; S' = S o gamma + P1 B' + N; Y^T = S R^^T + P1 C^T + V^T P^T
          float p1[4][4] = {};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_b2(Ah, 2 * np, kk, lane, f0, f1);
              mma3(p1[2 * np], fs[kk], f0);
              mma3(p1[2 * np + 1], fs[kk], f1);
            }
          FragA fp[2];
          fp[0] = frag_from_acc(p1[0], p1[1]);
          fp[1] = frag_from_acc(p1[2], p1[3]);
          float acc[8][4] = {};
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int nq = 0; nq < 4; ++nq) {
              FragB f0, f1;
              rm_bt2(Bp, 2 * nq, kk, lane, f0, f1);
              mma3(acc[2 * nq], fp[kk], f0);
              mma3(acc[2 * nq + 1], fp[kk], f1);
            }
          float yv[4][4] = {};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_b2(Rh, 2 * np, kk, lane, f0, f1);
              mma3(yv[2 * np], fs[kk], f0);
              mma3(yv[2 * np + 1], fs[kk], f1);
            }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_b2(Cm, 2 * np, kk, lane, f0, f1);
              mma3(yv[2 * np], fp[kk], f0);
              mma3(yv[2 * np + 1], fp[kk], f1);
            }
          bsync<3, 128>();  // V (operand) and N = V^T K' are in shared memory
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const FragA fv = rm_at(Vop, mt, kk, lane);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_b2(Pm, 2 * np, kk, lane, f0, f1);
              if (kVExact) {
                mma2(yv[2 * np], fv, f0);
                mma2(yv[2 * np + 1], fv, f1);
              } else {
                mma3(yv[2 * np], fv, f0);
                mma3(yv[2 * np + 1], fv, f1);
              }
            }
          }
#pragma unroll
          for (int nj = 0; nj < 8; ++nj) {
            const float4 nv = *reinterpret_cast<const float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4);
            const float2 gl = *reinterpret_cast<const float2*>(GL + nj * 8 + 2 * q);
            S[nj][0] = fmaf(S[nj][0], gl.x, acc[nj][0] + nv.x);
            S[nj][1] = fmaf(S[nj][1], gl.y, acc[nj][1] + nv.y);
            S[nj][2] = fmaf(S[nj][2], gl.x, acc[nj][2] + nv.z);
            S[nj][3] = fmaf(S[nj][3], gl.y, acc[nj][3] + nv.w);
          }
          const int i0 = mt * 16 + g;
#pragma unroll
          for (int nj = 0; nj < 4; ++nj) {
            const int tt = nj * 8 + 2 * q;
            ys[tt * LY::kSY + i0] = yv[nj][0];
            ys[(tt + 1) * LY::kSY + i0] = yv[nj][1];
            ys[tt * LY::kSY + i0 + 8] = yv[nj][2];
            ys[(tt + 1) * LY::kSY + i0 + 8] = yv[nj][3];
          }
          barrive<4, 128>();
        } else {
          // Q = G B'^T + DY^T C (rows i, 32 tokens); G' = G o gamma + Q A^ + DY^T R^
          float qv[4][4] = {};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_b2(Bp, 2 * np, kk, lane, f0, f1);
              mma3(qv[2 * np], fs[kk], f0);
              mma3(qv[2 * np + 1], fs[kk], f1);
            }
          bsync<3, 128>();  // N2 = DY^T C and N = DY^T R^ are in shared memory
#pragma unroll
          for (int nj = 0; nj < 4; ++nj) {
            const float4 n2 = *reinterpret_cast<const float4*>(nb2 + ((mt * 4 + nj) * 32 + lane) * 4);
            qv[nj][0] += n2.x; qv[nj][1] += n2.y; qv[nj][2] += n2.z; qv[nj][3] += n2.w;
          }
          FragA fq[2];
          fq[0] = frag_from_acc(qv[0], qv[1]);
          fq[1] = frag_from_acc(qv[2], qv[3]);
          float acc[8][4] = {};
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int nq = 0; nq < 4; ++nq) {
              FragB f0, f1;
              rm_bt2(Ah, 2 * nq, kk, lane, f0, f1);
              mma3(acc[2 * nq], fq[kk], f0);
              mma3(acc[2 * nq + 1], fq[kk], f1);
            }
#pragma unroll
          for (int nj = 0; nj < 8; ++nj) {
            const float4 nv = *reinterpret_cast<const float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4);
            const float2 gl = *reinterpret_cast<const float2*>(GL + nj * 8 + 2 * q);
            S[nj][0] = fmaf(S[nj][0], gl.x, acc[nj][0] + nv.x);
            S[nj][1] = fmaf(S[nj][1], gl.y, acc[nj][1] + nv.y);
            S[nj][2] = fmaf(S[nj][2], gl.x, acc[nj][2] + nv.z);
            S[nj][3] = fmaf(S[nj][3], gl.y, acc[nj][3] + nv.w);
          }
        }
      } else {
        // ---- token by token (decay too strong for the transition form); inputs from global memory
        float* FS = reinterpret_cast<float*>(sm + LY::oFS);
        const int i0 = mt * 16 + g;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(FS + i0 * LY::kSFS + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(FS + (i0 + 8) * LY::kSFS + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
        bsync<2, 64>();
        const int ti = tid >> 1, half = tid & 1, c0 = 32 * half;
        float Sr[32];
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) Sr[cc] = FS[ti * LY::kSFS + c0 + cc];
        auto cols8 = [&](const Tin* src, int tok, int cc, float (&o)[8]) {
          load8(src + base + (size_t)tok * tstride + c0 + cc, o);
        };
        for (int tt = 0; tt < nm; ++tt) {
          const int tok = WALK ? t0 + nm - 1 - tt : t0 + tt;
          const float vi = to_f32(v[base + (size_t)tok * tstride + rb * kR + ti]);
          if (!WALK) {
            float s = 0.f;
#pragma unroll
            for (int cc = 0; cc < 32; cc += 8) {
              float av[8];
              cols8(a, tok, cc, av);
#pragma unroll
              for (int u = 0; u < 8; ++u) s = fmaf(Sr[cc + u], av[u], s);
            }
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            float yy = 0.f;
#pragma unroll
            for (int cc = 0; cc < 32; cc += 8) {
              float wv[8], kv[8], bv[8], rv[8];
              cols8(w, tok, cc, wv);
              cols8(k, tok, cc, kv);
              cols8(b, tok, cc, bv);
              cols8(r, tok, cc, rv);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                Sr[cc + u] = fmaf(Sr[cc + u], wv[u], fmaf(vi, kv[u], s * bv[u]));
                yy = fmaf(Sr[cc + u], rv[u], yy);
              }
            }
            yy += __shfl_xor_sync(0xffffffffu, yy, 1);
            if (half == 0) y[base + (size_t)tok * tstride + rb * kR + ti] = yy;
          } else {
            // X_t = X'_t + dy_t r_t^T; dsa_t = X_t b_t; X'_{t-1} = X_t diag(w_t) + dsa_t a_t^T
            float s = 0.f;
#pragma unroll
            for (int cc = 0; cc < 32; cc += 8) {
              float rv[8], bv[8];
              cols8(r, tok, cc, rv);
              cols8(b, tok, cc, bv);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                Sr[cc + u] = fmaf(vi, rv[u], Sr[cc + u]);
                s = fmaf(Sr[cc + u], bv[u], s);
              }
            }
            s += __shfl_xor_sync(0xffffffffu, s, 1);
#pragma unroll
            for (int cc = 0; cc < 32; cc += 8) {
              float wv[8], av[8];
              cols8(w, tok, cc, wv);
              cols8(a, tok, cc, av);
#pragma unroll
              for (int u = 0; u < 8; ++u) Sr[cc + u] = fmaf(Sr[cc + u], wv[u], s * av[u]);
            }
          }
        }
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) FS[ti * LY::kSFS + c0 + cc] = Sr[cc];
        bsync<2, 64>();
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          const float2 x0 = *reinterpret_cast<const float2*>(FS + i0 * LY::kSFS + nj * 8 + 2 * q);
          const float2 x8 = *reinterpret_cast<const float2*>(FS + (i0 + 8) * LY::kSFS + nj * 8 + 2 * q);
          S[nj][0] = x0.x; S[nj][1] = x0.y; S[nj][2] = x8.x; S[nj][3] = x8.y;
        }
      }
      if (!WALK && ck != nullptr) {  // the state after chunk c
        float* dst = ck + ((size_t)bh * nchunks + c) * kD * kD;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(dst + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(dst + (size_t)(row + 8) * kD + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
      }
      __syncthreads();  // end of period n
    }
    if (sT != nullptr) {
#pragma unroll
      for (int nj = 0; nj < 8; ++nj) {
        *reinterpret_cast<float2*>(sT + sbase + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
        *reinterpret_cast<float2*>(sT + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q) =
            make_float2(S[nj][2], S[nj][3]);
      }
    }
    return;
  }

  if (warp < 4) {
    // =============================================================== v (forward) / dy (walk) warps
    const int mt = warp - 2;
    const int ot = tid - 64;
    auto issue_v = [&](int n) {
      constexpr int VPR = kR * (int)sizeof(TV) / 16;
      constexpr int EPV = 16 / (int)sizeof(TV);
      TV* dst = vraw(n);
      const int c = chunk_of(n), t0 = c * kL, nm = clen(c);
      for (int e = ot; e < nm * VPR; e += 64) {
        const int t = e / VPR, pc = e % VPR;
        cp_async16(dst + t * kR + pc * EPV, v + base + (size_t)(t0 + t) * tstride + rb * kR + pc * EPV);
      }
      cp_async_commit();
    };
    if (nsub > 0) issue_v(0);
    __syncthreads();

    for (int n = 0; n < nsub; ++n) {
      unsigned char* cb = buf(n);
      const int c = chunk_of(n), t0 = c * kL, nm = clen(c);
      if (n + 1 < nsub) {
        issue_v(n + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      bsync<5, 64>();
      if (!slow_of(cb)) {
        {  // V / DY (rows t, columns i of this CTA) as an operand, rows past the chunk zero
          const TV* vb = vraw(n);
          const int t = ot >> 1, c0 = (ot & 1) * 16;
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = t < nm ? to_f32(vb[t * kR + c0 + 8 * h8 + u]) : 0.f;
            rm_store8(Vop, t, c0 + 8 * h8, x);
          }
        }
        bsync<5, 64>();
        if (!WALK) {  // N = V^T K'
          const RM Kp = rm64(cb, Buf::cKp);
          float acc[8][4] = {};
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const FragA fv = rm_at(Vop, mt, kk, lane);
#pragma unroll
            for (int nq = 0; nq < 4; ++nq) {
              FragB f0, f1;
              rm_bt2(Kp, 2 * nq, kk, lane, f0, f1);
              if (kVExact) {
                mma2(acc[2 * nq], fv, f0);
                mma2(acc[2 * nq + 1], fv, f1);
              } else {
                mma3(acc[2 * nq], fv, f0);
                mma3(acc[2 * nq + 1], fv, f1);
              }
            }
          }
#pragma unroll
          for (int nj = 0; nj < 8; ++nj)
            *reinterpret_cast<float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4) =
                make_float4(acc[nj][0], acc[nj][1], acc[nj][2], acc[nj][3]);
          barrive<3, 128>();
          bsync<4, 128>();  // y staged
          for (int e = ot; e < nm * (kR / 4); e += 64) {
            const int t = e >> 3, i = (e & 7) * 4;
            *reinterpret_cast<float4*>(y + base + (size_t)(t0 + t) * tstride + rb * kR + i) =
                *reinterpret_cast<const float4*>(ys + t * LY::kSY + i);
          }
        } else {  // N2 = DY^T C (rows i, 32 tokens), N = DY^T R^ (rows i, 64 columns)
          const RM Rh = rm64(cb, Buf::cRh), Cm = rm32(cb, Buf::cC);
          float a2[4][4] = {}, acc[8][4] = {};
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const FragA fv = rm_at(Vop, mt, kk, lane);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              FragB f0, f1;
              rm_bt2(Cm, 2 * np, kk, lane, f0, f1);
              mma3(a2[2 * np], fv, f0);
              mma3(a2[2 * np + 1], fv, f1);
            }
#pragma unroll
            for (int nq = 0; nq < 4; ++nq) {
              FragB f0, f1;
              rm_bt2(Rh, 2 * nq, kk, lane, f0, f1);
              mma3(acc[2 * nq], fv, f0);
              mma3(acc[2 * nq + 1], fv, f1);
            }
          }
#pragma unroll
          for (int nj = 0; nj < 4; ++nj)
            *reinterpret_cast<float4*>(nb2 + ((mt * 4 + nj) * 32 + lane) * 4) =
                make_float4(a2[nj][0], a2[nj][1], a2[nj][2], a2[nj][3]);
#pragma unroll
          for (int nj = 0; nj < 8; ++nj)
            *reinterpret_cast<float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4) =
                make_float4(acc[nj][0], acc[nj][1], acc[nj][2], acc[nj][3]);
          barrive<3, 128>();
        }
      }
      __syncthreads();
    }
    return;
  }

  // ================================================================= load warps (4)
  const int lt = tid - 128;  // 0 .. 127
  const int lw = lt >> 5;
  float* const G = reinterpret_cast<float*>(sm + LY::oG);
  auto rawbuf = [&](int n) { return reinterpret_cast<Tin*>(sm + LY::oRaw + (n & 1) * LY::kRaw); };
  // cp.async: chunk n's operands (B', K', C, P, gamma_31, flag) into buf(n) and its w, a, r into raw(n)
  auto issue = [&](int n) {
    const int c = chunk_of(n), t0 = c * kL, nm = clen(c);
    unsigned char* cb = buf(n);
    const unsigned char* src = ops + ((size_t)bh * nchunks + c) * kOpBytes;
    copy_rm<false>(rm64(cb, Buf::cBp), 32, 64, const_cast<unsigned char*>(src + kOpBp), lt, 128);
    copy_rm<false>(rm64(cb, Buf::cKp), 32, 64, const_cast<unsigned char*>(src + kOpKp), lt, 128);
    copy_rm<false>(rm32(cb, Buf::cC), 32, 32, const_cast<unsigned char*>(src + kOpC), lt, 128);
    copy_rm<false>(rm32(cb, Buf::cP), 32, 32, const_cast<unsigned char*>(src + kOpP), lt, 128);
    if (lt < 17) cp_async16(cb + Buf::cGL + lt * 16, src + kOpGL + lt * 16);  // gamma_31 and the flag
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    Tin* dst = rawbuf(n);
    const Tin* srcs[3] = {w, a, r};
#pragma unroll
    for (int s3 = 0; s3 < 3; ++s3)
      for (int e = lt; e < nm * CPR; e += 128) {
        const int t = e / CPR, pc = e % CPR;
        cp_async16(dst + (s3 * kL + t) * kD + pc * EPC, srcs[s3] + base + (size_t)(t0 + t) * tstride + pc * EPC);
      }
    cp_async_commit();
  };
  // decays, A^ and R^ of chunk n into buf(n) (its copies have landed)
  auto rebuild = [&](int n) {
    const int c = chunk_of(n), nm = clen(c);
    unsigned char* cb = buf(n);
    if (slow_of(cb)) return;
    const Tin* rw = rawbuf(n);
    const Tin* ra = rw + kL * kD;
    const Tin* rr = rw + 2 * kL * kD;
    if (lt < kD) {
      const int j = lt;
      float gm = 1.f;
#pragma unroll 8
      for (int t = 0; t < kL; ++t) {
        gm *= t < nm ? to_f32(rw[t * kD + j]) : 1.f;
        G[t * kD + j] = gm;
      }
    }
    bsync<6, 128>();
    const RM Ah = rm64(cb, Buf::cAh), Rh = rm64(cb, Buf::cRh);
    for (int e = lt; e < 256; e += 128) {
      const int t = e >> 3, c0 = (e & 7) * 8;
      const bool ok = t < nm;
      float gt[8], gp[8], av[8], rv[8];
      raw8(G + t * kD + c0, gt);
      if (t > 0) {
        raw8(G + (t - 1) * kD + c0, gp);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) gp[u] = 1.f;
      }
      raw8(ra + t * kD + c0, av);
      raw8(rr + t * kD + c0, rv);
      float oa[8], orr[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        oa[u] = ok ? av[u] * gp[u] : 0.f;
        orr[u] = ok ? rv[u] * gt[u] : 0.f;
      }
      rm_store8(Ah, t, c0, oa);
      rm_store8(Rh, t, c0, orr);
    }
    bsync<6, 128>();  // G is free for the next chunk
  };
  if (nsub > 0) {
    issue(0);
    if (nsub > 1) issue(1);
    if (nsub > 1) cp_async_wait<1>(); else cp_async_wait<0>();
    bsync<6, 128>();
    rebuild(0);
  }
  __syncthreads();  // chunk 0's operands are in place
  for (int n = 0; n < nsub; ++n) {
    // buf(n + 2) held chunk n - 1 (done): refill; chunk n + 1's copies (issued a period ago) land
    if (n + 2 < nsub) {
      issue(n + 2);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    bsync<6, 128>();
    if (n + 1 < nsub) rebuild(n + 1);
    __syncthreads();  // end of period n
  }
}

template <typename Tin>
cudaError_t launch_prep_t(int B, int T, int H, int nchunks, const void* r, const void* w, const void* k,
                          const void* a, const void* b, unsigned char* ops, cudaStream_t stream) {
  using LY = PrepLay<Tin>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  auto kern = ops_prep_kernel<Tin>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)B * H * nchunks;
  kern<<<grid, kNTP, LY::kBytes, stream>>>(T, H, nchunks, (const Tin*)r, (const Tin*)w, (const Tin*)k,
                                           (const Tin*)a, (const Tin*)b, ops);
  return cudaGetLastError();
}

template <typename Tin, bool WALK>
cudaError_t launch_ochain_t(int B, int T, int H, int nchunks, const void* r, const void* w, const void* k,
                            const void* v, const void* a, const void* b, const unsigned char* ops, const float* s0,
                            float* y, float* ck, float* sT, cudaStream_t stream) {
  using TV = typename std::conditional<WALK, float, Tin>::type;
  using LY = ChainLay<Tin, TV>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  auto kern = ops_chain_kernel<Tin, WALK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)B * H * 2;
  kern<<<grid, kNTC, LY::kBytes, stream>>>(T, H, nchunks, (const Tin*)r, (const Tin*)w, (const Tin*)k, v,
                                           (const Tin*)a, (const Tin*)b, ops, s0, y, ck, sT);
  return cudaGetLastError();
}

}  // namespace

size_t transition_ops_bytes(int B, int T, int H) {
  const size_t C = T > 0 ? (size_t)((T + kL - 1) / kL) : 0;
  return (size_t)B * H * C * kOpBytes;
}

cudaError_t launch_transition_ops(const FwdArgs& p, unsigned char* ops, cudaStream_t stream) {
  if (p.nchunks == 0) return cudaSuccess;
  return p.bf16 ? launch_prep_t<__nv_bfloat16>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.in.a, p.in.b, ops,
                                               stream)
                : launch_prep_t<float>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.in.a, p.in.b, ops, stream);
}

cudaError_t launch_forward_from_ops(const FwdArgs& p, const unsigned char* ops, cudaStream_t stream) {
  return p.bf16 ? launch_ochain_t<__nv_bfloat16, false>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.in.v,
                                                        p.in.a, p.in.b, ops, p.h0, p.y, p.h_ckpt, p.hT, stream)
                : launch_ochain_t<float, false>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.in.v, p.in.a,
                                                p.in.b, ops, p.h0, p.y, p.h_ckpt, p.hT, stream);
}

cudaError_t launch_walk_from_ops(const BwdArgs& p, const unsigned char* ops, float* g_ends, cudaStream_t stream) {
  return p.bf16 ? launch_ochain_t<__nv_bfloat16, true>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.dy,
                                                       p.in.a, p.in.b, ops, p.dhT, nullptr, g_ends, p.dh0, stream)
                : launch_ochain_t<float, true>(p.B, p.T, p.H, p.nchunks, p.in.r, p.in.w, p.in.k, p.dy, p.in.a,
                                               p.in.b, ops, p.dhT, nullptr, g_ends, p.dh0, stream);
}

}  // namespace wkv7
