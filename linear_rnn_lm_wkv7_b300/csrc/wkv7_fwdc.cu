// WKV7 forward on sm_103a in sub-chunks of 16 tokens, the dense contractions on tensor cores.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
// architecture", Forward listing), per head, state S (rows i = value, columns j = key):
//     sa_t = S_{t-1} a_t;   S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T;   y_t = S_t r_t
// with S written out after every `chunk` tokens.
//
// Sub-chunk form (exact in real arithmetic).  Over 16 tokens t = 0..15 starting from S, with
// gamma_t = w_0 o .. o w_t (per column) and gamma_L = gamma_15:
//     A^_t = a_t o gamma_{t-1},  R^_t = r_t o gamma_t,  K~_s = k_s / gamma_s,  B~_s = b_s / gamma_s,
//     K-_s = k_s o gamma_L / gamma_s,  B-_s = b_s o gamma_L / gamma_s
//     M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T)
//     SA = (I - M_ab)^-1 (A^ S^T + M_ak V)                  (rows t: sa_t)
//     Y  = R^ S^T + M_rk V + M_rb SA                         (rows t: y_t)
//     S' = S diag(gamma_L) + V^T K- + SA^T B-
// Unrolling S_t over the sub-chunk gives these directly: sa_t and y_t are dots of the start state
// with decayed a_t / r_t plus the sub-chunk's own rank-one terms, coupled through sa by the unit
// lower-triangular system (I - M_ab).  The serial chain is one sub-chunk step per 16 tokens.
//
// Precision.  Products of fp32 operands on the tensor cores use three TF32 passes (x = hi + lo,
// hi lo + lo hi + hi hi), fp32 accumulation: ~1e-7 relative against the fp64 recurrence at the
// training shapes (one TF32 pass gives ~3e-4).  (I - M_ab)^-1, M_ak / M_rk times V and the decay
// factors are plain fp32.  1/gamma grows like (1/w)^16; a sub-chunk whose gamma_L falls below
// 1e-30 in some column is instead advanced token by token (exact, slow), so any w in (0, 1] is
// handled.
//
// Mapping: one CTA per (head, 32-row block), 12 warps.  Warps 0-1 hold the CTA's 32 x 64 slice of
// S as mma.sync m16n8k8 accumulator tiles (warp m = rows 16m..16m+15), run the chain and write y
// and sa; warps 2-11 prepare the next sub-chunk (decays, the four 16x16 coupling matrices and
// U = V^T K- on tensor cores, (I - M_ab)^-1 by forward substitution, a column per lane, the V corrections on tensor
// cores) one sub-chunk ahead.  One CTA barrier per sub-chunk.  An accumulator tile is reused
// directly as the A operand of the next product by permuting the contraction index inside each
// 8-block (logical k = q <-> column 2q, k = q + 4 <-> column 2q + 1); the B operands are stored in
// shared memory already split into hi/lo and paired to match.
//
// The same kernel runs the backward's state-gradient walk (GRAD): that recurrence, read from the
// last token down, has the forward's form with the inputs remapped (see FwdcPtrs and `issue`).
#include <type_traits>

#include "wkv7_device.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kL = 16;     // tokens per sub-chunk
constexpr int kR = 32;     // state rows per CTA
constexpr int kNT = 384;   // threads per CTA
constexpr int kNP = 320;   // preparing threads (warps 2-11)
constexpr int kChainThreads = 64;

// padded row strides: 16-byte (hi0, hi1, lo0, lo1) words for the split pair arrays, floats otherwise
constexpr int kSP = 36;    // [16][32 pairs] (+4): A^, R^, K~, B~
constexpr int kSM = 12;    // [16][8 pairs] (+4): (I - M_ab)^-1, M_rb
constexpr int kSJ = 66;    // [8 token pairs][64] (+2): K-, B-
constexpr int kSC = 24;    // [32][16] fp32 (+8): the V corrections of sa and y
constexpr int kSU = 72;    // [32][64] fp32 (+8): U = V^T K-, and the state in the token-by-token path
constexpr int kSO = 36;    // [16][32] fp32 (+4): y / sa staging
constexpr int kSF = 72;    // [16][64] fp32 (+8): K~, B~
constexpr int kSJ2 = 68;   // [8 token pairs][64] float2 (+4): K-
constexpr int kSV2 = 36;   // [8 token pairs][32] float2 (+4): V
constexpr float kMinDecay = 1e-30f;

template <typename Tin, typename TV>
struct Lay {
  // raw input stage (x2): w, k, a, b, r [kL][64] (Tin), then v [kL][32] (TV)
  static constexpr size_t kRaw = (5 * kL * kD * sizeof(Tin) + 15) / 16 * 16 + (kL * kR * sizeof(TV) + 15) / 16 * 16;
  static constexpr size_t oRaw = 0;
  // chain buffer (x2): what the chain reads for one sub-chunk
  static constexpr size_t cAH = 0;                          // uint4 [16][kSP]
  static constexpr size_t cRH = cAH + 16 * kSP * 16;
  static constexpr size_t cTI = cRH + 16 * kSP * 16;        // float [16][kSC]: (I - M_ab)^-1
  static constexpr size_t cMRB = cTI + 16 * kSC * 4;        // uint4 [16][kSM]
  static constexpr size_t cCAK = cMRB + 16 * kSM * 16;      // float [32][kSC]: V^T M_ak^T
  static constexpr size_t cCY = cCAK + 32 * kSC * 4;        // float [32][kSC]: V^T M_rk^T
  static constexpr size_t cU = cCY + 32 * kSC * 4;          // float [32][kSU]
  static constexpr size_t cBB = cU + 32 * kSU * 4;          // uint4 [8][kSJ]
  static constexpr size_t cGL = cBB + 8 * kSJ * 16;         // float [64]
  static constexpr size_t cMeta = cGL + 64 * 4;             // int [4]: token-by-token flag, tokens
  static constexpr size_t kChain = cMeta + 16;
  // in the token-by-token path the same buffer holds the fp32 inputs: w k a b r [16][64], v [16][32]
  static constexpr size_t cFW = 0;
  static constexpr size_t kFallbackInputs = (5 * kL * kD + kL * kR) * 4;
  static_assert(kFallbackInputs <= cCAK, "token-by-token inputs fit below the corrections");
  static constexpr size_t oChain = oRaw + 2 * kRaw;
  // preparation scratch
  static constexpr size_t oG = oChain + 2 * kChain;          // float [16][64] gamma
  static constexpr size_t oKT = oG + kL * kD * 4;            // float [16][kSF]: K~, B~
  static constexpr size_t oBT = oKT + 16 * kSF * 4;
  static constexpr size_t oKB = oBT + 16 * kSF * 4;          // float2 [8][kSJ2]: K- in token pairs
  static constexpr size_t oVP = oKB + 8 * kSJ2 * 8;          // float2 [8][kSV2]: V in token pairs
  static constexpr size_t oMAK = oVP + 8 * kSV2 * 8;          // uint4 [16][kSM] each: M_ak, M_rk split
  static constexpr size_t oMRK = oMAK + 16 * kSM * 16;
  static constexpr size_t oMAB = oMRK + 16 * kSM * 16;       // float [16][16]: M_ab
  // output staging (x2): y, sa [16][kSO]
  static constexpr size_t oOut = oMAB + 1024;
  static constexpr size_t kOut = 2 * kL * kSO * 4;
  // state of the token-by-token path: float [32][kSU]
  static constexpr size_t oFS = oOut + 2 * kOut;
  static constexpr size_t kBytes = oFS + kR * kSU * 4;
};

// ---------------------------------------------------------------- tensor-core helpers

// x = hi + lo, hi = x rounded to the nearest TF32 value (ties away from zero: adding half a TF32
// unit to the magnitude bits, then dropping the low 13), lo = x - hi exactly, |lo| <= 2^-11 |x|;
// the tensor core reads lo's top 19 bits.  Relative error ~2^-22 per product in three passes.
// (Finite x below 2^127 only -- every operand here is.)
__device__ __forceinline__ void split(float x, uint32_t& hi, uint32_t& lo) {
  hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}


// (hi x0, hi x1, lo x0, lo x1)
__device__ __forceinline__ uint4 split_pair(float x0, float x1) {
  uint4 q;
  split(x0, q.x, q.z);
  split(x1, q.y, q.w);
  return q;
}

struct FragA {
  uint32_t h[4], l[4];
};
struct FragB {
  uint32_t h[2], l[2];
};

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += A B in three TF32 passes, the small terms first
__device__ __forceinline__ void mma3(float (&d)[4], const FragA& a, const FragB& b) {
  mma_tf32(d, a.l, b.h[0], b.h[1]);
  mma_tf32(d, a.h, b.l[0], b.l[1]);
  mma_tf32(d, a.h, b.h[0], b.h[1]);
}

// An accumulator tile (rows g, g+8; columns 2q, 2q+1 of an 8-block) as the A operand of a product
// contracting over those columns, with k = q <-> column 2q and k = q + 4 <-> column 2q + 1.
__device__ __forceinline__ FragA frag_from_acc(const float (&c)[4]) {
  FragA a;
  split(c[0], a.h[0], a.l[0]);
  split(c[2], a.h[1], a.l[1]);
  split(c[1], a.h[2], a.l[2]);
  split(c[3], a.h[3], a.l[3]);
  return a;
}

// A operand from split pairs: row g -> (a0, a2), row g + 8 -> (a1, a3)
__device__ __forceinline__ FragA frag_a(uint4 r0, uint4 r8) {
  FragA a;
  a.h[0] = r0.x; a.h[2] = r0.y; a.l[0] = r0.z; a.l[2] = r0.w;
  a.h[1] = r8.x; a.h[3] = r8.y; a.l[1] = r8.z; a.l[3] = r8.w;
  return a;
}

// A operand from fp32 pairs: row g -> (a0, a2), row g + 8 -> (a1, a3), split here
__device__ __forceinline__ FragA frag_a2(float2 r0, float2 r8) {
  FragA a;
  split(r0.x, a.h[0], a.l[0]);
  split(r0.y, a.h[2], a.l[2]);
  split(r8.x, a.h[1], a.l[1]);
  split(r8.y, a.h[3], a.l[3]);
  return a;
}

// B operand from an fp32 pair (b0, b1), split here
__device__ __forceinline__ FragB frag_b2(float2 v) {
  FragB b;
  split(v.x, b.h[0], b.l[0]);
  split(v.y, b.h[1], b.l[1]);
  return b;
}

__device__ __forceinline__ FragB frag_b(uint4 q) {
  FragB b;
  b.h[0] = q.x; b.h[1] = q.y; b.l[0] = q.z; b.l[1] = q.w;
  return b;
}

__device__ __forceinline__ void bar_prep() { asm volatile("bar.sync 1, %0;\n" ::"n"(kNP) : "memory"); }
__device__ __forceinline__ void bar_chain() { asm volatile("bar.sync 2, %0;\n" ::"n"(kChainThreads) : "memory"); }
// preparing warps 1-9
__device__ __forceinline__ void bar_rest() { asm volatile("bar.sync 3, %0;\n" ::"n"(kNP - 32) : "memory"); }
// preparing warp 1 hands its M_ab tile to warp 0
__device__ __forceinline__ void bar_pair_sync() { asm volatile("bar.sync 4, 64;\n" ::: "memory"); }
__device__ __forceinline__ void bar_pair_arrive() { asm volatile("bar.arrive 4, 64;\n" ::: "memory"); }

template <typename Tin>
__device__ __forceinline__ float raw_at(const Tin* p) {
  return to_f32(*p);
}

// two consecutive raw values (the pair starts on an even element)
__device__ __forceinline__ float2 raw2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 raw2(const __nv_bfloat16* p) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(bf16_lo(u), bf16_hi(u));
}

// ---------------------------------------------------------------- the kernel

// Pointers of one call.  Forward: the inputs, s0 = h0, y, ck = h_ckpt, sT = hT, sa.  Gradient walk
// (GRAD): the inputs with v = dy (fp32), s0 = dhT, y = dv, ck = X at the chunk ends, sT = dh0,
// sa = dsa (every one of them laid out as in the forward).
struct FwdcPtrs {
  const void *r, *w, *k, *v, *a, *b;
  const float* s0;
  float *y, *ck, *sT, *sa;
};

// all-ones (bf16 or fp32 1.0) or all-zero 16 bytes
template <typename T>
__device__ __forceinline__ uint4 fill16(bool one) {
  const uint32_t u = !one ? 0u : (sizeof(T) == 2 ? 0x3f803f80u : 0x3f800000u);
  return make_uint4(u, u, u, u);
}

template <typename Tin, bool GRAD>
__global__ void __launch_bounds__(kNT, 1)
fwdc_kernel(int T, int H, int chunk, int nchunks, FwdcPtrs P) {
  using TV = typename std::conditional<GRAD, float, Tin>::type;
  using LY = Lay<Tin, TV>;
  const Tin* __restrict__ r = static_cast<const Tin*>(P.r);
  const Tin* __restrict__ w = static_cast<const Tin*>(P.w);
  const Tin* __restrict__ k = static_cast<const Tin*>(P.k);
  const TV* __restrict__ v = static_cast<const TV*>(P.v);
  const Tin* __restrict__ a = static_cast<const Tin*>(P.a);
  const Tin* __restrict__ b = static_cast<const Tin*>(P.b);
  const float* __restrict__ h0 = P.s0;
  float* __restrict__ y = P.y;
  float* __restrict__ h_ckpt = P.ck;
  float* __restrict__ hT = P.sT;
  float* __restrict__ sa_out = P.sa;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);

  const int bh = blockIdx.x >> 1;
  const int rb = blockIdx.x & 1;
  const int bi = bh / H;
  const int hi = bh - bi * H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t sbase = (size_t)bh * kD * kD;
  // Sub-chunk schedule over the steps.  Forward: steps = tokens, 16 per sub-chunk.  Gradient walk:
  // T + 1 steps, step s for token T - 1 - s (the last one yields dh0); a first sub-chunk of one
  // step and a second of ((T - 1) % 16) + 1 put every chunk end on a sub-chunk end.
  const int len2 = GRAD && T > 0 ? (T - 1) % kL + 1 : 0;
  const int nsub = GRAD ? (T > 0 ? 2 + (T - len2) / kL : 0) : (T + kL - 1) / kL;
  auto sub_start = [&](int m) { return GRAD ? (m == 0 ? 0 : (m == 1 ? 1 : 1 + len2 + kL * (m - 2))) : m * kL; };
  auto sub_len = [&](int m) { return GRAD ? (m == 0 ? 1 : (m == 1 ? len2 : kL)) : min(kL, T - m * kL); };

  auto raw_buf = [&](int m) { return reinterpret_cast<Tin*>(sm + LY::oRaw + (size_t)(m & 1) * LY::kRaw); };
  auto chain_buf = [&](int m) { return sm + LY::oChain + (size_t)(m & 1) * LY::kChain; };
  auto out_y = [&](int m) { return reinterpret_cast<float*>(sm + LY::oOut + (size_t)(m & 1) * LY::kOut); };
  auto out_sa = [&](int m) { return out_y(m) + kL * kSO; };

  if (warp < 2) {
    // =========================================================== chain warps
    const int mi = warp;
    const int g = lane >> 2, q = lane & 3;
    const int row = rb * kR + mi * 16 + g;  // rows row and row + 8 of the head
    float S[8][4];
#pragma unroll
    for (int nj = 0; nj < 8; ++nj) {
      if (h0 != nullptr) {
        const float2 s0 = __ldg(reinterpret_cast<const float2*>(h0 + sbase + (size_t)row * kD + nj * 8 + 2 * q));
        const float2 s8 = __ldg(reinterpret_cast<const float2*>(h0 + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q));
        S[nj][0] = s0.x; S[nj][1] = s0.y; S[nj][2] = s8.x; S[nj][3] = s8.y;
      } else {
        S[nj][0] = S[nj][1] = S[nj][2] = S[nj][3] = 0.f;
      }
    }
    __syncthreads();  // the preparation of sub-chunk 0 is done

    for (int n = 0; n < nsub; ++n) {
      const unsigned char* cb = chain_buf(n);
      const int* meta = reinterpret_cast<const int*>(cb + LY::cMeta);
      const int slow = meta[0];
      const int nm = meta[1];
      float* fy = out_y(n);
      float* fsa = out_sa(n);
      if (!slow) {
        const uint4* AH = reinterpret_cast<const uint4*>(cb + LY::cAH);
        const uint4* RH = reinterpret_cast<const uint4*>(cb + LY::cRH);
        const float* TI = reinterpret_cast<const float*>(cb + LY::cTI);
        const uint4* MRB = reinterpret_cast<const uint4*>(cb + LY::cMRB);
        const float* CAK = reinterpret_cast<const float*>(cb + LY::cCAK);
        const float* CY = reinterpret_cast<const float*>(cb + LY::cCY);
        const float* U = reinterpret_cast<const float*>(cb + LY::cU);
        const uint4* BB = reinterpret_cast<const uint4*>(cb + LY::cBB);
        const float* GL = reinterpret_cast<const float*>(cb + LY::cGL);
        const int i0 = mi * 16 + g;  // local rows i0, i0 + 8

        // P^T = V^T M_ak^T + S A^T and Y^T = V^T M_rk^T + S R^T (rows i, tokens t).  Every tensor-core
        // product accumulates from zero in two accumulators per tile (the tensor core's own
        // accumulation does not round to nearest) and is added to the rest with fp32 adds.
        float P[2][2][4], Y[2][2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) P[nt][0][e] = P[nt][1][e] = Y[nt][0][e] = Y[nt][1][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const FragA as = frag_from_acc(S[kk]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            mma3(P[nt][kk & 1], as, frag_b(AH[(nt * 8 + g) * kSP + kk * 4 + q]));
            mma3(Y[nt][kk & 1], as, frag_b(RH[(nt * 8 + g) * kSP + kk * 4 + q]));
          }
        }
        float Pt[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 c0 = *reinterpret_cast<const float2*>(CY + i0 * kSC + nt * 8 + 2 * q);
          const float2 c8 = *reinterpret_cast<const float2*>(CY + (i0 + 8) * kSC + nt * 8 + 2 * q);
          const float2 d0 = *reinterpret_cast<const float2*>(CAK + i0 * kSC + nt * 8 + 2 * q);
          const float2 d8 = *reinterpret_cast<const float2*>(CAK + (i0 + 8) * kSC + nt * 8 + 2 * q);
          const float cy[4] = {c0.x, c0.y, c8.x, c8.y}, cak[4] = {d0.x, d0.y, d8.x, d8.y};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            Pt[nt][e] = (P[nt][0][e] + P[nt][1][e]) + cak[e];
            Y[nt][0][e] = (Y[nt][0][e] + Y[nt][1][e]) + cy[e];
          }
        }

        // SA^T = P^T (I - M_ab)^-T
        float SA[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) SA[nt][0] = SA[nt][1] = SA[nt][2] = SA[nt][3] = 0.f;
        {
          const FragA p0 = frag_from_acc(Pt[0]);
          const FragA p1 = frag_from_acc(Pt[1]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            mma3(SA[nt], p0, frag_b2(*reinterpret_cast<const float2*>(TI + (nt * 8 + g) * kSC + 2 * q)));
            mma3(SA[nt], p1, frag_b2(*reinterpret_cast<const float2*>(TI + (nt * 8 + g) * kSC + 8 + 2 * q)));
          }
        }
        const FragA s0 = frag_from_acc(SA[0]);
        const FragA s1 = frag_from_acc(SA[1]);
        // Y^T += SA^T M_rb^T
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float yb[4] = {0.f, 0.f, 0.f, 0.f};
          mma3(yb, s0, frag_b(MRB[(nt * 8 + g) * kSM + q]));
          mma3(yb, s1, frag_b(MRB[(nt * 8 + g) * kSM + 4 + q]));
#pragma unroll
          for (int e = 0; e < 4; ++e) Y[nt][0][e] += yb[e];
        }
        // stage y and sa as [t][i]
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int t0 = nt * 8 + 2 * q;
          fy[t0 * kSO + i0] = Y[nt][0][0];
          fy[(t0 + 1) * kSO + i0] = Y[nt][0][1];
          fy[t0 * kSO + i0 + 8] = Y[nt][0][2];
          fy[(t0 + 1) * kSO + i0 + 8] = Y[nt][0][3];
          fsa[t0 * kSO + i0] = SA[nt][0];
          fsa[(t0 + 1) * kSO + i0] = SA[nt][1];
          fsa[t0 * kSO + i0 + 8] = SA[nt][2];
          fsa[(t0 + 1) * kSO + i0 + 8] = SA[nt][3];
        }
        // S <- S diag(gamma_L) + U + SA^T B-
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          const float2 gl = *reinterpret_cast<const float2*>(GL + nj * 8 + 2 * q);
          const float2 u0 = *reinterpret_cast<const float2*>(U + i0 * kSU + nj * 8 + 2 * q);
          const float2 u8 = *reinterpret_cast<const float2*>(U + (i0 + 8) * kSU + nj * 8 + 2 * q);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma3(d, s0, frag_b(BB[q * kSJ + nj * 8 + g]));
          mma3(d, s1, frag_b(BB[(4 + q) * kSJ + nj * 8 + g]));
          S[nj][0] = fmaf(S[nj][0], gl.x, u0.x + d[0]);
          S[nj][1] = fmaf(S[nj][1], gl.y, u0.y + d[1]);
          S[nj][2] = fmaf(S[nj][2], gl.x, u8.x + d[2]);
          S[nj][3] = fmaf(S[nj][3], gl.y, u8.y + d[3]);
        }
      } else {
        // ---- token by token (decay too strong for the sub-chunk form)
        float* FS = reinterpret_cast<float*>(sm + LY::oFS);
        const float* FW = reinterpret_cast<const float*>(cb + LY::cFW);
        const float* FK = FW + kL * kD;
        const float* FA = FK + kL * kD;
        const float* FB = FA + kL * kD;
        const float* FR = FB + kL * kD;
        const float* FV = FR + kL * kD;
        const int i0 = mi * 16 + g;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(FS + i0 * kSU + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(FS + (i0 + 8) * kSU + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
        bar_chain();
        const int ti = tid >> 1, half = tid & 1, c0 = 32 * half;
        float Sr[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) Sr[c] = FS[ti * kSU + c0 + c];
        for (int t = 0; t < nm; ++t) {
          float s = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) s = fmaf(Sr[c], FA[t * kD + c0 + c], s);
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          const float vi = FV[t * kR + ti];
          float yy = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            Sr[c] = fmaf(Sr[c], FW[t * kD + c0 + c], fmaf(vi, FK[t * kD + c0 + c], s * FB[t * kD + c0 + c]));
            yy = fmaf(Sr[c], FR[t * kD + c0 + c], yy);
          }
          yy += __shfl_xor_sync(0xffffffffu, yy, 1);
          if (half == 0) {
            fy[t * kSO + ti] = yy;
            fsa[t * kSO + ti] = s;
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) FS[ti * kSU + c0 + c] = Sr[c];
        bar_chain();
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          const float2 s0 = *reinterpret_cast<const float2*>(FS + i0 * kSU + nj * 8 + 2 * q);
          const float2 s8 = *reinterpret_cast<const float2*>(FS + (i0 + 8) * kSU + nj * 8 + 2 * q);
          S[nj][0] = s0.x; S[nj][1] = s0.y; S[nj][2] = s8.x; S[nj][3] = s8.y;
        }
        bar_chain();  // FS is free for the next sub-chunk
      }

      // y and sa of this sub-chunk to global memory (both chain warps have staged theirs)
      bar_chain();
      const int tau0 = sub_start(n);
      for (int e = tid; e < nm * (kR / 4); e += kChainThreads) {
        const int t = e >> 3, i = (e & 7) * 4;
        const float4 vy = *reinterpret_cast<const float4*>(fy + t * kSO + i);
        const float4 vs = *reinterpret_cast<const float4*>(fsa + t * kSO + i);
        if (!GRAD) {
          const size_t o = base + (size_t)(tau0 + t) * tstride + rb * kR + i;
          *reinterpret_cast<float4*>(y + o) = vy;
          if (sa_out != nullptr) *reinterpret_cast<float4*>(sa_out + o) = vs;
        } else {  // step s: y' is dv at token T-1-s, sa' is dsa at token T-s
          const int st = tau0 + t;
          if (st <= T - 1) *reinterpret_cast<float4*>(y + base + (size_t)(T - 1 - st) * tstride + rb * kR + i) = vy;
          if (st >= 1) *reinterpret_cast<float4*>(sa_out + base + (size_t)(T - st) * tstride + rb * kR + i) = vs;
        }
      }

      // the state after the sub-chunk's last step when that ends a chunk (forward: token 32c+31 or
      // T-1; gradient walk: step T-1-t for a chunk end t, i.e. X_t)
      const int tlast = tau0 + nm - 1;
      const bool at_end = GRAD ? (tlast < T && (tlast == 0 || (T - tlast) % chunk == 0))
                               : ((tlast + 1) % chunk == 0 || tlast == T - 1);
      const int cidx = GRAD ? (T - 1 - tlast) / chunk : tlast / chunk;
      if (h_ckpt != nullptr && at_end) {
        float* dst = h_ckpt + ((size_t)bh * nchunks + cidx) * kD * kD;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(dst + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(dst + (size_t)(row + 8) * kD + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
      }
      __syncthreads();  // end of period n
    }
    if (hT != nullptr) {
#pragma unroll
      for (int nj = 0; nj < 8; ++nj) {
        *reinterpret_cast<float2*>(hT + sbase + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
        *reinterpret_cast<float2*>(hT + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q) =
            make_float2(S[nj][2], S[nj][3]);
      }
    }
    return;
  }

  // ============================================================= preparing warps
  const int pt = tid - kChainThreads;  // 0 .. 319
  const int pw = pt >> 5;              // 0 .. 9
  const int g = lane >> 2, q = lane & 3;
  float* G = reinterpret_cast<float*>(sm + LY::oG);
  float* KT = reinterpret_cast<float*>(sm + LY::oKT);
  float* BT = reinterpret_cast<float*>(sm + LY::oBT);
  float2* KB = reinterpret_cast<float2*>(sm + LY::oKB);
  float2* VP = reinterpret_cast<float2*>(sm + LY::oVP);
  uint4* MAK = reinterpret_cast<uint4*>(sm + LY::oMAK);
  uint4* MRK = reinterpret_cast<uint4*>(sm + LY::oMRK);
  float* MAB = reinterpret_cast<float*>(sm + LY::oMAB);

  // cp.async copies of sub-chunk m's inputs; steps past the sub-chunk are not copied and read as
  // padding.  Gradient walk: slots w, k, a, b, r, v take w, r, b, a, k at tokens T - s (w, a, b) or
  // T - 1 - s (k, r) and dy at T - 1 - s; a step outside [0, T) gets w = 1 and zeros.
  auto issue = [&](int m) {
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    constexpr int VPR = kR * (int)sizeof(TV) / 16;
    constexpr int EPV = 16 / (int)sizeof(TV);
    Tin* dst = raw_buf(m);
    TV* dstv = reinterpret_cast<TV*>(dst + 5 * kL * kD);
    const int t0 = sub_start(m);
    const int nm = sub_len(m);
    const Tin* srcs[5] = {w, k, a, b, r};
    if (GRAD) {
      srcs[1] = r;
      srcs[2] = b;
      srcs[3] = a;
      srcs[4] = k;
    }
#pragma unroll
    for (int s5 = 0; s5 < 5; ++s5)
      for (int e = pt; e < nm * CPR; e += kNP) {
        const int t = e / CPR, pc = e % CPR;
        Tin* d = dst + (s5 * kL + t) * kD + pc * EPC;
        const int tok = !GRAD ? t0 + t : ((s5 == 0 || s5 == 2 || s5 == 3) ? T - (t0 + t) : T - 1 - (t0 + t));
        if (tok >= 0 && tok < T)
          cp_async16(d, srcs[s5] + base + (size_t)tok * tstride + pc * EPC);
        else
          *reinterpret_cast<uint4*>(d) = fill16<Tin>(s5 == 0);
      }
    for (int e = pt; e < nm * VPR; e += kNP) {
      const int t = e / VPR, pc = e % VPR;
      TV* d = dstv + t * kR + pc * EPV;
      const int tok = GRAD ? T - 1 - (t0 + t) : t0 + t;
      if (tok >= 0)
        cp_async16(d, v + base + (size_t)tok * tstride + rb * kR + pc * EPV);
      else
        *reinterpret_cast<uint4*>(d) = fill16<TV>(false);
    }
    cp_async_commit();
  };

  // everything the chain needs for sub-chunk m, into chain buffer m & 1 (its raw inputs have landed)
  auto prepare = [&](int m) {
    const Tin* raw = raw_buf(m);
    const Tin* rw = raw;
    const Tin* rk = raw + kL * kD;
    const Tin* ra = raw + 2 * kL * kD;
    const Tin* rbv = raw + 3 * kL * kD;
    const Tin* rr = raw + 4 * kL * kD;
    const TV* rv = reinterpret_cast<const TV*>(raw + 5 * kL * kD);
    unsigned char* cb = chain_buf(m);
    int* meta = reinterpret_cast<int*>(cb + LY::cMeta);
    const int nm = sub_len(m);

    // ---- P0: gamma_t = w_0 o .. o w_t down each column; V split in token pairs
    if (pt < kD) {
      const int j = pt;
      float wv[kL];
#pragma unroll
      for (int t = 0; t < kL; ++t) wv[t] = raw_at(rw + t * kD + j);  // all 16 rows: no dependent guards
#pragma unroll
      for (int t = 0; t < kL; ++t) wv[t] = t < nm ? wv[t] : 1.f;
      float gm = 1.f;
#pragma unroll
      for (int t = 0; t < kL; ++t) {
        gm *= wv[t];
        G[t * kD + j] = gm;
      }
      if (pt == 0) {
        meta[0] = 0;
        meta[1] = nm;
      }
    } else {
      for (int e = pt - kD; e < (kL / 2) * kR; e += kNP - kD) {
        const int tp = e >> 5, i = e & 31;
        const float v0 = 2 * tp < nm ? raw_at(rv + 2 * tp * kR + i) : 0.f;
        const float v1 = 2 * tp + 1 < nm ? raw_at(rv + (2 * tp + 1) * kR + i) : 0.f;
        VP[tp * kSV2 + i] = make_float2(v0, v1);
      }
    }
    bar_prep();

    // ---- P1: decayed vectors split for the tensor cores, by 2 x 2 blocks (tokens 2tp, 2tp+1; columns
    // 2jp, 2jp+1): column pairs for A^, R^, K~, B~ and token pairs for K-, B-; the decay guard
    {
      uint4* AH = reinterpret_cast<uint4*>(cb + LY::cAH);
      uint4* RH = reinterpret_cast<uint4*>(cb + LY::cRH);
      uint4* BB = reinterpret_cast<uint4*>(cb + LY::cBB);
      float* GL = reinterpret_cast<float*>(cb + LY::cGL);
      for (int e = pt; e < (kL / 2) * (kD / 2); e += kNP) {
        const int tp = e >> 5, jp = e & 31, j = 2 * jp;
        const int t0 = 2 * tp, t1 = t0 + 1;
        const float2 gprev = t0 > 0 ? *reinterpret_cast<const float2*>(G + (t0 - 1) * kD + j) : make_float2(1.f, 1.f);
        const float2 g0 = *reinterpret_cast<const float2*>(G + t0 * kD + j);
        const float2 g1 = *reinterpret_cast<const float2*>(G + t1 * kD + j);
        const float2 i0 = make_float2(__fdividef(1.f, g0.x), __fdividef(1.f, g0.y));
        const float2 i1 = make_float2(__fdividef(1.f, g1.x), __fdividef(1.f, g1.y));
        const float2 gl = *reinterpret_cast<const float2*>(G + (kL - 1) * kD + j);
        const float2 z = make_float2(0.f, 0.f);
        const bool v0 = t0 < nm, v1 = t1 < nm;
        // rows past the sub-chunk hold stale bits: load unconditionally, select zeros
        float2 a0 = raw2(ra + t0 * kD + j), a1 = raw2(ra + t1 * kD + j);
        float2 b0 = raw2(rbv + t0 * kD + j), b1 = raw2(rbv + t1 * kD + j);
        float2 k0 = raw2(rk + t0 * kD + j), k1 = raw2(rk + t1 * kD + j);
        float2 r0 = raw2(rr + t0 * kD + j), r1 = raw2(rr + t1 * kD + j);
        if (!v0) a0 = b0 = k0 = r0 = z;
        if (!v1) a1 = b1 = k1 = r1 = z;
        AH[t0 * kSP + jp] = split_pair(a0.x * gprev.x, a0.y * gprev.y);
        AH[t1 * kSP + jp] = split_pair(a1.x * g0.x, a1.y * g0.y);
        RH[t0 * kSP + jp] = split_pair(r0.x * g0.x, r0.y * g0.y);
        RH[t1 * kSP + jp] = split_pair(r1.x * g1.x, r1.y * g1.y);
        *reinterpret_cast<float2*>(KT + t0 * kSF + j) = make_float2(k0.x * i0.x, k0.y * i0.y);
        *reinterpret_cast<float2*>(KT + t1 * kSF + j) = make_float2(k1.x * i1.x, k1.y * i1.y);
        *reinterpret_cast<float2*>(BT + t0 * kSF + j) = make_float2(b0.x * i0.x, b0.y * i0.y);
        *reinterpret_cast<float2*>(BT + t1 * kSF + j) = make_float2(b1.x * i1.x, b1.y * i1.y);
        // gamma_L / gamma_t
        const float f00 = gl.x * i0.x, f01 = gl.y * i0.y, f10 = gl.x * i1.x, f11 = gl.y * i1.y;
        KB[tp * kSJ2 + j] = make_float2(k0.x * f00, k1.x * f10);
        KB[tp * kSJ2 + j + 1] = make_float2(k0.y * f01, k1.y * f11);
        BB[tp * kSJ + j] = split_pair(b0.x * f00, b1.x * f10);
        BB[tp * kSJ + j + 1] = split_pair(b0.y * f01, b1.y * f11);
      }
      if (pt < kD) {
        const float gl = G[(kL - 1) * kD + pt];
        GL[pt] = gl;
        if (!(gl >= kMinDecay)) meta[0] = 1;
      }
    }
    bar_prep();

    if (meta[0]) {
      // token-by-token sub-chunk: the chain reads fp32 inputs instead of the matrices
      float* FW = reinterpret_cast<float*>(cb + LY::cFW);
      for (int e = pt; e < 5 * kL * kD; e += kNP) {
        const int s5 = e / (kL * kD), t = (e - s5 * kL * kD) >> 6;
        FW[e] = t < nm ? raw_at(raw + e) : (s5 == 0 ? 1.f : 0.f);
      }
      for (int e = pt; e < kL * kR; e += kNP) FW[5 * kL * kD + e] = (e >> 5) < nm ? raw_at(rv + e) : 0.f;
      return;
    }

    // ---- P2: the coupling matrices (16 x 16, K = 64) and U = V^T K- (32 x 64, K = 16) on tensor cores.
    // Preparing warp 0 forms M_ab and goes straight on to (I - M_ab)^-1 (the longest dependent
    // path); warps 1-9 form M_ak, M_rb, M_rk and U, then C_AK = V^T M_ak^T and C_Y = V^T M_rk^T.
    {
      const uint4* AH = reinterpret_cast<const uint4*>(cb + LY::cAH);
      const uint4* RH = reinterpret_cast<const uint4*>(cb + LY::cRH);
      uint4* MRB = reinterpret_cast<uint4*>(cb + LY::cMRB);
      float* U = reinterpret_cast<float*>(cb + LY::cU);
      // one coupling-matrix tile: job = 4 x (R^ rows) + 2 x (K~ columns) + nt; k-steps in four
      // accumulators; A^-rows strictly lower (s < t), R^-rows lower with the diagonal
      auto mjob = [&](int job) {
        const int xr = job >> 2, yk = (job >> 1) & 1, nt = job & 1;
        const uint4* X = xr ? RH : AH;
        const float* Yv = yk ? KT : BT;
        float acc[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma3(acc[kk & 3], frag_a(X[g * kSP + kk * 4 + q], X[(g + 8) * kSP + kk * 4 + q]),
               frag_b2(*reinterpret_cast<const float2*>(Yv + (nt * 8 + g) * kSF + kk * 8 + 2 * q)));
        float sum[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sum[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
        const int s0 = nt * 8 + 2 * q;
        const int lim0 = xr ? g : g - 1, lim8 = xr ? g + 8 : g + 7;
        const float m00 = s0 <= lim0 ? sum[0] : 0.f;
        const float m01 = s0 + 1 <= lim0 ? sum[1] : 0.f;
        const float m80 = s0 <= lim8 ? sum[2] : 0.f;
        const float m81 = s0 + 1 <= lim8 ? sum[3] : 0.f;
        if (!xr && !yk) {  // M_ab: fp32 for the inverse
          *reinterpret_cast<float2*>(MAB + g * 16 + s0) = make_float2(m00, m01);
          *reinterpret_cast<float2*>(MAB + (g + 8) * 16 + s0) = make_float2(m80, m81);
        } else {           // split pairs [t][s / 2], the B operand of products contracting over s
          uint4* M = xr ? (yk ? MRK : MRB) : MAK;
          M[g * kSM + nt * 4 + q] = split_pair(m00, m01);
          M[(g + 8) * kSM + nt * 4 + q] = split_pair(m80, m81);
        }
      };
      // the eight U tiles of rows um*16 .. um*16+15, one accumulator each
      auto ujob8 = [&](int um) {
        float acc[8][4] = {};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const FragA av = frag_a2(VP[(kk * 4 + q) * kSV2 + um * 16 + g], VP[(kk * 4 + q) * kSV2 + um * 16 + g + 8]);
#pragma unroll
          for (int u = 0; u < 8; ++u) mma3(acc[u], av, frag_b2(KB[(kk * 4 + q) * kSJ2 + u * 8 + g]));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          *reinterpret_cast<float2*>(U + (um * 16 + g) * kSU + u * 8 + 2 * q) = make_float2(acc[u][0], acc[u][1]);
          *reinterpret_cast<float2*>(U + (um * 16 + g + 8) * kSU + u * 8 + 2 * q) = make_float2(acc[u][2], acc[u][3]);
        }
      };

      if (pw == 0) {
        mjob(0);
        bar_pair_sync();  // warp 1 has stored the other M_ab tile
        // ---- (I - M_ab)^-1, unit lower: column c solves (I - M_ab) x = e_c by forward substitution,
        // x_t = [t == c] + sum_{u < t} M_ab[t][u] x_u, in lane c's registers (lanes 16-31 repeat
        // columns 0-15); rows of M_ab are broadcast loads.  Stored fp32; the chain splits it.
        {
          const int c = lane & 15;
          float x[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            float acc = t == c ? 1.f : 0.f;
#pragma unroll
            for (int u = 0; u < t; ++u) acc = fmaf(MAB[t * 16 + u], x[u], acc);
            x[t] = acc;
          }
          float* TI = reinterpret_cast<float*>(cb + LY::cTI);
          if (lane < 16) {
#pragma unroll
            for (int t = 0; t < 16; ++t) TI[t * kSC + c] = x[t];
          }
        }
      } else {
        if (pw == 1) {
          mjob(1);
          bar_pair_arrive();
        } else if (pw <= 7) {
          mjob(pw);  // jobs 2-7: M_ak, M_rb, M_rk
        } else {
          ujob8(pw - 8);
        }
        bar_rest();
        if (pw <= 8) {  // C_AK (jb < 4) and C_Y tiles: (which, um, nt) = (jb >> 2, (jb >> 1) & 1, jb & 1)
          float* CAK = reinterpret_cast<float*>(cb + LY::cCAK);
          float* CY = reinterpret_cast<float*>(cb + LY::cCY);
          const int jb = pw - 1;
          const int which = jb >> 2, um = (jb >> 1) & 1, nt = jb & 1;
          const uint4* M = which ? MRK : MAK;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma3(acc, frag_a2(VP[(kk * 4 + q) * kSV2 + um * 16 + g], VP[(kk * 4 + q) * kSV2 + um * 16 + g + 8]),
                 frag_b(M[(nt * 8 + g) * kSM + kk * 4 + q]));
          float* C = which ? CY : CAK;
          *reinterpret_cast<float2*>(C + (um * 16 + g) * kSC + nt * 8 + 2 * q) = make_float2(acc[0], acc[1]);
          *reinterpret_cast<float2*>(C + (um * 16 + g + 8) * kSC + nt * 8 + 2 * q) = make_float2(acc[2], acc[3]);
        }
      }
    }
  };

  if (nsub > 0) {
    issue(0);
    if (nsub > 1) issue(1);
    if (nsub > 1) cp_async_wait<1>(); else cp_async_wait<0>();
    bar_prep();
    prepare(0);
  }
  __syncthreads();  // sub-chunk 0 prepared

  for (int n = 0; n < nsub; ++n) {
    if (n + 1 < nsub) {
      // raw buffer n & 1 held sub-chunk n, prepared in the previous period: refill with n + 2
      if (n + 2 < nsub) {
        issue(n + 2);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      bar_prep();  // sub-chunk n + 1's inputs are visible to every preparing thread
      prepare(n + 1);
    }
    __syncthreads();  // end of period n
  }
}

template <typename Tin, bool GRAD>
cudaError_t launch_fwdc_t(int B, int T, int H, int chunk, int nchunks, const FwdcPtrs& P, cudaStream_t stream) {
  using TV = typename std::conditional<GRAD, float, Tin>::type;
  using LY = Lay<Tin, TV>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  auto kern = fwdc_kernel<Tin, GRAD>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::kBytes);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)B * H * 2;
  kern<<<grid, kNT, LY::kBytes, stream>>>(T, H, chunk, nchunks, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_chunked(const FwdArgs& p, cudaStream_t stream) {
  const FwdcPtrs P{p.in.r, p.in.w, p.in.k, p.in.v, p.in.a, p.in.b, p.h0, p.y, p.h_ckpt, p.hT, p.sa};
  return p.bf16 ? launch_fwdc_t<__nv_bfloat16, false>(p.B, p.T, p.H, p.chunk, p.nchunks, P, stream)
                : launch_fwdc_t<float, false>(p.B, p.T, p.H, p.chunk, p.nchunks, P, stream);
}

cudaError_t launch_gwalk_chunked(const BwdArgs& p, float* dsa_ws, float* xck_ws, cudaStream_t stream) {
  const FwdcPtrs P{p.in.r, p.in.w, p.in.k, p.dy, p.in.a, p.in.b, p.dhT, p.dv, xck_ws, p.dh0, dsa_ws};
  return p.bf16 ? launch_fwdc_t<__nv_bfloat16, true>(p.B, p.T, p.H, p.chunk, p.nchunks, P, stream)
                : launch_fwdc_t<float, true>(p.B, p.T, p.H, p.chunk, p.nchunks, P, stream);
}

WKV7_DEBUG_READER(debug_word_fwdc)

}  // namespace wkv7
