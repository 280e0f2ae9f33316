// WKV7 forward on sm_103a as a chain of 32-token transition products, and the backward's
// state-gradient walk on the same kernel.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel architecture",
// Forward listing), per head, state S (rows i = value, columns j = key):
//     sa_t = S_{t-1} a_t;   S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T;   y_t = S_t r_t,
// with S written out after every chunk of 32 tokens.
//
// Transition form (exact in real arithmetic).  Over a chunk of 32 tokens from state S0, with
// gamma_t = w_0 o .. o w_t per column and
//     A^_t = a_t o gamma_{t-1},  R^_t = r_t o gamma_t,  K~_t = k_t / gamma_t,  B~_t = b_t / gamma_t,
//     K-_t = k_t o gamma_31 / gamma_t,  B-_t = b_t o gamma_31 / gamma_t,
//     M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T),
//     T = (I - M_ab)^-1,  B' = T^T B-,  C = M_rb T,
// the state after the chunk and the chunk's outputs are
//     S' = S0 diag(gamma_31) + S0 M' + V^T K',   M' = A^^T B',  K' = K- + M_ak^T B'
//     Y  = R' S0^T + P V,                        R' = R^ + C A^,  P = M_rk + C M_ak
// (unrolling the recurrence: sa_t and y_t are dots of S0 with decayed a_t / r_t plus the chunk's own
// rank-one terms, coupled through sa by the unit lower-triangular system (I - M_ab); eliminating sa
// leaves one 64 x 64 product per chunk on the serial path).  Everything but S0 M' is independent
// of the state and is prepared one chunk ahead.
//
// Precision: tensor-core products of fp32 operands as three bf16 products (hi hi + hi lo + lo hi,
// see wkv7_mma.cuh), ~2^-17 relative each, fp32 accumulation; the diagonal part S0 diag(gamma_31)
// in fp32.  1/gamma grows like prod(1/w); a chunk whose gamma_31 falls below 1e-20 in some column
// (or is not finite) is advanced token by token instead (exact fp32), so any w in [0, 1] works.
//
// Mapping: one CTA per (head, 32-row block), 12 warps, one CTA per SM.
//   warps 0-1  (chain): rows 16m..16m+15 of the CTA's slice of S as mma accumulators; per chunk they
//              store S as an operand for the output warps, form S M', add S o gamma_31 and V^T K',
//              and write the checkpoint;
//   warps 2-3  (output): V^T K' for the chain warps, then Y^T = S0 R'^T + V^T P^T, and y;
//   warps 4-11 (prep): the next chunk's decays, operands, coupling products, T (block forward
//              substitution on CUDA cores) and M', K', R', P, into the other of two buffers.
// One CTA barrier per chunk; the chain and output warps hand S and V^T K' over by named barriers.
//
// The same kernel runs the backward's state-gradient walk (GRAD): read from the last token down,
// that recurrence has the forward's form with w' = w_{t+1}, a' = b_{t+1}, b' = a_{t+1}, v' = dy_t,
// k' = r_t, r' = k_t over steps s = 0..T (token t = T-1-s; zeros and w' = 1 outside the sequence),
// started from dhT: y' is dv_t, the state after step s is the gradient X_t (including dy_t r_t^T) and
// after step T it is dh0.  Chunks of one step, then ((T-1) % 32) + 1 steps, then 32 put every
// checkpoint boundary at a chunk end.
#include <type_traits>

#include "wkv7_device.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace {

using namespace mma;

constexpr int kL = 32;       // tokens per chunk
constexpr int kR = 32;       // state rows per CTA
constexpr int kNT = 384;     // threads
constexpr int kNP = 256;     // prep threads (warps 4-11)
constexpr int kFirstPrep = 128;
constexpr float kMinGamma = 1e-20f;

// named barriers
constexpr int kBarPrep = 1;   // prep warps
constexpr int kBarChain = 2;  // chain warps
constexpr int kBarS = 3;      // chain warps arrive (S stored), output warps wait
constexpr int kBarN = 4;      // output warps arrive (V^T K' stored), chain warps wait
constexpr int kBarOut = 5;    // output warps

template <int ID, int N>
__device__ __forceinline__ void bsync() { asm volatile("bar.sync %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }
template <int ID, int N>
__device__ __forceinline__ void barrive() { asm volatile("bar.arrive %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }

// pair-tile array sizes in words (hi + lo) of an R x C matrix
__host__ __device__ constexpr int pt_words(int r, int c) { return r * c; }

template <typename Tin, typename TV>
struct Lay {
  // ---- prep scratch (byte offsets)
  static constexpr size_t oG = 0;                                   // float [32][64] gamma; then M_ab^T fp32
  static constexpr int kSMab = 36;                                  // row stride of M_ab^T [32][36]
  static constexpr size_t oU1 = oG + 32 * 64 * 4;                    // B~, K~ (PT 32x64 each); then T^T, B'^T, C
  static constexpr size_t oBt = oU1;
  static constexpr size_t oKt = oU1 + pt_words(32, 64) * 4;
  static constexpr size_t oTT = oU1;                                 // PT 32x32 (T^T)
  static constexpr size_t oBpT = oU1 + pt_words(32, 32) * 4;         // PT 64x32 (B'^T)
  static constexpr size_t oC = oBpT + pt_words(64, 32) * 4;          // PT 32x32 (C)
  static constexpr size_t oRh = oU1 + 2 * pt_words(32, 64) * 4;      // PT 32x64 (R^)
  static constexpr size_t oU2 = oRh + pt_words(32, 64) * 4;          // A^ (PT 32x64); then TI, E
  static constexpr size_t oAh = oU2;
  static constexpr int kSTI = 36;
  static constexpr size_t oTI = oU2;                                 // float [32][36]
  static constexpr size_t oE = oU2 + 32 * kSTI * 4;                  // float [16][16]
  static constexpr size_t oAhT = oU2 + pt_words(32, 64) * 4;         // PT 64x32 (A^^T)
  static constexpr size_t oBmT = oAhT + pt_words(64, 32) * 4;        // PT 64x32 (B-^T)
  static constexpr size_t oKmT = oBmT + pt_words(64, 32) * 4;        // PT 64x32 (K-^T)
  static constexpr size_t oMakT = oKmT + pt_words(64, 32) * 4;       // PT 32x32 (M_ak^T)
  static constexpr size_t oMrb = oMakT + pt_words(32, 32) * 4;       // PT 32x32 (M_rb)
  static constexpr size_t oMrk = oMrb + pt_words(32, 32) * 4;        // PT 32x32 (M_rk)
  static constexpr size_t kPrepEnd = oMrk + pt_words(32, 32) * 4;
  static_assert(oE + 16 * 16 * 4 <= oAhT, "TI and E fit in A^'s space");
  static_assert(oC + pt_words(32, 32) * 4 <= oRh, "T^T, B'^T, C fit in B~ and K~'s space");
  static_assert(32 * kSMab * 4 <= 32 * 64 * 4, "M_ab^T fits in gamma's space");
  // ---- chain buffers (x2): what one chunk's chain and output steps read
  static constexpr size_t cMT = 0;                                   // PT 64x64 (M'^T)
  static constexpr size_t cKpT = cMT + pt_words(64, 64) * 4;         // PT 64x32 (K'^T)
  static constexpr size_t cRp = cKpT + pt_words(64, 32) * 4;         // PT 32x64 (R')
  static constexpr size_t cP = cRp + pt_words(32, 64) * 4;           // PT 32x32 (P)
  static constexpr size_t cGL = cP + pt_words(32, 32) * 4;           // float [64] gamma_31
  static constexpr size_t cMeta = cGL + 64 * 4;                      // int [4]: token-by-token flag
  static constexpr size_t kChain = cMeta + 16;
  static constexpr size_t oChain = kPrepEnd;
  // ---- raw inputs of the chunk being prepared: w, k, a, b, r [32][64]
  static constexpr size_t oRaw = oChain + 2 * kChain;
  static constexpr size_t kRaw = 5 * kL * kD * sizeof(Tin);
  // ---- v of this CTA's rows, two chunks: [32 tokens][32 rows]
  static constexpr size_t oV = oRaw + kRaw;
  static constexpr size_t kV = kL * kR * sizeof(TV);
  // ---- chain / output exchange
  static constexpr size_t oS = oV + 2 * kV;                          // PT 32x64 (S of this CTA's rows)
  static constexpr size_t oVT = oS + pt_words(32, 64) * 4;           // PT 32x32 (V^T: rows i, columns t)
  static constexpr size_t oN = oVT + pt_words(32, 32) * 4;           // float [2 mt][8 nj][32 lanes][4]
  static constexpr int kSY = 36;
  static constexpr size_t oY = oN + 32 * 64 * 4;                     // float [32 t][36]
  static constexpr size_t oFS = oN;                                  // token-by-token path: float [32][68] (N and Y)
  static constexpr int kSFS = 68;
  static constexpr size_t kBytes = oY + kL * kSY * 4;
  static_assert(oFS + 32 * kSFS * 4 <= kBytes, "token-by-token state fits over N and Y");
};

// Pointers of one call.  Forward: the inputs, s0 = h0, y, ck = h_ckpt, sT = hT.  Gradient walk
// (GRAD): the inputs with v = dy (fp32), s0 = dhT, y = dv, ck = X at the chunk ends, sT = dh0.
struct ChainPtrs {
  const void *r, *w, *k, *v, *a, *b;
  const float* s0;
  float *y, *ck, *sT;
};

template <typename Tin, bool GRAD>
__global__ void __launch_bounds__(kNT, 1)
chain_kernel(int T, int H, int nchunks, ChainPtrs P) {
  using TV = typename std::conditional<GRAD, float, Tin>::type;
  using LY = Lay<Tin, TV>;
  constexpr bool kVExact = sizeof(TV) == 2;  // bf16 v: exact in the tensor-core operand
  const Tin* __restrict__ r = static_cast<const Tin*>(P.r);
  const Tin* __restrict__ w = static_cast<const Tin*>(P.w);
  const Tin* __restrict__ k = static_cast<const Tin*>(P.k);
  const TV* __restrict__ v = static_cast<const TV*>(P.v);
  const Tin* __restrict__ a = static_cast<const Tin*>(P.a);
  const Tin* __restrict__ b = static_cast<const Tin*>(P.b);
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

  // chunk schedule over the steps.  Forward: steps = tokens, 32 per chunk.  Walk: T + 1 steps, a
  // first chunk of one step and a second of ((T - 1) % 32) + 1 put every checkpoint on a chunk end.
  const int len2 = GRAD && T > 0 ? (T - 1) % kL + 1 : 0;
  const int nsub = GRAD ? (T > 0 ? 2 + (T - len2) / kL : 0) : (T + kL - 1) / kL;
  auto sub_start = [&](int m) { return GRAD ? (m == 0 ? 0 : (m == 1 ? 1 : 1 + len2 + kL * (m - 2))) : m * kL; };
  auto sub_len = [&](int m) { return GRAD ? (m == 0 ? 1 : (m == 1 ? len2 : kL)) : min(kL, T - m * kL); };
  // token of slot (w, k, a, b, r) at step st: forward the step itself; walk w, a, b at T - st and
  // k, r at T - 1 - st; the walk's slots w, k, a, b, r take w, r, b, a, k
  auto slot_token = [&](int s5, int st) {
    return !GRAD ? st : ((s5 == 0 || s5 == 2 || s5 == 3) ? T - st : T - 1 - st);
  };
  auto v_token = [&](int st) { return GRAD ? T - 1 - st : st; };

  unsigned char* const chain0 = sm + LY::oChain;
  auto chain_buf = [&](int m) { return chain0 + (size_t)(m & 1) * LY::kChain; };
  Tin* const raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  auto vbuf = [&](int m) { return reinterpret_cast<TV*>(sm + LY::oV + (size_t)(m & 1) * LY::kV); };

  if (warp < 2) {
    // =============================================================== chain warps
    const int mt = warp;
    const int row = rb * kR + mt * 16 + g;  // rows row, row + 8 of the head
    float S[8][4];
#pragma unroll
    for (int nj = 0; nj < 8; ++nj) {
      if (P.s0 != nullptr) {
        const float2 s0 = __ldg(reinterpret_cast<const float2*>(P.s0 + sbase + (size_t)row * kD + nj * 8 + 2 * q));
        const float2 s8 = __ldg(reinterpret_cast<const float2*>(P.s0 + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q));
        S[nj][0] = s0.x; S[nj][1] = s0.y; S[nj][2] = s8.x; S[nj][3] = s8.y;
      } else {
        S[nj][0] = S[nj][1] = S[nj][2] = S[nj][3] = 0.f;
      }
    }
    uint32_t* const pS = reinterpret_cast<uint32_t*>(sm + LY::oS);
    const float* const nb = reinterpret_cast<const float*>(sm + LY::oN);
    __syncthreads();  // chunk 0 prepared

    for (int n = 0; n < nsub; ++n) {
      const unsigned char* cb = chain_buf(n);
      const int slow = reinterpret_cast<const int*>(cb + LY::cMeta)[0] | reinterpret_cast<const int*>(cb + LY::cMeta)[1];
      const int tau0 = sub_start(n);
      const int nm = sub_len(n);
      if (!slow) {
        // S (the state before the chunk) as an operand for the output warps
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) store_acc(pS, pt_words(32, 64) / 2, 4, mt, nj, lane, S[nj]);
        barrive<kBarS, 128>();
        // S M'
        const uint32_t* pMT = reinterpret_cast<const uint32_t*>(cb + LY::cMT);
        float acc[8][4];
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) acc[nj][0] = acc[nj][1] = acc[nj][2] = acc[nj][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const FragA fa = frag_from_acc(S[2 * kk], S[2 * kk + 1]);
#pragma unroll
          for (int nj = 0; nj < 8; ++nj) mma3(acc[nj], fa, load_b(pMT, pt_words(64, 64) / 2, 4, nj, kk, lane));
        }
        bsync<kBarN, 128>();  // V^T K' is in shared memory
        const float* GL = reinterpret_cast<const float*>(cb + LY::cGL);
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          const float4 nv = *reinterpret_cast<const float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4);
          const float2 gl = *reinterpret_cast<const float2*>(GL + nj * 8 + 2 * q);
          S[nj][0] = fmaf(S[nj][0], gl.x, acc[nj][0] + nv.x);
          S[nj][1] = fmaf(S[nj][1], gl.y, acc[nj][1] + nv.y);
          S[nj][2] = fmaf(S[nj][2], gl.x, acc[nj][2] + nv.z);
          S[nj][3] = fmaf(S[nj][3], gl.y, acc[nj][3] + nv.w);
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
        bsync<kBarChain, 64>();
        const int ti = tid >> 1, half = tid & 1, c0 = 32 * half;
        float Sr[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) Sr[c] = FS[ti * LY::kSFS + c0 + c];
        const Tin* srcs[5] = {w, k, a, b, r};
        if (GRAD) {
          srcs[1] = r; srcs[2] = b; srcs[3] = a; srcs[4] = k;
        }
        // 8 columns of slot s5 at step st (w = 1 and zeros outside the sequence)
        auto cols8 = [&](int s5, int st, int c, float (&o)[8]) {
          const int tok = slot_token(s5, st);
          if (tok >= 0 && tok < T) {
            load8(srcs[s5] + base + (size_t)tok * tstride + c0 + c, o);
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) o[u] = s5 == 0 ? 1.f : 0.f;
          }
        };
        for (int t = 0; t < nm; ++t) {
          const int st = tau0 + t;
          const int vt = v_token(st);
          const float vi = (vt >= 0 && vt < T) ? to_f32(v[base + (size_t)vt * tstride + rb * kR + ti]) : 0.f;
          float s = 0.f;
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            float av[8];
            cols8(2, st, c, av);
#pragma unroll
            for (int u = 0; u < 8; ++u) s = fmaf(Sr[c + u], av[u], s);
          }
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          float yy = 0.f;
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            float wv[8], kv[8], bv[8], rv[8];
            cols8(0, st, c, wv);
            cols8(1, st, c, kv);
            cols8(3, st, c, bv);
            cols8(4, st, c, rv);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              Sr[c + u] = fmaf(Sr[c + u], wv[u], fmaf(vi, kv[u], s * bv[u]));
              yy = fmaf(Sr[c + u], rv[u], yy);
            }
          }
          yy += __shfl_xor_sync(0xffffffffu, yy, 1);
          if (half == 0) {
            if (!GRAD) {
              P.y[base + (size_t)st * tstride + rb * kR + ti] = yy;
            } else if (st <= T - 1) {
              P.y[base + (size_t)(T - 1 - st) * tstride + rb * kR + ti] = yy;
            }
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) FS[ti * LY::kSFS + c0 + c] = Sr[c];
        bsync<kBarChain, 64>();
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          const float2 s0 = *reinterpret_cast<const float2*>(FS + i0 * LY::kSFS + nj * 8 + 2 * q);
          const float2 s8 = *reinterpret_cast<const float2*>(FS + (i0 + 8) * LY::kSFS + nj * 8 + 2 * q);
          S[nj][0] = s0.x; S[nj][1] = s0.y; S[nj][2] = s8.x; S[nj][3] = s8.y;
        }
      }

      // the state after the chunk's last step when that is a checkpoint (forward: every chunk end;
      // walk: step T-1-t for a chunk end t, i.e. X_t)
      const int tlast = tau0 + nm - 1;
      const bool at_end = GRAD ? (tlast < T && (tlast == 0 || (T - tlast) % kL == 0)) : true;
      const int cidx = GRAD ? (T - 1 - tlast) / kL : n;
      if (P.ck != nullptr && at_end) {
        float* dst = P.ck + ((size_t)bh * nchunks + cidx) * kD * kD;
#pragma unroll
        for (int nj = 0; nj < 8; ++nj) {
          *reinterpret_cast<float2*>(dst + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
          *reinterpret_cast<float2*>(dst + (size_t)(row + 8) * kD + nj * 8 + 2 * q) = make_float2(S[nj][2], S[nj][3]);
        }
      }
      __syncthreads();  // end of period n
    }
    if (P.sT != nullptr) {
#pragma unroll
      for (int nj = 0; nj < 8; ++nj) {
        *reinterpret_cast<float2*>(P.sT + sbase + (size_t)row * kD + nj * 8 + 2 * q) = make_float2(S[nj][0], S[nj][1]);
        *reinterpret_cast<float2*>(P.sT + sbase + (size_t)(row + 8) * kD + nj * 8 + 2 * q) =
            make_float2(S[nj][2], S[nj][3]);
      }
    }
    return;
  }

  if (warp < 4) {
    // =============================================================== output warps
    const int mt = warp - 2;
    const int ot = tid - 64;  // 0 .. 63
    uint32_t* const pVT = reinterpret_cast<uint32_t*>(sm + LY::oVT);
    const uint32_t* const pS = reinterpret_cast<const uint32_t*>(sm + LY::oS);
    float* const nb = reinterpret_cast<float*>(sm + LY::oN);
    float* const ys = reinterpret_cast<float*>(sm + LY::oY);
    // v of this CTA's rows for chunk m into buffer m & 1 (rows past the chunk are not copied)
    auto issue_v = [&](int m) {
      constexpr int VPR = kR * (int)sizeof(TV) / 16;
      constexpr int EPV = 16 / (int)sizeof(TV);
      TV* dst = vbuf(m);
      const int t0 = sub_start(m), nm = sub_len(m);
      for (int e = ot; e < nm * VPR; e += 64) {
        const int t = e / VPR, pc = e % VPR;
        const int tok = v_token(t0 + t);
        if (tok >= 0 && tok < T)
          cp_async16(dst + t * kR + pc * EPV, v + base + (size_t)tok * tstride + rb * kR + pc * EPV);
        else
          *reinterpret_cast<uint4*>(dst + t * kR + pc * EPV) = make_uint4(0u, 0u, 0u, 0u);
      }
      cp_async_commit();
    };
    if (nsub > 0) issue_v(0);
    __syncthreads();  // chunk 0 prepared

    for (int n = 0; n < nsub; ++n) {
      const unsigned char* cb = chain_buf(n);
      const int slow = reinterpret_cast<const int*>(cb + LY::cMeta)[0] | reinterpret_cast<const int*>(cb + LY::cMeta)[1];
      const int tau0 = sub_start(n);
      const int nm = sub_len(n);
      if (n + 1 < nsub) {
        issue_v(n + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      bsync<kBarOut, 64>();  // v of chunk n has landed for both output warps
      if (!slow) {
        // V^T (rows i, columns t), steps past the chunk zero
        {
          const TV* vb = vbuf(n);
          for (int e = ot; e < 16 * kR; e += 64) {
            const int tp = e >> 5, i = e & 31;
            const int t0 = 2 * tp;
            const float x0 = t0 < nm ? to_f32(vb[t0 * kR + i]) : 0.f;
            const float x1 = t0 + 1 < nm ? to_f32(vb[(t0 + 1) * kR + i]) : 0.f;
            if (kVExact)
              pt_store_hi(pVT, i, t0, 2, x0, x1);
            else
              pt_store(pVT, pt_words(32, 32) / 2, i, t0, 2, x0, x1);
          }
        }
        bsync<kBarOut, 64>();
        // N = V^T K' (this warp's 16 rows, all 64 columns), for the chain warps
        {
          const uint32_t* pKpT = reinterpret_cast<const uint32_t*>(cb + LY::cKpT);
          float acc[8][4];
#pragma unroll
          for (int nj = 0; nj < 8; ++nj) acc[nj][0] = acc[nj][1] = acc[nj][2] = acc[nj][3] = 0.f;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const FragA fa = kVExact ? load_a_hi(pVT, 2, mt, kk, lane) : load_a(pVT, pt_words(32, 32) / 2, 2, mt, kk, lane);
#pragma unroll
            for (int nj = 0; nj < 8; ++nj) {
              const FragB fb = load_b(pKpT, pt_words(64, 32) / 2, 2, nj, kk, lane);
              if (kVExact) mma2(acc[nj], fa, fb); else mma3(acc[nj], fa, fb);
            }
          }
#pragma unroll
          for (int nj = 0; nj < 8; ++nj)
            *reinterpret_cast<float4*>(nb + ((mt * 8 + nj) * 32 + lane) * 4) =
                make_float4(acc[nj][0], acc[nj][1], acc[nj][2], acc[nj][3]);
        }
        barrive<kBarN, 128>();
        bsync<kBarS, 128>();  // S of the chunk's start is in shared memory
        // Y^T = S R'^T + V^T P^T: rows i of this warp, tokens t
        {
          const uint32_t* pRp = reinterpret_cast<const uint32_t*>(cb + LY::cRp);
          const uint32_t* pP = reinterpret_cast<const uint32_t*>(cb + LY::cP);
          float acc[4][4];
#pragma unroll
          for (int nj = 0; nj < 4; ++nj) acc[nj][0] = acc[nj][1] = acc[nj][2] = acc[nj][3] = 0.f;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const FragA fa = load_a(pS, pt_words(32, 64) / 2, 4, mt, kk, lane);
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) mma3(acc[nj], fa, load_b(pRp, pt_words(32, 64) / 2, 4, nj, kk, lane));
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const FragA fa = kVExact ? load_a_hi(pVT, 2, mt, kk, lane) : load_a(pVT, pt_words(32, 32) / 2, 2, mt, kk, lane);
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) {
              const FragB fb = load_b(pP, pt_words(32, 32) / 2, 2, nj, kk, lane);
              if (kVExact) mma2(acc[nj], fa, fb); else mma3(acc[nj], fa, fb);
            }
          }
          // stage as [t][i]
          const int i0 = mt * 16 + g;
#pragma unroll
          for (int nj = 0; nj < 4; ++nj) {
            const int t0 = nj * 8 + 2 * q;
            ys[t0 * LY::kSY + i0] = acc[nj][0];
            ys[(t0 + 1) * LY::kSY + i0] = acc[nj][1];
            ys[t0 * LY::kSY + i0 + 8] = acc[nj][2];
            ys[(t0 + 1) * LY::kSY + i0 + 8] = acc[nj][3];
          }
        }
        bsync<kBarOut, 64>();
        for (int e = ot; e < nm * (kR / 4); e += 64) {
          const int t = e >> 3, i = (e & 7) * 4;
          const float4 vy = *reinterpret_cast<const float4*>(ys + t * LY::kSY + i);
          const int st = tau0 + t;
          if (!GRAD) {
            *reinterpret_cast<float4*>(P.y + base + (size_t)st * tstride + rb * kR + i) = vy;
          } else if (st <= T - 1) {
            *reinterpret_cast<float4*>(P.y + base + (size_t)(T - 1 - st) * tstride + rb * kR + i) = vy;
          }
        }
      }
      __syncthreads();  // end of period n
    }
    return;
  }

  // ================================================================= prep warps
  const int pt = tid - kFirstPrep;  // 0 .. 255
  const int pw = pt >> 5;           // 0 .. 7
  float* const G = reinterpret_cast<float*>(sm + LY::oG);
  float* const MabT = reinterpret_cast<float*>(sm + LY::oG);
  uint32_t* const pBt = reinterpret_cast<uint32_t*>(sm + LY::oBt);
  uint32_t* const pKt = reinterpret_cast<uint32_t*>(sm + LY::oKt);
  uint32_t* const pRh = reinterpret_cast<uint32_t*>(sm + LY::oRh);
  uint32_t* const pAh = reinterpret_cast<uint32_t*>(sm + LY::oAh);
  uint32_t* const pAhT = reinterpret_cast<uint32_t*>(sm + LY::oAhT);
  uint32_t* const pBmT = reinterpret_cast<uint32_t*>(sm + LY::oBmT);
  uint32_t* const pKmT = reinterpret_cast<uint32_t*>(sm + LY::oKmT);
  uint32_t* const pMakT = reinterpret_cast<uint32_t*>(sm + LY::oMakT);
  uint32_t* const pMrb = reinterpret_cast<uint32_t*>(sm + LY::oMrb);
  uint32_t* const pMrk = reinterpret_cast<uint32_t*>(sm + LY::oMrk);
  float* const TI = reinterpret_cast<float*>(sm + LY::oTI);
  float* const E = reinterpret_cast<float*>(sm + LY::oE);
  uint32_t* const pTT = reinterpret_cast<uint32_t*>(sm + LY::oTT);
  uint32_t* const pBpT = reinterpret_cast<uint32_t*>(sm + LY::oBpT);
  uint32_t* const pC = reinterpret_cast<uint32_t*>(sm + LY::oC);
  constexpr int H3232 = pt_words(32, 32) / 2, H3264 = pt_words(32, 64) / 2, H6432 = pt_words(64, 32) / 2,
                H6464 = pt_words(64, 64) / 2;

  // cp.async copies of chunk m's w, k, a, b, r (rows past the chunk are not copied)
  auto issue_raw = [&](int m) {
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    const int t0 = sub_start(m), nm = sub_len(m);
    const Tin* srcs[5] = {w, k, a, b, r};
    if (GRAD) {
      srcs[1] = r; srcs[2] = b; srcs[3] = a; srcs[4] = k;
    }
#pragma unroll
    for (int s5 = 0; s5 < 5; ++s5)
      for (int e = pt; e < nm * CPR; e += kNP) {
        const int t = e / CPR, pc = e % CPR;
        const int tok = slot_token(s5, t0 + t);
        Tin* d = raw + (s5 * kL + t) * kD + pc * EPC;
        if (tok >= 0 && tok < T) {
          cp_async16(d, srcs[s5] + base + (size_t)tok * tstride + pc * EPC);
        } else {
          const uint32_t u = s5 != 0 ? 0u : (sizeof(Tin) == 2 ? 0x3f803f80u : 0x3f800000u);
          *reinterpret_cast<uint4*>(d) = make_uint4(u, u, u, u);
        }
      }
    cp_async_commit();
  };

  auto prepare = [&](int m) {  // also issues the copy of chunk m + 1 once chunk m's inputs are consumed
    unsigned char* cb = chain_buf(m);
    int* meta = reinterpret_cast<int*>(cb + LY::cMeta);
    float* GL = reinterpret_cast<float*>(cb + LY::cGL);
    const int nm = sub_len(m);
    const Tin* rw = raw;
    const Tin* rk = raw + kL * kD;
    const Tin* ra = raw + 2 * kL * kD;
    const Tin* rbv = raw + 3 * kL * kD;
    const Tin* rr = raw + 4 * kL * kD;

    // ---- S1a: gamma_t down each column; the token-by-token flag
    if (pt < kD) {
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
      if (lane == 0) meta[pw] = any != 0u;  // prep warps 0 and 1 hold the 64 columns
    }
    bsync<kBarPrep, kNP>();
    const bool slow = (meta[0] | meta[1]) != 0;
    if (!slow) {
      // ---- S1b: row pairs (t, j): A^, R^, K~, B~
      for (int e = pt; e < kL * (kD / 2); e += kNP) {
        const int t = e >> 5, j = 2 * (e & 31);
        const bool ok = t < nm;
        const float2 gt = *reinterpret_cast<const float2*>(G + t * kD + j);
        const float2 gp = t > 0 ? *reinterpret_cast<const float2*>(G + (t - 1) * kD + j) : make_float2(1.f, 1.f);
        const float ix = __frcp_rn(gt.x), iy = __frcp_rn(gt.y);
        const float a0 = ok ? to_f32(ra[t * kD + j]) : 0.f, a1 = ok ? to_f32(ra[t * kD + j + 1]) : 0.f;
        const float r0 = ok ? to_f32(rr[t * kD + j]) : 0.f, r1 = ok ? to_f32(rr[t * kD + j + 1]) : 0.f;
        const float k0 = ok ? to_f32(rk[t * kD + j]) : 0.f, k1 = ok ? to_f32(rk[t * kD + j + 1]) : 0.f;
        const float b0 = ok ? to_f32(rbv[t * kD + j]) : 0.f, b1 = ok ? to_f32(rbv[t * kD + j + 1]) : 0.f;
        pt_store(pAh, H3264, t, j, 4, a0 * gp.x, a1 * gp.y);
        pt_store(pRh, H3264, t, j, 4, r0 * gt.x, r1 * gt.y);
        pt_store(pKt, H3264, t, j, 4, k0 * ix, k1 * iy);
        pt_store(pBt, H3264, t, j, 4, b0 * ix, b1 * iy);
      }
      // ---- S1c: column pairs (t, t + 1; j): A^^T, B-^T, K-^T
      for (int e = pt; e < (kL / 2) * kD; e += kNP) {
        const int tp = e >> 6, j = e & 63;
        const int t0 = 2 * tp, t1 = t0 + 1;
        const float gl = G[(kL - 1) * kD + j];
        const float g0 = G[t0 * kD + j], g1 = G[t1 * kD + j];
        const float gp0 = t0 > 0 ? G[(t0 - 1) * kD + j] : 1.f;
        const bool ok0 = t0 < nm, ok1 = t1 < nm;
        const float a0 = ok0 ? to_f32(ra[t0 * kD + j]) : 0.f, a1 = ok1 ? to_f32(ra[t1 * kD + j]) : 0.f;
        const float b0 = ok0 ? to_f32(rbv[t0 * kD + j]) : 0.f, b1 = ok1 ? to_f32(rbv[t1 * kD + j]) : 0.f;
        const float k0 = ok0 ? to_f32(rk[t0 * kD + j]) : 0.f, k1 = ok1 ? to_f32(rk[t1 * kD + j]) : 0.f;
        const float f0 = gl * __frcp_rn(g0), f1 = gl * __frcp_rn(g1);
        pt_store(pAhT, H6432, j, t0, 2, a0 * gp0, a1 * g0);
        pt_store(pBmT, H6432, j, t0, 2, b0 * f0, b1 * f1);
        pt_store(pKmT, H6432, j, t0, 2, k0 * f0, k1 * f1);
      }
    }
    bsync<kBarPrep, kNP>();  // raw is free: the next chunk is copied in while this one is prepared
    if (m + 1 < nsub) issue_raw(m + 1);
    if (slow) return;

    // ---- S2: coupling products (m16 x n8 tiles, K = 64): M_ab^T = B~ A^^T and M_ak^T = K~ A^^T (rows t,
    // columns s, kept s > t), M_rb = R^ B~^T and M_rk = R^ K~^T (kept s <= t).  Tiles wholly outside
    // the kept triangle are stored as zeros (later products read them).
    for (int job = pw; job < 32; job += 8) {
      const int prod = job >> 3, mt = (job >> 2) & 1, nj = job & 3;
      const bool upper = prod < 2;
      const bool empty = upper ? (mt == 1 && nj < 2) : (mt == 0 && nj >= 2);
      const uint32_t* X = prod == 0 ? pBt : (prod == 1 ? pKt : pRh);
      const uint32_t* Y = prod <= 1 ? pAh : (prod == 2 ? pBt : pKt);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (!empty) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma3(acc, load_a(X, H3264, 4, mt, kk, lane), load_b(Y, H3264, 4, nj, kk, lane));
      }
      const int t0 = mt * 16 + g, s0 = nj * 8 + 2 * q;
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = t0 + ((e >> 1) << 3), s = s0 + (e & 1);
        const bool keep = upper ? (s > t) : (s <= t);
        c[e] = keep ? acc[e] : 0.f;
      }
      if (prod == 0) {
        *reinterpret_cast<float2*>(MabT + t0 * Lay<Tin, TV>::kSMab + s0) = make_float2(c[0], c[1]);
        *reinterpret_cast<float2*>(MabT + (t0 + 8) * Lay<Tin, TV>::kSMab + s0) = make_float2(c[2], c[3]);
      } else {
        store_acc(prod == 1 ? pMakT : (prod == 2 ? pMrb : pMrk), H3232, 2, mt, nj, lane, c);
      }
    }
    bsync<kBarPrep, kNP>();

    // ---- S3: T = (I - M_ab)^-1 (unit lower triangular) by blocks of 16: the diagonal blocks by forward
    // substitution, one column per lane (lanes 0-15: T11, lanes 16-31: T22); M_ab[t][u] = M_ab^T[u][t]
    constexpr int SM = Lay<Tin, TV>::kSMab;
    constexpr int ST = Lay<Tin, TV>::kSTI;
    if (pw == 0) {
      const int off = lane < 16 ? 0 : 16;
      const int c = lane & 15;
      float x[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        float acc = t == c ? 1.f : 0.f;
#pragma unroll
        for (int u = 0; u < t; ++u) acc = fmaf(MabT[(off + u) * SM + off + t], x[u], acc);
        x[t] = acc;
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) TI[(off + t) * ST + off + c] = x[t];
    }
    bsync<kBarPrep, kNP>();
    // E = A21 T11 (A21 = M_ab[16..31][0..15]), then T21 = T22 E
    {
      const int t = pt >> 4, s = pt & 15;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) acc = fmaf(MabT[u * SM + 16 + t], TI[u * ST + s], acc);
      E[t * 16 + s] = acc;
    }
    bsync<kBarPrep, kNP>();
    {
      const int t = pt >> 4, s = pt & 15;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) acc = fmaf(TI[(16 + t) * ST + 16 + u], E[u * 16 + s], acc);
      TI[(16 + t) * ST + s] = acc;
    }
    bsync<kBarPrep, kNP>();
    // T^T as pair tiles (rows s, columns t); T[t][s] = 0 for s > t
    for (int e = pt; e < 32 * 16; e += kNP) {
      const int s = e >> 4, t0 = 2 * (e & 15);
      const float x0 = s <= t0 ? TI[t0 * ST + s] : 0.f;
      const float x1 = s <= t0 + 1 ? TI[(t0 + 1) * ST + s] : 0.f;
      pt_store(pTT, H3232, s, t0, 2, x0, x1);
    }
    bsync<kBarPrep, kNP>();

    // ---- S4: B'^T = B-^T T (rows j, columns s, K = t) and C = M_rb T (rows t, columns s, K = u)
    for (int job = pw; job < 24; job += 8) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (job < 16) {
        const int mt = job >> 2, nj = job & 3;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if (kk == 1 || nj < 2)  // T[t < 16][s >= 16] = 0
            mma3(acc, load_a(pBmT, H6432, 2, mt, kk, lane), load_b(pTT, H3232, 2, nj, kk, lane));
        store_acc(pBpT, H6432, 2, mt, nj, lane, acc);
      } else {
        const int mt = (job - 16) >> 2, nj = (job - 16) & 3;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          if ((kk == 1 || nj < 2) && (mt == 1 || kk == 0))  // M_rb[t < 16][u >= 16] = 0
            mma3(acc, load_a(pMrb, H3232, 2, mt, kk, lane), load_b(pTT, H3232, 2, nj, kk, lane));
        store_acc(pC, H3232, 2, mt, nj, lane, acc);
      }
    }
    bsync<kBarPrep, kNP>();

    // ---- S5 (into the chain buffer): M'^T = B'^T A^ (rows j, columns j'), K'^T = K-^T + B'^T M_ak (rows j,
    // columns t), R' = R^ + C A^ (rows t, columns j), P = M_rk + C M_ak (rows t, columns s); K = 32 each
    {
      uint32_t* cMT = reinterpret_cast<uint32_t*>(cb + LY::cMT);
      uint32_t* cKpT = reinterpret_cast<uint32_t*>(cb + LY::cKpT);
      uint32_t* cRp = reinterpret_cast<uint32_t*>(cb + LY::cRp);
      uint32_t* cP = reinterpret_cast<uint32_t*>(cb + LY::cP);
      for (int job = pw; job < 72; job += 8) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (job < 32) {
          const int mt = job >> 3, nj = job & 7;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma3(acc, load_a(pBpT, H6432, 2, mt, kk, lane), load_b(pAhT, H6432, 2, nj, kk, lane));
          store_acc(cMT, H6464, 4, mt, nj, lane, acc);
        } else if (job < 48) {
          const int mt = (job - 32) >> 2, nj = (job - 32) & 3;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma3(acc, load_a(pBpT, H6432, 2, mt, kk, lane), load_b(pMakT, H3232, 2, nj, kk, lane));
          float add[4];
          load_acc_pos(pKmT, H6432, 2, mt, nj, lane, add);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += add[e];
          store_acc(cKpT, H6432, 2, mt, nj, lane, acc);
        } else if (job < 64) {
          const int mt = (job - 48) >> 3, nj = (job - 48) & 7;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma3(acc, load_a(pC, H3232, 2, mt, kk, lane), load_b(pAhT, H6432, 2, nj, kk, lane));
          float add[4];
          load_acc_pos(pRh, H3264, 4, mt, nj, lane, add);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += add[e];
          store_acc(cRp, H3264, 4, mt, nj, lane, acc);
        } else {
          const int mt = (job - 64) >> 2, nj = (job - 64) & 3;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma3(acc, load_a(pC, H3232, 2, mt, kk, lane), load_b(pMakT, H3232, 2, nj, kk, lane));
          float add[4];
          load_acc_pos(pMrk, H3232, 2, mt, nj, lane, add);
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += add[e];
          store_acc(cP, H3232, 2, mt, nj, lane, acc);
        }
      }
    }
  };

  if (nsub > 0) {
    issue_raw(0);
    cp_async_wait<0>();
    bsync<kBarPrep, kNP>();
    prepare(0);
  }
  __syncthreads();  // chunk 0 prepared

  for (int n = 0; n < nsub; ++n) {
    if (n + 1 < nsub) {
      cp_async_wait<0>();
      bsync<kBarPrep, kNP>();  // chunk n + 1's inputs are visible to every prep thread
      prepare(n + 1);
    }
    __syncthreads();  // end of period n
  }
}

template <typename Tin, bool GRAD>
cudaError_t launch_chain_t(int B, int T, int H, int nchunks, const ChainPtrs& P, cudaStream_t stream) {
  using TV = typename std::conditional<GRAD, float, Tin>::type;
  using LY = Lay<Tin, TV>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  auto kern = chain_kernel<Tin, GRAD>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::kBytes);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)B * H * 2;
  kern<<<grid, kNT, LY::kBytes, stream>>>(T, H, nchunks, P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_transition(const FwdArgs& p, cudaStream_t stream) {
  const ChainPtrs P{p.in.r, p.in.w, p.in.k, p.in.v, p.in.a, p.in.b, p.h0, p.y, p.h_ckpt, p.hT};
  return p.bf16 ? launch_chain_t<__nv_bfloat16, false>(p.B, p.T, p.H, p.nchunks, P, stream)
                : launch_chain_t<float, false>(p.B, p.T, p.H, p.nchunks, P, stream);
}

cudaError_t launch_gwalk_transition(const BwdArgs& p, float* xck_ws, cudaStream_t stream) {
  const ChainPtrs P{p.in.r, p.in.w, p.in.k, p.dy, p.in.a, p.in.b, p.dhT, p.dv, xck_ws, p.dh0};
  return p.bf16 ? launch_chain_t<__nv_bfloat16, true>(p.B, p.T, p.H, p.nchunks, P, stream)
                : launch_chain_t<float, true>(p.B, p.T, p.H, p.nchunks, P, stream);
}

}  // namespace wkv7
