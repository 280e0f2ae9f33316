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
//     M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T),
//     T = (I - M_ab)^-1,  B' = (T^T B~) diag(gamma_31),  C = M_rb T,
//     K' = K~ diag(gamma_31) + M_ak^T B',  P = M_rk + C M_ak,
// the state after the chunk and the chunk's outputs are, with P1 = S0 A^^T (32 tokens wide),
//     S' = S0 diag(gamma_31) + P1 B' + V^T K'
//     Y^T = S0 R^^T + P1 C^T + V^T P^T                         (columns t: y_t)
// (unrolling the recurrence: sa_t and y_t are dots of S0 with decayed a_t / r_t plus the chunk's own
// rank-one terms, coupled through sa by the unit lower-triangular system (I - M_ab); eliminating sa
// leaves two dependent products, S0 A^^T then P1 B', on the serial path per 32 tokens).  Everything
// but P1 and the products with S0 is independent of the state and is prepared one chunk ahead.
//
// Precision: tensor-core products of fp32 operands as three bf16 products (hi hi + hi lo + lo hi,
// wkv7_mma.cuh), ~2^-17 relative each, fp32 accumulation; S0 diag(gamma_31) in fp32.  1/gamma grows
// like prod(1/w); a chunk whose gamma_31 falls below 1e-20 in some column (or is not finite) is
// advanced token by token instead (exact fp32), so any w in [0, 1] works.
//
// Operands are stored once, row-major, as bf16 hi and lo arrays, and read with ldmatrix (.trans
// for the transposed uses).  Mapping: one CTA per (head, 32-row block), 12 warps, one CTA per SM.
//   warps 0-1  (chain): rows 16m..16m+15 of the CTA's slice of S as mma accumulators; per chunk
//              P1, S', Y (staged), the checkpoint;
//   warps 2-3  (v): the chunk's v slice as an operand and N = V^T K' for the chain warps, then y;
//   warps 4-11 (prep): the next chunk's decays, operands, coupling products, T (block forward
//              substitution on CUDA cores), B', C, K', P into the other of two buffers.
// One CTA barrier per chunk; the chain and v warps hand N and y over by named barriers.
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
constexpr int kLD64 = 72;    // row stride (bf16 elements) of 64-wide operands
constexpr int kLD32 = 40;    // of 32-wide operands
constexpr float kMinGamma = 1e-20f;

// named barriers
constexpr int kBarPrep = 1;   // prep warps
constexpr int kBarChain = 2;  // chain warps
constexpr int kBarN = 3;      // v warps arrive (V^T K' stored), chain warps wait
constexpr int kBarY = 4;      // chain warps arrive (y staged), v warps wait
constexpr int kBarV = 5;      // v warps

template <int ID, int N>
__device__ __forceinline__ void bsync() { asm volatile("bar.sync %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }
template <int ID, int N>
__device__ __forceinline__ void barrive() { asm volatile("bar.arrive %0, %1;\n" ::"n"(ID), "n"(N) : "memory"); }

__host__ __device__ constexpr int rmb(int rows, int ld) { return 2 * rows * ld * 2; }  // RM bytes, hi + lo

template <typename Tin, typename TV>
struct Lay {
  // ---- prep scratch
  static constexpr int oG = 0;                          // float [32][64] gamma
  static constexpr int oKt = oG + 32 * 64 * 4;          // RM 32x64: K~, B~
  static constexpr int oBt = oKt + rmb(32, kLD64);
  static constexpr int oMak = oBt + rmb(32, kLD64);     // RM 32x32: M_ak, M_rb, M_rk, T
  static constexpr int oMrb = oMak + rmb(32, kLD32);
  static constexpr int oMrk = oMrb + rmb(32, kLD32);
  static constexpr int oT = oMrk + rmb(32, kLD32);
  static constexpr int kSM = 36;
  static constexpr int oMab = oT + rmb(32, kLD32);      // float [32][36]: M_ab
  static constexpr int oTI = oMab + 32 * kSM * 4;       // float [32][36]: T
  static constexpr int oE = oTI + 32 * kSM * 4;         // float [16][16]
  static constexpr int kPrepEnd = oE + 16 * 16 * 4;
  // ---- chain buffers (x2): A^, R^, B', K' (RM 32x64), C, P (RM 32x32), gamma_31, flags
  static constexpr int cAh = 0;
  static constexpr int cRh = cAh + rmb(32, kLD64);
  static constexpr int cBp = cRh + rmb(32, kLD64);
  static constexpr int cKp = cBp + rmb(32, kLD64);
  static constexpr int cC = cKp + rmb(32, kLD64);
  static constexpr int cP = cC + rmb(32, kLD32);
  static constexpr int cGL = cP + rmb(32, kLD32);
  static constexpr int cMeta = cGL + 64 * 4;
  static constexpr int kChain = cMeta + 16;
  static constexpr int oChain = kPrepEnd;
  // ---- raw inputs of the chunk being prepared: w, k, a, b, r [32][64]
  static constexpr int oRaw = oChain + 2 * kChain;
  static constexpr int kRaw = 5 * kL * kD * (int)sizeof(Tin);
  // ---- v of this CTA's rows: raw [32 t][32 i] (x2), and as an operand V (RM 32 t x 32 i)
  static constexpr int oVraw = oRaw + kRaw;
  static constexpr int kVraw = kL * kR * (int)sizeof(TV);
  static constexpr int oVop = oVraw + 2 * kVraw;
  // ---- N (fp32, accumulator order [2 mt][8 nj][32 lanes][4]) and y staging [32 t][36]
  static constexpr int oN = oVop + rmb(32, kLD32);
  static constexpr int kSY = 36;
  static constexpr int oY = oN + 32 * 64 * 4;
  static constexpr int oFS = oN;                        // token-by-token path: float [32][68] over N and y
  static constexpr int kSFS = 68;
  static constexpr int kBytes = oY + kL * kSY * 4;
  static_assert(oFS + 32 * kSFS * 4 <= kBytes, "token-by-token state fits over N and y");
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
  auto chain_buf = [&](int m) { return chain0 + (m & 1) * LY::kChain; };
  auto bfp = [&](unsigned char* p, int off) { return reinterpret_cast<__nv_bfloat16*>(p + off); };
  auto cbuf_rm64 = [&](unsigned char* cb, int off) { return RM{bfp(cb, off), 32 * kLD64, kLD64}; };
  auto cbuf_rm32 = [&](unsigned char* cb, int off) { return RM{bfp(cb, off), 32 * kLD32, kLD32}; };
  Tin* const raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  auto vraw = [&](int m) { return reinterpret_cast<TV*>(sm + LY::oVraw + (m & 1) * LY::kVraw); };
  const RM Vop{bfp(sm, LY::oVop), 32 * kLD32, kLD32};
  float* const nb = reinterpret_cast<float*>(sm + LY::oN);
  float* const ys = reinterpret_cast<float*>(sm + LY::oY);
  auto slow_flag = [&](const unsigned char* cb) {
    const int* meta = reinterpret_cast<const int*>(cb + LY::cMeta);
    return (meta[0] | meta[1]) != 0;
  };

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
    __syncthreads();  // chunk 0 prepared

    for (int n = 0; n < nsub; ++n) {
      unsigned char* cb = chain_buf(n);
      const int tau0 = sub_start(n);
      const int nm = sub_len(n);
      if (!slow_flag(cb)) {
        const RM Ah = cbuf_rm64(cb, LY::cAh), Rh = cbuf_rm64(cb, LY::cRh), Bp = cbuf_rm64(cb, LY::cBp);
        const RM Cm = cbuf_rm32(cb, LY::cC), Pm = cbuf_rm32(cb, LY::cP);
        // A fragments of S (k = j), from the accumulators
        FragA fs[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) fs[kk] = frag_from_acc(S[2 * kk], S[2 * kk + 1]);
        // P1 = S A^^T (16 rows x 32 tokens)
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
        // P1 B' (16 rows x 64 columns)
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
        // Y^T = S R^^T + P1 C^T (+ V^T P^T once the v warps have stored V)
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
        bsync<kBarN, 128>();  // V (operand) and N = V^T K' are in shared memory
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
        // S <- S o gamma_31 + P1 B' + N
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
        // stage y as [t][i]
        const int i0 = mt * 16 + g;
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
          const int t0 = nj * 8 + 2 * q;
          ys[t0 * LY::kSY + i0] = yv[nj][0];
          ys[(t0 + 1) * LY::kSY + i0] = yv[nj][1];
          ys[t0 * LY::kSY + i0 + 8] = yv[nj][2];
          ys[(t0 + 1) * LY::kSY + i0 + 8] = yv[nj][3];
        }
        barrive<kBarY, 128>();
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
    // =============================================================== v warps
    const int mt = warp - 2;
    const int ot = tid - 64;  // 0 .. 63
    // v of this CTA's rows for chunk m into raw buffer m & 1 (steps outside the sequence zero)
    auto issue_v = [&](int m) {
      constexpr int VPR = kR * (int)sizeof(TV) / 16;
      constexpr int EPV = 16 / (int)sizeof(TV);
      TV* dst = vraw(m);
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
      unsigned char* cb = chain_buf(n);
      const int tau0 = sub_start(n);
      const int nm = sub_len(n);
      if (n + 1 < nsub) {
        issue_v(n + 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      bsync<kBarV, 64>();  // v of chunk n has landed for both v warps
      if (!slow_flag(cb)) {
        // V (rows t, columns i of this CTA) as an operand, steps past the chunk zero
        {
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
        bsync<kBarV, 64>();
        // N = V^T K' (this warp's 16 rows i, all 64 columns), for the chain warps
        {
          const RM Kp = cbuf_rm64(cb, LY::cKp);
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
        }
        barrive<kBarN, 128>();
        bsync<kBarY, 128>();  // y of the chunk is staged
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
  const RM Kt{bfp(sm, LY::oKt), 32 * kLD64, kLD64}, Bt{bfp(sm, LY::oBt), 32 * kLD64, kLD64};
  const RM Mak{bfp(sm, LY::oMak), 32 * kLD32, kLD32}, Mrb{bfp(sm, LY::oMrb), 32 * kLD32, kLD32};
  const RM Mrk{bfp(sm, LY::oMrk), 32 * kLD32, kLD32}, Tm{bfp(sm, LY::oT), 32 * kLD32, kLD32};
  float* const Mab = reinterpret_cast<float*>(sm + LY::oMab);
  float* const TI = reinterpret_cast<float*>(sm + LY::oTI);
  float* const E = reinterpret_cast<float*>(sm + LY::oE);
  constexpr int SM = LY::kSM;

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

  // everything the chain needs for chunk m, into chain buffer m & 1 (its raw inputs have landed);
  // issues the copy of chunk m + 1 once chunk m's inputs are consumed
  auto prepare = [&](int m) {
    unsigned char* cb = chain_buf(m);
    int* meta = reinterpret_cast<int*>(cb + LY::cMeta);
    float* GL = reinterpret_cast<float*>(cb + LY::cGL);
    const int nm = sub_len(m);
    const Tin* rw = raw;
    const Tin* rk = raw + kL * kD;
    const Tin* ra = raw + 2 * kL * kD;
    const Tin* rbv = raw + 3 * kL * kD;
    const Tin* rr = raw + 4 * kL * kD;
    const RM Ah = cbuf_rm64(cb, LY::cAh), Rh = cbuf_rm64(cb, LY::cRh), Bp = cbuf_rm64(cb, LY::cBp);
    const RM Kp = cbuf_rm64(cb, LY::cKp), Cm = cbuf_rm32(cb, LY::cC), Pm = cbuf_rm32(cb, LY::cP);

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
      // ---- S1b: one (token, 8 columns) block per thread: A^, R^ (chain buffer), K~, B~
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
    bsync<kBarPrep, kNP>();  // raw is free: the next chunk is copied in while this one is prepared
    if (m + 1 < nsub) issue_raw(m + 1);
    if (slow) return;

    // ---- S2: M_ab = tril(A^ B~^T, -1) (fp32), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T),
    // M_rk = tril(R^ K~^T): 16 jobs of (product, m-tile, pair of n-tiles), K = 64
    for (int job = pw; job < 16; job += 8) {
      const int prod = job >> 2, mt = (job >> 1) & 1, np = job & 1;
      const bool strict = prod < 2;
      float acc[2][4] = {};
      if (!(mt == 0 && np == 1)) {  // rows 0-15 x columns 16-31: above the diagonal
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
    bsync<kBarPrep, kNP>();

    // ---- S3: T = (I - M_ab)^-1 (unit lower triangular) by blocks of 16: the diagonal blocks by forward
    // substitution, one column per lane (lanes 0-15: T11, lanes 16-31: T22), then T21 = T22 A21 T11
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
    bsync<kBarPrep, kNP>();
    {
      const int t = pt >> 4, s = pt & 15;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) acc = fmaf(Mab[(16 + t) * SM + u], TI[u * SM + s], acc);
      E[t * 16 + s] = acc;
    }
    bsync<kBarPrep, kNP>();
    {
      const int t = pt >> 4, s = pt & 15;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) acc = fmaf(TI[(16 + t) * SM + 16 + u], E[u * 16 + s], acc);
      TI[(16 + t) * SM + s] = acc;
    }
    bsync<kBarPrep, kNP>();
    if (pt < 128) {  // T as an operand (rows t, columns u), zero above the diagonal: 8 columns per thread
      const int t = pt >> 2, u0 = (pt & 3) * 8;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = u0 + e <= t ? TI[t * SM + u0 + e] : 0.f;
      rm_store8(Tm, t, u0, x);
    }
    bsync<kBarPrep, kNP>();

    // ---- S4: B' = (T^T B~) diag(gamma_31) (rows s, columns j; K = t) and C = M_rb T (rows t, columns s;
    // K = u): 12 jobs of (product, m-tile, 2 n-tiles)
    for (int job = pw; job < 12; job += 8) {
      float acc[2][4] = {};
      if (job < 8) {
        const int mt = job >> 2, nq = job & 3;  // B' n-tiles 2nq, 2nq + 1
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (mt == 1 && kk == 0) continue;  // T^T[s >= 16][t < 16] = 0
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
          rm_store_acc(Bp, mt, 2 * nq + h, lane, acc[h]);
        }
      } else {
        const int mt = (job - 8) >> 1, np = (job - 8) & 1;  // C n-tiles 2np, 2np + 1
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (mt == 0 && kk == 1) continue;  // M_rb[t < 16][u >= 16] = 0
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
    bsync<kBarPrep, kNP>();

    // ---- S5: K' = K~ diag(gamma_31) + M_ak^T B' (rows t, columns j; K = s) and P = M_rk + C M_ak
    // (rows t, columns s; K = u): 12 jobs
    for (int job = pw; job < 12; job += 8) {
      float acc[2][4] = {};
      if (job < 8) {
        const int mt = job >> 2, nq = job & 3;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (mt == 1 && kk == 0) continue;  // M_ak^T[t >= 16][s < 16] = 0
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
          if (mt == 0 && kk == 1) continue;  // C[t < 16][u >= 16] = 0
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
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
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

WKV7_DEBUG_READER(debug_word_chain)

}  // namespace wkv7
