// WKV7 on sm_103a as chunk operators: every 32-token chunk's transition operator at once (a parallel
// kernel over all heads and chunks), then a short serial chain per head that applies them.
//
// Recurrence ("RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel architecture",
// Forward and Backward listings), per head, state S (rows i = value, columns j = key):
//     sa_t = S_{t-1} a_t;   S_t = S_{t-1} diag(w_t) + v_t k_t^T + sa_t b_t^T = S_{t-1} M_t + v_t k_t^T;
//     y_t = S_t r_t,        M_t = diag(w_t) + a_t b_t^T.
// Over a chunk of n <= 32 tokens from the state S_c before it, with A_{<=t} = M_0 .. M_t:
//     S_t = S_c A_{<=t} + U_{<=t},   U_{<=t} = sum_{s<=t} v_s k_s^T M_{s+1} .. M_t
//     S_end = S_c A_c + U_c          (A_c = A_{<=n-1}, U_c = U_{<=n-1})
//     Y_c^T = S_c Q_c + Y_intra^T    (column t of Q_c: A_{<=t} r_t; row t of Y_intra: U_{<=t} r_t)
// and the backward's state gradient (G: w.r.t. the state after the chunk, from every later token)
//     G_prev = G A_c^T + E_c,        E_c = DY^T Q_c^T   (row t of DY: dy_t).
// The operators in closed form (gamma_t = w_0 o .. o w_t per column, gamma_L = gamma_31, steps past n
// padded with w = 1 and zero inputs):
//     A^_t = a_t o gamma_{t-1},  R^_t = r_t o gamma_t,  K~_t = k_t / gamma_t,  B~_t = b_t / gamma_t,
//     M_ab = tril(A^ B~^T, -1), M_ak = tril(A^ K~^T, -1), M_rb = tril(R^ B~^T), M_rk = tril(R^ K~^T),
//     T = (I - M_ab)^-1,  B' = (T^T B~) diag(gamma_L),  C = M_rb T,
//     K' = K~ diag(gamma_L) + M_ak^T B',  P = M_rk + C M_ak,
//     A_c = diag(gamma_L) + A^^T B',  U_c = V^T K',  Q_c = (R^ + C A^)^T,  Y_intra = P V.
// (Unrolled over the chunk, sa is coupled through the unit lower-triangular system I - M_ab; T
// eliminates it.)  A chunk whose gamma_L falls below 1e-20 in some column, or above 1e37 (only decays
// w > 1 reach that) or is not finite, forms the same operators token by token instead (rows of A_c and
// U_c run the recurrence from I and 0), which divides by nothing.
//
// xop_prep_kernel: all chunks at once, two CTAs per SM each looping over chunks (the next chunk's inputs
// loaded during the current one's last products); writes A_c (bf16 hi + lo) and, forward, Q_c (bf16 hi +
// lo), U_c, Y_intra^T and the coupling matrices, or, backward, E_c, per chunk, into an operator block.
// xop_chain_kernel: one CTA per (head, block of R state rows); a producer warp streams the chunks'
// operator blocks into a ring of shared-memory stages with cp.async.bulk (one mbarrier per stage and
// direction); 2 R / 16 chain warps hold 16 state rows by 32 columns each as mma accumulators and apply
//     forward: y_c = S Q_c + Y_intra;  S = S A_c + U_c  (checkpoint after every chunk)
//     walk:    G_c written;   G = G A_c^T + E_c (G_c over E_c's block, accumulator order; dh0 at the end).
// xop_e_kernel: E_c from the Q_c a forward left in its blocks (the backward on the forward's operators).
// The walk on a forward's blocks with whole-head CTAs instead copies the chunk's dy rows beside A_c and Q_c,
// and the chain warps form E_c = DY^T Q_c^T at their own rows and columns, one chunk ahead (G_c then goes
// over U_c's block).
// Precision: products of fp32 operands as three bf16 products (hi hi + hi lo + lo hi, ~2^-17 each),
// fp32 accumulation (wkv7_mma.cuh).  Waits are bounded in time: past the limit a kernel sets the status
// word and returns.
#include "wkv7_device.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"

namespace wkv7 {
namespace {

using namespace mma;

constexpr int kL = 32;
constexpr int kLD64 = 72;
constexpr int kLD32 = 40;
constexpr float kMinGamma = 1e-20f;
constexpr float kMaxGamma = 1e37f;  // (1 / gamma by __fdividef, exact to a few ulp below 2^126)
constexpr unsigned long long kWaitNs = 2000000000ull;  // a stage wait gives up after 2 s

// ---- per-chunk operator block (bytes).  A_c and Q_c: bf16 hi array then lo array, rows unpadded, the
// 16-byte pieces of row j permuted (piece p stored at p ^ (j & 7) for A, p ^ ((j >> 1) & 3) for Q) so
// that ldmatrix reads of eight rows hit eight distinct bank groups.  X: U_c or E_c (fp32) in mma
// accumulator order [m-tile of 16 rows][n-tile of 8 columns][lane][4] (acc_order in wkv7_mma.cuh); the
// walk overwrites it with G in the same order.  The forward's blocks add Y: Y_intra^T (rows i, columns t;
// fp32) in the same order [i / 16][t / 8][lane][4], so that a chain CTA fetches its rows' part in one
// copy; and M: M_ak, M_rb, M_rk and T (5 KB each: bf16 hi rows then lo rows, 32 x 32 in rows of 40
// elements, the operand layout of shared memory, so that one bulk copy moves all four each way) for a
// backward that reuses them.  A backward alone uses only A, Q and X.
constexpr int kXA = 0;
constexpr int kXQ = 16384;
constexpr int kXX = 24576;
constexpr int kXY = 40960;
constexpr int kXM = 49152;
constexpr int kXMBytes = 20480;
constexpr int kXBytesFwd = kXM + kXMBytes;  // block stride of the forward's workspace (68 KB)
constexpr int kXBytesBwd = 40960;  // ... of a backward's own

// index (floats) of element (i, t) of a 64 x 32 fp32 matrix in mma accumulator order
__host__ __device__ __forceinline__ int acc_order32(int i, int t) {
  const int lane = (i & 7) * 4 + ((t & 7) >> 1);
  const int e = ((i >> 3) & 1) * 2 + (t & 1);
  return ((((i >> 4) * 4 + (t >> 3)) * 32 + lane) << 2) + e;
}
constexpr int kXHead = 256;  // status word(s) before the first block

__host__ __device__ __forceinline__ int swz_a(int j, int jp) { return j * 64 + (((jp >> 3) ^ (j & 7)) << 3) + (jp & 7); }
__host__ __device__ __forceinline__ int swz_q(int j, int t) {
  return j * 32 + (((t >> 3) ^ ((j >> 1) & 3)) << 3) + (t & 7);
}

__host__ __device__ constexpr int rmb(int rows, int ld) { return 2 * rows * ld * 2; }

// shared -> global bulk copy (16-byte aligned addresses, size a multiple of 16), in the issuing thread's
// bulk group; the generic-proxy writes it reads are made visible to the copy by fence_async_smem in every
// writing thread before a barrier
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* ssrc, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(gdst),
               "r"(static_cast<unsigned>(__cvta_generic_to_shared(ssrc))), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// ======================================================================================= prep

constexpr int kNTP = 256;

template <typename Tin, bool BWD>
struct XPrepLay {
  // region X: raw inputs + gamma first, then the coupling matrices
  static constexpr int kRawN = BWD ? 4 : 6;  // w, a, b, r (, k, v)
  static constexpr int kRaw = kRawN * kL * kD * (int)sizeof(Tin);
  static constexpr int oRaw = 0;
  static constexpr int oDyRaw = kRaw;  // backward: dy fp32 [32][64]
  static constexpr int oG = oDyRaw + (BWD ? kL * kD * 4 : 0);
  static constexpr int kXa = oG + kL * kD * 4;
  static constexpr int kSM = 36;
  static constexpr int oMab = 0;                        // fp32 [32][36]
  static constexpr int oTI = oMab + 32 * kSM * 4;       // fp32 [32][36]
  static constexpr int oE = oTI + 32 * kSM * 4;         // fp32 [16][16]
  static constexpr int oMak = oE + 16 * 16 * 4;         // RM 32 x 32 each
  static constexpr int oMrb = oMak + rmb(32, kLD32);
  static constexpr int oMrk = oMrb + rmb(32, kLD32);
  static constexpr int oT = oMrk + rmb(32, kLD32);
  static constexpr int kXb = oT + rmb(32, kLD32);
  static constexpr int kX = ((kXa > kXb ? kXa : kXb) + 127) / 128 * 128;
  // long-lived operands
  static constexpr int oAh = kX;
  static constexpr int oRh = oAh + rmb(32, kLD64);
  static constexpr int oBt = oRh + rmb(32, kLD64);  // B~, then K' (forward)
  static constexpr int oKt = oBt + rmb(32, kLD64);  // K~ (forward) or DY (backward)
  static constexpr int oV = oKt + rmb(32, kLD64);   // V (forward; hi only for bf16 inputs)
  static constexpr int kV = BWD ? 0 : (sizeof(Tin) == 2 ? 32 * kLD64 * 2 : rmb(32, kLD64));
  static constexpr int oBp = oV + kV;
  static constexpr int oC = oBp + rmb(32, kLD64);
  static constexpr int oP = oC + rmb(32, kLD32);  // P (forward) or Q as RM [64 j][32 t] (backward)
  static constexpr int kP = BWD ? rmb(64, kLD32) : rmb(32, kLD32);
  static constexpr int oGL = oP + kP;  // fp32 [64], then int [8]
  static constexpr int oBT = oGL + 64 * 4 + 32;  // fp32 [4][64]: block products of the gamma scan
  static constexpr int kBytes = oBT + 4 * 64 * 4;
  // token-by-token path: q_t as fp32 [64 j][33] over A^
  static constexpr int oQf = oAh;
  static_assert(64 * 33 * 4 <= rmb(32, kLD64), "q_t fit over A^");
};

template <typename Tin, bool BWD>
__global__ void __launch_bounds__(kNTP, 2)  // two CTAs per SM (bf16 inputs: ~93 KB of shared memory each)
xop_prep_kernel(int T, int H, int nchunks, int total, const Tin* __restrict__ r, const Tin* __restrict__ w,
                const Tin* __restrict__ k, const Tin* __restrict__ v, const Tin* __restrict__ a,
                const Tin* __restrict__ b, const float* __restrict__ dy, unsigned char* __restrict__ ops,
                size_t bstride, unsigned* __restrict__ status) {
  using LY = XPrepLay<Tin, BWD>;
  constexpr int SM = LY::kSM;
  constexpr bool kVExact = sizeof(Tin) == 2;
  extern __shared__ float4 smem4[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(smem4);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const size_t tstride = (size_t)H * kD;
  if (blockIdx.x == 0 && tid == 0 && status != nullptr) *status = 0u;

  auto bfp = [&](int off) { return reinterpret_cast<__nv_bfloat16*>(sm + off); };
  const RM Ah{bfp(LY::oAh), 32 * kLD64, kLD64}, Rh{bfp(LY::oRh), 32 * kLD64, kLD64};
  const RM Bt{bfp(LY::oBt), 32 * kLD64, kLD64}, Kt{bfp(LY::oKt), 32 * kLD64, kLD64};
  const RM Kp = Bt, DYm = Kt;
  const RM Vm{bfp(LY::oV), kVExact ? 0 : 32 * kLD64, kLD64};
  const RM Bp{bfp(LY::oBp), 32 * kLD64, kLD64};
  const RM Cm{bfp(LY::oC), 32 * kLD32, kLD32};
  const RM Pm{bfp(LY::oP), 32 * kLD32, kLD32};
  const RM Qs{bfp(LY::oP), 64 * kLD32, kLD32};
  const RM Mak{bfp(LY::oMak), 32 * kLD32, kLD32}, Mrb{bfp(LY::oMrb), 32 * kLD32, kLD32};
  const RM Mrk{bfp(LY::oMrk), 32 * kLD32, kLD32}, Tm{bfp(LY::oT), 32 * kLD32, kLD32};
  float* G = reinterpret_cast<float*>(sm + LY::oG);
  float* GL = reinterpret_cast<float*>(sm + LY::oGL);
  int* meta = reinterpret_cast<int*>(sm + LY::oGL + 256);
  Tin* raw = reinterpret_cast<Tin*>(sm + LY::oRaw);
  const Tin* rw = raw;
  const Tin* ra = raw + kL * kD;
  const Tin* rbv = raw + 2 * kL * kD;
  const Tin* rr = raw + 3 * kL * kD;
  const Tin* rk = raw + 4 * kL * kD;
  const Tin* rv = raw + 5 * kL * kD;
  float* dyr = reinterpret_cast<float*>(sm + LY::oDyRaw);
  float* Mab = reinterpret_cast<float*>(sm + LY::oMab);
  float* TI = reinterpret_cast<float*>(sm + LY::oTI);

  // A chunk's inputs (rows past the chunk are not copied) by cp.async.  The CTA loops over chunks
  // blockIdx.x, + gridDim.x, ...; the next chunk's inputs are issued once the current chunk's raw inputs
  // and coupling matrices are dead (before its last products).
  auto issue = [&](int jb) {
    const int ci_ = jb % nchunks, bh_ = jb / nchunks;
    const int bi_ = bh_ / H, hi_ = bh_ - bi_ * H;
    const int t0_ = ci_ * kL, nm_ = min(kL, T - t0_);
    const size_t base_ = ((size_t)bi_ * T * H + hi_) * kD;
    constexpr int CPR = kD * (int)sizeof(Tin) / 16;
    constexpr int EPC = 16 / (int)sizeof(Tin);
    const Tin* srcs[6] = {w, a, b, r, k, v};
#pragma unroll
    for (int s6 = 0; s6 < LY::kRawN; ++s6)
      for (int e = tid; e < nm_ * CPR; e += kNTP) {
        const int t = e / CPR, pc = e % CPR;
        cp_async16(raw + (s6 * kL + t) * kD + pc * EPC, srcs[s6] + base_ + (size_t)(t0_ + t) * tstride + pc * EPC);
      }
    if (BWD)
      for (int e = tid; e < nm_ * (kD / 4); e += kNTP) {
        const int t = e >> 4, pc = e & 15;
        cp_async16(dyr + t * kD + pc * 4, dy + base_ + (size_t)(t0_ + t) * tstride + pc * 4);
      }
    cp_async_commit();
  };
  if (blockIdx.x < total) issue(blockIdx.x);

  for (int job = blockIdx.x; job < total; job += gridDim.x) {
  const int ci = job % nchunks;
  const int bh = job / nchunks;
  const int t0 = ci * kL;
  const int nm = min(kL, T - t0);
  unsigned char* blk = ops + ((size_t)bh * nchunks + ci) * bstride;
  __nv_bfloat16* gA = reinterpret_cast<__nv_bfloat16*>(blk + kXA);
  __nv_bfloat16* gQ = reinterpret_cast<__nv_bfloat16*>(blk + kXQ);
  float* gX = reinterpret_cast<float*>(blk + kXX);
  float* gY = reinterpret_cast<float*>(blk + kXY);
  const int next = job + gridDim.x;
  cp_async_wait<0>();
  __syncthreads();

  {  // gamma_t down each column as a scan: column j, tokens 8 blk .. 8 blk + 7; the token-by-token flag
    float* BT = reinterpret_cast<float*>(sm + LY::oBT);
    const int j = tid & 63, blk = tid >> 6;
    float loc[8];
    float p = 1.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = 8 * blk + u;
      p *= t < nm ? to_f32(rw[t * kD + j]) : 1.f;
      loc[u] = p;
    }
    BT[blk * 64 + j] = p;
    __syncthreads();
    float pre = 1.f;
    for (int q2 = 0; q2 < blk; ++q2) pre *= BT[q2 * 64 + j];
#pragma unroll
    for (int u = 0; u < 8; ++u) G[(8 * blk + u) * kD + j] = pre * loc[u];
    bool bad = false;
    if (blk == 3) {
      const float gm = pre * p;
      GL[j] = gm;
      bad = !(gm >= kMinGamma) || !(gm <= kMaxGamma);
    }
    const unsigned any = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) meta[warp] = any != 0u;
  }
  __syncthreads();

  if ((meta[0] | meta[1] | meta[2] | meta[3] | meta[4] | meta[5] | meta[6] | meta[7]) != 0) {
    // ======== token by token: rows j of A_c from e_j (threads 0-63), rows i of U_c from 0 (64-127, forward)
    float* Qf = reinterpret_cast<float*>(sm + LY::oQf);
    if (tid < 64) {
      const int j = tid;
      float x[64];
#pragma unroll
      for (int u = 0; u < 64; ++u) x[u] = u == j ? 1.f : 0.f;
      for (int t = 0; t < nm; ++t) {
        float d = 0.f;
#pragma unroll
        for (int u = 0; u < 64; ++u) d = fmaf(x[u], to_f32(ra[t * kD + u]), d);
        float qv = 0.f;
#pragma unroll
        for (int u = 0; u < 64; ++u) {
          x[u] = fmaf(x[u], to_f32(rw[t * kD + u]), d * to_f32(rbv[t * kD + u]));
          qv = fmaf(x[u], to_f32(rr[t * kD + u]), qv);
        }
        Qf[j * 33 + t] = qv;
      }
      for (int t = nm; t < kL; ++t) Qf[j * 33 + t] = 0.f;
#pragma unroll
      for (int p8 = 0; p8 < 8; ++p8) {
        uint4 h, l;
        split2(x[p8 * 8 + 0], x[p8 * 8 + 1], h.x, l.x);
        split2(x[p8 * 8 + 2], x[p8 * 8 + 3], h.y, l.y);
        split2(x[p8 * 8 + 4], x[p8 * 8 + 5], h.z, l.z);
        split2(x[p8 * 8 + 6], x[p8 * 8 + 7], h.w, l.w);
        *reinterpret_cast<uint4*>(gA + swz_a(j, p8 * 8)) = h;
        *reinterpret_cast<uint4*>(gA + 4096 + swz_a(j, p8 * 8)) = l;
      }
    } else if (!BWD && tid < 128) {
      const int i = tid - 64;
      float u8[64];
#pragma unroll
      for (int u = 0; u < 64; ++u) u8[u] = 0.f;
      for (int t = 0; t < nm; ++t) {
        float d = 0.f;
#pragma unroll
        for (int u = 0; u < 64; ++u) d = fmaf(u8[u], to_f32(ra[t * kD + u]), d);
        const float vi = to_f32(rv[t * kD + i]);
        float yv = 0.f;
#pragma unroll
        for (int u = 0; u < 64; ++u) {
          u8[u] = fmaf(u8[u], to_f32(rw[t * kD + u]), fmaf(vi, to_f32(rk[t * kD + u]), d * to_f32(rbv[t * kD + u])));
          yv = fmaf(u8[u], to_f32(rr[t * kD + u]), yv);
        }
        gY[acc_order32(i, t)] = yv;
      }
      for (int t = nm; t < kL; ++t) gY[acc_order32(i, t)] = 0.f;
#pragma unroll
      for (int u = 0; u < 64; ++u) gX[acc_order(i, u)] = u8[u];
    }
    __syncthreads();
    if (!BWD) {
      for (int e = tid; e < 64 * 4; e += kNTP) {  // Q_c rows j, 8 tokens per piece
        const int j = e >> 2, p4 = e & 3;
        const float* src = Qf + j * 33 + p4 * 8;
        uint4 h, l;
        split2(src[0], src[1], h.x, l.x);
        split2(src[2], src[3], h.y, l.y);
        split2(src[4], src[5], h.z, l.z);
        split2(src[6], src[7], h.w, l.w);
        *reinterpret_cast<uint4*>(gQ + swz_q(j, p4 * 8)) = h;
        *reinterpret_cast<uint4*>(gQ + 2048 + swz_q(j, p4 * 8)) = l;
      }
    } else {
      for (int e = tid; e < 64 * 64; e += kNTP) {  // E_c[i][j] = sum_t dy_t[i] q_t[j]
        const int i = e >> 6, j = e & 63;
        float s = 0.f;
        for (int t = 0; t < nm; ++t) s = fmaf(dyr[t * kD + i], Qf[j * 33 + t], s);
        gX[acc_order(i, j)] = s;
      }
    }
    __syncthreads();  // the raw inputs and dy are read
    if (next < total) issue(next);
    continue;
  }

  {  // one (token, 8 columns) block per thread: A^, R^, B~, and K~, V (forward) or DY (backward)
    const int t = tid >> 3, c0 = (tid & 7) * 8;
    const bool ok = t < nm;
    float gt[8], gp[8], av[8], rv8[8], bv[8];
    raw8(G + t * kD + c0, gt);
    if (t > 0) {
      raw8(G + (t - 1) * kD + c0, gp);
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) gp[u] = 1.f;
    }
    raw8(ra + t * kD + c0, av);
    raw8(rr + t * kD + c0, rv8);
    raw8(rbv + t * kD + c0, bv);
    float oa[8], orr[8], ob[8], ig[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      ig[u] = __fdividef(1.f, gt[u]);
      oa[u] = ok ? av[u] * gp[u] : 0.f;
      orr[u] = ok ? rv8[u] * gt[u] : 0.f;
      ob[u] = ok ? bv[u] * ig[u] : 0.f;
    }
    rm_store8(Ah, t, c0, oa);
    rm_store8(Rh, t, c0, orr);
    rm_store8(Bt, t, c0, ob);
    if (!BWD) {
      float kv[8], vv[8], ok8[8];
      raw8(rk + t * kD + c0, kv);
      raw8(rv + t * kD + c0, vv);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ok8[u] = ok ? kv[u] * ig[u] : 0.f;
        vv[u] = ok ? vv[u] : 0.f;
      }
      rm_store8(Kt, t, c0, ok8);
      if (kVExact) rm_store8_hi(Vm, t, c0, vv); else rm_store8(Vm, t, c0, vv);
    } else {
      float d8[8];
      raw8(dyr + t * kD + c0, d8);
#pragma unroll
      for (int u = 0; u < 8; ++u) d8[u] = ok ? d8[u] : 0.f;
      rm_store8(DYm, t, c0, d8);
    }
  }
  __syncthreads();  // raw inputs and gamma consumed: the coupling matrices reuse their space

  // M_ab = tril(A^ B~^T, -1) (fp32), the only coupling matrix T needs: warps 0-2, one of its three nonzero
  // (m-tile, pair of n-tiles) each
  if (warp < 3) {
    const int mt = warp >= 1 ? 1 : 0, np = warp == 2 ? 1 : 0;  // (0, 0), (1, 0), (1, 1)
    float acc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const FragA fa = rm_a(Ah, mt, kk, lane);
      FragB fb[2];
      rm_b2(Bt, 2 * np, kk, lane, fb[0], fb[1]);
      mma3n<2>(acc, fa, fb);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tr = mt * 16 + g, sc = (2 * np + h) * 8 + 2 * q;
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] = sc + (e & 1) < tr + ((e >> 1) << 3) ? acc[h][e] : 0.f;
      *reinterpret_cast<float2*>(Mab + tr * SM + sc) = make_float2(c[0], c[1]);
      *reinterpret_cast<float2*>(Mab + (tr + 8) * SM + sc) = make_float2(c[2], c[3]);
    }
  }
  __syncthreads();

  // T = (I - M_ab)^-1 by blocks of 16 on warp 0: diagonal blocks by forward substitution (one column per
  // lane), then T21 = T22 A21 T11 on tensor cores.  Meanwhile warps 1-3 form (forward) M_ak = tril(A^ K~^T,
  // -1) and M_rk = tril(R^ K~^T) at one nonzero tile each (sharing K~), warps 4-6 M_rb = tril(R^ B~^T), and
  // warp 7 zeroes their blocks above the diagonal (rows 0-15, columns 16-31), which later products read.
  if (warp == 0) {
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
    tri_inverse_t21(Mab, TI, SM, lane);
  } else if (warp < 7) {
    const bool kside = warp <= 3;  // (M_ak, M_rk) or M_rb
    const int j = kside ? warp - 1 : warp - 4;
    const int mt = j >= 1 ? 1 : 0, np = j == 2 ? 1 : 0;
    if (!(BWD && kside)) {
      float acc[2][2][4] = {};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        FragB fb[2];
        rm_b2(kside ? Kt : Bt, 2 * np, kk, lane, fb[0], fb[1]);
        const FragA fr = rm_a(Rh, mt, kk, lane);
        if (kside) {
          const FragA fa = rm_a(Ah, mt, kk, lane);
          mma3n_two<2>(acc[0], fa, fb, acc[1], fr, fb);
        } else {
          mma3n<2>(acc[1], fr, fb);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int nj = 2 * np + h;
        const int tr = mt * 16 + g, sc = nj * 8 + 2 * q;
        float c0[4], c1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tt = tr + ((e >> 1) << 3), s2 = sc + (e & 1);
          c0[e] = s2 < tt ? acc[0][h][e] : 0.f;   // M_ak: strictly below the diagonal
          c1[e] = s2 <= tt ? acc[1][h][e] : 0.f;  // M_rk, M_rb: with the diagonal
        }
        if (kside) {
          rm_store_acc(Mak, mt, nj, lane, c0);
          rm_store_acc(Mrk, mt, nj, lane, c1);
        } else {
          rm_store_acc(Mrb, mt, nj, lane, c1);
        }
      }
    }
  } else {
    for (int e = lane; e < 3 * 2 * 16 * 2; e += 32) {  // (matrix, hi / lo, row, 16-byte piece)
      const int m = e >> 6, hl = (e >> 5) & 1, rr = (e >> 1) & 15, pc = e & 1;
      const RM& X = m == 0 ? Mrb : (m == 1 ? Mak : Mrk);
      if (BWD && m != 0) continue;
      *reinterpret_cast<uint4*>(X.p + hl * X.lo + rm_off(X, rr, 16 + 8 * pc, 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncthreads();
  if (tid < 128) {
    const int t = tid >> 2, u0 = (tid & 3) * 8;
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = u0 + e <= t ? TI[t * SM + u0 + e] : 0.f;
    rm_store8(Tm, t, u0, x);
  }
  __syncthreads();

  // B' = (T^T B~) diag(gamma_L) and C = M_rb T
  for (int job = warp; job < 12; job += 8) {
    float acc[2][4] = {};
    if (job < 8) {
      const int mt = job >> 2, nq = job & 3;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (mt == 1 && kk == 0) continue;
        const FragA fa = rm_at(Tm, mt, kk, lane);
        FragB f0, f1;
        rm_bt2(Bt, 2 * nq, kk, lane, f0, f1);
        {
          const FragB fb2[2] = {f0, f1};
          mma3n<2>(acc, fa, fb2);
        }
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
        {
          const FragB fb2[2] = {f0, f1};
          mma3n<2>(acc, fa, fb2);
        }
      }
      rm_store_acc(Cm, mt, 2 * np, lane, acc[0]);
      rm_store_acc(Cm, mt, 2 * np + 1, lane, acc[1]);
    }
  }
  if (!BWD) fence_async_smem();  // M_ak, M_rb, M_rk, T (written in earlier phases) for the bulk store below
  __syncthreads();
  // (forward) M_ak, M_rb, M_rk and T, contiguous in shared memory, into the block for a backward that
  // reuses them: one bulk copy, read by the end of this phase
  static_assert(LY::oMrb == LY::oMak + rmb(32, kLD32) && LY::oMrk == LY::oMrb + rmb(32, kLD32) &&
                    LY::oT == LY::oMrk + rmb(32, kLD32) && 4 * rmb(32, kLD32) == kXMBytes,
                "the coupling matrices are one contiguous block");
  if (!BWD && tid == 0) bulk_s2g(blk + kXM, sm + LY::oMak, kXMBytes);

  // A_c = diag(gamma_L) + A^^T B' and Q_c = R^^T + A^^T C^T (rows j); forward: K' = K~ diag(gamma_L) +
  // M_ak^T B' (over B~) and P = M_rk + C M_ak.  Warp w: the A_c tiles (m-tiles w >> 2 and (w >> 2) + 2,
  // n-tiles 2 (w & 3) + 0, 1; B' shared), then one Q_c tile, one K' tile and (w < 4) one P tile.
  {
    {
      const int mt0 = warp >> 2, p = warp & 3;
      float acc[2][2][4] = {};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        FragB fb[2];
        rm_bt2(Bp, 2 * p, kk, lane, fb[0], fb[1]);
        const FragA fa0 = rm_at(Ah, mt0, kk, lane), fa1 = rm_at(Ah, mt0 + 2, kk, lane);
        mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
      }
#pragma unroll
      for (int jb = 0; jb < 2; ++jb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int jr = (mt0 + 2 * jb) * 16 + g, col = (2 * p + h) * 8 + 2 * q;
          float* c = acc[jb][h];
          if (jr == col) c[0] += GL[col];
          if (jr == col + 1) c[1] += GL[col + 1];
          if (jr + 8 == col) c[2] += GL[col];
          if (jr + 8 == col + 1) c[3] += GL[col + 1];
          uint32_t hw, lw;
          split2(c[0], c[1], hw, lw);
          *reinterpret_cast<uint32_t*>(gA + swz_a(jr, col)) = hw;
          *reinterpret_cast<uint32_t*>(gA + 4096 + swz_a(jr, col)) = lw;
          split2(c[2], c[3], hw, lw);
          *reinterpret_cast<uint32_t*>(gA + swz_a(jr + 8, col)) = hw;
          *reinterpret_cast<uint32_t*>(gA + 4096 + swz_a(jr + 8, col)) = lw;
        }
    }
    {  // Q_c: m-tile w >> 1, n-tiles 2 (w & 1) + 0, 1
      const int mt = warp >> 1, p = warp & 1;
      float acc[2][4] = {};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        if (p == 0 && kk == 1) continue;  // C[t][s] = 0 for s > t
        const FragA fa = rm_at(Ah, mt, kk, lane);
        FragB fb[2];
        rm_b2(Cm, 2 * p, kk, lane, fb[0], fb[1]);
        mma3n<2>(acc, fa, fb);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jr = mt * 16 + g, tc = (2 * p + h) * 8 + 2 * q;
        acc[h][0] += rm_get1(Rh, tc, jr);
        acc[h][1] += rm_get1(Rh, tc + 1, jr);
        acc[h][2] += rm_get1(Rh, tc, jr + 8);
        acc[h][3] += rm_get1(Rh, tc + 1, jr + 8);
        if (BWD) {
          rm_store_acc(Qs, mt, 2 * p + h, lane, acc[h]);
        } else {
          uint32_t hw, lw;
          split2(acc[h][0], acc[h][1], hw, lw);
          *reinterpret_cast<uint32_t*>(gQ + swz_q(jr, tc)) = hw;
          *reinterpret_cast<uint32_t*>(gQ + 2048 + swz_q(jr, tc)) = lw;
          split2(acc[h][2], acc[h][3], hw, lw);
          *reinterpret_cast<uint32_t*>(gQ + swz_q(jr + 8, tc)) = hw;
          *reinterpret_cast<uint32_t*>(gQ + 2048 + swz_q(jr + 8, tc)) = lw;
        }
      }
    }
    if (!BWD) {
      {  // K': m-tile w >> 2, n-tiles 2 (w & 3) + 0, 1
        const int mt = warp >> 2, nq = warp & 3;
        float acc[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (mt == 1 && kk == 0) continue;
          const FragA fa = rm_at(Mak, mt, kk, lane);
          FragB fb[2];
          rm_bt2(Bp, 2 * nq, kk, lane, fb[0], fb[1]);
          mma3n<2>(acc, fa, fb);
        }
        // K~ is read here for the last time and K' written over B~ (read for the last time by B')
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
      }
      if (warp < 4) {  // P: m-tile w >> 1, n-tiles 2 (w & 1) + 0, 1
        const int mt = warp >> 1, np = warp & 1;
        float acc[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          if (mt == 0 && kk == 1) continue;
          const FragA fa = rm_a(Cm, mt, kk, lane);
          FragB fb[2];
          rm_bt2(Mak, 2 * np, kk, lane, fb[0], fb[1]);
          mma3n<2>(acc, fa, fb);
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
  }
  if (!BWD && tid == 0) bulk_wait_read_all();  // the bulk store has read the matrices
  __syncthreads();
  if (next < total) issue(next);  // the raw inputs and the coupling matrices are dead from here on

  // U_c = V^T K' (forward) or E_c = DY^T Q_c^T (backward), rows i in mma accumulator order: warp w forms
  // m-tiles w >> 2 and (w >> 2) + 2 at n-tiles 2 (w & 3) + 0, 1 (sharing K' or Q_c); the forward then forms
  // Y_intra^T = V^T P^T into the block
  {
    const int mt0 = warp >> 2, p = warp & 3;
    float acc[2][2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      FragB fb[2];
      if (BWD) {
        rm_b2(Qs, 2 * p, kk, lane, fb[0], fb[1]);
        const FragA fa0 = rm_at(DYm, mt0, kk, lane), fa1 = rm_at(DYm, mt0 + 2, kk, lane);
        mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
      } else {
        rm_bt2(Kp, 2 * p, kk, lane, fb[0], fb[1]);
        if (kVExact) {
          const FragA fa0 = rm_at_hi(Vm, mt0, kk, lane), fa1 = rm_at_hi(Vm, mt0 + 2, kk, lane);
          mma2n_two<2>(acc[0], fa0, acc[1], fa1, fb);
        } else {
          const FragA fa0 = rm_at(Vm, mt0, kk, lane), fa1 = rm_at(Vm, mt0 + 2, kk, lane);
          mma3n_two<2>(acc[0], fa0, fb, acc[1], fa1, fb);
        }
      }
    }
#pragma unroll
    for (int jb = 0; jb < 2; ++jb)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int idx = ((mt0 + 2 * jb) * 8 + 2 * p + h) * 32 + lane;
        if (WKV7_IN(idx, 1024, dbg::kXopPrep))
          reinterpret_cast<float4*>(gX)[idx] = make_float4(acc[jb][h][0], acc[jb][h][1], acc[jb][h][2], acc[jb][h][3]);
      }
  }
  if (!BWD) {  // Y_intra^T = V^T P^T (rows i, columns t): m-tile w >> 1, t n-tiles 2 (w & 1) + 0, 1
    const int mt = warp >> 1, p = warp & 1;
    float acc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (kk > p) continue;  // P[t][s] = 0 for s > t
      const FragA fa = kVExact ? rm_at_hi(Vm, mt, kk, lane) : rm_at(Vm, mt, kk, lane);  // A[i][s] = V[s][i]
      FragB fb[2];
      rm_b2(Pm, 2 * p, kk, lane, fb[0], fb[1]);  // B[s][t] = P[t][s]
      if (kVExact)
        mma2n<2>(acc, fa, fb);
      else
        mma3n<2>(acc, fa, fb);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int idx = (mt * 4 + 2 * p + h) * 32 + lane;
      if (WKV7_IN(idx, 512, dbg::kXopPrep))
        reinterpret_cast<float4*>(gY)[idx] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
    }
  }
  }  // chunks
  if (!BWD && tid == 0) bulk_wait_all();  // the last bulk store has landed before the CTA exits
}

// ====================================================================================== chain

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0u;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// wait for the phase of parity `parity` to complete; false once kWaitNs have passed
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long start = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - start > kWaitNs) return false;
  return true;
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16) completing on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// B fragments (n-tiles nt, nt + 1; k-tile kk) of A_c for S A_c: B[k = j][n = j'] = A_c[j][j']
__device__ __forceinline__ void ld_a_fwd(const __nv_bfloat16* sA, int nt, int kk, int lane, FragB& b0, FragB& b1) {
  const int j = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const __nv_bfloat16* p = sA + j * 64 + (((nt + (lane >> 4)) ^ (lane & 7)) << 3);
  uint32_t h[4], l[4];
  ldsm4<true>(h, p);
  ldsm4<true>(l, p + 4096);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}
// ... of A_c^T for G A_c^T: B[k = j'][n = j] = A_c[j][j']
__device__ __forceinline__ void ld_a_walk(const __nv_bfloat16* sA, int nt, int kk, int lane, FragB& b0, FragB& b1) {
  const int j = nt * 8 + (lane & 7) + ((lane >> 4) << 3);
  const __nv_bfloat16* p = sA + j * 64 + (((2 * kk + ((lane >> 3) & 1)) ^ (lane & 7)) << 3);
  uint32_t h[4], l[4];
  ldsm4<false>(h, p);
  ldsm4<false>(l, p + 4096);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}
// ... of Q_c for S Q_c: B[k = j][n = t] = Q_c[j][t]
__device__ __forceinline__ void ld_q_fwd(const __nv_bfloat16* sQ, int nt, int kk, int lane, FragB& b0, FragB& b1) {
  const int j = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const __nv_bfloat16* p = sQ + j * 32 + (((nt + (lane >> 4)) ^ ((j >> 1) & 3)) << 3);
  uint32_t h[4], l[4];
  ldsm4<true>(h, p);
  ldsm4<true>(l, p + 2048);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}

// B fragments of n-tiles nt, nt + 1 at k-tile kk for B[k][n] = Q_c[n][k] (rows j, tokens t) from an
// operator block's Q_c copied as is (hi then lo, pieces permuted as swz_q)
__device__ __forceinline__ void q_b2(const __nv_bfloat16* sq, int nt, int kk, int lane, FragB& b0, FragB& b1) {
  const int j = nt * 8 + (lane & 7) + ((lane >> 4) << 3);
  const int t = kk * 16 + ((lane >> 3) & 1) * 8;
  const int off = swz_q(j, t);
  uint32_t h[4], l[4];
  ldsm4<false>(h, sq + off);
  ldsm4<false>(l, sq + 2048 + off);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}


constexpr int kMaxStages = 5;     // stages in flight: as many as fit one CTA's shared memory, 3 to 5
constexpr int kSmemCap = 232448;  // shared memory per CTA (bytes)

// One chain CTA holds R state rows of a head: R / 16 row blocks of 16 rows, each split by columns between
// two warps (column half 0: columns 0-31, half 1: 32-63) so that a CTA keeps every SM sub-partition's
// tensor pipe busy.  A product over the state's columns (S A_c, S Q_c) needs the whole row block as its A
// operand: each warp forms the fragments of its own half from its accumulators and trades them with its
// partner once per chunk through shared memory (double-buffered by chunk parity, one named barrier per
// pair and chunk).
// EQ (the walk on the forward's operator blocks, which hold Q_c but no E_c): a stage holds A_c, Q_c and
// this CTA's rows of the chunk's dy (fp32, one row of R values per token, rows padded to R + 4 floats so
// that a warp's fragment loads fall in distinct banks), and each chain warp forms its own part of
// E_c = DY^T Q_c^T, one chunk ahead.  A_c and Q_c come in one bulk copy, dy in 16-byte cp.async pieces
// spread over the producer's lanes (small rows: one bulk copy per row would queue 32 short copies per
// stage); the stage's barrier expects lane 0's arrival with the bulk bytes plus one arrival per lane, made
// once the lane's pieces have landed (cp.async.wait_group, one stage behind the copies being issued) so that
// the arrival's release ordering covers them.
template <int R, bool WALK, bool EQ>
struct Stage {
  static_assert(WALK || !EQ, "E_c from Q_c in the walk only");
  static constexpr int kRB = R / 16;                             // row blocks
  static constexpr int kNW = 2 * kRB;                            // chain warps
  static constexpr int oA = 0;                                   // A_c (16 KB), then Q_c (forward, EQ: 8 KB)
  static constexpr int kAQ = (WALK && !EQ) ? 16384 : 24576;
  static constexpr int oX = kAQ;                                 // this CTA's rows of U_c / E_c, or of dy (EQ)
  static constexpr int kDyLd = R + 4;                            // EQ: dy row stride (floats)
  static constexpr int kX = EQ ? kL * kDyLd * 4 : kRB * 4096;
  static constexpr int oY = oX + kX;                             // forward: this CTA's rows of Y_intra^T
  static constexpr int kY = WALK ? 0 : kRB * 2048;
  static constexpr int kBytes = oY + kY;
  static constexpr int kHead = 256;                              // full[kNS], empty[kNS] mbarriers, flags
  static constexpr int oFlag = 128;                              // int [2][kNW] after the mbarriers
  static constexpr int kXch = 2 * kNW * 4 * 32 * 16;             // uint4 [2][kNW][4][32]
  static constexpr int kFit = (kSmemCap - kHead - kXch) / kBytes;
  static constexpr int kNS = kFit > kMaxStages ? kMaxStages : kFit;
  static constexpr int oXch = kHead + kNS * kBytes;
  static constexpr int kSmem = oXch + kXch;
  static_assert(kBytes % 128 == 0, "stage alignment");
  static_assert(kNS >= 3, "at least three stages");
  static_assert(2 * kNS * 8 <= oFlag && oFlag + 2 * kNW * 4 <= kHead, "barriers and flags fit the header");
};

template <int R, bool WALK, bool EQ>
__global__ void __launch_bounds__((2 * R / 16 + 1) * 32)
xop_chain_kernel(int T, int H, int nchunks, const unsigned char* __restrict__ ops, size_t bstride,
                 const float* __restrict__ s0, void* __restrict__ y, bool ybf, float* __restrict__ ck,
                 size_t ck_stride, float* __restrict__ sT, const float* __restrict__ dy, unsigned* __restrict__ status) {
  // forward: s0 = h0 (or null), y out (fp32, or bf16 rounded to nearest when ybf), ck = h_ckpt (or null;
  // ck_stride = 4096 floats), sT = hT.  walk: s0 = dhT (or null), y unused, ck = G over each block's X in accumulator order
  // (ck_stride = bstride / 4), sT = dh0; dy (EQ only): (B, T, H, 64) fp32.  bstride: bytes between operator blocks.
  using ST = Stage<R, WALK, EQ>;
  constexpr int NW = ST::kNW;
  constexpr int NB = 64 / R;
  extern __shared__ float4 smem4[];
  unsigned char* smc = reinterpret_cast<unsigned char*>(smem4);
  uint64_t* full = reinterpret_cast<uint64_t*>(smc);
  uint64_t* empty = full + ST::kNS;
  int* okf = reinterpret_cast<int*>(smc + ST::oFlag);
  uint4* xch = reinterpret_cast<uint4*>(smc + ST::oXch);
  constexpr int kNS = ST::kNS;
  auto stage = [&](int s) { return smc + ST::kHead + s * ST::kBytes; };
  const int bh = blockIdx.x / NB, rb = blockIdx.x - (blockIdx.x / NB) * NB;
  const int bi = bh / H, hi = bh - bi * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t tstride = (size_t)H * kD;
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const unsigned char* hops = ops + (size_t)bh * nchunks * bstride;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&full[s], EQ ? 33 : 1);
      mbar_init(&empty[s], NW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  if (warp == NW) {
    // ================= producer: chunk n into stage n % kNS once the chain warps have released it
    int issued = 0;
    bool ok = true;
    for (int n = 0; n < nchunks; ++n) {
      const int c = WALK ? nchunks - 1 - n : n;
      const int s = n % kNS;
      // every lane observes the release; the warp agrees on the outcome (a time limit could split it)
      if (n >= kNS && !__all_sync(0xffffffffu, mbar_wait(&empty[s], ((n / kNS) - 1) & 1))) {
        ok = false;
        break;
      }
      const int nm = min(kL, T - c * kL);
      unsigned char* st = stage(s);
      const unsigned char* src = hops + (size_t)c * bstride;
      if (EQ) {
        // A_c and Q_c in one bulk copy; the chunk's dy rows (this CTA's R values of each token) in 16-byte
        // pieces over the lanes, one cp.async group per chunk.  Rows past the chunk are not copied.  Then the
        // previous chunk's pieces of this lane have landed: its arrival releases them.
        if (lane == 0) {
          mbar_expect_tx(&full[s], ST::kAQ);
          bulk_g2s(st + ST::oA, src + kXA, ST::kAQ, &full[s]);
        }
        constexpr int kPPR = R / 4;  // 16-byte pieces per row
        for (int e = lane; e < nm * kPPR; e += 32) {
          const int t = e / kPPR, pc = e - t * kPPR;
          if (WKV7_IN(c * kL + t, T, dbg::kXopChain))
            cp_async16(st + ST::oX + (t * ST::kDyLd + pc * 4) * 4,
                       dy + base + (size_t)(c * kL + t) * tstride + rb * R + pc * 4);
        }
        cp_async_commit();
        if (n > 0) {
          cp_async_wait<1>();
          mbar_arrive(&full[(n - 1) % kNS]);
        }
      } else if (lane == 0) {
        mbar_expect_tx(&full[s], ST::kAQ + ST::kX + ST::kY);
        bulk_g2s(st + ST::oA, src + kXA, ST::kAQ, &full[s]);
        bulk_g2s(st + ST::oX, src + kXX + rb * ST::kX, ST::kX, &full[s]);
        if (!WALK) bulk_g2s(st + ST::oY, src + kXY + rb * ST::kY, ST::kY, &full[s]);
      }
      __syncwarp();
      issued = n + 1;
    }
    if (EQ && issued > 0) {  // the last issued chunk's pieces
      cp_async_wait<0>();
      mbar_arrive(&full[(issued - 1) % kNS]);
    }
    if (!ok) {
      if (lane == 0) atomicOr(status, 1u);
      // the copies already issued land before the CTA may exit
      for (int m = max(0, issued - kNS); m < issued; ++m) mbar_wait(&full[m % kNS], (m / kNS) & 1);
    }
    return;
  }

  // =================== chain warp: state rows rb * R + 16 pair + (g, g + 8), columns 32 half + ..
  const int pair = warp >> 1, half = warp & 1;
  const int g = lane >> 2, q = lane & 3;
  const int lrow = pair * 16 + g;  // row within the CTA's block
  const int row = rb * R + lrow;
  const size_t sbase = (size_t)bh * kD * kD;
  float S[4][4];  // n-tiles 4 half + 0 .. 3
#pragma unroll
  for (int nj = 0; nj < 4; ++nj) {
    const int col = (4 * half + nj) * 8 + 2 * q;
    if (s0 != nullptr) {
      const float2 x0 = __ldg(reinterpret_cast<const float2*>(s0 + sbase + (size_t)row * kD + col));
      const float2 x8 = __ldg(reinterpret_cast<const float2*>(s0 + sbase + (size_t)(row + 8) * kD + col));
      S[nj][0] = x0.x; S[nj][1] = x0.y; S[nj][2] = x8.x; S[nj][3] = x8.y;
    } else {
      S[nj][0] = S[nj][1] = S[nj][2] = S[nj][3] = 0.f;
    }
  }
  auto store_rows = [&](float* dst) {
    if (!WKV7_IN(row + 8, kD, dbg::kXopChain)) return;
#pragma unroll
    for (int nj = 0; nj < 4; ++nj) {
      const int col = (4 * half + nj) * 8 + 2 * q;
      *reinterpret_cast<float2*>(dst + (size_t)row * kD + col) = make_float2(S[nj][0], S[nj][1]);
      *reinterpret_cast<float2*>(dst + (size_t)(row + 8) * kD + col) = make_float2(S[nj][2], S[nj][3]);
    }
  };
  // EQ: E_c at this warp's rows and columns for the m-th chunk taken, into en: DY^T (rows i, tokens t; split
  // into bf16 hi + lo, zero past the chunk) times Q_c^T, the passes in the same order as the backward's
  // operator kernel forms E_c.  Formed one chunk ahead (chunk 0's before the loop), after the current
  // chunk's products, so that it stays off the chain's dependent path.
  float en[4][4];
  auto form_e = [&](int m) {
    const int cm = nchunks - 1 - m;
    const int nmm = min(kL, T - cm * kL);
    const unsigned char* stm = stage(m % kNS);
    const float* sdy = reinterpret_cast<const float*>(stm + ST::oX);
    const __nv_bfloat16* sqm = reinterpret_cast<const __nv_bfloat16*>(stm + kXQ);
    auto dyv = [&](int t, int i) { return t < nmm ? sdy[t * ST::kDyLd + i] : 0.f; };
#pragma unroll
    for (int nj = 0; nj < 4; ++nj) en[nj][0] = en[nj][1] = en[nj][2] = en[nj][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int t = kk * 16 + 2 * q;
      FragA fa;
      split2(dyv(t, lrow), dyv(t + 1, lrow), fa.h[0], fa.l[0]);
      split2(dyv(t, lrow + 8), dyv(t + 1, lrow + 8), fa.h[1], fa.l[1]);
      split2(dyv(t + 8, lrow), dyv(t + 9, lrow), fa.h[2], fa.l[2]);
      split2(dyv(t + 8, lrow + 8), dyv(t + 9, lrow + 8), fa.h[3], fa.l[3]);
      FragB fb[4];
      q_b2(sqm, 4 * half, kk, lane, fb[0], fb[1]);
      q_b2(sqm, 4 * half + 2, kk, lane, fb[2], fb[3]);
      mma3n<4>(en, fa, fb);
    }
  };
  if (EQ && nchunks > 0) {
    (void)mbar_wait(&full[0], 0);  // (a wait that gives up is met again, and acted on, in the loop)
    form_e(0);
  }

  for (int n = 0; n < nchunks; ++n) {
    const int c = WALK ? nchunks - 1 - n : n;
    const int s = n % kNS;
    const int par = n & 1;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (n / kNS) & 1));
    // this warp's half of the chunk-start state as A fragments (k-tiles 2 half, 2 half + 1), handed to
    // the partner; both warps of the pair learn whether either wait gave up, and leave together
    FragA own[2] = {frag_from_acc(S[0], S[1]), frag_from_acc(S[2], S[3])};
    {
      uint4* xo = xch + ((par * NW + warp) * 4) * 32 + lane;
      xo[0] = make_uint4(own[0].h[0], own[0].h[1], own[0].h[2], own[0].h[3]);
      xo[32] = make_uint4(own[0].l[0], own[0].l[1], own[0].l[2], own[0].l[3]);
      xo[64] = make_uint4(own[1].h[0], own[1].h[1], own[1].h[2], own[1].h[3]);
      xo[96] = make_uint4(own[1].l[0], own[1].l[1], own[1].l[2], own[1].l[3]);
      if (lane == 0) okf[par * NW + warp] = ok ? 1 : 0;
    }
    asm volatile("bar.sync %0, 64;\n" ::"r"(1 + pair) : "memory");
    if (!ok || okf[par * NW + (warp ^ 1)] == 0) {
      if (!ok && lane == 0) atomicOr(status, 1u);
      return;
    }
    FragA oth[2];
    {
      const uint4* xi = xch + ((par * NW + (warp ^ 1)) * 4) * 32 + lane;
      const uint4 a0 = xi[0], a1 = xi[32], a2 = xi[64], a3 = xi[96];
      oth[0].h[0] = a0.x; oth[0].h[1] = a0.y; oth[0].h[2] = a0.z; oth[0].h[3] = a0.w;
      oth[0].l[0] = a1.x; oth[0].l[1] = a1.y; oth[0].l[2] = a1.z; oth[0].l[3] = a1.w;
      oth[1].h[0] = a2.x; oth[1].h[1] = a2.y; oth[1].h[2] = a2.z; oth[1].h[3] = a2.w;
      oth[1].l[0] = a3.x; oth[1].l[1] = a3.y; oth[1].l[2] = a3.z; oth[1].l[3] = a3.w;
    }
    const unsigned char* st = stage(s);
    const __nv_bfloat16* sA = reinterpret_cast<const __nv_bfloat16*>(st + ST::oA);
    // the walk's G before this chunk, in accumulator order, over the block's X (E_c, already read into the
    // stage; or, EQ, the forward's U_c)
    if (WALK && ck != nullptr) {
      float4* dst = reinterpret_cast<float4*>(ck + ((size_t)bh * nchunks + c) * ck_stride) +
                    ((rb * ST::kRB + pair) * 8 + 4 * half) * 32 + lane;
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) dst[nj * 32] = make_float4(S[nj][0], S[nj][1], S[nj][2], S[nj][3]);
    }
    // S = S A_c + U_c (forward) or G = G A_c^T + E_c (walk) at this warp's columns; the forward also
    // y_c^T += S Q_c at tokens 16 half .. 16 half + 15 (rows i, columns t).  The own k-tiles go first;
    // per k-step the three bf16 passes go over all accumulators in turn, so that dependent mma into one
    // accumulator are 4 (walk) or 6 (forward) instructions apart.
    const int nm = min(kL, T - c * kL);
    const __nv_bfloat16* sQ = reinterpret_cast<const __nv_bfloat16*>(st + kXQ);
    float acc[4][4], ya[2][4];
    if (EQ) {
#pragma unroll
      for (int nj = 0; nj < 4; ++nj)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nj][e] = en[nj][e];
    } else {
      const float4* xs = reinterpret_cast<const float4*>(st + ST::oX) + (pair * 8 + 4 * half) * 32 + lane;
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) {
        const float4 u = xs[nj * 32];
        acc[nj][0] = u.x; acc[nj][1] = u.y; acc[nj][2] = u.z; acc[nj][3] = u.w;
      }
    }
    if (!WALK) {
      const float4* ys = reinterpret_cast<const float4*>(st + ST::oY) + (pair * 4 + 2 * half) * 32 + lane;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float4 u = ys[nt * 32];
        ya[nt][0] = u.x; ya[nt][1] = u.y; ya[nt][2] = u.z; ya[nt][3] = u.w;
      }
    }
#pragma unroll
    for (int ki = 0; ki < 4; ++ki) {
      const int kk = (2 * half + ki) & 3;
      const FragA& fa = ki < 2 ? own[ki] : oth[ki - 2];
      FragB fb[4], fq[2];
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        if (WALK)
          ld_a_walk(sA, 4 * half + 2 * np, kk, lane, fb[2 * np], fb[2 * np + 1]);
        else
          ld_a_fwd(sA, 4 * half + 2 * np, kk, lane, fb[2 * np], fb[2 * np + 1]);
      }
      if (!WALK) ld_q_fwd(sQ, 2 * half, kk, lane, fq[0], fq[1]);
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) mma16816(acc[nj], fa.l, fb[nj].h[0], fb[nj].h[1]);
      if (!WALK)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma16816(ya[nt], fa.l, fq[nt].h[0], fq[nt].h[1]);
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) mma16816(acc[nj], fa.h, fb[nj].l[0], fb[nj].l[1]);
      if (!WALK)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma16816(ya[nt], fa.h, fq[nt].l[0], fq[nt].l[1]);
#pragma unroll
      for (int nj = 0; nj < 4; ++nj) mma16816(acc[nj], fa.h, fb[nj].h[0], fb[nj].h[1]);
      if (!WALK)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma16816(ya[nt], fa.h, fq[nt].h[0], fq[nt].h[1]);
    }
    if (!WALK) {
      const size_t yo = base + (size_t)(c * kL) * tstride;
      auto put = [&](int t, int rr, float v) {
        const size_t o = yo + (size_t)t * tstride + rr;
        if (ybf)
          static_cast<__nv_bfloat16*>(y)[o] = __float2bfloat16_rn(v);
        else
          static_cast<float*>(y)[o] = v;
      };
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int tc = (2 * half + nt) * 8 + 2 * q;
        if (tc < nm) {
          put(tc, row, ya[nt][0]);
          put(tc, row + 8, ya[nt][2]);
        }
        if (tc + 1 < nm) {
          put(tc + 1, row, ya[nt][1]);
          put(tc + 1, row + 8, ya[nt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
    for (int nj = 0; nj < 4; ++nj)
#pragma unroll
      for (int e = 0; e < 4; ++e) S[nj][e] = acc[nj][e];
    if (EQ && n + 1 < nchunks) {
      (void)mbar_wait(&full[(n + 1) % kNS], ((n + 1) / kNS) & 1);  // (as above)
      form_e(n + 1);
    }
    if (!WALK && ck != nullptr) store_rows(ck + ((size_t)bh * nchunks + c) * ck_stride);
  }
  if (sT != nullptr) store_rows(sT + sbase);
}

template <typename Tin, bool BWD>
cudaError_t launch_prep_t(const FwdArgs* fa, const BwdArgs* ba, unsigned char* ops, size_t bstride, unsigned* status,
                          cudaStream_t stream) {
  using LY = XPrepLay<Tin, BWD>;
  static_assert(LY::kBytes <= 232448, "shared memory per CTA");
  auto kern = xop_prep_kernel<Tin, BWD>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
  if (err != cudaSuccess) return err;
  const int B = BWD ? ba->B : fa->B, T = BWD ? ba->T : fa->T, H = BWD ? ba->H : fa->H;
  const int C = BWD ? ba->nchunks : fa->nchunks;
  const TokenInputs& in = BWD ? ba->in : fa->in;
  const int total = B * H * C;
  const unsigned grid = (unsigned)min(total, 2 * num_sms());  // two CTAs per SM, each looping over its chunks
  kern<<<grid, kNTP, LY::kBytes, stream>>>(T, H, C, total, (const Tin*)in.r, (const Tin*)in.w, (const Tin*)in.k,
                                          (const Tin*)in.v, (const Tin*)in.a, (const Tin*)in.b,
                                          BWD ? ba->dy : nullptr, ops, bstride, status);
  return cudaGetLastError();
}

template <int R, bool WALK, bool EQ>
cudaError_t launch_chain_t(int B, int T, int H, int C, const unsigned char* ops, size_t bstride, const float* s0, void* y,
                           bool ybf, float* ck, size_t ck_stride, float* sT, const float* dy, unsigned* status,
                           cudaStream_t stream) {
  using ST = Stage<R, WALK, EQ>;
  static_assert(ST::kSmem <= 232448, "shared memory per CTA");
  auto kern = xop_chain_kernel<R, WALK, EQ>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ST::kSmem);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)B * H * (64 / R);
  kern<<<grid, (ST::kNW + 1) * 32, ST::kSmem, stream>>>(T, H, C, ops, bstride, s0, y, ybf, ck, ck_stride, sT, dy,
                                                        status);
  return cudaGetLastError();
}

// state rows per chain CTA.  Two CTAs of 32 rows per head (the head's operators read twice) while they fit
// one CTA per SM: measured faster than one 64-row CTA there (B12 T1024 H6 forward 115 vs 121 us, B4 T512
// H12 54 vs 57 us); whole heads past that (B2 T4096 H64: 636 vs 678 us).  WKV7_CHAIN_ROWS fixes the choice.
int chain_rows(int heads) {
#ifdef WKV7_CHAIN_ROWS
  (void)heads;
  return WKV7_CHAIN_ROWS;
#else
  return 2 * heads <= num_sms() ? 32 : 64;
#endif
}

template <bool WALK>
cudaError_t launch_chain(int rows, int B, int T, int H, int C, const unsigned char* ops, size_t bstride, const float* s0,
                         void* y, bool ybf, float* ck, size_t ck_stride, float* sT, unsigned* status,
                         cudaStream_t stream) {
  switch (rows) {
    case 64:
      return launch_chain_t<64, WALK, false>(B, T, H, C, ops, bstride, s0, y, ybf, ck, ck_stride, sT, nullptr, status,
                                             stream);
    case 32:
      return launch_chain_t<32, WALK, false>(B, T, H, C, ops, bstride, s0, y, ybf, ck, ck_stride, sT, nullptr, status,
                                             stream);
    default:
      return launch_chain_t<16, WALK, false>(B, T, H, C, ops, bstride, s0, y, ybf, ck, ck_stride, sT, nullptr, status,
                                             stream);
  }
}

// ================================================================================ E_c from the forward

constexpr int kNTE = 128;

// E_c = DY^T Q_c^T of every chunk from the Q_c that the forward left in the operator blocks: one CTA per
// chunk, warp w forms rows 16 w .. 16 w + 15 (all 64 columns) and writes them over U_c in accumulator
// order.  A_c stays as the forward wrote it.  DY is split as the backward's operator kernel splits it and
// the products run in the same order, so E_c of a closed-form chunk is the same as that kernel's.
__global__ void __launch_bounds__(kNTE)
xop_e_kernel(int T, int H, int nchunks, const float* __restrict__ dy, unsigned char* __restrict__ ops,
             size_t bstride, unsigned* __restrict__ status) {
  __shared__ __align__(128) __nv_bfloat16 sQ[2 * 64 * 32];
  __shared__ __align__(128) __nv_bfloat16 sDY[2 * kL * kLD64];
  __shared__ __align__(16) float sdy[kL * kD];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int job = blockIdx.x;
  const int ci = job % nchunks, bh = job / nchunks;
  const int bi = bh / H, hi = bh - bi * H;
  const int t0 = ci * kL, nm = min(kL, T - t0);
  const size_t base = ((size_t)bi * T * H + hi) * kD;
  const size_t tstride = (size_t)H * kD;
  unsigned char* blk = ops + ((size_t)bh * nchunks + ci) * bstride;
  if (job == 0 && tid == 0 && status != nullptr) *status = 0u;
  // Q_c (8 KB) and the chunk's dy rows (fp32, 256 bytes each) in flight together
  for (int e = tid; e < 512; e += kNTE) cp_async16(sQ + e * 8, blk + kXQ + e * 16);
  for (int e = tid; e < nm * (kD / 4); e += kNTE) {
    const int t = e >> 4, c = (e & 15) * 4;
    if (WKV7_IN(t0 + t, T, dbg::kXopPrep)) cp_async16(sdy + t * kD + c, dy + base + (size_t)(t0 + t) * tstride + c);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  const RM DYm{sDY, kL * kLD64, kLD64};
  for (int e = tid; e < kL * (kD / 4); e += kNTE) {  // split into hi + lo (rows past the chunk zero)
    const int t = e >> 4, c = (e & 15) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < nm) x = *reinterpret_cast<const float4*>(sdy + t * kD + c);
    rm_store(DYm, t, c, x.x, x.y);
    rm_store(DYm, t, c + 2, x.z, x.w);
  }
  __syncthreads();
  float acc[8][4] = {};
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const FragA fa = rm_at(DYm, warp, kk, lane);
    FragB fb[8];
#pragma unroll
    for (int np = 0; np < 4; ++np) q_b2(sQ, 2 * np, kk, lane, fb[2 * np], fb[2 * np + 1]);
    mma3n<8>(acc, fa, fb);
  }
  float4* gX = reinterpret_cast<float4*>(blk + kXX);
#pragma unroll
  for (int nj = 0; nj < 8; ++nj) gX[(warp * 8 + nj) * 32 + lane] = make_float4(acc[nj][0], acc[nj][1], acc[nj][2], acc[nj][3]);
}

}  // namespace

WKV7_DEBUG_READER(debug_word_xop)

size_t xop_workspace_bytes(int B, int T, int H, bool forward) {
  const size_t C = ((size_t)T + kL - 1) / kL;
  return kXHead + (size_t)B * H * C * (forward ? kXBytesFwd : kXBytesBwd);
}

cudaError_t launch_xop_forward(const FwdArgs& p, void* workspace, int rows, cudaStream_t stream) {
  if (p.nchunks == 0) return cudaSuccess;
  unsigned* status = static_cast<unsigned*>(workspace);
  unsigned char* ops = static_cast<unsigned char*>(workspace) + kXHead;
  cudaError_t err = p.bf16 ? launch_prep_t<__nv_bfloat16, false>(&p, nullptr, ops, kXBytesFwd, status, stream)
                           : launch_prep_t<float, false>(&p, nullptr, ops, kXBytesFwd, status, stream);
  if (err != cudaSuccess) return err;
  if (rows == 0) rows = chain_rows(p.B * p.H);
  return launch_chain<false>(rows, p.B, p.T, p.H, p.nchunks, ops, kXBytesFwd, p.h0, p.y, p.y_bf16, p.h_ckpt,
                             (size_t)kD * kD, p.hT, status, stream);
}

cudaError_t launch_xop_walk(const BwdArgs& p, void* workspace, bool from_forward, int rows, ChunkEnds* ends,
                            cudaStream_t stream) {
  unsigned* status = static_cast<unsigned*>(workspace);
  unsigned char* ops = static_cast<unsigned char*>(workspace) + kXHead;
  const size_t bstride = from_forward ? kXBytesFwd : kXBytesBwd;
  ends->g = reinterpret_cast<const float*>(ops + kXX);
  ends->flags = reinterpret_cast<int*>(ops + kXQ);  // Q_c's slot: free once the walk has run
  ends->stride = bstride / 4;
  ends->mats = from_forward ? ops + kXM : nullptr;
  if (rows == 0) rows = chain_rows(p.B * p.H);
  float* gck = reinterpret_cast<float*>(ops + kXX);
  // The walk on a forward's blocks.  With whole-head CTAs (64 rows: two chain warps per SM sub-partition)
  // the chain warps form E_c themselves, its products taking issue slots the dependent chain leaves idle
  // (measured: B2 T4096 H64 backward 54 us shorter than with the E_c kernel); with 32-row CTAs (one chain
  // warp per sub-partition) they lengthen the chain by about what the E_c kernel costs (B12 T1024 H6 1 us,
  // B4 T512 H12 4 us longer), so E_c is formed by that kernel there.  Both give the same E_c bit for bit.
  if (from_forward && rows == 64) {
    cudaError_t err = cudaMemsetAsync(status, 0, sizeof(unsigned), stream);
    if (err != cudaSuccess) return err;
    return launch_chain_t<64, true, true>(p.B, p.T, p.H, p.nchunks, ops, bstride, p.dhT, nullptr, false, gck,
                                          bstride / 4, p.dh0, p.dy, status, stream);
  }
  if (p.nchunks > 0) {  // (no chunks: the chain only copies dhT to dh0)
    cudaError_t err;
    if (from_forward) {
      xop_e_kernel<<<(unsigned)(p.B * p.H * p.nchunks), kNTE, 0, stream>>>(p.T, p.H, p.nchunks, p.dy, ops, bstride,
                                                                             status);
      err = cudaGetLastError();
    } else {
      err = p.bf16 ? launch_prep_t<__nv_bfloat16, true>(nullptr, &p, ops, bstride, status, stream)
                   : launch_prep_t<float, true>(nullptr, &p, ops, bstride, status, stream);
    }
    if (err != cudaSuccess) return err;
  }
  return launch_chain<true>(rows, p.B, p.T, p.H, p.nchunks, ops, bstride, p.dhT, nullptr, false, gck, bstride / 4,
                            p.dh0, status, stream);
}

}  // namespace wkv7
