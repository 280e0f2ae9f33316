// Tensor-core operands for the chunk kernels: warp-level bf16 mma (m16n8k16, fp32 accumulate) on
// fp32 values split as x = hi + lo (hi = x rounded to bf16, lo = the remainder rounded to bf16), so a
// product of two fp32 matrices is hi*hi + hi*lo + lo*hi (relative error ~2^-17 per product; the
// dropped lo*lo term and lo's own rounding are ~2^-18).  An operand that is already an exact bf16
// value (a bf16 input) has no lo part and takes two products.
//
// Pair tiles.  Every operand lives in shared memory as a "pair tile" array: an R x C fp32 matrix X
// (R, C multiples of 16) is cut into 16 x 16 tiles, each stored as 32 lanes x 4 words, where a word
// is the bf16 pair X[r][c], X[r][c+1] (c even).  For tile (r/16, c/16) and lane g*4 + q
// (g = r % 8, q = (c % 8) / 2) the four words are
//     w0 = (g, 2q)   w1 = (g, 2q + 8)   w2 = (g + 8, 2q)   w3 = (g + 8, 2q + 8)
// (tile-relative row, column).  hi and lo words are two separate arrays of the same shape.  One
// format serves both operands of mma.m16n8k16:
//   - as A (rows m, contraction k) of X[m][k]:  a0 = w0, a1 = w2, a2 = w1, a3 = w3;
//   - as B of a product contracting X's columns, B[k][n] = X[n][k] (i.e. "times X^T"): n-tile nt is
//     half (nt & 1) of tile row nt / 2: b0 = w[2 (nt & 1)], b1 = w[2 (nt & 1) + 1].
// A product contracting X's rows (B[k][n] = X[k][n]) takes the pair tiles of X^T instead.
// An accumulator tile (m-tile mt, n8-tile nj) holds c0, c1 = (g, 2q, 2q + 1) and c2, c3 = (g + 8, ...):
// exactly words w(nj & 1) and w(2 + (nj & 1)) of pair tile (mt, nj / 2) in the same lane, so a result
// is stored as an operand of the next product by its own lane with no shuffle.
#pragma once

#include "wkv7_debug.cuh"

#include <cuda_bf16.h>
#include <stdint.h>

namespace wkv7 {
namespace mma {

// packed bf16 pair (x in the low half) rounded to nearest
__device__ __forceinline__ uint32_t pack_bf16(float x, float y) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ float bf16_low(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_high(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// (x, y) -> hi pair, lo pair
__device__ __forceinline__ void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x, y);
  lo = pack_bf16(x - bf16_low(hi), y - bf16_high(hi));
}

// x + y of a split pair word (hi + lo), low and high element
__device__ __forceinline__ float2 join2(uint32_t hi, uint32_t lo) {
  return make_float2(bf16_low(hi) + bf16_low(lo), bf16_high(hi) + bf16_high(lo));
}

struct FragA {
  uint32_t h[4], l[4];
};
struct FragB {
  uint32_t h[2], l[2];
};

// (not volatile: the instruction only reads registers and writes its accumulator, so the compiler may
// interleave independent accumulators -- a product's three passes into one accumulator are dependent)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += A B for split A and B (small terms first)
__device__ __forceinline__ void mma3(float (&d)[4], const FragA& a, const FragB& b) {
  mma16816(d, a.l, b.h[0], b.h[1]);
  mma16816(d, a.h, b.l[0], b.l[1]);
  mma16816(d, a.h, b.h[0], b.h[1]);
}
// d += A B for an exact-bf16 A (hi only) and split B
__device__ __forceinline__ void mma2(float (&d)[4], const FragA& a, const FragB& b) {
  mma16816(d, a.h, b.l[0], b.l[1]);
  mma16816(d, a.h, b.h[0], b.h[1]);
}

// ---- pair-tile addressing: word index of element pair (r, c) (c even) in an array with `tc` tiles per
// tile row; the lo array sits `half` words after the hi array
__device__ __forceinline__ int pt_word(int r, int c, int tc) {
  const int tile = (r >> 4) * tc + (c >> 4);
  const int lane = (r & 7) * 4 + ((c & 7) >> 1);
  const int w = 2 * ((r >> 3) & 1) + ((c >> 3) & 1);
  return (tile * 32 + lane) * 4 + w;
}

// store the split pair (x at (r, c), y at (r, c + 1)) into pair tiles (hi at p, lo at p + half)
__device__ __forceinline__ void pt_store(uint32_t* p, int half, int r, int c, int tc, float x, float y) {
  uint32_t hi, lo;
  split2(x, y, hi, lo);
  const int i = pt_word(r, c, tc);
  p[i] = hi;
  p[i + half] = lo;
}
// exact-bf16 pair (hi only)
__device__ __forceinline__ void pt_store_hi(uint32_t* p, int r, int c, int tc, float x, float y) {
  p[pt_word(r, c, tc)] = pack_bf16(x, y);
}

// A operand of tile (mt, kk) for this lane
__device__ __forceinline__ FragA load_a(const uint32_t* p, int half, int tc, int mt, int kk, int lane) {
  const int i = ((mt * tc + kk) * 32 + lane) * 4;
  const uint4 h = *reinterpret_cast<const uint4*>(p + i);
  const uint4 l = *reinterpret_cast<const uint4*>(p + half + i);
  FragA a;
  a.h[0] = h.x; a.h[1] = h.z; a.h[2] = h.y; a.h[3] = h.w;
  a.l[0] = l.x; a.l[1] = l.z; a.l[2] = l.y; a.l[3] = l.w;
  return a;
}
// A operand, hi words only (exact bf16 values)
__device__ __forceinline__ FragA load_a_hi(const uint32_t* p, int tc, int mt, int kk, int lane) {
  const int i = ((mt * tc + kk) * 32 + lane) * 4;
  const uint4 h = *reinterpret_cast<const uint4*>(p + i);
  FragA a;
  a.h[0] = h.x; a.h[1] = h.z; a.h[2] = h.y; a.h[3] = h.w;
  a.l[0] = a.l[1] = a.l[2] = a.l[3] = 0u;
  return a;
}
// B operand of n-tile nt, k-tile kk (B[k][n] = X[n][k]) for this lane
__device__ __forceinline__ FragB load_b(const uint32_t* p, int half, int tc, int nt, int kk, int lane) {
  const int i = (((nt >> 1) * tc + kk) * 32 + lane) * 4 + 2 * (nt & 1);
  const uint2 h = *reinterpret_cast<const uint2*>(p + i);
  const uint2 l = *reinterpret_cast<const uint2*>(p + half + i);
  FragB b;
  b.h[0] = h.x; b.h[1] = h.y;
  b.l[0] = l.x; b.l[1] = l.y;
  return b;
}

// store accumulator tile (mt, nj) of a result into pair tiles by its own lane (see above)
__device__ __forceinline__ void store_acc(uint32_t* p, int half, int tc, int mt, int nj, int lane, const float (&c)[4]) {
  const int i = ((mt * tc + (nj >> 1)) * 32 + lane) * 4 + (nj & 1);
  uint32_t hi, lo;
  split2(c[0], c[1], hi, lo);
  p[i] = hi;
  p[i + half] = lo;
  split2(c[2], c[3], hi, lo);
  p[i + 2] = hi;
  p[i + 2 + half] = lo;
}
// the fp32 values (hi + lo) at the positions of accumulator tile (mt, nj) of this lane
__device__ __forceinline__ void load_acc_pos(const uint32_t* p, int half, int tc, int mt, int nj, int lane,
                                             float (&c)[4]) {
  const int i = ((mt * tc + (nj >> 1)) * 32 + lane) * 4 + (nj & 1);
  const float2 x = join2(p[i], p[i + half]);
  const float2 y = join2(p[i + 2], p[i + 2 + half]);
  c[0] = x.x; c[1] = x.y; c[2] = y.x; c[3] = y.y;
}

// A operand of k-tile kk built from this lane's accumulator tiles 2kk, 2kk + 1 of the same m-tile
__device__ __forceinline__ FragA frag_from_acc(const float (&c0)[4], const float (&c1)[4]) {
  FragA a;
  split2(c0[0], c0[1], a.h[0], a.l[0]);
  split2(c0[2], c0[3], a.h[1], a.l[1]);
  split2(c1[0], c1[1], a.h[2], a.l[2]);
  split2(c1[2], c1[3], a.h[3], a.l[3]);
  return a;
}

}  // namespace mma
}  // namespace wkv7

// ---------------------------------------------------------------------------------------------------
// Row-major operands read with ldmatrix.  A matrix X is stored once, row-major, as bf16 hi and lo
// arrays (lo `lo` elements after hi), `ld` elements per row (ld = 8 mod 64 -> the eight 16-byte rows of
// an 8 x 8 block fall in distinct banks).  ldmatrix hands out the mma fragments of X itself or, with
// .trans, of X^T, so one copy serves every product.
namespace wkv7 {
namespace mma {

template <bool TRANS>
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const __nv_bfloat16* p) {
  const unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(p));
  if (TRANS)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
  else
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
}

struct RM {
  __nv_bfloat16* p;  // hi array; lo array at p + lo
  int lo;
  int ld;
};

// element offset of (r, c) for an access of w elements from column c.  Rows: lo / ld (lo = 0: a hi-only
// array, rows unchecked); columns: ld - 8 (every array pads its rows by 8).  Debug builds record an
// out-of-range access and use offset 0 instead.
__device__ __forceinline__ int rm_off(const RM& x, int r, int c, int w) {
#ifdef WKV7_DEBUG_CHECKS
  const int rows = x.lo > 0 ? x.lo / x.ld : (1 << 30);
  if (!WKV7_IN(r, rows, dbg::kOperand) || !WKV7_IN(c, x.ld - 8, dbg::kOperand) ||
      !WKV7_IN(c + w - 1, x.ld - 8, dbg::kOperand))
    return 0;
#else
  (void)w;
#endif
  return r * x.ld + c;
}

// A fragment (m-tile mt, k-tile kk) of X[m][k]
__device__ __forceinline__ FragA rm_a(const RM& x, int mt, int kk, int lane) {
  const int off = rm_off(x, mt * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8, 8);
  FragA f;
  ldsm4<false>(f.h, x.p + off);
  ldsm4<false>(f.l, x.p + x.lo + off);
  return f;
}
__device__ __forceinline__ FragA rm_a_hi(const RM& x, int mt, int kk, int lane) {
  const int off = rm_off(x, mt * 16 + (lane & 15), kk * 16 + (lane >> 4) * 8, 8);
  FragA f;
  ldsm4<false>(f.h, x.p + off);
  f.l[0] = f.l[1] = f.l[2] = f.l[3] = 0u;
  return f;
}
// A fragment (mt, kk) of X^T, i.e. A[m][k] = X[k][m]
__device__ __forceinline__ FragA rm_at(const RM& x, int mt, int kk, int lane) {
  const int off = rm_off(x, kk * 16 + (lane & 7) + ((lane >> 4) << 3), mt * 16 + ((lane >> 3) & 1) * 8, 8);
  FragA f;
  ldsm4<true>(f.h, x.p + off);
  ldsm4<true>(f.l, x.p + x.lo + off);
  return f;
}
__device__ __forceinline__ FragA rm_at_hi(const RM& x, int mt, int kk, int lane) {
  const int off = rm_off(x, kk * 16 + (lane & 7) + ((lane >> 4) << 3), mt * 16 + ((lane >> 3) & 1) * 8, 8);
  FragA f;
  ldsm4<true>(f.h, x.p + off);
  f.l[0] = f.l[1] = f.l[2] = f.l[3] = 0u;
  return f;
}
// B fragments of n-tiles nt, nt + 1 at k-tile kk for B[k][n] = X[n][k] (a product "times X^T")
__device__ __forceinline__ void rm_b2(const RM& x, int nt, int kk, int lane, FragB& b0, FragB& b1, bool with_lo = true) {
  const int off = rm_off(x, nt * 8 + (lane & 7) + ((lane >> 4) << 3), kk * 16 + ((lane >> 3) & 1) * 8, 8);
  uint32_t h[4], l[4] = {0u, 0u, 0u, 0u};
  ldsm4<false>(h, x.p + off);
  if (with_lo) ldsm4<false>(l, x.p + x.lo + off);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}
// B fragments of n-tiles nt, nt + 1 at k-tile kk for B[k][n] = X[k][n] (a product "times X")
__device__ __forceinline__ void rm_bt2(const RM& x, int nt, int kk, int lane, FragB& b0, FragB& b1, bool with_lo = true) {
  const int off = rm_off(x, kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, nt * 8 + (lane >> 4) * 8, 8);
  uint32_t h[4], l[4] = {0u, 0u, 0u, 0u};
  ldsm4<true>(h, x.p + off);
  if (with_lo) ldsm4<true>(l, x.p + x.lo + off);
  b0.h[0] = h[0]; b0.h[1] = h[1]; b1.h[0] = h[2]; b1.h[1] = h[3];
  b0.l[0] = l[0]; b0.l[1] = l[1]; b1.l[0] = l[2]; b1.l[1] = l[3];
}
// split pair (x at (r, c), y at (r, c + 1)), c even
__device__ __forceinline__ void rm_store(const RM& x, int r, int c, float a, float b) {
  uint32_t hi, lo;
  split2(a, b, hi, lo);
  const int off = rm_off(x, r, c, 2);
  *reinterpret_cast<uint32_t*>(x.p + off) = hi;
  *reinterpret_cast<uint32_t*>(x.p + x.lo + off) = lo;
}
__device__ __forceinline__ void rm_store_hi(const RM& x, int r, int c, float a, float b) {
  *reinterpret_cast<uint32_t*>(x.p + rm_off(x, r, c, 2)) = pack_bf16(a, b);
}
// accumulator tile (mt, nj) of a result into X
__device__ __forceinline__ void rm_store_acc(const RM& x, int mt, int nj, int lane, const float (&c)[4]) {
  const int r = mt * 16 + (lane >> 2), col = nj * 8 + 2 * (lane & 3);
  rm_store(x, r, col, c[0], c[1]);
  rm_store(x, r + 8, col, c[2], c[3]);
}
// 8 split values to row r, columns c..c+7 (c a multiple of 8): two 16-byte stores
__device__ __forceinline__ void rm_store8(const RM& x, int r, int c, const float (&v)[8]) {
  uint4 h, l;
  split2(v[0], v[1], h.x, l.x);
  split2(v[2], v[3], h.y, l.y);
  split2(v[4], v[5], h.z, l.z);
  split2(v[6], v[7], h.w, l.w);
  const int off = rm_off(x, r, c, 8);
  *reinterpret_cast<uint4*>(x.p + off) = h;
  *reinterpret_cast<uint4*>(x.p + x.lo + off) = l;
}
// fp32 values (hi + lo) at (r, c), (r, c + 1)
__device__ __forceinline__ float2 rm_get2(const RM& x, int r, int c) {
  const int off = rm_off(x, r, c, 2);
  return join2(*reinterpret_cast<const uint32_t*>(x.p + off), *reinterpret_cast<const uint32_t*>(x.p + x.lo + off));
}
// fp32 value (hi + lo) at (r, c)
__device__ __forceinline__ float rm_get1(const RM& x, int r, int c) {
  const int off = rm_off(x, r, c, 1);
  return __bfloat162float(x.p[off]) + __bfloat162float(x.p[x.lo + off]);
}
// 8 values to row r, columns c..c+7 of an exact-bf16 operand (hi only): one 16-byte store
__device__ __forceinline__ void rm_store8_hi(const RM& x, int r, int c, const float (&v)[8]) {
  uint4 h;
  h.x = pack_bf16(v[0], v[1]);
  h.y = pack_bf16(v[2], v[3]);
  h.z = pack_bf16(v[4], v[5]);
  h.w = pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4*>(x.p + rm_off(x, r, c, 8)) = h;
}
// d[i] += A B[i] for split A and B, i < N: the three bf16 passes each over all N accumulators, so that
// dependent mma into one accumulator are N instructions apart
template <int N>
__device__ __forceinline__ void mma3n(float (&d)[N][4], const FragA& a, const FragB (&b)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) mma16816(d[i], a.l, b[i].h[0], b[i].h[1]);
#pragma unroll
  for (int i = 0; i < N; ++i) mma16816(d[i], a.h, b[i].l[0], b[i].l[1]);
#pragma unroll
  for (int i = 0; i < N; ++i) mma16816(d[i], a.h, b[i].h[0], b[i].h[1]);
}
// ... for an exact-bf16 A (hi only)
template <int N>
__device__ __forceinline__ void mma2n(float (&d)[N][4], const FragA& a, const FragB (&b)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) mma16816(d[i], a.h, b[i].l[0], b[i].l[1]);
#pragma unroll
  for (int i = 0; i < N; ++i) mma16816(d[i], a.h, b[i].h[0], b[i].h[1]);
}
// two products at once, d0[i] += A0 B0[i] and d1[i] += A1 B1[i] (all split), pass by pass over both
template <int N>
__device__ __forceinline__ void mma3n_two(float (&d0)[N][4], const FragA& a0, const FragB (&b0)[N], float (&d1)[N][4],
                                          const FragA& a1, const FragB (&b1)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.l, b0[i].h[0], b0[i].h[1]);
    mma16816(d1[i], a1.l, b1[i].h[0], b1[i].h[1]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.h, b0[i].l[0], b0[i].l[1]);
    mma16816(d1[i], a1.h, b1[i].l[0], b1[i].l[1]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.h, b0[i].h[0], b0[i].h[1]);
    mma16816(d1[i], a1.h, b1[i].h[0], b1[i].h[1]);
  }
}
// ... with exact-bf16 A0, A1 (hi only) and a split B shared by both: d0[i] += A0 B[i], d1[i] += A1 B[i]
template <int N>
__device__ __forceinline__ void mma2n_two(float (&d0)[N][4], const FragA& a0, float (&d1)[N][4], const FragA& a1,
                                          const FragB (&b)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.h, b[i].l[0], b[i].l[1]);
    mma16816(d1[i], a1.h, b[i].l[0], b[i].l[1]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.h, b[i].h[0], b[i].h[1]);
    mma16816(d1[i], a1.h, b[i].h[0], b[i].h[1]);
  }
}
// ... with an exact-bf16 B (hi only) shared by both: d0[i] += A0 B[i], d1[i] += A1 B[i]
template <int N>
__device__ __forceinline__ void mma2b_two(float (&d0)[N][4], const FragA& a0, float (&d1)[N][4], const FragA& a1,
                                          const FragB (&b)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.l, b[i].h[0], b[i].h[1]);
    mma16816(d1[i], a1.l, b[i].h[0], b[i].h[1]);
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mma16816(d0[i], a0.h, b[i].h[0], b[i].h[1]);
    mma16816(d1[i], a1.h, b[i].h[0], b[i].h[1]);
  }
}
// The off-diagonal block of T = (I - M)^-1 for a strictly lower 32 x 32 M (fp32, row stride sm) once the
// diagonal blocks T11, T22 are in TI (fp32, stride sm): T21 = T22 M21 T11, formed by one warp on tensor
// cores in transposed form (E^T = T11^T M21^T, then T21^T = E^T T22^T) and written into TI rows 16-31,
// columns 0-15.  Every lane of the warp calls it.
__device__ __forceinline__ void tri_inverse_t21(const float* M, float* TI, int sm, int lane) {
  const int g = lane >> 2, q = lane & 3;
  auto ld2 = [&](const float* p0, const float* p1, uint32_t& hw, uint32_t& lw) { split2(*p0, *p1, hw, lw); };
  FragA fa;  // T11^T: A[s][u] = T11[u][s]
  ld2(TI + (2 * q) * sm + g, TI + (2 * q + 1) * sm + g, fa.h[0], fa.l[0]);
  ld2(TI + (2 * q) * sm + g + 8, TI + (2 * q + 1) * sm + g + 8, fa.h[1], fa.l[1]);
  ld2(TI + (2 * q + 8) * sm + g, TI + (2 * q + 9) * sm + g, fa.h[2], fa.l[2]);
  ld2(TI + (2 * q + 8) * sm + g + 8, TI + (2 * q + 9) * sm + g + 8, fa.h[3], fa.l[3]);
  FragB fb[2];  // M21^T: B[u][t] = M[16 + t][u]
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float* row = M + (16 + nt * 8 + g) * sm;
    ld2(row + 2 * q, row + 2 * q + 1, fb[nt].h[0], fb[nt].l[0]);
    ld2(row + 2 * q + 8, row + 2 * q + 9, fb[nt].h[1], fb[nt].l[1]);
  }
  float et[2][4] = {};
  mma3n<2>(et, fa, fb);
  const FragA fe = frag_from_acc(et[0], et[1]);  // E^T as an A operand (rows s, k = t')
  FragB fc[2];  // T22^T: B[t'][t] = T22[t][t']
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float* row = TI + (16 + nt * 8 + g) * sm + 16;
    ld2(row + 2 * q, row + 2 * q + 1, fc[nt].h[0], fc[nt].l[0]);
    ld2(row + 2 * q + 8, row + 2 * q + 9, fc[nt].h[1], fc[nt].l[1]);
  }
  float tt[2][4] = {};
  mma3n<2>(tt, fe, fc);
  __syncwarp();
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {  // T21[t][s] from T21^T (rows s = g, g + 8; columns t = 8 nt + 2q, + 1)
    const int t = nt * 8 + 2 * q;
    TI[(16 + t) * sm + g] = tt[nt][0];
    TI[(17 + t) * sm + g] = tt[nt][1];
    TI[(16 + t) * sm + g + 8] = tt[nt][2];
    TI[(17 + t) * sm + g + 8] = tt[nt][3];
  }
}

// index (floats) of element (i, j) of a 64 x 64 fp32 matrix stored in mma accumulator order:
// [m-tile i / 16][n-tile j / 8][lane][4], lane = 4 (i % 8) + (j % 8) / 2, slot 2 ((i % 16) / 8) + j % 2
// (the order in which a warp's m16n8 accumulators leave or enter registers as one float4 per lane)
__host__ __device__ __forceinline__ int acc_order(int i, int j) {
  const int r = i & 15, c = j & 7;
  const int lane = (r & 7) * 4 + (c >> 1);
  const int e = (r >> 3) * 2 + (c & 1);
  return ((((i >> 4) * 8 + (j >> 3)) * 32 + lane) << 2) + e;
}

// d += A B for split A and an exact-bf16 B (hi only)
__device__ __forceinline__ void mma2b(float (&d)[4], const FragA& a, const FragB& b) {
  mma16816(d, a.l, b.h[0], b.h[1]);
  mma16816(d, a.h, b.h[0], b.h[1]);
}

}  // namespace mma
}  // namespace wkv7
