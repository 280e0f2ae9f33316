// Device helpers shared by the WKV7 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wkv7_debug.cuh"

namespace wkv7 {

constexpr int kD = 64;  // head size: the state is kD x kD fp32

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 pattern.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 consecutive inputs (16-byte aligned) as fp32, through the read-only path.
__device__ __forceinline__ void load8(const float* __restrict__ p, float (&o)[8]) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  const float4 y = __ldg(reinterpret_cast<const float4*>(p) + 1);
  o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
  o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* __restrict__ p, float (&o)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  o[0] = bf16_lo(u.x); o[1] = bf16_hi(u.x); o[2] = bf16_lo(u.y); o[3] = bf16_hi(u.y);
  o[4] = bf16_lo(u.z); o[5] = bf16_hi(u.z); o[6] = bf16_lo(u.w); o[7] = bf16_hi(u.w);
}

// 4 consecutive inputs (8-byte aligned for bf16, 16-byte for fp32) as fp32.
__device__ __forceinline__ float4 load4(const float* __restrict__ p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* __restrict__ p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

__device__ __forceinline__ void store8(float* p, const float (&o)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// ---- cp.async (16-byte pieces, global -> shared, bypassing L1)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// 8 values already in shared memory (16-byte aligned, input dtype) -> fp32
__device__ __forceinline__ void raw8(const float* p, float (&o)[8]) {
  const float4 x = reinterpret_cast<const float4*>(p)[0];
  const float4 y = reinterpret_cast<const float4*>(p)[1];
  o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
}
__device__ __forceinline__ void raw8(const __nv_bfloat16* p, float (&o)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  o[0] = bf16_lo(u.x); o[1] = bf16_hi(u.x); o[2] = bf16_lo(u.y); o[3] = bf16_hi(u.y);
  o[4] = bf16_lo(u.z); o[5] = bf16_hi(u.z); o[6] = bf16_lo(u.w); o[7] = bf16_hi(u.w);
}

__device__ __forceinline__ float2 lo2(float4 x) { return make_float2(x.x, x.y); }
__device__ __forceinline__ float2 hi2(float4 x) { return make_float2(x.z, x.w); }

// ---- row sums over the 16 lanes of a row group, each lane holding partials of 4 rows.
// Reduce-scatter: after 5 shuffles lane l (l16 = lane % 16) holds the full sum of row
// rs_row(l16) = 2*bit3 + bit2.  all_gather4 then hands every lane all four sums.
__device__ __forceinline__ int rs_row(int l16) { return ((l16 >> 3) & 1) * 2 + ((l16 >> 2) & 1); }

__device__ __forceinline__ float reduce_scatter4(const float (&x)[4], int l16) {
  const bool b3 = (l16 & 8) != 0, b2 = (l16 & 4) != 0;
  float k0 = b3 ? x[2] : x[0], k1 = b3 ? x[3] : x[1];
  const float s0 = b3 ? x[0] : x[2], s1 = b3 ? x[1] : x[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 8);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 8);
  float k = b2 ? k1 : k0;
  const float s = b2 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, s, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

__device__ __forceinline__ void all_gather4(float z, int l16, float (&out)[4]) {
  const int q = rs_row(l16);
  const float o = __shfl_xor_sync(0xffffffffu, z, 4);
  const float e0 = (q & 1) ? o : z;
  const float e1 = (q & 1) ? z : o;
  const float f0 = __shfl_xor_sync(0xffffffffu, e0, 8);
  const float f1 = __shfl_xor_sync(0xffffffffu, e1, 8);
  const bool hi = (q & 2) != 0;
  out[0] = hi ? f0 : e0;
  out[1] = hi ? f1 : e1;
  out[2] = hi ? e0 : f0;
  out[3] = hi ? e1 : f1;
}

// all-reduce of 4 rows over 16 lanes as a 4-level butterfly: more shuffles than
// reduce-scatter + all-gather but only 4 dependent steps (used on serial chains)
__device__ __forceinline__ void butterfly4(float (&x)[4]) {
#pragma unroll
  for (int m = 1; m < 16; m <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], m);
}

// ---- thread-block clusters: rank, split barrier, peer shared-memory stores
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// shared::cluster address of `p` (a shared-memory variable of this CTA) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_smem(const void* p, unsigned rank) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(s), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float2 bcast2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// 4 consecutive values already in shared memory (input dtype) -> fp32
__device__ __forceinline__ float4 raw4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 raw4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

// ---- sums over all 32 lanes of NV per-lane values (NV a power of two, 2 <= NV <= 32).
// Reduce-scatter: each level halves the values a lane keeps (it keeps the half selected by its
// lane bit, adds the partner's copy of that half); once one value is left the remaining levels
// are a plain butterfly.  Afterwards lane l holds the full sum of value index rs32_index<NV>(l).
template <int NV>
__device__ __forceinline__ int rs32_index(int lane) {
  int idx = 0, n = NV, mask = 16;
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    if (n > 1) {
      n >>= 1;
      if (lane & mask) idx += n;
    }
    mask >>= 1;
  }
  return idx;
}

template <int NV>
__device__ __forceinline__ float rs32(const float (&x)[NV], int lane) {
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = x[i];
  int n = NV;
#pragma unroll
  for (int mask = 16; mask >= 1; mask >>= 1) {
    if (n > 1) {
      const int h = n >> 1;
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int m = 0; m < NV / 2; ++m) {
        if (m < h) {
          const float keep = up ? v[h + m] : v[m];
          const float send = up ? v[m] : v[h + m];
          v[m] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
    }
  }
  return v[0];
}

// After rs32<2*NP>: lanes with lane bit 16 clear hold the first NP sums (index rs32_index).
// Hand every lane all NP of them.
template <int NP>
__device__ __forceinline__ void ag32_low(float u, int lane, float (&out)[NP]) {
  static_assert(NP == 2 || NP == 4 || NP == 8, "2, 4 or 8 values");
  const float t = __shfl_xor_sync(0xffffffffu, u, 16);
  float g[NP];
  g[0] = (lane & 16) ? t : u;  // value index = rs32_index<2*NP>(lane) with the top bit dropped
  // index bits of the remaining levels, lowest weight first: lane masks 16/NP ... 8
  int have = 1;
#pragma unroll
  for (int wgt = 1; wgt < NP; wgt <<= 1) {
    const int mask = 16 / (2 * NP) * 2 * wgt;  // lane mask carrying index weight `wgt`
    const bool up = (lane & mask) != 0;
    float o[NP / 2];
#pragma unroll
    for (int m = 0; m < NP / 2; ++m)
      if (m < have) o[m] = __shfl_xor_sync(0xffffffffu, g[m], mask);
#pragma unroll
    for (int m = NP / 2 - 1; m >= 0; --m) {
      if (m < have) {
        const float mine = g[m];
        g[m] = up ? o[m] : mine;
        g[have + m] = up ? mine : o[m];
      }
    }
    have <<= 1;
  }
#pragma unroll
  for (int i = 0; i < NP; ++i) out[i] = g[i];
}

// 4-wide dot products of 4 state rows with one float4 (two packed fp32x2 FMAs each)
__device__ __forceinline__ void dot4x4(const float2 (&S)[4][2], float4 c, float (&out)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p2 = __ffma2_rn(S[i][1], hi2(c), __fmul2_rn(S[i][0], lo2(c)));
    out[i] = p2.x + p2.y;
  }
}

// The same for R rows (R = 2 or 4)
template <int R>
__device__ __forceinline__ void dot_rows(const float2 (&S)[R][2], float4 c, float (&out)[R]) {
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const float2 p2 = __ffma2_rn(S[i][1], hi2(c), __fmul2_rn(S[i][0], lo2(c)));
    out[i] = p2.x + p2.y;
  }
}

// ---- row sums over the 16 lanes of a row group for R rows per lane (R = 2 or 4).
// rs16<R>: reduce-scatter (halving levels, then a plain butterfly); lane l16 ends with the
// full sum of row rs16_row<R>(l16); for R = 4 this is reduce_scatter4 / rs_row exactly.
// Every lane with l16 % (16/R) == 0 holds a distinct row.
template <int R>
__device__ __forceinline__ int rs16_row(int l16) {
  return R == 4 ? rs_row(l16) : ((l16 >> 3) & 1);
}

template <int R>
__device__ __forceinline__ float rs16(const float (&x)[R], int l16) {
  static_assert(R == 2 || R == 4, "2 or 4 rows");
  if constexpr (R == 4) {
    return reduce_scatter4(x, l16);
  } else {
    const bool b3 = (l16 & 8) != 0;
    float k = b3 ? x[1] : x[0];
    const float s = b3 ? x[0] : x[1];
    k += __shfl_xor_sync(0xffffffffu, s, 8);
    k += __shfl_xor_sync(0xffffffffu, k, 4);
    k += __shfl_xor_sync(0xffffffffu, k, 2);
    k += __shfl_xor_sync(0xffffffffu, k, 1);
    return k;
  }
}

// all-reduce of R rows over 16 lanes, 4 dependent levels (R = 4: butterfly4 exactly)
template <int R>
__device__ __forceinline__ void butterfly16(float (&x)[R]) {
#pragma unroll
  for (int m = 1; m < 16; m <<= 1)
#pragma unroll
    for (int i = 0; i < R; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], m);
}

}  // namespace wkv7
