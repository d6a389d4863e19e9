// Element-wise pieces of the backward kernels (fa_bwd.cu, fa_bwd_pair.cu,
// fa_bwd256.cu): recomputing the softmax weights P (section 7.1 of
// "FlashAttention V2 in depth") from the saved logsumexp over 64 columns
// held in registers, reading an fp32 accumulator out of tensor memory as
// packed bf16, and where a 128-column tile's packed bf16 lands in TMEM.
#pragma once

#include "sm103_primitives.cuh"

namespace fa {

using namespace dev;

// Packed column of the 16 columns [16 kk, 16 kk + 16) of a bf16 tile written
// by the element-wise warps of the 128-column kernels: warp half h holds
// columns [64 h, 64 h + 64) as bf16 pairs in [64 h, 64 h + 32) of its region
// (second = true: in [64 h + 32, 64 h + 64)).
__device__ __forceinline__ uint32_t packed_col(int kk, bool second) {
  return 64u * (kk >> 2) + (second ? 32u : 0u) + 8u * (kk & 3);
}

// Rows of 32 consecutive TMEM columns, NC columns from `taddr`, scaled and
// packed to bf16 pairs into w[NC / 2].
template <int NC>
__device__ __forceinline__ void tmem_read_pack(uint32_t taddr, float sc, uint32_t* w) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(taddr + 32 * c, a);
    tmem_ld_wait<32>(a);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[16 * c + i] = pack_bf16(__uint_as_float(a[2 * i]) * sc, __uint_as_float(a[2 * i + 1]) * sc);
  }
}

// P^T of 64 query columns [q_first, q_first + 64) of key row kr, in place:
// p = exp2(s * sl2 - L_q) with L per column.  MASK zeroes the weights the
// causal mask hides (kr > query; the caller passes the key row less the
// causal offset) and those of a key row past Nk (dead).
template <bool MASK>
__device__ __forceinline__ void p64_colL(uint32_t* s, const float* bl, float sl2, int kr, int q_first, bool dead,
                                         bool causal) {
#pragma unroll
  for (int e4 = 0; e4 < 16; ++e4) {
    const float4 l4 = reinterpret_cast<const float4*>(bl)[e4];
    const float2 a01 = __ffma2_rn(make_float2(__uint_as_float(s[4 * e4]), __uint_as_float(s[4 * e4 + 1])),
                                  make_float2(sl2, sl2), make_float2(-l4.x, -l4.y));
    const float2 a23 = __ffma2_rn(make_float2(__uint_as_float(s[4 * e4 + 2]), __uint_as_float(s[4 * e4 + 3])),
                                  make_float2(sl2, sl2), make_float2(-l4.z, -l4.w));
    float p0 = ex2_approx(a01.x), p1 = ex2_approx(a01.y), p2 = ex2_approx(a23.x), p3 = ex2_approx(a23.y);
    if (MASK) {
      const int col = q_first + 4 * e4;
      p0 = (dead || (causal && kr > col)) ? 0.f : p0;
      p1 = (dead || (causal && kr > col + 1)) ? 0.f : p1;
      p2 = (dead || (causal && kr > col + 2)) ? 0.f : p2;
      p3 = (dead || (causal && kr > col + 3)) ? 0.f : p3;
    }
    s[4 * e4] = __float_as_uint(p0);
    s[4 * e4 + 1] = __float_as_uint(p1);
    s[4 * e4 + 2] = __float_as_uint(p2);
    s[4 * e4 + 3] = __float_as_uint(p3);
  }
}

// P of 64 key columns [k_first, k_first + 64) of query row q, in place:
// p = exp2(s * sl2 - L) with one L for the row.  MASK zeroes keys past N and,
// with the causal mask, keys after q (the caller passes the query row plus
// the causal offset).
template <bool MASK>
__device__ __forceinline__ void p64_rowL(uint32_t* s, float L, float sl2, int q, int k_first, int N, bool causal) {
  const float2 sv = make_float2(sl2, sl2);
  const float2 lv = make_float2(-L, -L);
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const float2 a = __ffma2_rn(make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sv, lv);
    float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
    if (MASK) {
      const int k = k_first + e;
      p0 = (k >= N || (causal && k > q)) ? 0.f : p0;
      p1 = (k + 1 >= N || (causal && k + 1 > q)) ? 0.f : p1;
    }
    s[e] = __float_as_uint(p0);
    s[e + 1] = __float_as_uint(p1);
  }
}

}  // namespace fa
