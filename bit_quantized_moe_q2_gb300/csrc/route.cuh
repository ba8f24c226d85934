// Router building blocks shared by the routing kernels and the fused
// single-token layer kernel: error-free transforms, the per-expert Dot2
// logit of a 256-thread CTA, the ranking key and the warp top-k / softmax.
#pragma once

#include "internal.cuh"

namespace ds4 {

// ------------------------------------------------------------------- router
// Error-free transforms (Ogita, Rump, Oishi, "Accurate sum and dot product",
// SIAM J. Sci. Comput. 26(6), 2005): TwoProduct via FMA and Knuth's TwoSum.
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
  p = __fmul_rn(a, b);
  e = fmaf(a, b, -p);
}
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Dot2 partial of x . Wr_e for one 256-thread group (thread tid < 256 of
// the group holds the router row's float4 slices j = 4 (tid + 256 i) in
// wv, and the matching four bf16 values of x in xv[i]): four compensated
// chains per thread, merged with TwoSum, then across the warp; lane 0
// leaves the warp's (sum, error) in (ps, pc).
template <int NI>
__device__ __forceinline__ void route_dot2_regs(const uint2 (&xin)[NI], const float4 (&wv)[NI], int D, int tid,
                                                float &ps, float &pc) {
  const int lane = threadIdx.x & 31;
  float s4[4] = {0.f, 0.f, 0.f, 0.f}, c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = 4 * (tid + 256 * i);
    if (j < D) {
      const uint2 xv = xin[i];
      const float xs[4] = {bf16_bits_to_f32(xv.x & 0xFFFFu), bf16_bits_to_f32(xv.x >> 16),
                           bf16_bits_to_f32(xv.y & 0xFFFFu), bf16_bits_to_f32(xv.y >> 16)};
      const float ws4[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float p, pe, se;
        two_prod(xs[q], ws4[q], p, pe);
        two_sum(s4[q], p, s4[q], se);
        c4[q] = __fadd_rn(c4[q], __fadd_rn(pe, se));
      }
    }
  }
  float s = s4[0], c = __fadd_rn(c4[0], __fadd_rn(c4[1], __fadd_rn(c4[2], c4[3])));
#pragma unroll
  for (int q = 1; q < 4; ++q) {
    float se;
    two_sum(s, s4[q], s, se);
    c = __fadd_rn(c, se);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float so = __shfl_xor_sync(0xffffffffu, s, off);
    const float co = __shfl_xor_sync(0xffffffffu, c, off);
    float se;
    two_sum(s, so, s, se);
    c = __fadd_rn(c, __fadd_rn(co, se));
  }
  if (lane == 0) {
    ps = s;
    pc = c;
  }
}

// The partial above with x read from global memory (row xr).
template <int NI>
__device__ __forceinline__ void route_dot2_partial(const uint16_t *__restrict__ xr, const float4 (&wv)[NI], int D,
                                                   int tid, float &ps, float &pc) {
  uint2 xv[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = 4 * (tid + 256 * i);
    xv[i] = j < D ? __ldcg(reinterpret_cast<const uint2 *>(xr + j)) : make_uint2(0u, 0u);
  }
  route_dot2_regs<NI>(xv, wv, D, tid, ps, pc);
}

// The same partial for NT consecutive tokens (row stride D) at once: every
// token's arithmetic is exactly route_dot2_partial's, in the same order, but
// the NT independent load / reduction chains overlap (a CTA ranks a batch of
// tokens an NT-th of the latency apart).
template <int NI, int NT>
__device__ __forceinline__ void route_dot2_partial_n(const uint16_t *__restrict__ xr, int64_t stride,
                                                     const float4 (&wv)[NI], int D, int tid, float *ps,
                                                     float *pc) {
  const int lane = threadIdx.x & 31;
  float s4[NT][4], c4[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) s4[t][q] = c4[t][q] = 0.f;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = 4 * (tid + 256 * i);
    if (j < D) {
      uint2 xv[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) xv[t] = __ldcg(reinterpret_cast<const uint2 *>(xr + t * stride + j));
      const float ws4[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float xs[4] = {bf16_bits_to_f32(xv[t].x & 0xFFFFu), bf16_bits_to_f32(xv[t].x >> 16),
                             bf16_bits_to_f32(xv[t].y & 0xFFFFu), bf16_bits_to_f32(xv[t].y >> 16)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float p, pe, se;
          two_prod(xs[q], ws4[q], p, pe);
          two_sum(s4[t][q], p, s4[t][q], se);
          c4[t][q] = __fadd_rn(c4[t][q], __fadd_rn(pe, se));
        }
      }
    }
  }
  float s[NT], c[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    s[t] = s4[t][0];
    c[t] = __fadd_rn(c4[t][0], __fadd_rn(c4[t][1], __fadd_rn(c4[t][2], c4[t][3])));
#pragma unroll
    for (int q = 1; q < 4; ++q) {
      float se;
      two_sum(s[t], s4[t][q], s[t], se);
      c[t] = __fadd_rn(c[t], se);
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float so = __shfl_xor_sync(0xffffffffu, s[t], off);
      const float co = __shfl_xor_sync(0xffffffffu, c[t], off);
      float se;
      two_sum(s[t], so, s[t], se);
      c[t] = __fadd_rn(c[t], __fadd_rn(co, se));
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      ps[t] = s[t];
      pc[t] = c[t];
    }
  }
}

// Merge of the eight warp partials of column `col` (+ bias), rounded once.
__device__ __forceinline__ float route_dot2_merge(const float (*ps)[32], const float (*pc)[32], int col,
                                                  const float *bias_e) {
  float s = ps[0][col], c = pc[0][col];
  for (int ww = 1; ww < 8; ++ww) {
    float se;
    two_sum(s, ps[ww][col], s, se);
    c = __fadd_rn(c, __fadd_rn(pc[ww][col], se));
  }
  if (bias_e) {
    float se;
    two_sum(s, *bias_e, s, se);
    c = __fadd_rn(c, se);
  }
  return __fadd_rn(s, c);
}

// Ranking key of (logit, expert): a larger key ranks first.  The logit maps
// monotonically onto 32 bits with NaN lowest (below -inf) and -0 == +0; ties
// go to the lower expert id.
__device__ __forceinline__ uint64_t rank_key(float v, int e) {
  const uint32_t u = __float_as_uint(v) == 0x80000000u ? 0u : __float_as_uint(v);
  const uint32_t o = isnan(v) ? 0u : (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)o << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  const uint32_t o = (uint32_t)(key >> 32);
  if (o == 0u) return __uint_as_float(0x7FC00000u);  // NaN
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Top-k of one token's E <= 256 logits held in registers by one warp (entry
// lane + 32 j in v[j]): lane i < k receives the i-th selected (logit, id).
// k rounds of a warp-wide maximum of the ranking keys: the maximum of the
// high (logit) halves, then of the low (id) halves among the lanes holding
// that logit, each one warp reduction.
__device__ __forceinline__ void topk_select_warp(const float (&v)[8], int E, int k, float &my_v, int &my_e) {
  const int lane = threadIdx.x & 31;
  uint64_t key[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) key[j] = lane + 32 * j < E ? rank_key(v[j], lane + 32 * j) : 0ull;
  my_v = 0.f;
  my_e = -1;
  for (int i = 0; i < k; ++i) {
    uint64_t lb = key[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) lb = key[j] > lb ? key[j] : lb;
    const uint32_t bh = __reduce_max_sync(0xffffffffu, (uint32_t)(lb >> 32));
    const uint32_t bl = __reduce_max_sync(0xffffffffu, (uint32_t)(lb >> 32) == bh ? (uint32_t)lb : 0u);
    const uint64_t best = ((uint64_t)bh << 32) | bl;
    const int be = (int)(0xFFFFFFFFu - bl);
    if ((be & 31) == lane) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == (be >> 5)) key[j] = 0ull;
    }
    if (lane == i) {
      my_v = key_value(best);
      my_e = be;
    }
  }
}

// Softmax over the k selected logits (lane i < k holds the i-th): in
// double, summed in rank order, rounded once to fp32.
__device__ __forceinline__ float softmax_selected_warp(float my_v, int k) {
  const int lane = threadIdx.x & 31;
  const double m = (double)__shfl_sync(0xffffffffu, my_v, 0);
  const double ex = lane < k ? exp((double)my_v - m) : 0.0;
  double sum = 0.0;
  for (int i = 0; i < k; ++i) sum += __shfl_sync(0xffffffffu, ex, i);
  return (float)(ex / sum);
}

}  // namespace ds4
