// C-ABI entry points of libds4moe plus the small kernels of the hot path:
// block dequantisation, the router (compensated dot product), top-k with a
// softmax over the selected experts, token->expert bucketing and the
// weighted combine.  The expert GEMV/GEMM kernels live in ffn_decode.cu and
// ffn_prefill.cu.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "route.cuh"
#include "span.cuh"

using namespace ds4;

namespace ds4 {

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

cudaError_t span_control_abi(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline bool qtype_ok(int q) { return q == DS4MOE_Q4_1 || q == DS4MOE_Q2_K || q == DS4MOE_Q4_K; }

ds4moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DS4MOE_OK;
  fprintf(stderr, "ds4moe: CUDA error %s\n", cudaGetErrorString(e));
  return DS4MOE_ECUDA;
}

// ------------------------------------------------------------------ dequant
// Q4_1 ([Q41] "Q4_1 블록이 어떻게 생겼나"): one thread per (block, byte j);
// writes values j (low nibble) and j+16 (high nibble) as fmaf(d, q, m): d*q is
// exact in fp32, so this is the single rounding of d*q + m.
__global__ void k_dequant_q41(const uint8_t *__restrict__ blk, int64_t nb, float *__restrict__ out) {
  const int64_t n = nb * 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i >> 4;
    const int j = (int)(i & 15);
    const uint8_t *p = blk + b * kQ41Bytes;
    const float d = f16_bits_to_f32(p[0] | (p[1] << 8));
    const float m = f16_bits_to_f32(p[2] | (p[3] << 8));
    const uint32_t q = p[4 + j];
    out[b * 32 + j] = fmaf(d, (float)(q & 15u), m);
    out[b * 32 + j + 16] = fmaf(d, (float)(q >> 4), m);
  }
}

// Q2_K ([DS4-2] layout table and qs packing): one thread per (block, qs byte);
// qs byte 32h + l carries values 128h + l + 32s in bits 2s..2s+1.  d*sc and
// dmin*mn are exact, so fmaf(d*sc, q, -dmin*mn) is the single rounding.
__global__ void k_dequant_q2k(const uint8_t *__restrict__ blk, int64_t nb, float *__restrict__ out) {
  const int64_t n = nb * 64;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i >> 6;
    const int byte = (int)(i & 63), h = byte >> 5, l = byte & 31;
    const uint8_t *p = blk + b * kQ2KBytes;
    const float d = f16_bits_to_f32(p[80] | (p[81] << 8));
    const float dmin = f16_bits_to_f32(p[82] | (p[83] << 8));
    const uint32_t q = p[16 + byte];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int v = 128 * h + l + 32 * s;
      const uint32_t scb = p[v >> 4];
      out[b * 256 + v] = fmaf(d * (float)(scb & 15u), (float)((q >> (2 * s)) & 3u), -(dmin * (float)(scb >> 4)));
    }
  }
}

// Q4_K (standard k-quant reading of the 144-byte block): one thread per
// (block, qs byte); qs byte 32c + l carries value 64c + l (low nibble, sub-
// block 2c) and 64c + 32 + l (high nibble, sub-block 2c + 1).  d*sc and
// dmin*mn are exact, so fmaf(d*sc, q, -dmin*mn) is the single rounding.
__global__ void k_dequant_q4k(const uint8_t *__restrict__ blk, int64_t nb, float *__restrict__ out) {
  const int64_t n = nb * 128;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i >> 7;
    const int byte = (int)(i & 127), c = byte >> 5, l = byte & 31;
    const uint8_t *p = blk + b * kQ4KBytes;
    const float d = f16_bits_to_f32(p[0] | (p[1] << 8));
    const float dmin = f16_bits_to_f32(p[2] | (p[3] << 8));
    const uint32_t q = p[16 + byte];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t sc, mn;
      q4k_scale_min(p + 4, 2 * c + hh, sc, mn);
      out[b * 256 + 64 * c + 32 * hh + l] =
          fmaf(d * (float)sc, (float)((q >> (4 * hh)) & 15u), -(dmin * (float)mn));
    }
  }
}

// ------------------------------------------------------------------- router
// One warp computes x_t . Wr_e (+ bias) with Dot2: lanes own interleaved
// float4 slices, the (sum, error) pairs are merged across lanes with TwoSum,
// the bias is added with TwoSum, and the result is rounded once.  Every lane
// returns the same value.
__device__ __forceinline__ float dot2_row_warp(const uint16_t *__restrict__ xr, const float *__restrict__ wr, int D,
                                               const float *bias_e) {
  const int lane = threadIdx.x & 31;
  float s = 0.f, c = 0.f;
  for (int j = 4 * lane; j < D; j += 128) {
    const float4 wv = *reinterpret_cast<const float4 *>(wr + j);
    const uint2 xv = *reinterpret_cast<const uint2 *>(xr + j);
    const float xs[4] = {bf16_bits_to_f32(xv.x & 0xFFFFu), bf16_bits_to_f32(xv.x >> 16),
                         bf16_bits_to_f32(xv.y & 0xFFFFu), bf16_bits_to_f32(xv.y >> 16)};
    const float ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float p, pe, se;
      two_prod(xs[q], ws[q], p, pe);
      two_sum(s, p, s, se);
      c = __fadd_rn(c, __fadd_rn(pe, se));
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float so = __shfl_xor_sync(0xffffffffu, s, off);
    const float co = __shfl_xor_sync(0xffffffffu, c, off);
    float se;
    two_sum(s, so, s, se);
    c = __fadd_rn(c, __fadd_rn(co, se));
  }
  if (bias_e) {
    float se;
    two_sum(s, *bias_e, s, se);
    c = __fadd_rn(c, se);
  }
  return __fadd_rn(s, c);
}

// One warp per (t, e) (or per (listed token, e) when `list` is given, for
// the tokens the certified fast path handed back): exact logits.
__global__ void k_router_logits(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                                const float *__restrict__ bias, int T, int D, int E,
                                float *__restrict__ logits, const int32_t *__restrict__ list = nullptr,
                                const int32_t *__restrict__ count = nullptr) {
  const int lane = threadIdx.x & 31;
  const int64_t n = list ? (int64_t)*count * E : (int64_t)T * E;
  for (int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; gw < n;
       gw += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int t = list ? list[gw / E] : (int)(gw / E), e = (int)(gw % E);
    const float v = dot2_row_warp(x + (int64_t)t * D, Wr + (int64_t)e * D, D, bias ? bias + e : nullptr);
    if (lane == 0) logits[(int64_t)t * E + e] = v;
  }
}

// a ranks before b: larger first, NaN below everything, ties to lower id.
__device__ __forceinline__ bool ranks_before(float va, int a, float vb, int b) {
  if (b < 0) return a >= 0;
  if (a < 0) return false;
  const bool na = isnan(va), nb = isnan(vb);
  if (na || nb) return (na && nb) ? a < b : nb;
  if (va != vb) return va > vb;
  return a < b;
}

__device__ __forceinline__ void topk_softmax_warp(const float (&v)[8], int E, int k, int32_t *__restrict__ idx,
                                                  float *__restrict__ w) {
  const int lane = threadIdx.x & 31;
  float my_v;
  int my_e;
  topk_select_warp(v, E, k, my_v, my_e);
  const float wi = softmax_selected_warp(my_v, k);
  if (lane < k) {
    idx[lane] = my_e;
    w[lane] = wi;
  }
}

// One warp per token: top-k + softmax over logits already in memory
// (E <= 256 in registers; larger E re-reads its row each round).
__device__ __forceinline__ void topk_softmax_row(const float *__restrict__ logits, int t, int E, int k,
                                                 int32_t *__restrict__ idx, float *__restrict__ w) {
  const int lane = threadIdx.x & 31;
  const float *l = logits + (int64_t)t * E;
  if (E <= 256) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = lane + 32 * j < E ? l[lane + 32 * j] : 0.f;
    topk_softmax_warp(v, E, k, idx + (int64_t)t * k, w + (int64_t)t * k);
    return;
  }
  uint32_t taken = 0;  // bit j: entry lane + 32 j already selected
  float my_v = 0.f;
  int my_e = -1;
  for (int i = 0; i < k; ++i) {
    float bv = 0.f;
    int be = -1;
    for (int j = 0, e = lane; e < E; ++j, e += 32) {
      if (taken & (1u << j)) continue;
      const float v = l[e];
      if (ranks_before(v, e, bv, be)) { bv = v; be = e; }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ranks_before(ov, oe, bv, be)) { bv = ov; be = oe; }
    }
    if (be >= 0 && (be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == i) { my_v = bv; my_e = be; }
  }
  const double m = (double)__shfl_sync(0xffffffffu, my_v, 0);
  const double ex = lane < k ? exp((double)my_v - m) : 0.0;
  double sum = 0.0;
  for (int i = 0; i < k; ++i) sum += __shfl_sync(0xffffffffu, ex, i);
  if (lane < k) {
    idx[(int64_t)t * k + lane] = my_e;
    w[(int64_t)t * k + lane] = (float)(ex / sum);
  }
}

// With `list`, only the listed tokens (count of them).
__global__ void k_topk_softmax(const float *__restrict__ logits, int T, int E, int k,
                               int32_t *__restrict__ idx, float *__restrict__ w,
                               const int32_t *__restrict__ list = nullptr, const int32_t *__restrict__ count = nullptr) {
  const int n = list ? *count : T;
  for (int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5); gw < n;
       gw += (int)(((int64_t)gridDim.x * blockDim.x) >> 5))
    topk_softmax_row(logits, list ? list[gw] : gw, E, k, idx, w);
}

// ------------------------------------ routing with a selection-only bias
// Both logits of (t, e) from one Dot2 pass: the unbiased one rounded from
// the compensated (sum, error) pair, the biased one after adding the bias
// with TwoSum -- each equal to what the plain router computes for it.
__global__ void k_router_logits_both(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                                     const float *__restrict__ bias, int T, int D, int E, float *__restrict__ lb,
                                     float *__restrict__ lu) {
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)T * E;
  for (int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; gw < n;
       gw += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int t = (int)(gw / E), e = (int)(gw % E);
    const uint16_t *xr = x + (int64_t)t * D;
    const float *wr = Wr + (int64_t)e * D;
    float s = 0.f, c = 0.f;
    for (int j = 4 * lane; j < D; j += 128) {
      const float4 wv = *reinterpret_cast<const float4 *>(wr + j);
      const uint2 xv = *reinterpret_cast<const uint2 *>(xr + j);
      const float xs[4] = {bf16_bits_to_f32(xv.x & 0xFFFFu), bf16_bits_to_f32(xv.x >> 16),
                           bf16_bits_to_f32(xv.y & 0xFFFFu), bf16_bits_to_f32(xv.y >> 16)};
      const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float p, pe, se;
        two_prod(xs[q], w4[q], p, pe);
        two_sum(s, p, s, se);
        c = __fadd_rn(c, __fadd_rn(pe, se));
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float so = __shfl_xor_sync(0xffffffffu, s, off);
      const float co = __shfl_xor_sync(0xffffffffu, c, off);
      float se;
      two_sum(s, so, s, se);
      c = __fadd_rn(c, __fadd_rn(co, se));
    }
    const float vu = __fadd_rn(s, c);
    float sb, se;
    two_sum(s, bias[e], sb, se);
    const float vb = __fadd_rn(sb, __fadd_rn(c, se));
    if (lane == 0) {
      lu[(int64_t)t * E + e] = vu;
      lb[(int64_t)t * E + e] = vb;
    }
  }
}

// One warp per token (E <= 256): rank by the biased logits; weights are the
// softmax of the selected experts' unbiased logits shifted by their maximum,
// in double, summed in rank order, rounded once.
__global__ void k_topk_selbias(const float *__restrict__ lb, const float *__restrict__ lu, int T, int E, int k,
                               int32_t *__restrict__ idx, float *__restrict__ w) {
  const int lane = threadIdx.x & 31;
  for (int t = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5); t < T;
       t += (int)(((int64_t)gridDim.x * blockDim.x) >> 5)) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = lane + 32 * j < E ? lb[(int64_t)t * E + lane + 32 * j] : 0.f;
    float my_v;
    int my_e;
    topk_select_warp(v, E, k, my_v, my_e);
    const double u = lane < k ? (double)lu[(int64_t)t * E + my_e] : -INFINITY;
    double m = u;
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, off));
    const double ex = lane < k ? exp(u - m) : 0.0;
    double sum = 0.0;
    for (int i = 0; i < k; ++i) sum += __shfl_sync(0xffffffffu, ex, i);
    if (lane < k) {
      idx[(int64_t)t * k + lane] = my_e;
      w[(int64_t)t * k + lane] = (float)(ex / sum);
    }
  }
}

// ------------------------------------------------- certified router (large T)
// Approximate logits (no bias) for the certified fast path: a tiled fp32
// GEMM, 64 tokens x 64 experts per CTA and 4 x 4 outputs per thread.  Each
// output is a sum of 64-term FMA chains over consecutive 64-value chunks of
// K, each chunk started from zero and then added to the running total, so
// it carries at most 64 + D/64 roundings: |error| <= gamma_n * sum_j
// |x_j w_j| with gamma_n = n u / (1 - n u), u = 2^-24 (Higham, "Accuracy and
// Stability of Numerical Algorithms", 2nd ed., section 3.1).
constexpr int kRT = 64, kRK = 32;
// The staged K slices are stored transposed ([k][row]); row index XOR
// 8 ((k / 8) % 4) keeps the stores of one warp on distinct banks and the
// float4 groups read back intact.  The next slice is fetched into
// registers while the current one is multiplied (two shared buffers, one
// barrier per slice).  Arithmetic and its order are the plain tiled GEMM's.
__device__ __forceinline__ int router_sw(int k) { return 8 * ((k >> 3) & 3); }

__global__ void __launch_bounds__(256) k_router_approx(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                                                       int T, int D, int E, float *__restrict__ lg) {
  __shared__ __align__(16) float Xs[2][kRK][kRT + 4];
  __shared__ __align__(16) float Ws[2][kRK][kRT + 4];
  const int t0 = blockIdx.y * kRT, e0 = blockIdx.x * kRT;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int lr = tid >> 2, lc = (tid & 3) * 8;  // staging: row lr, k lc .. lc + 7
  const int t_ld = t0 + lr, e_ld = e0 + lr;
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  float4 wa = make_float4(0.f, 0.f, 0.f, 0.f), wb = wa;
  auto fetch = [&](int kc) {
    if (t_ld < T) xv = *reinterpret_cast<const uint4 *>(x + (int64_t)t_ld * D + kc + lc);
    if (e_ld < E) {
      wa = *reinterpret_cast<const float4 *>(Wr + (int64_t)e_ld * D + kc + lc);
      wb = *reinterpret_cast<const float4 *>(Wr + (int64_t)e_ld * D + kc + lc + 4);
    }
  };
  auto stage = [&](int b) {
    const int col = lr ^ router_sw(lc);  // the same for k = lc .. lc + 7
    const uint32_t wd[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      Xs[b][lc + 2 * q][col] = bf16_bits_to_f32(wd[q] & 0xFFFFu);
      Xs[b][lc + 2 * q + 1][col] = bf16_bits_to_f32(wd[q] >> 16);
    }
    const float w8[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) Ws[b][lc + q][col] = w8[q];
  };
  float tot[4][4], acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) tot[i][j] = acc[i][j] = 0.f;
  fetch(0);
  stage(0);
  __syncthreads();
  for (int kc = 0, b = 0; kc < D; kc += kRK, b ^= 1) {
    const bool more = kc + kRK < D;
    if (more) fetch(kc + kRK);
    // each output: 64-term FMA chains over consecutive 64-value chunks of K,
    // each started from zero and then added to the running total
    if ((kc & 63) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    }
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float4 xq = *reinterpret_cast<const float4 *>(&Xs[b][kk][(ty * 4) ^ router_sw(kk)]);
      const float4 wq = *reinterpret_cast<const float4 *>(&Ws[b][kk][(tx * 4) ^ router_sw(kk)]);
      const float xa[4] = {xq.x, xq.y, xq.z, xq.w}, wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wv[j], acc[i][j]);
    }
    if ((kc & 63) == 32) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[i][j] = __fadd_rn(tot[i][j], acc[i][j]);
    }
    if (more) stage(b ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) lg[(int64_t)t * E + e] = tot[i][j];
    }
  }
}

// Euclidean norms of the T rows of x and the E rows of Wr (one warp per
// row), rounded up so that |x_t . w_e| sums are bounded by xn[t] * wn[e]
// (Cauchy-Schwarz).
__global__ void k_row_norms(const uint16_t *__restrict__ x, int T, const float *__restrict__ Wr, int E, int D,
                            float *__restrict__ xn, float *__restrict__ wn) {
  const int lane = threadIdx.x & 31;
  for (int r = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5); r < T + E;
       r += (int)(((int64_t)gridDim.x * blockDim.x) >> 5)) {
    float ss = 0.f;
    if (r < T) {
      const uint16_t *xr = x + (int64_t)r * D;
      for (int j = 2 * lane; j < D; j += 64) {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(xr + j);
        const float a = bf16_bits_to_f32(v & 0xFFFFu), b = bf16_bits_to_f32(v >> 16);
        ss = fmaf(a, a, fmaf(b, b, ss));
      }
    } else {
      const float *wr = Wr + (int64_t)(r - T) * D;
      for (int j = lane; j < D; j += 32) ss = fmaf(wr[j], wr[j], ss);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    // the fp32 sum of squares is within (D/32 + 6) u of exact; 1 + 2^-10 covers it
    const float nv = sqrtf(ss) * (1.f + 0x1p-10f);
    if (lane == 0) (r < T ? xn[r] : wn[r - T]) = nv;
  }
}

// One warp per token: top-k over the approximate logits (+ bias); if every
// selected value minus its error bound stays above every unselected value
// plus its bound, the selected set is that of the exact logits, and only
// the k selected logits are recomputed exactly (Dot2) to order them and
// weight them.  Otherwise the token is handed back (list) for an exact pass
// over all E logits.
__global__ void k_topk_cert(const float *__restrict__ lg, const float *__restrict__ bias,
                            const float *__restrict__ xn, const float *__restrict__ wn,
                            const uint16_t *__restrict__ x, const float *__restrict__ Wr, int T, int D, int E,
                            int k, float gam, int32_t *__restrict__ idx, float *__restrict__ w,
                            int32_t *__restrict__ list, int32_t *__restrict__ count) {
  const int lane = threadIdx.x & 31;
  for (int t = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5); t < T;
       t += (int)(((int64_t)gridDim.x * blockDim.x) >> 5)) {
    float v[8], bd[8];
    bool finite = true;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      v[j] = 0.f;
      bd[j] = 0.f;
      if (e < E) {
        v[j] = __fadd_rn(lg[(int64_t)t * E + e], bias ? bias[e] : 0.f);
        bd[j] = gam * xn[t] * wn[e] + 0x1p-21f * fabsf(v[j]) + 0x1p-126f;
        finite &= isfinite(v[j]) && isfinite(bd[j]);
      }
    }
    float my_v;
    int my_e;
    topk_select_warp(v, E, k, my_v, my_e);
    uint32_t selm = 0;
    for (int i = 0; i < k; ++i) {
      const int se = __shfl_sync(0xffffffffu, my_e, i);
      if (se >= 0 && (se & 31) == lane) selm |= 1u << (se >> 5);
    }
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (lane + 32 * j >= E) continue;
      if ((selm >> j) & 1u) lo = fminf(lo, v[j] - bd[j]);
      else hi = fmaxf(hi, v[j] + bd[j]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    finite = __all_sync(0xffffffffu, finite);
    if (!finite || !(lo > hi)) {
      if (lane == 0) list[atomicAdd(count, 1)] = t;
      continue;
    }
    // exact logits of the selected experts, then order them exactly
    float ex = 0.f;
    for (int i = 0; i < k; ++i) {
      const int se = __shfl_sync(0xffffffffu, my_e, i);
      const float val = dot2_row_warp(x + (int64_t)t * D, Wr + (int64_t)se * D, D, bias ? bias + se : nullptr);
      if (lane == i) ex = val;
    }
    int rank = 0;
    for (int j = 0; j < k; ++j) {
      const float ov = __shfl_sync(0xffffffffu, ex, j);
      const int oe = __shfl_sync(0xffffffffu, my_e, j);
      if (lane < k && j != lane && ranks_before(ov, oe, ex, my_e)) ++rank;
    }
    float rv = 0.f;
    int re = -1;
    for (int r = 0; r < k; ++r) {
      const int src = __ffs(__ballot_sync(0xffffffffu, lane < k && rank == r)) - 1;
      const float vv = __shfl_sync(0xffffffffu, ex, src);
      const int ee = __shfl_sync(0xffffffffu, my_e, src);
      if (lane == r) { rv = vv; re = ee; }
    }
    const float wi = softmax_selected_warp(rv, k);
    if (lane < k) {
      idx[(int64_t)t * k + lane] = re;
      w[(int64_t)t * k + lane] = wi;
    }
  }
}

// fp16 copy of x and its sub-block (16-value) / block (32-value) sums for
// the tensor-core decode kernels, by `n` threads numbered from `i0`.
// bf16 -> fp16 is exact for |x| in [2^-14, 65504]; larger magnitudes are
// flagged as a data error.
__device__ __forceinline__ void convert_x(const uint16_t *__restrict__ x, int T, int D, uint16_t *__restrict__ x16,
                                          uint8_t *__restrict__ xs16, float *__restrict__ xs32,
                                          WsHeader *__restrict__ hdr, int i0, int n) {
  const int n32 = D / 32;
  for (int i = i0; i < T * n32; i += n) {
    const int t = i / n32, b32 = i % n32;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (int64_t)t * D + 32 * b32);
    uint4 *x16r = reinterpret_cast<uint4 *>(x16 + (int64_t)t * D + 32 * b32);
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldcg(xr + q);
    float s[2] = {0.f, 0.f};
    bool big = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t wd[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
      uint32_t o[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float lo = bf16_bits_to_f32(wd[r] & 0xFFFFu), hi = bf16_bits_to_f32(wd[r] >> 16);
        big |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
        o[r] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
        s[q >> 1] += lo + hi;
      }
      x16r[q] = make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int n16 = 2 * b32 + hh;
      const __half hi = __float2half_rn(s[hh]);
      const __half lo = __float2half_rn(s[hh] - __half2float(hi));
      uint16_t *rec = reinterpret_cast<uint16_t *>(xs16 + ((int64_t)t * (D / 256 + 1) + n16 / 16) * 64);
      rec[n16 & 15] = __half_as_ushort(hi);
      rec[16 + (n16 & 15)] = __half_as_ushort(lo);
      big |= fabsf(s[hh]) > 65504.f;
    }
    if (big) record_status(hdr, DS4MOE_EDEVICE);
    xs32[(int64_t)t * n32 + b32] = s[0] + s[1];
  }
}

// convert_x over a whole grid (the prefill's weight-streaming experts).
__global__ void k_convert_x(const uint16_t *__restrict__ x, int T, int D, uint16_t *__restrict__ x16,
                            uint8_t *__restrict__ xs16, float *__restrict__ xs32, WsHeader *__restrict__ hdr) {
  convert_x(x, T, D, x16, xs16, xs32, hdr, (int)(blockIdx.x * blockDim.x + threadIdx.x), (int)(gridDim.x * blockDim.x));
}

// Outputs of the bucketing step (pairs p = t*k + i grouped by expert).
struct BucketArgs {
  int32_t *idx;
  int P, E, T, D, k;
  WsHeader *hdr;
  int32_t *counts, *offs, *active, *perm, *inv, *lrank;
  Group *groups;
  const uint16_t *x;
  uint16_t *x16;
  uint8_t *xs16;
  float *xs32;
  float *w;
  int32_t *nvalid;
  float *out;
  int32_t *zero2;  // single-token chain: further counters the router grid zeroes
  int nzero2;
  int32_t *zero3;  // and the tagged hidden words of the tile-order grid
  int nzero3;
  // single token, layer input made here (nullptr otherwise): x = bf16 of
  // RMS-normalised (nrm_res + nrm_add), as k_residual_norm computes it; CTA 0
  // stores the sum to nrm_res_next and x to nrm_x
  const float *nrm_res, *nrm_add;
  float *nrm_res_next;
  uint16_t *nrm_x;
  float nrm_eps;
};

// Bucketing of a decode batch (P <= 32 pairs) by a CTA of 256 threads
// (E <= 256).  With `logits`, warp w ranks the experts of tokens w, w + 8,
// ... (writing idx, and the k selected logits to w: the routing weights are
// their softmax, computed later off the critical path by
// finish_routing_weights); then warp 0 sorts the pairs by (expert, pair
// index) with ballot-based radix ranking and cuts them into groups of
// <= kGroup.
__device__ __forceinline__ void bucket_small_warps(const BucketArgs &b, const float *__restrict__ logits) {
  __shared__ int32_t s_idx[32];
  __shared__ int32_t sorted_e[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int P = b.P, E = b.E, T = b.T, k = b.k;
  if (logits) {
    for (int t = wid; t < T; t += nw) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? __ldcg(logits + (int64_t)t * E + e) : 0.f;
      }
      float my_v;
      int my_e;
      topk_select_warp(v, E, k, my_v, my_e);
      if (lane < k) {
        s_idx[t * k + lane] = my_e;
        b.idx[(int64_t)t * k + lane] = my_e;
        b.w[(int64_t)t * k + lane] = my_v;
      }
    }
    __syncthreads();
  }
  if (wid != 0) return;
  if (!logits && lane < P) s_idx[lane] = __ldcg(b.idx + lane);
  __syncwarp();
  int e = -1;
  if (lane < P) {
    e = s_idx[lane];
    if (e < 0 || e >= E) { record_status(b.hdr, DS4MOE_EDEVICE); e = -1; }
  }
  const unsigned valid = __ballot_sync(0xffffffffu, e >= 0);
  // valid experts per token (for the fused combine); a token without any
  // gets a zero output row
  if (lane < T) {
    const int nvt = __popc(valid & (uint32_t)(((1ull << k) - 1ull) << (lane * k)));
    b.nvalid[lane] = nvt;
    if (nvt == 0)
      for (int c = 0; c < b.D; ++c) b.out[(int64_t)lane * b.D + c] = 0.f;
  }
  // rank of (expert, pair) among the 32 lanes, invalid pairs last (as
  // expert E): radix ranking over the keys (expert << 5 | lane), one ballot
  // per key bit, most significant first
  const uint32_t key = ((uint32_t)(e >= 0 ? e : E) << 5) | (uint32_t)lane;
  const int nbits = 5 + 32 - __clz(E);
  int rank = 0;
  uint32_t same = 0xffffffffu;
  for (int bit = nbits - 1; bit >= 0; --bit) {
    const uint32_t mine = (key >> bit) & 1u;
    const uint32_t ones = __ballot_sync(0xffffffffu, mine);
    if (mine) rank += __popc(same & ~ones);
    same &= mine ? ones : ~ones;
  }
  if (lane < P) b.inv[lane] = e >= 0 ? rank : -1;
  if (e >= 0) b.perm[rank] = lane;
  // sorted view: lane r holds the expert of the r-th pair
  if (e >= 0) sorted_e[rank] = e;
  __syncwarp();
  const int nv = __popc(valid);
  const int er = lane < nv ? sorted_e[lane] : -1;
  const int eprev = __shfl_up_sync(0xffffffffu, er, 1);
  const bool run_start = lane < nv && (lane == 0 || eprev != er);
  const unsigned starts = __ballot_sync(0xffffffffu, run_start);
  const int rs = 31 - __clz(starts & (0xffffffffu >> (31 - lane)));   // start of this lane's run
  const bool gstart = lane < nv && ((lane - rs) % kGroup == 0);
  const unsigned gmask = __ballot_sync(0xffffffffu, gstart);
  if (gstart) {
    int run_end = nv;
    const unsigned later = starts & ~(0xffffffffu >> (31 - lane));
    if (later) run_end = __ffs(later) - 1;
    b.groups[__popc(gmask & ((1u << lane) - 1u))] = Group{er, lane, min(kGroup, run_end - lane), 0};
  }
  if (lane == 0) {
    b.hdr->n_groups = __popc(gmask);
    b.hdr->n_active = __popc(starts);
  }
}

// MODE kRouteLogits only writes the logits (the bucketing kernel ranks
// them).  Otherwise the last CTA to finish (ticket counter in the workspace
// header) ranks the experts of every token: kRouteTopk writes idx and w;
// kRouteBucket (decode batches of <= 32 pairs) also sorts the pairs into
// expert groups for the FFN kernels, and every CTA first converts its slice
// of x for them -- the whole bucketing step without a kernel of its own.
enum { kRouteLogits = 0, kRouteTopk = 1, kRouteBucket = 2 };
template <int NI, int MODE>
__global__ void __launch_bounds__(256) k_route_small(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                                                     const float *__restrict__ bias, int T, int D, int E, int k,
                                                     float *__restrict__ logits, int32_t *__restrict__ idx,
                                                     float *__restrict__ w, WsHeader *__restrict__ hdr,
                                                     BucketArgs bk) {
  __shared__ float ps[8][32], pc[8][32];
  __shared__ uint32_t ticket;
  const SpanExit span_exit(DS4MOE_SPAN_ROUTE);
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // the router row is constant: fetch it before waiting for x
  float4 wv[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int j = 4 * (tid + 256 * i);
    wv[i] = j < D ? __ldg(reinterpret_cast<const float4 *>(Wr + (int64_t)e * D + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  ptx::pdl_wait();
  span_begin(DS4MOE_SPAN_ROUTE);
  ptx::pdl_launch_dependents();
  // single-token chain: the merged FFN grid's per-expert counters start at 0
  if (MODE == kRouteLogits && bk.counts && tid == 0) bk.counts[blockIdx.x] = 0;
  if (MODE == kRouteLogits && bk.zero2)
    for (int i = blockIdx.x * 256 + tid; i < bk.nzero2; i += gridDim.x * 256) bk.zero2[i] = 0;
  if (MODE == kRouteLogits && bk.zero3)
    for (int i = blockIdx.x * 256 + tid; i < bk.nzero3; i += gridDim.x * 256) bk.zero3[i] = 0;
  // the fp16 copy of x and its block sums for the multi-token FFN kernels,
  // spread over all CTAs of the router (not the single bucketing CTA)
  if (MODE != kRouteTopk && bk.xs16)
    convert_x(x, T, D, bk.x16, bk.xs16, bk.xs32, hdr, blockIdx.x * 256 + tid, gridDim.x * 256);
  if (MODE == kRouteLogits && bk.nrm_res) {
    // one token: the residual add and the RMS norm of k_residual_norm, with
    // its thread mapping and summation order (every CTA the same values)
    __shared__ float s_part[8];
    float4 v[NI];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int q = tid + 256 * i;
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (4 * q < D) {
        float4 a = __ldcg(reinterpret_cast<const float4 *>(bk.nrm_res) + q);
        const float4 o = __ldcg(reinterpret_cast<const float4 *>(bk.nrm_add) + q);
        a.x = __fadd_rn(a.x, o.x);
        a.y = __fadd_rn(a.y, o.y);
        a.z = __fadd_rn(a.z, o.z);
        a.w = __fadd_rn(a.w, o.w);
        v[i] = a;
        ss = fmaf(a.x, a.x, ss);
        ss = fmaf(a.y, a.y, ss);
        ss = fmaf(a.z, a.z, ss);
        ss = fmaf(a.w, a.w, ss);
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) s_part[wid] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) tot += s_part[ww];
    const float r = 1.0f / sqrtf(tot / (float)D + bk.nrm_eps);
    uint2 xv[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int q = tid + 256 * i;
      xv[i] = make_uint2((uint32_t)f32_to_bf16_bits(v[i].x * r) | ((uint32_t)f32_to_bf16_bits(v[i].y * r) << 16),
                         (uint32_t)f32_to_bf16_bits(v[i].z * r) | ((uint32_t)f32_to_bf16_bits(v[i].w * r) << 16));
      if (blockIdx.x == 0 && 4 * q < D) {
        reinterpret_cast<float4 *>(bk.nrm_res_next)[q] = v[i];
        reinterpret_cast<uint2 *>(bk.nrm_x)[q] = xv[i];
      }
    }
    route_dot2_regs<NI>(xv, wv, D, tid, ps[wid][0], pc[wid][0]);
    __syncthreads();
    if (wid == 0 && lane == 0) logits[e] = route_dot2_merge(ps, pc, 0, bias ? bias + e : nullptr);
    return;
  }
  for (int t0 = 0; t0 < T; t0 += 32) {
    const int nt = min(32, T - t0);
    int tt = 0;
    for (; tt + 4 <= nt; tt += 4)
      route_dot2_partial_n<NI, 4>(x + (int64_t)(t0 + tt) * D, D, wv, D, tid, &ps[wid][tt], &pc[wid][tt]);
    for (; tt < nt; ++tt) route_dot2_partial<NI>(x + (int64_t)(t0 + tt) * D, wv, D, tid, ps[wid][tt], pc[wid][tt]);
    __syncthreads();
    if (wid == 0 && lane < nt) logits[(int64_t)(t0 + lane) * E + e] = route_dot2_merge(ps, pc, lane, bias ? bias + e : nullptr);
    __syncthreads();
  }
  if (MODE == kRouteLogits) return;  // ranking done by the bucketing kernel
  // the last CTA to finish ranks the experts of every token
  __threadfence();
  __syncthreads();
  if (tid == 0) ticket = atomicAdd(&hdr->route_done, 1u);
  __syncthreads();
  if (ticket != (uint32_t)E - 1u) return;
  __threadfence();
  if (MODE == kRouteBucket) {
    bucket_small_warps(bk, logits);
  } else {
    for (int t = wid; t < T; t += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int ee = lane + 32 * j;
        v[j] = ee < E ? __ldcg(logits + (int64_t)t * E + ee) : 0.f;
      }
      topk_softmax_warp(v, E, k, idx + (int64_t)t * k, w + (int64_t)t * k);
    }
  }
  if (tid == 0) hdr->route_done = 0u;
}

// ---------------------------------------------------------------- bucketing
// One CTA (256 threads for the decode batch path, P <= 32, which leaves the
// expert offsets unwritten; else 1024).  Pairs p = t*k + i are grouped by expert, stable
// in p (hence in token order).  Phase A: warp w walks its contiguous slice of
// pairs 32 at a time and ranks each pair among same-expert pairs of the slice
// (__match_any_sync); Phase B: per-expert totals, exclusive offsets and
// per-warp bases; Phase C: scatter.  Also builds the list of active experts.
__global__ void __launch_bounds__(1024) k_bucket(int32_t *__restrict__ idx, int P, int E,
                                                 WsHeader *__restrict__ hdr, int32_t *__restrict__ counts,
                                                 int32_t *__restrict__ offs, int32_t *__restrict__ active,
                                                 int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                                                 int32_t *__restrict__ lrank, Group *__restrict__ groups,
                                                 const uint16_t *__restrict__ x, int T, int D,
                                                 uint16_t *__restrict__ x16, uint8_t *__restrict__ xs16,
                                                 float *__restrict__ xs32, const float *__restrict__ logits, int k,
                                                 float *__restrict__ w, int32_t *__restrict__ nvalid,
                                                 float *__restrict__ out) {
  extern __shared__ int32_t sm[];
  int32_t *wcnt = sm;              // [32][E]
  int32_t *soff = sm + 32 * E;     // [E + 1]
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nthr = blockDim.x;
  ptx::pdl_wait();  // idx (or the logits) and x come from the preceding grids
  ptx::pdl_launch_dependents();
  if (nthr <= 256) {  // the host picks 256 threads only for P <= 32
    // Small batch (decode): warps 0 and 1 rank, weight and sort, the other
    // warps convert x -- concurrently.
    BucketArgs b{idx, P, E, T, D, k, hdr, counts, offs, active, perm, inv, lrank, groups, x, x16, xs16, xs32, w,
                 nvalid, out};
    bucket_small_warps(b, logits);
    if (wid >= 2 && xs16) convert_x(x, T, D, x16, xs16, xs32, hdr, tid - 64, nthr - 64);
    return;
  }
  // fused decode path: rank the experts of every token here (E <= 256)
  if (logits) {
    for (int t = wid; t < T; t += nthr / 32) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        v[j] = e < E ? __ldcg(logits + (int64_t)t * E + e) : 0.f;
      }
      topk_softmax_warp(v, E, k, idx + (int64_t)t * k, w + (int64_t)t * k);
    }
    __syncthreads();
  }
  // valid experts per token (for the fused combine); a token without any
  // gets a zero output row here
  for (int t = tid; t < T; t += nthr) {
    int nv = 0;
    for (int i = 0; i < k; ++i) {
      const int e = __ldcg(idx + (int64_t)t * k + i);
      nv += e >= 0 && e < E;
    }
    nvalid[t] = nv;
    if (nv == 0)
      for (int c = 0; c < D; ++c) out[(int64_t)t * D + c] = 0.f;
  }
  if (xs16) convert_x(x, T, D, x16, xs16, xs32, hdr, tid, nthr);
  for (int i = tid; i < 32 * E; i += nthr) wcnt[i] = 0;
  __syncthreads();
  const int R = (P + 31) / 32;
  const int p0 = wid * R, p1 = min(P, p0 + R);
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    int e = -1;
    if (p < p1) {
      e = idx[p];
      if (e < 0 || e >= E) { record_status(hdr, DS4MOE_EDEVICE); e = -1; }
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(mask & ((1u << lane) - 1u));
    int base = 0;
    if (e >= 0) base = wcnt[wid * E + e];
    __syncwarp();
    if (e >= 0 && rank == 0) wcnt[wid * E + e] = base + __popc(mask);
    __syncwarp();
    if (p < p1) lrank[p] = e >= 0 ? base + rank : -1;
  }
  __syncthreads();
  // Phase B: totals and per-warp exclusive bases (one thread per expert)
  for (int e = tid; e < E; e += 1024) {
    int run = 0;
    for (int w2 = 0; w2 < 32; ++w2) {
      const int c = wcnt[w2 * E + e];
      wcnt[w2 * E + e] = run;
      run += c;
    }
    soff[e] = run;  // count, scanned below
    counts[e] = run;
  }
  __syncthreads();
  // exclusive scan of soff[0..E) (E <= 1024: one element per thread)
  {
    const int v = tid < E ? soff[tid] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int wt = warp_tot[lane], wi = wt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      warp_tot[lane] = wi - wt;  // exclusive
    }
    __syncthreads();
    const int excl = warp_tot[wid] + incl - v;
    __syncthreads();
    if (tid < E) { soff[tid] = excl; offs[tid] = excl; }
    if (tid == E - 1) offs[E] = excl + v;
    // active list: flags (count > 0) scanned the same way
    const int f = (tid < E && v > 0) ? 1 : 0;
    int fi = f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, fi, off);
      if (lane >= off) fi += o;
    }
    if (lane == 31) warp_tot[wid] = fi;
    __syncthreads();
    if (wid == 0) {
      int wt = warp_tot[lane], wi = wt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      warp_tot[lane] = wi - wt;
      if (lane == 31) hdr->n_active = wi;
    }
    __syncthreads();
    if (f) active[warp_tot[wid] + fi - 1] = tid;
    __syncthreads();
    // token groups: ceil(count / kGroup) per expert, numbered in expert order
    const int ng = (v + kGroup - 1) / kGroup;
    int gi = ng;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, gi, off);
      if (lane >= off) gi += o;
    }
    if (lane == 31) warp_tot[wid] = gi;
    __syncthreads();
    if (wid == 0) {
      int wt = warp_tot[lane], wi = wt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      warp_tot[lane] = wi - wt;
      if (lane == 31) hdr->n_groups = wi;
    }
    __syncthreads();
    if (tid < E) {
      const int g0 = warp_tot[wid] + gi - ng;
      for (int j = 0; j < ng; ++j) groups[g0 + j] = Group{tid, excl + kGroup * j, min(kGroup, v - kGroup * j), 0};
    }
  }
  __syncthreads();
  // Phase C: scatter
  for (int p = tid; p < P; p += 1024) {
    const int r = lrank[p];
    if (r < 0) { inv[p] = -1; continue; }
    const int e = idx[p];
    const int wslice = p / R;
    const int pos = soff[e] + wcnt[wslice * E + e] + r;
    perm[pos] = p;
    inv[p] = pos;
  }
}

// ------------------------------------------------------------- residual
// One CTA per token: x_res += out (fp32; out == nullptr: skip), then
// x_next = bf16_RNE(x_res * r), r = 1 / sqrt(mean(x_res^2) + eps), the sum of
// squares reduced in a fixed order (thread, warp, CTA).
constexpr int kNormThreads = 256;
// With `src`, the residual is read from src and the sum written to x_res.
__global__ void __launch_bounds__(kNormThreads) k_residual_norm(float *__restrict__ x_res, const float *__restrict__ out,
                                                               uint16_t *__restrict__ x_next, int D, float eps,
                                                               const float *__restrict__ src) {
  ptx::pdl_wait();  // out comes from the preceding grid
  ptx::pdl_launch_dependents();
  __shared__ float s_part[kNormThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  float4 *xr = reinterpret_cast<float4 *>(x_res + (int64_t)t * D);
  const float4 *xs = src ? reinterpret_cast<const float4 *>(src + (int64_t)t * D) : xr;
  const float4 *orow = out ? reinterpret_cast<const float4 *>(out + (int64_t)t * D) : nullptr;
  float ss = 0.f;
  for (int i = tid; i < D / 4; i += kNormThreads) {
    float4 v = xs[i];
    if (orow) {
      const float4 o = __ldcg(orow + i);
      v.x = __fadd_rn(v.x, o.x);
      v.y = __fadd_rn(v.y, o.y);
      v.z = __fadd_rn(v.z, o.z);
      v.w = __fadd_rn(v.w, o.w);
    }
    if (orow || src) xr[i] = v;
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((tid & 31) == 0) s_part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
  const float r = 1.0f / sqrtf(tot / (float)D + eps);
  uint2 *xn = reinterpret_cast<uint2 *>(x_next + (int64_t)t * D);
  for (int i = tid; i < D / 4; i += kNormThreads) {
    const float4 v = xr[i];
    xn[i] = make_uint2((uint32_t)f32_to_bf16_bits(v.x * r) | ((uint32_t)f32_to_bf16_bits(v.y * r) << 16),
                       (uint32_t)f32_to_bf16_bits(v.z * r) | ((uint32_t)f32_to_bf16_bits(v.w * r) << 16));
  }
}

// ------------------------------------------------------------- validation
// All three matrices in the 16-row tile order (the single-token kernel's
// weights; no other path reads that order).
inline bool layer_r16(const ds4moe_layer &L) {
  return L.q_gate == DS4MOE_Q2_K_R16 && L.q_up == DS4MOE_Q2_K_R16 && L.q_down == DS4MOE_Q2_K_R16;
}

ds4moe_status check_layer(const ds4moe_layer *L) {
  if (!L) return DS4MOE_EINVAL;
  if (L->q_gate == DS4MOE_IQ2_XXS || L->q_up == DS4MOE_IQ2_XXS || L->q_down == DS4MOE_IQ2_XXS)
    return DS4MOE_EUNSUPPORTED;
  if (!layer_r16(*L) && (!qtype_ok(L->q_gate) || !qtype_ok(L->q_up) || !qtype_ok(L->q_down)))
    return DS4MOE_EUNSUPPORTED;
  if (L->d_model <= 0 || L->d_ff <= 0 || L->n_expert < 1 || L->n_expert > 1024) return DS4MOE_EINVAL;
  if (L->d_model % block_vals(L->q_gate) || L->d_model % block_vals(L->q_up) ||
      L->d_ff % block_vals(L->q_down) || L->d_ff % 16 || L->d_model % 16)
    return DS4MOE_EINVAL;
  if (!L->gate || !L->up || !L->down) return DS4MOE_EINVAL;
  if (!aligned16(L->gate) || !aligned16(L->up) || !aligned16(L->down)) return DS4MOE_EINVAL;
  return DS4MOE_OK;
}

// The bucketing outputs inside a workspace laid out by ws_layout.
BucketArgs bucket_args(const ds4moe_layer &L, void *ws, const WsLayout &lay, const uint16_t *x, int32_t *idx,
                       float *w, int T, int k, float *out, bool sums) {
  return BucketArgs{idx, T * k, L.n_expert, T, L.d_model, k, ws_ptr<WsHeader>(ws, lay.hdr),
                    ws_ptr<int32_t>(ws, lay.counts), ws_ptr<int32_t>(ws, lay.offs), ws_ptr<int32_t>(ws, lay.active),
                    ws_ptr<int32_t>(ws, lay.perm), ws_ptr<int32_t>(ws, lay.inv), ws_ptr<int32_t>(ws, lay.lrank),
                    ws_ptr<Group>(ws, lay.groups), x, ws_ptr<uint16_t>(ws, lay.x16),
                    sums ? ws_ptr<uint8_t>(ws, lay.xs16) : nullptr, sums ? ws_ptr<float>(ws, lay.xs32) : nullptr, w,
                    ws_ptr<int32_t>(ws, lay.nvalid), out};
}

// Attributes of the routing chain's kernels, set once per device (kernel
// attributes are per device) under a lock; a failed set is returned to the
// caller and tried again on the next call.  One shared-memory carveout for
// every kernel of the chain: consecutive grids then never wait for an SM to
// reconfigure its L1 / shared split.
constexpr int kAttrDevices = 64;
cudaError_t chain_attributes() {
  static std::mutex mu;
  static std::atomic<bool> done[kAttrDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kAttrDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(k_bucket, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_bucket, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  for (auto kern : {k_route_small<1, kRouteLogits>, k_route_small<2, kRouteLogits>, k_route_small<4, kRouteLogits>,
                    k_route_small<8, kRouteLogits>, k_route_small<1, kRouteTopk>, k_route_small<2, kRouteTopk>,
                    k_route_small<4, kRouteTopk>, k_route_small<8, kRouteTopk>, k_route_small<1, kRouteBucket>,
                    k_route_small<2, kRouteBucket>, k_route_small<4, kRouteBucket>, k_route_small<8, kRouteBucket>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Bucketing, expert FFN and combine.  With `logits` (fused decode path) the
// bucketing kernel first ranks the experts of every token and writes idx / w;
// with `bucketed` the router kernel has already done the whole bucketing step.
ds4moe_status run_ffn(bool prefill, const ds4moe_layer *L, const uint16_t *x, const int32_t *idx,
                      const float *w, int32_t T, int32_t k, float *out, void *ws, size_t ws_bytes,
                      void *stream, const float *logits = nullptr, bool bucketed = false,
                      bool route_t1 = false, bool x_converted = false, bool x_late = false) {
  ds4moe_status st = check_layer(L);
  if (st != DS4MOE_OK) return st;
  if (T < 0 || k < 1 || k > 32 || k > L->n_expert) return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if ((int64_t)T * k > (1 << 24)) return DS4MOE_EINVAL;
  if (!x || !idx || !w || !out || !ws) return DS4MOE_EINVAL;
  if (!aligned16(x) || !aligned16(idx) || !aligned16(w) || !aligned16(out) || !aligned16(ws))
    return DS4MOE_EINVAL;
  if (layer_r16(*L) && (prefill || T != 1 || !t1r_ok(*L, k))) return DS4MOE_EUNSUPPORTED;
  const WsLayout lay = ws_layout(*L, T, k, prefill);
  if (ws_bytes < lay.total) return DS4MOE_ESPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FfnArgs a{};
  a.L = *L;
  a.x = x;
  a.x_late = x_late;
  a.w = w;
  a.T = T;
  a.k = k;
  a.out = out;
  a.hdr = ws_ptr<WsHeader>(ws, lay.hdr);
  a.offs = ws_ptr<int32_t>(ws, lay.offs);
  a.active = ws_ptr<int32_t>(ws, lay.active);
  a.perm = ws_ptr<int32_t>(ws, lay.perm);
  a.inv = ws_ptr<int32_t>(ws, lay.inv);
  a.h = ws_ptr<uint16_t>(ws, lay.h);
  a.y = ws_ptr<float>(ws, lay.y);
  a.groups = ws_ptr<Group>(ws, lay.groups);
  a.x16 = ws_ptr<uint16_t>(ws, lay.x16);
  a.xs16 = ws_ptr<uint8_t>(ws, lay.xs16);
  a.xs32 = ws_ptr<float>(ws, lay.xs32);
  a.hs16 = ws_ptr<uint8_t>(ws, lay.hs16);
  a.nvalid = ws_ptr<int32_t>(ws, lay.nvalid);
  if (layer_r16(*L)) {
    // one token over the tile-order weights: one grid does gate/up, SwiGLU,
    // down and the combine; it ranks the experts from the router's logits
    // or reads the caller's idx / w.  Its per-slot h-ready counters and
    // per-64-row combine counters start at zero (the fused router zeroes
    // them; here they are cleared first).
    a.lg = route_t1 ? logits : nullptr;
    a.idx_out = const_cast<int32_t *>(idx);
    a.ccnt = ws_ptr<int32_t>(ws, lay.cnt);
    cudaError_t e = cudaSuccess;
    if (!route_t1) {
      e = cudaMemsetAsync(a.h, 0, sizeof(int32_t) * (size_t)k * (size_t)L->d_ff, s);
      if (e == cudaSuccess) e = cudaMemsetAsync(a.ccnt, 0, sizeof(int32_t) * (size_t)(L->d_model / 64), s);
    }
    if (e == cudaSuccess) e = launch_ffn_t1r(a, s);
    return cuda_status(e);
  }
  const bool tc = prefill && prefill_tc_ok(*L);
  if (tc) {
    a.xp = ws_ptr<uint16_t>(ws, lay.xp);
    a.chunks_gu = ws_ptr<Chunk>(ws, lay.chunks_gu);
    a.chunks_dn = ws_ptr<Chunk>(ws, lay.chunks_dn);
    a.nchunks = ws_ptr<int32_t>(ws, lay.nchunks);
  }
  const bool sums = !tc && decode_mma_ok(*L);
  a.cnt = sums ? ws_ptr<int32_t>(ws, lay.cnt) : nullptr;
  const int E = L->n_expert, P = T * k;
  if (route_t1) {
    // single token: the FFN grids rank the experts from the logits
    a.lg = logits;
    a.idx_out = const_cast<int32_t *>(idx);
    a.hready = ws_ptr<int32_t>(ws, lay.counts);
    a.ccnt = ws_ptr<int32_t>(ws, lay.cnt);
  } else {
    a.w_logits = logits != nullptr && P <= 32;  // the small bucketing path leaves raw selected logits in w
  }
  const size_t smem = sizeof(int32_t) * (32 * (size_t)E + E + 1);
  cudaError_t e = chain_attributes();
  if (e != cudaSuccess) return cuda_status(e);
  if (!bucketed) {
    ProfScope prof("bucket", s);
    // the tensor-core prefill reads the expert offsets: always the full path
    const int threads = P <= 32 && !tc ? 256 : 1024;
    e = launch_pdl(k_bucket, dim3(1), dim3(threads), threads == 256 ? 0 : smem, s, const_cast<int32_t *>(idx), P, E, a.hdr,
                   ws_ptr<int32_t>(ws, lay.counts), ws_ptr<int32_t>(ws, lay.offs), ws_ptr<int32_t>(ws, lay.active),
                   ws_ptr<int32_t>(ws, lay.perm), ws_ptr<int32_t>(ws, lay.inv), ws_ptr<int32_t>(ws, lay.lrank),
                   ws_ptr<Group>(ws, lay.groups), x, (int)T, (int)L->d_model, ws_ptr<uint16_t>(ws, lay.x16),
                   sums && !x_converted ? ws_ptr<uint8_t>(ws, lay.xs16) : nullptr,
                   sums && !x_converted ? ws_ptr<float>(ws, lay.xs32) : nullptr,
                   logits, (int)k, const_cast<float *>(w), ws_ptr<int32_t>(ws, lay.nvalid), out);
  }
  if (e != cudaSuccess) return cuda_status(e);
  if (tc && prefill_split_ok(*L)) {
    // the experts with few pairs stream their weights through the
    // multi-token kernels, which read x as fp16 with its block sums
    ProfScope prof("convert_x", s);
    const int64_t work = (int64_t)T * (L->d_model / 32);
    const int grid = (int)((work + 255) / 256 < num_sms() * 8 ? (work + 255) / 256 : num_sms() * 8);
    k_convert_x<<<grid, 256, 0, s>>>(x, T, L->d_model, ws_ptr<uint16_t>(ws, lay.x16), ws_ptr<uint8_t>(ws, lay.xs16),
                                     ws_ptr<float>(ws, lay.xs32), a.hdr);
    e = cudaGetLastError();
  } else if (tc) {
    a.x16 = nullptr;  // no split: the grouped kernels do not run
  }
  if (e != cudaSuccess) return cuda_status(e);
  e = prefill ? launch_ffn_prefill(a, s) : launch_ffn_decode(a, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_combine(a, s);
  return cuda_status(e);
}

// ------------------------------------------------ expert-parallel data plane
// dst[j] = x[rows[j]] (bf16 rows of d_model values, 16-byte chunks); one
// thread per chunk.
__global__ void k_gather_rows(const uint4 *__restrict__ x, const int32_t *__restrict__ rows, int n, int nc,
                              uint4 *__restrict__ dst) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)n * nc) return;
  const int j = (int)(i / nc), c = (int)(i % nc);
  dst[i] = __ldg(x + (int64_t)rows[j] * nc + c);
}

// out[t][c] = sum_{i < k} w[t k + i] * y[pos[t k + i]][c], in rank order i,
// skipping pairs with pos < 0; one thread per output element.
__global__ void k_combine_pairs(const float *__restrict__ y, const int32_t *__restrict__ pos,
                                const float *__restrict__ w, int T, int k, int D, float *__restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)T * D) return;
  const int t = (int)(i / D), c = (int)(i % D);
  float acc = 0.f;
  for (int j = 0; j < k; ++j) {
    const int p = pos[(int64_t)t * k + j];
    if (p >= 0) acc = fmaf(w[(int64_t)t * k + j], y[(int64_t)p * D + c], acc);
  }
  out[i] = acc;
}

}  // namespace

// The layer input of a single-token tile-order layer formed inside its
// router grid: x = bf16(rmsnorm(res + add)), the sum stored to res_next
// (a buffer other than res) and x to `x`.
struct NormFuse {
  const float *res, *add;
  float *res_next;
  uint16_t *x;
  float eps;
};

// =================================================================== C ABI
extern "C" {

int32_t ds4moe_block_values(int32_t qtype) { return block_vals(qtype); }
int32_t ds4moe_block_bytes(int32_t qtype) { return block_bytes(qtype); }

int32_t ds4moe_prefill_small_pairs(const ds4moe_layer *L) {
  if (check_layer(L) != DS4MOE_OK) return -1;
  return prefill_tc_ok(*L) && prefill_split_ok(*L) ? kSmallPairs : 0;
}

const char *ds4moe_status_string(int32_t s) {
  switch (s) {
    case DS4MOE_OK: return "ok";
    case DS4MOE_EINVAL: return "invalid argument";
    case DS4MOE_EBLOCKER: return "lossless re-encode condition violated (BLOCKER)";
    case DS4MOE_EUNSUPPORTED: return "unsupported block format";
    case DS4MOE_ECUDA: return "CUDA error";
    case DS4MOE_ETIMEOUT: return "device wait timed out";
    case DS4MOE_EDEVICE: return "device-detected data error";
    case DS4MOE_ESPACE: return "workspace too small";
    default: return "unknown status";
  }
}

ds4moe_status ds4moe_dequant(int32_t qtype, const void *blocks, int64_t n_values, float *out,
                             void *stream) {
  if (qtype == DS4MOE_IQ2_XXS) return DS4MOE_EUNSUPPORTED;
  if (!qtype_ok(qtype)) return DS4MOE_EUNSUPPORTED;
  if (n_values < 0 || n_values % block_vals(qtype)) return DS4MOE_EINVAL;
  if (n_values == 0) return DS4MOE_OK;
  if (!blocks || !out || !aligned16(blocks) || !aligned16(out)) return DS4MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nb = n_values / block_vals(qtype);
  const int64_t work = qtype == DS4MOE_Q4_1 ? nb * 16 : qtype == DS4MOE_Q2_K ? nb * 64 : nb * 128;
  const int threads = 256;
  const int64_t want = (work + threads - 1) / threads;
  const int grid = (int)(want < (int64_t)num_sms() * 32 ? want : (int64_t)num_sms() * 32);
  ProfScope prof("dequant", s);
  if (qtype == DS4MOE_Q4_1)
    k_dequant_q41<<<grid, threads, 0, s>>>(static_cast<const uint8_t *>(blocks), nb, out);
  else if (qtype == DS4MOE_Q2_K)
    k_dequant_q2k<<<grid, threads, 0, s>>>(static_cast<const uint8_t *>(blocks), nb, out);
  else
    k_dequant_q4k<<<grid, threads, 0, s>>>(static_cast<const uint8_t *>(blocks), nb, out);
  return cuda_status(cudaGetLastError());
}

ds4moe_status ds4moe_repack(int32_t src_type, int32_t dst_type, const void *src, int64_t rows, int64_t cols,
                            void *dst, void *stream) {
  const bool to = src_type == DS4MOE_Q2_K && dst_type == DS4MOE_Q2_K_R16;
  const bool from = src_type == DS4MOE_Q2_K_R16 && dst_type == DS4MOE_Q2_K;
  if (!to && !from) return DS4MOE_EUNSUPPORTED;
  if (rows < 0 || cols < 0 || rows % 16 || cols % 256) return DS4MOE_EINVAL;
  if (rows == 0 || cols == 0) return DS4MOE_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return DS4MOE_EINVAL;
  const int64_t bytes = rows * (cols / 256) * kQ2KBytes;
  const char *a = static_cast<const char *>(src), *b = static_cast<const char *>(dst);
  if (a < b + bytes && b < a + bytes) return DS4MOE_EINVAL;  // overlapping
  return cuda_status(launch_repack(to, src, dst, rows, cols, static_cast<cudaStream_t>(stream)));
}

ds4moe_status ds4moe_profile_span(int32_t on, double *total_ns, int64_t *launches) {
  if (on < -1 || on > 1) return DS4MOE_EINVAL;
  if (total_ns)
    for (int i = 0; i < DS4MOE_SPAN_COUNT; ++i) total_ns[i] = 0.0;
  if (launches)
    for (int i = 0; i < DS4MOE_SPAN_COUNT; ++i) launches[i] = 0;
  cudaError_t e = span_control_abi(on, total_ns, launches);
  if (e == cudaSuccess) e = span_control_decode(on, total_ns, launches);
  if (e == cudaSuccess) e = span_control_t1r(on, total_ns, launches);
  if (e == cudaSuccess) e = span_control_prefill(on, total_ns, launches);
  if (e == cudaSuccess) e = span_control_shared(on, total_ns, launches);
  return cuda_status(e);
}

size_t ds4moe_shared_workspace_bytes(int32_t d_model, int32_t d_shared, int32_t T) {
  if (d_model <= 0 || d_shared < 0 || T < 0) return 0;
  return shared_ws_bytes(d_model, d_shared, T);
}

ds4moe_status ds4moe_shared_ffn(const uint16_t *w1, const uint16_t *w3, const uint16_t *w2, int32_t d_model,
                                int32_t d_shared, const uint16_t *x, int32_t T, float *out, int32_t accumulate,
                                void *ws, size_t ws_bytes, void *stream) {
  if (d_model <= 0 || d_model % 8 || d_shared < 0 || d_shared % 8 || T < 0 || (accumulate != 0 && accumulate != 1))
    return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!x || !out || !ws || !aligned16(x) || !aligned16(out) || !aligned16(ws)) return DS4MOE_EINVAL;
  if (d_shared > 0 && (!w1 || !w3 || !w2 || !aligned16(w1) || !aligned16(w3) || !aligned16(w2))) return DS4MOE_EINVAL;
  if (ws_bytes < shared_ws_bytes(d_model, d_shared, T)) return DS4MOE_ESPACE;
  return cuda_status(
      launch_shared_ffn(w1, w3, w2, d_model, d_shared, x, T, out, accumulate, ws, static_cast<cudaStream_t>(stream)));
}

size_t ds4moe_workspace_bytes(const ds4moe_layer *L, int32_t T, int32_t k, int32_t prefill) {
  if (!L || T < 0 || k < 1 || L->n_expert < 1 || L->d_model <= 0 || L->d_ff <= 0) return 0;
  return ws_layout(*L, T, k, prefill).total;
}

ds4moe_status ds4moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (!ws || !aligned16(ws) || ws_bytes < sizeof(WsHeader)) return DS4MOE_EINVAL;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

ds4moe_status ds4moe_route_topk(const uint16_t *x, const float *Wr, const float *bias, int32_t T,
                                int32_t d_model, int32_t n_expert, int32_t k, int32_t *idx, float *w,
                                float *logits, void *ws, size_t ws_bytes, void *stream) {
  if (T < 0 || d_model <= 0 || d_model % 4 || n_expert < 1 || n_expert > 1024 || k < 1 || k > 32 ||
      k > n_expert)
    return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!x || !Wr || !idx || !w || !ws) return DS4MOE_EINVAL;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(idx) || !aligned16(w) || !aligned16(ws) ||
      (bias && !aligned16(bias)) || (logits && !aligned16(logits)))
    return DS4MOE_EINVAL;
  if ((int64_t)d_model * 2 % 16) return DS4MOE_EINVAL;  // bf16 rows start 16-byte aligned
  ds4moe_layer shape{};
  shape.d_model = d_model;
  shape.d_ff = 16;
  shape.n_expert = n_expert;
  const WsLayout lay = ws_layout(shape, T, k, 0);
  // Large batches without a logits output take the certified fast path
  // (approximate fp32 GEMM + error bounds; exact Dot2 for the selected
  // experts and for tokens whose top-k boundary is within the bounds).
  const bool fast = !logits && T > 256 && n_expert <= 256 && d_model % 64 == 0;
  const size_t need = fast     ? lay.rlist + align256(sizeof(int32_t) * ((size_t)T + 64))
                      : logits ? sizeof(WsHeader)
                               : lay.logits + align256(sizeof(float) * (size_t)T * n_expert);
  if (ws_bytes < need) return DS4MOE_ESPACE;
  float *lg = logits ? logits : ws_ptr<float>(ws, lay.logits);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T <= 256 && n_expert <= 256 && d_model <= 8192) {
    WsHeader *hdr = static_cast<WsHeader *>(ws);
    ProfScope prof("route_topk", s);
    const int ni = (d_model + 1023) / 1024;
    auto kern = ni <= 1   ? k_route_small<1, kRouteTopk>
                : ni <= 2 ? k_route_small<2, kRouteTopk>
                : ni <= 4 ? k_route_small<4, kRouteTopk>
                          : k_route_small<8, kRouteTopk>;
    return cuda_status(launch_pdl(kern, dim3(n_expert), dim3(256), 0, s, x, Wr, bias, (int)T, (int)d_model,
                                  (int)n_expert, (int)k, lg, idx, w, hdr, BucketArgs{}));
  }
  if (fast) {
    float *xn = ws_ptr<float>(ws, lay.rnorm), *wn = xn + T;
    int32_t *cnt = ws_ptr<int32_t>(ws, lay.rlist), *list = cnt + 64;
    const int n_chain = 64 + d_model / 64 + 2;
    const float gam = (float)(n_chain * 0x1p-24 / (1.0 - n_chain * 0x1p-24));
    cudaError_t e;
    {
      ProfScope prof("router_norms", s);
      k_row_norms<<<num_sms() * 4, 256, 0, s>>>(x, T, Wr, n_expert, d_model, xn, wn);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    }
    {
      ProfScope prof("router_approx", s);
      k_router_approx<<<dim3((n_expert + kRT - 1) / kRT, (T + kRT - 1) / kRT), 256, 0, s>>>(x, Wr, T, d_model,
                                                                                         n_expert, lg);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    }
    if ((e = cudaMemsetAsync(cnt, 0, sizeof(int32_t), s)) != cudaSuccess) return cuda_status(e);
    {
      ProfScope prof("topk_cert", s);
      const int grid = (T + 7) / 8 < num_sms() * 8 ? (T + 7) / 8 : num_sms() * 8;
      k_topk_cert<<<grid, 256, 0, s>>>(lg, bias, xn, wn, x, Wr, T, d_model, n_expert, k, gam, idx, w, list, cnt);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    }
    {
      ProfScope prof("router_exact_tail", s);
      k_router_logits<<<num_sms() * 8, 256, 0, s>>>(x, Wr, bias, T, d_model, n_expert, lg, list, cnt);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
      k_topk_softmax<<<num_sms() * 2, 256, 0, s>>>(lg, T, n_expert, k, idx, w, list, cnt);
    }
    return cuda_status(cudaGetLastError());
  }
  const int64_t warps = (int64_t)T * n_expert;
  {
    ProfScope prof("router_logits", s);
    k_router_logits<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(x, Wr, bias, T, d_model, n_expert, lg);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  {
    ProfScope prof("topk_softmax", s);
    k_topk_softmax<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(lg, T, n_expert, k, idx, w);
  }
  return cuda_status(cudaGetLastError());
}

ds4moe_status ds4moe_route_topk_select_bias(const uint16_t *x, const float *Wr, const float *bias, int32_t T,
                                            int32_t d_model, int32_t n_expert, int32_t k, int32_t *idx, float *w,
                                            float *logits, void *ws, size_t ws_bytes, void *stream) {
  if (T < 0 || d_model <= 0 || d_model % 4 || n_expert < 1 || n_expert > 256 || k < 1 || k > 32 ||
      k > n_expert)
    return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!x || !Wr || !bias || !idx || !w || !ws) return DS4MOE_EINVAL;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(bias) || !aligned16(idx) || !aligned16(w) || !aligned16(ws) ||
      (logits && !aligned16(logits)))
    return DS4MOE_EINVAL;
  if ((int64_t)d_model * 2 % 16) return DS4MOE_EINVAL;
  ds4moe_layer shape{};
  shape.d_model = d_model;
  shape.d_ff = 16;
  shape.n_expert = n_expert;
  const WsLayout lay = ws_layout(shape, T, k, 0);
  const size_t plane = align256(sizeof(float) * (size_t)T * n_expert);
  if (ws_bytes < lay.logits + (logits ? 1 : 2) * plane) return DS4MOE_ESPACE;
  float *lb = ws_ptr<float>(ws, lay.logits);
  float *lu = logits ? logits : ws_ptr<float>(ws, lay.logits + plane);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t warps = (int64_t)T * n_expert;
  {
    ProfScope prof("router_logits_both", s);
    const int64_t blocks = (warps + 7) / 8;
    k_router_logits_both<<<(unsigned)(blocks < num_sms() * 64 ? blocks : num_sms() * 64), 256, 0, s>>>(
        x, Wr, bias, T, d_model, n_expert, lb, lu);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  {
    ProfScope prof("topk_selbias", s);
    const int blocks = (T + 7) / 8;
    k_topk_selbias<<<blocks < num_sms() * 8 ? blocks : num_sms() * 8, 256, 0, s>>>(lb, lu, T, n_expert, k, idx, w);
  }
  return cuda_status(cudaGetLastError());
}

ds4moe_status ds4moe_ffn_decode(const ds4moe_layer *L, const uint16_t *x, const int32_t *idx,
                                const float *w, int32_t T, int32_t k, float *out, void *ws,
                                size_t ws_bytes, void *stream) {
  return run_ffn(false, L, x, idx, w, T, k, out, ws, ws_bytes, stream);
}

ds4moe_status ds4moe_ffn_prefill(const ds4moe_layer *L, const uint16_t *x, const int32_t *idx,
                                 const float *w, int32_t T, int32_t k, float *out, void *ws,
                                 size_t ws_bytes, void *stream) {
  return run_ffn(true, L, x, idx, w, T, k, out, ws, ws_bytes, stream);
}

// ds4moe_moe_decode's body; with `nf` (one token on tile-order weights
// only), the router grid forms the layer input itself from the residual
// stream (NormFuse) instead of reading x.
static ds4moe_status moe_decode_impl(const ds4moe_layer *L, const uint16_t *x, const float *Wr, const float *bias,
                                     int32_t T, int32_t k, float *out, int32_t *idx, float *w, void *ws,
                                     size_t ws_bytes, void *stream, const NormFuse *nf) {
  ds4moe_status st = check_layer(L);
  if (st != DS4MOE_OK) return st;
  const int E = L->n_expert, D = L->d_model;
  if (T < 0 || k < 1 || k > 32 || k > E) return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!x || !Wr || !out || !idx || !w || !ws) return DS4MOE_EINVAL;
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(out) || !aligned16(idx) || !aligned16(w) || !aligned16(ws) ||
      (bias && !aligned16(bias)))
    return DS4MOE_EINVAL;
  const WsLayout lay = ws_layout(*L, T, k, 0);
  if (ws_bytes < lay.total) return DS4MOE_ESPACE;
  const bool r16 = layer_r16(*L);
  if (r16 && (T != 1 || !t1r_ok(*L, k))) return DS4MOE_EUNSUPPORTED;
  if (nf && (!r16 || D > 4096 || !nf->res || !nf->add || !nf->res_next || nf->x != x || !aligned16(nf->res) ||
             !aligned16(nf->add) || !aligned16(nf->res_next) || nf->res == nf->res_next))
    return DS4MOE_EINVAL;
  if (!r16 && (T > 256 || E > 256 || D > 8192 || D % 8)) {
    // the two-call path gives the same results for shapes the fused router does not cover
    st = ds4moe_route_topk(x, Wr, bias, T, D, E, k, idx, w, nullptr, ws, ws_bytes, stream);
    if (st != DS4MOE_OK) return st;
    return run_ffn(false, L, x, idx, w, T, k, out, ws, ws_bytes, stream);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float *lg = ws_ptr<float>(ws, lay.logits);
  const cudaError_t ea = chain_attributes();
  if (ea != cudaSuccess) return cuda_status(ea);
  if (T == 1 && (r16 || t1_chain_ok(*L))) {
    // one token on the single-token kernels: the router grid only writes the
    // logits, and every CTA of the FFN grids ranks the experts itself (no
    // grid waits on one CTA's ranking)
    ProfScope prof("route", s);
    const int ni = (D + 1023) / 1024;
    auto kern = ni <= 1   ? k_route_small<1, kRouteLogits>
                : ni <= 2 ? k_route_small<2, kRouteLogits>
                : ni <= 4 ? k_route_small<4, kRouteLogits>
                          : k_route_small<8, kRouteLogits>;
    BucketArgs zero{};
    zero.counts = ws_ptr<int32_t>(ws, lay.counts);  // one counter per expert, zeroed by CTA e
    zero.zero2 = ws_ptr<int32_t>(ws, lay.cnt);       // the merged grid's combine counters
    zero.nzero2 = (D + 63) / 64;
    if (r16) {  // the tile-order grid's hidden words: every call starts them untagged
      zero.zero3 = ws_ptr<int32_t>(ws, lay.h);
      zero.nzero3 = k * L->d_ff;
    }
    if (nf) {
      zero.nrm_res = nf->res;
      zero.nrm_add = nf->add;
      zero.nrm_res_next = nf->res_next;
      zero.nrm_x = nf->x;
      zero.nrm_eps = nf->eps;
    }
    const cudaError_t e = launch_pdl(kern, dim3(E), dim3(256), 0, s, x, Wr, bias, (int)T, (int)D, (int)E, (int)k, lg,
                                     idx, w, static_cast<WsHeader *>(ws), zero);
    if (e != cudaSuccess) return cuda_status(e);
    // with nf the router grid writes x: the FFN grid reads it after its dependency wait
    return run_ffn(false, L, x, idx, w, T, k, out, ws, ws_bytes, stream, lg, /*bucketed=*/true, /*route_t1=*/true,
                   /*x_converted=*/false, /*x_late=*/nf != nullptr);
  }
  // up to 32 pairs: the router's last CTA also does the bucketing
  const bool fused = T * k <= 32;
  {
    ProfScope prof(fused ? "route_bucket" : "route", s);
    const int ni = (D + 1023) / 1024;
    cudaError_t e;
    if (fused) {
      auto kern = ni <= 1   ? k_route_small<1, kRouteBucket>
                  : ni <= 2 ? k_route_small<2, kRouteBucket>
                  : ni <= 4 ? k_route_small<4, kRouteBucket>
                            : k_route_small<8, kRouteBucket>;
      e = launch_pdl(kern, dim3(E), dim3(256), 0, s, x, Wr, bias, (int)T, (int)D, (int)E, (int)k, lg, idx, w,
                     static_cast<WsHeader *>(ws), bucket_args(*L, ws, lay, x, idx, w, T, k, out, decode_mma_ok(*L)));
    } else {
      auto kern = ni <= 1   ? k_route_small<1, kRouteLogits>
                  : ni <= 2 ? k_route_small<2, kRouteLogits>
                  : ni <= 4 ? k_route_small<4, kRouteLogits>
                            : k_route_small<8, kRouteLogits>;
      BucketArgs cv{};  // the router grid also converts x for the multi-token kernels
      if (decode_mma_ok(*L)) {
        cv.x16 = ws_ptr<uint16_t>(ws, lay.x16);
        cv.xs16 = ws_ptr<uint8_t>(ws, lay.xs16);
        cv.xs32 = ws_ptr<float>(ws, lay.xs32);
      }
      e = launch_pdl(kern, dim3(E), dim3(256), 0, s, x, Wr, bias, (int)T, (int)D, (int)E, (int)k, lg, idx, w,
                     static_cast<WsHeader *>(ws), cv);
    }
    if (e != cudaSuccess) return cuda_status(e);
  }
  return run_ffn(false, L, x, idx, w, T, k, out, ws, ws_bytes, stream, lg, fused, false,
                 !fused && decode_mma_ok(*L));
}

ds4moe_status ds4moe_moe_decode(const ds4moe_layer *L, const uint16_t *x, const float *Wr, const float *bias,
                               int32_t T, int32_t k, float *out, int32_t *idx, float *w, void *ws,
                               size_t ws_bytes, void *stream) {
  return moe_decode_impl(L, x, Wr, bias, T, k, out, idx, w, ws, ws_bytes, stream, nullptr);
}

ds4moe_status ds4moe_gather_rows(const uint16_t *x, const int32_t *rows, int32_t n, int32_t d_model,
                                uint16_t *dst, void *stream) {
  if (n < 0 || d_model <= 0 || d_model % 8) return DS4MOE_EINVAL;
  if (n == 0) return DS4MOE_OK;
  if (!x || !rows || !dst || !aligned16(x) || !aligned16(dst)) return DS4MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nc = d_model / 8;
  const int64_t total = (int64_t)n * nc;
  ProfScope prof("gather_rows", s);
  k_gather_rows<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(reinterpret_cast<const uint4 *>(x), rows, (int)n, nc,
                                                                reinterpret_cast<uint4 *>(dst));
  return cuda_status(cudaGetLastError());
}

ds4moe_status ds4moe_combine_pairs(const float *y, const int32_t *pos, const float *w, int32_t T, int32_t k,
                                   int32_t d_model, float *out, void *stream) {
  if (T < 0 || k < 1 || k > 32 || d_model <= 0) return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!pos || !w || !out) return DS4MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t total = (int64_t)T * d_model;
  ProfScope prof("combine_pairs", s);
  k_combine_pairs<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(y, pos, w, (int)T, (int)k, (int)d_model, out);
  return cuda_status(cudaGetLastError());
}

ds4moe_status ds4moe_residual_norm(float *x_res, const float *out, uint16_t *x_next, int32_t T, int32_t d_model,
                                   float eps, void *stream) {
  if (T < 0 || d_model <= 0 || d_model % 4 || !(eps >= 0.f)) return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  if (!x_res || !x_next || !aligned16(x_res) || !aligned16(x_next) || (out && !aligned16(out)))
    return DS4MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope prof("residual_norm", s);
  return cuda_status(launch_pdl(k_residual_norm, dim3(T), dim3(kNormThreads), 0, s, x_res, out, x_next,
                                (int)d_model, eps, static_cast<const float *>(nullptr)));
}

ds4moe_status ds4moe_stack_decode(const ds4moe_layer *layers, const float *const *Wr, const float *const *bias,
                                  int32_t n_layers, int32_t T, int32_t k, float eps, float *x_res, uint16_t *x_bf16,
                                  float *out, int32_t *idx, float *w, void *ws, size_t ws_bytes, void *stream) {
  if (!layers || !Wr || n_layers < 1) return DS4MOE_EINVAL;
  if (T < 0 || k < 1 || k > 32) return DS4MOE_EINVAL;
  for (int l = 0; l < n_layers; ++l) {  // validate everything before launching anything
    const ds4moe_status st = check_layer(&layers[l]);
    if (st != DS4MOE_OK) return st;
    if (layers[l].d_model != layers[0].d_model || !Wr[l] || k > layers[l].n_expert) return DS4MOE_EINVAL;
    if (layer_r16(layers[l]) && (T != 1 || !t1r_ok(layers[l], k))) return DS4MOE_EUNSUPPORTED;
    if (ws_bytes < ws_layout(layers[l], T, k, 0).total) return DS4MOE_ESPACE;
  }
  if (T == 0) return DS4MOE_OK;
  if (!idx || !w || !aligned16(idx) || !aligned16(w)) return DS4MOE_EINVAL;
  const int D = layers[0].d_model;
  const size_t ldk = ((size_t)T * k + 3) & ~size_t(3);
  ds4moe_status st = ds4moe_residual_norm(x_res, nullptr, x_bf16, T, D, eps, stream);
  // one token over tile-order layers: each layer after the first forms its
  // input inside its router grid (residual add + norm of the previous
  // layer's output), the residual alternating between x_res and a
  // workspace buffer; the last layer's add + norm runs as its own grid
  bool fuse = T == 1 && D <= 4096;
  for (int l = 0; l < n_layers; ++l) fuse = fuse && layer_r16(layers[l]);
  // the second buffer past every layer's other regions (each layer's
  // workspace check covers its own offset plus the buffer)
  size_t res2 = 0;
  for (int l = 0; l < n_layers; ++l) res2 = std::max(res2, ws_layout(layers[l], T, k, 0).res2);
  float *res[2] = {x_res, ws_ptr<float>(ws, res2)};
  int cur = 0;
  for (int l = 0; l < n_layers && st == DS4MOE_OK; ++l) {
    if (fuse && l > 0) {
      const NormFuse nf{res[cur], out, res[cur ^ 1], x_bf16, eps};
      st = moe_decode_impl(&layers[l], x_bf16, Wr[l], bias ? bias[l] : nullptr, T, k, out, idx + l * ldk,
                           w + l * ldk, ws, ws_bytes, stream, &nf);
      cur ^= 1;
    } else {
      st = ds4moe_moe_decode(&layers[l], x_bf16, Wr[l], bias ? bias[l] : nullptr, T, k, out, idx + l * ldk,
                             w + l * ldk, ws, ws_bytes, stream);
      if (st == DS4MOE_OK && !fuse) st = ds4moe_residual_norm(x_res, out, x_bf16, T, D, eps, stream);
    }
  }
  if (st == DS4MOE_OK && fuse) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ProfScope prof("residual_norm", s);
    st = cuda_status(launch_pdl(k_residual_norm, dim3(T), dim3(kNormThreads), 0, s, x_res, static_cast<const float *>(out),
                                x_bf16, (int)D, eps, cur ? static_cast<const float *>(res[1]) : nullptr));
  }
  return st;
}

ds4moe_status ds4moe_stream_status(void *ws, void *stream) {
  if (!ws || !aligned16(ws)) return DS4MOE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t st = 0;
  cudaError_t e = cudaMemcpyAsync(&st, ws, sizeof(st), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_status(e);
  if (st != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyAsync(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return static_cast<ds4moe_status>(st);
}

}  // extern "C"

// ======================================================= allocation-free
// ds4moe_ffn_decode_noalloc: the decode FFN for callers that cannot allocate
// device memory themselves (see include/ds4moe.h).  Its scratch is this
// file-scope device array instead of a caller-provided workspace.  Host code
// must not pass the array's name to a kernel: on the host it is only a
// stand-in for the device symbol, so the device address is looked up once
// per device with cudaGetSymbolAddress and cached.
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // DS4MOE_NOALLOC_SCRATCH_BYTES
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

ds4moe_status noalloc_scratch(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return DS4MOE_ECUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (!p) return DS4MOE_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return DS4MOE_OK;
}

}  // namespace

extern "C" ds4moe_status ds4moe_ffn_decode_noalloc(const ds4moe_layer *L, const uint16_t *x,
                                                   const int32_t *idx, const float *w, int32_t T,
                                                   int32_t k, float *out, int32_t *status_out,
                                                   void *stream) {
  ds4moe_status st = check_layer(L);
  if (st != DS4MOE_OK) return st;
  if (T < 0 || k < 1 || k > 32 || k > L->n_expert) return DS4MOE_EINVAL;
  if (T == 0) return DS4MOE_OK;
  const size_t need = ws_layout(*L, T, k, 0).total;
  if (need > kNoAllocScratchBytes) {
    fprintf(stderr,
            "ds4moe_ffn_decode_noalloc: T=%d k=%d d_model=%d d_ff=%d n_expert=%d needs %zu bytes of "
            "scratch, above the fixed %zu-byte array; use ds4moe_ffn_decode with a workspace\n",
            T, k, L->d_model, L->d_ff, L->n_expert, need, kNoAllocScratchBytes);
    return DS4MOE_ESPACE;
  }
  void *scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != DS4MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's bytes: the status word and counters
  // in its header must start at zero; every other region is written before
  // it is read within a call
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(WsHeader), s);
  if (e != cudaSuccess) return cuda_status(e);
  st = run_ffn(false, L, x, idx, w, T, k, out, scratch, kNoAllocScratchBytes, stream);
  if (st != DS4MOE_OK) return st;
  if (status_out) {
    e = cudaMemcpyAsync(status_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return DS4MOE_OK;
}

