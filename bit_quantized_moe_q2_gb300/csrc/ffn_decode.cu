// Expert FFN for decode batches: dequant-fused GEMV over Q4_1 / Q2_K rows,
// gate+up fused with SwiGLU, then down, then the weighted combine.
#include "internal.cuh"

namespace ds4 {
namespace {

constexpr int kTok = 8;  // tokens handled per pass over a weight row

// Lane-partial dot products of one quantized row with up to kTok input rows.
// in(t, j) returns input value j of token slot t as fp32.
// Q4_1 ([Q41] "Q4_1 블록이 어떻게 생겼나"): y = d*q + m, value j low nibble of
// qs[j], value j+16 high nibble.
template <typename In>
__device__ __forceinline__ void row_dot_q41(const uint8_t *__restrict__ row, int cols, int nt, In in,
                                            float (&acc)[kTok]) {
  const int lane = threadIdx.x & 31;
  const int nb = cols / 32;
  for (int b = lane; b < nb; b += 32) {
    const uint8_t *p = row + (int64_t)b * kQ41Bytes;
    const float d = f16_bits_to_f32(p[0] | (p[1] << 8));
    const float m = f16_bits_to_f32(p[2] | (p[3] << 8));
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const uint32_t q = p[4 + j];
      const float w0 = fmaf(d, (float)(q & 15u), m), w1 = fmaf(d, (float)(q >> 4), m);
#pragma unroll
      for (int t = 0; t < kTok; ++t)
        if (t < nt) acc[t] = fmaf(w1, in(t, 32 * b + j + 16), fmaf(w0, in(t, 32 * b + j), acc[t]));
    }
  }
}

// Q2_K ([DS4-2] layout table / qs packing): qs byte 32h+l holds values
// 128h + l + 32s at bits 2s; sub-block n = v/16 has scale byte sc | mn << 4;
// y = d*sc*q - dmin*mn.
template <typename In>
__device__ __forceinline__ void row_dot_q2k(const uint8_t *__restrict__ row, int cols, int nt, In in,
                                            float (&acc)[kTok]) {
  const int lane = threadIdx.x & 31;
  const int nitems = cols / 256 * 64;
  for (int it = lane; it < nitems; it += 32) {
    const int b = it >> 6, by = it & 63, h = by >> 5, l = by & 31;
    const uint8_t *p = row + (int64_t)b * kQ2KBytes;
    const float d = f16_bits_to_f32(p[80] | (p[81] << 8));
    const float dmin = f16_bits_to_f32(p[82] | (p[83] << 8));
    const uint32_t q = p[16 + by];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int v = 128 * h + l + 32 * s;
      const uint32_t scb = p[v >> 4];
      const float wv = fmaf(d * (float)(scb & 15u), (float)((q >> (2 * s)) & 3u), -(dmin * (float)(scb >> 4)));
#pragma unroll
      for (int t = 0; t < kTok; ++t)
        if (t < nt) acc[t] = fmaf(wv, in(t, 256 * b + v), acc[t]);
    }
  }
}

template <typename In>
__device__ __forceinline__ void row_dot(int q, const uint8_t *row, int cols, int nt, In in, float (&acc)[kTok]) {
  if (q == DS4MOE_Q4_1) row_dot_q41(row, cols, nt, in, acc);
  else row_dot_q2k(row, cols, nt, in, acc);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// gate/up + SwiGLU: one warp per (active expert, hidden row r), all pairs of
// that expert in passes of kTok tokens.  h[pos, r] = bf16(silu(g) * u) where
// pos is the pair's position in expert-sorted order.
__global__ void __launch_bounds__(256) k_gate_up_simt(FfnArgs a) {
  const int D = a.L.d_model, F = a.L.d_ff, k = a.k;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)a.hdr->n_active * F;
  const int64_t rbg = row_bytes(a.L.q_gate, D), rbu = row_bytes(a.L.q_up, D);
  for (int64_t item = gw; item < items; item += nw) {
    const int ai = (int)(item / F), r = (int)(item % F);
    const int e = a.active[ai];
    const int pb = a.offs[e], pe = a.offs[e + 1];
    const uint8_t *grow = static_cast<const uint8_t *>(a.L.gate) + ((int64_t)e * F + r) * rbg;
    const uint8_t *urow = static_cast<const uint8_t *>(a.L.up) + ((int64_t)e * F + r) * rbu;
    for (int p0 = pb; p0 < pe; p0 += kTok) {
      const int nt = min(kTok, pe - p0);
      const uint16_t *xr[kTok];
#pragma unroll
      for (int t = 0; t < kTok; ++t) xr[t] = a.x + (int64_t)(a.perm[p0 + (t < nt ? t : 0)] / k) * D;
      auto in = [&](int t, int j) { return bf16_bits_to_f32(xr[t][j]); };
      float ag[kTok] = {}, au[kTok] = {};
      row_dot(a.L.q_gate, grow, D, nt, in, ag);
      row_dot(a.L.q_up, urow, D, nt, in, au);
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        const float g = warp_sum(ag[t]), u = warp_sum(au[t]);
        if (lane == t && t < nt) a.h[(int64_t)(p0 + t) * F + r] = f32_to_bf16_bits(silu(g) * u);
      }
    }
  }
}

// down: one warp per (active expert, output row c); y[pos, c] = W2[e][c] . h[pos]
__global__ void __launch_bounds__(256) k_down_simt(FfnArgs a) {
  const int D = a.L.d_model, F = a.L.d_ff;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)a.hdr->n_active * D;
  const int64_t rbd = row_bytes(a.L.q_down, F);
  for (int64_t item = gw; item < items; item += nw) {
    const int ai = (int)(item / D), c = (int)(item % D);
    const int e = a.active[ai];
    const int pb = a.offs[e], pe = a.offs[e + 1];
    const uint8_t *drow = static_cast<const uint8_t *>(a.L.down) + ((int64_t)e * D + c) * rbd;
    for (int p0 = pb; p0 < pe; p0 += kTok) {
      const int nt = min(kTok, pe - p0);
      const uint16_t *hr = a.h + (int64_t)p0 * F;
      auto in = [&](int t, int j) { return bf16_bits_to_f32(hr[(int64_t)t * F + j]); };
      float ay[kTok] = {};
      row_dot(a.L.q_down, drow, F, nt, in, ay);
#pragma unroll
      for (int t = 0; t < kTok; ++t) {
        const float yv = warp_sum(ay[t]);
        if (lane == t && t < nt) a.y[(int64_t)(p0 + t) * D + c] = yv;
      }
    }
  }
}

// out[t, c] = sum_{i<k} w[t,i] * y[inv[t,i], c], in rank order.
__global__ void k_combine(FfnArgs a) {
  const int D = a.L.d_model, k = a.k;
  const int64_t n4 = (int64_t)a.T * D / 4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = (i * 4) / D;
    const int c = (int)((i * 4) % D);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int pos = a.inv[t * k + j];
      if (pos < 0) continue;
      const float wt = a.w[t * k + j];
      const float4 yv = *reinterpret_cast<const float4 *>(a.y + (int64_t)pos * D + c);
      acc.x = fmaf(wt, yv.x, acc.x);
      acc.y = fmaf(wt, yv.y, acc.y);
      acc.z = fmaf(wt, yv.z, acc.z);
      acc.w = fmaf(wt, yv.w, acc.w);
    }
    *reinterpret_cast<float4 *>(a.out + t * D + c) = acc;
  }
}

}  // namespace

cudaError_t launch_ffn_decode(const FfnArgs &a, cudaStream_t s) {
  const int grid = num_sms() * 8;
  {
    ProfScope p("gate_up", s);
    k_gate_up_simt<<<grid, 256, 0, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    ProfScope p("down", s);
    k_down_simt<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const FfnArgs &a, cudaStream_t s) {
  const int64_t n4 = (int64_t)a.T * a.L.d_model / 4;
  const int grid = (int)((n4 + 255) / 256 < num_sms() * 16 ? (n4 + 255) / 256 : num_sms() * 16);
  {
    ProfScope p("combine", s);
    k_combine<<<grid, 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace ds4
