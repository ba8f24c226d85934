// Single-token (T = 1) decode over Q2_K weights in the 16-row tile order
// (DS4MOE_Q2_K_R16): the same 84 bytes per 256 values as the Q2_K block of
// "【#2】ds4.c 해독하기" (layout table: scales, qs, d, dmin), with the bytes of
// every 16 consecutive rows of one block column permuted so that each lane
// of a warp reads its tensor-core operands with one 16-byte load.
#pragma once

#include "internal.cuh"
#include "ptx.cuh"

namespace ds4 {

// ------------------------------------------------------------ tile order
// A tile-block is 16 rows x one 256-value block column: 16 * 84 = 1344
// bytes, at the byte offset the 16 rows' blocks of that column would take in
// the plain layout (a 16-row tile of a matrix stays where it was; a tile is
// its tile-blocks in column order).  Within a tile-block (lane L = 4 g + c,
// rows g and g + 8, sub-blocks s = 0 .. 15 of 16 values):
//   [0, 1024)     codes.  Half h (values 128 h .. 128 h + 127) of lane L:
//                 16 bytes at 512 h + 16 L, four words
//                   (row g, s = 8h + c), (row g+8, 8h + c),
//                   (row g, 8h + c + 4), (row g+8, 8h + c + 4);
//                 value v (0 .. 15) of a sub-block sits at bit
//                 16 (v & 1) + 2 (v >> 1) of its word.
//   [1024, 1280)  scale bytes (sc | mn << 4).  Lane L: 8 bytes at 1024 + 8 L,
//                 words for rows g and g + 8, each
//                   b(2c) | b(2c + 8) << 8 | b(2c + 1) << 16 | b(2c + 9) << 24.
//   [1280, 1344)  row r's fp16 d and dmin at 1280 + 4 r (as in the block).
constexpr uint32_t kR16Rows = 16;
constexpr uint32_t kR16TileBlock = kR16Rows * kQ2KBytes;  // 1344
constexpr uint32_t kR16Scales = 1024, kR16Dmin = 1280;

// Bit position of value v of a sub-block in its code word.
__host__ __device__ constexpr uint32_t r16_code_bit(uint32_t v) { return 16u * (v & 1u) + 2u * (v >> 1); }

// ------------------------------------------------------ operand scheme
// mma.sync.m16n8k16 (A 16 x 16 row-major, B 16 x 8, fp32 D).  Per 128-value
// half of a block, K slots 2n, 2n + 1 of every MMA carry two values of
// sub-block n of the half and the activation operand is block-diagonal
// (column n is non-zero only in slots 2n, 2n + 1), so after the eight MMAs
// of a half D[row][n] is the code-dot of sub-block n alone; its scale is one
// fp32 FMA per 16 weights, and the minima are one more MMA per block.
//
// MMA i (0 .. 7) of a half takes values 2i, 2i + 1 of every sub-block.  Its
// A registers are code words masked to the field of value 2i (low half) and
// 2i + 1 (high half): for i < 5 the field at bits 2i and 16 + 2i, for i >= 5
// the word shifted right by 10 and the field at 2 (i - 5).  A 2-bit field at
// bit 2e of an fp16 half is the subnormal q * 2^(2e - 24), exact, so each A
// register costs one AND (and every fifth a shift).  The activation operand
// of MMA i carries x * 2^(8 - 2 e_i + sigma): every product is then
// q * x * 2^(sigma - 16), whatever the field position.  sigma <= 0 keeps the
// largest operand below 2^16 (exact binary16), sigma = 0 whenever
// max |x| < 128.
__host__ __device__ constexpr int r16_field(int i) { return i < 5 ? i : i - 5; }

// Activation operands of one 256-value block: x[h][i] for MMA i of half h
// (b0, b1), m for the minima MMA (columns 0 / 1: hi / lo parts of the 16
// sub-block sums), and the factors that undo the operand scaling.
struct R16B {
  uint32_t x[2][8][2];
  uint32_t m[2];
  float k1;  // 2^(40 - sigma): D * sc-as-subnormal -> exact units
  float k2;  // 2^(20 - sigma_m): minima MMA -> exact units
};

__device__ __forceinline__ float2 r16_h2_to_f2(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, sizeof(h));
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t r16_pack_h2(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// src: the block's 256 activations as bf16 bit patterns, in device memory
// (read through L2) or, with SMEM, in shared memory.  Lane (g, c) owns
// sub-block g of each half when g == c (b0) or g == c + 4 (b1); every lane
// reads sub-block 8h + g so that the block maximum is a plain warp reduction.
template <bool SMEM = false>
__device__ __forceinline__ void r16_load_b(R16B &B, const uint16_t *__restrict__ src, int g, int c) {
  float v[2][16];
  float mx = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 *p = reinterpret_cast<const uint4 *>(src + 16 * (8 * h + g));
    const uint4 q0 = SMEM ? p[0] : __ldcg(p);
    const uint4 q1 = SMEM ? p[1] : __ldcg(p + 1);
    const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[h][i] = bf16_bits_to_f32((wd[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
      mx = fmaxf(mx, fabsf(v[h][i]));
    }
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  // exponent of the block maximum (0 for a zero block; NaN / inf clamp)
  const int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 : -127;
  const int sig = max(-60, min(0, 7 - ex)), sigm = max(-60, min(0, 10 - ex));
  B.k1 = __uint_as_float((uint32_t)(127 + 40 - sig) << 23);
  B.k2 = __uint_as_float((uint32_t)(127 + 20 - sigm) << 23);
  const bool own0 = g == c, own1 = g == c + 4;
  uint32_t shl[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += v[h][i];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = __uint_as_float((uint32_t)(127 + 8 - 2 * r16_field(i) + sig) << 23);
      const uint32_t p = r16_pack_h2(v[h][2 * i] * f, v[h][2 * i + 1] * f);
      B.x[h][i][0] = own0 ? p : 0u;
      B.x[h][i][1] = own1 ? p : 0u;
    }
    // hi / lo binary16 parts of the scaled sub-block sum
    const float ss = s * __uint_as_float((uint32_t)(127 + sigm) << 23);
    const __half hi = __float2half_rn(ss);
    const __half lo = __float2half_rn(ss - __half2float(hi));
    shl[h] = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
  }
  // minima operand: K slot s = sub-block s of the block; lane (g, c) holds
  // slots 2c, 2c + 1 (b0) and 2c + 8, 2c + 9 (b1) of column g (0: hi, 1: lo)
  const int sh = 16 * (g & 1);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t a = __shfl_sync(0xffffffffu, shl[h], 8 * c);      // sub-block 8h + 2c
    const uint32_t b = __shfl_sync(0xffffffffu, shl[h], 8 * c + 4);  // sub-block 8h + 2c + 1
    const uint32_t p = ((a >> sh) & 0xFFFFu) | (((b >> sh) & 0xFFFFu) << 16);
    B.m[h] = g < 2 ? p : 0u;
  }
}

// Sum over the four lanes of a quad (the c index).
__device__ __forceinline__ float r16_quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// One 256-value block column of NM tile-blocks (tb[m], shared memory) against
// one activation block: this lane's share of
//   d * sum(sc * q * x) - dmin * sum(mn * xsum)
// for rows g (y[m][0]) and g + 8 (y[m][1]); a quad sum over c completes it.
template <int NM>
__device__ __forceinline__ void r16_block(const uint8_t *const (&tb)[NM], int g, int lane, const R16B &B,
                                          float (&y)[NM][2]) {
  uint32_t S[NM][2], dd[NM][2];
  float sacc[NM][2];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const uint2 s2 = *reinterpret_cast<const uint2 *>(tb[m] + kR16Scales + 8 * lane);
    S[m][0] = s2.x;
    S[m][1] = s2.y;
    dd[m][0] = ptx::lds32(tb[m] + kR16Dmin + 4 * g);
    dd[m][1] = ptx::lds32(tb[m] + kR16Dmin + 4 * (g + 8));
    sacc[m][0] = sacc[m][1] = 0.f;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 W[NM], Ws[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      W[m] = *reinterpret_cast<const uint4 *>(tb[m] + 512 * h + 16 * lane);
      Ws[m] = make_uint4(W[m].x >> 10, W[m].y >> 10, W[m].z >> 10, W[m].w >> 10);
    }
    float C[NM][4];
#pragma unroll
    for (int m = 0; m < NM; ++m) C[m][0] = C[m][1] = C[m][2] = C[m][3] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t mask = 0x00030003u << (2 * r16_field(i));
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint4 &w = i < 5 ? W[m] : Ws[m];
        const uint32_t A[4] = {w.x & mask, w.y & mask, w.z & mask, w.w & mask};
        ptx::mma_f16(C[m], A, B.x[h][i][0], B.x[h][i][1]);
      }
    }
    // sc of sub-blocks 8h + 2c, 8h + 2c + 1 as fp16 subnormals sc * 2^-24
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint32_t s0 = (h ? S[m][0] >> 8 : S[m][0]) & 0x000F000Fu;
      const uint32_t s1 = (h ? S[m][1] >> 8 : S[m][1]) & 0x000F000Fu;
      const float2 f0 = r16_h2_to_f2(s0), f1 = r16_h2_to_f2(s1);
      sacc[m][0] = fmaf(f0.x, C[m][0], fmaf(f0.y, C[m][1], sacc[m][0]));
      sacc[m][1] = fmaf(f1.x, C[m][2], fmaf(f1.y, C[m][3], sacc[m][1]));
    }
  }
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    // minima: mn * 2^-20 (high nibbles) against the sub-block sums
    const uint32_t Am[4] = {S[m][0] & 0x00F000F0u, S[m][1] & 0x00F000F0u, (S[m][0] >> 8) & 0x00F000F0u,
                            (S[m][1] >> 8) & 0x00F000F0u};
    float M[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_f16(M, Am, B.m[0], B.m[1]);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float2 dm = r16_h2_to_f2(dd[m][r]);
      y[m][r] = fmaf(dm.x * B.k1, sacc[m][r], -(dm.y * B.k2) * (M[2 * r] + M[2 * r + 1]));
    }
  }
}

}  // namespace ds4
