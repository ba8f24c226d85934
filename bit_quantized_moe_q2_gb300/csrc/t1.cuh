// Single-token (T = 1) decode building blocks shared by the stand-alone
// FFN kernels and the fused layer kernel.
#pragma once

#include "internal.cuh"
#include "ptx.cuh"
#include "route.cuh"

namespace ds4 {

// ================================================== single-token decode
// With one token (T = 1) every expert group holds one pair, and the n = 8
// side of the MMA is better spent on eight Q2_K sub-blocks than on tokens.
// Per 128-value half of a 256-value block, K slots 2n, 2n+1 of every MMA
// carry two values of sub-block n, and the activation operand is placed
// block-diagonally (column n sees only K slots 2n, 2n+1), so after the eight
// MMAs of a half, D[row][n] is the code-dot of sub-block n alone.  The
// per-(row, sub-block) scale is then one fp32 FMA per 16 weights in the
// epilogue, and the mins one more MMA per block (mn codes x sub-block sums).
//
// Codes enter as fp16 subnormals: masking the 2-bit field at bit 2p of the
// low byte of each fp16 half leaves q * 2^(2p - 24) exactly, one LOP per
// operand register; the power of two is folded into the block scale.  Lane
// quad c handles sub-blocks c and c + 4 of a half, which share the qs bytes
// 16 (c & 1) .. +15 at code positions c / 2 and c / 2 + 2, and D columns
// 2c, 2c+1, which both sit at code position c.
//
// Each consumer warp owns one 256-value block column of K and keeps its
// activation operands in registers; a producer warp streams 16-row tiles
// into a ring of shared-memory stages with bulk copies.
struct T1Lane {
  uint32_t m1, m2;  // code fields at positions c/2 and c/2 + 2, both fp16 halves
  uint32_t qoff;    // this lane's 16 qs bytes within a 32-byte half
  uint32_t rot;     // word order rotation of lanes with odd c (spreads banks)
  uint32_t soff;    // scale word holding bytes 2c, 2c+1 of a half
  uint32_t ssel;    // PRMT selector: (byte 2c, 0, byte 2c+1, 0)
  float kd;         // 2^(48 - 2c): undoes sc's 2^-24 and the columns' 2^(2c-24)
};

__device__ __forceinline__ T1Lane t1_lane(int c) {
  T1Lane L;
  L.m1 = 0x00030003u << (2 * (c >> 1));
  L.m2 = L.m1 << 4;
  L.qoff = 16u * (c & 1);
  L.rot = 2u * (c & 1);
  L.soff = 4u * (c >> 1);
  const uint32_t b = 2u * (c & 1);
  L.ssel = b | (4u << 4) | ((b + 1u) << 8) | (4u << 12);
  L.kd = __uint_as_float((uint32_t)(127 + 48 - 2 * c) << 23);
  return L;
}

// Activation operands of one 256-value block of one token: x[h][s] for the
// eight MMAs of half h, m for the mins MMA (columns 0 / 1: hi / lo parts of
// the 16 sub-block sums).
struct T1B {
  uint32_t x[2][8][2];
  uint32_t m[2];
};

__device__ __forceinline__ uint32_t pack_h2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// src: the block's 256 activations, bf16 (BF16 = true) or fp16 bits.
template <bool BF16>
__device__ __forceinline__ void t1_load_b(T1B &B, const uint16_t *__restrict__ src, int g, int c) {
  const bool own0 = g == c, own1 = g == c + 4;
  uint16_t shi[2], slo[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // sub-block 8h + g of the block, natural order
    const uint4 v0 = __ldcg(reinterpret_cast<const uint4 *>(src + 16 * (8 * h + g)));
    const uint4 v1 = __ldcg(reinterpret_cast<const uint4 *>(src + 16 * (8 * h + g)) + 1);
    const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint16_t f[16];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t bits = (wd[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
      float v;
      if (BF16) {
        v = bf16_bits_to_f32(bits);
        f[i] = __half_as_ushort(__float2half_rn(v));
      } else {
        v = f16_bits_to_f32(bits);
        f[i] = (uint16_t)bits;
      }
      s += v;
    }
    // K step 2 wd + beta: values 4 (wd ^ rot) + beta and + 2
#pragma unroll
    for (int wdi = 0; wdi < 4; ++wdi) {
#pragma unroll
      for (int beta = 0; beta < 2; ++beta) {
        const uint32_t p0 = pack_h2(f[4 * wdi + beta], f[4 * wdi + 2 + beta]);
        const uint32_t p1 = pack_h2(f[4 * (wdi ^ 2) + beta], f[4 * (wdi ^ 2) + 2 + beta]);
        const uint32_t p = (c & 1) ? p1 : p0;
        B.x[h][2 * wdi + beta][0] = own0 ? p : 0u;
        B.x[h][2 * wdi + beta][1] = own1 ? p : 0u;
      }
    }
    const __half hi = __float2half_rn(s);
    shi[h] = __half_as_ushort(hi);
    slo[h] = __half_as_ushort(__float2half_rn(s - __half2float(hi)));
  }
  // mins operand: K slots 2c, 2c+1 = sub-blocks 2c, 2c+1 (half 0) and
  // 2c+8, 2c+9 (half 1); their sums live in lanes 4 (2c) and 4 (2c + 1)
  uint32_t mv[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint16_t h0 = (uint16_t)__shfl_sync(0xffffffffu, (uint32_t)shi[h], 8 * c);
    const uint16_t h1 = (uint16_t)__shfl_sync(0xffffffffu, (uint32_t)shi[h], 8 * c + 4);
    const uint16_t l0 = (uint16_t)__shfl_sync(0xffffffffu, (uint32_t)slo[h], 8 * c);
    const uint16_t l1 = (uint16_t)__shfl_sync(0xffffffffu, (uint32_t)slo[h], 8 * c + 4);
    mv[h] = g == 0 ? pack_h2(h0, h1) : g == 1 ? pack_h2(l0, l1) : 0u;
  }
  B.m[0] = mv[0];
  B.m[1] = mv[1];
}

// Shared-memory layout of a staged 16-row tile: row r starts at
// r * rowb + gap * (r >> gsh); the tile arrives as 16 >> gsh bulk copies of
// (rowb << gsh) bytes, each followed by a gap-byte hole.  The gap makes the 8
// rows g = 0 .. 7 that a warp's lane quads read together start in 8 distinct
// 16-byte bank groups (with R = rowb / 16):
//   R odd:          no gap, the whole tile in one copy (R g mod 8 distinct);
//   R = 4 (mod 8):  16 bytes every 2 rows (4 g + g / 2 mod 8 distinct);
//   R = 2, 6 (mod 8): 16 bytes every 4 rows (2 g + g / 4, 6 g + g / 4);
//   R = 0 (mod 8):  16 bytes after every row (stride R + 1, odd).
// Fewer, larger copies matter: a bulk copy of a 1.3 KB row lands noticeably
// later than one of 2.7 KB carrying the same bytes.
struct T1Tile {
  uint32_t rowb, gap, gsh;
};
__host__ __device__ constexpr T1Tile t1_tile(uint32_t rowb) {
  return ((rowb / 16) & 1u)       ? T1Tile{rowb, 0u, 4u}
         : ((rowb / 16) % 8 == 4) ? T1Tile{rowb, 16u, 1u}
         : ((rowb / 16) % 8 == 0) ? T1Tile{rowb, 16u, 0u}
                                  : T1Tile{rowb, 16u, 2u};
}
__host__ __device__ constexpr uint32_t t1_tile_bytes(T1Tile t) { return 16u * t.rowb + (16u >> t.gsh) * t.gap; }
__host__ __device__ constexpr uint32_t t1_row_off(T1Tile t, uint32_t r) { return r * t.rowb + t.gap * (r >> t.gsh); }
__host__ __device__ constexpr uint32_t t1_copies(T1Tile t) { return 16u >> t.gsh; }
__host__ __device__ constexpr uint32_t t1_copy_bytes(T1Tile t) { return t.rowb << t.gsh; }

// Issue copy i (< t1_copies) of the 16 rows starting at src into the tile at dst.
__device__ __forceinline__ void t1_tile_copy(uint8_t *dst, const uint8_t *src, T1Tile t, uint32_t i, uint64_t *bar) {
  ptx::bulk_g2s(dst + i * (t1_copy_bytes(t) + t.gap), src + (size_t)i * t1_copy_bytes(t), t1_copy_bytes(t), bar);
}

// One Q2_K block column of NM tiles of 16 staged rows each (tile m, row r at
// mat[m] + t1_row_off(tl, r)), against one activation block: this lane's
// share of
// d * sum(sc * q * x) - dmin * sum(mn * xsum) for rows g and g + 8 of every
// matrix.  Even and odd K steps accumulate separately, so 2 NM MMA chains
// are in flight.
template <int NM>
__device__ __forceinline__ void t1_block(const uint8_t *const (&mat)[NM], T1Tile tl, int g, const T1B &B,
                                         const T1Lane &L, float (&y)[NM][2]) {
  const uint8_t *row[NM][2];
  uint32_t sp[NM][2][2], dd[NM][2];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      row[m][r] = mat[m] + t1_row_off(tl, (uint32_t)(g + 8 * r));
      // scale bytes of sub-blocks (2c, 2c+1) of half 0 and (8+2c, 9+2c) of half 1
      sp[m][r][0] = __byte_perm(ptx::lds32(row[m][r] + L.soff), 0u, L.ssel);
      sp[m][r][1] = __byte_perm(ptx::lds32(row[m][r] + 8 + L.soff), 0u, L.ssel);
      dd[m][r] = ptx::lds32(row[m][r] + 80);
    }
  }
  float sacc[NM][2];
#pragma unroll
  for (int m = 0; m < NM; ++m) sacc[m][0] = sacc[m][1] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t wq[NM][2][4];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) wq[m][r][i] = ptx::lds32(row[m][r] + 16 + 32 * h + L.qoff + 4 * (i ^ L.rot));
    float C[NM][2][4];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) C[m][0][j] = C[m][1][j] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint32_t A[4] = {wq[m][0][i] & L.m1, wq[m][1][i] & L.m1, wq[m][0][i] & L.m2, wq[m][1][i] & L.m2};
        ptx::mma_f16(C[m][0], A, B.x[h][2 * i][0], B.x[h][2 * i][1]);
      }
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const uint32_t ua = wq[m][0][i] >> 8, ub = wq[m][1][i] >> 8;
        const uint32_t A[4] = {ua & L.m1, ub & L.m1, ua & L.m2, ub & L.m2};
        ptx::mma_f16(C[m][1], A, B.x[h][2 * i + 1][0], B.x[h][2 * i + 1][1]);
      }
    }
    // sc of sub-blocks 8h + 2c, 8h + 2c + 1 as fp16 subnormals sc * 2^-24
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const uint32_t sca = sp[m][0][h] & 0x000F000Fu, scb = sp[m][1][h] & 0x000F000Fu;
      sacc[m][0] = fmaf(f16_bits_to_f32(sca & 0xFFFFu), C[m][0][0] + C[m][1][0], sacc[m][0]);
      sacc[m][0] = fmaf(f16_bits_to_f32(sca >> 16), C[m][0][1] + C[m][1][1], sacc[m][0]);
      sacc[m][1] = fmaf(f16_bits_to_f32(scb & 0xFFFFu), C[m][0][2] + C[m][1][2], sacc[m][1]);
      sacc[m][1] = fmaf(f16_bits_to_f32(scb >> 16), C[m][0][3] + C[m][1][3], sacc[m][1]);
    }
  }
  // mins: mn * 2^-20 (high nibbles) against the sub-block sums
  const float k20 = 1048576.f;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const uint32_t Am[4] = {sp[m][0][0] & 0x00F000F0u, sp[m][1][0] & 0x00F000F0u, sp[m][0][1] & 0x00F000F0u,
                            sp[m][1][1] & 0x00F000F0u};
    float M[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_f16(M, Am, B.m[0], B.m[1]);
#pragma unroll
    for (int r = 0; r < 2; ++r)
      y[m][r] = fmaf(f16_bits_to_f32(dd[m][r] & 0xFFFFu) * L.kd, sacc[m][r],
                     -f16_bits_to_f32(dd[m][r] >> 16) * k20 * (M[2 * r] + M[2 * r + 1]));
  }
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Last-arriver election over the consumer warps of a stage: every warp
// publishes its partials, then counts itself; the warp that completes the
// count returns true (and resets the counter) and may read all partials.
__device__ __forceinline__ bool t1_last_arriver(int *cnt, int nwarps) {
  const int lane = threadIdx.x & 31;
  int last = 0;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    last = atomicAdd(cnt, 1) == nwarps - 1;
    if (last) {
      *cnt = 0;
      __threadfence_block();
    }
  }
  return __shfl_sync(0xffffffffu, last, 0) != 0;
}

// Shared-memory layout of the single-token kernels: nstage stages, then
// the full / empty barriers, the per-stage partials and the per-stage
// arrival counters.
struct T1Smem {
  uint64_t *full, *empty;
  float *red;  // [nstage][nwarps][32]
  int *cnt;    // [nstage]
};
__device__ __forceinline__ T1Smem t1_smem(uint8_t *smem, int nstage, uint32_t stage_bytes, int nwarps) {
  T1Smem t;
  t.full = reinterpret_cast<uint64_t *>(smem + (size_t)nstage * stage_bytes);
  t.empty = t.full + nstage;
  t.red = reinterpret_cast<float *>(t.empty + nstage);
  t.cnt = reinterpret_cast<int *>(t.red + (size_t)nstage * nwarps * 32);
  return t;
}
__host__ __device__ constexpr size_t t1_smem_bytes(int nstage, uint32_t stage_bytes, int nwarps) {
  return (size_t)nstage * stage_bytes + 16 * (size_t)nstage + (size_t)nstage * nwarps * 32 * 4 + 4 * (size_t)nstage;
}

// With one token there are at most k <= 32 groups: every CTA keeps them in
// shared memory, so no unit waits on a global load for its expert.
constexpr int kT1MaxGroups = 32;

// Routing of the single token from the router's E <= 256 logits, by one
// warp of every CTA that needs it (each computes the same result from the
// same logits, so no grid waits on another one's ranking): the k experts in
// rank order (descending logit, ties to the lower id), then one group per
// selected expert in ascending expert order -- the selected experts are
// distinct, so every group holds one pair and pair i sits at position
// inv[i] of the expert-sorted order.  With `publish` (one CTA of the chain)
// the warp also writes idx and the softmax weights over the selected (the
// call's outputs) and the bucketing outputs the later grids read.
__device__ __forceinline__ void t1_route_warp(const FfnArgs &a, Group *s_grp, int *s_ngrp, bool publish,
                                              float *s_lv = nullptr, int *s_inv = nullptr) {
  const int lane = threadIdx.x & 31, E = a.L.n_expert, k = a.k;
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? __ldcg(a.lg + e) : 0.f;
  }
  float my_v;
  int my_e;
  topk_select_warp(v, E, k, my_v, my_e);
  int pos = 0;  // experts selected with a smaller id
  for (int j = 0; j < k; ++j) pos += __shfl_sync(0xffffffffu, my_e, j) < my_e;
  if (lane < k) s_grp[pos] = Group{my_e, pos, 1, 0};
  if (lane == 0) *s_ngrp = k;
  if (s_lv && lane < k) {
    s_lv[lane] = my_v;  // slot i's logit and sorted position, for a later warp
    s_inv[lane] = pos;
  }
  if (publish) {
    const float wt = softmax_selected_warp(my_v, k);
    if (lane < k) {
      a.idx_out[lane] = my_e;
      const_cast<float *>(a.w)[lane] = wt;
      const_cast<int32_t *>(a.inv)[lane] = pos;
      const_cast<int32_t *>(a.perm)[pos] = lane;
      const_cast<Group *>(a.groups)[pos] = Group{my_e, pos, 1, 0};
    }
    if (lane == 0) {
      const_cast<int32_t *>(a.nvalid)[0] = k;
      a.hdr->n_groups = k;
      a.hdr->n_active = k;
    }
  }
}
// The routing weights (softmax over the k selected logits, by one warp) into
// s_w, and with `publish` the call's routing outputs, from what
// t1_route_warp left in shared memory.
__device__ __forceinline__ void t1_weights_warp(const FfnArgs &a, const Group *s_grp, const float *s_lv,
                                                const int *s_inv, float *s_w, bool publish) {
  const int lane = threadIdx.x & 31, k = a.k;
  const float wt = softmax_selected_warp(lane < k ? s_lv[lane] : 0.f, k);
  if (lane < k) s_w[lane] = wt;
  if (publish) {
    if (lane < k) {
      const int pos = s_inv[lane];
      a.idx_out[lane] = s_grp[pos].e;
      const_cast<float *>(a.w)[lane] = wt;
      const_cast<int32_t *>(a.inv)[lane] = pos;
      const_cast<int32_t *>(a.perm)[pos] = lane;
      const_cast<Group *>(a.groups)[pos] = s_grp[pos];
    }
    if (lane == 0) {
      const_cast<int32_t *>(a.nvalid)[0] = k;
      a.hdr->n_groups = k;
      a.hdr->n_active = k;
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void t1_load_groups(const FfnArgs &a, Group *s_grp, int *s_ngrp) {
  if (threadIdx.x < 32) {
    const int n = __ldcg(&a.hdr->n_groups);
    if (threadIdx.x < n) {
      const int4 v = __ldcg(reinterpret_cast<const int4 *>(a.groups + threadIdx.x));
      s_grp[threadIdx.x] = Group{v.x, v.y, v.z, v.w};
    }
    if (threadIdx.x == 0) *s_ngrp = n;
  }
  __syncthreads();
}

}  // namespace ds4

namespace ds4 {

// ------------------------------------------------------- Q4_K single token
// The same scheme for Q4_K blocks (8 sub-blocks of 32 values, 4-bit codes,
// 6-bit scales and mins): column n of every MMA is sub-block n, K slots 2n,
// 2n+1 carry two of its values, and the 16 K steps of a block cover all 32.
// Lane quad c reads sub-block c (qs bytes 32 (c/2) .. +31) and c + 4 (bytes
// 32 (c/2 + 2) ..), both in nibble c & 1: masking the nibble leaves the
// subnormal q * 2^-24 (low) or q * 2^-20 (high), so D column 2c is scaled by
// 2^24 and column 2c + 1 by 2^20.  K step 2i + beta of a sub-block holds its
// values 4i + beta and 4i + 2 + beta.  The activation operands use T1B with
// K step s in x[s / 8][s % 8]; the mins MMA pairs each sub-block's mn (twice)
// with the hi and lo parts of its sum in column 0.

__device__ __forceinline__ void q4k_sc_mn_pair(const uint32_t (&s3)[3], int j, uint32_t &sc, uint32_t &mn) {
  // scales[12] as three little-endian words
  const auto byte = [&](int b) { return (s3[b >> 2] >> (8 * (b & 3))) & 0xFFu; };
  if (j < 4) {
    sc = byte(j) & 63u;
    mn = byte(j + 4) & 63u;
  } else {
    sc = (byte(j + 4) & 15u) | ((byte(j - 4) >> 6) << 4);
    mn = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
  }
}

// src: the block's 256 activations, bf16 (BF16 = true) or fp16 bits.
template <bool BF16>
__device__ __forceinline__ void t1_load_b_q4k(T1B &B, const uint16_t *__restrict__ src, int g, int c) {
  const bool own0 = g == c, own1 = g == c + 4;
  // sub-block g: values 32 g .. 32 g + 31
  uint16_t f[32];
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(src + 32 * g) + q);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t bits = (wd[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
      float val;
      if (BF16) {
        val = bf16_bits_to_f32(bits);
        f[8 * q + i] = __half_as_ushort(__float2half_rn(val));
      } else {
        val = f16_bits_to_f32(bits);
        f[8 * q + i] = (uint16_t)bits;
      }
      s += val;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int beta = 0; beta < 2; ++beta) {
      const uint32_t p = pack_h2(f[4 * i + beta], f[4 * i + 2 + beta]);
      const int st = 2 * i + beta;
      B.x[st >> 3][st & 7][0] = own0 ? p : 0u;
      B.x[st >> 3][st & 7][1] = own1 ? p : 0u;
    }
  const __half hi = __float2half_rn(s);
  const uint16_t shi = __half_as_ushort(hi), slo = __half_as_ushort(__float2half_rn(s - __half2float(hi)));
  const uint32_t hl = pack_h2(shi, slo);
  // lanes of column 0 (g == 0): (hi, lo) of sub-blocks c and c + 4
  const uint32_t m0 = __shfl_sync(0xffffffffu, hl, 4 * c);
  const uint32_t m1 = __shfl_sync(0xffffffffu, hl, 4 * c + 16);
  B.m[0] = g == 0 ? m0 : 0u;
  B.m[1] = g == 0 ? m1 : 0u;
}

// One Q4_K block column of NM 16-row tiles (tile m, row r at mat[m] +
// t1_row_off(tl, r)) against one activation block: this lane's share of
// d * sum(sc * q * x) - dmin * sum(mn * xsum) for rows g and g + 8.
template <int NM>
__device__ __forceinline__ void t1_block_q4k(const uint8_t *const (&mat)[NM], T1Tile tl, int g, int c,
                                             const T1B &B, float (&y)[NM][2]) {
  const uint32_t mask = (c & 1) ? 0x00F000F0u : 0x000F000Fu;
  const float k0 = 16777216.f, k1 = 1048576.f;  // 2^24, 2^20
  const uint32_t offa = 16u + 32u * (uint32_t)(c >> 1), offb = offa + 64u;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    uint4 qa[2][2], qb[2][2];  // [row][16-byte half]
    uint32_t dd[2], s3[2][3];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint8_t *row = mat[m] + t1_row_off(tl, (uint32_t)(g + 8 * r));
      dd[r] = ptx::lds32(row);
#pragma unroll
      for (int q = 0; q < 3; ++q) s3[r][q] = ptx::lds32(row + 4 + 4 * q);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        qa[r][q] = *reinterpret_cast<const uint4 *>(row + offa + 16 * q);
        qb[r][q] = *reinterpret_cast<const uint4 *>(row + offb + 16 * q);
      }
    }
    float C[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const auto word = [](const uint4 (&v)[2], int k) {
        const uint4 &h = v[k >> 2];
        return (k & 3) == 0 ? h.x : (k & 3) == 1 ? h.y : (k & 3) == 2 ? h.z : h.w;
      };
      const uint32_t wa0 = word(qa[0], i), wa1 = word(qa[1], i), wb0 = word(qb[0], i), wb1 = word(qb[1], i);
      {
        const uint32_t A[4] = {wa0 & mask, wa1 & mask, wb0 & mask, wb1 & mask};
        const int st = 2 * i;
        ptx::mma_f16(C[0], A, B.x[st >> 3][st & 7][0], B.x[st >> 3][st & 7][1]);
      }
      {
        const uint32_t A[4] = {(wa0 >> 8) & mask, (wa1 >> 8) & mask, (wb0 >> 8) & mask, (wb1 >> 8) & mask};
        const int st = 2 * i + 1;
        ptx::mma_f16(C[1], A, B.x[st >> 3][st & 7][0], B.x[st >> 3][st & 7][1]);
      }
    }
    // scales of the lane's columns (sub-blocks 2c, 2c + 1) and mins of the
    // sub-blocks whose K slots it holds (c, c + 4)
    uint32_t Am[4];
    float sacc[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      uint32_t sc0, mn0, sc1, mn1, scx, mnc, mnc4;
      q4k_sc_mn_pair(s3[r], 2 * c, sc0, mn0);
      q4k_sc_mn_pair(s3[r], 2 * c + 1, sc1, mn1);
      q4k_sc_mn_pair(s3[r], c, scx, mnc);
      q4k_sc_mn_pair(s3[r], c + 4, scx, mnc4);
      sacc[r] = fmaf((float)sc0 * k0, C[0][2 * r] + C[1][2 * r], (float)sc1 * k1 * (C[0][2 * r + 1] + C[1][2 * r + 1]));
      // fp16 mn (exact small integers), duplicated in both halves
      const uint32_t hc = __half_as_ushort(__uint2half_rn(mnc)), hc4 = __half_as_ushort(__uint2half_rn(mnc4));
      Am[r] = hc | (hc << 16);
      Am[2 + r] = hc4 | (hc4 << 16);
    }
    float M[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_f16(M, Am, B.m[0], B.m[1]);
#pragma unroll
    for (int r = 0; r < 2; ++r)
      y[m][r] = fmaf(f16_bits_to_f32(dd[r] & 0xFFFFu), sacc[r], -f16_bits_to_f32(dd[r] >> 16) * M[2 * r]);
  }
}

}  // namespace ds4
