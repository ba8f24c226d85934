// Expert FFN for decode batches.
//
// Tensor-core path (mma.sync m16n8k16, bf16 operands, fp32 accumulate):
// the 2-bit / 4-bit codes are turned into exact bf16 A-operands in
// registers (a magic-number OR places the code in the mantissa of 128.0), so
// each tensor-core product is exact; per-16-value Q2_K scales are folded into
// the operand with one packed bf16 FMA (sc * q <= 45 is exact in bf16), the
// Q2_K mins and the Q4_1 (d, m) are applied per block in an fp32 epilogue.
// Weight rows are staged into shared memory by bulk asynchronous copies (TMA,
// non-tensor form) completing on mbarriers, two stages per warp.  Tokens of
// one expert (up to 8 per group) fill the n = 8 side of the MMA.
//
//   gate/up: one CTA per (token group, 16-row tile); each warp owns one K
//            slice of both matrices, the slices are summed in shared memory,
//            then h = bf16(silu(g) * u) and the 16-row sub-block sums of h.
//   down:    one warp per (token group, 16-row tile), full K.
//
// A SIMT path covers shapes whose rows cannot be staged with 16-byte bulk
// copies (row bytes not a multiple of 16).
#include "internal.cuh"
#include "ptx.cuh"

namespace ds4 {
namespace {

constexpr int kTok = kGroup;            // tokens per pass (= MMA n)
constexpr uint32_t kMagic = 0x43004300u;  // bf16x2 (128, 128)
constexpr uint32_t kOne = 0x3F803F80u;    // bf16x2 (1, 1)
constexpr uint32_t kNeg128 = 0xC300C300u; // bf16x2 (-128, -128)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ======================================================= tensor-core tiles
// Per-lane view of the m16n8k16 fragments: lane = 4 g + c; A rows g and
// g + 8; B column (token) g; D rows g, g + 8 x tokens 2c, 2c + 1.  K slots
// (2c, 2c+1) hold values 4c, 4c+1 of a 16-value run and slots (2c+8, 2c+9)
// values 4c+2, 4c+3, so B is a natural-order 64-bit load of 4 activations.

// Q2_K scale folding constants for code position s' (the code sits at bit
// 2 s' of each bf16 half, i.e. the operand is 128 + 4^s' q):
//   s1 = sc * 4^-s',  s0 = -128 * sc * 4^-s'  from v = 128 + sc:
//   s1 = v * 4^-s' - 128 * 4^-s',  s0 = v * (-128 * 4^-s') + 16384 * 4^-s'.
__device__ __forceinline__ void q2k_consts(uint32_t v, int sp, uint32_t &s1, uint32_t &s0) {
  const uint32_t f1 = sp == 0 ? 0x3F803F80u : sp == 1 ? 0x3E803E80u : 0x3D803D80u;   // 4^-s'
  const uint32_t f0 = sp == 0 ? 0xC300C300u : sp == 1 ? 0xC200C200u : 0xC100C100u;   // -128 * 4^-s'
  const uint32_t g0 = sp == 0 ? 0x46804680u : sp == 1 ? 0x45804580u : 0x44804480u;   // 16384 * 4^-s'
  s1 = ptx::fma_bf16x2(v, f1, f0);
  s0 = ptx::fma_bf16x2(v, f0, g0);
}

// This lane's activations for one 256-value segment: the B fragments of the
// 16 sixteen-value runs (token g, values 16n + 4c .. 16n + 4c + 3) and, for
// Q2_K mins, the sub-block-sum fragments (hi and lo parts).
struct SegIn {
  uint2 bx[16];
  uint2 shi, slo;
};

__device__ __forceinline__ void load_seg(SegIn &in, const uint16_t *__restrict__ xb,
                                         const uint8_t *__restrict__ sums, int c) {
#pragma unroll
  for (int n = 0; n < 16; ++n) in.bx[n] = xb ? ptx::ldg_nc_v2(xb + 16 * n + 4 * c) : make_uint2(0u, 0u);
  in.shi = sums ? ptx::ldg_nc_v2(sums + 8 * c) : make_uint2(0u, 0u);
  in.slo = sums ? ptx::ldg_nc_v2(sums + 32 + 8 * c) : make_uint2(0u, 0u);
}

// One Q2_K 256-value block of 16 staged rows (row g at blk_a, g + 8 at
// blk_b): acc += d * (sum sc*q*x) - dmin * (sum mn*xsum).
__device__ __forceinline__ void q2k_block(const uint8_t *__restrict__ blk_a, const uint8_t *__restrict__ blk_b,
                                          const SegIn &in, int c, float (&acc)[4]) {
  uint32_t qa[4], qb[4], sa[4], sb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    qa[j] = ptx::lds32(blk_a + 16 + 4 * (4 * j + c));
    qb[j] = ptx::lds32(blk_b + 16 + 4 * (4 * j + c));
    sa[j] = ptx::lds32(blk_a + 4 * j);
    sb[j] = ptx::lds32(blk_b + 4 * j);
  }
  const uint32_t dda = ptx::lds32(blk_a + 80), ddb = ptx::lds32(blk_b + 80);
  uint32_t scma[4], scmb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    scma[j] = sa[j] & 0x0F0F0F0Fu;
    scmb[j] = sb[j] & 0x0F0F0F0Fu;
  }
  float dm[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a01 = __byte_perm(qa[j], 0, 0x4140), a23 = __byte_perm(qa[j], 0, 0x4342);
    const uint32_t b01 = __byte_perm(qb[j], 0, 0x4140), b23 = __byte_perm(qb[j], 0, 0x4342);
    const uint32_t a01s = __byte_perm(qa[j] >> 2, 0, 0x4140), a23s = __byte_perm(qa[j] >> 2, 0, 0x4342);
    const uint32_t b01s = __byte_perm(qb[j] >> 2, 0, 0x4140), b23s = __byte_perm(qb[j] >> 2, 0, 0x4342);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int n = 8 * (j >> 1) + 2 * s + (j & 1);  // 16-value sub-block of this MMA
      const int sp = s < 3 ? s : 2;                   // s = 3 is read from the >> 2 copy
      const uint32_t mask = 0x00030003u << (2 * sp);
      const uint32_t sel = 0x4040u | ((uint32_t)(n & 3) << 8) | (uint32_t)(n & 3);
      uint32_t s1a, s0a, s1b, s0b;
      q2k_consts(__byte_perm(scma[n >> 2], 0x43434343u, sel), sp, s1a, s0a);
      q2k_consts(__byte_perm(scmb[n >> 2], 0x43434343u, sel), sp, s1b, s0b);
      uint32_t A[4];
      A[0] = ptx::fma_bf16x2(ptx::and_or(s < 3 ? a01 : a01s, mask, kMagic), s1a, s0a);
      A[1] = ptx::fma_bf16x2(ptx::and_or(s < 3 ? b01 : b01s, mask, kMagic), s1b, s0b);
      A[2] = ptx::fma_bf16x2(ptx::and_or(s < 3 ? a23 : a23s, mask, kMagic), s1a, s0a);
      A[3] = ptx::fma_bf16x2(ptx::and_or(s < 3 ? b23 : b23s, mask, kMagic), s1b, s0b);
      ptx::mma_bf16(dm[j & 1], A, in.bx[n].x, in.bx[n].y);
    }
  }
  // mins: D_min[r][t] = sum_n mn[r][n] * xsum[n][t] (xsum = hi + lo); lane
  // quad c takes scale bytes 2c, 2c+1 and 2c+8, 2c+9, high nibble = min
  float dn[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t sel = (c & 1) ? 0x4342u : 0x4140u;
    uint32_t Am[4];
    Am[0] = ptx::fma_bf16x2(ptx::and_or(__byte_perm(sa[c >> 1], 0, sel) >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    Am[1] = ptx::fma_bf16x2(ptx::and_or(__byte_perm(sb[c >> 1], 0, sel) >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    Am[2] = ptx::fma_bf16x2(ptx::and_or(__byte_perm(sa[2 + (c >> 1)], 0, sel) >> 4, 0x000F000Fu, kMagic), kOne,
                            kNeg128);
    Am[3] = ptx::fma_bf16x2(ptx::and_or(__byte_perm(sb[2 + (c >> 1)], 0, sel) >> 4, 0x000F000Fu, kMagic), kOne,
                            kNeg128);
    ptx::mma_bf16(dn, Am, in.shi.x, in.shi.y);
    ptx::mma_bf16(dn, Am, in.slo.x, in.slo.y);
  }
  const float da = f16_bits_to_f32(dda & 0xFFFFu), dmina = f16_bits_to_f32(dda >> 16);
  const float db = f16_bits_to_f32(ddb & 0xFFFFu), dminb = f16_bits_to_f32(ddb >> 16);
  acc[0] = fmaf(da, dm[0][0] + dm[1][0], fmaf(-dmina, dn[0], acc[0]));
  acc[1] = fmaf(da, dm[0][1] + dm[1][1], fmaf(-dmina, dn[1], acc[1]));
  acc[2] = fmaf(db, dm[0][2] + dm[1][2], fmaf(-dminb, dn[2], acc[2]));
  acc[3] = fmaf(db, dm[0][3] + dm[1][3], fmaf(-dminb, dn[3], acc[3]));
}

// Eight Q4_1 blocks (one 256-value segment): per block
// acc += d * (sum q*x) + m * (sum x).  xs_a / xs_b: the 8 block sums of
// tokens 2c and 2c + 1 (or nullptr).
__device__ __forceinline__ void q41_seg(const uint8_t *__restrict__ seg_a, const uint8_t *__restrict__ seg_b,
                                        const SegIn &in, const float *__restrict__ xs_a,
                                        const float *__restrict__ xs_b, int c, float (&acc)[4]) {
  float xsa[8], xsb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    xsa[i] = xs_a ? xs_a[i] : 0.f;
    xsb[i] = xs_b ? xs_b[i] : 0.f;
  }
#pragma unroll
  for (int bb = 0; bb < 8; ++bb) {
    const uint8_t *blk_a = seg_a + kQ41Bytes * bb, *blk_b = seg_b + kQ41Bytes * bb;
    const uint32_t qa = ptx::lds32(blk_a + 4 + 4 * c), qb = ptx::lds32(blk_b + 4 + 4 * c);
    const uint32_t dma = ptx::lds32(blk_a), dmb = ptx::lds32(blk_b);
    const uint32_t a01 = __byte_perm(qa, 0, 0x4140), a23 = __byte_perm(qa, 0, 0x4342);
    const uint32_t b01 = __byte_perm(qb, 0, 0x4140), b23 = __byte_perm(qb, 0, 0x4342);
    uint32_t lo[4], hi[4];
    lo[0] = ptx::fma_bf16x2(ptx::and_or(a01, 0x000F000Fu, kMagic), kOne, kNeg128);
    lo[1] = ptx::fma_bf16x2(ptx::and_or(b01, 0x000F000Fu, kMagic), kOne, kNeg128);
    lo[2] = ptx::fma_bf16x2(ptx::and_or(a23, 0x000F000Fu, kMagic), kOne, kNeg128);
    lo[3] = ptx::fma_bf16x2(ptx::and_or(b23, 0x000F000Fu, kMagic), kOne, kNeg128);
    hi[0] = ptx::fma_bf16x2(ptx::and_or(a01 >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    hi[1] = ptx::fma_bf16x2(ptx::and_or(b01 >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    hi[2] = ptx::fma_bf16x2(ptx::and_or(a23 >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    hi[3] = ptx::fma_bf16x2(ptx::and_or(b23 >> 4, 0x000F000Fu, kMagic), kOne, kNeg128);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_bf16(d, lo, in.bx[2 * bb].x, in.bx[2 * bb].y);
    ptx::mma_bf16(d, hi, in.bx[2 * bb + 1].x, in.bx[2 * bb + 1].y);
    const float da = f16_bits_to_f32(dma & 0xFFFFu), ma = f16_bits_to_f32(dma >> 16);
    const float db = f16_bits_to_f32(dmb & 0xFFFFu), mb = f16_bits_to_f32(dmb >> 16);
    acc[0] = fmaf(da, d[0], fmaf(ma, xsa[bb], acc[0]));
    acc[1] = fmaf(da, d[1], fmaf(ma, xsb[bb], acc[1]));
    acc[2] = fmaf(db, d[2], fmaf(mb, xsa[bb], acc[2]));
    acc[3] = fmaf(db, d[3], fmaf(mb, xsb[bb], acc[3]));
  }
}

// Bytes of one 256-value segment of a row.
template <int Q>
constexpr int seg_bytes() { return Q == DS4MOE_Q2_K ? kQ2KBytes : 8 * kQ41Bytes; }

template <int Q>
__device__ __forceinline__ void seg_rows(const uint8_t *ra, const uint8_t *rb, const SegIn &in,
                                         const float *xs_a, const float *xs_b, int c, float (&acc)[4]) {
  if constexpr (Q == DS4MOE_Q2_K) q2k_block(ra, rb, in, c, acc);
  else q41_seg(ra, rb, in, xs_a, xs_b, c, acc);
}

// ------------------------------------------------------------ staging
struct Stage {
  uint64_t *bar;
  uint8_t *buf;
};

// Issue the bulk copies of 16 rows x `chunk` bytes (row r from src + r * stride)
// into dst (row stride `chunk`), lanes 0..15; completes on bar.
__device__ __forceinline__ void stage_rows(uint8_t *dst, const uint8_t *src, int64_t stride, uint32_t chunk,
                                           uint64_t *bar, int lane_base) {
  const int lane = threadIdx.x & 31;
  const int r = lane - lane_base;
  if (r >= 0 && r < 16) ptx::bulk_g2s(dst + r * chunk, src + r * stride, chunk, bar);
}

// ============================================================ gate / up
// CTA = kp warps; warp w owns K chunk w of both matrices.  Shared memory per
// warp: two stages of [16 gate rows | 16 up rows] x chunk bytes.
template <int QG, int QU>
__global__ void __launch_bounds__(256) k_gate_up_mma(FfnArgs a, int kp, uint32_t chg, uint32_t chu) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff;
  const uint32_t stage_bytes = 16u * (chg + chu);
  uint8_t *wbuf = smem + (size_t)w * 2 * stage_bytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kp * 2 * stage_bytes);  // [kp][2]
  float *red = reinterpret_cast<float *>(bars + 2 * kp);                              // [kp][32][8]
  uint64_t *mybar = bars + 2 * w;
  if (lane == 0) {
    ptx::mbar_init(&mybar[0], 1);
    ptx::mbar_init(&mybar[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const int ntile = F / 16;
  const int U = a.hdr->n_groups * ntile;
  const int64_t rbg = row_bytes(QG, D), rbu = row_bytes(QU, D);
  const int kvals = D / kp;  // values per K chunk (same for gate and up)
  const uint8_t *gate = static_cast<const uint8_t *>(a.L.gate);
  const uint8_t *up = static_cast<const uint8_t *>(a.L.up);

  auto issue = [&](int u, int st) {
    const Group grp = a.groups[u / ntile];
    const int row0 = (u % ntile) * 16;
    uint8_t *dst = wbuf + (size_t)st * stage_bytes;
    if (lane == 0) ptx::mbar_arrive_expect_tx(&mybar[st], stage_bytes);
    __syncwarp();
    const uint8_t *gs = gate + ((int64_t)grp.e * F + row0) * rbg + (int64_t)w * chg;
    const uint8_t *us = up + ((int64_t)grp.e * F + row0) * rbu + (int64_t)w * chu;
    stage_rows(dst, gs, rbg, chg, &mybar[st], 0);
    stage_rows(dst + 16 * chg, us, rbu, chu, &mybar[st], 16);
  };

  uint32_t phase[2] = {0u, 0u};
  int u = blockIdx.x;
  if (u < U) issue(u, 0);
  if (u + (int)gridDim.x < U) issue(u + gridDim.x, 1);
  bool timed_out = false;
  for (int it = 0; u < U; u += gridDim.x, ++it) {
    const int st = it & 1;
    const Group grp = a.groups[u / ntile];
    const int row0 = (u % ntile) * 16;
    if (!timed_out && !ptx::mbar_wait(&mybar[st], phase[st])) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    phase[st] ^= 1u;
    const uint8_t *buf = wbuf + (size_t)st * stage_bytes;
    // this lane's token (B column g) and the tokens of its D columns 2c, 2c+1
    const int k0 = w * kvals;
    const uint16_t *xb = nullptr;
    const uint8_t *sums = nullptr;
    const float *xs_a = nullptr, *xs_b = nullptr;
    if (g < grp.nt) {
      const int t = a.perm[grp.p0 + g] / a.k;
      xb = a.x + (int64_t)t * D + k0;
      sums = a.xs16 + ((int64_t)t * (D / 256 + 1) + k0 / 256) * 64;
    }
    if (2 * c < grp.nt) xs_a = a.xs32 + (int64_t)(a.perm[grp.p0 + 2 * c] / a.k) * (D / 32) + k0 / 32;
    if (2 * c + 1 < grp.nt) xs_b = a.xs32 + (int64_t)(a.perm[grp.p0 + 2 * c + 1] / a.k) * (D / 32) + k0 / 32;
    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    if (!timed_out) {
      const uint8_t *ga = buf + g * chg, *gb = buf + (g + 8) * chg;
      const uint8_t *ua = buf + 16 * chg + g * chu, *ub = buf + 16 * chg + (g + 8) * chu;
      for (int sg = 0; sg < kvals / 256; ++sg) {
        SegIn in;
        load_seg(in, xb ? xb + 256 * sg : nullptr, sums ? sums + 64 * sg : nullptr, c);
        const float *xa = xs_a ? xs_a + 8 * sg : nullptr, *xbb = xs_b ? xs_b + 8 * sg : nullptr;
        seg_rows<QG>(ga + seg_bytes<QG>() * sg, gb + seg_bytes<QG>() * sg, in, xa, xbb, c, ag);
        seg_rows<QU>(ua + seg_bytes<QU>() * sg, ub + seg_bytes<QU>() * sg, in, xa, xbb, c, au);
      }
    }
    __syncwarp();
    if (u + 2 * (int)gridDim.x < U && !timed_out) issue(u + 2 * gridDim.x, st);
    // K-slice partials -> shared, summed in fixed warp order
    float *r = red + ((size_t)w * 32 + lane) * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[i] = ag[i];
      r[4 + i] = au[i];
    }
    __syncthreads();
    if (w == 0) {
      float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ww = 0; ww < kp; ++ww) {
        const float *q = red + ((size_t)ww * 32 + lane) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gs[i] += q[i];
          us[i] += q[4 + i];
        }
      }
      // h for rows (g, g+8) x tokens (2c, 2c+1); zero for absent tokens
      float hsum[2] = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = row0 + g + 8 * (i >> 1);
        const int tok = 2 * c + (i & 1);
        if (tok < grp.nt) {
          const uint16_t hb = f32_to_bf16_bits(silu(gs[i]) * us[i]);
          a.h[(int64_t)(grp.p0 + tok) * F + row] = hb;
          hsum[i & 1] += bf16_bits_to_f32(hb);
        }
      }
      // sub-block sums of h over the tile's 16 rows (for the down kernel's mins)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        hsum[i] += __shfl_xor_sync(0xffffffffu, hsum[i], 4);
        hsum[i] += __shfl_xor_sync(0xffffffffu, hsum[i], 8);
        hsum[i] += __shfl_xor_sync(0xffffffffu, hsum[i], 16);
      }
      if (g == 0) {
        const int n16 = row0 / 16;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = 2 * c + i;
          if (tok < grp.nt) {
            const uint16_t hi = f32_to_bf16_bits(hsum[i]);
            const uint16_t lo = f32_to_bf16_bits(hsum[i] - bf16_bits_to_f32(hi));
            uint16_t *rec = reinterpret_cast<uint16_t *>(
                a.hs16 + ((int64_t)(grp.p0 + tok) * (F / 256 + 1) + n16 / 16) * 64);
            rec[sums_slot(n16 & 15)] = hi;
            rec[16 + sums_slot(n16 & 15)] = lo;
          }
        }
      }
    }
    __syncthreads();
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out) {
    for (int st = 0; st < 2; ++st) ptx::mbar_wait(&mybar[st], phase[st], 1u << 20);
  }
}

// ================================================================ down
// One warp per (token group, 16-row tile) over the full K (= d_ff); CTA of
// `nw` independent warps, two stages each.
template <int QD>
__global__ void __launch_bounds__(256) k_down_mma(FfnArgs a, uint32_t chd) {
  static_assert(QD == DS4MOE_Q2_K, "the tensor-core down kernel reads Q2_K rows");
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int nw = blockDim.x >> 5;
  const int D = a.L.d_model, F = a.L.d_ff;
  const uint32_t stage_bytes = 16u * chd;
  uint8_t *wbuf = smem + (size_t)w * 2 * stage_bytes;
  uint64_t *mybar = reinterpret_cast<uint64_t *>(smem + (size_t)nw * 2 * stage_bytes) + 2 * w;
  if (lane == 0) {
    ptx::mbar_init(&mybar[0], 1);
    ptx::mbar_init(&mybar[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const int ntile = D / 16;
  const int U = a.hdr->n_groups * ntile;
  const int64_t rbd = row_bytes(QD, F);
  const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
  const int gw = blockIdx.x * nw + w, nwarps = gridDim.x * nw;

  auto issue = [&](int u, int st) {
    const Group grp = a.groups[u / ntile];
    const int row0 = (u % ntile) * 16;
    if (lane == 0) ptx::mbar_arrive_expect_tx(&mybar[st], stage_bytes);
    __syncwarp();
    stage_rows(wbuf + (size_t)st * stage_bytes, down + ((int64_t)grp.e * D + row0) * rbd, rbd, chd, &mybar[st], 0);
  };

  uint32_t phase[2] = {0u, 0u};
  int u = gw;
  if (u < U) issue(u, 0);
  if (u + nwarps < U) issue(u + nwarps, 1);
  bool timed_out = false;
  for (int it = 0; u < U; u += nwarps, ++it) {
    const int st = it & 1;
    const Group grp = a.groups[u / ntile];
    const int row0 = (u % ntile) * 16;
    if (!timed_out && !ptx::mbar_wait(&mybar[st], phase[st])) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    phase[st] ^= 1u;
    const uint16_t *xb = nullptr;
    const uint8_t *sums = nullptr;
    if (g < grp.nt) {
      xb = a.h + (int64_t)(grp.p0 + g) * F;
      sums = a.hs16 + (int64_t)(grp.p0 + g) * (F / 256 + 1) * 64;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (!timed_out) {
      const uint8_t *rows = wbuf + (size_t)st * stage_bytes;
      const uint8_t *ra = rows + g * chd, *rb = rows + (g + 8) * chd;
      for (int sg = 0; sg < F / 256; ++sg) {
        SegIn in;
        load_seg(in, xb ? xb + 256 * sg : nullptr, sums ? sums + 64 * sg : nullptr, c);
        q2k_block(ra + kQ2KBytes * sg, rb + kQ2KBytes * sg, in, c, acc);
      }
    }
    __syncwarp();
    if (u + 2 * nwarps < U && !timed_out) issue(u + 2 * nwarps, st);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * c + (i & 1);
      if (tok < grp.nt) a.y[(int64_t)(grp.p0 + tok) * D + row0 + g + 8 * (i >> 1)] = acc[i];
    }
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out) {
    for (int st = 0; st < 2; ++st) ptx::mbar_wait(&mybar[st], phase[st], 1u << 20);
  }
}

// ============================================================ SIMT path
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

// gate/up + SwiGLU, SIMT: one warp per (token group, hidden row).
__global__ void __launch_bounds__(256) k_gate_up_simt(FfnArgs a) {
  const int D = a.L.d_model, F = a.L.d_ff, k = a.k;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)a.hdr->n_groups * F;
  const int64_t rbg = row_bytes(a.L.q_gate, D), rbu = row_bytes(a.L.q_up, D);
  for (int64_t item = gw; item < items; item += nw) {
    const Group grp = a.groups[item / F];
    const int r = (int)(item % F);
    const uint8_t *grow = static_cast<const uint8_t *>(a.L.gate) + ((int64_t)grp.e * F + r) * rbg;
    const uint8_t *urow = static_cast<const uint8_t *>(a.L.up) + ((int64_t)grp.e * F + r) * rbu;
    const uint16_t *xr[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) xr[t] = a.x + (int64_t)(a.perm[grp.p0 + (t < grp.nt ? t : 0)] / k) * D;
    auto in = [&](int t, int j) { return bf16_bits_to_f32(xr[t][j]); };
    float ag[kTok] = {}, au[kTok] = {};
    row_dot(a.L.q_gate, grow, D, grp.nt, in, ag);
    row_dot(a.L.q_up, urow, D, grp.nt, in, au);
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
      const float gv = warp_sum(ag[t]), uv = warp_sum(au[t]);
      if (lane == t && t < grp.nt) a.h[(int64_t)(grp.p0 + t) * F + r] = f32_to_bf16_bits(silu(gv) * uv);
    }
  }
}

// down, SIMT: one warp per (token group, output row).
__global__ void __launch_bounds__(256) k_down_simt(FfnArgs a) {
  const int D = a.L.d_model, F = a.L.d_ff;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)a.hdr->n_groups * D;
  const int64_t rbd = row_bytes(a.L.q_down, F);
  for (int64_t item = gw; item < items; item += nw) {
    const Group grp = a.groups[item / D];
    const int c = (int)(item % D);
    const uint8_t *drow = static_cast<const uint8_t *>(a.L.down) + ((int64_t)grp.e * D + c) * rbd;
    const uint16_t *hr = a.h + (int64_t)grp.p0 * F;
    auto in = [&](int t, int j) { return bf16_bits_to_f32(hr[(int64_t)t * F + j]); };
    float ay[kTok] = {};
    row_dot(a.L.q_down, drow, F, grp.nt, in, ay);
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
      const float yv = warp_sum(ay[t]);
      if (lane == t && t < grp.nt) a.y[(int64_t)(grp.p0 + t) * D + c] = yv;
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

// ------------------------------------------------------------ dispatch
// K split of gate/up: largest kp in {8, 4, 2, 1} whose per-warp chunks of
// both matrices are whole blocks of a multiple of 16 bytes.
int pick_kp(int D, int qg, int qu) {
  for (int kp = 8; kp >= 1; kp >>= 1) {
    if (D % kp) continue;
    const int kv = D / kp;
    if (kv % 256) continue;
    bool ok = true;
    for (int q : {qg, qu}) {
      if (kv % block_vals(q)) { ok = false; break; }
      if (((int64_t)kv / block_vals(q) * block_bytes(q)) % 16) ok = false;
    }
    if (ok) return kp;
  }
  return 0;
}

template <int QG, int QU>
cudaError_t launch_gate_up_mma(const FfnArgs &a, cudaStream_t s, int kp) {
  const int D = a.L.d_model;
  const uint32_t chg = (uint32_t)(D / kp / block_vals(QG) * block_bytes(QG));
  const uint32_t chu = (uint32_t)(D / kp / block_vals(QU) * block_bytes(QU));
  const size_t smem = (size_t)kp * 2 * 16 * (chg + chu) + 16 * kp + (size_t)kp * 32 * 8 * sizeof(float);
  auto kern = k_gate_up_mma<QG, QU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kp * 32, smem);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * (per_sm > 0 ? per_sm : 1);
  ProfScope p("gate_up", s);
  kern<<<grid, kp * 32, smem, s>>>(a, kp, chg, chu);
  return cudaGetLastError();
}

template <int QD>
cudaError_t launch_down_mma(const FfnArgs &a, cudaStream_t s) {
  const int F = a.L.d_ff;
  const uint32_t chd = (uint32_t)row_bytes(QD, F);
  const int nw = 4;
  const size_t smem = (size_t)nw * 2 * 16 * chd + 16 * nw;
  auto kern = k_down_mma<QD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nw * 32, smem);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * (per_sm > 0 ? per_sm : 1);
  ProfScope p("down", s);
  kern<<<grid, nw * 32, smem, s>>>(a, chd);
  return cudaGetLastError();
}

}  // namespace

// The tensor-core kernels need rows that split into 16-byte-multiple bulk
// copies and stages that fit in shared memory; other shapes use SIMT.
bool decode_mma_ok(const ds4moe_layer &L) {
  const int kp = pick_kp(L.d_model, L.q_gate, L.q_up);
  if (kp == 0) return false;
  const int64_t st = 16 * (row_bytes(L.q_gate, L.d_model) + row_bytes(L.q_up, L.d_model)) / kp;
  if (2 * st * kp > 200 * 1024) return false;
  const int64_t rbd = row_bytes(L.q_down, L.d_ff);
  return L.q_down == DS4MOE_Q2_K && L.d_ff % 256 == 0 && rbd % 16 == 0 && 2 * 16 * 4 * rbd <= 200 * 1024;
}

cudaError_t launch_ffn_decode(const FfnArgs &a, cudaStream_t s) {
  const ds4moe_layer &L = a.L;
  if (decode_mma_ok(L)) {
    const int kp = pick_kp(L.d_model, L.q_gate, L.q_up);
    cudaError_t e;
    if (L.q_gate == DS4MOE_Q2_K && L.q_up == DS4MOE_Q2_K) e = launch_gate_up_mma<DS4MOE_Q2_K, DS4MOE_Q2_K>(a, s, kp);
    else if (L.q_gate == DS4MOE_Q4_1 && L.q_up == DS4MOE_Q4_1) e = launch_gate_up_mma<DS4MOE_Q4_1, DS4MOE_Q4_1>(a, s, kp);
    else if (L.q_gate == DS4MOE_Q2_K) e = launch_gate_up_mma<DS4MOE_Q2_K, DS4MOE_Q4_1>(a, s, kp);
    else e = launch_gate_up_mma<DS4MOE_Q4_1, DS4MOE_Q2_K>(a, s, kp);
    if (e != cudaSuccess) return e;
    return launch_down_mma<DS4MOE_Q2_K>(a, s);
  }
  const int grid = num_sms() * 8;
  {
    ProfScope p("gate_up_simt", s);
    k_gate_up_simt<<<grid, 256, 0, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    ProfScope p("down_simt", s);
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
