// Expert FFN for decode batches.
//
// Tensor-core path (mma.sync m16n8k16, fp16 operands, fp32 accumulate).
// The codes become exact fp16 A-operands in registers:
//  - multi-token kernels: a code field ORed under the fp16 exponent of 1024
//    reads as 1024 + 4^s q, and one packed fp16 FMA with (sc 4^-s,
//    -1024 sc 4^-s) folds the Q2_K sub-block scale in exactly (sc q <= 45);
//    B is the fp16 rounding of the tokens' activations (values beyond the
//    fp16 range are flagged), up to 8 tokens of one expert on the n = 8 side;
//  - single-token kernels (t1.cuh): a 2-bit field at bit 2e of a 16-bit half
//    is the fp16 subnormal q 2^(2e - 24), used as is after one mask, and the
//    activation operand is pre-scaled by a power of two per field position,
//    so every product is exact.
// The Q2_K mins and the Q4_1 / Q4_K (d, m) are applied per sub-block or block
// in an fp32 epilogue, against sub-block sums of the activations carried as
// hi + lo fp16 pairs.  Weight rows are staged into shared memory by bulk
// asynchronous copies (TMA, non-tensor form) completing on mbarriers.
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
#include "span.cuh"
#include "t1.cuh"

namespace ds4 {
namespace {

constexpr int kTok = kGroup;  // tokens per pass (= MMA n)

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

// fp16x2 constants
constexpr uint32_t kMagicH = 0x64006400u;    // (1024, 1024)
constexpr uint32_t kOneH = 0x3C003C00u;      // (1, 1)
constexpr uint32_t kNeg1024H = 0xE400E400u;  // (-1024, -1024)
constexpr uint32_t kSixteenthH = 0x2C002C00u; // (1/16, 1/16)
constexpr uint32_t kNeg64H = 0xD400D400u;    // (-64, -64)

// Per-lane Q2_K constants.  Lane quad c walks the four 16-value sub-blocks
// 4c .. 4c+3 of every 256-value block (one sub-block per 4 consecutive MMAs,
// values 4j .. 4j+3 in MMA j); those sub-blocks sit in qs half c/2 at code
// positions s = 2 (c & 1) (sub-blocks 4c, 4c+1) and s + 1 (4c+2, 4c+3).
// A code at position s becomes the fp16 operand 1024 + 4^s q (one OR with
// the magic exponent), and the scale fold is exact:
//   (1024 + 4^s q) * (sc 4^-s) + (-1024 sc 4^-s) = sc q  (<= 45).
struct Q2kLane {
  uint32_t mask[2];  // code field of position s, s + 1 in both fp16 lanes
  uint32_t f1[2];    // 4^-s
  uint32_t f0[2];    // -1024 * 4^-s
};

__device__ __forceinline__ Q2kLane q2k_lane(int c) {
  Q2kLane k;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int s = 2 * (c & 1) + i;
    k.mask[i] = 0x00030003u << (2 * s);
    const uint32_t p = (uint32_t)(15 - 2 * s);            // fp16 exponent field of 4^-s
    k.f1[i] = (p << 10) | (p << 26);
    const uint32_t q = (uint32_t)(25 - 2 * s) | 0x20u;    // -(1024 * 4^-s): sign + exponent 25 - 2s
    k.f0[i] = (q << 10) | (q << 26);
  }
  return k;
}

// This lane's activations (fp16) for one 256-value segment.
// Q2_K mapping: bx[4i + j] = values 64c + 16i + 4j .. +3 (contiguous per lane);
// shi / slo = hi and lo parts of the sums of sub-blocks 4c .. 4c+3.
// Q4_1 mapping: bx[2b + h] = values 32b + 16h + 4c .. +3.
struct SegIn {
  uint2 bx[16];
  uint2 shi, slo;
};

template <int Q>
__device__ __forceinline__ void load_seg(SegIn &in, const uint16_t *__restrict__ xb,
                                         const uint8_t *__restrict__ sums, int c) {
  if constexpr (Q == DS4MOE_Q2_K || Q == DS4MOE_Q4_K) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint4 t = make_uint4(0u, 0u, 0u, 0u);
      if (xb) t = *reinterpret_cast<const uint4 *>(xb + 64 * c + 8 * u);
      in.bx[2 * u] = make_uint2(t.x, t.y);
      in.bx[2 * u + 1] = make_uint2(t.z, t.w);
    }
    in.shi = sums ? *reinterpret_cast<const uint2 *>(sums + 8 * c) : make_uint2(0u, 0u);
    in.slo = sums ? *reinterpret_cast<const uint2 *>(sums + 32 + 8 * c) : make_uint2(0u, 0u);
  } else {
#pragma unroll
    for (int n = 0; n < 16; ++n)
      in.bx[n] = xb ? *reinterpret_cast<const uint2 *>(xb + 32 * (n >> 1) + 16 * (n & 1) + 4 * c)
                    : make_uint2(0u, 0u);
    in.shi = in.slo = make_uint2(0u, 0u);
  }
}

// One Q2_K 256-value block of 16 staged rows (row g at blk_a, g + 8 at
// blk_b): acc += d * (sum sc*q*x) - dmin * (sum mn*xsum).
__device__ __forceinline__ void q2k_block(const uint8_t *__restrict__ blk_a, const uint8_t *__restrict__ blk_b,
                                          const SegIn &in, const Q2kLane &kl, int c, float (&acc)[4]) {
  const uint8_t *qsa = blk_a + 16 + 32 * (c >> 1), *qsb = blk_b + 16 + 32 * (c >> 1);
  const uint32_t swa = ptx::lds32(blk_a + 4 * c), swb = ptx::lds32(blk_b + 4 * c);
  const uint32_t dda = ptx::lds32(blk_a + 80), ddb = ptx::lds32(blk_b + 80);
  const uint32_t scma = swa & 0x0F0F0F0Fu, scmb = swb & 0x0F0F0F0Fu;
  // scale folding constants of sub-blocks 4c + i, rows a and b
  uint32_t s1a[4], s0a[4], s1b[4], s0b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t sel = 0x4040u | ((uint32_t)i << 8) | (uint32_t)i;   // (1024 + sc, 1024 + sc)
    s1a[i] = ptx::fma_f16x2(__byte_perm(scma, 0x64646464u, sel), kl.f1[i >> 1], kl.f0[i >> 1]);
    s1b[i] = ptx::fma_f16x2(__byte_perm(scmb, 0x64646464u, sel), kl.f1[i >> 1], kl.f0[i >> 1]);
    s0a[i] = ptx::mul_f16x2(s1a[i], kNeg1024H);
    s0b[i] = ptx::mul_f16x2(s1b[i], kNeg1024H);
  }
  float dm[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {            // qs word (4 consecutive values) of this lane
    const uint32_t qa = ptx::lds32(qsa + 4 * wi), qb = ptx::lds32(qsb + 4 * wi);
    const uint32_t a01 = __byte_perm(qa, 0, 0x4140), a23 = __byte_perm(qa, 0, 0x4342);
    const uint32_t b01 = __byte_perm(qb, 0, 0x4140), b23 = __byte_perm(qb, 0, 0x4342);
    const int j = wi & 3;
#pragma unroll
    for (int si = 0; si < 2; ++si) {          // code position s + si -> sub-block i
      const int i = (wi >> 2) + 2 * si;
      uint32_t A[4];
      A[0] = ptx::fma_f16x2(ptx::and_or(a01, kl.mask[si], kMagicH), s1a[i], s0a[i]);
      A[1] = ptx::fma_f16x2(ptx::and_or(b01, kl.mask[si], kMagicH), s1b[i], s0b[i]);
      A[2] = ptx::fma_f16x2(ptx::and_or(a23, kl.mask[si], kMagicH), s1a[i], s0a[i]);
      A[3] = ptx::fma_f16x2(ptx::and_or(b23, kl.mask[si], kMagicH), s1b[i], s0b[i]);
      ptx::mma_f16(dm[j & 1], A, in.bx[4 * i + j].x, in.bx[4 * i + j].y);
    }
  }
  // mins: D_min[r][t] = sum over sub-blocks 4c..4c+3 (K slots 2c, 2c+1,
  // 2c+8, 2c+9) of mn[r][n] * xsum[n][t], xsum = hi + lo
  float dn[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t ma = (swa >> 4) & 0x0F0F0F0Fu, mb = (swb >> 4) & 0x0F0F0F0Fu;
    uint32_t Am[4];
    Am[0] = ptx::fma_f16x2(__byte_perm(ma, 0, 0x4140) | kMagicH, kOneH, kNeg1024H);
    Am[1] = ptx::fma_f16x2(__byte_perm(mb, 0, 0x4140) | kMagicH, kOneH, kNeg1024H);
    Am[2] = ptx::fma_f16x2(__byte_perm(ma, 0, 0x4342) | kMagicH, kOneH, kNeg1024H);
    Am[3] = ptx::fma_f16x2(__byte_perm(mb, 0, 0x4342) | kMagicH, kOneH, kNeg1024H);
    ptx::mma_f16(dn, Am, in.shi.x, in.shi.y);
    ptx::mma_f16(dn, Am, in.slo.x, in.slo.y);
  }
  const float da = f16_bits_to_f32(dda & 0xFFFFu), dmina = f16_bits_to_f32(dda >> 16);
  const float db = f16_bits_to_f32(ddb & 0xFFFFu), dminb = f16_bits_to_f32(ddb >> 16);
  acc[0] = fmaf(da, dm[0][0] + dm[1][0], fmaf(-dmina, dn[0], acc[0]));
  acc[1] = fmaf(da, dm[0][1] + dm[1][1], fmaf(-dmina, dn[1], acc[1]));
  acc[2] = fmaf(db, dm[0][2] + dm[1][2], fmaf(-dminb, dn[2], acc[2]));
  acc[3] = fmaf(db, dm[0][3] + dm[1][3], fmaf(-dminb, dn[3], acc[3]));
}

// One Q4_K 256-value block of 16 staged rows (row g at blk_a, g + 8 at
// blk_b), the same activation mapping as Q2_K: lane quad c owns values
// 64c .. 64c + 63, i.e. qs bytes 32c .. 32c + 31, whose low nibbles are
// sub-block 2c and high nibbles sub-block 2c + 1 (32 values each).  qs word
// wi (values 4wi .. 4wi + 3 of each half) feeds two MMAs: the low nibbles
// against bx[wi], the high ones against bx[8 + wi].  A code under the fp16
// exponent of 1024 reads as 1024 + q (low) or 1024 + 16 q (high); one packed
// fp16 FMA with (sc, -1024 sc) or (sc / 16, -64 sc) leaves sc * q <= 945,
// exact.  The mins take one MMA pair against the 16-value sub-block sums:
// sub-block j's mn sits in the K slots of its two 16-value halves.
__device__ __forceinline__ void q4k_block(const uint8_t *__restrict__ blk_a, const uint8_t *__restrict__ blk_b,
                                          const SegIn &in, int c, float (&acc)[4]) {
  const uint32_t dda = ptx::lds32(blk_a), ddb = ptx::lds32(blk_b);
  uint32_t sa[3], sb[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    sa[q] = ptx::lds32(blk_a + 4 + 4 * q);
    sb[q] = ptx::lds32(blk_b + 4 + 4 * q);
  }
  uint32_t sca[2], mna[2], scb[2], mnb[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    q4k_sc_mn_pair(sa, 2 * c + h, sca[h], mna[h]);
    q4k_sc_mn_pair(sb, 2 * c + h, scb[h], mnb[h]);
  }
  // scale-fold constants: low nibbles (sub-block 2c) and high (2c + 1), rows a / b
  const auto h2 = [](float v) {
    const uint32_t b = __half_as_ushort(__float2half_rn(v));
    return b | (b << 16);
  };
  const uint32_t s1a0 = h2((float)sca[0]), s0a0 = h2(-1024.f * (float)sca[0]);
  const uint32_t s1b0 = h2((float)scb[0]), s0b0 = h2(-1024.f * (float)scb[0]);
  const uint32_t s1a1 = h2((float)sca[1] * 0.0625f), s0a1 = h2(-64.f * (float)sca[1]);
  const uint32_t s1b1 = h2((float)scb[1] * 0.0625f), s0b1 = h2(-64.f * (float)scb[1]);
  const uint8_t *qsa = blk_a + 16 + 32 * c, *qsb = blk_b + 16 + 32 * c;
  float dm[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    const uint32_t qa = ptx::lds32(qsa + 4 * wi), qb = ptx::lds32(qsb + 4 * wi);
    const uint32_t a01 = __byte_perm(qa, 0, 0x4140), a23 = __byte_perm(qa, 0, 0x4342);
    const uint32_t b01 = __byte_perm(qb, 0, 0x4140), b23 = __byte_perm(qb, 0, 0x4342);
    uint32_t A[4];
    A[0] = ptx::fma_f16x2(ptx::and_or(a01, 0x000F000Fu, kMagicH), s1a0, s0a0);
    A[1] = ptx::fma_f16x2(ptx::and_or(b01, 0x000F000Fu, kMagicH), s1b0, s0b0);
    A[2] = ptx::fma_f16x2(ptx::and_or(a23, 0x000F000Fu, kMagicH), s1a0, s0a0);
    A[3] = ptx::fma_f16x2(ptx::and_or(b23, 0x000F000Fu, kMagicH), s1b0, s0b0);
    ptx::mma_f16(dm[wi & 1], A, in.bx[wi].x, in.bx[wi].y);
    A[0] = ptx::fma_f16x2(ptx::and_or(a01, 0x00F000F0u, kMagicH), s1a1, s0a1);
    A[1] = ptx::fma_f16x2(ptx::and_or(b01, 0x00F000F0u, kMagicH), s1b1, s0b1);
    A[2] = ptx::fma_f16x2(ptx::and_or(a23, 0x00F000F0u, kMagicH), s1a1, s0a1);
    A[3] = ptx::fma_f16x2(ptx::and_or(b23, 0x00F000F0u, kMagicH), s1b1, s0b1);
    ptx::mma_f16(dm[wi & 1], A, in.bx[8 + wi].x, in.bx[8 + wi].y);
  }
  // mins: K slots 2c, 2c + 1 (16-value sums 4c, 4c + 1) carry mn of
  // sub-block 2c, slots 2c + 8, 2c + 9 (sums 4c + 2, 4c + 3) mn of 2c + 1
  float dn[4] = {0.f, 0.f, 0.f, 0.f};
  {
    uint32_t Am[4];
    Am[0] = h2((float)mna[0]);
    Am[1] = h2((float)mnb[0]);
    Am[2] = h2((float)mna[1]);
    Am[3] = h2((float)mnb[1]);
    ptx::mma_f16(dn, Am, in.shi.x, in.shi.y);
    ptx::mma_f16(dn, Am, in.slo.x, in.slo.y);
  }
  const float da = f16_bits_to_f32(dda & 0xFFFFu), dmina = f16_bits_to_f32(dda >> 16);
  const float db = f16_bits_to_f32(ddb & 0xFFFFu), dminb = f16_bits_to_f32(ddb >> 16);
  acc[0] = fmaf(da, dm[0][0] + dm[1][0], fmaf(-dmina, dn[0], acc[0]));
  acc[1] = fmaf(da, dm[0][1] + dm[1][1], fmaf(-dmina, dn[1], acc[1]));
  acc[2] = fmaf(db, dm[0][2] + dm[1][2], fmaf(-dminb, dn[2], acc[2]));
  acc[3] = fmaf(db, dm[0][3] + dm[1][3], fmaf(-dminb, dn[3], acc[3]));
}

// Eight Q4_1 blocks (one 256-value segment): per block
// acc += d * (sum q*x) + m * (sum x).  Low nibbles -> 1024 + q, high
// nibbles -> 1024 + 16 q, both turned into exact q by one packed FMA.
// xs_a / xs_b: the 8 block sums of tokens 2c and 2c + 1 (or nullptr).
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
    lo[0] = ptx::fma_f16x2(ptx::and_or(a01, 0x000F000Fu, kMagicH), kOneH, kNeg1024H);
    lo[1] = ptx::fma_f16x2(ptx::and_or(b01, 0x000F000Fu, kMagicH), kOneH, kNeg1024H);
    lo[2] = ptx::fma_f16x2(ptx::and_or(a23, 0x000F000Fu, kMagicH), kOneH, kNeg1024H);
    lo[3] = ptx::fma_f16x2(ptx::and_or(b23, 0x000F000Fu, kMagicH), kOneH, kNeg1024H);
    hi[0] = ptx::fma_f16x2(ptx::and_or(a01, 0x00F000F0u, kMagicH), kSixteenthH, kNeg64H);
    hi[1] = ptx::fma_f16x2(ptx::and_or(b01, 0x00F000F0u, kMagicH), kSixteenthH, kNeg64H);
    hi[2] = ptx::fma_f16x2(ptx::and_or(a23, 0x00F000F0u, kMagicH), kSixteenthH, kNeg64H);
    hi[3] = ptx::fma_f16x2(ptx::and_or(b23, 0x00F000F0u, kMagicH), kSixteenthH, kNeg64H);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    ptx::mma_f16(d, lo, in.bx[2 * bb].x, in.bx[2 * bb].y);
    ptx::mma_f16(d, hi, in.bx[2 * bb + 1].x, in.bx[2 * bb + 1].y);
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
constexpr int seg_bytes() { return Q == DS4MOE_Q2_K ? kQ2KBytes : Q == DS4MOE_Q4_K ? kQ4KBytes : 8 * kQ41Bytes; }

template <int Q>
__device__ __forceinline__ void seg_rows(const uint8_t *ra, const uint8_t *rb, const SegIn &in, const Q2kLane &kl,
                                         const float *xs_a, const float *xs_b, int c, float (&acc)[4]) {
  if constexpr (Q == DS4MOE_Q2_K) q2k_block(ra, rb, in, kl, c, acc);
  else if constexpr (Q == DS4MOE_Q4_K) q4k_block(ra, rb, in, c, acc);
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

// ============================================================ tile driver
// One staged 16-row tile chunk (row g at buf + g * ch) against this lane's
// token activations: nseg 256-value segments.
template <int Q>
__device__ __forceinline__ void tile_rows(const uint8_t *buf, uint32_t ch, int nseg, const uint16_t *xb,
                                          const uint8_t *sums, const float *xs_a, const float *xs_b,
                                          const Q2kLane &kl, int g, int c, float (&acc)[4]) {
  const uint8_t *ra = buf + g * ch, *rb = buf + (g + 8) * ch;
  for (int sg = 0; sg < nseg; ++sg) {
    SegIn in;
    load_seg<Q>(in, xb ? xb + 256 * sg : nullptr, sums ? sums + 64 * sg : nullptr, c);
    seg_rows<Q>(ra + seg_bytes<Q>() * sg, rb + seg_bytes<Q>() * sg, in, kl, xs_a ? xs_a + 8 * sg : nullptr,
                xs_b ? xs_b + 8 * sg : nullptr, c, acc);
  }
}

// ============================================================ gate / up
// CTA = 2 kp warps: warp w < kp computes K chunk w of the gate tile, warp
// kp + w the same chunk of the up tile.  Each warp stages its 16 rows x chunk
// bytes in two shared-memory stages; the K partials are summed in shared
// memory in a fixed order, then h = bf16(silu(g) * u) and the tile's
// sub-block sums of h are written.
template <int QG, int QU, bool FIN>
__global__ void __launch_bounds__(512) k_gate_up_mma(FfnArgs a, int kp, uint32_t chg, uint32_t chu) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_GATE_UP_MMA);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff;
  const bool is_up = w >= kp;
  const int part = is_up ? w - kp : w;
  const uint32_t ch = is_up ? chu : chg;
  const uint32_t stage_bytes = 16u * ch;
  uint8_t *wbuf = smem + (is_up ? (size_t)kp * 32 * chg + (size_t)part * 32 * chu : (size_t)part * 32 * chg);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kp * 32 * (chg + chu));  // [2 kp][2]
  float *red = reinterpret_cast<float *>(bars + 4 * kp);                              // [2 kp][32][4]
  uint64_t *mybar = bars + 2 * w;
  if (lane == 0) {
    ptx::mbar_init(&mybar[0], 1);
    ptx::mbar_init(&mybar[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const Q2kLane kl = q2k_lane(c);
  // groups, permutation, fp16 x and its sums come from the bucketing grid
  ptx::pdl_wait();
  span_begin(DS4MOE_SPAN_GATE_UP_MMA);
  ptx::pdl_launch_dependents();
  if (FIN && blockIdx.x == 0 && w == 0) finish_routing_weights(const_cast<float *>(a.w), a.T, a.k);
  clear_combine_counters(a, threadIdx.x, blockDim.x);
  const int ntile = F / 16;
  const int U = __ldcg(&a.hdr->n_groups) * ntile;
  const int64_t rb = is_up ? row_bytes(QU, D) : row_bytes(QG, D);
  const uint8_t *mat = static_cast<const uint8_t *>(is_up ? a.L.up : a.L.gate);
  const int kvals = D / kp, k0 = part * kvals;

  auto load_group = [&](int u) {
    const int4 v = __ldcg(reinterpret_cast<const int4 *>(a.groups + u / ntile));
    return Group{v.x, v.y, v.z, v.w};
  };
  // Every warp of the CTA works on the same unit, so the units' groups and
  // token ids live in a small shared ring: the group of unit it + 3 is
  // fetched during iteration it and its token ids during it + 1, so neither
  // dependent global load sits on a unit's critical path.
  __shared__ Group s_gq[4];
  __shared__ int s_tq[4][kGroup];  // token of pair p0 + j of the slot's group
  const int G = gridDim.x;
  auto tokens_of = [&](int slot, int j) {  // token id of pair j of the slot's group (-1 past its end)
    const Group gr = s_gq[slot];
    return j < gr.nt ? __ldcg(a.perm + gr.p0 + j) / a.k : -1;
  };
  auto issue = [&](int u, int st, const Group &grp) {
    const int row0 = (u % ntile) * 16;
    if (lane == 0) ptx::mbar_arrive_expect_tx(&mybar[st], stage_bytes);
    __syncwarp();
    stage_rows(wbuf + (size_t)st * stage_bytes, mat + ((int64_t)grp.e * F + row0) * rb + (int64_t)part * ch, rb,
               ch, &mybar[st], 0);
  };

  uint32_t phase = 0u;  // bit st: parity of stage st
  int u = blockIdx.x;
  // ring invariant at the top of iteration it: groups of units it .. it + 2
  // and token ids of units it, it + 1 are in slots (it + i) & 3
  if (threadIdx.x < 3 && u + G * (int)threadIdx.x < U) s_gq[threadIdx.x] = load_group(u + G * (int)threadIdx.x);
  __syncthreads();
  if (threadIdx.x < 2 * kGroup && u + G * (int)(threadIdx.x / kGroup) < U)
    s_tq[threadIdx.x / kGroup][threadIdx.x % kGroup] = tokens_of(threadIdx.x / kGroup, threadIdx.x % kGroup);
  __syncthreads();
  if (u < U) issue(u, 0, s_gq[0]);
  if (u + G < U) issue(u + G, 1, s_gq[1]);
  bool timed_out = false;
  for (int it = 0; u < U; u += G, ++it) {
    const int st = it & 1, sl = it & 3;
    const Group grp = s_gq[sl];
    const int row0 = (u % ntile) * 16;
    // prefetch (stored after this unit's arithmetic): thread 0 the group of
    // unit it + 3, threads 32 .. 32 + kGroup - 1 the token ids of unit it + 2
    Group gpre{};
    int tpre = -1;
    const bool pre_g = threadIdx.x == 0 && u + 3 * G < U;
    const bool pre_t = threadIdx.x >= 32 && threadIdx.x < 32 + kGroup && u + 2 * G < U;
    if (pre_g) gpre = load_group(u + 3 * G);
    if (pre_t) tpre = tokens_of((it + 2) & 3, (int)threadIdx.x - 32);
    if (!timed_out && !ptx::mbar_wait(&mybar[st], (phase >> st) & 1u)) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    phase ^= 1u << st;
    // this lane's token (B column g) and the tokens of its D columns 2c, 2c+1
    const uint16_t *xb = nullptr;
    const uint8_t *sums = nullptr;
    const float *xs_a = nullptr, *xs_b = nullptr;
    if (g < grp.nt) {
      const int t = s_tq[sl][g];
      xb = a.x16 + (int64_t)t * D + k0;
      sums = a.xs16 + ((int64_t)t * (D / 256 + 1) + k0 / 256) * 64;
    }
    if (2 * c < grp.nt) xs_a = a.xs32 + (int64_t)s_tq[sl][2 * c] * (D / 32) + k0 / 32;
    if (2 * c + 1 < grp.nt) xs_b = a.xs32 + (int64_t)s_tq[sl][2 * c + 1] * (D / 32) + k0 / 32;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (!timed_out) {
      const uint8_t *buf = wbuf + (size_t)st * stage_bytes;
      if (is_up) tile_rows<QU>(buf, ch, kvals / 256, xb, sums, xs_a, xs_b, kl, g, c, acc);
      else tile_rows<QG>(buf, ch, kvals / 256, xb, sums, xs_a, xs_b, kl, g, c, acc);
    }
    __syncwarp();
    if (u + 2 * G < U && !timed_out) issue(u + 2 * G, st, s_gq[(it + 2) & 3]);
    float *r = red + ((size_t)w * 32 + lane) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = acc[i];
    // slot (it + 3) & 3 held unit it - 1, which no warp reads any more
    if (pre_g) s_gq[(it + 3) & 3] = gpre;
    if (pre_t) s_tq[(it + 2) & 3][threadIdx.x - 32] = tpre;
    __syncthreads();
    if (w == 0) {
      float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
      for (int p = 0; p < kp; ++p) {
        const float *qg = red + ((size_t)p * 32 + lane) * 4, *qu = red + ((size_t)(kp + p) * 32 + lane) * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gs[i] += qg[i];
          us[i] += qu[i];
        }
      }
      // h for rows (g, g+8) x tokens (2c, 2c+1)
      float hsum[2] = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = row0 + g + 8 * (i >> 1);
        const int tok = 2 * c + (i & 1);
        if (tok < grp.nt) {
          // h is rounded to bf16 (the definition), then stored as the fp16
          // operand of the down kernel (exact for |h| in [2^-14, 65504])
          const float hv = bf16_bits_to_f32(f32_to_bf16_bits(silu(gs[i]) * us[i]));
          if (fabsf(hv) > 65504.f) record_status(a.hdr, DS4MOE_EDEVICE);
          a.h[(int64_t)(grp.p0 + tok) * F + row] = __half_as_ushort(__float2half_rn(hv));
          hsum[i & 1] += hv;
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
            const __half hi = __float2half_rn(hsum[i]);
            const __half lo = __float2half_rn(hsum[i] - __half2float(hi));
            uint16_t *rec = reinterpret_cast<uint16_t *>(
                a.hs16 + ((int64_t)(grp.p0 + tok) * (F / 256 + 1) + n16 / 16) * 64);
            rec[n16 & 15] = __half_as_ushort(hi);
            rec[16 + (n16 & 15)] = __half_as_ushort(lo);
          }
        }
      }
    }
    __syncthreads();
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out) {
    for (int st = 0; st < 2; ++st) ptx::mbar_wait(&mybar[st], (phase >> st) & 1u, 1u << 20);
  }
}

// ====================================================== gate / up, persistent
// T > 1 with gate and up in one format (Q2_K or Q4_1), d_model <= 4096: one
// CTA per SM with nbk = d_model / 256 consumer warps (warp w: 256-value K
// block w of both the gate and the up tile), a producer warp that streams
// whole 16-row gate + up tiles (one or a few bulk copies each, the T = 1
// bank-group layout) into a ring, and a reducer warp.  Each CTA takes a
// contiguous range of the (token group, 16-row tile) units, so consecutive
// units mostly share their token group and a consumer loads that group's
// activation operand into registers only when the group changes.  The
// reducer sums the K partials in a fixed order (warp 0 .. nbk - 1), applies
// SwiGLU and writes h and its sub-block sums, the operands of the down
// kernels, exactly as the one-CTA-per-unit kernel does.
constexpr int kMtMaxK = 16;  // consumer warps: d_model <= 4096
constexpr int kMtPart = 2;   // partial-sum slots between the consumers and the reducer

size_t gate_up_mt_smem(uint32_t tile, int nbk, int nstage) {
  return (size_t)nstage * 2 * tile + (size_t)kMtPart * nbk * 32 * 2 * sizeof(float4) +
         sizeof(uint64_t) * (2 * (size_t)nstage + 2 * kMtPart);
}

template <int Q, bool FIN>
__global__ void __launch_bounds__((kMtMaxK + 2) * 32, 1) k_gate_up_mt(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_GATE_UP_MMA);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nbk = D / 256;
  const int64_t rb = row_bytes(Q, D);
  const T1Tile tl = t1_tile((uint32_t)rb);
  const uint32_t tile = t1_tile_bytes(tl), stage = 2u * tile;
  const int wprod = nbk, wred = nbk + 1;
  // shared memory: stages (gate tile | up tile) | partials | barriers
  float4 *red = reinterpret_cast<float4 *>(smem + (size_t)nstage * stage);  // [kMtPart][nbk][32][2]
  uint64_t *full = reinterpret_cast<uint64_t *>(red + (size_t)kMtPart * nbk * 64);
  uint64_t *empty = full + nstage, *pfull = empty + nstage, *pempty = pfull + kMtPart;
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&full[st], 1);
      ptx::mbar_init(&empty[st], nbk);
    }
    for (int pt = 0; pt < kMtPart; ++pt) {
      ptx::mbar_init(&pfull[pt], nbk);
      ptx::mbar_init(&pempty[pt], 1);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const Q2kLane kl = q2k_lane(c);
  // groups, permutation, fp16 x and its sums come from the bucketing grid
  ptx::pdl_wait();
  span_begin(DS4MOE_SPAN_GATE_UP_MMA);
  ptx::pdl_launch_dependents();
  if (FIN && blockIdx.x == 0 && w == wred) finish_routing_weights(const_cast<float *>(a.w), a.T, a.k);
  clear_combine_counters(a, threadIdx.x, blockDim.x);
  const int ntile = F / 16;
  const int U = __ldcg(&a.hdr->n_groups) * ntile, G = gridDim.x;
  const int u0 = (int)((int64_t)blockIdx.x * U / G), u1 = (int)((int64_t)(blockIdx.x + 1) * U / G);
  auto load_group = [&](int gi) {
    const int4 v = __ldcg(reinterpret_cast<const int4 *>(a.groups + gi));
    return Group{v.x, v.y, v.z, v.w};
  };
  bool timed_out = false;
  if (w == wprod) {
    const uint8_t *gate = static_cast<const uint8_t *>(a.L.gate), *up = static_cast<const uint8_t *>(a.L.up);
    const uint32_t nc = t1_copies(tl);
    int gi = -1, issued = 0;
    Group grp{};
    for (int u = u0; u < u1; ++u, ++issued) {
      const int it = u - u0, st = it % nstage;
      if (it >= nstage && !ptx::mbar_wait(&empty[st], ((it / nstage) & 1) ^ 1)) {
        if (lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        break;
      }
      if (u / ntile != gi) {
        gi = u / ntile;
        grp = load_group(gi);
      }
      const int64_t row0 = (int64_t)grp.e * F + (u % ntile) * 16;
      uint8_t *dst = smem + (size_t)st * stage;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&full[st], 32u * (uint32_t)rb);
      __syncwarp();
      if ((uint32_t)lane < 2u * nc) {
        const uint32_t mat = (uint32_t)lane / nc, i = (uint32_t)lane % nc;
        t1_tile_copy(dst + mat * tile, (mat == 0 ? gate : up) + row0 * rb, tl, i, &full[st]);
      }
      __syncwarp();
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (lane == 0)
      for (int it = issued - nstage > 0 ? issued - nstage : 0; it < issued; ++it)
        ptx::mbar_wait(&full[it % nstage], (uint32_t)(it / nstage) & 1u, 1u << 20);
  } else if (w < nbk) {
    int gi = -1;
    SegIn in;
    const float *xs_a = nullptr, *xs_b = nullptr;
    const uint32_t og = t1_row_off(tl, (uint32_t)g), og8 = t1_row_off(tl, (uint32_t)g + 8u);
    const uint32_t kb = (uint32_t)w * (uint32_t)seg_bytes<Q>();
    for (int u = u0; u < u1; ++u) {
      const int it = u - u0, st = it % nstage;
      if (u / ntile != gi) {
        // a new token group: this lane's token (B column g), the tokens of
        // its D columns 2c, 2c + 1, and K block w of their activations
        gi = u / ntile;
        const Group grp = load_group(gi);
        const int tg = g < grp.nt ? __ldcg(a.perm + grp.p0 + g) / a.k : -1;
        const int ta = 2 * c < grp.nt ? __ldcg(a.perm + grp.p0 + 2 * c) / a.k : -1;
        const int tb = 2 * c + 1 < grp.nt ? __ldcg(a.perm + grp.p0 + 2 * c + 1) / a.k : -1;
        load_seg<Q>(in, tg >= 0 ? a.x16 + (int64_t)tg * D + 256 * w : nullptr,
                    tg >= 0 ? a.xs16 + ((int64_t)tg * (D / 256 + 1) + w) * 64 : nullptr, c);
        xs_a = ta >= 0 ? a.xs32 + (int64_t)ta * (D / 32) + 8 * w : nullptr;
        xs_b = tb >= 0 ? a.xs32 + (int64_t)tb * (D / 32) + 8 * w : nullptr;
      }
      if (!timed_out && !ptx::mbar_wait(&full[st], (uint32_t)(it / nstage) & 1u)) {
        if (lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
      if (!timed_out) {
        const uint8_t *sp = smem + (size_t)st * stage;
        seg_rows<Q>(sp + og + kb, sp + og8 + kb, in, kl, xs_a, xs_b, c, ag);
        seg_rows<Q>(sp + tile + og + kb, sp + tile + og8 + kb, in, kl, xs_a, xs_b, c, au);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      // partial slot it % kMtPart: free once the reducer has read unit it - kMtPart
      const int pt = it % kMtPart;
      if (it >= kMtPart && !ptx::mbar_wait(&pempty[pt], ((uint32_t)(it / kMtPart) & 1u) ^ 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      float4 *rp = red + (((size_t)pt * nbk + w) * 32 + lane) * 2;
      rp[0] = make_float4(ag[0], ag[1], ag[2], ag[3]);
      rp[1] = make_float4(au[0], au[1], au[2], au[3]);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pfull[pt]);
    }
  } else if (w == wred) {
    int gi = -1;
    Group grp{};
    for (int u = u0; u < u1; ++u) {
      const int it = u - u0, pt = it % kMtPart;
      if (u / ntile != gi) {
        gi = u / ntile;
        grp = load_group(gi);
      }
      if (!ptx::mbar_wait(&pfull[pt], (uint32_t)(it / kMtPart) & 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      float gs[4] = {0.f, 0.f, 0.f, 0.f}, us[4] = {0.f, 0.f, 0.f, 0.f};
      for (int p = 0; p < nbk; ++p) {  // K blocks in order: a fixed summation order
        const float4 *q = red + (((size_t)pt * nbk + p) * 32 + lane) * 2;
        const float4 qg = q[0], qu = q[1];
        gs[0] += qg.x; gs[1] += qg.y; gs[2] += qg.z; gs[3] += qg.w;
        us[0] += qu.x; us[1] += qu.y; us[2] += qu.z; us[3] += qu.w;
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pempty[pt]);
      const int row0 = (u % ntile) * 16;
      // h for rows (g, g + 8) x tokens (2c, 2c + 1)
      float hsum[2] = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = row0 + g + 8 * (i >> 1);
        const int tok = 2 * c + (i & 1);
        if (tok < grp.nt) {
          // h is rounded to bf16 (the definition), then stored as the fp16
          // operand of the down kernel (exact for |h| in [2^-14, 65504])
          const float hv = bf16_bits_to_f32(f32_to_bf16_bits(silu(gs[i]) * us[i]));
          if (fabsf(hv) > 65504.f) record_status(a.hdr, DS4MOE_EDEVICE);
          a.h[(int64_t)(grp.p0 + tok) * F + row] = __half_as_ushort(__float2half_rn(hv));
          hsum[i & 1] += hv;
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
            const __half hi = __float2half_rn(hsum[i]);
            const __half lo = __float2half_rn(hsum[i] - __half2float(hi));
            uint16_t *rec = reinterpret_cast<uint16_t *>(
                a.hs16 + ((int64_t)(grp.p0 + tok) * (F / 256 + 1) + n16 / 16) * 64);
            rec[n16 & 15] = __half_as_ushort(hi);
            rec[16 + (n16 & 15)] = __half_as_ushort(lo);
          }
        }
      }
    }
  }
}

// ================================================================ down
// Weighted combine fused into the down kernel: each warp counts, per token of
// its group, one arrival at (token, 16-row tile); the warp that brings the
// count to the token's number of valid experts sums that tile of
// out[t] = sum_{i<k} w[t,i] * y[inv[t,i]] in rank order (so the result does
// not depend on which warp finishes last) and resets the counter.
__device__ __forceinline__ void combine_tile(const FfnArgs &a, const Group &grp, int tile, int ntile) {
  const int lane = threadIdx.x & 31;
  const int D = a.L.d_model, k = a.k;
  __threadfence();  // this lane's y stores are visible before it is counted
  __syncwarp();
  int tok = -1;
  bool last = false;
  if (lane < grp.nt) {
    tok = __ldcg(a.perm + grp.p0 + lane) / k;
    const int old = atomicAdd(a.cnt + (int64_t)tok * ntile + tile, 1);
    last = old == __ldcg(a.nvalid + tok) - 1;
    if (last) a.cnt[(int64_t)tok * ntile + tile] = 0;
  }
  unsigned lm = __ballot_sync(0xffffffffu, last);
  while (lm) {
    const int src = __ffs(lm) - 1;
    lm &= lm - 1u;
    const int t = __shfl_sync(0xffffffffu, tok, src);
    __threadfence();  // the other experts' y tiles are visible after the count
    if (lane < 16) {
      const int row = tile * 16 + lane;
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int pos = __ldcg(a.inv + (int64_t)t * k + j);
        if (pos < 0) continue;
        acc = fmaf(__ldcg(a.w + (int64_t)t * k + j), __ldcg(a.y + (int64_t)pos * D + row), acc);
      }
      a.out[(int64_t)t * D + row] = acc;
    }
  }
}

// One warp per (token group, 16-row tile) over the full K (= d_ff), NST
// shared-memory stages per warp.  The first tiles are prefetched before the
// dependency wait: the token groups were complete before the gate/up grid
// (whose h this kernel reads) launched it.
template <int NST>
__global__ void __launch_bounds__(256) k_down_mma(FfnArgs a, uint32_t chd) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_DOWN_MMA);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int nw = blockDim.x >> 5;
  const int D = a.L.d_model, F = a.L.d_ff;
  const Q2kLane kl = q2k_lane(c);
  const uint32_t stage_bytes = 16u * chd;
  uint8_t *wbuf = smem + (size_t)w * NST * stage_bytes;
  uint64_t *mybar = reinterpret_cast<uint64_t *>(smem + (size_t)nw * NST * stage_bytes) + NST * w;
  if (lane == 0) {
    for (int st = 0; st < NST; ++st) ptx::mbar_init(&mybar[st], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const int ntile = D / 16;
  const int U = __ldcg(&a.hdr->n_groups) * ntile;
  const int64_t rbd = row_bytes(DS4MOE_Q2_K, F);
  const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
  const int gw = blockIdx.x * nw + w, nwarps = gridDim.x * nw;

  auto load_group = [&](int u) {
    const int4 v = __ldcg(reinterpret_cast<const int4 *>(a.groups + u / ntile));
    return Group{v.x, v.y, v.z, v.w};
  };
  auto issue = [&](int u, int st) {
    const Group grp = load_group(u);
    const int row0 = (u % ntile) * 16;
    if (lane == 0) ptx::mbar_arrive_expect_tx(&mybar[st], stage_bytes);
    __syncwarp();
    stage_rows(wbuf + (size_t)st * stage_bytes, down + ((int64_t)grp.e * D + row0) * rbd, rbd, chd, &mybar[st], 0);
  };

  uint32_t phase = 0u;
  int u = gw;
  for (int st = 0; st < NST; ++st)
    if (u + st * nwarps < U) issue(u + st * nwarps, st);
  ptx::pdl_wait();  // h and its sums come from the gate/up grid
  span_begin(DS4MOE_SPAN_DOWN_MMA);
  ptx::pdl_launch_dependents();
  bool timed_out = false;
  for (int it = 0; u < U; u += nwarps, ++it) {
    const int st = NST == 1 ? 0 : it % NST;
    const Group grp = load_group(u);
    const int row0 = (u % ntile) * 16;
    if (!timed_out && !ptx::mbar_wait(&mybar[st], (phase >> st) & 1u)) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    phase ^= 1u << st;
    const uint16_t *xb = nullptr;
    const uint8_t *sums = nullptr;
    if (g < grp.nt) {
      xb = a.h + (int64_t)(grp.p0 + g) * F;
      sums = a.hs16 + (int64_t)(grp.p0 + g) * (F / 256 + 1) * 64;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (!timed_out) tile_rows<DS4MOE_Q2_K>(wbuf + (size_t)st * stage_bytes, chd, F / 256, xb, sums, nullptr, nullptr,
                                          kl, g, c, acc);
    __syncwarp();
    if (u + NST * nwarps < U && !timed_out) issue(u + NST * nwarps, st);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 2 * c + (i & 1);
      if (tok < grp.nt) a.y[(int64_t)(grp.p0 + tok) * D + row0 + g + 8 * (i >> 1)] = acc[i];
    }
    if (a.cnt) combine_tile(a, grp, u % ntile, ntile);
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out) {
    for (int st = 0; st < NST; ++st) ptx::mbar_wait(&mybar[st], (phase >> st) & 1u, 1u << 20);
  }
}

// ================================================================ down, persistent
// T > 1, Q2_K or Q4_K down, d_ff in {1024, 2048, 4096}: one CTA per SM, 16 consumer
// warps over units of kDmtTpw * 16 / nbk 16-row tiles (nbk = d_ff / 256): warp
// w takes K block w % nbk of tiles w / nbk + (16 / nbk) j, j < kDmtTpw, and
// keeps that K block of its token group's h (the operand the gate/up kernels
// wrote) in registers while consecutive units share the group -- each CTA
// takes a contiguous range of units.  A producer warp streams the unit's
// tiles (the single-token bank-group layout) into a ring; a reducer warp sums
// each tile's K partials in order and writes y.  The weighted combine runs
// as its own grid.  Two tiles per warp and unit halve the unit's fixed cost
// (ring and partial hand-offs) per MMA.
constexpr int kDmtWarps = 16;
constexpr int kDmtTpw = 2;

size_t down_mt_smem(uint32_t tile, int tpu, int nstage) {
  return (size_t)nstage * tpu * kDmtTpw * tile + (size_t)kMtPart * kDmtWarps * kDmtTpw * 32 * sizeof(float4) +
         sizeof(uint64_t) * (2 * (size_t)nstage + 2 * kMtPart);
}

template <int Q>
__global__ void __launch_bounds__((kDmtWarps + 2) * 32, 1) k_down_mt(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_DOWN_MMA);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nbk = F / 256, tpu = kDmtWarps / nbk;
  const int64_t rbd = row_bytes(Q, F);
  const T1Tile tl = t1_tile((uint32_t)rbd);
  const int upt = tpu * kDmtTpw;  // tiles per unit
  const uint32_t tile = t1_tile_bytes(tl), stage = (uint32_t)upt * tile;
  const int wprod = kDmtWarps, wred = kDmtWarps + 1;
  float4 *red = reinterpret_cast<float4 *>(smem + (size_t)nstage * stage);  // [kMtPart][kDmtTpw][16][32]
  uint64_t *full = reinterpret_cast<uint64_t *>(red + (size_t)kMtPart * kDmtWarps * kDmtTpw * 32);
  uint64_t *empty = full + nstage, *pfull = empty + nstage, *pempty = pfull + kMtPart;
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&full[st], 1);
      ptx::mbar_init(&empty[st], kDmtWarps);
    }
    for (int pt = 0; pt < kMtPart; ++pt) {
      ptx::mbar_init(&pfull[pt], kDmtWarps);
      ptx::mbar_init(&pempty[pt], 1);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const Q2kLane kl = q2k_lane(c);
  const int ntu = D / (16 * upt);  // units per token group
  // the token groups were complete before the gate/up grid (whose h this
  // kernel reads) launched it: the producer starts before the dependency wait
  const int U = __ldcg(&a.hdr->n_groups) * ntu, G = gridDim.x;
  const int u0 = (int)((int64_t)blockIdx.x * U / G), u1 = (int)((int64_t)(blockIdx.x + 1) * U / G);
  auto load_group = [&](int gi) {
    const int4 v = __ldcg(reinterpret_cast<const int4 *>(a.groups + gi));
    return Group{v.x, v.y, v.z, v.w};
  };
  bool timed_out = false;
  if (w == wprod) {
    const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
    const uint32_t nc = t1_copies(tl);
    int gi = -1, issued = 0;
    Group grp{};
    for (int u = u0; u < u1; ++u, ++issued) {
      const int it = u - u0, st = it % nstage;
      if (it >= nstage && !ptx::mbar_wait(&empty[st], ((it / nstage) & 1) ^ 1)) {
        if (lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        break;
      }
      if (u / ntu != gi) {
        gi = u / ntu;
        grp = load_group(gi);
      }
      const int64_t row0 = (int64_t)grp.e * D + (int64_t)(u % ntu) * 16 * upt;
      uint8_t *dst = smem + (size_t)st * stage;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&full[st], (uint32_t)(16 * upt) * (uint32_t)rbd);
      __syncwarp();
      for (uint32_t ci = (uint32_t)lane; ci < (uint32_t)upt * nc; ci += 32u) {  // upt * nc may exceed 32
        const uint32_t m = ci / nc, i = ci % nc;
        t1_tile_copy(dst + m * tile, down + (row0 + 16 * (int64_t)m) * rbd, tl, i, &full[st]);
      }
      __syncwarp();
    }
    if (lane == 0)
      for (int it = issued - nstage > 0 ? issued - nstage : 0; it < issued; ++it)
        ptx::mbar_wait(&full[it % nstage], (uint32_t)(it / nstage) & 1u, 1u << 20);
  }
  ptx::pdl_wait();  // h and its sums come from the gate/up grid
  span_begin(DS4MOE_SPAN_DOWN_MMA);
  ptx::pdl_launch_dependents();
  if (w < kDmtWarps) {
    const int m = w / nbk, kbw = w % nbk;
    int gi = -1;
    SegIn in;
    const uint32_t og = t1_row_off(tl, (uint32_t)g) + (uint32_t)(kbw * seg_bytes<Q>()),
                   og8 = t1_row_off(tl, (uint32_t)g + 8u) + (uint32_t)(kbw * seg_bytes<Q>());
    for (int u = u0; u < u1; ++u) {
      const int it = u - u0, st = it % nstage;
      if (u / ntu != gi) {
        gi = u / ntu;
        const Group grp = load_group(gi);
        const int p = grp.p0 + g;  // this lane's pair (B column g)
        load_seg<Q>(in, g < grp.nt ? a.h + (int64_t)p * F + 256 * kbw : nullptr,
                              g < grp.nt ? a.hs16 + ((int64_t)p * (F / 256 + 1) + kbw) * 64 : nullptr, c);
      }
      if (!timed_out && !ptx::mbar_wait(&full[st], (uint32_t)(it / nstage) & 1u)) {
        if (lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      float acc[kDmtTpw][4];
#pragma unroll
      for (int j = 0; j < kDmtTpw; ++j) {
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        if (!timed_out) {
          const uint8_t *sp = smem + (size_t)st * stage + (size_t)(m + tpu * j) * tile;
          seg_rows<Q>(sp + og, sp + og8, in, kl, nullptr, nullptr, c, acc[j]);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      const int pt = it % kMtPart;
      if (it >= kMtPart && !ptx::mbar_wait(&pempty[pt], ((uint32_t)(it / kMtPart) & 1u) ^ 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
#pragma unroll
      for (int j = 0; j < kDmtTpw; ++j)
        red[(((size_t)pt * kDmtTpw + j) * kDmtWarps + w) * 32 + lane] =
            make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pfull[pt]);
    }
  } else if (w == wred) {
    int gi = -1;
    Group grp{};
    for (int u = u0; u < u1; ++u) {
      const int it = u - u0, pt = it % kMtPart;
      if (u / ntu != gi) {
        gi = u / ntu;
        grp = load_group(gi);
      }
      if (!ptx::mbar_wait(&pfull[pt], (uint32_t)(it / kMtPart) & 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      const int row0 = (u % ntu) * 16 * upt;
      for (int mt = 0; mt < upt; ++mt) {  // tile mt = m + tpu j of the unit
        const int j = mt / tpu, m = mt % tpu;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kb = 0; kb < nbk; ++kb) {  // K blocks in order: a fixed summation order
          const float4 q = red[(((size_t)pt * kDmtTpw + j) * kDmtWarps + m * nbk + kb) * 32 + lane];
          v[0] += q.x;
          v[1] += q.y;
          v[2] += q.z;
          v[3] += q.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = 2 * c + (i & 1);
          if (tok < grp.nt) a.y[(int64_t)(grp.p0 + tok) * D + row0 + 16 * mt + g + 8 * (i >> 1)] = v[i];
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pempty[pt]);
    }
  }
}

// gate/up + SwiGLU for T = 1: warps 0 .. nb-1 consume block w of d_model for
// the 16 gate and 16 up rows of a tile, warp nb produces.  Units (group,
// 16-row tile) are dealt to the CTAs round-robin; the warp that finishes a
// unit last sums the blocks and writes h.
template <bool FIN, int FMT>
__global__ void __launch_bounds__(17 * 32, 1) k_gate_up_t1(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_GATE_UP_T1);
  constexpr int kBB = FMT == DS4MOE_Q4_K ? kQ4KBytes : kQ2KBytes;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nb = D / 256;
  const T1Tile tl = t1_tile((uint32_t)(kBB * nb));
  const uint32_t tile_bytes = t1_tile_bytes(tl), stage_bytes = 2u * tile_bytes;
  const uint32_t ncp = t1_copies(tl);
  const T1Smem sm = t1_smem(smem, nstage, stage_bytes, nb);
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&sm.full[st], 1);
      ptx::mbar_init(&sm.empty[st], nb);
      sm.cnt[st] = 0;
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const T1Lane L = t1_lane(c);
  T1B B;
  // the activations are the call's input: loaded before the dependency wait
  if (w < nb) {
    if constexpr (FMT == DS4MOE_Q4_K) t1_load_b_q4k<true>(B, a.x + 256 * w, g, c);
    else t1_load_b<true>(B, a.x + 256 * w, g, c);
  }
  ptx::pdl_wait();  // groups (or the logits) come from the routing grid
  span_begin(DS4MOE_SPAN_GATE_UP_T1);
  ptx::pdl_launch_dependents();
  const int ntile = F / 16;
  __shared__ Group s_grp[kT1MaxGroups];
  __shared__ int s_ngrp;
  if (a.lg) {
    // the producer warp ranks the experts (the consumers hold x)
    if (w == nb) t1_route_warp(a, s_grp, &s_ngrp, blockIdx.x == 0);
    __syncthreads();
  } else {
    t1_load_groups(a, s_grp, &s_ngrp);
  }
  if (w == nb) clear_combine_counters(a, lane, 32);
  // units dealt round-robin: at any moment the CTAs read neighbouring tiles,
  // so DRAM sees a few long sequential streams instead of one short range
  // per CTA (the activations are the same for every unit)
  const int U = s_ngrp * ntile;
  const int u0 = blockIdx.x, ustep = gridDim.x;
  const int nunits = u0 < U ? (U - u0 + ustep - 1) / ustep : 0;
  auto load_group = [&](int u) { return s_grp[u / ntile]; };
  if (w == nb) {
    // producer
    const uint8_t *gate = static_cast<const uint8_t *>(a.L.gate), *up = static_cast<const uint8_t *>(a.L.up);
    for (int u = u0, it = 0; u < U; u += ustep, ++it) {
      const int st = it % nstage;
      if (it >= nstage && !ptx::mbar_wait(&sm.empty[st], ((it / nstage) - 1) & 1)) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        break;
      }
      const Group grp = load_group(u);
      const int row0 = (u % ntile) * 16;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&sm.full[st], 32u * tl.rowb);
      __syncwarp();
      // gate tile, then up tile: ncp copies each
      if ((uint32_t)lane < 2u * ncp) {
        const uint32_t mat = (uint32_t)lane / ncp, i = (uint32_t)lane % ncp;
        const uint8_t *src = (mat == 0 ? gate : up) + ((int64_t)grp.e * F + row0) * tl.rowb;
        t1_tile_copy(smem + (size_t)st * stage_bytes + mat * tile_bytes, src, tl, i, &sm.full[st]);
      }
      if (FIN && blockIdx.x == 0 && it == nstage - 1) finish_routing_weights(const_cast<float *>(a.w), a.T, a.k);
    }
    if (FIN && blockIdx.x == 0 && nunits < nstage) finish_routing_weights(const_cast<float *>(a.w), a.T, a.k);
    return;
  }
  bool timed_out = false;
  int it = 0;
  for (int u = u0; u < U; u += ustep, ++it) {
    const int st = it % nstage;
    if (!timed_out && !ptx::mbar_wait(&sm.full[st], (it / nstage) & 1)) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    float y[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (!timed_out) {
      const uint8_t *sb = smem + (size_t)st * stage_bytes + kBB * w;
      const uint8_t *const mats[2] = {sb, sb + tile_bytes};
      if constexpr (FMT == DS4MOE_Q4_K) t1_block_q4k<2>(mats, tl, g, c, B, y);
      else t1_block<2>(mats, tl, g, B, L, y);
    }
    // partials of this block: gate rows g, g+8 at [g], [g+8], up at [16+g], [24+g]
    float *r = sm.red + ((size_t)st * nb + w) * 32;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float v = quad_sum(y[m][q]);
        if (c == 0) r[16 * m + 8 * q + g] = v;
      }
    if (t1_last_arriver(&sm.cnt[st], nb)) {
      // lane l: gate row l (l < 16) or up row l - 16, blocks summed in order
      const float *rr = sm.red + (size_t)st * nb * 32 + lane;
      float sv = 0.f;
      for (int p = 0; p < nb; ++p) sv += rr[32 * p];
      const float us = __shfl_down_sync(0xffffffffu, sv, 16);
      const Group grp = load_group(u);
      const int row0 = (u % ntile) * 16;
      float hv = 0.f;
      // a group holds more than one slot only when the token names its
      // expert more than once: every slot gets the same h
      if (lane < 16) {
        // h rounded to bf16 (the definition), stored as the fp16 operand of
        // the down kernel (exact for |h| in [2^-14, 65504])
        hv = bf16_bits_to_f32(f32_to_bf16_bits(silu(sv) * us));
        if (fabsf(hv) > 65504.f) record_status(a.hdr, DS4MOE_EDEVICE);
        uint16_t *hp = a.h + (int64_t)grp.p0 * F + row0 + lane;
        const uint16_t hb = __half_as_ushort(__float2half_rn(hv));
#pragma unroll 1
        for (int j = 0; j < grp.nt; ++j, hp += F) *hp = hb;
      }
#pragma unroll
      for (int off = 8; off; off >>= 1) hv += __shfl_xor_sync(0xffffffffu, hv, off);
      if (lane < grp.nt) {
        const int n16 = row0 / 16;
        const __half hi = __float2half_rn(hv);
        const __half lo = __float2half_rn(hv - __half2float(hi));
        uint16_t *rec =
            reinterpret_cast<uint16_t *>(a.hs16 + ((int64_t)(grp.p0 + lane) * (F / 256 + 1) + n16 / 16) * 64);
        rec[n16 & 15] = __half_as_ushort(hi);
        rec[16 + (n16 & 15)] = __half_as_ushort(lo);
      }
    }
    // the stage (weights and partials) may be refilled once every warp is here
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sm.empty[st]);
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out && lane == 0) {
    for (int j = it - nstage > 0 ? it - nstage : 0; j < it; ++j)
      ptx::mbar_wait(&sm.full[j % nstage], (j / nstage) & 1, 1u << 20);
  }
}

// down for T = 1: warps 0 .. nb-1 consume block w of d_ff for a 16-row tile
// of one expert (its h loaded when the group changes), warp nb produces;
// contiguous unit ranges per CTA, so a CTA sees at most a few groups.  The
// warp finishing a unit last writes y; the weighted combine is a grid of
// its own (a fused one would count arrivals per tile across CTAs, and its
// fences cost more than the launch).
template <int FMT>
__global__ void __launch_bounds__(9 * 32, 2) k_down_t1(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_DOWN_T1);
  constexpr int kBB = FMT == DS4MOE_Q4_K ? kQ4KBytes : kQ2KBytes;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nb = F / 256;
  const T1Tile tl = t1_tile((uint32_t)(kBB * nb));
  const uint32_t stage_bytes = t1_tile_bytes(tl);
  const T1Smem sm = t1_smem(smem, nstage, stage_bytes, nb);
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&sm.full[st], 1);
      ptx::mbar_init(&sm.empty[st], nb);
      sm.cnt[st] = 0;
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int ntile = D / 16;
  // the groups (or the logits) were complete before the gate/up grid
  // launched this one
  __shared__ Group s_grp[kT1MaxGroups];
  __shared__ int s_ngrp;
  if (a.lg) {
    if (w == 0) t1_route_warp(a, s_grp, &s_ngrp, false);
    __syncthreads();
  } else {
    t1_load_groups(a, s_grp, &s_ngrp);
  }
  const int U = s_ngrp * ntile;
  const int u0 = (int)((int64_t)U * blockIdx.x / gridDim.x);
  const int u1 = (int)((int64_t)U * (blockIdx.x + 1) / gridDim.x);
  auto load_group = [&](int u) { return s_grp[u / ntile]; };
  if (w == nb) {
    const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
    for (int u = u0, it = 0; u < u1; ++u, ++it) {
      const int st = it % nstage;
      if (it >= nstage && !ptx::mbar_wait(&sm.empty[st], ((it / nstage) - 1) & 1)) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        break;
      }
      const Group grp = load_group(u);
      const int row0 = (u % ntile) * 16;
      if (lane == 0) ptx::mbar_arrive_expect_tx(&sm.full[st], 16u * tl.rowb);
      __syncwarp();
      if ((uint32_t)lane < t1_copies(tl))
        t1_tile_copy(smem + (size_t)st * stage_bytes, down + ((int64_t)grp.e * D + row0) * tl.rowb, tl, (uint32_t)lane,
                     &sm.full[st]);
    }
    return;
  }
  const T1Lane L = t1_lane(c);
  T1B B;
  ptx::pdl_wait();  // h comes from the gate/up grid
  span_begin(DS4MOE_SPAN_DOWN_T1);
  ptx::pdl_launch_dependents();
  bool timed_out = false;
  int it = 0, cur = -1;
  for (int u = u0; u < u1; ++u, ++it) {
    const int st = it % nstage;
    const Group grp = load_group(u);
    if (grp.p0 != cur) {
      if constexpr (FMT == DS4MOE_Q4_K) t1_load_b_q4k<false>(B, a.h + (int64_t)grp.p0 * F + 256 * w, g, c);
      else t1_load_b<false>(B, a.h + (int64_t)grp.p0 * F + 256 * w, g, c);
      cur = grp.p0;
    }
    if (!timed_out && !ptx::mbar_wait(&sm.full[st], (it / nstage) & 1)) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    float y[1][2] = {{0.f, 0.f}};
    if (!timed_out) {
      const uint8_t *const mats[1] = {smem + (size_t)st * stage_bytes + kBB * w};
      if constexpr (FMT == DS4MOE_Q4_K) t1_block_q4k<1>(mats, tl, g, c, B, y);
      else t1_block<1>(mats, tl, g, B, L, y);
    }
    float *r = sm.red + ((size_t)st * nb + w) * 32;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float v = quad_sum(y[0][q]);
      if (c == 0) r[8 * q + g] = v;
    }
    if (t1_last_arriver(&sm.cnt[st], nb)) {
      const int row0 = (u % ntile) * 16;
      if (lane < 16) {
        const float *rr = sm.red + (size_t)st * nb * 32 + lane;
        float sv = 0.f;
        for (int p = 0; p < nb; ++p) sv += rr[32 * p];
        float *yp = a.y + (int64_t)grp.p0 * D + row0 + lane;
#pragma unroll 1
        for (int j = 0; j < grp.nt; ++j, yp += D) *yp = sv;  // one slot per naming of the expert
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sm.empty[st]);
  }
  if (timed_out && lane == 0) {
    for (int j = it - nstage > 0 ? it - nstage : 0; j < it; ++j)
      ptx::mbar_wait(&sm.full[j % nstage], (j / nstage) & 1, 1u << 20);
  }
}

// Poll budget and target offset of the merged grid's h-ready wait (a
// fault-injection hook for tests: ds4moe_debug_sync_wait).
__device__ int32_t g_sync_budget = 1 << 24;
__device__ int32_t g_sync_extra = 0;

// The single-token expert FFN as one persistent grid (Q2_K gate, up and
// down, d_model = 2 d_ff): one CTA per SM with nbg = d_model / 256 consumer
// warps and one producer.  Every CTA runs its gate/up units first (16 gate +
// 16 up rows of one selected expert, dealt round-robin, exactly as the
// gate/up kernel), then its down items (64 rows of one expert's down matrix,
// dealt in reverse round-robin so that the CTAs holding an extra gate/up
// unit hold fewer down items).  The producer streams both kinds through one
// ring of stages, so the down weights land while gate/up still computes and
// no grid boundary separates the two.  A down item of expert slot j waits
// (bounded) until all d_ff / 16 gate/up units of slot j have published their
// h.  Cross-CTA synchronisation stays off the consumer warps: the warp that
// finishes a gate/up unit only sets the unit's bit in a shared-memory mask,
// and a sync warp per CTA publishes the completed units (one GPU-scope fence
// for every batch, then relaxed adds on hready[]), then waits on hready[] for
// the experts of the CTA's down items and hands them to the consumers
// through a second shared-memory mask.  A GPU-scope fence in the finishing
// consumer warp instead costs it about as much as the unit's arithmetic, and
// every consumer warp polling global counters slows the publishing down.
// The weighted combine is fused the same way: the warp that finishes a down
// item only sets its bit in a third mask; the sync warp counts the item on
// its 64 output rows (ccnt, fence-release / fence-acquire), and if it was
// the last of the k items over those rows, sums w_i y_i in rank order, as
// the combine kernel does.  The sync warp also forms the routing weights
// (and in CTA 0 writes the call's routing outputs), off the producer's path.
// Consumer warp w
// takes K block w % nbd of the down rows and tiles 2 (w / nbd), +1 of the
// item, so both kinds of work run the same two-tile block kernel.  Arithmetic
// and summation order are those of the two separate kernels, so y is
// bit-identical to theirs.
__global__ void __launch_bounds__(18 * 32, 1) k_ffn_t1(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_FFN_T1);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nbg = D / 256, nbd = F / 256;
  const T1Tile tg = t1_tile((uint32_t)(kQ2KBytes * nbg)), td = t1_tile((uint32_t)(kQ2KBytes * nbd));
  const uint32_t tile_g = t1_tile_bytes(tg), tile_d = t1_tile_bytes(td);
  const uint32_t stage_bytes = 2u * tile_g > 4u * tile_d ? 2u * tile_g : 4u * tile_d;
  const T1Smem sm = t1_smem(smem, nstage, stage_bytes, nbg);
  __shared__ uint32_t s_done, s_hok, s_ddone;  // gate/up units finished; experts with h ready; down items finished
  __shared__ float s_lv[kT1MaxGroups], s_w[kT1MaxGroups];  // per slot: selected logit, routing weight
  __shared__ int s_inv[kT1MaxGroups];                      // per slot: position in expert order
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&sm.full[st], 1);
      ptx::mbar_init(&sm.empty[st], nbg);
      sm.cnt[st] = 0;
    }
    s_done = 0u;
    s_hok = 0u;
    s_ddone = 0u;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const T1Lane L = t1_lane(c);
  T1B B;
  if (w < nbg) t1_load_b<true>(B, a.x + 256 * w, g, c);  // the call's input: before the dependency wait
  ptx::pdl_wait();  // the logits come from the router grid
  span_begin(DS4MOE_SPAN_FFN_T1);
  ptx::pdl_launch_dependents();
  __shared__ Group s_grp[kT1MaxGroups];
  __shared__ int s_ngrp;
  if (w == nbg) t1_route_warp(a, s_grp, &s_ngrp, false, s_lv, s_inv);
  __syncthreads();
  const int ntg = F / 16, ntd = D / 64;  // gate/up units and down items per expert
  const int Ug = s_ngrp * ntg, Ud = s_ngrp * ntd, G = gridDim.x;
  const int ng = (int)blockIdx.x < Ug ? (Ug - (int)blockIdx.x + G - 1) / G : 0;
  const int rb = G - 1 - (int)blockIdx.x;
  const int nd = rb < Ud ? (Ud - rb + G - 1) / G : 0;
  const int n = ng + nd;
  if (w == nbg + 1) {
    // sync warp: the routing weights (CTA 0 also writes the routing outputs)
    t1_weights_warp(a, s_grp, s_lv, s_inv, s_w, blockIdx.x == 0);
    // then, interleaved: publish this CTA's gate/up units as they finish, and
    // hand each expert of its down items to the consumers once its h is out
    const uint32_t all = ng >= 32 ? 0xffffffffu : (1u << ng) - 1u;
    const uint32_t dall = nd >= 32 ? 0xffffffffu : (1u << nd) - 1u;
    uint32_t pub = 0, dpub = 0, polls = 0, hpolls = 0;
    const uint32_t hbudget = (uint32_t)g_sync_budget;
    const int32_t htarget = ntg + g_sync_extra;
    int t = 0, prev = -1;
    while (pub != all || t < nd || dpub != dall) {
      bool progress = false;
      uint32_t m = 0;
      if (lane == 0) m = *reinterpret_cast<volatile uint32_t *>(&s_done) & ~pub;
      m = __shfl_sync(0xffffffffu, m, 0);  // one view of the mask for the whole warp
      if (m) {
        if (lane == 0) {
          __threadfence_block();  // the units' h writes, seen through s_done
          ptx::fence_acq_rel_gpu();
          for (uint32_t r = m; r; r &= r - 1u)
            ptx::red_relaxed_add(a.hready + ((int)blockIdx.x + G * (__ffs(r) - 1)) / ntg, 1);
        }
        pub |= m;
        progress = true;
      }
      while (t < nd && (rb + G * t) / ntd == prev) ++t;  // same expert as the previous item
      if (t < nd) {
        const int j = (rb + G * t) / ntd;
        int ready = 0;
        if (lane == 0) {
          ready = ptx::ld_acquire(a.hready + j) >= htarget;
          if (!ready && ++hpolls > hbudget) {
            // the wait ran out: record it, and hand the expert over anyway
            // so that the grid still finishes
            record_status(a.hdr, DS4MOE_ETIMEOUT);
            ready = 1;
          }
        }
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          if (lane == 0) {
            __threadfence_block();
            atomicOr(&s_hok, 1u << j);
            hpolls = 0;
          }
          prev = j;
          ++t;
          progress = true;
        }
      }
      // finished down items: count each on its rows; the last one combines
      uint32_t dm = 0;
      if (lane == 0) dm = *reinterpret_cast<volatile uint32_t *>(&s_ddone) & ~dpub;
      dm = __shfl_sync(0xffffffffu, dm, 0);
      if (dm) {
        if (lane == 0) {
          __threadfence_block();  // the items' y writes, seen through s_ddone
          ptx::fence_acq_rel_gpu();
        }
        for (uint32_t r = dm; r; r &= r - 1u) {
          const int v = rb + G * (__ffs(r) - 1), row0 = (v % ntd) * 64;
          int last = 0;
          if (lane == 0) {
            last = atomicAdd(a.ccnt + row0 / 64, 1) == s_ngrp - 1;
            if (last) ptx::fence_acq_rel_gpu();  // acquires the other items' y
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          __syncwarp();
          if (last) {
            // out rows row0 + lane and row0 + 32 + lane: sum over the k slots in rank order
            float o0 = 0.f, o1 = 0.f;
            for (int i0 = 0; i0 < a.k; i0 += 8) {
              float y0[8], y1[8];
#pragma unroll
              for (int ii = 0; ii < 8; ++ii) {
                const int i = i0 + ii;
                const float *ys = a.y + (int64_t)(i < a.k ? s_inv[i] : 0) * D + row0 + lane;
                y0[ii] = i < a.k ? __ldcg(ys) : 0.f;
                y1[ii] = i < a.k ? __ldcg(ys + 32) : 0.f;
              }
#pragma unroll
              for (int ii = 0; ii < 8; ++ii)
                if (i0 + ii < a.k) {
                  o0 = fmaf(s_w[i0 + ii], y0[ii], o0);
                  o1 = fmaf(s_w[i0 + ii], y1[ii], o1);
                }
            }
            a.out[row0 + lane] = o0;
            a.out[row0 + 32 + lane] = o1;
          }
        }
        dpub |= dm;
        progress = true;
      }
      if (!progress) {
        if (++polls > (1u << 24)) {
          record_status(a.hdr, DS4MOE_ETIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    return;
  }
  if (w == nbg) {
    // producer: one item per stage, gate/up units then down items
    const uint8_t *gate = static_cast<const uint8_t *>(a.L.gate), *up = static_cast<const uint8_t *>(a.L.up);
    const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
    const uint32_t cg = t1_copies(tg), cd = t1_copies(td);
    int st = 0;
    uint32_t ph = 0;
    for (int it = 0; it < n; ++it) {
      if (it >= nstage && !ptx::mbar_wait(&sm.empty[st], ph ^ 1u)) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        break;
      }
      uint8_t *dst = smem + (size_t)st * stage_bytes;
      if (it < ng) {
        const int u = (int)blockIdx.x + G * it;
        const Group grp = s_grp[u / ntg];
        const int row0 = (u % ntg) * 16;
        if (lane == 0) ptx::mbar_arrive_expect_tx(&sm.full[st], 32u * tg.rowb);
        __syncwarp();
        if ((uint32_t)lane < 2u * cg) {
          const uint32_t mat = (uint32_t)lane / cg, i = (uint32_t)lane % cg;
          t1_tile_copy(dst + mat * tile_g, (mat == 0 ? gate : up) + ((int64_t)grp.e * F + row0) * tg.rowb, tg, i,
                       &sm.full[st]);
        }
      } else {
        const int v = rb + G * (it - ng);
        const Group grp = s_grp[v / ntd];
        const int row0 = (v % ntd) * 64;
        if (lane == 0) ptx::mbar_arrive_expect_tx(&sm.full[st], 64u * td.rowb);
        __syncwarp();
        if ((uint32_t)lane < 4u * cd) {
          const uint32_t tile = (uint32_t)lane / cd, i = (uint32_t)lane % cd;
          t1_tile_copy(dst + tile * tile_d, down + ((int64_t)grp.e * D + row0 + 16 * (int)tile) * td.rowb, td, i,
                       &sm.full[st]);
        }
      }
      if (++st == nstage) {
        st = 0;
        ph ^= 1u;
      }
    }
    return;
  }
  bool timed_out = false;
  int st = 0, it = 0, cur = -1;
  uint32_t ph = 0;
  for (; it < n; ++it) {
    const bool gu = it < ng;
    int j, row0;
    if (gu) {
      const int u = (int)blockIdx.x + G * it;
      j = u / ntg;
      row0 = (u % ntg) * 16;
    } else {
      const int v = rb + G * (it - ng);
      j = v / ntd;
      row0 = (v % ntd) * 64;
      if (j != cur) {
        // h of slot j: wait until the sync warp has seen all of it published
        uint32_t polls = 0;
        while (!((*reinterpret_cast<volatile uint32_t *>(&s_hok) >> j) & 1u)) {
          if (++polls > (1u << 24)) {
            record_status(a.hdr, DS4MOE_ETIMEOUT);
            break;
          }
          __nanosleep(32);
        }
        __threadfence_block();  // this lane's h loads after the sync warp's acquire
        t1_load_b<false>(B, a.h + (int64_t)s_grp[j].p0 * F + 256 * (w % nbd), g, c);
        cur = j;
      }
    }
    if (!timed_out && !ptx::mbar_wait(&sm.full[st], ph)) {
      record_status(a.hdr, DS4MOE_ETIMEOUT);
      timed_out = true;
    }
    float y[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (!timed_out) {
      const uint8_t *sb = smem + (size_t)st * stage_bytes;
      if (gu) {
        const uint8_t *const mats[2] = {sb + kQ2KBytes * w, sb + tile_g + kQ2KBytes * w};
        t1_block<2>(mats, tg, g, B, L, y);
      } else {
        const uint8_t *t0 = sb + 2u * (uint32_t)(w / nbd) * tile_d + kQ2KBytes * (w % nbd);
        const uint8_t *const mats[2] = {t0, t0 + tile_d};
        t1_block<2>(mats, td, g, B, L, y);
      }
    }
    // partials: [16 m + 8 q + g] (gate/up: m = gate / up; down: m = tile)
    float *r = sm.red + ((size_t)st * nbg + w) * 32;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float v = quad_sum(y[m][q]);
        if (c == 0) r[16 * m + 8 * q + g] = v;
      }
    if (t1_last_arriver(&sm.cnt[st], nbg)) {
      const Group grp = s_grp[j];
      const float *rr = sm.red + (size_t)st * nbg * 32 + lane;
      if (gu) {
        float sv = 0.f;
        for (int p = 0; p < nbg; ++p) sv += rr[32 * p];
        const float us = __shfl_down_sync(0xffffffffu, sv, 16);
        if (lane < 16) {
          const float hv = bf16_bits_to_f32(f32_to_bf16_bits(silu(sv) * us));
          if (fabsf(hv) > 65504.f) record_status(a.hdr, DS4MOE_EDEVICE);
          uint16_t *hp = a.h + (int64_t)grp.p0 * F + row0 + lane;
          const uint16_t hb = __half_as_ushort(__float2half_rn(hv));
#pragma unroll 1
          for (int jj = 0; jj < grp.nt; ++jj, hp += F) *hp = hb;
        }
        // hand the unit to the sync warp
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicOr(&s_done, 1u << it);
        }
      } else {
        // rows row0 + lane (K blocks of warps 0 .. nbd-1) and row0 + 32 + lane
        float s0 = 0.f, s1 = 0.f;
        for (int p = 0; p < nbd; ++p) {
          s0 += rr[32 * p];
          s1 += rr[32 * (nbd + p)];
        }
        float *yp = a.y + (int64_t)grp.p0 * D + row0 + lane;
#pragma unroll 1
        for (int jj = 0; jj < grp.nt; ++jj, yp += D) {
          yp[0] = s0;
          yp[32] = s1;
        }
        // hand the item to the sync warp (it counts it for the combine)
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          atomicOr(&s_ddone, 1u << (it - ng));
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&sm.empty[st]);
    if (++st == nstage) {
      st = 0;
      ph ^= 1u;
    }
  }
  // no copy may still be landing in shared memory when the CTA exits
  if (timed_out && lane == 0) {
    for (int jj = it - nstage > 0 ? it - nstage : 0; jj < it; ++jj)
      ptx::mbar_wait(&sm.full[jj % nstage], (jj / nstage) & 1, 1u << 20);
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

// Q4_K row: lane items are (block, qs byte); byte 32c + l holds values
// 64c + l (low nibble) and 64c + 32 + l (high nibble).
template <typename In>
__device__ __forceinline__ void row_dot_q4k(const uint8_t *__restrict__ row, int cols, int nt, In in,
                                            float (&acc)[kTok]) {
  const int lane = threadIdx.x & 31;
  const int nitems = cols / 256 * 128;
  for (int it = lane; it < nitems; it += 32) {
    const int b = it >> 7, by = it & 127, c = by >> 5, l = by & 31;
    const uint8_t *p = row + (int64_t)b * kQ4KBytes;
    const float d = f16_bits_to_f32(p[0] | (p[1] << 8));
    const float dmin = f16_bits_to_f32(p[2] | (p[3] << 8));
    const uint32_t q = p[16 + by];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t sc, mn;
      q4k_scale_min(p + 4, 2 * c + hh, sc, mn);
      const int v = 64 * c + 32 * hh + l;
      const float wv = fmaf(d * (float)sc, (float)((q >> (4 * hh)) & 15u), -(dmin * (float)mn));
#pragma unroll
      for (int t = 0; t < kTok; ++t)
        if (t < nt) acc[t] = fmaf(wv, in(t, 256 * b + v), acc[t]);
    }
  }
}

template <typename In>
__device__ __forceinline__ void row_dot(int q, const uint8_t *row, int cols, int nt, In in, float (&acc)[kTok]) {
  if (q == DS4MOE_Q4_1) row_dot_q41(row, cols, nt, in, acc);
  else if (q == DS4MOE_Q2_K) row_dot_q2k(row, cols, nt, in, acc);
  else row_dot_q4k(row, cols, nt, in, acc);
}

// gate/up + SwiGLU, SIMT: one warp per (token group, hidden row).
__global__ void __launch_bounds__(256) k_gate_up_simt(FfnArgs a) {
  const int D = a.L.d_model, F = a.L.d_ff, k = a.k;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t items = (int64_t)a.hdr->n_groups * F;
  const int64_t rbg = row_bytes(a.L.q_gate, D), rbu = row_bytes(a.L.q_up, D);
  if (a.w_logits && gw == 0) finish_routing_weights(const_cast<float *>(a.w), a.T, k);
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
  ptx::pdl_wait();  // y comes from the down grid
  const int D = a.L.d_model, k = a.k;
  const int64_t n4 = (int64_t)a.T * D / 4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = (i * 4) / D;
    const int c = (int)((i * 4) % D);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // eight slots at a time: every (position, weight) load, then every y
    // load, issued before the first use (one round trip each, not k)
    for (int j0 = 0; j0 < k; j0 += 8) {
      int pos[8];
      float wt[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        pos[jj] = j < k ? __ldcg(a.inv + t * k + j) : -1;
        wt[jj] = j < k ? __ldcg(a.w + t * k + j) : 0.f;
      }
      float4 yv[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        yv[jj] = pos[jj] >= 0 ? __ldcg(reinterpret_cast<const float4 *>(a.y + (int64_t)pos[jj] * D + c))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        if (pos[jj] < 0) continue;
        acc.x = fmaf(wt[jj], yv[jj].x, acc.x);
        acc.y = fmaf(wt[jj], yv[jj].y, acc.y);
        acc.z = fmaf(wt[jj], yv[jj].z, acc.z);
        acc.w = fmaf(wt[jj], yv[jj].w, acc.w);
      }
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
  const size_t smem = (size_t)kp * 32 * (chg + chu) + 32 * kp + (size_t)2 * kp * 32 * 4 * sizeof(float);
  // a separate instantiation for the batches whose routing weights are still
  // logits keeps the main loop's code of the other one untouched
  auto kern = a.w_logits ? k_gate_up_mma<QG, QU, true> : k_gate_up_mma<QG, QU, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 2 * kp * 32, smem);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * (per_sm > 0 ? per_sm : 1);
  ProfScope p("gate_up", s);
  return launch_pdl(kern, dim3(grid), dim3(2 * kp * 32), smem, s, a, kp, chg, chu);
}

constexpr size_t kT1SmemGateUp = 227 * 1024, kT1SmemDown = 100 * 1024;

// The persistent multi-token gate/up kernel: gate and up in one format (Q2_K,
// Q4_1 or Q4_K) with
// rows that split into 16-byte bulk copies, d_model <= 4096, two stages fit.
bool gate_up_mt_ok(const ds4moe_layer &L) {
  if (L.q_gate != L.q_up || (L.q_gate != DS4MOE_Q2_K && L.q_gate != DS4MOE_Q4_1 && L.q_gate != DS4MOE_Q4_K))
    return false;
  if (L.d_model % 256 || L.d_model > 256 * kMtMaxK) return false;
  const int64_t rb = row_bytes(L.q_gate, L.d_model);
  if (rb % 16) return false;
  return gate_up_mt_smem(t1_tile_bytes(t1_tile((uint32_t)rb)), L.d_model / 256, 2) <= kT1SmemGateUp;
}

template <int Q>
cudaError_t launch_gate_up_mt(const FfnArgs &a, cudaStream_t s) {
  const int nbk = a.L.d_model / 256;
  const uint32_t tile = t1_tile_bytes(t1_tile((uint32_t)row_bytes(Q, a.L.d_model)));
  int nstage = 6;
  while (nstage > 2 && gate_up_mt_smem(tile, nbk, nstage) > kT1SmemGateUp) --nstage;
  const size_t smem = gate_up_mt_smem(tile, nbk, nstage);
  auto kern = a.w_logits ? k_gate_up_mt<Q, true> : k_gate_up_mt<Q, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p("gate_up", s);
  return launch_pdl(kern, dim3(num_sms()), dim3(32 * (nbk + 2)), smem, s, a, nstage);
}

cudaError_t launch_gate_up_t1(const FfnArgs &a, cudaStream_t s) {
  const int nb = a.L.d_model / 256;
  const bool q4k = a.L.q_gate == DS4MOE_Q4_K;
  const uint32_t stage = 2 * t1_tile_bytes(t1_tile((uint32_t)(block_bytes(a.L.q_gate) * nb)));
  int nstage = 6;
  while (nstage > 2 && t1_smem_bytes(nstage, stage, nb) > kT1SmemGateUp) --nstage;
  const size_t smem = t1_smem_bytes(nstage, stage, nb);
  if (smem > kT1SmemGateUp) return cudaErrorInvalidValue;
  auto kern = q4k ? (a.w_logits ? k_gate_up_t1<true, DS4MOE_Q4_K> : k_gate_up_t1<false, DS4MOE_Q4_K>)
                  : (a.w_logits ? k_gate_up_t1<true, DS4MOE_Q2_K> : k_gate_up_t1<false, DS4MOE_Q2_K>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p("gate_up", s);
  return launch_pdl(kern, dim3(num_sms()), dim3(32 * (nb + 1)), smem, s, a, nstage);
}

// The merged single-token grid: Q2_K gate, up and down with d_model = 2 d_ff
// (<= 4096), d_ff a multiple of 1024, within the single-token chain (the
// grid ranks the experts itself and the router grid zeroes hready).
bool t1_merged_ok(const ds4moe_layer &L, int k) {
  // every CTA tracks its gate/up units and its down items in 32-bit masks
  return L.q_gate == DS4MOE_Q2_K && L.q_up == DS4MOE_Q2_K && L.q_down == DS4MOE_Q2_K && L.d_model == 2 * L.d_ff &&
         L.d_ff % 1024 == 0 && L.d_model <= 4096 && L.n_expert <= 256 &&
         ((int64_t)k * (L.d_ff / 16) + num_sms() - 1) / num_sms() <= 32 &&
         ((int64_t)k * (L.d_model / 64) + num_sms() - 1) / num_sms() <= 32;
}

bool t1_merged_path(const FfnArgs &a) {
  return a.T == 1 && a.lg && a.hready && a.ccnt && t1_merged_ok(a.L, a.k);
}

cudaError_t launch_ffn_t1(const FfnArgs &a, cudaStream_t s) {
  const int nbg = a.L.d_model / 256, nbd = a.L.d_ff / 256;
  const uint32_t tile_g = t1_tile_bytes(t1_tile((uint32_t)(kQ2KBytes * nbg)));
  const uint32_t tile_d = t1_tile_bytes(t1_tile((uint32_t)(kQ2KBytes * nbd)));
  const uint32_t stage = 2 * tile_g > 4 * tile_d ? 2 * tile_g : 4 * tile_d;
  int nstage = 8;
  while (nstage > 2 && t1_smem_bytes(nstage, stage, nbg) > kT1SmemGateUp) --nstage;
  const size_t smem = t1_smem_bytes(nstage, stage, nbg);
  if (smem > kT1SmemGateUp) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_ffn_t1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p("ffn_t1", s);
  return launch_pdl(k_ffn_t1, dim3(num_sms()), dim3(32 * (nbg + 2)), smem, s, a, nstage);
}

cudaError_t launch_down_t1(const FfnArgs &a, cudaStream_t s) {
  const int nb = a.L.d_ff / 256;
  const uint32_t stage = t1_tile_bytes(t1_tile((uint32_t)(block_bytes(a.L.q_down) * nb)));
  int nstage = 8;
  while (nstage > 2 && t1_smem_bytes(nstage, stage, nb) > kT1SmemDown) --nstage;
  const size_t smem = t1_smem_bytes(nstage, stage, nb);
  if (smem > kT1SmemDown) return cudaErrorInvalidValue;
  auto kern = a.L.q_down == DS4MOE_Q4_K ? k_down_t1<DS4MOE_Q4_K> : k_down_t1<DS4MOE_Q2_K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * (nb + 1), smem);
  if (e != cudaSuccess) return e;
  ProfScope p("down", s);
  return launch_pdl(kern, dim3(num_sms() * (per_sm > 0 ? per_sm : 1)), dim3(32 * (nb + 1)), smem, s, a, nstage);
}

// Single-token kernels: Q2_K or Q4_K (gate and up alike), one consumer warp
// per 256-value block of K (at most 16 for gate/up, 8 for down), rows split
// into 16-byte units.
bool t1_gate_up_ok(const ds4moe_layer &L) {
  return (L.q_gate == DS4MOE_Q2_K || L.q_gate == DS4MOE_Q4_K) && L.q_up == L.q_gate && L.d_model % 1024 == 0 &&
         L.d_model <= 4096 && L.d_ff % 16 == 0;
}
bool t1_down_ok(const ds4moe_layer &L) {
  return (L.q_down == DS4MOE_Q2_K || L.q_down == DS4MOE_Q4_K) && L.d_ff % 1024 == 0 && L.d_ff <= 2048 &&
         L.d_model % 16 == 0;
}

// The persistent multi-token down kernel: Q2_K or Q4_K rows that split into
// 16-byte bulk copies, d_ff / 256 dividing its 16 consumer warps, whole
// units of rows.
bool down_mt_ok(const ds4moe_layer &L) {
  if ((L.q_down != DS4MOE_Q2_K && L.q_down != DS4MOE_Q4_K) || L.d_ff % 256) return false;
  const int nbk = L.d_ff / 256;
  if (nbk > kDmtWarps || kDmtWarps % nbk) return false;
  const int64_t rbd = row_bytes(L.q_down, L.d_ff);
  if (rbd % 16 || L.d_model % (16 * kDmtTpw * (kDmtWarps / nbk))) return false;
  return down_mt_smem(t1_tile_bytes(t1_tile((uint32_t)rbd)), kDmtWarps / nbk, 2) <= kT1SmemGateUp;
}

cudaError_t launch_down_mt(const FfnArgs &a, cudaStream_t s) {
  const int tpu = kDmtWarps / (a.L.d_ff / 256);
  const uint32_t tile = t1_tile_bytes(t1_tile((uint32_t)row_bytes(a.L.q_down, a.L.d_ff)));
  int nstage = 8;
  while (nstage > 2 && down_mt_smem(tile, tpu, nstage) > kT1SmemGateUp) --nstage;
  const size_t smem = down_mt_smem(tile, tpu, nstage);
  auto kern = a.L.q_down == DS4MOE_Q4_K ? k_down_mt<DS4MOE_Q4_K> : k_down_mt<DS4MOE_Q2_K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p("down", s);
  return launch_pdl(kern, dim3(num_sms()), dim3(32 * (kDmtWarps + 2)), smem, s, a, nstage);
}

cudaError_t launch_down_mma(const FfnArgs &a, cudaStream_t s) {
  const int F = a.L.d_ff;
  const uint32_t chd = (uint32_t)row_bytes(DS4MOE_Q2_K, F);
  // one stage per warp and as many warps as shared memory allows: every
  // tile of a small batch is in flight at once
  const int nw = 8;
  const size_t smem = (size_t)nw * 16 * chd + 8 * nw;
  auto kern = k_down_mma<1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nw * 32, smem);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * (per_sm > 0 ? per_sm : 1);
  ProfScope p("down", s);
  return launch_pdl(kern, dim3(grid), dim3(nw * 32), smem, s, a, chd);
}

}  // namespace

bool t1_chain_ok(const ds4moe_layer &L) { return t1_gate_up_ok(L) && t1_down_ok(L) && L.n_expert <= 256; }

// Prefill: the experts with few pairs go to the persistent weight-streaming
// kernels (token groups in a.groups, their count in the header), the rest to
// the tensor-core grouped GEMMs; both write h and y by sorted pair.
bool prefill_split_ok(const ds4moe_layer &L) { return gate_up_mt_ok(L) && down_mt_ok(L); }

cudaError_t launch_gate_up_groups(const FfnArgs &a, cudaStream_t s) {
  const int q = a.L.q_gate;
  return q == DS4MOE_Q2_K   ? launch_gate_up_mt<DS4MOE_Q2_K>(a, s)
         : q == DS4MOE_Q4_K ? launch_gate_up_mt<DS4MOE_Q4_K>(a, s)
                            : launch_gate_up_mt<DS4MOE_Q4_1>(a, s);
}

cudaError_t launch_down_groups(const FfnArgs &a, cudaStream_t s) { return launch_down_mt(a, s); }

// The tensor-core kernels need rows that split into 16-byte-multiple bulk
// copies and stages that fit in shared memory; other shapes use SIMT.
bool decode_mma_ok(const ds4moe_layer &L) {
  // the persistent kernels (one-format gate/up of Q2_K / Q4_1 / Q4_K, Q2_K or
  // Q4_K down), or the per-unit ones (Q4_1 / Q2_K gate and up, Q2_K down)
  if (gate_up_mt_ok(L) && down_mt_ok(L)) return true;
  const auto mma_fmt = [](int q) { return q == DS4MOE_Q4_1 || q == DS4MOE_Q2_K; };
  if (!mma_fmt(L.q_gate) || !mma_fmt(L.q_up)) return false;
  if (L.d_model % 16) return false;
  const int kp = pick_kp(L.d_model, L.q_gate, L.q_up);
  if (kp == 0) return false;
  const int64_t st = 16 * (row_bytes(L.q_gate, L.d_model) + row_bytes(L.q_up, L.d_model)) / kp;
  if (2 * st * kp > 200 * 1024) return false;
  const int64_t rbd = row_bytes(L.q_down, L.d_ff);
  return L.q_down == DS4MOE_Q2_K && L.d_ff % 256 == 0 && rbd % 16 == 0 && 8 * 16 * rbd <= 200 * 1024;
}

// Whether this call's down step runs k_down_mt (whose weighted combine is the
// separate combine grid) rather than a kernel with the combine fused.
bool down_mt_runs(const FfnArgs &a) {
  const ds4moe_layer &L = a.L;
  if (t1_merged_path(a)) return false;
  const bool t1g = a.T == 1 && t1_gate_up_ok(L), t1d = a.T == 1 && t1_down_ok(L);
  return (decode_mma_ok(L) || (t1g && t1d)) && !t1d && down_mt_ok(L);
}

cudaError_t launch_ffn_decode(const FfnArgs &a, cudaStream_t s) {
  const ds4moe_layer &L = a.L;
  // single token: the sub-block-column kernels where the format allows;
  // both h producers (single-token and multi-token gate/up) write the fp16
  // operand both down kernels read, so they combine freely
  if (t1_merged_path(a)) return launch_ffn_t1(a, s);
  const bool t1g = a.T == 1 && t1_gate_up_ok(L), t1d = a.T == 1 && t1_down_ok(L);
  if (decode_mma_ok(L) || (t1g && t1d)) {
    const int kp = pick_kp(L.d_model, L.q_gate, L.q_up);
    cudaError_t e;
    if (t1g) e = launch_gate_up_t1(a, s);
    else if (gate_up_mt_ok(L))
      e = L.q_gate == DS4MOE_Q2_K   ? launch_gate_up_mt<DS4MOE_Q2_K>(a, s)
          : L.q_gate == DS4MOE_Q4_K ? launch_gate_up_mt<DS4MOE_Q4_K>(a, s)
                                    : launch_gate_up_mt<DS4MOE_Q4_1>(a, s);
    else if (L.q_gate == DS4MOE_Q2_K && L.q_up == DS4MOE_Q2_K) e = launch_gate_up_mma<DS4MOE_Q2_K, DS4MOE_Q2_K>(a, s, kp);
    else if (L.q_gate == DS4MOE_Q4_1 && L.q_up == DS4MOE_Q4_1) e = launch_gate_up_mma<DS4MOE_Q4_1, DS4MOE_Q4_1>(a, s, kp);
    else if (L.q_gate == DS4MOE_Q2_K) e = launch_gate_up_mma<DS4MOE_Q2_K, DS4MOE_Q4_1>(a, s, kp);
    else e = launch_gate_up_mma<DS4MOE_Q4_1, DS4MOE_Q2_K>(a, s, kp);
    if (e != cudaSuccess) return e;
    if (t1d) return launch_down_t1(a, s);
    return down_mt_runs(a) ? launch_down_mt(a, s) : launch_down_mma(a, s);
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
  if (t1_merged_path(a)) return cudaSuccess;                        // fused into the merged grid
  if (a.cnt && !(a.T == 1 && t1_down_ok(a.L)) && !down_mt_runs(a)) return cudaSuccess;  // fused into the down kernel
  const int64_t n4 = (int64_t)a.T * a.L.d_model / 4;
  const int grid = (int)((n4 + 255) / 256 < num_sms() * 16 ? (n4 + 255) / 256 : num_sms() * 16);
  ProfScope p("combine", s);
  return launch_pdl(k_combine, dim3(grid), dim3(256), 0, s, a);
}

cudaError_t span_control_decode(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4

extern "C" ds4moe_status ds4moe_debug_sync_wait(int32_t budget_polls, int32_t extra_target) {
  if (budget_polls < 1 || extra_target < 0) return DS4MOE_EINVAL;
  cudaError_t e = cudaMemcpyToSymbol(ds4::g_sync_budget, &budget_polls, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(ds4::g_sync_extra, &extra_target, sizeof(int32_t));
  if (e == cudaSuccess) e = ds4::t1r_set_sync_hook(budget_polls, extra_target);
  return e == cudaSuccess ? DS4MOE_OK : DS4MOE_ECUDA;
}
