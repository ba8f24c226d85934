// Expert FFN for prefill chunks (large T): per-expert grouped GEMMs on the
// fifth-generation tensor cores (tcgen05.mma, fp32 accumulators in TMEM).
//
// The pages' expert FFN (DeepSeek-V4-Flash model card, routed experts; the
// Q4_1 / Q2_K block layouts of the ggml quantization notes) is, per expert e
// and its sorted token pairs P_e:
//   H[p] = bf16(silu(Wg_e x_p) * (Wu_e x_p)),   Y[p] = Wd_e H[p].
// Each weight byte is dequantized once per token chunk and multiplied
// against every token of the chunk.  A tcgen05.mma with M = 128 and K = 16
// costs the tensor pipe about the same time for any N up to 256 (measured),
// so the operands are oriented to fill N: gate/up take the chunk's tokens as
// A (M = 128) and 128 gate rows + the same 128 up rows as B (N = 256), one
// MMA producing g and u side by side; down takes 128 weight rows as A and
// the chunk's tokens (up to 256) as B.
//
// One persistent CTA per SM, warp-specialised:
//   warps 0-7   dequantize the staged blocks into fp16 A tiles (K-major,
//               128-byte swizzle, the layout the MMA descriptors name)
//   warps 8-11  epilogue: TMEM -> registers (lane quadrant = warp % 4),
//               SwiGLU + bf16 rounding (gate/up) or fp32 y (down), store
//   warp 12     TMA: quantized weight rows -> shared memory (2-D, u32 boxes)
//   warp 13     TMA: fp16 activations (x gathered by pair, or h) -> B tiles
//   warp 14     TMEM allocation and tcgen05.mma issue (one thread)
// Rings of shared-memory stages hand data between roles on mbarriers; every
// wait is bounded and gives up (status DS4MOE_ETIMEOUT) instead of hanging.
//
// Numerics.  Gate/up are exact up to fp32 accumulation for every format:
// the scaled code (Q4_1: d*q; Q2_K / Q4_K: d*(sc*q), sc*q an exact fp16
// integer) is carried as two fp16 tiles, RN(.) and its exact FMA residual,
// each multiplied against the same x tile; the block minima (Q4_1: m;
// Q2_K / Q4_K: -dmin*mn as a hi/lo pair) enter through extra K-steps against
// the hi and lo fp16 parts of the x block sums (precomputed per pair:
// 32-value blocks, 16-value sub-blocks for Q2_K).  Rounding gate/up weights
// to fp16 instead would perturb g and u by ~2^-12 relative, enough to flip
// the bf16 rounding of a few percent of h.  Down weights are rounded once
// to fp16 (Q2_K / Q4_K: RN(RN(d*sc)*q + RN(-dmin*mn)); Q4_1: RN(d*q + m))
// -- h is final by then, and the effect on y is ~2e-4 relative.
// Activations are exact in fp16 (bf16 values; larger than the fp16 range is
// flagged); products are exact and accumulate in fp32.
//
// Experts with few pairs of a call (at most kSmallPairs) do not come here:
// on layers the persistent multi-token kernels take, they stream their
// weights through those kernels (token groups from k_chunks), which write h
// and y at the same sorted pair rows.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "span.cuh"

namespace ds4 {
namespace {

constexpr int kTileM = 128;   // weight rows per tile (MMA M)
constexpr int kStepK = 64;    // K values per pipeline step: one 128-byte swizzle row of fp16
constexpr int kDqWarps = 8;   // 256 dequant threads: two per tile row
constexpr int kEpiWarp0 = 8;  // epilogue warps 8..11
constexpr int kQWarp = 12, kBWarp = 13, kMmaWarp = 14;
constexpr int kThreads = 15 * 32;
constexpr int kTmemCols = 512;
constexpr int kBRowsPerLoad = 32;  // B tiles arrive in TMA boxes of 32 rows x 64 fp16

// Staged quantized rows: 4 whole blocks of a row per stage.
template <int Q>
struct QFmt;
template <>
struct QFmt<DS4MOE_Q4_1> {
  static constexpr int kVals = 128, kBytes = 80;
};
template <>
struct QFmt<DS4MOE_Q2_K> {
  static constexpr int kVals = 1024, kBytes = 336;
};
template <>
struct QFmt<DS4MOE_Q4_K> {
  static constexpr int kVals = 256, kBytes = 144;
};

// Gate/up K-steps come in groups of kMain main steps of 64 values and one
// extra step for the minima of the group's blocks (the window); the
// prefill layer's d_model is a multiple of kWinVals.
constexpr int kWinSteps = 16, kWinVals = kWinSteps * kStepK;

// Gate/up staging per weight format: kStageSteps K-steps per shared-memory
// stage, kRowBytes bytes per weight row of a stage, kMain main steps per
// minima step, and whether the minima carry a lo part (the block minimum
// is exact in fp16 for Q4_1; for Q2_K / Q4_K dmin * mn is split in two).
//   Q4_1: 4 blocks (80 B) per stage, 2 K-steps.
//   Q4_K: half a super-block per stage: the 16-byte header and 64 code
//         bytes for half 0 (words 0..19 of the block), words 16..35 for
//         half 1 (the header is kept from half 0); 2 K-steps.
//   Q2_K: one super-block per stage, as the 96 bytes from the 16-byte
//         boundary at or below it (a tensor-map box must be a multiple of
//         16 bytes wide; the block starts at byte 4 (sb % 4) of the staged
//         row, and for the row's last block the 96 bytes end at the row's
//         end); 4 K-steps; its 16-value sub-blocks give 32 minima per 8
//         K-steps, so a minima step follows every 8 main steps.
template <int Q>
struct GuFmt;
template <>
struct GuFmt<DS4MOE_Q4_1> {
  static constexpr int kStageSteps = 2, kRowBytes = 80, kMain = 16;
  static constexpr bool kMinLo = false;
};
template <>
struct GuFmt<DS4MOE_Q4_K> {
  static constexpr int kStageSteps = 2, kRowBytes = 80, kMain = 16;
  static constexpr bool kMinLo = true;
};
template <>
struct GuFmt<DS4MOE_Q2_K> {
  static constexpr int kStageSteps = 4, kRowBytes = 96, kMain = 8;
  static constexpr bool kMinLo = true;
};
static_assert(GuFmt<DS4MOE_Q4_1>::kRowBytes == GuFmt<DS4MOE_Q4_K>::kRowBytes, "one tensor-map box for both");

// NMAT = 2: gate and up (exact hi/lo tiles) share each B tile (SwiGLU
// epilogue); NMAT = 1: down.
template <int NMAT, int QA, int BN>
struct TcCfg {
  static constexpr int kSA = NMAT == 2 ? 2 : 4;
  static constexpr int kSB = NMAT == 2 ? 3 : 2;
  static constexpr int kSQ = (NMAT == 2 || QA == DS4MOE_Q2_K) ? 2 : 4;
  static constexpr int kATile = kTileM * kStepK * 2;
  static constexpr int kTiles = NMAT == 2 ? 4 : 1;  // gate hi, up hi, gate lo, up lo
  static constexpr int kASlot = kTiles * kATile;
  static constexpr int kBSlot = BN * kStepK * 2;
  static constexpr int kRowQ = NMAT == 2 ? GuFmt<QA>::kRowBytes : QFmt<QA>::kBytes;
  static constexpr int kQMat = kTileM * kRowQ;
  static constexpr int kQSlot = NMAT * kQMat;
  static constexpr int kNB = kTmemCols / (NMAT * BN);  // TMEM accumulator buffers
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kSA * kASlot;
  static constexpr int kOffQ = kOffB + kSB * kBSlot;
  static constexpr int kOffBar = kOffQ + kSQ * kQSlot;
  static constexpr int kNBars = 2 * (kSQ + kSA + kSB + kNB) + 1;
  static constexpr int kSmem = kOffBar + kNBars * 8 + 16 + 1024;  // + TMEM holder, abort flag, alignment slack
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kOffB % 1024 == 0 && kOffQ % 1024 == 0 && kASlot % 1024 == 0 && kBSlot % 1024 == 0,
                "swizzled tiles start on 1024-byte boundaries");
  static_assert(kNB >= 1, "TMEM holds at least one accumulator set");
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), start address advanced by 32 B per K = 16 slice.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__device__ __forceinline__ uint32_t f16_idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of 16-byte chunk `lc` (K values 8 lc .. 8 lc + 7) of row r in
// a 128 x 64 fp16 tile with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int r, int lc) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((lc ^ (r & 7)) << 4));
}

__device__ __forceinline__ void sts128(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

constexpr uint32_t kMagic1024 = 0x64006400u;

// One Q4_1 block (32 values) of tile row r -> fp16 chunks 4 hb .. 4 hb + 3.
// Value j is the low nibble of qs[j], value j + 16 the high nibble; the code
// enters as the exact fp16 (1024 + q) or (64 + q), minus the base, then
// RN(q * d + m) in one fp16 FMA.
__device__ __forceinline__ bool dq_q41(const uint8_t *blk, uint8_t *tile, int r, int hb) {
  const uint32_t dm = ptx::lds32(blk);
  const uint32_t d2 = __byte_perm(dm, 0, 0x1010), m2 = __byte_perm(dm, 0, 0x3232);
  uint32_t lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = ptx::lds32(blk + 4 + 4 * i);
    const uint32_t p01 = __byte_perm(w, 0, 0x4140), p23 = __byte_perm(w, 0, 0x4342);
    lo[2 * i] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p01, 0x000F000Fu, kMagic1024), kMagic1024), d2, m2);
    lo[2 * i + 1] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p23, 0x000F000Fu, kMagic1024), kMagic1024), d2, m2);
    hi[2 * i] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p01, 0x00F000F0u, 0x54005400u), 0x54005400u), d2, m2);
    hi[2 * i + 1] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p23, 0x00F000F0u, 0x54005400u), 0x54005400u), d2, m2);
  }
  sts128(tile + sw128_off(r, 4 * hb + 0), lo[0], lo[1], lo[2], lo[3]);
  sts128(tile + sw128_off(r, 4 * hb + 1), lo[4], lo[5], lo[6], lo[7]);
  sts128(tile + sw128_off(r, 4 * hb + 2), hi[0], hi[1], hi[2], hi[3]);
  sts128(tile + sw128_off(r, 4 * hb + 3), hi[4], hi[5], hi[6], hi[7]);
  // the largest magnitude is at q = 0 or q = 15
  const float d = f16_bits_to_f32(dm & 0xFFFFu), m = f16_bits_to_f32(dm >> 16);
  return fabsf(m) > 65504.f || fabsf(fmaf(d, 15.f, m)) > 65504.f;
}

// One Q4_1 block of tile row r as two exact fp16 parts: hi = RN(d*q) and
// lo = d*q - hi (an FMA residual, exact barring underflow), written to chunks
// 4 hb .. 4 hb + 3 of the hi and lo tiles.  Returns m (fp16 bits); its
// contribution m * sum(x over the block) is added by the window's extra step.
__device__ __forceinline__ uint32_t dq_q41_exact(const uint8_t *blk, uint8_t *thi, uint8_t *tlo, int r, int hb,
                                                 bool &big) {
  const uint32_t dm = ptx::lds32(blk);
  const uint32_t d2 = __byte_perm(dm, 0, 0x1010);
  uint32_t hi[16], lo[16];  // value pairs (2i, 2i+1) in K order
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = ptx::lds32(blk + 4 + 4 * i);
    const uint32_t p01 = __byte_perm(w, 0, 0x4140), p23 = __byte_perm(w, 0, 0x4342);
    const uint32_t q[4] = {ptx::sub_f16x2(ptx::and_or(p01, 0x000F000Fu, kMagic1024), kMagic1024),
                           ptx::sub_f16x2(ptx::and_or(p23, 0x000F000Fu, kMagic1024), kMagic1024),
                           ptx::sub_f16x2(ptx::and_or(p01, 0x00F000F0u, 0x54005400u), 0x54005400u),
                           ptx::sub_f16x2(ptx::and_or(p23, 0x00F000F0u, 0x54005400u), 0x54005400u)};
    const int pi[4] = {2 * i, 2 * i + 1, 8 + 2 * i, 9 + 2 * i};  // values 4i, 4i+2, 16+4i, 18+4i
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h = ptx::mul_f16x2(q[j], d2);
      hi[pi[j]] = h;
      lo[pi[j]] = ptx::fma_f16x2(q[j], d2, h ^ 0x80008000u);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sts128(thi + sw128_off(r, 4 * hb + c), hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
    sts128(tlo + sw128_off(r, 4 * hb + c), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
  }
  big |= fabsf(f16_bits_to_f32(dm & 0xFFFFu)) * 15.f > 65504.f;
  return dm >> 16;
}

// Half hb of quarter qq of one Q2_K block (values 64 qq + 32 hb .. +31,
// sub-blocks 4 qq + 2 hb and +1) of tile row r -> fp16 chunks 4 hb .. +3.
// Value i's code sits at bits 2s of qs[32 (i / 128) + i % 32], s =
// (i % 128) / 32; masked in place under the fp16 base 1024 / 4^s it reads
// as base + q exactly.
__device__ __forceinline__ bool dq_q2k(const uint8_t *blk, int qq, uint8_t *tile, int r, int hb) {
  const int h = qq >> 1, s = 2 * (qq & 1) + hb;
  const uint32_t scw = ptx::lds32(blk + 4 * qq);
  const uint32_t ddm = ptx::lds32(blk + 80);
  const float d = f16_bits_to_f32(ddm & 0xFFFFu), dmin = f16_bits_to_f32(ddm >> 16);
  uint32_t a2[2], b2[2];
  bool big = false;
#pragma unroll
  for (int sb = 0; sb < 2; ++sb) {
    const uint32_t byte = (scw >> (8 * (2 * hb + sb))) & 0xFFu;
    const float a = d * (float)(byte & 15u), b = -dmin * (float)(byte >> 4);
    big |= fabsf(a) * 3.f > 65504.f || fabsf(b) > 65504.f;
    const uint32_t ah = __half_as_ushort(__float2half_rn(a)), bh = __half_as_ushort(__float2half_rn(b));
    a2[sb] = ah | (ah << 16);
    b2[sb] = bh | (bh << 16);
  }
  const uint32_t mask = (3u << (2 * s)) * 0x00010001u;
  const uint32_t magic = ((uint32_t)(25 - 2 * s) << 10) * 0x00010001u;
  uint32_t v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = ptx::lds32(blk + 16 + 32 * h + 4 * i);
    const uint32_t p01 = __byte_perm(w, 0, 0x4140), p23 = __byte_perm(w, 0, 0x4342);
    const int sb = i >> 2;
    v[2 * i] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p01, mask, magic), magic), a2[sb], b2[sb]);
    v[2 * i + 1] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(p23, mask, magic), magic), a2[sb], b2[sb]);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) sts128(tile + sw128_off(r, 4 * hb + c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  return big;
}

// Duplicate the low / high fp16 of a word into both halves.
__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }
__device__ __forceinline__ uint32_t f16_dup(float v) {
  const uint32_t h = __half_as_ushort(__float2half_rn(v));
  return h | (h << 16);
}

// Q4_K sub-block j's 6-bit scale and min from the 12 scale bytes held in
// three words (bytes 0..3, 4..7, 8..11).
__device__ __forceinline__ void q4k_sm_regs(uint32_t w0, uint32_t w1, uint32_t w2, int j, uint32_t &sc,
                                            uint32_t &mn) {
  const uint32_t bj = ((j < 4 ? w0 : w1) >> (8 * (j & 3))) & 0xFFu;           // byte j
  const uint32_t bj4 = ((j < 4 ? w1 : w2) >> (8 * (j & 3))) & 0xFFu;          // byte j + 4
  const uint32_t bjm4 = (w0 >> (8 * (j & 3))) & 0xFFu;                         // byte j - 4 (j >= 4)
  if (j < 4) {
    sc = bj & 63u;
    mn = bj4 & 63u;
  } else {
    sc = (bj4 & 15u) | ((bjm4 >> 6) << 4);
    mn = (bj4 >> 4) | ((bj >> 6) << 4);
  }
}

// The exact gate/up tiles of 32 values v_i = d sc q_i - dmin mn (Q2_K and
// Q4_K): the integer sc q_i is exact in fp16 (one FMA removes the code
// field's base), hi = RN(d (sc q)) and lo = d (sc q) - hi (an FMA residual,
// exact barring underflow).  The minimum -dmin mn is returned split the
// same way: mh = RN(-dmin mn), ml = -dmin mn - mh.

// Half hb of quarter qq of a Q2_K super-block (values 64 qq + 32 hb .. +31,
// sub-blocks 4 qq + 2 hb and + 1): hi / lo chunks 4 hb .. + 3 of row r,
// and the two sub-blocks' (mh0, mh1) and (ml0, ml1) pairs.
__device__ __forceinline__ void dq_q2k_exact(const uint8_t *blk, int qq, int hb, uint8_t *thi, uint8_t *tlo, int r,
                                             uint32_t &mhp, uint32_t &mlp, bool &big) {
  const int h = qq >> 1, s = 2 * (qq & 1) + hb;
  const uint32_t scw = ptx::lds32(blk + 4 * qq);
  const uint32_t ddm = ptx::lds32(blk + 80);
  const uint32_t d2 = dup_lo(ddm);
  const float d = f16_bits_to_f32(ddm & 0xFFFFu), dmin = f16_bits_to_f32(ddm >> 16);
  const float magic = (float)(1 << (10 - 2 * s));
  uint32_t sc2[2], nms2[2];
  uint32_t mn2 = 0;
#pragma unroll
  for (int sb = 0; sb < 2; ++sb) {
    const uint32_t byte = (scw >> (8 * (2 * hb + sb))) & 0xFFu;
    const float sc = (float)(byte & 15u);
    sc2[sb] = f16_dup(sc);
    nms2[sb] = f16_dup(-magic * sc);
    mn2 |= (uint32_t)__half_as_ushort(__float2half_rn((float)(byte >> 4))) << (16 * sb);
  }
  const uint32_t ndm2 = f16_dup(-dmin);
  mhp = ptx::mul_f16x2(mn2, ndm2);
  mlp = ptx::fma_f16x2(mn2, ndm2, mhp ^ 0x80008000u);
  const uint32_t mask = (3u << (2 * s)) * 0x00010001u;
  const uint32_t base = ((uint32_t)(25 - 2 * s) << 10) * 0x00010001u;
  uint32_t hi[16], lo[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = ptx::lds32(blk + 16 + 32 * h + 4 * i);
    const uint32_t p[2] = {__byte_perm(w, 0, 0x4140), __byte_perm(w, 0, 0x4342)};
    const int sb = i >> 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t scq = ptx::fma_f16x2(ptx::and_or(p[j], mask, base), sc2[sb], nms2[sb]);
      hi[2 * i + j] = ptx::mul_f16x2(scq, d2);
      lo[2 * i + j] = ptx::fma_f16x2(scq, d2, hi[2 * i + j] ^ 0x80008000u);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sts128(thi + sw128_off(r, 4 * hb + c), hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
    sts128(tlo + sw128_off(r, 4 * hb + c), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
  }
  big |= fabsf(d) * 45.f > 65504.f || fabsf(dmin) * 15.f > 65504.f;
}

// Q4_K sub-block j (32 values, nibble hb of the 32 code bytes at qs32) of
// a super-block whose header (d, dmin, 12 scale bytes) is `hd`: hi / lo
// chunks 4 hb .. + 3 of row r; returns mh | ml << 16.
__device__ __forceinline__ uint32_t dq_q4k_exact(const uint8_t *qs32, const uint4 &hd, int j, int hb, uint8_t *thi,
                                                 uint8_t *tlo, int r, bool &big) {
  const uint32_t d2 = dup_lo(hd.x);
  const float d = f16_bits_to_f32(hd.x & 0xFFFFu), dmin = f16_bits_to_f32(hd.x >> 16);
  uint32_t sc, mn;
  q4k_sm_regs(hd.y, hd.z, hd.w, j, sc, mn);
  const float magic = hb ? 64.f : 1024.f;
  const uint32_t sc2 = f16_dup((float)sc), nms2 = f16_dup(-magic * (float)sc);
  const uint32_t mask = hb ? 0x00F000F0u : 0x000F000Fu, base = hb ? 0x54005400u : kMagic1024;
  uint32_t hi[16], lo[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = ptx::lds32(qs32 + 4 * i);
    const uint32_t p[2] = {__byte_perm(w, 0, 0x4140), __byte_perm(w, 0, 0x4342)};
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const uint32_t scq = ptx::fma_f16x2(ptx::and_or(p[jj], mask, base), sc2, nms2);
      hi[2 * i + jj] = ptx::mul_f16x2(scq, d2);
      lo[2 * i + jj] = ptx::fma_f16x2(scq, d2, hi[2 * i + jj] ^ 0x80008000u);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sts128(thi + sw128_off(r, 4 * hb + c), hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
    sts128(tlo + sw128_off(r, 4 * hb + c), lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
  }
  big |= fabsf(d) * 945.f > 65504.f || fabsf(dmin) * 63.f > 65504.f;
  const uint32_t mn2 = f16_dup((float)mn), ndm2 = f16_dup(-dmin);
  const uint32_t mh = ptx::mul_f16x2(mn2, ndm2), ml = ptx::fma_f16x2(mn2, ndm2, mh ^ 0x80008000u);
  return (mh & 0xFFFFu) | (ml << 16);
}

// Q4_K down: K-step kk of the super-block `blk` (144 bytes), sub-block
// 2 kk + hb, rounded once to fp16 as RN(RN(d sc) q + RN(-dmin mn)) into
// chunks 4 hb .. + 3 of row r.  Returns whether a value left the fp16 range.
__device__ __forceinline__ bool dq_q4k(const uint8_t *blk, int kk, uint8_t *tile, int r, int hb) {
  const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
  const float d = f16_bits_to_f32(hd.x & 0xFFFFu), dmin = f16_bits_to_f32(hd.x >> 16);
  uint32_t sc, mn;
  q4k_sm_regs(hd.y, hd.z, hd.w, 2 * kk + hb, sc, mn);
  const float a = d * (float)sc, b = -dmin * (float)mn;
  const uint32_t a2 = f16_dup(a), b2 = f16_dup(b);
  const uint32_t mask = hb ? 0x00F000F0u : 0x000F000Fu, base = hb ? 0x54005400u : kMagic1024;
  uint32_t v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w = ptx::lds32(blk + 16 + 32 * kk + 4 * i);
    v[2 * i] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(__byte_perm(w, 0, 0x4140), mask, base), base), a2, b2);
    v[2 * i + 1] = ptx::fma_f16x2(ptx::sub_f16x2(ptx::and_or(__byte_perm(w, 0, 0x4342), mask, base), base), a2, b2);
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) sts128(tile + sw128_off(r, 4 * hb + c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
  return fabsf(a) * 15.f > 65504.f || fabsf(b) > 65504.f;
}

struct TcArgs {
  const Chunk *chunks;
  const int32_t *nchunks;
  int K;     // reduction length
  int rows;  // weight rows per expert = output features
  void *out; // gate/up: h fp16 [P][rows]; down: y fp32 [P][rows]
  WsHeader *hdr;
};

__device__ __forceinline__ void tc_fail(WsHeader *hdr, volatile int *abort_flag) {
  record_status(hdr, DS4MOE_ETIMEOUT);
  *abort_flag = 1;
}

template <int NMAT, int QA, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_ffn_tc(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
             const __grid_constant__ CUtensorMap mB, TcArgs a) {
  using C = TcCfg<NMAT, QA, BN>;
  constexpr int QV = QFmt<QA>::kVals, QB = QFmt<QA>::kBytes;
  extern __shared__ uint8_t smem_raw[];
  const SpanExit span_exit(NMAT == 2 ? DS4MOE_SPAN_GATE_UP_TC : DS4MOE_SPAN_DOWN_TC);
  span_begin(NMAT == 2 ? DS4MOE_SPAN_GATE_UP_TC : DS4MOE_SPAN_DOWN_TC);
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = sm + C::kOffA, *sB = sm + C::kOffB, *sQ = sm + C::kOffQ;
  uint64_t *qfull = reinterpret_cast<uint64_t *>(sm + C::kOffBar);
  uint64_t *qempty = qfull + C::kSQ, *afull = qempty + C::kSQ, *aempty = afull + C::kSA;
  uint64_t *bfull = aempty + C::kSA, *bempty = bfull + C::kSB, *tfull = bempty + C::kSB, *tempty = tfull + C::kNB;
  uint64_t *drain = tempty + C::kNB;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSQ; ++i) { ptx::mbar_init(&qfull[i], 1); ptx::mbar_init(&qempty[i], kDqWarps); }
    for (int i = 0; i < C::kSA; ++i) { ptx::mbar_init(&afull[i], kDqWarps); ptx::mbar_init(&aempty[i], 1); }
    for (int i = 0; i < C::kSB; ++i) { ptx::mbar_init(&bfull[i], 1); ptx::mbar_init(&bempty[i], 1); }
    for (int i = 0; i < C::kNB; ++i) { ptx::mbar_init(&tfull[i], 1); ptx::mbar_init(&tempty[i], 4); }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int MT = a.rows / kTileM;
  const int nunits = *a.nchunks * MT;
  // gate/up: kMain main steps per minima step (16 for Q4_1 / Q4_K, 8 for Q2_K)
  constexpr int kMain = NMAT == 2 ? GuFmt<QA>::kMain : 1;
  const int nks = a.K / kStepK;                                      // main K-steps
  const int nsteps = NMAT == 2 ? nks + nks / kMain : nks;           // + the minima steps
  // gate/up step s: main step (s / (kMain + 1)) * kMain + s % (kMain + 1),
  // or the minima step of group s / (kMain + 1) when s % (kMain + 1) == kMain
  auto is_min_step = [](int s) { return NMAT == 2 && s % (kMain + 1) == kMain; };

  if (warp < kDqWarps) {
    // ---------------------------------------------------------- dequant
    const int r = (warp * 32 + lane) >> 1, hb = lane & 1;
    int qit = 0, ait = 0;
    bool big = false, ok = true;
    // every lane waits; the warp acts on the unanimous result so that it
    // never diverges around __syncwarp
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(~0u, ptx::mbar_wait_or_abort(bar, parity, abort_flag));
    };
    auto publish = [&](int aslot) {
      ptx::fence_proxy_async();  // generic-proxy tile writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&afull[aslot]);
    };
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
      if constexpr (NMAT == 2) {
        using G = GuFmt<QA>;
        constexpr int kSS = G::kStageSteps;
        for (int grp = 0; grp < nks / kMain && ok; ++grp) {
          // per main step: Q4_1 the block minimum m; Q4_K mh | ml << 16 of its
          // sub-block; Q2_K the (mh0, mh1) and (ml0, ml1) pairs at 2 kk, 2 kk + 1
          uint32_t mg[16], mu[16];
          const uint8_t *qrow = nullptr;
          int qslot = 0;
          uint4 hg = make_uint4(0u, 0u, 0u, 0u), hu = hg;  // Q4_K: the super-block headers
#pragma unroll
          for (int kk = 0; kk < kMain; ++kk) {
            if (!ok) break;
            if (kk % kSS == 0) {
              qslot = qit % C::kSQ;
              if (!wait_all(&qfull[qslot], (qit / C::kSQ) & 1)) { ok = false; break; }
              qrow = sQ + qslot * C::kQSlot + r * G::kRowBytes;
            }
            const int aslot = ait % C::kSA;
            if (!wait_all(&aempty[aslot], ((ait / C::kSA) & 1) ^ 1)) { ok = false; break; }
            uint8_t *tile = sA + aslot * C::kASlot;
            // B tiles of 256 rows: gate rows 0..127 then up rows 128..255, hi then lo
            if constexpr (QA == DS4MOE_Q4_1) {
              const int b = 2 * (kk & 1) + hb;  // a stage (4 blocks) feeds two K-steps
              mg[kk] = dq_q41_exact(qrow + 20 * b, tile, tile + 2 * C::kATile, r, hb, big);
              mu[kk] = dq_q41_exact(qrow + C::kQMat + 20 * b, tile + C::kATile, tile + 3 * C::kATile, r, hb, big);
            } else if constexpr (QA == DS4MOE_Q4_K) {
              const int j = kk & 1, hf = (kk >> 1) & 1;  // step j of super-block half hf
              if ((kk & 3) == 0) {
                hg = *reinterpret_cast<const uint4 *>(qrow);
                hu = *reinterpret_cast<const uint4 *>(qrow + C::kQMat);
              }
              const int sub = 2 * (2 * hf + j) + hb;
              mg[kk] = dq_q4k_exact(qrow + 16 + 32 * j, hg, sub, hb, tile, tile + 2 * C::kATile, r, big);
              mu[kk] = dq_q4k_exact(qrow + C::kQMat + 16 + 32 * j, hu, sub, hb, tile + C::kATile,
                                    tile + 3 * C::kATile, r, big);
            } else {
              const int sb = grp * (kMain / kSS) + kk / kSS;  // super-block of the row
              const int off = 4 * (sb & 3);
              dq_q2k_exact(qrow + off, kk & 3, hb, tile, tile + 2 * C::kATile, r, mg[2 * kk], mg[2 * kk + 1], big);
              dq_q2k_exact(qrow + C::kQMat + off, kk & 3, hb, tile + C::kATile, tile + 3 * C::kATile, r, mu[2 * kk],
                           mu[2 * kk + 1], big);
            }
            publish(aslot);
            ++ait;
            if (kk % kSS == kSS - 1) {
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&qempty[qslot]);
              ++qit;
            }
          }
          if (!ok) break;
          // minima step: its 64 columns pair with the hi and lo parts of the
          // x block sums (32 hb + 2 kk (+1): the 32-value block 2 kk + hb of
          // a Q4_1 / Q4_K window; 32 hb + 4 kk + 2 s (+1): the 16-value
          // sub-block 4 kk + 2 hb + s of a Q2_K group); the hi tiles take m
          // (or mh), the lo tiles ml
          const int aslot = ait % C::kSA;
          if (!wait_all(&aempty[aslot], ((ait / C::kSA) & 1) ^ 1)) { ok = false; break; }
          uint8_t *tile = sA + aslot * C::kASlot;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t gh[4], uh[4], gl[4], ul[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if constexpr (QA == DS4MOE_Q2_K) {
                const int kk = 2 * c + (i >> 1);
                gh[i] = (i & 1) ? dup_hi(mg[2 * kk]) : dup_lo(mg[2 * kk]);
                uh[i] = (i & 1) ? dup_hi(mu[2 * kk]) : dup_lo(mu[2 * kk]);
                gl[i] = (i & 1) ? dup_hi(mg[2 * kk + 1]) : dup_lo(mg[2 * kk + 1]);
                ul[i] = (i & 1) ? dup_hi(mu[2 * kk + 1]) : dup_lo(mu[2 * kk + 1]);
              } else {
                gh[i] = dup_lo(mg[4 * c + i]);
                uh[i] = dup_lo(mu[4 * c + i]);
                gl[i] = dup_hi(mg[4 * c + i]);
                ul[i] = dup_hi(mu[4 * c + i]);
              }
            }
            sts128(tile + sw128_off(r, 4 * hb + c), gh[0], gh[1], gh[2], gh[3]);
            sts128(tile + C::kATile + sw128_off(r, 4 * hb + c), uh[0], uh[1], uh[2], uh[3]);
            if constexpr (G::kMinLo) {
              sts128(tile + 2 * C::kATile + sw128_off(r, 4 * hb + c), gl[0], gl[1], gl[2], gl[3]);
              sts128(tile + 3 * C::kATile + sw128_off(r, 4 * hb + c), ul[0], ul[1], ul[2], ul[3]);
            }
          }
          publish(aslot);
          ++ait;
        }
      } else {
        for (int qs = 0; qs < a.K / QV && ok; ++qs, ++qit) {
          const int qslot = qit % C::kSQ;
          if (!wait_all(&qfull[qslot], (qit / C::kSQ) & 1)) { ok = false; break; }
          const uint8_t *qrow = sQ + qslot * C::kQSlot + r * QB;
          for (int kk = 0; kk < QV / kStepK; ++kk, ++ait) {
            const int aslot = ait % C::kSA;
            if (!wait_all(&aempty[aslot], ((ait / C::kSA) & 1) ^ 1)) { ok = false; break; }
            uint8_t *tile = sA + aslot * C::kASlot;
            if constexpr (QA == DS4MOE_Q4_1)
              big |= dq_q41(qrow + 20 * (2 * kk + hb), tile, r, hb);
            else if constexpr (QA == DS4MOE_Q4_K)
              big |= dq_q4k(qrow, kk, tile, r, hb);
            else
              big |= dq_q2k(qrow + 84 * (kk >> 2), kk & 3, tile, r, hb);
            publish(aslot);
          }
          __syncwarp();
          if (ok && lane == 0) ptx::mbar_arrive(&qempty[qslot]);
        }
      }
    }
    if (!ok) tc_fail(a.hdr, abort_flag);
    if (big) record_status(a.hdr, DS4MOE_EDEVICE);
  } else if (warp < kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue
    const int sub = warp & 3, row = 32 * sub + lane;
    int tit = 0;
    bool big = false;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++tit) {
      const Chunk ch = a.chunks[u / MT];
      const int mt = u % MT, tb = tit % C::kNB;
      if (!__all_sync(~0u, ptx::mbar_wait_or_abort(&tfull[tb], (tit / C::kNB) & 1, abort_flag))) {
        tc_fail(a.hdr, abort_flag);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(32 * sub) << 16) + (uint32_t)(tb * NMAT * BN);
      const int64_t grow = (int64_t)mt * kTileM + row;
      if constexpr (NMAT == 2) {
        // lane = token of the chunk; columns 0..127 = g, 128..255 = u of the
        // tile's 128 rows: 256 contiguous bytes of h per token
        const int tok = row;
        uint4 *H = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + (int64_t)(ch.p0 + tok) * a.rows +
                                             (int64_t)mt * kTileM);
#pragma unroll 1
        for (int c0 = 0; c0 < kTileM; c0 += 32) {
          uint32_t g[32], v[32];
          ptx::tmem_ld32x2_wait(tbase + c0, tbase + kTileM + c0, g, v);
          if (tok < ch.n) {
            uint32_t hp[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float h0 = bf16_bits_to_f32(f32_to_bf16_bits(silu(__uint_as_float(g[j])) * __uint_as_float(v[j])));
              const float h1 =
                  bf16_bits_to_f32(f32_to_bf16_bits(silu(__uint_as_float(g[j + 1])) * __uint_as_float(v[j + 1])));
              big |= !(fabsf(h0) <= 65504.f) || !(fabsf(h1) <= 65504.f);
              hp[j >> 1] = (uint32_t)__half_as_ushort(__float2half_rn(h0)) |
                           ((uint32_t)__half_as_ushort(__float2half_rn(h1)) << 16);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) H[c0 / 8 + q] = make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
          }
        }
      }
      for (int j0 = 0; NMAT == 1 && j0 < ch.n; j0 += 32) {
        {
          uint32_t y[32];
          ptx::tmem_ld32_wait(tbase + j0, y);
          float *Y = static_cast<float *>(a.out);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j0 + j < ch.n) Y[(int64_t)(ch.p0 + j0 + j) * a.rows + grow] = __uint_as_float(y[j]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[tb]);
    }
    if (big) record_status(a.hdr, DS4MOE_EDEVICE);
  } else if (warp == kQWarp) {
    // ------------------------------------------------ weight stages
    constexpr int kSteps = NMAT == 2 ? GuFmt<QA>::kStageSteps : QV / kStepK;  // K-steps per stage
    const int nst = a.K / (kSteps * kStepK);                                   // stages per row
    if (lane == 0) {
      // TMA tiles of 128 rows; x in u32 words: Q4_1 20 per stage; Q4_K
      // 36 per super-block, half 1 from word 16; Q2_K the 24 words from the
      // 16-byte boundary at or below super-block qs (21 qs words in); down:
      // one stage's bytes
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Chunk ch = a.chunks[u / MT];
        const int row0 = ch.e * a.rows + (u % MT) * kTileM;
        for (int qs = 0; qs < nst; ++qs, ++it) {
          const int slot = it % C::kSQ;
          if (!ptx::mbar_wait_or_abort(&qempty[slot], ((it / C::kSQ) & 1) ^ 1, abort_flag)) { ok = false; break; }
          const int x = NMAT == 2 && QA == DS4MOE_Q4_K   ? (qs >> 1) * 36 + (qs & 1) * 16
                        : NMAT == 2 && QA == DS4MOE_Q2_K ? (21 * qs) & ~3
                                                         : qs * (C::kRowQ / 4);
          ptx::mbar_arrive_expect_tx(&qfull[slot], C::kQSlot);
          ptx::tma_load_2d(sQ + slot * C::kQSlot, &mA0, x, row0, &qfull[slot]);
          if constexpr (NMAT == 2) ptx::tma_load_2d(sQ + slot * C::kQSlot + C::kQMat, &mA1, x, row0, &qfull[slot]);
        }
      }
      if (!ok) {
        tc_fail(a.hdr, abort_flag);
        for (int j = it - C::kSQ < 0 ? 0 : it - C::kSQ; j < it; ++j)  // let issued copies land
          ptx::mbar_wait(&qfull[j % C::kSQ], (j / C::kSQ) & 1, 1u << 20);
      }
    }
    __syncwarp();
  } else if (warp == kBWarp) {
    // ------------------------------------------------- TMA: activations
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Chunk ch = a.chunks[u / MT];
        const int nload = (ch.n + kBRowsPerLoad - 1) / kBRowsPerLoad;
        for (int s = 0; s < nsteps; ++s, ++it) {
          const int slot = it % C::kSB;
          // column of the step: main K-steps first in each window, then the
          // window's block sums (stored after the D values of each row)
          const int col = NMAT == 2 ? (is_min_step(s) ? a.K + kStepK * (s / (kMain + 1))
                                                      : kStepK * ((s / (kMain + 1)) * kMain + s % (kMain + 1)))
                                    : kStepK * s;
          if (!ptx::mbar_wait_or_abort(&bempty[slot], ((it / C::kSB) & 1) ^ 1, abort_flag)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&bfull[slot], nload * kBRowsPerLoad * kStepK * 2);
          for (int j = 0; j < nload; ++j)
            ptx::tma_load_2d(sB + slot * C::kBSlot + j * kBRowsPerLoad * kStepK * 2, &mB, col,
                             ch.p0 + j * kBRowsPerLoad, &bfull[slot]);
        }
      }
      if (!ok) {
        tc_fail(a.hdr, abort_flag);
        for (int j = it - C::kSB < 0 ? 0 : it - C::kSB; j < it; ++j)
          ptx::mbar_wait(&bfull[j % C::kSB], (j / C::kSB) & 1, 1u << 20);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issue
    if (lane == 0) {
      int ait = 0, bit = 0, tit = 0;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++tit) {
        const Chunk ch = a.chunks[u / MT];
        const uint32_t idesc = f16_idesc(kTileM, (ch.n + 15) & ~15);
        const uint32_t idesc_gu = f16_idesc(kTileM, 2 * kTileM);  // M = 128 tokens, N = 256 rows
        const int tb = tit % C::kNB;
        if (!ptx::mbar_wait_or_abort(&tempty[tb], ((tit / C::kNB) & 1) ^ 1, abort_flag)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dcol = tmem + (uint32_t)(tb * NMAT * BN);
        for (int s = 0; s < nsteps; ++s, ++ait, ++bit) {
          const int aslot = ait % C::kSA, bslot = bit % C::kSB;
          if (!ptx::mbar_wait_or_abort(&afull[aslot], (ait / C::kSA) & 1, abort_flag) ||
              !ptx::mbar_wait_or_abort(&bfull[bslot], (bit / C::kSB) & 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sA + aslot * C::kASlot), b0 = ptx::smem_u32(sB + bslot * C::kBSlot);
          if constexpr (NMAT == 2) {
            // tokens (the B ring's tile) as A, the 256 weight rows as B
            const bool lo_too = !is_min_step(s) || GuFmt<QA>::kMinLo;
#pragma unroll
            for (int kk = 0; kk < kStepK / 16; ++kk) {
              const uint64_t xd = sw128_desc(b0 + 32 * kk);
              ptx::umma_f16(dcol, xd, sw128_desc(a0 + 32 * kk), idesc_gu, (s | kk) != 0);
              if (lo_too) ptx::umma_f16(dcol, xd, sw128_desc(a0 + 2 * C::kATile + 32 * kk), idesc_gu, 1);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kStepK / 16; ++kk)
              ptx::umma_f16(dcol, sw128_desc(a0 + 32 * kk), sw128_desc(b0 + 32 * kk), idesc, (s | kk) != 0);
          }
          issued = true;
          ptx::umma_commit(&aempty[aslot]);
          ptx::umma_commit(&bempty[bslot]);
        }
        if (ok) ptx::umma_commit(&tfull[tb]);
      }
      if (!ok) {
        tc_fail(a.hdr, abort_flag);
        if (issued) {  // let the issued MMAs finish before TMEM is freed
          ptx::umma_commit(drain);
          ptx::mbar_wait(drain, 0, 1u << 20);
        }
      }
    }
    __syncwarp();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// x of every sorted pair as fp16 (exact for bf16 values within the fp16
// range; larger magnitudes are flagged), row stride ld.  After the D values
// each row carries the hi and lo fp16 parts of its block sums, in the order
// the gate/up minima steps read them:
//   sums = 1 (Q4_1 / Q4_K): 32-value block b at
//            D + 64 (b / 32) + 32 (b % 2) + 2 ((b % 32) / 2) (+1 for lo);
//   sums = 2 (Q2_K): 16-value sub-block g at
//            D + 64 (g / 32) + 32 ((g % 4) / 2) + 4 ((g % 32) / 4) + 2 (g % 2) (+1).
__global__ void k_xperm(const uint16_t *__restrict__ x, const int32_t *__restrict__ perm,
                        const int32_t *__restrict__ offs, int E, int k, int D, int ld, int sums,
                        uint16_t *__restrict__ xp, WsHeader *__restrict__ hdr) {
  const int nv = offs[E];
  const int nb = D / 32;
  bool big = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)nv * nb;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / nb;
    const int b = (int)(i % nb);
    const int t = perm[p] / k;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * D + 32 * b);
    uint4 *dst = reinterpret_cast<uint4 *>(xp + p * ld + 32 * b);
    float hsum[2] = {0.f, 0.f};  // values 0..15 and 16..31 of the block
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 q = __ldg(src + v);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = bf16_bits_to_f32(wd[j] & 0xFFFFu), hi = bf16_bits_to_f32(wd[j] >> 16);
        big |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
        hsum[v >> 1] += lo + hi;
        o[j] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    auto put = [&](float sum, int64_t col) {
      const __half sh = __float2half_rn(sum);
      const __half sl = __float2half_rn(sum - __half2float(sh));
      big |= !(fabsf(sum) <= 65504.f);
      *reinterpret_cast<uint32_t *>(xp + p * ld + col) =
          (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(sl) << 16);
    };
    if (sums == 1) {
      put(hsum[0] + hsum[1], D + 64 * (b >> 5) + 32 * (b & 1) + 2 * ((b & 31) >> 1));
    } else if (sums == 2) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int g = 2 * b + hh;
        put(hsum[hh], D + 64 * (g >> 5) + 32 * ((g & 3) >> 1) + 4 * ((g & 31) >> 2) + 2 * (g & 1));
      }
    }
  }
  if (big) record_status(hdr, DS4MOE_EDEVICE);
}

// Token chunks per expert for both tensor-core kernels (one CTA, E <= 1024
// threads).  With `small` > 0, an expert with 1 .. small pairs gets token
// groups of <= kGroup pairs for the weight-streaming kernels instead, in
// expert order, their count in hdr->n_groups.
__global__ void __launch_bounds__(1024) k_chunks(const int32_t *__restrict__ offs, int E, Chunk *__restrict__ cgu,
                                                 Chunk *__restrict__ cdn, int32_t *__restrict__ nchunks, int small,
                                                 Group *__restrict__ groups, WsHeader *__restrict__ hdr) {
  __shared__ int s1[1024], s2[1024], s3[1024];
  const int e = threadIdx.x;
  const int n = e < E ? offs[e + 1] - offs[e] : 0;
  const bool grouped = n <= small;
  const int a1 = grouped ? 0 : (n + kChunkGateUp - 1) / kChunkGateUp;
  const int a2 = grouped ? 0 : (n + kChunkDown - 1) / kChunkDown;
  const int a3 = grouped ? (n + kGroup - 1) / kGroup : 0;
  s1[e] = a1;
  s2[e] = a2;
  s3[e] = a3;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v1 = e >= o ? s1[e - o] : 0, v2 = e >= o ? s2[e - o] : 0, v3 = e >= o ? s3[e - o] : 0;
    __syncthreads();
    s1[e] += v1;
    s2[e] += v2;
    s3[e] += v3;
    __syncthreads();
  }
  if (e < E) {
    const int p0 = offs[e];
    for (int j = 0, b = s1[e] - a1; j < a1; ++j, ++b)
      cgu[b] = Chunk{e, p0 + j * kChunkGateUp, min(kChunkGateUp, n - j * kChunkGateUp), 0};
    for (int j = 0, b = s2[e] - a2; j < a2; ++j, ++b)
      cdn[b] = Chunk{e, p0 + j * kChunkDown, min(kChunkDown, n - j * kChunkDown), 0};
    for (int j = 0, b = s3[e] - a3; j < a3; ++j, ++b)
      groups[b] = Group{e, p0 + j * kGroup, min(kGroup, n - j * kGroup), 0};
  }
  if (e == 1023) {
    nchunks[0] = s1[1023];
    nchunks[1] = s2[1023];
    if (small > 0) hdr->n_groups = s3[1023];
  }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Weight blocks of all experts as a 2-D u32 array [E * rows][row_bytes / 4];
// boxes of one stage (qbytes / 4 words) x 128 rows, no swizzle.
bool map_weights(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t nrows, int qbytes) {
  const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)nrows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(qbytes / 4), (cuuint32_t)kTileM};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// fp16 activations [rows][cols]; boxes of 64 values x 32 rows, 128-byte swizzle.
bool map_acts(CUtensorMap *m, const void *base, int64_t cols, int64_t nrows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)nrows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kStepK, (cuuint32_t)kBRowsPerLoad};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAT, int QA, int BN>
cudaError_t launch_tc(const CUtensorMap &mA0, const CUtensorMap &mA1, const CUtensorMap &mB, const TcArgs &ta,
                      int max_units, cudaStream_t s, const char *name) {
  using C = TcCfg<NMAT, QA, BN>;
  auto kern = k_ffn_tc<NMAT, QA, BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = max_units < num_sms() ? (max_units > 0 ? max_units : 1) : num_sms();
  ProfScope p(name, s);
  kern<<<grid, kThreads, C::kSmem, s>>>(mA0, mA1, mB, ta);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_ok(const ds4moe_layer &L) {
  const int D = L.d_model, F = L.d_ff;
  if (L.q_gate != L.q_up) return false;
  if (L.q_gate != DS4MOE_Q4_1 && L.q_gate != DS4MOE_Q4_K && L.q_gate != DS4MOE_Q2_K) return false;
  if (L.q_down == DS4MOE_Q2_K) {
    if (F % QFmt<DS4MOE_Q2_K>::kVals) return false;
  } else if (L.q_down == DS4MOE_Q4_1) {
    if (F % QFmt<DS4MOE_Q4_1>::kVals) return false;
  } else if (L.q_down == DS4MOE_Q4_K) {
    if (F % QFmt<DS4MOE_Q4_K>::kVals) return false;
  } else {
    return false;
  }
  if (D % kWinVals || D % kTileM || F % kTileM) return false;
  if (!encode_fn()) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  return major == 10;
}

cudaError_t launch_ffn_prefill(const FfnArgs &a, cudaStream_t s) {
  const ds4moe_layer &L = a.L;
  if (!a.xp || !prefill_tc_ok(L)) return launch_ffn_decode(a, s);
  const int D = L.d_model, F = L.d_ff, E = L.n_expert, P = a.T * a.k;
  cudaError_t e;
  {
    ProfScope p("xperm", s);
    const int64_t work = (int64_t)P * (D / 32);
    const int grid = (int)((work + 255) / 256 < num_sms() * 8 ? (work + 255) / 256 : num_sms() * 8);
    k_xperm<<<grid, 256, 0, s>>>(a.x, a.perm, a.offs, E, a.k, D, xp_cols(D), L.q_gate == DS4MOE_Q2_K ? 2 : 1,
                                 a.xp, a.hdr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // experts with few pairs: the weight-streaming kernels (x as fp16 with its
  // sums for them was converted before this call)
  const bool split = a.x16 && a.xs16 && a.xs32 && prefill_split_ok(L);
  {
    ProfScope p("chunks", s);
    k_chunks<<<1, 1024, 0, s>>>(a.offs, E, a.chunks_gu, a.chunks_dn, a.nchunks, split ? kSmallPairs : 0,
                                const_cast<Group *>(a.groups), a.hdr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap mg, mu, md, mx, mh;
  if (!map_acts(&mx, a.xp, xp_cols(D), P) || !map_acts(&mh, a.h, F, P)) return cudaErrorInvalidValue;
  const int qg = L.q_gate, qd = L.q_down;
  const int gbytes = qg == DS4MOE_Q2_K ? GuFmt<DS4MOE_Q2_K>::kRowBytes : GuFmt<DS4MOE_Q4_1>::kRowBytes;
  if (!map_weights(&mg, L.gate, row_bytes(qg, D), (int64_t)E * F, gbytes) ||
      !map_weights(&mu, L.up, row_bytes(qg, D), (int64_t)E * F, gbytes))
    return cudaErrorInvalidValue;
  const int dbytes = qd == DS4MOE_Q2_K ? QFmt<DS4MOE_Q2_K>::kBytes
                     : qd == DS4MOE_Q4_K ? QFmt<DS4MOE_Q4_K>::kBytes
                                         : QFmt<DS4MOE_Q4_1>::kBytes;
  if (!map_weights(&md, L.down, row_bytes(qd, F), (int64_t)E * D, dbytes)) return cudaErrorInvalidValue;
  const int ne = E < P ? E : P;
  TcArgs gu{a.chunks_gu, a.nchunks, D, F, a.h, a.hdr};
  const int gu_units = (ne + P / kChunkGateUp) * (F / kTileM);
  e = qg == DS4MOE_Q2_K   ? launch_tc<2, DS4MOE_Q2_K, kChunkGateUp>(mg, mu, mx, gu, gu_units, s, "gate_up_tc")
      : qg == DS4MOE_Q4_K ? launch_tc<2, DS4MOE_Q4_K, kChunkGateUp>(mg, mu, mx, gu, gu_units, s, "gate_up_tc")
                          : launch_tc<2, DS4MOE_Q4_1, kChunkGateUp>(mg, mu, mx, gu, gu_units, s, "gate_up_tc");
  if (e != cudaSuccess) return e;
  if (split && (e = launch_gate_up_groups(a, s)) != cudaSuccess) return e;
  TcArgs dn{a.chunks_dn, a.nchunks + 1, F, D, a.y, a.hdr};
  const int dn_units = (ne + P / kChunkDown) * (D / kTileM);
  e = qd == DS4MOE_Q2_K   ? launch_tc<1, DS4MOE_Q2_K, kChunkDown>(md, md, mh, dn, dn_units, s, "down_tc")
      : qd == DS4MOE_Q4_K ? launch_tc<1, DS4MOE_Q4_K, kChunkDown>(md, md, mh, dn, dn_units, s, "down_tc")
                          : launch_tc<1, DS4MOE_Q4_1, kChunkDown>(md, md, mh, dn, dn_units, s, "down_tc");
  if (e != cudaSuccess) return e;
  return split ? launch_down_groups(a, s) : cudaSuccess;
}

cudaError_t span_control_prefill(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4
