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
// Numerics.  Gate/up (Q4_1) are exact up to fp32 accumulation: d*q is
// carried as two fp16 tiles, RN(d*q) and the exact FMA residual
// d*q - RN(d*q), each multiplied against the same x tile; the block minima
// enter through extra K-steps that multiply m against the hi and lo fp16
// parts of the 32-value block sums of x (precomputed per pair).  Rounding
// gate/up weights to fp16 instead would perturb g and u by ~2^-12 relative,
// enough to flip the bf16 rounding of a few percent of h.  Down weights are
// rounded once to fp16 (Q2_K: RN(RN(d*sc)*q + RN(-dmin*mn)); Q4_1:
// RN(d*q + m)) -- h is final by then, and the effect on y is ~2e-4
// relative.  Activations are exact in fp16 (bf16 values; larger than the
// fp16 range is flagged); products are exact and accumulate in fp32.
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

// Gate/up K-steps come in windows of 16 x 64 values (32 Q4_1 blocks) and
// one extra step for the block minima of the window.
constexpr int kWinSteps = 16, kWinVals = kWinSteps * kStepK;

// NMAT = 2: gate and up (Q4_1, exact hi/lo tiles) share each B tile
// (SwiGLU epilogue); NMAT = 1: down.
template <int NMAT, int QA, int BN>
struct TcCfg {
  static_assert(NMAT == 1 || QA == DS4MOE_Q4_1, "exact gate/up tiles are built from Q4_1 blocks");
  static constexpr int kSA = NMAT == 2 ? 2 : 4;
  static constexpr int kSB = NMAT == 2 ? 3 : 2;
  static constexpr int kSQ = QA == DS4MOE_Q2_K ? 2 : (NMAT == 2 ? 2 : 4);
  static constexpr int kATile = kTileM * kStepK * 2;
  static constexpr int kTiles = NMAT == 2 ? 4 : 1;  // gate hi, up hi, gate -lo, up -lo
  static constexpr int kASlot = kTiles * kATile;
  static constexpr int kBSlot = BN * kStepK * 2;
  static constexpr int kQMat = kTileM * QFmt<QA>::kBytes;
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
  const int nks = a.K / kStepK;                                      // main K-steps
  const int nsteps = NMAT == 2 ? nks + nks / kWinSteps : nks;       // + one minima step per window
  // gate/up step s: main step (s / 17) * 16 + s % 17, or the minima step of
  // window s / 17 when s % 17 == 16
  auto is_min_step = [](int s) { return NMAT == 2 && s % (kWinSteps + 1) == kWinSteps; };

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
        for (int win = 0; win < a.K / kWinVals && ok; ++win) {
          uint32_t mg[kWinSteps], mu[kWinSteps];
          const uint8_t *qrow = nullptr;
          int qslot = 0;
#pragma unroll
          for (int kk = 0; kk < kWinSteps; ++kk) {
            if (!ok) break;
            if ((kk & 1) == 0) {  // a Q4_1 stage (4 blocks) feeds two K-steps
              qslot = qit % C::kSQ;
              if (!wait_all(&qfull[qslot], (qit / C::kSQ) & 1)) { ok = false; break; }
              qrow = sQ + qslot * C::kQSlot + r * QB;
            }
            const int aslot = ait % C::kSA;
            if (!wait_all(&aempty[aslot], ((ait / C::kSA) & 1) ^ 1)) { ok = false; break; }
            uint8_t *tile = sA + aslot * C::kASlot;
            const int b = 2 * (kk & 1) + hb;
            // B tiles of 256 rows: gate rows 0..127 then up rows 128..255, hi then lo
            mg[kk] = dq_q41_exact(qrow + 20 * b, tile, tile + 2 * C::kATile, r, hb, big);
            mu[kk] = dq_q41_exact(qrow + C::kQMat + 20 * b, tile + C::kATile, tile + 3 * C::kATile, r, hb, big);
            publish(aslot);
            ++ait;
            if (kk & 1) {
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&qempty[qslot]);
              ++qit;
            }
          }
          if (!ok) break;
          // minima step: column 32 hb + 2 kk (+1) of the window's extra K-step
          // holds m of block 2 kk + hb, against the hi (lo) part of its x sum
          const int aslot = ait % C::kSA;
          if (!wait_all(&aempty[aslot], ((ait / C::kSA) & 1) ^ 1)) { ok = false; break; }
          uint8_t *tile = sA + aslot * C::kASlot;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t g4[4], u4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              g4[i] = mg[4 * c + i] | (mg[4 * c + i] << 16);
              u4[i] = mu[4 * c + i] | (mu[4 * c + i] << 16);
            }
            sts128(tile + sw128_off(r, 4 * hb + c), g4[0], g4[1], g4[2], g4[3]);
            sts128(tile + C::kATile + sw128_off(r, 4 * hb + c), u4[0], u4[1], u4[2], u4[3]);
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
    // ------------------------------------------------ TMA: weight blocks
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const Chunk ch = a.chunks[u / MT];
        const int row0 = ch.e * a.rows + (u % MT) * kTileM;
        for (int qs = 0; qs < a.K / QV; ++qs, ++it) {
          const int slot = it % C::kSQ;
          if (!ptx::mbar_wait_or_abort(&qempty[slot], ((it / C::kSQ) & 1) ^ 1, abort_flag)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&qfull[slot], C::kQSlot);
          ptx::tma_load_2d(sQ + slot * C::kQSlot, &mA0, qs * (QB / 4), row0, &qfull[slot]);
          if constexpr (NMAT == 2) ptx::tma_load_2d(sQ + slot * C::kQSlot + C::kQMat, &mA1, qs * (QB / 4), row0, &qfull[slot]);
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
          const int col = NMAT == 2 ? (is_min_step(s) ? a.K + kStepK * (s / (kWinSteps + 1))
                                                      : kStepK * ((s / (kWinSteps + 1)) * kWinSteps + s % (kWinSteps + 1)))
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
            const bool lo_too = !is_min_step(s);
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
// range; larger magnitudes are flagged), row stride ld.  With `sums`, each
// row also carries the hi and lo fp16 parts of its 32-value block sums after
// the D values, in the order the gate/up minima steps read them: block b at
// D + 64 (b / 32) + 32 (b % 2) + 2 ((b % 32) / 2) (+1 for lo).
__global__ void k_xperm(const uint16_t *__restrict__ x, const int32_t *__restrict__ perm,
                        const int32_t *__restrict__ offs, int E, int k, int D, int ld, bool sums,
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
    float sum = 0.f;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 q = __ldg(src + v);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = bf16_bits_to_f32(wd[j] & 0xFFFFu), hi = bf16_bits_to_f32(wd[j] >> 16);
        big |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
        sum += lo + hi;
        o[j] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (sums) {
      const __half sh = __float2half_rn(sum);
      const __half sl = __float2half_rn(sum - __half2float(sh));
      big |= !(fabsf(sum) <= 65504.f);
      const int64_t col = D + 64 * (b >> 5) + 32 * (b & 1) + 2 * ((b & 31) >> 1);
      *reinterpret_cast<uint32_t *>(xp + p * ld + col) =
          (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(sl) << 16);
    }
  }
  if (big) record_status(hdr, DS4MOE_EDEVICE);
}

// Token chunks per expert for both kernels (one CTA, E <= 1024 threads).
__global__ void __launch_bounds__(1024) k_chunks(const int32_t *__restrict__ offs, int E, Chunk *__restrict__ cgu,
                                                 Chunk *__restrict__ cdn, int32_t *__restrict__ nchunks) {
  __shared__ int s1[1024], s2[1024];
  const int e = threadIdx.x;
  const int n = e < E ? offs[e + 1] - offs[e] : 0;
  const int a1 = (n + kChunkGateUp - 1) / kChunkGateUp, a2 = (n + kChunkDown - 1) / kChunkDown;
  s1[e] = a1;
  s2[e] = a2;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v1 = e >= o ? s1[e - o] : 0, v2 = e >= o ? s2[e - o] : 0;
    __syncthreads();
    s1[e] += v1;
    s2[e] += v2;
    __syncthreads();
  }
  if (e < E) {
    const int p0 = offs[e];
    for (int j = 0, b = s1[e] - a1; j < a1; ++j, ++b)
      cgu[b] = Chunk{e, p0 + j * kChunkGateUp, min(kChunkGateUp, n - j * kChunkGateUp), 0};
    for (int j = 0, b = s2[e] - a2; j < a2; ++j, ++b)
      cdn[b] = Chunk{e, p0 + j * kChunkDown, min(kChunkDown, n - j * kChunkDown), 0};
  }
  if (e == 1023) {
    nchunks[0] = s1[1023];
    nchunks[1] = s2[1023];
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
  if (L.q_gate != DS4MOE_Q4_1 || L.q_up != DS4MOE_Q4_1) return false;
  if (L.q_down == DS4MOE_Q2_K) {
    if (F % QFmt<DS4MOE_Q2_K>::kVals) return false;
  } else if (L.q_down == DS4MOE_Q4_1) {
    if (F % QFmt<DS4MOE_Q4_1>::kVals) return false;
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
    k_xperm<<<grid, 256, 0, s>>>(a.x, a.perm, a.offs, E, a.k, D, xp_cols(D), true, a.xp, a.hdr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope p("chunks", s);
    k_chunks<<<1, 1024, 0, s>>>(a.offs, E, a.chunks_gu, a.chunks_dn, a.nchunks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  CUtensorMap mg, mu, md, mx, mh;
  if (!map_weights(&mg, L.gate, row_bytes(L.q_gate, D), (int64_t)E * F, QFmt<DS4MOE_Q4_1>::kBytes) ||
      !map_weights(&mu, L.up, row_bytes(L.q_up, D), (int64_t)E * F, QFmt<DS4MOE_Q4_1>::kBytes) ||
      !map_acts(&mx, a.xp, xp_cols(D), P) || !map_acts(&mh, a.h, F, P))
    return cudaErrorInvalidValue;
  const bool dq2 = L.q_down == DS4MOE_Q2_K;
  if (!map_weights(&md, L.down, row_bytes(L.q_down, F), (int64_t)E * D,
                   dq2 ? QFmt<DS4MOE_Q2_K>::kBytes : QFmt<DS4MOE_Q4_1>::kBytes))
    return cudaErrorInvalidValue;
  const int ne = E < P ? E : P;
  TcArgs gu{a.chunks_gu, a.nchunks, D, F, a.h, a.hdr};
  e = launch_tc<2, DS4MOE_Q4_1, kChunkGateUp>(mg, mu, mx, gu, (ne + P / kChunkGateUp) * (F / kTileM), s,
                                              "gate_up_tc");
  if (e != cudaSuccess) return e;
  TcArgs dn{a.chunks_dn, a.nchunks + 1, F, D, a.y, a.hdr};
  const int dn_units = (ne + P / kChunkDown) * (D / kTileM);
  if (dq2) return launch_tc<1, DS4MOE_Q2_K, kChunkDown>(md, md, mh, dn, dn_units, s, "down_tc");
  return launch_tc<1, DS4MOE_Q4_1, kChunkDown>(md, md, mh, dn, dn_units, s, "down_tc");
}

cudaError_t span_control_prefill(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4
