// The shared expert: an unquantised (bf16) SwiGLU FFN that runs for every
// token and is added to the routed combine with weight one.  "【#2】ds4.c
// 해독하기" (summary bullets and the README's Model Weights bullets) keeps it,
// like the projections and the routing, out of the 2-bit recipe: only the
// routed experts are quantised.  Per token t:
//   h[t] = bf16(silu(w1 x[t]) * (w3 x[t])),  out[t] (+)= w2 h[t]
// with w1, w3 [Fs x D] and w2 [D x Fs] bf16, row-major; fp32 accumulation
// over the exact bf16 products.
//
// Two paths:
//  - up to kSimtTokens (8) tokens: bandwidth-bound GEMVs on the CUDA cores, one
//    warp per hidden unit (gate/up) or output row (down), 16-byte loads
//    along the row, tokens in groups of eight, a fixed-order warp reduction;
//  - more tokens: persistent tcgen05 GEMMs.  A = 128 tokens x 64 K of the
//    activations (x or h), B = 256 weight rows x 64 K (gate/up: 128 rows of
//    w1 then the same 128 rows of w3; down: 256 rows of w2), both brought by
//    TMA in the 128-byte-swizzled K-major layout, bf16 x bf16 -> fp32 in
//    TMEM (two 256-column accumulators), epilogue: SwiGLU to bf16 h, or the
//    fp32 output (added to out when accumulating).
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "span.cuh"

namespace ds4 {
namespace {

constexpr int kSimtTokens = 8;   // at most this many tokens take the GEMV path
constexpr int kGT = 8;           // tokens per group in the GEMV kernels
constexpr int kGemvWarps = 4;    // warps (rows) per CTA of the GEMV kernels

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ GEMV path
// One warp per hidden unit f: g = w1[f] . x[t], u = w3[f] . x[t] for every
// token, h[t][f] = bf16(silu(g) * u).
__global__ void __launch_bounds__(32 * kGemvWarps) k_shared_gu_simt(const uint16_t *__restrict__ w1,
                                                        const uint16_t *__restrict__ w3,
                                                        const uint16_t *__restrict__ x, int D, int Fs, int T,
                                                        uint16_t *__restrict__ h) {
  const int lane = threadIdx.x & 31;
  const int f = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
  if (f >= Fs) return;
  const uint4 *r1 = reinterpret_cast<const uint4 *>(w1 + (int64_t)f * D);
  const uint4 *r3 = reinterpret_cast<const uint4 *>(w3 + (int64_t)f * D);
  const int nc = D / 8;
  for (int t0 = 0; t0 < T; t0 += kGT) {
    const int nt = T - t0 < kGT ? T - t0 : kGT;
    float g[kGT], u[kGT];
#pragma unroll
    for (int t = 0; t < kGT; ++t) g[t] = u[t] = 0.f;
#pragma unroll 4
    for (int c = lane; c < nc; c += 32) {
      float a[8], b[8];
      bf16x8_to_f32(__ldg(r1 + c), a);
      bf16x8_to_f32(__ldg(r3 + c), b);
#pragma unroll
      for (int t = 0; t < kGT; ++t)
        if (t < nt) {
          float xv[8];
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(x + (int64_t)(t0 + t) * D) + c), xv);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            g[t] = fmaf(a[j], xv[j], g[t]);
            u[t] = fmaf(b[j], xv[j], u[t]);
          }
        }
    }
    float mine = 0.f;
#pragma unroll
    for (int t = 0; t < kGT; ++t)
      if (t < nt) {
        const float gs = warp_sum(g[t]), us = warp_sum(u[t]);
        if (lane == t) mine = silu(gs) * us;
      }
    if (lane < nt) h[(int64_t)(t0 + lane) * Fs + f] = f32_to_bf16_bits(mine);
  }
}

// One warp per output row d: y = w2[d] . h[t]; out[t][d] = y or out + y.
__global__ void __launch_bounds__(32 * kGemvWarps) k_shared_down_simt(const uint16_t *__restrict__ w2,
                                                          const uint16_t *__restrict__ h, int D, int Fs, int T,
                                                          float *__restrict__ out, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int d = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
  if (d >= D) return;
  const uint4 *r2 = reinterpret_cast<const uint4 *>(w2 + (int64_t)d * Fs);
  const int nc = Fs / 8;
  for (int t0 = 0; t0 < T; t0 += kGT) {
    const int nt = T - t0 < kGT ? T - t0 : kGT;
    float y[kGT];
#pragma unroll
    for (int t = 0; t < kGT; ++t) y[t] = 0.f;
#pragma unroll 4
    for (int c = lane; c < nc; c += 32) {
      float a[8];
      bf16x8_to_f32(__ldg(r2 + c), a);
#pragma unroll
      for (int t = 0; t < kGT; ++t)
        if (t < nt) {
          float hv[8];
          bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4 *>(h + (int64_t)(t0 + t) * Fs) + c), hv);
#pragma unroll
          for (int j = 0; j < 8; ++j) y[t] = fmaf(a[j], hv[j], y[t]);
        }
    }
    float mine = 0.f;
#pragma unroll
    for (int t = 0; t < kGT; ++t)
      if (t < nt) {
        const float s = warp_sum(y[t]);
        if (lane == t) mine = s;
      }
    if (lane < nt) {
      float *o = out + (int64_t)(t0 + lane) * D + d;
      *o = accumulate ? *o + mine : mine;
    }
  }
}

// ------------------------------------------------------ tensor-core path
constexpr int kTok = 128;     // tokens per tile (MMA M)
constexpr int kRows = 256;    // weight rows per tile (MMA N)
constexpr int kK = 64;        // K values per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kATile = kTok * kK * 2;     // 16 KB
constexpr int kBTile = kRows * kK * 2;    // 32 KB
constexpr int kStage = kATile + kBTile;   // 48 KB
constexpr int kAccCols = kRows;           // fp32 columns per accumulator
constexpr int kTmemCols = 2 * kAccCols;   // two accumulators
constexpr int kTmaWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2;
constexpr int kDenseThreads = 6 * 32;
constexpr int kDenseSmem = kStages * kStage + 1024 + 256;  // stages, alignment slack, barriers + TMEM holder

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart; the start address advances 32 bytes per K = 16 slice.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16 with bf16 A and B (K-major), fp32 D.
__device__ __forceinline__ uint32_t bf16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct DenseArgs {
  int T, K;          // tokens, reduction length
  int nrt;           // weight-row tiles (gate/up: Fs / 128; down: D / 256)
  int ldo;           // output row length (gate/up: Fs; down: D)
  void *out;         // gate/up: h bf16 [T][Fs]; down: out fp32 [T][D]
  int accumulate;    // down: add to out
  WsHeader *hdr;
};

// GATEUP: B = 128 rows of w1 (map mB0) and the same 128 rows of w3 (mB1);
// otherwise B = 256 rows of w2 (two 128-row boxes of mB0).
template <bool GATEUP>
__global__ void __launch_bounds__(kDenseThreads, 1)
    k_shared_tc(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                const __grid_constant__ CUtensorMap mB1, DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const SpanExit span_exit(GATEUP ? DS4MOE_SPAN_SHARED_GATE_UP_TC : DS4MOE_SPAN_SHARED_DOWN_TC);
  span_begin(GATEUP ? DS4MOE_SPAN_SHARED_GATE_UP_TC : DS4MOE_SPAN_SHARED_DOWN_TC);
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + kStages * kStage);
  uint64_t *empty = full + kStages, *tfull = empty + kStages, *tempty = tfull + 2, *drain = tempty + 2;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], 4);
    }
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
  const int ntt = (a.T + kTok - 1) / kTok, nunits = ntt * a.nrt, nks = a.K / kK;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int t0 = (u / a.nrt) * kTok, r0 = (u % a.nrt) * (GATEUP ? kTok : kRows);
        for (int s = 0; s < nks; ++s, ++it) {
          const int slot = it % kStages;
          if (!ptx::mbar_wait_or_abort(&empty[slot], ((it / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
          uint8_t *st = sm + slot * kStage;
          // full boxes: rows past the last token (or matrix row) arrive as zeros
          ptx::mbar_arrive_expect_tx(&full[slot], kStage);
          ptx::tma_load_2d(st, &mA, s * kK, t0, &full[slot]);
          ptx::tma_load_2d(st + kATile, &mB0, s * kK, r0, &full[slot]);
          if (GATEUP)
            ptx::tma_load_2d(st + kATile + kBTile / 2, &mB1, s * kK, r0, &full[slot]);
          else
            ptx::tma_load_2d(st + kATile + kBTile / 2, &mB0, s * kK, r0 + kTok, &full[slot]);
        }
      }
      if (!ok) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        *abort_flag = 1;
        for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)  // let issued copies land
          ptx::mbar_wait(&full[j % kStages], (j / kStages) & 1, 1u << 20);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = bf16_idesc(kTok, kRows);
      int it = 0, tit = 0;
      bool ok = true, issued = false;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++tit) {
        const int tb = tit & 1;
        if (!ptx::mbar_wait_or_abort(&tempty[tb], ((tit >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dcol = tmem + (uint32_t)(tb * kAccCols);
        for (int s = 0; s < nks; ++s, ++it) {
          const int slot = it % kStages;
          if (!ptx::mbar_wait_or_abort(&full[slot], (it / kStages) & 1, abort_flag)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sm + slot * kStage), b0 = a0 + kATile;
#pragma unroll
          for (int kk = 0; kk < kK / 16; ++kk)
            ptx::umma_f16(dcol, sw128_desc(a0 + 32 * kk), sw128_desc(b0 + 32 * kk), idesc, (s | kk) != 0);
          issued = true;
          ptx::umma_commit(&empty[slot]);
        }
        if (ok) ptx::umma_commit(&tfull[tb]);
      }
      if (!ok) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        *abort_flag = 1;
        if (issued) {  // let the issued MMAs finish before TMEM is freed
          ptx::umma_commit(drain);
          ptx::mbar_wait(drain, 0, 1u << 20);
        }
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // epilogue warps 2..5: TMEM lanes 32 (warp % 4) .. +31 = tokens of the tile
    const int sub = warp & 3, row = 32 * sub + lane;
    int tit = 0;
    bool big = false;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++tit) {
      const int tb = tit & 1;
      if (!__all_sync(~0u, ptx::mbar_wait_or_abort(&tfull[tb], (tit >> 1) & 1, abort_flag))) {
        record_status(a.hdr, DS4MOE_ETIMEOUT);
        *abort_flag = 1;
        break;
      }
      ptx::tc_fence_after();
      const int tok = (u / a.nrt) * kTok + row, r0 = (u % a.nrt) * (GATEUP ? kTok : kRows);
      const uint32_t tbase = tmem + ((uint32_t)(32 * sub) << 16) + (uint32_t)(tb * kAccCols);
      if constexpr (GATEUP) {
        uint4 *H = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + (int64_t)tok * a.ldo + r0);
#pragma unroll 1
        for (int c0 = 0; c0 < kTok; c0 += 32) {
          uint32_t g[32], v[32];
          ptx::tmem_ld32x2_wait(tbase + c0, tbase + kTok + c0, g, v);
          if (tok < a.T) {
            uint32_t hp[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float h0 = silu(__uint_as_float(g[j])) * __uint_as_float(v[j]);
              const float h1 = silu(__uint_as_float(g[j + 1])) * __uint_as_float(v[j + 1]);
              big |= !(fabsf(h0) < 3.0e38f) || !(fabsf(h1) < 3.0e38f);
              hp[j >> 1] = (uint32_t)f32_to_bf16_bits(h0) | ((uint32_t)f32_to_bf16_bits(h1) << 16);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) H[c0 / 8 + q] = make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
          }
        }
      } else {
        float *O = static_cast<float *>(a.out) + (int64_t)tok * a.ldo + r0;
#pragma unroll 1
        for (int c0 = 0; c0 < kRows; c0 += 32) {
          uint32_t y[32];
          ptx::tmem_ld32_wait(tbase + c0, y);
          if (tok < a.T) {
            float4 *o4 = reinterpret_cast<float4 *>(O + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 v = make_float4(__uint_as_float(y[4 * q]), __uint_as_float(y[4 * q + 1]),
                                     __uint_as_float(y[4 * q + 2]), __uint_as_float(y[4 * q + 3]));
              if (a.accumulate) {
                const float4 p = o4[q];
                v.x += p.x;
                v.y += p.y;
                v.z += p.z;
                v.w += p.w;
              }
              o4[q] = v;
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[tb]);
    }
    if (big) record_status(a.hdr, DS4MOE_EDEVICE);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
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

// bf16 matrix [rows][cols], row-major; boxes of 64 values x 128 rows,
// 128-byte swizzle (the canonical K-major layout of one MMA operand slice).
bool map_bf16(CUtensorMap *m, const void *base, int64_t cols, int64_t rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kK, (cuuint32_t)kTok};
  const cuuint32_t es[2] = {1, 1};
  return encode_tiled()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool GATEUP>
cudaError_t launch_dense(const CUtensorMap &mA, const CUtensorMap &mB0, const CUtensorMap &mB1, const DenseArgs &da,
                         cudaStream_t s) {
  auto kern = k_shared_tc<GATEUP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  if (e != cudaSuccess) return e;
  const int units = (da.T + kTok - 1) / kTok * da.nrt;
  const int grid = units < num_sms() ? units : num_sms();
  ProfScope p(GATEUP ? "shared_gate_up_tc" : "shared_down_tc", s);
  kern<<<grid, kDenseThreads, kDenseSmem, s>>>(mA, mB0, mB1, da);
  return cudaGetLastError();
}

bool tc_shape_ok(int D, int Fs) {
  if (D % kRows || Fs % kTok || D % kK || Fs % kK) return false;
  if (!encode_tiled()) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  return major == 10;
}

}  // namespace

size_t shared_ws_bytes(int D, int Fs, int T) {
  (void)D;
  return align256(sizeof(WsHeader)) + align256(sizeof(uint16_t) * (size_t)T * (size_t)(Fs > 0 ? Fs : 0));
}

bool shared_uses_tc(int D, int Fs, int T) { return T > kSimtTokens && tc_shape_ok(D, Fs); }

cudaError_t launch_shared_ffn(const uint16_t *w1, const uint16_t *w3, const uint16_t *w2, int D, int Fs,
                              const uint16_t *x, int T, float *out, int accumulate, void *ws, cudaStream_t s) {
  WsHeader *hdr = static_cast<WsHeader *>(ws);
  uint16_t *h = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + align256(sizeof(WsHeader)));
  cudaError_t e;
  if (Fs == 0) return accumulate ? cudaSuccess : cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * D, s);
  if (shared_uses_tc(D, Fs, T)) {
    CUtensorMap mx, m1, m3, m2, mh;
    if (!map_bf16(&mx, x, D, T) || !map_bf16(&m1, w1, D, Fs) || !map_bf16(&m3, w3, D, Fs) ||
        !map_bf16(&m2, w2, Fs, D) || !map_bf16(&mh, h, Fs, T))
      return cudaErrorInvalidValue;
    DenseArgs gu{T, D, Fs / kTok, Fs, h, 0, hdr};
    if ((e = launch_dense<true>(mx, m1, m3, gu, s)) != cudaSuccess) return e;
    DenseArgs dn{T, Fs, D / kRows, D, out, accumulate, hdr};
    return launch_dense<false>(mh, m2, m2, dn, s);
  }
  {
    ProfScope p("shared_gate_up_simt", s);
    k_shared_gu_simt<<<(Fs + kGemvWarps - 1) / kGemvWarps, 32 * kGemvWarps, 0, s>>>(w1, w3, x, D, Fs, T, h);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ProfScope p("shared_down_simt", s);
  k_shared_down_simt<<<(D + kGemvWarps - 1) / kGemvWarps, 32 * kGemvWarps, 0, s>>>(w2, h, D, Fs, T, out, accumulate);
  return cudaGetLastError();
}

cudaError_t span_control_shared(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4
