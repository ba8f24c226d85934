// Internal declarations shared by the ds4moe translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/ds4moe.h"

namespace ds4 {

// ------------------------------------------------------------ formats
constexpr int kQ41Vals = 32, kQ41Bytes = 20;
constexpr int kQ2KVals = 256, kQ2KBytes = 84;
constexpr int kQ4KVals = 256, kQ4KBytes = 144;

// The 16-row tile order of Q2_K keeps its 84 bytes per 256 values.
__host__ __device__ inline int block_vals(int q) {
  return q == DS4MOE_Q4_1 ? kQ41Vals
         : (q == DS4MOE_Q2_K || q == DS4MOE_Q2_K_R16) ? kQ2KVals
         : q == DS4MOE_Q4_K ? kQ4KVals : 0;
}
__host__ __device__ inline int block_bytes(int q) {
  return q == DS4MOE_Q4_1 ? kQ41Bytes
         : (q == DS4MOE_Q2_K || q == DS4MOE_Q2_K_R16) ? kQ2KBytes
         : q == DS4MOE_Q4_K ? kQ4KBytes : 0;
}

// Q4_K sub-block j's 6-bit scale and min from the 12 packed bytes.
__device__ __forceinline__ void q4k_scale_min(const uint8_t *s12, int j, uint32_t &sc, uint32_t &mn) {
  if (j < 4) {
    sc = s12[j] & 63u;
    mn = s12[j + 4] & 63u;
  } else {
    sc = (s12[j + 4] & 15u) | ((uint32_t)(s12[j - 4] >> 6) << 4);
    mn = (uint32_t)(s12[j + 4] >> 4) | ((uint32_t)(s12[j] >> 6) << 4);
  }
}
__host__ __device__ inline int64_t row_bytes(int q, int cols) {
  return (int64_t)(cols / block_vals(q)) * block_bytes(q);
}

// ---------------------------------------------------------- workspace
// Every region starts on a 256-byte boundary.  The header holds the sticky
// device status word and small counters.
struct WsHeader {
  uint32_t status;     // 0 or a ds4moe_status recorded by a kernel
  int32_t n_active;    // experts with >= 1 routed pair (set by bucketing)
  uint32_t route_done; // last-block counter of the fused router
  int32_t n_groups;    // token groups (<= kGroup pairs of one expert each)
  uint32_t pad[60];
};

// A token group: up to kGroup consecutive expert-sorted pairs of one expert.
constexpr int kGroup = 8;
struct Group {
  int32_t e, p0, nt, pad;
};

// Sub-block sums of an activation row for the tensor-core kernels: per
// 256-value block a 64-byte record of 16 fp16 "hi" parts then 16 fp16 "lo"
// parts (sum of sub-block n ~= hi[n] + lo[n]), in sub-block order.
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

// A token chunk of the prefill grouped GEMMs: n <= BN consecutive
// expert-sorted pairs p0 .. p0+n-1, all routed to expert e.
struct Chunk {
  int32_t e, p0, n, pad;
};
// Token-chunk widths of the prefill kernels (gate/up and down).
constexpr int kChunkGateUp = 128, kChunkDown = 256;
// Row length of the gathered prefill activations: D fp16 values, then the
// hi/lo fp16 parts of the block sums (D/32 blocks of 32 values for Q4_1 /
// Q4_K gate/up, D/16 sub-blocks of 16 for Q2_K: room for the larger).
inline int64_t xp_cols(int64_t D) { return D + D / 8; }

struct WsLayout {
  size_t hdr, logits, rnorm, rlist, counts, offs, active, perm, inv, lrank, groups, x16, xs16, xs32, hs16, h, y, nvalid, cnt,
      xp, chunks_gu, chunks_dn, nchunks, res2, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline WsLayout ws_layout(const ds4moe_layer &L, int T, int k, int prefill) {
  WsLayout w{};
  size_t o = 0;
  const size_t E = (size_t)L.n_expert, P = (size_t)T * (size_t)k;
  w.hdr = o;     o += align256(sizeof(WsHeader));
  w.logits = o;  o += align256(sizeof(float) * (size_t)T * E);
  w.rnorm = o;   o += align256(sizeof(float) * ((size_t)T + E));    // router fast path: row norms of x, Wr
  w.rlist = o;   o += align256(sizeof(int32_t) * ((size_t)T + 64)); // count, then tokens handed back
  w.counts = o;  o += align256(sizeof(int32_t) * E);
  w.offs = o;    o += align256(sizeof(int32_t) * (E + 1));
  w.active = o;  o += align256(sizeof(int32_t) * E);
  w.perm = o;    o += align256(sizeof(int32_t) * P);
  w.inv = o;     o += align256(sizeof(int32_t) * P);
  w.lrank = o;   o += align256(sizeof(int32_t) * P);
  w.groups = o;  o += align256(sizeof(Group) * P);
  w.x16 = o;     o += align256(sizeof(uint16_t) * (size_t)T * (size_t)L.d_model);
  w.xs16 = o;    o += align256((size_t)T * (size_t)(L.d_model / 256 + 1) * 64);
  w.xs32 = o;    o += align256(sizeof(float) * (size_t)T * (size_t)(L.d_model / 32 + 1));
  w.hs16 = o;    o += align256(P * (size_t)(L.d_ff / 256 + 1) * 64);
  // h: bf16 per element; the tile-order single-token grid stores each as a
  // tagged 32-bit word
  const bool r16 = L.q_gate == DS4MOE_Q2_K_R16;
  w.h = o;       o += align256((r16 ? sizeof(uint32_t) : sizeof(uint16_t)) * P * (size_t)L.d_ff);
  w.y = o;       o += align256(sizeof(float) * P * (size_t)L.d_model);
  w.nvalid = o;  o += align256(sizeof(int32_t) * (size_t)T);
  w.cnt = o;     o += align256(sizeof(int32_t) * (size_t)T * (size_t)(L.d_model / 16));
  w.res2 = o;    o += align256(sizeof(float) * (size_t)T * (size_t)L.d_model);  // the stack's second residual buffer
  if (prefill) {  // tensor-core prefill: x gathered in pair order, token chunks
    const size_t ne = E < P ? E : P;
    w.xp = o;        o += align256(sizeof(uint16_t) * P * (size_t)xp_cols(L.d_model));
    w.chunks_gu = o; o += align256(sizeof(Chunk) * (ne + P / kChunkGateUp + 1));
    w.chunks_dn = o; o += align256(sizeof(Chunk) * (ne + P / kChunkDown + 1));
    w.nchunks = o;   o += align256(2 * sizeof(int32_t));
  }
  w.total = o;
  return w;
}

template <typename T>
inline T *ws_ptr(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

// ------------------------------------------------------- device helpers
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ void record_status(WsHeader *hdr, uint32_t code) {
  atomicCAS(&hdr->status, 0u, code);
}

// Round-to-nearest-even fp32 -> bf16 bit pattern (hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Routing weights of a decode batch of P = T * k <= 32 pairs, by one warp:
// w[t*k + i] holds the i-th selected logit of token t (descending), and is
// replaced by exp(l_i - l_0) / sum_j exp(l_j - l_0), in double, summed in
// rank order, rounded once to fp32 -- one lane per pair.
__device__ __forceinline__ void finish_routing_weights(float *w, int T, int k) {
  const int lane = threadIdx.x & 31, P = T * k;
  const int base = lane < P ? lane - lane % k : 0;
  const float v = lane < P ? w[lane] : 0.f;
  const double m = (double)__shfl_sync(0xffffffffu, v, base);
  const double ex = lane < P ? exp((double)v - m) : 0.0;
  double sum = 0.0;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, base + j < 32 ? base + j : 0);
  if (lane < P) w[lane] = (float)(ex / sum);
}

// ------------------------------------------------------- launch entry points
// (defined in ffn_decode.cu / ffn_prefill.cu; called from ds4moe_abi.cu)
struct FfnArgs {
  ds4moe_layer L;
  const uint16_t *x;
  int x_late;  // x is written by the preceding grid: read it only after the dependency wait
  const float *w;
  int T, k;
  float *out;
  WsHeader *hdr;
  const int32_t *offs, *active, *perm, *inv;
  const Group *groups;
  const uint16_t *x16;  // [T][D] x as fp16 (tensor-core path)
  const uint8_t *xs16;  // [T][D/256][64 B] sub-block sums of x
  const float *xs32;    // [T][D/32] block sums of x
  uint8_t *hs16;        // [P][F/256][64 B] sub-block sums of h
  uint16_t *h;          // [P][F] hidden: fp16 (tensor-core path) or bf16 (SIMT)
  float *y;
  const int32_t *nvalid;  // [T] experts in range per token
  int32_t *cnt;           // [T][D/16] arrival counters of the fused combine (nullptr: separate combine)
  int w_logits;           // w holds the k selected logits per token: the gate/up grid turns them into weights
  // single-token chain only (nullptr otherwise): the FFN grids rank the
  // experts themselves from the router's logits [E]; CTA 0 of the gate/up
  // grid writes idx_out / w and the bucketing outputs
  const float *lg;
  int32_t *idx_out;
  // merged single-token FFN grid only: per selected expert, the gate/up
  // units that have published their h (zeroed by the router grid)
  int32_t *hready;
  int32_t *ccnt;  // and per 64 output rows, the down items finished (zeroed by the router grid)
  // tensor-core prefill only (nullptr otherwise)
  uint16_t *xp;           // [P][D] x of each sorted pair, fp16
  Chunk *chunks_gu, *chunks_dn;
  int32_t *nchunks;       // [2]: chunk counts of chunks_gu / chunks_dn
};

// The combine's arrival counters start every call at zero: the gate/up grid
// clears them (the down grid reads them only after that grid completes).
// The workspace regions move with the call's sizes, so what the previous
// call left there cannot be relied on.
// `tid` of `nthr` threads per CTA take part.
__device__ __forceinline__ void clear_combine_counters(const FfnArgs &a, int tid, int nthr) {
  if (!a.cnt) return;
  const int64_t n = (int64_t)a.T * (a.L.d_model / 16);
  for (int64_t i = blockIdx.x * (int64_t)nthr + tid; i < n; i += (int64_t)gridDim.x * nthr) a.cnt[i] = 0;
}

cudaError_t launch_ffn_decode(const FfnArgs &a, cudaStream_t s);
// Single-token FFN over DS4MOE_Q2_K_R16 weights (ffn_t1r.cu): the layer
// shapes it takes, its launch, the repacking kernels, the fault-injection
// hook of its h-ready wait and its device-side span record.
bool t1r_ok(const ds4moe_layer &L, int k);
cudaError_t launch_ffn_t1r(const FfnArgs &a, cudaStream_t s);
// shared expert (shared_ffn.cu)
size_t shared_ws_bytes(int D, int Fs, int T);
bool shared_uses_tc(int D, int Fs, int T);
cudaError_t launch_shared_ffn(const uint16_t *w1, const uint16_t *w3, const uint16_t *w2, int D, int Fs,
                              const uint16_t *x, int T, float *out, int accumulate, void *ws, cudaStream_t s);
cudaError_t launch_repack(bool to_r16, const void *src, void *dst, int64_t rows, int64_t cols, cudaStream_t s);
cudaError_t t1r_set_sync_hook(int32_t budget, int32_t extra);
cudaError_t launch_ffn_prefill(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_combine(const FfnArgs &a, cudaStream_t s);
bool decode_mma_ok(const ds4moe_layer &L);
// Both single-token FFN kernels apply (the single-token chain of the fused
// decode entry ranks the experts inside them).
bool t1_chain_ok(const ds4moe_layer &L);
bool prefill_tc_ok(const ds4moe_layer &L);
// Prefill split (ffn_decode.cu): layers whose formats the persistent
// multi-token kernels take send experts with at most kSmallPairs pairs to
// them (one token group of <= 8 pairs streams the expert's weights once).
constexpr int kSmallPairs = 16;
bool prefill_split_ok(const ds4moe_layer &L);
cudaError_t launch_gate_up_groups(const FfnArgs &a, cudaStream_t s);
cudaError_t launch_down_groups(const FfnArgs &a, cudaStream_t s);

int num_sms();

// Launch with programmatic stream serialization (the kernel overlaps the
// tail of the preceding grid and must call ptx::pdl_wait before consuming
// its outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Brackets one kernel launch with CUDA events while profiling is enabled
// (ds4moe_profile_enable); a no-op otherwise and during stream capture.
class ProfScope {
 public:
  ProfScope(const char *name, cudaStream_t s);
  ~ProfScope();
  ProfScope(const ProfScope &) = delete;
  ProfScope &operator=(const ProfScope &) = delete;

 private:
  const char *name_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace ds4
