/*
 * ds4moe -- routed-MoE expert FFN over low-bit block-quantized weights
 * (Q4_1 and Q2_K) for one NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; no CUDA, PyTorch or C++ types cross
 * this boundary.  A "stream" argument is a cudaStream_t passed as void*
 * (NULL = the legacy default stream).  Device pointers must come from
 * cudaMalloc-class allocations on the current device.
 *
 * Sources of the operations (web pages):
 *  [DS4-1] molayo1419.me, "ds4.c 해독하기 1/8": DeepSeek V4 Flash shape --
 *          256 routed experts per layer, 6 used per token, 43 layers.
 *  [DS4-2] molayo1419.me, "【#2】ds4.c 해독하기": the routed-expert-only
 *          2-bit recipe (w1 = gate, w2 = down, w3 = up; expert matrices
 *          4096 x 2048); the Q2_K type trait (256 values / 84 bytes), its
 *          layout table and its qs packing expression.
 *  [Q41]   thakicloud.com, "자체 저비트 포맷을 llama.cpp로 옮기기: 복원값이
 *          비트까지 같은 GGUF Q4_1 재부호화": the Q4_1 block ("Q4_1 블록이 어떻게
 *          생겼나"), the lossless re-encode and its two conditions ("무손실이
 *          성립하는 조건 두 개", "실제로 돌린 코드"), explicit bits/group ("비트
 *          폭과 그룹 크기는 메타데이터에서만 읽습니다"), block order along the
 *          input dimension ("텐서 이름과 KV 메타데이터").
 *
 * Conventions
 *  - The caller owns every buffer.  Nothing here allocates device memory on
 *    the compute path; scratch lives in a caller-provided workspace whose size
 *    ds4moe_workspace_bytes() returns.
 *  - Device entry points are asynchronous on `stream`.  Errors that the host
 *    can see (bad sizes, NULL or misaligned pointers, unsupported formats,
 *    too small a workspace) return before anything is launched.  Errors that
 *    only the device can see (an expert id out of range, a bounded wait that
 *    gave up) are recorded in a status word inside the workspace and reported
 *    by ds4moe_stream_status(); kernels never trap.
 *  - Alignment: every device pointer must be 16-byte aligned.
 *  - Weight tensors are experts-major: expert e of a [rows x cols] matrix
 *    starts at byte e * rows * row_bytes, row r at + r * row_bytes, and a row
 *    is cols / block_values consecutive blocks along the input axis.
 *    gate (w1) and up (w3) are [d_ff x d_model], down (w2) is [d_model x d_ff].
 *  - Activations x are bf16 bit patterns (uint16_t), row-major [T, d_model].
 *  - T == 0 is a no-op that returns DS4MOE_OK.
 */
#ifndef DS4MOE_H
#define DS4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS4MOE_OK = 0,
  DS4MOE_EINVAL = 1,       /* invalid argument (host-detected, nothing launched) */
  DS4MOE_EBLOCKER = 2,     /* lossless re-encode condition violated ([Q41]) */
  DS4MOE_EUNSUPPORTED = 3, /* block format not supported (e.g. IQ2_XXS) */
  DS4MOE_ECUDA = 4,        /* a CUDA runtime call failed */
  DS4MOE_ETIMEOUT = 5,     /* a bounded device-side wait gave up */
  DS4MOE_EDEVICE = 6,      /* device-detected data error (expert id out of range) */
  DS4MOE_ESPACE = 7        /* workspace smaller than ds4moe_workspace_bytes() */
} ds4moe_status;

/* Block formats.  These ids are this library's own, not ggml's. */
typedef enum {
  DS4MOE_Q4_1 = 1,   /* 32 values in 20 bytes: fp16 d @0, fp16 m @2, qs[16] @4;
                        value j = low nibble of qs[j], value j+16 = high nibble;
                        y = d*q + m  ([Q41] "Q4_1 블록이 어떻게 생겼나") */
  DS4MOE_Q2_K = 2,   /* 256 values in 84 bytes: scales[16] @0 (sc | mn << 4 per
                        16 values), qs[64] @16, fp16 d @80, fp16 dmin @82;
                        value i: code (qs[32*(i/128) + i%32] >> 2*((i%128)/32)) & 3,
                        y = d*sc*q - dmin*mn  ([DS4-2] layout table and packing) */
  DS4MOE_IQ2_XXS = 3, /* named by [DS4-2]; its grid codebook is not given there:
                        every entry point returns DS4MOE_EUNSUPPORTED */
  DS4MOE_Q4_K = 4,   /* 256 values in 144 bytes ([DS4-2] type table; the layout
                        is the standard k-quant reading): fp16 d @0, fp16 dmin
                        @2, scales[12] @4, qs[128] @16.  Sub-block j = values
                        32j..32j+31: j < 4: sc = s[j] & 63, mn = s[j+4] & 63;
                        j >= 4: sc = (s[j+4] & 15) | (s[j-4] >> 6) << 4,
                        mn = (s[j+4] >> 4) | (s[j] >> 6) << 4.  Value 64c+l
                        (l < 32): low nibble of qs[32c+l]; 64c+32+l: its high
                        nibble.  y = d*sc*q - dmin*mn.  Dequant and the FFN
                        entry points (SIMT kernels) take it. */
  DS4MOE_Q2_K_R16 = 5 /* the Q2_K blocks above in a 16-row tile order, made by
                        ds4moe_repack: the same 84 bytes per 256 values and the
                        same values, each 16-row x 256-column tile-block of a
                        matrix keeping the 16 x 84 bytes the plain layout gives
                        it, permuted inside (lane L = 4g + c, rows g, g+8):
                        [0,1024) codes, half h of lane L at 512h + 16L as four
                        words (row g, sub-block 8h+c), (g+8, 8h+c), (g, 8h+c+4),
                        (g+8, 8h+c+4), value v of a sub-block at bit
                        16(v&1) + 2(v>>1); [1024,1280) scale bytes, lane L at
                        1024 + 8L: per row g, g+8 the word s[2c] | s[2c+8]<<8 |
                        s[2c+1]<<16 | s[2c+9]<<24; [1280,1344) row r's d, dmin
                        at 1280 + 4r.  Matrices need rows % 16 == 0.  Taken by
                        the single-token decode (ds4moe_moe_decode,
                        ds4moe_ffn_decode and ds4moe_ffn_decode_noalloc at T = 1,
                        ds4moe_stack_decode at T = 1) when gate, up and down are
                        all in this order and d_model = 2 d_ff, d_model a
                        multiple of 512 up to 4096; everything else returns
                        DS4MOE_EUNSUPPORTED (ds4moe_dequant included: repack to
                        DS4MOE_Q2_K first). */
} ds4moe_qtype;

/* One routed-MoE layer's expert weights (device pointers, 16-byte aligned). */
typedef struct {
  int32_t d_model;   /* D: input/output width (multiple of the gate/up block size) */
  int32_t d_ff;      /* F: hidden width (multiple of the down block size and of 16) */
  int32_t n_expert;  /* E: routed experts in this layer, 1..1024 */
  int32_t q_gate, q_up, q_down;  /* ds4moe_qtype of each matrix */
  const void *gate;  /* [E][F rows][D/bv * bb bytes]  w1 */
  const void *up;    /* [E][F rows][D/bv * bb bytes]  w3 */
  const void *down;  /* [E][D rows][F/bv * bb bytes]  w2 */
} ds4moe_layer;

/* Values and bytes per block of a format (0 if unknown). */
int32_t ds4moe_block_values(int32_t qtype);
int32_t ds4moe_block_bytes(int32_t qtype);

/* Human-readable name of a status code (static string). */
const char *ds4moe_status_string(int32_t status);

/*
 * ds4moe_quantize_ref -- HOST, synchronous.  Packs integer codes and their
 * scales into blocks; nothing is recomputed or rounded.
 *
 * out_type == DS4MOE_Q4_1: the lossless re-encode of [Q41] ("무손실이
 *   성립하는 조건 두 개", "실제로 돌린 코드").  `codes` holds n_values codes,
 *   one per byte, each < 2^bits; scale_f16[g] / min_f16[g] are the fp16 bit
 *   patterns of group g (n_values / group entries each).  Each 32-value block
 *   copies its group's (scale, min) into (d, m) and folds its codes into
 *   nibbles.  bits and group are explicit and never inferred from a byte
 *   count ([Q41] "비트 폭과 그룹 크기는 메타데이터에서만 읽습니다").
 *   Returns DS4MOE_EBLOCKER if group % 32 != 0, bits > 4 or any code >=
 *   2^bits (no fallback); DS4MOE_EINVAL if bits < 1, group < 1, n_values %
 *   group != 0 or a pointer is NULL.  sub_sc / sub_mn must be NULL.
 * out_type == DS4MOE_Q2_K: packs 2-bit codes ([DS4-2] layout table and qs
 *   packing).  bits must be 2 and group 256; scale_f16 / min_f16 hold d and
 *   dmin per 256 values; sub_sc / sub_mn hold the 4-bit scale and min of each
 *   16-value sub-block (n_values / 16 entries, one per byte).  Codes > 3 or
 *   nibbles > 15 return DS4MOE_EBLOCKER.
 * out_type == DS4MOE_Q4_K: packs 4-bit codes into the 144-byte layout
 *   above.  bits must be 4 and group 256; scale_f16 / min_f16 hold d and dmin
 *   per 256 values; sub_sc / sub_mn the 6-bit scale and min of each 32-value
 *   sub-block (n_values / 32 entries).  Codes > 15 or fields > 63 return
 *   DS4MOE_EBLOCKER.
 * out_type == DS4MOE_IQ2_XXS: DS4MOE_EUNSUPPORTED.
 * out_bytes must be at least n_values / block_values * block_bytes
 * (DS4MOE_ESPACE otherwise).  `out_blocks` is host memory.
 */
ds4moe_status ds4moe_quantize_ref(int32_t out_type, int32_t bits, int32_t group,
                                  const uint8_t *codes, const uint16_t *scale_f16,
                                  const uint16_t *min_f16, const uint8_t *sub_sc,
                                  const uint8_t *sub_mn, int64_t n_values,
                                  void *out_blocks, size_t out_bytes);

/*
 * ds4moe_quantize_f32 -- DEVICE, asynchronous on `stream`.  Quantizes
 * n_values fp32 values `x` (device, rows of `cols` values) into Q2_K or Q4_1
 * blocks `out` (device, out_bytes >= n_values / block_values * block_bytes).
 * [DS4-2], section on the Q2_K block writer: a scale and a minimum per
 * 16-value sub-block, values rounded to 2-bit codes; with an importance
 * matrix the weighted writer scores the error by column importance.  The
 * pages give no search; this one (fp32, fixed order, deterministic):
 *   Q2_K  per sub-block lo = min(0, min x), hi = max x, a = (hi - lo) / 3,
 *         b = -lo; d = f16(max a / 15), dmin = f16(max b / 15); sc = rint(a /
 *         d), mn = rint(b / dmin) clamped to 0..15; nearest codes 0..3.
 *   Q4_1  d = f16((max - min) / 15), m = f16(min); nearest codes 0..15.
 *   importance (device, `cols` fp32 weights, one per column; NULL: none):
 *         every sub-block tries (sc, mn) +-1 (Q4_1: d and m one binary16
 *         step each way) and keeps the first candidate with the least
 *         sum importance * (x - y)^2, the plain choice tried first.
 * cols must be a multiple of the block size dividing n_values when
 * importance is given.  Host errors: EUNSUPPORTED (other formats), EINVAL
 * (sizes, NULL or unaligned pointers), ESPACE (out_bytes, or ws_bytes <
 * 256).  Device-detected: a block holding a non-finite value is written as
 * zeros and DS4MOE_EDEVICE is recorded in `ws` (read it with
 * ds4moe_stream_status).  `ws`: a workspace from ds4moe_workspace_init.
 */
ds4moe_status ds4moe_quantize_f32(int32_t qtype, const float *x, const float *importance, int64_t n_values,
                                  int64_t cols, void *out, size_t out_bytes, void *ws, size_t ws_bytes,
                                  void *stream);

/*
 * ds4moe_repack -- DEVICE, asynchronous on `stream`.  Rewrites a Q2_K matrix
 * between the plain block layout (DS4MOE_Q2_K) and the 16-row tile order
 * (DS4MOE_Q2_K_R16) above, in either direction: (src_type, dst_type) =
 * (DS4MOE_Q2_K, DS4MOE_Q2_K_R16) or the reverse.  A bijection on the bytes:
 * every value, scale and d / dmin is kept, so repacking back gives the input
 * bit for bit.  [DS4-2]'s layout table and qs packing define the values; the
 * tile order is this library's (it lets a tensor-core lane read its 64 codes
 * with one 16-byte load), not the pages'.
 * src, dst: device, 16-byte aligned, rows * cols / 256 * 84 bytes each, not
 * overlapping.  rows % 16 == 0 and cols % 256 == 0; an experts-major [E][R][C]
 * tensor is rows = E * R.  Host errors: EINVAL (sizes, NULL or misaligned
 * pointers, src == dst), EUNSUPPORTED (any other pair of formats).
 */
ds4moe_status ds4moe_repack(int32_t src_type, int32_t dst_type, const void *src, int64_t rows,
                            int64_t cols, void *dst, void *stream);

/*
 * ds4moe_dequant -- DEVICE.  Decodes n_values values of `blocks` (device,
 * qtype layout above) into fp32 `out` (device).  The result is the single
 * fp32 rounding of the exact decoded value (d*q + m, or d*sc*q - dmin*mn),
 * so it is unique bit for bit.  n_values must be a multiple of the block
 * size.
 */
ds4moe_status ds4moe_dequant(int32_t qtype, const void *blocks, int64_t n_values,
                             float *out, void *stream);

/*
 * ds4moe_workspace_bytes -- bytes of device workspace needed by
 * ds4moe_route_topk + ds4moe_ffn_decode / ds4moe_ffn_prefill for this layer
 * shape, T tokens and top-k (one workspace serves all three calls).  Returns
 * 0 for invalid arguments.  `prefill` selects the prefill path's layout.
 */
size_t ds4moe_workspace_bytes(const ds4moe_layer *L, int32_t T, int32_t k,
                              int32_t prefill);

/*
 * ds4moe_workspace_init -- DEVICE.  Zeroes the workspace (its status word;
 * every other region, the combine's arrival counters included, is written
 * by each call before it is read, so one workspace may serve calls of any
 * sizes it is large enough for).  Call once after allocating it.
 */
ds4moe_status ds4moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * ds4moe_route_topk -- DEVICE.  Router of one layer ([DS4-1] model shape:
 * top-6 of 256 experts per token; scoring per the library's reading: plain
 * logits with a softmax over the selected experts).
 *   logits[t,e] = sum_j x[t,j] * Wr[e,j] (+ bias[e]), computed with a
 *     compensated (twice-working-precision) dot product and rounded once to
 *     fp32;
 *   idx[t, 0..k) = the k largest logits, descending, ties to the lower
 *     expert id, NaN below -inf;
 *   w[t,i] = exp(l_i - l_0) / sum_j exp(l_j - l_0) over the k selected.
 * x: bf16 [T, d_model]; Wr: fp32 [n_expert, d_model]; bias: fp32 [n_expert]
 * or NULL; idx: int32 [T, k]; w: fp32 [T, k]; logits: fp32 [T, n_expert] or
 * NULL.  1 <= k <= min(n_expert, 32), d_model % 4 == 0.  `ws` is the layer
 * workspace (ds4moe_workspace_bytes).
 */
ds4moe_status ds4moe_route_topk(const uint16_t *x, const float *Wr, const float *bias,
                                int32_t T, int32_t d_model, int32_t n_expert, int32_t k,
                                int32_t *idx, float *w, float *logits, void *ws,
                                size_t ws_bytes, void *stream);

/*
 * ds4moe_route_topk_select_bias -- DEVICE.  Routing variant with the bias
 * used for selection only (DeepSeek-style): the k experts with the largest
 * biased logits fp32(x . Wr_e + bias_e) are selected (descending, ties to the
 * lower id, NaN lowest) and w is the softmax of their UNBIASED logits
 * fp32(x . Wr_e), shifted by the largest of them, in double, summed in rank
 * order, rounded once.  Both logits come from one compensated (Dot2) pass
 * and each equals the plain router's value for it.  Same arguments as
 * ds4moe_route_topk, except: bias is required; n_expert <= 256; `logits`
 * (nullable) receives the unbiased logits.  ws must hold the layout's
 * logits region plus one (with `logits`) or two T x n_expert fp32 planes.
 */
ds4moe_status ds4moe_route_topk_select_bias(const uint16_t *x, const float *Wr, const float *bias, int32_t T,
                                            int32_t d_model, int32_t n_expert, int32_t k, int32_t *idx, float *w,
                                            float *logits, void *ws, size_t ws_bytes, void *stream);

/*
 * ds4moe_ffn_decode -- DEVICE.  Routed expert FFN + combine for a decode
 * batch (small T):
 *   for each (t, i): e = idx[t,i];
 *     g = W1[e] x_t, u = W3[e] x_t  (dequant fused into the contraction),
 *     h = bf16(silu(g) * u), silu(z) = z / (1 + exp(-z)),
 *     y_{t,i} = W2[e] h;
 *   out[t] = sum_{i<k} w[t,i] * y_{t,i}, summed in rank order i = 0..k-1.
 * x: bf16 [T, d_model]; idx: int32 [T, k] (from ds4moe_route_topk or the
 * caller); w: fp32 [T, k]; out: fp32 [T, d_model].  Pairs whose expert id is
 * out of range are skipped and flag DS4MOE_EDEVICE in the workspace status.
 * Accuracy: fp32 accumulation over exact integer codes; max |err| <=
 * 2e-3 * max |exact| (tested against a double-precision oracle).
 */
ds4moe_status ds4moe_ffn_decode(const ds4moe_layer *L, const uint16_t *x,
                                const int32_t *idx, const float *w, int32_t T,
                                int32_t k, float *out, void *ws, size_t ws_bytes,
                                void *stream);

/*
 * ds4moe_ffn_prefill -- DEVICE.  Same contract as ds4moe_ffn_decode for a
 * prefill chunk (large T, e.g. the 4096-token chunk of [DS4-1]'s distributed
 * prefill): tokens are bucketed per expert and each expert runs as a grouped
 * GEMM.  On layers where ds4moe_prefill_small_pairs() is n > 0, an expert
 * with 1 .. n pairs of the call streams its weights through the multi-token
 * decode kernels instead (the results agree to the same tolerance).
 */
ds4moe_status ds4moe_ffn_prefill(const ds4moe_layer *L, const uint16_t *x,
                                 const int32_t *idx, const float *w, int32_t T,
                                 int32_t k, float *out, void *ws, size_t ws_bytes,
                                 void *stream);

/*
 * ds4moe_prefill_small_pairs -- HOST.  The pair count at or below which
 * ds4moe_ffn_prefill sends an expert of this layer to the weight-streaming
 * kernels, 0 if it sends every expert to the grouped GEMMs (or takes the
 * decode kernels for the whole layer).  Returns -1 for an invalid layer.
 * Needs the CUDA device (reads its compute capability).
 */
int32_t ds4moe_prefill_small_pairs(const ds4moe_layer *L);

/*
 * ds4moe_moe_decode -- DEVICE.  One decode step of a routed-MoE layer in
 * one call: ds4moe_route_topk followed by ds4moe_ffn_decode, with the same
 * results (idx / w are written as outputs), but scheduled as one chain of
 * kernels.  Up to 32 (token, expert) pairs, the router's last CTA ranks and
 * buckets; beyond that the router grid also converts x for the FFN kernels
 * and the bucketing kernel ranks.  The weighted combine runs inside the
 * down projection.  At T = 1, the router grid writes only the logits and
 * the FFN grids rank the experts themselves.  On all-Q2_K layers with
 * d_model = 2 d_ff, one grid then runs gate/up, SwiGLU, down and the
 * combine.  Same arguments and constraints as those two calls; `ws` must
 * hold ds4moe_workspace_bytes(L, T, k, 0) bytes.
 */
ds4moe_status ds4moe_moe_decode(const ds4moe_layer *L, const uint16_t *x, const float *Wr,
                                const float *bias, int32_t T, int32_t k, float *out,
                                int32_t *idx, float *w, void *ws, size_t ws_bytes,
                                void *stream);

/*
 * ds4moe_residual_norm -- DEVICE.  The step between layers of a decode
 * stack ([DS4-1]: 43 routed-MoE layers): per token t,
 *   x_res[t] += out[t]                 (fp32, one rounding per element),
 *   x_next[t] = bf16_RNE(x_res[t] / sqrt(mean_j x_res[t,j]^2 + eps)),
 * the next layer's input.  With out == NULL only the normalisation runs.
 * x_res / out: fp32 [T, d_model]; x_next: bf16 bit patterns [T, d_model].
 * The normalisation (an RMS norm with unit weight) is this library's reading
 * of the stack: the pages give only x += moe(x), and with their weight
 * distributions an unnormalised residual overflows within a few layers.
 * The sum of squares is an fp32 reduction in a fixed order, so x_next may
 * differ from an exact evaluation by one bf16 ulp where x / rms lies within
 * ~1e-6 relative of a rounding boundary.
 */
#define DS4MOE_STACK_RMS_EPS 1e-6f
ds4moe_status ds4moe_residual_norm(float *x_res, const float *out, uint16_t *x_next,
                                   int32_t T, int32_t d_model, float eps, void *stream);

/*
 * ds4moe_stack_decode -- DEVICE.  One decode step through n_layers routed-MoE
 * layers: x_bf16 = norm(x_res) (ds4moe_residual_norm with out = NULL); then
 * for each layer l, ds4moe_moe_decode(layers[l], x_bf16, Wr[l], bias[l]) ->
 * out and ds4moe_residual_norm(x_res, out, x_bf16).  Exactly the kernels and
 * results of making those calls one by one (no host synchronisation;
 * capturable into a CUDA graph).
 *   layers, Wr, bias: HOST arrays of n_layers entries (layer descriptors and
 *     device pointers; bias[l] may be NULL, bias itself may be NULL);
 *   x_res: fp32 [T, d_model], updated in place;
 *   x_bf16: bf16 [T, d_model] and out: fp32 [T, d_model], scratch that hold
 *     the normalised input after the last layer / its output on return;
 *   idx, w: int32 / fp32 [n_layers][ldk], ldk = T * k rounded up to a
 *     multiple of 4 (so every layer's slice stays 16-byte aligned), each
 *     layer's routing [T, k] at the start of its slice.
 * All layers share one workspace of max_l ds4moe_workspace_bytes(layers[l],
 * T, k, 0) bytes.  Same constraints as ds4moe_moe_decode for every layer.
 */
ds4moe_status ds4moe_stack_decode(const ds4moe_layer *layers, const float *const *Wr,
                                  const float *const *bias, int32_t n_layers, int32_t T,
                                  int32_t k, float eps, float *x_res, uint16_t *x_bf16,
                                  float *out, int32_t *idx, float *w, void *ws,
                                  size_t ws_bytes, void *stream);

/*
 * ds4moe_stream_status -- synchronizes `stream`, then reads and clears the
 * device status word of `ws`.  Returns DS4MOE_OK, the recorded device error
 * (DS4MOE_EDEVICE, DS4MOE_ETIMEOUT) or DS4MOE_ECUDA if the stream itself
 * failed.
 */
ds4moe_status ds4moe_stream_status(void *ws, void *stream);

/*
 * ds4moe_ffn_decode_noalloc -- DEVICE.  The same computation and arguments
 * as ds4moe_ffn_decode, for callers that cannot allocate device memory or
 * hand the library a workspace: an application whose memory is owned by a
 * host framework's own pool or arena (an allocation behind its back breaks
 * its accounting and out-of-memory handling), a per-token decode loop that
 * cannot afford cudaMalloc's implicit device synchronisation and unbounded
 * latency, or a fixed plug-in interface with no place to pass a workspace
 * pointer.  (The paper has no counterpart; this is a property of this
 * library's interface only.)
 *
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  Its scratch is one fixed device array of
 * DS4MOE_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library, which every GPU
 * that loads the library holds until the process exits.  A call whose
 * sizes need more scratch than that (ds4moe_workspace_bytes(L, T, k, 0) >
 * DS4MOE_NOALLOC_SCRATCH_BYTES; e.g. the 4096 x 2048, 256-expert, top-6
 * shape fits up to 16 tokens) returns DS4MOE_ESPACE, prints why on stderr
 * and launches nothing.
 *
 * All calls on a device share that one array and it keeps the previous
 * call's contents; each call clears the part that must start at zero.
 * Calls whose work can overlap on the GPU (different streams, or different
 * host threads without ordering) race on the array: order them on one
 * stream.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  The cached address belongs to the device's primary
 * context: after cudaDeviceReset (or anything else that destroys that
 * context) it is stale, so do not call this entry point again on that
 * device in the same process.
 *
 * status_out: optional device int32; receives this call's device status
 * (0 or DS4MOE_EDEVICE for an expert id out of range), asynchronously.
 */
#define DS4MOE_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
ds4moe_status ds4moe_ffn_decode_noalloc(const ds4moe_layer *L, const uint16_t *x,
                                        const int32_t *idx, const float *w, int32_t T,
                                        int32_t k, float *out, int32_t *status_out,
                                        void *stream);

/*
 * Expert-parallel data plane (no counterpart in the pages' single-process
 * engine; the pages split the model across machines by layer slices,
 * "【#6】ds4.c 분석하기").  With the experts of a layer partitioned across
 * ranks, a rank sends each (token, selected expert) pair's activations to
 * the expert's owner, the owner runs the expert FFN on the pairs it
 * receives (ds4moe_ffn_decode / ds4moe_ffn_prefill with k = 1, weight 1),
 * and the outputs come back to the token's rank for the combine.  The
 * exchange itself is the caller's (e.g. NCCL all-to-all).
 *
 * ds4moe_gather_rows -- DEVICE, asynchronous: dst[j] = x[rows[j]] for
 * j < n; x and dst bf16 [.][d_model], d_model a multiple of 8, both 16-byte
 * aligned; rows int32 [n], each in range (not checked on the device).
 *
 * ds4moe_combine_pairs -- DEVICE, asynchronous: out[t][c] =
 * sum_{i < k} w[t k + i] * y[pos[t k + i]][c] in rank order i (fp32 FMA
 * chain), skipping pairs with pos < 0 (an expert id out of range); y fp32
 * [.][d_model] (the returned expert outputs), pos int32 [T k] (row of pair
 * t k + i in y), w fp32 [T k], out fp32 [T][d_model].
 *
 * Host errors: EINVAL (sizes, alignment, null pointers), ECUDA.
 */
ds4moe_status ds4moe_gather_rows(const uint16_t *x, const int32_t *rows, int32_t n, int32_t d_model,
                                 uint16_t *dst, void *stream);
ds4moe_status ds4moe_combine_pairs(const float *y, const int32_t *pos, const float *w, int32_t T,
                                   int32_t k, int32_t d_model, float *out, void *stream);

/*
 * ds4moe_shared_ffn -- DEVICE, asynchronous on `stream`.  The shared expert
 * of the model ("【#2】ds4.c 해독하기", summary bullets and the README's Model
 * Weights bullets: only the routed experts are quantised; the shared expert,
 * like the projections and the routing, keeps its precision and runs for
 * every token).  The pages give no width, so d_shared is the caller's.
 * Reading: bf16 weights, the routed experts' SwiGLU with h rounded to bf16,
 * output added to the routed combine with weight one.  Per token t:
 *   h[t] = bf16(silu(w1 x[t]) * (w3 x[t])),
 *   out[t] = w2 h[t]            (accumulate = 0)
 *   out[t] = out[t] + w2 h[t]   (accumulate = 1: after ds4moe_moe_decode /
 *                                ds4moe_ffn_decode has written the combine)
 * fp32 accumulation over the exact bf16 products.
 *
 * w1, w3: [d_shared][d_model] bf16 bit patterns, row-major; w2:
 * [d_model][d_shared]; x: [T][d_model] bf16; out: [T][d_model] fp32.  All
 * device pointers 16-byte aligned; d_model and d_shared multiples of 8
 * (d_shared may be 0: out = 0, or unchanged when accumulating).  Up to 8
 * tokens run bandwidth-bound GEMVs on the CUDA cores; more tokens, with
 * d_model a multiple of 256 and d_shared of 128, run tcgen05 GEMMs with TMA
 * operands (other shapes keep the GEMVs).
 *
 * ws: caller-owned workspace of at least ds4moe_shared_workspace_bytes
 * (status word + h [T][d_shared] bf16), initialised once with
 * ds4moe_workspace_init before its first use (as for the routed entry
 * points); ds4moe_stream_status(ws) reports and clears a device-side error
 * (a bounded wait that gave up: DS4MOE_ETIMEOUT; a non-finite h:
 * DS4MOE_EDEVICE).  Host errors:
 * EINVAL (sizes, alignment, null pointers, accumulate not 0 / 1), ESPACE
 * (workspace too small), ECUDA.  Calls sharing a workspace must not overlap.
 */
size_t ds4moe_shared_workspace_bytes(int32_t d_model, int32_t d_shared, int32_t T);
ds4moe_status ds4moe_shared_ffn(const uint16_t *w1, const uint16_t *w3, const uint16_t *w2,
                                int32_t d_model, int32_t d_shared, const uint16_t *x, int32_t T,
                                float *out, int32_t accumulate, void *ws, size_t ws_bytes,
                                void *stream);

/*
 * ds4moe_debug_sync_wait -- HOST, synchronous; a fault-injection hook for
 * tests of failure detection (no counterpart in the pages).  It applies to
 * the single-token fused decode on all-Q2_K layers with d_model = 2 d_ff:
 * ds4moe_moe_decode at T = 1, and each layer of ds4moe_stack_decode.  That
 * path runs the expert FFN as one grid whose CTAs wait on each other.  Every
 * CTA waits until all gate/up units of an expert have published h before
 * its down work on that expert.
 *
 * The hook sets, for later calls on the current device, two things about
 * that wait:
 *   budget_polls  polls before the wait gives up (default 1 << 24, about a
 *                 second);
 *   extra_target  added to the count the wait needs (default 0).
 * With extra_target > 0 the wait cannot succeed.  It gives up after
 * budget_polls polls, records DS4MOE_ETIMEOUT in the workspace status word,
 * and the grid finishes normally, so the CUDA context stays usable.
 * Restore the defaults with (1 << 24, 0).
 *
 * Host errors: EINVAL if budget_polls < 1 or extra_target < 0; ECUDA if the
 * device copy fails.  Call it only while none of this library's kernels is
 * running.
 */
ds4moe_status ds4moe_debug_sync_wait(int32_t budget_polls, int32_t extra_target);

/*
 * Per-kernel timing (tracing aid).  ds4moe_profile_enable(1) clears the
 * totals and, until ds4moe_profile_enable(0), brackets every kernel the
 * library launches with a pair of CUDA events recorded on the launch stream
 * (skipped while that stream is being captured into a CUDA graph).
 * ds4moe_profile_count() synchronizes on the pending events and returns the
 * number of distinct kernels seen; ds4moe_profile_entry(i, ...) returns the
 * i-th kernel's name (static storage, valid until the next enable), total
 * milliseconds and launch count.
 */
ds4moe_status ds4moe_profile_enable(int32_t on);
int32_t ds4moe_profile_count(void);
ds4moe_status ds4moe_profile_entry(int32_t i, const char **name, double *total_ms,
                                   int64_t *launches);

/*
 * Device-side kernel spans (tracing aid).  For each kernel below, while
 * recording is on, every launch adds %globaltimer from the first CTA past its
 * grid-dependency wait to the last warp's exit -- a kernel's duration inside
 * a replayed CUDA graph, where events cannot bracket it -- and counts the
 * launch.
 *
 * ds4moe_profile_span(on, total_ns, launches) writes the totals recorded so
 * far into total_ns[DS4MOE_SPAN_COUNT] / launches[DS4MOE_SPAN_COUNT] (either
 * may be NULL; indexed by ds4moe_span_kernel); with on = 1 or 0 it then
 * clears them and switches recording on or off for later launches on the
 * current device (on = -1: read only).  Call it only while none of this
 * library's kernels is running.  EINVAL for another `on`; ECUDA if a device
 * copy fails.
 */
typedef enum {
  DS4MOE_SPAN_ROUTE = 0,        /* decode router grid: logits (+ top-k, bucketing) */
  DS4MOE_SPAN_FFN_T1 = 1,       /* single-token merged FFN grid, plain blocks */
  DS4MOE_SPAN_FFN_T1R = 2,      /* single-token FFN grid, DS4MOE_Q2_K_R16 */
  DS4MOE_SPAN_GATE_UP_MMA = 3,  /* multi-token decode gate/up + SwiGLU (either kernel) */
  DS4MOE_SPAN_DOWN_MMA = 4,     /* multi-token decode down (either kernel) */
  DS4MOE_SPAN_GATE_UP_TC = 5,   /* prefill tensor-core gate/up + SwiGLU */
  DS4MOE_SPAN_DOWN_TC = 6,      /* prefill tensor-core down */
  DS4MOE_SPAN_SHARED_GATE_UP_TC = 7,  /* shared expert, tensor-core gate/up + SwiGLU */
  DS4MOE_SPAN_SHARED_DOWN_TC = 8,     /* shared expert, tensor-core down */
  DS4MOE_SPAN_GATE_UP_T1 = 9,   /* single-token gate/up + SwiGLU (separate path, Q2_K / Q4_K) */
  DS4MOE_SPAN_DOWN_T1 = 10,     /* single-token down (separate path) */
  DS4MOE_SPAN_COUNT = 11
} ds4moe_span_kernel;
ds4moe_status ds4moe_profile_span(int32_t on, double *total_ns, int64_t *launches);

#ifdef __cplusplus
}
#endif

#endif /* DS4MOE_H */
