// Single-token (T = 1) routed-MoE expert FFN over Q2_K weights in the
// 16-row tile order (DS4MOE_Q2_K_R16), and the repacking between that order
// and the plain Q2_K block layout of "【#2】ds4.c 해독하기" (layout table and
// qs packing).  The arithmetic is the model's expert FFN (w1 = gate, w3 = up,
// w2 = down, SwiGLU, combine weighted by the routing weights over the top-k
// experts of "ds4.c 해독하기 1/8").
#include <stdio.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "route.cuh"
#include "span.cuh"
#include "t1r.cuh"

namespace ds4 {

// ================================================================ repacking
// One warp per tile-block (16 rows x one 256-value block column).  Q2_K
// value i of a row: code (qs[32 (i / 128) + i % 32] >> 2 ((i % 128) / 32)) & 3,
// so the 16 values of sub-block s are qs[32 (s / 8) + 16 (s % 2) + v] at bit
// 2 ((s % 8) / 2), v = 0 .. 15.
__device__ __forceinline__ uint32_t q2k_subblock_word(const uint8_t *blk, int s) {
  const uint8_t *q = blk + 16 + 32 * (s >> 3) + 16 * (s & 1);
  const int sh = 2 * ((s & 7) >> 1);
  uint32_t w = 0;
#pragma unroll
  for (int v = 0; v < 16; ++v) w |= (uint32_t)((q[v] >> sh) & 3) << r16_code_bit((uint32_t)v);
  return w;
}

__global__ void k_repack_to_r16(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int64_t ntile,
                                int nb, int64_t rowb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t tbk = wid; tbk < ntile * nb; tbk += nwarp) {
    const int64_t tile = tbk / nb;
    const int b = (int)(tbk % nb);
    const uint8_t *rows = src + tile * 16 * rowb + (int64_t)b * kQ2KBytes;  // row r at + r * rowb
    uint8_t *o = dst + tile * 16 * rowb + (int64_t)b * kR16TileBlock;
    const uint8_t *rg = rows + g * rowb, *rg8 = rows + (g + 8) * rowb;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v;
      v.x = q2k_subblock_word(rg, 8 * h + c);
      v.y = q2k_subblock_word(rg8, 8 * h + c);
      v.z = q2k_subblock_word(rg, 8 * h + c + 4);
      v.w = q2k_subblock_word(rg8, 8 * h + c + 4);
      *reinterpret_cast<uint4 *>(o + 512 * h + 16 * lane) = v;
    }
    uint2 s;
    s.x = rg[2 * c] | (uint32_t)rg[2 * c + 8] << 8 | (uint32_t)rg[2 * c + 1] << 16 | (uint32_t)rg[2 * c + 9] << 24;
    s.y = rg8[2 * c] | (uint32_t)rg8[2 * c + 8] << 8 | (uint32_t)rg8[2 * c + 1] << 16 | (uint32_t)rg8[2 * c + 9] << 24;
    *reinterpret_cast<uint2 *>(o + kR16Scales + 8 * lane) = s;
    if (lane < 16) {
      const uint8_t *r = rows + lane * rowb + 80;
      *reinterpret_cast<uint32_t *>(o + kR16Dmin + 4 * lane) =
          r[0] | (uint32_t)r[1] << 8 | (uint32_t)r[2] << 16 | (uint32_t)r[3] << 24;
    }
  }
}

// The inverse: every byte of the 16 plain blocks gathered from the tile-block.
__global__ void k_repack_from_r16(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int64_t ntile, int nb,
                                  int64_t rowb) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t tbk = wid; tbk < ntile * nb; tbk += nwarp) {
    const int64_t tile = tbk / nb;
    const int b = (int)(tbk % nb);
    const uint8_t *t = src + tile * 16 * rowb + (int64_t)b * kR16TileBlock;
    uint8_t *rows = dst + tile * 16 * rowb + (int64_t)b * kQ2KBytes;
    for (int idx = lane; idx < 16 * kQ2KBytes; idx += 32) {
      const int r = idx / kQ2KBytes, pos = idx % kQ2KBytes, g = r & 7, rr = r >> 3;
      uint32_t byte;
      if (pos < 16) {  // scale byte of sub-block pos
        const int s = pos, c = (s & 7) >> 1;
        const int sel = (s >= 8 ? 1 : 0) + 2 * (s & 1);  // byte of b(2c) | b(2c+8) << 8 | b(2c+1) << 16 | b(2c+9) << 24
        byte = t[kR16Scales + 8 * (4 * g + c) + 4 * rr + sel];
      } else if (pos < 80) {  // qs byte j: codes of sub-blocks 8 (j / 32) + 2 s' + (j % 32) / 16 at bit 2 s'
        const int j = pos - 16, hh = j >> 5, l = j & 31, v = l & 15;
        byte = 0;
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
          const int m = 2 * sp + (l >> 4);  // sub-block within the half
          const int c = m & 3, wsel = (m >= 4 ? 2 : 0) + rr;
          const uint32_t word = *reinterpret_cast<const uint32_t *>(t + 512 * hh + 16 * (4 * g + c) + 4 * wsel);
          byte |= ((word >> r16_code_bit((uint32_t)v)) & 3u) << (2 * sp);
        }
      } else {
        byte = t[kR16Dmin + 4 * r + (pos - 80)];
      }
      rows[r * rowb + pos] = (uint8_t)byte;
    }
  }
}

cudaError_t launch_repack(bool to_r16, const void *src, void *dst, int64_t rows, int64_t cols, cudaStream_t s) {
  const int nb = (int)(cols / 256);
  const int64_t rowb = (int64_t)nb * kQ2KBytes, ntile = rows / 16;
  const int64_t warps = ntile * nb;
  const int64_t blocks64 = (warps + 7) / 8;
  const int blocks = (int)(blocks64 < (int64_t)num_sms() * 64 ? blocks64 : (int64_t)num_sms() * 64);
  ProfScope p("repack", s);
  if (to_r16)
    k_repack_to_r16<<<blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), ntile, nb, rowb);
  else
    k_repack_from_r16<<<blocks, 256, 0, s>>>(static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), ntile, nb,
                                             rowb);
  return cudaGetLastError();
}

// ============================================= single-token FFN over R16
// Poll budget and target offset of the h-ready wait (fault-injection hook of
// ds4moe_debug_sync_wait, set for this kernel by t1r_set_sync_hook).
__device__ int32_t g_t1r_budget = 1 << 24;
__device__ int32_t g_t1r_extra = 0;

constexpr int kT1rMaxConsumers = 16;  // one per 256-value block of d_model <= 4096
constexpr int kT1rPart = 3;           // partial-sum slots between the consumers and the reducer
constexpr uint32_t kT1rHTag = 1u << 16;  // tag of a hidden word written in this call
constexpr int kT1rMaxWarps = kT1rMaxConsumers + 3;

// Order-preserving 32-bit key of a logit: larger logit, larger key; -0 ties
// with +0; NaN ranks below -inf (key 1); 0 marks an absent or already taken
// expert.
__device__ __forceinline__ uint32_t t1r_key(float f) {
  const uint32_t u = f == 0.f ? 0u : __float_as_uint(f);
  if (f != f) return 1u;
  return ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) + 1u;
}

// The k largest of E <= 256 logits (lane holds e = lane + 32 jj in v[jj]),
// in rank order (descending logit, ties to the lower expert id): lane i < k
// receives rank i's logit and expert.  Keys stay in registers: per rank one
// warp max of the keys, then one warp min of the ids holding that key.
__device__ __forceinline__ void t1r_topk(const float (&v)[8], int E, int k, float &my_v, int &my_e) {
  const int lane = threadIdx.x & 31;
  uint32_t key[8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) key[jj] = lane + 32 * jj < E ? t1r_key(v[jj]) : 0u;
  my_v = 0.f;
  my_e = -1;
  for (int i = 0; i < k; ++i) {
    uint32_t lb = key[0];
#pragma unroll
    for (int jj = 1; jj < 8; ++jj) lb = key[jj] > lb ? key[jj] : lb;
    const uint32_t best = __reduce_max_sync(0xffffffffu, lb);
    uint32_t mine = 0xFFFFu;
#pragma unroll
    for (int jj = 7; jj >= 0; --jj)
      if (key[jj] == best) mine = (uint32_t)(lane + 32 * jj);
    const uint32_t be = __reduce_min_sync(0xffffffffu, mine);
    float bv = 0.f;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj)
      if ((uint32_t)(lane + 32 * jj) == be) {
        bv = v[jj];
        key[jj] = 0u;
      }
    bv = __shfl_sync(0xffffffffu, bv, (int)(be & 31u));
    if (lane == i) {
      my_v = bv;
      my_e = (int)be;
    }
  }
}

// Work of one call (T = 1, top-k, all three matrices Q2_K_R16, d_model =
// 2 d_ff): per valid routing slot j, d_ff / 16 gate/up units (16 gate + 16
// up rows, all of K) and d_model / 64 down items (64 rows, all of K).  Unit
// u of all slots goes to CTA u mod G, down item v to CTA G - 1 - v mod G, in
// increasing order; every role of a CTA walks the same list.
struct T1rItem {
  bool gu;
  int j, row0;
};
constexpr int kT1rMaxItems = 64;  // per CTA
__device__ __forceinline__ T1rItem t1r_item(int it, int ng, int G, int ntg, int ntd) {
  T1rItem r;
  r.gu = it < ng;
  if (r.gu) {
    const int u = (int)blockIdx.x + G * it;
    r.j = u / ntg;
    r.row0 = 16 * (u % ntg);
  } else {
    const int v = G - 1 - (int)blockIdx.x + G * (it - ng);
    r.j = v / ntd;
    r.row0 = 64 * (v % ntd);
  }
  return r;
}
// The list packed in shared memory once per CTA: gu << 31 | j << 16 | row0.
__device__ __forceinline__ uint32_t t1r_pack(T1rItem t) {
  return (t.gu ? 0x80000000u : 0u) | ((uint32_t)t.j << 16) | (uint32_t)t.row0;
}
__device__ __forceinline__ T1rItem t1r_unpack(uint32_t p) {
  return T1rItem{(p >> 31) != 0u, (int)((p >> 16) & 0x7FFFu), (int)(p & 0xFFFFu)};
}

// One persistent grid (one CTA per SM) with nbg = d_model / 256 consumer
// warps, a producer warp, a reducer warp and a sync warp.
//  - Routing: the sync warp of every CTA ranks the router's logits (top-k,
//    descending, ties to the lower id; softmax over the selected), or reads
//    the caller's idx / w; slots whose expert id is out of range are skipped
//    (DS4MOE_EDEVICE).  CTA 0 writes the call's routing outputs.
//  - Producer: one bulk copy per 21.5 KB tile (gate/up) or per 43 KB item
//    (down) into a ring of at most three stages (deeper rings put more
//    bytes in flight ahead of the h hand-over's reads and measured slower).
//  - Consumer warp w: K block w of a gate/up unit (gate and up together), or
//    K block w % nbd of two 16-row tiles of a down item; operands of its
//    block in registers (x for gate/up, h of the slot for down); writes the
//    16 + 16 row partials of its block to shared memory.
//  - Reducer: per item, the nbg partials in a fixed order; gate/up: h =
//    bf16(silu(g) * u), stored as a tagged 32-bit word (bf16 | 1 << 16) in a
//    buffer the router grid (or the host path) clears before the call;
//    down: y of the slot, then per 64 output rows a counter; the last of
//    the slots to arrive sums w_i * y_i in rank order.
//  - Sync: the softmax of the selected logits, then for each slot of the
//    CTA's down items, polls (bounded) until every word of its h carries
//    the tag, stages it in shared memory as bf16 and releases the consumers
//    through a per-slot mbarrier.  A word is written once per call, so a
//    reader that sees the tag sees the value: no fence on the hand-over.
// Every wait is bounded: a wait that gives up records DS4MOE_ETIMEOUT and
// the grid still finishes (the CUDA context stays usable).  All CTAs must
// be resident together, as in any persistent grid with one CTA per SM.
__global__ void __launch_bounds__(kT1rMaxWarps * 32, 1) k_ffn_t1r(FfnArgs a, int nstage) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SpanExit span_exit(DS4MOE_SPAN_FFN_T1R);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = lane >> 2, c = lane & 3;
  const int D = a.L.d_model, F = a.L.d_ff, nbg = D / 256, nbd = F / 256;
  const uint32_t sb = 2u * (uint32_t)nbg * kR16TileBlock;  // gate + up tile = four 16-row down tiles
  const uint32_t tile_g = (uint32_t)nbg * kR16TileBlock, tile_d = (uint32_t)nbd * kR16TileBlock;
  const int wprod = nbg, wred = nbg + 1, wsync = nbg + 2;
  uint32_t *hw = reinterpret_cast<uint32_t *>(a.h);  // [k][F] tagged hidden words
  // shared memory: stages | staged h | partials | barriers (every region a
  // multiple of 16 bytes, so the 16-byte accesses to the first three stay aligned)
  uint16_t *s_h = reinterpret_cast<uint16_t *>(smem + (size_t)nstage * sb);    // [2][F] staged h (bf16 bits)
  float *red = reinterpret_cast<float *>(s_h + 2 * (size_t)F);                  // [kT1rPart][nbg][32]
  uint64_t *full = reinterpret_cast<uint64_t *>(red + (size_t)kT1rPart * nbg * 32);
  uint64_t *empty = full + nstage, *pfull = full + 2 * nstage, *pempty = pfull + kT1rPart;
  uint64_t *hfull = pempty + kT1rPart;  // [2]: h of a slot staged in shared memory
  uint64_t *hempty = hfull + 2;          // [2]: every consumer has built its operands from it
  uint64_t *wready = hempty + 2;         // the routing weights are in s_w
  __shared__ int s_e[32];
  __shared__ float s_v[32], s_w[32];
  __shared__ int s_kv;
  __shared__ uint32_t s_items[kT1rMaxItems];
  if (threadIdx.x == 0) {
    for (int st = 0; st < nstage; ++st) {
      ptx::mbar_init(&full[st], 1);
      ptx::mbar_init(&empty[st], nbg);
    }
    for (int pt = 0; pt < kT1rPart; ++pt) {
      ptx::mbar_init(&pfull[pt], nbg);
      ptx::mbar_init(&pempty[pt], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&hfull[b], 1);
      ptx::mbar_init(&hempty[b], nbg);
    }
    ptx::mbar_init(wready, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  R16B B;
  // the call's input: ready before the router grid started, unless that
  // grid forms it (x_late)
  if (!a.x_late && w < nbg) r16_load_b(B, a.x + 256 * w, g, c);
  ptx::pdl_wait();
  span_begin(DS4MOE_SPAN_FFN_T1R);
  ptx::pdl_launch_dependents();
  if (a.x_late && w < nbg) r16_load_b(B, a.x + 256 * w, g, c);
  if (w == wsync) {
    // the experts of the single token: all that the producer needs
    const int k = a.k, E = a.L.n_expert;
    int my_e = -1;
    float my_v = 0.f;
    if (a.lg) {
      float v[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int e = lane + 32 * jj;
        v[jj] = e < E ? __ldcg(a.lg + e) : 0.f;
      }
      t1r_topk(v, E, k, my_v, my_e);
    } else if (lane < k) {
      my_e = __ldcg(a.idx_out + lane);
      my_v = __ldcg(a.w + lane);  // the caller's weight
    }
    const bool ok = lane < k && my_e >= 0 && my_e < E;
    if (lane < k && !ok && blockIdx.x == 0) record_status(a.hdr, DS4MOE_EDEVICE);
    const uint32_t okm = __ballot_sync(0xffffffffu, ok);
    if (lane < k) s_v[lane] = my_v;
    if (ok) s_e[__popc(okm & ((1u << lane) - 1u))] = my_e;
    if (lane == 0) s_kv = __popc(okm);
  }
  __syncthreads();
  const int kv = s_kv, G = gridDim.x;
  const int ntg = F / 16, ntd = D / 64;
  const int Ug = kv * ntg, Ud = kv * ntd;
  const int ng = (int)blockIdx.x < Ug ? (Ug - (int)blockIdx.x + G - 1) / G : 0;
  const int rb = G - 1 - (int)blockIdx.x;
  const int nd = rb < Ud ? (Ud - rb + G - 1) / G : 0;
  const int n = ng + nd;
  if (kv == 0 && blockIdx.x == 0)  // no valid slot: the combine of nothing
    for (int i = threadIdx.x; i < D; i += blockDim.x) a.out[i] = 0.f;
  // this CTA's work list, in order, for every role
  if ((int)threadIdx.x < n) s_items[threadIdx.x] = t1r_pack(t1r_item((int)threadIdx.x, ng, G, ntg, ntd));
  __syncthreads();
  bool timed_out = false;
  if (w == wprod) {
    const uint8_t *gate = static_cast<const uint8_t *>(a.L.gate), *up = static_cast<const uint8_t *>(a.L.up);
    const uint8_t *down = static_cast<const uint8_t *>(a.L.down);
    const int64_t rbg = (int64_t)nbg * kQ2KBytes, rbd = (int64_t)nbd * kQ2KBytes;  // row bytes
    for (int it = 0; it < n; ++it) {
      const int st = it % nstage;
      const uint32_t ph = (uint32_t)(it / nstage) & 1u;
      if (it >= nstage && !ptx::mbar_wait(&empty[st], ph ^ 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      const T1rItem t = t1r_unpack(s_items[it]);
      uint8_t *dst = smem + (size_t)st * sb;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&full[st], sb);
        const int64_t e = s_e[t.j];
        if (t.gu) {
          ptx::bulk_g2s(dst, gate + (e * F + t.row0) * rbg, tile_g, &full[st]);
          ptx::bulk_g2s(dst + tile_g, up + (e * F + t.row0) * rbg, tile_g, &full[st]);
        } else {
          ptx::bulk_g2s(dst, down + (e * D + t.row0) * rbd, sb, &full[st]);
        }
      }
      __syncwarp();
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (lane == 0)
      for (int it = n - nstage > 0 ? n - nstage : 0; it < n; ++it)
        ptx::mbar_wait(&full[it % nstage], (uint32_t)(it / nstage) & 1u, 1u << 20);
  } else if (w < nbg) {
    int cur = -1, q = -1;  // the slot whose h the operands hold; its staging index
    for (int it = 0; it < n; ++it) {
      const int st = it % nstage;
      const uint32_t ph = (uint32_t)(it / nstage) & 1u;
      const T1rItem t = t1r_unpack(s_items[it]);
      if (!t.gu && t.j != cur) {
        // h of slot j, staged in shared memory by the sync warp once every
        // unit has published it (buffer q % 2 of the staging ring)
        ++q;
        if (!ptx::mbar_wait(&hfull[q & 1], (uint32_t)(q >> 1) & 1u)) {
          if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
          timed_out = true;
        }
        r16_load_b<true>(B, s_h + (size_t)(q & 1) * F + 256 * (w % nbd), g, c);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&hempty[q & 1]);
        cur = t.j;
      }
      if (!ptx::mbar_wait(&full[st], ph)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      // gate/up: K block w of the gate and the up tile; down: K block w % nbd
      // of tiles 2 (w / nbd) and + 1 (one call site keeps the loop's code small)
      const uint8_t *sp = smem + (size_t)st * sb;
      const uint8_t *t0 = t.gu ? sp + kR16TileBlock * w
                               : sp + 2u * (uint32_t)(w / nbd) * tile_d + kR16TileBlock * (w % nbd);
      const uint8_t *const tb[2] = {t0, t0 + (t.gu ? tile_g : tile_d)};
      float y[2][2];
      r16_block<2>(tb, g, lane, B, y);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&empty[st]);
      float q[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int r = 0; r < 2; ++r) q[m][r] = r16_quad_sum(y[m][r]);
      // partial slot it % kT1rPart: free once the reducer has read item it - kT1rPart
      const int pt = it % kT1rPart;
      if (it >= kT1rPart && !ptx::mbar_wait(&pempty[pt], ((uint32_t)(it / kT1rPart) & 1u) ^ 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      // partials [16 m + 8 r + g]: gate/up m = gate / up, down m = tile of the pair
      float *rp = red + ((size_t)pt * nbg + w) * 32;
      if (c == 0) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
          for (int r = 0; r < 2; ++r) rp[16 * m + 8 * r + g] = q[m][r];
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pfull[pt]);
    }
  } else if (w == wred) {
    for (int it = 0; it < n; ++it) {
      const int pt = it % kT1rPart;
      const T1rItem t = t1r_unpack(s_items[it]);
      if (!ptx::mbar_wait(&pfull[pt], (uint32_t)(it / kT1rPart) & 1u)) {
        if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
        timed_out = true;
      }
      const float *rr = red + (size_t)pt * nbg * 32 + lane;
      float v0 = 0.f, v1 = 0.f;
      if (t.gu) {
#pragma unroll
        for (int p = 0; p < kT1rMaxConsumers; ++p)
          if (p < nbg) v0 += rr[32 * p];
      } else {
#pragma unroll
        for (int p = 0; p < kT1rMaxConsumers / 2; ++p)
          if (p < nbd) {
            v0 += rr[32 * p];
            v1 += rr[32 * (nbd + p)];
          }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&pempty[pt]);
      if (t.gu) {
        // lanes 0 .. 15: gate rows row0 + lane; lanes 16 .. 31: up rows
        const float us = __shfl_down_sync(0xffffffffu, v0, 16);
        // h as tagged 32-bit words (bf16 | 1 << 16): a reader that sees the
        // tag sees this call's value, with no fence or counter (every call
        // starts the words at zero)
        if (lane < 16)
          hw[(int64_t)t.j * F + t.row0 + lane] = (uint32_t)f32_to_bf16_bits(silu(v0) * us) | kT1rHTag;
      } else {
        // rows row0 + lane (tiles 0, 1) and row0 + 32 + lane (tiles 2, 3)
        float *yp = a.y + (int64_t)t.j * D + t.row0 + lane;
        yp[0] = v0;
        yp[32] = v1;
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          ptx::fence_acq_rel_gpu();
          last = atomicAdd(a.ccnt + t.row0 / 64, 1) == kv - 1;
          if (last) ptx::fence_acq_rel_gpu();  // acquires the other slots' y
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          if (!ptx::mbar_wait(wready, 0u)) {
            if (!timed_out && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);
            timed_out = true;
          }
          float o0 = 0.f, o1 = 0.f;
          for (int j0 = 0; j0 < kv; j0 += 8) {
            float y0[8], y1[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj < kv ? j0 + jj : 0;
              const float *ys = a.y + (int64_t)j * D + t.row0 + lane;
              y0[jj] = __ldcg(ys);
              y1[jj] = __ldcg(ys + 32);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
              if (j0 + jj < kv) {
                o0 = fmaf(s_w[j0 + jj], y0[jj], o0);
                o1 = fmaf(s_w[j0 + jj], y1[jj], o1);
              }
          }
          a.out[t.row0 + lane] = o0;
          a.out[t.row0 + 32 + lane] = o1;
        }
      }
    }
  } else if (w == wsync) {
    {
      // the routing weights (softmax over the selected logits, in double,
      // while the producer's first copies are in flight: only the combine
      // needs them), then the call's routing outputs from CTA 0
      const int k = a.k, E = a.L.n_expert;
      const float v = lane < k ? s_v[lane] : 0.f;
      const float my_w = a.lg ? softmax_selected_warp(v, k) : v;
      int my_e = -1;
      if (lane < k) my_e = a.lg ? s_e[lane] : __ldcg(a.idx_out + lane);
      if (a.lg && blockIdx.x == 0 && lane < k) {
        // ranked experts: every slot is valid and in rank order
        a.idx_out[lane] = my_e;
        const_cast<float *>(a.w)[lane] = my_w;
      }
      const bool ok = lane < k && my_e >= 0 && my_e < E;
      const uint32_t okm = __ballot_sync(0xffffffffu, ok);
      if (ok) s_w[__popc(okm & ((1u << lane) - 1u))] = my_w;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(wready);
    }
    // Then, for each slot of this CTA's down items in order: wait until its
    // staging buffer is free and every word of its h carries this call's
    // tag (all d_ff gate/up units of the slot, from every CTA, have written
    // it), and stage it in shared memory as bf16.
    const uint32_t budget = (uint32_t)g_t1r_budget;
    const uint32_t tag = kT1rHTag * (1u + (uint32_t)g_t1r_extra);  // the hook makes the tag unreachable
    int prev = -1, q = -1;
    for (int tt = 0; tt < nd; ++tt) {
      const int j = t1r_unpack(s_items[ng + tt]).j;
      if (j == prev) continue;
      prev = j;
      ++q;
      if (q >= 2 && lane == 0 && !ptx::mbar_wait(&hempty[q & 1], (uint32_t)((q >> 1) - 1) & 1u))
        record_status(a.hdr, DS4MOE_ETIMEOUT);
      __syncwarp();
      const uint4 *src = reinterpret_cast<const uint4 *>(hw + (int64_t)j * F);  // 4 words per load
      uint2 *dst = reinterpret_cast<uint2 *>(s_h + (size_t)(q & 1) * F);       // 4 bf16 per store
      constexpr int R = kT1rMaxConsumers / 2;  // loads per lane and pass: F / 4 / 32 / 2 <= 8
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t polls = 0;
        for (;;) {
          uint4 v[R];
          bool ok = true;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int i = lane + 32 * (r + R * pass);
            if (i < F / 4) {
              v[r] = __ldcg(src + i);
              ok &= (v[r].x & 0xFFFF0000u) == tag && (v[r].y & 0xFFFF0000u) == tag &&
                    (v[r].z & 0xFFFF0000u) == tag && (v[r].w & 0xFFFF0000u) == tag;
            }
          }
          const bool all = __all_sync(0xffffffffu, ok);
          if (all || ++polls > budget) {
            if (!all && lane == 0) record_status(a.hdr, DS4MOE_ETIMEOUT);  // hand it over anyway
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const int i = lane + 32 * (r + R * pass);
              if (i < F / 4)
                dst[i] = make_uint2((v[r].x & 0xFFFFu) | (v[r].y << 16), (v[r].z & 0xFFFFu) | (v[r].w << 16));
            }
            break;
          }
          __nanosleep(64);
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&hfull[q & 1]);
    }
  }
}

// Shared memory of the grid for nbg consumer warps and nstage stages.
size_t t1r_smem_bytes(int nbg, int nstage) {
  return (size_t)nstage * 2u * (size_t)nbg * kR16TileBlock + (size_t)kT1rPart * nbg * 32 * sizeof(float) +
         sizeof(uint64_t) * (2 * (size_t)nstage + 2 * kT1rPart + 5) +
         2 * sizeof(uint16_t) * 128 * (size_t)nbg;  // two staged h of d_ff values
}

constexpr size_t kT1rSmemMax = 227 * 1024;

bool t1r_ok(const ds4moe_layer &L, int k) {
  const int64_t G = num_sms();
  const int64_t items = ((int64_t)k * (L.d_ff / 16) + G - 1) / G + ((int64_t)k * (L.d_model / 64) + G - 1) / G;
  return items <= kT1rMaxItems && L.q_gate == DS4MOE_Q2_K_R16 && L.q_up == DS4MOE_Q2_K_R16 && L.q_down == DS4MOE_Q2_K_R16 &&
         L.d_model == 2 * L.d_ff && L.d_model % 512 == 0 && L.d_model <= 256 * kT1rMaxConsumers && L.n_expert <= 256 &&
         k <= 32 && t1r_smem_bytes(L.d_model / 256, 2) <= kT1rSmemMax;
}

cudaError_t launch_ffn_t1r(const FfnArgs &a, cudaStream_t s) {
  const int nbg = a.L.d_model / 256;
  int nstage = 3;
  while (nstage > 2 && t1r_smem_bytes(nbg, nstage) > kT1rSmemMax) --nstage;
  const size_t smem = t1r_smem_bytes(nbg, nstage);
  cudaError_t e = cudaFuncSetAttribute(k_ffn_t1r, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope p("ffn_t1r", s);
  return launch_pdl(k_ffn_t1r, dim3(num_sms()), dim3(32 * (nbg + 3)), smem, s, a, nstage);
}

cudaError_t t1r_set_sync_hook(int32_t budget, int32_t extra) {
  cudaError_t e = cudaMemcpyToSymbol(g_t1r_budget, &budget, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_t1r_extra, &extra, sizeof(int32_t));
  return e;
}

cudaError_t span_control_t1r(int on, double *total_ns, int64_t *launches) {
  return span_control_unit(on, total_ns, launches);
}

}  // namespace ds4
