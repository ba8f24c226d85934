/*
 * CPU oracle for the routed-MoE expert FFN over Q4_1 / Q2_K weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It is deliberately plain and slow: one value at a time,
 * fp64 arithmetic, no blocking, no fusion.  It shares no code, header, table
 * or constant generator with the CUDA path.
 *
 * Sources (web pages this oracle is written from):
 *  [DS4-1]  molayo1419.me, "ds4.c 해독하기 1/8" -- DeepSeek V4 Flash shape
 *           (43 layers, 256 routed experts, n_expert_used = 6).
 *  [DS4-2]  molayo1419.me, "【#2】ds4.c 해독하기" -- asymmetric 2-bit
 *           quantisation: the quants.c type-trait table (Q2_K = 256 values in
 *           84 bytes), the ds4q_write_q2_k_block_ref layout table
 *           (scales @0, qs @16, d @80, dmin @82) and the qs_out packing
 *           expression; w1 = gate, w2 = down, w3 = up.
 *  [Q41]    thakicloud.com, "자체 저비트 포맷을 llama.cpp로 옮기기: 복원값이
 *           비트까지 같은 GGUF Q4_1 재부호화" -- sections "Q4_1 블록이 어떻게
 *           생겼나" (the 20-byte block and its nibble order), "무손실이 성립하는
 *           조건 두 개" (the two lossless conditions), "실제로 돌린 코드" (the
 *           block writer), "비트 폭과 그룹 크기는 메타데이터에서만 읽습니다"
 *           (bits and group are explicit), "텐서 이름과 KV 메타데이터" (ne[0]
 *           is the input dimension; row-major [out, in] equals block order).
 *
 * Readings where the pages are silent or truncated: the 4th term of the Q2_K packing expression is the 6-bit shift
 * of value l+96; the low nibble of a Q2_K scale byte is the scale and the
 * high nibble the min; the min is subtracted; router scoring is a plain
 * dot product (+ optional bias) with a softmax over the k selected experts;
 * top-k ties go to the lower expert id and NaN ranks below -inf; the FFN is
 * SwiGLU, silu(gate) * up, with the hidden activation rounded to bf16;
 * expert tensors are experts-major; in the 43-layer stack ([DS4-1]) the
 * residual stream stays fp32 (x += moe(..) with one fp32 rounding) and each
 * layer reads bf16(x / rms(x)), an RMS normalisation with unit weight --
 * without it the stated weight distributions overflow within a few layers;
 * the unquantised shared expert is bf16, the same SwiGLU, added with weight
 * one.
 *
 * Pins: every function here is checked by tests/test_oracle_*.py against
 * facts the pages fix or mathematics fixes (hand-derived golden blocks,
 * single-code bit positions, exact closed forms, brute force, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_EBLOCKER = 2, ORC_EUNSUPPORTED = 3 };
enum { ORC_Q4_1 = 1, ORC_Q2_K = 2, ORC_Q4_K = 4 };

/* ---------------------------------------------------------------- formats */

/* [DS4-2] type-trait table: Q2_K holds 256 values in 84 bytes.
 * [Q41] "Q4_1 블록이 어떻게 생겼나": Q4_1 holds 32 values in 20 bytes. */
int orc_block_values(int qtype) {
  return qtype == ORC_Q4_1 ? 32 : qtype == ORC_Q2_K ? 256 : qtype == ORC_Q4_K ? 256 : 0;
}
int orc_block_bytes(int qtype) {
  return qtype == ORC_Q4_1 ? 20 : qtype == ORC_Q2_K ? 84 : qtype == ORC_Q4_K ? 144 : 0;
}

/* IEEE binary16 -> double, exact (normals, subnormals, inf, NaN). */
double orc_f16(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(1024 + f), e - 25);
  return sign ? -v : v;
}

/* bf16 -> double, exact. */
double orc_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bf16 bit pattern, round to nearest, ties to even, done on the
 * integer significand of the double so that there is exactly one rounding. */
uint16_t orc_round_bf16(double v) {
  uint64_t u;
  memcpy(&u, &v, 8);
  uint16_t s = (uint16_t)((u >> 48) & 0x8000);
  int E = (int)((u >> 52) & 0x7FF);
  uint64_t M = u & ((1ULL << 52) - 1);
  if (E == 0x7FF) return M ? (uint16_t)(s | 0x7FC0) : (uint16_t)(s | 0x7F80);
  if (E == 0) return s; /* double subnormals are far below bf16's range */
  uint64_t sig = (1ULL << 52) | M;     /* value = sig * 2^(E - 1075) */
  int e = E - 1023;                    /* value = 1.x * 2^e */
  /* bf16 keeps 8 significand bits for e >= -126; below that the quantum is
   * fixed at 2^-133. Number of low significand bits to drop: */
  int drop = 52 - 7;
  if (e < -126) drop += (-126 - e);
  if (drop > 60) return s;            /* rounds to zero */
  uint64_t rem = sig & ((1ULL << drop) - 1), half = 1ULL << (drop - 1);
  uint64_t q = sig >> drop;
  if (rem > half || (rem == half && (q & 1))) q++;
  /* q is the significand in units of the quantum 2^(e - 7) (normal) or
   * 2^-133 (subnormal). Re-assemble. */
  if (e < -126) {
    /* q < 2^7 subnormal, q == 2^7 becomes the smallest normal */
    if (q >= 128) return (uint16_t)(s | (1 << 7) | (q - 128));
    return (uint16_t)(s | q);
  }
  if (q == 256) { q = 128; e += 1; }  /* carry into the exponent */
  if (e > 127) return (uint16_t)(s | 0x7F80);
  return (uint16_t)(s | ((e + 127) << 7) | (q - 128));
}

void orc_round_bf16_array(const double *in, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(in[i]);
}

static void put16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }
static uint16_t get16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------------ Q4_1 */
/* [Q41] "Q4_1 블록이 어떻게 생겼나": fp16 d, fp16 m, uint8 qs[16]; value j
 * sits in the low 4 bits of qs[j], value j+16 in the high 4 bits of qs[j];
 * the decoded value is d * q + m. */

int orc_q41_pack(const uint8_t *codes, const uint16_t *d, const uint16_t *m,
                 int64_t nb, uint8_t *out) {
  for (int64_t b = 0; b < nb; ++b) {
    uint8_t *blk = out + 20 * b;
    const uint8_t *q = codes + 32 * b;
    put16(blk + 0, d[b]);
    put16(blk + 2, m[b]);
    for (int j = 0; j < 16; ++j) {
      if (q[j] > 15 || q[j + 16] > 15) return ORC_EBLOCKER;
      blk[4 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
    }
  }
  return ORC_OK;
}

void orc_q41_unpack(const uint8_t *blocks, int64_t nb, uint8_t *codes,
                    uint16_t *d, uint16_t *m) {
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t *blk = blocks + 20 * b;
    d[b] = get16(blk + 0);
    m[b] = get16(blk + 2);
    for (int j = 0; j < 16; ++j) {
      codes[32 * b + j] = blk[4 + j] & 0x0F;
      codes[32 * b + j + 16] = blk[4 + j] >> 4;
    }
  }
}

/* One decoded value: d*q + m. d*q is exact in double (11 x 4 bits) and so is
 * the sum (fp16 exponents span < 53 bits), so the cast is the single
 * rounding of the exact value to fp32. */
static float q41_value(const uint8_t *blk, int j) {
  double d = orc_f16(get16(blk + 0)), m = orc_f16(get16(blk + 2));
  int q = j < 16 ? (blk[4 + j] & 0x0F) : (blk[4 + j - 16] >> 4);
  return (float)(d * (double)q + m);
}

void orc_q41_dequant(const uint8_t *blocks, int64_t nb, float *out) {
  for (int64_t b = 0; b < nb; ++b)
    for (int j = 0; j < 32; ++j) out[32 * b + j] = q41_value(blocks + 20 * b, j);
}

/* [Q41] "무손실이 성립하는 조건 두 개" + "실제로 돌린 코드" + "비트 폭과 그룹
 * 크기는 메타데이터에서만 읽습니다": re-encode asymmetric codes with an
 * explicit bit width and group size into Q4_1.  Lossless iff the group is a
 * multiple of 32 (a group never straddles a block; its (scale, min) pair is
 * copied into group/32 blocks) and the bit width is at most 4 (codes fit a
 * nibble).  Violations, or a code outside the declared bit range, are a
 * BLOCKER: nothing is recomputed, clipped or regrouped. */
int orc_q41_reencode(int bits, int group, const uint8_t *codes,
                     const uint16_t *scale, const uint16_t *mins, int64_t n,
                     uint8_t *out) {
  if (bits < 1 || group < 1 || n < 0) return ORC_EINVAL;
  if (group % 32 != 0 || bits > 4) return ORC_EBLOCKER;
  if (n % group != 0) return ORC_EINVAL;
  int maxc = (1 << bits) - 1;
  for (int64_t i = 0; i < n; ++i)
    if (codes[i] > maxc) return ORC_EBLOCKER;
  int64_t nb = n / 32;
  for (int64_t b = 0; b < nb; ++b) {
    int64_t g = (32 * b) / group; /* the group this block lies in */
    uint8_t *blk = out + 20 * b;
    put16(blk + 0, scale[g]);
    put16(blk + 2, mins[g]);
    for (int j = 0; j < 16; ++j)
      blk[4 + j] = (uint8_t)(codes[32 * b + j] | (codes[32 * b + j + 16] << 4));
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ Q2_K */
/* [DS4-2] layout table: scales[16] at byte 0 (one scale/min nibble pair per
 * 16-value sub-block), qs[64] at byte 16 (256 2-bit codes), fp16 d at 80,
 * fp16 dmin at 82.  Packing expression: for j in {0, 128} and l in 0..31,
 * qs[j/4 + l] = L[j+l] | L[j+l+32] << 2 | L[j+l+64] << 4 | (reading: the
 * truncated 4th term) L[j+l+96] << 6.  Reading: low nibble = scale, high
 * nibble = min, value = d*sc*q - dmin*mn. */

static int q2k_qs_index(int i) { return 32 * (i / 128) + (i % 32); }
static int q2k_qs_shift(int i) { return 2 * ((i % 128) / 32); }

int orc_q2k_pack(const uint8_t *codes, const uint8_t *sc, const uint8_t *mn,
                 const uint16_t *d, const uint16_t *dmin, int64_t nb,
                 uint8_t *out) {
  for (int64_t b = 0; b < nb; ++b) {
    uint8_t *blk = out + 84 * b;
    memset(blk, 0, 84);
    for (int n = 0; n < 16; ++n) {
      uint8_t s = sc[16 * b + n], m = mn[16 * b + n];
      if (s > 15 || m > 15) return ORC_EBLOCKER;
      blk[n] = (uint8_t)(s | (m << 4));
    }
    for (int i = 0; i < 256; ++i) {
      uint8_t q = codes[256 * b + i];
      if (q > 3) return ORC_EBLOCKER;
      blk[16 + q2k_qs_index(i)] |= (uint8_t)(q << q2k_qs_shift(i));
    }
    put16(blk + 80, d[b]);
    put16(blk + 82, dmin[b]);
  }
  return ORC_OK;
}

void orc_q2k_unpack(const uint8_t *blocks, int64_t nb, uint8_t *codes,
                    uint8_t *sc, uint8_t *mn, uint16_t *d, uint16_t *dmin) {
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t *blk = blocks + 84 * b;
    for (int n = 0; n < 16; ++n) {
      sc[16 * b + n] = blk[n] & 0x0F;
      mn[16 * b + n] = blk[n] >> 4;
    }
    for (int i = 0; i < 256; ++i)
      codes[256 * b + i] = (blk[16 + q2k_qs_index(i)] >> q2k_qs_shift(i)) & 3;
    d[b] = get16(blk + 80);
    dmin[b] = get16(blk + 82);
  }
}

/* d*sc*q (<= 17 significand bits) and dmin*mn (<= 15) are exact in double and
 * so is their difference; the cast is the one rounding to fp32. */
static float q2k_value(const uint8_t *blk, int i) {
  double d = orc_f16(get16(blk + 80)), dmin = orc_f16(get16(blk + 82));
  int n = i / 16;
  int sc = blk[n] & 0x0F, mn = blk[n] >> 4;
  int q = (blk[16 + q2k_qs_index(i)] >> q2k_qs_shift(i)) & 3;
  return (float)(d * (double)sc * (double)q - dmin * (double)mn);
}

void orc_q2k_dequant(const uint8_t *blocks, int64_t nb, float *out) {
  for (int64_t b = 0; b < nb; ++b)
    for (int i = 0; i < 256; ++i) out[256 * b + i] = q2k_value(blocks + 84 * b, i);
}

/* ------------------------------------------- Q2_K in the 16-row tile order
 * A storage order of this library's own (the pages give none): the bytes of
 * the Q2_K blocks above, permuted within every 16-row x 256-column
 * tile-block of a matrix (rows % 16 == 0, cols % 256 == 0).  The tile-block
 * of rows 16t .. 16t+15 and block column b keeps the 1344 bytes the plain
 * layout gives those 16 blocks: byte offset (16t) * row_bytes + b * 1344.
 * For row r (r8 = r mod 8, upper = r >= 8) and value i of the block
 * (sub-block s = i / 16, v = i mod 16, half h = s / 8, m = s mod 8):
 *   the code sits in the 32-bit little-endian word at
 *     512 h + 16 (4 r8 + m mod 4) + 4 (2 (m >= 4) + upper),
 *   at bit 16 (v mod 2) + 2 (v / 2);
 *   the scale byte of (r, s) is byte (s >= 8) + 2 (s mod 2) of the word at
 *     1024 + 8 (4 r8 + (s mod 8) / 2) + 4 upper;
 *   row r's d and dmin (block bytes 80 .. 83) are bytes 1280 + 4 r .. +3. */

static int64_t r16_code_word(int r, int i) {
  const int s = i / 16, h = s / 8, m = s % 8;
  return 512 * h + 16 * (4 * (r % 8) + m % 4) + 4 * (2 * (m >= 4) + (r >= 8));
}
static int r16_code_bit(int i) { return 16 * ((i % 16) % 2) + 2 * ((i % 16) / 2); }
static int64_t r16_scale_byte(int r, int s) {
  return 1024 + 8 * (4 * (r % 8) + (s % 8) / 2) + 4 * (r >= 8) + (s >= 8) + 2 * (s % 2);
}

static int r16_shape_ok(int64_t rows, int64_t cols) {
  return rows >= 0 && cols >= 0 && rows % 16 == 0 && cols % 256 == 0;
}

/* Plain Q2_K blocks -> tile order, one value (and one scale byte) at a time. */
int orc_q2k_to_r16(const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst) {
  if (!r16_shape_ok(rows, cols)) return ORC_EINVAL;
  const int64_t nb = cols / 256, rowb = nb * 84;
  memset(dst, 0, (size_t)(rows * rowb));
  for (int64_t t = 0; t < rows / 16; ++t)
    for (int64_t b = 0; b < nb; ++b) {
      uint8_t *tile = dst + 16 * t * rowb + 1344 * b;
      for (int r = 0; r < 16; ++r) {
        const uint8_t *blk = src + (16 * t + r) * rowb + 84 * b;
        for (int i = 0; i < 256; ++i) {
          const int q = (blk[16 + q2k_qs_index(i)] >> q2k_qs_shift(i)) & 3;
          const int64_t wo = r16_code_word(r, i);
          const int bit = r16_code_bit(i);
          tile[wo + bit / 8] |= (uint8_t)(q << (bit % 8));
        }
        for (int n = 0; n < 16; ++n) tile[r16_scale_byte(r, n)] = blk[n];
        for (int j = 0; j < 4; ++j) tile[1280 + 4 * r + j] = blk[80 + j];
      }
    }
  return ORC_OK;
}

/* The inverse: tile order -> plain Q2_K blocks. */
int orc_q2k_from_r16(const uint8_t *src, int64_t rows, int64_t cols, uint8_t *dst) {
  if (!r16_shape_ok(rows, cols)) return ORC_EINVAL;
  const int64_t nb = cols / 256, rowb = nb * 84;
  memset(dst, 0, (size_t)(rows * rowb));
  for (int64_t t = 0; t < rows / 16; ++t)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t *tile = src + 16 * t * rowb + 1344 * b;
      for (int r = 0; r < 16; ++r) {
        uint8_t *blk = dst + (16 * t + r) * rowb + 84 * b;
        for (int i = 0; i < 256; ++i) {
          const int64_t wo = r16_code_word(r, i);
          const int bit = r16_code_bit(i);
          const int q = (tile[wo + bit / 8] >> (bit % 8)) & 3;
          blk[16 + q2k_qs_index(i)] |= (uint8_t)(q << q2k_qs_shift(i));
        }
        for (int n = 0; n < 16; ++n) blk[n] = tile[r16_scale_byte(r, n)];
        for (int j = 0; j < 4; ++j) blk[80 + j] = tile[1280 + 4 * r + j];
      }
    }
  return ORC_OK;
}

/* Value (row, column) of a tile-order matrix read in place: the same value
 * the plain block gives, d * sc * q - dmin * mn rounded once to fp32. */
int orc_r16_dequant(const uint8_t *src, int64_t rows, int64_t cols, float *out) {
  if (!r16_shape_ok(rows, cols)) return ORC_EINVAL;
  const int64_t nb = cols / 256, rowb = nb * 84;
  for (int64_t row = 0; row < rows; ++row)
    for (int64_t col = 0; col < cols; ++col) {
      const int r = (int)(row % 16), i = (int)(col % 256);
      const uint8_t *tile = src + (row - r) * rowb + 1344 * (col / 256);
      const int bit = r16_code_bit(i);
      const int q = (tile[r16_code_word(r, i) + bit / 8] >> (bit % 8)) & 3;
      const int sb = tile[r16_scale_byte(r, i / 16)];
      const double d = orc_f16(get16(tile + 1280 + 4 * r)), dmin = orc_f16(get16(tile + 1282 + 4 * r));
      out[row * cols + col] = (float)(d * (double)(sb & 15) * (double)q - dmin * (double)(sb >> 4));
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------ Q4_K
 * [DS4-2] type-trait table: Q4_K holds 256 values in 144 bytes; the pages
 * give no layout.  Reading (the standard k-quant order, as for Q2_K): fp16 d
 * @0, fp16 dmin @2, scales[12] @4 packing eight 6-bit (scale, min) pairs,
 * qs[128] @16 holding 4-bit codes.  Sub-block j (values 32j .. 32j+31):
 * for j < 4 sc = scales[j] & 63, mn = scales[j + 4] & 63; for j >= 4
 * sc = (scales[j + 4] & 15) | (scales[j - 4] >> 6) << 4,
 * mn = (scales[j + 4] >> 4) | (scales[j] >> 6) << 4.  Value 64 c + l
 * (l < 32) is the low nibble of qs[32 c + l], value 64 c + 32 + l its high
 * nibble.  y = d * sc * q - dmin * mn (one rounding: d * sc * q has at most
 * 21 significant bits, dmin * mn at most 17). */
static void q4k_scale_min(const uint8_t *sc12, int j, int *sc, int *mn) {
  if (j < 4) {
    *sc = sc12[j] & 63;
    *mn = sc12[j + 4] & 63;
  } else {
    *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
    *mn = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
  }
}
static int q4k_qs_index(int i) { return 32 * (i / 64) + (i % 32); }
static int q4k_qs_shift(int i) { return 4 * ((i % 64) / 32); }

int orc_q4k_pack(const uint8_t *codes, const uint8_t *sc, const uint8_t *mn, const uint16_t *d,
                 const uint16_t *dmin, int64_t nb, uint8_t *out) {
  for (int64_t b = 0; b < nb; ++b) {
    uint8_t *blk = out + b * 144;
    memset(blk, 0, 144);
    put16(blk, d[b]);
    put16(blk + 2, dmin[b]);
    uint8_t *s12 = blk + 4;
    for (int j = 0; j < 8; ++j) {
      const int S = sc[b * 8 + j], Mn = mn[b * 8 + j];
      if (S > 63 || Mn > 63) return ORC_EBLOCKER;
      if (j < 4) {
        s12[j] |= (uint8_t)(S & 63);
        s12[j + 4] |= (uint8_t)(Mn & 63);
      } else {
        s12[j + 4] |= (uint8_t)((S & 15) | ((Mn & 15) << 4));
        s12[j - 4] |= (uint8_t)((S >> 4) << 6);
        s12[j] |= (uint8_t)((Mn >> 4) << 6);
      }
    }
    for (int i = 0; i < 256; ++i) {
      const int q = codes[b * 256 + i];
      if (q > 15) return ORC_EBLOCKER;
      blk[16 + q4k_qs_index(i)] |= (uint8_t)(q << q4k_qs_shift(i));
    }
  }
  return ORC_OK;
}

void orc_q4k_unpack(const uint8_t *blocks, int64_t nb, uint8_t *codes, uint8_t *sc, uint8_t *mn, uint16_t *d,
                    uint16_t *dmin) {
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t *blk = blocks + b * 144;
    d[b] = get16(blk);
    dmin[b] = get16(blk + 2);
    for (int j = 0; j < 8; ++j) {
      int S, Mn;
      q4k_scale_min(blk + 4, j, &S, &Mn);
      sc[b * 8 + j] = (uint8_t)S;
      mn[b * 8 + j] = (uint8_t)Mn;
    }
    for (int i = 0; i < 256; ++i) codes[b * 256 + i] = (uint8_t)((blk[16 + q4k_qs_index(i)] >> q4k_qs_shift(i)) & 15);
  }
}

static float q4k_value(const uint8_t *blk, int i) {
  int S, Mn;
  q4k_scale_min(blk + 4, i / 32, &S, &Mn);
  const int q = (blk[16 + q4k_qs_index(i)] >> q4k_qs_shift(i)) & 15;
  /* exact products in double, one rounding to fp32 */
  return (float)(orc_f16(get16(blk)) * S * q - orc_f16(get16(blk + 2)) * Mn);
}

void orc_q4k_dequant(const uint8_t *blocks, int64_t nb, float *out) {
  for (int64_t b = 0; b < nb; ++b)
    for (int i = 0; i < 256; ++i) out[b * 256 + i] = q4k_value(blocks + b * 144, i);
}

int orc_dequant(int qtype, const uint8_t *blocks, int64_t n_values, float *out) {
  int bv = orc_block_values(qtype);
  if (!bv) return ORC_EUNSUPPORTED;
  if (n_values % bv) return ORC_EINVAL;
  if (qtype == ORC_Q4_1) orc_q41_dequant(blocks, n_values / 32, out);
  else if (qtype == ORC_Q2_K) orc_q2k_dequant(blocks, n_values / 256, out);
  else orc_q4k_dequant(blocks, n_values / 256, out);
  return ORC_OK;
}

/* --------------------------------------------------------------- routing */
/* [DS4-1] model shape: 256 routed experts, 6 used per token.  The pages do
 * not print the router; reading: logit[t,e] = sum_j x[t,j] * Wr[e,j]
 * (+ bias[e]), every product exact in double (bf16 x fp32 = 32 bits), the sum
 * accumulated in double in index order and rounded once to fp32. */
void orc_router_logits(const uint16_t *x, const float *Wr, const float *bias,
                       int T, int D, int E, float *logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int j = 0; j < D; ++j)
        acc += orc_bf16(x[(int64_t)t * D + j]) * (double)Wr[(int64_t)e * D + j];
      if (bias) acc += (double)bias[e];
      logits[(int64_t)t * E + e] = (float)acc;
    }
}

/* a ranks before b: larger logit first, NaN below everything, ties -> lower id */
static int ranks_before(float va, int a, float vb, int b) {
  int na = isnan(va), nb = isnan(vb);
  if (na || nb) {
    if (na && nb) return a < b;
    return nb; /* a is a number, b is NaN */
  }
  if (va != vb) return va > vb;
  return a < b;
}

/* Top-k by (logit desc, id asc), then w_i = exp(l_i - m) / sum_j exp(l_j - m)
 * over the k selected, m = the largest selected logit, in double, rounded to
 * fp32.  Selection is k passes of a plain linear scan. */
void orc_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx,
                      float *w) {
  char *taken = (char *)malloc((size_t)E);
  double *ex = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  for (int t = 0; t < T; ++t) {
    const float *l = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int i = 0; i < k; ++i) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
      }
      taken[best] = 1;
      idx[(int64_t)t * k + i] = best;
    }
    double m = (double)l[idx[(int64_t)t * k]];
    double s = 0.0;
    for (int i = 0; i < k; ++i) {
      ex[i] = exp((double)l[idx[(int64_t)t * k + i]] - m);
      s += ex[i];
    }
    for (int i = 0; i < k; ++i) w[(int64_t)t * k + i] = (float)(ex[i] / s);
  }
  free(taken);
  free(ex);
}

/* ------------------------------------------------------------------- FFN */
/* Expert matrices are experts-major: expert e of a [rows x cols] matrix
 * starts at e * rows * row_bytes, row r at + r * row_bytes, and a row holds
 * its cols values as cols / block_values consecutive blocks ([Q41] "텐서
 * 이름과 KV 메타데이터": ne[0] is the input dimension and row-major [out, in]
 * order is block order).  gate = w1 and up = w3 are [d_ff x d_model],
 * down = w2 is [d_model x d_ff] ([DS4-2]). */

static int64_t row_bytes(int qtype, int cols) {
  return (int64_t)cols / orc_block_values(qtype) * orc_block_bytes(qtype);
}

/* out[r - row0] = sum_j W[r, j] * in[j] for r in [row0, row0 + nrows), in
 * double over the exact fp32 weights (one row dequantised at a time). */
int orc_matvec_rows(int qtype, const uint8_t *mat, int rows, int cols, int row0,
                    int nrows, const double *in, double *out) {
  if (!orc_block_values(qtype)) return ORC_EUNSUPPORTED;
  if (cols <= 0 || cols % orc_block_values(qtype) || row0 < 0 || nrows < 0 ||
      row0 + nrows > rows)
    return ORC_EINVAL;
  int64_t rb = row_bytes(qtype, cols);
  float *rowbuf = (float *)malloc(sizeof(float) * (size_t)cols);
  for (int r = row0; r < row0 + nrows; ++r) {
    orc_dequant(qtype, mat + (int64_t)r * rb, cols, rowbuf);
    double acc = 0.0;
    for (int j = 0; j < cols; ++j) acc += (double)rowbuf[j] * in[j];
    out[r - row0] = acc;
  }
  free(rowbuf);
  return ORC_OK;
}

/* One (token, expert) pair: g = Wg x, u = Wu x, h = bf16(silu(g) * u) with
 * silu(z) = z / (1 + exp(-z)), y = Wd h (y kept in double). */
int orc_expert_ffn(int D, int F, int qg, const uint8_t *gate, int qu,
                   const uint8_t *up, int qd, const uint8_t *down, int e,
                   const uint16_t *x, double *y, uint16_t *h_out,
                   double *g_out, double *u_out) {
  if (!orc_block_values(qg) || !orc_block_values(qu) || !orc_block_values(qd))
    return ORC_EUNSUPPORTED;
  if (D <= 0 || F <= 0 || D % orc_block_values(qg) || D % orc_block_values(qu) ||
      F % orc_block_values(qd))
    return ORC_EINVAL;
  double *xin = (double *)malloc(sizeof(double) * (size_t)D);
  double *g = (double *)malloc(sizeof(double) * (size_t)F);
  double *u = (double *)malloc(sizeof(double) * (size_t)F);
  double *h = (double *)malloc(sizeof(double) * (size_t)F);
  for (int j = 0; j < D; ++j) xin[j] = orc_bf16(x[j]);
  orc_matvec_rows(qg, gate + (int64_t)e * F * row_bytes(qg, D), F, D, 0, F, xin, g);
  orc_matvec_rows(qu, up + (int64_t)e * F * row_bytes(qu, D), F, D, 0, F, xin, u);
  for (int r = 0; r < F; ++r) {
    double silu = g[r] / (1.0 + exp(-g[r]));
    uint16_t hb = orc_round_bf16(silu * u[r]);
    if (h_out) h_out[r] = hb;
    h[r] = orc_bf16(hb);
  }
  if (g_out) memcpy(g_out, g, sizeof(double) * (size_t)F);
  if (u_out) memcpy(u_out, u, sizeof(double) * (size_t)F);
  orc_matvec_rows(qd, down + (int64_t)e * D * row_bytes(qd, F), D, F, 0, D, h, y);
  free(xin); free(g); free(u); free(h);
  return ORC_OK;
}

/* Whole layer: out[t, c] = sum_{i<k} w[t,i] * y_{t,i}[c] in double, summed in
 * rank order i = 0..k-1, rounded once to fp32. */
int orc_moe_ffn(int D, int F, int E, int qg, const uint8_t *gate, int qu,
                const uint8_t *up, int qd, const uint8_t *down,
                const uint16_t *x, const int32_t *idx, const float *w, int T,
                int k, float *out) {
  if (!orc_block_values(qg) || !orc_block_values(qu) || !orc_block_values(qd))
    return ORC_EUNSUPPORTED;
  if (D % orc_block_values(qg) || D % orc_block_values(qu) ||
      F % orc_block_values(qd))
    return ORC_EINVAL;
  for (int64_t i = 0; i < (int64_t)T * k; ++i)
    if (idx[i] < 0 || idx[i] >= E) return ORC_EINVAL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    double *acc = (double *)calloc((size_t)D, sizeof(double));
    double *y = (double *)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < k; ++i) {
      orc_expert_ffn(D, F, qg, gate, qu, up, qd, down, idx[(int64_t)t * k + i],
                     x + (int64_t)t * D, y, NULL, NULL, NULL);
      double wi = (double)w[(int64_t)t * k + i];
      for (int c = 0; c < D; ++c) acc[c] += wi * y[c];
    }
    for (int c = 0; c < D; ++c) out[(int64_t)t * D + c] = (float)acc[c];
    free(acc); free(y);
  }
  return ORC_OK;
}

/* ---------------------------------------------------------- shared expert */
/* [DS4-2] (summary bullets and the README's Model Weights bullets): only the
 * routed experts are quantised; the shared expert, like the projections and
 * the routing, keeps its original precision and runs for every token.
 * Reading: its three matrices are bf16 (w1 = gate and w3 = up [Fs x D],
 * w2 = down [D x Fs], row-major), the same SwiGLU as a routed expert with
 * the hidden activation rounded to bf16, and its output is added to the
 * routed combine with weight one.  Per token t:
 *   g = w1 x, u = w3 x (double over the exact bf16 products),
 *   h = bf16(silu(g) * u), y = w2 h (double),
 *   out[t, :] = fp32(base[t, :] + y), or fp32(y) when base is NULL. */
int orc_shared_ffn(int D, int Fs, const uint16_t *w1, const uint16_t *w3, const uint16_t *w2, int T,
                   const uint16_t *x, const float *base, float *out) {
  if (D <= 0 || Fs < 0 || T < 0) return ORC_EINVAL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < T; ++t) {
    double *h = (double *)malloc(sizeof(double) * (size_t)(Fs > 0 ? Fs : 1));
    const uint16_t *xt = x + (int64_t)t * D;
    for (int f = 0; f < Fs; ++f) {
      double g = 0.0, u = 0.0;
      for (int j = 0; j < D; ++j) {
        const double xj = orc_bf16(xt[j]);
        g += orc_bf16(w1[(int64_t)f * D + j]) * xj;
        u += orc_bf16(w3[(int64_t)f * D + j]) * xj;
      }
      const double silu = g / (1.0 + exp(-g));
      h[f] = orc_bf16(orc_round_bf16(silu * u));
    }
    for (int c = 0; c < D; ++c) {
      double y = 0.0;
      for (int f = 0; f < Fs; ++f) y += orc_bf16(w2[(int64_t)c * Fs + f]) * h[f];
      if (base) y += (double)base[(int64_t)t * D + c];
      out[(int64_t)t * D + c] = (float)y;
    }
    free(h);
  }
  return ORC_OK;
}

/* ----------------------------------------------------------- layer stack */
/* [DS4-1] stacks 43 routed-MoE layers.  Reading (see header): the residual
 * x_res stays fp32, x_res += out rounds once to fp32 (done by the caller in
 * fp32), and a layer's input is bf16_RNE(x_res / sqrt(mean(x_res^2) + eps)),
 * evaluated here in fp64 per token. */
void orc_rmsnorm_bf16(const float *x, int64_t T, int64_t D, double eps, uint16_t *out) {
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t j = 0; j < D; ++j) ss += (double)x[t * D + j] * (double)x[t * D + j];
    const double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t j = 0; j < D; ++j) out[t * D + j] = orc_round_bf16((double)x[t * D + j] * r);
  }
}

/* ------------------------------------------------ float-input quantizer
 * [DS4-2], section on the Q2_K block writer: a scale and a minimum are
 * estimated per 16-value sub-block and every value is rounded to a 2-bit
 * code 0..3; with an importance matrix the weighted writer scores the
 * quantisation error with the per-column importance and so changes which
 * scales and codes are chosen.  The pages give neither search, so this is a
 * plain reading (the same one the CUDA path implements, decision by
 * decision in fp32, so that the integer codes can be compared bit for bit):
 *
 *   Q2_K, per sub-block s:  lo = min(0, min x), hi = max x,
 *     a_s = (hi - lo) / 3, b_s = -lo;  d = f16(max a_s / 15),
 *     dmin = f16(max b_s / 15), sc_s = clamp(rint(a_s / d), 0, 15),
 *     mn_s = clamp(rint(b_s / dmin), 0, 15), q = clamp(rint((x + dmin mn) /
 *     (d sc)), 0, 3)  (a zero step gives code 0).
 *   Q4_1, per 32-value block: d = f16((max - min) / 15), m = f16(min),
 *     q = clamp(rint((x - m) / d), 0, 15).
 *   With importance w (one weight per column): every sub-block (Q2_K) tries
 *   (sc, mn) in {sc-1, sc, sc+1} x {mn-1, mn, mn+1} (Q4_1: d and m each
 *   also one fp16 step down and up), codes re-chosen for each candidate,
 *   and keeps the first candidate with the least sum w (x - y)^2 -- the
 *   plain choice is tried first, so the weighted error never grows.
 *
 * All arithmetic is fp32 with one rounding per operation (no contraction);
 * f16() rounds to nearest even.
 */

/* IEEE binary32 -> binary16, round to nearest even (finite inputs). */
uint16_t orc_f32_to_f16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (a > 0x7F800000u ? 0x200u : 0u));
  const int e = (int)(a >> 23) - 127;
  uint32_t mant = (a & 0x7FFFFFu) | (a ? 0x800000u : 0u); /* 24-bit significand */
  if (a == 0) return sign;
  if (e > 15) return (uint16_t)(sign | 0x7C00u); /* overflow -> inf */
  /* target exponent field and how many significand bits to drop */
  int shift;
  uint32_t exp_field;
  if (e >= -14) {
    exp_field = (uint32_t)(e + 15);
    shift = 13;
  } else {
    exp_field = 0;
    shift = 13 + (-14 - e);
    if (shift > 24) return sign; /* below half of the smallest subnormal */
  }
  uint32_t q = mant >> shift;
  const uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) ++q;
  if (exp_field == 0) return (uint16_t)(sign | q); /* may round up into the normal range: same bits */
  /* q holds the implicit bit (0x400); a carry out of the significand (q =
   * 0x800) moves into the exponent field by itself */
  const uint32_t h = (exp_field << 10) + (q - 0x400u);
  if (h >= 0x7C00u) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | h);
}

static float f16f(uint16_t h) { return (float)orc_f16(h); }

/* next representable binary16 above (dir > 0) or below (dir < 0) */
static uint16_t f16_step(uint16_t h, int dir) {
  if ((h & 0x7FFFu) == 0) return dir > 0 ? 0x0001u : 0x8001u;
  const int neg = (h & 0x8000u) != 0;
  return (uint16_t)((dir > 0) != neg ? h + 1u : h - 1u);
}

static int clampi(int v, int lo, int hi) { return v < lo ? lo : v > hi ? hi : v; }

static int code_of(float x, float step, float off, int qmax) {
  /* nearest code for x ~ step * q + off; the clamp is done on the float so
   * that a huge quotient (tiny step) stays well defined */
  if (!(step > 0.0f)) return 0;
  float r = rintf((x - off) / step);
  if (r < 0.0f) r = 0.0f;
  if (r > (float)qmax) r = (float)qmax;
  return (int)r;
}

/* Q2_K: codes and weighted error of one sub-block for scale A = d*sc and
 * offset B = dmin*mn (value = A q - B) */
static float q2k_sub_err(const float *x, const float *w, float A, float B, uint8_t *q) {
  float err = 0.0f;
  for (int i = 0; i < 16; ++i) {
    const int c = code_of(x[i], A, -B, 3);
    if (q) q[i] = (uint8_t)c;
    const float y = A * (float)c - B;
    const float e = x[i] - y;
    err = err + (w ? w[i] : 1.0f) * (e * e);
  }
  return err;
}

static void quantize_q2k_block(const float *x, const float *w, uint8_t *blk) {
  float a[16], b[16];
  float amax = 0.0f, bmax = 0.0f;
  for (int s = 0; s < 16; ++s) {
    float lo = x[16 * s], hi = x[16 * s];
    for (int i = 1; i < 16; ++i) {
      const float v = x[16 * s + i];
      if (v < lo) lo = v;
      if (v > hi) hi = v;
    }
    if (!(lo < 0.0f)) lo = 0.0f;
    a[s] = (hi - lo) / 3.0f;
    b[s] = 0.0f - lo;
    if (a[s] > amax) amax = a[s];
    if (b[s] > bmax) bmax = b[s];
  }
  const uint16_t dh = orc_f32_to_f16(amax / 15.0f), mh = orc_f32_to_f16(bmax / 15.0f);
  const float d = f16f(dh), dmin = f16f(mh);
  uint8_t codes[256], sc[16], mn[16];
  for (int s = 0; s < 16; ++s) {
    int scs = d > 0.0f ? clampi((int)rintf(a[s] / d), 0, 15) : 0;
    int mns = dmin > 0.0f ? clampi((int)rintf(b[s] / dmin), 0, 15) : 0;
    if (w) {
      float best = q2k_sub_err(x + 16 * s, w + 16 * s, d * (float)scs, dmin * (float)mns, NULL);
      int bsc = scs, bmn = mns;
      for (int ds = -1; ds <= 1; ++ds)
        for (int dm = -1; dm <= 1; ++dm) {
          const int cs = scs + ds, cm = mns + dm;
          if ((ds == 0 && dm == 0) || cs < 0 || cs > 15 || cm < 0 || cm > 15) continue;
          const float e = q2k_sub_err(x + 16 * s, w + 16 * s, d * (float)cs, dmin * (float)cm, NULL);
          if (e < best) {
            best = e;
            bsc = cs;
            bmn = cm;
          }
        }
      scs = bsc;
      mns = bmn;
    }
    sc[s] = (uint8_t)scs;
    mn[s] = (uint8_t)mns;
    q2k_sub_err(x + 16 * s, NULL, d * (float)scs, dmin * (float)mns, codes + 16 * s);
  }
  memset(blk, 0, 84);
  for (int s = 0; s < 16; ++s) blk[s] = (uint8_t)(sc[s] | (mn[s] << 4));
  for (int i = 0; i < 256; ++i) blk[16 + q2k_qs_index(i)] |= (uint8_t)(codes[i] << q2k_qs_shift(i));
  put16(blk + 80, dh);
  put16(blk + 82, mh);
}

static float q41_err(const float *x, const float *w, float D, float M, uint8_t *q) {
  float err = 0.0f;
  for (int j = 0; j < 32; ++j) {
    const int c = code_of(x[j], D, M, 15);
    if (q) q[j] = (uint8_t)c;
    const float y = D * (float)c + M;
    const float e = x[j] - y;
    err = err + (w ? w[j] : 1.0f) * (e * e);
  }
  return err;
}

static void quantize_q41_block(const float *x, const float *w, uint8_t *blk) {
  float lo = x[0], hi = x[0];
  for (int j = 1; j < 32; ++j) {
    if (x[j] < lo) lo = x[j];
    if (x[j] > hi) hi = x[j];
  }
  uint16_t dh = orc_f32_to_f16((hi - lo) / 15.0f), mh = orc_f32_to_f16(lo);
  if (w) {
    float best = q41_err(x, w, f16f(dh), f16f(mh), NULL);
    const uint16_t d0 = dh, m0 = mh;
    for (int dd = -1; dd <= 1; ++dd)
      for (int dm = -1; dm <= 1; ++dm) {
        if (dd == 0 && dm == 0) continue;
        const uint16_t cd = dd ? f16_step(d0, dd) : d0, cm = dm ? f16_step(m0, dm) : m0;
        const float D = f16f(cd), M = f16f(cm);
        if (!(D >= 0.0f) || (cd & 0x7C00u) == 0x7C00u || (cm & 0x7C00u) == 0x7C00u) continue;
        const float e = q41_err(x, w, D, M, NULL);
        if (e < best) {
          best = e;
          dh = cd;
          mh = cm;
        }
      }
  }
  uint8_t q[32];
  q41_err(x, NULL, f16f(dh), f16f(mh), q);
  put16(blk, dh);
  put16(blk + 2, mh);
  for (int j = 0; j < 16; ++j) blk[4 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/* x: n_values floats, row-major rows of `cols` values (cols a multiple of
 * the block size); importance: NULL or `cols` weights, one per column. */
int orc_quantize_f32(int qtype, const float *x, const float *importance, int64_t n_values, int64_t cols,
                     uint8_t *out) {
  const int bv = orc_block_values(qtype), bb = orc_block_bytes(qtype);
  if (!bv || n_values < 0 || n_values % bv || (importance && (cols <= 0 || cols % bv || n_values % cols)))
    return ORC_EINVAL;
  for (int64_t i = 0; i < n_values; ++i)
    if (!isfinite(x[i])) return ORC_EINVAL;
  const int64_t nb = n_values / bv;
  for (int64_t b = 0; b < nb; ++b) {
    const float *w = importance ? importance + (b * bv) % cols : NULL;
    if (qtype == ORC_Q2_K) quantize_q2k_block(x + b * bv, w, out + b * bb);
    else quantize_q41_block(x + b * bv, w, out + b * bb);
  }
  return ORC_OK;
}

/* sum over values of w_col * (x - dequant(x))^2, in double (test helper) */
double orc_weighted_sq_error(int qtype, const float *x, const float *importance, int64_t n_values, int64_t cols,
                             const uint8_t *blocks) {
  float *y = (float *)malloc(sizeof(float) * (size_t)(n_values ? n_values : 1));
  if (!y) return -1.0;
  orc_dequant(qtype, blocks, n_values, y);
  double s = 0.0;
  for (int64_t i = 0; i < n_values; ++i) {
    const double e = (double)x[i] - (double)y[i];
    s += (importance ? (double)importance[i % cols] : 1.0) * e * e;
  }
  free(y);
  return s;
}

/* Routing variant with the bias used for selection only (the DeepSeek-style
 * reading of a selection bias): experts are ranked by the biased logit
 * lb = fp32(x . Wr_e + bias_e) (ties to the lower id, NaN lowest), and the
 * weights are the softmax of the selected experts' unbiased logits
 * lu = fp32(x . Wr_e), shifted by their maximum, summed in rank order in
 * double and rounded once. */
void orc_topk_softmax_selbias(const float *lb, const float *lu, int T, int E, int k, int32_t *idx, float *w) {
  char *taken = (char *)malloc((size_t)E);
  double *ex = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  for (int t = 0; t < T; ++t) {
    const float *l = lb + (int64_t)t * E, *u = lu + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int i = 0; i < k; ++i) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
      }
      taken[best] = 1;
      idx[(int64_t)t * k + i] = best;
    }
    double m = -INFINITY;
    for (int i = 0; i < k; ++i) {
      const double v = (double)u[idx[(int64_t)t * k + i]];
      if (v > m) m = v;
    }
    double s = 0.0;
    for (int i = 0; i < k; ++i) {
      ex[i] = exp((double)u[idx[(int64_t)t * k + i]] - m);
      s += ex[i];
    }
    for (int i = 0; i < k; ++i) w[(int64_t)t * k + i] = (float)(ex[i] / s);
  }
  free(taken);
  free(ex);
}
