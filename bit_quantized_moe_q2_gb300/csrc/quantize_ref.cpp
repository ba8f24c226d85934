// ds4moe_quantize_ref: host-side packing of integer codes into Q4_1 / Q2_K /
// Q4_K blocks.  Nothing is recomputed or rounded; the block bytes are a pure
// re-arrangement of the given codes and fp16 scale patterns.
#include <cstring>

#include "../../include/ds4moe.h"

namespace {

inline void store_le16(unsigned char *p, uint16_t v) {
  p[0] = static_cast<unsigned char>(v);
  p[1] = static_cast<unsigned char>(v >> 8);
}

// [Q41] "무손실이 성립하는 조건 두 개" / "실제로 돌린 코드": a group of `group`
// values spans group/32 whole blocks; each block takes the group's fp16
// (scale, min) verbatim as (d, m) and folds codes j and j+16 into the low
// and high nibble of qs[j].
ds4moe_status pack_q41(int bits, int group, const uint8_t *codes, const uint16_t *scale,
                       const uint16_t *mins, int64_t n, unsigned char *out) {
  if (group % 32 != 0 || bits > 4) return DS4MOE_EBLOCKER;
  const unsigned limit = 1u << bits;
  for (int64_t i = 0; i < n; ++i)
    if (codes[i] >= limit) return DS4MOE_EBLOCKER;
  const int64_t blocks_per_group = group / 32;
  for (int64_t g = 0; g < n / group; ++g) {
    for (int64_t bb = 0; bb < blocks_per_group; ++bb) {
      const int64_t blk = g * blocks_per_group + bb;
      unsigned char *o = out + blk * 20;
      store_le16(o, scale[g]);
      store_le16(o + 2, mins[g]);
      const uint8_t *c = codes + blk * 32;
      for (int j = 0; j < 16; ++j) o[4 + j] = static_cast<unsigned char>(c[j] | (c[16 + j] << 4));
    }
  }
  return DS4MOE_OK;
}

// [DS4-2] layout table and qs packing: scales[n] = sc | mn << 4 at byte n,
// qs at byte 16 with byte 32h + l = L[128h+l] | L[128h+l+32] << 2 |
// L[128h+l+64] << 4 | L[128h+l+96] << 6, d at 80, dmin at 82.
ds4moe_status pack_q2k(const uint8_t *codes, const uint16_t *d, const uint16_t *dmin,
                       const uint8_t *sc, const uint8_t *mn, int64_t n, unsigned char *out) {
  for (int64_t i = 0; i < n; ++i)
    if (codes[i] > 3) return DS4MOE_EBLOCKER;
  for (int64_t i = 0; i < n / 16; ++i)
    if (sc[i] > 15 || mn[i] > 15) return DS4MOE_EBLOCKER;
  for (int64_t b = 0; b < n / 256; ++b) {
    unsigned char *o = out + b * 84;
    const uint8_t *L = codes + b * 256;
    for (int s = 0; s < 16; ++s) o[s] = static_cast<unsigned char>(sc[b * 16 + s] | (mn[b * 16 + s] << 4));
    for (int half = 0; half < 2; ++half)
      for (int l = 0; l < 32; ++l) {
        const uint8_t *q = L + 128 * half + l;
        o[16 + 32 * half + l] = static_cast<unsigned char>(q[0] | (q[32] << 2) | (q[64] << 4) | (q[96] << 6));
      }
    store_le16(o + 80, d[b]);
    store_le16(o + 82, dmin[b]);
  }
  return DS4MOE_OK;
}

// Q4_K (the 144-byte k-quant layout of include/ds4moe.h): fp16 d @0, dmin
// @2, eight 6-bit (sc, mn) pairs folded into scales[12] @4 (sub-blocks 0..3
// in the low 6 bits of bytes j and j+4, sub-blocks 4..7 as low / high
// nibbles of bytes j+4 with their top two bits in the top bits of bytes j-4
// and j), codes at 16 + 32c + l (value 64c + l low nibble, 64c + 32 + l high).
ds4moe_status pack_q4k(const uint8_t *codes, const uint16_t *d, const uint16_t *dmin,
                       const uint8_t *sc, const uint8_t *mn, int64_t n, unsigned char *out) {
  for (int64_t i = 0; i < n; ++i)
    if (codes[i] > 15) return DS4MOE_EBLOCKER;
  for (int64_t i = 0; i < n / 32; ++i)
    if (sc[i] > 63 || mn[i] > 63) return DS4MOE_EBLOCKER;
  for (int64_t b = 0; b < n / 256; ++b) {
    unsigned char *o = out + b * 144;
    std::memset(o, 0, 144);
    store_le16(o, d[b]);
    store_le16(o + 2, dmin[b]);
    unsigned char *s12 = o + 4;
    for (int j = 0; j < 8; ++j) {
      const unsigned S = sc[b * 8 + j], Mn = mn[b * 8 + j];
      if (j < 4) {
        s12[j] = static_cast<unsigned char>(s12[j] | S);
        s12[j + 4] = static_cast<unsigned char>(s12[j + 4] | Mn);
      } else {
        s12[j + 4] = static_cast<unsigned char>(s12[j + 4] | (S & 15u) | ((Mn & 15u) << 4));
        s12[j - 4] = static_cast<unsigned char>(s12[j - 4] | ((S >> 4) << 6));
        s12[j] = static_cast<unsigned char>(s12[j] | ((Mn >> 4) << 6));
      }
    }
    const uint8_t *L = codes + b * 256;
    for (int c = 0; c < 4; ++c)
      for (int l = 0; l < 32; ++l)
        o[16 + 32 * c + l] = static_cast<unsigned char>(L[64 * c + l] | (L[64 * c + 32 + l] << 4));
  }
  return DS4MOE_OK;
}

}  // namespace

extern "C" ds4moe_status ds4moe_quantize_ref(int32_t out_type, int32_t bits, int32_t group,
                                             const uint8_t *codes, const uint16_t *scale_f16,
                                             const uint16_t *min_f16, const uint8_t *sub_sc,
                                             const uint8_t *sub_mn, int64_t n_values, void *out_blocks,
                                             size_t out_bytes) {
  if (out_type == DS4MOE_IQ2_XXS) return DS4MOE_EUNSUPPORTED;
  if (out_type != DS4MOE_Q4_1 && out_type != DS4MOE_Q2_K && out_type != DS4MOE_Q4_K) return DS4MOE_EUNSUPPORTED;
  if (n_values < 0 || bits < 1 || group < 1) return DS4MOE_EINVAL;
  if (n_values == 0) return DS4MOE_OK;
  if (!codes || !scale_f16 || !min_f16 || !out_blocks) return DS4MOE_EINVAL;
  unsigned char *out = static_cast<unsigned char *>(out_blocks);
  if (out_type == DS4MOE_Q4_1) {
    if (sub_sc || sub_mn) return DS4MOE_EINVAL;
    if (group % 32 != 0 || bits > 4) return DS4MOE_EBLOCKER;
    if (n_values % group) return DS4MOE_EINVAL;
    if (out_bytes < static_cast<size_t>(n_values / 32) * 20) return DS4MOE_ESPACE;
    return pack_q41(bits, group, codes, scale_f16, min_f16, n_values, out);
  }
  if (out_type == DS4MOE_Q4_K) {
    if (bits != 4 || group != 256 || !sub_sc || !sub_mn) return DS4MOE_EINVAL;
    if (n_values % 256) return DS4MOE_EINVAL;
    if (out_bytes < static_cast<size_t>(n_values / 256) * 144) return DS4MOE_ESPACE;
    return pack_q4k(codes, scale_f16, min_f16, sub_sc, sub_mn, n_values, out);
  }
  if (bits != 2 || group != 256 || !sub_sc || !sub_mn) return DS4MOE_EINVAL;
  if (n_values % 256) return DS4MOE_EINVAL;
  if (out_bytes < static_cast<size_t>(n_values / 256) * 84) return DS4MOE_ESPACE;
  return pack_q2k(codes, scale_f16, min_f16, sub_sc, sub_mn, n_values, out);
}
