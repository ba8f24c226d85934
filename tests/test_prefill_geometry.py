"""Index arithmetic of the tensor-core prefill kernels, checked on the host:
the weight-stage tensor-map boxes stay inside their rows and 16-byte aligned,
each covers the bytes its dequant threads read, and the activation rows'
block-sum columns form a one-to-one map into the row's tail.  The formulas
are those of ffn_prefill.cu (stage x coordinates, in-stage offsets, k_xperm's
column maps)."""
import pytest

Q2K_BYTES, Q4K_BYTES, Q41_BYTES = 84, 144, 20


@pytest.mark.parametrize("d_model", [1024, 2048, 4096, 8192])
def test_q2k_gate_up_stage_boxes(d_model):
    nsb = d_model // 256                 # super-blocks per row (d_model % 1024 == 0)
    row = nsb * Q2K_BYTES
    assert row % 16 == 0
    for sb in range(nsb):
        x = (21 * sb) & ~3               # box start in u32 words
        start, end = 4 * x, 4 * x + 96   # 24-word box
        assert start % 16 == 0 and 0 <= start and end <= row
        off = 4 * (sb % 4)               # where the dequant threads find the super-block
        assert start + off == Q2K_BYTES * sb
        assert off + Q2K_BYTES <= 96     # the whole super-block is in the box


@pytest.mark.parametrize("d_model", [1024, 2048, 4096])
def test_q4k_gate_up_stage_boxes(d_model):
    nsb = d_model // 256
    row = nsb * Q4K_BYTES
    for qs in range(2 * nsb):            # half a super-block per stage
        sb, half = qs >> 1, qs & 1
        x = sb * 36 + half * 16          # 20-word box
        start, end = 4 * x, 4 * x + 80
        assert start % 16 == 0 and end <= row
        if half == 0:                    # header (d, dmin, 12 scale bytes) at the box's start
            assert start == Q4K_BYTES * sb
        for j in range(2):               # K-step j of the stage: 32 code bytes at box offset 16 + 32 j
            code0 = Q4K_BYTES * sb + 16 + 32 * (2 * half + j)
            assert start + 16 + 32 * j == code0 and 16 + 32 * j + 32 <= 80


@pytest.mark.parametrize("d_model", [1024, 4096])
def test_q41_gate_up_stage_boxes(d_model):
    row = (d_model // 32) * Q41_BYTES
    for qs in range(d_model // 128):     # four blocks (two K-steps) per stage
        x = qs * 20
        assert (4 * x) % 16 == 0 and 4 * x + 80 <= row


@pytest.mark.parametrize("d_model", [1024, 2048, 4096])
def test_block_sum_columns_are_one_to_one(d_model):
    cols = d_model + d_model // 8        # the gathered row: D values, then the sums
    # 32-value blocks (Q4_1 / Q4_K): block b at D + 64 (b / 32) + 32 (b % 2) + 2 ((b % 32) / 2), lo one on
    seen = set()
    for b in range(d_model // 32):
        c = d_model + 64 * (b >> 5) + 32 * (b & 1) + 2 * ((b & 31) >> 1)
        seen |= {c, c + 1}
    assert len(seen) == 2 * (d_model // 32) and max(seen) < d_model + d_model // 16
    # 16-value sub-blocks (Q2_K): g at D + 64 (g / 32) + 32 ((g % 4) / 2) + 4 ((g % 32) / 4) + 2 (g % 2)
    seen = set()
    for g in range(d_model // 16):
        c = d_model + 64 * (g >> 5) + 32 * ((g & 3) >> 1) + 4 * ((g & 31) >> 2) + 2 * (g & 1)
        seen |= {c, c + 1}
    assert len(seen) == 2 * (d_model // 16) and max(seen) < cols


def test_q2k_minima_columns_match_the_dequant_threads():
    """Q2_K minima step: thread hb writes columns 32 hb + 8 c + 2 i (+1) from
    step kk = 2 c + i / 2, sub-block s = i % 2, i.e. sub-block 4 kk + 2 hb + s
    of the 8-step group -- the column k_xperm gives that sub-block's sum."""
    for hb in range(2):
        for c in range(4):
            for i in range(4):
                kk, s = 2 * c + (i >> 1), i & 1
                col = 32 * hb + 8 * c + 2 * i
                g = 4 * kk + 2 * hb + s                       # sub-block within the group
                assert col == 32 * ((g & 3) >> 1) + 4 * ((g & 31) >> 2) + 2 * (g & 1)
