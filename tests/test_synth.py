"""The seeded generator: deterministic, counter-based (any slice regenerates
identically), uniform codes, normal values rounded correctly to fp16/bf16."""
import numpy as np

import synth


def test_streams_are_deterministic_and_sliceable():
    k = synth.key(3, 1, synth.T_GATE, 7, synth.F_CODES)
    a = synth.codes(k, 10000, 2)
    assert np.array_equal(a, synth.codes(k, 10000, 2))
    for start, n in ((0, 1), (31, 97), (5000, 4999), (9999, 1)):
        assert np.array_equal(synth.codes(k, n, 2, start=start), a[start:start + n])
    b = synth.abs_normal_f16(k, 300, 0.01)
    assert np.array_equal(synth.abs_normal_f16(k, 100, 0.01, start=150), b[150:250])
    assert synth.key(3, 1, synth.T_GATE, 7, 0) != synth.key(3, 1, synth.T_UP, 7, 0)


def test_codes_are_uniform():
    for bits in (2, 3, 4):
        c = synth.codes(synth.key(0, 0, 0, 0, bits), 1 << 20, bits)
        h = np.bincount(c, minlength=1 << bits)
        assert h.size == 1 << bits
        exp = c.size / h.size
        chi2 = ((h - exp) ** 2 / exp).sum()
        assert chi2 < 3 * h.size + 30


def test_normals_moments_and_rounding():
    k = synth.key(9, 0, synth.T_X, 0, 0)
    x = synth.normal_bf16(k, 200000, 1.0)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(xv.mean()) < 0.01 and abs(xv.std() - 1.0) < 0.01
    h = synth.abs_normal_f16(k, 200000, 0.01)
    hv = h.view(np.float16).astype(np.float64)
    assert hv.min() >= 0 and abs(hv.mean() - 0.01 * np.sqrt(2 / np.pi)) < 2e-4
    # fp16 rounding agrees with numpy's correctly rounded float64 -> float16
    v = np.random.default_rng(0).standard_normal(50000) * 10.0 ** np.random.default_rng(1).integers(-9, 5, 50000)
    ours = np.array([synth._L().synth_round_f16(float(t)) for t in v[:5000]], np.uint16)
    assert np.array_equal(ours, v[:5000].astype(np.float16).view(np.uint16))


def test_workload_recipes():
    w = synth.WORKLOADS[2]
    f = synth.matrix_fields(w, 0, synth.T_GATE, 3, row0=0, nrows=2)
    assert f.qtype == "q4_1" and f.bits == 3 and f.group == 32 and f.codes.max() <= 7
    # min = -4 * scale, exactly
    assert np.array_equal(f.minv.view(np.float16).astype(np.float64),
                          -4 * f.scale.view(np.float16).astype(np.float64))
    w0 = synth.WORKLOADS[0]
    f0 = synth.matrix_fields(w0, 0, synth.T_UP, 1, row0=0, nrows=2)
    assert f0.bits == 4 and np.array_equal(f0.minv.view(np.float16).astype(np.float64),
                                           -8 * f0.scale.view(np.float16).astype(np.float64))
    fd = synth.matrix_fields(w0, 0, synth.T_DOWN, 1, row0=0, nrows=2)
    assert fd.qtype == "q2_k" and fd.codes.max() <= 3 and fd.sc.max() <= 15 and fd.mn.max() <= 15
    assert synth.matrix_shape(w0, synth.T_DOWN) == (4096, 2048)
