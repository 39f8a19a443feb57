"""Pins of the oracle's FP8 (E4M3, per-row scale) weight format against the format's definition:
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest
finite 448, smallest normal 2^-6, subnormals m * 2^-9; rounding to the nearest code, ties to even,
saturating at 448.  The values below are worked out by hand from that definition."""
import numpy as np
import pytest

from oracle.oracle import oracle_lib, quantize_fp8

# (value, code): each follows from value = (1 + m/8) * 2^(e - 7) for e >= 1, m/8 * 2^-6 for e = 0
EXACT = [
    (0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (2.0 ** -6, 0x08),          # smallest normal: e = 1, m = 0
    (2.0 ** -9, 0x01),          # smallest subnormal
    (7 * 2.0 ** -9, 0x07),      # largest subnormal
    (3.0, 0x44),                # 1.5 * 2^1: e = 8, m = 4
    (240.0, 0x77),              # 1.875 * 2^7: e = 14, m = 7
    (256.0, 0x78),              # 2^8: e = 15, m = 0
    (0.3125, 0x2A),             # 1.25 * 2^-2: e = 5, m = 2
]
ROUNDED = [
    (1.0625, 0x38),             # halfway between 1.0 (m = 0) and 1.125 (m = 1): the even code
    (1.1875, 0x3A),             # halfway between 1.125 (m = 1) and 1.25 (m = 2): the even code
    (1.06, 0x38), (1.07, 0x39),  # either side of that midpoint
    (-0.3, 0xAA),               # 0.3 = 1.2 * 2^-2 is nearer 1.25 * 2^-2 than 1.125 * 2^-2
    (2.0 ** -10, 0x00),         # halfway between 0 and the smallest subnormal: 0 is even
    (1.5 * 2.0 ** -9, 0x02),    # halfway between codes 1 and 2: the even code
    (464.0, 0x7E),              # above 448 (the next step would be 480, the NaN code): saturates
    (1.0e6, 0x7E), (-1.0e6, 0xFE),
]


@pytest.fixture(scope="module")
def lib():
    return oracle_lib()


@pytest.mark.parametrize("value,code", EXACT + ROUNDED)
def test_codes_of_hand_computed_values(lib, value, code):
    assert lib.orc_fp8_from_f32(value) == code


@pytest.mark.parametrize("value,code", EXACT)
def test_values_of_codes(lib, value, code):
    assert lib.orc_fp8_to_f32(code) == value


def test_every_finite_code_round_trips_and_codes_increase(lib):
    vals = [lib.orc_fp8_to_f32(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))          # 0x00..0x7E increase
    assert np.isnan(lib.orc_fp8_to_f32(0x7F)) and np.isnan(lib.orc_fp8_to_f32(0xFF))
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert lib.orc_fp8_from_f32(lib.orc_fp8_to_f32(c)) == c
        if c < 0x7F:
            assert lib.orc_fp8_to_f32(c | 0x80) == -lib.orc_fp8_to_f32(c)


def test_midpoints_go_to_the_even_code_and_other_points_to_the_nearest(lib):
    vals = [float(lib.orc_fp8_to_f32(c)) for c in range(0x7F)]
    rng = np.random.default_rng(0)
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2  # exact in fp32: two codes' values have <= 4 significant bits
        assert np.float32(mid) == mid
        assert lib.orc_fp8_from_f32(mid) == (c if c % 2 == 0 else c + 1)
        for x in rng.uniform(vals[c], vals[c + 1], size=4).astype(np.float32):
            got = lib.orc_fp8_from_f32(float(x))
            want = c if abs(float(x) - vals[c]) < abs(vals[c + 1] - float(x)) else c + 1
            if abs(float(x) - vals[c]) != abs(vals[c + 1] - float(x)):
                assert got == want


def test_row_quantization(lib):
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((37, 200)) * 0.02).astype(np.float32)
    w[5] = 0.0                                        # an all-zero row
    bits = (w.view(np.uint32) >> 16).astype(np.uint16)  # truncation gives valid bf16 patterns
    wf = (bits.astype(np.uint32) << 16).view(np.float32)
    q, s = quantize_fp8(bits, lib)
    amax = np.abs(wf).max(axis=1)
    want_s = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    assert np.array_equal(s, want_s)
    assert np.all(q[5] == 0) and s[5] == 1.0
    for r in range(37):
        if r == 5:
            continue
        k = int(np.argmax(np.abs(wf[r])))
        assert q[r, k] in (0x7E, 0xFE)               # the row maximum lands on +-448
        v = np.array([lib.orc_fp8_to_f32(int(c)) for c in q[r]], dtype=np.float64) * float(s[r])
        big = np.abs(wf[r]) >= 2.0 ** -6 * float(s[r])
        rel = np.abs(v[big] - wf[r][big]) / np.abs(wf[r][big])
        assert rel.max() <= 2.0 ** -4 + 1e-6         # half a unit in the last of 3 mantissa bits


def test_fp8_gemv_is_the_scaled_exact_sum(lib):
    rng = np.random.default_rng(2)
    q = rng.integers(0, 256, size=(23, 96), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x10                      # no NaN codes
    s = rng.uniform(1e-4, 1e-2, size=23).astype(np.float32)
    x = rng.standard_normal(96).astype(np.float32)
    y = np.empty(23, dtype=np.float32)
    lib.orc_gemv_fp8(q.ctypes.data, s.ctypes.data, x.ctypes.data, None, 23, 96, y.ctypes.data, 1)
    vals = np.array([lib.orc_fp8_to_f32(c) for c in range(256)], dtype=np.float64)
    want = (vals[q] @ x.astype(np.float64)) * s.astype(np.float64)
    assert np.allclose(y, want.astype(np.float32), rtol=1e-6, atol=0)


def test_fp8_decoder_stays_near_the_bf16_decoder():
    """The FP8 oracle on the tiny shape: every projection takes its own quantized weight (a slot
    mix-up would land far from the bf16 result), within the error of 3-bit mantissas."""
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300 import workloads
    wl = workloads.generate("tiny", seed=0)
    a = OracleDecoder(wl)
    b = OracleDecoder(wl, fp8=True)
    for i in range(4):
        la = a.step(int(wl.tokens[i]), i).astype(np.float64)
        lb = b.step(int(wl.tokens[i]), i).astype(np.float64)
        rel = np.linalg.norm(lb - la) / np.linalg.norm(la)
        assert 1e-4 < rel < 0.1, rel


# ---- the oracle's quantization and FP8 decode step against independent restatements ----
def test_oracle_quantization_and_gemv_match_numpy_restatements(lib):
    from persistent_decode_megakernel_gb300 import workloads
    import oracle_pins as pins
    pins.pin_fp8_quantize_and_gemv(lib, workloads.generate("tiny", seed=0))


def test_fp8_decoder_matches_torch_restatement_on_dequantized_weights(lib):
    from oracle import OracleDecoder
    from persistent_decode_megakernel_gb300 import workloads
    import oracle_pins as pins
    pins.pin_fp8_decoder_vs_torch(lib, workloads.generate("tiny", seed=0), 8, lambda wl: OracleDecoder(wl, fp8=True))
