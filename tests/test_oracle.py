"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one step of the oracle against something independent:
numpy's float16 casts (a library routine), hand-packed words, hand-derived
worked examples, closed forms, brute-force sums, and invariants of the
method (trivial g_idx == no g_idx; act-order is a row permutation).  A few
tests plant a plausible mistake (a dropped "+1", a reversed nibble order) in
a copy of the oracle's inputs and check that the tolerance catches it.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def pack_rows(q: np.ndarray) -> np.ndarray:
    """Test-side packer: q [K, N] codes -> [K/8, N] int32, code 8i+r in bits 4r..4r+3."""
    K, N = q.shape
    words = np.zeros((K // 8, N), np.uint64)
    for r in range(8):
        words |= q[r::8, :].astype(np.uint64) << np.uint64(4 * r)
    return words.astype(np.uint32).view(np.int32)


def pack_cols(z: np.ndarray) -> np.ndarray:
    """Test-side packer: z [G, N] codes -> [G, N/8] int32, code 8j+r in bits 4r..4r+3."""
    G, N = z.shape
    words = np.zeros((G, N // 8), np.uint64)
    for r in range(8):
        words |= z[:, r::8].astype(np.uint64) << np.uint64(4 * r)
    return words.astype(np.uint32).view(np.int32)


def h(v) -> np.ndarray:
    return np.asarray(v, np.float16)


# ------------------------------------------------------------------- fp16

def test_half_to_double_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.half_bits_to_f64(bits)
    lib = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(lib[~nan]))


def test_double_to_half_matches_numpy_rounding():
    g = np.random.default_rng(1234)
    vals = [g.standard_normal(200000) * 10.0 ** g.uniform(-9, 5, 200000)]
    # every fp16 value, the midpoints between neighbours (ties) and points
    # just either side of them
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    finite = np.sort(allh[np.isfinite(allh)])
    mid = (finite[:-1] + finite[1:]) / 2.0
    vals += [finite, mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)]
    # overflow edge and tiny subnormals
    vals.append(np.array([65504.0, 65519.0, 65519.999, 65520.0, 65536.0, 1e6, -65520.0,
                          2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26,
                          2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 0.0, -0.0, np.inf, -np.inf]))
    v = np.concatenate(vals)
    mine = oracle.f64_to_half_bits(v)
    with np.errstate(over="ignore"):
        lib = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(mine, lib)


def test_double_to_half_nan():
    out = oracle.f64_to_half_bits(np.array([np.nan]))
    assert np.isnan(out.view(np.float16)[0])


# ----------------------------------------------------------------- unpack

def _golden_words():
    rows = []
    with open(os.path.join(GOLDEN, "unpack_words.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), [int(p) for p in parts[1:]]))
    return rows


@pytest.mark.parametrize("word,codes", _golden_words())
def test_unpack_hand_packed_words(word, codes):
    w = np.array([word], np.uint32).view(np.int32)
    # qweight: one word per column, the eight codes run down K
    q = oracle.unpack_qweight(np.tile(w, (1, 8)).reshape(1, 8), 8, 8)
    assert q[:, 0].tolist() == codes
    assert (q == q[:, :1]).all()
    # qzeros: the eight codes run along N
    z = oracle.unpack_qzeros(w.reshape(1, 1), 1, 8)
    assert z[0].tolist() == codes


def test_unpack_round_trip_all_values_all_positions():
    g = np.random.default_rng(5)
    K, N, G = 64, 48, 4
    q = g.integers(0, 16, size=(K, N)).astype(np.uint8)
    q[:16, 0] = np.arange(16)            # every value ...
    for r in range(8):                   # ... at every nibble position
        q[r::8, 1] = (np.arange(K // 8) + r) % 16
    z = g.integers(0, 16, size=(G, N)).astype(np.uint8)
    z[0, :16] = np.arange(16)
    assert np.array_equal(oracle.unpack_qweight(pack_rows(q), K, N), q)
    assert np.array_equal(oracle.unpack_qzeros(pack_cols(z), G, N), z)


# --------------------------------------------------------------- bf16

def test_bf16_to_double_exhaustive():
    """Every bf16 pattern against numpy: the float32 whose upper half it is."""
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):                # signalling NaN patterns
        expect = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = oracle.bf16_bits_to_f64(bits.astype(np.uint16))
    nan = np.isnan(expect)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], expect[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(expect[~nan]))


def test_bf16_hand_values():
    b = np.array([0x3F80, 0xC020, 0x0001, 0x7F7F, 0x4000, 0x3C00], np.uint16)
    assert oracle.bf16_bits_to_f64(b).tolist() == [1.0, -2.5, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 2.0,
                                                    2.0 ** -7]


def test_bf16_tolerance_covers_output_rounding_only():
    """The bf16 bound admits y_ref rounded to bf16 and rejects an error of a
    whole bf16 unit in the last place on a value just above a power of two."""
    y_ref = np.array([[1.0 + 2 ** -8 * 0.999, 3.0]])
    x = np.zeros((1, 64), np.uint16)                   # x = 0: only the relative term is left
    w16 = np.zeros((64, 2), np.uint16)
    tol = oracle.tolerance_rows_bf16(x, w16, y_ref, 64)
    assert (np.abs(np.array([[1.0, 3.0]]) - y_ref) <= tol).all()
    assert not (np.abs(np.array([[1.0 + 2 ** -7 + 2 ** -6, 3.0]]) - y_ref) <= tol).all()


# ------------------------------------------------------------- 8-bit

def pack_rows8(q: np.ndarray) -> np.ndarray:
    """Test-side packer: 8-bit q [K, N] -> [K/4, N] int32, code 4i+r in bits 8r..8r+7."""
    K, N = q.shape
    words = np.zeros((K // 4, N), np.uint64)
    for r in range(4):
        words |= q[r::4, :].astype(np.uint64) << np.uint64(8 * r)
    return words.astype(np.uint32).view(np.int32)


def pack_cols8(z: np.ndarray) -> np.ndarray:
    G, N = z.shape
    words = np.zeros((G, N // 4), np.uint64)
    for r in range(4):
        words |= z[:, r::4].astype(np.uint64) << np.uint64(8 * r)
    return words.astype(np.uint32).view(np.int32)


@pytest.mark.parametrize("word,codes", [
    (0x04030201, [1, 2, 3, 4]),
    (0xFF80007F, [0x7F, 0x00, 0x80, 0xFF]),       # a negative int32: the top byte is 255
    (0x00000000, [0, 0, 0, 0]),
    (0xF00F0FF0, [0xF0, 0x0F, 0x0F, 0xF0]),
])
def test_unpack8_hand_packed_words(word, codes):
    w = np.array([word], np.uint32).view(np.int32)
    q = oracle.unpack_qweight8(np.tile(w, (1, 4)).reshape(1, 4), 4, 4)
    assert q[:, 0].tolist() == codes and (q == q[:, :1]).all()
    z = oracle.unpack_qzeros8(w.reshape(1, 1), 1, 4)
    assert z[0].tolist() == codes


def test_unpack8_round_trip_all_byte_values():
    g = np.random.default_rng(15)
    K, N, G = 1024, 16, 4
    q = g.integers(0, 256, size=(K, N)).astype(np.uint8)
    for r in range(4):                   # every value at every byte position
        q[r::4, 0] = (np.arange(K // 4) + r) % 256
    z = g.integers(0, 256, size=(G, N)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_qweight8(pack_rows8(q), K, N), q)
    assert np.array_equal(oracle.unpack_qzeros8(pack_cols8(z), G, N), z)


def test_8bit_closed_forms():
    """Every code 200, stored zero 100, unit scale: w = 200 - 101 (GPTQ) or
    200 - 100 (GPTQ_V2); codes 255 against zero 255: -1 / 0."""
    K, N = 32, 8
    for code, zero in ((200, 100), (255, 255), (0, 255)):
        qw = pack_rows8(np.full((K, N), code, np.uint8))
        qz = pack_cols8(np.full((1, N), zero, np.uint8))
        s = np.ones((1, N), np.float16)
        for zo in (1, 0):
            dq = oracle.dequantize_layer(qw, qz, s, None, K, N, -1, zero_offset=zo, bits=8)
            assert (dq.w64 == float(code - zero - zo)).all()
            assert (dq.w16.view(np.float16).astype(np.float64) == float(code - zero - zo)).all()


def test_8bit_uneven_groups_brute_force_tiny():
    """A 16 x 8 layer with 8-bit codes and groups of 5 and 11 rows, element by
    element from the packing (byte k % 4 of word k / 4; byte n % 4 of zero
    word n / 4), rounded by numpy's float16 cast."""
    g = np.random.default_rng(17)
    K, N, gs = 16, 8, 8
    qw = g.integers(0, 2**32, size=(K // 4, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    qz = g.integers(0, 2**32, size=(2, N // 4), dtype=np.uint64).astype(np.uint32).view(np.int32)
    s = g.uniform(0.0002, 0.002, size=(2, N)).astype(np.float16)
    gi = np.array([0] * 5 + [1] * 11, np.int32)[g.permutation(K)]
    dq = oracle.dequantize_layer(qw, qz, s, gi, K, N, gs, bits=8)
    for k in range(K):
        for n in range(N):
            q = (int(qw.view(np.uint32)[k // 4, n]) >> (8 * (k % 4))) & 0xFF
            z = (int(qz.view(np.uint32)[gi[k], n // 4]) >> (8 * (n % 4))) & 0xFF
            w = float(s[gi[k], n]) * (q - z - 1)
            assert dq.q[k, n] == q and dq.z[gi[k], n] == z
            assert dq.w16[k, n] == np.float16(w).view(np.uint16)


def test_8bit_layer_with_nibble_codes_equals_4bit_layer():
    """Codes and zeros below 16 packed as an 8-bit and as a 4-bit checkpoint
    describe the same weights: both oracle routes agree bit for bit."""
    g = np.random.default_rng(16)
    K, N, gs = 256, 32, 64
    q = g.integers(0, 16, size=(K, N)).astype(np.uint8)
    z = g.integers(0, 16, size=(K // gs, N)).astype(np.uint8)
    s = g.uniform(0.002, 0.02, size=(K // gs, N)).astype(np.float16)
    gi = (g.permutation(K) // gs).astype(np.int32)
    d4 = oracle.dequantize_layer(pack_rows(q), pack_cols(z), s, gi, K, N, gs)
    d8 = oracle.dequantize_layer(pack_rows8(q), pack_cols8(z), s, gi, K, N, gs, bits=8)
    assert np.array_equal(d4.w16, d8.w16) and np.array_equal(d4.q, d8.q) and np.array_equal(d4.z, d8.z)


# ----------------------------------------------------------- group map

def test_row_groups_trivial_and_errors():
    gr, G = oracle.row_groups(None, 256, 64)
    assert G == 4 and np.array_equal(gr, np.arange(256) // 64)
    gr, G = oracle.row_groups(None, 256, -1)
    assert G == 1 and not gr.any()
    with pytest.raises(ValueError):
        oracle.row_groups(None, 256, 48)          # does not divide K
    with pytest.raises(ValueError):
        oracle.row_groups(None, 256, 0)
    bad = np.arange(256, dtype=np.int32) // 64
    bad[7] = 4
    with pytest.raises(ValueError):
        oracle.row_groups(bad, 256, 64)
    bad[7] = -1
    with pytest.raises(ValueError):
        oracle.row_groups(bad, 256, 64)


# ---------------------------------------------------------------- dequant

def test_dequant_unit_scale_is_exact_integer():
    g = np.random.default_rng(7)
    K, N = 32, 16
    q = g.integers(0, 16, (K, N)).astype(np.uint8)
    z = g.integers(0, 16, (1, N)).astype(np.uint8)
    s = np.ones((1, N), np.float16).view(np.uint16)
    w16, w64 = oracle.dequant(q, z, s, np.zeros(K, np.int32), K, N)
    expect = q.astype(np.int64) - z.astype(np.int64) - 1
    assert np.array_equal(w64, expect.astype(np.float64))
    assert np.array_equal(w16.view(np.float16).astype(np.float64), expect.astype(np.float64))


def test_dequant_power_of_two_scale_and_numpy_cast():
    g = np.random.default_rng(8)
    K, N, G = 64, 32, 2
    q = g.integers(0, 16, (K, N)).astype(np.uint8)
    z = g.integers(0, 16, (G, N)).astype(np.uint8)
    gr = (np.arange(K) // 32).astype(np.int32)
    # powers of two scale exactly
    s2 = (2.0 ** g.integers(-20, 3, (G, N))).astype(np.float16)
    w16, w64 = oracle.dequant(q, z, s2.view(np.uint16), gr, K, N)
    iq = q.astype(np.float64) - z[gr].astype(np.float64) - 1
    assert np.array_equal(w64, s2.astype(np.float64)[gr] * iq)
    # arbitrary fp16 scales: one rounding of the exact product, as numpy casts it
    s = g.uniform(1e-4, 3.0, (G, N)).astype(np.float16)
    w16, w64 = oracle.dequant(q, z, s.view(np.uint16), gr, K, N)
    exact = s.astype(np.float64)[gr] * iq
    assert np.array_equal(w64, exact)
    assert np.array_equal(w16, exact.astype(np.float16).view(np.uint16))


# ------------------------------------------------------- GPTQ_V2 zeros

def test_v2_zero_convention_closed_forms():
    """GPTQ_V2 ("Inference Backends", "Concepts": a checkpoint format distinct
    from GPTQ), read as the same layout with the effective zero stored as is:
    codes equal to the stored zero dequantize to exactly 0 (under GPTQ they
    give -s), and with unit scales w is the integer q - z."""
    g = np.random.default_rng(70)
    K, N = 64, 24
    z = g.integers(0, 16, (1, N)).astype(np.uint8)
    q = np.repeat(z, K, axis=0)
    s = g.uniform(1e-3, 2.0, (1, N)).astype(np.float16)
    gr = np.zeros(K, np.int32)
    w16, w64 = oracle.dequant(q, z, s.view(np.uint16), gr, K, N, zero_offset=0)
    assert np.all(w64 == 0.0) and np.all(w16.view(np.float16) == 0)
    w16, w64 = oracle.dequant(q, z, s.view(np.uint16), gr, K, N, zero_offset=1)
    assert np.array_equal(w64, np.repeat(-s.astype(np.float64), K, axis=0))
    q = g.integers(0, 16, (K, N)).astype(np.uint8)
    one = np.ones((1, N), np.float16).view(np.uint16)
    w16, w64 = oracle.dequant(q, z, one, gr, K, N, zero_offset=0)
    assert np.array_equal(w64, (q.astype(np.int64) - z.astype(np.int64)).astype(np.float64))


def test_v2_layer_equals_v1_layer_with_zeros_minus_one():
    """Through the packed checkpoint: a GPTQ_V2 layer whose stored zeros are
    z + 1 is the GPTQ layer with stored zeros z (z <= 14), bit for bit."""
    g = np.random.default_rng(71)
    K, N, gs = 256, 64, 64
    G = K // gs
    q = g.integers(0, 16, (K, N)).astype(np.uint8)
    z = g.integers(0, 15, (G, N)).astype(np.uint8)
    scales = g.uniform(0.002, 0.02, (G, N)).astype(np.float16)
    v1 = oracle.dequantize_layer(pack_rows(q), pack_cols(z), scales, None, K, N, gs, zero_offset=1)
    v2 = oracle.dequantize_layer(pack_rows(q), pack_cols(z + 1), scales, None, K, N, gs, zero_offset=0)
    assert np.array_equal(v1.w16, v2.w16) and np.array_equal(v1.w64, v2.w64)


# ------------------------------------------------------------- packing

def test_pack_round_trips_exact_weights():
    """Weights that are exactly s * (q - z) (power-of-two scales) pack back to
    q, with the GPTQ zero stored as z - 1 and the GPTQ_V2 zero as z; the
    layout matches an independent packer; dequantizing gives the weights."""
    g = np.random.default_rng(80)
    K, N, gs = 128, 64, 32
    G = K // gs
    q = g.integers(0, 16, (K, N)).astype(np.int64)
    z = g.integers(1, 16, (G, N)).astype(np.int64)
    s = (2.0 ** g.integers(-12, -2, (G, N))).astype(np.float16)
    gr = np.arange(K) // gs
    w = (s.astype(np.float64)[gr] * (q - z[gr])).astype(np.float16)
    assert np.array_equal(w.astype(np.float64), s.astype(np.float64)[gr] * (q - z[gr]))
    for off in (1, 0):
        qw, qz = oracle.pack(w.view(np.uint16), s.view(np.uint16), z.astype(np.int32), None, K, N, gs, off)
        assert np.array_equal(qw, pack_rows(q.astype(np.uint8)))
        assert np.array_equal(qz, pack_cols((z - off).astype(np.uint8)))
        dq = oracle.dequantize_layer(qw, qz, s, None, K, N, gs, zero_offset=off)
        assert np.array_equal(dq.w16, w.view(np.uint16))


def test_pack_rounding_clamping_and_symmetric_zero():
    """Hand-worked codes, unit scale: ties go to even (2.5 -> 2, 3.5 -> 4,
    -0.5 -> 0), out-of-range quotients clamp to 0 and 15, no zeros means
    the symmetric zero 8 (stored 7 for GPTQ)."""
    K, N = 8, 8
    vals = np.array([2.5, 3.5, -0.5, 0.49, -100.0, 100.0, 6.5, -7.5], np.float16)
    w = np.tile(vals[:, None], (1, N))
    one = np.ones((1, N), np.float16)
    qw, qz = oracle.pack(w.view(np.uint16), one.view(np.uint16), None, None, K, N, -1, 1)
    codes = [(int(qw[0, 0]) >> (4 * r)) & 0xF for r in range(8)]
    assert codes == [8 + 2, 8 + 4, 8 + 0, 8 + 0, 0, 15, 8 + 6, 8 - 8]
    assert all(((int(qz[0, 0]) & 0xFFFFFFFF) >> (4 * r)) & 0xF == 7 for r in range(8))


def test_pack_follows_act_order_groups():
    """With an act-order g_idx each row takes the scale and zero of its own
    group: packing through g_idx equals packing each row against its group."""
    g = np.random.default_rng(81)
    K, N, gs = 64, 16, 16
    G = K // gs
    g_idx = (g.permutation(K) // gs).astype(np.int32)
    s = g.uniform(0.01, 0.1, (G, N)).astype(np.float16)
    z = g.integers(0, 16, (G, N)).astype(np.int32)
    w = g.normal(0, 0.3, (K, N)).astype(np.float16)
    qw, _ = oracle.pack(w.view(np.uint16), s.view(np.uint16), z, g_idx, K, N, gs, 0)
    q = oracle.unpack_qweight(qw, K, N).astype(np.int64)
    sf = s.astype(np.float32)[g_idx]
    expect = np.clip(np.rint(w.astype(np.float32) / sf) + z[g_idx], 0, 15)
    assert np.array_equal(q, expect.astype(np.int64))


# --------------------------------------------------------------- products

def test_linear_matches_numpy_matmul():
    g = np.random.default_rng(9)
    M, K, N = 5, 96, 40
    x = g.standard_normal((M, K))
    w = g.standard_normal((K, N))
    b = g.standard_normal(N)
    y = oracle.linear_f64(x, w, b, nthreads=3)
    ref = x @ w + b
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(x).sum() * np.abs(w).max())


def test_linear_brute_force_tiny():
    g = np.random.default_rng(10)
    M, K, N = 3, 16, 8
    x = g.standard_normal((M, K))
    w = g.standard_normal((K, N))
    b = g.standard_normal(N)
    y = oracle.linear_f64(x, w, b, nthreads=2)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):            # ascending k, then bias
                acc += x[m, k] * w[k, n]
            acc += b[n]
            assert y[m, n] == acc         # same order, so bitwise equal


def test_one_hot_x_selects_dequantized_row():
    layer = synthetic.make_layer(128, 64, 32, bias=True, key=(11,))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, None, 128, 64, 32)
    for k in (0, 1, 31, 32, 77, 127):
        x = np.zeros((1, 128), np.float16)
        x[0, k] = 1.0
        y = oracle.reference_output(x, dq, layer.bias)
        expect = dq.w16.view(np.float16).astype(np.float64)[k] + layer.bias.astype(np.float64)
        assert np.array_equal(y[0], expect)


def test_closed_form_all_equal_codes():
    K, N, c, z0 = 256, 16, 11, 4
    q = np.full((K, N), c, np.uint8)
    z = np.full((2, N), z0, np.uint8)
    g = np.random.default_rng(12)
    # dyadic x so every partial sum is exact in fp64
    x = (g.integers(-64, 64, (3, K)) / 16.0).astype(np.float16)
    bias = (g.integers(-8, 8, N) / 4.0).astype(np.float16)
    dq = oracle.dequantize_layer(pack_rows(q), pack_cols(z), np.ones((2, N), np.float16),
                                 None, K, N, 128)
    y = oracle.reference_output(x, dq, bias)
    expect = (c - z0 - 1) * x.astype(np.float64).sum(axis=1, keepdims=True) + bias.astype(np.float64)
    assert np.array_equal(y, expect)


def test_golden_worked_examples():
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        spec = json.load(f)
    for case in spec["cases"]:
        def arr(key, dt):
            v = case[key]
            return None if v is None else np.array([[int(s, 16) for s in row] for row in v] if isinstance(v[0], list)
                                                    else [int(s, 16) for s in v], dtype=np.uint64)
        K, N, gs = case["K"], case["N"], case["groupsize"]
        qw = arr("qweight_hex", None).astype(np.uint32).view(np.int32)
        qz = arr("qzeros_hex", None).astype(np.uint32).view(np.int32)
        sc = arr("scales_fp16_hex", None).astype(np.uint16)
        xb = arr("x_fp16_hex", None).astype(np.uint16)
        bb = case["bias_fp16_hex"]
        bias = None if bb is None else np.array([int(s, 16) for s in bb], np.uint16)
        gidx = None if "g_idx" not in case else np.array(case["g_idx"], np.int32)
        dq = oracle.dequantize_layer(qw, qz, sc, gidx, K, N, gs)
        assert [int(v) for v in dq.w16[0]] == [int(s, 16) for s in case["w16_row0_hex"]]
        y = oracle.reference_output(xb, dq, bias)
        assert np.array_equal(y, np.array(case["y"], np.float64)), case["comment"]


# ---------------------------------------------------------------- g_idx

def test_trivial_gidx_equals_none():
    layer = synthetic.make_layer(256, 64, 64, key=(13,))
    x = synthetic.activations(4, 256, key=(13, 4))
    gi = (np.arange(256) // 64).astype(np.int32)
    a = oracle.linear_layer(layer.qweight, layer.qzeros, layer.scales, None, None, x, 256, 64, 64)
    b = oracle.linear_layer(layer.qweight, layer.qzeros, layer.scales, gi, None, x, 256, 64, 64)
    assert np.array_equal(a[0].w16, b[0].w16)
    assert np.array_equal(a[1], b[1])


def test_act_order_is_a_row_permutation():
    """y(x, W, g_idx) == y(x[:, P], W[P, :], g_idx[P]); with g_idx[P] sorted
    this is the plain grouped layer on the permuted operands."""
    K, N, gs = 256, 32, 64
    layer = synthetic.make_layer(K, N, gs, act_order=True, key=(14,))
    x = synthetic.activations(3, K, key=(14, 3))
    q = oracle.unpack_qweight(layer.qweight, K, N)
    P = np.argsort(layer.g_idx, kind="stable")
    assert np.array_equal(layer.g_idx[P], np.arange(K) // gs)
    dq_a, y_a, _, _ = oracle.linear_layer(layer.qweight, layer.qzeros, layer.scales, layer.g_idx,
                                          None, x, K, N, gs)
    dq_b, y_b, _, _ = oracle.linear_layer(pack_rows(q[P]), layer.qzeros, layer.scales, None,
                                          None, np.ascontiguousarray(x[:, P]), K, N, gs)
    assert np.array_equal(dq_a.w16[P], dq_b.w16)
    assert np.allclose(y_a, y_b, rtol=1e-12, atol=1e-12 * np.abs(y_a).max())


# ------------------------------------------------------------ tolerance

def test_single_layer_reference_within_tolerance_of_exact():
    layer, x = synthetic.single_layer()
    dq, y_ref, y_exact, tol = oracle.linear_layer(layer.qweight, layer.qzeros, layer.scales, None,
                                                  None, x, 1024, 1024, 128)
    assert np.all(np.abs(y_ref - y_exact) <= tol)
    assert np.all(tol > 0)


def test_tolerance_catches_planted_mistakes():
    """Plant two plausible errors in the oracle's inputs and make sure the
    stated tolerance rejects them: dropping the +1 on the zero point, and
    reading the nibbles high-first."""
    K, N, gs = 1024, 256, 128
    layer = synthetic.make_layer(K, N, gs, key=(15,))
    x = synthetic.activations(2, K, key=(15, 2))
    dq, y_ref, _, tol = oracle.linear_layer(layer.qweight, layer.qzeros, layer.scales, None,
                                            None, x, K, N, gs)
    # (a) no +1: equivalent to an effective zero one smaller
    z = oracle.unpack_qzeros(layer.qzeros, dq.G, N).astype(np.int64)
    # z - 1 would go negative for z = 0: emulate through the weights instead
    w_wrong = dq.w64 + layer.scales.astype(np.float64)[dq.gr]
    y_wrong = oracle.linear_f64(oracle.half_bits_to_f64(x.view(np.uint16)), w_wrong)
    assert np.any(np.abs(y_wrong - y_ref) > tol)
    # (b) nibbles read high-first
    q = oracle.unpack_qweight(layer.qweight, K, N)
    q_rev = q.reshape(K // 8, 8, N)[:, ::-1, :].reshape(K, N)
    dq_rev = oracle.dequantize_layer(pack_rows(q_rev), layer.qzeros, layer.scales, None, K, N, gs)
    y_rev = oracle.reference_output(x, dq_rev)
    assert np.any(np.abs(y_rev - y_ref) > tol)
    del z


def test_tolerance_hand_computed_values():
    """The fp16 bound against values worked out by hand (not by re-evaluating
    its formula).  K = 64, so sqrt(K) = 8.  x has two rows whose largest
    magnitudes differ (|-4| in row 0, 0.5 in row 1); the largest |w| is |-2|.
    With the maxima global over the whole x and w16:
        1e-2 * 8 * 4 * 2 / 64 = 0.01
    so every element's bound is 0.01 + 0.002 |y_ref|:
        y_ref  =  1, -10,  0   |  100,  0.5,  -3
        bound  = 0.012, 0.03, 0.01 | 0.21, 0.011, 0.016
    A bound with K instead of sqrt(K) (0.08 + ...), without the /64
    (0.64 + ...), with |y_ref| dropped, or with the maxima taken per row (row 1
    would give 0.00125 + ...) misses these values."""
    x = np.zeros((2, 64), np.float16)
    x[0, 5], x[0, 9] = -4.0, 3.5
    x[1, 0], x[1, 63] = 0.5, -0.25
    w = np.zeros((64, 3), np.float16)
    w[7, 1], w[40, 2] = -2.0, 1.75
    y_ref = np.array([[1.0, -10.0, 0.0], [100.0, 0.5, -3.0]])
    tol = oracle.tolerance(x.view(np.uint16), w.view(np.uint16), y_ref, 64)
    expect = np.array([[0.012, 0.03, 0.01], [0.21, 0.011, 0.016]])
    np.testing.assert_allclose(tol, expect, rtol=1e-12, atol=0)


# ------------------------------------------------------------- fp32 x

def test_f32_to_double_matches_numpy_on_sampled_patterns():
    """The binary32 decoder against numpy's float32 reinterpretation: 2^20
    seeded random bit patterns plus every exponent at the fraction's ends,
    signed zeros, the subnormal range's ends, the largest finite values and
    infinities; NaN patterns decode to NaN."""
    g = np.random.default_rng(21)
    rnd = g.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    e = np.arange(256, dtype=np.uint32) << 23
    ends = np.concatenate([e, e | 1, e | 0x7FFFFF, e | 0x400000])
    special = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0xFF7FFFFF,
                        0x7F800000, 0xFF800000], np.uint32)
    bits = np.concatenate([rnd, ends, ends | 0x80000000, special])
    got = oracle.f32_bits_to_f64(bits)
    with np.errstate(invalid="ignore"):
        want = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_f32_hand_values():
    """Values worked out from the binary32 layout by hand."""
    cases = {0x3F800000: 1.0, 0xC0000000: -2.0, 0x00000001: 2.0 ** -149, 0x00800000: 2.0 ** -126,
             0x7F7FFFFF: (2.0 - 2.0 ** -23) * 2.0 ** 127, 0x3EAAAAAB: 11184811 * 2.0 ** -25,
             0x00400000: 2.0 ** -127}
    for bits, v in cases.items():
        assert oracle.f32_bits_to_f64(np.array([bits], np.uint32))[0] == v, hex(bits)


def test_f32_tolerance_hand_computed_values():
    """The fp32-activation bound (per-row max|x|) against hand-worked values.
    K = 64 (sqrt 8), largest |w| = 2.  Row 0 has max|x| = 4, row 1 has 0.5:
        row 0: 1e-2 * 8 * 4 * 2 / 64 = 0.01      row 1: ... * 0.5 ... = 0.00125
    plus 0.002 |y_ref|:  y_ref = 1, -10 | 100, 0.5
        bound = 0.012, 0.03 | 0.20125, 0.00225"""
    x = np.zeros((2, 64), np.float32)
    x[0, 3], x[0, 8] = -4.0, 2.5
    x[1, 1] = 0.5
    w = np.zeros((64, 2), np.float16)
    w[10, 0] = -2.0
    y_ref = np.array([[1.0, -10.0], [100.0, 0.5]])
    tol = oracle.tolerance_rows_f32(x.view(np.uint32), w.view(np.uint16), y_ref, 64)
    np.testing.assert_allclose(tol, np.array([[0.012, 0.03], [0.20125, 0.00225]]), rtol=1e-12, atol=0)


def test_f32_reference_is_the_definition_on_a_tiny_layer():
    """y for fp32 x by brute force: explicit nested sums over the exact
    double values of x and of the dequantized weights."""
    K, N, gs = 16, 8, 8
    layer = synthetic.make_layer(K, N, gs, key=(23,))
    dq = oracle.dequantize_layer(layer.qweight, layer.qzeros, layer.scales, None, K, N, gs)
    xb = synthetic.activations_f32(3, K, key=(23, 3), row_scales=[1.0, 1e6, 1e-6])
    x = xb.view(np.float32).astype(np.float64)
    w = dq.w16.view(np.float16).astype(np.float64)
    y = oracle.reference_output_f32(xb, dq)
    for m in range(3):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[m, k] * w[k, n]
            assert y[m, n] == acc
