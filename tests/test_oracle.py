"""Pins for the CPU oracle, against what the pages and plain mathematics fix.

No GPU.  Each test pins the oracle to something other than itself: values
decoded by hand from the pages' bit layout, the pages' second description of
the decoder (three permuted signed 64-entry tables indexed by I0, I1, I2),
the reflection structure of the codebook, closed forms, textbook integer
matrix products, and exact rational arithmetic.

Pages: "11 billion parameters on a phone" (Graphcore Research blog),
sections "Bit layout", "Fusing sign selection into lookups", "Absolute-value
centroids and sign selection", "Output channel packing", "Format decoding on
Arm CPUs"; "Llama-Mobile: Efficient 2.7-Bit Quantization of VLMs", section
3.4 (Eq. 1, domains, bits per element, alpha = absmax / 127).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import s3d8_inputs as si

HERE = os.path.dirname(os.path.abspath(__file__))


def hand_table():
    """C[q][d] = 4q + d + 1, the table the golden fixture was decoded with."""
    return np.array([[4 * q + d + 1 for d in range(3)] for q in range(32)], dtype=np.int8)


def load_fixture():
    rows = []
    with open(os.path.join(HERE, "golden", "byte_layout.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            rows.append([int(tok[0], 16)] + [int(t) for t in tok[1:]])
    return rows


def signed_tables_from_pages(C):
    """The decoder as the blog's "Format decoding on Arm CPUs" describes it.

    Each column of the 32 x 3 absolute table is expanded over both signs into
    a 64-entry signed table: components 0 and 2 in sign-minor order (index =
    2Q + s), component 1 in sign-major order (index = 32 s + Q).
    """
    C = np.asarray(C, dtype=np.int64)
    T0 = np.zeros(64, np.int64)
    T1 = np.zeros(64, np.int64)
    T2 = np.zeros(64, np.int64)
    for q in range(32):
        for s in (0, 1):
            sign = -1 if s else 1
            T0[2 * q + s] = sign * C[q, 0]
            T1[32 * s + q] = sign * C[q, 1]
            T2[2 * q + s] = sign * C[q, 2]
    return T0, T1, T2


def decode_by_pages_lut(b, tables):
    """Three lookups with indices built by the blog's 5 logical operations."""
    T0, T1, T2 = tables
    i0 = b & 0x3F
    i1 = (b >> 1) & 0x3F
    i2 = i0 ^ (b >> 7)
    return int(T0[i0]), int(T1[i1]), int(T2[i2])


def dense_by_pages_lut(packed, C, N):
    tables = signed_tables_from_pages(C)
    G, K = packed.shape
    W = np.zeros((3 * G, K), np.int64)
    lut = np.array([decode_by_pages_lut(b, tables) for b in range(256)], dtype=np.int64)
    for d in range(3):
        W[d::3] = lut[packed.astype(np.int64), d]
    return W[:N]


def some_tables():
    rng = np.random.default_rng(1234)
    yield hand_table()
    yield rng.integers(0, 128, size=(32, 3)).astype(np.int8)        # includes 0 and 127
    t = rng.integers(1, 128, size=(32, 3)).astype(np.int8)
    t[0] = 0
    t[31] = 127
    yield t
    yield np.zeros((32, 3), np.int8)


# --------------------------------------------------------------------------
# Byte layout
# --------------------------------------------------------------------------

def test_fixture_fields_and_values():
    C = hand_table()
    for b, Q, S0, S1, S2, I0, I1, I2, w0, w1, w2 in load_fixture():
        assert oracle.byte_fields(b) == (Q, S0, S1, S2), hex(b)
        assert oracle.pack_byte(Q, S0, S1, S2) == b, hex(b)
        # the fixture's indices are the blog's I0 / I1 / I2 of the same byte
        assert (b & 0x3F, (b >> 1) & 0x3F, (b & 0x3F) ^ (b >> 7)) == (I0, I1, I2)
        assert (I0, I1, I2) == (2 * Q + S0, 32 * S1 + Q, 2 * Q + S2)
        got = tuple(oracle.decode_component(b, C, d) for d in range(3))
        assert got == (w0, w1, w2), hex(b)


@pytest.mark.parametrize("which", range(4))
def test_exhaustive_decode_matches_pages_lut_reading(which):
    C = list(some_tables())[which]
    tables = signed_tables_from_pages(C)
    for b in range(256):
        want = decode_by_pages_lut(b, tables)
        got = tuple(oracle.decode_component(b, C, d) for d in range(3))
        assert got == want, (hex(b), got, want)


def test_layout_is_a_bijection():
    seen = set()
    for b in range(256):
        f = oracle.byte_fields(b)
        assert 0 <= f[0] < 32 and all(s in (0, 1) for s in f[1:])
        assert oracle.pack_byte(*f) == b
        seen.add(f)
    assert len(seen) == 256


def test_reflections():
    """The 256 signed codewords are the 8 sign reflections of 32 absolute rows
    (blog, "Absolute-value centroids and sign selection"); in the physical
    layout each reflection is a fixed XOR on the byte."""
    rng = np.random.default_rng(7)
    C = rng.integers(1, 128, size=(32, 3)).astype(np.int8)
    flips = {0x41: (-1, -1, -1), 0x81: (-1, 1, 1), 0x40: (1, -1, 1), 0x80: (1, 1, -1)}
    for b in range(256):
        base = [oracle.decode_component(b, C, d) for d in range(3)]
        assert [abs(v) for v in base] == [int(C[oracle.byte_fields(b)[0], d]) for d in range(3)]
        for mask, sgn in flips.items():
            got = [oracle.decode_component(b ^ mask, C, d) for d in range(3)]
            assert got == [s * v for s, v in zip(sgn, base)], (hex(b), hex(mask))
    # the 8 reflections of one row are all distinct when the row has no zero
    row = {tuple(oracle.decode_component(b, C, d) for d in range(3)) for b in range(256)
           if oracle.byte_fields(b)[0] == 5}
    assert len(row) == 8


def test_output_channel_packing_and_padding():
    """Byte (g, k) feeds channels 3g, 3g+1, 3g+2 at column k; N is padded up to
    a multiple of 3 and the pad lanes never reach an output."""
    rng = np.random.default_rng(3)
    C = rng.integers(1, 128, size=(32, 3)).astype(np.int8)
    for N in (1, 2, 3, 4, 5, 7, 96):
        G = oracle.groups(N)
        K = 32
        packed = rng.integers(0, 256, size=(G, K), dtype=np.uint8)
        W = oracle.decode(packed, C, N)
        assert W.shape == (N, K)
        np.testing.assert_array_equal(W.astype(np.int64), dense_by_pages_lut(packed, C, N))
        # flipping every pad-lane sign selector changes nothing
        if 3 * G > N:
            Q = np.array([[oracle.byte_fields(b)[0] for b in r] for r in packed], np.int32)
            S = np.zeros((3 * G, K), np.int32)
            for g in range(G):
                for k in range(K):
                    f = oracle.byte_fields(int(packed[g, k]))
                    S[3 * g:3 * g + 3, k] = f[1:]
            S[N:] ^= 1
            packed2 = oracle.pack(Q, S)
            assert not np.array_equal(packed2, packed)
            np.testing.assert_array_equal(oracle.decode(packed2, C, N), W)


def test_pack_roundtrip_matrix():
    rng = np.random.default_rng(11)
    G, K = 5, 48
    Q = rng.integers(0, 32, size=(G, K)).astype(np.int32)
    S = rng.integers(0, 2, size=(3 * G, K)).astype(np.int32)
    packed = oracle.pack(Q, S)
    for g in range(G):
        for k in range(K):
            f = oracle.byte_fields(int(packed[g, k]))
            assert f == (Q[g, k], S[3 * g, k], S[3 * g + 1, k], S[3 * g + 2, k])


# --------------------------------------------------------------------------
# Accumulation: textbook integer products and closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 2, 16), (3, 4, 32), (5, 5, 256), (4, 96, 256),
                                   (2, 7, 48)])
def test_linear_acc_matches_textbook_matmul(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    C = rng.integers(0, 128, size=(32, 3)).astype(np.int8)
    packed = rng.integers(0, 256, size=(oracle.groups(N), K), dtype=np.uint8)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    W = dense_by_pages_lut(packed, C, N)
    want = xq.astype(np.int64) @ W.T
    acc, bad = oracle.linear_acc(packed, C, xq, N)
    assert bad == 0
    np.testing.assert_array_equal(acc, want)
    ms = rng.integers(0, M, size=17)
    ns = rng.integers(0, N, size=17)
    np.testing.assert_array_equal(oracle.linear_acc_at(packed, C, xq, N, ms, ns), want[ms, ns])


def test_constant_bytes_closed_form():
    """All bytes equal with every selector positive: acc[m, 3g+d] = C[Q][d] * sum_k xq[m, k]."""
    rng = np.random.default_rng(5)
    C = rng.integers(1, 128, size=(32, 3)).astype(np.int8)
    M, N, K = 3, 9, 64
    for Q in (0, 17, 31):
        b = oracle.pack_byte(Q, 0, 0, 0)
        packed = np.full((oracle.groups(N), K), b, np.uint8)
        xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        acc, _ = oracle.linear_acc(packed, C, xq, N)
        rs = xq.astype(np.int64).sum(axis=1)
        for n in range(N):
            np.testing.assert_array_equal(acc[:, n], int(C[Q, n % 3]) * rs)
        # the all-negative reflection negates every accumulator exactly
        acc_neg, _ = oracle.linear_acc(packed ^ np.uint8(0x41), C, xq, N)
        np.testing.assert_array_equal(acc_neg, -acc)


def test_int32_edge():
    """|acc| <= 127 * 127 * K; at K = 14336 the extreme 231,225,344 still fits
    int32, and at K = 133,145 it does not."""
    C = np.full((32, 3), 127, np.int8)
    for K, fits in ((14336, True), (133145, False)):
        packed = np.full((1, K), oracle.pack_byte(3, 0, 0, 0), np.uint8)
        xq = np.full((1, K), 127, np.int8)
        acc, bad = oracle.linear_acc(packed, C, xq, 3)
        assert (acc == 16129 * K).all()
        assert (bad == 0) == fits
    assert 16129 * 14336 == 231_225_344


# --------------------------------------------------------------------------
# Activation quantisation (per-token absmax INT8)
# --------------------------------------------------------------------------

def bf16(vals):
    return si.f32_to_bf16_bits(np.asarray(vals, np.float32))


def test_quantize_ties_to_even_with_unit_scale():
    # absmax 127 gives s = 127 / 127 = 1 exactly, so x / s = x
    x = bf16([[127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, 126.5, 0.0, -127.0, 64.0, 1.0, -1.0,
               0.25, 0.75]])
    xq, xs = oracle.quantize_act(x)
    assert xs[0] == np.float32(1.0)
    assert xq.tolist() == [[127, 2, 4, -2, -4, 0, 2, 0, 126, 0, -127, 64, 1, -1, 0, 1]]


def test_quantize_zero_row_and_signs():
    rng = np.random.default_rng(9)
    xf = rng.standard_normal((4, 64)).astype(np.float32)
    xf[2] = 0.0
    x = bf16(xf)
    xq, xs = oracle.quantize_act(x)
    assert xs[2] == 0.0 and (xq[2] == 0).all()
    xneg = x ^ np.uint16(0x8000)          # flip the bf16 sign bit: exact negation
    xneg[2] = 0
    xqn, xsn = oracle.quantize_act(xneg)
    np.testing.assert_array_equal(xsn, xs)
    np.testing.assert_array_equal(xqn, -xq)


def test_quantize_properties():
    rng = np.random.default_rng(10)
    x = si.activations(rng, 8, 512, outliers=True)
    xf = si.bf16_bits_to_f32(x).astype(np.float64)
    xq, xs = oracle.quantize_act(x)
    amax = np.abs(xf).max(axis=1)
    # the scale is absmax / 127 rounded once to fp32
    for m in range(8):
        exact = Fraction(float(amax[m])) / 127
        half_ulp = Fraction(float(np.spacing(np.float32(xs[m])))) / 2
        assert abs(Fraction(float(xs[m])) - exact) <= half_ulp
        # the absmax element lands on +-127
        assert np.abs(xq[m]).max() == 127
        r = xf[m] / float(xs[m])
        assert np.all(np.abs(r - xq[m]) <= 0.5 + 1e-5)
    # scaling a row by 2 (exact in bf16) doubles the scale and keeps the codes
    x2 = si.f32_to_bf16_bits(si.bf16_bits_to_f32(x) * np.float32(2.0))
    xq2, xs2 = oracle.quantize_act(x2)
    np.testing.assert_array_equal(xq2, xq)
    np.testing.assert_array_equal(xs2, xs * np.float32(2.0))


def test_quantize_agrees_with_fp64_rounding_away_from_ties():
    rng = np.random.default_rng(12)
    x = si.activations(rng, 16, 1024)
    xf = si.bf16_bits_to_f32(x).astype(np.float64)
    xq, xs = oracle.quantize_act(x)
    r = xf / xs.astype(np.float64)[:, None]
    frac = np.abs(r - np.floor(r) - 0.5)
    safe = frac > 1e-4
    np.testing.assert_array_equal(xq[safe], np.rint(r[safe]).astype(np.int8))


# --------------------------------------------------------------------------
# Output scaling and bits per element
# --------------------------------------------------------------------------

def test_linear_out_exact_rationals():
    rng = np.random.default_rng(13)
    M, N = 3, 5
    acc = rng.integers(-2**31, 2**31, size=(M, N)).astype(np.int64)
    xs = rng.random(M).astype(np.float32)
    cs = si.f32_to_bf16_bits(rng.random(N).astype(np.float32) * 0.01)
    out = oracle.linear_out(acc, xs, cs)
    csf = si.bf16_bits_to_f32(cs)
    for m in range(M):
        for n in range(N):
            exact = Fraction(float(xs[m])) * int(acc[m, n]) * Fraction(float(csf[n]))
            assert abs(Fraction(out[m, n]) - exact) <= abs(exact) * Fraction(2, 2**52)


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096), (4096, 4096), (4096, 1024)])
def test_bits_per_element_closed_form(K, N):
    """Buffer sizes give 8/3 + 16/K bits per element up to padding and the
    96-byte table (Llama-Mobile section 3.4)."""
    G = oracle.groups(N)
    bits = 8 * G * K + 16 * N + 8 * 96
    bpp = bits / (N * K)
    slack = (8 * (3 * G - N) * K / 3 + 8 * 96) / (N * K)
    assert abs(bpp - (8 / 3 + 16 / K)) <= slack + 1e-12
    assert 2.66 < bpp < 2.68


def test_bits_per_element_whole_text_stack():
    total_bits = 0
    total_params = 0
    for _, K, N in list(si.LLAMA_11B_LAYER) * si.LLAMA_11B_LAYERS + [si.LLAMA_11B_HEAD]:
        total_bits += 8 * si.groups(N) * K + 16 * N + 8 * 96
        total_params += N * K
    bpp = total_bits / total_params
    # the pages report 2.68 bits/parameter for the whole VLM
    assert 2.66 < bpp < 2.69


def test_input_bf16_conversion_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    f = (rng.standard_normal(4096) * np.exp(rng.uniform(-30, 30, 4096))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(si.f32_to_bf16_bits(f), want)


# --------------------------------------------------------------------------
# Direct-cast encoder (Llama-Mobile paper, section 3.4 "Quantization":
# alpha = absmax / 127, s = sign with W >= 0 positive, q = nearest centroid of
# |W| / alpha in L2, the lowest index winning a tie)
# --------------------------------------------------------------------------

def _bf16_exact(vals):
    """float -> bf16 bits for values that bf16 holds exactly."""
    a = np.asarray(vals, np.float32)
    b = si.f32_to_bf16_bits(a)
    assert np.array_equal(si.bf16_bits_to_f32(b), a)
    return b


def test_encode_hand_worked_case():
    # Hand table: C[q] = (4q+1, 4q+2, 4q+3).  Both columns scaled by 1/64, and
    # every row holds a +-127/64, so alpha = 1/64 exactly for the three rows.
    #  column 0: (125, -126, 127) is centroid 31 itself, signs (+, -, +);
    #  column 1: (127, 127, 1) in magnitude, signs (-, +, -).  With
    #    f(q) = (4q - 126)^2 + (4q - 125)^2 + (4q + 2)^2:
    #    f(20) = 2116 + 2025 + 6724 = 10865, f(21) = 1764 + 1681 + 7396 = 10841,
    #    f(22) = 1444 + 1369 + 8100 = 10913, and f is a parabola in q: q = 21.
    C = hand_table()
    w = _bf16_exact(np.array([[125, -127], [-126, 127], [127, -1]], np.float32) / 64)
    packed, cs = oracle.encode(w, C)
    assert np.array_equal(si.bf16_bits_to_f32(cs), np.full(3, 1 / 64, np.float32))
    # fields by the pages' layout: S0 is w0's sign, S1 w1's sign, S2 w2's sign
    assert oracle.byte_fields(int(packed[0, 0])) == (31, 0, 1, 0)
    assert oracle.byte_fields(int(packed[0, 1])) == (21, 1, 0, 1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_encode_roundtrips_exactly_representable_weights(seed):
    # W = s * C[q] * alpha with alpha a power of two and one column that holds
    # 127 * alpha in every row, so |W| / alpha is C[q] exactly: distance 0 and,
    # with all-distinct table rows, the only nearest centroid.
    rng = np.random.default_rng(seed)
    C = rng.permutation(np.arange(1, 97)).reshape(32, 3).astype(np.int8)
    C[31] = 127                                   # centroid 31 = (127, 127, 127)
    N, K = 3 * 5, 40
    Q = rng.integers(0, 32, size=(N // 3, K))
    Q[:, 0] = 31
    S = rng.integers(0, 2, size=(N, K))
    alpha = 2.0 ** rng.integers(-12, -4, size=N)
    W = np.zeros((N, K))
    for n in range(N):
        W[n] = (1 - 2 * S[n]) * C[Q[n // 3], n % 3] * alpha[n]
    packed, cs = oracle.encode(_bf16_exact(W), C)
    assert np.array_equal(si.bf16_bits_to_f32(cs).astype(np.float64), alpha)
    # decode by the pages' own signed-table construction, independent of the oracle
    assert np.array_equal(dense_by_pages_lut(packed, C, N), (1 - 2 * S) * C[Q.repeat(3, 0), np.tile([0, 1, 2], N // 3)[:, None]])


def test_encode_tie_goes_to_lowest_index():
    C = hand_table()
    C[9] = C[4]                                   # a duplicate row later in the table
    C[20] = C[4]
    w = _bf16_exact(np.array([[17, 127], [18, 127], [19, 127]], np.float32))   # alpha = 1, C[4]
    packed, _ = oracle.encode(w, C)
    assert oracle.byte_fields(int(packed[0, 0]))[0] == 4
    # a point exactly halfway between two centroids on one axis
    C = np.zeros((32, 3), np.int8)
    C[:, 0] = np.arange(32) * 4
    w = _bf16_exact(np.array([[42, 127], [0, 0], [0, 0]], np.float32))     # 42: midway 40 / 44
    packed, _ = oracle.encode(w, C)
    assert oracle.byte_fields(int(packed[0, 0]))[0] == 10


def test_encode_signs_zeros_and_zero_channels():
    C = hand_table()
    pz, nz = 0x0000, 0x8000                        # +0 and -0 in bf16
    w = np.array([[pz, nz, 0x3F80], [nz, pz, 0xBF80], [0, 0, 0]], np.uint16)   # row 2 all zero
    packed, cs = oracle.encode(w, C)
    assert cs[2] == 0                              # alpha of an all-zero channel is 0
    for k in range(3):
        Q, S0, S1, S2 = oracle.byte_fields(int(packed[0, k]))
        assert S2 == 0                             # zero channel: positive
        # -0 >= 0, so both zero forms take the positive selector
        if k < 2:
            assert (S0, S1) == (0, 0)
    assert oracle.byte_fields(int(packed[0, 2]))[1:3] == (0, 1)
    # a zero group is (0, 0, 0): nearest is the row of least norm, centroid 0 here
    assert oracle.byte_fields(int(packed[0, 0]))[0] == 0


def test_encode_pads_missing_channels_positive_and_zero():
    C = hand_table()
    rng = np.random.default_rng(7)
    for N in (1, 2, 4, 5):
        W = si.f32_to_bf16_bits(rng.standard_normal((N, 16)).astype(np.float32))
        packed, cs = oracle.encode(W, C)
        assert packed.shape == (si.groups(N), 16) and cs.shape == (N,)
        g = (N - 1) // 3
        for k in range(16):
            f = oracle.byte_fields(int(packed[g, k]))
            for d in range(N - 3 * g, 3):
                assert f[1 + d] == 0
        # the padded components enter the distance as 0
        Cf = C.astype(np.float64)
        csf = si.bf16_bits_to_f32(cs).astype(np.float64)
        Wf = si.bf16_bits_to_f32(W).astype(np.float64)
        for k in range(16):
            wp = np.zeros(3)
            for d in range(N - 3 * g):
                wp[d] = abs(Wf[3 * g + d, k]) / csf[3 * g + d]
            dist = ((Cf - wp) ** 2).sum(1)
            q = oracle.byte_fields(int(packed[g, k]))[0]
            assert dist[q] <= dist.min() * (1 + 1e-5) + 1e-3


@pytest.mark.parametrize("N,K,seed", [(12, 64, 0), (7, 33, 1), (30, 16, 2)])
def test_encode_picks_a_nearest_centroid_and_the_right_scales(N, K, seed):
    rng = np.random.default_rng(seed)
    C = si.centroids(rng)
    Wf32 = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Wf32[0, 3] = 0.25                              # an outlier channel
    W = si.f32_to_bf16_bits(Wf32)
    Wf = si.bf16_bits_to_f32(W).astype(np.float64)
    packed, cs = oracle.encode(W, C)
    alpha = si.bf16_bits_to_f32(cs).astype(np.float64)
    amax = np.abs(Wf).max(1)
    # alpha is absmax / 127 to bf16 precision (8 significant bits)
    assert np.all(np.abs(127 * alpha - amax) <= amax * 2.0 ** -8)
    # decoded signs follow the weights' signs; magnitudes are the chosen centroid
    dense = dense_by_pages_lut(packed, C, N)
    G = si.groups(N)
    Cf = C.astype(np.float64)
    for g in range(G):
        ch = [3 * g + d for d in range(3) if 3 * g + d < N]
        for k in range(K):
            q = oracle.byte_fields(int(packed[g, k]))[0]
            wp = np.zeros(3)
            for d, n in enumerate(ch):
                wp[d] = abs(Wf[n, k]) / alpha[n]
                assert dense[n, k] == (C[q, d] if Wf[n, k] >= 0 else -int(C[q, d]))
            dist = ((Cf - wp) ** 2).sum(1)
            # the fp32 decision may differ from exact arithmetic only within rounding
            assert dist[q] <= dist.min() * (1 + 1e-5) + 1e-3
            # and no centroid before q is strictly nearer by more than rounding
            assert np.all(dist[:q] >= dist[q] - (dist[q] * 1e-5 + 1e-3))


def test_encode_then_decode_is_a_fixed_point():
    # Encoding the decoded weights s * alpha * C[q] (exactly representable when
    # alpha is a power of two and a channel holds 127) gives the same bytes back.
    rng = np.random.default_rng(3)
    C = si.centroids(rng)
    C[0] = 127
    N, K = 9, 24
    packed = si.packed_bytes(rng, si.groups(N), K)
    packed[:, 0] = oracle.pack_byte(0, 0, 0, 0)
    dense = dense_by_pages_lut(packed, C, N).astype(np.float64)
    assert len({tuple(r) for r in C.tolist()}) == 32     # the nearest centroid is unique
    W = _bf16_exact(dense * 2.0 ** -9)
    again, cs = oracle.encode(W, C)
    assert np.all(si.bf16_bits_to_f32(cs) == np.float32(2.0 ** -9))
    assert np.array_equal(again, packed)


# --------------------------------------------------------------------------
# Centroid fit (Llama-Mobile paper, section 3.4 "Quantization": Lloyd-Max
# with k-means++ initialisation on the zero-padded |W| / alpha 3-vectors, then
# Round).  Draws are 32 caller-supplied 32-bit integers.
# --------------------------------------------------------------------------

GRID_X = (13, 40, 68, 96)
GRID_Z = (12, 60)


def cluster_centres():
    """31 grid centres 28+ apart, plus (127, 127, 127)."""
    cs = [(x, y, z) for x in GRID_X for y in GRID_X for z in GRID_Z]
    cs.remove((96, 96, 60))
    cs.append((127, 127, 127))
    return np.array(cs, np.float64)


def weights_from_points(Wp, alpha_exp=-8, seed=0):
    """bf16 weights whose scaled magnitudes are the given points [G, K, 3]:
    W = s * W' * 2^alpha_exp with random signs; every channel must hold 127."""
    rng = np.random.default_rng(seed)
    G, K, _ = Wp.shape
    W = np.zeros((3 * G, K))
    for d in range(3):
        W[d::3] = Wp[:, :, d] * (2.0 ** alpha_exp)
    W *= 1 - 2 * rng.integers(0, 2, size=W.shape)
    return _bf16_exact(W)


def draws(seed):
    return np.random.default_rng(seed).integers(0, 2 ** 32, 32, dtype=np.uint64).astype(np.uint32)


def clustered_points(G=16, K=256, seed=0, half_up=()):
    """Each point is a cluster centre plus an offset of +-0.5 on one axis
    (means within 0.5 / count of the centre), or {0, +1} in x for the centres in
    half_up (mean x.5 when the count is even)."""
    rng = np.random.default_rng(seed)
    cs = cluster_centres()
    Wp = np.zeros((G, K, 3))
    lab = rng.permutation(np.arange(G * K) % 32).reshape(G, K)
    lab[:, 0] = 31                                   # every row holds (127, 127, 127)
    counts = {}
    for g in range(G):
        for k in range(K):
            c = lab[g, k]
            i = counts.get(c, 0)
            counts[c] = i + 1
            off = np.zeros(3)
            if c != 31:
                if c in half_up:
                    off[0] = i % 2
                else:
                    off[i % 3] = 0.5 if (i // 3) % 2 == 0 else -0.5
            Wp[g, k] = cs[c] + off
    return Wp, lab, counts


def sorted_rows(a):
    a = np.asarray(a)
    return a[np.lexsort(a.T[::-1])]


def test_fit_recovers_well_separated_clusters():
    Wp, lab, counts = clustered_points()
    W = weights_from_points(Wp)
    cf, C = oracle.fit_centroids(W, draws(1), iters=8)
    assert np.array_equal(sorted_rows(C.astype(np.int64)), sorted_rows(cluster_centres().astype(np.int64)))
    # the fp32 centroids are the cluster means, within the 2^-20 grid of the sums
    means = np.array([Wp[lab == c].mean(0) for c in range(32)])
    assert np.allclose(sorted_rows(cf.astype(np.float64)), sorted_rows(means), atol=2e-6)


def test_fit_rounds_half_to_even():
    # clusters (13, y, z) and (40, y, z) take x in {c, c+1} equally: mean c + 0.5
    half = [i for i, c in enumerate(cluster_centres()) if c[0] in (13.0, 40.0)
            and c[1] == 13.0 and c[2] == 12.0]
    Wp, lab, counts = clustered_points(seed=3, half_up=half)
    assert all(counts[c] % 2 == 0 for c in half)
    W = weights_from_points(Wp, seed=3)
    cf, C = oracle.fit_centroids(W, draws(4), iters=8)
    got = {tuple(r) for r in C.astype(np.int64).tolist()}
    assert (14, 13, 12) in got and (13, 13, 12) not in got    # 13.5 -> 14
    assert (40, 13, 12) in got and (41, 13, 12) not in got    # 40.5 -> 40
    assert np.isclose(cf.astype(np.float64), 13.5).any() and np.isclose(cf.astype(np.float64), 40.5).any()


def test_fit_with_fewer_distinct_points_than_centroids():
    # one packed row, 16 distinct points on a line (rows 1, 2 all zero): k-means++
    # never draws a point already covered while any weight is left, so all 16
    # become centroids; every point then sits on its own centroid
    xs = np.array([0, 3, 8, 10, 20, 33, 47, 51, 64, 70, 80, 90, 100, 110, 120, 127], np.float64)
    Wp = np.zeros((1, 16, 3))
    Wp[0, :, 0] = xs
    W = np.zeros((3, 16), np.uint16)
    W[0] = _bf16_exact(xs)                          # alpha = 1 exactly
    cf, C = oracle.fit_centroids(W, draws(5), iters=3)
    assert set(cf[:, 0].tolist()) == set(xs.tolist())
    assert np.all(cf[:, 1:] == 0)
    assert set(C[:, 0].astype(np.int64).tolist()) == set(xs.astype(np.int64).tolist())


def test_kmeanspp_second_centre_follows_d2_weights():
    # first centre fixed at point 0 (x = 0) by r[0] = 0; over a fine grid of r[1]
    # the second centre must be point p with frequency D2_p / sum D2 = x_p^2 / sum x^2
    xs = np.array([0, 3, 8, 10, 20, 33, 47, 51, 64, 70, 80, 90, 100, 110, 120, 127], np.float64)
    W = np.zeros((3, 16), np.uint16)
    W[0] = _bf16_exact(xs)
    T = 2048
    hits = dict.fromkeys(xs.tolist(), 0)
    for j in range(T):
        r = np.zeros(32, np.uint32)
        r[1] = int((j + 0.5) / T * 2 ** 32)
        cf, _ = oracle.fit_centroids(W, r, iters=0)
        assert cf[0, 0] == 0.0
        hits[float(cf[1, 0])] += 1
    p = xs ** 2 / (xs ** 2).sum()
    freq = np.array([hits[x] for x in xs.tolist()]) / T
    assert np.all(np.abs(freq - p) <= 2.0 / T), np.abs(freq - p).max()


def _points_f64(W):
    Wf = si.bf16_bits_to_f32(W).astype(np.float64)
    N, K = Wf.shape
    G = si.groups(N)
    amax = np.abs(Wf).max(1)
    alpha = si.bf16_bits_to_f32(si.f32_to_bf16_bits((amax / 127).astype(np.float32))).astype(np.float64)
    P = np.zeros((G, K, 3))
    for n in range(N):
        if alpha[n] > 0:
            P[n // 3, :, n % 3] = np.abs(Wf[n]) / alpha[n]
    return P.reshape(-1, 3)


def test_lloyd_step_moves_centroids_to_the_means_of_their_points():
    rng = np.random.default_rng(8)
    W = si.f32_to_bf16_bits((rng.standard_normal((31, 128)) * 0.02).astype(np.float32))
    r = draws(9)
    c0, _ = oracle.fit_centroids(W, r, iters=0)
    c1, _ = oracle.fit_centroids(W, r, iters=1)
    P = _points_f64(W)
    d = ((P[:, None, :] - c0.astype(np.float64)[None]) ** 2).sum(2)
    lab = d.argmin(1)
    for l in range(32):
        if (lab == l).any():
            assert np.allclose(c1[l], P[lab == l].mean(0), atol=2e-6, rtol=1e-6), l
        else:
            assert np.array_equal(c1[l], c0[l])          # an empty cluster stays put


def test_lloyd_objective_never_increases():
    rng = np.random.default_rng(10)
    W = si.f32_to_bf16_bits((rng.standard_normal((45, 96)) * 0.02).astype(np.float32))
    P = _points_f64(W)
    r = draws(11)
    prev = np.inf
    for it in range(7):
        c, _ = oracle.fit_centroids(W, r, iters=it)
        sse = ((P[:, None, :] - c.astype(np.float64)[None]) ** 2).sum(2).min(1).sum()
        assert sse <= prev * (1 + 1e-9) + 1e-6, (it, sse, prev)
        prev = sse


# --------------------------------------------------------------------------
# Fake-quant forward (paper section 3.4: in QAT the weight is quantised in the
# forward pass with the centroids frozen and rebuilt by Eq. 1)
# --------------------------------------------------------------------------

def test_fake_quant_keeps_exactly_representable_weights():
    # s * alpha * C[q] with alpha a power of two and 127 in every channel is its
    # own quantisation: the forward pass returns the weights bit for bit
    rng = np.random.default_rng(12)
    C = rng.permutation(np.arange(1, 97)).reshape(32, 3).astype(np.int8)
    C[31] = 127
    N, K = 12, 48
    Q = rng.integers(0, 32, size=(N // 3, K))
    Q[:, 0] = 31
    S = rng.integers(0, 2, size=(N, K))
    alpha = 2.0 ** rng.integers(-12, -4, size=N)
    W = np.zeros((N, K))
    for n in range(N):
        W[n] = (1 - 2 * S[n]) * C[Q[n // 3], n % 3] * alpha[n]
    Wb = _bf16_exact(W)
    assert np.array_equal(oracle.fake_quant(Wb, C), Wb)


def test_fake_quant_is_scale_times_signed_centroid():
    # every output is +-alpha_n times an entry of column n mod 3 of the table,
    # with the weight's sign (0 for a zero channel), within one bf16 rounding
    rng = np.random.default_rng(13)
    C = si.centroids(rng)
    N, K = 14, 64
    W = si.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    W[5] = 0
    out = si.bf16_bits_to_f32(oracle.fake_quant(W, C)).astype(np.float64)
    Wf = si.bf16_bits_to_f32(W).astype(np.float64)
    alpha = np.abs(Wf).max(1) / 127
    assert np.all(out[5] == 0)
    for n in range(N):
        if n == 5:
            continue
        ratio = np.abs(out[n]) / alpha[n]
        col = C[:, n % 3].astype(np.float64)
        near = np.abs(ratio[:, None] - col[None, :]).min(1)
        assert np.all(near <= col.max() * 2.0 ** -7), n     # bf16 alpha and bf16 rounding
        assert np.all(np.sign(out[n]) == np.sign(Wf[n]) * (out[n] != 0))


def test_fake_quant_error_is_the_nearest_centroid_error():
    # per 3-vector, the reconstruction error in units of alpha is the distance to
    # the nearest centroid, so no other table row reconstructs the vector better
    rng = np.random.default_rng(14)
    C = si.centroids(rng)
    N, K = 9, 40
    W = si.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    out = si.bf16_bits_to_f32(oracle.fake_quant(W, C)).astype(np.float64)
    Wf = si.bf16_bits_to_f32(W).astype(np.float64)
    _, cs = oracle.encode(W, C)
    a = si.bf16_bits_to_f32(cs).astype(np.float64)
    Cf = C.astype(np.float64)
    for g in range(N // 3):
        for k in range(K):
            wp = np.array([abs(Wf[3 * g + d, k]) / a[3 * g + d] for d in range(3)])
            got = np.array([abs(out[3 * g + d, k]) / a[3 * g + d] for d in range(3)])
            err = np.sqrt(((got - wp) ** 2).sum())
            best = np.sqrt(((Cf - wp) ** 2).sum(1).min())
            # the bf16 rounding of alpha C moves each component by at most
            # 127 * 2^-9 (in units of alpha): sqrt(3) * 0.25 < 0.5 in total
            assert err <= best + 0.5
