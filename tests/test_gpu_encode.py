"""GPU parity of the direct-cast encoder (s3d8_encode) with the oracle.

Bit-exact: the bf16 channel scales and every packed byte.  Weights follow the
recipe of a trained layer (bf16 N(0, 0.02) with 1 % outliers x 20, per-channel
spread); the tables are the recipe's random int8 1..127 rows.  Special cases:
exact ties between centroids, points on a midway plane, all-zero channels,
-0, values that hit a centroid exactly, padded channels (N mod 3 = 1, 2),
the smallest and ragged shapes, and a full 4096 x 14336 gate matrix checked on
sampled packed rows (the oracle encodes those rows' three channels alone,
which fixes their scales and bytes).
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import bf16_bits, dev, i8, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def weights(rng, N, K):
    w = rng.standard_normal((N, K)) * 0.02 * rng.uniform(0.5, 2.0, size=(N, 1))
    out = rng.random((N, K)) < 0.01
    w[out] *= 20
    return si.f32_to_bf16_bits(w.astype(np.float32))


def run_gpu(w_bits, C):
    packed, cs = s3d8.encode(bf16_bits(w_bits), i8(C))
    torch.cuda.synchronize()
    return to_np(packed), to_np(cs.view(torch.int16)).view(np.uint16)


def assert_same(w_bits, C):
    want_p, want_s = oracle.encode(w_bits, C)
    got_p, got_s = run_gpu(w_bits, C)
    assert np.array_equal(got_s, want_s), np.argwhere(got_s != want_s)[:5]
    bad = np.argwhere(got_p != want_p)
    assert bad.size == 0, (bad[:5], got_p[tuple(bad[0])], want_p[tuple(bad[0])])


@pytest.mark.parametrize("N,K,seed", [(3, 16, 0), (1, 16, 1), (2, 32, 2), (4, 48, 3),
                                      (5, 4096, 4), (96, 256, 5), (241, 1040, 6),
                                      (722, 2112, 7), (1024, 4096, 8)])
def test_encode_matches_oracle(N, K, seed):
    rng = np.random.default_rng(seed)
    assert_same(weights(rng, N, K), si.centroids(rng))


def test_encode_ties_midpoints_zeros_and_exact_hits():
    rng = np.random.default_rng(11)
    N, K = 30, 64
    C = si.centroids(rng)
    C[7] = C[3]                                     # duplicate rows: the first must win
    C[19] = C[3]
    C[20] = [40, 0, 0]
    C[21] = [44, 0, 0]
    alpha = 2.0 ** rng.integers(-12, -5, size=N)
    W = np.clip(rng.standard_normal((N, K)) * 40, -126, 126) * alpha[:, None]
    W[:, 0] = 127 * alpha                           # every channel's absmax: alpha exact
    g = rng.integers(0, N // 3, size=40)
    k = rng.integers(1, K, size=40)
    for i, (gg, kk) in enumerate(zip(g, k)):
        q = [3, 20, 21][i % 3]
        s = rng.integers(0, 2, size=3)
        for d in range(3):
            W[3 * gg + d, kk] = (1 - 2 * s[d]) * C[q, d] * alpha[3 * gg + d]
    for d in range(3):                              # a point midway between C[20] and C[21]
        W[3 + d, 5] = [42, 0, 0][d] * alpha[3 + d]
    W[6:9, 7] = 0.0
    W[9:12, 9] = -0.0
    W[12] = 0.0                                      # a whole zero channel
    bits = si.f32_to_bf16_bits(W.astype(np.float32))
    bits[13, 3] = 0x8000                             # -0 next to a live channel
    assert_same(bits, C)


@pytest.mark.parametrize("N", [1, 2, 4, 5, 7, 8])
def test_encode_padded_groups(N):
    rng = np.random.default_rng(20 + N)
    assert_same(weights(rng, N, 96), si.centroids(rng))


def test_encode_table_with_zero_and_max_entries():
    rng = np.random.default_rng(31)
    C = rng.integers(0, 128, size=(32, 3)).astype(np.int8)
    C[0] = 0
    C[31] = 127
    assert_same(weights(rng, 48, 512), C)


def test_encode_full_gate_matrix_sampled_rows():
    name, K, N = "gate", 4096, 14336
    gen = torch.Generator(device=dev()).manual_seed(5)
    w = (torch.randn((N, K), device=dev(), generator=gen) * 0.02).to(torch.bfloat16)
    C = torch.randint(1, 128, (32, 3), dtype=torch.int8, device=dev(), generator=gen)
    packed, cs = s3d8.encode(w, C)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    G = si.groups(N)
    gs = np.concatenate([[0, 1, G - 1], rng.integers(0, G, 29)])
    Cn = to_np(C)
    for g in gs:
        rows = to_np(w[3 * g:3 * g + 3].view(torch.int16)).view(np.uint16)
        want_p, want_s = oracle.encode(rows, Cn)
        got_s = to_np(cs[3 * g:3 * g + 3].view(torch.int16)).view(np.uint16)
        assert np.array_equal(got_s, want_s), g
        assert np.array_equal(to_np(packed[g]), want_p[0]), g


def test_encode_decode_roundtrip_on_device():
    # decoding what the encoder wrote must give s * C[q] with s the sign of W
    rng = np.random.default_rng(41)
    N, K = 60, 256
    C = si.centroids(rng)
    w = weights(rng, N, K)
    packed, _ = s3d8.encode(bf16_bits(w), i8(C))
    dense = to_np(s3d8.decode(packed, i8(C), N))
    wf = si.bf16_bits_to_f32(w)
    assert np.all((dense >= 0) == (wf >= 0))
    mags = np.abs(dense.astype(np.int64))
    for d in range(3):
        assert np.all(np.isin(mags[d::3], C[:, d].astype(np.int64)))


def test_encode_argument_checks():
    C = torch.zeros((32, 3), dtype=torch.int8, device=dev())
    w = torch.zeros((6, 24), dtype=torch.bfloat16, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:                # K % 16 != 0
        s3d8.encode(w, C)
    assert e.value.status == -1
    buf = torch.zeros((6 * 32 + 8,), dtype=torch.bfloat16, device=dev())
    w = buf[1:1 + 6 * 32].view(6, 32)                       # not 16-byte aligned
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.encode(w, C)
    assert e.value.status == -2
    w = torch.zeros((0, 32), dtype=torch.bfloat16, device=dev())
    p, cs = s3d8.encode(w, C)                               # empty: nothing launched
    assert p.shape == (0, 32) and cs.shape == (0,)
    w = torch.zeros((6, 32), dtype=torch.bfloat16, device=dev())
    small = torch.zeros((s3d8.ENCODE_WORKSPACE_BYTES - 16,), dtype=torch.uint8, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.encode(w, C, workspace=small)
    assert e.value.status == -6


def test_scaled_magnitude_is_the_ieee_quotient():
    # Every finite bf16 x against every bf16 significand of alpha at three
    # exponents, and alphas at the edges of the fast path's range (2^-50,
    # 2^50) and just outside it, subnormal and tiny: the device quotient must
    # equal numpy's IEEE fp32 division bit for bit wherever |x| <= 2^20 alpha.
    xs = np.arange(0x10000, dtype=np.uint32)
    xs = xs[(xs & 0x7F80) != 0x7F80].astype(np.uint16)         # finite only
    sig = np.arange(128, dtype=np.uint32)
    alphas = [((127 + e) << 7) | sig for e in (0, -9, 6)]
    alphas.append(np.array([0x0001, 0x0040, 0x0080, 0x0D80, 0x0E00, 0x0E01, 0x3F80,
                            0x6580, 0x6600, 0x6601, 0x7F00, 0x7F7F], np.uint32))
    alphas = np.concatenate(alphas).astype(np.uint16)
    ax = np.abs(si.bf16_bits_to_f32(xs)).astype(np.float64)
    X, A = [], []
    for a in alphas:
        af = float(si.bf16_bits_to_f32(np.array([a], np.uint16))[0])
        keep = xs[ax <= af * 2.0 ** 20]
        X.append(keep)
        A.append(np.full(keep.shape, a, np.uint16))
    X = np.concatenate(X)
    A = np.concatenate(A)
    got = to_np(s3d8.selftest_scaled_abs(bf16_bits(X), bf16_bits(A)))
    want = np.abs(si.bf16_bits_to_f32(X)) / si.bf16_bits_to_f32(A)   # fp32 / fp32, IEEE
    assert want.dtype == np.float32 and X.size > 4_000_000
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (bad.size, X[bad[:4]], A[bad[:4]], got[bad[:4]], want[bad[:4]])
    zero = to_np(s3d8.selftest_scaled_abs(bf16_bits(xs[:1000]), bf16_bits(np.zeros(1000, np.uint16))))
    assert np.all(zero == 0)


# --------------------------------------------------------------------------
# QAT fake-quant forward (s3d8_fake_quant) and its straight-through backward
# --------------------------------------------------------------------------

def run_fake_quant(w_bits, C):
    w_hat, cs = s3d8.fake_quant(bf16_bits(w_bits), i8(C))
    torch.cuda.synchronize()
    return (to_np(w_hat.view(torch.int16)).view(np.uint16),
            to_np(cs.view(torch.int16)).view(np.uint16))


@pytest.mark.parametrize("N,K,seed", [(3, 16, 0), (1, 16, 1), (2, 32, 2), (5, 4096, 4),
                                      (241, 1040, 6), (1024, 4096, 8)])
def test_fake_quant_matches_oracle(N, K, seed):
    rng = np.random.default_rng(50 + seed)
    w = weights(rng, N, K)
    C = si.centroids(rng)
    got_w, got_s = run_fake_quant(w, C)
    want_s = oracle.encode(w, C)[1]
    assert np.array_equal(got_s, want_s)
    want_w = oracle.fake_quant(w, C)
    bad = np.argwhere(got_w != want_w)
    assert bad.size == 0, bad[:4]


def test_fake_quant_zero_channels_and_negative_zero():
    rng = np.random.default_rng(60)
    w = weights(rng, 12, 64)
    w[4] = 0
    w[7] = 0x8000                     # a whole channel of -0
    w[9, 3] = 0x8000
    C = si.centroids(rng)
    C[5] = 0
    got_w, _ = run_fake_quant(w, C)
    assert np.array_equal(got_w, oracle.fake_quant(w, C))


def test_fake_quant_straight_through_gradient():
    # forward uses Q(theta); the gradient reaching theta is the gradient with
    # respect to Q(theta), unchanged
    rng = np.random.default_rng(61)
    N, K, M = 48, 256, 8
    theta = bf16_bits(weights(rng, N, K)).requires_grad_(True)
    C = i8(si.centroids(rng))
    x = torch.randn((M, K), device=dev()).to(torch.bfloat16)
    r = torch.randn((M, N), device=dev()).to(torch.bfloat16)
    w_hat = s3d8.FakeQuantSTE.apply(theta, C)
    (x @ w_hat.t() * r).float().sum().backward()
    leaf = s3d8.fake_quant(theta.detach(), C)[0].requires_grad_(True)
    (x @ leaf.t() * r).float().sum().backward()
    assert torch.equal(theta.grad, leaf.grad)
    assert torch.equal(w_hat.detach(), leaf.detach())


def test_fake_quant_argument_checks():
    C = torch.zeros((32, 3), dtype=torch.int8, device=dev())
    w = torch.zeros((6, 24), dtype=torch.bfloat16, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.fake_quant(w, C)
    assert e.value.status == -1
    w = torch.zeros((6, 32), dtype=torch.bfloat16, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.fake_quant(w, C, workspace=torch.zeros((64,), dtype=torch.uint8, device=dev()))
    assert e.value.status == -6
