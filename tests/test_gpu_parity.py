"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bar: activation codes and scales, decoded int8 weights and int32 accumulators
bit-exact; bf16 outputs within |gpu - ref| <= 1e-3 + 1e-2 |ref| of the fp64
oracle.  Inputs follow the seeded recipe in s3d8_inputs; the oracle never sees
anything the GPU produced.
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import (assert_out_close, bf16_bits, bf16_to_f64, dev, f32, guarded, i8, to_np,
                      u8)

pytestmark = pytest.mark.gpu

ALGOS = [s3d8.ALGO_GEMV, s3d8.ALGO_TC, s3d8.ALGO_TMEM]
MAX_M = {s3d8.ALGO_TMEM: 64}   # token limits of the bounded algorithms
ALGO_IDS = {s3d8.ALGO_AUTO: "auto", s3d8.ALGO_GEMV: "gemv", s3d8.ALGO_SKINNY: "skinny",
            s3d8.ALGO_TC: "tc", s3d8.ALGO_TMEM: "tmem"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def rand_case(M, N, K, seed, outliers=False):
    rng = np.random.default_rng(seed)
    C = si.centroids(rng)
    packed = si.packed_bytes(rng, si.groups(N), K)
    cs = si.chan_scale(rng, N)
    x = si.activations(rng, M, K, outliers)
    return C, packed, cs, x


def gpu_linear(C, packed, cs, xq, xs, N, algo):
    return s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs), N, algo=algo)


def gpu_acc(C, packed, xq, N, algo):
    return to_np(s3d8.linear_acc_i32(u8(packed), i8(C), i8(xq), N, algo=algo)).astype(np.int64)


# --------------------------------------------------------------------------
# Activation quantisation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,outliers", [(4, 256, False), (1, 16, False), (3, 48, False),
                                          (1, 4096, False), (1, 14336, False), (7, 1040, True),
                                          (64, 14336, True), (2048, 14336, False),
                                          # both sides of each row-width class of the
                                          # standalone kernel (2048 / 4096 / 8192 / 16384
                                          # columns held in registers, longer rows two-pass)
                                          (2, 2048, False), (3, 2064, True), (2, 8192, True),
                                          (3, 8208, False), (3, 16384, True), (2, 16400, True),
                                          (2, 40960, False)])
def test_quantize_act_bitexact(M, K, outliers):
    rng = np.random.default_rng(M * 7 + K)
    x = si.activations(rng, M, K, outliers)
    if M > 2:
        x[1] = 0                      # an all-zero row
    xq_o, xs_o = oracle.quantize_act(x)
    xq, xs = s3d8.quantize_act(bf16_bits(x))
    np.testing.assert_array_equal(to_np(xs), xs_o)
    np.testing.assert_array_equal(to_np(xq), xq_o)


def _all_bf16_up_to(amax_bits):
    # every finite bf16 value with |x| <= bf16(amax), both signs, plus amax itself
    pos = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    pos = pos[si.bf16_bits_to_f32(pos) <= si.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0]]
    vals = np.concatenate([pos, pos | np.uint16(0x8000), np.array([amax_bits], np.uint16)])
    pad = (-len(vals)) % 16
    return np.concatenate([vals, np.zeros(pad, np.uint16)])


@pytest.mark.parametrize("amax", [1.0, 3.7, 127.0, 0.0078125, 6.0e-31, 2.5e35, 1.0e-38])
def test_quantize_exhaustive_bf16(amax):
    """Every bf16 value below a row's absmax, through both GPU quantisers (the
    standalone kernel and the one fused into the grouped linear launch)."""
    a_bits = int(si.f32_to_bf16_bits(np.array([amax], np.float32))[0])
    row = _all_bf16_up_to(a_bits)[None, :]
    xq_o, xs_o = oracle.quantize_act(row)
    xq, xs = s3d8.quantize_act(bf16_bits(row))
    np.testing.assert_array_equal(to_np(xs), xs_o)
    np.testing.assert_array_equal(to_np(xq), xq_o)
    # fused path: slices of at most 28672 values that all contain the absmax
    rng = np.random.default_rng(a_bits)
    vals = row[0]
    C = si.centroids(rng)
    for start in range(0, vals.size, 28656):
        part = np.concatenate([vals[start:start + 28656], np.array([a_bits], np.uint16)])
        part = np.concatenate([part, np.zeros((-part.size) % 16, np.uint16)])[None, :]
        K = part.shape[1]
        pq_o, ps_o = oracle.quantize_act(part)
        xq_out = torch.empty((1, K), dtype=torch.int8, device=dev())
        xs_out = torch.empty((1,), dtype=torch.float32, device=dev())
        N = 3
        packed = si.packed_bytes(rng, 1, K)
        s3d8.linear_batch([dict(packed=u8(packed), centroids=i8(C), chan_scale=bf16_bits(
            si.chan_scale(rng, N)), N=N, x=bf16_bits(part), xq_out=xq_out, xscale_out=xs_out)], 1)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np(xs_out), ps_o)
        np.testing.assert_array_equal(to_np(xq_out), pq_o)


def test_quantize_act_ties_and_guards():
    # absmax 127 gives a unit scale: halves round to even
    vals = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, 126.5, 0.0, -127.0, 64.0, 1.0, -1.0,
            0.25, 0.75]
    x = si.f32_to_bf16_bits(np.array([vals], np.float32))
    xq_o, xs_o = oracle.quantize_act(x)
    xq, check_q = guarded((1, 16), torch.int8, 99)
    xs, check_s = guarded((1,), torch.float32, -7.0)
    s3d8.quantize_act(bf16_bits(x), xq, xs)
    torch.cuda.synchronize()
    check_q()
    check_s()
    np.testing.assert_array_equal(to_np(xq), xq_o)
    assert to_np(xs)[0] == 1.0


# --------------------------------------------------------------------------
# Standalone unpack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(96, 256), (1, 16), (2, 32), (4, 48), (5, 64), (7, 1040),
                                 (1024, 4096), (14336, 4096), (4096, 14336)])
def test_decode_bitexact(N, K):
    rng = np.random.default_rng(N + K)
    C = si.centroids(rng)
    packed = si.packed_bytes(rng, si.groups(N), K)
    want = oracle.decode(packed, C, N)
    w, check = guarded((N, K), torch.int8, 77)
    s3d8.decode(u8(packed), i8(C), N, w)
    torch.cuda.synchronize()
    check()
    np.testing.assert_array_equal(to_np(w), want)


def test_decode_every_byte_every_table():
    """All 256 byte values against tables with 0 and 127 entries."""
    rng = np.random.default_rng(5)
    packed = np.tile(np.arange(256, dtype=np.uint8), (4, 1))   # 4 groups x 256 columns
    for C in (rng.integers(0, 128, (32, 3)).astype(np.int8), np.full((32, 3), 127, np.int8),
              np.zeros((32, 3), np.int8)):
        for N in (12, 11, 10):
            want = oracle.decode(packed, C, N)
            np.testing.assert_array_equal(to_np(s3d8.decode(u8(packed), i8(C), N)), want)


# --------------------------------------------------------------------------
# Linear: exact int32 accumulators and bf16 output
# --------------------------------------------------------------------------

SMALL = [(1, 1, 16), (2, 2, 32), (3, 4, 48), (4, 96, 256), (5, 5, 256), (7, 100, 1040),
         (8, 33, 512), (9, 1000, 512), (16, 64, 2048), (17, 10, 64)]


@pytest.mark.parametrize("algo", ALGOS, ids=lambda a: ALGO_IDS[a])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_linear_small_exact(M, N, K, algo):
    C, packed, cs, x = rand_case(M, N, K, seed=M * 100003 + N * 101 + K)
    xq, xs = oracle.quantize_act(x)
    ref, acc_o = oracle.linear(packed, C, cs, xq, xs, N)
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, N, algo), acc_o)
    out, check = guarded((M, N), torch.bfloat16, 3.0)
    s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs), N, out=out, algo=algo)
    torch.cuda.synchronize()
    check()
    assert_out_close(bf16_to_f64(out), ref)


@pytest.mark.parametrize("algo", ALGOS, ids=lambda a: ALGO_IDS[a])
def test_tiny_config(algo):
    """K=256, N=96, M=4 with the seeded recipe (the small case)."""
    mat, x = si.tiny_case(0)
    xq, xs = oracle.quantize_act(x)
    ref, acc_o = oracle.linear(mat.packed, mat.C, mat.chan_scale, xq, xs, mat.N)
    np.testing.assert_array_equal(gpu_acc(mat.C, mat.packed, xq, mat.N, algo), acc_o)
    assert_out_close(bf16_to_f64(gpu_linear(mat.C, mat.packed, mat.chan_scale, xq, xs, mat.N, algo)),
                     ref)


def _plain_linear(packed, C, cs, xq, xs, N):
    """out through the exported s3d8_linear symbol itself, called with ctypes
    (workspace sized by s3d8_linear_workspace_size with the automatic choice)."""
    M, K = xq.shape
    lib = s3d8.load()
    need = int(lib.s3d8_linear_workspace_size(M, N, K, s3d8.ALGO_AUTO))
    ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev())
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    st = lib.s3d8_linear(packed.data_ptr(), C.data_ptr(), cs.data_ptr(), xq.data_ptr(),
                         xs.data_ptr(), M, N, K, out.data_ptr(), ws.data_ptr() if need else None,
                         need, torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.s3d8_status_string(st)
    return out


def test_plain_entry_point_s3d8_linear():
    """The literal boundary call s3d8_linear on the small case (K=256, N=96,
    M=4) and on two projections of an 11B layer at M = 1 (gate 4096 -> 14336,
    down 14336 -> 4096): within tolerance of the oracle, and bit for bit equal
    to s3d8_linear_ex with the automatic algorithm."""
    mat, x = si.tiny_case(0)
    cases = [(mat, x)]
    for m in si.layer_matrices(layer=0, seed=0):
        if m.name in ("gate", "down"):
            cases.append((m, si.acts(1, m.K, seed=0, index=len(cases))))
    for mat, x in cases:
        xq, xs = oracle.quantize_act(x)
        ref, _ = oracle.linear(mat.packed, mat.C, mat.chan_scale, xq, xs, mat.N)
        args = (u8(mat.packed), i8(mat.C), bf16_bits(mat.chan_scale), i8(xq), f32(xs))
        got = _plain_linear(*args, mat.N)
        ex = torch.empty_like(got)
        M, K = xq.shape
        ws = torch.empty((max(1, s3d8.workspace_size(M, mat.N, K)),), dtype=torch.uint8, device=dev())
        st = s3d8.load().s3d8_linear_ex(*(a.data_ptr() for a in args), M, mat.N, K, ex.data_ptr(),
                                        ws.data_ptr(), ws.numel(), s3d8.ALGO_AUTO,
                                        torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(got), ref)
        np.testing.assert_array_equal(to_np(got.view(torch.int16)), to_np(ex.view(torch.int16)))


@pytest.mark.parametrize("algo", [s3d8.ALGO_AUTO] + ALGOS, ids=lambda a: ALGO_IDS[a])
def test_llama_layer_decode_m1_full(algo):
    """Every projection of one 11B decoder layer at M = 1, compared in full."""
    for i, mat in enumerate(si.layer_matrices(layer=0, seed=0)):
        x = si.acts(1, mat.K, seed=0, index=i)
        xq, xs = oracle.quantize_act(x)
        ref, acc_o = oracle.linear(mat.packed, mat.C, mat.chan_scale, xq, xs, mat.N)
        np.testing.assert_array_equal(gpu_acc(mat.C, mat.packed, xq, mat.N, algo), acc_o,
                                      err_msg=mat.name)
        got = bf16_to_f64(gpu_linear(mat.C, mat.packed, mat.chan_scale, xq, xs, mat.N, algo))
        assert_out_close(got, ref)


def sample_positions(M, N, rng, count=1500):
    ms = list(rng.integers(0, M, count)) + [0, 0, M - 1, M - 1, M // 2]
    ns = list(rng.integers(0, N, count)) + [0, N - 1, 0, N - 1, N - 2]
    return np.array(ms, np.int64), np.array(ns, np.int64)


@pytest.mark.parametrize("algo", [s3d8.ALGO_AUTO] + ALGOS, ids=lambda a: ALGO_IDS[a])
@pytest.mark.parametrize("M", list(si.DECODE_SWEEP_M) + list(si.PREFILL_M))
@pytest.mark.parametrize("shape", si.SWEEP_SHAPES, ids=lambda s: s[0])
def test_sweep_sampled(shape, M, algo):
    """Batched decode (with 1 % activation outliers) and prefill sizes at full
    shape; the oracle computes a sample of outputs one by one."""
    if M > MAX_M.get(algo, M):
        pytest.skip(f"{ALGO_IDS[algo]} takes up to {MAX_M[algo]} tokens")
    name, K, N = shape
    mat = si.matrix(name, K, N, seed=2)
    x = si.acts(M, K, seed=2, outliers=M <= 64)
    xq, xs = oracle.quantize_act(x)
    acc = gpu_acc(mat.C, mat.packed, xq, N, algo)
    out = bf16_to_f64(gpu_linear(mat.C, mat.packed, mat.chan_scale, xq, xs, N, algo))
    rng = np.random.default_rng(M)
    ms, ns = sample_positions(M, N, rng)
    want = oracle.linear_acc_at(mat.packed, mat.C, xq, N, ms, ns)
    np.testing.assert_array_equal(acc[ms, ns], want)
    ref = xs.astype(np.float64)[ms] * want * si.bf16_bits_to_f32(mat.chan_scale).astype(
        np.float64)[ns]
    assert_out_close(out[ms, ns], ref)
    # property at any size: the bf16 output is the epilogue of the exact accumulators
    csf = si.bf16_bits_to_f32(mat.chan_scale).astype(np.float64)
    full_ref = xs.astype(np.float64)[:, None] * acc * csf[None, :]
    assert_out_close(out, full_ref)


@pytest.mark.parametrize("algo", ALGOS, ids=lambda a: ALGO_IDS[a])
@pytest.mark.parametrize("K", [16, 4096, 14336])
def test_int32_extremes(K, algo):
    """All centroids 127, all codes 127: acc = +-16129 K (231,225,344 at K = 14336)."""
    C = np.full((32, 3), 127, np.int8)
    M, N = 3, 8
    G = si.groups(N)
    pos = oracle.pack_byte(9, 0, 0, 0)
    packed = np.full((G, K), pos, np.uint8)
    packed[1] ^= 0x41                 # group 1: all three weights negative
    packed[2] ^= 0x80                 # group 2: only component 2 negative
    xq = np.full((M, K), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127                 # alternating signs
    acc_o, bad = oracle.linear_acc(packed, C, xq, N)
    assert bad == 0
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, N, algo), acc_o)
    assert acc_o[0, 0] == 16129 * K and acc_o[0, 3] == -16129 * K


@pytest.mark.parametrize("M", [3, 40])
def test_tmem_int32_extremes_across_chunks(M):
    """The tensor-memory path at the int32 edge with tiles of many 1024-column
    chunks (100 row tiles leave one K range per tile: 14 chunk sums carried in
    int32 up to 16129 * 14336 = 231,225,344; with 40 tokens the K ranges are
    capped at one chunk and the CTAs walk several tiles).  Every weight is +-127
    with one sign per packed row, so acc[m, 3g + d] = sign(g) * 127 * sum_k xq[m, k]
    in closed form; a sample is also checked against the oracle."""
    C = np.full((32, 3), 127, np.int8)
    K, N = 14336, 3 * 128 * 100
    G = si.groups(N)
    packed = np.full((G, K), oracle.pack_byte(9, 0, 0, 0), np.uint8)
    packed[1::7] ^= 0x41              # every 7th packed row: all three weights negative
    xq = np.full((M, K), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127                 # alternating signs: row sum 0
    sign = np.ones(G, np.int64)
    sign[1::7] = -1
    want = 127 * xq.astype(np.int64).sum(axis=1)[:, None] * np.repeat(sign, 3)[None, :N]
    got = gpu_acc(C, packed, xq, N, s3d8.ALGO_TMEM)
    np.testing.assert_array_equal(got, want)
    assert want[0, 0] == 16129 * K and want[0, 3] == -16129 * K
    rng = np.random.default_rng(M)
    ms, ns = sample_positions(M, N, rng, count=200)
    np.testing.assert_array_equal(got[ms, ns], oracle.linear_acc_at(packed, C, xq, N, ms, ns))


@pytest.mark.parametrize("algo", ALGOS, ids=lambda a: ALGO_IDS[a])
def test_zero_activation_row_gives_zero(algo):
    C, packed, cs, x = rand_case(3, 30, 64, seed=4)
    x[1] = 0
    xq, xs = oracle.quantize_act(x)
    out = to_np(gpu_linear(C, packed, cs, xq, xs, 30, algo).float())
    assert (out[1] == 0).all()


TC_TILES = [(128, 240, 64), (129, 241, 1040), (300, 722, 2112), (256, 480, 3072),
            (1, 3, 16), (17, 1201, 1024),
            # from 384 tokens two SMs share each 256-token tile (240 or 192
            # channels, each SM decoding its 40 or 32 packed rows, fp16); from 1537
            # tokens on rows of up to 8192 columns and from 2049 on longer rows,
            # 256 channels of weights expanded to bf16 first: the odd SM's rows
            # past M, partial pair tiles, one K block, split and unsplit K, both
            # sides of both boundaries
            (384, 241, 1040), (520, 722, 2112), (768, 480, 3072), (400, 3, 16),
            (1000, 1201, 4096), (2048, 96, 14336), (640, 257, 1024), (512, 512, 2048),
            (768, 722, 2112), (769, 241, 1040), (1024, 96, 14336), (1025, 96, 14336),
            (1023, 722, 2112), (1024, 241, 1040), (1300, 3, 64),
            (1536, 241, 1040), (1537, 241, 1040), (2049, 96, 14336), (1700, 3, 64),
            # expanded-weight tiles narrower than 256 channels (192 and 128: each
            # drain thread writes 96 or 64 columns) with 16-byte aligned rows
            (1600, 1344, 128), (1600, 1024, 64)]


@pytest.mark.parametrize("M,N,K", TC_TILES)
def test_tc_tiles_and_tails(M, N, K):
    """Tensor-core path in full against the oracle: whole and ragged 128-token and
    240-channel tiles, K ragged against the 64-column block and the 1024-column
    exact chunk, on one SM per tile (small M) and on SM pairs (M >= 384:
    decoding the weight tiles inside the GEMM below 1537 tokens, or 2049 on rows
    longer than 8192 columns; on weights expanded to bf16 first above)."""
    C, packed, cs, x = rand_case(M, N, K, seed=M * 7919 + N * 31 + K)
    xq, xs = oracle.quantize_act(x)
    ref, acc_o = oracle.linear(packed, C, cs, xq, xs, N)
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, N, s3d8.ALGO_TC), acc_o)
    out, check = guarded((M, N), torch.bfloat16, 3.0)
    s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs), N, out=out, algo=s3d8.ALGO_TC)
    torch.cuda.synchronize()
    check()
    assert_out_close(bf16_to_f64(out), ref)


def test_retired_algorithm_value_is_rejected():
    """Algorithm value 2 (the retired register-fragment path) returns
    S3D8_ERR_UNSUPPORTED before any launch."""
    C, packed, cs, x = rand_case(16, 9, 64, seed=9)
    xq, xs = oracle.quantize_act(x)
    with pytest.raises(s3d8.S3D8Error) as e:
        gpu_acc(C, packed, xq, 9, s3d8.ALGO_SKINNY)
    assert e.value.status == -3


# Tensor-memory path: 128-row tiles (ragged last tile, N not a multiple of 3),
# tiles of several 1024-column chunks (few K splits when there are many row
# tiles), more tiles than SMs (a second tile per CTA), K ragged against the
# 64-column block, and 1..64 tokens (N of the MMA 16..64).
TMEM_CASES = [(1, 4, 16), (5, 241, 1040), (16, 722, 2112), (17, 1201, 3088), (33, 96, 256),
              (64, 480, 14336), (8, 38401, 4096), (64, 61441, 256), (48, 3000, 1104),
              (64, 29569, 1088)]   # 231 row tiles, 17-block tiles: chunk sums in shared memory


@pytest.mark.parametrize("M,N,K", TMEM_CASES)
def test_tmem_in_full(M, N, K):
    C, packed, cs, x = rand_case(M, N, K, seed=M * 17 + N * 3 + K)
    xq, xs = oracle.quantize_act(x)
    ref, acc_o = oracle.linear(packed, C, cs, xq, xs, N)
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, N, s3d8.ALGO_TMEM), acc_o)
    out, check = guarded((M, N), torch.bfloat16, 3.0, pad=65)
    s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs), N, out=out, algo=s3d8.ALGO_TMEM)
    torch.cuda.synchronize()
    check()
    assert_out_close(bf16_to_f64(out), ref)


def test_tmem_rejects_more_than_64_tokens():
    C, packed, cs, x = rand_case(65, 9, 64, seed=10)
    xq, xs = oracle.quantize_act(x)
    with pytest.raises(s3d8.S3D8Error) as e:
        gpu_acc(C, packed, xq, 9, s3d8.ALGO_TMEM)
    assert e.value.status == -3


@pytest.mark.parametrize("M", [130, 390, 1100])
def test_tc_unaligned_outputs(M):
    """Output views that are only 2- (bf16) or 4-byte (int32) aligned take the
    scalar store path and still match (one-SM and both SM-pair kernels)."""
    N, K = 480, 256
    C, packed, cs, x = rand_case(M, N, K, seed=5)
    xq, xs = oracle.quantize_act(x)
    ref, acc_o = oracle.linear(packed, C, cs, xq, xs, N)
    out, check = guarded((M, N), torch.bfloat16, 3.0, pad=65)
    s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs), N, out=out, algo=s3d8.ALGO_TC)
    acc, check_acc = guarded((M, N), torch.int32, 7, pad=33)
    s3d8.linear_acc_i32(u8(packed), i8(C), i8(xq), N, algo=s3d8.ALGO_TC, acc=acc)
    torch.cuda.synchronize()
    check()
    check_acc()
    assert_out_close(bf16_to_f64(out), ref)
    np.testing.assert_array_equal(to_np(acc).astype(np.int64), acc_o)


@pytest.mark.parametrize("M", [200, 400, 1030])
def test_tc_adversarial_chunk_sums(M):
    """Every product +16129 over 1024 columns is the largest partial sum an exact
    fp32 chunk holds (16,516,096 < 2^24); two chunks in a row must still add
    exactly in int32 (K = 2048 + 1024 + 16).  One SM per tile (200 tokens), SM
    pairs decoding packed tiles (400) and SM pairs on expanded weights (1030)."""
    C = np.full((32, 3), 127, np.int8)
    N, K = 243, 3088
    packed = np.full((si.groups(N), K), oracle.pack_byte(3, 0, 0, 0), np.uint8)
    xq = np.full((M, K), 127, np.int8)
    xq[1::2, 1024:2048] = -127        # odd rows: the middle chunk cancels the first
    acc_o, bad = oracle.linear_acc(packed, C, xq, N)
    assert bad == 0
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, N, s3d8.ALGO_TC), acc_o)
    assert acc_o[0, 0] == 16129 * K


def test_empty_and_rejected_calls():
    packed = torch.zeros((2, 32), dtype=torch.uint8, device=dev())
    C = torch.zeros((32, 3), dtype=torch.int8, device=dev())
    cs = torch.zeros((5,), dtype=torch.bfloat16, device=dev())
    xq = torch.zeros((0, 32), dtype=torch.int8, device=dev())
    xs = torch.zeros((0,), dtype=torch.float32, device=dev())
    out = s3d8.linear(packed, C, cs, xq, xs, 5)
    assert out.shape == (0, 5)
    # misaligned packed (1-byte offset view) is rejected before any launch
    big = torch.zeros((2 * 32 + 16,), dtype=torch.uint8, device=dev())
    mis = big[1:1 + 64].view(2, 32)
    xq1 = torch.zeros((1, 32), dtype=torch.int8, device=dev())
    xs1 = torch.ones((1,), dtype=torch.float32, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.linear(mis, C, cs, xq1, xs1, 5)
    assert e.value.status == -2
    # K not a multiple of 16
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.linear(torch.zeros((2, 24), dtype=torch.uint8, device=dev()), C, cs,
                    torch.zeros((1, 24), dtype=torch.int8, device=dev()), xs1, 5)
    assert e.value.status == -1
    assert s3d8.device_status() == 0


def test_bounded_wait_reports_timeout_and_recovers():
    """A wait that nothing completes ends with S3D8_ERR_TIMEOUT in the status
    word (no fault, no hang); the status clears on read and work continues."""
    assert s3d8.device_status() == 0
    s3d8.selftest_wait_timeout(2000)
    assert s3d8.device_status() == -5
    assert s3d8.device_status() == 0
    C, packed, cs, x = rand_case(2, 9, 64, seed=77)
    xq, xs = oracle.quantize_act(x)
    _, acc_o = oracle.linear(packed, C, cs, xq, xs, 9)
    np.testing.assert_array_equal(gpu_acc(C, packed, xq, 9, s3d8.ALGO_GEMV), acc_o)
    assert s3d8.device_status() == 0
