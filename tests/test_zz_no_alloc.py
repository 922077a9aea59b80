"""The no-allocation tensor-core entry point, s3d8_linear_tc_noalloc.

Some callers cannot allocate device memory (code inside an allocator or pool
callback, a real-time loop that must not wait on the driver's allocator, a host
that owns all device memory).  This entry point serves them with a fixed
scratch array inside the library instead of caller workspace.  Its results
must match the fp64 oracle within the parity tolerance, and, since every path
sums the products exactly in int32 and applies the same bf16 epilogue, the
ordinary entry point (s3d8_linear_ex with the tensor-core algorithm) bit for
bit, call after call, although every call reuses the same scratch.  Shapes of
384 tokens and more are included: there the ordinary entry point runs an
SM-pair GEMM (decoding packed tiles itself, or on pre-expanded weights from
1537 tokens on these rows), while this one keeps the one-SM GEMM and that
kernel's own K-split plan.  Kept in a file that pytest collects last.
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import assert_out_close, bf16_bits, bf16_to_f64, dev, f32, i8, to_np, u8

pytestmark = pytest.mark.gpu

# Outputs the oracle checks one by one on shapes too large for a full product.
SAMPLES = 600


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def _case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    C = si.centroids(rng)
    packed = si.packed_bytes(rng, si.groups(N), K)
    cs = si.chan_scale(rng, N)
    xq, xs = oracle.quantize_act(si.activations(rng, M, K, False))
    return (packed, C, cs, xq, xs), (u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs))


def _check_with_oracle(host, got, M, N, full, seed):
    packed, C, cs, xq, xs = host
    if full:
        ref, _ = oracle.linear(packed, C, cs, xq, xs, N)
        assert_out_close(got, ref)
        return
    rng = np.random.default_rng(seed)
    ms = np.concatenate([[0, M - 1, M - 1, 0], rng.integers(0, M, SAMPLES)]).astype(np.int64)
    ns = np.concatenate([[0, N - 1, 0, N - 1], rng.integers(0, N, SAMPLES)]).astype(np.int64)
    acc = oracle.linear_acc_at(packed, C, xq, N, ms, ns)
    csf = si.bf16_bits_to_f32(cs).astype(np.float64)
    assert_out_close(got[ms, ns], xs.astype(np.float64)[ms] * acc * csf[ns])


# (M, N, K, compare with the oracle in full): the second of each pair is smaller
# than the first, so stale scratch from the first call sits beyond what the
# second one writes.  On the 152 SMs of a GB300, 512 x 96, 2047 x 481 and
# 384 x 2048 split K (int32 partials in the scratch); 2047 x 14336 does not.
CASES = [
    [(300, 722, 2112, True), (130, 481, 1040, True)],
    [(2047, 481, 4096, False), (512, 96, 4096, True)],
    [(2047, 14336, 4096, False), (384, 2048, 4096, False)],
]


@pytest.mark.parametrize("pair", CASES, ids=lambda p: "-".join(f"{c[0]}x{c[1]}x{c[2]}" for c in p))
def test_noalloc_matches_oracle_and_workspace_entry_on_consecutive_calls(pair):
    for i, (M, N, K, full) in enumerate(pair):
        host, (packed, C, cs, xq, xs) = _case(M, N, K, 11 + i + 7 * M)
        want = s3d8.linear(packed, C, cs, xq, xs, N, algo=s3d8.ALGO_TC)
        out = torch.full((M, N), 5.0, dtype=torch.bfloat16, device=dev())
        s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np(out.view(torch.int16)), to_np(want.view(torch.int16)))
        _check_with_oracle(host, bf16_to_f64(out), M, N, full, seed=M + N)


def test_noalloc_takes_no_device_memory():
    M, N, K = 256, 480, 4096
    host, (packed, C, cs, xq, xs) = _case(M, N, K, 13)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)   # first call does the set-up
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    _check_with_oracle(host, bf16_to_f64(out), M, N, True, seed=0)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    M, K, N = 4096, 4096, 3          # 2 M K + 256 bytes > 32 MiB
    assert 2 * M * K + 256 > s3d8.NOALLOC_SCRATCH_BYTES
    packed = torch.zeros((1, K), dtype=torch.uint8, device=dev())
    C = torch.zeros((32, 3), dtype=torch.int8, device=dev())
    cs = torch.ones((N,), dtype=torch.bfloat16, device=dev())
    xq = torch.zeros((M, K), dtype=torch.int8, device=dev())
    xs = torch.ones((M,), dtype=torch.float32, device=dev())
    out = torch.zeros((M, N), dtype=torch.bfloat16, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)
    assert e.value.status == -6
    assert bool((out == 0).all())
