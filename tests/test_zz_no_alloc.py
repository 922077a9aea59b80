"""The no-allocation tensor-core entry point, s3d8_linear_tc_noalloc.

Some callers cannot allocate device memory (code inside an allocator or pool
callback, a real-time loop that must not wait on the driver's allocator, a host
that owns all device memory).  This entry point serves them with a fixed
scratch array inside the library instead of caller workspace.  Its results
must match the ordinary entry point (s3d8_linear_ex with the tensor-core
algorithm) within the parity tolerance, call after call, although every call
reuses the same scratch.  Kept in a file that pytest collects last.
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import assert_out_close, bf16_bits, bf16_to_f64, dev, f32, i8, u8

pytestmark = pytest.mark.gpu


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
    return u8(packed), i8(C), bf16_bits(cs), i8(xq), f32(xs)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    # the second call is smaller than the first, so stale scratch from the first
    # call sits beyond what the second one writes
    for M, N, K, seed in [(300, 722, 2112, 11), (130, 481, 1040, 12)]:
        packed, C, cs, xq, xs = _case(M, N, K, seed)
        want = s3d8.linear(packed, C, cs, xq, xs, N, algo=s3d8.ALGO_TC)
        out = torch.full((M, N), 5.0, dtype=torch.bfloat16, device=dev())
        s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)
        torch.cuda.synchronize()
        assert_out_close(bf16_to_f64(out), bf16_to_f64(want))


def test_noalloc_takes_no_device_memory():
    M, N, K = 256, 480, 4096
    packed, C, cs, xq, xs = _case(M, N, K, 13)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)   # first call does the set-up
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        s3d8.linear_tc_noalloc(packed, C, cs, xq, xs, N, out)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    want = s3d8.linear(packed, C, cs, xq, xs, N, algo=s3d8.ALGO_TC)
    assert_out_close(bf16_to_f64(out), bf16_to_f64(want))


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
