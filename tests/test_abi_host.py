"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, export every entry point that
include/s3d8.h declares, and reject bad arguments before it makes any CUDA
call.  The rejection tests pass non-null dummy addresses that are never
dereferenced; they run only on a machine without a CUDA device so that no
code path can ever hand such an address to a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

import s3d8_a8_linear_gb300 as s3d8
from s3d8_a8_linear_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _has_cuda_device():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


no_device_only = pytest.mark.skipif(_has_cuda_device(),
                                    reason="dummy-pointer rejection tests run only without a GPU")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return s3d8.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "s3d8.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(s3d8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("s3d8_quantize_act", "s3d8_linear", "s3d8_decode", "s3d8_linear_ex",
               "s3d8_linear_acc_i32", "s3d8_linear_workspace_size", "s3d8_device_status",
               "s3d8_status_string", "s3d8_version", "s3d8_encode"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (s3d8_[a-z0-9_]+)$", out, flags=re.M))
    missing = [fn for fn in declared_functions() if fn not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for fn in declared_functions():
        getattr(lib, fn)


def test_debug_build_exports_the_same_symbols():
    """The debug-checks variant (in-kernel bounds checks) builds here and exports
    every declared entry point too."""
    path = _build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (s3d8_[a-z0-9_]+)$", out, flags=re.M))
    missing = [fn for fn in declared_functions() if fn not in exported]
    assert not missing, f"declared but not exported by the debug build: {missing}"


def test_status_strings(lib):
    for code, word in ((0, b"ok"), (-1, b"invalid"), (-2, b"misaligned"), (-3, b"unsupported"),
                       (-4, b"CUDA"), (-5, b"timed out"), (-6, b"workspace"), (-7, b"bounds")):
        assert word in lib.s3d8_status_string(code)
    assert lib.s3d8_version() >= 100


A16 = 0x10000        # dummy, 16-byte aligned, never dereferenced
A16B = 0x20000
A16C = 0x30000


@no_device_only
def test_linear_rejects_bad_shapes(lib):
    f = lib.s3d8_linear
    ok_ptrs = (A16, A16B, A16C, A16, A16B)
    for K in (0, 8, 15, 17, 100, 133145, -16):
        assert f(*ok_ptrs, 1, 3, K, A16C, None, 0, None) == -1, K
    assert f(*ok_ptrs, -1, 3, 16, A16C, None, 0, None) == -1
    assert f(*ok_ptrs, 1, -3, 16, A16C, None, 0, None) == -1
    assert f(*ok_ptrs, (1 << 24) + 1, 3, 16, A16C, None, 0, None) == -1


@no_device_only
def test_linear_rejects_null_and_misaligned(lib):
    f = lib.s3d8_linear
    base = [A16, A16B, A16C, A16, A16B]
    for i in range(5):
        args = list(base)
        args[i] = None
        assert f(*args, 2, 3, 32, A16C, None, 0, None) == -1, i
    assert f(*base, 2, 3, 32, None, None, 0, None) == -1
    mis = list(base)
    mis[0] = A16 + 8     # packed must be 16-byte aligned
    assert f(*mis, 2, 3, 32, A16C, None, 0, None) == -2
    mis = list(base)
    mis[3] = A16 + 4     # xq must be 16-byte aligned
    assert f(*mis, 2, 3, 32, A16C, None, 0, None) == -2
    mis = list(base)
    mis[4] = A16 + 2     # xscale must be 4-byte aligned
    assert f(*mis, 2, 3, 32, A16C, None, 0, None) == -2
    assert f(*base, 2, 3, 32, A16C + 1, None, 0, None) == -2


@no_device_only
def test_empty_calls_are_no_ops(lib):
    # M == 0 or N == 0 returns OK without touching any pointer (all NULL here)
    assert lib.s3d8_linear(None, None, None, None, None, 0, 3, 32, None, None, 0, None) == 0
    assert lib.s3d8_linear(None, None, None, None, None, 2, 0, 32, None, None, 0, None) == 0
    assert lib.s3d8_quantize_act(None, 0, 32, None, None, None) == 0
    assert lib.s3d8_decode(None, None, 0, 32, None, None) == 0
    assert lib.s3d8_linear_acc_i32(None, None, None, 0, 5, 32, None, None, 0, 0, None) == 0
    assert lib.s3d8_encode(None, None, 0, 32, None, None, None, 0, None) == 0
    assert lib.s3d8_selftest_scaled_abs(None, None, 0, None, None) == 0
    assert lib.s3d8_fake_quant(None, None, 0, 32, None, None, None, 0, None) == 0


@no_device_only
def test_other_entry_points_reject(lib):
    assert lib.s3d8_quantize_act(A16, 2, 24, A16B, A16C, None) == -1        # K % 16
    assert lib.s3d8_quantize_act(A16 + 2, 2, 32, A16B, A16C, None) == -2    # x alignment
    assert lib.s3d8_quantize_act(None, 2, 32, A16B, A16C, None) == -1
    assert lib.s3d8_decode(A16, A16B, 5, 20, A16C, None) == -1
    assert lib.s3d8_decode(A16 + 1, A16B, 5, 32, A16C, None) == -2
    assert lib.s3d8_decode(A16, A16B, 5, 32, A16C + 8, None) == -2
    assert lib.s3d8_linear_acc_i32(A16, A16B, A16C, 2, 5, 32, None, None, 0, 0, None) == -1
    assert lib.s3d8_linear_acc_i32(A16, A16B, A16C, 2, 5, 32, A16 + 2, None, 0, 0, None) == -2
    assert lib.s3d8_linear_ex(A16, A16B, A16C, A16, A16B, 2, 3, 32, A16C, None, 0, 7, None) == -1
    assert lib.s3d8_linear_ex(A16, A16B, A16C, A16, A16B, 2, 3, 32, A16C, None, 0, -1, None) == -1
    assert lib.s3d8_linear_ex(A16, A16B, A16C, A16, A16B, 2, 3, 32, A16C, None, 0, 5, None) == -1
    # the tensor-memory algorithm takes at most 64 tokens
    assert lib.s3d8_linear_ex(A16, A16B, A16C, A16, A16B, 65, 3, 32, A16C, None, 0, 4, None) == -3
    enc = lib.s3d8_encode
    WS = 16384
    assert enc(A16, A16B, 6, 24, A16C, A16, A16B, WS, None) == -1            # K % 16
    assert enc(A16, None, 6, 32, A16C, A16, A16B, WS, None) == -1
    assert enc(A16 + 8, A16B, 6, 32, A16C, A16, A16B, WS, None) == -2        # w alignment
    assert enc(A16, A16B, 6, 32, A16C + 4, A16, A16B, WS, None) == -2        # packed
    assert enc(A16, A16B, 6, 32, A16C, A16 + 1, A16B, WS, None) == -2        # scales
    assert enc(A16, A16B, 6, 32, A16C, A16, None, WS, None) == -6            # no workspace
    assert enc(A16, A16B, 6, 32, A16C, A16, A16B, WS - 1, None) == -6        # too small
    assert enc(A16, A16B, 6, 32, A16C, A16, A16B + 8, WS, None) == -2        # ws alignment
    fit = lib.s3d8_fit_centroids
    assert fit(A16, 6, 32, A16B, 1, A16C, A16, A16B, 16, None) == -6             # ws too small
    assert fit(A16, 0, 32, A16B, 1, A16C, A16, A16B, 1 << 30, None) == -1        # no points
    assert fit(A16, 6, 24, A16B, 1, A16C, A16, A16B, 1 << 30, None) == -1        # K % 16
    assert fit(A16, 6, 32, A16B, -1, A16C, A16, A16B, 1 << 30, None) == -1       # iters
    assert fit(A16, 6, 32, None, 1, A16C, A16, A16B, 1 << 30, None) == -1
    assert fit(A16 + 8, 6, 32, A16B, 1, A16C, A16, A16B, 1 << 30, None) == -2
    assert fit(A16, 6, 32, A16B, 1, A16C, A16, A16B + 16, 1 << 30, None) == -2   # ws alignment
    assert lib.s3d8_fit_workspace_size(6, 24) == 0
    fq = lib.s3d8_fake_quant
    assert fq(A16, A16B, 6, 24, A16C, A16, A16B, WS, None) == -1                # K % 16
    assert fq(A16, A16B, 6, 32, A16C + 8, A16, A16B, WS, None) == -2            # w_hat alignment
    assert fq(A16, A16B, 6, 32, A16C, A16, None, WS, None) == -6
    assert lib.s3d8_selftest_scaled_abs(A16, A16B, -1, A16C, None) == -1
    assert lib.s3d8_selftest_scaled_abs(A16 + 1, A16B, 4, A16C, None) == -2


def test_linear_workspace_sizes(lib):
    """Workspace of the tensor-memory decode GEMM: a 256-byte alignment pad and
    nsplit int32 partial sums [M, N], for some split count 1..K/64 (it depends
    on the SM count; the kernel reads the int8 codes themselves); no workspace
    past 64 tokens or for the 8-token GEMV, and the automatic choice takes it
    for 16 tokens on a 14336 x 4096 matrix."""
    ws = lib.s3d8_linear_workspace_size
    M, N, K = 16, 14336, 4096
    t = ws(M, N, K, 4)
    rest = t - 256
    assert rest > 0 and rest % (M * N * 4) == 0 and 1 <= rest // (M * N * 4) <= K // 64
    assert ws(M, N, K, 0) == t
    assert ws(65, 9, 64, 4) == 0
    assert ws(8, N, K, 1) == 0
    assert ws(0, N, K, 0) == 0 and ws(M, N, 0, 0) == 0
    assert ws(64, 4096, 14336, 4) > 0


def test_tc_workspace_marks_the_weight_expansion(lib):
    """The tensor-core workspace holds a 16-bit copy of the weights [N, K] only
    where the path expands them first: from 1537 tokens on rows of up to 8192
    columns, from 2049 on longer rows (below, the SM pairs decode the packed
    tiles inside the GEMM); the 16-bit activation copy grows with M throughout."""
    ws = lib.s3d8_linear_workspace_size
    for N, K, last_fused in ((14336, 4096, 1536), (4096, 14336, 2048), (14336, 8192, 1536), (14336, 8208, 2048)):
        before, after = ws(last_fused, N, K, 3), ws(last_fused + 1, N, K, 3)
        assert before < N * K * 2 + last_fused * K * 2, (N, K)
        assert after >= N * K * 2 + (last_fused + 1) * K * 2, (N, K)
        assert ws(384, N, K, 3) < N * K * 2


def test_binding_refuses_cpu_tensors(lib):
    import torch

    packed = torch.zeros((1, 16), dtype=torch.uint8)
    C = torch.zeros((32, 3), dtype=torch.int8)
    with pytest.raises(ValueError):
        s3d8.decode(packed, C, 3)


@no_device_only
def test_batch_rejects(lib):
    job = s3d8.LinearJob()
    job.packed, job.centroids, job.chan_scale_bf16, job.xq = A16, A16B, A16C, A16
    job.xscale, job.out_bf16, job.N, job.K = A16B, A16C, 3, 32
    arr = (s3d8.LinearJob * 9)(*([job] * 9))
    assert lib.s3d8_linear_batch(arr, 9, 1, None) == -1          # more than 8 jobs
    assert lib.s3d8_linear_batch(None, 2, 1, None) == -1
    assert lib.s3d8_linear_batch(arr, 2, 9, None) == -3          # M > 8
    assert lib.s3d8_linear_batch(arr, 0, 1, None) == 0
    assert lib.s3d8_linear_batch(arr, 2, 0, None) == 0
    both = s3d8.LinearJob.from_buffer_copy(job)
    both.x_bf16 = A16
    assert lib.s3d8_linear_batch((s3d8.LinearJob * 1)(both), 1, 1, None) == -1   # x and xq
    bad_k = s3d8.LinearJob.from_buffer_copy(job)
    bad_k.K = 40
    assert lib.s3d8_linear_batch((s3d8.LinearJob * 1)(bad_k), 1, 1, None) == -1
    mis = s3d8.LinearJob.from_buffer_copy(job)
    mis.packed = A16 + 4
    assert lib.s3d8_linear_batch((s3d8.LinearJob * 1)(mis), 1, 1, None) == -2
