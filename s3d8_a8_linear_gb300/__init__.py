"""GB300 (sm_103a) S3D8 W2.7A8 linear layer: thin Python binding.

Every step of the layer runs in the CUDA library ``_build/libs3d8.so`` behind
the C ABI of ``include/s3d8.h``; this module only checks tensor dtypes,
shapes and devices, and passes raw device pointers and the current CUDA
stream.  There is no CPU or PyTorch fallback: if the library has not been
built, every call raises.

Format: "11 billion parameters on a phone" (Graphcore Research blog),
sections "Bit layout" and "Output channel packing"; math: "Llama-Mobile:
Efficient 2.7-Bit Quantization of VLMs", section 3.4, Eq. 1.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

ALGO_AUTO, ALGO_GEMV, ALGO_SKINNY, ALGO_TC, ALGO_TMEM = 0, 1, 2, 3, 4

STATUS = {
    0: "ok",
    -1: "invalid argument",
    -2: "misaligned pointer",
    -3: "unsupported",
    -4: "CUDA error",
    -5: "timeout",
    -6: "workspace",
    -7: "bounds check failed (debug build)",
}

_lib = None

MAX_BATCH = 8


class LinearJob(ctypes.Structure):
    """Mirror of s3d8_linear_job (include/s3d8.h)."""
    _fields_ = [("packed", ctypes.c_void_p), ("centroids", ctypes.c_void_p),
                ("chan_scale_bf16", ctypes.c_void_p), ("x_bf16", ctypes.c_void_p),
                ("xq", ctypes.c_void_p), ("xscale", ctypes.c_void_p), ("xq_out", ctypes.c_void_p),
                ("xscale_out", ctypes.c_void_p), ("out_bf16", ctypes.c_void_p),
                ("acc", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class S3D8Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status} ({msg})")
        self.status = status


def _debug_variant() -> bool:
    """S3D8_LIBRARY=debug selects the build with in-kernel bounds checks."""
    return os.environ.get("S3D8_LIBRARY", "") == "debug"


def library_path() -> str:
    return _build.DEBUG_LIB if _debug_variant() else _build.LIB


def load(build_if_missing: bool = False):
    """Load the CUDA library (optionally building it first)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing and not _debug_variant():
            raise RuntimeError(
                f"S3D8 CUDA library missing at {path}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        _build.build(debug=_debug_variant())
    L = ctypes.CDLL(path)
    P, I64, SZ, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    L.s3d8_quantize_act.argtypes = [P, I64, I64, P, P, P]
    L.s3d8_decode.argtypes = [P, P, I64, I64, P, P]
    L.s3d8_encode.argtypes = [P, P, I64, I64, P, P, P, SZ, P]
    L.s3d8_selftest_scaled_abs.argtypes = [P, P, I64, P, P]
    L.s3d8_fake_quant.argtypes = [P, P, I64, I64, P, P, P, SZ, P]
    L.s3d8_fit_workspace_size.argtypes = [I64, I64]
    L.s3d8_fit_workspace_size.restype = SZ
    L.s3d8_fit_centroids.argtypes = [P, I64, I64, P, ctypes.c_int32, P, P, P, SZ, P]
    L.s3d8_linear_workspace_size.argtypes = [I64, I64, I64, I]
    L.s3d8_linear_workspace_size.restype = SZ
    L.s3d8_linear.argtypes = [P, P, P, P, P, I64, I64, I64, P, P, SZ, P]
    L.s3d8_linear_ex.argtypes = [P, P, P, P, P, I64, I64, I64, P, P, SZ, I, P]
    L.s3d8_linear_acc_i32.argtypes = [P, P, P, I64, I64, I64, P, P, SZ, I, P]
    L.s3d8_linear_batch.argtypes = [ctypes.POINTER(LinearJob), I, I64, P]
    L.s3d8_selftest_wait_timeout.argtypes = [I64, P]
    L.s3d8_linear_tc_noalloc.argtypes = [P, P, P, P, P, I64, I64, I64, P, P]
    L.s3d8_device_status.argtypes = [P]
    L.s3d8_status_string.argtypes = [I]
    L.s3d8_status_string.restype = ctypes.c_char_p
    L.s3d8_version.argtypes = []
    for fn in ("s3d8_quantize_act", "s3d8_decode", "s3d8_encode", "s3d8_selftest_scaled_abs",
               "s3d8_fit_centroids", "s3d8_fake_quant",
               "s3d8_linear", "s3d8_linear_ex",
               "s3d8_linear_acc_i32", "s3d8_linear_batch", "s3d8_selftest_wait_timeout",
               "s3d8_device_status", "s3d8_version"):
        getattr(L, fn).restype = I
    _lib = L
    return L


def _check(fn: str, status: int):
    if status != 0:
        raise S3D8Error(fn, status, load().s3d8_status_string(status).decode())


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dev(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def groups(N: int) -> int:
    return (N + 2) // 3


def quantize_act(x: torch.Tensor, xq: torch.Tensor | None = None,
                 xscale: torch.Tensor | None = None):
    """Per-token INT8 quantisation of bf16 x[M, K] -> (xq int8 [M, K], xscale fp32 [M])."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xscale is None:
        xscale = torch.empty((M,), dtype=torch.float32, device=x.device)
    st = load().s3d8_quantize_act(_dev(x, "x", torch.bfloat16), M, K,
                                  _dev(xq, "xq", torch.int8, (M, K)),
                                  _dev(xscale, "xscale", torch.float32, (M,)), _stream(x.device))
    _check("s3d8_quantize_act", st)
    return xq, xscale


def decode(packed: torch.Tensor, centroids: torch.Tensor, N: int,
           w: torch.Tensor | None = None) -> torch.Tensor:
    """S3D8 -> dense int8 W[N, K]."""
    G, K = packed.shape
    if G != groups(N):
        raise ValueError(f"packed has {G} rows, expected ceil(N/3) = {groups(N)}")
    if w is None:
        w = torch.empty((N, K), dtype=torch.int8, device=packed.device)
    st = load().s3d8_decode(_dev(packed, "packed", torch.uint8),
                            _dev(centroids, "centroids", torch.int8, (32, 3)), N, K,
                            _dev(w, "w", torch.int8, (N, K)), _stream(packed.device))
    _check("s3d8_decode", st)
    return w


ENCODE_WORKSPACE_BYTES = 16384


def encode(w: torch.Tensor, centroids: torch.Tensor, packed: torch.Tensor | None = None,
           chan_scale: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Direct-cast encoder: bf16 W[N, K] + int8 C[32, 3] -> (packed uint8
    [ceil(N/3), K], chan_scale bf16 [N])."""
    if w.dim() != 2:
        raise ValueError("w must be 2-D [N, K]")
    N, K = w.shape
    if packed is None:
        packed = torch.empty((groups(N), K), dtype=torch.uint8, device=w.device)
    if chan_scale is None:
        chan_scale = torch.empty((N,), dtype=torch.bfloat16, device=w.device)
    if workspace is None:
        workspace = torch.empty((ENCODE_WORKSPACE_BYTES,), dtype=torch.uint8, device=w.device)
    st = load().s3d8_encode(_dev(w, "w", torch.bfloat16),
                            _dev(centroids, "centroids", torch.int8, (32, 3)), N, K,
                            _dev(packed, "packed", torch.uint8, (groups(N), K)),
                            _dev(chan_scale, "chan_scale", torch.bfloat16, (N,)),
                            _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                            _stream(w.device))
    _check("s3d8_encode", st)
    return packed, chan_scale


def fake_quant(w: torch.Tensor, centroids: torch.Tensor, w_hat: torch.Tensor | None = None,
               chan_scale: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """QAT fake-quant forward: bf16 W[N, K] -> (w_hat bf16 [N, K] = s alpha
    C[q][n mod 3], chan_scale bf16 [N])."""
    if w.dim() != 2:
        raise ValueError("w must be 2-D [N, K]")
    N, K = w.shape
    if w_hat is None:
        w_hat = torch.empty((N, K), dtype=torch.bfloat16, device=w.device)
    if chan_scale is None:
        chan_scale = torch.empty((N,), dtype=torch.bfloat16, device=w.device)
    if workspace is None:
        workspace = torch.empty((ENCODE_WORKSPACE_BYTES,), dtype=torch.uint8, device=w.device)
    st = load().s3d8_fake_quant(_dev(w, "w", torch.bfloat16),
                                _dev(centroids, "centroids", torch.int8, (32, 3)), N, K,
                                _dev(w_hat, "w_hat", torch.bfloat16, (N, K)),
                                _dev(chan_scale, "chan_scale", torch.bfloat16, (N,)),
                                _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                                _stream(w.device))
    _check("s3d8_fake_quant", st)
    return w_hat, chan_scale


class FakeQuantSTE(torch.autograd.Function):
    """Q(theta) in the forward pass (s3d8_fake_quant), identity in the
    backward pass (straight-through estimator): the QAT weight path."""

    @staticmethod
    def forward(ctx, w, centroids):
        w_hat, _ = fake_quant(w.detach(), centroids)
        return w_hat

    @staticmethod
    def backward(ctx, grad):
        return grad, None


def fit_workspace_size(N: int, K: int) -> int:
    return int(load().s3d8_fit_workspace_size(N, K))


def fit_centroids(w: torch.Tensor, draws: torch.Tensor, iters: int,
                  workspace: torch.Tensor | None = None):
    """Lloyd-Max centroid fit from k-means++ on the scaled 3-vectors of bf16
    W[N, K]; draws: 32 int32 (read as uint32) on the device.  Returns (fp32
    centroids [32, 3], int8 table [32, 3])."""
    if w.dim() != 2:
        raise ValueError("w must be 2-D [N, K]")
    N, K = w.shape
    cf = torch.empty((32, 3), dtype=torch.float32, device=w.device)
    C = torch.empty((32, 3), dtype=torch.int8, device=w.device)
    if workspace is None:
        workspace = torch.empty((max(fit_workspace_size(N, K), 1),), dtype=torch.uint8,
                                device=w.device)
    st = load().s3d8_fit_centroids(_dev(w, "w", torch.bfloat16), N, K,
                                   _dev(draws, "draws", torch.int32, (32,)), int(iters),
                                   _dev(cf, "cf", torch.float32), _dev(C, "C", torch.int8),
                                   _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                                   _stream(w.device))
    _check("s3d8_fit_centroids", st)
    return cf, C


def selftest_scaled_abs(x: torch.Tensor, alpha: torch.Tensor) -> torch.Tensor:
    """|x| / alpha elementwise (bf16 inputs, fp32 result) through the encoder's
    device code; for checking it against IEEE division."""
    n = x.numel()
    out = torch.empty((n,), dtype=torch.float32, device=x.device)
    st = load().s3d8_selftest_scaled_abs(_dev(x, "x", torch.bfloat16),
                                         _dev(alpha, "alpha", torch.bfloat16, tuple(x.shape)), n,
                                         _dev(out, "out", torch.float32), _stream(x.device))
    _check("s3d8_selftest_scaled_abs", st)
    return out


def workspace_size(M: int, N: int, K: int, algo: int = ALGO_AUTO) -> int:
    return int(load().s3d8_linear_workspace_size(M, N, K, algo))


def _workspace(M, N, K, algo, device, workspace):
    need = workspace_size(M, N, K, algo)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=device)
    if workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    return workspace, workspace.numel()


def linear(packed: torch.Tensor, centroids: torch.Tensor, chan_scale: torch.Tensor,
           xq: torch.Tensor, xscale: torch.Tensor, N: int, out: torch.Tensor | None = None,
           algo: int = ALGO_AUTO, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """out[M, N] bf16 = xscale[m] * chan_scale[n] * sum_k xq[m,k] Wq[n,k]."""
    G, K = packed.shape
    if G != groups(N):
        raise ValueError(f"packed has {G} rows, expected ceil(N/3) = {groups(N)}")
    M = xq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=packed.device)
    ws, ws_bytes = _workspace(M, N, K, algo, packed.device, workspace)
    args = (_dev(packed, "packed", torch.uint8), _dev(centroids, "centroids", torch.int8, (32, 3)),
            _dev(chan_scale, "chan_scale", torch.bfloat16, (N,)), _dev(xq, "xq", torch.int8, (M, K)),
            _dev(xscale, "xscale", torch.float32, (M,)), M, N, K,
            _dev(out, "out", torch.bfloat16, (M, N)),
            None if ws is None else ws.data_ptr(), ws_bytes)
    if algo == ALGO_AUTO:   # the plain entry point: the library picks the algorithm
        _check("s3d8_linear", load().s3d8_linear(*args, _stream(packed.device)))
    else:
        _check("s3d8_linear_ex", load().s3d8_linear_ex(*args, algo, _stream(packed.device)))
    return out


NOALLOC_SCRATCH_BYTES = 32 << 20


def linear_tc_noalloc(packed: torch.Tensor, centroids: torch.Tensor, chan_scale: torch.Tensor,
                      xq: torch.Tensor, xscale: torch.Tensor, N: int,
                      out: torch.Tensor) -> torch.Tensor:
    """The tensor-core linear into the caller's `out` without any device
    allocation, neither here nor in the library: its scratch is a fixed array of
    NOALLOC_SCRATCH_BYTES inside the library (the tensor-core workspace of the
    shape must fit).  For
    callers that cannot allocate device memory.  Calls that overlap on the GPU
    share that array and race; order them on one stream."""
    G, K = packed.shape
    if G != groups(N):
        raise ValueError(f"packed has {G} rows, expected ceil(N/3) = {groups(N)}")
    M = xq.shape[0]
    st = load().s3d8_linear_tc_noalloc(
        _dev(packed, "packed", torch.uint8), _dev(centroids, "centroids", torch.int8, (32, 3)),
        _dev(chan_scale, "chan_scale", torch.bfloat16, (N,)), _dev(xq, "xq", torch.int8, (M, K)),
        _dev(xscale, "xscale", torch.float32, (M,)), M, N, K,
        _dev(out, "out", torch.bfloat16, (M, N)), _stream(packed.device))
    _check("s3d8_linear_tc_noalloc", st)
    return out


def linear_acc_i32(packed: torch.Tensor, centroids: torch.Tensor, xq: torch.Tensor, N: int,
                   algo: int = ALGO_AUTO, acc: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Exact int32 accumulators acc[M, N] = sum_k xq[m,k] Wq[n,k]."""
    G, K = packed.shape
    if G != groups(N):
        raise ValueError(f"packed has {G} rows, expected ceil(N/3) = {groups(N)}")
    M = xq.shape[0]
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=packed.device)
    ws, ws_bytes = _workspace(M, N, K, algo, packed.device, workspace)
    st = load().s3d8_linear_acc_i32(
        _dev(packed, "packed", torch.uint8), _dev(centroids, "centroids", torch.int8, (32, 3)),
        _dev(xq, "xq", torch.int8, (M, K)), M, N, K, _dev(acc, "acc", torch.int32, (M, N)),
        None if ws is None else ws.data_ptr(), ws_bytes, algo, _stream(packed.device))
    _check("s3d8_linear_acc_i32", st)
    return acc


def linear_batch(jobs, M: int):
    """Several independent S3D8 linears with the same token count M (1..8) in one
    launch.  Each job is a dict with keys packed, centroids, chan_scale, N and
    either x (bf16 [M, K], quantised inside the launch) or xq + xscale; optional
    out (bf16 [M, N]), acc (int32 [M, N], replaces out), xq_out, xscale_out.
    Returns the list of output tensors (out, or acc when given)."""
    if len(jobs) > MAX_BATCH:
        raise ValueError(f"at most {MAX_BATCH} jobs per launch")
    arr = (LinearJob * max(1, len(jobs)))()
    results = []
    device = None
    for i, j in enumerate(jobs):
        packed, C, N = j["packed"], j["centroids"], int(j["N"])
        G, K = packed.shape
        if G != groups(N):
            raise ValueError(f"job {i}: packed has {G} rows, expected ceil(N/3) = {groups(N)}")
        device = packed.device
        d = arr[i]
        d.packed = _dev(packed, "packed", torch.uint8)
        d.centroids = _dev(C, "centroids", torch.int8, (32, 3))
        d.N, d.K = N, K
        if j.get("x") is not None:
            d.x_bf16 = _dev(j["x"], "x", torch.bfloat16, (M, K))
            if j.get("xq_out") is not None:
                d.xq_out = _dev(j["xq_out"], "xq_out", torch.int8, (M, K))
            if j.get("xscale_out") is not None:
                d.xscale_out = _dev(j["xscale_out"], "xscale_out", torch.float32, (M,))
        else:
            d.xq = _dev(j["xq"], "xq", torch.int8, (M, K))
            if j.get("xscale") is not None:
                d.xscale = _dev(j["xscale"], "xscale", torch.float32, (M,))
        if j.get("acc") is not None:
            d.acc = _dev(j["acc"], "acc", torch.int32, (M, N))
            results.append(j["acc"])
        else:
            out = j.get("out")
            if out is None:
                out = torch.empty((M, N), dtype=torch.bfloat16, device=packed.device)
            d.out_bf16 = _dev(out, "out", torch.bfloat16, (M, N))
            d.chan_scale_bf16 = _dev(j["chan_scale"], "chan_scale", torch.bfloat16, (N,))
            results.append(out)
    st = load().s3d8_linear_batch(arr, len(jobs), M, _stream(device))
    _check("s3d8_linear_batch", st)
    return results


def selftest_wait_timeout(polls: int = 1000) -> None:
    """Run the bounded-wait failure path once (see include/s3d8.h)."""
    _check("s3d8_selftest_wait_timeout", load().s3d8_selftest_wait_timeout(polls, _stream(None)))


def device_status() -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    return int(load().s3d8_device_status(_stream(None)))
