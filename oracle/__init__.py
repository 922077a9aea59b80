"""Plain CPU oracle for the S3D8 W2.7A8 linear layer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the CPU
baseline leg of the benchmark may import this package; the product path
(``s3d8_a8_linear_gb300``) never does, and the two share no code.

The arithmetic lives in ``s3d8_oracle.c`` (plain scalar C, fp32 where the
activation quantiser fixes fp32, int64 accumulation, fp64 output).  This
module only compiles it with gcc, loads it and marshals numpy arrays.

Sources followed (cited per function in the C file):
  "Llama-Mobile: Efficient 2.7-Bit Quantization of VLMs", section 3.4, Eq. 1;
  "11 billion parameters on a phone", sections "Bit layout" and
  "Output channel packing".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "s3d8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libs3d8_oracle.so")

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, plain -O2, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        L = _lib
        L.s3d8o_byte_fields.argtypes = [ctypes.c_uint8] + [ctypes.POINTER(I32)] * 4
        L.s3d8o_byte_fields.restype = None
        L.s3d8o_pack_byte.argtypes = [I32, I32, I32, I32]
        L.s3d8o_pack_byte.restype = ctypes.c_uint8
        L.s3d8o_decode_component.argtypes = [ctypes.c_uint8, P, I32]
        L.s3d8o_decode_component.restype = I32
        L.s3d8o_decode.argtypes = [P, P, I64, I64, P]
        L.s3d8o_decode.restype = None
        L.s3d8o_pack.argtypes = [P, P, I64, I64, P]
        L.s3d8o_pack.restype = None
        L.s3d8o_quantize_act.argtypes = [P, I64, I64, P, P]
        L.s3d8o_quantize_act.restype = None
        L.s3d8o_linear_acc.argtypes = [P, P, P, I64, I64, I64, P]
        L.s3d8o_linear_acc.restype = I64
        L.s3d8o_linear_acc_at.argtypes = [P, P, P, I64, I64, I64, P, P, I64, P]
        L.s3d8o_linear_acc_at.restype = None
        L.s3d8o_linear_out.argtypes = [P, P, P, I64, I64, P]
        L.s3d8o_encode.argtypes = [P, P, I64, I64, P, P]
        L.s3d8o_encode.restype = I32
        L.s3d8o_fit_centroids.argtypes = [P, I64, I64, P, I32, P, P]
        L.s3d8o_fit_centroids.restype = I32
        L.s3d8o_fake_quant.argtypes = [P, P, I64, I64, P]
        L.s3d8o_fake_quant.restype = I32
        L.s3d8o_linear_out.restype = None
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _as(a, dtype, shape=None) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    if shape is not None:
        assert a.shape == tuple(shape), f"expected shape {shape}, got {a.shape}"
    return a


def groups(N: int) -> int:
    """Packed rows: ceil(N / 3)."""
    return (N + 2) // 3


def byte_fields(b: int):
    """(Q, S0, S1, S2) of one packed byte."""
    vals = [ctypes.c_int32() for _ in range(4)]
    lib().s3d8o_byte_fields(ctypes.c_uint8(b), *[ctypes.byref(v) for v in vals])
    return tuple(v.value for v in vals)


def pack_byte(Q: int, S0: int, S1: int, S2: int) -> int:
    return int(lib().s3d8o_pack_byte(Q, S0, S1, S2))


def decode_component(b: int, C: np.ndarray, d: int) -> int:
    C = _as(C, np.int8, (32, 3))
    return int(lib().s3d8o_decode_component(ctypes.c_uint8(b), _ptr(C), d))


def decode(packed: np.ndarray, C: np.ndarray, N: int) -> np.ndarray:
    """Dense int8 W[N, K] from packed[ceil(N/3), K]."""
    packed = _as(packed, np.uint8)
    G, K = packed.shape
    assert G == groups(N)
    C = _as(C, np.int8, (32, 3))
    w = np.empty((N, K), dtype=np.int8)
    lib().s3d8o_decode(_ptr(packed), _ptr(C), N, K, _ptr(w))
    return w


def pack(Q: np.ndarray, S: np.ndarray) -> np.ndarray:
    """packed[G, K] from Q[G, K] (0..31) and S[3G, K] (0/1)."""
    Q = _as(Q, np.int32)
    S = _as(S, np.int32)
    G, K = Q.shape
    assert S.shape == (3 * G, K)
    out = np.empty((G, K), dtype=np.uint8)
    lib().s3d8o_pack(_ptr(Q), _ptr(S), G, K, _ptr(out))
    return out


def quantize_act(x_bf16_bits: np.ndarray):
    """(xq int8 [M, K], xscale fp32 [M]) from bf16 bit patterns [M, K]."""
    x = _as(x_bf16_bits, np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), dtype=np.int8)
    xs = np.empty((M,), dtype=np.float32)
    lib().s3d8o_quantize_act(_ptr(x), M, K, _ptr(xq), _ptr(xs))
    return xq, xs


def linear_acc(packed: np.ndarray, C: np.ndarray, xq: np.ndarray, N: int):
    """(acc int64 [M, N], number of entries outside int32)."""
    packed = _as(packed, np.uint8)
    G, K = packed.shape
    assert G == groups(N)
    xq = _as(xq, np.int8)
    M = xq.shape[0]
    assert xq.shape == (M, K)
    C = _as(C, np.int8, (32, 3))
    acc = np.empty((M, N), dtype=np.int64)
    bad = lib().s3d8o_linear_acc(_ptr(packed), _ptr(C), _ptr(xq), M, N, K, _ptr(acc))
    return acc, int(bad)


def linear_acc_at(packed, C, xq, N: int, ms, ns) -> np.ndarray:
    """acc[ms[i], ns[i]] for each i (int64)."""
    packed = _as(packed, np.uint8)
    G, K = packed.shape
    assert G == groups(N)
    xq = _as(xq, np.int8)
    M = xq.shape[0]
    C = _as(C, np.int8, (32, 3))
    ms = _as(ms, np.int64)
    ns = _as(ns, np.int64)
    assert ms.shape == ns.shape and ms.ndim == 1
    assert (ms >= 0).all() and (ms < M).all() and (ns >= 0).all() and (ns < N).all()
    out = np.empty(ms.shape, dtype=np.int64)
    lib().s3d8o_linear_acc_at(_ptr(packed), _ptr(C), _ptr(xq), M, N, K, _ptr(ms), _ptr(ns),
                              ms.size, _ptr(out))
    return out


def linear_out(acc: np.ndarray, xscale: np.ndarray, chan_scale_bits: np.ndarray) -> np.ndarray:
    """fp64 out[M, N] = xscale[m] * acc[m, n] * alpha[n]."""
    acc = _as(acc, np.int64)
    M, N = acc.shape
    xscale = _as(xscale, np.float32, (M,))
    cs = _as(chan_scale_bits, np.uint16, (N,))
    out = np.empty((M, N), dtype=np.float64)
    lib().s3d8o_linear_out(_ptr(acc), _ptr(xscale), _ptr(cs), M, N, _ptr(out))
    return out


def linear(packed, C, chan_scale_bits, xq, xscale, N: int):
    """Full layer: (fp64 out [M, N], int64 acc [M, N])."""
    acc, bad = linear_acc(packed, C, xq, N)
    assert bad == 0, "accumulator outside int32"
    return linear_out(acc, xscale, chan_scale_bits), acc


def encode(w_bf16_bits: np.ndarray, C: np.ndarray):
    """Direct-cast encoder: bf16 weights [N, K] and a 32x3 table -> (packed
    [ceil(N/3), K] uint8, chan_scale [N] bf16 bits).  Paper section 3.4,
    "Quantization" (forward pass with frozen centroids)."""
    w = _as(w_bf16_bits, np.uint16)
    N, K = w.shape
    C = _as(C, np.int8, (32, 3))
    packed = np.empty((groups(N), K), np.uint8)
    cs = np.empty((N,), np.uint16)
    if lib().s3d8o_encode(_ptr(w), _ptr(C), N, K, _ptr(packed), _ptr(cs)) != 0:
        raise MemoryError("oracle encoder scratch")
    return packed, cs


def fit_centroids(w_bf16_bits: np.ndarray, r: np.ndarray, iters: int):
    """Lloyd-Max centroid fit from k-means++ (paper section 3.4,
    "Quantization"): bf16 weights [N, K], 32 uint32 draws -> (fp32 centroids
    [32, 3], int8 table [32, 3])."""
    w = _as(w_bf16_bits, np.uint16)
    N, K = w.shape
    r = _as(r, np.uint32, (32,))
    cf = np.empty((32, 3), np.float32)
    C = np.empty((32, 3), np.int8)
    if lib().s3d8o_fit_centroids(_ptr(w), N, K, _ptr(r), int(iters), _ptr(cf), _ptr(C)) != 0:
        raise MemoryError("oracle fit scratch")
    return cf, C


def fake_quant(w_bf16_bits: np.ndarray, C: np.ndarray) -> np.ndarray:
    """QAT fake-quant forward: bf16 W [N, K] -> bf16 bits of s alpha C[q][n mod 3]
    (paper section 3.4, Eq. 1 applied to the direct cast)."""
    w = _as(w_bf16_bits, np.uint16)
    N, K = w.shape
    C = _as(C, np.int8, (32, 3))
    out = np.empty((N, K), np.uint16)
    if lib().s3d8o_fake_quant(_ptr(w), _ptr(C), N, K, _ptr(out)) != 0:
        raise MemoryError("oracle fake-quant scratch")
    return out
