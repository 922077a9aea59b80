"""Helpers shared by the GPU parity tests: device copies and comparisons."""
import numpy as np
import torch

TOL_ABS = 1e-3
TOL_REL = 1e-2


def dev():
    return torch.device("cuda:0")


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(dev())


def i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int8)).to(dev())


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev())


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(
        torch.bfloat16).to(dev())


def to_np(t):
    return t.cpu().numpy()


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def assert_out_close(got, ref):
    """|gpu - ref| <= 1e-3 + 1e-2 |ref| element by element (bf16 vs fp64 oracle)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    excess = np.abs(got - ref) - (TOL_ABS + TOL_REL * np.abs(ref))
    if not (excess <= 0).all():
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"out outside tolerance at {i}: got {got[i]}, ref {ref[i]}")


def guarded(shape, dtype, fill, pad=64):
    """A tensor view with `pad` guard elements on both sides, and a checker that
    the guards were left untouched.  An odd pad gives a view that is not
    16-byte aligned."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device=dev())
    view = buf[pad:pad + n].view(*shape)

    def check():
        lo = buf[:pad]
        hi = buf[pad + n:]
        assert bool((lo == fill).all()) and bool((hi == fill).all()), "write outside the output"

    return view, check
