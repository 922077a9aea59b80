"""GPU parity on the full 40-layer 11B-shaped text stack at M = 1 plus the LM head.

Every one of the 281 matrices (40 x 7 projections, each with its own centroid
table, and the 4096 -> 128256 head) runs through the grouped decode launch with
the activation quantisation fused, one launch per layer as a decoder would
issue it.  Four layers and the head are compared with the fp64 oracle in full,
the other layers on 64 outputs per matrix (first, last and random channels)
that the oracle computes one by one.  Each layer (and the head) runs twice:
once with bf16 outputs, checked within the parity tolerance, and once with the
raw int32 accumulators, which must equal the oracle's exact sums.  About
3.08 GB of packed weights in total; the layers are generated, checked and freed
one at a time.
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import assert_out_close, bf16_bits, bf16_to_f64, dev, i8, to_np, u8

pytestmark = pytest.mark.gpu

SEED = 4
FULL_LAYERS = (0, 13, 26, 39)
INPUT_K = {"attn": 4096, "o": 4096, "mlp": 4096, "down": 14336}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def _job(m, x):
    return dict(packed=u8(m.packed), centroids=i8(m.C), chan_scale=bf16_bits(m.chan_scale),
                N=m.N, x=bf16_bits(x))


def _acc_job(job):
    """The same job writing int32 accumulators instead of bf16 outputs."""
    j = dict(job)
    j["acc"] = torch.empty((1, job["N"]), dtype=torch.int32, device=dev())
    return j


def test_text_stack_40_layers_and_head():
    total = 0
    for layer in range(si.LLAMA_11B_LAYERS):
        mats = si.layer_matrices(layer=layer, seed=SEED)
        acts = {a: si.acts(1, K, seed=SEED, index=layer * 4 + i)
                for i, (a, K) in enumerate(INPUT_K.items())}
        jobs = [_job(m, acts[si.LLAMA_11B_INPUT_OF[m.name]]) for m in mats]
        outs = s3d8.linear_batch(jobs, 1)
        accs = s3d8.linear_batch([_acc_job(j) for j in jobs], 1)
        torch.cuda.synchronize()
        q = {a: oracle.quantize_act(x) for a, x in acts.items()}
        rng = np.random.default_rng(layer)
        for m, out, acc_gpu in zip(mats, outs, accs):
            xq, xs = q[si.LLAMA_11B_INPUT_OF[m.name]]
            got = bf16_to_f64(out)
            acc_got = to_np(acc_gpu).astype(np.int64)
            if layer in FULL_LAYERS:
                ref, acc_ref = oracle.linear(m.packed, m.C, m.chan_scale, xq, xs, m.N)
                assert_out_close(got, ref)
                np.testing.assert_array_equal(acc_got, acc_ref, err_msg=f"layer {layer} {m.name}")
            else:
                ns = np.concatenate([[0, 1, 2, m.N - 1], rng.integers(0, m.N, 60)]).astype(np.int64)
                acc = oracle.linear_acc_at(m.packed, m.C, xq, m.N, np.zeros_like(ns), ns)
                csf = si.bf16_bits_to_f32(m.chan_scale).astype(np.float64)
                assert_out_close(got[0, ns], float(xs[0]) * acc * csf[ns])
                np.testing.assert_array_equal(acc_got[0, ns], acc, err_msg=f"layer {layer} {m.name}")
            total += m.packed.size
        del jobs, outs, accs
    head = si.head_matrix(seed=SEED)
    x = si.acts(1, head.K, seed=SEED, index=si.LLAMA_11B_LAYERS * 4)
    job = _job(head, x)
    (out,) = s3d8.linear_batch([job], 1)
    (acc_gpu,) = s3d8.linear_batch([_acc_job(job)], 1)
    torch.cuda.synchronize()
    xq, xs = oracle.quantize_act(x)
    ref, acc_ref = oracle.linear(head.packed, head.C, head.chan_scale, xq, xs, head.N)
    assert_out_close(bf16_to_f64(out), ref)
    np.testing.assert_array_equal(to_np(acc_gpu).astype(np.int64), acc_ref, err_msg="head")
    total += head.packed.size
    assert total == 3_084_091_392   # packed bytes of the whole stack
