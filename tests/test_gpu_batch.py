"""GPU parity of the grouped decode launch (s3d8_linear_batch) against the oracle.

Covers fused activation quantisation (codes and scales bit-exact, optional
copies returned), pre-quantised jobs, int32 accumulators, partial K slices,
N not a multiple of 3, M = 1..8, and the rejection of unsupported sizes.
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import assert_out_close, bf16_bits, bf16_to_f64, dev, f32, i8, to_np, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def mat_dev(m):
    return dict(packed=u8(m.packed), centroids=i8(m.C), chan_scale=bf16_bits(m.chan_scale), N=m.N)


def test_layer_fused_m1():
    """The seven projections of a decoder layer in one launch, activations
    quantised inside the launch, each compared in full with the oracle: the
    bf16 outputs within the parity tolerance, and, from a second launch that
    writes int32 accumulators instead, the exact sums bit for bit."""
    mats = si.layer_matrices(layer=3, seed=1)
    acts = {a: si.acts(1, K, seed=1, index=i) for i, (a, K) in
            enumerate({"attn": 4096, "o": 4096, "mlp": 4096, "down": 14336}.items())}
    jobs, refs, qref = [], [], {}
    for m in mats:
        a = si.LLAMA_11B_INPUT_OF[m.name]
        if a not in qref:
            qref[a] = oracle.quantize_act(acts[a])
        xq_o, xs_o = qref[a]
        ref, acc_o = oracle.linear(m.packed, m.C, m.chan_scale, xq_o, xs_o, m.N)
        refs.append((m.name, ref, a, acc_o))
        j = mat_dev(m)
        j["x"] = bf16_bits(acts[a])
        j["xq_out"] = torch.empty((1, m.K), dtype=torch.int8, device=dev())
        j["xscale_out"] = torch.empty((1,), dtype=torch.float32, device=dev())
        jobs.append(j)
    outs = s3d8.linear_batch(jobs, 1)
    acc_jobs = [dict(j, acc=torch.empty((1, j["N"]), dtype=torch.int32, device=dev())) for j in jobs]
    accs = s3d8.linear_batch(acc_jobs, 1)
    torch.cuda.synchronize()
    for (name, ref, a, acc_o), j, out, acc in zip(refs, jobs, outs, accs):
        assert_out_close(bf16_to_f64(out), ref)
        np.testing.assert_array_equal(to_np(acc).astype(np.int64), acc_o, err_msg=name)
        np.testing.assert_array_equal(to_np(j["xq_out"]), qref[a][0], err_msg=name)
        np.testing.assert_array_equal(to_np(j["xscale_out"]), qref[a][1], err_msg=name)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8])
def test_mixed_jobs_exact(M):
    rng = np.random.default_rng(40 + M)
    shapes = [(96, 256), (7, 16), (1000, 5008), (50, 4096 + 16), (4096, 2048)]
    if M <= 2:
        shapes.append((301, 14336))
    jobs, expect = [], []
    for i, (N, K) in enumerate(shapes):
        C = si.centroids(rng)
        packed = si.packed_bytes(rng, si.groups(N), K)
        cs = si.chan_scale(rng, N)
        x = si.activations(rng, M, K, outliers=True)
        xq_o, xs_o = oracle.quantize_act(x)
        acc_o, bad = oracle.linear_acc(packed, C, xq_o, N)
        assert bad == 0
        j = dict(packed=u8(packed), centroids=i8(C), chan_scale=bf16_bits(cs), N=N)
        fused = (i % 2 == 0) and M * K <= 28672
        if fused:
            j["x"] = bf16_bits(x)
        else:
            j["xq"], j["xscale"] = i8(xq_o), f32(xs_o)
        if i % 3 == 1:
            j["acc"] = torch.empty((M, N), dtype=torch.int32, device=dev())
            expect.append(("acc", acc_o))
        else:
            expect.append(("out", oracle.linear_out(acc_o, xs_o, cs)))
        jobs.append(j)
    outs = s3d8.linear_batch(jobs, M)
    torch.cuda.synchronize()
    for (kind, want), got in zip(expect, outs):
        if kind == "acc":
            np.testing.assert_array_equal(to_np(got).astype(np.int64), want)
        else:
            assert_out_close(bf16_to_f64(got), want)


def test_single_job_matches_linear_and_ties():
    # unit scale (absmax 127): halves round to even inside the fused quantiser
    K, N = 512, 33
    rng = np.random.default_rng(3)
    vals = rng.choice(np.array([2.5, -3.5, 0.5, 1.5, -0.5, 126.5, 0.0, 64.0], np.float32), K)
    vals[7] = 127.0
    x = si.f32_to_bf16_bits(vals[None, :])
    C = si.centroids(rng)
    packed = si.packed_bytes(rng, si.groups(N), K)
    cs = si.chan_scale(rng, N)
    xq_o, xs_o = oracle.quantize_act(x)
    assert xs_o[0] == 1.0
    ref, _ = oracle.linear(packed, C, cs, xq_o, xs_o, N)
    j = dict(packed=u8(packed), centroids=i8(C), chan_scale=bf16_bits(cs), N=N, x=bf16_bits(x),
             xq_out=torch.empty((1, K), dtype=torch.int8, device=dev()))
    out = s3d8.linear_batch([j], 1)[0]
    single = s3d8.linear(u8(packed), i8(C), bf16_bits(cs), i8(xq_o), f32(xs_o), N)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(j["xq_out"]), xq_o)
    assert_out_close(bf16_to_f64(out), ref)
    np.testing.assert_array_equal(to_np(out.view(torch.int16)), to_np(single.view(torch.int16)))


def test_zero_activation_and_unsupported():
    rng = np.random.default_rng(8)
    K, N = 256, 12
    C, packed, cs = si.centroids(rng), si.packed_bytes(rng, si.groups(N), K), si.chan_scale(rng, N)
    x = np.zeros((2, K), np.uint16)
    out = s3d8.linear_batch([dict(packed=u8(packed), centroids=i8(C), chan_scale=bf16_bits(cs), N=N,
                                  x=bf16_bits(x))], 2)[0]
    assert (to_np(out.float()) == 0).all()
    # fused quantisation needs M * K <= 28672
    K2 = 14336
    big = dict(packed=u8(si.packed_bytes(rng, si.groups(N), K2)), centroids=i8(C),
               chan_scale=bf16_bits(cs), N=N,
               x=bf16_bits(si.activations(rng, 3, K2)))
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.linear_batch([big], 3)
    assert e.value.status == -3
    with pytest.raises(ValueError):
        s3d8.linear_batch([big] * 9, 3)
