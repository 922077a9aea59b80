"""GPU parity of the centroid fit (s3d8_fit_centroids) with the oracle.

Bit-exact: the fp32 centroids after k-means++ and every Lloyd iteration, and
the rounded int8 table.  Every sum in the method is an exact integer (fixed
point, 2^-20 grid) and every decision an fp32 comparison taken in the same
operation order on both sides, so the two runs take the same steps.  Cases:
random weights of several shapes (N mod 3 = 0, 1, 2), planted well-separated
clusters, means exactly half-way between integers, fewer distinct points than
centroids, 0 iterations (k-means++ alone), and a full 4096 x 14336 gate
matrix (one iteration).
"""
import numpy as np
import pytest
import torch

import oracle
import s3d8_a8_linear_gb300 as s3d8
import s3d8_inputs as si
from gpu_util import bf16_bits, dev, to_np
from test_oracle import clustered_points, cluster_centres, draws, weights_from_points

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    s3d8.load(build_if_missing=True)
    torch.cuda.set_device(0)
    yield
    assert s3d8.device_status() == 0


def dev_draws(r):
    return torch.from_numpy(np.ascontiguousarray(r, np.uint32).view(np.int32)).to(dev())


def assert_fit_same(W, r, iters):
    want_cf, want_C = oracle.fit_centroids(W, r, iters)
    cf, C = s3d8.fit_centroids(bf16_bits(W), dev_draws(r), iters)
    torch.cuda.synchronize()
    got_cf = to_np(cf)
    assert np.array_equal(got_cf.view(np.uint32), want_cf.view(np.uint32)), \
        np.argwhere(got_cf != want_cf)[:4]
    assert np.array_equal(to_np(C), want_C)


def weights(rng, N, K):
    w = rng.standard_normal((N, K)) * 0.02 * rng.uniform(0.5, 2.0, size=(N, 1))
    w[rng.random((N, K)) < 0.01] *= 20
    return si.f32_to_bf16_bits(w.astype(np.float32))


@pytest.mark.parametrize("N,K,iters,seed", [(48, 256, 8, 0), (31, 128, 5, 1), (7, 64, 3, 2),
                                            (100, 1040, 6, 3), (2, 512, 4, 4), (66, 96, 0, 5)])
def test_fit_matches_oracle(N, K, iters, seed):
    rng = np.random.default_rng(seed)
    assert_fit_same(weights(rng, N, K), draws(100 + seed), iters)


def test_fit_planted_clusters_and_half_way_means():
    Wp, _, _ = clustered_points()
    assert_fit_same(weights_from_points(Wp), draws(1), 8)
    half = [i for i, c in enumerate(cluster_centres()) if c[0] in (13.0, 40.0)
            and c[1] == 13.0 and c[2] == 12.0]
    Wp, _, _ = clustered_points(seed=3, half_up=half)
    assert_fit_same(weights_from_points(Wp, seed=3), draws(4), 8)


def test_fit_fewer_distinct_points_than_centroids():
    W = np.zeros((3, 16), np.uint16)
    W[0] = si.f32_to_bf16_bits(np.array([0, 3, 8, 10, 20, 33, 47, 51, 64, 70, 80, 90, 100, 110,
                                         120, 127], np.float32))
    assert_fit_same(W, draws(5), 3)
    assert_fit_same(np.zeros((6, 32), np.uint16), draws(6), 2)     # every point at 0


def test_fit_medium_matrix():
    rng = np.random.default_rng(7)
    assert_fit_same(weights(rng, 1024, 4096), draws(7), 3)


def test_fit_full_gate_matrix_one_iteration():
    rng = np.random.default_rng(8)
    W = si.f32_to_bf16_bits((rng.standard_normal((14336, 4096)) * 0.02).astype(np.float32))
    assert_fit_same(W, draws(8), 1)


def test_fit_argument_checks():
    w = torch.zeros((6, 32), dtype=torch.bfloat16, device=dev())
    r = dev_draws(draws(0))
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.fit_centroids(w, r, -1)
    assert e.value.status == -1
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.fit_centroids(torch.zeros((6, 24), dtype=torch.bfloat16, device=dev()), r, 1)
    assert e.value.status == -1
    small = torch.empty((s3d8.fit_workspace_size(6, 32) - 256,), dtype=torch.uint8, device=dev())
    with pytest.raises(s3d8.S3D8Error) as e:
        s3d8.fit_centroids(w, r, 1, workspace=small)
    assert e.value.status == -6
