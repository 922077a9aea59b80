"""The seeded input recipe (s3d8_inputs), checked by its properties on the CPU:
the field ranges and distributions the workloads name (centroids uniform in
[1, 127], uniform packed bytes, |N(0, 0.02)|/127 channel scales, N(0, 1)
activations, 1 % outliers at 20x), determinism per seed and index, and the
Llama-3.2-11B shapes."""
import numpy as np

import s3d8_inputs as si


def test_same_seed_same_fields_other_index_other_fields():
    a, b = si.matrix("q", 256, 96, seed=3, index=1), si.matrix("q", 256, 96, seed=3, index=1)
    c = si.matrix("q", 256, 96, seed=3, index=2)
    for f in ("C", "packed", "chan_scale"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
        assert not np.array_equal(getattr(a, f), getattr(c, f))
    assert np.array_equal(si.acts(4, 256, seed=3), si.acts(4, 256, seed=3))
    assert not np.array_equal(si.acts(4, 256, seed=3, index=0), si.acts(4, 256, seed=3, index=1))


def test_centroid_tables_are_uniform_on_1_to_127():
    tables = np.stack([si.matrix("t", 16, 3, seed=0, index=i).C for i in range(400)]).astype(np.int64)
    assert tables.shape == (400, 32, 3)
    assert tables.min() == 1 and tables.max() == 127
    # uniform on 1..127: mean 64, standard deviation sqrt((127^2 - 1) / 12)
    assert abs(tables.mean() - 64.0) < 0.5
    assert abs(tables.std() - np.sqrt((127 ** 2 - 1) / 12)) < 0.5
    counts = np.bincount(tables.ravel(), minlength=128)[1:]
    assert counts.min() > 0.75 * counts.mean()


def test_packed_bytes_are_uniform():
    m = si.matrix("gate", 4096, 14336, seed=0)
    assert m.packed.shape == (si.groups(14336), 4096) and m.packed.dtype == np.uint8
    counts = np.bincount(m.packed.ravel(), minlength=256).astype(np.float64)
    expected = m.packed.size / 256
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    assert chi2 < 400   # 255 degrees of freedom: mean 255, sd ~22.6


def test_channel_scales_are_half_normal_over_127():
    s = si.bf16_bits_to_f32(si.matrix("gate", 16, 14336 * 8, seed=1).chan_scale).astype(np.float64)
    assert (s >= 0).all()
    sigma = 0.02 / 127
    assert abs(s.mean() / (sigma * np.sqrt(2 / np.pi)) - 1) < 0.02      # half-normal mean
    assert abs(np.sqrt((s ** 2).mean()) / sigma - 1) < 0.02              # second moment sigma^2


def test_activations_are_standard_normal_with_one_percent_outliers_at_20x():
    M, K = 64, 4096
    base = si.bf16_bits_to_f32(si.acts(M, K, seed=2)).astype(np.float64)
    assert abs(base.mean()) < 0.01 and abs(base.std() - 1) < 0.01
    out = si.bf16_bits_to_f32(si.acts(M, K, seed=2, outliers=True)).astype(np.float64)
    moved = out != base
    # the outliers reuse the plain draw and scale 1 % of the positions by 20
    assert moved.sum() == (M * K) // 100
    ratio = out[moved] / base[moved]
    assert np.all(np.abs(ratio - 20) < 20 * 2 ** -7)


def test_llama_11b_shapes():
    params = sum(K * N for _, K, N in si.LLAMA_11B_LAYER)
    assert params == 218_103_808
    assert [m.packed.shape for m in si.layer_matrices(0)] == [(si.groups(N), K) for _, K, N in si.LLAMA_11B_LAYER]
    assert si.LLAMA_11B_HEAD == ("head", 4096, 128256) and si.LLAMA_11B_LAYERS == 40
    m, x = si.tiny_case()
    assert (m.K, m.N, x.shape) == (256, 96, (4, 256))
