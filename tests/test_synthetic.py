"""The seeded input recipe (no GPU): deterministic, shaped and distributed as stated."""
import numpy as np

import synthetic


def test_deterministic_and_seed_dependent():
    w = synthetic.custom(192, 4, 2, seed=123)
    a = synthetic.make_inputs(w)
    b = synthetic.make_inputs(w)
    for x, y in zip(a, b):
        assert x.dtype == np.float16 and np.array_equal(x.view(np.uint16), y.view(np.uint16))
    c = synthetic.make_inputs(synthetic.custom(192, 4, 2, seed=124))
    assert not np.array_equal(a[0], c[0])


def test_shapes_and_layouts():
    w = synthetic.WORKLOADS["t128_h4_kv2"]
    q, k, vT = synthetic.make_inputs(w)
    assert q.shape == (4, 128, 64) and k.shape == (2, 128, 64) and vT.shape == (2, 64, 128)
    assert vT.flags["C_CONTIGUOUS"]
    assert 0.9 < float(q.astype(np.float64).std()) < 1.1


def test_workload_table():
    names = list(synthetic.WORKLOADS)
    assert names[3] == synthetic.HEADLINE
    w = synthetic.WORKLOADS[synthetic.HEADLINE]
    assert (w.T, w.heads, w.kv_heads) == (8192, 32, 8)
    assert w.causal_flops == 4 * 8192 ** 2 * 64 * 32 / 2
    for w in synthetic.WORKLOADS.values():
        assert w.T % 64 == 0 and w.heads % w.kv_heads == 0


def test_profile_shapes_apart_from_workloads():
    assert not set(synthetic.PROFILE_SHAPES) & set(synthetic.WORKLOADS)
    for name, w in synthetic.PROFILE_SHAPES.items():
        assert synthetic.lookup(name) is w
        assert w.T % 64 == 0 and w.heads % w.kv_heads == 0
    assert synthetic.lookup(synthetic.HEADLINE) is synthetic.WORKLOADS[synthetic.HEADLINE]


def test_peaked_and_outlier_recipes():
    w = synthetic.custom(388, 2, 1, seed=5, qk_scale=4.0)
    q, k, _ = synthetic.make_inputs(w)
    assert 3.6 < float(q.astype(np.float64).std()) < 4.4
    w = synthetic.custom(388, 2, 1, seed=5, k_outlier_every=97, k_outlier_scale=16.0,
                         v_uniform=True)
    q, k, vT = synthetic.make_inputs(w)
    norms = np.linalg.norm(k[0].astype(np.float64), axis=1)
    out = (np.arange(388) + 1) % 97 == 0
    assert out.sum() == 4 and norms[out].min() > 4 * norms[~out].max()
    assert float(np.abs(vT.astype(np.float64)).max()) <= 1.0
