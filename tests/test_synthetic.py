"""The seeded input generator produces the shapes and distributions the
workloads prescribe."""
import numpy as np

import synthetic


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-39, 65504.0], np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6)
    got = synthetic.bf16_bits_to_f32(synthetic.f32_to_bf16_bits(x))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == np.float32(1.015625)
    assert got[3] == -2.5 and got[5] == 65536.0
    assert np.isfinite(got).all()


def test_chain16_shapes_and_ranges():
    inp = synthetic.chain16()
    B, N, Hk, Hv, d = 1, 16, 16, 48, 128
    assert inp["q"].shape == (B, N, Hk, d) and inp["q"].dtype == np.uint16
    assert inp["v"].shape == (B, N, Hv, d)
    assert inp["alpha"].shape == (B, N, Hv) and inp["alpha"].dtype == np.float32
    assert np.all((inp["alpha"] > 0.9) & (inp["alpha"] < 1.0))
    assert np.all((inp["beta"] > 0) & (inp["beta"] < 1))
    norms = np.linalg.norm(inp["k_f64"], axis=-1)
    assert np.all(np.abs(norms - 1) < 2 ** -7)
    assert inp["cache"].shape == (1, Hv, d, d)
    assert abs(inp["cache"].std() - 0.05) < 0.002
    assert 0 <= inp["accept"][0] < N
    assert inp["parent"][0].tolist() == list(range(-1, N - 1))


def test_tree22_structure():
    inp = synthetic.tree22()
    par = inp["parent"][0]
    assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, 22))
    depth = [1] * 22
    for i in range(1, 22):
        depth[i] = depth[par[i]] + 1
    assert max(depth) <= 16
    assert 0 <= inp["accept"][0] < 22


def test_tiny_and_seeds_are_deterministic():
    a, b = synthetic.tiny_chain(), synthetic.tiny_chain()
    for key in ("q", "k", "v", "alpha", "beta", "cache"):
        assert np.array_equal(a[key], b[key])
    assert a["q"].dtype == np.float32
    assert np.all((a["alpha"] > 0) & (a["alpha"] < 1))
    l0, l1 = synthetic.batched8x16_layer(0), synthetic.batched8x16_layer(1)
    assert not np.array_equal(l0["v"], l1["v"])
    assert sorted(l0["slot"].tolist()) == list(range(8))


def test_prefill_shapes():
    inp = synthetic.prefill8192(T=100)
    assert inp["q"].shape == (100, 16, 128) and inp["v"].shape == (100, 48, 128)
    assert inp["state"].shape == (48, 128, 128)


def test_batched8x22_layers_share_trees_not_inputs():
    """The batched tree workload: eight 22-node trees drawn once for the batch
    (the same in every layer, depth within the cap, parents before children),
    one slot permutation and accepted node per sequence, fresh per-layer
    q/k/v, gates and states."""
    l0, l1 = synthetic.batched8x22_layer(0), synthetic.batched8x22_layer(5)
    for key in ("parent", "slot", "accept"):
        assert np.array_equal(l0[key], l1[key]), key
    assert not np.array_equal(l0["k"], l1["k"]) and not np.array_equal(l0["cache"], l1["cache"])
    par = l0["parent"]
    assert par.shape == (8, 22) and np.all(par[:, 0] == -1)
    n = np.arange(1, 22)
    assert np.all((par[:, 1:] >= 0) & (par[:, 1:] < n))
    assert sorted(l0["slot"].tolist()) == list(range(8))
    assert np.all((l0["accept"] >= 0) & (l0["accept"] < 22))
    for b in range(8):
        depth = [0] * 22
        for i in range(22):
            depth[i] = 1 if par[b, i] < 0 else depth[par[b, i]] + 1
        assert max(depth) <= 16
