"""Trees verified without snapshots (the per-block solve) on the GPU against
the oracle, through the C ABI: tree shapes up to 64 nodes (a node's path
spans both halves of a warp's lanes past 32 nodes), bf16 and fp32 inputs, the
8- and 16-column tiles, raw-projection inputs, and the malformed-tree and
depth-cap paths."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, canaries_ok, dev, guarded, torch

pytestmark = pytest.mark.gpu


def _shape(name, N, rng):
    n = np.arange(N)
    if name == "star":
        p = np.where(n == 0, -1, 0)
    elif name == "path":
        p = n - 1
    elif name == "broom":
        p = np.where(n < N // 2, n - 1, N // 2 - 1)
    else:
        p = synthetic.random_tree(rng, N, depth_cap=64)
    p = np.asarray(p, np.int32)
    p[0] = -1
    return p


def _run(gdn, inp, *, tile=0, max_depth=0, prep=False, q=None, k=None, a=None, b=None):
    t = torch()
    B, N, Hv, dv = inp["B"], inp["N"], inp["Hv"], inp["dv"]
    o, o_back = guarded((B, N, Hv, dv), fill=float("nan"))
    depth = t.zeros((B, N), dtype=t.int32, device="cuda")
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gdn.gdn_verify_tree(dev(inp["q"] if q is None else q), dev(inp["k"] if k is None else k),
                        dev(inp["v"]), dev(inp["alpha"] if a is None else a),
                        dev(inp["beta"] if b is None else b), dev(inp["cache"]), None, o,
                        dev(inp["parent"]), depth_out=depth, slot=dev(inp["slot"]),
                        n_slots=inp["n_slots"], status=st, tile_cols=tile, max_depth=max_depth,
                        prep=prep)
    t.cuda.synchronize()
    assert canaries_ok(o_back, o.numel())
    return int(st.item()), o.cpu().numpy(), depth.cpu().numpy()


@pytest.mark.parametrize("N", [1, 7, 33, 64])
@pytest.mark.parametrize("shape", ["star", "path", "broom", "random"])
def test_snapshot_free_tree_shapes(gpu_lib, N, shape):
    rng = np.random.default_rng(9600 + N)
    inp = synthetic.make_verify_inputs(B=2, N=N, Hk=2, Hv=4, dk=128, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05,
                                       seed=9600 + 3 * N + len(shape), tree=True, n_slots=3,
                                       depth_cap=64)
    inp = dict(inp, parent=np.stack([_shape(shape, N, rng) for _ in range(2)]))
    st, o, depth = _run(gpu_lib, inp)
    assert st == 0
    ost, _, oo = oracle.verify_inputs(inp)
    assert ost == oracle.OK
    assert_close(o, oo, f"{shape} N={N} o")
    assert np.array_equal(depth, oracle.tree_depth(inp["parent"])[1])


@pytest.mark.parametrize("dtype,tile", [("f32", 0), ("f32", 8), ("bf16", 8)])
def test_snapshot_free_tree_dtypes_and_tiles(gpu_lib, dtype, tile):
    inp = synthetic.make_verify_inputs(B=3, N=40, Hk=2, Hv=6, dk=64, dv=48, dtype=dtype,
                                       alpha_kind="near_one", state_sigma=0.05, seed=9700 + tile,
                                       tree=True, depth_cap=64)
    st, o, _ = _run(gpu_lib, inp, tile=tile)
    assert st == 0
    ost, _, oo = oracle.verify_inputs(inp)
    assert_close(o, oo, f"{dtype} tile={tile} o")


def test_snapshot_free_tree_from_raw_projections(gpu_lib):
    """gdn_verify_tree_prep without snapshots: raw q/k projections and gate
    pre-activations, against the oracle on the oracle-prepared inputs."""
    rng = np.random.default_rng(9800)
    B, N, Hk, Hv, dk, dv = 2, 45, 2, 6, 128, 32
    q = rng.standard_normal((B, N, Hk, dk)) * rng.uniform(0.2, 5.0, (B, N, Hk, 1))
    k = rng.standard_normal((B, N, Hk, dk)) * rng.uniform(0.2, 5.0, (B, N, Hk, 1))
    qs, ks = (synthetic.f32_to_bf16_bits(x.astype(np.float32)) for x in (q, k))
    q64, k64 = (synthetic.bf16_bits_to_f32(x).astype(np.float64) for x in (qs, ks))
    a = (rng.standard_normal((B, N, Hv)) * 2.0 - 2.5).astype(np.float32)
    b = (rng.standard_normal((B, N, Hv)) * 1.5).astype(np.float32)
    inp = synthetic.make_verify_inputs(B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=9801,
                                       tree=True, depth_cap=64)
    st, o, _ = _run(gpu_lib, inp, prep=True, q=qs, k=ks, a=a, b=b)
    assert st == 0
    qn, kn, al, be = oracle.prepare_inputs(q64, k64, a, b)
    ost, _, oo = oracle.verify(qn, kn, inp["v_f64"], al, be, inp["cache"], inp["slot"],
                               inp["parent"], B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                               n_slots=inp["n_slots"])
    assert ost == oracle.OK
    assert_close(o, oo, "snapshot-free prep tree o")


def test_snapshot_free_tree_errors_skip_only_the_bad_sequence(gpu_lib):
    """A malformed parent array or a tree deeper than the cap skips only its
    own sequence (outputs left untouched) and reports GDN_ERR_BAD_TREE."""
    inp = synthetic.make_verify_inputs(B=3, N=12, Hk=1, Hv=2, dk=32, dv=16, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=9900,
                                       tree=True)
    n = np.arange(12)
    par = np.stack([np.where(n == 0, -1, 0), n - 1, np.where(n < 4, n - 1, 3)]).astype(np.int32)
    inp = dict(inp, parent=par)
    st, o, depth = _run(gpu_lib, inp, max_depth=6)
    assert st == gpu_lib.GDN_ERR_BAD_TREE
    assert np.all(np.isnan(o[1])), "the too-deep path must be skipped"
    assert np.array_equal(depth[1], n + 1), "the skipped tree still reports its depths"
    ost, _, oo = oracle.verify_inputs(inp)
    for b in (0, 2):
        assert_close(o[b], oo[b], f"sequence {b}")
    bad = dict(inp, parent=par.copy())
    bad["parent"][2, 5] = 7
    st, o, _ = _run(gpu_lib, bad)
    assert st == gpu_lib.GDN_ERR_BAD_TREE
    assert np.all(np.isnan(o[2])) and not np.any(np.isnan(o[:2]))
