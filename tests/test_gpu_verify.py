"""CUDA verify / commit path against the CPU oracle, element by element,
on the same seeded inputs, through the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import (assert_close, canaries_ok, dev, guarded, torch, verify_on_gpu)

pytestmark = pytest.mark.gpu


def _oracle(inp, tree=None):
    st, snap, o = oracle.verify_inputs(inp, tree=tree)
    assert st == oracle.OK
    return snap, o


def test_tiny_chain_verify_and_commit(gpu_lib):
    """4-node chain, 2 heads, d = 16, fp32 everything; commit node 2."""
    inp = synthetic.tiny_chain()
    out = verify_on_gpu(gpu_lib, inp)
    snap, o = _oracle(inp)
    assert out["status"] == 0
    assert_close(out["o"], o, "tiny o")
    assert_close(out["snap"], snap, "tiny snapshots")
    t = torch()
    acc = t.tensor([synthetic.tiny_chain_accept()], dtype=t.int32, device="cuda")
    st = t.zeros(1, dtype=t.int32, device="cuda")
    cache = out["cache_t"]
    gpu_lib.gdn_commit_accepted(out["snap_t"], acc, cache, B=1, N=4, Hv=2, dk=16, dv=16,
                                slot=out["slot_t"], n_slots=1, status=st)
    t.cuda.synchronize()
    assert st.item() == 0
    got = cache.cpu().numpy()[inp["slot"][0]]
    assert np.array_equal(got, out["snap"][0, 2]), "commit is not a bit-exact copy"
    assert_close(got, snap[0, 2], "committed state vs oracle")


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (16, 2), (8, 1)])
def test_chain16_full(gpu_lib, tile):
    """Single-sequence chain of 16, 16 q/k heads, 48 value heads, d = 128, bf16
    inputs; every output and every snapshot, in every tile shape."""
    inp = synthetic.chain16()
    out = verify_on_gpu(gpu_lib, inp, tile_cols=tile[0], row_warps=tile[1])
    snap, o = _oracle(inp)
    assert out["status"] == 0
    assert_close(out["o"], o, "chain16 o")
    assert_close(out["snap"], snap, "chain16 snapshots")


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (16, 2), (8, 1)])
def test_tree22_full(gpu_lib, tile):
    """DDTree of 22 nodes: per-node states from the parent, depths bit-exact,
    commit of the accepted node."""
    inp = synthetic.tree22()
    out = verify_on_gpu(gpu_lib, inp, tile_cols=tile[0], row_warps=tile[1])
    snap, o = _oracle(inp)
    assert out["status"] == 0
    assert_close(out["o"], o, "tree22 o")
    assert_close(out["snap"], snap, "tree22 snapshots")
    st, depth = oracle.tree_depth(inp["parent"])
    assert st == oracle.OK and np.array_equal(out["depth"], depth)
    t = torch()
    acc = dev(inp["accept"])
    gpu_lib.gdn_commit_accepted(out["snap_t"], acc, out["cache_t"], B=1, N=22, Hv=48, dk=128,
                                dv=128, slot=out["slot_t"], n_slots=inp["n_slots"])
    t.cuda.synchronize()
    got = out["cache_t"].cpu().numpy()[inp["slot"][0]]
    assert np.array_equal(got, out["snap"][0, inp["accept"][0]])


@pytest.mark.parametrize("tile", [(16, 1), (16, 2), (8, 1)])
def test_single_path_tree_matches_chain(gpu_lib, tile):
    """A tree that is one path is the chain.  The tree kernel reduces u = H^T k
    at every node while the chain kernel takes u from the previous node's
    look-ahead, so the two agree to rounding, and each matches the oracle."""
    inp = synthetic.chain16(seed=99)
    a = verify_on_gpu(gpu_lib, inp, tree=False, tile_cols=tile[0], row_warps=tile[1])
    b = verify_on_gpu(gpu_lib, inp, tree=True, tile_cols=tile[0], row_warps=tile[1])
    snap, o = _oracle(inp)
    for out, kind in ((a, "chain"), (b, "single-path tree")):
        assert_close(out["snap"], snap, f"{kind} snapshots")
        assert_close(out["o"], o, f"{kind} o")
    assert_close(b["snap"], a["snap"], "tree vs chain snapshots")
    assert b["depth"][0].tolist() == list(range(1, 17))


def test_batched_48_layers_as_benchmarked(gpu_lib):
    """8 sequences x chain of 16 x 48 layers, each layer with its own inputs and
    cache, then one commit over all 48 layers; layers 0, 23 and 47 are compared
    with the oracle in full, the commit of every layer bit-exactly."""
    t = torch()
    L, B, N, Hv, d = synthetic.BATCHED_LAYERS, 8, 16, 48, 128
    cache = t.empty((L, B, Hv, d, d), dtype=t.float32, device="cuda")
    snaps = t.empty((L, B, N, Hv, d, d), dtype=t.float32, device="cuda")
    outs = t.empty((L, B, N, Hv, d), dtype=t.float32, device="cuda")
    acc = dev(synthetic.batched8x16_layer(0)["accept"])
    slot = dev(synthetic.batched8x16_layer(0)["slot"])
    inputs = {}
    for l in range(L):
        inp = synthetic.batched8x16_layer(l)
        cache[l].copy_(dev(inp["cache"]))
        if l in (0, 23, 47):
            inputs[l] = inp
        gpu_lib.gdn_verify_chain(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                                 dev(inp["beta"]), cache[l], snaps[l], outs[l], slot=slot,
                                 n_slots=B)
    gpu_lib.gdn_commit_accepted(snaps, acc, cache, B=B, N=N, Hv=Hv, dk=d, dv=d, n_layers=L,
                                snap_layer_stride=B * N * Hv * d * d,
                                cache_layer_stride=B * Hv * d * d, slot=slot, n_slots=B)
    t.cuda.synchronize()
    for l, inp in inputs.items():
        snap, o = _oracle(inp)
        assert_close(outs[l].cpu().numpy(), o, f"layer {l} o")
        assert_close(snaps[l].cpu().numpy(), snap, f"layer {l} snapshots")
    acc_n, slot_n = acc.cpu().numpy(), slot.cpu().numpy()
    for b in range(B):
        got = cache[:, slot_n[b]]
        want = snaps[:, b, acc_n[b]]
        assert t.equal(got, want), f"commit of sequence {b}"


@pytest.mark.parametrize("shape", [
    dict(B=1, N=1, Hk=1, Hv=1, dk=128, dv=128),     # single node
    dict(B=3, N=64, Hk=2, Hv=6, dk=128, dv=128),    # maximum block, several sequences
    dict(B=2, N=5, Hk=1, Hv=3, dk=64, dv=48),       # dv not a multiple of 32
    dict(B=2, N=7, Hk=4, Hv=4, dk=32, dv=16),
    dict(B=1, N=3, Hk=1, Hv=2, dk=16, dv=32),
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tree", [False, True])
def test_edge_shapes(gpu_lib, shape, dtype, tree):
    inp = synthetic.make_verify_inputs(dtype=dtype, alpha_kind="near_one", state_sigma=0.05,
                                       seed=1234 + shape["N"], tree=tree, n_slots=shape["B"] + 2,
                                       **shape)
    out = verify_on_gpu(gpu_lib, inp)
    snap, o = _oracle(inp)
    assert out["status"] == 0
    assert_close(out["o"], o, "o")
    assert_close(out["snap"], snap, "snapshots")
    if tree:
        assert np.array_equal(out["depth"], oracle.tree_depth(inp["parent"])[1])


def test_unit_decay_gates_f32(gpu_lib):
    """alpha = exp(-softplus(z)) spans (0, 1), fp32 inputs, d = 128."""
    inp = synthetic.make_verify_inputs(B=2, N=16, Hk=2, Hv=6, dk=128, dv=128, dtype="f32",
                                       alpha_kind="unit", state_sigma=0.1, seed=77, tree=True)
    out = verify_on_gpu(gpu_lib, inp)
    snap, o = _oracle(inp)
    assert_close(out["o"], o, "o")
    assert_close(out["snap"], snap, "snapshots")


def test_empty_batch_is_a_no_op(gpu_lib):
    t = torch()
    z = t.zeros((0, 4, 1, 16), dtype=t.float32, device="cuda")
    zv = t.zeros((0, 4, 1, 16), dtype=t.float32, device="cuda")
    ab = t.zeros((0, 4, 1), dtype=t.float32, device="cuda")
    cache = t.zeros((1, 1, 16, 16), device="cuda")
    snap = t.zeros((0, 4, 1, 16, 16), device="cuda")
    o = t.zeros((0, 4, 1, 16), device="cuda")
    gpu_lib.gdn_verify_chain(z, z, zv, ab, ab, cache, snap, o, n_slots=1)
    gpu_lib.gdn_commit_accepted(snap, t.zeros(0, dtype=t.int32, device="cuda"), cache, B=0,
                                N=4, Hv=1, dk=16, dv=16)
    t.cuda.synchronize()


@pytest.mark.parametrize("dk", [32, 64])
def test_device_errors_skip_only_the_bad_sequence(gpu_lib, dk):
    """A malformed tree, a bad slot and a bad accept index are reported in the
    status word; the other sequences are still computed correctly (d_k = 64
    runs on two row warps per block)."""
    t = torch()
    inp = synthetic.make_verify_inputs(B=3, N=6, Hk=1, Hv=2, dk=dk, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=5, tree=True)
    good_snap, good_o = _oracle(inp)
    bad = dict(inp)
    bad["parent"] = inp["parent"].copy()
    bad["parent"][1, 3] = 4          # forward reference
    out = verify_on_gpu(gpu_lib, bad)
    assert out["status"] == gpu_lib.GDN_ERR_BAD_TREE
    for b in (0, 2):
        assert_close(out["o"][b], good_o[b], f"sequence {b} o")
    assert not np.any(out["snap"][1]), "the bad sequence must be skipped"

    bad = dict(inp)
    bad["slot"] = inp["slot"].copy()
    bad["slot"][2] = 99
    out = verify_on_gpu(gpu_lib, bad)
    assert out["status"] == gpu_lib.GDN_ERR_SLOT_RANGE
    assert_close(out["snap"][0], good_snap[0], "sequence 0 snapshots")

    out = verify_on_gpu(gpu_lib, inp)
    cache = out["cache_t"]
    before = cache.clone()
    st = t.zeros(1, dtype=t.int32, device="cuda")
    acc = t.tensor([2, 6, 0], dtype=t.int32, device="cuda")   # 6 is out of range
    gpu_lib.gdn_commit_accepted(out["snap_t"], acc, cache, B=3, N=6, Hv=2, dk=dk, dv=32,
                                slot=out["slot_t"], n_slots=inp["n_slots"], status=st)
    t.cuda.synchronize()
    assert st.item() == gpu_lib.GDN_ERR_ACCEPT_RANGE
    s = inp["slot"]
    assert t.equal(cache[s[1]], before[s[1]])
    assert t.equal(cache[s[0]], out["snap_t"][0, 2]) and t.equal(cache[s[2]], out["snap_t"][2, 0])


def test_rounds_of_verify_and_commit_match_one_sequential_run(gpu_lib):
    """Several speculative rounds on the GPU (verify from the cache, commit the
    accepted prefix) reach the state of one token-by-token run over the
    accepted tokens (oracle), i.e. speculation does not change the state."""
    t = torch()
    rng = np.random.default_rng(8)
    Hk, Hv, d, N = 2, 6, 128, 16
    first = synthetic.make_verify_inputs(B=1, N=N, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype="bf16",
                                         alpha_kind="near_one", state_sigma=0.05, seed=300)
    cache = dev(first["cache"])
    start = first["cache"][first["slot"][0]].astype(np.float64)
    slot = dev(first["slot"])
    acc_parts = {key: [] for key in ("q_f64", "k_f64", "v_f64", "alpha", "beta")}
    for r in range(5):
        inp = first if r == 0 else synthetic.make_verify_inputs(
            B=1, N=N, Hk=Hk, Hv=Hv, dk=d, dv=d, dtype="bf16", alpha_kind="near_one",
            state_sigma=0.05, seed=300 + r)
        snap = t.empty((1, N, Hv, d, d), device="cuda")
        o = t.empty((1, N, Hv, d), device="cuda")
        gpu_lib.gdn_verify_chain(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                                 dev(inp["beta"]), cache, snap, o, slot=slot, n_slots=1)
        L = int(rng.integers(1, N + 1))
        gpu_lib.gdn_commit_accepted(snap, t.tensor([L - 1], dtype=t.int32, device="cuda"), cache,
                                    B=1, N=N, Hv=Hv, dk=d, dv=d, slot=slot, n_slots=1)
        for key in acc_parts:
            acc_parts[key].append(inp[key][0, :L])
    t.cuda.synchronize()
    cat = {key: np.concatenate(v) for key, v in acc_parts.items()}
    T = cat["alpha"].shape[0]
    st, final, _ = oracle.prefill_step(cat["q_f64"], cat["k_f64"], cat["v_f64"], cat["alpha"],
                                       cat["beta"], start, T=T, Hk=Hk, Hv=Hv, dk=d, dv=d)
    assert st == oracle.OK
    assert_close(cache.cpu().numpy()[0], final, "state after rounds")


def test_outputs_have_guard_canaries_after_commit(gpu_lib):
    """The commit writes exactly the accepted slots of the cache and nothing past it."""
    t = torch()
    inp = synthetic.chain16(seed=5)
    out = verify_on_gpu(gpu_lib, inp)
    n = 48 * 128 * 128
    cache, back = guarded((1, 48, 128, 128))
    cache.copy_(out["cache_t"])
    gpu_lib.gdn_commit_accepted(out["snap_t"], dev(inp["accept"]), cache, B=1, N=16, Hv=48,
                                dk=128, dv=128, slot=t.zeros(1, dtype=t.int32, device="cuda"),
                                n_slots=1)
    t.cuda.synchronize()
    assert canaries_ok(back, n)


@pytest.mark.parametrize("shape", ["star", "path", "broom", "two_paths"])
def test_tree_kernel_level_shapes(gpu_lib, shape):
    """The tree kernel walks depth levels with four warps: a star (one level of
    63 nodes), a path (64 levels of one node: every node on the same warp), a
    broom (a path then a fan) and two interleaved paths (siblings alternate,
    so parents are read back from snapshots written by another warp); three
    sequences with different trees, all against the oracle, depths exact."""
    B, N = 3, 64
    inp = synthetic.make_verify_inputs(B=B, N=N, Hk=2, Hv=4, dk=128, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05,
                                       seed=9100 + len(shape), tree=True, n_slots=B + 1,
                                       depth_cap=64)
    par = np.empty((B, N), np.int32)
    for b in range(B):
        n = np.arange(N)
        if shape == "star":
            p = np.where(n == 0, -1, 0)
        elif shape == "path":
            p = n - 1
        elif shape == "broom":
            p = np.where(n < 20 + b, n - 1, 19 + b)
            p[0] = -1
        else:
            p = np.where(n <= 2, n - 1, n - 2)
            p[0], p[1], p[2] = -1, 0, 0
        par[b] = p
    inp = dict(inp, parent=par)
    out = verify_on_gpu(gpu_lib, inp)
    snap, o = _oracle(inp)
    assert out["status"] == 0
    assert_close(out["o"], o, f"{shape} o")
    assert_close(out["snap"], snap, f"{shape} snapshots")
    st, depth = oracle.tree_depth(par)
    assert st == oracle.OK and np.array_equal(out["depth"], depth)


def test_tree_depth_cap_skips_only_the_deep_tree(gpu_lib):
    """max_depth: a star (depth 2), a path (depth 8) and a broom (a path of 4
    then a fan: depth 5) under a cap of 5.  The path is skipped and reported
    as GDN_ERR_BAD_TREE, its depths still written; the others match the
    oracle run under the same cap.  At a cap of 8 nothing is skipped."""
    t = torch()
    B, N = 3, 8
    inp = synthetic.make_verify_inputs(B=B, N=N, Hk=1, Hv=2, dk=128, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=77,
                                       tree=True)
    n = np.arange(N)
    par = np.stack([np.where(n == 0, -1, 0), n - 1, np.where(n < 4, n - 1, 3)]).astype(np.int32)
    inp = dict(inp, parent=par)
    for cap, want in ((5, gpu_lib.GDN_ERR_BAD_TREE), (8, 0)):
        snap, snap_back = guarded((B, N, 2, 128, 32))
        o, o_back = guarded((B, N, 2, 32))
        st = t.zeros(1, dtype=t.int32, device="cuda")
        depth = t.full((B, N), -9, dtype=t.int32, device="cuda")
        gpu_lib.gdn_verify_tree(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                                dev(inp["beta"]), dev(inp["cache"]), snap, o, dev(par),
                                depth_out=depth, slot=dev(inp["slot"]), n_slots=inp["n_slots"],
                                status=st, max_depth=cap)
        t.cuda.synchronize()
        assert st.item() == want
        assert canaries_ok(snap_back, snap.numel()) and canaries_ok(o_back, o.numel())
        ost, ref_snap, ref_o = oracle.verify(
            inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"], inp["beta"], inp["cache"],
            inp["slot"], par, B=B, N=N, Hk=1, Hv=2, dk=128, dv=32, n_slots=inp["n_slots"],
            max_depth=cap)
        assert ost == (oracle.ERR_BAD_TREE if want else oracle.OK)
        _, ref_depth = oracle.tree_depth(par)
        assert np.array_equal(depth.cpu().numpy(), ref_depth)
        got_snap, got_o = snap.cpu().numpy(), o.cpu().numpy()
        for b in range(B):
            if want and b == 1:
                assert not np.any(got_snap[b]) and not np.any(got_o[b]), "deep tree not skipped"
                continue
            assert_close(got_snap[b], ref_snap[b], f"cap {cap} sequence {b} snapshots")
            assert_close(got_o[b], ref_o[b], f"cap {cap} sequence {b} o")


def test_tree_shape_follows_parents_rewritten_between_launches(gpu_lib):
    """One parent buffer rewritten on the launch stream before each of eight
    back-to-back tree verifies, as a drafter that reuses its buffer would (the
    tree kernel reads the parent array before its programmatic wait to work
    the shape out early and reads it again after the wait): every launch
    follows the array as its predecessors on the stream left it, against the
    oracle, depths exact.  Launches of 48 blocks, so the early analysis runs."""
    t = torch()
    B, N, Hk, Hv, dk, dv = 2, 22, 2, 6, 128, 64
    inp = synthetic.make_verify_inputs(B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=31337,
                                       tree=True)
    rng = np.random.default_rng(31338)
    n = np.arange(N)
    trees = [inp["parent"],
             np.stack([synthetic.random_tree(rng, N) for _ in range(B)]),
             np.stack([np.where(n == 0, -1, 0)] * B),          # a star
             np.stack([n - 1] * B)]                              # a path
    trees = [np.ascontiguousarray(p, dtype=np.int32) for p in trees]
    q, k, v = dev(inp["q"]), dev(inp["k"]), dev(inp["v"])
    alpha, beta, cache, slot = dev(inp["alpha"]), dev(inp["beta"]), dev(inp["cache"]), dev(inp["slot"])
    srcs = [dev(p) for p in trees]
    parent = t.empty_like(srcs[0])
    st = t.zeros(1, dtype=t.int32, device="cuda")
    runs = []
    for i in (0, 1, 2, 3, 1, 0, 3, 2):
        parent.copy_(srcs[i])
        snap = t.empty((B, N, Hv, dk, dv), device="cuda")
        o = t.empty((B, N, Hv, dv), device="cuda")
        depth = t.empty((B, N), dtype=t.int32, device="cuda")
        gpu_lib.gdn_verify_tree(q, k, v, alpha, beta, cache, snap, o, parent, depth_out=depth,
                                slot=slot, n_slots=inp["n_slots"], status=st)
        runs.append((i, snap, o, depth))
    t.cuda.synchronize()
    assert st.item() == 0
    refs = {}
    for i, snap, o, depth in runs:
        if i not in refs:
            refs[i] = _oracle(dict(inp, parent=trees[i])), oracle.tree_depth(trees[i])[1]
        (ref_snap, ref_o), ref_depth = refs[i]
        assert np.array_equal(depth.cpu().numpy(), ref_depth), f"tree {i}: depths"
        assert_close(o.cpu().numpy(), ref_o, f"tree {i} o")
        assert_close(snap.cpu().numpy(), ref_snap, f"tree {i} snapshots")
