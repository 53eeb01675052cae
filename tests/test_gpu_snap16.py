"""16-bit persisted states on the GPU (gdn_verify_chain_f16, gdn_verify_tree_f16,
gdn_commit_accepted_f16) against the fp32 path and the oracle, through the C
ABI.  The bar for a binary16 snapshot is the float bar plus its own rounding:
|gpu - oracle| <= 2e-3 * rms(oracle) + 2^-11 * |oracle| element by element
(2^-11 is the unit roundoff of round-to-nearest binary16)."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import TOL, assert_close, dev, torch, verify_on_gpu

pytestmark = pytest.mark.gpu

U16 = 2.0 ** -11


def assert_close16(gpu, ref, what, ulps=1):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    excess = np.abs(gpu - ref) - ulps * U16 * np.abs(ref)
    e = float(np.max(excess)) / rms
    assert e <= TOL, f"{what}: binary16 excess error {e:.3e} x rms > {TOL}"


def _run16(gdn, inp, tile=0):
    t = torch()
    B, N, Hv, dk, dv = inp["B"], inp["N"], inp["Hv"], inp["dk"], inp["dv"]
    snap16 = t.full((B, N, Hv, dk, dv), float("nan"), dtype=t.float16, device="cuda")
    o = t.empty((B, N, Hv, dv), device="cuda")
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gdn.gdn_verify_chain_f16(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                             dev(inp["beta"]), dev(inp["cache"]), snap16, o,
                             slot=dev(inp["slot"]), n_slots=inp["n_slots"], status=st,
                             tile_cols=tile)
    t.cuda.synchronize()
    assert st.item() == 0
    return snap16, o


@pytest.mark.parametrize("tile", [0, 8])
def test_chain16_f16_snapshots(gpu_lib, tile):
    inp = synthetic.chain16()
    ref = verify_on_gpu(gpu_lib, inp, tile_cols=tile)
    snap16, o = _run16(gpu_lib, inp, tile)
    s16 = snap16.cpu().numpy()
    assert np.array_equal(o.cpu().numpy(), ref["o"]), "outputs must not change"
    assert np.array_equal(s16.view(np.uint16), ref["snap"].astype(np.float16).view(np.uint16)), \
        "binary16 snapshots are not the round-to-nearest-even of the fp32 states"
    st, osnap, oo = oracle.verify_inputs(inp)
    assert st == oracle.OK
    assert_close(o.cpu().numpy(), oo, "o")
    assert_close16(s16, osnap, "binary16 snapshots vs oracle")


def test_batched_f16_snapshots_and_commit(gpu_lib):
    t = torch()
    inp = synthetic.make_verify_inputs(B=4, N=16, Hk=4, Hv=12, dk=128, dv=128, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=7800,
                                       n_slots=6)
    snap16, _ = _run16(gpu_lib, inp)
    cache = dev(inp["cache"])
    acc = inp["accept"].copy()
    acc[2] = 16                      # out of range: sequence 2 keeps its state
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gpu_lib.gdn_commit_accepted_f16(snap16, dev(acc), cache, B=4, N=16, Hv=12, dk=128, dv=128,
                                    slot=dev(inp["slot"]), n_slots=6, status=st)
    t.cuda.synchronize()
    assert st.item() == gpu_lib.GDN_ERR_ACCEPT_RANGE
    got = cache.cpu().numpy()
    s16 = snap16.cpu().numpy()
    for b in range(4):
        sl = inp["slot"][b]
        if b == 2:
            assert np.array_equal(got[sl], inp["cache"][sl])
        else:
            assert np.array_equal(got[sl], s16[b, acc[b]].astype(np.float32)), f"commit {b}"


def test_rounds_with_f16_commits(gpu_lib):
    """Blocks verified with binary16 snapshots and committed through them:
    the committed state carries one binary16 rounding per block; the oracle
    takes the same rounding of its own accepted state."""
    t = torch()
    rng = np.random.default_rng(7900)
    Hk, Hv, dk, dv, N = 2, 6, 128, 128, 16
    cache_t = None
    ocache = None
    for r in range(5):
        inp = synthetic.make_verify_inputs(B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                           alpha_kind="near_one", state_sigma=0.05,
                                           seed=7900 + r, n_slots=1, slot_perm=False)
        if cache_t is None:
            cache_t = dev(inp["cache"])
            ocache = inp["cache"].astype(np.float64)
        snap16 = t.empty((1, N, Hv, dk, dv), dtype=t.float16, device="cuda")
        o = t.empty((1, N, Hv, dv), device="cuda")
        gpu_lib.gdn_verify_chain_f16(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                                     dev(inp["alpha"]), dev(inp["beta"]), cache_t, snap16, o,
                                     slot=dev(inp["slot"]), n_slots=1)
        L = int(rng.integers(1, N + 1))
        gpu_lib.gdn_commit_accepted_f16(snap16, dev(np.array([L - 1], np.int32)), cache_t, B=1,
                                        N=N, Hv=Hv, dk=dk, dv=dv, slot=dev(inp["slot"]),
                                        n_slots=1)
        st, osnap, _ = oracle.verify(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                     inp["beta"], ocache, inp["slot"], None, B=1, N=N, Hk=Hk,
                                     Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        ocache = osnap[0, L - 1][None].astype(np.float16).astype(np.float64)
    t.cuda.synchronize()
    assert_close16(cache_t.cpu().numpy(), ocache, "state after 5 binary16 commits", ulps=2)


def _run_tree16(gdn, inp, tile=0, row_warps=0, max_depth=0):
    t = torch()
    B, N, Hv, dk, dv = inp["B"], inp["N"], inp["Hv"], inp["dk"], inp["dv"]
    snap16 = t.full((B, N, Hv, dk, dv), float("nan"), dtype=t.float16, device="cuda")
    o = t.full((B, N, Hv, dv), float("nan"), device="cuda")
    st = t.zeros(1, dtype=t.int32, device="cuda")
    depth = t.zeros((B, N), dtype=t.int32, device="cuda")
    gdn.gdn_verify_tree_f16(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                            dev(inp["beta"]), dev(inp["cache"]), snap16, o, dev(inp["parent"]),
                            depth_out=depth, slot=dev(inp["slot"]), n_slots=inp["n_slots"],
                            status=st, tile_cols=tile, row_warps=row_warps, max_depth=max_depth)
    t.cuda.synchronize()
    return int(st.item()), snap16, o, depth


TREE_WARPS = 4      # warps of a tree block
STASH_SLOTS = 3      # stashed states per depth level


def rounded_edges(parent):
    """For each node, whether the level-by-level tree walk continues it from
    its parent's binary16 snapshot (True) rather than from the parent's exact
    fp32 state.  The walk keeps a parent exact when the warp that formed it
    takes the child next (its registers), or when the parent is one of the
    first STASH_SLOTS nodes of its depth that have children (the shared-memory
    stash); the root starts from the fp32 cache.  The warps of a block take
    the nodes of each depth level round robin, in index order."""
    N = len(parent)
    depth = [0] * N
    for n in range(N):
        depth[n] = 1 if parent[n] < 0 else depth[parent[n]] + 1
    has_child = [False] * N
    for n in range(1, N):
        has_child[parent[n]] = True
    stashed = [False] * N
    for n in range(N):
        rank = sum(1 for m in range(n) if has_child[m] and depth[m] == depth[n])
        stashed[n] = has_child[n] and rank < STASH_SLOTS
    order = sorted(range(N), key=lambda n: (depth[n], n))
    held = [-1] + [-2] * (TREE_WARPS - 1)     # warp 0 starts with the cached state
    rounded = [False] * N
    for d in range(1, max(depth) + 1):
        level = [n for n in order if depth[n] == d]
        for i, n in enumerate(level):
            w = i % TREE_WARPS
            p = parent[n]
            rounded[n] = p >= 0 and held[w] != p and not stashed[p]
            held[w] = n
    return rounded


def rounded_walk_reference(inp, b):
    """The oracle stepped node by node over sequence b's tree, each node
    continuing from its parent's oracle state, rounded to binary16 (nearest
    even) exactly where rounded_edges() says the walk re-reads it.
    Returns (snap [N][Hv][dk][dv], o [N][Hv][dv]) in float64."""
    N, Hk, Hv, dk, dv = inp["N"], inp["Hk"], inp["Hv"], inp["dk"], inp["dv"]
    parent = [int(x) for x in inp["parent"][b]]
    rnd = rounded_edges(parent)
    snaps = np.zeros((N, Hv, dk, dv))
    outs = np.zeros((N, Hv, dv))
    cache0 = inp["cache"][inp["slot"][b]].astype(np.float64)
    for n in range(N):
        p = parent[n]
        src = cache0 if p < 0 else snaps[p]
        if rnd[n]:
            src = src.astype(np.float16).astype(np.float64)
        sl = (slice(b, b + 1), slice(n, n + 1))
        st, snap, o = oracle.verify(inp["q_f64"][sl], inp["k_f64"][sl], inp["v_f64"][sl],
                                    inp["alpha"][sl], inp["beta"][sl], src[None],
                                    np.zeros(1, np.int32), None, B=1, N=1, Hk=Hk, Hv=Hv, dk=dk,
                                    dv=dv)
        assert st == oracle.OK
        snaps[n], outs[n] = snap[0, 0], o[0, 0]
    return snaps, outs


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (8, 1)])
def test_tree22_f16_snapshots(gpu_lib, tile):
    """The DDTree block with binary16 snapshots: every parent of the test tree
    is kept exact (registers or the stash), so every persisted state is within
    the binary16 bar of the plain oracle and the outputs within the float
    bar; depths exact."""
    inp = synthetic.tree22()
    assert not any(rounded_edges([int(x) for x in inp["parent"][0]]))
    st, snap16, o, depth = _run_tree16(gpu_lib, inp, *tile)
    assert st == 0
    ost, osnap, oo = oracle.verify_inputs(inp)
    assert ost == oracle.OK
    assert_close(o.cpu().numpy(), oo, "tree22 o")
    assert_close16(snap16.cpu().numpy(), osnap, "tree22 binary16 snapshots vs oracle")
    assert np.array_equal(depth.cpu().numpy(), oracle.tree_depth(inp["parent"])[1])


def test_rounded_walk_reference_is_the_oracle_on_exact_trees():
    """Pin of the reference used below: with no rounded edge (a path, whose
    every parent is stashed) stepping the oracle node by node equals the
    oracle's own tree run."""
    inp = synthetic.make_verify_inputs(B=1, N=12, Hk=1, Hv=2, dk=16, dv=16, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=9250,
                                       tree=True)
    inp = dict(inp, parent=np.arange(-1, 11, dtype=np.int32)[None])
    assert not any(rounded_edges(list(range(-1, 11))))
    snaps, outs = rounded_walk_reference(inp, 0)
    st, osnap, oo = oracle.verify_inputs(inp)
    assert st == oracle.OK
    assert np.allclose(snaps, osnap[0], rtol=1e-12, atol=1e-14)
    assert np.allclose(outs, oo[0], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("shape", ["star", "path", "broom", "random"])
def test_tree64_f16_snapshots(gpu_lib, shape):
    """64-node trees of several shapes, three sequences, binary16 snapshots.
    A node whose parent is neither in a warp's registers nor stashed continues
    from the parent's binary16 snapshot, as an f16 intermediate cache does:
    compared with the oracle stepped over the same tree with the same
    roundings (snapshots at the binary16 bar, outputs at the float bar)."""
    B, N = 3, 64
    inp = synthetic.make_verify_inputs(B=B, N=N, Hk=2, Hv=4, dk=128, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05,
                                       seed=9300 + len(shape), tree=True, n_slots=B + 1,
                                       depth_cap=64)
    if shape != "random":
        n = np.arange(N)
        p = {"star": np.where(n == 0, -1, 0), "path": n - 1,
             "broom": np.where(n < 24, n - 1, 23)}[shape].astype(np.int32)
        p[0] = -1
        inp = dict(inp, parent=np.tile(p, (B, 1)))
    st, snap16, o, depth = _run_tree16(gpu_lib, inp)
    assert st == 0
    s16, og = snap16.cpu().numpy(), o.cpu().numpy()
    for b in range(B):
        rsnap, ro = rounded_walk_reference(inp, b)
        assert_close(og[b], ro, f"{shape} o, sequence {b}")
        assert_close16(s16[b], rsnap, f"{shape} binary16 snapshots, sequence {b}")
    if shape == "random":
        assert any(any(rounded_edges([int(x) for x in inp["parent"][b]])) for b in range(B)), \
            "the random trees must exercise the rounded re-read"
    assert np.array_equal(depth.cpu().numpy(), oracle.tree_depth(inp["parent"])[1])


def test_tree_f16_depth_cap_and_bad_tree(gpu_lib):
    """The binary16 tree path reports a tree deeper than max_depth and a
    malformed parent array as GDN_ERR_BAD_TREE and skips only that sequence."""
    inp = synthetic.make_verify_inputs(B=3, N=8, Hk=1, Hv=2, dk=128, dv=32, dtype="bf16",
                                       alpha_kind="near_one", state_sigma=0.05, seed=9400,
                                       tree=True)
    n = np.arange(8)
    par = np.stack([np.where(n == 0, -1, 0), n - 1, np.where(n < 4, n - 1, 3)]).astype(np.int32)
    inp = dict(inp, parent=par)
    st, snap16, o, _ = _run_tree16(gpu_lib, inp, max_depth=5)
    assert st == gpu_lib.GDN_ERR_BAD_TREE
    s16 = snap16.cpu().numpy()
    assert np.all(np.isnan(s16[1])), "the too-deep tree must be skipped"
    ost, osnap, _ = oracle.verify_inputs(inp)
    for b in (0, 2):
        assert_close16(s16[b], osnap[b], f"sequence {b}")
    bad = dict(inp, parent=par.copy())
    bad["parent"][2, 5] = 6
    st, snap16, _, _ = _run_tree16(gpu_lib, bad)
    assert st == gpu_lib.GDN_ERR_BAD_TREE
    assert np.all(np.isnan(snap16.cpu().numpy()[2]))


def test_tree_rounds_with_f16_commits(gpu_lib):
    """Tree blocks verified with binary16 snapshots and committed through them
    (accepted node of each block), against an oracle that rounds its own
    accepted state the same way."""
    t = torch()
    Hk, Hv, dk, dv, N = 2, 6, 128, 128, 22
    cache_t, ocache = None, None
    for r in range(4):
        inp = synthetic.make_verify_inputs(B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                           alpha_kind="near_one", state_sigma=0.05,
                                           seed=9500 + r, n_slots=1, slot_perm=False, tree=True)
        if cache_t is None:
            cache_t = dev(inp["cache"])
            ocache = inp["cache"].astype(np.float64)
        snap16 = t.empty((1, N, Hv, dk, dv), dtype=t.float16, device="cuda")
        o = t.empty((1, N, Hv, dv), device="cuda")
        gpu_lib.gdn_verify_tree_f16(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                                    dev(inp["alpha"]), dev(inp["beta"]), cache_t, snap16, o,
                                    dev(inp["parent"]), slot=dev(inp["slot"]), n_slots=1)
        acc = int(inp["accept"][0])
        gpu_lib.gdn_commit_accepted_f16(snap16, dev(np.array([acc], np.int32)), cache_t, B=1,
                                        N=N, Hv=Hv, dk=dk, dv=dv, slot=dev(inp["slot"]),
                                        n_slots=1)
        st, osnap, _ = oracle.verify(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                     inp["beta"], ocache, inp["slot"], inp["parent"], B=1, N=N,
                                     Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        ocache = osnap[0, acc][None].astype(np.float16).astype(np.float64)
    t.cuda.synchronize()
    assert_close16(cache_t.cpu().numpy(), ocache, "state after 4 binary16 tree commits", ulps=2)
