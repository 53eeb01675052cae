"""Checkpoint-and-replay commit on the GPU (gdn_verify_chain without snapshots,
gdn_replay_accepted) against the oracle's replay, element by element, through
the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, canaries_ok, dev, guarded, torch, verify_on_gpu

pytestmark = pytest.mark.gpu


def _oracle_replay(inp, accept, tree):
    cache = np.ascontiguousarray(inp["cache"], dtype=np.float64).copy()
    st = oracle.replay(inp["k_f64"], inp["v_f64"], inp["alpha"], inp["beta"], cache,
                       inp["slot"], inp["parent"] if tree else None, accept, B=inp["B"],
                       N=inp["N"], Hk=inp["Hk"], Hv=inp["Hv"], dk=inp["dk"], dv=inp["dv"],
                       n_slots=inp["n_slots"])
    return st, cache


def _gpu_replay(gdn, inp, accept, tree, cache_t=None, tile_cols=0, row_warps=0, status=None):
    t = torch()
    cache_t = dev(inp["cache"]) if cache_t is None else cache_t
    st = t.zeros(1, dtype=t.int32, device="cuda") if status is None else status
    gdn.gdn_replay_accepted(dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]),
                            cache_t, dev(np.asarray(accept, np.int32)),
                            parent=dev(inp["parent"]) if tree else None, slot=dev(inp["slot"]),
                            n_slots=inp["n_slots"], status=st, tile_cols=tile_cols,
                            row_warps=row_warps)
    t.cuda.synchronize()
    return int(st.item()), cache_t


def _inputs(tree, *, B=4, N=16, Hk=4, Hv=12, dk=128, dv=128, dtype="bf16", seed=7100):
    return synthetic.make_verify_inputs(B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype=dtype,
                                        alpha_kind="near_one", state_sigma=0.05, seed=seed,
                                        tree=tree, n_slots=B + 2)


@pytest.mark.parametrize("tile", [0, 16, 8])
def test_chain_verify_without_snapshots(gpu_lib, tile):
    """A chain verified with snapshots=None gives the same outputs as with them."""
    inp = synthetic.chain16()
    t = torch()
    out = verify_on_gpu(gpu_lib, inp, tile_cols=tile)
    o, o_back = guarded((1, 16, 48, 128), fill=float("nan"))
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gpu_lib.gdn_verify_chain(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                             dev(inp["beta"]), dev(inp["cache"]), None, o, slot=dev(inp["slot"]),
                             n_slots=inp["n_slots"], status=st, tile_cols=tile)
    t.cuda.synchronize()
    assert st.item() == 0 and canaries_ok(o_back, o.numel())
    assert np.array_equal(o.cpu().numpy(), out["o"])


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (16, 2), (8, 1)])
def test_chain_replay_matches_persisted_state_bitwise(gpu_lib, tile):
    """Along a chain the replay repeats the verify kernel's arithmetic: with the
    same tile, the committed state is bit for bit the persisted snapshot of the
    accepted node, and within tolerance of the oracle's replay."""
    inp = _inputs(False)
    out = verify_on_gpu(gpu_lib, inp, tile_cols=tile[0], row_warps=tile[1])
    accept = inp["accept"]
    st, cache_t = _gpu_replay(gpu_lib, inp, accept, False, tile_cols=tile[0],
                              row_warps=tile[1])
    assert st == 0
    cache = cache_t.cpu().numpy()
    ost, ocache = _oracle_replay(inp, accept, False)
    assert ost == oracle.OK
    for b in range(inp["B"]):
        sl = inp["slot"][b]
        assert np.array_equal(cache[sl], out["snap"][b, accept[b]]), f"sequence {b}"
        assert_close(cache[sl], ocache[sl], f"replayed state, sequence {b}")
    for sl in set(range(inp["n_slots"])) - set(inp["slot"].tolist()):
        assert np.array_equal(cache[sl], inp["cache"][sl]), "a slot outside the batch changed"


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (16, 2), (8, 1)])
def test_tree_replay_matches_oracle(gpu_lib, tile):
    """Tree: the ancestors of the accepted node from the root, from the cache."""
    inp = _inputs(True, seed=7200)
    accept = inp["accept"]
    st, cache_t = _gpu_replay(gpu_lib, inp, accept, True, tile_cols=tile[0], row_warps=tile[1])
    assert st == 0
    cache = cache_t.cpu().numpy()
    ost, ocache = _oracle_replay(inp, accept, True)
    assert ost == oracle.OK
    out = verify_on_gpu(gpu_lib, inp, tile_cols=tile[0], row_warps=tile[1])
    for b in range(inp["B"]):
        sl = inp["slot"][b]
        assert_close(cache[sl], ocache[sl], f"tree replay, sequence {b}")
        assert_close(cache[sl], out["snap"][b, accept[b]], f"tree replay vs persisted, {b}")


def test_tree22_replay_every_node(gpu_lib):
    """Every node of the tree22 block as the accepted one."""
    base = synthetic.tree22()
    for node in range(22):
        acc = np.array([node], np.int32)
        st, cache_t = _gpu_replay(gpu_lib, base, acc, True)
        assert st == 0
        ost, ocache = _oracle_replay(base, acc, True)
        sl = base["slot"][0]
        assert_close(cache_t.cpu().numpy()[sl], ocache[sl], f"tree22 node {node}")


@pytest.mark.parametrize("shape", [dict(dk=16, dv=16, Hk=1, Hv=3, N=1),
                                   dict(dk=32, dv=48, Hk=2, Hv=2, N=64),
                                   dict(dk=64, dv=32, Hk=1, Hv=2, N=7, dtype="f32")])
def test_replay_edge_shapes(gpu_lib, shape):
    for tree in (False, True):
        inp = _inputs(tree, B=3, seed=7300 + shape["N"], **shape)
        st, cache_t = _gpu_replay(gpu_lib, inp, inp["accept"], tree)
        assert st == 0
        ost, ocache = _oracle_replay(inp, inp["accept"], tree)
        for b in range(3):
            sl = inp["slot"][b]
            assert_close(cache_t.cpu().numpy()[sl], ocache[sl], f"{shape} tree={tree} b={b}")


def test_replay_errors_skip_only_the_bad_sequence(gpu_lib):
    inp = _inputs(True, B=2, seed=7400)
    t = torch()
    for kind in ("accept", "tree", "slot"):
        acc = inp["accept"].copy()
        case = dict(inp)
        if kind == "accept":
            acc[1] = 16
            want = -6
        elif kind == "tree":
            par = inp["parent"].copy()
            par[1, 5] = 9
            case["parent"] = par
            want = -5
        else:
            slot = inp["slot"].copy()
            slot[1] = inp["n_slots"] + 3
            case["slot"] = slot
            want = -7
        st, cache_t = _gpu_replay(gpu_lib, case, acc, True)
        assert st == want, (kind, st)
        cache = cache_t.cpu().numpy()
        ost, ocache = _oracle_replay(case, acc, True)
        assert ost == want
        sl0 = case["slot"][0]
        assert_close(cache[sl0], ocache[sl0], f"{kind}: the valid sequence commits")
        if kind != "slot":
            sl1 = case["slot"][1]
            assert np.array_equal(cache[sl1], inp["cache"][sl1]), f"{kind}: skipped sequence"
    t.cuda.synchronize()


def test_rounds_of_verify_and_replay_equal_sequential(gpu_lib):
    """Blocks verified without snapshots, each committed by replay from the
    cache, equal one token-by-token run over the accepted tokens."""
    t = torch()
    rng = np.random.default_rng(7500)
    Hk, Hv, dk, dv, N = 2, 6, 128, 128, 16
    start = None
    cache_t = None
    acc_tok = {key: [] for key in ("q_f64", "k_f64", "v_f64", "alpha", "beta")}
    for r in range(5):
        inp = synthetic.make_verify_inputs(B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                           alpha_kind="near_one", state_sigma=0.05,
                                           seed=7500 + r, n_slots=1, slot_perm=False)
        if cache_t is None:
            cache_t = dev(inp["cache"])
            start = inp["cache"][0].astype(np.float64)
        o, _ = guarded((1, N, Hv, dv))
        gpu_lib.gdn_verify_chain(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                                 dev(inp["beta"]), cache_t, None, o, slot=dev(inp["slot"]),
                                 n_slots=1)
        L = int(rng.integers(1, N + 1))
        st, cache_t = _gpu_replay(gpu_lib, inp, np.array([L - 1], np.int32), False,
                                  cache_t=cache_t)
        assert st == 0
        for key in acc_tok:
            acc_tok[key].append(inp[key][0, :L])
    cat = [np.concatenate(acc_tok[key]) for key in ("q_f64", "k_f64", "v_f64", "alpha", "beta")]
    st, sT, _ = oracle.prefill_step(*cat, start, T=cat[0].shape[0], Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    assert st == oracle.OK
    t.cuda.synchronize()
    assert_close(cache_t.cpu().numpy()[0], sT, "rounds of verify + replay")


def test_rounds_of_tree_verify_and_replay_equal_sequential(gpu_lib):
    """DDTree blocks verified without snapshots (the per-block solve), each
    committed by replaying the accepted node's ancestor path from the cache:
    every round's outputs match the oracle's verify of that block from the
    oracle's own running state, and after five rounds the cached state equals
    one token-by-token run over the accepted paths."""
    t = torch()
    Hk, Hv, dk, dv, N = 2, 6, 128, 64, 22
    start = None
    cache_t = None
    ocache = None
    acc_tok = {key: [] for key in ("q_f64", "k_f64", "v_f64", "alpha", "beta")}
    for r in range(5):
        inp = synthetic.make_verify_inputs(B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                           alpha_kind="near_one", state_sigma=0.05,
                                           seed=7600 + r, n_slots=1, slot_perm=False, tree=True)
        if cache_t is None:
            cache_t = dev(inp["cache"])
            start = inp["cache"][0].astype(np.float64)
            ocache = inp["cache"].astype(np.float64)
        o, o_back = guarded((1, N, Hv, dv), fill=float("nan"))
        st_t = t.zeros(1, dtype=t.int32, device="cuda")
        gpu_lib.gdn_verify_tree(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                                dev(inp["beta"]), cache_t, None, o, dev(inp["parent"]),
                                slot=dev(inp["slot"]), n_slots=1, status=st_t)
        t.cuda.synchronize()
        assert st_t.item() == 0 and canaries_ok(o_back, o.numel())
        ost, osnap, oo = oracle.verify(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                       inp["beta"], ocache, inp["slot"], inp["parent"], B=1, N=N,
                                       Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        assert ost == oracle.OK
        assert_close(o.cpu().numpy(), oo, f"round {r} outputs")
        acc = int(inp["accept"][0])
        st, cache_t = _gpu_replay(gpu_lib, inp, np.array([acc], np.int32), True, cache_t=cache_t)
        assert st == 0
        ocache = osnap[0, acc][None]
        path, nd = [], acc
        while nd >= 0:
            path.append(nd)
            nd = int(inp["parent"][0, nd])
        path.reverse()
        for key in acc_tok:
            acc_tok[key].append(inp[key][0, path])
    cat = [np.concatenate(acc_tok[key]) for key in ("q_f64", "k_f64", "v_f64", "alpha", "beta")]
    st, sT, _ = oracle.prefill_step(*cat, start, T=cat[0].shape[0], Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    assert st == oracle.OK
    t.cuda.synchronize()
    assert_close(cache_t.cpu().numpy()[0], sT, "rounds of tree verify + replay")


@pytest.mark.parametrize("tile", [(0, 0), (16, 1), (8, 1)])
def test_tree_verify_without_snapshots_then_replay(gpu_lib, tile):
    """A draft tree verified with snapshots=None (nothing persisted) gives the
    oracle's outputs, and the replay commit of the accepted node (the
    ancestors re-run from the cached state) gives the oracle's accepted
    state: the whole round persists no per-node state."""
    t = torch()
    inp = _inputs(True, seed=7300)
    o, o_back = guarded((inp["B"], inp["N"], inp["Hv"], inp["dv"]), fill=float("nan"))
    st = t.zeros(1, dtype=t.int32, device="cuda")
    cache_t = dev(inp["cache"])
    gpu_lib.gdn_verify_tree(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                            dev(inp["beta"]), cache_t, None, o, dev(inp["parent"]),
                            slot=dev(inp["slot"]), n_slots=inp["n_slots"], status=st,
                            tile_cols=tile[0], row_warps=tile[1])
    t.cuda.synchronize()
    assert st.item() == 0 and canaries_ok(o_back, o.numel())
    ost, osnap, oo = oracle.verify_inputs(inp)
    assert ost == oracle.OK
    assert_close(o.cpu().numpy(), oo, "tree o without snapshots")
    accept = inp["accept"]
    rst, cache_t = _gpu_replay(gpu_lib, inp, accept, True, cache_t=cache_t)
    assert rst == 0
    ost, ocache = _oracle_replay(inp, accept, True)
    assert ost == oracle.OK
    got = cache_t.cpu().numpy()
    for b in range(inp["B"]):
        sl = inp["slot"][b]
        assert_close(got[sl], ocache[sl], f"replayed state, sequence {b}")


def test_tree22_without_snapshots_matches_persisting_outputs(gpu_lib):
    """tree22: the snapshot-free verify gives the persisting verify's outputs
    within the float bar (the two run different kernels)."""
    t = torch()
    inp = synthetic.tree22()
    out = verify_on_gpu(gpu_lib, inp)
    o = t.empty((1, 22, 48, 128), device="cuda")
    gpu_lib.gdn_verify_tree(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                            dev(inp["beta"]), dev(inp["cache"]), None, o, dev(inp["parent"]),
                            slot=dev(inp["slot"]), n_slots=inp["n_slots"])
    t.cuda.synchronize()
    assert_close(o.cpu().numpy(), out["o"], "snapshot-free tree22 o vs persisting verify")
