"""Index-table commit on the GPU (gdn_commit_index, then a verify that reads
its state from the previous block's snapshot region) against the copy commit
and the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, dev, torch

pytestmark = pytest.mark.gpu


def test_commit_index_matches_oracle(gpu_lib):
    t = torch()
    rng = np.random.default_rng(7600)
    B, N, base = 300, 16, 41
    acc = rng.integers(0, N, B).astype(np.int32)
    acc[[5, 77]] = [N, -1]
    slot_t = dev(np.full(B, -3, np.int32))
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gpu_lib.gdn_commit_index(dev(acc), slot_t, N=N, base_slot=base, status=st)
    t.cuda.synchronize()
    want = np.full(B, -3, np.int32)
    assert oracle.commit_index(acc, want, N=N, base=base) == oracle.ERR_ACCEPT_RANGE
    assert st.item() == gpu_lib.GDN_ERR_ACCEPT_RANGE
    assert np.array_equal(slot_t.cpu().numpy(), want)


@pytest.mark.parametrize("tree", [False, True])
def test_rounds_through_the_index_table_equal_copy_commit(gpu_lib, tree):
    """Several blocks: (a) verify, copy commit into the cache; (b) verify
    writing into one snapshot region that the next verify also reads from
    through the slot table (in place).  Every block's outputs and snapshots
    are bit-identical, and the last state matches the oracle."""
    t = torch()
    B, N, Hk, Hv, dk, dv = 4, 16, 4, 12, 128, 128
    blocks = [synthetic.make_verify_inputs(B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                           alpha_kind="near_one", state_sigma=0.05,
                                           seed=7700 + r, tree=tree, n_slots=B)
              for r in range(3)]
    hs = Hv * dk * dv
    cache_a = dev(blocks[0]["cache"])
    slot_a = dev(blocks[0]["slot"])
    region = t.empty((B * N, Hv, dk, dv), device="cuda")
    cache_b = dev(blocks[0]["cache"])
    slot_b = dev(blocks[0]["slot"])
    ocache = np.ascontiguousarray(blocks[0]["cache"], dtype=np.float64).copy()
    for r, inp in enumerate(blocks):
        ins = [dev(inp[n]) for n in ("q", "k", "v", "alpha", "beta")]
        par = dev(inp["parent"]) if tree else None
        acc = dev(inp["accept"])
        snap_a = t.empty((B, N, Hv, dk, dv), device="cuda")
        o_a = t.empty((B, N, Hv, dv), device="cuda")
        o_b = t.empty((B, N, Hv, dv), device="cuda")
        # (a) copy commit
        if tree:
            gpu_lib.gdn_verify_tree(*ins, cache_a, snap_a, o_a, par, slot=slot_a, n_slots=B)
        else:
            gpu_lib.gdn_verify_chain(*ins, cache_a, snap_a, o_a, slot=slot_a, n_slots=B)
        gpu_lib.gdn_commit_accepted(snap_a, acc, cache_a, B=B, N=N, Hv=Hv, dk=dk, dv=dv,
                                    slot=slot_a, n_slots=B)
        # (b) index table: block 0 reads the cache, later blocks the region
        src, nsl = (cache_b, B) if r == 0 else (region, B * N)
        snap_b = region.view(B, N, Hv, dk, dv)
        if tree:
            gpu_lib.gdn_verify_tree(*ins, src, snap_b, o_b, par, slot=slot_b, n_slots=nsl)
        else:
            gpu_lib.gdn_verify_chain(*ins, src, snap_b, o_b, slot=slot_b, n_slots=nsl)
        t.cuda.synchronize()
        assert t.equal(o_a, o_b), f"block {r}: outputs differ"
        assert t.equal(snap_a, snap_b), f"block {r}: snapshots differ"
        slot_b = t.empty(B, dtype=t.int32, device="cuda")
        gpu_lib.gdn_commit_index(acc, slot_b, N=N, base_slot=0)
        # oracle: the same blocks with copy commits
        st, osnap, _ = oracle.verify(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                     inp["beta"], ocache, blocks[0]["slot"],
                                     inp["parent"] if tree else None, B=B, N=N, Hk=Hk, Hv=Hv,
                                     dk=dk, dv=dv, n_slots=B)
        assert st == oracle.OK
        assert oracle.commit(osnap, inp["accept"], ocache, blocks[0]["slot"], B=B, N=N, Hv=Hv,
                             dk=dk, dv=dv, n_slots=B) == oracle.OK
    t.cuda.synchronize()
    flat = region.view(B * N, hs).cpu().numpy()
    for b in range(B):
        got = flat[int(slot_b[b].item())].reshape(Hv, dk, dv)
        assert_close(got, ocache[blocks[0]["slot"][b]], f"final state of sequence {b}")
