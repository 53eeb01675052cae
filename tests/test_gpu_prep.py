"""Verify and replay from raw projections on the GPU (gdn_verify_chain_prep,
gdn_verify_tree_prep, gdn_replay_accepted_prep) against the oracle run on the
oracle-prepared inputs, through the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, dev, guarded, torch

pytestmark = pytest.mark.gpu


def _raw_block(seed, *, B=3, N=16, Hk=4, Hv=12, dk=128, dv=128, dtype="bf16", tree=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hk, dk)) * rng.uniform(0.2, 5.0, (B, N, Hk, 1))
    k = rng.standard_normal((B, N, Hk, dk)) * rng.uniform(0.2, 5.0, (B, N, Hk, 1))
    k[0, 3, 1] = 0.0                                   # a zero key stays zero
    v = rng.standard_normal((B, N, Hv, dv))
    if dtype == "bf16":
        qs, ks, vs = (synthetic.f32_to_bf16_bits(x.astype(np.float32)) for x in (q, k, v))
        q64, k64, v64 = (synthetic.bf16_bits_to_f32(x).astype(np.float64) for x in (qs, ks, vs))
    else:
        qs, ks, vs = (x.astype(np.float32) for x in (q, k, v))
        q64, k64, v64 = (x.astype(np.float64) for x in (qs, ks, vs))
    a = (rng.standard_normal((B, N, Hv)) * 2.0 - 2.5).astype(np.float32)
    b = (rng.standard_normal((B, N, Hv)) * 1.5).astype(np.float32)
    n_slots = B + 1
    cache = (rng.standard_normal((n_slots, Hv, dk, dv)) * 0.05).astype(np.float32)
    slot = rng.permutation(n_slots)[:B].astype(np.int32)
    parent = (np.stack([synthetic.random_tree(rng, N) for _ in range(B)]).astype(np.int32)
              if tree else None)
    accept = rng.integers(0, N, B).astype(np.int32)
    return dict(q=qs, k=ks, v=vs, q64=q64, k64=k64, v64=v64, a=a, b=b, cache=cache, slot=slot,
                parent=parent, accept=accept, B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv,
                n_slots=n_slots)


def _oracle(blk):
    qn, kn, al, be = oracle.prepare_inputs(blk["q64"], blk["k64"], blk["a"], blk["b"])
    st, snap, o = oracle.verify(qn, kn, blk["v64"], al, be, blk["cache"], blk["slot"],
                                blk["parent"], B=blk["B"], N=blk["N"], Hk=blk["Hk"],
                                Hv=blk["Hv"], dk=blk["dk"], dv=blk["dv"], n_slots=blk["n_slots"])
    assert st == oracle.OK
    return kn, al, be, snap, o


@pytest.mark.parametrize("tree", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_from_raw_projections(gpu_lib, tree, dtype):
    t = torch()
    blk = _raw_block(8300 + 2 * tree + (dtype == "f32"), dtype=dtype, tree=tree)
    B, N, Hv, dk, dv = blk["B"], blk["N"], blk["Hv"], blk["dk"], blk["dv"]
    snap, _ = guarded((B, N, Hv, dk, dv))
    o, _ = guarded((B, N, Hv, dv))
    st = t.zeros(1, dtype=t.int32, device="cuda")
    args = (dev(blk["q"]), dev(blk["k"]), dev(blk["v"]), dev(blk["a"]), dev(blk["b"]),
            dev(blk["cache"]), snap, o)
    if tree:
        gpu_lib.gdn_verify_tree(*args, dev(blk["parent"]), slot=dev(blk["slot"]),
                                n_slots=blk["n_slots"], status=st, prep=True)
    else:
        gpu_lib.gdn_verify_chain(*args, slot=dev(blk["slot"]), n_slots=blk["n_slots"], status=st,
                                 prep=True)
    t.cuda.synchronize()
    assert st.item() == 0
    _, _, _, osnap, oo = _oracle(blk)
    assert np.all(np.isfinite(o.cpu().numpy()))
    assert_close(o.cpu().numpy(), oo, f"o ({dtype}, tree={tree})")
    assert_close(snap.cpu().numpy(), osnap, f"snapshots ({dtype}, tree={tree})")


@pytest.mark.parametrize("tree", [False, True])
def test_replay_from_raw_projections(gpu_lib, tree):
    t = torch()
    blk = _raw_block(8400 + tree, tree=tree)
    cache = dev(blk["cache"])
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gpu_lib.gdn_replay_accepted(dev(blk["k"]), dev(blk["v"]), dev(blk["a"]), dev(blk["b"]), cache,
                                dev(blk["accept"]),
                                parent=None if blk["parent"] is None else dev(blk["parent"]),
                                slot=dev(blk["slot"]), n_slots=blk["n_slots"], status=st,
                                prep=True)
    t.cuda.synchronize()
    assert st.item() == 0
    _, _, _, osnap, _ = _oracle(blk)
    got = cache.cpu().numpy()
    for b in range(blk["B"]):
        assert_close(got[blk["slot"][b]], osnap[b, blk["accept"][b]], f"replayed state {b}")
