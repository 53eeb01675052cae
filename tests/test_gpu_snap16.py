"""16-bit persisted states on the GPU (gdn_verify_chain_f16,
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
