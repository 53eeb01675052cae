"""Chunked prefill on the GPU against the step-by-step oracle, element by
element, through the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, canaries_ok, dev, guarded, torch

pytestmark = pytest.mark.gpu


def run_prefill(gdn, inp):
    t = torch()
    T, Hk, Hv, dk, dv = inp["T"], inp["Hk"], inp["Hv"], inp["dk"], inp["dv"]
    q, k, v = dev(inp["q"]), dev(inp["k"]), dev(inp["v"])
    alpha, beta = dev(inp["alpha"]), dev(inp["beta"])
    state, s_back = guarded((Hv, dk, dv))
    state.copy_(dev(inp["state"]))
    o, o_back = guarded((T, Hv, dv), fill=float("nan"))
    wbytes = gdn.gdn_prefill_workspace_bytes(T, Hk, Hv, dk, dv, 64)
    ws = t.empty(max(wbytes, 16), dtype=t.uint8, device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    gdn.gdn_prefill_chunked(q, k, v, alpha, beta, state, o, ws, status=status)
    t.cuda.synchronize()
    assert status.item() == 0, "a bounded wait inside the prefill expired"
    assert canaries_ok(s_back, state.numel()), "state buffer overrun"
    assert canaries_ok(o_back, o.numel()), "output buffer overrun"
    return state.cpu().numpy(), o.cpu().numpy()


def oracle_prefill(inp, heads=None):
    st, H, O = oracle.prefill_step(inp["q_f64"], inp["k_f64"], inp["v_f64"], inp["alpha"],
                                   inp["beta"], inp["state"], T=inp["T"], Hk=inp["Hk"],
                                   Hv=inp["Hv"], dk=inp["dk"], dv=inp["dv"], heads=heads)
    assert st == oracle.OK
    return H, O


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("heads", [(1, 3), (2, 2), (4, 12)])
def test_prefill_ragged_lengths(gpu_lib, T, heads):
    Hk, Hv = heads
    inp = synthetic.make_prefill_inputs(T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="near_one", state_sigma=0.05,
                                        seed=4000 + T + Hv)
    H, O = run_prefill(gpu_lib, inp)
    Hr, Or = oracle_prefill(inp)
    assert_close(O, Or, f"prefill o T={T}")
    assert_close(H, Hr, f"prefill state T={T}")


def test_prefill_extreme_decay(gpu_lib):
    """Gates near zero on part of the sequence: the log decay spans hundreds
    across a chunk, beyond what a product of two exponentials can hold in
    fp32, so the preparation takes each decay ratio from its own exponential."""
    inp = synthetic.make_prefill_inputs(T=192, Hk=1, Hv=3, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="unit", state_sigma=0.1, seed=4343)
    inp["alpha"][64:128] = np.float32(1e-3)       # chunk 1: log decay spans ~440
    H, O = run_prefill(gpu_lib, inp)
    Hr, Or = oracle_prefill(inp)
    assert_close(O, Or, "o")
    assert_close(H, Hr, "state")


@pytest.mark.parametrize("heads", [(1, 4), (2, 16)])
def test_prefill_many_value_heads_per_qk_head(gpu_lib, heads):
    """More than three value heads share a q/k head: the preparation runs in
    several passes over the value heads (4 = 3 + 1, 8 = 3 + 3 + 2)."""
    Hk, Hv = heads
    inp = synthetic.make_prefill_inputs(T=130, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="near_one", state_sigma=0.05,
                                        seed=4500 + Hv)
    H, O = run_prefill(gpu_lib, inp)
    Hr, Or = oracle_prefill(inp)
    assert_close(O, Or, f"prefill o heads={heads}")
    assert_close(H, Hr, f"prefill state heads={heads}")


def test_prefill_wide_decay(gpu_lib):
    """alpha = exp(-softplus(z)) over (0, 1): decays within a chunk reach ~1e-20."""
    inp = synthetic.make_prefill_inputs(T=256, Hk=2, Hv=6, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="unit", state_sigma=0.1, seed=4242)
    H, O = run_prefill(gpu_lib, inp)
    Hr, Or = oracle_prefill(inp)
    assert_close(O, Or, "o")
    assert_close(H, Hr, "state")


@pytest.mark.parametrize("group", [0, 8, 15])
def test_prefill8192_sampled_heads(gpu_lib, group):
    """The 8192-token, 16/48-head workload as benchmarked; one q/k head group
    (3 value heads, i.e. every column slab) compared with the step oracle."""
    inp = synthetic.prefill8192()
    H, O = run_prefill(gpu_lib, inp)
    h0 = 3 * group
    Hr, Or = oracle_prefill(inp, heads=(h0, 3))
    assert_close(O[:, h0:h0 + 3], Or[:, h0:h0 + 3], f"o heads {h0}..{h0 + 2}")
    assert_close(H[h0:h0 + 3], Hr[h0:h0 + 3], f"state heads {h0}..{h0 + 2}")
    # heads the oracle did not run keep finite outputs everywhere
    assert np.isfinite(O).all() and np.isfinite(H).all()


def test_prefill_empty_is_a_no_op(gpu_lib):
    t = torch()
    z = t.zeros((0, 1, 128), dtype=t.bfloat16, device="cuda")
    zv = t.zeros((0, 3, 128), dtype=t.bfloat16, device="cuda")
    ab = t.zeros((0, 3), dtype=t.float32, device="cuda")
    state = t.randn((3, 128, 128), device="cuda")
    before = state.clone()
    o = t.zeros((0, 3, 128), device="cuda")
    gpu_lib.gdn_prefill_chunked(z, z, zv, ab, ab, state, o, None)
    t.cuda.synchronize()
    assert t.equal(state, before)


def test_prefill_rejects_short_workspace(gpu_lib):
    t = torch()
    inp = synthetic.make_prefill_inputs(T=100, Hk=1, Hv=3, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="near_one", state_sigma=0.05, seed=1)
    need = gpu_lib.gdn_prefill_workspace_bytes(100, 1, 3, 128, 128, 64)
    ws = t.empty(need - 16, dtype=t.uint8, device="cuda")
    with pytest.raises(gpu_lib.GdnError) as e:
        gpu_lib.gdn_prefill_chunked(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                                    dev(inp["alpha"]), dev(inp["beta"]), dev(inp["state"]),
                                    t.empty((100, 3, 128), device="cuda"), ws)
    assert e.value.code == gpu_lib.GDN_ERR_WORKSPACE


def _slice(inp, a, b):
    """Tokens a .. b-1 of a prefill input (the state is the caller's)."""
    out = dict(inp, T=b - a)
    for key in ("q", "k", "v", "q_f64", "k_f64", "v_f64", "alpha", "beta"):
        out[key] = np.ascontiguousarray(inp[key][a:b])
    return out


def test_prefill_split_across_calls(gpu_lib):
    """A sequence prefilled in three calls of ragged lengths (the state passed
    from call to call through the in/out state buffer) gives the outputs and
    final state of one step-by-step run over the whole sequence."""
    inp = synthetic.make_prefill_inputs(T=333, Hk=2, Hv=6, dk=128, dv=128, dtype="bf16",
                                        alpha_kind="near_one", state_sigma=0.05, seed=4500)
    Hr, Or = oracle_prefill(inp)
    state = inp["state"]
    outs = []
    for a, b in ((0, 100), (100, 164), (164, 333)):
        part = dict(_slice(inp, a, b), state=state)
        state, o = run_prefill(gpu_lib, part)
        outs.append(o)
    assert_close(np.concatenate(outs), Or, "split prefill o")
    assert_close(state, Hr, "split prefill state")


def test_prefill_then_chain_verify(gpu_lib):
    """The serving path: a prompt prefilled, then a 16-position block verified
    from the prefill's final state, equals one step-by-step run over the prompt
    and the block (the block's outputs and its last snapshot)."""
    t = torch()
    Hk, Hv, dk, dv, T, N = 2, 6, 128, 128, 130, 16
    inp = synthetic.make_prefill_inputs(T=T + N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                        alpha_kind="near_one", state_sigma=0.05, seed=4600)
    Hr, Or = oracle_prefill(inp)
    state, _ = run_prefill(gpu_lib, _slice(inp, 0, T))
    blk = _slice(inp, T, T + N)
    cache = dev(state[None].astype(np.float32))
    snap = t.empty((1, N, Hv, dk, dv), device="cuda")
    o = t.empty((1, N, Hv, dv), device="cuda")
    st = t.zeros(1, dtype=t.int32, device="cuda")
    gpu_lib.gdn_verify_chain(dev(blk["q"][None]), dev(blk["k"][None]), dev(blk["v"][None]),
                             dev(blk["alpha"][None]), dev(blk["beta"][None]), cache, snap, o,
                             n_slots=1, status=st)
    t.cuda.synchronize()
    assert st.item() == 0
    assert_close(o.cpu().numpy()[0], Or[T:], "verify after prefill: o")
    assert_close(snap.cpu().numpy()[0, N - 1], Hr, "verify after prefill: last state")
