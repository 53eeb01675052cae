"""gdn_prefill_chunked_noalloc: the chunked prefill for callers that cannot
allocate device memory (for example a plugin whose host engine owns every
device allocation, or a path where cudaMalloc's implicit synchronisation is not
allowed and no workspace was reserved).  It runs on scratch built into the
library instead of a caller workspace; these checks call it through the C ABI
and compare it with gdn_prefill_chunked on the same inputs, twice in a row,
since consecutive calls share (and leave behind) the same scratch.

The file name makes pytest collect it after every other test file."""
import numpy as np
import pytest

import synthetic
from gpu_helpers import TOL, dev, torch

pytestmark = pytest.mark.gpu


def _with_workspace(gdn, inp):
    t = torch()
    state = dev(inp["state"]).clone()
    o = t.empty((inp["T"], inp["Hv"], inp["dv"]), device="cuda")
    need = gdn.gdn_prefill_workspace_bytes(inp["T"], inp["Hk"], inp["Hv"], inp["dk"],
                                           inp["dv"], 64)
    ws = t.empty(need, dtype=t.uint8, device="cuda")
    gdn.gdn_prefill_chunked(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha"]),
                            dev(inp["beta"]), state, o, ws)
    t.cuda.synchronize()
    return state.cpu().numpy(), o.cpu().numpy()


def _no_alloc(gdn, inp):
    t = torch()
    state = dev(inp["state"]).clone()
    o = t.empty((inp["T"], inp["Hv"], inp["dv"]), device="cuda")
    gdn.gdn_prefill_chunked_noalloc(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                                    dev(inp["alpha"]), dev(inp["beta"]), state, o)
    t.cuda.synchronize()
    return state.cpu().numpy(), o.cpu().numpy()


def _close(a, ref, what):
    err = float(np.max(np.abs(a - ref))) / float(np.sqrt(np.mean(ref.astype(np.float64) ** 2)))
    assert err <= TOL, f"{what}: {err:.3e} > {TOL}"


@pytest.mark.parametrize("shape", [dict(T=200, Hk=2, Hv=6),     # ragged last chunk
                                   dict(T=640, Hk=16, Hv=48)])  # the largest that fits
def test_no_alloc_matches_workspace_call_twice(gpu_lib, shape):
    inp = synthetic.make_prefill_inputs(dk=128, dv=128, dtype="bf16", alpha_kind="near_one",
                                        state_sigma=0.05, seed=9000 + shape["T"], **shape)
    need = gpu_lib.gdn_prefill_workspace_bytes(shape["T"], shape["Hk"], shape["Hv"], 128, 128,
                                               64)
    assert need <= gpu_lib.PREFILL_NOALLOC_SCRATCH_BYTES
    ref_state, ref_o = _with_workspace(gpu_lib, inp)
    for call in range(2):
        state, o = _no_alloc(gpu_lib, inp)
        _close(o, ref_o, f"output, call {call}")
        _close(state, ref_state, f"final state, call {call}")


def test_no_alloc_rejects_problems_beyond_its_scratch(gpu_lib):
    t = torch()
    T, Hk, Hv = 704, 16, 48   # 11 chunks x 48 heads: just over 16 MiB
    assert gpu_lib.gdn_prefill_workspace_bytes(T, Hk, Hv, 128, 128, 64) > \
        gpu_lib.PREFILL_NOALLOC_SCRATCH_BYTES
    q = t.zeros((T, Hk, 128), dtype=t.bfloat16, device="cuda")
    v = t.zeros((T, Hv, 128), dtype=t.bfloat16, device="cuda")
    g = t.ones((T, Hv), device="cuda")
    state = t.randn((Hv, 128, 128), device="cuda")
    before = state.clone()
    o = t.empty((T, Hv, 128), device="cuda")
    with pytest.raises(gpu_lib.GdnError) as e:
        gpu_lib.gdn_prefill_chunked_noalloc(q, q, v, g, g, state, o)
    assert e.value.code == gpu_lib.GDN_ERR_SCRATCH_LIMIT
    t.cuda.synchronize()
    assert t.equal(state, before)
