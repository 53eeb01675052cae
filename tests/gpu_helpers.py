"""Shared helpers for the GPU parity tests: move synthetic inputs to the
device, allocate outputs with guard canaries, compare with the oracle."""
from __future__ import annotations

import numpy as np

TOL = 2e-3          # max |gpu - oracle| <= TOL * rms(oracle), per tensor
CANARY = -7.25e30   # written past every output buffer, must survive each call
GUARD = 64          # canary floats after each output


def torch():
    import torch as _t
    return _t


def dev(a):
    """numpy -> cuda tensor; uint16 arrays are bf16 bit patterns."""
    t = torch()
    if a.dtype == np.uint16:
        return t.from_numpy(a.view(np.int16).copy()).cuda().view(t.bfloat16)
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(shape, dtype=None, fill=0.0):
    """A contiguous float32 device tensor of `shape` followed by GUARD canaries;
    returns (view, backing)."""
    t = torch()
    n = int(np.prod(shape))
    back = t.full((n + GUARD,), CANARY, dtype=dtype or t.float32, device="cuda")
    back[:n] = fill
    return back[:n].view(*shape), back


def canaries_ok(back, n):
    return bool((back[n:] == CANARY).all().item())


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(gpu - ref))) / rms


def assert_close(gpu, ref, what, tol=TOL):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{what}: max|gpu-oracle|/rms = {e:.3e} > {tol:.1e}"
    return e


def verify_on_gpu(gdn, inp, *, tree=None, tile_cols=0, row_warps=0, status=True,
                  cache=None):
    """Run gdn_verify_chain / gdn_verify_tree on a synthetic input dict.
    Returns dict of numpy outputs plus the device tensors used."""
    t = torch()
    tree = inp["tree"] if tree is None else tree
    B, N, Hv, dk, dv = inp["B"], inp["N"], inp["Hv"], inp["dk"], inp["dv"]
    q, k, v = dev(inp["q"]), dev(inp["k"]), dev(inp["v"])
    alpha, beta = dev(inp["alpha"]), dev(inp["beta"])
    cache_t = dev(inp["cache"]) if cache is None else cache
    slot = dev(inp["slot"])
    snap, snap_back = guarded((B, N, Hv, dk, dv))
    o, o_back = guarded((B, N, Hv, dv))
    st = t.zeros(1, dtype=t.int32, device="cuda") if status else None
    depth = None
    if tree:
        parent = dev(inp["parent"])
        depth = t.zeros((B, N), dtype=t.int32, device="cuda")
        gdn.gdn_verify_tree(q, k, v, alpha, beta, cache_t, snap, o, parent, depth_out=depth,
                            slot=slot, n_slots=inp["n_slots"], status=st, tile_cols=tile_cols,
                            row_warps=row_warps)
    else:
        gdn.gdn_verify_chain(q, k, v, alpha, beta, cache_t, snap, o, slot=slot,
                             n_slots=inp["n_slots"], status=st, tile_cols=tile_cols,
                             row_warps=row_warps)
    t.cuda.synchronize()
    assert canaries_ok(snap_back, snap.numel()), "snapshot buffer overrun"
    assert canaries_ok(o_back, o.numel()), "output buffer overrun"
    return dict(snap=snap.cpu().numpy(), o=o.cpu().numpy(),
                status=None if st is None else int(st.item()),
                depth=None if depth is None else depth.cpu().numpy(),
                snap_t=snap, cache_t=cache_t, slot_t=slot)
