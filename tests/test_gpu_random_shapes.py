"""Seeded random verify shapes on the GPU against the oracle: head sizes,
block lengths, batch sizes, GQA ratios, input dtypes, tile widths and tree
depth caps drawn together, so that combinations no hand-written case names
(a deep narrow tree on 8-column tiles, a one-node block in fp32, ...) are
compared element by element too."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import assert_close, verify_on_gpu

pytestmark = pytest.mark.gpu


def _draw(i):
    rng = np.random.default_rng(6100 + i)
    dk = int(rng.choice([16, 32, 64, 128]))
    dv = int(rng.choice([16, 32, 48, 128]))
    hk = int(rng.choice([1, 2]))
    wc = int(rng.choice([0, 8, 16]))
    return dict(dk=dk, dv=dv, N=int(rng.integers(1, 65)), B=int(rng.integers(1, 5)), Hk=hk,
                Hv=hk * int(rng.choice([1, 2, 3])), dtype=str(rng.choice(["bf16", "f32"])),
                tree=bool(rng.integers(0, 2)), wc=wc if wc == 0 or dv % wc == 0 else 0,
                cap=int(rng.choice([2, 4, 16, 64])), seed=6100 + i)


@pytest.mark.parametrize("i", range(16))
def test_random_verify_shape(gpu_lib, i):
    c = _draw(i)
    inp = synthetic.make_verify_inputs(B=c["B"], N=c["N"], Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"],
                                       dv=c["dv"], dtype=c["dtype"], alpha_kind="near_one",
                                       state_sigma=0.05, seed=c["seed"], tree=c["tree"],
                                       n_slots=c["B"] + 1, depth_cap=c["cap"])
    out = verify_on_gpu(gpu_lib, inp, tile_cols=c["wc"])
    st, snap, o = oracle.verify_inputs(inp)
    assert st == oracle.OK and out["status"] == 0, c
    assert_close(out["o"], o, f"o {c}")
    assert_close(out["snap"], snap, f"snapshots {c}")
    if c["tree"]:
        assert np.array_equal(out["depth"], oracle.tree_depth(inp["parent"])[1]), c
