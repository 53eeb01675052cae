"""Convolution-history commit on the GPU (gdn_conv_commit) against the oracle,
bit for bit, through the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic
from gpu_helpers import dev, torch

pytestmark = pytest.mark.gpu

C_QKV = 2 * 16 * 128 + 48 * 128   # q, k and v channels of one GDN layer


def _values(rng, shape, dtype):
    x = rng.standard_normal(shape).astype(np.float32)
    if dtype == "bf16":
        return synthetic.f32_to_bf16_bits(x)
    return x


def _as_f64(a):
    return (synthetic.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


def _run(gdn, x, state, accept, parent=None, slot=None, status=None):
    t = torch()
    st_t = dev(state)
    gdn.gdn_conv_commit(dev(x), st_t, dev(np.asarray(accept, np.int32)),
                        parent=None if parent is None else dev(parent),
                        slot=None if slot is None else dev(slot), status=status)
    t.cuda.synchronize()
    return st_t


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("tree", [False, True])
def test_conv_commit_matches_oracle(gpu_lib, dtype, tree):
    rng = np.random.default_rng(8000 + tree)
    B, N, W, n_slots = 4, 16, 3, 6
    x = _values(rng, (B, N, C_QKV), dtype)
    state = _values(rng, (n_slots, C_QKV, W), dtype)
    slot = rng.permutation(n_slots)[:B].astype(np.int32)
    parent = (np.stack([synthetic.random_tree(rng, N) for _ in range(B)]).astype(np.int32)
              if tree else None)
    accept = rng.integers(0, N, B).astype(np.int32)
    accept[0] = 0            # a path shorter than the window
    got = _run(gpu_lib, x, state, accept, parent, slot).cpu()
    got = got.view(torch().int16).numpy().view(np.uint16) if dtype == "bf16" else got.numpy()
    want = _as_f64(state).copy()
    assert oracle.conv_commit(_as_f64(x), want, slot, parent, accept) == oracle.OK
    assert np.array_equal(_as_f64(got), want)


@pytest.mark.parametrize("W", [1, 8])
def test_conv_commit_window_sizes_and_rounds(gpu_lib, W):
    t = torch()
    rng = np.random.default_rng(8100 + W)
    C, N = 300, 5
    state0 = rng.standard_normal((2, C, W)).astype(np.float32)
    st_t = dev(state0)
    want = state0.astype(np.float64)
    for r in range(6):
        x = rng.standard_normal((1, N, C)).astype(np.float32)
        acc = np.array([int(rng.integers(0, N))], np.int32)
        gpu_lib.gdn_conv_commit(dev(x), st_t, dev(acc), slot=dev(np.array([1], np.int32)))
        assert oracle.conv_commit(x, want, np.array([1], np.int32), None, acc) == oracle.OK
    t.cuda.synchronize()
    assert np.array_equal(st_t.cpu().numpy().astype(np.float64), want)


def test_conv_commit_errors_skip_only_the_bad_sequence(gpu_lib):
    t = torch()
    rng = np.random.default_rng(8200)
    B, N, C, W = 2, 8, 700, 3
    x = rng.standard_normal((B, N, C)).astype(np.float32)
    state = rng.standard_normal((3, C, W)).astype(np.float32)
    parent = np.stack([synthetic.random_tree(rng, N) for _ in range(B)]).astype(np.int32)
    cases = [(np.array([3, N], np.int32), parent, np.array([0, 1], np.int32),
              gpu_lib.GDN_ERR_ACCEPT_RANGE),
             (np.array([3, 4], np.int32), parent, np.array([0, 7], np.int32),
              gpu_lib.GDN_ERR_SLOT_RANGE)]
    bad_tree = parent.copy()
    bad_tree[1, 5] = 6
    cases.append((np.array([3, 4], np.int32), bad_tree, np.array([0, 1], np.int32),
                  gpu_lib.GDN_ERR_BAD_TREE))
    for acc, par, slot, code in cases:
        st = t.zeros(1, dtype=t.int32, device="cuda")
        got = _run(gpu_lib, x, state, acc, par, slot, status=st).cpu().numpy()
        assert st.item() == code
        want = state.astype(np.float64)
        assert oracle.conv_commit(x, want, slot, par, acc, n_slots=3) == code
        assert np.array_equal(got.astype(np.float64), want)
