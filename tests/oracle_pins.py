"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (closed forms, invariants, exact-rational brute force, a worked
example done by hand).  Each check takes no arguments, calls the oracle through
the `oracle` package, and raises AssertionError on a mismatch; test_oracle_pins
runs them on the real oracle and test_oracle_mutants on deliberately broken
copies of it (every planted mistake must trip at least one check).
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers
def _case(rng, *, B=2, N=5, Hk=2, Hv=4, dk=4, dv=4, tree=False, alpha=None, beta=None,
          unit_k=True, n_slots=None):
    n_slots = B if n_slots is None else n_slots
    q = rng.standard_normal((B, N, Hk, dk))
    k = rng.standard_normal((B, N, Hk, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, N, Hv, dv))
    a = rng.uniform(0.3, 1.0, (B, N, Hv)) if alpha is None else np.full((B, N, Hv), alpha)
    b = rng.uniform(0.0, 1.0, (B, N, Hv)) if beta is None else np.full((B, N, Hv), beta)
    cache = rng.standard_normal((n_slots, Hv, dk, dv)) * 0.5
    slot = rng.permutation(n_slots)[:B].astype(np.int32)
    if tree:
        parent = np.full((B, N), -1, np.int32)
        for bb in range(B):
            for i in range(1, N):
                parent[bb, i] = rng.integers(0, i)
    else:
        parent = None
    return dict(q=q, k=k, v=v, alpha=a, beta=b, cache=cache, slot=slot, parent=parent, B=B,
                N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv)


_DEFAULT = object()


def _run(c, parent=_DEFAULT, cache=None, v=None, precision="f64"):
    par = c["parent"] if parent is _DEFAULT else parent
    st, snap, o = oracle.verify(c["q"], c["k"], c["v"] if v is None else v, c["alpha"],
                                c["beta"], c["cache"] if cache is None else cache, c["slot"], par,
                                B=c["B"], N=c["N"], Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"],
                                dv=c["dv"], precision=precision)
    assert st == oracle.OK, st
    return snap, o


def _src_state(c, snap, b, n, h):
    par = c["parent"]
    p = (n - 1) if par is None else par[b, n]
    return c["cache"][c["slot"][b], h] if p < 0 else snap[b, p, h]


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol:.1e} x {scale:.3g}"


# --------------------------------------------------------------- the checks
def check_golden_hand_example():
    """Worked by hand in exact decimals (tests/golden/hand_d2_tree.json)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_d2_tree.json")))
    I, E = g["inputs"], g["expected"]
    N = len(I["parent"])
    sh = lambda x: np.array(x, dtype=np.float64).reshape(1, N, 1, 2)  # noqa: E731
    st, snap, o = oracle.verify(sh(I["q"]), sh(I["k"]), sh(I["v"]),
                                np.array(I["alpha"]).reshape(1, N, 1),
                                np.array(I["beta"]).reshape(1, N, 1),
                                np.array(I["H0"]).reshape(1, 1, 2, 2), np.zeros(1, np.int32),
                                np.array(I["parent"], np.int32).reshape(1, N), B=1, N=N, Hk=1,
                                Hv=1, dk=2, dv=2)
    assert st == oracle.OK
    _close(snap[0, :, 0], np.array(E["H"]), 1e-14, "hand example H")
    _close(o[0, :, 0], np.array(E["o"]), 1e-14, "hand example o")
    st, depth = oracle.tree_depth(np.array(I["parent"], np.int32).reshape(1, N))
    assert st == oracle.OK and depth[0].tolist() == E["depth"]


def check_identity_gate():
    """beta = 0, alpha = 1: the state never changes and o = S q."""
    rng = np.random.default_rng(11)
    for tree in (False, True):
        c = _case(rng, alpha=1.0, beta=0.0, tree=tree)
        snap, o = _run(c)
        G = c["Hv"] // c["Hk"]
        for b in range(c["B"]):
            for n in range(c["N"]):
                for h in range(c["Hv"]):
                    H0 = c["cache"][c["slot"][b], h]
                    assert np.array_equal(snap[b, n, h], H0), "state moved with beta=0, alpha=1"
                    _close(o[b, n, h], H0.T @ c["q"][b, n, h // G], 1e-13, "o = S q")


def check_delta_rule_closed_form():
    """beta = 1 and |k| = 1: after the update S k = v exactly, for any alpha."""
    rng = np.random.default_rng(12)
    for tree in (False, True):
        c = _case(rng, beta=1.0, tree=tree)
        snap, _ = _run(c)
        G = c["Hv"] // c["Hk"]
        for b in range(c["B"]):
            for n in range(c["N"]):
                for h in range(c["Hv"]):
                    Sk = snap[b, n, h].T @ c["k"][b, n, h // G]
                    _close(Sk, c["v"][b, n, h], 1e-12, "S k = v")


def check_zero_decay():
    """alpha = 0: the old state is forgotten, S_n = beta v k^T, o = beta (k.q) v."""
    rng = np.random.default_rng(13)
    c = _case(rng, alpha=0.0)
    snap, o = _run(c)
    G = c["Hv"] // c["Hk"]
    for b in range(c["B"]):
        for n in range(c["N"]):
            for h in range(c["Hv"]):
                kk, qq, vv, be = (c["k"][b, n, h // G], c["q"][b, n, h // G], c["v"][b, n, h],
                                  c["beta"][b, n, h])
                _close(snap[b, n, h], be * np.outer(kk, vv), 1e-14, "rank-1 state")
                _close(o[b, n, h], be * (kk @ qq) * vv, 1e-13, "o for alpha=0")


def check_scalar_closed_form():
    """d_k = d_v = 1: s_n = a_n s_{n-1} + b_n with a = alpha(1 - beta k^2),
    b = beta v k (a first-order linear recurrence), whose solution is
    s_N = (prod a) s_0 + sum_m (prod_{j>m} a_j) b_m."""
    rng = np.random.default_rng(14)
    c = _case(rng, B=1, N=7, Hk=1, Hv=1, dk=1, dv=1, unit_k=False)
    snap, o = _run(c)
    al, be = c["alpha"][0, :, 0], c["beta"][0, :, 0]
    kk, vv, qq = c["k"][0, :, 0, 0], c["v"][0, :, 0, 0], c["q"][0, :, 0, 0]
    a = al * (1 - be * kk * kk)
    bterm = be * vv * kk
    s0 = c["cache"][c["slot"][0], 0, 0, 0]
    for n in range(c["N"]):
        s = np.prod(a[: n + 1]) * s0 + sum(np.prod(a[m + 1: n + 1]) * bterm[m] for m in range(n + 1))
        _close(snap[0, n, 0, 0, 0], s, 1e-13, f"scalar s_{n}")
        _close(o[0, n, 0, 0], s * qq[n], 1e-13, f"scalar o_{n}")


def check_linearity():
    """For fixed k, q, alpha, beta the map (S_0, V) -> (S_n, o) is linear."""
    rng = np.random.default_rng(15)
    c = _case(rng, tree=True)
    s_full, o_full = _run(c)
    s_h0, o_h0 = _run(c, v=np.zeros_like(c["v"]))
    s_v, o_v = _run(c, cache=np.zeros_like(c["cache"]))
    _close(s_full, s_h0 + s_v, 1e-13, "superposition (state)")
    _close(o_full, o_h0 + o_v, 1e-13, "superposition (o)")
    s_c, o_c = _run(c, cache=2.5 * c["cache"], v=2.5 * c["v"])
    _close(s_c, 2.5 * s_full, 1e-13, "homogeneity (state)")
    _close(o_c, 2.5 * o_full, 1e-13, "homogeneity (o)")


def check_column_independence():
    """Permuting the d_v columns of S_0 and of v permutes every output the same way."""
    rng = np.random.default_rng(16)
    c = _case(rng, dv=6, tree=True)
    perm = rng.permutation(c["dv"])
    s1, o1 = _run(c)
    s2, o2 = _run(c, cache=c["cache"][..., perm], v=c["v"][..., perm])
    _close(s2, s1[..., perm], 1e-14, "column permutation (state)")
    _close(o2, o1[..., perm], 1e-14, "column permutation (o)")


def check_contraction():
    """v = 0, alpha <= 1, 0 <= beta <= 2, |k| = 1: |S_n|_F never grows; at
    alpha = 1, beta = 2 the step is a Householder reflection and keeps the norm."""
    rng = np.random.default_rng(17)
    for alpha, beta, equal in ((None, None, False), (1.0, 2.0, True)):
        c = _case(rng, tree=True, alpha=alpha, beta=beta)
        if alpha is None:
            c["beta"] = rng.uniform(0.0, 2.0, c["beta"].shape)
        snap, _ = _run(c, v=np.zeros_like(c["v"]))
        for b in range(c["B"]):
            for n in range(c["N"]):
                for h in range(c["Hv"]):
                    before = np.linalg.norm(_src_state(c, snap, b, n, h))
                    after = np.linalg.norm(snap[b, n, h])
                    assert after <= before * (1 + 1e-13), "norm grew"
                    if equal:
                        assert abs(after - before) <= 1e-12 * before, "reflection changed norm"


def check_tree_matches_chain_and_paths():
    """A single-path tree is the chain, bit for bit; every tree node equals the
    chain run over its root-to-node ancestor path; a star tree starts every
    non-root node from node 0's state."""
    rng = np.random.default_rng(18)
    c = _case(rng, N=7)
    chain_s, chain_o = _run(c, parent=None)
    line = np.tile(np.arange(-1, c["N"] - 1, dtype=np.int32), (c["B"], 1))
    tree_s, tree_o = _run(c, parent=line)
    assert np.array_equal(chain_s, tree_s) and np.array_equal(chain_o, tree_o)

    c = _case(rng, N=8, tree=True)
    ts, to = _run(c)
    for b in range(c["B"]):
        for n in range(c["N"]):
            path = []
            m = n
            while m >= 0:
                path.append(m)
                m = c["parent"][b, m]
            path = path[::-1]
            sub = {key: c[key][b:b + 1, path] for key in ("q", "k", "v", "alpha", "beta")}
            st, ss, so = oracle.verify(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"],
                                       c["cache"], c["slot"][b:b + 1], None, B=1, N=len(path),
                                       Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"], dv=c["dv"])
            assert st == oracle.OK
            assert np.array_equal(ss[0, -1], ts[b, n]), f"tree node {n} != its ancestor chain"
            assert np.array_equal(so[0, -1], to[b, n])

    c = _case(rng, N=6, tree=True)
    c["parent"][:, 1:] = 0
    ss, so = _run(c)
    for b in range(c["B"]):
        for i in range(2, c["N"]):
            sub = {key: c[key][b:b + 1, [0, i]] for key in ("q", "k", "v", "alpha", "beta")}
            st, s2, o2 = oracle.verify(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"],
                                       c["cache"], c["slot"][b:b + 1], None, B=1, N=2,
                                       Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"], dv=c["dv"])
            assert np.array_equal(s2[0, 1], ss[b, i]) and np.array_equal(o2[0, 1], so[b, i])


def _fraction_verify(c, b):
    """Exact rational arithmetic, the recurrence in its literal matrix form
    S_n = alpha S_src (I - beta k k^T) + beta v k^T, o_n = S_n q_n, S = H^T.
    Value head h reads q/k head h // (Hv/Hk).  Returns per-node S and o."""
    F = Fraction
    dk, dv, G = c["dk"], c["dv"], c["Hv"] // c["Hk"]
    out_S, out_o = {}, {}
    for h in range(c["Hv"]):
        H0 = c["cache"][c["slot"][b], h]
        S0 = [[F(float(H0[i][j])) for i in range(dk)] for j in range(dv)]
        states = []
        for n in range(c["N"]):
            p = (n - 1) if c["parent"] is None else int(c["parent"][b, n])
            S = S0 if p < 0 else states[p]
            k = [F(float(x)) for x in c["k"][b, n, h // G]]
            q = [F(float(x)) for x in c["q"][b, n, h // G]]
            v = [F(float(x)) for x in c["v"][b, n, h]]
            a, be = F(float(c["alpha"][b, n, h])), F(float(c["beta"][b, n, h]))
            P = [[(F(1) if i == m else F(0)) - be * k[i] * k[m] for m in range(dk)]
                 for i in range(dk)]
            SP = [[sum(S[j][i] * P[i][m] for i in range(dk)) for m in range(dk)]
                  for j in range(dv)]
            Sn = [[a * SP[j][m] + be * v[j] * k[m] for m in range(dk)] for j in range(dv)]
            states.append(Sn)
            out_S[(n, h)] = Sn
            out_o[(n, h)] = [sum(Sn[j][m] * q[m] for m in range(dk)) for j in range(dv)]
    return out_S, out_o


def check_exact_rational_bruteforce():
    """Tiny cases in exact rationals vs the float64 and long-double oracle."""
    rng = np.random.default_rng(19)
    for dk, dv, tree in ((2, 2, False), (3, 2, True), (2, 3, True)):
        c = _case(rng, B=2, N=4, Hk=2, Hv=4, dk=dk, dv=dv, tree=tree, n_slots=3)
        snap, o = _run(c)
        snap_ld, o_ld = _run(c, precision="ld")
        for b in range(c["B"]):
            S_ex, o_ex = _fraction_verify(c, b)
            for (n, h), S in S_ex.items():
                H = np.array([[float(S[j][i]) for j in range(dv)] for i in range(dk)])
                _close(snap[b, n, h], H, 1e-13, f"exact state b{b} n{n} h{h}")
                _close(o[b, n, h], np.array([float(x) for x in o_ex[(n, h)]]), 1e-13,
                       f"exact o b{b} n{n} h{h}")
        _close(snap_ld, snap, 1e-14, "long double vs double")
        _close(o_ld, o, 1e-14, "long double vs double (o)")


def check_tree_depth_and_validation():
    rng = np.random.default_rng(20)
    N = 12
    parent = np.full((3, N), -1, np.int32)
    for b in range(3):
        for i in range(1, N):
            parent[b, i] = rng.integers(0, i)
    st, depth = oracle.tree_depth(parent)
    assert st == oracle.OK
    for b in range(3):
        for i in range(N):
            d, m = 0, i
            while m >= 0:
                d, m = d + 1, parent[b, m]
            assert depth[b, i] == d
    for bad in ([0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]):
        st, _ = oracle.tree_depth(np.array([bad], np.int32))
        assert st == oracle.ERR_BAD_TREE, bad
    # a bad tree skips its sequence and reports the error; the good one still runs
    c = _case(rng, B=2, N=4, tree=True)
    c["parent"][1] = [-1, 0, 2, 1]
    st, snap, o = oracle.verify(c["q"], c["k"], c["v"], c["alpha"], c["beta"], c["cache"],
                                c["slot"], c["parent"], B=2, N=4, Hk=c["Hk"], Hv=c["Hv"],
                                dk=c["dk"], dv=c["dv"])
    assert st == oracle.ERR_BAD_TREE
    assert not np.any(snap[1]) and np.any(snap[0])
    # the depth cap: a path of 6 nodes has depth 6 and a star depth 2 (counted
    # by hand, root = 1); a cap at the depth keeps the tree, one below rejects it
    path = np.array([[-1, 0, 1, 2, 3, 4]], np.int32)
    star = np.array([[-1, 0, 0, 0, 0, 0]], np.int32)
    for tree, deepest in ((path, 6), (star, 2)):
        st, depth = oracle.tree_depth(tree, max_depth=deepest)
        assert st == oracle.OK and int(depth.max()) == deepest
        st, _ = oracle.tree_depth(tree, max_depth=deepest - 1)
        assert st == oracle.ERR_BAD_TREE
    c = _case(rng, B=2, N=6, tree=True)
    c["parent"][0], c["parent"][1] = path[0], star[0]
    common = dict(B=2, N=6, Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"], dv=c["dv"])
    args = (c["q"], c["k"], c["v"], c["alpha"], c["beta"], c["cache"], c["slot"], c["parent"])
    st, snap_free, o_free = oracle.verify(*args, **common)
    assert st == oracle.OK
    st, snap_cap, o_cap = oracle.verify(*args, max_depth=6, **common)
    assert st == oracle.OK and np.array_equal(snap_cap, snap_free) and np.array_equal(o_cap, o_free)
    st, snap_cap, o_cap = oracle.verify(*args, max_depth=5, **common)
    assert st == oracle.ERR_BAD_TREE
    assert not np.any(snap_cap[0]) and np.array_equal(snap_cap[1], snap_free[1])


def check_commit():
    """Commit copies snap[layer][b][accept[b]] into cache[layer][slot[b]] and
    nothing else; bad accept / slot values are reported and skipped."""
    rng = np.random.default_rng(21)
    L, B, N, Hv, dk, dv, n_slots = 3, 2, 5, 2, 3, 4, 4
    snap = rng.standard_normal((L, B, N, Hv, dk, dv))
    cache = rng.standard_normal((L, n_slots, Hv, dk, dv))
    before = cache.copy()
    acc = np.array([4, 1], np.int32)
    slot = np.array([3, 0], np.int32)
    st = oracle.commit(snap, acc, cache, slot, B=B, N=N, Hv=Hv, dk=dk, dv=dv, n_layers=L,
                       snap_layer_stride=B * N * Hv * dk * dv,
                       cache_layer_stride=n_slots * Hv * dk * dv, n_slots=n_slots)
    assert st == oracle.OK
    for l in range(L):
        for s in range(n_slots):
            if s in slot:
                b = int(np.nonzero(slot == s)[0][0])
                assert np.array_equal(cache[l, s], snap[l, b, acc[b]])
            else:
                assert np.array_equal(cache[l, s], before[l, s])
    for bad_acc, bad_slot, err in (([5, 1], [3, 0], oracle.ERR_ACCEPT_RANGE),
                                   ([-1, 1], [3, 0], oracle.ERR_ACCEPT_RANGE),
                                   ([0, 1], [4, 0], oracle.ERR_SLOT_RANGE)):
        cache2 = before.copy()
        st = oracle.commit(snap, np.array(bad_acc, np.int32), cache2,
                           np.array(bad_slot, np.int32), B=B, N=N, Hv=Hv, dk=dk, dv=dv,
                           n_layers=L, snap_layer_stride=B * N * Hv * dk * dv,
                           cache_layer_stride=n_slots * Hv * dk * dv, n_slots=n_slots)
        assert st == err
        # the good sequence (b = 1) is still committed
        assert np.array_equal(cache2[0, 0], snap[0, 1, 1])


def chunked_reference(q, k, v, alpha, beta, state, chunk):
    """Chunked (WY / UT-transform) evaluation of the same recurrence, float64,
    one value head: q, k [T][dk], v [T][dv], alpha, beta [T], state H [dk][dv].

    Inside a chunk with cumulative decay g_t = prod_{s<=t} alpha_s and
    delta_t = beta_t (v_t - alpha_t H_{t-1}^T k_t), the rows of Delta solve
    (I + A) Delta = diag(beta) (V - diag(g) K H) with
    A[t][s] = beta_t (g_t / g_s) (k_t . k_s) for s < t; then
    O = diag(g) Q H + (causal(g_t / g_s) * Q K^T) Delta and
    H <- g_C H + K^T diag(g_C / g) Delta."""
    T = q.shape[0]
    H = state.copy()
    O = np.zeros((T, v.shape[1]))
    for t0 in range(0, T, chunk):
        sl = slice(t0, min(T, t0 + chunk))
        Q, K, V, a, b = q[sl], k[sl], v[sl], alpha[sl], beta[sl]
        C = Q.shape[0]
        g = np.cumprod(a)
        ratio = g[:, None] / g[None, :]
        A = np.tril(b[:, None] * ratio * (K @ K.T), -1)
        X = b[:, None] * (V - g[:, None] * (K @ H))
        Delta = np.linalg.solve(np.eye(C) + A, X)
        O[sl] = g[:, None] * (Q @ H) + (np.tril(ratio) * (Q @ K.T)) @ Delta
        H = g[-1] * H + K.T @ ((g[-1] / g)[:, None] * Delta)
    return H, O


def check_chunked_equals_step():
    """The chunked form (C = 1, 4, 64) reaches the step recurrence's result."""
    rng = np.random.default_rng(22)
    Hk, Hv, dk, dv = 1, 2, 8, 6
    for T in (1, 63, 64, 65, 200):
        q = rng.standard_normal((T, Hk, dk))
        k = rng.standard_normal((T, Hk, dk))
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        v = rng.standard_normal((T, Hv, dv))
        al = rng.uniform(0.85, 1.0, (T, Hv))
        be = rng.uniform(0.0, 1.0, (T, Hv))
        s0 = rng.standard_normal((Hv, dk, dv)) * 0.1
        st, sT, o = oracle.prefill_step(q, k, v, al, be, s0, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        for C in (1, 4, 64):
            for h in range(Hv):
                Hc, Oc = chunked_reference(q[:, 0], k[:, 0], v[:, h], al[:, h], be[:, h], s0[h], C)
                _close(Hc, sT[h], 1e-10, f"chunked state T={T} C={C}")
                _close(Oc, o[:, h], 1e-10, f"chunked o T={T} C={C}")


def check_rounds_equal_sequential():
    """verify -> commit(accepted) -> verify the next block from the cache, for
    several rounds, equals one token-by-token run over the accepted tokens
    (speculation is lossless; the replayed prefix equals the persisted state)."""
    rng = np.random.default_rng(23)
    Hk, Hv, dk, dv, N = 2, 4, 4, 3, 5
    cache = rng.standard_normal((2, Hv, dk, dv)) * 0.3
    slot = np.array([1], np.int32)
    start = cache[1].copy()
    acc_q, acc_k, acc_v, acc_a, acc_b = [], [], [], [], []
    for _ in range(4):
        c = _case(rng, B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        st, snap, o = oracle.verify(c["q"], c["k"], c["v"], c["alpha"], c["beta"], cache, slot,
                                    None, B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        L = int(rng.integers(1, N + 1))
        st = oracle.commit(snap, np.array([L - 1], np.int32), cache, slot, B=1, N=N, Hv=Hv,
                           dk=dk, dv=dv, n_slots=2)
        assert st == oracle.OK
        for lst, key in ((acc_q, "q"), (acc_k, "k"), (acc_v, "v"), (acc_a, "alpha"),
                         (acc_b, "beta")):
            lst.append(c[key][0, :L])
    cat = [np.concatenate(x) for x in (acc_q, acc_k, acc_v, acc_a, acc_b)]
    T = cat[0].shape[0]
    st, sT, _ = oracle.prefill_step(*cat, start, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    assert st == oracle.OK
    _close(cache[1], sT, 1e-13, "rounds of verify+commit vs sequential")


def check_replay_equals_persist():
    """Checkpoint-and-replay commit: re-running each sequence's accepted path
    (a chain prefix, or a tree node's ancestors from the root) from the cached
    state gives the state the verify block persisted for that node; rounds of
    verify -> replay commit equal one token-by-token run over the accepted
    tokens; a bad accept index, slot or parent array leaves the cache alone."""
    rng = np.random.default_rng(31)
    for tree in (False, True):
        c = _case(rng, B=3, N=6, Hk=2, Hv=4, dk=4, dv=3, tree=tree, n_slots=4)
        snap, _ = _run(c)
        acc = rng.integers(0, c["N"], c["B"]).astype(np.int32)
        cache = np.ascontiguousarray(c["cache"], dtype=np.float64).copy()
        st = oracle.replay(c["k"], c["v"], c["alpha"], c["beta"], cache, c["slot"], c["parent"],
                           acc, B=c["B"], N=c["N"], Hk=c["Hk"], Hv=c["Hv"], dk=c["dk"],
                           dv=c["dv"])
        assert st == oracle.OK, st
        for b in range(c["B"]):
            _close(cache[c["slot"][b]], snap[b, acc[b]], 1e-13,
                   f"replay of node {acc[b]} ({'tree' if tree else 'chain'}) vs persisted")
        untouched = sorted(set(range(4)) - set(int(x) for x in c["slot"]))
        for s_ in untouched:
            _close(cache[s_], c["cache"][s_], 0.0, "slot not in the batch is untouched")
    # rounds with the replay commit
    Hk, Hv, dk, dv, N = 2, 4, 4, 3, 5
    cache = rng.standard_normal((2, Hv, dk, dv)) * 0.3
    slot = np.array([1], np.int32)
    start = cache[1].copy()
    acc_l = {key: [] for key in ("q", "k", "v", "alpha", "beta")}
    for _ in range(4):
        c = _case(rng, B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        L = int(rng.integers(1, N + 1))
        st = oracle.replay(c["k"], c["v"], c["alpha"], c["beta"], cache, slot, None,
                           np.array([L - 1], np.int32), B=1, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        for key in acc_l:
            acc_l[key].append(c[key][0, :L])
    cat = [np.concatenate(acc_l[key]) for key in ("q", "k", "v", "alpha", "beta")]
    st, sT, _ = oracle.prefill_step(*cat, start, T=cat[0].shape[0], Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    assert st == oracle.OK
    _close(cache[1], sT, 1e-13, "rounds of verify+replay vs sequential")
    # errors: the offending sequence is skipped, the other one still commits
    c = _case(rng, B=2, N=4, Hk=1, Hv=2, dk=2, dv=2, tree=True)
    cases = (  # (accept, slot, parent, status, bad sequence)
        (np.array([4, 1], np.int32), c["slot"], c["parent"], oracle.ERR_ACCEPT_RANGE, 0),
        (np.array([2, 3], np.int32), np.array([0, 5], np.int32), c["parent"],
         oracle.ERR_SLOT_RANGE, 1),
        (np.array([2, 3], np.int32), c["slot"], None, oracle.ERR_BAD_TREE, 1),
    )
    for acc, slot, par, code, bad_b in cases:
        if par is None:
            par = c["parent"].copy()
            par[1, 2] = 3
        cache = np.ascontiguousarray(c["cache"], dtype=np.float64).copy()
        st = oracle.replay(c["k"], c["v"], c["alpha"], c["beta"], cache, slot, par, acc, B=2,
                           N=4, Hk=1, Hv=2, dk=2, dv=2, n_slots=2)
        assert st == code, (st, code)
        good_b = 1 - bad_b
        _, snap, _ = oracle.verify(c["q"], c["k"], c["v"], c["alpha"], c["beta"], c["cache"],
                                   slot, c["parent"], B=2, N=4, Hk=1, Hv=2, dk=2, dv=2,
                                   n_slots=2)
        _close(cache[int(slot[good_b])], snap[good_b, acc[good_b]], 1e-13,
               "the valid sequence still commits")
        if 0 <= int(slot[bad_b]) < 2:
            _close(cache[int(slot[bad_b])], c["cache"][int(slot[bad_b])], 0.0,
                   "a skipped sequence keeps its cached state")


def check_index_commit_equals_copy():
    """Index-table commit: a block that starts from the previous block's
    snapshot region through the slot table computes exactly what it computes
    after the accepted states were copied into the cache; a bad accept index
    leaves its slot alone."""
    rng = np.random.default_rng(37)
    B, N, Hk, Hv, dk, dv = 3, 5, 2, 4, 4, 3
    for tree in (False, True):
        c1 = _case(rng, B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, tree=tree)
        snap1, _ = _run(c1)
        acc = rng.integers(0, N, B).astype(np.int32)
        # (a) copy commit into the cache, then block 2 from the cache
        cache = np.ascontiguousarray(c1["cache"], dtype=np.float64).copy()
        assert oracle.commit(snap1, acc, cache, c1["slot"], B=B, N=N, Hv=Hv, dk=dk,
                             dv=dv) == oracle.OK
        c2 = _case(rng, B=B, N=N, Hk=Hk, Hv=Hv, dk=dk, dv=dv, tree=tree)
        st, snap_a, o_a = oracle.verify(c2["q"], c2["k"], c2["v"], c2["alpha"], c2["beta"],
                                        cache, c1["slot"], c2["parent"], B=B, N=N, Hk=Hk,
                                        Hv=Hv, dk=dk, dv=dv)
        assert st == oracle.OK
        # (b) index commit, then block 2 from block 1's snapshot region
        base = 7
        slot = np.full(B, -1, np.int32)
        assert oracle.commit_index(acc, slot, N=N, base=base) == oracle.OK
        assert [int(x) for x in slot] == [base + b * N + int(acc[b]) for b in range(B)]
        region = np.zeros((base + B * N, Hv, dk, dv))
        region[base:] = snap1.reshape(B * N, Hv, dk, dv)
        st, snap_b, o_b = oracle.verify(c2["q"], c2["k"], c2["v"], c2["alpha"], c2["beta"],
                                        region, slot, c2["parent"], B=B, N=N, Hk=Hk, Hv=Hv,
                                        dk=dk, dv=dv)
        assert st == oracle.OK
        assert np.array_equal(snap_a, snap_b) and np.array_equal(o_a, o_b), \
            "index-table commit differs from copy commit"
    slot = np.array([3, 4], np.int32)
    assert oracle.commit_index(np.array([1, 5], np.int32), slot, N=5) == oracle.ERR_ACCEPT_RANGE
    assert [int(x) for x in slot] == [1, 4], "a bad accept index must leave its slot alone"


def check_conv_history_commit():
    """Convolution history: after rounds of chain blocks each committed at
    its accepted boundary, every channel holds the last W inputs of the whole
    accepted token stream (the first history included); a tree commit equals
    the chain commit over the accepted node's ancestor path; a short path
    keeps the newest part of the old history; bad sequences are skipped."""
    rng = np.random.default_rng(41)
    C, W, N = 5, 4, 6
    hist0 = rng.standard_normal((2, C, W))
    state = hist0.copy()
    slot = np.array([1], np.int32)
    stream = [hist0[1].T]                          # [W][C], oldest first
    for _ in range(5):
        x = rng.standard_normal((1, N, C))
        L = int(rng.integers(1, N + 1))
        assert oracle.conv_commit(x, state, slot, None, np.array([L - 1], np.int32)) == oracle.OK
        stream.append(x[0, :L])
    tokens = np.concatenate(stream)                # [T][C]
    assert np.array_equal(state[1], tokens[-W:].T), "history is not the last W inputs"
    assert np.array_equal(state[0], hist0[0]), "another slot changed"
    # tree == chain over the ancestor path
    par = np.array([[-1, 0, 0, 1, 3, 2, 4]], np.int32)
    x = rng.standard_normal((1, 7, C))
    for acc in range(7):
        t_state = hist0.copy()
        assert oracle.conv_commit(x, t_state, slot, par, np.array([acc], np.int32)) == oracle.OK
        path = []
        m = acc
        while m >= 0:
            path.insert(0, m)
            m = par[0, m]
        c_state = hist0.copy()
        xc = x[:, path]
        assert oracle.conv_commit(xc, c_state, slot, None,
                                  np.array([len(path) - 1], np.int32)) == oracle.OK
        assert np.array_equal(t_state, c_state), f"tree node {acc} != chain over its path"
    # a path shorter than W keeps the newest W - L old entries
    s2 = hist0.copy()
    assert oracle.conv_commit(x, s2, slot, None, np.array([1], np.int32)) == oracle.OK
    assert np.array_equal(s2[1][:, :W - 2], hist0[1][:, 2:])
    assert np.array_equal(s2[1][:, W - 2:], x[0, :2].T)
    # errors
    s3 = hist0.copy()
    xb = rng.standard_normal((2, N, C))
    st = oracle.conv_commit(xb, s3, np.array([0, 1], np.int32), None,
                            np.array([2, N], np.int32))
    assert st == oracle.ERR_ACCEPT_RANGE
    assert np.array_equal(s3[1], hist0[1]), "a skipped sequence keeps its history"
    assert np.array_equal(s3[0][:, W - 3:], xb[0, :3].T)


def check_input_preparation():
    """Raw projections -> inputs: unit-norm q and k in the same direction (a
    zero vector stays zero); alpha = exp(-softplus(a)) equals 1/(1+e^a) (the
    closed form of the composition) and lies in (0, 1), falling with a;
    beta = sigmoid(b) with beta(b) + beta(-b) = 1 and beta(0) = 1/2."""
    rng = np.random.default_rng(43)
    q = rng.standard_normal((3, 5, 2, 8)) * 3.0
    k = rng.standard_normal((3, 5, 2, 8)) * 0.1
    k[1, 2, 0] = 0.0
    a = rng.standard_normal((3, 5, 4)) * 4.0
    b = rng.standard_normal((3, 5, 4)) * 4.0
    qn, kn, al, be = oracle.prepare_inputs(q, k, a, b)
    for x, xn in ((q, qn), (k, kn)):
        norms = np.linalg.norm(xn, axis=-1)
        zero = np.linalg.norm(x, axis=-1) == 0
        _close(norms[~zero], np.ones(int((~zero).sum())), 1e-14, "unit norm")
        assert np.all(xn[zero] == 0), "a zero vector must stay zero"
        cos = np.sum(xn * x, axis=-1)[~zero] / np.linalg.norm(x, axis=-1)[~zero]
        _close(cos, np.ones_like(cos), 1e-14, "same direction")
    _close(al, 1.0 / (1.0 + np.exp(a)), 1e-14, "alpha closed form")
    assert np.all((al > 0) & (al < 1))
    order = np.argsort(a.ravel())
    assert np.all(np.diff(al.ravel()[order]) <= 0), "alpha must fall as a rises"
    _, _, _, be_neg = oracle.prepare_inputs(q, k, a, -b)
    _close(be + be_neg, np.ones_like(be), 1e-14, "sigmoid symmetry")
    _, _, _, half = oracle.prepare_inputs(q, k, a, np.zeros_like(b))
    _close(half, np.full_like(half, 0.5), 0.0, "sigmoid(0)")


def block_form_reference(H0, K, V, Q, alpha, beta, parent):
    """The whole block at once (float64, one value head): with G(n) the sum of
    log alpha over the root-to-n path and the deltas solved first from
        delta_n = beta_n v_n - beta_n e^G(n) H0^T k_n
                  - sum_{m strict ancestor of n} beta_n e^(G(n)-G(m)) (k_m . k_n) delta_m,
    every state is H_n = e^G(n) H0 + sum_{m on the path} e^(G(n)-G(m)) k_m delta_m^T."""
    N = K.shape[0]
    G = np.zeros(N)
    anc = [[] for _ in range(N)]
    for n in range(N):
        p = parent[n]
        G[n] = np.log(alpha[n]) + (G[p] if p >= 0 else 0.0)
        anc[n] = (anc[p] + [p]) if p >= 0 else []
    X = K @ H0
    KK = K @ K.T
    D = np.zeros((N, V.shape[1]))
    for n in range(N):
        D[n] = beta[n] * V[n] - beta[n] * np.exp(G[n]) * X[n]
        for m in anc[n]:
            D[n] -= beta[n] * np.exp(G[n] - G[m]) * KK[n, m] * D[m]
    S = np.array([np.exp(G[n]) * H0 + sum(np.exp(G[n] - G[m]) * np.outer(K[m], D[m])
                                          for m in anc[n] + [n]) for n in range(N)])
    return S, np.einsum("nij,ni->nj", S, Q)


def check_block_form_equals_recurrence():
    """All deltas first, then every state from the cached one: the same states
    and outputs as the node-by-node recurrence, for chains and trees."""
    rng = np.random.default_rng(24)
    for tree in (False, True):
        N, dk, dv = 12, 8, 6
        parent = np.array([-1] + [int(rng.integers(0, i)) if tree else i - 1
                                  for i in range(1, N)], np.int32)
        K = rng.standard_normal((N, dk))
        K /= np.linalg.norm(K, axis=1, keepdims=True)
        Q, V = rng.standard_normal((N, dk)), rng.standard_normal((N, dv))
        al, be = rng.uniform(0.5, 1.0, N), rng.uniform(0.0, 1.0, N)
        H0 = rng.standard_normal((dk, dv))
        S, O = block_form_reference(H0, K, V, Q, al, be, parent)
        st, snap, o = oracle.verify(Q[None, :, None], K[None, :, None], V[None, :, None],
                                    al[None, :, None], be[None, :, None], H0[None, None],
                                    np.zeros(1, np.int32), parent[None] if tree else None, B=1,
                                    N=N, Hk=1, Hv=1, dk=dk, dv=dv)
        assert st == oracle.OK
        _close(S, snap[0, :, 0], 1e-12, "block form states")
        _close(O, o[0, :, 0], 1e-12, "block form outputs")


ALL_CHECKS = [
    check_golden_hand_example, check_identity_gate, check_delta_rule_closed_form,
    check_zero_decay, check_scalar_closed_form, check_linearity, check_column_independence,
    check_contraction, check_tree_matches_chain_and_paths, check_exact_rational_bruteforce,
    check_tree_depth_and_validation, check_commit, check_chunked_equals_step,
    check_rounds_equal_sequential, check_block_form_equals_recurrence,
    check_replay_equals_persist, check_index_commit_equals_copy, check_conv_history_commit,
    check_input_preparation,
]
