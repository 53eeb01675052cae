"""CPU-only checks of the C ABI: the library builds and loads, exports every
function include/gdn.h declares, the struct layout matches, and host-side
argument checks reject bad calls before anything is launched (these calls
never reach the GPU)."""
import ctypes
import os
import re

import pytest

import hybrid_gated_deltanet_delta_gb300 as gdn
from hybrid_gated_deltanet_delta_gb300 import build as gdn_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gdn_build.build()
    return gdn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gdn_verify_chain", "gdn_verify_tree", "gdn_commit_accepted",
                 "gdn_commit_index", "gdn_conv_commit", "gdn_replay_accepted", "gdn_prefill_chunked", "gdn_prefill_workspace_bytes",
                 "gdn_status_string", "gdn_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared in gdn.h but not exported"


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include "gdn.h"\n#include <stdio.h>\n#include <stddef.h>\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(gdn_verify_args),'
                   ' offsetof(gdn_verify_args, cache_slot_stride),'
                   ' offsetof(gdn_verify_args, n_slots), offsetof(gdn_verify_args, row_warps),'
                   ' offsetof(gdn_verify_args, max_depth));'
                   'return 0;}\n')
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)])
    size, off_stride, off_slots, off_rw, off_md = map(
        int, subprocess.check_output([str(exe)]).split())
    A = gdn.VerifyArgs
    assert ctypes.sizeof(A) == size
    assert A.cache_slot_stride.offset == off_stride
    assert A.n_slots.offset == off_slots and A.row_warps.offset == off_rw
    assert A.max_depth.offset == off_md


def test_version_and_status_strings(lib):
    assert lib.gdn_version() == 3
    assert gdn.status_string(gdn.GDN_ERR_BAD_TREE) == "GDN_ERR_BAD_TREE"
    assert gdn.status_string(gdn.GDN_ERR_TIMEOUT) == "GDN_ERR_TIMEOUT"
    assert gdn.status_string(12345) == "GDN_ERR_UNKNOWN"


def _args(**kw):
    a = gdn.VerifyArgs()
    base = dict(q=0x10000, k=0x20000, v=0x30000, alpha=0x40000, beta=0x50000,
                state_cache=0x60000, snapshots=0x70000, o=0x80000, cache_slot_stride=48 * 128 * 128,
                n_slots=1, B=1, N=16, Hk=16, Hv=48, dk=128, dv=128, in_dtype=gdn.GDN_BF16)
    base.update(kw)
    for key, val in base.items():
        setattr(a, key, val)
    return a


@pytest.mark.parametrize("change, want", [
    (dict(N=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(Hv=47), gdn.GDN_ERR_INVALID_ARG),
    (dict(in_dtype=7), gdn.GDN_ERR_INVALID_ARG),
    (dict(N=65), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dv=40), gdn.GDN_ERR_UNSUPPORTED),
    (dict(q=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(alpha=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(v=0x30008), gdn.GDN_ERR_MISALIGNED),
    (dict(o=0x80004), gdn.GDN_ERR_MISALIGNED),
    (dict(alpha=0x40002), gdn.GDN_ERR_MISALIGNED),
    (dict(n_slots=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(cache_slot_stride=100), gdn.GDN_ERR_INVALID_ARG),
    (dict(cache_slot_stride=48 * 128 * 128 + 2), gdn.GDN_ERR_MISALIGNED),
    (dict(tile_cols=24), gdn.GDN_ERR_UNSUPPORTED),
    (dict(tile_cols=32, row_warps=1), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dk=64, row_warps=4), gdn.GDN_ERR_UNSUPPORTED),
    (dict(dk=32, row_warps=2), gdn.GDN_ERR_UNSUPPORTED),
    (dict(tile_cols=8, row_warps=2), gdn.GDN_ERR_UNSUPPORTED),
    (dict(B=0), gdn.GDN_OK),
])
def test_verify_host_checks(lib, change, want):
    a = _args(**change)
    assert lib.gdn_verify_chain(ctypes.byref(a), None) == want
    assert lib.gdn_verify_tree(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None) == want


def test_verify_tree_rejects_negative_depth_cap(lib):
    """max_depth = 0 means no cap; a negative cap is an argument error (tree
    call only: a chain ignores the field, so its call would launch)."""
    a = _args(max_depth=-1)
    assert lib.gdn_verify_tree(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None) == \
        gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_tree_prep(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None) == \
        gdn.GDN_ERR_INVALID_ARG


def test_verify_tree_needs_parent(lib):
    assert lib.gdn_verify_tree(ctypes.byref(_args()), None, None, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_chain(None, None) == gdn.GDN_ERR_INVALID_ARG


def test_verify_without_snapshots_checks_q(lib):
    """Chains and trees may skip persistence (commit by replay); the other
    arguments are still checked (calls that fail before any launch)."""
    a = _args(snapshots=0, q=0)
    assert lib.gdn_verify_chain(ctypes.byref(a), None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_tree(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None) == \
        gdn.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("change, acc, want", [
    (dict(N=0), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(B=-1), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(Hv=47), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(N=65), 0xA0000, gdn.GDN_ERR_UNSUPPORTED),
    (dict(dk=96), 0xA0000, gdn.GDN_ERR_UNSUPPORTED),
    (dict(k=0), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(state_cache=0), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(beta=0), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(), 0, gdn.GDN_ERR_INVALID_ARG),
    (dict(), 0xA0002, gdn.GDN_ERR_MISALIGNED),
    (dict(v=0x30008), 0xA0000, gdn.GDN_ERR_MISALIGNED),
    (dict(n_slots=0), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(cache_slot_stride=100), 0xA0000, gdn.GDN_ERR_INVALID_ARG),
    (dict(tile_cols=24), 0xA0000, gdn.GDN_ERR_UNSUPPORTED),
    (dict(B=0), 0xA0000, gdn.GDN_OK),
])
def test_replay_host_checks(lib, change, acc, want):
    """gdn_replay_accepted needs no q, snapshots or o; everything else is
    checked as for verify (these calls never launch)."""
    a = _args(q=0, snapshots=0, o=0, **change)
    assert lib.gdn_replay_accepted(ctypes.byref(a), None, ctypes.c_void_p(acc), None) == want
    assert lib.gdn_replay_accepted(ctypes.byref(a), ctypes.c_void_p(0x90000),
                                   ctypes.c_void_p(acc), None) == want


@pytest.mark.parametrize("args, want", [
    ((0xA0000, -1, 16, 0, 0xB0000, None), gdn.GDN_ERR_INVALID_ARG),
    ((0xA0000, 4, 0, 0, 0xB0000, None), gdn.GDN_ERR_INVALID_ARG),
    ((0xA0000, 4, 16, -2, 0xB0000, None), gdn.GDN_ERR_INVALID_ARG),
    ((0xA0000, 1 << 27, 64, 0, 0xB0000, None), gdn.GDN_ERR_UNSUPPORTED),
    ((None, 4, 16, 0, 0xB0000, None), gdn.GDN_ERR_INVALID_ARG),
    ((0xA0000, 4, 16, 0, None, None), gdn.GDN_ERR_INVALID_ARG),
    ((0xA0002, 4, 16, 0, 0xB0000, None), gdn.GDN_ERR_MISALIGNED),
    ((0xA0000, 4, 16, 0, 0xB0001, None), gdn.GDN_ERR_MISALIGNED),
    ((0xA0000, 0, 16, 0, None, None), gdn.GDN_OK),
])
def test_commit_index_host_checks(lib, args, want):
    acc, B, N, base, slot, status = args
    P = ctypes.c_void_p
    lib.gdn_commit_index.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P]
    assert lib.gdn_commit_index(acc, B, N, base, slot, status, None) == want


def test_f16_entry_points_host_checks(lib):
    """The binary16 variants check their own pointers (calls that never launch)."""
    a = _args()
    assert lib.gdn_verify_chain_f16(ctypes.byref(a), None, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_chain_f16(ctypes.byref(a), ctypes.c_void_p(0x70008), None) == \
        gdn.GDN_ERR_MISALIGNED
    a = _args(q=0)
    assert lib.gdn_verify_chain_f16(ctypes.byref(a), ctypes.c_void_p(0x70000), None) == \
        gdn.GDN_ERR_INVALID_ARG
    a = _args()
    assert lib.gdn_verify_tree_f16(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None,
                                   None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_tree_f16(ctypes.byref(a), ctypes.c_void_p(0x90000), None,
                                   ctypes.c_void_p(0x70008), None) == gdn.GDN_ERR_MISALIGNED
    assert lib.gdn_verify_tree_f16(ctypes.byref(a), None, None, ctypes.c_void_p(0x70000),
                                   None) == gdn.GDN_ERR_INVALID_ARG
    f = lib.gdn_commit_accepted_f16
    assert f(None, 0, 0x20000, 0x30000, 48 * 128 * 128, 0, None, 1, 1, 16, 48, 128, 128, 1,
             None, None) == gdn.GDN_ERR_INVALID_ARG
    assert f(0x10008, 0, 0x20000, 0x30000, 48 * 128 * 128, 0, None, 1, 1, 16, 48, 128, 128, 1,
             None, None) == gdn.GDN_ERR_MISALIGNED
    assert f(0x10000, 0, 0x20000, 0x30000, 48 * 128 * 128, 0, None, 1, 0, 16, 48, 128, 128, 1,
             None, None) == gdn.GDN_OK


@pytest.mark.parametrize("change, want", [
    (dict(dtype=5), gdn.GDN_ERR_INVALID_ARG),
    (dict(B=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(N=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(W=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(W=9), gdn.GDN_ERR_UNSUPPORTED),
    (dict(stride=10), gdn.GDN_ERR_INVALID_ARG),
    (dict(x=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(acc=None), gdn.GDN_ERR_INVALID_ARG),
    (dict(x=0x10001), gdn.GDN_ERR_MISALIGNED),
    (dict(dtype=0, state=0x30002), gdn.GDN_ERR_MISALIGNED),
    (dict(acc=0x20002), gdn.GDN_ERR_MISALIGNED),
    (dict(B=0), gdn.GDN_OK),
])
def test_conv_commit_host_checks(lib, change, want):
    b = dict(x=0x10000, dtype=gdn.GDN_BF16, state=0x30000, stride=10240 * 3, slot=None,
             n_slots=1, parent=None, acc=0x20000, B=1, N=16, C=10240, W=3, status=None)
    b.update(change)
    assert lib.gdn_conv_commit(b["x"], b["dtype"], b["state"], b["stride"], b["slot"],
                               b["n_slots"], b["parent"], b["acc"], b["B"], b["N"], b["C"],
                               b["W"], b["status"], None) == want


@pytest.mark.parametrize("change, want", [
    (dict(N=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(dk=96), gdn.GDN_ERR_UNSUPPORTED),
    (dict(q=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(v=0x30008), gdn.GDN_ERR_MISALIGNED),
    (dict(B=0), gdn.GDN_OK),
])
def test_prep_entry_points_host_checks(lib, change, want):
    """The raw-projection variants run the same checks (calls that never launch)."""
    a = _args(**change)
    assert lib.gdn_verify_chain_prep(ctypes.byref(a), None) == want
    assert lib.gdn_verify_tree_prep(ctypes.byref(a), ctypes.c_void_p(0x90000), None, None) == want
    r = _args(snapshots=0, o=0, **change)
    if "q" not in change:
        assert lib.gdn_replay_accepted_prep(ctypes.byref(r), None, ctypes.c_void_p(0xA0000),
                                            None) == want


def _commit(lib, **kw):
    base = dict(snap=0x10000, sls=0, acc=0x20000, cache=0x30000, css=48 * 128 * 128, cls=0,
                slot=None, n_slots=1, B=1, N=16, Hv=48, dk=128, dv=128, L=1, status=None)
    base.update(kw)
    b = base
    return lib.gdn_commit_accepted(b["snap"], b["sls"], b["acc"], b["cache"], b["css"], b["cls"],
                                   b["slot"], b["n_slots"], b["B"], b["N"], b["Hv"], b["dk"],
                                   b["dv"], b["L"], b["status"], None)


@pytest.mark.parametrize("change, want", [
    (dict(B=0), gdn.GDN_OK),
    (dict(L=0), gdn.GDN_OK),
    (dict(N=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(snap=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(acc=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(cache=0x30004), gdn.GDN_ERR_MISALIGNED),
    (dict(sls=6), gdn.GDN_ERR_MISALIGNED),
    (dict(css=5), gdn.GDN_ERR_INVALID_ARG),
    (dict(n_slots=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(dk=3, dv=3, Hv=1, css=16), gdn.GDN_ERR_MISALIGNED),
    (dict(cls=-4), gdn.GDN_ERR_INVALID_ARG),
])
def test_commit_host_checks(lib, change, want):
    assert _commit(lib, **change) == want


@pytest.mark.parametrize("noalloc", [False, True])
def test_prefill_host_checks(lib, noalloc):
    P = 0x100000
    ok = dict(q=P, k=P, v=P, dt=gdn.GDN_BF16, a=P, b=P, T=128, Hk=16, Hv=48, dk=128, dv=128,
              C=64, s=P, o=P, w=P, wb=1 << 40, st=None)

    def call(**kw):
        x = dict(ok)
        x.update(kw)
        head = (x["q"], x["k"], x["v"], x["dt"], x["a"], x["b"], x["T"], x["Hk"], x["Hv"],
                x["dk"], x["dv"], x["C"], x["s"], x["o"])
        if noalloc:
            return lib.gdn_prefill_chunked_noalloc(*head, x["st"], None)
        return lib.gdn_prefill_chunked(*head, x["w"], x["wb"], x["st"], None)

    assert call(T=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(Hv=47) == gdn.GDN_ERR_INVALID_ARG
    assert call(dt=5) == gdn.GDN_ERR_INVALID_ARG
    assert call(dt=gdn.GDN_F32) == gdn.GDN_ERR_UNSUPPORTED   # host-side, before any launch
    assert call(dk=64) == gdn.GDN_ERR_UNSUPPORTED
    assert call(C=32) == gdn.GDN_ERR_UNSUPPORTED
    assert call(s=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(o=P + 4) == gdn.GDN_ERR_MISALIGNED
    assert call(st=P + 2) == gdn.GDN_ERR_MISALIGNED
    assert call(q=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(a=P + 1) == gdn.GDN_ERR_MISALIGNED
    assert call(T=0) == gdn.GDN_OK
    if noalloc:
        # 11 chunks x 48 value heads of workspace do not fit the built-in scratch
        assert call(T=704) == gdn.GDN_ERR_SCRATCH_LIMIT
    else:
        need = lib.gdn_prefill_workspace_bytes(128, 16, 48, 128, 128, 64)
        if need > 0:
            assert call(w=0) == gdn.GDN_ERR_WORKSPACE
            assert call(wb=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert lib.gdn_prefill_workspace_bytes(-1, 16, 48, 128, 128, 64) == 0


def test_nvtx_ranges_switch_on_without_changing_results(tmp_path):
    """GDN_NVTX=1 wraps every entry point in an NVTX range; host-side checks
    return the same codes with the ranges on (run in a fresh process, since
    the switch is read once per process)."""
    import subprocess
    import sys

    code = ("import ctypes, hybrid_gated_deltanet_delta_gb300 as g; lib = g.load(); "
            "a = g.VerifyArgs(); "
            "assert lib.gdn_verify_chain(ctypes.byref(a), None) == g.GDN_ERR_INVALID_ARG; "
            "assert lib.gdn_verify_chain(None, None) == g.GDN_ERR_INVALID_ARG; "
            "assert lib.gdn_commit_index(None, 1, 4, 0, None, None, None) == "
            "g.GDN_ERR_INVALID_ARG; print('ok')")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for val in ("1", "0"):
        env = dict(os.environ, GDN_NVTX=val, PYTHONPATH=root)
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True,
                             text=True, cwd=root, timeout=120)
        assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        gdn.load(str(tmp_path / "missing.so"))
