"""Host-side accounting of bench.py, on the CPU: the algorithmic byte and flop
counts behind the roofline figures, written out term by term here from the
tensors each call moves, the clock summary's throttle detection, the traffic
lookup in profile summaries, and one line of the reference arm."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_verify_bytes_chain16_by_tensor():
    # 1 sequence, 16 nodes, 16 q/k heads, 48 value heads, d = 128, bf16 inputs
    state = 48 * 128 * 128 * 4
    snapshots = 16 * state
    q_and_k = 2 * 16 * 16 * 128 * 2
    v = 16 * 48 * 128 * 2
    gates = 2 * 16 * 48 * 4
    o = 16 * 48 * 128 * 4
    assert bench.verify_bytes(1, 16, 16, 48, 128, 128) == \
        state + snapshots + q_and_k + v + gates + o == 54_204_416


def test_verify_bytes_variants():
    base = bench.verify_bytes(1, 22, 16, 48, 128, 128, tree=True)
    assert base == 73_351_600   # parents in and depths out: 2 x 22 x 4 bytes on top
    assert base - bench.verify_bytes(1, 22, 16, 48, 128, 128) == 2 * 22 * 4
    no_snap = bench.verify_bytes(1, 16, 16, 48, 128, 128, persist=False)
    assert bench.verify_bytes(1, 16, 16, 48, 128, 128) - no_snap == 16 * 48 * 128 * 128 * 4
    f16 = bench.verify_bytes(1, 16, 16, 48, 128, 128, snap_bytes=2)
    assert bench.verify_bytes(1, 16, 16, 48, 128, 128) - f16 == 16 * 48 * 128 * 128 * 2
    assert bench.verify_bytes(8, 16, 16, 48, 128, 128) == 433_635_328
    assert bench.commit_bytes(8, 48, 128, 128, n_layers=48) == 2 * 8 * 48 * 128 * 128 * 4 * 48


def test_prefill_flops_by_product():
    T, Hk, Hv, d, C = 8192, 16, 48, 128, 64
    chunks = T // C
    per_qk_head = 2 * (C * C * d)                 # K K^T, Q K^T
    per_v_head = 3 * (C * d * d) + 2 * (C * C * d)  # K H, Q H, K^T D'; T X, P Delta
    want = 2 * chunks * (Hk * per_qk_head + Hv * per_v_head)
    assert bench.prefill_flops(T, Hk, Hv, d, d) == want
    assert abs(want - 55.83e9) < 0.01e9


def test_clock_summary_flags_throttling():
    s = bench.ClockSampler(None)
    s.samples = [(1.0, ["2070", "2070", "900", "Not Active", "Not Active", "Not Active",
                        "Active"]),
                 (2.0, ["1500", "2070", "950", "Active", "Not Active", "Not Active",
                        "Not Active"]),
                 (9.0, ["300", "2070", "100", "Active", "Active", "Active", "Active"])]
    out = s.summary(0.5, 2.5)
    assert out["sm_max_mhz"] == 2070.0
    assert "hw_slowdown" in out["reasons"] and "sw_power_cap" in out["reasons"]
    assert "hw_thermal_slowdown" not in out["reasons"]   # the 9.0 s sample is outside


def test_profiled_traffic_needs_matching_source_hash(tmp_path, monkeypatch):
    sha = bench.source_sha(bench.KERNEL_SOURCES["verify"])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "x.md").write_text(
        f"bench-traffic: kernel=verify workload=chain16 source_sha={sha} "
        f"dram_bytes_per_launch=123\n"
        f"bench-traffic: kernel=verify workload=tree22 source_sha=0000000000000000 "
        f"dram_bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_sha", lambda files: sha)
    assert bench.profiled_traffic("verify", "chain16") == 123
    assert bench.profiled_traffic("verify", "tree22") is None   # stale: sources changed


@pytest.mark.timeout(600)
def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "node-heads/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_tree_walk_stats():
    """Rounds and L2 parent reads of the level walk reported by the tree22
    shape sweep: the test tree takes 8 rounds with every parent on chip; a
    star takes 1 + ceil(21 / 4) rounds; a level with four parents that have
    children puts the fourth one's children on L2 unless a warp still holds
    it."""
    import bench
    import synthetic

    st = bench.tree_walk_stats([int(x) for x in synthetic.tree22()["parent"][0]])
    assert st == {"depth": 6, "rounds": 8, "parents_read_from_l2": 0}
    star = [-1] + [0] * 21
    assert bench.tree_walk_stats(star) == {"depth": 2, "rounds": 7, "parents_read_from_l2": 0}
    # level 2 holds nodes 1..5, each with one child (nodes 6..10); nodes 1-3
    # are stashed, 4 and 5 are not.  Round robin: level 2 puts nodes 1..5 on
    # warps 0, 1, 2, 3, 0 and level 3 nodes 6..10 on the same warps, so node 9
    # finds its parent 4 in warp 3's registers, but warp 0 has formed node 6
    # since node 5: node 10 reads node 5 back through L2
    wide = [-1, 0, 0, 0, 0, 0, 1, 2, 3, 4, 5]
    assert bench.tree_walk_stats(wide) == {"depth": 3, "rounds": 5, "parents_read_from_l2": 1}
