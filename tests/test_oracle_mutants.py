"""Plant plausible mistakes in a private copy of the oracle (on the CPU) and
check that the pins catch every one of them.  A pin set that let a dropped
term, a flipped sign, a transposed operand or a wrong index through would not
be worth trusting."""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.cpp")

MUTANTS = {
    "flipped_sign_in_erase": ("alpha * (s - beta * u[j] * k[i])",
                              "alpha * (s + beta * u[j] * k[i])"),
    "dropped_write_term": ("+ beta * v[j] * k[i];", ";"),
    "decay_on_write_term": ("+ beta * v[j] * k[i];", "+ alpha * beta * v[j] * k[i];"),
    "transposed_readout": ("acc += H[(int64_t)i * dv + j] * k[i];",
                           "acc += H[(int64_t)j * dv + i] * k[i];"),
    "output_reads_key": ("acc += H[(int64_t)i * dv + j] * q[i];",
                         "acc += H[(int64_t)i * dv + j] * k[i];"),
    "tree_ignores_parent": ("int src = par ? par[n] : n - 1;", "int src = n - 1;"),
    "wrong_head_group": ("const int hk = h / G;", "const int hk = h % Hk;"),
    "commit_wrong_node": ("(((int64_t)b * N + a) * Hv + h) * hs;",
                          "(((int64_t)b * N + (N - 1)) * Hv + h) * hs;"),
    "commit_ignores_slot": ("double* to = cache + l * cache_layer_stride + sl * cache_slot_stride",
                            "double* to = cache + l * cache_layer_stride + b * cache_slot_stride"),
    "depth_off_by_one": ("depth[n] = depth[p] + 1;", "depth[n] = depth[p] + (p > 0);"),
    "depth_cap_off_by_one": ("if (depth[n] > max_depth) return ERR_BAD_TREE;",
                             "if (depth[n] >= max_depth) return ERR_BAD_TREE;"),
    "prefill_drops_decay": ("alpha[(int64_t)t * Hv + h],\n",
                            "1.0 + 0 * alpha[(int64_t)t * Hv + h],\n"),
    "replay_drops_root": ("for (int m = acc; m >= 0; m = par[m]) path.insert",
                          "for (int m = acc; m > 0; m = par[m]) path.insert"),
    "conv_keeps_oldest": ("for (int w = 0; w < W; ++w) h[w] = seq[seq.size() - W + w];",
                          "for (int w = 0; w < W; ++w) h[w] = seq[w];"),
    "conv_ignores_parent": ("for (int m = acc; m >= 0; m = par[m]) path.insert(path.begin(), m);\n"
                            "    } else {\n      for (int m = 0; m <= acc; ++m) path.push_back(m);\n"
                            "    }\n    for (int c = 0; c < C; ++c) {",
                            "for (int m = 0; m <= acc; ++m) path.push_back(m);\n"
                            "    } else {\n      for (int m = 0; m <= acc; ++m) path.push_back(m);\n"
                            "    }\n    for (int c = 0; c < C; ++c) {"),
    "prep_gate_sign": ("ab_alpha[i] = std::exp(-softplus);", "ab_alpha[i] = std::exp(softplus - 2 * a);"),
    "prep_skips_norm": ("for (int i = 0; i < d; ++i) x[i] *= inv;", "for (int i = 0; i < d; ++i) x[i] *= 1.0;"),
    "index_commit_wrong_stride": ("slot[b] = base + b * N + accept[b];",
                                  "slot[b] = base + b * (N - 1) + accept[b];"),
    "replay_chain_short": ("for (int m = 0; m <= acc; ++m) path.push_back(m);",
                           "for (int m = 0; m < acc; ++m) path.push_back(m);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    cpp = tmp_path / "mutant.cpp"
    cpp.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fPIC", "-shared", str(cpp), "-o",
                           str(so)])
    lib = oracle.bind(ctypes.CDLL(str(so)))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check()
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
