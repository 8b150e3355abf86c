"""Host logic of bench.py that feeds its JSON line, on CPU.

* The algorithmic flops count visible (row, key) pairs through each node's
  depth; here they are counted instead by brute force over the oracle's mask
  bytes, for random trees of every shape rule.
* The algorithmic bytes are recomputed from their definition for both mask
  forms and the prefix skip.
* The committed DRAM traffic is reported only while the kernel sources it
  was measured on are unchanged; comments and layout do not count as a
  change, code does."""
import importlib.util
import json
import os

import numpy as np
import pytest

import oracle
from speculative_decode_mla_tree_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_cpu_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _small(rule, seed):
    return W.make_workload("b", 3, [40, 7, 90], rule, [9, 1, 17], 4096, seed=seed)


@pytest.mark.parametrize("rule", ["uniform", "chain", "branch3", "branch4d8"])
def test_flops_equal_visible_pairs(bench, rule):
    w = _small(rule, 5)
    kv_indices, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr,
                                                    w.out_cache_loc, w.qo_indptr)
    _, mask = oracle.tree_mask_pack(w.parents, w.qo_indptr, kv_indptr)
    visible = int(np.count_nonzero(mask))
    _, flops = bench.alg_cost(w)
    assert flops == 2 * (576 + 512) * w.heads * visible


def test_bytes_from_definition(bench):
    w = _small("uniform", 9)
    H = w.heads
    want_bytes_mask, want_bits_mask, want_bits_skip = 0, 0, 0
    for b in range(w.batch):
        n, P = w.tree_sizes[b], w.prefix_lens[b]
        L = P + n
        common = L * 1152 + L * 4 + n * H * (1152 + 1024 + 4)
        want_bytes_mask += common + n * L
        want_bits_mask += common + n * 4 * ((L + 31) // 32)
        want_bits_skip += common + n * 4 * ((L + 31) // 32 - P // 32)
    assert bench.alg_cost(w)[0] == want_bytes_mask
    assert bench.alg_cost(w, mask_bits=True)[0] == want_bits_mask
    assert bench.alg_cost(w, mask_bits=True, skip_prefix=True)[0] == want_bits_skip


def test_traffic_only_for_current_sources(bench, tmp_path, monkeypatch):
    h = bench._kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "verify_c5": {"dram_bytes_per_launch": 123.0, "source_hash": h},
        "verify_c3": {"dram_bytes_per_launch": 456.0, "source_hash": "0" * 16},
    }))
    csrc = os.path.join(ROOT, "speculative_decode_mla_tree_gb300", "csrc")
    os.symlink(os.path.dirname(csrc), tmp_path / "speculative_decode_mla_tree_gb300")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("verify_c5") == 123.0
    assert bench._traffic("verify_c3") is None      # measured on other sources
    assert bench._traffic("verify_c1") is None      # never measured


def test_committed_traffic_names_its_sources(bench):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for key, e in t.items():
        assert key.startswith("verify_c")
        assert e["dram_bytes_per_launch"] > 0
        assert len(e["source_hash"]) == 16


def test_source_hash_ignores_comments_not_code(bench):
    base = 'int f(int x) {\n  return x + 1;  // one more\n}\nconst char* s = "a // b /* c */";\n'
    same = ('/* header\n   text */\nint f(int x)\n{\n    return x + 1;\n}\n'
            'const char* s = "a // b /* c */";  // the string keeps its slashes\n')
    other = 'int f(int x) {\n  return x + 2;  // one more\n}\nconst char* s = "a // b /* c */";\n'
    lit = 'int f(int x) {\n  return x + 1;  // one more\n}\nconst char* s = "a //  b /* c */";\n'
    t = bench._code_tokens
    assert t(base) == t(same)
    assert t(base) != t(other)
    assert t(base) != t(lit)      # white space inside a literal is code
    assert "one more" not in t(base) and "// b /* c */" in t(base)
