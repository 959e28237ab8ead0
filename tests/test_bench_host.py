"""bench.py on the host: the reference arm's JSON line carries the contract's
keys, and the workload arithmetic the roofline uses agrees with the oracle's
chunk plan and budget rule (no GPU needed)."""
import json
import math
import os
import subprocess
import sys

import pytest

import kv_synth as ks
from oracle import kv2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("cfg", [ks.TINY, ks.LLAMA_16K, ks.QWEN_32K, ks.LLAMA_128K], ids=lambda c: c.name)
def test_workload_arithmetic_matches_the_oracle_plan(cfg):
    w = bench.algorithmic_work(cfg)
    ch = kv2.chunk_plan(cfg.N, cfg.sinks, cfg.m, cfg.rho)
    assert w["Q"] == sum(c.nq for c in ch)
    assert w["k"] == kv2.budget_count(cfg.budget, cfg.N)
    # pass 2 multiplies each chunk's queries by its own keys only
    col = cfg.L * cfg.Hq * 2 * cfg.d * sum(c.nq * (c.hi - c.lo) for c in ch)
    assert w["flops_colmax_per_launch"] == col
    # pass 1 sees the whole cache plus the causal triangle of appended keys
    lse = cfg.L * cfg.Hq * 2 * cfg.d * sum(c.nq * cfg.N + c.nq * (c.nq + 1) / 2 for c in ch)
    assert math.isclose(w["flops_lse_per_launch"], lse, rel_tol=1e-12)
    assert w["flops_lse"] == lse * cfg.passes or math.isclose(w["flops_lse"], lse * cfg.passes, rel_tol=1e-12)


def test_decode_bytes_count_every_kept_row_once():
    cfg = ks.DECODE_128K
    assert bench.decode_bytes(cfg) == cfg.n_seg * cfg.kept * 512 + cfg.n_seg * cfg.G * (256 + 512 + 4)


def test_epicache_evict_compact_bytes_hand_worked():
    """Blocks of 4, 4, 2 tokens; budgets 5 and 12.  Layer 0 reaches 8 > 5
    (reads 8 scores, writes 5 indices, moves 5 rows), then 5 + 2 = 7 > 5
    (7 scores, 5 indices, 5 rows); layer 1 stays at or under 12.  Each kept
    row moves K and V (256 B each, read and written) and its int32 position
    (read and written): 1032 B per row and KV head; scores and indices are
    4 B each."""
    import types
    cfg = types.SimpleNamespace(L=2, Hkv=3, block=4, sinks=2, n_hist=10)
    step1 = 8 * 4 + 5 * 4 + 5 * 1032
    step2 = 7 * 4 + 5 * 4 + 5 * 1032
    assert bench.epi_evict_compact_bytes(cfg, [5, 12]) == 3 * (step1 + step2)


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
                          "tiny-4k", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "tiny-4k"
