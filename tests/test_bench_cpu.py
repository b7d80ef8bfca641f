"""CPU checks of bench.py's host logic: the algorithmic pair counts behind
the roofline figures, the schedules, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_pair_counts_match_oracle_key_sets():
    import bench

    T = bench.T
    for alpha in (0.5, 0.5 + 5 / 15, 1.0, 1.5):
        for W in (6, 8, 12):
            slots = o.interp_slots(bench.FIB, alpha, W)
            ok = np.zeros((len(slots), T), dtype=bool)
            for a, sl in enumerate(slots):
                lo = sl["s"] if sl["kind"] == "win" else sl["c"]
                ok[a, lo:] = lo < T
            rung_rows = [a for a, sl in enumerate(slots) if sl["kind"] == "rung"]
            pairs, rung = bench.pair_counts(alpha, W)
            assert pairs == ok.sum() and rung == ok[rung_rows].sum()


def test_pair_counts_take_other_base_lists():
    import bench

    pow2 = [1 << j for j in range(11)]
    slots = o.interp_slots(pow2, 0.5 + 9 / 15, 8)
    T = bench.T
    want = sum(max(0, T - (sl["s"] if sl["kind"] == "win" else sl["c"])) for sl in slots)
    assert bench.pair_counts(0.5 + 9 / 15, 8, pow2)[0] == want


def test_step_order():
    """The timed step runs every layer's forward first, then the backwards
    from the last layer to the first; --order layerwise pairs them per layer."""
    import bench

    calls = []

    class FakeLayer:
        def __init__(self, i):
            self.i = i

        def run_fwd(self, stream):
            calls.append(("fwd", self.i))

        def run_bwd(self, stream):
            calls.append(("bwd", self.i))

        def run(self, stream):
            self.run_fwd(stream)
            self.run_bwd(stream)

    layers = [FakeLayer(i) for i in range(3)]
    saved = bench.ORDER
    try:
        bench.ORDER = "training"
        bench.run_layers(layers, None)
        assert calls == [("fwd", 0), ("fwd", 1), ("fwd", 2), ("bwd", 2), ("bwd", 1), ("bwd", 0)]
        calls.clear()
        bench.ORDER = "layerwise"
        bench.run_layers(layers, None)
        assert calls == [("fwd", 0), ("bwd", 0), ("fwd", 1), ("bwd", 1), ("fwd", 2), ("bwd", 2)]
    finally:
        bench.ORDER = saved


def test_schedules_match_oracle():
    import bench

    assert bench.alphas("linear") == o.alpha_schedule(16, o.SCHED_LINEAR)
    assert bench.alphas("coprime") == o.alpha_schedule(16, o.SCHED_COPRIME, 7)
    assert bench.alphas("fixed") == [1.0] * 16


def test_unique_bytes_per_token():
    """bf16 rows of 64 dims: a query-head tensor is 8 x 128 B per token, a
    KV-head tensor 2 x 128 B."""
    import bench

    qh, kvh = 8 * 128, 2 * 128
    assert bench.UNIQUE_BYTES_PER_TOKEN == 4 * qh + 4 * kvh == 5120  # Q O dO dQ, K V dK dV
    assert bench.KERNEL_BYTES_PER_TOKEN["fwd"] == 2 * qh + 2 * kvh      # Q, O, K, V
    assert bench.KERNEL_BYTES_PER_TOKEN["bwd_q"] == 4 * qh + 2 * kvh    # Q, O, dO, dQ, K, V
    assert bench.KERNEL_BYTES_PER_TOKEN["bwd_kv"] == 2 * qh + 2 * kvh   # Q, dO, dK, dV


def test_reference_arm_json_line():
    import time

    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["warmup"] >= 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["seq_len"] == 1024 and d["config"]["global_batch"] == 32
    # the timed steps fit in the run that printed them; the scale to the
    # workload's step (32 sequences x 16 layers) is a separate field
    assert d["steps"] * d["ms_per_step"] * 1e-3 <= wall
    assert d["sample_scale"]["factor"] == 32 * 16
    assert abs(d["value"] - 32 * 1024 / (d["sample_scale"]["workload_ms_per_step"] * 1e-3)) <= 1e-2 * d["value"]
