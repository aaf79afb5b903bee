"""Host-side pieces of bench.py (no GPU): its defaults keep the timing rules, and its launch counts follow
the kernels one call of each entry point launches."""
import os
import sys

import datagen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_defaults_keep_the_timing_rules(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert a.config == "prefill_128k" and a.impl == "ours"


def test_prefill_launch_count():
    # select 1, B* inversion 4, then per query slab: schedule 3, tiles 1, combine 1
    cfg = datagen.CONFIGS["prefill_128k"]
    assert bench.prefill_slabs(cfg) == 1
    assert bench.prefill_launches(cfg) == 10


def test_backward_launch_count():
    # inversion 4 and rowdot 1, then per slab: schedule 3, mark_repeats 1, index lse 2, main 1, index 1
    assert bench.bwd_launches(datagen.CONFIGS["prefill_128k"]) == 13
    two = datagen.make_config("two_slabs", N=180000, H_q=8, H_kv=2, d=128, d_I=128, Bk=128, k=8, needles=0)
    assert bench.bwd_launches(two) == 21


def test_varlen_mix_fills_the_cells():
    for N, Bk in ((131072, 128), (8192, 64), (32768, 128)):
        lengths = bench.varlen_mix(N, Bk)
        assert sum(lengths) == N
        assert all(x > 0 for x in lengths)
        assert all(x % Bk == 0 for x in lengths[:-1])
