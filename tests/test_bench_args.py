"""bench.py's workload selection on the CPU: --config N, or a serving batch of B full rows
(--batch B --context L); both flags are needed together."""
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def _args(**kw):
    base = dict(config=3, batch=0, context=0)
    base.update(kw)
    return types.SimpleNamespace(**base)


def test_serving_batch_workload():
    w = bench.base_workload(_args(config=1, batch=6, context=40))
    assert tuple(w.q.shape) == (6, 32, 128)
    assert tuple(w.k.shape) == (6, 8, 40, 128)
    assert w.seq_lens.tolist() == [40] * 6                  # every row full
    assert w.name == "serving bf16 B6 Hq32 Hkv8 d128 L40"
    again = workloads.serving_case(6, 40)                   # seeded: the same values
    assert bool((again.k == w.k).all()) and bool((again.q == w.q).all())


def test_config_workload_by_default():
    w = bench.base_workload(_args(config=1))
    assert w.name == workloads.config1().name


@pytest.mark.parametrize("kw", [dict(batch=4), dict(context=64), dict(batch=-1, context=8)])
def test_serving_flags_go_together(kw):
    with pytest.raises(SystemExit):
        bench.base_workload(_args(**kw))
