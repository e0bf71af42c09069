"""Host logic of bench.py that feeds the reported roofline: the algorithmic bytes and FLOPs
of one latent-attention launch (by definition, independent of the kernels), the peak
figures, and the traffic record lookup."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_latent_kv_70_b300 import inputs as I  # noqa: E402


def test_dsv3_bytes_and_flops():
    cache, total, flops = bench.algorithmic(I.dsv3())
    assert cache == 64 * 4096 * 1152                          # 301,989,888 B of cache rows
    assert total == cache + 64 * 128 * (576 * 2 + 512 * 4 + 4)  # q_cat in, o_lat and lse out
    assert total == 328_237_056
    assert flops == 2 * 128 * (576 + 512) * 64 * 4096          # 73.0 GFLOP
    assert flops / total == pytest.approx(222.4, abs=0.1)       # FLOP per algorithmic byte


def test_causal_two_token_pairs():
    # With S = 2 causal, the first query token reads T-1 rows and the second T.
    case = I.make_case("c", 3, 2, 16, [5, 1, 64], causal=True, seed=0)
    _, _, flops = bench.algorithmic(case)
    pairs = (4 + 5) + (0 + 1) + (63 + 64)
    assert flops == 2 * 16 * (576 + 512) * pairs


def test_ragged_cache_bytes_follow_the_lengths():
    case = I.ragged_paged()
    cache, _, _ = bench.algorithmic(case)
    assert cache == 1152 * sum(case.seqlens)


def test_peaks_are_read():
    hbm, tf, tf_sus, kind = bench.measured_peaks()
    assert kind in ("measured", "fallback")
    assert hbm > 0 and tf > 0 and 0 < tf_sus <= tf * 1.05


def test_traffic_record_only_for_known_workloads():
    assert bench.recorded_traffic("no_such_workload") is None
