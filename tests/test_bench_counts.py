"""The benchmark's algorithmic counts against a plain enumeration (CPU only).

The roofline numbers divide these counts by measured times, so they are pinned here to a count
made the long way: every conv output position of every level, k x k multiply-adds each."""
import pytest

import bench
from memory_bound_cnn_gb300.inputs import WORKLOADS


def enumerated_macs(s):
    """Multiply-adds of one forward pass: the base conv at every pixel plus, at every level, the
    four subband convs at every level position (each k x k)."""
    macs = s.k * s.k * s.H * s.W
    h, w = s.H, s.W
    for _ in range(s.L):
        h, w = (h + 1) // 2, (w + 1) // 2
        macs += 4 * s.k * s.k * h * w
    return s.B * s.C * macs


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_algorithmic_counts_match_enumeration(name):
    for s in WORKLOADS[name]:
        a = bench.algorithmic(s)
        n = s.B * s.C * s.H * s.W
        e = 4 if s.dtype == "f32" else 2
        assert a["fwd_flop"] == pytest.approx(2 * enumerated_macs(s), rel=1e-12)
        assert a["bwd_flop"] == pytest.approx(2 * a["fwd_flop"], rel=1e-12)  # dx and dW: one forward each
        assert a["fwd_bytes"] == 2 * n * e                                     # x in, y out
        assert a["bwd_bytes"] == 3 * n * e                                     # x, dy in, dx out


def test_whole_job_throughput_counts_every_rank():
    assert bench.whole_job_throughput(10**9, 1, 1.0) == pytest.approx(1.0)
    assert bench.whole_job_throughput(10**9, 4, 2.0) == pytest.approx(2.0)
