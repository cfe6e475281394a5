"""Host-side helpers of the benchmark (no GPU).

The bench reports the product kernel's DRAM traffic from a committed ncu
summary, which is valid only for the kernel source it was captured from: the
record carries that source's SHA-256 and the bench must drop the figure as soon
as the source differs.  The algorithmic byte count per Newton-Schulz phase is
computed from the shapes and must agree with the per-layer figure the summary
states (X read twice and X' written: 6mn bytes; A and B written and read once:
8m^2 bytes, bf16).
"""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _bench():
    import bench
    return bench


def test_traffic_record_matches_current_kernel_source_or_is_dropped(tmp_path, monkeypatch):
    b = _bench()
    rec = b.traffic_record()
    src = os.path.join(ROOT, "newton_schulz_owner_gb300", "csrc", "ns_gemm.cu")
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    with open(os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")) as f:
        stored = json.load(f)
    if stored["source_sha256"] == h:
        assert rec is not None and rec["dram_bytes_per_ns_phase"] > 0
    else:
        assert rec is None
    # a record for another source is never reported
    fake_root = tmp_path / "repo"
    (fake_root / "profiles").mkdir(parents=True)
    (fake_root / "newton_schulz_owner_gb300" / "csrc").mkdir(parents=True)
    (fake_root / "newton_schulz_owner_gb300" / "csrc" / "ns_gemm.cu").write_text("// other\n")
    stored["source_sha256"] = h
    (fake_root / "profiles" / "ns_gemm_traffic.json").write_text(json.dumps(stored))
    monkeypatch.setattr(b, "ROOT", str(fake_root))
    assert b.traffic_record() is None


def test_layer_traffic_record_is_above_the_algorithmic_bytes():
    b = _bench()
    with open(os.path.join(ROOT, "profiles", "ns_gemm_traffic.json")) as f:
        stored = json.load(f)
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (14336, 4096),
              (14336, 4096), (4096, 14336)]
    alg = sum(6 * min(r, c) * max(r, c) + 8 * min(r, c) ** 2 for r, c in shapes)
    assert alg == pytest.approx(1996.49e6, rel=1e-5)
    # DRAM traffic cannot be below what the products must move at least once
    assert stored["dram_bytes_per_layer_iteration"] >= alg
    assert stored["dram_bytes_per_ns_phase"] == pytest.approx(
        stored["dram_bytes_per_layer_iteration"] * 32 * 5)
    assert callable(b.blas_name) and isinstance(b.blas_name(), str) and b.blas_name()


def test_trace_summary_splits_pair_time():
    """Two launches of two pairs each (four CTAs), hand-made timestamps in ns:
    launch 0 runs 0..1000 (pair 0 MMA 100..900, pair 1 MMA 100..500, exits at
    600), launch 1 starts after a 200 ns gap and runs 1200..2000 (both pairs
    MMA 1300..1900).  Window 2000 ns x 2 pairs = 4000 pair-ns; MMA-active
    800 + 400 + 600 + 600 = 2400; resident 1000 + 600 + 800 + 800 = 3200."""
    import torch
    b = _bench()
    T = lambda v: torch.tensor(v, dtype=torch.int64)
    rec = {"launch": T([0, 0, 0, 0, 1, 1, 1, 1]), "cta": T([0, 1, 2, 3, 0, 1, 2, 3]),
           "kind": T([0] * 8), "tiles": T([2] * 8),
           "t_entry": T([0, 0, 0, 0, 1200, 1200, 1200, 1200]),
           "t_mma_first": T([100, 0, 100, 0, 1300, 0, 1300, 0]),
           "t_mma_last": T([900, 0, 500, 0, 1900, 0, 1900, 0]),
           "t_exit": T([1000, 1000, 600, 600, 2000, 2000, 2000, 2000])}
    s = b.trace_summary(rec, step_ms=0.003)
    assert s["launches"] == 2 and s["pairs"] == 2
    assert s["product_window_ms"] == pytest.approx(2000e-6)
    assert s["mma_active_frac"] == pytest.approx(2400 / 4000)
    assert s["fill_drain_frac"] == pytest.approx(800 / 4000)
    assert s["not_resident_frac"] == pytest.approx(800 / 4000)
    assert s["launch_gaps_ms"] == pytest.approx(200e-6)
    assert s["recoverable_ms_upper_bound"] == pytest.approx(1600e-6 / 2)


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 5, 8])
def test_bench_flop_counts_agree_with_the_oracle(steps):
    """The bench counts algorithmic flops itself (its GPU leg does not touch
    the oracle); both counts must agree with the oracle's."""
    import oracle
    b = _bench()
    shapes = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336), (300, 7), (1, 1)]
    assert b.ns_flops(shapes, steps) == pytest.approx(oracle.ns_flops_algorithmic(shapes, steps))
    assert b.gram_flops(shapes, steps) == pytest.approx(
        oracle.gram_ns_flops_algorithmic(shapes, steps))


@pytest.mark.parametrize("layers", [1, 3, 28, 32])
@pytest.mark.parametrize("groups", [1, 2, 4, 6, 8])
@pytest.mark.parametrize("taper", [False, True])
def test_e2e_groups_cover_every_layer_once(layers, groups, taper):
    b = _bench()
    g = b.e2e_group_bounds(layers, groups, taper)
    assert g[0][0] == 0 and g[-1][1] == layers
    assert all(lo < hi for lo, hi in g)
    assert all(g[k][1] == g[k + 1][0] for k in range(len(g) - 1))
    assert len(g) <= max(1, min(groups, layers))
    if taper and layers >= 16 and groups >= 4:
        sizes = [hi - lo for lo, hi in g]
        assert sizes[0] < max(sizes) and sizes[-1] < max(sizes)


def test_nominal_flops_count_every_product_in_full():
    b = _bench()
    s = [(1024, 4096)]
    m, n = 1024, 4096
    assert b.nominal_flops(s, 5) == pytest.approx(5 * (2 * m * m * n + 2 * m ** 3 + 2 * m * m * n))
    assert b.nominal_flops(s, 5) > b.ns_flops(s, 5)


def test_clock_sampler_keeps_only_samples_inside_the_window():
    """A short timed region is summarised from its own samples: idle samples
    before and after it (maximum clock, low power) do not enter the median."""
    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = _bench().ClockSampler(0)
    s.proc = FakeProc()
    row = "0, {mhz}, 2070, {w}, 0x0, Not Active, Not Active, Not Active, {cap}"
    s.lines = [(0.0, row.format(mhz=2070, w=200, cap="Not Active")),
               (1.0, row.format(mhz=1500, w=1300, cap="Active")),
               (1.2, row.format(mhz=1520, w=1350, cap="Active")),
               (1.4, row.format(mhz=1480, w=1340, cap="Active")),
               (3.0, row.format(mhz=2070, w=210, cap="Not Active"))]
    inside = s.stop(window=(0.9, 1.5))
    assert inside["samples"] == 3 and inside["sm_mhz"] == 1500
    assert inside["power_w_median"] == 1340 and inside["reasons"] == ["sw_power_cap"]
    s.proc = FakeProc()
    everything = s.stop()
    assert everything["samples"] == 5 and everything["sm_mhz"] == 1520
