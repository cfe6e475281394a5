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
