"""Tracing of the product launches (dmuon_trace_begin / dmuon_trace_end).

A traced Newton-Schulz call must give the same bits as an untraced one, and
its records must be complete and consistent: one record per CTA of every
product launch, launches numbered in order, every CTA pair's stamps ordered
entry <= first MMA <= last MMA <= exit for the CTA that issues the MMAs (the
first of the pair), the other CTA's MMA stamps zero, and the MMA thread's wait
cycles within its MMA span.  Launches beyond the buffer are not traced, and
nothing is recorded once tracing has ended.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [(256, 1024), (1024, 256), (300, 7), (129, 257), (512, 512)]


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    from newton_schulz_owner_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from newton_schulz_owner_gb300 import dmuon
    return dmuon


def _call(dm, ws, packed, offsets, steps=3):
    dm.ns_batched(SHAPES, packed, offsets, ws, ns_steps=steps)
    assert dm.stream_status(ws) == dm.OK


def test_trace_records_are_complete_and_change_nothing(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    _, off, oel = dm.plan(SHAPES)
    src = torch.zeros(sum(oel), dtype=torch.bfloat16, device="cuda")
    for i, (r, c) in enumerate(SHAPES):
        src[off[i]:off[i] + r * c].view(r, c).copy_(
            wl.random_matrix((r, c), 40 + i, "cuda", 1.0, torch.bfloat16))
    ws = torch.zeros(dm.workspace_bytes(SHAPES), dtype=torch.uint8, device="cuda")
    plain = src.clone()
    _call(dm, ws, plain, off)
    traced = src.clone()
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    dm.trace_begin(buf)
    _call(dm, ws, traced, off)
    rec = dm.trace_end(buf)
    assert torch.equal(plain.view(torch.int16), traced.view(torch.int16))

    n = rec["cta"].numel()
    assert n > 0 and n % 2 == 0
    launches = sorted(set(rec["launch"].tolist()))
    assert launches == list(range(len(launches)))
    # 3 steps x (X X^T, A A, B X), each split by orientation: at least 9 launches
    assert len(launches) >= 9
    for L in launches:
        m = rec["launch"] == L
        ctas = sorted(rec["cta"][m].tolist())
        assert ctas == list(range(len(ctas))) and len(ctas) % 2 == 0
        assert len(set(rec["kind"][m].tolist())) == 1 and int(rec["kind"][m][0]) in (0, 1, 2, 3)
    lead = rec["cta"] % 2 == 0
    has = lead & (rec["t_mma_first"] > 0)
    assert bool((rec["t_entry"][has] <= rec["t_mma_first"][has]).all())
    assert bool((rec["t_mma_first"][has] <= rec["t_mma_last"][has]).all())
    assert bool((rec["t_mma_last"][has] <= rec["t_exit"][has]).all())
    assert bool((rec["t_entry"] <= rec["t_exit"]).all())
    assert bool((rec["t_mma_first"][~lead] == 0).all()) and bool((rec["mma_span_cycles"][~lead] == 0).all())
    waits = rec["wait_operand_cycles"][has] + rec["wait_accum_cycles"][has]
    assert bool((waits <= rec["mma_span_cycles"][has]).all())

    # a buffer with room for a few records: the launches that fit are traced
    # (numbered from 0), the others are not, and nothing is written past it
    cap = 24
    small = torch.zeros((cap + 4) * dm.TRACE_RECORD_BYTES, dtype=torch.uint8, device="cuda")
    dm.trace_begin(small[:cap * dm.TRACE_RECORD_BYTES])
    _call(dm, ws, src.clone(), off)
    rec2 = dm.trace_end(small)
    assert 0 < rec2["cta"].numel() <= cap
    got = sorted(set(rec2["launch"].tolist()))
    assert got == list(range(len(got))) and len(got) < len(launches)
    assert not bool(small[cap * dm.TRACE_RECORD_BYTES:].any())
    # after trace_end nothing is recorded
    before = buf.clone()
    _call(dm, ws, src.clone(), off)
    torch.cuda.synchronize()
    assert torch.equal(before, buf)
