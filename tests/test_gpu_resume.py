"""Checkpoint/resume and run-to-run bit identity of the whole owner-side step.

The DMuon home page ("Key Features", "Bit-Identical Correctness") states that
its paths give identical loss trajectories and that this was tested via a
checkpoint restart.  The single-GPU analogue here: the step's only state is
(W, M), so three steps in one run must equal two steps, a save of (W, M), a
fresh owner (new packed buffer and workspace) restored from the save, and a
third step -- bit for bit.  And two independent runs on the same inputs must
agree bit for bit (no atomics, fixed reduction orders).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [(512, 512), (128, 512), (128, 512), (512, 512), (1400, 512), (1400, 512), (512, 1400),
          (300, 7)]


def _run(dm, wl, steps, restore=None, start=0):
    own = dm.MuonOwner(SHAPES)
    if restore is None:
        W = [wl.random_matrix(s, 700 + i, "cuda", 0.02, torch.bfloat16) for i, s in enumerate(SHAPES)]
        M = [torch.zeros(s, device="cuda") for s in SHAPES]
    else:
        W = [w.clone().cuda() for w in restore[0]]
        M = [m.clone().cuda() for m in restore[1]]
    for k in range(start, start + steps):
        G = [wl.random_matrix(s, 10_000 * (k + 1) + i, "cuda", 1e-3, torch.bfloat16)
             for i, s in enumerate(SHAPES)]
        own.step(G, M, W, lr=0.02, beta=0.95, ns_steps=5)
        assert own.status() == dm.OK
    torch.cuda.synchronize()
    return [w.cpu() for w in W], [m.cpu() for m in M]


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


def _same(a, b):
    return all(torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))
               for x, y in zip(a, b))


def test_resume_from_saved_state_is_bit_identical(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    W3, M3 = _run(dm, wl, 3)
    W2, M2 = _run(dm, wl, 2)
    W3r, M3r = _run(dm, wl, 1, restore=(W2, M2), start=2)
    assert _same(W3, W3r) and _same(M3, M3r)
    assert not _same(W3, W2)          # the third step did change the weights


@pytest.mark.parametrize("variant", [0, 1])
def test_overlapped_step_equals_three_separate_calls(dm, variant):
    """dmuon_muon_step runs the memory-bound kernels of later and earlier buckets
    on a second stream next to the current bucket's products, bucket by bucket;
    the result must be the same bits as pack, Newton-Schulz and update called one
    after another over all buckets -- with the standard form and with the Gram
    variant (whose rule gives the rectangular matrices here the Gram form)."""
    from newton_schulz_owner_gb300 import workloads as wl
    if variant == 1:
        assert any(dm.ns_variant_for(s, 5, dm.NS_GRAM) == dm.NS_GRAM for s in SHAPES)
    outs = []
    for mode in ("whole", "three"):
        own = dm.MuonOwner(SHAPES, variant=variant)
        W = [wl.random_matrix(s, 700 + i, "cuda", 0.02, torch.bfloat16) for i, s in enumerate(SHAPES)]
        M = [torch.zeros(s, device="cuda") for s in SHAPES]
        for k in range(2):
            G = [wl.random_matrix(s, 10_000 * (k + 1) + i, "cuda", 1e-3, torch.bfloat16)
                 for i, s in enumerate(SHAPES)]
            if mode == "whole":
                own.step(G, M, W, lr=0.02, beta=0.95, ns_steps=5)
            else:
                dm.pack(SHAPES, G, M, 0.95, own.packed, own.offsets, own.workspace)
                dm.ns_batched(SHAPES, own.packed, own.offsets, own.workspace, ns_steps=5,
                              variant=variant, use_pack_norms=True)
                dm.unpack_update(SHAPES, W, 0.02, own.packed, own.offsets, own.workspace)
            assert own.status() == dm.OK
        torch.cuda.synchronize()
        outs.append(([w.cpu() for w in W], [m.cpu() for m in M],
                     [own.packed_view(i).cpu() for i in range(len(SHAPES))]))
    for a, b in zip(outs[0], outs[1]):
        assert _same(a, b)


def test_two_runs_are_bit_identical(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    a = _run(dm, wl, 2)
    b = _run(dm, wl, 2)
    assert _same(a[0], b[0]) and _same(a[1], b[1])
