"""The whole owner-side step captured once into a CUDA graph and replayed.

A training loop that runs the same step every iteration can capture it and
replay it without re-planning or re-launching from the host.  The library's
tables are written by a kernel (so they are part of the graph), and the step's
second stream forks from and joins the caller's stream through events (so it
is captured as graph edges).  Replaying the graph over two steps, with each
step's gradients copied into the captured buffers, must give the same bits as
calling dmuon_muon_step eagerly.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [(512, 512), (128, 512), (1400, 512), (512, 1400), (300, 7), (7, 300)]


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


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_whole_step_replayed_from_a_cuda_graph_matches_eager_calls(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    W0 = [wl.random_matrix(s, 900 + i, "cuda", 0.02, torch.bfloat16) for i, s in enumerate(SHAPES)]
    Gs = [[wl.random_matrix(s, 20_000 * (k + 1) + i, "cuda", 1e-3, torch.bfloat16)
           for i, s in enumerate(SHAPES)] for k in range(2)]

    # eager reference (also performs the library's one-time device set-up)
    own_e = dm.MuonOwner(SHAPES)
    W_e = [w.clone() for w in W0]
    M_e = [torch.zeros(s, device="cuda") for s in SHAPES]
    for k in range(2):
        own_e.step(Gs[k], M_e, W_e, lr=0.02, beta=0.95, ns_steps=5)
    assert own_e.status() == dm.OK
    torch.cuda.synchronize()

    # captured once, replayed per step
    own_g = dm.MuonOwner(SHAPES)
    W_g = [w.clone() for w in W0]
    M_g = [torch.zeros(s, device="cuda") for s in SHAPES]
    G_static = [torch.empty(s, dtype=torch.bfloat16, device="cuda") for s in SHAPES]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        own_g.step(G_static, M_g, W_g, lr=0.02, beta=0.95, ns_steps=5)
    # capture enqueues nothing: state is untouched until the first replay
    torch.cuda.synchronize()
    assert all(torch.equal(_bits(a), _bits(b)) for a, b in zip(W_g, W0))
    for k in range(2):
        for dst, src in zip(G_static, Gs[k]):
            dst.copy_(src)
        graph.replay()
    torch.cuda.synchronize()
    assert own_g.status() == dm.OK

    for a, b in zip(W_g, W_e):
        assert torch.equal(_bits(a), _bits(b))
    for a, b in zip(M_g, M_e):
        assert torch.equal(_bits(a), _bits(b))
    for i in range(len(SHAPES)):
        assert torch.equal(_bits(own_g.packed_view(i)), _bits(own_e.packed_view(i)))
