"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (each derived from the arithmetic):
  * momentum, update (fp32 math): relative Frobenius error <= 1e-5
  * packed U, bf16 weights: within 1 bf16 ulp of RNE of the fp64 value (the
    fp32 result can sit on the other side of a rounding boundary); where
    W - lr*s*O cancels to about zero, within fp32 rounding of the operands
  * ns_steps = 0 (normalisation only): <= 5e-3 relative Frobenius (two bf16
    roundings of at most 2^-9 each)
  * Newton-Schulz with bf16 operands, fp32 accumulation: <= 2e-2 relative
    Frobenius per matrix for ns_steps <= 5, 4e-2 for 8 steps
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

NS_TOL = {0: 5e-3, 1: 2e-2, 2: 2e-2, 3: 2e-2, 5: 2e-2, 8: 4e-2}

# wide and tall (rows > cols: the working layout keeps the parameter's own
# orientation) shapes with ragged tiles in every dimension
ODD_SHAPES = [(1, 1), (1, 5), (5, 1), (7, 300), (300, 7), (129, 257), (257, 129), (64, 64),
              (256, 1024), (1024, 256), (1000, 1000), (96, 4096), (4096, 96), (130, 130),
              (8, 8200), (8200, 8), (333, 1500), (1500, 333)]


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from newton_schulz_owner_gb300 import build_lib
    import os
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from newton_schulz_owner_gb300 import dmuon
    return dmuon


@pytest.fixture(scope="module")
def wl():
    from newton_schulz_owner_gb300 import workloads
    return workloads


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def bf16_ulp_dist(gpu_bf16: torch.Tensor, ref64: np.ndarray) -> int:
    """Max distance in bf16 ulps between a bf16 tensor and RNE(ref64)."""
    ref = torch.from_numpy(oracle.round_bf16(ref64)).to(torch.bfloat16)
    a = gpu_bf16.detach().cpu().view(torch.int16).to(torch.int32)
    b = ref.view(torch.int16).to(torch.int32)
    # map sign-magnitude to a monotone integer line
    a = torch.where(a < 0, -(a & 0x7FFF), a)
    b = torch.where(b < 0, -(b & 0x7FFF), b)
    return int((a - b).abs().max().item()) if a.numel() else 0


def bf16_update_ok(w_gpu: torch.Tensor, w_ref64: np.ndarray, w0: np.ndarray,
                   step64: np.ndarray) -> bool:
    """Elementwise: within 1 bf16 ulp of RNE(w_ref64), or -- where W - lr*s*O
    cancels to (almost) zero and ulps lose meaning -- within fp32 rounding of
    the operands (lr*s is rounded to fp32 before the fused multiply-add)."""
    ref = torch.from_numpy(oracle.round_bf16(w_ref64)).to(torch.bfloat16)
    a = w_gpu.detach().cpu().view(torch.int16).to(torch.int32)
    b = ref.view(torch.int16).to(torch.int32)
    a = torch.where(a < 0, -(a & 0x7FFF), a)
    b = torch.where(b < 0, -(b & 0x7FFF), b)
    ulps = (a - b).abs().numpy()
    diff = np.abs(np64(w_gpu) - w_ref64)
    return bool(np.all((ulps <= 1) | (diff <= 2.0 ** -22 * (np.abs(w0) + np.abs(step64)))))


class PackedSet:
    """Packed buffer + workspace for a shape list, with canary guards."""

    def __init__(self, dm, shapes, variant=0, guard=True, n_owners=1):
        self.shapes = shapes
        own, off, oel = dm.plan(shapes, n_owners)
        g = 128 if guard else 0
        # shift every segment by a guard gap so that stray writes land in canaries
        self.offsets = [o + g * (i + 1) for i, o in enumerate(off)]
        total = sum(oel) + g * (len(shapes) + 2)
        self.packed = torch.empty(max(total, 128), dtype=torch.bfloat16, device="cuda")
        self.canary = torch.tensor([0x7F7F], dtype=torch.int16).view(torch.bfloat16).item()
        self.packed.fill_(self.canary)
        self.ws_bytes = dm.workspace_bytes(shapes, variant)
        self.ws_full = torch.zeros(self.ws_bytes + 4096, dtype=torch.uint8, device="cuda")
        self.ws_full[self.ws_bytes:] = 0xA5
        self.workspace = self.ws_full[:self.ws_bytes]

    def view(self, i):
        r, c = self.shapes[i]
        o = self.offsets[i]
        return self.packed[o:o + r * c].view(r, c)

    def guards_intact(self):
        mask = torch.ones_like(self.packed, dtype=torch.bool)
        for i, (r, c) in enumerate(self.shapes):
            mask[self.offsets[i]:self.offsets[i] + r * c] = False
        bad = (self.packed[mask].view(torch.int16) != 0x7F7F).sum().item()
        tail = (self.ws_full[self.ws_bytes:] != 0xA5).sum().item()
        return bad == 0 and tail == 0


def run_ns(dm, ps, steps, variant=0, abc=None):
    dm.ns_batched(ps.shapes, ps.packed, ps.offsets, ps.workspace, ns_steps=steps,
                  variant=variant, abc=abc, ws_bytes=ps.ws_bytes)
    assert dm.stream_status(ps.workspace) == dm.OK


# ------------------------------------------------------------------ NS
@pytest.mark.parametrize("steps", [0, 1, 2, 5, 8])
def test_ns_batched_odd_shapes(dm, wl, steps):
    ps = PackedSet(dm, ODD_SHAPES)
    ins = []
    for i, s in enumerate(ODD_SHAPES):
        u = wl.random_matrix(s, 100 + i, "cuda", 1.0, torch.bfloat16)
        ps.view(i).copy_(u)
        ins.append(np64(u))
    run_ns(dm, ps, steps)
    assert ps.guards_intact()
    for i, s in enumerate(ODD_SHAPES):
        ref = oracle.newton_schulz(ins[i], steps)
        err = rel(np64(ps.view(i)), ref)
        assert err <= NS_TOL[steps], f"{s} steps={steps}: rel err {err:.3e}"


# m and n on both sides of the product kernel's boundaries: a pipeline stage
# carries 128 of the reduction dimension, a tile 256 rows and columns, a TMA box
# 64; both orientations
BOUNDARY_SHAPES = [(127, 384), (128, 385), (129, 383), (255, 511), (256, 513), (257, 640),
                   (383, 129), (384, 128), (385, 127), (511, 255), (513, 256), (640, 257),
                   (384, 384), (385, 385), (63, 129), (129, 63)]


@pytest.mark.parametrize("steps,variant", [(1, 0), (5, 0), (5, 1)])
def test_ns_stage_and_tile_boundaries(dm, wl, steps, variant):
    """Shapes whose m and n fall just below, on and just above the multiples of
    64, 128 and 256 that the product kernel's boxes, stages and tiles use, in
    both orientations; with the Gram rule, the shapes it gives the Gram form are
    checked against the oracle's Gram iteration."""
    ps = PackedSet(dm, BOUNDARY_SHAPES, variant=variant)
    ins = []
    for i, s in enumerate(BOUNDARY_SHAPES):
        u = wl.random_matrix(s, 900 + i, "cuda", 1.0, torch.bfloat16)
        ps.view(i).copy_(u)
        ins.append(np64(u))
    run_ns(dm, ps, steps, variant=variant)
    assert ps.guards_intact()
    n_gram = 0
    for i, s in enumerate(BOUNDARY_SHAPES):
        gram = dm.ns_variant_for(s, steps, variant) == dm.NS_GRAM
        n_gram += gram
        ref = (oracle.gram_newton_schulz if gram else oracle.newton_schulz)(ins[i], steps)
        err = rel(np64(ps.view(i)), ref)
        assert err <= NS_TOL[steps], f"{s} steps={steps} gram={gram}: rel err {err:.3e}"
    if variant == dm.NS_GRAM:
        assert n_gram > 0


@pytest.mark.parametrize("steps", [0, 1])
def test_ns_eps_is_added_to_the_norm(dm, wl, steps):
    """With ||U|| ~ 1e-3 and eps = 1e-3, X0 = U / (||U|| + eps) is about half of
    U / ||U||: the GPU result must follow the oracle with that eps and differ
    clearly from the default eps."""
    shapes = [(64, 200), (300, 7), (256, 256)]
    ps = PackedSet(dm, shapes)
    ins = []
    for i, s in enumerate(shapes):
        u = wl.random_matrix(s, 400 + i, "cuda", 1.0, torch.float32)
        u = (u / u.norm() * 1e-3).to(torch.bfloat16)
        ps.view(i).copy_(u)
        ins.append(np64(u))
    dm.ns_batched(ps.shapes, ps.packed, ps.offsets, ps.workspace, ns_steps=steps, eps=1e-3,
                  ws_bytes=ps.ws_bytes)
    assert dm.stream_status(ps.workspace) == dm.OK
    for i, s in enumerate(shapes):
        got = np64(ps.view(i))
        ref = oracle.newton_schulz(ins[i], steps, eps=1e-3)
        default = oracle.newton_schulz(ins[i], steps)
        assert rel(got, ref) <= NS_TOL[steps], f"{s}: rel err {rel(got, ref):.3e}"
        assert rel(got, default) > 10 * NS_TOL[steps], f"{s}: eps had no effect"


def test_ns_phase_isolation(dm, wl):
    """abc = (1,0,0) returns X0; (0,1,0) gives X0 X0^T X0; (0,0,1) gives (X0 X0^T)^2 X0.
    Separates the symmetric products and the full product when one is wrong."""
    shapes = [(256, 1024), (1024, 256), (129, 257), (300, 7)]
    for abc in ((1.0, 0.0, 0.0), (0.0, 1.0, 0.0), (0.0, 0.0, 1.0)):
        ps = PackedSet(dm, shapes)
        ins = []
        for i, s in enumerate(shapes):
            u = wl.random_matrix(s, 7 + i, "cuda", 1.0, torch.bfloat16)
            ps.view(i).copy_(u)
            ins.append(np64(u))
        run_ns(dm, ps, 1, abc=abc)
        for i, s in enumerate(shapes):
            ref = oracle.newton_schulz(ins[i], 1, abc=abc)
            err = rel(np64(ps.view(i)), ref)
            assert err <= 2e-2, f"abc={abc} {s}: rel err {err:.3e}"


def test_ns_eight_steps_band(dm, wl):
    shapes = [(256, 1024), (512, 512)]
    ps = PackedSet(dm, shapes)
    ins = []
    for i, s in enumerate(shapes):
        u = wl.random_matrix(s, 300 + i, "cuda", 1.0, torch.bfloat16)
        ps.view(i).copy_(u)
        ins.append(np64(u))
    run_ns(dm, ps, 8)
    for i, s in enumerate(shapes):
        out = np64(ps.view(i))
        assert rel(out, oracle.newton_schulz(ins[i], 8)) <= NS_TOL[8]
        sv = np.linalg.svd(out, compute_uv=False)
        assert sv.max() <= 1.2025 * 1.02


def test_ns_deterministic(dm, wl):
    shapes = [(1000, 1000), (300, 7), (256, 1024)]
    outs = []
    for _ in range(2):
        ps = PackedSet(dm, shapes)
        for i, s in enumerate(shapes):
            ps.view(i).copy_(wl.random_matrix(s, 55 + i, "cuda", 1.0, torch.bfloat16))
        run_ns(dm, ps, 5)
        outs.append(ps.packed.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_ns_zero_matrix_gives_zero(dm):
    shapes = [(64, 200), (200, 64)]
    ps = PackedSet(dm, shapes)
    for i in range(2):
        ps.view(i).zero_()
    run_ns(dm, ps, 5)
    for i in range(2):
        assert not torch.any(ps.view(i).float() != 0)


@pytest.mark.parametrize("steps", [1, 3, 5])
def test_gram_variant(dm, wl, steps):
    shapes = [(128, 512), (512, 128), (200, 900), (900, 200), (64, 4096), (300, 300), (7, 300),
              (300, 7)]
    ps = PackedSet(dm, shapes, variant=dm.NS_GRAM)
    ins = []
    for i, s in enumerate(shapes):
        u = wl.random_matrix(s, 900 + i, "cuda", 1.0, torch.bfloat16)
        ps.view(i).copy_(u)
        ins.append(np64(u))
    run_ns(dm, ps, steps, variant=dm.NS_GRAM)
    assert ps.guards_intact()
    for i, s in enumerate(shapes):
        gram = dm.ns_variant_for(s, steps, dm.NS_GRAM) == dm.NS_GRAM
        ref = (oracle.gram_newton_schulz if gram else oracle.newton_schulz)(ins[i], steps)
        err = rel(np64(ps.view(i)), ref)
        assert err <= NS_TOL[steps], f"gram {s} steps={steps}: rel err {err:.3e}"


# ------------------------------------------------------------------ pack / update
@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16])
def test_pack_momentum(dm, wl, gdt):
    shapes = [(256, 1024), (300, 7), (7, 300), (1, 1), (129, 257)]
    ps = PackedSet(dm, shapes)
    grads = [wl.random_matrix(s, 40 + i, "cuda", 1e-3, gdt) for i, s in enumerate(shapes)]
    moms = [wl.random_matrix(s, 60 + i, "cuda", 1e-3, torch.float32) for i, s in enumerate(shapes)]
    m0 = [np64(m) for m in moms]
    dm.pack(shapes, grads, moms, 0.95, ps.packed, ps.offsets, ps.workspace)
    assert dm.stream_status(ps.workspace) == dm.OK
    assert ps.guards_intact()
    for i, s in enumerate(shapes):
        m_ref, u_ref = oracle.nesterov_momentum(np64(grads[i]), m0[i], 0.95)
        assert rel(np64(moms[i]), m_ref) <= 1e-5
        assert bf16_ulp_dist(ps.view(i), u_ref) <= 1


def test_pack_then_ns_uses_fp32_norm(dm, wl):
    shapes = [(256, 1024), (1024, 256)]
    ps = PackedSet(dm, shapes)
    grads = [wl.random_matrix(s, 70 + i, "cuda", 1.0, torch.float32) for i, s in enumerate(shapes)]
    moms = [torch.zeros(s, device="cuda") for s in shapes]
    dm.pack(shapes, grads, moms, 0.95, ps.packed, ps.offsets, ps.workspace)
    dm.ns_batched(shapes, ps.packed, ps.offsets, ps.workspace, ns_steps=0, use_pack_norms=True,
                  ws_bytes=ps.ws_bytes)
    assert dm.stream_status(ps.workspace) == dm.OK
    for i, s in enumerate(shapes):
        _, u = oracle.nesterov_momentum(np64(grads[i]), np.zeros(s), 0.95)
        assert rel(np64(ps.view(i)), oracle.newton_schulz(u, 0)) <= 5e-3


@pytest.mark.parametrize("wdt", [torch.float32, torch.bfloat16])
def test_unpack_update(dm, wl, wdt):
    shapes = [(256, 1024), (1024, 256), (300, 7), (3, 3)]
    ps = PackedSet(dm, shapes)
    for i, s in enumerate(shapes):
        ps.view(i).copy_(wl.random_matrix(s, 80 + i, "cuda", 0.03, torch.bfloat16))
    ws = [wl.random_matrix(s, 90 + i, "cuda", 0.02, wdt) for i, s in enumerate(shapes)]
    w0 = [np64(w) for w in ws]
    dm.unpack_update(shapes, ws, 0.02, ps.packed, ps.offsets, ps.workspace)
    assert dm.stream_status(ps.workspace) == dm.OK
    for i, s in enumerate(shapes):
        ref = oracle.apply_update(w0[i], np64(ps.view(i)), 0.02)
        if wdt == torch.float32:
            assert rel(np64(ws[i]) - w0[i], ref - w0[i]) <= 1e-5
        else:
            assert bf16_update_ok(ws[i], ref, w0[i], ref - w0[i])


# ------------------------------------------------------------------ whole step
def _muon_case(dm, wl, shapes, gdt, wdt, steps=2, variant=0, seed=0, ns_steps=5):
    """`steps` whole owner-side steps against the oracle, each step fed the
    GPU's weights from before it (so that every step is checked on its own)
    and the oracle's carried momentum.

    fp32 weights: dW = W' - W within the NS tolerance of the oracle's dW.
    bf16 weights: W' - W'_64 = (bf16 rounding of the result) + lr*s*(O_64 - O),
    so its norm is bounded by the rounding residual of RNE(W'_64) (25% slack
    for the other side of a rounding boundary) plus the NS tolerance on the
    update itself."""
    from newton_schulz_owner_gb300.dmuon import MuonOwner
    own = MuonOwner(shapes, variant=variant)
    ws = [wl.random_matrix(s, seed + 500 + i, "cuda", 0.02, wdt) for i, s in enumerate(shapes)]
    ms = [torch.zeros(s, device="cuda") for s in shapes]
    m_ref = [np.zeros(s) for s in shapes]
    worst = 0.0
    for step in range(steps):
        gs = [wl.random_matrix(s, seed + 1000 * step + i, "cuda", 1e-3 if gdt == torch.bfloat16
                               else 1.0, gdt) for i, s in enumerate(shapes)]
        w_before = [np64(w) for w in ws]
        own.step(gs, ms, ws, lr=0.02, beta=0.95, ns_steps=ns_steps)
        assert own.status() == dm.OK
        for i, s in enumerate(shapes):
            m_ref[i], o_ref, w_new = oracle.muon_step(
                np64(gs[i]), m_ref[i], w_before[i], lr=0.02, beta=0.95, ns_steps=ns_steps,
                variant="gram" if dm.ns_variant_for(s, ns_steps, variant) == dm.NS_GRAM
                else "standard")
            assert rel(np64(ms[i]), m_ref[i]) <= 1e-5, f"momentum {s}"
            err_o = rel(np64(own.packed_view(i)), o_ref)
            assert err_o <= NS_TOL[ns_steps], f"step {step} {s}: O rel err {err_o:.3e}"
            if wdt == torch.float32:
                err = rel(np64(ws[i]) - w_before[i], w_new - w_before[i])
                assert err <= NS_TOL[ns_steps], f"step {step} {s}: dW rel err {err:.3e}"
            else:
                resid = np.linalg.norm(oracle.round_bf16(w_new) - w_new)
                bound = 1.25 * resid + NS_TOL[ns_steps] * np.linalg.norm(w_new - w_before[i])
                dist = float(np.linalg.norm(np64(ws[i]) - w_new))
                assert dist <= bound, f"step {step} {s}: |W - W_64| {dist:.3e} > {bound:.3e}"
                err = dist / max(bound, 1e-30)
            worst = max(worst, err)
    return worst


def test_muon_step_single_256x1024_fp32(dm, wl):
    _muon_case(dm, wl, [(256, 1024)], torch.float32, torch.float32)


def test_muon_step_mixed_projection_set(dm, wl):
    shapes = [(256, 256), (64, 256), (64, 256), (256, 256), (700, 256), (700, 256), (256, 700)]
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.float32)


def test_muon_step_several_wide_and_tall_buckets(dm, wl):
    """Several wide and several tall buckets with ragged sizes: each product
    runs as one launch per run of same-orientation buckets, and the whole step
    pipelines over all buckets on two streams."""
    shapes = [(256, 700), (700, 256), (300, 900), (900, 300), (256, 256), (129, 520),
              (520, 129), (700, 256), (64, 1000), (1000, 64)]
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.float32, seed=17)


def test_muon_step_bf16_weights_ragged_buckets(dm, wl):
    """bf16 gradients and bf16 weights over several ragged wide and tall
    buckets (the pipelined whole step), two steps with carried momentum."""
    shapes = [(129, 520), (520, 129), (300, 900), (900, 300), (257, 257), (64, 1000),
              (1000, 64), (7, 300)]
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.bfloat16, seed=23)


@pytest.mark.parametrize("variant", [0, 1])
def test_nan_and_inf_propagate_to_their_own_matrix_only(dm, wl, variant):
    """A NaN in one gradient and an Inf in another: those two matrices' O and
    W become NaN everywhere, exactly as in the oracle (X0 = U/||U|| is NaN at
    the bad element, and every product spreads it over the whole matrix); the
    momentum keeps the bad value at its element only; every other matrix of the
    same call, in the same buckets, matches the oracle as usual.  With the Gram
    rule the rectangular matrices take the Gram form, whose products spread the
    bad value the same way."""
    shapes = [(256, 700), (256, 700), (256, 700), (700, 256), (700, 256), (300, 300)]
    own = dm.MuonOwner(shapes, variant=variant)
    ws = [wl.random_matrix(s, 1500 + i, "cuda", 0.02, torch.bfloat16) for i, s in enumerate(shapes)]
    ms = [torch.zeros(s, device="cuda") for s in shapes]
    gs = [wl.random_matrix(s, 1600 + i, "cuda", 1e-3, torch.bfloat16) for i, s in enumerate(shapes)]
    gs[1][17, 301] = float("nan")
    gs[3][600, 5] = float("inf")
    w0 = [np64(w) for w in ws]
    own.step(gs, ms, ws, lr=0.02, beta=0.95, ns_steps=5)
    assert own.status() == dm.OK
    n_gram = 0
    for i, s in enumerate(shapes):
        gram = dm.ns_variant_for(s, 5, variant) == dm.NS_GRAM
        n_gram += gram
        m_ref, o_ref, w_ref = oracle.muon_step(np64(gs[i]), np.zeros(s), w0[i], lr=0.02,
                                               beta=0.95, ns_steps=5,
                                               variant="gram" if gram else "standard")
        m_gpu, o_gpu, w_gpu = np64(ms[i]), np64(own.packed_view(i)), np64(ws[i])
        if i in (1, 3):
            assert np.isnan(o_ref).all() and np.isnan(w_ref).all()
            assert np.isnan(o_gpu).all(), f"#{i}: O not NaN everywhere"
            assert np.isnan(w_gpu).all(), f"#{i}: W not NaN everywhere"
            bad = ~np.isfinite(m_ref)
            assert bad.sum() == 1
            assert np.array_equal(~np.isfinite(m_gpu), bad)
            assert np.array_equal(np.isnan(m_gpu), np.isnan(m_ref))
            assert rel(m_gpu[~bad], m_ref[~bad]) <= 1e-5
        else:
            assert np.isfinite(o_gpu).all() and np.isfinite(w_gpu).all(), f"#{i} touched"
            assert rel(m_gpu, m_ref) <= 1e-5
            assert rel(o_gpu, o_ref) <= NS_TOL[5], f"#{i}: O rel err {rel(o_gpu, o_ref):.3e}"
    assert n_gram == (5 if variant == 1 else 0)


def test_two_owners_on_two_streams_run_concurrently_and_match(dm, wl):
    """Two owners with different matrices step on two caller streams at once
    (each with its own companion stream); the results equal the same steps
    run one owner after the other on one stream, bit for bit."""
    sets = [[(256, 700), (700, 256), (300, 300)], [(512, 128), (128, 512), (257, 520)]]

    def run(concurrent):
        owners = [dm.MuonOwner(sh) for sh in sets]
        W = [[wl.random_matrix(s, 2000 + 10 * k + i, "cuda", 0.02, torch.bfloat16)
              for i, s in enumerate(sh)] for k, sh in enumerate(sets)]
        M = [[torch.zeros(s, device="cuda") for s in sh] for sh in sets]
        G = [[[wl.random_matrix(s, 3000 * (step + 1) + 10 * k + i, "cuda", 1e-3, torch.bfloat16)
               for i, s in enumerate(sh)] for k, sh in enumerate(sets)] for step in range(2)]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()] if concurrent else \
            [torch.cuda.current_stream()] * 2
        torch.cuda.synchronize()
        # both owners' steps are enqueued back to back, with no host wait between
        for step in range(2):
            for k in range(2):
                with torch.cuda.stream(streams[k]):
                    owners[k].step(G[step][k], M[k], W[k], lr=0.02, beta=0.95, ns_steps=5,
                                   stream=streams[k])
        torch.cuda.synchronize()
        for k in range(2):
            assert owners[k].status(streams[k]) == dm.OK
        return [[w.clone() for w in wk] for wk in W], [[m.clone() for m in mk] for mk in M]

    Wc, Mc = run(True)
    Ws, Ms = run(False)
    for k in range(2):
        for a, b in zip(Wc[k], Ws[k]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        for a, b in zip(Mc[k], Ms[k]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("ns_steps", [0, 1, 2, 8])
def test_muon_step_other_step_counts(dm, wl, ns_steps):
    """The pipelined step places its memory-bound pieces by product launch, and
    the launches per bucket follow the step count: a ragged multi-bucket step
    at 1, 2 and 8 Newton-Schulz steps, against the oracle; and at 0 steps (no
    products: O is the normalised U, and the step runs its three parts in
    turn)."""
    shapes = [(256, 700), (700, 256), (300, 900), (900, 300), (256, 256), (64, 1000)]
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.float32, steps=1, seed=29,
               ns_steps=ns_steps)


@pytest.mark.parametrize("ns_steps", [3, 8])
def test_muon_step_gram_variant_other_step_counts(dm, wl, ns_steps):
    """The Gram form's positions in the pipelined step (their launch count
    depends on the step count), next to standard ones."""
    shapes = [(256, 256), (64, 256), (700, 256), (256, 700), (300, 900)]
    assert any(dm.ns_variant_for(s, ns_steps, dm.NS_GRAM) == dm.NS_GRAM for s in shapes)
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.float32, steps=1, variant=1, seed=31,
               ns_steps=ns_steps)


def test_muon_step_gram_variant(dm, wl):
    shapes = [(256, 256), (64, 256), (700, 256), (256, 700)]
    _muon_case(dm, wl, shapes, torch.bfloat16, torch.float32, variant=1)


# ------------------------------------------------------------------ failure path
def test_bounded_wait_timeout_is_reported_and_context_survives(dm, wl):
    ps = PackedSet(dm, [(64, 128)])
    dm.debug_wait_timeout(ps.workspace, 2000)
    assert dm.stream_status(ps.workspace) == dm.ERR_TIMEOUT
    assert dm.stream_status(ps.workspace) == dm.OK     # cleared once read
    u = wl.random_matrix((64, 128), 3, "cuda", 1.0, torch.bfloat16)
    ps.view(0).copy_(u)
    run_ns(dm, ps, 5)
    assert rel(np64(ps.view(0)), oracle.newton_schulz(np64(u), 5)) <= 2e-2
