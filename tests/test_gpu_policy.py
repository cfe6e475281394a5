"""The Newton-Schulz variant rule, measured and checked on the GPU.

The DMuon home page names Gram Newton-Schulz ("VLA and VLM"; closing credits)
but gives no rule for when to use it.  The library's rule (dmuon_ns_variant_for)
uses the Gram form only where it saves work and, by step count, only from an
aspect ratio n/m upward at which the bf16 Gram iteration stays within the
Newton-Schulz tolerance.  This test measures that error directly: every shape
of a grid of aspect ratios (wide and tall, two sizes, seeded Gaussian inputs
as in the benchmark workloads) runs through the C ABI with the Gram form
forced on (DMUON_NS_GRAM_ALL), with the standard form, and with the rule
(DMUON_NS_GRAM), at several step counts, against the fp64 oracle.

The grid is the one the rule's bands were calibrated on.  Checked: wherever
the rule picks Gram, the forced-Gram error is below 0.9 x the tolerance (the
rule is safe); every result of the rule's call is within the tolerance of the
oracle, and so is the standard form at every step count; the model projection
sets' MLP and k/v shapes (aspect 2.67-7) get the Gram form at 3, 5 and 8 steps;
and a call with exactly dmuon_workspace_bytes succeeds at every step count.
Run with `-s` to print the measured table.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

# aspect ratios n/m: a grid plus those of the model projection sets' matrices
# (Llama-3.2-3B MLP 2.67, Llama-3.1-8B MLP 3.5, Qwen2.5-7B MLP 5.29, Qwen2.5-1.5B
# MLP 5.83, Qwen2.5-1.5B k/v 6, Qwen2.5-7B k/v 7)
RATIOS = [1.25, 1.5, 1.75, 2.0, 2.5, 2.67, 3.0, 3.5, 4.0, 5.29, 5.83, 7.0, 8.0]
STEPS = [2, 3, 4, 5, 6, 7, 8, 9, 10]
SIZES = [(256, True), (448, True), (1024, False)]   # (m, also the tall orientation)
MARGIN = 0.9     # the rule may pick Gram only where its error is below 0.9 x tolerance


def tol(k):
    return 2e-2 if k <= 5 else 4e-2


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


def shapes():
    """(shape, m, ratio) of every grid point."""
    out = []
    for m, tall in SIZES:
        for r in RATIOS:
            n = int(round(r * m))
            out.append(((m, n), m, r))
            if tall:
                out.append(((n, m), m, r))
    return out


def run(dm, shp, ins, steps, variant):
    _, off, oel = dm.plan(shp)
    packed = torch.zeros(max(sum(oel), 128), dtype=torch.bfloat16, device="cuda")
    for i, (r, c) in enumerate(shp):
        packed[off[i]:off[i] + r * c].view(r, c).copy_(ins[i])
    ws = torch.zeros(dm.workspace_bytes(shp, variant), dtype=torch.uint8, device="cuda")
    dm.ns_batched(shp, packed, off, ws, ns_steps=steps, variant=variant)
    assert dm.stream_status(ws) == dm.OK
    return [packed[off[i]:off[i] + r * c].view(r, c).double().cpu().numpy()
            for i, (r, c) in enumerate(shp)]


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_gram_rule_against_measured_error(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    grid = shapes()
    shp = [g[0] for g in grid]
    ins = [wl.random_matrix(s, 7000 + i, "cuda", 1.0, torch.bfloat16) for i, s in enumerate(shp)]
    ins64 = [u.double().cpu().numpy() for u in ins]
    worst = {}   # (m, ratio, steps) -> (forced-Gram error, standard error, rule error, rule pick)
    bad = []
    for k in STEPS:
        out_all = run(dm, shp, ins, k, dm.NS_GRAM_ALL)
        out_std = run(dm, shp, ins, k, dm.NS_STANDARD)
        out_pol = run(dm, shp, ins, k, dm.NS_GRAM)
        for i, s in enumerate(shp):
            ref = oracle.newton_schulz(ins64[i], k)
            e_all, e_std, e_pol = rel(out_all[i], ref), rel(out_std[i], ref), rel(out_pol[i], ref)
            pick = dm.ns_variant_for(s, k, dm.NS_GRAM)
            key = (grid[i][1], grid[i][2], k)
            w = worst.get(key, (0.0, 0.0, 0.0, pick))
            worst[key] = (max(w[0], e_all), max(w[1], e_std), max(w[2], e_pol), pick)
            if e_pol > tol(k):
                bad.append(f"{s} steps={k}: the rule's result is off by {e_pol:.3e}")
            if e_std > tol(k):
                bad.append(f"{s} steps={k}: standard off by {e_std:.3e}")
            if pick == dm.NS_GRAM and e_all > MARGIN * tol(k):
                bad.append(f"{s} steps={k}: the rule picks Gram but its error is {e_all:.3e}")
    print("\n     m  aspect  steps  gram_forced  standard      rule  rule_pick")
    for (m, r, k), (ea, es, ep, pick) in sorted(worst.items()):
        print(f"{m:6d} {r:7.2f} {k:6d}  {ea:11.3e}  {es:8.3e}  {ep:8.3e}  "
              f"{'gram' if pick == dm.NS_GRAM else 'standard'}")
    assert not bad, "\n".join(bad)
    # the projection sets' MLP and k/v matrices (n/m = 2.67 .. 7) take the Gram
    # form at 3, 5 and 8 steps; their square q/o matrices keep the standard form
    for k in (3, 5, 8):
        for s in ((14336, 4096), (3584, 18944), (8960, 1536), (8192, 3072), (1024, 4096),
                  (512, 3584), (256, 1536), (1024, 3072)):
            assert dm.ns_variant_for(s, k, dm.NS_GRAM) == dm.NS_GRAM, (s, k)
        assert dm.ns_variant_for((4096, 4096), k, dm.NS_GRAM) == dm.NS_STANDARD


def test_pack_then_gram_call_reads_its_own_norms(dm):
    """dmuon_pack plans every matrix as standard; a following Gram call plans
    some as Gram, which reorders its buckets.  The norm partial sums must
    still be found per matrix: here the first matrix goes Gram (so it moves
    behind the square one in the Gram call's bucket order)."""
    from newton_schulz_owner_gb300 import workloads as wl
    shp = [(128, 700), (300, 300), (700, 128), (256, 256), (64, 900)]
    assert dm.ns_variant_for(shp[0], 5, dm.NS_GRAM) == dm.NS_GRAM
    _, off, oel = dm.plan(shp)
    packed = torch.zeros(sum(oel), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(dm.workspace_bytes(shp, dm.NS_GRAM), dtype=torch.uint8, device="cuda")
    grads = [wl.random_matrix(s, 8100 + i, "cuda", 1.0, torch.float32) for i, s in enumerate(shp)]
    moms = [torch.zeros(s, device="cuda") for s in shp]
    dm.pack(shp, grads, moms, 0.95, packed, off, ws)
    dm.ns_batched(shp, packed, off, ws, ns_steps=5, variant=dm.NS_GRAM, use_pack_norms=True)
    assert dm.stream_status(ws) == dm.OK
    for i, (r, c) in enumerate(shp):
        _, u = oracle.nesterov_momentum(grads[i].double().cpu().numpy(), np.zeros((r, c)), 0.95)
        got = packed[off[i]:off[i] + r * c].view(r, c).double().cpu().numpy()
        err = rel(got, oracle.newton_schulz(u, 5))
        assert err <= 2e-2, f"{(r, c)}: rel err {err:.3e}"
