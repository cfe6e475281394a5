"""Newton-Schulz at the library's size limits.

DMUON_MAX_M (32768) bounds the short side of a matrix and DMUON_MAX_N (1048576)
the long side; at those sizes the fp64 oracle cannot run the dense iteration in
a test.  The inputs here are scaled partial permutations instead:
U = sum_k v_k e_{r_k} e_{c_k}^T with m distinct random rows r_k and columns c_k.
Their singular values are |v_k| with the unit vectors as singular vectors, so
the Newton-Schulz image keeps the pattern, each value becoming
sign(v_k) * p^steps(|v_k| / (||v|| + eps)) (p the quintic), and every other
element stays exactly zero: a product of zero rows and columns is zero, and
the diagonal shift of B only meets rows of X that are zero.  The oracle gives
each scalar through its own 1 x 1 iteration, on an input x whose normalisation
x / (|x| + eps) equals that ratio.  The nonzeros fall in random tiles, so the
check covers the tile indexing, strides and tensor-map coordinates of the
largest launches the library accepts, in both orientations.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

CASES = [(32768, 32768), (32768, 40000), (40000, 32768), (64, 1048576), (1048576, 64)]
STEPS = 5
TOL = 2e-2   # the Newton-Schulz tolerance on the pattern's values (bf16 operands)


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


def expected_values(v: np.ndarray, steps: int) -> np.ndarray:
    """sign(v) * p^steps(|v| / (||v|| + eps)) from the oracle's 1 x 1 iteration."""
    eps = oracle.NS_EPS
    y = np.abs(v) / (np.linalg.norm(v) + eps)
    out = np.empty_like(v)
    for k, (yk, vk) in enumerate(zip(y, v)):
        x = yk * eps / (1.0 - yk)          # x / (|x| + eps) == yk
        out[k] = np.sign(vk) * float(oracle.newton_schulz(np.array([[x]]), steps)[0, 0])
    return out


@pytest.mark.timeout(900)
@pytest.mark.parametrize("shape", CASES)
def test_partial_permutation_at_the_size_limits(dm, shape):
    r, c = shape
    m = min(r, c)
    assert max(r, c) <= dm.MAX_N and m <= dm.MAX_M
    g = torch.Generator().manual_seed(r * 7 + c)
    rows = torch.randperm(r, generator=g)[:m]
    cols = torch.randperm(c, generator=g)[:m]
    mag = 0.25 + torch.rand(m, generator=g, dtype=torch.float64)
    sgn = torch.where(torch.rand(m, generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    v = (mag * sgn).to(torch.bfloat16)       # the exact values the GPU sees

    shapes = [shape]
    _, offsets, owner_elems = dm.plan(shapes)
    packed = torch.zeros(owner_elems[0], dtype=torch.bfloat16, device="cuda")
    U = packed[offsets[0]:offsets[0] + r * c].view(r, c)
    rows_d, cols_d = rows.cuda(), cols.cuda()
    U[rows_d, cols_d] = v.cuda()
    ws = torch.zeros(dm.workspace_bytes(shapes), dtype=torch.uint8, device="cuda")
    dm.ns_batched(shapes, packed, offsets, ws, ns_steps=STEPS)
    assert dm.stream_status(ws) == dm.OK

    want = expected_values(v.double().numpy(), STEPS)
    got = U[rows_d, cols_d].double().cpu().numpy()
    err = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    assert err <= TOL, f"{shape}: pattern values rel err {err:.3e}"
    # nothing outside the pattern: the output's whole mass sits on it
    total = 0.0
    for r0 in range(0, r, 4096):
        total += float(U[r0:r0 + 4096].float().pow(2).sum(dtype=torch.float64))
    on_pattern = float((U[rows_d, cols_d].double() ** 2).sum())
    assert total == pytest.approx(on_pattern, rel=1e-6), \
        f"{shape}: {total - on_pattern:.3e} of squared mass outside the pattern"
    del packed, ws
    torch.cuda.empty_cache()
