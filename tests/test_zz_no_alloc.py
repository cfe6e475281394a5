"""The allocation-free Newton-Schulz call, dmuon_ns_batched_noalloc.

Some callers cannot allocate device memory: a host framework that owns every
device allocation, a plugin that may only touch the buffers it is handed, or a
latency-critical loop that cannot afford cudaMalloc's implicit
synchronisation.  For them the library keeps a fixed scratch array of its own.
These tests call that entry point through the C ABI and check it against
dmuon_ns_batched (which runs on a caller workspace) on two calls in a row with
different inputs, so the second call runs on scratch that still holds the
first call's data; and they check that a problem too large for the array is
refused before anything runs.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2   # bf16-operand Newton-Schulz, 5 steps: relative Frobenius per matrix
SHAPES = [(256, 1024), (300, 7), (129, 257), (64, 64), (1, 5)]


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


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_noalloc_matches_workspace_call_on_two_calls_in_a_row(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    _, offsets, owner_elems = dm.plan(SHAPES)
    total = sum(owner_elems)
    ws = torch.zeros(dm.workspace_bytes(SHAPES), dtype=torch.uint8, device="cuda")
    lib = dm.lib()
    for call, seed in enumerate((31, 57)):
        ref = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        for i, (r, c) in enumerate(SHAPES):
            ref[offsets[i]:offsets[i] + r * c].view(r, c).copy_(
                wl.random_matrix((r, c), seed + i, "cuda", 1.0, torch.bfloat16))
        out = ref.clone()
        dm.ns_batched(SHAPES, ref, offsets, ws, ns_steps=5)
        stream = torch.cuda.current_stream().cuda_stream
        st = lib.dmuon_ns_batched_noalloc(len(SHAPES), dm._shapes(SHAPES), out.data_ptr(),
                                          dm._i64(offsets), 5, dm.NS_STANDARD, None,
                                          ctypes.c_float(1e-7), stream)
        assert st == dm.OK, dm.status_string(st)
        torch.cuda.synchronize()
        assert dm.stream_status(ws) == dm.OK
        for i, (r, c) in enumerate(SHAPES):
            a = out[offsets[i]:offsets[i] + r * c]
            b = ref[offsets[i]:offsets[i] + r * c]
            err = _rel(a, b)
            assert err <= NS_TOL, f"call {call} matrix {i} {(r, c)}: rel err {err:.3e}"


def test_noalloc_refuses_problems_beyond_its_scratch(dm):
    big = [(4096, 4096)]
    assert dm.workspace_bytes(big) > dm.NOALLOC_SCRATCH_BYTES
    packed = torch.zeros(4096 * 4096, dtype=torch.bfloat16, device="cuda")
    before = packed.clone()
    st = dm.lib().dmuon_ns_batched_noalloc(1, dm._shapes(big), packed.data_ptr(), dm._i64([0]),
                                           5, dm.NS_STANDARD, None, ctypes.c_float(1e-7), None)
    assert st == dm.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(packed, before)
