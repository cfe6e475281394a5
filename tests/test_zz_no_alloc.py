"""The allocation-free Newton-Schulz call, dmuon_ns_batched_noalloc.

Some callers cannot allocate device memory: a host framework that owns every
device allocation, a plugin that may only touch the buffers it is handed, or a
latency-critical loop that cannot afford cudaMalloc's implicit
synchronisation.  For them the library keeps a fixed scratch array of its own.

These tests call that entry point through the C ABI and check that
  * on two calls in a row -- the second with other shapes and other values, so
    that anything left over from the first call in the shared array would
    change its result -- the output is bit for bit the output of
    dmuon_ns_batched (the same kernels on a caller workspace), and every matrix
    is within the Newton-Schulz tolerance of the fp64 oracle;
  * a bounded device wait that gives up on the array's error word is reported
    by dmuon_noalloc_status, cleared once read, and leaves the call usable;
  * a problem too large for the array is refused before anything runs.
This file is collected last on purpose, and each test also passes when it runs
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2   # bf16-operand Newton-Schulz, 5 steps: relative Frobenius per matrix
# The second list reuses some working shapes of the first (same slots, other
# values) and adds others, so the second call's tables and buffers are laid out
# over what the first call left in the array.
CALLS = [
    (31, [(256, 1024), (300, 7), (129, 257), (64, 64), (1, 5)]),
    (57, [(129, 257), (700, 300), (256, 1024), (5, 1), (64, 64), (1000, 96)]),
]


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
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _noalloc(dm, shapes, packed, offsets, stream, ns_steps=5):
    return dm.lib().dmuon_ns_batched_noalloc(len(shapes), dm._shapes(shapes), packed.data_ptr(),
                                             dm._i64(offsets), ns_steps, dm.NS_STANDARD, None,
                                             ctypes.c_float(1e-7), stream)


def test_noalloc_equals_workspace_call_bit_for_bit_on_two_calls_in_a_row(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    stream = torch.cuda.current_stream().cuda_stream
    for call, (seed, shapes) in enumerate(CALLS):
        _, offsets, owner_elems = dm.plan(shapes)
        total = sum(owner_elems)
        ws = torch.zeros(dm.workspace_bytes(shapes), dtype=torch.uint8, device="cuda")
        ref = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        ins = []
        for i, (r, c) in enumerate(shapes):
            u = wl.random_matrix((r, c), seed + i, "cuda", 1.0, torch.bfloat16)
            ref[offsets[i]:offsets[i] + r * c].view(r, c).copy_(u)
            ins.append(u.double().cpu().numpy())
        out = ref.clone()
        dm.ns_batched(shapes, ref, offsets, ws, ns_steps=5)
        assert dm.stream_status(ws) == dm.OK
        st = _noalloc(dm, shapes, out, offsets, stream)
        assert st == dm.OK, dm.status_string(st)
        assert dm.noalloc_status() == dm.OK
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"call {call}: the allocation-free result differs from dmuon_ns_batched"
        for i, (r, c) in enumerate(shapes):
            got = out[offsets[i]:offsets[i] + r * c].view(r, c).double().cpu().numpy()
            err = _rel(got, oracle.newton_schulz(ins[i], 5))
            assert err <= NS_TOL, f"call {call} matrix {i} {(r, c)}: rel err {err:.3e}"


def test_noalloc_reports_a_device_timeout_and_stays_usable(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    stream = torch.cuda.current_stream().cuda_stream
    dm.debug_wait_timeout(None, 2000)          # a wait on the array's error word runs out
    assert dm.noalloc_status() == dm.ERR_TIMEOUT
    assert dm.noalloc_status() == dm.OK        # cleared once read
    shapes = [(64, 128)]
    u = wl.random_matrix((64, 128), 3, "cuda", 1.0, torch.bfloat16)
    packed = torch.zeros(64 * 128, dtype=torch.bfloat16, device="cuda")
    packed.view(64, 128).copy_(u)
    assert _noalloc(dm, shapes, packed, [0], stream) == dm.OK
    assert dm.noalloc_status() == dm.OK
    err = _rel(packed.view(64, 128).double().cpu().numpy(),
               oracle.newton_schulz(u.double().cpu().numpy(), 5))
    assert err <= NS_TOL


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


def test_noalloc_gram_variant_equals_workspace_call(dm):
    """The same call with the Gram variant: the rule gives the rectangular
    matrices the Gram form and the square one the standard form, in the built-in
    array exactly as in a caller workspace (bit for bit), each within the
    tolerance of the oracle's form for it."""
    from newton_schulz_owner_gb300 import workloads as wl
    shapes = [(128, 512), (512, 128), (200, 700), (256, 256), (96, 900)]
    assert dm.ns_variant_for((128, 512), 5, dm.NS_GRAM) == dm.NS_GRAM
    _, offsets, owner_elems = dm.plan(shapes)
    assert dm.workspace_bytes(shapes, dm.NS_GRAM) <= dm.NOALLOC_SCRATCH_BYTES
    ws = torch.zeros(dm.workspace_bytes(shapes, dm.NS_GRAM), dtype=torch.uint8, device="cuda")
    ref = torch.zeros(sum(owner_elems), dtype=torch.bfloat16, device="cuda")
    ins = []
    for i, (r, c) in enumerate(shapes):
        u = wl.random_matrix((r, c), 77 + i, "cuda", 1.0, torch.bfloat16)
        ref[offsets[i]:offsets[i] + r * c].view(r, c).copy_(u)
        ins.append(u.double().cpu().numpy())
    out = ref.clone()
    dm.ns_batched(shapes, ref, offsets, ws, ns_steps=5, variant=dm.NS_GRAM)
    assert dm.stream_status(ws) == dm.OK
    stream = torch.cuda.current_stream().cuda_stream
    st = dm.lib().dmuon_ns_batched_noalloc(len(shapes), dm._shapes(shapes), out.data_ptr(),
                                           dm._i64(offsets), 5, dm.NS_GRAM, None,
                                           ctypes.c_float(1e-7), stream)
    assert st == dm.OK, dm.status_string(st)
    assert dm.noalloc_status() == dm.OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    for i, (r, c) in enumerate(shapes):
        gram = dm.ns_variant_for((r, c), 5, dm.NS_GRAM) == dm.NS_GRAM
        want = (oracle.gram_newton_schulz if gram else oracle.newton_schulz)(ins[i], 5)
        got = out[offsets[i]:offsets[i] + r * c].view(r, c).double().cpu().numpy()
        err = _rel(got, want)
        assert err <= NS_TOL, f"{(r, c)} gram={gram}: rel err {err:.3e}"
