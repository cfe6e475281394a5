"""GPU parity of dmuon_adamw (AdamW for the parameters Muon does not own)
against the fp64 oracle, through the C ABI.

Tolerances: moments and fp32 parameter changes <= 1e-5 relative Frobenius
(fp32 arithmetic); bf16 parameters within 1 bf16 ulp of RNE(fp64), or within
fp32 rounding of the operands where the update cancels to about zero."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

SIZES = [(1,), (7,), (8192,), (8193,), (33, 65), (4096,), (0,), (128256, 16)]


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


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def rel(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


@pytest.mark.parametrize("pdt,gdt", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                     (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("misaligned", [False, True])
def test_adamw_matches_oracle_over_three_steps(dm, pdt, gdt, misaligned):
    from newton_schulz_owner_gb300 import workloads as wl
    gen = torch.Generator(device="cuda").manual_seed(5)
    off = 1 if misaligned else 0     # views one element in: scalar path
    def mk(shape, std, dtype):
        n = int(np.prod(shape))
        base = torch.randn(n + off, generator=gen, device="cuda").mul_(std).to(dtype)
        return base[off:].view(shape)
    ps = [mk(s, 0.02, pdt) for s in SIZES]
    ms = [mk(s, 0.0, torch.float32).zero_() for s in SIZES]
    vs = [mk(s, 0.0, torch.float32).zero_() for s in SIZES]
    ref_p = [np64(p) for p in ps]
    ref_m = [np.zeros(s) for s in SIZES]
    ref_v = [np.zeros(s) for s in SIZES]
    ws = torch.zeros(dm.adamw_workspace_bytes(len(SIZES)), dtype=torch.uint8, device="cuda")
    for t in range(1, 4):
        gs = [mk(s, 1e-2, gdt) for s in SIZES]
        p_before = [np64(p) for p in ps]
        dm.adamw(ps, gs, ms, vs, t, ws, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
        assert dm.stream_status(ws) == dm.OK
        for i, s in enumerate(SIZES):
            if int(np.prod(s)) == 0:
                continue
            # the oracle runs from the GPU's own previous state, isolating this step
            rp, rm, rv = oracle.adamw_step(p_before[i], np64(gs[i]), ref_m[i], ref_v[i], t)
            assert rel(np64(ms[i]), rm) <= 1e-5, f"m {s} t={t}"
            assert rel(np64(vs[i]), rv) <= 1e-5, f"v {s} t={t}"
            if pdt == torch.float32:
                assert rel(np64(ps[i]) - p_before[i], rp - p_before[i]) <= 1e-5, f"p {s} t={t}"
            else:
                ref = torch.from_numpy(oracle.round_bf16(rp)).to(torch.bfloat16)
                a = ps[i].detach().cpu().view(torch.int16).to(torch.int32)
                b = ref.view(torch.int16).to(torch.int32)
                a = torch.where(a < 0, -(a & 0x7FFF), a)
                b = torch.where(b < 0, -(b & 0x7FFF), b)
                ulps = (a - b).abs().numpy()
                diff = np.abs(np64(ps[i]) - rp)
                ok = (ulps <= 1) | (diff <= 2.0 ** -22 * (np.abs(p_before[i]) + 1e-3))
                assert ok.all(), f"p bf16 {s} t={t}"
            ref_m[i], ref_v[i] = np64(ms[i]), np64(vs[i])


def test_adamw_argument_errors(dm):
    import ctypes
    lib = dm.lib()
    ws = torch.zeros(dm.adamw_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    p = torch.zeros(8, device="cuda")
    ptr = (ctypes.c_void_p * 1)(p.data_ptr())
    ptrf = ctypes.cast(ptr, ctypes.POINTER(ctypes.c_void_p))
    n = dm._i64([8])
    args = lambda step, b1, ws_bytes: lib.dmuon_adamw(1, n, ptr, dm.F32, ptr, dm.F32, ptrf, ptrf,
                                                      1e-3, b1, 0.999, 1e-8, 0.01, step,
                                                      ws.data_ptr(), ws_bytes, None)
    assert args(0, 0.9, ws.numel()) == dm.ERR_INVALID_ARG        # step counts from 1
    assert args(1, 1.0, ws.numel()) == dm.ERR_INVALID_ARG        # beta1 must be < 1
    assert args(1, 0.9, 16) == dm.ERR_WORKSPACE
