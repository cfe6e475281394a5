"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, plans owners/offsets exactly like the oracle, sizes its workspace, and
rejects bad arguments before touching a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dmuon.h")


@pytest.fixture(scope="module")
def dm():
    from newton_schulz_owner_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from newton_schulz_owner_gb300 import dmuon
    return dmuon


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dmuon_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("dmuon_plan", "dmuon_workspace_bytes", "dmuon_pack", "dmuon_ns_batched",
              "dmuon_muon_step", "dmuon_stream_status", "dmuon_status_string"):
        assert f in names


def test_library_exports_every_declared_symbol(dm):
    lib = ctypes.CDLL(dm.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(dm.EXPORTED)


def test_status_strings_and_version(dm):
    assert dm.status_string(0) == "ok"
    assert "timed out" in dm.status_string(dm.ERR_TIMEOUT)
    assert dm.version() >= 100


SHAPE_SETS = [
    [(7, 300), (256, 1536), (1, 1), (64, 64), (300, 7), (5, 129)] * 3,
    [(1536, 1536), (256, 1536), (256, 1536), (1536, 1536), (8960, 1536), (8960, 1536), (1536, 8960)],
    [(3, 3)],
    [(0, 5), (4, 4), (5, 0)],
]


@pytest.mark.parametrize("shapes", SHAPE_SETS)
@pytest.mark.parametrize("n_owners", [1, 2, 3, 8])
def test_plan_matches_oracle_exactly(dm, shapes, n_owners):
    own, off, oel = dm.plan(shapes, n_owners)
    o_own, o_off, o_oel = oracle.pack_plan(shapes, n_owners)
    assert own == o_own and off == o_off and oel == o_oel


def test_plan_llama_3b_eight_owners_balanced(dm):
    from newton_schulz_owner_gb300 import workloads as wl
    w = wl.WORKLOADS["llama-3.2-3b"]
    shapes = w.shapes()
    own, off, oel = dm.plan(shapes, 8)
    assert (own, off, oel) == oracle.pack_plan(shapes, 8)
    loads = [sum(r * c for (r, c), o in zip(shapes, own) if o == k) for k in range(8)]
    assert max(loads) - min(loads) <= max(r * c for r, c in shapes)


def test_workspace_bytes(dm):
    shapes = [(256, 1024), (1024, 256), (7, 300)]
    a = dm.workspace_bytes(shapes, dm.NS_STANDARD)
    g = dm.workspace_bytes([(256, 1024), (1024, 256)], dm.NS_GRAM)
    assert a > 2 * 2 * (256 * 1024 + 1024 * 256)  # two X buffers at least
    assert g > 0
    assert dm.workspace_bytes(shapes, 7) == 0          # bad variant
    assert dm.workspace_bytes([(-1, 3)], 0) == 0       # bad shape
    assert dm.workspace_bytes([(40000, 40000)], 0) == 0  # beyond DMUON_MAX_M


def _raw_ns(dm, n, shapes, packed, offsets, steps, variant, ws, ws_bytes, abc=None):
    lib = dm.lib()
    sh = dm._shapes(shapes)
    off = dm._i64(offsets) if offsets is not None else None
    return lib.dmuon_ns_batched(n, sh, packed, off, steps, variant, abc, 1e-7, 0, ws, ws_bytes,
                                None)


def test_argument_errors_return_before_any_launch(dm):
    shapes = [(256, 1024)]
    need = dm.workspace_bytes(shapes)
    P, W = 1 << 20, 1 << 24     # fake, 256-aligned addresses: never dereferenced
    assert _raw_ns(dm, 1, shapes, P, [0], -1, 0, W, need) == dm.ERR_INVALID_ARG
    assert _raw_ns(dm, 1, shapes, P, [0], 5, 9, W, need) == dm.ERR_INVALID_ARG
    assert _raw_ns(dm, 1, shapes, P + 2, [0], 5, 0, W, need) == dm.ERR_ALIGNMENT
    assert _raw_ns(dm, 1, shapes, P, [0], 5, 0, W + 16, need) == dm.ERR_ALIGNMENT
    assert _raw_ns(dm, 1, shapes, P, [64], 5, 0, W, need) == dm.ERR_ALIGNMENT
    assert _raw_ns(dm, 1, shapes, P, [0], 5, 0, W, need - 1) == dm.ERR_WORKSPACE
    assert _raw_ns(dm, 1, shapes, None, [0], 5, 0, W, need) == dm.ERR_INVALID_ARG
    assert _raw_ns(dm, 1, shapes, P, None, 5, 0, W, need) == dm.ERR_INVALID_ARG
    assert _raw_ns(dm, 1, [(-3, 4)], P, [0], 5, 0, W, need) == dm.ERR_INVALID_ARG
    nan_abc = (ctypes.c_float * 3)(float("nan"), 0.0, 0.0)
    assert _raw_ns(dm, 1, shapes, P, [0], 5, 0, W, need, nan_abc) == dm.ERR_INVALID_ARG
    # an empty problem is a no-op
    assert _raw_ns(dm, 0, [], P, [], 5, 0, W, need) == dm.OK
    lib = dm.lib()
    sh = dm._shapes(shapes)
    nullp = (ctypes.c_void_p * 1)()
    # null per-matrix gradient pointer
    assert lib.dmuon_pack(1, sh, nullp, dm.BF16, nullp, 0.95, P, dm._i64([0]), W, need,
                          None) == dm.ERR_INVALID_ARG
    # bad dtype
    gp = (ctypes.c_void_p * 1)(P)
    assert lib.dmuon_pack(1, sh, gp, 5, gp, 0.95, P, dm._i64([0]), W, need,
                          None) == dm.ERR_INVALID_ARG
    assert lib.dmuon_unpack_update(1, sh, gp, 7, 0.02, P, dm._i64([0]), W, need,
                                   None) == dm.ERR_INVALID_ARG
    assert lib.dmuon_debug_wait_timeout(W, 100, 0, None) == dm.ERR_INVALID_ARG
    assert lib.dmuon_plan(1, sh, 0, (ctypes.c_int * 1)(), dm._i64([0]),
                          dm._i64([0])) == dm.ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib.util
    import shutil
    pkg = tmp_path / "newton_schulz_owner_gb300"
    pkg.mkdir()
    src = os.path.join(ROOT, "newton_schulz_owner_gb300", "dmuon.py")
    shutil.copy(src, pkg / "dmuon.py")
    spec = importlib.util.spec_from_file_location("dmuon_nolib", pkg / "dmuon.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_ns_variant_rule_properties(dm):
    """The Gram rule (host only): standard unless Gram saves work (n > m and at
    least 2 steps) and the step count is one the rule was measured for (2..10);
    never for square matrices; the same for a matrix and its transpose; for a
    fixed step count the Gram aspect ratios form one interval (a band); the
    band edges sit where the measurement put them; GRAM_ALL takes every n > m,
    STANDARD none."""
    ratios = [1.0 + 0.05 * i for i in range(1, 200)]           # 1.05 .. 10.95
    for k in range(0, 14):
        for m in (64, 333, 1024):
            assert dm.ns_variant_for((m, m), k, dm.NS_GRAM) == dm.NS_STANDARD
            picks = []
            for r in ratios:
                n = int(round(r * m))
                got = dm.ns_variant_for((m, n), k, dm.NS_GRAM)
                assert got == dm.ns_variant_for((n, m), k, dm.NS_GRAM)
                if k < 2 or k > 10:
                    assert got == dm.NS_STANDARD
                picks.append(got)
                assert dm.ns_variant_for((m, n), k, dm.NS_GRAM_ALL) == dm.NS_GRAM
                assert dm.ns_variant_for((m, n), k, dm.NS_STANDARD) == dm.NS_STANDARD
            on = [i for i, p in enumerate(picks) if p == dm.NS_GRAM]
            if on:   # one contiguous band
                assert on == list(range(on[0], on[-1] + 1)), (m, k)
    m = 1024
    edge = {5: [(1.5, 0), (1.75, 1), (7.0, 1), (7.5, 0)], 8: [(1.25, 0), (1.5, 1), (8.0, 1), (8.5, 0)],
            10: [(1.5, 0), (1.75, 1), (5.83, 1), (6.5, 0)], 3: [(1.25, 1), (8.0, 1), (9.0, 0)]}
    for k, pts in edge.items():
        for r, want in pts:
            got = dm.ns_variant_for((m, int(round(r * m))), k, dm.NS_GRAM)
            assert got == (dm.NS_GRAM if want else dm.NS_STANDARD), (k, r)
    with pytest.raises(dm.DMuonError):
        dm.ns_variant_for((4, 8), -1, dm.NS_GRAM)
    with pytest.raises(dm.DMuonError):
        dm.ns_variant_for((4, 8), 5, 7)


def test_binding_size_limits_match_the_header(dm):
    """The binding's MAX_M / MAX_N mirror DMUON_MAX_M / DMUON_MAX_N, and the
    library accepts a matrix exactly at both limits and refuses one beyond."""
    text = open(os.path.join(ROOT, "include", "dmuon.h")).read()
    assert int(re.search(r"#define DMUON_MAX_M (\d+)", text).group(1)) == dm.MAX_M
    assert int(re.search(r"#define DMUON_MAX_N (\d+)", text).group(1)) == dm.MAX_N
    assert dm.workspace_bytes([(dm.MAX_M, dm.MAX_M)], 0) > 0
    assert dm.workspace_bytes([(64, dm.MAX_N)], 0) > 0
    assert dm.workspace_bytes([(dm.MAX_N, 64)], 0) > 0
    assert dm.workspace_bytes([(64, dm.MAX_N + 1)], 0) == 0
    assert dm.workspace_bytes([(dm.MAX_M + 1, dm.MAX_M + 1)], 0) == 0
