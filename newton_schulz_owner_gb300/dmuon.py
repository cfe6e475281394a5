"""ctypes binding of ``libdmuon.so`` (declared in ``include/dmuon.h``).

Argument marshalling only: every step of the Muon step runs in the library's
CUDA kernels.  PyTorch provides device memory and the CUDA stream.  Importing
this module raises ``ImportError`` if the library has not been built, so no
caller can silently fall back to another implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdmuon.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m newton_schulz_owner_gb300.build_lib` (or __graft_entry__.build())")
_lib = ctypes.CDLL(_LIB_PATH)

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = \
    0, -1, -2, -3, -4, -5, -6
F32, BF16 = 0, 1
NS_STANDARD, NS_GRAM, NS_GRAM_ALL = 0, 1, 2
PACK_ALIGN_ELEMS = 128
DEFAULT_ABC = (3.4445, -4.7750, 2.0315)

EXPORTED = ("dmuon_plan", "dmuon_workspace_bytes", "dmuon_ns_variant_for", "dmuon_pack", "dmuon_ns_batched",
            "dmuon_unpack_update", "dmuon_muon_step", "dmuon_stream_status",
            "dmuon_debug_wait_timeout", "dmuon_ns_batched_noalloc", "dmuon_noalloc_status",
            "dmuon_adamw",
            "dmuon_adamw_workspace_bytes", "dmuon_status_string", "dmuon_version",
            "dmuon_launch_count", "dmuon_trace_begin", "dmuon_trace_end")
NOALLOC_SCRATCH_BYTES = 64 << 20
# largest short side m and long side n of a matrix the library accepts
MAX_M, MAX_N = 32768, 1048576


class Shape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


_vp, _i, _f, _sz, _i64p = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, \
    ctypes.POINTER(ctypes.c_int64)
_ShapeP = ctypes.POINTER(Shape)
_VPP = ctypes.POINTER(ctypes.c_void_p)

_lib.dmuon_plan.argtypes = [_i, _ShapeP, _i, ctypes.POINTER(ctypes.c_int), _i64p, _i64p]
_lib.dmuon_plan.restype = _i
_lib.dmuon_workspace_bytes.argtypes = [_i, _ShapeP, _i]
_lib.dmuon_workspace_bytes.restype = _sz
_lib.dmuon_ns_variant_for.argtypes = [ctypes.c_int64, ctypes.c_int64, _i, _i]
_lib.dmuon_ns_variant_for.restype = _i
_lib.dmuon_pack.argtypes = [_i, _ShapeP, _VPP, _i, _VPP, _f, _vp, _i64p, _vp, _sz, _vp]
_lib.dmuon_pack.restype = _i
_lib.dmuon_ns_batched.argtypes = [_i, _ShapeP, _vp, _i64p, _i, _i, ctypes.POINTER(ctypes.c_float),
                                  _f, _i, _vp, _sz, _vp]
_lib.dmuon_ns_batched.restype = _i
_lib.dmuon_unpack_update.argtypes = [_i, _ShapeP, _VPP, _i, _f, _vp, _i64p, _vp, _sz, _vp]
_lib.dmuon_unpack_update.restype = _i
_lib.dmuon_muon_step.argtypes = [_i, _ShapeP, _VPP, _i, _VPP, _VPP, _i, _f, _f, _i, _i, _vp,
                                 _i64p, _vp, _sz, _vp]
_lib.dmuon_muon_step.restype = _i
_lib.dmuon_ns_batched_noalloc.argtypes = [_i, _ShapeP, _vp, _i64p, _i, _i,
                                          ctypes.POINTER(ctypes.c_float), _f, _vp]
_lib.dmuon_ns_batched_noalloc.restype = _i
_lib.dmuon_noalloc_status.argtypes = [_vp]
_lib.dmuon_noalloc_status.restype = _i
_lib.dmuon_adamw_workspace_bytes.argtypes = [_i]
_lib.dmuon_adamw_workspace_bytes.restype = _sz
_d = ctypes.c_double
_lib.dmuon_adamw.argtypes = [_i, _i64p, _VPP, _i, _VPP, _i, _VPP, _VPP, _d, _d, _d, _d, _d, _i,
                             _vp, _sz, _vp]
_lib.dmuon_adamw.restype = _i
_lib.dmuon_stream_status.argtypes = [_vp, _vp]
_lib.dmuon_stream_status.restype = _i
_lib.dmuon_debug_wait_timeout.argtypes = [_vp, _sz, _i, _vp]
_lib.dmuon_debug_wait_timeout.restype = _i
_lib.dmuon_status_string.argtypes = [_i]
_lib.dmuon_status_string.restype = ctypes.c_char_p
_lib.dmuon_version.argtypes = []
_lib.dmuon_version.restype = _i
_lib.dmuon_launch_count.argtypes = [_i]
_lib.dmuon_launch_count.restype = ctypes.c_longlong
_lib.dmuon_trace_begin.argtypes = [_vp, _sz]
_lib.dmuon_trace_begin.restype = _i
_lib.dmuon_trace_end.argtypes = []
_lib.dmuon_trace_end.restype = ctypes.c_longlong
TRACE_RECORD_BYTES = 72


class DMuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    return _lib


def library_path() -> str:
    return _LIB_PATH


def status_string(status: int) -> str:
    return _lib.dmuon_status_string(int(status)).decode()


def version() -> int:
    return int(_lib.dmuon_version())


def launch_count(reset: bool = False) -> int:
    """Kernels the library launched from this host thread since the last reset."""
    return int(_lib.dmuon_launch_count(1 if reset else 0))


def _check(status: int, where: str) -> None:
    if status != OK:
        raise DMuonError(status, where)


def _shapes(shapes: Sequence[Tuple[int, int]]):
    arr = (Shape * max(1, len(shapes)))()
    for i, (r, c) in enumerate(shapes):
        arr[i].rows, arr[i].cols = int(r), int(c)
    return arr


def _ptrs(ts) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(ts)))()
    for i, t in enumerate(ts):
        arr[i] = t if isinstance(t, int) else t.data_ptr()
    return arr


def _i64(vals) -> ctypes.Array:
    arr = (ctypes.c_int64 * max(1, len(vals)))()
    for i, v in enumerate(vals):
        arr[i] = int(v)
    return arr


def _dtype(t) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: expected bfloat16 or float32")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _addr(t) -> int:
    return t if isinstance(t, int) else t.data_ptr()


# ------------------------------------------------------------------ calls
def plan(shapes: Sequence[Tuple[int, int]], n_owners: int = 1) -> Tuple[List[int], List[int], List[int]]:
    """Owner map, packed offsets and owner buffer sizes (host only)."""
    n = len(shapes)
    own = (ctypes.c_int * max(1, n))()
    off = (ctypes.c_int64 * max(1, n))()
    oel = (ctypes.c_int64 * max(1, n_owners))()
    _check(_lib.dmuon_plan(n, _shapes(shapes), int(n_owners), own, off, oel), "dmuon_plan")
    return list(own[:n]), list(off[:n]), list(oel[:n_owners])


def workspace_bytes(shapes: Sequence[Tuple[int, int]], variant: int = NS_STANDARD) -> int:
    return int(_lib.dmuon_workspace_bytes(len(shapes), _shapes(shapes), int(variant)))


def ns_variant_for(shape: Tuple[int, int], ns_steps: int, variant: int = NS_GRAM) -> int:
    """The Newton-Schulz form (NS_STANDARD or NS_GRAM) a call with `variant`
    runs on one matrix of this shape at `ns_steps` steps (host only)."""
    st = int(_lib.dmuon_ns_variant_for(int(shape[0]), int(shape[1]), int(ns_steps), int(variant)))
    if st < 0:
        raise DMuonError(st, "dmuon_ns_variant_for")
    return st


def pack(shapes, grads, momenta, beta, packed, offsets, workspace, stream=None) -> None:
    n = len(shapes)
    gdt = _dtype(grads[0]) if n else BF16
    _check(_lib.dmuon_pack(n, _shapes(shapes), _ptrs(grads), gdt, _ptrs(momenta), float(beta),
                           _addr(packed), _i64(offsets), _addr(workspace), workspace.numel()
                           if hasattr(workspace, "numel") else 0, _stream(stream)), "dmuon_pack")


def ns_batched(shapes, packed, offsets, workspace, ns_steps: int = 5, variant: int = NS_STANDARD,
               abc: Optional[Sequence[float]] = None, eps: float = 1e-7,
               use_pack_norms: bool = False, stream=None, ws_bytes: Optional[int] = None) -> None:
    n = len(shapes)
    abc_arr = None if abc is None else (ctypes.c_float * 3)(*[float(v) for v in abc])
    wsb = ws_bytes if ws_bytes is not None else workspace.numel()
    _check(_lib.dmuon_ns_batched(n, _shapes(shapes), _addr(packed), _i64(offsets), int(ns_steps),
                                 int(variant), abc_arr, float(eps), int(bool(use_pack_norms)),
                                 _addr(workspace), wsb, _stream(stream)), "dmuon_ns_batched")


def ns_batched_noalloc(shapes, packed, offsets, ns_steps: int = 5, variant: int = NS_STANDARD,
                       abc: Optional[Sequence[float]] = None, eps: float = 1e-7,
                       stream=None) -> None:
    """dmuon_ns_batched on the library's built-in scratch array (no workspace,
    no device allocation); problems up to NOALLOC_SCRATCH_BYTES of workspace."""
    abc_arr = None if abc is None else (ctypes.c_float * 3)(*[float(v) for v in abc])
    _check(_lib.dmuon_ns_batched_noalloc(len(shapes), _shapes(shapes), _addr(packed),
                                         _i64(offsets), int(ns_steps), int(variant), abc_arr,
                                         float(eps), _stream(stream)),
           "dmuon_ns_batched_noalloc")


def noalloc_status(stream=None) -> int:
    """Synchronise the stream and report (and clear) the error word of the
    built-in scratch array used by :func:`ns_batched_noalloc`."""
    return int(_lib.dmuon_noalloc_status(_stream(stream)))


def unpack_update(shapes, weights, lr, packed, offsets, workspace, stream=None) -> None:
    n = len(shapes)
    wdt = _dtype(weights[0]) if n else BF16
    _check(_lib.dmuon_unpack_update(n, _shapes(shapes), _ptrs(weights), wdt, float(lr),
                                    _addr(packed), _i64(offsets), _addr(workspace),
                                    workspace.numel(), _stream(stream)), "dmuon_unpack_update")


def muon_step(shapes, grads, momenta, weights, packed, offsets, workspace, lr: float = 0.02,
              beta: float = 0.95, ns_steps: int = 5, variant: int = NS_STANDARD,
              stream=None) -> None:
    n = len(shapes)
    gdt = _dtype(grads[0]) if n else BF16
    wdt = _dtype(weights[0]) if n else BF16
    _check(_lib.dmuon_muon_step(n, _shapes(shapes), _ptrs(grads), gdt, _ptrs(momenta),
                                _ptrs(weights), wdt, float(lr), float(beta), int(ns_steps),
                                int(variant), _addr(packed), _i64(offsets), _addr(workspace),
                                workspace.numel(), _stream(stream)), "dmuon_muon_step")


def adamw_workspace_bytes(n: int) -> int:
    return int(_lib.dmuon_adamw_workspace_bytes(int(n)))


def adamw(params, grads, exp_avgs, exp_avg_sqs, step: int, workspace, lr: float = 1e-3,
          betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.01,
          stream=None) -> None:
    """One AdamW step over a list of tensors (one kernel launch)."""
    n = len(params)
    pdt = _dtype(params[0]) if n else F32
    gdt = _dtype(grads[0]) if n else F32
    numel = _i64([p.numel() for p in params])
    _check(_lib.dmuon_adamw(n, numel, _ptrs(params), pdt, _ptrs(grads), gdt, _ptrs(exp_avgs),
                            _ptrs(exp_avg_sqs), float(lr), float(betas[0]), float(betas[1]),
                            float(eps), float(weight_decay), int(step), _addr(workspace),
                            workspace.numel(), _stream(stream)), "dmuon_adamw")


def stream_status(workspace=None, stream=None) -> int:
    return int(_lib.dmuon_stream_status(_stream(stream),
                                        None if workspace is None else _addr(workspace)))


def debug_wait_timeout(workspace, budget_us: int, stream=None) -> None:
    """Make a bounded device wait run out; workspace None targets the built-in
    scratch array of :func:`ns_batched_noalloc`."""
    ws = None if workspace is None else _addr(workspace)
    nbytes = 0 if workspace is None else workspace.numel()
    _check(_lib.dmuon_debug_wait_timeout(ws, nbytes, int(budget_us), _stream(stream)),
           "dmuon_debug_wait_timeout")


def trace_begin(buffer) -> None:
    """Record one timestamp record per CTA of every product launch into
    `buffer` (a uint8 CUDA tensor) until :func:`trace_end`."""
    _check(_lib.dmuon_trace_begin(_addr(buffer), buffer.numel()), "dmuon_trace_begin")


def trace_end(buffer):
    """Stop tracing; return the records as a dict of int64 CPU tensors (read
    after the traced work has completed)."""
    n = int(_lib.dmuon_trace_end())
    raw = buffer[:n * TRACE_RECORD_BYTES].cpu()
    u32 = raw.view(torch.int32).view(n, 18).to(torch.int64) & 0xFFFFFFFF
    u64 = raw.view(torch.int64).view(n, 9)
    return {"launch": u32[:, 0], "cta": u32[:, 1], "kind": u32[:, 2], "tiles": u32[:, 3],
            "t_entry": u64[:, 2], "t_mma_first": u64[:, 3], "t_mma_last": u64[:, 4],
            "t_exit": u64[:, 5], "mma_span_cycles": u64[:, 6], "wait_operand_cycles": u64[:, 7],
            "wait_accum_cycles": u64[:, 8]}


class MuonOwner:
    """One owner's Muon state for a fixed list of matrix shapes.

    Holds the packed bf16 buffer and the workspace (both allocated through
    PyTorch), and runs :func:`muon_step` on caller tensors.  Home page ("What
    DMuon Can Do"): each owner runs Muon once per step for the matrices it owns;
    "Z2 vs Z3 Modes": those matrices share one contiguous packed buffer.
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], n_owners: int = 1,
                 variant: int = NS_STANDARD, device="cuda"):
        self.shapes = [(int(r), int(c)) for r, c in shapes]
        self.variant = int(variant)
        self.owner_of, self.offsets, self.owner_elems = plan(self.shapes, n_owners)
        total = max(sum(self.owner_elems), PACK_ALIGN_ELEMS)
        self.packed = torch.empty(total, dtype=torch.bfloat16, device=device)
        self.ws_bytes = workspace_bytes(self.shapes, self.variant)
        if self.ws_bytes == 0:
            raise DMuonError(ERR_INVALID_ARG, "dmuon_workspace_bytes")
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)

    def step(self, grads, momenta, weights, lr: float = 0.02, beta: float = 0.95,
             ns_steps: int = 5, stream=None) -> None:
        muon_step(self.shapes, grads, momenta, weights, self.packed, self.offsets, self.workspace,
                  lr=lr, beta=beta, ns_steps=ns_steps, variant=self.variant, stream=stream)

    def packed_view(self, i: int) -> torch.Tensor:
        r, c = self.shapes[i]
        o = self.offsets[i]
        return self.packed[o:o + r * c].view(r, c)

    def status(self, stream=None) -> int:
        return stream_status(self.workspace, stream)
