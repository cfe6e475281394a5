"""fp64 CPU oracle for the DMuon owner-side Muon step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  It imports nothing from the CUDA
library and the CUDA library imports nothing from it.
"""
from .muon_oracle import (  # noqa: F401
    NS_COEFFS, NS_EPS, DEFAULT_LR, DEFAULT_NS_STEPS, DEFAULT_BETA,
    PACK_ALIGN_BYTES, PACK_ALIGN_ELEMS,
    nesterov_momentum, ns_working_matrix, ns_normalise, newton_schulz,
    gram_newton_schulz, update_scale, apply_update, muon_step, round_bf16,
    lpt_assign, pack_plan, ns_flops_algorithmic, gram_ns_flops_algorithmic,
    adamw_step, ADAMW_DEFAULT_LR, ADAMW_DEFAULT_BETAS, ADAMW_DEFAULT_EPS, ADAMW_DEFAULT_WD,
)
