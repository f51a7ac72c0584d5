"""Owner-side Muon update for one GB300 (sm_103a): momentum accumulate,
Newton-Schulz orthogonalisation in Gram or original space on tcgen05 tensor
cores, and the scaled apply, behind the C ABI in include/muon_ns.h.

Importing the package does not load the CUDA library; the first call does.
"""
from .binding import (  # noqa: F401
    AdamwTail, MuonError, MuonUpdater, adamw_tail, bucket_plan, cost_estimate, debug_bounded_wait,
    debug_bounded_wait_static, debug_gemm, device_status, library_path, load, measure_costs, muon_step, new_workspace,
    ns_batched, ns_batched_static, owned, partition, profile_enable, profile_records, resolve_schedule,
    sched_code, schedule_candidates, static_status, tune_schedules, workspace_bytes,
)
