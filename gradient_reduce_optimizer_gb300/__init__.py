"""GB300-native fused data-parallel step.

Bucketed gradient reduction over R emulated replicas, one AdamW step and the
redistribution of the updated bf16 parameters to every replica, in one pass
per element on sm_103a (CoCoNet's fused ReduceScatter-optimizer-AllGather,
run at DDP bucket granularity in reverse layer order).

* ``capi``      -- Python binding of the C ABI (include/cc_dp.h).
* ``workloads`` -- parameter-shape lists and seeded synthetic inputs.
* ``build``     -- in-tree build of ``libcc_dp.so`` for sm_103a.
"""
from . import capi, workloads  # noqa: F401
from .capi import (CCError, cc_accumulate_local, cc_bucket_ready_layers,  # noqa: F401
                   cc_device_status, cc_fused_dp_bucket, cc_fused_dp_shard,
                   cc_fused_dp_step, cc_fused_dp_step_accum, cc_inject_launch_failure,
                   cc_l2_flush, cc_last_error, cc_overlap_bench, cc_plan_buckets,
                   cc_status_string, cc_tp_allreduce, cc_tp_overlap_bench,
                   cc_unfused_dp_step, cc_unfused_dp_step_noalloc)
