"""GB300-native ZeRO sharded mixed-precision optimizer step.

The compute lives in libzero.so (C ABI: include/zero.h; CUDA kernels for
sm_103a in csrc/); this package is its Python binding.  ``engine`` wires a
model's backward pass into it; ``workloads`` holds the seeded synthetic
parameter groups used by the tests and the benchmark.
"""
from .zero import (AMP_STATE_BYTES, ZERO_BF16, ZERO_FP16, ZERO_PART_FLAT,  # noqa: F401
                   ZERO_PART_ROUND_ROBIN, ZERO_REDUCE_AVG, ZERO_REDUCE_SUM, AdamW, AmpConfig,
                   AmpState, FloorProbe, Plan, ReduceScatterBucketAmp, ReduceScatterRange,
                   Zero3Pass, ZeroError, ZeroStep,
                   amp_state_tensor, lib, read_amp_state, zero_adamw_shard_step, zero_allgather,
                   zero_amp_init, zero_amp_workspace_bytes, zero_cpu_adamw_shard_step,
                   zero_init_shards, zero_last_error, zero_launch_count, zero_memory_bytes,
                   zero_offload_step, zero_offload_step_amp,
                   zero_plan_describe, zero_plan_destroy, zero_plan_info, zero_plan_partitions,
                   zero_plan_segments, zero_plan_shard, zero_plan_total, zero_reduce_scatter,
                   zero_reduce_scatter_bucket_amp, zero_reduce_scatter_range,
                   zero_floor_probe, zero_selftest_wait_timeout, zero_step, zero_step_amp,
                   zero_step_amp_noalloc, zero_step_amp_reduced, zero_step_amp_shards,
                   zero_sync, zero_version, zero_zero3_pass)
