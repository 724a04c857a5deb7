"""GB300-native ZeRO sharded mixed-precision optimizer step.

The compute lives in libzero.so (C ABI: include/zero.h; CUDA kernels for
sm_103a in csrc/); this package is its Python binding.  ``workloads`` holds the
seeded synthetic parameter groups used by the tests and the benchmark.
"""
from .zero import (AMP_STATE_BYTES, AdamW, AmpConfig, AmpState, amp_state_tensor,  # noqa: F401
                   read_amp_state, zero_amp_init, zero_amp_workspace_bytes, zero_step_amp)
from .zero import Zero3Pass, zero_step_amp_noalloc, zero_zero3_pass  # noqa: F401
from .zero import (AdamW, Plan, ZeroError, ZeroStep, lib, zero_adamw_shard_step,  # noqa: F401
                   zero_allgather, zero_init_shards, zero_last_error, zero_launch_count,
                   zero_memory_bytes, zero_plan_partitions, zero_reduce_scatter, zero_step,
                   zero_sync, zero_version, ZERO_BF16, ZERO_FP16, ZERO_PART_FLAT,
                   ZERO_PART_ROUND_ROBIN, ZERO_REDUCE_AVG, ZERO_REDUCE_SUM)
