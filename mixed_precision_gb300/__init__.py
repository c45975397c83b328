"""GB300-native ZeRO-1/2 gradient-and-optimizer step.

The product is the C-ABI library libzero_gb300.so (declared in include/zero.h,
hand-written CUDA for sm_103a). ``_abi`` binds its entry points one for one;
``engine.ZeroStep`` owns the device buffers of one layout. No CPU fallback
exists: without the built library every call raises.
"""
from ._abi import (ZERO_BF16, ZERO_MAX_ELEMS, ZERO_STATE_BLOB_BYTES, zero_accumulate, zero_gather_bucket,
                   zero_loss_scale_state_async, zero_state_blob_decode, zero_scaler_restore, zero_selftest_wait_timeout,
                   zero_selftest_layout_timeout,
                   zero_state_export_params, zero_state_import_params, ZERO_F16, ZERO_F32, ZeroError, zero_bucket_range, zero_config,
                   zero_gather_params, zero_hparams, zero_last_error, zero_layout_create,
                   zero_layout_destroy, zero_layout_info, zero_layout_query,
                   zero_layout_set_allocator, zero_loss_scale_state, zero_param_offset,
                   zero_scaler_cfg, zero_scaler_state, zero_set_step_events, zero_shard_range, zero_state_bind,
                   zero_state_bind_alternate, zero_step_speculative, zero_step_speculative_tensors,
                   zero_state_export, zero_state_import, zero_state_init, zero_step,
                   zero_step_host, zero_step_per_tensor_launch, zero_step_tensors, lib)

__all__ = [n for n in dir() if n.startswith("zero_") or n.startswith("ZERO_")] + ["ZeroError", "lib"]
