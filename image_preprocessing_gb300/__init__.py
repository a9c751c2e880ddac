"""GB300-native fused image normalisation (FusedNormalization on sm_103a).

One memory pass over a uint8 NHWC batch: ToTensor, per-channel Normalize,
optional horizontal flip and optional erase rectangle per image, binary32 or
binary16 output in NHWC, NCHW or 4-channel NHWC.  The work runs in the CUDA
kernels of libtrfn.so (C ABI in include/tr_fused_norm.h); this package is
its thin binding plus the seeded synthetic-input generators (synth).
"""
from .api import (LAUNCH_OVERLAP_PREVIOUS, LAYOUT_NCHW, LAYOUT_NHWC, LAYOUT_NHWC4, OUT_F16, OUT_F32, PRESETS, STAGE_FAST,
                  STAGE_REPRODUCIBLE, VARIANT_AUTO, Staging, tr_stage_zone_bytes,
                  VARIANT_GENERIC, VARIANT_TILED, TransferStation, out_shape, tr_device_status,
                  tr_fused_norm, tr_fused_norm_batches, tr_fused_norm_crop, tr_fused_norm_geometry, tr_fused_norm_plan, tr_fused_norm_sampled, tr_launch_count, tr_norm_preset, tr_sample_aug_params,
                  tr_sample_aug_params_device,
                  tr_ts_slot_bytes, tr_tune_tiled, tr_validate_aug_params, tr_workspace_bytes)
from ._native import LIB_PATH, TrError

__all__ = [
    "LAUNCH_OVERLAP_PREVIOUS", "LAYOUT_NCHW", "LAYOUT_NHWC", "LAYOUT_NHWC4", "OUT_F16", "OUT_F32", "PRESETS", "VARIANT_AUTO",
    "VARIANT_GENERIC", "VARIANT_TILED", "TransferStation", "out_shape", "tr_device_status", "tr_fused_norm",
    "tr_fused_norm_batches",
    "tr_fused_norm_crop", "tr_fused_norm_geometry", "tr_sample_aug_params_device", "tr_fused_norm_sampled",
    "tr_fused_norm_plan", "tr_launch_count", "tr_norm_preset", "tr_sample_aug_params", "tr_ts_slot_bytes",
    "tr_tune_tiled", "tr_workspace_bytes",
    "tr_validate_aug_params", "LIB_PATH", "TrError", "STAGE_FAST", "STAGE_REPRODUCIBLE", "Staging",
    "tr_stage_zone_bytes",
]
