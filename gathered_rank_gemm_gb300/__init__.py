"""Multi-LoRA shrink/expand over an unsorted mixed-adapter batch, for GB300 (sm_103a).

The compute lives in the CUDA library ``libgathered_rank_gemm.so`` (C ABI in
``include/gathered_rank_gemm.h``); ``binding`` is its thin ctypes wrapper and
``workloads`` draws seeded synthetic inputs.  The wrappers take bf16 tensors,
or fp16 tensors for the stacked-weight calls (routed to the ``*_f16`` entry
points).
"""
from .binding import (LoraError, LoraMetadata, lora_apply_noalloc, lora_expand,  # noqa: F401
                      lora_expand_paged, lora_expand_partials, lora_prepare_metadata,
                      lora_read_status, lora_shrink, lora_shrink_expand,
                      lora_shrink_expand_kernels, lora_shrink_expand_paged,
                      lora_shrink_expand_workspace_size, lora_shrink_paged,
                      lora_shrink_partials, lora_workspace_size)

__all__ = ["LoraError", "LoraMetadata", "lora_apply_noalloc", "lora_expand",
           "lora_expand_paged", "lora_expand_partials", "lora_prepare_metadata",
           "lora_read_status", "lora_shrink", "lora_shrink_expand", "lora_shrink_expand_kernels",
           "lora_shrink_expand_paged", "lora_shrink_expand_workspace_size", "lora_shrink_paged",
           "lora_shrink_partials", "lora_workspace_size"]
