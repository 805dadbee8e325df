"""Decode and prefill attention over a paged (block-table) or contiguous
(reqId x S) KV cache, with KV append, copy-on-write block copy and block swap
to host memory (pre-emption), as hand-written sm_103a CUDA kernels behind a C
ABI (include/pkv.h).  This package is the thin Python binding; build the
library with ``build.build()``."""
from .binding import (BlockManager, PkvError, VmmBuffer, block_copy, block_swap,
                      BM_RETIRED, BM_RUNNING, BM_SWAPPED, BM_RECOMPUTE, PREEMPT_RECOMPUTE,
                      PREEMPT_SWAP, contig_decode_attention, contig_decode_step,
                      decode_num_splits, decode_uses_tensor_cores, paged_decode_step,
                      paged_decode_attention_shared,
                      shared_decode_launches,
                      paged_prefill_attention, contig_prefill_attention,
                      decode_workspace_size, get_checked, get_device_error, kv_append, lib,
                      paged_decode_attention, set_checked, set_decode_variant, get_decode_variant,
                      set_split_tiles, VARIANT_AUTO, VARIANT_SPLIT, VARIANT_TC_8X3,
                      VARIANT_TC_12X2)

__all__ = ["BlockManager", "PkvError", "VmmBuffer", "block_copy", "block_swap", "BM_RETIRED",
           "BM_RUNNING", "BM_SWAPPED", "BM_RECOMPUTE", "PREEMPT_RECOMPUTE", "PREEMPT_SWAP",
           "contig_decode_attention", "contig_decode_step",
           "paged_decode_step", "paged_decode_attention_shared", "paged_prefill_attention",
           "contig_prefill_attention",
           "decode_num_splits", "decode_uses_tensor_cores", "shared_decode_launches",
           "decode_workspace_size", "get_checked", "get_device_error", "kv_append", "lib",
           "paged_decode_attention", "set_checked", "set_split_tiles", "set_decode_variant",
           "get_decode_variant", "VARIANT_AUTO", "VARIANT_SPLIT", "VARIANT_TC_8X3",
           "VARIANT_TC_12X2"]
