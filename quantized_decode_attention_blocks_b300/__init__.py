"""KVarN-style quantized KV cache for B300 (sm_103a).

The compute lives in libkvarn.so (CUDA kernels behind the C ABI of
include/kvarn.h); this package is its thin Python binding.
"""
from .kvarn import (Config, KvarnError, alloc_decode_workspace, alloc_fp16_decode_workspace,
                    alloc_fp8_decode_workspace, alloc_fp8_pool, fp8_decode_workspace_bytes,
                    kvarn_fp8_decode_attention, kvarn_fp8_write_blocks,
                    kvarn_snapkv_gather, kvarn_snapkv_select, snapkv_workspace_bytes,
                    alloc_fp16_pool, alloc_pool, alloc_tails, fp16_decode_workspace_bytes,
                    kvarn_fp16_decode_attention, kvarn_fp16_write_blocks,
                    config_from_string, config_validate, decode_split_plan, decode_workspace_bytes,
                    kvarn_append_token, kvarn_chunk_attention, kvarn_decode_attention,
                    kvarn_decode_attention_noalloc, kvarn_dequantize_pages, kvarn_dequantize_records,
                    kvarn_quantize_blocks, lib, page_bytes, status_string, version)

__all__ = ["Config", "KvarnError", "alloc_decode_workspace", "alloc_fp16_decode_workspace",
           "alloc_fp8_decode_workspace", "alloc_fp8_pool", "fp8_decode_workspace_bytes",
           "kvarn_fp8_decode_attention", "kvarn_fp8_write_blocks",
           "kvarn_snapkv_gather", "kvarn_snapkv_select", "snapkv_workspace_bytes",
           "alloc_fp16_pool", "alloc_pool", "alloc_tails", "fp16_decode_workspace_bytes",
           "kvarn_fp16_decode_attention", "kvarn_fp16_write_blocks",
           "config_from_string", "config_validate", "decode_split_plan", "decode_workspace_bytes",
           "kvarn_append_token", "kvarn_chunk_attention", "kvarn_decode_attention",
           "kvarn_decode_attention_noalloc", "kvarn_dequantize_pages", "kvarn_dequantize_records",
           "kvarn_quantize_blocks", "lib", "page_bytes", "status_string", "version"]
