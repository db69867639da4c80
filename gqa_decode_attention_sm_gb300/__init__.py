"""GB300 (sm_103a) single-token grouped-query decode attention.

The compute path is libgqa_decode.so (hand-written CUDA kernels behind a C
ABI, include/gqa_decode.h); ``api`` is a thin PyTorch binding over it.
Importing the package does not load the library; the first call does, and
raises if the library has not been built (there is no fallback path).
"""
from .api import (GqaError, Prepared, append_kv, append_kv_paged, combine_stage, get_status, gqa_decode, gqa_decode_fp8kv,
                  gqa_decode_int8kv, gqa_decode_paged, gqa_decode_verify, launch, plan, prepare, split_stage,
                  workspace_init, workspace_size)

__all__ = ["GqaError", "Prepared", "append_kv", "append_kv_paged", "combine_stage", "get_status", "gqa_decode", "gqa_decode_fp8kv",
           "gqa_decode_int8kv", "gqa_decode_paged", "gqa_decode_verify", "launch", "plan", "prepare", "split_stage",
           "workspace_init", "workspace_size"]
