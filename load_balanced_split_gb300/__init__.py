"""Load-balanced split-KV GQA decode attention for GB300 (sm_103a).

The compute path is the C-ABI library libhpa (include/hpa.h, sources in
csrc/); `hpa` is its ctypes binding.  Nothing here computes on the CPU.
"""
from .hpa import (KV_BF16, KV_E4M3, HpaError, Workspace, decode_step,  # noqa: F401
                  hpa_arrivals_elems, hpa_combine, hpa_decode_attn, hpa_decode_attn_allheads,
                  hpa_decode_attn_combine_noalloc, hpa_default_num_ctas_allheads,
                  hpa_decode_attn_mma, hpa_default_num_ctas_mma,
                  hpa_decode_attn_fused, hpa_decode_attn_tc, hpa_default_num_ctas_tc,
                  hpa_decode_attn_traced, hpa_default_num_ctas, hpa_max_segments, hpa_plan,
                  hpa_plan_static, hpa_plan_weighted, hpa_selftest_wait_timeout, hpa_static_num_ctas,
                  hpa_static_taskmap_bytes, hpa_store_kv, hpa_taskmap_bytes, lib,
                  trace_summary)
