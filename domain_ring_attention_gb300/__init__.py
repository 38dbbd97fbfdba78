"""Sharded ring attention for one GB300 (sm_103a).

Python surface of the C-ABI library (include/st_attn.h); the functions keep
the C names.  See ``_lib`` for the marshalling and ``workloads`` for the
seeded synthetic inputs.
"""
from ._lib import (  # noqa: F401
    Layout,
    StAttnError,
    load,
    st_attn_bwd,
    st_attn_fwd,
    st_attn_fwd_host,
    st_attn_fwd_partials,
    st_attn_merge,
    st_attn_workspace_size,
    st_permute,
    st_proj_gemm,
    st_gated_mlp,
    st_halo_exchange,
    st_conv2d_sharded,
    st_group_norm_sharded,
    st_ring_workspace_size,
    st_ring_fwd_step,
    st_ring_bwd_step,
    st_ring_fwd_local,
    st_ring_bwd_local,
    st_attn_bwd_delta,
    st_convert_f32,
    st_fp16_scaled_copy,
    ST_DTYPE_BF16,
    ST_DTYPE_F32,
)
