"""Absorbed Multi-Head Latent Attention decode for B300 (sm_103a).

The computation lives in the CUDA library ``libmla.so`` (C ABI in
``include/mla.h``); this package only loads it and marshals arguments.
"""
from ._lib import (  # noqa: F401
    EXPORTED, LIB_PATH, MLA_BF16, MLA_DEV_BAD_LENGTH, MLA_DEV_BAD_POSITION, MLA_DEV_TIMEOUT, MLA_DEV_SMEM_ALIGN,
    MLA_ERR_CUDA, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_F32, MLA_OK,
    MlaCacheLayout, MlaDims, MlaError, load, make_cache_layout, make_dims, mla_append_workspace_size,
    mla_cache_append, mla_cache_append_ex, mla_cache_append_fp8, mla_copy_from_host, mla_decode_absorbed, mla_decode_absorbed_ex,
    mla_decode_absorbed_multi, mla_decode_absorbed_fp8, mla_decode_prepare_beside, fp8_row_bytes, mla_decode_workspace_size, mla_launch_count, mla_profile_events,
    mla_project_out, mla_project_output, mla_project_output_merged, mla_merge_output_weights,
    mla_project_query, mla_project_query_latent, mla_set_wait_limit_ns, status_string,
)
