"""GB300 (sm_103a) differential attention (forward, backward, cache forward) behind a C ABI.

The public functions carry the names of the C entry points in
include/diffattn.h and take torch tensors for device memory and streams.
"""
from ._lib import (  # noqa: F401
    DTYPE_BF16,
    DTYPE_F32,
    DiffAttnDesc,
    DiffAttnError,
    DiffAttnKvDesc,
    DiffAttnMergeDesc,
    DiffAttnOutProjDesc,
    DiffAttnRopeDesc,
    DiffAttnRopeQ,
    diffattn_bwd,
    diffattn_bwd_workspace_size,
    diffattn_fwd,
    diffattn_fwd_lambda,
    diffattn_fwd_kernel,
    diffattn_fwd_rope_q,
    diffattn_fwd_train,
    diffattn_fwd_kvcache,
    diffattn_fwd_kvcache_lambda,
    diffattn_fwd_kvcache_noalloc,
    diffattn_fwd_kvcache_workspace_size,
    diffattn_get_device_status,
    diffattn_lambda,
    diffattn_lambda_bwd,
    diffattn_lambda_init,
    diffattn_merge_partials,
    diffattn_out_proj,
    diffattn_rope_k,
    diffattn_rope_qk,
    diffattn_rope_tables,
    diffattn_set_fault_injection,
    diffattn_set_wait_timeout_ns,
    diffattn_status_string,
    kv_desc,
    load_library,
)
from ._build import LIB_PATH, build  # noqa: F401
