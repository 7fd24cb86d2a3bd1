"""CSA2 global-attention decode path on GB300 (sm_103a).

The compute lives in ``libcsa2.so`` (C ABI, include/csa2.h); this package is
its ctypes binding (``_lib``) plus the decode-step compositions (``decode``)
that chain the entry points on one CUDA stream.  There is no fallback: if the
library is not built, importing the binding raises.
"""
from ._lib import (  # noqa: F401
    CSA2_IDX_MXFP4, CSA2_KV_NVFP4, CSA2_OP_BUILD_CACHE, CSA2_OP_DECODE, CSA2_OP_DECODE_HOST, CSA2_OP_DECODE_MQ,
    CSA2_OP_DECODE_REINDEX, CSA2_OP_SPARSE_ATTN, csa2_build_cache, csa2_decode_reindex, csa2_index_key_proj,
    csa2_profile_events,
    CSA2_OP_TOPK, CSA2_OUT_BF16, CSA2_OUT_F32, CSA2_SWA_MXFP8, CSA2Error, EXPORTS, LIB_PATH, csa2_check_bounded_wait,
    csa2_decode,
    csa2_decode_host, csa2_decode_mq, csa2_entry_bytes, csa2_fp4_pack, csa2_get_device_status, csa2_index_score,
    csa2_index_score_mq, csa2_params, csa2_sparse_attn, csa2_topk, csa2_topk_noalloc, csa2_workspace_size,
    default_params, load,
)

load()
