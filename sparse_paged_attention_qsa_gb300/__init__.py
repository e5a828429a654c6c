"""GB300 (sm_103a) QSA sparse decode path: paged top-512 block selection and
FP16 sparse paged attention, plus the side-cache metadata builder that feeds
them and a weighted paged MQA indexer with its per-row top-k, as hand-written
CUDA kernels behind the C ABI in include/qsa.h, include/qsa_metadata.h and
include/qsa_indexer.h.  This package is the Python binding (ctypes, marshalling
only), the in-tree build, and the seeded workload generators."""
from .binding import (  # noqa: F401
    COMPRESS_RATIO, DERR_CMP_PAGE, DERR_KV_PAGE, DERR_REQUEST, DERR_TIMEOUT, EXPORTED, LIB_PATH,
    OUT_WIDTH, TOKEN_TOPK, TOPK_BLOCKS, QSAError, declare_signatures, load_library,
    qsa_attention_workspace_bytes,
    qsa_build_metadata, qsa_decode, qsa_paged_mqa_logits, qsa_select_attend,
    qsa_select_attend_fused_rows, qsa_select_attend_fused_cluster,
    qsa_select_attend_workspace_bytes,
    qsa_top_k_per_row_decode, qsa_select_paged_tokens, qsa_select_workspace_bytes, qsa_sparse_attention)
