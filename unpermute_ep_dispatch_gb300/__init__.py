"""GB300-native single-GPU MoE expert-parallel token permute / unpermute.

The path has four steps, each a hand-written CUDA kernel for sm_103a behind a
C ABI (``include/epd.h``, ``libepd.so``):

1. ``ep_dispatch_layout`` -- per-expert / per-rank / per-RDMA-node token counts
   and ``is_token_in_rank`` from ``topk_idx`` (plus each pair's rank inside its
   expert, kept in the caller's workspace);
2. ``ep_scan_offsets``    -- ``expert_start_loc``, the exclusive prefix sum of
   the expert counts;
3. ``ep_permute``         -- the ep_scatter copy into the expert-contiguous
   buffer, with ``m_indices`` and ``output_index``;
4. ``ep_unpermute``       -- the topk-weighted, fp32-accumulated combine.

``ep_dispatch_layout_offsets`` runs steps 1 and 2 in one launch and
``ep_dispatch`` steps 1 to 3 in one call (one kernel for a small batch).
The Python functions of the same names only marshal torch tensors into the C
calls; the library is loaded on first use and its absence is an error.
"""
from . import workloads  # noqa: F401  (CPU-only input generator)
from ._binding import (  # noqa: F401,E402
    EPD_BF16, EPD_ERR_CAPACITY, EPD_ERR_CUDA, EPD_ERR_INVALID_ARG, EPD_ERR_INVALID_EXPERT,
    EPD_ERR_TIMEOUT, EPD_ERR_UNSUPPORTED, EPD_FP8_E4M3, EPD_OK, EpdError, check_status,
    aligned_capacity, ep_dispatch, ep_dispatch_layout, ep_dispatch_layout_offsets,
    ep_dispatch_lowlatency, ep_permute,
    ep_permute_ex, ep_permute_lowlatency, ep_scan_offsets, ep_scan_offsets_aligned,
    ep_unpermute, epd_workspace_bytes,
    epd_workspace_init, load_library, new_status, new_workspace, status_string, version,
)
