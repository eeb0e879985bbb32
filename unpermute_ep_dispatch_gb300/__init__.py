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

The Python functions of the same names only marshal torch tensors into the C
calls; the library is loaded on first use and its absence is an error.
"""
from . import workloads  # noqa: F401  (CPU-only input generator)
