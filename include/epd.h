/*
 * epd.h -- C ABI of libepd: single-GPU MoE expert-parallel token permute and
 * unpermute for GB300 (sm_103a).
 *
 * The path, in the order a caller runs it on one stream:
 *   1. ep_dispatch_layout  counts per expert / simulated rank / simulated RDMA
 *                          node and the is_token_in_rank mask;
 *   2. ep_scan_offsets     expert_start_loc = exclusive prefix sum of the counts;
 *   3. ep_permute          ep_scatter: token rows into the expert-contiguous
 *                          buffer, with m_indices and output_index;
 *   4. ep_unpermute        combine: the topk-weighted sum of each token's expert
 *                          output rows, accumulated in fp32.
 * ep_dispatch_layout_offsets runs steps 1 and 2 in one launch, and ep_dispatch
 * steps 1 to 3 in one call (a single kernel for a decode-sized batch).
 * Nothing in between goes back to the host: every count, offset and total stays
 * in device memory, and the permuted buffer is sized at the T*k upper bound.
 *
 * Conventions shared by every call:
 *   - The caller owns all memory. libepd never allocates or frees device or
 *     host memory. Every pointer argument except the stream is a device
 *     pointer unless stated otherwise.
 *   - Every call is asynchronous on the caller's stream, does not synchronise
 *     and touches no host memory (the stream replaces DeepEP's previous_event /
 *     async_finish pair).
 *   - The return value reports argument errors, found on the host before any
 *     launch (EPD_ERR_INVALID_ARG, EPD_ERR_UNSUPPORTED), and launch errors
 *     (EPD_ERR_CUDA). A call that returns an error has launched nothing.
 *   - Errors that depend on the data (an expert id outside [-1, E), a slot
 *     outside the buffer, a look-back wait that gave up) are written to the
 *     caller's device word `status` with an atomic compare-and-swap from 0, so
 *     the first error sticks until the caller clears the word. Kernels never
 *     trap: the offending pair is skipped and the call completes.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the kernel before it on the stream drains, and waits
 *     (griddepcontrol.wait) before it reads what that kernel may write; every
 *     libepd kernel waits before it lets its own dependents start. Calls on one
 *     stream may follow each other in any order on one workspace -- two layout
 *     calls back to back included: a layout kernel takes its tile ticket before
 *     that wait from a counter that every call returns to zero, and reads the
 *     rest of the workspace only after it.
 *   - Sizes: T = num_tokens >= 0, k = num_topk in [0, EPD_MAX_TOPK],
 *     E = num_experts in [1, EPD_MAX_EXPERTS], R = num_ranks with E % R == 0,
 *     N = num_rdma_ranks with R % N == 0, T*k <= INT32_MAX.
 *     Expert e lives on simulated rank e / (E/R); rank r on node r / (R/N).
 *
 * Page references (page title, section):
 *   [P1] "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题"
 *   [P2] "高性能专家并行（EP）内核解剖学解读"
 *   [P3] "[MoE] Deepseek的All-to-all通信: DeepEP代码解读"
 */
#ifndef EPD_H
#define EPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EPD_API __attribute__((visibility("default")))
#else
#define EPD_API
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *epd_stream_t;

typedef enum {
    EPD_OK = 0,
    EPD_ERR_INVALID_ARG = 1,    /* bad size, null or misaligned pointer, mismatched workspace */
    EPD_ERR_UNSUPPORTED = 2,    /* valid but beyond a documented limit */
    EPD_ERR_CUDA = 3,           /* a CUDA call failed; epd_last_cuda_error() has the cause */
    EPD_ERR_INVALID_EXPERT = 4, /* (status word) topk_idx held an id outside [-1, E) */
    EPD_ERR_TIMEOUT = 5,        /* (status word) a bounded look-back wait gave up */
    EPD_ERR_CAPACITY = 6,       /* (status word) a slot fell outside [0, capacity_rows) */
} epd_status_t;

typedef enum {
    EPD_BF16 = 0,      /* rows of H bfloat16 values (2H bytes), H % 8 == 0 */
    EPD_FP8_E4M3 = 1,  /* rows of H float8_e4m3fn values (H bytes) plus H/128 fp32
                          scales per row, H % 128 == 0 */
} epd_dtype_t;

#define EPD_MAX_EXPERTS 4096
#define EPD_MAX_TOPK 64
#define EPD_MAX_ALIGNMENT 4096

/* Human-readable name of a status code (static string; never NULL). */
EPD_API const char *epd_status_string(int code);

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
EPD_API int epd_version(void);

/*
 * The cudaError_t code of the last CUDA failure seen by a libepd call on this
 * host thread (0 if none). libepd reads and clears the CUDA runtime's
 * last-error state when a launch fails, so the caller's own error checks are
 * not disturbed; this is where the cause is kept.
 */
EPD_API int epd_last_cuda_error(void);

/*
 * Workspace size in bytes for one layout -> permute chain over T tokens, k
 * picks, E experts, R ranks and N nodes. The workspace holds the per-pair rank
 * inside its expert (T*k int32), the per-expert counts and, for batches beyond
 * one thread-block cluster, the per-tile state of the layout's single-pass
 * look-back (whose count rows, when the batch runs as several clusters, hold the
 * counts each cluster publishes). Returns 0 for invalid sizes. Host-only
 * arithmetic.
 */
EPD_API size_t epd_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks,
                           int num_rdma_ranks);

/*
 * Zero-fills `workspace` (device, `bytes` long) on `stream`. A workspace must
 * be zero-filled once before its first use; the layout call keeps it reusable
 * from then on, for calls of any shape that fits (its look-back state words and
 * the counts clusters publish are tagged with a call counter and a mark no other
 * workspace data carries). A
 * workspace serves one stream at a time: calls on different streams that
 * overlap on the GPU and share a workspace race.
 */
EPD_API epd_status_t epd_workspace_init(void *workspace, size_t bytes, epd_stream_t stream);

/*
 * Step 1 -- dispatch layout. [P3] "Dispatch", get_dispatch_layout docstring:
 * from topk_idx [T, k] int64 (row-major; -1 = no selection) compute
 *   tokens_per_expert    [E] int32: number of (t, j) with topk_idx[t, j] == e;
 *   tokens_per_rank      [R] int32: number of tokens with a pick on rank r
 *                                   (a token counts once per rank);
 *   tokens_per_rdma_rank [N] int32: number of tokens with a pick on node n
 *                                   (once per node); may be NULL (DeepEP
 *                                   returns None for one node);
 *   is_token_in_rank  [T, R] uint8: 1 if token t has a pick on rank r, else 0
 *                                   (torch.bool layout); may be NULL.
 * and, in `workspace` (epd_workspace_bytes(T, k, E, R, N) bytes), the rank of
 * every pair among the pairs of its expert in token-major (t, then j) order,
 * which ep_permute turns into slots. The ranks come from per-tile counts and
 * an exclusive prefix over token tiles: for up to 16 x 8192 pairs (E <= 1024)
 * the tiles are the blocks of thread-block clusters of 2-16 blocks, which
 * exchange their counts through distributed shared memory -- one cluster, or,
 * where one cluster of 16 would need 8 chunks of 32 pairs per warp, up to 8
 * clusters that all fit on the device at once, whose last blocks publish each
 * cluster's counts in the workspace for the later clusters (a later cluster waits
 * for the earlier ones to run: should other work hold the SMs they need for about
 * a second, the wait gives up with EPD_ERR_TIMEOUT); larger batches use
 * a single-pass decoupled look-back over tiles taken in ticket order. Every way
 * the result does not depend on the order in which blocks run. Ids outside
 * [-1, E) set EPD_ERR_INVALID_EXPERT in *status and are treated as -1.
 */
EPD_API epd_status_t ep_dispatch_layout(const int64_t *topk_idx, int num_tokens, int num_topk,
                                int num_experts, int num_ranks, int num_rdma_ranks,
                                int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                int32_t *tokens_per_rdma_rank, uint8_t *is_token_in_rank,
                                void *workspace, int32_t *status, epd_stream_t stream);

/*
 * Steps 1 and 2 in one launch: ep_dispatch_layout, and the block of the last
 * token tile, once it has the totals, also writes expert_start_loc and *total_rows exactly as
 * ep_scan_offsets_aligned(tokens_per_expert, alignment) would (alignment 1 gives
 * ep_scan_offsets). Saves one launch and one kernel per pass; same arguments and
 * errors as ep_dispatch_layout otherwise.
 */
EPD_API epd_status_t ep_dispatch_layout_offsets(const int64_t *topk_idx, int num_tokens,
                                                int num_topk, int num_experts, int num_ranks,
                                                int num_rdma_ranks, int32_t *tokens_per_expert,
                                                int32_t *tokens_per_rank,
                                                int32_t *tokens_per_rdma_rank,
                                                uint8_t *is_token_in_rank, int alignment,
                                                int32_t *expert_start_loc, int32_t *total_rows,
                                                void *workspace, int32_t *status,
                                                epd_stream_t stream);

/*
 * Step 2 -- expert offsets. [P2] "5. 缓冲区布局与发送" (the first source starts
 * at 0, each next one where the previous ended) and [P1] 2.2.4 (ep_scatter
 * scans, then scatters): expert_start_loc[e] = sum of tokens_per_expert[e'] for
 * e' < e; *total_rows (device int32) = the sum of all counts. A negative count
 * sets EPD_ERR_INVALID_ARG in *status.
 */
EPD_API epd_status_t ep_scan_offsets(const int32_t *tokens_per_expert, int num_experts,
                             int32_t *expert_start_loc, int32_t *total_rows, int32_t *status,
                             epd_stream_t stream);

/*
 * Step 2 with expert alignment (the grouped-GEMM contiguous layout). [P1] 3.3
 * and 4 (deepgemm_moe_permute pads every expert to block_m = 256 rows;
 * compute_aligned_M) and [P3] "Dispatch" (dispatch's expert_alignment): every
 * expert's region holds round_up(tokens_per_expert[e], alignment) rows;
 * expert_start_loc[e] = sum of the padded counts of e' < e, *total_rows = the sum
 * of all padded counts. alignment in [1, EPD_MAX_ALIGNMENT]; 1 gives
 * ep_scan_offsets. A buffer of round_up(T*k + E*(alignment-1), alignment) rows
 * always holds the padded regions. ep_permute fills them and marks the padding
 * rows with m_indices = -1.
 */
EPD_API epd_status_t ep_scan_offsets_aligned(const int32_t *tokens_per_expert, int num_experts,
                                             int alignment, int32_t *expert_start_loc,
                                             int32_t *total_rows, int32_t *status,
                                             epd_stream_t stream);

/*
 * Step 3 -- permute (ep_scatter). [P1] 2.2 (ep_scatter into input_tensor,
 * input_tensor_scale, m_indices, output_index) and 3.3 (m_indices pre-set to
 * -1 so that unwritten rows are skipped): for every pair (t, j) with expert
 * e = topk_idx[t, j] != -1, its slot is s = expert_start_loc[e] + (rank of the
 * pair inside e, from ep_dispatch_layout's workspace) and
 *   out[s, :]         = x[t, :]        (row bytes copied verbatim),
 *   out_scale[s, :]   = x_scale[t, :]  (fp8 only, H/128 floats),
 *   m_indices[s]      = e,
 *   output_index[t,j] = s;
 * pairs with no selection get output_index = -1, and m_indices[s] = -1 for
 * every row s in [0, capacity_rows) that no pair fills (alignment padding and
 * the rows after the last region). expert_start_loc may come from
 * ep_scan_offsets or ep_scan_offsets_aligned. Rows of out and out_scale that no
 * pair fills are not written.
 *   x:            [T, H] dtype rows, 16-byte aligned;
 *   x_scale:      [T, H/128] float32 for EPD_FP8_E4M3, NULL for EPD_BF16;
 *   out:          [capacity_rows, H] dtype, 16-byte aligned;
 *   out_scale:    [capacity_rows, H/128] float32 (fp8) or NULL (bf16);
 *   m_indices:    [capacity_rows] int32;  output_index: [T, k] int32;
 *   capacity_rows >= T*k (the exact-allocation upper bound with alignment 1;
 *   with aligned offsets it must also hold the padded regions),
 *   capacity_rows <= INT32_MAX.
 * `workspace` must hold the layout of the same topk_idx (same T and k); a
 * mismatch sets EPD_ERR_INVALID_ARG in *status and writes nothing.
 * Over the whole expert range the kernel asks L2 for up to 32 MB of x's first
 * rows before it waits for the previous kernel on the stream (a prefetch: it
 * changes no value any load returns), marked evict-last, and releases each line
 * (evict-first) when it reads the row.
 */
EPD_API epd_status_t ep_permute(const void *x, epd_dtype_t dtype, const float *x_scale,
                        const int64_t *topk_idx, int num_tokens, int num_topk, int hidden,
                        int num_experts, const int32_t *expert_start_loc, const void *workspace,
                        int64_t capacity_rows, void *out, float *out_scale, int32_t *m_indices,
                        int32_t *output_index, int32_t *status, epd_stream_t stream);

/*
 * Steps 1 to 3 in one call: the dispatch layout with its (aligned) offsets, then
 * the permute over the whole expert range with row-major scales -- exactly the
 * outputs of ep_dispatch_layout_offsets followed by ep_permute on the same
 * arguments, workspace state included. A small batch (T*k <= 4096, T <= 1024,
 * E <= 1024, R and N <= 64; a decode step) runs as one kernel in which every
 * block counts and scans the whole batch's picks itself and copies its own
 * tokens' rows; larger batches run the two kernels. Arguments, layouts and errors
 * as in those two calls; tokens_per_rdma_rank and is_token_in_rank may be NULL.
 * capacity_rows must hold the (aligned) total (a slot outside sets
 * EPD_ERR_CAPACITY). The pages have no single call for these steps (DeepEP
 * computes the layout in get_dispatch_layout before dispatch).
 */
EPD_API epd_status_t ep_dispatch(const void *x, epd_dtype_t dtype, const float *x_scale,
                                 const int64_t *topk_idx, int num_tokens, int num_topk,
                                 int hidden, int num_experts, int num_ranks, int num_rdma_ranks,
                                 int alignment, int32_t *tokens_per_expert,
                                 int32_t *tokens_per_rank, int32_t *tokens_per_rdma_rank,
                                 uint8_t *is_token_in_rank, int32_t *expert_start_loc,
                                 int32_t *total_rows, void *workspace, int64_t capacity_rows,
                                 void *out, float *out_scale, int32_t *m_indices,
                                 int32_t *output_index, int32_t *status, epd_stream_t stream);

/*
 * Output options of ep_permute_ex.
 *   expert_begin, expert_end: the view -- only pairs whose expert is in
 *     [expert_begin, expert_end) are placed (0 and num_experts for all
 *     experts). A simulated rank r of R holds [r*E/R, (r+1)*E/R). Rows are
 *     relative to the view's first region: a pair's row is
 *     expert_start_loc[e] - expert_start_loc[expert_begin] + its rank inside e,
 *     m_indices holds the local id e - expert_begin, and pairs outside the view
 *     get output_index = -1.
 *   scale_cols: 32-bit scale words per token (H/128 fp32 scales, or
 *     ceil(H/512) words of four packed UE8M0 exponent bytes); 0 for none.
 *   scale_col_major: 0 stores word c of row s at out_scale[s * scale_cols + c];
 *     1 stores it at out_scale[c * scale_ld + s] (column-major, the layout a
 *     TMA-fed grouped GEMM reads), scale_ld >= capacity_rows.
 */
typedef struct {
    int expert_begin;
    int expert_end;
    int scale_cols;
    int scale_col_major;
    int64_t scale_ld;
} epd_permute_view_t;

/*
 * Step 3 with output options: a per-rank view ([P1] 3.1.2 and 7: after dispatch
 * a rank's topk ids are local, rank_expert_offset maps them; [P1] 3.3:
 * deepgemm_moe_permute over local_num_experts) and scale layouts ([P1] 2.2:
 * UE8M0 scales as an int tensor [ceil(H/512), M] viewed transposed; [P3]
 * low_latency_dispatch docstring: scales column-major for TMA). Rows are any
 * row_bytes (a multiple of 16) copied verbatim; `view` is a host pointer.
 * capacity_rows must hold the view's regions (a slot outside sets
 * EPD_ERR_CAPACITY). Otherwise as ep_permute, which is this call with the whole
 * expert range and row-major fp32 scales. With column-major scales of more than
 * 16 words per row and a view of at least a quarter of the experts the call
 * enqueues two kernels: the row copy, which parks each filled row's source token
 * in m_indices, then a pass that writes the scales down their columns (coalesced)
 * and the final m_indices; m_indices is only meaningful once both have run.
 */
EPD_API epd_status_t ep_permute_ex(const void *x, int64_t row_bytes, const void *x_scale,
                                   const int64_t *topk_idx, int num_tokens, int num_topk,
                                   int num_experts, const int32_t *expert_start_loc,
                                   const void *workspace, int64_t capacity_rows,
                                   const epd_permute_view_t *view, void *out, void *out_scale,
                                   int32_t *m_indices, int32_t *output_index, int32_t *status,
                                   epd_stream_t stream);

/*
 * Low-latency dispatch layout with the fused cast. [P2] "3. 解决方案：固定矩形 vs.
 * 精确分配" strategy A (a fixed rectangle of rows per expert, sized for the worst
 * case, no count exchange first) and [P3] "low_latency模式" (low_latency_dispatch:
 * bf16 tokens cast to fp8 e4m3 on the way, one fp32 scale per 128 columns with
 * the last two dimensions column-major, recv_count, per-row source info).
 * Experts [expert_begin, expert_end) each own rows_per_expert rows; the r-th pick
 * of expert e in token-major order (the pair ranks ep_dispatch_layout left in
 * `workspace`) goes to row (e - expert_begin) * rows_per_expert + r -- no
 * ep_scan_offsets is needed. For every token with a pick in the view and every
 * 128-column block c:
 *   amax = max |x[t, 128c .. 128c+127]|, scale = amax / 448 (fp32; 1 if amax = 0),
 *   q = e4m3(x / scale), fp32 division, round to nearest even, saturating at 448,
 * written to every row the token goes to.
 *   x_bf16:    [T, H] bfloat16, H % 128 == 0, 16-byte aligned;
 *   out_q:     [E_view, rows_per_expert, H] e4m3 bytes, 8-byte aligned;
 *   out_scale: [E_view, H/128, rows_per_expert] float32;
 *   recv_count [E_view] int32: rows used per expert (at most rows_per_expert);
 *   output_index [T, k] int32: row of each pair, -1 for no pick, other experts,
 *     or a pick that found its rectangle full (EPD_ERR_CAPACITY in *status);
 *   src_token [E_view, rows_per_expert] int32: token of each used row; may be NULL.
 * Rows at and beyond recv_count are not written. ep_unpermute combines expert
 * outputs laid out in the same rectangles.
 */
EPD_API epd_status_t ep_permute_lowlatency(const void *x_bf16, const int64_t *topk_idx,
                                           int num_tokens, int num_topk, int hidden,
                                           int num_experts, int expert_begin, int expert_end,
                                           int64_t rows_per_expert, const void *workspace,
                                           void *out_q, float *out_scale, int32_t *recv_count,
                                           int32_t *output_index, int32_t *src_token,
                                           int32_t *status, epd_stream_t stream);

/*
 * The low-latency dispatch in one call: the same outputs as ep_dispatch_layout (its
 * pair ranks only) followed by ep_permute_lowlatency, without the layout's count
 * outputs ([P3] low_latency_dispatch returns recv_count, not a layout). A
 * decode-sized batch (T*k <= 4096, T <= 1024, E <= 1024, a block's bf16 rows
 * within 96 KiB) runs as one kernel in which every block ranks its own tokens'
 * picks against the batch itself -- a fixed rectangle needs no offsets -- and
 * casts its own rows; the workspace is then not touched. Larger batches run the
 * layout kernel (which needs `workspace` sized by epd_workspace_bytes(T, k, E, R,
 * N)) and then ep_permute_lowlatency. Arguments, layouts, results and errors as in
 * ep_permute_lowlatency.
 */
EPD_API epd_status_t ep_dispatch_lowlatency(const void *x_bf16, const int64_t *topk_idx,
                                            int num_tokens, int num_topk, int hidden,
                                            int num_experts, int num_ranks, int num_rdma_ranks,
                                            int expert_begin, int expert_end,
                                            int64_t rows_per_expert, void *workspace, void *out_q,
                                            float *out_scale, int32_t *recv_count,
                                            int32_t *output_index, int32_t *src_token,
                                            int32_t *status, epd_stream_t stream);

/*
 * Step 4 -- unpermute (combine). [P3] "Dispatch" (combine is the reverse of
 * dispatch; topk_weights are fp32 [T, k]):
 *   y[t, h] = bf16( sum over j with output_index[t, j] != -1, in j order, of
 *                   topk_weights[t, j] * expert_out[output_index[t, j], h] )
 * with every product and sum in fp32 (no fused multiply-add) and one
 * round-to-nearest-even to bf16. A token with no valid pair gets +0.
 *   expert_out:   [capacity_rows, H] bfloat16, 16-byte aligned;
 *   output_index: [T, k] int32 (from ep_permute); topk_weights: [T, k] float32;
 *   y:            [T, H] bfloat16, 16-byte aligned; H % 8 == 0.
 * A slot outside [-1, capacity_rows) sets EPD_ERR_CAPACITY and is skipped.
 */
EPD_API epd_status_t ep_unpermute(const void *expert_out, int64_t capacity_rows,
                          const int32_t *output_index, const float *topk_weights, int num_tokens,
                          int num_topk, int hidden, void *y, int32_t *status, epd_stream_t stream);

/*
 * Allocation-free variant of ep_dispatch_layout. The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory at
 * the moment they need the layout -- for example code running inside an
 * inference engine or plugin whose device memory is planned up front and
 * handed out by the host framework, or code that must not touch the allocator
 * on a hot serving path. Such callers own the inputs and outputs but have no
 * way to provide the workspace.
 *
 * It computes exactly what ep_dispatch_layout computes (tokens_per_expert,
 * tokens_per_rank, tokens_per_rdma_rank, is_token_in_rank, same arguments and
 * errors) but keeps its scratch -- the look-back state and the per-pair ranks --
 * in a file-scope device array of EPD_NOALLOC_SCRATCH_BYTES (8 MiB) inside
 * libepd. Every GPU that loads the library holds that array until the process
 * exits. The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *   - Sizes whose scratch need, epd_workspace_bytes(T, k, E, R, N), exceeds
 *     EPD_NOALLOC_SCRATCH_BYTES are rejected with EPD_ERR_UNSUPPORTED before
 *     anything is launched (T*k up to about 1.8 million pairs fits at E = 256,
 *     R = 32, N = 4, k = 8).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the previous call's contents.
 *     Nothing needs clearing between calls, whatever their shapes: every call
 *     leaves the tile ticket and finished-block count at zero, and the
 *     look-back only accepts state words tagged with the running call's
 *     counter, never an earlier call's ranks, counts or states. Calls in order
 *     on one stream are safe; calls that overlap on the GPU (other streams)
 *     race with each other.
 *   - The per-pair ranks it leaves in the shared array are not an input to
 *     ep_permute; a caller running the whole path uses ep_dispatch_layout with
 *     its own workspace.
 */
#define EPD_NOALLOC_SCRATCH_BYTES (8u << 20)

EPD_API epd_status_t ep_dispatch_layout_noalloc(const int64_t *topk_idx, int num_tokens,
                                                int num_topk, int num_experts, int num_ranks,
                                                int num_rdma_ranks, int32_t *tokens_per_expert,
                                                int32_t *tokens_per_rank,
                                                int32_t *tokens_per_rdma_rank,
                                                uint8_t *is_token_in_rank, int32_t *status,
                                                epd_stream_t stream);

/*
 * Test hook for failure detection, not part of the path: runs ep_dispatch_layout
 * in its tile form (whatever the batch size) with the look-back wait bounded by
 * `spin_limit` polls and with token tile
 * `stalled_tile` never publishing its state, so that every later tile's wait
 * runs out. The call still completes; *status then holds EPD_ERR_TIMEOUT and
 * the counts are meaningless. The workspace stays reusable afterwards.
 */
EPD_API epd_status_t epd_test_layout_stalled_tile(const int64_t *topk_idx, int num_tokens, int num_topk,
                                          int num_experts, int num_ranks, int num_rdma_ranks,
                                          int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                          int32_t *tokens_per_rdma_rank,
                                          uint8_t *is_token_in_rank, void *workspace,
                                          int32_t *status, int stalled_tile,
                                          uint32_t spin_limit, epd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EPD_H */
