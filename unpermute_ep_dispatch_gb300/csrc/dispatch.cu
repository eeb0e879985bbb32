// dispatch.cu -- steps 1 to 3 in one call: ep_dispatch.
//
// The same results as ep_dispatch_layout_offsets followed by ep_permute (whole
// expert range, row-major scales): "[MoE] Deepseek的All-to-all通信: DeepEP代码解读",
// section "Dispatch" (get_dispatch_layout: tokens per expert, rank and RDMA node,
// is_token_in_rank) and "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题",
// sections 2.2 and 3.3 (ep_scatter: offsets by prefix sum, rows and scales into
// the expert-contiguous buffer, m_indices, output_index).
//
// A small batch (a decode step: T*k up to 4096 pairs, T up to 1024, E up to 1024,
// R and N up to 64, a block's rows within 96 KiB) is one kernel, with no hand-off
// between blocks. Every block:
//   * bulk-loads its own tokens' rows into shared memory and their scale words
//     into registers right after the dependency wait, before anything else;
//   * reads the whole batch's picks into shared memory and counts them per expert,
//     and, apart, those that come before its own first pair;
//   * finds the ranks of its own tokens' pairs (a pair's rank inside its expert is
//     the number of earlier pairs, in row-major order, with the same expert): the
//     count before the block plus the block's own earlier pairs with that expert;
//   * scans the counts itself -- a few thousand pairs cost less than a second
//     kernel and the cross-block hand-off -- and so knows every offset;
//   * writes its slots, bulk-stores each row to its k slots, writes its slice of
//     m_indices and its tokens' is_token_in_rank rows;
//   * counts the batch's tokens per rank and per node from each token's bit masks
//     (a bit-matrix transpose of each warp's masks; every block counts the batch).
// Block 0 also writes all the counts, the offsets and the total, and leaves the
// workspace as the layout kernel would (header, counts, pair ranks), so a later
// ep_permute on the same workspace sees the same state. Larger batches run the
// layout and permute kernels.
#include <atomic>

#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kThreads = 256;
constexpr int kSmallPairs = 4096;     // T*k of the one-kernel form
constexpr int kSmallExperts = 1024;   // E of the one-kernel form
constexpr int kSmallTokens = 1024;    // T of the one-kernel form (block 0 counts every token)
constexpr int kSmallBlockPairs = 128; // pairs of one block's tokens
constexpr size_t kSmallRowBytes = 96 * 1024;  // shared memory for one block's rows
constexpr uint32_t kWaitLimit = 1u << 24;      // mbarrier polls before the row wait gives up

struct SmallArgs {
    const uint8_t *x;
    int64_t row_bytes;
    const uint32_t *x_scale;
    int scale_cols;
    const int64_t *topk;
    int T, k, E, R, N, epr, rpn, alignment;
    int rank_shift, node_shift;  // log2(E/R), log2(R/N) when powers of two, else -1
    int32_t *per_expert, *per_rank, *per_node;
    uint8_t *in_rank;
    int32_t *start_out, *total_out;
    WsHeader *hdr;
    int32_t *pair_rank, *ws_counts;
    int64_t capacity;
    uint8_t *out;
    uint32_t *out_scale;
    int32_t *m_indices, *output_index, *status;
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Shared memory of the one-kernel form beyond its static arrays: the block's rows.
__host__ __device__ inline size_t small_row_stride(int64_t row_bytes) {
    return align_up((size_t)row_bytes, 128);
}

__global__ void __launch_bounds__(kThreads) small_dispatch_kernel(SmallArgs a) {
    extern __shared__ __align__(128) uint8_t s_rows[];  // [tokens of the block][row stride]
    __shared__ int16_t s_e[kSmallPairs];    // expert of every pair of the batch, -1 = none
    __shared__ int s_cnt[kSmallExperts];    // pairs per expert
    __shared__ int s_before[kSmallExperts]; // pairs per expert before this block's first pair
    __shared__ int s_start[kSmallExperts];  // (aligned) offsets
    __shared__ uint8_t s_rank_of[kSmallExperts], s_node_of[64];
    __shared__ int s_rank[kSmallBlockPairs];
    __shared__ int s_total, s_pairs;
    __shared__ bool s_rows_ok;
    __shared__ int s_col[128];  // the batch's tokens per rank [0, R) and per node [64, 64 + N)
    __shared__ __align__(8) uint64_t s_bar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P_all = a.T * a.k;
    const int t_begin = (int)((int64_t)a.T * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)a.T * (blockIdx.x + 1) / gridDim.x);
    const int nt = t_end - t_begin;
    const size_t stride = small_row_stride(a.row_bytes);
    const bool copy = a.k > 0 && nt > 0;
    for (int e = tid; e < a.E; e += kThreads) {
        s_cnt[e] = 0;
        s_before[e] = 0;
        s_rank_of[e] = (uint8_t)(e / a.epr);
    }
    for (int r = tid; r < a.R; r += kThreads) s_node_of[r] = (uint8_t)(r / a.rpn);
    for (int i = tid; i < 128; i += kThreads) s_col[i] = 0;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init_fence();
    }
    pdl_wait();  // topk_idx and the rows may come from the previous kernel

    // the block's rows, by bulk copy into shared memory: they depend on nothing
    if (tid == 0 && copy) {
        mbar_expect_tx(&s_bar, (uint32_t)(nt * a.row_bytes));
        for (int tl = 0; tl < nt; ++tl)
            bulk_load(s_rows + tl * stride, a.x + (int64_t)(t_begin + tl) * a.row_bytes,
                      (uint32_t)a.row_bytes, &s_bar);
    }
    // and their scale words, into the registers of warps 1 and 2 (which store them)
    const int nsc = a.k > 0 ? nt * a.scale_cols : 0;
    uint32_t sc = 0;
    if (tid >= 32 && tid < 96 && tid - 32 < nsc)
        sc = a.x_scale[(int64_t)t_begin * a.scale_cols + tid - 32];

    // the batch's picks: all of a thread's loads are issued first (one round trip, not
    // one per pick), then parked in shared memory and counted per expert, and those
    // before this block's first pair once more (the base of its pairs' ranks); ids
    // outside [-1, E) are reported (by block 0) and skipped
    const int p0 = t_begin * a.k, q_end = nt * a.k;
    constexpr int kPicksPerThread = kSmallPairs / kThreads;
    int64_t pv[kPicksPerThread];
#pragma unroll
    for (int i = 0; i < kPicksPerThread; ++i) {
        const int p = tid + i * kThreads;
        pv[i] = p < P_all ? __ldg(a.topk + p) : -1;
    }
#pragma unroll
    for (int i = 0; i < kPicksPerThread; ++i) {
        const int p = tid + i * kThreads;
        if (p >= P_all) break;
        const int64_t v = pv[i];
        const bool ok = v >= 0 && v < a.E;
        if ((v < -1 || v >= a.E) && blockIdx.x == 0) report(a.status, EPD_ERR_INVALID_EXPERT);
        s_e[p] = ok ? (int16_t)v : (int16_t)-1;
        if (ok) {
            atomicAdd(&s_cnt[(int)v], 1);
            if (p < p0) atomicAdd(&s_before[(int)v], 1);
        }
    }
    __syncthreads();

    // warp 0: exclusive prefix sum of the (aligned) counts, each lane a contiguous run
    // of up to 32 experts, then a shuffle scan of the runs. Meanwhile one thread per
    // pair of this block: its rank inside its expert (the number of earlier pairs of
    // the batch with the same expert) is the count before the block plus the block's
    // own earlier pairs with that expert.
    if (warp == 0) {
        const int per = (a.E + 31) / 32;
        const int e0 = min(a.E, lane * per), e1 = min(a.E, e0 + per);
        const int A = a.alignment;
        auto padded = [A](int c) { return A == 1 ? c : (c + A - 1) / A * A; };
        int run = 0, pairs = 0;
        for (int e = e0; e < e1; ++e) {
            const int c = s_cnt[e];
            pairs += c;
            run += padded(c);
        }
        const int incl = warp_incl_scan(run, lane);
        pairs = warp_sum(pairs);
        int pos = incl - run;
        for (int e = e0; e < e1; ++e) {
            s_start[e] = pos;
            pos += padded(s_cnt[e]);
        }
        if (lane == 31) {
            s_total = incl;
            s_pairs = pairs;
        }
    } else {
        for (int q = tid - 32; q < q_end; q += kThreads - 32) {
            const int e = s_e[p0 + q];
            int r = 0;
            if (e >= 0) {
                r = s_before[e];
                for (int q2 = 0; q2 < q; ++q2) r += s_e[p0 + q2] == e;
            }
            s_rank[q] = r;
        }
    }
    __syncthreads();

    // the slot of this block's pair q (-1 for no pick, or past the buffer); every warp
    // that needs slots computes them itself, so no barrier separates them from the
    // copies
    auto slot_of = [&](int q) {
        const int e = s_e[p0 + q];
        if (e < 0) return -1;
        const int64_t sl = (int64_t)s_start[e] + s_rank[q];
        return sl < a.capacity ? (int)sl : -1;
    };

    // warp 0 writes the block's slots (output_index and the workspace's pair ranks)
    // and moves the rows: once they have landed, lane i issues the bulk stores of
    // pairs i, i + 32, ... from shared memory. Meanwhile warps 1 and 2 copy the scale
    // words (the ones loaded at the start), warp 3 writes this block's slice of
    // m_indices, and warps 4..7 build the batch's token masks, write this block's
    // is_token_in_rank rows and count the batch's tokens per rank and per node.
    bool issued = false;  // this lane of warp 0 has bulk stores in flight
    if (warp == 0) {
        constexpr int kPerLane = kSmallBlockPairs / 32;
        int sl[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int q = lane + 32 * i;
            sl[i] = -1;
            if (q < q_end) {
                const int e = s_e[p0 + q];
                sl[i] = slot_of(q);
                if (e >= 0 && sl[i] < 0) report(a.status, EPD_ERR_CAPACITY);
                a.output_index[p0 + q] = sl[i];
                a.pair_rank[p0 + q] = e >= 0 ? s_rank[q] : -1;
            }
        }
        bool landed = true;
        if (copy) {
            if (lane == 0) landed = mbar_wait_bounded(&s_bar, 0u, kWaitLimit);
            landed = __shfl_sync(0xffffffffu, landed, 0);
            if (lane == 0) {
                s_rows_ok = landed;
                if (!landed) report(a.status, EPD_ERR_TIMEOUT);
            }
            if (landed) {
                fence_proxy_async_smem();
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    const int q = lane + 32 * i;
                    if (q >= q_end || sl[i] < 0) continue;
                    bulk_store(a.out + (int64_t)sl[i] * a.row_bytes, s_rows + (q / a.k) * stride,
                               (uint32_t)a.row_bytes);
                    issued = true;
                }
                if (issued) bulk_commit();
            }
        }
    } else if (warp <= 2) {
        const int wt = tid - 32;
        for (int i = wt; i < nsc; i += 64) {  // the first word of each thread is in sc
            const int tl = i / a.scale_cols, c = i - tl * a.scale_cols;
            const uint32_t v = i == wt ? sc : a.x_scale[(int64_t)t_begin * a.scale_cols + i];
            for (int j = 0; j < a.k; ++j) {
                const int s = slot_of(tl * a.k + j);
                if (s >= 0) a.out_scale[(int64_t)s * a.scale_cols + c] = v;
            }
        }
    } else if (warp == 3) {
        // row s belongs to the last expert whose region starts at or before s, and
        // holds it when it is among the region's first count rows (else -1: padding
        // or rows past the last region)
        const int64_t m0 = a.capacity * blockIdx.x / gridDim.x;
        const int64_t m1 = a.capacity * (blockIdx.x + 1) / gridDim.x;
        for (int64_t s = m0 + lane; s < m1; s += 32) {
            int lo = 0, hi = a.E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((int64_t)s_start[mid] <= s) lo = mid;
                else hi = mid - 1;
            }
            const int64_t st = s_start[lo];
            a.m_indices[s] = (s >= st && s < st + s_cnt[lo]) ? lo : -1;
        }
    } else {
        // warps 4..7, one lane per token of the batch: the token's rank and node bit
        // masks from its picks (R, N <= 64 in this form); its is_token_in_rank row when
        // it is one of this block's tokens; and the batch's tokens per rank and per node
        // by counting the columns of each warp's masks. Every block counts the whole
        // batch (a few hundred tokens); block 0 writes the counts.
        const bool words = (a.R & 3) == 0 && (reinterpret_cast<uintptr_t>(a.in_rank) & 3) == 0;
        const bool fastm = a.rank_shift >= 0 && a.node_shift >= 0 && a.R <= 32 && a.N <= 32;
        for (int t0 = (warp - 4) * 32; t0 < a.T; t0 += 128) {
            const int t = t0 + lane;
            unsigned long long rm = 0, nm = 0;
            if (t < a.T) {
                const int16_t *row = s_e + t * a.k;
                if (fastm) {  // shifts, 32-bit masks
                    const int rs = a.rank_shift, ns = a.node_shift;
                    uint32_t r32 = 0u, n32 = 0u;
                    for (int j = 0; j < a.k; ++j) {
                        const int e = row[j];
                        const int r = e >> rs;
                        r32 |= e >= 0 ? 1u << r : 0u;
                        n32 |= e >= 0 ? 1u << (r >> ns) : 0u;
                    }
                    rm = r32;
                    nm = n32;
                } else {
                    for (int j = 0; j < a.k; ++j) {
                        const int e = row[j];
                        if (e < 0) continue;
                        const int r = s_rank_of[e];
                        rm |= 1ull << r;
                        nm |= 1ull << s_node_of[r];
                    }
                }
                if (a.in_rank && t >= t_begin && t < t_end) {
                    uint8_t *dst = a.in_rank + (int64_t)t * a.R;
                    if (words) {
                        for (int w4 = 0; w4 < (a.R >> 2); ++w4)
                            reinterpret_cast<int *>(dst)[w4] = spread4((uint32_t)(rm >> (4 * w4)));
                    } else {
                        for (int r = 0; r < a.R; ++r) dst[r] = (uint8_t)((rm >> r) & 1ull);
                    }
                }
            }
            for (int g = 0; g < 2; ++g) {
                if (32 * g < a.R) {
                    const int c = bit_column_count((uint32_t)(rm >> (32 * g)), lane);
                    if (c) atomicAdd(&s_col[32 * g + lane], c);
                }
                if (a.per_node && 32 * g < a.N) {
                    const int c = bit_column_count((uint32_t)(nm >> (32 * g)), lane);
                    if (c) atomicAdd(&s_col[64 + 32 * g + lane], c);
                }
            }
        }
    }
    __syncthreads();

    // block 0: per-expert, per-rank and per-node counts, offsets and total, and the
    // workspace header and counts
    if (blockIdx.x == 0) {
        for (int c = tid; c < a.R; c += kThreads) a.per_rank[c] = s_col[c];
        if (a.per_node)
            for (int c = tid; c < a.N; c += kThreads) a.per_node[c] = s_col[64 + c];
        for (int e = tid; e < a.E; e += kThreads) {
            a.per_expert[e] = s_cnt[e];
            a.ws_counts[e] = s_cnt[e];
            a.start_out[e] = s_start[e];
        }
        if (tid == 0) {
            *a.total_out = s_total;
            a.hdr->total_pairs = s_pairs;
            a.hdr->num_tokens = a.T;
            a.hdr->num_topk = a.k;
        }
    }
    // the bulk stores read shared memory until they have read it (their writes then
    // complete on their own: the grid's completion covers them); loads that outlived
    // a wait that gave up land before the block's shared memory is released
    if (issued) bulk_wait_read<0>();
    if (tid == 0 && copy && !s_rows_ok) mbar_wait_bounded(&s_bar, 0u, kWaitLimit);
    pdl_trigger();
}

}  // namespace
}  // namespace epd

extern "C" epd_status_t ep_dispatch(const void *x, epd_dtype_t dtype, const float *x_scale,
                                    const int64_t *topk_idx, int num_tokens, int num_topk,
                                    int hidden, int num_experts, int num_ranks,
                                    int num_rdma_ranks, int alignment, int32_t *tokens_per_expert,
                                    int32_t *tokens_per_rank, int32_t *tokens_per_rdma_rank,
                                    uint8_t *is_token_in_rank, int32_t *expert_start_loc,
                                    int32_t *total_rows, void *workspace, int64_t capacity_rows,
                                    void *out, float *out_scale, int32_t *m_indices,
                                    int32_t *output_index, int32_t *status, epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk, H = hidden, E = num_experts;
    const int R = num_ranks, N = num_rdma_ranks;
    if (!topology_ok(T, k, E, R, N) || H <= 0) return EPD_ERR_INVALID_ARG;
    if (alignment < 1 || alignment > EPD_MAX_ALIGNMENT) return EPD_ERR_INVALID_ARG;
    if (capacity_rows < (int64_t)T * k || capacity_rows > INT32_MAX) return EPD_ERR_INVALID_ARG;
    int64_t row_bytes;
    int scale_cols;
    if (dtype == EPD_BF16) {
        if (H % 8 != 0 || x_scale != nullptr || out_scale != nullptr) return EPD_ERR_INVALID_ARG;
        row_bytes = 2 * (int64_t)H;
        scale_cols = 0;
    } else if (dtype == EPD_FP8_E4M3) {
        if (H % 128 != 0) return EPD_ERR_INVALID_ARG;
        if (((int64_t)T * k > 0 && x_scale == nullptr) || (capacity_rows > 0 && out_scale == nullptr))
            return EPD_ERR_INVALID_ARG;
        if (!aligned4(x_scale) || !aligned4(out_scale)) return EPD_ERR_INVALID_ARG;
        row_bytes = H;
        scale_cols = H / 128;
    } else {
        return EPD_ERR_INVALID_ARG;
    }
    if (!tokens_per_expert || !tokens_per_rank || !expert_start_loc || !total_rows || !workspace ||
        !status)
        return EPD_ERR_INVALID_ARG;
    if (!aligned4(tokens_per_expert) || !aligned4(tokens_per_rank) ||
        (tokens_per_rdma_rank && !aligned4(tokens_per_rdma_rank)) || !aligned4(expert_start_loc) ||
        !aligned4(total_rows) || !aligned16(workspace) || !aligned4(status))
        return EPD_ERR_INVALID_ARG;
    if (capacity_rows > 0 && (!m_indices || !aligned4(m_indices))) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 &&
        (!x || !topk_idx || !out || !output_index || !aligned16(x) || !aligned16(out) ||
         !aligned8(topk_idx) || !aligned4(output_index)))
        return EPD_ERR_INVALID_ARG;

    const int grid_cap = 2 * sm_count();
    const int grid = T < 1 ? 1 : (T < grid_cap ? T : grid_cap);
    const int tokens_per_block = T > 0 ? (T + grid - 1) / grid : 0;
    const size_t smem = (size_t)tokens_per_block * small_row_stride(row_bytes);
    const bool small = (int64_t)T * k <= kSmallPairs && T <= kSmallTokens && E <= kSmallExperts &&
                       R <= 64 && N <= 64 && (int64_t)tokens_per_block * k <= kSmallBlockPairs &&
                       smem <= kSmallRowBytes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!small) {
        const epd_status_t st = ep_dispatch_layout_offsets(
            topk_idx, T, k, E, R, N, tokens_per_expert, tokens_per_rank, tokens_per_rdma_rank,
            is_token_in_rank, alignment, expert_start_loc, total_rows, workspace, status, stream);
        if (st != EPD_OK) return st;
        return ep_permute(x, dtype, x_scale, topk_idx, T, k, H, E, expert_start_loc, workspace,
                          capacity_rows, out, out_scale, m_indices, output_index, status, stream);
    }
    char *ws = static_cast<char *>(workspace);
    SmallArgs a;
    a.x = static_cast<const uint8_t *>(x);
    a.row_bytes = row_bytes;
    a.x_scale = reinterpret_cast<const uint32_t *>(x_scale);
    a.scale_cols = scale_cols;
    a.topk = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.R = R;
    a.N = N;
    a.epr = E / R;
    auto log2_exact = [](int v) {
        int b = 0;
        while ((1 << b) < v) ++b;
        return (1 << b) == v ? b : -1;
    };
    a.rank_shift = log2_exact(E / R);
    a.node_shift = log2_exact(R / N);
    a.rpn = R / N;
    a.alignment = alignment;
    a.per_expert = tokens_per_expert;
    a.per_rank = tokens_per_rank;
    a.per_node = tokens_per_rdma_rank;
    a.in_rank = is_token_in_rank;
    a.start_out = expert_start_loc;
    a.total_out = total_rows;
    a.hdr = reinterpret_cast<WsHeader *>(ws);
    a.pair_rank = reinterpret_cast<int32_t *>(ws + ws_pair_rank_off());
    a.ws_counts = reinterpret_cast<int32_t *>(ws + ws_counts_off(T, k));
    a.capacity = capacity_rows;
    a.out = static_cast<uint8_t *>(out);
    a.out_scale = reinterpret_cast<uint32_t *>(out_scale);
    a.m_indices = m_indices;
    a.output_index = output_index;
    a.status = status;
    // the static arrays and up to kSmallRowBytes of rows exceed the default 48 KiB
    // limit: opt in once per device
    static std::atomic<bool> opted[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return record_cuda_error();
    if (dev < 0 || dev >= 64 || !opted[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(small_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmallRowBytes) != cudaSuccess)
            return record_cuda_error();
        if (dev >= 0 && dev < 64) opted[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(small_dispatch_kernel, grid, kThreads, smem, s, a);
}
