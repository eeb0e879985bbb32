// lowlatency.cu -- the fixed-rectangle (low-latency) dispatch layout with the
// fused bf16 -> fp8 cast.
//
// "高性能专家并行（EP）内核解剖学解读", section "3. 解决方案：固定矩形 vs. 精确分配",
// strategy A: every expert owns a fixed rectangle of rows sized for the worst
// case, so no count has to be exchanged before the rows move.
// "[MoE] Deepseek的All-to-all通信: DeepEP代码解读", section "low_latency模式"
// (low_latency_dispatch): bf16 tokens are cast to fp8 on the way, one fp32 scale
// per 128 columns, the scales' last two dimensions column-major, recv_count per
// expert and the source of every received row.
//
// The r-th pick of expert e (token-major order: the pair ranks left in the
// workspace by ep_dispatch_layout) goes to row (e - e_begin) * rows + r; no
// offset scan is needed. Work units are (token, two 128-column blocks); a
// half-warp owns one block: 16-byte bf16 loads, the block's absolute maximum by
// half-warp shuffles, scale = amax / 448 and q = e4m3(x / scale) with IEEE
// divisions and the saturating round-to-nearest-even conversion, then 8-byte
// stores of the quantised block to each row the token goes to. Each warp checks
// the workspace header itself and issues the loads that do not depend on a slot
// (the header, the picks and their ranks, and over wide views the row) before its
// first store.
#include <cuda_fp8.h>

#include <atomic>

#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct LLArgs {
    const uint8_t *x;  // bf16 [T, H]
    int T, k, H, E, e_begin, e_end;
    int64_t rows;      // rows per expert rectangle
    const int64_t *topk;
    const int32_t *pair_rank;
    const int32_t *counts;
    const WsHeader *hdr;
    uint8_t *out_q;      // e4m3 [E_view, rows, H]
    float *out_scale;    // [E_view, H/128, rows]
    int32_t *recv_count;
    int32_t *output_index;
    int32_t *src_token;  // [E_view, rows] or null
    int32_t *status;
};

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void __launch_bounds__(kThreads) lowlatency_kernel(LLArgs a) {
    __shared__ int s_row[kWarps][EPD_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();  // pair ranks and counts come from the layout kernel
    // Each warp checks the workspace header itself, and every load that does not
    // depend on a slot (the header, the row, the picks and their ranks) is issued
    // before the first store, which waits for the header check's result.
    int hdr_ok = 0;
    if (lane == 0) hdr_ok = a.hdr->num_tokens == a.T && a.hdr->num_topk == a.k;
    bool checked = false;

    const int C = a.H >> 7;                // 128-column blocks per row
    const int upt = (C + 1) >> 1;          // units (block pairs) per token
    const int64_t units = (int64_t)a.T * upt;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u_end = units * (gw + 1) / nw;
    const int half = lane >> 4, hl = lane & 15;
    // rows are loaded before their slots are known over views of at least a quarter
    // of the experts (nearly every token is copied); a narrow view copies few tokens
    // and loads a row only once it has a slot
    const bool early = a.k > 0 && 4 * (a.e_end - a.e_begin) >= a.E;
    int cur_t = -1;
    bool any = false;
    for (int64_t u = units * gw / nw; u < u_end; ++u) {
        const int t = (int)(u / upt);
        const int ch = (int)(u - (int64_t)t * upt);
        const int c = 2 * ch + half;       // this half-warp's block
        const bool active = c < C;
        const uint8_t *src = a.x + ((int64_t)t * a.H + 128 * c + 8 * hl) * 2;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (active && early) raw = ld_stream16(src);
        if (t != cur_t) {
            cur_t = t;
            int64_t pe[2];
            int32_t pr[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {  // k <= 64: at most two picks per lane
                const int j = lane + 32 * q;
                pe[q] = -1;
                pr[q] = -1;
                if (j < a.k) {
                    const int64_t idx = (int64_t)t * a.k + j;
                    pe[q] = a.topk[idx];
                    pr[q] = a.pair_rank[idx];
                }
            }
            if (!checked) {
                checked = true;
                if (!__shfl_sync(0xffffffffu, hdr_ok, 0)) {
                    if (blockIdx.x == 0 && threadIdx.x == 0) report(a.status, EPD_ERR_INVALID_ARG);
                    return;
                }
            }
            int has = 0;
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int j = lane + 32 * q;
                if (j >= a.k) continue;
                const int64_t idx = (int64_t)t * a.k + j;
                const int64_t e = pe[q];
                int row = -1;
                if (e >= a.e_begin && e < a.e_end) {
                    const int64_t r = pr[q];
                    if (r >= 0 && r < a.rows) {
                        row = (int)((e - a.e_begin) * a.rows + r);
                        if (ch == 0 && a.src_token) a.src_token[row] = t;
                    } else if (ch == 0) {
                        report(a.status, EPD_ERR_CAPACITY);  // the rectangle is full
                    }
                }
                if (ch == 0) a.output_index[idx] = row;
                s_row[warp][j] = row;
                has |= (row >= 0);
            }
            any = __any_sync(0xffffffffu, has);
            __syncwarp();
        }
        if (!any) continue;
        if (active && !early) raw = ld_stream16(src);
        float v[8];
        float amax = 0.0f;
        if (active) {
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (!active) continue;
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        uint2 q;
        q.x = e4m3x4(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale), __fdiv_rn(v[2], scale),
                     __fdiv_rn(v[3], scale));
        q.y = e4m3x4(__fdiv_rn(v[4], scale), __fdiv_rn(v[5], scale), __fdiv_rn(v[6], scale),
                     __fdiv_rn(v[7], scale));
        for (int j = 0; j < a.k; ++j) {
            const int row = s_row[warp][j];
            if (row < 0) continue;
            *reinterpret_cast<uint2 *>(a.out_q + (int64_t)row * a.H + 128 * c + 8 * hl) = q;
            if (hl == 0) {
                const int64_t el = row / a.rows, r = row - el * a.rows;
                a.out_scale[(el * C + c) * a.rows + r] = scale;
            }
        }
    }
    // recv_count by block 0 (after its warps' units: off the path of the rows)
    if (blockIdx.x == 0 && __shfl_sync(0xffffffffu, hdr_ok, 0))
        for (int e = threadIdx.x; e < a.e_end - a.e_begin; e += kThreads) {
            const int64_t c = a.counts[a.e_begin + e];
            a.recv_count[e] = (int32_t)(c < a.rows ? c : a.rows);
        }
    pdl_trigger();
}

// ----------------------------------------------------------------------------- one kernel
// ep_dispatch_lowlatency for a decode-sized batch: no layout kernel. Blocks
// (x, y) share the token run x: every one reads the batch's picks into shared
// memory and ranks the run's pairs (the number of earlier pairs, in row-major
// order, with the same expert: the picks before the run are counted per expert as
// they are parked), which is all a fixed rectangle needs; it
// bulk-loads the run's bf16 rows into shared memory as it starts and casts the
// units (token, two 128-column blocks) u = y, y + gridDim.y, ... from there. Blocks
// with y = 0 write output_index and src_token; block (0, 0) counts the view's
// experts for recv_count.
constexpr int kLLSmallPairs = 4096;
constexpr int kLLSmallExperts = 1024;
constexpr int kLLSmallTokens = 1024;
constexpr int kLLSmallBlockPairs = 128;
constexpr size_t kLLSmallRowBytes = 96 * 1024;
constexpr uint32_t kLLWaitLimit = 1u << 24;

struct LLSmallArgs {
    const uint8_t *x;  // bf16 [T, H]
    int T, k, H, E, e_begin, e_end;
    int64_t rows;
    const int64_t *topk;
    uint8_t *out_q;
    float *out_scale;
    int32_t *recv_count, *output_index, *src_token, *status;
};

__host__ __device__ inline size_t ll_row_stride(int H) { return align_up((size_t)H * 2, 128); }

__global__ void __launch_bounds__(kThreads) lowlatency_small_kernel(LLSmallArgs a) {
    extern __shared__ __align__(128) uint8_t s_x[];  // the block's bf16 rows
    __shared__ int16_t s_e[kLLSmallPairs];
    __shared__ int s_cnt[kLLSmallExperts];            // block 0: picks per expert of the view
    __shared__ int s_before[kLLSmallExperts];         // picks per expert before the run's first
    __shared__ int s_rank[kLLSmallBlockPairs], s_row[kLLSmallBlockPairs];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_ok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P_all = a.T * a.k;
    const int EV = a.e_end - a.e_begin;
    const int t_begin = (int)((int64_t)a.T * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)a.T * (blockIdx.x + 1) / gridDim.x);
    const int nt = t_end - t_begin;
    const size_t stride = ll_row_stride(a.H);
    const bool copy = a.k > 0 && nt > 0;
    const bool lead = blockIdx.y == 0;                  // writes the run's indices
    const bool first = lead && blockIdx.x == 0;         // writes recv_count
    if (first)
        for (int e = tid; e < EV; e += kThreads) s_cnt[e] = 0;
    for (int e = tid; e < a.E; e += kThreads) s_before[e] = 0;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init_fence();
    }
    pdl_wait();  // topk_idx and the rows may come from the previous kernel

    if (tid == 0 && copy) {
        const uint32_t bytes = (uint32_t)a.H * 2;
        mbar_expect_tx(&s_bar, (uint32_t)nt * bytes);
        for (int tl = 0; tl < nt; ++tl)
            bulk_load(s_x + tl * stride, a.x + (int64_t)(t_begin + tl) * bytes, bytes, &s_bar);
    }
    // the batch's picks: all of a thread's loads are issued first (one round trip),
    // then parked in shared memory; those before the run's first pair are counted per
    // expert (the base of the run's ranks)
    const int p0 = t_begin * a.k, q_end = nt * a.k;
    constexpr int kPicksPerThread = kLLSmallPairs / kThreads;
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
        if ((v < -1 || v >= a.E) && first) report(a.status, EPD_ERR_INVALID_EXPERT);
        s_e[p] = ok ? (int16_t)v : (int16_t)-1;
        if (ok && p < p0) atomicAdd(&s_before[(int)v], 1);
    }
    __syncthreads();
    if (first)
        for (int p = tid; p < P_all; p += kThreads) {
            const int e = s_e[p];
            if (e >= a.e_begin && e < a.e_end) atomicAdd(&s_cnt[e - a.e_begin], 1);
        }
    // ranks of the run's pairs (the view's picks only get rows): the count before the
    // run plus the run's own earlier pairs with the same expert
    for (int q = tid; q < q_end; q += kThreads) {
        const int e = s_e[p0 + q];
        int r = 0;
        if (e >= a.e_begin && e < a.e_end) {
            r = s_before[e];
            for (int q2 = 0; q2 < q; ++q2) r += s_e[p0 + q2] == e;
        }
        s_rank[q] = r;
    }
    __syncthreads();
    // rows in the rectangles; a pick past its rectangle is dropped and reported
    for (int q = tid; q < q_end; q += kThreads) {
        const int p = p0 + q;
        const int e = s_e[p];
        int row = -1;
        if (e >= a.e_begin && e < a.e_end) {
            const int64_t r = s_rank[q];
            if (r < a.rows) {
                row = (int)((e - a.e_begin) * a.rows + r);
                if (lead && a.src_token) a.src_token[row] = t_begin + q / a.k;
            } else if (lead) {
                report(a.status, EPD_ERR_CAPACITY);
            }
        }
        if (lead) a.output_index[p] = row;
        s_row[q] = row;
    }
    if (first) {
        __syncthreads();
        for (int e = tid; e < EV; e += kThreads) {
            const int64_t c = s_cnt[e];
            a.recv_count[e] = (int32_t)(c < a.rows ? c : a.rows);
        }
    }
    // the rows have landed (every thread observes the barrier before reading them)
    if (tid == 0) s_ok = 1;
    __syncthreads();
    if (copy && !mbar_wait_bounded(&s_bar, 0u, kLLWaitLimit)) {
        if (tid == 0) report(a.status, EPD_ERR_TIMEOUT);
        s_ok = 0;
    }
    __syncthreads();
    // cast: units of (token, two 128-column blocks), a half-warp per block
    const int C = a.H >> 7, upt = (C + 1) >> 1;
    const int half = lane >> 4, hl = lane & 15;
    if (s_ok && copy)
        for (int u = blockIdx.y * kWarps + warp; u < nt * upt; u += gridDim.y * kWarps) {
            const int tl = u / upt, ch = u - tl * upt;
            const int c = 2 * ch + half;
            const int *rows = s_row + tl * a.k;
            bool any = false;
            for (int j = 0; j < a.k; ++j) any |= rows[j] >= 0;
            if (!any) continue;  // warp-uniform: the token has no row in the view
            const bool active = c < C;
            float v[8];
            float amax = 0.0f;
            if (active) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(s_x + tl * stride + (128 * c + 8 * hl) * 2);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(w[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (!active) continue;
            const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
            uint2 qv;
            qv.x = e4m3x4(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale), __fdiv_rn(v[2], scale),
                          __fdiv_rn(v[3], scale));
            qv.y = e4m3x4(__fdiv_rn(v[4], scale), __fdiv_rn(v[5], scale), __fdiv_rn(v[6], scale),
                          __fdiv_rn(v[7], scale));
            for (int j = 0; j < a.k; ++j) {
                const int row = rows[j];
                if (row < 0) continue;
                *reinterpret_cast<uint2 *>(a.out_q + (int64_t)row * a.H + 128 * c + 8 * hl) = qv;
                if (hl == 0) {
                    const int64_t el = row / a.rows, r = row - el * a.rows;
                    a.out_scale[(el * C + c) * a.rows + r] = scale;
                }
            }
        }
    // loads that outlived a wait that gave up land before shared memory is released
    if (tid == 0 && copy && !s_ok) mbar_wait_bounded(&s_bar, 0u, kLLWaitLimit);
    pdl_trigger();
}

}  // namespace
}  // namespace epd

extern "C" epd_status_t ep_permute_lowlatency(const void *x_bf16, const int64_t *topk_idx,
                                              int num_tokens, int num_topk, int hidden,
                                              int num_experts, int expert_begin, int expert_end,
                                              int64_t rows_per_expert, const void *workspace,
                                              void *out_q, float *out_scale, int32_t *recv_count,
                                              int32_t *output_index, int32_t *src_token,
                                              int32_t *status, epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk, H = hidden, E = num_experts;
    if (T < 0 || k < 0 || k > EPD_MAX_TOPK || E < 1 || E > EPD_MAX_EXPERTS) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > INT32_MAX || H < 128 || H % 128 != 0) return EPD_ERR_INVALID_ARG;
    if (expert_begin < 0 || expert_end > E || expert_begin >= expert_end) return EPD_ERR_INVALID_ARG;
    const int64_t EV = expert_end - expert_begin;
    if (rows_per_expert < 0 || EV * rows_per_expert > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if (!workspace || !recv_count || !status || !aligned16(workspace) || !aligned4(recv_count) ||
        !aligned4(status))
        return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (!x_bf16 || !topk_idx || !output_index)) return EPD_ERR_INVALID_ARG;
    if (EV * rows_per_expert > 0 && (!out_q || !out_scale)) return EPD_ERR_INVALID_ARG;
    if ((x_bf16 && !aligned16(x_bf16)) || (topk_idx && !aligned8(topk_idx)) ||
        (out_q && !aligned8(out_q)) || !aligned4(out_scale) || !aligned4(output_index) ||
        !aligned4(src_token))
        return EPD_ERR_INVALID_ARG;
    const char *ws = static_cast<const char *>(workspace);
    LLArgs a;
    a.x = static_cast<const uint8_t *>(x_bf16);
    a.T = T;
    a.k = k;
    a.H = H;
    a.E = E;
    a.e_begin = expert_begin;
    a.e_end = expert_end;
    a.rows = rows_per_expert;
    a.topk = topk_idx;
    a.pair_rank = reinterpret_cast<const int32_t *>(ws + ws_pair_rank_off());
    a.counts = reinterpret_cast<const int32_t *>(ws + ws_counts_off(T, k));
    a.hdr = reinterpret_cast<const WsHeader *>(ws);
    a.out_q = static_cast<uint8_t *>(out_q);
    a.out_scale = out_scale;
    a.recv_count = recv_count;
    a.output_index = output_index;
    a.src_token = src_token;
    a.status = status;
    static const int resident = blocks_per_sm(lowlatency_kernel, kThreads, 0);
    const int64_t units = (int64_t)T * ((H / 128 + 1) / 2);
    const int64_t want = (units + kWarps - 1) / kWarps;
    const int64_t full = (int64_t)sm_count() * resident;
    const int grid = (int)(want < 1 ? 1 : (want < full ? want : full));
    return launch_pdl(lowlatency_kernel, grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream),
                      a);
}

extern "C" epd_status_t ep_dispatch_lowlatency(const void *x_bf16, const int64_t *topk_idx,
                                               int num_tokens, int num_topk, int hidden,
                                               int num_experts, int num_ranks, int num_rdma_ranks,
                                               int expert_begin, int expert_end,
                                               int64_t rows_per_expert, void *workspace,
                                               void *out_q, float *out_scale,
                                               int32_t *recv_count, int32_t *output_index,
                                               int32_t *src_token, int32_t *status,
                                               epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk, H = hidden, E = num_experts;
    if (!topology_ok(T, k, E, num_ranks, num_rdma_ranks)) return EPD_ERR_INVALID_ARG;
    if (H < 128 || H % 128 != 0) return EPD_ERR_INVALID_ARG;
    if (expert_begin < 0 || expert_end > E || expert_begin >= expert_end) return EPD_ERR_INVALID_ARG;
    const int64_t EV = expert_end - expert_begin;
    if (rows_per_expert < 0 || EV * rows_per_expert > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if (!workspace || !recv_count || !status || !aligned16(workspace) || !aligned4(recv_count) ||
        !aligned4(status))
        return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (!x_bf16 || !topk_idx || !output_index)) return EPD_ERR_INVALID_ARG;
    if (EV * rows_per_expert > 0 && (!out_q || !out_scale)) return EPD_ERR_INVALID_ARG;
    if ((x_bf16 && !aligned16(x_bf16)) || (topk_idx && !aligned8(topk_idx)) ||
        (out_q && !aligned8(out_q)) || !aligned4(out_scale) || !aligned4(output_index) ||
        !aligned4(src_token))
        return EPD_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int grid_cap = 2 * sm_count();
    const int grid = T < 1 ? 1 : (T < grid_cap ? T : grid_cap);
    const int tokens_per_block = T > 0 ? (T + grid - 1) / grid : 0;
    const size_t smem = (size_t)tokens_per_block * ll_row_stride(H);
    const bool small = (int64_t)T * k <= kLLSmallPairs && T <= kLLSmallTokens &&
                       E <= kLLSmallExperts && (int64_t)tokens_per_block * k <= kLLSmallBlockPairs &&
                       smem <= kLLSmallRowBytes;
    if (!small) {
        const epd_status_t st = layout_ranks_only(topk_idx, T, k, E, num_ranks, num_rdma_ranks,
                                                  workspace, status, s);
        if (st != EPD_OK) return st;
        return ep_permute_lowlatency(x_bf16, topk_idx, T, k, H, E, expert_begin, expert_end,
                                     rows_per_expert, workspace, out_q, out_scale, recv_count,
                                     output_index, src_token, status, stream);
    }
    static std::atomic<bool> opted[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return record_cuda_error();
    if (dev < 0 || dev >= 64 || !opted[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(lowlatency_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kLLSmallRowBytes) != cudaSuccess)
            return record_cuda_error();
        if (dev >= 0 && dev < 64) opted[dev].store(true, std::memory_order_release);
    }
    LLSmallArgs a;
    a.x = static_cast<const uint8_t *>(x_bf16);
    a.T = T;
    a.k = k;
    a.H = H;
    a.E = E;
    a.e_begin = expert_begin;
    a.e_end = expert_end;
    a.rows = rows_per_expert;
    a.topk = topk_idx;
    a.out_q = static_cast<uint8_t *>(out_q);
    a.out_scale = out_scale;
    a.recv_count = recv_count;
    a.output_index = output_index;
    a.src_token = src_token;
    a.status = status;
    // blocks per token run: enough to give every warp one unit of the cast, within
    // four blocks per SM in all
    const int upt = (H / 128 + 1) / 2;
    const int units_per_run = tokens_per_block * upt;
    int split = (units_per_run + kWarps - 1) / kWarps;
    const int split_cap = (4 * sm_count()) / grid;
    split = split < 1 ? 1 : (split > split_cap ? (split_cap < 1 ? 1 : split_cap) : split);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, (unsigned)split);
    cfg.blockDim = dim3((unsigned)kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, lowlatency_small_kernel, a);
    return record_cuda_error();
}
