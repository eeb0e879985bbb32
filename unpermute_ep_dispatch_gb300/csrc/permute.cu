// permute.cu -- step 3 of the path: permute (ep_scatter).
//
// "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题", sections 2.2 and
// 3.3: every token row (with its fp8 scale row) is copied into the
// expert-contiguous buffer once per selected expert; m_indices names the expert
// of each buffer row, output_index the row each (token, pick) pair went to,
// and rows no pair fills carry m_indices = -1.
//
// The slot of pair (t, j) with expert e is expert_start_loc[e] plus the pair's
// rank inside e, which the layout kernel left in the workspace, so every token
// is independent and the cost per token does not depend on the routing skew.
// The work is cut into units of (token, 1 KiB of its row) and a persistent grid
// (resident blocks x SMs) gives every warp an equal contiguous run of units, so
// no SM idles in a tail wave. Each unit is read once (16-byte streaming loads
// that bypass L1) and written k times with 16-byte coalesced stores: every
// warp-wide store covers 512 contiguous bytes of a destination row.
#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnitVecs = 64;  // 16-byte vectors per work unit (1 KiB of a row)

struct PermuteArgs {
    const uint8_t *x;
    int64_t row_bytes;
    const float *x_scale;
    int scale_cols;
    const int64_t *topk;
    int T, k, E;
    const int32_t *start;
    const int32_t *pair_rank;
    const WsHeader *hdr;
    int64_t capacity;
    uint8_t *out;
    float *out_scale;
    int32_t *m_indices;
    int32_t *output_index;
    int32_t *status;
};

__global__ void __launch_bounds__(kThreads) permute_kernel(PermuteArgs a) {
    __shared__ int s_slot[kWarps][EPD_MAX_TOPK];
    __shared__ int s_ok, s_P;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();  // offsets and pair ranks come from the previous kernels
    pdl_trigger();
    if (threadIdx.x == 0) {
        const bool ok = a.hdr->num_tokens == a.T && a.hdr->num_topk == a.k;
        s_ok = ok;
        s_P = ok ? max(0, a.hdr->total_pairs) : 0;
        if (!ok && blockIdx.x == 0) report(a.status, EPD_ERR_INVALID_ARG);
    }
    __syncthreads();
    if (!s_ok) return;

    const int64_t row_vecs = a.row_bytes >> 4;
    const int upt = (int)((row_vecs + kUnitVecs - 1) / kUnitVecs);  // units per token
    const int64_t units = (int64_t)a.T * upt;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u_end = units * (gw + 1) / nw;
    int cur_t = -1;
    bool any = false;
    for (int64_t u = units * gw / nw; u < u_end; ++u) {
        const int t = (int)(u / upt);
        const int ch = (int)(u - (int64_t)t * upt);
        if (t != cur_t) {
            // slots of this token's picks; the unit holding chunk 0 records them
            cur_t = t;
            int has = 0;
            __syncwarp();
            for (int j = lane; j < a.k; j += 32) {
                const int64_t idx = (int64_t)t * a.k + j;
                const int64_t e = a.topk[idx];
                int s = -1;
                if (e >= 0 && e < a.E) {
                    const int64_t sl = (int64_t)a.start[e] + a.pair_rank[idx];
                    if (sl >= 0 && sl < a.capacity) s = (int)sl;
                    else if (ch == 0) report(a.status, EPD_ERR_CAPACITY);
                }
                if (ch == 0) {
                    a.output_index[idx] = s;
                    if (s >= 0) a.m_indices[s] = (int)e;
                }
                s_slot[warp][j] = s;
                has |= (s >= 0);
            }
            any = __any_sync(0xffffffffu, has);
            __syncwarp();
        }
        if (!any) continue;  // no valid pick: nothing to copy

        const uint8_t *src = a.x + (int64_t)t * a.row_bytes;
        const int64_t c0 = (int64_t)ch * kUnitVecs + lane, c1 = c0 + 32;
        const uint4 v0 = c0 < row_vecs ? ld_stream16(src + (c0 << 4)) : make_uint4(0, 0, 0, 0);
        const uint4 v1 = c1 < row_vecs ? ld_stream16(src + (c1 << 4)) : make_uint4(0, 0, 0, 0);
        for (int j = 0; j < a.k; ++j) {
            const int s = s_slot[warp][j];
            if (s < 0) continue;
            uint8_t *dst = a.out + (int64_t)s * a.row_bytes;
            if (c0 < row_vecs) st16(dst + (c0 << 4), v0);
            if (c1 < row_vecs) st16(dst + (c1 << 4), v1);
        }
        if (ch == 0) {  // fp8 scale row travels with chunk 0
            for (int c = lane; c < a.scale_cols; c += 32) {
                const float sv = a.x_scale[(int64_t)t * a.scale_cols + c];
                for (int j = 0; j < a.k; ++j) {
                    const int s = s_slot[warp][j];
                    if (s >= 0) a.out_scale[(int64_t)s * a.scale_cols + c] = sv;
                }
            }
        }
    }

    // rows [P, capacity) hold no pair
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t s = s_P + (int64_t)blockIdx.x * kThreads + threadIdx.x; s < a.capacity; s += stride)
        a.m_indices[s] = -1;
}

}  // namespace
}  // namespace epd

extern "C" epd_status_t ep_permute(const void *x, epd_dtype_t dtype, const float *x_scale,
                                   const int64_t *topk_idx, int num_tokens, int num_topk,
                                   int hidden, int num_experts, const int32_t *expert_start_loc,
                                   const void *workspace, int64_t capacity_rows, void *out,
                                   float *out_scale, int32_t *m_indices, int32_t *output_index,
                                   int32_t *status, epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk, H = hidden, E = num_experts;
    if (T < 0 || k < 0 || k > EPD_MAX_TOPK || E < 1 || E > EPD_MAX_EXPERTS || H <= 0)
        return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > INT32_MAX) return EPD_ERR_INVALID_ARG;
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
    if (!expert_start_loc || !workspace || !status) return EPD_ERR_INVALID_ARG;
    if (capacity_rows > 0 && !m_indices) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (!output_index || !topk_idx || !x || !out)) return EPD_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (out && !aligned16(out)) || (topk_idx && !aligned8(topk_idx)) ||
        !aligned4(expert_start_loc) || !aligned16(workspace) || !aligned4(m_indices) ||
        !aligned4(output_index) || !aligned4(status))
        return EPD_ERR_INVALID_ARG;

    const char *ws = static_cast<const char *>(workspace);
    PermuteArgs a;
    a.x = static_cast<const uint8_t *>(x);
    a.row_bytes = row_bytes;
    a.x_scale = x_scale;
    a.scale_cols = scale_cols;
    a.topk = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.start = expert_start_loc;
    a.pair_rank = reinterpret_cast<const int32_t *>(ws + ws_pair_rank_off());
    a.hdr = reinterpret_cast<const WsHeader *>(ws);
    a.capacity = capacity_rows;
    a.out = static_cast<uint8_t *>(out);
    a.out_scale = out_scale;
    a.m_indices = m_indices;
    a.output_index = output_index;
    a.status = status;

    static int resident = 0;
    if (resident == 0) resident = blocks_per_sm(permute_kernel, kThreads, 0);
    const int64_t units = (int64_t)T * ((row_bytes / 16 + kUnitVecs - 1) / kUnitVecs);
    const int64_t want = (units + kWarps - 1) / kWarps;
    const int64_t full = (int64_t)sm_count() * resident;
    const int grid = (int)(want < 1 ? 1 : (want < full ? want : full));
    return launch_pdl(permute_kernel, grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream), a);
}
