// unpermute.cu -- step 4 of the path: unpermute (combine).
//
// "[MoE] Deepseek的All-to-all通信: DeepEP代码解读", section "Dispatch": the
// weights travel with the tokens as fp32 topk_weights [T, k] and combine is the
// reverse of dispatch. For every token t and column h
//     y[t, h] = bf16( sum over valid j, in j order, of w[t, j] * eo[slot(t, j), h] )
// with each product and each sum rounded to fp32 (no fused multiply-add) and
// one round-to-nearest-even at the end.
//
// The work is cut into units of (token, 32*U 16-byte column chunks) and a
// persistent grid (resident blocks x SMs) gives every warp an equal contiguous
// run of units. For a group of KT picks a lane issues all KT x U row loads
// before any arithmetic, so each warp keeps KT * U * 512 bytes of gathers in
// flight. Loads bypass L1 (each expert-output row is read exactly once); y is
// written with 16-byte coalesced stores.
#include <cuda_bf16.h>

#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct UnpermuteArgs {
    const uint8_t *eo;  // [capacity, H] bf16
    int64_t capacity;
    const int32_t *output_index;
    const float *w;
    int T, k;
    int64_t row_vecs;  // H / 8
    uint8_t *y;        // [T, H] bf16
    int32_t *status;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

__device__ __forceinline__ void accum8(float (&acc)[8], float w, const uint4 &v) {
    acc[0] = __fadd_rn(acc[0], __fmul_rn(w, bf16_lo(v.x)));
    acc[1] = __fadd_rn(acc[1], __fmul_rn(w, bf16_hi(v.x)));
    acc[2] = __fadd_rn(acc[2], __fmul_rn(w, bf16_lo(v.y)));
    acc[3] = __fadd_rn(acc[3], __fmul_rn(w, bf16_hi(v.y)));
    acc[4] = __fadd_rn(acc[4], __fmul_rn(w, bf16_lo(v.z)));
    acc[5] = __fadd_rn(acc[5], __fmul_rn(w, bf16_hi(v.z)));
    acc[6] = __fadd_rn(acc[6], __fmul_rn(w, bf16_lo(v.w)));
    acc[7] = __fadd_rn(acc[7], __fmul_rn(w, bf16_hi(v.w)));
}

template <int KT, int U>
__global__ void __launch_bounds__(kThreads) unpermute_kernel(UnpermuteArgs a) {
    __shared__ int s_slot[kWarps][EPD_MAX_TOPK];
    __shared__ float s_w[kWarps][EPD_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();  // output_index (and the expert outputs) come from earlier kernels
    pdl_trigger();
    const int64_t row_bytes = a.row_vecs << 4;
    constexpr int kUnitVecs = 32 * U;
    const int upt = (int)((a.row_vecs + kUnitVecs - 1) / kUnitVecs);  // units per token
    const int64_t units = (int64_t)a.T * upt;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t u_end = units * (gw + 1) / nw;
    int cur_t = -1;
    for (int64_t u = units * gw / nw; u < u_end; ++u) {
        const int t = (int)(u / upt);
        const int ch = (int)(u - (int64_t)t * upt);
        if (t != cur_t) {
            cur_t = t;
            __syncwarp();
            for (int j = lane; j < a.k; j += 32) {
                const int64_t idx = (int64_t)t * a.k + j;
                int s = a.output_index[idx];
                if (s < -1 || (int64_t)s >= a.capacity) {
                    if (ch == 0) report(a.status, EPD_ERR_CAPACITY);
                    s = -1;
                }
                s_slot[warp][j] = s;
                s_w[warp][j] = a.w[idx];
            }
            __syncwarp();
        }
        const int64_t c0 = (int64_t)ch * kUnitVecs + lane;
        float acc[U][8];
#pragma unroll
        for (int uu = 0; uu < U; ++uu)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[uu][i] = 0.0f;
        for (int jg = 0; jg < a.k; jg += KT) {
            uint4 v[KT][U];
#pragma unroll
            for (int jj = 0; jj < KT; ++jj) {
                const int j = jg + jj;
                const int s = j < a.k ? s_slot[warp][j] : -1;
                const uint8_t *src = a.eo + (int64_t)(s < 0 ? 0 : s) * row_bytes;
#pragma unroll
                for (int uu = 0; uu < U; ++uu) {
                    const int64_t c = c0 + uu * 32;
                    v[jj][uu] = (s >= 0 && c < a.row_vecs) ? ld_stream16(src + (c << 4))
                                                           : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int jj = 0; jj < KT; ++jj) {
                const int j = jg + jj;
                if (j >= a.k || s_slot[warp][j] < 0) continue;
                const float wj = s_w[warp][j];
#pragma unroll
                for (int uu = 0; uu < U; ++uu) accum8(acc[uu], wj, v[jj][uu]);
            }
        }
        uint8_t *dst = a.y + (int64_t)t * row_bytes;
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            const int64_t c = c0 + uu * 32;
            if (c < a.row_vecs) {
                uint4 o;
                o.x = pack_bf16(acc[uu][0], acc[uu][1]);
                o.y = pack_bf16(acc[uu][2], acc[uu][3]);
                o.z = pack_bf16(acc[uu][4], acc[uu][5]);
                o.w = pack_bf16(acc[uu][6], acc[uu][7]);
                st16(dst + (c << 4), o);
            }
        }
    }
}

template <int KT, int U>
epd_status_t launch(const UnpermuteArgs &a, cudaStream_t stream) {
    static const int resident = blocks_per_sm(unpermute_kernel<KT, U>, kThreads, 0);
    const int64_t units = (int64_t)a.T * ((a.row_vecs + 32 * U - 1) / (32 * U));
    const int64_t want = (units + kWarps - 1) / kWarps;
    const int64_t full = (int64_t)sm_count() * resident;
    const int grid = (int)(want < 1 ? 1 : (want < full ? want : full));
    return launch_pdl(unpermute_kernel<KT, U>, grid, kThreads, 0, stream, a);
}

}  // namespace
}  // namespace epd

extern "C" epd_status_t ep_unpermute(const void *expert_out, int64_t capacity_rows,
                                     const int32_t *output_index, const float *topk_weights,
                                     int num_tokens, int num_topk, int hidden, void *y,
                                     int32_t *status, epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk, H = hidden;
    if (T < 0 || k < 0 || k > EPD_MAX_TOPK || H <= 0 || H % 8 != 0) return EPD_ERR_INVALID_ARG;
    if (capacity_rows < 0 || capacity_rows > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if (!status || !aligned4(status)) return EPD_ERR_INVALID_ARG;
    if (T == 0) return EPD_OK;
    if (!y || !aligned16(y)) return EPD_ERR_INVALID_ARG;
    if (k > 0) {
        if (!output_index || !topk_weights || !aligned4(output_index) || !aligned4(topk_weights))
            return EPD_ERR_INVALID_ARG;
        if (capacity_rows > 0 && (!expert_out || !aligned16(expert_out))) return EPD_ERR_INVALID_ARG;
    }
    UnpermuteArgs a;
    a.eo = static_cast<const uint8_t *>(expert_out);
    a.capacity = capacity_rows;
    a.output_index = output_index;
    a.w = topk_weights;
    a.T = T;
    a.k = k;
    a.row_vecs = H / 8;
    a.y = static_cast<uint8_t *>(y);
    a.status = status;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (k <= 1) return launch<1, 4>(a, s);
    if (k <= 2) return launch<2, 4>(a, s);
    if (k <= 4) return launch<4, 2>(a, s);
    return launch<8, 2>(a, s);
}
