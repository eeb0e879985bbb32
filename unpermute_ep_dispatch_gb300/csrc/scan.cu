// scan.cu -- step 2 of the path: expert offsets.
//
// "高性能专家并行（EP）内核解剖学解读", section "5. 缓冲区布局与发送": once the
// counts are known the buffer layout follows from a prefix sum -- the first
// source starts at 0, each next one where the previous ended.
// "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题", 2.2.4: ep_scatter
// first scans the counts into expert_start_loc, then scatters.
//
// With an alignment A > 1 every count is first rounded up to a multiple of A
// (the padded regions of a grouped-GEMM contiguous layout).
// E <= 4096 values fit one block: 1024 threads each own 4 consecutive counts,
// a warp-shuffle scan and a scan of the 32 warp totals give every thread its
// exclusive base. The cross-block part of the path's prefix work (counts
// accumulated over token tiles) is the layout kernel's decoupled look-back.
#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
static_assert(kScanThreads * kScanItems >= EPD_MAX_EXPERTS, "one block covers every expert");

__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int32_t *__restrict__ counts, int E, int alignment,
                int32_t *__restrict__ start, int32_t *__restrict__ total, int32_t *status) {
    __shared__ int s_warp[kScanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();  // the counts come from the layout kernel
    pdl_trigger();
    int v[kScanItems];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        const int idx = tid * kScanItems + i;
        v[i] = idx < E ? counts[idx] : 0;
        if (v[i] < 0) {
            report(status, EPD_ERR_INVALID_ARG);
            v[i] = 0;
        }
        v[i] = (v[i] + alignment - 1) / alignment * alignment;  // the expert's padded rows
        sum += v[i];
    }
    // inclusive scan of the thread sums inside the warp
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = s_warp[lane];
        int wincl = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wincl, o);
            if (lane >= o) wincl += n;
        }
        s_warp[lane] = wincl - wv;  // exclusive base of each warp
        if (lane == 31) *total = wincl;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - sum;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        const int idx = tid * kScanItems + i;
        if (idx < E) start[idx] = run;
        run += v[i];
    }
}

}  // namespace
}  // namespace epd

extern "C" epd_status_t ep_scan_offsets_aligned(const int32_t *tokens_per_expert,
                                                int num_experts, int alignment,
                                                int32_t *expert_start_loc, int32_t *total_rows,
                                                int32_t *status, epd_stream_t stream) {
    using namespace epd;
    if (num_experts < 1 || num_experts > EPD_MAX_EXPERTS) return EPD_ERR_INVALID_ARG;
    if (alignment < 1 || alignment > EPD_MAX_ALIGNMENT) return EPD_ERR_INVALID_ARG;
    if (!tokens_per_expert || !expert_start_loc || !total_rows || !status) return EPD_ERR_INVALID_ARG;
    if (!aligned4(tokens_per_expert) || !aligned4(expert_start_loc) || !aligned4(total_rows) ||
        !aligned4(status))
        return EPD_ERR_INVALID_ARG;
    return launch_pdl(scan_kernel, 1, kScanThreads, 0, reinterpret_cast<cudaStream_t>(stream),
                      tokens_per_expert, num_experts, alignment, expert_start_loc, total_rows,
                      status);
}

extern "C" epd_status_t ep_scan_offsets(const int32_t *tokens_per_expert, int num_experts,
                                        int32_t *expert_start_loc, int32_t *total_rows,
                                        int32_t *status, epd_stream_t stream) {
    return ep_scan_offsets_aligned(tokens_per_expert, num_experts, 1, expert_start_loc,
                                   total_rows, status, stream);
}
