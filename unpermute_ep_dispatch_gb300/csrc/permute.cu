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
#include <atomic>

#include "epd_common.cuh"

namespace epd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnitVecs = 64;  // 16-byte vectors per work unit (1 KiB of a row)

struct PermuteArgs {
    const uint8_t *x;
    int64_t row_bytes;
    const uint32_t *x_scale;  // 32-bit scale words (fp32 scales or packed UE8M0 bytes)
    int scale_cols;
    int scale_col_major;      // 0: out_scale[s * scale_cols + c]; 1: out_scale[c * scale_ld + s]
    int64_t scale_ld;
    int e_begin, e_end;       // experts of the view; rows are relative to start[e_begin]
    const int64_t *topk;
    int T, k, E;
    const int32_t *start;
    const int32_t *pair_rank;
    const int32_t *counts;  // per-expert counts the layout left in the workspace
    const WsHeader *hdr;
    int64_t capacity;
    uint8_t *out;
    uint32_t *out_scale;
    int32_t *m_indices;
    int32_t *output_index;
    int32_t *status;
    // column-major scales: the permute leaves each filled row's source token in
    // m_indices and scale_gather_kernel writes the scales and the final m_indices
    int defer_scales;
    // whole expert range, bulk-copy kernel: blocks [0, pf_stride) (the first resident
    // wave) prefetch the rows of blocks b, b + pf_stride, ... below pf_blocks into L2
    int pf_stride, pf_blocks;
};

// m_indices over the whole buffer from the expert segments: row s belongs to the
// last expert whose region starts at or before s (experts that share a start have
// empty regions), and holds that expert when it is among the region's first
// count rows, else -1 (alignment padding, or rows after the last region). Works
// for plain and aligned offsets alike. `seg_start` / `seg_count` are the view's
// nseg offsets and counts (shared or global memory); g is the row in the
// offsets' coordinates. Returns the expert relative to the view, or -1.
__device__ __forceinline__ int row_expert(const int32_t *seg_start, const int32_t *seg_count,
                                          int nseg, int64_t g) {
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {  // last segment with start <= g
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)seg_start[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    const int64_t st = seg_start[lo];
    return (g >= st && g < st + seg_count[lo]) ? lo : -1;
}

__device__ __forceinline__ void fill_m_indices(const PermuteArgs &a, const int32_t *seg_start,
                                               const int32_t *seg_count, int64_t base,
                                               int64_t first, int64_t stride) {
    const int nseg = a.e_end - a.e_begin;
    for (int64_t s = first; s < a.capacity; s += stride)
        a.m_indices[s] = row_expert(seg_start, seg_count, nseg, s + base);
}

// Row of the scale word c of buffer row s.
__device__ __forceinline__ int64_t scale_index(const PermuteArgs &a, int64_t s, int c) {
    return a.scale_col_major ? (int64_t)c * a.scale_ld + s : s * a.scale_cols + c;
}

__global__ void __launch_bounds__(kThreads) permute_kernel(PermuteArgs a) {
    __shared__ int s_slot[kWarps][EPD_MAX_TOPK];
    __shared__ int s_ok;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();  // offsets and pair ranks come from the previous kernels
    if (threadIdx.x == 0) {
        const bool ok = a.hdr->num_tokens == a.T && a.hdr->num_topk == a.k;
        s_ok = ok;
        if (!ok && blockIdx.x == 0) report(a.status, EPD_ERR_INVALID_ARG);
    }
    __syncthreads();
    if (!s_ok) return;
    const int64_t base = a.start[a.e_begin];  // first row of the view in offset coordinates

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
                if (e >= a.e_begin && e < a.e_end) {
                    const int64_t sl = (int64_t)a.start[e] - base + a.pair_rank[idx];
                    if (sl >= 0 && sl < a.capacity) s = (int)sl;
                    else if (ch == 0) report(a.status, EPD_ERR_CAPACITY);
                }
                if (ch == 0) {
                    a.output_index[idx] = s;
                    if (s >= 0 && a.defer_scales) a.m_indices[s] = t;
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
        if (ch == 0 && !a.defer_scales) {  // fp8 scale row travels with chunk 0
            for (int c = lane; c < a.scale_cols; c += 32) {
                const uint32_t sv = a.x_scale[(int64_t)t * a.scale_cols + c];
                for (int j = 0; j < a.k; ++j) {
                    const int s = s_slot[warp][j];
                    if (s >= 0) a.out_scale[scale_index(a, s, c)] = sv;
                }
            }
        }
    }

    // the next kernel may be scheduled now: triggering only after the row copies keeps
    // its blocks from holding SM resources while this kernel streams
    pdl_trigger();
    if (!a.defer_scales)
        fill_m_indices(a, a.start + a.e_begin, a.counts + a.e_begin, base,
                       (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);
}

// ----------------------------------------------------------------------------- bulk-copy variant
// Blocks over contiguous runs of tokens. For a batch of tokens all threads first
// resolve the slots; then warp 0 streams the rows through a ring of shared-memory
// stages -- one bulk load of each row from HBM and, as soon as it lands, k bulk
// stores of it to its slots, issued by k lanes at once -- while the other warps copy
// the small fp8 scale rows. The row copies run on the TMA engine instead of the
// load/store units, whose store queue limits the register variant above.
constexpr int kTmaThreads = 256;
constexpr size_t kTmaStageBudget = 64 * 1024;  // shared memory for row stages (a few blocks per SM)
constexpr int kTmaMaxStages = 16;
constexpr uint32_t kTmaWaitLimit = 1u << 24;    // mbarrier polls before a wait gives up
constexpr int kTmaSegMax = 1024;  // views of at most this many experts keep their offsets in shared memory

__host__ __device__ inline int tma_batch_tokens(int k) {
    const int b = k > 0 ? 4096 / k : 512;
    return b < 1 ? 1 : (b > 512 ? 512 : b);
}

struct TmaSmem {
    int stages;
    size_t row_stride, slots_off, list_off, bars_off, seg_off, total;  // seg_off 0: not staged
};

__host__ __device__ inline TmaSmem tma_smem(int64_t row_bytes, int k, int nseg) {
    TmaSmem m;
    m.row_stride = align_up((size_t)row_bytes, 128);
    const size_t fit = kTmaStageBudget / m.row_stride;
    m.stages = (int)(fit < (size_t)kTmaMaxStages ? fit : (size_t)kTmaMaxStages);
    const int B = tma_batch_tokens(k);
    m.slots_off = (size_t)m.stages * m.row_stride;
    m.list_off = align_up(m.slots_off + (size_t)B * (k > 0 ? k : 1) * 4, 16);
    m.bars_off = align_up(m.list_off + (size_t)B * 4, 16);
    const size_t bars_end = m.bars_off + (size_t)m.stages * 8;
    m.seg_off = nseg <= kTmaSegMax ? align_up(bars_end, 16) : 0;
    m.total = m.seg_off ? m.seg_off + 2 * (size_t)nseg * 4 : bars_end;
    return m;
}

__global__ void __launch_bounds__(kTmaThreads) permute_tma_kernel(PermuteArgs a) {
    extern __shared__ __align__(128) uint8_t tsm[];
    __shared__ int s_ok, s_n, s_failed;
    const int nseg = a.e_end - a.e_begin;
    const TmaSmem L = tma_smem(a.row_bytes, a.k, nseg);
    uint8_t *stage = tsm;
    int *s_slot = reinterpret_cast<int *>(tsm + L.slots_off);  // [batch tokens][k]
    int *s_list = reinterpret_cast<int *>(tsm + L.list_off);   // tokens of the batch with a slot
    uint64_t *bars = reinterpret_cast<uint64_t *>(tsm + L.bars_off);
    int32_t *s_seg = reinterpret_cast<int32_t *>(tsm + L.seg_off);  // [nseg] offsets, [nseg] counts
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = tma_batch_tokens(a.k);
    const int S = L.stages;
    const uint32_t bytes = (uint32_t)a.row_bytes;
    const int t_begin = (int)((int64_t)a.T * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)a.T * (blockIdx.x + 1) / gridDim.x);
    // Over the whole expert range nearly every token is copied, so the block's first
    // rows are loaded before their slots are known (a token without a valid pick is
    // loaded and not stored); a view copies few of the tokens and loads after.
    const bool whole = a.e_begin == 0 && a.e_end == a.E && a.k > 0;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        mbar_init_fence();
    }
    // Before the dependency wait, the first resident wave asks L2 for the rows of the
    // first blocks (up to kPrefetchBytes), marked to stay (evict-last): the layout kernel
    // that usually runs just before is latency-bound and leaves HBM idle, and the
    // prefetched lines outlast the rows this kernel writes meanwhile. A prefetch
    // changes no value a load returns, so it is safe whatever ran before. Every row
    // is then loaded with an evict-first policy, which releases the line.
    if (whole && warp == 0 && (int)blockIdx.x < a.pf_stride) {
        const uint64_t keep = l2_policy_evict_last();
        for (int b = blockIdx.x; b < a.pf_blocks; b += a.pf_stride) {
            const int tb = (int)((int64_t)a.T * b / gridDim.x);
            const int te = (int)((int64_t)a.T * (b + 1) / gridDim.x);
            for (int t = tb + lane; t < te; t += 32)
                bulk_prefetch_l2(a.x + (int64_t)t * a.row_bytes, bytes, keep);
        }
    }
    const uint64_t release = l2_policy_evict_first();
    pdl_wait();  // offsets and pair ranks come from the previous kernels
    // rows of the first batch loaded ahead (by thread 0)
    const int pre = whole ? min(S - 1, min(B, t_end - t_begin)) : 0;
    if (tid == 0) {
        if (whole) {
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(&bars[i], bytes);
                bulk_load_policy(stage + i * L.row_stride,
                                 a.x + (int64_t)(t_begin + i) * a.row_bytes, bytes, &bars[i],
                                 release);
            }
        }
        const bool ok = a.hdr->num_tokens == a.T && a.hdr->num_topk == a.k;
        s_ok = ok;
        s_failed = 0;
        if (!ok && blockIdx.x == 0) report(a.status, EPD_ERR_INVALID_ARG);
    }
    // the view's offsets and counts, read once per block (slots and m_indices use them)
    if (L.seg_off)
        for (int i = tid; i < nseg; i += kTmaThreads) {
            s_seg[i] = a.start[a.e_begin + i];
            s_seg[nseg + i] = a.counts[a.e_begin + i];
        }
    __syncthreads();
    if (!s_ok) {
        if (tid == 0)  // loads issued ahead land before the block's shared memory is released
            for (int i = 0; i < pre; ++i) mbar_wait_bounded(&bars[i], 0u, kTmaWaitLimit);
        return;
    }
    const int32_t *seg_start = L.seg_off ? s_seg : a.start + a.e_begin;
    const int32_t *seg_count = L.seg_off ? s_seg + nseg : a.counts + a.e_begin;
    const int64_t base = seg_start[0];  // first row of the view in offset coordinates

    uint32_t seq = 0;  // rows this block has loaded so far: row r uses stage r % S, phase r / S
    for (int b0 = t_begin; b0 < t_end; b0 += B) {
        const int nb = min(B, t_end - b0);
        if (tid == 0) s_n = 0;  // counted into after the next barrier
        for (int i = tid; i < nb * a.k; i += kTmaThreads) {
            const int tl = i / a.k;
            const int64_t idx = (int64_t)(b0 + tl) * a.k + (i - tl * a.k);
            const int64_t e = a.topk[idx];
            int s = -1;
            if (e >= a.e_begin && e < a.e_end) {
                const int64_t sl = (int64_t)seg_start[e - a.e_begin] - base + a.pair_rank[idx];
                if (sl >= 0 && sl < a.capacity) {
                    s = (int)sl;
                } else {
                    report(a.status, EPD_ERR_CAPACITY);
                }
            }
            a.output_index[idx] = s;
            if (s >= 0 && a.defer_scales) a.m_indices[s] = b0 + tl;
            s_slot[i] = s;
        }
        __syncthreads();
        if (!whole) {
            for (int tl = tid; tl < nb; tl += kTmaThreads) {
                bool any = false;
                for (int j = 0; j < a.k; ++j) any |= s_slot[tl * a.k + j] >= 0;
                if (any) s_list[atomicAdd(&s_n, 1)] = tl;  // copy order does not change the result
            }
            __syncthreads();
        }
        if (warp == 0) {
            // Warp 0 streams the rows: lane 0 issues the loads, every lane waits on the
            // landed stage's barrier, and lanes j < k issue the k stores of the row at
            // once (each lane in its own bulk group).
            const int n = whole ? nb : s_n;
            int issued = b0 == t_begin ? pre : 0, landed = 0;
            auto token = [&](int i) { return whole ? i : s_list[i]; };
            auto load = [&](int i) {
                const uint32_t r = seq + i, st = r % S;
                mbar_expect_tx(&bars[st], bytes);
                bulk_load_policy(stage + st * L.row_stride,
                                 a.x + (int64_t)(b0 + token(i)) * a.row_bytes, bytes, &bars[st],
                                 release);
            };
            const int first = min(n, S - 1);
            if (lane == 0)
                for (int i = issued; i < first; ++i) load(i);
            issued = max(issued, first);
            for (; landed < n; ++landed) {
                const uint32_t r = seq + landed, st = r % S;
                const bool ok = mbar_wait_bounded(&bars[st], (r / S) & 1u, kTmaWaitLimit);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) {
                        report(a.status, EPD_ERR_TIMEOUT);
                        s_failed = 1;
                    }
                    break;
                }
                fence_proxy_async_smem();
                const int *sl = s_slot + token(landed) * a.k;
                for (int j = lane; j < a.k; j += 32)
                    if (sl[j] >= 0)
                        bulk_store(a.out + (int64_t)sl[j] * a.row_bytes, stage + st * L.row_stride,
                                   bytes);
                bulk_commit();
                if (issued < n) {
                    bulk_wait_read<1>();  // this lane's stores of row r - 1 have left its stage
                    __syncwarp();         // and every other lane's: the stage is free again
                    if (lane == 0) load(issued);
                    ++issued;
                }
            }
            if (s_failed && lane == 0) {  // let every load still in flight land before the block exits
                for (int i = landed; i < issued; ++i) {
                    const uint32_t r = seq + i;
                    mbar_wait_bounded(&bars[r % S], (r / S) & 1u, kTmaWaitLimit);
                }
            }
            seq += issued;
            bulk_wait_read<0>();  // stages are reused by the next batch
        } else if (a.scale_cols > 0 && !a.defer_scales) {
            // fp8 scale rows with plain loads and stores, while thread 0 streams rows
            const int nthreads = kTmaThreads - 32;
            const int t2 = tid - 32;
            if (t2 >= 0) {
                for (int i = t2; i < nb * a.scale_cols; i += nthreads) {
                    const int tl = i / a.scale_cols, c = i - tl * a.scale_cols;
                    const uint32_t sv = a.x_scale[(int64_t)(b0 + tl) * a.scale_cols + c];
                    for (int j = 0; j < a.k; ++j) {
                        const int sl = s_slot[tl * a.k + j];
                        if (sl >= 0) a.out_scale[scale_index(a, sl, c)] = sv;
                    }
                }
            }
        }
        __syncthreads();
        if (s_failed) break;
    }

    if (!a.defer_scales)
        fill_m_indices(a, seg_start, seg_count, base, (int64_t)blockIdx.x * kTmaThreads + tid,
                       (int64_t)gridDim.x * kTmaThreads);
    // the stages must stay valid until the last stores have read them; their writes
    // complete on their own (the grid's completion covers them)
    if (warp == 0) bulk_wait_read<0>();
    // the next kernel may be scheduled now: triggering only after the row copies keeps
    // its blocks from holding SM resources while this kernel streams
    pdl_trigger();
}

// ----------------------------------------------------------------------------- column-major scales
// Scales whose buffer is column-major ([scale_cols][ld], the layout a TMA load of
// one expert's scale tile wants) are written after the rows: scattered across
// the permutation, every pick would store scale_cols words ld apart. Here one
// thread owns one buffer row: it reads the row's source token (left in m_indices
// by the permute), gathers that token's scale words (one cached row of x_scale)
// and stores them down its column, so each warp-wide store covers 32 consecutive
// rows of one column. It then writes the row's final m_indices.
__global__ void __launch_bounds__(kThreads) scale_gather_kernel(PermuteArgs a) {
    __shared__ int32_t s_seg[2 * kTmaSegMax];
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    const int nseg = a.e_end - a.e_begin;
    const bool staged = nseg <= kTmaSegMax;
    pdl_wait();  // source tokens come from the permute
    if (tid == 0) s_ok = a.hdr->num_tokens == a.T && a.hdr->num_topk == a.k;
    if (staged)
        for (int i = tid; i < nseg; i += kThreads) {
            s_seg[i] = a.start[a.e_begin + i];
            s_seg[nseg + i] = a.counts[a.e_begin + i];
        }
    __syncthreads();
    pdl_trigger();
    if (!s_ok) return;  // the permute reported the workspace and wrote nothing
    const int32_t *seg_start = staged ? s_seg : a.start + a.e_begin;
    const int32_t *seg_count = staged ? s_seg + nseg : a.counts + a.e_begin;
    const int64_t base = seg_start[0];
    const int C = a.scale_cols;
    for (int64_t s = (int64_t)blockIdx.x * kThreads + tid; s < a.capacity;
         s += (int64_t)gridDim.x * kThreads) {
        const int e = row_expert(seg_start, seg_count, nseg, s + base);
        if (e >= 0) {
            const int t = a.m_indices[s];
            if (t >= 0 && t < a.T) {  // a permute that gave up early leaves rows unset
                const uint32_t *src = a.x_scale + (int64_t)t * C;
                uint32_t *dst = a.out_scale + s;
                int c = 0;
                for (; c + 8 <= C; c += 8) {
                    uint32_t v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = __ldg(src + c + q);
#pragma unroll
                    for (int q = 0; q < 8; ++q) dst[(int64_t)(c + q) * a.scale_ld] = v[q];
                }
                for (; c < C; ++c) dst[(int64_t)c * a.scale_ld] = __ldg(src + c);
            }
        }
        a.m_indices[s] = e;
    }
}

}  // namespace
}  // namespace epd

namespace epd {
namespace {

epd_status_t permute_rows_launch(PermuteArgs &a, int64_t T, int k, cudaStream_t cs);

// Rows the bulk-copy kernel prefetches into L2 before its dependency wait (measured on
// GB300, steps of layout -> permute -> combine: 32 MB gains 3.1 us at dsv3_fp8 and
// 5.2 us at skew_bf16, as much as 48 or 64 MB, and costs least when nothing runs
// before the permute to hide it; without the evict-last mark the prefetched lines
// were gone by the time they were read).
constexpr int64_t kPrefetchBytes = 32ll << 20;

epd_status_t permute_launch(PermuteArgs &a, int64_t T, int k, cudaStream_t cs) {
    // The separate pass pays off when the scattered stores it replaces are many:
    // more than 16 words per row (fp32 per-128 scales of a 4096-wide row and up;
    // packed UE8M0 words of a 7168-wide row are 14) over a view holding at least a
    // quarter of the experts (a narrow view fills few rows but the pass walks all).
    a.defer_scales = a.scale_cols > 16 && a.scale_col_major && a.capacity > 0 &&
                     4 * (int64_t)(a.e_end - a.e_begin) >= a.E;
    const epd_status_t st = permute_rows_launch(a, T, k, cs);
    if (st != EPD_OK || !a.defer_scales) return st;
    const int64_t want = (a.capacity + kThreads - 1) / kThreads;
    const int64_t full = 8 * (int64_t)sm_count();
    const int grid = (int)(want < full ? want : full);
    return launch_pdl(scale_gather_kernel, grid, kThreads, 0, cs, a);
}

epd_status_t permute_rows_launch(PermuteArgs &a, int64_t T, int k, cudaStream_t cs) {
    // bulk-copy kernel when at least two row stages fit in shared memory
    const TmaSmem L = tma_smem(a.row_bytes, k, a.e_end - a.e_begin);
    if (L.stages >= 2) {
        // the kernel's shared-memory limit, raised per device (a function attribute
        // applies to the current device only)
        static std::atomic<size_t> opted_by_dev[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return record_cuda_error();
        std::atomic<size_t> scratch{0};
        std::atomic<size_t> &opted = (dev >= 0 && dev < 64) ? opted_by_dev[dev] : scratch;
        if (L.total > opted.load(std::memory_order_acquire)) {
            int optin = 0;
            if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
                return record_cuda_error();
            if (L.total + 64 <= (size_t)optin) {
                if (cudaFuncSetAttribute(permute_tma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.total) != cudaSuccess)
                    return record_cuda_error();
                opted.store(L.total, std::memory_order_release);
            }
        }
        if (L.total <= opted.load(std::memory_order_acquire)) {
            // Whole waves of short token runs: the grid is a whole number of resident
            // waves (1..8), each block about six tokens; the hardware hands the next run
            // to whichever block slot frees first, and no wave is left part-full at the
            // end. Measured on GB300 (step / permute chained): prefill_bf16 78.8 / 38.6
            // us at 2 waves of ~7 tokens against 81.7 / 41.5 at 3.5 waves of 4; dsv3_fp8
            // flat from 6 to 8 waves; skew_bf16 best at 8 waves. A view of a few experts
            // copies few rows: there the blocks' fixed costs dominate and three blocks per
            // SM stay best.
            const int64_t sms = sm_count();
            // resident blocks per SM at this shared-memory size (the last size asked is
            // kept per device: (bytes << 8 | blocks))
            static std::atomic<unsigned long long> occ_by_dev[64];
            std::atomic<unsigned long long> occ_scratch{0};
            std::atomic<unsigned long long> &occ =
                (dev >= 0 && dev < 64) ? occ_by_dev[dev] : occ_scratch;
            const unsigned long long o = occ.load(std::memory_order_acquire);
            int per_sm = (o >> 8) == L.total ? (int)(o & 0xffu) : 0;
            if (per_sm == 0) {
                per_sm = blocks_per_sm(permute_tma_kernel, kTmaThreads, L.total);
                occ.store((unsigned long long)L.total << 8 | (unsigned)(per_sm & 0xff),
                          std::memory_order_release);
            }
            const int64_t slots = sms * per_sm;
            const bool wide = 4 * (int64_t)(a.e_end - a.e_begin) >= a.E;
            int64_t g;
            if (wide) {
                int64_t waves = (T + 3 * slots) / (6 * slots);  // round(T / (6 slots))
                waves = waves < 1 ? 1 : (waves > 8 ? 8 : waves);
                g = waves * slots;
            } else {
                g = 3 * sms;
            }
            if (g > T) g = T;
            const int grid = (int)(g < 1 ? 1 : g);
            // the L2 prefetch: the first wave's blocks, for up to kPrefetchBytes of rows
            a.pf_stride = (int)slots;
            const int64_t block_bytes = (T + grid - 1) / grid * a.row_bytes;
            const int64_t pf = kPrefetchBytes / (block_bytes > 0 ? block_bytes : 1);
            a.pf_blocks = (int)(pf < grid ? pf : grid);
            return launch_pdl(permute_tma_kernel, grid, kTmaThreads, L.total, cs, a);
        }
    }
    static const int resident = blocks_per_sm(permute_kernel, kThreads, 0);
    const int64_t units = T * ((a.row_bytes / 16 + kUnitVecs - 1) / kUnitVecs);
    const int64_t want = (units + kWarps - 1) / kWarps;
    const int64_t full = (int64_t)sm_count() * resident;
    const int grid = (int)(want < 1 ? 1 : (want < full ? want : full));
    return launch_pdl(permute_kernel, grid, kThreads, 0, cs, a);
}

// Checks shared by both entry points; fills the common fields of `a`.
epd_status_t permute_common(PermuteArgs &a, const void *x, int64_t row_bytes,
                            const int64_t *topk_idx, int T, int k, int E,
                            const int32_t *expert_start_loc, const void *workspace,
                            int64_t capacity_rows, void *out, int32_t *m_indices,
                            int32_t *output_index, int32_t *status) {
    if (T < 0 || k < 0 || k > EPD_MAX_TOPK || E < 1 || E > EPD_MAX_EXPERTS) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if (row_bytes <= 0 || row_bytes % 16 != 0) return EPD_ERR_INVALID_ARG;
    if (capacity_rows < 0 || capacity_rows > INT32_MAX) return EPD_ERR_INVALID_ARG;
    if (!expert_start_loc || !workspace || !status) return EPD_ERR_INVALID_ARG;
    if (capacity_rows > 0 && !m_indices) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (!output_index || !topk_idx || !x || !out)) return EPD_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (out && !aligned16(out)) || (topk_idx && !aligned8(topk_idx)) ||
        !aligned4(expert_start_loc) || !aligned16(workspace) || !aligned4(m_indices) ||
        !aligned4(output_index) || !aligned4(status))
        return EPD_ERR_INVALID_ARG;
    const char *ws = static_cast<const char *>(workspace);
    a.x = static_cast<const uint8_t *>(x);
    a.row_bytes = row_bytes;
    a.topk = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.start = expert_start_loc;
    a.pair_rank = reinterpret_cast<const int32_t *>(ws + ws_pair_rank_off());
    a.counts = reinterpret_cast<const int32_t *>(ws + ws_counts_off(T, k));
    a.hdr = reinterpret_cast<const WsHeader *>(ws);
    a.capacity = capacity_rows;
    a.out = static_cast<uint8_t *>(out);
    a.m_indices = m_indices;
    a.output_index = output_index;
    a.status = status;
    a.pf_stride = 0;  // no prefetch unless the bulk-copy launch sets it
    a.pf_blocks = 0;
    return EPD_OK;
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
    const int T = num_tokens, k = num_topk, H = hidden;
    if (T < 0 || k < 0 || H <= 0) return EPD_ERR_INVALID_ARG;
    if (capacity_rows < (int64_t)T * k) return EPD_ERR_INVALID_ARG;
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
    PermuteArgs a;
    const epd_status_t st = permute_common(a, x, row_bytes, topk_idx, T, k, num_experts,
                                           expert_start_loc, workspace, capacity_rows, out,
                                           m_indices, output_index, status);
    if (st != EPD_OK) return st;
    a.x_scale = reinterpret_cast<const uint32_t *>(x_scale);
    a.scale_cols = scale_cols;
    a.scale_col_major = 0;
    a.scale_ld = 0;
    a.out_scale = reinterpret_cast<uint32_t *>(out_scale);
    a.e_begin = 0;
    a.e_end = num_experts;
    return permute_launch(a, T, k, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" epd_status_t ep_permute_ex(const void *x, int64_t row_bytes, const void *x_scale,
                                      const int64_t *topk_idx, int num_tokens, int num_topk,
                                      int num_experts, const int32_t *expert_start_loc,
                                      const void *workspace, int64_t capacity_rows,
                                      const epd_permute_view_t *view, void *out, void *out_scale,
                                      int32_t *m_indices, int32_t *output_index, int32_t *status,
                                      epd_stream_t stream) {
    using namespace epd;
    if (view == nullptr) return EPD_ERR_INVALID_ARG;
    const epd_permute_view_t v = *view;
    if (v.expert_begin < 0 || v.expert_end > num_experts || v.expert_begin >= v.expert_end)
        return EPD_ERR_INVALID_ARG;
    if (v.scale_cols < 0 || (v.scale_col_major != 0 && v.scale_col_major != 1))
        return EPD_ERR_INVALID_ARG;
    if (v.scale_cols > 0) {
        if ((num_tokens > 0 && num_topk > 0 && x_scale == nullptr) ||
            (capacity_rows > 0 && out_scale == nullptr) || !aligned4(x_scale) || !aligned4(out_scale))
            return EPD_ERR_INVALID_ARG;
        if (v.scale_col_major && v.scale_ld < capacity_rows) return EPD_ERR_INVALID_ARG;
    }
    PermuteArgs a;
    const epd_status_t st = permute_common(a, x, row_bytes, topk_idx, num_tokens, num_topk,
                                           num_experts, expert_start_loc, workspace,
                                           capacity_rows, out, m_indices, output_index, status);
    if (st != EPD_OK) return st;
    a.x_scale = static_cast<const uint32_t *>(x_scale);
    a.scale_cols = v.scale_cols;
    a.scale_col_major = v.scale_col_major;
    a.scale_ld = v.scale_ld;
    a.out_scale = static_cast<uint32_t *>(out_scale);
    a.e_begin = v.expert_begin;
    a.e_end = v.expert_end;
    return permute_launch(a, num_tokens, num_topk, reinterpret_cast<cudaStream_t>(stream));
}
