// epd_common.cuh -- helpers shared by libepd's CUDA translation units:
// workspace layout, argument checks, PTX wrappers for the memory-model
// operations the look-back needs, and 16-byte streaming loads / stores.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "epd.h"

namespace epd {

// ---------------------------------------------------------------------------- workspace
// Byte layout of the caller's workspace. The header and the per-pair ranks sit
// at fixed offsets that depend on T*k only, so ep_permute (which is not given
// R and N) finds them; the look-back state follows.
struct WsHeader {
    uint32_t ticket;       // next token tile to hand out (dynamic tile order); wraps to 0
                           // by itself once a call has handed out all its tiles
    uint32_t done;         // layout blocks of the running call that finished; wraps to 0
    uint64_t epoch;        // call counter; look-back states carry it
    int32_t total_pairs;   // P of the last layout call
    int32_t num_tokens;    // T of the last layout call
    int32_t num_topk;      // k of the last layout call
    uint32_t pad[9];
};
static_assert(sizeof(WsHeader) == 64, "header is one 64-byte block");

constexpr size_t kAlign = 256;
constexpr int kLayoutTilePairs = 1024;    // (token, pick) pairs per tile of 4- and 8-warp blocks
constexpr int kLayoutWideChunks = 4;      // 32-pair chunks per warp of 16- and 32-warp blocks
constexpr int kLayoutMaxTileTokens = 2048;

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Warps per layout block: each warp keeps a private E-wide histogram in shared
// memory (at most 64 KiB of histograms), so fewer warps for larger E.
__host__ __device__ inline int layout_warps(int E) {
    return E <= 512 ? 32 : E <= 1024 ? 16 : E <= 2048 ? 8 : 4;
}

// (token, pick) pairs per tile of the layout's tile form: four 32-pair chunks per warp of
// a 16- or 32-warp block (E <= 1024: fewer tiles, a shorter look-back), 1024 pairs for
// the narrow blocks of E > 1024.
__host__ __device__ inline int layout_tile_pairs(int E) {
    const int W = layout_warps(E);
    return W >= 16 ? W * 32 * kLayoutWideChunks : kLayoutTilePairs;
}

// Tokens per layout tile: at most layout_tile_pairs(E) pairs and at most 2048 tokens (one
// 64-bit rank mask and one node mask per token stay in shared memory).
__host__ __device__ inline int layout_tile_tokens(int k, int E) {
    const int t = k > 0 ? layout_tile_pairs(E) / k : kLayoutMaxTileTokens;
    return t < 1 ? 1 : (t < kLayoutMaxTileTokens ? t : kLayoutMaxTileTokens);
}

struct WsLayout {
    size_t header_off, pair_rank_off, counts_off, state_off, agg_off, incl_off, total;
    int tiles, cols, cols_pad;
};

__host__ __device__ inline size_t ws_pair_rank_off() { return kAlign; }

// The layout's per-expert counts, kept for ep_permute (which needs T, k and E only).
__host__ __device__ inline size_t ws_counts_off(int T, int k) {
    return align_up(kAlign + (size_t)T * (size_t)k * 4, kAlign);
}

__host__ __device__ inline WsLayout ws_layout(int T, int k, int E, int R, int N) {
    WsLayout w;
    int tile = layout_tile_tokens(k, E);
    w.tiles = T > 0 ? (T + tile - 1) / tile : 1;
    w.cols = E + R + N;
    w.cols_pad = (int)align_up((size_t)w.cols, 32);
    w.header_off = 0;
    w.pair_rank_off = ws_pair_rank_off();
    w.counts_off = ws_counts_off(T, k);
    w.state_off = align_up(w.counts_off + (size_t)E * 4, kAlign);
    w.agg_off = align_up(w.state_off + (size_t)w.tiles * 8, kAlign);  // 64-bit state words
    w.incl_off = align_up(w.agg_off + (size_t)w.tiles * w.cols_pad * 4, kAlign);
    w.total = align_up(w.incl_off + (size_t)w.tiles * w.cols_pad * 4, kAlign);
    return w;
}

// ---------------------------------------------------------------------------- host checks
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

inline bool topology_ok(int T, int k, int E, int R, int N) {
    if (T < 0 || k < 0 || k > EPD_MAX_TOPK) return false;
    if (E < 1 || E > EPD_MAX_EXPERTS) return false;
    if (R < 1 || R > E || E % R != 0) return false;
    if (N < 1 || N > R || R % N != 0) return false;
    if ((int64_t)T * (int64_t)k > INT32_MAX) return false;
    return true;
}

int sm_count();  // multiprocessors of the current device (cached per device)

// The layout kernel for its workspace only (no count outputs); layout.cu.
epd_status_t layout_ranks_only(const int64_t *topk_idx, int T, int k, int E, int R, int N,
                               void *workspace, int32_t *status, cudaStream_t stream);

// Reads and clears the CUDA runtime's last error, keeps its code for
// epd_last_cuda_error() and maps it to EPD_OK / EPD_ERR_CUDA.
epd_status_t record_cuda_error();
int last_cuda_error();

inline epd_status_t launch_status() { return record_cuda_error(); }

// Launch with programmatic dependent launch: the kernel may be scheduled while
// the previous kernel on the stream drains, and waits (griddepcontrol.wait)
// before it touches memory that kernel wrote. Hides the launch gap between the
// four steps of the path.
template <typename... KArgs, typename... Args>
inline epd_status_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                               cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return record_cuda_error();
}

// The same with the grid cut into thread-block clusters of `cluster` blocks.
template <typename... KArgs, typename... Args>
inline epd_status_t launch_pdl_cluster(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                                       int cluster, cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return record_cuda_error();
}

// Resident blocks of `kernel` per SM at `block` threads and `smem` dynamic bytes.
template <typename K>
inline int blocks_per_sm(K kernel, int block, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = 1;
    }
    return n;
}

// ---------------------------------------------------------------------------- device helpers
__device__ __forceinline__ void report(int32_t *status, int code) {
    atomicCAS(status, 0, code);
}

// Wait until the previous kernel on the stream has completed and its writes
// are visible (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel on the stream to be scheduled (it still waits for this
// one to complete before reading what this one writes).
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_acquire_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Streaming 16-byte load that does not allocate in L1 (each row is read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st16(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Lane b gets the number of lanes of the warp whose word x has bit b set: the warp's
// 32 x 32 bit matrix is transposed by five butterfly exchanges of half-blocks, and
// each lane then counts the bits of its row.
__device__ __forceinline__ int bit_column_count(uint32_t x, int lane) {
#pragma unroll
    for (int j = 16; j >= 1; j >>= 1) {
        const uint32_t m = j == 16 ? 0x0000ffffu
                         : j == 8  ? 0x00ff00ffu
                         : j == 4  ? 0x0f0f0f0fu
                         : j == 2  ? 0x33333333u
                                   : 0x55555555u;
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
        x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y & m) << j));
    }
    return __popc(x);
}

// The low four bits of b spread to the four bytes of a word (byte i = bit i).
__device__ __forceinline__ int spread4(uint32_t b) { return (int)(((b & 0xFu) * 0x00204081u) & 0x01010101u); }

// ---------------------------------------------------------------------------- thread-block clusters
// Index of this block's cluster in the grid (x).
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Rank of this block inside its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Split cluster barrier: every thread of every block of the cluster arrives (its
// earlier writes, shared memory of other blocks included, are released) and later
// waits (acquiring what the others released). Called by all threads, uniformly.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Barrier `id` (1..15; 0 is __syncthreads) over the first `threads` threads of the
// block (a multiple of 32, whole warps, each of them calling it).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Arrival that publishes nothing: only "this block is running" (no ordering of the
// block's earlier writes).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return r;
}

// 16-byte store to another block's shared memory (an address from cluster_map).
__device__ __forceinline__ void cluster_st_v4(uint32_t addr, const int4 &v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------- bulk copies
// Shared-memory address of a generic pointer to this block's shared memory.
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes initialised mbarriers visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after `limit` polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Global -> shared bulk copy (bytes % 16 == 0, both addresses 16-byte aligned),
// completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// L2 eviction-priority policies for the cache hints below (fraction 1: every access
// made with the policy).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Asks L2 to fetch `bytes` at `src` (16-byte aligned, a multiple of 16 bytes) with
// the given eviction policy. A hint only: it changes no value any load returns (L2
// is where every write lands), so it may be issued before the dependency wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
                 "r"(bytes), "l"(policy)
                 : "memory");
}

// bulk_load with an L2 eviction policy for the lines it reads.
__device__ __forceinline__ void bulk_load_policy(void *dst_smem, const void *src, uint32_t bytes,
                                                 uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Shared -> global bulk copy in the current bulk group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace epd
