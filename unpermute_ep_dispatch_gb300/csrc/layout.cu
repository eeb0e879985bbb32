// layout.cu -- step 1 of the path: the dispatch layout.
//
// "[MoE] Deepseek的All-to-all通信: DeepEP代码解读", section "Dispatch"
// (get_dispatch_layout docstring): from topk_idx [T, k] (-1 = no selection)
// count the tokens sent to each expert, each rank and each RDMA node, and mark
// is_token_in_rank. The pages skip the kernel body; this one is designed for
// sm_103a from the definition.
//
// The batch is cut into token tiles, one per block: the blocks of one
// thread-block cluster for batches up to 16 x 8192 pairs (they exchange their
// counts through distributed shared memory) -- or of several clusters, where one
// cluster of 16 would need eight 32-pair chunks per warp (each cluster's last block
// publishes the cluster's counts in global memory for the later clusters) -- else
// one block per tile of layout_tile_pairs(E) pairs in ticket order (a block only
// ever waits on blocks already running). Inside a tile:
//   * each warp zeroes its private histogram row while its picks are in flight,
//     then walks a contiguous run of the tile's (token, pick) pairs in row-major
//     order, 32 at a time; lanes holding the same expert find each other through a
//     per-warp shared-memory word per expert (each clears it, sets its lane bit,
//     then reads the word), and the lowest of them adds the group's size to the
//     warp's private histogram; the picks are parked in shared memory for the
//     token masks;
//   * an exclusive scan across the warps' histograms (one thread per expert)
//     gives each pair its rank among the tile's pairs of the same expert, in
//     (t, j) order; beside it, other warps build each token's rank and node bit
//     masks and count the tile's tokens per rank and per node;
//   * the tile's counts (experts, ranks, nodes) reach the later tiles: in a
//     cluster, by stores into their shared memory and one cluster barrier (then,
//     with several clusters, through the published cluster counts); else they are
//     published and read with a single-pass decoupled look-back (a warp polls the
//     states of up to 32 earlier tiles at once and stops at the nearest one that
//     has published its inclusive prefix);
//   * prefix + warp base + rank inside the warp = the pair's rank inside its
//     expert over the whole batch, stored in the workspace for ep_permute;
//   * the last tile (the last ticket, or the grid's last block) writes the totals
//     (and, for ep_dispatch_layout_offsets, the expert offsets) from eight warps
//     while the others store the pair ranks.
// A tile-form call with a single tile takes no ticket and publishes nothing.
// Every value is an integer sum, so the outputs are the same whichever order the
// blocks run in. Waits are bounded: a wait that runs out sets EPD_ERR_TIMEOUT and
// the block carries on.
#include <atomic>
#include <cstddef>

#include "epd_common.cuh"

namespace epd {
namespace {

// A tile's 64-bit state word is kStateMark | call counter << 2 | flag. Nothing else
// the library writes into a workspace has the top bit of a 64-bit word set (every
// other int32 there is >= -1, and two -1 words would need a call counter of 2^61),
// so leftovers of a call of another shape -- pair ranks, counts -- or of an
// earlier call never read as a published state.
constexpr uint64_t kStateMark = 1ull << 63;
constexpr uint32_t kStateAgg = 1;   // tile published its own counts
constexpr uint32_t kStateIncl = 2;  // tile published counts of itself and all earlier tiles
constexpr uint32_t kDefaultSpinLimit = 1u << 19;  // polls with back-off: about a second
// A cluster's published count (several clusters): kStateMark | call counter << 21 |
// count. Counts stay below 2^21 (the form is used for at most 2^20 pairs) and the
// call counter keeps 42 bits. Leftovers never read as current: an int32 pair whose
// upper word is >= 0 lacks the mark, one whose upper word is -1 would need a counter
// with its 31 top bits set, and an earlier call's word carries another counter
// unless 2^42 calls lie between them.
constexpr int kAggValueBits = 21;
constexpr uint64_t kAggValueMask = (1ull << kAggValueBits) - 1;
constexpr uint64_t kAggEpochMask = (1ull << 42) - 1;
constexpr int kMaxClusters = 8;

struct LayoutArgs {
    const int64_t *topk;
    int T, k, E, R, N, epr, rpn;
    int32_t *per_expert, *per_rank, *per_node;
    uint8_t *in_rank;
    WsHeader *hdr;
    int32_t *pair_rank;
    int32_t *ws_counts;
    uint64_t *state;
    int32_t *agg, *incl;
    int tiles, tile_tokens, cols, cols_pad;
    int csize, ccount;  // cluster form: blocks per cluster and clusters (tiles = csize * ccount)
    uint64_t *gagg;     // cluster form, ccount > 1: [ccount][cols_pad] published cluster counts
    int rank_shift, node_shift;  // log2(E/R), log2(R/N) when powers of two, else -1
    int32_t *start_out;  // optional: expert offsets written by the last tile (fused step 2)
    int32_t *total_out;
    int alignment;
    int32_t *status;
    int stalled_tile;
    uint32_t spin_limit;
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// kChunks: 32-pair chunks per warp at most (a tile holds up to W * 32 * kChunks pairs).
// kForm 1 (one cluster) and 2 (several): the tiles are the blocks of thread-block
// clusters that all run at once (tile = cluster index * blocks per cluster + rank in
// the cluster); each block pushes its counts into the shared memory of every later
// block of its cluster and one cluster barrier completes every prefix inside the
// cluster (no ticket). With several clusters, each cluster's last block then
// publishes the cluster's counts in global memory (self-tagged 64-bit words) and the
// blocks of later clusters add those of the clusters before theirs. kForm 0: tiles
// are handed out by ticket and chained by the decoupled look-back.
// Byte offsets of the layout kernel's shared-memory regions; every region that is
// read or written with 16-byte vectors starts on a 16-byte boundary.
struct LayoutSmem {
    size_t rmask, nmask, hist, lanes, agg, excl, rank_of, node_of, pick, stage, total;
};

__host__ __device__ inline LayoutSmem layout_smem(int E, int W, int cols_pad, int tile_tokens,
                                                  int64_t tile_pairs, int stage_rows) {
    LayoutSmem m;
    m.rmask = 0;
    m.nmask = m.rmask + (size_t)tile_tokens * 8;
    m.hist = m.nmask + (size_t)tile_tokens * 8;
    m.lanes = align_up(m.hist + (size_t)W * (E + 1) * 4, 16);
    m.agg = align_up(m.lanes + (W >= 16 ? (size_t)W * E * 4 : 0), 16);
    m.excl = m.agg + (size_t)cols_pad * 4;
    m.rank_of = m.excl + (size_t)cols_pad * 4;
    m.node_of = m.rank_of + (size_t)E * 4;
    m.pick = align_up(m.node_of + (size_t)E * 4, 16);
    m.stage = align_up(m.pick + (size_t)tile_pairs * 2, 16);
    m.total = m.stage + (size_t)stage_rows * cols_pad * 4;
    return m;
}

template <int W, int kChunks, int kForm>
__global__ void __launch_bounds__(W * 32, 1) layout_kernel(LayoutArgs a) {
    constexpr int kThreads = W * 32;
    constexpr bool kCluster = kForm >= 1, kMulti = kForm == 2;
    // lane-mask words per warp and expert for E <= 1024 (16 or 32 warps); wider
    // expert sets keep their shared memory for the histograms and use ballots
    constexpr bool kLaneWords = W >= 16;
    extern __shared__ int4 smem_raw[];
    char *sm = reinterpret_cast<char *>(smem_raw);
    const LayoutSmem L = layout_smem(a.E, W, a.cols_pad, a.tile_tokens,
                                     (int64_t)a.tile_tokens * a.k, 0);
    unsigned long long *tok_rmask = reinterpret_cast<unsigned long long *>(sm + L.rmask);  // ranks
    unsigned long long *tok_nmask = reinterpret_cast<unsigned long long *>(sm + L.nmask);  // nodes
    // [W][E + 1] warp histograms -> warp bases; rows padded by one word so that the
    // per-expert scan across warps (stride of one row) hits 32 different banks
    const int hws = a.E + 1;
    int *hw = reinterpret_cast<int *>(sm + L.hist);
    // [W][E] per warp and expert: the lanes of the warp's current chunk holding that
    // expert (a bit mask), zero between chunks
    uint32_t *lanes_of = reinterpret_cast<uint32_t *>(sm + L.lanes);
    int *col_agg = reinterpret_cast<int *>(sm + L.agg);    // [cols_pad] this tile's counts
    int *col_excl = reinterpret_cast<int *>(sm + L.excl);  // [cols_pad] counts of earlier tiles
    int *rank_of = reinterpret_cast<int *>(sm + L.rank_of);  // [E] simulated rank of each expert
    int *node_of = reinterpret_cast<int *>(sm + L.node_of);  // [R] simulated node of each rank
    int16_t *s_pick = reinterpret_cast<int16_t *>(sm + L.pick);  // [tile pairs] expert or -1
    // cluster: [tiles][cols_pad] counts of the earlier blocks, sent by each of them
    int *s_stage = reinterpret_cast<int *>(sm + L.stage);
    __shared__ int s_tile;
    __shared__ uint64_t s_epoch;
    __shared__ int s_win_aggs, s_win_incl, s_win_done;
    __shared__ int s_red[W], s_red2[W];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < a.cols_pad; i += kThreads) {
        col_agg[i] = 0;
        col_excl[i] = 0;
    }
    for (int e = tid; e < a.E; e += kThreads) rank_of[e] = e / a.epr;
    for (int r = tid; r < a.R; r += kThreads) node_of[r] = r / a.rpn;
    // cluster: this block has started; the other blocks store into its shared memory
    // only once every block has arrived here (nothing written so far is read by
    // another block, so the arrival orders no writes)
    if constexpr (kCluster) cluster_arrive_relaxed();
    // The tile ticket is taken before the dependency wait. It wraps to 0 by itself once
    // all `tiles` tickets of a call are handed out, and the next kernel on the stream
    // can only start once every block of this one has taken its ticket (the trigger
    // below follows it), so a layout call issued right after this one -- on the same
    // workspace -- starts from ticket 0 whatever the timing. Everything else the call
    // reads from the workspace (the call counter, the look-back state) and topk_idx
    // (which the kernel before may write) is read after the wait, when every earlier
    // call has completed. A call with one tile needs none of it (no look-back).
    const bool multi = !kCluster && a.tiles > 1;  // ticket, look-back and call counter
    if (tid == 0)
        s_tile = kMulti ? (int)(cluster_id_x() * a.csize + cluster_ctarank())
                 : kCluster ? (int)cluster_ctarank()
                 : multi ? (int)atomicInc(&a.hdr->ticket, (unsigned)(a.tiles - 1)) : 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // the call counter, read before this block's cluster barrier: once a cluster's
    // counts are published, every block of that cluster has read it
    if (tid == 0) s_epoch = (multi || kMulti) ? ld_relaxed_gpu(&a.hdr->epoch) : 0ull;
    const int tile = s_tile;
    const int crank = kMulti ? tile % a.csize : tile;  // rank inside the cluster
    const int t0 = tile * a.tile_tokens;
    const int ntok = max(0, min(a.tile_tokens, a.T - t0));
    const int npairs = ntok * a.k;
    const int64_t pair0 = (int64_t)t0 * a.k;

    // (1) warp w owns a contiguous run of cpw 32-pair chunks of the tile, in
    // row-major order: pairs [32 cpw w, 32 cpw (w + 1)) (warp-major order, which the
    // scan across warps relies on). A full tile has kChunks chunks per warp; a
    // partial one spreads its pairs over all warps, and chunks past its last pair
    // are skipped. All of a lane's picks are loaded at once, then each chunk is
    // ranked: lanes holding the same expert find each other through the expert's
    // lane-mask word, and the lowest of them adds the group's size to the warp's
    // private histogram.
    int pe[kChunks], pr[kChunks];
    const int cpw = max(1, min(kChunks, (npairs + kThreads - 1) / kThreads));
    const int p_base = warp * 32 * cpw + lane;
    const int live = min(cpw, max(0, (npairs - (p_base - lane) + 31) >> 5));
    int64_t pv[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int p = p_base + 32 * c;
        pv[c] = (c < cpw && p < npairs) ? __ldg(a.topk + pair0 + p) : -1;
    }
    // while the picks are in flight, the warp zeroes its own histogram row (the lane
    // words need no zeroing: each chunk clears the words it uses before setting them)
    int *my_hist = hw + warp * hws;
    for (int i = lane; i < hws; i += 32) my_hist[i] = 0;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int64_t v = pv[c];
        pe[c] = (v >= 0 && v < a.E) ? (int)v : -1;
        if (v < -1 || v >= a.E) report(a.status, EPD_ERR_INVALID_EXPERT);
    }
    // the picks, for the per-token rank and node masks of step (3)
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int p = p_base + 32 * c;
        if (c < live && p < npairs) s_pick[p] = (int16_t)pe[c];
    }
    uint32_t *my_lanes = lanes_of + warp * a.E;
    __syncwarp();  // the row is zero for every lane of the warp
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        pr[c] = 0;
        if (c >= live) continue;
        const int e = pe[c];
        // the lanes holding the same expert: every lane clears the expert's word, then
        // sets its bit in it, then reads the word back (a shared-memory atomic OR and a
        // load cost a fraction of the one-ballot-per-id-bit search they replace); every
        // lane reads the group's count before the group's lowest lane adds to it; the
        // warp stays converged (whole-warp syncs only). The syncs of the next chunk
        // order its reads after this chunk's count update.
        uint32_t peers;
        if constexpr (kLaneWords) {
            if (e >= 0) my_lanes[e] = 0u;
            __syncwarp();
            if (e >= 0) atomicOr(&my_lanes[e], 1u << lane);
            __syncwarp();
            peers = e >= 0 ? my_lanes[e] : 0u;
        } else {
            // E > 1024: one ballot per id bit instead (no lane words: shared memory)
            peers = __ballot_sync(0xffffffffu, e >= 0);
#pragma unroll
            for (int b = 0; b < 12; ++b) {  // ids below 4096; higher bits are 0 for valid lanes
                const uint32_t set = __ballot_sync(0xffffffffu, (e >> b) & 1);
                peers &= ((e >> b) & 1) ? set : ~set;
            }
        }
        const int before = __popc(peers & lanemask_lt());
        const int base = e >= 0 ? my_hist[e] : 0;
        pr[c] = base + before;
        __syncwarp();
        if (e >= 0 && before == 0) my_hist[e] = base + __popc(peers);
        if constexpr (!kLaneWords) __syncwarp();
    }

    __syncthreads();

    // (2) exclusive scan of the warp histograms per expert: one thread per expert
    // walks the W rows (consecutive experts are consecutive words: no bank
    // conflicts), and the tile's count per expert
    for (int e = tid; e < a.E; e += kThreads) {
        constexpr int G = W < 8 ? W : 8;  // rows loaded per batch
        int run = 0;
#pragma unroll
        for (int w0 = 0; w0 < W; w0 += G) {
            int v[G];
#pragma unroll
            for (int q = 0; q < G; ++q) v[q] = hw[(w0 + q) * hws + e];
#pragma unroll
            for (int q = 0; q < G; ++q) {
                hw[(w0 + q) * hws + e] = run;
                run += v[q];
            }
        }
        col_agg[e] = run;
    }

    // (3) one lane per token, warps taken from the top so that they run beside the
    // scan above: the ranks and nodes the token reaches (read from its picks in
    // shared memory), as bit masks when R, N <= 64 (a token counts once per rank and
    // once per node) -- 32-bit masks from shifts alone when R, N <= 32 and E/R, R/N
    // are powers of two, the top-8 row as one 16-byte load -- and the tile's tokens
    // per rank and per node by counting the columns of the warp's masks; for R or N
    // above 64 each token counts its distinct ranks or nodes by comparing its picks
    const bool small_r = a.R <= 64, small_n = a.N <= 64;
    const bool fastm = a.rank_shift >= 0 && a.node_shift >= 0 && a.R <= 32 && a.N <= 32;
    for (int base = (W - 1 - warp) * 32; base < ntok; base += kThreads) {
        const int tl = base + lane;
        unsigned long long rm = 0, nm = 0;
        if (tl < ntok && fastm) {
            // shifts for rank and node, R, N <= 32: 32-bit masks, no table look-ups;
            // top-8 rows loaded as one 16-byte vector
            const int16_t *row = s_pick + tl * a.k;
            uint32_t r32 = 0u, n32 = 0u;
            const int rs = a.rank_shift, ns = a.node_shift;
            if (a.k == 8) {
                const uint4 v = *reinterpret_cast<const uint4 *>(row);
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int e = (int)(int16_t)(wv[j >> 1] >> (16 * (j & 1)));
                    const int r = e >> rs;
                    r32 |= e >= 0 ? 1u << r : 0u;
                    n32 |= e >= 0 ? 1u << (r >> ns) : 0u;
                }
            } else {
                for (int j = 0; j < a.k; ++j) {
                    const int e = row[j];
                    const int r = e >> rs;
                    r32 |= e >= 0 ? 1u << r : 0u;
                    n32 |= e >= 0 ? 1u << (r >> ns) : 0u;
                }
            }
            rm = r32;
            nm = n32;
            tok_rmask[tl] = rm;
            tok_nmask[tl] = nm;
        } else if (tl < ntok) {
            const int16_t *row = s_pick + tl * a.k;
            for (int j = 0; j < a.k; ++j) {
                const int e = row[j];
                if (e < 0) continue;
                const int r = a.rank_shift >= 0 ? e >> a.rank_shift : rank_of[e];
                const int n = a.node_shift >= 0 ? r >> a.node_shift : node_of[r];
                if (small_r) rm |= 1ull << r;
                if (small_n) nm |= 1ull << n;
                if (!small_r || !small_n) {
                    bool new_r = !small_r, new_n = !small_n;
                    for (int j2 = 0; j2 < j && (new_r || new_n); ++j2) {
                        const int e2 = row[j2];
                        if (e2 < 0) continue;
                        const int r2 = rank_of[e2];
                        if (r2 == r) new_r = false;
                        if (node_of[r2] == n) new_n = false;
                    }
                    if (new_r) atomicAdd(&col_agg[a.E + r], 1);
                    if (new_n) atomicAdd(&col_agg[a.E + a.R + n], 1);
                }
            }
            tok_rmask[tl] = rm;
            tok_nmask[tl] = nm;
        }
        // lane b of group g ends up with the warp's count for bit 32 g + b
        for (int g = 0; g < 2; ++g) {
            if (small_r && 32 * g < a.R) {
                const int cr = bit_column_count((uint32_t)(rm >> (32 * g)), lane);
                if (cr) atomicAdd(&col_agg[a.E + 32 * g + lane], cr);
            }
            if (small_n && 32 * g < a.N) {
                const int cn = bit_column_count((uint32_t)(nm >> (32 * g)), lane);
                if (cn) atomicAdd(&col_agg[a.E + a.R + 32 * g + lane], cn);
            }
        }
    }
    __syncthreads();

    if constexpr (kCluster) {
        // (4') every block of the cluster has started: send this tile's counts, as 16-byte
        // vectors, into row `tile` of the staging area of every later block -- the expert
        // columns to each of them, all columns to the last one (which writes the totals)
        cluster_wait_acquire();
        const int later = a.csize - 1 - crank;
        const int nv_e = (a.E + 3) >> 2, nv_all = a.cols_pad >> 2;
        const int n_mid = later > 0 ? (later - 1) * nv_e : 0;
        const int n_send = later > 0 ? n_mid + nv_all : 0;
        const int4 *row = reinterpret_cast<const int4 *>(col_agg);
        int *dst_row = s_stage + crank * a.cols_pad;
        for (int i = tid; i < n_send; i += kThreads) {
            int d, v;
            if (i < n_mid) {
                d = i / nv_e;
                v = i - d * nv_e;
                d += crank + 1;
            } else {
                d = a.csize - 1;
                v = i - n_mid;
            }
            cluster_st_v4(cluster_map(dst_row + 4 * v, (uint32_t)d), row[v]);
        }
        cluster_arrive_release();
    }

    // (4) publish this tile's counts (tile 0 has no predecessor: its counts are its
    // prefix). The block barrier orders every thread's stores before thread 0's
    // release store of the state word.
    const bool publish = multi && tile != a.stalled_tile;
    const uint64_t epoch = s_epoch;  // written by thread 0 before the barriers above
    const uint64_t tag = kStateMark | (epoch << 2);
    int32_t *my_agg = a.agg + (size_t)tile * a.cols_pad;
    int32_t *my_incl = a.incl + (size_t)tile * a.cols_pad;
    if (multi) {
        for (int c = tid; c < a.cols; c += kThreads) {
            if (tile == 0) my_incl[c] = col_agg[c];
            else my_agg[c] = col_agg[c];
        }
        __syncthreads();
    }
    if (tid == 0 && publish)
        st_release_gpu(&a.state[tile], tag | (tile == 0 ? kStateIncl : kStateAgg));

    // is_token_in_rank rows of the tile, after publishing (nothing waits on them):
    // one contiguous [ntok, R] byte block, written in coalesced 4-byte words where
    // it is 4-byte aligned
    if (a.in_rank) {
        uint8_t *blk = a.in_rank + (int64_t)t0 * a.R;
        const int nbytes = ntok * a.R;
        if (small_r && (a.R & 15) == 0 && (reinterpret_cast<uintptr_t>(a.in_rank) & 15) == 0) {
            // one token per thread: its row of R bytes as 16-byte vectors, byte r = bit r
            // of the token's rank mask (rows are 16-byte aligned as R % 16 == 0)
            for (int tl = tid; tl < ntok; tl += kThreads) {
                const unsigned long long m = tok_rmask[tl];
                int4 *dst = reinterpret_cast<int4 *>(blk + (int64_t)tl * a.R);
                for (int v = 0; v < (a.R >> 4); ++v) {
                    const uint32_t bits = (uint32_t)(m >> (16 * v));
                    dst[v] = make_int4(spread4(bits), spread4(bits >> 4), spread4(bits >> 8),
                                       spread4(bits >> 12));
                }
            }
        } else if (small_r && (a.R & 3) == 0 && (reinterpret_cast<uintptr_t>(blk) & 3) == 0) {
            // each word holds 4 ranks of one token: spread 4 mask bits into 4 bytes
            const int wpr = a.R >> 2;  // words per row
            uint32_t *words = reinterpret_cast<uint32_t *>(blk);
            for (int wi = tid; wi < (nbytes >> 2); wi += kThreads) {
                const int tl = wi / wpr;
                const uint32_t m = (uint32_t)(tok_rmask[tl] >> ((wi - tl * wpr) << 2)) & 0xFu;
                words[wi] = (m & 1u) | ((m & 2u) << 7) | ((m & 4u) << 14) | ((m & 8u) << 21);
            }
        } else {
            for (int i = tid; i < nbytes; i += kThreads) {
                const int tl = i / a.R, r = i - tl * a.R;
                bool hit = false;
                if (small_r) {
                    hit = (tok_rmask[tl] >> r) & 1ull;
                } else {
                    const int16_t *row = s_pick + tl * a.k;
                    for (int j = 0; j < a.k && !hit; ++j) {
                        const int e = row[j];
                        hit = e >= 0 && rank_of[e] == r;
                    }
                }
                blk[i] = hit ? 1 : 0;
            }
        }
    }

    // cluster: the barrier completes once every block's rows have landed, and no block
    // touches another's shared memory after it (so any block may exit); the prefix of
    // this tile is the sum of the rows of the earlier tiles
    if constexpr (kCluster) {
        cluster_wait_acquire();
        const int ncol = crank == a.csize - 1 ? a.cols : a.E;
        for (int c = tid; c < ncol; c += kThreads) {
            int sum = 0;
            for (int t = 0; t < crank; ++t) sum += s_stage[t * a.cols_pad + c];
            col_excl[c] = sum;
        }
        __syncthreads();
        if constexpr (kMulti) {
            // several clusters: the last block of every cluster but the last publishes
            // the cluster's counts (all columns); the blocks of cluster g add those of
            // clusters 0..g-1 to their prefixes (all columns for the grid's last block,
            // which writes the totals), loading every word at once and polling again,
            // bounded, only where a cluster has not published yet
            const int cid = tile / a.csize;
            const uint64_t mark = kStateMark | ((s_epoch & kAggEpochMask) << kAggValueBits);
            if (crank == a.csize - 1 && cid < a.ccount - 1) {
                uint64_t *mine = a.gagg + (size_t)cid * a.cols_pad;
                for (int c = tid; c < a.cols; c += kThreads)
                    st_relaxed_gpu(&mine[c], mark | (uint64_t)(uint32_t)(col_excl[c] + col_agg[c]));
            }
            if (cid > 0) {
                const int ncol2 = tile == a.tiles - 1 ? a.cols : a.E;
                for (int c = tid; c < ncol2; c += kThreads) {
                    uint64_t v[kMaxClusters - 1];
#pragma unroll
                    for (int g = 0; g < kMaxClusters - 1; ++g)
                        v[g] = g < cid ? ld_relaxed_gpu(a.gagg + (size_t)g * a.cols_pad + c) : mark;
                    int sum = 0;
#pragma unroll
                    for (int g = 0; g < kMaxClusters - 1; ++g) {
                        if (g >= cid) break;
                        uint32_t polls = 0;
                        unsigned ns = 32;
                        while ((v[g] & ~kAggValueMask) != mark) {
                            if (++polls >= a.spin_limit) {
                                report(a.status, EPD_ERR_TIMEOUT);
                                v[g] = mark;
                                break;
                            }
                            __nanosleep(ns);
                            if (ns < 256) ns <<= 1;
                            v[g] = ld_relaxed_gpu(a.gagg + (size_t)g * a.cols_pad + c);
                        }
                        sum += (int)(v[g] & kAggValueMask);
                    }
                    col_excl[c] += sum;
                }
            }
            __syncthreads();
            // every block of the call has read the call counter (the clusters before
            // published, this cluster passed its barrier): advance it for the next call
            if (tile == a.tiles - 1 && tid == 0) a.hdr->epoch = s_epoch + 1;
        }
    }

    // (5) decoupled look-back over earlier tiles
    if (multi && tile > 0) {
        int pos = tile - 1;
        while (true) {
            if (warp == 0) {
                const int idx = pos - lane;
                uint32_t polls = 0;
                unsigned ns = 32;
                int win_aggs = 0, win_incl = -1, done = 1;
                while (true) {
                    uint32_t st = kStateIncl;  // before tile 0: an empty inclusive prefix
                    if (idx >= 0) {
                        const uint64_t v = ld_acquire_gpu(&a.state[idx]);
                        st = ((v & ~3ull) == tag) ? (uint32_t)(v & 3ull) : 0u;
                    }
                    const uint32_t incl_mask = __ballot_sync(0xffffffffu, st == kStateIncl);
                    const uint32_t wait_mask = __ballot_sync(0xffffffffu, st == 0);
                    const uint32_t need =
                        incl_mask ? (((incl_mask & (0u - incl_mask)) << 1) - 1u) : 0xffffffffu;
                    if ((wait_mask & need) == 0) {
                        if (incl_mask) {
                            const int first = __ffs(incl_mask) - 1;
                            win_aggs = first;
                            win_incl = pos - first;  // negative when it is the empty prefix
                            done = 1;
                        } else {
                            win_aggs = 32;
                            win_incl = -1;
                            done = 0;
                        }
                        break;
                    }
                    if (++polls >= a.spin_limit) {
                        if (lane == 0) report(a.status, EPD_ERR_TIMEOUT);
                        win_aggs = 0;
                        win_incl = -1;
                        done = 1;
                        break;
                    }
                    __nanosleep(ns);
                    if (ns < 256) ns <<= 1;
                }
                if (lane == 0) {
                    s_win_aggs = win_aggs;
                    s_win_incl = win_incl;
                    s_win_done = done;
                }
            }
            __syncthreads();
            const int wa = s_win_aggs, wi = s_win_incl, wdone = s_win_done;
            for (int c = tid; c < a.cols; c += kThreads) {
                // all window rows are loaded at once: one L2 round trip, not one per row
                const int32_t *col = a.agg + (size_t)pos * a.cols_pad + c;
                int sum = 0;
#pragma unroll
                for (int l = 0; l < 32; ++l)
                    if (l < wa) sum += __ldcg(col - (size_t)l * a.cols_pad);
                if (wi >= 0) sum += __ldcg(a.incl + (size_t)wi * a.cols_pad + c);
                col_excl[c] += sum;
            }
            __syncthreads();
            if (wdone) break;
            pos -= 32;
        }
        // (6) publish the inclusive prefix. Tiles 1..32 reach the empty prefix before
        // tile 0 inside their first window, so only a call with more than 33 tiles
        // has a later tile that can stop on it (none needs it: aggregates suffice).
        if (a.tiles > 33 && tile < a.tiles - 1) {
            for (int c = tid; c < a.cols; c += kThreads) my_incl[c] = col_excl[c] + col_agg[c];
            __syncthreads();
            if (tid == 0 && publish) st_release_gpu(&a.state[tile], tag | kStateIncl);
        }
    }

    // (7) the last tile (in ticket order, or the cluster's last block) holds the
    // totals. For E <= 1024 the first 8 warps write them while the others store the
    // pair ranks: each of their 256 threads owns a contiguous run of experts (their
    // counts, their sum P and, for the fused step 2, the exclusive prefix sum of the
    // padded counts by a shuffle scan of the runs, then of the 8 warps' sums, between
    // barriers of those 8 warps only); warp 8 writes the per-rank and per-node counts.
    const bool last = tile == a.tiles - 1;
    const bool warp_totals = a.E <= 1024;  // W >= 16 warps
    auto padded = [&](int c) {
        return a.alignment == 1 ? c : (c + a.alignment - 1) / a.alignment * a.alignment;
    };
    if (last && warp_totals && warp < 8) {
        const int per = (a.E + 255) >> 8;
        const int e0 = min(a.E, tid * per), e1 = min(a.E, e0 + per);
        int part = 0, run = 0;
        for (int e = e0; e < e1; ++e) {
            const int tot = col_excl[e] + col_agg[e];
            if (a.per_expert) a.per_expert[e] = tot;
            a.ws_counts[e] = tot;
            part += tot;
            run += padded(tot);
        }
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        part = warp_sum(part);
        if (lane == 31) {
            s_red[warp] = incl;
            s_red2[warp] = part;
        }
        named_barrier_sync(1, 256);
        if (warp == 0) {
            const int v = lane < 8 ? s_red[lane] : 0;
            int wincl = v;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, wincl, o);
                if (lane >= o) wincl += n;
            }
            const int P = warp_sum(lane < 8 ? s_red2[lane] : 0);
            if (lane < 8) s_red[lane] = wincl - v;
            if (lane == 7) {
                a.hdr->total_pairs = P;
                a.hdr->num_tokens = a.T;
                a.hdr->num_topk = a.k;
                if (a.start_out) *a.total_out = wincl;
            }
        }
        if (a.start_out) {
            named_barrier_sync(1, 256);
            int pos = s_red[warp] + incl - run;
            for (int e = e0; e < e1; ++e) {
                a.start_out[e] = pos;
                pos += padded(col_excl[e] + col_agg[e]);
            }
        }
    } else if (last && warp_totals && warp == 8) {
        for (int c = a.E + lane; c < a.cols; c += 32) {
            const int tot = col_excl[c] + col_agg[c];
            if (c < a.E + a.R) {
                if (a.per_rank) a.per_rank[c - a.E] = tot;
            }
            else if (a.per_node) a.per_node[c - a.E - a.R] = tot;
        }
    }

    // (8) rank of every pair inside its expert over the whole batch
    const int *my_base = hw + warp * hws;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        const int p = p_base + 32 * c;
        if (c < cpw && p < npairs) {
            const int e = pe[c];
            a.pair_rank[pair0 + p] = e >= 0 ? col_excl[e] + my_base[e] + pr[c] : -1;
        }
    }

    // (8') the totals for E > 1024 (blocks of 4 or 8 warps): each thread owns a
    // contiguous run of experts; a warp-shuffle scan of the runs, then of the warps'
    // sums
    if (last && !warp_totals) {
        const int per = (a.E + kThreads - 1) / kThreads;
        const int e0 = min(a.E, tid * per), e1 = min(a.E, e0 + per);
        int part = 0, run = 0;
        for (int e = e0; e < e1; ++e) {
            const int tot = col_excl[e] + col_agg[e];
            if (a.per_expert) a.per_expert[e] = tot;
            a.ws_counts[e] = tot;
            part += tot;
            run += padded(tot);
        }
        for (int c = a.E + tid; c < a.cols; c += kThreads) {
            const int tot = col_excl[c] + col_agg[c];
            if (c < a.E + a.R) {
                if (a.per_rank) a.per_rank[c - a.E] = tot;
            }
            else if (a.per_node) a.per_node[c - a.E - a.R] = tot;
        }
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        part = warp_sum(part);
        if (lane == 31) {
            s_red[warp] = incl;
            s_red2[warp] = part;
        }
        __syncthreads();
        if (warp == 0) {
            const int v = lane < W ? s_red[lane] : 0;
            int wincl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, wincl, o);
                if (lane >= o) wincl += n;
            }
            const int P = warp_sum(lane < W ? s_red2[lane] : 0);
            if (lane < W) s_red[lane] = wincl - v;
            if (lane == 31) {
                a.hdr->total_pairs = P;
                a.hdr->num_tokens = a.T;
                a.hdr->num_topk = a.k;
                if (a.start_out) *a.total_out = wincl;
            }
        }
        if (a.start_out) {
            __syncthreads();
            int pos = s_red[warp] + incl - run;
            for (int e = e0; e < e1; ++e) {
                a.start_out[e] = pos;
                pos += padded(col_excl[e] + col_agg[e]);
            }
        }
    }

    // (9) the last block to finish advances the call counter for the next call (which
    // reads it only after its dependency wait, once this call has completed); the
    // finished-block count wraps back to 0 by itself
    if (multi) {
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atomicInc(&a.hdr->done, (unsigned)(a.tiles - 1));
            if (prev == (unsigned)a.tiles - 1) {
                a.hdr->epoch = epoch + 1;
                __threadfence();
            }
        }
    }
}

size_t layout_smem_bytes(int E, int cols_pad, int tile_tokens, int64_t tile_pairs,
                         int stage_rows) {
    return layout_smem(E, layout_warps(E), cols_pad, tile_tokens, tile_pairs, stage_rows).total;
}

constexpr int kMaxCluster = 16;         // blocks of the cluster form (non-portable above 8)
constexpr int kClusterMaxChunks = 8;    // 32-pair chunks per warp in the cluster form

// Raises the kernel's dynamic shared-memory limit to `smem` if needed (per device).
template <typename K>
epd_status_t opt_in_smem(K kernel, size_t smem) {
    if (smem <= 48 * 1024) return EPD_OK;
    // the opt-in limit covers static and dynamic shared memory together
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
        return record_cuda_error();
    if (smem + fa.sharedSizeBytes > (size_t)optin) return EPD_ERR_UNSUPPORTED;
    if ((int)smem > fa.maxDynamicSharedSizeBytes &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return record_cuda_error();
    return EPD_OK;
}

template <int W, int CH>
epd_status_t launch_tiles(const LayoutArgs &a, size_t smem, cudaStream_t stream) {
    auto kernel = layout_kernel<W, CH, 0>;
    const epd_status_t st = opt_in_smem(kernel, smem);
    if (st != EPD_OK) return st;
    return launch_pdl(kernel, a.tiles, W * 32, smem, stream, a);
}

// How many clusters of C blocks of layout_kernel<W, CH, F> with `smem` bytes each
// can run at once on the current device, 0 if none (the answer for the last size
// asked is kept per device and cluster width).
template <int W, int CH, int F>
int cluster_capacity(int C, size_t smem) {
    static std::atomic<unsigned long long> last[64][2];  // (smem << 8 | count) + 1, 0 = unknown
    auto kernel = layout_kernel<W, CH, F>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int slot = C > 8 ? 1 : 0;
    std::atomic<unsigned long long> *cache =
        (dev >= 0 && dev < 64) ? &last[dev][slot] : nullptr;
    if (cache) {
        const unsigned long long v = cache->load(std::memory_order_acquire);
        if (v != 0 && ((v - 1) >> 8) == smem) return (int)((v - 1) & 0xffu);
    }
    bool fits = opt_in_smem(kernel, smem) == EPD_OK;
    if (fits && C > 8 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        fits = false;
    }
    int n = 0;
    if (fits) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)C);
        cfg.blockDim = dim3((unsigned)(W * 32));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    }
    n = n < 0 ? 0 : (n > 255 ? 255 : n);
    if (cache) cache->store(((unsigned long long)smem << 8 | (unsigned)n) + 1,
                            std::memory_order_release);
    return n;
}

template <int W, int CH, int F>
epd_status_t launch_cluster(const LayoutArgs &a, size_t smem, cudaStream_t stream) {
    return launch_pdl_cluster(layout_kernel<W, CH, F>, a.tiles, W * 32, smem, a.csize, stream, a);
}

// Form F = 1 (one cluster) takes 1..8 chunks per warp; F = 2 (several clusters) 1..4.
template <int W, int F>
int cluster_capacity_any(int CH, int C, size_t smem) {
    switch (CH) {
        case 1: return cluster_capacity<W, 1, F>(C, smem);
        case 2: return cluster_capacity<W, 2, F>(C, smem);
        case 4: return cluster_capacity<W, 4, F>(C, smem);
        default: return F == 1 ? cluster_capacity<W, 8, 1>(C, smem) : 0;
    }
}

template <int W, int F>
epd_status_t launch_cluster_any(int CH, const LayoutArgs &a, size_t smem, cudaStream_t stream) {
    switch (CH) {
        case 1: return launch_cluster<W, 1, F>(a, smem, stream);
        case 2: return launch_cluster<W, 2, F>(a, smem, stream);
        case 4: return launch_cluster<W, 4, F>(a, smem, stream);
        default: return F == 1 ? launch_cluster<W, 8, 1>(a, smem, stream) : EPD_ERR_UNSUPPORTED;
    }
}

// The cluster form for a batch of `pairs` (token, pick) pairs: blocks per cluster C (a
// power of two, 2..16, about one block per 1024 pairs), clusters G and chunks per warp,
// or C = 0 when the batch fits one tile, exceeds what the form holds, or the device
// cannot co-schedule the clusters. A batch that would give one cluster of 16 blocks
// kMultiMinChunks or more chunks per warp is spread over up to kMaxClusters clusters
// that all fit on the device at once, one block per SM, when the workspace's
// look-back rows (which then hold the clusters' published counts: 2 G rows of 32-bit
// words) are enough.
struct ClusterPlan {
    int C, G, chunks, tile_tokens;
    size_t smem;
};

constexpr int kMultiMinChunks = 8;

// Shared memory per block that keeps two of them off one SM (per device).
size_t one_block_per_sm_smem() {
    static std::atomic<int> by_dev[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int v = (dev >= 0 && dev < 64) ? by_dev[dev].load(std::memory_order_acquire) : 0;
    if (v == 0) {
        int per_sm = 0;
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        v = (int)align_up((size_t)per_sm / 2 + 1024, 16);
        if (dev >= 0 && dev < 64) by_dev[dev].store(v, std::memory_order_release);
    }
    return (size_t)v;
}

ClusterPlan plan_cluster(int T, int k, int E, int cols_pad, int ws_tiles) {
    ClusterPlan p = {0, 1, 0, 0, 0};
    const int W = layout_warps(E);
    const int64_t pairs = (int64_t)T * k;
    if (W < 16 || pairs <= kLayoutTilePairs) return p;
    int C = 2;
    while (C < kMaxCluster && (int64_t)C * kLayoutTilePairs < pairs) C *= 2;
    for (; C >= 2; C /= 2) {
        const int tt = (T + C - 1) / C;
        const int64_t tp = (int64_t)tt * k;
        if (tt > kLayoutMaxTileTokens || tp > (int64_t)W * 32 * kClusterMaxChunks) return p;
        int ch = 1;
        while ((int64_t)ch * W * 32 < tp) ch *= 2;
        const size_t smem = layout_smem_bytes(E, cols_pad, tt, tp, C);
        const int n = W == 32 ? cluster_capacity_any<32, 1>(ch, C, smem)
                              : cluster_capacity_any<16, 1>(ch, C, smem);
        if (n >= 1) {
            p.C = C;
            p.chunks = ch;
            p.tile_tokens = tt;
            p.smem = smem;
            break;
        }
    }
    if (p.C != kMaxCluster || p.chunks < kMultiMinChunks || pairs >= (1ll << kAggValueBits))
        return p;
    const size_t one = one_block_per_sm_smem();
    for (int G = p.chunks < kMaxClusters ? p.chunks : kMaxClusters; G >= 2; G /= 2) {
        if (2 * G > ws_tiles) continue;
        const int tt = (T + C * G - 1) / (C * G);
        const int64_t tp = (int64_t)tt * k;
        int ch = 1;
        while ((int64_t)ch * W * 32 < tp) ch *= 2;
        size_t smem = layout_smem_bytes(E, cols_pad, tt, tp, C);
        if (smem < one) smem = one;
        const int n = W == 32 ? cluster_capacity_any<32, 2>(ch, C, smem)
                              : cluster_capacity_any<16, 2>(ch, C, smem);
        if (n >= G) {
            p.G = G;
            p.chunks = ch;
            p.tile_tokens = tt;
            p.smem = smem;
            break;
        }
    }
    return p;
}

epd_status_t layout_launch(int32_t *start_out, int32_t *total_out, int alignment,
                           const int64_t *topk_idx, int T, int k, int E, int R, int N,
                           int32_t *per_expert, int32_t *per_rank, int32_t *per_node,
                           uint8_t *in_rank, void *workspace, int32_t *status, int stalled_tile,
                           uint32_t spin_limit, cudaStream_t stream) {
    if (!topology_ok(T, k, E, R, N)) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (topk_idx == nullptr || !aligned8(topk_idx))) return EPD_ERR_INVALID_ARG;
    // the count outputs are optional only for the internal ranks-only launch
    if (status == nullptr || workspace == nullptr || (per_expert == nullptr) != (per_rank == nullptr))
        return EPD_ERR_INVALID_ARG;
    if (!aligned4(per_expert) || !aligned4(per_rank) || !aligned4(status) ||
        (per_node && !aligned4(per_node)) || !aligned16(workspace))
        return EPD_ERR_INVALID_ARG;
    if (spin_limit == 0) return EPD_ERR_INVALID_ARG;

    const WsLayout w = ws_layout(T, k, E, R, N);
    char *ws = static_cast<char *>(workspace);
    LayoutArgs a;
    a.topk = topk_idx;
    a.T = T;
    a.k = k;
    a.E = E;
    a.R = R;
    a.N = N;
    a.epr = E / R;
    a.rpn = R / N;
    a.per_expert = per_expert;
    a.per_rank = per_rank;
    a.per_node = per_node;
    a.in_rank = in_rank;
    a.hdr = reinterpret_cast<WsHeader *>(ws + w.header_off);
    a.pair_rank = reinterpret_cast<int32_t *>(ws + w.pair_rank_off);
    a.ws_counts = reinterpret_cast<int32_t *>(ws + w.counts_off);
    a.state = reinterpret_cast<uint64_t *>(ws + w.state_off);
    a.agg = reinterpret_cast<int32_t *>(ws + w.agg_off);
    a.incl = reinterpret_cast<int32_t *>(ws + w.incl_off);
    a.tiles = w.tiles;
    a.tile_tokens = layout_tile_tokens(k, E);
    a.start_out = start_out;
    a.total_out = total_out;
    a.alignment = alignment;
    auto log2_exact = [](int v) {
        int b = 0;
        while ((1 << b) < v) ++b;
        return (1 << b) == v ? b : -1;
    };
    a.rank_shift = log2_exact(a.epr);
    a.node_shift = log2_exact(a.rpn);
    a.cols = w.cols;
    a.cols_pad = w.cols_pad;
    a.status = status;
    a.stalled_tile = stalled_tile;
    a.spin_limit = spin_limit;
    // the failure-detection hook needs the look-back, so it always runs the tile form
    a.csize = 1;
    a.ccount = 1;
    a.gagg = nullptr;
    const ClusterPlan cp = stalled_tile < 0 ? plan_cluster(T, k, E, w.cols_pad, w.tiles)
                                            : ClusterPlan{0, 1, 0, 0, 0};
    if (cp.C > 0) {
        a.csize = cp.C;
        a.ccount = cp.G;
        a.tiles = cp.C * cp.G;
        a.tile_tokens = cp.tile_tokens;
        a.gagg = reinterpret_cast<uint64_t *>(ws + w.agg_off);
        if (cp.G > 1)
            return layout_warps(E) == 32 ? launch_cluster_any<32, 2>(cp.chunks, a, cp.smem, stream)
                                         : launch_cluster_any<16, 2>(cp.chunks, a, cp.smem, stream);
        return layout_warps(E) == 32 ? launch_cluster_any<32, 1>(cp.chunks, a, cp.smem, stream)
                                     : launch_cluster_any<16, 1>(cp.chunks, a, cp.smem, stream);
    }
    const size_t smem = layout_smem_bytes(E, w.cols_pad, a.tile_tokens,
                                          (int64_t)a.tile_tokens * k, 0);
    // a batch of one warp chunk per warp (a decode step) takes the one-chunk build
    if (a.tiles == 1 && (int64_t)T * k <= 1024 && layout_warps(E) == 32)
        return launch_tiles<32, 1>(a, smem, stream);
    switch (layout_warps(E)) {  // one tile of layout_tile_pairs(E) pairs per block
        case 32: return launch_tiles<32, kLayoutWideChunks>(a, smem, stream);
        case 16: return launch_tiles<16, kLayoutWideChunks>(a, smem, stream);
        case 8: return launch_tiles<8, kLayoutTilePairs / 256>(a, smem, stream);
        default: return launch_tiles<4, kLayoutTilePairs / 128>(a, smem, stream);
    }
}

}  // namespace

namespace {
thread_local int g_last_cuda_error = 0;
}

int last_cuda_error() { return g_last_cuda_error; }

epd_status_t record_cuda_error() {
    const cudaError_t e = cudaGetLastError();  // consume it: the caller's runtime state stays clean
    g_last_cuda_error = (int)e;
    return e == cudaSuccess ? EPD_OK : EPD_ERR_CUDA;
}

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace epd

extern "C" {

const char *epd_status_string(int code) {
    switch (code) {
        case EPD_OK: return "ok";
        case EPD_ERR_INVALID_ARG: return "invalid argument";
        case EPD_ERR_UNSUPPORTED: return "unsupported size";
        case EPD_ERR_CUDA: return "CUDA launch error";
        case EPD_ERR_INVALID_EXPERT: return "expert id outside [-1, E)";
        case EPD_ERR_TIMEOUT: return "look-back wait gave up";
        case EPD_ERR_CAPACITY: return "slot outside the permuted buffer";
        default: return "unknown status";
    }
}

int epd_version(void) { return 10000; }

int epd_last_cuda_error(void) { return epd::last_cuda_error(); }

size_t epd_workspace_bytes(int num_tokens, int num_topk, int num_experts, int num_ranks,
                           int num_rdma_ranks) {
    if (!epd::topology_ok(num_tokens, num_topk, num_experts, num_ranks, num_rdma_ranks)) return 0;
    return epd::ws_layout(num_tokens, num_topk, num_experts, num_ranks, num_rdma_ranks).total;
}

epd_status_t epd_workspace_init(void *workspace, size_t bytes, epd_stream_t stream) {
    if (workspace == nullptr || bytes < sizeof(epd::WsHeader)) return EPD_ERR_INVALID_ARG;
    cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream));
    return epd::record_cuda_error();
}

epd_status_t ep_dispatch_layout(const int64_t *topk_idx, int num_tokens, int num_topk,
                                int num_experts, int num_ranks, int num_rdma_ranks,
                                int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                int32_t *tokens_per_rdma_rank, uint8_t *is_token_in_rank,
                                void *workspace, int32_t *status, epd_stream_t stream) {
    if (!tokens_per_expert || !tokens_per_rank) return EPD_ERR_INVALID_ARG;
    return epd::layout_launch(nullptr, nullptr, 1, topk_idx, num_tokens, num_topk, num_experts, num_ranks,
                              num_rdma_ranks, tokens_per_expert, tokens_per_rank,
                              tokens_per_rdma_rank, is_token_in_rank, workspace, status, -1,
                              epd::kDefaultSpinLimit, reinterpret_cast<cudaStream_t>(stream));
}

epd_status_t ep_dispatch_layout_offsets(const int64_t *topk_idx, int num_tokens, int num_topk,
                                        int num_experts, int num_ranks, int num_rdma_ranks,
                                        int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                        int32_t *tokens_per_rdma_rank, uint8_t *is_token_in_rank,
                                        int alignment, int32_t *expert_start_loc,
                                        int32_t *total_rows, void *workspace, int32_t *status,
                                        epd_stream_t stream) {
    if (alignment < 1 || alignment > EPD_MAX_ALIGNMENT || !expert_start_loc || !total_rows ||
        !epd::aligned4(expert_start_loc) || !epd::aligned4(total_rows) || !tokens_per_expert ||
        !tokens_per_rank)
        return EPD_ERR_INVALID_ARG;
    return epd::layout_launch(expert_start_loc, total_rows, alignment, topk_idx, num_tokens,
                              num_topk, num_experts, num_ranks, num_rdma_ranks, tokens_per_expert,
                              tokens_per_rank, tokens_per_rdma_rank, is_token_in_rank, workspace,
                              status, -1, epd::kDefaultSpinLimit,
                              reinterpret_cast<cudaStream_t>(stream));
}

epd_status_t epd_test_layout_stalled_tile(const int64_t *topk_idx, int num_tokens, int num_topk,
                                          int num_experts, int num_ranks, int num_rdma_ranks,
                                          int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                          int32_t *tokens_per_rdma_rank,
                                          uint8_t *is_token_in_rank, void *workspace,
                                          int32_t *status, int stalled_tile,
                                          uint32_t spin_limit, epd_stream_t stream) {
    if (stalled_tile < 0 || spin_limit > epd::kDefaultSpinLimit || !tokens_per_expert ||
        !tokens_per_rank)
        return EPD_ERR_INVALID_ARG;
    return epd::layout_launch(nullptr, nullptr, 1, topk_idx, num_tokens, num_topk, num_experts, num_ranks,
                              num_rdma_ranks, tokens_per_expert, tokens_per_rank,
                              tokens_per_rdma_rank, is_token_in_rank, workspace, status,
                              stalled_tile, spin_limit, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace epd {
// The layout kernel for its workspace only (pair ranks, counts, header): no
// count outputs. Used by ep_dispatch_lowlatency for batches beyond its one-kernel
// form.
epd_status_t layout_ranks_only(const int64_t *topk_idx, int T, int k, int E, int R, int N,
                               void *workspace, int32_t *status, cudaStream_t stream) {
    return layout_launch(nullptr, nullptr, 1, topk_idx, T, k, E, R, N, nullptr, nullptr, nullptr,
                         nullptr, workspace, status, -1, kDefaultSpinLimit, stream);
}
}  // namespace epd

// ---------------------------------------------------------------------------- allocation-free variant
// Scratch for ep_dispatch_layout_noalloc: a file-scope device array that every
// GPU loading this library holds until the process exits. Host code must not
// pass `g_noalloc_scratch` itself to a kernel (on the host it names a host-side
// stand-in); it passes the device address resolved by cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EPD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void *> g_noalloc_addr[kMaxDevices];

// Device address of the scratch on the current device, resolved once per device.
epd_status_t noalloc_scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return epd::record_cuda_error();
    if (dev < 0 || dev >= kMaxDevices) return EPD_ERR_UNSUPPORTED;
    void *p = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            epd::record_cuda_error();
            return EPD_ERR_CUDA;
        }
        g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return EPD_OK;
}

}  // namespace

extern "C" epd_status_t ep_dispatch_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk,
                                        int num_experts, int num_ranks, int num_rdma_ranks,
                                        int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                                        int32_t *tokens_per_rdma_rank,
                                        uint8_t *is_token_in_rank, int32_t *status,
                                        epd_stream_t stream) {
    using namespace epd;
    const int T = num_tokens, k = num_topk;
    if (!topology_ok(T, k, num_experts, num_ranks, num_rdma_ranks)) return EPD_ERR_INVALID_ARG;
    if ((int64_t)T * k > 0 && (topk_idx == nullptr || !aligned8(topk_idx))) return EPD_ERR_INVALID_ARG;
    if (!tokens_per_expert || !tokens_per_rank || !status || !aligned4(tokens_per_expert) ||
        !aligned4(tokens_per_rank) || !aligned4(status) ||
        (tokens_per_rdma_rank && !aligned4(tokens_per_rdma_rank)))
        return EPD_ERR_INVALID_ARG;
    if (ws_layout(T, k, num_experts, num_ranks, num_rdma_ranks).total > EPD_NOALLOC_SCRATCH_BYTES)
        return EPD_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const epd_status_t st = noalloc_scratch_address(&scratch);
    if (st != EPD_OK) return st;
    // Nothing is cleared between calls: every call leaves the tile ticket and the
    // finished-block count at zero, and the look-back only accepts state words tagged
    // with the running call's counter, so the leftovers of an earlier call of any shape
    // (ranks, counts, older states) in the shared array are never read as published.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return layout_launch(nullptr, nullptr, 1, topk_idx, T, k, num_experts, num_ranks, num_rdma_ranks,
                         tokens_per_expert, tokens_per_rank, tokens_per_rdma_rank,
                         is_token_in_rank, scratch, status, -1, kDefaultSpinLimit, s);
}

