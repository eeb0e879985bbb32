/*
 * epd_oracle.c -- plain, slow, single-threaded CPU oracle for the single-GPU
 * MoE expert-parallel token permute / unpermute path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load this library. The product path never
 * links, imports or calls it, and it shares no code, header or table with the
 * CUDA library: every function below is written out from the definitions on the
 * pages, in plain loops, with no blocking, fusion or reordering.
 *
 * Sources (page title, section):
 *   [P1] "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题"
 *        (refactoring vLLM's EP high-throughput path after SGLang), sections
 *        2.2 / 2.2.4 (pre_permute + ep_scatter: "scan, then scatter") and
 *        3.3 (deepgemm_moe_permute: m_indices / inv_perm initialised to -1).
 *   [P2] "高性能专家并行（EP）内核解剖学解读" (anatomy of high-performance EP
 *        kernels), sections "任务设定与数据流" (8 GPUs on 2 nodes, 2 experts per
 *        GPU, top-2 of 16) and "5. 缓冲区布局与发送" (buffer layout by prefix sum).
 *   [P3] "[MoE] Deepseek的All-to-all通信: DeepEP代码解读" (reading DeepEP),
 *        section "Dispatch" (get_dispatch_layout and dispatch docstrings;
 *        "combine is similar to dispatch").
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - expert e belongs to simulated rank e / (E/R); rank r to simulated RDMA
 *     node r / (R/N) (contiguous blocks);
 *   - per-rank and per-node counts count tokens, once per rank / node;
 *   - slots inside one expert are assigned in token-major (t, then j) order;
 *   - output_index is -1 for a pair with no selection; m_indices is -1 on the
 *     rows [P, capacity) that no pair fills;
 *   - the combine is the weighted sum over the valid pairs of a token, formed
 *     here in fp64 and rounded once to bf16 (round to nearest, ties to even);
 *     a token with no valid pair gives +0.
 *
 * Build: gcc -O2 -ffp-contract=off -std=c11 -fPIC -shared (single-threaded).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum {
    ORC_OK = 0,
    ORC_ERR_INVALID_ARG = 1,
    ORC_ERR_INVALID_EXPERT = 4,
    ORC_ERR_CAPACITY = 6,
};

double oracle_double_from_bf16(uint16_t b);

/* Simulated topology: [P2] "任务设定与数据流" places 2 experts on each of 8 GPUs
 * and the 8 GPUs on 2 nodes; contiguous blocks are the plain reading. */
static int rank_of_expert(int64_t e, int E, int R) { return (int)(e / (E / R)); }
static int node_of_rank(int r, int R, int N) { return r / (R / N); }

static int check_topology(int T, int k, int E, int R, int N) {
    if (T < 0 || k < 0 || E < 1 || R < 1 || N < 1) return ORC_ERR_INVALID_ARG;
    if (E % R != 0 || R % N != 0) return ORC_ERR_INVALID_ARG;
    return ORC_OK;
}

/*
 * Dispatch layout -- [P3] "Dispatch", get_dispatch_layout docstring:
 *   num_tokens_per_expert[e] = number of (t, j) with topk_idx[t, j] == e;
 *   is_token_in_rank[t, r]   = token t is sent to rank r;
 *   num_tokens_per_rank[r]   = number of tokens sent to rank r;
 *   num_tokens_per_rdma_rank[n] = number of tokens sent to RDMA node n.
 * -1 means "no selection". Any other id outside [0, E) is rejected.
 * tokens_per_rdma_rank and is_token_in_rank may be NULL (not computed).
 */
int oracle_dispatch_layout(const int64_t *topk_idx, int T, int k, int E, int R, int N,
                           int32_t *tokens_per_expert, int32_t *tokens_per_rank,
                           int32_t *tokens_per_rdma_rank, uint8_t *is_token_in_rank) {
    int rc = check_topology(T, k, E, R, N);
    if (rc != ORC_OK) return rc;
    for (int64_t i = 0; i < (int64_t)T * k; ++i) {
        int64_t e = topk_idx[i];
        if (e < -1 || e >= E) return ORC_ERR_INVALID_EXPERT;
    }

    for (int e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int r = 0; r < R; ++r) tokens_per_rank[r] = 0;
    if (tokens_per_rdma_rank)
        for (int n = 0; n < N; ++n) tokens_per_rdma_rank[n] = 0;

    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t e = topk_idx[(int64_t)t * k + j];
            if (e >= 0) tokens_per_expert[e] += 1;
        }
        /* token t is sent to rank r if any of its selections lives on r */
        for (int r = 0; r < R; ++r) {
            int in_rank = 0;
            for (int j = 0; j < k; ++j) {
                int64_t e = topk_idx[(int64_t)t * k + j];
                if (e >= 0 && rank_of_expert(e, E, R) == r) in_rank = 1;
            }
            if (is_token_in_rank) is_token_in_rank[(int64_t)t * R + r] = (uint8_t)in_rank;
            tokens_per_rank[r] += in_rank;
        }
        /* token t is sent to node n if it is sent to any rank of n */
        if (tokens_per_rdma_rank) {
            for (int n = 0; n < N; ++n) {
                int in_node = 0;
                for (int j = 0; j < k; ++j) {
                    int64_t e = topk_idx[(int64_t)t * k + j];
                    if (e >= 0 && node_of_rank(rank_of_expert(e, E, R), R, N) == n) in_node = 1;
                }
                tokens_per_rdma_rank[n] += in_node;
            }
        }
    }
    return ORC_OK;
}

/*
 * Expert offsets -- [P2] "5. 缓冲区布局与发送": the first source starts at index
 * 0 and each next one starts where the previous one ended, i.e. the exclusive
 * prefix sum of the counts. [P1] 2.2.4: ep_scatter "scans, then scatters"
 * into expert_start_loc. *total = sum of all counts.
 */
int oracle_scan_offsets(const int32_t *tokens_per_expert, int E, int32_t *expert_start_loc,
                        int32_t *total) {
    if (E < 1) return ORC_ERR_INVALID_ARG;
    int64_t run = 0;
    for (int e = 0; e < E; ++e) {
        expert_start_loc[e] = (int32_t)run;
        run += tokens_per_expert[e];
    }
    *total = (int32_t)run;
    return ORC_OK;
}

/*
 * Aligned expert offsets -- [P1] 3.3 / 4 (deepgemm_moe_permute and
 * compute_aligned_M: every expert's rows are padded to a multiple of the
 * alignment, block_m = 256, so the grouped GEMM sees whole blocks) and [P3]
 * "Dispatch" (the dispatch docstring's expert_alignment: "align the number of
 * tokens received by each local expert"): expert e's region holds
 * round_up(count[e], alignment) rows, regions follow each other in expert
 * order; *total = sum of the padded counts. alignment = 1 is the plain scan.
 */
int oracle_scan_offsets_aligned(const int32_t *tokens_per_expert, int E, int alignment,
                                int32_t *expert_start_loc, int32_t *total) {
    if (E < 1 || alignment < 1) return ORC_ERR_INVALID_ARG;
    int64_t run = 0;
    for (int e = 0; e < E; ++e) {
        expert_start_loc[e] = (int32_t)run;
        int64_t c = tokens_per_expert[e];
        run += (c + alignment - 1) / alignment * alignment;
    }
    *total = (int32_t)run;
    return ORC_OK;
}

/*
 * Permute (ep_scatter) -- [P1] 2.2 and 3.3: each token row (and its fp8 scale
 * row) is copied, byte for byte, to one row of the expert-contiguous buffer per
 * selected expert; m_indices[row] = expert of that row, output_index[t, j] =
 * the row that pair (t, j) went to. Pairs are visited token-major, so rows
 * within one expert follow (t, j) order. Pairs with no selection get
 * output_index = -1; rows [P, capacity) get m_indices = -1 ([P1] 3.3: the
 * buffer is pre-filled with -1 so unwritten rows are skipped downstream).
 *
 * x: T rows of row_bytes bytes; x_scale: T rows of scale_cols floats, or NULL.
 * out: capacity rows of row_bytes; out_scale: capacity rows of scale_cols.
 * Rows of out / out_scale at and beyond P are left untouched.
 */
int oracle_permute(const uint8_t *x, int64_t row_bytes, const float *x_scale, int scale_cols,
                   const int64_t *topk_idx, int T, int k, int E,
                   const int32_t *expert_start_loc, int64_t capacity,
                   uint8_t *out, float *out_scale, int32_t *m_indices, int32_t *output_index) {
    if (T < 0 || k < 0 || E < 1 || row_bytes < 0 || capacity < 0) return ORC_ERR_INVALID_ARG;
    int32_t fill_count[E];
    for (int e = 0; e < E; ++e) fill_count[e] = 0;
    for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t e = topk_idx[(int64_t)t * k + j];
            if (e < -1 || e >= E) return ORC_ERR_INVALID_EXPERT;
            if (e == -1) {
                output_index[(int64_t)t * k + j] = -1;
                continue;
            }
            int64_t s = (int64_t)expert_start_loc[e] + fill_count[e];
            fill_count[e] += 1;
            if (s < 0 || s >= capacity) return ORC_ERR_CAPACITY;
            output_index[(int64_t)t * k + j] = (int32_t)s;
            m_indices[s] = (int32_t)e;
            memcpy(out + s * row_bytes, x + (int64_t)t * row_bytes, (size_t)row_bytes);
            if (x_scale != NULL && scale_cols > 0)
                memcpy(out_scale + s * scale_cols, x_scale + (int64_t)t * scale_cols,
                       (size_t)scale_cols * sizeof(float));
        }
    }
    return ORC_OK;
}

/*
 * Permute with output options -- the receiver-side view of one simulated rank
 * and the scale layouts a grouped GEMM reads:
 *   - local view ([P1] 3.1.2 and 7: after dispatch a rank holds its own experts
 *     under local ids, expert - rank_expert_offset; [P1] 3.3 deepgemm_moe_permute
 *     over local_num_experts): only pairs whose expert is in [e_begin, e_end)
 *     are placed; the buffer starts at the region of e_begin, so a pair's row
 *     is expert_start_loc[e] - expert_start_loc[e_begin] + its rank inside e;
 *     m_indices holds the local id e - e_begin; other pairs get -1;
 *   - scales ([P1] 2.2: input_tensor_scale [M, H/128], or for UE8M0 an int
 *     tensor [ceil(H/512), M] viewed transposed; [P3] low_latency_dispatch
 *     docstring: scales column-major for TMA): each token's scale row of
 *     scale_cols 32-bit words (fp32 scales or packed UE8M0 bytes) is copied to
 *     row s either row-major (out_scale[s * scale_cols + c]) or column-major
 *     (out_scale[c * scale_ld + s]).
 * Rows no pair fills keep m_indices = -1; out and out_scale rows no pair fills
 * are not written.
 */
int oracle_permute_ex(const uint8_t *x, int64_t row_bytes, const uint32_t *x_scale,
                      int scale_cols, int scale_col_major, int64_t scale_ld,
                      const int64_t *topk_idx, int T, int k, int E, int e_begin, int e_end,
                      const int32_t *expert_start_loc, int64_t capacity, uint8_t *out,
                      uint32_t *out_scale, int32_t *m_indices, int32_t *output_index) {
    if (T < 0 || k < 0 || E < 1 || row_bytes < 0 || capacity < 0) return ORC_ERR_INVALID_ARG;
    if (e_begin < 0 || e_end > E || e_begin >= e_end) return ORC_ERR_INVALID_ARG;
    if (scale_col_major && scale_ld < capacity) return ORC_ERR_INVALID_ARG;
    int32_t fill_count[E];
    for (int e = 0; e < E; ++e) fill_count[e] = 0;
    for (int64_t s = 0; s < capacity; ++s) m_indices[s] = -1;
    const int64_t base = expert_start_loc[e_begin];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t e = topk_idx[(int64_t)t * k + j];
            if (e < -1 || e >= E) return ORC_ERR_INVALID_EXPERT;
            if (e < e_begin || e >= e_end) {  /* no pick, or an expert of another view */
                output_index[(int64_t)t * k + j] = -1;
                continue;
            }
            int64_t s = (int64_t)expert_start_loc[e] - base + fill_count[e];
            fill_count[e] += 1;
            if (s < 0 || s >= capacity) return ORC_ERR_CAPACITY;
            output_index[(int64_t)t * k + j] = (int32_t)s;
            m_indices[s] = (int32_t)(e - e_begin);
            memcpy(out + s * row_bytes, x + (int64_t)t * row_bytes, (size_t)row_bytes);
            for (int c = 0; c < scale_cols; ++c) {
                uint32_t v = x_scale[(int64_t)t * scale_cols + c];
                if (scale_col_major) out_scale[(int64_t)c * scale_ld + s] = v;
                else out_scale[s * scale_cols + c] = v;
            }
        }
    }
    return ORC_OK;
}

/*
 * bf16 from a double, round to nearest, ties to even, written from the format's
 * definition (8 significant bits, fp32's exponent range, subnormal spacing
 * 2^-133): scale to the spacing of the value's binade, round the scaled value to
 * an integer with ties to even, scale back. Overflow gives infinity.
 */
uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int ex;
    (void)frexp(a, &ex);          /* a in [2^(ex-1), 2^ex) */
    int lead = ex - 1;
    if (lead < -126) lead = -126; /* below the normal range the spacing stays 2^-133 */
    double spacing = ldexp(1.0, lead - 7);
    double scaled = a / spacing;  /* exact: division by a power of two */
    double rounded = nearbyint(scaled); /* default mode: nearest, ties to even */
    double result = rounded * spacing;
    if (result >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)result;      /* exact: result has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFF));
}

/*
 * float8 e4m3 (the "fn" variant: bias 7, 3 mantissa bits, largest finite 448,
 * no infinities) from a float, round to nearest, ties to even, saturating to
 * +-448; written from the format's definition (subnormal spacing 2^-9). NaN
 * gives 0x7F.
 */
uint8_t oracle_e4m3_from_float(float v) {
    if (isnan(v)) return (uint8_t)0x7F;
    uint8_t sign = signbit(v) ? (uint8_t)0x80 : (uint8_t)0;
    double a = fabs((double)v);
    if (a == 0.0) return sign;
    int ex;
    (void)frexp(a, &ex);
    int lead = ex - 1;
    if (lead < -6) lead = -6;         /* below the normal range the spacing stays 2^-9 */
    double spacing = ldexp(1.0, lead - 3);
    double r = nearbyint(a / spacing) * spacing;
    if (r > 448.0) r = 448.0;         /* saturate */
    if (r == 0.0) return sign;
    int rex;
    (void)frexp(r, &rex);
    int e = rex - 1;                  /* r in [2^e, 2^(e+1)) */
    uint8_t bits;
    if (e < -6) {                     /* subnormal: r = m * 2^-9, m in 1..7 */
        bits = (uint8_t)(r / ldexp(1.0, -9));
    } else {
        int m = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);
        bits = (uint8_t)(((e + 7) << 3) | m);
    }
    return (uint8_t)(sign | bits);
}

/*
 * Low-latency dispatch layout with the fused cast -- [P2] "3. 解决方案：固定矩形
 * vs. 精确分配", strategy A (one fixed rectangle per expert, sized for the worst
 * case, padded slots) and [P3] "low_latency模式" (low_latency_dispatch: bf16
 * tokens cast to fp8 on the way, one fp32 scale per 128 columns with the last
 * two dimensions column-major, recv_count per expert, per-row source info; no
 * count exchange first). Experts [e_begin, e_end) each own rows_per_expert rows:
 * the r-th pick of expert e in token-major order goes to row
 * (e - e_begin) * rows_per_expert + r. A pick that finds its rectangle full is
 * dropped (output_index -1) and *overflow is set.
 *   cast, per token t and 128-column block c:
 *     amax = max |x[t, 128c .. 128c+127]|,  scale = amax / 448 (fp32), 1 if amax = 0,
 *     q[h] = e4m3(x[t, h] / scale) with the division in fp32;
 *   out_q [E_view, rows_per_expert, H] e4m3 bytes; out_scale [E_view, H/128,
 *   rows_per_expert] (column-major per expert); recv_count [E_view] = rows used;
 *   src_token [E_view, rows_per_expert] = the token of each used row.
 * Rows beyond recv_count are not written.
 */
int oracle_permute_lowlatency(const uint16_t *x, int T, int k, int H, const int64_t *topk_idx,
                              int E, int e_begin, int e_end, int64_t rows_per_expert,
                              uint8_t *out_q, float *out_scale, int32_t *recv_count,
                              int32_t *output_index, int32_t *src_token, int *overflow) {
    if (T < 0 || k < 0 || H <= 0 || H % 128 != 0 || E < 1 || rows_per_expert < 0)
        return ORC_ERR_INVALID_ARG;
    if (e_begin < 0 || e_end > E || e_begin >= e_end) return ORC_ERR_INVALID_ARG;
    const int C = H / 128;
    const int EV = e_end - e_begin;
    *overflow = 0;
    for (int e = 0; e < EV; ++e) recv_count[e] = 0;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t e = topk_idx[(int64_t)t * k + j];
            if (e < -1 || e >= E) return ORC_ERR_INVALID_EXPERT;
            output_index[(int64_t)t * k + j] = -1;
            if (e < e_begin || e >= e_end) continue;
            int64_t r = recv_count[e - e_begin];
            if (r >= rows_per_expert) {
                *overflow = 1;
                continue;
            }
            recv_count[e - e_begin] += 1;
            int64_t row = (e - e_begin) * rows_per_expert + r;
            output_index[(int64_t)t * k + j] = (int32_t)row;
            src_token[row] = t;
            for (int c = 0; c < C; ++c) {
                float amax = 0.0f;
                for (int h = 128 * c; h < 128 * (c + 1); ++h) {
                    float v = fabsf((float)oracle_double_from_bf16(x[(int64_t)t * H + h]));
                    if (v > amax) amax = v;
                }
                float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
                out_scale[((e - e_begin) * (int64_t)C + c) * rows_per_expert + r] = scale;
                for (int h = 128 * c; h < 128 * (c + 1); ++h) {
                    float v = (float)oracle_double_from_bf16(x[(int64_t)t * H + h]);
                    out_q[row * H + h] = oracle_e4m3_from_float(v / scale);
                }
            }
        }
    }
    return ORC_OK;
}

double oracle_double_from_bf16(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Unpermute (combine) -- [P3] "Dispatch": the weights travel with the tokens
 * (topk_weights, fp32) and combine is the reverse of dispatch. For every token
 * t and column h:
 *     y[t, h] = bf16( sum over j with output_index[t, j] != -1 of
 *                     topk_weights[t, j] * expert_out[output_index[t, j], h] )
 * The sum is formed in fp64 in j order and rounded once. A token with no valid
 * pair gives +0.
 */
int oracle_unpermute(const uint16_t *expert_out, int64_t capacity, const int32_t *output_index,
                     const float *topk_weights, int T, int k, int H, uint16_t *y) {
    if (T < 0 || k < 0 || H < 0 || capacity < 0) return ORC_ERR_INVALID_ARG;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t s = output_index[(int64_t)t * k + j];
            if (s < -1 || (int64_t)s >= capacity) return ORC_ERR_CAPACITY;
        }
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t s = output_index[(int64_t)t * k + j];
                if (s < 0) continue;
                acc += (double)topk_weights[(int64_t)t * k + j] *
                       oracle_double_from_bf16(expert_out[(int64_t)s * H + h]);
            }
            y[(int64_t)t * H + h] = oracle_bf16_from_double(acc);
        }
    }
    return ORC_OK;
}
