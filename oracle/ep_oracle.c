/*
 * ep_oracle.c -- plain, slow CPU oracle for the expert-parallel (EP) layout,
 * dispatch and combine path.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The product
 * path (the CUDA library) shares no code with it and never calls it.
 *
 * Every function is a nested loop over the definition, single-threaded, in
 * the order the definition states.  Integer/index outputs and byte copies
 * are exact; floating point follows the precision the method fixes:
 *   - combine accumulates in fp32, biases first, then destination ranks in
 *     ascending order, one final round-to-nearest-even to bf16;
 *   - the FP8 cast works in fp32: amax over a 128-channel group, scale =
 *     amax/448 and inverse 448/amax as two IEEE divisions, e4m3 with
 *     round-to-nearest-even and saturation to +-448;
 *   - low-latency combine is an fp32 fused multiply-add chain over top-k
 *     slots in slot order.
 * Build with -ffp-contract=off so that no other fused operation appears.
 *
 * Sources (page title, section):
 *   [P1] "DeepEP Normal vs Low-Latency 双模式深度分析" -- low-latency
 *        dispatch excerpt of internode_ll.cu (per-token FP8 cast, per-expert
 *        slot, message put), receive-side layout excerpt (slots indexed
 *        [local_expert][src_rank][max_tokens]); expert -> rank map
 *        dst_rank = expert / num_local_experts.
 *   [P2] "Normal vs Low-Latency: 双通信哲学在 DeepEP V1/V2/DeepGEMM 中的三系统比较"
 *        -- message package: a 16-byte header (source token index and three
 *        reserved ints), then the hidden payload, then the FP8 scales.
 *   [P3] "第 4 章 V1：布局、dispatch 与 combine" -- §4.1 layout (tokens per
 *        rank, per RDMA rank, per expert, is_token_in_rank) and the dispatch
 *        handle (rank / channel prefix matrices, recv_src_idx, send_head),
 *        expert_alignment; §4.2 combine with bias_0/bias_1; §4.3 the
 *        low-latency API (packed_recv_count, packed_recv_src_info,
 *        packed_recv_layout_range); §4.4 combine sums without weights and
 *        the top-k weights are reduced separately.
 *
 * Where the pages leave a step open the reading taken is stated beside the
 * code (receive order, channel convention, FP8 clamp, UE8M0 rule, LL slot
 * order).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_CAPACITY 1
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_EXPERT (-2)
#define ORACLE_INCONSISTENT (-3)
#define ORACLE_NO_MEMORY (-4)

/* ------------------------------------------------------------------------
 * Number formats
 * ---------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays NaN. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, 0x7f/0xff are NaN, largest finite 448 = 1.75 * 2^8.
 * Subnormals: exponent field 0 encodes m * 2^-9 for m = 0..7. */
float oracle_e4m3_to_f32(uint8_t c) {
    int sign = (c >> 7) & 1;
    int ef = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (ef == 0xf && m == 7) return NAN;
    if (ef == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, ef - 7);
    return (float)(sign ? -v : v);
}

/* binary32 -> e4m3, round to nearest with ties to even, saturating to the
 * largest finite magnitude (448) instead of producing NaN for large values. */
uint8_t oracle_f32_to_e4m3(float f) {
    if (isnan(f)) return 0x7f;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7e;
    /* Quantum of the binade that holds a: 2^(eb-3) for a in [2^eb, 2^(eb+1)),
     * eb >= -6; below 2^-6 the subnormal quantum 2^-9 applies. */
    int eb = 0;
    if (a > 0.0) {
        int e2;
        frexp(a, &e2); /* a = mant * 2^e2, mant in [0.5, 1) */
        eb = e2 - 1;
    }
    if (eb < -6) eb = -6;
    double quantum = ldexp(1.0, eb - 3);
    double n = nearbyint(a / quantum); /* exact quotient; default mode rounds half to even */
    double v = n * quantum;            /* a representable magnitude, <= 448 */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));
    int e2;
    frexp(v, &e2);
    int ev = e2 - 1; /* v in [2^ev, 2^(ev+1)) */
    int mant = (int)(v / ldexp(1.0, ev - 3)) - 8;
    return sign | (uint8_t)(((ev + 7) << 3) | mant);
}

/* Smallest integer e with 2^e >= s, for finite s > 0. */
static int ceil_log2(float s) {
    int e2;
    float m = frexpf(s, &e2); /* s = m * 2^e2, m in [0.5, 1) */
    return (m == 0.5f) ? e2 - 1 : e2;
}

/*
 * One 128-channel group -> e4m3 codes and its scale ([P1] low-latency
 * dispatch excerpt: per-128 amax, scale and inverse scale; [P3] §4.4: FP8
 * input with one fp32 scale per 128 channels).
 *
 *   amax  = max(max_i |x_i|, 1e-4)        (the clamp guards the division)
 *   s     = amax / 448                    (IEEE division, fp32)
 *   round_scale == 0:  scale = s,   q_i = e4m3(x_i * (448 / amax))
 *   round_scale != 0:  e = smallest integer with 2^e >= s,
 *                      scale = 2^e, q_i = e4m3(x_i * 2^-e)
 * *exp_out receives e (only meaningful when round_scale != 0).
 */
void oracle_fp8_quantize_group(const uint16_t* x, int n, int round_scale,
                               uint8_t* q, float* scale_out, int* exp_out) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(oracle_bf16_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    if (amax < 1e-4f) amax = 1e-4f;
    float s = amax / 448.0f;
    if (!round_scale) {
        float inv = 448.0f / amax;
        for (int i = 0; i < n; ++i) q[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(x[i]) * inv);
        *scale_out = s;
        if (exp_out) *exp_out = 0;
    } else {
        int e = ceil_log2(s);
        float inv = ldexpf(1.0f, -e);
        for (int i = 0; i < n; ++i) q[i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(x[i]) * inv);
        *scale_out = ldexpf(1.0f, e);
        if (exp_out) *exp_out = e;
    }
}

/* ------------------------------------------------------------------------
 * Layout ([P3] §4.1: get_dispatch_layout(topk_idx, num_experts))
 *
 * topk_idx [R][T][K] int64, -1 = masked slot.  Expert e lives on rank
 * e / (E/R) ([P1] dst_rank = expert / num_local_experts).
 *   num_tokens_per_expert[s][e] = #(t,k) with topk_idx[s][t][k] == e
 *   is_token_in_rank[s][t][r]   = 1 iff some slot of (s,t) maps to rank r
 *   num_tokens_per_rank[s][r]   = #t with is_token_in_rank[s][t][r]
 *   num_tokens_per_rdma_rank[s][n] = #t with a hit in node n (8 ranks per
 *     node), computed only when the pointer is non-NULL.
 *
 * Rank masking ([P1] low-latency receive excerpt: mask_buffer and
 * is_rank_masked; the pages show it in the low-latency path only): when
 * rank_mask is non-NULL, a slot whose source rank s or whose destination
 * rank e / EL has rank_mask != 0 counts as a masked slot (-1).  Reading, the
 * same as the low-latency dispatch's: a masked rank neither sends nor
 * receives, so the layout -- and the record, dispatch and combine that
 * follow from it -- leaves it out.  An expert id out of range is an error
 * whatever the mask.
 * ---------------------------------------------------------------------- */
int oracle_get_dispatch_layout(int R, int T, int K, int E, const int64_t* topk_idx, const int32_t* rank_mask,
                               int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                               int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank) {
    if (R <= 0 || T < 0 || K <= 0 || E <= 0 || E % R != 0) return ORACLE_BAD_ARG;
    const int EL = E / R;
    const int NN = (R + 7) / 8;
    memset(num_tokens_per_rank, 0, sizeof(int32_t) * (size_t)R * R);
    memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)R * E);
    memset(is_token_in_rank, 0, (size_t)R * T * R);
    if (num_tokens_per_rdma_rank) memset(num_tokens_per_rdma_rank, 0, sizeof(int32_t) * (size_t)R * NN);
    for (int s = 0; s < R; ++s) {
        for (int t = 0; t < T; ++t) {
            uint8_t* hit = is_token_in_rank + ((size_t)s * T + t) * R;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[((size_t)s * T + t) * K + k];
                if (e == -1) continue;
                if (e < 0 || e >= E) return ORACLE_BAD_EXPERT;
                if (rank_mask && (rank_mask[s] != 0 || rank_mask[e / EL] != 0)) continue;
                num_tokens_per_expert[(size_t)s * E + e] += 1;
                hit[e / EL] = 1;
            }
            for (int r = 0; r < R; ++r)
                if (hit[r]) num_tokens_per_rank[(size_t)s * R + r] += 1;
            if (num_tokens_per_rdma_rank) {
                for (int n = 0; n < NN; ++n) {
                    int any = 0;
                    for (int r = 8 * n; r < 8 * n + 8 && r < R; ++r) any |= hit[r];
                    if (any) num_tokens_per_rdma_rank[(size_t)s * NN + n] += 1;
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Dispatch bookkeeping: prefix matrices and receive rows ([P3] §4.1 the
 * handle (rank_prefix_matrix, channel_prefix_matrix,
 * recv_channel_prefix_matrix, recv_src_idx, is_token_in_rank, send_head)
 * and num_recv_tokens_per_expert_list with expert_alignment).
 *
 * Readings:
 *  - receive order inside destination rank r: source rank ascending, then
 *    token index ascending (channels are contiguous token ranges, so the
 *    channel order gives the same sequence);
 *  - C channels, channel c owns tokens [c*chunk, min(T,(c+1)*chunk)) with
 *    chunk = ceil(T/C);
 *    channel_prefix[s][r][c]      = #hits of (s -> r) among t < end(c)
 *                                    (inclusive prefix over channels);
 *    recv_channel_prefix[r][s][c] = first receive row of channel c of
 *                                    source s inside r
 *                                  = rank_prefix[s-1][r] + #hits among t < start(c);
 *  - rank_prefix[s][r] = sum over s' <= s of num_tokens_per_rank[s'][r];
 *  - send_head[s][t][r] = the absolute receive row of (s,t) in rank r, or
 *    -1 when (s,t) is not sent to r (one GPU has no ring buffer to index);
 *  - recv_src_idx[r][row] = t for every row below the capacity;
 *  - num_recv_tokens_per_expert[r][j] = sum_s num_tokens_per_expert[s][r*EL+j]
 *    rounded up to a multiple of expert_alignment.
 * Returns ORACLE_CAPACITY when a rank receives more than cap rows (rows at
 * or past cap are not recorded in recv_src_idx), ORACLE_INCONSISTENT when
 * num_tokens_per_rank does not match is_token_in_rank.
 * ---------------------------------------------------------------------- */
int oracle_dispatch_notify(int R, int T, int E, int C, int A, int64_t cap,
                           const int32_t* num_tokens_per_rank, const uint8_t* is_token_in_rank,
                           const int32_t* num_tokens_per_expert,
                           int32_t* rank_prefix_matrix, int32_t* channel_prefix_matrix,
                           int32_t* recv_channel_prefix_matrix, int32_t* num_recv,
                           int32_t* send_head, int32_t* recv_src_idx,
                           int32_t* num_recv_tokens_per_expert) {
    if (R <= 0 || T < 0 || E <= 0 || E % R != 0 || C <= 0 || A <= 0 || cap < 0) return ORACLE_BAD_ARG;
    const int EL = E / R;
    int status = ORACLE_OK;

    for (int r = 0; r < R; ++r) {
        int32_t acc = 0;
        for (int s = 0; s < R; ++s) {
            acc += num_tokens_per_rank[(size_t)s * R + r];
            rank_prefix_matrix[(size_t)s * R + r] = acc;
        }
        num_recv[r] = acc;
    }

    const int chunk = (T + C - 1) / C;
    for (int s = 0; s < R; ++s) {
        for (int r = 0; r < R; ++r) {
            int32_t before_rank = s > 0 ? rank_prefix_matrix[(size_t)(s - 1) * R + r] : 0;
            for (int c = 0; c < C; ++c) {
                int start = c * chunk < T ? c * chunk : T;
                int end = (c + 1) * chunk < T ? (c + 1) * chunk : T;
                int32_t n_end = 0, n_start = 0;
                for (int t = 0; t < end; ++t) {
                    int h = is_token_in_rank[((size_t)s * T + t) * R + r] != 0;
                    n_end += h;
                    if (t < start) n_start += h;
                }
                channel_prefix_matrix[((size_t)s * R + r) * C + c] = n_end;
                recv_channel_prefix_matrix[((size_t)r * R + s) * C + c] = before_rank + n_start;
            }
        }
    }

    for (int r = 0; r < R; ++r) {
        int64_t row = 0;
        for (int s = 0; s < R; ++s) {
            int32_t sent = 0;
            for (int t = 0; t < T; ++t) {
                size_t g = (size_t)s * T + t;
                if (is_token_in_rank[g * R + r]) {
                    send_head[g * R + r] = (int32_t)row;
                    if (row < cap) recv_src_idx[(size_t)r * cap + row] = t;
                    ++row;
                    ++sent;
                } else {
                    send_head[g * R + r] = -1;
                }
            }
            if (sent != num_tokens_per_rank[(size_t)s * R + r]) status = ORACLE_INCONSISTENT;
        }
        if (row > cap && status == ORACLE_OK) status = ORACLE_CAPACITY;
    }

    for (int r = 0; r < R; ++r) {
        for (int j = 0; j < EL; ++j) {
            int64_t sum = 0;
            for (int s = 0; s < R; ++s) sum += num_tokens_per_expert[(size_t)s * E + (size_t)r * EL + j];
            num_recv_tokens_per_expert[(size_t)r * EL + j] = (int32_t)(((sum + A - 1) / A) * A);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * Node-level (RDMA rank) record of a two-level dispatch ([P3] §4.2: the
 * internode handle adds RDMA channel prefix matrices and RDMA rank prefix
 * sums; [P1]: 8 NVLink peers per node, the GPUs of a node share one RDMA
 * rank in normal mode, and the RDMA team is the ranks with the same GPU
 * index).  Whole nodes only: R > 8 and R % 8 == 0; rank r = 8 n + l is
 * GPU l of node n, NN = R / 8.
 *
 * A token "goes to node n" when it is sent to at least one rank of node n:
 * source (m, l) moves it once over RDMA, to rank (n, l), which forwards it
 * over NVLink.  With the channels of oracle_dispatch_notify:
 *   rdma_channel_prefix[s][n][c] = #t < end(c) of source s that go to node n
 *                                  (inclusive prefix over channels)
 *   recv_rdma_rank_prefix[r][m]  = for r = (n, l): #t of the sources (m', l),
 *                                  m' <= m, that go to node n (inclusive
 *                                  prefix over source nodes)
 * The rank-level matrices are those of oracle_dispatch_notify.
 * ---------------------------------------------------------------------- */
int oracle_rdma_prefix(int R, int T, int C, const uint8_t* is_token_in_rank,
                       int32_t* rdma_channel_prefix, int32_t* recv_rdma_rank_prefix) {
    if (R <= 8 || R % 8 != 0 || T < 0 || C <= 0) return ORACLE_BAD_ARG;
    const int NN = R / 8;
    const int chunk = (T + C - 1) / C;
    for (int s = 0; s < R; ++s)
        for (int n = 0; n < NN; ++n)
            for (int c = 0; c < C; ++c) {
                int end = (c + 1) * chunk < T ? (c + 1) * chunk : T;
                int32_t count = 0;
                for (int t = 0; t < end; ++t) {
                    int goes = 0;
                    for (int r = 8 * n; r < 8 * n + 8; ++r)
                        goes |= is_token_in_rank[((size_t)s * T + t) * R + r] != 0;
                    count += goes;
                }
                rdma_channel_prefix[((size_t)s * NN + n) * C + c] = count;
            }
    for (int r = 0; r < R; ++r) {
        const int n = r / 8, l = r % 8;
        int32_t acc = 0;
        for (int m = 0; m < NN; ++m) {
            acc += rdma_channel_prefix[((size_t)(8 * m + l) * NN + n) * C + (C - 1)];
            recv_rdma_rank_prefix[(size_t)r * NN + m] = acc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Normal dispatch ([P3] §4.1 intranode_dispatch; §4.4 FP8 input).
 * For every token (s,t) in the list (all tokens when tokens == NULL) and
 * every rank r with row = send_head[s][t][r] in [0, cap):
 *   mode 0 (bf16):      recv_x[r][row][:] = x[s][t][:]               (bytes)
 *   mode 1 (bf16->FP8): recv_x[r][row][:] = e4m3 codes of x[s][t],
 *                       recv_x_scales[r][row][g] = scale of group g
 *   mode 2 (FP8 in):    e4m3 bytes and the input's scales are copied
 *   recv_topk_idx[r][row][k]     = topk_idx[s][t][k] mod EL when that
 *                                  expert lives on r, else -1
 *   recv_topk_weights[r][row][k] = topk_weights[s][t][k] under the same
 *                                  condition, else 0
 * ---------------------------------------------------------------------- */
int oracle_dispatch(int R, int T, int H, int K, int E, int64_t cap, int mode,
                    const void* x, const float* x_scales,
                    const int64_t* topk_idx, const float* topk_weights,
                    const int32_t* send_head, const int64_t* tokens, int64_t n_tokens,
                    void* recv_x, float* recv_x_scales,
                    int64_t* recv_topk_idx, float* recv_topk_weights) {
    if (R <= 0 || T < 0 || H <= 0 || K <= 0 || E <= 0 || E % R != 0 || cap < 0) return ORACLE_BAD_ARG;
    if (mode < 0 || mode > 2) return ORACLE_BAD_ARG;
    if (mode != 0 && (H % 128 != 0 || recv_x_scales == NULL)) return ORACLE_BAD_ARG;
    if (mode == 2 && x_scales == NULL) return ORACLE_BAD_ARG;
    const int EL = E / R;
    const int G = H / 128;
    const int64_t total = (int64_t)R * T;
    const int64_t count = tokens ? n_tokens : total;
    uint8_t* qrow = NULL;
    float* srow = NULL;
    if (mode == 1) {
        qrow = (uint8_t*)malloc((size_t)H);
        srow = (float*)malloc(sizeof(float) * (size_t)G);
        if (!qrow || !srow) { free(qrow); free(srow); return ORACLE_NO_MEMORY; }
    }
    for (int64_t i = 0; i < count; ++i) {
        int64_t g = tokens ? tokens[i] : i;
        if (g < 0 || g >= total) continue;
        if (mode == 1) {
            const uint16_t* xr = (const uint16_t*)x + (size_t)g * H;
            for (int grp = 0; grp < G; ++grp)
                oracle_fp8_quantize_group(xr + grp * 128, 128, 0, qrow + grp * 128, srow + grp, NULL);
        }
        for (int r = 0; r < R; ++r) {
            int64_t row = send_head[(size_t)g * R + r];
            if (row < 0 || row >= cap) continue;
            size_t dst = (size_t)r * cap + row;
            if (mode == 0) {
                memcpy((uint16_t*)recv_x + dst * H, (const uint16_t*)x + (size_t)g * H, sizeof(uint16_t) * H);
            } else if (mode == 1) {
                memcpy((uint8_t*)recv_x + dst * H, qrow, (size_t)H);
                memcpy(recv_x_scales + dst * G, srow, sizeof(float) * G);
            } else {
                memcpy((uint8_t*)recv_x + dst * H, (const uint8_t*)x + (size_t)g * H, (size_t)H);
                memcpy(recv_x_scales + dst * G, x_scales + (size_t)g * G, sizeof(float) * G);
            }
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx ? topk_idx[(size_t)g * K + k] : -1;
                int mine = e >= 0 && e / EL == r;
                if (recv_topk_idx) recv_topk_idx[dst * K + k] = mine ? e % EL : -1;
                if (recv_topk_weights && topk_weights)
                    recv_topk_weights[dst * K + k] = mine ? topk_weights[(size_t)g * K + k] : 0.0f;
            }
        }
    }
    free(qrow);
    free(srow);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Normal combine ([P3] §4.2 combine(x, handle, topk_weights, bias); §4.4
 * the combine adds without weights, top-k weights are reduced separately).
 * For every token (s,t) in the list and every channel h:
 *   acc = float(bias0) + float(bias1)          (a missing bias counts +0)
 *   for r = 0..R-1 with row = send_head[s][t][r] in [0, cap):
 *       acc = acc + float(y[r][row][h])         (fp32)
 *   out[s][t][h] = bf16_rne(acc), or acc when out_fp32
 *   combined_topk_weights[s][t][k] = 0, then += recv_topk_weights[r][row][k]
 *                                    over the same ranks in the same order
 * ---------------------------------------------------------------------- */
int oracle_combine(int R, int T, int H, int K, int64_t cap, const int32_t* send_head,
                   const uint16_t* y, const float* recv_topk_weights,
                   const uint16_t* bias0, const uint16_t* bias1, int out_fp32,
                   const int64_t* tokens, int64_t n_tokens,
                   void* out, float* combined_topk_weights) {
    if (R <= 0 || T < 0 || H <= 0 || K <= 0 || cap < 0) return ORACLE_BAD_ARG;
    const int64_t total = (int64_t)R * T;
    const int64_t count = tokens ? n_tokens : total;
    for (int64_t i = 0; i < count; ++i) {
        int64_t g = tokens ? tokens[i] : i;
        if (g < 0 || g >= total) continue;
        for (int h = 0; h < H; ++h) {
            float b0 = bias0 ? oracle_bf16_to_f32(bias0[(size_t)g * H + h]) : 0.0f;
            float b1 = bias1 ? oracle_bf16_to_f32(bias1[(size_t)g * H + h]) : 0.0f;
            float acc = b0 + b1;
            for (int r = 0; r < R; ++r) {
                int64_t row = send_head[(size_t)g * R + r];
                if (row < 0 || row >= cap) continue;
                acc = acc + oracle_bf16_to_f32(y[((size_t)r * cap + row) * H + h]);
            }
            if (out_fp32) ((float*)out)[(size_t)g * H + h] = acc;
            else ((uint16_t*)out)[(size_t)g * H + h] = oracle_f32_to_bf16(acc);
        }
        if (combined_topk_weights && recv_topk_weights) {
            for (int k = 0; k < K; ++k) {
                float w = 0.0f;
                for (int r = 0; r < R; ++r) {
                    int64_t row = send_head[(size_t)g * R + r];
                    if (row < 0 || row >= cap) continue;
                    w = w + recv_topk_weights[((size_t)r * cap + row) * K + k];
                }
                combined_topk_weights[(size_t)g * K + k] = w;
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Low-latency dispatch ([P1] low-latency dispatch and receive-layout
 * excerpts; [P2] message package; [P3] §4.3).
 *
 * One message per valid slot (s,t,k), e = topk_idx[s][t][k], destination
 * rank d = e / EL, local expert j = e mod EL:
 *   bytes [0,16)          int32 t, then three int32 zeros
 *   bytes [16,16+P)       payload: bf16 row (P = 2H) or e4m3 codes (P = H)
 *   bytes [16+P, msg)     FP8 only, 4*H/128 bytes: fp32 scales, or with
 *                         use_ue8m0 the bytes e_g + 127 at offset g and
 *                         zeros after the first H/128 bytes
 * use_ue8m0 implies round_scale (power-of-two scales).
 *
 * Reading (slot order): the rows of local expert j on rank d form one
 * packed array of R*maxT slots; source ranks occupy consecutive blocks in
 * ascending order, and inside a block the slots follow (token, k) order:
 *   cnt[s][e]   = #valid slots of source s routed to e
 *   begin[e][s] = sum over s' < s of cnt[s'][e]
 *   row(s,t,k)  = begin[e][s] + #slots (t',k') < (t,k) of source s with e
 *   packed_recv_count[d][j]     = sum_s cnt[s][e]
 *   packed_recv_layout_range[d][j][s] = (cnt[s][e] << 32) | begin[e][s]
 * The messages are written to msgs_by_slot[s][t][k][:] (indexed by slot;
 * the receive buffer holds the same bytes at [d][j][row]); slot_row gets
 * the row, -1 for masked slots and for rows past the R*maxT capacity.
 *
 * Rank masking ([P1] low-latency receive excerpt: a rank that timed out is
 * marked in mask_buffer, and is_rank_masked skips sends to it): when
 * rank_mask is non-NULL, a slot whose destination rank d or whose source
 * rank s has rank_mask != 0 is treated as a masked slot (-1): no message, not
 * counted, slot_row -1.  Reading: a masked rank neither receives nor sends.
 * ---------------------------------------------------------------------- */
int64_t oracle_ll_msg_bytes(int H, int use_fp8) {
    return use_fp8 ? 16 + (int64_t)H + 4 * (int64_t)(H / 128) : 16 + 2 * (int64_t)H;
}

/* The expert of slot i of source s, or -1 when the slot is masked or either rank is masked. */
static int64_t ll_slot_expert(const int64_t* topk_idx, size_t i, int s, int EL, const int32_t* rank_mask) {
    int64_t e = topk_idx[i];
    if (e < 0) return -1;
    if (rank_mask && (rank_mask[s] != 0 || rank_mask[e / EL] != 0)) return -1;
    return e;
}

int oracle_ll_dispatch(int R, int T, int maxT, int H, int K, int E, const uint16_t* x,
                       const int64_t* topk_idx, const int32_t* rank_mask, int use_fp8, int round_scale,
                       int use_ue8m0, uint8_t* msgs_by_slot, int32_t* slot_row,
                       int32_t* packed_recv_count, int64_t* packed_recv_layout_range) {
    if (R <= 0 || T < 0 || T > maxT || H <= 0 || K <= 0 || E <= 0 || E % R != 0) return ORACLE_BAD_ARG;
    if (use_fp8 && H % 128 != 0) return ORACLE_BAD_ARG;
    if (use_ue8m0) round_scale = 1;
    const int EL = E / R;
    const int G = H / 128;
    const int64_t msg = oracle_ll_msg_bytes(H, use_fp8);
    const int64_t slots_per_expert = (int64_t)R * maxT;
    int status = ORACLE_OK;

    int64_t* cnt = (int64_t*)calloc((size_t)R * E, sizeof(int64_t));
    int64_t* begin = (int64_t*)calloc((size_t)R * E, sizeof(int64_t));
    int64_t* running = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    uint8_t* q = (uint8_t*)malloc((size_t)H);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
    int* ex = (int*)malloc(sizeof(int) * (size_t)(G > 0 ? G : 1));
    if (!cnt || !begin || !running || !q || !sc || !ex) {
        free(cnt); free(begin); free(running); free(q); free(sc); free(ex);
        return ORACLE_NO_MEMORY;
    }

    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[((size_t)s * T + t) * K + k];
                if (e == -1) continue;
                if (e < 0 || e >= E) { status = ORACLE_BAD_EXPERT; goto done; }
                e = ll_slot_expert(topk_idx, ((size_t)s * T + t) * K + k, s, EL, rank_mask);
                if (e < 0) continue;
                cnt[(size_t)s * E + e] += 1;
            }
    for (int e = 0; e < E; ++e) {
        int64_t acc = 0;
        for (int s = 0; s < R; ++s) {
            begin[(size_t)e * R + s] = acc;
            acc += cnt[(size_t)s * E + e];
        }
        int d = e / EL, j = e % EL;
        packed_recv_count[(size_t)d * EL + j] = (int32_t)(acc < slots_per_expert ? acc : slots_per_expert);
        if (acc > slots_per_expert) status = ORACLE_CAPACITY;
        for (int s = 0; s < R; ++s)
            packed_recv_layout_range[((size_t)d * EL + j) * R + s] =
                (int64_t)(((uint64_t)cnt[(size_t)s * E + e] << 32) | (uint64_t)(uint32_t)begin[(size_t)e * R + s]);
    }

    for (int s = 0; s < R; ++s) {
        memset(running, 0, sizeof(int64_t) * (size_t)E);
        for (int t = 0; t < T; ++t) {
            const uint16_t* xr = x + ((size_t)s * T + t) * H;
            if (use_fp8)
                for (int grp = 0; grp < G; ++grp)
                    oracle_fp8_quantize_group(xr + grp * 128, 128, round_scale, q + grp * 128, sc + grp, ex + grp);
            for (int k = 0; k < K; ++k) {
                size_t slot = ((size_t)s * T + t) * K + k;
                uint8_t* m = msgs_by_slot + slot * msg;
                memset(m, 0, (size_t)msg);
                int64_t e = ll_slot_expert(topk_idx, slot, s, EL, rank_mask);
                if (e < 0) { slot_row[slot] = -1; continue; }
                int64_t row = begin[(size_t)e * R + s] + running[e];
                running[e] += 1;
                if (row >= slots_per_expert) { slot_row[slot] = -1; continue; }
                slot_row[slot] = (int32_t)row;
                int32_t header[4] = {t, 0, 0, 0};
                memcpy(m, header, sizeof header);
                if (!use_fp8) {
                    memcpy(m + 16, xr, sizeof(uint16_t) * H);
                } else {
                    memcpy(m + 16, q, (size_t)H);
                    uint8_t* tail = m + 16 + H;
                    if (use_ue8m0) {
                        for (int grp = 0; grp < G; ++grp) tail[grp] = (uint8_t)(ex[grp] + 127);
                    } else {
                        memcpy(tail, sc, sizeof(float) * G);
                    }
                }
            }
        }
    }
done:
    free(cnt); free(begin); free(running); free(q); free(sc); free(ex);
    return status;
}

/* ------------------------------------------------------------------------
 * Low-latency combine ([P1] combine excerpt names; [P3] §4.3
 * low_latency_combine(x, topk_idx, topk_weights, handle)).  The expert
 * outputs y sit in the packed receive layout [R][EL][R*maxT][H] (bf16).
 * For every token (s,t) in the list and channel h:
 *   acc = 0; for k = 0..K-1 with a valid slot (row = slot_row[s][t][k] >= 0):
 *       acc = fma(topk_weights[s][t][k], float(y[d][j][row][h]), acc)
 *   out[s][t][h] = bf16_rne(acc)
 * ---------------------------------------------------------------------- */
int oracle_ll_combine(int R, int T, int maxT, int H, int K, int E, const uint16_t* y,
                      const int64_t* topk_idx, const float* topk_weights, const int32_t* slot_row,
                      const int64_t* tokens, int64_t n_tokens, uint16_t* out) {
    if (R <= 0 || T < 0 || T > maxT || H <= 0 || K <= 0 || E <= 0 || E % R != 0) return ORACLE_BAD_ARG;
    const int EL = E / R;
    const int64_t total = (int64_t)R * T;
    const int64_t count = tokens ? n_tokens : total;
    for (int64_t i = 0; i < count; ++i) {
        int64_t g = tokens ? tokens[i] : i;
        if (g < 0 || g >= total) continue;
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[(size_t)g * K + k];
                int32_t row = slot_row[(size_t)g * K + k];
                if (e < 0 || row < 0) continue;
                size_t d = (size_t)(e / EL), j = (size_t)(e % EL);
                float v = oracle_bf16_to_f32(y[((d * EL + j) * (size_t)R * maxT + row) * H + h]);
                acc = fmaf(topk_weights[(size_t)g * K + k], v, acc);
            }
            out[(size_t)g * H + h] = oracle_f32_to_bf16(acc);
        }
    }
    return ORACLE_OK;
}
