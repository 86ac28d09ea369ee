/*
 * ep.h -- C ABI of the single-GPU expert-parallel (EP) layout / dispatch /
 * combine engine for GB300 (sm_103a).
 *
 * The R "ranks" of an expert-parallel group are virtual partitions of one
 * GPU's memory: every tensor carries the rank as its leading axis, and a
 * "send" to rank r is a store into r's slice.  The operations are those of
 * the DeepEP Buffer API described on the pages
 *   [P1] "DeepEP Normal vs Low-Latency 双模式深度分析"
 *   [P2] "Normal vs Low-Latency: 双通信哲学在 DeepEP V1/V2/DeepGEMM 中的三系统比较"
 *   [P3] "第 4 章 V1：布局、dispatch 与 combine"
 * restated for one GPU with all R ranks batched into one call.
 *
 * Conventions (every entry point):
 *  - Tensor pointers are DEVICE pointers on the handle's device, allocated and
 *    owned by the caller, C-contiguous row-major, with the shapes given
 *    below.  Payload tensors (x, recv_x, combine inputs/outputs, low-latency
 *    message buffers) must be 16-byte aligned; the others need their natural
 *    alignment.  The handle is the only library-owned object.
 *  - Notation: R ranks, T tokens per rank in this call, H hidden size,
 *    E experts, K top-k, EL = E/R local experts per rank, C channels,
 *    cap = recv_capacity, maxT = num_max_tokens, G = H/128 scale groups.
 *    Expert e lives on rank e / EL as local expert e % EL ([P1]:
 *    dst_rank = expert / num_local_experts).  topk_idx entries are expert
 *    ids in [0, E) or -1 for a masked slot.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns after enqueueing its kernels.
 *    Calls on one handle must not overlap on the GPU -- issue them on one
 *    stream, or order them with events: the handle holds the dispatch record,
 *    the status word and the counters its kernels share.
 *  - Argument errors found on the host are returned at once and nothing is
 *    enqueued.  Errors found by the kernels (an expert id out of range,
 *    counts that disagree with is_token_in_rank, a receive buffer that is
 *    too small, an expired wait) are recorded in the handle's device status
 *    word -- the first one wins -- and are read with ep_handle_status().
 *    Kernels never trap; a capacity error skips the rows that do not fit
 *    and writes nothing out of bounds.
 *  - Nothing here allocates memory except ep_handle_create().
 */
#ifndef EP_GB300_EP_H
#define EP_GB300_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ep_stream_t; /* same type as cudaStream_t */

typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,   /* host: bad pointer, size, alignment, dtype or mode combination  */
    EP_ERR_CAPACITY = 2,      /* device: a receive buffer has fewer rows than the layout needs   */
    EP_ERR_TIMEOUT = 3,       /* device: a bounded wait expired                                  */
    EP_ERR_CUDA = 4,          /* a CUDA runtime call failed (message in ep_last_error())         */
    EP_ERR_UNSUPPORTED = 5,   /* host: sizes outside what the kernels were built for             */
    EP_ERR_INCONSISTENT = 6,  /* device: num_tokens_per_rank disagrees with is_token_in_rank      */
    EP_ERR_BAD_EXPERT = 7,    /* device: an expert id outside [-1, E)                            */
    EP_ERR_STATE = 8          /* host: a cached / combine call without the dispatch it relies on */
} ep_status;

typedef enum ep_dtype {
    EP_BF16 = 0,     /* bfloat16, 2 bytes                                   */
    EP_FP8_E4M3 = 1, /* OCP e4m3 ("e4m3fn"), 1 byte, largest finite 448      */
    EP_FP32 = 2      /* IEEE binary32                                       */
} ep_dtype;

/* Sizes fixed for the lifetime of a handle (the Buffer of [P1]/[P3]). */
typedef struct ep_config {
    int32_t num_ranks;        /* R: 1..32                                                       */
    int32_t num_max_tokens;   /* maxT: most tokens per rank in one call; for low-latency mode
                                 this is num_max_dispatch_tokens_per_rank ([P3] §4.3)            */
    int32_t hidden;           /* H: multiple of 8; a multiple of 128 for FP8 payloads and of
                                 512 for FP8 low-latency messages (16-byte message size)         */
    int32_t num_experts;      /* E: multiple of R, at most 2048                                 */
    int32_t num_topk;         /* K: 1..32                                                       */
    int32_t num_channels;     /* C >= 1: channels of the prefix matrices; the pages' tests run
                                 24 SMs, i.e. 12 channels ([P1] num_channels = num_sms / 2)     */
    int32_t expert_alignment; /* A >= 1: per-expert receive counts are rounded up to A ([P3] §4.1) */
    int32_t max_sms;          /* 0: the data kernels may fill the GPU; n > 0: they keep at most n
                                 SMs' worth of CTAs resident at once and leave the rest of the
                                 GPU to concurrent work ([P1] get_theoretical_num_sms and
                                 prefer_overlap_with_compute; ep_theoretical_num_sms suggests n) */
    int64_t recv_capacity;    /* cap: rows per destination rank in normal-mode receive buffers
                                 (the num_worst_tokens bound of [P3] §4.1); 0 disables normal mode */
} ep_config;

typedef struct ep_handle ep_handle;

/* Which handle array ep_handle_export() copies. */
typedef enum ep_handle_field {
    EP_FIELD_RANK_PREFIX_MATRIX = 0,         /* int32 [R][R]                                  */
    EP_FIELD_CHANNEL_PREFIX_MATRIX = 1,      /* int32 [R][R][C]                               */
    EP_FIELD_RECV_CHANNEL_PREFIX_MATRIX = 2, /* int32 [R][R][C]                               */
    EP_FIELD_RECV_SRC_IDX = 3,               /* int32 [R][cap]                                */
    EP_FIELD_SEND_HEAD = 4,                  /* int32 [R][maxT][R] (first T*R*... rows valid) */
    EP_FIELD_NUM_RECV = 5,                   /* int32 [R]                                     */
    EP_FIELD_LL_SLOT_ROW = 6,                /* int32 [R][maxT][K]                            */
    /* The node-level record of the two-level layout ("第 4 章 V1：布局、dispatch 与
     * combine" §4.2, the internode handle), kept when the ranks form two or more
     * whole nodes of 8 (R > 8, R % 8 == 0): rank r = 8n + l is GPU l of node n,
     * NN = R / 8.  The GPUs of a node share one RDMA rank and the RDMA team is
     * the ranks with the same GPU index ("DeepEP Normal vs Low-Latency 双模式深度
     * 分析"), so rank (n, l) receives over RDMA the tokens of the sources (m, l)
     * that reach node n.  Exporting either otherwise is EP_ERR_UNSUPPORTED. */
    EP_FIELD_RDMA_CHANNEL_PREFIX_MATRIX = 7, /* int32 [R][NN][C]: [s][n][c] = tokens t < end of
                                                channel c of source s that reach any rank of node n */
    EP_FIELD_RECV_RDMA_RANK_PREFIX_SUM = 8   /* int32 [R][NN]: [r][m], r = (n, l) = tokens of the
                                                sources (m', l), m' <= m, that reach node n      */
} ep_handle_field;

/* ------------------------------------------------------------------ handle */

/* Create a handle on the current CUDA device: validates `cfg` and allocates
 * (cudaMalloc, once) the device arrays of the dispatch record -- the prefix
 * matrices, recv_src_idx, send_head, the low-latency slot map -- and the
 * status word.  On success *out owns them; release with ep_handle_destroy(). */
ep_status ep_handle_create(const ep_config* cfg, ep_handle** out);

/* Free the handle's device memory (synchronises the device first).  NULL is a no-op. */
void ep_handle_destroy(ep_handle* h);

/* Synchronise `stream`, then return the first device-detected error recorded
 * since the last reset (EP_OK if none).  reset != 0 clears the word. */
ep_status ep_handle_status(ep_handle* h, ep_stream_t stream, int32_t reset);

/* Synchronise `stream` and copy the per-rank receive counts of the last
 * normal dispatch (num_recv[r] = rank_prefix_matrix[R-1][r]) to host memory
 * host_num_recv[R]. */
ep_status ep_handle_num_recv(ep_handle* h, int32_t* host_num_recv, ep_stream_t stream);

/* Byte size of one handle array, and an asynchronous copy of it to `dst`
 * (device or host memory, `bytes` >= that size). */
size_t ep_handle_field_bytes(const ep_handle* h, ep_handle_field field);
ep_status ep_handle_export(const ep_handle* h, ep_handle_field field, void* dst, size_t bytes,
                           ep_stream_t stream);

/* Static text for a status code; thread-local detail of the last failing call. */
const char* ep_status_string(ep_status s);
const char* ep_last_error(void);

/* ------------------------------------------------------------------ layout */

/* get_dispatch_layout ([P3] §4.1): from topk_idx [R][T][K] (int64) compute
 *   num_tokens_per_rank[s][r]      int32 [R][R]    tokens of rank s with an expert on rank r
 *   num_tokens_per_rdma_rank[s][n] int32 [R][ceil(R/8)] tokens of s with an expert in node n
 *                                  (8 ranks per node, [P1] NVL peers); may be NULL
 *   num_tokens_per_expert[s][e]    int32 [R][E]    top-k slots of s that chose e
 *   is_token_in_rank[s][t][r]      uint8 [R][T][R] 1 iff token (s,t) has an expert on r
 * Every output element is written.  An id outside [-1, E) sets EP_ERR_BAD_EXPERT.
 * With ranks masked in the handle's mask buffer (ep_update_mask_buffer), a
 * slot whose source rank s or whose destination rank e / EL is masked counts
 * as a masked slot (-1): a masked rank neither sends nor receives.  The
 * record, dispatch and combine built from this layout then leave it out. */
ep_status ep_get_dispatch_layout(ep_handle* h, int32_t num_tokens, const int64_t* topk_idx,
                                 int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                                 int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                                 ep_stream_t stream);

/* -------------------------------------------------------- normal dispatch */

/* How ep_dispatch() obtains the dispatch record. */
typedef enum ep_dispatch_mode {
    EP_DISPATCH_FRESH = 0,    /* build the record from the layout inputs, then move the rows          */
    EP_DISPATCH_CACHED = 1,   /* reuse the record of an earlier dispatch; no top-k inputs or outputs  */
    EP_DISPATCH_PREPARED = 2  /* use the record that ep_notify_dispatch() just built for this call;
                                 top-k inputs and outputs as in fresh mode, layout inputs NULL        */
} ep_dispatch_mode;

/* The notify step of a dispatch ([P1] notify_dispatch; [P3] §4.1 the
 * prefix matrices, recv_src_idx, send_head and num_recv_tokens_per_expert):
 * builds the handle's dispatch record for num_tokens tokens per rank from
 * num_tokens_per_rank [R][R], is_token_in_rank [R][T][R] and
 * num_tokens_per_expert [R][E], and writes num_recv_tokens_per_expert
 * [R][EL] (aligned).  Exactly what the fresh mode of ep_dispatch() does
 * first; call it on its own to read the receive counts
 * (ep_handle_num_recv) before moving any row, then ep_dispatch() in
 * EP_DISPATCH_PREPARED mode with the same num_tokens. */
ep_status ep_notify_dispatch(ep_handle* h, int32_t num_tokens, const int32_t* num_tokens_per_rank,
                             const uint8_t* is_token_in_rank, const int32_t* num_tokens_per_expert,
                             int32_t* num_recv_tokens_per_expert, ep_stream_t stream);

/* ep_get_dispatch_layout() followed by ep_notify_dispatch(), in one launch
 * ([P3] §4.1: the layout, then the notify step of the dispatch).  The layout
 * outputs are written as by ep_get_dispatch_layout() (num_tokens_per_rdma_rank
 * optional) and the dispatch record and num_recv_tokens_per_expert [R][EL] as
 * by ep_notify_dispatch(); follow with ep_dispatch() in EP_DISPATCH_PREPARED
 * mode with the same num_tokens.
 * With num_tokens >= 1 this is one pass of a decoupled look-back scan: CTAs
 * take tiles of 512 tokens in (source, token) order -- the receive order of
 * every destination rank -- publish their per-rank and per-node hit counts,
 * and add up those of the earlier tiles; with two or more whole nodes of 8
 * ranks it also writes the node-level record.  With num_tokens == 0 the two
 * steps run one after the other.  The rank mask applies as in
 * ep_get_dispatch_layout().  Every wait is bounded and a timeout sets
 * EP_ERR_TIMEOUT in the status word.  Errors as the two calls it stands for. */
ep_status ep_layout_notify(ep_handle* h, int32_t num_tokens, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                           int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                           uint8_t* is_token_in_rank, int32_t* num_recv_tokens_per_expert, ep_stream_t stream);

/* Normal-mode dispatch ([P3] §4.1 intranode_dispatch).
 *
 * `cached` takes an ep_dispatch_mode.  Fresh mode (EP_DISPATCH_FRESH): first
 * builds the dispatch record in the handle from num_tokens_per_rank [R][R],
 * is_token_in_rank [R][T][R] and num_tokens_per_expert [R][E] (the layout
 * outputs), as ep_notify_dispatch() does:
 *   rank_prefix_matrix[s][r] = sum_{s'<=s} num_tokens_per_rank[s'][r]
 *   receive rows: inside rank r, tokens arrive ordered by source rank, then
 *     token index; send_head[s][t][r] = that row, or -1 if not sent
 *   recv_src_idx[r][row] = t
 *   channel_prefix_matrix[s][r][c] = hits of (s -> r) among tokens before
 *     the end of channel c (channel c = tokens [c*ceil(T/C), (c+1)*ceil(T/C)))
 *   recv_channel_prefix_matrix[r][s][c] = first row of that channel in r
 *   num_recv_tokens_per_expert[r][j] (int32 [R][EL], output) = received
 *     top-k slots of local expert j, rounded up to expert_alignment
 *   with two or more whole nodes of 8 ranks ([P3] §4.2, the two-level
 *     layout), the node-level record as well (EP_FIELD_RDMA_CHANNEL_PREFIX_MATRIX,
 *     EP_FIELD_RECV_RDMA_RANK_PREFIX_SUM): a token counts once per node it
 *     reaches, whatever the number of that node's ranks
 * Cached mode (EP_DISPATCH_CACHED): reuses the record of the last fresh or
 * prepared dispatch on this handle with the same num_tokens; topk_idx,
 * topk_weights, the three layout inputs, recv_topk_* and
 * num_recv_tokens_per_expert must be NULL ([P3] §4.1: a cached handle takes
 * no top-k inputs).  Prepared mode (EP_DISPATCH_PREPARED): the record of the
 * ep_notify_dispatch() call just made with the same num_tokens; the layout
 * inputs and num_recv_tokens_per_expert must be NULL, top-k as in fresh mode.
 *
 * Payload (both modes), for every (s,t) and every rank r it is sent to:
 *   x_dtype == EP_BF16, cast_to_fp8 == 0: recv_x[r][row] = x[s][t] (bf16 [.][.][H])
 *   x_dtype == EP_BF16, cast_to_fp8 != 0: recv_x[r][row] = e4m3 codes of
 *       x[s][t] and recv_x_scales[r][row][g] (fp32 [R][cap][G]) = the scale of
 *       group g: amax = max(max|x| over the 128 channels, 1e-4),
 *       scale = amax/448, code = e4m3_rne_satfinite(x * (448/amax))
 *   x_dtype == EP_FP8_E4M3: x holds e4m3 codes and x_scales [R][T][G] fp32
 *       its scales ([P3] §4.4 FP8 input); both are copied
 * Top-k metadata (fresh mode, optional): recv_topk_idx[r][row][k] (int64
 *   [R][cap][K]) = local expert id if slot k's expert lives on r, else -1;
 *   recv_topk_weights[r][row][k] (fp32) = topk_weights[s][t][k] then, else 0.
 * recv_x and recv_x_scales are [R][cap][...] with rank r's rows starting at
 * r*cap; rows at or past num_recv[r] are not written.  */
ep_status ep_dispatch(ep_handle* h, int32_t num_tokens,
                      const void* x, ep_dtype x_dtype, const float* x_scales, int32_t cast_to_fp8,
                      const int64_t* topk_idx, const float* topk_weights,
                      const int32_t* num_tokens_per_rank, const uint8_t* is_token_in_rank,
                      const int32_t* num_tokens_per_expert,
                      void* recv_x, float* recv_x_scales, int64_t* recv_topk_idx,
                      float* recv_topk_weights, int32_t* num_recv_tokens_per_expert,
                      int32_t cached, ep_stream_t stream);

/* --------------------------------------------------------- normal combine */

/* Normal-mode combine ([P3] §4.2; §4.4: the combine adds the returned rows
 * without weights, the top-k weights are reduced separately).  With the
 * record of the last fresh dispatch, for every token (s,t) and channel h:
 *   acc = float(bias_0[s][t][h]) + float(bias_1[s][t][h])   (a NULL bias counts 0)
 *   acc += float(x[r][send_head[s][t][r]][h]) for r = 0..R-1 that received it
 *   combined_x[s][t][h] = bf16_rne(acc)  (out_dtype EP_BF16), or acc (EP_FP32)
 * all in fp32 in exactly that order.  x is the expert output in the receive
 * layout, bf16 [R][cap][H]; bias_0/bias_1 bf16 [R][T][H] or NULL;
 * combined_x [R][T][H].  If topk_weights (fp32 [R][cap][K], the dispatched
 * recv_topk_weights) and combined_topk_weights (fp32 [R][T][K]) are both
 * given: combined_topk_weights[s][t][k] = sum over the same ranks, in the
 * same order, of topk_weights[r][row][k].  Tokens sent nowhere get the bias
 * sum (or 0) and zero weights. */
ep_status ep_combine(ep_handle* h, const void* x, const float* topk_weights,
                     const void* bias_0, const void* bias_1,
                     void* combined_x, ep_dtype out_dtype, float* combined_topk_weights,
                     ep_stream_t stream);

/* --------------------------------------------------- low-latency dispatch */

/* Bytes of one low-latency message ([P2] message package): a 16-byte header,
 * the payload (H e4m3 codes, or 2H bytes of bf16) and, for FP8, 4*G bytes of
 * scales.  16 + H + 4*H/128 or 16 + 2*H. */
int64_t ep_ll_msg_bytes(int32_t hidden, int32_t use_fp8);

/* Low-latency dispatch ([P1] low-latency dispatch / receive excerpts, [P2],
 * [P3] §4.3).  x bf16 [R][T][H] with T <= maxT, topk_idx int64 [R][T][K]
 * (8-byte aligned).
 * One message per valid slot (s,t,k) with e = topk_idx[s][t][k] goes to
 *   recv_msgs[d][j][row]  (uint8 [R][EL][R*maxT][msg_bytes]),  d = e/EL, j = e%EL
 * The rows of (d,j) are packed: source ranks in ascending order, each
 * source's slots in (token, k) order, so rows [0, packed_recv_count[d][j])
 * are valid.  Message: int32 {t, 0, 0, 0}; payload (bf16 copy, or e4m3 codes
 * of the per-128-channel cast); FP8 tail: fp32 scales, or with use_ue8m0
 * the exponent bytes e_g + 127 at tail[g] and zeros in tail[G..4G).
 * round_scale (implied by use_ue8m0) rounds each scale up to a power of two,
 * 2^e with e the smallest integer such that 2^e >= amax/448, and casts
 * x * 2^-e.  Outputs: packed_recv_count int32 [R][EL];
 * packed_recv_layout_range int64 [R][EL][R] = (count << 32) | begin of each
 * source's block; cumulative_local_expert_recv_stats (int32 [R][EL], may be
 * NULL) gets += packed_recv_count.  The slot -> row map stays in the handle
 * for ep_ll_combine().  Rows past R*maxT set EP_ERR_CAPACITY and are skipped. */
ep_status ep_ll_dispatch(ep_handle* h, int32_t num_tokens, const void* x, const int64_t* topk_idx,
                         int32_t use_fp8, int32_t round_scale, int32_t use_ue8m0,
                         void* recv_msgs, int32_t* packed_recv_count,
                         int64_t* packed_recv_layout_range,
                         int32_t* cumulative_local_expert_recv_stats, ep_stream_t stream);

/* ---------------------------------------------------- low-latency combine */

/* Low-latency combine ([P3] §4.3 low_latency_combine(x, topk_idx,
 * topk_weights, handle)), using the slot map of the last ep_ll_dispatch on
 * this handle.  x: expert outputs bf16 [R][EL][R*maxT][H] in the packed row
 * order; topk_idx int64 [R][T][K] and topk_weights fp32 [R][T][K] as given
 * to that dispatch.  For every token and channel:
 *   acc = 0; for k = 0..K-1 with a valid slot:
 *       acc = fmaf(topk_weights[s][t][k], float(x[d][j][row][h]), acc)
 *   combined_x[s][t][h] = bf16_rne(acc)          (bf16 [R][T][H]) */
ep_status ep_ll_combine(ep_handle* h, const void* x, const int64_t* topk_idx,
                        const float* topk_weights, void* combined_x, ep_stream_t stream);

/* ep_ll_combine() with strided expert-output rows: row (e, row) of x starts at
 * x + (e * R*maxT + row) * x_row_bytes (x 16-byte aligned; x_row_bytes a
 * multiple of 16, at least 2*H; the first 2*H bytes of a row are the bf16
 * outputs).  This is the zero-copy combine input of [P3] §4.3 (low-latency
 * combine can take its input straight from the communication buffer): after a
 * bf16 ep_ll_dispatch, x = recv_msgs + 16 with x_row_bytes =
 * ep_ll_msg_bytes(H, 0) reads the expert outputs written over the message
 * payloads in place.  EP_ERR_INVALID_ARG for a bad stride or alignment;
 * otherwise as ep_ll_combine(), which is this call with x_row_bytes = 2*H. */
ep_status ep_ll_combine_strided(ep_handle* h, const void* x, int64_t x_row_bytes, const int64_t* topk_idx,
                                const float* topk_weights, void* combined_x, ep_stream_t stream);

/* ------------------------------------------------------- rank masking */

/* The handle's mask buffer ([P1] low-latency: mask_buffer, is_rank_masked,
 * query / update / clean_mask_buffer): one int32 per rank, all zero after
 * ep_handle_create().  A masked rank neither sends nor receives:
 *  - ep_ll_dispatch() treats every slot whose source or destination rank is
 *    masked as a masked slot (no message, not counted, no contribution in
 *    ep_ll_combine());
 *  - the normal-mode layout (ep_get_dispatch_layout(), ep_layout_notify())
 *    does the same, so such slots are not counted in num_tokens_per_expert,
 *    the token does not go to that rank in is_token_in_rank and the counts,
 *    and the record, dispatch and combine built from that layout leave the
 *    rank out (it receives no row; its tokens go nowhere and combine to the
 *    bias sum).  ep_notify_dispatch() and a fresh ep_dispatch() follow the
 *    layout they are given; a cached dispatch or a combine follows its record,
 *    i.e. the mask as it was when the layout was computed.
 * The pages show the mask on the low-latency path only; the normal path
 * applies it the same way.
 *   update: asynchronously set (masked != 0) or clear one rank's entry;
 *   query:  synchronise `stream` and copy the R entries to host_mask[R];
 *   clean:  asynchronously clear every entry. */
ep_status ep_update_mask_buffer(ep_handle* h, int32_t rank, int32_t masked, ep_stream_t stream);
ep_status ep_query_mask_buffer(ep_handle* h, int32_t* host_mask, ep_stream_t stream);
ep_status ep_clean_mask_buffer(ep_handle* h, ep_stream_t stream);

/* Self-test of the bounded device waits (no counterpart on the pages): one
 * kernel waits, at most max_iterations (1..2^20) polls, on an mbarrier phase
 * that nothing completes.  The wait gives up, records EP_ERR_TIMEOUT in the
 * status word and masks `rank` -- what the pages' receiver does with a
 * source rank that never delivers -- and the kernel returns.  Nothing hangs
 * or traps; read the outcome with ep_handle_status() / ep_query_mask_buffer(). */
ep_status ep_selftest_bounded_wait(ep_handle* h, uint32_t max_iterations, int32_t rank, ep_stream_t stream);

/* ------------------------------------- low-latency dispatch, no allocation */

/* Capacity of the fixed count scratch of ep_ll_dispatch_noalloc(): int32
 * entries, one per (source rank, expert) pair, so num_ranks * num_experts
 * may not exceed it.  64 KiB of device memory per GPU that loads the library. */
#define EP_LL_NOALLOC_MAX_COUNTS 16384

/* No counterpart on the pages: this is an addition of this library for
 * callers that must not allocate device memory -- an engine plugin whose
 * enqueue path may not allocate, a server that reserves all device memory at
 * start-up, or a latency-critical loop that cannot take the synchronisation
 * cudaMalloc/cudaFree may cause.  It computes what ep_ll_dispatch() computes
 * on a handle with no rank masked -- there is no handle, so no mask buffer
 * applies and every rank sends and receives -- and every buffer is the
 * caller's, including the slot map and the status word:
 *   slot_row (int32 [R][maxT][K]): slot_row[s][t][k] is the row of slot
 *     (s, t, k) among the packed rows of its expert e = topk_idx[s][t][k],
 *     i.e. its message is recv_msgs[e / EL][e % EL][slot_row[s][t][k]]; -1
 *     for a masked slot or a row past R*maxT.  Entries of tokens t >=
 *     num_tokens are not written.  ep_ll_dispatch() keeps the same map in
 *     its handle (EP_FIELD_LL_SLOT_ROW), and ep_ll_combine() reads only that
 *     copy: no entry point of this library combines from a caller's
 *     slot_row, so a caller of this function gathers the expert outputs back
 *     with the map itself.
 *   status (one device int32): the kernels set it to the first error code and
 *     never clear it; the caller zeroes it.
 * The per-(source, expert) counts the kernels pass between them live in a
 * file-scope __device__ array of EP_LL_NOALLOC_MAX_COUNTS entries, so
 * num_ranks * num_experts beyond that is rejected with EP_ERR_UNSUPPORTED
 * before anything is enqueued.  The function calls no cudaMalloc, cudaFree
 * or other allocating routine.  Its first call on a device looks up the
 * array's device address and the launch shapes for that device; make that
 * first call before any stream capture.  Every call on a device shares the
 * array (it keeps the last call's counts, and nothing in it needs clearing),
 * so calls whose kernels may overlap on the GPU -- on different streams
 * without an ordering between them -- race and must not be issued.
 * Other sizes, layouts and errors as for ep_ll_dispatch(). */
ep_status ep_ll_dispatch_noalloc(int32_t num_ranks, int32_t num_tokens, int32_t num_max_tokens,
                                 int32_t hidden, int32_t num_experts, int32_t num_topk, const void* x,
                                 const int64_t* topk_idx, int32_t use_fp8, int32_t round_scale,
                                 int32_t use_ue8m0, void* recv_msgs, int32_t* packed_recv_count,
                                 int64_t* packed_recv_layout_range,
                                 int32_t* cumulative_local_expert_recv_stats, int32_t* slot_row,
                                 int32_t* status, ep_stream_t stream);

/* ------------------------------------------------------------ launch model
 * The SM-count model of [P1] (get_theoretical_num_sms, elastic.py), with the
 * one link of a single GPU -- HBM -- as the bottleneck.  All host-side; no
 * device call. */

/* Expected number of distinct groups hit by one token's top-k experts, for
 * num_experts experts split evenly into num_groups groups and the k experts
 * drawn uniformly without replacement ([P1] get_expected_topk):
 *   num_groups * (1 - C(E - E/G, k) / C(E, k)).
 * With G = num_ranks this is rho, the expected destination ranks per token.
 * Returns -1 (and sets ep_last_error) unless 1 <= G <= E, E % G == 0 and
 * 1 <= k <= E. */
double ep_expected_topk(int32_t num_groups, int32_t num_experts, int32_t num_topk);

/* Inputs of ep_theoretical_num_sms: bandwidths in GB/s. */
typedef struct ep_sm_model {
    double hbm_gbs;       /* HBM bandwidth the data kernels can reach (read + write bytes)   */
    double sm_read_gbs;   /* reads one SM of the data kernels sustains                       */
    double sm_write_gbs;  /* writes one SM of the data kernels sustains                      */
    int32_t num_device_sms;
    int32_t prefer_overlap_with_compute; /* 0: never fewer than min(64, num_device_sms) SMs  */
} ep_sm_model;

/* SMs a dispatch (for_combine == 0) or combine (for_combine != 0) needs to
 * keep HBM busy, by the steps of [P1] get_theoretical_num_sms with
 * rho = ep_expected_topk(num_ranks, num_experts, num_topk).  Per received
 * row, a dispatch reads 1/rho source rows and writes one row, a combine reads
 * one row and writes 1/rho rows, and HBM carries 1 + 1/rho rows:
 *   sms = max(hbm / (1 + 1/rho) * read / sm_read, hbm / (1 + 1/rho) * write / sm_write)
 *   sms = align_up(max(4, ceil(1.25 * sms)), 2)
 *   sms = max(sms, 64) unless prefer_overlap_with_compute; then min(sms, num_device_sms).
 * Returns -1 (and sets ep_last_error) for invalid arguments. */
int32_t ep_theoretical_num_sms(const ep_sm_model* model, int32_t num_ranks, int32_t num_experts, int32_t num_topk,
                               int32_t for_combine);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_EP_H */
