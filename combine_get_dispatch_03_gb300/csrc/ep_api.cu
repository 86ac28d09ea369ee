// ep_api.cu -- the C ABI: handle lifetime, argument validation, launches.
//
// The handle plays the role of the Buffer object of the pages ("第 4 章 V1：
// 布局、dispatch 与 combine" §4.1-§4.3): it fixes the sizes, owns the device
// arrays of the dispatch record (rank / channel prefix matrices,
// recv_src_idx, send_head; with two or more whole nodes of 8 ranks the
// node-level prefix matrices of the two-level layout; the low-latency slot
// map) and the status word that
// kernels use to report errors without trapping.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "ep_common.cuh"
#include "ep_kernels.h"
#include "ep_trace.h"

namespace ep {
cudaError_t plan_dispatch_combine(LaunchPlan* plan, int hidden);
cudaError_t plan_ll(LaunchPlan* plan, int num_experts);
}  // namespace ep

struct ep_handle {
    ep_config cfg;
    int device = -1;
    ep::LaunchPlan plan;
    void* dmem = nullptr;
    size_t dmem_bytes = 0;
    int32_t* status = nullptr;
    int32_t* rank_prefix = nullptr;          // [R][R]
    int32_t* channel_prefix = nullptr;       // [R][R][C]
    int32_t* recv_channel_prefix = nullptr;  // [R][R][C]
    int32_t* num_recv = nullptr;             // [R]
    int32_t* recv_src_idx = nullptr;         // [R][cap]
    int32_t* send_head = nullptr;            // [R][maxT][R]
    int32_t* ll_slot = nullptr;              // [R][maxT][K]
    int32_t* ll_cnt = nullptr;               // [R][E]
    int32_t* rank_mask = nullptr;            // [R], nonzero = masked
    int32_t* rdma_channel_prefix = nullptr;    // [R][NN][C], NN = R / 8 whole nodes (see has_nodes)
    int32_t* recv_rdma_rank_prefix = nullptr;  // [R][NN]
    int32_t* claims = nullptr;                 // [2]: the combine's next token and finished warps
    int32_t* layout_scratch = nullptr;         // tile states of the one-pass layout + record scan
    int normal_tokens = -1;                  // T of the current dispatch record, -1 = none
    bool prepared = false;                   // record built by ep_notify_dispatch, not yet used
    int ll_tokens = -1;                      // T of the last LL dispatch, -1 = none
};

namespace {

thread_local std::string g_last_error;

ep_status fail(ep_status code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

ep_status cuda_fail(cudaError_t err, const char* what) {
    return fail(EP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

// Two or more whole nodes of 8 ranks: the handle keeps the node-level record.
bool has_nodes(const ep_config& c) { return c.num_ranks > 8 && c.num_ranks % 8 == 0; }

// The node-level arrays the notify fills (0: channel prefix, 1: receive prefix), NULL without whole nodes.
int32_t* node_record(const ep_handle* h, int which) {
    if (!has_nodes(h->cfg)) return nullptr;
    return which == 0 ? h->rdma_channel_prefix : h->recv_rdma_rank_prefix;
}

#define EP_CHECK_ARG(cond, ...)                                  \
    do {                                                         \
        if (!(cond)) return fail(EP_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

// Makes the handle's device current for the duration of a call.
class DeviceGuard {
public:
    explicit DeviceGuard(int device) {
        cudaGetDevice(&prev_);
        if (prev_ != device) cudaSetDevice(device);
        restore_ = prev_ != device;
    }
    ~DeviceGuard() {
        if (restore_) cudaSetDevice(prev_);
    }

private:
    int prev_ = 0;
    bool restore_ = false;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

ep_status check_config(const ep_config* c) {
    if (c == nullptr) return fail(EP_ERR_INVALID_ARG, "config is NULL");
    if (c->num_ranks < 1 || c->num_ranks > ep::kMaxRanks)
        return fail(EP_ERR_UNSUPPORTED, "num_ranks %d outside [1, %d]", c->num_ranks, ep::kMaxRanks);
    if (c->num_max_tokens < 0) return fail(EP_ERR_INVALID_ARG, "num_max_tokens %d < 0", c->num_max_tokens);
    if (c->hidden < 8 || c->hidden % 8 != 0)
        return fail(EP_ERR_INVALID_ARG, "hidden %d must be a positive multiple of 8", c->hidden);
    if (c->num_experts < 1 || c->num_experts % c->num_ranks != 0)
        return fail(EP_ERR_INVALID_ARG, "num_experts %d must be a positive multiple of num_ranks %d",
                    c->num_experts, c->num_ranks);
    if (c->num_experts > ep::kMaxExperts)
        return fail(EP_ERR_UNSUPPORTED, "num_experts %d > %d", c->num_experts, ep::kMaxExperts);
    if (c->num_topk < 1 || c->num_topk > ep::kMaxTopk)
        return fail(EP_ERR_UNSUPPORTED, "num_topk %d outside [1, %d]", c->num_topk, ep::kMaxTopk);
    if (c->num_channels < 1) return fail(EP_ERR_INVALID_ARG, "num_channels %d < 1", c->num_channels);
    if (c->expert_alignment < 1) return fail(EP_ERR_INVALID_ARG, "expert_alignment %d < 1", c->expert_alignment);
    if (c->max_sms < 0) return fail(EP_ERR_INVALID_ARG, "max_sms %d < 0", c->max_sms);
    if (c->recv_capacity < 0 || c->recv_capacity > INT32_MAX)
        return fail(EP_ERR_INVALID_ARG, "recv_capacity %lld outside [0, 2^31)",
                    static_cast<long long>(c->recv_capacity));
    const int64_t ll_rows = static_cast<int64_t>(c->num_ranks) * c->num_max_tokens;
    if (ll_rows > INT32_MAX) return fail(EP_ERR_UNSUPPORTED, "num_ranks * num_max_tokens exceeds 2^31");
    // the top-k slots of one rank are indexed in int32
    if (static_cast<int64_t>(c->num_max_tokens) * c->num_topk > INT32_MAX)
        return fail(EP_ERR_UNSUPPORTED, "num_max_tokens * num_topk exceeds 2^31");
    return EP_OK;
}

ep_status check_tokens(const ep_handle* h, int32_t num_tokens) {
    if (num_tokens < 0 || num_tokens > h->cfg.num_max_tokens)
        return fail(EP_ERR_INVALID_ARG, "num_tokens %d outside [0, num_max_tokens=%d]", num_tokens,
                    h->cfg.num_max_tokens);
    return EP_OK;
}

}  // namespace

namespace ep {
// Lets other translation units of the library set the thread's ep_last_error() text.
void record_error(const char* message) { g_last_error = message ? message : ""; }
}  // namespace ep

extern "C" {

const char* ep_status_string(ep_status s) {
    switch (s) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_CAPACITY: return "receive buffer capacity exceeded";
        case EP_ERR_TIMEOUT: return "device wait timed out";
        case EP_ERR_CUDA: return "CUDA runtime error";
        case EP_ERR_UNSUPPORTED: return "unsupported size";
        case EP_ERR_INCONSISTENT: return "num_tokens_per_rank disagrees with is_token_in_rank";
        case EP_ERR_BAD_EXPERT: return "expert id out of range";
        case EP_ERR_STATE: return "no prior dispatch for this call";
    }
    return "unknown status";
}

const char* ep_last_error(void) { return g_last_error.c_str(); }

int64_t ep_ll_msg_bytes(int32_t hidden, int32_t use_fp8) {
    if (hidden <= 0) return -1;
    return use_fp8 ? 16 + static_cast<int64_t>(hidden) + 4 * static_cast<int64_t>(hidden / 128)
                   : 16 + 2 * static_cast<int64_t>(hidden);
}

ep_status ep_handle_create(const ep_config* cfg, ep_handle** out) {
    EP_TRACE();
    if (out == nullptr) return fail(EP_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    ep_status st = check_config(cfg);
    if (st != EP_OK) return st;

    ep_handle* h = new ep_handle();
    h->cfg = *cfg;
    cudaError_t err = cudaGetDevice(&h->device);
    if (err != cudaSuccess) {
        delete h;
        return cuda_fail(err, "cudaGetDevice");
    }
    err = cudaDeviceGetAttribute(&h->plan.num_sms, cudaDevAttrMultiProcessorCount, h->device);
    if (err == cudaSuccess && cfg->max_sms > 0 && cfg->max_sms < h->plan.num_sms) {
        h->plan.num_sms = cfg->max_sms;
        h->plan.sm_limited = true;
    }
    if (err == cudaSuccess) err = ep::plan_dispatch_combine(&h->plan, cfg->hidden);
    if (err == cudaSuccess) err = ep::plan_ll(&h->plan, cfg->num_experts);
    if (err != cudaSuccess) {
        delete h;
        return cuda_fail(err, "planning launches");
    }

    const size_t R = cfg->num_ranks, C = cfg->num_channels, T = cfg->num_max_tokens, K = cfg->num_topk;
    const size_t E = cfg->num_experts, cap = static_cast<size_t>(cfg->recv_capacity);
    const size_t NN = (R + 7) / 8;
    const size_t scan_words = ep::layout_scan_scratch_words(cfg->num_ranks, cfg->num_experts, cfg->num_max_tokens);
    const size_t sizes[] = {1, R * R, R * R * C, R * R * C, R, R * cap, R * T * R, R * T * K, R * E, R,
                            R * NN * C, R * NN, 2, scan_words};
    int32_t** slots[] = {&h->status,   &h->rank_prefix,  &h->channel_prefix, &h->recv_channel_prefix,
                         &h->num_recv, &h->recv_src_idx, &h->send_head,      &h->ll_slot,
                         &h->ll_cnt,   &h->rank_mask,    &h->rdma_channel_prefix, &h->recv_rdma_rank_prefix,
                         &h->claims,   &h->layout_scratch};
    size_t total = 0;
    for (size_t s : sizes) total += align_up(s * sizeof(int32_t), 256);
    err = cudaMalloc(&h->dmem, total);
    if (err != cudaSuccess) {
        delete h;
        return cuda_fail(err, "cudaMalloc(handle)");
    }
    h->dmem_bytes = total;
    size_t off = 0;
    for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
        *slots[i] = reinterpret_cast<int32_t*>(static_cast<char*>(h->dmem) + off);
        off += align_up(sizes[i] * sizeof(int32_t), 256);
    }
    err = cudaMemset(h->dmem, 0, total);  // the status word, the claim counters and the scan's tickets start at 0
    if (err != cudaSuccess) {
        cudaFree(h->dmem);
        delete h;
        return cuda_fail(err, "cudaMemset(handle)");
    }
    *out = h;
    return EP_OK;
}

void ep_handle_destroy(ep_handle* h) {
    EP_TRACE();
    if (h == nullptr) return;
    DeviceGuard guard(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->dmem);
    delete h;
}

ep_status ep_handle_status(ep_handle* h, ep_stream_t stream, int32_t reset) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    DeviceGuard guard(h->device);
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "cudaStreamSynchronize");
    int32_t word = 0;
    err = cudaMemcpy(&word, h->status, sizeof word, cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_fail(err, "reading the status word");
    if (reset && word != 0) {
        err = cudaMemset(h->status, 0, sizeof(int32_t));
        if (err != cudaSuccess) return cuda_fail(err, "clearing the status word");
    }
    if (word != 0) fail(static_cast<ep_status>(word), "device reported: %s", ep_status_string(static_cast<ep_status>(word)));
    return static_cast<ep_status>(word);
}

ep_status ep_handle_num_recv(ep_handle* h, int32_t* host_num_recv, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr || host_num_recv == nullptr) return fail(EP_ERR_INVALID_ARG, "NULL argument");
    if (h->normal_tokens < 0) return fail(EP_ERR_STATE, "no normal dispatch on this handle yet");
    DeviceGuard guard(h->device);
    cudaError_t err = cudaMemcpyAsync(host_num_recv, h->num_recv, sizeof(int32_t) * h->cfg.num_ranks,
                                      cudaMemcpyDefault, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "reading num_recv");
    return EP_OK;
}

size_t ep_handle_field_bytes(const ep_handle* h, ep_handle_field field) {
    if (h == nullptr) return 0;
    const size_t R = h->cfg.num_ranks, C = h->cfg.num_channels, T = h->cfg.num_max_tokens;
    const size_t K = h->cfg.num_topk, cap = static_cast<size_t>(h->cfg.recv_capacity);
    switch (field) {
        case EP_FIELD_RANK_PREFIX_MATRIX: return sizeof(int32_t) * R * R;
        case EP_FIELD_CHANNEL_PREFIX_MATRIX:
        case EP_FIELD_RECV_CHANNEL_PREFIX_MATRIX: return sizeof(int32_t) * R * R * C;
        case EP_FIELD_RECV_SRC_IDX: return sizeof(int32_t) * R * cap;
        case EP_FIELD_SEND_HEAD: return sizeof(int32_t) * R * T * R;
        case EP_FIELD_NUM_RECV: return sizeof(int32_t) * R;
        case EP_FIELD_LL_SLOT_ROW: return sizeof(int32_t) * R * T * K;
        case EP_FIELD_RDMA_CHANNEL_PREFIX_MATRIX: return has_nodes(h->cfg) ? sizeof(int32_t) * R * (R / 8) * C : 0;
        case EP_FIELD_RECV_RDMA_RANK_PREFIX_SUM: return has_nodes(h->cfg) ? sizeof(int32_t) * R * (R / 8) : 0;
    }
    return 0;
}

ep_status ep_handle_export(const ep_handle* h, ep_handle_field field, void* dst, size_t bytes,
                           ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr || dst == nullptr) return fail(EP_ERR_INVALID_ARG, "NULL argument");
    const bool node_field =
        field == EP_FIELD_RDMA_CHANNEL_PREFIX_MATRIX || field == EP_FIELD_RECV_RDMA_RANK_PREFIX_SUM;
    if (node_field && !has_nodes(h->cfg))
        return fail(EP_ERR_UNSUPPORTED,
                    "the node-level record needs two or more whole nodes of 8 ranks (handle has %d ranks)",
                    h->cfg.num_ranks);
    const size_t need = ep_handle_field_bytes(h, field);
    if (need == 0 && field != EP_FIELD_RECV_SRC_IDX && field != EP_FIELD_SEND_HEAD && field != EP_FIELD_LL_SLOT_ROW)
        return fail(EP_ERR_INVALID_ARG, "unknown field %d", static_cast<int>(field));
    if (bytes < need) return fail(EP_ERR_INVALID_ARG, "destination holds %zu bytes, %zu needed", bytes, need);
    const int32_t* src = nullptr;
    switch (field) {
        case EP_FIELD_RANK_PREFIX_MATRIX: src = h->rank_prefix; break;
        case EP_FIELD_CHANNEL_PREFIX_MATRIX: src = h->channel_prefix; break;
        case EP_FIELD_RECV_CHANNEL_PREFIX_MATRIX: src = h->recv_channel_prefix; break;
        case EP_FIELD_RECV_SRC_IDX: src = h->recv_src_idx; break;
        case EP_FIELD_SEND_HEAD: src = h->send_head; break;
        case EP_FIELD_NUM_RECV: src = h->num_recv; break;
        case EP_FIELD_LL_SLOT_ROW: src = h->ll_slot; break;
        case EP_FIELD_RDMA_CHANNEL_PREFIX_MATRIX: src = h->rdma_channel_prefix; break;
        case EP_FIELD_RECV_RDMA_RANK_PREFIX_SUM: src = h->recv_rdma_rank_prefix; break;
        default: return fail(EP_ERR_INVALID_ARG, "unknown field %d", static_cast<int>(field));
    }
    if (need == 0) return EP_OK;
    DeviceGuard guard(h->device);
    cudaError_t err = cudaMemcpyAsync(dst, src, need, cudaMemcpyDefault, stream);
    if (err != cudaSuccess) return cuda_fail(err, "copying a handle field");
    return EP_OK;
}

ep_status ep_get_dispatch_layout(ep_handle* h, int32_t num_tokens, const int64_t* topk_idx,
                                 int32_t* num_tokens_per_rank, int32_t* num_tokens_per_rdma_rank,
                                 int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    ep_status st = check_tokens(h, num_tokens);
    if (st != EP_OK) return st;
    const ep_config& c = h->cfg;
    EP_CHECK_ARG(num_tokens == 0 || topk_idx != nullptr, "topk_idx is NULL");
    EP_CHECK_ARG(num_tokens_per_rank && num_tokens_per_expert && is_token_in_rank, "a layout output is NULL");
    EP_CHECK_ARG(aligned8(topk_idx) && aligned4(num_tokens_per_rank) && aligned4(num_tokens_per_expert) &&
                     aligned4(num_tokens_per_rdma_rank) && aligned16(is_token_in_rank),
                 "misaligned layout pointer");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_get_dispatch_layout(topk_idx, h->rank_mask, c.num_ranks, num_tokens, c.num_topk,
                                                     c.num_experts, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                                     num_tokens_per_expert, is_token_in_rank, h->status, stream);
    if (err != cudaSuccess) return cuda_fail(err, "get_dispatch_layout launch");
    return EP_OK;
}

ep_status ep_dispatch(ep_handle* h, int32_t num_tokens, const void* x, ep_dtype x_dtype, const float* x_scales,
                      int32_t cast_to_fp8, const int64_t* topk_idx, const float* topk_weights,
                      const int32_t* num_tokens_per_rank, const uint8_t* is_token_in_rank,
                      const int32_t* num_tokens_per_expert, void* recv_x, float* recv_x_scales,
                      int64_t* recv_topk_idx, float* recv_topk_weights, int32_t* num_recv_tokens_per_expert,
                      int32_t cached, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    ep_status st = check_tokens(h, num_tokens);
    if (st != EP_OK) return st;
    const ep_config& c = h->cfg;
    EP_CHECK_ARG(c.recv_capacity > 0, "handle was created with recv_capacity 0 (normal mode disabled)");
    EP_CHECK_ARG(x_dtype == EP_BF16 || x_dtype == EP_FP8_E4M3, "x_dtype must be EP_BF16 or EP_FP8_E4M3");
    int mode = ep::kModeBf16;
    if (x_dtype == EP_FP8_E4M3) {
        EP_CHECK_ARG(!cast_to_fp8, "cast_to_fp8 needs a bf16 input");
        mode = ep::kModeFp8In;
    } else if (cast_to_fp8) {
        mode = ep::kModeCastFp8;
    }
    if (mode != ep::kModeBf16) {
        if (c.hidden % ep::kFp8Group != 0)
            return fail(EP_ERR_UNSUPPORTED, "FP8 payloads need hidden %% 128 == 0 (hidden %d)", c.hidden);
        EP_CHECK_ARG(recv_x_scales != nullptr && aligned4(recv_x_scales), "FP8 dispatch needs recv_x_scales");
        if (mode == ep::kModeFp8In) EP_CHECK_ARG(num_tokens == 0 || (x_scales && aligned4(x_scales)), "FP8 input needs x_scales");
    } else {
        EP_CHECK_ARG(x_scales == nullptr && recv_x_scales == nullptr, "bf16 dispatch takes no scales");
    }
    EP_CHECK_ARG(num_tokens == 0 || (x != nullptr && aligned16(x)), "x must be a 16-byte aligned device pointer");
    EP_CHECK_ARG(recv_x != nullptr && aligned16(recv_x), "recv_x must be a 16-byte aligned device pointer");

    EP_CHECK_ARG(cached == EP_DISPATCH_FRESH || cached == EP_DISPATCH_CACHED || cached == EP_DISPATCH_PREPARED,
                 "unknown dispatch mode %d", cached);
    if (cached == EP_DISPATCH_PREPARED) {
        EP_CHECK_ARG(num_tokens_per_rank == nullptr && is_token_in_rank == nullptr && num_tokens_per_expert == nullptr &&
                         num_recv_tokens_per_expert == nullptr,
                     "prepared dispatch takes no layout arguments (ep_notify_dispatch had them)");
        if (!h->prepared || h->normal_tokens != num_tokens)
            return fail(EP_ERR_STATE, "prepared dispatch without an ep_notify_dispatch for %d tokens", num_tokens);
        EP_CHECK_ARG((recv_topk_idx == nullptr && recv_topk_weights == nullptr) || topk_idx != nullptr,
                     "recv_topk_* outputs need topk_idx");
        EP_CHECK_ARG(recv_topk_weights == nullptr || topk_weights != nullptr, "recv_topk_weights needs topk_weights");
        EP_CHECK_ARG(aligned8(topk_idx) && aligned4(topk_weights) && aligned8(recv_topk_idx) &&
                         aligned4(recv_topk_weights),
                     "misaligned top-k pointer");
    } else if (cached == EP_DISPATCH_CACHED) {
        EP_CHECK_ARG(topk_idx == nullptr && topk_weights == nullptr && num_tokens_per_rank == nullptr &&
                         is_token_in_rank == nullptr && num_tokens_per_expert == nullptr &&
                         recv_topk_idx == nullptr && recv_topk_weights == nullptr &&
                         num_recv_tokens_per_expert == nullptr,
                     "cached dispatch takes no top-k or layout arguments");
        if (h->normal_tokens < 0) return fail(EP_ERR_STATE, "cached dispatch without a prior fresh dispatch");
        if (h->normal_tokens != num_tokens)
            return fail(EP_ERR_STATE, "cached dispatch with %d tokens, the record holds %d", num_tokens,
                        h->normal_tokens);
    } else {
        EP_CHECK_ARG(num_tokens_per_rank && is_token_in_rank && num_tokens_per_expert && num_recv_tokens_per_expert,
                     "fresh dispatch needs the layout inputs and num_recv_tokens_per_expert");
        EP_CHECK_ARG(aligned4(num_tokens_per_rank) && aligned16(is_token_in_rank) && aligned4(num_tokens_per_expert) &&
                         aligned4(num_recv_tokens_per_expert),
                     "misaligned layout pointer");
        EP_CHECK_ARG((recv_topk_idx == nullptr && recv_topk_weights == nullptr) || topk_idx != nullptr,
                     "recv_topk_* outputs need topk_idx");
        EP_CHECK_ARG(recv_topk_weights == nullptr || topk_weights != nullptr, "recv_topk_weights needs topk_weights");
        EP_CHECK_ARG(aligned8(topk_idx) && aligned4(topk_weights) && aligned8(recv_topk_idx) &&
                         aligned4(recv_topk_weights),
                     "misaligned top-k pointer");
    }

    DeviceGuard guard(h->device);
    cudaError_t err;
    if (cached == EP_DISPATCH_FRESH) {
        err = ep::launch_dispatch_notify(c.num_ranks, num_tokens, c.num_experts, c.num_channels, c.expert_alignment,
                                         c.recv_capacity, num_tokens_per_rank, is_token_in_rank,
                                         num_tokens_per_expert, h->rank_prefix, h->channel_prefix,
                                         h->recv_channel_prefix, h->num_recv, h->send_head, h->recv_src_idx,
                                         num_recv_tokens_per_expert, node_record(h, 0), node_record(h, 1),
                                         h->status, stream);
        if (err != cudaSuccess) return cuda_fail(err, "dispatch_notify launch");
        h->normal_tokens = num_tokens;
    }
    h->prepared = false;
    const bool with_topk = cached != EP_DISPATCH_CACHED;
    err = ep::launch_dispatch(h->plan, mode, c.num_ranks, num_tokens, c.hidden, c.num_topk,
                              c.num_experts / c.num_ranks, c.recv_capacity, x, x_scales,
                              with_topk ? topk_idx : nullptr, with_topk ? topk_weights : nullptr, h->send_head,
                              recv_x, recv_x_scales, recv_topk_idx, recv_topk_weights, h->status, stream);
    if (err != cudaSuccess) return cuda_fail(err, "dispatch launch");
    return EP_OK;
}

ep_status ep_notify_dispatch(ep_handle* h, int32_t num_tokens, const int32_t* num_tokens_per_rank,
                             const uint8_t* is_token_in_rank, const int32_t* num_tokens_per_expert,
                             int32_t* num_recv_tokens_per_expert, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    ep_status st = check_tokens(h, num_tokens);
    if (st != EP_OK) return st;
    const ep_config& c = h->cfg;
    EP_CHECK_ARG(c.recv_capacity > 0, "handle was created with recv_capacity 0 (normal mode disabled)");
    EP_CHECK_ARG(num_tokens_per_rank && is_token_in_rank && num_tokens_per_expert && num_recv_tokens_per_expert,
                 "the layout inputs and num_recv_tokens_per_expert are required");
    EP_CHECK_ARG(aligned4(num_tokens_per_rank) && aligned16(is_token_in_rank) && aligned4(num_tokens_per_expert) &&
                     aligned4(num_recv_tokens_per_expert),
                 "misaligned layout pointer");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_dispatch_notify(
        c.num_ranks, num_tokens, c.num_experts, c.num_channels, c.expert_alignment, c.recv_capacity,
        num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert, h->rank_prefix, h->channel_prefix,
        h->recv_channel_prefix, h->num_recv, h->send_head, h->recv_src_idx, num_recv_tokens_per_expert,
        node_record(h, 0), node_record(h, 1), h->status, stream);
    if (err != cudaSuccess) return cuda_fail(err, "dispatch_notify launch");
    h->normal_tokens = num_tokens;
    h->prepared = true;
    return EP_OK;
}

ep_status ep_layout_notify(ep_handle* h, int32_t num_tokens, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
                           int32_t* num_tokens_per_rdma_rank, int32_t* num_tokens_per_expert,
                           uint8_t* is_token_in_rank, int32_t* num_recv_tokens_per_expert, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    ep_status st = check_tokens(h, num_tokens);
    if (st != EP_OK) return st;
    const ep_config& c = h->cfg;
    EP_CHECK_ARG(c.recv_capacity > 0, "handle was created with recv_capacity 0 (normal mode disabled)");
    EP_CHECK_ARG(num_tokens == 0 || topk_idx != nullptr, "topk_idx is NULL");
    EP_CHECK_ARG(num_tokens_per_rank && num_tokens_per_expert && is_token_in_rank && num_recv_tokens_per_expert,
                 "a layout output or num_recv_tokens_per_expert is NULL");
    EP_CHECK_ARG(aligned8(topk_idx) && aligned4(num_tokens_per_rank) && aligned4(num_tokens_per_expert) &&
                     aligned4(num_tokens_per_rdma_rank) && aligned16(is_token_in_rank) &&
                     aligned4(num_recv_tokens_per_expert),
                 "misaligned layout pointer");
    DeviceGuard guard(h->device);
    cudaError_t err;
    if (num_tokens >= 1) {
        // one pass: a decoupled look-back scan over token tiles in receive order
        err = ep::launch_layout_scan(topk_idx, h->rank_mask, c.num_ranks, num_tokens, c.num_topk, c.num_experts,
                                     c.num_channels, c.expert_alignment, c.recv_capacity, num_tokens_per_rank,
                                     num_tokens_per_rdma_rank, num_tokens_per_expert, is_token_in_rank,
                                     h->rank_prefix, h->channel_prefix, h->recv_channel_prefix, h->num_recv,
                                     h->send_head, h->recv_src_idx, num_recv_tokens_per_expert, node_record(h, 0),
                                     node_record(h, 1), reinterpret_cast<uint32_t*>(h->layout_scratch), h->status,
                                     stream);
        if (err != cudaSuccess) return cuda_fail(err, "layout scan launch");
    } else {
        // no tokens: the two calls it stands for (their kernels write the empty record)
        err = ep::launch_get_dispatch_layout(topk_idx, h->rank_mask, c.num_ranks, num_tokens, c.num_topk,
                                             c.num_experts, num_tokens_per_rank, num_tokens_per_rdma_rank,
                                             num_tokens_per_expert, is_token_in_rank, h->status, stream);
        if (err == cudaSuccess)
            err = ep::launch_dispatch_notify(
                c.num_ranks, num_tokens, c.num_experts, c.num_channels, c.expert_alignment, c.recv_capacity,
                num_tokens_per_rank, is_token_in_rank, num_tokens_per_expert, h->rank_prefix, h->channel_prefix,
                h->recv_channel_prefix, h->num_recv, h->send_head, h->recv_src_idx, num_recv_tokens_per_expert,
                node_record(h, 0), node_record(h, 1), h->status, stream);
        if (err != cudaSuccess) return cuda_fail(err, "layout / notify launch");
    }
    h->normal_tokens = num_tokens;
    h->prepared = true;
    return EP_OK;
}

ep_status ep_combine(ep_handle* h, const void* x, const float* topk_weights, const void* bias_0,
                     const void* bias_1, void* combined_x, ep_dtype out_dtype, float* combined_topk_weights,
                     ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    if (h->normal_tokens < 0) return fail(EP_ERR_STATE, "combine without a prior dispatch");
    const ep_config& c = h->cfg;
    const int T = h->normal_tokens;
    EP_CHECK_ARG(out_dtype == EP_BF16 || out_dtype == EP_FP32, "out_dtype must be EP_BF16 or EP_FP32");
    EP_CHECK_ARG(x != nullptr && aligned16(x), "x must be a 16-byte aligned device pointer");
    EP_CHECK_ARG(T == 0 || (combined_x != nullptr && aligned16(combined_x)),
                 "combined_x must be a 16-byte aligned device pointer");
    EP_CHECK_ARG(aligned16(bias_0) && aligned16(bias_1), "biases must be 16-byte aligned");
    EP_CHECK_ARG((topk_weights == nullptr) == (combined_topk_weights == nullptr),
                 "topk_weights and combined_topk_weights go together");
    EP_CHECK_ARG(aligned4(topk_weights) && aligned4(combined_topk_weights), "misaligned weights");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_combine(h->plan, out_dtype == EP_FP32, c.num_ranks, T, c.hidden, c.num_topk,
                                         c.recv_capacity, h->send_head, x, topk_weights, bias_0, bias_1, combined_x,
                                         combined_topk_weights, reinterpret_cast<uint32_t*>(h->claims), stream);
    if (err != cudaSuccess) return cuda_fail(err, "combine launch");
    return EP_OK;
}

ep_status ep_ll_dispatch(ep_handle* h, int32_t num_tokens, const void* x, const int64_t* topk_idx, int32_t use_fp8,
                         int32_t round_scale, int32_t use_ue8m0, void* recv_msgs, int32_t* packed_recv_count,
                         int64_t* packed_recv_layout_range, int32_t* cumulative_local_expert_recv_stats,
                         ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    ep_status st = check_tokens(h, num_tokens);
    if (st != EP_OK) return st;
    const ep_config& c = h->cfg;
    EP_CHECK_ARG(!use_ue8m0 || use_fp8, "use_ue8m0 needs use_fp8");
    if (use_fp8 && c.hidden % 512 != 0)
        return fail(EP_ERR_UNSUPPORTED, "FP8 low-latency messages need hidden %% 512 == 0 (hidden %d)", c.hidden);
    EP_CHECK_ARG(num_tokens == 0 || (x != nullptr && aligned16(x) && topk_idx != nullptr && aligned8(topk_idx)),
                 "x (16-byte aligned) and topk_idx are required");
    EP_CHECK_ARG(recv_msgs != nullptr && aligned16(recv_msgs), "recv_msgs must be a 16-byte aligned device pointer");
    EP_CHECK_ARG(packed_recv_count && packed_recv_layout_range && aligned4(packed_recv_count) &&
                     aligned8(packed_recv_layout_range) && aligned4(cumulative_local_expert_recv_stats),
                 "packed_recv_count / packed_recv_layout_range missing or misaligned");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_ll_dispatch(h->plan, c.num_ranks, num_tokens, c.num_max_tokens, c.hidden, c.num_topk,
                                             c.num_experts, x, topk_idx, use_fp8 != 0, round_scale != 0,
                                             use_ue8m0 != 0, h->rank_mask, h->ll_slot, h->ll_cnt, recv_msgs, packed_recv_count,
                                             packed_recv_layout_range, cumulative_local_expert_recv_stats, h->status,
                                             stream);
    if (err != cudaSuccess) return cuda_fail(err, "low-latency dispatch launch");
    h->ll_tokens = num_tokens;
    return EP_OK;
}

ep_status ep_ll_combine_strided(ep_handle* h, const void* x, int64_t x_row_bytes, const int64_t* topk_idx,
                                const float* topk_weights, void* combined_x, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    if (h->ll_tokens < 0) return fail(EP_ERR_STATE, "low-latency combine without a prior low-latency dispatch");
    const ep_config& c = h->cfg;
    const int T = h->ll_tokens;
    EP_CHECK_ARG(x != nullptr && aligned16(x), "x must be a 16-byte aligned device pointer");
    EP_CHECK_ARG(x_row_bytes >= 2 * static_cast<int64_t>(c.hidden) && x_row_bytes % 16 == 0,
                 "x_row_bytes %lld must be a multiple of 16 and at least 2 * hidden = %d",
                 static_cast<long long>(x_row_bytes), 2 * c.hidden);
    EP_CHECK_ARG(T == 0 || (topk_idx && topk_weights && combined_x && aligned8(topk_idx) && aligned4(topk_weights) &&
                            aligned16(combined_x)),
                 "topk_idx, topk_weights and a 16-byte aligned combined_x are required");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_ll_combine(h->plan, c.num_ranks, T, c.num_max_tokens, c.hidden, c.num_topk,
                                            c.num_experts, x, x_row_bytes, topk_idx, topk_weights, h->ll_slot,
                                            combined_x, stream);
    if (err != cudaSuccess) return cuda_fail(err, "low-latency combine launch");
    return EP_OK;
}

ep_status ep_ll_combine(ep_handle* h, const void* x, const int64_t* topk_idx, const float* topk_weights,
                        void* combined_x, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    return ep_ll_combine_strided(h, x, 2 * static_cast<int64_t>(h->cfg.hidden), topk_idx, topk_weights, combined_x,
                                 stream);
}

ep_status ep_update_mask_buffer(ep_handle* h, int32_t rank, int32_t masked, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    EP_CHECK_ARG(rank >= 0 && rank < h->cfg.num_ranks, "rank %d outside [0, %d)", rank, h->cfg.num_ranks);
    DeviceGuard guard(h->device);
    cudaError_t err = cudaMemsetAsync(h->rank_mask + rank, 0, sizeof(int32_t), stream);
    if (err == cudaSuccess && masked) err = cudaMemsetAsync(h->rank_mask + rank, 1, 1, stream);
    if (err != cudaSuccess) return cuda_fail(err, "updating the mask buffer");
    return EP_OK;
}

ep_status ep_query_mask_buffer(ep_handle* h, int32_t* host_mask, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr || host_mask == nullptr) return fail(EP_ERR_INVALID_ARG, "NULL argument");
    DeviceGuard guard(h->device);
    cudaError_t err = cudaMemcpyAsync(host_mask, h->rank_mask, sizeof(int32_t) * h->cfg.num_ranks, cudaMemcpyDefault,
                                      stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_fail(err, "reading the mask buffer");
    return EP_OK;
}

ep_status ep_clean_mask_buffer(ep_handle* h, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    DeviceGuard guard(h->device);
    cudaError_t err = cudaMemsetAsync(h->rank_mask, 0, sizeof(int32_t) * h->cfg.num_ranks, stream);
    if (err != cudaSuccess) return cuda_fail(err, "clearing the mask buffer");
    return EP_OK;
}

ep_status ep_selftest_bounded_wait(ep_handle* h, uint32_t max_iterations, int32_t rank, ep_stream_t stream) {
    EP_TRACE();
    if (h == nullptr) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    EP_CHECK_ARG(rank >= 0 && rank < h->cfg.num_ranks, "rank %d outside [0, %d)", rank, h->cfg.num_ranks);
    EP_CHECK_ARG(max_iterations >= 1 && max_iterations <= (1u << 20), "max_iterations must lie in [1, 2^20]");
    DeviceGuard guard(h->device);
    cudaError_t err = ep::launch_bounded_wait_selftest(max_iterations, rank, h->rank_mask, h->status, stream);
    if (err != cudaSuccess) return cuda_fail(err, "self-test launch");
    return EP_OK;
}

}  // extern "C"
