// ep_noalloc.cu -- low-latency dispatch for callers that cannot allocate device memory.
//
// ep_ll_dispatch() keeps its per-(source rank, expert) slot counts in memory
// that ep_handle_create() obtains with cudaMalloc.  Some callers cannot do
// that: a plugin running inside an inference engine whose enqueue path must
// not allocate, a server that reserves all device memory once at start-up and
// forbids later allocations, or a latency-critical loop that cannot afford
// the device-wide synchronisation cudaMalloc/cudaFree may cause.  For them,
// ep_ll_dispatch_noalloc() runs the same kernels with that count array in a
// fixed-size file-scope __device__ array instead, and takes every other
// buffer (slot map, status word included) from the caller.  It has no handle,
// so no rank mask applies.
//
// The array lives in the library image, so every GPU that loads the library
// holds its 64 KiB until the process exits.  All calls on a device share it:
// two calls whose kernels overlap on the GPU (different streams without an
// ordering between them) race on it.  Nothing in it needs clearing between
// calls: the count kernel overwrites every entry that the later kernels read.
#include <mutex>

#include "ep_common.cuh"
#include "ep_kernels.h"
#include "ep_trace.h"

namespace ep {
cudaError_t plan_ll(LaunchPlan* plan, int num_experts);
void record_error(const char* message);
}  // namespace ep

namespace {

constexpr int64_t kScratchCounts = EP_LL_NOALLOC_MAX_COUNTS;  // int32 entries, R * E at most

static __device__ __align__(256) int32_t g_ll_count_scratch[kScratchCounts];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    int32_t* scratch = nullptr;  // device address of g_ll_count_scratch on this device
    ep::LaunchPlan plan;
};

DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

ep_status reject(ep_status code, const char* message) {
    ep::record_error(message);
    return code;
}

// Once per device, with that device current: the scratch array's device
// address (host code only sees a host-side stand-in under its name) and the
// launch shapes of the kernels.
ep_status setup_device(int device, DeviceSetup** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[device];
    if (!s.ready) {
        int32_t* ptr = nullptr;
        cudaError_t err = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_ll_count_scratch);
        if (err != cudaSuccess) return reject(EP_ERR_CUDA, "cudaGetSymbolAddress of the low-latency count scratch failed");
        err = cudaDeviceGetAttribute(&s.plan.num_sms, cudaDevAttrMultiProcessorCount, device);
        if (err == cudaSuccess) err = ep::plan_ll(&s.plan, ep::kMaxExperts);
        if (err != cudaSuccess) return reject(EP_ERR_CUDA, "planning the low-latency launches failed");
        s.scratch = ptr;
        s.ready = true;
    }
    *out = &s;
    return EP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" ep_status ep_ll_dispatch_noalloc(int32_t num_ranks, int32_t num_tokens, int32_t num_max_tokens,
                                            int32_t hidden, int32_t num_experts, int32_t num_topk, const void* x,
                                            const int64_t* topk_idx, int32_t use_fp8, int32_t round_scale,
                                            int32_t use_ue8m0, void* recv_msgs, int32_t* packed_recv_count,
                                            int64_t* packed_recv_layout_range,
                                            int32_t* cumulative_local_expert_recv_stats, int32_t* slot_row,
                                            int32_t* status, ep_stream_t stream) {
    EP_TRACE();
    const int R = num_ranks, T = num_tokens, maxT = num_max_tokens, H = hidden, E = num_experts, K = num_topk;
    if (R < 1 || R > ep::kMaxRanks) return reject(EP_ERR_UNSUPPORTED, "num_ranks outside [1, 32]");
    if (E < 1 || E % R != 0 || E > ep::kMaxExperts)
        return reject(EP_ERR_INVALID_ARG, "num_experts must be a positive multiple of num_ranks, at most 2048");
    if (static_cast<int64_t>(R) * E > kScratchCounts)
        return reject(EP_ERR_UNSUPPORTED,
                      "num_ranks * num_experts exceeds the fixed count scratch of ep_ll_dispatch_noalloc "
                      "(EP_LL_NOALLOC_MAX_COUNTS entries); use ep_ll_dispatch with a handle");
    if (K < 1 || K > ep::kMaxTopk) return reject(EP_ERR_UNSUPPORTED, "num_topk outside [1, 32]");
    if (maxT < 0 || T < 0 || T > maxT) return reject(EP_ERR_INVALID_ARG, "num_tokens must lie in [0, num_max_tokens]");
    if (static_cast<int64_t>(R) * maxT > INT32_MAX || static_cast<int64_t>(maxT) * K > INT32_MAX)
        return reject(EP_ERR_UNSUPPORTED, "num_ranks * num_max_tokens or num_max_tokens * num_topk exceeds 2^31");
    if (H < 8 || H % 8 != 0) return reject(EP_ERR_INVALID_ARG, "hidden must be a positive multiple of 8");
    if (use_ue8m0 && !use_fp8) return reject(EP_ERR_INVALID_ARG, "use_ue8m0 needs use_fp8");
    if (use_fp8 && H % 512 != 0)
        return reject(EP_ERR_UNSUPPORTED, "FP8 low-latency messages need hidden % 512 == 0");
    if (T > 0 && (x == nullptr || !aligned(x, 16) || topk_idx == nullptr || !aligned(topk_idx, 8)))
        return reject(EP_ERR_INVALID_ARG, "x (16-byte aligned) and topk_idx are required");
    if (recv_msgs == nullptr || !aligned(recv_msgs, 16) || packed_recv_count == nullptr ||
        packed_recv_layout_range == nullptr || !aligned(packed_recv_layout_range, 8) || slot_row == nullptr ||
        status == nullptr || !aligned(status, 4) || !aligned(cumulative_local_expert_recv_stats, 4))
        return reject(EP_ERR_INVALID_ARG, "an output pointer is missing or misaligned");

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return reject(EP_ERR_CUDA, "no usable current CUDA device");
    DeviceSetup* s = nullptr;
    ep_status st = setup_device(device, &s);
    if (st != EP_OK) return st;
    cudaError_t err = ep::launch_ll_dispatch(s->plan, R, T, maxT, H, K, E, x, topk_idx, use_fp8 != 0,
                                             round_scale != 0, use_ue8m0 != 0, nullptr, slot_row, s->scratch,
                                             recv_msgs,
                                             packed_recv_count, packed_recv_layout_range,
                                             cumulative_local_expert_recv_stats, status, stream);
    if (err != cudaSuccess) return reject(EP_ERR_CUDA, cudaGetErrorString(err));
    return EP_OK;
}
