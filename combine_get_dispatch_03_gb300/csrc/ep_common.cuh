// ep_common.cuh -- device helpers shared by the EP kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep.h"

namespace ep {

constexpr int kWarpSize = 32;
constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMaxRanks = 32;
constexpr int kMaxTopk = 32;
constexpr int kMaxExperts = 2048;
constexpr int kFp8Group = 128;

// First device-detected error wins; the host reads the word through ep_handle_status().
__device__ __forceinline__ void report(int32_t* status, ep_status code) {
    atomicCAS(status, 0, static_cast<int32_t>(code));
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & (kWarpSize - 1); }

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 16-byte read of data that no thread writes during the kernel; no L1 allocation.
__device__ __forceinline__ int4 ld_stream_v4(const int4* p) {
    int4 v;
    asm("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte store that is not kept in L1.
__device__ __forceinline__ void st_stream_v4(int4* p, const int4& v) {
    asm volatile("st.global.L1::no_allocate.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream_v2(int2* p, const int2& v) {
    asm volatile("st.global.L1::no_allocate.v2.s32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// bf16 pair packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const int4& v, float (&f)[8]) {
    const uint32_t w[4] = {static_cast<uint32_t>(v.x), static_cast<uint32_t>(v.y), static_cast<uint32_t>(v.z),
                           static_cast<uint32_t>(v.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
}

// Eight floats -> eight bf16 (round to nearest even) packed in 16 bytes.
__device__ __forceinline__ int4 pack8_bf16(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // .x = low half
        w[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return make_int4(static_cast<int>(w[0]), static_cast<int>(w[1]), static_cast<int>(w[2]),
                     static_cast<int>(w[3]));
}

// Two floats -> two e4m3 codes (round to nearest even, saturate to +-448); `a` in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Per-128-channel FP8 scale of one group whose |x| maximum is `amax_raw`.
//   amax = max(amax_raw, 1e-4); s = amax / 448 (IEEE division)
//   round_scale == false: scale = s,   multiplier = 448 / amax (IEEE division)
//   round_scale == true:  e = smallest integer with 2^e >= s, read off the
//                         bits of s; scale = 2^e, multiplier = 2^-e
struct Fp8Scale {
    float scale;
    float mult;
    int exponent;
};

__device__ __forceinline__ Fp8Scale fp8_scale(float amax_raw, bool round_scale) {
    const float amax = fmaxf(amax_raw, 1e-4f);
    const float s = __fdiv_rn(amax, 448.0f);
    Fp8Scale r;
    if (!round_scale) {
        r.scale = s;
        r.mult = __fdiv_rn(448.0f, amax);
        r.exponent = 0;
    } else {
        // s is a positive normal binary32 (s >= 1e-4/448 > 2^-126).
        const uint32_t u = __float_as_uint(s);
        const int biased = static_cast<int>(u >> 23);
        const int e = (u & 0x7fffffu) ? biased - 126 : biased - 127;
        r.exponent = e;
        r.scale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        r.mult = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    }
    return r;
}

// Eight bf16 (one int4) times `mult`, cast to eight e4m3 codes (8 bytes).
__device__ __forceinline__ int2 cast8_e4m3(const float (&f)[8], float mult) {
    uint32_t lo = static_cast<uint32_t>(e4m3x2(__fmul_rn(f[0], mult), __fmul_rn(f[1], mult))) |
                  (static_cast<uint32_t>(e4m3x2(__fmul_rn(f[2], mult), __fmul_rn(f[3], mult))) << 16);
    uint32_t hi = static_cast<uint32_t>(e4m3x2(__fmul_rn(f[4], mult), __fmul_rn(f[5], mult))) |
                  (static_cast<uint32_t>(e4m3x2(__fmul_rn(f[6], mult), __fmul_rn(f[7], mult))) << 16);
    return make_int2(static_cast<int>(lo), static_cast<int>(hi));
}

__device__ __forceinline__ float absmax8(const float (&f)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return m;
}

}  // namespace ep

// ---------------------------------------------------------------------------
// Bulk (1D TMA) copies and mbarriers, written out in PTX.
// ---------------------------------------------------------------------------
namespace ep {

// Iteration cap of every mbarrier wait; a wait that reaches it reports
// EP_ERR_TIMEOUT instead of spinning on (each try_wait may itself suspend).
constexpr uint32_t kMaxWaitIterations = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(arrivals) : "memory");
}

// Make initialised barriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity; false if the cap was reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t max_iterations = kMaxWaitIterations) {
    for (uint32_t it = 0; it < max_iterations; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// global -> shared bulk copy completing `bytes` of transaction on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst_smem)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// shared -> global bulk copy in the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic shared-memory writes before later bulk copies read them.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Per-thread asynchronous global -> shared copies of 4 or 8 bytes (naturally aligned).
__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_8(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have landed.  The
// arrival is not added to the barrier's expected count: initialise the barrier for it.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Acquire load / release store of one word in global memory, at GPU scope: the flags through
// which CTAs of one launch publish results to one another.
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation, so it may be scheduled while the previous
// kernel on the stream is still running; it therefore waits for that kernel's
// completion (and memory flush) before touching any global memory, then lets
// the next kernel be scheduled.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warm passes.  A kernel launched early sits at its grid-dependency wait while the previous kernel
// runs.  After a call's stream of stores has gone through L2 its code is cold: the first block
// after the wait took 1000-1900 SM cycles in the low-latency count kernel (clock64 stamps), about
// 450 once its code was cached.  A kernel whose body runs twice -- pass 0 before the wait with every global load and
// store switched off and its loops cut short, pass 1 after the wait for real -- fetches that code
// while it would otherwise only wait.  Only short single-wave kernels use it: in a grid of many
// waves every later CTA would pay for a pass 0 of its own.  The pass count is opaque to the
// compiler so that both passes run one copy of the body.
__device__ __forceinline__ int warm_passes() {
    int n = 2;
    asm volatile("" : "+r"(n));
    return n;
}

// Launch `kernel` with programmatic stream serialisation (and a 1-D cluster when cluster_x > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ep
