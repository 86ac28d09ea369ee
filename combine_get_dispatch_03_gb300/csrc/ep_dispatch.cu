// ep_dispatch.cu -- normal-mode dispatch and combine data movement.
//
// Dispatch ("第 4 章 V1：布局、dispatch 与 combine" §4.1): each source token
// row is read from HBM once and written to every destination rank that hosts
// one of its experts, at the row the notify kernel assigned (send_head).  In
// FP8 mode the per-128-channel amax, scale and e4m3 cast happen in registers
// between the read and the writes ("DeepEP Normal vs Low-Latency
// 双模式深度分析", low-latency dispatch excerpt: per-group amax, scale,
// inverse scale, cast).
//
// Combine (same chapter §4.2 and §4.4): each output token gathers the rows
// that its destination ranks hold, adds them in fp32 in ascending rank order
// after the two optional biases, and writes bf16 (or fp32) once; the top-k
// weights are summed separately over the same ranks.
//
// Both are HBM-bound permutations (about 0 flops per byte): a persistent
// grid of (SM count x resident CTAs), one warp per token, 16-byte vector
// accesses with several in flight per lane.
#include "ep_common.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kDispatchUnroll = 4;  // 16-byte vectors in flight per lane (payload read)
constexpr int kCombineUnroll = 2;   // 16-byte columns per lane per pass
// Source rows loaded together before accumulation: all of them up to 8 ranks (one batch), else
// batches of 4 (measured on the 7168-wide workloads: 452 against 460 us at R = 8, and 1351
// against 1399 us at R = 16, for the 8- and 4-row batches respectively).
constexpr int kCombineFanInSmallR = 8;
constexpr int kCombineFanIn = 4;
constexpr int kCombineWeightRanks = 8;  // source ranks whose top-k weights are loaded ahead of the rows
constexpr bool kUseBulkDispatch = true;  // bulk-copy (TMA 1D) dispatch where the rows fit in shared memory
// Shared memory for the stages of one CTA (bf16, cast, FP8 input).  The cast keeps the fewest
// stages (see bulk_stages) so that more CTAs -- and their cast work -- share an SM; measured on the
// 7168-wide workloads, with one round of the stages per CTA (a CTA takes at most `stages` tokens):
// 652 us for fp8_zipf with two stages against 692 us with three stages and two rounds.
constexpr uint32_t kBulkStageBudget[3] = {65536u, 45056u, 65536u};
constexpr int kBulkCastWarps = 4;  // warps of a cast CTA

// Row of rank `lane` for token g, or -1 (not sent / past capacity).
__device__ __forceinline__ int32_t dest_row(const int32_t* send_head, int64_t g, int R, int64_t cap, int lane) {
    int32_t row = -1;
    if (lane < R) {
        row = __ldg(send_head + g * R + lane);
        if (row >= cap) row = -1;
    }
    return row;
}

template <int kMode>
__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_kernel(int R, int T, int H, int K, int EL, int64_t cap, const void* __restrict__ x,
                    const float* __restrict__ x_scales, const int64_t* __restrict__ topk_idx,
                    const float* __restrict__ topk_weights, const int32_t* __restrict__ send_head,
                    void* __restrict__ recv_x, float* __restrict__ recv_x_scales,
                    int64_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_weights) {
    pdl_enter();
    constexpr int kWarps = kDispatchThreads / kWarpSize;
    const int lane = lane_id();
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int G = H / kFp8Group;

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + threadIdx.x / kWarpSize; g < n_tokens;
         g += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int32_t row = dest_row(send_head, g, R, cap, lane);
        const unsigned dst = __ballot_sync(kFullMask, row >= 0);
        if (dst == 0u) continue;

        // Top-k metadata of each destination.
        if (recv_topk_idx != nullptr || recv_topk_weights != nullptr) {
            int64_t e = -1;
            float w = 0.0f;
            if (lane < K) {
                e = __ldg(topk_idx + g * K + lane);
                if (topk_weights != nullptr) w = __ldg(topk_weights + g * K + lane);
            }
            for (unsigned m = dst; m; m &= m - 1) {
                const int r = __ffs(m) - 1;
                const int64_t rr = __shfl_sync(kFullMask, row, r);
                if (lane < K) {
                    const bool mine = e >= 0 && static_cast<int>(e) / EL == r;
                    const int64_t o = (static_cast<int64_t>(r) * cap + rr) * K + lane;
                    if (recv_topk_idx != nullptr) recv_topk_idx[o] = mine ? e % EL : -1;
                    if (recv_topk_weights != nullptr) recv_topk_weights[o] = mine ? w : 0.0f;
                }
            }
        }

        if constexpr (kMode == kModeBf16 || kMode == kModeFp8In) {
            // Byte copy of the row (bf16: 2H bytes; FP8 input: H bytes) plus FP8 scales.
            const int n16 = kMode == kModeBf16 ? H / 8 : H / 16;
            const int4* src = reinterpret_cast<const int4*>(x) + g * n16;
            int4* base = reinterpret_cast<int4*>(recv_x);
            for (int i0 = 0; i0 < n16; i0 += kWarpSize * kDispatchUnroll) {
                int4 v[kDispatchUnroll];
#pragma unroll
                for (int u = 0; u < kDispatchUnroll; ++u) {
                    const int i = i0 + u * kWarpSize + lane;
                    if (i < n16) v[u] = ld_stream_v4(src + i);
                }
                for (unsigned m = dst; m; m &= m - 1) {
                    const int r = __ffs(m) - 1;
                    const int64_t rr = __shfl_sync(kFullMask, row, r);
                    int4* d = base + (static_cast<int64_t>(r) * cap + rr) * n16;
#pragma unroll
                    for (int u = 0; u < kDispatchUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (i < n16) st_stream_v4(d + i, v[u]);
                    }
                }
            }
            if constexpr (kMode == kModeFp8In) {
                const float* ssrc = x_scales + g * G;
                for (unsigned m = dst; m; m &= m - 1) {
                    const int r = __ffs(m) - 1;
                    const int64_t rr = __shfl_sync(kFullMask, row, r);
                    float* d = recv_x_scales + (static_cast<int64_t>(r) * cap + rr) * G;
                    for (int i = lane; i < G; i += kWarpSize) d[i] = __ldg(ssrc + i);
                }
            }
        } else {
            // bf16 -> e4m3 with one fp32 scale per 128 channels.  Lane l of a
            // warp pass covers 8 channels; lanes 0-15 and 16-31 each hold one group.
            const int n16 = H / 8;
            const int4* src = reinterpret_cast<const int4*>(x) + g * n16;
            int2* base = reinterpret_cast<int2*>(recv_x);
            for (int i0 = 0; i0 < n16; i0 += kWarpSize * kDispatchUnroll) {
                int4 v[kDispatchUnroll];
#pragma unroll
                for (int u = 0; u < kDispatchUnroll; ++u) {
                    const int i = i0 + u * kWarpSize + lane;
                    v[u] = i < n16 ? ld_stream_v4(src + i) : make_int4(0, 0, 0, 0);
                }
                int2 q[kDispatchUnroll];
                float sc[kDispatchUnroll];
#pragma unroll
                for (int u = 0; u < kDispatchUnroll; ++u) {
                    float f[8];
                    unpack8(v[u], f);
                    float amax = absmax8(f);
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
                    const Fp8Scale fs = fp8_scale(amax, false);
                    q[u] = cast8_e4m3(f, fs.mult);
                    sc[u] = fs.scale;
                }
                for (unsigned m = dst; m; m &= m - 1) {
                    const int r = __ffs(m) - 1;
                    const int64_t rr = __shfl_sync(kFullMask, row, r);
                    const int64_t drow = static_cast<int64_t>(r) * cap + rr;
                    int2* d = base + drow * n16;
#pragma unroll
                    for (int u = 0; u < kDispatchUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (i < n16) {
                            st_stream_v2(d + i, q[u]);
                            if ((lane & 15) == 0) recv_x_scales[drow * G + i / 16] = sc[u];
                        }
                    }
                }
            }
        }
    }
}

// Bulk-copy dispatch: CTA b takes the contiguous tokens [b * per_cta, (b + 1) *
// per_cta) and walks them through `stages` shared-memory row buffers; the grid
// covers all tokens, so the rows in flight on the GPU stay a contiguous window
// of the token order (a grid-stride walk spreads them out as CTAs drift apart,
// and measured about 10 % slower on HBM).  Warp 0 lane 0 loads a row with
// one bulk copy (completion counted on the stage's mbarrier), all stages at
// the start, and writes it to every destination row with one bulk store each;
// the stores of token j form one bulk group, and a stage is refilled (only
// when a CTA has more tokens than stages) one token later, after its group has
// read it and a block barrier has ordered its metadata's last use.  In cast mode all warps of the
// CTA turn the staged bf16 row into e4m3 codes + fp32 scales in a second
// buffer first.  A wait that reaches its iteration cap reports
// EP_ERR_TIMEOUT, lets the loads already issued land, and leaves.
struct BulkSmem {
    uint32_t in_stride, out_stride, meta_bytes, total;
};

__host__ __device__ __forceinline__ uint32_t align128(uint32_t v) { return (v + 127u) & ~127u; }

__host__ __device__ __forceinline__ BulkSmem bulk_smem(int mode, int H, int stages) {
    BulkSmem b;
    const uint32_t in_bytes = mode == kModeFp8In ? H : 2 * H;
    b.in_stride = align128(in_bytes);
    b.out_stride = mode == kModeCastFp8 ? align128(H + 4 * (H / kFp8Group)) : 0;
    b.meta_bytes = align128(64 + stages * (32 * 4 + 32 * 8 + 32 * 4) + 16);
    b.total = b.meta_bytes + stages * (b.in_stride + b.out_stride);
    return b;
}

template <int kMode>
__global__ void dispatch_bulk_kernel(int R, int T, int H, int K, int EL, int64_t cap, int stages, int per_cta,
                                     bool scales_bulk,
                                     const uint8_t* __restrict__ x, const float* __restrict__ x_scales,
                                     const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_weights,
                                     const int32_t* __restrict__ send_head, uint8_t* __restrict__ recv_x,
                                     float* __restrict__ recv_x_scales, int64_t* __restrict__ recv_topk_idx,
                                     float* __restrict__ recv_topk_weights, int32_t* status) {
    pdl_enter();
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = stages;
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const bool warp0 = tid < kWarpSize;
    const int G = H / kFp8Group;
    const uint32_t in_bytes = kMode == kModeFp8In ? H : 2 * H;
    const uint32_t out_bytes = kMode == kModeBf16 ? 2 * H : H;  // payload bytes of one destination row
    const BulkSmem lay = bulk_smem(kMode, H, S);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                       // [S], S <= 8
    int32_t* s_row = reinterpret_cast<int32_t*>(smem + 64);                   // [S][32]
    int64_t* s_idx = reinterpret_cast<int64_t*>(smem + 64 + S * 128);         // [S][32]
    float* s_w = reinterpret_cast<float*>(smem + 64 + S * 384);               // [S][32]
    int32_t* s_flag = reinterpret_cast<int32_t*>(smem + 64 + S * 512);          // [2]
    uint8_t* in_base = smem + lay.meta_bytes;
    uint8_t* out_base = in_base + S * lay.in_stride;

    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t n_local = first < n_tokens ? (n_tokens - first < per_cta ? n_tokens - first : per_cta) : 0;
    if (n_local == 0) return;
    if (tid == 0) {
        // one arrival with the row's transaction bytes + one per warp-0 lane for its metadata copies
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1 + kWarpSize);
        fence_barrier_init();
    }
    __syncthreads();

    // Warp 0: start the copies of the token's destination rows, top-k slots and row;
    // all of them complete on the stage's barrier, so nothing here waits.
    auto produce = [&](int64_t j) {
        const int s = static_cast<int>(j % S);
        const int64_t g = first + j;
        if (lane < R) cp_async_4(&s_row[s * 32 + lane], send_head + g * R + lane);
        if (topk_idx != nullptr && lane < K) {
            cp_async_8(&s_idx[s * 32 + lane], topk_idx + g * K + lane);
            if (topk_weights != nullptr) cp_async_4(&s_w[s * 32 + lane], topk_weights + g * K + lane);
        }
        cp_async_arrive(&bars[s]);
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[s], in_bytes);
            bulk_load(in_base + s * lay.in_stride, x + g * in_bytes, in_bytes, &bars[s]);
        }
    };

    if (warp0) {
        const int64_t pro = n_local < S ? n_local : S;  // every stage starts full
        for (int64_t j = 0; j < pro; ++j) produce(j);
    }
    int64_t j = 0;
    for (; j < n_local; ++j) {
        const int s = static_cast<int>(j % S);
        // One flag per token parity: thread 0 may write token j+1's flag while a slower warp still
        // reads token j's, but not token j+2's before every warp has passed token j+1's barrier.
        if (tid == 0) s_flag[j & 1] = mbar_wait_bounded(&bars[s], static_cast<uint32_t>((j / S) & 1)) ? 1 : 0;
        __syncthreads();
        if (s_flag[j & 1] == 0) break;
        const uint8_t* payload = in_base + s * lay.in_stride;
        if constexpr (kMode == kModeCastFp8) {
            const int4* xin = reinterpret_cast<const int4*>(payload);
            uint8_t* qo = out_base + s * lay.out_stride;
            float* so = reinterpret_cast<float*>(qo + H);
            const int n16 = H / 8;
            for (int i0 = (tid / kWarpSize) * kWarpSize; i0 < n16; i0 += blockDim.x) {
                const int i = i0 + lane;
                float f[8];
                unpack8(i < n16 ? xin[i] : make_int4(0, 0, 0, 0), f);
                float amax = absmax8(f);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
                const Fp8Scale fs = fp8_scale(amax, false);
                if (i < n16) {
                    reinterpret_cast<int2*>(qo)[i] = cast8_e4m3(f, fs.mult);
                    if ((lane & 15) == 0) so[i / 16] = fs.scale;
                }
            }
            fence_async_smem();
            __syncthreads();
            payload = qo;
        }
        // Top-k metadata and FP8 scales of every destination: warp 1 when the CTA has
        // several warps (it then runs beside warp 0's stores and refill), else warp 0.
        const int meta_warp = blockDim.x > kWarpSize ? 1 : 0;
        if (tid / kWarpSize == meta_warp) {
            int32_t row = lane < R ? s_row[s * 32 + lane] : -1;
            if (row >= cap) row = -1;
            const unsigned dst = __ballot_sync(kFullMask, row >= 0);
            const int64_t g = first + j;
            int e = -1;
            float w = 0.0f;
            if (lane < K && topk_idx != nullptr) {
                e = static_cast<int>(s_idx[s * 32 + lane]);
                if (topk_weights != nullptr) w = s_w[s * 32 + lane];
            }
            for (unsigned m = dst; m; m &= m - 1) {
                const int r = __ffs(m) - 1;
                const int64_t drow = static_cast<int64_t>(r) * cap + s_row[s * 32 + r];
                if ((recv_topk_idx != nullptr || recv_topk_weights != nullptr) && lane < K) {
                    const bool mine = e >= 0 && e / EL == r;
                    if (recv_topk_idx != nullptr) recv_topk_idx[drow * K + lane] = mine ? e % EL : -1;
                    if (recv_topk_weights != nullptr) recv_topk_weights[drow * K + lane] = mine ? w : 0.0f;
                }
                if (kMode == kModeFp8In)
                    for (int i = lane; i < G; i += kWarpSize) recv_x_scales[drow * G + i] = __ldg(x_scales + g * G + i);
                if (kMode == kModeCastFp8 && !scales_bulk) {
                    const float* so = reinterpret_cast<const float*>(payload + H);
                    for (int i = lane; i < G; i += kWarpSize) recv_x_scales[drow * G + i] = so[i];
                }
            }
        }
        if (warp0) {
            int32_t row = lane < R ? s_row[s * 32 + lane] : -1;
            if (row >= cap) row = -1;
            const unsigned dst = __ballot_sync(kFullMask, row >= 0);
            if (lane == 0) {
                for (unsigned m = dst; m; m &= m - 1) {
                    const int r = __ffs(m) - 1;
                    const int64_t drow = static_cast<int64_t>(r) * cap + s_row[s * 32 + r];
                    bulk_store(recv_x + drow * out_bytes, payload, out_bytes);
                    if (kMode == kModeCastFp8 && scales_bulk)
                        bulk_store(recv_x_scales + drow * G, payload + H, 4 * G);
                }
                bulk_commit();
            }
            // Refill the stage that token j-1 used with token j-1+S, once its stores have read
            // it; its metadata was read before this iteration's block barrier.  (A CTA takes at
            // most S tokens unless max_sms caps the grid, so this is rare.)
            if (j >= 1 && j - 1 + S < n_local) {
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                produce(j - 1 + S);
            }
        }
    }
    if (j < n_local && tid == 0) {
        report(status, EP_ERR_TIMEOUT);
        // Let the row loads already issued land before this CTA's shared memory is released.
        const int64_t last = j + S - 1 > S ? j + S - 1 : S;  // tokens loaded so far
        const int64_t issued = last < n_local ? last : n_local;
        for (int64_t k = j + 1; k < issued; ++k) mbar_wait_bounded(&bars[k % S], static_cast<uint32_t>((k / S) & 1));
    }
    if (tid == 0) bulk_wait_all();
}

template <bool kOutF32, int kFanIn>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(int R, int T, int H, int K, int64_t cap, const int32_t* __restrict__ send_head,
                   const int4* __restrict__ y, const float* __restrict__ recv_w, const int4* __restrict__ bias0,
                   const int4* __restrict__ bias1, void* __restrict__ out, float* __restrict__ cw,
                   uint32_t* __restrict__ work) {
    pdl_enter();
    constexpr int kWarps = kCombineThreads / kWarpSize;
    const int lane = lane_id();
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int n16 = H / 8;

    // With work != nullptr, tokens are claimed one at a time from a counter shared by every warp
    // (work[0]), so warps whose tokens hit fewer ranks take more tokens and all finish together
    // (a token's cost is its number of source rows); the last warp to finish (work[1]) resets
    // both counters for the next launch.  Without it (about one token per warp) the warps stride
    // over the tokens.  Either way the next token and its send_head row are fetched one ahead.
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    auto claim = [&]() -> int64_t {
        uint32_t v = 0;
        if (lane == 0) v = atomicAdd(work, 1u);
        return static_cast<int64_t>(__shfl_sync(kFullMask, v, 0));
    };
    int64_t g = work != nullptr ? claim() : static_cast<int64_t>(blockIdx.x) * kWarps + threadIdx.x / kWarpSize;
    int32_t next_row = g < n_tokens ? dest_row(send_head, g, R, cap, lane) : -1;
    while (g < n_tokens) {
        const int32_t row = next_row;
        const int64_t g_next = work != nullptr ? claim() : g + stride;
        if (g_next < n_tokens) next_row = dest_row(send_head, g_next, R, cap, lane);
        const unsigned src_ranks = __ballot_sync(kFullMask, row >= 0);

        // Top-k weights of the first kCombineWeightRanks source ranks: loaded now, summed (in
        // rank order) after the rows, so their latency hides behind the row loads.
        const bool with_w = cw != nullptr && recv_w != nullptr;
        float wv[kCombineWeightRanks];
        unsigned w_left = src_ranks;
        if (with_w) {
#pragma unroll
            for (int j = 0; j < kCombineWeightRanks; ++j) {
                const int r = w_left ? __ffs(w_left) - 1 : 0;
                const int64_t rr = __shfl_sync(kFullMask, row, r);
                wv[j] = (w_left && lane < K) ? __ldg(recv_w + (static_cast<int64_t>(r) * cap + rr) * K + lane) : 0.0f;
                if (w_left) w_left &= w_left - 1;
            }
        }

        for (int i0 = 0; i0 < n16; i0 += kWarpSize * kCombineUnroll) {
            float acc[kCombineUnroll][8];
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u) {
                const int i = i0 + u * kWarpSize + lane;
                float f0[8], f1[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) f0[q] = f1[q] = 0.0f;
                if (i < n16) {
                    if (bias0 != nullptr) unpack8(ld_stream_v4(bias0 + g * n16 + i), f0);
                    if (bias1 != nullptr) unpack8(ld_stream_v4(bias1 + g * n16 + i), f1);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[u][q] = __fadd_rn(f0[q], f1[q]);
            }
            unsigned m = src_ranks;
            while (m) {
                int rk[kFanIn];
                int64_t rr[kFanIn];
#pragma unroll
                for (int j = 0; j < kFanIn; ++j) {
                    rk[j] = m ? __ffs(m) - 1 : -1;
                    if (m) m &= m - 1;
                    rr[j] = __shfl_sync(kFullMask, row, rk[j] < 0 ? 0 : rk[j]);
                }
                int4 v[kFanIn][kCombineUnroll];
#pragma unroll
                for (int j = 0; j < kFanIn; ++j)
#pragma unroll
                    for (int u = 0; u < kCombineUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (rk[j] >= 0 && i < n16)
                            v[j][u] = ld_stream_v4(y + (static_cast<int64_t>(rk[j]) * cap + rr[j]) * n16 + i);
                    }
#pragma unroll
                for (int j = 0; j < kFanIn; ++j) {
                    if (rk[j] < 0) continue;
#pragma unroll
                    for (int u = 0; u < kCombineUnroll; ++u) {
                        float f[8];
                        unpack8(v[j][u], f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[u][q] = __fadd_rn(acc[u][q], f[q]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kCombineUnroll; ++u) {
                const int i = i0 + u * kWarpSize + lane;
                if (i >= n16) continue;
                if constexpr (kOutF32) {
                    float4* o = reinterpret_cast<float4*>(out) + (g * n16 + i) * 2;
                    o[0] = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
                    o[1] = make_float4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
                } else {
                    reinterpret_cast<int4*>(out)[g * n16 + i] = pack8_bf16(acc[u]);
                }
            }
        }

        if (with_w) {
            float acc = 0.0f;
            const int nw = __popc(src_ranks);
#pragma unroll
            for (int j = 0; j < kCombineWeightRanks; ++j)
                if (j < nw) acc = acc + wv[j];
            for (unsigned m = w_left; m; m &= m - 1) {  // ranks past the first kCombineWeightRanks
                const int r = __ffs(m) - 1;
                const int64_t rr = __shfl_sync(kFullMask, row, r);
                if (lane < K) acc = acc + __ldg(recv_w + (static_cast<int64_t>(r) * cap + rr) * K + lane);
            }
            if (lane < K) cw[g * K + lane] = acc;
        }
        g = g_next;
    }
    if (work != nullptr && lane == 0) {
        __threadfence();  // this warp's claims come before its count of finished warps
        if (atomicAdd(work + 1, 1u) == static_cast<uint32_t>(gridDim.x) * kWarps - 1u) {
            atomicExch(work, 0u);
            atomicExch(work + 1, 0u);
        }
    }
}

template <typename Kernel>
int resident_blocks(Kernel k, int threads, int num_sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return per_sm * num_sms;
}

int clamp_grid(int planned, int64_t warps_needed, int warps_per_block) {
    const int64_t need = (warps_needed + warps_per_block - 1) / warps_per_block;
    return static_cast<int>(need < planned ? (need > 0 ? need : 1) : planned);
}

}  // namespace

int bulk_stages(int mode, int H, bool sm_limited) {
    // The cast: one stage (the bf16 row and its codes + scales, 22 KB at 7168 channels), so 9 CTAs share
    // an SM (fp8_zipf: 636.2 against 638.7 us with two stages; the low-latency FP8 dispatch gained the
    // same way) -- unless max_sms caps the grid: a CTA then takes more tokens than it has stages, and
    // the refill of token j-1's stage at token j needs two.  Otherwise kBulkStageBudget[mode] bytes of
    // row buffers per CTA, between 2 and 8 stages.
    if (mode == kModeCastFp8 && !sm_limited) return 1;
    const uint32_t per = bulk_smem(mode, H, 1).in_stride + bulk_smem(mode, H, 1).out_stride;
    int s = static_cast<int>(kBulkStageBudget[mode] / per);
    return s < 2 ? 2 : (s > 8 ? 8 : s);
}

// FP8 input: a second warp writes the top-k metadata and the copied scales beside warp 0's row
// stores (measured on fp8_zipf: 563 -> 541 us).  bf16 rows keep one warp: with twice the bytes
// per row the metadata hides behind the stores (two warps measured 0.4 % slower).
int bulk_threads(int mode) {
    return mode == kModeCastFp8 ? kBulkCastWarps * kWarpSize : (mode == kModeFp8In ? 2 * kWarpSize : kWarpSize);
}

template <int kMode>
cudaError_t plan_bulk(LaunchPlan* plan, int H) {
    const int S = bulk_stages(kMode, H, plan->sm_limited);
    const uint32_t smem = bulk_smem(kMode, H, S).total;
    plan->bulk_stages[kMode] = 0;
    if (smem > 200u * 1024u) return cudaSuccess;  // rows too long to stage: the register kernel is used
    cudaError_t err = cudaFuncSetAttribute(dispatch_bulk_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_bulk_kernel<kMode>, bulk_threads(kMode), smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaSuccess;
    plan->bulk_stages[kMode] = S;
    plan->bulk_smem[kMode] = smem;
    plan->bulk_resident[kMode] = per_sm * plan->num_sms;
    return cudaSuccess;
}

cudaError_t plan_dispatch_combine(LaunchPlan* plan, int H) {
    const int n = plan->num_sms;
    cudaError_t err = plan_bulk<kModeBf16>(plan, H);
    if (err == cudaSuccess && H % kFp8Group == 0) err = plan_bulk<kModeCastFp8>(plan, H);
    if (err == cudaSuccess && H % kFp8Group == 0) err = plan_bulk<kModeFp8In>(plan, H);
    if (err != cudaSuccess) return err;
    plan->dispatch_blocks[kModeBf16] = resident_blocks(dispatch_kernel<kModeBf16>, kDispatchThreads, n);
    plan->dispatch_blocks[kModeCastFp8] = resident_blocks(dispatch_kernel<kModeCastFp8>, kDispatchThreads, n);
    plan->dispatch_blocks[kModeFp8In] = resident_blocks(dispatch_kernel<kModeFp8In>, kDispatchThreads, n);
    plan->combine_blocks[0] = resident_blocks(combine_kernel<false, kCombineFanIn>, kCombineThreads, n);
    plan->combine_blocks[1] = resident_blocks(combine_kernel<true, kCombineFanIn>, kCombineThreads, n);
    plan->combine_blocks[2] = resident_blocks(combine_kernel<false, kCombineFanInSmallR>, kCombineThreads, n);
    plan->combine_blocks[3] = resident_blocks(combine_kernel<true, kCombineFanInSmallR>, kCombineThreads, n);
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const LaunchPlan& plan, int mode, int R, int T, int H, int K, int EL, int64_t cap,
                            const void* x, const float* x_scales, const int64_t* topk_idx,
                            const float* topk_weights, const int32_t* send_head, void* recv_x,
                            float* recv_x_scales, int64_t* recv_topk_idx, float* recv_topk_weights,
                            int32_t* status, cudaStream_t stream) {
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    if (n_tokens == 0) return cudaSuccess;
    if (kUseBulkDispatch && plan.bulk_stages[mode] > 0) {
        const int S = plan.bulk_stages[mode];
        // contiguous token blocks: enough CTAs to fill the GPU once, at most one round of the stages
        const int64_t fill = (n_tokens + plan.bulk_resident[mode] - 1) / plan.bulk_resident[mode];
        // (with max_sms, one resident wave takes all tokens)
        const int cap_cta = plan.sm_limited ? INT32_MAX : S;
        const int per_cta = static_cast<int>(fill < 1 ? 1 : (fill > cap_cta ? cap_cta : fill));
        if (S < 2 && per_cta > 1) return cudaErrorInvalidValue;  // the refill of a stage needs two stages
        const int grid = static_cast<int>((n_tokens + per_cta - 1) / per_cta);
        const uint32_t smem = plan.bulk_smem[mode];
        const int threads = bulk_threads(mode);
        const int G = H / kFp8Group;
        const bool scales_bulk = (G % 4 == 0) && ((reinterpret_cast<uintptr_t>(recv_x_scales) & 15u) == 0);
        const uint8_t* xb = static_cast<const uint8_t*>(x);
        uint8_t* rb = static_cast<uint8_t*>(recv_x);
        auto kernel = mode == kModeBf16 ? dispatch_bulk_kernel<kModeBf16>
                      : mode == kModeCastFp8 ? dispatch_bulk_kernel<kModeCastFp8>
                                             : dispatch_bulk_kernel<kModeFp8In>;
        return launch_kernel(kernel, dim3(grid), dim3(threads), smem, stream, 1, R, T, H, K, EL, cap, S, per_cta,
                             scales_bulk, xb, x_scales, topk_idx, topk_weights, send_head, rb, recv_x_scales,
                             recv_topk_idx, recv_topk_weights, status);
    }
    const int grid = clamp_grid(plan.dispatch_blocks[mode], n_tokens, kDispatchThreads / kWarpSize);
    auto kernel = mode == kModeBf16 ? dispatch_kernel<kModeBf16>
                  : mode == kModeCastFp8 ? dispatch_kernel<kModeCastFp8>
                                         : dispatch_kernel<kModeFp8In>;
    return launch_kernel(kernel, dim3(grid), dim3(kDispatchThreads), 0, stream, 1, R, T, H, K, EL, cap, x, x_scales,
                         topk_idx, topk_weights, send_head, recv_x, recv_x_scales, recv_topk_idx, recv_topk_weights);
}

cudaError_t launch_combine(const LaunchPlan& plan, bool out_fp32, int R, int T, int H, int K, int64_t cap,
                           const int32_t* send_head, const void* y, const float* recv_topk_weights,
                           const void* bias0, const void* bias1, void* out, float* combined_topk_weights,
                           uint32_t* work, cudaStream_t stream) {
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    if (n_tokens == 0) return cudaSuccess;
    const bool small_r = R <= kCombineFanInSmallR;
    const int grid = clamp_grid(plan.combine_blocks[(out_fp32 ? 1 : 0) + (small_r ? 2 : 0)], n_tokens,
                                kCombineThreads / kWarpSize);
    const int4* yv = static_cast<const int4*>(y);
    const int4* b0 = static_cast<const int4*>(bias0);
    const int4* b1 = static_cast<const int4*>(bias1);
    auto kernel = small_r ? (out_fp32 ? combine_kernel<true, kCombineFanInSmallR>
                                      : combine_kernel<false, kCombineFanInSmallR>)
                          : (out_fp32 ? combine_kernel<true, kCombineFanIn> : combine_kernel<false, kCombineFanIn>);
    // Claimed tokens once there are two or more per warp: on normal_v3 the combine went from 450.0 to
    // 444.8 us, and combine_heavy from 1351 to 1338 us.  With about one token per warp the claims are
    // pure latency (+4 us on the L2-resident normal_small step), so the warps stride instead.
    const int64_t warps = static_cast<int64_t>(grid) * (kCombineThreads / kWarpSize);
    uint32_t* claims = n_tokens >= 2 * warps ? work : nullptr;
    return launch_kernel(kernel, dim3(grid), dim3(kCombineThreads), 0, stream, 1, R, T, H, K, cap, send_head, yv,
                         recv_topk_weights, b0, b1, out, combined_topk_weights, claims);
}

}  // namespace ep
