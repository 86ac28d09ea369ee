// ep_ll.cu -- low-latency (LL) dispatch and combine.
//
// LL dispatch ("DeepEP Normal vs Low-Latency 双模式深度分析", low-latency
// dispatch and receive-layout excerpts; "Normal vs Low-Latency: 双通信哲学在
// DeepEP V1/V2/DeepGEMM 中的三系统比较", message package; "第 4 章 V1：布局、
// dispatch 与 combine" §4.3): every valid top-k slot (s, t, k) becomes one
// message -- 16-byte header {t, 0, 0, 0}, payload, FP8 scales -- in the receive
// rows of its expert e: recv_msgs[e][row] with e = d*EL + j.  The pages take a
// slot with an atomicAdd on a per-expert counter, whose order depends on
// timing; here the rows are fixed beforehand so the layout is deterministic:
//   1. ll_count (one CTA per source rank): stable rank of each slot among the
//      slots of the same (source, expert), in (token, k) order, and the count;
//   2. ll_finish: begin of each source block = prefix over sources (one warp
//      per expert); packed_recv_count, packed_recv_layout_range, receive
//      stats; and the final row of every slot, which stays in the handle for
//      the combine;
//   3. ll_dispatch: read + cast the row once into a complete message in
//      shared memory, then one bulk store per destination slot (a register
//      kernel, one warp per token, serves messages too long to stage).
// LL combine (§4.3): one warp per token gathers its K expert outputs and
// accumulates w_k * y in fp32 with fused multiply-adds in slot order.  The
// expert-output rows may be strided (row stride >= 2H bytes): the bf16
// payloads of the dispatch messages themselves, written over in place by the
// experts, serve as the combine input with no copy (the zero-copy combine
// buffer of §4.3).
#include "ep_common.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kLLCountThreadsLarge = 1024;  // the count kernel's block while its histograms fit in smem
constexpr int kFinishThreads = 256;
constexpr int kLLUnroll = 4;
constexpr int kLLCombineUnroll = 2;
constexpr int kLLCombineFanIn = 4;         // slots loaded together before accumulation
constexpr int kLLCombineFanInSmallK = 8;   // ... with top-k up to 8: every slot in one batch

template <int kThreads>
__global__ void __launch_bounds__(kThreads)
    ll_count_kernel(int R, int T, int maxT, int K, int E, const int64_t* __restrict__ topk_idx,
                    const int32_t* __restrict__ rank_mask, int32_t* __restrict__ slot, int32_t* __restrict__ cnt,
                    int32_t* status) {
    constexpr int kWarps = kThreads / kWarpSize;
    constexpr int kScanChunk = kWarps < 16 ? kWarps : 16;
    static_assert(kWarps % kScanChunk == 0, "whole scan chunks");
    extern __shared__ __align__(16) int32_t smem[];
    int32_t* s_warp = smem;                   // [kWarps][E]: per-warp count -> exclusive prefix
    int32_t* s_run = smem + kWarps * E;  // [E]: slots of this source seen so far
    const int s = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int warp = tid / kWarpSize;
    const int n = T * K;
    const int64_t* idx_s = topk_idx + static_cast<int64_t>(s) * T * K;
    int32_t* slot_s = slot + static_cast<int64_t>(s) * maxT * K;

    __shared__ int32_t s_mask[kMaxRanks];  // rank mask (0 everywhere without one)
    const bool any_mask = rank_mask != nullptr;
    const int EL = E / R;
    // a warm pass first (see warm_passes): no global access, one chunk
    const int passes = warm_passes();
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        const bool live = pass == passes - 1;  // the pass after the grid-dependency wait
        if (live) pdl_enter();
        const int n_pass = live ? n : (n < kThreads ? n : kThreads);
        for (int e = tid; e < E; e += kThreads) s_run[e] = 0;
        if (tid < kMaxRanks) s_mask[tid] = live && rank_mask != nullptr && tid < R ? __ldg(rank_mask + tid) : 0;
        int64_t next = live && tid < n ? __ldg(idx_s + tid) : -1;  // the next chunk's entry, loaded one chunk ahead
        for (int base = 0; base < n_pass; base += kThreads) {
            for (int i = tid; i < kWarps * E / 4; i += kThreads)  // kWarps * E is a multiple of 4
                reinterpret_cast<int4*>(s_warp)[i] = make_int4(0, 0, 0, 0);
            __syncthreads();
            const int i = base + tid;
            const int64_t v = next;
            if (live && base + kThreads + tid < n) next = __ldg(idx_s + base + kThreads + tid);
            int e = -1;
            if (i < n) {
                if (v >= 0 && v < E) e = static_cast<int>(v);
                else if (v != -1 && live) report(status, EP_ERR_BAD_EXPERT);
                // a masked rank neither sends nor receives
                if (e >= 0 && any_mask && (s_mask[s] != 0 || s_mask[e / EL] != 0)) e = -1;
            }
            const unsigned peers = __match_any_sync(kFullMask, e);
            const int before = __popc(peers & lanemask_lt());
            if (e >= 0 && before == 0) s_warp[warp * E + e] = __popc(peers);
            __syncthreads();
            // per expert: exclusive prefix over the warps, in chunks of 16 whose loads are all issued
            // before the stores (a load after a store to the same array would wait for it)
            for (int x = tid; x < E; x += kThreads) {
                int32_t run = s_run[x];
#pragma unroll
                for (int w0 = 0; w0 < kWarps; w0 += kScanChunk) {
                    int32_t c[kScanChunk];
#pragma unroll
                    for (int u = 0; u < kScanChunk; ++u) c[u] = s_warp[(w0 + u) * E + x];
#pragma unroll
                    for (int u = 0; u < kScanChunk; ++u) {
                        s_warp[(w0 + u) * E + x] = run;
                        run += c[u];
                    }
                }
                s_run[x] = run;
            }
            __syncthreads();
            if (live && i < n) slot_s[i] = e >= 0 ? s_warp[warp * E + e] + before : -1;
            __syncthreads();
        }
        if (live)
            for (int e = tid; e < E; e += kThreads) cnt[static_cast<int64_t>(s) * E + e] = s_run[e];
        __syncthreads();  // shared memory is rewritten by the next pass
    }
}

// One pass of ll_finish_kernel; `live` false: no global access (the warm pass).
__device__ __forceinline__ void ll_finish_pass(bool live, int R, int T, int maxT, int K, int E, int expert_blocks,
                                               const int64_t* __restrict__ topk_idx, const int32_t* __restrict__ cnt,
                                               int32_t* __restrict__ slot, int32_t* __restrict__ packed_recv_count,
                                               int64_t* __restrict__ layout_range, int32_t* __restrict__ stats,
                                               int32_t* status, int32_t* s_begin) {
    const int64_t slots = static_cast<int64_t>(R) * maxT;
    if (static_cast<int>(blockIdx.x) < expert_blocks) {
        const int lane = lane_id();
        const int warps = blockDim.x / kWarpSize;
        const int e = blockIdx.x * warps + threadIdx.x / kWarpSize;
        if (e >= E) return;
        const int32_t c = live && lane < R ? __ldg(cnt + static_cast<int64_t>(lane) * E + e) : 0;
        int32_t incl = c;
#pragma unroll
        for (int off = 1; off < kWarpSize; off <<= 1) {
            const int32_t o = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off) incl += o;
        }
        const int32_t begin = incl - c;
        if (live && lane < R)
            layout_range[static_cast<int64_t>(e) * R + lane] =
                static_cast<int64_t>((static_cast<uint64_t>(static_cast<uint32_t>(c)) << 32) |
                                     static_cast<uint32_t>(begin));
        const int32_t total = __shfl_sync(kFullMask, incl, kWarpSize - 1);
        if (live && lane == 0) {
            if (total > slots) report(status, EP_ERR_CAPACITY);
            const int32_t n = static_cast<int32_t>(total < slots ? total : slots);
            packed_recv_count[e] = n;
            if (stats != nullptr) stats[e] += n;
        }
        return;
    }
    const int64_t n_slots = static_cast<int64_t>(R) * T * K;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x - expert_blocks) * blockDim.x;
    const int64_t i = i0 + threadIdx.x;
    // With E <= blockDim and every slot of the CTA from one source, the CTA sums the begins of
    // that source's blocks for all experts into shared memory while its slots' expert ids and
    // positions load: loads that need no expert id, so a slot waits for one round of loads
    // instead of two.
    const int64_t i_last = (i0 + blockDim.x < n_slots ? i0 + blockDim.x : n_slots) - 1;
    const int s_first = static_cast<int>(i0 / (static_cast<int64_t>(T) * K));
    const bool table = E <= static_cast<int>(blockDim.x) && i0 < n_slots &&
                       s_first == static_cast<int>(i_last / (static_cast<int64_t>(T) * K));
    const bool active = i < n_slots;
    int s = 0;
    int64_t v = -1;
    int32_t pos = -1;
    int32_t* sp = nullptr;
    if (active) {
        s = static_cast<int>(i / (static_cast<int64_t>(T) * K));
        sp = slot + static_cast<int64_t>(s) * maxT * K + (i - static_cast<int64_t>(s) * T * K);
        if (live) {
            v = __ldg(topk_idx + i);
            pos = *sp;
        }
    }
    if (table) {
        const int e = threadIdx.x;
        if (e < E) {
            int32_t part[kMaxRanks];
#pragma unroll
            for (int q = 0; q < kMaxRanks; ++q)
                part[q] = live && q < s_first ? __ldg(cnt + static_cast<int64_t>(q) * E + e) : 0;
            int32_t b = 0;
#pragma unroll
            for (int q = 0; q < kMaxRanks; ++q) b += part[q];
            s_begin[e] = b;
        }
        __syncthreads();
    }
    if (!active) return;
    int32_t row = -1;
    if (v >= 0 && v < E && pos >= 0) {
        int64_t begin = 0;
        if (table) {
            begin = s_begin[v];
        } else {
            // the counts of the earlier sources, all loads in flight at once (R <= kMaxRanks)
            int32_t part[kMaxRanks];
#pragma unroll
            for (int sp2 = 0; sp2 < kMaxRanks; ++sp2)
                part[sp2] = sp2 < s ? __ldg(cnt + static_cast<int64_t>(sp2) * E + v) : 0;
#pragma unroll
            for (int sp2 = 0; sp2 < kMaxRanks; ++sp2) begin += part[sp2];
        }
        if (begin + pos < slots) row = static_cast<int32_t>(begin + pos);
    }
    if (live) *sp = row;
}

// Blocks [0, expert_blocks): one warp per expert e; lane s holds the count of
// source s, a warp scan gives each source block's begin (R <= 32).  The other
// blocks: one thread per top-k slot turns its position within (source, expert)
// into the final row, begin(e, s) + position, or -1 past the R * maxT capacity.
// A warm pass first (see warm_passes).
__global__ void ll_finish_kernel(int R, int T, int maxT, int K, int E, int expert_blocks,
                                 const int64_t* __restrict__ topk_idx, const int32_t* __restrict__ cnt,
                                 int32_t* __restrict__ slot, int32_t* __restrict__ packed_recv_count,
                                 int64_t* __restrict__ layout_range, int32_t* __restrict__ stats, int32_t* status) {
    __shared__ int32_t s_begin[kFinishThreads];
    const int passes = warm_passes();
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        const bool live = pass == passes - 1;
        if (live) pdl_enter();
        ll_finish_pass(live, R, T, maxT, K, E, expert_blocks, topk_idx, cnt, slot, packed_recv_count, layout_range,
                       stats, status, s_begin);
        __syncthreads();  // s_begin is rewritten by the next pass
    }
}

// Bulk-copy low-latency dispatch: CTA b takes the contiguous tokens [b * per_cta,
// (b + 1) * per_cta) -- the grid covers all tokens, so the messages in flight
// stay a contiguous window of the token order -- and walks them through
// `stages` shared-memory buffers.  A stage holds one complete message
// (header, payload, FP8 scales) -- for bf16 the row is loaded straight into the
// payload position -- and warp 0 lane 0 writes it to every valid slot's row with
// one bulk store each.  In FP8 mode the CTA's warps first cast the staged bf16
// row into the message.  Slot rows and expert ids arrive by cp.async on the
// stage's barrier.  Bounded waits as in the normal bulk dispatch.
__host__ __device__ __forceinline__ uint32_t ll_align128(uint32_t v) { return (v + 127u) & ~127u; }

struct LLBulkSmem {
    uint32_t in_stride, msg_stride, meta_bytes, total;
};

__host__ __device__ __forceinline__ LLBulkSmem ll_bulk_smem(bool fp8, int H, int64_t msg_bytes, int stages) {
    LLBulkSmem b;
    b.in_stride = fp8 ? ll_align128(2 * H) : 0;
    b.msg_stride = ll_align128(static_cast<uint32_t>(msg_bytes));
    b.meta_bytes = ll_align128(64 + stages * (32 * 4 + 32 * 8) + 16);
    b.total = b.meta_bytes + stages * (b.in_stride + b.msg_stride);
    return b;
}

template <bool kFp8>
__global__ void ll_dispatch_bulk_kernel(int R, int T, int maxT, int H, int K, int E, int stages, int per_cta,
                                        const uint8_t* __restrict__ x, const int64_t* __restrict__ topk_idx,
                                        bool round_scale, bool use_ue8m0, const int32_t* __restrict__ slot,
                                        uint8_t* __restrict__ recv_msgs, int64_t msg_bytes, int32_t* status) {
    pdl_enter();
    extern __shared__ __align__(128) uint8_t bulk_smem_raw[];
    uint8_t* smem = bulk_smem_raw;
    const int S = stages;
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const bool warp0 = tid < kWarpSize;
    const int G = H / kFp8Group;
    const uint32_t row_bytes = 2 * H;
    const LLBulkSmem lay = ll_bulk_smem(kFp8, H, msg_bytes, S);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    int32_t* s_row = reinterpret_cast<int32_t*>(smem + 64);            // [S][32]
    int64_t* s_idx = reinterpret_cast<int64_t*>(smem + 64 + S * 128);  // [S][32]
    int32_t* s_flag = reinterpret_cast<int32_t*>(smem + 64 + S * 384);            // [2]
    uint8_t* msg_base = smem + lay.meta_bytes;
    uint8_t* in_base = msg_base + S * lay.msg_stride;
    const int64_t slots = static_cast<int64_t>(R) * maxT;
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * per_cta;
    const int64_t n_local = first < n_tokens ? (n_tokens - first < per_cta ? n_tokens - first : per_cta) : 0;
    if (n_local == 0) return;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1 + kWarpSize);
        fence_barrier_init();
    }
    __syncthreads();

    auto produce = [&](int64_t j) {
        const int st = static_cast<int>(j % S);
        const int64_t g = first + j;
        const int64_t s = g / T;
        const int64_t t = g - s * T;
        if (lane < K) {
            cp_async_4(&s_row[st * 32 + lane], slot + (s * maxT + t) * K + lane);
            cp_async_8(&s_idx[st * 32 + lane], topk_idx + g * K + lane);
        }
        cp_async_arrive(&bars[st]);
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[st], row_bytes);
            uint8_t* dst = kFp8 ? in_base + st * lay.in_stride : msg_base + st * lay.msg_stride + 16;
            bulk_load(dst, x + g * row_bytes, row_bytes, &bars[st]);
        }
    };

    if (warp0) {
        const int64_t pro = n_local < S ? n_local : S;  // every stage starts full
        for (int64_t j = 0; j < pro; ++j) produce(j);
    }
    int64_t j = 0;
    for (; j < n_local; ++j) {
        const int st = static_cast<int>(j % S);
        // one flag per token parity, as in the normal bulk dispatch
        if (tid == 0) s_flag[j & 1] = mbar_wait_bounded(&bars[st], static_cast<uint32_t>((j / S) & 1)) ? 1 : 0;
        __syncthreads();
        if (s_flag[j & 1] == 0) break;
        uint8_t* msg = msg_base + st * lay.msg_stride;
        const int64_t g = first + j;
        if constexpr (kFp8) {
            const int4* xin = reinterpret_cast<const int4*>(in_base + st * lay.in_stride);
            int2* q = reinterpret_cast<int2*>(msg + 16);
            uint8_t* tail = msg + 16 + H;
            const int n16 = H / 8;
            for (int i0 = (tid / kWarpSize) * kWarpSize; i0 < n16; i0 += blockDim.x) {
                const int i = i0 + lane;
                float f[8];
                unpack8(i < n16 ? xin[i] : make_int4(0, 0, 0, 0), f);
                float amax = absmax8(f);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
                const Fp8Scale fs = fp8_scale(amax, round_scale);
                if (i < n16) {
                    q[i] = cast8_e4m3(f, fs.mult);
                    if ((lane & 15) == 0) {
                        if (use_ue8m0) tail[i / 16] = static_cast<uint8_t>(fs.exponent + 127);
                        else reinterpret_cast<float*>(tail)[i / 16] = fs.scale;
                    }
                }
            }
            if (use_ue8m0)
                for (int w = tid; w < (3 * G) / 4; w += blockDim.x) reinterpret_cast<uint32_t*>(tail + G)[w] = 0u;
        }
        if (tid == 0) *reinterpret_cast<int4*>(msg) = make_int4(static_cast<int>(g % T), 0, 0, 0);
        fence_async_smem();
        __syncthreads();
        if (warp0) {
            int64_t dst_row = -1;
            if (lane < K) {
                const int64_t e = s_idx[st * 32 + lane];
                const int32_t row = s_row[st * 32 + lane];
                if (e >= 0 && e < E && row >= 0 && row < slots) dst_row = e * slots + row;
            }
            const unsigned dst = __ballot_sync(kFullMask, dst_row >= 0);
            for (unsigned m = dst; m; m &= m - 1) {
                const int k = __ffs(m) - 1;
                const int64_t r = __shfl_sync(kFullMask, dst_row, k);
                if (lane == 0) bulk_store(recv_msgs + r * msg_bytes, msg, static_cast<uint32_t>(msg_bytes));
            }
            if (lane == 0) bulk_commit();
            if (j + S < n_local) {  // refill this token's stage once its stores have read it
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                produce(j + S);
            }
        }
    }
    if (j < n_local && tid == 0) {
        report(status, EP_ERR_TIMEOUT);
        const int64_t issued = (j + S < n_local) ? j + S : n_local;
        for (int64_t k = j + 1; k < issued; ++k) mbar_wait_bounded(&bars[k % S], static_cast<uint32_t>((k / S) & 1));
    }
    if (tid == 0) bulk_wait_all();
}

// One warp per source token.  kFp8: e4m3 payload + scales (fp32, or UE8M0 bytes).
template <bool kFp8>
__global__ void __launch_bounds__(kLLDispatchThreads)
    ll_dispatch_kernel(int R, int T, int maxT, int H, int K, int E, const int4* __restrict__ x,
                       const int64_t* __restrict__ topk_idx, bool round_scale, bool use_ue8m0,
                       const int32_t* __restrict__ slot, uint8_t* __restrict__ recv_msgs, int64_t msg_bytes) {
    pdl_enter();
    constexpr int kWarps = kLLDispatchThreads / kWarpSize;
    const int lane = lane_id();
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int64_t slots = static_cast<int64_t>(R) * maxT;
    const int n16 = H / 8;
    const int G = H / kFp8Group;

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + threadIdx.x / kWarpSize; g < n_tokens;
         g += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int s = static_cast<int>(g / T);
        const int t = static_cast<int>(g - static_cast<int64_t>(s) * T);
        // Lane k owns slot k: destination expert and final row.
        int e = -1;
        int64_t row = -1;
        if (lane < K) {
            const int64_t v = __ldg(topk_idx + g * K + lane);
            const int32_t r = __ldg(slot + (static_cast<int64_t>(s) * maxT + t) * K + lane);
            if (v >= 0 && v < E && r >= 0 && r < slots) {
                e = static_cast<int>(v);
                row = r;
            }
        }
        const unsigned dst = __ballot_sync(kFullMask, row >= 0);
        if (dst == 0u) continue;

        // Header {t, 0, 0, 0}.
        for (unsigned m = dst; m; m &= m - 1) {
            const int k = __ffs(m) - 1;
            const int ek = __shfl_sync(kFullMask, e, k);
            const int64_t rk = __shfl_sync(kFullMask, row, k);
            if (lane == 0)
                st_stream_v4(reinterpret_cast<int4*>(recv_msgs + (static_cast<int64_t>(ek) * slots + rk) * msg_bytes),
                             make_int4(t, 0, 0, 0));
        }

        const int4* src = x + g * n16;
        if constexpr (!kFp8) {
            for (int i0 = 0; i0 < n16; i0 += kWarpSize * kLLUnroll) {
                int4 v[kLLUnroll];
#pragma unroll
                for (int u = 0; u < kLLUnroll; ++u) {
                    const int i = i0 + u * kWarpSize + lane;
                    if (i < n16) v[u] = ld_stream_v4(src + i);
                }
                for (unsigned m = dst; m; m &= m - 1) {
                    const int k = __ffs(m) - 1;
                    const int ek = __shfl_sync(kFullMask, e, k);
                    const int64_t rk = __shfl_sync(kFullMask, row, k);
                    int4* d = reinterpret_cast<int4*>(recv_msgs + (static_cast<int64_t>(ek) * slots + rk) * msg_bytes + 16);
#pragma unroll
                    for (int u = 0; u < kLLUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (i < n16) st_stream_v4(d + i, v[u]);
                    }
                }
            }
        } else {
            for (int i0 = 0; i0 < n16; i0 += kWarpSize * kLLUnroll) {
                int4 v[kLLUnroll];
#pragma unroll
                for (int u = 0; u < kLLUnroll; ++u) {
                    const int i = i0 + u * kWarpSize + lane;
                    v[u] = i < n16 ? ld_stream_v4(src + i) : make_int4(0, 0, 0, 0);
                }
                int2 q[kLLUnroll];
                float sc[kLLUnroll];
                int ex[kLLUnroll];
#pragma unroll
                for (int u = 0; u < kLLUnroll; ++u) {
                    float f[8];
                    unpack8(v[u], f);
                    float amax = absmax8(f);
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, off));
                    const Fp8Scale fs = fp8_scale(amax, round_scale);
                    q[u] = cast8_e4m3(f, fs.mult);
                    sc[u] = fs.scale;
                    ex[u] = fs.exponent;
                }
                for (unsigned m = dst; m; m &= m - 1) {
                    const int k = __ffs(m) - 1;
                    const int ek = __shfl_sync(kFullMask, e, k);
                    const int64_t rk = __shfl_sync(kFullMask, row, k);
                    uint8_t* msg = recv_msgs + (static_cast<int64_t>(ek) * slots + rk) * msg_bytes;
                    int2* d = reinterpret_cast<int2*>(msg + 16);
                    uint8_t* tail = msg + 16 + H;
#pragma unroll
                    for (int u = 0; u < kLLUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (i < n16) {
                            st_stream_v2(d + i, q[u]);
                            if ((lane & 15) == 0) {
                                if (use_ue8m0) tail[i / 16] = static_cast<uint8_t>(ex[u] + 127);
                                else reinterpret_cast<float*>(tail)[i / 16] = sc[u];
                            }
                        }
                    }
                }
            }
            if (use_ue8m0) {
                // Bytes [G, 4G) of the scale tail are zero (G is a multiple of 4).
                for (unsigned m = dst; m; m &= m - 1) {
                    const int k = __ffs(m) - 1;
                    const int ek = __shfl_sync(kFullMask, e, k);
                    const int64_t rk = __shfl_sync(kFullMask, row, k);
                    uint32_t* z = reinterpret_cast<uint32_t*>(recv_msgs + (static_cast<int64_t>(ek) * slots + rk) * msg_bytes +
                                                              16 + H + G);
                    for (int w = lane; w < (3 * G) / 4; w += kWarpSize) z[w] = 0u;
                }
            }
        }
    }
}

template <int kFanIn>
__global__ void __launch_bounds__(kLLCombineThreads)
    ll_combine_kernel(int R, int T, int maxT, int H, int K, int E, const int4* __restrict__ y, int64_t y_row16,
                      const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_weights,
                      const int32_t* __restrict__ slot, int4* __restrict__ out) {
    pdl_enter();
    constexpr int kWarps = kLLCombineThreads / kWarpSize;
    const int lane = lane_id();
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    const int64_t slots = static_cast<int64_t>(R) * maxT;
    const int n16 = H / 8;

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + threadIdx.x / kWarpSize; g < n_tokens;
         g += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int s = static_cast<int>(g / T);
        const int t = static_cast<int>(g - static_cast<int64_t>(s) * T);
        int64_t src_row = -1;  // flat row e * slots + row
        float w = 0.0f;
        if (lane < K) {
            const int64_t v = __ldg(topk_idx + g * K + lane);
            const int32_t r = __ldg(slot + (static_cast<int64_t>(s) * maxT + t) * K + lane);
            if (v >= 0 && v < E && r >= 0 && r < slots) {
                src_row = v * slots + r;
                w = __ldg(topk_weights + g * K + lane);
            }
        }
        const unsigned valid = __ballot_sync(kFullMask, src_row >= 0);

        for (int i0 = 0; i0 < n16; i0 += kWarpSize * kLLCombineUnroll) {
            float acc[kLLCombineUnroll][8];
#pragma unroll
            for (int u = 0; u < kLLCombineUnroll; ++u)
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[u][q] = 0.0f;
            unsigned m = valid;
            while (m) {
                int kk[kFanIn];
                int64_t sr[kFanIn];
                float wk[kFanIn];
#pragma unroll
                for (int j = 0; j < kFanIn; ++j) {
                    kk[j] = m ? __ffs(m) - 1 : -1;
                    if (m) m &= m - 1;
                    const int srcl = kk[j] < 0 ? 0 : kk[j];
                    sr[j] = __shfl_sync(kFullMask, src_row, srcl);
                    wk[j] = __shfl_sync(kFullMask, w, srcl);
                }
                int4 v[kFanIn][kLLCombineUnroll];
#pragma unroll
                for (int j = 0; j < kFanIn; ++j)
#pragma unroll
                    for (int u = 0; u < kLLCombineUnroll; ++u) {
                        const int i = i0 + u * kWarpSize + lane;
                        if (kk[j] >= 0 && i < n16) v[j][u] = ld_stream_v4(y + sr[j] * y_row16 + i);
                    }
#pragma unroll
                for (int j = 0; j < kFanIn; ++j) {
                    if (kk[j] < 0) continue;
#pragma unroll
                    for (int u = 0; u < kLLCombineUnroll; ++u) {
                        float f[8];
                        unpack8(v[j][u], f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[u][q] = __fmaf_rn(wk[j], f[q], acc[u][q]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kLLCombineUnroll; ++u) {
                const int i = i0 + u * kWarpSize + lane;
                if (i < n16) out[g * n16 + i] = pack8_bf16(acc[u]);
            }
        }
    }
}

// Self-test of the bounded waits: one thread waits, with a small iteration cap, on
// an mbarrier whose phase nothing completes.  The wait must give up, record
// EP_ERR_TIMEOUT and mark `rank` in the mask buffer -- what a receiver does
// with a source rank that never delivers ([P1] low-latency receive excerpt).
__global__ void bounded_wait_selftest_kernel(uint32_t max_iterations, int rank, int32_t* rank_mask,
                                             int32_t* status) {
    pdl_enter();
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(&bar, 0, max_iterations)) {
        report(status, EP_ERR_TIMEOUT);
        if (rank_mask != nullptr) atomicExch(rank_mask + rank, 1);
    }
}

template <typename Kernel>
int resident_blocks(Kernel k, int threads, int num_sms, size_t smem = 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return per_sm * num_sms;
}

int clamp_grid(int planned, int64_t warps_needed, int warps_per_block) {
    const int64_t need = (warps_needed + warps_per_block - 1) / warps_per_block;
    return static_cast<int>(need < planned ? (need > 0 ? need : 1) : planned);
}

size_t ll_count_smem(int E, int threads) {
    return sizeof(int32_t) * static_cast<size_t>(threads / kWarpSize + 1) * E;
}

constexpr size_t kLLCountMaxSmem = 200u * 1024u;

// One chunk of 1024 top-k entries per pass while the per-warp histograms fit in shared memory
// (measured: 57.0 against 58.6 us per ll_v3 dispatch), else 512-thread passes.
int ll_count_threads(int E) {
    return ll_count_smem(E, kLLCountThreadsLarge) <= kLLCountMaxSmem ? kLLCountThreadsLarge : kLLCountThreads;
}

}  // namespace

constexpr uint32_t kLLBulkMaxSmem = 200u * 1024u;  // larger messages use the register kernel
constexpr int kLLBulkRoundsPerCta = 1;              // bulk LL dispatch: at most stages x this tokens per CTA

cudaError_t plan_ll(LaunchPlan* plan, int num_experts) {
    (void)num_experts;  // every expert count is served by the limits set below
    const int n = plan->num_sms;
    plan->ll_dispatch_blocks[0] = resident_blocks(ll_dispatch_kernel<false>, kLLDispatchThreads, n);
    plan->ll_dispatch_blocks[1] = resident_blocks(ll_dispatch_kernel<true>, kLLDispatchThreads, n);
    plan->ll_combine_blocks = resident_blocks(ll_combine_kernel<kLLCombineFanIn>, kLLCombineThreads, n);
    plan->ll_combine_blocks_small_k = resident_blocks(ll_combine_kernel<kLLCombineFanInSmallK>, kLLCombineThreads, n);
    cudaError_t err = cudaFuncSetAttribute(ll_dispatch_bulk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kLLBulkMaxSmem));
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(ll_dispatch_bulk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kLLBulkMaxSmem));
    if (err != cudaSuccess) return err;
    // both block sizes may be chosen per call (the allocation-free entry point plans for the most
    // experts and launches with fewer), so both may use the whole budget
    err = cudaFuncSetAttribute(ll_count_kernel<kLLCountThreadsLarge>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kLLCountMaxSmem));
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(ll_count_kernel<kLLCountThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kLLCountMaxSmem));
}

cudaError_t launch_ll_dispatch(const LaunchPlan& plan, int R, int T, int maxT, int H, int K, int E,
                               const void* x, const int64_t* topk_idx, bool use_fp8, bool round_scale,
                               bool use_ue8m0, const int32_t* rank_mask, int32_t* slot, int32_t* cnt,
                               void* recv_msgs, int32_t* packed_recv_count, int64_t* layout_range,
                               int32_t* stats, int32_t* status, cudaStream_t stream) {
    const int count_threads = ll_count_threads(E);
    auto count_kernel = count_threads == kLLCountThreadsLarge ? ll_count_kernel<kLLCountThreadsLarge>
                                                              : ll_count_kernel<kLLCountThreads>;
    cudaError_t err = launch_kernel(count_kernel, dim3(R), dim3(count_threads), ll_count_smem(E, count_threads), stream,
                                    1, R, T, maxT, K, E, topk_idx, rank_mask, slot, cnt, status);
    if (err != cudaSuccess) return err;
    const int fin_threads = kFinishThreads;
    const int expert_blocks = (E + fin_threads / kWarpSize - 1) / (fin_threads / kWarpSize);
    const int64_t n_slots = static_cast<int64_t>(R) * T * K;
    const int slot_blocks = static_cast<int>((n_slots + fin_threads - 1) / fin_threads);
    err = launch_kernel(ll_finish_kernel, dim3(expert_blocks + slot_blocks), dim3(fin_threads), 0, stream, 1, R, T,
                        maxT, K, E, expert_blocks, topk_idx, static_cast<const int32_t*>(cnt), slot,
                        packed_recv_count, layout_range, stats, status);
    if (err != cudaSuccess) return err;
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    if (n_tokens == 0) return cudaSuccess;
    const int64_t msg = ep_ll_msg_bytes(H, use_fp8 ? 1 : 0);
    const bool rs = round_scale || use_ue8m0;
    // Bulk-copy kernel.  FP8: one stage (the bf16 row and its message, 22 KB at 7168 channels) and one
    // token per CTA, so 9 CTAs -- 36 casting warps -- share an SM (measured on ll_v3 against two stages
    // and 5 CTAs per SM: 56.3 against 57.5 us per dispatch, and 59.0 against 61.1 us from a cold L2;
    // three or four stages, more tokens per CTA, or the row loaded into registers instead of staged
    // were all slower).  bf16: about 64 KB of stages per CTA, 2..8 stages.
    const uint32_t per_stage = ll_bulk_smem(use_fp8, H, msg, 1).total - ll_bulk_smem(use_fp8, H, msg, 0).total;
    int S = static_cast<int>(65536u / per_stage);
    S = use_fp8 ? 1 : (S < 2 ? 2 : (S > 8 ? 8 : S));
    const uint32_t smem = ll_bulk_smem(use_fp8, H, msg, S).total;
    if (smem <= kLLBulkMaxSmem) {
        // contiguous token blocks: enough CTAs to fill the GPU once (CTAs resident per SM from the
        // shared memory: 227 KB per SM, 1 KB reserved per CTA), at most one round of the stages
        int per_sm = static_cast<int>((227u * 1024u) / (smem + 1024u));
        per_sm = per_sm < 1 ? 1 : (per_sm > 32 ? 32 : per_sm);
        const int64_t resident = static_cast<int64_t>(per_sm) * plan.num_sms;
        const int64_t fill = (n_tokens + resident - 1) / resident;
        const int cap_cta = plan.sm_limited ? INT32_MAX : S * kLLBulkRoundsPerCta;  // max_sms: one wave
        const int per_cta = static_cast<int>(fill < 1 ? 1 : (fill > cap_cta ? cap_cta : fill));
        const int grid = static_cast<int>((n_tokens + per_cta - 1) / per_cta);
        auto kernel = use_fp8 ? ll_dispatch_bulk_kernel<true> : ll_dispatch_bulk_kernel<false>;
        return launch_kernel(kernel, dim3(grid), dim3(use_fp8 ? 4 * kWarpSize : kWarpSize), smem, stream, 1, R, T,
                             maxT, H, K, E, S, per_cta, static_cast<const uint8_t*>(x), topk_idx, rs, use_ue8m0,
                             static_cast<const int32_t*>(slot), static_cast<uint8_t*>(recv_msgs), msg, status);
    }
    const int grid = clamp_grid(plan.ll_dispatch_blocks[use_fp8 ? 1 : 0], n_tokens, kLLDispatchThreads / kWarpSize);
    auto kernel = use_fp8 ? ll_dispatch_kernel<true> : ll_dispatch_kernel<false>;
    return launch_kernel(kernel, dim3(grid), dim3(kLLDispatchThreads), 0, stream, 1, R, T, maxT, H, K, E,
                         static_cast<const int4*>(x), topk_idx, rs, use_ue8m0, static_cast<const int32_t*>(slot),
                         static_cast<uint8_t*>(recv_msgs), msg);
}

cudaError_t launch_ll_combine(const LaunchPlan& plan, int R, int T, int maxT, int H, int K, int E,
                              const void* y, int64_t y_row_bytes, const int64_t* topk_idx, const float* topk_weights,
                              const int32_t* slot, void* out, cudaStream_t stream) {
    const int64_t n_tokens = static_cast<int64_t>(R) * T;
    if (n_tokens == 0) return cudaSuccess;
    const bool small_k = K <= kLLCombineFanInSmallK;
    const int grid = clamp_grid(small_k ? plan.ll_combine_blocks_small_k : plan.ll_combine_blocks, n_tokens,
                                kLLCombineThreads / kWarpSize);
    auto kernel = small_k ? ll_combine_kernel<kLLCombineFanInSmallK> : ll_combine_kernel<kLLCombineFanIn>;
    return launch_kernel(kernel, dim3(grid), dim3(kLLCombineThreads), 0, stream, 1, R, T, maxT, H, K, E,
                         static_cast<const int4*>(y), y_row_bytes / 16, topk_idx, topk_weights, slot,
                         static_cast<int4*>(out));
}

cudaError_t launch_bounded_wait_selftest(uint32_t max_iterations, int rank, int32_t* rank_mask, int32_t* status,
                                         cudaStream_t stream) {
    return launch_kernel(bounded_wait_selftest_kernel, dim3(1), dim3(kWarpSize), 0, stream, 1, max_iterations, rank,
                         rank_mask, status);
}

}  // namespace ep
