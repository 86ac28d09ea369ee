// ep_layout.cu -- routing layout and dispatch bookkeeping kernels.
//
// get_dispatch_layout ("第 4 章 V1：布局、dispatch 与 combine" §4.1): per source
// rank, counts of tokens per destination rank / RDMA node / expert and the
// is_token_in_rank mask.  dispatch_notify (same section, the handle's prefix
// matrices, recv_src_idx and send_head): every hit (s, t, r) gets its receive
// row, ordered by source rank then token, with channel prefix matrices at
// the boundaries of C contiguous token ranges.
//
// Both kernels run one CTA per source rank: the per-rank work is a few
// hundred KB of routing data, so a single CTA with every load of a round in
// flight reads it in a couple of microseconds, and keeping a source rank in
// one CTA makes its token scan a block-local scan (no cross-CTA waiting and
// no scratch memory).  A second grid slot (blockIdx.x == R) of the notify
// kernel folds the R x R and R x E summaries.
#include "ep_common.cuh"
#include "ep_kernels.h"

namespace ep {

namespace {

constexpr int kLayoutRound = 4096;  // tokens per round of the layout kernel (mask staging in smem)
constexpr int kLayoutUnroll = 8;    // top-k entries in flight per thread
constexpr int kNotifyTPT = 4;       // tokens per thread per notify round
constexpr int kNotifyRound = kNotifyThreads * kNotifyTPT;
constexpr int kNotifyWarps = kNotifyThreads / kWarpSize;

// Mask of destination ranks of one token from its R-byte is_token_in_rank row.
__device__ __forceinline__ uint32_t load_rank_mask(const uint8_t* row, int R) {
    uint32_t m = 0;
    if ((R & 3) == 0) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
        for (int i = 0; i < R / 4; ++i) {
            const uint32_t v = __ldg(w + i);
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if ((v >> (8 * b)) & 0xffu) m |= 1u << (4 * i + b);
        }
    } else {
        for (int r = 0; r < R; ++r)
            if (__ldg(row + r)) m |= 1u << r;
    }
    return m;
}

__device__ __forceinline__ void store_rank_mask(uint8_t* row, int R, uint32_t m) {
    if ((R & 3) == 0) {
        uint32_t* w = reinterpret_cast<uint32_t*>(row);
        for (int i = 0; i < R / 4; ++i) {
            uint32_t v = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) v |= ((m >> (4 * i + b)) & 1u) << (8 * b);
            w[i] = v;
        }
    } else {
        for (int r = 0; r < R; ++r) row[r] = static_cast<uint8_t>((m >> r) & 1u);
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
    get_dispatch_layout_kernel(const int64_t* __restrict__ topk_idx, int R, int T, int K, int E, int EL,
                               int32_t* __restrict__ tpr, int32_t* __restrict__ tprdma,
                               int32_t* __restrict__ tpe, uint8_t* __restrict__ itr, int32_t* status) {
    extern __shared__ int32_t s_expert[];  // [E]
    __shared__ uint32_t s_mask[kLayoutRound];
    __shared__ int32_t s_rank[kMaxRanks];
    __shared__ int32_t s_node[kMaxRanks / 8];

    const int s = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int NN = (R + 7) / 8;
    for (int i = tid; i < E; i += kLayoutThreads) s_expert[i] = 0;
    if (tid < kMaxRanks) s_rank[tid] = 0;
    if (tid < kMaxRanks / 8) s_node[tid] = 0;

    const int64_t* idx_s = topk_idx + static_cast<int64_t>(s) * T * K;
    uint8_t* itr_s = itr + static_cast<int64_t>(s) * T * R;

    for (int round = 0; round < T; round += kLayoutRound) {
        const int len = min(kLayoutRound, T - round);
        for (int i = tid; i < len; i += kLayoutThreads) s_mask[i] = 0;
        __syncthreads();

        // Phase A: flat walk over this round's top-k entries (coalesced 8-byte loads).
        const int64_t e_begin = static_cast<int64_t>(round) * K;
        const int64_t e_end = static_cast<int64_t>(round + len) * K;
        for (int64_t i0 = e_begin + tid; i0 < e_end; i0 += kLayoutUnroll * kLayoutThreads) {
            int64_t v[kLayoutUnroll];
#pragma unroll
            for (int u = 0; u < kLayoutUnroll; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * kLayoutThreads;
                v[u] = i < e_end ? __ldg(idx_s + i) : -1;
            }
#pragma unroll
            for (int u = 0; u < kLayoutUnroll; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * kLayoutThreads;
                const int64_t e = v[u];
                if (i >= e_end || e == -1) continue;
                if (e < 0 || e >= E) {
                    report(status, EP_ERR_BAD_EXPERT);
                    continue;
                }
                atomicAdd(&s_expert[e], 1);
                atomicOr(&s_mask[static_cast<int>(i / K) - round], 1u << (static_cast<int>(e) / EL));
            }
        }
        __syncthreads();

        // Phase B: per token, the mask row and the per-rank / per-node counts.
        for (int tl0 = 0; tl0 < len; tl0 += kLayoutThreads) {
            const int tl = tl0 + tid;
            const uint32_t m = tl < len ? s_mask[tl] : 0u;
            if (tl < len) store_rank_mask(itr_s + static_cast<int64_t>(round + tl) * R, R, m);
            for (int r = 0; r < R; ++r) {
                const unsigned b = __ballot_sync(kFullMask, (m >> r) & 1u);
                if (lane == 0 && b) atomicAdd(&s_rank[r], __popc(b));
            }
            for (int n = 0; n < NN; ++n) {
                const unsigned b = __ballot_sync(kFullMask, ((m >> (8 * n)) & 0xffu) != 0u);
                if (lane == 0 && b) atomicAdd(&s_node[n], __popc(b));
            }
        }
        __syncthreads();
    }

    for (int i = tid; i < E; i += kLayoutThreads) tpe[static_cast<int64_t>(s) * E + i] = s_expert[i];
    if (tid < R) tpr[s * R + tid] = s_rank[tid];
    if (tprdma != nullptr && tid < NN) tprdma[s * NN + tid] = s_node[tid];
}

// One CTA per source rank s (blockIdx.x < R): block-local scan of the R hit
// columns over the tokens of s.  blockIdx.x == R: rank_prefix_matrix, num_recv
// and the aligned per-expert receive counts.
__global__ void __launch_bounds__(kNotifyThreads)
    dispatch_notify_kernel(int R, int T, int E, int C, int A, int64_t cap, const int32_t* __restrict__ tpr,
                           const uint8_t* __restrict__ itr, const int32_t* __restrict__ tpe,
                           int32_t* __restrict__ rank_prefix, int32_t* __restrict__ channel_prefix,
                           int32_t* __restrict__ recv_channel_prefix, int32_t* __restrict__ num_recv,
                           int32_t* __restrict__ send_head, int32_t* __restrict__ recv_src_idx,
                           int32_t* __restrict__ num_recv_per_expert, int32_t* status) {
    const int tid = threadIdx.x;
    const int s = blockIdx.x;

    if (s == R) {
        for (int r = tid; r < R; r += kNotifyThreads) {
            int32_t acc = 0;
            for (int sp = 0; sp < R; ++sp) {
                acc += __ldg(tpr + sp * R + r);
                rank_prefix[sp * R + r] = acc;
            }
            num_recv[r] = acc;
            if (acc > cap) report(status, EP_ERR_CAPACITY);
        }
        for (int e = tid; e < E; e += kNotifyThreads) {
            int64_t sum = 0;
            for (int sp = 0; sp < R; ++sp) sum += __ldg(tpe + static_cast<int64_t>(sp) * E + e);
            num_recv_per_expert[e] = static_cast<int32_t>(((sum + A - 1) / A) * A);
        }
        return;
    }

    __shared__ int32_t s_base[kMaxRanks];  // rows of rank r taken by sources < s
    __shared__ int32_t s_run[kMaxRanks];   // hits of (s -> r) in earlier rounds
    __shared__ int32_t s_cnt[kMaxRanks][kNotifyTPT * kNotifyWarps + 1];

    const int lane = lane_id();
    const int warp = tid / kWarpSize;
    if (tid < R) {
        int32_t acc = 0;
        for (int sp = 0; sp < s; ++sp) acc += __ldg(tpr + sp * R + tid);
        s_base[tid] = acc;
        s_run[tid] = 0;
    }
    const int chunk = max(1, (T + C - 1) / C);
    const uint8_t* itr_s = itr + static_cast<int64_t>(s) * T * R;
    int32_t* head_s = send_head + static_cast<int64_t>(s) * T * R;
    __syncthreads();

    for (int round = 0; round < T; round += kNotifyRound) {
        uint32_t mask[kNotifyTPT];
#pragma unroll
        for (int j = 0; j < kNotifyTPT; ++j) {
            const int t = round + j * kNotifyThreads + tid;
            mask[j] = t < T ? load_rank_mask(itr_s + static_cast<int64_t>(t) * R, R) : 0u;
        }
        // Per-warp hit counts of every (slot j, warp) group of 32 consecutive tokens.
#pragma unroll
        for (int j = 0; j < kNotifyTPT; ++j)
            for (int r = 0; r < R; ++r) {
                const unsigned b = __ballot_sync(kFullMask, (mask[j] >> r) & 1u);
                if (lane == 0) s_cnt[r][j * kNotifyWarps + warp] = __popc(b);
            }
        __syncthreads();
        // Warp r turns column r into exclusive prefixes (plus the earlier rounds' hits).
        if (warp < R) {
            constexpr int kPer = kNotifyTPT * kNotifyWarps / kWarpSize;
            int32_t v[kPer];
            int32_t local = 0;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                v[i] = s_cnt[warp][lane * kPer + i];
                local += v[i];
            }
            int32_t incl = local;
#pragma unroll
            for (int off = 1; off < kWarpSize; off <<= 1) {
                const int32_t o = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += o;
            }
            const int32_t before = s_run[warp];
            int32_t run = before + incl - local;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                s_cnt[warp][lane * kPer + i] = run;
                run += v[i];
            }
            __syncwarp();
            if (lane == kWarpSize - 1) s_run[warp] = before + incl;
        }
        __syncthreads();
        // Rows, recv_src_idx and the channel boundaries.
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int j = 0; j < kNotifyTPT; ++j) {
            const int t = round + j * kNotifyThreads + tid;
            const bool live = t < T;
            const bool boundary = live && (t % chunk) == 0;
            const int c = t / chunk;
            for (int r = 0; r < R; ++r) {
                const bool bit = (mask[j] >> r) & 1u;
                const unsigned b = __ballot_sync(kFullMask, bit);
                const int32_t excl = s_cnt[r][j * kNotifyWarps + warp] + __popc(b & lt);
                if (!live) continue;
                int32_t row = -1;
                if (bit) {
                    row = s_base[r] + excl;
                    if (row < cap) recv_src_idx[static_cast<int64_t>(r) * cap + row] = t;
                }
                head_s[static_cast<int64_t>(t) * R + r] = row;
                if (boundary) {
                    recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = s_base[r] + excl;
                    if (c > 0) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c - 1] = excl;
                }
            }
        }
        __syncthreads();
    }

    // Channels that end at T (or hold no token) and the consistency check.
    if (tid < R) {
        const int r = tid;
        const int32_t total = s_run[r];
        if (total != __ldg(tpr + s * R + r)) report(status, EP_ERR_INCONSISTENT);
        for (int c = 0; c < C; ++c) {
            const int64_t start = min(static_cast<int64_t>(T), static_cast<int64_t>(c) * chunk);
            const int64_t end = min(static_cast<int64_t>(T), static_cast<int64_t>(c + 1) * chunk);
            if (end == T) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c] = total;
            if (start == T) recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = s_base[r] + total;
        }
    }
}

}  // namespace

cudaError_t launch_get_dispatch_layout(const int64_t* topk_idx, int R, int T, int K, int E, int32_t* tpr,
                                       int32_t* tprdma, int32_t* tpe, uint8_t* itr, int32_t* status,
                                       cudaStream_t stream) {
    const size_t smem = sizeof(int32_t) * static_cast<size_t>(E);
    get_dispatch_layout_kernel<<<R, kLayoutThreads, smem, stream>>>(topk_idx, R, T, K, E, E / R, tpr, tprdma,
                                                                     tpe, itr, status);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_notify(int R, int T, int E, int C, int A, int64_t cap, const int32_t* tpr,
                                   const uint8_t* itr, const int32_t* tpe, int32_t* rank_prefix,
                                   int32_t* channel_prefix, int32_t* recv_channel_prefix, int32_t* num_recv,
                                   int32_t* send_head, int32_t* recv_src_idx, int32_t* num_recv_per_expert,
                                   int32_t* status, cudaStream_t stream) {
    dispatch_notify_kernel<<<R + 1, kNotifyThreads, 0, stream>>>(R, T, E, C, A, cap, tpr, itr, tpe, rank_prefix,
                                                                 channel_prefix, recv_channel_prefix, num_recv,
                                                                 send_head, recv_src_idx, num_recv_per_expert,
                                                                 status);
    return cudaGetLastError();
}

}  // namespace ep
