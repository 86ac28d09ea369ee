// ep_layout.cu -- routing layout and dispatch bookkeeping kernels.
//
// get_dispatch_layout ("第 4 章 V1：布局、dispatch 与 combine" §4.1): per source
// rank, counts of tokens per destination rank / RDMA node / expert and the
// is_token_in_rank mask.  dispatch_notify (same section, the handle's prefix
// matrices, recv_src_idx and send_head): every hit (s, t, r) gets its receive
// row, ordered by source rank then token, with channel prefix matrices at
// the boundaries of C contiguous token ranges.  When the ranks form two or
// more whole nodes of 8 (the two-level layout of §4.2 of the same page; rank
// r = 8 n + l is GPU l of node n) the notify also builds the node-level
// record: per source and node, the tokens that reach any rank of the node at
// every channel end; per rank (n, l), the inclusive prefix over source nodes
// m of the tokens of source (m, l) that reach node n -- the tokens (n, l)
// receives over RDMA, since the GPUs of a node share one RDMA rank and the
// RDMA team is the ranks with the same GPU index ("DeepEP Normal vs
// Low-Latency 双模式深度分析").
//
// The two separate kernels (ep_get_dispatch_layout, ep_notify_dispatch) give
// each source rank one thread-block cluster of kClusterCtas CTAs; CTA q of the
// cluster owns the q-th contiguous slice of that rank's tokens.  Partial
// counts are exchanged through distributed shared memory after a cluster
// barrier, so a kernel is one launch with no global scratch, no atomics on
// global memory and no waiting on other launches.  ep_layout_notify runs both
// steps as one pass of a decoupled look-back scan (layout_scan_kernel, below).
// With ranks masked in the handle's mask buffer, the layout leaves out every
// slot that starts or ends on a masked rank (the mask buffer of the
// low-latency receive excerpt of the same page, applied to the normal path).
#include <cooperative_groups.h>

#include "ep_common.cuh"
#include "ep_kernels.h"

namespace cg = cooperative_groups;

namespace ep {

namespace {

constexpr int kClusterCtas = 8;      // CTAs per source rank (portable cluster size)
constexpr int kLayoutRound = 2048;   // tokens of one round of the layout kernel (mask staging in smem)
constexpr int kLayoutUnroll = 8;     // top-k entries in flight per thread
constexpr int kNotifyWarps = kNotifyThreads / kWarpSize;
constexpr int kRanksPerNode = 8;     // NVLink peers of one node
constexpr int kMaxNodes = kMaxRanks / kRanksPerNode;
constexpr int kMaxColumns = kMaxRanks + kMaxNodes;  // notify count columns: ranks, then nodes

// Mask of destination ranks of one token from its R-byte is_token_in_rank row (L2 loads: the
// one-launch layout + notify reads rows that the same launch wrote).
__device__ __forceinline__ uint32_t load_rank_mask(const uint8_t* row, int R) {
    uint32_t m = 0;
    if ((R & 3) == 0) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(row);
        for (int i = 0; i < R / 4; ++i) {
            const uint32_t v = __ldcg(w + i);
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if ((v >> (8 * b)) & 0xffu) m |= 1u << (4 * i + b);
        }
    } else {
        for (int r = 0; r < R; ++r)
            if (__ldcg(row + r)) m |= 1u << r;
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

// Column col of a token's hits: rank col for col < R, else whether any rank of node col - R is hit.
__device__ __forceinline__ bool column_bit(uint32_t m, int col, int R) {
    return col < R ? ((m >> col) & 1u) != 0u
                   : ((m >> (kRanksPerNode * (col - R))) & ((1u << kRanksPerNode) - 1u)) != 0u;
}

// Token slice [lo, hi) of CTA q of a cluster over T tokens.
__device__ __forceinline__ void cluster_slice(int T, int q, int& lo, int& hi) {
    const int per = (T + kClusterCtas - 1) / kClusterCtas;
    lo = min(T, q * per);
    hi = min(T, lo + per);
}

// Layout of source s by CTA q of its cluster: the slice's tokens are marked in is_token_in_rank,
// counted per expert, per destination rank and per node.  Slots that start or end on a rank of
// `rmask` (bit r: rank r masked) are left out as if they were -1.  Leaves the slice's hits per rank in
// s_cnt[0, R) and per node in s_cnt[R, R + ceil(R/8)) -- read by the rest of the cluster -- and
// writes the source's totals (tpr, tprdma when given, tpe).  Ends with a cluster barrier.
__device__ __forceinline__ void layout_source(const cg::cluster_group& cluster, int s, int q,
                                              const int64_t* __restrict__ topk_idx, uint32_t rmask, int R, int T,
                                              int K, int E, int EL, int32_t* __restrict__ tpr,
                                              int32_t* __restrict__ tprdma, int32_t* __restrict__ tpe,
                                              uint8_t* __restrict__ itr, int32_t* status, int32_t* s_expert,
                                              int32_t* s_cnt) {
    __shared__ uint32_t s_mask[kLayoutRound];
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int NN = (R + kRanksPerNode - 1) / kRanksPerNode;
    const bool src_masked = (rmask >> s) & 1u;
    for (int i = tid; i < E; i += kLayoutThreads) s_expert[i] = 0;
    if (tid < kMaxColumns) s_cnt[tid] = 0;

    int lo, hi;
    cluster_slice(T, q, lo, hi);
    const int64_t* idx_s = topk_idx + static_cast<int64_t>(s) * T * K;
    uint8_t* itr_s = itr + static_cast<int64_t>(s) * T * R;

    for (int round = lo; round < hi; round += kLayoutRound) {
        const int len = min(kLayoutRound, hi - round);
        for (int i = tid; i < len; i += kLayoutThreads) s_mask[i] = 0;
        __syncthreads();
        // Flat walk over this round's top-k entries (coalesced 8-byte loads, several in flight).
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
                const int d = static_cast<int>(e) / EL;
                if (src_masked || ((rmask >> d) & 1u)) continue;  // a masked rank neither sends nor receives
                atomicAdd(&s_expert[e], 1);
                atomicOr(&s_mask[static_cast<int>(i / K) - round], 1u << d);
            }
        }
        __syncthreads();
        // Per token: the mask row and the per-rank / per-node counts.
        for (int tl0 = 0; tl0 < len; tl0 += kLayoutThreads) {
            const int tl = tl0 + tid;
            const uint32_t m = tl < len ? s_mask[tl] : 0u;
            if (tl < len) store_rank_mask(itr_s + static_cast<int64_t>(round + tl) * R, R, m);
            for (int r = 0; r < R; ++r) {
                const unsigned b = __ballot_sync(kFullMask, (m >> r) & 1u);
                if (lane == 0 && b) atomicAdd(&s_cnt[r], __popc(b));
            }
            for (int n = 0; n < NN; ++n) {
                const unsigned b = __ballot_sync(kFullMask, column_bit(m, R + n, R));
                if (lane == 0 && b) atomicAdd(&s_cnt[R + n], __popc(b));
            }
        }
        __syncthreads();
    }

    // Sum the cluster's partial counts: CTA q writes the entries i with i % kClusterCtas == q.
    cluster.sync();
    for (int e = q + kClusterCtas * tid; e < E; e += kClusterCtas * kLayoutThreads) {
        int32_t sum = 0;
        for (int p = 0; p < kClusterCtas; ++p) sum += cluster.map_shared_rank(s_expert, p)[e];
        tpe[static_cast<int64_t>(s) * E + e] = sum;
    }
    if (q == 0 && tid < R) {
        int32_t sum = 0;
        for (int p = 0; p < kClusterCtas; ++p) sum += cluster.map_shared_rank(s_cnt, p)[tid];
        tpr[s * R + tid] = sum;
    }
    if (q == 1 && tprdma != nullptr && tid < NN) {
        int32_t sum = 0;
        for (int p = 0; p < kClusterCtas; ++p) sum += cluster.map_shared_rank(s_cnt, p)[R + tid];
        tprdma[s * NN + tid] = sum;
    }
    cluster.sync();  // keep every CTA's shared memory alive until the sums are read
}

// grid (kClusterCtas, R), cluster (kClusterCtas, 1, 1).
__global__ void __launch_bounds__(kLayoutThreads)
    get_dispatch_layout_kernel(const int64_t* __restrict__ topk_idx, const int32_t* __restrict__ rank_mask, int R,
                               int T, int K, int E, int EL, int32_t* __restrict__ tpr, int32_t* __restrict__ tprdma,
                               int32_t* __restrict__ tpe, uint8_t* __restrict__ itr, int32_t* status) {
    pdl_enter();
    extern __shared__ int32_t s_expert[];  // [E]
    __shared__ int32_t s_cnt[kMaxColumns];
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = lane_id();
    const uint32_t rmask = __ballot_sync(kFullMask, rank_mask != nullptr && lane < R && __ldg(rank_mask + lane) != 0);
    layout_source(cluster, blockIdx.y, static_cast<int>(cluster.block_rank()), topk_idx, rmask, R, T, K, E, EL, tpr,
                  tprdma, tpe, itr, status, s_expert, s_cnt);
}

// The summary of the dispatch record: rank_prefix_matrix, num_recv and the aligned
// per-expert receive counts (cluster R of the notify grid).
__device__ __forceinline__ void notify_summary(int q, int R, int E, int A, int64_t cap,
                                               const int32_t* __restrict__ tpr, const int32_t* __restrict__ tpe,
                                               int32_t* __restrict__ rank_prefix, int32_t* __restrict__ num_recv,
                                               int32_t* __restrict__ num_recv_per_expert, int32_t* status) {
    const int tid = threadIdx.x;
    const int per = kNotifyThreads * kClusterCtas;
    for (int r = q * kNotifyThreads + tid; r < R; r += per) {
        int32_t acc = 0;
        for (int sp = 0; sp < R; ++sp) {
            acc += __ldcg(tpr + sp * R + r);
            rank_prefix[sp * R + r] = acc;
        }
        num_recv[r] = acc;
        if (acc > cap) report(status, EP_ERR_CAPACITY);
    }
    for (int e = q * kNotifyThreads + tid; e < E; e += per) {
        int64_t sum = 0;
        for (int sp = 0; sp < R; ++sp) sum += __ldcg(tpe + static_cast<int64_t>(sp) * E + e);
        num_recv_per_expert[e] = static_cast<int32_t>(((sum + A - 1) / A) * A);
    }
}

// The rows of source s, CTA q of its cluster, given the slice's hits per column in s_cnt (every
// CTA of the cluster has filled its s_cnt before this is entered): send_head, recv_src_idx, the
// channel prefix matrices and, with NN > 0 node columns, the node-level channel prefix matrix.
__device__ __forceinline__ void notify_source(const cg::cluster_group& cluster, int s, int q, int R, int NN, int T,
                                              int C, int64_t cap, const int32_t* __restrict__ tpr,
                                              const uint8_t* __restrict__ itr, int32_t* __restrict__ channel_prefix,
                                              int32_t* __restrict__ recv_channel_prefix,
                                              int32_t* __restrict__ rdma_channel_prefix,
                                              int32_t* __restrict__ send_head, int32_t* __restrict__ recv_src_idx,
                                              int32_t* status, const int32_t* s_cnt) {
    __shared__ int32_t s_base[kMaxRanks];                  // rows taken by earlier sources
    __shared__ int32_t s_before[kMaxColumns];              // hits of this source before the current round
    __shared__ int32_t s_warp[kMaxColumns][kNotifyWarps];  // per-warp counts -> exclusive prefixes
    __shared__ int32_t s_total[kMaxColumns];               // hits of the current round
    static_assert(kNotifyWarps == kWarpSize, "the column scan gives one lane per warp");
    static_assert(kMaxColumns <= kNotifyThreads, "one thread per column");
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int warp = tid / kWarpSize;
    const int NC = R + NN;
    int lo, hi;
    cluster_slice(T, q, lo, hi);
    const uint8_t* itr_s = itr + static_cast<int64_t>(s) * T * R;
    int32_t* head_s = send_head + static_cast<int64_t>(s) * T * R;

    // Hits before this slice: earlier slices of this source; rows before it also count earlier sources.
    if (tid < NC) {
        int32_t before = 0;
        for (int p = 0; p < q; ++p) before += cluster.map_shared_rank(s_cnt, p)[tid];
        s_before[tid] = before;
    }
    if (tid < R) {
        int32_t base = 0;
        for (int sp = 0; sp < s; ++sp) base += __ldcg(tpr + sp * R + tid);
        s_base[tid] = base;
        if (q == kClusterCtas - 1) {
            // this slice ends the source: the per-source total must match the counts
            const int32_t total = s_before[tid] + s_cnt[tid];
            if (total != __ldcg(tpr + s * R + tid)) report(status, EP_ERR_INCONSISTENT);
        }
    }
    cluster.sync();  // peers are done reading this CTA's s_cnt

    const int chunk = max(1, (T + C - 1) / C);
    const unsigned lt = lanemask_lt();
    for (int t0 = lo; t0 < hi; t0 += kNotifyThreads) {
        const int t = t0 + tid;
        const bool live = t < hi;
        const uint32_t m = live ? load_rank_mask(itr_s + static_cast<int64_t>(t) * R, R) : 0u;
        for (int col = 0; col < NC; ++col) {
            const unsigned b = __ballot_sync(kFullMask, column_bit(m, col, R));
            if (lane == 0) s_warp[col][warp] = __popc(b);
        }
        __syncthreads();
        // warp w scans columns w, w + 32, ...: exclusive prefix over the warps of this round
        for (int col = warp; col < NC; col += kNotifyWarps) {
            const int32_t v = s_warp[col][lane];
            int32_t incl = v;
#pragma unroll
            for (int off = 1; off < kWarpSize; off <<= 1) {
                const int32_t o = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += o;
            }
            s_warp[col][lane] = s_before[col] + incl - v;
            if (lane == kWarpSize - 1) s_total[col] = incl;
        }
        __syncthreads();
        int32_t rows[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r >= R) break;
            const bool bit = (m >> r) & 1u;
            const unsigned b = __ballot_sync(kFullMask, bit);
            const int32_t excl = s_warp[r][warp] + __popc(b & lt);  // hits of (s -> r) before t
            rows[r] = bit ? s_base[r] + excl : -1;
            if (live && (t % chunk) == 0) {
                const int c = t / chunk;
                recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = s_base[r] + excl;
                if (c > 0) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c - 1] = excl;
            }
        }
        for (int n = 0; n < NN; ++n) {  // node columns: tokens of s that reach node n, before t
            const unsigned b = __ballot_sync(kFullMask, column_bit(m, R + n, R));
            if (live && t > 0 && (t % chunk) == 0)
                rdma_channel_prefix[(static_cast<int64_t>(s) * NN + n) * C + t / chunk - 1] =
                    s_warp[R + n][warp] + __popc(b & lt);
        }
        if (live) {
            int32_t* dst = head_s + static_cast<int64_t>(t) * R;
            if ((R & 3) == 0) {
#pragma unroll
                for (int r = 0; r < kMaxRanks; r += 4) {
                    if (r >= R) break;
                    reinterpret_cast<int4*>(dst)[r / 4] = make_int4(rows[r], rows[r + 1], rows[r + 2], rows[r + 3]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < kMaxRanks; ++r) {
                    if (r >= R) break;
                    dst[r] = rows[r];
                }
            }
#pragma unroll
            for (int r = 0; r < kMaxRanks; ++r) {
                if (r >= R) break;
                if (rows[r] >= 0 && rows[r] < cap) recv_src_idx[static_cast<int64_t>(r) * cap + rows[r]] = t;
            }
        }
        // the next round starts after this round's hits
        __syncthreads();
        if (tid < NC) s_before[tid] += s_total[tid];
        __syncthreads();
    }

    // Channels that end at T (or hold no token): written by the last slice of the source.
    if (q == kClusterCtas - 1 && tid < R) {
        const int r = tid;
        const int32_t total = __ldcg(tpr + s * R + r);
        for (int c = 0; c < C; ++c) {
            const int64_t start = min(static_cast<int64_t>(T), static_cast<int64_t>(c) * chunk);
            const int64_t end = min(static_cast<int64_t>(T), static_cast<int64_t>(c + 1) * chunk);
            if (end == T) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c] = total;
            if (start == T) recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = s_base[r] + total;
        }
    }
    if (q == kClusterCtas - 1 && tid >= R && tid < NC) {
        const int n = tid - R;  // s_before now holds the source's whole count for the column
        for (int c = 0; c < C; ++c)
            if (min(static_cast<int64_t>(T), static_cast<int64_t>(c + 1) * chunk) == T)
                rdma_channel_prefix[(static_cast<int64_t>(s) * NN + n) * C + c] = s_before[tid];
    }
}

// grid (kClusterCtas, R + 1), cluster (kClusterCtas, 1, 1).  Cluster s < R: the
// rows of source s, and with NN > 0 node columns its row of the node-level
// channel prefix matrix.  Cluster R: rank_prefix_matrix, num_recv and the
// aligned per-expert receive counts.  Counts are kept per column: R rank
// columns, then NN node columns (0 when there is no node-level record).
__global__ void __launch_bounds__(kNotifyThreads)
    dispatch_notify_kernel(int R, int NN, int T, int E, int C, int A, int64_t cap,
                           const int32_t* __restrict__ tpr, const uint8_t* __restrict__ itr,
                           const int32_t* __restrict__ tpe, int32_t* __restrict__ rank_prefix,
                           int32_t* __restrict__ channel_prefix, int32_t* __restrict__ recv_channel_prefix,
                           int32_t* __restrict__ rdma_channel_prefix, int32_t* __restrict__ num_recv,
                           int32_t* __restrict__ send_head, int32_t* __restrict__ recv_src_idx,
                           int32_t* __restrict__ num_recv_per_expert, int32_t* status) {
    pdl_enter();
    __shared__ int32_t s_cnt[kMaxColumns];  // hits of this CTA's slice, per column
    cg::cluster_group cluster = cg::this_cluster();
    const int q = static_cast<int>(cluster.block_rank());
    const int s = blockIdx.y;
    if (s == R) {
        notify_summary(q, R, E, A, cap, tpr, tpe, rank_prefix, num_recv, num_recv_per_expert, status);
        return;
    }
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int NC = R + NN;
    int lo, hi;
    cluster_slice(T, q, lo, hi);
    const uint8_t* itr_s = itr + static_cast<int64_t>(s) * T * R;
    if (tid < kMaxColumns) s_cnt[tid] = 0;
    __syncthreads();
    // Pass 1: hits of this slice per column.
    for (int t0 = lo; t0 < hi; t0 += kNotifyThreads) {
        const int t = t0 + tid;
        const uint32_t m = t < hi ? load_rank_mask(itr_s + static_cast<int64_t>(t) * R, R) : 0u;
        for (int col = 0; col < NC; ++col) {
            const unsigned b = __ballot_sync(kFullMask, column_bit(m, col, R));
            if (lane == 0 && b) atomicAdd(&s_cnt[col], __popc(b));
        }
    }
    cluster.sync();
    notify_source(cluster, s, q, R, NN, T, C, cap, tpr, itr, channel_prefix, recv_channel_prefix,
                  rdma_channel_prefix, send_head, recv_src_idx, status, s_cnt);
}

// One CTA, after the notify, R = 8 NN: recv_rdma_rank_prefix[r][m] for r = (n, l)
// = sum over m' <= m of the last channel of the node-level channel prefix
// matrix of source (m', l) towards node n.
__global__ void __launch_bounds__(kMaxRanks * kMaxNodes)
    node_prefix_kernel(int R, int NN, int C, const int32_t* __restrict__ rdma_channel_prefix,
                       int32_t* __restrict__ recv_rdma_rank_prefix) {
    pdl_enter();
    const int i = threadIdx.x;
    if (i >= R * NN) return;
    const int r = i / NN, m = i % NN;
    const int n = r / kRanksPerNode, l = r % kRanksPerNode;
    int32_t acc = 0;
    for (int mp = 0; mp <= m; ++mp)
        acc += rdma_channel_prefix[(static_cast<int64_t>(kRanksPerNode * mp + l) * NN + n) * C + C - 1];
    recv_rdma_rank_prefix[i] = acc;
}

// ---------------------------------------------------------------------------
// Layout and record in one pass: a single decoupled look-back scan.  The receive rows of every
// destination rank follow the (source, token) order, so one scan over the tokens of all sources,
// in that order, with one counter per destination rank, gives every row.  CTAs take tiles of
// kScanTile tokens of one source by ticket, in (source, token) order -- a CTA only ever waits for
// tiles whose CTAs started before it, so the waits end -- and for its tile:
//   1. marks is_token_in_rank, counts the slots per expert and, per column -- R destination ranks,
//      then ceil(R/8) nodes of 8 ranks -- the hits of each warp (ballots), then publishes the
//      tile's per-column totals with state "aggregate";
//   2. looks back over the earlier tiles, adding aggregates until one publishes state
//      "inclusive", then publishes its own inclusive prefixes: over all earlier tiles (rank
//      columns: the rows before the tile) and over this source's earlier tiles (every column:
//      the channel prefix matrices).  A tile reaches "inclusive" only after every earlier tile
//      published its aggregate, so the nearest inclusive tile ends both sums, however many
//      tiles a source has;
//   3. writes each token's send_head row (the exclusive prefix + the hits before the token in
//      the tile), recv_src_idx and the channel prefix entries (rank and, with whole nodes, node
//      columns) at channel starts.
// The last tile of a source writes the source's totals; the last CTA to finish writes the
// summary (num_recv, aligned per-expert receive counts and, with whole nodes, the node receive
// prefix) and resets the tickets for the next launch.  Every wait is bounded (EP_ERR_TIMEOUT).
// Published states carry the launch's epoch (a counter in the scratch that each launch
// advances), so stale states of an earlier launch never match and CUDA-graph replays need no
// reset.  With a rank mask, slots that start or end on a masked rank are left out as if they
// were -1 (a masked rank neither sends nor receives).
constexpr int kScanTile = 512;   // tokens per tile = threads per CTA (1024 measured 0.3 % slower on the step)
constexpr int kScanWarps = kScanTile / kWarpSize;
static_assert(kScanWarps <= kWarpSize, "the column scan gives one lane per warp");
constexpr int kScanAggregate = 1, kScanInclusive = 2;

// Per-tile words of the scratch, NC = R + ceil(R/8) columns: the state word, then the tile's
// per-column hits [NC], its inclusive prefix over all earlier tiles for the rank columns [R], its
// inclusive prefix over this source's tiles for every column [NC], and its expert histogram [E].
// The scratch starts with 4 words: [0] next ticket, [1] finished tiles, [2] epoch, [3] unused.
struct ScanWords {
    int NC, agg, incl, sincl, hist;
    int64_t per_tile;
};

__host__ __device__ __forceinline__ ScanWords scan_words(int R, int E) {
    ScanWords w;
    w.NC = R + (R + kRanksPerNode - 1) / kRanksPerNode;
    w.agg = 1;
    w.incl = w.agg + w.NC;
    w.sincl = w.incl + R;
    w.hist = w.sincl + w.NC;
    w.per_tile = w.hist + E;
    return w;
}

// All lanes of the calling warp wait (bounded) until tile k published at least `state` in this
// epoch; returns the state word, or 0 if the wait gave up.
__device__ __forceinline__ uint32_t scan_wait(const uint32_t* word, uint32_t epoch, uint32_t state) {
    for (uint32_t it = 0; it < kMaxWaitIterations; ++it) {
        const uint32_t f = ld_acquire_u32(word);
        if ((f >> 2) == (epoch & 0x3fffffffu) && (f & 3u) >= state) return f;
    }
    return 0u;
}

// Bit r set: rank r is masked (rank_mask may be NULL).  Every lane of the calling warp gets it.
__device__ __forceinline__ uint32_t masked_ranks(const int32_t* rank_mask, int R) {
    const int lane = lane_id();
    return __ballot_sync(kFullMask, rank_mask != nullptr && lane < R && __ldg(rank_mask + lane) != 0);
}

__global__ void __launch_bounds__(kScanTile)
    layout_scan_kernel(const int64_t* __restrict__ topk_idx, const int32_t* __restrict__ rank_mask, int R, int T,
                       int K, int E, int C, int A, int64_t cap, int32_t* __restrict__ tpr,
                       int32_t* __restrict__ tprdma, int32_t* __restrict__ tpe, uint8_t* __restrict__ itr,
                       int32_t* __restrict__ rank_prefix, int32_t* __restrict__ channel_prefix,
                       int32_t* __restrict__ recv_channel_prefix, int32_t* __restrict__ num_recv,
                       int32_t* __restrict__ send_head, int32_t* __restrict__ recv_src_idx,
                       int32_t* __restrict__ num_recv_per_expert, int32_t* __restrict__ rdma_channel_prefix,
                       int32_t* __restrict__ recv_rdma_rank_prefix, uint32_t* __restrict__ scratch,
                       int32_t* status) {
    pdl_enter();
    extern __shared__ int32_t s_hist[];                    // [E]: slots per expert
    __shared__ uint32_t s_mask[kScanTile];                 // destination ranks of each token of the tile
    __shared__ int32_t s_wpre[kMaxColumns][kScanWarps];    // per-warp hits -> exclusive prefix in the tile
    __shared__ int32_t s_agg[kMaxColumns];                 // the tile's hits per column
    __shared__ int32_t s_excl[kMaxRanks];                  // hits of every earlier tile (rows before the tile)
    __shared__ int32_t s_ws[kMaxColumns];                  // hits of this source's earlier tiles
    __shared__ int32_t s_tile, s_ok, s_last;
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x;
    const int lane = lane_id();
    const int warp = tid / kWarpSize;
    const int EL = E / R;
    const int NN = (R + kRanksPerNode - 1) / kRanksPerNode;
    const ScanWords W = scan_words(R, E);
    const int NC = W.NC;
    const int tiles_per_src = (T + kScanTile - 1) / kScanTile;
    const int n_tiles = R * tiles_per_src;
    uint32_t* tiles = scratch + 4;

    if (tid == 0) {
        s_tile = static_cast<int>(atomicAdd(scratch, 1u));
        s_epoch = ld_acquire_u32(scratch + 2);
        s_ok = 1;
    }
    for (int i = tid; i < E; i += kScanTile) s_hist[i] = 0;
    s_mask[tid] = 0u;
    const uint32_t rmask = masked_ranks(rank_mask, R);
    __syncthreads();
    const int tile = s_tile;
    const uint32_t epoch = s_epoch;
    const uint32_t tag = (epoch & 0x3fffffffu) << 2;
    const int s = tile / tiles_per_src;
    const int j = tile - s * tiles_per_src;
    const int t0 = j * kScanTile;
    const int len = min(kScanTile, T - t0);
    uint32_t* my = tiles + static_cast<int64_t>(tile) * W.per_tile;
    const bool src_masked = (rmask >> s) & 1u;

    // 1. the tile's layout: one flat walk over its top-k entries, several loads in flight
    const int64_t* idx_t = topk_idx + (static_cast<int64_t>(s) * T + t0) * K;
    const int64_t n_ent = static_cast<int64_t>(len) * K;
    for (int64_t i0 = tid; i0 < n_ent; i0 += static_cast<int64_t>(kLayoutUnroll) * kScanTile) {
        int64_t v[kLayoutUnroll];
#pragma unroll
        for (int u = 0; u < kLayoutUnroll; ++u) {
            const int64_t i = i0 + static_cast<int64_t>(u) * kScanTile;
            v[u] = i < n_ent ? __ldg(idx_t + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kLayoutUnroll; ++u) {
            const int64_t i = i0 + static_cast<int64_t>(u) * kScanTile;
            const int64_t e = v[u];
            if (i >= n_ent || e == -1) continue;
            if (e < 0 || e >= E) {
                report(status, EP_ERR_BAD_EXPERT);
                continue;
            }
            const int d = static_cast<int>(e) / EL;
            if (src_masked || ((rmask >> d) & 1u)) continue;  // a masked rank neither sends nor receives
            atomicAdd(&s_hist[e], 1);
            atomicOr(&s_mask[static_cast<int>(i / K)], 1u << d);
        }
    }
    __syncthreads();
    const bool live = tid < len;
    const int t = t0 + tid;
    const uint32_t m = live ? s_mask[tid] : 0u;
    if (live) store_rank_mask(itr + (static_cast<int64_t>(s) * T + t) * R, R, m);
    for (int c = 0; c < NC; ++c) {
        const unsigned b = __ballot_sync(kFullMask, column_bit(m, c, R));
        if (lane == 0) s_wpre[c][warp] = __popc(b);
    }
    __syncthreads();
    for (int c = warp; c < NC; c += kScanWarps) {  // exclusive prefix of column c's hits over the warps of the tile
        const int32_t v = lane < kScanWarps ? s_wpre[c][lane] : 0;
        int32_t incl = v;
#pragma unroll
        for (int off = 1; off < kWarpSize; off <<= 1) {
            const int32_t o = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane < kScanWarps) s_wpre[c][lane] = incl - v;
        if (lane == kWarpSize - 1) s_agg[c] = incl;
    }
    __syncthreads();
    // publish the aggregate (and the histogram the source's last tile sums)
    if (tid < NC) my[W.agg + tid] = static_cast<uint32_t>(s_agg[tid]);
    for (int i = tid; i < E; i += kScanTile) my[W.hist + i] = static_cast<uint32_t>(s_hist[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_u32(my, tag | kScanAggregate);

    // 2. look back: warp c sums column c's hits of the earlier tiles.  Lane i reads tile
    //    (tile - 1 - i) of a window of 32, so one round of loads covers the window; the sums stop
    //    at the nearest tile that published its inclusive prefixes -- for a rank column the prefix
    //    over all tiles, and for every column the prefix over its own source's tiles.
    for (int c = warp; c < NC; c += kScanWarps) {
        const bool rank_col = c < R;
        int32_t excl = 0, ws = 0;
        bool ok = true;
        for (int k0 = tile - 1; k0 >= 0; k0 -= kWarpSize) {
            const int k = k0 - lane;
            uint32_t f = 1u;
            int32_t agg = 0, inc = 0, sinc = 0;
            if (k >= 0) {
                const uint32_t* w = tiles + static_cast<int64_t>(k) * W.per_tile;
                f = scan_wait(w, epoch, kScanAggregate);
                if (f != 0u) {
                    agg = static_cast<int32_t>(__ldcg(w + W.agg + c));
                    if ((f & 3u) == kScanInclusive) {
                        if (rank_col) inc = static_cast<int32_t>(__ldcg(w + W.incl + c));
                        sinc = static_cast<int32_t>(__ldcg(w + W.sincl + c));
                    }
                }
            }
            if (__any_sync(kFullMask, f == 0u)) {
                ok = false;
                break;
            }
            const bool same = k >= 0 && k >= tile - j;  // tile k is an earlier tile of this source
            const unsigned inclusive = __ballot_sync(kFullMask, k >= 0 && (f & 3u) == kScanInclusive);
            const int first = inclusive ? __ffs(inclusive) - 1 : kWarpSize;
            int32_t part = lane < first ? agg : (lane == first ? inc : 0);
            int32_t spart = same ? (lane < first ? agg : (lane == first ? sinc : 0)) : 0;
#pragma unroll
            for (int off = kWarpSize / 2; off > 0; off >>= 1) {
                part += __shfl_xor_sync(kFullMask, part, off);
                spart += __shfl_xor_sync(kFullMask, spart, off);
            }
            excl += part;
            ws += spart;
            if (inclusive) break;
        }
        if (lane == 0) {
            if (rank_col) {
                s_excl[c] = excl;
                my[W.incl + c] = static_cast<uint32_t>(excl + s_agg[c]);
            }
            s_ws[c] = ws;
            my[W.sincl + c] = static_cast<uint32_t>(ws + s_agg[c]);
            if (!ok) s_ok = 0;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        st_release_u32(my, tag | kScanInclusive);  // published even after a timeout, so no later tile waits on it
        if (!s_ok) report(status, EP_ERR_TIMEOUT);
    }

    // 3. rows, recv_src_idx and the channel prefix entries of the tile's tokens
    if (s_ok) {
        const int chunk = max(1, (T + C - 1) / C);
        const unsigned lt = lanemask_lt();
        const bool channel_start = live && (t % chunk) == 0;
        int32_t rows[kMaxRanks];
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r >= R) break;
            const bool bit = (m >> r) & 1u;
            const unsigned b = __ballot_sync(kFullMask, bit);
            const int32_t before = s_wpre[r][warp] + __popc(b & lt);  // hits of (s -> r) in the tile before t
            const int32_t row = s_excl[r] + before;
            rows[r] = bit ? row : -1;
            if (channel_start) {
                const int c = t / chunk;
                recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = row;
                if (c > 0) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c - 1] = s_ws[r] + before;
            }
        }
        if (rdma_channel_prefix != nullptr) {  // node columns: tokens of s that reach node n, before t
            for (int n = 0; n < NN; ++n) {
                const unsigned b = __ballot_sync(kFullMask, column_bit(m, R + n, R));
                if (channel_start && t > 0)
                    rdma_channel_prefix[(static_cast<int64_t>(s) * NN + n) * C + t / chunk - 1] =
                        s_ws[R + n] + s_wpre[R + n][warp] + __popc(b & lt);
            }
        }
        if (live) {
            int32_t* dst = send_head + (static_cast<int64_t>(s) * T + t) * R;
            if ((R & 3) == 0) {
#pragma unroll
                for (int r = 0; r < kMaxRanks; r += 4) {
                    if (r >= R) break;
                    reinterpret_cast<int4*>(dst)[r / 4] = make_int4(rows[r], rows[r + 1], rows[r + 2], rows[r + 3]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < kMaxRanks; ++r) {
                    if (r >= R) break;
                    dst[r] = rows[r];
                }
            }
#pragma unroll
            for (int r = 0; r < kMaxRanks; ++r) {
                if (r >= R) break;
                if (rows[r] >= 0 && rows[r] < cap) recv_src_idx[static_cast<int64_t>(r) * cap + rows[r]] = t;
            }
        }
        // the source's last tile: its totals, the channels that end at T, its expert and node counts
        if (j == tiles_per_src - 1) {
            if (tid < R) {
                const int r = tid;
                const int32_t total = s_ws[r] + s_agg[r];
                const int32_t base = s_excl[r] - s_ws[r];
                tpr[s * R + r] = total;
                rank_prefix[s * R + r] = s_excl[r] + s_agg[r];
                for (int c = 0; c < C; ++c) {
                    const int64_t start = min(static_cast<int64_t>(T), static_cast<int64_t>(c) * chunk);
                    const int64_t end = min(static_cast<int64_t>(T), static_cast<int64_t>(c + 1) * chunk);
                    if (end == T) channel_prefix[(static_cast<int64_t>(s) * R + r) * C + c] = total;
                    if (start == T) recv_channel_prefix[(static_cast<int64_t>(r) * R + s) * C + c] = base + total;
                }
            } else if (tid < NC) {
                const int n = tid - R;
                const int32_t total = s_ws[tid] + s_agg[tid];
                if (tprdma != nullptr) tprdma[s * NN + n] = total;
                if (rdma_channel_prefix != nullptr)
                    for (int c = 0; c < C; ++c)
                        if (min(static_cast<int64_t>(T), static_cast<int64_t>(c + 1) * chunk) == T)
                            rdma_channel_prefix[(static_cast<int64_t>(s) * NN + n) * C + c] = total;
            }
            // every earlier tile of the source has published its histogram: the look-back above
            // reached an inclusive tile, and a tile is inclusive only after all earlier ones
            for (int i = tid; i < E; i += kScanTile) {
                int32_t sum = s_hist[i];
                for (int k = tile - j; k < tile; ++k)
                    sum += static_cast<int32_t>(__ldcg(tiles + static_cast<int64_t>(k) * W.per_tile + W.hist + i));
                tpe[static_cast<int64_t>(s) * E + i] = sum;
            }
        }
    }

    // the last CTA to finish: summary, and the next launch's tickets
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(scratch + 1, 1u) == static_cast<uint32_t>(n_tiles) - 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int r = tid; r < R; r += kScanTile) {
        const int32_t total = __ldcg(rank_prefix + (R - 1) * R + r);
        num_recv[r] = total;
        if (total > cap) report(status, EP_ERR_CAPACITY);
    }
    for (int e = tid; e < E; e += kScanTile) {
        int64_t sum = 0;
        for (int sp = 0; sp < R; ++sp) sum += __ldcg(tpe + static_cast<int64_t>(sp) * E + e);
        num_recv_per_expert[e] = static_cast<int32_t>(((sum + A - 1) / A) * A);
    }
    if (recv_rdma_rank_prefix != nullptr && tid < R * NN) {
        // rank (n, l) receives over RDMA the tokens of the sources (m, l) that reach node n
        const int r = tid / NN, mm = tid % NN;
        const int n = r / kRanksPerNode, l = r % kRanksPerNode;
        int32_t acc = 0;
        for (int mp = 0; mp <= mm; ++mp)
            acc += __ldcg(rdma_channel_prefix + (static_cast<int64_t>(kRanksPerNode * mp + l) * NN + n) * C + C - 1);
        recv_rdma_rank_prefix[tid] = acc;
    }
    if (tid == 0) {
        scratch[0] = 0u;
        scratch[1] = 0u;
        __threadfence();
        st_release_u32(scratch + 2, epoch + 1u);
    }
}

}  // namespace

cudaError_t launch_get_dispatch_layout(const int64_t* topk_idx, const int32_t* rank_mask, int R, int T, int K, int E,
                                       int32_t* tpr, int32_t* tprdma, int32_t* tpe, uint8_t* itr, int32_t* status,
                                       cudaStream_t stream) {
    return launch_kernel(get_dispatch_layout_kernel, dim3(kClusterCtas, R, 1), dim3(kLayoutThreads, 1, 1),
                         sizeof(int32_t) * static_cast<size_t>(E), stream, kClusterCtas, topk_idx, rank_mask, R, T, K,
                         E, E / R, tpr, tprdma, tpe, itr, status);
}

cudaError_t launch_dispatch_notify(int R, int T, int E, int C, int A, int64_t cap, const int32_t* tpr,
                                   const uint8_t* itr, const int32_t* tpe, int32_t* rank_prefix,
                                   int32_t* channel_prefix, int32_t* recv_channel_prefix, int32_t* num_recv,
                                   int32_t* send_head, int32_t* recv_src_idx, int32_t* num_recv_per_expert,
                                   int32_t* rdma_channel_prefix, int32_t* recv_rdma_rank_prefix, int32_t* status,
                                   cudaStream_t stream) {
    const bool nodes = rdma_channel_prefix != nullptr && recv_rdma_rank_prefix != nullptr;
    if (nodes && (R <= kRanksPerNode || R % kRanksPerNode != 0)) return cudaErrorInvalidValue;
    const int NN = nodes ? R / kRanksPerNode : 0;
    cudaError_t err = launch_kernel(dispatch_notify_kernel, dim3(kClusterCtas, R + 1, 1), dim3(kNotifyThreads, 1, 1),
                                    0, stream, kClusterCtas, R, NN, T, E, C, A, cap, tpr, itr, tpe, rank_prefix,
                                    channel_prefix, recv_channel_prefix, rdma_channel_prefix, num_recv, send_head,
                                    recv_src_idx, num_recv_per_expert, status);
    if (err != cudaSuccess || !nodes) return err;
    return launch_kernel(node_prefix_kernel, dim3(1, 1, 1), dim3(kMaxRanks * kMaxNodes, 1, 1), 0, stream, 1, R, NN, C,
                         static_cast<const int32_t*>(rdma_channel_prefix), recv_rdma_rank_prefix);
}

size_t layout_scan_scratch_words(int R, int E, int max_tokens) {
    const int64_t tiles = static_cast<int64_t>(R) * ((max_tokens + kScanTile - 1) / kScanTile);
    return static_cast<size_t>(4 + tiles * scan_words(R, E).per_tile);
}

cudaError_t launch_layout_scan(const int64_t* topk_idx, const int32_t* rank_mask, int R, int T, int K, int E, int C,
                               int A, int64_t cap, int32_t* tpr, int32_t* tprdma, int32_t* tpe, uint8_t* itr,
                               int32_t* rank_prefix, int32_t* channel_prefix, int32_t* recv_channel_prefix,
                               int32_t* num_recv, int32_t* send_head, int32_t* recv_src_idx,
                               int32_t* num_recv_per_expert, int32_t* rdma_channel_prefix,
                               int32_t* recv_rdma_rank_prefix, uint32_t* scratch, int32_t* status,
                               cudaStream_t stream) {
    const bool nodes = rdma_channel_prefix != nullptr || recv_rdma_rank_prefix != nullptr;
    if (T < 1 || (nodes && (rdma_channel_prefix == nullptr || recv_rdma_rank_prefix == nullptr ||
                            R <= kRanksPerNode || R % kRanksPerNode != 0)))
        return cudaErrorInvalidValue;
    const int64_t n_tiles = static_cast<int64_t>(R) * ((T + kScanTile - 1) / kScanTile);
    if (n_tiles > INT32_MAX) return cudaErrorInvalidValue;
    const size_t smem = sizeof(int32_t) * static_cast<size_t>(E);
    return launch_kernel(layout_scan_kernel, dim3(static_cast<unsigned>(n_tiles)), dim3(kScanTile), smem, stream, 1,
                         topk_idx, rank_mask, R, T, K, E, C, A, cap, tpr, tprdma, tpe, itr, rank_prefix, channel_prefix,
                         recv_channel_prefix, num_recv, send_head, recv_src_idx, num_recv_per_expert,
                         rdma_channel_prefix, recv_rdma_rank_prefix, scratch, status);
}

}  // namespace ep
