// Receiving-side row plan (the layout the grouped GEMM reads its rows in).
//
// Rows of local expert e are ordered by (source rank, token, slot): the entry
// (rk, t, j) of the routing table goes to row
//     base[e][rk] + #{entries (rk, t', j') routed to e with (t', j') before (t, j)}.
// Entries are stored in exactly that order (rank-major, then token, then slot), so
// each source rank's entries are cut into C contiguous chunks, one warp per chunk:
//  1. every warp counts its chunk's entries per local expert;
//  2. the block turns the counts into expert offsets, segment offsets and send
//     counts (a scan in (expert, source rank) order) and gives every chunk its
//     first row per expert;
//  3. every warp walks its chunk again and places each entry, stably (lanes with
//     the same expert are ranked with match_any), so the plan is deterministic.
// Untimed set-up work: it stands in for the dispatch step that precedes the
// down-projection.
#include "ep_internal.h"

namespace ep {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanUnroll = 8;  // 32-entry steps whose routing ids are loaded at once

// The local expert of each of this lane's next kPlanUnroll entries (one per 32-entry
// step starting at i0), or -1 (routed elsewhere, past the chunk, or malformed).
__device__ __forceinline__ void load_keys(const int32_t *ids, int64_t i0, int64_t hi, int lane,
                                          int n_experts, int El, int my_rank,
                                          int (&key)[kPlanUnroll], bool &bad)
{
    int g[kPlanUnroll];
#pragma unroll
    for (int u = 0; u < kPlanUnroll; ++u) {
        const int64_t i = i0 + 32 * u + lane;
        g[u] = i < hi ? __ldg(ids + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kPlanUnroll; ++u) {
        const int64_t i = i0 + 32 * u + lane;
        key[u] = -1;
        if (i < hi) {
            if (g[u] < 0 || g[u] >= n_experts)
                bad = true;
            else if (g[u] / El == my_rank)
                key[u] = g[u] % El;
        }
    }
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const PlanParams p)
{
    extern __shared__ int smem[];
    const int R = p.n_ranks, El = p.El, k = p.top_k;
    const int C = kPlanWarps / R;           // chunks per source rank (>= 4)
    int *chunk = smem;                      // [R][C][El]: counts, then first rows
    int *seg = chunk + R * C * El;          // [El][R]: rows per (expert, source rank)
    __shared__ int s_warp_sum[kPlanWarps];
    __shared__ int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < R * C * El; i += blockDim.x)
        chunk[i] = 0;
    __syncthreads();

    const int64_t Tk = static_cast<int64_t>(p.T) * k;
    const int64_t L = (Tk + C - 1) / C;     // entries per chunk
    const int n_experts = R * El;
    const bool has_chunk = warp < R * C;  // R * C <= 32: spare warps only help with steps 2
    const int rk = has_chunk ? warp / C : 0, c = has_chunk ? warp % C : 0;
    const int64_t lo = has_chunk ? c * L : 0;
    const int64_t hi = has_chunk ? (lo + L < Tk ? lo + L : Tk) : 0;
    const int32_t *ids = p.topk_ids + static_cast<int64_t>(rk) * Tk;
    int *cnt = chunk + (rk * C + c) * El;

    // ---- 1. per-chunk counts
    const unsigned lt_mask = (1u << lane) - 1u;
    bool bad_id = false;
    for (int64_t i0 = lo; i0 < hi; i0 += 32 * kPlanUnroll) {
        int key[kPlanUnroll];
        load_keys(ids, i0, hi, lane, n_experts, El, p.my_rank, key, bad_id);
#pragma unroll
        for (int u = 0; u < kPlanUnroll; ++u) {
            const unsigned peers = __match_any_sync(0xffffffffu, key[u]);
            if (key[u] >= 0 && (peers & lt_mask) == 0)
                cnt[key[u]] += __popc(peers);  // the lowest lane of each group; chunks are private
            __syncwarp();
        }
    }
    if (__syncthreads_or(bad_id) && threadIdx.x == 0)
        atomicOr(p.status, EP_STATUS_ROUTING);

    // ---- 2. offsets: seg[e][rk] = rows of (e, rk); exclusive scan in (e, rk) order
    for (int q = threadIdx.x; q < El * R; q += blockDim.x) {
        const int e = q / R, r = q % R;
        int s = 0;
        for (int cc = 0; cc < C; ++cc)
            s += chunk[(r * C + cc) * El + e];
        seg[q] = s;
    }
    __syncthreads();
    // block-wide exclusive scan of seg[0 .. El*R): each thread scans a contiguous run
    const int n = El * R;
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int a0 = threadIdx.x * per, a1 = a0 + per < n ? a0 + per : n;
    int local = 0;
    for (int q = a0; q < a1; ++q)
        local += seg[q];
    int incl = local;  // inclusive scan of the per-thread sums across the block
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += v;
    }
    if (lane == 31)
        s_warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = s_warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d)
                v += u;
        }
        s_warp_sum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int total = s_warp_sum[kPlanWarps - 1];
    int run = (warp > 0 ? s_warp_sum[warp - 1] : 0) + incl - local;  // exclusive start
    if (threadIdx.x == 0)
        s_ok = static_cast<int64_t>(total) <= p.max_rows;
    __syncthreads();
    const bool ok = s_ok;
    for (int q = a0; q < a1; ++q) {
        const int e = q / R, r = q % R;
        const int rows = seg[q];
        p.seg_offsets[e * (R + 1) + r] = ok ? run : 0;
        p.send_counts[q] = ok ? rows : 0;
        if (r == 0)
            p.expert_offsets[e] = ok ? run : 0;
        if (r == R - 1)
            p.seg_offsets[e * (R + 1) + R] = ok ? run + rows : 0;
        seg[q] = run;  // now the first row of (e, r)
        run += rows;
    }
    if (threadIdx.x == 0) {
        p.expert_offsets[El] = ok ? total : 0;
        *p.m_total = ok ? total : 0;
        if (!ok)
            atomicOr(p.status, EP_STATUS_CAPACITY);  // does not fit: empty plan, flagged
    }
    __syncthreads();
    if (!ok)
        return;
    // first row of every (chunk, expert): the segment start plus earlier chunks' rows
    for (int q = threadIdx.x; q < El * R; q += blockDim.x) {
        const int e = q / R, r = q % R;
        int row = seg[e * R + r];
        for (int cc = 0; cc < C; ++cc) {
            int *x = &chunk[(r * C + cc) * El + e];
            const int rows = *x;
            *x = row;
            row += rows;
        }
    }
    __syncthreads();

    // ---- 3. placement
    if (!has_chunk)
        return;
    bool unused = false;
    for (int64_t i0 = lo; i0 < hi; i0 += 32 * kPlanUnroll) {
        int key[kPlanUnroll];
        load_keys(ids, i0, hi, lane, n_experts, El, p.my_rank, key, unused);
#pragma unroll
        for (int u = 0; u < kPlanUnroll; ++u) {
            const unsigned peers = __match_any_sync(0xffffffffu, key[u]);
            int pos = 0;
            if (key[u] >= 0)
                pos = cnt[key[u]] + __popc(peers & lt_mask);
            __syncwarp();
            if (key[u] >= 0 && (peers & lt_mask) == 0)
                cnt[key[u]] += __popc(peers);
            __syncwarp();
            if (key[u] >= 0) {
                const int64_t i = i0 + 32 * u + lane;
                const int t = static_cast<int>(i / k), j = static_cast<int>(i % k);
                reinterpret_cast<int2 *>(p.src_info)[pos] = make_int2(t, j);
                p.gather_idx[pos] = static_cast<int32_t>(rk * Tk + i);
            }
        }
    }
}

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s)
{
    const int C = kPlanWarps / p.n_ranks;
    const size_t smem =
        sizeof(int) * (static_cast<size_t>(p.n_ranks) * C * p.El + static_cast<size_t>(p.El) *
                                                                        p.n_ranks);
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(
            plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess)
            return err;
    }
    plan_kernel<<<1, kPlanThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
