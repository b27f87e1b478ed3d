// Receiving-side row plan (the layout the grouped GEMM reads its rows in).
//
// One block, one warp per source rank. Pass 1 counts the rows of every
// (local expert, source rank) pair; one thread turns the counts into expert and
// segment offsets; pass 2 walks each source rank's routing entries in order and
// gives every entry routed here its row, stably (token, then slot), so the
// result is deterministic. Untimed set-up work: it stands in for the dispatch
// step that precedes the down-projection.
#include "ep_internal.h"

namespace ep {

__global__ void __launch_bounds__(EP_MAX_RANKS * 32, 1) plan_kernel(const PlanParams p)
{
    extern __shared__ int smem[];
    const int R = p.n_ranks, El = p.El, k = p.top_k;
    int *counts = smem;              // [El][R]
    int *base = counts + El * R;     // [El][R]
    int *running = base + El * R;    // [R][El]
    __shared__ int s_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < El * R; i += blockDim.x) {
        counts[i] = 0;
        running[i] = 0;
    }
    __syncthreads();

    const int64_t Tk = static_cast<int64_t>(p.T) * k;
    const int n_experts = R * El;
    bool bad_id = false;
    if (warp < R) {
        const int32_t *ids = p.topk_ids + warp * Tk;
        for (int64_t i = lane; i < Tk; i += 32) {
            const int g = ids[i];
            if (g < 0 || g >= n_experts) {
                bad_id = true;
                continue;
            }
            if (g / El == p.my_rank)
                atomicAdd(&counts[(g % El) * R + warp], 1);
        }
    }
    if (__syncthreads_or(bad_id) && threadIdx.x == 0)
        atomicOr(p.status, EP_STATUS_ROUTING);

    if (threadIdx.x == 0) {
        int64_t row = 0;
        for (int e = 0; e < El; ++e) {
            p.expert_offsets[e] = static_cast<int32_t>(row);
            for (int rk = 0; rk < R; ++rk) {
                base[e * R + rk] = static_cast<int>(row);
                p.seg_offsets[e * (R + 1) + rk] = static_cast<int32_t>(row);
                p.send_counts[e * R + rk] = counts[e * R + rk];
                row += counts[e * R + rk];
            }
            p.seg_offsets[e * (R + 1) + R] = static_cast<int32_t>(row);
        }
        p.expert_offsets[El] = static_cast<int32_t>(row);
        s_ok = row <= p.max_rows;
        if (!s_ok) {
            // does not fit: publish an empty plan and flag it
            for (int e = 0; e <= El; ++e)
                p.expert_offsets[e] = 0;
            for (int i = 0; i < El * (R + 1); ++i)
                p.seg_offsets[i] = 0;
            for (int i = 0; i < El * R; ++i)
                p.send_counts[i] = 0;
            atomicOr(p.status, EP_STATUS_CAPACITY);
            row = 0;
        }
        *p.m_total = static_cast<int32_t>(row);
    }
    __syncthreads();
    if (!s_ok || warp >= R)
        return;

    const unsigned lt_mask = (1u << lane) - 1u;
    const int32_t *ids = p.topk_ids + warp * Tk;
    int *run = running + warp * El;
    for (int64_t c = 0; c < Tk; c += 32) {
        const int64_t i = c + lane;
        int key = -1;  // local expert of this entry, or -1
        if (i < Tk) {
            const int g = ids[i];
            if (g >= 0 && g < n_experts && g / El == p.my_rank)
                key = g % El;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        int pos = 0;
        if (key >= 0)
            pos = base[key * R + warp] + run[key] + __popc(peers & lt_mask);
        __syncwarp();
        if (key >= 0 && (peers & lt_mask) == 0)  // lowest lane of the group advances the count
            run[key] += __popc(peers);
        __syncwarp();
        if (key >= 0) {
            const int t = static_cast<int>(i / k), j = static_cast<int>(i % k);
            p.src_info[2 * static_cast<int64_t>(pos) + 0] = t;
            p.src_info[2 * static_cast<int64_t>(pos) + 1] = j;
            p.gather_idx[pos] = static_cast<int32_t>(warp * Tk + i);
        }
    }
}

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s)
{
    const size_t smem = sizeof(int) * 3 * static_cast<size_t>(p.El) * p.n_ranks;
    plan_kernel<<<1, EP_MAX_RANKS * 32, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
