// The send step on its own: the unfused comparator of the fused GEMM + send.
//
// "EpiloguePeerSink" with the sink disabled stores the output tile to the local C
// (the null sink); this kernel then does what the fused epilogue does in place:
// every row m < m_total goes to the receive buffer of the rank that owns its
// token, at (src_idx*top_k + src_topk)*msg_bytes ("P3PeerSendConfig"), and the
// rank is signalled as "ep_signal_completion" does: count words, then the rank
// flag (or, per expert, epoch-tagged count words). One launch sends every local
// expert, so instead of an election per expert the last thread block to finish
// publishes all count words and the flags.
//
// Memory-bound copy: one warp per row at a time, 16-byte loads and stores, each
// row's bytes contiguous on both sides; grid = a few blocks per SM.
#include "ep_internal.h"
#include "ep_ptx.cuh"

namespace ep {

constexpr int kScatterThreads = 256;

// Destination of row m, or nullptr (EP_STATUS_BOUNDS raised) when the plan sends
// it outside the receive buffer.
__device__ __forceinline__ uint8_t *scatter_destination(const ScatterParams &p, int m)
{
    int lo = 0, hi = p.El - 1;  // the last expert whose first row is <= m owns m
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.expert_offsets + mid) <= m)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int R = p.n_ranks;
    const int *seg = p.seg_offsets + lo * (R + 1);
    int dst = -1;
    for (int rk = 0; rk < R; ++rk)
        if (m >= __ldg(seg + rk) && m < __ldg(seg + rk + 1))
            dst = rk;
    const int2 si = __ldg(reinterpret_cast<const int2 *>(p.src_info) + m);
    if (dst < 0 || si.x < 0 || si.x >= p.max_tokens || si.y < 0 || si.y >= p.top_k)
        return nullptr;
    return p.recv_buf[dst] + (static_cast<int64_t>(si.x) * p.top_k + si.y) * p.msg_bytes;
}

__global__ void __launch_bounds__(kScatterThreads) scatter_kernel(const ScatterParams p)
{
    const int lane = threadIdx.x & 31;
    const int warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int n_warps = (gridDim.x * blockDim.x) >> 5;
    int64_t m_total = __ldg(p.expert_offsets + p.El);
    m_total = m_total < 0 ? 0 : (m_total > p.max_rows ? p.max_rows : m_total);
    const int chunks = p.N / 8;  // 16-byte pieces of a bf16 row

    bool bad = false;
    for (int64_t m = warp_id; m < m_total; m += n_warps) {
        uint8_t *dst = scatter_destination(p, static_cast<int>(m));
        if (dst == nullptr) {
            bad = true;
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(p.C + m * p.N * 2);
        for (int c = lane; c < chunks; c += 32)
            st_global_v4(dst + c * 16, __ldg(src + c));
    }
    if (bad && lane == 0)
        atomicOr(p.status, EP_STATUS_BOUNDS);

    // every block releases its rows (gpu scope) through the block counter; the last
    // one acquires them all (gpu scope) and signals every expert towards every
    // destination behind system-scope releases, which carry the rows cumulatively
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const bool last = atomicAdd(p.block_counter, 1) == static_cast<int>(gridDim.x) - 1;
        if (last)
            fence_acq_rel_gpu();
        s_last = last;
    }
    __syncthreads();
    if (!s_last)
        return;
    const int R = p.n_ranks;
    if (p.signal_mode == EP_SIGNAL_PER_EXPERT) {
        // every count word is its expert's arrival signal, tagged with the epoch and
        // released by a system-scope fence of the thread that stores it (after the
        // barrier that orders it behind the acquire above); no rank flag
        const uint64_t tag = (p.epoch & 0xFFFFFFFFull) << 32;
        if (threadIdx.x < p.El * R)
            fence_acq_rel_sys();
        for (int i = threadIdx.x; i < p.El * R; i += blockDim.x) {
            const int e = i / R, dst = i % R;
            st_relaxed_sys_u64(p.recv_count[dst] + static_cast<int64_t>(e) * R + p.my_rank,
                               tag | static_cast<uint32_t>(__ldg(p.send_counts + e * R + dst)));
        }
        __syncthreads();
        if (threadIdx.x == 0)
            *reinterpret_cast<volatile int *>(p.block_counter) = 0;
        return;
    }
    for (int i = threadIdx.x; i < p.El * R; i += blockDim.x) {
        const int e = i / R, dst = i % R;
        volatile uint64_t *w = p.recv_count[dst] + static_cast<int64_t>(e) * R + p.my_rank;
        *w = static_cast<uint64_t>(__ldg(p.send_counts + e * R + dst));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        fence_acq_rel_sys();  // every row and count word before any flag
        for (int dst = 0; dst < R; ++dst)
            st_relaxed_sys_u64(p.recv_count[dst] + static_cast<int64_t>(p.El) * R + p.my_rank,
                               p.epoch);
        *reinterpret_cast<volatile int *>(p.block_counter) = 0;  // re-armed for the next call
    }
}

cudaError_t launch_scatter(const ScatterParams &p, int num_sms, cudaStream_t s)
{
    scatter_kernel<<<4 * num_sms, kScatterThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
