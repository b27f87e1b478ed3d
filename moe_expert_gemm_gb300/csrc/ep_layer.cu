// The steps of a MoE layer that precede the fused down-projection, for running a
// whole layer on these kernels: the dispatch (every routed token row brought to
// the rank that owns its expert, in plan order) and the gated activation between
// the up/gate projection and the down-projection. The up/gate projection itself is
// the grouped GEMM with the sink disabled (rows to a local buffer).
//
// Both are memory-bound copies / elementwise passes: one warp per row at a time,
// 16-byte accesses, a few blocks per SM.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"

namespace ep {

constexpr int kLayerThreads = 256;

// A_in[m] = x_{rk}[t] for the row m = (source rank rk, token t, slot j) of the plan
// (gather_idx[m] = (rk*T + t)*top_k + j).
__global__ void __launch_bounds__(kLayerThreads) dispatch_gather_kernel(const DispatchParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    int64_t m_total = __ldg(p.expert_offsets + p.El);
    m_total = m_total < 0 ? 0 : (m_total > p.max_rows ? p.max_rows : m_total);
    const int chunks = p.hidden / 8;  // 16-byte pieces of a bf16 row
    const int64_t Tk = static_cast<int64_t>(p.T) * p.top_k;
    bool bad = false;
    for (int64_t m = warp_id; m < m_total; m += n_warps) {
        const int64_t gi = __ldg(p.gather_idx + m);
        const int64_t rk = gi / Tk, t = (gi - rk * Tk) / p.top_k;
        if (gi < 0 || rk >= p.n_ranks || t >= p.max_tokens) {
            bad = true;
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x[rk] + t * p.hidden * 2);
        uint4 *dst = reinterpret_cast<uint4 *>(p.A_in + m * p.hidden * 2);
        for (int c = lane; c < chunks; c += 32)
            dst[c] = __ldg(src + c);
    }
    if (bad && lane == 0)
        atomicOr(p.status, EP_STATUS_BOUNDS);
}

// A[m][i] = bf16( SiLU(G[m][i]) * G[m][I + i] ) for i < I, m < m_total: the gate
// half first, the up half second.
__global__ void __launch_bounds__(kLayerThreads) swiglu_kernel(const SwigluParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    int64_t m_total = __ldg(p.expert_offsets + p.El);
    m_total = m_total < 0 ? 0 : (m_total > p.max_rows ? p.max_rows : m_total);
    const int chunks = p.inter / 8;
    for (int64_t m = warp_id; m < m_total; m += n_warps) {
        const uint4 *gate = reinterpret_cast<const uint4 *>(p.G + m * 2 * p.inter * 2);
        const uint4 *up = gate + chunks;
        uint4 *out = reinterpret_cast<uint4 *>(p.A + m * p.inter * 2);
        for (int c = lane; c < chunks; c += 32) {
            const uint4 g4 = __ldcs(gate + c), u4 = __ldcs(up + c);
            const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
            const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float g0 = __uint_as_float(gw[h] << 16), g1 = __uint_as_float(gw[h] & 0xFFFF0000u);
                const float u0 = __uint_as_float(uw[h] << 16), u1 = __uint_as_float(uw[h] & 0xFFFF0000u);
                __nv_bfloat162 b = __float22bfloat162_rn(make_float2(silu_f32(g0) * u0, silu_f32(g1) * u1));
                o[h] = *reinterpret_cast<uint32_t *>(&b);
            }
            out[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

cudaError_t launch_dispatch_gather(const DispatchParams &p, int num_sms, cudaStream_t s)
{
    dispatch_gather_kernel<<<4 * num_sms, kLayerThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_swiglu(const SwigluParams &p, int num_sms, cudaStream_t s)
{
    swiglu_kernel<<<4 * num_sms, kLayerThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
