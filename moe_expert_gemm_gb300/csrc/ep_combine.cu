// Gate-weighted combine on the receiving rank.
//
// "ep_signal_completion" (ep_ord_r): a fused consumer acquires one rank-completion
// flag per source rank instead of one word per expert; the single system-scope
// release of the elected producer carries all of that rank's rows and counts. The
// sum itself, out[t] = sum_j g[t, j] * row(t, j), is the combine role the
// "P3PeerSendConfig" description names (EPCombineKernel), whose receive layout is
// (src_idx*top_k + src_topk)*msg_bytes + byte_off.
//
// HBM-bound: every received byte is read once and every output byte written
// once. R threads per block acquire the R source flags (bounded waits), then each
// warp handles 256 contiguous columns of one token: 32 lanes x 16-byte loads of
// each of the token's top_k rows, fp32 accumulation in slot order, one 16-byte
// streaming store. The grid is one wave of 8 blocks per SM with a grid-stride loop.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"

namespace ep {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ void accumulate_row(float (&acc)[8], float g, uint4 raw)
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        acc[2 * h] = fmaf(g, __uint_as_float(w[h] << 16), acc[2 * h]);
        acc[2 * h + 1] = fmaf(g, __uint_as_float(w[h] & 0xFFFF0000u), acc[2 * h + 1]);
    }
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p)
{
    __shared__ int s_ok;
    if (threadIdx.x == 0)
        s_ok = 1;
    __syncthreads();
    if (threadIdx.x < p.n_ranks) {
        // one thread per source rank acquires that rank's flag (bounded wait)
        const uint64_t *flag = p.recv_count + static_cast<int64_t>(p.El) * p.n_ranks + threadIdx.x;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_sys_u64(flag) != p.epoch) {
            if (globaltimer_ns() - t0 > p.timeout_ns) {
                atomicOr(p.status, EP_STATUS_TIMEOUT);
                s_ok = 0;
                break;
            }
            __nanosleep(100);
        }
    }
    __syncthreads();
    if (!s_ok)
        return;

    const int lane = threadIdx.x & 31;
    const int warps = kCombineThreads / 32;
    const int k = p.top_k;
    const int64_t vec_per_row = p.N / 8;  // 16-byte vectors of one output row
    const int64_t units_per_row = (vec_per_row + 31) / 32;
    const int64_t units = static_cast<int64_t>(p.T) * units_per_row;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); u < units;
         u += static_cast<int64_t>(gridDim.x) * warps) {
        const int64_t t = u / units_per_row;
        const int64_t v = (u - t * units_per_row) * 32 + lane;
        if (v >= vec_per_row)
            continue;
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            acc[c] = 0.f;
        const uint8_t *rows = p.recv_buf + t * k * p.msg_bytes + v * 16;
        const float *g = p.gates + t * k;
        int j = 0;
        for (; j + 4 <= k; j += 4) {
            uint4 r[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                r[jj] = __ldcs(reinterpret_cast<const uint4 *>(rows + (j + jj) * p.msg_bytes));
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                accumulate_row(acc, __ldg(g + j + jj), r[jj]);
        }
        for (; j < k; ++j)
            accumulate_row(acc, __ldg(g + j),
                           __ldcs(reinterpret_cast<const uint4 *>(rows + j * p.msg_bytes)));
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            __nv_bfloat162 b = __float22bfloat162_rn(make_float2(acc[2 * h], acc[2 * h + 1]));
            o[h] = *reinterpret_cast<uint32_t *>(&b);
        }
        __stcs(reinterpret_cast<uint4 *>(p.out + (t * p.N + v * 8) * 2),
               make_uint4(o[0], o[1], o[2], o[3]));
    }
}

cudaError_t launch_combine(const CombineParams &p, int num_sms, cudaStream_t s)
{
    const int64_t units = static_cast<int64_t>(p.T) * ((p.N / 8 + 31) / 32);
    int64_t blocks = (units + 7) / 8;
    const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kCombineThreads);
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    combine_kernel<<<static_cast<int>(blocks), kCombineThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
