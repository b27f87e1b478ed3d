// Gate-weighted combine on the receiving rank.
//
// "ep_signal_completion" (ep_ord_r): a fused consumer acquires one rank-completion
// flag per source rank instead of one word per expert; the single system-scope
// release of the elected producer carries all of that rank's rows and counts. In
// the per-expert mode the consumer instead acquires, per token, the count words of
// that token's experts (combine_kernel_per_expert). The
// sum itself, out[t] = sum_j g[t, j] * row(t, j), is the combine role the
// "P3PeerSendConfig" description names (EPCombineKernel), whose receive layout is
// (src_idx*top_k + src_topk)*msg_bytes + byte_off.
//
// HBM-bound: every received byte is read once and every output byte written
// once. R threads per block acquire the R source flags (bounded waits), then a warp
// handles units of 256 contiguous columns of one token: 32 lanes x 16-byte loads of
// each of the token's top_k rows, fp32 accumulation in slot order, one 16-byte
// streaming store. A warp takes several consecutive units at a time (8 / top_k;
// for top_k >= 8 on large calls 16 / top_k) and issues all their loads before
// accumulating, so each thread keeps 8-16 16-byte loads in flight. The grid is one
// resident wave (four for the 16-load form) with a grid-stride loop.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"

namespace ep {

constexpr int kCombineThreads = 256;
constexpr int kLoads = 8;  // 16-byte row loads a thread keeps in flight (at least)

// Units a warp reduces at once for a compile-time top_k: about kLoads row loads per
// thread in flight (one unit for run-time top_k).
template <int K>
constexpr int units_at_once()
{
    return K == 0 ? 1 : (K >= kLoads ? 1 : kLoads / K);
}

__device__ __forceinline__ void store_out(const CombineParams &p, int64_t t, int64_t v,
                                          const float (&acc)[8])
{
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 b = __float22bfloat162_rn(make_float2(acc[2 * h], acc[2 * h + 1]));
        o[h] = *reinterpret_cast<uint32_t *>(&b);
    }
    __stcs(reinterpret_cast<uint4 *>(p.out + (t * p.N + v * 8) * 2),
           make_uint4(o[0], o[1], o[2], o[3]));
}

__device__ __forceinline__ void accumulate_row(float (&acc)[8], float g, uint4 raw)
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        acc[2 * h] = fmaf(g, __uint_as_float(w[h] << 16), acc[2 * h]);
        acc[2 * h + 1] = fmaf(g, __uint_as_float(w[h] & 0xFFFF0000u), acc[2 * h + 1]);
    }
}

// Acquire every source rank's flag (one thread per rank, bounded wait); false when
// a wait ran out (EP_STATUS_TIMEOUT raised, the block must not read the rows).
__device__ __forceinline__ bool acquire_source_flags(const CombineParams &p)
{
    __shared__ int s_ok;
    if (threadIdx.x == 0)
        s_ok = 1;
    __syncthreads();
    if (threadIdx.x < p.n_ranks) {
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
    return s_ok != 0;
}

// top_k known at compile time: a warp takes U consecutive units and issues all U*K
// loads before accumulating any of them.
template <int K, int U>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p)
{
    if (!acquire_source_flags(p))
        return;
    if (p.overlap_previous == EP_OVERLAP_ANY)
        griddep_wait();  // gates (and out) may belong to the kernel before this one
    const int lane = threadIdx.x & 31;
    const int warps = kCombineThreads / 32;
    const int64_t vec_per_row = p.N / 8;  // 16-byte vectors of one output row
    const int64_t units_per_row = (vec_per_row + 31) / 32;
    const int64_t units = static_cast<int64_t>(p.T) * units_per_row;
    for (int64_t u0 = (static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5)) * U;
         u0 < units; u0 += static_cast<int64_t>(gridDim.x) * warps * U) {
        uint4 r[U][K];
        int64_t tt[U], vv[U];
        bool live[U];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            const int64_t u = u0 + uu;
            tt[uu] = u / units_per_row;
            vv[uu] = (u - tt[uu] * units_per_row) * 32 + lane;
            live[uu] = u < units && vv[uu] < vec_per_row;
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (live[uu])
                    r[uu][j] = __ldcs(reinterpret_cast<const uint4 *>(
                        p.recv_buf + (tt[uu] * K + j) * p.msg_bytes + vv[uu] * 16));
        }
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            if (!live[uu])
                continue;
            float acc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[c] = 0.f;
            const float *g = p.gates + tt[uu] * K;
#pragma unroll
            for (int j = 0; j < K; ++j)
                accumulate_row(acc, __ldg(g + j), r[uu][j]);
            store_out(p, tt[uu], vv[uu], acc);
        }
    }
}

// EP_SIGNAL_PER_EXPERT: wait for (acquire) the count word of global expert g in this
// rank's count buffer, (epoch mod 2^32) << 32 | rows, which g's owner releases once
// all of g's rows are written. Bounded; after one wait of the block has run out,
// later waits give up at once instead of each waiting out the limit.
__device__ __forceinline__ bool expert_arrived(const CombineParams &p, int g, volatile int *gave_up)
{
    const int rk = g / p.El, e = g - rk * p.El;
    const uint64_t *w = p.recv_count + static_cast<int64_t>(e) * p.n_ranks + rk;
    const uint32_t tag = static_cast<uint32_t>(p.epoch);
    if (static_cast<uint32_t>(ld_acquire_sys_u64(w) >> 32) == tag)
        return true;
    if (*gave_up)
        return false;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(100);
        if (static_cast<uint32_t>(ld_acquire_sys_u64(w) >> 32) == tag)
            return true;
        if (*gave_up)
            return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            atomicOr(p.status, EP_STATUS_TIMEOUT);
            *gave_up = 1;
            return false;
        }
    }
}

// EP_SIGNAL_PER_EXPERT: the warp's lanes acquire the count words of token t's
// top_k experts (warp-collective); true when all arrived. A malformed expert id
// counts as never arriving and raises EP_STATUS_ROUTING.
__device__ __forceinline__ bool token_arrived(const CombineParams &p, int64_t t, int k, int lane,
                                              volatile int *gave_up)
{
    const int n_experts = p.n_ranks * p.El;
    bool ok = true;
    for (int j = lane; j < k; j += 32) {
        const int g = __ldg(p.topk_ids + t * k + j);
        if (g < 0 || g >= n_experts) {
            atomicOr(p.status, EP_STATUS_ROUTING);
            ok = false;
        } else {
            ok = expert_arrived(p, g, gave_up) && ok;
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();  // the acquiring lanes' reads precede every lane's row loads
    return ok;
}

// EP_SIGNAL_PER_EXPERT consumer: every warp takes a contiguous range of (token,
// 256-column unit) work items and, whenever its range enters a new token, acquires
// that token's experts; then it reduces the token's units U at a time, all U*K row
// loads issued before accumulating. A token whose experts have
// all arrived is reduced whatever the other experts are doing; one whose expert
// never arrives is left unwritten (EP_STATUS_TIMEOUT). K = 0: top_k known at run
// time only.
template <int K, int U>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel_per_expert(const CombineParams p)
{
    __shared__ int s_gave_up;
    if (threadIdx.x == 0)
        s_gave_up = 0;
    if (p.overlap_previous == EP_OVERLAP_ANY)
        griddep_wait();  // the routing and gates may belong to the kernel before this one
    __syncthreads();
    volatile int *gave_up = &s_gave_up;
    const int k = K == 0 ? p.top_k : K;
    const int lane = threadIdx.x & 31;
    const int64_t vec_per_row = p.N / 8;
    const int64_t units_per_row = (vec_per_row + 31) / 32;
    const int64_t units = static_cast<int64_t>(p.T) * units_per_row;
    const int64_t n_warps = static_cast<int64_t>(gridDim.x) * (kCombineThreads / 32);
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5);
    const int64_t per = (units + n_warps - 1) / n_warps;
    const int64_t u_end = (gw + 1) * per < units ? (gw + 1) * per : units;
    for (int64_t u = gw * per; u < u_end;) {
        const int64_t t = u / units_per_row;
        const int64_t stop = (t + 1) * units_per_row < u_end ? (t + 1) * units_per_row : u_end;
        if (token_arrived(p, t, k, lane, gave_up)) {
            const uint8_t *rows_t = p.recv_buf + t * k * p.msg_bytes;
            const float *g = p.gates + t * k;
            for (int64_t u0 = u; u0 < stop; u0 += U) {
                int64_t vv[U];
                bool live[U];
#pragma unroll
                for (int uu = 0; uu < U; ++uu) {
                    vv[uu] = (u0 + uu - t * units_per_row) * 32 + lane;
                    live[uu] = u0 + uu < stop && vv[uu] < vec_per_row;
                }
                if constexpr (K > 0) {
                    uint4 r[U][K];
#pragma unroll
                    for (int uu = 0; uu < U; ++uu)
#pragma unroll
                        for (int jj = 0; jj < K; ++jj)
                            if (live[uu])
                                r[uu][jj] = __ldcs(reinterpret_cast<const uint4 *>(
                                    rows_t + jj * p.msg_bytes + vv[uu] * 16));
#pragma unroll
                    for (int uu = 0; uu < U; ++uu) {
                        if (!live[uu])
                            continue;
                        float acc[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            acc[c] = 0.f;
#pragma unroll
                        for (int jj = 0; jj < K; ++jj)
                            accumulate_row(acc, __ldg(g + jj), r[uu][jj]);
                        store_out(p, t, vv[uu], acc);
                    }
                } else {
                    // run-time top_k: one unit, rows streamed kLoads at a time
                    if (!live[0])
                        continue;
                    float acc[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        acc[c] = 0.f;
                    for (int j = 0; j < k; j += kLoads) {
                        uint4 rr[kLoads];
#pragma unroll
                        for (int jj = 0; jj < kLoads; ++jj)
                            if (j + jj < k)
                                rr[jj] = __ldcs(reinterpret_cast<const uint4 *>(
                                    rows_t + (j + jj) * p.msg_bytes + vv[0] * 16));
#pragma unroll
                        for (int jj = 0; jj < kLoads; ++jj)
                            if (j + jj < k)
                                accumulate_row(acc, __ldg(g + j + jj), rr[jj]);
                    }
                    store_out(p, t, vv[0], acc);
                }
            }
        }
        u = stop;
    }
}

// any other top_k: one unit at a time, its rows streamed kLoads at a time
__global__ void __launch_bounds__(kCombineThreads) combine_kernel_any(const CombineParams p)
{
    if (!acquire_source_flags(p))
        return;
    if (p.overlap_previous == EP_OVERLAP_ANY)
        griddep_wait();  // gates (and out) may belong to the kernel before this one
    const int lane = threadIdx.x & 31;
    const int warps = kCombineThreads / 32;
    const int k = p.top_k;
    const int64_t vec_per_row = p.N / 8;
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
        for (int j = 0; j < k; j += kLoads) {
            uint4 r[kLoads];
#pragma unroll
            for (int jj = 0; jj < kLoads; ++jj)
                if (j + jj < k)
                    r[jj] = __ldcs(reinterpret_cast<const uint4 *>(rows + (j + jj) * p.msg_bytes));
#pragma unroll
            for (int jj = 0; jj < kLoads; ++jj)
                if (j + jj < k)
                    accumulate_row(acc, __ldg(g + j + jj), r[jj]);
        }
        store_out(p, t, v, acc);
    }
}

// Launch; with overlap_previous as a programmatic dependent of the previous kernel
// on the stream (it may start once that kernel's thread blocks have signalled).
static cudaError_t launch_with(void (*kern)(CombineParams), int blocks, const CombineParams &p,
                               cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(kCombineThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.overlap_previous ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename Kern>
static int blocks_for(Kern kern, int num_sms, int64_t work_blocks, int waves = 1)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCombineThreads, 0) !=
            cudaSuccess ||
        per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    const int64_t cap = static_cast<int64_t>(waves) * num_sms * per_sm;  // resident waves
    int64_t b = work_blocks < cap ? work_blocks : cap;
    return static_cast<int>(b < 1 ? 1 : b);
}

// Per call, the kernel form: U = units_at_once<K>(), or twice that for top_k >= kLoads
// when every resident warp would get at least kWideUnits units (16 loads in flight
// per thread: the fp8 prefill combine 177 -> 162 us, 0.88 -> 0.95 of the copy
// bandwidth; on smaller calls the fewer, longer warps cost more at the tail). The
// wide form's grid is up to four resident waves: a combine launched behind the send
// starts on SMs as the send's blocks leave, and smaller blocks spread the work over
// the SMs that free up last (the narrow form keeps one wave: its blocks are short,
// and each extra block acquires the flags again).
constexpr int64_t kWideUnits = 32;

template <int K>
static cudaError_t launch_form(const CombineParams &p, int num_sms, cudaStream_t s,
                               void (*narrow)(CombineParams), void (*wide)(CombineParams))
{
    constexpr int U = units_at_once<K>();
    const int64_t units = static_cast<int64_t>(p.T) * ((p.N / 8 + 31) / 32);
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, narrow, kCombineThreads, 0) !=
            cudaSuccess ||
        per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
    }
    const int64_t resident_warps = static_cast<int64_t>(num_sms) * per_sm * (kCombineThreads / 32);
    if (K >= kLoads && wide != nullptr && units >= kWideUnits * resident_warps) {
        const int b = blocks_for(wide, num_sms, (units + 16 * U - 1) / (16 * U), 4);
        return launch_with(wide, b, p, s);
    }
    const int b = blocks_for(narrow, num_sms, (units + 8 * U - 1) / (8 * U));
    return launch_with(narrow, b, p, s);
}

template <int K>
static cudaError_t launch_k(const CombineParams &p, int num_sms, cudaStream_t s)
{
    constexpr int U = units_at_once<K>();
    if constexpr (K >= kLoads)
        return launch_form<K>(p, num_sms, s, combine_kernel<K, U>, combine_kernel<K, 2 * U>);
    else
        return launch_form<K>(p, num_sms, s, combine_kernel<K, U>, nullptr);
}

template <int K>
static cudaError_t launch_per_expert(const CombineParams &p, int num_sms, cudaStream_t s)
{
    constexpr int U = units_at_once<K>();
    if constexpr (K >= kLoads)
        return launch_form<K>(p, num_sms, s, combine_kernel_per_expert<K, U>,
                              combine_kernel_per_expert<K, 2 * U>);
    else
        return launch_form<K>(p, num_sms, s, combine_kernel_per_expert<K, U>, nullptr);
}

cudaError_t launch_combine(const CombineParams &p, int num_sms, cudaStream_t s)
{
    if (p.signal_mode == EP_SIGNAL_PER_EXPERT) {
        switch (p.top_k) {
        case 1:
            return launch_per_expert<1>(p, num_sms, s);
        case 2:
            return launch_per_expert<2>(p, num_sms, s);
        case 4:
            return launch_per_expert<4>(p, num_sms, s);
        case 8:
            return launch_per_expert<8>(p, num_sms, s);
        default:
            return launch_per_expert<0>(p, num_sms, s);
        }
    }
    switch (p.top_k) {
    case 1:
        return launch_k<1>(p, num_sms, s);
    case 2:
        return launch_k<2>(p, num_sms, s);
    case 4:
        return launch_k<4>(p, num_sms, s);
    case 8:
        return launch_k<8>(p, num_sms, s);
    default: {
        const int64_t units = static_cast<int64_t>(p.T) * ((p.N / 8 + 31) / 32);
        const int b = blocks_for(combine_kernel_any, num_sms, (units + 7) / 8);
        return launch_with(combine_kernel_any, b, p, s);
    }
    }
}

}  // namespace ep
