// grouped_gemm_combine_send_noalloc: the fused GEMM + combine send for callers
// that cannot allocate device memory.
//
// Some hosts own every device allocation themselves and forbid allocating from
// inside their per-call path: inference engines that run kernels from a plugin's
// enqueue callback, or serving loops with a fixed memory budget, where cudaMalloc
// could implicitly synchronise the device and stall unrelated streams, or
// fragment a pool the host manages. Such a caller can hand over its inputs and
// outputs but not the two small counter arrays the fused kernel also needs
// (tile-completion counters and per-destination election counters). This file
// keeps those counters in a file-scope device array instead.
//
// The array holds EP_NOALLOC_SCRATCH_INTS int32 words: EP_MAX_LOCAL_EXPERTS tile
// counters followed by EP_MAX_RANKS election counters (1056 bytes). Every GPU that
// loads the library keeps it until the process exits. Host code cannot use the
// array's name as a device address, so the first call on each device asks the
// runtime for that device's address of the array (cudaGetSymbolAddress, with the
// device current) and caches it.
#include <mutex>

#include "ep_internal.h"

static __device__ __align__(256) int32_t g_send_scratch[EP_NOALLOC_SCRATCH_INTS];

namespace {

constexpr int kMaxDevices = 128;

// Device address of g_send_scratch on the current device (nullptr on error).
int32_t *scratch_address()
{
    static std::mutex mu;
    static int32_t *addr[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_send_scratch) != cudaSuccess || !p)
            return nullptr;
        addr[dev] = static_cast<int32_t *>(p);
    }
    return addr[dev];
}

}  // namespace

extern "C" int grouped_gemm_combine_send_noalloc(const ep_config *cfg, const ep_send_args *args,
                                                 ep_stream_t stream)
{
    if (!cfg || !args)
        return EP_ERR_INVALID_ARG;
    if (cfg->n_local_experts < 1 || cfg->n_ranks < 1)
        return EP_ERR_INVALID_ARG;
    // the counters of one call must fit the array
    if (cfg->n_local_experts > EP_MAX_LOCAL_EXPERTS || cfg->n_ranks > EP_MAX_RANKS)
        return EP_ERR_UNSUPPORTED;
    int32_t *scratch = scratch_address();
    if (!scratch)
        return EP_ERR_CUDA;
    ep_send_args a = *args;
    a.atomic_counter = scratch;
    a.rank_completion_counter = scratch + EP_MAX_LOCAL_EXPERTS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (a.p3_control >= 0) {
        // the array keeps the last call's contents (a call that ended with a status
        // bit may leave counts behind): both counter sets must start at zero
        if (cudaMemsetAsync(scratch, 0, sizeof(int32_t) * EP_NOALLOC_SCRATCH_INTS, s) !=
            cudaSuccess)
            return EP_ERR_CUDA;
    }
    return grouped_gemm_combine_send(cfg, &a, stream);
}
