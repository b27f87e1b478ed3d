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
// array's name as a device address, so every call asks the runtime for the current
// device's address of the array (cudaGetSymbolAddress, with that device current)
// and remembers it. A call made while its stream is being captured into a graph
// uses the remembered address instead (looking it up may load the module, which a
// capture forbids), so the first call on a device must come before any capture.
// Looking the address up again on every other call keeps it right after the
// device's primary context was destroyed and re-created (cudaDeviceReset), which
// reloads the module and may move the array.
#include <mutex>

#include "ep_internal.h"

static __device__ __align__(256) int32_t g_send_scratch[EP_NOALLOC_SCRATCH_INTS];

namespace {

constexpr int kMaxDevices = 128;

// Device address of g_send_scratch on the current device (nullptr on error).
// Outside stream capture it is looked up afresh and remembered; during a capture
// the remembered address is used (nullptr if this device has none yet).
int32_t *scratch_address(cudaStream_t s)
{
    static std::mutex mu;
    static int32_t *addr[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (cap == cudaStreamCaptureStatusNone) {
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t *scratch = scratch_address(s);
    if (!scratch)
        return EP_ERR_CUDA;
    ep_send_args a = *args;
    a.atomic_counter = scratch;
    a.rank_completion_counter = scratch + EP_MAX_LOCAL_EXPERTS;
    // every check of the allocating entry point, before anything is enqueued
    ep::PreparedSend ps;
    const int rc = ep::prepare_send(cfg, &a, &ps);
    if (rc != EP_OK)
        return rc;
    if (a.p3_control >= 0) {
        // the array keeps the last call's contents (a call that ended with a status
        // bit may leave counts behind): both counter sets must start at zero
        if (cudaMemsetAsync(scratch, 0, sizeof(int32_t) * EP_NOALLOC_SCRATCH_INTS, s) !=
            cudaSuccess)
            return EP_ERR_CUDA;
    }
    return ep::launch_prepared_send(ps, s);
}
