// Receive buffers shared between the processes of an expert-parallel group on one
// node: a rank exports the device buffers its peers write (its receive buffer and
// its receive-count buffer) as CUDA IPC handles, and every other process of the
// group maps them into its own address space, so that its fused send writes them by
// plain stores ("ep_signal_completion": direct memory access when the target
// device is on the same node; "P3PeerSendConfig": recv_buf_ptrs, one pointer per
// rank).
//
// A handle names a whole cudaMalloc allocation, while the caller's buffer may start
// inside one (a caching allocator hands out pieces of larger blocks), so the handle
// carries the buffer's offset from the allocation's base.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "ep_internal.h"

namespace {

using AddressRangeFn = PFN_cuMemGetAddressRange_v3020;

AddressRangeFn address_range_fn()
{
    static AddressRangeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 3020, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddressRangeFn>(p);
    });
    return fn;
}

static_assert(sizeof(cudaIpcMemHandle_t) == EP_IPC_HANDLE_BYTES, "IPC handle size");

}  // namespace

extern "C" {

int ep_ipc_export(const void *dev_ptr, ep_ipc_handle *out)
{
    if (!dev_ptr || !out)
        return EP_ERR_INVALID_ARG;
    AddressRangeFn range = address_range_fn();
    if (!range)
        return EP_ERR_CUDA;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, reinterpret_cast<CUdeviceptr>(dev_ptr)) != CUDA_SUCCESS)
        return EP_ERR_INVALID_ARG;  // not device memory of this context
    cudaIpcMemHandle_t h;
    if (cudaIpcGetMemHandle(&h, reinterpret_cast<void *>(base)) != cudaSuccess)
        return EP_ERR_CUDA;  // e.g. memory not from cudaMalloc
    std::memset(out, 0, sizeof *out);
    std::memcpy(out->handle, &h, sizeof h);
    out->offset = static_cast<uint64_t>(reinterpret_cast<CUdeviceptr>(dev_ptr) - base);
    out->bytes = static_cast<uint64_t>(size) - out->offset;
    return EP_OK;
}

int ep_ipc_import(const ep_ipc_handle *h, void **dev_ptr)
{
    if (!h || !dev_ptr)
        return EP_ERR_INVALID_ARG;
    *dev_ptr = nullptr;
    cudaIpcMemHandle_t mh;
    std::memcpy(&mh, h->handle, sizeof mh);
    void *base = nullptr;
    if (cudaIpcOpenMemHandle(&base, mh, cudaIpcMemLazyEnablePeerAccess) != cudaSuccess)
        return EP_ERR_CUDA;
    *dev_ptr = static_cast<uint8_t *>(base) + h->offset;
    return EP_OK;
}

int ep_ipc_close(const ep_ipc_handle *h, void *dev_ptr)
{
    if (!h || !dev_ptr)
        return EP_ERR_INVALID_ARG;
    void *base = static_cast<uint8_t *>(dev_ptr) - h->offset;
    return cudaIpcCloseMemHandle(base) == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // extern "C"
