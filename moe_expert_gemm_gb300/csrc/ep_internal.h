// Launch-side definitions shared by the host API and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder comes from the runtime's driver entry point)
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_ep.h"

namespace ep {

constexpr int BM = 128;          // rows per tile (tcgen05 M, one TMEM lane per row)
constexpr int kRowBytesK = 128;  // bytes of K per stage and row: one 128-byte swizzle atom

// Everything the fused GEMM + send kernel reads besides the two operand tensor maps.
struct SendParams {
    // sink disabled (bf16 kernels, output warps storing): the local C as a tensor map,
    // box 64 columns x 32 rows with the 128-byte swizzle of the staging buffers
    CUtensorMap tmap_c;
    int c_tma;         // tmap_c is valid
    int n_ranks, my_rank, El, top_k, K, N, max_tokens;
    int n_blocks;      // column blocks per expert (N / BN)
    int m_fastest;     // tile order within an expert: row blocks fastest (else column blocks)
    int num_k_blocks;  // K / (elements per 128 bytes)
    int64_t msg_bytes;
    int64_t max_rows;
    const int32_t *expert_offsets;
    const int32_t *src_info;
    const int32_t *seg_offsets;
    const int32_t *send_counts;
    uint8_t *recv_buf[EP_MAX_RANKS];
    uint64_t *recv_count[EP_MAX_RANKS];
    int32_t *atomic_counter;
    int32_t *rank_counter;
    uint64_t epoch;
    int sink_enabled;  // p3_control >= 0
    int signal_mode;   // EP_SIGNAL_RANK_FLAG or EP_SIGNAL_PER_EXPERT
    int act_swiglu;    // sink disabled: gate/up column halves -> SiLU(gate) * up
    int64_t c_row_bytes;  // local C row pitch (N*2, or N with the activation)
    uint8_t *C;        // local output when the sink is disabled
    uint32_t *status;
    uint64_t timeout_ns;
    const float *a_scales;
    const float *w_scales;
    uint64_t *trace;    // optional per-tile timestamps
    int trace_records;  // records per thread block
    int overlap_previous;  // launched as a programmatic dependent of the previous kernel
};

// Launch of a fused send kernel, as a programmatic dependent of the previous kernel
// on the stream when p.overlap_previous is set.
template <typename Kern>
inline cudaError_t launch_send_kernel(Kern kern, int grid, int threads, int smem,
                                      const CUtensorMap &ta, const CUtensorMap &tb,
                                      const SendParams &p, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.overlap_previous ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, p);
}

// The unfused send step (local C rows to the receive buffers, then signalling).
struct ScatterParams {
    int n_ranks, my_rank, El, top_k, N, max_tokens;
    int64_t msg_bytes;
    int64_t max_rows;
    const uint8_t *C;
    const int32_t *expert_offsets;
    const int32_t *src_info;
    const int32_t *seg_offsets;
    const int32_t *send_counts;
    uint8_t *recv_buf[EP_MAX_RANKS];
    uint64_t *recv_count[EP_MAX_RANKS];
    int32_t *block_counter;
    uint64_t epoch;
    uint32_t *status;
    int signal_mode;
};

// The layer steps around the fused down-projection (ep_layer.cu).
struct DispatchParams {
    int n_ranks, El, top_k, T, max_tokens, hidden;
    int64_t max_rows;
    const uint8_t *x[EP_MAX_RANKS];
    const int32_t *gather_idx;
    const int32_t *expert_offsets;
    uint8_t *A_in;
    uint32_t *status;
};

struct SwigluParams {
    int El, inter;
    int64_t max_rows;
    const uint8_t *G;
    uint8_t *A;
    const int32_t *expert_offsets;
};

struct PlanParams {
    int n_ranks, my_rank, El, top_k, T;
    int64_t max_rows;
    const int32_t *topk_ids;
    int32_t *expert_offsets, *src_info, *seg_offsets, *send_counts, *gather_idx, *m_total;
    uint32_t *status;
};

struct CombineParams {
    int n_ranks, El, top_k, T, N;
    int64_t msg_bytes;
    const uint8_t *recv_buf;
    const uint64_t *recv_count;
    const float *gates;
    uint8_t *out;
    uint64_t epoch;
    uint64_t timeout_ns;
    uint32_t *status;
    const int32_t *topk_ids;  // EP_SIGNAL_PER_EXPERT: [T][top_k] global expert ids
    int signal_mode;
    int overlap_previous;  // EP_OVERLAP_*: programmatic dependent of the previous kernel
};

// A checked grouped_gemm_combine_send call, ready to launch: prepare_send runs every
// host check (returning EP_ERR_* with nothing enqueued), encodes the tensor maps and
// picks the kernel; launch_prepared_send enqueues it (EP_OK or EP_ERR_CUDA).
struct PreparedSend {
    enum Kind { kBf16, kPair, kFp8 };
    CUtensorMap ta, tb;
    SendParams p;
    int kind, bn, send_warps, grid, max_pairs;
};
int prepare_send(const ep_config *cfg, const ep_send_args *a, PreparedSend *out);
int launch_prepared_send(const PreparedSend &ps, cudaStream_t s);

// Kernel launchers; each returns the launch's cudaError_t.
cudaError_t launch_plan(const PlanParams &p, cudaStream_t s);
cudaError_t launch_gemm_send_bf16(const CUtensorMap &ta, const CUtensorMap &tb,
                                  const SendParams &p, int bn, int send_warps, int grid,
                                  cudaStream_t s);
cudaError_t launch_gemm_send_fp8(const CUtensorMap &ta, const CUtensorMap &tb,
                                 const SendParams &p, int bn, int grid, cudaStream_t s);
cudaError_t launch_gemm_send_bf16_pair(const CUtensorMap &ta, const CUtensorMap &tb,
                                       const SendParams &p, int send_warps, int max_pairs,
                                       cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_scatter(const ScatterParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_dispatch_gather(const DispatchParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_swiglu(const SwigluParams &p, int num_sms, cudaStream_t s);

}  // namespace ep
