// Host side of the C ABI: argument checks, TMA descriptors, launches.
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>
#include <mutex>

#include "ep_internal.h"

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn tensor_map_encoder()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int sm_count()
{
    static std::mutex mu;
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
        return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// 2-D tiled map over a row-major [outer][inner] array, 128-byte swizzle, zero fill
// outside the array.
bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer)
{
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t elem_strides[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_config(const ep_config *c)
{
    if (!c)
        return EP_ERR_INVALID_ARG;
    if (c->n_ranks < 1 || c->my_rank < 0 || c->my_rank >= c->n_ranks)
        return EP_ERR_INVALID_ARG;
    if (c->n_ranks > EP_MAX_RANKS)
        return EP_ERR_UNSUPPORTED;  // direct-store reach is 8 ranks
    if (c->n_local_experts < 1 || c->top_k < 1 ||
        static_cast<int64_t>(c->top_k) > static_cast<int64_t>(c->n_ranks) * c->n_local_experts)
        return EP_ERR_INVALID_ARG;
    if (c->n_local_experts > EP_MAX_LOCAL_EXPERTS)
        return EP_ERR_UNSUPPORTED;
    if (c->num_tokens < 0 || c->max_tokens_per_rank < 1 || c->num_tokens > c->max_tokens_per_rank)
        return EP_ERR_INVALID_ARG;
    if (c->K < 1 || c->N < 1 || c->msg_bytes != 2 * static_cast<int64_t>(c->N))
        return EP_ERR_INVALID_ARG;
    if (c->dtype != EP_BF16 && c->dtype != EP_FP8_1D2D)
        return EP_ERR_INVALID_ARG;
    if (c->send_warps != -1 && c->send_warps != 0 && c->send_warps != 4)
        return EP_ERR_INVALID_ARG;
    if (c->signal_mode != EP_SIGNAL_RANK_FLAG && c->signal_mode != EP_SIGNAL_PER_EXPERT)
        return EP_ERR_INVALID_ARG;
    // every index the kernels form from (token, slot) stays in 32 bits
    if (static_cast<int64_t>(c->max_tokens_per_rank) * c->n_ranks * c->top_k >= INT32_MAX)
        return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

// Column tile of the fp8 kernel: 256 where N allows it (half the operand traffic per
// FLOP of a 128-wide tile, two fp32 partial buffers in TMEM), else 128 (four buffers).
int fp8_tile_n(int N)
{
    return N % 256 == 0 ? 256 : 128;
}

// Tile order within an expert that moves fewer bytes from DRAM, with `conc` tiles
// in flight: column blocks fastest re-reads the expert's W once per group of
// concurrent row blocks; row blocks fastest re-reads its A once per group of
// concurrent column blocks.
bool pick_m_fastest(int64_t rows, int64_t tile_rows, int64_t n_blocks, int64_t K, int64_t N,
                    int64_t elem, int64_t conc)
{
    const int64_t m_blocks = (rows + tile_rows - 1) / tile_rows;
    if (m_blocks <= 1 || conc < 1)
        return false;
    const int64_t a_bytes = rows * K * elem, w_bytes = N * K * elem;
    const int64_t rows_per_wave = conc / n_blocks > 0 ? conc / n_blocks : 1;
    const int64_t cols_per_wave = conc / m_blocks > 0 ? conc / m_blocks : 1;
    const int64_t n_fast = a_bytes + (m_blocks + rows_per_wave - 1) / rows_per_wave * w_bytes;
    const int64_t m_fast = w_bytes + (n_blocks + cols_per_wave - 1) / cols_per_wave * a_bytes;
    return m_fast < n_fast;
}

int cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

}  // namespace

extern "C" {

int ep_plan_sizes(const ep_config *cfg, int64_t *max_rows)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!max_rows)
        return EP_ERR_INVALID_ARG;
    const int64_t per_token = cfg->top_k < cfg->n_local_experts ? cfg->top_k : cfg->n_local_experts;
    *max_rows = static_cast<int64_t>(cfg->num_tokens) * cfg->n_ranks * per_token;
    return EP_OK;
}

int ep_plan(const ep_config *cfg, const int32_t *topk_ids, const ep_plan_out *out,
            ep_stream_t stream)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!out || !out->expert_offsets || !out->src_info || !out->seg_offsets ||
        !out->send_counts || !out->gather_idx || !out->m_total || !out->status)
        return EP_ERR_INVALID_ARG;
    if (cfg->num_tokens > 0 && !topk_ids)
        return EP_ERR_INVALID_ARG;
    if (out->max_rows < 0 || out->max_rows > INT32_MAX)
        return EP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(out->src_info) & 7u)
        return EP_ERR_INVALID_ARG;  // written as (src_idx, src_topk) pairs
    ep::PlanParams p;
    p.n_ranks = cfg->n_ranks;
    p.my_rank = cfg->my_rank;
    p.El = cfg->n_local_experts;
    p.top_k = cfg->top_k;
    p.T = cfg->num_tokens;
    p.max_rows = out->max_rows;
    p.topk_ids = topk_ids;
    p.expert_offsets = out->expert_offsets;
    p.src_info = out->src_info;
    p.seg_offsets = out->seg_offsets;
    p.send_counts = out->send_counts;
    p.gather_idx = out->gather_idx;
    p.m_total = out->m_total;
    p.status = out->status;
    return cuda_status(ep::launch_plan(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace ep {

// Every host check of grouped_gemm_combine_send, the tensor maps and the launch
// parameters; nothing is enqueued.
int prepare_send(const ep_config *cfg, const ep_send_args *a, PreparedSend *out)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!a)
        return EP_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == EP_FP8_1D2D;
    // dedicated send warps exist in the single-CTA bf16 kernel
    if (fp8 && cfg->send_warps == 4)
        return EP_ERR_UNSUPPORTED;
    if (a->p3_control < 0 && a->local_activation != EP_ACT_NONE) {
        if (a->local_activation != EP_ACT_SWIGLU)
            return EP_ERR_INVALID_ARG;
        // the activation pairs the two 128-column halves of a 256-column tile
        if (fp8 || cfg->N % 256 != 0 || cfg->send_warps == 4)
            return EP_ERR_UNSUPPORTED;
    }
    if (!fp8 && (cfg->K % 64 != 0 || cfg->N % 64 != 0))
        return EP_ERR_UNSUPPORTED;  // whole 128-byte K atoms and 64-column output chunks
    // fp8: one 128-wide scale block per K step, whole 128-column weight-scale blocks
    if (fp8 && (cfg->K % 128 != 0 || cfg->N % 128 != 0))
        return EP_ERR_UNSUPPORTED;
    if (fp8 && (!a->a_scales || !a->w_scales ||
                (reinterpret_cast<uintptr_t>(a->a_scales) & 3u) ||
                (reinterpret_cast<uintptr_t>(a->w_scales) & 3u)))
        return EP_ERR_INVALID_ARG;
    const int R = cfg->n_ranks;
    const bool sink = a->p3_control >= 0;
    if (!a->A || !a->W || !a->expert_offsets || !a->src_info || !a->seg_offsets ||
        !a->send_counts || !a->status)
        return EP_ERR_INVALID_ARG;
    if (a->trace && (a->trace_records < 1 || a->trace_records > (1 << 20) ||
                     (reinterpret_cast<uintptr_t>(a->trace) & 7u)))
        return EP_ERR_INVALID_ARG;
    if (!aligned16(a->A) || !aligned16(a->W))
        return EP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(a->src_info) & 7u)
        return EP_ERR_INVALID_ARG;  // read as (src_idx, src_topk) pairs
    if (a->max_rows < 1 || a->max_rows > INT32_MAX)
        return EP_ERR_INVALID_ARG;
    if (sink) {
        if (!a->atomic_counter || !a->rank_completion_counter)
            return EP_ERR_INVALID_ARG;
        for (int r = 0; r < R; ++r)
            if (!a->recv_buf_ptrs[r] || !a->recv_count_ptrs[r] || !aligned16(a->recv_buf_ptrs[r]) ||
                (reinterpret_cast<uintptr_t>(a->recv_count_ptrs[r]) & 7u))
                return EP_ERR_INVALID_ARG;
    } else if (!a->C || !aligned16(a->C)) {
        return EP_ERR_INVALID_ARG;
    }
    const int num_sms = sm_count();
    if (num_sms <= 0)
        return EP_ERR_CUDA;

    const int bn = fp8 ? fp8_tile_n(cfg->N)
                       : (cfg->N % 256 == 0 ? 256 : (cfg->N % 128 == 0 ? 128 : 64));
    const int El = cfg->n_local_experts;
    const int elem = fp8 ? 1 : 2;
    const int box_k = 128 / elem;  // one 128-byte swizzle atom of K per stage
    const CUtensorMapDataType dt =
        fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // bf16 256-column tiles run on CTA pairs (each CTA loads half of the W block) when
    // an expert's expected rows, T*top_k/E_l, fill a 256-row pair tile; with fewer rows
    // (decode) the pair's extra padded MMA rows cost more than the traffic saved. The
    // fp8 kernel stays on single CTAs: its per-K-block hand-off of partial buffers
    // between MMA and promotion would cross the pair every K block.
    const int64_t rows_per_expert =
        static_cast<int64_t>(cfg->num_tokens) * cfg->top_k / cfg->n_local_experts;
    const bool pair = !fp8 && bn == 256 && rows_per_expert >= 2 * ep::BM;
    CUtensorMap ta, tb;
    if (!encode_2d(&ta, dt, a->A, cfg->K, a->max_rows, static_cast<uint64_t>(cfg->K) * elem,
                   box_k, ep::BM))
        return EP_ERR_CUDA;
    if (!encode_2d(&tb, dt, a->W, cfg->K, static_cast<uint64_t>(El) * cfg->N,
                   static_cast<uint64_t>(cfg->K) * elem, box_k,
                   static_cast<uint32_t>(pair ? bn / 2 : bn)))
        return EP_ERR_CUDA;

    ep::SendParams p;
    std::memset(&p, 0, sizeof p);
    p.n_ranks = R;
    p.my_rank = cfg->my_rank;
    p.El = El;
    p.top_k = cfg->top_k;
    p.K = cfg->K;
    p.N = cfg->N;
    p.max_tokens = cfg->max_tokens_per_rank;
    p.n_blocks = cfg->N / bn;
    p.num_k_blocks = cfg->K / box_k;
    p.msg_bytes = cfg->msg_bytes;
    p.max_rows = a->max_rows;
    p.expert_offsets = a->expert_offsets;
    p.src_info = a->src_info;
    p.seg_offsets = a->seg_offsets;
    p.send_counts = a->send_counts;
    for (int r = 0; r < R; ++r) {
        p.recv_buf[r] = a->recv_buf_ptrs[r];
        p.recv_count[r] = a->recv_count_ptrs[r];
    }
    p.atomic_counter = a->atomic_counter;
    p.rank_counter = a->rank_completion_counter;
    p.epoch = a->epoch;
    p.sink_enabled = sink ? 1 : 0;
    p.signal_mode = cfg->signal_mode;
    p.act_swiglu = !sink && a->local_activation == EP_ACT_SWIGLU ? 1 : 0;
    p.c_row_bytes = static_cast<int64_t>(cfg->N) * (p.act_swiglu ? 1 : 2);
    p.C = static_cast<uint8_t *>(a->C);
    p.status = a->status;
    p.timeout_ns = a->timeout_ns > 0 ? static_cast<uint64_t>(a->timeout_ns) : kDefaultTimeoutNs;
    p.a_scales = a->a_scales;
    p.w_scales = a->w_scales;
    p.trace = a->trace;
    p.trace_records = a->trace ? static_cast<int>(a->trace_records) : 0;
    p.overlap_previous = a->overlap_previous ? 1 : 0;
    // sink disabled ("EpiloguePeerSink" disabled: the local C store is the epilogue's
    // own): the bf16 output warps store whole 32-row groups of C with TMA
    if (!sink && !fp8 && cfg->send_warps != 4) {
        const int64_t c_cols = p.c_row_bytes / 2;
        if (!encode_2d(&p.tmap_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->C,
                           static_cast<uint64_t>(c_cols), static_cast<uint64_t>(a->max_rows),
                           static_cast<uint64_t>(p.c_row_bytes), 64, 32))
            return EP_ERR_CUDA;
        p.c_tma = 1;
    }

    // the plan lives on the device, so size the grid by the worst-case tile count
    const int64_t max_tiles = ((a->max_rows + ep::BM - 1) / ep::BM + El) * p.n_blocks;
    const int grid = static_cast<int>(max_tiles < num_sms ? (max_tiles < 1 ? 1 : max_tiles)
                                                          : num_sms);
    p.m_fastest = pick_m_fastest(rows_per_expert, pair ? 2 * ep::BM : ep::BM, p.n_blocks, cfg->K,
                                 cfg->N, elem, pair ? num_sms / 2 : grid) ? 1 : 0;
    out->ta = ta;
    out->tb = tb;
    out->p = p;
    out->bn = bn;
    out->send_warps = cfg->send_warps;
    out->grid = grid;
    out->kind = pair ? PreparedSend::kPair : fp8 ? PreparedSend::kFp8 : PreparedSend::kBf16;
    if (pair) {
        const int64_t pair_tiles = ((a->max_rows + 2 * ep::BM - 1) / (2 * ep::BM) + El) * p.n_blocks;
        out->max_pairs = static_cast<int>(
            pair_tiles < num_sms / 2 ? (pair_tiles < 1 ? 1 : pair_tiles) : num_sms / 2);
    }
    return EP_OK;
}

int launch_prepared_send(const PreparedSend &ps, cudaStream_t s)
{
    switch (ps.kind) {
    case PreparedSend::kPair:
        return cuda_status(
            launch_gemm_send_bf16_pair(ps.ta, ps.tb, ps.p, ps.send_warps, ps.max_pairs, s));
    case PreparedSend::kFp8:
        return cuda_status(launch_gemm_send_fp8(ps.ta, ps.tb, ps.p, ps.bn, ps.grid, s));
    default:
        return cuda_status(
            launch_gemm_send_bf16(ps.ta, ps.tb, ps.p, ps.bn, ps.send_warps, ps.grid, s));
    }
}

}  // namespace ep

extern "C" {

int grouped_gemm_combine_send(const ep_config *cfg, const ep_send_args *a, ep_stream_t stream)
{
    ep::PreparedSend ps;
    const int rc = ep::prepare_send(cfg, a, &ps);
    if (rc != EP_OK)
        return rc;
    return ep::launch_prepared_send(ps, reinterpret_cast<cudaStream_t>(stream));
}

int ep_scatter_send(const ep_config *cfg, const ep_scatter_args *a, ep_stream_t stream)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!a || !a->C || !a->expert_offsets || !a->src_info || !a->seg_offsets ||
        !a->send_counts || !a->block_counter || !a->status)
        return EP_ERR_INVALID_ARG;
    if (!aligned16(a->C) || (reinterpret_cast<uintptr_t>(a->src_info) & 7u) ||
        (reinterpret_cast<uintptr_t>(a->block_counter) & 3u))
        return EP_ERR_INVALID_ARG;
    if (a->max_rows < 1 || a->max_rows > INT32_MAX || cfg->N % 8 != 0)
        return EP_ERR_INVALID_ARG;
    const int R = cfg->n_ranks;
    ep::ScatterParams p;
    std::memset(&p, 0, sizeof p);
    for (int r = 0; r < R; ++r) {
        if (!a->recv_buf_ptrs[r] || !a->recv_count_ptrs[r] || !aligned16(a->recv_buf_ptrs[r]) ||
            (reinterpret_cast<uintptr_t>(a->recv_count_ptrs[r]) & 7u))
            return EP_ERR_INVALID_ARG;
        p.recv_buf[r] = static_cast<uint8_t *>(a->recv_buf_ptrs[r]);
        p.recv_count[r] = a->recv_count_ptrs[r];
    }
    const int num_sms = sm_count();
    if (num_sms <= 0)
        return EP_ERR_CUDA;
    p.n_ranks = R;
    p.my_rank = cfg->my_rank;
    p.El = cfg->n_local_experts;
    p.top_k = cfg->top_k;
    p.N = cfg->N;
    p.max_tokens = cfg->max_tokens_per_rank;
    p.msg_bytes = cfg->msg_bytes;
    p.max_rows = a->max_rows;
    p.C = static_cast<const uint8_t *>(a->C);
    p.expert_offsets = a->expert_offsets;
    p.src_info = a->src_info;
    p.seg_offsets = a->seg_offsets;
    p.send_counts = a->send_counts;
    p.block_counter = a->block_counter;
    p.epoch = a->epoch;
    p.status = a->status;
    p.signal_mode = cfg->signal_mode;
    return cuda_status(ep::launch_scatter(p, num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch_gather(const ep_config *cfg, const ep_dispatch_args *a, ep_stream_t stream)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!a || !a->gather_idx || !a->expert_offsets || !a->A_in || !a->status)
        return EP_ERR_INVALID_ARG;
    if (a->hidden < 8 || a->hidden % 8 != 0 || !aligned16(a->A_in) || a->max_rows < 1 ||
        a->max_rows > INT32_MAX)
        return EP_ERR_INVALID_ARG;
    ep::DispatchParams p;
    std::memset(&p, 0, sizeof p);
    for (int r = 0; r < cfg->n_ranks; ++r) {
        if (!a->x_ptrs[r] || !aligned16(a->x_ptrs[r]))
            return EP_ERR_INVALID_ARG;
        p.x[r] = static_cast<const uint8_t *>(a->x_ptrs[r]);
    }
    const int num_sms = sm_count();
    if (num_sms <= 0)
        return EP_ERR_CUDA;
    p.n_ranks = cfg->n_ranks;
    p.El = cfg->n_local_experts;
    p.top_k = cfg->top_k;
    p.T = cfg->num_tokens;
    p.max_tokens = cfg->max_tokens_per_rank;
    p.hidden = a->hidden;
    p.max_rows = a->max_rows;
    p.gather_idx = a->gather_idx;
    p.expert_offsets = a->expert_offsets;
    p.A_in = static_cast<uint8_t *>(a->A_in);
    p.status = a->status;
    return cuda_status(
        ep::launch_dispatch_gather(p, num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_swiglu(const ep_config *cfg, const ep_swiglu_args *a, ep_stream_t stream)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!a || !a->G || !a->A || !a->expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (a->inter < 8 || a->inter % 8 != 0 || !aligned16(a->G) || !aligned16(a->A) ||
        a->max_rows < 1 || a->max_rows > INT32_MAX)
        return EP_ERR_INVALID_ARG;
    const int num_sms = sm_count();
    if (num_sms <= 0)
        return EP_ERR_CUDA;
    ep::SwigluParams p;
    p.El = cfg->n_local_experts;
    p.inter = a->inter;
    p.max_rows = a->max_rows;
    p.G = static_cast<const uint8_t *>(a->G);
    p.A = static_cast<uint8_t *>(a->A);
    p.expert_offsets = a->expert_offsets;
    return cuda_status(ep::launch_swiglu(p, num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_combine_reduce(const ep_config *cfg, const ep_combine_args *a, ep_stream_t stream)
{
    int rc = check_config(cfg);
    if (rc != EP_OK)
        return rc;
    if (!a || !a->recv_buf || !a->recv_count || !a->status)
        return EP_ERR_INVALID_ARG;
    if (cfg->num_tokens > 0 && (!a->gates || !a->out))
        return EP_ERR_INVALID_ARG;
    if (cfg->signal_mode == EP_SIGNAL_PER_EXPERT && cfg->num_tokens > 0 && !a->topk_ids)
        return EP_ERR_INVALID_ARG;  // the per-token wait needs the token's experts
    if (cfg->N % 8 != 0 || !aligned16(a->recv_buf) || (a->out && !aligned16(a->out)) ||
        (reinterpret_cast<uintptr_t>(a->recv_count) & 7u))
        return EP_ERR_INVALID_ARG;
    if (a->overlap_previous < EP_OVERLAP_NONE || a->overlap_previous > EP_OVERLAP_INPUTS_READY)
        return EP_ERR_INVALID_ARG;
    const int num_sms = sm_count();
    if (num_sms <= 0)
        return EP_ERR_CUDA;
    ep::CombineParams p;
    p.n_ranks = cfg->n_ranks;
    p.El = cfg->n_local_experts;
    p.top_k = cfg->top_k;
    p.T = cfg->num_tokens;
    p.N = cfg->N;
    p.msg_bytes = cfg->msg_bytes;
    p.recv_buf = a->recv_buf;
    p.recv_count = a->recv_count;
    p.gates = a->gates;
    p.out = static_cast<uint8_t *>(a->out);
    p.epoch = a->epoch;
    p.timeout_ns = a->timeout_ns > 0 ? static_cast<uint64_t>(a->timeout_ns) : kDefaultTimeoutNs;
    p.status = a->status;
    p.topk_ids = a->topk_ids;
    p.signal_mode = cfg->signal_mode;
    p.overlap_previous = a->overlap_previous;
    return cuda_status(ep::launch_combine(p, num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

const char *ep_strerror(int code)
{
    switch (code) {
    case EP_OK:
        return "ok";
    case EP_ERR_INVALID_ARG:
        return "invalid argument";
    case EP_ERR_UNSUPPORTED:
        return "unsupported configuration";
    case EP_ERR_CUDA:
        return "CUDA runtime error";
    default:
        break;
    }
    if (code > 0) {
        if (code & EP_STATUS_TIMEOUT)
            return "device status: bounded wait timed out";
        if (code & EP_STATUS_BOUNDS)
            return "device status: destination outside the receive buffer";
        if (code & EP_STATUS_CAPACITY)
            return "device status: routed rows exceed the plan capacity";
        if (code & EP_STATUS_ROUTING)
            return "device status: expert id out of range";
        if (code & EP_STATUS_INTERNAL)
            return "device status: inconsistent tensor-memory allocation in a CTA pair";
    }
    return "unknown code";
}

}  // extern "C"
