/*
 * moe_ep.h -- C ABI of the fused MoE expert-parallel down-projection:
 * grouped expert GEMM whose epilogue scatters rows straight into the combine
 * receive buffers of the token-owning ranks, completion signalling, and the
 * gate-weighted combine.
 *
 * Sources (Modular MAX Mojo API pages):
 *   "EpiloguePeerSink"     (linalg/matmul/gpu/sm100_structured/structured_kernels/output_writer)
 *   "P3PeerSendConfig"     (same directory)
 *   "ep_signal_completion" (shmem/ep_comm)
 *
 * General rules.
 *  - Every entry point is asynchronous on the caller's stream (`ep_stream_t`, a
 *    cudaStream_t; NULL is the legacy default stream) and returns EP_OK when the
 *    work was enqueued, or a negative EP_ERR_* code when the host found a problem,
 *    in which case nothing was launched.
 *  - The caller allocates and owns every buffer. The library allocates no device
 *    memory and keeps no per-call state (it caches only the SM count and kernel
 *    attributes of each device).
 *  - Problems found on the device (a destination outside the receive buffer, a
 *    bounded wait that ran out, a plan that does not fit) never trap: the kernel
 *    ORs an EP_STATUS_* bit into the caller's `status` word, skips the offending
 *    access and returns. Read the word after the stream has synchronised.
 *  - All device pointers must be 16-byte aligned.
 *  - Logical ranks: on one GPU, the receive buffers of the other ranks are simply
 *    other device allocations; with peer access they may be peer memory.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *ep_stream_t;

/* recv_buf_ptrs on "P3PeerSendConfig" is a StaticTuple of 8 pointers: at most
 * 8 ranks reachable by direct stores. */
#define EP_MAX_RANKS 8
/* Local experts per rank supported by one launch. */
#define EP_MAX_LOCAL_EXPERTS 256

/* host return codes */
#define EP_OK 0
#define EP_ERR_INVALID_ARG (-1)
#define EP_ERR_UNSUPPORTED (-2)
#define EP_ERR_CUDA (-3)

/* device status bits, OR-ed into *status */
#define EP_STATUS_BOUNDS 0x1u   /* a row's destination lay outside the receive buffer: row skipped */
#define EP_STATUS_TIMEOUT 0x2u  /* a bounded wait ran out (pipeline barrier or rank flag) */
#define EP_STATUS_CAPACITY 0x4u /* ep_plan: routed rows exceed max_rows; the plan is empty */
#define EP_STATUS_ROUTING 0x8u  /* ep_plan: an expert id outside [0, n_ranks*n_local_experts) */
#define EP_STATUS_INTERNAL 0x10u /* a CTA pair found inconsistent tensor-memory bases: no work done */

/* completion signalling ("ep_signal_completion") */
#define EP_SIGNAL_RANK_FLAG 0  /* ep_ord_r with has_rank_flag: plain count words, an
                                  acquire-release election, the elected producer
                                  release-stores the rank flag of every destination; the
                                  consumer acquires one flag per source rank */
#define EP_SIGNAL_PER_EXPERT 1 /* without ep_ord_r: every expert's count word is its own
                                  arrival signal, released once the expert's rows are
                                  written; no election, no rank flag; the consumer
                                  acquires, per token, the words of that token's experts */

/* operand types */
#define EP_BF16 0     /* bf16 A and W, fp32 accumulation, bf16 rows */
#define EP_FP8_1D2D 1 /* e4m3 A (1x128 fp32 scales) and W (128x128 fp32 scales), bf16 rows */

/*
 * Problem description shared by all calls.
 *   n_ranks              ranks taking part (1..EP_MAX_RANKS)   ["P3PeerSendConfig" n_ranks]
 *   my_rank              the rank this call plays               ["P3PeerSendConfig" my_rank]
 *   n_local_experts      experts per rank, E_l; global expert g lives on rank g / E_l at
 *                        local slot g % E_l                     ["ep_signal_completion"
 *                                                                n_experts_per_device]
 *   top_k                experts per token                      ["P3PeerSendConfig" top_k]
 *   num_tokens           tokens per source rank in this batch (T)
 *   max_tokens_per_rank  token capacity of each receive buffer (>= num_tokens)
 *                                                               ["P3PeerSendConfig"]
 *   K, N                 down-projection: rows of K inputs give rows of N outputs
 *   msg_bytes            bytes of one received row; must equal 2*N (bf16 rows)
 *   dtype                EP_BF16 or EP_FP8_1D2D
 *   send_warps           warps reserved for the sink above the output warps
 *                        ("EpiloguePeerSink" SendWarps): 0 runs the send inside the
 *                        output warps; 4 adds four send warps, one per output warp,
 *                        that store the rows the output warps stage (bf16 only, on
 *                        single CTAs and on CTA pairs; fp8 gives EP_ERR_UNSUPPORTED);
 *                        -1 lets the library choose (today: inside the output
 *                        warps). Any other value gives EP_ERR_INVALID_ARG.
 *   signal_mode          EP_SIGNAL_RANK_FLAG or EP_SIGNAL_PER_EXPERT; producers and
 *                        consumers of one exchange must use the same mode.
 */
typedef struct {
    int32_t n_ranks;
    int32_t my_rank;
    int32_t n_local_experts;
    int32_t top_k;
    int32_t num_tokens;
    int32_t max_tokens_per_rank;
    int32_t K;
    int32_t N;
    int32_t msg_bytes;
    int32_t dtype;
    int32_t send_warps;
    int32_t signal_mode;
} ep_config;

/* ------------------------------------------------------------------ plan */

/*
 * Receiving-side row plan of rank cfg->my_rank (the layout a dispatch step
 * produces and the grouped GEMM consumes). Rows of local expert e are
 * contiguous, ordered by source rank, then source token index, then top-k slot.
 * All arrays are device memory owned by the caller:
 *   expert_offsets [E_l+1]       first row of each local expert; [E_l] = row count
 *   src_info       [max_rows][2] (src_idx, src_topk) of each row ["P3PeerSendConfig"
 *                                src_info_ptr]
 *   seg_offsets    [E_l][R+1]    first row of each (expert, source rank) segment
 *   send_counts    [E_l][R]      rows of expert e from source rank rk: the count that
 *                                ep_signal_completion publishes to rk
 *   gather_idx     [max_rows]    flat routing index (rk*T + t)*top_k + j of each row
 *   m_total        [1]           row count
 *   status         [1]           EP_STATUS_* bits (OR-ed)
 * max_rows is the capacity of src_info / gather_idx (and of the A operand).
 * src_info is read and written as 8-byte pairs: it must be 8-byte aligned, else
 * EP_ERR_INVALID_ARG (here and in grouped_gemm_combine_send).
 */
typedef struct {
    int32_t *expert_offsets;
    int32_t *src_info;
    int32_t *seg_offsets;
    int32_t *send_counts;
    int32_t *gather_idx;
    int32_t *m_total;
    uint32_t *status;
    int64_t max_rows;
} ep_plan_out;

/* Worst-case row count of one rank: num_tokens * n_ranks * min(top_k, E_l).
 * Host only. Returns EP_OK or EP_ERR_INVALID_ARG. */
int ep_plan_sizes(const ep_config *cfg, int64_t *max_rows);

/*
 * Build the plan of cfg->my_rank from topk_ids, a device array
 * [n_ranks][num_tokens][top_k] of global expert ids. One small kernel; the
 * result is deterministic. If the rows exceed out->max_rows the kernel sets
 * EP_STATUS_CAPACITY and writes an empty plan (all offsets and counts 0).
 */
int ep_plan(const ep_config *cfg, const int32_t *topk_ids, const ep_plan_out *out,
            ep_stream_t stream);

/* -------------------------------------------- grouped GEMM + combine send */

/*
 * Runtime state of the fused send ("P3PeerSendConfig" fields, plus operands).
 *   A                [max_rows][K] bf16 or e4m3, row-major, rows in plan order. Rows at
 *                    or past the plan's row count are read (and ignored).
 *   a_scales         EP_FP8_1D2D only: [max_rows][K/128] fp32
 *   W                [E_l][N][K] bf16 or e4m3 (each expert's [N, K] weight, K contiguous)
 *   w_scales         EP_FP8_1D2D only: [E_l][N/128][K/128] fp32
 *   expert_offsets, src_info, seg_offsets, send_counts   the plan of my_rank (ep_plan)
 *   max_rows         rows allocated for A (and src_info)
 *   recv_buf_ptrs    [n_ranks] receive buffers, max_tokens_per_rank*top_k*msg_bytes bytes
 *                    each. The row of (src_idx, src_topk) from the token-owning rank goes
 *                    to byte (src_idx*top_k + src_topk)*msg_bytes + 2*n of that rank's
 *                    buffer ("P3PeerSendConfig" recv_buf_layout).
 *   recv_count_ptrs  [n_ranks] receive-count buffers, E_l*n_ranks + n_ranks uint64 words
 *                    each: word e*n_ranks + rk holds the rows expert e of rank rk sent
 *                    ("P3PeerSendConfig" recv_count_layout); word E_l*n_ranks + rk is
 *                    rank rk's completion flag ("ep_signal_completion" rank_flag_offset,
 *                    the buffer tail). With EP_SIGNAL_RANK_FLAG a count word holds the
 *                    row count and the flag the epoch; with EP_SIGNAL_PER_EXPERT a
 *                    count word holds (epoch mod 2^32) << 32 | rows and the flag words
 *                    are not written.
 *   atomic_counter   [E_l] int32 tile-completion counters of my_rank's experts
 *   rank_completion_counter  [n_ranks] int32 election counters. In one call every
 *                    expert's completion signals every destination (count 0 for an
 *                    empty segment), so the per-destination counters would always
 *                    hold the same value: element 0 elects the last expert for all
 *                    destinations, the other elements are not used.
 *                    Both counter arrays must be zero before the first call; every
 *                    call that completes without a status bit leaves them at zero.
 *   epoch            value released into the rank flags (or the count words' high
 *                    half); use a new value per call (e.g. 1, 2, 3, ...) so a consumer
 *                    can tell calls apart.
 *   p3_control       >= 0: the sink owns the output (no local C); < 0: the sink is
 *                    disabled and rows go to the local C instead, with no signalling
 *                    ("EpiloguePeerSink" p3_control: negative disables the sink).
 *   C                [max_rows][N] bf16, used only when p3_control < 0.
 *   status           device word for EP_STATUS_* bits.
 *   trace            optional (NULL: off) per-tile timestamps ("P3PeerSendConfig" fields
 *                    trace_ptr / trace_on / send_stamp_ptr): thread block b owns the
 *                    2 + 4*trace_records words starting at b*(2 + 4*trace_records):
 *                    [0] tiles it processed, [1] %globaltimer (ns) at its start, then
 *                    one record per tile (the first trace_records tiles):
 *                    {tile | expert << 32 | completed-the-expert << 63,
 *                     time the accumulator was ready, time the tile's rows were all
 *                     stored, time its completion counting (and signalling) ended}.
 *                    Allocate at least (#SMs) * (2 + 4*trace_records) words. Where two
 *                    thread blocks share a tile (bf16, 256-column tiles: CTA pairs),
 *                    each records it.
 *   timeout_ns       limit of each bounded wait inside the kernel (0: 2 s).
 *   trace_records    records per thread block in `trace` (>= 1 when trace is set).
 *   overlap_previous nonzero: launch as a programmatic dependent of the previous kernel
 *                    on `stream`. The thread blocks then start while that kernel is
 *                    still finishing and do their set-up (barriers, tensor memory,
 *                    descriptor prefetch) meanwhile, and wait for its completion and
 *                    memory before reading or writing any global memory, so the
 *                    previous kernel may produce the plan or the operands.
 *   local_activation with p3_control < 0 only (else ignored): EP_ACT_NONE stores the
 *                    rows as they are; EP_ACT_SWIGLU makes the call the up/gate
 *                    projection of a gated MLP with the activation in its epilogue:
 *                    W's rows come in interleaved 128-row blocks (rows 256b..256b+127
 *                    are the gate rows of intermediate indices 128b..128b+127, the next
 *                    128 rows the up rows of the same indices), and C receives
 *                    [max_rows][N/2] bf16 rows bf16(SiLU(gate) * up) computed from the
 *                    fp32 accumulators (SiLU(x) = x / (1 + e^-x), fp32). Needs bf16,
 *                    N % 256 == 0 and send_warps != 4, else EP_ERR_UNSUPPORTED.
 */
#define EP_ACT_NONE 0
#define EP_ACT_SWIGLU 1

typedef struct {
    const void *A;
    const float *a_scales;
    const void *W;
    const float *w_scales;
    const int32_t *expert_offsets;
    const int32_t *src_info;
    const int32_t *seg_offsets;
    const int32_t *send_counts;
    int64_t max_rows;
    uint8_t *recv_buf_ptrs[EP_MAX_RANKS];
    uint64_t *recv_count_ptrs[EP_MAX_RANKS];
    int32_t *atomic_counter;
    int32_t *rank_completion_counter;
    uint64_t epoch;
    int32_t p3_control;
    void *C;
    uint32_t *status;
    uint64_t *trace;
    int64_t timeout_ns;
    int64_t trace_records;
    int32_t local_activation;
    int32_t overlap_previous;
} ep_send_args;

/*
 * One persistent kernel: for every local expert e and every 128-row tile of its
 * rows (256-row tiles on CTA pairs, bf16) and every column block, Y_e = A_e * W_e^T
 * on the tensor cores (fp32 accumulation), rounded to bf16 and written row by row to
 * the receive buffer of the rank that owns each row's token. No local C tensor
 * exists ("EpiloguePeerSink" Enabled: the local store and its TMA descriptor are
 * dead).
 * EP_SIGNAL_RANK_FLAG: the count words are plain progress stores (made once, at the
 * start of the call, before any release); when the last tile of expert e is done,
 * an acquire-release increment of the election counter; the completion that sees
 * E_l-1 release-stores (system scope) `epoch` into every destination's flag word for
 * my_rank ("ep_signal_completion", ep_ord_r with has_rank_flag). EP_SIGNAL_PER_EXPERT: the count words, tagged with
 * the epoch, are released for each expert; no election, no flag. Experts with no
 * rows signal count 0.
 */
int grouped_gemm_combine_send(const ep_config *cfg, const ep_send_args *args,
                              ep_stream_t stream);

/*
 * grouped_gemm_combine_send_noalloc -- the same fused GEMM + send for callers
 * that cannot allocate device memory. The pages have no counterpart to this entry
 * point; it exists for library users.
 *
 * Who needs it: hosts that own every device allocation and forbid allocating
 * inside their per-call path (an inference engine running kernels from a
 * plugin's enqueue callback, a serving loop with a fixed memory budget), because
 * cudaMalloc can implicitly synchronise the device and stall other streams, or
 * break up a pool the host manages. Such a caller still passes every input and
 * output in `args`, but not the counter arrays: args->atomic_counter and
 * args->rank_completion_counter are ignored. The library keeps both in one
 * file-scope device array of EP_NOALLOC_SCRATCH_INTS int32 words
 * (EP_MAX_LOCAL_EXPERTS tile counters, then EP_MAX_RANKS election counters;
 * 1056 bytes) that every GPU loading the library holds until the process exits.
 *
 * Behaviour:
 *  - n_local_experts > EP_MAX_LOCAL_EXPERTS or n_ranks > EP_MAX_RANKS: returns
 *    EP_ERR_UNSUPPORTED, nothing is enqueued. Every check of
 *    grouped_gemm_combine_send runs before anything is enqueued, so a call that
 *    returns an error enqueues nothing.
 *  - Each call outside stream capture looks up the current device's address of
 *    the array (with that device current), so the address stays right after a
 *    cudaDeviceReset. A call on a stream being captured uses the address found
 *    by the last earlier call on that device: make the first call on a device
 *    before any stream capture (else EP_ERR_CUDA).
 *  - Every call shares the array and it keeps the last call's contents, so each
 *    call first clears it with an asynchronous memset on `stream` (no allocation).
 *    Calls that overlap on the GPU (e.g. on two streams at once) race on the
 *    counters: issue them in order on one stream.
 *  - overlap_previous gives no overlap here: the kernel launches behind that
 *    memset, so it starts only after the previous work on `stream` has ended.
 *  - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 * Everything else (arguments, results, signalling, status bits) is exactly as for
 * grouped_gemm_combine_send.
 */
#define EP_NOALLOC_SCRATCH_INTS (EP_MAX_LOCAL_EXPERTS + EP_MAX_RANKS)

int grouped_gemm_combine_send_noalloc(const ep_config *cfg, const ep_send_args *args,
                                      ep_stream_t stream);

/* ------------------------------------------------------- unfused send */

/*
 * ep_scatter_send -- the send step on its own, for the unfused comparator
 * ("EpiloguePeerSink" disabled, i.e. the null sink: the grouped GEMM stores its
 * output tile to the local C, here grouped_gemm_combine_send with p3_control < 0,
 * and a separate kernel then moves the rows). It reads the local C produced that
 * way and delivers exactly what the fused call delivers: every row to
 * (src_idx*top_k + src_topk)*msg_bytes of its destination's receive buffer
 * ("P3PeerSendConfig"), the count words, and the rank flag of my_rank in every
 * destination's count buffer ("ep_signal_completion"), the flag after all rows
 * and counts (one launch sends every expert, so the last thread block to finish
 * signals all of them at once).
 *   C                [max_rows][N] bf16, row m = output row m in plan order
 *   expert_offsets, src_info, seg_offsets, send_counts   the plan (ep_plan)
 *   max_rows         rows allocated for C (and src_info)
 *   recv_buf_ptrs, recv_count_ptrs, epoch, status   as for grouped_gemm_combine_send
 *   block_counter    one int32 in device memory, 0 before the first call; the call
 *                    that uses it re-arms it to 0
 * Errors: as for grouped_gemm_combine_send (EP_ERR_INVALID_ARG for NULL or
 * misaligned pointers, src_info not 8-byte aligned; EP_STATUS_BOUNDS for a row
 * whose destination lies outside the receive buffer, which is skipped).
 */
typedef struct {
    const void *C;
    const int32_t *expert_offsets;
    const int32_t *src_info;
    const int32_t *seg_offsets;
    const int32_t *send_counts;
    int64_t max_rows;
    void *recv_buf_ptrs[EP_MAX_RANKS];
    uint64_t *recv_count_ptrs[EP_MAX_RANKS];
    int32_t *block_counter;
    uint64_t epoch;
    uint32_t *status;
} ep_scatter_args;

int ep_scatter_send(const ep_config *cfg, const ep_scatter_args *args, ep_stream_t stream);

/* ------------------------------------------------------------- MoE layer */

/*
 * The steps before the down-projection, for running a whole MoE layer on this
 * library: dispatch, the up/gate projection, the gated activation. The pages
 * describe only the down-projection and its combine; they imply the dispatch
 * through the plan's row order and src_info. The up/gate projection is
 * grouped_gemm_combine_send itself with p3_control < 0 (rows to a local buffer),
 * called with K = hidden size and N = 2 * intermediate size (msg_bytes = 2*N).
 *
 * ep_dispatch_gather -- every routed token row to the rank that owns its expert,
 * in plan order.
 *   x_ptrs          [n_ranks] source ranks' tokens, [max_tokens_per_rank][hidden]
 *                   bf16 each (peer memory or, on one GPU, other allocations)
 *   gather_idx, expert_offsets   the plan of my_rank (ep_plan)
 *   max_rows        rows allocated for A_in
 *   hidden          row length in elements, a multiple of 8
 *   A_in            [max_rows][hidden] bf16 out: row m = x_rk[t] for the plan's
 *                   row m = (rk, t, j)
 *   status          EP_STATUS_BOUNDS for a gather index outside the token tables
 *                   (that row skipped)
 */
typedef struct {
    const void *x_ptrs[EP_MAX_RANKS];
    const int32_t *gather_idx;
    const int32_t *expert_offsets;
    int64_t max_rows;
    int32_t hidden;
    void *A_in;
    uint32_t *status;
} ep_dispatch_args;

int ep_dispatch_gather(const ep_config *cfg, const ep_dispatch_args *args, ep_stream_t stream);

/*
 * ep_swiglu -- the gated activation between the up/gate and down projections:
 *   A[m][i] = bf16( SiLU(G[m][i]) * G[m][inter + i] ),  SiLU(x) = x / (1 + e^-x),
 * in fp32 from the bf16 G, rounded to nearest even once, for m below the plan's
 * row count.
 *   G               [max_rows][2*inter] bf16: the up/gate GEMM's rows, gate half first
 *   A               [max_rows][inter] bf16 out: the down-projection's A
 *   expert_offsets  the plan of my_rank (row count at [E_l])
 *   inter           a multiple of 8
 */
typedef struct {
    const void *G;
    void *A;
    const int32_t *expert_offsets;
    int64_t max_rows;
    int32_t inter;
} ep_swiglu_args;

int ep_swiglu(const ep_config *cfg, const ep_swiglu_args *args, ep_stream_t stream);

/* --------------------------------------------------------------- combine */

/*
 * Gate-weighted combine on rank cfg->my_rank.
 *   recv_buf    this rank's receive buffer (layout above)
 *   recv_count  this rank's receive-count buffer (layout above)
 *   gates       [num_tokens][top_k] fp32
 *   out         [num_tokens][N] bf16: out[t][n] = bf16(sum_j gates[t][j] * row(t, j)[n])
 *   epoch       the flag value to wait for from every source rank
 *   timeout_ns  limit of the flag wait (0: 2 s); on expiry EP_STATUS_TIMEOUT is set
 *               and the affected outputs are left unwritten
 *   topk_ids    EP_SIGNAL_PER_EXPERT only: this rank's routing, [num_tokens][top_k]
 *               global expert ids (the table ep_plan reads, rank my_rank's part)
 *   overlap_previous  EP_OVERLAP_NONE (0): launch after the previous work on `stream`
 *               has ended. EP_OVERLAP_ANY: launch as a programmatic dependent of the
 *               previous kernel on `stream`; the combine reads no row before acquiring
 *               the signal that releases it, and reads the gates, the routing and `out`
 *               only after the previous kernel has completed and its memory is visible
 *               (with the rank flags it acquires the flags first, so that this wait
 *               overlaps the end of a send). EP_OVERLAP_INPUTS_READY: the same launch
 *               for a caller that guarantees the previous kernel writes none of the
 *               gates, the routing and `out` (e.g. it is this library's fused send):
 *               no wait, so the combine's reads start while that kernel finishes.
 * EP_SIGNAL_RANK_FLAG: each thread block acquires every source rank's flag once
 * (system scope) before reading the rows, as the fused consumer of
 * "ep_signal_completion" does. EP_SIGNAL_PER_EXPERT: before reducing a token, the
 * warp acquires the count words of that token's top_k experts, so tokens whose
 * experts have all arrived are reduced even while other experts are still sending.
 */
#define EP_OVERLAP_NONE 0
#define EP_OVERLAP_ANY 1
#define EP_OVERLAP_INPUTS_READY 2

typedef struct {
    const uint8_t *recv_buf;
    const uint64_t *recv_count;
    const float *gates;
    void *out;
    uint64_t epoch;
    int64_t timeout_ns;
    uint32_t *status;
    const int32_t *topk_ids;
    int32_t overlap_previous;
} ep_combine_args;

int ep_combine_reduce(const ep_config *cfg, const ep_combine_args *args, ep_stream_t stream);

/* ------------------------------------------------- peers in other processes */

/*
 * Sharing receive buffers between the processes of an expert-parallel group on one
 * node, one rank per process. "ep_signal_completion" sends by direct memory access
 * when the target device is on the same node, and "P3PeerSendConfig" holds one
 * receive-buffer pointer per rank (recv_buf_ptrs): each rank exports the buffers
 * its peers write (its receive buffer and its receive-count buffer), every other
 * rank imports them and passes the imported pointers in ep_send_args.recv_buf_ptrs /
 * recv_count_ptrs. The kernels then store rows, count words and flags there exactly
 * as into local buffers (plain stores, system-scope releases). Carrying the handle
 * bytes from process to process is the caller's business (any host channel).
 *
 * ep_ipc_export  dev_ptr: a device buffer of the calling process, allocated with
 *                cudaMalloc (directly, or inside a block of a caching allocator; not
 *                VMM or stream-ordered pool memory). Fills *out with a CUDA IPC handle
 *                of the allocation holding it, dev_ptr's offset in that allocation
 *                and the bytes from dev_ptr to the allocation's end.
 *                EP_ERR_INVALID_ARG for NULL or a pointer that is not device memory
 *                of the current context; EP_ERR_CUDA if the runtime refuses a handle.
 * ep_ipc_import  maps an exported buffer of another process into this one (on the
 *                current device; peer access is enabled when that is another GPU)
 *                and returns its address in *dev_ptr. A process cannot import its own
 *                handles. EP_ERR_CUDA if the runtime refuses.
 * ep_ipc_close   unmaps a buffer ep_ipc_import mapped (same handle and address).
 * The exporting process must keep the buffer allocated until every importer has
 * closed it: a store into a buffer whose owner freed it is an invalid access.
 * These three calls are synchronous host calls (no stream).
 */
#define EP_IPC_HANDLE_BYTES 64

typedef struct {
    uint8_t handle[EP_IPC_HANDLE_BYTES];
    uint64_t offset;
    uint64_t bytes;
} ep_ipc_handle;

int ep_ipc_export(const void *dev_ptr, ep_ipc_handle *out);
int ep_ipc_import(const ep_ipc_handle *h, void **dev_ptr);
int ep_ipc_close(const ep_ipc_handle *h, void *dev_ptr);

/* Static description of a return code or status bit set. */
const char *ep_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EP_H */
