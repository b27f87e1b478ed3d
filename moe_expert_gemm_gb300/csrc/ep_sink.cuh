// The sink side of the fused expert GEMM, shared by the bf16 and fp8 kernels:
// tile schedule, per-row destination resolution, the hand-off of finished tiles
// to a completion warp, and the completion signalling.
//
// "EpiloguePeerSink": the finished output tile goes to the peers that own its rows
// instead of to the local C; rows m_abs <= m < m_end of the tile's group.
// "P3PeerSendConfig": row (src_idx, src_topk) lands at
// (src_idx*top_k + src_topk)*msg_bytes + byte_off of its rank's receive buffer; the
// count of expert e from rank rk sits at e*n_ranks + rk.
// "ep_signal_completion" (ep_ord_r, has_rank_flag): plain count stores before an
// acquire-release election on a per-destination counter bounded by the local
// expert count; the elected producer publishes the rank flag in the buffer tail.
#pragma once

#include "ep_internal.h"
#include "ep_ptx.cuh"

namespace ep {

constexpr int kQueue = 64;        // finished-tile queue, epilogue -> completion warp
constexpr int kCountCache = 512;  // send counts kept in shared memory when E_l * R fits

// Shared-memory state of the sink, one per thread block.
struct SinkShared {
    uint8_t *recv[EP_MAX_RANKS];
    uint64_t *cnt[EP_MAX_RANKS];
    int tile_start[EP_MAX_LOCAL_EXPERTS + 1];
    int eoff[EP_MAX_LOCAL_EXPERTS + 1];
    int counts[kCountCache];  // send_counts[e * R + dst], when E_l * R <= kCountCache
    int4 queue[kQueue];       // {expert, trace record or -1, tiles of the expert, 0}
    int q_head, q_tail, q_done, abort_flag;
    uint32_t tmem_slot;
};

__device__ __forceinline__ void raise_abort(uint32_t *status, volatile int *abort_flag)
{
    atomicOr(status, EP_STATUS_TIMEOUT);
    *abort_flag = 1;
}

// Completion signalling ("ep_signal_completion", ep_ord_r with has_rank_flag) is a
// chain of acquire-release steps kept as short as possible, because the completion
// of the last expert ends the call:
//  1. the count words are plain progress stores whose values the plan fixes, so block
//     0's completion thread stores all of them (store_counts, every expert) before
//     its first release; every release after that (its tile-counter RMWs, then the
//     election) carries them to whoever acquires;
//  2. each finished tile: one acquire-release RMW on its expert's tile counter
//     (gpu scope: all producers of the rank share its GPU), which releases the
//     tile's rows (stored by the output warps before the hand-off) and, for the
//     tile that completes the expert, acquires every other tile of it;
//  3. elect_and_publish, once per completed expert: one acquire-release RMW on the
//     election counter. In one fused call every expert completion signals every
//     destination (empty segments with count 0), so the per-destination counters
//     of the pages would move in lockstep: counter 0 elects the last expert for all
//     destinations at once. The elected block has acquired every other expert's
//     release through that RMW chain; its one system-scope fence is the single
//     system-scope release that carries the whole rank (cumulatively) to the peers,
//     followed by the rank flag of every destination. It re-arms the counter.
__device__ __forceinline__ void store_counts(const SendParams &p, const SinkShared *sh, int e)
{
    const int R = p.n_ranks;
    const bool cached = p.El * R <= kCountCache;
    int c[EP_MAX_RANKS];
#pragma unroll
    for (int dst = 0; dst < EP_MAX_RANKS; ++dst)
        c[dst] = dst < R ? (cached ? sh->counts[e * R + dst] : __ldg(p.send_counts + e * R + dst))
                         : 0;
#pragma unroll
    for (int dst = 0; dst < EP_MAX_RANKS; ++dst) {
        if (dst < R) {
            volatile uint64_t *w = sh->cnt[dst] + static_cast<int64_t>(e) * R + p.my_rank;
            *w = static_cast<uint64_t>(c[dst]);
        }
    }
}

// EP_SIGNAL_PER_EXPERT: the count word is the expert's arrival signal, tagged with
// the call's epoch ((epoch mod 2^32) << 32 | rows) and stored after the caller's
// system-scope fence (a release by the PTX release pattern); no election, no flag.
__device__ __forceinline__ void store_tagged_counts(const SendParams &p, const SinkShared *sh,
                                                    int e)
{
    const int R = p.n_ranks;
    const bool cached = p.El * R <= kCountCache;
    const uint64_t tag = (p.epoch & 0xFFFFFFFFull) << 32;
#pragma unroll
    for (int dst = 0; dst < EP_MAX_RANKS; ++dst) {
        if (dst < R) {
            const int c = cached ? sh->counts[e * R + dst] : __ldg(p.send_counts + e * R + dst);
            st_relaxed_sys_u64(sh->cnt[dst] + static_cast<int64_t>(e) * R + p.my_rank,
                               tag | static_cast<uint32_t>(c));
        }
    }
}

static __device__ __noinline__ void elect_and_publish(const SendParams &p, const SinkShared *sh)
{
    const int old = atom_add_acq_rel_gpu(&p.rank_counter[0], 1);
    if (old != p.El - 1)
        return;
    // last expert of this rank: re-arm the counter for the next call and publish the
    // whole rank through the rank flag of every destination
    *reinterpret_cast<volatile int *>(&p.rank_counter[0]) = 0;
    fence_acq_rel_sys();
    const int R = p.n_ranks;
#pragma unroll
    for (int dst = 0; dst < EP_MAX_RANKS; ++dst)
        if (dst < R)
            st_relaxed_sys_u64(sh->cnt[dst] + static_cast<int64_t>(p.El) * R + p.my_rank, p.epoch);
}

struct TileCoord {
    int e, m_abs, m_end, nb;
};

// Tiles are numbered expert by expert. Within an expert either the column block
// runs fastest (concurrent blocks share A rows and sweep W: best when W is the
// smaller operand) or the row block does (concurrent blocks share a W block and
// sweep A: best when A is smaller). A row block has `tile_rows` rows (128, or 256
// for a CTA pair).
__device__ __forceinline__ TileCoord decode_tile(int t, const int *tile_start, const int *eoff,
                                                 int El, int n_blocks, int tile_rows = BM,
                                                 bool m_fastest = false)
{
    // the largest expert whose first tile is <= t owns t (empty experts share starts)
    int lo = 0, hi = El - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    TileCoord c;
    c.e = lo;
    const int local = t - tile_start[lo];
    int mt;
    if (m_fastest) {
        const int m_blocks = (eoff[lo + 1] - eoff[lo] + tile_rows - 1) / tile_rows;
        c.nb = local / m_blocks;
        mt = local - c.nb * m_blocks;
    } else {
        mt = local / n_blocks;
        c.nb = local - mt * n_blocks;
    }
    c.m_abs = eoff[lo] + mt * tile_rows;
    c.m_end = eoff[lo + 1];
    return c;
}

// Called by every thread of the block: destination pointers, expert row ranges
// (made monotone and clamped to the rows of A so that a malformed plan cannot send
// reads past the plan arrays) and the tile table. Ends with __syncthreads.
__device__ __forceinline__ void sink_prologue(const SendParams &p, SinkShared *sh,
                                              int tile_rows = BM)
{
    const int El = p.El;
    if (threadIdx.x < EP_MAX_RANKS) {
        sh->recv[threadIdx.x] = p.recv_buf[threadIdx.x];
        sh->cnt[threadIdx.x] = p.recv_count[threadIdx.x];
    }
    if (threadIdx.x == 0) {
        sh->q_head = 0;
        sh->q_tail = 0;
        sh->q_done = 0;
        sh->abort_flag = 0;
    }
    // one pass issues both loads of a thread before either store
    const int n_cnt = p.sink_enabled && El * p.n_ranks <= kCountCache ? El * p.n_ranks : 0;
    const int n_all = n_cnt > El + 1 ? n_cnt : El + 1;
    for (int i = threadIdx.x; i < n_all; i += blockDim.x) {
        const int eo = i <= El ? __ldg(p.expert_offsets + i) : 0;
        const int cn = i < n_cnt ? __ldg(p.send_counts + i) : 0;
        if (i <= El)
            sh->eoff[i] = eo;
        if (i < n_cnt)
            sh->counts[i] = cn;
    }
    __syncthreads();
    if ((threadIdx.x >> 5) == 2) {
        // one warp, 32 experts at a time. Made monotone and clamped, the offsets are
        // min(max(0, raw_0 .. raw_e), max_rows): a prefix maximum, then the clamp.
        const int lane = threadIdx.x & 31;
        const int max_rows = static_cast<int>(p.max_rows);
        int carry = 0;
        for (int base = 0; base <= El; base += 32) {
            const int e = base + lane;
            int m = e <= El ? sh->eoff[e] : 0;
            m = m > carry ? m : carry;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, m, d);
                if (lane >= d)
                    m = o > m ? o : m;
            }
            carry = __shfl_sync(0xffffffffu, m, 31);
            if (e <= El)
                sh->eoff[e] = m < max_rows ? m : max_rows;
        }
        __syncwarp();
        // tile table: exclusive prefix sum of the experts' tile counts
        int acc = 0;
        for (int base = 0; base < El; base += 32) {
            const int e = base + lane;
            const int t = e < El
                              ? (sh->eoff[e + 1] - sh->eoff[e] + tile_rows - 1) / tile_rows * p.n_blocks
                              : 0;
            int incl = t;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += o;
            }
            if (e < El)
                sh->tile_start[e] = acc + incl - t;
            acc += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            sh->tile_start[El] = acc;
    }
    __syncthreads();
}

// Destination of row m of tile c: its slot in the receive buffer of the rank that
// owns its token (sink on), or its row of the local C (sink off). nullptr when the
// row lies past the group (m >= m_end) or its destination is outside the buffer
// (then EP_STATUS_BOUNDS is raised and the row is skipped).
__device__ __forceinline__ uint8_t *resolve_row(const SendParams &p, const SinkShared *sh,
                                                const TileCoord &c, int m)
{
    if (m >= c.m_end)
        return nullptr;
    if (!p.sink_enabled)
        return p.C + static_cast<int64_t>(m) * p.c_row_bytes;
    const int R = p.n_ranks;
    const int *seg = p.seg_offsets + c.e * (R + 1);
    int dst = -1;
    for (int rk = 0; rk < R; ++rk)
        if (m >= __ldg(seg + rk) && m < __ldg(seg + rk + 1))
            dst = rk;
    const int2 si = __ldg(reinterpret_cast<const int2 *>(p.src_info) + m);
    if (dst < 0 || si.x < 0 || si.x >= p.max_tokens || si.y < 0 || si.y >= p.top_k) {
        atomicOr(p.status, EP_STATUS_BOUNDS);
        return nullptr;
    }
    return sh->recv[dst] + (static_cast<int64_t>(si.x) * p.top_k + si.y) * p.msg_bytes;
}

__device__ __forceinline__ uint64_t *trace_block(const SendParams &p)
{
    return p.trace ? p.trace + static_cast<int64_t>(blockIdx.x) * (2 + 4 * p.trace_records)
                   : nullptr;
}

// One epilogue thread hands a finished tile (all of whose rows have been stored,
// as ordered by a barrier over the epilogue threads) to the completion warp.
// Bounded wait for a free slot; false when it gave up.
__device__ __forceinline__ bool push_tile_done(const SendParams &p, SinkShared *sh, int e,
                                               int record, int tiles_e)
{
    volatile int *head = &sh->q_head;
    volatile int *tail = &sh->q_tail;
    volatile int *abort_flag = &sh->abort_flag;
    const uint64_t t0 = globaltimer_ns();
    while (*tail - *head >= kQueue) {
        if (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns)
            return false;
    }
    const int tl = *tail;
    sh->queue[tl % kQueue] = make_int4(e, record, tiles_e, 0);
    __threadfence_block();
    *tail = tl + 1;
    return true;
}

// The epilogue has no more tiles (or gave up).
__device__ __forceinline__ void close_queue(SinkShared *sh)
{
    __threadfence_block();
    *reinterpret_cast<volatile int *>(&sh->q_done) = 1;
}

// Completion warp, one thread: counts finished tiles per expert (one acquire-release
// RMW per tile) and runs the signalling of every expert this block completes (rank
// flag: the election; per expert: one system-scope fence, tagged count words). Block
// 0 first stores every count word of the rank (rank flag) and signals the experts
// without rows, which have no tile to complete.
static __device__ void completion_loop(const SendParams &p, SinkShared *sh)
{
    volatile int *head_p = &sh->q_head;
    volatile int *tail_p = &sh->q_tail;
    volatile int *done_p = &sh->q_done;
    volatile int *abort_flag = &sh->abort_flag;
    uint64_t *trace = trace_block(p);
    const bool per_expert = p.signal_mode == EP_SIGNAL_PER_EXPERT;
    if (blockIdx.x == 0) {
        // every count word of the rank, before this thread's first release
        if (!per_expert)
            for (int e = 0; e < p.El; ++e)
                store_counts(p, sh, e);
        bool any_empty = false;
        for (int e = 0; e < p.El; ++e)
            any_empty |= sh->eoff[e + 1] == sh->eoff[e];
        if (any_empty) {
            if (per_expert)
                fence_acq_rel_sys();
            for (int e = 0; e < p.El; ++e) {
                if (sh->eoff[e + 1] == sh->eoff[e]) {
                    if (per_expert)
                        store_tagged_counts(p, sh, e);
                    else
                        elect_and_publish(p, sh);
                }
            }
        }
    }
    int head = 0;
    uint64_t t0 = globaltimer_ns();
    while (true) {
        const int tail = *tail_p;
        if (head < tail) {
            __threadfence_block();
            int4 ent[8];
            int n = 0;
            while (head < tail && n < 8)
                ent[n++] = sh->queue[(head++) % kQueue];
            __threadfence_block();
            *head_p = head;
            // each tile's rows released into its expert's tile counter; the tile that
            // completes the expert acquires the expert's other tiles
            bool last[8];
            bool any = false;
            for (int j = 0; j < n; ++j) {
                const int old = atom_add_acq_rel_gpu(&p.atomic_counter[ent[j].x], 1);
                last[j] = old == ent[j].z - 1;
                any |= last[j];
            }
            // per expert: the completed experts' rows go to the peers directly (each
            // count word is a system-scope release); with the rank flag, the election
            // releases them on this GPU
            if (any && per_expert)
                fence_acq_rel_sys();
            for (int j = 0; j < n; ++j) {
                if (last[j]) {
                    *reinterpret_cast<volatile int *>(&p.atomic_counter[ent[j].x]) = 0;
                    if (per_expert)
                        store_tagged_counts(p, sh, ent[j].x);
                    else
                        elect_and_publish(p, sh);
                }
                if (trace && ent[j].y >= 0) {
                    uint64_t *rec = trace + 2 + 4 * ent[j].y;
                    if (last[j])
                        rec[0] |= 1ull << 63;
                    rec[3] = globaltimer_ns();
                }
            }
            t0 = globaltimer_ns();
            continue;
        }
        if (*done_p) {
            __threadfence_block();
            if (*tail_p == head)
                break;
            continue;
        }
        if (*abort_flag)
            break;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
            raise_abort(p.status, abort_flag);
            break;
        }
    }
}

}  // namespace ep
