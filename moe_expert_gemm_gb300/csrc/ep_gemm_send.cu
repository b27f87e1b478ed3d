// Grouped expert GEMM (bf16) with the EP-combine send fused into its epilogue.
//
// "EpiloguePeerSink" (Modular MAX Mojo API, sm100_structured output_writer): the
// epilogue hands its finished output tile to a sink instead of storing it to the
// local C; with the sink enabled the local store and its TMA descriptor do not
// exist. "P3PeerSendConfig": each valid row m of a tile (m < m_end) goes to the
// receive buffer of the rank owning its token, at
// (src_idx*top_k + src_topk)*msg_bytes + byte_off. "ep_signal_completion"
// (shmem/ep_comm, ep_ord_r with has_rank_flag): per-expert count words are plain
// stores made before an acquire-release election on a per-destination counter;
// the producer elected last publishes the rank flag.
//
// Design for sm_103a: one persistent CTA per SM walks a static schedule of
// (expert, 128-row block, BN-column block) tiles. Warp 0 issues TMA loads of A and
// W into a STAGES-deep ring of 128-byte-swizzled shared-memory tiles; warp 1
// allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16 per instruction) into
// one of two TMEM accumulators; warps 2-5 (one per TMEM lane quarter) drain an
// accumulator with tcgen05.ld, round to bf16, stage 32 rows x 64 columns per warp
// in shared memory and write each row's 128 contiguous bytes to its destination
// with 16-byte stores (8 lanes per row). The double-buffered accumulator lets the
// MMA of tile i+1 run while tile i is being sent. After a barrier over the four
// epilogue warps, the finished tile goes to warp 6, which counts tiles per expert
// and runs the completion signalling, off the output path.
//
// Variants: SEND = 4 adds four send warps (7-10) that store the rows the epilogue
// warps stage in two slots each ("EpiloguePeerSink" SendWarps). With the sink
// disabled the rows go to the local C, optionally through the gated activation
// (act_swiglu: each sub-tile pairs gate columns with the up columns BN/2 further on).
//
// Every wait is bounded (timeout_ns of %globaltimer): on expiry the kernel sets
// EP_STATUS_TIMEOUT, the other roles stop at their next wait, outstanding TMA
// loads and MMAs are waited for (again bounded), TMEM is freed and the CTA exits.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"
#include "ep_sink.cuh"

namespace ep {

// A staging slot's row destinations, handed with the slot from an epilogue warp to
// its send warp.
struct SendSlotMeta {
    unsigned long long row_base[32];
    int col_byte;
    int pad[3];
};

// SEND = 0: the output warps store their rows themselves. SEND = 4: four dedicated
// send warps ("EpiloguePeerSink" SendWarps), one per output warp, drain two staging
// slots per output warp, so that reading TMEM and rounding the next 64 columns
// overlaps the stores of the previous ones.
template <int BN, int STAGES, int SEND>
struct GemmLayout {
    static constexpr int kABytes = BM * kRowBytesK;
    static constexpr int kBBytes = BN * kRowBytesK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiWarps = 4;
    static constexpr int kSlots = SEND ? 2 : 1;    // staging slots per output warp
    static constexpr int kWarpStaging = 32 * 128;  // 32 rows x 64 bf16 columns
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStaging = kOffB + STAGES * kBBytes;
    static constexpr int kOffMeta = kOffStaging + kEpiWarps * kSlots * kWarpStaging;
    static constexpr int kOffBars =
        kOffMeta + (SEND ? kEpiWarps * kSlots * static_cast<int>(sizeof(SendSlotMeta)) : 0);
    // full, empty, acc_full x2, acc_empty x2, mma_done (+ slot_full, slot_empty per slot)
    static constexpr int kNumBars = 2 * STAGES + 5 + (SEND ? 2 * kEpiWarps * kSlots : 0);
    static constexpr int kOffSink = (kOffBars + kNumBars * 8 + 15) / 16 * 16;
    static constexpr int kEnd = kOffSink + static_cast<int>(sizeof(SinkShared));
    static constexpr int kSmemBytes = kEnd + 1024;  // slack to align the base to 1024
    static constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators
    // TMA, MMA, 4 output warps, completion (+ send warps)
    static constexpr int kThreads = 224 + 32 * SEND;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM columns");
    static_assert(SEND == 0 || SEND == kEpiWarps, "send warps: none, or one per output warp");
};

template <int BN, int STAGES, int SEND>
__global__ void __launch_bounds__(224 + 32 * SEND, 1)
    gemm_send_bf16_kernel(const __grid_constant__ CUtensorMap tmap_a,
                          const __grid_constant__ CUtensorMap tmap_b,
                          const __grid_constant__ SendParams p)
{
    using L = GemmLayout<BN, STAGES, SEND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBars);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *acc_full = bars + 2 * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *slot_full = mma_done + 1;  // [output warp][slot], SEND only
    uint64_t *slot_empty = slot_full + L::kEpiWarps * L::kSlots;
    SendSlotMeta *meta = reinterpret_cast<SendSlotMeta *>(smem + L::kOffMeta);
    SinkShared *sh = reinterpret_cast<SinkShared *>(smem + L::kOffSink);
    volatile int *abort_flag = &sh->abort_flag;
    const int El = p.El;

    // ---------------------------------------------------------------- prologue
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], L::kEpiWarps);
        }
        mbar_init(mma_done, 1);
        if (SEND) {
            for (int j = 0; j < L::kEpiWarps * L::kSlots; ++j) {
                mbar_init(&slot_full[j], 1);
                mbar_init(&slot_empty[j], 1);
            }
        }
        fence_mbar_init();
    }
    // the allocation and the descriptor prefetches overlap the prologue's loads
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(&sh->tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmap_a);
        tma_prefetch_map(&tmap_b);
    }
    griddep_wait();  // from here on global memory may be what the previous kernel wrote
    sink_prologue(p, sh);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_slot;
    const int total_tiles = sh->tile_start[El];

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t used_mask = 0, last_parity = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const TileCoord c = decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, BM, p.m_fastest);
                const int w_row = c.e * p.N + c.nb * BN;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
                    tma_load_2d(smem + L::kOffA + stage * L::kABytes, &tmap_a, &full[stage],
                                kb * 64, c.m_abs);
                    tma_load_2d(smem + L::kOffB + stage * L::kBBytes, &tmap_b, &full[stage],
                                kb * 64, w_row);
                    used_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                raise_abort(p.status, abort_flag);
            // loads complete whether or not anyone consumes them: wait for the last
            // one of every stage before the block may exit
            volatile int no_abort = 0;
            for (int s = 0; s < STAGES; ++s)
                if (used_mask & (1u << s))
                    mbar_wait(&full[s], (last_parity >> s) & 1u, p.timeout_ns, &no_abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(1u, BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++i) {
                const int as = i & 1;
                const uint32_t aphase = (i >> 1) & 1;
                if (!mbar_wait(&acc_empty[as], aphase ^ 1u, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * BN);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + L::kOffA + stage * L::kABytes);
                    const uint32_t b_addr = smem_u32(smem + L::kOffB + stage * L::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(d_tmem, desc_kmajor_sw128(a_addr + kk * 32),
                                desc_kmajor_sw128(b_addr + kk * 32), idesc,
                                (kb | kk) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(&acc_full[as]);
            }
            if (!ok)
                raise_abort(p.status, abort_flag);
            // every MMA issued so far has finished once this commit lands
            mma_commit(mma_done);
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, p.timeout_ns, &no_abort);
        }
        __syncwarp();
    } else if (warp < 6) {
        // --------------------------------------------------- epilogue + sink
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int epi_tid = threadIdx.x - 64;
        const uint32_t stg =
            smem_u32(smem + L::kOffStaging + (warp - 2) * L::kSlots * L::kWarpStaging);
        uint64_t *trace = epi_tid == 0 ? trace_block(p) : nullptr;
        if (trace)
            trace[1] = globaltimer_ns();

        bool ok = true;
        bool push_ok = true;  // epi_tid 0: the last hand-off to the completion warp succeeded
                              // (SEND: every wait of this warp for a free slot succeeded)
        int k_sub = 0;        // SEND: sub-tiles this warp has handed to its send warp
        const bool act = SEND == 0 && p.act_swiglu;  // gated-MLP epilogue (local C only)
        int i = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++i) {
            const TileCoord c = decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, BM, p.m_fastest);
            const int as = i & 1;
            const uint32_t aphase = (i >> 1) & 1;
            // resolve this thread's row destination while the MMA runs
            uint8_t *row_base = resolve_row(p, sh, c, c.m_abs + q * 32 + lane);

            ok = mbar_wait(&acc_full[as], aphase, p.timeout_ns, abort_flag) && push_ok;
            // all four epilogue warps take the same decision, so none is left waiting
            // at a named barrier that another has abandoned
            ok = named_bar_and(2, 128, ok);
            if (!ok)
                break;
            tc_fence_after();
            uint64_t *rec = (trace && i < p.trace_records) ? trace + 2 + 4 * i : nullptr;
            if (rec) {
                rec[0] = static_cast<uint64_t>(t) | (static_cast<uint64_t>(c.e) << 32);
                rec[1] = globaltimer_ns();
            }

            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(as * BN);
#pragma unroll 1
            for (int sub = 0; sub < (act ? BN / 128 : BN / 64); ++sub) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(t_row + sub * 64, v0);
                tmem_ld_32x32b_x32(t_row + sub * 64 + 32, v1);
                if (act) {
                    // gated MLP: this sub-tile's gate columns and, BN/2 further on, the
                    // up columns of the same intermediate indices
                    uint32_t u0[32], u1[32];
                    tmem_ld_32x32b_x32(t_row + BN / 2 + sub * 64, u0);
                    tmem_ld_32x32b_x32(t_row + BN / 2 + sub * 64 + 32, u1);
                    tmem_ld_wait();
                    tmem_regs_ready(v0);
                    tmem_regs_ready(v1);
                    tmem_regs_ready(u0);
                    tmem_regs_ready(u1);
#pragma unroll
                    for (int c2 = 0; c2 < 32; ++c2) {
                        swiglu_inplace(v0[c2], u0[c2]);
                        swiglu_inplace(v1[c2], u1[c2]);
                    }
                } else {
                    tmem_ld_wait();
                    tmem_regs_ready(v0);
                    tmem_regs_ready(v1);
                }
                const int col_byte = (c.nb * (act ? BN / 2 : BN) + sub * 64) * 2;
                uint32_t buf = stg;
                int slot = 0;
                if constexpr (SEND != 0) {
                    // wait until the send warp has drained this slot's previous contents
                    slot = (warp - 2) * L::kSlots + (k_sub % L::kSlots);
                    buf = stg + (k_sub % L::kSlots) * L::kWarpStaging;
                    const uint32_t sph = (k_sub / L::kSlots) & 1;
                    push_ok = mbar_wait(&slot_empty[slot], sph ^ 1u, p.timeout_ns, abort_flag) &&
                              push_ok;
                }
                // sink disabled, whole 32-row groups of the expert leave as one TMA store
                // from the staging buffer (the map's 128-byte swizzle is the buffer's);
                // the previous store of this warp must have read the buffer
                const int group_row = c.m_abs + q * 32;
                const bool tma_group = SEND == 0 && p.c_tma && group_row + 32 <= c.m_end;
                if (SEND == 0 && p.c_tma) {
                    if (lane == 0)
                        bulk_wait_read_all();
                    __syncwarp();
                }
                // fp32 -> bf16 (nearest even), this thread's row, 8 chunks of 16 bytes
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t *v = ch < 4 ? v0 + ch * 8 : v1 + (ch - 4) * 8;
                    uint32_t w[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        __nv_bfloat162 b = __float22bfloat162_rn(
                            make_float2(__uint_as_float(v[2 * h]), __uint_as_float(v[2 * h + 1])));
                        w[h] = *reinterpret_cast<uint32_t *>(&b);
                    }
                    st_shared_v4(buf + lane * 128 + ((ch ^ (lane & 7)) << 4),
                                 make_uint4(w[0], w[1], w[2], w[3]));
                }
                if constexpr (SEND != 0) {
                    // hand the slot, with its rows' destinations, to the send warp
                    meta[slot].row_base[lane] = reinterpret_cast<unsigned long long>(row_base);
                    if (lane == 0)
                        meta[slot].col_byte = col_byte;
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&slot_full[slot]);
                    ++k_sub;
                    continue;
                }
                if (tma_group) {
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmap_c, buf, col_byte / 2, group_row);
                        bulk_commit();
                    }
                    continue;
                }
                __syncwarp();
                // 8 lanes per row: each row's 128 bytes leave as one contiguous segment
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int row = it * 4 + (lane >> 3);
                    const int ch = lane & 7;
                    const unsigned long long base = __shfl_sync(
                        0xffffffffu, reinterpret_cast<unsigned long long>(row_base), row);
                    const uint4 val = ld_shared_v4(stg + row * 128 + ((ch ^ (row & 7)) << 4));
                    if (base != 0ull)
                        st_global_v4(reinterpret_cast<uint8_t *>(base) + col_byte + ch * 16, val);
                }
                __syncwarp();
            }
            // accumulator drained: hand it back to the MMA warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[as]);

            if (SEND != 0) {
                // the send warps hand the tile to the completion warp; a failed wait
                // for a slot is voted on at the next tile (or reported after the loop)
                push_ok = __all_sync(0xffffffffu, push_ok);
            } else if (p.sink_enabled) {
                // all 128 sink threads' stores of this tile precede the hand-off to the
                // completion warp, which counts the tile; a failed hand-off is voted
                // on at the next tile (or reported after the loop)
                named_bar_sync(1, 128);
                if (epi_tid == 0) {
                    if (rec)
                        rec[2] = globaltimer_ns();
                    const int tiles_e = (c.m_end - sh->eoff[c.e] + BM - 1) / BM * p.n_blocks;
                    push_ok = push_tile_done(p, sh, c.e, rec ? i : -1, tiles_e);
                }
            } else if (rec) {
                rec[2] = rec[3] = globaltimer_ns();
            }
        }
        // the local C's TMA stores have completed before the block ends
        if (SEND == 0 && p.c_tma && lane == 0)
            bulk_wait_all();
        if (epi_tid == 0) {
            if (trace)
                trace[0] = static_cast<uint64_t>(i);
            if (SEND == 0)
                close_queue(sh);
        }
        if ((!ok || !push_ok) && lane == 0)
            raise_abort(p.status, abort_flag);
    } else if (warp == 6) {
        // ------------------------------------------- completion counting + signalling
        if (lane == 0 && p.sink_enabled)
            completion_loop(p, sh);
        __syncwarp();
    } else if constexpr (SEND != 0) {
        // ------------------------------------------------------------ send warps
        // Send warp sw drains the slots of output warp sw in order: each row's 128
        // bytes of a sub-tile leave as one contiguous segment (8 lanes per row). After
        // a tile's last sub-tile the send warps meet at a barrier, which is also their
        // vote, and one thread hands the tile to the completion warp.
        const int sw = warp - 7;
        const int send_tid = threadIdx.x - 224;
        uint64_t *trace = send_tid == 0 ? trace_block(p) : nullptr;
        bool ok = true;
        bool push_ok = true;  // send_tid 0: the last hand-off succeeded
        int k = 0;
        int i = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++i) {
            const TileCoord c =
                decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, BM, p.m_fastest);
            for (int sub = 0; sub < BN / 64; ++sub, ++k) {
                const int slot = sw * L::kSlots + (k % L::kSlots);
                const uint32_t sph = (k / L::kSlots) & 1;
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&slot_full[slot], sph, p.timeout_ns, abort_flag));
                if (!ok)
                    break;
                const uint32_t buf = smem_u32(smem + L::kOffStaging + slot * L::kWarpStaging);
                const int col_byte = meta[slot].col_byte;
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int row = it * 4 + (lane >> 3);
                    const int ch = lane & 7;
                    const unsigned long long base = meta[slot].row_base[row];
                    const uint4 val = ld_shared_v4(buf + row * 128 + ((ch ^ (row & 7)) << 4));
                    if (base != 0ull)
                        st_global_v4(reinterpret_cast<uint8_t *>(base) + col_byte + ch * 16, val);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&slot_empty[slot]);
            }
            // every send thread's stores of this tile precede the hand-off
            ok = named_bar_and(3, 32 * SEND, ok && push_ok);
            if (!ok)
                break;
            if (send_tid == 0) {
                uint64_t *rec = (trace && i < p.trace_records) ? trace + 2 + 4 * i : nullptr;
                if (p.sink_enabled) {
                    if (rec)
                        rec[2] = globaltimer_ns();
                    const int tiles_e = (c.m_end - sh->eoff[c.e] + BM - 1) / BM * p.n_blocks;
                    push_ok = push_tile_done(p, sh, c.e, rec ? i : -1, tiles_e);
                } else if (rec) {
                    rec[2] = rec[3] = globaltimer_ns();
                }
            }
        }
        if (send_tid == 0)
            close_queue(sh);
        if ((!ok || !push_ok) && lane == 0)
            raise_abort(p.status, abort_flag);
    }

    // --------------------------------------------------------------- teardown
    // a combine launched behind this kernel may start now: it reads nothing before
    // acquiring the flags (or count words) this kernel releases
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
}

template <int BN, int STAGES, int SEND>
static cudaError_t launch_bn(const CUtensorMap &ta, const CUtensorMap &tb, const SendParams &p,
                             int grid, cudaStream_t s)
{
    using L = GemmLayout<BN, STAGES, SEND>;
    auto kern = gemm_send_bf16_kernel<BN, STAGES, SEND>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_send_kernel(kern, grid, L::kThreads, L::kSmemBytes, ta, tb, p, s);
}

cudaError_t launch_gemm_send_bf16(const CUtensorMap &ta, const CUtensorMap &tb,
                                  const SendParams &p, int bn, int send_warps, int grid,
                                  cudaStream_t s)
{
    if (send_warps == 4) {
        // the second staging slot of each output warp takes the room of one stage
        switch (bn) {
        case 256:
            return launch_bn<256, 3, 4>(ta, tb, p, grid, s);
        case 128:
            return launch_bn<128, 5, 4>(ta, tb, p, grid, s);
        case 64:
            return launch_bn<64, 7, 4>(ta, tb, p, grid, s);
        default:
            return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 256:
        return launch_bn<256, 4, 0>(ta, tb, p, grid, s);
    case 128:
        return launch_bn<128, 6, 0>(ta, tb, p, grid, s);
    case 64:
        return launch_bn<64, 8, 0>(ta, tb, p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace ep
