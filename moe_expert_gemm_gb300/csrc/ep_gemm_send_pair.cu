// Grouped expert GEMM (bf16) with the fused EP-combine send, on CTA pairs.
//
// Same computation and sink as the single-CTA kernel ("EpiloguePeerSink",
// "P3PeerSendConfig", "ep_signal_completion"); this variant spends half the
// shared-memory operand traffic per FLOP. Two CTAs of a cluster share one
// 256 x 256 tile of one expert: CTA r loads its 128 rows of A and the 128-row
// half r of the W block, and the even CTA issues tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 16), which reads the A and B halves from both CTAs'
// shared memory and writes rows 128 r .. 128 r + 127 of the accumulator into the
// TMEM of CTA r. Each CTA then drains and sends its own 128 rows exactly as the
// single-CTA kernel does.
//
// Pair protocol:
//  * both CTAs allocate and later free TMEM together (cta_group::2);
//  * every stage's TMA loads of both CTAs complete on the even CTA's full barrier,
//    which expects the bytes of both;
//  * the even CTA's commits reach both CTAs' stage-free and accumulator-full
//    barriers (multicast), and both CTAs' epilogues release an accumulator on the
//    even CTA's barrier;
//  * a cluster barrier after set-up (all barriers initialised, TMEM allocated) and
//    one before the TMEM is freed (no MMA still writing the peer's TMEM).
// All waits except these two cluster barriers are bounded; every role reaches
// the final cluster barrier on every path.
//
// SEND = 4 adds four send warps (7-10), one per output warp, that store the rows
// the output warps stage in two slots each ("EpiloguePeerSink" SendWarps: the
// output warps go back to reading the accumulator while the previous 64 columns
// leave); the second slot takes the room of one operand stage.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"
#include "ep_sink.cuh"

namespace ep {

// A staging slot's row destinations, handed with the slot from an output warp to its
// send warp (SEND = 4).
struct PairSlotMeta {
    unsigned long long row_base[32];
    int col_byte;
    int pad[3];
};

template <int SEND>
struct PairLayout {
    static constexpr int BN = 256;
    static constexpr int STAGES = SEND ? 5 : 6;
    static constexpr int kAccStages = 2;              // TMEM accumulators per CTA
    static constexpr int kTileRows = 2 * BM;          // rows of a pair tile
    static constexpr int kABytes = BM * kRowBytesK;   // this CTA's 128 rows of A
    static constexpr int kBBytes = (BN / 2) * kRowBytesK;  // this CTA's half of the W block
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kEpiWarps = 4;
    static constexpr int kSlots = SEND ? 2 : 1;    // staging slots per output warp
    static constexpr int kWarpStaging = 32 * 128;  // 32 rows x 64 bf16 columns
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffStaging = kOffB + STAGES * kBBytes;
    static constexpr int kOffMeta = kOffStaging + kEpiWarps * kSlots * kWarpStaging;
    static constexpr int kOffBars =
        kOffMeta + (SEND ? kEpiWarps * kSlots * static_cast<int>(sizeof(PairSlotMeta)) : 0);
    // full, empty, acc_full x2, acc_empty x2, mma_done (+ slot_full, slot_empty per slot)
    static constexpr int kNumBars = 2 * STAGES + 5 + (SEND ? 2 * kEpiWarps * kSlots : 0);
    static constexpr int kOffSink = (kOffBars + kNumBars * 8 + 15) / 16 * 16;
    static constexpr int kEnd = kOffSink + static_cast<int>(sizeof(SinkShared));
    static constexpr int kSmemBytes = kEnd + 1024;
    static constexpr uint32_t kTmemCols = kAccStages * BN;
    // TMA, MMA, 4 output warps, completion (+ send warps)
    static constexpr int kThreads = 224 + 32 * SEND;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(SEND == 0 || SEND == kEpiWarps, "send warps: none, or one per output warp");
};

template <int SEND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(224 + 32 * SEND, 1)
    gemm_send_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                               const __grid_constant__ CUtensorMap tmap_b,
                               const __grid_constant__ SendParams p)
{
    using L = PairLayout<SEND>;
    constexpr int BN = L::BN;
    constexpr int STAGES = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBars);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *acc_full = bars + 2 * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *slot_full = mma_done + 1;  // [output warp][slot], SEND only
    uint64_t *slot_empty = slot_full + L::kEpiWarps * L::kSlots;
    PairSlotMeta *meta = reinterpret_cast<PairSlotMeta *>(smem + L::kOffMeta);
    SinkShared *sh = reinterpret_cast<SinkShared *>(smem + L::kOffSink);
    volatile int *abort_flag = &sh->abort_flag;
    const int El = p.El;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < L::kAccStages; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 2 * L::kEpiWarps);  // both CTAs' epilogue warps
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
        tmem_alloc_pair(&sh->tmem_slot, L::kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tmap_a);
        tma_prefetch_map(&tmap_b);
    }
    griddep_wait();  // from here on global memory may be what the previous kernel wrote
    sink_prologue(p, sh, L::kTileRows);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = sh->tmem_slot;
    // the pair MMA writes both CTAs' TMEM at one address: both allocations must agree
    const uint32_t peer_base = ld_shared_cluster_u32(mapa_shared(smem_u32(&sh->tmem_slot), rank ^ 1u));
    const bool tmem_ok = peer_base == tmem_base;
    if (!tmem_ok && threadIdx.x == 0)
        atomicOr(p.status, EP_STATUS_INTERNAL);
    const int total_tiles = tmem_ok ? sh->tile_start[El] : 0;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t used_mask = 0, last_parity = 0;
            bool ok = true;
            for (int t = pair; t < total_tiles && ok; t += n_pairs) {
                const TileCoord c =
                    decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, L::kTileRows, p.m_fastest);
                const int a_row = c.m_abs + static_cast<int>(rank) * BM;
                const int w_row = c.e * p.N + c.nb * BN + static_cast<int>(rank) * (BN / 2);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait_cluster(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_lead = mapa_shared(smem_u32(&full[stage]), 0);
                    if (leader)
                        mbar_arrive_expect_tx(&full[stage], 2 * L::kStageBytes);
                    tma_load_2d_pair(smem + L::kOffA + stage * L::kABytes, &tmap_a, full_lead,
                                     kb * 64, a_row);
                    tma_load_2d_pair(smem + L::kOffB + stage * L::kBBytes, &tmap_b, full_lead,
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
            volatile int no_abort = 0;
            if (leader) {
                // the even CTA's full barriers count both CTAs' loads
                for (int s = 0; s < STAGES; ++s)
                    if (used_mask & (1u << s))
                        mbar_wait_cluster(&full[s], (last_parity >> s) & 1u, p.timeout_ns,
                                          &no_abort);
            } else if (!ok) {
                // give loads already issued time to land before this CTA may exit
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = make_idesc(1u, 2 * BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int i = 0;
            for (int t = pair; t < total_tiles && ok; t += n_pairs, ++i) {
                const int as = i % L::kAccStages;
                const uint32_t aphase = (i / L::kAccStages) & 1;
                if (!mbar_wait_cluster(&acc_empty[as], aphase ^ 1u, p.timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(as * BN);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait_cluster(&full[stage], phase, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + L::kOffA + stage * L::kABytes);
                    const uint32_t b_addr = smem_u32(smem + L::kOffB + stage * L::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_pair(d_tmem, desc_kmajor_sw128(a_addr + kk * 32),
                                     desc_kmajor_sw128(b_addr + kk * 32), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                    mma_commit_pair(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit_pair(&acc_full[as], 0x3);
            }
            if (!ok)
                raise_abort(p.status, abort_flag);
            mma_commit_pair(mma_done, 0x1);
            volatile int no_abort = 0;
            mbar_wait_cluster(mma_done, 0, p.timeout_ns, &no_abort);
        }
        __syncwarp();
    } else if (warp < 6) {
        // --------------------------------------------------- epilogue + sink
        const int q = warp & 3;
        const int epi_tid = threadIdx.x - 64;
        // this output warp's staging slots (one, or two with send warps)
        const uint32_t stg =
            smem_u32(smem + L::kOffStaging + (warp - 2) * L::kSlots * L::kWarpStaging);
        uint64_t *trace = epi_tid == 0 ? trace_block(p) : nullptr;
        if (trace)
            trace[1] = globaltimer_ns();
        uint32_t acc_empty_lead[L::kAccStages];
#pragma unroll
        for (int a = 0; a < L::kAccStages; ++a)
            acc_empty_lead[a] = mapa_shared(smem_u32(&acc_empty[a]), 0);

        bool ok = true;
        bool push_ok = true;  // SEND: every wait of this warp for a free slot succeeded
        int k_sub = 0;        // SEND: sub-tiles this warp has handed to its send warp
        const bool act = SEND == 0 && p.act_swiglu != 0;  // gated-MLP epilogue (local C only)
        int i = 0;
        for (int t = pair; t < total_tiles; t += n_pairs, ++i) {
            const TileCoord c =
                decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, L::kTileRows, p.m_fastest);
            const int as = i % L::kAccStages;
            const uint32_t aphase = (i / L::kAccStages) & 1;
            const int row0 = c.m_abs + static_cast<int>(rank) * BM;
            uint8_t *row_base = resolve_row(p, sh, c, row0 + q * 32 + lane);

            ok = mbar_wait_cluster(&acc_full[as], aphase, p.timeout_ns, abort_flag) && push_ok;
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
                const int group_row = c.m_abs + static_cast<int>(rank) * BM + q * 32;
                const bool tma_group = SEND == 0 && p.c_tma && group_row + 32 <= c.m_end;
                if (SEND == 0 && p.c_tma) {
                    if (lane == 0)
                        bulk_wait_read_all();
                    __syncwarp();
                }
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
            // this CTA's half of the accumulator is drained: tell the even CTA
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(acc_empty_lead[as]);

            if (SEND != 0) {
                // the send warps hand the tile to the completion warp; a failed wait
                // for a slot is voted on at the next tile (or reported after the loop)
                push_ok = __all_sync(0xffffffffu, push_ok);
            } else if (p.sink_enabled) {
                named_bar_sync(1, 128);
                if (epi_tid == 0) {
                    if (rec)
                        rec[2] = globaltimer_ns();
                    // each CTA counts its half of every pair tile of the expert
                    const int tiles_e =
                        2 * ((c.m_end - sh->eoff[c.e] + L::kTileRows - 1) / L::kTileRows) *
                        p.n_blocks;
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
        // vote, and one thread hands this CTA's half of the tile to the completion warp.
        const int sw = warp - 7;
        const int send_tid = threadIdx.x - 224;
        uint64_t *trace = send_tid == 0 ? trace_block(p) : nullptr;
        bool ok = true;
        bool push_ok = true;  // send_tid 0: the last hand-off succeeded
        int k = 0;
        int i = 0;
        for (int t = pair; t < total_tiles; t += n_pairs, ++i) {
            const TileCoord c =
                decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, L::kTileRows, p.m_fastest);
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
                    // each CTA counts its half of every pair tile of the expert
                    const int tiles_e =
                        2 * ((c.m_end - sh->eoff[c.e] + L::kTileRows - 1) / L::kTileRows) *
                        p.n_blocks;
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

    // a combine launched behind this kernel may start now: it reads nothing before
    // acquiring the flags (or count words) this kernel releases
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no MMA of the pair is still writing either CTA's TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, L::kTmemCols);
    }
}

template <int SEND>
static cudaError_t launch_pair(const CUtensorMap &ta, const CUtensorMap &tb, const SendParams &p,
                               int max_pairs, cudaStream_t s)
{
    using L = PairLayout<SEND>;
    auto kern = gemm_send_bf16_pair_kernel<SEND>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    // persistent: as many pairs as can be resident at once (clusters are placed
    // within a GPC), and never more than there are pair tiles
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * max_pairs, 1, 1);
    cfg.blockDim = dim3(L::kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = s;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess ||
        active < 1) {
        (void)cudaGetLastError();
        active = max_pairs;
    }
    const int pairs = active < max_pairs ? active : max_pairs;
    return launch_send_kernel(kern, 2 * pairs, L::kThreads, L::kSmemBytes, ta, tb, p, s);
}

cudaError_t launch_gemm_send_bf16_pair(const CUtensorMap &ta, const CUtensorMap &tb,
                                       const SendParams &p, int send_warps, int max_pairs,
                                       cudaStream_t s)
{
    return send_warps == 4 ? launch_pair<4>(ta, tb, p, max_pairs, s)
                           : launch_pair<0>(ta, tb, p, max_pairs, s);
}

}  // namespace ep
