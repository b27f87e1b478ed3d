// Grouped expert GEMM with blockwise fp8 operands (the "blockwise_fp8_1d2d"
// family named in the "P3PeerSendConfig" description: 1x128 activation scales,
// 128x128 weight scales), with the same fused EP-combine send as the bf16 kernel.
//
// y[m, n] = sum_kb sa[m, kb] * sw[e, n/128, kb] * sum_{k in kb} a8[m, k] * w8[n, k]
//
// The scales are arbitrary fp32 values, so they cannot ride on the tensor cores'
// power-of-two block scaling: every 128-wide K block is its own fp32 partial sum
// on the tensor cores, and warps outside the MMA path scale and accumulate the
// partials ("promotion") in registers.
//
// Design for sm_103a, one persistent CTA per SM, 352 threads, column tile BN = 256
// (128 where N is not a multiple of 256). The kernel stays on single CTAs: with two
// partial buffers the MMA -> promotion -> MMA hand-off is on the critical path of
// every K block, and across a CTA pair that round trip doubles.
//  warp 0     TMA: A box 128 (K bytes) x 128 rows, W box 128 x BN, 128-byte swizzle;
//             one stage is exactly one scale block (3 stages; 5 for BN 128: the
//             shared memory left holds the output tile).
//  warp 1     TMEM (512 columns = 512/BN fp32 partial buffers of 128 x BN) and the MMA:
//             tcgen05.mma kind::f8f6f4, e4m3 x e4m3, M 128, N BN, K 32 per instruction;
//             one partial per K block, buffers in rotation.
//  warp 2     completion counting + signalling (shared with the bf16 kernel).
//  warps 3-10 promotion + epilogue: warp w reads TMEM lane quarter w % 4 and column
//             half (w - 3) / 4; each thread keeps its row's BN/2 fp32 accumulators
//             (as pairs, updated with paired FMAs), adds sa[m, kb] * sw[e, n/128, kb] *
//             partial per K block, then rounds to bf16 into a shared-memory tile
//             buffer; once both halves of the tile's rows are staged, the thread of
//             each row's first half sends the whole row (BN columns, contiguous at the
//             destination) with one bulk copy. The copies run on the TMA engine while
//             the warps promote the next tile; a tile goes to the completion warp once
//             its copies have completed (at the next tile's epilogue, or after the last
//             tile), so the rows it signals are written.
#include <cuda_bf16.h>

#include "ep_internal.h"
#include "ep_ptx.cuh"
#include "ep_sink.cuh"

namespace ep {

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Tile number i of this block (expert e), whose rows have all been written, goes to
// the completion warp.
__device__ __forceinline__ bool push_written_tile(const SendParams &p, SinkShared *sh,
                                                  uint64_t *trace, int e, int i)
{
    const int rec = (trace && i < p.trace_records) ? i : -1;
    if (rec >= 0)
        trace[2 + 4 * rec + 2] = globaltimer_ns();
    const int tiles_e = (sh->eoff[e + 1] - sh->eoff[e] + BM - 1) / BM * p.n_blocks;
    return push_tile_done(p, sh, e, rec, tiles_e);
}

template <int BN_>
struct Fp8Layout {
    static constexpr int BN = BN_;
    static constexpr int STAGES = BN == 128 ? 5 : 3;
    static constexpr int kBufs = 512 / BN;    // fp32 partial buffers that fit in TMEM
    static constexpr int kHalfCols = BN / 2;  // columns per promotion warp
    static constexpr int kABytes = BM * kRowBytesK;  // 128 rows x 128 e4m3
    static constexpr int kBBytes = BN * kRowBytesK;  // BN rows x 128 e4m3
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kPromoWarps = 8;
    static constexpr int kTilePitch = BN * 2 + 16;  // a bf16 output row + 16 bytes: rows
                                                     // of a warp's stores hit all banks
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffTile = kOffB + STAGES * kBBytes;
    static constexpr int kOffBars = kOffTile + BM * kTilePitch;
    static constexpr int kNumBars = 2 * STAGES + 2 * kBufs + 1;  // full, empty, pfull, pfree, done
    static constexpr int kOffSink = (kOffBars + kNumBars * 8 + 15) / 16 * 16;
    static constexpr int kEnd = kOffSink + static_cast<int>(sizeof(SinkShared));
    static constexpr int kSmemBytes = kEnd + 1024;
    static constexpr uint32_t kTmemCols = kBufs * BN;  // all 512 columns
    static_assert(kBufs * BN == 512, "the partial buffers fill the allocation");
    static constexpr int kThreads = 32 * (3 + kPromoWarps);
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// The per-K-block hand-offs (stages, partial buffers) spin on test_wait instead of
// suspending in try_wait: their round trip is on the critical path of every K block.
__device__ __forceinline__ bool fp8_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns,
                                         volatile int *abort)
{
    return mbar_spin<false>(bar, parity, timeout_ns, abort);
}

template <int BN_>
__global__ void __launch_bounds__(352, 1)
    gemm_send_fp8_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ SendParams p)
{
    using L = Fp8Layout<BN_>;
    constexpr int BN = L::BN;
    constexpr int STAGES = L::STAGES;
    constexpr int NBUF = L::kBufs;
    constexpr int HC = L::kHalfCols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBars);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *pfull = bars + 2 * STAGES;
    uint64_t *pfree = pfull + NBUF;
    uint64_t *mma_done = pfree + NBUF;
    SinkShared *sh = reinterpret_cast<SinkShared *>(smem + L::kOffSink);
    volatile int *abort_flag = &sh->abort_flag;
    const int El = p.El;
    const int nkb = p.num_k_blocks;  // K / 128: one scale block per K block

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pfree[b], L::kPromoWarps);
        }
        mbar_init(mma_done, 1);
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
                const TileCoord c =
                    decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, BM, p.m_fastest);
                const int w_row = c.e * p.N + c.nb * BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!fp8_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
                    tma_load_2d(smem + L::kOffA + stage * L::kABytes, &tmap_a, &full[stage],
                                kb * 128, c.m_abs);
                    tma_load_2d(smem + L::kOffB + stage * L::kBBytes, &tmap_b, &full[stage],
                                kb * 128, w_row);
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
                    fp8_wait(&full[s], (last_parity >> s) & 1u, p.timeout_ns, &no_abort);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(0u, BM, BN);  // e4m3 x e4m3 -> fp32
            int stage = 0;
            uint32_t phase = 0;
            uint32_t g = 0;  // K blocks issued so far (selects the partial buffer)
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t pb = g % NBUF, pph = (g / NBUF) & 1u;
                    if (!fp8_wait(&pfree[pb], pph ^ 1u, p.timeout_ns, abort_flag) ||
                        !fp8_wait(&full[stage], phase, p.timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + L::kOffA + stage * L::kABytes);
                    const uint32_t b_addr = smem_u32(smem + L::kOffB + stage * L::kBBytes);
                    const uint32_t d_tmem = tmem_base + pb * BN;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f8(d_tmem, desc_kmajor_sw128(a_addr + kk * 32),
                               desc_kmajor_sw128(b_addr + kk * 32), idesc, kk != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    mma_commit(&pfull[pb]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                raise_abort(p.status, abort_flag);
            mma_commit(mma_done);
            volatile int no_abort = 0;
            fp8_wait(mma_done, 0, p.timeout_ns, &no_abort);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------- completion counting + signalling
        if (lane == 0 && p.sink_enabled)
            completion_loop(p, sh);
        __syncwarp();
    } else {
        // --------------------------------------------- promotion + epilogue + sink
        const int q = warp & 3;            // TMEM lane quarter
        const int half = (warp - 3) >> 2;  // column half of the tile
        const int ptid = threadIdx.x - 96;  // 0..255
        // this thread's row of the tile buffer (its HC columns)
        const uint32_t trow = smem_u32(smem + L::kOffTile) + (q * 32 + lane) * L::kTilePitch +
                              half * HC * 2;
        int pend_e = -1;  // expert of the previous tile, whose copies may be in flight
        const int row = q * 32 + lane;
        const int n_scale_blocks = p.N / 128;
        uint64_t *trace = ptid == 0 ? trace_block(p) : nullptr;
        if (trace)
            trace[1] = globaltimer_ns();

        bool ok = true;
        bool push_ok = true;
        uint32_t g = 0;
        int i = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++i) {
            const TileCoord c =
                decode_tile(t, sh->tile_start, sh->eoff, El, p.n_blocks, BM, p.m_fastest);
            const int m = c.m_abs + row;
            uint8_t *row_base = resolve_row(p, sh, c, m);
            // scale rows (rows past the tile's group read the last row's scales: unused)
            const int m_s = m < p.max_rows ? m : static_cast<int>(p.max_rows) - 1;
            const float *sa = p.a_scales + static_cast<int64_t>(m_s) * nkb;
            const float *sw = p.w_scales +
                              (static_cast<int64_t>(c.e) * n_scale_blocks +
                               (c.nb * BN + half * HC) / 128) * nkb;
            // HC fp32 accumulators of this thread's row, as pairs
            uint64_t acc[HC / 2];
#pragma unroll
            for (int j = 0; j < HC / 2; ++j)
                acc[j] = 0ull;
            float sa_next = __ldg(sa), sw_next = __ldg(sw);
            bool ok_t = push_ok;
            for (int kb = 0; kb < nkb && ok_t; ++kb, ++g) {
                const float s = sa_next * sw_next;
                const uint64_t s2 = pack_f32x2(__float_as_uint(s), __float_as_uint(s));
                if (kb + 1 < nkb) {
                    sa_next = __ldg(sa + kb + 1);
                    sw_next = __ldg(sw + kb + 1);
                }
                const uint32_t pb = g % NBUF, pph = (g / NBUF) & 1u;
                ok_t = fp8_wait(&pfull[pb], pph, p.timeout_ns, abort_flag);
                ok_t = __all_sync(0xffffffffu, ok_t);
                if (!ok_t)
                    break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       pb * BN + half * HC;
                // HC/16 groups of 16 columns; the load of group j+1 is in flight while
                // group j is scaled and added
                constexpr int NG = HC / 16;
                uint32_t buf0[16], buf1[16];
                tmem_ld_32x32b_x16(taddr, buf0);
                tmem_ld_wait();
                tmem_regs_ready(buf0);
#pragma unroll
                for (int j = 0; j < NG; ++j) {
                    uint32_t(&cur)[16] = (j & 1) ? buf1 : buf0;
                    uint32_t(&nxt)[16] = (j & 1) ? buf0 : buf1;
                    if (j + 1 < NG)
                        tmem_ld_32x32b_x16(taddr + (j + 1) * 16, nxt);
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        acc[j * 8 + h] = fma_f32x2(pack_f32x2(cur[2 * h], cur[2 * h + 1]), s2,
                                                   acc[j * 8 + h]);
                    if (j + 1 < NG) {
                        tmem_ld_wait();
                        tmem_regs_ready(nxt);
                    }
                }
                // partial read: hand the buffer back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&pfree[pb]);
            }
            ok = named_bar_and(2, 256, ok_t);
            if (!ok)
                break;
            uint64_t *rec = (trace && i < p.trace_records) ? trace + 2 + 4 * i : nullptr;
            if (rec) {
                rec[0] = static_cast<uint64_t>(t) | (static_cast<uint64_t>(c.e) << 32);
                rec[1] = globaltimer_ns();
            }

            // the previous tile's copies have read the buffer and written their rows:
            // hand that tile to the completion warp
            bulk_wait_all();
            fence_proxy_async_global();
            named_bar_sync(1, 256);
            if (ptid == 0 && pend_e >= 0 && p.sink_enabled)
                push_ok = push_written_tile(p, sh, trace, pend_e, i - 1) && push_ok;
            // this thread's half row in bf16 into the buffer
#pragma unroll
            for (int ch = 0; ch < HC / 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint64_t a2 = acc[ch * 4 + h];
                    __nv_bfloat162 b = __float22bfloat162_rn(
                        make_float2(__uint_as_float(static_cast<uint32_t>(a2)),
                                    __uint_as_float(static_cast<uint32_t>(a2 >> 32))));
                    w[h] = *reinterpret_cast<uint32_t *>(&b);
                }
                st_shared_v4(trow + ch * 16, make_uint4(w[0], w[1], w[2], w[3]));
            }
            fence_proxy_async_shared();
            // both halves of every row are staged: one copy per row (its BN columns are
            // contiguous at the destination), issued by the thread of its first half
            named_bar_sync(1, 256);
            if (half == 0 && row_base != nullptr)
                bulk_store(row_base + c.nb * BN * 2, trow, BN * 2);
            bulk_commit();
            pend_e = c.e;
            if (!p.sink_enabled && rec)
                rec[2] = rec[3] = globaltimer_ns();
        }
        // the last tile's copies
        bulk_wait_all();
        fence_proxy_async_global();
        named_bar_sync(1, 256);
        if (ptid == 0 && pend_e >= 0 && p.sink_enabled && ok)
            push_ok = push_written_tile(p, sh, trace, pend_e, i - 1) && push_ok;
        if (ptid == 0) {
            if (trace)
                trace[0] = static_cast<uint64_t>(i);
            close_queue(sh);
            if (!push_ok)
                raise_abort(p.status, abort_flag);
        }
        if (!ok && lane == 0)
            raise_abort(p.status, abort_flag);
    }

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

template <int BN>
static cudaError_t launch_fp8_bn(const CUtensorMap &ta, const CUtensorMap &tb,
                                 const SendParams &p, int grid, cudaStream_t s)
{
    using L = Fp8Layout<BN>;
    auto kern = gemm_send_fp8_kernel<BN>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    return launch_send_kernel(kern, grid, L::kThreads, L::kSmemBytes, ta, tb, p, s);
}

cudaError_t launch_gemm_send_fp8(const CUtensorMap &ta, const CUtensorMap &tb,
                                 const SendParams &p, int bn, int grid, cudaStream_t s)
{
    switch (bn) {
    case 256:
        return launch_fp8_bn<256>(ta, tb, p, grid, s);
    case 128:
        return launch_fp8_bn<128>(ta, tb, p, grid, s);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace ep
