/*
 * Oracle for the fused MoE expert GEMM + EP-combine path -- TEST INFRASTRUCTURE.
 *
 * A plain, slow, obviously correct CPU restatement of what the path computes,
 * written from these pages:
 *   [P1] "EpiloguePeerSink" (Modular MAX Mojo API, linalg/matmul/gpu/sm100_structured/
 *        structured_kernels/output_writer): send_tile takes the finished output tile
 *        instead of the local store; rows m_abs <= m < m_end of the tile's group.
 *   [P2] "P3PeerSendConfig" (same directory), description: the two row-major
 *        linear-index formulas recv_count_layout((e, rk)) and
 *        recv_buf_layout((src_idx, src_topk, byte_off)); fields src_info_ptr,
 *        recv_buf_ptrs[8], n_ranks, top_k, msg_bytes, max_tokens_per_rank.
 *   [P3] "ep_signal_completion" (Modular MAX Mojo API, shmem/ep_comm): plain per-expert
 *        count stores, an acquire-release election on a per-destination counter
 *        bounded by the local expert count, and one release of a rank flag kept in
 *        the tail of the receive-count buffer.
 * The gate-weighted combine (the consumer the P2 description calls EPCombineKernel)
 * is the plain sum over a token's top_k received rows, each scaled by its gate.
 *
 * Only the test suite, the package entry's smoke check and the benchmark's CPU
 * baseline load this library. The product path never does. It shares no code
 * with the CUDA path: no header, helper, table or constant.
 *
 * Arithmetic: double accumulation, bf16 round-to-nearest-even at the received
 * row and at the combined output, e4m3 decoded from its bit definition.
 * Loops only; threads split independent rows and nothing else.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* bf16 bit pattern -> value: the high half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* value -> bf16, rounded once, to nearest, ties to even (8 significant bits,
 * exponent range of binary32, subnormals down to 2^-133, overflow to infinity). */
uint16_t orc_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    frexp(a, &e);           /* a = f * 2^e with 0.5 <= f < 1: leading bit has weight 2^(e-1) */
    int q = e - 1 - 7;      /* weight of the last of the 7 kept fraction bits */
    if (q < -133)
        q = -133;           /* subnormal spacing 2^-126 * 2^-7 */
    double r = nearbyint(ldexp(a, -q));  /* default rounding mode: nearest, ties to even */
    double v = ldexp(r, q);
    if (v >= 0x1p128)
        return sign | 0x7F80;
    float f = (float)v;     /* exact: at most 8 significant bits, within binary32 range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* OCP 8-bit E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * subnormals at exponent 0, S.1111.111 is NaN, no infinities. */
double orc_e4m3_to_double(uint8_t b)
{
    int s = b >> 7, E = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);          /* (m/8) * 2^-6 */
    else
        v = ldexp(8.0 + (double)m, E - 10); /* (1 + m/8) * 2^(E-7) */
    return s ? -v : v;
}

void orc_bf16_to_double_n(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_to_double(h[i]);
}

void orc_bf16_from_double_n(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_from_double(x[i]);
}

void orc_e4m3_to_double_n(const uint8_t *b, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_to_double(b[i]);
}

/* ---------------------------------------------------------- index formulas */

/* [P2] recv_count_layout((e, rk)) = e*n_ranks + rk */
int64_t orc_recv_count_index(int64_t e, int64_t rk, int64_t n_ranks)
{
    return e * n_ranks + rk;
}

/* [P2] recv_buf_layout((src_idx, src_topk, byte_off)) = (src_idx*top_k + src_topk)*msg_bytes + byte_off */
int64_t orc_recv_buf_offset(int64_t src_idx, int64_t src_topk, int64_t byte_off,
                            int64_t top_k, int64_t msg_bytes)
{
    return (src_idx * top_k + src_topk) * msg_bytes + byte_off;
}

/* -------------------------------------------------------------------- plan */

/*
 * Rows that one producer rank receives, in the receiving layout's order.
 * Expert g lives on rank g / El at local slot g % El. Within local expert e the
 * rows are ordered by source rank, then token index, then top-k slot.
 * Outputs:
 *   expert_offsets[El+1]   first row of each local expert
 *   src_info[rows][2]      (src_idx, src_topk) of each row (the P2 src_info_ptr)
 *   seg_offsets[El][R+1]   first row of each (expert, source rank) segment
 *   send_counts[El][R]     rows of expert e that came from (and go back to) rank rk
 *   gather_idx[rows]       flat index (rk*T + t)*k + j of the row's routing entry
 *   m_total                row count
 * Returns 0, -1 when the rows exceed max_rows, -2 for an expert id out of range.
 */
int orc_plan(int R, int El, int T, int k, int rank, const int32_t *topk_ids, int64_t max_rows,
             int32_t *expert_offsets, int32_t *src_info, int32_t *seg_offsets,
             int32_t *send_counts, int32_t *gather_idx, int32_t *m_total)
{
    int64_t n_entries = (int64_t)R * T * k;
    for (int64_t i = 0; i < n_entries; i++)
        if (topk_ids[i] < 0 || topk_ids[i] >= R * El)
            return -2;
    int64_t row = 0;
    for (int e = 0; e < El; e++) {
        int g = rank * El + e;
        expert_offsets[e] = (int32_t)row;
        for (int rk = 0; rk < R; rk++) {
            seg_offsets[e * (R + 1) + rk] = (int32_t)row;
            int64_t count = 0;
            for (int t = 0; t < T; t++) {
                for (int j = 0; j < k; j++) {
                    int64_t flat = ((int64_t)rk * T + t) * k + j;
                    if (topk_ids[flat] != g)
                        continue;
                    if (row >= max_rows)
                        return -1;
                    src_info[2 * row + 0] = t;
                    src_info[2 * row + 1] = j;
                    gather_idx[row] = (int32_t)flat;
                    row++;
                    count++;
                }
            }
            send_counts[e * R + rk] = (int32_t)count;
        }
        seg_offsets[e * (R + 1) + R] = (int32_t)row;
    }
    expert_offsets[El] = (int32_t)row;
    *m_total = (int32_t)row;
    return 0;
}

/* ------------------------------------------------------------- expert rows */

enum { ORC_BF16 = 0, ORC_FP8_1D2D = 1 };

typedef struct {
    int dtype;
    const void *A;
    const float *sa;
    const void *W;
    const float *sw;
    const int32_t *expert_offsets;
    int El, K, N;
    const int64_t *rows;
    int64_t n_rows;
    uint16_t *Y;   /* bf16 rows, or NULL */
    double *Yd;    /* unrounded rows, or NULL */
    int64_t lo, hi;
    int status;
} rows_job;

static int expert_of_row(const int32_t *expert_offsets, int El, int64_t m)
{
    for (int e = 0; e < El; e++)
        if (m >= expert_offsets[e] && m < expert_offsets[e + 1])
            return e;
    return -1;
}

static double operand_a(const rows_job *j, int64_t m, int kk)
{
    if (j->dtype == ORC_BF16)
        return orc_bf16_to_double(((const uint16_t *)j->A)[m * j->K + kk]);
    /* blockwise fp8, 1x128 activation scales: value = e4m3 * sa[m][kk/128] */
    return orc_e4m3_to_double(((const uint8_t *)j->A)[m * j->K + kk]) *
           (double)j->sa[m * (j->K / 128) + kk / 128];
}

static double operand_w(const rows_job *j, int e, int n, int kk)
{
    int64_t idx = ((int64_t)e * j->N + n) * j->K + kk;
    if (j->dtype == ORC_BF16)
        return orc_bf16_to_double(((const uint16_t *)j->W)[idx]);
    /* blockwise fp8, 128x128 weight scales: value = e4m3 * sw[e][n/128][kk/128] */
    int64_t s = ((int64_t)e * (j->N / 128) + n / 128) * (j->K / 128) + kk / 128;
    return orc_e4m3_to_double(((const uint8_t *)j->W)[idx]) * (double)j->sw[s];
}

static void *rows_worker(void *arg)
{
    rows_job *j = (rows_job *)arg;
    double *a = (double *)malloc(sizeof(double) * (size_t)j->K);
    if (!a) {
        j->status = -3;
        return NULL;
    }
    for (int64_t r = j->lo; r < j->hi; r++) {
        int64_t m = j->rows[r];
        int e = expert_of_row(j->expert_offsets, j->El, m);
        if (e < 0) {
            j->status = -1;
            continue;
        }
        for (int kk = 0; kk < j->K; kk++)
            a[kk] = operand_a(j, m, kk);
        for (int n = 0; n < j->N; n++) {
            /* Y_e[m, n] = sum_k A[m, k] * W_e[n, k] */
            double acc = 0.0;
            for (int kk = 0; kk < j->K; kk++)
                acc += a[kk] * operand_w(j, e, n, kk);
            if (j->Y)
                j->Y[r * j->N + n] = orc_bf16_from_double(acc);
            if (j->Yd)
                j->Yd[r * j->N + n] = acc;
        }
    }
    free(a);
    return NULL;
}

/*
 * Down-projection rows of one producer rank: for every requested absolute row m
 * of expert e (expert_offsets[e] <= m < expert_offsets[e+1]),
 * Y[r][n] = bf16(sum_k A[m][k] * W[e][n][k]), r the position of m in `rows`;
 * Yd (if not NULL) receives the same sums unrounded.
 * Returns 0, or -1 if a row lies in no expert.
 */
int orc_expert_rows2(int dtype, const void *A, const float *a_scales, const void *W,
                     const float *w_scales, const int32_t *expert_offsets, int El, int K, int N,
                     const int64_t *rows, int64_t n_rows, uint16_t *Y, double *Yd, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n_rows)
        nthreads = (int)(n_rows > 0 ? n_rows : 1);
    rows_job *jobs = (rows_job *)calloc((size_t)nthreads, sizeof(rows_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -3;
    }
    for (int i = 0; i < nthreads; i++) {
        rows_job *j = &jobs[i];
        j->dtype = dtype; j->A = A; j->sa = a_scales; j->W = W; j->sw = w_scales;
        j->expert_offsets = expert_offsets; j->El = El; j->K = K; j->N = N;
        j->rows = rows; j->n_rows = n_rows; j->Y = Y; j->Yd = Yd;
        j->lo = n_rows * i / nthreads;
        j->hi = n_rows * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, rows_worker, j);
    }
    int status = 0;
    for (int i = 0; i < nthreads; i++) {
        pthread_join(th[i], NULL);
        if (jobs[i].status)
            status = jobs[i].status;
    }
    free(jobs);
    free(th);
    return status;
}

int orc_expert_rows(int dtype, const void *A, const float *a_scales, const void *W,
                    const float *w_scales, const int32_t *expert_offsets, int El, int K, int N,
                    const int64_t *rows, int64_t n_rows, uint16_t *Y, int nthreads)
{
    return orc_expert_rows2(dtype, A, a_scales, W, w_scales, expert_offsets, El, K, N, rows,
                            n_rows, Y, NULL, nthreads);
}

/* ----------------------------------------------------------------- scatter */

/*
 * [P1] send_tile / [P2] recv_buf_layout: every computed row m of local expert e
 * goes to the receive buffer of the rank that owns its token (the source rank of
 * its segment), at byte (src_idx*top_k + src_topk)*msg_bytes + 2*n for column n.
 * hits[dst][src_idx*top_k + src_topk] counts the writes of each slot, so a caller
 * can check that every (token, slot) is written exactly once.
 * Returns the number of rows whose destination falls outside the receive buffer
 * (those rows are skipped).
 */
int64_t orc_scatter(const uint16_t *Y, const int64_t *rows, int64_t n_rows, int N,
                    const int32_t *expert_offsets, const int32_t *src_info,
                    const int32_t *seg_offsets, int El, int R, int top_k, int64_t msg_bytes,
                    int64_t max_tokens, uint8_t **recv_bufs, int32_t *hits)
{
    int64_t bad = 0;
    int64_t slots = max_tokens * top_k;
    for (int64_t r = 0; r < n_rows; r++) {
        int64_t m = rows[r];
        int e = expert_of_row(expert_offsets, El, m);
        int dst = -1;
        for (int rk = 0; e >= 0 && rk < R; rk++)
            if (m >= seg_offsets[e * (R + 1) + rk] && m < seg_offsets[e * (R + 1) + rk + 1])
                dst = rk;
        int64_t src_idx = src_info[2 * m + 0];
        int64_t src_topk = src_info[2 * m + 1];
        if (dst < 0 || src_idx < 0 || src_idx >= max_tokens || src_topk < 0 ||
            src_topk >= top_k || 2 * (int64_t)N > msg_bytes) {
            bad++;
            continue;
        }
        hits[(int64_t)dst * slots + src_idx * top_k + src_topk] += 1;
        for (int n = 0; n < N; n++) {
            int64_t off = orc_recv_buf_offset(src_idx, src_topk, 2 * (int64_t)n, top_k, msg_bytes);
            uint16_t v = Y[r * N + n];
            recv_bufs[dst][off + 0] = (uint8_t)(v & 0xFF);  /* little-endian bf16 */
            recv_bufs[dst][off + 1] = (uint8_t)(v >> 8);
        }
    }
    return bad;
}

/* -------------------------------------------------------------- signalling */

/*
 * [P3] Completion signalling of one producer rank, as one sequential history in
 * which the rank's experts complete in slot order. For each expert e and every
 * destination dst:
 *   1. plain store recv_counts[dst][e*R + rank] = send_counts[e][dst]  (P2 recv_count_layout)
 *   2. election: old = rank_counter[dst]++  (the acquire-release counter)
 *   3. the producer that sees old == El-1 stores recv_counts[dst][El*R + rank] = epoch
 *      (the dedicated rank flag in the tail of the receive-count buffer).
 * Each event is logged as (kind 0 = count / 1 = flag, expert, dst, old counter).
 * Returns the number of logged events.
 */
int orc_signal(int R, int El, int rank, const int32_t *send_counts, uint64_t epoch,
               uint64_t **recv_counts, int32_t *rank_counter, int32_t *log)
{
    int n = 0;
    for (int e = 0; e < El; e++) {
        for (int dst = 0; dst < R; dst++) {
            recv_counts[dst][orc_recv_count_index(e, rank, R)] =
                (uint64_t)send_counts[e * R + dst];
            int old = rank_counter[dst]++;
            log[4 * n + 0] = 0; log[4 * n + 1] = e; log[4 * n + 2] = dst; log[4 * n + 3] = old;
            n++;
            if (old == El - 1) {
                recv_counts[dst][(int64_t)El * R + rank] = epoch;
                log[4 * n + 0] = 1; log[4 * n + 1] = e; log[4 * n + 2] = dst; log[4 * n + 3] = old;
                n++;
            }
        }
    }
    return n;
}

/* ----------------------------------------------------------------- combine */

typedef struct {
    const uint8_t *recv;
    const float *gates;
    int k, N;
    int64_t msg_bytes;
    const int64_t *tokens;
    uint16_t *out;
    int64_t lo, hi;
} combine_job;

static void *combine_worker(void *arg)
{
    combine_job *j = (combine_job *)arg;
    for (int64_t r = j->lo; r < j->hi; r++) {
        int64_t t = j->tokens[r];
        for (int n = 0; n < j->N; n++) {
            /* out[t, n] = sum_j g[t, j] * recv[t, j, n], slots in order */
            double acc = 0.0;
            for (int s = 0; s < j->k; s++) {
                int64_t off = orc_recv_buf_offset(t, s, 2 * (int64_t)n, j->k, j->msg_bytes);
                uint16_t v = (uint16_t)(j->recv[off] | ((uint16_t)j->recv[off + 1] << 8));
                acc += (double)j->gates[t * j->k + s] * orc_bf16_to_double(v);
            }
            j->out[r * j->N + n] = orc_bf16_from_double(acc);
        }
    }
    return NULL;
}

/* The exact gate-weighted sum of exact rows: out[t][n] = sum_j g[t][j] * rows[t][j][n],
 * no rounding anywhere (the value the rounded path approximates). */
void orc_combine_exact(const double *rows, const float *gates, int top_k, int N, int64_t n_tokens,
                       double *out)
{
    for (int64_t t = 0; t < n_tokens; t++)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int s = 0; s < top_k; s++)
                acc += (double)gates[t * top_k + s] * rows[(t * top_k + s) * (int64_t)N + n];
            out[t * N + n] = acc;
        }
}

/* Gate-weighted combine of the requested tokens of one destination rank. */
void orc_combine(const uint8_t *recv, const float *gates, int top_k, int N, int64_t msg_bytes,
                 const int64_t *tokens, int64_t n_tokens, uint16_t *out, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > n_tokens)
        nthreads = (int)(n_tokens > 0 ? n_tokens : 1);
    combine_job *jobs = (combine_job *)calloc((size_t)nthreads, sizeof(combine_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return;
    }
    for (int i = 0; i < nthreads; i++) {
        combine_job *j = &jobs[i];
        j->recv = recv; j->gates = gates; j->k = top_k; j->N = N; j->msg_bytes = msg_bytes;
        j->tokens = tokens; j->out = out;
        j->lo = n_tokens * i / nthreads;
        j->hi = n_tokens * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, combine_worker, j);
    }
    for (int i = 0; i < nthreads; i++)
        pthread_join(th[i], NULL);
    free(jobs);
    free(th);
}
