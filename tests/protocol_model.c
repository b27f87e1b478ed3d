/*
 * The completion-signalling protocol on host threads (C11 atomics), for the
 * orderings the kernels rely on. Producer threads stand for the thread blocks: tile t
 * of expert e of rank r writes its share of the expert's rows into every
 * destination's buffer and increments the expert's tile counter with an
 * acquire-release RMW; the one that completes the expert (sees TILES - 1) re-arms
 * the tile counter and then
 *   rank-flag mode ("ep_signal_completion", ep_ord_r with has_rank_flag): the count
 *     words are plain (relaxed) stores made at the start of the call by the thread
 *     standing for block 0 of the rank (tile 0 of expert 0), before its own release;
 *     the completer increments the rank's election counter with an acquire-release
 *     RMW (every expert completion signals every destination, so one counter serves
 *     all of them); the producer that sees E_l - 1 re-arms it, takes a release fence
 *     and stores the rank flag of every destination;
 *     a consumer per destination waits for each source rank's flag, takes an
 *     acquire fence and reads every row and count word of that rank;
 *   per-expert mode: takes a release fence and stores each count word tagged with
 *     the epoch; the consumer acquires each expert's word and reads that expert's rows.
 * Threads sleep for random short spans between steps, so the interleavings vary
 * with the seed. Every wait is bounded; a producer told to fail never signals.
 *
 * usage: protocol_model R E TILES ROWS EPOCHS MODE SEED [FAIL_RANK FAIL_EXPERT]
 *   MODE 0 rank flag, 1 per expert, and two planted mistakes the checks must catch:
 *   2 the rank flag is stored by the first expert to finish instead of the last;
 *   3 block 0 stores the count words after its release instead of before it.
 *   Prints one line:
 *   "epochs N errors X timeouts Y elections Z" (Z = elections over all epochs).
 */
#define _POSIX_C_SOURCE 200809L  /* pthread barriers, clock_gettime */
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

enum { MAX_R = 8, MAX_E = 8, MAX_TILES = 4, MAX_ROWS = 256 };

static int R, E, TILES, ROWS, EPOCHS, MODE, FAIL_R = -1, FAIL_E = -1;
static uint64_t SEED;
static const double TIMEOUT_S = 0.05;

static _Atomic uint64_t payload[MAX_R][MAX_R][MAX_E][MAX_ROWS]; /* [dst][src][e][row] */
static _Atomic uint64_t counts[MAX_R][MAX_E * MAX_R];            /* [dst][e*R + src] */
static _Atomic uint64_t flags[MAX_R][MAX_R];                     /* [dst][src] */
static _Atomic int rank_counter[MAX_R];                          /* [src] */
static _Atomic int tile_counter[MAX_R][MAX_E];                   /* [src][e] */
static atomic_int errors, timeouts, elections;
static pthread_barrier_t epoch_bar;

static uint64_t mix(uint64_t x)
{
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdull;
    x ^= x >> 33;
    x *= 0xc4ceb9fe1a85ec53ull;
    x ^= x >> 33;
    return x;
}

static uint64_t row_value(int ep, int dst, int src, int e, int i)
{
    return ((uint64_t)ep << 40) ^ mix(((uint64_t)dst << 48) ^ ((uint64_t)src << 32) ^ ((uint64_t)e << 16) ^ (uint64_t)i);
}

static double now_s(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec + 1e-9 * ts.tv_nsec;
}

static void jitter(uint64_t *rng)
{
    *rng = mix(*rng + 0x9e3779b97f4a7c15ull);
    for (volatile int k = (int)(*rng % 2000); k > 0; --k) {
    }
}

struct producer {
    int src, e, tile;
};

static void *producer_main(void *arg)
{
    const struct producer *p = arg;
    uint64_t rng = SEED ^ mix((uint64_t)((p->src * MAX_E + p->e) * MAX_TILES + p->tile + 1));
    const int block0 = p->e == 0 && p->tile == 0;  /* stands for block 0 of the rank */
    for (int ep = 1; ep <= EPOCHS; ++ep) {
        pthread_barrier_wait(&epoch_bar);
        if (block0 && (MODE == 0 || MODE == 2)) {  /* every count word, before any release */
            for (int dst = 0; dst < R; ++dst)
                for (int e = 0; e < E; ++e)
                    atomic_store_explicit(&counts[dst][e * R + p->src], (uint64_t)ROWS + (uint64_t)ep,
                                          memory_order_relaxed);
            jitter(&rng);
        }
        for (int dst = 0; dst < R; ++dst) {
            for (int i = p->tile; i < ROWS; i += TILES)
                atomic_store_explicit(&payload[dst][p->src][p->e][i], row_value(ep, dst, p->src, p->e, i),
                                      memory_order_relaxed);
            jitter(&rng);
        }
        const int fail = p->src == FAIL_R && p->e == FAIL_E;
        int completes = 0;
        if (!fail)
            completes = atomic_fetch_add_explicit(&tile_counter[p->src][p->e], 1, memory_order_acq_rel) ==
                        TILES - 1;
        if (completes) {
            atomic_store_explicit(&tile_counter[p->src][p->e], 0, memory_order_relaxed);
            jitter(&rng);
            if (MODE != 1) {
                const int last = MODE == 2 ? 0 : E - 1;
                const int old = atomic_fetch_add_explicit(&rank_counter[p->src], 1, memory_order_acq_rel);
                if (old == E - 1)  /* the last increment re-arms the counter */
                    atomic_store_explicit(&rank_counter[p->src], 0, memory_order_relaxed);
                if (old == last) {
                    atomic_thread_fence(memory_order_release);
                    for (int dst = 0; dst < R; ++dst) {
                        atomic_fetch_add(&elections, 1);
                        atomic_store_explicit(&flags[dst][p->src], (uint64_t)ep, memory_order_relaxed);
                    }
                }
            } else {
                atomic_thread_fence(memory_order_release);
                for (int dst = 0; dst < R; ++dst)
                    atomic_store_explicit(&counts[dst][p->e * R + p->src],
                                          ((uint64_t)ep << 32) | (uint64_t)ROWS, memory_order_relaxed);
            }
        }
        if (block0 && MODE == 3) {  /* planted: the count words after this block's release */
            jitter(&rng);
            jitter(&rng);
            for (int dst = 0; dst < R; ++dst)
                for (int e = 0; e < E; ++e)
                    atomic_store_explicit(&counts[dst][e * R + p->src], (uint64_t)ROWS + (uint64_t)ep,
                                          memory_order_relaxed);
        }
        pthread_barrier_wait(&epoch_bar); /* every consumer has finished the epoch */
    }
    return NULL;
}

static int check_rows(int ep, int dst, int src, int e)
{
    int bad = 0;
    for (int i = 0; i < ROWS; ++i)
        bad |= atomic_load_explicit(&payload[dst][src][e][i], memory_order_relaxed) !=
               row_value(ep, dst, src, e, i);
    return bad;
}

static void *consumer_main(void *arg)
{
    const int dst = (int)(intptr_t)arg;
    for (int ep = 1; ep <= EPOCHS; ++ep) {
        pthread_barrier_wait(&epoch_bar);
        const double t0 = now_s();
        for (int src = 0; src < R; ++src) {
            if (MODE != 1) {
                int ok = 1;
                while (atomic_load_explicit(&flags[dst][src], memory_order_relaxed) != (uint64_t)ep) {
                    if (now_s() - t0 > TIMEOUT_S) {
                        ok = 0;
                        break;
                    }
                }
                if (!ok) {
                    atomic_fetch_add(&timeouts, 1);
                    continue;
                }
                atomic_thread_fence(memory_order_acquire);
                int bad = 0;
                for (int e = 0; e < E; ++e) {
                    bad |= atomic_load_explicit(&counts[dst][e * R + src], memory_order_relaxed) !=
                           (uint64_t)ROWS + (uint64_t)ep;
                    bad |= check_rows(ep, dst, src, e);
                }
                if (bad)
                    atomic_fetch_add(&errors, 1);
            } else {
                for (int e = 0; e < E; ++e) {
                    int ok = 1;
                    while (atomic_load_explicit(&counts[dst][e * R + src], memory_order_acquire) >> 32 !=
                           (uint64_t)ep) {
                        if (now_s() - t0 > TIMEOUT_S) {
                            ok = 0;
                            break;
                        }
                    }
                    if (!ok) {
                        atomic_fetch_add(&timeouts, 1);
                        continue;
                    }
                    if (check_rows(ep, dst, src, e))
                        atomic_fetch_add(&errors, 1);
                }
            }
        }
        pthread_barrier_wait(&epoch_bar);
    }
    return NULL;
}

int main(int argc, char **argv)
{
    if (argc < 8)
        return 2;
    R = atoi(argv[1]);
    E = atoi(argv[2]);
    TILES = atoi(argv[3]);
    ROWS = atoi(argv[4]);
    EPOCHS = atoi(argv[5]);
    MODE = atoi(argv[6]);
    SEED = strtoull(argv[7], NULL, 10);
    if (argc >= 10) {
        FAIL_R = atoi(argv[8]);
        FAIL_E = atoi(argv[9]);
    }
    if (R < 1 || R > MAX_R || E < 1 || E > MAX_E || TILES < 1 || TILES > MAX_TILES || ROWS < TILES ||
        ROWS > MAX_ROWS || EPOCHS < 1)
        return 2;
    const int n_prod = R * E * TILES;
    pthread_barrier_init(&epoch_bar, NULL, (unsigned)(n_prod + R));
    pthread_t th[MAX_R * MAX_E * MAX_TILES + MAX_R];
    static struct producer ps[MAX_R * MAX_E * MAX_TILES];
    for (int i = 0; i < n_prod; ++i) {
        ps[i].src = i / (E * TILES);
        ps[i].e = (i / TILES) % E;
        ps[i].tile = i % TILES;
        pthread_create(&th[i], NULL, producer_main, &ps[i]);
    }
    for (int d = 0; d < R; ++d)
        pthread_create(&th[n_prod + d], NULL, consumer_main, (void *)(intptr_t)d);
    for (int i = 0; i < n_prod + R; ++i)
        pthread_join(th[i], NULL);
    printf("epochs %d errors %d timeouts %d elections %d\n", EPOCHS, atomic_load(&errors),
           atomic_load(&timeouts), atomic_load(&elections));
    return 0;
}
