/*
 * CPU oracle for the tile-centric AllGather->GEMM and GEMM->ReduceScatter path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load this file's library.  The CUDA
 * path never calls it, links it or shares a line of code with it.
 *
 * Everything here is the plain definition of what the path computes, written
 * out in fp64 so a reader can check it against the pages by eye:
 *
 *   - "Triton-distributed Semantics", section "AllGather and GEMM Overlapping":
 *     the producer gathers every rank's tiles into one buffer and the consumer
 *     multiplies the gathered matrix.  Result: G = concat_r(A_r) along rows,
 *     C = G * B.
 *   - same page, section "GEMM and ReduceScatter Overlapping": per-rank GEMM
 *     partials are reduced and each row block is scattered to its rank.
 *     Result: S = sum_r A_r * B_r, out_j = rows of block j of S.
 *   - "Distributed Architecture Design", section 5.3 (remote addresses of
 *     symm_at): an address in the own slice moves to rank pe's slice by
 *     subtracting the own slice's base and adding rank pe's.
 *   - "Triton-distributed Semantics", section "Threadblock Swizzling": the row
 *     tile index is rotated by rank * tiles_per_pe modulo the tile count.
 *
 * Precision: bf16 inputs are decoded exactly to fp64; every product of two
 * bf16 values is exact in fp64 (8 + 8 significant bits); sums are fp64 and
 * taken in ascending k (and ascending rank for the reduction).  Outputs are
 * rounded once, fp64 -> bf16, round-to-nearest-even.  Build with
 * -ffp-contract=off so no fused multiply-add changes a rounding (it could not
 * here, since each product is exact, but the flag keeps that obvious).
 *
 * No BLAS, no blocking, no reordering of any sum.  Loops over rows may run in
 * parallel (OpenMP); that changes no arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int opw_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bf16 codec                                                                */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper 16 bits of an IEEE binary32; widening is exact. */
double opw_oracle_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round an fp64 value to the nearest bf16, ties to even, in ONE rounding step
 * (not through binary32, which would round twice).
 *
 * bf16 has an 8-bit significand and the binary32 exponent range, so for
 * |x| in [2^e, 2^(e+1)) with e >= -126 the spacing is 2^(e-7); below 2^-126
 * (subnormal range) the spacing is fixed at 2^-133.  Divide by the spacing
 * (exact: a power of two), round to an integer with ties-to-even, multiply
 * back.  Results at or above 2^128 overflow to infinity.  NaN stays NaN
 * (canonical quiet NaN with the input's sign).
 */
uint16_t opw_oracle_f64_to_bf16(double x)
{
    uint64_t bits;
    memcpy(&bits, &x, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 48) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
    const double a = fabs(x);
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);           /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;        /* subnormal: fixed spacing */
    const int q = e - 7;           /* spacing 2^q */
    const double units = nearbyint(ldexp(a, -q));  /* default mode: ties-to-even */
    const double r = ldexp(units, q);
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);

    /* r is exactly representable as bf16, hence as binary32: take its top half. */
    const float rf = (float)r;
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void opw_oracle_bf16_decode_array(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = opw_oracle_bf16_to_f64(in[i]);
}

void opw_oracle_bf16_encode_array(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = opw_oracle_f64_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* symm_at                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * "Distributed Architecture Design", section 5.3: subtract the local heap
 * base to get the symmetric offset, add the target PE's heap base.
 */
uint64_t opw_oracle_symm_at(uint64_t ptr, uint64_t heap_base_self, uint64_t heap_base_pe)
{
    return heap_base_pe + (ptr - heap_base_self);
}

/*
 * In this build all R logical ranks share one allocation: rank r's heap
 * base is heap + rank_off[r].  A symmetric object at offset `off` of every
 * rank's slice therefore lives at heap + rank_off[r] + off on rank r.
 */
static const uint8_t* rank_ptr(const uint8_t* heap, const int64_t* rank_off, int r, int64_t off)
{
    const uint64_t self_base = (uint64_t)(uintptr_t)heap + (uint64_t)rank_off[0];
    const uint64_t local = self_base + (uint64_t)off;
    const uint64_t pe_base = (uint64_t)(uintptr_t)heap + (uint64_t)rank_off[r];
    return (const uint8_t*)(uintptr_t)opw_oracle_symm_at(local, self_base, pe_base);
}

/* ------------------------------------------------------------------------ */
/* AllGather                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * "AllGather and GEMM Overlapping": every rank's shard A_r ([M_r, K] bf16,
 * row-major, at symmetric offset a_off) lands in the gathered buffer G
 * ([R*M_r, K]) at rows r*M_r .. r*M_r+M_r-1.  A bit copy.
 */
void opw_oracle_allgather(const uint8_t* heap, const int64_t* rank_off, int R, int64_t a_off,
                          int64_t M_r, int64_t K, uint16_t* G)
{
    for (int r = 0; r < R; ++r) {
        const uint16_t* A_r = (const uint16_t*)rank_ptr(heap, rank_off, r, a_off);
        memcpy(G + (int64_t)r * M_r * K, A_r, (size_t)(M_r * K) * sizeof(uint16_t));
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * C[i][j] = sum_{k=0..K-1} A[i][k] * B[k][j], fp64, terms added in ascending
 * k.  A is [M, K] (row stride lda), B is [K, N] (row stride ldb), both bf16
 * row-major; C is [M, N] fp64 (row stride ldc).
 *
 * The loop runs k outside j so B is read row by row, but each C[i][j] still
 * receives its K terms one after another in ascending k: the order of every
 * sum is the definition's.
 */
void opw_oracle_gemm_f64(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                         int64_t M, int64_t N, int64_t K, double* C, int64_t ldc)
{
    double* Bd = (double*)malloc((size_t)(K * N) * sizeof(double));
    if (!Bd) return;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) Bd[k * N + j] = opw_oracle_bf16_to_f64(B[k * ldb + j]);

#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * ldc;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = opw_oracle_bf16_to_f64(A[i * lda + k]);
            const double* b = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) c[j] += a * b[j];
        }
    }
    free(Bd);
}

/* One row of the same product, for sampled checks: c[j] = sum_k a[k]*B[k][j]. */
static void gemm_row_f64(const uint16_t* a, const uint16_t* B, int64_t ldb, int64_t N, int64_t K,
                         double* c)
{
    for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double av = opw_oracle_bf16_to_f64(a[k]);
        const uint16_t* b = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) c[j] += av * opw_oracle_bf16_to_f64(b[j]);
    }
}

/* ------------------------------------------------------------------------ */
/* AG-GEMM                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * Form the gathered matrix explicitly, then multiply:
 *   G = concat_r(A_r)  ([R*M_r, K] bf16),  C = G * B  ([R*M_r, N] fp64).
 * The caller rounds C to bf16 with opw_oracle_bf16_encode_array.
 */
void opw_oracle_ag_gemm(const uint8_t* heap, const int64_t* rank_off, int R, int64_t a_off,
                        int64_t M_r, int64_t N, int64_t K, const uint16_t* B,
                        uint16_t* G, double* C)
{
    opw_oracle_allgather(heap, rank_off, R, a_off, M_r, K, G);
    opw_oracle_gemm_f64(G, K, B, N, (int64_t)R * M_r, N, K, C, N);
}

/*
 * Selected rows of the same C, for sizes where the whole product is too slow
 * on the CPU.  Row i of G is row i mod M_r of shard i / M_r.
 */
void opw_oracle_ag_gemm_rows(const uint8_t* heap, const int64_t* rank_off, int R, int64_t a_off,
                             int64_t M_r, int64_t N, int64_t K, const uint16_t* B,
                             int64_t n_rows, const int64_t* rows, double* C_rows)
{
    (void)R;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
        const int64_t i = rows[t];
        const int r = (int)(i / M_r);
        const uint16_t* A_r = (const uint16_t*)rank_ptr(heap, rank_off, r, a_off);
        gemm_row_f64(A_r + (i % M_r) * K, B, N, N, K, C_rows + t * N);
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM-RS                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * "GEMM and ReduceScatter Overlapping": rank r holds A_r ([M, K_r]) and B_r
 * ([K_r, N]) at symmetric offsets a_off / b_off.  The partial products are
 * reduced across ranks and row block j (rows j*M/R .. (j+1)*M/R-1) of the
 * sum is delivered to rank j:
 *
 *   P_r = A_r * B_r           (fp64, ascending k)
 *   S   = P_0 + P_1 + ... + P_{R-1}   (fp64, ascending rank, from S = 0)
 *   out_j = bf16_rne(S[j*M/R : (j+1)*M/R, :])  written at rank j's out_off.
 *
 * S ([M, N] fp64) is returned; the bf16 blocks are written into heap_out,
 * a buffer laid out like the heap (same rank_off table).
 */
void opw_oracle_gemm_rs(const uint8_t* heap, const int64_t* rank_off, int R,
                        int64_t a_off, int64_t b_off, int64_t out_off,
                        int64_t M, int64_t N, int64_t K_r, double* S, uint8_t* heap_out)
{
    double* P = (double*)malloc((size_t)(M * N) * sizeof(double));
    if (!P) return;
    for (int64_t i = 0; i < M * N; ++i) S[i] = 0.0;
    for (int r = 0; r < R; ++r) {
        const uint16_t* A_r = (const uint16_t*)rank_ptr(heap, rank_off, r, a_off);
        const uint16_t* B_r = (const uint16_t*)rank_ptr(heap, rank_off, r, b_off);
        opw_oracle_gemm_f64(A_r, K_r, B_r, N, M, N, K_r, P, N);
        for (int64_t i = 0; i < M * N; ++i) S[i] = S[i] + P[i];
    }
    free(P);

    const int64_t Mb = M / R;
    for (int j = 0; j < R; ++j) {
        uint16_t* out_j = (uint16_t*)(uintptr_t)rank_ptr(heap_out, rank_off, j, out_off);
        opw_oracle_bf16_encode_array(S + (int64_t)j * Mb * N, out_j, Mb * N);
    }
}

/* Selected rows of S (fp64), same definition. */
void opw_oracle_gemm_rs_rows(const uint8_t* heap, const int64_t* rank_off, int R,
                             int64_t a_off, int64_t b_off, int64_t M, int64_t N, int64_t K_r,
                             int64_t n_rows, const int64_t* rows, double* S_rows)
{
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
        const int64_t i = rows[t];
        double* s = S_rows + t * N;
        double* p = (double*)malloc((size_t)N * sizeof(double));
        for (int64_t j = 0; j < N; ++j) s[j] = 0.0;
        for (int r = 0; r < R; ++r) {
            const uint16_t* A_r = (const uint16_t*)rank_ptr(heap, rank_off, r, a_off);
            const uint16_t* B_r = (const uint16_t*)rank_ptr(heap, rank_off, r, b_off);
            gemm_row_f64(A_r + i * K_r, B_r, N, N, K_r, p);
            for (int64_t j = 0; j < N; ++j) s[j] = s[j] + p[j];
        }
        free(p);
    }
}

/*
 * Information-only variant that follows the fp32 reading of the reduction:
 * each partial is rounded to binary32, then the partials are summed in
 * binary32 in ascending rank order.  Not the parity target (the parity
 * target is the fp64 sum rounded once to bf16); used to report how far the
 * fp32 reduction itself moves the result.
 */
void opw_oracle_gemm_rs_rows_f32(const uint8_t* heap, const int64_t* rank_off, int R,
                                 int64_t a_off, int64_t b_off, int64_t M, int64_t N, int64_t K_r,
                                 int64_t n_rows, const int64_t* rows, float* S_rows)
{
    (void)M;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_rows; ++t) {
        const int64_t i = rows[t];
        float* s = S_rows + t * N;
        double* p = (double*)malloc((size_t)N * sizeof(double));
        for (int64_t j = 0; j < N; ++j) s[j] = 0.0f;
        for (int r = 0; r < R; ++r) {
            const uint16_t* A_r = (const uint16_t*)rank_ptr(heap, rank_off, r, a_off);
            const uint16_t* B_r = (const uint16_t*)rank_ptr(heap, rank_off, r, b_off);
            gemm_row_f64(A_r + i * K_r, B_r, N, N, K_r, p);
            for (int64_t j = 0; j < N; ++j) s[j] = s[j] + (float)p[j];
        }
        free(p);
    }
}

/* ------------------------------------------------------------------------ */
/* Signals                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * SET semantics ("Distributed Architecture Design", 2.3 SignalOp: SET sets
 * the signal to the given value): after a launch that publishes every tile
 * with epoch e, every slot holds e.
 */
void opw_oracle_expected_flags(int64_t n_slots, int64_t epoch, int64_t* out)
{
    for (int64_t i = 0; i < n_slots; ++i) out[i] = epoch;
}

/*
 * Batched signals with SignalOp ADD ("Distributed Architecture Design", 2.3:
 * an ADD increments the signal by its operand; "Triton-distributed
 * Semantics", Best Practices 4: tiles that are always consumed together may
 * share one signal).  One counter per row of flag tiles; every launch adds 1
 * for each of the row's T_k k-tiles, starting from 0 after a reset.  After
 * the launches with epochs 1..e every counter holds e * T_k, which is also the
 * value a consumer waits for to know the whole row is in.
 */
void opw_oracle_expected_row_counters(int64_t n_rows, int64_t epoch, int64_t T_k, int64_t* out)
{
    for (int64_t i = 0; i < n_rows; ++i) out[i] = epoch * T_k;
}

/* ------------------------------------------------------------------------ */
/* Consumer schedule (threadblock swizzle)                                   */
/* ------------------------------------------------------------------------ */

/*
 * "Threadblock Swizzling": pid_m = (pid_m + rank * tiles_per_pe) % total_tiles,
 * so that each PE starts on its own rows.  This is that formula.
 */
int64_t opw_oracle_swizzle_row(int64_t pid_m, int64_t rank, int64_t tiles_per_pe, int64_t total_tiles)
{
    return (pid_m + rank * tiles_per_pe) % total_tiles;
}

/*
 * The consumer schedule built on it.  The GPU plays one PE, rank `rank`, and
 * computes all T_M x T_N output tiles (T_M row tiles, T_N column tiles) with
 * a persistent grid of G consumers.  Every consumer follows one order of the
 * tiles: row tiles in groups of group_rows consecutive rows, the column index
 * outermost inside a group (so consumers working at the same time share the
 * column tiles of B) and running backwards in every second group (so a group
 * starts on the column tiles the previous one used last), and every row tile
 * pid_m renamed so that the PE starts
 * on its own rows and then moves on to the other ranks' rows.  With visit ==
 * NULL the renaming is the page's formula swizzle_row(pid_m, rank,
 * tiles_per_pe, T_M): rank+1's rows next, then rank+2's, ... (the order a
 * ring delivers them).  Otherwise visit[k] names the rank whose rows come
 * k-th (the PE's own rank first, then the others in the order they arrive):
 * pid_m -> visit[pid_m / tiles_per_pe] * tiles_per_pe + pid_m % tiles_per_pe.
 * Consumer c takes positions c, c+G, c+2G, ... of that order.  Writes
 * consumer c's tile indices (q = m*T_N + n) in visit order to out and
 * returns how many.
 */
int64_t opw_oracle_consumer_order(int64_t T_M, int64_t T_N, int64_t G, int64_t c,
                                  int64_t group_rows, int64_t rank, int64_t tiles_per_pe,
                                  const int64_t* visit, int64_t* out)
{
    int64_t count = 0;
    for (int64_t pos = c; pos < T_M * T_N; pos += G) {
        const int64_t first = (pos / (group_rows * T_N)) * group_rows;  /* group's first row */
        const int64_t rows = T_M - first < group_rows ? T_M - first : group_rows;
        const int64_t local = pos - first * T_N;
        const int64_t pid_m = first + local % rows;
        const int64_t col = local / rows;
        /* successive groups sweep the columns in alternating directions */
        const int64_t pid_n = (first / group_rows) % 2 == 0 ? col : T_N - 1 - col;
        const int64_t m = visit == NULL
                              ? opw_oracle_swizzle_row(pid_m, rank, tiles_per_pe, T_M)
                              : visit[pid_m / tiles_per_pe] * tiles_per_pe + pid_m % tiles_per_pe;
        out[count++] = m * T_N + pid_n;
    }
    return count;
}

/* ------------------------------------------------------------------------ */
/* Ring AllReduce                                                            */
/* ------------------------------------------------------------------------ */

/*
 * "Triton-distributed Semantics", "Example: Ring AllReduce with Overlap".
 * R ranks each hold n fp32 values at symmetric offset data_off, viewed as R
 * chunks of n/R values.  Reduce-scatter: in R-1 steps each rank adds its own
 * copy of a chunk to the partial sum it receives from the previous rank
 * (reduced = local + incoming) and passes it on; the partial for chunk c
 * starts at rank c, so its sum is taken in ring order c, c+1, ..., c-1:
 *     S_c = x_{c-1}[c] + ( ... + (x_{c+2}[c] + (x_{c+1}[c] + x_c[c])) ... )
 * in binary32 (indices mod R).  All-gather: R-1 more steps copy each finished
 * chunk around the ring, so every rank ends with every S_c.  The result
 * written at each rank's out_off is therefore concat_c(S_c) on every rank.
 *
 * Writes rank j's result at heap_out + rank_off[j] + out_off.
 */
void opw_oracle_ring_allreduce(const uint8_t* heap, const int64_t* rank_off, int R,
                               int64_t data_off, int64_t out_off, int64_t n, uint8_t* heap_out)
{
    const int64_t chunk = n / R;
    float* S = (float*)malloc((size_t)n * sizeof(float));
    if (!S) return;
    for (int c = 0; c < R; ++c) {
        const float* x_c = (const float*)rank_ptr(heap, rank_off, c, data_off);
        for (int64_t i = 0; i < chunk; ++i) S[c * chunk + i] = x_c[c * chunk + i];
        for (int k = 1; k < R; ++k) {
            const int r = (c + k) % R;
            const float* x_r = (const float*)rank_ptr(heap, rank_off, r, data_off);
            for (int64_t i = 0; i < chunk; ++i) {
                const float local = x_r[c * chunk + i];
                const float incoming = S[c * chunk + i];
                S[c * chunk + i] = local + incoming;
            }
        }
    }
    for (int j = 0; j < R; ++j) {
        float* out_j = (float*)(uintptr_t)rank_ptr(heap_out, rank_off, j, out_off);
        memcpy(out_j, S, (size_t)n * sizeof(float));
    }
    free(S);
}

/* ------------------------------------------------------------------------ */
/* All-to-all                                                                */
/* ------------------------------------------------------------------------ */

/*
 * Aboleth README, Tier-2 all-to-all: every rank puts slice `peer` of its send
 * buffer into the peer's receive buffer at position RANK, then signals the
 * peer.  The plain result: rank j's receive buffer holds, at slot r, slice j
 * of rank r's send buffer:
 *     recv_j[r*B .. (r+1)*B) = send_r[j*B .. (j+1)*B)    for all ranks r, j
 * (B bytes per slice; the slot r == j is the rank's own slice, copied too).
 * Written into heap_out, laid out like the heap.
 */
void opw_oracle_alltoall(const uint8_t* heap, const int64_t* rank_off, int R, int64_t send_off,
                         int64_t recv_off, int64_t B, uint8_t* heap_out)
{
    for (int j = 0; j < R; ++j) {
        uint8_t* recv_j = (uint8_t*)(uintptr_t)rank_ptr(heap_out, rank_off, j, recv_off);
        for (int r = 0; r < R; ++r) {
            const uint8_t* send_r = rank_ptr(heap, rank_off, r, send_off);
            memcpy(recv_j + (int64_t)r * B, send_r + (int64_t)j * B, (size_t)B);
        }
    }
}
