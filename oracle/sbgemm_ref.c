/*
 * Oracle for the strided batched product  C <- alpha * A * B  (optionally + C).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct CPU
 * statement of what the CUDA library computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * constant with the CUDA library, and the library never calls it.
 *
 * Definition followed (StaleyNET "GPU Implementation", section "The matrix
 * product"): for a batch of matrix pairs, C <- alpha * A * B, optionally adding
 * the previous C.  Each input is described by the memory distance between
 * neighbouring rows and neighbouring columns, so a transposed read is the same
 * memory with the two distances exchanged; a third distance steps between the
 * matrices of the batch.  Element (b, i, j) of an operand X is X[b*bs + i*rs + j*cs]
 * with distances counted in fp32 elements.
 *
 * Readings where the page is silent:
 *  - "optionally + C" adds the previous C unscaled: ref = alpha*(A*B) + C0.
 *  - Without accumulation the previous C is not read at all.
 *  - Strides are in elements and may be zero or negative for A and B.
 *
 * For every output element the oracle forms, in fp64,
 *     s     = sum_{k=0..K-1} A[b,m,k] * B[b,k,n]       (k increasing)
 *     t     = sum_{k=0..K-1} |A[b,m,k] * B[b,k,n]|
 *     ref   = alpha * s + (accumulate ? C0[b,m,n] : 0)
 *     bound = |alpha| * t + (accumulate ? |C0[b,m,n]| : 0)
 * Products of two fp32 values are exact in fp64.  `bound` is the scale the
 * tolerance of a GPU result is measured against.
 *
 * Parity pins for this file live in tests/test_oracle.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float* A; int64_t rsA, csA, bsA;
    const float* B; int64_t rsB, csB, bsB;
    const float* C0; int64_t rsC, csC, bsC;
    int64_t M, N, K, batch;
    double alpha;
    int accumulate;
    double* ref;      /* dense [batch][M][N] */
    double* bound;    /* dense [batch][M][N], may be NULL */
    int nthreads;
    int thread;
    int reverse;      /* walk this thread's rows last-to-first */
} oracle_job;

/* One output row (b, m): every n of that row, each sum in increasing k. */
static void oracle_row(const oracle_job* j, int64_t b, int64_t m,
                       double* acc, double* mag) {
    const int64_t N = j->N, K = j->K;
    for (int64_t n = 0; n < N; ++n) { acc[n] = 0.0; mag[n] = 0.0; }
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)j->A[b * j->bsA + m * j->rsA + k * j->csA];
        const float* brow = j->B + b * j->bsB + k * j->rsB;
        for (int64_t n = 0; n < N; ++n) {
            const double p = a * (double)brow[n * j->csB];
            acc[n] += p;
            mag[n] += fabs(p);
        }
    }
    double* out = j->ref + (b * j->M + m) * N;
    double* bnd = j->bound ? j->bound + (b * j->M + m) * N : NULL;
    for (int64_t n = 0; n < N; ++n) {
        double r = j->alpha * acc[n];
        double t = fabs(j->alpha) * mag[n];
        if (j->accumulate) {
            const double c0 = (double)j->C0[b * j->bsC + m * j->rsC + n * j->csC];
            r += c0;
            t += fabs(c0);
        }
        out[n] = r;
        if (bnd) bnd[n] = t;
    }
}

static void* oracle_worker(void* arg) {
    const oracle_job* j = (const oracle_job*)arg;
    const int64_t rows = j->batch * j->M;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    double* mag = (double*)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    if (!acc || !mag) { free(acc); free(mag); return (void*)1; }
    /* Rows are independent; thread t takes rows t, t+T, t+2T, ... */
    int64_t count = rows > j->thread ? (rows - 1 - j->thread) / j->nthreads + 1 : 0;
    for (int64_t i = 0; i < count; ++i) {
        int64_t step = j->reverse ? count - 1 - i : i;
        int64_t r = j->thread + step * j->nthreads;
        oracle_row(j, r / j->M, r % j->M, acc, mag);
    }
    free(acc);
    free(mag);
    return NULL;
}

/* Full product.  Returns 0 on success, -1 on a bad argument, -2 on a thread or
 * allocation failure. */
int sbgemm_ref(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
               const float* B, int64_t rsB, int64_t csB, int64_t bsB,
               const float* C0, int64_t rsC, int64_t csC, int64_t bsC,
               int64_t M, int64_t N, int64_t K, int64_t batch,
               float alpha, int accumulate,
               double* ref, double* bound, int nthreads, int reverse) {
    if (M < 0 || N < 0 || K < 0 || batch < 0) return -1;
    if (M == 0 || N == 0 || batch == 0) return 0;
    if (!ref || (K > 0 && (!A || !B)) || (accumulate && !C0)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    oracle_job base = {A, rsA, csA, bsA, B, rsB, csB, bsB, C0, rsC, csC, bsC,
                       M, N, K, batch, (double)alpha, accumulate, ref, bound,
                       nthreads, 0, reverse};
    oracle_job jobs[256];
    pthread_t tid[256];
    int started = 0, failed = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].thread = t;
        if (t == nthreads - 1) break;     /* the calling thread runs the last */
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) != 0) { failed = 1; break; }
        ++started;
    }
    if (!failed && oracle_worker(&jobs[nthreads - 1]) != NULL) failed = 1;
    for (int t = 0; t < started; ++t) {
        void* rv = NULL;
        pthread_join(tid[t], &rv);
        if (rv != NULL) failed = 1;
    }
    return failed ? -2 : 0;
}

/* The same definition at selected outputs only: idx holds n_points triples
 * (b, m, n).  Used where the full product is too large for the CPU. */
int sbgemm_ref_points(const float* A, int64_t rsA, int64_t csA, int64_t bsA,
                      const float* B, int64_t rsB, int64_t csB, int64_t bsB,
                      const float* C0, int64_t rsC, int64_t csC, int64_t bsC,
                      int64_t M, int64_t N, int64_t K, int64_t batch,
                      float alpha, int accumulate,
                      const int64_t* idx, int64_t n_points,
                      double* ref, double* bound) {
    if (M < 0 || N < 0 || K < 0 || batch < 0 || n_points < 0) return -1;
    for (int64_t p = 0; p < n_points; ++p) {
        const int64_t b = idx[3 * p], m = idx[3 * p + 1], n = idx[3 * p + 2];
        if (b < 0 || b >= batch || m < 0 || m >= M || n < 0 || n >= N) return -1;
        double s = 0.0, t = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double prod = (double)A[b * bsA + m * rsA + k * csA] *
                                (double)B[b * bsB + k * rsB + n * csB];
            s += prod;
            t += fabs(prod);
        }
        double r = (double)alpha * s;
        double u = fabs((double)alpha) * t;
        if (accumulate) {
            const double c0 = (double)C0[b * bsC + m * rsC + n * csC];
            r += c0;
            u += fabs(c0);
        }
        ref[p] = r;
        if (bound) bound[p] = u;
    }
    return 0;
}

/*
 * Fused epilogue (test infrastructure, as above).
 *
 * The fusion a linear layer asks for ("PyTorch demystified 3", section
 * "Summary": add the bias term in the matmul kernel instead of a second pass)
 * extended by an activation, in the usual epilogue order:
 *     z   = alpha * s + (accumulate ? C0 : 0) + D[b,m,n]
 *     out = act(z)
 * D is an addend laid out like any operand (its own row, column and batch
 * strides; zero strides broadcast, so a per-column bias has rs = 0, cs = 1).
 * The activations are the mathematical functions the pages name: ReLU and the
 * two GELUs of "Chapter 09 CUDA backend" (section "Elementwise": Relu,
 * GeluTanh, GeluExact), the sigmoid of "PyTorch demystified 3" and the SiLU of
 * "rvllm CUDA path" (silu(gate)), each evaluated in fp64 with the C library:
 *     0 none       z
 *     1 relu       max(z, 0)
 *     2 sigmoid    1 / (1 + e^-z)
 *     3 silu       z * sigmoid(z)
 *     4 gelu_tanh  z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3)))
 *     5 gelu_erf   z/2 * (1 + erf(z / sqrt(2)))
 * Returns -1 for an unknown activation.
 */
static int oracle_act(int act, double z, double* out) {
    switch (act) {
        case 0: *out = z; return 0;
        case 1: *out = z > 0.0 ? z : 0.0; return 0;
        case 2: *out = 1.0 / (1.0 + exp(-z)); return 0;
        case 3: *out = z / (1.0 + exp(-z)); return 0;
        case 4: {
            const double c = sqrt(2.0 / acos(-1.0));   /* sqrt(2 / pi) */
            *out = 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
            return 0;
        }
        case 5: *out = 0.5 * z * (1.0 + erf(z / sqrt(2.0))); return 0;
        default: return -1;
    }
}

/* out[i] = act(z[i]) for n values. */
int sbgemm_ref_activation(int act, const double* z, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if (oracle_act(act, z[i], &out[i]) != 0) return -1;
    return 0;
}

/* Adds D to product results and applies the activation, at the outputs
 * listed in idx (n_points triples (b, m, n)); z and bound are updated in
 * place (z += D, bound += |D|) and out receives act(z).  D may be NULL. */
int sbgemm_ref_epilogue_points(const float* D, int64_t rsD, int64_t csD, int64_t bsD,
                               int act, const int64_t* idx, int64_t n_points,
                               double* z, double* bound, double* out) {
    for (int64_t p = 0; p < n_points; ++p) {
        const int64_t b = idx[3 * p], m = idx[3 * p + 1], n = idx[3 * p + 2];
        if (D) {
            const double d = (double)D[b * bsD + m * rsD + n * csD];
            z[p] += d;
            if (bound) bound[p] += fabs(d);
        }
        if (oracle_act(act, z[p], &out[p]) != 0) return -1;
    }
    return 0;
}

/*
 * Fused attention (test infrastructure, as above).
 *
 * The three steps of "rvllm CUDA path", section "What's basic about it"
 * (scores, softmax, then probs @ V), here without the scores ever leaving the
 * computation, for a batch of (sequence, head) problems laid out by strides
 * like the product's operands:
 *     s[n]  = alpha * sum_d Q[b,m,d] * K[b,n,d]        (fp64)
 *     masked keys (causal: n > position(m)) drop out of the softmax,
 *     position(m) = (m mod q_len) + N - q_len,
 *     P[n]  = exp(s[n] - max_n s) / sum_n exp(s[n] - max_n s)   (the three
 *             passes of the page's softmax: max, sum of exponentials, divide)
 *     O[b,m,e] = sum_n P[n] * V[b,n,e]
 * and, for the tolerance of a GPU result,
 *     weight[b,m,e] = sum_n P[n] * |V[b,n,e]|
 *     smag[b,m]     = max over kept n of |alpha| * sum_d |Q[b,m,d] * K[b,n,d]|.
 * Stacked grouped-query heads are rows m of one batch entry with q_len the
 * rows per head ("rvllm CUDA path", section "Matmuls go to cuBLAS").
 * Returns 0, or -1 on a bad argument.
 */
int sbgemm_ref_attention(const float* Q, int64_t rsQ, int64_t csQ, int64_t bsQ,
                         const float* K, int64_t rsK, int64_t csK, int64_t bsK,
                         const float* V, int64_t rsV, int64_t csV, int64_t bsV,
                         int64_t M, int64_t N, int64_t D, int64_t Dv, int64_t batch,
                         float alpha, int causal, int64_t q_len,
                         double* O, double* weight, double* smag) {
    if (M < 0 || N <= 0 || D < 0 || Dv < 0 || batch < 0) return -1;
    if (causal && (q_len <= 0 || q_len > N)) return -1;
    double* s = (double*)malloc((size_t)N * sizeof(double));
    double* mag = (double*)malloc((size_t)N * sizeof(double));
    if (!s || !mag) { free(s); free(mag); return -1; }
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t m = 0; m < M; ++m) {
            const int64_t kept = causal ? (m % q_len) + N - q_len + 1 : N;
            double mx = -INFINITY, big = 0.0;
            for (int64_t n = 0; n < kept; ++n) {
                double acc = 0.0, t = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    const double prod = (double)Q[b * bsQ + m * rsQ + d * csQ] *
                                        (double)K[b * bsK + n * rsK + d * csK];
                    acc += prod;
                    t += fabs(prod);
                }
                s[n] = (double)alpha * acc;
                mag[n] = fabs((double)alpha) * t;
                if (s[n] > mx) mx = s[n];
                if (mag[n] > big) big = mag[n];
            }
            double l = 0.0;
            for (int64_t n = 0; n < kept; ++n) {
                s[n] = exp(s[n] - mx);
                l += s[n];
            }
            for (int64_t e = 0; e < Dv; ++e) {
                double o = 0.0, w = 0.0;
                for (int64_t n = 0; n < kept; ++n) {
                    const double v = (double)V[b * bsV + n * rsV + e * csV];
                    o += s[n] * v;
                    w += s[n] * fabs(v);
                }
                O[(b * M + m) * Dv + e] = o / l;
                if (weight) weight[(b * M + m) * Dv + e] = w / l;
            }
            if (smag) smag[b * M + m] = big;
        }
    }
    free(s);
    free(mag);
    return 0;
}

/*
 * Paged key / value cache read (test infrastructure, as above).
 *
 * "rvllm CUDA path", section "The kernels": the cache is one buffer shaped
 * [num_blocks][block_size][n_kv_heads][head_dim]; a sequence's context
 * position pos lives in the block that the sequence's row of the block table
 * names for pos / block_size, at offset pos % block_size inside it.  This
 * copies the rows of positions 0..len-1 of one (sequence, head) into a
 * contiguous [len][head_dim] buffer, the gather step the page describes, so
 * that attention over paged keys is this gather followed by
 * sbgemm_ref_attention.  Returns 0, or -1 if a position needs a table entry
 * past max_blocks or a block id outside [0, num_blocks) (nothing is read
 * from the cache then).
 */
int sbgemm_ref_kv_gather(const float* cache, int64_t num_blocks, int64_t block_size,
                         int64_t n_kv_heads, int64_t head_dim,
                         const int32_t* block_table, int64_t max_blocks,
                         int64_t seq, int64_t head, int64_t len, float* out) {
    if (num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim < 0 ||
        max_blocks <= 0 || seq < 0 || head < 0 || head >= n_kv_heads || len < 0)
        return -1;
    for (int64_t pos = 0; pos < len; ++pos) {
        const int64_t block_pos = pos / block_size;
        const int64_t offset = pos % block_size;
        if (block_pos >= max_blocks) return -1;
        const int64_t block = block_table[seq * max_blocks + block_pos];
        if (block < 0 || block >= num_blocks) return -1;
        const float* row = cache + ((block * block_size + offset) * n_kv_heads + head) * head_dim;
        for (int64_t d = 0; d < head_dim; ++d) out[pos * head_dim + d] = row[d];
    }
    return 0;
}
