/*
 * fp64 reference of the multi-LoRA batched linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may call this code; the library's compute path never does.
 * It shares no code with the CUDA path.
 *
 * What it computes, for every selected token row t and output column o:
 *
 *   y[t,o] = sum_i W[o,i] x[t,i]
 *          + sum over j with slot[t,j] != -1 of
 *                c_j * sum_q B_s[o,q] * (sum_i A_s[q,i] x[t,i]),   s = slot[t,j]
 *   c_j    = scale[t,j] * alpha_s / r_s        (plain LoRA)
 *   c_j    = scale[t,j] * alpha_s / sqrt(r_s)  (rsLoRA)
 *
 * Sources:
 * - "Multi-LoRA Serving Explained" (sevydevy.com), the LoRA-basics section:
 *   B is d x r, A is r x k, the layer computes W x + B(A x), the side path
 *   scaled by alpha / r; the batched-serving section: one shared base product
 *   plus each token's own side path, slot -1 meaning "base model only".
 * - "[RFC] Per-request activation of multiple LoRA adapters" (vLLM issue
 *   51940), "Proposed Change / Semantics": base(x) + sum_i s_i (alpha_i/r_i)
 *   B_i A_i x, unused slots of a token filled with the sentinel.
 * - "[vLLM] LoRA" (secrett2633 blog), PEFTHelper: alpha / sqrt(r) under rsLoRA.
 *
 * Adapters are given unpadded (A_s is [r_s, K], B_s is [D, r_s], row-major),
 * exactly as the pages define them; r_s is the adapter's true rank.
 * Parenthesisation follows the definition: A x first (r_s numbers), then B.
 * Sentinel and zero-scale pairs contribute nothing: the row is the base sum.
 *
 * Error behaviour: a slot id below -1, at or above n_slots, or naming a slot
 * with no adapter (A_s == NULL) makes the call return ORACLE_ERR_BAD_SLOT
 * before anything is written.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_ERR_BAD_SLOT 1
#define ORACLE_ERR_ARG 2
#define ORACLE_ERR_OOM 3

typedef struct {
    int T, K, D, J, n_slots;
    const double* x;
    const double* W;
    const int32_t* token_slots;
    const double* scales;
    const double* const* A;
    const double* const* B;
    const int32_t* rank;
    const double* alpha;
    const int32_t* rslora;
    int n_rows, n_cols;
    const int32_t* rows;
    const int32_t* cols;
    double* y;
    int row_begin, row_end;
    int failed;
} work_t;

static double adapter_coefficient(double alpha, int r, int rslora) {
    return rslora ? alpha / sqrt((double)r) : alpha / (double)r;
}

static void* run_rows(void* arg) {
    work_t* w = (work_t*)arg;
    int r_cap = 0;
    for (int s = 0; s < w->n_slots; ++s)
        if (w->A[s] && w->rank[s] > r_cap) r_cap = w->rank[s];
    double* v = (double*)malloc(sizeof(double) * (size_t)(w->J > 0 ? w->J : 1) * (size_t)(r_cap > 0 ? r_cap : 1));
    double* c = (double*)malloc(sizeof(double) * (size_t)(w->J > 0 ? w->J : 1));
    if (!v || !c) {
        free(v);
        free(c);
        w->failed = 1;
        return 0;
    }
    for (int ri = w->row_begin; ri < w->row_end; ++ri) {
        const int t = w->rows ? w->rows[ri] : ri;
        const double* xt = w->x + (size_t)t * (size_t)w->K;
        /* side path, first factor: v_j = A_s x_t (r_s numbers per active j) */
        for (int j = 0; j < w->J; ++j) {
            const int s = w->token_slots[(size_t)t * (size_t)w->J + (size_t)j];
            c[j] = 0.0;
            if (s == -1) continue;
            const double sc = w->scales ? w->scales[(size_t)t * (size_t)w->J + (size_t)j] : 1.0;
            c[j] = sc * adapter_coefficient(w->alpha[s], w->rank[s], w->rslora[s]);
            const double* As = w->A[s];
            for (int q = 0; q < w->rank[s]; ++q) {
                double acc = 0.0;
                for (int i = 0; i < w->K; ++i) acc += As[(size_t)q * (size_t)w->K + (size_t)i] * xt[i];
                v[(size_t)j * (size_t)r_cap + (size_t)q] = acc;
            }
        }
        for (int ci = 0; ci < w->n_cols; ++ci) {
            const int o = w->cols ? w->cols[ci] : ci;
            const double* Wo = w->W + (size_t)o * (size_t)w->K;
            double acc = 0.0;
            for (int i = 0; i < w->K; ++i) acc += Wo[i] * xt[i];
            for (int j = 0; j < w->J; ++j) {
                const int s = w->token_slots[(size_t)t * (size_t)w->J + (size_t)j];
                if (s == -1) continue;
                const int r = w->rank[s];
                const double* Bo = w->B[s] + (size_t)o * (size_t)r;
                double side = 0.0;
                for (int q = 0; q < r; ++q) side += Bo[q] * v[(size_t)j * (size_t)r_cap + (size_t)q];
                acc += c[j] * side;
            }
            w->y[(size_t)ri * (size_t)w->n_cols + (size_t)ci] = acc;
        }
    }
    free(v);
    free(c);
    return 0;
}

/*
 * rows/cols select the output sub-matrix (NULL = all T rows / all D columns);
 * y is [n_rows, n_cols] row-major. scales NULL means every scale is 1.
 * n_threads > 1 splits the selected rows across POSIX threads (each row is
 * computed by one thread, in the order written above).
 */
int oracle_mlora_linear(int T, int K, int D, int J, const double* x, const double* W,
                        const int32_t* token_slots, const double* scales, int n_slots,
                        const double* const* A, const double* const* B, const int32_t* rank,
                        const double* alpha, const int32_t* rslora, int n_rows,
                        const int32_t* rows, int n_cols, const int32_t* cols, double* y,
                        int n_threads) {
    if (T < 0 || K < 0 || D < 0 || J < 0 || n_slots < 0 || n_rows < 0 || n_cols < 0) return ORACLE_ERR_ARG;
    if ((T > 0 && K > 0 && !x) || (D > 0 && K > 0 && !W) || (T > 0 && J > 0 && !token_slots)) return ORACLE_ERR_ARG;
    if ((n_rows > 0 && n_cols > 0 && !y) || (n_slots > 0 && (!A || !B || !rank || !alpha || !rslora)))
        return ORACLE_ERR_ARG;
    for (int i = 0; i < n_rows; ++i)
        if (rows && (rows[i] < 0 || rows[i] >= T)) return ORACLE_ERR_ARG;
    for (int i = 0; i < n_cols; ++i)
        if (cols && (cols[i] < 0 || cols[i] >= D)) return ORACLE_ERR_ARG;
    if (!rows && n_rows != T) return ORACLE_ERR_ARG;
    if (!cols && n_cols != D) return ORACLE_ERR_ARG;
    for (int s = 0; s < n_slots; ++s)
        if (A[s] && (!B[s] || rank[s] < 1)) return ORACLE_ERR_ARG;
    for (long p = 0; p < (long)T * (long)J; ++p) {
        const int s = token_slots[p];
        if (s == -1) continue;
        if (s < -1 || s >= n_slots || !A[s]) return ORACLE_ERR_BAD_SLOT;
    }
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_rows) n_threads = n_rows > 0 ? n_rows : 1;
    if (n_threads > 512) n_threads = 512;
    work_t* jobs = (work_t*)calloc((size_t)n_threads, sizeof(work_t));
    pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
    int* started = (int*)calloc((size_t)n_threads, sizeof(int));
    if (!jobs || !tids || !started) {
        free(jobs);
        free(tids);
        free(started);
        return ORACLE_ERR_OOM;
    }
    for (int k = 0; k < n_threads; ++k) {
        work_t w = {T, K, D, J, n_slots, x, W, token_slots, scales, A, B, rank, alpha, rslora,
                    n_rows, n_cols, rows, cols, y, 0, 0, 0};
        w.row_begin = (int)((long)n_rows * k / n_threads);
        w.row_end = (int)((long)n_rows * (k + 1) / n_threads);
        jobs[k] = w;
    }
    for (int k = 1; k < n_threads; ++k) {
        if (pthread_create(&tids[k], 0, run_rows, &jobs[k]) == 0)
            started[k] = 1;
        else
            run_rows(&jobs[k]);
    }
    run_rows(&jobs[0]);
    int failed = jobs[0].failed;
    for (int k = 1; k < n_threads; ++k) {
        if (started[k]) pthread_join(tids[k], 0);
        failed |= jobs[k].failed;
    }
    free(jobs);
    free(tids);
    free(started);
    return failed ? ORACLE_ERR_OOM : ORACLE_OK;
}
