/*
 * dspark_oracle.c — plain, slow, fp64 CPU oracle of the DSpark per-round hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header or table with the CUDA library; the two meet only through
 * the seeded synthetic inputs.
 *
 * Every function follows the method's definition step by step, in double precision,
 * from inputs converted exactly (fp32 -> fp64, bf16 -> fp64).  No blocking, fusion
 * or reordering beyond what the definition states.  OpenMP runs independent requests
 * in parallel; each request's arithmetic is sequential and in a fixed order.
 *
 * Sources (web pages about the DSpark paper, arXiv 2607.05147):
 *   [EXPL]  numb3r33 blog, "DSpark: confidence-scheduled speculative decoding"
 *   [VLLM]  vllmbangkok blog, "DSpark: Confidence-Scheduled Speculative Decoding with
 *           Semi-Autoregressive Generation"
 *   [KB]    edgeai1 knowledge base, "DSpark 精读"
 *   [FR]    mkdocs.reaper.mx, "3 · DSpark"
 *   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 *           SC'11 — the Philox4x32-10 counter-based generator.
 *
 * Parity pins: every function here is pinned by the not-gpu tests (worked examples
 * printed on the pages, closed forms, brute-force law at V=8, chi-square over 10^6
 * seeded trials, brute-force scheduler optimum).  No function is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_EARLY_STOP 0
#define ORC_FULL_SEARCH 1
#define ORC_CAPACITY_K 2
#define ORC_FIXED 3

#define ORC_STREAM_DRAFT 0u
#define ORC_STREAM_ACCEPT 1u
#define ORC_STREAM_CORRECT 2u

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [PHILOX]: S-box free bijection built from two 32x32->64
 * multiplications per round, 10 rounds, key bumped by the Weyl constants
 * (golden ratio and sqrt(3)-1 fractions) between rounds.                    */
/* ------------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint64_t MUL_A = 0xD2511F53u, MUL_B = 0xCD9E8D57u;
    const uint32_t WEYL_A = 0x9E3779B9u, WEYL_B = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += WEYL_A;
            k1 += WEYL_B;
        }
        uint64_t pa = MUL_A * (uint64_t)c0;
        uint64_t pb = MUL_B * (uint64_t)c2;
        uint32_t hi_a = (uint32_t)(pa >> 32), lo_a = (uint32_t)pa;
        uint32_t hi_b = (uint32_t)(pb >> 32), lo_b = (uint32_t)pb;
        uint32_t n0 = hi_b ^ c1 ^ k0;
        uint32_t n1 = lo_b;
        uint32_t n2 = hi_a ^ c3 ^ k1;
        uint32_t n3 = lo_a;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The counter layout of the method's random draws ("counter-based RNG keyed by
 * (seed, request, position)"): counter = (lo32 req_id, lo32 round,
 * stream<<24 | position, chunk), key = (lo32 seed, hi32 seed).  Element v of a
 * vocabulary row takes word v%4 of chunk v/4.  Returns the raw 32-bit word.  */
uint32_t orc_draw_bits(uint64_t seed, uint64_t req_id, uint64_t round, uint32_t stream,
                       uint32_t position, uint32_t chunk, uint32_t lane) {
    uint32_t ctr[4] = {(uint32_t)req_id, (uint32_t)round, (stream << 24) | position, chunk};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[lane & 3u];
}

/* Uniform in (0,1): the top 24 bits, centred in their cell: ((b>>8)+1/2) / 2^24. */
double orc_uniform(uint32_t bits) { return ((double)(bits >> 8) + 0.5) * (1.0 / 16777216.0); }

/* Standard Gumbel from a uniform: g = -ln(-ln u).  ln u is taken as log1p(u-1),
 * u-1 being exact in binary64, so the tail u -> 1 keeps full relative accuracy. */
double orc_gumbel(double u) { return -log(-log1p(u - 1.0)); }

static double orc_load(const void* base, int dtype, size_t idx) {
    if (dtype == ORC_F32) return (double)((const float*)base)[idx];
    uint16_t b = ((const uint16_t*)base)[idx];
    uint32_t f = ((uint32_t)b) << 16;
    float x;
    memcpy(&x, &f, sizeof x);
    return (double)x;
}

static int orc_threads(int want) {
#ifdef _OPENMP
    if (want > 0) return want;
    return omp_get_max_threads();
#else
    (void)want;
    return 1;
#endif
}

/* z = (U_k + W1[x_prev,:] W2) / T over the whole vocabulary ([EXPL] "Markov sequential
 * head": p_k(v|x_{k-1}) = softmax(U_k(v) + B(x_{k-1},v)), B(x,:) = W1[x,:] W2; [KB] §2
 * writes the same law with the anchor x_0 conditioning position 1).  The temperature
 * divides the whole logit row. */
static void orc_draft_logits(int V, int rank, int dtype_u, int dtype_w, const void* U, size_t u_row,
                             const void* W1, const void* W2, int x_prev, double temperature,
                             double* z) {
    for (int v = 0; v < V; ++v) z[v] = 0.0;
    for (int i = 0; i < rank; ++i) {
        double w1 = orc_load(W1, dtype_w, (size_t)x_prev * rank + i);
        for (int v = 0; v < V; ++v) z[v] += w1 * orc_load(W2, dtype_w, (size_t)i * V + v);
    }
    for (int v = 0; v < V; ++v) z[v] = (orc_load(U, dtype_u, u_row + v) + z[v]) / temperature;
}

/* z = (U_row + a W2) / T for an explicit factor row a[rank] (the head's state). */
static void orc_row_logits(int V, int rank, int dtype_u, int dtype_w, const void* U, size_t u_row,
                           const double* arow, const void* W2, double temperature, double* z) {
    for (int v = 0; v < V; ++v) z[v] = 0.0;
    for (int i = 0; i < rank; ++i) {
        const double w1 = arow[i];
        for (int v = 0; v < V; ++v) z[v] += w1 * orc_load(W2, dtype_w, (size_t)i * V + v);
    }
    for (int v = 0; v < V; ++v) z[v] = (orc_load(U, dtype_u, u_row + v) + z[v]) / temperature;
}

static double orc_logsumexp(const double* z, int V) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (z[v] > m) m = z[v];
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp(z[v] - m);
    return m + log(s);
}

/* argmax_v (score_v + g_v), g_v standard Gumbel from the given stream/position,
 * restricted to v with valid[v] != 0 (valid == NULL: all).  Lowest v wins ties.
 * Also reports the runner-up and the key margin between the two. */
static int orc_gumbel_argmax(const double* score, const unsigned char* valid, int V, uint64_t seed,
                             uint64_t req_id, uint64_t round, uint32_t stream, uint32_t position,
                             int* runner_up, double* margin) {
    int best = -1, second = -1;
    double kbest = -INFINITY, ksecond = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (valid && !valid[v]) continue;
        double g = orc_gumbel(orc_uniform(orc_draw_bits(seed, req_id, round, stream, position,
                                                        (uint32_t)v >> 2, (uint32_t)v & 3u)));
        double key = score[v] + g;
        if (best < 0 || key > kbest) {
            second = best; ksecond = kbest;
            best = v; kbest = key;
        } else if (second < 0 || key > ksecond) {
            second = v; ksecond = key;
        }
    }
    if (runner_up) *runner_up = second;
    if (margin) *margin = (second < 0) ? INFINITY : kbest - ksecond;
    return best;
}

static double orc_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* Stage 1 — Markov-head draft loop with the confidence head.                 */
/* ------------------------------------------------------------------------- */
/* For each request r and k = 1..gamma (x_0 = anchor):
 *   z      = (U[r,k-1,:] + W1[x_{k-1},:] W2) / T                     [EXPL] Markov head
 *   lse_k  = log sum_v exp z_v ;  x_k = argmax_v z_v + g_v (Gumbel-max draw of
 *            softmax(z), stream 0 at position k)                      [VLLM] §4.1
 *   logq_k = z_{x_k} - lse_k
 *   c_k    = sigmoid(kappa * (w_h . h[r,k-1,:] + w_e . W1[x_{k-1},:] + b) / T_k)
 *            (linear + sigmoid on [h_k ; W1[x_{k-1}]], [KB] §4; per-position
 *            temperature of sequential temperature scaling, [EXPL] "Sequential
 *            temperature scaling"; kappa scales the raw logit).
 * Diagnostics: runner_up / margin of the Gumbel draw (boundary-case rule). */
int orc_markov_draft(int R, int gamma, int V, int rank, int d, int dtype_u, int dtype_w, int dtype_h,
                     const void* U, const void* W1, const void* W2, const void* h,
                     const float* conf_w, double conf_b, double conf_logit_scale,
                     const float* conf_temp, double temperature, const int32_t* x0,
                     const int64_t* req_id, uint64_t seed, uint64_t round, int32_t* x_out,
                     double* logq_out, double* lse_out, double* conf_out, int32_t* runner_up_out,
                     double* margin_out, int nthreads) {
    if (R < 0 || gamma < 1 || V < 1 || rank < 1 || d < 0 || temperature <= 0.0) return 1;
    int nt = orc_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int r = 0; r < R; ++r) {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        int x_prev = x0[r];
        for (int k = 1; k <= gamma; ++k) {
            size_t row = ((size_t)r * gamma + (k - 1));
            orc_draft_logits(V, rank, dtype_u, dtype_w, U, row * (size_t)V, W1, W2, x_prev,
                             temperature, z);
            double lse = orc_logsumexp(z, V);
            int ru = -1;
            double mg = 0.0;
            int xk = orc_gumbel_argmax(z, NULL, V, seed, (uint64_t)req_id[r], round,
                                       ORC_STREAM_DRAFT, (uint32_t)k, &ru, &mg);
            double s_h = 0.0;
            for (int i = 0; i < d; ++i) s_h += (double)conf_w[i] * orc_load(h, dtype_h, row * (size_t)d + i);
            double s_e = 0.0;
            for (int i = 0; i < rank; ++i)
                s_e += (double)conf_w[d + i] * orc_load(W1, dtype_w, (size_t)x_prev * rank + i);
            double logit = conf_logit_scale * (s_h + s_e + conf_b);
            double c = orc_sigmoid(logit / (double)conf_temp[k - 1]);
            x_out[row] = xk;
            logq_out[row] = z[xk] - lse;
            lse_out[row] = lse;
            conf_out[row] = c;
            if (runner_up_out) runner_up_out[row] = ru;
            if (margin_out) margin_out[row] = mg;
            x_prev = xk;
        }
        free(z);
    }
    return 0;
}

/* Full draft distribution q_k(. | x_prev) for one request/position (test helper). */
int orc_draft_distribution(int V, int rank, int dtype_u, int dtype_w, const void* U_row,
                           const void* W1, const void* W2, int x_prev, double temperature,
                           double* q_out) {
    orc_draft_logits(V, rank, dtype_u, dtype_w, U_row, 0, W1, W2, x_prev, temperature, q_out);
    double lse = orc_logsumexp(q_out, V);
    for (int v = 0; v < V; ++v) q_out[v] = exp(q_out[v] - lse);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Stage 2 — confidence scheduler.                                            */
/* ------------------------------------------------------------------------- */
typedef struct {
    double a;
    int depth; /* j, 1-based */
    int req;   /* r */
} orc_cand;

/* (a desc, depth asc, request asc): a is non-increasing along each request's chain,
 * so with depth ascending on ties a request's prefix is always admitted in order
 * ([EXPL] "Greedy prefix allocation"). */
static int orc_cand_cmp(const void* pa, const void* pb) {
    const orc_cand* a = (const orc_cand*)pa;
    const orc_cand* b = (const orc_cand*)pb;
    if (a->a > b->a) return -1;
    if (a->a < b->a) return 1;
    if (a->depth != b->depth) return a->depth < b->depth ? -1 : 1;
    if (a->req != b->req) return a->req < b->req ? -1 : 1;
    return 0;
}

/* a_{r,j} = prod_{i<=j} c_{r,i}, multiplied left to right in binary64 ([KB] §4,
 * [FR] §3.3), then sorted globally. */
static void orc_sorted_candidates(int R, int gamma, const float* conf, orc_cand* out) {
    for (int r = 0; r < R; ++r) {
        double a = 1.0;
        for (int j = 1; j <= gamma; ++j) {
            a = a * (double)conf[(size_t)r * gamma + (j - 1)];
            orc_cand c = {a, j, r};
            out[(size_t)r * gamma + (j - 1)] = c;
        }
    }
    qsort(out, (size_t)R * gamma, sizeof(orc_cand), orc_cand_cmp);
}

/* Theta(n) = tau(n) * SPS(R + n) along the admission path, tau(n) = R + sum of the
 * first n sorted a's ([KB] §4: B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a),
 * maximise tau * SPS(B); [EXPL] "Scheduler objective"). */
static void orc_theta_path(int R, int N, const orc_cand* sorted, const double* sps, double* tau,
                           double* theta) {
    tau[0] = (double)R;
    theta[0] = tau[0] * sps[R];
    for (int n = 1; n <= N; ++n) {
        tau[n] = tau[n - 1] + sorted[n - 1].a;
        theta[n] = tau[n] * sps[R + n];
    }
}

static int orc_full_search(int N, const double* theta) {
    int best = 0;
    for (int n = 1; n <= N; ++n)
        if (theta[n] > theta[best]) best = n;
    return best;
}

/* Modes:
 *  EARLY_STOP  — admit in sorted order, stop at the first n with Theta(n+1) <= Theta(n)
 *                (non-anticipating ideal scheduler, [EXPL] "Losslessness and
 *                non-anticipation", [KB] §4 "首次不增").
 *  FULL_SEARCH — n* = argmax_n Theta(n), smallest n on ties ([VLLM] §4.2.2, jagged SPS).
 *  CAPACITY_K  — K = FULL_SEARCH count on the stale confidences conf_hist; admit the
 *                top-K by the current order ([EXPL] "Async scheduler in practice").
 *  FIXED       — l_r = min(fixed_len, gamma) for every request (scheduler off).
 * Diagnostics (boundary-case rule): diag[0] = smallest relative Theta gap met by a
 * decision on the path, diag[1] = relative gap between the a's either side of the cut. */
int orc_schedule(int R, int gamma, const float* conf, const double* sps, int sps_len, int mode,
                 const float* conf_hist, int fixed_len, int32_t* ell_out, int32_t* B_out,
                 double* tau_out, double* diag) {
    int N = R * gamma;
    if (R < 0 || gamma < 1 || sps_len < R * (gamma + 1) + 1) return 1;
    if (mode == ORC_CAPACITY_K && conf_hist == NULL) return 1;
    orc_cand* cand = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(N > 0 ? N : 1));
    double* tau = (double*)malloc(sizeof(double) * (size_t)(N + 1));
    double* theta = (double*)malloc(sizeof(double) * (size_t)(N + 1));
    orc_sorted_candidates(R, gamma, conf, cand);
    orc_theta_path(R, N, cand, sps, tau, theta);
    for (int r = 0; r < R; ++r) ell_out[r] = 0;
    double gap = INFINITY, tie = INFINITY;
    int nstar = 0;
    if (mode == ORC_FIXED) {
        int L = fixed_len < 0 ? 0 : (fixed_len > gamma ? gamma : fixed_len);
        double t = (double)R;
        for (int r = 0; r < R; ++r) {
            double a = 1.0;
            for (int j = 1; j <= L; ++j) {
                a = a * (double)conf[(size_t)r * gamma + (j - 1)];
                t += a;
            }
            ell_out[r] = L;
        }
        *B_out = R + R * L;
        *tau_out = t;
        if (diag) { diag[0] = INFINITY; diag[1] = INFINITY; }
        free(cand); free(tau); free(theta);
        return 0;
    }
    if (mode == ORC_EARLY_STOP) {
        nstar = N;
        for (int n = 0; n < N; ++n) {
            double g = fabs(theta[n + 1] - theta[n]) / theta[n];
            if (g < gap) gap = g;
            if (theta[n + 1] <= theta[n]) { nstar = n; break; }
        }
    } else if (mode == ORC_FULL_SEARCH) {
        nstar = orc_full_search(N, theta);
        for (int n = 0; n <= N; ++n) {
            if (n == nstar) continue;
            double g = fabs(theta[nstar] - theta[n]) / theta[nstar];
            if (g < gap) gap = g;
        }
    } else if (mode == ORC_CAPACITY_K) {
        orc_cand* hc = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(N > 0 ? N : 1));
        double* ht = (double*)malloc(sizeof(double) * (size_t)(N + 1));
        double* hth = (double*)malloc(sizeof(double) * (size_t)(N + 1));
        orc_sorted_candidates(R, gamma, conf_hist, hc);
        orc_theta_path(R, N, hc, sps, ht, hth);
        int K = orc_full_search(N, hth);
        for (int n = 0; n <= N; ++n) {
            if (n == K) continue;
            double g = fabs(hth[K] - hth[n]) / hth[K];
            if (g < gap) gap = g;
        }
        nstar = K < N ? K : N;
        free(hc); free(ht); free(hth);
    } else {
        free(cand); free(tau); free(theta);
        return 1;
    }
    if (nstar > 0 && nstar < N) {
        double hi = cand[nstar - 1].a, lo = cand[nstar].a;
        tie = (hi - lo) / hi;
    }
    for (int n = 0; n < nstar; ++n) ell_out[cand[n].req] += 1;
    *B_out = R + nstar;
    *tau_out = tau[nstar];
    if (diag) { diag[0] = gap; diag[1] = tie; }
    free(cand); free(tau); free(theta);
    return 0;
}

/* Theta path along the sorted order, for tests: writes a_(n) (n=1..N) and Theta(n). */
int orc_schedule_path(int R, int gamma, const float* conf, const double* sps, double* a_sorted,
                      int32_t* req_sorted, int32_t* depth_sorted, double* theta_out) {
    int N = R * gamma;
    orc_cand* cand = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(N > 0 ? N : 1));
    double* tau = (double*)malloc(sizeof(double) * (size_t)(N + 1));
    orc_sorted_candidates(R, gamma, conf, cand);
    orc_theta_path(R, N, cand, sps, tau, theta_out);
    for (int n = 0; n < N; ++n) {
        a_sorted[n] = cand[n].a;
        req_sorted[n] = cand[n].req;
        depth_sorted[n] = cand[n].depth;
    }
    free(cand); free(tau);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Stage 3 — exact speculative-sampling verification.                         */
/* ------------------------------------------------------------------------- */
/* For request r with verify length l = ell[r]:
 *   for j = 1..l: p_t = softmax(target[r,j-1,:] / T); accept x_j iff
 *       u_j < p_t(x_j) / q_j(x_j), u_j uniform from stream 1 at position j
 *       (min(1, p/q) acceptance, [EXPL] "One-token exactness"); stop at the first
 *       rejection ([EXPL] "Why only the longest accepted prefix survives").
 *   n_acc = accepted count.
 *   if n_acc < l: j* = n_acc+1, q = softmax(z) with z the draft logits of position j*
 *       (recomputed from U, W1[x_{j*-1}], W2 and normalised by the draft's lse),
 *       p = softmax(target[r,j*-1]/T), rho = (p - q)_+, y drawn from rho/sum(rho) as
 *       argmax_{rho_v>0} ln rho_v + g_v (stream 2 at position j*) — residual
 *       correction ([EXPL] "One-token exactness").  If no rho_v > 0 (rounding only),
 *       y is drawn from p with the same Gumbels.
 *   else (every verified draft accepted, including l = 0): bonus token
 *       y = argmax_v target[r,l,v]/T + g_v (stream 2 at position l+1) ([EXPL] "Prefix
 *       survival and accepted length"; [KB] §6 counts it in tau).
 *   tokens = x_1..x_{n_acc}, y;  n_out = n_acc + 1.
 * Diagnostics per request: acc_margin[r*gamma + j-1] = u_j - ratio_j for tested j;
 * corr_margin[r] = Gumbel key margin of the correction draw; corr_rho[r*2 + 0/1] =
 * rho/max(p,q) of winner/runner-up for a residual draw (1 for a bonus draw).
 * With the recurrent head (state != NULL, [R,gamma,rank] stored states), the residual's
 * bias row is state[r,j*-1,:] W2 instead of W1[x_{j*-1},:] W2. */
int orc_verify(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
               const void* target, const void* U, const void* W1, const void* W2,
               const int32_t* x0, const int32_t* x, const double* logq, const double* lse_q,
               const int32_t* ell, double temperature, const int64_t* req_id, uint64_t seed,
               uint64_t round, int32_t* n_acc_out, int32_t* tokens_out, int32_t* n_out,
               double* acc_margin, double* corr_margin, double* corr_rho, int32_t* corr_kind,
               const double* state, int nthreads) {
    if (R < 0 || gamma < 1 || V < 1 || temperature <= 0.0) return 1;
    for (int r = 0; r < R; ++r)
        if (ell[r] < 0 || ell[r] > gamma) return 1;
    int nt = orc_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int r = 0; r < R; ++r) {
        double* t = (double*)malloc(sizeof(double) * (size_t)V);
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        unsigned char* pos = (unsigned char*)malloc((size_t)V);
        const int l = ell[r];
        const uint64_t rid = (uint64_t)req_id[r];
        for (int j = 0; j < gamma; ++j)
            if (acc_margin) acc_margin[(size_t)r * gamma + j] = NAN;
        int n_acc = 0;
        for (int j = 1; j <= l; ++j) {
            size_t trow = ((size_t)r * (gamma + 1) + (j - 1)) * (size_t)V;
            for (int v = 0; v < V; ++v) t[v] = orc_load(target, dtype_t, trow + v) / temperature;
            double lse_t = orc_logsumexp(t, V);
            int xj = x[(size_t)r * gamma + (j - 1)];
            double lp = t[xj] - lse_t;
            double ratio = exp(lp - logq[(size_t)r * gamma + (j - 1)]);
            double u = orc_uniform(orc_draw_bits(seed, rid, round, ORC_STREAM_ACCEPT, (uint32_t)j, 0u, 0u));
            if (acc_margin) acc_margin[(size_t)r * gamma + (j - 1)] = u - ratio;
            if (u < ratio) n_acc += 1;
            else break;
        }
        int y, ru = -1;
        double mg = INFINITY;
        int kind;
        if (n_acc < l) {
            int js = n_acc + 1;
            int xprev = (js == 1) ? x0[r] : x[(size_t)r * gamma + (js - 2)];
            size_t urow = ((size_t)r * gamma + (js - 1)) * (size_t)V;
            if (state)
                orc_row_logits(V, rank, dtype_u, dtype_w, U, urow, state + ((size_t)r * gamma + (js - 1)) * rank, W2,
                               temperature, z);
            else
                orc_draft_logits(V, rank, dtype_u, dtype_w, U, urow, W1, W2, xprev, temperature, z);
            double lq = lse_q[(size_t)r * gamma + (js - 1)];
            size_t trow = ((size_t)r * (gamma + 1) + (js - 1)) * (size_t)V;
            for (int v = 0; v < V; ++v) t[v] = orc_load(target, dtype_t, trow + v) / temperature;
            double lse_t = orc_logsumexp(t, V);
            int any = 0;
            double* score = z; /* reuse: score_v = ln rho_v */
            double* rho_rel = (double*)malloc(sizeof(double) * (size_t)V);
            for (int v = 0; v < V; ++v) {
                double p = exp(t[v] - lse_t);
                double q = exp(z[v] - lq);
                double rho = p - q;
                double mx = p > q ? p : q;
                rho_rel[v] = mx > 0.0 ? rho / mx : 0.0;
                pos[v] = rho > 0.0;
                any |= pos[v];
                score[v] = rho > 0.0 ? log(rho) : -INFINITY;
            }
            if (any) {
                y = orc_gumbel_argmax(score, pos, V, seed, rid, round, ORC_STREAM_CORRECT,
                                      (uint32_t)js, &ru, &mg);
                kind = 1;
                if (corr_rho) {
                    corr_rho[(size_t)r * 2 + 0] = rho_rel[y];
                    corr_rho[(size_t)r * 2 + 1] = ru >= 0 ? rho_rel[ru] : 1.0;
                }
            } else {
                y = orc_gumbel_argmax(t, NULL, V, seed, rid, round, ORC_STREAM_CORRECT,
                                      (uint32_t)js, &ru, &mg);
                kind = 2;
                if (corr_rho) { corr_rho[(size_t)r * 2 + 0] = 0.0; corr_rho[(size_t)r * 2 + 1] = 0.0; }
            }
            free(rho_rel);
        } else {
            size_t trow = ((size_t)r * (gamma + 1) + l) * (size_t)V;
            for (int v = 0; v < V; ++v) t[v] = orc_load(target, dtype_t, trow + v) / temperature;
            y = orc_gumbel_argmax(t, NULL, V, seed, rid, round, ORC_STREAM_CORRECT,
                                  (uint32_t)(l + 1), &ru, &mg);
            kind = 0;
            if (corr_rho) { corr_rho[(size_t)r * 2 + 0] = 1.0; corr_rho[(size_t)r * 2 + 1] = 1.0; }
        }
        for (int j = 0; j <= gamma; ++j) tokens_out[(size_t)r * (gamma + 1) + j] = -1;
        for (int j = 0; j < n_acc; ++j) tokens_out[(size_t)r * (gamma + 1) + j] = x[(size_t)r * gamma + j];
        tokens_out[(size_t)r * (gamma + 1) + n_acc] = y;
        n_acc_out[r] = n_acc;
        n_out[r] = n_acc + 1;
        if (corr_margin) corr_margin[r] = mg;
        if (corr_kind) corr_kind[r] = kind;
        free(t); free(z); free(pos);
    }
    return 0;
}

/* Many independent scheduler problems of the same shape, one after another (used by
 * the law tests, which run 10^6 small batches). */
/* Fixed confidence cutoff ([VLLM] "Verify smarter, not longer: the role of confidence
 * scheduling": draft tokens whose confidence is below a fixed cutoff are dropped before
 * verification).  Verification needs a prefix, so request r keeps its leading tokens
 * with c >= threshold: l_r = the first j with c_{r,j} < threshold, minus one (gamma if
 * none).  B and tau as in every mode: B = R + sum l_r, tau = R + sum_r sum_{j<=l_r} a_{r,j}
 * with a the left-to-right product of the confidences. */
int orc_schedule_threshold(int R, int gamma, const float* conf, double threshold, int32_t* ell_out,
                           int32_t* B_out, double* tau_out) {
    if (R < 0 || gamma < 1) return 1;
    double t = (double)R;
    long long B = R;
    for (int r = 0; r < R; ++r) {
        double a = 1.0;
        int l = 0;
        while (l < gamma && (double)conf[(size_t)r * gamma + l] >= threshold) {
            a = a * (double)conf[(size_t)r * gamma + l];
            t += a;
            ++l;
        }
        ell_out[r] = l;
        B += l;
    }
    *B_out = (int32_t)B;
    *tau_out = t;
    return 0;
}

int orc_schedule_many(int nbatch, int R, int gamma, const float* conf, const double* sps,
                      int sps_len, int mode, const float* conf_hist, int fixed_len,
                      int32_t* ell_out) {
    for (int b = 0; b < nbatch; ++b) {
        int32_t B;
        double tau;
        const size_t off = (size_t)b * R * gamma;
        int rc = orc_schedule(R, gamma, conf + off, sps, sps_len, mode,
                              conf_hist ? conf_hist + off : NULL, fixed_len,
                              ell_out + (size_t)b * R, &B, &tau, NULL);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Stage 1, RNN variant — recurrent sequential head.                          */
/* ------------------------------------------------------------------------- */
/* [EXPL] "RNN sequential head": s_k = f(s_{k-1}, E(x_{k-1}), h_k), z_k = U_k + W_o s_k;
 * [KB] §2: f concatenates the recurrent state, the previous token's embedding and the
 * position's backbone hidden state and accumulates the block prefix with a gated
 * update.  The gate's form is not printed; read as the update-gate cell
 *   a       = [s_{k-1}; E[x_{k-1}]] Wse + h_k Wh + b          (2*ns pre-activations)
 *   g       = sigmoid(a[0:ns]),  c = tanh(a[ns:2ns])
 *   s_k     = (1 - g) * s_{k-1} + g * c
 * with s_0 = 0.  The state is kept in the weights' storage type (fp32, or bf16 rounded to
 * nearest-even), so s_k here is the exact cell output rounded once to that type.       */
static double orc_round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    frexp(v, &e);                       /* |v| in [2^(e-1), 2^e) */
    const double ulp = ldexp(1.0, e - 8); /* 8 significant bits */
    return rint(v / ulp) * ulp;         /* default rounding: to nearest, ties to even */
}

static double orc_round_storage(double v, int dtype) {
    return dtype == ORC_BF16 ? orc_round_bf16(v) : (double)(float)v;
}

/* One cell update.  s_prev [ns] (stored values), Wse [(ns+ne), 2ns], Wh [d, 2ns]
 * (dtype_w), bgc [2ns], h row of d elements at h_row (dtype_h) -> s_out [ns]. */
int orc_rnn_cell(int ns, int ne, int d, int dtype_w, int dtype_h, const double* s_prev, int x_prev,
                 const void* E, const void* Wse, const void* Wh, const float* bgc, const void* h,
                 size_t h_row, double* s_out) {
    if (ns < 1 || ne < 0 || d < 0) return 1;
    const int n2 = 2 * ns;
    double* a = (double*)malloc(sizeof(double) * (size_t)n2);
    for (int c = 0; c < n2; ++c) {
        double acc = (double)bgc[c];
        for (int i = 0; i < ns; ++i) acc += s_prev[i] * orc_load(Wse, dtype_w, (size_t)i * n2 + c);
        for (int i = 0; i < ne; ++i)
            acc += orc_load(E, dtype_w, (size_t)x_prev * ne + i) * orc_load(Wse, dtype_w, (size_t)(ns + i) * n2 + c);
        for (int i = 0; i < d; ++i) acc += orc_load(h, dtype_h, h_row + i) * orc_load(Wh, dtype_w, (size_t)i * n2 + c);
        a[c] = acc;
    }
    for (int c = 0; c < ns; ++c) {
        const double g = orc_sigmoid(a[c]);
        const double cand = tanh(a[ns + c]);
        s_out[c] = orc_round_storage((1.0 - g) * s_prev[c] + g * cand, dtype_w);
    }
    free(a);
    return 0;
}

/* One draft position given its factor row: x = Gumbel-max draw of softmax(z) (stream 0 at
 * `position`), lse, logq = z_x - lse, and the runner-up / key margin of the draw. */
int orc_draft_row(int V, int rank, int dtype_u, int dtype_w, const void* U_row, const double* arow,
                  const void* W2, double temperature, uint64_t seed, uint64_t req_id, uint64_t round,
                  uint32_t position, int32_t* x_out, double* lse_out, double* logq_out, int32_t* runner_up,
                  double* margin) {
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    orc_row_logits(V, rank, dtype_u, dtype_w, U_row, 0, arow, W2, temperature, z);
    const double lse = orc_logsumexp(z, V);
    int ru = -1;
    double mg = 0.0;
    const int x = orc_gumbel_argmax(z, NULL, V, seed, req_id, round, ORC_STREAM_DRAFT, position, &ru, &mg);
    *x_out = x;
    *lse_out = lse;
    *logq_out = z[x] - lse;
    if (runner_up) *runner_up = ru;
    if (margin) *margin = mg;
    free(z);
    return 0;
}

/* Confidence of the recurrent head for given states: c[r,k] = sigmoid(kappa (w_h .
 * h[r,k-1,:] + w_s . state[r,k-1,:] + b) / T_k), conf_w = [w_h (d); w_s (ns)]. */
int orc_rnn_confidence(int R, int gamma, int d, int ns, int dtype_h, const void* h, const double* state,
                       const float* conf_w, double conf_b, double conf_logit_scale, const float* conf_temp,
                       double* conf_out) {
    for (int r = 0; r < R; ++r)
        for (int k = 1; k <= gamma; ++k) {
            const size_t row = (size_t)r * gamma + (k - 1);
            double s_h = 0.0, s_s = 0.0;
            for (int i = 0; i < d; ++i) s_h += (double)conf_w[i] * orc_load(h, dtype_h, row * (size_t)d + i);
            for (int i = 0; i < ns; ++i) s_s += (double)conf_w[d + i] * state[row * (size_t)ns + i];
            conf_out[row] = orc_sigmoid(conf_logit_scale * (s_h + s_s + conf_b) / (double)conf_temp[k - 1]);
        }
    return 0;
}

/* The draft loop with the recurrent head, per request r (x_0 = anchor, s_0 = 0):
 *   s_k = cell(s_{k-1}, x_{k-1}, h[r,k-1,:]);  z = (U[r,k-1,:] + s_k W_o) / T;
 *   x_k, lse_k, logq_k as for the Markov head (stream 0 at position k);
 *   c_k = sigmoid(kappa (w_h . h[r,k-1,:] + w_s . s_k + b) / T_k)  (the state takes the
 *   place of the Markov head's factor row in the confidence input).
 * state_out [R,gamma,ns]: the stored states s_1..s_gamma. */
int orc_rnn_draft(int R, int gamma, int V, int ns, int ne, int d, int dtype_u, int dtype_w, int dtype_h,
                  const void* U, const void* E, const void* Wse, const void* Wh, const float* bgc,
                  const void* Wo, const void* h, const float* conf_w, double conf_b, double conf_logit_scale,
                  const float* conf_temp, double temperature, const int32_t* x0, const int64_t* req_id,
                  uint64_t seed, uint64_t round, int32_t* x_out, double* logq_out, double* lse_out,
                  double* conf_out, double* state_out, int32_t* runner_up_out, double* margin_out,
                  int nthreads) {
    if (R < 0 || gamma < 1 || V < 1 || ns < 1 || ne < 0 || d < 0 || temperature <= 0.0) return 1;
    int nt = orc_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int r = 0; r < R; ++r) {
        double* s = (double*)calloc((size_t)ns, sizeof(double));
        double* sn = (double*)malloc(sizeof(double) * (size_t)ns);
        int x_prev = x0[r];
        for (int k = 1; k <= gamma; ++k) {
            const size_t row = (size_t)r * gamma + (k - 1);
            orc_rnn_cell(ns, ne, d, dtype_w, dtype_h, s, x_prev, E, Wse, Wh, bgc, h, row * (size_t)d, sn);
            memcpy(s, sn, sizeof(double) * (size_t)ns);
            int32_t xk, ru;
            double lse, logq, mg;
            orc_draft_row(V, ns, dtype_u, dtype_w, (const char*)U + row * (size_t)V * (dtype_u == ORC_BF16 ? 2 : 4),
                          s, Wo, temperature, seed, (uint64_t)req_id[r], round, (uint32_t)k, &xk, &lse, &logq,
                          &ru, &mg);
            double s_h = 0.0;
            for (int i = 0; i < d; ++i) s_h += (double)conf_w[i] * orc_load(h, dtype_h, row * (size_t)d + i);
            double s_s = 0.0;
            for (int i = 0; i < ns; ++i) s_s += (double)conf_w[d + i] * s[i];
            const double logit = conf_logit_scale * (s_h + s_s + conf_b);
            x_out[row] = xk;
            logq_out[row] = logq;
            lse_out[row] = lse;
            conf_out[row] = orc_sigmoid(logit / (double)conf_temp[k - 1]);
            if (state_out) memcpy(state_out + row * (size_t)ns, s, sizeof(double) * (size_t)ns);
            if (runner_up_out) runner_up_out[row] = ru;
            if (margin_out) margin_out[row] = mg;
            x_prev = xk;
        }
        free(s);
        free(sn);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Sequential temperature scaling (STS) of the confidence head.               */
/* ------------------------------------------------------------------------- */
/* [EXPL] "Sequential temperature scaling": c_k = sigmoid(z_k / T_k); calibrate position 1,
 * freeze it, then calibrate the cumulative survival through position 2, and so on left
 * to right.  [FR] §3.2: a per-position temperature search minimising the expected
 * calibration error of the cumulative product prod_{i<=k} c_i on held-out data.
 * Held-out sample n: confidence logits z[n, 1..gamma] (before the temperature) and the
 * number of accepted drafts L_n when the whole block was verified, so the survival
 * outcome at position k is 1[L_n >= k].
 * ECE over M equal-width bins of [0,1] (bin of p: min(floor(p M), M-1)):
 *   ECE = sum_b |sum_{n in b} (p_n - o_n)| / N
 * (the bin-weighted gap |mean p - mean o| of the usual definition).  T_k is the grid
 * temperature with the smallest ECE of p_n = prod_{i<k} sigmoid(z_{n,i}/T_i) *
 * sigmoid(z_{n,k}/T), the first one on ties.                                */
static int orc_bin(double p, int M) {
    int b = (int)floor(p * M);
    if (b < 0) b = 0;
    if (b > M - 1) b = M - 1;
    return b;
}

/* ECE at position k (1-based) for temperature T, given the frozen T_1..T_{k-1}. */
double orc_sts_ece(int N, int gamma, const float* z, const int32_t* acc_len, const double* T_prev, int k,
                   double T, int M) {
    double* gap = (double*)calloc((size_t)M, sizeof(double));
    for (int n = 0; n < N; ++n) {
        double p = 1.0;
        for (int i = 1; i < k; ++i) p *= orc_sigmoid((double)z[(size_t)n * gamma + (i - 1)] / T_prev[i - 1]);
        p *= orc_sigmoid((double)z[(size_t)n * gamma + (k - 1)] / T);
        const double o = acc_len[n] >= k ? 1.0 : 0.0;
        gap[orc_bin(p, M)] += p - o;
    }
    double e = 0.0;
    for (int b = 0; b < M; ++b) e += fabs(gap[b]);
    free(gap);
    return e / N;
}

int orc_sts_fit(int N, int gamma, const float* z, const int32_t* acc_len, const double* grid, int G, int M,
                double* T_out, double* ece_out) {
    if (N < 1 || gamma < 1 || G < 1 || M < 1) return 1;
    for (int k = 1; k <= gamma; ++k) {
        int best = 0;
        double best_e = INFINITY;
        for (int g = 0; g < G; ++g) {
            const double e = orc_sts_ece(N, gamma, z, acc_len, T_out, k, grid[g], M);
            if (e < best_e) {
                best_e = e;
                best = g;
            }
        }
        T_out[k - 1] = grid[best];
        ece_out[k - 1] = best_e;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Acceptance-overlap diagnostic.                                             */
/* ------------------------------------------------------------------------- */
/* For request r and drafted position j (1-based) the expected acceptance of the
 * draft token is the overlap of the two distributions ([EXPL] "Total variation
 * label"; [EXPL] "Speculative sampling in one picture"):
 *   c*_j = sum_v min(q_j(v), p_j(v)) = 1 - (1/2) ||q_j - p_j||_1
 * with q_j = softmax((U[r,j-1,:] + W1[x_{j-1},:] W2)/T) the draft distribution at
 * position j (x_0 the anchor) and p_j = softmax(target[r,j-1,:]/T) the target
 * distribution that verifies position j.  Positions j <= n_r are evaluated, n_r =
 * ell[r] (ell == NULL: every position); the others are set to NaN. */
int orc_acceptance_overlap(int R, int gamma, int V, int rank, int dtype_t, int dtype_u, int dtype_w,
                           const void* target, const void* U, const void* W1, const void* W2,
                           const int32_t* x0, const int32_t* x, const int32_t* ell,
                           double temperature, double* out, int nthreads) {
    if (R < 0 || gamma < 1 || V < 1 || rank < 1 || temperature <= 0.0) return 1;
    if (ell)
        for (int r = 0; r < R; ++r)
            if (ell[r] < 0 || ell[r] > gamma) return 1;
    int nt = orc_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int r = 0; r < R; ++r) {
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        double* t = (double*)malloc(sizeof(double) * (size_t)V);
        const int n = ell ? ell[r] : gamma;
        for (int j = 1; j <= gamma; ++j) {
            const size_t row = (size_t)r * gamma + (j - 1);
            if (j > n) {
                out[row] = NAN;
                continue;
            }
            const int xprev = (j == 1) ? x0[r] : x[(size_t)r * gamma + (j - 2)];
            orc_draft_logits(V, rank, dtype_u, dtype_w, U, row * (size_t)V, W1, W2, xprev, temperature, z);
            const double lq = orc_logsumexp(z, V);
            const size_t trow = ((size_t)r * (gamma + 1) + (j - 1)) * (size_t)V;
            for (int v = 0; v < V; ++v) t[v] = orc_load(target, dtype_t, trow + v) / temperature;
            const double lt = orc_logsumexp(t, V);
            double c = 0.0;
            for (int v = 0; v < V; ++v) {
                const double q = exp(z[v] - lq), p = exp(t[v] - lt);
                c += q < p ? q : p;
            }
            out[row] = c;
        }
        free(z);
        free(t);
    }
    return 0;
}

int orc_max_threads(void) { return orc_threads(0); }
