/*
 * retention_oracle.c -- plain, slow, fp64 CPU oracle of the RetNet retention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library; both sides only receive the same seeded inputs.
 *
 * Sources (page title, then section / equation on that page):
 *   [RN2]  "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）"
 *          sections "Retention" (eqs. (1)-(7)), "門控多尺度 Retention",
 *          "Retention Score 歸一化", "訓練/推理" paragraphs.
 *   [RVW]  "[論文レビュー] Retentive Network: A Successor to Transformer for Large
 *          Language Models", ABSTRACT (three paradigms: parallel, recurrent,
 *          chunkwise recurrent).
 *
 * The formulas of [RN2] were lost when the page was extracted to text; the
 * surrounding sentences survive.  Every function below states the reading it
 * implements.  All readings are the plainest ones consistent with that text:
 *   - decay matrix  D[n][m] = gamma^(n-m) for n >= m, 0 otherwise (0-based);
 *   - parallel form (eq.5):  O = (Q K^T (.) D) V;
 *   - recurrent form (eq.6): S_n = gamma S_{n-1} + K_n^T V_n,  o_n = Q_n S_n
 *     (the output reads the state after the update);
 *   - chunkwise form (eq.7), chunk length B, chunk i covering rows iB..iB+B-1:
 *       R_i  = K_[i]^T (V_[i] (.) zeta) + gamma^B R_{i-1},  zeta_r = gamma^(B-1-r)
 *       O_[i] = (Q_[i] K_[i]^T (.) D_B) V_[i] + (Q_[i] R_{i-1}) (.) xi,  xi_j = gamma^(j+1)
 *     with D_B the B x B block of D and R_{-1} the incoming state (zero by default);
 *   - real-valued inputs, so the conjugate transpose of eq.(4) is a plain transpose;
 *   - Q and K arrive already position-rotated (the xPos factor of eqs.(2)-(3) is
 *     absorbed into the inputs), so no rotation happens here.
 *
 * Layouts (all row-major, contiguous, fp64):
 *   q, k : [b][H][N][dk]      v, o : [b][H][N][dv]
 *   state: [b][H][dk][dv]     gamma: [H]
 *   y    : [b][H][N][dv]      g, out: [b][N][H*dv]   (token-major, like X W_G)
 *
 * Every function returns 0 on success and -1 on an argument it cannot handle.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_NORM_SCALE 1u  /* QK^T / sqrt(dk)                              */
#define ORACLE_NORM_DECAY 2u  /* row n of D divided by sqrt(sum_m D[n][m])    */
#define ORACLE_NORM_ROWSUM 4u /* R row n divided by max(|sum_m R[n][m]|, 1)   */

/* gamma^e for an integer e >= 0, with 0^0 = 1 (C99 pow guarantees pow(x,0)=1). */
static double gpow(double gamma, long e) { return pow(gamma, (double)e); }

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += a[i] * b[i];
    return s;
}

/*
 * Parallel form, [RN2] "Retention" 1) (eq.5, Fig.3a), with the optional score
 * normalisations of [RN2] "Retention Score 歸一化":
 *   R[n][m] = (q_n . k_m) [/ sqrt(dk)] * D[n][m] [/ sqrt(sum_{i<=n} D[n][i])]
 *   R[n][.] /= max(|sum_m R[n][m]|, 1)            (ROWSUM flag)
 *   O = R V
 * The row sum of D is accumulated term by term (its definition), not from a
 * closed form, so that the closed form can serve as an independent check.
 */
int oracle_parallel(const double* q, const double* k, const double* v, double* o,
                    int b, int H, int N, int dk, int dv, const double* gamma,
                    unsigned flags) {
    if (b < 0 || H < 0 || N < 0 || dk <= 0 || dv <= 0) return -1;
    if (N == 0 || b == 0 || H == 0) return 0;
    double* R = (double*)malloc(sizeof(double) * (size_t)N * (size_t)N);
    if (!R) return -1;
    for (int bi = 0; bi < b; ++bi)
        for (int h = 0; h < H; ++h) {
            size_t u = (size_t)bi * H + h;
            const double* Q = q + u * (size_t)N * dk;
            const double* K = k + u * (size_t)N * dk;
            const double* V = v + u * (size_t)N * dv;
            double* O = o + u * (size_t)N * dv;
            double g = gamma[h];
            for (int n = 0; n < N; ++n) {
                double drow = 0.0; /* sum_m D[n][m] */
                for (int m = 0; m <= n; ++m) drow += gpow(g, n - m);
                for (int m = 0; m < N; ++m) {
                    double r = 0.0;
                    if (m <= n) {
                        double s = dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk);
                        if (flags & ORACLE_NORM_SCALE) s /= sqrt((double)dk);
                        double d = gpow(g, n - m);
                        if (flags & ORACLE_NORM_DECAY) d /= sqrt(drow);
                        r = s * d;
                    }
                    R[(size_t)n * N + m] = r;
                }
                if (flags & ORACLE_NORM_ROWSUM) {
                    double rs = 0.0;
                    for (int m = 0; m < N; ++m) rs += R[(size_t)n * N + m];
                    double den = fabs(rs) > 1.0 ? fabs(rs) : 1.0;
                    for (int m = 0; m < N; ++m) R[(size_t)n * N + m] /= den;
                }
            }
            for (int n = 0; n < N; ++n) {
                double* on = O + (size_t)n * dv;
                for (int c = 0; c < dv; ++c) on[c] = 0.0;
                for (int m = 0; m < N; ++m) {
                    double r = R[(size_t)n * N + m];
                    if (r == 0.0) continue;
                    const double* vm = V + (size_t)m * dv;
                    for (int c = 0; c < dv; ++c) on[c] += r * vm[c];
                }
            }
        }
    free(R);
    return 0;
}

/*
 * Recurrent form, [RN2] "Retention" 2) (eq.6, Fig.3b):
 *   S_n = gamma S_{n-1} + k_n^T v_n,   o_n = q_n S_n.
 * state_in (nullable -> zero) is S_{-1}; state_out (nullable) receives S_{N-1}.
 */
int oracle_recurrent(const double* q, const double* k, const double* v, double* o,
                     int b, int H, int N, int dk, int dv, const double* gamma,
                     const double* state_in, double* state_out) {
    if (b < 0 || H < 0 || N < 0 || dk <= 0 || dv <= 0) return -1;
    size_t SS = (size_t)dk * dv;
    double* S = (double*)malloc(sizeof(double) * SS);
    if (!S) return -1;
    for (int bi = 0; bi < b; ++bi)
        for (int h = 0; h < H; ++h) {
            size_t u = (size_t)bi * H + h;
            const double* Q = q + u * (size_t)N * dk;
            const double* K = k + u * (size_t)N * dk;
            const double* V = v + u * (size_t)N * dv;
            double* O = o + u * (size_t)N * dv;
            double g = gamma[h];
            if (state_in) memcpy(S, state_in + u * SS, sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            for (int n = 0; n < N; ++n) {
                const double* qn = Q + (size_t)n * dk;
                const double* kn = K + (size_t)n * dk;
                const double* vn = V + (size_t)n * dv;
                for (int a = 0; a < dk; ++a)
                    for (int c = 0; c < dv; ++c)
                        S[(size_t)a * dv + c] = g * S[(size_t)a * dv + c] + kn[a] * vn[c];
                double* on = O + (size_t)n * dv;
                for (int c = 0; c < dv; ++c) on[c] = 0.0;
                for (int a = 0; a < dk; ++a)
                    for (int c = 0; c < dv; ++c) on[c] += qn[a] * S[(size_t)a * dv + c];
            }
            if (state_out) memcpy(state_out + u * SS, S, sizeof(double) * SS);
        }
    free(S);
    return 0;
}

/*
 * One decode step of the recurrent form, [RN2] "Retention" 2) (eq.6), and the
 * inference paragraph (O(1) per token).  q,k:[b][H][dk] v:[b][H][dv];
 * state:[b][H][dk][dv] is read and overwritten with the updated S; o:[b][H][dv]
 * is read from the updated state.
 */
int oracle_recurrent_step(const double* q, const double* k, const double* v,
                          double* state, double* o, int b, int H, int dk, int dv,
                          const double* gamma) {
    if (b < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    return oracle_recurrent(q, k, v, o, b, H, 1, dk, dv, gamma, state, state);
}

/*
 * Chunkwise recurrent form, [RN2] "Retention" 3) (eq.7): inside a chunk the
 * parallel form, across chunks the recurrent state R.  Literal steps for each
 * chunk i (0-based, rows iB..iB+B-1, j and r index rows inside the chunk):
 *   inner[j]  = sum_{r<=j} (q_j . k_r) gamma^(j-r) v_r
 *   cross[j]  = (q_j R_{i-1}) * xi_j,               xi_j   = gamma^(j+1)
 *   O[iB+j]   = inner[j] + cross[j]
 *   R_i       = sum_r zeta_r k_r^T v_r + gamma^B R_{i-1},  zeta_r = gamma^(B-1-r)
 * Requires N % chunk == 0 (a ragged final chunk is not read as anything).
 */
int oracle_chunkwise(const double* q, const double* k, const double* v, double* o,
                     int b, int H, int N, int dk, int dv, int chunk,
                     const double* gamma, const double* state_in, double* state_out) {
    if (b < 0 || H < 0 || N < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return -1;
    if (N % chunk != 0) return -1;
    int B = chunk;
    size_t SS = (size_t)dk * dv;
    double* R = (double*)malloc(sizeof(double) * SS);
    double* Rn = (double*)malloc(sizeof(double) * SS);
    double* xi = (double*)malloc(sizeof(double) * (size_t)B);
    double* zeta = (double*)malloc(sizeof(double) * (size_t)B);
    if (!R || !Rn || !xi || !zeta) { free(R); free(Rn); free(xi); free(zeta); return -1; }
    for (int bi = 0; bi < b; ++bi)
        for (int h = 0; h < H; ++h) {
            size_t u = (size_t)bi * H + h;
            const double* Q = q + u * (size_t)N * dk;
            const double* K = k + u * (size_t)N * dk;
            const double* V = v + u * (size_t)N * dv;
            double* O = o + u * (size_t)N * dv;
            double g = gamma[h];
            double gB = gpow(g, B);
            for (int j = 0; j < B; ++j) { xi[j] = gpow(g, j + 1); zeta[j] = gpow(g, B - 1 - j); }
            if (state_in) memcpy(R, state_in + u * SS, sizeof(double) * SS);
            else memset(R, 0, sizeof(double) * SS);
            for (int i = 0; i < N / B; ++i) {
                const double* Qi = Q + (size_t)i * B * dk;
                const double* Ki = K + (size_t)i * B * dk;
                const double* Vi = V + (size_t)i * B * dv;
                double* Oi = O + (size_t)i * B * dv;
                for (int j = 0; j < B; ++j) {
                    double* oj = Oi + (size_t)j * dv;
                    const double* qj = Qi + (size_t)j * dk;
                    for (int c = 0; c < dv; ++c) oj[c] = 0.0;
                    /* inner-chunk parallel part */
                    for (int r = 0; r <= j; ++r) {
                        double p = dot(qj, Ki + (size_t)r * dk, dk) * gpow(g, j - r);
                        const double* vr = Vi + (size_t)r * dv;
                        for (int c = 0; c < dv; ++c) oj[c] += p * vr[c];
                    }
                    /* cross-chunk part from the incoming state */
                    for (int a = 0; a < dk; ++a) {
                        double qa = qj[a] * xi[j];
                        const double* Ra = R + (size_t)a * dv;
                        for (int c = 0; c < dv; ++c) oj[c] += qa * Ra[c];
                    }
                }
                /* state update */
                for (size_t e = 0; e < SS; ++e) Rn[e] = gB * R[e];
                for (int r = 0; r < B; ++r) {
                    const double* kr = Ki + (size_t)r * dk;
                    const double* vr = Vi + (size_t)r * dv;
                    for (int a = 0; a < dk; ++a) {
                        double ka = kr[a] * zeta[r];
                        double* Ra = Rn + (size_t)a * dv;
                        for (int c = 0; c < dv; ++c) Ra[c] += ka * vr[c];
                    }
                }
                double* t = R; R = Rn; Rn = t;
            }
            if (state_out) memcpy(state_out + u * SS, R, sizeof(double) * SS);
        }
    free(R); free(Rn); free(xi); free(zeta);
    return 0;
}

/*
 * Brute-force definition, no matrices: o_n[c] = sum_{m<=n} gamma^(n-m) (q_n . k_m) v_m[c].
 * This is eq.(5) without normalisation written as a single sum per output entry.
 */
int oracle_brute(const double* q, const double* k, const double* v, double* o,
                 int b, int H, int N, int dk, int dv, const double* gamma) {
    if (b < 0 || H < 0 || N < 0 || dk <= 0 || dv <= 0) return -1;
    for (int bi = 0; bi < b; ++bi)
        for (int h = 0; h < H; ++h) {
            size_t u = (size_t)bi * H + h;
            for (int n = 0; n < N; ++n)
                for (int c = 0; c < dv; ++c) {
                    double acc = 0.0;
                    for (int m = 0; m <= n; ++m) {
                        double qk = 0.0;
                        for (int a = 0; a < dk; ++a)
                            qk += q[(u * N + n) * dk + a] * k[(u * N + m) * dk + a];
                        acc += gpow(gamma[h], n - m) * qk * v[(u * N + m) * dv + c];
                    }
                    o[(u * N + n) * dv + c] = acc;
                }
        }
    return 0;
}

/*
 * Gated multi-scale retention epilogue, [RN2] "門控多尺度 Retention":
 *   Y = GroupNorm_h(head outputs): one group per (token, head) over its dv
 *   channels (each head normalised separately), biased variance, eps inside
 *   the square root; optional per-channel affine (weight, bias over H*dv
 *   channels; NULL means identity);
 *   out = swish(G) (.) Y,  swish(x) = x * sigmoid(x)  (the [RZL17] gate, beta=1).
 * The output projection W_O is not part of this step.
 * y:[b][H][N][dv] (head-major, as the retention forms produce it);
 * g, out:[b][N][H*dv] (token-major, as X W_G is laid out).
 */
int oracle_msr_epilogue(const double* y, const double* g, double* out, int b, int H,
                        int N, int dv, double eps, const double* weight,
                        const double* bias) {
    if (b < 0 || H < 0 || N < 0 || dv <= 0 || eps < 0.0) return -1;
    size_t C = (size_t)H * dv;
    for (int bi = 0; bi < b; ++bi)
        for (int n = 0; n < N; ++n)
            for (int h = 0; h < H; ++h) {
                const double* yr = y + (((size_t)bi * H + h) * N + n) * dv;
                double mu = 0.0;
                for (int c = 0; c < dv; ++c) mu += yr[c];
                mu /= dv;
                double var = 0.0;
                for (int c = 0; c < dv; ++c) var += (yr[c] - mu) * (yr[c] - mu);
                var /= dv;
                double inv = 1.0 / sqrt(var + eps);
                for (int c = 0; c < dv; ++c) {
                    size_t ch = (size_t)h * dv + c;
                    double yn = (yr[c] - mu) * inv;
                    if (weight) yn *= weight[ch];
                    if (bias) yn += bias[ch];
                    size_t gi = ((size_t)bi * N + n) * C + ch;
                    double gv = g[gi];
                    double sw = gv / (1.0 + exp(-gv));
                    out[gi] = sw * yn;
                }
            }
    return 0;
}

/*
 * Gradient of the chunkwise form.  [RN2] "訓練/推理" says training runs the
 * parallel and chunkwise forms; the pages print no backward pass, so this is the
 * exact derivative of what eq.(7) computes.  For every chunk length eq.(7) gives,
 * per (batch, head), with S0 the incoming state (zero when state_in is NULL):
 *   o_n     = gamma^(n+1) q_n S0 + sum_{m<=n} gamma^(n-m) (q_n . k_m) v_m
 *   S_final = gamma^N S0 + sum_m gamma^(N-1-m) k_m^T v_m
 * and the scalar  L = sum_n dout_n . o_n + <dstate_out, S_final>  (dstate_out NULL
 * means zero).  Its partial derivatives, written out entry by entry:
 *   dq_n[a] = sum_{m<=n} gamma^(n-m) (dout_n . v_m) k_m[a]
 *             + gamma^(n+1) sum_c dout_n[c] S0[a][c]
 *   dk_m[a] = sum_{n>=m} gamma^(n-m) (dout_n . v_m) q_n[a]
 *             + gamma^(N-1-m) sum_c dstate_out[a][c] v_m[c]
 *   dv_m[c] = sum_{n>=m} gamma^(n-m) (q_n . k_m) dout_n[c]
 *             + gamma^(N-1-m) sum_a k_m[a] dstate_out[a][c]
 *   dS0[a][c] = sum_n gamma^(n+1) q_n[a] dout_n[c] + gamma^N dstate_out[a][c]
 * Layouts as above; dout like o, dq/dk like q, dv like v, dstate_in and
 * dstate_out like state.  dstate_in may be NULL (not computed).
 */
int oracle_chunkwise_backward(const double* q, const double* k, const double* v,
                              const double* dout, const double* state_in,
                              const double* dstate_out, double* dq, double* dk, double* dv,
                              double* dstate_in, int b, int H, int N, int dk_, int dv_,
                              const double* gamma) {
    if (b < 0 || H < 0 || N < 0 || dk_ <= 0 || dv_ <= 0) return -1;
    size_t SS = (size_t)dk_ * dv_;
    for (int bi = 0; bi < b; ++bi)
        for (int h = 0; h < H; ++h) {
            size_t u = (size_t)bi * H + h;
            const double* Q = q + u * (size_t)N * dk_;
            const double* K = k + u * (size_t)N * dk_;
            const double* V = v + u * (size_t)N * dv_;
            const double* DO = dout + u * (size_t)N * dv_;
            const double* S0 = state_in ? state_in + u * SS : NULL;
            const double* DS = dstate_out ? dstate_out + u * SS : NULL;
            double g = gamma[h];
            for (int n = 0; n < N; ++n) {
                const double* don = DO + (size_t)n * dv_;
                double* dqn = dq + (u * N + n) * dk_;
                for (int a = 0; a < dk_; ++a) dqn[a] = 0.0;
                for (int m = 0; m <= n; ++m) {
                    double w = gpow(g, n - m) * dot(don, V + (size_t)m * dv_, dv_);
                    const double* km = K + (size_t)m * dk_;
                    for (int a = 0; a < dk_; ++a) dqn[a] += w * km[a];
                }
                if (S0) {
                    double f = gpow(g, n + 1);
                    for (int a = 0; a < dk_; ++a)
                        dqn[a] += f * dot(don, S0 + (size_t)a * dv_, dv_);
                }
            }
            for (int m = 0; m < N; ++m) {
                const double* km = K + (size_t)m * dk_;
                const double* vm = V + (size_t)m * dv_;
                double* dkm = dk + (u * N + m) * dk_;
                double* dvm = dv + (u * N + m) * dv_;
                for (int a = 0; a < dk_; ++a) dkm[a] = 0.0;
                for (int c = 0; c < dv_; ++c) dvm[c] = 0.0;
                for (int n = m; n < N; ++n) {
                    double gd = gpow(g, n - m);
                    const double* qn = Q + (size_t)n * dk_;
                    const double* don = DO + (size_t)n * dv_;
                    double wk = gd * dot(don, vm, dv_);
                    double wv = gd * dot(qn, km, dk_);
                    for (int a = 0; a < dk_; ++a) dkm[a] += wk * qn[a];
                    for (int c = 0; c < dv_; ++c) dvm[c] += wv * don[c];
                }
                if (DS) {
                    double f = gpow(g, N - 1 - m);
                    for (int a = 0; a < dk_; ++a)
                        dkm[a] += f * dot(DS + (size_t)a * dv_, vm, dv_);
                    for (int c = 0; c < dv_; ++c) {
                        double s = 0.0;
                        for (int a = 0; a < dk_; ++a) s += km[a] * DS[(size_t)a * dv_ + c];
                        dvm[c] += f * s;
                    }
                }
            }
            if (dstate_in) {
                double* D0 = dstate_in + u * SS;
                for (int a = 0; a < dk_; ++a)
                    for (int c = 0; c < dv_; ++c) {
                        double s = DS ? gpow(g, N) * DS[(size_t)a * dv_ + c] : 0.0;
                        for (int n = 0; n < N; ++n)
                            s += gpow(g, n + 1) * Q[(size_t)n * dk_ + a] * DO[(size_t)n * dv_ + c];
                        D0[(size_t)a * dv_ + c] = s;
                    }
            }
        }
    return 0;
}

/*
 * RG-LRU scan of the Griffin page ("Griffin ：將門控線性循環與局部注意力混合以實現
 * 高效的語言模型", section "實門線性循環單元 (RG-LRU)", its four equations), a second
 * linear recurrence.  Per batch row, channel d and step t, from the gate
 * pre-activations (the two projections W_a x_t + b_a and W_x x_t + b_x are plain
 * matrix products outside this step):
 *   r_t = sigmoid(gate_a_t)             recurrence gate
 *   i_t = sigmoid(gate_x_t)             input gate
 *   a   = sigmoid(lambda_d)             so 0 <= a <= 1
 *   a_t = a^(c r_t)                     (the page fixes c = 8)
 *   h_t = a_t h_{t-1} + sqrt(1 - a_t^2) (i_t x_t),   y_t = h_t
 * with h_{-1} = h0 (NULL means zero).  Written as the definition, with pow; the page
 * evaluates a_t in log space, which is the same number.
 * x, gate_a, gate_x, y: [b][T][D]; lambda: [D]; h0, h_last: [b][D] (h_last nullable).
 */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

int oracle_rglru(const double* x, const double* gate_a, const double* gate_x,
                 const double* lambda_, const double* h0, double* y, double* h_last,
                 int b, int T, int D, double c) {
    if (b < 0 || T < 0 || D <= 0 || !(c >= 0.0)) return -1;
    for (int bi = 0; bi < b; ++bi)
        for (int d = 0; d < D; ++d) {
            double h = h0 ? h0[(size_t)bi * D + d] : 0.0;
            double a = sigmoid(lambda_[d]);
            for (int t = 0; t < T; ++t) {
                size_t e = ((size_t)bi * T + t) * D + d;
                double r = sigmoid(gate_a[e]);
                double i = sigmoid(gate_x[e]);
                double at = pow(a, c * r);
                h = at * h + sqrt(1.0 - at * at) * (i * x[e]);
                y[e] = h;
            }
            if (h_last) h_last[(size_t)bi * D + d] = h;
        }
    return 0;
}

/*
 * xPos rotation, [RN2] "Retention", eqs.(2)-(3) (their formulas were lost; the prose
 * survives): Q_n becomes Q_n e^{i n theta} and K_m becomes K_m e^{i m theta}, so that
 * the score of eq.(4), taken with the conjugate transpose, depends on n - m only (a
 * relative position embedding).  Reading for real inputs: the pair of coordinates
 * (2j, 2j+1) is one complex number z = x_{2j} + i x_{2j+1}, multiplied by
 * e^{i p theta_j} at position p = pos0 + n:
 *   out_{2j}   = x_{2j} cos(p theta_j) - x_{2j+1} sin(p theta_j)
 *   out_{2j+1} = x_{2j} sin(p theta_j) + x_{2j+1} cos(p theta_j)
 * x, out: [b][H][N][d] (d even), theta: [d/2].
 */
int oracle_xpos_rotate(const double* x, double* out, int b, int H, int N, int d,
                       const double* theta, long long pos0) {
    if (b < 0 || H < 0 || N < 0 || d <= 0 || d % 2 != 0) return -1;
    for (long long row = 0; row < (long long)b * H * N; ++row) {
        long long p = pos0 + row % N;
        const double* xr = x + row * d;
        double* orow = out + row * d;
        for (int j = 0; j < d / 2; ++j) {
            double ang = (double)p * theta[j];
            double cs = cos(ang), sn = sin(ang);
            double x0 = xr[2 * j], x1 = xr[2 * j + 1];
            orow[2 * j] = x0 * cs - x1 * sn;
            orow[2 * j + 1] = x0 * sn + x1 * cs;
        }
    }
    return 0;
}
