/*
 * ORACLE for the exact speculative verify path of a hybrid gated-delta-net
 * (GDN) / attention decoder.  TEST INFRASTRUCTURE ONLY: the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark call it; the product
 * path never does.  It shares no code, header or constant table with the CUDA
 * library.
 *
 * Plain, slow, obviously-correct C.  Every floating-point operation runs in
 * double precision; a value is rounded to bf16 (round to nearest, ties to
 * even) exactly where the model stores a bf16 tensor: projection outputs,
 * beta and gate, GDN output o, attention output, gated attention output,
 * SwiGLU product, residual stream, RMSNorm output and the KV cache.  The GDN
 * state is kept in double.  Logits are left in double.
 *
 * Sources.  The pages describe a recipe that makes speculative decoding of a
 * GDN/attention hybrid bit-exact:
 *   [post]   "Follow-up to my earlier post on Qwen3.8-27B decode speed"
 *            (r/LocalLLaMA post, feedman.me copy): verify must step the GDN
 *            recurrence through the decode kernel, with beta in the decode
 *            dtype rather than fp32, and must run attention as one decode row
 *            per draft position; outputs are compared token id by token id
 *            and logprob by logprob against decoding without speculation.
 *   [card]   "Qwen3.8-27B Bit-Exact Spec-Decode 1x RTX PRO 6000 SGLang"
 *            (recipe card), summary: the same two verify changes plus a
 *            small-M GEMM route that yields the same bits.
 * The pages name the GDN recurrence but never print it; the oracle uses the
 * standard gated delta rule
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T ,   o_t = S_t q_t
 * with S_t of shape [dv][dk].  Because the method's whole claim is that
 * verifying k draft tokens gives exactly the bits of decoding them one at a
 * time, the oracle has NO verify code at all: verify(k) is k calls of
 * orc_decode_token.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - decoder layer = x + mixer(rmsnorm(x)), then h + swiglu_mlp(rmsnorm(h));
 *   - rmsnorm(x) = x / sqrt(mean(x^2) + eps) * (1 + w);
 *   - GDN input projection columns = [q | k | v | b | a]; q and k are
 *     L2-normalised per head (x / sqrt(sum x^2 + 1e-6)); beta = sigmoid(b),
 *     gate = exp(-softplus(a)), both rounded to bf16 before use; no q scale;
 *   - the complete GDN layer (optional, off in the configurations the pages'
 *     measurements concern) adds, as in gated-delta-net decoders: fewer q/k
 *     heads than v heads (v head h reads q/k head h / (Hv/Hk)); a depthwise
 *     causal convolution of width Kc with SiLU over the q|k|v channels, whose
 *     state is the Kc-1 previous inputs; and an output RMSNorm per v head
 *     gated by silu(z), z a further Hv*dv projection columns placed after v,
 *     with the (1 + w) gain of the block's other norms;
 *   - attention input projection columns = [q | gate | k | v]; no RoPE;
 *     scale 1/sqrt(hd); output rounded to bf16, then times sigmoid(gate);
 *   - softplus(x) = x for x > 20, else log1p(exp(x));
 *   - argmax ties go to the lowest index; the accepted count is the number
 *     of leading drafts equal to the target's argmax.
 *
 * Pins (tests that do not run this code against itself): bf16 rounding is
 * checked exhaustively over all float bit patterns against an independent
 * bracket-and-compare rounding; GEMM against one-hot closed forms and exact
 * integer products; the GDN step against the 1x1 closed form, a brute-force
 * 2x2 case in exact rationals, and the delta-rule invariants; attention
 * against L=1, identical keys, a dominant key and scipy's softmax; RMSNorm,
 * SwiGLU and the gates against constant-vector closed forms and scipy; the
 * causal convolution against numpy's convolution, its impulse response and
 * its state; the gated norm against closed forms; grouped heads against the
 * ungrouped step on repeated q/k; the complete GDN layer's column layout
 * against repeated projection rows, a zeroed z block and a numpy composition.
 * orc_decode_token composes pinned functions; its composition (column blocks,
 * gate, MLP layout, both residuals) is pinned against numpy compositions of
 * the pinned parts.
 *
 * Second evaluation.  Compiled with ORC_F32 defined, every accumulation and
 * every elementwise evaluation runs in single precision instead (the type
 * `real` below; the GDN state is rounded to single precision after each
 * step), with the bf16 storage points unchanged.  That build is never the
 * reference: the tests use the distance between its results and the double
 * build's to size the tolerance of whole-block comparisons, since it shows
 * how far a faithful fp32 evaluation of the same arithmetic lands from the
 * exact one.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef ORC_F32
typedef float real;
#define EXP expf
#define LOG1P log1pf
#define SQRT sqrtf
#else
typedef double real;
#define EXP exp
#define LOG1P log1p
#define SQRT sqrt
#endif

/* ------------------------------------------------------------------ bf16 */

double orc_bf16_val(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Nearest bf16 to x, ties to even.  x is scaled by a power of two so that the
 * bf16 grid around it becomes the integers, rounded with nearbyint (the FPU's
 * default mode is round-half-even), and scaled back; both scalings are exact. */
uint16_t orc_bf16_rne(double x) {
    if (isnan(x)) return signbit(x) ? 0xFFC0u : 0x7FC0u;
    if (isinf(x)) return signbit(x) ? 0xFF80u : 0x7F80u;
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    int e;
    frexp(x, &e);                  /* |x| = m 2^e, 0.5 <= m < 1 */
    int sh = e - 8;                /* 8 significant bits */
    if (sh < -133) sh = -133;      /* bf16 subnormal spacing is 2^-133 */
    double q = nearbyint(ldexp(x, -sh));
    double r = ldexp(q, sh);
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? 0xFF80u : 0x7F80u;
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double orc_bf16_round(double x) { return orc_bf16_val(orc_bf16_rne(x)); }

void orc_round_bf16_array(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_bf16_rne(x[i]);
}

/* Exhaustive-check helper: rounds float bit patterns [lo, hi) and stores the
 * bf16 patterns.  Loops in C only to keep the exhaustive pin fast. */
void orc_bf16_rne_f32_range(uint64_t lo, uint64_t hi, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = (int64_t)lo; i < (int64_t)hi; ++i) {
        uint32_t u = (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        out[i - (int64_t)lo] = orc_bf16_rne((double)f);
    }
}

/* ------------------------------------------------------------ elementwise */

static real sigmoid(real x) { return (real)1 / ((real)1 + EXP(-x)); }
static real softplus(real x) { return x > (real)20 ? x : LOG1P(EXP(x)); }
static real silu(real x) { return x * sigmoid(x); }

/* ----------------------------------------------------------------- GEMM */

/* Y[m][n] = sum_k X[m][k] * W[n][k], double accumulation in index order.
 * X is [M][ldx] bf16, W is [N][K] bf16 (row-major, the layout the model
 * stores), Y is [M][N] double.  [post]: the small-M route must give the same
 * bits for any row count; the value it approximates is this dot product. */
void orc_gemm(const uint16_t* X, int64_t ldx, const uint16_t* W, int M, int N, int K, double* Y) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t* w = W + (int64_t)n * K;
        for (int m = 0; m < M; ++m) {
            const uint16_t* x = X + (int64_t)m * ldx;
            real acc = 0;
            for (int k = 0; k < K; ++k) acc += (real)orc_bf16_val(x[k]) * (real)orc_bf16_val(w[k]);
            Y[(int64_t)m * N + n] = acc;
        }
    }
}

/* ---------------------------------------------------------- norms, MLP */

/* y = bf16( x / sqrt(mean(x^2) + eps) * (1 + w) ) */
void orc_rmsnorm(const uint16_t* x, const uint16_t* w, int H, double eps, uint16_t* y) {
    real ss = 0;
    for (int i = 0; i < H; ++i) ss += (real)orc_bf16_val(x[i]) * (real)orc_bf16_val(x[i]);
    real inv = (real)1 / SQRT(ss / (real)H + (real)eps);
    for (int i = 0; i < H; ++i)
        y[i] = orc_bf16_rne((real)orc_bf16_val(x[i]) * inv * ((real)1 + (real)orc_bf16_val(w[i])));
}

/* y = bf16( silu(g) * u ) */
void orc_swiglu(const uint16_t* g, const uint16_t* u, int n, uint16_t* y) {
    for (int i = 0; i < n; ++i) y[i] = orc_bf16_rne(silu((real)orc_bf16_val(g[i])) * (real)orc_bf16_val(u[i]));
}

/* beta = bf16(sigmoid(b)), gate = bf16(exp(-softplus(a))): the decode dtype
 * for both ([post]: the faulty verify kept beta in fp32). */
void orc_gdn_gates(const uint16_t* b, const uint16_t* a, int n, uint16_t* beta, uint16_t* gate) {
    for (int i = 0; i < n; ++i) {
        beta[i] = orc_bf16_rne(sigmoid((real)orc_bf16_val(b[i])));
        gate[i] = orc_bf16_rne(EXP(-softplus((real)orc_bf16_val(a[i]))));
    }
}

/* y = x / sqrt(sum x^2 + eps) */
void orc_l2norm(const double* x, int n, double eps, double* y) {
    real ss = 0;
    for (int i = 0; i < n; ++i) ss += (real)x[i] * (real)x[i];
    real d = SQRT(ss + (real)eps);
    for (int i = 0; i < n; ++i) y[i] = (real)x[i] / d;
}

/* ---------------------------------------------------------------- GDN */

/* One step of the gated delta rule on one head, written as the matrix
 * product it is:  S <- a * S * (I - b k k^T) + b v k^T ;  o = S q.
 * S is [dv][dk] row-major double; q, k have dk entries, v has dv; o gets dv
 * doubles (unrounded).  O(dv dk^2): slow on purpose, no refactoring. */
void orc_gdn_step(double* S, const double* q, const double* k, const double* v,
                  double beta, double gate, int dk, int dv, double* o) {
    real* P = (real*)malloc(sizeof(real) * (size_t)dk * dk);   /* I - b k k^T */
    real* T = (real*)malloc(sizeof(real) * (size_t)dv * dk);
    const real b = (real)beta, a = (real)gate;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dk; ++j) P[i * dk + j] = (real)(i == j ? 1 : 0) - b * (real)k[i] * (real)k[j];
    for (int r = 0; r < dv; ++r)
        for (int j = 0; j < dk; ++j) {
            real acc = 0;
            for (int i = 0; i < dk; ++i) acc += (real)S[r * dk + i] * P[i * dk + j];
            T[r * dk + j] = a * acc + b * (real)v[r] * (real)k[j];
        }
    for (int i = 0; i < dv * dk; ++i) S[i] = T[i];
    for (int r = 0; r < dv; ++r) {
        real acc = 0;
        for (int j = 0; j < dk; ++j) acc += (real)S[r * dk + j] * (real)q[j];
        o[r] = acc;
    }
    free(P);
    free(T);
}

/* A head's step from bf16 inputs as the model feeds it: q and k L2-normalised
 * in double when l2 != 0 (left as given otherwise), beta/gate already bf16;
 * o is rounded to bf16. */
void orc_gdn_step_bf16(double* S, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       uint16_t beta, uint16_t gate, int dk, int dv, int l2, uint16_t* o) {
    double* qd = (double*)malloc(sizeof(double) * dk);
    double* kd = (double*)malloc(sizeof(double) * dk);
    double* vd = (double*)malloc(sizeof(double) * dv);
    double* od = (double*)malloc(sizeof(double) * dv);
    for (int i = 0; i < dk; ++i) { qd[i] = orc_bf16_val(q[i]); kd[i] = orc_bf16_val(k[i]); }
    for (int i = 0; i < dv; ++i) vd[i] = orc_bf16_val(v[i]);
    if (l2) { orc_l2norm(qd, dk, 1e-6, qd); orc_l2norm(kd, dk, 1e-6, kd); }
    orc_gdn_step(S, qd, kd, vd, orc_bf16_val(beta), orc_bf16_val(gate), dk, dv, od);
    for (int i = 0; i < dv; ++i) o[i] = orc_bf16_rne(od[i]);
    free(qd); free(kd); free(vd); free(od);
}

/* Batched heads for one step: S [H][dv][dk], q/k [H][dk], v [H][dv],
 * beta/gate [H], o [H][dv]. */
void orc_gdn_step_heads(double* S, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* beta, const uint16_t* gate, int H, int dk, int dv, int l2,
                        uint16_t* o) {
#pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
        orc_gdn_step_bf16(S + (int64_t)h * dv * dk, q + (int64_t)h * dk, k + (int64_t)h * dk,
                          v + (int64_t)h * dv, beta[h], gate[h], dk, dv, l2, o + (int64_t)h * dv);
}

/* Grouped heads: v head h (of Hv) reads q and k of head h / (Hv / Hk).
 * S [Hv][dv][dk], q/k [Hk][dk], v [Hv][dv], beta/gate [Hv], o [Hv][dv]. */
void orc_gdn_step_heads_grouped(double* S, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const uint16_t* beta, const uint16_t* gate, int Hv, int Hk, int dk, int dv,
                                int l2, uint16_t* o) {
    int group = Hv / Hk;
#pragma omp parallel for schedule(static)
    for (int h = 0; h < Hv; ++h)
        orc_gdn_step_bf16(S + (int64_t)h * dv * dk, q + (int64_t)(h / group) * dk, k + (int64_t)(h / group) * dk,
                          v + (int64_t)h * dv, beta[h], gate[h], dk, dv, l2, o + (int64_t)h * dv);
}

/* One step of a depthwise causal convolution of width Kc over C channels,
 * then SiLU.  The window of channel c is its Kc-1 previous inputs (state,
 * [Kc-1][C], oldest row first) followed by x[c]; tap j = 0 meets the oldest:
 *     y[c] = bf16( silu( sum_j w[c][j] * window_c[j] ) ).
 * Afterwards the state forgets its oldest row and keeps x as its newest, so
 * it always holds the last Kc-1 inputs (bf16 values moved, never rounded). */
void orc_conv_step(uint16_t* state, const uint16_t* x, const uint16_t* w, int C, int Kc, uint16_t* y) {
    for (int c = 0; c < C; ++c) {
        real acc = 0;
        for (int j = 0; j < Kc - 1; ++j)
            acc += (real)orc_bf16_val(w[(int64_t)c * Kc + j]) * (real)orc_bf16_val(state[(int64_t)j * C + c]);
        acc += (real)orc_bf16_val(w[(int64_t)c * Kc + Kc - 1]) * (real)orc_bf16_val(x[c]);
        y[c] = orc_bf16_rne(silu(acc));
    }
    for (int j = 0; j + 1 < Kc - 1; ++j) memcpy(state + (int64_t)j * C, state + (int64_t)(j + 1) * C, sizeof(uint16_t) * C);
    if (Kc > 1) memcpy(state + (int64_t)(Kc - 2) * C, x, sizeof(uint16_t) * C);
}

/* The gated output norm of one head: y = bf16( o / sqrt(mean(o^2) + eps) * (1 + w) * silu(z) ). */
void orc_gated_norm(const uint16_t* o, const uint16_t* z, const uint16_t* w, int n, double eps, uint16_t* y) {
    real ss = 0;
    for (int i = 0; i < n; ++i) ss += (real)orc_bf16_val(o[i]) * (real)orc_bf16_val(o[i]);
    real inv = (real)1 / SQRT(ss / (real)n + (real)eps);
    for (int i = 0; i < n; ++i)
        y[i] = orc_bf16_rne((real)orc_bf16_val(o[i]) * inv * ((real)1 + (real)orc_bf16_val(w[i])) *
                            silu((real)orc_bf16_val(z[i])));
}

/* ---------------------------------------------------------- attention */

/* One decode row: softmax(q K^T * scale) V over positions [0, len), explicit
 * full softmax in double (no online or split form).  K and V are [pos][hd]
 * with row stride ld; out gets hd unrounded doubles.  [post]: verify runs
 * attention as one decode row per draft position; a decode row is this. */
void orc_attn_row(const uint16_t* q, const uint16_t* K, const uint16_t* V, int64_t ld,
                  int len, int hd, double scale, double* out) {
    real* s = (real*)malloc(sizeof(real) * (len > 0 ? len : 1));
    real m = -INFINITY;
    for (int j = 0; j < len; ++j) {
        real acc = 0;
        for (int d = 0; d < hd; ++d) acc += (real)orc_bf16_val(q[d]) * (real)orc_bf16_val(K[(int64_t)j * ld + d]);
        s[j] = acc * (real)scale;
        if (s[j] > m) m = s[j];
    }
    real l = 0;
    for (int j = 0; j < len; ++j) { s[j] = EXP(s[j] - m); l += s[j]; }
    for (int d = 0; d < hd; ++d) {
        real acc = 0;
        for (int j = 0; j < len; ++j) acc += s[j] * (real)orc_bf16_val(V[(int64_t)j * ld + d]);
        out[d] = acc / l;
    }
    free(s);
}

/* Rows of a verify block as the model issues them: q [R][Hq][hd] (row stride
 * q_ld), caches [Hkv][Lmax][hd]; row r sees len0 + r positions; out is
 * bf16 [R][Hq][hd].  Each (row, head) is an independent orc_attn_row. */
void orc_attn_rows(const uint16_t* q, int64_t q_ld, const uint16_t* kc, const uint16_t* vc,
                   int Lmax, int len0, int R, int Hq, int Hkv, int hd, double scale, uint16_t* out,
                   int64_t out_ld) {
    int G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; ++r)
        for (int h = 0; h < Hq; ++h) {
            double* o = (double*)malloc(sizeof(double) * hd);
            int g = h / G;
            orc_attn_row(q + r * q_ld + (int64_t)h * hd, kc + (int64_t)g * Lmax * hd,
                         vc + (int64_t)g * Lmax * hd, hd, len0 + r, hd, scale, o);
            for (int d = 0; d < hd; ++d) out[r * out_ld + (int64_t)h * hd + d] = orc_bf16_rne(o[d]);
            free(o);
        }
}

/* ---------------------------------------------------- argmax / accept */

/* Lowest index among the maxima. */
int orc_argmax(const double* x, int n) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (x[i] > x[best]) best = i;
    return best;
}

/* Greedy acceptance at temperature 0: tokens[0] is the last committed token,
 * tokens[1..k-1] are drafts, pred[j] is the target's argmax after position j.
 * Returns how many drafts are accepted (leading j with pred[j] == tokens[j+1]). */
int orc_accept(const int32_t* tokens, const int32_t* pred, int k) {
    int n = 0;
    while (n < k - 1 && pred[n] == tokens[n + 1]) ++n;
    return n;
}

/* ------------------------------------------------------ hybrid stack */

typedef struct {
    int H, V, F, n_layers;
    const int32_t* kind;        /* [n_layers]: 0 GDN, 1 attention */
    int gdn_h, gdn_dk, gdn_dv;
    int at_hq, at_hkv, at_hd;
    double eps;
    int gdn_hk;                 /* q/k heads of a GDN layer (gdn_h v heads) */
    int gdn_conv;               /* causal convolution width Kc (0: none) */
    int gdn_onorm;              /* 1: gated output norm with z columns */
} orc_cfg;

typedef struct {
    const uint16_t* embed;             /* [V][H] */
    const uint16_t* const* norm1;      /* [L] -> [H] */
    const uint16_t* const* w_in;       /* [L] -> [in][H] */
    const uint16_t* const* w_out;      /* [L] -> [H][inner] */
    const uint16_t* const* norm2;      /* [L] -> [H] */
    const uint16_t* const* w_gu;       /* [L] -> [2F][H], gate rows then up rows */
    const uint16_t* const* w_down;     /* [L] -> [H][F] */
    const uint16_t* final_norm;        /* [H] */
    const uint16_t* lm_head;           /* [V][H] */
    const uint16_t* const* conv_w;     /* [L] -> [C][Kc] (GDN layers with a convolution) */
    const uint16_t* const* onorm;      /* [L] -> [dv] (GDN layers with the gated output norm) */
} orc_weights;

typedef struct {
    double* const* S;        /* [L] -> GDN state [heads][dv][dk] (NULL for attention layers) */
    uint16_t* const* kc;     /* [L] -> [hkv][Lmax][hd] (NULL for GDN layers) */
    uint16_t* const* vc;
    int Lmax;
    int len;                 /* tokens already in the KV cache */
    uint16_t* const* conv;   /* [L] -> convolution state [Kc-1][C] bf16 (GDN layers with a convolution) */
} orc_seq;

/* y = bf16(x @ W^T) for one row */
static void proj(const uint16_t* x, const uint16_t* W, int N, int K, uint16_t* y) {
    double* t = (double*)malloc(sizeof(double) * N);
    orc_gemm(x, K, W, 1, N, K, t);
    orc_round_bf16_array(t, y, N);
    free(t);
}

static void residual(uint16_t* x, const uint16_t* y, int n) {
    for (int i = 0; i < n; ++i) x[i] = orc_bf16_rne(orc_bf16_val(x[i]) + orc_bf16_val(y[i]));
}

/* Input-projection widths (columns of w_in). */
int orc_gdn_in_dim(const orc_cfg* c) {
    return 2 * c->gdn_hk * c->gdn_dk + c->gdn_h * c->gdn_dv * (c->gdn_onorm ? 2 : 1) + 2 * c->gdn_h;
}
/* Channels the convolution runs over: q | k | v. */
int orc_gdn_conv_dim(const orc_cfg* c) { return 2 * c->gdn_hk * c->gdn_dk + c->gdn_h * c->gdn_dv; }
int orc_attn_in_dim(const orc_cfg* c) { return 2 * c->at_hq * c->at_hd + 2 * c->at_hkv * c->at_hd; }

static void gdn_mixer(const orc_cfg* c, double* S, uint16_t* conv_state, const uint16_t* conv_w,
                      const uint16_t* onorm, const uint16_t* xn, const uint16_t* Win, const uint16_t* Wout,
                      uint16_t* y) {
    int Hg = c->gdn_h, Hk = c->gdn_hk, dk = c->gdn_dk, dv = c->gdn_dv;
    int in = orc_gdn_in_dim(c), inner = Hg * dv, C = orc_gdn_conv_dim(c);
    uint16_t* p = (uint16_t*)malloc(sizeof(uint16_t) * in);
    uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * C);
    uint16_t* beta = (uint16_t*)malloc(sizeof(uint16_t) * Hg);
    uint16_t* gate = (uint16_t*)malloc(sizeof(uint16_t) * Hg);
    uint16_t* o = (uint16_t*)malloc(sizeof(uint16_t) * inner);
    proj(xn, Win, in, c->H, p);
    const uint16_t* qkv = p;
    if (c->gdn_conv > 0) {
        orc_conv_step(conv_state, p, conv_w, C, c->gdn_conv, u);
        qkv = u;
    }
    const uint16_t* q = qkv;
    const uint16_t* k = qkv + Hk * dk;
    const uint16_t* v = qkv + 2 * Hk * dk;
    const uint16_t* z = p + C;                       /* only with the gated output norm */
    const uint16_t* b = p + C + (c->gdn_onorm ? inner : 0);
    const uint16_t* a = b + Hg;
    orc_gdn_gates(b, a, Hg, beta, gate);
    orc_gdn_step_heads_grouped(S, q, k, v, beta, gate, Hg, Hk, dk, dv, 1, o);
    if (c->gdn_onorm)
        for (int h = 0; h < Hg; ++h) orc_gated_norm(o + h * dv, z + h * dv, onorm, dv, c->eps, o + h * dv);
    proj(o, Wout, c->H, inner, y);
    free(p); free(u); free(beta); free(gate); free(o);
}

static void attn_mixer(const orc_cfg* c, orc_seq* s, int layer, const uint16_t* xn,
                       const uint16_t* Win, const uint16_t* Wout, uint16_t* y) {
    int Hq = c->at_hq, Hkv = c->at_hkv, hd = c->at_hd;
    int in = orc_attn_in_dim(c), inner = Hq * hd;
    uint16_t* p = (uint16_t*)malloc(sizeof(uint16_t) * in);
    uint16_t* o = (uint16_t*)malloc(sizeof(uint16_t) * inner);
    proj(xn, Win, in, c->H, p);
    const uint16_t* q = p;
    const uint16_t* g = p + inner;
    const uint16_t* k = p + 2 * inner;
    const uint16_t* v = k + Hkv * hd;
    uint16_t* kc = s->kc[layer];
    uint16_t* vc = s->vc[layer];
    for (int h = 0; h < Hkv; ++h) {
        memcpy(kc + ((int64_t)h * s->Lmax + s->len) * hd, k + h * hd, sizeof(uint16_t) * hd);
        memcpy(vc + ((int64_t)h * s->Lmax + s->len) * hd, v + h * hd, sizeof(uint16_t) * hd);
    }
    orc_attn_rows(q, inner, kc, vc, s->Lmax, s->len + 1, 1, Hq, Hkv, hd, 1.0 / sqrt((double)hd), o, inner);
    for (int i = 0; i < inner; ++i) o[i] = orc_bf16_rne((real)orc_bf16_val(o[i]) * sigmoid((real)orc_bf16_val(g[i])));
    proj(o, Wout, c->H, inner, y);
    free(p); free(o);
}

/* Layer l of the stack for one position (s->len): the residual row x (bf16 [H]) in place through
 * x <- x + mixer(rmsnorm(x)), then x <- x + down(silu(gate) * up) of rmsnorm(x), each sum
 * rounded to bf16; mid (bf16 [H], or NULL) receives x between the two.  The layer's GDN state and
 * convolution state advance one step, or the position's K/V land at s->len; s->len is left as
 * it is. */
void orc_layer_token(const orc_cfg* c, const orc_weights* w, orc_seq* s, int l, uint16_t* x, uint16_t* mid) {
    int H = c->H, F = c->F;
    uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * H);
    uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * H);
    uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * 2 * F);
    uint16_t* act = (uint16_t*)malloc(sizeof(uint16_t) * F);
    orc_rmsnorm(x, w->norm1[l], H, c->eps, xn);
    if (c->kind[l] == 0)
        gdn_mixer(c, s->S[l], c->gdn_conv > 0 ? s->conv[l] : NULL, c->gdn_conv > 0 ? w->conv_w[l] : NULL,
                  c->gdn_onorm ? w->onorm[l] : NULL, xn, w->w_in[l], w->w_out[l], y);
    else attn_mixer(c, s, l, xn, w->w_in[l], w->w_out[l], y);
    residual(x, y, H);
    if (mid) memcpy(mid, x, sizeof(uint16_t) * H);
    orc_rmsnorm(x, w->norm2[l], H, c->eps, xn);
    proj(xn, w->w_gu[l], 2 * F, H, gu);
    orc_swiglu(gu, gu + F, F, act);
    proj(act, w->w_down[l], H, F, y);
    residual(x, y, H);
    free(xn); free(y); free(gu); free(act);
}

/* One decode step of one sequence: token in, logits [V] (double) out; the
 * GDN states advance one step, the token's K/V land at position len, and
 * len grows by one. */
void orc_decode_token(const orc_cfg* c, const orc_weights* w, orc_seq* s, int32_t token, double* logits) {
    int H = c->H;
    uint16_t* x = (uint16_t*)malloc(sizeof(uint16_t) * H);
    uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * H);
    memcpy(x, w->embed + (int64_t)token * H, sizeof(uint16_t) * H);
    for (int l = 0; l < c->n_layers; ++l) orc_layer_token(c, w, s, l, x, NULL);
    orc_rmsnorm(x, w->final_norm, H, c->eps, xn);
    orc_gemm(xn, H, w->lm_head, 1, c->V, H, logits);
    s->len += 1;
    free(x); free(xn);
}
