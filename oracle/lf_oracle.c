/*
 * lf_oracle.c -- plain, slow CPU reference of batch-1 decoder decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this library.  It
 * shares no code, header, table or constant generator with the CUDA library,
 * and the CUDA library never calls it.
 *
 * What it computes follows the KOG monokernel write-up (shivam2003.com,
 * "KOG LaneFormer-2B & the monokernel"):
 *   - batch-1 decode, one token per step, FP16 weights streamed once per
 *     token ("A worked bandwidth ceiling"; model table "Precision: FP16");
 *   - GEMV partial products accumulated in FP32 ("The fused operations,
 *     briefly", QKV-projection bullet);
 *   - Gumbel-max sampling, argmax_i(logit_i + g_i) ("The fused operations,
 *     briefly", sampling bullet);
 * and, where those pages are silent, the plain Llama-style decoder that the
 * workload definitions name: pre-norm RMSNorm blocks, rotate-half RoPE,
 * causal GQA attention over an FP16 KV cache, SwiGLU FFN, final RMSNorm and an
 * untied LM head.  Every reading taken where the pages are silent is listed in
 * the repository's design notes.
 *
 * Precision: activations and every accumulation are IEEE FP32, each dot
 * product summed left to right in index order; K and V are rounded to FP16
 * (round to nearest even) when stored in the cache.  Build with
 * -ffp-contract=off so that no multiply-add is fused and the result is the
 * same on x86-64 and aarch64.  OpenMP only splits independent output rows or
 * heads across threads; it does not change any sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the IEEE 754 encoding.           */
/* ------------------------------------------------------------------------ */

ORC_API float orc_half_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t expo = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t mant = (uint32_t)h & 0x3FFu;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)mant, -24);                  /* subnormal: m * 2^-24 */
    } else if (expo == 31) {
        mag = mant ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(mant | 0x400u), (int)expo - 25);  /* (1024+m) * 2^(e-25) */
    }
    return sign ? -mag : mag;
}

/* Round a float to the nearest binary16, ties to even. */
ORC_API uint16_t orc_float_to_half(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    float a = fabsf(f);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00u);  /* rounds to infinity */
    if (a < ldexpf(1.0f, -14)) {
        /* subnormal range: quantum 2^-24; rint rounds half to even */
        float q = rintf(ldexpf(a, 24));
        return (uint16_t)(sign | (uint16_t)q);           /* q == 1024 gives the smallest normal */
    }
    int e;
    frexpf(a, &e);                                       /* a = fr * 2^e, fr in [0.5, 1) */
    /* a in [2^(e-1), 2^e); binary16 quantum there is 2^(e-1-10) */
    float q = rintf(ldexpf(a, 11 - e));                  /* in [1024, 2048] */
    int expo = e - 1 + 15;
    uint32_t m = (uint32_t)q;
    if (m == 2048u) { m = 1024u; expo += 1; }
    if (expo >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(expo << 10) | (uint16_t)(m - 1024u));
}

/* ------------------------------------------------------------------------ */
/* Building blocks                                                           */
/* ------------------------------------------------------------------------ */

/* RMSNorm: out_i = x_i * (1 / sqrt(sum_j x_j^2 / d + eps)) * g_i. */
ORC_API void orc_rmsnorm(const float *x, const uint16_t *g, int d, float eps, float *out)
{
    float ss = 0.0f;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int i = 0; i < d; ++i) out[i] = (x[i] * inv) * orc_half_to_float(g[i]);
}

/* y_r = sum_k W[r, k] * x_k, W row-major FP16 [n_rows, k_dim], FP32 sum in index order. */
ORC_API void orc_matvec(const uint16_t *W, const float *x, int n_rows, int k_dim, float *y)
{
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < n_rows; ++r) {
        const uint16_t *row = W + (size_t)r * (size_t)k_dim;
        float acc = 0.0f;
        for (int k = 0; k < k_dim; ++k) acc += orc_half_to_float(row[k]) * x[k];
        y[r] = acc;
    }
}

/* FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite value 448), decoded from the
 * format definition: exponent field 0 gives the subnormals m/8 * 2^-6. */
ORC_API float orc_e4m3_to_float(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const float mag = e == 0 ? ldexpf((float)m / 8.0f, -6) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -mag : mag;
}

/* y = diag(scale) . decode(C) . x for an [n_rows, k_dim] matrix of E4M3 codes
 * with one FP32 scale per row (weight-only FP8; the pages' FP8 streaming,
 * shivam2003.com, "Scaling the idea to frontier models"): each row's dot
 * product of the decoded codes with x in FP32, index order, then times the
 * row's scale. */
ORC_API void orc_matvec_fp8(const uint8_t *C, const float *scale, const float *x, int n_rows, int k_dim, float *y)
{
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < n_rows; ++r) {
        const uint8_t *row = C + (size_t)r * (size_t)k_dim;
        float acc = 0.0f;
        for (int k = 0; k < k_dim; ++k) acc += orc_e4m3_to_float(row[k]) * x[k];
        y[r] = acc * scale[r];
    }
}

/* MXFP4 (OCP Microscaling FP4; the pages' "FP8/MXFP4" streaming,
 * shivam2003.com, "Scaling the idea to frontier models").  Elements are E2M1
 * (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no infinities or NaN):
 * exponent field 0 gives the subnormals m * 0.5, so the magnitudes are 0,
 * 0.5, 1, 1.5, 2, 3, 4 and 6.  Blocks of 32 consecutive elements of a row
 * share one E8M0 scale, 2^(E - 127), with E = 255 meaning NaN. */
ORC_API float orc_e2m1_to_float(uint8_t nib)
{
    const int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    const float mag = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
    return s ? -mag : mag;
}
ORC_API float orc_e8m0_to_float(uint8_t e)
{
    if (e == 255) return NAN;
    return ldexpf(1.0f, (int)e - 127);
}

/* y = decode(C, S) . x for an [n_rows, k_dim] MXFP4 matrix: C holds two
 * elements per byte (element k of a row in the low nibble of byte k/2 for
 * even k, in the high nibble for odd k), S one E8M0 scale per 32 elements
 * ([n_rows, k_dim/32]).  Weight (r, k) = e2m1(C) * e8m0(S[r][k/32]), exact in
 * FP32; each row's dot product with x in FP32, index order. */
ORC_API void orc_matvec_mxfp4(const uint8_t *C, const uint8_t *S, const float *x, int n_rows, int k_dim, float *y)
{
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < n_rows; ++r) {
        const uint8_t *row = C + (size_t)r * (size_t)(k_dim / 2);
        const uint8_t *sc = S + (size_t)r * (size_t)(k_dim / 32);
        float acc = 0.0f;
        for (int k = 0; k < k_dim; ++k) {
            const uint8_t nib = (k & 1) ? (uint8_t)(row[k / 2] >> 4) : (uint8_t)(row[k / 2] & 15);
            const float w = orc_e2m1_to_float(nib) * orc_e8m0_to_float(sc[k / 32]);
            acc += w * x[k];
        }
        y[r] = acc;
    }
}

/* Rotate-half RoPE of one head vector v[hd] at position pos:
 * for i < hd/2, theta_i = pos * base^(-2i/hd) (in double), and
 *   v[i]        <- v[i] cos - v[i+hd/2] sin
 *   v[i+hd/2]   <- v[i+hd/2] cos + v[i] sin      (FP32 arithmetic). */
ORC_API void orc_rope(float *v, int hd, int pos, float base)
{
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow((double)base, -2.0 * (double)i / (double)hd);
        double ang = (double)pos * inv_freq;
        float c = (float)cos(ang), s = (float)sin(ang);
        float a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

/* Softmax-weighted sum for one query head over ctx cached positions:
 *   s_j = (q . K_j) * scale,  p = softmax(s) (max subtracted),  o = sum_j p_j V_j.
 * K, V: FP16 rows of hd values, row j at K + j*hd.  scores: scratch [ctx]. */
ORC_API void orc_attend_head(const float *q, const uint16_t *K, const uint16_t *V, int ctx, int hd,
                             float scale, float *scores, float *out)
{
    float m = -INFINITY;
    for (int j = 0; j < ctx; ++j) {
        const uint16_t *kj = K + (size_t)j * hd;
        float dot = 0.0f;
        for (int i = 0; i < hd; ++i) dot += q[i] * orc_half_to_float(kj[i]);
        scores[j] = dot * scale;
        if (scores[j] > m) m = scores[j];
    }
    float sum = 0.0f;
    for (int j = 0; j < ctx; ++j) { scores[j] = expf(scores[j] - m); sum += scores[j]; }
    for (int j = 0; j < ctx; ++j) scores[j] = scores[j] / sum;
    for (int i = 0; i < hd; ++i) out[i] = 0.0f;
    for (int j = 0; j < ctx; ++j) {
        const uint16_t *vj = V + (size_t)j * hd;
        for (int i = 0; i < hd; ++i) out[i] += scores[j] * orc_half_to_float(vj[i]);
    }
}

/* SiLU(z) = z / (1 + e^-z). */
ORC_API float orc_silu(float z) { return z / (1.0f + expf(-z)); }

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with     */
/* Weyl key bumps between rounds.                                            */
/* ------------------------------------------------------------------------ */

#define ORC_PHILOX_M0 0xD2511F53u
#define ORC_PHILOX_M1 0xCD9E8D57u
#define ORC_PHILOX_W0 0x9E3779B9u
#define ORC_PHILOX_W1 0xBB67AE85u

ORC_API void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += ORC_PHILOX_W0; k1 += ORC_PHILOX_W1; }
        uint64_t p0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Gumbel noise for vocabulary entry i of the step at position pos:
 *   r = word (i mod 4) of Philox4x32-10(counter = (i div 4, pos, 0, 0), key = seed),
 *   u = (2 * (r >> 9) + 1) * 2^-24 in (0, 1)   (exact in FP32),
 *   g = -log(-log(u)). */
ORC_API float orc_gumbel(uint64_t seed, int pos, int i)
{
    uint32_t ctr[4] = {(uint32_t)i >> 2, (uint32_t)pos, 0u, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t r[4];
    orc_philox4x32_10(ctr, key, r);
    uint32_t w = r[i & 3];
    float u = (float)((w >> 9) * 2u + 1u) * 0x1p-24f;
    return -logf(-logf(u));
}

/* Order used for "largest logits": larger value first, equal values by lower index. */
static const float *g_sort_logits;
static int orc_cmp_desc(const void *a, const void *b)
{
    int ia = *(const int *)a, ib = *(const int *)b;
    float va = g_sort_logits[ia], vb = g_sort_logits[ib];
    if (va > vb) return -1;
    if (va < vb) return 1;
    return (ia < ib) ? -1 : (ia > ib);
}

/* Token choice for one step.
 *   temperature <= 0 or top_k == 1: greedy argmax (lowest index among equal maxima).
 *   otherwise: S = the top_k largest logits (top_k <= 0 or >= V: all of them);
 *   token = argmax_{i in S} (logit_i / T + g_i), equal scores resolved to the lower index. */
ORC_API int orc_sample(const float *logits, int V, float temperature, int top_k, uint64_t seed, int pos)
{
    if (temperature <= 0.0f || top_k == 1) {
        int best = 0;
        for (int i = 1; i < V; ++i) if (logits[i] > logits[best]) best = i;
        return best;
    }
    int k = (top_k <= 0 || top_k >= V) ? V : top_k;
    int *idx = (int *)malloc(sizeof(int) * (size_t)V);
    for (int i = 0; i < V; ++i) idx[i] = i;
    if (k < V) {
        g_sort_logits = logits;
        qsort(idx, (size_t)V, sizeof(int), orc_cmp_desc);
    }
    int tok = -1;
    float best = -INFINITY;
    for (int j = 0; j < k; ++j) {
        int i = idx[j];
        float score = logits[i] / temperature + orc_gumbel(seed, pos, i);
        if (tok < 0 || score > best || (score == best && i < tok)) { best = score; tok = i; }
    }
    free(idx);
    return tok;
}

/* ------------------------------------------------------------------------ */
/* The decoder                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab, max_seq;
    float rope_theta, rms_eps;
} orc_config;

typedef struct {
    const uint16_t *embed;      /* [V, d] */
    const uint16_t *attn_norm;  /* [L, d] */
    const uint16_t *wq;         /* [L, Q, d] */
    const uint16_t *wk;         /* [L, KV, d] */
    const uint16_t *wv;         /* [L, KV, d] */
    const uint16_t *wo;         /* [L, d, Q] */
    const uint16_t *ffn_norm;   /* [L, d] */
    const uint16_t *w_gate;     /* [L, F, d] */
    const uint16_t *w_up;       /* [L, F, d] */
    const uint16_t *w_down;     /* [L, d, F] */
    const uint16_t *final_norm; /* [d] */
    const uint16_t *lm_head;    /* [V, d] */
} orc_weights;

typedef struct {
    orc_config c;
    orc_weights w;
    uint16_t *kcache;   /* [L][H_kv][max_seq][hd] FP16 */
    uint16_t *vcache;
    int pos;            /* position of the pending token */
    int pending;        /* token fed to the next forward pass, -1 if none */
    int *window;        /* [L] attention window of each layer in positions, 0 = the whole cache */
    /* FP8 weights: the eight projection pointers of w hold E4M3 codes, and
     * scale[i] the per-row FP32 scales of matrix i (wq, wk, wv, wo, w_gate,
     * w_up, w_down, lm_head); fp8 = 0: FP16 weights */
    int fp8;
    const float *scale[8];
    /* MXFP4 weights: the eight projection pointers hold packed E2M1 codes and
     * bscale[i] the E8M0 block scales of matrix i ([rows, cols/32]) */
    int mxfp4;
    const uint8_t *bscale[8];
    /* Mixture-of-experts FFN: n_experts = E > 0 experts per layer, top_k of
     * them active per token; w_gate / w_up are then [L, E, F, d], w_down
     * [L, E, d, F] (F = ffn_dim per expert) and router [L, E, d] */
    int n_experts, top_k;
    const uint16_t *router;
    float *ffn_acc;     /* [d] */
    float *rlogit;      /* [E] */
    /* activations */
    float *x, *xn, *q, *k, *v, *attn, *tmp, *gate, *up, *hbuf, *scores;
} orc_model;

ORC_API orc_model *orc_create(const orc_config *c, const orc_weights *w)
{
    if (!c || !w || c->n_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0) return NULL;
    orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
    m->c = *c;
    m->w = *w;
    size_t kv = (size_t)c->n_layers * c->n_kv_heads * (size_t)c->max_seq * c->head_dim;
    m->kcache = (uint16_t *)calloc(kv, 2);
    m->vcache = (uint16_t *)calloc(kv, 2);
    int d = c->d_model, Q = c->n_heads * c->head_dim, KV = c->n_kv_heads * c->head_dim, F = c->ffn_dim;
    m->x = (float *)calloc((size_t)d, 4);
    m->xn = (float *)calloc((size_t)d, 4);
    m->q = (float *)calloc((size_t)Q, 4);
    m->k = (float *)calloc((size_t)KV, 4);
    m->v = (float *)calloc((size_t)KV, 4);
    m->attn = (float *)calloc((size_t)Q, 4);
    m->tmp = (float *)calloc((size_t)(d > c->vocab ? d : c->vocab), 4);
    m->gate = (float *)calloc((size_t)F, 4);
    m->up = (float *)calloc((size_t)F, 4);
    m->hbuf = (float *)calloc((size_t)F, 4);
    m->scores = (float *)calloc((size_t)c->n_heads * (size_t)c->max_seq, 4);
    m->window = (int *)calloc((size_t)c->n_layers, sizeof(int));
    if (!m->kcache || !m->vcache || !m->scores || !m->window) { free(m); return NULL; }
    m->pos = 0;
    m->pending = -1;
    return m;
}

ORC_API void orc_destroy(orc_model *m)
{
    if (!m) return;
    free(m->ffn_acc); free(m->rlogit);
    free(m->kcache); free(m->vcache);
    free(m->x); free(m->xn); free(m->q); free(m->k); free(m->v); free(m->attn);
    free(m->tmp); free(m->gate); free(m->up); free(m->hbuf); free(m->scores); free(m->window);
    free(m);
}

ORC_API void orc_reset(orc_model *m) { m->pos = 0; m->pending = -1; }

/* Sliding-window attention (shivam2003.com, model table and "Why GQA and
 * sliding windows": some layers attend only to a window of recent positions,
 * so that the KV cache they read stops growing with the context).  window[l]
 * = W > 0: the query at position p of layer l attends to the W positions
 * max(0, p-W+1) .. p; W = 0: to every cached position.  NULL clears them. */
/* Switch the model to FP8 weights (see orc_model); NULL scales switch back. */
ORC_API void orc_set_fp8(orc_model *m, const float *const *scales)
{
    m->fp8 = scales != NULL;
    for (int i = 0; i < 8; ++i) m->scale[i] = scales ? scales[i] : NULL;
}

/* Switch the model to MXFP4 weights (see orc_model); NULL switches back. */
ORC_API void orc_set_mxfp4(orc_model *m, const uint8_t *const *bscales)
{
    m->mxfp4 = bscales != NULL;
    for (int i = 0; i < 8; ++i) m->bscale[i] = bscales ? bscales[i] : NULL;
}

/* Switch the model to a mixture-of-experts FFN (see orc_model; FP16
 * weights).  n_experts = 0 switches back to the dense FFN.  Returns 0, or -1
 * for top_k outside [1, min(n_experts, 8)] or n_experts above 64. */
ORC_API int orc_set_moe(orc_model *m, int n_experts, int top_k, const uint16_t *router)
{
    if (n_experts == 0) {
        m->n_experts = 0;
        return 0;
    }
    if (n_experts < 1 || n_experts > 64 || top_k < 1 || top_k > 8 || top_k > n_experts || !router) return -1;
    if (!m->ffn_acc) m->ffn_acc = (float *)calloc((size_t)m->c.d_model, 4);
    if (!m->rlogit) m->rlogit = (float *)calloc(64, 4);
    if (!m->ffn_acc || !m->rlogit) return -1;
    m->n_experts = n_experts;
    m->top_k = top_k;
    m->router = router;
    return 0;
}

/* Top-k routing of one token (the plain mixture-of-experts reading of the
 * pages' "only the active experts' weights stream per token", shivam2003.com,
 * "Scaling the idea to frontier models"): the k largest router logits, ties
 * to the lower expert index, in decreasing order; gate_j = softmax over the
 * k selected logits (FP32, the largest subtracted). */
ORC_API void orc_route(const float *logits, int n_experts, int top_k, int *sel, float *gate)
{
    unsigned long long used = 0ull;
    for (int j = 0; j < top_k; ++j) {
        int best = -1;
        for (int e = 0; e < n_experts; ++e)
            if (!(used >> e & 1ull) && (best < 0 || logits[e] > logits[best])) best = e;
        used |= 1ull << best;
        sel[j] = best;
    }
    float sum = 0.0f;
    for (int j = 0; j < top_k; ++j) {
        gate[j] = expf(logits[sel[j]] - logits[sel[0]]);
        sum += gate[j];
    }
    for (int j = 0; j < top_k; ++j) gate[j] = gate[j] / sum;
}

/* Projection `which` (0 wq .. 7 lm_head) of layer l: y = W x. */
static void orc_project(const orc_model *m, int which, int l, int n_rows, int k_dim, const float *x, float *y)
{
    const orc_weights *w = &m->w;
    const uint16_t *base[8] = {w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down, w->lm_head};
    const size_t off = (size_t)l * (size_t)n_rows * (size_t)k_dim;
    if (m->mxfp4)
        orc_matvec_mxfp4((const uint8_t *)base[which] + off / 2, m->bscale[which] + off / 32, x, n_rows, k_dim, y);
    else if (m->fp8)
        orc_matvec_fp8((const uint8_t *)base[which] + off, m->scale[which] + (size_t)l * n_rows, x, n_rows, k_dim, y);
    else
        orc_matvec(base[which] + off, x, n_rows, k_dim, y);
}

/* Timing hook: make `token` the pending token at position `pos` without
 * running the forward passes of positions 0 .. pos-1 (their cache rows keep
 * what they hold: zeros in a fresh model).  The work of a decode step depends
 * on its position, not on the cached values, so decode steps after this time
 * like steps at that context.  Returns 0, or -1 for a position or token out of
 * range.  Parity tests never call it. */
ORC_API int orc_skip_to(orc_model *m, int pos, int token)
{
    if (pos < 0 || pos >= m->c.max_seq || token < 0 || token >= m->c.vocab) return -1;
    m->pos = pos;
    m->pending = token;
    return 0;
}

ORC_API void orc_set_windows(orc_model *m, const int *window)
{
    for (int l = 0; l < m->c.n_layers; ++l) m->window[l] = window ? (window[l] > 0 ? window[l] : 0) : 0;
}
ORC_API int orc_pos(const orc_model *m) { return m->pos; }
ORC_API int orc_pending(const orc_model *m) { return m->pending; }
ORC_API const uint16_t *orc_kcache(const orc_model *m) { return m->kcache; }
ORC_API const uint16_t *orc_vcache(const orc_model *m) { return m->vcache; }

ORC_API int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One forward pass of `token` at position m->pos.  Appends K and V of this
 * position to the cache, writes the V logits if `logits` is not NULL, and
 * advances the position.  Returns 0, or -1 if the cache is full. */
ORC_API int orc_forward(orc_model *m, int token, float *logits)
{
    const orc_config *c = &m->c;
    const orc_weights *w = &m->w;
    int L = c->n_layers, d = c->d_model, Hq = c->n_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
    int F = c->ffn_dim, Q = Hq * hd, KV = Hkv * hd, group = Hq / Hkv;
    int p = m->pos;
    if (p >= c->max_seq || token < 0 || token >= c->vocab) return -1;
    float scale = 1.0f / sqrtf((float)hd);

    for (int i = 0; i < d; ++i) m->x[i] = orc_half_to_float(w->embed[(size_t)token * d + i]);

    for (int l = 0; l < L; ++l) {
        /* attention block */
        orc_rmsnorm(m->x, w->attn_norm + (size_t)l * d, d, c->rms_eps, m->xn);
        orc_project(m, 0, l, Q, d, m->xn, m->q);
        orc_project(m, 1, l, KV, d, m->xn, m->k);
        orc_project(m, 2, l, KV, d, m->xn, m->v);
        for (int h = 0; h < Hq; ++h) orc_rope(m->q + h * hd, hd, p, c->rope_theta);
        for (int g = 0; g < Hkv; ++g) orc_rope(m->k + g * hd, hd, p, c->rope_theta);
        for (int g = 0; g < Hkv; ++g) {
            size_t base = (((size_t)l * Hkv + g) * (size_t)c->max_seq + (size_t)p) * hd;
            for (int i = 0; i < hd; ++i) {
                m->kcache[base + i] = orc_float_to_half(m->k[g * hd + i]);
                m->vcache[base + i] = orc_float_to_half(m->v[g * hd + i]);
            }
        }
        /* positions j0 .. p: the whole cache, or the layer's window */
        int j0 = 0;
        if (m->window[l] > 0 && p + 1 > m->window[l]) j0 = p + 1 - m->window[l];
        #pragma omp parallel for schedule(static)
        for (int h = 0; h < Hq; ++h) {
            int g = h / group;
            size_t base = (((size_t)l * Hkv + g) * (size_t)c->max_seq + (size_t)j0) * hd;
            orc_attend_head(m->q + h * hd, m->kcache + base, m->vcache + base, p + 1 - j0, hd, scale,
                            m->scores + (size_t)h * c->max_seq, m->attn + h * hd);
        }
        orc_project(m, 3, l, d, Q, m->attn, m->tmp);
        for (int i = 0; i < d; ++i) m->x[i] = m->x[i] + m->tmp[i];

        /* FFN block */
        orc_rmsnorm(m->x, w->ffn_norm + (size_t)l * d, d, c->rms_eps, m->xn);
        if (m->n_experts > 0) {
            /* mixture of experts: y = sum_j gate_j * expert_{e_j}(xn) */
            const int E = m->n_experts;
            int sel[8];
            float gate[8];
            orc_matvec(m->router + (size_t)l * E * d, m->xn, E, d, m->rlogit);
            orc_route(m->rlogit, E, m->top_k, sel, gate);
            for (int i = 0; i < d; ++i) m->ffn_acc[i] = 0.0f;
            for (int j = 0; j < m->top_k; ++j) {
                const size_t ex = (size_t)l * E + (size_t)sel[j];
                orc_matvec(w->w_gate + ex * F * d, m->xn, F, d, m->gate);
                orc_matvec(w->w_up + ex * F * d, m->xn, F, d, m->up);
                for (int i = 0; i < F; ++i) m->hbuf[i] = orc_silu(m->gate[i]) * m->up[i];
                orc_matvec(w->w_down + ex * d * F, m->hbuf, d, F, m->tmp);
                for (int i = 0; i < d; ++i) m->ffn_acc[i] = m->ffn_acc[i] + gate[j] * m->tmp[i];
            }
            for (int i = 0; i < d; ++i) m->x[i] = m->x[i] + m->ffn_acc[i];
        } else {
            orc_project(m, 4, l, F, d, m->xn, m->gate);
            orc_project(m, 5, l, F, d, m->xn, m->up);
            for (int i = 0; i < F; ++i) m->hbuf[i] = orc_silu(m->gate[i]) * m->up[i];
            orc_project(m, 6, l, d, F, m->hbuf, m->tmp);
            for (int i = 0; i < d; ++i) m->x[i] = m->x[i] + m->tmp[i];
        }
    }
    if (logits) {
        orc_rmsnorm(m->x, w->final_norm, d, c->rms_eps, m->xn);
        orc_project(m, 7, 0, c->vocab, d, m->xn, logits);
    }
    m->pos = p + 1;
    return 0;
}

/* Prefill: forward passes of tokens[0 .. n-2]; tokens[n-1] becomes the pending
 * token.  Returns 0, or -1 on a bad argument or a full cache. */
ORC_API int orc_prefill(orc_model *m, const int32_t *tokens, int n)
{
    /* positions used: the pending token (if any), tokens[0 .. n-2], and one
     * more for tokens[n-1] when it is later decoded */
    if (n < 1 || m->pos + (m->pending >= 0 ? 1 : 0) + n > m->c.max_seq) return -1;
    if (m->pending >= 0) {
        /* a pending token from an earlier call is consumed first */
        if (orc_forward(m, m->pending, NULL)) return -1;
    }
    for (int i = 0; i < n - 1; ++i)
        if (orc_forward(m, tokens[i], NULL)) return -1;
    m->pending = tokens[n - 1];
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Prefill in blocks of positions (long prompts for stored test data)       */
/* ------------------------------------------------------------------------ */

/* Y[t][r] = sum_k W[r, k] * X[t][k] for the T rows of X: the sum of
 * orc_matvec for every t, formed the same way (FP32 products of the decoded
 * weight and x, added left to right in index order), with each weight row
 * decoded from FP16 once for all T inputs.  XT holds X transposed, [k_dim][Tp]
 * with Tp = T rounded up to a multiple of 8 (zero-padded), so that eight
 * independent sums advance together. */
static void orc_block_matvec(const uint16_t *W, const float *XT, int T, int Tp, int n_rows, int k_dim, float *Y)
{
    #pragma omp parallel
    {
        float *wrow = (float *)malloc(sizeof(float) * (size_t)k_dim);
        #pragma omp for schedule(static)
        for (int r = 0; r < n_rows; ++r) {
            const uint16_t *row = W + (size_t)r * (size_t)k_dim;
            for (int k = 0; k < k_dim; ++k) wrow[k] = orc_half_to_float(row[k]);
            for (int t0 = 0; t0 < Tp; t0 += 8) {
                float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
                for (int k = 0; k < k_dim; ++k) {
                    const float w = wrow[k];
                    const float *xk = XT + (size_t)k * (size_t)Tp + t0;
                    #pragma omp simd
                    for (int u = 0; u < 8; ++u) acc[u] += w * xk[u];
                }
                for (int u = 0; u < 8 && t0 + u < T; ++u) Y[(size_t)(t0 + u) * (size_t)n_rows + r] = acc[u];
            }
        }
        free(wrow);
    }
}

/* orc_attend_head on K and V rows already converted to FP32 (the conversion
 * is exact, so the values are the same): the same scores, each q . K_j summed
 * over i in index order, eight positions j at a time as independent sums; the
 * same softmax; o_i += p_j V_j,i over j in order.  Equal to orc_attend_head
 * bit for bit (the blocked-prefill test compares the two paths). */
static void orc_attend_head_f32(const float *q, const float *K, const float *V, int ctx, int hd, float scale,
                                float *scores, float *out)
{
    float m = -INFINITY;
    int j = 0;
    for (; j + 8 <= ctx; j += 8) {
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        const float *kj = K + (size_t)j * hd;
        for (int i = 0; i < hd; ++i) {
            const float qi = q[i];
            for (int u = 0; u < 8; ++u) acc[u] += qi * kj[(size_t)u * hd + i];
        }
        for (int u = 0; u < 8; ++u) {
            scores[j + u] = acc[u] * scale;
            if (scores[j + u] > m) m = scores[j + u];
        }
    }
    for (; j < ctx; ++j) {
        const float *kj = K + (size_t)j * hd;
        float dot = 0.0f;
        for (int i = 0; i < hd; ++i) dot += q[i] * kj[i];
        scores[j] = dot * scale;
        if (scores[j] > m) m = scores[j];
    }
    float sum = 0.0f;
    for (j = 0; j < ctx; ++j) { scores[j] = expf(scores[j] - m); sum += scores[j]; }
    for (j = 0; j < ctx; ++j) scores[j] = scores[j] / sum;
    for (int i = 0; i < hd; ++i) out[i] = 0.0f;
    for (j = 0; j < ctx; ++j) {
        const float pj = scores[j];
        const float *vj = V + (size_t)j * hd;
        #pragma omp simd
        for (int i = 0; i < hd; ++i) out[i] += pj * vj[i];
    }
}

/* X [T][k_dim] -> XT [k_dim][Tp], zero-padded to Tp columns. */
static void orc_transpose_pad(const float *X, int T, int Tp, int k_dim, float *XT)
{
    for (int k = 0; k < k_dim; ++k) {
        float *dst = XT + (size_t)k * (size_t)Tp;
        for (int t = 0; t < T; ++t) dst[t] = X[(size_t)t * (size_t)k_dim + k];
        for (int t = T; t < Tp; ++t) dst[t] = 0.0f;
    }
}

/* The forward passes of orc_prefill -- the pending token (if any), then
 * tokens[0 .. n-2], tokens[n-1] left pending -- taken `block` positions at a
 * time.  Nothing in the arithmetic of one position changes: every norm,
 * product, sum (index order), rotation, rounding of K and V to FP16 and
 * softmax is orc_forward's, and attention at position p reads cache rows
 * j0 .. p exactly as it would after the earlier forward passes (the block's
 * K and V rows of a layer are stored before that layer's attention runs).
 * Only the order in which independent positions are visited changes: within
 * a layer every position of the block goes through one projection before the
 * next starts, so each weight row is decoded once per block instead of once
 * per position, and attention reads FP32 copies of the cache rows
 * (orc_attend_head_f32).  The cache and the pending state therefore equal those of
 * orc_prefill bit for bit (checked by a test).  Dense FP16 models only (FP8,
 * MXFP4 and mixture-of-experts models: orc_prefill).  Returns 0, or -1 on a
 * bad argument, a full cache, an unsupported model or a failed allocation. */
ORC_API int orc_prefill_blocked(orc_model *m, const int32_t *tokens, int n, int block)
{
    const orc_config *c = &m->c;
    const orc_weights *w = &m->w;
    const int L = c->n_layers, d = c->d_model, Hq = c->n_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
    const int F = c->ffn_dim, Q = Hq * hd, KV = Hkv * hd, group = Hq / Hkv;
    if (n < 1 || block < 1 || m->fp8 || m->mxfp4 || m->n_experts > 0) return -1;
    const int has_pending = m->pending >= 0;
    const int n_pass = n - 1 + has_pending;
    if (m->pos + n_pass + 1 > c->max_seq) return -1;
    for (int i = 0; i < n; ++i) if (tokens[i] < 0 || tokens[i] >= c->vocab) return -1;
    const float scale = 1.0f / sqrtf((float)hd);
    const int Tp_max = (block + 7) / 8 * 8;
    const int wide = Q > F ? (Q > d ? Q : d) : (F > d ? F : d);
    float *X = (float *)malloc(sizeof(float) * (size_t)block * d);
    float *XN = (float *)malloc(sizeof(float) * (size_t)block * wide);
    float *XT = (float *)malloc(sizeof(float) * (size_t)Tp_max * wide);
    float *Yq = (float *)malloc(sizeof(float) * (size_t)block * Q);
    float *Yk = (float *)malloc(sizeof(float) * (size_t)block * KV);
    float *Yv = (float *)malloc(sizeof(float) * (size_t)block * KV);
    float *A = (float *)malloc(sizeof(float) * (size_t)block * Q);
    float *G = (float *)malloc(sizeof(float) * (size_t)block * F);
    float *U = (float *)malloc(sizeof(float) * (size_t)block * F);
    float *Y = (float *)malloc(sizeof(float) * (size_t)block * d);
    int nthr = 1;
#ifdef _OPENMP
    nthr = omp_get_max_threads();
#endif
    float *scr = (float *)malloc(sizeof(float) * (size_t)nthr * (size_t)c->max_seq);
    /* FP32 copies of the cache rows (exact), converted once per row */
    const size_t kv_elems = (size_t)L * Hkv * (size_t)c->max_seq * hd;
    float *kf = (float *)malloc(sizeof(float) * kv_elems);
    float *vf = (float *)malloc(sizeof(float) * kv_elems);
    int rc = 0;
    if (!X || !XN || !XT || !Yq || !Yk || !Yv || !A || !G || !U || !Y || !scr || !kf || !vf) rc = -1;
    for (int l = 0; rc == 0 && l < L; ++l)
        for (int g = 0; g < Hkv; ++g) {
            const size_t base = ((size_t)l * Hkv + g) * (size_t)c->max_seq * hd;
            for (size_t i = 0; i < (size_t)m->pos * hd; ++i) {
                kf[base + i] = orc_half_to_float(m->kcache[base + i]);
                vf[base + i] = orc_half_to_float(m->vcache[base + i]);
            }
        }
    for (int b0 = 0; rc == 0 && b0 < n_pass; b0 += block) {
        const int T = n_pass - b0 < block ? n_pass - b0 : block;
        const int Tp = (T + 7) / 8 * 8;
        const int p0 = m->pos;
        for (int t = 0; t < T; ++t) {
            const int i = b0 + t;   /* pass i: the pending token first, then the prompt */
            const int tok = has_pending ? (i == 0 ? m->pending : tokens[i - 1]) : tokens[i];
            for (int k = 0; k < d; ++k) X[(size_t)t * d + k] = orc_half_to_float(w->embed[(size_t)tok * d + k]);
        }
        for (int l = 0; l < L; ++l) {
            /* attention block */
            for (int t = 0; t < T; ++t)
                orc_rmsnorm(X + (size_t)t * d, w->attn_norm + (size_t)l * d, d, c->rms_eps, XN + (size_t)t * d);
            orc_transpose_pad(XN, T, Tp, d, XT);
            orc_block_matvec(w->wq + (size_t)l * Q * d, XT, T, Tp, Q, d, Yq);
            orc_block_matvec(w->wk + (size_t)l * KV * d, XT, T, Tp, KV, d, Yk);
            orc_block_matvec(w->wv + (size_t)l * KV * d, XT, T, Tp, KV, d, Yv);
            for (int t = 0; t < T; ++t) {
                const int p = p0 + t;
                for (int h = 0; h < Hq; ++h) orc_rope(Yq + (size_t)t * Q + h * hd, hd, p, c->rope_theta);
                for (int g = 0; g < Hkv; ++g) orc_rope(Yk + (size_t)t * KV + g * hd, hd, p, c->rope_theta);
                for (int g = 0; g < Hkv; ++g) {
                    const size_t base = (((size_t)l * Hkv + g) * (size_t)c->max_seq + (size_t)p) * hd;
                    for (int i = 0; i < hd; ++i) {
                        m->kcache[base + i] = orc_float_to_half(Yk[(size_t)t * KV + g * hd + i]);
                        m->vcache[base + i] = orc_float_to_half(Yv[(size_t)t * KV + g * hd + i]);
                        kf[base + i] = orc_half_to_float(m->kcache[base + i]);
                        vf[base + i] = orc_half_to_float(m->vcache[base + i]);
                    }
                }
            }
            #pragma omp parallel for schedule(dynamic, 1)
            for (int th = 0; th < T * Hq; ++th) {
                const int t = th / Hq, h = th % Hq, g = h / group, p = p0 + t;
                int j0 = 0;
                if (m->window[l] > 0 && p + 1 > m->window[l]) j0 = p + 1 - m->window[l];
                int me = 0;
#ifdef _OPENMP
                me = omp_get_thread_num();
#endif
                const size_t base = (((size_t)l * Hkv + g) * (size_t)c->max_seq + (size_t)j0) * hd;
                orc_attend_head_f32(Yq + (size_t)t * Q + h * hd, kf + base, vf + base, p + 1 - j0, hd, scale,
                                    scr + (size_t)me * c->max_seq, A + (size_t)t * Q + h * hd);
            }
            orc_transpose_pad(A, T, Tp, Q, XT);
            orc_block_matvec(w->wo + (size_t)l * d * Q, XT, T, Tp, d, Q, Y);
            for (size_t i = 0; i < (size_t)T * d; ++i) X[i] = X[i] + Y[i];

            /* FFN block */
            for (int t = 0; t < T; ++t)
                orc_rmsnorm(X + (size_t)t * d, w->ffn_norm + (size_t)l * d, d, c->rms_eps, XN + (size_t)t * d);
            orc_transpose_pad(XN, T, Tp, d, XT);
            orc_block_matvec(w->w_gate + (size_t)l * F * d, XT, T, Tp, F, d, G);
            orc_block_matvec(w->w_up + (size_t)l * F * d, XT, T, Tp, F, d, U);
            for (size_t i = 0; i < (size_t)T * F; ++i) G[i] = orc_silu(G[i]) * U[i];
            orc_transpose_pad(G, T, Tp, F, XT);
            orc_block_matvec(w->w_down + (size_t)l * d * F, XT, T, Tp, d, F, Y);
            for (size_t i = 0; i < (size_t)T * d; ++i) X[i] = X[i] + Y[i];
        }
        m->pos = p0 + T;
    }
    if (rc == 0) m->pending = tokens[n - 1];
    free(X); free(XN); free(XT); free(Yq); free(Yk); free(Yv); free(A); free(G); free(U); free(Y); free(scr);
    free(kf); free(vf);
    return rc;
}

/* n_steps decode steps.  Step i runs the forward pass of the pending token at
 * position pos, chooses a token from its logits (orc_sample, keyed by that
 * position), writes it to out_tokens[i] and makes it the pending token -- or,
 * if force_tokens is not NULL, makes force_tokens[i] the pending token
 * instead (teacher forcing on a fixed input sequence).  If logits_out is not
 * NULL, step i's logits go to logits_out[i * V ...].  Returns 0 or -1. */
ORC_API int orc_decode(orc_model *m, int n_steps, float temperature, int top_k, uint64_t seed,
                       const int32_t *force_tokens, int32_t *out_tokens, float *logits_out)
{
    int V = m->c.vocab;
    if (m->pending < 0 || m->pos + n_steps > m->c.max_seq) return -1;
    float *lg = logits_out ? NULL : (float *)malloc(sizeof(float) * (size_t)V);
    for (int i = 0; i < n_steps; ++i) {
        float *dst = logits_out ? logits_out + (size_t)i * V : lg;
        int p = m->pos;
        if (orc_forward(m, m->pending, dst)) { free(lg); return -1; }
        int tok = orc_sample(dst, V, temperature, top_k, seed, p);
        out_tokens[i] = tok;
        m->pending = force_tokens ? force_tokens[i] : tok;
    }
    free(lg);
    return 0;
}
