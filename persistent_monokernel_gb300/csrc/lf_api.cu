// lf_api.cu -- host runtime behind include/lf.h: validation, the static work
// partition, allocation, the repack of the weights into per-CTA streams, the
// RoPE table, and the launches of the persistent kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/lf.h"
#include "lf_internal.cuh"
#include "lf_prefill.h"

extern "C" cudaError_t lfk_set_smem(int smem_bytes);
extern "C" cudaError_t lfk_launch_monokernel(const lfk::Params *p, int smem_bytes, cudaStream_t stream,
                                             int cooperative);
extern "C" cudaError_t lfk_occupancy(int smem_bytes, int *blocks_per_sm);
extern "C" unsigned lfk_smem_bytes(int ring_bytes, int a_floats, int lm_rows_max, int L);
extern "C" cudaError_t lfk_launch_mxfp4_interleave(const void *codes, const void *scales, size_t rows, int cols,
                                                   void *out, cudaStream_t stream);
extern "C" cudaError_t lfk_launch_repack(lfk::Geo g, int P, const lfk::CtaPlan *plans, const void *wq,
                                         const void *wk, const void *wv, const void *wo, const void *wg,
                                         const void *wu, const void *wd, const void *head, void *dst,
                                         cudaStream_t stream);

namespace {

constexpr int kAttnMinLen = 64;         // fewest positions per split-KV piece
constexpr long long kDefaultTimeoutNs = 2000000000LL;

// Tuning override of the shortest split-KV piece, LF_ATTN_MIN_LEN (positions).
int attn_min_len_from_env()
{
    const char *v = std::getenv("LF_ATTN_MIN_LEN");
    long n = v ? std::strtol(v, nullptr, 10) : kAttnMinLen;
    return n < 16 ? 16 : (n > (1 << 20) ? (1 << 20) : (int)n);
}

}  // namespace

struct lf_handle {
    lf_config cfg;
    lfk::Geo g;
    int P = 0, sm_count = 0;
    std::vector<lfk::CtaPlan> plans;
    lfk::CtaPlan *d_plans = nullptr;
    uint8_t *wstream = nullptr;
    size_t wstream_bytes = 0;
    const __half *embed = nullptr, *attn_norm = nullptr, *ffn_norm = nullptr, *final_norm = nullptr;
    __half *kc = nullptr, *vc = nullptr;
    float2 *rope = nullptr;
    float *qbuf = nullptr, *attn = nullptr, *xattn = nullptr, *hbuf = nullptr, *xout = nullptr, *apart = nullptr;
    float *kvf = nullptr;
    int *win = nullptr;            // [L] attention window per layer, or null (every layer: the whole cache)
    const __half *router = nullptr;  // mixture of experts: the caller's [L][E][d] router rows (read in place)
    float *wsc = nullptr;          // FP8 weights: copies of the eight per-row scale arrays, back to back
    size_t wsc_off[8] = {};
    int max_split = 1;
    unsigned *counters = nullptr;  // one allocation: slice counters, attn_done, lm_done, tok_cnt, gbar
    size_t counters_bytes = 0;
    unsigned *sig = nullptr, *attn_done = nullptr, *lm_done = nullptr, *tok_cnt = nullptr, *gbar = nullptr;
    unsigned long long *lm_part = nullptr;
    int *tok_buf = nullptr, *tok_seq = nullptr;
    unsigned *status = nullptr, *abort_flag = nullptr;
    int ring_bytes = 0, a_floats = 0, lm_rows_max = 0, smem_bytes = 0;
    // sequence state
    int pos = 0;
    int has_pending = 0;
    unsigned epoch = 0, tok_count = 0, gbar_count = 0;
    int sched = LF_SCHED_FLAGS;
    lf_status latched = LF_OK;
    cudaStream_t last_stream = nullptr;
    // lf_generate staging
    int32_t *stage_in = nullptr, *stage_out = nullptr;
    int stage_cap = 0;
    // optional stage trace
    unsigned long long *trace = nullptr;
    int trace_steps = 0;
    int attn_min_len = kAttnMinLen;
    // batched prefill (cfg.prefill_block != 0): row-major projection copy,
    // FP8 row scales in the same layout, workspace, token staging, cuBLAS
    int pf_block = 0;
    __half *pf_w = nullptr;
    float *pf_s = nullptr;
    uint8_t *pf_ws = nullptr;
    int *pf_tok = nullptr;
    lfp_maps pf_maps;              // TMA tensor maps of the prefill GEMM operands
    size_t pf_bytes = 0;
    size_t pf_woff[4] = {}, pf_soff[4] = {};   // [qkv, o, gu, d] element offsets
};

namespace {

template <class T>
cudaError_t dalloc(T **p, size_t count)
{
    return cudaMalloc(reinterpret_cast<void **>(p), std::max<size_t>(count, 1) * sizeof(T));
}

void free_all(lf_handle *h)
{
    void *ptrs[] = {h->d_plans, h->wstream, h->kc, h->vc, h->rope, h->qbuf, h->attn, h->xattn, h->hbuf,
                    h->xout, h->apart, h->kvf, h->win, h->wsc, h->counters, h->lm_part, h->tok_buf, h->tok_seq, h->status,
                    h->stage_in, h->stage_out, h->trace, h->pf_w, h->pf_s, h->pf_ws, h->pf_tok};
    for (void *p : ptrs)
        if (p) cudaFree(p);
}

// The activations between GEMV stages start as zeros whenever the pass count
// restarts: a zero carries the parity of no pass 0 value (the tags of
// lfk::Params::attn, xattn, hbuf, xout).
cudaError_t clear_activations(lf_handle *h)
{
    const lfk::Geo &g = h->g;
    cudaError_t e = cudaMemset(h->attn, 0, sizeof(float) * (size_t)g.L * g.Q);
    if (e == cudaSuccess) e = cudaMemset(h->qbuf, 0, sizeof(float) * (size_t)g.L * g.Q);
    if (e == cudaSuccess) e = cudaMemset(h->kvf, 0, sizeof(float) * (size_t)g.L * 2 * g.KV);
    if (e == cudaSuccess) e = cudaMemset(h->xattn, 0, sizeof(float) * (size_t)g.L * g.d);
    if (e == cudaSuccess) e = cudaMemset(h->hbuf, 0, sizeof(float) * (size_t)g.L * g.F);
    if (e == cudaSuccess) e = cudaMemset(h->xout, 0, sizeof(float) * (size_t)g.L * g.d);
    return e;
}

lf_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return LF_OK;
    if (e == cudaErrorMemoryAllocation) return LF_ERR_OUT_OF_MEMORY;
    if (e == cudaErrorCooperativeLaunchTooLarge) return LF_ERR_NOT_RESIDENT;
    return LF_ERR_CUDA;
}

lf_status validate_config(const lf_config &c)
{
    if (c.n_layers <= 0 || c.d_model <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 ||
        c.ffn_dim <= 0 || c.vocab <= 0 || c.max_seq <= 0 || !(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f) ||
        c.n_ctas < 0 || c.wait_timeout_ns < 0)
        return LF_ERR_INVALID_ARG;
    if (c.head_dim != 64 && c.head_dim != 128) return LF_ERR_NOT_SUPPORTED;
    if (c.n_heads % c.n_kv_heads != 0 || lfk::MAX_GROUP % (c.n_heads / c.n_kv_heads) != 0) return LF_ERR_NOT_SUPPORTED;
    const long long Q = (long long)c.n_heads * c.head_dim;
    if (c.d_model % lfk::KC || Q % lfk::KC || c.ffn_dim % lfk::KC) return LF_ERR_NOT_SUPPORTED;
    const long long most = (long long)lfk::MAX_SLICES * lfk::KC;
    if (c.d_model > most || Q > most || c.ffn_dim > most) return LF_ERR_NOT_SUPPORTED;
    if (c.layer_window)
        for (int l = 0; l < c.n_layers; ++l)
            if (c.layer_window[l] < 0) return LF_ERR_INVALID_ARG;
    if (c.weight_format != LF_WEIGHTS_FP16 && c.weight_format != LF_WEIGHTS_FP8_E4M3 &&
        c.weight_format != LF_WEIGHTS_MXFP4)
        return LF_ERR_NOT_SUPPORTED;
    if (c.prefill_block < LF_PREFILL_AUTO) return LF_ERR_INVALID_ARG;
    if (c.n_experts < 0 || c.top_k_experts < 0) return LF_ERR_INVALID_ARG;
    if (c.n_experts > 0) {
        // mixture of experts: up to 64 experts, 1..8 active, FP16 weights
        if (c.n_experts > lfk::MAX_EXPERTS || c.top_k_experts < 1 || c.top_k_experts > lfk::MAX_ACTIVE_EXPERTS ||
            c.top_k_experts > c.n_experts)
            return LF_ERR_NOT_SUPPORTED;
        if (c.weight_format != LF_WEIGHTS_FP16) return LF_ERR_NOT_SUPPORTED;
        if ((long long)c.top_k_experts * c.ffn_dim > (long long)lfk::MAX_SLICES * lfk::KC) return LF_ERR_NOT_SUPPORTED;
    }
    return LF_OK;
}

// The batched prefill's arguments that do not change between calls.
lfp_args prefill_args(const lf_handle *h)
{
    const lfk::Geo &g = h->g;
    lfp_args a;
    a.g = g;
    a.block = h->pf_block;
    a.n = 0;
    a.pos0 = 0;
    a.eps = h->cfg.rms_eps;
    a.tokens = h->pf_tok;
    a.embed = h->embed;
    a.attn_norm = h->attn_norm;
    a.ffn_norm = h->ffn_norm;
    a.wqkv = h->pf_w + h->pf_woff[0];
    a.wo = h->pf_w + h->pf_woff[1];
    a.wgu = h->pf_w + h->pf_woff[2];
    a.wd = h->pf_w + h->pf_woff[3];
    const bool fp8 = h->pf_s != nullptr;
    a.sqkv = fp8 ? h->pf_s + h->pf_soff[0] : nullptr;
    a.so = fp8 ? h->pf_s + h->pf_soff[1] : nullptr;
    a.sgu = fp8 ? h->pf_s + h->pf_soff[2] : nullptr;
    a.sd = fp8 ? h->pf_s + h->pf_soff[3] : nullptr;
    a.router = h->router;
    a.rope = h->rope;
    a.win = h->win;
    a.kc = h->kc;
    a.vc = h->vc;
    a.status = h->status;
    a.sms = h->sm_count;
    a.attn_stamps = h->trace_steps > 0 ? h->trace : nullptr;   // with tracing on: the prefill attention's stamps
    a.ws = lfp_carve(h->pf_ws, g, h->pf_block, h->sm_count);
    return a;
}

// Batched prefill state: the eight layer projections copied row-major as FP16
// into four stacked arrays [L, Q+2KV, d] (q, k, v rows), [L, d, Q],
// [L, 2F, d] (gate and up rows interleaved in blocks of 128 units, so that
// one 256-row GEMM tile holds a unit's gate and up rows) and [L, d, F] --
// FP8 models: the decoded codes, with the row scales gathered into the same
// row order -- plus the block workspace, a token staging buffer and the
// GEMMs' tensor maps.
lf_status setup_prefill(lf_handle *h, const lf_weights *w)
{
    const lfk::Geo &g = h->g;
    int block = h->cfg.prefill_block;
    if (block == LF_PREFILL_AUTO) {
        // The attention of a block runs (block / 128) x Hq CTAs, one per SM at a
        // time: the fraction of its waves' SM slots those fill is
        // n / (ceil(n / SMs) * SMs).  Take the largest block (a multiple of
        // 128, at most 1,024: larger blocks make better GEMMs) whose fill is at
        // least 80 % of the best block's.
        const int sms = std::max(1, h->sm_count);
        auto fill = [&](int b) {
            const long long n = (long long)(b / 128) * g.Hq;
            const long long waves = (n + sms - 1) / sms;
            return (double)n / (double)(waves * sms);
        };
        double best = 0.0;
        for (int b = 128; b <= 1024; b += 128) best = std::max(best, fill(b));
        block = 128;
        for (int b = 1024; b >= 128; b -= 128)
            if (fill(b) >= 0.8 * best) {
                block = b;
                break;
            }
    }
    h->pf_block = std::min(block, g.max_seq);
    const size_t L = g.L, d = g.d, Q = g.Q, KV = g.KV, F = g.F, NQKV = Q + 2 * KV;
    // mixture of experts: gate/up [L][E][2 Fe][d] and down [L][E][d][Fe]
    const size_t nexp = (size_t)lfk::n_expert_parts(g), Fw = g.E > 0 ? (size_t)g.Fe : F;
    const size_t wlen[4] = {L * NQKV * d, L * d * Q, L * nexp * 2 * Fw * d, L * nexp * d * Fw};
    const size_t slen[4] = {L * NQKV, L * d, L * 2 * F, L * d};
    size_t wt = 0, st = 0;
    for (int i = 0; i < 4; ++i) {
        h->pf_woff[i] = wt;
        h->pf_soff[i] = st;
        wt += wlen[i];
        st += slen[i];
    }
    const bool fp8 = g.fmt == lfk::FMT_FP8, mx = g.fmt == lfk::FMT_MXFP4;
    const void *bsc[7] = {w->wq_scale, w->wk_scale, w->wv_scale, w->wo_scale, w->w_gate_scale, w->w_up_scale,
                          w->w_down_scale};
    if (mx) {
        // the FP16 copy is exact only for block scales 2^-23 .. 2^13 (E 104 .. 140)
        const size_t nsc[7] = {L * Q * d / 32, L * KV * d / 32, L * KV * d / 32, L * d * Q / 32,
                               L * F * d / 32, L * F * d / 32, L * d * F / 32};
        for (int i = 0; i < 7; ++i) {
            unsigned lo = 0, hi = 0;
            const cudaError_t er = lfp_byte_range(static_cast<const uint8_t *>(bsc[i]), nsc[i], &lo, &hi);
            if (er != cudaSuccess) return from_cuda(er);
            if (lo < 104u || hi > 140u) return LF_ERR_NOT_SUPPORTED;
        }
    }
    const size_t ws_bytes = lfp_workspace_bytes(g, h->pf_block, h->sm_count);
    cudaError_t e = dalloc(&h->pf_w, wt);
    if (e == cudaSuccess && fp8) e = dalloc(&h->pf_s, st);
    if (e == cudaSuccess) e = dalloc(&h->pf_ws, ws_bytes);
    if (e == cudaSuccess) e = dalloc(&h->pf_tok, (size_t)g.max_seq);
    if (e != cudaSuccess) return from_cuda(e);
    h->pf_bytes = wt * sizeof(__half) + (fp8 ? st * sizeof(float) : 0) + ws_bytes + (size_t)g.max_seq * sizeof(int);
    // A [units, cols] matrix (gate or up rows) into the interleaved gate/up
    // layout: its rows of units 128b .. 128b+127 go to rows 256b + half*128 ..
    // (elem bytes per value: 2 for the FP16 weights, 4 for the FP8 row scales).
    auto interleave = [](void *dst, const void *src, size_t units, size_t cols, size_t elem, int half) {
        const size_t blk = 128 * cols * elem;
        return cudaMemcpy2D(static_cast<uint8_t *>(dst) + (size_t)half * blk, 2 * blk, src, blk, blk, units / 128,
                            cudaMemcpyDeviceToDevice);
    };
    if (g.E > 0 && e == cudaSuccess) {
        // each expert's gate and up rows interleaved; the down projections in the caller's layout
        const size_t ge = Fw * d;
        for (size_t le = 0; le < L * nexp && e == cudaSuccess; ++le) {
            __half *dst = h->pf_w + h->pf_woff[2] + le * 2 * ge;
            e = interleave(dst, static_cast<const __half *>(w->w_gate) + le * ge, Fw, d, sizeof(__half), 0);
            if (e == cudaSuccess)
                e = interleave(dst, static_cast<const __half *>(w->w_up) + le * ge, Fw, d, sizeof(__half), 1);
        }
        if (e == cudaSuccess)
            e = cudaMemcpy(h->pf_w + h->pf_woff[3], w->w_down, wlen[3] * sizeof(__half), cudaMemcpyDeviceToDevice);
    }
    // per matrix: source, rows, cols, destination array, row offset inside a
    // layer (gate/up: which half of the interleaved blocks)
    struct Part {
        const void *src;
        size_t rows, cols;
        int arr;
        size_t row0;
    };
    const Part parts[7] = {{w->wq, Q, d, 0, 0},      {w->wk, KV, d, 0, Q},     {w->wv, KV, d, 0, Q + KV},
                           {w->wo, d, Q, 1, 0},      {w->w_gate, F, d, 2, 0},  {w->w_up, F, d, 2, 1},
                           {w->w_down, d, F, 3, 0}};
    const size_t arr_rows[4] = {NQKV, d, 2 * F, d};
    __half *tmp = nullptr;   // decoded gate/up matrix of one layer before interleaving (FP8, MXFP4)
    if (g.E == 0 && (fp8 || mx) && e == cudaSuccess) e = dalloc(&tmp, F * d);
    for (int i = 0; i < (g.E > 0 ? 4 : 7) && e == cudaSuccess; ++i) {
        const Part &pt = parts[i];
        const size_t n = pt.rows * pt.cols;
        const bool gu = pt.arr == 2;
        for (size_t l = 0; l < L && e == cudaSuccess; ++l) {
            __half *layer = h->pf_w + h->pf_woff[pt.arr] + l * arr_rows[pt.arr] * pt.cols;
            __half *dst = gu ? tmp : layer + pt.row0 * pt.cols;
            if (mx) {
                e = lfp_decode_mxfp4(static_cast<const uint8_t *>(pt.src) + l * n / 2,
                                     static_cast<const uint8_t *>(bsc[i]) + l * n / 32, pt.rows, (int)pt.cols, dst,
                                     nullptr);
            } else if (fp8) {
                e = lfp_decode_e4m3(static_cast<const uint8_t *>(pt.src) + l * n, dst, n, nullptr);
                const float *ssrc = h->wsc + h->wsc_off[i] + l * pt.rows;
                float *sl = h->pf_s + h->pf_soff[pt.arr] + l * arr_rows[pt.arr];
                if (e == cudaSuccess)
                    e = gu ? interleave(sl, ssrc, pt.rows, 1, sizeof(float), (int)pt.row0)
                           : cudaMemcpy(sl + pt.row0, ssrc, pt.rows * sizeof(float), cudaMemcpyDeviceToDevice);
            } else if (gu) {
                e = interleave(layer, static_cast<const __half *>(pt.src) + l * n, pt.rows, pt.cols, sizeof(__half),
                               (int)pt.row0);
            } else {
                e = cudaMemcpy(dst, static_cast<const __half *>(pt.src) + l * n, n * sizeof(__half),
                               cudaMemcpyDeviceToDevice);
            }
            if (e == cudaSuccess && gu && (fp8 || mx))
                e = interleave(layer, tmp, pt.rows, pt.cols, sizeof(__half), (int)pt.row0);
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (tmp) cudaFree(tmp);
    if (e != cudaSuccess) return from_cuda(e);
    lfp_args a = prefill_args(h);
    e = cudaMemset(a.ws.tile_cnt, 0, 1024 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    if (lfp_make_maps(&a, &h->pf_maps) != 0) return LF_ERR_CUDA;
    return LF_OK;
}

lf_status launch(lf_handle *h, const lfk::Params &p, cudaStream_t stream)
{
    const int coop = (p.sched == lfk::SCHED_MULTI) ? 0 : 1;
    cudaError_t e = lfk_launch_monokernel(&p, h->smem_bytes, stream, coop);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return from_cuda(e);
    }
    return LF_OK;
}

lfk::Params base_params(lf_handle *h)
{
    lfk::Params p;
    std::memset(&p, 0, sizeof(p));
    p.g = h->g;
    p.P = h->P;
    p.eps = h->cfg.rms_eps;
    p.plans = h->d_plans;
    p.wstream = h->wstream;
    p.embed = h->embed;
    p.attn_norm = h->attn_norm;
    p.ffn_norm = h->ffn_norm;
    p.final_norm = h->final_norm;
    p.kc = h->kc;
    p.vc = h->vc;
    p.rope = h->rope;
    p.qbuf = h->qbuf;
    p.attn = h->attn;
    p.xattn = h->xattn;
    p.hbuf = h->hbuf;
    p.xout = h->xout;
    p.apart = h->apart;
    p.kvf = h->kvf;
    p.win = h->win;
    p.router = h->router;
    for (int i = 0; i < 8; ++i) p.wsc[i] = h->wsc ? h->wsc + h->wsc_off[i] : nullptr;
    p.max_split = h->max_split;
    p.sig = h->sig;
    p.attn_done = h->attn_done;
    p.lm_done = h->lm_done;
    p.tok_cnt = h->tok_cnt;
    p.gbar = h->gbar;
    p.lm_part = h->lm_part;
    p.tok_buf = h->tok_buf;
    p.tok_seq = h->tok_seq;
    p.status = h->status;
    p.abort_flag = h->abort_flag;
    p.timeout_ns = h->cfg.wait_timeout_ns > 0 ? h->cfg.wait_timeout_ns : kDefaultTimeoutNs;
    p.fault_step = h->cfg.fault_step;
    p.ring_bytes = h->ring_bytes;
    p.a_floats = h->a_floats;
    p.lm_rows_max = h->lm_rows_max;
    p.attn_min_len = h->attn_min_len;
    p.sched = h->sched;
    p.only_layer = -1;
    p.only_stage = -1;
    p.trace = h->trace;
    p.trace_steps = h->trace_steps;
    return p;
}

// Runs the steps of one prefill or decode call under the current schedule.
lf_status run_steps(lf_handle *h, lfk::Params p, cudaStream_t stream)
{
    if (p.sched != lfk::SCHED_MULTI) return launch(h, p, stream);
    // multi-kernel ablation: one launch per (step, layer, stage) + one for the LM head
    const int L = h->g.L;
    const int n = p.n_steps;
    for (int i = 0; i < n; ++i) {
        lfk::Params q = p;
        q.n_steps = 1;
        q.pos0 = p.pos0 + i;
        q.epoch0 = p.epoch0 + (unsigned)i;
        q.tok_base = p.tok_base + (unsigned)i;
        q.fault_step = -1;
        q.trace = nullptr;
        if (p.mode == lfk::MODE_PREFILL) {
            q.has_pending = (p.has_pending && i == 0) ? 1 : 0;
            q.prompt = p.prompt + (i - (p.has_pending ? 1 : 0));
            if (q.has_pending) q.prompt = p.prompt;
        } else {
            q.out_tokens = p.out_tokens + i;
            q.debug_logits = p.debug_logits ? p.debug_logits + (size_t)i * h->g.V : nullptr;
            q.force_tokens = p.force_tokens ? p.force_tokens + i : nullptr;
        }
        for (int l = 0; l < L; ++l) {
            for (int s = 0; s < 5; ++s) {
                q.only_layer = l;
                q.only_stage = s;
                lf_status st = launch(h, q, stream);
                if (st != LF_OK) return st;
            }
        }
        if (p.mode == lfk::MODE_DECODE) {
            q.only_layer = 0;
            q.only_stage = 5;
            lf_status st = launch(h, q, stream);
            if (st != LF_OK) return st;
        }
    }
    return LF_OK;
}

}  // namespace

extern "C" {

int32_t lf_abi_version(void) { return LF_ABI_VERSION; }

const char *lf_error_string(lf_status s)
{
    switch (s) {
    case LF_OK: return "LF_OK";
    case LF_ERR_INVALID_ARG: return "LF_ERR_INVALID_ARG: invalid argument";
    case LF_ERR_OUT_OF_MEMORY: return "LF_ERR_OUT_OF_MEMORY: allocation failed";
    case LF_ERR_CAPACITY: return "LF_ERR_CAPACITY: not enough KV-cache positions left";
    case LF_ERR_NOT_RESIDENT: return "LF_ERR_NOT_RESIDENT: the persistent grid cannot be co-resident";
    case LF_ERR_CUDA: return "LF_ERR_CUDA: a CUDA runtime call failed";
    case LF_ERR_TIMEOUT: return "LF_ERR_TIMEOUT: a device-side wait ran out";
    case LF_ERR_NOT_SUPPORTED: return "LF_ERR_NOT_SUPPORTED: shape or option not supported";
    case LF_ERR_STATE: return "LF_ERR_STATE: call not valid in the current state";
    }
    return "unknown lf_status";
}

lf_status lf_create(const lf_config *cfg, const lf_weights *w, lf_handle **out)
{
    if (!cfg || !w || !out) return LF_ERR_INVALID_ARG;
    *out = nullptr;
    lf_status st = validate_config(*cfg);
    if (st != LF_OK) return st;
    const void *need[] = {w->embed, w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm,
                          w->w_gate, w->w_up, w->w_down, w->final_norm, w->lm_head};
    for (const void *p : need)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return LF_ERR_INVALID_ARG;   // bulk copies need 16 B
    if (cfg->n_experts > 0 ? (!w->w_router || (reinterpret_cast<uintptr_t>(w->w_router) & 15u)) : w->w_router != nullptr)
        return LF_ERR_INVALID_ARG;
    const bool fp8 = cfg->weight_format == LF_WEIGHTS_FP8_E4M3;
    const bool mxfp4 = cfg->weight_format == LF_WEIGHTS_MXFP4;
    const void *scales_v[8] = {w->wq_scale, w->wk_scale, w->wv_scale, w->wo_scale,
                               w->w_gate_scale, w->w_up_scale, w->w_down_scale, w->lm_head_scale};
    const float *scales[8];
    for (int i = 0; i < 8; ++i) {
        const void *p = scales_v[i];
        scales[i] = static_cast<const float *>(p);
        // FP8: FP32 row scales (4-byte aligned); MXFP4: E8M0 block scales (bytes); FP16: none
        if (fp8 ? (!p || (reinterpret_cast<uintptr_t>(p) & 3u)) : mxfp4 ? !p : p != nullptr)
            return LF_ERR_INVALID_ARG;
    }

    lf_handle *h = new (std::nothrow) lf_handle();
    if (!h) return LF_ERR_OUT_OF_MEMORY;
    h->cfg = *cfg;
    h->cfg.layer_window = nullptr;   // the caller's array is copied to the device below
    h->attn_min_len = attn_min_len_from_env();
    lfk::Geo &g = h->g;
    g.L = cfg->n_layers;
    g.d = cfg->d_model;
    g.Hq = cfg->n_heads;
    g.Hkv = cfg->n_kv_heads;
    g.hd = cfg->head_dim;
    g.E = cfg->n_experts;
    g.topk = g.E > 0 ? cfg->top_k_experts : 1;
    g.Fe = cfg->ffn_dim;
    g.F = g.topk * g.Fe;
    g.V = cfg->vocab;
    g.Q = g.Hq * g.hd;
    g.KV = g.Hkv * g.hd;
    g.group = g.Hq / g.Hkv;
    g.max_seq = cfg->max_seq;
    g.fmt = fp8 ? lfk::FMT_FP8 : mxfp4 ? lfk::FMT_MXFP4 : lfk::FMT_FP16;
    g.crb = lfk::fmt_crb(g.fmt);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
    int optin = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        delete h;
        return from_cuda(e);
    }

    // ---- grid size: one CTA per SM, and every CTA owns rows of every GEMV stage
    int P = cfg->n_ctas > 0 ? std::min(cfg->n_ctas, h->sm_count) : h->sm_count;
    for (int s = 0; s < lfk::N_GEMV; ++s) P = std::min(P, lfk::stage_geom(g, s).units);
    h->P = P;

    // ---- static partition and per-CTA stream offsets
    h->plans.resize(P);
    unsigned long long base = 0;
    int lm_rows_max = 0;
    for (int b = 0; b < P; ++b) {
        lfk::CtaPlan &pl = h->plans[b];
        for (int s = 0; s < lfk::N_GEMV; ++s) {
            const int U = lfk::stage_geom(g, s).units;
            pl.u0[s] = lfk::cta_unit_start(U, P, b);
            pl.u1[s] = lfk::cta_unit_start(U, P, b + 1);
        }
        unsigned long long off = 0;
        for (int s = 0; s < 4; ++s) {
            const lfk::StageGeom sg = lfk::stage_geom(g, s);
            pl.stage_off[s] = off;
            // gate/up and down hold every expert's rows (down: Fe columns each)
            const int nexp = (s == lfk::ST_GU || s == lfk::ST_D) ? lfk::n_expert_parts(g) : 1;
            const int kcols = s == lfk::ST_D ? g.Fe : sg.K;
            off += (unsigned long long)nexp * (pl.u1[s] - pl.u0[s]) * sg.rows_per_unit * (kcols / lfk::KC) *
                   (unsigned long long)g.crb;
        }
        pl.layer_bytes = off;
        pl.lm_off = off * (unsigned long long)g.L;
        const unsigned long long lm_bytes =
            (unsigned long long)(pl.u1[lfk::ST_LM] - pl.u0[lfk::ST_LM]) * (g.d / lfk::KC) * (unsigned long long)g.crb;
        pl.base = base;
        base += pl.lm_off + lm_bytes;
        lm_rows_max = std::max(lm_rows_max, pl.u1[lfk::ST_LM] - pl.u0[lfk::ST_LM]);
    }
    h->wstream_bytes = base;
    h->lm_rows_max = lm_rows_max;

    // ---- shared memory: everything but the ring, then the largest ring that fits
    h->max_split = std::max(1, P / g.Hkv);
    h->a_floats = lfk::scratch_floats(g, h->max_split);
    const unsigned rest = lfk_smem_bytes(0, h->a_floats, lm_rows_max, g.L);
    if ((int)rest + 2 * lfk::ATT_CHUNK_BYTES > optin) {
        delete h;
        return LF_ERR_NOT_SUPPORTED;
    }
    h->ring_bytes = (int)(((unsigned)optin - rest) / 1024u * 1024u);
    while ((int)lfk_smem_bytes(h->ring_bytes, h->a_floats, lm_rows_max, g.L) > optin)
        h->ring_bytes -= 1024;
    h->smem_bytes = (int)lfk_smem_bytes(h->ring_bytes, h->a_floats, lm_rows_max, g.L);
    if (h->ring_bytes < 2 * lfk::ATT_CHUNK_BYTES) {
        delete h;
        return LF_ERR_NOT_SUPPORTED;
    }
    int per_sm = 0;
    e = lfk_occupancy(h->smem_bytes, &per_sm);
    if (e != cudaSuccess) {
        delete h;
        return from_cuda(e);
    }
    if (per_sm < 1 || per_sm * h->sm_count < P) {
        delete h;
        return LF_ERR_NOT_RESIDENT;
    }

    // ---- allocations
    const size_t kv_elems = (size_t)g.L * g.Hkv * (size_t)g.max_seq * g.hd;
    const size_t sig_words = (size_t)g.L * lfk::sig_layout(g).per_layer * lfk::SIG_STRIDE;
    const size_t n_attn_done = (size_t)g.L * g.Hkv;
    const size_t n_words = sig_words + (n_attn_done + 3) * lfk::CNT_STRIDE;
    h->counters_bytes = n_words * sizeof(unsigned);
    if ((e = dalloc(&h->d_plans, (size_t)P)) != cudaSuccess || (e = dalloc(&h->wstream, h->wstream_bytes)) != cudaSuccess ||
        (e = dalloc(&h->kc, kv_elems)) != cudaSuccess || (e = dalloc(&h->vc, kv_elems)) != cudaSuccess ||
        (e = dalloc(&h->rope, (size_t)g.max_seq * (g.hd / 2))) != cudaSuccess ||
        (e = dalloc(&h->qbuf, (size_t)g.L * g.Q)) != cudaSuccess ||
        (e = dalloc(&h->attn, (size_t)g.L * g.Q)) != cudaSuccess ||
        (e = dalloc(&h->xattn, (size_t)g.L * g.d)) != cudaSuccess ||
        (e = dalloc(&h->hbuf, (size_t)g.L * g.F)) != cudaSuccess ||
        (e = dalloc(&h->xout, (size_t)g.L * g.d)) != cudaSuccess ||
        (e = dalloc(&h->apart, (size_t)g.L * g.Hq * h->max_split * (g.hd + 2))) != cudaSuccess ||
        (e = dalloc(&h->kvf, (size_t)g.L * 2 * g.KV)) != cudaSuccess ||
        (e = dalloc(&h->counters, n_words)) != cudaSuccess ||
        (e = dalloc(&h->lm_part, (size_t)P * lfk::MAX_TOPK)) != cudaSuccess ||
        (e = dalloc(&h->tok_buf, 1)) != cudaSuccess || (e = dalloc(&h->tok_seq, (size_t)g.max_seq)) != cudaSuccess ||
        (e = dalloc(&h->status, 8)) != cudaSuccess) {
        free_all(h);
        delete h;
        return from_cuda(e);
    }
    if (fp8) {
        const size_t rows[8] = {(size_t)g.L * g.Q, (size_t)g.L * g.KV, (size_t)g.L * g.KV, (size_t)g.L * g.d,
                                (size_t)g.L * g.F, (size_t)g.L * g.F, (size_t)g.L * g.d, (size_t)g.V};
        size_t total = 0;
        for (int i = 0; i < 8; ++i) {
            h->wsc_off[i] = total;
            total += rows[i];
        }
        e = dalloc(&h->wsc, total);
        for (int i = 0; i < 8 && e == cudaSuccess; ++i)
            e = cudaMemcpy(h->wsc + h->wsc_off[i], scales[i], rows[i] * sizeof(float), cudaMemcpyDeviceToDevice);
        if (e != cudaSuccess) {
            free_all(h);
            delete h;
            return from_cuda(e);
        }
    }
    bool windowed = false;
    if (cfg->layer_window)
        for (int l = 0; l < g.L; ++l) windowed = windowed || cfg->layer_window[l] > 0;
    if (windowed) {
        e = dalloc(&h->win, (size_t)g.L);
        if (e == cudaSuccess) e = cudaMemcpy(h->win, cfg->layer_window, sizeof(int) * g.L, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            free_all(h);
            delete h;
            return from_cuda(e);
        }
    }
    h->sig = h->counters;
    h->attn_done = h->counters + sig_words;
    h->lm_done = h->attn_done + n_attn_done * lfk::CNT_STRIDE;
    h->tok_cnt = h->lm_done + lfk::CNT_STRIDE;
    h->gbar = h->tok_cnt + lfk::CNT_STRIDE;
    h->abort_flag = h->status + 4;
    h->embed = static_cast<const __half *>(w->embed);
    h->router = static_cast<const __half *>(w->w_router);
    h->attn_norm = static_cast<const __half *>(w->attn_norm);
    h->ffn_norm = static_cast<const __half *>(w->ffn_norm);
    h->final_norm = static_cast<const __half *>(w->final_norm);

    // ---- RoPE table: theta_i = pos * base^(-2i/hd) in double, cos/sin rounded to FP32
    std::vector<float2> rope((size_t)g.max_seq * (g.hd / 2));
    for (int pos = 0; pos < g.max_seq; ++pos)
        for (int i = 0; i < g.hd / 2; ++i) {
            const double inv_freq = std::pow((double)cfg->rope_theta, -2.0 * (double)i / (double)g.hd);
            const double ang = (double)pos * inv_freq;
            rope[(size_t)pos * (g.hd / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    e = cudaMemcpy(h->rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->d_plans, h->plans.data(), P * sizeof(lfk::CtaPlan), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(h->counters, 0, h->counters_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, 8 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(h->tok_buf, 0, sizeof(int));
    if (e == cudaSuccess) e = clear_activations(h);
    // the cache starts as zeros: rows past the current position are finite when a
    // prefill attention chunk reads them (their probabilities are 0)
    if (e == cudaSuccess) e = cudaMemset(h->kc, 0, kv_elems * sizeof(__half));
    if (e == cudaSuccess) e = cudaMemset(h->vc, 0, kv_elems * sizeof(__half));
    if (e == cudaSuccess && !mxfp4)
        e = lfk_launch_repack(g, P, h->d_plans, w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down,
                              w->lm_head, h->wstream, nullptr);
    if (e == cudaSuccess && mxfp4) {
        // codes and block scales -> rows of 144-byte column groups (temporary), then the usual repack
        const void *codes[8] = {w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down, w->lm_head};
        const size_t rows[8] = {(size_t)g.L * g.Q, (size_t)g.L * g.KV, (size_t)g.L * g.KV, (size_t)g.L * g.d,
                                (size_t)g.L * g.F, (size_t)g.L * g.F, (size_t)g.L * g.d, (size_t)g.V};
        const int cols[8] = {g.d, g.d, g.d, g.Q, g.d, g.d, g.F, g.d};
        uint8_t *tmp[8] = {};
        for (int i = 0; i < 8 && e == cudaSuccess; ++i) {
            e = dalloc(&tmp[i], rows[i] * (size_t)(cols[i] / lfk::KC) * (size_t)g.crb);
            if (e == cudaSuccess) e = lfk_launch_mxfp4_interleave(codes[i], scales_v[i], rows[i], cols[i], tmp[i], nullptr);
        }
        if (e == cudaSuccess)
            e = lfk_launch_repack(g, P, h->d_plans, tmp[0], tmp[1], tmp[2], tmp[3], tmp[4], tmp[5], tmp[6], tmp[7],
                                  h->wstream, nullptr);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        for (uint8_t *t : tmp)
            if (t) cudaFree(t);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = lfk_set_smem(h->smem_bytes);
    if (e != cudaSuccess) {
        free_all(h);
        delete h;
        return from_cuda(e);
    }
    if (cfg->prefill_block != 0) {
        st = setup_prefill(h, w);
        if (st != LF_OK) {
            free_all(h);
            delete h;
            return st;
        }
    }
    *out = h;
    return LF_OK;
}

void lf_destroy(lf_handle *h)
{
    if (!h) return;
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
}

lf_status lf_prefill(lf_handle *h, const int32_t *tokens_dev, int32_t n, void *stream)
{
    if (!h || !tokens_dev || n < 1) return LF_ERR_INVALID_ARG;
    if (h->latched != LF_OK) return LF_ERR_STATE;
    const int steps = (h->has_pending ? 1 : 0) + n - 1;
    if ((long long)h->pos + steps + 1 > h->g.max_seq) return LF_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (steps > 0 && h->pf_block > 0) {
        // batched: the pending token, then tokens_dev[0 .. n-2]
        const int hp = h->has_pending ? 1 : 0;
        cudaError_t e = cudaSuccess;
        if (hp) e = cudaMemcpyAsync(h->pf_tok, h->tok_buf, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess && n > 1)
            e = cudaMemcpyAsync(h->pf_tok + hp, tokens_dev, sizeof(int32_t) * (size_t)(n - 1),
                                cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return from_cuda(e);
        lfp_args a = prefill_args(h);
        a.n = steps;
        a.pos0 = h->pos;
        if (lfp_run(&a, &h->pf_maps, s) != 0) return LF_ERR_CUDA;
        h->pos += steps;   // the monokernel's counters and epoch are untouched
    } else if (steps > 0) {
        lfk::Params p = base_params(h);
        p.mode = lfk::MODE_PREFILL;
        p.n_steps = steps;
        p.pos0 = h->pos;
        p.has_pending = h->has_pending;
        p.prompt = tokens_dev;
        p.epoch0 = h->epoch;
        p.tok_base = h->tok_count;
        p.gbar_base = h->gbar_count;
        p.fault_step = -1;
        lf_status st = run_steps(h, p, s);
        if (st != LF_OK) return st;
        h->epoch += (unsigned)steps;
        h->pos += steps;
        if (h->sched == LF_SCHED_GRID_BARRIER) h->gbar_count += (unsigned)steps * 5u * (unsigned)h->g.L;
    }
    cudaError_t e = cudaMemcpyAsync(h->tok_buf, tokens_dev + (n - 1), sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return from_cuda(e);
    h->has_pending = 1;
    h->last_stream = s;
    return LF_OK;
}

lf_status lf_decode(lf_handle *h, int32_t n_steps, const lf_sampling *sp, uint64_t seed, int32_t *out_tokens_dev,
                    void *stream)
{
    if (!h || !sp || !out_tokens_dev || n_steps < 1) return LF_ERR_INVALID_ARG;
    if (sp->top_k < 0 || sp->top_k > LF_MAX_TOP_K) return LF_ERR_NOT_SUPPORTED;
    if (h->latched != LF_OK || !h->has_pending) return LF_ERR_STATE;
    if ((long long)h->pos + n_steps > h->g.max_seq) return LF_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    lfk::Params p = base_params(h);
    p.mode = lfk::MODE_DECODE;
    p.n_steps = n_steps;
    p.pos0 = h->pos;
    p.out_tokens = out_tokens_dev;
    p.debug_logits = sp->debug_logits_dev;
    p.force_tokens = sp->force_tokens_dev;
    p.temperature = sp->temperature;
    p.top_k = sp->top_k;
    p.seed = seed;
    p.epoch0 = h->epoch;
    p.tok_base = h->tok_count;
    p.gbar_base = h->gbar_count;
    lf_status st = run_steps(h, p, s);
    if (st != LF_OK) return st;
    h->epoch += (unsigned)n_steps;
    h->tok_count += (unsigned)n_steps;
    h->pos += n_steps;
    if (h->sched == LF_SCHED_GRID_BARRIER) h->gbar_count += (unsigned)n_steps * (5u * (unsigned)h->g.L + 1u);
    h->last_stream = s;
    return LF_OK;
}

lf_status lf_sync(lf_handle *h)
{
    if (!h) return LF_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(h->last_stream);
    if (e != cudaSuccess) return from_cuda(e);
    unsigned st[4] = {0, 0, 0, 0};
    e = cudaMemcpy(st, h->status, sizeof(st), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (st[0] == (unsigned)lfk::STATUS_TIMEOUT) h->latched = LF_ERR_TIMEOUT;
    else if (st[0] != 0u) h->latched = LF_ERR_INVALID_ARG;
    return h->latched;
}

lf_status lf_reset(lf_handle *h)
{
    if (!h) return LF_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(h->counters, 0, h->counters_bytes);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, 8 * sizeof(unsigned));
    if (e == cudaSuccess) e = clear_activations(h);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    h->pos = 0;
    h->has_pending = 0;
    h->epoch = h->tok_count = h->gbar_count = 0;
    h->latched = LF_OK;
    return LF_OK;
}

lf_status lf_set_schedule(lf_handle *h, int32_t schedule)
{
    if (!h) return LF_ERR_INVALID_ARG;
    if (schedule != LF_SCHED_FLAGS && schedule != LF_SCHED_GRID_BARRIER && schedule != LF_SCHED_MULTI_KERNEL)
        return LF_ERR_INVALID_ARG;
    // the expert choice lives in shared memory for the rest of the launch
    if (schedule == LF_SCHED_MULTI_KERNEL && h->g.E > 0) return LF_ERR_NOT_SUPPORTED;
    h->sched = schedule;
    return LF_OK;
}

lf_status lf_get_info(const lf_handle *h, lf_info *out)
{
    if (!h || !out) return LF_ERR_INVALID_ARG;
    out->n_ctas = h->P;
    out->threads_per_cta = lfk::NTHREADS;
    out->smem_bytes = h->smem_bytes;
    out->ring_bytes = h->ring_bytes;
    out->sm_count = h->sm_count;
    out->position = h->pos;
    out->has_pending = h->has_pending;
    out->schedule = h->sched;
    out->weight_stream_bytes = (int64_t)h->wstream_bytes;
    out->kv_cache_bytes = (int64_t)(2ull * h->g.L * h->g.Hkv * (size_t)h->g.max_seq * h->g.hd * 2ull);
    out->prefill_block = h->pf_block;
    out->prefill_bytes = (int64_t)h->pf_bytes;
    return LF_OK;
}

lf_status lf_generate(lf_handle *h, const int32_t *prompt_host, int32_t n_prompt, int32_t n_steps,
                      const lf_sampling *sp, uint64_t seed, int32_t *out_host, void *stream)
{
    if (!h || !prompt_host || !out_host || !sp || n_prompt < 1 || n_steps < 1) return LF_ERR_INVALID_ARG;
    const int need = std::max(n_prompt, n_steps);
    if (need > h->stage_cap) {
        if (h->stage_in) cudaFree(h->stage_in);
        if (h->stage_out) cudaFree(h->stage_out);
        h->stage_in = h->stage_out = nullptr;
        h->stage_cap = 0;
        cudaError_t e = dalloc(&h->stage_in, (size_t)need);
        if (e == cudaSuccess) e = dalloc(&h->stage_out, (size_t)need);
        if (e != cudaSuccess) return from_cuda(e);
        h->stage_cap = need;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(h->stage_in, prompt_host, sizeof(int32_t) * n_prompt, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return from_cuda(e);
    lf_status st = lf_prefill(h, h->stage_in, n_prompt, stream);
    if (st != LF_OK) return st;
    st = lf_decode(h, n_steps, sp, seed, h->stage_out, stream);
    if (st != LF_OK) return st;
    e = cudaMemcpyAsync(out_host, h->stage_out, sizeof(int32_t) * n_steps, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return from_cuda(e);
    return lf_sync(h);
}

}  // extern "C"

extern "C" {

lf_status lf_enable_trace(lf_handle *h, int32_t max_steps)
{
    if (!h || max_steps < 0) return LF_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    if (h->trace) cudaFree(h->trace);
    h->trace = nullptr;
    h->trace_steps = 0;
    if (max_steps == 0) return LF_OK;
    const size_t n = (size_t)max_steps * lfk::trace_slots(h->g.L) * h->P * lfk::TR_N;
    e = dalloc(&h->trace, n);
    if (e == cudaSuccess) e = cudaMemset(h->trace, 0, n * sizeof(unsigned long long));
    if (e != cudaSuccess) return from_cuda(e);
    h->trace_steps = max_steps;
    return LF_OK;
}

lf_status lf_read_trace(lf_handle *h, uint64_t *host_out, int64_t capacity, int64_t *n_out)
{
    if (!h || !n_out) return LF_ERR_INVALID_ARG;
    const size_t n = h->trace ? (size_t)h->trace_steps * lfk::trace_slots(h->g.L) * h->P * lfk::TR_N : 0;
    *n_out = (int64_t)n;
    if (!host_out) return LF_OK;
    if (capacity < (int64_t)n) return LF_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess && n) e = cudaMemcpy(host_out, h->trace, n * sizeof(uint64_t), cudaMemcpyDeviceToHost);
    return from_cuda(e);
}

}  // extern "C"
