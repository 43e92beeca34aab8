// lf_noalloc.cu -- lf_generate_noalloc: one prefill + decode request that
// allocates no device memory.
//
// Some callers cannot call cudaMalloc at request time: a plugin running inside
// a host framework that owns every device allocation through its own pool, code
// that must not touch the allocator while other work is being captured or
// replayed, or a process whose device memory is fully reserved up front.  For
// them this file keeps all scratch of one request -- the static work
// partition, the RoPE table, the FP16 KV cache, the per-layer activations, the
// readiness counters, the attention partials and the sampling candidates -- in
// one file-scope __device__ array of LF_NOALLOC_SCRATCH_BYTES, and streams the
// weights straight from the caller's row-major buffers (no repacked copy).
//
// Set-up: the first call on a device looks up the array's device address with
// cudaGetSymbolAddress (with that device current) and caches it; that first
// call should therefore come before any stream capture.  Every later call on
// the device reuses the same array, which keeps the previous call's contents;
// each call clears the counters and status words it relies on.  Calls whose
// work overlaps on the GPU race on the array, and so do calls from two host
// threads at once -- also on two different GPUs, since the host staging
// buffers below are shared by the whole process: serialise them.  Once any
// work is queued, every error return first synchronizes the stream, so that
// no queued copy or kernel still uses the array when the call returns.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "../../include/lf.h"
#include "lf_internal.cuh"

extern "C" unsigned lfk_smem_bytes(int ring_bytes, int a_floats, int lm_rows_max, int L);
extern "C" cudaError_t lfk_set_smem_direct(int smem_bytes);
extern "C" cudaError_t lfk_launch_monokernel_direct(const lfk::Params *p, const void *wq, const void *wk,
                                                    const void *wv, const void *wo, const void *wg, const void *wu,
                                                    const void *wd, const void *head, int smem_bytes,
                                                    cudaStream_t stream);

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxCtas = 1024;
constexpr int kAttnMinLen = 64;
constexpr long long kTimeoutNs = 2000000000LL;

// The scratch.  Every GPU that loads the library holds these bytes until the
// process exits.
__device__ __align__(256) unsigned char lf_noalloc_scratch[LF_NOALLOC_SCRATCH_BYTES];

void *g_scratch[kMaxDevices];       // device address of lf_noalloc_scratch, per device
int g_smem_set[kMaxDevices];        // dynamic shared memory size set for the kernel, per device

// Host staging for the partition and the RoPE table (static: no host allocation either).
lfk::CtaPlan h_plans[kMaxCtas];
float2 h_rope[LF_NOALLOC_SCRATCH_BYTES / sizeof(float2)];

// Error return once work that touches the scratch array is queued on `st`:
// wait for that work first, so that nothing still reads or writes the array
// when the call returns and the caller may retry at once.  The wait's own
// error is ignored (the call already failed).
lf_status drain_and_fail(cudaStream_t st, lf_status s)
{
    (void)cudaStreamSynchronize(st);
    return s;
}

size_t carve(size_t &off, size_t bytes)
{
    const size_t at = off;
    off = (off + bytes + 255) / 256 * 256;
    return at;
}

}  // namespace

extern "C" LF_API lf_status lf_generate_noalloc(const lf_config *cfg, const lf_weights *w,
                                                const int32_t *prompt_dev, int32_t n_prompt, int32_t n_steps,
                                                const lf_sampling *sp, uint64_t seed, int32_t *out_tokens_dev,
                                                void *stream)
{
    if (!cfg || !w || !prompt_dev || !sp || !out_tokens_dev || n_prompt < 1 || n_steps < 1) return LF_ERR_INVALID_ARG;
    const void *need[] = {w->embed, w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm,
                          w->w_gate, w->w_up, w->w_down, w->final_norm, w->lm_head};
    for (const void *p : need)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return LF_ERR_INVALID_ARG;   // bulk copies need 16 B
    if (cfg->n_layers <= 0 || cfg->d_model <= 0 || cfg->n_heads <= 0 || cfg->n_kv_heads <= 0 || cfg->ffn_dim <= 0 ||
        cfg->vocab <= 0 || cfg->max_seq <= 0 || cfg->n_ctas < 0 || !(cfg->rope_theta > 0.f) || !(cfg->rms_eps >= 0.f))
        return LF_ERR_INVALID_ARG;
    if (cfg->head_dim != 64 && cfg->head_dim != 128) return LF_ERR_NOT_SUPPORTED;
    if (cfg->n_heads % cfg->n_kv_heads || lfk::MAX_GROUP % (cfg->n_heads / cfg->n_kv_heads)) return LF_ERR_NOT_SUPPORTED;
    if (cfg->d_model % lfk::KC || (cfg->n_heads * cfg->head_dim) % lfk::KC || cfg->ffn_dim % lfk::KC)
        return LF_ERR_NOT_SUPPORTED;
    const long long most = (long long)lfk::MAX_SLICES * lfk::KC;
    if (cfg->d_model > most || (long long)cfg->n_heads * cfg->head_dim > most || cfg->ffn_dim > most)
        return LF_ERR_NOT_SUPPORTED;
    if (sp->top_k < 0 || sp->top_k > LF_MAX_TOP_K) return LF_ERR_NOT_SUPPORTED;
    if (cfg->weight_format != LF_WEIGHTS_FP16 || cfg->prefill_block != 0 || cfg->n_experts != 0)
        return LF_ERR_NOT_SUPPORTED;
    if (cfg->layer_window)
        for (int l = 0; l < cfg->n_layers; ++l)
            if (cfg->layer_window[l] < 0) return LF_ERR_INVALID_ARG;
    {
        // pageable copies and a stream synchronize cannot be captured: refuse a capturing stream up front
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) return LF_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return LF_ERR_NOT_SUPPORTED;
    }
    // the forward passes use positions 0 .. n_prompt + n_steps - 2 (the bound of
    // lf_prefill followed by lf_decode on a handle)
    if ((long long)n_prompt - 1 + n_steps > cfg->max_seq) return LF_ERR_CAPACITY;

    lfk::Geo g;
    g.L = cfg->n_layers;
    g.d = cfg->d_model;
    g.Hq = cfg->n_heads;
    g.Hkv = cfg->n_kv_heads;
    g.hd = cfg->head_dim;
    g.F = cfg->ffn_dim;
    g.V = cfg->vocab;
    g.Q = g.Hq * g.hd;
    g.KV = g.Hkv * g.hd;
    g.group = g.Hq / g.Hkv;
    g.max_seq = cfg->max_seq;
    g.fmt = lfk::FMT_FP16;
    g.E = 0;
    g.topk = 1;
    g.Fe = g.F;
    g.crb = lfk::fmt_crb(lfk::FMT_FP16);

    // ---- device, grid and the static partition (as lf_create)
    int dev = 0, sm = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return LF_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LF_ERR_NOT_SUPPORTED;
    int P = cfg->n_ctas > 0 ? (cfg->n_ctas < sm ? cfg->n_ctas : sm) : sm;
    for (int s = 0; s < lfk::N_GEMV; ++s) P = P < lfk::stage_geom(g, s).units ? P : lfk::stage_geom(g, s).units;
    if (P > kMaxCtas) P = kMaxCtas;
    int lm_rows_max = 0;
    for (int b = 0; b < P; ++b) {
        lfk::CtaPlan &pl = h_plans[b];
        std::memset(&pl, 0, sizeof(pl));
        for (int s = 0; s < lfk::N_GEMV; ++s) {
            const int U = lfk::stage_geom(g, s).units;
            pl.u0[s] = lfk::cta_unit_start(U, P, b);
            pl.u1[s] = lfk::cta_unit_start(U, P, b + 1);
        }
        const int n_lm = pl.u1[lfk::ST_LM] - pl.u0[lfk::ST_LM];
        lm_rows_max = n_lm > lm_rows_max ? n_lm : lm_rows_max;
    }
    const int max_split = P / g.Hkv > 1 ? P / g.Hkv : 1;
    const int a_floats = lfk::scratch_floats(g, max_split);
    const unsigned rest = lfk_smem_bytes(0, a_floats, lm_rows_max, g.L);
    if ((int)rest + 2 * lfk::ATT_CHUNK_BYTES > optin) return LF_ERR_NOT_SUPPORTED;
    int ring = (int)(((unsigned)optin - rest) / 1024u * 1024u);
    while ((int)lfk_smem_bytes(ring, a_floats, lm_rows_max, g.L) > optin) ring -= 1024;
    if (ring < 2 * lfk::ATT_CHUNK_BYTES) return LF_ERR_NOT_SUPPORTED;   // as lf_create: one K/V sub-block must fit
    const int smem = (int)lfk_smem_bytes(ring, a_floats, lm_rows_max, g.L);

    // ---- scratch layout inside the static array
    const size_t kv_elems = (size_t)g.L * g.Hkv * (size_t)g.max_seq * g.hd;
    const size_t sig_words = (size_t)g.L * lfk::sig_layout(g).per_layer * lfk::SIG_STRIDE;
    const size_t n_attn_done = (size_t)g.L * g.Hkv;
    const size_t cnt_words = sig_words + (n_attn_done + 3) * lfk::CNT_STRIDE;
    const size_t rope_elems = (size_t)g.max_seq * (g.hd / 2);
    size_t off = 0;
    const size_t o_plans = carve(off, sizeof(lfk::CtaPlan) * P);
    const size_t o_k = carve(off, 2 * kv_elems), o_v = carve(off, 2 * kv_elems);
    const size_t o_rope = carve(off, sizeof(float2) * rope_elems);
    const size_t o_q = carve(off, 4ull * g.L * g.Q), o_attn = carve(off, 4ull * g.L * g.Q);
    const size_t o_xattn = carve(off, 4ull * g.L * g.d), o_h = carve(off, 4ull * g.L * g.F);
    const size_t o_xout = carve(off, 4ull * g.L * g.d);
    const size_t o_apart = carve(off, 4ull * g.L * g.Hq * max_split * (g.hd + 2));
    const size_t o_kvf = carve(off, 4ull * g.L * 2 * g.KV);
    const size_t o_cnt = carve(off, 4 * cnt_words);
    const size_t o_lm = carve(off, 8ull * P * lfk::MAX_TOPK);
    const size_t o_tok = carve(off, 4ull * (1 + g.max_seq));
    const size_t o_status = carve(off, 4 * 8);
    bool windowed = false;
    if (cfg->layer_window)
        for (int l = 0; l < g.L; ++l) windowed = windowed || cfg->layer_window[l] > 0;
    const size_t o_win = windowed ? carve(off, sizeof(int) * g.L) : 0;
    if (off > (size_t)LF_NOALLOC_SCRATCH_BYTES) return LF_ERR_CAPACITY;

    // ---- per-device set-up: device address of the scratch array, kernel smem limit
    if (!g_scratch[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, lf_noalloc_scratch);
        if (e != cudaSuccess || !ptr) return LF_ERR_CUDA;
        g_scratch[dev] = ptr;
    }
    if (g_smem_set[dev] < smem) {
        if (lfk_set_smem_direct(smem) != cudaSuccess) return LF_ERR_CUDA;
        g_smem_set[dev] = smem;
    }
    unsigned char *base = static_cast<unsigned char *>(g_scratch[dev]);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    for (int pos = 0; pos < g.max_seq; ++pos)
        for (int i = 0; i < g.hd / 2; ++i) {
            const double inv_freq = std::pow((double)cfg->rope_theta, -2.0 * (double)i / (double)g.hd);
            const double ang = (double)pos * inv_freq;
            h_rope[(size_t)pos * (g.hd / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    e = cudaMemcpyAsync(base + o_plans, h_plans, sizeof(lfk::CtaPlan) * P, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + o_rope, h_rope, sizeof(float2) * rope_elems, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_cnt, 0, 4 * cnt_words, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_status, 0, 4 * 8, st);
    // the pass count restarts at 0: the activations between GEMV stages start as zeros
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_attn, 0, 4ull * g.L * g.Q, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_q, 0, 4ull * g.L * g.Q, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_kvf, 0, 4ull * g.L * 2 * g.KV, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_xattn, 0, 4ull * g.L * g.d, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_h, 0, 4ull * g.L * g.F, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(base + o_xout, 0, 4ull * g.L * g.d, st);
    if (e == cudaSuccess && windowed)
        e = cudaMemcpyAsync(base + o_win, cfg->layer_window, sizeof(int) * g.L, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return drain_and_fail(st, LF_ERR_CUDA);

    lfk::Params p;
    std::memset(&p, 0, sizeof(p));
    p.g = g;
    p.P = P;
    p.eps = cfg->rms_eps;
    p.plans = reinterpret_cast<const lfk::CtaPlan *>(base + o_plans);
    p.embed = static_cast<const __half *>(w->embed);
    p.attn_norm = static_cast<const __half *>(w->attn_norm);
    p.ffn_norm = static_cast<const __half *>(w->ffn_norm);
    p.final_norm = static_cast<const __half *>(w->final_norm);
    p.kc = reinterpret_cast<__half *>(base + o_k);
    p.vc = reinterpret_cast<__half *>(base + o_v);
    p.rope = reinterpret_cast<const float2 *>(base + o_rope);
    p.qbuf = reinterpret_cast<float *>(base + o_q);
    p.attn = reinterpret_cast<float *>(base + o_attn);
    p.xattn = reinterpret_cast<float *>(base + o_xattn);
    p.hbuf = reinterpret_cast<float *>(base + o_h);
    p.xout = reinterpret_cast<float *>(base + o_xout);
    p.apart = reinterpret_cast<float *>(base + o_apart);
    p.kvf = reinterpret_cast<float *>(base + o_kvf);
    p.win = windowed ? reinterpret_cast<const int *>(base + o_win) : nullptr;
    p.max_split = max_split;
    unsigned *cnt = reinterpret_cast<unsigned *>(base + o_cnt);
    p.sig = cnt;
    p.attn_done = cnt + sig_words;
    p.lm_done = p.attn_done + n_attn_done * lfk::CNT_STRIDE;
    p.tok_cnt = p.lm_done + lfk::CNT_STRIDE;
    p.gbar = p.tok_cnt + lfk::CNT_STRIDE;
    p.lm_part = reinterpret_cast<unsigned long long *>(base + o_lm);
    p.tok_buf = reinterpret_cast<int *>(base + o_tok);
    p.tok_seq = p.tok_buf + 1;
    p.status = reinterpret_cast<unsigned *>(base + o_status);
    p.abort_flag = p.status + 4;
    p.timeout_ns = cfg->wait_timeout_ns > 0 ? cfg->wait_timeout_ns : kTimeoutNs;
    p.fault_step = -1;
    p.ring_bytes = ring;
    p.a_floats = a_floats;
    p.lm_rows_max = lm_rows_max;
    p.attn_min_len = kAttnMinLen;
    p.sched = lfk::SCHED_FLAGS;
    p.only_layer = -1;
    p.only_stage = -1;

    // ---- prefill: forward passes of prompt[0 .. n_prompt-2]
    if (n_prompt > 1) {
        lfk::Params q = p;
        q.mode = lfk::MODE_PREFILL;
        q.n_steps = n_prompt - 1;
        q.prompt = prompt_dev;
        e = lfk_launch_monokernel_direct(&q, w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down, w->lm_head,
                                         smem, st);
        if (e != cudaSuccess)
            return drain_and_fail(st, e == cudaErrorCooperativeLaunchTooLarge ? LF_ERR_NOT_RESIDENT : LF_ERR_CUDA);
    }
    e = cudaMemcpyAsync(p.tok_buf, prompt_dev + (n_prompt - 1), sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return drain_and_fail(st, LF_ERR_CUDA);

    // ---- decode n_steps tokens
    lfk::Params q = p;
    q.mode = lfk::MODE_DECODE;
    q.n_steps = n_steps;
    q.pos0 = n_prompt - 1;
    q.epoch0 = (unsigned)(n_prompt - 1);
    q.out_tokens = out_tokens_dev;
    q.debug_logits = sp->debug_logits_dev;
    q.force_tokens = sp->force_tokens_dev;
    q.temperature = sp->temperature;
    q.top_k = sp->top_k;
    q.seed = seed;
    e = lfk_launch_monokernel_direct(&q, w->wq, w->wk, w->wv, w->wo, w->w_gate, w->w_up, w->w_down, w->lm_head,
                                     smem, st);
    if (e != cudaSuccess)
        return drain_and_fail(st, e == cudaErrorCooperativeLaunchTooLarge ? LF_ERR_NOT_RESIDENT : LF_ERR_CUDA);

    // ---- wait for the request and report the device status
    unsigned status[4] = {0, 0, 0, 0};
    e = cudaMemcpyAsync(status, p.status, sizeof(status), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return drain_and_fail(st, LF_ERR_CUDA);
    if (status[0] == (unsigned)lfk::STATUS_TIMEOUT) return LF_ERR_TIMEOUT;
    if (status[0] != 0u) return LF_ERR_INVALID_ARG;
    return LF_OK;
}
