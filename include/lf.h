/*
 * lf.h -- C ABI of the batch-1 decode monokernel library (liblf.so).
 *
 * One handle holds one decoder (weights, FP16 KV cache, decode state) on one
 * GPU.  The whole per-token pass -- embedding gather, RMSNorm, QKV GEMV, RoPE,
 * KV append, attention over the cache, output projection, SwiGLU FFN, final
 * norm, LM-head GEMV and sampling -- runs inside ONE persistent kernel per
 * lf_decode / lf_prefill call, with no kernel launch and no host round trip
 * between tokens.  This follows the "monokernel" of the KOG LaneFormer
 * write-up (shivam2003.com, "KOG LaneFormer-2B & the monokernel", section
 * "Pillar 3 -- the monokernel runtime": the kernel launches once and stays
 * resident until the token is produced), extended here to n_steps tokens per
 * launch.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 *     The caller owns every buffer it passes.  Device buffers must stay
 *     valid until the work queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Calls are asynchronous on it unless stated otherwise.
 *   - A handle is single-threaded and single-stream: do not call into one
 *     handle from two threads at once, or queue work for it on two streams.
 *   - Every call returns an lf_status.  No entry point aborts the process,
 *     throws, or traps on the device.  Errors found on the host are returned
 *     at once and leave the handle unchanged.  An error found on the device
 *     (a bounded wait that ran out) is latched in the handle: lf_sync
 *     returns it, and every later call returns LF_ERR_STATE until lf_reset.
 *   - All tensors are row-major.  Weight matrices use the nn.Linear layout
 *     [out_features, in_features] and are FP16 (IEEE binary16).
 */
#ifndef LF_H
#define LF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LF_API __attribute__((visibility("default")))
#else
#define LF_API
#endif

#define LF_ABI_VERSION 6
#define LF_MAX_TOP_K 64          /* largest top_k that lf_decode accepts (besides 0) */
#define LF_PREFILL_AUTO (-1)     /* lf_config.prefill_block: batched prefill, block size chosen by the library */

typedef enum {
    LF_OK = 0,
    LF_ERR_INVALID_ARG = 1,      /* NULL pointer, bad size or shape */
    LF_ERR_OUT_OF_MEMORY = 2,    /* a device or host allocation failed */
    LF_ERR_CAPACITY = 3,         /* the request needs more than max_seq positions */
    LF_ERR_NOT_RESIDENT = 4,     /* the persistent grid cannot be co-resident on this GPU */
    LF_ERR_CUDA = 5,             /* a CUDA runtime call failed */
    LF_ERR_TIMEOUT = 6,          /* a device-side wait ran past wait_timeout_ns (latched) */
    LF_ERR_NOT_SUPPORTED = 7,    /* shape outside what the kernels handle (see lf_config) */
    LF_ERR_STATE = 8             /* call not valid in the current state (no pending token, latched error) */
} lf_status;

/* Schedules: how the stages of the per-token pass wait for each other.
 * LF_SCHED_FLAGS is the library's design; the other two are ablations that
 * reproduce the overheads the monokernel write-up removes. */
typedef enum {
    /* One persistent launch; every stage waits only for the counters of the
     * data it reads (per-dependency waits: stackfutures.com, "The
     * Monokernel", "Targeted synchronization"). */
    LF_SCHED_FLAGS = 0,
    /* One persistent launch; a grid-wide arrival-counter barrier after every
     * stage (the atomic-counter grid sync that shivam2003.com, "Cross-GPU
     * synchronization without atomics", measured at 7.59-7.88 us). */
    LF_SCHED_GRID_BARRIER = 1,
    /* One kernel launch per stage and layer, on the stream (the generic
     * stack of shivam2003.com, "Why standard frameworks leave the bandwidth
     * on the table": one kernel per stage/layer). */
    LF_SCHED_MULTI_KERNEL = 2
} lf_schedule;

/* Decoder shape.  Supported: head_dim 64 or 128; n_heads a multiple of
 * n_kv_heads with n_heads / n_kv_heads <= 8; d_model, n_heads * head_dim and
 * ffn_dim multiples of 256; vocab >= 1; max_seq >= 1. */
typedef struct {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_heads;         /* query heads */
    int32_t n_kv_heads;      /* key/value heads (GQA groups are contiguous: query head h uses KV head h / (n_heads / n_kv_heads)) */
    int32_t head_dim;
    int32_t ffn_dim;
    int32_t vocab;
    int32_t max_seq;         /* KV-cache capacity in positions */
    float rope_theta;        /* RoPE base, e.g. 10000 */
    float rms_eps;           /* RMSNorm epsilon, e.g. 1e-5 */
    int64_t wait_timeout_ns; /* bound of every device-side wait; 0 selects 2e9 (2 s) */
    int32_t n_ctas;          /* persistent grid size; 0 selects one CTA per SM (capped at d_model) */
    int32_t fault_step;      /* test hook: -1 (off), or the decode step (within one lf_decode call)
                                at which layer 0's QKV stage withholds its readiness signal, so
                                that the consumers' bounded waits run out */
    /* Sliding-window attention (shivam2003.com, model table and "Why GQA and
     * sliding windows": windowed layers bound the KV cache each token reads).
     * NULL: every layer attends to the whole cache.  Otherwise a HOST array
     * of n_layers windows, copied by lf_create: layer_window[l] = W > 0 makes
     * the query at position p of layer l attend to positions
     * max(0, p-W+1) .. p only; 0 keeps the whole cache.  The KV cache still
     * holds every position (max_seq). */
    const int32_t *layer_window;
    /* Format of the eight projection matrices (wq .. w_down, lm_head):
     * LF_WEIGHTS_FP16 (0), or LF_WEIGHTS_FP8_E4M3 (1): weight-only FP8 (the
     * pages' FP8 streaming, shivam2003.com, "Scaling the idea to frontier
     * models"), one byte per weight in OCP E4M3 (no infinities, 448 largest)
     * and one FP32 scale per output row in the lf_weights *_scale arrays; the
     * matrix applied is diag(scale) . decode(codes), dot products in FP32 with
     * the scale applied to each finished row sum.  Or LF_WEIGHTS_MXFP4 (2):
     * OCP Microscaling FP4 (the pages' "FP8/MXFP4", same section), two E2M1
     * elements per byte (element 2i in the low nibble of byte i; magnitudes
     * 0, 0.5, 1, 1.5, 2, 3, 4, 6) and one E8M0 scale byte, 2^(E-127), per 32
     * consecutive elements of a row in the *_scale arrays; weight (r, k) =
     * e2m1 * 2^(E-127), dot products in FP32.  The embedding and the norm
     * gains stay FP16.  lf_generate_noalloc takes FP16 weights only.  The
     * batched prefill of an MXFP4 model (prefill_block > 0) uses the weights
     * decoded to FP16, which is exact for block scales 2^-23 .. 2^13 (E 104
     * .. 140); lf_create rejects other scales there with NOT_SUPPORTED. */
    int32_t weight_format;
    /* Prefill implementation.  0: lf_prefill runs the prompt as repeated
     * decode steps inside the monokernel (one position per step, the
     * weights streamed once per position).  B > 0: batched prefill over
     * blocks of up to B positions (min(B, max_seq)): per layer, the
     * projections of the whole block as the library's tensor-core GEMMs
     * (tcgen05, with the RMSNorm, RoPE, KV append, SwiGLU and residual work
     * fused into their epilogues) and a causal flash-style attention over the
     * cache, the same arithmetic per position (FP32 activations, FP16
     * weights and cache).  lf_create then keeps a row-major FP16 copy of the
     * seven layer projections (FP8 models: the decoded codes; the scales are
     * applied to the sums) and a workspace that grows with B;
     * lf_info.prefill_bytes reports them.  B = LF_PREFILL_AUTO: batched, with
     * the library's choice of B (lf_info.prefill_block reports it): the
     * largest multiple of 128 up to 1024 (and at most max_seq) whose causal
     * attention grid -- one CTA per 128 query rows and query head, one CTA per
     * SM at a time -- fills its waves to at least 80 % of the best such
     * block's fill (896 for 20 heads on 152 SMs, 1024 for 16 or 32).
     * lf_generate_noalloc takes 0 only. */
    int32_t prefill_block;
    /* Mixture-of-experts FFN (the pages: only the active experts' weights
     * stream per token, shivam2003.com, "Scaling the idea to frontier
     * models").  n_experts = 0: the dense SwiGLU FFN.  n_experts = E in
     * [1, 64]: every layer holds E SwiGLU experts of ffn_dim hidden units
     * (lf_weights.w_gate / w_up [L, E, ffn_dim, d], w_down [L, E, d,
     * ffn_dim]) and a router lf_weights.w_router [L, E, d]; per token and
     * layer the kernel forms the router logits W_router . xn (xn the FFN's
     * RMSNorm output), takes the top_k_experts in [1, min(8, E)] largest
     * (ties to the lower index), weights expert j by the softmax of the
     * chosen logits, and streams only the chosen experts' rows.  Needs FP16
     * weights, top_k_experts * ffn_dim <= 16384 and a schedule other than
     * LF_SCHED_MULTI_KERNEL.  The batched prefill (prefill_block > 0) routes
     * the block's tokens the same way and runs grouped GEMMs over the tokens
     * routed to each expert, sized on the device (no host round trip). */
    int32_t n_experts;
    int32_t top_k_experts;
} lf_config;

#define LF_WEIGHTS_FP16 0
#define LF_WEIGHTS_FP8_E4M3 1
#define LF_WEIGHTS_MXFP4 2

/* Device pointers to the caller's weights (row-major, stacked over layers):
 * FP16, or for lf_config.weight_format = LF_WEIGHTS_FP8_E4M3 the eight
 * projections as E4M3 bytes with FP32 per-row scales, or for
 * LF_WEIGHTS_MXFP4 as packed E2M1 codes ([.., rows, cols/2] bytes) with E8M0
 * block scales ([.., rows, cols/32] bytes).  L = n_layers,
 * d = d_model, Q = n_heads*head_dim, KV = n_kv_heads*head_dim, F = ffn_dim,
 * V = vocab.  lf_create copies the projection matrices, the LM head and the
 * scales into library-owned memory (a per-CTA streaming layout for the
 * matrices); the caller may free those after lf_create returns.  embed and
 * the three norm-gain tensors are read in place by every decode step and must
 * outlive the handle.  Every matrix pointer must be 16-byte aligned (the
 * kernels read them with bulk copies); the scale pointers are NULL for FP16
 * weights, 4-byte aligned for FP8 and any byte address for MXFP4. */
typedef struct {
    const void *embed;       /* [V, d]      read in place */
    const void *attn_norm;   /* [L, d]      read in place */
    const void *wq;          /* [L, Q, d]   copied */
    const void *wk;          /* [L, KV, d]  copied */
    const void *wv;          /* [L, KV, d]  copied */
    const void *wo;          /* [L, d, Q]   copied */
    const void *ffn_norm;    /* [L, d]      read in place */
    const void *w_gate;      /* [L, F, d]   copied */
    const void *w_up;        /* [L, F, d]   copied */
    const void *w_down;      /* [L, d, F]   copied */
    const void *final_norm;  /* [d]         read in place */
    const void *lm_head;     /* [V, d]      copied (untied from embed) */
    /* FP8: FP32 scale of every row of the matrix of the same name (shapes
     * below); MXFP4: uint8 E8M0 scale of every 32 elements of a row (the
     * shapes below with a last dimension of cols/32); FP16: NULL */
    const void *wq_scale;      /* [L, Q]  */
    const void *wk_scale;      /* [L, KV] */
    const void *wv_scale;      /* [L, KV] */
    const void *wo_scale;      /* [L, d]  */
    const void *w_gate_scale;  /* [L, F]  */
    const void *w_up_scale;    /* [L, F]  */
    const void *w_down_scale;  /* [L, d]  */
    const void *lm_head_scale; /* [V]     */
    /* Mixture of experts only (lf_config.n_experts > 0), else NULL: the
     * router rows [L, E, d] FP16, read in place (must outlive the handle),
     * 16-byte aligned */
    const void *w_router;
} lf_weights;

/* Token choice, after the Gumbel-max trick of shivam2003.com ("The fused
 * operations, briefly", sampling: argmax_i(logit_i + g_i) samples the
 * softmax without normalising):
 *   temperature <= 0 or top_k == 1: greedy argmax (lowest index among equal maxima);
 *   otherwise S = the top_k largest logits (all of them if top_k == 0; equal
 *   logits ordered by lower index) and the token is
 *   argmax_{i in S} (logit_i / temperature + g_i), equal scores to the lower index,
 *   g_i = -log(-log(u_i)), u_i = (2 * (r_i >> 9) + 1) * 2^-24, r_i = word (i mod 4) of
 *   Philox4x32-10(counter = (i / 4, p, 0, 0), key = (seed low 32, seed high 32)),
 *   p = position of the token whose logits are sampled.
 * top_k must be 0 or in [1, LF_MAX_TOP_K]. */
typedef struct {
    float temperature;
    int32_t top_k;
    float *debug_logits_dev;          /* NULL, or [n_steps, V] FP32: every step's logits */
    const int32_t *force_tokens_dev;  /* NULL, or [n_steps]: step i feeds force_tokens[i] to step
                                         i+1 instead of its own choice (the choice is still
                                         written to out_tokens); teacher forcing for tests */
} lf_sampling;

typedef struct lf_handle lf_handle;

typedef struct {
    int32_t n_ctas;              /* persistent grid size */
    int32_t threads_per_cta;
    int32_t smem_bytes;          /* dynamic shared memory per CTA */
    int32_t ring_bytes;          /* weight-ring bytes per CTA */
    int32_t sm_count;
    int32_t position;            /* position of the pending token (tokens decoded or prefilled so far) */
    int32_t has_pending;         /* 1 if a pending token is set */
    int32_t schedule;            /* current lf_schedule */
    int64_t weight_stream_bytes; /* bytes of the library's repacked weight copy */
    int64_t kv_cache_bytes;      /* bytes of the FP16 K and V caches */
    int32_t prefill_block;       /* lf_config.prefill_block as used (0: prefill in the monokernel) */
    int64_t prefill_bytes;       /* bytes of the batched prefill's weight copy and workspace (0 if off) */
} lf_info;

/* Validate cfg, allocate the KV cache, activations, counters and the
 * repacked weight copy on the current device, build the RoPE table and the
 * static work partition, and check that the persistent grid fits.  Runs one
 * repack kernel on the legacy default stream and synchronizes.  On success
 * *out receives a handle with no pending token at position 0.
 * Errors: INVALID_ARG (NULL or not 16-byte aligned weight pointers,
 * non-positive sizes, a negative window, prefill_block below LF_PREFILL_AUTO), NOT_SUPPORTED
 * (shape: head_dim other than 64 or 128, d_model, n_heads*head_dim or
 * ffn_dim not a multiple of 256 or above 16384; an unknown weight_format;
 * MXFP4 block scales outside 2^-23 .. 2^13 with prefill_block > 0; an
 * expert configuration outside the limits of lf_config.n_experts),
 * OUT_OF_MEMORY,
 * NOT_RESIDENT, CUDA (also: a tensor map of the batched prefill could not
 * be encoded). */
LF_API lf_status lf_create(const lf_config *cfg, const lf_weights *weights, lf_handle **out);

/* Release every library-owned allocation.  Synchronizes the device first.
 * Accepts NULL. */
LF_API void lf_destroy(lf_handle *h);

/* Prefill (the per-token decode pass of shivam2003.com, "KOG LaneFormer-2B
 * & the monokernel", sections "Pillar 3 -- the monokernel runtime" and "The
 * fused operations, briefly", run once per prompt position without sampling):
 * runs the forward pass of the pending token (if any) and of
 * tokens_dev[0 .. n-2] at consecutive positions, appending their K and V to
 * the cache, and makes tokens_dev[n-1] the pending token.  No logits are
 * computed.  With lf_config.prefill_block = 0 the passes are repeated decode
 * steps in one persistent launch; with B > 0 they run batched, B positions
 * per pass (see lf_config.prefill_block), on the same stream.  tokens_dev: device int32 [n], each in [0, vocab).
 * Errors: INVALID_ARG (n < 1, NULL), CAPACITY (not enough positions left for
 * these tokens plus the pending one), STATE (latched device error). */
LF_API lf_status lf_prefill(lf_handle *h, const int32_t *tokens_dev, int32_t n, void *stream);

/* n_steps decode steps in one persistent launch (shivam2003.com, "KOG
 * LaneFormer-2B & the monokernel", section "Pillar 3 -- the monokernel
 * runtime": the kernel stays resident until the token is produced; here it
 * stays resident for n_steps tokens, feeding each sampled token to the next
 * step on the device).  Step i runs the forward
 * pass of the pending token at the current position, chooses a token from
 * its logits (lf_sampling), writes it to out_tokens_dev[i] (device int32
 * [n_steps]) and makes it the pending token.  The position advances by
 * n_steps.  Errors: INVALID_ARG, NOT_SUPPORTED (top_k), CAPACITY (position +
 * n_steps > max_seq), STATE (no pending token, or latched device error). */
LF_API lf_status lf_decode(lf_handle *h, int32_t n_steps, const lf_sampling *sp, uint64_t seed,
                    int32_t *out_tokens_dev, void *stream);

/* Host-buffer convenience: copies prompt_host[0 .. n_prompt-1] to the device,
 * prefills it, decodes n_steps tokens and copies them to out_host, then
 * synchronizes `stream` and returns the device status.  Uses library-owned
 * staging buffers; both host buffers may be pageable or pinned. */
LF_API lf_status lf_generate(lf_handle *h, const int32_t *prompt_host, int32_t n_prompt, int32_t n_steps,
                      const lf_sampling *sp, uint64_t seed, int32_t *out_host, void *stream);

/* Synchronize the stream of the last call and return the latched device
 * status: LF_OK; LF_ERR_TIMEOUT if a bounded wait ran out; LF_ERR_INVALID_ARG
 * if a token id fed to a forward pass was outside [0, vocab) (the kernel
 * substituted 0 for it and stopped). */
LF_API lf_status lf_sync(lf_handle *h);

/* Forget the sequence: position 0, no pending token, counters and the
 * latched device error cleared.  Synchronizes the device. */
LF_API lf_status lf_reset(lf_handle *h);

/* Select the schedule used by later lf_prefill / lf_decode calls.  Errors:
 * INVALID_ARG (unknown schedule), NOT_SUPPORTED (LF_SCHED_MULTI_KERNEL on a
 * mixture-of-experts handle: the expert choice is kept in shared memory
 * within one launch). */
LF_API lf_status lf_set_schedule(lf_handle *h, int32_t schedule);

/* Fill *out with the handle's launch geometry and state. */
LF_API lf_status lf_get_info(const lf_handle *h, lf_info *out);

/* Stage trace (profiling aid).  lf_enable_trace(h, n) makes every later
 * lf_prefill / lf_decode launch of the persistent schedules record, for its
 * first n steps, eight %globaltimer stamps (ns) per (step, slot, CTA): [0] the
 * stage was entered, [1] its inputs were ready, [2] its inputs were loaded,
 * [3] it was published, [4] GEMV: first tile done / attention: K/V positions
 * done, [5] GEMV: first weight chunk in hand / attention: piece partial
 * published, [6] and [7] the producer warp issued the stage's first and last
 * weight (or K/V) chunk, [8] (a count, not a time) GEMV chunks that had not
 * landed in shared memory when first asked for.  slot = 5 * layer + {0 QKV,
 * 1 attention, 2 O, 3 gate/up, 4 down}; slot 5 * n_layers is the LM head and
 * sampling.  Layout: [step][slot][cta][9] uint64, zero where nothing was
 * recorded.  n = 0 disables tracing.  lf_read_trace synchronizes the device,
 * sets *n_out to the number of words and, if host_out is not NULL, copies
 * them there (capacity in words). */
LF_API lf_status lf_enable_trace(lf_handle *h, int32_t max_steps);
LF_API lf_status lf_read_trace(lf_handle *h, uint64_t *host_out, int64_t capacity, int64_t *n_out);

/* Size of the device array that lf_generate_noalloc uses as scratch. */
#define LF_NOALLOC_SCRATCH_BYTES (8u << 20)

/* One whole request -- prefill of prompt_dev[0 .. n_prompt-1], then n_steps
 * decode steps written to out_tokens_dev -- that makes no device allocation.
 * The write-up these kernels follow has no counterpart of this entry point:
 * it exists for callers that cannot call cudaMalloc when a request arrives,
 * such as a plugin inside a host framework that owns every device allocation
 * through its own pool, or a process whose device memory is reserved up front.
 *
 * cfg and w are as for lf_create, but nothing is copied: the kernels stream
 * the projection matrices and the LM head straight from the caller's buffers
 * (row-major, nn.Linear layout), so every buffer in w must stay valid until
 * the call returns.  prompt_dev (device int32 [n_prompt]) and out_tokens_dev
 * (device int32 [n_steps]) belong to the caller; sp works as for lf_decode.
 * The forward passes use positions 0 .. n_prompt + n_steps - 2, so
 * n_prompt - 1 + n_steps must not exceed cfg->max_seq (the bound of
 * lf_prefill followed by lf_decode on a handle); cfg->fault_step is ignored.
 *
 * All scratch -- partition, RoPE table, FP16 KV cache, activations, counters,
 * attention partials, sampling candidates -- lives in one file-scope device
 * array of LF_NOALLOC_SCRATCH_BYTES (8 MiB), which every GPU that loads the
 * library holds until the process exits.  A request whose scratch would not
 * fit (mainly the KV cache: 4 * n_layers * n_kv_heads * max_seq * head_dim
 * bytes) is rejected with LF_ERR_CAPACITY before any work is queued.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit.  Every
 * call copies from pageable host memory and synchronizes `stream`, so no call
 * can be captured into a CUDA graph: a call on a capturing stream returns
 * LF_ERR_NOT_SUPPORTED before any work is queued.  Every call reuses the same array and
 * clears the counters it relies on; calls whose work overlaps on the GPU race
 * on the array.  The host staging buffers of the partition and the RoPE table
 * are shared by the whole process, so calls from two host threads at once
 * race even when they use different GPUs: serialise them.  Once a call has
 * queued work on `stream`, every error return first synchronizes `stream`,
 * so that no copy or kernel of the failed call still uses the array.
 * The call synchronizes `stream` and returns the device status (LF_OK,
 * LF_ERR_TIMEOUT, or LF_ERR_INVALID_ARG for a token id outside [0, vocab)).
 * Other errors: INVALID_ARG, NOT_SUPPORTED (also: FP8 or MXFP4 weights,
 * prefill_block other than 0, a mixture of experts, a capturing stream), CAPACITY,
 * NOT_RESIDENT, CUDA. */
LF_API lf_status lf_generate_noalloc(const lf_config *cfg, const lf_weights *w, const int32_t *prompt_dev,
                                     int32_t n_prompt, int32_t n_steps, const lf_sampling *sp, uint64_t seed,
                                     int32_t *out_tokens_dev, void *stream);

/* Static string naming a status code. */
LF_API const char *lf_error_string(lf_status s);

/* Microbenchmark of grid synchronisation on the current device (no handle).
 * mode 0: one-hop readiness flag -- a token is passed round a ring of n_ctas
 * CTAs `iters` times, each hop a gpu-scope release add by one CTA and an
 * acquire poll by the next; *ns_out = nanoseconds per hop.
 * mode 1: arrival-counter grid barrier over n_ctas CTAs, `iters` times;
 * *ns_out = nanoseconds per barrier.
 * Both run as one cooperative launch of n_ctas one-warp CTAs on the legacy
 * default stream and synchronize the device.  Waits are bounded (1 s).
 * Errors: INVALID_ARG (mode, n_ctas < 2, iters < 1, NULL), NOT_RESIDENT
 * (n_ctas above the SM count), OUT_OF_MEMORY, TIMEOUT, CUDA. */
LF_API lf_status lf_sync_latency(int32_t mode, int32_t n_ctas, int32_t iters, double *ns_out);

/* LF_ABI_VERSION of the built library. */
LF_API int32_t lf_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LF_H */
