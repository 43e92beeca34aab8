// lf_prefill.h -- internal interface of the batched prefill (lf_prefill.cu),
// called by the host runtime (lf_api.cu) when a handle was created with
// lf_config.prefill_block > 0.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "lf_internal.cuh"

// Device scratch of one block of T <= block positions (all row-major).
struct lfp_workspace {
    float *X;           // [T, d]   residual stream
    __half *Xh, *Xl;    // [T, max(d, Q, F)] FP16 head / remainder of a projection input
    float *Y;           // [T, max(Q + 2 KV, d)] projection output
    float *Qr;          // [T, Q]   q after RoPE
    float *A;           // [T, Q]   attention output
    float *GU;          // [T, 2F]  gate and up projections
    // mixture of experts only (null otherwise)
    float *R;           // [T, E]   router logits
    int *sel;           // [T, 8]   chosen experts, slot by slot
    float *gate;        // [T, 8]   their gates (index t * 8 + j)
    int *list;          // [E, T]   per expert: t * 8 + j of the tokens routed to it, in token order
    int *cnt;           // [E]      list lengths
    __half *Xgh, *Xgl;  // [T, d]   FFN input rows gathered for one expert
    __half *Hh, *Hl;    // [T, Fe]  gated hidden units of one expert
    float *Yk;          // [T, k, d] expert outputs per slot
};

// Bytes of the workspace for blocks of `block` positions, and its carving.
size_t lfp_workspace_bytes(const lfk::Geo &g, int block);
lfp_workspace lfp_carve(void *base, const lfk::Geo &g, int block);

struct lfp_args {
    lfk::Geo g;
    int block;                  // positions per pass
    int n;                      // positions to run (tokens[0 .. n-1] at positions pos0 .. pos0+n-1)
    int pos0;
    float eps;
    const int *tokens;          // [n] device
    const __half *embed, *attn_norm, *ffn_norm;
    // row-major FP16 projections per layer, fused where the inputs are shared:
    // [L, Q + 2 KV, d] q/k/v rows, [L, d, Q], [L, 2F, d] gate rows then up rows,
    // [L, d, F]; FP8 models: the decoded E4M3 codes, and the FP32 row scales of
    // the same layouts (null for FP16 models); MXFP4 models: the decoded
    // weights; mixture of experts: wgu [L, E, 2 Fe, d], wd [L, E, d, Fe]
    const __half *wqkv, *wo, *wgu, *wd;
    const float *sqkv, *so, *sgu, *sd;
    const __half *router;       // mixture of experts: the caller's [L, E, d] router rows, else null
    const float2 *rope;         // [max_seq, hd/2] (cos, sin)
    const int *win;             // [L] windows, or null
    __half *kc, *vc;            // KV cache, group-swizzled rows
    unsigned *status;           // [8]: status[0..3] error record, status[4] abort flag
    void *cublas;               // cublasHandle_t
    lfp_workspace ws;
};

// Runs the passes on `stream`.  0 on success; 1 a launch or copy failed; 2/3 cuBLAS failed.  With a
// mixture of experts each layer reads its per-expert token counts back to the host (the stream is
// synchronized once per layer and block) to size the experts' GEMMs.
extern "C" int lfp_run(const lfp_args *a, cudaStream_t stream);
// cuBLAS handle lifetime (kept out of lf_api.cu so that only this file includes cuBLAS).
extern "C" int lfp_cublas_create(void **out);
extern "C" void lfp_cublas_destroy(void *h);
// E4M3 codes -> FP16 (exact: every finite E4M3 value is an FP16 value).
extern "C" cudaError_t lfp_decode_e4m3(const uint8_t *src, __half *dst, size_t n, cudaStream_t stream);
// MXFP4 matrix [rows, cols] (packed E2M1 codes, E8M0 scales per 32) -> FP16, exact for scales 2^-23 .. 2^13.
extern "C" cudaError_t lfp_decode_mxfp4(const uint8_t *codes, const uint8_t *scales, size_t rows, int cols,
                                         __half *dst, cudaStream_t stream);
// Smallest and largest of n device bytes (synchronous).
extern "C" cudaError_t lfp_byte_range(const uint8_t *s, size_t n, unsigned *lo, unsigned *hi);
