// lf_prefill.h -- internal interface of the batched prefill (lf_prefill.cu),
// called by the host runtime (lf_api.cu) when a handle was created with
// lf_config.prefill_block > 0.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cuda.h>

#include "lf_internal.cuh"

// Device scratch of one block of T <= block positions (all row-major).
struct lfp_workspace {
    float *X;           // [T, d]   residual stream
    __half *Xh, *Xl;    // [T, d]   the next RMSNorm's input x * gain, FP16 head / remainder (GEMM operand)
    float *SS;          // [T, d/128] partial sums of squares of x per 128-column group
    float *Qr;          // [T, Q]   q after RoPE
    __half *Ah, *Al;    // [T, Q]   attention output, head / remainder (GEMM operand)
    __half *Hh, *Hl;    // [T, F]   SiLU(gate) * up, head / remainder; mixture of experts: [E * T, Fe]
    // mixture of experts only (null otherwise)
    float *R;           // [T, E]   router logits
    int *sel;           // [T, 8]   chosen experts, slot by slot
    float *gate;        // [T, 8]   their gates (index t * 8 + j)
    int *list;          // [E, T]   per expert: t * 8 + j of the tokens routed to it, in token order
    int *cnt;           // [E]      list lengths (read on the device: no host round trip)
    __half *Xgh, *Xgl;  // [E * T, d] FFN input rows gathered per expert
    float *Yk;          // [T, k, d] expert outputs per slot
    // split-K GEMMs: partial tiles and per-tile arrival counters (zeroed once)
    float *part;        // [sms * 128 * 256]
    unsigned *tile_cnt; // [1024]
};

// Bytes of the workspace for blocks of `block` positions on a device of
// `sms` SMs, and its carving.
size_t lfp_workspace_bytes(const lfk::Geo &g, int block, int sms);
lfp_workspace lfp_carve(void *base, const lfk::Geo &g, int block, int sms);

struct lfp_args {
    lfk::Geo g;
    int block;                  // positions per pass
    int n;                      // positions to run (tokens[0 .. n-1] at positions pos0 .. pos0+n-1)
    int pos0;
    float eps;
    const int *tokens;          // [n] device
    const __half *embed, *attn_norm, *ffn_norm;
    // row-major FP16 projections per layer, fused where the inputs are shared:
    // [L, Q + 2 KV, d] q/k/v rows; [L, d, Q]; [L, 2F, d] gate and up rows
    // interleaved in blocks of 128 units (128 gate rows, then the same units'
    // up rows); [L, d, F].  FP8 models: the decoded E4M3 codes, and the FP32
    // row scales in the same row order (null for FP16 models); MXFP4 models:
    // the decoded weights; mixture of experts: wgu [L, E, 2 Fe, d] (interleaved
    // the same way per expert), wd [L, E, d, Fe]
    const __half *wqkv, *wo, *wgu, *wd;
    const float *sqkv, *so, *sgu, *sd;
    const __half *router;       // mixture of experts: the caller's [L, E, d] router rows, else null
    const float2 *rope;         // [max_seq, hd/2] (cos, sin)
    const int *win;             // [L] windows, or null
    __half *kc, *vc;            // KV cache, group-swizzled rows
    unsigned *status;           // [8]: status[0..3] error record, status[4] abort flag
    int sms;                    // SMs of the device (GEMM tiling and split-K)
    // optional per-CTA %globaltimer stamps of layer 1's attention in the first
    // block ([grid][8]; profiling aid, null = off)
    unsigned long long *attn_stamps;
    lfp_workspace ws;
};

// TMA tensor maps of the GEMM operands (built once per handle: the workspace
// and the weight copies do not move).
struct lfp_maps {
    CUtensorMap xh, xl, ah, al, hh, hl, xgh, xgl, wgu;
    CUtensorMap wqkv[2], wo[2], wd[2];   // weight boxes of 128 and 256 rows (the two tile widths)
    CUtensorMap kc, vc;                  // the KV cache as [L * Hkv * max_seq, hd] rows (head_dim 128)
};

// Builds the tensor maps of a->ws and a->w*.  0 on success.
extern "C" int lfp_make_maps(const lfp_args *a, lfp_maps *m);
// Runs the passes on `stream`: five launches per layer and block (the QKV,
// O, gate/up and down GEMMs with fused epilogues, and the attention -- on
// the tensor cores through tcgen05 for head_dim 128, warp-level MMA
// fragments for 64), plus the block's embedding gather; a mixture of experts routes, gathers and runs
// grouped GEMMs sized on the device.  0 on success; 1 a launch failed.
extern "C" int lfp_run(const lfp_args *a, const lfp_maps *m, cudaStream_t stream);
// E4M3 codes -> FP16 (exact: every finite E4M3 value is an FP16 value).
extern "C" cudaError_t lfp_decode_e4m3(const uint8_t *src, __half *dst, size_t n, cudaStream_t stream);
// MXFP4 matrix [rows, cols] (packed E2M1 codes, E8M0 scales per 32) -> FP16, exact for scales 2^-23 .. 2^13.
extern "C" cudaError_t lfp_decode_mxfp4(const uint8_t *codes, const uint8_t *scales, size_t rows, int cols,
                                         __half *dst, cudaStream_t stream);
// Smallest and largest of n device bytes (synchronous).
extern "C" cudaError_t lfp_byte_range(const uint8_t *s, size_t n, unsigned *lo, unsigned *hi);
