// lf_gemm.h -- tensor-core GEMM of the batched prefill (lf_gemm.cu): one
// output tile per CTA, operands staged by TMA into 128-byte-swizzled shared
// memory, tcgen05.mma (FP16 x FP16 -> FP32) into TMEM, and an epilogue fused
// with the stage that consumes the projection (RoPE + KV store, residual +
// next RMSNorm's input, SwiGLU).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "lf_internal.cuh"

namespace lfg {

constexpr int BM = 128;   // rows of A (positions) per tile
constexpr int BK = 64;    // K per pipeline stage (128 bytes of FP16: one swizzle row)

// Epilogues.  Rows are positions (or, grouped, the rows routed to one expert).
enum Epi {
    EPI_STORE = 0,    // Y[r][n] = acc (x colscale): plain product, for tests
    EPI_QKV = 1,      // x inv(r) (x colscale), RoPE on q and k heads, q to Qr, K/V rounded into the cache
    EPI_RESID = 2,    // X[r][n] += acc (x colscale); then (X x gain_next) split into Xh/Xl and the row's
                      // sum of squares over the tile into ss_out (skipped when gain_next is null)
    EPI_GU = 3,       // tile = 128 gate rows then their 128 up rows: h = SiLU(g inv) (u inv) split into Hh/Hl
    EPI_GU_MOE = 4,   // EPI_GU for one expert's gathered rows, h also x the token-slot's gate
    EPI_D_MOE = 5     // expert output rows scattered to their (token, slot) places of Yk
};

struct GemmParams {
    int M;            // rows that exist (grouped: the largest possible count; cnt[e] decides)
    int N, K;
    int a_row0;       // first row of A's tensor map (grouped: + e * a_group_rows)
    int a_group_rows;
    int b_row0;       // first row of B's tensor map (grouped: + e * N)
    const int *cnt;   // grouped: rows of group e (null: M rows, no groups)
    // outputs and epilogue inputs
    float *Y;
    int ldy;
    const float *colscale;     // FP8 weights: per-output-column scale, or null
    const float *ss_in;        // [rows][ss_n] partial sums of squares of the RMSNorm input
    int ss_n;
    int dnorm;                 // length of the normed vector (d)
    float eps;
    // EPI_QKV
    lfk::Geo g;
    int pos0, layer;
    const float2 *rope;
    float *Qr;
    __half *kc, *vc;
    // EPI_RESID
    float *X;
    const __half *gain_next;
    __half *Xh, *Xl;
    float *ss_out;
    // EPI_GU / EPI_GU_MOE / EPI_D_MOE
    __half *Hh, *Hl;
    int ldh;
    const int *list;           // grouped rows: t * 8 + slot of row r of group e at list[e * a_group_rows + r]
    const float *gatev;        // [T * 8] gates
    float *Yk;                 // [T, k, d]
    int topk;
    unsigned *status;          // error record (timeouts)
    // split-K (groups == 1 only): the K steps of each tile are cut into
    // `splits` contiguous ranges, one CTA each; every CTA writes its partial
    // tile to part[(tile * splits + s)], and the last one to arrive adds the
    // partials in split order (the same sum whichever CTA is last) and runs
    // the epilogue.  tile_cnt: one zeroed counter per tile, left zeroed.
    int splits;
    float *part;
    unsigned *tile_cnt;
    // optional %globaltimer stamps per CTA (profiling aid, null = off):
    // [cta][4] = entry, first stage landed, last MMA done, epilogue done
    unsigned long long *stamps;
};

}  // namespace lfg

// A [rows, K] (FP16 head and remainder, row-major) x B [rows, K]^T (FP16,
// row-major) into the epilogue `epi`, tile width bn (128 or 256; EPI_GU and
// EPI_GU_MOE need 256); the tensor maps cover the whole arrays.
// grid = (N / bn, ceil(M / 128), groups x splits).  pdl = 1 launches it as a
// programmatic dependent of the previous kernel on the stream (its prologue
// overlaps that kernel's tail; it waits for that kernel before any global
// memory access).
extern "C" cudaError_t lfg_launch(int epi, int bn, const CUtensorMap *a_hi, const CUtensorMap *a_lo,
                                  const CUtensorMap *b, const lfg::GemmParams *p, int groups, int pdl,
                                  cudaStream_t stream);
// Tile width and split count for an M x N x K product on `sms` SMs, from a
// time model of this kernel (waves x (fixed cost + K steps per CTA x cost
// per step) + the split reduction); K is split only while the split CTAs fit
// in one wave and each keeps at least 8 K steps (the partial buffer holds
// sms tiles of 128 x 256).
extern "C" void lfg_plan(int M, int N, int K, int sms, int allow_bn128, int *bn, int *splits);
// 2-D tensor map of a row-major FP16 matrix [rows, cols] read in boxes of
// box_rows x 64 columns with the 128-byte swizzle.  0 on success.
extern "C" int lfg_tensor_map(CUtensorMap *out, const void *base, unsigned long long rows, unsigned long long cols,
                              int box_rows);
