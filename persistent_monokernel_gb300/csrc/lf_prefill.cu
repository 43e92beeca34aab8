// lf_prefill.cu -- batched prefill: the prompt's forward passes over blocks
// of positions at once instead of one decode step per position.  The
// projections of a block are dense GEMMs (T positions x rows x columns), so
// they run on the tensor cores through cuBLAS (FP16 operands, FP32
// accumulation); the causal attention of the block is a flash-style kernel
// of warp-level tensor-core fragments over the cached K/V rows; RMSNorm,
// RoPE, the KV append, SwiGLU and the residual adds are small elementwise
// kernels.  The decode path stays the monokernel: this only fills the KV
// cache, the step before it, with the same arithmetic per position.
//
// Numerics follow the decode path: activations are FP32; every projection
// input is split into an FP16 head and an FP16 remainder (x = hi + lo, about
// 22 significant bits) and multiplied twice with FP32 accumulation, so the
// GEMMs keep FP32-level accuracy against the FP16 weights; q and the softmax
// probabilities are split the same way in the attention products; RMSNorm,
// RoPE (the same FP32 table), SiLU and the softmax are FP32; K and V are
// rounded to FP16 (RNE) into the group-swizzled cache rows the decode kernels
// read.
#include <cublas_v2.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "lf_internal.cuh"
#include "lf_prefill.h"
#include "lf_ptx.cuh"

namespace lfp {

using lfk::Geo;

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    const int nw = blockDim.x >> 5;
    for (int i = 0; i < nw; ++i) t += red[i];
    __syncthreads();
    return t;
}

__device__ __forceinline__ void split_store(float v, __half *hi, __half *lo, size_t i)
{
    const __half h = __float2half_rn(v);
    hi[i] = h;
    lo[i] = __float2half_rn(v - __half2float(h));
}

// X[t] = FP32 embedding row of token tok[t].  Ids outside [0, V) read row 0,
// record STATUS_BAD_TOKEN (where = 400, step = t) and raise the abort flag,
// as the decode path does, so that the next persistent launch stops at once.
__global__ void gather_embed(const int *tok, const __half *E, int d, int V, float *X, unsigned *status, int t_base)
{
    const int t = blockIdx.x;
    int id = tok[t];
    if ((unsigned)id >= (unsigned)V) {
        if (threadIdx.x == 0 && atomicCAS(status, 0u, (unsigned)lfk::STATUS_BAD_TOKEN) == 0u) {
            status[1] = 400u;
            status[2] = 0u;
            status[3] = (unsigned)(t_base + t);
        }
        if (threadIdx.x == 0) atomicExch(status + 4, 1u);
        id = 0;
    }
    for (int i = threadIdx.x; i < d; i += blockDim.x) X[(size_t)t * d + i] = __half2float(E[(size_t)id * d + i]);
}

// RMSNorm of row t times the gain, split into FP16 head and remainder.
__global__ void rmsnorm_split(const float *X, const __half *gain, int d, float eps, __half *Xh, __half *Xl)
{
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float *x = X + (size_t)t * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    const float inv = 1.0f / sqrtf(block_sum(ss, red) / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        split_store(x[i] * inv * __half2float(gain[i]), Xh, Xl, (size_t)t * d + i);
}

// Elementwise split of an FP32 array into FP16 head and remainder.
__global__ void split_f32(const float *A, size_t n, __half *Ah, __half *Al)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        split_store(A[i], Ah, Al, i);
}

// h[t][r] = SiLU(gate[t][r]) * up[t][r] from the fused [T, 2F] projection, split.
__global__ void silu_mul_split(const float *GU, int T, int F, __half *Hh, __half *Hl)
{
    const size_t n = (size_t)T * F;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / F, r = i % F;
        const float gt = GU[t * 2 * F + r], up = GU[t * 2 * F + F + r];
        split_store(gt / (1.0f + expf(-gt)) * up, Hh, Hl, i);
    }
}

__global__ void resid_add(float *X, const float *Y, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        X[i] += Y[i];
}

// FP8 models: Y[t][c] *= s[c] for the N columns of a [T, ldc] output (the
// per-row weight scale, applied after the sum as the decode epilogue does).
__global__ void scale_cols(float *Y, int T, int ldc, int N, const float *s)
{
    const size_t n = (size_t)T * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / N, c = i % N;
        Y[t * ldc + c] *= s[c];
    }
}

__global__ void decode_e4m3(const uint8_t *src, __half *dst, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)src[i], __NV_E4M3));
}

// MXFP4 -> FP16: element k of row r is the E2M1 nibble k (low nibble first)
// times 2^(E - 127) of its 32-element block; exact in FP16 for block scales
// 2^-23 .. 2^13 (lf_create checks them with lfp_byte_range before the decode).
__global__ void decode_mxfp4(const uint8_t *codes, const uint8_t *scales, size_t rows, int cols, __half *dst)
{
    const size_t n = rows * (size_t)cols;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / cols;
        const int k = (int)(i % cols);
        const unsigned byte = codes[r * (size_t)(cols / 2) + k / 2];
        const unsigned nib = (k & 1) ? byte >> 4 : byte & 15u;
        const int ex = (int)((nib >> 1) & 3u), man = (int)(nib & 1u);
        // E2M1: exponent field 0 is the subnormal m * 0.5, else 2^(e-1) * (1 + m/2)
        float mag = ex == 0 ? 0.5f * (float)man : ldexpf(1.0f + 0.5f * (float)man, ex - 1);
        mag = ldexpf(mag, (int)scales[r * (size_t)(cols / 32) + k / 32] - 127);
        dst[i] = __float2half_rn((nib & 8u) ? -mag : mag);
    }
}

__global__ void byte_min_max(const uint8_t *s, size_t n, unsigned *out)
{
    unsigned lo = 255u, hi = 0u;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        lo = min(lo, (unsigned)s[i]);
        hi = max(hi, (unsigned)s[i]);
    }
    atomicMin(out, lo);
    atomicMax(out + 1, hi);
}

// ---- mixture of experts

// Token t's top-k experts from its router logits (ties to the lower index)
// and the softmax of the chosen logits: one warp per token, the monokernel's rule.
__global__ void route_tokens(const float *R, int E, int k, int *sel, float *gate)
{
    const int t = blockIdx.x, lane = threadIdx.x;
    float v0 = lane < E ? R[(size_t)t * E + lane] : -INFINITY;
    float v1 = lane + 32 < E ? R[(size_t)t * E + lane + 32] : -INFINITY;
    float top[8];
    for (int j = 0; j < k; ++j) {
        float bv = v0;
        int bi = lane;
        if (v1 > bv) {
            bv = v1;
            bi = lane + 32;
        }
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi == lane) v0 = -INFINITY;
        else if (bi == lane + 32) v1 = -INFINITY;
        top[j] = bv;
        if (lane == 0) sel[(size_t)t * 8 + j] = min(bi, E - 1);
    }
    if (lane == 0) {
        float sum = 0.f;
        for (int j = 0; j < k; ++j) sum += expf(top[j] - top[0]);
        for (int j = 0; j < k; ++j) gate[(size_t)t * 8 + j] = expf(top[j] - top[0]) / sum;
    }
}

// Per expert (one block each, 256 threads): the (token, slot) pairs routed to
// it, in token order, as t * 8 + j, and their count.
__global__ void build_lists(const int *sel, int T, int k, int *list, int *cnt)
{
    __shared__ int wsum[8];
    const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int base = 0;
    for (int c0 = 0; c0 < T; c0 += 256) {
        const int t = c0 + threadIdx.x;
        int j = -1;
        if (t < T)
            for (int jj = 0; jj < k; ++jj)
                if (sel[(size_t)t * 8 + jj] == e) j = jj;
        const unsigned m = __ballot_sync(0xffffffffu, j >= 0);
        if (lane == 0) wsum[warp] = __popc(m);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < 8; ++w) {
            if (w < warp) before += wsum[w];
            total += wsum[w];
        }
        if (j >= 0) list[(size_t)e * T + base + before + __popc(m & ((1u << lane) - 1u))] = t * 8 + j;
        base += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) cnt[e] = base;
}

// Row i of the gathered input: the FFN input row of token list[i] / 8.
__global__ void gather_rows(const __half *Xh, const __half *Xl, const int *list, int d, __half *Gh, __half *Gl)
{
    const size_t i = blockIdx.x, t = (size_t)(list[i] >> 3);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        Gh[i * d + c] = Xh[t * d + c];
        Gl[i * d + c] = Xl[t * d + c];
    }
}

// h = gate * SiLU(g) * u for the n gathered rows of one expert, split.
__global__ void silu_mul_gate_split(const float *GU, int n, int Fe, const int *list, const float *gatev,
                                    __half *Hh, __half *Hl)
{
    const size_t total = (size_t)n * Fe;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / Fe, c = i % Fe;
        const float gt = GU[r * 2 * Fe + c], up = GU[r * 2 * Fe + Fe + c];
        split_store(gatev[list[r]] * (gt / (1.0f + expf(-gt)) * up), Hh, Hl, i);
    }
}

// The expert's output row i goes to its (token, slot) place.
__global__ void scatter_rows(const float *Y, const int *list, int d, int k, float *Yk)
{
    const size_t i = blockIdx.x;
    const int tj = list[i];
    float *dst = Yk + ((size_t)(tj >> 3) * k + (tj & 7)) * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) dst[c] = Y[i * d + c];
}

// X[t] += the slots' outputs, summed in slot order.
__global__ void combine_slots(float *X, const float *Yk, int k, int d)
{
    const size_t t = blockIdx.x;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc += Yk[(t * k + j) * d + c];
        X[t * d + c] += acc;
    }
}

// RoPE on the q and k heads of row t (rotate-half pairs (j, j + hd/2), the
// FP32 table), q to Qr, K after RoPE and V rounded to FP16 into the cache at
// position pos0 + t of layer l.  Thread u: pair unit u of the fused [q; k; v] row.
__global__ void rope_store(const float *Y, int pos0, int l, Geo g, const float2 *rope, float *Qr, __half *kc,
                           __half *vc)
{
    const int t = blockIdx.x;
    const int half = g.hd / 2;
    const int N = g.Q + 2 * g.KV;
    const int pos = pos0 + t;
    for (int u = threadIdx.x; u < N / 2; u += blockDim.x) {
        const int hh = u / half, j = u % half;
        const float *y = Y + (size_t)t * N + (size_t)hh * g.hd;
        const float v0 = y[j], v1 = y[j + half];
        if (hh < g.Hq + g.Hkv) {
            const float2 cs = rope[(size_t)pos * half + j];
            const float r0 = v0 * cs.x - v1 * cs.y;
            const float r1 = v1 * cs.x + v0 * cs.y;
            if (hh < g.Hq) {
                float *q = Qr + (size_t)t * g.Q + (size_t)hh * g.hd;
                q[j] = r0;
                q[j + half] = r1;
            } else {
                __half *kr = kc + (((size_t)l * g.Hkv + (hh - g.Hq)) * g.max_seq + pos) * g.hd;
                kr[lfk::kv_swz(pos, j)] = __float2half_rn(r0);
                kr[lfk::kv_swz(pos, j + half)] = __float2half_rn(r1);
            }
        } else {
            __half *vr = vc + (((size_t)l * g.Hkv + (hh - g.Hq - g.Hkv)) * g.max_seq + pos) * g.hd;
            vr[lfk::kv_swz(pos, j)] = __float2half_rn(v0);
            vr[lfk::kv_swz(pos, j + half)] = __float2half_rn(v1);
        }
    }
}

// ------------------------------------------------------------- attention

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, unsigned src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int FA_BM = 64;   // query rows of a CTA: four warps of 16
constexpr int FA_BN = 64;   // cached positions per K/V chunk (chunks start at multiples of 64)

template <int HD>
constexpr int fa_smem_bytes()
{
    return (2 * FA_BM + 4 * FA_BN) * HD * 2;   // q head + remainder, K and V double-buffered
}

// Causal attention of the block's rows t0 .. t0+63 (positions pos0 + t) for
// query head blockIdx.y.  Row t attends to cached positions
// attn_first_pos(pos, W) .. pos, which include the block's own rows (written
// by rope_store before this launch).  K/V chunks of 64 positions are copied
// into shared memory verbatim (the cache's group swizzle makes the fragment
// loads conflict-free), double-buffered with cp.async; each warp owns 16 query
// rows and runs, per chunk, S = Q K^T (q as head + remainder: two products),
// the masked online softmax in FP32 (running max and sum per row), and
// O += P V (p as head + remainder).  Output rows are FP32, normalised by the
// final sum.
template <int HD>
__global__ void __launch_bounds__(128) attn_flash(const float *Qr, const __half *kc, const __half *vc, int T, int pos0,
                                                  int l, Geo g, const int *win, float *A)
{
    constexpr int ROW = HD * 2;     // bytes of one FP16 row
    constexpr int KS = HD / 16;     // k-steps of Q K^T
    constexpr int NO = HD / 8;      // n-tiles of O
    constexpr int NS = FA_BN / 8;   // n-tiles of S
    extern __shared__ __align__(128) uint8_t fsm[];
    const uint32_t sqh = lfk::smem_u32(fsm), sql = sqh + FA_BM * ROW;
    const uint32_t sk = sql + FA_BM * ROW, sv = sk + 2 * FA_BN * ROW;
    const int blk = gridDim.x - 1 - blockIdx.x;   // the longest rows first
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;      // fragment coordinates of this lane
    const int t0 = blk * FA_BM;
    const int nrow = min(FA_BM, T - t0);
    const int gkv = h / g.group;
    const int W = win ? win[l] : 0;
    const float scale = 1.0f / sqrtf((float)HD);

    // q rows as FP16 head and remainder, group-swizzled by row
    for (int i = threadIdx.x; i < FA_BM * HD / 2; i += blockDim.x) {
        const int r = i / (HD / 2), c = (i % (HD / 2)) * 2;
        const float2 v =
            *reinterpret_cast<const float2 *>(Qr + (size_t)(t0 + min(r, nrow - 1)) * g.Q + (size_t)h * HD + c);
        __half h0, r0, h1, r1;
        lfk::split_h(v.x, h0, r0);
        lfk::split_h(v.y, h1, r1);
        const int off = r * ROW + lfk::kv_swz(r, c) * 2;
        *reinterpret_cast<unsigned *>(fsm + off) = lfk::pack_h2(h0, h1);
        *reinterpret_cast<unsigned *>(fsm + FA_BM * ROW + off) = lfk::pack_h2(r0, r1);
    }

    const int pos_hi = pos0 + t0 + nrow - 1;
    const int c_begin = lfk::attn_first_pos(pos0 + t0, W) / FA_BN, c_end = pos_hi / FA_BN;
    const size_t head_base = ((size_t)l * g.Hkv + gkv) * g.max_seq * HD;
    const __half *kb = kc + head_base, *vb = vc + head_base;
    // chunk c -> buffer buf; rows past the block's last position are zero-filled
    auto load = [&](int c, int buf) {
        constexpr int PIECES = FA_BN * HD / 8;
        for (int i = threadIdx.x; i < PIECES; i += blockDim.x) {
            const int r = i / (HD / 8), q16 = i % (HD / 8);
            const int p = c * FA_BN + r;
            const bool ok = p <= pos_hi;
            const size_t src = (size_t)(ok ? p : pos_hi) * HD + q16 * 8;
            const uint32_t dst = (uint32_t)(buf * FA_BN * ROW + r * ROW + q16 * 16);
            cp_async16(sk + dst, kb + src, ok ? 16u : 0u);
            cp_async16(sv + dst, vb + src, ok ? 16u : 0u);
        }
        cp_async_commit();
    };

    const int wr0 = warp * 16;
    const bool live = wr0 < nrow;
    const int rowa = wr0 + gq, rowb = rowa + 8;
    const int pa = pos0 + t0 + min(rowa, nrow - 1), pb = pos0 + t0 + min(rowb, nrow - 1);
    const int fa = lfk::attn_first_pos(pa, W), fb = lfk::attn_first_pos(pb, W);
    const int wlo = pos0 + t0 + min(wr0, nrow - 1), whi = pos0 + t0 + min(wr0 + 15, nrow - 1);
    const int wfirst = lfk::attn_first_pos(wlo, W);

    float o[NO][4];
#pragma unroll
    for (int i = 0; i < NO; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

    load(c_begin, 0);
    for (int c = c_begin, it = 0; c <= c_end; ++c, ++it) {
        const int buf = it & 1;
        if (c < c_end) {
            load(c + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int cbase = c * FA_BN;
        if (live && cbase <= whi && cbase + FA_BN - 1 >= wfirst) {
            const uint32_t kbuf = sk + buf * FA_BN * ROW, vbuf = sv + buf * FA_BN * ROW;
            float s[NS][4];
#pragma unroll
            for (int i = 0; i < NS; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                unsigned ah[4], al[4];
                {
                    const int m = lane >> 3, r = wr0 + (m & 1) * 8 + (lane & 7), grp = 2 * kk + (m >> 1);
                    const uint32_t off = r * ROW + ((grp ^ (r & 7)) << 4);
                    lfk::ldsm_x4(ah, sqh + off);
                    lfk::ldsm_x4(al, sql + off);
                }
#pragma unroll
                for (int nb = 0; nb < FA_BN / 16; ++nb) {
                    unsigned bk[4];
                    const int m = lane >> 3, r = nb * 16 + (m >> 1) * 8 + (lane & 7), grp = 2 * kk + (m & 1);
                    lfk::ldsm_x4(bk, kbuf + r * ROW + ((grp ^ (r & 7)) << 4));
                    lfk::mma16816(s[2 * nb], ah[0], ah[1], ah[2], ah[3], bk[0], bk[1]);
                    lfk::mma16816(s[2 * nb], al[0], al[1], al[2], al[3], bk[0], bk[1]);
                    lfk::mma16816(s[2 * nb + 1], ah[0], ah[1], ah[2], ah[3], bk[2], bk[3]);
                    lfk::mma16816(s[2 * nb + 1], al[0], al[1], al[2], al[3], bk[2], bk[3]);
                }
            }
            // mask, online softmax (rows a = gq, b = gq + 8 of the warp's 16)
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NS; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int p = cbase + nt * 8 + 2 * tq + (e & 1);
                    const bool ok = e < 2 ? (p <= pa && p >= fa) : (p <= pb && p >= fb);
                    const float v = ok ? s[nt][e] * scale : -INFINITY;
                    s[nt][e] = v;
                    if (e < 2) mxa = fmaxf(mxa, v);
                    else mxb = fmaxf(mxb, v);
                }
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
            const float refa = na == -INFINITY ? 0.f : na, refb = nb == -INFINITY ? 0.f : nb;
            const float ca = __expf(ma - refa), cb = __expf(mb - refb);   // 0 while the max was -inf
            ma = na;
            mb = nb;
            la *= ca;
            lb *= cb;
#pragma unroll
            for (int i = 0; i < NO; ++i) {
                o[i][0] *= ca;
                o[i][1] *= ca;
                o[i][2] *= cb;
                o[i][3] *= cb;
            }
#pragma unroll
            for (int nt = 0; nt < NS; ++nt) {
                s[nt][0] = __expf(s[nt][0] - refa);
                s[nt][1] = __expf(s[nt][1] - refa);
                s[nt][2] = __expf(s[nt][2] - refb);
                s[nt][3] = __expf(s[nt][3] - refb);
                la += s[nt][0] + s[nt][1];
                lb += s[nt][2] + s[nt][3];
            }
            // O += P V: P (16 x 64) as the A operand straight from the score
            // accumulators, V rows as the B operand through transposing loads
#pragma unroll
            for (int kk = 0; kk < FA_BN / 16; ++kk) {
                unsigned ph[4], pl[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float *src = &s[2 * kk + (q >> 1)][(q & 1) * 2];
                    __half h0, r0, h1, r1;
                    lfk::split_h(src[0], h0, r0);
                    lfk::split_h(src[1], h1, r1);
                    ph[q] = lfk::pack_h2(h0, h1);
                    pl[q] = lfk::pack_h2(r0, r1);
                }
#pragma unroll
                for (int nb = 0; nb < HD / 16; ++nb) {
                    unsigned bv[4];
                    const int m = lane >> 3, r = kk * 16 + (m & 1) * 8 + (lane & 7), grp = 2 * nb + (m >> 1);
                    lfk::ldsm_x4_t(bv, vbuf + r * ROW + ((grp ^ (r & 7)) << 4));
                    lfk::mma16816(o[2 * nb], ph[0], ph[1], ph[2], ph[3], bv[0], bv[1]);
                    lfk::mma16816(o[2 * nb], pl[0], pl[1], pl[2], pl[3], bv[0], bv[1]);
                    lfk::mma16816(o[2 * nb + 1], ph[0], ph[1], ph[2], ph[3], bv[2], bv[3]);
                    lfk::mma16816(o[2 * nb + 1], pl[0], pl[1], pl[2], pl[3], bv[2], bv[3]);
                }
            }
        }
        __syncthreads();   // every warp is done with this buffer before it is refilled
    }

    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    if (!live) return;
    const float ia = 1.0f / la, ib = 1.0f / lb;
#pragma unroll
    for (int i = 0; i < NO; ++i) {
        const int col = h * HD + i * 8 + 2 * tq;
        if (rowa < nrow)
            *reinterpret_cast<float2 *>(A + (size_t)(t0 + rowa) * g.Q + col) = make_float2(o[i][0] * ia, o[i][1] * ia);
        if (rowb < nrow)
            *reinterpret_cast<float2 *>(A + (size_t)(t0 + rowb) * g.Q + col) = make_float2(o[i][2] * ib, o[i][3] * ib);
    }
}

// ------------------------------------------------------------- host side

// Y[T x N] (row-major, leading dimension ldc) = X W^T for W [N x K] row-major
// and X = Xh + Xl [T x K] row-major: two FP16 GEMMs into one FP32 result.
cublasStatus_t gemm2(cublasHandle_t cb, const __half *W, int N, int K, const __half *Xh, const __half *Xl, int T,
                     float *Y, int ldc)
{
    const float one = 1.0f, zero = 0.0f;
    cublasStatus_t st = cublasGemmEx(cb, CUBLAS_OP_T, CUBLAS_OP_N, N, T, K, &one, W, CUDA_R_16F, K, Xh, CUDA_R_16F,
                                     K, &zero, Y, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (st != CUBLAS_STATUS_SUCCESS) return st;
    return cublasGemmEx(cb, CUBLAS_OP_T, CUBLAS_OP_N, N, T, K, &one, W, CUDA_R_16F, K, Xl, CUDA_R_16F, K, &one, Y,
                        CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
}

int grid_for(size_t n) { return (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, 8 * 1024)); }

// The mixture-of-experts FFN of layer l for the block's T rows (input in
// w.Xh / w.Xl): router GEMM, routing, then per expert with tokens a gather,
// the gate/up GEMM, the gated SiLU product, the down GEMM and a scatter to
// the (token, slot) places; the slots are summed into the residual in order.
int moe_ffn(const lfp_args *a, cublasHandle_t cb, cudaStream_t s, int l, int T, int *cnt_host)
{
    const Geo &g = a->g;
    const lfp_workspace &w = a->ws;
    const int E = g.E, k = g.topk, Fe = g.Fe, d = g.d;
    if (gemm2(cb, a->router + (size_t)l * E * d, E, d, w.Xh, w.Xl, T, w.R, E)) return 3;
    route_tokens<<<T, 32, 0, s>>>(w.R, E, k, w.sel, w.gate);
    build_lists<<<E, 256, 0, s>>>(w.sel, T, k, w.list, w.cnt);
    if (cudaMemcpyAsync(cnt_host, w.cnt, sizeof(int) * E, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return 1;
    for (int e = 0; e < E; ++e) {
        const int n = cnt_host[e];
        if (n <= 0) continue;
        const int *lst = w.list + (size_t)e * T;
        const size_t ex = (size_t)l * E + e;
        gather_rows<<<n, 256, 0, s>>>(w.Xh, w.Xl, lst, d, w.Xgh, w.Xgl);
        if (gemm2(cb, a->wgu + ex * 2 * Fe * d, 2 * Fe, d, w.Xgh, w.Xgl, n, w.GU, 2 * Fe)) return 3;
        silu_mul_gate_split<<<grid_for((size_t)n * Fe), 256, 0, s>>>(w.GU, n, Fe, lst, w.gate, w.Hh, w.Hl);
        if (gemm2(cb, a->wd + ex * d * Fe, d, Fe, w.Hh, w.Hl, n, w.Y, d)) return 3;
        scatter_rows<<<n, 256, 0, s>>>(w.Y, lst, d, k, w.Yk);
    }
    combine_slots<<<T, 256, 0, s>>>(w.X, w.Yk, k, d);
    return 0;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace lfp

// The workspace's parts, carved from `base` (or only sized when base is null).
static size_t lfp_layout(const lfk::Geo &g, int block, uint8_t *base, lfp_workspace *w)
{
    using lfp::align256;
    const size_t T = (size_t)block;
    const size_t kmax = (size_t)std::max(g.d, std::max(g.Q, g.F));
    const size_t ymax = (size_t)std::max(g.Q + 2 * g.KV, g.d);
    size_t o = 0;
    auto take = [&](size_t bytes) -> void * {
        void *p = base ? static_cast<void *>(base + o) : nullptr;
        o += align256(bytes);
        return p;
    };
    *w = lfp_workspace{};
    w->X = static_cast<float *>(take(T * g.d * 4));
    w->Xh = static_cast<__half *>(take(T * kmax * 2));
    w->Xl = static_cast<__half *>(take(T * kmax * 2));
    w->Y = static_cast<float *>(take(T * ymax * 4));
    w->Qr = static_cast<float *>(take(T * g.Q * 4));
    w->A = static_cast<float *>(take(T * g.Q * 4));
    w->GU = static_cast<float *>(take(T * 2 * g.F * 4));
    if (g.E > 0) {
        w->R = static_cast<float *>(take(T * g.E * 4));
        w->sel = static_cast<int *>(take(T * 8 * 4));
        w->gate = static_cast<float *>(take(T * 8 * 4));
        w->list = static_cast<int *>(take((size_t)g.E * T * 4));
        w->cnt = static_cast<int *>(take((size_t)g.E * 4));
        w->Xgh = static_cast<__half *>(take(T * g.d * 2));
        w->Xgl = static_cast<__half *>(take(T * g.d * 2));
        w->Hh = static_cast<__half *>(take(T * g.Fe * 2));
        w->Hl = static_cast<__half *>(take(T * g.Fe * 2));
        w->Yk = static_cast<float *>(take(T * g.topk * g.d * 4));
    }
    return o;
}

size_t lfp_workspace_bytes(const lfk::Geo &g, int block)
{
    lfp_workspace w;
    return lfp_layout(g, block, nullptr, &w);
}

lfp_workspace lfp_carve(void *base, const lfk::Geo &g, int block)
{
    lfp_workspace w;
    lfp_layout(g, block, static_cast<uint8_t *>(base), &w);
    return w;
}

extern "C" int lfp_cublas_create(void **out)
{
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return 1;
    // FP32 accumulation throughout; no reduced-precision split reductions
    if (cublasSetMathMode(h, CUBLAS_MATH_DISALLOW_REDUCED_PRECISION_REDUCTION) != CUBLAS_STATUS_SUCCESS) {
        cublasDestroy(h);
        return 1;
    }
    *out = h;
    return 0;
}

extern "C" void lfp_cublas_destroy(void *h)
{
    if (h) cublasDestroy(static_cast<cublasHandle_t>(h));
}

extern "C" cudaError_t lfp_decode_e4m3(const uint8_t *src, __half *dst, size_t n, cudaStream_t stream)
{
    lfp::decode_e4m3<<<lfp::grid_for(n), 256, 0, stream>>>(src, dst, n);
    return cudaGetLastError();
}

extern "C" cudaError_t lfp_decode_mxfp4(const uint8_t *codes, const uint8_t *scales, size_t rows, int cols,
                                         __half *dst, cudaStream_t stream)
{
    lfp::decode_mxfp4<<<lfp::grid_for(rows * (size_t)cols), 256, 0, stream>>>(codes, scales, rows, cols, dst);
    return cudaGetLastError();
}

extern "C" cudaError_t lfp_byte_range(const uint8_t *s, size_t n, unsigned *lo, unsigned *hi)
{
    unsigned *d = nullptr;
    cudaError_t e = cudaMalloc(&d, 2 * sizeof(unsigned));
    const unsigned init[2] = {255u, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(d, init, sizeof(init), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        lfp::byte_min_max<<<lfp::grid_for(n), 256>>>(s, n, d);
        e = cudaGetLastError();
    }
    unsigned res[2] = {255u, 0u};
    if (e == cudaSuccess) e = cudaMemcpy(res, d, sizeof(res), cudaMemcpyDeviceToHost);
    if (d) cudaFree(d);
    *lo = res[0];
    *hi = res[1];
    return e;
}

extern "C" int lfp_run(const lfp_args *a, cudaStream_t s)
{
    using namespace lfp;
    const Geo &g = a->g;
    cublasHandle_t cb = static_cast<cublasHandle_t>(a->cublas);
    if (cublasSetStream(cb, s) != CUBLAS_STATUS_SUCCESS) return 2;
    const int d = g.d, Q = g.Q, F = g.F, NQKV = g.Q + 2 * g.KV;
    const int fa_smem = g.hd == 64 ? fa_smem_bytes<64>() : fa_smem_bytes<128>();
    cudaError_t e = g.hd == 64
                        ? cudaFuncSetAttribute(attn_flash<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem)
                        : cudaFuncSetAttribute(attn_flash<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem);
    if (e != cudaSuccess) return 1;
    const lfp_workspace &w = a->ws;
    std::vector<int> cnt_host(g.E > 0 ? g.E : 1);
    for (int t0 = 0; t0 < a->n; t0 += a->block) {
        const int T = std::min(a->block, a->n - t0);
        const int pos0 = a->pos0 + t0;
        const dim3 fa_grid((T + FA_BM - 1) / FA_BM, g.Hq);
        gather_embed<<<T, 256, 0, s>>>(a->tokens + t0, a->embed, d, g.V, w.X, a->status, t0);
        for (int l = 0; l < g.L; ++l) {
            // attention block
            rmsnorm_split<<<T, 256, 0, s>>>(w.X, a->attn_norm + (size_t)l * d, d, a->eps, w.Xh, w.Xl);
            if (gemm2(cb, a->wqkv + (size_t)l * NQKV * d, NQKV, d, w.Xh, w.Xl, T, w.Y, NQKV)) return 3;
            if (a->sqkv)
                scale_cols<<<grid_for((size_t)T * NQKV), 256, 0, s>>>(w.Y, T, NQKV, NQKV, a->sqkv + (size_t)l * NQKV);
            rope_store<<<T, 256, 0, s>>>(w.Y, pos0, l, g, a->rope, w.Qr, a->kc, a->vc);
            if (g.hd == 64)
                attn_flash<64><<<fa_grid, 128, fa_smem, s>>>(w.Qr, a->kc, a->vc, T, pos0, l, g, a->win, w.A);
            else
                attn_flash<128><<<fa_grid, 128, fa_smem, s>>>(w.Qr, a->kc, a->vc, T, pos0, l, g, a->win, w.A);
            split_f32<<<grid_for((size_t)T * Q), 256, 0, s>>>(w.A, (size_t)T * Q, w.Xh, w.Xl);
            if (gemm2(cb, a->wo + (size_t)l * d * Q, d, Q, w.Xh, w.Xl, T, w.Y, d)) return 3;
            if (a->so) scale_cols<<<grid_for((size_t)T * d), 256, 0, s>>>(w.Y, T, d, d, a->so + (size_t)l * d);
            resid_add<<<grid_for((size_t)T * d), 256, 0, s>>>(w.X, w.Y, (size_t)T * d);
            // SwiGLU block (or the mixture of experts)
            rmsnorm_split<<<T, 256, 0, s>>>(w.X, a->ffn_norm + (size_t)l * d, d, a->eps, w.Xh, w.Xl);
            if (g.E > 0) {
                const int r = moe_ffn(a, cb, s, l, T, cnt_host.data());
                if (r) return r;
                continue;
            }
            if (gemm2(cb, a->wgu + (size_t)l * 2 * F * d, 2 * F, d, w.Xh, w.Xl, T, w.GU, 2 * F)) return 3;
            if (a->sgu)
                scale_cols<<<grid_for((size_t)T * 2 * F), 256, 0, s>>>(w.GU, T, 2 * F, 2 * F,
                                                                       a->sgu + (size_t)l * 2 * F);
            silu_mul_split<<<grid_for((size_t)T * F), 256, 0, s>>>(w.GU, T, F, w.Xh, w.Xl);
            if (gemm2(cb, a->wd + (size_t)l * d * F, d, F, w.Xh, w.Xl, T, w.Y, d)) return 3;
            if (a->sd) scale_cols<<<grid_for((size_t)T * d), 256, 0, s>>>(w.Y, T, d, d, a->sd + (size_t)l * d);
            resid_add<<<grid_for((size_t)T * d), 256, 0, s>>>(w.X, w.Y, (size_t)T * d);
        }
        if (cudaGetLastError() != cudaSuccess) return 1;
    }
    return 0;
}
