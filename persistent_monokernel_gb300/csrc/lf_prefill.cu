// lf_prefill.cu -- batched prefill: the prompt's forward passes over blocks
// of positions at once instead of one decode step per position.  The
// projections of a block are dense GEMMs (T positions x rows x columns) on
// the sm_103a tensor cores (lf_gemm.cu: tcgen05.mma, TMA-staged operands,
// TMEM accumulators), each with the elementwise work that follows it fused
// into its epilogue; the causal attention of the block is a flash-style
// kernel of warp-level tensor-core fragments over the cached K/V rows.  Per
// layer and block, five launches:
//
//   QKV GEMM   (x g) . Wqkv^T, x the RMSNorm factor, RoPE, q out, K/V into the cache
//   attention  causal over the cache, output split for the O GEMM
//   O GEMM     residual add, then the FFN RMSNorm's input (x g_ffn, split) and
//              its per-tile sums of squares
//   GU GEMM    x the RMSNorm factor, SiLU(gate) * up, split for the down GEMM
//   D GEMM     residual add, then the next layer's RMSNorm input the same way
//
// The decode path stays the monokernel: this only fills the KV cache, the
// step before it, with the same arithmetic per position.
//
// Numerics follow the decode path: activations are FP32; every projection
// input is split into an FP16 head and an FP16 remainder (x = hi + lo, about
// 22 significant bits) and multiplied twice with FP32 accumulation, so the
// GEMMs keep FP32-level accuracy against the FP16 weights; q and the softmax
// probabilities are split the same way in the attention products; RMSNorm,
// RoPE (the same FP32 table), SiLU and the softmax are FP32; K and V are
// rounded to FP16 (RNE) into the group-swizzled cache rows the decode kernels
// read.  The RMSNorm gain multiplies the GEMM input and the factor
// 1/sqrt(mean(x^2) + eps) the GEMM output (the same product, rounded in a
// different order); the mean comes from per-128-column partial sums written
// by the kernel that produced x.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "lf_gemm.h"
#include "lf_internal.cuh"

extern "C" cudaError_t lfa_launch(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const float *Qr, int T, int pos0,
                                  int l, lfk::Geo g, const int *win, __half *Ah, __half *Al, unsigned *status,
                                  unsigned long long *stamps, cudaStream_t stream);
extern "C" int lfa_cache_map(CUtensorMap *out, const void *cache, unsigned long long rows);
#include "lf_prefill.h"
#include "lf_ptx.cuh"

namespace lfp {

using lfk::Geo;

constexpr int NG = 128;   // columns per partial sum of squares (the O / down GEMM tile width)

__device__ __forceinline__ void split_store(float v, __half *hi, __half *lo, size_t i)
{
    const __half h = __float2half_rn(v);
    hi[i] = h;
    lo[i] = __float2half_rn(v - __half2float(h));
}

// The next RMSNorm's input for row t of X: X x gain split into Xh / Xl, and
// the sum of squares of every 128-column group into SS[t][group].  One block
// of 128 threads per row.
__device__ __forceinline__ void norm_prep_row(const float *x, const __half *gain, int d, __half *Xh, __half *Xl,
                                              float *ss, size_t t)
{
    __shared__ float red[4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int g0 = 0; g0 < d; g0 += NG) {
        const int c = g0 + threadIdx.x;
        const float v = x[c];
        split_store(v * __half2float(gain[c]), Xh, Xl, t * d + c);
        float s = v * v;
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) red[warp] = s;
        __syncthreads();
        if (threadIdx.x == 0) ss[t * (d / NG) + g0 / NG] = (red[0] + red[1]) + (red[2] + red[3]);
        __syncthreads();
    }
}

// X[t] = FP32 embedding row of token tok[t], then layer 0's RMSNorm input.
// Ids outside [0, V) read row 0, record STATUS_BAD_TOKEN (where = 400, step =
// t) and raise the abort flag, as the decode path does, so that the next
// persistent launch stops at once.
__global__ void __launch_bounds__(128) embed_prep(const int *tok, const __half *E, int d, int V, const __half *gain,
                                                  float *X, __half *Xh, __half *Xl, float *SS, unsigned *status,
                                                  int t_base)
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
    float *x = X + (size_t)t * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) x[i] = __half2float(E[(size_t)id * d + i]);
    __syncthreads();
    norm_prep_row(x, gain, d, Xh, Xl, SS, (size_t)t);
}


int grid_for(size_t n) { return (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, 8 * 1024)); }

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
// it, in token order, as t * 8 + j, at list[e * ld ..], and their count.
__global__ void build_lists(const int *sel, int T, int k, int ld, int *list, int *cnt)
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
        if (j >= 0) list[(size_t)e * ld + base + before + __popc(m & ((1u << lane) - 1u))] = t * 8 + j;
        base += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) cnt[e] = base;
}


// Router logits of token t: W_r . (x g), times the RMSNorm factor (the
// monokernel's order: FP32 dots of the FP16 router rows with x * gain, then
// the positive scale).  One block of 256 threads per token; warp w takes
// experts w, w + 8, ...
__global__ void __launch_bounds__(256) router_logits(const float *X, const __half *gain, const __half *Wr, int E, int d,
                                                     float eps, float *R)
{
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *x = X + (size_t)t * d;
    __shared__ float red[8];
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    for (int e = warp; e < E; e += 8) {
        const __half *row = Wr + (size_t)e * d;
        float acc = 0.f;
        for (int i = lane; i < d; i += 32) acc = fmaf(__half2float(row[i]), x[i] * __half2float(gain[i]), acc);
#pragma unroll
        for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) R[(size_t)t * E + e] = acc * inv;
    }
}

// Row i of expert e's gathered GEMM input: the FFN input row (split) of the
// token of list[e][i]; rows past the expert's count stay untouched.
__global__ void gather_rows(const __half *Xh, const __half *Xl, const int *list, const int *cnt, int T, int d,
                            __half *Gh, __half *Gl)
{
    const int i = blockIdx.x, e = blockIdx.y;
    if (i >= cnt[e]) return;
    const size_t row = (size_t)e * T + i, t = (size_t)(list[row] >> 3);
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        Gh[row * d + c] = Xh[t * d + c];
        Gl[row * d + c] = Xl[t * d + c];
    }
}

// X[t] += the slots' expert outputs (slot order), then the next RMSNorm's
// input of the row (skipped after the last layer: gain null).
__global__ void __launch_bounds__(128) combine_prep(float *X, const float *Yk, int k, int d, const __half *gain,
                                                    __half *Xh, __half *Xl, float *SS)
{
    const size_t t = blockIdx.x;
    float *x = X + t * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j) acc += Yk[(t * k + j) * d + c];
        x[c] += acc;
    }
    __syncthreads();
    if (gain) norm_prep_row(x, gain, d, Xh, Xl, SS, t);
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
// O += P V (p as head + remainder).  Output rows, normalised by the final
// sum, are stored as FP16 head and remainder: the O projection's GEMM operand.
template <int HD>
__global__ void __launch_bounds__(128) attn_flash(const float *Qr, const __half *kc, const __half *vc, int T, int pos0,
                                                  int l, Geo g, const int *win, __half *Ah, __half *Al)
{
    constexpr int ROW = HD * 2;     // bytes of one FP16 row
    constexpr int KS = HD / 16;     // k-steps of Q K^T
    constexpr int NO = HD / 8;      // n-tiles of O
    constexpr int NS = FA_BN / 8;   // n-tiles of S
    extern __shared__ __align__(128) uint8_t fsm[];
    const uint32_t sqh = lfk::smem_u32(fsm), sql = sqh + FA_BM * ROW;
    const uint32_t sk = sql + FA_BM * ROW, sv = sk + 2 * FA_BN * ROW;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // launched as a programmatic dependent
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
        __half h0, r0, h1, r1;
        if (rowa < nrow) {
            const size_t o0 = (size_t)(t0 + rowa) * g.Q + col;
            lfk::split_h(o[i][0] * ia, h0, r0);
            lfk::split_h(o[i][1] * ia, h1, r1);
            *reinterpret_cast<unsigned *>(Ah + o0) = lfk::pack_h2(h0, h1);
            *reinterpret_cast<unsigned *>(Al + o0) = lfk::pack_h2(r0, r1);
        }
        if (rowb < nrow) {
            const size_t o1 = (size_t)(t0 + rowb) * g.Q + col;
            lfk::split_h(o[i][2] * ib, h0, r0);
            lfk::split_h(o[i][3] * ib, h1, r1);
            *reinterpret_cast<unsigned *>(Ah + o1) = lfk::pack_h2(h0, h1);
            *reinterpret_cast<unsigned *>(Al + o1) = lfk::pack_h2(r0, r1);
        }
    }
}

// ------------------------------------------------------------- host side

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace lfp

// The workspace's parts, carved from `base` (or only sized when base is null).
static size_t lfp_layout(const lfk::Geo &g, int block, int sms, uint8_t *base, lfp_workspace *w)
{
    using lfp::align256;
    const size_t T = (size_t)block;
    const size_t hrows = g.E > 0 ? (size_t)g.E * T : T;   // hidden rows: per expert when routed
    const size_t hcols = g.E > 0 ? (size_t)g.Fe : (size_t)g.F;
    size_t o = 0;
    auto take = [&](size_t bytes) -> void * {
        void *p = base ? static_cast<void *>(base + o) : nullptr;
        o += align256(bytes);
        return p;
    };
    *w = lfp_workspace{};
    w->X = static_cast<float *>(take(T * g.d * 4));
    w->Xh = static_cast<__half *>(take(T * g.d * 2));
    w->Xl = static_cast<__half *>(take(T * g.d * 2));
    w->SS = static_cast<float *>(take(T * (g.d / lfp::NG) * 4));
    w->Qr = static_cast<float *>(take(T * g.Q * 4));
    w->Ah = static_cast<__half *>(take(T * g.Q * 2));
    w->Al = static_cast<__half *>(take(T * g.Q * 2));
    w->Hh = static_cast<__half *>(take(hrows * hcols * 2));
    w->Hl = static_cast<__half *>(take(hrows * hcols * 2));
    if (g.E > 0) {
        w->R = static_cast<float *>(take(T * g.E * 4));
        w->sel = static_cast<int *>(take(T * 8 * 4));
        w->gate = static_cast<float *>(take(T * 8 * 4));
        w->list = static_cast<int *>(take((size_t)g.E * T * 4));
        w->cnt = static_cast<int *>(take((size_t)g.E * 4));
        w->Xgh = static_cast<__half *>(take((size_t)g.E * T * g.d * 2));
        w->Xgl = static_cast<__half *>(take((size_t)g.E * T * g.d * 2));
        w->Yk = static_cast<float *>(take(T * g.topk * g.d * 4));
    }
    w->part = static_cast<float *>(take((size_t)sms * 128 * 256 * 4));
    w->tile_cnt = static_cast<unsigned *>(take(1024 * 4));
    return o;
}

size_t lfp_workspace_bytes(const lfk::Geo &g, int block, int sms)
{
    lfp_workspace w;
    return lfp_layout(g, block, sms, nullptr, &w);
}

lfp_workspace lfp_carve(void *base, const lfk::Geo &g, int block, int sms)
{
    lfp_workspace w;
    lfp_layout(g, block, sms, static_cast<uint8_t *>(base), &w);
    return w;
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

// Tensor maps of the GEMM operands: the workspace's split activations and
// the four stacked weight arrays.  0 on success.
extern "C" int lfp_make_maps(const lfp_args *a, lfp_maps *m)
{
    const lfk::Geo &g = a->g;
    const lfp_workspace &w = a->ws;
    const unsigned long long T = (unsigned long long)a->block, L = (unsigned long long)g.L;
    const unsigned long long d = g.d, Q = g.Q, NQKV = g.Q + 2 * g.KV;
    int r = 0;
    r |= lfg_tensor_map(&m->xh, w.Xh, T, d, lfg::BM);
    r |= lfg_tensor_map(&m->xl, w.Xl, T, d, lfg::BM);
    r |= lfg_tensor_map(&m->ah, w.Ah, T, Q, lfg::BM);
    r |= lfg_tensor_map(&m->al, w.Al, T, Q, lfg::BM);
    for (int i = 0; i < 2; ++i) {
        r |= lfg_tensor_map(&m->wqkv[i], a->wqkv, L * NQKV, d, 128 << i);
        r |= lfg_tensor_map(&m->wo[i], a->wo, L * d, Q, 128 << i);
    }
    if (g.hd == 128) {
        const unsigned long long rows = L * (unsigned long long)g.Hkv * (unsigned long long)g.max_seq;
        r |= lfa_cache_map(&m->kc, a->kc, rows);
        r |= lfa_cache_map(&m->vc, a->vc, rows);
    }
    if (g.E > 0) {
        const unsigned long long E = g.E, Fe = g.Fe;
        r |= lfg_tensor_map(&m->hh, w.Hh, E * T, Fe, lfg::BM);
        r |= lfg_tensor_map(&m->hl, w.Hl, E * T, Fe, lfg::BM);
        r |= lfg_tensor_map(&m->xgh, w.Xgh, E * T, d, lfg::BM);
        r |= lfg_tensor_map(&m->xgl, w.Xgl, E * T, d, lfg::BM);
        r |= lfg_tensor_map(&m->wgu, a->wgu, L * E * 2 * Fe, d, 256);
        for (int i = 0; i < 2; ++i) r |= lfg_tensor_map(&m->wd[i], a->wd, L * E * d, Fe, 128 << i);
    } else {
        const unsigned long long F = g.F;
        r |= lfg_tensor_map(&m->hh, w.Hh, T, F, lfg::BM);
        r |= lfg_tensor_map(&m->hl, w.Hl, T, F, lfg::BM);
        r |= lfg_tensor_map(&m->wgu, a->wgu, L * 2 * F, d, 256);
        for (int i = 0; i < 2; ++i) r |= lfg_tensor_map(&m->wd[i], a->wd, L * d, F, 128 << i);
    }
    return r ? 1 : 0;
}

extern "C" int lfp_run(const lfp_args *a, const lfp_maps *m, cudaStream_t s)
{
    using namespace lfp;
    const Geo &g = a->g;
    const int d = g.d, NQKV = g.Q + 2 * g.KV;
    const int fa_smem = g.hd == 64 ? fa_smem_bytes<64>() : fa_smem_bytes<128>();
    cudaError_t e = g.hd == 64
                        ? cudaFuncSetAttribute(attn_flash<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem)
                        : cudaFuncSetAttribute(attn_flash<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, fa_smem);
    if (e != cudaSuccess) return 1;
    const lfp_workspace &w = a->ws;
    // tile width and split count per product; the weight map whose box matches the width
    auto plan = [&](lfg::GemmParams &q, int M, bool allow128) {
        int bn = 256, sp = 1;
        lfg_plan(M, q.N, q.K, a->sms, allow128 ? 1 : 0, &bn, &sp);
        q.splits = sp;
        q.part = w.part;
        q.tile_cnt = w.tile_cnt;
        return bn;
    };
    for (int t0 = 0; t0 < a->n; t0 += a->block) {
        const int T = std::min(a->block, a->n - t0);
        const int pos0 = a->pos0 + t0;
        const dim3 fa_grid((T + FA_BM - 1) / FA_BM, g.Hq);
        embed_prep<<<T, 128, 0, s>>>(a->tokens + t0, a->embed, d, g.V, a->attn_norm, w.X, w.Xh, w.Xl, w.SS, a->status,
                                     t0);
        for (int l = 0; l < g.L; ++l) {
            const __half *next_gain = l + 1 < g.L ? a->attn_norm + (size_t)(l + 1) * d : nullptr;
            lfg::GemmParams p = {};
            p.M = T;
            p.g = g;
            p.eps = a->eps;
            p.ss_in = w.SS;
            p.ss_n = d / NG;
            p.dnorm = d;
            p.status = a->status;
            // ---- attention block
            lfg::GemmParams q = p;
            q.N = NQKV;
            q.K = d;
            q.b_row0 = l * NQKV;
            q.colscale = a->sqkv ? a->sqkv + (size_t)l * NQKV : nullptr;
            q.pos0 = pos0;
            q.layer = l;
            q.rope = a->rope;
            q.Qr = w.Qr;
            q.kc = a->kc;
            q.vc = a->vc;
            const int bq = plan(q, T, true);
            if (lfg_launch(lfg::EPI_QKV, bq, &m->xh, &m->xl, &m->wqkv[bq / 256], &q, 1, 1, s) != cudaSuccess) return 1;
            if (g.hd == 128) {
                if (lfa_launch(&m->kc, &m->vc, w.Qr, T, pos0, l, g, a->win, w.Ah, w.Al, a->status,
                               l == 1 && t0 == 0 ? a->attn_stamps : nullptr, s) != cudaSuccess)
                    return 1;
            } else {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = fa_grid;
                cfg.blockDim = dim3(128);
                cfg.dynamicSmemBytes = (size_t)fa_smem;
                cfg.stream = s;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaLaunchKernelEx(&cfg, attn_flash<64>, (const float *)w.Qr, (const __half *)a->kc,
                                       (const __half *)a->vc, T, pos0, l, g, a->win, w.Ah, w.Al) != cudaSuccess)
                    return 1;
            }
            lfg::GemmParams o = p;
            o.N = d;
            o.K = g.Q;
            o.b_row0 = l * d;
            o.colscale = a->so ? a->so + (size_t)l * d : nullptr;
            o.X = w.X;
            o.gain_next = a->ffn_norm + (size_t)l * d;
            o.Xh = w.Xh;
            o.Xl = w.Xl;
            o.ss_out = w.SS;
            const int bo = plan(o, T, true);
            if (lfg_launch(lfg::EPI_RESID, bo, &m->ah, &m->al, &m->wo[bo / 256], &o, 1, 1, s) != cudaSuccess) return 1;
            // ---- SwiGLU block
            if (g.E > 0) {
                const int E = g.E, k = g.topk, Fe = g.Fe;
                router_logits<<<T, 256, 0, s>>>(w.X, a->ffn_norm + (size_t)l * d, a->router + (size_t)l * E * d, E, d,
                                                a->eps, w.R);
                route_tokens<<<T, 32, 0, s>>>(w.R, E, k, w.sel, w.gate);
                build_lists<<<E, 256, 0, s>>>(w.sel, T, k, a->block, w.list, w.cnt);
                gather_rows<<<dim3(T, E), 256, 0, s>>>(w.Xh, w.Xl, w.list, w.cnt, a->block, d, w.Xgh, w.Xgl);
                lfg::GemmParams u = p;
                u.M = T;
                u.N = 2 * Fe;
                u.K = d;
                u.a_group_rows = a->block;
                u.b_row0 = l * E * 2 * Fe;
                u.cnt = w.cnt;
                u.list = w.list;
                u.gatev = w.gate;
                u.Hh = w.Hh;
                u.Hl = w.Hl;
                u.ldh = Fe;
                if (lfg_launch(lfg::EPI_GU_MOE, 256, &m->xgh, &m->xgl, &m->wgu, &u, E, 1, s) != cudaSuccess) return 1;
                lfg::GemmParams dn = p;
                dn.M = T;
                dn.N = d;
                dn.K = Fe;
                dn.a_group_rows = a->block;
                dn.b_row0 = l * E * d;
                dn.cnt = w.cnt;
                dn.list = w.list;
                dn.Yk = w.Yk;
                dn.topk = k;
                if (lfg_launch(lfg::EPI_D_MOE, 128, &m->hh, &m->hl, &m->wd[0], &dn, E, 1, s) != cudaSuccess) return 1;
                combine_prep<<<T, 128, 0, s>>>(w.X, w.Yk, k, d, next_gain, w.Xh, w.Xl, w.SS);
                continue;
            }
            lfg::GemmParams u = p;
            u.N = 2 * g.F;
            u.K = d;
            u.b_row0 = l * 2 * g.F;
            u.colscale = a->sgu ? a->sgu + (size_t)l * 2 * g.F : nullptr;
            u.Hh = w.Hh;
            u.Hl = w.Hl;
            u.ldh = g.F;
            plan(u, T, false);
            if (lfg_launch(lfg::EPI_GU, 256, &m->xh, &m->xl, &m->wgu, &u, 1, 1, s) != cudaSuccess) return 1;
            lfg::GemmParams dn = p;
            dn.N = d;
            dn.K = g.F;
            dn.b_row0 = l * d;
            dn.colscale = a->sd ? a->sd + (size_t)l * d : nullptr;
            dn.X = w.X;
            dn.gain_next = next_gain;
            dn.Xh = w.Xh;
            dn.Xl = w.Xl;
            dn.ss_out = w.SS;
            const int bd = plan(dn, T, true);
            if (lfg_launch(lfg::EPI_RESID, bd, &m->hh, &m->hl, &m->wd[bd / 256], &dn, 1, 1, s) != cudaSuccess) return 1;
        }
        if (cudaGetLastError() != cudaSuccess) return 1;
    }
    return 0;
}
