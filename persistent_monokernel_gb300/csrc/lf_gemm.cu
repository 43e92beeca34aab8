// lf_gemm.cu -- the batched prefill's projections on the sm_103a tensor cores.
//
// C = A . B^T with A the block's activations [positions, K] and B a weight
// matrix [rows, K] (nn.Linear layout), both K-major FP16.  The activations
// come as an FP16 head and remainder (x = hi + lo, about 22 significant
// bits), so every K step issues two MMAs on the same weight tile and the FP32
// accumulator in TMEM sums hi . W^T + lo . W^T: FP32-level activations against
// FP16 weights, as the decode GEMVs compute them.
//
// One CTA computes one 128 x BN output tile (BN 128 or 256): warp 4 streams
// the A-head, A-remainder and B tiles of each 64-wide K step into a ring of
// shared-memory stages with 2-D TMA loads (128-byte swizzle); warp 5
// allocates the TMEM accumulator and issues the tcgen05.mma instructions from
// one thread, each stage released back to the loader by a tcgen05.commit;
// warps 0-3 wait for the last commit, read the accumulator with tcgen05.ld
// (warp w: TMEM lanes 32w .. 32w+31 = the tile's rows) and run the epilogue of
// the stage that consumes the projection, so that no separate elementwise
// kernel touches the result.  Every wait is bounded by %globaltimer; on
// expiry the CTA records a timeout in the status word, drains its copies and
// MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lf_gemm.h"
#include "lf_internal.cuh"
#include "lf_ptx.cuh"
#include "lf_tc.cuh"

namespace lfg {

using namespace lftc;

constexpr int NTHR = 192;                        // warps 0-3 epilogue, 4 loader, 5 MMA
constexpr long long kWaitNs = 2000000000LL;      // bound of every wait

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 3 : 4;
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + B_BYTES;
    static constexpr uint32_t SMEM = STAGES * STAGE_BYTES + 1024 /* barriers */ + 1024 /* alignment */;
};

struct Shared {
    uint64_t *full, *empty, *accf;
    uint32_t *tmem_slot;
    volatile int *abort_s;
};

// Bounded wait on one mbarrier phase.  On expiry: record a timeout (where,
// the CTA) once and raise the CTA's abort flag.
__device__ bool wait_phase(uint64_t *bar, unsigned parity, const Shared &sh, unsigned *status, unsigned where)
{
    if (lfk::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = lfk::globaltimer_ns();
    for (unsigned it = 0;; ++it) {
        if (lfk::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*sh.abort_s) return false;
            if ((long long)(lfk::globaltimer_ns() - t0) > kWaitNs) {
                *sh.abort_s = 1;
                if (status && atomicCAS(status, 0u, (unsigned)lfk::STATUS_TIMEOUT) == 0u) {
                    status[1] = where;
                    status[2] = blockIdx.x;
                    status[3] = blockIdx.y;
                }
                if (status) atomicExch(status + 4, 1u);
                return false;
            }
        }
    }
}
// The same without recording anything (teardown: copies or MMAs that must
// have finished before shared memory or TMEM is released).
__device__ void settle_phase(uint64_t *bar, unsigned parity)
{
    const unsigned long long t0 = lfk::globaltimer_ns();
    while (!lfk::mbar_try_wait(bar, parity))
        if ((long long)(lfk::globaltimer_ns() - t0) > kWaitNs) return;
}

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }

__device__ __forceinline__ void split_h(float v, __half &hi, __half &lo)
{
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));
}

// 1 / sqrt(mean of squares + eps) of the RMSNorm input of row `row`, from its
// partial sums of squares.
__device__ __forceinline__ float row_inv(const GemmParams &p, int row)
{
    const float *s = p.ss_in + (size_t)row * p.ss_n;
    float t = 0.f;
    for (int i = 0; i < p.ss_n; ++i) t += s[i];
    return 1.0f / sqrtf(t / (float)p.dnorm + p.eps);
}

// ---------------------------------------------------------------- epilogues
// Warp w owns rows m0 + 32 w .. +31 of the tile.  tcgen05.ld hands thread i
// row i's values of a 32-column chunk; the chunk goes through a padded
// 32 x 33 shared-memory buffer so that the global accesses that follow are
// row by row with lane = column (coalesced).  Per-row values (the RMSNorm
// factor, the position, the routed token) are computed by the row's own
// thread and broadcast with a shuffle.

struct Rows {
    int m0w;     // first row of the warp
    int rows;    // rows that exist
    int lane;
};

__device__ __forceinline__ void stage(float *buf, const uint32_t (&v)[32], int lane)
{
#pragma unroll
    for (int j = 0; j < 32; ++j) buf[lane * 33 + j] = u2f(v[j]);
    __syncwarp();
}

template <int BN>
__device__ void epi_store(const GemmParams &p, uint32_t tb, const Rows &R, int n0, float *buf)
{
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        stage(buf, v, R.lane);
        const int col = n0 + c * 32 + R.lane;
        const float cs = p.colscale ? p.colscale[col] : 1.f;
        for (int r = 0; r < 32 && R.m0w + r < R.rows; ++r) p.Y[(size_t)(R.m0w + r) * p.ldy + col] = buf[r * 33 + R.lane] * cs;
        __syncwarp();
    }
}

// Fused q/k/v rows (a tile covers whole heads: BN is a multiple of hd): the
// RMSNorm factor of the row, then per rotate-half pair (j, j + hd/2) of a q
// or k head the rotation by the position's (cos, sin); q goes to Qr in FP32,
// k and v are rounded to FP16 into the cache rows (group-swizzled, as the
// decode kernels read them).
template <int BN>
__device__ void epi_qkv(const GemmParams &p, uint32_t tb, const Rows &R, int n0, int m0, float *buf, float2 *rt,
                        int tid)
{
    const lfk::Geo &g = p.g;
    const int hd = g.hd, half = hd / 2, hstep = half / 32;
    // the (cos, sin) rows of the tile's positions, copied into shared memory at once
    {
        const int P16 = half / 2;   // 16-byte pieces of one position's half-row of float2
        for (int i = tid; i < 128 * P16; i += 128) {
            const int rr = i / P16, q = i % P16;
            const bool ok = m0 + rr < R.rows;
            cp_async16(smem_u32(rt + rr * half + q * 2), p.rope + (size_t)(p.pos0 + (ok ? m0 + rr : m0)) * half + q * 2,
                       ok ? 16u : 0u);
        }
        cp_async_wait_all();
        asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    const int wr = R.m0w - m0;
    const int myrow = R.m0w + R.lane;
    const float myinv = myrow < R.rows ? row_inv(p, myrow) : 0.f;
    float *bufb = buf + 32 * 33;
#pragma unroll 1
    for (int c0 = 0; c0 < BN / 32; ++c0) {
        if ((c0 / hstep) & 1) continue;
        const int c1 = c0 + hstep;
        {
            uint32_t a[32], b[32];
            tmem_ld32(tb + (uint32_t)(c0 * 32), a);
            tmem_ld32(tb + (uint32_t)(c1 * 32), b);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                buf[R.lane * 33 + j] = u2f(a[j]);
                bufb[R.lane * 33 + j] = u2f(b[j]);
            }
            __syncwarp();
        }
        const int col0 = n0 + c0 * 32;
        const int hh = col0 / hd, j = col0 % hd + R.lane;   // this lane's pair (j, j + half)
        float s0 = 1.f, s1 = 1.f;
        if (p.colscale) {
            s0 = p.colscale[col0 + R.lane];
            s1 = p.colscale[col0 + half + R.lane];
        }
        for (int r = 0; r < 32; ++r) {
            const float inv = __shfl_sync(0xffffffffu, myinv, r);
            const int row = R.m0w + r;
            if (row >= R.rows) break;
            const int pos = p.pos0 + row;
            const float v0 = buf[r * 33 + R.lane] * s0 * inv, v1 = bufb[r * 33 + R.lane] * s1 * inv;
            if (hh < g.Hq + g.Hkv) {
                const float2 t = rt[(wr + r) * half + j];
                const float r0 = v0 * t.x - v1 * t.y, r1 = v1 * t.x + v0 * t.y;
                if (hh < g.Hq) {
                    float *q = p.Qr + (size_t)row * g.Q + (size_t)hh * hd;
                    q[j] = r0;
                    q[j + half] = r1;
                } else {
                    __half *kr = p.kc + (((size_t)p.layer * g.Hkv + (hh - g.Hq)) * g.max_seq + pos) * hd;
                    kr[lfk::kv_swz(pos, j)] = __float2half_rn(r0);
                    kr[lfk::kv_swz(pos, j + half)] = __float2half_rn(r1);
                }
            } else {
                __half *vr = p.vc + (((size_t)p.layer * g.Hkv + (hh - g.Hq - g.Hkv)) * g.max_seq + pos) * hd;
                vr[lfk::kv_swz(pos, j)] = __float2half_rn(v0);
                vr[lfk::kv_swz(pos, j + half)] = __float2half_rn(v1);
            }
        }
        __syncwarp();
    }
}

// Residual add into X (FP32, [rows, N]); then the next RMSNorm's input: X x
// gain_next split into Xh / Xl, and the row's sum of squares over each group
// of 128 columns into ss_out[row][group].  The tile of X is first copied into
// shared memory with 16-byte async copies (all in flight at once), so the
// row-by-row pass below issues only stores.
template <int BN>
__device__ void epi_resid(const GemmParams &p, uint32_t tb, const Rows &R, int n0, int m0, float *buf, float *xt,
                          int tid)
{
    constexpr int P16 = BN / 4;
    for (int i = tid; i < 128 * P16; i += 128) {
        const int rr = i / P16, q = i % P16;
        const int row = m0 + rr;
        const bool ok = row < R.rows;
        cp_async16(smem_u32(xt + rr * BN + q * 4), p.X + (size_t)(ok ? row : m0) * p.N + n0 + q * 4, ok ? 16u : 0u);
    }
    cp_async_wait_all();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int wr = R.m0w - m0;   // the warp's first row within the tile
    float ss = 0.f;              // this thread's row, the current 128-column group
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        stage(buf, v, R.lane);
        const int cl = c * 32 + R.lane, col = n0 + cl;
        const float cs = p.colscale ? p.colscale[col] : 1.f;
        const float gn = p.gain_next ? __half2float(p.gain_next[col]) : 0.f;
        for (int r = 0; r < 32; ++r) {
            const int row = R.m0w + r;
            if (row >= R.rows) break;
            const size_t o = (size_t)row * p.N + col;
            const float x = xt[(wr + r) * BN + cl] + buf[r * 33 + R.lane] * cs;
            p.X[o] = x;
            if (p.gain_next) {
                __half hi, lo;
                split_h(x * gn, hi, lo);
                p.Xh[o] = hi;
                p.Xl[o] = lo;
            }
            buf[r * 33 + R.lane] = x;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float x = buf[R.lane * 33 + j];
            ss = fmaf(x, x, ss);
        }
        __syncwarp();
        if ((c & 3) == 3) {   // one partial sum of squares per 128 columns
            const int myrow = R.m0w + R.lane;
            if (myrow < R.rows && p.gain_next) p.ss_out[(size_t)myrow * (p.N / 128) + (n0 + c * 32) / 128] = ss;
            ss = 0.f;
        }
    }
}

// Gate/up tile (BN = 256: columns 0..127 are the gate rows of units
// u0 .. u0+127, columns 128..255 their up rows): h = SiLU(g inv) (u inv),
// split into Hh / Hl.  Grouped (mixture of experts): the row is one routed
// (token, slot), h is also scaled by its gate, and the RMSNorm factor is the
// token's.
template <bool MOE>
__device__ void epi_gu(const GemmParams &p, uint32_t tb, const Rows &R, int e, float *buf)
{
    const int myrow = R.m0w + R.lane;
    int mytok = myrow;
    float mygw = 1.f;
    if (MOE && myrow < R.rows) {
        const int tj = p.list[(size_t)e * p.a_group_rows + myrow];
        mytok = tj >> 3;
        mygw = p.gatev[tj];
    }
    const float myinv = myrow < R.rows ? row_inv(p, mytok) : 0.f;
    const int u0 = blockIdx.x * 128;
    float *bufb = buf + 32 * 33;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        {
            uint32_t gv[32], uv[32];
            tmem_ld32(tb + (uint32_t)(c * 32), gv);
            tmem_ld32(tb + (uint32_t)(128 + c * 32), uv);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                buf[R.lane * 33 + j] = u2f(gv[j]);
                bufb[R.lane * 33 + j] = u2f(uv[j]);
            }
            __syncwarp();
        }
        const int unit = u0 + c * 32 + R.lane;
        float sg = 1.f, su = 1.f;
        if (p.colscale) {
            sg = p.colscale[2 * u0 + c * 32 + R.lane];
            su = p.colscale[2 * u0 + 128 + c * 32 + R.lane];
        }
        for (int r = 0; r < 32; ++r) {
            const float inv = __shfl_sync(0xffffffffu, myinv, r);
            const float gw = __shfl_sync(0xffffffffu, mygw, r);
            const int row = R.m0w + r;
            if (row >= R.rows) break;
            const float gt = buf[r * 33 + R.lane] * sg * inv, up = bufb[r * 33 + R.lane] * su * inv;
            float hv = gt / (1.0f + expf(-gt)) * up;
            if (MOE) hv *= gw;
            const size_t hrow = MOE ? (size_t)e * p.a_group_rows + row : (size_t)row;
            __half hi, lo;
            split_h(hv, hi, lo);
            p.Hh[hrow * p.ldh + unit] = hi;
            p.Hl[hrow * p.ldh + unit] = lo;
        }
        __syncwarp();
    }
}

// Down-projection rows of one expert, scattered to their (token, slot) places.
template <int BN>
__device__ void epi_d_moe(const GemmParams &p, uint32_t tb, const Rows &R, int e, int n0, float *buf)
{
    const int myrow = R.m0w + R.lane;
    const int mytj = myrow < R.rows ? p.list[(size_t)e * p.a_group_rows + myrow] : 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        stage(buf, v, R.lane);
        for (int r = 0; r < 32; ++r) {
            const int tj = __shfl_sync(0xffffffffu, mytj, r);
            if (R.m0w + r >= R.rows) break;
            float *dst = p.Yk + ((size_t)(tj >> 3) * p.topk + (tj & 7)) * p.N + n0 + c * 32;
            dst[R.lane] = buf[r * 33 + R.lane];
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------- split-K

// AND of a predicate over the four epilogue warps (named barrier 1, 128 threads).
__device__ __forceinline__ bool epi_all(bool pred)
{
    unsigned r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((unsigned)pred)
        : "memory");
    return r != 0;
}

// Called by the four epilogue warps of every split CTA of a tile: each writes
// its partial tile (thread = row, 32-column chunks, 128 contiguous bytes each)
// to part[tile * S + split], then counts itself in the tile's counter.  The
// CTA that arrives last sums the S partials in split order -- the same sum
// whichever CTA it is -- and stores the sum back into its TMEM accumulator
// for the epilogue (returns true); the others return false.
template <int BN>
__device__ bool reduce_splits(const GemmParams &p, uint32_t tb, int warp, int lane, int split, int S, const Shared &sh)
{
    constexpr int NC = BN / 32;
    const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
    const size_t row = (size_t)(warp * 32 + lane);
    // partial s, chunk c: [32 columns][128 rows], so that a warp's 32 rows of
    // one column are 128 contiguous bytes
    auto chunk = [&](int s, int c) { return p.part + ((tile * S + s) * NC + c) * (32 * 128) + row; };
#pragma unroll 1
    for (int c = 0; c < NC; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        float *dst = chunk(split, c);
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[j * 128] = u2f(v[j]);
    }
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
    if (warp == 0 && lane == 0) {
        const unsigned old = atomicAdd(p.tile_cnt + tile, 1u);
        const bool last = old == (unsigned)S - 1u;
        if (last) p.tile_cnt[tile] = 0u;             // ready for the next product
        sh.abort_s[1] = last ? 1 : 0;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (!sh.abort_s[1]) return false;
    __threadfence();
#pragma unroll 1
    for (int c = 0; c < NC; ++c) {
        float acc[32];
        {
            const float *src = chunk(0, c);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = __ldcg(src + j * 128);
        }
        for (int s = 1; s < S; ++s) {
            const float *src = chunk(s, c);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] += __ldcg(src + j * 128);
        }
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(acc[j]);
        tmem_st32(tb + (uint32_t)(c * 32), v);
    }
    tmem_st_wait();
    fence_before_sync();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    fence_after_sync();
    return true;
}

// ---------------------------------------------------------------- the kernel

template <int BN, int EPI>
__global__ void __launch_bounds__(NTHR, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_ah, const __grid_constant__ CUtensorMap tm_al,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ GemmParams p)
{
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
    Shared sh;
    sh.full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    sh.empty = sh.full + C::STAGES;
    sh.accf = sh.empty + C::STAGES;
    sh.tmem_slot = reinterpret_cast<uint32_t *>(sh.accf + 1);
    sh.abort_s = reinterpret_cast<volatile int *>(sh.tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.splits > 1 ? p.splits : 1;
    const int e = blockIdx.z / S, split = blockIdx.z % S;
    const int rows = p.cnt ? p.cnt[e] : p.M;
    const int m0 = blockIdx.y * BM;
    if (m0 >= rows) return;                          // the whole CTA: nothing to compute
    const int n0 = blockIdx.x * BN;
    const int a_y = p.a_row0 + e * p.a_group_rows + m0;
    const int b_y = p.b_row0 + e * p.N + n0;
    const int nk_all = p.K / BK;
    const int kb = (int)((long long)split * nk_all / S), ke = (int)((long long)(split + 1) * nk_all / S);
    const int nk = ke - kb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            lfk::mbar_init(&sh.full[s], 1);
            lfk::mbar_init(&sh.empty[s], 1);
        }
        lfk::mbar_init(sh.accf, 1);
        sh.abort_s[0] = 0;
        sh.abort_s[1] = 0;
        lfk::mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(sh.tmem_slot, BN);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *sh.tmem_slot;
    const size_t cta = ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    if (p.stamps && threadIdx.x == 0) p.stamps[cta * 4] = lfk::globaltimer_ns();
    // launched as a programmatic dependent of the previous kernel: everything
    // above overlapped its tail; nothing below touches global memory before
    // that kernel has finished and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tm_ah);
            prefetch_tmap(&tm_al);
            prefetch_tmap(&tm_b);
            int issued = 0;
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % C::STAGES;
                const unsigned ph = (unsigned)(kt / C::STAGES) & 1u;
                if (!wait_phase(&sh.empty[s], ph ^ 1u, sh, p.status, 500)) break;
                lfk::mbar_arrive_expect_tx(&sh.full[s], C::STAGE_BYTES);
                uint8_t *st = smem + (size_t)s * C::STAGE_BYTES;
                const int kx = (kb + kt) * BK;
                tma_load_2d(st, &tm_ah, kx, a_y, &sh.full[s]);
                tma_load_2d(st + C::A_BYTES, &tm_al, kx, a_y, &sh.full[s]);
                tma_load_2d(st + 2 * C::A_BYTES, &tm_b, kx, b_y, &sh.full[s]);
                issued = kt + 1;
            }
            // every copy this thread issued has landed before the CTA can exit
            for (int kt = issued > C::STAGES ? issued - C::STAGES : 0; kt < issued; ++kt)
                settle_phase(&sh.full[kt % C::STAGES], (unsigned)(kt / C::STAGES) & 1u);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);
            for (int kt = 0; kt < nk; ++kt) {
                const int s = kt % C::STAGES;
                const unsigned ph = (unsigned)(kt / C::STAGES) & 1u;
                if (!wait_phase(&sh.full[s], ph, sh, p.status, 501)) break;
                if (kt == 0 && p.stamps) p.stamps[cta * 4 + 1] = lfk::globaltimer_ns();
                fence_after_sync();
                const uint32_t base = smem_u32(smem + (size_t)s * C::STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t bd = sdesc_kmajor_sw128(base + 2 * C::A_BYTES + (uint32_t)kk * 32u);
                    mma_f16(tmem, sdesc_kmajor_sw128(base + (uint32_t)kk * 32u), bd, IDESC, (kt | kk) != 0);
                    mma_f16(tmem, sdesc_kmajor_sw128(base + C::A_BYTES + (uint32_t)kk * 32u), bd, IDESC, 1u);
                }
                commit(&sh.empty[s]);                // the stage is free once these MMAs are done
            }
            commit(sh.accf);                         // every issued MMA done: the accumulator is final
        }
    } else {
        const bool ok = wait_phase(sh.accf, 0u, sh, p.status, 502);
        fence_after_sync();
        if (p.stamps && threadIdx.x == 0) p.stamps[cta * 4 + 2] = lfk::globaltimer_ns();
        const uint32_t tb = tmem + ((uint32_t)(warp * 32) << 16);
        // one decision for the four epilogue warps (they meet at named barriers below)
        bool run = epi_all(ok && !*sh.abort_s);
        if (run && S > 1) run = reduce_splits<BN>(p, tb, warp, lane, split, S, sh);
        if (run) {
            // the stage buffers are free once every MMA is done: two 32 x 33 staging buffers per warp
            float *buf = reinterpret_cast<float *>(smem) + warp * (2 * 32 * 33);
            // after the staging buffers (4 x 8.25 KB): the tile's inputs of the epilogue
            float *ein = reinterpret_cast<float *>(smem + 36 * 1024);
            const Rows R{m0 + warp * 32, rows, lane};
            const int tid = threadIdx.x;   // 0..127 in warps 0-3
            if constexpr (EPI == EPI_STORE) epi_store<BN>(p, tb, R, n0, buf);
            else if constexpr (EPI == EPI_QKV) epi_qkv<BN>(p, tb, R, n0, m0, buf, reinterpret_cast<float2 *>(ein), tid);
            else if constexpr (EPI == EPI_RESID) epi_resid<BN>(p, tb, R, n0, m0, buf, ein, tid);
            else if constexpr (EPI == EPI_GU) epi_gu<false>(p, tb, R, e, buf);
            else if constexpr (EPI == EPI_GU_MOE) epi_gu<true>(p, tb, R, e, buf);
            else epi_d_moe<BN>(p, tb, R, e, n0, buf);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (p.stamps && threadIdx.x == 0) p.stamps[cta * 4 + 3] = lfk::globaltimer_ns();
    if (warp == 5) {
        if (lane == 0) settle_phase(sh.accf, 0u);    // no MMA still writes TMEM
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, BN);
    }
}

template <int BN, int EPI>
cudaError_t launch_one(const CUtensorMap *a_hi, const CUtensorMap *a_lo, const CUtensorMap *b, const GemmParams *p,
                       int groups, int pdl, cudaStream_t stream)
{
    using C = Cfg<BN>;
    static bool attr_set[64] = {};  // the shared-memory limit is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const int S = p->splits > 1 ? p->splits : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p->N / BN), (unsigned)((p->M + BM - 1) / BM), (unsigned)(groups * S));
    cfg.blockDim = dim3(NTHR);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<BN, EPI>, *a_hi, *a_lo, *b, *p);
}

}  // namespace lfg

extern "C" cudaError_t lfg_launch(int epi, int bn, const CUtensorMap *a_hi, const CUtensorMap *a_lo,
                                  const CUtensorMap *b, const lfg::GemmParams *p, int groups, int pdl,
                                  cudaStream_t stream)
{
    using namespace lfg;
    if (p->N % bn || p->K % BK || p->M < 1 || groups < 1) return cudaErrorInvalidValue;
    if (p->splits > 1 && (groups != 1 || !p->part || !p->tile_cnt || p->splits > p->K / BK)) return cudaErrorInvalidValue;
    if (bn == 128) {
        switch (epi) {
        case EPI_STORE: return launch_one<128, EPI_STORE>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_QKV: return launch_one<128, EPI_QKV>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_RESID: return launch_one<128, EPI_RESID>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_D_MOE: return launch_one<128, EPI_D_MOE>(a_hi, a_lo, b, p, groups, pdl, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    if (bn == 256) {
        switch (epi) {
        case EPI_STORE: return launch_one<256, EPI_STORE>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_QKV: return launch_one<256, EPI_QKV>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_RESID: return launch_one<256, EPI_RESID>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_D_MOE: return launch_one<256, EPI_D_MOE>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_GU: return launch_one<256, EPI_GU>(a_hi, a_lo, b, p, groups, pdl, stream);
        case EPI_GU_MOE: return launch_one<256, EPI_GU_MOE>(a_hi, a_lo, b, p, groups, pdl, stream);
        default: return cudaErrorInvalidValue;
        }
    }
    return cudaErrorInvalidValue;
}

extern "C" void lfg_plan(int M, int N, int K, int sms, int allow_bn128, int *bn, int *splits)
{
    // Time model of one product, in microseconds, fitted to GB300 runs of this
    // kernel: per wave of CTAs (one CTA per SM) a fixed cost F (pipeline fill,
    // epilogue, launch) plus the K steps of one CTA at k_w per step (128-wide
    // tiles reach a lower fraction of the tensor peak than 256-wide ones), plus
    // the partial-tile reduction when K is split.
    const int mt = (M + lfg::BM - 1) / lfg::BM, nk = K / lfg::BK;
    const double F = 5.0, k128 = 0.42, k256 = 0.62;
    double best = 1e300;
    *bn = N % 256 == 0 ? 256 : 128;
    *splits = 1;
    for (int w = 128; w <= 256; w += 128) {
        if (N % w || (w == 128 && !allow_bn128)) continue;
        const int tiles = (N / w) * mt;
        for (int s = 1; s <= 4; ++s) {
            if (s > 1 && (nk / s < 8 || tiles * s > sms)) break;   // split CTAs fit one wave (and the partial buffer)
            const int waves = (tiles * s + sms - 1) / sms;
            const double t = waves * (F + ((nk + s - 1) / s) * (w == 128 ? k128 : k256)) + (s > 1 ? 3.0 + 2.0 * s : 0.0);
            if (t < best) {
                best = t;
                *bn = w;
                *splits = s;
            }
        }
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the library
// links the CUDA runtime statically and not libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

extern "C" int lfg_tensor_map(CUtensorMap *out, const void *base, unsigned long long rows, unsigned long long cols,
                              int box_rows)
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return 1;
        fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    if ((reinterpret_cast<uintptr_t>(base) & 15u) || (cols * 2) % 16 || box_rows < 1 || box_rows > 256) return 2;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)lfg::BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 3;
}

// Test hook: Y [M, N] (FP32, row-major) = (Xh + Xl) [M, K] . W [N, K]^T through
// the tensor-core GEMM with the plain-store epilogue; all pointers device,
// row-major FP16 inputs; splits > 1 cuts K into that many ranges (part: at
// least tiles x splits x 128 x bn floats, tile_cnt: tiles zeroed counters).
// Synchronous.  0 on success.
extern "C" __attribute__((visibility("default"))) int lfg_gemm_test(const void *xh, const void *xl, const void *w,
                                                                    int M, int N, int K, int bn, int splits,
                                                                    float *part, unsigned *tile_cnt, float *Y)
{
    CUtensorMap ta, tl, tb;
    if (lfg_tensor_map(&ta, xh, (unsigned long long)M, (unsigned long long)K, lfg::BM) ||
        lfg_tensor_map(&tl, xl, (unsigned long long)M, (unsigned long long)K, lfg::BM) ||
        lfg_tensor_map(&tb, w, (unsigned long long)N, (unsigned long long)K, bn))
        return 1;
    lfg::GemmParams p = {};
    p.M = M;
    p.N = N;
    p.K = K;
    p.Y = Y;
    p.ldy = N;
    p.splits = splits;
    p.part = part;
    p.tile_cnt = tile_cnt;
    const cudaError_t e = lfg_launch(lfg::EPI_STORE, bn, &ta, &tl, &tb, &p, 1, 0, nullptr);
    if (e != cudaSuccess) return 2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

// Benchmark hook: the same product as lfg_gemm_test, launched `reps` times
// back to back on the legacy stream between two CUDA events; *us_out = mean
// microseconds per launch.  0 on success.
extern "C" __attribute__((visibility("default"))) int lfg_gemm_bench(const void *xh, const void *xl, const void *w,
                                                                     int M, int N, int K, int bn, int splits,
                                                                     float *part, unsigned *tile_cnt, float *Y,
                                                                     int reps, float *us_out,
                                                                     unsigned long long *stamps)
{
    CUtensorMap ta, tl, tb;
    if (lfg_tensor_map(&ta, xh, (unsigned long long)M, (unsigned long long)K, lfg::BM) ||
        lfg_tensor_map(&tl, xl, (unsigned long long)M, (unsigned long long)K, lfg::BM) ||
        lfg_tensor_map(&tb, w, (unsigned long long)N, (unsigned long long)K, bn))
        return 1;
    lfg::GemmParams p = {};
    p.M = M;
    p.N = N;
    p.K = K;
    p.Y = Y;
    p.ldy = N;
    p.splits = splits;
    p.part = part;
    p.tile_cnt = tile_cnt;
    cudaEvent_t e0, e1;
    if (stamps) {   // one extra launch that records the per-CTA stamps
        p.stamps = stamps;
        if (lfg_launch(lfg::EPI_STORE, bn, &ta, &tl, &tb, &p, 1, 0, nullptr) != cudaSuccess) return 2;
        p.stamps = nullptr;
    }
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    if (lfg_launch(lfg::EPI_STORE, bn, &ta, &tl, &tb, &p, 1, 0, nullptr) != cudaSuccess) return 2;
    cudaEventRecord(e0, nullptr);
    for (int i = 0; i < reps; ++i) lfg_launch(lfg::EPI_STORE, bn, &ta, &tl, &tb, &p, 1, 0, nullptr);
    cudaEventRecord(e1, nullptr);
    const cudaError_t e = cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *us_out = ms * 1000.f / (float)reps;
    return e == cudaSuccess ? 0 : 3;
}
