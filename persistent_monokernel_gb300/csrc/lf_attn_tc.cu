// lf_attn_tc.cu -- the batched prefill's causal attention on the sm_103a
// tensor cores (head_dim 128).
//
// One CTA takes 128 query rows of one query head and walks the cached
// positions they attend to in chunks of 64 (flash-attention order):
//
//   S   = Q K^T            tcgen05.mma, Q as FP16 head + remainder (two MMAs),
//                          K straight from the cache rows, FP32 in TMEM
//   P   = exp2(S - m)      two threads per query row (TMEM lane = row): mask,
//                          running maximum and sum, P split into FP16 head and
//                          remainder written to shared memory
//   O  += P V              tcgen05.mma with V as an MN-major operand (the cache
//                          rows need no transpose), FP32 in TMEM
//
// Warp 8 streams K and V of each chunk with 2-D TMA loads into a ring of three
// stages; warp 9 owns TMEM and issues the MMAs from one thread, ordering them
// S(c+2) after PV(c) so that the softmax of chunk c+1 overlaps the MMAs;
// warps 0-7 run the softmax and the output, two threads per query row (warps
// w and w + 4 share TMEM lanes 32 (w mod 4) ..; each takes half of a chunk's
// positions and half of the output's dimensions).  The running maximum is a lazy
// reference: O and the sum are rescaled only when a row's maximum rises more
// than 8 (log2 units) above it, which leaves the quotient O / l exact in
// exact arithmetic and keeps every exponent bounded.
//
// The cache rows are group-swizzled (16-byte group g of position p at g XOR
// (p mod 8)), so a chunk of 64 rows starting at a multiple of 64 lands in
// shared memory already in the 128-byte-swizzle layout the MMA descriptors
// describe: K as a K-major operand, V as an MN-major one.  Positions past the
// last one a chunk's rows attend to are masked to probability 0; the cache is
// zero-filled at creation so that their values are finite.
//
// Every wait is bounded by %globaltimer; on expiry the CTA records a timeout
// in the status word, settles its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lf_internal.cuh"
#include "lf_ptx.cuh"
#include "lf_tc.cuh"

namespace lfa {

using namespace lftc;

constexpr int HD = 128;
constexpr int BM = 128;                  // query rows per CTA
constexpr int BN = 64;                   // cached positions per chunk
constexpr int STAGES = 3;
constexpr int NTHR = 320;                // warps 0-7 softmax / output, 8 loads, 9 MMA
constexpr int W_LOAD = 8, W_MMA = 9, NSM = 256;   // softmax threads: two per query row
constexpr long long kWaitNs = 2000000000LL;

// shared memory (offsets from a 1,024-byte aligned base)
constexpr uint32_t Q_ATOM = BM * 128;                 // 128 rows x 64 dims (FP16)
constexpr uint32_t Q_BYTES = 2 * Q_ATOM;              // head dims 0-63, 64-127
constexpr uint32_t KV_ATOM = BN * 128;                // 64 positions x 64 dims
constexpr uint32_t STAGE_BYTES = 4 * KV_ATOM;         // K halves, then V halves
constexpr uint32_t P_BYTES = BM * 128;                // 128 rows x 64 positions (FP16)
constexpr uint32_t OFF_QH = 0, OFF_QL = Q_BYTES, OFF_KV = 2 * Q_BYTES;
constexpr uint32_t OFF_P = OFF_KV + STAGES * STAGE_BYTES;   // [2 buffers][head, remainder]
constexpr uint32_t OFF_BAR = OFF_P + 4 * P_BYTES;   // 224 KB
constexpr uint32_t SMEM = 232448;   // the opt-in maximum: the data, the barriers and the base's alignment slack

// TMEM columns: S buffers 0 and 1, then O
constexpr uint32_t T_S0 = 0, T_S1 = BN, T_O = 2 * BN, T_COLS = 256;

struct Bars {
    uint64_t kv_full[STAGES], kv_empty[STAGES];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
    uint64_t q_ready, o_done;
    uint32_t tmem;
    int abort;
    float xmax[2][2][BM];   // [chunk parity][key half][row]: the halves' maxima; then the halves' sums
};

__device__ bool wait_phase(uint64_t *bar, unsigned parity, Bars *b, unsigned *status, unsigned where)
{
    if (lfk::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = lfk::globaltimer_ns();
    for (unsigned it = 0;; ++it) {
        if (lfk::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*reinterpret_cast<volatile int *>(&b->abort)) return false;
            if ((long long)(lfk::globaltimer_ns() - t0) > kWaitNs) {
                *reinterpret_cast<volatile int *>(&b->abort) = 1;
                if (atomicCAS(status, 0u, (unsigned)lfk::STATUS_TIMEOUT) == 0u) {
                    status[1] = where;
                    status[2] = blockIdx.x;
                    status[3] = blockIdx.y;
                }
                atomicExch(status + 4, 1u);
                return false;
            }
        }
    }
}
__device__ void settle_phase(uint64_t *bar, unsigned parity)
{
    const unsigned long long t0 = lfk::globaltimer_ns();
    while (!lfk::mbar_try_wait(bar, parity))
        if ((long long)(lfk::globaltimer_ns() - t0) > kWaitNs) return;
}

// AND of a predicate over the softmax warps 0-7 (named barrier 1, 256 threads).
__device__ __forceinline__ bool rows_all(bool pred)
{
    unsigned r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((unsigned)pred)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void rows_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// 2^x on the special-function unit (about 2 ulp; exact 0 for -inf).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// MN-major 128-byte-swizzle descriptor (8-row groups along K 1,024 bytes
// apart; one 64-element atom along MN): start, LBO (unused with one atom),
// SBO 1,024, version 1, SWIZZLE_128B.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(KV_ATOM >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// kind::f16, FP16 A and B, FP32 D; B MN-major when b_mn.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn)
{
    return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t sw128(int row, int chunk16) { return (uint32_t)(row * 128 + ((chunk16 ^ (row & 7)) << 4)); }

__global__ void __launch_bounds__(NTHR, 1)
    attn_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const float *Qr,
            int T, int pos0, int l, lfk::Geo g, const int *win, __half *Ah, __half *Al, unsigned *status,
            unsigned long long *stamps)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~uintptr_t(1023));
    Bars *b = reinterpret_cast<Bars *>(smem + OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the aligned layout must fit the allocation (the base's alignment slack is small)
    if ((uint32_t)(smem - smem_raw) + OFF_BAR + (uint32_t)sizeof(Bars) > SMEM) {
        if (threadIdx.x == 0 && atomicCAS(status, 0u, (unsigned)lfk::STATUS_TIMEOUT) == 0u) status[1] = 609;
        return;
    }
    const int blk = gridDim.x - 1 - blockIdx.x;      // the longest rows first
    const int h = blockIdx.y, gkv = h / g.group;
    const int t0 = blk * BM, nrow = min(BM, T - t0);
    const int W = win ? win[l] : 0;
    const int pos_hi = pos0 + t0 + nrow - 1;
    const int c_begin = lfk::attn_first_pos(pos0 + t0, W) / BN, c_end = pos_hi / BN;
    const int nc = c_end - c_begin + 1;
    const int kv_row0 = (l * g.Hkv + gkv) * g.max_seq;   // first cache row of this KV head

    asm volatile("griddepcontrol.wait;" ::: "memory");   // launched as a programmatic dependent
    // optional %globaltimer stamps per CTA (profiling aid): entry, q staged,
    // first scores in hand, last P handed over, output done, chunk count
    unsigned long long *stp = stamps ? stamps + ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * 8 : nullptr;
    if (stp && threadIdx.x == 0) {
        stp[0] = lfk::globaltimer_ns();
        stp[5] = (unsigned long long)nc;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            lfk::mbar_init(&b->kv_full[s], 1);
            lfk::mbar_init(&b->kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            lfk::mbar_init(&b->s_full[i], 1);
            lfk::mbar_init(&b->s_free[i], NSM);
            lfk::mbar_init(&b->p_full[i], NSM);
            lfk::mbar_init(&b->pv_done[i], 1);
        }
        lfk::mbar_init(&b->q_ready, NSM);
        lfk::mbar_init(&b->o_done, 1);
        b->abort = 0;
        lfk::mbar_fence_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(&b->tmem, T_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = b->tmem;

    if (warp == W_LOAD) {
        // ---- K and V of every chunk, in order, into the stage ring
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int i = 0; i < nc; ++i) {
                const int s = i % STAGES;
                if (!wait_phase(&b->kv_empty[s], ((unsigned)(i / STAGES) & 1u) ^ 1u, b, status, 600)) break;
                lfk::mbar_arrive_expect_tx(&b->kv_full[s], STAGE_BYTES);
                uint8_t *st = smem + OFF_KV + (size_t)s * STAGE_BYTES;
                const int y = kv_row0 + (c_begin + i) * BN;
                tma_load_2d(st, &tm_k, 0, y, &b->kv_full[s]);
                tma_load_2d(st + KV_ATOM, &tm_k, 64, y, &b->kv_full[s]);
                tma_load_2d(st + 2 * KV_ATOM, &tm_v, 0, y, &b->kv_full[s]);
                tma_load_2d(st + 3 * KV_ATOM, &tm_v, 64, y, &b->kv_full[s]);
                issued = i + 1;
            }
            for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                settle_phase(&b->kv_full[i % STAGES], (unsigned)(i / STAGES) & 1u);
        }
    } else if (warp == W_MMA) {
        // ---- MMAs: S(0), S(1), then per chunk PV(c) and S(c+2)
        if (lane == 0) {
            const uint32_t sb = smem_u32(smem);
            auto issue_s = [&](int i) -> bool {
                const int s = i % STAGES;
                if (!wait_phase(&b->kv_full[s], (unsigned)(i / STAGES) & 1u, b, status, 601)) return false;
                if (i >= 2 && !wait_phase(&b->s_free[i & 1], (unsigned)((i - 2) / 2) & 1u, b, status, 602)) return false;
                fence_after_sync();
                const uint32_t kb = sb + OFF_KV + (uint32_t)s * STAGE_BYTES;
                const uint32_t d = tmem + ((i & 1) ? T_S1 : T_S0);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk / 4) * Q_ATOM + (uint32_t)(kk % 4) * 32u;
                    const uint64_t bd = sdesc_kmajor_sw128(kb + (uint32_t)(kk / 4) * KV_ATOM + (uint32_t)(kk % 4) * 32u);
                    mma_f16(d, sdesc_kmajor_sw128(sb + OFF_QH + off), bd, idesc(BM, BN, false), kk != 0);
                    mma_f16(d, sdesc_kmajor_sw128(sb + OFF_QL + off), bd, idesc(BM, BN, false), 1u);
                }
                commit(&b->s_full[i & 1]);
                return true;
            };
            bool ok = wait_phase(&b->q_ready, 0u, b, status, 603);
            if (ok) ok = issue_s(0);
            if (ok && nc > 1) ok = issue_s(1);
            for (int i = 0; ok && i < nc; ++i) {
                if (!wait_phase(&b->p_full[i & 1], (unsigned)(i / 2) & 1u, b, status, 604)) break;
                fence_after_sync();
                const int s = i % STAGES;
                const uint32_t vb = sb + OFF_KV + (uint32_t)s * STAGE_BYTES + 2 * KV_ATOM;
                const uint32_t pb = sb + OFF_P + (uint32_t)(i & 1) * 2 * P_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t ph = sdesc_kmajor_sw128(pb + (uint32_t)kk * 32u);
                    const uint64_t pl = sdesc_kmajor_sw128(pb + P_BYTES + (uint32_t)kk * 32u);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // 16 positions = two 8-row groups of the V half (1,024 bytes each)
                        const uint64_t vd = sdesc_mnmajor_sw128(vb + (uint32_t)half * KV_ATOM + (uint32_t)kk * 2048u);
                        const uint32_t d = tmem + T_O + (uint32_t)half * 64u;
                        mma_f16(d, ph, vd, idesc(BM, 64, true), (i | kk) != 0);
                        mma_f16(d, pl, vd, idesc(BM, 64, true), 1u);
                    }
                }
                commit(&b->pv_done[i & 1]);
                commit(&b->kv_empty[s]);
                if (i + 2 < nc) ok = issue_s(i + 2);
            }
            commit(&b->o_done);
        }
    } else {
        // ---- softmax and output: two threads per query row; thread (r, hf)
        // takes positions 32 hf .. 32 hf + 31 of every chunk and head
        // dimensions 64 hf .. 64 hf + 63 of the output
        const int r = threadIdx.x & 127, hf = threadIdx.x >> 7;   // TMEM lane r (warp % 4 = r / 32)
        const bool live = r < nrow;
        const int pos = pos0 + t0 + (live ? r : nrow - 1);
        const int first = lfk::attn_first_pos(pos, W);
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        // q tile -> FP16 head / remainder in the 128-byte-swizzle K-major layout
        // (coalesced: consecutive threads take consecutive 8-element groups of a row)
        {
            const int tid = threadIdx.x;
#pragma unroll 4
            for (int it = 0; it < BM * (HD / 8) / NSM; ++it) {
                const int idx = it * NSM + tid, row = idx / (HD / 8), c16 = idx % (HD / 8);
                const float *q = Qr + (size_t)(t0 + min(row, nrow - 1)) * g.Q + (size_t)h * HD + c16 * 8;
                const float4 a = *reinterpret_cast<const float4 *>(q);
                const float4 c = *reinterpret_cast<const float4 *>(q + 4);
                const float v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
                unsigned hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __half h0, r0, h1, r1;
                    lfk::split_h(v[2 * j], h0, r0);
                    lfk::split_h(v[2 * j + 1], h1, r1);
                    hw[j] = lfk::pack_h2(h0, h1);
                    lw[j] = lfk::pack_h2(r0, r1);
                }
                const uint32_t o = (uint32_t)(c16 / 8) * Q_ATOM + sw128(row, c16 % 8);
                *reinterpret_cast<uint4 *>(smem + OFF_QH + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(smem + OFF_QL + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
        fence_async_smem();
        lfk::mbar_arrive(&b->q_ready);
        if (stp && threadIdx.x == 0) stp[1] = lfk::globaltimer_ns();
        const float sl2 = 1.4426950408889634f / sqrtf((float)HD);   // scale x log2(e)
        float mref = -INFINITY, lsum = 0.f;
        bool run = true;
        for (int i = 0; i < nc && run; ++i) {
            run = wait_phase(&b->s_full[i & 1], (unsigned)(i / 2) & 1u, b, status, 605);
            run = rows_all(run);
            if (!run) break;
            if (stp && threadIdx.x == 0 && i == 0) stp[2] = lfk::globaltimer_ns();
            fence_after_sync();
            float sv[32];
            {
                uint32_t u[32];
                tmem_ld32(tl + ((i & 1) ? T_S1 : T_S0) + (uint32_t)(32 * hf), u);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(u[j]);
            }
            fence_before_sync();
            lfk::mbar_arrive(&b->s_free[i & 1]);
            const int kb = (c_begin + i) * BN + 32 * hf;
            float mh = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = kb + j;
                const bool ok = live && key <= pos && key >= first;
                sv[j] = ok ? sv[j] * sl2 : -INFINITY;
                mh = fmaxf(mh, sv[j]);
            }
            b->xmax[i & 1][hf][r] = mh;
            rows_sync();
            const float mx = fmaxf(b->xmax[i & 1][0][r], b->xmax[i & 1][1][r]);
            // lazy reference maximum: rescale O and l only when the row's maximum rises by more than 8
            const bool resc = mx > mref + 8.0f;
            if (!rows_all(!resc)) {
                // some row rescales: O must be complete up to chunk i-1 first
                if (i > 0) run = wait_phase(&b->pv_done[(i - 1) & 1], (unsigned)((i - 1) / 2) & 1u, b, status, 606);
                run = rows_all(run);
                if (!run) break;
                fence_after_sync();
                const float alpha = resc ? ex2(mref - mx) : 1.0f;   // 0 when mref is -inf
                if (resc) {
                    lsum *= alpha;
                    mref = mx;
                }
                if (i > 0) {
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t oc = tl + T_O + (uint32_t)(64 * hf + 32 * c);
                        uint32_t o[32];
                        tmem_ld32(oc, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(oc, o);
                    }
                    tmem_st_wait();
                }
            }
            // P buffer (i & 1) is free once PV(i-2) is done
            if (i >= 2) run = wait_phase(&b->pv_done[i & 1], (unsigned)((i - 2) / 2) & 1u, b, status, 607);
            run = rows_all(run);
            if (!run) break;
            uint8_t *ph = smem + OFF_P + (size_t)(i & 1) * 2 * P_BYTES, *pl = ph + P_BYTES;
            const bool none = mref == -INFINITY;
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) {
                unsigned hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float p0 = none ? 0.f : ex2(sv[c16 * 8 + 2 * j] - mref);
                    const float p1 = none ? 0.f : ex2(sv[c16 * 8 + 2 * j + 1] - mref);
                    lsum += p0 + p1;
                    __half h0, r0, h1, r1;
                    lfk::split_h(p0, h0, r0);
                    lfk::split_h(p1, h1, r1);
                    hw[j] = lfk::pack_h2(h0, h1);
                    lw[j] = lfk::pack_h2(r0, r1);
                }
                const uint32_t o = sw128(r, 4 * hf + c16);
                *reinterpret_cast<uint4 *>(ph + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(pl + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_async_smem();
            fence_before_sync();
            lfk::mbar_arrive(&b->p_full[i & 1]);
            if (stp && threadIdx.x == 0) stp[3] = lfk::globaltimer_ns();
        }
        // ---- output: O / l (the two halves' sums added), split into FP16 head and remainder
        if (run) run = wait_phase(&b->o_done, 0u, b, status, 608);
        run = rows_all(run);
        if (stp && threadIdx.x == 0) stp[4] = lfk::globaltimer_ns();
        if (run) {
            fence_after_sync();
            b->xmax[0][hf][r] = lsum;
            rows_sync();
            const float tot = b->xmax[0][0][r] + b->xmax[0][1][r];
            const float inv = live ? 1.0f / tot : 0.f;
            __half *dh = Ah + (size_t)(t0 + r) * g.Q + (size_t)h * HD + 64 * hf;
            __half *dl = Al + (size_t)(t0 + r) * g.Q + (size_t)h * HD + 64 * hf;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                tmem_ld32(tl + T_O + (uint32_t)(64 * hf + 32 * c), o);
                tmem_ld_wait();
                if (!live) continue;
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    unsigned hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __half h0, r0, h1, r1;
                        lfk::split_h(__uint_as_float(o[j + 2 * u]) * inv, h0, r0);
                        lfk::split_h(__uint_as_float(o[j + 2 * u + 1]) * inv, h1, r1);
                        hw[u] = lfk::pack_h2(h0, h1);
                        lw[u] = lfk::pack_h2(r0, r1);
                    }
                    *reinterpret_cast<uint4 *>(dh + c * 32 + j) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(dl + c * 32 + j) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (stp && threadIdx.x == 0) stp[6] = lfk::globaltimer_ns();
    if (warp == W_MMA) {
        if (lane == 0) settle_phase(&b->o_done, 0u);   // no MMA still writes TMEM
        __syncwarp();
        fence_after_sync();
        tmem_dealloc(tmem, T_COLS);
    }
}

}  // namespace lfa

// Causal attention of a prefill block (head_dim 128) on the tensor cores:
// q rows from Qr [T, Q] (FP32), K and V from the cache (tensor maps over the
// cache as [L * Hkv * max_seq, 128] FP16 rows, boxes of 64 rows x 64
// columns, no swizzle), output split into Ah / Al [T, Q].  Launched as a
// programmatic dependent of the previous kernel on `stream`.
extern "C" cudaError_t lfa_launch(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const float *Qr, int T, int pos0,
                                  int l, lfk::Geo g, const int *win, __half *Ah, __half *Al, unsigned *status,
                                  unsigned long long *stamps, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(lfa::attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lfa::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    if (g.hd != lfa::HD) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((T + lfa::BM - 1) / lfa::BM), (unsigned)g.Hq);
    cfg.blockDim = dim3(lfa::NTHR);
    cfg.dynamicSmemBytes = lfa::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lfa::attn_tc, *tm_k, *tm_v, Qr, T, pos0, l, g, win, Ah, Al, status, stamps);
}

// Tensor map of a KV cache [rows, 128] FP16 for lfa_launch (boxes of 64 x 64,
// no swizzle: the rows are stored pre-swizzled).  0 on success.
extern "C" int lfa_cache_map(CUtensorMap *out, const void *cache, unsigned long long rows)
{
    typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);
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
    const cuuint64_t dims[2] = {(cuuint64_t)lfa::HD, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)lfa::HD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)lfa::BN};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(cache), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 3;
}

static_assert(lfa::OFF_BAR + sizeof(lfa::Bars) <= lfa::SMEM, "attention shared memory layout");
