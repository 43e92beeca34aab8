// lf_kernel.cu -- the persistent decode monokernel for sm_103a.
//
// One CTA per SM runs every stage of every decode step, as in the KOG
// monokernel (shivam2003.com, "Pillar 3 -- the monokernel runtime"):
//
//   for step:                                    (one token)
//     for layer:
//       QKV   rmsnorm(x) . [Wq;Wk;Wv] -> RoPE -> q, K/V cache append (FP16)
//       ATTN  split-KV attention pieces -> the last piece of a KV head combines
//       O     x += Wo . attn
//       GU    h = SiLU(Wg . rmsnorm(x)) * (Wu . rmsnorm(x))
//       D     x += Wd . h
//     LM      logits = Whead . rmsnorm(x) -> per-CTA candidates -> the last CTA samples
//
// Warp roles.  Warp NCW (the producer) streams this CTA's weights -- repacked
// at handle creation into one contiguous per-CTA stream in consumption order
// -- and the K/V sub-blocks of its attention pieces through a shared-memory
// byte ring with 1-D TMA bulk copies carrying an L2 evict-first hint
// (shivam2003.com, "Weight streaming -- keeping HBM saturated": non-temporal
// weight loads, and weights for the next stages fetched while the current
// one still runs).  It never waits for activations, so the ring fills ahead
// across stage, layer and token boundaries.  Warps 0..NCW-1 (the consumers)
// compute.
//
// Synchronisation.  In the default schedule a stage waits only for the
// counters of the data it reads (stackfutures.com, "The Monokernel":
// per-dependency waits instead of a global barrier).  Producers publish with
// red.release.gpu; consumers poll with ld.acquire.gpu.  Counters only grow:
// stage s of layer l is complete for forward pass e when its counter reaches
// (e + 1) * (number of CTAs that publish it).  Every wait is bounded by a
// %globaltimer deadline; on expiry the kernel records the error, raises an
// abort flag that every other wait also polls, drains its in-flight copies
// and returns.
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "lf_internal.cuh"
#include "lf_ptx.cuh"

namespace lfk {

// ---------------------------------------------------------------- shared memory

struct SmemLayout {
    unsigned res, full, empty, chunk_end, red, hist, misc, plan;
    unsigned ring, acta, lmkeys, win, total;
};

__host__ __device__ inline unsigned align_up(unsigned x, unsigned a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int ring_bytes, int a_floats, int lm_rows_max, int L)
{
    // Fixed-size parts first: their offsets are compile-time constants, so
    // their addresses cost no registers; the ring, the attention scratch and
    // the LM keys follow at offsets that depend on the model.
    SmemLayout s;
    unsigned o = 0;
    s.res = o;       o = align_up(o + 4u * PART_BUFS * NCW * PART_STRIDE, 128);
    s.full = o;      o += 8u * TICKETS;
    s.empty = o;     o += 8u * TICKETS;
    s.chunk_end = o; o += 8u * TICKETS;
    s.red = o;       o = align_up(o + 4u * 64u, 16);
    s.hist = o;      o = align_up(o + 4u * 256u, 16);
    s.misc = o;      o = align_up(o + 4u * 64u, 128);
    s.plan = o;      o = align_up(o + (unsigned)sizeof(CtaPlan), 128);
    s.ring = o;      o = align_up(o + (unsigned)ring_bytes, 128);
    s.acta = o;      o = align_up(o + 4u * (unsigned)a_floats, 128);
    s.lmkeys = o;    o = align_up(o + 8u * (unsigned)lm_rows_max, 128);
    s.win = o;       o = align_up(o + 4u * (unsigned)L, 128);   // attention window of each layer
    // the GEMV reads whole 8-row blocks: keep 7 rows of readable bytes after the ring
    const unsigned slack_end = s.ring + (unsigned)ring_bytes + 7u * KC_BYTES;
    s.total = o > slack_end ? o : align_up(slack_end, 128);
    return s;
}

// misc word indices.  M_TCNT + b / M_TRED + b: consumer arrivals at / reducer
// passes over partial-sum buffer b (cumulative).  M_LMDONE: decode steps
// whose LM-head keys are complete.
// Mixture of experts: M_ROUTE counts the expert choices made in this launch;
// M_SEL + 8 * (l & 1) + j and M_GATE + 8 * (l & 1) + j hold slot j's expert
// and gate (FP32 bits) of layer l.
enum { M_FLAG = 0, M_TOKEN = 1, M_DIGIT = 2, M_REMAIN = 3, M_LMDONE = 6, M_ROUTE = 7,
       M_TCNT = 16, M_TRED = 24, M_SEL = 32, M_GATE = 48 };

struct Ctx {
    const Params *p;
    const CtaPlan *plan;  // this CTA's partition, copied to shared memory (global reads
                          // after an ld.acquire miss L1 and cost an L2 round trip)
    uint8_t *ring;
    float *acta;      // attention scratch
    unsigned long long *lmkeys;
    float *res;
    uint64_t *full, *empty;
    unsigned long long *chunk_end;
    float *red;
    unsigned *hist;
    unsigned *misc;
    const int *win;   // [L] attention window of each layer (0: whole cache), in shared memory
    int b;            // CTA index
    int tid, warp, lane;
};

// Stage ids for the multi-kernel schedule's stage filter.
enum { SID_QKV = 0, SID_ATTN = 1, SID_O = 2, SID_GU = 3, SID_D = 4, SID_LM = 5 };

__device__ __forceinline__ bool stage_active(const Params &p, int layer, int sid)
{
    if (p.only_stage < 0) return true;
    return p.only_stage == sid && (sid == SID_LM || p.only_layer == layer);
}

__device__ __forceinline__ void trace_mark(const Ctx &c, int step, int slot, int stamp)
{
    const Params &p = *c.p;
    if (p.trace && c.tid == 0 && step < p.trace_steps)
        p.trace[(((size_t)step * trace_slots(p.g.L) + slot) * p.P + c.b) * TR_N + stamp] = globaltimer_ns();
}
__device__ __forceinline__ void trace_mark_producer(const Ctx &c, int step, int slot, int stamp)
{
    const Params &p = *c.p;
    if (p.trace && step < p.trace_steps)
        p.trace[(((size_t)step * trace_slots(p.g.L) + slot) * p.P + c.b) * TR_N + stamp] = globaltimer_ns();
}

// ---------------------------------------------------------------- bounded waits

__device__ __forceinline__ void raise_error(const Params &p, unsigned code, unsigned where, unsigned layer,
                                            unsigned step)
{
    if (atomicCAS(p.status, 0u, code) == 0u) {
        p.status[1] = where;
        p.status[2] = layer;
        p.status[3] = step;
    }
    atomicExch(p.abort_flag, 1u);
}

// Spin until (int)(*ctr - target) >= 0.  Returns false on timeout or abort.
// The spin loops live out of line (one copy each) to keep the kernel's
// executed code small; callers try once inline first.
__device__ __forceinline__ bool wait_counter_slow(const Params &p, const unsigned *ctr, unsigned target, unsigned where,
                                               unsigned layer, unsigned step)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        if ((int)(ld_acquire(ctr) - target) >= 0) return true;
        if ((it & 31u) == 31u) {
            if (ld_relaxed(p.abort_flag)) return false;
            unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > p.timeout_ns) {
                raise_error(p, STATUS_TIMEOUT, where, layer, step);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_counter(const Params &p, const unsigned *ctr, unsigned target, unsigned where,
                                             unsigned layer, unsigned step)
{
    if ((int)(ld_acquire(ctr) - target) >= 0) return true;
    return wait_counter_slow(p, ctr, target, where, layer, step);
}

__device__ __forceinline__ bool wait_mbar_slow(const Params &p, uint64_t *bar, unsigned parity, unsigned where)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (ld_relaxed(p.abort_flag)) return false;
            unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > p.timeout_ns) {
                raise_error(p, STATUS_TIMEOUT, where, 0xFFFFu, 0xFFFFu);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_mbar(const Params &p, uint64_t *bar, unsigned parity, unsigned where)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_mbar_slow(p, bar, parity, where);
}

// ---------------------------------------------------------------- ring cursors

// Both sides place chunks identically: a chunk that would cross the end of the
// ring starts at offset 0 instead.
struct ConsRing {
    unsigned n = 0;       // chunks consumed
    unsigned off = 0;     // read offset
    unsigned waited = 0;  // chunks that had not landed when first asked for (for the trace)
    __device__ __forceinline__ const uint8_t *acquire(const Ctx &c, unsigned bytes, bool &ab)
    {
        if (off + bytes > (unsigned)c.p->ring_bytes) off = 0;
        const uint8_t *ptr = c.ring + off;
        off += bytes;
        bool fail = ab;
        if (!fail && !mbar_try_wait(&c.full[n % TICKETS], (n / TICKETS) & 1u)) {
            ++waited;
            fail = !wait_mbar(*c.p, &c.full[n % TICKETS], (n / TICKETS) & 1u, 100);
        }
        if (__any_sync(0xffffffffu, fail)) {
            ab = true;
            return nullptr;
        }
        return ptr;
    }
    __device__ __forceinline__ void release(const Ctx &c)
    {
        __syncwarp();
        if (c.lane == 0) mbar_arrive(&c.empty[n % TICKETS]);
        ++n;
    }
    // A chunk owned by one warp: the other warps only advance their cursor;
    // the owner releases it for all NCW consumer warps at once.
    __device__ __forceinline__ void skip(const Ctx &c, unsigned bytes)
    {
        if (off + bytes > (unsigned)c.p->ring_bytes) off = 0;
        off += bytes;
        ++n;
    }
    __device__ __forceinline__ void release_own(const Ctx &c)
    {
        __syncwarp();
        if (c.lane == 0) mbar_arrive_cnt(&c.empty[n % TICKETS], NCW);
        ++n;
    }
};

struct ProdRing {
    unsigned n = 0, off = 0, tail_n = 0;
    unsigned long long alloc = 0, tail_b = 0;
    uint64_t pol = 0;     // weights: read once per token, L2 evict-first
    uint64_t pol_kv = 0;  // KV cache
    // Reserve `bytes` of ring and a ticket; returns the ring offset or -1 on abort.
    __device__ __forceinline__ int reserve(const Ctx &c, unsigned bytes)
    {
        const unsigned RB = (unsigned)c.p->ring_bytes;
        if (off + bytes > RB) {
            alloc += RB - off;
            off = 0;
        }
        while (n - tail_n >= (unsigned)TICKETS || alloc + bytes - tail_b > RB) {
            if (!wait_mbar(*c.p, &c.empty[tail_n % TICKETS], (tail_n / TICKETS) & 1u, 101)) return -1;
            tail_b = c.chunk_end[tail_n % TICKETS];
            ++tail_n;
        }

        c.chunk_end[n % TICKETS] = alloc + bytes;
        int o = (int)off;
        off += bytes;
        alloc += bytes;
        return o;
    }
    __device__ __forceinline__ bool emit(const Ctx &c, const void *src, unsigned bytes)
    {
        int o = reserve(c, bytes);
        if (o < 0) return false;
        uint64_t *bar = &c.full[n % TICKETS];
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(c.ring + o, src, bytes, bar, pol);
        ++n;
        return true;
    }
    // K and V rows of one attention sub-block (L2 policy pol_kv).
    __device__ bool emit2(const Ctx &c, const void *src0, const void *src1, unsigned half_bytes)
    {
        int o = reserve(c, 2 * half_bytes);
        if (o < 0) return false;
        uint64_t *bar = &c.full[n % TICKETS];
        mbar_arrive_expect_tx(bar, 2 * half_bytes);
        bulk_g2s(c.ring + o, src0, half_bytes, bar, pol_kv);
        bulk_g2s(c.ring + o + half_bytes, src1, half_bytes, bar, pol_kv);
        ++n;
        return true;
    }
    // After an abort: wait (bounded) until every issued copy has landed, so
    // that no TMA write into shared memory is in flight when the CTA exits.
    __device__ void drain(const Ctx &c)
    {
        unsigned first = (n > (unsigned)TICKETS && n - TICKETS > tail_n) ? n - TICKETS : tail_n;
        for (unsigned k = first; k < n; ++k) {
            unsigned long long t0 = globaltimer_ns();
            while (!mbar_try_wait(&c.full[k % TICKETS], (k / TICKETS) & 1u)) {
                if ((long long)(globaltimer_ns() - t0) > c.p->timeout_ns) break;
            }
        }
    }
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

__device__ __forceinline__ float dot8(uint4 w, float4 xa, float4 xb, float acc)
{
    float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
    float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
    float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&w.z));
    float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&w.w));
    acc = fmaf(f0.x, xa.x, acc);
    acc = fmaf(f0.y, xa.y, acc);
    acc = fmaf(f1.x, xa.z, acc);
    acc = fmaf(f1.y, xa.w, acc);
    acc = fmaf(f2.x, xb.x, acc);
    acc = fmaf(f2.y, xb.y, acc);
    acc = fmaf(f3.x, xb.z, acc);
    acc = fmaf(f3.y, xb.w, acc);
    return acc;
}

// Packed FP32 arithmetic for the weight chunks: rows r and r + 1 share one
// fma.rn.f32x2 per column (the .x half carries row r, the .y half row r + 1),
// so a lane issues half the FMA instructions while each row keeps its own
// chain of single-rounded FMAs in column order.  fa / fb: the lane's 8 decoded
// weights of the two rows (column pairs), xd: the 8 input values, each
// duplicated into both halves.
__device__ __forceinline__ float2 h2f2(unsigned w) { return __half22float2(*reinterpret_cast<const __half2 *>(&w)); }
__device__ __forceinline__ void dup8(const float4 &xa, const float4 &xb, float2 (&xd)[8])
{
    xd[0] = make_float2(xa.x, xa.x); xd[1] = make_float2(xa.y, xa.y);
    xd[2] = make_float2(xa.z, xa.z); xd[3] = make_float2(xa.w, xa.w);
    xd[4] = make_float2(xb.x, xb.x); xd[5] = make_float2(xb.y, xb.y);
    xd[6] = make_float2(xb.z, xb.z); xd[7] = make_float2(xb.w, xb.w);
}
__device__ __forceinline__ float2 dot8_pair(const float2 (&fa)[4], const float2 (&fb)[4], const float2 (&xd)[8],
                                            float2 acc)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = __ffma2_rn(make_float2(fa[i].x, fb[i].x), xd[2 * i], acc);
        acc = __ffma2_rn(make_float2(fa[i].y, fb[i].y), xd[2 * i + 1], acc);
    }
    return acc;
}

__device__ __forceinline__ float gumbel_dev(unsigned long long seed, int pos, int i)
{
    uint4 r = philox4x32_10(make_uint4((unsigned)i >> 2, (unsigned)pos, 0u, 0u),
                            make_uint2((unsigned)(seed & 0xFFFFFFFFull), (unsigned)(seed >> 32)));
    unsigned w = (i & 3) == 0 ? r.x : (i & 3) == 1 ? r.y : (i & 3) == 2 ? r.z : r.w;
    float u = (float)((w >> 9) * 2u + 1u) * 0x1p-24f;
    return -logf(-logf(u));
}

// ---------------------------------------------------------------- tagged activations

// The parity a value of forward pass e carries in its lowest mantissa bit
// (pass 0 carries 1, so the zero-filled buffers of a fresh or reset handle
// never pass for pass 0's values).
__device__ __forceinline__ unsigned pass_tag(unsigned e) { return (e & 1u) ^ 1u; }
__device__ __forceinline__ float tag_value(float v, unsigned tag) { return __uint_as_float((__float_as_uint(v) & ~1u) | tag); }
// Stores v with the tag (a relaxed gpu-scope store: the readers poll it with
// relaxed gpu-scope loads).
__device__ __forceinline__ void st_tagged(float *dst, float v, unsigned tag)
{
    asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(dst), "f"(tag_value(v, tag)) : "memory");
}
__device__ __forceinline__ bool tagged_ok(float v, unsigned tag) { return (__float_as_uint(v) & 1u) == tag; }
__device__ __forceinline__ float4 ld_relaxed_f4(const float *ptr)
{
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(ptr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float ld_relaxed_f(const float *ptr)
{
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(ptr) : "memory");
    return v;
}

// ---------------------------------------------------------------- stage plumbing

__device__ __forceinline__ unsigned *sig_ptr(const Params &p, int l, int idx)
{
    return p.sig + ((size_t)l * sig_layout(p.g).per_layer + idx) * SIG_STRIDE;
}

// Spin (one thread) until the cumulative shared-memory count *w reaches
// target.  Returns false on timeout or abort.
__device__ __forceinline__ bool wait_smem_ge(const Params &p, const unsigned *w, unsigned target, unsigned where,
                                             unsigned layer, unsigned step)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        if ((int)(*reinterpret_cast<const volatile unsigned *>(w) - target) >= 0) return true;
        if ((it & 255u) == 255u) {
            if (ld_relaxed(p.abort_flag)) return false;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > p.timeout_ns) {
                raise_error(p, STATUS_TIMEOUT, where, layer, step);
                return false;
            }
        }
    }
}

// Warp-wide poll of 8 tagged values per lane (columns 8 lane .. 8 lane + 7
// of a 256-element slice at src) until every value of the warp carries
// `tag`; the values arrive in xa, xb.  Returns false on timeout or abort.
__device__ bool poll_slice(const Params &p, const float *src, unsigned tag, float4 &xa, float4 &xb, unsigned where,
                           int l, int step)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        xa = ld_relaxed_f4(src);
        xb = ld_relaxed_f4(src + 4);
        const bool ok = tagged_ok(xa.x, tag) && tagged_ok(xa.y, tag) && tagged_ok(xa.z, tag) &&
                        tagged_ok(xa.w, tag) && tagged_ok(xb.x, tag) && tagged_ok(xb.y, tag) &&
                        tagged_ok(xb.z, tag) && tagged_ok(xb.w, tag);
        if (__all_sync(0xffffffffu, ok)) return true;
        // after two misses, back off briefly: warps that ran ahead of their
        // input (no chunk in a stage) would otherwise keep L2 busy with polls
        // that the stages still being computed wait behind
        if (it >= 2) __nanosleep(64);
        if ((it & 15u) == 15u) {
            bool stop = ld_relaxed(p.abort_flag) != 0u;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if (!stop && (long long)(now - t0) > p.timeout_ns) {
                if ((threadIdx.x & 31) == 0) raise_error(p, STATUS_TIMEOUT, where, l, step);
                stop = true;
            }
            if (__any_sync(0xffffffffu, stop)) return false;
        }
    }
}
// The same for one tagged value (one thread).
__device__ bool poll_value(const Params &p, const float *src, unsigned tag, float &v, unsigned where, int l, int step)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        v = ld_relaxed_f(src);
        if (tagged_ok(v, tag)) return true;
        if ((it & 15u) == 15u) {
            if (ld_relaxed(p.abort_flag)) return false;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > p.timeout_ns) {
                raise_error(p, STATUS_TIMEOUT, where, l, step);
                return false;
            }
        }
    }
}

// The same for four tagged values (one thread).
__device__ bool poll_f4(const Params &p, const float *src, unsigned tag, float4 &v, unsigned where, int l, int step)
{
    unsigned long long t0 = 0;
    for (unsigned it = 0;; ++it) {
        v = ld_relaxed_f4(src);
        if (tagged_ok(v.x, tag) && tagged_ok(v.y, tag) && tagged_ok(v.z, tag) && tagged_ok(v.w, tag)) return true;
        if ((it & 15u) == 15u) {
            if (ld_relaxed(p.abort_flag)) return false;
            const unsigned long long now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > p.timeout_ns) {
                raise_error(p, STATUS_TIMEOUT, where, l, step);
                return false;
            }
        }
    }
}

// Count the outputs [e0, e0 + n) of a stage in the readiness counters of the
// groups of `per` elements they fall in (`base`: counter of group 0).  Called
// by one lane after __syncwarp or a barrier; the single gpu-scope fence turns
// the relaxed adds into releases of every store the group made before.
__device__ __forceinline__ void publish_range(unsigned *base, int e0, int n, int per)
{
    fence_acq_rel_gpu();
    const int end = e0 + n;
    for (int e = e0; e < end;) {
        const int grp = e / per;
        const int stop = min(end, (grp + 1) * per);
        red_relaxed_add(base + (size_t)grp * SIG_STRIDE, (unsigned)(stop - e));
        e = stop;
    }
}

// Grid-barrier schedule: index of the barrier that closes (step, layer, slot).
// Slots 0..4 close QKV, attention, O, GU and D of a layer; slot 5 closes the
// LM head and sampling of a decode step.
__device__ __forceinline__ unsigned gbar_index(const Params &p, int step, int l, int slot)
{
    const unsigned per_step = 5u * (unsigned)p.g.L + (p.mode == MODE_DECODE ? 1u : 0u);
    const unsigned in_step = slot == 5 ? 5u * (unsigned)p.g.L : (unsigned)l * 5u + (unsigned)slot;
    return p.gbar_base + (unsigned)step * per_step + in_step;
}

// The grid barrier a sub-stage waits for in the barrier schedule: the one
// that closes the previous sub-stage (false: none, the first sub-stage of the
// call).
__device__ __forceinline__ bool grid_barrier_before(const Params &p, int step, int l, int sid, unsigned &idx)
{
    int gstep = step, gl = l, gslot = sid - 1;
    if (sid == SID_QKV) {
        if (l > 0) {
            gl = l - 1;
            gslot = 4;
        } else {
            if (step == 0) return false;
            gstep = step - 1;
            gl = p.g.L - 1;
            gslot = p.mode == MODE_DECODE ? 5 : 4;
        }
    } else if (sid == SID_LM) {
        gl = p.g.L - 1;
        gslot = 4;
    }
    idx = gbar_index(p, gstep, gl, gslot);
    return true;
}

// Consumer-side dependency wait: thread 0 polls, then the consumer warps
// meet at a named barrier that also ORs the abort state.  Returns true if
// the CTA must stop.
__device__ __forceinline__ bool cons_wait(const Ctx &c, const unsigned *ctr, unsigned target, unsigned where, int l, int step,
                          bool ab)
{
    if (c.tid == 0 && !ab) ab = !wait_counter(*c.p, ctr, target, where, l, step);
    return cons_sync_or(ab);
}

// Arrival of this CTA at the grid barrier (barrier schedule), after all
// consumer writes of the sub-stage.
__device__ __forceinline__ bool cons_grid_arrive(const Ctx &c, bool ab)
{
    ab = cons_sync_or(ab);
    if (ab) return true;
    if (c.tid == 0) {
        fence_acq_rel_gpu();
        red_release_add(c.p->gbar, 1u);
    }
    return false;
}

__device__ __forceinline__ int stage_of(int sid)
{
    return sid == SID_QKV ? ST_QKV : sid == SID_O ? ST_O : sid == SID_GU ? ST_GU : sid == SID_D ? ST_D : ST_LM;
}

// Input of a GEMV stage: the FP32 vector (null for layer 0's QKV, which reads
// the FP16 embedding row of the step's token) and the RMSNorm gain row (null
// for the O and down projections).  The vector's values are tagged with the
// pass that wrote them (see pass_tag).
struct StageIn {
    const float *src32;
    const __half *gain;
};

__device__ __forceinline__ StageIn stage_input(const Params &p, int s, int l)
{
    const Geo &g = p.g;
    StageIn in;
    in.src32 = nullptr;
    in.gain = nullptr;
    if (s == ST_QKV) {
        in.gain = p.attn_norm + (size_t)l * g.d;
        if (l > 0) in.src32 = p.xout + (size_t)(l - 1) * g.d;
    } else if (s == ST_O) {
        in.src32 = p.attn + (size_t)l * g.Q;
    } else if (s == ST_GU) {
        in.src32 = p.xattn + (size_t)l * g.d;
        in.gain = p.ffn_norm + (size_t)l * g.d;
    } else if (s == ST_D) {
        in.src32 = p.hbuf + (size_t)l * g.F;
    } else {
        in.src32 = p.xout + (size_t)(g.L - 1) * g.d;
        in.gain = p.final_norm;
    }
    return in;
}

// A warp's position in the CTA's sequence of sub-stages, advanced identically
// by the consumer warps and the reducer: tiles passed (the partial-sum buffer
// sequence) and, with a mixture of experts, expert choices made.
struct PipeState {
    unsigned seq = 0, routes = 0;
};

// Token fed to forward pass `step` (decode: after its counter was acquired).
// An id outside [0, V) is reported (LF_ERR_INVALID_ARG via lf_sync) and
// replaced by 0, so that no embedding read leaves the table.
__device__ __forceinline__ int step_token(const Params &p, int step)
{
    int t;
    if (p.mode == MODE_PREFILL) {
        if (p.has_pending) t = step == 0 ? __ldcg(p.tok_buf) : __ldg(p.prompt + step - 1);
        else t = __ldg(p.prompt + step);
    } else {
        t = step == 0 ? __ldcg(p.tok_buf) : __ldcg(p.tok_seq + step - 1);
    }
    if ((unsigned)t >= (unsigned)p.g.V) {
        raise_error(p, STATUS_BAD_TOKEN, 300, 0, (unsigned)step);
        t = 0;
    }
    return t;
}

// FP32 scale of row `part` of unit `unit` of stage s, layer l (FP8 weights),
// from the caller's per-row scales.
__device__ __forceinline__ float row_scale(const Params &p, int s, int l, int unit, int part)
{
    const Geo &g = p.g;
    switch (s) {
    case ST_QKV: {
        const int half = g.hd / 2;
        const int hh = unit / half, j = unit % half;
        const int r = hh * g.hd + j + part * half;
        if (r < g.Q) return __ldg(p.wsc[0] + (size_t)l * g.Q + r);
        if (r < g.Q + g.KV) return __ldg(p.wsc[1] + (size_t)l * g.KV + (r - g.Q));
        return __ldg(p.wsc[2] + (size_t)l * g.KV + (r - g.Q - g.KV));
    }
    case ST_O: return __ldg(p.wsc[3] + (size_t)l * g.d + unit);
    case ST_GU: return __ldg(p.wsc[part ? 5 : 4] + (size_t)l * g.F + unit);
    case ST_D: return __ldg(p.wsc[6] + (size_t)l * g.d + unit);
    default: return __ldg(p.wsc[7] + unit);
    }
}

// ---------------------------------------------------------------- GEMV stages

// One weight chunk (R rows x 256 columns, row-major, R <= 32) consumed by one
// warp: lane l holds the 8 input values of columns 8l..8l+7 (xa, xb) and
// accumulates all R rows, so each lane carries R independent FMA chains
// (advanced two rows per packed FMA).
__device__ __forceinline__ void gemv_chunk(const Ctx &c, const uint8_t *ch, int R, const float4 &xa, const float4 &xb,
                                           float (&acc)[TILE_ROWS])
{
    // 32-bit shared addresses: the lane's 16 bytes of row r sit at chunk + r * 512 + lane * 16.
    const uint32_t a0 = smem_u32(ch) + (uint32_t)c.lane * 16u;
    float2 xd[8];
    dup8(xa, xb, xd);
    // Rows in blocks of 8 at constant offsets: one branch per block, so the 8
    // loads issue together and the 8 FMA chains interleave.  The last block
    // may read up to 7 rows past the chunk (inside the ring, or in the slack
    // the shared-memory layout keeps after it); those sums land in lanes
    // >= R after the row reduction and are never used.
#pragma unroll
    for (int rb = 0; rb < TILE_ROWS; rb += 8) {
        if (rb < R) {
            uint4 wv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) wv[r] = lds_u4(a0 + (uint32_t)(rb + r) * KC_BYTES);
#pragma unroll
            for (int r = 0; r < 8; r += 2) {
                const float2 fa[4] = {h2f2(wv[r].x), h2f2(wv[r].y), h2f2(wv[r].z), h2f2(wv[r].w)};
                const float2 fb[4] = {h2f2(wv[r + 1].x), h2f2(wv[r + 1].y), h2f2(wv[r + 1].z), h2f2(wv[r + 1].w)};
                const float2 o = dot8_pair(fa, fb, xd, make_float2(acc[rb + r], acc[rb + r + 1]));
                acc[rb + r] = o.x;
                acc[rb + r + 1] = o.y;
            }
        }
    }
}

// The same for an FP8 chunk (R rows x 256 E4M3 codes, 256 bytes per row): lane
// l's 8 bytes of row r are decoded pairwise to FP16 (cvt.rn.f16x2.e4m3x2) and
// then to FP32 before the (packed) FMAs; the row's scale is applied to the
// finished sum.
__device__ __forceinline__ float2 e4m3x2_f2(unsigned short v)
{
    unsigned h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}
__device__ __forceinline__ uint2 lds_u2(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ void gemv_chunk_fp8(const Ctx &c, const uint8_t *ch, int R, const float4 &xa, const float4 &xb,
                                               float (&acc)[TILE_ROWS])
{
    constexpr uint32_t RB = KC;                        // bytes of one row
    const uint32_t a0 = smem_u32(ch) + (uint32_t)c.lane * 8u;
    float2 xd[8];
    dup8(xa, xb, xd);
#pragma unroll
    for (int rb = 0; rb < TILE_ROWS; rb += 8) {
        if (rb < R) {
            uint2 wv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) wv[r] = lds_u2(a0 + (uint32_t)(rb + r) * RB);
#pragma unroll
            for (int r = 0; r < 8; r += 2) {
                const float2 fa[4] = {e4m3x2_f2((unsigned short)(wv[r].x & 0xFFFFu)),
                                      e4m3x2_f2((unsigned short)(wv[r].x >> 16)),
                                      e4m3x2_f2((unsigned short)(wv[r].y & 0xFFFFu)),
                                      e4m3x2_f2((unsigned short)(wv[r].y >> 16))};
                const float2 fb[4] = {e4m3x2_f2((unsigned short)(wv[r + 1].x & 0xFFFFu)),
                                      e4m3x2_f2((unsigned short)(wv[r + 1].x >> 16)),
                                      e4m3x2_f2((unsigned short)(wv[r + 1].y & 0xFFFFu)),
                                      e4m3x2_f2((unsigned short)(wv[r + 1].y >> 16))};
                const float2 o = dot8_pair(fa, fb, xd, make_float2(acc[rb + r], acc[rb + r + 1]));
                acc[rb + r] = o.x;
                acc[rb + r + 1] = o.y;
            }
        }
    }
}

// The same for an MXFP4 chunk (R rows x 144 bytes: 128 bytes of packed E2M1
// codes, then the E8M0 scales of the row's eight 32-column blocks): lane l's
// 4 code bytes (columns 8l..8l+7, one quarter of block l/4) are decoded
// pairwise to FP16 (cvt.rn.f16x2.e2m1x2, exact), multiplied with x in FP32,
// and the lane's partial sum is scaled by its block's 2^(E-127) (exact) before
// it joins the row's accumulator.
__device__ __forceinline__ void e2m1x8_h2(unsigned w, unsigned &h0, unsigned &h1, unsigned &h2, unsigned &h3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}
// 2^(e - 127) for an E8M0 byte: the FP32 with that exponent field (e = 0:
// the subnormal 2^-127; e = 255: NaN).
__device__ __forceinline__ float e8m0_f(unsigned e)
{
    return e == 0u ? __uint_as_float(0x00400000u) : e == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float(e << 23);
}
// Rows r and r + 1 (codes wa / wb, block scales sa / sb) with packed FMAs:
// per row the product of column 0, seven FMAs, then the scaled partial joins
// the accumulator.
__device__ __forceinline__ float2 dot8_mxfp4_pair(unsigned wa, unsigned sa, unsigned wb, unsigned sb,
                                                  const float2 (&xd)[8], float2 acc)
{
    unsigned a0, a1, a2, a3, b0, b1, b2, b3;
    e2m1x8_h2(wa, a0, a1, a2, a3);
    e2m1x8_h2(wb, b0, b1, b2, b3);
    const float2 fa[4] = {h2f2(a0), h2f2(a1), h2f2(a2), h2f2(a3)};
    const float2 fb[4] = {h2f2(b0), h2f2(b1), h2f2(b2), h2f2(b3)};
    float2 part = __fmul2_rn(make_float2(fa[0].x, fb[0].x), xd[0]);
    part = __ffma2_rn(make_float2(fa[0].y, fb[0].y), xd[1], part);
#pragma unroll
    for (int i = 1; i < 4; ++i) {
        part = __ffma2_rn(make_float2(fa[i].x, fb[i].x), xd[2 * i], part);
        part = __ffma2_rn(make_float2(fa[i].y, fb[i].y), xd[2 * i + 1], part);
    }
    return __ffma2_rn(part, make_float2(e8m0_f(sa), e8m0_f(sb)), acc);
}
__device__ __forceinline__ unsigned lds_u32(uint32_t a)
{
    unsigned v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ unsigned lds_u8(uint32_t a)
{
    unsigned short v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void gemv_chunk_mxfp4(const Ctx &c, const uint8_t *ch, int R, const float4 &xa,
                                                 const float4 &xb, float (&acc)[TILE_ROWS])
{
    constexpr uint32_t RB = fmt_crb(FMT_MXFP4);        // bytes of one row
    const uint32_t a0 = smem_u32(ch) + (uint32_t)c.lane * 4u;
    const uint32_t s0 = smem_u32(ch) + 128u + (uint32_t)(c.lane >> 2);
    float2 xd[8];
    dup8(xa, xb, xd);
#pragma unroll
    for (int rb = 0; rb < TILE_ROWS; rb += 8) {
        if (rb < R) {
            unsigned wv[8], sv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                wv[r] = lds_u32(a0 + (uint32_t)(rb + r) * RB);
                sv[r] = lds_u8(s0 + (uint32_t)(rb + r) * RB);
            }
#pragma unroll
            for (int r = 0; r < 8; r += 2) {
                const float2 o = dot8_mxfp4_pair(wv[r], sv[r], wv[r + 1], sv[r + 1], xd,
                                                 make_float2(acc[rb + r], acc[rb + r + 1]));
                acc[rb + r] = o.x;
                acc[rb + r + 1] = o.y;
            }
        }
    }
}

// Sum each of 32 per-lane values over the warp; afterwards lane r holds the
// sum of value r (31 shuffles: each level hands half of the values to the
// partner lane).
__device__ __forceinline__ float reduce_rows32(float (&v)[TILE_ROWS], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

__device__ __forceinline__ float2 h2f(unsigned w) { return __half22float2(*reinterpret_cast<const __half2 *>(&w)); }

// Consumer side of a GEMV stage.  Chunk j of the stage (tile by tile, column
// group by column group, as the producer streams them) belongs to warp
// j mod NCW.  Before a chunk the warp reads the lane's 8 input values of the
// chunk's column group in place, polling until all carry the pass's tag (no
// counter, no staging copy), adds their squares to the RMSNorm sum (tile 0
// covers every slice once) and applies the gain.  After
// each tile the warp reduces its 32 row sums over the lanes and hands them to
// the reducer through a rotating partial-sum buffer.
// Mixture of experts: every CTA chooses the layer's active experts itself,
// from the gate/up stage's input, read in place (the pages: only the
// active experts' weights stream per token), so the choice costs no grid-wide
// hop.  Warp w forms the router logits of experts w, w + 8, ... as FP32 dot
// products of the FP16 router rows with x * gain (the RMSNorm factor is a
// positive scale, applied afterwards); warp 0 scales them, takes the top k
// (ties to the lower index) and the softmax of the chosen logits, and
// publishes experts and gates in shared memory for the producer, which then
// streams only those experts' rows, and for the reducer.  Returns true if the
// CTA must stop.
__device__ __forceinline__ bool route_experts(const Ctx &c, PipeState &ps, int l, int step, bool ab)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    const unsigned tag = pass_tag(p.epoch0 + (unsigned)step);
    const float *xsrc = p.xattn + (size_t)l * g.d;
    const __half *gsrc = p.ffn_norm + (size_t)l * g.d;
    // the FFN input, staged in the attention scratch (free during the FFN):
    // slice k by warp k mod NCW, so that each warp waits for at most a few
    // slices and the polls of the eight warps overlap
    float *xs = c.acta;
    bool fail = ab;
    for (int k = c.warp; k < g.d / KC && !fail; k += NCW) {
        float4 xa, xb;
        if (!poll_slice(p, xsrc + (size_t)k * KC + c.lane * 8, tag, xa, xb, 141, l, step)) {
            fail = true;
            break;
        }
        reinterpret_cast<float4 *>(xs + (size_t)k * KC + c.lane * 8)[0] = xa;
        reinterpret_cast<float4 *>(xs + (size_t)k * KC + c.lane * 8)[1] = xb;
    }
    if (cons_sync_or(fail)) return true;
    float *logit = reinterpret_cast<float *>(c.hist);
    float ss = 0.f;
    const __half *wr = p.router + (size_t)l * g.E * g.d;
    for (int e = c.warp; e < g.E; e += NCW) {
        const __half *row = wr + (size_t)e * g.d;
        float acc = 0.f;
        for (int i = c.lane * 8; i < g.d; i += 256) {
            float4 xa = lds_f4(smem_u32(xs + i)), xb = lds_f4(smem_u32(xs + i + 4));
            if (e == 0) {
                ss = fmaf(xa.x, xa.x, ss); ss = fmaf(xa.y, xa.y, ss);
                ss = fmaf(xa.z, xa.z, ss); ss = fmaf(xa.w, xa.w, ss);
                ss = fmaf(xb.x, xb.x, ss); ss = fmaf(xb.y, xb.y, ss);
                ss = fmaf(xb.z, xb.z, ss); ss = fmaf(xb.w, xb.w, ss);
            }
            const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(gsrc + i));
            const float2 g0 = h2f(gv.x), g1 = h2f(gv.y), g2 = h2f(gv.z), g3 = h2f(gv.w);
            xa.x *= g0.x; xa.y *= g0.y; xa.z *= g1.x; xa.w *= g1.y;
            xb.x *= g2.x; xb.y *= g2.y; xb.z *= g3.x; xb.w *= g3.y;
            acc = dot8(__ldg(reinterpret_cast<const uint4 *>(row + i)), xa, xb, acc);
        }
        acc = warp_sum(acc);
        if (c.lane == 0) logit[e] = acc;
    }
    if (cons_sync_or(fail)) return true;
    if (c.warp == 0) {
        const float inv = 1.0f / sqrtf(warp_sum(ss) / (float)g.d + p.eps);
        float v0 = c.lane < g.E ? logit[c.lane] * inv : -INFINITY;
        float v1 = c.lane + 32 < g.E ? logit[c.lane + 32] * inv : -INFINITY;
        __syncwarp();
        const int b = 8 * (l & 1);
        float *top = logit + MAX_EXPERTS;   // the chosen logits, in order
        for (int j = 0; j < g.topk; ++j) {
            float bv = v0;
            int bi = c.lane;
            if (v1 > bv) {
                bv = v1;
                bi = c.lane + 32;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi == c.lane) v0 = -INFINITY;
            else if (bi == c.lane + 32) v1 = -INFINITY;
            if (c.lane == 0) {
                top[j] = bv;
                // (bi < E for any finite logits; the clamp keeps a NaN logit's
                // choice inside the stream)
                c.misc[M_SEL + b + j] = (unsigned)min(bi, g.E - 1);
            }
        }
        if (c.lane == 0) {
            float sum = 0.f;
            for (int j = 0; j < g.topk; ++j) sum += expf(top[j] - top[0]);
            for (int j = 0; j < g.topk; ++j) c.misc[M_GATE + b + j] = __float_as_uint(expf(top[j] - top[0]) / sum);
            __threadfence_block();
            *reinterpret_cast<volatile unsigned *>(&c.misc[M_ROUTE]) = ps.routes + 1u;
        }
    }
    ps.routes++;
    return false;
}

template <int FMT, bool MOE>
__device__ __forceinline__ bool stage_gemv(const Ctx &c, ConsRing &rc, PipeState &ps, int s, int l, int step, bool ab)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    const CtaPlan &pl = *c.plan;
    const StageGeom sg = stage_geom(g, s);
    const StageIn in = stage_input(p, s, l);
    const bool fp16 = in.src32 == nullptr;
    const bool norm = in.gain != nullptr;
    const int tslot = s == ST_LM ? 5 * g.L : 5 * l + (s == ST_QKV ? 0 : s + 1);
    const int nslices = sg.K / KC;
    const unsigned tag = pass_tag(p.epoch0 + (unsigned)step);
    // layer 0's QKV: the embedding row of the step's token, read in place
    const __half *emb_row = nullptr;
    if (fp16 && !ab) {
        int tok = 0;
        bool ok = true;
        if (c.lane == 0) {
            if (p.mode == MODE_DECODE && step > 0 && p.sched == SCHED_FLAGS)
                ok = wait_counter(p, p.tok_cnt, p.tok_base + (unsigned)step, 133, l, step);
            if (ok) tok = step_token(p, step);
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        tok = __shfl_sync(0xffffffffu, tok, 0);
        if (!ok) ab = true;
        emb_row = p.embed + (size_t)tok * g.d;
    }
    const int u0 = pl.u0[s], n = pl.u1[s] - u0;
    const int nt = tiles_of(n, sg.rows_per_unit);
    // gate/up: the CTA's tiles once per active expert (slot); the weights of
    // slot j's expert arrive through the ring like any other tile
    const int nslot = (MOE && s == ST_GU) ? g.topk : 1;
    int jc = 0;
    bool first = true;
    for (int jt = 0; jt < nslot * nt && !ab; ++jt) {
        const int t = MOE ? jt % nt : jt;
        int a, bnd;
        tile_range(u0, n, nt, t, a, bnd);
        const int R = (bnd - a) * sg.rows_per_unit;
        const unsigned bytes = (unsigned)R * (unsigned)fmt_crb(FMT);
        float acc[TILE_ROWS];
#pragma unroll
        for (int r = 0; r < TILE_ROWS; ++r) acc[r] = 0.f;
        float ss = 0.f;
        bool mine = false;
        for (int k = 0; k < nslices; ++k, ++jc) {
            if (jc % NCW != c.warp) {
                rc.skip(c, bytes);
                continue;
            }
            // the gain first (it does not depend on the input: its load
            // overlaps the poll)
            uint4 gv = make_uint4(0u, 0u, 0u, 0u);
            if (norm) gv = __ldg(reinterpret_cast<const uint4 *>(in.gain + (size_t)k * KC) + c.lane);
            // the lane's 8 input values, straight from global memory: fixed
            // (the embedding row) or polled until they carry this pass's tag
            float4 xa, xb;
            if (fp16) {
                const uint4 hv = __ldg(reinterpret_cast<const uint4 *>(emb_row + (size_t)k * KC) + c.lane);
                const float2 f0 = h2f(hv.x), f1 = h2f(hv.y), f2 = h2f(hv.z), f3 = h2f(hv.w);
                xa = make_float4(f0.x, f0.y, f1.x, f1.y);
                xb = make_float4(f2.x, f2.y, f3.x, f3.y);
            } else if (!poll_slice(p, in.src32 + (size_t)k * KC + c.lane * 8, tag, xa, xb, 121, l, step)) {
                ab = true;
                break;
            }
            if (first) {
                trace_mark(c, step, tslot, TR_READY);
                first = false;
            }
            if (norm) {
                if (jt == 0) {
                    ss = fmaf(xa.x, xa.x, ss); ss = fmaf(xa.y, xa.y, ss);
                    ss = fmaf(xa.z, xa.z, ss); ss = fmaf(xa.w, xa.w, ss);
                    ss = fmaf(xb.x, xb.x, ss); ss = fmaf(xb.y, xb.y, ss);
                    ss = fmaf(xb.z, xb.z, ss); ss = fmaf(xb.w, xb.w, ss);
                }
                const float2 g0 = h2f(gv.x), g1 = h2f(gv.y), g2 = h2f(gv.z), g3 = h2f(gv.w);
                xa.x *= g0.x; xa.y *= g0.y; xa.z *= g1.x; xa.w *= g1.y;
                xb.x *= g2.x; xb.y *= g2.y; xb.z *= g3.x; xb.w *= g3.y;
            }
            const uint8_t *ch = rc.acquire(c, bytes, ab);
            if (ab) break;
            if constexpr (FMT == FMT_FP8) gemv_chunk_fp8(c, ch, R, xa, xb, acc);
            else if constexpr (FMT == FMT_MXFP4) gemv_chunk_mxfp4(c, ch, R, xa, xb, acc);
            else gemv_chunk(c, ch, R, xa, xb, acc);
            mine = true;
            rc.release_own(c);
        }
        if (ab) break;
        // ---- per-warp row sums -> partial buffer of this tile
        const float v = mine ? reduce_rows32(acc, c.lane) : 0.f;
        const float ssw = (norm && jt == 0) ? warp_sum(ss) : 0.f;
        const unsigned seq = ps.seq++;
        const int buf = (int)(seq % PART_BUFS);
        const unsigned use = seq / PART_BUFS;
        // the reducer must be done with the buffer's previous use
        bool ok = true;
        if (c.lane == 0 && use > 0) ok = wait_smem_ge(p, &c.misc[M_TRED + buf], use, 110, l, step);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
            ab = true;
            break;
        }
        float *part = c.res + ((size_t)buf * NCW + c.warp) * PART_STRIDE;
        part[c.lane] = v;
        if (c.lane == 0) part[TILE_ROWS] = ssw;
        __syncwarp();
        if (c.lane == 0) {
            __threadfence_block();
            atomicAdd(&c.misc[M_TCNT + buf], 1u);
        }
    }
    if (ab) return true;
    if (c.warp == 0 && c.lane == 0) trace_mark_producer(c, step, tslot, TR_X1);
    return false;
}

// Reducer side of a GEMV stage: for each tile, in the consumers' order, wait
// for the eight warps' partials, sum them in warp order and run the stage
// epilogue (lane i: unit a + i; pair stages: rows i and i + nu): QKV outputs
// are counted in their heads' readiness counters, the others stored tagged.
template <bool MOE>
__device__ __forceinline__ bool reduce_stage(const Ctx &c, PipeState &ps, int s, int l, int step, bool ab)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    const CtaPlan &pl = *c.plan;
    const StageGeom sg = stage_geom(g, s);
    const SigLayout sl = sig_layout(g);
    const int pos = p.pos0 + step;
    const bool norm = s != ST_O && s != ST_D;
    const int tslot = s == ST_LM ? 5 * g.L : 5 * l + (s == ST_QKV ? 0 : s + 1);
    // layer 0's O residual is the embedding row of the step's token
    const int tok = (l == 0 && s == ST_O) ? __shfl_sync(0xffffffffu, c.lane == 0 ? step_token(p, step) : 0, 0) : 0;
    const bool withhold = p.mode == MODE_DECODE && step == p.fault_step && l == 0 && s == ST_QKV;
    const int u0 = pl.u0[s], n = pl.u1[s] - u0;
    const int nt = tiles_of(n, sg.rows_per_unit);
    const int nslot = (MOE && s == ST_GU) ? g.topk : 1;
    const bool moe = MOE && s == ST_GU;
    if (moe) {
        // the layer's expert choice (made by the consumers before any gate/up tile)
        bool ok = true;
        if (c.lane == 0) ok = wait_smem_ge(p, &c.misc[M_ROUTE], ps.routes + 1u, 113, l, step);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) return true;
        __threadfence_block();
        ps.routes++;
    }
    float inv = 1.f;
    const unsigned tag = pass_tag(p.epoch0 + (unsigned)step);
    bool rfail = false;
    for (int jt = 0; jt < nslot * nt; ++jt) {
        const int t = MOE ? jt % nt : jt, slot = MOE ? jt / nt : 0;
        int a, bnd;
        tile_range(u0, n, nt, t, a, bnd);
        const int nu = bnd - a;
        const unsigned seq = ps.seq++;
        const int buf = (int)(seq % PART_BUFS);
        const unsigned use = seq / PART_BUFS;
        // the epilogue's other inputs (RoPE row, residual) do not depend on
        // the partials: load them while the consumers finish the tile
        const int u = a + min(c.lane, nu - 1);
        // FP8 weights: the scales of the lane's rows (pair stages: both rows)
        float sc0 = 1.f, sc1 = 1.f;
        if (g.fmt == FMT_FP8) {
            sc0 = row_scale(p, s, l, u, 0);
            if (sg.rows_per_unit == 2) sc1 = row_scale(p, s, l, u, 1);
        }
        float2 pre = make_float2(0.f, 0.f);
        if (s == ST_QKV) {
            const int half = g.hd / 2;
            if (u / half < g.Hq + g.Hkv) pre = __ldg(p.rope + (size_t)pos * half + u % half);
        } else if (s == ST_O && l == 0) {
            pre.x = __half2float(p.embed[(size_t)tok * g.d + u]);
        } else if (s == ST_O || s == ST_D) {
            // the residual, tagged: this pass's value (in place long before: the stage consumed it)
            const float *src = s == ST_O ? p.xout + (size_t)(l - 1) * g.d + u : p.xattn + (size_t)l * g.d + u;
            if (!poll_value(p, src, tag, pre.x, 114, l, step)) rfail = true;
        }
        if (__any_sync(0xffffffffu, rfail)) return true;
        bool ok = true;
        if (c.lane == 0) ok = wait_smem_ge(p, &c.misc[M_TCNT + buf], (use + 1u) * NCW, 111, l, step);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) return true;
        if (jt == nslot * nt - 1 && c.lane == 0) trace_mark_producer(c, step, tslot, TR_X2);
        __threadfence_block();
        const volatile float *part = c.res + (size_t)buf * NCW * PART_STRIDE;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) sum += part[w * PART_STRIDE + c.lane];
        if (norm && jt == 0) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) tot += part[w * PART_STRIDE + TILE_ROWS];
            inv = 1.0f / sqrtf(tot / (float)sg.K + p.eps);
        }
        __syncwarp();
        if (c.lane == 0) {
            __threadfence_block();
            *reinterpret_cast<volatile unsigned *>(&c.misc[M_TRED + buf]) = use + 1u;
        }
        // ---- epilogue: lane i handles unit a + i (pair stages: rows i and i + nu)
        float partner = __shfl_sync(0xffffffffu, sum, (c.lane + nu) & 31);
        if (g.fmt == FMT_FP8) {
            sum *= sc0;
            partner *= sc1;
        }
        if (c.lane < nu) {
            if (s == ST_QKV) {
                const int half = g.hd / 2;
                const int hh = u / half, j = u % half;
                const float v0 = sum * inv, v1 = partner * inv;
                // q (tagged), and the K/V cache row (FP16) plus its tagged
                // FP32 copy in kvf, which the attention reads for this position
                if (hh < g.Hq + g.Hkv) {
                    const float2 cs = pre;
                    const float r0 = v0 * cs.x - v1 * cs.y;
                    const float r1 = v1 * cs.x + v0 * cs.y;
                    if (hh < g.Hq) {
                        float *q = p.qbuf + (size_t)l * g.Q + (size_t)hh * g.hd;
                        if (!withhold) {
                            st_tagged(q + j, r0, tag);
                            st_tagged(q + j + half, r1, tag);
                        }
                    } else {
                        const int kvh = hh - g.Hq;
                        __half *kr = p.kc + (((size_t)l * g.Hkv + kvh) * g.max_seq + pos) * g.hd;
                        const __half k0 = __float2half_rn(r0), k1 = __float2half_rn(r1);
                        kr[kv_swz(pos, j)] = k0;
                        kr[kv_swz(pos, j + half)] = k1;
                        float *kf = p.kvf + ((size_t)l * 2 * g.Hkv + kvh) * g.hd;
                        st_tagged(kf + j, __half2float(k0), tag);
                        st_tagged(kf + j + half, __half2float(k1), tag);
                    }
                } else {
                    const int kvh = hh - g.Hq - g.Hkv;
                    __half *vr = p.vc + (((size_t)l * g.Hkv + kvh) * g.max_seq + pos) * g.hd;
                    const __half w0 = __float2half_rn(v0), w1 = __float2half_rn(v1);
                    vr[kv_swz(pos, j)] = w0;
                    vr[kv_swz(pos, j + half)] = w1;
                    float *vf = p.kvf + ((size_t)(l * 2 + 1) * g.Hkv + kvh) * g.hd;
                    st_tagged(vf + j, __half2float(w0), tag);
                    st_tagged(vf + j + half, __half2float(w1), tag);
                }
                if (hh >= g.Hq) fence_proxy_async_global();   // K/V rows are read by TMA in later steps
            } else if (s == ST_O) {
                const float v = pre.x + sum;
                st_tagged(p.xattn + (size_t)l * g.d + u, v, tag);
            } else if (s == ST_GU) {
                const float gt = sum * inv, up = partner * inv;
                float hv = gt / (1.0f + expf(-gt)) * up;
                if (moe)   // slot j's gate weights its expert's hidden units
                    hv *= __uint_as_float(*reinterpret_cast<const volatile unsigned *>(
                        &c.misc[M_GATE + 8 * (l & 1) + slot]));
                st_tagged(p.hbuf + (size_t)l * g.F + (size_t)slot * g.Fe + u, hv, tag);
            } else if (s == ST_D) {
                const float v = pre.x + sum;
                st_tagged(p.xout + (size_t)l * g.d + u, v, tag);
            } else {
                const float logit = sum * inv;
                if (p.debug_logits) p.debug_logits[(size_t)step * g.V + u] = logit;
                float keyv = logit;
                const bool all_vocab = p.temperature > 0.f && p.top_k != 1 && (p.top_k <= 0 || p.top_k >= g.V);
                if (all_vocab) keyv = logit / p.temperature + gumbel_dev(p.seed, pos, u);
                c.lmkeys[u - u0] = sel_key(keyv, u);
            }
        }
        __syncwarp();
        // q, k, v go to the attention stage by counters (their consumers are
        // the attention pieces and the TMA copies of the K/V rows); the other
        // outputs are tagged and need none
        if (s == ST_QKV) {
            __syncwarp();
            if (c.lane == 0 && !withhold) publish_range(sig_ptr(p, l, sl.qkvh), a, nu, g.hd / 2);
        }
    }
    if (c.lane == 0) {
        trace_mark_producer(c, step, tslot, TR_DONE);
        if (s == ST_LM) {
            __threadfence_block();
            *reinterpret_cast<volatile unsigned *>(&c.misc[M_LMDONE]) = (unsigned)step + 1u;
        } else if (p.sched == SCHED_GRID && !withhold) {
            fence_acq_rel_gpu();
            red_release_add(p.gbar, 1u);
        }
    }
    __syncwarp();
    return ab;
}

// The reducer warp walks the same sub-stages as the consumers.
template <bool MOE>
__device__ void reducer(const Ctx &c)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    const int n_sub = 5 * g.L + (p.mode == MODE_DECODE ? 1 : 0);
    PipeState ps;
    for (int step = 0; step < p.n_steps; ++step) {
        for (int k = 0; k < n_sub; ++k) {
            const bool lm = k == 5 * g.L;
            const int l = lm ? g.L - 1 : k / 5;
            const int sid = lm ? SID_LM : k % 5;
            if (!stage_active(p, l, sid) || sid == SID_ATTN) continue;
            if (reduce_stage<MOE>(c, ps, stage_of(sid), l, step, false)) return;
        }
    }
}

// ---------------------------------------------------------------- attention

// One split-KV piece: positions [j0, j1) of KV head gkv for the G query heads
// that share it (j0 = w0 + cpiece * per, where w0 is the first position the
// layer attends to: 0, or pos + 1 - W in a layer with a sliding window of W).
//
// The piece is a small dense contraction on the tensor cores (warp-level
// mma.sync m16n8k16, FP16 operands, FP32 accumulators).  The K/V rows sit in
// the ring as [position][hd] FP16 rows (group-swizzled, kv_swz); the ring's
// 16-position slabs go round-robin to the eight consumer warps.  Per slab a
// warp forms the scores S[h][j] = q_h . k_j for all G heads at once (the G
// query rows padded to 16, K^T as the B operand loaded with ldmatrix), runs an
// online softmax per head in FP32 (running max m, running sum l), and adds
// P V into its output, computed transposed, O^T[dim][h] = V^T P^T, so that
// the score accumulators are the B operand of the second product without
// leaving registers.  q and the probabilities p are each split into an FP16
// head and an FP16 remainder (two products each), which keeps them accurate to
// about 2^-22: the sums are FP32 like the rest of the path.  Position pos
// (written by this step's QKV stage) is staged from the cache and added by one
// warp with plain FP32 arithmetic.  The warps' states are merged pairwise
// through shared memory.
template <int HD>
__device__ __forceinline__ bool attn_piece(const Ctx &c, ConsRing &rc, int l, int step, int gkv, int cpiece, int w0,
                                        const AttnSplit &sp, bool ab)
{
    constexpr int S = ATT_CHUNK_BYTES / (4 * HD);     // positions per ring sub-block
    constexpr int SPB = S / 16;                         // 16-position slabs per sub-block
    constexpr int KS = HD / 16;                         // 16-wide k-steps over the head dimension
    constexpr int ROW = HD * 2;                         // bytes of one K or V row
    constexpr int H2 = HD / 2;
    const Params &p = *c.p;
    const Geo &g = p.g;
    const int G = g.group;                              // query heads of the group (<= 8)
    const int TT = (G + 1) / 2;                         // lanes t < TT hold output columns of real heads
    const int pos = p.pos0 + step;
    const int j0 = w0 + cpiece * sp.per;
    const int j1 = min(j0 + sp.per, pos + 1);
    const int jr = min(j1, pos);
    const float scale = 1.0f / sqrtf((float)HD);
    const int hq0 = gkv * G;
    const int gq = c.lane >> 2, tq = c.lane & 3;        // mma fragment coordinates of this lane

    // ---- shared scratch: q [G][HD] FP32, fresh K and V rows [2][HD] FP16, merge states
    float *qs = c.acta;
    __half *fresh = reinterpret_cast<__half *>(qs + G * HD);
    float *ws = qs + G * HD + HD;                       // [4][8 * TT][HD / 4] outputs, then [4][8] m and l
    float *wml = ws + (NCW / 2) * 8 * TT * (HD / 4);
    uint4 *qfr = reinterpret_cast<uint4 *>(wml + 2 * (NCW / 2) * 8);   // [KS][32 lanes] q fragments
    const bool has_fresh = pos >= j0 && pos < j1;
    // ---- this step's q of the group's heads and (the piece holding position
    // pos) the fresh K and V rows of gkv: tagged, polled in place.  The
    // monokernel prefill first waits for the heads' readiness counters (its
    // passes are not ordered by a token chain); decode needs no counter.
    if (p.sched == SCHED_FLAGS && p.mode == MODE_PREFILL) {
        const SigLayout sl = sig_layout(g);
        const unsigned target = (unsigned)H2 * (p.epoch0 + (unsigned)step + 1u);
        if (c.tid < G + 2 && !ab) {
            const int hh = c.tid < G ? hq0 + c.tid : (c.tid == G ? g.Hq + gkv : g.Hq + g.Hkv + gkv);
            ab = !wait_counter(p, sig_ptr(p, l, sl.qkvh + hh), target, 140, l, step);
        }
        if (cons_sync_or(ab)) return true;
    }
    if (!ab) {
        const unsigned tag = pass_tag(p.epoch0 + (unsigned)step);
        const float *qsrc = p.qbuf + (size_t)l * g.Q + (size_t)hq0 * HD;
        for (int i = c.tid; i < G * HD / 4 && !ab; i += NCT) {
            float4 v;
            if (!poll_f4(p, qsrc + 4 * i, tag, v, 140, l, step)) ab = true;
            reinterpret_cast<float4 *>(qs)[i] = v;
        }
        if (has_fresh) {
            // K then V as FP16 in plain order (the values are FP16 already:
            // the conversion is exact and clears the tag)
            for (int i = c.tid; i < HD / 2 && !ab; i += NCT) {
                const int r = (4 * i) / HD, e = (4 * i) % HD;   // r 0: K, 1: V
                const float *src = p.kvf + ((size_t)(l * 2 + r) * g.Hkv + gkv) * HD + e;
                float4 v;
                if (!poll_f4(p, src, tag, v, 142, l, step)) ab = true;
                __half2 *dst = reinterpret_cast<__half2 *>(fresh) + (r * HD + e) / 2;
                dst[0] = __floats2half2_rn(v.x, v.y);
                dst[1] = __floats2half2_rn(v.z, v.w);
            }
        }
    }
    if (cons_sync_or(ab)) return true;

    // ---- q fragments (A operand, rows = heads, padded to 16), one table for
    // all warps: entry [k][lane] = (a0 head, a2 head, a0 remainder, a2
    // remainder) of row lane/4, columns 16k + 2(lane%4) (+1) and 16k + 8 +
    // 2(lane%4) (+1); rows >= G and rows 8..15 are zero
    for (int i = c.tid; i < KS * 32; i += NCT) {
        const int k = i / 32, gi = (i % 32) >> 2, ti = i & 3;
        uint4 fr = make_uint4(0u, 0u, 0u, 0u);
        if (gi < G) {
            const float *qr = qs + gi * HD + 16 * k + 2 * ti;
            __half h0, r0, h1, r1;
            split_h(qr[0], h0, r0);
            split_h(qr[1], h1, r1);
            fr.x = pack_h2(h0, h1);
            fr.z = pack_h2(r0, r1);
            split_h(qr[8], h0, r0);
            split_h(qr[9], h1, r1);
            fr.y = pack_h2(h0, h1);
            fr.w = pack_h2(r0, r1);
        }
        qfr[i] = fr;
    }
    if (cons_sync_or(ab)) return true;
    const uint32_t qfa = smem_u32(qfr) + (uint32_t)c.lane * 16u;
    // ---- per-warp state, per lane: running max and (partial) sum of heads
    // 2tq and 2tq+1, and O^T tiles o[d][0..3] = O[2tq][16d+gq],
    // O[2tq+1][16d+gq], O[2tq][16d+gq+8], O[2tq+1][16d+gq+8]
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    float o[KS][4];
#pragma unroll
    for (int d = 0; d < KS; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    // ldmatrix row addresses (lanes 8i..8i+7 address matrix i, row = lane & 7):
    // K as the A operand of S^T = K Q^T: matrices (positions 0-7 | 8-15) x
    // (group 2k | 2k+1) in the order a0..a3; V for V^T: (positions 0-7 | 8-15)
    // outer, (group 2d | 2d+1) inner, transposed
    const int krw = (c.lane & 7) + (((c.lane >> 3) & 1) << 3), kgp = c.lane >> 4;
    const int vrw = (c.lane & 7) + ((c.lane >> 4) << 3), vgp = (c.lane >> 3) & 1;

    // one 16-position slab: positions q0 .. q0+nv-1 (nv in 1..16), rows at kb/vb
    auto slab = [&](uint32_t kb, uint32_t vb, int q0, int nv) {
        const int kpos = q0 + krw, vpos = q0 + vrw;     // positions of the rows this lane addresses
        const uint32_t krow = kb + (uint32_t)krw * ROW, vrow = vb + (uint32_t)vrw * ROW;
        // S^T[pos][head]: sc0 = (gq, 2tq), sc1 = (gq, 2tq+1), sc2 = (gq+8, 2tq), sc3 = (gq+8, 2tq+1)
        float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            unsigned a[4];
            ldsm_x4(a, krow + (uint32_t)((((2 * k + kgp) ^ (kpos & 7))) << 4));
            const uint4 qb = lds_u4(qfa + (uint32_t)k * 512u);
            mma16816(st, a[0], a[1], a[2], a[3], qb.x, qb.y);
            mma16816(st, a[0], a[1], a[2], a[3], qb.z, qb.w);
        }
        float sc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[i] = st[i] * scale;
        if (gq >= nv) sc[0] = sc[1] = -INFINITY;
        if (gq + 8 >= nv) sc[2] = sc[3] = -INFINITY;
        // maxima of heads 2tq, 2tq+1 over the slab (lanes of equal tq)
        float xa = fmaxf(sc[0], sc[2]), xb = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int sh = 4; sh <= 16; sh <<= 1) {
            xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, sh));
            xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, sh));
        }
        const float na = fmaxf(ma, xa), nb2 = fmaxf(mb, xb);   // finite: nv >= 1
        const float ca = __expf(ma - na), cb = __expf(mb - nb2);   // 0 while the max is -inf
        ma = na;
        mb = nb2;
        const float p0 = __expf(sc[0] - na), p1 = __expf(sc[1] - nb2), p2 = __expf(sc[2] - na), p3 = __expf(sc[3] - nb2);
        la = fmaf(la, ca, p0 + p2);
        lb = fmaf(lb, cb, p1 + p3);
        // P^T as the B operand of O^T = V^T P^T: the 8x8 blocks (positions 0-7 |
        // 8-15) x heads, transposed in registers
        __half h0, r0, h1, r1, h2, r2, h3, r3;
        split_h(p0, h0, r0);
        split_h(p1, h1, r1);
        split_h(p2, h2, r2);
        split_h(p3, h3, r3);
        const unsigned pb0h = movm_t(pack_h2(h0, h1)), pb1h = movm_t(pack_h2(h2, h3));
        const unsigned pb0r = movm_t(pack_h2(r0, r1)), pb1r = movm_t(pack_h2(r2, r3));
        // V^T as the A operand (rows = dims, columns = positions), positions past nv zeroed
        const unsigned keep0 = (2 * tq < nv ? 0x0000FFFFu : 0u) | (2 * tq + 1 < nv ? 0xFFFF0000u : 0u);
        const unsigned keep1 = (8 + 2 * tq < nv ? 0x0000FFFFu : 0u) | (9 + 2 * tq < nv ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int d = 0; d < KS; ++d) {
            o[d][0] *= ca;
            o[d][1] *= cb;
            o[d][2] *= ca;
            o[d][3] *= cb;
            unsigned a[4];
            ldsm_x4_t(a, vrow + (uint32_t)((((2 * d + vgp) ^ (vpos & 7))) << 4));
            // matrices (transposed): 0 = positions 0-7 x dims 16d..16d+7, 1 = positions 0-7 x dims
            // 16d+8.., 2 = positions 8-15 x dims 16d.., 3 = positions 8-15 x dims 16d+8.. --
            // exactly the A fragments a0..a3 of V^T (rows gq / gq+8, columns 2tq / 8+2tq)
            const unsigned va0 = a[0] & keep0, va1 = a[1] & keep0, va2 = a[2] & keep1, va3 = a[3] & keep1;
            mma16816(o[d], va0, va1, va2, va3, pb0h, pb1h);
            mma16816(o[d], va0, va1, va2, va3, pb0r, pb1r);
        }
    };

    const int nring = jr > j0 ? ceil_div(jr - j0, S) : 0;
    int nslab = 0;
    for (int blk = 0; blk < nring; ++blk) {
        const int nb = min(S, jr - (j0 + blk * S));
        const uint8_t *ch = rc.acquire(c, 4u * (unsigned)nb * HD, ab);
        if (ab) break;
        const uint32_t kb = smem_u32(ch), vb = kb + (uint32_t)nb * ROW;
        const int q0 = j0 + blk * S;
#pragma unroll 1
        for (int sl = 0; sl < SPB; ++sl) {
            const int nv = min(16, nb - 16 * sl);
            if (nv > 0) {
                if ((nslab + sl) % NCW == c.warp)
                    slab(kb + (uint32_t)(16 * sl) * ROW, vb + (uint32_t)(16 * sl) * ROW, q0 + 16 * sl, nv);
            }
        }
        nslab += ceil_div(nb, 16);
        rc.release(c);
    }
    if (!ab && has_fresh && nslab % NCW == c.warp) {
        // position pos: scores q_h . k for all heads (lane: HD/32 elements), then one online-softmax step
        constexpr int EL = HD / 32;
        float kf[EL], vlo[KS], vhi[KS];
#pragma unroll
        for (int e = 0; e < EL; ++e) kf[e] = __half2float(fresh[c.lane * EL + e]);
#pragma unroll
        for (int d = 0; d < KS; ++d) {
            vlo[d] = __half2float(fresh[HD + 16 * d + gq]);
            vhi[d] = __half2float(fresh[HD + 16 * d + gq + 8]);
        }
        float sa = 0.f, sb = 0.f;                        // scores of heads 2tq, 2tq+1 (0 for padding heads)
        for (int h = 0; h < G; ++h) {
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < EL; ++e) dot = fmaf(qs[h * HD + c.lane * EL + e], kf[e], dot);
            dot = warp_sum(dot) * scale;
            if (h == 2 * tq) sa = dot;
            if (h == 2 * tq + 1) sb = dot;
        }
        const float na = fmaxf(ma, sa), nb2 = fmaxf(mb, sb);
        const float ca = __expf(ma - na), cb = __expf(mb - nb2);
        const float pa = __expf(sa - na), pb = __expf(sb - nb2);
        la = fmaf(la, ca, gq == 0 ? pa : 0.f);
        lb = fmaf(lb, cb, gq == 0 ? pb : 0.f);
        ma = na;
        mb = nb2;
#pragma unroll
        for (int d = 0; d < KS; ++d) {
            o[d][0] = fmaf(o[d][0], ca, pa * vlo[d]);
            o[d][1] = fmaf(o[d][1], cb, pb * vlo[d]);
            o[d][2] = fmaf(o[d][2], ca, pa * vhi[d]);
            o[d][3] = fmaf(o[d][3], cb, pb * vhi[d]);
        }
    }
    trace_mark(c, step, 5 * l + 1, TR_X1);
#pragma unroll
    for (int sh = 4; sh <= 16; sh <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, sh);
        lb += __shfl_xor_sync(0xffffffffu, lb, sh);
    }

    // ---- merge the warps pairwise (warp w + st into warp w, st = 4, 2, 1):
    // state = (m, l) of heads 2tq, 2tq+1 and the O^T tiles of the lanes t < TT
    for (int st = NCW / 2; st >= 1; st >>= 1) {
        const bool sender = c.warp >= st && c.warp < 2 * st, taker = c.warp < st;
        const int slot = sender ? c.warp - st : c.warp;
        if (sender) {
            if (tq < TT) {
                float *dst = ws + ((size_t)slot * 8 * TT + gq * TT + tq) * (HD / 4);
#pragma unroll
                for (int d = 0; d < KS; ++d)
                    reinterpret_cast<float4 *>(dst)[d] = make_float4(o[d][0], o[d][1], o[d][2], o[d][3]);
            }
            if (gq == 0) {
                wml[slot * 16 + 2 * tq] = ma;
                wml[slot * 16 + 2 * tq + 1] = mb;
                wml[slot * 16 + 8 + 2 * tq] = la;
                wml[slot * 16 + 9 + 2 * tq] = lb;
            }
        }
        if (cons_sync_or(ab)) return true;
        if (taker) {
            const float moa = wml[slot * 16 + 2 * tq], mob = wml[slot * 16 + 2 * tq + 1];
            const float loa = wml[slot * 16 + 8 + 2 * tq], lob = wml[slot * 16 + 9 + 2 * tq];
            const float Ma = fmaxf(ma, moa), Mb = fmaxf(mb, mob);
            const float fa0 = (ma == -INFINITY) ? 0.f : __expf(ma - Ma), fb0 = (moa == -INFINITY) ? 0.f : __expf(moa - Ma);
            const float fa1 = (mb == -INFINITY) ? 0.f : __expf(mb - Mb), fb1 = (mob == -INFINITY) ? 0.f : __expf(mob - Mb);
            if (tq < TT) {
                const float *src = ws + ((size_t)slot * 8 * TT + gq * TT + tq) * (HD / 4);
#pragma unroll
                for (int d = 0; d < KS; ++d) {
                    const float4 v = reinterpret_cast<const float4 *>(src)[d];
                    o[d][0] = fmaf(o[d][0], fa0, v.x * fb0);
                    o[d][1] = fmaf(o[d][1], fa1, v.y * fb1);
                    o[d][2] = fmaf(o[d][2], fa0, v.z * fb0);
                    o[d][3] = fmaf(o[d][3], fa1, v.w * fb1);
                }
            }
            la = fmaf(la, fa0, loa * fb0);
            lb = fmaf(lb, fa1, lob * fb1);
            ma = Ma;
            mb = Mb;
        }
        if (cons_sync_or(ab)) return true;
    }
    // ---- warp 0 holds the piece: (o, m, l) per head into the partials
    if (c.warp == 0) {
        float *base = p.apart + (((size_t)l * g.Hq + hq0) * p.max_split + cpiece) * (HD + 2);
        const size_t hstride = (size_t)p.max_split * (HD + 2);
        if (2 * tq < G) {
            float *ha = base + (size_t)(2 * tq) * hstride;
#pragma unroll
            for (int d = 0; d < KS; ++d) {
                ha[16 * d + gq] = o[d][0];
                ha[16 * d + gq + 8] = o[d][2];
            }
            if (gq == 0) {
                ha[HD] = ma;
                ha[HD + 1] = la;
            }
        }
        if (2 * tq + 1 < G) {
            float *hb = base + (size_t)(2 * tq + 1) * hstride;
#pragma unroll
            for (int d = 0; d < KS; ++d) {
                hb[16 * d + gq] = o[d][1];
                hb[16 * d + gq + 8] = o[d][3];
            }
            if (gq == 0) {
                hb[HD] = mb;
                hb[HD + 1] = lb;
            }
        }
    }
    if (cons_sync_or(ab)) return true;
    if (c.tid == 0) {
        const unsigned old = atom_add_acq_rel(p.attn_done + ((size_t)l * g.Hkv + gkv) * CNT_STRIDE, 1u);
        c.misc[M_FLAG] = (old == (unsigned)sp.n_split - 1u) ? 1u : 0u;
    }
    if (cons_sync_or(ab)) return true;
    trace_mark(c, step, 5 * l + 1, TR_X2);
    if (c.misc[M_FLAG] == 0u) return false;

    // ---- this CTA holds the last piece of KV head gkv: combine all pieces,
    // attn = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c, M = max_c m_c.
    // The (m, l) table goes to shared memory while each thread loads o of 16
    // pieces for two output elements at once: one L2 round trip per 16 pieces.
    if (c.tid == 0) st_relaxed(p.attn_done + ((size_t)l * g.Hkv + gkv) * CNT_STRIDE, 0u);
    constexpr int PB = 16;
    const int ns = sp.n_split;
    const float *base = p.apart + ((size_t)l * g.Hq + hq0) * p.max_split * (HD + 2);
    float2 *mls = reinterpret_cast<float2 *>(c.acta);  // [G][ns] (m, l); the scratch is free after the merge
    const int n_el = G * HD;
    const int n_it = ceil_div(n_el, 2 * NCT);           // the same for every thread
    float o0[PB], o1[PB];
    auto load_batch = [&](int it, int c0) {
        const int e0 = c.tid + it * 2 * NCT, e1 = e0 + NCT;
        const float *s0 = base + (size_t)(e0 / HD) * p.max_split * (HD + 2) + e0 % HD;
        const float *s1 = base + (size_t)(e1 / HD) * p.max_split * (HD + 2) + e1 % HD;
#pragma unroll
        for (int k = 0; k < PB; ++k) {
            if (c0 + k < ns && e0 < n_el) o0[k] = __ldcg(s0 + (size_t)(c0 + k) * (HD + 2));
            if (c0 + k < ns && e1 < n_el) o1[k] = __ldcg(s1 + (size_t)(c0 + k) * (HD + 2));
        }
    };
    load_batch(0, 0);                                   // in flight while the table loads
    for (int idx = c.tid; idx < G * ns; idx += NCT) {
        const int h = idx / ns, cc = idx % ns;
        mls[idx] = __ldcg(reinterpret_cast<const float2 *>(base + ((size_t)h * p.max_split + cc) * (HD + 2) + HD));
    }
    if (cons_sync_or(ab)) return true;
    for (int it = 0; it < n_it; ++it) {
        const int e0 = c.tid + it * 2 * NCT, e1 = e0 + NCT;
        const int h0 = min(e0, n_el - 1) / HD, h1 = min(e1, n_el - 1) / HD;
        float M0 = -INFINITY, n0 = 0.f, d0 = 0.f, M1 = -INFINITY, n1 = 0.f, d1 = 0.f;
        for (int c0 = 0; c0 < ns; c0 += PB) {
            if (it > 0 || c0 > 0) load_batch(it, c0);
            float B0 = M0, B1 = M1;
#pragma unroll
            for (int k = 0; k < PB; ++k) {
                if (c0 + k < ns) {
                    B0 = fmaxf(B0, mls[h0 * ns + c0 + k].x);
                    B1 = fmaxf(B1, mls[h1 * ns + c0 + k].x);
                }
            }
            const float a0 = __expf(M0 - B0), a1 = __expf(M1 - B1);
            n0 *= a0; d0 *= a0; n1 *= a1; d1 *= a1;
#pragma unroll
            for (int k = 0; k < PB; ++k) {
                if (c0 + k < ns) {
                    const float2 q0 = mls[h0 * ns + c0 + k], q1 = mls[h1 * ns + c0 + k];
                    const float w0 = __expf(q0.x - B0), w1 = __expf(q1.x - B1);
                    if (e0 < n_el) { n0 = fmaf(w0, o0[k], n0); d0 = fmaf(w0, q0.y, d0); }
                    if (e1 < n_el) { n1 = fmaf(w1, o1[k], n1); d1 = fmaf(w1, q1.y, d1); }
                }
            }
            M0 = B0;
            M1 = B1;
        }
        const unsigned tg = pass_tag(p.epoch0 + (unsigned)step);
        if (e0 < n_el) st_tagged(p.attn + (size_t)l * g.Q + (size_t)hq0 * HD + e0, n0 / d0, tg);
        if (e1 < n_el) st_tagged(p.attn + (size_t)l * g.Q + (size_t)hq0 * HD + e1, n1 / d1, tg);
    }
    // the outputs are tagged (no count); the barrier keeps the (m, l) table in
    // the scratch until every thread has read it
    return cons_sync_or(ab);
}

// ---------------------------------------------------------------- LM head selection

// k-th largest of n distinct 64-bit keys (k >= 1, k <= n), by an 8-pass
// most-significant-digit radix select over the consumer threads.  `keys`
// may be shared or global memory; stride/width describe a [rows][stride]
// array of which the first `width` entries of each row are used.
__device__ __forceinline__ bool radix_select(const Ctx &c, const unsigned long long *keys, int rows, int stride, int width, int k,
                             bool global_mem, unsigned long long &tau, bool ab)
{
    unsigned long long prefix = 0ull, mask = 0ull;
    unsigned remain = (unsigned)k;
    const int n = rows * width;
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int i = c.tid; i < 256; i += NCT) c.hist[i] = 0u;
        if (cons_sync_or(ab)) return true;
        for (int i = c.tid; i < n; i += NCT) {
            const int r = i / width, j = i % width;
            const unsigned long long key = global_mem ? __ldcg(keys + (size_t)r * stride + j) : keys[(size_t)r * stride + j];
            if ((key & mask) == prefix) atomicAdd(&c.hist[(key >> shift) & 255u], 1u);
        }
        if (cons_sync_or(ab)) return true;
        if (c.warp == 0) {
            // lane L covers bins 255-8L .. 248-8L (high to low)
            unsigned cnt[8];
            unsigned tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cnt[q] = c.hist[255 - 8 * c.lane - q];
                tot += cnt[q];
            }
            unsigned incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned v = __shfl_up_sync(0xffffffffu, incl, o);
                if (c.lane >= o) incl += v;
            }
            const unsigned excl = incl - tot;
            if (excl < remain && remain <= incl) {
                unsigned cum = excl;
                for (int q = 0; q < 8; ++q) {
                    if (cum + cnt[q] >= remain) {
                        c.misc[M_DIGIT] = 255u - 8u * c.lane - q;
                        c.misc[M_REMAIN] = remain - cum;
                        break;
                    }
                    cum += cnt[q];
                }
            }
        }
        if (cons_sync_or(ab)) return true;
        const unsigned digit = c.misc[M_DIGIT];
        remain = c.misc[M_REMAIN];
        prefix |= (unsigned long long)digit << shift;
        mask |= 0xFFull << shift;
    }
    tau = prefix;
    return false;
}

// Token choice after the LM-head tiles of this CTA have put their selection
// keys in shared memory: per-CTA candidates, then the last CTA to arrive picks
// the token and publishes it.
__device__ __forceinline__ bool stage_lm_sample(const Ctx &c, int step, bool ab)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    const CtaPlan &pl = *c.plan;
    const int pos = p.pos0 + step;
    if (cons_sync_or(ab)) return true;

    const bool greedy = !(p.temperature > 0.f) || p.top_k == 1;
    const bool all_vocab = !greedy && (p.top_k <= 0 || p.top_k >= g.V);
    const int nloc = pl.u1[ST_LM] - pl.u0[ST_LM];
    unsigned long long *part = p.lm_part + (size_t)c.b * MAX_TOPK;
    if (greedy || all_vocab) {
        unsigned long long best = 0ull;
        for (int i = c.tid; i < nloc; i += NCT) best = c.lmkeys[i] > best ? c.lmkeys[i] : best;
        best = warp_max_u64(best);
        if (c.lane == 0) reinterpret_cast<unsigned long long *>(c.red)[c.warp] = best;
        if (cons_sync_or(ab)) return true;
        if (c.tid == 0) {
            unsigned long long m = 0ull;
            for (int w = 0; w < NCW; ++w) {
                unsigned long long v = reinterpret_cast<unsigned long long *>(c.red)[w];
                m = v > m ? v : m;
            }
            part[0] = m;
        }
    } else {
        const int k = p.top_k;
        const int kloc = min(k, nloc);
        unsigned long long tau;
        if (radix_select(c, c.lmkeys, 1, nloc, nloc, kloc, false, tau, ab)) return true;
        if (c.tid == 0) c.misc[M_FLAG] = 0u;
        if (cons_sync_or(ab)) return true;
        for (int i = c.tid; i < nloc; i += NCT) {
            const unsigned long long key = c.lmkeys[i];
            if (key >= tau) part[atomicAdd(&c.misc[M_FLAG], 1u)] = key;
        }
        for (int j = kloc + c.tid; j < k; j += NCT) part[j] = 0ull;
    }
    if (cons_sync_or(ab)) return true;
    if (c.tid == 0) {
        fence_acq_rel_gpu();
        const unsigned old = atom_add_acq_rel(p.lm_done, 1u);
        c.misc[M_FLAG] = (old == (unsigned)p.P - 1u) ? 1u : 0u;
    }
    if (cons_sync_or(ab)) return true;
    const bool last = c.misc[M_FLAG] != 0u;
    if (last) {
        if (c.tid == 0) st_relaxed(p.lm_done, 0u);
        unsigned long long best = 0ull;
        if (greedy || all_vocab) {
            for (int i = c.tid; i < p.P; i += NCT) {
                const unsigned long long v = __ldcg(p.lm_part + (size_t)i * MAX_TOPK);
                best = v > best ? v : best;
            }
        } else {
            const int k = p.top_k;
            unsigned long long tau;
            if (radix_select(c, p.lm_part, p.P, MAX_TOPK, k, k, true, tau, ab)) return true;
            for (int i = c.tid; i < p.P * k; i += NCT) {
                const unsigned long long key = __ldcg(p.lm_part + (size_t)(i / k) * MAX_TOPK + (i % k));
                if (key >= tau) {
                    const int idx = sel_key_index(key);
                    const float score = sel_key_value(key) / p.temperature + gumbel_dev(p.seed, pos, idx);
                    const unsigned long long sk = sel_key(score, idx);
                    best = sk > best ? sk : best;
                }
            }
        }
        best = warp_max_u64(best);
        if (c.lane == 0) reinterpret_cast<unsigned long long *>(c.red)[c.warp] = best;
        if (cons_sync_or(ab)) return true;
        if (c.tid == 0) {
            unsigned long long m = 0ull;
            for (int w = 0; w < NCW; ++w) {
                unsigned long long v = reinterpret_cast<unsigned long long *>(c.red)[w];
                m = v > m ? v : m;
            }
            const int tok = sel_key_index(m);
            p.out_tokens[step] = tok;
            const int next = p.force_tokens ? __ldg(p.force_tokens + step) : tok;
            p.tok_seq[step] = next;
            if (step == p.n_steps - 1) p.tok_buf[0] = next;
            fence_acq_rel_gpu();
            red_release_add(p.tok_cnt, 1u);
        }
    }
    if (p.sched == SCHED_GRID) {
        if (cons_sync_or(ab)) return true;
        if (c.tid == 0) red_release_add(p.gbar, 1u);
    }
    return cons_sync_or(ab);
}

// ---------------------------------------------------------------- consumer

// The consumer walks the sub-stages of every step -- for each layer QKV,
// attention, O, gate/up, down, then the LM head -- through ONE loop body, so
// that each stage's code exists once in the kernel and stays warm in the
// instruction cache from one layer to the next.
template <int FMT, bool MOE>
__device__ void consumer(const Ctx &c)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    ConsRing rc;
    PipeState ps;
    const bool ab = false;
    const bool decode = p.mode == MODE_DECODE;
    const int n_sub = 5 * g.L + (decode ? 1 : 0);
    // A GEMV stage has no consumer barrier, so a warp without chunks in it
    // may run ahead to the next point where the consumer warps meet (a named
    // barrier, which cannot time out).  A warp whose GEMV stage gives up (the
    // abort flag is then set) therefore does not exit at once: it walks on to
    // that next meeting point and joins it with the abort bit, so that every
    // warp leaves there, or reaches the end if none is left.
    bool failed = false;
    for (int step = 0; step < p.n_steps; ++step) {
        for (int k = 0; k < n_sub; ++k) {
            const bool lm = k == 5 * g.L;
            const int l = lm ? g.L - 1 : k / 5;
            const int sid = lm ? SID_LM : k % 5;
            if (!stage_active(p, l, sid)) continue;
            if (failed) {
                unsigned idx;
                const bool meets = sid == SID_ATTN || lm || (MOE && sid == SID_GU) ||
                                   (p.sched == SCHED_GRID && grid_barrier_before(p, step, l, sid, idx));
                if (meets) {
                    (void)cons_sync_or(true);
                    return;
                }
                continue;
            }
            trace_mark(c, step, k, TR_ENTER);
            if (sid == SID_ATTN) {
                // barrier schedule: the whole QKV stage, everywhere (the flag
                // schedule waits per unit inside attn_piece)
                unsigned idx;
                if (p.sched == SCHED_GRID && grid_barrier_before(p, step, l, sid, idx)) {
                    if (cons_wait(c, p.gbar, (idx + 1u) * (unsigned)p.P, 2, l, step, ab)) return;
                }
                trace_mark(c, step, k, TR_READY);
                const int pos = p.pos0 + step;
                const int w0 = attn_first_pos(pos, c.win[l]);    // first attended position
                const AttnSplit sp = attn_split(pos + 1 - w0, p.P, g.Hkv, p.attn_min_len);
                const int U = g.Hkv * sp.n_split;
                for (int u = attn_unit_first(c.b, l, U, p.P); u < U; u += p.P) {
                    const int gkv = u / sp.n_split, cp = u % sp.n_split;
                    const bool stop = (g.hd == 128) ? attn_piece<128>(c, rc, l, step, gkv, cp, w0, sp, ab)
                                                    : attn_piece<64>(c, rc, l, step, gkv, cp, w0, sp, ab);
                    if (stop) return;
                }
                // every CTA's consumers meet once per attention stage, with or
                // without pieces (a meeting point of the walk after a failure)
                if (cons_sync_or(ab)) return;
                if (p.sched == SCHED_GRID && cons_grid_arrive(c, ab)) return;
                trace_mark(c, step, k, TR_DONE);
            } else {
                // barrier schedule: the whole previous sub-stage, everywhere
                unsigned idx;
                if (p.sched == SCHED_GRID && grid_barrier_before(p, step, l, sid, idx)) {
                    if (cons_wait(c, p.gbar, (idx + 1u) * (unsigned)p.P, 3, l, step, ab)) return;
                }
                if (MOE && sid == SID_GU && route_experts(c, ps, l, step, ab)) return;
                if (stage_gemv<FMT, MOE>(c, rc, ps, stage_of(sid), l, step, ab)) {
                    if (lm) {   // the other warps meet after the LM head's tiles
                        (void)cons_sync_or(true);
                        return;
                    }
                    failed = true;
                    continue;
                }
                if (lm) {
                    // the reducer's keys of every LM-head tile of this CTA
                    bool fail = false;
                    if (c.tid == 0) fail = !wait_smem_ge(p, &c.misc[M_LMDONE], (unsigned)step + 1u, 112, l, step);
                    if (cons_sync_or(fail)) return;
                    if (stage_lm_sample(c, step, ab)) return;
                }
            }
        }
    }
}

// ---------------------------------------------------------------- caller-layout weight rows

struct RepackSrc {
    const uint8_t *wq, *wk, *wv, *wo, *wg, *wu, *wd, *head;
};

// Row `part` of unit `unit` of stage s, layer l, in the caller's row-major
// weights, or for MXFP4 in the chunk-interleaved copy lf_create builds: a row
// of `cols` columns takes cols / 256 * g.crb bytes either way.
__device__ const uint8_t *src_row(const Geo &g, const RepackSrc &w, int s, int l, int unit, int part, int e = 0)
{
    // gate/up/down of a mixture of experts: [L][E][rows][cols]; dense: E = 1, Fe = F
    const size_t rd = (size_t)(g.d / KC) * g.crb, rq = (size_t)(g.Q / KC) * g.crb, rf = (size_t)(g.Fe / KC) * g.crb;
    const size_t le = (size_t)l * n_expert_parts(g) + e;
    switch (s) {
    case ST_QKV: {
        const int half = g.hd / 2;
        const int hh = unit / half, j = unit % half;
        const int r = hh * g.hd + j + part * half;  // row of the fused [q; k; v] space
        if (r < g.Q) return w.wq + ((size_t)l * g.Q + r) * rd;
        if (r < g.Q + g.KV) return w.wk + ((size_t)l * g.KV + (r - g.Q)) * rd;
        return w.wv + ((size_t)l * g.KV + (r - g.Q - g.KV)) * rd;
    }
    case ST_O: return w.wo + ((size_t)l * g.d + unit) * rq;
    case ST_GU: return (part ? w.wu : w.wg) + (le * g.Fe + unit) * rd;
    case ST_D: return w.wd + (le * g.d + unit) * rf;
    default: return w.head + (size_t)unit * rd;
    }
}

// ---------------------------------------------------------------- producer

// Mixture of experts: the stream holds the gate/up and down rows of every
// expert of the layer, expert after expert (gate/up: the CTA's tiles with
// d/256 chunks each; down: the CTA's tiles with Fe/256 chunks each), and only
// the active experts' parts are sent, in the consumers' order: gate/up slot by
// slot; down tile by tile, each tile's chunks slot by slot.
__device__ __forceinline__ bool produce_moe(const Ctx &c, ProdRing &pr, int s, int l)
{
    // slot j's expert, chosen by the consumers for this layer
    auto sel = [&c, l](int j) {
        return (int)*reinterpret_cast<const volatile unsigned *>(&c.misc[M_SEL + 8 * (l & 1) + j]);
    };
    const Params &p = *c.p;
    const Geo &g = p.g;
    const CtaPlan &pl = *c.plan;
    const StageGeom sg = stage_geom(g, s);
    const int u0 = pl.u0[s], n = pl.u1[s] - u0;
    const int nt = tiles_of(n, sg.rows_per_unit);
    const uint8_t *base = p.wstream + pl.base + (unsigned long long)l * pl.layer_bytes + pl.stage_off[s];
    const int nch = (s == ST_GU ? g.d : g.Fe) / KC;
    const unsigned long long part = (unsigned long long)n * sg.rows_per_unit * nch * (unsigned long long)g.crb;
    if (s == ST_GU) {
        for (int j = 0; j < g.topk; ++j) {
            const uint8_t *src = base + (unsigned long long)sel(j) * part;
            for (int t = 0; t < nt; ++t) {
                int a, bnd;
                tile_range(u0, n, nt, t, a, bnd);
                const unsigned bytes = (unsigned)((bnd - a) * sg.rows_per_unit) * (unsigned)g.crb;
                for (int k = 0; k < nch; ++k) {
                    if (!pr.emit(c, src, bytes)) return false;
                    src += bytes;
                }
            }
        }
        return true;
    }
    unsigned long long toff = 0;   // offset of tile t inside an expert's part
    for (int t = 0; t < nt; ++t) {
        int a, bnd;
        tile_range(u0, n, nt, t, a, bnd);
        const unsigned bytes = (unsigned)((bnd - a) * sg.rows_per_unit) * (unsigned)g.crb;
        for (int j = 0; j < g.topk; ++j) {
            const uint8_t *src = base + (unsigned long long)sel(j) * part + toff;
            for (int k = 0; k < nch; ++k) {
                if (!pr.emit(c, src, bytes)) return false;
                src += bytes;
            }
        }
        toff += (unsigned long long)bytes * nch;
    }
    return true;
}

__device__ __forceinline__ bool produce_tiles(const Ctx &c, ProdRing &pr, int s, int l, int step)
{
    const Params &p = *c.p;
    const CtaPlan &pl = *c.plan;
    const StageGeom sg = stage_geom(p.g, s);
    const int u0 = pl.u0[s], n = pl.u1[s] - u0;
    const int nt = tiles_of(n, sg.rows_per_unit);
    const uint8_t *src = p.wstream + pl.base +
                         (s == ST_LM ? pl.lm_off : (unsigned long long)l * pl.layer_bytes + pl.stage_off[s]);
    for (int t = 0; t < nt; ++t) {
        int a, bnd;
        tile_range(u0, n, nt, t, a, bnd);
        const int R = (bnd - a) * sg.rows_per_unit;
        const unsigned bytes = (unsigned)R * (unsigned)chunk_row_bytes(p.g);
        const int nch = sg.K / KC;
        for (int k = 0; k < nch; ++k) {
            if (!pr.emit(c, src, bytes)) return false;
            src += bytes;
        }
    }
    return true;
}

// Producer variant used by lf_generate_noalloc, whose weights stay in the
// caller's row-major layout: each chunk (R rows x 256 columns) is gathered
// with one 512-byte bulk copy per row into the same ring layout.
__device__ __forceinline__ bool produce_tiles_direct(const Ctx &c, ProdRing &pr, const RepackSrc &w, int s, int l, int step)
{
    const Params &p = *c.p;
    const CtaPlan &pl = *c.plan;
    const StageGeom sg = stage_geom(p.g, s);
    const int u0 = pl.u0[s], n = pl.u1[s] - u0;
    const int nt = tiles_of(n, sg.rows_per_unit);
    for (int t = 0; t < nt; ++t) {
        int a, bnd;
        tile_range(u0, n, nt, t, a, bnd);
        const int nu = bnd - a;
        const int R = nu * sg.rows_per_unit;
        const unsigned row_bytes = (unsigned)chunk_row_bytes(p.g);
        const int nch = sg.K / KC;
        for (int k = 0; k < nch; ++k) {
            const int o = pr.reserve(c, (unsigned)R * row_bytes);
            if (o < 0) return false;
            uint64_t *bar = &c.full[pr.n % TICKETS];
            mbar_arrive_expect_tx(bar, (unsigned)R * row_bytes);
            for (int r = 0; r < R; ++r) {
                const int unit = a + (sg.rows_per_unit == 2 ? r % nu : r);
                const int part = sg.rows_per_unit == 2 ? r / nu : 0;
                const uint8_t *src = src_row(p.g, w, s, l, unit, part) + (size_t)k * row_bytes;
                bulk_g2s(c.ring + o + r * row_bytes, src, row_bytes, bar, pr.pol);
            }
            ++pr.n;
        }
    }
    return true;
}

template <bool kDirect, bool MOE>
__device__ void producer(const Ctx &c, const RepackSrc *w)
{
    const Params &p = *c.p;
    const Geo &g = p.g;
    ProdRing pr;
    int step_now = 0;
    auto tiles = [&step_now](const Ctx &cc, ProdRing &r, const RepackSrc *ws, int s, int l) {
        if constexpr (kDirect) return produce_tiles_direct(cc, r, *ws, s, l, step_now);
        else return produce_tiles(cc, r, s, l, step_now);
    };
    pr.pol = policy_evict_first();
    // K/V rows are read again by the next step: they keep the normal L2
    // priority while the cache the call reads fits in L2, and are streamed
    // evict-first like the weights once it cannot stay resident anyway
    {
        const long long ctx_end = (long long)p.pos0 + p.n_steps;
        const long long kv_read = ctx_end * (long long)p.g.L * p.g.KV * 4;   // K + V, FP16, every layer
        pr.pol_kv = kv_read > (128ll << 20) ? policy_evict_first() : policy_evict_normal();
    }
    bool ok = true;
    const int n_sub = 5 * g.L + (p.mode == MODE_DECODE ? 1 : 0);
    unsigned routes = 0;   // expert choices consumed (mixture of experts)
    for (int step = 0; step < p.n_steps && ok; ++step) {
        step_now = step;
        const unsigned e = p.epoch0 + (unsigned)step;
        const int pos = p.pos0 + step;
        for (int k = 0; k < n_sub && ok; ++k) {
            const bool lm = k == 5 * g.L;
            const int l = lm ? 0 : k / 5;
            const int sid = lm ? SID_LM : k % 5;
            if (!stage_active(p, l, sid)) continue;
            trace_mark_producer(c, step, k, TR_P0);
            if (sid != SID_ATTN) {
                const int st = sid == SID_QKV ? ST_QKV : sid == SID_O ? ST_O : sid == SID_GU ? ST_GU
                                                       : sid == SID_D ? ST_D : ST_LM;
                if (MOE && (st == ST_GU || st == ST_D)) {
                    if (st == ST_GU) {
                        // the consumers' expert choice for this layer
                        ok = wait_smem_ge(p, &c.misc[M_ROUTE], routes + 1u, 104, l, step);
                        ++routes;
                    }
                    if (ok) ok = produce_moe(c, pr, st, l);
                    trace_mark_producer(c, step, k, TR_P1);
                    continue;
                }
                ok = tiles(c, pr, w, st, l);
                trace_mark_producer(c, step, k, TR_P1);
                continue;
            }
            const int w0 = attn_first_pos(pos, c.win[l]);
            const AttnSplit sp = attn_split(pos + 1 - w0, p.P, g.Hkv, p.attn_min_len);
            const int U = g.Hkv * sp.n_split;
            const int S = attn_sub_positions(g.hd);
            for (int u = attn_unit_first(c.b, l, U, p.P); u < U && ok; u += p.P) {
                const int gkv = u / sp.n_split, cp = u % sp.n_split;
                const int j0 = w0 + cp * sp.per;
                const int jr = min(min(j0 + sp.per, pos + 1), pos);
                if (jr > j0 && step > 0) {
                    // position pos - 1 of step > 0 was written by the previous
                    // step's QKV stage: its key and value heads of gkv
                    const SigLayout sl = sig_layout(g);
                    const unsigned prev = (unsigned)(g.hd / 2) * e;
                    ok = wait_counter(p, sig_ptr(p, l, sl.qkvh + g.Hq + gkv), prev, 102, l, step) &&
                         wait_counter(p, sig_ptr(p, l, sl.qkvh + g.Hq + g.Hkv + gkv), prev, 103, l, step);
                    fence_proxy_async_global();
                }
                const size_t base = (((size_t)l * g.Hkv + gkv) * g.max_seq) * g.hd;
                for (int jb = j0; jb < jr && ok; jb += S) {
                    const int nb = min(S, jr - jb);
                    const unsigned hb = (unsigned)nb * g.hd * 2u;
                    ok = pr.emit2(c, p.kc + base + (size_t)jb * g.hd, p.vc + base + (size_t)jb * g.hd, hb);
                }
            }
            trace_mark_producer(c, step, k, TR_P1);
        }
    }
    if (!ok) pr.drain(c);
}

// ---------------------------------------------------------------- kernel

template <bool kDirect, int FMT, bool MOE = false>
__device__ __forceinline__ void monokernel_body(const Params &p, const RepackSrc *w)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const SmemLayout L = smem_layout(p.ring_bytes, p.a_floats, p.lm_rows_max, p.g.L);
    Ctx c;
    c.p = &p;
    c.ring = smem + L.ring;
    c.acta = reinterpret_cast<float *>(smem + L.acta);
    c.lmkeys = reinterpret_cast<unsigned long long *>(smem + L.lmkeys);
    c.res = reinterpret_cast<float *>(smem + L.res);
    c.full = reinterpret_cast<uint64_t *>(smem + L.full);
    c.empty = reinterpret_cast<uint64_t *>(smem + L.empty);
    c.chunk_end = reinterpret_cast<unsigned long long *>(smem + L.chunk_end);
    c.red = reinterpret_cast<float *>(smem + L.red);
    c.hist = reinterpret_cast<unsigned *>(smem + L.hist);
    c.misc = reinterpret_cast<unsigned *>(smem + L.misc);
    {
        int *win = reinterpret_cast<int *>(smem + L.win);
        for (int i = threadIdx.x; i < p.g.L; i += blockDim.x) win[i] = p.win ? p.win[i] : 0;
        c.win = win;
    }
    CtaPlan *plan_s = reinterpret_cast<CtaPlan *>(smem + L.plan);
    c.plan = plan_s;
    c.b = blockIdx.x;
    c.tid = threadIdx.x;
    c.warp = threadIdx.x >> 5;
    c.lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < TICKETS; ++i) {
            mbar_init(&c.full[i], 1);
            mbar_init(&c.empty[i], NCW);
        }
        mbar_fence_init();
        *plan_s = p.plans[blockIdx.x];
        for (int i = 0; i < 64; ++i) c.misc[i] = 0u;
    }
    __syncthreads();
    if (c.warp == W_PROD) {
        if (c.lane == 0) producer<kDirect, MOE>(c, w);
        return;
    }
    if (c.warp == W_RED) {
        reducer<MOE>(c);
        return;
    }
    consumer<FMT, MOE>(c);
}

__global__ void __launch_bounds__(NTHREADS, 1) lf_monokernel(const __grid_constant__ Params p)
{
    monokernel_body<false, FMT_FP16>(p, nullptr);
}

// The same kernel for FP8 (E4M3) projection weights.
__global__ void __launch_bounds__(NTHREADS, 1) lf_monokernel_fp8(const __grid_constant__ Params p)
{
    monokernel_body<false, FMT_FP8>(p, nullptr);
}

// The same kernel for a mixture-of-experts FFN (FP16 weights).
__global__ void __launch_bounds__(NTHREADS, 1) lf_monokernel_moe(const __grid_constant__ Params p)
{
    monokernel_body<false, FMT_FP16, true>(p, nullptr);
}

// The same kernel for MXFP4 projection weights.
__global__ void __launch_bounds__(NTHREADS, 1) lf_monokernel_mxfp4(const __grid_constant__ Params p)
{
    monokernel_body<false, FMT_MXFP4>(p, nullptr);
}

// Same kernel, streaming weights from the caller's layout (lf_generate_noalloc).
__global__ void __launch_bounds__(NTHREADS, 1) lf_monokernel_direct(const __grid_constant__ Params p,
                                                                   const __grid_constant__ RepackSrc w)
{
    monokernel_body<true, FMT_FP16>(p, &w);
}

// ---------------------------------------------------------------- repack

// Copy the caller's weights into the per-CTA streams, using the same tile
// enumeration as the producer.  One block per CTA stream.
__global__ void lf_repack_kernel(Geo g, const CtaPlan *plans, RepackSrc w, uint8_t *dst)
{
    const CtaPlan pl = plans[blockIdx.x];
    for (int l = 0; l < g.L + 1; ++l) {
        const int s_lo = (l < g.L) ? ST_QKV : ST_LM;
        const int s_hi = (l < g.L) ? ST_D : ST_LM;
        for (int s = s_lo; s <= s_hi; ++s) {
            const StageGeom sg = stage_geom(g, s);
            const int u0 = pl.u0[s], n = pl.u1[s] - u0;
            const int nt = tiles_of(n, sg.rows_per_unit);
            uint8_t *out = dst + pl.base + (s == ST_LM ? pl.lm_off : (unsigned long long)l * pl.layer_bytes + pl.stage_off[s]);
            // gate/up and down: every expert's rows, expert after expert
            const int nexp = (s == ST_GU || s == ST_D) ? n_expert_parts(g) : 1;
            const int nch = (s == ST_D ? g.Fe : sg.K) / KC;
            for (int e = 0; e < nexp; ++e) {
                for (int t = 0; t < nt; ++t) {
                    int a, bnd;
                    tile_range(u0, n, nt, t, a, bnd);
                    const int nu = bnd - a;
                    const int R = nu * sg.rows_per_unit;
                    const int v16 = chunk_row_bytes(g) / 16;   // 16-byte words of one row of a chunk
                    for (int k = 0; k < nch; ++k) {
                        // chunk: R rows x 256 columns, stored row r -> (unit a + r % nu, part r / nu)
                        for (int q = threadIdx.x; q < R * v16; q += blockDim.x) {
                            const int r = q / v16, rem = q % v16;
                            const int unit = a + (sg.rows_per_unit == 2 ? r % nu : r);
                            const int part = sg.rows_per_unit == 2 ? r / nu : 0;
                            const uint4 *srow =
                                reinterpret_cast<const uint4 *>(src_row(g, w, s, l < g.L ? l : 0, unit, part, e));
                            reinterpret_cast<uint4 *>(out)[q] = srow[(size_t)k * v16 + rem];
                        }
                        out += (size_t)R * chunk_row_bytes(g);
                    }
                }
            }
        }
    }
}

// MXFP4: one matrix ([rows, cols] elements: codes [rows, cols/2], E8M0 scales
// [rows, cols/32]) rewritten as rows of cols/256 groups of 144 bytes (128
// code bytes, 8 scale bytes, 8 zero bytes), the row layout the repack copies
// into the streams.  One thread per 16 output bytes.
__global__ void lf_mxfp4_interleave_kernel(const uint8_t *codes, const uint8_t *scales, size_t rows, int cols,
                                           uint8_t *out)
{
    const int ng = cols / KC;
    const size_t n16 = rows * (size_t)ng * 9;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
        const size_t rg = i / 9;
        const int q = (int)(i % 9);
        const size_t r = rg / ng;
        const int gidx = (int)(rg % ng);
        uint4 v;
        if (q < 8) {
            v = *reinterpret_cast<const uint4 *>(codes + r * (size_t)(cols / 2) + (size_t)gidx * 128 + q * 16);
        } else {
            const uint8_t *sp = scales + r * (size_t)(cols / 32) + (size_t)gidx * 8;
            uint8_t b[16] = {};
            for (int k = 0; k < 8; ++k) b[k] = sp[k];
            v = *reinterpret_cast<const uint4 *>(b);
        }
        *reinterpret_cast<uint4 *>(out + i * 16) = v;
    }
}

}  // namespace lfk

// ---------------------------------------------------------------- launch hooks used by lf_api.cu

extern "C" cudaError_t lfk_set_smem(int smem_bytes)
{
    cudaError_t e = cudaFuncSetAttribute(lfk::lf_monokernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lfk::lf_monokernel_fp8, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lfk::lf_monokernel_mxfp4, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lfk::lf_monokernel_moe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    return e;
}

extern "C" cudaError_t lfk_launch_monokernel(const lfk::Params *p, int smem_bytes, cudaStream_t stream,
                                             int cooperative)
{
    void *args[] = {const_cast<lfk::Params *>(p)};
    const void *fn = p->g.fmt == lfk::FMT_FP8     ? (const void *)lfk::lf_monokernel_fp8
                     : p->g.fmt == lfk::FMT_MXFP4 ? (const void *)lfk::lf_monokernel_mxfp4
                     : p->g.E > 0                 ? (const void *)lfk::lf_monokernel_moe
                                                  : (const void *)lfk::lf_monokernel;
    if (cooperative)
        return cudaLaunchCooperativeKernel(fn, dim3(p->P), dim3(lfk::NTHREADS), args, (size_t)smem_bytes, stream);
    return cudaLaunchKernel(fn, dim3(p->P), dim3(lfk::NTHREADS), args, (size_t)smem_bytes, stream);
}

extern "C" cudaError_t lfk_occupancy(int smem_bytes, int *blocks_per_sm)
{
    cudaError_t e = lfk_set_smem(smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, lfk::lf_monokernel, lfk::NTHREADS,
                                                        (size_t)smem_bytes);
}

extern "C" unsigned lfk_smem_bytes(int ring_bytes, int a_floats, int lm_rows_max, int L)
{
    return lfk::smem_layout(ring_bytes, a_floats, lm_rows_max, L).total;
}

extern "C" cudaError_t lfk_launch_repack(lfk::Geo g, int P, const lfk::CtaPlan *plans, const void *wq, const void *wk,
                                         const void *wv, const void *wo, const void *wg, const void *wu,
                                         const void *wd, const void *head, void *dst, cudaStream_t stream)
{
    lfk::RepackSrc w{(const uint8_t *)wq, (const uint8_t *)wk, (const uint8_t *)wv, (const uint8_t *)wo,
                     (const uint8_t *)wg, (const uint8_t *)wu, (const uint8_t *)wd, (const uint8_t *)head};
    lfk::lf_repack_kernel<<<P, 256, 0, stream>>>(g, plans, w, (uint8_t *)dst);
    return cudaGetLastError();
}

extern "C" cudaError_t lfk_set_smem_direct(int smem_bytes)
{
    return cudaFuncSetAttribute(lfk::lf_monokernel_direct, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

extern "C" cudaError_t lfk_launch_monokernel_direct(const lfk::Params *p, const void *wq, const void *wk,
                                                    const void *wv, const void *wo, const void *wg, const void *wu,
                                                    const void *wd, const void *head, int smem_bytes,
                                                    cudaStream_t stream)
{
    lfk::RepackSrc w{(const uint8_t *)wq, (const uint8_t *)wk, (const uint8_t *)wv, (const uint8_t *)wo,
                     (const uint8_t *)wg, (const uint8_t *)wu, (const uint8_t *)wd, (const uint8_t *)head};
    void *args[] = {const_cast<lfk::Params *>(p), &w};
    return cudaLaunchCooperativeKernel((const void *)lfk::lf_monokernel_direct, dim3(p->P), dim3(lfk::NTHREADS),
                                       args, (size_t)smem_bytes, stream);
}

extern "C" cudaError_t lfk_launch_mxfp4_interleave(const void *codes, const void *scales, size_t rows, int cols,
                                                   void *out, cudaStream_t stream)
{
    const size_t n16 = rows * (size_t)(cols / lfk::KC) * 9;
    const int grid = (int)std::min<size_t>((n16 + 255) / 256, 8192);
    lfk::lf_mxfp4_interleave_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(codes),
                                                              static_cast<const uint8_t *>(scales), rows, cols,
                                                              static_cast<uint8_t *>(out));
    return cudaGetLastError();
}
