// lf_internal.cuh -- shapes, static work partition and the kernel parameter
// block, shared by the host runtime (lf_api.cu) and the kernels (lf_kernel.cu).
//
// The partition is fixed when a handle is created, in the spirit of the
// "compile-time work partition" of the KOG monokernel (shivam2003.com,
// "Compile-time work partition (no scheduler)"): every CTA of the persistent
// grid knows, for every stage, which weight rows it owns and where their
// bytes sit in its own contiguous weight stream.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace lfk {

constexpr int KC = 256;               // weight columns per column group (32 lanes x 8 FP16)
constexpr int KC_BYTES = KC * 2;      // bytes of one row of one column group
constexpr int TILE_ROWS = 32;         // rows of one GEMV tile (4 per consumer warp)
constexpr int NCW = 8;                // consumer warps
constexpr int NCT = NCW * 32;         // consumer threads
// Warp roles after the consumers: the producer streams weights into the ring,
// the reducer sums tile partials and runs the stage epilogues.
constexpr int W_PROD = NCW, W_RED = NCW + 1;
constexpr int NTHREADS = NCT + 64;
constexpr int TICKETS = 32;           // ring slots in flight (mbarrier pairs)
constexpr int ATT_CHUNK_BYTES = 32768;// K + V bytes of one attention sub-block
constexpr int MAX_TOPK = 64;
constexpr int MAX_GROUP = 8;          // query heads per KV head
constexpr int CNT_STRIDE = 32;        // uint32 words between counters (one 128-byte line each)
constexpr int SIG_STRIDE = 8;         // uint32 words between slice readiness counters (one 32-byte sector)
constexpr int PART_BUFS = 8;          // rotating per-tile partial-sum buffers of a GEMV stage
constexpr int PART_STRIDE = TILE_ROWS + 1;  // per warp: 32 row sums + the sum of squares of x
constexpr int MAX_SLICES = 64;        // 256-element slices of one activation vector (length <= 16384)

enum Stage { ST_QKV = 0, ST_O = 1, ST_GU = 2, ST_D = 3, ST_LM = 4, N_GEMV = 5 };
enum Mode { MODE_PREFILL = 0, MODE_DECODE = 1 };
enum Sched { SCHED_FLAGS = 0, SCHED_GRID = 1, SCHED_MULTI = 2 };
enum StatusCode { STATUS_OK = 0, STATUS_BAD_TOKEN = 1, STATUS_TIMEOUT = 6 };

// Formats of the projection weights in the per-CTA streams.  One row of one
// column group (256 weights) of a chunk takes fmt_crb(fmt) bytes: FP16 512; FP8
// E4M3 256 (per-row FP32 scales applied in the epilogue); MXFP4 144 = 128 bytes
// of packed E2M1 codes (element 2i in the low nibble of byte i), the E8M0
// scales of the group's eight 32-element blocks, and 8 bytes of padding that
// keep every chunk a multiple of 16 bytes for the bulk copies.
enum WeightFmt { FMT_FP16 = 0, FMT_FP8 = 1, FMT_MXFP4 = 2 };
__host__ __device__ constexpr int fmt_crb(int fmt) { return fmt == FMT_FP16 ? 512 : fmt == FMT_FP8 ? 256 : 144; }

struct Geo {
    int L, d, Hq, Hkv, hd, F, V, Q, KV, group, max_seq;
    int fmt;            // WeightFmt of the eight projections
    int crb;            // fmt_crb(fmt)
    // FFN: E = 0 dense (topk = 1, Fe = F); E > 0: mixture of E experts of
    // Fe hidden units each, topk active per token, and F = topk * Fe, the
    // length of the hidden vector h (the active experts' units, slot by slot)
    int E, topk, Fe;
};
constexpr int MAX_EXPERTS = 64;          // router logits: two per lane of one warp
constexpr int MAX_ACTIVE_EXPERTS = 8;    // expert slots in shared memory per layer
// Experts whose weights a stage's stream holds per layer (1 for a dense FFN).
__host__ __device__ inline int n_expert_parts(const Geo &g) { return g.E > 0 ? g.E : 1; }
// Bytes of one row of one column group (256 weights) of a projection in the stream.
__host__ __device__ inline int chunk_row_bytes(const Geo &g) { return g.crb; }

struct StageGeom {
    int units;          // work units of the stage
    int rows_per_unit;  // 2 for RoPE pairs (QKV) and gate/up pairs (GU), else 1
    int K;              // columns (input length)
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// QKV units are row pairs (i, i + hd/2) of one head of the fused [q; k; v]
// row space, so that RoPE's rotate-half partners land in the same tile.
// GU units are (gate row r, up row r) pairs, so that SiLU(gate) * up is
// formed where both rows were computed.
__host__ __device__ inline StageGeom stage_geom(const Geo &g, int s)
{
    switch (s) {
    case ST_QKV: return {(g.Q + 2 * g.KV) / 2, 2, g.d};
    case ST_O: return {g.d, 1, g.Q};
    case ST_GU: return {g.Fe, 2, g.d};     // per slot (active expert)
    case ST_D: return {g.d, 1, g.F};
    default: return {g.V, 1, g.d};
    }
}

__host__ __device__ inline int units_per_tile(int rpu) { return TILE_ROWS / rpu; }
__host__ __device__ inline int tiles_of(int n_units, int rpu)
{
    return n_units <= 0 ? 0 : ceil_div(n_units, units_per_tile(rpu));
}
// Units [a, b) of tile t when n units starting at u0 are split into nt near-equal tiles.
__host__ __device__ inline void tile_range(int u0, int n, int nt, int t, int &a, int &b)
{
    a = u0 + (int)((long long)t * n / nt);
    b = u0 + (int)((long long)(t + 1) * n / nt);
}
// First unit owned by CTA b when U units are split contiguously over P CTAs.
__host__ __device__ inline int cta_unit_start(int U, int P, int b) { return (int)((long long)b * U / P); }

// Split-KV attention: the ctx positions of each KV head are cut into n_split
// contiguous pieces of `per` positions (the last may be shorter; none is
// empty), at most P / Hkv pieces per head, at least min_len positions each.
struct AttnSplit { int n_split, per; };
__host__ __device__ inline AttnSplit attn_split(int ctx, int P, int Hkv, int min_len)
{
    int maxs = P / Hkv;
    if (maxs < 1) maxs = 1;
    int n0 = ceil_div(ctx, min_len);
    if (n0 > maxs) n0 = maxs;
    if (n0 < 1) n0 = 1;
    int per = ceil_div(ctx, n0);
    return {ceil_div(ctx, per), per};
}
// Attention unit u of layer l (u in [0, U), U = Hkv * n_split) runs on CTA (u + l*U) mod P.
__host__ __device__ inline int attn_unit_first(int b, int l, int U, int P)
{
    long long r = ((long long)b - (long long)l * U) % P;
    if (r < 0) r += P;
    return (int)r;
}
__host__ __device__ inline int attn_sub_positions(int hd) { return ATT_CHUNK_BYTES / (4 * hd); }
// KV-cache row layout: element j of the row of position p sits at
// kv_swz(p, j): its 16-byte group (8 FP16 values) j/8 is XOR-ed with p mod 8,
// so that 8 consecutive positions' groups j/8 fall in 8 different shared-
// memory bank quads once a block of rows is copied into the ring, and the
// tensor-core fragment loads (ldmatrix, 8 rows x 16 bytes) are conflict-free.
__host__ __device__ inline int kv_swz(int p, int j) { return ((((j >> 3) ^ (p & 7)) << 3) | (j & 7)); }
// First position the query at `pos` attends to in a layer of window W
// (W > 0: the W most recent positions, itself included; 0: the whole cache).
__host__ __device__ inline int attn_first_pos(int pos, int W) { return (W > 0 && pos + 1 > W) ? pos + 1 - W : 0; }

// Per-CTA plan: unit ranges of the five GEMV stages and the byte offsets of
// this CTA's weight stream.  The stream of CTA b is laid out as
//   [layer 0: QKV tiles | O tiles | GU tiles | D tiles] ... [layer L-1: ...] [LM-head tiles]
// and each tile as K/256 chunks of (R rows x 256 columns), row-major inside
// a chunk.
// Readiness counters of one layer, cumulative over forward passes (cleared by
// lf_create and lf_reset).  Every slot is a uint32 SIG_STRIDE words apart.
//   qkvh[h]   RoPE pair-units of head h written by the QKV stage (query heads,
//             then key heads, then value heads): hd/2 per pass
// Only the attention stage's inputs go by counters (their readers include
// TMA copies of the K/V rows, which cannot check values); the GEMV stages'
// inputs are tagged activations (Params::attn, xattn, hbuf, xout).
struct SigLayout {
    int qkvh, per_layer;
};
__host__ __device__ inline SigLayout sig_layout(const Geo &g)
{
    SigLayout s;
    s.qkvh = 0;
    s.per_layer = g.Hq + 2 * g.Hkv;
    return s;
}

// Attention scratch (floats) in shared memory: q of the group [G][hd],
// the staged fresh K and V rows (hd floats' worth of FP16), the states that
// half of the warps hand to the other half in one round of the merge (4 warps
// x 8 x ceil(G/2) lanes x hd/4 output values, then [4][8] running maxima and
// sums) and the table of q's tensor-core fragments (hd/16 x 32 lanes x 4
// words); or, in the combine, the (m, l) table [G][max_split].
__host__ __device__ inline int attn_scratch_floats(const Geo &g, int max_split)
{
    const int piece = g.group * g.hd + g.hd + (NCW / 2) * 8 * ((g.group + 1) / 2) * (g.hd / 4) + 2 * (NCW / 2) * 8 +
                      (g.hd / 16) * 32 * 4;
    const int combine = 2 * g.group * max_split;
    return piece > combine ? piece : combine;
}

// The shared-memory scratch (Params::a_floats): the attention's, or with a
// mixture of experts at least the FFN input the router stages (d floats);
// rounded to whole float4s.
__host__ __device__ inline int scratch_floats(const Geo &g, int max_split)
{
    int a = attn_scratch_floats(g, max_split);
    if (g.E > 0 && g.d > a) a = g.d;
    return (a + 3) / 4 * 4;
}

struct CtaPlan {
    int u0[N_GEMV], u1[N_GEMV];
    unsigned long long base;          // byte offset of the stream in the repacked buffer
    unsigned long long layer_bytes;   // bytes of one layer's four stages
    unsigned long long stage_off[4];  // offset of each stage inside a layer
    unsigned long long lm_off;        // offset of the LM-head tiles from base
};

struct Params {
    Geo g;
    int P;                       // persistent CTAs
    float eps;
    const CtaPlan *plans;
    const uint8_t *wstream;      // repacked FP16 weights
    const __half *embed, *attn_norm, *ffn_norm, *final_norm;
    __half *kc, *vc;             // [L][Hkv][max_seq][hd]
    const float2 *rope;          // [max_seq][hd/2] (cos, sin)
    float *qbuf;                 // [L][Q]   RoPE'd queries (tagged, see below)
    // Tagged activations: the lowest mantissa bit of every value holds the
    // parity of the forward pass that wrote it (pass e: (e & 1) ^ 1, so the
    // zeros these buffers start from match no pass 0 value).  Their readers
    // take them straight from global memory, polling until every value they
    // need carries the current pass's parity: no counter, no writer fence.
    // Every pass rewrites every value, and every value is read by the same
    // threads in every pass of a launch: having seen pass e - 1's value, a
    // thread cannot see an older one (coherence of one location), so a value
    // of pass e - 2 is never taken for one of pass e; a launch's first pass
    // is ordered after the previous launch.
    float *attn;                 // [L][Q]   attention output
    float *xattn;                // [L][d]   residual after attention
    float *hbuf;                 // [L][F]   SiLU(gate) * up
    float *xout;                 // [L][d]   residual after FFN
    float *kvf;                  // [L][2][Hkv][hd] this pass's K and V rows (tagged FP32 copies of
                                 // the FP16 values the cache holds) for the attention's fresh position
    float *apart;                // [L][Hq][max_split][hd + 2]  (o[hd], m, l) per piece
    const int *win;              // [L] attention window per layer in positions (0: whole cache), or null
    // FP8 weights (g.fmt == FMT_FP8): per-row FP32 scales of wq, wk, wv, wo, w_gate,
    // w_up, w_down, lm_head in the caller's row order ([L][rows], [V])
    const float *wsc[8];
    const __half *router;        // [L][E][d] FP16 router rows (mixture of experts), or null
    int max_split;
    unsigned *sig;               // [L][sig_layout().per_layer] readiness counters
    unsigned *attn_done;         // [L][Hkv] pieces of each KV head that have published
    unsigned *lm_done, *tok_cnt, *gbar;
    unsigned long long *lm_part; // [P][MAX_TOPK] 64-bit selection keys
    int *tok_buf;                // [1] pending token
    int *tok_seq;                // [max_seq] token fed to step i + 1
    unsigned *status;            // first error code (0 = none)
    unsigned *abort_flag;
    // per call
    int mode;
    int n_steps;
    int pos0;                    // position of step 0's input token
    int has_pending;             // prefill: step 0 consumes the pending token first
    const int *prompt;
    int *out_tokens;
    float *debug_logits;
    const int *force_tokens;
    float temperature;
    int top_k;                   // 0 = whole vocabulary
    unsigned long long seed;
    unsigned epoch0;             // forward passes since the counters were cleared
    unsigned tok_base;           // sampled tokens since the counters were cleared
    unsigned gbar_base;          // grid barriers since the counters were cleared
    long long timeout_ns;
    int fault_step;
    int ring_bytes;
    int a_floats;                // attention scratch (attn_scratch_floats, rounded to 4)
    int lm_rows_max;
    int attn_min_len;
    int sched;
    // multi-kernel schedule: run only stage `only_stage` of layer `only_layer` of step 0
    int only_layer, only_stage;
    // optional %globaltimer trace: [step][slot][cta][4] (slot = 5 * layer + stage, LM = 5 * L)
    unsigned long long *trace;
    int trace_steps;
};

// Trace stamps per (step, slot, CTA), %globaltimer ns.  GEMV stages: consumer
// warp 0 entered the stage, the first chunk's input values were read, the
// reducer stored the last tile, consumer warp 0 finished its last chunk (X1),
// the last tile's partials were complete (X2); TR_LOADED is not used.
// Attention: entered, inputs ready, K/V positions done (X1), piece partial
// published (X2), stage done.  The producer adds when it issued the first and
// the last chunk of the sub-stage (P0, P1).  TR_WAITS is a count: weight
// chunks of the stage that had not landed when warp 0 first asked for them.
enum TraceStamp { TR_ENTER = 0, TR_READY = 1, TR_LOADED = 2, TR_DONE = 3, TR_X1 = 4, TR_X2 = 5, TR_P0 = 6, TR_P1 = 7,
                  TR_WAITS = 8, TR_N = 9 };
__host__ __device__ inline int trace_slots(int L) { return 5 * L + 1; }

}  // namespace lfk
