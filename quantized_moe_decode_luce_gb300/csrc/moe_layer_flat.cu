// moe_layer_flat.cu -- the one-launch routed-MoE FFN layer for layers whose
// q8_1 rows of h do not fit shared memory (speculative verify: five tokens,
// H = 4096, I = 2048, tens of experts): router select + weights, the q8_1
// quantization of the input, the expert grouping, the gate/up pair with its
// SwiGLU, the q8_1 quantization of h, the down product and the masked
// route-weighted combine with the shared expert.  luce_moe_layer (in
// moe_layer.cu) sends such layers here.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving".  The arithmetic of every step is the one of the
// separate operations ([PR826] commits "fused DS4.1 decode kernels", "RDNA4
// Q8_0 gate/up pair" and "fused routed combine and q8_1 inputs for the hybrid
// owners"): the same per-lane block order and warp sums, so h, hq and y equal
// those of luce_moe_glu_pair + luce_moe_down_combine bit for bit.  The launch
// structure is our own:
//
//  * Cost balance.  Every CTA takes an equal slice of the shared expert's I
//    rows and an equal cost share of the flat list of the routed experts'
//    rows (a row of an expert with c columns costs GU_ROW_COST + c); and an
//    equal cost share of the down items of the flat list of (virtual expert,
//    output row) (DN_ROW_COST + c each).
//  * One producer warp streams the CTA's stages in order through a ring of
//    shared-memory slots with cp.async.bulk (evict-first L2 policy).  The copy
//    engine of an SM keeps about four bulk copies in flight (measured on
//    GB300: four copies of 16 KB reach ~7 TB/s, of 4 KB ~2.3 TB/s), so every
//    copy is at least 16 KB where the rows allow: a gate/up part is RU gate
//    rows and RU up rows with RU rbg >= 16 KB; part j goes to consumer group
//    j mod NG, each of the group's RU warps taking one row pair for every
//    column of the part's expert.
//  * h goes to global memory; after a device-wide barrier each CTA quantizes
//    an equal share of the q8_1 blocks of h; after a second one each CTA
//    copies the hq rows of the (at most a few) experts its down items touch
//    into shared memory, computes y for its items and stores it in the
//    caller's workspace; after a third, each CTA combines an equal share of
//    the output rows in slot order.
//  * The device-wide barrier: the grid is launched cooperatively (every CTA
//    resident), one 64-bit monotonic arrival count in caller memory (no
//    reset), bounded waits (LUCE_FAULT_TIMEOUT, LUCE_FAULT_DESYNC).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_layer_flat)

namespace {

using namespace luce;

constexpr int CW = 16;               // consumer warps
constexpr int CTHREADS = CW * 32;
constexpr int THREADS = CTHREADS + 32; // + the producer warp
constexpr int BAR_CONS = 1;          // named barrier of the consumer threads
constexpr int BAR_SEL = 2;           // the ranking (every thread)
constexpr int BAR_TABLES = 3;        // one token: the tables, tables warp -> consumers
constexpr int BAR_PLAN = 4;          // several tokens: the tables, producer warp -> warps 0 and 1
constexpr int RT0 = CTHREADS / 2;    // threads below quantize x; warp RT0 / 32 builds the tables
constexpr int MAX_T = 8;
constexpr int MAX_R = 64;  // T * k
constexpr int MAX_E = 256; // experts (selection bit masks of MAX_E / 32 words)
constexpr int MAX_V = MAX_R + 1;
constexpr int RB_MAX = 64; // down rows per row block (y buffer rows)
// Cost of a gate/up row pair and of a down row with c columns, in units of
// one column's dot products: streaming the row through the ring costs
// about as much as that many dots (measured on the verify layer: the time
// per CTA follows these weights).
constexpr int GU_ROW_COST = 6;
constexpr int DN_ROW_COST = 3;
constexpr unsigned FULL = 0xffffffffu;

struct LayerArgs {
    const float *logits, *bias, *x;
    const uint8_t *wg, *wu, *wd;    // routed: [E][I][rbg], [E][I][rbg], [E][H][rbd]
    const uint8_t *wsg, *wsu, *wsd; // shared expert or null
    int T, E, k, H, I;
    float clamp;
    int32_t *ids;
    float *weights;
    uint32_t *xq; // [T][nbH] q8_1 blocks (9 words)
    int32_t *counts, *offsets, *routes;
    float *h;     // [T*k+T][I]
    uint32_t *hq; // [T*k+T][nbI] q8_1 blocks
    float *out;   // [T][H]
    unsigned long long *sync; // arrivals of every barrier (monotonic), first word of the workspace
    int nbH, nbI, rbg, rbd;
    int RU;          // rows of a gate/up part = warps of a consumer group
    int NG;          // consumer groups that take gate/up parts (<= CW / RU)
    int stage_bytes; // one ring slot
    int NS;          // ring slots
    int SR;          // down rows per stage
    int RB;          // rows of a full row block (<= RB_MAX)
    int flat;        // down items split flat over (expert, row), y through ws_y, combine after a third barrier
    float *ws_y;     // [T*k+T][H] y values (flat), in the caller's workspace
    int xstride;     // words of an activation row in shared memory
    int hstride;     // words of an hq row in shared memory
    int hq_rows;     // hq rows held in shared memory
    int evict_first;
};

// Device-wide barrier number `nth` (1, 2) of this launch among the n CTAs of a
// cooperative grid, called by one thread per CTA after a CTA barrier that
// follows the CTA's stores (the release of the arrival covers them).  `count`
// (64-bit, never wraps) only grows: every barrier of every launch adds n, and
// all launches that share it have the same n.  c0, read after the previous
// launch has completed, is a multiple of n; this barrier ends at c0 + nth n.
// Returns false if the wait ran out (never in a correct run).
__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ bool grid_barrier(unsigned long long *count, unsigned n, unsigned long long c0, int nth)
{
    const unsigned long long target = (c0 / n + (unsigned long long)nth) * n;
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(count) : "memory");
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; i++) {
        if (ld_acquire_gpu_u64(count) >= target)
            return true;
        __nanosleep(32); // 152 pollers of one word: leave the L2 slice room for the arrivals
        if ((i & 15u) == 0u && global_timer_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// Warp sums of two values per lane: lanes 0..15 end with the sum of a, lanes
// 16..31 with the sum of b.  Each addition pairs the same lanes as warp_sum.
__device__ __forceinline__ float reduce2(float a, float b, int lane)
{
    const bool h16 = lane & 16;
    float v = (h16 ? b : a) + __shfl_xor_sync(FULL, h16 ? a : b, 16);
    v += __shfl_xor_sync(FULL, v, 8);
    v += __shfl_xor_sync(FULL, v, 4);
    v += __shfl_xor_sync(FULL, v, 2);
    v += __shfl_xor_sync(FULL, v, 1);
    return v;
}

// q8_1 rule for one block held by 4 lanes (lane 4i + j holds x[8j .. 8j+7] of
// block i of the warp's 8): the same arithmetic as quantize_q8_1_warp (the
// maximum and the integer sum do not depend on the order).  The words go to
// out_words (and to gout when it is not null).
__device__ __forceinline__ void quantize_q8_1_quad(const float (&v)[8], bool valid, uint32_t *out_words,
                                                   uint32_t *gout, int qj)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++)
        amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float dd = amax == 0.0f ? 1.0f : d; // an all-zero block: codes 0, no division by 0
    int q[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        q[i] = (int)roundf(__fdiv_rn(v[i], dd));
        sum += q[i];
    }
    sum += __shfl_xor_sync(FULL, sum, 1);
    sum += __shfl_xor_sync(FULL, sum, 2);
    if (!valid)
        return;
    const uint32_t w0 = (uint32_t)(q[0] & 0xff) | (uint32_t)(q[1] & 0xff) << 8 | (uint32_t)(q[2] & 0xff) << 16 |
                        (uint32_t)(q[3] & 0xff) << 24;
    const uint32_t w1 = (uint32_t)(q[4] & 0xff) | (uint32_t)(q[5] & 0xff) << 8 | (uint32_t)(q[6] & 0xff) << 16 |
                        (uint32_t)(q[7] & 0xff) << 24;
    uint32_t w00 = 0;
    if (qj == 0) {
        const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
        const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sum)));
        w00 = d16 | (s16 << 16);
    }
    if (out_words) {
        out_words[1 + 2 * qj] = w0;
        out_words[2 + 2 * qj] = w1;
        if (qj == 0)
            out_words[0] = w00;
    }
    if (gout) {
        gout[1 + 2 * qj] = w0;
        gout[2 + 2 * qj] = w1;
        if (qj == 0)
            gout[0] = w00;
    }
}

__device__ __forceinline__ void load8(const float *p, float (&v)[8], bool cg)
{
    const float4 *p4 = reinterpret_cast<const float4 *>(p);
    const float4 a = cg ? __ldcg(p4) : p4[0];
    const float4 b = cg ? __ldcg(p4 + 1) : p4[1];
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
    v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

// Word offset of q8_1 block b in an activation row staged in shared memory:
// with the ROWMAP_PAIRS mapping, blocks b and b + 32 (read by one load
// instruction) sit 16 banks apart.
__device__ __forceinline__ int xblock_word(int b, int pad) { return b * Q8_1_WORDS + pad * (b >> 5); }

// This CTA's work.  Gate/up parts: shared ones first (rows [s0, s1) of the
// shared expert in pieces aligned to RU), then routed ones (flat rows
// [q0, q1) of the routed virtual experts, v-major, in pieces aligned to RU;
// RU divides I, so no piece crosses an expert).  Down: rows [n0, n0 + nrows)
// in nrb row blocks of rpb rows (the last one rlast); a row block's NV * rows
// items (v-major) are cut into stages of SR items.
struct LayerPlan {
    int NVr, NV;
    int s0, s1, ps0, NPs;
    int q0, q1, pr0;
    int NPr, NPglu;
    int n0, nrows, nrb, rpb, rlast, spr, slast, NPd;
    int it0, it1; // flat down items of this CTA
    int SR;       // down items per stage (whole experts' row runs where they fit)
};

// Bounded wait that parks the thread in hardware until the phase completes
// (or a 10 us suspend hint runs out), so a waiter wakes as soon as its data
// or slot is there instead of after a back-off sleep.
__device__ __forceinline__ bool mbar_wait_parked(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 10000))
            return true;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// The items where CTAs b and b + 1 of nb start in a list of nv runs of M
// items, an item of run v costing w(v) > 0: the first item of the first run
// whose cost prefix exceeds b / nb of the total cost, offset into that run
// by the rest of that share over the run's item cost.  Warp-collective
// (every lane gets the results): the run costs are summed and scanned across
// the lanes, in exact 64-bit integers, so the results are the ones the plain
// sequential walk over the runs gives.
template <typename Wf>
__device__ void split_at_warp(int nv, unsigned M, Wf w, int b, int nb, int lane, int &r0, int &r1)
{
    // r0 for CTA b, r1 for CTA b + 1 (the same walk, two targets)
    unsigned long long tot = 0;
    #pragma unroll 1
    for (int v0 = 0; v0 < nv; v0 += 32) {
        const int v = v0 + lane;
        unsigned long long c = v < nv ? (unsigned long long)w(v) * M : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            c += __shfl_xor_sync(FULL, c, o);
        tot += c;
    }
    const unsigned long long t0 = tot * (unsigned)b / (unsigned)nb, t1 = tot * (unsigned)(b + 1) / (unsigned)nb;
    r0 = r1 = nv * (int)M;
    bool f0 = false, f1 = false;
    unsigned long long base = 0;
    #pragma unroll 1
    for (int v0 = 0; v0 < nv && !f1; v0 += 32) {
        const int v = v0 + lane;
        const int wv = v < nv ? w(v) : 1;
        const unsigned long long c = v < nv ? (unsigned long long)wv * M : 0ull;
        unsigned long long incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(FULL, incl, o);
            if (lane >= o)
                incl += y;
        }
        incl += base;
        const unsigned b0 = __ballot_sync(FULL, v < nv && incl > t0);
        const unsigned b1 = __ballot_sync(FULL, v < nv && incl > t1);
        if (!f0 && b0) {
            const int L = __ffs(b0) - 1;
            const unsigned long long acc = __shfl_sync(FULL, incl - c, L);
            const int wl = __shfl_sync(FULL, wv, L);
            r0 = (v0 + L) * (int)M + (int)((t0 - acc) / (unsigned)wl);
            f0 = true;
        }
        if (b1) {
            const int L = __ffs(b1) - 1;
            const unsigned long long acc = __shfl_sync(FULL, incl - c, L);
            const int wl = __shfl_sync(FULL, wv, L);
            r1 = (v0 + L) * (int)M + (int)((t1 - acc) / (unsigned)wl);
            f1 = true;
        }
        base = __shfl_sync(FULL, incl, 31);
    }
}

// The routed gate/up rows where CTAs b and b + 1 of nb start: the rows of the nvr
// virtual experts are laid end to end and split so that every CTA gets an
// equal share of their cost, a row of an expert with c columns costing
// GU_ROW_COST + c.  vcols == null: every expert has one column (equal rows;
// any thread).  Otherwise warp-collective.  Monotone in b; b = nb gives the
// end of the rows.
__device__ void routed_rows_at(const LayerArgs &a, int nvr, const int *vcols, int b, int nb, int lane, int &r0,
                               int &r1)
{
    if (!vcols) {
        r0 = (int)((unsigned)nvr * (unsigned)a.I * (unsigned)b / (unsigned)nb); // <= 2^21 * 152
        r1 = (int)((unsigned)nvr * (unsigned)a.I * (unsigned)(b + 1) / (unsigned)nb);
        return;
    }
    split_at_warp(nvr, (unsigned)a.I, [&](int v) { return GU_ROW_COST + vcols[v]; }, b, nb, lane, r0, r1);
}

// The flat down items (v, n) = v H + n where CTAs b and b + 1 of nb start: items of
// virtual expert v (the shared expert last, with T columns) cost DN_ROW_COST
// + its columns, and every CTA gets an equal share of the cost.  vcols ==
// null: equal items (any thread); otherwise warp-collective.
__device__ void down_items_at(const LayerArgs &a, int nvr, int nv, const int *vcols, int b, int nb, int lane, int &r0,
                              int &r1)
{
    if (!vcols) {
        r0 = (int)((unsigned)nv * (unsigned)a.H * (unsigned)b / (unsigned)nb); // <= 65 * 2^15 * 152
        r1 = (int)((unsigned)nv * (unsigned)a.H * (unsigned)(b + 1) / (unsigned)nb);
        return;
    }
    split_at_warp(nv, (unsigned)a.H, [&](int v) { return DN_ROW_COST + (v < nvr ? vcols[v] : a.T); }, b, nb, lane,
                  r0, r1);
}

// (vcols != null: warp-collective.  with_down == false: the flat down split
// is left to the caller, it0 = it1 = NPd = 0.)
__device__ LayerPlan make_plan(const LayerArgs &a, int nvr, int bx, int nb, const int *vcols = nullptr, int lane = 0,
                               bool with_down = true)
{
    LayerPlan q;
    const int RU = a.RU;
    q.NVr = nvr;
    q.NV = nvr + (a.wsg ? 1 : 0);
    q.s0 = q.s1 = q.ps0 = q.NPs = 0;
    if (a.wsg) {
        q.s0 = (int)((unsigned)a.I * (unsigned)bx / (unsigned)nb);
        q.s1 = (int)((unsigned)a.I * (unsigned)(bx + 1) / (unsigned)nb);
        q.ps0 = q.s0 / RU;
        q.NPs = q.s1 > q.s0 ? (q.s1 + RU - 1) / RU - q.ps0 : 0;
    }
    routed_rows_at(a, nvr, vcols, bx, nb, lane, q.q0, q.q1);
    q.pr0 = q.q0 / RU;
    q.NPr = q.q1 > q.q0 ? (q.q1 + RU - 1) / RU - q.pr0 : 0;
    q.NPglu = q.NPs + q.NPr;
    q.n0 = (int)((unsigned)a.H * (unsigned)bx / (unsigned)nb);
    q.nrows = (int)((unsigned)a.H * (unsigned)(bx + 1) / (unsigned)nb) - q.n0;
    q.it0 = q.it1 = 0;
    if (a.flat) {
        if (with_down)
            down_items_at(a, nvr, q.NV, vcols, bx, nb, lane, q.it0, q.it1);
        q.nrb = q.rpb = q.rlast = q.spr = q.slast = 0;
        q.SR = a.SR;
        q.NPd = (q.it1 - q.it0 + q.SR - 1) / q.SR;
        return q;
    }
    q.nrb = (q.nrows + a.RB - 1) / a.RB;
    q.rpb = q.nrb ? (q.nrows + q.nrb - 1) / q.nrb : 0;
    q.rlast = q.nrows - (q.nrb - 1) * q.rpb;
    // a stage holds whole experts' runs of rpb rows when one fits (one bulk
    // copy each: few, large copies keep the copy engine at full bandwidth)
    q.SR = q.rpb > 0 && q.rpb <= a.SR ? (a.SR / q.rpb) * q.rpb : a.SR;
    q.spr = q.nrb ? (q.NV * q.rpb + q.SR - 1) / q.SR : 0;
    q.slast = q.nrb ? (q.NV * q.rlast + q.SR - 1) / q.SR : 0;
    q.NPd = q.nrb ? (q.nrb - 1) * q.spr + q.slast : 0;
    return q;
}

// Gate/up part j: virtual expert v (NVr: the shared expert), rows [i0, i0 + n).
__device__ __forceinline__ void part_rows(const LayerArgs &a, const LayerPlan &P, int j, int &v, int &i0, int &n)
{
    if (j < P.NPs) {
        const int r0 = max(P.s0, (P.ps0 + j) * a.RU), r1 = min(P.s1, (P.ps0 + j + 1) * a.RU);
        v = P.NVr;
        i0 = r0;
        n = r1 - r0;
    } else {
        const int p = P.pr0 + (j - P.NPs);
        const int f0 = max(P.q0, p * a.RU), f1 = min(P.q1, (p + 1) * a.RU);
        v = (int)(f0 / a.I);
        i0 = f0 - v * a.I;
        n = (int)(f1 - f0);
    }
}

// Row block and the items of down stage d.
__device__ __forceinline__ void down_stage(const LayerArgs &a, const LayerPlan &P, int d, int &rb, int &nr0,
                                           int &rows, int &i0, int &i1)
{
    rb = d / max(P.spr, 1);
    int sp;
    if (rb >= P.nrb - 1) {
        rb = P.nrb - 1;
        sp = d - (P.nrb - 1) * P.spr;
    } else {
        sp = d - rb * P.spr;
    }
    nr0 = P.n0 + rb * P.rpb;
    rows = rb == P.nrb - 1 ? P.rlast : P.rpb;
    i0 = sp * P.SR;
    i1 = min(P.NV * rows, i0 + P.SR);
}

// Stage s of a CTA into slot s % NS: a gate/up part (gate rows at 0, up
// rows at RU rbg) or a down stage (its items' weight rows in item order).
// v_e maps routed virtual experts to experts.  Called by one thread; kept out
// of line (two call sites, off the arithmetic's path).
__device__ __noinline__ void issue_stage(const LayerArgs &a, const LayerPlan &P, int s, uint8_t *ring, uint64_t *full,
                                         uint64_t pol, const int *v_e)
{
    const int slot = s % a.NS;
    uint8_t *dst = ring + (size_t)slot * a.stage_bytes;
    const int E = a.E;
    if (s < P.NPglu) {
        int v, i0, n;
        part_rows(a, P, s, v, i0, n);
        const bool routed = v < P.NVr;
        const int e = routed ? v_e[v] : E;
        const uint8_t *g = routed ? a.wg + ((size_t)e * a.I + i0) * a.rbg : a.wsg + (size_t)i0 * a.rbg;
        const uint8_t *u = routed ? a.wu + ((size_t)e * a.I + i0) * a.rbg : a.wsu + (size_t)i0 * a.rbg;
        const uint32_t bytes = (uint32_t)(n * a.rbg);
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        bulk_copy_g2s(dst, g, bytes, &full[slot], pol);
        bulk_copy_g2s(dst + (size_t)a.RU * a.rbg, u, bytes, &full[slot], pol);
        return;
    }
    // down items [i0, i1) of a list whose item i is virtual expert i / rows,
    // row base + i mod rows
    int i0, i1;
    int rows, base;
    if (a.flat) {
        i0 = P.it0 + (s - P.NPglu) * P.SR;
        i1 = min(P.it1, i0 + P.SR);
        rows = a.H;
        base = 0;
    } else {
        int rb, nr0, ii0, ii1;
        down_stage(a, P, s - P.NPglu, rb, nr0, rows, ii0, ii1);
        i0 = ii0;
        i1 = ii1;
        base = nr0;
    }
    mbar_arrive_expect_tx(&full[slot], (uint32_t)((i1 - i0) * a.rbd));
    #pragma unroll 1
    for (int i = i0; i < i1;) {
        const int v = i / rows, m = i - v * rows;
        const int cnt = min(i1 - i, rows - m);
        const int e = v < P.NVr ? v_e[v] : E;
        const uint8_t *src = e < E ? a.wd + ((size_t)e * a.H + base + m) * a.rbd : a.wsd + (size_t)(base + m) * a.rbd;
        bulk_copy_g2s(dst + (size_t)(i - i0) * a.rbd, src, (uint32_t)(cnt * a.rbd), &full[slot], pol);
        i += cnt;
    }
}

template <int TT, bool FLAT>
__global__ void __launch_bounds__(THREADS, 1) k_moe_layer(const LayerArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * a.stage_bytes);
    uint64_t *empty = full + a.NS;
    uint32_t *act = reinterpret_cast<uint32_t *>(empty + a.NS); // x rows, later the hq rows (16-byte aligned)
    const int R = a.T * a.k;
    const int nslots = R + (a.wsg ? a.T : 0);
    const size_t act_words = max((size_t)a.T * a.xstride, (size_t)a.hq_rows * a.hstride);
    float *scores = reinterpret_cast<float *>(act + act_words); // [T][E] logit + bias
    float *lsm = scores + (size_t)a.T * a.E;                   // [T][E] logits

    __shared__ int ids_s[MAX_R], routes_s[MAX_R];
    __shared__ float w_s[MAX_R];
    __shared__ int cnt_s[MAX_E], off_s[MAX_E + 1];
    __shared__ int v_e[MAX_V], v_first[MAX_V], v_ncols[MAX_V];
    __shared__ uint32_t sel_bits[MAX_T][MAX_E / 32]; // expert e selected by token t
    __shared__ int s_abort;
    __shared__ int s_issued; // stages requested so far (written by the producer after each request)
    __shared__ int s_nvr;   // routed virtual experts
    __shared__ LayerPlan s_plan; // several tokens: the plan (warp 0) ...
    __shared__ int s_it[2];      // ... and its down split (warp 1)
    __shared__ unsigned long long s_c0; // barrier count at the start


    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, k = a.k;
    const bool cta0 = blockIdx.x == 0;
    const int nb = gridDim.x, bx = blockIdx.x;
    const int RU = a.RU, NG = a.NG;
    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();
    const int gmap = (a.nbH % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN; // gate/up row mapping
    const int xpad = gmap == ROWMAP_PAIRS ? 16 : 0;
    const int dmap = a.nbI == 32 ? ROWMAP_TWO_ROWS : (a.nbI % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN;
    const int hpad = dmap == ROWMAP_PAIRS ? 16 : 0;

    // With one token the router selects k experts, so the plan is known
    // before the routing.
    const LayerPlan P1 = make_plan(a, T == 1 ? k : 0, bx, nb);
    if (tid == CTHREADS) {
        #pragma unroll 1
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW); // every consumer warp, or a group's warps CW / RU times each
        }
        fence_mbar_init();
        s_abort = 0;
        s_issued = 0;
    }
    __syncthreads(); // barriers initialized
    // (The producer requests every stage after the routing: requesting the
    // shared expert's first stages before it, while the routing runs, measured
    // slower on the verify layer.)
    int issued = 0; // producer lane 0: stages requested
    if (warp == CW) {
        // the inputs of the routing into L2 (a hint)
        for (int i = lane; i < (T * E + 31) / 32; i += 32)
            prefetch_line_l2(a.logits + 32 * i);
        for (int i = lane; a.bias && i < (E + 31) / 32; i += 32)
            prefetch_line_l2(a.bias + 32 * i);
    }
    pdl_wait();
    pdl_trigger();
    if (tid == 0)
        s_c0 = ld_acquire_gpu_u64(a.sync); // every earlier launch's barriers have ended

    bool dead = false;
    // Waits for stage s (slot s % NS, use s / NS); false if this CTA gave up
    // (warp-collective: every lane takes the same branch).  Consumer groups
    // take the gate/up parts round-robin and share the ring's slots, so a
    // group may reach part s while the slot still shows an older use of the
    // same parity: it first waits until the producer has requested stage s
    // (s_issued > s; the request arms the slot's phase for this use), and only
    // then for the phase's parity.  Every consumer warp consumes the down
    // stages in order, after every gate/up part.
    auto wait_stage = [&](int s) -> bool {
        if (__any_sync(FULL, *(volatile int *)&s_abort != 0))
            dead = true;
        if (dead)
            return false;
        bool req = *(volatile int *)&s_issued > s;
        if (!__all_sync(FULL, req)) {
            const unsigned long long t0 = global_timer_ns();
            for (;;) {
                __nanosleep(32);
                req = *(volatile int *)&s_issued > s;
                if (__all_sync(FULL, req) || __any_sync(FULL, *(volatile int *)&s_abort != 0) ||
                    __any_sync(FULL, global_timer_ns() - t0 > WAIT_LIMIT_NS))
                    break;
            }
        }
        __threadfence_block(); // the request's arrival before the parity test
        const bool got =
            __all_sync(FULL, req) && __all_sync(FULL, mbar_wait_parked(&full[s % a.NS], (uint32_t)(s / a.NS) & 1u));
        if (!got) {
            if (lane == 0) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
            }
            dead = true;
            return false;
        }
        return true;
    };

    // x -> q8_1 into shared memory (CTA 0 also stores xq) by warps
    // [w0, w0 + nw): 8 blocks per warp and pass, 4 lanes per block, XP
    // passes' loads in flight at once (warp-collective)
    const int nbx = T * a.nbH;
    auto quantize_x = [&](int w0, int nw) {
        constexpr int XP = 4;
        const int qj = lane & 3;
        const int step = nw * 8;
        #pragma unroll 1
        for (int base0 = (warp - w0) * 8; base0 < nbx; base0 += XP * step) { // warp-uniform trip count
            float v[XP][8];
#pragma unroll
            for (int q = 0; q < XP; q++) {
                const int b = base0 + q * step + (lane >> 2);
                if (b < nbx) {
                    load8(a.x + (size_t)b * QK + qj * 8, v[q], false);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; i++)
                        v[q][i] = 0.0f;
                }
            }
#pragma unroll
            for (int q = 0; q < XP; q++) {
                if (base0 + q * step >= nbx)
                    break; // warp-uniform
                const int b = base0 + q * step + (lane >> 2);
                const bool valid = b < nbx;
                const int bt = valid ? b / a.nbH : 0, bg = valid ? b - bt * a.nbH : 0;
                quantize_q8_1_quad(v[q], valid, act + (size_t)bt * a.xstride + xblock_word(bg, xpad),
                                   cta0 && valid ? a.xq + (size_t)b * Q8_1_WORDS : nullptr, qj);
            }
        }
    };

    // ---------------- routing ----------------
    // Scores (a NaN ranks below every number) and the rank of every (token,
    // expert) pair by `nthr` threads starting at thread `t0` (four threads per
    // pair): expert e of token t takes slot #{e' ranked before e} when that is
    // below k, the (score descending, index ascending) order of the
    // sequential selection.  Named barrier `bar` among the nthr threads.
    auto route_rank = [&](int t0, int nthr, int bar) {
        const int rt = tid - t0;
        #pragma unroll 1
        for (int i0 = rt; i0 < T * E; i0 += 2 * nthr) {
            float l[2], bb[2];
#pragma unroll
            for (int q = 0; q < 2; q++) { // every load in flight before the first use
                const int i = i0 + q * nthr;
                l[q] = i < T * E ? a.logits[i] : 0.0f;
                bb[q] = (a.bias && i < T * E) ? a.bias[i % E] : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 2; q++) {
                const int i = i0 + q * nthr;
                if (i < T * E) {
                    lsm[i] = l[q];
                    const float sc = a.bias ? __fadd_rn(l[q], bb[q]) : l[q];
                    scores[i] = sc == sc ? sc : -INFINITY;
                }
            }
        }
        #pragma unroll 1
        for (int i = rt; i < MAX_T * (MAX_E / 32); i += nthr)
            (&sel_bits[0][0])[i] = 0u;
        named_barrier(bar, nthr);
        const int npair = T * E;
        const int qj = lane & 3; // four threads per pair
        #pragma unroll 1
        for (int base = 0; base < npair; base += nthr / 4) { // warp-uniform trip count
            const int p = base + (rt >> 2);
            int rank = 0, t = 0, e = 0;
            if (p < npair) {
                t = p / E;
                e = p - t * E;
                const float *sc = scores + (size_t)t * E;
                const float v = sc[e];
                // thread qj takes experts qj, qj + 4, ...: the four threads of a
                // pair read four neighbouring words (no bank conflict)
#pragma unroll 8
                for (int e2 = qj; e2 < E; e2 += 4) {
                    const float o = sc[e2];
                    rank += (o > v || (o == v && e2 < e)) ? 1 : 0;
                }
            }
            rank += __shfl_xor_sync(FULL, rank, 1);
            rank += __shfl_xor_sync(FULL, rank, 2);
            if (p < npair && qj == 0 && rank < k) {
                ids_s[t * k + rank] = e;
                atomicOr(&sel_bits[t][e >> 5], 1u << (e & 31));
            }
        }
        named_barrier(bar, nthr);
    };
    // The expert tables (one warp): virtual expert v is the v-th selected
    // expert in index order; its columns are the routes that chose it, in
    // route order, at [first, first + ncols) of the route list.
    auto build_tables = [&]() {
        int nact = 0, offp = 0;
        #pragma unroll 1
        for (int c = 0; c < E; c += 32) { // warp-uniform trip count
            const int e = c + lane;
            int cnt = 0;
            if (e < E)
                #pragma unroll 1
                for (int t = 0; t < T; t++)
                    cnt += (sel_bits[t][e >> 5] >> (e & 31)) & 1u;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const unsigned bal = __ballot_sync(FULL, cnt > 0);
            const int v = nact + __popc(bal & ((1u << lane) - 1u));
            const int off = offp + incl - cnt;
            if (e < E) {
                cnt_s[e] = cnt;
                off_s[e] = off;
            }
            if (cnt > 0) {
                v_e[v] = e;
                v_first[v] = off;
                v_ncols[v] = cnt;
            }
            nact += __popc(bal);
            offp += __shfl_sync(FULL, incl, 31);
        }
        if (lane == 0) {
            off_s[E] = offp;
            s_nvr = nact;
            if (a.wsg) {
                v_e[nact] = E;
                v_first[nact] = R;
                v_ncols[nact] = T;
            }
        }
    };
    // route weights (one softmax per token) and the route list: route
    // r = t k + j goes to position pos(r), the routes ahead of it in (expert,
    // route) order (one warp)
    auto weights_routes = [&]() {
        #pragma unroll 1
        for (int t = 0; t < T; t++) {
            const float sel0 = lane < k ? lsm[t * E + ids_s[t * k + lane]] : 0.0f;
            const float sel1 = lane + 32 < k ? lsm[t * E + ids_s[t * k + lane + 32]] : 0.0f;
            route_softmax_warp(sel0, sel1, k, w_s + t * k, lane);
        }
        // the routes ahead of r = t k + j: every route of a lower expert
        // (off_s[e]) and the routes of expert e from earlier tokens (a
        // token selects k distinct experts)
        #pragma unroll 1
        for (int r = lane; r < R; r += 32) {
            const int e = ids_s[r], t = r / k;
            int pos = off_s[e];
            #pragma unroll 1
            for (int t2 = 0; t2 < t; t2++)
                pos += (int)((sel_bits[t2][e >> 5] >> (e & 31)) & 1u);
            routes_s[pos] = r;
        }
    };
    // Several tokens: the route weights of token t (one warp; CTA 0 also
    // stores them), the route list (one warp) and CTA 0's copy of the rest of
    // the tables (one warp)
    auto token_weights = [&](int t) {
        const float sel0 = lane < k ? lsm[t * E + ids_s[t * k + lane]] : 0.0f;
        const float sel1 = lane + 32 < k ? lsm[t * E + ids_s[t * k + lane + 32]] : 0.0f;
        route_softmax_warp(sel0, sel1, k, w_s + t * k, lane);
        __syncwarp();
        if (cta0)
            for (int j = lane; j < k; j += 32)
                a.weights[t * k + j] = w_s[t * k + j];
    };
    auto route_positions = [&]() {
        #pragma unroll 1
        for (int r = lane; r < R; r += 32) {
            const int e = ids_s[r], t = r / k;
            int pos = off_s[e];
            #pragma unroll 1
            for (int t2 = 0; t2 < t; t2++)
                pos += (int)((sel_bits[t2][e >> 5] >> (e & 31)) & 1u);
            routes_s[pos] = r;
        }
    };
    auto store_rest = [&]() {
        #pragma unroll 1
        for (int i = lane; i < R; i += 32) {
            a.ids[i] = ids_s[i];
            a.routes[i] = routes_s[i];
        }
        #pragma unroll 1
        for (int e = lane; e < E; e += 32) {
            a.counts[e] = cnt_s[e];
            a.offsets[e] = off_s[e];
        }
        if (lane == 0)
            a.offsets[E] = off_s[E];
    };
    // CTA 0 stores the routing tables (one warp)
    auto store_tables = [&]() {
        #pragma unroll 1
        for (int i = lane; i < R; i += 32) {
            a.ids[i] = ids_s[i];
            a.weights[i] = w_s[i];
            a.routes[i] = routes_s[i];
        }
        #pragma unroll 1
        for (int e = lane; e < E; e += 32) {
            a.counts[e] = cnt_s[e];
            a.offsets[e] = off_s[e];
        }
        if (lane == 0)
            a.offsets[E] = off_s[E];
    };

    // Every warp ranks the experts.  With one token the first half of the
    // consumer warps then quantizes x, the producer derives the routed virtual
    // experts (the selected experts in index order) and starts requesting
    // their rows at once, while warp RT0 / 32 builds the tables the consumers
    // need (expert columns, route list, weights, CTA 0's copy); the consumers
    // meet it at BAR_TABLES before their first routed part.  With more tokens
    // every consumer warp quantizes x; then the producer warp builds the
    // tables and the route list, warps 0 and 1 make this CTA's plan from the
    // tables, warps 2 .. T + 1 weigh one token's routes each, and every warp
    // waits for all of it.
    route_rank(0, THREADS, BAR_SEL); // every warp
    const int wsel = RT0 / 32; // the tables warp (one token)
    if (T == 1 ? tid < RT0 : tid < CTHREADS)
        quantize_x(0, T == 1 ? RT0 / 32 : CW);
    if (T == 1) {
        if (warp == CW) {
            // virtual expert v = the v-th selected expert in index order
            int nv = 0;
            #pragma unroll 1
            for (int j = 0; j < (E + 31) / 32; j++) {
                const uint32_t m = sel_bits[0][j];
                if ((m >> lane) & 1u)
                    v_e[nv + __popc(m & ((1u << lane) - 1u))] = lane + 32 * j;
                nv += __popc(m);
            }
            __syncwarp();
        } else if (warp == wsel) {
            build_tables();
            __syncwarp();
            weights_routes();
            __syncwarp();
            if (cta0)
                store_tables();
        }
    } else {
        __syncthreads(); // selections and x in shared memory
        if (warp == CW) {
            build_tables();
            __syncwarp();
            named_barrier_arrive(BAR_PLAN, 3 * 32); // the tables for warps 0 and 1
            route_positions();
            __syncwarp();
            if (cta0)
                store_rest();
        } else if (warp >= 2 && warp < 2 + T) {
            token_weights(warp - 2); // (T <= 8: warps 2 .. 9)
        } else if (warp < 2) {
            named_barrier(BAR_PLAN, 3 * 32);
            if (warp == 0) {
                const LayerPlan q = make_plan(a, s_nvr, bx, nb, v_ncols, lane, false);
                if (lane == 0)
                    s_plan = q;
            } else {
                int i0, i1;
                down_items_at(a, s_nvr, s_nvr + (a.wsg ? 1 : 0), v_ncols, bx, nb, lane, i0, i1);
                if (lane == 0) {
                    s_it[0] = i0;
                    s_it[1] = i1;
                }
            }
        }
        __syncthreads(); // tables, weights, route list and plan in shared memory
    }
    const LayerPlan P = [&]() {
        if (T == 1)
            return P1;
        LayerPlan q = s_plan;
        if (a.flat) {
            q.it0 = s_it[0];
            q.it1 = s_it[1];
            q.NPd = (q.it1 - q.it0 + q.SR - 1) / q.SR;
        }
        return q;
    }();

    if (warp == CW) {
        // ---------------- the producer: every stage of this CTA ----------------
        if (lane != 0)
            return;
        const int NST = P.NPglu + P.NPd;
        #pragma unroll 1
        while (issued < NST) {
            if (*(volatile int *)&s_abort)
                break;
            const int slot = issued % a.NS, use = issued / a.NS;
            // the slot's previous stage released by its consumers (the wait
            // sleeps rather than spins)
            if (use > 0 && !mbar_wait_parked(&empty[slot], (uint32_t)(use - 1) & 1u)) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
                break;
            }
            issue_stage(a, P, issued, ring, full, pol, v_e);
            issued++;
            __threadfence_block(); // the stage's expect_tx arrival before its count
            *(volatile int *)&s_issued = issued;
        }
        // no bulk copy may still be writing shared memory when the CTA exits
        #pragma unroll 1
        for (int u = 0; u < a.NS && u < issued; u++) {
            const int last = issued - 1 - u; // the last use of slot last % NS
            if (!mbar_wait_bounded(&full[last % a.NS], (uint32_t)(last / a.NS) & 1u))
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers ----------------
    if (T == 1)
        named_barrier(BAR_CONS, CTHREADS); // all of x is quantized
    // one token: the tables warp arrives at BAR_TABLES; every other consumer
    // warp meets it once, before its first routed part
    bool tables_seen = T != 1 || warp == wsel;
    if (T == 1 && warp == wsel)
        named_barrier_arrive(BAR_TABLES, CTHREADS);

    // ---------------- gate/up parts -> h ----------------
    // one token: this lane's x blocks stay in registers for every row
    constexpr int XR = 4;
    const int nblg = rowmap_blocks(gmap, a.nbH, lane);
    // one token: this lane's x blocks stay in registers (the host sends one
    // token whose rows have more than XR blocks per lane to the TT = 2 kernel)
    constexpr bool x_regs = TT == 1;
    Q81Block xreg[XR];
    if constexpr (x_regs) {
#pragma unroll
        for (int j = 0; j < XR; j++) {
            if (j < nblg) {
                load_q8_1_any(act + xblock_word(rowmap_block(gmap, lane, j), xpad), xreg[j]);
            } else {
                xreg[j].d = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; i++)
                    xreg[j].q[i] = 0;
            }
        }
    }
    const int grp = warp / RU, wl = warp - grp * RU;
    #pragma unroll 1
    for (int j = grp; grp < NG && j < P.NPglu; j += NG) {
        int v, i0, n;
        part_rows(a, P, j, v, i0, n);
        if (!tables_seen && j >= P.NPs) {
            named_barrier(BAR_TABLES, CTHREADS);
            tables_seen = true;
        }
        if (wait_stage(j) && wl < n) {
            const uint8_t *st = ring + (size_t)(j % a.NS) * a.stage_bytes;
            const uint8_t *grow = st + (size_t)wl * a.rbg;
            const uint8_t *urow = st + (size_t)(RU + wl) * a.rbg;
            const uint32_t gsa = smem_addr(grow), usa = smem_addr(urow);
            const int i = i0 + wl;
            const bool routed = v < P.NVr;
            if constexpr (x_regs) {
                float ag = 0.0f, au = 0.0f;
#pragma unroll
                for (int jj = 0; jj < XR; jj++) {
                    if (jj < nblg) {
                        const int b = rowmap_block(gmap, lane, jj);
                        Q80Block gbk, ubk;
                        load_q8_0_sh(gsa, b, gbk);
                        load_q8_0_sh(usa, b, ubk);
                        const int sg = dot_q8_block(gbk.q, xreg[jj].q);
                        const int su = dot_q8_block(ubk.q, xreg[jj].q);
                        ag = fmaf(gbk.d * xreg[jj].d, (float)sg, ag);
                        au = fmaf(ubk.d * xreg[jj].d, (float)su, au);
                    }
                }
                const float sm = reduce2(ag, au, lane);
                const float u = __shfl_sync(FULL, sm, 16);
                if (lane == 0) {
                    const int slot = routed ? routes_s[v_first[v]] : R;
                    a.h[(size_t)slot * a.I + i] = swiglu(sm, u, a.clamp);
                }
            } else {
                const int first = routed ? v_first[v] : 0, ncols = routed ? v_ncols[v] : T;
                // NC columns at a time, NC a constant: no column slot of the
                // unrolled loops is predicated off
                auto cols = [&](int c0, auto ncc) {
                    constexpr int NC = decltype(ncc)::value;
                    uint32_t xsa[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++)
                        xsa[c] = smem_addr(act + (size_t)(routed ? routes_s[first + c0 + c] / k : c0 + c) * a.xstride);
                    float ag[NC], au[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++)
                        ag[c] = au[c] = 0.0f;
                    for (int jj = 0; jj < nblg; jj++) {
                        const int b = rowmap_block(gmap, lane, jj);
                        Q80Block gbk, ubk;
                        load_q8_0_sh(gsa, b, gbk);
                        load_q8_0_sh(usa, b, ubk);
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            Q81Block xb;
                            load_q8_1_sh(xsa[c] + 4u * (uint32_t)xblock_word(b, xpad), xb);
                            const int sg = dot_q8_block(gbk.q, xb.q);
                            const int su = dot_q8_block(ubk.q, xb.q);
                            ag[c] = fmaf(gbk.d * xb.d, (float)sg, ag[c]);
                            au[c] = fmaf(ubk.d * xb.d, (float)su, au[c]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < NC; c++) {
                        const float sm = reduce2(ag[c], au[c], lane);
                        const float u = __shfl_sync(FULL, sm, 16);
                        if (lane == 0) {
                            const int slot = routed ? routes_s[first + c0 + c] : R + c0 + c;
                            a.h[(size_t)slot * a.I + i] = swiglu(sm, u, a.clamp);
                        }
                    }
                };
                #pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += TT) {
                    const int nc = min(TT, ncols - c0);
                    if (TT >= 4 && nc >= 4)
                        cols(c0, std::integral_constant<int, (TT >= 4 ? 4 : 1)>{});
                    else if (TT >= 3 && nc == 3)
                        cols(c0, std::integral_constant<int, (TT >= 3 ? 3 : 1)>{});
                    else if (TT >= 2 && nc == 2)
                        cols(c0, std::integral_constant<int, (TT >= 2 ? 2 : 1)>{});
                    else
                        cols(c0, std::integral_constant<int, 1>{});
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !dead)
            mbar_arrive_count(&empty[j % a.NS], (uint32_t)(CW / RU)); // this warp is done with the stage
    }

    if (!tables_seen)
        named_barrier(BAR_TABLES, CTHREADS); // a warp without routed parts

    // ---------------- device-wide barriers, q8_1 of h ----------------
    auto barrier = [&](int nth) {
        named_barrier(BAR_CONS, CTHREADS); // this CTA's stores are done
        if (tid == 0 && !*(volatile int *)&s_abort && !grid_barrier(a.sync, gridDim.x, s_c0, nth)) {
            atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT | LUCE_FAULT_DESYNC);
            *(volatile int *)&s_abort = 1;
        }
        named_barrier(BAR_CONS, CTHREADS);
    };
    auto item_cols = [&](int v, int &first, int &ncols) {
        const bool routed = v < P.NVr;
        first = routed ? v_first[v] : R;
        ncols = routed ? v_ncols[v] : T;
    };
    auto col_slot = [&](int v, int first, int c) { return v < P.NVr ? routes_s[first + c] : R + c; };
    const int nhb = nslots * a.nbI;
    barrier(1); // every h value is stored
    // this CTA's share of the q8_1 blocks of h: blocks bx + nb q for q = 8
    // warp + i (+ 8 CW per pass), 4 lanes per block
    if (!*(volatile int *)&s_abort) {
        const int qj = lane & 3;
        #pragma unroll 1
        for (int base = warp * 8; base * nb + bx < nhb; base += CW * 8) { // warp-uniform trip count
            const int ub = (base + (lane >> 2)) * nb + bx; // blocks bx, bx + nb, ...
            const bool valid = ub < nhb;
            float vv[8];
            if (valid) {
                const int slot = ub / a.nbI, b = ub - slot * a.nbI;
                load8(a.h + (size_t)slot * a.I + b * QK + qj * 8, vv, true);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    vv[i] = 0.0f;
            }
            quantize_q8_1_quad(vv, valid, nullptr, valid ? a.hq + (size_t)ub * Q8_1_WORDS : nullptr, qj);
        }
    }
    barrier(2); // every q8_1 block of h is stored
    // The hq rows this CTA reads into shared memory (the padding of the
    // ROWMAP_PAIRS rows in place): all rows (split by output rows), or row
    // (v - v_lo) T + c = column c of virtual expert v for the experts this
    // CTA's flat items touch.
    const int v_lo = FLAT ? (int)(P.it0 / a.H) : 0;
    const int v_hi = FLAT ? (P.it1 > P.it0 ? (int)((P.it1 - 1) / a.H) : v_lo) : 0;
    const int nhrows = FLAT ? (v_hi - v_lo + 1) * T : nslots;
    if (FLAT && nhrows > a.hq_rows && tid == 0 && !*(volatile int *)&s_abort) {
        // (the host sizes hq_rows for every split; never expected)
        atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        *(volatile int *)&s_abort = 1;
    }
    named_barrier(BAR_CONS, CTHREADS);
    // (16-byte loads by every consumer thread: a few KB, so one round trip
    // to L2 rather than many small bulk copies)
    if (!*(volatile int *)&s_abort) {
        const int n4 = a.nbI * Q8_1_WORDS / 4; // uint4 per row
        const int run4 = 32 * Q8_1_WORDS / 4;  // uint4 per 32 blocks
        #pragma unroll 1
        for (int idx = tid; idx < nhrows * n4; idx += CTHREADS) {
            const int r = idx / n4, w4 = idx - r * n4;
            int slot = r;
            if (FLAT) {
                int first, ncols;
                item_cols(v_lo + r / T, first, ncols);
                slot = r % T < ncols ? col_slot(v_lo + r / T, first, r % T) : 0;
            }
            const uint4 val = __ldcg(reinterpret_cast<const uint4 *>(a.hq + (size_t)slot * a.nbI * Q8_1_WORDS) + w4);
            reinterpret_cast<uint4 *>(act + (size_t)r * a.hstride)[w4 + (hpad / 4) * (w4 / run4)] = val;
        }
    }
    named_barrier(BAR_CONS, CTHREADS); // the hq rows are in shared memory

    // ---------------- down rows, combine ----------------
    // out[t][n] for rows [nr0, nr0 + rows): sum_j fl(w * y) in slot order,
    // then + shared; y(slot, m) reads the y values
    auto combine = [&](int nr0, int rows, auto y) {
        if (dead || *(volatile int *)&s_abort)
            return;
        #pragma unroll 1
        for (int idx = tid; idx < T * rows; idx += CTHREADS) {
            const int t = idx / rows, m = idx - t * rows;
            float acc = 0.0f;
            #pragma unroll 1
            for (int j = 0; j < k; j++) {
                const int e = ids_s[t * k + j];
                if (e >= 0)
                    acc = __fadd_rn(acc, __fmul_rn(w_s[t * k + j], y(t * k + j, m)));
            }
            if (a.wsd)
                acc = __fadd_rn(acc, y(R + t, m));
            a.out[(size_t)t * a.H + nr0 + m] = acc;
        }
    };
    // Down items [ia, ib) of a list whose item i is virtual expert v = i /
    // rows, row m = i mod rows; the item's weight row sits in stage
    // (i - ib0) / SR of the down stages at stage number sd0, row
    // (i - ib0) mod SR.  Each warp takes a contiguous chunk of the items;
    // with rows of 32 blocks its two half-warps take neighbouring items (rows
    // 16 banks apart), else the whole warp takes each item.  Every column of
    // an item's expert is computed; hrow(v, first, c) is the column's hq row in
    // shared memory, put(slot, v, m, y) stores y.  The warp first waits for
    // the stages of its chunk.
    const bool two = dmap == ROWMAP_TWO_ROWS;
    const int nbl = rowmap_blocks(dmap, a.nbI, lane);
    int dw = -1; // the last down stage this warp waited for (stage number - d0)
    const int d0 = P.NPglu;
    auto down_items = [&](int ia, int ib, int ib0, int sd0, int rows, auto hrow, auto put, int wi, int nwc) {
        const int ni = ib - ia;
        const int c0i = ia + ni * wi / nwc, c1i = ia + ni * (wi + 1) / nwc;
        if (c1i > c0i) {
            const int dn = sd0 + (c1i - 1 - ib0) / P.SR; // the chunk's last stage
            const int da = sd0 + (c0i - ib0) / P.SR;     // and its first
            if (dw < da - 1)
                dw = da - 1; // (stages before the chunk's first: not read by this warp)
            while (dw < dn && !dead) {
                ++dw;
                wait_stage(d0 + dw);
            }
        }
        if (dead)
            return;
        const int h = two ? (lane >> 4) : 0;
        const int step = two ? 2 : 1;
        int i = c0i + h;
        int v = i / rows, m = i - v * rows;
        if constexpr (TT == 1) {
            // One token: every expert has one column.  Neighbouring items share
            // their expert, so the lane keeps that column's hq blocks in
            // registers while it does (shared-memory bandwidth bounds this
            // loop: each weight byte is read once, each hq row once per run of
            // items).
            constexpr int XC = 4;
            if (rowmap_blocks(dmap, a.nbI, 0) <= XC) { // warp-uniform
                Q81Block xc[XC];
                int vc = -1;
                int r = i - ib0, d = r / P.SR;
                uint32_t slot_sa = smem_addr(ring + (size_t)((d0 + sd0 + d) % a.NS) * a.stage_bytes);
                #pragma unroll 1
                for (int q = c0i; q < c1i; q += step) {
                    const bool live = i < c1i;
                    int first = 0, ncols = 0;
                    if (live) {
                        item_cols(v, first, ncols);
                        if (v != vc) {
                            const uint32_t xsa = smem_addr(hrow(v, first, 0));
#pragma unroll
                            for (int jb = 0; jb < XC; jb++)
                                if (jb < nbl)
                                    load_q8_1_sh(xsa + 4u * (uint32_t)xblock_word(rowmap_block(dmap, lane, jb), hpad),
                                                 xc[jb]);
                            vc = v;
                        }
                    }
                    const uint32_t wsa = live ? slot_sa + (uint32_t)((r - d * P.SR) * a.rbd) : smem_addr(ring);
                    float acc = 0.0f;
#pragma unroll
                    for (int jb = 0; jb < XC; jb++) {
                        if (jb < nbl && live) {
                            Q80Block wb;
                            load_q8_0_sh(wsa, rowmap_block(dmap, lane, jb), wb);
                            acc = fmaf(wb.d * xc[jb].d, (float)dot_q8_block(wb.q, xc[jb].q), acc);
                        }
                    }
                    const float y = two ? half_warp_sum(acc) : warp_sum(acc);
                    if (live && (two ? (lane & 15) : lane) == 0)
                        put(col_slot(v, first, 0), v, m, y);
                    i += step;
                    m += step;
                    r += step;
                    while (m >= rows) {
                        m -= rows;
                        v++;
                    }
                    if (r - d * P.SR >= P.SR) {
                        d = r / P.SR;
                        slot_sa = smem_addr(ring + (size_t)((d0 + sd0 + d) % a.NS) * a.stage_bytes);
                    }
                }
                return;
            }
        }
        if (!two) {
            // Two items at a time (their dot chains interleave; each item's
            // arithmetic and order are those of the one-item loop below).  Two
            // items of the same expert share their hq blocks.
            #pragma unroll 1
            for (int q = c0i; q < c1i; q += 2) { // warp-uniform
                const bool live1 = q + 1 < c1i;
                int v1 = v, m1 = m + 1;
                if (m1 >= rows) {
                    m1 -= rows;
                    v1++;
                }
                int first0 = 0, nc0 = 0, first1 = 0, nc1 = 0;
                item_cols(v, first0, nc0);
                if (live1)
                    item_cols(v1, first1, nc1);
                const int r0 = i - ib0, d0s = r0 / P.SR;
                const uint8_t *wr0 =
                    ring + (size_t)((d0 + sd0 + d0s) % a.NS) * a.stage_bytes + (size_t)(r0 - d0s * P.SR) * a.rbd;
                const int r1 = r0 + 1, d1s = r1 / P.SR;
                const uint8_t *wr1 =
                    ring + (size_t)((d0 + sd0 + d1s) % a.NS) * a.stage_bytes + (size_t)(r1 - d1s * P.SR) * a.rbd;
                const bool same = live1 && v1 == v;
                const int ncm = max(nc0, nc1);
                // NC columns at a time, NC a constant, and the common case of
                // two items of one expert (same column count, shared hq
                // blocks) apart: no slot of the unrolled loops is predicated off
                auto pass = [&](int cb, auto ncc, auto samec) {
                    constexpr int NC = decltype(ncc)::value;
                    constexpr bool SAME = decltype(samec)::value;
                    float acc0[NC], acc1[NC];
                    uint32_t xs0[NC], xs1[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++) {
                        acc0[c] = acc1[c] = 0.0f;
                        xs0[c] = smem_addr(SAME || cb + c < nc0 ? hrow(v, first0, cb + c) : act);
                        xs1[c] = SAME ? 0u : smem_addr(live1 && cb + c < nc1 ? hrow(v1, first1, cb + c) : act);
                    }
                    const uint32_t wsa0 = smem_addr(wr0), wsa1 = smem_addr(live1 ? wr1 : wr0);
                    for (int jb = 0; jb < nbl; jb++) {
                        const int b = rowmap_block(dmap, lane, jb);
                        Q80Block wb0, wb1;
                        load_q8_0_sh(wsa0, b, wb0);
                        load_q8_0_sh(wsa1, b, wb1);
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            if (SAME || cb + c < nc0) {
                                Q81Block xb;
                                load_q8_1_sh(xs0[c] + 4u * (uint32_t)xblock_word(b, hpad), xb);
                                acc0[c] = fmaf(wb0.d * xb.d, (float)dot_q8_block(wb0.q, xb.q), acc0[c]);
                                if (SAME)
                                    acc1[c] = fmaf(wb1.d * xb.d, (float)dot_q8_block(wb1.q, xb.q), acc1[c]);
                            }
                            if (!SAME && live1 && cb + c < nc1) {
                                Q81Block xb;
                                load_q8_1_sh(xs1[c] + 4u * (uint32_t)xblock_word(b, hpad), xb);
                                acc1[c] = fmaf(wb1.d * xb.d, (float)dot_q8_block(wb1.q, xb.q), acc1[c]);
                            }
                        }
                    }
#pragma unroll
                    for (int c = 0; c < NC; c++) {
                        if (SAME || cb + c < nc0) {
                            const float y = warp_sum(acc0[c]);
                            if (lane == 0)
                                put(col_slot(v, first0, cb + c), v, m, y);
                        }
                        if (SAME || (live1 && cb + c < nc1)) {
                            const float y = warp_sum(acc1[c]);
                            if (lane == 0)
                                put(col_slot(v1, first1, cb + c), v1, m1, y);
                        }
                    }
                };
                auto pass_n = [&](int cb, auto samec) {
                    const int nc = min(TT, ncm - cb);
                    if (TT >= 4 && nc >= 4)
                        pass(cb, std::integral_constant<int, (TT >= 4 ? 4 : 1)>{}, samec);
                    else if (TT >= 3 && nc == 3)
                        pass(cb, std::integral_constant<int, (TT >= 3 ? 3 : 1)>{}, samec);
                    else if (TT >= 2 && nc == 2)
                        pass(cb, std::integral_constant<int, (TT >= 2 ? 2 : 1)>{}, samec);
                    else
                        pass(cb, std::integral_constant<int, 1>{}, samec);
                };
                #pragma unroll 1
                for (int cb = 0; cb < ncm; cb += TT) {
                    if (same)
                        pass_n(cb, std::true_type{});
                    else
                        pass_n(cb, std::false_type{});
                }
                i += 2;
                m += 2;
                while (m >= rows) {
                    m -= rows;
                    v++;
                }
            }
            return;
        }
        // warp-uniform trip count: the chunk's item pairs (or items)
        #pragma unroll 1
        for (int q = c0i; q < c1i; q += step) {
            const bool live = i < c1i;
            int first = 0, ncols = 0;
            if (live)
                item_cols(v, first, ncols);
            const int r = i - ib0, d = r / P.SR;
            const uint8_t *wr = ring + (size_t)((d0 + sd0 + d) % a.NS) * a.stage_bytes + (size_t)(r - d * P.SR) * a.rbd;
            const int ncmax = two ? max(ncols, __shfl_xor_sync(FULL, ncols, 16)) : ncols;
            #pragma unroll 1
            for (int cb = 0; cb < ncmax; cb += TT) {
                float acc[TT];
                const uint32_t *xr[TT];
#pragma unroll
                for (int c = 0; c < TT; c++) {
                    acc[c] = 0.0f;
                    xr[c] = cb + c < ncols ? hrow(v, first, cb + c) : act;
                }
                const uint32_t wsa = smem_addr(live ? wr : ring);
                uint32_t xsa[TT];
#pragma unroll
                for (int c = 0; c < TT; c++)
                    xsa[c] = smem_addr(xr[c]);
                for (int jb = 0; jb < nbl; jb++) {
                    const int b = rowmap_block(dmap, lane, jb);
                    Q80Block wb;
                    load_q8_0_sh(wsa, b, wb);
#pragma unroll
                    for (int c = 0; c < TT; c++) {
                        if (cb + c < ncols) {
                            Q81Block xb;
                            load_q8_1_sh(xsa[c] + 4u * (uint32_t)xblock_word(b, hpad), xb);
                            acc[c] = fmaf(wb.d * xb.d, (float)dot_q8_block(wb.q, xb.q), acc[c]);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < TT; c++) {
                    if (cb + c < ncmax) {
                        const float y = two ? half_warp_sum(acc[c]) : warp_sum(acc[c]);
                        if ((two ? (lane & 15) : lane) == 0 && cb + c < ncols)
                            put(col_slot(v, first, cb + c), v, m, y);
                    }
                }
            }
            i += step;
            m += step;
            while (m >= rows) {
                m -= rows;
                v++;
            }
        }
    };
    auto release = [&](int da, int db, uint32_t cnt) {
        __syncwarp();
        if (lane == 0 && !dead)
            #pragma unroll 1
            for (int d = da; d < db; d++) {
                if (d > dw) {
                    // a stage this warp did not wait for: its slot's previous use
                    // is released by every warp once the stage is requested
                    const unsigned long long t0 = global_timer_ns();
                    while (*(volatile int *)&s_issued <= d0 + d) {
                        if (*(volatile int *)&s_abort || global_timer_ns() - t0 > WAIT_LIMIT_NS)
                            break;
                        __nanosleep(64);
                    }
                    __threadfence_block();
                }
                mbar_arrive_count(&empty[(d0 + d) % a.NS], cnt);
            }
    };
    // flat items [it0, it1) of the list over (v, n), n < H; y to the workspace
    {
        const int it0 = (int)P.it0, ni = (int)(P.it1 - P.it0);
        auto hrow = [&](int v, int, int c) -> const uint32_t * {
            return act + (size_t)((v - v_lo) * T + c) * a.hstride;
        };
        auto put = [&](int slot, int, int n, float y) { a.ws_y[(size_t)slot * a.H + n] = y; };
        if (!two) {
            // As the gate/up parts: down stage d goes to consumer group d mod
            // NG, whose RU warps each take a contiguous quarter (1 / RU) of its
            // items and release the stage with CW / RU arrivals each, so the
            // groups run on their own and the producer refills a slot as soon
            // as its group is done with it.
            const int grp = warp / a.RU, wl = warp - grp * a.RU;
            #pragma unroll 1
            for (int d = grp; d < P.NPd; d += a.NG) {
                down_items(it0 + d * P.SR, it0 + min(ni, (d + 1) * P.SR), it0, 0, a.H, hrow, put, wl, a.RU);
                release(d, d + 1, (uint32_t)(CW / a.RU));
            }
        } else {
            // Rows go two to a warp: stages one at a time, each warp taking
            // its share of the stage's items, then releasing it, so the
            // producer keeps the rest of the ring in flight.
            #pragma unroll 1
            for (int w = 0; w < P.NPd; w++) {
                down_items(it0 + w * P.SR, it0 + min(ni, (w + 1) * P.SR), it0, 0, a.H, hrow, put, warp, CW);
                release(w, w + 1, 1u);
            }
        }
    }
    barrier(3); // every y value is stored
    combine(P.n0, P.nrows, [&](int slot, int m) { return __ldcg(a.ws_y + (size_t)slot * a.H + P.n0 + m); });
}

// The dynamic shared memory attribute, once per device and template instance
// (thread-safe).
template <int TT, bool FLAT>
luce_status launch_layer(const LayerArgs &a, cudaStream_t stream, size_t smem)
{
    static luce_host::SmemLimit limit;
    auto kern = k_moe_layer<TT, FLAT>;
    if (limit.raise(kern, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_UNSUPPORTED;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    if (occ < 1)
        return LUCE_ERR_UNSUPPORTED;
    // one CTA per SM whatever the shape, so every call sharing a barrier
    // count has the same grid
    const int grid = luce_host::sm_count();
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    luce_host::make_config(cfg, attr, dim3(grid), dim3(THREADS), smem, stream);
    attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
    attr[cfg.numAttrs].val.cooperative = 1;
    cfg.numAttrs++;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        limit.forget();
        return LUCE_ERR_CUDA;
    }
    return LUCE_OK;
}

} // namespace

using namespace luce_host;

extern "C" __attribute__((visibility("hidden"))) luce_status luce_internal_moe_layer_flat(const float *logits, const float *bias, const float *x,
                                      const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                                      const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_gate,
                                      const luce_block_q8_0 *ws_up, const luce_block_q8_0 *ws_down, int T, int E,
                                      int k, int H, int I, float clamp, int32_t *ids, float *weights,
                                      luce_block_q8_1 *xq, int32_t *counts, int32_t *offsets, int32_t *routes,
                                      float *h, luce_block_q8_1 *hq, float *out, void *workspace,
                                      size_t workspace_bytes, void *stream)
{
    if (T < 0 || E < 1 || k < 1 || k > E || k > 64 || H <= 0 || I <= 0 || H % 256 != 0 || I % 256 != 0 ||
        H / 32 > 1024 || I / 32 > 1024 || !(clamp == clamp))
        return LUCE_ERR_INVALID_ARG;
    const bool has_ws = ws_gate != nullptr;
    if ((ws_up != nullptr) != has_ws || (ws_down != nullptr) != has_ws)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!logits || !x || !w_gate || !w_up || !w_down || !ids || !weights || !xq || !counts || !offsets || !routes ||
        !h || !hq || !out || !workspace)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || (bias && !aligned(bias, 4)) || !aligned(x, 16) || !aligned(w_gate, 16) ||
        !aligned(w_up, 16) || !aligned(w_down, 16) ||
        (has_ws && (!aligned(ws_gate, 16) || !aligned(ws_up, 16) || !aligned(ws_down, 16))) || !aligned(ids, 4) ||
        !aligned(weights, 4) || !aligned(xq, 4) || !aligned(counts, 4) || !aligned(offsets, 4) ||
        !aligned(routes, 4) || !aligned(h, 16) || !aligned(hq, 16) || !aligned(out, 4) || !aligned(workspace, 16))
        return LUCE_ERR_INVALID_ARG;
    if (T > MAX_T || T * k > MAX_R || E > MAX_E)
        return LUCE_ERR_UNSUPPORTED;

    LayerArgs a;
    a.logits = logits;
    a.bias = bias;
    a.x = x;
    a.wg = reinterpret_cast<const uint8_t *>(w_gate);
    a.wu = reinterpret_cast<const uint8_t *>(w_up);
    a.wd = reinterpret_cast<const uint8_t *>(w_down);
    a.wsg = reinterpret_cast<const uint8_t *>(ws_gate);
    a.wsu = reinterpret_cast<const uint8_t *>(ws_up);
    a.wsd = reinterpret_cast<const uint8_t *>(ws_down);
    a.T = T;
    a.E = E;
    a.k = k;
    a.H = H;
    a.I = I;
    a.clamp = clamp;
    a.ids = ids;
    a.weights = weights;
    a.xq = reinterpret_cast<uint32_t *>(xq);
    a.counts = counts;
    a.offsets = offsets;
    a.routes = routes;
    a.h = h;
    a.hq = reinterpret_cast<uint32_t *>(hq);
    a.out = out;
    a.sync = reinterpret_cast<unsigned long long *>(workspace);
    a.nbH = H / 32;
    a.nbI = I / 32;
    a.rbg = a.nbH * Q8_0_BYTES;
    a.rbd = a.nbI * Q8_0_BYTES;
    a.evict_first = g_tuning.evict_first;
    const int nb = sm_count();
    const int nslots = T * k + (has_ws ? T : 0);
    // activation rows (x during gate/up, then hq) in shared memory, padded so
    // that the row mappings' loads spread over the banks
    const bool gpairs = a.nbH % 64 == 0;
    a.xstride = a.nbH * Q8_1_WORDS + (gpairs ? 16 * (a.nbH / 32) : 0);
    const int dmap = a.nbI == 32 ? 1 : (a.nbI % 64 == 0) ? 2 : 0;
    a.hstride = a.nbI * Q8_1_WORDS + (dmap == 2 ? 16 * (a.nbI / 32) : dmap == 1 ? 16 : 0);
    a.hstride = (a.hstride + 3) & ~3; // rows 16-byte aligned
    // Down work: an equal share of the flat (expert, row) item list per CTA,
    // the hq rows of the few experts it touches in shared memory, y through
    // the workspace.
    a.flat = 1;
    {
        // a CTA's cost share over the cheapest items (cost DN_ROW_COST + 1
        // each, of at most DN_ROW_COST + T)
        const long long nv_max = std::min(E, T * k) + (has_ws ? 1 : 0);
        const long long items_max =
            ((long long)(DN_ROW_COST + T) * nv_max * H + (DN_ROW_COST + 1LL) * nb - 1) / ((DN_ROW_COST + 1LL) * nb) +
            1;
        const int span = (int)((items_max + H - 1) / H) + 1; // experts a range of items_max can touch
        a.hq_rows = span * T;
    }
    a.ws_y = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + 16);
    const int max_rows = (H + nb - 1) / nb;
    a.RB = std::min(RB_MAX, max_rows);
    const size_t act_bytes = 4 * std::max((size_t)T * a.xstride, (size_t)a.hq_rows * a.hstride);
    const size_t fixed = act_bytes +
                         (size_t)2 * T * E * sizeof(float);
    const size_t budget = (size_t)g_tuning.layer_budget_kb * 1024;
    // Gate/up parts of RU row pairs: RU gate rows and RU up rows, one bulk
    // copy each, RU warps per consumer group.  The copy engine of an SM keeps
    // about four bulk copies in flight (measured on GB300: four 16 KB copies
    // per SM reach ~7 TB/s, four 4 KB copies ~2.3 TB/s), so a copy should be
    // at least 16 KB: the smallest RU <= 16 with RU rbg >= 16 KB, halved while
    // the ring holds fewer than two stages.  CW / RU consumer groups take the
    // parts round-robin and share every slot of the ring.
    if (budget < fixed + 2 * ((size_t)std::max(2 * a.rbg, a.rbd) + 16))
        return LUCE_ERR_UNSUPPORTED;
    const size_t ring = budget - fixed;
    int RU = 1;
    while (RU < 16 && (size_t)RU * a.rbg < 16 * 1024)
        RU *= 2;
    while (RU > 1 && ring / ((size_t)std::max(2 * RU * a.rbg, a.rbd) + 16) < 2)
        RU /= 2;
    a.RU = RU;
    a.stage_bytes = std::max(2 * RU * a.rbg, a.rbd);
    const int ns = (int)std::min<size_t>(32, ring / ((size_t)a.stage_bytes + 16));
    a.NG = CW / RU; // consumer groups share the slots (ordered by the producer's request count)
    a.SR = a.stage_bytes / a.rbd;
    a.NS = ns;
    if (a.NS < 2)
        return LUCE_ERR_UNSUPPORTED;
    const size_t smem = (size_t)a.NS * a.stage_bytes + (size_t)2 * a.NS * sizeof(uint64_t) + fixed;
    cudaStream_t st = as_stream(stream);
    // kernels by columns per expert (more go four at a time) and down split;
    // one token keeps its x blocks in registers when a row gives a lane at
    // most 4 of them
    const bool xregs = T == 1 && (a.nbH % 64 == 0 ? a.nbH / 32 : (a.nbH + 31) / 32) <= 4;
    if (xregs)
        return launch_layer<1, true>(a, st, smem);
    if (T <= 2)
        return launch_layer<2, true>(a, st, smem);
    return launch_layer<4, true>(a, st, smem);
}
