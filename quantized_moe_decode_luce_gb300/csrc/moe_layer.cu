// moe_layer.cu -- one whole routed-MoE FFN layer of a decode or verify step
// in ONE launch: router select + weights, the q8_1 quantization of the input,
// the expert grouping, the gate/up pair with its SwiGLU, the q8_1
// quantization of h, the down product and the masked route-weighted combine
// with the shared expert.  Its C-ABI entry point is luce_moe_layer.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving".  The arithmetic of every step is the one of the
// separate operations ([PR826] commits "fused DS4.1 decode kernels", "RDNA4
// Q8_0 gate/up pair" and "fused routed combine and q8_1 inputs for the hybrid
// owners"); each fused step repeats the replaced step's arithmetic in the same
// order, so the results equal those of luce_moe_prep + luce_moe_glu_pair +
// luce_moe_down_combine bit for bit.  The launch structure is our own:
//
//  * Every CTA routes the T <= 8 tokens itself (a few hundred logits) and
//    quantizes x into its own shared memory; CTA 0 also stores the routing
//    tables and xq.  Selection is by rank: expert e of token t takes slot
//    #{e' : (s_e', e') before (s_e, e)} when that is below k, which is the
//    (score descending, index ascending) order of the sequential selection.
//  * Work per CTA: an equal share of all gate/up ROWS of the active experts
//    (the shared expert last) and an equal share of the down output rows n,
//    so every CTA streams the same bytes.  One producer warp streams the
//    CTA's gate/up parts and then its down stages through a ring of
//    shared-memory stages with cp.async.bulk; the down rows do not depend on
//    h, so they arrive while the gate/up rows are computed.  Sixteen
//    consumer warps compute, in two groups that take alternate stages (the
//    ring has an even number of stages, so every use of a slot falls to the
//    same group, in order); they never issue copies.
//  * The gate/up part stores h in fp32.  The down product needs all of h:
//    each CTA arrives at a device-wide barrier.  The grid is launched
//    cooperatively, so all of its CTAs are resident at once and the barrier
//    cannot wait for a CTA that has not started.  Its state (a monotonic
//    arrival count) lives in caller memory and needs no reset, so graph
//    replays need no host update.  Its wait is bounded (LUCE_FAULT_TIMEOUT).
//  * Then h -> q8_1 (the q8_1 rule of the separate kernels): when all of hq
//    fits in 24 KB every CTA quantizes all of it into its own shared memory
//    (CTA 0 also stores it); otherwise each CTA quantizes and stores its
//    share and a second barrier follows.
//  * Each CTA computes its down rows from shared memory, keeps every y in
//    shared memory and combines out[t][n] in slot order with separately
//    rounded products and sums, then adds the shared expert.
//  * Warp sums use a reduce-scatter butterfly (several sums per pass) whose
//    additions pair the lanes exactly as a full butterfly does, so every sum
//    is bitwise the one of the separate kernels.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_layer)

namespace {

using namespace luce;

// Consumer warps in two groups of GW that take alternate ring stages; warp CW
// streams the weights.  Named barriers: 1 + group (a group), 3 (all consumers).
constexpr int GW = 8;
constexpr int CW = 2 * GW;
constexpr int GTHREADS = GW * 32;
constexpr int CTHREADS = CW * 32;
constexpr int THREADS = CTHREADS + 32;
constexpr int BAR_ALL = 3;
constexpr int BAR_ROUTE = 4;                 // the routing warps GW .. CW
constexpr int RTHREADS = THREADS - GTHREADS; // routing threads (E <= this)
constexpr int MAX_T = 8;
constexpr int MAX_R = 64;  // T * k
constexpr int MAX_E = 256; // one thread per expert in the grouping
constexpr int MAX_V = MAX_R + 1;
constexpr int RB_MAX = 64; // down rows per row block (y buffer rows)
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
    unsigned long long *sync; // arrivals of every barrier (monotonic)
    int nbH, nbI, rbg, rbd;
    int RU;          // gate/up rows per part
    int stage_bytes; // one ring stage
    int NS;          // ring stages
    int SR;          // down rows per stage
    int hs_on;       // every CTA holds all of hq in shared memory
    int hs_own;      // ... quantized by itself from h (else staged from hq after a second barrier)
    int hq_bulk;     // stage hq with one bulk copy (else 16-byte loads)
    int prefetch;
    int evict_first;
};

// Device-wide barrier of the n CTAs of a cooperative grid, called by one
// thread per CTA after a CTA barrier that follows the CTA's stores (the
// release of the arrival covers them).  `count` (64-bit, never wraps) only
// grows: every barrier of every launch adds n, and all launches that share it
// have the same n.  A CTA reads c before arriving; the CTAs already counted
// in this barrier do not change floor(c / n), so the barrier ends when the
// count reaches (floor(c / n) + 1) n.  Arrival is a reduction (no reply to
// wait for).  Returns false if the wait ran out (never in a correct run).
__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ bool grid_barrier(unsigned long long *count, unsigned n)
{
    const unsigned long long c0 = ld_acquire_gpu_u64(count);
    const unsigned long long target = (c0 / n + 1ull) * n;
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(count) : "memory");
    const unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; i++) {
        if (ld_acquire_gpu_u64(count) >= target)
            return true;
        if ((i & 15u) == 0u && global_timer_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// Warp sums of four values per lane: lane L ends with the sum of
// v[(L >> 3) & 3].  Each addition pairs the same lanes, in the same order, as
// the full butterfly of warp_sum, so each sum is bitwise warp_sum's.
__device__ __forceinline__ float reduce4(float v0, float v1, float v2, float v3, int lane)
{
    const bool h16 = lane & 16, h8 = lane & 8;
    const float k0 = (h16 ? v2 : v0) + __shfl_xor_sync(FULL, h16 ? v0 : v2, 16);
    const float k1 = (h16 ? v3 : v1) + __shfl_xor_sync(FULL, h16 ? v1 : v3, 16);
    float k = (h8 ? k1 : k0) + __shfl_xor_sync(FULL, h8 ? k0 : k1, 8);
    k += __shfl_xor_sync(FULL, k, 4);
    k += __shfl_xor_sync(FULL, k, 2);
    k += __shfl_xor_sync(FULL, k, 1);
    return k;
}

// q8_1 rule for one block held by 4 lanes (lane 4i + j holds x[8j .. 8j+7] of
// block i of the warp's 8): the same arithmetic as quantize_q8_1_warp (the
// maximum and the integer sum do not depend on the order).
__device__ __forceinline__ void quantize_q8_1_quad(const float (&v)[8], bool valid, uint32_t *out_words, int qj)
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
    out_words[1 + 2 * qj] = w0;
    out_words[2 + 2 * qj] = w1;
    if (qj == 0) {
        const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
        const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sum)));
        out_words[0] = d16 | (s16 << 16);
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

// A gate/up part: rows [row, row + len) of virtual expert v (len <= RU, not
// crossing an expert).  Parts follow each other over the CTA's row range.
struct Part {
    int v, row, len;
};

__device__ __forceinline__ Part part_at(int gr, int r1, int I, int RU)
{
    Part p;
    p.v = gr / I;
    p.row = gr - p.v * I;
    p.len = min(min(RU, I - p.row), r1 - gr);
    return p;
}

template <int NC>
__global__ void __launch_bounds__(THREADS, 1) k_moe_layer(const LayerArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * a.stage_bytes);
    uint64_t *empty = full + a.NS;
    uint32_t *xs = reinterpret_cast<uint32_t *>(empty + a.NS); // [T][nbH][9], 16-byte aligned
    const int R = a.T * a.k;
    const int nslots = R + a.T;
    // x rows: block g of token t at word t * xstride + 9 g + xpad (g / 32): blocks g
    // and g + 32, read by one load instruction, sit 16 banks apart
    const int gmap = (a.nbH % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN; // gate/up row mapping
    const int xpad = gmap == ROWMAP_PAIRS ? 16 : 0;
    const int xstride = a.nbH * Q8_1_WORDS + xpad * (a.nbH >> 5);
    uint32_t *hs = xs + (size_t)a.T * xstride; // [nslots][nbI][9]
    float *ybuf = reinterpret_cast<float *>(hs + (a.hs_on ? (size_t)nslots * a.nbI * Q8_1_WORDS : 0)); // [nslots][RB]
    float *scores = ybuf + (size_t)nslots * RB_MAX; // [T][E] logit + bias
    float *lsm = scores + (size_t)a.T * a.E;        // [T][E] logits

    __shared__ int ids_s[MAX_R], pos_s[MAX_R], routes_s[MAX_R];
    __shared__ float w_s[MAX_R];
    __shared__ int cnt_s[MAX_E], off_s[MAX_E + 1];
    __shared__ int v_e[MAX_V], v_first[MAX_V], v_ncols[MAX_V];
    __shared__ int wcnt[RTHREADS / 32];
    __shared__ int s_abort;
    __shared__ int s_xnext; // next x block to quantize
    __shared__ int s_nvr;   // routed virtual experts
    __shared__ __align__(8) uint64_t hq_bar; // the bulk copy of hq

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, k = a.k;
    const bool cta0 = blockIdx.x == 0;
    const int nb = gridDim.x, bx = blockIdx.x;
    const int half_bytes = a.RU * a.rbg;
    // This CTA's slice of the shared expert's gate/up rows, [s0, s1): it does
    // not depend on the routing, so its parts are requested at once and (for
    // a single pass of x) computed while the other warps route.
    const int s0 = a.wsg ? (int)((unsigned)(a.I * bx) / (unsigned)nb) : 0;
    const int s1 = a.wsg ? (int)((unsigned)(a.I * (bx + 1)) / (unsigned)nb) : 0;
    const int NPs = (s1 - s0 + a.RU - 1) / a.RU; // shared parts: RU rows each, the last shorter
    const int NPe = min(NPs, a.NS);              // of them requested before the routing
    const int nbx = T * a.nbH;                   // x blocks
    const bool early = NPe > 0 && nbx <= GTHREADS / 4; // group 0 quantizes x in one pass, then takes them
    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();
    auto issue_shared = [&](int qq) {
        const uint32_t slot = (uint32_t)(qq % a.NS);
        uint8_t *dst = ring + (size_t)slot * a.stage_bytes;
        const int row = s0 + qq * a.RU, len = min(a.RU, s1 - row);
        const uint32_t bytes = (uint32_t)(len * a.rbg);
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        bulk_copy_g2s(dst, a.wsg + (size_t)row * a.rbg, bytes, &full[slot], pol);
        bulk_copy_g2s(dst + half_bytes, a.wsu + (size_t)row * a.rbg, bytes, &full[slot], pol);
    };
    if (tid == CTHREADS) {
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&hq_bar, 1);
        fence_mbar_init();
        s_abort = 0;
        s_xnext = 0;
    }
    __syncthreads(); // barriers initialized
    if (tid == CTHREADS) {
        // weights do not depend on the previous kernel: request them before waiting for it
        for (int qq = 0; qq < NPe; qq++)
            issue_shared(qq);
        if (a.wsd && a.prefetch) {
            // and warm L2 with this CTA's slice of the shared expert's down rows
            const size_t tot_d = (size_t)a.H * a.rbd; // a multiple of 16
            const size_t cd = ((tot_d / nb) + 15) & ~size_t(15);
            const size_t od = cd * bx;
            if (od < tot_d)
                prefetch_l2(a.wsd + od, (uint32_t)min(cd, tot_d - od));
        }
    }
    pdl_wait();
    pdl_trigger();

    // ---------------- consumer helpers ----------------
    const int grp = warp / GW, wl = warp - grp * GW; // consumer group, warp within it
    const int gtid = tid - grp * GTHREADS;
    bool dead = false;
    // waits for stage qq; false if this CTA gave up (now or earlier)
    auto wait_stage = [&](int qq) -> bool {
        // warp-uniform: every lane takes the same branch to the __all_sync
        if (__any_sync(FULL, *(volatile int *)&s_abort != 0))
            dead = true;
        if (dead)
            return false;
        const uint32_t slot = (uint32_t)(qq % a.NS), use = (uint32_t)(qq / a.NS);
        const bool got = __all_sync(FULL, mbar_wait_bounded(&full[slot], use & 1u));
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
    auto release_stage = [&](int qq) {
        named_barrier(1 + grp, GTHREADS); // every warp of the group is done with the stage
        if (gtid == 0 && !dead)
            mbar_arrive(&empty[qq % a.NS]);
    };
    auto cta_barrier = [&]() {
        named_barrier(BAR_ALL, CTHREADS);
        if (tid == 0 && !grid_barrier(a.sync, gridDim.x)) {
            atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
            *(volatile int *)&s_abort = 1;
        }
        named_barrier(BAR_ALL, CTHREADS);
    };

    // x -> q8_1 into shared memory (CTA 0 also stores xq): a warp claims 8
    // blocks at a time, 4 lanes per block
    auto quantize_x = [&]() {
        const int qj = lane & 3;
        for (;;) { // warp-uniform trip count
            int base = 0;
            if (lane == 0)
                base = atomicAdd(&s_xnext, 8);
            base = __shfl_sync(FULL, base, 0);
            if (base >= nbx)
                break;
            const int b = base + (lane >> 2);
            const bool valid = b < nbx;
            float v[8];
            if (valid) {
                load8(a.x + (size_t)b * QK + qj * 8, v, false);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    v[i] = 0.0f;
            }
            const int bt = valid ? b / a.nbH : 0, bg = valid ? b - bt * a.nbH : 0;
            uint32_t *dst = xs + (size_t)bt * xstride + (size_t)bg * Q8_1_WORDS + xpad * (bg >> 5);
            quantize_q8_1_quad(v, valid, dst, qj);
            if (cta0 && valid) {
                uint32_t *g = a.xq + (size_t)b * Q8_1_WORDS;
                g[1 + 2 * qj] = dst[1 + 2 * qj]; // this lane's own words
                g[2 + 2 * qj] = dst[2 + 2 * qj];
                if (qj == 0)
                    g[0] = dst[0];
            }
        }
    };

    // one token (NC == 1): this lane's x blocks stay in registers for every row
    constexpr int XR = 4;
    const int nblg = rowmap_blocks(gmap, a.nbH, lane);
    const bool x_regs = NC == 1 && a.T == 1 && nblg <= XR;
    Q81Block xreg[XR];
    auto load_xregs = [&]() {
#pragma unroll
        for (int j = 0; j < XR; j++) {
            if (x_regs && j < nblg) {
                const int b = rowmap_block(gmap, lane, j);
                load_q8_1_any(xs + (size_t)b * Q8_1_WORDS + xpad * (b >> 5), xreg[j]);
            } else {
                xreg[j].d = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; i++)
                    xreg[j].q[i] = 0;
            }
        }
    };

    // gate/up rows [row, row + len) of one part in stage qq -> h; columns of
    // a routed expert (first, ncols) or, routed == false, the T shared tokens
    auto glu_part = [&](int qq, int row0, int len, bool routed, int first, int ncols) {
        if (wait_stage(qq)) {
            const uint8_t *st = ring + (size_t)(qq % a.NS) * a.stage_bytes;
            for (int i = wl; i < len; i += GW) {
                const int row = row0 + i;
                const uint8_t *grow = st + (size_t)i * a.rbg;
                const uint8_t *urow = st + half_bytes + (size_t)i * a.rbg;
                for (int c0 = 0; c0 < ncols; c0 += NC) {
                    const int nc = min(NC, ncols - c0);
                    const uint32_t *xc[NC];
                    int rr[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++) {
                        const int cc = c0 + (c < nc ? c : 0);
                        rr[c] = routed ? routes_s[first + cc] : R + cc; // h row
                        xc[c] = xs + (size_t)(routed ? rr[c] / k : cc) * xstride;
                    }
                    float ag[NC], au[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++)
                        ag[c] = au[c] = 0.0f;
                    if (x_regs) {
                        // one token: its x blocks are in registers
#pragma unroll
                        for (int j = 0; j < XR; j++) {
                            if (j < nblg) {
                                const int b = rowmap_block(gmap, lane, j);
                                Q80Block gbk, ubk;
                                load_q8_0_smem(grow, b, gbk);
                                load_q8_0_smem(urow, b, ubk);
                                const int sg = dot_q8_block(gbk.q, xreg[j].q);
                                const int su = dot_q8_block(ubk.q, xreg[j].q);
                                ag[0] = fmaf(gbk.d * xreg[j].d, (float)sg, ag[0]);
                                au[0] = fmaf(ubk.d * xreg[j].d, (float)su, au[0]);
                            }
                        }
                    } else {
                        for (int j = 0; j < nblg; j++) {
                            const int b = rowmap_block(gmap, lane, j);
                            Q80Block gbk, ubk;
                            load_q8_0_smem(grow, b, gbk);
                            load_q8_0_smem(urow, b, ubk);
#pragma unroll
                            for (int c = 0; c < NC; c++) {
                                if (c < nc) {
                                    Q81Block xb;
                                    load_q8_1_any(xc[c] + (size_t)b * Q8_1_WORDS + xpad * (b >> 5), xb);
                                    const int sg = dot_q8_block(gbk.q, xb.q);
                                    const int su = dot_q8_block(ubk.q, xb.q);
                                    ag[c] = fmaf(gbk.d * xb.d, (float)sg, ag[c]);
                                    au[c] = fmaf(ubk.d * xb.d, (float)su, au[c]);
                                }
                            }
                        }
                    }
                    // two columns per pass: g0, u0, g1, u1 at lanes 0, 8, 16, 24
#pragma unroll
                    for (int c = 0; c < NC; c += 2) {
                        if (c < nc) {
                            const bool two = c + 1 < nc;
                            const float g1 = two ? ag[(c + 1) % NC] : 0.0f;
                            const float u1 = two ? au[(c + 1) % NC] : 0.0f;
                            const float sm = reduce4(ag[c], au[c], g1, u1, lane);
                            const float u = __shfl_down_sync(FULL, sm, 8); // lane 0: u0, lane 16: u1
                            if (lane == 0)
                                a.h[(size_t)rr[c] * a.I + row] = swiglu(sm, u, a.clamp);
                            if (two && lane == 16)
                                a.h[(size_t)rr[(c + 1) % NC] * a.I + row] = swiglu(sm, u, a.clamp);
                        }
                    }
                }
            }
        }
        release_stage(qq);
    };

    // ---------------- 1-3. x -> q8_1 (warps 0 .. GW-1) while warps GW .. CW route ----------------
    if (warp < GW) {
        quantize_x();
        if (early) {
            named_barrier(1, GTHREADS); // all of x is quantized (one pass, by this group)
            load_xregs();
            for (int qq = 0; qq < NPe; qq += 2) { // group 0's stages: the even ones
                const int row = s0 + qq * a.RU;
                glu_part(qq, row, min(a.RU, s1 - row), false, 0, T);
            }
        }
    } else {
        const int rt = tid - GTHREADS;      // routing threads 0 .. RTHREADS-1
        const int rw = warp - GW;           // routing warp
        for (int i = rt; i < T * E; i += RTHREADS) {
            const float l = a.logits[i];
            lsm[i] = l;
            scores[i] = a.bias ? __fadd_rn(l, a.bias[i % E]) : l;
        }
        for (int i = rt; i < R; i += RTHREADS)
            ids_s[i] = -1;
        named_barrier(BAR_ROUTE, RTHREADS);
        // selection by rank, 4 threads per (token, expert)
        {
            const int npair = T * E;
            const int qj = lane & 3;
            const int qE = (E + 3) >> 2;
            for (int base = 0; base < npair; base += RTHREADS / 4) { // warp-uniform trip count
                const int p = base + (rt >> 2);
                int rank = 0;
                int t = 0, e = 0;
                if (p < npair) {
                    t = p / E;
                    e = p - t * E;
                    const float *sc = scores + (size_t)t * E;
                    const float v = sc[e];
                    const int e_end = min(E, (qj + 1) * qE);
                    for (int e2 = qj * qE; e2 < e_end; e2++) {
                        const float o = sc[e2];
                        rank += (o > v || (o == v && e2 < e)) ? 1 : 0;
                    }
                }
                rank += __shfl_xor_sync(FULL, rank, 1);
                rank += __shfl_xor_sync(FULL, rank, 2);
                if (p < npair && qj == 0 && rank < k)
                    ids_s[t * k + rank] = e;
            }
        }
        named_barrier(BAR_ROUTE, RTHREADS);
        // weights (routing warp t) and grouping
        if (rw < T) {
            const int t = rw;
            float sel0 = 0.0f, sel1 = 0.0f;
            if (lane < k) {
                const int e = ids_s[t * k + lane];
                sel0 = e >= 0 ? lsm[t * E + e] : 0.0f;
            }
            if (lane + 32 < k) {
                const int e = ids_s[t * k + lane + 32];
                sel1 = e >= 0 ? lsm[t * E + e] : 0.0f;
            }
            route_softmax_warp(sel0, sel1, k, w_s + t * k, lane);
        }
        if (rt < R) {
            // slot of route r in the (expert, route) order; masked routes have none
            const int e = ids_s[rt];
            int pos = -1;
            if (e >= 0) {
                pos = 0;
                for (int r2 = 0; r2 < R; r2++) {
                    const int e2 = ids_s[r2];
                    pos += (e2 >= 0 && (e2 < e || (e2 == e && r2 < rt))) ? 1 : 0;
                }
            }
            pos_s[rt] = pos;
        }
        {
            const int e = rt; // E <= RTHREADS
            int c = 0, o = 0;
            if (e < E) {
                for (int r2 = 0; r2 < R; r2++) {
                    const int e2 = ids_s[r2];
                    c += e2 == e ? 1 : 0;
                    o += (e2 >= 0 && e2 < e) ? 1 : 0;
                }
                cnt_s[e] = c;
                off_s[e] = o;
            }
            if (e == 0) {
                int nvalid = 0;
                for (int r2 = 0; r2 < R; r2++)
                    nvalid += ids_s[r2] >= 0 ? 1 : 0;
                off_s[E] = nvalid;
            }
            const unsigned bal = __ballot_sync(FULL, e < E && c > 0);
            if (lane == 0)
                wcnt[rw] = __popc(bal);
        }
        named_barrier(BAR_ROUTE, RTHREADS);
        if (rt < R) {
            if (pos_s[rt] >= 0)
                routes_s[pos_s[rt]] = rt;
            if (rt >= off_s[E])
                routes_s[rt] = -1;
        }
        {
            const int e = rt;
            const bool act = e < E && cnt_s[e] > 0;
            const unsigned bal = __ballot_sync(FULL, act);
            int before = __popc(bal & ((1u << lane) - 1u));
            for (int w = 0; w < rw; w++)
                before += wcnt[w];
            if (act) {
                v_e[before] = e;
                v_first[before] = off_s[e];
                v_ncols[before] = cnt_s[e];
            }
            if (rt == 0) {
                int nvr = 0;
                for (int w = 0; w < RTHREADS / 32; w++)
                    nvr += wcnt[w];
                s_nvr = nvr;
                if (a.wsg) {
                    v_e[nvr] = E;
                    v_first[nvr] = 0;
                    v_ncols[nvr] = T;
                }
            }
        }
        named_barrier(BAR_ROUTE, RTHREADS);
        if (cta0) {
            for (int i = rt; i < R; i += RTHREADS) {
                a.ids[i] = ids_s[i];
                a.weights[i] = w_s[i];
                a.routes[i] = routes_s[i];
            }
            for (int e = rt; e < E; e += RTHREADS) {
                a.counts[e] = cnt_s[e];
                a.offsets[e] = off_s[e];
            }
            if (rt == 0)
                a.offsets[E] = off_s[E];
        }
        if (!early)
            quantize_x(); // what is left of x (with the early stage, group 0 alone quantizes all of it)
    }
    __syncthreads(); // routing tables and all of x are in shared memory

    // ---------------- 4. this CTA's work ----------------
    // gate/up: the shared slice [s0, s1), then the routed rows [r0, r1) of all
    // NVr * I routed rows (expert major); down output rows [dn0, dn1)
    // (unsigned 32-bit: NVr * I <= 64 * 32768 rows, times at most 1024 CTAs < 2^32)
    const int NVr = s_nvr;
    const int NV = NVr + (a.wsg ? 1 : 0);
    const int NRr = NVr * a.I;
    const int r0 = (int)((unsigned)(NRr * bx) / (unsigned)nb), r1 = (int)((unsigned)(NRr * (bx + 1)) / (unsigned)nb);
    const int dn0 = a.H * bx / nb, dn1 = a.H * (bx + 1) / nb;
    // down rows in nrb row blocks of rpb rows (the last may be shorter); a row
    // block's NV * rows items (expert major) are cut into stages of SR rows
    const int SR = a.SR;
    int nrb, rpb, rlast, spr, slast, NPd;
    auto plan_down = [&]() {
        const int nrows = dn1 - dn0;
        nrb = (nrows + RB_MAX - 1) / RB_MAX;
        rpb = nrb ? (nrows + nrb - 1) / nrb : 0;
        rlast = nrows - (nrb - 1) * rpb;
        spr = nrb ? (NV * rpb + SR - 1) / SR : 0;     // stages of a full row block
        slast = nrb ? (NV * rlast + SR - 1) / SR : 0; // stages of the last one
        NPd = nrb ? (nrb - 1) * spr + slast : 0;
    };
    auto down_stage = [&](int d, int &rb, int &sp) {
        rb = d / max(spr, 1);
        if (rb >= nrb - 1) {
            rb = nrb - 1;
            sp = d - (nrb - 1) * spr;
        } else {
            sp = d - rb * spr;
        }
    };

    if (warp == CW) {
        // ---------------- the producer: every stage of this CTA, in order ----------------
        if (lane != 0)
            return;
        int NPg = NPs;
        for (int gr = r0; gr < r1; NPg++)
            gr += part_at(gr, r1, a.I, a.RU).len;
        plan_down();
        const int NP = NPg + NPd;
        int gr = r0;
        int issued = NPe; // the first shared parts went out before the routing
        for (; issued < NP; issued++) {
            const uint32_t slot = (uint32_t)(issued % a.NS), use = (uint32_t)(issued / a.NS);
            if (use > 0 && !mbar_wait_bounded(&empty[slot], (use - 1) & 1u)) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
                break;
            }
            if (*(volatile int *)&s_abort)
                break;
            uint8_t *dst = ring + (size_t)slot * a.stage_bytes;
            if (issued < NPs) {
                issue_shared(issued);
            } else if (issued < NPg) {
                const Part pt = part_at(gr, r1, a.I, a.RU);
                gr += pt.len;
                const int e = v_e[pt.v];
                const uint8_t *gsrc = a.wg + ((size_t)e * a.I + pt.row) * a.rbg;
                const uint8_t *usrc = a.wu + ((size_t)e * a.I + pt.row) * a.rbg;
                const uint32_t bytes = (uint32_t)(pt.len * a.rbg);
                mbar_arrive_expect_tx(&full[slot], 2 * bytes);
                bulk_copy_g2s(dst, gsrc, bytes, &full[slot], pol);
                bulk_copy_g2s(dst + half_bytes, usrc, bytes, &full[slot], pol);
            } else {
                int rb, sp;
                down_stage(issued - NPg, rb, sp);
                const int nr0 = dn0 + rb * rpb;
                const int rows = rb == nrb - 1 ? rlast : rpb;
                const int i0 = sp * SR, i1 = min(NV * rows, i0 + SR);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)((i1 - i0) * a.rbd));
                for (int i = i0; i < i1;) {
                    const int v = i / rows, m = i - v * rows;
                    const int cnt = min(i1 - i, rows - m);
                    const int e = v_e[v];
                    const uint8_t *src = e < E ? a.wd + ((size_t)e * a.H + nr0 + m) * a.rbd
                                               : a.wsd + (size_t)(nr0 + m) * a.rbd;
                    bulk_copy_g2s(dst + (size_t)(i - i0) * a.rbd, src, (uint32_t)(cnt * a.rbd), &full[slot], pol);
                    i += cnt;
                }
            }
        }
        // no bulk copy may still be writing shared memory when the CTA exits
        const int n_slots = issued < a.NS ? issued : a.NS;
        for (int sl = 0; sl < n_slots; sl++) {
            const int last_use = (issued - 1 - sl) / a.NS;
            if (!mbar_wait_bounded(&full[sl], (uint32_t)last_use & 1u))
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        }
        return;
    }

    // ---------------- 5. gate/up rows -> h (consumer warps) ----------------
    if (!(early && grp == 0))
        load_xregs();
    int q = 0;
    {
        int gr = r0;
        for (; q < NPs || gr < r1; q++) {
            if (q < NPs) {
                if ((q & 1) != grp || (early && grp == 0 && q < NPe))
                    continue; // the other group's stage, or one group 0 took before the routing
                const int row = s0 + q * a.RU;
                glu_part(q, row, min(a.RU, s1 - row), false, 0, T);
                continue;
            }
            const Part pt = part_at(gr, r1, a.I, a.RU);
            gr += pt.len;
            if ((q & 1) != grp)
                continue; // the other group's stage
            glu_part(q, pt.row, pt.len, true, v_first[pt.v], v_ncols[pt.v]);
        }
    }
    plan_down(); // q is now the first down stage

    // ---------------- 6. all of h is stored: h -> q8_1 ----------------
    cta_barrier();
    const int ibytes_w = a.nbI * Q8_1_WORDS; // words per hq row
    {
        // blocks u = (slot, g) of the live slots: the routes, then the shared
        // tokens.  All of them (every CTA, rotated so that the CTAs do not
        // all start on the same lines) or this CTA's share; the loads of four
        // passes are issued before any block is quantized.
        const int nlive = R + (a.wsd ? T : 0);
        const int U = nlive * a.nbI;
        const bool own = a.hs_on && a.hs_own;
        const int u0 = own ? 0 : (int)((long long)U * bx / nb);
        const int u1 = own ? U : (int)((long long)U * (bx + 1) / nb);
        const int rot = own ? (int)(((long long)bx * 67) % U) : 0;
        const int qj = lane & 3;
        constexpr int NQ = CTHREADS / 4; // quads of all consumer warps
        if (!*(volatile int *)&s_abort) {
            for (int base = u0; base < u1; base += 4 * NQ) { // warp-uniform trip count
                float v[4][8];
                int uu[4];
                bool val[4];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int w = base + j * NQ + (tid >> 2);
                    int u = w - u0 + rot;
                    u = (u >= u1 - u0 ? u - (u1 - u0) : u) + u0;
                    const int slot = u / a.nbI, g = u - slot * a.nbI;
                    uu[j] = u;
                    val[j] = w < u1 && (slot >= R || ids_s[slot] >= 0);
                    if (val[j]) {
                        load8(a.h + (size_t)slot * a.I + (size_t)g * QK + qj * 8, v[j], true); // other CTAs' h
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            v[j][i] = 0.0f;
                    }
                }
#pragma unroll 1
                for (int j = 0; j < 4; j++) {
                    // pass j's values by selects (one copy of the quantizer, no local memory)
                    float vj[8];
#pragma unroll
                    for (int i = 0; i < 8; i++)
                        vj[i] = j == 0 ? v[0][i] : j == 1 ? v[1][i] : j == 2 ? v[2][i] : v[3][i];
                    const bool ok = j == 0 ? val[0] : j == 1 ? val[1] : j == 2 ? val[2] : val[3];
                    if (!__any_sync(FULL, ok))
                        continue; // a warp with no block in this pass does no work
                    const int u = ok ? (j == 0 ? uu[0] : j == 1 ? uu[1] : j == 2 ? uu[2] : uu[3]) : 0;
                    uint32_t *dst = (own ? hs : a.hq) + (size_t)u * Q8_1_WORDS;
                    quantize_q8_1_quad(vj, ok, dst, qj);
                    if (own && cta0 && ok) {
                        uint32_t *gq = a.hq + (size_t)u * Q8_1_WORDS;
                        gq[1 + 2 * qj] = dst[1 + 2 * qj]; // this lane's own words
                        gq[2 + 2 * qj] = dst[2 + 2 * qj];
                        if (qj == 0)
                            gq[0] = dst[0];
                    }
                }
            }
        }
        if (own) {
            named_barrier(BAR_ALL, CTHREADS);
        } else {
            cta_barrier(); // every CTA's share of hq is stored
            if (a.hs_on && !*(volatile int *)&s_abort) {
                if (a.hq_bulk) {
                    // all of hq into shared memory with one bulk copy (the rows
                    // are multiples of 16 bytes); the proxy fence orders the
                    // other CTAs' stores, seen through the barrier, before it
                    const uint32_t bytes = (uint32_t)(nlive * ibytes_w * 4);
                    if (tid == 0) {
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        mbar_arrive_expect_tx(&hq_bar, bytes);
                        bulk_copy_g2s(hs, a.hq, bytes, &hq_bar, l2_evict_normal_policy());
                    }
                    if (!__all_sync(FULL, mbar_wait_bounded(&hq_bar, 0))) {
                        if (lane == 0) {
                            atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                            *(volatile int *)&s_abort = 1;
                        }
                    }
                } else {
                    // all of hq into shared memory: 16-byte loads at L2, each CTA
                    // starting at another offset (rows are multiples of 16 bytes)
                    const int n4 = nlive * ibytes_w / 4;
                    const int r4 = (int)(((long long)bx * 37) % n4);
                    const uint4 *src4 = reinterpret_cast<const uint4 *>(a.hq);
                    uint4 *dst4 = reinterpret_cast<uint4 *>(hs);
#pragma unroll 4
                    for (int i = tid; i < n4; i += CTHREADS) {
                        const int j = i + r4 < n4 ? i + r4 : i + r4 - n4;
                        dst4[j] = __ldcg(src4 + j);
                    }
                }
                named_barrier(BAR_ALL, CTHREADS);
            }
        }
    }

    // ---------------- 7. down rows, combine ----------------
    for (int d = 0; d < NPd; d++, q++) {
        int rb, sp;
        down_stage(d, rb, sp);
        const int nr0 = dn0 + rb * rpb;
        const int rows = rb == nrb - 1 ? rlast : rpb;
        const int i0 = sp * SR, i1 = min(NV * rows, i0 + SR);
        const bool mine = (q & 1) == grp;
        if (mine && wait_stage(q)) {
            const uint8_t *st = ring + (size_t)(q % a.NS) * a.stage_bytes;
            const uint32_t *xbase = a.hs_on ? hs : a.hq;
            const int ni = i1 - i0;
            if (a.nbI == 32) {
                // two rows per warp (ROWMAP_TWO_ROWS): half h of the warp walks the
                // items 2 p + h, p = wl, wl + GW, ..., and their columns, two units
                // per pass; a half-warp reduce-scatter leaves the sums at lanes
                // 0, 8 (half 0) and 16, 24 (half 1)
                const int h = lane >> 4;
                int p = wl, col = 0;
                const uint32_t *xlast = nullptr;
                Q81Block xb[2];
                while (__any_sync(FULL, 2 * p + h < ni)) { // warp-uniform trip count
                    const uint8_t *wr[2];
                    const uint32_t *xr[2];
                    int yo[2];
                    bool live[2];
#pragma unroll
                    for (int z = 0; z < 2; z++) {
                        const int it = 2 * p + h;
                        live[z] = it < ni;
                        wr[z] = st;
                        xr[z] = xbase;
                        yo[z] = 0;
                        if (live[z]) {
                            const int i = i0 + it;
                            const int v = i / rows, m = i - v * rows;
                            const int ys = v_e[v] < E ? routes_s[v_first[v] + col] : R + col; // hq row = y slot
                            wr[z] = st + (size_t)it * a.rbd;
                            xr[z] = xbase + (size_t)ys * ibytes_w;
                            yo[z] = ys * RB_MAX + m;
                            if (++col == v_ncols[v]) {
                                col = 0;
                                p += GW;
                            }
                        }
                    }
                    float acc[2] = {0.0f, 0.0f};
#pragma unroll
                    for (int z = 0; z < 2; z++) {
                        if (live[z]) {
                            if (xr[z] != xlast) { // this half's activation blocks, reloaded on a new hq row
                                xlast = xr[z];
#pragma unroll
                                for (int j = 0; j < 2; j++) {
                                    const uint32_t *xw = xr[z] + (size_t)rowmap_block(ROWMAP_TWO_ROWS, lane, j) * Q8_1_WORDS;
                                    if (a.hs_on) {
                                        load_q8_1_any(xw, xb[j]);
                                    } else {
                                        xb[j].d = half_bits_to_float(__ldcg(xw));
#pragma unroll
                                        for (int w = 0; w < 8; w++)
                                            xb[j].q[w] = (int)__ldcg(xw + 1 + w);
                                    }
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 2; j++) {
                                Q80Block wb;
                                load_q8_0_smem(wr[z], rowmap_block(ROWMAP_TWO_ROWS, lane, j), wb);
                                acc[z] = fmaf(wb.d * xb[j].d, (float)dot_q8_block(wb.q, xb[j].q), acc[z]);
                            }
                        }
                    }
                    const bool h8 = lane & 8;
                    float y = (h8 ? acc[1] : acc[0]) + __shfl_xor_sync(FULL, h8 ? acc[0] : acc[1], 8);
                    y += __shfl_xor_sync(FULL, y, 4);
                    y += __shfl_xor_sync(FULL, y, 2);
                    y += __shfl_xor_sync(FULL, y, 1);
                    const int z = (lane >> 3) & 1;
                    if ((lane & 7) == 0 && (z ? live[1] : live[0]))
                        ybuf[z ? yo[1] : yo[0]] = y;
                }
            } else {
                // 32 lanes per unit (item, column), four units per pass
                const int dmap = (a.nbI % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN;
                const int nbl = rowmap_blocks(dmap, a.nbI, lane);
                int it = wl, col = 0;
                while (it < ni) {
                    const uint8_t *wr[4];
                    const uint32_t *xr[4];
                    int yo[4];
                    int nu = 0;
#pragma unroll
                    for (int z = 0; z < 4; z++) {
                        wr[z] = st;
                        xr[z] = xbase;
                        yo[z] = 0;
                        if (it < ni) {
                            const int i = i0 + it;
                            const int v = i / rows, m = i - v * rows;
                            const int ys = v_e[v] < E ? routes_s[v_first[v] + col] : R + col; // hq row = y slot
                            wr[z] = st + (size_t)it * a.rbd;
                            xr[z] = xbase + (size_t)ys * ibytes_w;
                            yo[z] = ys * RB_MAX + m;
                            nu++;
                            if (++col == v_ncols[v]) {
                                col = 0;
                                it += GW;
                            }
                        }
                    }
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    for (int j = 0; j < nbl; j++) {
                        const int b = rowmap_block(dmap, lane, j);
                        Q81Block xb; // the activation block, kept while the units share their hq row
#pragma unroll
                        for (int z = 0; z < 4; z++) {
                            if (z < nu) {
                                Q80Block wb;
                                load_q8_0_smem(wr[z], b, wb);
                                if (z == 0 || xr[z] != xr[z - 1]) {
                                    const uint32_t *xw = xr[z] + (size_t)b * Q8_1_WORDS;
                                    if (a.hs_on) {
                                        load_q8_1_any(xw, xb);
                                    } else {
                                        xb.d = half_bits_to_float(__ldcg(xw));
#pragma unroll
                                        for (int w = 0; w < 8; w++)
                                            xb.q[w] = (int)__ldcg(xw + 1 + w);
                                    }
                                }
                                acc[z] = fmaf(wb.d * xb.d, (float)dot_q8_block(wb.q, xb.q), acc[z]);
                            }
                        }
                    }
                    const float y = reduce4(acc[0], acc[1], acc[2], acc[3], lane);
                    const int z = lane >> 3;
                    const int yz = z == 0 ? yo[0] : z == 1 ? yo[1] : z == 2 ? yo[2] : yo[3];
                    if ((lane & 7) == 0 && z < nu)
                        ybuf[yz] = y;
                }
            }
        }
        if (mine)
            release_stage(q);
        if (sp == (rb == nrb - 1 ? slast : spr) - 1) {
            named_barrier(BAR_ALL, CTHREADS); // both groups' y of the row block are in ybuf
            // out[t][n] = sum_j fl(w * y) in slot order, then + shared
            if (!dead && !*(volatile int *)&s_abort) {
                for (int idx = tid; idx < T * rows; idx += CTHREADS) {
                    const int t = idx / rows, m = idx - t * rows;
                    float acc = 0.0f;
                    for (int j = 0; j < k; j++) {
                        const int e = ids_s[t * k + j];
                        if (e >= 0)
                            acc = __fadd_rn(acc, __fmul_rn(w_s[t * k + j], ybuf[(t * k + j) * RB_MAX + m]));
                    }
                    if (a.wsd)
                        acc = __fadd_rn(acc, ybuf[(R + t) * RB_MAX + m]);
                    a.out[(size_t)t * a.H + nr0 + m] = acc;
                }
            }
            named_barrier(BAR_ALL, CTHREADS); // ybuf is free for the next row block
        }
    }
}

// Cooperative launch (every CTA resident at once), with the programmatic
// attribute when enabled.  The dynamic shared memory attribute is set once
// per device and template instance.
template <int NC>
luce_status launch_layer(const LayerArgs &a, cudaStream_t stream, size_t smem, int cps)
{
    static size_t smem_set[64] = {0};
    auto kern = k_moe_layer<NC>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return LUCE_ERR_CUDA;
    if (smem_set[dev] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return LUCE_ERR_UNSUPPORTED;
        }
        smem_set[dev] = smem;
    }
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, THREADS, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    if (occ < 1)
        return LUCE_ERR_UNSUPPORTED;
    const int grid = luce_host::sm_count() * std::min(occ, std::max(1, cps));
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    luce_host::make_config(cfg, attr, dim3(grid), dim3(THREADS), smem, stream);
    attr[cfg.numAttrs].id = cudaLaunchAttributeCooperative;
    attr[cfg.numAttrs].val.cooperative = 1;
    cfg.numAttrs++;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    return LUCE_OK;
}

} // namespace

using namespace luce_host;

extern "C" luce_status luce_moe_layer(const float *logits, const float *bias, const float *x,
                                      const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                                      const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_gate,
                                      const luce_block_q8_0 *ws_up, const luce_block_q8_0 *ws_down, int T, int E,
                                      int k, int H, int I, float clamp, int32_t *ids, float *weights,
                                      luce_block_q8_1 *xq, int32_t *counts, int32_t *offsets, int32_t *routes,
                                      float *h, luce_block_q8_1 *hq, float *out, uint32_t *sync, void *stream)
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
        !h || !hq || !out || !sync)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || (bias && !aligned(bias, 4)) || !aligned(x, 16) || !aligned(w_gate, 16) ||
        !aligned(w_up, 16) || !aligned(w_down, 16) ||
        (has_ws && (!aligned(ws_gate, 16) || !aligned(ws_up, 16) || !aligned(ws_down, 16))) || !aligned(ids, 4) ||
        !aligned(weights, 4) || !aligned(xq, 4) || !aligned(counts, 4) || !aligned(offsets, 4) ||
        !aligned(routes, 4) || !aligned(h, 16) || !aligned(hq, 16) || !aligned(out, 4) || !aligned(sync, 8))
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
    a.sync = reinterpret_cast<unsigned long long *>(sync);
    a.nbH = H / 32;
    a.nbI = I / 32;
    a.rbg = a.nbH * Q8_0_BYTES;
    a.rbd = a.nbI * Q8_0_BYTES;
    const Tuning &tu = g_tuning;
    // a gate/up part (RU gate rows + RU up rows) of about part_kb, but at
    // least one row per warp while a part stays under twice that
    int RU = 32;
    while (RU > 1 && 2 * RU * a.rbg > tu.layer_part_kb * 1024 &&
           !(RU <= CW && 2 * RU * a.rbg <= 2 * tu.layer_part_kb * 1024))
        RU /= 2;
    a.RU = RU;
    a.stage_bytes = std::max(2 * RU * a.rbg, a.rbd);
    a.SR = a.stage_bytes / a.rbd;
    a.prefetch = tu.layer_prefetch;
    a.evict_first = tu.evict_first;
    const int nslots = T * k + T;
    const size_t hs_bytes = (size_t)nslots * a.nbI * Q8_1_BYTES;
    a.hs_on = hs_bytes <= 24 * 1024 ? 1 : 0;
    a.hs_own = tu.layer_hs_own;
    a.hq_bulk = tu.layer_hq_bulk;
    const size_t xrow = (size_t)a.nbH * Q8_1_BYTES + (a.nbH % 64 == 0 ? (size_t)64 * (a.nbH / 32) : 0);
    const size_t fixed = (size_t)T * xrow + (a.hs_on ? hs_bytes : 0) +
                         (size_t)nslots * RB_MAX * sizeof(float) + (size_t)2 * T * E * sizeof(float);
    const size_t budget = (size_t)tu.layer_budget_kb * 1024;
    if (budget < fixed + 2 * ((size_t)a.stage_bytes + 16))
        return LUCE_ERR_UNSUPPORTED;
    a.NS = (int)std::min<size_t>(16, (budget - fixed) / ((size_t)a.stage_bytes + 16));
    a.NS -= a.NS & 1; // even: each slot always falls to the same consumer group
    const size_t smem = (size_t)a.NS * a.stage_bytes + (size_t)2 * a.NS * sizeof(uint64_t) + fixed;
    cudaStream_t st = as_stream(stream);
    if (T <= 1)
        return launch_layer<1>(a, st, smem, tu.layer_cps);
    if (T <= 2)
        return launch_layer<2>(a, st, smem, tu.layer_cps);
    if (T <= 4)
        return launch_layer<4>(a, st, smem, tu.layer_cps);
    return launch_layer<8>(a, st, smem, tu.layer_cps);
}
