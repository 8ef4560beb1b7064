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
//    A NaN score ranks below every number, so the order is total and every
//    token selects exactly k distinct experts.
//  * Gate/up work per CTA: an equal share of all 32-row groups of the active
//    experts (the shared expert last; a CTA takes its shared groups first).
//    A group is the span of one q8_1 block of h, so the CTA that computes a
//    group's h also quantizes it, in the group's epilogue, and stores h and
//    hq.  Down work per CTA: an equal share of the output rows n.
//  * One producer warp streams the CTA's stages through a ring of shared
//    memory with cp.async.bulk: two halves, one per consumer group of eight
//    warps (group c takes the CTA's groups j = c, c + 2, ...), each half a
//    queue of its own; after the gate/up parts come the down stages,
//    alternating between the halves.  The down rows do not depend on h, so
//    they arrive while h is computed.  The consumer warps never issue copies;
//    each warp releases a stage by its own arrival.
//  * With one token the routing yields k experts, so the plan is known
//    before the routing: the producer requests the first shared group at
//    once and starts on the routed experts as soon as the ranks exist.
//  * The down product needs all of hq: each CTA arrives at a device-wide
//    barrier.  The grid is launched cooperatively, so all of its CTAs are
//    resident at once and the barrier cannot wait for a CTA that has not
//    started.  Its state (a monotonic arrival count) lives in caller memory
//    and needs no reset, so graph replays need no host update.  Its wait is
//    bounded (LUCE_FAULT_TIMEOUT).  While thread 0 waits, the other warps
//    list the CTA's down work units (item, column).
//  * After the barrier each CTA copies all of hq into shared memory (one bulk
//    copy when it fits in 24 KB), computes its down rows from shared memory,
//    keeps every y in shared memory and combines out[t][n] in slot order with
//    separately rounded products and sums, then adds the shared expert.
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

// Consumer warps in two groups of GW, each with its half of the ring; warp CW
// streams the weights.  Named barriers: 1 + group (a group), 3 (all consumers).
constexpr int GW = 8;
constexpr int CW = 2 * GW;
constexpr int GTHREADS = GW * 32;
constexpr int CTHREADS = CW * 32;
constexpr int THREADS = CTHREADS + 32;
constexpr int BAR_ALL = 3;
constexpr int BAR_ROUTE = 4;                 // the routing warps GW .. CW
constexpr int BAR_TABLES = 5;                // routing done: the consumers wait (the producer arrives when T > 1)
constexpr int RTHREADS = THREADS - GTHREADS; // routing threads (E <= this)
constexpr int MAX_T = 8;
constexpr int MAX_R = 64;  // T * k
constexpr int MAX_E = 256; // experts (selection bit masks of MAX_E / 32 words)
constexpr int MAX_V = MAX_R + 1;
constexpr int RB_MAX = 64; // down rows per row block (y buffer rows)
constexpr int HB_STRIDE = MAX_T + 1; // h of a 32-row group: [32][HB_STRIDE]
constexpr int MAX_UNITS = 4 * 32 * HB_STRIDE / 2; // down work units listed in the h buffers (8 B each)
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
    int hs_on;       // every CTA stages all of hq in shared memory
    int hq_bulk;     // stage hq with one bulk copy (else 16-byte loads)
    int prefetch;
    int evict_first;
    int dsplit; // down rows by weight (else an even split)
    int psleep; // producer back-off (ns) while no slot is free
    int down_early; // down stages as soon as a slot is free (else after every gate/up part)
};

// Device-wide barrier of the n CTAs of a cooperative grid, called by one
// thread per CTA after a CTA barrier that follows the CTA's stores (the
// release of the arrival covers them).  `count` (64-bit, never wraps) only
// grows: every barrier of every launch adds n, and all launches that share it
// have the same n.  A CTA reads c0 at any time after the previous barrier on
// `count` has ended and before its own arrival (the kernel does it at its
// start); the CTAs already counted in this barrier do not change
// floor(c0 / n), so the barrier ends when the count reaches
// (floor(c0 / n) + 1) n.  Arrival is a reduction (no reply to wait for).
// Returns false if the wait ran out (never in a correct run).
__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait that parks the thread in hardware until the phase completes
// (or a 10 us suspend hint runs out), so a waiter wakes as soon as its data
// is there instead of after a back-off sleep.
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

__device__ bool grid_barrier(unsigned long long *count, unsigned n, unsigned long long c0)
{
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

// Warp sums of eight values per lane: lane L ends with the sum of
// v[(L >> 2) & 7].  As in reduce4, each addition pairs the same lanes, in the
// same order, as the butterfly of warp_sum, so each sum is bitwise warp_sum's.
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane)
{
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float k[4];
#pragma unroll
    for (int i = 0; i < 4; i++)
        k[i] = (h16 ? v[4 + i] : v[i]) + __shfl_xor_sync(FULL, h16 ? v[i] : v[4 + i], 16);
    float m[2];
#pragma unroll
    for (int i = 0; i < 2; i++)
        m[i] = (h8 ? k[2 + i] : k[i]) + __shfl_xor_sync(FULL, h8 ? k[i] : k[2 + i], 8);
    float n = (h4 ? m[1] : m[0]) + __shfl_xor_sync(FULL, h4 ? m[0] : m[1], 4);
    n += __shfl_xor_sync(FULL, n, 2);
    n += __shfl_xor_sync(FULL, n, 1);
    return n;
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

// This CTA's work (see make_plan in the kernel).
struct LayerPlan {
    int NVr, NV;            // routed virtual experts; all of them
    int g0, g1, nsh, ngr;   // gate/up groups [g0, g1), nsh shared ones, ngr in all
    int dn0, nrows;         // down rows [dn0, dn0 + nrows)
    int nrb, rpb, rlast;    // row blocks, their rows, the last one's rows
    int spr, slast, NPd;    // stages of a full row block, of the last one, in all
    int nglu0, nglu1, s1;   // gate/up parts of ring half 0 and 1; down stages start in half s1
    int nd0, nd1;           // down stages of half 0 and 1
};

// Row block and stage within it of down stage d.
__device__ __forceinline__ void down_stage(const LayerPlan &P, int d, int &rb, int &sp)
{
    rb = d / max(P.spr, 1);
    if (rb >= P.nrb - 1) {
        rb = P.nrb - 1;
        sp = d - (P.nrb - 1) * P.spr;
    } else {
        sp = d - rb * P.spr;
    }
}

// Ring half and sequence number within it of down stage d: the down stages
// alternate between the halves, starting with the half that has fewer
// gate/up parts (s = 1: half 1).
__device__ __forceinline__ void down_slot_of(const LayerPlan &P, int d, int &hh, int &n)
{
    hh = (d & 1) ^ P.s1;
    const int pos = d >> 1;
    n = (hh ? P.nglu1 : P.nglu0) + pos;
}

template <int NC>
__global__ void __launch_bounds__(THREADS, 1) k_moe_layer(const LayerArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * a.stage_bytes);
    uint64_t *empty = full + a.NS;
    uint32_t *xs = reinterpret_cast<uint32_t *>(empty + a.NS); // [T][xstride], 16-byte aligned
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
    float *hbuf = lsm + (size_t)a.T * a.E;          // [2 groups][2 buffers][32][HB_STRIDE]

    __shared__ int ids_s[MAX_R], routes_s[MAX_R];
    __shared__ float w_s[MAX_R];
    __shared__ int cnt_s[MAX_E], off_s[MAX_E + 1];
    __shared__ int v_e[MAX_V], v_first[MAX_V], v_ncols[MAX_V];
    __shared__ uint32_t sel_bits[MAX_T][MAX_E / 32]; // expert e selected by token t
    __shared__ int s_abort;
    __shared__ int s_xnext; // next x block to quantize
    __shared__ int s_nvr;   // routed virtual experts
    __shared__ __align__(8) uint64_t hq_bar; // the bulk copy of hq
    __shared__ unsigned long long s_c0;       // barrier count at the start

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, E = a.E, k = a.k;
    const bool cta0 = blockIdx.x == 0;
    const int nb = gridDim.x, bx = blockIdx.x;
    const int half_bytes = a.RU * a.rbg;
    const int G32 = a.I / 32;  // 32-row groups per expert
    const int PPG = 32 / a.RU; // parts per group
    const int HALF = a.NS / 2; // ring slots of each consumer group
    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();

    // This CTA's gate/up groups: [g0, g1) of all NV * G32 groups (virtual expert
    // major, the shared expert last), taken shared ones first; the j-th group
    // it takes goes to consumer group j % 2, each with its own half of the
    // ring.  No weight is requested before the routing: bulk copies in flight
    // hold back this SM's other memory accesses (the routing's loads of the
    // logits and of x among them), and requesting the shared expert's first
    // parts before the routing measured slower (20.9 vs 20.3 us per decode
    // layer).
    const int nbx = T * a.nbH; // x blocks
    // part p of a group: RU gate rows then RU up rows into half c, sequence n
    auto issue_part = [&](int c, int n, int gi, int p, const uint8_t *wg_e, const uint8_t *wu_e) {
        const uint32_t slot = (uint32_t)(c * HALF + n % HALF);
        uint8_t *dst = ring + (size_t)slot * a.stage_bytes;
        const size_t row = (size_t)(gi % G32) * 32 + (size_t)p * a.RU;
        const uint32_t bytes = (uint32_t)(a.RU * a.rbg);
        mbar_arrive_expect_tx(&full[slot], 2 * bytes);
        bulk_copy_g2s(dst, wg_e + row * a.rbg, bytes, &full[slot], pol);
        bulk_copy_g2s(dst + half_bytes, wu_e + row * a.rbg, bytes, &full[slot], pol);
    };
    if (tid == CTHREADS) {
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GW); // the warps of a consumer group
        }
        mbar_init(&hq_bar, 1);
        fence_mbar_init();
        s_abort = 0;
        s_xnext = 0;
    }
    __syncthreads(); // barriers initialized
    if (tid == CTHREADS) {
        if (a.wsd && a.prefetch) {
            // warm L2 with this CTA's slice of the shared expert's down rows (a
            // hint: no bulk copy, so the routing's loads are not held back)
            const size_t tot_d = (size_t)a.H * a.rbd; // a multiple of 16
            const size_t cd = ((tot_d / nb) + 15) & ~size_t(15);
            const size_t od = cd * bx;
            if (od < tot_d)
                prefetch_l2(a.wsd + od, (uint32_t)min(cd, tot_d - od));
        }
    }
    if (warp == GW + 1) {
        // the inputs of the routing and of the quantization into L2 (a hint:
        // whatever the previous kernel still writes reaches L2 as well)
        for (int i = lane; i < (T * E + 31) / 32; i += 32)
            prefetch_line_l2(a.logits + 32 * i);
        for (int i = lane; a.bias && i < (E + 31) / 32; i += 32)
            prefetch_line_l2(a.bias + 32 * i);
        for (int i = lane; i < T * a.H / 32; i += 32)
            prefetch_line_l2(a.x + 32 * i);
    }
    pdl_wait();
    pdl_trigger();
    // the barrier count before this launch's barrier (every earlier one has ended)
    if (tid == 0)
        s_c0 = ld_acquire_gpu_u64(a.sync);

    // ---------------- helpers ----------------
    // ---------------- consumer helpers ----------------
    const int grp = warp / GW, wl = warp - grp * GW; // consumer group, warp within it
    bool dead = false;
    // waits for the stage in `slot`, use `use`; false if this CTA gave up
    auto wait_slot = [&](int slot, int use) -> bool {
        // warp-uniform: every lane takes the same branch to the __all_sync
        if (__any_sync(FULL, *(volatile int *)&s_abort != 0))
            dead = true;
        if (dead)
            return false;
        const bool got = __all_sync(FULL, mbar_wait_parked(&full[slot], (uint32_t)use & 1u));
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

    // Down rows [m0, m1) of this CTA (warp-collective).  By weight (dsplit):
    // each CTA should stream about the same bytes, gate/up groups plus down
    // rows, so D(b), the down rows of the CTAs before b, is the cost not yet
    // covered by their groups at the even share b / nb, in rows of all nv
    // experts, made non-decreasing by a suffix minimum (D(nb) = H).  Every
    // CTA evaluates the same expressions, so neighbours agree on their
    // boundary.  Otherwise an even split.
    auto down_rows = [&](int nv, int &m0, int &m1) {
        if (a.dsplit && nv > 0) {
            m0 = a.H;
            m1 = a.H;
            const unsigned ng = (unsigned)(nv * G32);
            const float Cg = 64.0f * (float)a.nbH, Cd = (float)nv * (float)a.nbI; // bytes / 34
            const float W = (float)ng * Cg + (float)a.H * Cd;
            for (int b = bx + lane; b < nb; b += 32) {
                const float gb = (float)((ng * (unsigned)b) / (unsigned)nb) * Cg;
                const float r = floorf((W * (float)b / (float)nb - gb) / Cd);
                const int d = r <= 0.0f ? 0 : r >= (float)a.H ? a.H : (int)r;
                m0 = min(m0, d);
                if (b > bx)
                    m1 = min(m1, d);
            }
            m0 = __reduce_min_sync(FULL, m0);
            m1 = __reduce_min_sync(FULL, m1);
        } else {
            m0 = a.H * bx / nb;
            m1 = a.H * (bx + 1) / nb;
        }
    };
    // This CTA's work once nvr, the routed virtual experts, is known
    // (warp-collective).  Gate/up: groups [g0, g1) of all NV * G32 (virtual
    // expert major, the shared expert last), shared ones taken first.  Down:
    // rows [dn0, dn0 + nrows) in nrb row blocks of rpb rows (the last one
    // rlast); a row block's NV * rows items (expert major) are cut into
    // stages of SR rows.  Each half of the ring takes the gate/up parts of its
    // consumer group's groups, then down stages, alternately, starting with
    // the half that has fewer gate/up parts.  (Unsigned 32-bit: NV * G32 <= 65 * 1024, times at most 1024
    // CTAs, stays below 2^32.)
    auto make_plan = [&](int nvr) {
        LayerPlan q;
        q.NVr = nvr;
        q.NV = nvr + (a.wsg ? 1 : 0);
        const unsigned NG = (unsigned)(q.NV * G32);
        q.g0 = (int)(NG * (unsigned)bx / (unsigned)nb);
        q.g1 = (int)(NG * (unsigned)(bx + 1) / (unsigned)nb);
        q.nsh = a.wsg ? max(0, q.g1 - max(q.g0, nvr * G32)) : 0;
        q.ngr = q.g1 - q.g0;
        int m0, m1;
        down_rows(q.NV, m0, m1);
        q.dn0 = m0;
        q.nrows = m1 - m0;
        q.nrb = (q.nrows + RB_MAX - 1) / RB_MAX;
        q.rpb = q.nrb ? (q.nrows + q.nrb - 1) / q.nrb : 0;
        q.rlast = q.nrows - (q.nrb - 1) * q.rpb;
        q.spr = q.nrb ? (q.NV * q.rpb + a.SR - 1) / a.SR : 0;
        q.slast = q.nrb ? (q.NV * q.rlast + a.SR - 1) / a.SR : 0;
        q.NPd = q.nrb ? (q.nrb - 1) * q.spr + q.slast : 0;
        q.nglu0 = ((q.ngr + 1) / 2) * PPG;
        q.nglu1 = (q.ngr / 2) * PPG;
        q.s1 = q.nglu1 < q.nglu0 ? 1 : 0;
        q.nd0 = q.s1 ? q.NPd / 2 : (q.NPd + 1) / 2;
        q.nd1 = q.NPd - q.nd0;
        return q;
    };
    const int SR = a.SR;

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
    constexpr int XR = 2;
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


    // One token with whole rows per warp (RU a multiple of GW): each warp
    // holds the lane partial sums of its four rows of a group (gate, up) and
    // reduces them once, when the group is done.
    const bool defer = x_regs && a.RU % GW == 0;
    const int rpw = a.RU / GW; // rows of a part per warp
    float dacc[8];
#pragma unroll
    for (int q = 0; q < 8; q++)
        dacc[q] = 0.0f;
    // rows [p RU, (p + 1) RU) of a 32-row group from the stage in `slot` -> hb
    // (h of the group's rows, 32 x HB_STRIDE); columns of a routed expert
    // (first, ncols) or, routed == false, the T shared tokens
    auto glu_part = [&](int slot, int use, int p, bool routed, int first, int ncols, float *hb) {
        if (wait_slot(slot, use)) {
            const uint8_t *st = ring + (size_t)slot * a.stage_bytes;
            for (int i = wl; i < a.RU; i += GW) {
                const int prow = p * a.RU + i; // row within the group
                const uint8_t *grow = st + (size_t)i * a.rbg;
                const uint8_t *urow = st + half_bytes + (size_t)i * a.rbg;
                for (int c0 = 0; c0 < ncols; c0 += NC) {
                    const int nc = min(NC, ncols - c0);
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
                        const uint32_t *xc[NC]; // x row of each column's token
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            const int cc = c0 + (c < nc ? c : 0);
                            xc[c] = xs + (size_t)(routed ? routes_s[first + cc] / k : cc) * xstride;
                        }
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
                    if (defer) {
                        // one token: the row's partial sums wait for one
                        // reduction of the warp's four rows of the group
                        const int r = p * rpw + (i - wl) / GW;
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            if (q == r) {
                                dacc[2 * q] = ag[0];
                                dacc[2 * q + 1] = au[0];
                            }
                        }
                        continue;
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
                                hb[prow * HB_STRIDE + c0 + c] = swiglu(sm, u, a.clamp);
                            if (two && lane == 16)
                                hb[prow * HB_STRIDE + c0 + c + 1] = swiglu(sm, u, a.clamp);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !dead)
            mbar_arrive(&empty[slot]); // this warp is done with the stage
    };
    // one token: h of this warp's four rows of a finished group -> hb (the
    // sums of row r at lanes 8 r (gate) and 8 r + 4 (up))
    auto glu_finish = [&](float *hb) {
        const float n = reduce8(dacc, lane);
        const float u = __shfl_down_sync(FULL, n, 4);
        if ((lane & 7) == 0) {
            const int r = lane >> 3;
            const int prow = (r / rpw) * a.RU + wl + GW * (r % rpw);
            hb[prow * HB_STRIDE] = swiglu(n, u, a.clamp);
        }
    };
    // a finished 32-row group in hb -> h and its q8_1 blocks (warp per column)
    auto glu_epilogue = [&](int gi, bool routed, int first, int ncols, const float *hb) {
        if (dead || *(volatile int *)&s_abort)
            return;
        const int grow0 = (gi % G32) * 32;
        for (int c = wl; c < ncols; c += GW) {
            const int r = routed ? routes_s[first + c] : R + c;
            const float hv = hb[lane * HB_STRIDE + c];
            a.h[(size_t)r * a.I + grow0 + lane] = hv;
            quantize_q8_1_warp(hv, a.hq + ((size_t)r * a.nbI + grow0 / 32) * Q8_1_WORDS, lane);
        }
    };

    // ---------------- 1-3. routing, x -> q8_1 ----------------
    // Scores and ranks by the routing warps GW .. CW (the producer among
    // them); a NaN score ranks below every number and ties go to the lower
    // index, a total order, so each token selects exactly k distinct experts.
    auto route_rank = [&]() {
        const int rt = tid - GTHREADS; // routing threads 0 .. RTHREADS-1
        for (int i = rt; i < T * E; i += RTHREADS) {
            const float l = a.logits[i];
            lsm[i] = l;
            const float sc = a.bias ? __fadd_rn(l, a.bias[i % E]) : l;
            scores[i] = sc == sc ? sc : -INFINITY;
        }
        for (int i = rt; i < MAX_T * (MAX_E / 32); i += RTHREADS)
            (&sel_bits[0][0])[i] = 0u;
        named_barrier(BAR_ROUTE, RTHREADS);
        // rank of every (token, expert) pair, four threads per pair
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
#pragma unroll 4
                for (int e2 = qj * qE; e2 < e_end; e2++) {
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
        named_barrier(BAR_ROUTE, RTHREADS);
    };
    // The expert tables (one warp): virtual expert v is the v-th selected
    // expert in index order; its columns are the routes that chose it, in
    // route order, at [first, first + ncols) of the route list.
    auto build_tables = [&]() {
        int nact = 0, offp = 0;
        for (int c = 0; c < E; c += 32) { // warp-uniform trip count
            const int e = c + lane;
            int cnt = 0;
            if (e < E)
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
                v_first[nact] = 0;
                v_ncols[nact] = T;
            }
        }
    };
    // route weights (routing warp w0 + t for token t) and the route list:
    // route r = t k + j goes to position pos(r), the routes ahead of it in
    // (expert, route) order; threads [r0, r0 + rn) of the routing warps
    auto weights_routes = [&](int w0, int r0, int rn) {
        const int rt = tid - GTHREADS, t = warp - GW - w0;
        if (t >= 0 && t < T) {
            const float sel0 = lane < k ? lsm[t * E + ids_s[t * k + lane]] : 0.0f;
            const float sel1 = lane + 32 < k ? lsm[t * E + ids_s[t * k + lane + 32]] : 0.0f;
            route_softmax_warp(sel0, sel1, k, w_s + t * k, lane);
        }
        for (int r = rt - r0; r >= 0 && r < R; r += rn) {
            const int e = ids_s[r];
            int pos = 0;
            for (int r2 = 0; r2 < R; r2++) {
                const int e2 = ids_s[r2];
                pos += (e2 < e || (e2 == e && r2 < r)) ? 1 : 0;
            }
            routes_s[pos] = r;
        }
    };

    LayerPlan P;
    if (warp == CW) {
        // ---------------- the producer: every stage of this CTA ----------------
        // With one token the plan is known at once (k experts); the producer
        // then needs only the selection itself, the v-th selected expert.
        if (T == 1)
            P = make_plan(k);
        route_rank();
        if (T != 1) {
            build_tables();
            __syncwarp();
            named_barrier_arrive(BAR_TABLES, THREADS);
            P = make_plan(s_nvr);
        }
        if (lane != 0)
            return;
        // expert of routed virtual expert v
        auto vexp = [&](int v) -> int {
            if (T != 1)
                return v_e[v];
            for (int w = 0; w < (E + 31) / 32; w++) {
                const uint32_t m = sel_bits[0][w];
                const int c = __popc(m);
                if (v < c)
                    return 32 * w + (int)__fns(m, 0u, v + 1);
                v -= c;
            }
            return E; // not reached: a token selects k experts
        };
        auto group_of = [&](int j) { return j < P.nsh ? P.g1 - P.nsh + j : P.g0 + (j - P.nsh); };
        int n[2] = {0, 0};    // stages requested per half
        int dq[2] = {0, 0};   // down stages requested per half
        const int nglu[2] = {P.nglu0, P.nglu1};
        unsigned long long t_idle = 0;
        for (uint32_t it = 0;;) {
            bool left = false, moved = false;
            for (int h = 0; h < 2; h++) {
                int d = -1; // the next stage of half h: a gate/up part, or down stage d
                if (n[h] >= nglu[h]) {
                    if (!a.down_early && (n[0] < nglu[0] || n[1] < nglu[1])) {
                        left = true; // down stages wait until every gate/up part is requested
                        continue;
                    }
                    const int i = dq[h];
                    d = 2 * i + (h ^ P.s1);
                    if (d >= P.NPd)
                        continue;
                }
                left = true;
                const int slot = h * HALF + n[h] % HALF, use = n[h] / HALF;
                if (use > 0 && !mbar_test_wait(&empty[slot], (uint32_t)(use - 1) & 1u))
                    continue;
                if (d < 0) {
                    const int j = h + 2 * (n[h] / PPG), p = n[h] % PPG;
                    const int gi = group_of(j);
                    const int v = gi / G32;
                    const bool routed = v < P.NVr;
                    const int e = routed ? vexp(v) : E;
                    issue_part(h, n[h], gi, p, routed ? a.wg + (size_t)e * a.I * a.rbg : a.wsg,
                               routed ? a.wu + (size_t)e * a.I * a.rbg : a.wsu);
                } else {
                    uint8_t *dst = ring + (size_t)slot * a.stage_bytes;
                    int rb, sp;
                    down_stage(P, d, rb, sp);
                    const int nr0 = P.dn0 + rb * P.rpb;
                    const int rows = rb == P.nrb - 1 ? P.rlast : P.rpb;
                    const int i0 = sp * SR, i1 = min(P.NV * rows, i0 + SR);
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)((i1 - i0) * a.rbd));
                    for (int i = i0; i < i1;) {
                        const int v = i / rows, m = i - v * rows;
                        const int cnt = min(i1 - i, rows - m);
                        const int e = v < P.NVr ? vexp(v) : E;
                        const uint8_t *src = e < E ? a.wd + ((size_t)e * a.H + nr0 + m) * a.rbd
                                                   : a.wsd + (size_t)(nr0 + m) * a.rbd;
                        bulk_copy_g2s(dst + (size_t)(i - i0) * a.rbd, src, (uint32_t)(cnt * a.rbd), &full[slot],
                                      pol);
                        i += cnt;
                    }
                    dq[h]++;
                }
                n[h]++;
                moved = true;
            }
            if (!left || *(volatile int *)&s_abort)
                break;
            if (moved) {
                t_idle = 0;
                continue;
            }
            if (a.psleep)
                __nanosleep((unsigned)a.psleep); // leave the issue slots to the consumer warps
            if ((++it & 31u) == 0u) {
                const unsigned long long now = global_timer_ns();
                if (t_idle == 0) {
                    t_idle = now;
                } else if (now - t_idle > WAIT_LIMIT_NS) {
                    atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                    *(volatile int *)&s_abort = 1;
                    break;
                }
            }
        }
        // no bulk copy may still be writing shared memory when the CTA exits
        for (int h = 0; h < 2; h++) {
            for (int u = 0; u < HALF && u < n[h]; u++) {
                const int last = n[h] - 1 - u; // the last use of slot h * HALF + last % HALF
                if (!mbar_wait_bounded(&full[h * HALF + last % HALF], (uint32_t)(last / HALF) & 1u))
                    atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
            }
        }
        return;
    }
    if (warp < GW) {
        quantize_x();
    } else {
        route_rank();
        if (T == 1) {
            // the producer does without the tables: warp GW builds them for
            // the consumers while the others weigh and order the routes
            if (warp == GW)
                build_tables();
            else
                weights_routes(1, 32, RTHREADS - 64);
        } else {
            weights_routes(0, 0, RTHREADS - 32);
        }
        quantize_x(); // what is left of x
    }
    // tables, weights, route list and x are in shared memory
    named_barrier(BAR_TABLES, T == 1 ? CTHREADS : THREADS);
    if (cta0 && warp >= GW) {
        const int rt = tid - GTHREADS;
        for (int i = rt; i < R; i += RTHREADS - 32) {
            a.ids[i] = ids_s[i];
            a.weights[i] = w_s[i];
            a.routes[i] = routes_s[i];
        }
        for (int e = rt; e < E; e += RTHREADS - 32) {
            a.counts[e] = cnt_s[e];
            a.offsets[e] = off_s[e];
        }
        if (rt == 0)
            a.offsets[E] = off_s[E];
    }
    P = make_plan(T == 1 ? k : s_nvr);
    auto group_of = [&](int j) { return j < P.nsh ? P.g1 - P.nsh + j : P.g0 + (j - P.nsh); };
    auto down_slot = [&](int d, int &hh, int &n) { down_slot_of(P, d, hh, n); };

    // ---------------- 4. gate/up groups -> h, hq (consumer group grp takes j = grp, grp + 2, ...) ----------------
    load_xregs();
    {
        int n = 0;  // stages of this group's half
        int lb = 0; // h buffer
        for (int j = grp; j < P.ngr; j += 2, lb ^= 1) {
            const int gi = group_of(j);
            const int v = gi / G32;
            const bool routed = v < P.NVr;
            const int first = routed ? v_first[v] : 0, ncols = routed ? v_ncols[v] : T;
            float *hb = hbuf + (size_t)(grp * 2 + lb) * 32 * HB_STRIDE;
            for (int p = 0; p < PPG; p++, n++) {
                glu_part(grp * HALF + n % HALF, n / HALF, p, routed, first, ncols, hb);
            }
            if (defer)
                glu_finish(hb);
            named_barrier(1 + grp, GTHREADS); // all 32 rows of the group are in hb
            glu_epilogue(gi, routed, first, ncols, hb);
        }
    }

    // ---------------- 5. every CTA's hq is stored ----------------
    // One row block whose down stages all fit the ring at once (no slot is
    // used twice by down stages): the work units (item, column) are listed
    // while thread 0 waits at the device-wide barrier, in the h buffers
    // (free by then), and each warp then walks its units in one go.
    const int nunits = P.nrows * (off_s[E] + (a.wsd ? T : 0));
    const bool by_units = P.nrb == 1 && P.nd0 <= HALF && P.nd1 <= HALF && nunits <= MAX_UNITS;
    uint2 *units = reinterpret_cast<uint2 *>(hbuf);
    named_barrier(BAR_ALL, CTHREADS); // this CTA's h and hq are stored
    if (warp == 0) {
        if (lane == 0) {
            if (!grid_barrier(a.sync, gridDim.x, s_c0)) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
            } else if (a.hs_on && a.hq_bulk) {
                // all of hq into shared memory with one bulk copy, requested as
                // soon as the barrier ends (the proxy fence orders the other
                // CTAs' stores, seen through the barrier, before it)
                const uint32_t bytes = (uint32_t)((R + (a.wsd ? T : 0)) * a.nbI * Q8_1_WORDS * 4);
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(&hq_bar, bytes);
                bulk_copy_g2s(hs, a.hq, bytes, &hq_bar, l2_evict_normal_policy());
            }
        }
        __syncwarp();
    } else if (by_units) {
        // unit (item i = v rows + m, column c) is number rows F(v) + m ncols(v) + c,
        // F(v) the columns of the virtual experts before v: item order
        const int fsh = off_s[E];
        for (int i = tid - 32; i < P.NV * P.nrows; i += CTHREADS - 32) {
            const int v = i / P.nrows, m = i - v * P.nrows;
            const bool routed = v < P.NVr;
            const int nc = routed ? v_ncols[v] : T;
            const int F = routed ? v_first[v] : fsh;
            const int d = i / SR;
            int hh, nq;
            down_slot(d, hh, nq);
            const uint32_t woff = (uint32_t)((hh * HALF + nq % HALF) * a.stage_bytes + (i - d * SR) * a.rbd);
            for (int c = 0; c < nc; c++) {
                const int ys = routed ? routes_s[F + c] : R + c; // hq row = y slot
                units[P.nrows * F + m * nc + c] = make_uint2(woff, (uint32_t)ys | ((uint32_t)m << 8) | ((uint32_t)d << 16));
            }
        }
    }
    named_barrier(BAR_ALL, CTHREADS); // every CTA's hq is stored
    const int ibytes_w = a.nbI * Q8_1_WORDS; // words per hq row
    {
        const int nlive = R + (a.wsd ? T : 0);
        if (a.hs_on && !*(volatile int *)&s_abort) {
                if (a.hq_bulk) {
                    // all of hq in shared memory: the bulk copy thread 0
                    // requested as soon as the device-wide barrier ended
                    if (!__all_sync(FULL, mbar_wait_parked(&hq_bar, 0))) {
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

    // ---------------- 6. down rows (all consumer warps), combine ----------------
    const uint32_t *xbase = a.hs_on ? hs : a.hq;
    // Units of work: item i0 + it of a row block (virtual expert v = i / rows,
    // row m = i - v rows), it in [0, ni), times each of its columns.  rowp(it)
    // is the item's weight row in shared memory; ensure(it) makes sure the
    // stages up to that of item it have landed (warp-collective, uniform it).
    // The y values go to ybuf.
    auto down_units = [&](int ni, int i0, int rows, auto rowp, auto ensure) {
        if (a.nbI == 32) {
            // two rows per warp (ROWMAP_TWO_ROWS): half h of the warp walks the
            // items 2 p + h, p = warp, warp + CW, ..., and their columns, two units
            // per pass; a half-warp reduce-scatter leaves the sums at lanes
            // 0, 8 (half 0) and 16, 24 (half 1)
            const int h = lane >> 4;
            int p = warp, col = 0;
            const uint32_t *xlast = nullptr;
            Q81Block xb[2];
            while (__any_sync(FULL, 2 * p + h < ni)) { // warp-uniform trip count
                // the stages of the items this pass may reach
                ensure(__reduce_max_sync(FULL, min(ni - 1, 2 * (p + CW) + h)));
                const uint8_t *wr[2];
                const uint32_t *xr[2];
                int yo[2];
                bool live[2];
#pragma unroll
                for (int z = 0; z < 2; z++) {
                    const int it = 2 * p + h;
                    live[z] = it < ni;
                    wr[z] = ring;
                    xr[z] = xbase;
                    yo[z] = 0;
                    if (live[z]) {
                        const int i = i0 + it;
                        const int v = i / rows, m = i - v * rows;
                        const int ys = v_e[v] < E ? routes_s[v_first[v] + col] : R + col; // hq row = y slot
                        wr[z] = rowp(it);
                        xr[z] = xbase + (size_t)ys * ibytes_w;
                        yo[z] = ys * RB_MAX + m;
                        if (++col == v_ncols[v]) {
                            col = 0;
                            p += CW;
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
            int it = warp, col = 0;
            while (it < ni) {
                ensure(min(ni - 1, it + 3 * CW)); // the stages of the items this pass may reach
                const uint8_t *wr[4];
                const uint32_t *xr[4];
                int yo[4];
                int nu = 0;
#pragma unroll
                for (int z = 0; z < 4; z++) {
                    wr[z] = ring;
                    xr[z] = xbase;
                    yo[z] = 0;
                    if (it < ni) {
                        const int i = i0 + it;
                        const int v = i / rows, m = i - v * rows;
                        const int ys = v_e[v] < E ? routes_s[v_first[v] + col] : R + col; // hq row = y slot
                        wr[z] = rowp(it);
                        xr[z] = xbase + (size_t)ys * ibytes_w;
                        yo[z] = ys * RB_MAX + m;
                        nu++;
                        if (++col == v_ncols[v]) {
                            col = 0;
                            it += CW;
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
    };
    // out rows [nr0, nr0 + rows) from ybuf
    auto combine = [&](int nr0, int rows) {
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
    };
    if (by_units) {
        int dw = -1; // the last stage this warp waited for
        auto ensure = [&](int dn) { // warp-uniform dn
            while (dw < dn) {
                int hh, nq;
                down_slot(++dw, hh, nq);
                wait_slot(hh * HALF + nq % HALF, nq / HALF);
            }
        };
        if (a.nbI == 32) {
            // half-warps (16 lanes, ROWMAP_TWO_ROWS) take units hw, hw + 32, ...,
            // UZ at a time; sums by the half-warp butterfly.  (Two at a time:
            // a pass waits only for the stages of its units, so the first pass
            // runs while later stages still land; measured faster than 1, 3, 4
            // or 6.)
            constexpr int UZ = 2;
            const int hw = 2 * warp + (lane >> 4);
            for (int base = 0; base < nunits; base += 32 * UZ) { // uniform trip count
                uint2 ud[UZ];
                int dmax = -1;
#pragma unroll
                for (int z = 0; z < UZ; z++) {
                    const int u = base + hw + 32 * z;
                    ud[z] = u < nunits ? units[u] : make_uint2(0u, 0u);
                    if (u < nunits)
                        dmax = max(dmax, (int)(ud[z].y >> 16));
                }
                ensure(__reduce_max_sync(FULL, dmax));
                float acc[UZ];
#pragma unroll
                for (int z = 0; z < UZ; z++) {
                    acc[z] = 0.0f;
                    const int u = base + hw + 32 * z;
                    if (u < nunits) {
                        const uint8_t *wr = ring + ud[z].x;
                        const uint32_t *xr = xbase + (size_t)(ud[z].y & 0xffu) * ibytes_w;
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            const int b = rowmap_block(ROWMAP_TWO_ROWS, lane, j);
                            Q81Block xb;
                            const uint32_t *xw = xr + (size_t)b * Q8_1_WORDS;
                            if (a.hs_on) {
                                load_q8_1_any(xw, xb);
                            } else {
                                xb.d = half_bits_to_float(__ldcg(xw));
#pragma unroll
                                for (int w = 0; w < 8; w++)
                                    xb.q[w] = (int)__ldcg(xw + 1 + w);
                            }
                            Q80Block wb;
                            load_q8_0_smem(wr, b, wb);
                            acc[z] = fmaf(wb.d * xb.d, (float)dot_q8_block(wb.q, xb.q), acc[z]);
                        }
                    }
                }
#pragma unroll
                for (int z = 0; z < UZ; z++) {
                    const float y = half_warp_sum(acc[z]);
                    const int u = base + hw + 32 * z;
                    if ((lane & 15) == 0 && u < nunits)
                        ybuf[(ud[z].y & 0xffu) * RB_MAX + ((ud[z].y >> 8) & 0xffu)] = y;
                }
            }
        } else {
            // warps (32 lanes) take units warp, warp + CW, ..., four at a time
            const int dmap = (a.nbI % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN;
            const int nbl = rowmap_blocks(dmap, a.nbI, lane);
            for (int base = warp; base < nunits; base += 4 * CW) {
                uint2 ud[4];
                int dmax = -1;
#pragma unroll
                for (int z = 0; z < 4; z++) {
                    const int u = base + CW * z;
                    ud[z] = u < nunits ? units[u] : make_uint2(0u, 0u);
                    if (u < nunits)
                        dmax = max(dmax, (int)(ud[z].y >> 16));
                }
                ensure(dmax);
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int j = 0; j < nbl; j++) {
                    const int b = rowmap_block(dmap, lane, j);
#pragma unroll
                    for (int z = 0; z < 4; z++) {
                        if (base + CW * z < nunits) {
                            Q80Block wb;
                            load_q8_0_smem(ring + ud[z].x, b, wb);
                            Q81Block xb;
                            const uint32_t *xw = xbase + (size_t)(ud[z].y & 0xffu) * ibytes_w + (size_t)b * Q8_1_WORDS;
                            if (a.hs_on) {
                                load_q8_1_any(xw, xb);
                            } else {
                                xb.d = half_bits_to_float(__ldcg(xw));
#pragma unroll
                                for (int w = 0; w < 8; w++)
                                    xb.q[w] = (int)__ldcg(xw + 1 + w);
                            }
                            acc[z] = fmaf(wb.d * xb.d, (float)dot_q8_block(wb.q, xb.q), acc[z]);
                        }
                    }
                }
                const float y = reduce4(acc[0], acc[1], acc[2], acc[3], lane);
                const int z = lane >> 3;
                const uint32_t yd = z == 0 ? ud[0].y : z == 1 ? ud[1].y : z == 2 ? ud[2].y : ud[3].y;
                if ((lane & 7) == 0 && base + CW * z < nunits)
                    ybuf[(yd & 0xffu) * RB_MAX + ((yd >> 8) & 0xffu)] = y;
            }
        }
        named_barrier(BAR_ALL, CTHREADS); // every y value is in ybuf
        combine(P.dn0, P.nrows);
        return;
    }
    for (int d = 0; d < P.NPd; d++) {
        int rb, sp;
        down_stage(P, d, rb, sp);
        const int nr0 = P.dn0 + rb * P.rpb;
        const int rows = rb == P.nrb - 1 ? P.rlast : P.rpb;
        const int i0 = sp * SR, i1 = min(P.NV * rows, i0 + SR);
        int hh, nq;
        down_slot(d, hh, nq);
        const int slot = hh * HALF + nq % HALF, use = nq / HALF;
        if (wait_slot(slot, use)) {
            const uint8_t *st = ring + (size_t)slot * a.stage_bytes;
            down_units(i1 - i0, i0, rows, [&](int it) -> const uint8_t * { return st + (size_t)it * a.rbd; },
                       [](int) {});
        }
        const bool rb_end = sp == (rb == P.nrb - 1 ? P.slast : P.spr) - 1;
        if (nq + HALF < (hh ? P.nglu1 + P.nd1 : P.nglu0 + P.nd0)) {
            // the producer reuses the slot: every consumer warp must be done with it
            named_barrier(BAR_ALL, CTHREADS);
            if (tid == 0 && !dead)
                mbar_arrive_count(&empty[slot], GW);
        }
        if (rb_end) {
            named_barrier(BAR_ALL, CTHREADS); // the row block's y values are in ybuf
            combine(nr0, rows);
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
    static luce_host::SmemLimit limit;
    auto kern = k_moe_layer<NC>;
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
        limit.forget();
        return LUCE_ERR_CUDA;
    }
    return LUCE_OK;
}

} // namespace

using namespace luce_host;

// The flat-split kernel for layers whose q8_1 rows of h exceed 24 KB
// (moe_layer_flat.cu); same arguments and checks.
extern "C" __attribute__((visibility("hidden"))) luce_status
luce_internal_moe_layer_flat(const float *logits, const float *bias, const float *x, const luce_block_q8_0 *w_gate,
                             const luce_block_q8_0 *w_up, const luce_block_q8_0 *w_down,
                             const luce_block_q8_0 *ws_gate, const luce_block_q8_0 *ws_up,
                             const luce_block_q8_0 *ws_down, int T, int E, int k, int H, int I, float clamp,
                             int32_t *ids, float *weights, luce_block_q8_1 *xq, int32_t *counts, int32_t *offsets,
                             int32_t *routes, float *h, luce_block_q8_1 *hq, float *out, void *workspace,
                             size_t workspace_bytes, void *stream);

// The grouped tensor-core path for many tokens (moe_tc.cu); same arguments.
extern "C" __attribute__((visibility("hidden"))) luce_status
luce_internal_moe_layer_tc(const float *logits, const float *bias, const float *x, const luce_block_q8_0 *w_gate,
                           const luce_block_q8_0 *w_up, const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_gate,
                           const luce_block_q8_0 *ws_up, const luce_block_q8_0 *ws_down, int T, int E, int k, int H,
                           int I, float clamp, int32_t *ids, float *weights, luce_block_q8_1 *xq, int32_t *counts,
                           int32_t *offsets, int32_t *routes, float *h, luce_block_q8_1 *hq, float *out,
                           void *workspace, size_t workspace_bytes, void *stream);
extern "C" __attribute__((visibility("hidden"))) size_t luce_internal_moe_layer_tc_bytes(int T, int k, int H, int I);

// Whether a shape goes to the grouped tensor-core path: more tokens or routes
// than the one-launch kernels take.
static bool tc_shape(int T, int k) { return T > MAX_T || (long long)T * k > MAX_R; }

extern "C" size_t luce_moe_layer_workspace_bytes(int T, int k, int H, int I)
{
    if (T < 0 || k < 0 || H < 0 || I < 0)
        return 0;
    if (T > 0 && k > 0 && tc_shape(T, k))
        return luce_internal_moe_layer_tc_bytes(T, k, H, I);
    return 16 + (size_t)T * (size_t)(k + 1) * (size_t)H * sizeof(float); // barrier count, y values
}

extern "C" luce_status luce_moe_layer(const float *logits, const float *bias, const float *x,
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
    if (workspace_bytes < luce_moe_layer_workspace_bytes(T, k, H, I))
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || (bias && !aligned(bias, 4)) || !aligned(x, 16) || !aligned(w_gate, 16) ||
        !aligned(w_up, 16) || !aligned(w_down, 16) ||
        (has_ws && (!aligned(ws_gate, 16) || !aligned(ws_up, 16) || !aligned(ws_down, 16))) || !aligned(ids, 4) ||
        !aligned(weights, 4) || !aligned(xq, 4) || !aligned(counts, 4) || !aligned(offsets, 4) ||
        !aligned(routes, 4) || !aligned(h, 16) || !aligned(hq, 16) || !aligned(out, 4) || !aligned(workspace, 16))
        return LUCE_ERR_INVALID_ARG;
    if (tc_shape(T, k))
        return luce_internal_moe_layer_tc(logits, bias, x, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, T, E, k, H, I,
                                          clamp, ids, weights, xq, counts, offsets, routes, h, hq, out, workspace,
                                          workspace_bytes, stream);
    if (E > MAX_E)
        return LUCE_ERR_UNSUPPORTED;
    {
        // large q8_1 rows of h (speculative verify): the flat-split kernel
        const size_t hs = (size_t)(T * k + T) * (size_t)(I / 32) * Q8_1_BYTES;
        if (hs > 24 * 1024)
            return luce_internal_moe_layer_flat(logits, bias, x, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, T, E,
                                                k, H, I, clamp, ids, weights, xq, counts, offsets, routes, h, hq, out,
                                                workspace, workspace_bytes, stream);
    }

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
    a.sync = reinterpret_cast<unsigned long long *>(workspace); // the barrier count: the workspace's first word
    a.nbH = H / 32;
    a.nbI = I / 32;
    a.rbg = a.nbH * Q8_0_BYTES;
    a.rbd = a.nbI * Q8_0_BYTES;
    const Tuning &tu = g_tuning;
    // a gate/up part (RU gate rows + RU up rows) of about part_kb, but at
    // least one row per warp while a part stays under twice that
    int RU = 32;
    while (RU > 1 && 2 * RU * a.rbg > tu.layer_part_kb * 1024 &&
           !(RU <= GW && 2 * RU * a.rbg <= 2 * tu.layer_part_kb * 1024))
        RU /= 2;
    a.RU = RU;
    a.stage_bytes = std::max(2 * RU * a.rbg, a.rbd);
    a.SR = a.stage_bytes / a.rbd;
    a.prefetch = tu.layer_prefetch;
    a.dsplit = tu.layer_dsplit;
    a.psleep = tu.layer_psleep;
    a.down_early = tu.layer_down_early;
    a.evict_first = tu.evict_first;
    const int nslots = T * k + T;
    const size_t hs_bytes = (size_t)nslots * a.nbI * Q8_1_BYTES;
    a.hs_on = hs_bytes <= 24 * 1024 ? 1 : 0;
    a.hq_bulk = tu.layer_hq_bulk;
    const size_t xrow = (size_t)a.nbH * Q8_1_BYTES + (a.nbH % 64 == 0 ? (size_t)64 * (a.nbH / 32) : 0);
    const size_t fixed = (size_t)T * xrow + (a.hs_on ? hs_bytes : 0) +
                         (size_t)nslots * RB_MAX * sizeof(float) + (size_t)2 * T * E * sizeof(float) +
                         (size_t)4 * 32 * HB_STRIDE * sizeof(float);
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
