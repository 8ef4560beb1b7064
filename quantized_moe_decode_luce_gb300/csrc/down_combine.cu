// down_combine.cu -- the Q8_0 x q8_1 down product of every route and of the
// shared expert, fused with the masked route-weighted combine, and its C-ABI
// entry point.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving", commit "fused routed combine and q8_1 inputs for
// the hybrid owners": masking, weighting and summing the routes is one
// launch, and its combine rounds each product and each sum on its own, the
// way the separate operations did.
//
// GB300 shape (our own): a CTA owns a slab of RN output rows n for a tile of
// tokens and streams those RN rows of EVERY active (virtual) expert, one
// cp.async.bulk stage per expert, through a shared-memory ring; each weight
// row crosses HBM once per token tile (once per step for decode and verify,
// where one tile holds every token).  Each consumer warp takes whole stages
// (all RN rows of one expert) when the ring allows it, else every warp takes
// part in every stage.  Each route's product y stays in shared memory, so
// the combine needs no second pass and no atomics: one thread sums out[t][n]
// over the k slots in slot order with separately rounded products and sums
// (__fmul_rn / __fadd_rn), then adds the shared expert.  Deterministic; no
// global scratch.
//
// With programmatic dependent launch the CTAs start while the gate/up kernel
// still runs: the routing tables (written two launches earlier) are read and
// the weight rows are requested before waiting for h.
#include <algorithm>
#include <climits>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_down)

namespace {

using namespace luce;

constexpr int NCU = 32; // columns per virtual expert
constexpr int CW = 4;   // consumer warps
constexpr int RN = 8;   // output rows per CTA
constexpr int RPW = RN / CW; // rows of a stage per consumer warp

struct DownArgs {
    const uint8_t *wd;    // [E][H][rowbytes]
    const uint8_t *wsd;   // [H][rowbytes] or null
    const uint32_t *hq;   // [T*k+T][nbI] q8_1 blocks (9 words)
    const int32_t *ids;   // [T][k]
    const float *weights; // [T][k]
    const int32_t *offsets, *routes;
    float *out; // [T][H]
    int T, k, E, H, I;
    int nbI, rowbytes;
    int TT; // tokens per tile
    int NS; // ring stages
    int hs_rows; // activation rows staged in shared memory (0: read through L1)
    int evict_first;
    int coop;    // all consumer warps on every stage (rings of fewer than CW stages)
};

struct VUnit {
    const uint8_t *w; // RN rows of this expert
    int e;            // expert (E = shared)
    int first;        // index into routes[] of the expert's first route in the tile
    int col0, ncols;
};

// y of the NR rows row0, row0 + rstep, ... of one stage for the nc columns
// whose activation rows are xc[] and whose y slots are ys[].  Rows of 32
// blocks go two at a time (ROWMAP_TWO_ROWS: lanes 0..15 on row 2q, lanes
// 16..31 on row 2q + 1, each lane on blocks l and l + 16, then a half-warp
// sum); other rows take all 32 lanes (ROWMAP_PAIRS or ROWMAP_PLAIN, then a
// warp sum).
template <int NR, int NC>
__device__ __forceinline__ void stage_dots(const uint8_t *st, int rowbytes, int row0, int rstep,
                                           const uint32_t *const (&xc)[NC], const int (&ys)[NC], int nc, int nbI,
                                           int lane, float *ybuf)
{
    if (nbI == 32) {
        constexpr int NP = NR / 2;
        static_assert(NR % 2 == 0, "rows go in pairs");
        const int h = lane >> 4;
        float acc[NP][NC];
#pragma unroll
        for (int i = 0; i < NP; i++)
#pragma unroll
            for (int c = 0; c < NC; c++)
                acc[i][c] = 0.0f;
#pragma unroll
        for (int j = 0; j < 2; j++) {
            const int b = rowmap_block(ROWMAP_TWO_ROWS, lane, j);
            Q81Block xb[NC];
#pragma unroll
            for (int c = 0; c < NC; c++)
                if (c < nc)
                    load_q8_1_any(xc[c] + (size_t)b * Q8_1_WORDS, xb[c]);
#pragma unroll
            for (int i = 0; i < NP; i++) {
                Q80Block wb;
                load_q8_0_smem(st + (size_t)(row0 + (2 * i + h) * rstep) * rowbytes, b, wb);
#pragma unroll
                for (int c = 0; c < NC; c++)
                    if (c < nc)
                        acc[i][c] = fmaf(wb.d * xb[c].d, (float)dot_q8_block(wb.q, xb[c].q), acc[i][c]);
            }
        }
#pragma unroll
        for (int c = 0; c < NC; c++) {
            if (c < nc) {
#pragma unroll
                for (int i = 0; i < NP; i++) {
                    const float y = half_warp_sum(acc[i][c]);
                    if ((lane & 15) == 0)
                        ybuf[ys[c] * RN + row0 + (2 * i + h) * rstep] = y;
                }
            }
        }
        return;
    }
    const int map = (nbI % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN;
    float acc[NR][NC];
#pragma unroll
    for (int i = 0; i < NR; i++)
#pragma unroll
        for (int c = 0; c < NC; c++)
            acc[i][c] = 0.0f;
    const int nbl = rowmap_blocks(map, nbI, lane);
    for (int j = 0; j < nbl; j++) {
        const int b = rowmap_block(map, lane, j);
        Q81Block xb[NC];
#pragma unroll
        for (int c = 0; c < NC; c++)
            if (c < nc)
                load_q8_1_any(xc[c] + (size_t)b * Q8_1_WORDS, xb[c]);
#pragma unroll
        for (int i = 0; i < NR; i++) {
            Q80Block wb;
            load_q8_0_smem(st + (size_t)(row0 + i * rstep) * rowbytes, b, wb);
#pragma unroll
            for (int c = 0; c < NC; c++)
                if (c < nc)
                    acc[i][c] = fmaf(wb.d * xb[c].d, (float)dot_q8_block(wb.q, xb[c].q), acc[i][c]);
        }
    }
#pragma unroll
    for (int c = 0; c < NC; c++) {
        if (c < nc) {
#pragma unroll
            for (int i = 0; i < NR; i++) {
                const float y = warp_sum(acc[i][c]);
                if (lane == 0)
                    ybuf[ys[c] * RN + row0 + i * rstep] = y;
            }
        }
    }
}

template <int NC, bool COOP>
__global__ void __launch_bounds__((CW + 1) * 32, 2) k_down_combine(const DownArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int stage_bytes = RN * a.rowbytes;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * stage_bytes);
    uint64_t *empty = full + a.NS;
    uint64_t *hs_bar = empty + a.NS;                            // staged activation rows landed
    uint32_t *hs = reinterpret_cast<uint32_t *>(hs_bar + 2);    // [hs_rows][nbI][9], 16-byte aligned
    float *ybuf = reinterpret_cast<float *>(hs + (size_t)a.hs_rows * a.nbI * Q8_1_WORDS); // [TT*k + TT][RN]
    int *vpre = reinterpret_cast<int *>(ybuf + (size_t)(a.TT * a.k + a.TT) * RN); // [E + 1]
    int *vlo = vpre + a.E + 1;                         // [E]: first route of the tile
    int *vcnt = vlo + a.E;                             // [E]: routes of the tile
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * a.TT, t1 = min(a.T, t0 + a.TT);
    const int n0 = blockIdx.y * RN;
    const int ntok = t1 - t0;
    if (tid == 0) {
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(hs_bar, 1);
        fence_mbar_init();
        s_abort = 0;
    }
    // routes of expert e that belong to tokens [t0, t1): a sub-range, since an
    // expert's routes are sorted by r = t*k + j.  (Grouping output: two
    // launches back, complete even when this grid started early.)
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int lo = a.offsets[e], hi = a.offsets[e + 1];
        int first = lo, end = hi;
        if (t0 > 0 || t1 < a.T) {
            const int rlo = t0 * a.k, rhi = t1 * a.k;
            int b = lo, c = hi;
            while (b < c) { // first route >= rlo
                const int m = (b + c) >> 1;
                if (a.routes[m] < rlo)
                    b = m + 1;
                else
                    c = m;
            }
            first = b;
            c = hi;
            while (b < c) { // first route >= rhi
                const int m = (b + c) >> 1;
                if (a.routes[m] < rhi)
                    b = m + 1;
                else
                    c = m;
            }
            end = b;
        }
        vlo[e] = first;
        vcnt[e] = end - first;
        vpre[e + 1] = (end - first + NCU - 1) / NCU;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < a.E; base += 32) {
            const int e = base + lane;
            int inc = e < a.E ? vpre[e + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o)
                    inc += v;
            }
            if (e < a.E)
                vpre[e + 1] = carry + inc;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0)
            vpre[0] = 0;
    }
    __syncthreads();
    const int NVr = vpre[a.E];
    const int NV = NVr + (a.wsd ? (ntok + NCU - 1) / NCU : 0);

    auto decode = [&](int v) {
        VUnit r;
        if (v < NVr) {
            int lo = 0, hi = a.E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (vpre[mid] <= v)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            r.e = lo;
            r.first = vlo[lo];
            r.col0 = (v - vpre[lo]) * NCU;
            r.ncols = min(NCU, vcnt[lo] - r.col0);
            r.w = a.wd + ((size_t)lo * a.H + n0) * a.rowbytes;
        } else {
            r.e = a.E;
            r.first = 0;
            r.col0 = (v - NVr) * NCU;
            r.ncols = min(NCU, ntok - r.col0);
            r.w = a.wsd + (size_t)n0 * a.rowbytes;
        }
        return r;
    };

    if (warp == CW) {
        // ---------------- producer: weights only, no wait on the gate/up kernel ----------------
        if (lane != 0)
            return;
        const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();
        uint32_t q = 0;
        for (int v = 0; v < NV; v++, q++) {
            const VUnit un = decode(v);
            const uint32_t slot = q % a.NS, use = q / a.NS;
            if (use > 0 && !mbar_wait_bounded(&empty[slot], (use - 1) & 1u)) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
                break;
            }
            if (*(volatile int *)&s_abort)
                break;
            mbar_arrive_expect_tx(&full[slot], (uint32_t)stage_bytes);
            bulk_copy_g2s(ring + (size_t)slot * stage_bytes, un.w, (uint32_t)stage_bytes, &full[slot], pol);
        }
        const uint32_t n_slots = (q < (uint32_t)a.NS ? q : (uint32_t)a.NS);
        for (uint32_t slot = 0; slot < n_slots; slot++) {
            const uint32_t last_use = (q - 1 - slot) / a.NS;
            if (!mbar_wait_bounded(&full[slot], last_use & 1u))
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers: wait for h, then one warp per stage ----------------
    pdl_wait();
    pdl_trigger();
    const int xstride = a.nbI * Q8_1_WORDS; // words per activation row
    const bool hs_on = a.hs_rows > 0;
    bool dead = false;
    if (hs_on) {
        // one bulk copy per activation row of the tile: the routed slots of
        // kept routes, then the shared expert's tokens
        if (tid == 0) {
            const int nslots = ntok * a.k + (a.wsd ? ntok : 0);
            const uint32_t xrow = (uint32_t)(xstride * 4);
            uint32_t bytes = 0;
            for (int ys = 0; ys < nslots; ys++) {
                if (ys < ntok * a.k) {
                    const int e = a.ids[t0 * a.k + ys];
                    if (e >= 0 && e < a.E)
                        bytes += xrow;
                } else {
                    bytes += xrow;
                }
            }
            mbar_arrive_expect_tx(hs_bar, bytes);
            for (int ys = 0; ys < nslots; ys++) {
                int row;
                if (ys < ntok * a.k) {
                    row = t0 * a.k + ys;
                    const int e = a.ids[row];
                    if (e < 0 || e >= a.E)
                        continue;
                } else {
                    row = a.T * a.k + t0 + (ys - ntok * a.k);
                }
                bulk_copy_g2s(hs + (size_t)ys * xstride, a.hq + (size_t)row * xstride, xrow, hs_bar,
                              l2_evict_normal_policy());
            }
        }
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(hs_bar, 0))) {
            if (lane == 0) {
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                *(volatile int *)&s_abort = 1;
            }
            dead = true;
        }
    }
    // Two ways to consume the ring, both safe for its parity waits (a warp
    // must never wait on a slot's use u while use u - 1 may be pending):
    //  * one warp per stage (all RN rows): warp v % CW takes stage v.  The host
    //    picks this when the ring holds every stage or NS is a multiple of CW,
    //    so that every use of a slot falls to the same warp, in order.
    //  * coop: every consumer warp takes part in every stage, in order, RN / CW
    //    rows each (rings of fewer than CW stages).
    for (int v = COOP ? 0 : warp; v < NV; v += COOP ? 1 : CW) {
        const VUnit un = decode(v);
        int my_r = 0, my_slot = 0; // column `lane`: its hq row and its y slot
        if (lane < un.ncols) {
            if (un.e < a.E) {
                my_r = a.routes[un.first + un.col0 + lane];
                my_slot = my_r - t0 * a.k;
            } else {
                const int t = t0 + un.col0 + lane;
                my_r = a.T * a.k + t;
                my_slot = ntok * a.k + (t - t0);
            }
        }
        const uint32_t slot = (uint32_t)v % a.NS, use = (uint32_t)v / a.NS;
        // warp-uniform: every lane takes the same branch to the __all_sync
        if (__any_sync(0xffffffffu, *(volatile int *)&s_abort != 0))
            dead = true;
        if (!dead) {
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], use & 1u));
            if (!got) {
                if (lane == 0) {
                    atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                    *(volatile int *)&s_abort = 1;
                }
                dead = true;
            }
        }
        if (!dead) {
            const uint8_t *st = ring + (size_t)slot * stage_bytes;
            // columns per pass: at most 4 (registers)
            constexpr int NCC = NC > 4 ? 4 : NC;
            for (int c0 = 0; c0 < un.ncols; c0 += NCC) {
                const int nc = min(NCC, un.ncols - c0);
                // warp-collective shuffles stay outside the lane-dependent block loop
                const uint32_t *xc[NCC]; // activation row of each column (shared or global)
                int ys[NCC];
#pragma unroll
                for (int c = 0; c < NCC; c++) {
                    const int cc = c0 + (c < nc ? c : 0);
                    const int r = __shfl_sync(0xffffffffu, my_r, cc);
                    ys[c] = __shfl_sync(0xffffffffu, my_slot, cc);
                    xc[c] = hs_on ? hs + (size_t)ys[c] * xstride : a.hq + (size_t)r * xstride;
                }
                if (COOP)
                    stage_dots<RPW, NCC>(st, a.rowbytes, warp, CW, xc, ys, nc, a.nbI, lane, ybuf);
                else
                    stage_dots<RN, NCC>(st, a.rowbytes, 0, 1, xc, ys, nc, a.nbI, lane, ybuf);
            }
        }
        if (COOP) {
            named_barrier(1, CW * 32); // every consumer warp is done with the stage
            if (tid == 0 && !dead)
                mbar_arrive(&empty[slot]);
        } else {
            __syncwarp();
            if (lane == 0 && !dead)
                mbar_arrive(&empty[slot]);
        }
    }
    named_barrier(1, CW * 32);
    if (dead || *(volatile int *)&s_abort)
        return;
    // combine: out[t][n] = sum_j fl(w * y) in slot order, then + shared
    for (int idx = tid; idx < ntok * RN; idx += CW * 32) {
        const int tl = idx / RN, i = idx % RN;
        const int t = t0 + tl;
        float acc = 0.0f;
        for (int j = 0; j < a.k; j++) {
            const int e = a.ids[(size_t)t * a.k + j];
            if (e >= 0 && e < a.E)
                acc = __fadd_rn(acc, __fmul_rn(a.weights[(size_t)t * a.k + j], ybuf[(tl * a.k + j) * RN + i]));
        }
        if (a.wsd)
            acc = __fadd_rn(acc, ybuf[(ntok * a.k + tl) * RN + i]);
        a.out[(size_t)t * a.H + n0 + i] = acc;
    }
}

template <int NC, bool COOP>
luce_status launch_down(const DownArgs &a, dim3 grid, size_t smem, cudaStream_t stream)
{
    static luce_host::SmemLimit limit;
    auto kern = k_down_combine<NC, COOP>;
    if (limit.raise(kern, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    const luce_status st = luce_host::launch(kern, grid, dim3((CW + 1) * 32), smem, stream, a);
    if (st != LUCE_OK)
        limit.forget();
    return st;
}

template <int NC>
luce_status launch_down_mode(const DownArgs &a, dim3 grid, size_t smem, cudaStream_t stream)
{
    return a.coop ? launch_down<NC, true>(a, grid, smem, stream) : launch_down<NC, false>(a, grid, smem, stream);
}

} // namespace

using namespace luce_host;

extern "C" luce_status luce_moe_down_combine(const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_down,
                                             const luce_block_q8_1 *hq, const int32_t *ids, const float *weights,
                                             const int32_t *offsets, const int32_t *routes, int T, int k, int E,
                                             int H, int I, float *out, int variant, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 64 || (int64_t)T * k > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 256 != 0 || I % 256 != 0 || I / 32 > 1024 || H > (1 << 19))
        return LUCE_ERR_INVALID_ARG;
    if (variant != 0)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!w_down || !hq || !ids || !weights || !offsets || !routes || !out)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(w_down, 16) || (ws_down && !aligned(ws_down, 16)) || !aligned(hq, 16) || !aligned(ids, 4) ||
        !aligned(weights, 4) || !aligned(offsets, 4) || !aligned(routes, 4) || !aligned(out, 4))
        return LUCE_ERR_INVALID_ARG;
    DownArgs a;
    a.wd = reinterpret_cast<const uint8_t *>(w_down);
    a.wsd = reinterpret_cast<const uint8_t *>(ws_down);
    a.hq = reinterpret_cast<const uint32_t *>(hq);
    a.ids = ids;
    a.weights = weights;
    a.offsets = offsets;
    a.routes = routes;
    a.out = out;
    a.T = T;
    a.k = k;
    a.E = E;
    a.H = H;
    a.I = I;
    a.nbI = I / 32;
    a.rowbytes = a.nbI * Q8_0_BYTES;
    // y buffer: (TT*k + TT) slots x RN floats, at most 32 KB
    const int per_tok = (k + 1) * RN * (int)sizeof(float);
    a.TT = std::max(1, std::min(T, (32 * 1024) / per_tok));
    // ring: every stage of a CTA at once when it fits in ~100 KB
    const long long Tk = (long long)a.TT * k;
    const long long nv_up = std::min<long long>(E, Tk) + Tk / NCU + (ws_down ? (a.TT + NCU - 1) / NCU : 0);
    const int stage = RN * a.rowbytes;
    a.NS = (int)std::max<long long>(2, std::min<long long>(nv_up, ((long long)g_tuning.down_budget_kb * 1024) / stage));
    // a ring that is reused is consumed one warp per stage only when NS is a
    // multiple of CW (each slot then always falls to the same warp)
    a.coop = 0;
    if (a.NS < nv_up) {
        if (a.NS >= CW)
            a.NS -= a.NS % CW;
        else
            a.coop = 1;
    }
    a.evict_first = g_tuning.evict_first;
    // activation rows of a tile in shared memory when they fit in 24 KB (a row
    // is a multiple of 16 bytes since I % 256 == 0)
    const size_t xrow = (size_t)a.nbI * Q8_1_BYTES;
    const int slots = a.TT * k + (ws_down ? a.TT : 0);
    a.hs_rows = (g_tuning.down_stage && (size_t)slots * xrow <= 24 * 1024) ? slots : 0;
    const size_t smem = (size_t)a.NS * stage + (size_t)(2 * a.NS + 2) * sizeof(uint64_t) + (size_t)a.hs_rows * xrow +
                        (size_t)(a.TT * k + a.TT) * RN * sizeof(float) + (size_t)(3 * E + 1) * sizeof(int);
    const int tiles = (T + a.TT - 1) / a.TT;
    dim3 grid((unsigned)tiles, (unsigned)(H / RN));
    const int maxcols = std::min(a.TT, NCU);
    cudaStream_t st = as_stream(stream);
    if (maxcols <= 1)
        return launch_down_mode<1>(a, grid, smem, st);
    if (maxcols <= 2)
        return launch_down_mode<2>(a, grid, smem, st);
    if (maxcols <= 4)
        return launch_down_mode<4>(a, grid, smem, st);
    return launch_down_mode<8>(a, grid, smem, st);
}
