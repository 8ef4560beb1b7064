// glu_pair.cu -- the Q8_0 x q8_1 gate/up products of every routed token and
// of the shared expert, fused with the (clamped) SwiGLU and the q8_1
// quantization of its output, and its C-ABI entry point.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving".  What the kernel computes follows the commit
// "RDNA4 Q8_0 gate/up pair" (both matrices read with one load of each
// activation fragment, each product with its own partial sums and
// reduction, the GLU in the epilogue) and the commit "fused DS4.1 decode
// kernels" (one expert grouping per layer, so each selected expert's
// weights cross HBM once).  Its GB300 shape is our own:
//
//  * Work is a flat list of 32-row GROUPS.  A virtual expert is an expert with
//    up to 32 of its routed columns (tokens); experts with more columns, and
//    the shared expert (all T tokens), are split into several.  Each virtual
//    expert has I/32 groups (one q8_1 block of h per column and group).
//  * Each CTA takes a contiguous range of whole groups and quantizes every
//    group it computed from its own shared memory, so no CTA ever waits for
//    another.  Two CTAs run per SM with ~108 KB rings each: measured on the
//    decode stack, this beats both one CTA per SM with a larger ring and
//    ranges balanced at a finer grain (whose groups shared by two CTAs cost
//    more in their epilogue than the balance gains), and it leaves room for
//    the down kernel's CTAs to start early under programmatic launch.
//  * Thread 0 streams each CTA's parts (RU gate rows + RU up rows, ~35-70 KB)
//    into a ring of shared-memory stages (~175-210 KB: a decode step's whole
//    share of the weights is requested at once) with cp.async.bulk
//    completing on per-stage mbarriers, and refills a stage once every warp
//    has passed the CTA barrier that ends its part.
//  * A lane owns Q8_0 blocks b = lane, lane + 32, ... of a row.  The q8_1
//    activation rows of the current virtual expert's columns are staged in
//    shared memory (when they fit) and each block is loaded once for the gate
//    AND the up row.  Block sums are exact int32 dp4a sums; the fp32 partials
//    are reduced across the warp.
//  * Every mbarrier wait is bounded (LUCE_FAULT_TIMEOUT, never expected); a
//    CTA that gives up keeps every CTA barrier in step, skips the arithmetic,
//    and drains its copies in flight before it exits.
//  * With programmatic dependent launch the CTAs start while the previous
//    kernel (the grouping) still runs: they prefetch their slice of the
//    shared expert's rows into L2 (those rows are needed whatever the
//    routing is) and then wait for the grouping's results.
#include <algorithm>
#include <climits>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_glu)

namespace {

using namespace luce;

constexpr int NCU = 32;          // columns per virtual expert (<= 32: one per lane)
constexpr int HB_STRIDE = NCU + 1;
constexpr int CW = 8;            // warps per CTA
constexpr int THREADS = CW * 32;

struct GluArgs {
    const uint8_t *wg, *wu;   // [E][I][rowbytes]
    const uint8_t *wsg, *wsu; // [I][rowbytes] or null
    const uint32_t *xq;       // [T][nb] q8_1 blocks, as 9 words each
    const int32_t *offsets;   // [E+1]
    const int32_t *routes;    // [T*k]
    float *h;                 // [T*k+T][I]
    uint32_t *hq;             // [T*k+T][I/32] q8_1 blocks
    int T, k, E, H, I;
    float clamp;
    int nb, rowbytes;
    int RU;      // rows per part (divides 32)
    int NS;      // stages (one part each) in the ring
    int xs_cols; // activation columns staged in shared memory (0: read through L1)
    int prefetch; // warm L2 with the shared expert before waiting
    int evict_first;
};

struct Group {
    const uint8_t *g, *u; // gate / up rows of this virtual expert
    int v;                // virtual expert
    int e;                // expert (E = shared)
    int col0, ncols;      // column range within the expert's routes / tokens
    int grp;              // 32-row group
};

__device__ __forceinline__ Group decode_group(const GluArgs &a, const int *vpre, int NVr, long long gi)
{
    const int G = a.I / 32;
    Group r;
    r.v = (int)(gi / G);
    r.grp = (int)(gi % G);
    if (r.v < NVr) {
        // the largest e with vpre[e] <= v owns virtual expert v
        int lo = 0, hi = a.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (vpre[mid] <= r.v)
                lo = mid;
            else
                hi = mid - 1;
        }
        r.e = lo;
        r.col0 = (r.v - vpre[lo]) * NCU;
        r.ncols = min(NCU, a.offsets[lo + 1] - a.offsets[lo] - r.col0);
        r.g = a.wg + (size_t)lo * a.I * a.rowbytes;
        r.u = a.wu + (size_t)lo * a.I * a.rowbytes;
    } else {
        r.e = a.E;
        r.col0 = (r.v - NVr) * NCU;
        r.ncols = min(NCU, a.T - r.col0);
        r.g = a.wsg;
        r.u = a.wsu;
    }
    return r;
}

template <int NC>
__global__ void __launch_bounds__(THREADS) k_glu_pair(const GluArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int half_bytes = a.RU * a.rowbytes;
    const int stage_bytes = 2 * half_bytes;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * stage_bytes);
    // lane -> block mapping of the weight rows (conflict-free for nb % 64 == 0)
    const int map = (a.nb % 64 == 0) ? ROWMAP_PAIRS : ROWMAP_PLAIN;
    // staged activation rows: block b at word 9 b + xpad (b / 32), so that
    // blocks b and b + 32 (read by one load instruction) sit 16 banks apart
    const int xpad = map == ROWMAP_PAIRS ? 16 : 0;
    const int xs_stride = a.nb * Q8_1_WORDS + xpad * (a.nb >> 5);
    uint32_t *xs = reinterpret_cast<uint32_t *>(full + a.NS); // [xs_cols][xs_stride]
    int *vpre = reinterpret_cast<int *>(xs + (size_t)a.xs_cols * xs_stride); // [E + 1]
    float *hbuf = reinterpret_cast<float *>(vpre + a.E + 1); // [2][32][HB_STRIDE]
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < a.NS; s++)
            mbar_init(&full[s], 1);
        fence_mbar_init();
        s_abort = 0;
        // before the grouping has finished: warm L2 with this CTA's slice of
        // the shared expert (needed whatever the routing)
        if (a.wsg && a.prefetch) {
            const size_t total = (size_t)a.I * a.rowbytes; // multiple of 16
            const size_t chunk = ((total / gridDim.x) + 15) & ~size_t(15);
            const size_t off = chunk * blockIdx.x;
            if (off < total) {
                const uint32_t n = (uint32_t)min(chunk, total - off);
                prefetch_l2(a.wsg + off, n);
                prefetch_l2(a.wsu + off, n);
            }
        }
    }
    pdl_wait();
    pdl_trigger();
    // virtual experts per expert, then an inclusive scan: vpre[e] = first v of e
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int cnt = a.offsets[e + 1] - a.offsets[e];
        vpre[e + 1] = (cnt + NCU - 1) / NCU;
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
    const int NV = NVr + (a.wsg ? (a.T + NCU - 1) / NCU : 0);
    const int G = a.I / 32;
    const long long NG = (long long)NV * G; // groups
    const long long g0 = NG * blockIdx.x / gridDim.x, g1 = NG * (blockIdx.x + 1) / gridDim.x;
    const int PPG = 32 / a.RU; // parts per group
    const long long NP = (g1 - g0) * PPG;
    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();

    // thread 0 requests part q (of this CTA's NP) into stage q % NS
    auto issue = [&](long long q) {
        const Group gr = decode_group(a, vpre, NVr, g0 + q / PPG);
        const int p = (int)(q % PPG);
        const size_t row0 = (size_t)gr.grp * 32 + (size_t)p * a.RU;
        const uint32_t slot = (uint32_t)(q % a.NS);
        uint8_t *dst = ring + (size_t)slot * stage_bytes;
        mbar_arrive_expect_tx(&full[slot], (uint32_t)stage_bytes);
        bulk_copy_g2s(dst, gr.g + row0 * a.rowbytes, (uint32_t)half_bytes, &full[slot], pol);
        bulk_copy_g2s(dst + half_bytes, gr.u + row0 * a.rowbytes, (uint32_t)half_bytes, &full[slot], pol);
    };
    long long issued = 0, waited = 0; // thread 0: parts requested / seen complete
    if (tid == 0) {
        for (; issued < NP && issued < a.NS; issued++)
            issue(issued);
    }

    const int xstride = a.nb * Q8_1_WORDS; // words per activation row
    bool dead = false;
    int cur_v = -1;
    int my_t = 0, my_r = 0; // lane c holds column c's token and h row
    bool x_in_smem = false;
    long long q = 0;
    int par = 0;
    for (long long gi = g0; gi < g1; gi++, par ^= 1) {
        const Group gr = decode_group(a, vpre, NVr, gi);
        if (gr.v != cur_v) {
            cur_v = gr.v;
            my_t = 0;
            my_r = 0;
            if (lane < gr.ncols) {
                if (gr.e < a.E) {
                    my_r = a.routes[a.offsets[gr.e] + gr.col0 + lane];
                    my_t = my_r / a.k;
                } else {
                    my_t = gr.col0 + lane;
                    my_r = a.T * a.k + my_t;
                }
            }
            x_in_smem = gr.ncols <= a.xs_cols;
            if (x_in_smem) {
                // stage the columns' q8_1 rows: warp w copies columns w, w+CW, ...
                // (every warp is past the previous part's barrier)
                for (int c = warp; c < gr.ncols; c += CW) {
                    const int t = __shfl_sync(0xffffffffu, my_t, c);
                    const uint32_t *src = a.xq + (size_t)t * xstride;
                    uint32_t *dst = xs + (size_t)c * xs_stride;
                    for (int w = lane; w < xstride; w += 32)
                        dst[w + xpad * ((w / Q8_1_WORDS) >> 5)] = __ldg(src + w);
                }
                __syncthreads();
            }
        }
        float *hb = hbuf + par * 32 * HB_STRIDE;
        for (int p = 0; p < PPG; p++, q++) {
            const uint32_t slot = (uint32_t)(q % a.NS), use = (uint32_t)(q / a.NS);
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
                } else if (tid == 0) {
                    waited = q + 1;
                }
            }
            if (!dead) {
                const uint8_t *st = ring + (size_t)slot * stage_bytes;
                for (int i = warp; i < a.RU; i += CW) {
                    const int prow = p * a.RU + i; // row within the group
                    const uint8_t *grow = st + (size_t)i * a.rowbytes;
                    const uint8_t *urow = st + half_bytes + (size_t)i * a.rowbytes;
                    for (int c0 = 0; c0 < gr.ncols; c0 += NC) {
                        const int nc = min(NC, gr.ncols - c0);
                        const uint32_t *xc[NC]; // activation row of each column (shared or global)
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            const int cc = c0 + (c < nc ? c : 0);
                            const int t = __shfl_sync(0xffffffffu, my_t, cc);
                            xc[c] = x_in_smem ? xs + (size_t)cc * xs_stride : a.xq + (size_t)t * xstride;
                        }
                        float ag[NC], au[NC];
#pragma unroll
                        for (int c = 0; c < NC; c++)
                            ag[c] = au[c] = 0.0f;
                        const int xp = x_in_smem ? xpad : 0;
                        const int nbl = rowmap_blocks(map, a.nb, lane);
                        for (int j = 0; j < nbl; j++) {
                            const int b = rowmap_block(map, lane, j);
                            Q80Block gb, ub;
                            load_q8_0_smem(grow, b, gb);
                            load_q8_0_smem(urow, b, ub);
#pragma unroll
                            for (int c = 0; c < NC; c++) {
                                if (c < nc) {
                                    Q81Block xb;
                                    load_q8_1_any(xc[c] + (size_t)b * Q8_1_WORDS + xp * (b >> 5), xb);
                                    const int sg = dot_q8_block(gb.q, xb.q);
                                    const int su = dot_q8_block(ub.q, xb.q);
                                    ag[c] = fmaf(gb.d * xb.d, (float)sg, ag[c]);
                                    au[c] = fmaf(ub.d * xb.d, (float)su, au[c]);
                                }
                            }
                        }
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            if (c < nc) {
                                const float g = warp_sum(ag[c]);
                                const float uu = warp_sum(au[c]);
                                if (lane == 0)
                                    hb[prow * HB_STRIDE + c0 + c] = swiglu(g, uu, a.clamp);
                            }
                        }
                    }
                }
            }
            __syncthreads(); // every warp is done with this stage
            if (tid == 0 && !*(volatile int *)&s_abort && issued < NP) {
                issue(issued); // into the stage just released
                issued++;
            }
        }
        // all 32 rows of the group are in hb (the barrier ending its last part)
        if (!dead && !*(volatile int *)&s_abort) {
            for (int c = warp; c < gr.ncols; c += CW) {
                const int r = __shfl_sync(0xffffffffu, my_r, c);
                const float v = hb[lane * HB_STRIDE + c];
                a.h[(size_t)r * a.I + (size_t)gr.grp * 32 + lane] = v;
                quantize_q8_1_warp(v, a.hq + ((size_t)r * G + gr.grp) * Q8_1_WORDS, lane);
            }
        }
    }
    // no bulk copy may still be writing shared memory when the CTA exits (only
    // after a timeout can a requested part be left unwaited; each stage holds
    // at most one of them, since nothing is requested after the abort)
    if (tid == 0) {
        for (long long r = waited; r < issued; r++) {
            if (!mbar_wait_bounded(&full[r % a.NS], (uint32_t)(r / a.NS) & 1u))
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        }
    }
}

// Per template instance and device: the dynamic shared memory set on the
// kernel (cached, so that steady-state calls make no attribute call).
template <int NC>
luce_status launch_glu(const GluArgs &a, cudaStream_t stream, size_t smem, int grid)
{
    static luce_host::SmemLimit limit;
    auto kern = k_glu_pair<NC>;
    if (limit.raise(kern, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    const luce_status st = luce_host::launch(kern, dim3(grid), dim3(THREADS), smem, stream, a);
    if (st != LUCE_OK)
        limit.forget();
    return st;
}

} // namespace

using namespace luce_host;

extern "C" luce_status luce_moe_glu_pair(const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                                         const luce_block_q8_0 *ws_gate, const luce_block_q8_0 *ws_up,
                                         const luce_block_q8_1 *xq, const int32_t *offsets, const int32_t *routes,
                                         int T, int k, int E, int H, int I, float clamp, float *h,
                                         luce_block_q8_1 *hq, int variant, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 64 || (int64_t)T * k > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 256 != 0 || I % 256 != 0 || H / 32 > 1024 || I > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (variant != 0 || (ws_gate == nullptr) != (ws_up == nullptr) || !(clamp == clamp))
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!w_gate || !w_up || !xq || !offsets || !routes || !h || !hq)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(w_gate, 16) || !aligned(w_up, 16) || (ws_gate && (!aligned(ws_gate, 16) || !aligned(ws_up, 16))) ||
        !aligned(xq, 16) || !aligned(hq, 16) || !aligned(h, 4) || !aligned(offsets, 4) || !aligned(routes, 4))
        return LUCE_ERR_INVALID_ARG;

    GluArgs a;
    a.wg = reinterpret_cast<const uint8_t *>(w_gate);
    a.wu = reinterpret_cast<const uint8_t *>(w_up);
    a.wsg = reinterpret_cast<const uint8_t *>(ws_gate);
    a.wsu = reinterpret_cast<const uint8_t *>(ws_up);
    a.xq = reinterpret_cast<const uint32_t *>(xq);
    a.offsets = offsets;
    a.routes = routes;
    a.h = h;
    a.hq = reinterpret_cast<uint32_t *>(hq);
    a.T = T;
    a.k = k;
    a.E = E;
    a.H = H;
    a.I = I;
    a.clamp = clamp;
    a.nb = H / 32;
    a.rowbytes = a.nb * Q8_0_BYTES;
    const Tuning &tu = g_tuning;
    // a part (RU gate rows + RU up rows) of about 35 KB, but at least one row
    // per warp while a part stays under 72 KB
    int RU = 32;
    while (RU > 1 && 2 * RU * a.rowbytes > tu.glu_part_kb * 1024 &&
           !(RU <= CW && 2 * RU * a.rowbytes <= 2 * tu.glu_part_kb * 1024))
        RU /= 2;
    a.RU = RU;
    // activation rows in shared memory when up to 32 columns fit in 40 KB
    const int maxcols = std::min(T, NCU);
    const size_t xrow = (size_t)a.nb * Q8_1_BYTES;
    const size_t xrow_pad = xrow + (a.nb % 64 == 0 ? (size_t)64 * (a.nb / 32) : 0); // staged row with bank padding
    a.xs_cols = (tu.glu_xs && maxcols * xrow_pad <= 40 * 1024) ? maxcols : 0;
    a.prefetch = tu.glu_prefetch;
    a.evict_first = tu.evict_first;
    const size_t stage = (size_t)2 * RU * a.rowbytes;
    const size_t fixed = (size_t)a.xs_cols * xrow_pad + (size_t)(E + 1) * sizeof(int) +
                         (size_t)2 * 32 * HB_STRIDE * sizeof(float) + 64;
    const size_t budget = (size_t)tu.glu_budget_kb * 1024;
    int NS = (int)std::min<size_t>(16, (budget - fixed) / (stage + 8));
    NS = std::max(NS, 2);
    a.NS = NS;
    const size_t smem = (size_t)NS * stage + (size_t)NS * sizeof(uint64_t) + fixed;
    const int grid = sm_count() * std::max(1, tu.glu_cps);
    cudaStream_t st = as_stream(stream);
    if (maxcols <= 1)
        return launch_glu<1>(a, st, smem, grid);
    if (maxcols <= 2)
        return launch_glu<2>(a, st, smem, grid);
    if (maxcols <= 4)
        return launch_glu<4>(a, st, smem, grid);
    return launch_glu<8>(a, st, smem, grid);
}
