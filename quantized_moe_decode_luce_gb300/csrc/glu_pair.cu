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
//  * Work is a flat list of PARTS.  A virtual expert is an expert with up to
//    32 of its routed columns (tokens); experts with more columns, and the
//    shared expert (all T tokens), are split into several.  Each virtual
//    expert has I/32 row groups (one q8_1 block of h per column and group),
//    and a group is cut into parts of RU gate rows + RU up rows (~35 KB).
//  * The CTAs take equal contiguous ranges of parts, so every SM streams the
//    same number of bytes.  A group whose parts all fall in one CTA is
//    quantized from that CTA's shared memory.  At most two groups per CTA
//    (the ends of its range) are shared with a neighbour: each side writes
//    its rows of h, and the side whose parts complete the group (a
//    per-group counter in the caller's workspace) quantizes it from L2 and
//    resets the counter.  No CTA ever waits for another.
//  * Thread 0 streams the CTA's parts into a ring of shared-memory stages
//    with cp.async.bulk completing on per-stage mbarriers, and refills a
//    stage once every warp has passed the CTA barrier that ends its part.
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
    unsigned int *group_cnt;  // [nv_max * I/32] zero-filled counters, left zero-filled
    const uint8_t *wd, *wsd;  // down weights to prefetch into L2, or null
    int T, k, E, H, I;
    float clamp;
    int nb, rowbytes;
    int RU;      // rows per part (divides 32)
    int NS;      // stages (one part each) in the ring
    int xs_cols; // activation columns staged in shared memory (0: read through L1)
    int prefetch; // warm L2 with the shared expert before waiting
    int evict_first;
    int l2pf;     // prefetch this CTA's own parts into L2 (per thread)
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
    uint32_t *xs = reinterpret_cast<uint32_t *>(full + a.NS); // [xs_cols][nb][9]
    int *vpre = reinterpret_cast<int *>(xs + (size_t)a.xs_cols * a.nb * Q8_1_WORDS); // [E + 1]
    float *hbuf = reinterpret_cast<float *>(vpre + a.E + 1); // [2][32][HB_STRIDE]
    __shared__ int s_abort, s_last;

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
    const int CL = 32 / a.RU;                    // parts per group
    const long long NPT = (long long)NV * G * CL; // parts of the call
    const long long u0 = NPT * blockIdx.x / gridDim.x, u1 = NPT * (blockIdx.x + 1) / gridDim.x;
    const long long NP = u1 - u0;
    const uint64_t pol = a.evict_first ? l2_evict_first_policy() : l2_evict_normal_policy();

    // thread 0 requests part q (of this CTA's NP) into stage q % NS
    auto issue = [&](long long q) {
        const long long u = u0 + q;
        const Group gr = decode_group(a, vpre, NVr, u / CL);
        const int p = (int)(u % CL);
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
    // Parts beyond the first ring-full: ask L2 for them now, through the
    // load/store path (one 128-byte line per thread and instruction), so that
    // their bulk copies later hit L2.  The bulk-copy engine of an SM moves far
    // less than its share of HBM bandwidth, and these requests use the rest.
    if (a.l2pf) {
        for (long long q = a.NS + warp; q < NP; q += CW) {
            const long long u = u0 + q;
            const Group gr = decode_group(a, vpre, NVr, u / CL);
            const size_t row0 = (size_t)gr.grp * 32 + (size_t)(u % CL) * a.RU;
            for (int off = lane * 128; off < half_bytes; off += 32 * 128) {
                prefetch_line_l2(gr.g + row0 * a.rowbytes + off);
                prefetch_line_l2(gr.u + row0 * a.rowbytes + off);
            }
        }
    }
    // The following down product's rows of the active experts (and of the
    // shared expert): this CTA's slice of them, into L2.
    if (a.wd) {
        const size_t dbytes = (size_t)a.H * (a.I / 32) * Q8_0_BYTES; // one expert's down matrix
        const int nact = NVr > 0 ? a.E : 0;
        const size_t per = ((dbytes / gridDim.x) + 127) & ~size_t(127);
        const size_t lo = per * blockIdx.x, hi = min(dbytes, lo + per);
        for (int e = 0; e < nact; e++) {
            if (vpre[e + 1] == vpre[e])
                continue; // no routes for this expert
            const uint8_t *base = a.wd + (size_t)e * dbytes;
            for (size_t off = lo + (size_t)tid * 128; off < hi; off += (size_t)THREADS * 128)
                prefetch_line_l2(base + off);
        }
        if (a.wsd)
            for (size_t off = lo + (size_t)tid * 128; off < hi; off += (size_t)THREADS * 128)
                prefetch_line_l2(a.wsd + off);
    }

    const int xstride = a.nb * Q8_1_WORDS; // words per activation row
    bool dead = false;
    int cur_v = -1;
    int my_t = 0, my_r = 0; // lane c holds column c's token and h row
    bool x_in_smem = false;
    long long cur_g = -1;
    int par = 1;
    for (long long q = 0; q < NP; q++) {
        const long long u = u0 + q;
        const long long gi = u / CL;
        const int p = (int)(u % CL);
        const Group gr = decode_group(a, vpre, NVr, gi);
        if (gi != cur_g) {
            cur_g = gi;
            par ^= 1;
        }
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
                    uint32_t *dst = xs + (size_t)c * xstride;
                    for (int w = lane; w < xstride; w += 32)
                        dst[w] = __ldg(src + w);
                }
                __syncthreads();
            }
        }
        float *hb = hbuf + par * 32 * HB_STRIDE;
        const uint32_t slot = (uint32_t)(q % a.NS), use = (uint32_t)(q / a.NS);
        if (!dead && *(volatile int *)&s_abort)
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
                        xc[c] = x_in_smem ? xs + (size_t)cc * xstride : a.xq + (size_t)t * xstride;
                    }
                    float ag[NC], au[NC];
#pragma unroll
                    for (int c = 0; c < NC; c++)
                        ag[c] = au[c] = 0.0f;
                    for (int b = lane; b < a.nb; b += 32) {
                        Q80Block gb, ub;
                        load_q8_0_smem(grow, b, gb);
                        load_q8_0_smem(urow, b, ub);
#pragma unroll
                        for (int c = 0; c < NC; c++) {
                            if (c < nc) {
                                Q81Block xb;
                                load_q8_1_any(xc[c] + (size_t)b * Q8_1_WORDS, xb);
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
        __syncthreads(); // every warp is done with this stage and with hb's rows
        if (tid == 0 && !*(volatile int *)&s_abort && issued < NP) {
            issue(issued); // into the stage just released
            issued++;
        }
        // the end of this CTA's share of the group?
        if (p == CL - 1 || q == NP - 1) {
            const bool ok = !dead && !*(volatile int *)&s_abort;
            const int pfirst = (q - p >= 0) ? 0 : (int)(p - q); // first part of the group in this CTA
            const bool whole = pfirst == 0 && p == CL - 1;
            if (whole) {
                if (ok) {
                    for (int c = warp; c < gr.ncols; c += CW) {
                        const int r = __shfl_sync(0xffffffffu, my_r, c);
                        const float v = hb[lane * HB_STRIDE + c];
                        a.h[(size_t)r * a.I + (size_t)gr.grp * 32 + lane] = v;
                        quantize_q8_1_warp(v, a.hq + ((size_t)r * G + gr.grp) * Q8_1_WORDS, lane);
                    }
                }
            } else {
                // a group shared with a neighbouring CTA: write this side's rows
                const int r0 = pfirst * a.RU, nrows = (p - pfirst + 1) * a.RU;
                if (ok) {
                    for (int c = warp; c < gr.ncols; c += CW) {
                        const int r = __shfl_sync(0xffffffffu, my_r, c);
                        if (lane < nrows)
                            a.h[(size_t)r * a.I + (size_t)gr.grp * 32 + r0 + lane] =
                                hb[(r0 + lane) * HB_STRIDE + c];
                    }
                }
                __threadfence();
                __syncthreads();
                if (tid == 0) {
                    unsigned int *cnt = a.group_cnt + (size_t)gr.v * G + gr.grp;
                    const unsigned int mine = (unsigned)(p - pfirst + 1);
                    const unsigned int old = ok ? atomicAdd(cnt, mine) : 0u;
                    const bool last = ok && old + mine == (unsigned)CL;
                    if (last)
                        *cnt = 0u; // every part has arrived: leave the counter zero
                    s_last = last ? 1 : 0;
                }
                __syncthreads();
                if (s_last) {
                    __threadfence();
                    for (int c = warp; c < gr.ncols; c += CW) {
                        const int r = __shfl_sync(0xffffffffu, my_r, c);
                        const float v = __ldcg(&a.h[(size_t)r * a.I + (size_t)gr.grp * 32 + lane]);
                        quantize_q8_1_warp(v, a.hq + ((size_t)r * G + gr.grp) * Q8_1_WORDS, lane);
                    }
                }
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
    static size_t smem_set[64] = {0};
    auto kern = k_glu_pair<NC>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return LUCE_ERR_CUDA;
    if (smem_set[dev] < smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LUCE_ERR_CUDA;
        smem_set[dev] = smem;
    }
    return luce_host::launch(kern, dim3(grid), dim3(THREADS), smem, stream, a);
}

// Upper bound of the number of virtual experts of a call.
long long max_virtual_experts(int T, int k, int E, bool shared)
{
    const long long Tk = (long long)T * k;
    return std::min<long long>(E, Tk) + Tk / NCU + (shared ? (T + NCU - 1) / NCU : 0);
}

} // namespace

using namespace luce_host;

extern "C" size_t luce_moe_glu_workspace_bytes(int T, int k, int E, int I)
{
    if (T <= 0 || k <= 0 || E <= 0 || I <= 0)
        return 0;
    // one counter per (virtual expert, 32-row group), with the shared expert
    return (size_t)max_virtual_experts(T, k, E, true) * (size_t)(I / 32) * sizeof(unsigned int);
}

extern "C" luce_status luce_moe_glu_pair(const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                                         const luce_block_q8_0 *ws_gate, const luce_block_q8_0 *ws_up,
                                         const luce_block_q8_1 *xq, const int32_t *offsets, const int32_t *routes,
                                         int T, int k, int E, int H, int I, float clamp, float *h,
                                         luce_block_q8_1 *hq, void *workspace, size_t workspace_bytes,
                                         const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_down, int variant,
                                         void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 64 || (int64_t)T * k > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || H % 256 != 0 || I % 256 != 0 || H / 32 > 1024 || I > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (variant != 0 || (ws_gate == nullptr) != (ws_up == nullptr) || !(clamp == clamp))
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!w_gate || !w_up || !xq || !offsets || !routes || !h || !hq || !workspace)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(w_gate, 16) || !aligned(w_up, 16) || (ws_gate && (!aligned(ws_gate, 16) || !aligned(ws_up, 16))) ||
        !aligned(xq, 16) || !aligned(hq, 16) || !aligned(h, 4) || !aligned(offsets, 4) || !aligned(routes, 4) ||
        !aligned(workspace, 4))
        return LUCE_ERR_INVALID_ARG;
    if (workspace_bytes < luce_moe_glu_workspace_bytes(T, k, E, I))
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
    a.group_cnt = reinterpret_cast<unsigned int *>(workspace);
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
    a.xs_cols = (tu.glu_xs && maxcols * xrow <= 40 * 1024) ? maxcols : 0;
    a.prefetch = tu.glu_prefetch;
    a.evict_first = tu.evict_first;
    a.l2pf = tu.glu_l2pf;
    a.wd = tu.glu_down_pf ? reinterpret_cast<const uint8_t *>(w_down) : nullptr;
    a.wsd = (tu.glu_down_pf && w_down) ? reinterpret_cast<const uint8_t *>(ws_down) : nullptr;
    const size_t stage = (size_t)2 * RU * a.rowbytes;
    const size_t fixed = (size_t)a.xs_cols * xrow + (size_t)(E + 1) * sizeof(int) +
                         (size_t)2 * 32 * HB_STRIDE * sizeof(float) + 64;
    const size_t budget = (size_t)tu.glu_budget_kb * 1024;
    int NS = (int)std::min<size_t>(16, (budget > fixed ? budget - fixed : 0) / (stage + 8));
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
