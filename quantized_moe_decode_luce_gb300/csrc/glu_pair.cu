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
//  * Persistent CTAs (one per SM) take contiguous ranges of whole groups, so
//    every group is quantized from shared memory by the CTA that computed it
//    and no CTA ever waits for another.  Whole groups are a coarse unit, but
//    one SM can pull several times its even share of HBM bandwidth, so the
//    bytes per CTA need not be balanced finely: what matters is that every
//    SM keeps enough requests in flight.
//  * One producer thread streams each group as parts of RU gate rows + RU up
//    rows (~35 KB) into a ring of shared-memory stages (~175 KB: a decode
//    step's whole share of the weights is requested at once) with
//    cp.async.bulk completing on per-stage mbarriers; eight consumer warps
//    compute from shared memory and release each stage on its "empty"
//    mbarrier.
//  * A consumer lane owns Q8_0 blocks b = lane, lane + 32, ... of a row.  The
//    q8_1 activation rows of the current virtual expert's columns are staged
//    in shared memory (when they fit) and each block is loaded once for the
//    gate AND the up row.  Block sums are exact int32 dp4a sums; the fp32
//    partials are reduced across the warp.
//  * Every device wait is bounded (LUCE_FAULT_TIMEOUT, never expected); a CTA
//    that gives up drains its copies in flight before it exits.
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
constexpr int CW = 8;            // consumer warps
constexpr int THREADS = (CW + 1) * 32;

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
    int RU;     // rows per part (divides 32)
    int CL;     // parts per 32-row group
    int NS;     // stages (one part each) in the ring
    int xs_cols; // activation columns staged in shared memory (0: read through L1)
};

struct Part {
    const uint8_t *g, *u; // gate / up rows of this virtual expert
    int v;                // virtual expert
    int e;                // expert (E = shared)
    int col0, ncols;      // column range within the expert's routes / tokens
    int grp, p;           // 32-row group, part within the group
};

__device__ __forceinline__ Part decode_part(const GluArgs &a, const int *vpre, int NVr, long long u)
{
    const int G = a.I / 32;
    const long long per_v = (long long)G * a.CL;
    Part r;
    r.v = (int)(u / per_v);
    const int rem = (int)(u % per_v);
    r.grp = rem / a.CL;
    r.p = rem % a.CL;
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
__global__ void __launch_bounds__(THREADS, 1) k_glu_pair(const GluArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int half_bytes = a.RU * a.rowbytes;
    const int stage_bytes = 2 * half_bytes;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * stage_bytes);
    uint64_t *empty = full + a.NS;
    uint32_t *xs = reinterpret_cast<uint32_t *>(empty + a.NS); // [xs_cols][nb][9]
    int *vpre = reinterpret_cast<int *>(xs + (size_t)a.xs_cols * a.nb * Q8_1_WORDS); // [E + 1]
    float *hbuf = reinterpret_cast<float *>(vpre + a.E + 1); // [2][32][HB_STRIDE]
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    // Before the grouping has finished: warm L2 with this CTA's slice of the
    // shared expert (needed whatever the routing), then wait for it.
    if (a.wsg && warp == CW && lane == 0) {
        const size_t total = (size_t)a.I * a.rowbytes; // multiple of 16
        const size_t chunk = ((total / gridDim.x) + 15) & ~size_t(15);
        const size_t off = chunk * blockIdx.x;
        if (off < total) {
            const uint32_t n = (uint32_t)min(chunk, total - off);
            prefetch_l2(a.wsg + off, n);
            prefetch_l2(a.wsu + off, n);
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

    if (warp == CW) {
        // ---------------- producer: one thread streams the parts ----------------
        if (lane != 0)
            return;
        const uint64_t pol = l2_evict_first_policy();
        uint32_t q = 0;
        bool stop = false;
        for (long long gi = g0; gi < g1 && !stop; gi++) {
            const Part pt = decode_part(a, vpre, NVr, gi * a.CL);
            for (int p = 0; p < a.CL; p++, q++) {
                const uint32_t slot = q % a.NS, use = q / a.NS;
                if (use > 0 && !mbar_wait_bounded(&empty[slot], (use - 1) & 1u)) {
                    atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                    *(volatile int *)&s_abort = 1;
                    stop = true;
                    break;
                }
                if (*(volatile int *)&s_abort) {
                    stop = true;
                    break;
                }
                const size_t row0 = (size_t)pt.grp * 32 + (size_t)p * a.RU;
                uint8_t *dst = ring + (size_t)slot * stage_bytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)stage_bytes);
                bulk_copy_g2s(dst, pt.g + row0 * a.rowbytes, (uint32_t)half_bytes, &full[slot], pol);
                bulk_copy_g2s(dst + half_bytes, pt.u + row0 * a.rowbytes, (uint32_t)half_bytes, &full[slot], pol);
            }
        }
        // no bulk copy may still be writing shared memory when the CTA exits
        const uint32_t n_slots = (q < (uint32_t)a.NS ? q : (uint32_t)a.NS);
        for (uint32_t slot = 0; slot < n_slots; slot++) {
            const uint32_t last_use = (q - 1 - slot) / a.NS;
            if (!mbar_wait_bounded(&full[slot], last_use & 1u))
                atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
        }
        return;
    }

    // ---------------- consumers ----------------
    const int cthreads = CW * 32;
    const int xstride = a.nb * Q8_1_WORDS; // words per activation row
    bool dead = false;
    int cur_v = -1;
    int my_t = 0, my_r = 0; // lane c holds column c's token and h row
    bool x_in_smem = false;
    uint32_t q = 0;
    int par = 0;
    for (long long gi = g0; gi < g1; gi++, par ^= 1) {
        const Part pt = decode_part(a, vpre, NVr, gi * a.CL);
        if (pt.v != cur_v) {
            cur_v = pt.v;
            my_t = 0;
            my_r = 0;
            if (lane < pt.ncols) {
                if (pt.e < a.E) {
                    my_r = a.routes[a.offsets[pt.e] + pt.col0 + lane];
                    my_t = my_r / a.k;
                } else {
                    my_t = pt.col0 + lane;
                    my_r = a.T * a.k + my_t;
                }
            }
            x_in_smem = pt.ncols <= a.xs_cols;
            if (x_in_smem) {
                // stage the columns' q8_1 rows: warp w copies columns w, w+CW, ...
                // (every warp is past the previous group's products: the group
                // barrier below; the epilogue does not read xs)
                for (int c = warp; c < pt.ncols; c += CW) {
                    const int t = __shfl_sync(0xffffffffu, my_t, c);
                    const uint32_t *src = a.xq + (size_t)t * xstride;
                    uint32_t *dst = xs + (size_t)c * xstride;
                    for (int w = lane; w < xstride; w += 32)
                        dst[w] = __ldg(src + w);
                }
                named_barrier(1, cthreads);
            }
        }
        float *hb = hbuf + par * 32 * HB_STRIDE;
        for (int p = 0; p < a.CL; p++, q++) {
            const uint32_t slot = q % a.NS, use = q / a.NS;
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
                }
            }
            if (!dead) {
                const uint8_t *st = ring + (size_t)slot * stage_bytes;
                for (int i = warp; i < a.RU; i += CW) {
                    const int prow = p * a.RU + i; // row within the 32-row group
                    const uint8_t *grow = st + (size_t)i * a.rowbytes;
                    const uint8_t *urow = st + half_bytes + (size_t)i * a.rowbytes;
                    for (int c0 = 0; c0 < pt.ncols; c0 += NC) {
                        const int nc = min(NC, pt.ncols - c0);
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
            __syncwarp();
            if (lane == 0 && !dead)
                mbar_arrive(&empty[slot]);
        }
        // the group is complete: h and its q8_1 block per column
        named_barrier(1, cthreads);
        if (!dead && !*(volatile int *)&s_abort) {
            for (int c = warp; c < pt.ncols; c += CW) {
                const int r = __shfl_sync(0xffffffffu, my_r, c);
                const float v = hb[lane * HB_STRIDE + c];
                a.h[(size_t)r * a.I + (size_t)pt.grp * 32 + lane] = v;
                quantize_q8_1_warp(v, a.hq + ((size_t)r * G + pt.grp) * Q8_1_WORDS, lane);
            }
        }
    }
}

// Per template instance and device: the dynamic shared memory the kernel may
// use (cached, so that steady-state calls make no attribute calls).
template <int NC>
luce_status launch_glu(const GluArgs &a, cudaStream_t stream, size_t smem)
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
    return luce_host::launch(kern, dim3(luce_host::sm_count()), dim3(THREADS), smem, stream, a);
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
    // a part (RU gate rows + RU up rows) of about 35 KB, but at least one row
    // per consumer warp while a part stays under 72 KB
    int RU = 32;
    while (RU > 1 && 2 * RU * a.rowbytes > 36 * 1024 && !(RU <= CW && 2 * RU * a.rowbytes <= 72 * 1024))
        RU /= 2;
    a.RU = RU;
    a.CL = 32 / RU;
    // activation rows in shared memory when up to 32 columns fit in 40 KB
    const int maxcols = std::min(T, NCU);
    const size_t xrow = (size_t)a.nb * Q8_1_BYTES;
    a.xs_cols = (maxcols * xrow <= 40 * 1024) ? maxcols : 0;
    const size_t stage = (size_t)2 * RU * a.rowbytes;
    const size_t fixed = (size_t)a.xs_cols * xrow + (size_t)(E + 1) * sizeof(int) +
                         (size_t)2 * 32 * HB_STRIDE * sizeof(float) + 64;
    const size_t budget = 216 * 1024;
    int NS = (int)std::min<size_t>(16, (budget - fixed) / (stage + 16));
    NS = std::max(NS, 2);
    a.NS = NS;
    const size_t smem = (size_t)NS * stage + (size_t)2 * NS * sizeof(uint64_t) + fixed;
    cudaStream_t st = as_stream(stream);
    if (maxcols <= 1)
        return launch_glu<1>(a, st, smem);
    if (maxcols <= 2)
        return launch_glu<2>(a, st, smem);
    if (maxcols <= 4)
        return launch_glu<4>(a, st, smem);
    return launch_glu<8>(a, st, smem);
}
