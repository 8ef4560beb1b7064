// glu_pair.cu -- the Q8_0 x q8_1 gate/up products of every routed token and
// of the shared expert, fused with the (clamped) SwiGLU and the q8_1
// quantization of its output, and its C-ABI entry point.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving".  The design follows what the page's commit "RDNA4
// Q8_0 gate/up pair" describes (both matrices read with one load of each
// activation fragment, each product with its own partial sums and reduction,
// the GLU in the epilogue) and the commit "fused DS4.1 decode kernels" (one
// expert grouping per layer, so each selected expert's weights cross HBM once).
// Its GB300 shape is our own:
//
//  * Work unit = (virtual expert, group of 32 rows).  A virtual expert is an
//    expert with up to `ncu` of its routed columns (tokens); experts with
//    more columns, and the shared expert (all T tokens), are split into
//    several.  32 rows make one q8_1 block of h per column, so the epilogue
//    quantizes locally, with no cross-CTA exchange.
//  * Persistent CTAs take contiguous ranges of units.  One producer thread
//    streams the gate and up rows of each unit through a ring of shared-memory
//    stages with cp.async.bulk (no tensor map: rows are contiguous runs of
//    34-byte blocks, 16-byte aligned because H % 256 == 0), completing on
//    per-stage mbarriers; consumer warps compute from shared memory and free
//    each stage on its "empty" mbarrier.
//  * A consumer lane owns Q8_0 blocks b = lane, lane + 32, ... of a row;
//    the q8_1 activation block of each column is loaded once (read-only
//    path, L1-resident) and used for the gate AND the up row.  Block sums are
//    exact int32 dp4a sums; the fp32 partials are reduced across the warp.
//  * Every device wait is bounded (LUCE_FAULT_TIMEOUT, never expected); a
//    CTA that gives up drains its copies in flight before it exits.
#include <algorithm>
#include <climits>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_glu)

namespace {

using namespace luce;

constexpr int NCU_MAX = 32;      // columns per virtual expert (<= 32: one per lane)
constexpr int HB_STRIDE = NCU_MAX + 1;

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
    int S;   // row pairs per stage (divides 32)
    int NS;  // stages in the ring
    int ncu; // columns per virtual expert
};

struct Unit {
    const uint8_t *g, *u; // gate / up rows of this virtual expert
    int e;                // expert (E = shared)
    int col0, ncols;      // column range within the expert's routes / tokens
    int grp;              // 32-row group
};

__device__ __forceinline__ Unit decode_unit(const GluArgs &a, const int *vpre, int NVr, long long u)
{
    const int G = a.I / 32;
    const int v = (int)(u / G);
    Unit r;
    r.grp = (int)(u % G);
    if (v < NVr) {
        // the largest e with vpre[e] <= v is the expert owning virtual expert v
        int lo = 0, hi = a.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (vpre[mid] <= v)
                lo = mid;
            else
                hi = mid - 1;
        }
        r.e = lo;
        r.col0 = (v - vpre[lo]) * a.ncu;
        const int cnt = a.offsets[lo + 1] - a.offsets[lo];
        r.ncols = min(a.ncu, cnt - r.col0);
        r.g = a.wg + (size_t)lo * a.I * a.rowbytes;
        r.u = a.wu + (size_t)lo * a.I * a.rowbytes;
    } else {
        r.e = a.E;
        r.col0 = (v - NVr) * a.ncu;
        r.ncols = min(a.ncu, a.T - r.col0);
        r.g = a.wsg;
        r.u = a.wsu;
    }
    return r;
}

template <int CW, int NC>
__global__ void __launch_bounds__((CW + 1) * 32) k_glu_pair(const GluArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int stage_bytes = 2 * a.S * a.rowbytes;
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.NS * stage_bytes);
    uint64_t *empty = full + a.NS;
    int *vpre = reinterpret_cast<int *>(empty + a.NS); // [E + 1]
    float *hbuf = reinterpret_cast<float *>(vpre + a.E + 1 + 1);
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wpart = min(a.S, CW); // consumer warps that touch one stage
    if (tid == 0) {
        for (int s = 0; s < a.NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], wpart);
        }
        fence_mbar_init();
        s_abort = 0;
    }
    // virtual experts per expert, then an inclusive scan: vpre[e] = first v of e
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int cnt = a.offsets[e + 1] - a.offsets[e];
        vpre[e + 1] = (cnt + a.ncu - 1) / a.ncu;
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
    const int NV = NVr + (a.wsg ? (a.T + a.ncu - 1) / a.ncu : 0);
    const long long N = (long long)NV * (a.I / 32);
    const long long u0 = N * blockIdx.x / gridDim.x, u1 = N * (blockIdx.x + 1) / gridDim.x;
    const int STG = 32 / a.S;

    if (warp == CW) {
        // ---------------- producer: one thread streams the rows ----------------
        if (lane != 0)
            return;
        const uint64_t pol = l2_evict_first_policy();
        const uint32_t half = (uint32_t)(a.S * a.rowbytes);
        uint32_t q = 0;
        bool ok = true;
        for (long long u = u0; u < u1 && ok; u++) {
            const Unit un = decode_unit(a, vpre, NVr, u);
            for (int s = 0; s < STG; s++, q++) {
                const uint32_t slot = q % a.NS, use = q / a.NS;
                if (use > 0 && !mbar_wait_bounded(&empty[slot], (use - 1) & 1u)) {
                    atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
                    *(volatile int *)&s_abort = 1;
                    ok = false;
                    break;
                }
                if (*(volatile int *)&s_abort) {
                    ok = false;
                    break;
                }
                const size_t row0 = (size_t)un.grp * 32 + (size_t)s * a.S;
                uint8_t *dst = ring + (size_t)slot * stage_bytes;
                mbar_arrive_expect_tx(&full[slot], 2 * half);
                bulk_copy_g2s(dst, un.g + row0 * a.rowbytes, half, &full[slot], pol);
                bulk_copy_g2s(dst + half, un.u + row0 * a.rowbytes, half, &full[slot], pol);
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
    bool dead = false;
    uint32_t q = 0;
    for (long long u = u0; u < u1; u++) {
        const Unit un = decode_unit(a, vpre, NVr, u);
        // lane c holds column c: its token t and its h row r
        int my_t = 0, my_r = 0;
        if (lane < un.ncols) {
            if (un.e < a.E) {
                my_r = a.routes[a.offsets[un.e] + un.col0 + lane];
                my_t = my_r / a.k;
            } else {
                my_t = un.col0 + lane;
                my_r = a.T * a.k + my_t;
            }
        }
        for (int s = 0; s < STG; s++, q++) {
            const uint32_t slot = q % a.NS, use = q / a.NS;
            // this warp's row pairs in the stage: p = s*S + i with p % CW == warp
            const int first = ((warp - s * a.S) % CW + CW) % CW;
            if (first >= a.S)
                continue;
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
                for (int i = first; i < a.S; i += CW) {
                    const int p = s * a.S + i; // row within the 32-row group
                    const uint8_t *grow = st + (size_t)i * a.rowbytes;
                    const uint8_t *urow = st + (size_t)(a.S + i) * a.rowbytes;
                    for (int c0 = 0; c0 < un.ncols; c0 += NC) {
                        const int nc = min(NC, un.ncols - c0);
                        int tcol[NC];
#pragma unroll
                        for (int c = 0; c < NC; c++)
                            tcol[c] = __shfl_sync(0xffffffffu, my_t, c0 + (c < nc ? c : 0));
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
                                    load_q8_1_global(a.xq + ((size_t)tcol[c] * a.nb + b) * Q8_1_WORDS, xb);
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
                                    hbuf[p * HB_STRIDE + c0 + c] = swiglu(g, uu, a.clamp);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && !dead)
                mbar_arrive(&empty[slot]);
        }
        named_barrier(1, cthreads);
        if (!dead && !*(volatile int *)&s_abort) {
            // epilogue: per column, the 32 h values of this row group -> h, hq
            for (int c = warp; c < un.ncols; c += CW) {
                const int r = __shfl_sync(0xffffffffu, my_r, c);
                const float v = hbuf[lane * HB_STRIDE + c];
                a.h[(size_t)r * a.I + (size_t)un.grp * 32 + lane] = v;
                quantize_q8_1_warp(v, a.hq + ((size_t)r * (a.I / 32) + un.grp) * Q8_1_WORDS, lane);
            }
        }
        named_barrier(1, cthreads);
    }
}

// Per template instance and device: the dynamic shared memory the kernel may
// use and its occupancy at that size (cached, so that steady-state calls make
// no attribute or occupancy queries).
struct LaunchCache {
    size_t smem = 0;
    int occ = 0;
};

template <int CW, int NC>
luce_status launch_glu(const GluArgs &a, cudaStream_t stream, int grid_cap)
{
    static LaunchCache cache[64];
    auto kern = k_glu_pair<CW, NC>;
    const size_t smem = (size_t)a.NS * 2 * a.S * a.rowbytes + (size_t)2 * a.NS * sizeof(uint64_t) +
                        (size_t)(a.E + 2) * sizeof(int) + (size_t)32 * HB_STRIDE * sizeof(float);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return LUCE_ERR_CUDA;
    LaunchCache &c = cache[dev];
    if (c.smem != smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return LUCE_ERR_CUDA;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (CW + 1) * 32, smem) != cudaSuccess ||
            occ < 1)
            return LUCE_ERR_CUDA;
        c.smem = smem;
        c.occ = occ;
    }
    const int grid = std::max(1, std::min(grid_cap, luce_host::sm_count() * c.occ));
    kern<<<grid, (CW + 1) * 32, smem, stream>>>(a);
    return luce_host::launch_status();
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
    a.ncu = NCU_MAX;
    // stage = S gate rows + S up rows, about 16-32 KB; ring of about 96 KB
    int S = 1;
    while (S < 32 && 2 * (2 * S) * a.rowbytes <= 36 * 1024)
        S *= 2;
    a.S = S;
    const int stage = 2 * S * a.rowbytes;
    a.NS = std::max(2, std::min(8, (96 * 1024) / stage));
    // an upper bound on the number of units, to size the grid
    const long long Tk = (long long)T * k;
    const long long nv_up = std::min<long long>(E, Tk) + Tk / NCU_MAX + (ws_gate ? (T + NCU_MAX - 1) / NCU_MAX : 0);
    const long long units = nv_up * (I / 32);
    const int cap = (int)std::min<long long>(units, INT_MAX);
    const int maxcols = std::min(T, NCU_MAX);
    cudaStream_t st = as_stream(stream);
    if (maxcols <= 1)
        return launch_glu<4, 1>(a, st, cap);
    if (maxcols <= 2)
        return launch_glu<4, 2>(a, st, cap);
    if (maxcols <= 4)
        return launch_glu<4, 4>(a, st, cap);
    return launch_glu<4, 8>(a, st, cap);
}
