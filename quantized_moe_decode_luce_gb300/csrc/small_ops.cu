// small_ops.cu -- router select + weights, q8_1 quantization, expert
// grouping and the argmax pair/pick, with their C-ABI entry points.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving" (section named at each use).
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

#include <cooperative_groups.h>

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_small_ops)

namespace {

using namespace luce;

// ---------------------------------------------------------------------------
// Router select + weights ([PR826], commit "fused DS4.1 decode kernels").
// One warp per token.  The E scores (logit + bias, one fp32 add) are staged in
// shared memory; k rounds of a warp arg-max pick the best untaken score,
// ties to the lower expert index (the (value, index) order is total, so the
// butterfly reduction gives every lane the same winner).  The weights are a
// softmax over the selected, unbiased logits.
constexpr int ROUTE_WARPS = 4;

__global__ void __launch_bounds__(ROUTE_WARPS * 32)
    k_route_topk(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k,
                 int32_t *__restrict__ ids, float *__restrict__ weights)
{
    extern __shared__ float s_scores[];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * ROUTE_WARPS + warp;
    if (t >= T)
        return;
    float *s = s_scores + warp * E;
    const float *l = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
        const float v = bias ? __fadd_rn(l[e], bias[e]) : l[e];
        s[e] = v == v ? v : -INFINITY; // a NaN score ranks below every number
    }
    __syncwarp();

    const int n_i = (E + 31) >> 5;
    uint32_t taken = 0;
    float sel0 = 0.0f, sel1 = 0.0f; // unbiased logit of slot lane and lane + 32
    for (int j = 0; j < k; j++) {
        float bv = 0.0f;
        int bi = INT_MAX;
        for (int i = 0; i < n_i; i++) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                const float v = s[e];
                if (bi == INT_MAX || v > bv) {
                    bv = v;
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        if (lane == 0)
            ids[(size_t)t * k + j] = bi;
        if (j == lane)
            sel0 = l[bi];
        else if (j == lane + 32)
            sel1 = l[bi];
    }
    route_softmax_warp(sel0, sel1, k, weights + (size_t)t * k, lane);
}

// ---------------------------------------------------------------------------
// q8_1 quantization ([PR826], commit "fused DS4.1 decode kernels": the q8_1
// activation memo).  One warp per 32-value block; a row of K values is K/32
// consecutive blocks, so the whole [T][K] input is one flat run of blocks.
constexpr int QUANT_WARPS = 8;

__global__ void __launch_bounds__(QUANT_WARPS * 32)
    k_quantize_q8_1(const float *__restrict__ x, int64_t n_blocks, uint32_t *__restrict__ out)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t b = (int64_t)blockIdx.x * QUANT_WARPS + (threadIdx.x >> 5);
    if (b >= n_blocks)
        return;
    const float v = x[b * QK + lane];
    quantize_q8_1_warp(v, out + b * Q8_1_WORDS, lane);
}

// ---------------------------------------------------------------------------
// Expert grouping ([PR826], commit "fused DS4.1 decode kernels").  One CTA.
// Warp w owns a contiguous segment of routes and counts it into its own
// histogram row; the exclusive scan of the totals gives the offsets, and a
// per-(warp, expert) running base makes the scatter stable in r: within a
// 32-route chunk, lanes with the same expert take consecutive slots in lane
// order (match + popcount), then the group's last lane advances the base.
constexpr int GROUP_THREADS = 1024;

// The grouping by one CTA of GROUP_THREADS threads.  ids_src may be global or
// shared memory; hist [nw*E] and excl [E+1] are shared scratch.
__device__ void group_body(const int32_t *ids_src, int R, int E, int nw, int *hist, int *excl,
                           int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ routes)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < nw * E; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();
    const int seg = (R + nw - 1) / nw;
    const int r0 = warp * seg, r1 = min(R, r0 + seg);
    if (warp < nw) {
        for (int r = r0 + lane; r < r1; r += 32) {
            const int e = ids_src[r];
            if (e >= 0 && e < E)
                atomicAdd(&hist[warp * E + e], 1);
            else if (e >= E)
                atomicOr(&g_fault_word, LUCE_FAULT_BAD_ID);
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < nw; w++)
            c += hist[w * E + e];
        excl[e] = c;
        counts[e] = c;
    }
    __syncthreads();
    if (warp == 0) { // exclusive scan of the counts, 32 at a time
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? excl[e] : 0;
            int inc = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o)
                    inc += v;
            }
            if (e < E)
                excl[e] = carry + inc - c;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0)
            excl[E] = carry;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += blockDim.x)
        offsets[e] = excl[e];
    for (int e = tid; e < E; e += blockDim.x) {
        int run = excl[e];
        for (int w = 0; w < nw; w++) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    if (warp < nw) {
        const unsigned lt = (1u << lane) - 1u;
        for (int base = r0; base < r1; base += 32) {
            const int r = base + lane;
            const int e = r < r1 ? ids_src[r] : -1;
            const bool ok = e >= 0 && e < E;
            const unsigned m = __match_any_sync(0xffffffffu, ok ? e : -1);
            int pos = 0;
            if (ok)
                pos = hist[warp * E + e] + __popc(m & lt);
            __syncwarp();
            if (ok) {
                routes[pos] = r;
                if (lane == 31 - __clz(m))
                    hist[warp * E + e] += __popc(m);
            }
            __syncwarp();
        }
    }
    const int total = excl[E];
    for (int r = total + tid; r < R; r += blockDim.x)
        routes[r] = -1;
}

__global__ void __launch_bounds__(GROUP_THREADS)
    k_moe_group(const int32_t *__restrict__ ids, int R, int E, int nw, int32_t *__restrict__ counts,
                int32_t *__restrict__ offsets, int32_t *__restrict__ routes)
{
    extern __shared__ int s_mem[];
    pdl_wait();
    pdl_trigger();
    group_body(ids, R, E, nw, s_mem, s_mem + nw * E, counts, offsets, routes);
}

// ---------------------------------------------------------------------------
// Fused prep: router select + weights, q8_1 quantization of the FFN input
// and expert grouping in ONE launch of one CTA ([PR826], commit "fused DS4.1
// decode kernels": the router's select and weights in one launch, one
// expert grouping per layer, the q8_1 activation memo).  For T <= 32 tokens
// and E <= 256 experts: warp t routes token t with its scores in registers
// (EPL per lane), all 32 warps then quantize the T*H/32 blocks, and after a
// CTA barrier the same CTA groups the routes from shared memory.
struct PrepArgs {
    const float *logits, *bias, *x;
    int T, E, k, H;
    int32_t *ids;
    float *weights;
    uint32_t *xq;
    int32_t *counts, *offsets, *routes;
};

template <int EPL>
__device__ __forceinline__ void route_token_regs(const float *__restrict__ l, const float *__restrict__ bias, int E,
                                                 int k, int32_t *ids_s, int32_t *ids_g, float *w_g, int lane)
{
    float sc[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float v = bias ? __fadd_rn(l[e], bias[e]) : l[e];
            sc[i] = v == v ? v : -INFINITY; // a NaN score ranks below every number
        } else {
            sc[i] = 0.0f;
            taken |= 1u << i;
        }
    }
    float sel0 = 0.0f, sel1 = 0.0f;
    for (int j = 0; j < k; j++) {
        float bv = 0.0f;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            if (!((taken >> i) & 1u) && (bi == INT_MAX || sc[i] > bv)) {
                bv = sc[i];
                bi = lane + 32 * i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        if (lane == 0) {
            ids_s[j] = bi;
            ids_g[j] = bi;
        }
        if (j == lane)
            sel0 = l[bi];
        else if (j == lane + 32)
            sel1 = l[bi];
    }
    route_softmax_warp(sel0, sel1, k, w_g, lane);
}

template <int EPL>
__global__ void __launch_bounds__(GROUP_THREADS) k_moe_prep(const PrepArgs a)
{
    extern __shared__ int s_mem[];
    int *ids_s = s_mem;                  // [T*k]
    int *hist = ids_s + a.T * a.k;       // [32*E]
    int *excl = hist + 32 * a.E;         // [E+1]
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < a.T) {
        const size_t o = (size_t)warp * a.k;
        route_token_regs<EPL>(a.logits + (size_t)warp * a.E, a.bias, a.E, a.k, ids_s + o, a.ids + o,
                              a.weights + o, lane);
    }
    const int nbl = a.T * (a.H / QK);
    for (int b = warp; b < nbl; b += 32)
        quantize_q8_1_warp(a.x[(size_t)b * QK + lane], a.xq + (size_t)b * Q8_1_WORDS, lane);
    __syncthreads();
    group_body(ids_s, a.T * a.k, a.E, 32, hist, excl, a.counts, a.offsets, a.routes);
}

// Small prep: T <= 8 tokens, T*k <= 64 routes, E <= 256 experts (decode and
// verify).  512 threads: warp t routes token t while the other warps share
// the quantization of the input blocks; after one CTA barrier, warp 0 alone groups
// the routes with shuffles (no further CTA barrier): lane l counts experts
// l, l+32, ..., a warp scan gives the offsets, and route r's slot is its
// expert's offset plus the number of earlier routes of that expert.
constexpr int PREP_SMALL_THREADS = 512;
constexpr int PREP_SMALL_MAX_T = 8;
constexpr int PREP_SMALL_MAX_R = 64;

template <int EPL>
__global__ void __launch_bounds__(PREP_SMALL_THREADS) k_moe_prep_small(const PrepArgs a)
{
    __shared__ int ids_s[PREP_SMALL_MAX_R];
    __shared__ int s_off[256];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = PREP_SMALL_THREADS / 32;
    if (warp < a.T) {
        const size_t o = (size_t)warp * a.k;
        route_token_regs<EPL>(a.logits + (size_t)warp * a.E, a.bias, a.E, a.k, ids_s + o, a.ids + o,
                              a.weights + o, lane);
    }
    // the routing warps do not quantize: the other warps share the blocks
    const int nbl = a.T * (a.H / QK);
    if (warp >= a.T)
        for (int b = warp - a.T; b < nbl; b += nwarps - a.T)
            quantize_q8_1_warp(a.x[(size_t)b * QK + lane], a.xq + (size_t)b * Q8_1_WORDS, lane);
    __syncthreads();
    if (warp != 0)
        return;
    const int R = a.T * a.k;
    // counts of experts lane + 32 i, then an exclusive scan in expert order
    int cnt[EPL];
#pragma unroll
    for (int i = 0; i < EPL; i++)
        cnt[i] = 0;
    for (int r = 0; r < R; r++) {
        const int e = ids_s[r];
#pragma unroll
        for (int i = 0; i < EPL; i++)
            cnt[i] += (e == lane + 32 * i) ? 1 : 0;
    }
    int carry = 0;
    int off[EPL];
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        int inc = cnt[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o)
                inc += v;
        }
        off[i] = carry + inc - cnt[i];
        carry += __shfl_sync(0xffffffffu, inc, 31);
        const int e = lane + 32 * i;
        if (e < a.E) {
            a.counts[e] = cnt[i];
            a.offsets[e] = off[i];
            s_off[e] = off[i];
        }
    }
    if (lane == 0)
        a.offsets[a.E] = carry;
    __syncwarp();
    // route r goes to its expert's offset plus the earlier routes of that expert
    for (int r = lane; r < R; r += 32) {
        const int e = ids_s[r];
        if (e < 0 || e >= a.E)
            continue;
        int before = 0;
        for (int q = 0; q < r; q++)
            before += (ids_s[q] == e) ? 1 : 0;
        a.routes[s_off[e] + before] = r;
    }
    for (int r = carry + lane; r < R; r += 32)
        a.routes[r] = -1;
}

// ---------------------------------------------------------------------------
// Argmax pair/pick ([PR826], commit "fused DS4.1 decode kernels").  CTA
// (c, r) reduces chunk c of row r to a (value, index) pair; the CTA that
// arrives last on the row's counter picks among the C pairs and resets the
// counter.  The (greater value, then lower index) order is total, so the
// result does not depend on which CTA finishes last.
constexpr int ARGMAX_THREADS = 256;

struct ArgPair {
    float v;
    int i;
};

__device__ __forceinline__ void better(float &bv, int &bi, float ov, int oi)
{
    if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
    }
}

__device__ __forceinline__ void block_argmax(float &bv, int &bi)
{
    __shared__ float sv[ARGMAX_THREADS / 32];
    __shared__ int si[ARGMAX_THREADS / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, ov, oi);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sv[warp] = bv;
        si[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        bv = lane < ARGMAX_THREADS / 32 ? sv[lane] : 0.0f;
        bi = lane < ARGMAX_THREADS / 32 ? si[lane] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            better(bv, bi, ov, oi);
        }
    }
}

__global__ void __launch_bounds__(ARGMAX_THREADS)
    k_argmax(const float *__restrict__ logits, int64_t V, int64_t L, int C, bool vec4, ArgPair *__restrict__ pairs,
             unsigned int *__restrict__ counters, int32_t *__restrict__ idx, float *__restrict__ val, int64_t v0)
{
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x, r = blockIdx.y;
    const int64_t lo = (int64_t)c * L, hi = min(V, lo + L);
    const float *row = logits + (int64_t)r * V;
    float bv = 0.0f;
    int bi = INT_MAX;
    if (vec4) {
        const float4 *p = reinterpret_cast<const float4 *>(row + lo);
        const int64_t n4 = (hi - lo) >> 2;
        for (int64_t i = threadIdx.x; i < n4; i += ARGMAX_THREADS) {
            const float4 q = __ldcs(p + i);
            const int base = (int)(lo + 4 * i);
            better(bv, bi, q.x, base);
            better(bv, bi, q.y, base + 1);
            better(bv, bi, q.z, base + 2);
            better(bv, bi, q.w, base + 3);
        }
        for (int64_t i = lo + 4 * n4 + threadIdx.x; i < hi; i += ARGMAX_THREADS)
            better(bv, bi, row[i], (int)i);
    } else {
        for (int64_t i = lo + threadIdx.x; i < hi; i += ARGMAX_THREADS)
            better(bv, bi, __ldcs(row + i), (int)i);
    }
    block_argmax(bv, bi);
    __shared__ bool s_last;
    if (threadIdx.x == 0) {
        pairs[(size_t)r * C + c] = ArgPair{bv, bi};
        __threadfence();
        const unsigned ticket = atomicAdd(&counters[r], 1u);
        s_last = (ticket == (unsigned)(C - 1));
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    bv = 0.0f;
    bi = INT_MAX;
    for (int i = threadIdx.x; i < C; i += ARGMAX_THREADS) {
        const float ov = __ldcg(&pairs[(size_t)r * C + i].v);
        const int oi = __ldcg(&pairs[(size_t)r * C + i].i);
        better(bv, bi, ov, oi);
    }
    block_argmax(bv, bi);
    if (threadIdx.x == 0) {
        idx[r] = (int32_t)(bi + v0); // the shard's first column is column v0 of the vocabulary
        if (val)
            val[r] = bv;
        counters[r] = 0u;
    }
}

// Chunking of an argmax row: a pure function of (R, V), so the workspace size
// does not depend on the device.
// Rows of at least ARGMAX_CLUSTER_MIN values: one cluster of AC = 16 CTAs
// per row (a non-portable cluster size, allowed per device), each CTA an
// equal slice of it (all its loads in flight: ~8 float4 a thread at V =
// 129,280), the CTAs' pairs joined through distributed shared memory by rank
// 0; no second pass through global memory and no atomics.  Measured 1.3 us
// faster than the two-pass kernel at 5 x 129,280 (8-CTA clusters: 0.2 us).
constexpr int AC = 16;
constexpr int64_t ARGMAX_CLUSTER_MIN = 8 * 2048;

__global__ void __cluster_dims__(AC, 1, 1) __launch_bounds__(ARGMAX_THREADS)
    k_argmax_cluster(const float *__restrict__ logits, int64_t V, int64_t L, bool vec4, int32_t *__restrict__ idx,
                     float *__restrict__ val, int64_t v0)
{
    namespace cg = cooperative_groups;
    pdl_wait();
    pdl_trigger();
    cg::cluster_group cl = cg::this_cluster();
    const int c = (int)cl.block_rank(), r = blockIdx.y;
    const int64_t lo = (int64_t)c * L, hi = min(V, lo + L);
    const float *row = logits + (int64_t)r * V;
    float bv = 0.0f;
    int bi = INT_MAX;
    if (lo < hi) {
        if (vec4) {
            const float4 *p = reinterpret_cast<const float4 *>(row + lo);
            const int n4 = (int)((hi - lo) >> 2);
            // every load of the slice in flight before the first comparison
            constexpr int U = 8;
            for (int i0 = threadIdx.x; i0 < n4; i0 += U * ARGMAX_THREADS) {
                float4 q[U];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const int i = i0 + u * ARGMAX_THREADS;
                    q[u] = i < n4 ? __ldcs(p + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const int i = i0 + u * ARGMAX_THREADS;
                    if (i < n4) {
                        const int base = (int)(lo + 4 * (int64_t)i);
                        better(bv, bi, q[u].x, base);
                        better(bv, bi, q[u].y, base + 1);
                        better(bv, bi, q[u].z, base + 2);
                        better(bv, bi, q[u].w, base + 3);
                    }
                }
            }
            for (int64_t i = lo + 4 * (int64_t)n4 + threadIdx.x; i < hi; i += ARGMAX_THREADS)
                better(bv, bi, row[i], (int)i);
        } else {
#pragma unroll 4
            for (int64_t i = lo + threadIdx.x; i < hi; i += ARGMAX_THREADS)
                better(bv, bi, __ldcs(row + i), (int)i);
        }
    }
    block_argmax(bv, bi);
    __shared__ float s_v;
    __shared__ int s_i;
    if (threadIdx.x == 0) {
        s_v = bv;
        s_i = bi;
    }
    cl.sync(); // every CTA's pair is in its shared memory
    if (c == 0 && threadIdx.x < 32) {
        float ov = 0.0f;
        int oi = INT_MAX;
        if (threadIdx.x < AC) {
            ov = *cl.map_shared_rank(&s_v, (unsigned)threadIdx.x);
            oi = *cl.map_shared_rank(&s_i, (unsigned)threadIdx.x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float pv = __shfl_xor_sync(0xffffffffu, ov, o);
            const int pi = __shfl_xor_sync(0xffffffffu, oi, o);
            better(ov, oi, pv, pi);
        }
        if (threadIdx.x == 0) {
            idx[r] = (int32_t)(oi + v0); // the shard's first column is column v0 of the vocabulary
            if (val)
                val[r] = ov;
        }
    }
    cl.sync(); // rank 0 has read every CTA's pair before any CTA exits
}

// Whether 16-CTA clusters are allowed for k_argmax_cluster on this device
// (the attribute is set once per device; a refusal or a failed launch turns
// the path off for the device).
std::atomic<int> g_argmax_cluster[64];
bool argmax_cluster_ok()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return false;
    }
    int st = g_argmax_cluster[dev].load(std::memory_order_acquire);
    if (st == 0) {
        st = cudaFuncSetAttribute(k_argmax_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess
                 ? 1
                 : -1;
        if (st < 0)
            (void)cudaGetLastError();
        g_argmax_cluster[dev].store(st, std::memory_order_release);
    }
    return st > 0;
}
void argmax_cluster_off()
{
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64)
        g_argmax_cluster[dev].store(-1, std::memory_order_release);
}

void argmax_chunks(int R, int64_t V, int64_t &L, int &C)
{
    const int64_t want = R > 0 ? std::max<int64_t>(1, 320 / R) : 1;
    L = std::max<int64_t>(2048, (V + want - 1) / want);
    L = (L + 3) & ~int64_t(3);
    C = (int)((V + L - 1) / L);
}

size_t argmax_pairs_bytes(int R, int C) { return ((size_t)R * C * sizeof(ArgPair) + 15) & ~size_t(15); }

} // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_glu(unsigned int *bits);
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_down(unsigned int *bits);
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_layer(unsigned int *bits);
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_layer_flat(unsigned int *bits);
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_tc(unsigned int *bits);
extern "C" __attribute__((visibility("hidden"))) cudaError_t luce_internal_fault_q4k(unsigned int *bits);

namespace luce_host {
Tuning g_tuning;
static int g_pdl = 0;
bool pdl_enabled() { return __atomic_load_n(&g_pdl, __ATOMIC_RELAXED) != 0; }

int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            return 148;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}
} // namespace luce_host

using namespace luce_host;

extern "C" const char *luce_status_string(luce_status s)
{
    switch (s) {
    case LUCE_OK:
        return "ok";
    case LUCE_ERR_INVALID_ARG:
        return "invalid argument";
    case LUCE_ERR_UNSUPPORTED:
        return "unsupported shape";
    case LUCE_ERR_CUDA:
        return "CUDA error";
    }
    return "unknown status";
}

extern "C" int luce_version(void) { return 300; }

extern "C" luce_status luce_set_pdl(int enable)
{
    __atomic_store_n(&luce_host::g_pdl, enable ? 1 : 0, __ATOMIC_RELAXED);
    return LUCE_OK;
}

extern "C" luce_status luce_get_fault(unsigned int *bits)
{
    if (!bits)
        return LUCE_ERR_INVALID_ARG;
    *bits = 0;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return LUCE_ERR_CUDA;
    cudaError_t e1 = luce_internal_fault_small_ops(bits);
    cudaError_t e2 = luce_internal_fault_glu(bits);
    cudaError_t e3 = luce_internal_fault_down(bits);
    cudaError_t e4 = luce_internal_fault_layer(bits);
    cudaError_t e5 = luce_internal_fault_q4k(bits);
    cudaError_t e6 = luce_internal_fault_layer_flat(bits);
    cudaError_t e7 = luce_internal_fault_tc(bits);
    return (e1 == cudaSuccess && e2 == cudaSuccess && e3 == cudaSuccess && e4 == cudaSuccess && e5 == cudaSuccess &&
            e6 == cudaSuccess && e7 == cudaSuccess)
               ? LUCE_OK
               : LUCE_ERR_CUDA;
}

extern "C" luce_status luce_route_topk(const float *logits, const float *bias, int T, int E, int k, int32_t *ids,
                                       float *weights, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 64)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!logits || !ids || !weights || !aligned(logits, 4) || !aligned(ids, 4) || !aligned(weights, 4) ||
        (bias && !aligned(bias, 4)))
        return LUCE_ERR_INVALID_ARG;
    const int blocks = (T + ROUTE_WARPS - 1) / ROUTE_WARPS;
    const size_t smem = (size_t)ROUTE_WARPS * E * sizeof(float);
    return launch(k_route_topk, dim3(blocks), dim3(ROUTE_WARPS * 32), smem, as_stream(stream), logits, bias, T, E,
                  k, ids, weights);
}

extern "C" luce_status luce_quantize_q8_1(const float *x, int T, int K, luce_block_q8_1 *xq, void *stream)
{
    if (T < 0 || K <= 0 || K % QK != 0)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!x || !xq || !aligned(x, 4) || !aligned(xq, 4))
        return LUCE_ERR_INVALID_ARG;
    const int64_t nb = (int64_t)T * (K / QK);
    const int64_t blocks = (nb + QUANT_WARPS - 1) / QUANT_WARPS;
    if (blocks > INT_MAX)
        return LUCE_ERR_INVALID_ARG;
    return launch(k_quantize_q8_1, dim3((unsigned)blocks), dim3(QUANT_WARPS * 32), 0, as_stream(stream), x, nb,
                  reinterpret_cast<uint32_t *>(xq));
}

extern "C" luce_status luce_moe_group(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                                      int32_t *routes, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > 64 || (int64_t)T * k > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4))
        return LUCE_ERR_INVALID_ARG;
    if (T > 0 && (!ids || !routes || !aligned(ids, 4) || !aligned(routes, 4)))
        return LUCE_ERR_INVALID_ARG;
    const int R = T * k;
    const int nw = std::max(1, std::min(32, 8192 / E));
    const size_t smem = ((size_t)nw * E + E + 1) * sizeof(int);
    return launch(k_moe_group, dim3(1), dim3(GROUP_THREADS), smem, as_stream(stream), ids, R, E, nw, counts, offsets,
                  routes);
}

extern "C" size_t luce_argmax_workspace_bytes(int R, int64_t V)
{
    if (R <= 0 || V <= 0)
        return 0;
    int64_t L;
    int C;
    argmax_chunks(R, V, L, C);
    return argmax_pairs_bytes(R, C) + (((size_t)R * sizeof(unsigned int) + 15) & ~size_t(15));
}

extern "C" luce_status luce_argmax(const float *logits, int R, int64_t V, int32_t *idx, float *val,
                                   void *workspace, size_t workspace_bytes, void *stream)
{
    if (R < 0 || V < 1 || V >= ((int64_t)1 << 31) || R > 65535)
        return LUCE_ERR_INVALID_ARG;
    if (R == 0)
        return LUCE_OK;
    if (!logits || !idx || !workspace || !aligned(logits, 4) || !aligned(idx, 4) || !aligned(workspace, 8) ||
        (val && !aligned(val, 4)))
        return LUCE_ERR_INVALID_ARG;
    if (workspace_bytes < luce_argmax_workspace_bytes(R, V))
        return LUCE_ERR_INVALID_ARG;
    int64_t L;
    int C;
    argmax_chunks(R, V, L, C);
    ArgPair *pairs = reinterpret_cast<ArgPair *>(workspace);
    unsigned int *counters =
        reinterpret_cast<unsigned int *>(reinterpret_cast<uint8_t *>(workspace) + argmax_pairs_bytes(R, C));
    const bool vec4 = (V % 4 == 0) && aligned(logits, 16);
    if (V >= ARGMAX_CLUSTER_MIN && argmax_cluster_ok()) {
        // (the workspace is not used on this path; the two-pass kernel below
        // remains for short rows and for a device without 16-CTA clusters)
        const int64_t Lc = (((V + AC - 1) / AC) + 3) & ~int64_t(3);
        if (launch(k_argmax_cluster, dim3((unsigned)AC, (unsigned)R), dim3(ARGMAX_THREADS), 0, as_stream(stream),
                   logits, V, Lc, vec4, idx, val, (int64_t)0) == LUCE_OK)
            return LUCE_OK;
        argmax_cluster_off();
    }
    dim3 grid((unsigned)C, (unsigned)R);
    return launch(k_argmax, grid, dim3(ARGMAX_THREADS), 0, as_stream(stream), logits, V, L, C, vec4, pairs, counters,
                  idx, val, (int64_t)0);
}

extern "C" luce_status luce_argmax_shard(const float *logits, int R, int64_t Vs, int64_t v0, int32_t *idx, float *val,
                                         void *workspace, size_t workspace_bytes, void *stream)
{
    if (R < 0 || Vs < 1 || v0 < 0 || v0 + Vs > ((int64_t)1 << 31) - 1 || R > 65535)
        return LUCE_ERR_INVALID_ARG;
    if (R == 0)
        return LUCE_OK;
    if (!logits || !idx || !workspace || !aligned(logits, 4) || !aligned(idx, 4) || !aligned(workspace, 8) ||
        (val && !aligned(val, 4)))
        return LUCE_ERR_INVALID_ARG;
    if (workspace_bytes < luce_argmax_workspace_bytes(R, Vs))
        return LUCE_ERR_INVALID_ARG;
    int64_t L;
    int C;
    argmax_chunks(R, Vs, L, C);
    ArgPair *pairs = reinterpret_cast<ArgPair *>(workspace);
    unsigned int *counters =
        reinterpret_cast<unsigned int *>(reinterpret_cast<uint8_t *>(workspace) + argmax_pairs_bytes(R, C));
    const bool vec4 = (Vs % 4 == 0) && aligned(logits, 16);
    if (Vs >= ARGMAX_CLUSTER_MIN && argmax_cluster_ok()) {
        const int64_t Lc = (((Vs + AC - 1) / AC) + 3) & ~int64_t(3);
        if (launch(k_argmax_cluster, dim3((unsigned)AC, (unsigned)R), dim3(ARGMAX_THREADS), 0, as_stream(stream),
                   logits, Vs, Lc, vec4, idx, val, v0) == LUCE_OK)
            return LUCE_OK;
        argmax_cluster_off();
    }
    dim3 grid((unsigned)C, (unsigned)R);
    return launch(k_argmax, grid, dim3(ARGMAX_THREADS), 0, as_stream(stream), logits, Vs, L, C, vec4, pairs, counters,
                  idx, val, v0);
}

extern "C" luce_status luce_moe_prep(const float *logits, const float *bias, const float *x, int T, int E, int k, int H,
                                     int32_t *ids, float *weights, luce_block_q8_1 *xq, int32_t *counts,
                                     int32_t *offsets, int32_t *routes, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 64 || H <= 0 || H % QK != 0 ||
        (int64_t)T * k > (1 << 20))
        return LUCE_ERR_INVALID_ARG;
    if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4))
        return LUCE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !x || !ids || !weights || !xq || !routes || !aligned(logits, 4) || !aligned(x, 4) ||
                  !aligned(ids, 4) || !aligned(weights, 4) || !aligned(xq, 4) || !aligned(routes, 4) ||
                  (bias && !aligned(bias, 4))))
        return LUCE_ERR_INVALID_ARG;
    if (T == 0 || T > 32 || E > 256) {
        // the general path: three launches
        luce_status st = luce_route_topk(logits, bias, T, E, k, ids, weights, stream);
        if (st == LUCE_OK)
            st = luce_quantize_q8_1(x, T, H, xq, stream);
        if (st == LUCE_OK)
            st = luce_moe_group(ids, T, k, E, counts, offsets, routes, stream);
        return st;
    }
    PrepArgs a{logits, bias, x, T, E, k, H, ids, weights, reinterpret_cast<uint32_t *>(xq), counts, offsets, routes};
    const size_t smem = ((size_t)T * k + 32 * (size_t)E + E + 1) * sizeof(int);
    const int epl = (E + 31) / 32;
    cudaStream_t st = as_stream(stream);
    if (T <= PREP_SMALL_MAX_T && T * k <= PREP_SMALL_MAX_R) {
        const dim3 g1(1), b1(PREP_SMALL_THREADS);
        if (epl <= 1)
            return launch(k_moe_prep_small<1>, g1, b1, 0, st, a);
        if (epl <= 2)
            return launch(k_moe_prep_small<2>, g1, b1, 0, st, a);
        if (epl <= 4)
            return launch(k_moe_prep_small<4>, g1, b1, 0, st, a);
        return launch(k_moe_prep_small<8>, g1, b1, 0, st, a);
    }
    if (epl <= 1)
        return launch(k_moe_prep<1>, dim3(1), dim3(GROUP_THREADS), smem, st, a);
    if (epl <= 2)
        return launch(k_moe_prep<2>, dim3(1), dim3(GROUP_THREADS), smem, st, a);
    if (epl <= 4)
        return launch(k_moe_prep<4>, dim3(1), dim3(GROUP_THREADS), smem, st, a);
    return launch(k_moe_prep<8>, dim3(1), dim3(GROUP_THREADS), smem, st, a);
}

// ===========================================================================
// luce_argmax_noalloc: the argmax pair/pick with library-owned scratch.
//
// Some callers cannot allocate device memory at all: a host application that
// owns every device allocation and gives this library none, or a loop that
// must never call into the CUDA allocator.  They cannot provide the
// workspace luce_argmax needs, so this entry point keeps its scratch (the
// per-chunk pairs and the per-row counters) in a fixed array of device memory
// that the library holds from load to exit on every GPU that loads it.
// ===========================================================================
namespace {
constexpr size_t kNoallocScratchBytes = 16384; // the fixed maximum
constexpr int kNoallocMaxRows = 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];
} // namespace

extern "C" luce_status luce_argmax_noalloc(const float *logits, int R, int64_t V, int32_t *idx, float *val,
                                           void *stream)
{
    if (R < 0 || V < 1 || V >= ((int64_t)1 << 31))
        return LUCE_ERR_INVALID_ARG;
    if (R == 0)
        return LUCE_OK;
    if (!logits || !idx || !aligned(logits, 4) || !aligned(idx, 4) || (val && !aligned(val, 4)))
        return LUCE_ERR_INVALID_ARG;
    const size_t need = luce_argmax_workspace_bytes(R, V);
    if (R > kNoallocMaxRows || need > kNoallocScratchBytes)
        return LUCE_ERR_UNSUPPORTED; // beyond the fixed scratch: use luce_argmax with a workspace
    // the array's device address in the current context, looked up on every
    // call (in host code its name is only a stand-in, and a cached address
    // would outlive a reset context or belong to another device)
    void *base = nullptr;
    if (cudaGetSymbolAddress(&base, g_noalloc_scratch) != cudaSuccess || base == nullptr) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    int64_t L;
    int C;
    argmax_chunks(R, V, L, C);
    ArgPair *pairs = reinterpret_cast<ArgPair *>(base);
    unsigned int *counters =
        reinterpret_cast<unsigned int *>(reinterpret_cast<uint8_t *>(base) + argmax_pairs_bytes(R, C));
    // the row counters must start at zero whatever an earlier call left
    if (cudaMemsetAsync(counters, 0, (size_t)R * sizeof(unsigned int), as_stream(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    const bool vec4 = (V % 4 == 0) && aligned(logits, 16);
    dim3 grid((unsigned)C, (unsigned)R);
    return launch(k_argmax, grid, dim3(ARGMAX_THREADS), 0, as_stream(stream), logits, V, L, C, vec4, pairs, counters,
                  idx, val, (int64_t)0);
}
