// edge_ops.cu -- the steps either side of the routed-MoE FFN: the RMS norm
// and the router logits before it, the pick of a vocabulary split across
// ranks after it, and the two pieces of an expert-parallel split (masking the
// routes a rank does not own, summing the ranks' partial outputs), with their
// C-ABI entry points.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving" (section named at each use).
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

namespace {

using namespace luce;


// ---------------------------------------------------------------------------
// RMS norm + router logits ([PR826], commit "fused DS4.1 decode kernels": the
// RMS norm among the launches it fuses; the HC pre-mix commit: an RMS norm
// whose sum of squares and products run in F32).  The standard RMS norm,
// xn_i = x_i * r * gamma_i with r = 1 / sqrt(mean_i x_i^2 + eps), and the
// router logits logits[t][e] = sum_i W_r[e][i] xn_i with W_r in F32.
//
// Grid (E / RW experts, T / tpc token tiles), RW warps: every CTA normalizes
// its tile's tokens into shared memory (warp t sums token t's squares), then
// warp w streams router row e = blockIdx.x RW + w once for all the tile's
// tokens.  CTAs of the first expert chunk also store xn.
//
// With a residual r the normed row is that of x + r (one fp32 add per value,
// the sum stored by the first expert chunk): the residual add before the norm
// in the same launch.
//
// ROW (one token, H <= 4 x 32 x WP, gamma 16-byte aligned): every warp holds
// the whole row in registers instead -- its lane's slice of x, of gamma
// (requested before the programmatic-launch wait, like the router row) and of
// its router row -- and sums the squares itself, so the token's path after
// the wait has no shared memory and no block barrier.  The lane slices, the
// order of every sum and every rounding are the tiled path's, so both give
// the same bits.
constexpr int RW = 8;   // warps (router rows) per CTA
constexpr int TPC = 8;  // most tokens per tile
constexpr int WP = 16;  // router-row float4 per lane requested before the wait
// warps (router rows) per CTA on the register path: its threads hold ~200
// registers, and small CTAs leave room on their SMs for the next kernel's
// CTAs (the one-launch layer, whose CTAs must all be resident) to be placed
// while the router runs
constexpr int RW_ROW = 2;

template <bool ROW>
__global__ void __launch_bounds__(RW * 32)
    k_rmsnorm_router(const float *__restrict__ x, const float *__restrict__ res, float *__restrict__ xsum,
                     const float *__restrict__ gamma, float eps, const float *__restrict__ w_router, int T, int E,
                     int H, int tpc, float *__restrict__ xn, float *__restrict__ logits)
{
    extern __shared__ __align__(16) float xs[]; // [tpc][H] normed rows
    __shared__ float rs[TPC];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * tpc, nt = min(tpc, T - t0);
    const int H4 = H >> 2;
    const int e = blockIdx.x * (ROW ? RW_ROW : RW) + warp;
    const float4 *wr = reinterpret_cast<const float4 *>(w_router + (size_t)min(e, E - 1) * H);
    const float4 zero4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // the router row does not depend on the previous kernel: its first
    // WP float4 per lane are requested before waiting for that kernel
    float4 wpre[WP];
#pragma unroll
    for (int u = 0; u < WP; u++) {
        const int i = lane + 32 * u;
        wpre[u] = (e < E && i < H4) ? __ldg(wr + i) : zero4;
    }
    if constexpr (ROW) {
        float4 gv[WP], xv[WP];
#pragma unroll
        for (int u = 0; u < WP; u++) {
            const int i = lane + 32 * u;
            gv[u] = i < H4 ? __ldg(reinterpret_cast<const float4 *>(gamma) + i) : zero4;
        }
        pdl_wait();
        pdl_trigger();
        const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)t0 * H);
#pragma unroll
        for (int u = 0; u < WP; u++) {
            const int i = lane + 32 * u;
            xv[u] = i < H4 ? xr[i] : zero4;
        }
        if (res != nullptr) {
            const float4 *rr = reinterpret_cast<const float4 *>(res + (size_t)t0 * H);
            float4 rv[WP];
#pragma unroll
            for (int u = 0; u < WP; u++) {
                const int i = lane + 32 * u;
                rv[u] = i < H4 ? rr[i] : zero4;
            }
#pragma unroll
            for (int u = 0; u < WP; u++) {
                xv[u].x = __fadd_rn(xv[u].x, rv[u].x);
                xv[u].y = __fadd_rn(xv[u].y, rv[u].y);
                xv[u].z = __fadd_rn(xv[u].z, rv[u].z);
                xv[u].w = __fadd_rn(xv[u].w, rv[u].w);
            }
            if (xsum != nullptr && blockIdx.x == 0 && warp == 1) {
                float4 *so = reinterpret_cast<float4 *>(xsum + (size_t)t0 * H);
#pragma unroll
                for (int u = 0; u < WP; u++)
                    if (lane + 32 * u < H4)
                        so[lane + 32 * u] = xv[u];
            }
        }
        float ss = 0.0f;
#pragma unroll
        for (int u = 0; u < WP; u++) {
            if (lane + 32 * u < H4) {
                ss = fmaf(xv[u].x, xv[u].x, ss);
                ss = fmaf(xv[u].y, xv[u].y, ss);
                ss = fmaf(xv[u].z, xv[u].z, ss);
                ss = fmaf(xv[u].w, xv[u].w, ss);
            }
        }
        ss = warp_sum(ss);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
        const bool store = xn != nullptr && blockIdx.x == 0 && warp == 0;
        float4 *xo = reinterpret_cast<float4 *>(xn + (size_t)t0 * H);
        float acc = 0.0f;
#pragma unroll
        for (int u = 0; u < WP; u++) {
            const int i = lane + 32 * u;
            if (i < H4) {
                float4 v;
                v.x = __fmul_rn(__fmul_rn(xv[u].x, r), gv[u].x);
                v.y = __fmul_rn(__fmul_rn(xv[u].y, r), gv[u].y);
                v.z = __fmul_rn(__fmul_rn(xv[u].z, r), gv[u].z);
                v.w = __fmul_rn(__fmul_rn(xv[u].w, r), gv[u].w);
                if (store)
                    xo[i] = v;
                acc = fmaf(wpre[u].x, v.x, acc);
                acc = fmaf(wpre[u].y, v.y, acc);
                acc = fmaf(wpre[u].z, v.z, acc);
                acc = fmaf(wpre[u].w, v.w, acc);
            }
        }
        acc = warp_sum(acc);
        if (e < E && lane == 0)
            logits[(size_t)t0 * E + e] = acc;
        return;
    }
    pdl_wait();
    pdl_trigger();
    if (warp < nt) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)(t0 + warp) * H);
        const float4 *rr = res ? reinterpret_cast<const float4 *>(res + (size_t)(t0 + warp) * H) : nullptr;
        float ss = 0.0f;
#pragma unroll 8
        for (int i = lane; i < H4; i += 32) {
            float4 v = xr[i];
            if (rr != nullptr) {
                const float4 q = rr[i];
                v.x = __fadd_rn(v.x, q.x);
                v.y = __fadd_rn(v.y, q.y);
                v.z = __fadd_rn(v.z, q.z);
                v.w = __fadd_rn(v.w, q.w);
            }
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0)
            rs[warp] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
    }
    __syncthreads();
    const bool store = xn != nullptr && blockIdx.x == 0;
    const bool store_sum = res != nullptr && xsum != nullptr && blockIdx.x == 0;
    for (int j = threadIdx.x; j < nt * H; j += RW * 32) {
        const int t = j / H, i = j - t * H;
        float xi = x[(size_t)(t0 + t) * H + i];
        if (res != nullptr) {
            xi = __fadd_rn(xi, res[(size_t)(t0 + t) * H + i]);
            if (store_sum)
                xsum[(size_t)(t0 + t) * H + i] = xi;
        }
        const float v = __fmul_rn(__fmul_rn(xi, rs[t]), gamma[i]);
        xs[j] = v;
        if (store)
            xn[(size_t)(t0 + t) * H + i] = v;
    }
    __syncthreads();
    if (e >= E)
        return;
    float acc[TPC];
#pragma unroll
    for (int t = 0; t < TPC; t++)
        acc[t] = 0.0f;
    auto dot4 = [&](const float4 q, int i) {
#pragma unroll
        for (int t = 0; t < TPC; t++) {
            if (t < nt) {
                const float4 v = reinterpret_cast<const float4 *>(xs + (size_t)t * H)[i];
                acc[t] = fmaf(q.x, v.x, acc[t]);
                acc[t] = fmaf(q.y, v.y, acc[t]);
                acc[t] = fmaf(q.z, v.z, acc[t]);
                acc[t] = fmaf(q.w, v.w, acc[t]);
            }
        }
    };
#pragma unroll
    for (int u = 0; u < WP; u++) {
        const int i = lane + 32 * u;
        if (i < H4)
            dot4(wpre[u], i);
    }
#pragma unroll 8 // eight row loads in flight per lane
    for (int i = lane + 32 * WP; i < H4; i += 32) {
        const float4 q = __ldg(wr + i);
        dot4(q, i);
    }
#pragma unroll
    for (int t = 0; t < TPC; t++) {
        if (t < nt) {
            const float s = warp_sum(acc[t]);
            if (lane == 0)
                logits[(size_t)(t0 + t) * E + e] = s;
        }
    }
}

// ---------------------------------------------------------------------------
// Pick across vocabulary shards ([PR826], commit "fused DS4.1 decode
// kernels": the argmax pair/pick of a vocabulary split across ranks; the
// cluster runtime commit: the greedy verify head with its vocabulary split
// across the ranks).  Shard s gave (vals[s][r], idxs[s][r]), its first
// maximum and that column's index in the whole vocabulary; the pick keeps the
// largest value, ties to the lower index.  One thread per row.
__global__ void __launch_bounds__(256)
    k_argmax_pick(const float *__restrict__ vals, const int32_t *__restrict__ idxs, int S, int R,
                  int32_t *__restrict__ idx, float *__restrict__ val)
{
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 256 + threadIdx.x;
    if (r >= R)
        return;
    float bv = vals[r];
    int32_t bi = idxs[r];
    for (int s = 1; s < S; s++) {
        const float v = vals[(size_t)s * R + r];
        const int32_t i = idxs[(size_t)s * R + r];
        if (v > bv || (v == bv && i < bi)) {
            bv = v;
            bi = i;
        }
    }
    idx[r] = bi;
    if (val)
        val[r] = bv;
}

// ---------------------------------------------------------------------------
// Expert-parallel split ([PR826], the cluster runtime commit: each rank holds
// a share of the routed experts and the ranks sum their outputs every layer;
// the review of moe_combine_masked_kernel: routes a rank does not own reach
// it masked to id -1).  The mask keeps the ids of [e0, e1) and sets the
// others to -1; the sum adds two ranks' partial outputs, one rounding each.
__global__ void __launch_bounds__(256)
    k_ep_mask(const int32_t *ids, int64_t n, int e0, int e1, int32_t *out) // in place allowed
{
    pdl_wait();
    pdl_trigger();
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        const int32_t e = ids[i];
        out[i] = (e >= e0 && e < e1) ? e : -1;
    }
}

__global__ void __launch_bounds__(256)
    k_add_f32(const float *a, const float *b, float *out, int64_t n) // in place allowed
{
    pdl_wait();
    pdl_trigger();
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
        out[i] = __fadd_rn(a[i], b[i]);
}

unsigned grid_for(int64_t n)
{
    const int64_t blocks = (n + 255) / 256;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)luce_host::sm_count() * 8));
}

} // namespace

using namespace luce_host;

// both entry points: res / xsum are NULL for the plain norm
static luce_status rmsnorm_router(const float *x, const float *res, float *xsum, const float *gamma, float eps,
                           const float *w_router, int T, int E, int H, float *xn, float *logits, void *stream)
{
    if (T < 0 || E < 1 || H < 4 || H % 4 != 0 || H > 12288 || !(eps >= 0.0f) || !std::isfinite(eps))
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!x || !gamma || !w_router || !logits || !aligned(x, 16) || !aligned(gamma, 4) || !aligned(w_router, 16) ||
        !aligned(logits, 4) || (xn && !aligned(xn, 4)) || (res && !aligned(res, 16)) || (xsum && !aligned(xsum, 4)))
        return LUCE_ERR_INVALID_ARG;
    if (xsum) {
        // the sum is stored while other CTAs still read x and r
        const size_t n = (size_t)T * H * sizeof(float);
        auto overlaps = [n](const void *a, const void *b) {
            const uintptr_t p = reinterpret_cast<uintptr_t>(a), q = reinterpret_cast<uintptr_t>(b);
            return p < q + n && q < p + n;
        };
        if (overlaps(xsum, x) || overlaps(xsum, res))
            return LUCE_ERR_INVALID_ARG;
    }
    // a tile's normed rows stay within 64 KB of shared memory (the kernel's
    // dynamic shared memory limit is raised to that once per device)
    const int tpc = std::max(1, std::min(TPC, 16384 / H));
    const int64_t tiles = ((int64_t)T + tpc - 1) / tpc;
    const int64_t chunks = ((int64_t)E + RW - 1) / RW;
    if (tiles > 65535 || chunks > INT_MAX)
        return LUCE_ERR_INVALID_ARG;
    // one token whose row fits the registers: the row path (xn and the sum
    // then need 16-byte alignment too, as their stores are float4)
    if (T == 1 && H <= 4 * 32 * WP && aligned(gamma, 16) && (!xn || aligned(xn, 16)) && (!xsum || aligned(xsum, 16)))
        return launch(k_rmsnorm_router<true>, dim3((unsigned)((E + RW_ROW - 1) / RW_ROW), 1u), dim3(RW_ROW * 32), 0,
                      as_stream(stream), x, res, xsum, gamma, eps, w_router, T, E, H, 1, xn, logits);
    const size_t smem = (size_t)tpc * H * sizeof(float);
    static SmemLimit limit;
    if (limit.raise(k_rmsnorm_router<false>, 64 * 1024) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    const luce_status st = launch(k_rmsnorm_router<false>, dim3((unsigned)chunks, (unsigned)tiles), dim3(RW * 32),
                                  smem, as_stream(stream), x, res, xsum, gamma, eps, w_router, T, E, H, tpc, xn,
                                  logits);
    if (st != LUCE_OK)
        limit.forget();
    return st;
}

extern "C" luce_status luce_rmsnorm_router(const float *x, const float *gamma, float eps, const float *w_router, int T,
                                           int E, int H, float *xn, float *logits, void *stream)
{
    return rmsnorm_router(x, nullptr, nullptr, gamma, eps, w_router, T, E, H, xn, logits, stream);
}

extern "C" luce_status luce_add_rmsnorm_router(const float *x, const float *residual, float *x_sum,
                                               const float *gamma, float eps, const float *w_router, int T, int E,
                                               int H, float *xn, float *logits, void *stream)
{
    if (!residual && T > 0)
        return LUCE_ERR_INVALID_ARG;
    return rmsnorm_router(x, residual, x_sum, gamma, eps, w_router, T, E, H, xn, logits, stream);
}

extern "C" luce_status luce_argmax_pick(const float *vals, const int32_t *idxs, int S, int R, int32_t *idx, float *val,
                                        void *stream)
{
    if (S < 1 || R < 0)
        return LUCE_ERR_INVALID_ARG;
    if (R == 0)
        return LUCE_OK;
    if (!vals || !idxs || !idx || !aligned(vals, 4) || !aligned(idxs, 4) || !aligned(idx, 4) ||
        (val && !aligned(val, 4)))
        return LUCE_ERR_INVALID_ARG;
    return launch(k_argmax_pick, dim3((unsigned)((R + 255) / 256)), dim3(256), 0, as_stream(stream), vals, idxs, S, R,
                  idx, val);
}

extern "C" luce_status luce_ep_mask(const int32_t *ids, int64_t n, int e0, int e1, int32_t *ids_out, void *stream)
{
    if (n < 0 || e0 < 0 || e1 < e0)
        return LUCE_ERR_INVALID_ARG;
    if (n == 0)
        return LUCE_OK;
    if (!ids || !ids_out || !aligned(ids, 4) || !aligned(ids_out, 4))
        return LUCE_ERR_INVALID_ARG;
    return launch(k_ep_mask, dim3(grid_for(n)), dim3(256), 0, as_stream(stream), ids, n, e0, e1, ids_out);
}

extern "C" luce_status luce_add_f32(const float *a, const float *b, float *out, int64_t n, void *stream)
{
    if (n < 0)
        return LUCE_ERR_INVALID_ARG;
    if (n == 0)
        return LUCE_OK;
    if (!a || !b || !out || !aligned(a, 4) || !aligned(b, 4) || !aligned(out, 4))
        return LUCE_ERR_INVALID_ARG;
    return launch(k_add_f32, dim3(grid_for(n)), dim3(256), 0, as_stream(stream), a, b, out, n);
}
