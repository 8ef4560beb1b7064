// q4k_ops.cu -- the gate/up pair with its SwiGLU and the down product with
// the masked route-weighted combine for Q4_K expert weights, with their
// C-ABI entry points.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving": commit "fused DS4.1 decode kernels" (wide Q4_K
// products among the layer's matrix products), commit "RDNA4 Q8_0 gate/up
// pair" (gate and up on one load of the activations, the GLU in the
// epilogue), commit "fused routed combine and q8_1 inputs for the hybrid
// owners" (masked combine, each product and sum rounded on its own).
//
// Format (the ggml K-quant the pages name): a super-block of 256 values in
// 144 bytes -- fp16 d, fp16 dmin, 12 bytes packing eight 6-bit scales sc_j
// and mins m_j, 128 bytes of 4-bit codes; sub-block j (32 values) takes the
// low (j even) or high (j odd) nibbles of bytes 32 (j / 2) ...  Against a
// q8_1 activation block (d8, s8 = d8 sum q8, codes) sub-block j contributes
// d sc_j d8 isum_j - dmin m_j s8, isum_j the exact int32 sum of codes times
// activation codes.
//
// Design: one warp per dot product row; a lane takes a pair of sub-blocks
// (2c, 2c + 1) of a super-block, whose codes are the same 32 bytes (low and
// high nibbles), with 16-byte loads of the super-block header and codes;
// dp4a on nibble-masked words.  A gate/up block stages the token's q8_1 row
// in shared memory once and owns 32 consecutive h values (two rows per warp),
// one q8_1 block of h, which it quantizes itself when asked (no separate
// quantization launch).  The down/combine warps take one route slot per
// half-warp when a row has at most 16 sub-block pairs (four slots per half in
// flight), the shared expert as the last slot of the same pass.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_q4k)

namespace {

using namespace luce;

constexpr int Q4K_BYTES = 144;
constexpr int QKK = 256;
constexpr int WARPS = 8;           // warps per down/combine block
constexpr int GW = 16;             // warps per gate/up block
constexpr int GR = QK / GW;        // h rows per gate/up warp: a block's GW x GR rows are one q8_1 block

// (sc, m) of sub-blocks 2c and 2c + 1 from the 12 scale bytes held as three
// little-endian words
__device__ __forceinline__ void scale_min_pair(const uint32_t (&sw)[3], int c, int (&sc)[2], int (&m)[2])
{
    auto byte = [&](int i) -> int { return (int)((sw[i >> 2] >> (8 * (i & 3))) & 0xffu); };
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int j = 2 * c + h;
        if (j < 4) {
            sc[h] = byte(j) & 63;
            m[h] = byte(j + 4) & 63;
        } else {
            sc[h] = (byte(j + 4) & 15) | ((byte(j - 4) >> 6) << 4);
            m[h] = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
        }
    }
}

// The weight bytes of sub-block pair p (sub-blocks 2c and 2c + 1 of
// super-block p / 4) of a Q4_K row: the super-block header and the pair's 32
// code bytes.
struct Q4Pair {
    uint4 hd, q0, q1;
};

__device__ __forceinline__ Q4Pair q4k_pair_load(const uint8_t *__restrict__ w_row, int p)
{
    const int sb = p >> 2, c = p & 3;
    const uint4 *qp = reinterpret_cast<const uint4 *>(w_row + (size_t)sb * Q4K_BYTES + 16 + 32 * c);
    return {__ldg(reinterpret_cast<const uint4 *>(w_row + (size_t)sb * Q4K_BYTES)), __ldg(qp), __ldg(qp + 1)};
}

// Loaded sub-block pair p of a Q4_K row times a q8_1 row, added to acc.
template <bool XS = false>
__device__ __forceinline__ float q4k_pair_fma(const Q4Pair &wp, const uint32_t *__restrict__ x_row, int p, float acc)
{
    {
        const int sb = p >> 2, c = p & 3;
        const uint4 hd = wp.hd, q0 = wp.q0, q1 = wp.q1;
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
        const uint32_t sw[3] = {hd.y, hd.z, hd.w};
        int sc[2], m[2];
        scale_min_pair(sw, c, sc, m);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint32_t *xb = x_row + (size_t)(8 * sb + 2 * c + h) * Q8_1_WORDS;
            const uint32_t xd = XS ? xb[0] : __ldg(xb);
            int isum = 0;
#pragma unroll
            for (int w = 0; w < 8; w++)
                isum = __dp4a((int)((qw[w] >> (4 * h)) & 0x0F0F0F0Fu), (int)(XS ? xb[1 + w] : __ldg(xb + 1 + w)), isum);
            const float d8 = half_bits_to_float(xd), s8 = half_bits_to_float(xd >> 16);
            acc = fmaf(d * (float)sc[h] * d8, (float)isum, acc);
            acc = fmaf(-dmin * (float)m[h], s8, acc);
        }
    }
    return acc;
}

// Sub-block pair p of a Q4_K row times a q8_1 row, added to acc.
template <bool XS = false>
__device__ __forceinline__ float q4k_pair_dot(const uint8_t *__restrict__ w_row, const uint32_t *__restrict__ x_row,
                                              int p, float acc)
{
    return q4k_pair_fma<XS>(q4k_pair_load(w_row, p), x_row, p, acc);
}

// This lane's part of a Q4_K row (K values) times a q8_1 row: pairs
// p = lane, lane + 32, ... of the row's K / 64 sub-block pairs.
__device__ __forceinline__ float q4k_lane_dot(const uint8_t *__restrict__ w_row, const uint32_t *__restrict__ x_row,
                                              int K, int lane)
{
    float acc = 0.0f;
    const int P = K >> 6;
    for (int p = lane; p < P; p += 32)
        acc = q4k_pair_dot(w_row, x_row, p, acc);
    return acc;
}

// Gate/up rows -> h (and its q8_1 block).  Block (32-row block b of h,
// route or shared row r); warp w computes h[r][i] for i = 32 b + GR w + j,
// j < GR, with the loads of its GR gate and GR up rows in flight together.
// With hq the block's 32 values are then quantized by warp 0 into
// hq[r][b] (the q8_1 rule of luce_quantize_q8_1, the same bits).  Under
// programmatic launch a CTA releases the next kernel only once its stores are
// issued: released at the start, the next kernel's CTAs became resident and
// waited beside this kernel's, which made the pair slower than with a third
// launch between them.
__global__ void __launch_bounds__(GW * 32)
    k_glu_q4k(const uint8_t *__restrict__ wg, const uint8_t *__restrict__ wu, const uint8_t *__restrict__ wsg,
              const uint8_t *__restrict__ wsu, const uint32_t *__restrict__ xq, const int32_t *__restrict__ ids, int T,
              int k, int E, int H, int I, float clamp, float *__restrict__ h, uint32_t *__restrict__ hq)
{
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.y, i0 = blockIdx.x * QK + warp * GR;
    extern __shared__ uint32_t xs[]; // the token's q8_1 row
    __shared__ float hs[QK];
    const uint8_t *G, *U;
    const size_t rowb = (size_t)(H / QKK) * Q4K_BYTES;
    if (r < T * k) {
        const int e = ids[r];
        if (e < 0)
            return; // masked route (the whole block: r is the block's)
        if (e >= E) {
            if (threadIdx.x == 0 && blockIdx.x == 0)
                atomicOr(&g_fault_word, LUCE_FAULT_BAD_ID);
            return;
        }
        G = wg + ((size_t)e * I + i0) * rowb;
        U = wu + ((size_t)e * I + i0) * rowb;
    } else {
        G = wsg + (size_t)i0 * rowb;
        U = wsu + (size_t)i0 * rowb;
    }
    {
        const int tt = r < T * k ? r / k : r - T * k;
        const uint32_t *xr = xq + (size_t)tt * (H / QK) * Q8_1_WORDS;
        for (int w = threadIdx.x; w < (H / QK) * Q8_1_WORDS; w += GW * 32)
            xs[w] = __ldg(xr + w);
        __syncthreads();
    }
    float gl[GR], ul[GR];
#pragma unroll
    for (int j = 0; j < GR; j++)
        gl[j] = ul[j] = 0.0f;
    for (int p = lane; p < (H >> 6); p += 32) {
#pragma unroll
        for (int j = 0; j < GR; j++) {
            gl[j] = q4k_pair_dot<true>(G + (size_t)j * rowb, xs, p, gl[j]);
            ul[j] = q4k_pair_dot<true>(U + (size_t)j * rowb, xs, p, ul[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < GR; j++) {
        const float g = warp_sum(gl[j]);
        const float u = warp_sum(ul[j]);
        const float v = swiglu(g, u, clamp);
        if (lane == 0) {
            h[(size_t)r * I + i0 + j] = v;
            hs[warp * GR + j] = v;
        }
    }
    if (hq == nullptr) {
        pdl_trigger();
        return;
    }
    __syncthreads();
    if (warp == 0)
        quantize_q8_1_warp(hs[lane], hq + ((size_t)r * (I / QK) + blockIdx.x) * Q8_1_WORDS, lane);
    pdl_trigger();
}

// Down rows and the combine.  Block (chunk of WARPS output rows, token t);
// warp w: out[t][n] for n = blockIdx.x WARPS + w, the k route slots in slot
// order with each product and sum rounded, then the shared expert.  The next
// kernel is released once the out values are stored (as in k_glu_q4k).  On
// rows of at most 16 sub-block pairs the route ids and weights and the first
// pass's weight bytes are read before the wait for the previous kernel (the
// gate/up launch, which writes only h and hq): the weight stream starts while
// that kernel drains.
__global__ void __launch_bounds__(WARPS * 32)
    k_down_combine_q4k(const uint8_t *__restrict__ wd, const uint8_t *__restrict__ wsd,
                       const uint32_t *__restrict__ hq, const int32_t *__restrict__ ids,
                       const float *__restrict__ weights, int T, int k, int E, int H, int I, float *__restrict__ out)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.y, n = blockIdx.x * WARPS + warp;
    const size_t rowb = (size_t)(I / QKK) * Q4K_BYTES;
    const size_t hrow = (size_t)(I / QK) * Q8_1_WORDS;
    float acc = 0.0f;
    if ((I >> 6) <= 16) {
        // A row has at most 16 sub-block pairs: each half-warp takes a slot
        // (half 0 the even ones, half 1 the odd ones), one pair per lane, four
        // slots per half in flight at once; slot k is the shared expert, so
        // its row is read in the same pass as the routed ones and still joins
        // the combine last, unweighted.  The half-warp butterfly adds the same
        // values in the same order as the warp butterfly over a warp whose
        // upper 16 lanes hold zeros (and the two halves reduce alike), so
        // every y is the one-slot-per-warp y.
        const int P = I >> 6, hh = lane >> 4, pl = lane & 15;
        const int ns = k + (wsd ? 1 : 0);
        constexpr int SJ = 8; // slots per pass (four per half)
        for (int j0 = 0; j0 < ns; j0 += SJ) {
            float part[SJ / 2];
            bool live[SJ / 2];
            Q4Pair wp[SJ / 2];
#pragma unroll
            for (int q = 0; q < SJ / 2; q++) {
                const int j = j0 + 2 * q + hh;
                const int e = j < k ? ids[t * k + j] : -1;
                if (e >= E && pl == 0 && n == 0)
                    atomicOr(&g_fault_word, LUCE_FAULT_BAD_ID);
                const bool sh = j == k && wsd != nullptr;
                live[q] = sh || (e >= 0 && e < E);
                const uint8_t *wrow = sh ? wsd + (size_t)n * rowb : wd + ((size_t)e * H + n) * rowb;
                if (live[q] && pl < P)
                    wp[q] = q4k_pair_load(wrow, pl);
            }
            if (j0 == 0)
                pdl_wait(); // hq is the previous kernel's
#pragma unroll
            for (int q = 0; q < SJ / 2; q++) {
                const int j = j0 + 2 * q + hh;
                const bool sh = j == k && wsd != nullptr;
                const uint32_t *hr = hq + (size_t)(sh ? T * k + t : t * k + j) * hrow;
                part[q] = live[q] && pl < P ? q4k_pair_fma(wp[q], hr, pl, 0.0f) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < SJ / 2; q++) {
                const float y = half_warp_sum(part[q]);
                const float y0 = __shfl_sync(0xffffffffu, y, 0), y1 = __shfl_sync(0xffffffffu, y, 16);
                const bool l0 = __shfl_sync(0xffffffffu, live[q], 0), l1 = __shfl_sync(0xffffffffu, live[q], 16);
                const int j = j0 + 2 * q;
                if (l0)
                    acc = __fadd_rn(acc, j == k ? y0 : __fmul_rn(weights[t * k + j], y0));
                if (l1)
                    acc = __fadd_rn(acc, j + 1 == k ? y1 : __fmul_rn(weights[t * k + j + 1], y1));
            }
        }
        if (lane == 0)
            out[(size_t)t * H + n] = acc;
        pdl_trigger();
        return;
    }
    pdl_wait();
    // SB slots at a time: their lane dots do not depend on one another, so
    // the loads of all of them are in flight together; the sums then join
    // the combine in slot order
    constexpr int SB = 8;
    for (int j0 = 0; j0 < k; j0 += SB) {
        float yl[SB];
        bool live[SB];
#pragma unroll
        for (int jj = 0; jj < SB; jj++) {
            const int j = j0 + jj;
            const int e = j < k ? ids[t * k + j] : -1;
            if (e >= E && lane == 0 && n == 0)
                atomicOr(&g_fault_word, LUCE_FAULT_BAD_ID);
            live[jj] = e >= 0 && e < E;
            yl[jj] = live[jj] ? q4k_lane_dot(wd + ((size_t)e * H + n) * rowb, hq + (size_t)(t * k + j) * hrow, I, lane)
                              : 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < SB; jj++) {
            const float y = warp_sum(yl[jj]);
            if (live[jj])
                acc = __fadd_rn(acc, __fmul_rn(weights[t * k + j0 + jj], y));
        }
    }
    if (wsd) {
        const float y = warp_sum(q4k_lane_dot(wsd + (size_t)n * rowb, hq + ((size_t)T * k + t) * hrow, I, lane));
        acc = __fadd_rn(acc, y);
    }
    if (lane == 0)
        out[(size_t)t * H + n] = acc;
    pdl_trigger();
}

} // namespace

using namespace luce_host;

extern "C" luce_status luce_moe_glu_q4k(const luce_block_q4_k *w_gate, const luce_block_q4_k *w_up,
                                        const luce_block_q4_k *ws_gate, const luce_block_q4_k *ws_up,
                                        const luce_block_q8_1 *xq, const int32_t *ids, int T, int k, int E, int H,
                                        int I, float clamp, float *h, luce_block_q8_1 *hq, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 64 || H <= 0 || I <= 0 || H % QKK != 0 ||
        I % QKK != 0 || !(clamp == clamp))
        return LUCE_ERR_INVALID_ARG;
    const bool has_ws = ws_gate != nullptr;
    if ((ws_up != nullptr) != has_ws)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!w_gate || !w_up || !xq || !ids || !h || !aligned(w_gate, 16) || !aligned(w_up, 16) ||
        (has_ws && (!aligned(ws_gate, 16) || !aligned(ws_up, 16))) || !aligned(xq, 4) || !aligned(ids, 4) ||
        !aligned(h, 4) || (hq && !aligned(hq, 4)))
        return LUCE_ERR_INVALID_ARG;
    const int rows = T * k + (has_ws ? T : 0);
    if ((int64_t)T * k > (1 << 20) || rows > 65535)
        return LUCE_ERR_INVALID_ARG;
    // one block per 32 h values (I % 256 == 0, so no partial block)
    return launch(k_glu_q4k, dim3((unsigned)(I / QK), (unsigned)rows), dim3(GW * 32),
                  (size_t)(H / QK) * Q8_1_WORDS * 4,
                  as_stream(stream), reinterpret_cast<const uint8_t *>(w_gate), reinterpret_cast<const uint8_t *>(w_up),
                  reinterpret_cast<const uint8_t *>(ws_gate), reinterpret_cast<const uint8_t *>(ws_up),
                  reinterpret_cast<const uint32_t *>(xq), ids, T, k, E, H, I, clamp, h,
                  reinterpret_cast<uint32_t *>(hq));
}

extern "C" luce_status luce_moe_down_combine_q4k(const luce_block_q4_k *w_down, const luce_block_q4_k *ws_down,
                                                 const luce_block_q8_1 *hq, const int32_t *ids, const float *weights,
                                                 int T, int k, int E, int H, int I, float *out, void *stream)
{
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || k > 64 || H <= 0 || I <= 0 || H % QKK != 0 ||
        I % QKK != 0)
        return LUCE_ERR_INVALID_ARG;
    if (T == 0)
        return LUCE_OK;
    if (!w_down || !hq || !ids || !weights || !out || !aligned(w_down, 16) || (ws_down && !aligned(ws_down, 16)) ||
        !aligned(hq, 4) || !aligned(ids, 4) || !aligned(weights, 4) || !aligned(out, 4))
        return LUCE_ERR_INVALID_ARG;
    if (T > 65535)
        return LUCE_ERR_INVALID_ARG;
    return launch(k_down_combine_q4k, dim3((unsigned)((H + WARPS - 1) / WARPS), (unsigned)T), dim3(WARPS * 32), 0,
                  as_stream(stream), reinterpret_cast<const uint8_t *>(w_down),
                  reinterpret_cast<const uint8_t *>(ws_down), reinterpret_cast<const uint32_t *>(hq), ids, weights, T,
                  k, E, H, I, out);
}
