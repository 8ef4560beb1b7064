/*
 * luce_moe.h -- C ABI of the GB300 (sm_103a) routed-MoE FFN decode library.
 *
 * The library computes the routed mixture-of-experts FFN step of an LLM
 * decode or speculative-verify pass on Q8_0-quantized experts, plus the
 * exact greedy argmax over a vocabulary of logits.  It is a from-scratch
 * design of the operations described on the page Lucebox PR #826
 * "feat(ds41): two-box expert-parallel serving" (cited below as [PR826],
 * with the section of the page: a commit subject, a code review, or a part
 * of the PR description).
 *
 * Conventions shared by every entry point:
 *   - All array pointers are DEVICE pointers, owned by the caller.  The
 *     library never allocates, frees or retains memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream: LUCE_OK means the
 *     work was validated and enqueued, nothing more.  Outputs are ready when
 *     the stream reaches that point.
 *   - Arguments are validated on the host before anything is launched; a
 *     bad argument returns LUCE_ERR_INVALID_ARG (or LUCE_ERR_UNSUPPORTED for
 *     a valid shape this library has no kernel for) with nothing enqueued.
 *     A launch failure returns LUCE_ERR_CUDA.  No C++ exception crosses the
 *     ABI.  T == 0 (or R == 0) is a valid empty call that enqueues nothing.
 *   - Route ids < 0 are masked routes ([PR826], review "moe_combine_masked_
 *     kernel indexes valid with an unchecked (possibly -1) route id"): they
 *     are skipped by grouping, products and combine.  Ids >= E are invalid
 *     data; kernels skip them and raise LUCE_FAULT_BAD_ID (luce_get_fault).
 *   - Outputs never alias inputs.
 *
 * Data layouts (row-major, little-endian):
 *   luce_block_q8_0  32 int8 codes q and an fp16 scale d; value = d*q.
 *                    34 bytes.  The ggml block_q8_0 layout the page names
 *                    (review of the commit "whole-row-lane slice").
 *   luce_block_q8_1  fp16 d, fp16 s = d*sum(q), 32 int8 codes; 36 bytes.
 *                    The q8_1 activation rows of [PR826], commit "fused
 *                    DS4.1 decode kernels" (the q8_1 activation memo).
 *   A Q8_0 matrix [rows][K] is rows*K/32 blocks, row after row.
 *   Expert weights: w_gate, w_up [E][I][H/32] blocks; w_down [E][H][I/32].
 *   The shared expert's weights have the same shapes without the E axis.
 */
#ifndef LUCE_MOE_H
#define LUCE_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LUCE_API __attribute__((visibility("default")))
#else
#define LUCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LUCE_OK = 0,
    LUCE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or shape     */
    LUCE_ERR_UNSUPPORTED = 2, /* valid but not supported by this library   */
    LUCE_ERR_CUDA = 3         /* a CUDA runtime call or launch failed      */
} luce_status;

typedef struct {
    uint16_t d;    /* fp16 scale */
    int8_t qs[32]; /* codes      */
} luce_block_q8_0;

typedef struct {
    uint16_t d;    /* fp16 scale d = max|x| / 127 */
    uint16_t s;    /* fp16 d * sum(qs)            */
    int8_t qs[32]; /* codes round(x / d)          */
} luce_block_q8_1;

typedef struct {
    uint16_t d;          /* fp16 super-block scale                       */
    uint16_t dmin;       /* fp16 super-block scale of the mins           */
    uint8_t scales[12];  /* eight 6-bit scales and eight 6-bit mins      */
    uint8_t qs[128];     /* 256 4-bit codes (see luce_moe_glu_q4k)       */
} luce_block_q4_k;

/* Device fault bits (luce_get_fault). */
#define LUCE_FAULT_BAD_ID 0x1u  /* a route id >= E was seen and skipped          */
#define LUCE_FAULT_TIMEOUT 0x2u /* a bounded device wait gave up (never expected) */
#define LUCE_FAULT_DESYNC 0x4u  /* a device-wide barrier of luce_moe_layer gave up: its count is out of step
                                   with the grid, so zero the `sync` word before the next call */

/* ------------------------------------------------------------------------
 * luce_route_topk -- router select + weights in one launch.
 * [PR826], commit "fused DS4.1 decode kernels": the router's selection and
 * its weights, both read from one set of logits, run as a single launch.
 *
 * Per token t: score_e = logits[t][e] + bias[e] (fp32 add).  The k largest
 * scores are selected, best first; equal scores go to the lower index.
 * weights[t][j] = softmax over the k selected UNBIASED logits (max-
 * subtracted, fp32 expf).  The bias only steers selection.
 *
 *   logits  [T][E] fp32          bias [E] fp32, or NULL for none
 *   ids     [T][k] int32 out     weights [T][k] fp32 out
 * Requires 1 <= E <= 1024, 1 <= k <= min(E, 64), T >= 0, 4-byte alignment.
 */
LUCE_API luce_status luce_route_topk(const float *logits, const float *bias, int T, int E, int k, int32_t *ids,
                            float *weights, void *stream);

/* ------------------------------------------------------------------------
 * luce_quantize_q8_1 -- quantize fp32 rows to q8_1 blocks, once per layer.
 * [PR826], commit "fused DS4.1 decode kernels" (the q8_1 activation memo,
 * reused by every reshape) and commit "fused routed combine and q8_1 inputs
 * for the hybrid owners" (the FFN input is quantized once, to the q8_1 rows
 * the matrix-vector kernels read).
 *
 * Per 32-value block: amax = max|x|, d = amax / 127 (fp32 IEEE division),
 * q = roundf(x / d) (half away from zero; 0 when amax == 0), stored
 * d16 = fp16(d) and s16 = fp16(d * sum(q)), fp16 round to nearest even.
 *
 *   x   [T][K] fp32 (4-byte aligned)      xq [T][K/32] luce_block_q8_1 out
 * Requires K % 32 == 0, K > 0, xq 4-byte aligned.
 */
LUCE_API luce_status luce_quantize_q8_1(const float *x, int T, int K, luce_block_q8_1 *xq, void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_group -- group the T*k routes by expert (one counting sort per
 * layer, shared by gate, up and down).  [PR826], commit "fused DS4.1 decode
 * kernels": a single grouping per MoE layer serves gate, up and down.
 *
 * Route r = t*k + j has expert ids[r].  Outputs:
 *   counts  [E]    number of routes of expert e (masked routes excluded)
 *   offsets [E+1]  offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   routes  [T*k]  routes[offsets[e] .. offsets[e+1]) = the route indices
 *                  r of expert e in increasing r; the tail after
 *                  offsets[E] is filled with -1.
 * One CTA, no atomics on the order: the result is unique and deterministic.
 * Requires 1 <= E <= 1024, 1 <= k <= 64, T*k <= 2^20, 4-byte alignment.
 */
LUCE_API luce_status luce_moe_group(const int32_t *ids, int T, int k, int E, int32_t *counts, int32_t *offsets,
                           int32_t *routes, void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_glu_pair -- the Q8_0 gate/up products of every routed token and
 * of the shared expert, fused with the (clamped) SwiGLU and the q8_1
 * quantization of its result.  [PR826], commit "RDNA4 Q8_0 gate/up pair"
 * (both matrices read with one load of each activation fragment, the GLU
 * written in the epilogue) and commit "fused routed combine ..." (the
 * clamped routed SwiGLU).
 *
 * For each expert e with routes (from luce_moe_group), for each of its
 * routes r = t*k + j and each row i < I:
 *   g = W_gate[e][i] . xq[t],  u = W_up[e][i] . xq[t]
 *   h[r][i] = silu(g) * u                                  (clamp <= 0)
 *   h[r][i] = silu(min(g, clamp)) * min(max(u, -clamp), clamp)   (clamp > 0)
 * where a row dot is sum_b d_w[b] * d_x[b] * isum[b] with exact int32 block
 * sums isum[b] (dp4a) accumulated in fp32.  If ws_gate/ws_up are given, the
 * shared expert is computed for every token t into row T*k + t.
 * hq[r] = q8_1(h[r]) with the rule of luce_quantize_q8_1, from exactly the
 * fp32 h values stored.  Rows of masked routes are not written.
 *
 *   w_gate, w_up   [E][I][H/32] Q8_0        ws_gate, ws_up [I][H/32] or NULL
 *   xq             [T][H/32] q8_1           offsets [E+1], routes [T*k]
 *   h              [T*k + T][I] fp32 out    hq [T*k + T][I/32] q8_1 out
 *   variant        0 = automatic (only one kernel exists in this library)
 * Requires H % 256 == 0, I % 256 == 0, H/32 <= 1024; w_*, xq, hq 16-byte
 * aligned; ws_gate and ws_up both given or both NULL.
 */
LUCE_API luce_status luce_moe_glu_pair(const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                              const luce_block_q8_0 *ws_gate, const luce_block_q8_0 *ws_up,
                              const luce_block_q8_1 *xq, const int32_t *offsets, const int32_t *routes, int T, int k,
                              int E, int H, int I, float clamp, float *h, luce_block_q8_1 *hq, int variant,
                              void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_down_combine -- the Q8_0 down product of every route and of the
 * shared expert, fused with the masked, route-weighted combine.  [PR826],
 * commit "fused routed combine and q8_1 inputs for the hybrid owners": masking
 * the routes, weighting them and summing them is one launch, and the masked
 * combine rounds every product and every sum on its own.
 *
 *   y[r][n]  = W_down[ids[r]][n] . hq[r]        (fp32, as in luce_moe_glu_pair)
 *   yS[t][n] = Ws_down[n] . hq[T*k + t]         (if ws_down is given)
 *   out[t][n] = 0; for j = 0..k-1 with ids[t*k+j] >= 0:
 *                    out = out + w[t][j] * y[t*k+j][n]   (product rounded,
 *                                                         then sum rounded)
 *               then out = out + yS[t][n]
 * No floating-point atomics: each out element is summed by one thread in
 * slot order, so the result is deterministic.
 *
 *   w_down [E][H][I/32] Q8_0    ws_down [H][I/32] or NULL
 *   hq [T*k + T][I/32] q8_1     ids, weights [T][k]   offsets, routes as above
 *   out [T][H] fp32 out         variant 0 = automatic
 * Requires H % 256 == 0 (H >= 256), I % 256 == 0, I/32 <= 1024; w_*, hq
 * 16-byte aligned.
 */
LUCE_API luce_status luce_moe_down_combine(const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_down,
                                  const luce_block_q8_1 *hq, const int32_t *ids, const float *weights,
                                  const int32_t *offsets, const int32_t *routes, int T, int k, int E, int H, int I,
                                  float *out, int variant, void *stream);

/* ------------------------------------------------------------------------
 * luce_argmax -- exact greedy argmax per row, as a "pair/pick": each CTA
 * reduces a chunk of a row to a (value, index) pair and one CTA picks among
 * the row's pairs (rows of 16,384 values or more: one cluster of CTAs per
 * row, the pairs joined in distributed shared memory; shorter rows: the
 * last CTA of the row to finish picks from pairs in the workspace).
 * [PR826], commit "fused DS4.1 decode kernels": the greedy token comes from
 * an exact argmax done as pairs and a pick.
 *
 * idx[r] = the lowest index of the maximum of logits[r][0..V) (float
 * comparison: -0 == +0 is a tie; inputs must hold no NaN); val[r] = that
 * maximum (val may be NULL).
 *
 *   logits [R][V] fp32          idx [R] int32 out      val [R] fp32 out or NULL
 *   workspace, workspace_bytes  device scratch of at least
 *                               luce_argmax_workspace_bytes(R, V) bytes,
 *                               8-byte aligned, ZERO-FILLED before its first
 *                               use.  Each call leaves it zero-filled again,
 *                               so one buffer serves any number of calls on
 *                               one stream; calls that overlap on the GPU
 *                               must not share it.
 * Requires 1 <= V < 2^31, R >= 0, logits 4-byte aligned.
 */
LUCE_API luce_status luce_argmax(const float *logits, int R, int64_t V, int32_t *idx, float *val, void *workspace,
                        size_t workspace_bytes, void *stream);
LUCE_API size_t luce_argmax_workspace_bytes(int R, int64_t V);

/* ------------------------------------------------------------------------
 * luce_argmax_noalloc -- the same argmax as luce_argmax, for callers that
 * cannot allocate device memory: a host application that owns every device
 * allocation and hands this library none, or a loop that must never call
 * into the CUDA allocator.  Such callers cannot supply the workspace of
 * luce_argmax, so this call uses scratch that the library itself holds: a
 * fixed 16 KB array of device memory that exists on every GPU that loads the
 * library, from load to exit.  (The pages have no counterpart of this call;
 * it exists only for such callers.)
 *
 *   logits [R][V] fp32   idx [R] int32 out   val [R] fp32 out or NULL
 * Results are identical to luce_argmax.  Allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library routine.  R above 1024 rows, or a
 * (R, V) whose scratch need (luce_argmax_workspace_bytes) exceeds 16 KB,
 * returns LUCE_ERR_UNSUPPORTED: use luce_argmax with a workspace instead.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture begins.
 * Every call clears the part of the array that must start at zero.  All
 * calls share the one array, so calls that overlap on the GPU (on different
 * streams, or from different host threads) race: order them on one stream.
 */
LUCE_API luce_status luce_argmax_noalloc(const float *logits, int R, int64_t V, int32_t *idx, float *val,
                                         void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_glu_q4k / luce_moe_down_combine_q4k -- the gate/up pair with its
 * SwiGLU and the down product with the masked route-weighted combine, for
 * Q4_K expert weights.  [PR826], commit "fused DS4.1 decode kernels" (wide
 * Q4_K products among the layer's products); the arithmetic around the dot
 * products is that of luce_moe_glu_pair and luce_moe_down_combine.
 *
 * Q4_K (the ggml K-quant the pages name; the pages do not define it): a
 * super-block of 256 values, luce_block_q4_k, 144 bytes.  Sub-block j
 * (values 32 j .. 32 j + 31) has a 6-bit scale sc_j and a 6-bit min m_j:
 * for j < 4, sc_j = scales[j] & 63 and m_j = scales[j + 4] & 63; for j >= 4,
 * sc_j = (scales[j + 4] & 15) | (scales[j - 4] >> 6) << 4 and
 * m_j = (scales[j + 4] >> 4) | (scales[j] >> 6) << 4.  Its codes q are the low
 * (j even) or high (j odd) nibbles of qs[32 (j / 2) .. 32 (j / 2) + 31], and
 * value i is d sc_j q_i - dmin m_j.  Against a q8_1 block (d8, s8, codes)
 * sub-block j contributes d sc_j d8 isum_j - dmin m_j s8, with the stored
 * fp16 s8 (isum_j: exact int32 sum of code products).
 *
 * luce_moe_glu_q4k: w_gate, w_up [E][I][H/256] blocks (16-byte aligned);
 *   ws_gate, ws_up [I][H/256] or both NULL; xq [T][H/32] q8_1; ids [T][k]
 *   (id < 0: masked, its h row untouched; id >= E: skipped and
 *   LUCE_FAULT_BAD_ID).  h [T*k (+T)][I] fp32 out: h = silu(g) u, or the
 *   clamped form when clamp > 0 (as luce_moe_glu_pair).  hq [T*k (+T)][I/32]
 *   q8_1 out or NULL: h quantized by the rule of luce_quantize_q8_1 (the same
 *   bits) in the same launch; rows of masked or skipped routes are left
 *   untouched in both.  With hq NULL, quantize h with luce_quantize_q8_1.
 * luce_moe_down_combine_q4k: w_down [E][H][I/256] (16-byte aligned), ws_down
 *   [H][I/256] or NULL, hq [T*k (+T)][I/32] q8_1, ids [T][k], weights [T][k]
 *   fp32 -> out [T][H] fp32, the combine of luce_moe_down_combine (slot
 *   order, each product and sum rounded, shared expert last).
 * Requires H % 256 == 0, I % 256 == 0, 1 <= k <= min(E, 64), E <= 1024.
 * Gate/up: one block per 32 values of h (two rows per warp); down: one warp
 * per output value.  Every weight row is read once per column that needs it.
 */
LUCE_API luce_status luce_moe_glu_q4k(const luce_block_q4_k *w_gate, const luce_block_q4_k *w_up,
                                      const luce_block_q4_k *ws_gate, const luce_block_q4_k *ws_up,
                                      const luce_block_q8_1 *xq, const int32_t *ids, int T, int k, int E, int H,
                                      int I, float clamp, float *h, luce_block_q8_1 *hq, void *stream);
LUCE_API luce_status luce_moe_down_combine_q4k(const luce_block_q4_k *w_down, const luce_block_q4_k *ws_down,
                                               const luce_block_q8_1 *hq, const int32_t *ids, const float *weights,
                                               int T, int k, int E, int H, int I, float *out, void *stream);

/* ------------------------------------------------------------------------
 * luce_argmax_shard / luce_argmax_pick -- the greedy token of a vocabulary
 * split into S shards (one per rank).  [PR826], commit "fused DS4.1 decode
 * kernels" (the argmax pair/pick over a vocabulary split across ranks, exact)
 * and the cluster runtime commit (the greedy verify head with its vocabulary
 * split across the ranks).
 *
 * luce_argmax_shard: the argmax of one shard, logits [R][Vs] fp32 whose
 *   column 0 is column v0 of the whole vocabulary: idx[r] = v0 + the lowest
 *   index of the shard row's maximum, val[r] = that maximum.  Same kernel,
 *   workspace (luce_argmax_workspace_bytes(R, Vs), zero-filled, left zero)
 *   and rules as luce_argmax.  Requires v0 >= 0 and v0 + Vs < 2^31.
 * luce_argmax_pick: vals [S][R] fp32 and idxs [S][R] int32 are the shards'
 *   results (shard-major, as gathered from the ranks); idx[r] / val[r] (val
 *   may be NULL) = the pair with the largest value, among equal values the
 *   lower index.  With shards covering disjoint column ranges this is
 *   exactly luce_argmax of the whole rows.  S >= 1, R >= 0; 4-byte aligned.
 */
LUCE_API luce_status luce_argmax_shard(const float *logits, int R, int64_t Vs, int64_t v0, int32_t *idx, float *val,
                                       void *workspace, size_t workspace_bytes, void *stream);
LUCE_API luce_status luce_argmax_pick(const float *vals, const int32_t *idxs, int S, int R, int32_t *idx, float *val,
                                      void *stream);

/* ------------------------------------------------------------------------
 * luce_rmsnorm_router -- the step before the router: the RMS norm of the
 * hidden rows and the router logits of the normed rows.  [PR826], commit
 * "fused DS4.1 decode kernels" (the RMS norm among the fused launches) and
 * the HC pre-mix commit (an RMS norm with its sum of squares and products in
 * F32).  The pages do not spell out either formula; this is the standard RMS
 * norm and a plain product with an F32 router matrix:
 *   xn[t][i]     = x[t][i] * r_t * gamma[i],  r_t = 1 / sqrt(mean_i x[t][i]^2 + eps)
 *   logits[t][e] = sum_i w_router[e][i] * xn[t][i]
 * in fp32 (IEEE square root and divisions; the sums in the kernel's order,
 * graded by tolerance against a double-precision oracle).
 *
 *   x [T][H] fp32 (16-byte aligned)    gamma [H] fp32    eps >= 0, finite
 *   w_router [E][H] fp32 (16-byte aligned)
 *   xn [T][H] fp32 out or NULL (not stored); must not overlap x
 *   logits [T][E] fp32 out (the input of luce_route_topk / luce_moe_layer)
 * Requires H % 4 == 0, 4 <= H <= 12288, E >= 1, T >= 0.  Under programmatic
 * launch (luce_set_pdl) the kernel reads w_router (and, for one token with
 * H <= 2048 and a 16-byte aligned gamma, gamma) before it waits for the
 * previous kernel, so that kernel must write neither.
 */
LUCE_API luce_status luce_rmsnorm_router(const float *x, const float *gamma, float eps, const float *w_router, int T,
                                         int E, int H, float *xn, float *logits, void *stream);

/* ------------------------------------------------------------------------
 * luce_add_rmsnorm_router -- luce_rmsnorm_router of the residual sum: the
 * residual add that makes a layer's input (the previous layer's input plus
 * its output) folded into the same launch as the norm and the router logits.
 * The pages list the RMS norm among the launches that the decode path fuses
 * ([PR826], commit "fused DS4.1 decode kernels"); the add is one fp32
 * addition per value:
 *   s[t][i] = x[t][i] + residual[t][i]     (fp32, round to nearest)
 * and then xn and logits exactly as luce_rmsnorm_router computes them from s
 * (the same bits as luce_add_f32 followed by luce_rmsnorm_router).
 *
 *   x, residual [T][H] fp32, both 16-byte aligned
 *   x_sum [T][H] fp32 out or NULL (not stored); must not overlap x or residual
 *   gamma, eps, w_router, xn, logits, T, E, H as for luce_rmsnorm_router
 * residual may be NULL only when T == 0.  Under programmatic launch the
 * previous kernel may write x and residual but neither w_router nor gamma.
 */
LUCE_API luce_status luce_add_rmsnorm_router(const float *x, const float *residual, float *x_sum,
                                             const float *gamma, float eps, const float *w_router, int T, int E,
                                             int H, float *xn, float *logits, void *stream);

/* ------------------------------------------------------------------------
 * luce_ep_mask / luce_add_f32 -- the two pieces of an expert-parallel split
 * of the step.  [PR826], the cluster runtime commit (each rank holds a share
 * of the routed experts, and the ranks sum their outputs every MoE layer) and
 * the review "moe_combine_masked_kernel indexes valid with an unchecked
 * (possibly -1) route id" (routes a rank does not own reach it as id -1).
 * A rank owning routed experts [e0, e1) masks the router's ids, runs
 * luce_moe_group, luce_moe_glu_pair and luce_moe_down_combine with the
 * masked ids (one rank also passes the shared expert), and the partial
 * outputs are summed.
 *
 * luce_ep_mask: ids_out[i] = ids[i] if e0 <= ids[i] < e1, else -1, for
 *   n int32 entries (ids_out may equal ids).  0 <= e0 <= e1.
 * luce_add_f32: out[i] = a[i] + b[i] (fp32, one rounding), n entries; out
 *   may equal a or b.
 */
LUCE_API luce_status luce_ep_mask(const int32_t *ids, int64_t n, int e0, int e1, int32_t *ids_out, void *stream);
LUCE_API luce_status luce_add_f32(const float *a, const float *b, float *out, int64_t n, void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_prep -- luce_route_topk, luce_quantize_q8_1 (K = H) and
 * luce_moe_group in ONE launch (one CTA) when T <= 32 and E <= 256, else the
 * three launches in that order.  Same arguments, outputs and results as the
 * three calls.  [PR826], commit "fused DS4.1 decode kernels": the verify
 * step's many short per-layer kernels are merged, among them the router's
 * selection and weights, the expert grouping and the q8_1 activation memo.
 */
LUCE_API luce_status luce_moe_prep(const float *logits, const float *bias, const float *x, int T, int E, int k,
                                   int H, int32_t *ids, float *weights, luce_block_q8_1 *xq, int32_t *counts,
                                   int32_t *offsets, int32_t *routes, void *stream);

/* ------------------------------------------------------------------------
 * luce_moe_layer -- one whole MoE FFN layer in ONE launch: the results of
 * luce_moe_prep, then luce_moe_glu_pair, then luce_moe_down_combine on the
 * same arguments, bit for bit (ids, weights, xq, counts, offsets, routes, h,
 * hq and out are all written).  [PR826], commits "fused DS4.1 decode
 * kernels" (select and weights, grouping, q8_1 memo), "RDNA4 Q8_0 gate/up
 * pair" and "fused routed combine and q8_1 inputs for the hybrid owners";
 * the single launch is this library's own.
 *
 *   logits [T][E] f32, bias [E] f32 or NULL, x [T][H] f32 (16-byte aligned);
 *   w_gate, w_up [E][I][H/32] and w_down [E][H][I/32] Q8_0 blocks;
 *   ws_gate, ws_up [I][H/32] and ws_down [H][I/32]: all three or none;
 *   clamp as in luce_moe_glu_pair; outputs as in the three calls.  h
 *   [T*k+T][I] f32 (16-byte aligned) is required: the launch keeps h there
 *   between its gate/up and down parts.
 *   workspace: workspace_bytes >= luce_moe_layer_workspace_bytes(T, k, H, I)
 *   bytes of device memory (16-byte aligned) owned by the caller, all zero
 *   before the first call.  Its first 8 bytes are a 64-bit count of
 *   device-wide barrier arrivals that only grows (no reset, so CUDA-graph
 *   replays need no host update); from byte 16 on it holds the y values
 *   [T*k+T][H] f32 of large layers between two barriers (contents need no
 *   initialisation).  The grid is always one CTA per SM, so calls of any
 *   shape may share one workspace on one device, one at a time (one stream
 *   or ordered streams); calls that may run at the same time need distinct
 *   workspaces.  If luce_get_fault reports LUCE_FAULT_DESYNC or
 *   LUCE_FAULT_TIMEOUT after this call, zero the first 8 bytes again before
 *   the next call.
 *
 * The grid is launched cooperatively (all CTAs resident at once) and every
 * CTA routes the tokens itself.  Two structures, chosen by the size of hq
 * ((T*k+T) * I/32 * 36 bytes):
 *   hq <= 24 KB (decode): each CTA takes an equal share of the 32-row gate/up
 *   groups (shared expert and routed experts) and quantizes the groups it
 *   computes; one device-wide barrier; each CTA then copies all of hq into
 *   shared memory, computes an equal share of the output rows of every
 *   expert and combines them itself.
 *   hq > 24 KB (verify, wide layers): each CTA takes a byte-balanced slice
 *   of the gate/up rows and stores h; barrier; each CTA quantizes an equal
 *   share of the q8_1 blocks of h; barrier; each CTA takes an equal share of
 *   the flat (expert, output row) list and writes y to the workspace;
 *   barrier; each CTA combines an equal share of the out elements.
 * Every barrier wait is bounded (LUCE_FAULT_TIMEOUT, LUCE_FAULT_DESYNC).
 * Supported: 1 <= T <= 8, T*k <= 64, E <= 256 (else LUCE_ERR_UNSUPPORTED,
 * and the three calls serve); H, I multiples of 256 up to 32768.  Argument
 * errors as in the three calls, plus a workspace too small or misaligned.
 * Not allowed inside a kernel that the caller runs concurrently with another
 * cooperative grid on the same device.
 */
LUCE_API size_t luce_moe_layer_workspace_bytes(int T, int k, int H, int I);
LUCE_API luce_status luce_moe_layer(const float *logits, const float *bias, const float *x,
                                    const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
                                    const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_gate,
                                    const luce_block_q8_0 *ws_up, const luce_block_q8_0 *ws_down, int T, int E, int k,
                                    int H, int I, float clamp, int32_t *ids, float *weights, luce_block_q8_1 *xq,
                                    int32_t *counts, int32_t *offsets, int32_t *routes, float *h,
                                    luce_block_q8_1 *hq, float *out, void *workspace, size_t workspace_bytes,
                                    void *stream);

/* ------------------------------------------------------------------------
 * luce_set_pdl -- process-wide switch (default 0 = off) for programmatic
 * dependent launch: each library kernel may then start before the previous
 * kernel on the stream has finished, run its prologue, and wait on the GPU
 * before it reads that kernel's results.  Kernels of other code never start
 * early (they do not signal), so expert weights written by any earlier
 * kernel are safe.  One extra rule holds while it is on:
 * luce_moe_down_combine reads ids, weights, offsets and routes before it
 * waits, and luce_moe_down_combine_q4k ids, weights and its weight rows, so
 * the call that produced them must not be the launch immediately before it
 * (in the order prep/group, glu_pair, down_combine, or route, glu_q4k,
 * down_combine_q4k, it never is).
 */
LUCE_API luce_status luce_set_pdl(int enable);

/* ------------------------------------------------------------------------
 * Diagnostics. */

/* Short English name of a status code (static storage). */
LUCE_API const char *luce_status_string(luce_status s);

/* Read and clear the device fault bits (LUCE_FAULT_*) raised by kernels on
 * the current device.  Synchronizes the device.  Returns LUCE_OK or
 * LUCE_ERR_CUDA; *bits receives the OR of all faults since the last call. */
LUCE_API luce_status luce_get_fault(unsigned int *bits);

/* Library version (major * 10000 + minor * 100 + patch). */
LUCE_API int luce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LUCE_MOE_H */
