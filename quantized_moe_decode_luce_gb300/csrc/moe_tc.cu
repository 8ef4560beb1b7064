// moe_tc.cu -- the routed-MoE FFN layer for many tokens (prefill) on the
// fifth-generation tensor cores: a grouped GEMM per expert for the gate/up
// pair and one for the down product, both with the pages' Q8_0 x q8_1 block
// arithmetic.  Reached through luce_moe_layer when T > 8.
//
// Pages cited by title: [PR826] = Lucebox PR #826 "feat(ds41): two-box
// expert-parallel serving".  Commit "fused DS4.1 decode kernels" routes wide
// quantized products over many rows to a matrix-core path, and commit
// "ROCmFP2 expert prefill on RDNA4 matrix cores" runs the routed-expert
// products of large batches as one grouped matrix product per expert; the
// arithmetic is that of commit "RDNA4 Q8_0 gate/up pair": per 32-value block
// b, the int32 sum isum_b = sum qw * qx, scaled by fp16(d_w) * fp16(d_x) and
// accumulated in fp32.  The tensor-core mapping below is this library's own.
//
// Exactness.  The tensor cores of this GPU have no int8 kind for tcgen05.mma,
// so the int8 codes go in as fp16 values: every code in [-127, 127] is an
// exact fp16 number, every product (at most 127^2) and every sum of the 32
// products of one block (at most 516,128 < 2^24) is an exact fp32 integer.
// Each 32-value block is accumulated into a tensor-memory region of its own
// (two K = 16 MMAs), so the MMA returns isum_b exactly, as a dp4a chain
// would; the CUDA cores then apply the block's two scales in fp32.
//
// Work items: (expert, 128 weight rows, up to 64 of the expert's tokens).
// Tokens are in expert-group order (the position p of a route in routes[]);
// the shared expert's tokens follow at p = T*k + t.  A persistent grid (one
// CTA per SM) takes items round-robin; each item streams its 128 rows over
// all K in stages of 8 blocks (272 bytes a row).
//
// CTA roles (11 warps):
//  * warp 8 -- TMA: per stage one 2D tile of each weight matrix (128 rows x
//    272 bytes, the Q8_0 rows seen as u16 elements, landing dense) and four
//    128-byte-swizzled tiles of the activation codes (fp16, the tensor core's
//    K-major layout), all completing on the stage's mbarrier; and an L2
//    prefetch of the weight tiles two stages ahead.
//  * warp 9 -- cp.async copies of the activation block scales ([block][token]).
//  * warp 10, one thread -- issues tcgen05.mma (A from tensor memory, B from
//    shared memory) and the tcgen05.commit arrivals.
//  * warps 0-7 -- lane quarter q = warp & 3 (rows 32q .. 32q+31, the tensor
//    memory lanes this warp may access), half h = warp >> 2.  They turn the
//    raw int8 codes of their rows into fp16 pairs in tensor memory
//    (tcgen05.st; the gate pair: half 0 converts gate, half 1 up; the down
//    product: half h converts the blocks of parity h), then read each block's
//    exact sums back (tcgen05.ld) and accumulate isum * (d_w * d_x) in
//    registers with packed fp32x2 multiply/FMA (half h takes the 16-token
//    chunks h and h + 2).  At the end of an item the gate pair forms
//    h = SwiGLU(g, u), stores h, its q8_1 blocks (each 32-row lane quarter is
//    one q8_1 block of h per token) and the fp16 codes and scales the down
//    product reads; the down product stores y.
// A warp converts block b while the sums of block b - 2 load from tensor
// memory, then applies their scales; so the MMAs of two blocks are in flight
// behind the scale work.  Every wait is bounded: on timeout the kernel raises
// LUCE_FAULT_TIMEOUT, the other roles leave at their next wait, and the CTA
// drains its copies and MMAs and frees its tensor memory before returning.
#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include <cuda.h> // CUtensorMap and its enums (the encoder is reached through the runtime's entry-point query)

#include "common.cuh"

LUCE_DEFINE_FAULT_WORD(luce_internal_fault_tc)

namespace {

using namespace luce;

constexpr int TM = 128;       // weight rows of one item (MMA M)
constexpr int TN = 64;        // tokens of one item at most (four 16-token chunks)
constexpr int SKB = 8;        // 32-value blocks per stage
constexpr int RA = 3;          // A slots in tensor memory
constexpr int RD = 3;          // D slots in tensor memory
constexpr int LAG = 2;         // a warp converts block b, then applies the scales of block b - LAG
constexpr int EPQ = 2;                   // convert + epilogue warps per tensor-memory lane quarter
constexpr int EPI_WARPS = 4 * EPQ;       // warps 0 .. EPI_WARPS-1
constexpr int CPW = 4 / EPQ;             // 16-token chunks per epilogue warp
constexpr int PROD_WARP0 = EPI_WARPS;    // producers: tensor-map tiles, activation block scales
constexpr int MMA_WARP = EPI_WARPS + 2;
constexpr int TC_THREADS = (EPI_WARPS + 3) * 32;
static_assert(EPQ == 2 || EPQ == 4, "chunk and conversion split");
constexpr int FULL_ARRIVALS = 33; // a stage is full: the tiles' arrival + bytes, 32 lanes of scale copies
// A slot reuse needs no wait of its own: a warp converts block b after it applied the
// scales of block b - LAG - 1 = b - RA, whose MMAs (the last readers of that slot) it
// waited for then.
static_assert(RA == LAG + 1 && LAG < RD, "slot reuse ordering");
constexpr uint32_t TMEM_COLS = 512;
constexpr int RAW_ROW = SKB * Q8_0_BYTES; // 272: one row's stage of raw Q8_0 blocks
constexpr int RAW_MAT = TM * RAW_ROW;     // 34,816
constexpr int B_ATOM = TN * 128;          // one 64-value K column of the activation tile (1024-aligned)
constexpr int B_BYTES = 4 * B_ATOM;       // 256 K values of TN tokens, fp16
constexpr int DX_BYTES = 2048;            // activation block scales [block][token] (SKB * TN * 4, padded)
constexpr int PF_STAGES = 2;              // weight tiles are prefetched into L2 this many stages ahead
static_assert(B_ATOM % 1024 == 0 && SKB * TN * 4 <= DX_BYTES, "stage layout");

template <int NMAT> struct Stage {
    static constexpr int b_off = 0; // 1024-aligned (swizzle atoms)
    static constexpr int raw_off = B_BYTES;
    static constexpr int dx_off = raw_off + NMAT * RAW_MAT;
    static constexpr int bytes = dx_off + DX_BYTES;
    static constexpr int count = NMAT == 2 ? 2 : 3;
    static_assert(bytes % 1024 == 0, "stages keep the swizzle atoms 1024-byte aligned");
};

// Tensor memory columns: A slots first (16 columns = 32 fp16 codes of a row
// per matrix), then D slots (TN columns = TN tokens per matrix).
constexpr int A_COLS = RA * 32;
__device__ __forceinline__ uint32_t acol(int slot, int m) { return (uint32_t)(slot * 32 + 16 * m); }
__device__ __forceinline__ uint32_t dcol(int slot, int m) { return (uint32_t)(A_COLS + slot * 2 * TN + TN * m); }
static_assert(A_COLS + RD * 2 * TN <= (int)TMEM_COLS, "tensor memory budget");

struct TcItem {
    int e;  // expert, or -1: the shared expert
    int m0; // first weight row
    int p0; // first token position
    int n;  // tokens (1 .. TN)
};

struct TcArgs {
    // tensor maps (2D tiles, copied by the TMA unit):
    //  tm_w[m] / tm_ws[m]: Q8_0 rows of matrix m (routed: E*M rows; shared: M rows) seen as
    //    u16 elements, nbK*17 to a row; box = 136 elements (8 blocks, 272 bytes) x 128 rows
    //  tm_b: activation codes fp16 [P][K]; box = 64 values (128 bytes) x 64 rows, 128-byte swizzle
    CUtensorMap tm_w[2], tm_ws[2], tm_b;
    const float *bscale;  // activation block scales [P][nbK]
    const TcItem *items;
    const int *nitems;
    int M, nbK;
    // gate/up epilogue
    const int32_t *routes;
    int Tk;
    float clamp;
    float *h;        // [Tk + T][M], route-slot order
    uint32_t *hq;    // [Tk + T][M/32] q8_1 blocks
    uint16_t *h16;   // [P][M] fp16 codes of hq, token-position order
    float *hscale;   // [P][M/32]
    // down epilogue
    float *y; // [P][M]
};

// ---------------------------------------------------------------------------
// tcgen05 / cp.async wrappers (sm_100 family PTX).
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// One arrival on `bar` once every cp.async this thread issued before has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Hint: bring one 2D tile of a tensor map into L2.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// One 2D tile of a tensor map into shared memory, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(16u >> 4) << 16;   // leading byte offset (unused by this layout)
    d |= (uint64_t)(1024u >> 4) << 32; // stride byte offset: next 8 rows
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp16 A and B, fp32 D, both K-major, M = 128.
__device__ __forceinline__ uint32_t mma_idesc(int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, bool acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)acc));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                     taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                 "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Four int8 codes -> two fp16 pairs holding the same integers: bias to
// unsigned (c + 128), place each byte under the exponent of 1024 (fp16
// 0x64XX = 1024 + XX), subtract 1152.  Exact for every code.
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// Bounded wait for the CTA's pipeline.  A wait that gives up raises the fault
// bit and the abort flag; every other wait of the CTA then gives up at its
// next poll.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    // each poll parks the thread in hardware until the phase completes (or a
    // suspend-time hint of 10 us runs out), so a waiting thread takes no issue
    // slots from the warps that work, and wakes at once
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 10000))
            return true;
        if (*abort_flag)
            return false;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicOr(&g_fault_word, LUCE_FAULT_TIMEOUT);
            return false;
        }
    }
}

// The same wait for a whole converged warp: every lane polls, and one poll
// instruction gives every lane the same answer, so the warp stays converged
// for the .sync.aligned tensor-memory instructions that follow.
__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int lane)
{
    (void)lane;
    const bool ok = tc_wait(bar, parity, abort_flag);
    __syncwarp();
    return ok;
}

// Block j of a row's stage sits at byte 34 j, inside the three 16-byte
// chunks starting at chunk (34 j) >> 4 (the row starts 16-byte aligned):
// its fp16 scale at byte o = 34 j - 16 ((34 j) >> 4) of that 48-byte window,
// its 32 codes at o + 2 .. o + 33.
template <int J> __device__ __forceinline__ uint32_t win_d16(const uint32_t (&W)[12])
{
    constexpr int o = 34 * J - 16 * ((34 * J) >> 4);
    return (o & 3) ? (W[o >> 2] >> 16) : (W[o >> 2] & 0xffffu);
}

template <int J> __device__ __forceinline__ void win_codes(const uint32_t (&W)[12], uint32_t (&c)[8])
{
    constexpr int o = 34 * J - 16 * ((34 * J) >> 4) + 2; // first code byte
    constexpr int w0 = o >> 2;
#pragma unroll
    for (int m = 0; m < 8; m++) {
        if constexpr ((o & 3) == 0)
            c[m] = W[w0 + m];
        else
            c[m] = __byte_perm(W[w0 + m], W[w0 + m + 1], 0x5432);
    }
}

template <int J> __device__ __forceinline__ void load_window(const uint8_t *row, uint32_t (&W)[12])
{
    constexpr int c0 = (34 * J) >> 4;
#pragma unroll
    for (int i = 0; i < 3; i++) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * (c0 + i));
        W[4 * i] = v.x;
        W[4 * i + 1] = v.y;
        W[4 * i + 2] = v.z;
        W[4 * i + 3] = v.w;
    }
}

// A ring position: slot index and phase parity, advanced one block at a time
// (no division by the ring size).
template <int R> struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next()
    {
        if (++slot == R) {
            slot = 0;
            phase ^= 1;
        }
    }
};

// The scales of one finished block, applied in two halves around the
// conversion of a later block so that the tensor-memory loads overlap it.
// begin: wait for the block's sums, start loading chunk c0 (matrix 0), read
// the block's weight scales.  finish: acc[cc][m][i] += isum * (d_w[m] *
// d_x[i]) for the chunks c = c0 + EPQ cc below nch (pairs of tokens in packed
// fp32 arithmetic; the chunks after the first are loaded here).
template <int NMAT> struct EpiBlock {
    uint32_t dv[NMAT][16];
    float dw[NMAT];
    const float *dxj;
    uint32_t dslot;
};

template <int NMAT>
__device__ __forceinline__ bool epi_begin(EpiBlock<NMAT> &eb, const uint8_t *stage, int rowoff, int j,
                                          const Ring<RD> &dr, uint64_t *dfull, uint32_t tl, int c0, int nch,
                                          volatile int *abort_flag)
{
    using S = Stage<NMAT>;
    if (!tc_wait(&dfull[dr.slot], dr.phase, abort_flag))
        return false;
    __syncwarp();
    tc_fence_after();
    eb.dslot = dr.slot;
    // (loaded whether or not chunk c0 holds tokens: no branch around the asm outputs, which
    // keeps them in registers; matrix 1 is loaded in epi_finish, so fewer registers are held)
    tmem_ld16(tl + dcol(dr.slot, 0) + 16 * c0, eb.dv[0]);
#pragma unroll
    for (int m = 0; m < NMAT; m++)
        eb.dw[m] =
            half_bits_to_float(*reinterpret_cast<const uint16_t *>(stage + rowoff + m * RAW_MAT + Q8_0_BYTES * j));
    eb.dxj = reinterpret_cast<const float *>(stage + S::dx_off) + j * TN;
    return true;
}

template <int NMAT>
__device__ __forceinline__ void epi_fma(float2 (&acc)[NMAT][8], const uint32_t (&dv)[NMAT][16], const float (&dw)[NMAT],
                                        const float *dx)
{
    const float4 *x4 = reinterpret_cast<const float4 *>(dx);
#pragma unroll
    for (int i4 = 0; i4 < 4; i4++) {
        const float4 x = x4[i4];
#pragma unroll
        for (int m = 0; m < NMAT; m++) {
            const float2 w2 = make_float2(dw[m], dw[m]);
            const float2 s0 = __fmul2_rn(w2, make_float2(x.x, x.y));
            const float2 s1 = __fmul2_rn(w2, make_float2(x.z, x.w));
            acc[m][2 * i4] = __ffma2_rn(make_float2(__uint_as_float(dv[m][4 * i4]), __uint_as_float(dv[m][4 * i4 + 1])),
                                        s0, acc[m][2 * i4]);
            acc[m][2 * i4 + 1] = __ffma2_rn(
                make_float2(__uint_as_float(dv[m][4 * i4 + 2]), __uint_as_float(dv[m][4 * i4 + 3])), s1,
                acc[m][2 * i4 + 1]);
        }
    }
}

template <int NMAT>
__device__ __forceinline__ void epi_finish(float2 (&acc)[CPW][NMAT][8], EpiBlock<NMAT> &eb, uint32_t tl, int c0,
                                           int nch)
{
    if constexpr (NMAT == 2)
        tmem_ld16(tl + dcol(eb.dslot, 1) + 16 * c0, eb.dv[1]);
    tmem_wait_ld();
    if (c0 < nch)
        epi_fma<NMAT>(acc[0], eb.dv, eb.dw, eb.dxj + 16 * c0);
#pragma unroll
    for (int cc = 1; cc < CPW; cc++) {
        const int c = c0 + EPQ * cc;
        if (c < nch) {
            uint32_t dv[NMAT][16];
#pragma unroll
            for (int m = 0; m < NMAT; m++)
                tmem_ld16(tl + dcol(eb.dslot, m) + 16 * c, dv[m]);
            tmem_wait_ld();
            epi_fma<NMAT>(acc[cc], dv, eb.dw, eb.dxj + 16 * c);
        }
    }
}

// ---------------------------------------------------------------------------
template <int NMAT>
__global__ void __launch_bounds__(TC_THREADS, 1) k_moe_tc(const __grid_constant__ TcArgs a)
{
    using S = Stage<NMAT>;
    constexpr int NS = S::count;
    extern __shared__ uint8_t smraw[];
    __shared__ uint64_t full[NS], sfree[NS], afull[RA], dfull[RD], dfree[RD], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_word;
    volatile int *abort_flag = &abort_word;
    uint8_t *sm = smraw + ((1024u - (smem_addr(smraw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], FULL_ARRIVALS);
            mbar_init(&sfree[s], 1 + EPI_WARPS);
        }
        for (int i = 0; i < RA; i++)
            mbar_init(&afull[i], EPI_WARPS);
        for (int i = 0; i < RD; i++) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dfree[i], EPI_WARPS);
        }
        mbar_init(&drain, 1);
        abort_word = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    pdl_wait(); // items, activation codes and scales come from the previous launches
    const int nitems = *a.nitems;
    const int nst = a.nbK / SKB;

    if (warp == PROD_WARP0 || warp == PROD_WARP0 + 1) {
        // ------------------------------------------------------------ producers
        const int pw = warp - PROD_WARP0;
        uint32_t gs = 0;
        for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
            const TcItem item = a.items[it];
            const int npad = (item.n + 15) & ~15;
            for (int st = 0; st < nst; st++, gs++) {
                const int s = (int)(gs % NS);
                if (!tc_wait_warp(&sfree[s], ((gs / NS) & 1) ^ 1, abort_flag, lane))
                    goto out_prod;
                uint8_t *stg = sm + s * S::bytes;
                if (pw == 0) {
                    // the weight tiles of every matrix (128 rows x 8 blocks each) and the
                    // activation tile (64 token rows x 256 codes, four swizzled 64-code columns)
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(NMAT * RAW_MAT + B_BYTES));
                        const int wy = item.e >= 0 ? item.e * a.M + item.m0 : item.m0;
#pragma unroll
                        for (int m = 0; m < NMAT; m++)
                            tma_load_2d(stg + S::raw_off + m * RAW_MAT, item.e >= 0 ? &a.tm_w[m] : &a.tm_ws[m],
                                        st * (RAW_ROW / 2), wy, &full[s]);
#pragma unroll
                        for (int kc = 0; kc < 4; kc++)
                            tma_load_2d(stg + S::b_off + kc * B_ATOM, &a.tm_b, st * (SKB * QK) + kc * 64, item.p0,
                                        &full[s]);
                        // the weight tiles PF_STAGES ahead (this item's, else the CTA's next item's) into L2
                        int pst = st + PF_STAGES, pit = it;
                        if (pst >= nst) {
                            pst -= nst;
                            pit += gridDim.x;
                        }
                        if (pit < nitems) {
                            const TcItem pi = pit == it ? item : a.items[pit];
                            const int py = pi.e >= 0 ? pi.e * a.M + pi.m0 : pi.m0;
#pragma unroll
                            for (int m = 0; m < NMAT; m++)
                                tma_prefetch_2d(pi.e >= 0 ? &a.tm_w[m] : &a.tm_ws[m], pst * (RAW_ROW / 2), py);
                        }
                    }
                } else {
                    // block scales, transposed to [block][token]
                    for (int i = lane; i < npad * SKB; i += 32) {
                        const int row = i >> 3, j = i & 7;
                        const int src = item.p0 + min(row, item.n - 1);
                        cp_async4(stg + S::dx_off + (j * TN + row) * 4, a.bscale + (size_t)src * a.nbK + st * SKB + j);
                    }
                    cp_async_arrive(&full[s]);
                }
            }
        }
    out_prod:
        cp_async_wait_all();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            Ring<NS> sr;
            Ring<RA> ar;
            Ring<RD> dr;
            for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
                const TcItem item = a.items[it];
                const int npad = (item.n + 15) & ~15;
                const uint32_t idesc = mma_idesc(npad);
                for (int st = 0; st < nst; st++, sr.next()) {
                    if (!tc_wait(&full[sr.slot], sr.phase, abort_flag))
                        goto out_mma;
                    // the scale copies landed through the generic proxy; the tensor core reads through the async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    const uint32_t bbase = smem_addr(sm + sr.slot * S::bytes + S::b_off);
                    for (int j = 0; j < SKB; j++, ar.next(), dr.next()) {
                        if (!tc_wait(&afull[ar.slot], ar.phase, abort_flag))
                            goto out_mma;
                        if (!tc_wait(&dfree[dr.slot], dr.phase ^ 1, abort_flag))
                            goto out_mma;
                        tc_fence_after();
#pragma unroll
                        for (int sk = 0; sk < 2; sk++) {
                            const uint64_t bd = sw128_desc(bbase + (j >> 1) * B_ATOM + (j & 1) * 64 + sk * 32);
#pragma unroll
                            for (int m = 0; m < NMAT; m++)
                                mma_ts(tmem + dcol(dr.slot, m), tmem + acol(ar.slot, m) + 8 * sk, bd, idesc, sk > 0);
                        }
                        mma_commit(&dfull[dr.slot]);
                    }
                    mma_commit(&sfree[sr.slot]);
                }
            }
        out_mma:
            // every MMA issued has completed before the tensor memory is freed
            mma_commit(&drain);
            (void)tc_wait(&drain, 0, abort_flag);
        }
        __syncwarp();
    } else if (warp < EPI_WARPS) {
        // ------------------------------------------------------------ convert + epilogue
        const int q = warp & 3, w2 = warp >> 2;
        const int r = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        // conversion: the gate pair -- matrix w2 & 1, the blocks j with
        // j mod (EPQ / 2) = w2 >> 1; the down product -- the blocks j with
        // j mod EPQ = w2.  Epilogue: token chunks w2 + EPQ cc.
        const int mc = NMAT == 2 ? (w2 & 1) : 0;
        const int rowoff = S::raw_off + r * RAW_ROW; // this row in a stage's raw weights
        Ring<NS> sr;                                 // stage being converted
        Ring<RA> ar;                                 // A slot being written
        Ring<RD> dr;                                 // D slot whose scales are applied next
        for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
            const TcItem item = a.items[it];
            const int nch = (item.n + 15) >> 4;
            float2 acc[CPW][NMAT][8];
#pragma unroll
            for (int cc = 0; cc < CPW; cc++)
#pragma unroll
                for (int m = 0; m < NMAT; m++)
#pragma unroll
                    for (int i = 0; i < 8; i++)
                        acc[cc][m][i] = make_float2(0.0f, 0.0f);

            for (int st = 0; st < nst; st++, sr.next()) {
                const int s = (int)sr.slot;
                const int sprev = s == 0 ? NS - 1 : s - 1;
                if (!tc_wait_warp(&full[s], sr.phase, abort_flag, lane))
                    goto out_epi;
                const uint8_t *myrow = sm + s * S::bytes + rowoff + mc * RAW_MAT;
                // one block J: start the scales of the block LAG back (same stage for
                // J >= LAG, else the previous one), convert block J into A slot ar
                // while those loads run, finish the scales, then one fence for both
                // arrivals; the template arguments need J as a constant, hence a macro
#define LUCE_TC_STEP(J)                                                                                              \
    {                                                                                                                \
        const bool has_epi = (J) >= LAG || st > 0;                                                                   \
        const int es = (J) >= LAG ? s : sprev;                                                                       \
        constexpr int ej = ((J) + SKB - LAG) % SKB;                                                                  \
        EpiBlock<NMAT> eb;                                                                                           \
        if (has_epi && !epi_begin<NMAT>(eb, sm + es * S::bytes, rowoff, ej, dr, dfull, tl, w2, nch, abort_flag))     \
            goto out_epi;                                                                                            \
        const bool conv = NMAT == 2 ? (((J) & (EPQ / 2 - 1)) == (w2 >> 1)) : (((J) % EPQ) == w2);                  \
        if (conv) {                                                                                                  \
            uint32_t W[12], cw[8];                                                                                   \
            load_window<J>(myrow, W);                                                                                \
            win_codes<J>(W, cw);                                                                                     \
            _Pragma("unroll") for (int hf = 0; hf < 2; hf++) {                                                      \
                uint32_t hv[8];                                                                                      \
                _Pragma("unroll") for (int m = 0; m < 4; m++)                                                       \
                    codes_to_half2(cw[4 * hf + m], hv[2 * m], hv[2 * m + 1]);                                        \
                tmem_st8(tl + acol(ar.slot, mc) + 8 * hf, hv);                                                       \
            }                                                                                                        \
        }                                                                                                            \
        if (has_epi)                                                                                                 \
            epi_finish<NMAT>(acc, eb, tl, w2, nch);                                                                  \
        if (conv)                                                                                                    \
            tmem_wait_st();                                                                                          \
        tc_fence_before();                                                                                           \
        __syncwarp();                                                                                                \
        if (lane == 0) {                                                                                             \
            mbar_arrive(&afull[ar.slot]);                                                                            \
            if (has_epi) {                                                                                           \
                mbar_arrive(&dfree[dr.slot]);                                                                        \
                if (ej == SKB - 1)                                                                                   \
                    mbar_arrive(&sfree[es]);                                                                         \
            }                                                                                                        \
        }                                                                                                            \
        ar.next();                                                                                                   \
        if (has_epi)                                                                                                 \
            dr.next();                                                                                               \
    }
                LUCE_TC_STEP(0)
                LUCE_TC_STEP(1)
                LUCE_TC_STEP(2)
                LUCE_TC_STEP(3)
                LUCE_TC_STEP(4)
                LUCE_TC_STEP(5)
                LUCE_TC_STEP(6)
                LUCE_TC_STEP(7)
#undef LUCE_TC_STEP
            }
            {
                // the item's last LAG blocks (indices SKB - LAG .. SKB - 1 of its last stage)
                const int s = sr.slot == 0 ? NS - 1 : (int)sr.slot - 1;
#pragma unroll
                for (int k2 = LAG; k2 >= 1; k2--) {
                    EpiBlock<NMAT> eb;
                    if (!epi_begin<NMAT>(eb, sm + s * S::bytes, rowoff, SKB - k2, dr, dfull, tl, w2, nch, abort_flag))
                        goto out_epi;
                    epi_finish<NMAT>(acc, eb, tl, w2, nch);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&dfree[dr.slot]);
                        if (k2 == 1)
                            mbar_arrive(&sfree[s]);
                    }
                    dr.next();
                }
            }

            // ---- the item's results: chunks w2 + EPQ cc of the tokens, rows 32q .. 32q+31
#pragma unroll
            for (int cc = 0; cc < CPW; cc++) {
                const int c = w2 + EPQ * cc;
                if (c >= nch)
                    continue;
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int n = 16 * c + i;
                    if (n >= item.n)
                        continue; // (not break: the loop stays unrolled and acc stays in registers)
                    const int p = item.p0 + n;
                    const int col = item.m0 + r;
                    if constexpr (NMAT == 2) {
                        const float g = (i & 1) ? acc[cc][0][i >> 1].y : acc[cc][0][i >> 1].x;
                        const float u = (i & 1) ? acc[cc][1][i >> 1].y : acc[cc][1][i >> 1].x;
                        const float hv = swiglu(g, u, a.clamp);
                        const int row = item.e >= 0 ? a.routes[p] : p;
                        a.h[(size_t)row * a.M + col] = hv;
                        const int blk = (item.m0 >> 5) + q;
                        int code;
                        uint32_t d16;
                        quantize_q8_1_warp(hv, a.hq + ((size_t)row * (a.M / QK) + blk) * Q8_1_WORDS, lane, code, d16);
                        a.h16[(size_t)p * a.M + col] = __half_as_ushort(__int2half_rn(code));
                        if (lane == 0)
                            a.hscale[(size_t)p * (a.M / QK) + blk] = half_bits_to_float(d16);
                    } else {
                        a.y[(size_t)p * a.M + col] = (i & 1) ? acc[cc][0][i >> 1].y : acc[cc][0][i >> 1].x;
                    }
                }
            }
        }
    out_epi:;
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == MMA_WARP)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

// ---------------------------------------------------------------------------
// Work lists (one CTA): the shared expert's token slices first, then every
// routed expert's; an expert with n tokens takes ceil(n / 64) slices of equal
// size.  Each (expert, slice) gives one item per 128 weight rows, slices of
// the same rows next to each other so that they meet in L2.
constexpr int ITEM_THREADS = 1024;

__global__ void __launch_bounds__(ITEM_THREADS) k_tc_items(const int32_t *counts, const int32_t *offsets, int E, int T,
                                                            int k, int has_shared, int mt_glu, int mt_down,
                                                            TcItem *glu_items, TcItem *down_items, int *nitems)
{
    __shared__ int scan[ITEM_THREADS];
    __shared__ int base_shared;
    pdl_wait();
    const int tid = threadIdx.x;
    const int Tk = T * k;
    // slices of expert e = tid (several experts per thread when E > ITEM_THREADS is not allowed by the host)
    const int e = tid;
    const int n = e < E ? counts[e] : 0;
    const int ns = (n + TN - 1) / TN;
    scan[tid] = ns;
    __syncthreads();
    for (int off = 1; off < ITEM_THREADS; off <<= 1) {
        const int v = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    const int sh_ns = has_shared ? (T + TN - 1) / TN : 0;
    if (tid == 0)
        base_shared = sh_ns;
    __syncthreads();
    const int total = base_shared + scan[ITEM_THREADS - 1];
    const int first = base_shared + scan[tid] - ns; // this expert's first slice
    auto emit = [&](int ex, int slice0, int nsl, int cnt, int p_base) {
        for (int j = 0; j < nsl; j++) {
            const int a0 = (int)((long long)j * cnt / nsl), a1 = (int)((long long)(j + 1) * cnt / nsl);
            for (int m = 0; m < mt_glu; m++)
                glu_items[(size_t)slice0 * mt_glu + (size_t)m * nsl + j] = TcItem{ex, m * TM, p_base + a0, a1 - a0};
            for (int m = 0; m < mt_down; m++)
                down_items[(size_t)slice0 * mt_down + (size_t)m * nsl + j] = TcItem{ex, m * TM, p_base + a0, a1 - a0};
        }
    };
    if (e < E && ns > 0)
        emit(e, first, ns, n, offsets[e]);
    if (tid == 0 && sh_ns > 0)
        emit(-1, 0, sh_ns, T, Tk);
    if (tid == 0) {
        nitems[0] = total * mt_glu;
        nitems[1] = total * mt_down;
    }
}

// Activation codes as fp16 in token-position order, their block scales, and
// the position of every kept route (inv[r] = p).
__global__ void __launch_bounds__(128) k_tc_gather(const uint32_t *xq, const int32_t *offsets, const int32_t *routes,
                                                    int E, int T, int k, int nbH, uint16_t *x16, float *xscale,
                                                    int32_t *inv)
{
    pdl_wait();
    const int p = blockIdx.x;
    const int Tk = T * k;
    int t;
    if (p < Tk) {
        if (p >= offsets[E])
            return;
        const int rr = routes[p];
        t = rr / k;
        if (threadIdx.x == 0)
            inv[rr] = p;
    } else {
        t = p - Tk;
    }
    for (int b = threadIdx.x; b < nbH; b += blockDim.x) {
        const uint32_t *src = xq + ((size_t)t * nbH + b) * Q8_1_WORDS;
        uint32_t hv[16];
#pragma unroll
        for (int m = 0; m < 8; m++)
            codes_to_half2(src[1 + m], hv[2 * m], hv[2 * m + 1]);
        uint4 *dst = reinterpret_cast<uint4 *>(x16 + (size_t)p * nbH * QK + (size_t)b * QK);
#pragma unroll
        for (int i = 0; i < 4; i++)
            dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
        xscale[(size_t)p * nbH + b] = half_bits_to_float(src[0]);
    }
}

// out[t][n] = sum over kept slots j, in order, of fl(w[t][j] * y[inv[t k + j]][n]),
// each product and sum rounded, then + y of the shared expert.
__global__ void __launch_bounds__(256) k_tc_combine(const float *y, const int32_t *ids, const float *weights,
                                                     const int32_t *inv, int T, int k, int E, int H, int has_shared,
                                                     float *out)
{
    pdl_wait();
    const int t = blockIdx.y;
    const int n = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (n >= H)
        return;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j = 0; j < k; j++) {
        const int e = ids[t * k + j];
        if (e < 0 || e >= E)
            continue;
        const float w = weights[t * k + j];
        const float4 v = *reinterpret_cast<const float4 *>(y + (size_t)inv[t * k + j] * H + n);
        acc.x = __fadd_rn(acc.x, __fmul_rn(w, v.x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(w, v.y));
        acc.z = __fadd_rn(acc.z, __fmul_rn(w, v.z));
        acc.w = __fadd_rn(acc.w, __fmul_rn(w, v.w));
    }
    if (has_shared) {
        const float4 v = *reinterpret_cast<const float4 *>(y + ((size_t)T * k + t) * H + n);
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
    }
    float *o = out + (size_t)t * H + n; // (out is only 4-byte aligned)
    o[0] = acc.x;
    o[1] = acc.y;
    o[2] = acc.z;
    o[3] = acc.w;
}

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the workspace start, 256-aligned).
struct TcLayout {
    size_t x16, xscale, h16, hscale, y, inv, glu_items, down_items, nitems, total;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool tc_layout(int T, int k, int H, int I, TcLayout &L)
{
    if (T <= 0 || k <= 0 || H <= 0 || I <= 0)
        return false;
    const size_t Tk = (size_t)T * k, P = Tk + T;
    const size_t slices = Tk + Tk / TN + 1 + ((size_t)T + TN - 1) / TN;
    size_t o = 16; // the barrier count of the small-T kernels
    o = align256(o);
    L.x16 = o;
    o = align256(o + P * H * 2);
    L.xscale = o;
    o = align256(o + P * (H / QK) * 4);
    L.h16 = o;
    o = align256(o + P * I * 2);
    L.hscale = o;
    o = align256(o + P * (I / QK) * 4);
    L.y = o;
    o = align256(o + P * H * 4);
    L.inv = o;
    o = align256(o + Tk * 4);
    L.glu_items = o;
    o = align256(o + slices * (I / TM) * sizeof(TcItem));
    L.down_items = o;
    o = align256(o + slices * (H / TM) * sizeof(TcItem));
    L.nitems = o;
    o = align256(o + 2 * sizeof(int));
    L.total = o;
    return true;
}

// cuTensorMapEncodeTiled, from the driver through the runtime's entry-point
// query (no link against the driver library); looked up once.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// Q8_0 rows [rows][nbK][34] as u16 elements; box = 8 blocks x 128 rows, no swizzle.
bool map_q8_0_rows(CUtensorMap *m, const void *base, long long rows, int nbK)
{
    EncodeTiledFn f = encode_tiled();
    if (!f || !base)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)nbK * (Q8_0_BYTES / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)nbK * Q8_0_BYTES};
    const cuuint32_t box[2] = {RAW_ROW / 2, TM};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 codes [P][K]; box = 64 codes (128 bytes) x 64 rows, 128-byte swizzle (rows past P read as zero).
bool map_codes(CUtensorMap *m, const void *base, long long rows, int K)
{
    EncodeTiledFn f = encode_tiled();
    if (!f || !base)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, TN};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAT> luce_status launch_tc(const TcArgs &args, cudaStream_t stream)
{
    static luce_host::SmemLimit limit;
    const size_t smem = (size_t)Stage<NMAT>::count * Stage<NMAT>::bytes + 1024;
    auto kern = k_moe_tc<NMAT>;
    if (limit.raise(kern, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_UNSUPPORTED;
    }
    const luce_status st = luce_host::launch(kern, dim3(luce_host::sm_count()), dim3(TC_THREADS), smem, stream, args);
    if (st != LUCE_OK)
        limit.forget();
    return st;
}

} // namespace

extern "C" __attribute__((visibility("hidden"))) size_t luce_internal_moe_layer_tc_bytes(int T, int k, int H, int I)
{
    TcLayout L;
    return tc_layout(T, k, H, I, L) ? L.total : 0;
}

// The prefill layer: route + quantize + group (the separate operations), then
// the work lists and gathered activation codes, the gate/up grouped GEMM, the
// down grouped GEMM and the combine.  Arguments were validated by
// luce_moe_layer; this adds the limits of this path.
extern "C" __attribute__((visibility("hidden"))) luce_status luce_internal_moe_layer_tc(
    const float *logits, const float *bias, const float *x, const luce_block_q8_0 *w_gate, const luce_block_q8_0 *w_up,
    const luce_block_q8_0 *w_down, const luce_block_q8_0 *ws_gate, const luce_block_q8_0 *ws_up,
    const luce_block_q8_0 *ws_down, int T, int E, int k, int H, int I, float clamp, int32_t *ids, float *weights,
    luce_block_q8_1 *xq, int32_t *counts, int32_t *offsets, int32_t *routes, float *h, luce_block_q8_1 *hq,
    float *out, void *workspace, size_t workspace_bytes, void *stream)
{
    using namespace luce_host;
    TcLayout L;
    if (E > ITEM_THREADS || T > 65535 || H % 256 != 0 || I % 256 != 0 || !tc_layout(T, k, H, I, L))
        return LUCE_ERR_UNSUPPORTED;
    if (workspace_bytes < L.total)
        return LUCE_ERR_INVALID_ARG;
    if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) || (ws_gate && !aligned(ws_gate, 16)) ||
        (ws_up && !aligned(ws_up, 16)) || (ws_down && !aligned(ws_down, 16)))
        return LUCE_ERR_INVALID_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *x16 = reinterpret_cast<uint16_t *>(ws + L.x16);
    float *xscale = reinterpret_cast<float *>(ws + L.xscale);
    uint16_t *h16 = reinterpret_cast<uint16_t *>(ws + L.h16);
    float *hscale = reinterpret_cast<float *>(ws + L.hscale);
    float *y = reinterpret_cast<float *>(ws + L.y);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    TcItem *glu_items = reinterpret_cast<TcItem *>(ws + L.glu_items);
    TcItem *down_items = reinterpret_cast<TcItem *>(ws + L.down_items);
    int *nitems = reinterpret_cast<int *>(ws + L.nitems);
    const bool shared = ws_gate != nullptr;
    const int Tk = T * k;
    cudaStream_t st = as_stream(stream);

    // the tensor maps first: a failure launches nothing
    const long long P = (long long)Tk + T;
    TcArgs g{}, d{};
    if (!map_q8_0_rows(&g.tm_w[0], w_gate, (long long)E * I, H / QK) ||
        !map_q8_0_rows(&g.tm_w[1], w_up, (long long)E * I, H / QK) || !map_codes(&g.tm_b, x16, P, H) ||
        !map_q8_0_rows(&d.tm_w[0], w_down, (long long)E * H, I / QK) || !map_codes(&d.tm_b, h16, P, I) ||
        (shared && (!map_q8_0_rows(&g.tm_ws[0], ws_gate, I, H / QK) || !map_q8_0_rows(&g.tm_ws[1], ws_up, I, H / QK) ||
                    !map_q8_0_rows(&d.tm_ws[0], ws_down, H, I / QK))))
        return LUCE_ERR_CUDA;
    g.bscale = xscale;
    g.items = glu_items;
    g.nitems = nitems;
    g.M = I;
    g.nbK = H / QK;
    g.routes = routes;
    g.Tk = Tk;
    g.clamp = clamp;
    g.h = h;
    g.hq = reinterpret_cast<uint32_t *>(hq);
    g.h16 = h16;
    g.hscale = hscale;
    d.bscale = hscale;
    d.items = down_items;
    d.nitems = nitems + 1;
    d.M = H;
    d.nbK = I / QK;
    d.y = y;

    luce_status s = luce_route_topk(logits, bias, T, E, k, ids, weights, stream);
    if (s == LUCE_OK)
        s = luce_quantize_q8_1(x, T, H, xq, stream);
    if (s == LUCE_OK)
        s = luce_moe_group(ids, T, k, E, counts, offsets, routes, stream);
    if (s == LUCE_OK)
        s = launch(k_tc_items, dim3(1), dim3(ITEM_THREADS), 0, st, (const int32_t *)counts, (const int32_t *)offsets, E,
                   T, k, (int)shared, I / TM, H / TM, glu_items, down_items, nitems);
    if (s == LUCE_OK)
        s = launch(k_tc_gather, dim3((unsigned)(Tk + (shared ? T : 0))), dim3(128), 0, st,
                   reinterpret_cast<const uint32_t *>(xq), (const int32_t *)offsets, (const int32_t *)routes, E, T, k,
                   H / QK, x16, xscale, inv);
    if (s == LUCE_OK)
        s = launch_tc<2>(g, st);
    if (s == LUCE_OK)
        s = launch_tc<1>(d, st);
    if (s != LUCE_OK)
        return s;
    return launch(k_tc_combine, dim3((unsigned)((H / 4 + 255) / 256), (unsigned)T), dim3(256), 0, st, (const float *)y,
                  (const int32_t *)ids, (const float *)weights, (const int32_t *)inv, T, k, E, H, (int)shared, out);
}
