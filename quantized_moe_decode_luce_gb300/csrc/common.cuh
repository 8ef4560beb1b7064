// common.cuh -- device helpers shared by the kernels of libluce_moe.
//
// Q8_0 / q8_1 block access, the q8_1 quantization rule, the warp reductions,
// and the Blackwell asynchronous-copy machinery (mbarrier + cp.async.bulk)
// used to stream expert weights into shared memory.  Host-side argument
// checks live here too.
#pragma once

#include <math.h>

#include <atomic>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/luce_moe.h"

namespace luce {

constexpr int QK = 32;
constexpr int Q8_0_BYTES = 34;
constexpr int Q8_1_BYTES = 36;
constexpr int Q8_1_WORDS = 9;
// A bounded device wait gives up after this many nanoseconds and raises
// LUCE_FAULT_TIMEOUT.  Nothing in a correct run waits longer than a few
// microseconds; the bound only keeps a defect from hanging the GPU.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// ---------------------------------------------------------------------------
// Fault word: one per translation unit (no relocatable device code).  Each
// .cu file defines it through LUCE_DEFINE_FAULT_WORD and exposes a host
// reader; luce_get_fault ORs them.
#define LUCE_DEFINE_FAULT_WORD(name)                                                    \
    static __device__ unsigned int g_fault_word;                                        \
    extern "C" __attribute__((visibility("hidden"))) cudaError_t name(unsigned int *bits) \
    {                                                                                   \
        unsigned int v = 0, zero = 0;                                                   \
        cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v));              \
        if (e == cudaSuccess)                                                           \
            e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero));                  \
        *bits |= v;                                                                     \
        return e;                                                                       \
    }

// ---------------------------------------------------------------------------
// Small device helpers.
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16)
{
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// q8_1 rule for one block held by a warp (lane i holds x[i]):
// amax = max|x|, d = amax / 127 (IEEE), q = roundf(x / d) (0 if amax == 0),
// d16 = fp16(d), s16 = fp16(d * sum(q)) (round to nearest even).  The block
// is written as 9 little-endian 32-bit words: d16 | s16 << 16, then the
// codes four to a word.
// The lane's code and the block's fp16 d bits are returned in q_out and
// d16_out (every lane gets d16).
__device__ __forceinline__ void quantize_q8_1_warp(float x, uint32_t *__restrict__ out_words, int lane, int &q_out,
                                                   uint32_t &d16_out)
{
    const float amax = warp_max(fabsf(x));
    const float d = __fdiv_rn(amax, 127.0f);
    // an all-zero block divides its zeros by 1 (codes 0) instead of by 0
    const int q = (int)roundf(__fdiv_rn(x, amax == 0.0f ? 1.0f : d));
    const int sum = warp_sum_i(q);
    uint32_t byte = (uint32_t)(q & 0xff);
    uint32_t w = byte;
    w |= __shfl_down_sync(0xffffffffu, byte, 1) << 8;
    w |= __shfl_down_sync(0xffffffffu, byte, 2) << 16;
    w |= __shfl_down_sync(0xffffffffu, byte, 3) << 24;
    const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
    if (lane == 0) {
        const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sum)));
        out_words[0] = d16 | (s16 << 16);
    }
    if ((lane & 3) == 0)
        out_words[1 + (lane >> 2)] = w;
    q_out = q;
    d16_out = d16;
}

__device__ __forceinline__ void quantize_q8_1_warp(float x, uint32_t *__restrict__ out_words, int lane)
{
    int q;
    uint32_t d16;
    quantize_q8_1_warp(x, out_words, lane, q, d16);
}

// ---------------------------------------------------------------------------
// A Q8_0 block b of a row that starts 16-byte aligned sits at byte 34*b:
// 4-byte aligned for even b, 2 bytes off for odd b.  Nine aligned words
// starting at (34*b) & ~3 hold the whole block either way; a funnel shift
// by 16 (even b) or 32 (odd b) extracts the scale and the eight code words.
struct Q80Block {
    float d;
    uint32_t q[8];
};

__device__ __forceinline__ void load_q8_0_smem(const uint8_t *row, int b, Q80Block &blk)
{
    const uint32_t *p = reinterpret_cast<const uint32_t *>(row + ((34 * b) & ~3));
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; i++)
        w[i] = p[i];
    const uint32_t sh = (b & 1) ? 32u : 16u;
    blk.d = half_bits_to_float(__funnelshift_rc(w[0], w[1], sh - 16u));
#pragma unroll
    for (int i = 0; i < 8; i++)
        blk.q[i] = __funnelshift_rc(w[i], w[i + 1], sh);
}

// The same block read through a shared-memory address (explicit ld.shared,
// whatever the compiler can prove about a generic pointer).
__device__ __forceinline__ uint32_t lds32(uint32_t saddr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ void load_q8_0_sh(uint32_t row_saddr, int b, Q80Block &blk)
{
    const uint32_t p = row_saddr + ((34u * (uint32_t)b) & ~3u);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; i++)
        w[i] = lds32(p + 4u * i);
    const uint32_t sh = (b & 1) ? 32u : 16u;
    blk.d = half_bits_to_float(__funnelshift_rc(w[0], w[1], sh - 16u));
#pragma unroll
    for (int i = 0; i < 8; i++)
        blk.q[i] = __funnelshift_rc(w[i], w[i + 1], sh);
}

// Which blocks of a Q8_0 row (nb blocks of 34 B, row start 16-byte aligned)
// a lane takes, and in which order it accumulates them.  34-byte blocks b and
// b + 32 start 272 words, i.e. 16 banks, apart, and so do two consecutive rows
// of 32 blocks; the mappings below make each 32-bit load instruction of a warp
// touch 32 distinct shared-memory banks.
//   ROWMAP_PAIRS (nb % 64 == 0): 32 lanes per row; block j of lane L is
//     64 (j >> 1) + 16 (j & 1) + (L & 15) + 32 (L >> 4).
//   ROWMAP_TWO_ROWS (nb == 32, where used): 16 lanes per row, lanes 16..31 on
//     the next row; block j of lane L is (L & 15) + 16 j.
//   ROWMAP_PLAIN (otherwise): 32 lanes per row; block j of lane L is L + 32 j.
// Every kernel that reduces the same row uses the same mapping, so partial
// sums are formed and added in the same order everywhere.
enum RowMap { ROWMAP_PLAIN = 0, ROWMAP_TWO_ROWS = 1, ROWMAP_PAIRS = 2 };

__device__ __forceinline__ int rowmap_blocks(int map, int nb, int lane)
{
    return map == ROWMAP_PAIRS ? (nb >> 5) : map == ROWMAP_TWO_ROWS ? 2 : ((nb - lane + 31) >> 5);
}

__device__ __forceinline__ int rowmap_block(int map, int lane, int j)
{
    return map == ROWMAP_PAIRS ? ((j >> 1) << 6) + ((j & 1) << 4) + (lane & 15) + ((lane >> 4) << 5)
         : map == ROWMAP_TWO_ROWS ? (lane & 15) + (j << 4)
                                  : lane + (j << 5);
}

// Sum over each half-warp (lanes 0..15 and 16..31 separately): the tree of
// warp_sum without its first level.
__device__ __forceinline__ float half_warp_sum(float v)
{
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// q8_1 block from global memory (read-only path, L1-cached): scale + codes.
struct Q81Block {
    float d;
    int q[8];
};

__device__ __forceinline__ void load_q8_1_global(const uint32_t *__restrict__ words, Q81Block &blk)
{
    blk.d = half_bits_to_float(__ldg(words));
#pragma unroll
    for (int i = 0; i < 8; i++)
        blk.q[i] = (int)__ldg(words + 1 + i);
}

// q8_1 block through a generic pointer (shared or global memory).
__device__ __forceinline__ void load_q8_1_any(const uint32_t *words, Q81Block &blk)
{
    blk.d = half_bits_to_float(words[0]);
#pragma unroll
    for (int i = 0; i < 8; i++)
        blk.q[i] = (int)words[1 + i];
}

// q8_1 block through a shared-memory address.
__device__ __forceinline__ void load_q8_1_sh(uint32_t saddr, Q81Block &blk)
{
    blk.d = half_bits_to_float(lds32(saddr));
#pragma unroll
    for (int i = 0; i < 8; i++)
        blk.q[i] = (int)lds32(saddr + 4u + 4u * i);
}

// Exact int32 block sum of 32 int8 products; four independent partial sums
// keep the dp4a dependency chains short (integer addition is exact, so the
// result does not depend on the grouping).
__device__ __forceinline__ int dot_q8_block(const uint32_t (&w)[8], const int (&x)[8])
{
    int s0 = __dp4a((int)w[0], x[0], 0);
    int s1 = __dp4a((int)w[1], x[1], 0);
    int s2 = __dp4a((int)w[2], x[2], 0);
    int s3 = __dp4a((int)w[3], x[3], 0);
    s0 = __dp4a((int)w[4], x[4], s0);
    s1 = __dp4a((int)w[5], x[5], s1);
    s2 = __dp4a((int)w[6], x[6], s2);
    s3 = __dp4a((int)w[7], x[7], s3);
    return (s0 + s1) + (s2 + s3);
}

// SwiGLU of the pages: silu(g) * u, optionally silu(min(g, L)) * clamp(u, -L, L).
__device__ __forceinline__ float swiglu(float g, float u, float clamp)
{
    if (clamp > 0.0f) {
        g = fminf(g, clamp);
        u = fminf(fmaxf(u, -clamp), clamp);
    }
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(s, u);
}

// Router weights of one token, held by a warp: lane j < k holds sel0 = the
// unbiased logit of slot j, lane j + 32 < k holds sel1 = that of slot j + 32.
// w[j] = exp(l_j - m) / sum_i exp(l_i - m), m the largest selected logit; the
// sum is a butterfly over the lanes, so every lane sees the same value.
__device__ __forceinline__ void route_softmax_warp(float sel0, float sel1, int k, float *w_out, int lane)
{
    const bool has0 = lane < k, has1 = lane + 32 < k;
    float m = has0 ? sel0 : -INFINITY;
    if (has1)
        m = fmaxf(m, sel1);
    m = warp_max(m);
    const float e0 = has0 ? expf(__fsub_rn(sel0, m)) : 0.0f;
    const float e1 = has1 ? expf(__fsub_rn(sel1, m)) : 0.0f;
    const float den = warp_sum(__fadd_rn(e0, e1));
    if (has0)
        w_out[lane] = __fdiv_rn(e0, den);
    if (has1)
        w_out[lane + 32] = __fdiv_rn(e1, den);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk asynchronous copy (global -> shared), sm_90+ PTX.
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_count(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Whether the phase of `parity` has completed, without waiting.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps (up to `ns` nanoseconds) until it completes, instead of spinning and
// taking issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most WAIT_LIMIT_NS.
// Returns false (and the caller raises LUCE_FAULT_TIMEOUT) if it gave up.
// Between polls the thread sleeps (backing off from 32 to 256 ns), so that
// waiting warps leave the issue slots to the warps that work.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    uint32_t ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity))
            return true;
        ns = ns < 256 ? 2 * ns : 256;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS)
            return false;
    }
}

// L2 policy for weights that are streamed once per step.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to shared memory, completing `bytes` of transaction on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch.  pdl_wait: wait until the kernels this grid
// depends on have completed and their writes are visible (a no-op when the
// grid was launched without the programmatic attribute).  pdl_trigger: let
// the next kernel on the stream start its prologue early.  Every kernel of
// this library triggers only after its own pdl_wait, so a kernel that starts
// early may still read the outputs of kernels two launches back.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Prefetch `bytes` (multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier among `nthreads` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrival at a named barrier without waiting (the threads that wait there
// with named_barrier see the memory writes made before the arrival).
__device__ __forceinline__ void named_barrier_arrive(int id, int nthreads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_line_l2(const void *p)
{
    asm volatile("prefetch.L2 [%0];" ::"l"(p));
}

} // namespace luce

// ---------------------------------------------------------------------------
// Host-side helpers.
namespace luce_host {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Maps the last launch error to a status (and clears it).
inline luce_status launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? LUCE_OK : LUCE_ERR_CUDA;
}

// Number of SMs of the current device (cached per device, thread-safe).
int sm_count();

// The dynamic shared memory limit of ONE kernel (one object per kernel or
// template instance), raised on the current device to at least `bytes` by
// the first call that needs it; later calls make no attribute call.  Safe
// from several host threads.  After a failed launch the caller calls forget()
// so that the next call sets the attribute again (a reset context starts
// from the default limit).
struct SmemLimit {
    std::atomic<size_t> set[64];
    std::mutex mu;
    template <class Kernel> cudaError_t raise(Kernel kern, size_t bytes)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 0 || dev >= 64)
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (set[dev].load(std::memory_order_acquire) >= bytes)
            return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu);
        if (set[dev].load(std::memory_order_relaxed) >= bytes)
            return cudaSuccess;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e == cudaSuccess)
            set[dev].store(bytes, std::memory_order_release);
        return e;
    }
    void forget()
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64)
            set[dev].store(0, std::memory_order_release);
    }
};

// Launch-shape parameters of the streaming kernels.  The values here are the
// library's choices; they are plain data so that a tuning build can sweep
// them, and every setting computes the same result.
// Defaults measured on GB300 with the 43-layer decode stack (graph + PDL):
// two gate/up CTAs per SM with ~108 KB rings leave room for the down kernel's
// CTAs to start early and stream their weights while the gate/up kernel runs.
struct Tuning {
    int glu_part_kb = 36;     // target bytes of one part (RU gate + RU up rows)
    int glu_budget_kb = 108;  // shared-memory ring budget per CTA
    int glu_cps = 2;          // gate/up CTAs per SM
    int glu_xs = 1;           // stage activation rows in shared memory
    int glu_prefetch = 1;     // warm L2 with the shared expert before waiting
    int down_budget_kb = 100; // down/combine ring budget per CTA
    int down_stage = 1;       // stage the tile's activation rows in shared memory
    int evict_first = 1;      // stream weights with the L2 evict-first policy
    int layer_part_kb = 36;   // whole-layer kernel: bytes of one gate/up part
    int layer_budget_kb = 222; // whole-layer kernel: shared memory per CTA
    int layer_cps = 1;        // whole-layer kernel: CTAs per SM
    int layer_prefetch = 1;   // whole-layer kernel: warm L2 with the shared expert
    int layer_dsplit = 0;     // whole-layer kernel: down rows split by weight across CTAs
    int layer_psleep = 64;    // whole-layer kernel: producer back-off in ns while the ring is full
    int layer_down_early = 0; // whole-layer kernel: down stages before every gate/up part is requested
    int layer_hq_bulk = 1;    // whole-layer kernel: stage a shared hq with one bulk copy
};
extern Tuning g_tuning;

// Whether kernels are launched with the programmatic-dependent-launch
// attribute (luce_set_pdl; process-wide, default off).
bool pdl_enabled();

// Launch configuration with the PDL attribute when enabled.  `attr` must
// hold one entry.
inline void make_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr, dim3 grid, dim3 block, size_t smem,
                        cudaStream_t stream)
{
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int n = 0;
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        n++;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
}

// Launch `kern` with cudaLaunchKernelEx, with the PDL attribute when enabled.
template <typename... KArgs, typename... Args>
luce_status launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    make_config(cfg, attr, grid, block, smem, stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return LUCE_ERR_CUDA;
    }
    return LUCE_OK;
}

} // namespace luce_host
