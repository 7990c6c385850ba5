// Shared device helpers of the DynaSpec GB300 kernels: bf16 unpacking, streaming loads,
// the Philox4x32-10 generator, warp reductions and the softmax/argmax partial-state
// algebra every head and verify reduction uses.
#pragma once
#include <utility>

#include <atomic>
#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/dynaspec.h"

namespace ds {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------------------
// bf16 <-> fp32.  A bf16 value is the top half of an fp32 word, so widening is a shift.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// fp32 -> bf16, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f)
{
    const uint32_t u = __float_as_uint(f);
    return uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

// Dot product of 8 packed bf16 (one 16-byte vector) with 8 fp32 values.
__device__ __forceinline__ float dot8(uint4 w, const float4 x0, const float4 x1, float acc)
{
    acc = fmaf(bf16lo(w.x), x0.x, acc);
    acc = fmaf(bf16hi(w.x), x0.y, acc);
    acc = fmaf(bf16lo(w.y), x0.z, acc);
    acc = fmaf(bf16hi(w.y), x0.w, acc);
    acc = fmaf(bf16lo(w.z), x1.x, acc);
    acc = fmaf(bf16hi(w.z), x1.y, acc);
    acc = fmaf(bf16lo(w.w), x1.z, acc);
    acc = fmaf(bf16hi(w.w), x1.w, acc);
    return acc;
}

// 16-byte streaming load through the non-coherent path, not kept in L1: LM-head rows are
// read once per draft position.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// L2 eviction-priority policies for loads that carry a cache hint: data read once (the LM-head
// rows of one draft position) is marked to leave L2 first; data every draft position reads
// again (the router weights) is marked to leave it last.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ld_stream with an L2 cache policy.
__device__ __forceinline__ uint4 ld_stream_hint(const uint4 *p, uint64_t policy)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(policy));
    return r;
}

__device__ __forceinline__ void set_status(int32_t *st, int32_t bit)
{
    if (st) atomicOr(st, bit);
}

// ---------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of two 32x32->64 multiplies whose halves are crossed over the four
// lanes and xored with a key that advances by the golden-ratio Weyl constants.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        // one widening multiply per product gives both halves
        const uint64_t p0 = uint64_t(0xD2511F53u) * c.x;
        const uint64_t p1 = uint64_t(0xCD9E8D57u) * c.z;
        const uint32_t lo0 = uint32_t(p0), hi0 = uint32_t(p0 >> 32);
        const uint32_t lo1 = uint32_t(p1), hi1 = uint32_t(p1 >> 32);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// -log(u) for u in (0, 1) on the hardware base-2 logarithm, kept accurate near u = 1, where the
// result is small: there t = 1 - u is exact and -log(1 - t) = t + t^2/2 + t^3/3 + ... is summed
// to t^7/7 (t < 1/16: truncation below 1e-9 relative).  Elsewhere the base-2 logarithm's
// relative error (about 2^-22) carries over to the result.
__device__ __forceinline__ float neg_log_unit(float u)
{
    const float t = 1.f - u;
    if (t < 0.0625f) {
        float p = 1.f / 7.f;
        p = fmaf(p, t, 1.f / 6.f);
        p = fmaf(p, t, 1.f / 5.f);
        p = fmaf(p, t, 1.f / 4.f);
        p = fmaf(p, t, 1.f / 3.f);
        p = fmaf(p, t, 1.f / 2.f);
        p = fmaf(p, t, 1.f);
        return p * t;
    }
    return -0.69314718055994531f * __log2f(u);
}

// Gumbel noise g = -log(-log u) of a 32-bit word w: u = (2 (w >> 9) + 1) 2^-24 in (0, 1).  The
// inner logarithm is neg_log_unit; the outer one's argument E = -log u lies in [6e-8, 17.4],
// where the base-2 logarithm's absolute error (about 2^-22 ln 2) is far below the noise scale.
__device__ __forceinline__ float gumbel_from_word(uint32_t x)
{
    const float u = float(2u * (x >> 9) + 1u) * 5.9604644775390625e-8f;   // * 2^-24, exact
    return -0.69314718055994531f * __log2f(neg_log_unit(u));
}

// The Philox block of shortlist entries 4q .. 4q+3 (j >> 2 = q; entry j's index in its list) for
// draft position `pos`, head row `row`: counter (q, pos, row, 0), key = the seed's halves.
__device__ __forceinline__ uint4 gumbel_block(uint64_t seed, uint32_t q, uint32_t pos, uint32_t row)
{
    return philox4x32_10(make_uint4(q, pos, row, 0u), uint32_t(seed), uint32_t(seed >> 32));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &w, uint32_t i)
{
    return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// Gumbel noise of shortlist entry j: word j & 3 of its block.
__device__ __forceinline__ float gumbel(uint64_t seed, uint32_t j, uint32_t pos, uint32_t row)
{
    return gumbel_from_word(word_of(gumbel_block(seed, j >> 2, pos, row), j & 3u));
}

// ---------------------------------------------------------------------------------------
// Softmax statistics + sampled argmax as one associative partial state.
//   m, s : running max of x and sum of exp(x - m)  (x = logit / Te)
//   key  : best sampling key so far, v its full-vocabulary id, j its index in the list;
//          a larger key wins, equal keys go to the lower v.
// ---------------------------------------------------------------------------------------
struct Stat {
    float m, s, key;
    int v, j;
};

__device__ __forceinline__ Stat stat_empty() { return Stat{-INFINITY, 0.f, -INFINITY, -1, -1}; }

__device__ __forceinline__ void stat_add(Stat &a, float x, float key, int v, int j)
{
    if (x > a.m) {
        a.s = a.s * __expf(a.m - x) + 1.f;   // exp(-inf) = 0 for the first element
        a.m = x;
    } else {
        a.s += __expf(x - a.m);
    }
    if (key > a.key || (key == a.key && (unsigned)v < (unsigned)a.v)) {
        a.key = key; a.v = v; a.j = j;
    }
}

// The states of each group of kWidth lanes (a power of two <= 32) reduced to one, which every
// lane of the group ends with.  Two passes of exchanges whose steps are all commutative, so both
// lanes of a pair compute the same value and the result does not depend on timing: the maximum
// and the best key first, then the sums, each scaled once to the common maximum (one
// exponential per lane instead of two per merge level).
template <int kWidth = 32>
__device__ __forceinline__ Stat stat_reduce_lanes(const Stat &mine)
{
    float m = mine.m, key = mine.key;
    int v = mine.v, j = mine.j;
#pragma unroll
    for (int o = 1; o < kWidth; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float k2 = __shfl_xor_sync(0xFFFFFFFFu, key, o);
        const int v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int j2 = __shfl_xor_sync(0xFFFFFFFFu, j, o);
        m = fmaxf(m, m2);
        const bool take = v2 >= 0 && (v < 0 || k2 > key || (k2 == key && v2 < v));
        key = take ? k2 : key;
        v = take ? v2 : v;
        j = take ? j2 : j;
    }
    float s = mine.m == -INFINITY ? 0.f : mine.s * __expf(mine.m - m);
#pragma unroll
    for (int o = 1; o < kWidth; o <<= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return Stat{m, s, key, v, j};
}

// n states (in registers) merged in index order into one: the maximum and the best key, then
// the sums scaled to the maximum (independent exponentials), added in index order.
template <int n>
__device__ __forceinline__ Stat stat_merge_n(const Stat (&q)[n])
{
    Stat r = q[0];
#pragma unroll
    for (int f = 1; f < n; ++f) {
        r.m = fmaxf(r.m, q[f].m);
        const bool take = q[f].v >= 0 && (r.v < 0 || q[f].key > r.key || (q[f].key == r.key && q[f].v < r.v));
        r.key = take ? q[f].key : r.key;
        r.v = take ? q[f].v : r.v;
        r.j = take ? q[f].j : r.j;
    }
    float s = 0.f;
#pragma unroll
    for (int f = 0; f < n; ++f) s += q[f].m == -INFINITY ? 0.f : q[f].s * __expf(q[f].m - r.m);
    r.s = s;
    return r;
}


__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

__device__ __forceinline__ Stat ld_stat(const Stat *p)
{
    const volatile Stat *q = (const volatile Stat *)p;
    return Stat{q->m, q->s, q->key, q->v, q->j};
}

__device__ __forceinline__ void st_stat(Stat *p, const Stat &a)
{
    volatile Stat *q = (volatile Stat *)p;
    q->m = a.m; q->s = a.s; q->key = a.key; q->v = a.v; q->j = a.j;
}

// Atomic add with acquire and release semantics at GPU scope: the calling thread's earlier
// memory operations (and, through a barrier before it, those of its block) are ordered before
// the add, and the values other threads released by their adds on the same counter are visible
// to what the caller does after it.  No separate fence is needed on either side.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *counter, unsigned x)
{
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(prev) : "l"(counter), "r"(x) : "memory");
    return prev;
}

// "Am I the last block of this group to finish?"  Every block calls it once, after its
// results are stored; the returning `true` block may read all of them.  The barrier before
// the add orders the block's stores before thread 0's release; the last block's acquire, and
// the barrier after it, make every block's stores visible to all of its threads.  The last
// block resets the counter; the next launch sees the reset (kernel boundary).
__device__ __forceinline__ bool last_block_done(unsigned *counter, unsigned nblocks)
{
    __shared__ bool is_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        is_last = atom_add_acq_rel_gpu(counter, 1u) == nblocks - 1;
        if (is_last) *counter = 0u;
    }
    __syncthreads();
    return is_last;
}

// ---------------------------------------------------------------------------------------
// mbarrier primitives.  Every wait is bounded: a wait that runs
// past its budget returns false and the caller records DS_DEV_TIMEOUT and winds down.
// ---------------------------------------------------------------------------------------
constexpr long long kWaitBudgetCycles = 2000000000LL;    // about one second at 2 GHz

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

// Programmatic dependent launch.  A kernel launched with the programmatic-serialization
// attribute (launch_pdl) may begin while the kernel before it in the stream still runs, once
// every block of that kernel has called pdl_allow (or exited); its blocks then call pdl_wait,
// which returns when the earlier kernel has completed and its writes are visible (at once for
// a kernel launched without the attribute).  Only launch latency is hidden: nothing is read
// before pdl_wait.
__device__ __forceinline__ void pdl_allow() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Fetch the 128-byte line holding p into L2 (a hint: nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

}  // namespace ds

// ---------------------------------------------------------------------------------------
// Host-side helpers
// ---------------------------------------------------------------------------------------
#define DS_TRY_LAUNCH()                                                 \
    do {                                                                \
        if (cudaPeekAtLastError() != cudaSuccess) {                     \
            (void)cudaGetLastError();                                   \
            return DS_ERR_CUDA;                                         \
        }                                                               \
    } while (0)

namespace ds {
// A named NVTX range around a library call's host side: a profiler that collects NVTX shows
// each stage's launches under the call's name.  Without such a tool attached it costs a check.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Budget (SM clock cycles) of the kernels' bounded pipeline waits, process-wide; set by
// ds_set_wait_budget (tests make it tiny to see a wait give up), kWaitBudgetCycles otherwise.
inline std::atomic<long long> &wait_budget_cell()
{
    static std::atomic<long long> cell{kWaitBudgetCycles};
    return cell;
}
inline long long wait_budget() { return wait_budget_cell().load(std::memory_order_relaxed); }

// Multiprocessors of the current device, looked up once per device: grids are sized from it, so a
// process driving GPUs of different sizes (or two host threads on different devices) gets each
// device's own count.  A racing first lookup stores the same value twice, which is harmless.
// 0 if the device cannot be named or queried.
inline int sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per device
// (the attribute belongs to the device, so a process driving several GPUs sets it on each).
// `done` holds one bit per device already set; concurrent first calls may both set it, which is
// harmless.  False if the device cannot be named or the call fails.
template <class K>
inline bool smem_limit_once(K kernel, size_t bytes, std::atomic<unsigned long long> &done)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) != cudaSuccess)
        return false;
    done.fetch_or(bit, std::memory_order_release);
    return true;
}
}  // namespace ds
