// Gathered-row GEMM on the 5th-generation tensor cores (tcgen05, accumulator in tensor memory).
//
//   out[u][r] = sum_k A[row(u)][k] * Bop[r][k]      u < n_rows (a list of rows of A), r < R
//
// A is a row-major bf16 matrix whose rows are picked through a list (the union of the
// shortlists for the gathered head, or simply 0..n-1 for the router layers); Bop holds the R
// bf16 vectors every picked row is scored against.  A policy object (`Ep`) names the picked
// rows and consumes finished accumulator columns, so the same kernel serves the head (which
// scatters logits into per-list positions) and the router layers (bias, activation, dense
// output).  Accumulation is fp32 in tensor memory.
//
// Work: tiles of 128 picked rows (the MMA's M side) x all R vectors (N = 16*MT, zero padded) x
// the full depth d, each tile swept in k-stages of kCols columns.  The (tile, k-stage) units,
// in tile order, are split into equal contiguous ranges, one per CTA of a persistent grid (a
// stream-K split), so every SM streams the same number of A bytes whatever the list size; a
// tile whose stages fall into several CTAs is finished by the last of them, which adds the
// parts in k order (so results do not depend on timing).
//
// Per CTA the work is split between warp roles that meet only at mbarriers (no CTA-wide
// barrier inside the main loop):
//   * producers (8 warps) copy each stage into one of kStages shared-memory slots with
//     cp.async, every thread a fixed 16-byte column chunk of a fixed set of rows, and arrive
//     on the slot's `full` barrier when their copies land (cp.async.mbarrier.arrive);
//   * one thread issues the stage's MMAs (M=128, N=16*MT, K=16 each) into one of two tensor-
//     memory accumulators and commits them to the slot's `empty` barrier, and at a tile's end
//     to the accumulator's `full` barrier;
//   * epilogue warps (8) read a finished accumulator with tcgen05.ld, release it, and hand
//     the values to the policy while the next tile is being multiplied into the other one.
// A slot holds the 128 A rows and the N B rows for its columns in the 128-byte-swizzled
// K-major layout the MMA descriptors describe (8-row x 128-byte atoms, 16-byte chunk c of row
// r at c ^ (r & 7)).
//
// Every pipeline wait on an mbarrier is bounded (the budget comes from the host) and also gives
// up when another role has failed; a wait that gives up sets DS_DEV_TIMEOUT.  Producers leave
// no copy in flight, the MMA thread waits for its own MMAs to finish whatever happened to the
// pipeline (bounded by the full default budget), and the tensor memory is freed after a final
// barrier.
#pragma once
#include "common.cuh"

namespace ds {
namespace tc {

constexpr int kRows = 128;                  // A rows per tile (MMA M)
constexpr int kThreads = 544;               // 8 epilogue warps, 8 producer warps, 1 MMA warp
constexpr int kMaxGrid = 160;               // CTAs of one launch (<= SMs in use)

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// MT = N / 16 for R vectors: 16, 32, 48, 64, 80 or 128 columns.
__host__ __device__ constexpr int mt_for(int R)
{
    return R <= 16 ? 1 : R <= 32 ? 2 : R <= 48 ? 3 : R <= 64 ? 4 : R <= 80 ? 5 : 8;
}

template <int MT> struct Cfg {
    static constexpr int N = 16 * MT;
    static constexpr int kAtoms = MT >= 8 ? 1 : 2;             // 64-column atoms per stage
    static constexpr int kCols = kAtoms * 64;                  // columns of d per stage
    static constexpr int kABytes = kAtoms * kRows * 128;       // A part of a stage
    static constexpr int kBBytes = kAtoms * N * 128;           // B part of a stage
    static constexpr int kStageBytes = kABytes + kBBytes;
    // as many slots as fit, except three at N = 80, which measured faster than the four that fit
    // (the bytes in flight do not set the pace from three slots up)
    static constexpr int kStages = MT == 5 ? 3 : cmin(8, (220 * 1024) / kStageBytes);
    // two accumulators of N columns (the epilogue drains one while the MMAs fill the other)
    static constexpr int kTmemCols = 2 * N <= 32 ? 32 : 2 * N <= 64 ? 64 : 2 * N <= 128 ? 128 : 256;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 /* align */;
    static_assert(kStages >= 3, "the pipeline needs three slots");
    static_assert(kSmem + 2560 <= 232448, "dynamic + static shared memory per CTA");
};

// Bytes of the partial-tile buffer a launch with `grid` CTAs and R vectors needs (two 128 x N
// fp32 parts per CTA: its first and its last tile).
inline size_t parts_bytes(int R, int grid)
{
    return size_t(2) * size_t(grid) * kRows * size_t(16 * mt_for(R)) * sizeof(float);
}

struct Operands {
    const uint16_t *A;       // [*, d] bf16, rows picked by the policy
    const uint16_t *B;       // [R, d] bf16
    int d, R;
    int32_t *status;
    long long wait_budget;   // cycles a pipeline wait may take before it gives up
};

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes));
}
// Wait until every cp.async this thread issued has landed.  The producers never commit groups
// (their copies complete through cp.async.mbarrier.arrive), and wait_all commits the pending
// ones before waiting, so it covers them; a bare wait_group would not.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);             // start address
    d |= uint64_t(1) << 16;                             // leading byte offset (unused, K-major SW128)
    d |= uint64_t((1024u >> 4) & 0x3FFFu) << 32;        // stride byte offset: next 8-row group
    d |= uint64_t(1) << 46;                             // descriptor version
    d |= uint64_t(2) << 61;                             // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Policy interface (all device, const):
//   int n_rows()                          picked rows (read once per CTA)
//   void pick(int u, int &v, int &c)      A row of list entry u (-1: none) and a tag c
//   void col_info(int r, int &i, long long &l)  per-vector values the epilogue keeps in smem
//   int row_aux(int v)                    per-row value loaded at the tile's epilogue
//   State                                 per-thread epilogue state, value-initialised
//   void emit(st, x[16], cb, v, c, aux, s_i, s_l)  accumulator row of A row v, columns cb..cb+15
//   void finish(st)                       called once by every thread of every CTA at the end
//                                         (also by CTAs without work), e.g. to fold st
// NoState is the State of policies that keep none.
struct NoState {};
// Warp roles.  Warps 0-7: epilogue (warp w reads TMEM lanes 32(w%4) .. +31 = A rows of the
// tile, and every other 16-column group starting at 16(w/4)).  Warps 8-15: producers (256
// threads of cp.async).  Warp 16: TMEM owner and MMA issuer (one thread).
constexpr int kEpiWarps = 8;
constexpr int kProdBase = 256;                  // first producer thread
constexpr int kProducers = 256;
constexpr int kMmaWarp = 16;
static_assert(kThreads == kProdBase + kProducers + 32, "warp roles");

// Wait for a phase of an mbarrier, giving up after `budget` cycles or when another role failed.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, unsigned parity, volatile int *fail, long long budget)
{
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (*fail) return false;
        if (clock64() - t0 > budget) return false;
    }
    return true;
}

// Wait for this thread's own asynchronous work to finish before its resources are released: a
// failure elsewhere does not end this wait, and its budget is the full default one whatever the
// pipeline budget is.
__device__ __forceinline__ bool wait_drain(uint64_t *bar, unsigned parity)
{
    const long long t0 = clock64();
    while (!mbar_test(bar, parity))
        if (clock64() - t0 > kWaitBudgetCycles) return false;
    return true;
}

// Arrive on `bar` once all of this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" :: "n"(kEpiWarps * 32) : "memory"); }

template <int MT, class Ep>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(Operands op, Ep ep, float *__restrict__ parts, unsigned *__restrict__ tile_cnt)
{
    using C = Cfg<MT>;
    constexpr int STG = C::kStages;
    constexpr int CPR = C::kAtoms * 8;                         // 16-byte chunks per row per stage
    constexpr int RPP = kProducers / CPR;                      // rows per pass of the producers
    constexpr int APASS = kRows / RPP;                         // A-row passes per stage
    constexpr int BPASS = (C::N + RPP - 1) / RPP;              // B-row passes per stage
    static_assert(kRows % RPP == 0 && RPP % 8 == 0, "row passes share their swizzle phase");
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[STG], empty[STG], acc_full[2], acc_empty[2], mma_idle;
    __shared__ int32_t s_ci[C::N];
    __shared__ long long s_cl[C::N];
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail, s_last, s_stop;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = op.d, R = op.R;
    const int nU = ep.n_rows();
    const int ntiles = (nU + kRows - 1) / kRows;
    const int nks = (d + C::kCols - 1) / C::kCols;             // stages per tile
    const long long total = 1LL * ntiles * nks;                // < 2^31 by the host's limits
    const int grid = gridDim.x, bid = blockIdx.x;
    const int g0 = int(total * bid / grid), g1 = int(total * (bid + 1) / grid);
    typename Ep::State est{};
    if (g0 >= g1) { ep.finish(est); return; }                  // uniform: no stage for this CTA
    constexpr uint32_t idesc = umma_idesc_bf16(kRows, C::N);
    // the CTA whose range holds unit i, the first tile of CTA c, and the owner of the unit
    // after CTA c's range (CTAs with empty ranges own nothing)
    auto cta_of = [&](long long i) { return int(((i + 1) * grid - 1) / total); };
    auto first_tile = [&](int c) { return int((total * c / grid) / nks); };
    auto next_owner = [&](int c) { return cta_of(total * (c + 1) / grid); };

    if (tid == 0) {
        for (int i = 0; i < STG; ++i) { mbar_init(&full[i], kProducers); mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], kEpiWarps); }
        mbar_init(&mma_idle, 1);
        mbar_fence_init();
        s_fail = 0;
    }
    for (int r = tid; r < C::N; r += kThreads) {
        int ci = -1;
        long long cl = 0;
        if (r < R) ep.col_info(r, ci, cl);
        s_ci[r] = ci;
        s_cl[r] = cl;
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(uint32_t(C::kTmemCols)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = s_tmem;
    volatile int *fail = &s_fail;
    const uint32_t smem0 = smem_u32(sm);

    if (tid >= kProdBase && tid < kProdBase + kProducers) {
        // ---------------- producers: fill slot li % STG with stage i, then arrive on full[]
        const int p = tid - kProdBase;
        const int ch = p % CPR, prow = p / CPR;
        const int coff = (ch >> 3) * 64 + (ch & 7) * 8;        // column of the chunk inside a stage
        const uint32_t dst0 = uint32_t((ch >> 3) * (kRows * 128) + prow * 128 + (((ch & 7) ^ (prow & 7)) << 4));
        const uint32_t bdst0 = uint32_t((ch >> 3) * (C::N * 128) + prow * 128 + (((ch & 7) ^ (prow & 7)) << 4));
        const uint16_t *bsrc[BPASS];
#pragma unroll
        for (int j = 0; j < BPASS; ++j) {
            const int r = prow + RPP * j;
            bsrc[j] = r < R ? op.B + size_t(r) * d + coff : nullptr;
        }
        const uint16_t *asrc[APASS];
        int t = g0 / nks, ks = g0 - t * nks, slot = 0, use = 0, cur_t = -1;
        for (int i = g0; i < g1; ++i) {
            if (use > 0 && !wait_phase(&empty[slot], unsigned(use - 1) & 1u, fail, op.wait_budget)) {
                s_fail = 1;
                set_status(op.status, DS_DEV_TIMEOUT);
                break;
            }
            if (t != cur_t) {                                  // this thread's rows of tile t
#pragma unroll
                for (int j = 0; j < APASS; ++j) {
                    const int u = t * kRows + prow + RPP * j;
                    int v = -1, c = -1;
                    if (u < nU) ep.pick(u, v, c);
                    asrc[j] = v >= 0 ? op.A + size_t(v) * d + coff : nullptr;
                }
                cur_t = t;
            }
            const int k0 = ks * C::kCols;
            const bool kin = k0 + coff < d;
            const uint32_t As = smem0 + uint32_t(slot * C::kStageBytes);
            const uint32_t Bs = As + C::kABytes;
#pragma unroll
            for (int j = 0; j < APASS; ++j) {
                const bool ok = kin && asrc[j] != nullptr;
                cp_async16(As + dst0 + uint32_t(j * RPP * 128), ok ? asrc[j] + k0 : op.A, ok ? 16 : 0);
            }
#pragma unroll
            for (int j = 0; j < BPASS; ++j) {
                if (prow + RPP * j < C::N) {
                    const bool ok = kin && bsrc[j] != nullptr;
                    cp_async16(Bs + bdst0 + uint32_t(j * RPP * 128), ok ? bsrc[j] + k0 : op.B, ok ? 16 : 0);
                }
            }
            cp_async_arrive(&full[slot]);
            if (++slot == STG) { slot = 0; ++use; }
            if (++ks == nks) { ks = 0; ++t; }
        }
        cp_async_wait_all();                                   // nothing in flight when the role ends
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer: one thread
        if (lane == 0) {
            int t = g0 / nks, ks = g0 - t * nks, slot = 0, use = 0, lt = 0;
            bool ok = true;
            for (int i = g0; i < g1 && ok; ++i) {
                const bool first = ks == 0 || i == g0;
                const int buf = lt & 1;
                if (first && lt >= 2 && !wait_phase(&acc_empty[buf], unsigned(lt / 2 - 1) & 1u, fail, op.wait_budget)) { ok = false; break; }
                if (!wait_phase(&full[slot], unsigned(use) & 1u, fail, op.wait_budget)) { ok = false; break; }
                proxy_fence_async();                           // the producers' copies -> tensor core
                fence_after();
                const uint32_t As = smem0 + uint32_t(slot * C::kStageBytes);
                const uint32_t Bs = As + C::kABytes;
                const uint32_t dacc = tmem + uint32_t(buf * C::N);
#pragma unroll
                for (int at = 0; at < C::kAtoms; ++at) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = umma_desc_sw128(As + at * (kRows * 128) + kk * 32);
                        const uint64_t bd = umma_desc_sw128(Bs + at * (C::N * 128) + kk * 32);
                        mma(dacc, ad, bd, idesc, (first && at == 0 && kk == 0) ? 0u : 1u);
                    }
                }
                commit(&empty[slot]);                          // frees the slot when these MMAs finish
                if (ks == nks - 1 || i == g1 - 1) { commit(&acc_full[buf]); ++lt; }
                if (++slot == STG) { slot = 0; ++use; }
                if (++ks == nks) { ks = 0; ++t; }
            }
            if (!ok) { s_fail = 1; set_status(op.status, DS_DEV_TIMEOUT); }
            commit(&mma_idle);                                 // completes once every MMA issued has
            // the tensor memory is freed below, so this waits for the MMAs in flight even when
            // the pipeline has failed
            if (!wait_drain(&mma_idle, 0u)) { s_fail = 1; set_status(op.status, DS_DEV_TIMEOUT); }
        }
        __syncwarp();
    } else if (warp < kEpiWarps) {
        // ---------------- epilogue: a TMEM lane quarter and every other 16-column group per warp
        const int wq = warp & 3;
        const int row = wq * 32 + lane;                        // A row of the tile
        const uint32_t tq = tmem + (uint32_t(wq * 32) << 16);
        const int cb0 = (warp >> 2) * 16;
        int t = g0 / nks, lt = 0;
        for (;;) {
            const long long ts = 1LL * t * nks;                // the tile's first unit
            if (ts >= g1) break;
            const bool whole = ts >= g0 && ts + nks <= g1;
            const int buf = lt & 1;
            int v = -1, c = -1;
            const int u = t * kRows + row;
            if (u < nU) ep.pick(u, v, c);
            const int aux = ep.row_aux(v);
            if (!wait_phase(&acc_full[buf], unsigned(lt / 2) & 1u, fail, op.wait_budget)) {
                s_fail = 1;
                set_status(op.status, DS_DEV_TIMEOUT);
            }
            // the epilogue warps meet at named barriers, so they stop together: every warp has
            // waited (or given up) before thread 0 takes one snapshot of the failure flag
            epi_sync();
            if (tid == 0) s_stop = *fail;
            epi_sync();
            if (s_stop) break;
            fence_after();
            const int mine = 2 * bid + (t == first_tile(bid) ? 0 : 1);
            // 16 columns at a time: emit them (whole tile) or store them as this CTA's part
#pragma unroll 1
            for (int cb = cb0; cb < C::N; cb += 32) {
                uint32_t r16[16];
                ld16(tq + uint32_t(buf * C::N + cb), r16);
                float xs[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) xs[e] = __uint_as_float(r16[e]);
                if (whole) {
                    ep.emit(est, xs, cb, v, c, aux, s_ci, s_cl);
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(parts + (size_t(mine) * kRows + row) * C::N + cb);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        __stcg(dst + e, make_float4(xs[4 * e], xs[4 * e + 1], xs[4 * e + 2], xs[4 * e + 3]));
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);      // the MMA may reuse this buffer
            if (!whole) {
                // the last CTA of the tile adds the parts in k (= CTA) order
                epi_sync();
                const int cf = cta_of(ts), cl = cta_of(ts + nks - 1);
                if (tid == 0) {
                    int nparts = 1;                            // CTAs that own stages of tile t
                    for (int cc = cf; cc != cl; cc = next_owner(cc)) ++nparts;
                    // the epilogue barrier orders the warps' part stores before this release
                    s_last = atom_add_acq_rel_gpu(&tile_cnt[t], 1u) == unsigned(nparts - 1);
                    if (s_last) tile_cnt[t] = 0u;
                }
                epi_sync();
                if (s_last) {
#pragma unroll 1
                    for (int cb = cb0; cb < C::N; cb += 32) {
                        float xs[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) xs[e] = 0.f;
                        for (int cc = cf;; cc = next_owner(cc)) {
                            const int pslot = 2 * cc + (t == first_tile(cc) ? 0 : 1);
                            const float4 *src = reinterpret_cast<const float4 *>(parts + (size_t(pslot) * kRows + row) * C::N + cb);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 pv = __ldcg(src + e);
                                xs[4 * e] += pv.x; xs[4 * e + 1] += pv.y; xs[4 * e + 2] += pv.z; xs[4 * e + 3] += pv.w;
                            }
                            if (cc == cl) break;
                        }
                        ep.emit(est, xs, cb, v, c, aux, s_ci, s_cl);
                    }
                }
                epi_sync();                                    // s_last is read before the next tile
            }
            ++lt;
            ++t;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(uint32_t(C::kTmemCols)) : "memory");
    ep.finish(est);
}

// Host: launch gemm_kernel<MT, Ep> on `grid` CTAs (sets the shared-memory limit once per
// instantiation and device).  `parts` holds parts_bytes(R, grid) bytes; `tile_cnt` one zeroed counter per
// tile (left zero).
template <int MT, class Ep>
ds_status launch(const Operands &op, const Ep &ep, float *parts, unsigned *tile_cnt, int grid, cudaStream_t stream)
{
    static std::atomic<unsigned long long> smem_set{0};
    if (!smem_limit_once(gemm_kernel<MT, Ep>, Cfg<MT>::kSmem, smem_set)) return DS_ERR_CUDA;
    gemm_kernel<MT, Ep><<<grid, kThreads, Cfg<MT>::kSmem, stream>>>(op, ep, parts, tile_cnt);
    DS_TRY_LAUNCH();
    return DS_OK;
}

// Dispatch on the number of B vectors.
template <class Ep>
ds_status launch_for(const Operands &op, const Ep &ep, float *parts, unsigned *tile_cnt, int grid, cudaStream_t stream)
{
    switch (mt_for(op.R)) {
    case 1: return launch<1>(op, ep, parts, tile_cnt, grid, stream);
    case 2: return launch<2>(op, ep, parts, tile_cnt, grid, stream);
    case 3: return launch<3>(op, ep, parts, tile_cnt, grid, stream);
    case 4: return launch<4>(op, ep, parts, tile_cnt, grid, stream);
    case 5: return launch<5>(op, ep, parts, tile_cnt, grid, stream);
    default: return launch<8>(op, ep, parts, tile_cnt, grid, stream);
    }
}

}  // namespace tc
}  // namespace ds
