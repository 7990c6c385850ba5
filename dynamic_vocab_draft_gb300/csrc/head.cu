// Gathered LM head: logits over the shortlist only, fused with the softmax statistics and
// the greedy / Gumbel-max draft draw.
//
// DynaSpec summary, Technical Details > System Modules "Gathered LM Head" (a fused index-
// select + GEMM) and Novel Architectural Elements ("Dynamic Vocabulary Head"; "gathering and
// matrix multiplication without intermediate memory overhead"); Limitations: the gathered
// multiplication costs more per row than a dense one.  W[V_S] is never materialised: every
// kernel streams the selected rows of W straight from HBM.
//
// Two shapes:
//   * per-row lists (batch-1 chain drafting): a GEMV over gathered rows.  One warp per W row,
//     16-byte streaming loads (a W row is contiguous, so a gather is still a coalesced
//     stream), the hidden state in shared memory, a warp-shuffle dot, and the epilogue
//     folded into a per-warp softmax/argmax state; blocks combine through a last-block pass.
//   * a union of lists (batched chain drafting, tree drafting): W is read once over the
//     union of the lists' clusters and every union row is scored against all B*G head rows on
//     the tensor cores; the epilogue keeps the (row, token) pairs whose list selects the
//     token's cluster.
#include "common.cuh"

namespace ds {
namespace {

int num_sms()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    }
    return n;
}

// ---------------------------------------------------------------------------------------
// Per-row gathered GEMV
// ---------------------------------------------------------------------------------------
constexpr int kGvWarps = 16;           // one 512-thread block per SM
constexpr int kHeadSideSms = 8;        // SMs a batch-1 head leaves to the side stream
constexpr int kGvMaxD = 16384;
constexpr int kGvMaxBlocks = 1024;     // per list; bounds the partials in the workspace

struct HeadArgs {
    const uint16_t *H;
    const uint16_t *W;
    int V, d;
    const int32_t *vs_offsets, *vs_ids;
    float T, inv_te;
    uint64_t seed;
    int pos;
    float *logits, *row_max, *row_sumexp;
    int32_t *token, *token_idx;
    int32_t *status;
};

__device__ __forceinline__ void write_row(const HeadArgs &a, int r, const Stat &s)
{
    if (a.row_max) a.row_max[r] = s.m;
    if (a.row_sumexp) a.row_sumexp[r] = s.s;
    a.token[r] = s.v;
    a.token_idx[r] = s.j;
}

// Rows are streamed in groups of kGvG 16-byte loads per lane (4 KB of a row per warp at a
// time).  The loads of the warp's next group -- the second half of the row, or the first half
// of its next row -- are issued before the current group is multiplied, so every warp keeps
// 4-8 KB in flight while it computes; 16 warps per SM hold ~100 KB in flight.  The id of the
// warp's next row is prefetched one row ahead.
//
// grid (gx, B): block (x, b) handles rows j = x*16 + warp, step gx*16, of list b.
constexpr int kGvG = 8;                // loads per lane per group (256 bf16 per load round)

__device__ __forceinline__ void load_group(uint4 (&buf)[kGvG], const uint16_t *W, int v, int d, int k0, int lane)
{
    const uint4 *row = reinterpret_cast<const uint4 *>(W + size_t(v) * d);
#pragma unroll
    for (int u = 0; u < kGvG; ++u) {
        const int k = k0 + (u * 32 + lane) * 8;
        buf[u] = k < d ? ld_stream(row + (k >> 3)) : make_uint4(0, 0, 0, 0);
    }
}

// h is kept in shared memory as bf16: one 16-byte load gives the 8 values a W vector meets.
__device__ __forceinline__ void dot_group(const uint4 (&buf)[kGvG], const uint4 *hs, int d, int k0, int lane,
                                          float &a0, float &a1)
{
#pragma unroll
    for (int u = 0; u < kGvG; ++u) {
        const int k = k0 + (u * 32 + lane) * 8;
        if (k < d) {
            const uint4 x = hs[k >> 3];
            const uint4 w = buf[u];
            a0 = fmaf(bf16lo(w.x), bf16lo(x.x), a0);
            a1 = fmaf(bf16hi(w.x), bf16hi(x.x), a1);
            a0 = fmaf(bf16lo(w.y), bf16lo(x.y), a0);
            a1 = fmaf(bf16hi(w.y), bf16hi(x.y), a1);
            a0 = fmaf(bf16lo(w.z), bf16lo(x.z), a0);
            a1 = fmaf(bf16hi(w.z), bf16hi(x.z), a1);
            a0 = fmaf(bf16lo(w.w), bf16lo(x.w), a0);
            a1 = fmaf(bf16hi(w.w), bf16hi(x.w), a1);
        }
    }
}

__global__ void __launch_bounds__(kGvWarps * 32, 1)
head_gemv_kernel(HeadArgs a, Stat *__restrict__ partials, unsigned *__restrict__ counters)
{
    extern __shared__ uint4 hs[];                 // h as bf16, d / 8 vectors
    __shared__ Stat warp_stat[kGvWarps];
    const int b = blockIdx.y;
    const int d = a.d;
    const uint4 *h = reinterpret_cast<const uint4 *>(a.H + size_t(b) * d);
    for (int k = threadIdx.x; k < d / 8; k += blockDim.x) hs[k] = h[k];
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int base = a.vs_offsets[b];
    const int n = a.vs_offsets[b + 1] - base;
    const int32_t *ids = a.vs_ids + base;
    float *lout = a.logits + base;
    const int stride = gridDim.x * kGvWarps;
    const int ngroups = (d + kGvG * 256 - 1) / (kGvG * 256);     // groups per row
    Stat st = stat_empty();

    int j = blockIdx.x * kGvWarps + warp;
    if (j < n) {
        auto safe = [&](int v) { return (v >= 0 && v < a.V) ? v : 0; };
        int v = ids[j];
        int jn = j + stride;
        int vn = jn < n ? ids[jn] : 0;                              // next row's id, one row ahead
        uint4 cur[kGvG], nxt[kGvG];
        load_group(cur, a.W, safe(v), d, 0, lane);
        int g = 0;
        float a0 = 0.f, a1 = 0.f;
        float gum = 0.f;
        if (a.T > 0.f && lane == 0 && v >= 0 && v < a.V) gum = gumbel(a.seed, uint32_t(v), uint32_t(a.pos), uint32_t(b));
        for (;;) {
            // issue the next group's loads before multiplying the current one
            const bool more_in_row = g + 1 < ngroups;
            const bool have_next = more_in_row || jn < n;
            if (more_in_row) load_group(nxt, a.W, safe(v), d, (g + 1) * kGvG * 256, lane);
            else if (jn < n) load_group(nxt, a.W, safe(vn), d, 0, lane);
            dot_group(cur, hs, d, g * kGvG * 256, lane, a0, a1);
            if (!more_in_row) {
                const float acc = warp_sum(a0 + a1);
                if (lane == 0) {
                    if (v < 0 || v >= a.V) {
                        set_status(a.status, DS_DEV_BAD_INDEX);
                        lout[j] = 0.f;
                    } else {
                        lout[j] = acc;
                        const float x = acc * a.inv_te;
                        stat_add(st, x, a.T > 0.f ? x + gum : acc, v, j);
                    }
                }
                a0 = a1 = 0.f;
                if (jn >= n) break;
                j = jn; v = vn;
                jn = j + stride;
                vn = jn < n ? ids[jn] : 0;
                g = 0;
                if (a.T > 0.f && lane == 0 && v >= 0 && v < a.V) gum = gumbel(a.seed, uint32_t(v), uint32_t(a.pos), uint32_t(b));
            } else {
                ++g;
            }
            if (!have_next) break;
#pragma unroll
            for (int u = 0; u < kGvG; ++u) cur[u] = nxt[u];
        }
    }
    if (lane == 0) warp_stat[warp] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        Stat c = warp_stat[0];
        for (int w = 1; w < kGvWarps; ++w) c = stat_merge(c, warp_stat[w]);
        st_stat(&partials[size_t(b) * kGvMaxBlocks + blockIdx.x], c);
    }
    if (!last_block_done(&counters[b], gridDim.x)) return;
    if (warp != 0) return;
    // Final combine in a fixed order: lane l folds partials l, l+32, ...; then a fixed tree.
    Stat c = stat_empty();
    for (int i = lane; i < int(gridDim.x); i += 32) c = stat_merge(c, ld_stat(&partials[size_t(b) * kGvMaxBlocks + i]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Stat other = shfl_xor_stat(c, o);
        c = (lane & o) ? stat_merge(other, c) : stat_merge(c, other);
    }
    if (lane == 0) write_row(a, b, c);
}

// ---------------------------------------------------------------------------------------
// Helpers of the union path.
// ---------------------------------------------------------------------------------------
constexpr int kUnMaxRows = 128;                 // head rows

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N)); }

struct UnionArgs {
    HeadArgs h;
    int B, G, R, M;
    const int32_t *cpos, *rank, *union_ids, *union_cluster, *union_count;
};

// ---------------------------------------------------------------------------------------
// Union path on the 5th-generation tensor cores (tcgen05, accumulator in tensor memory).
//
// Work: tiles of 128 union rows of W (the MMA's M side) x all head rows (N = 16*MT) x the full
// depth d, each tile swept in k-stages of kCols columns.  The (tile, k-stage) units, in tile
// order, are split into equal contiguous ranges, one per CTA of a persistent grid (a stream-K
// split), so every SM streams the same number of W bytes whatever the union size; a tile
// whose stages fall into several CTAs is finished by the last of them, which adds the parts
// in k order.
//
// Per CTA one software pipeline runs across its tiles: kStages shared-memory slots, loads
// kLook stages ahead of the stage being multiplied, and the MMAs of stage i are waited for
// only when their slot is refilled two stages later, so the loads never wait on the tensor
// core.  A slot holds the 128 W rows and the N head rows for its columns in the 128-byte-
// swizzled K-major layout the MMA descriptors describe (8-row x 128-byte atoms, 16-byte chunk
// c of row r at c ^ (r & 7)).  All threads fill slots with cp.async; one thread issues the
// MMAs (M=128, N=16*MT, K=16 each) and commits them to the slot's mbarrier.  The 128 x N fp32
// accumulator lives in tensor memory; at a tile's end the epilogue reads it with tcgen05.ld
// (the four warps of each TMEM lane quarter split the columns, each warp its 32 lanes = W
// rows) and scatters the selected logits while the next stages' loads are in flight.
// ---------------------------------------------------------------------------------------
constexpr int kTcRows = 128;
constexpr int kTcThreads = 512;
constexpr int kUnionMaxGrid = 160;              // CTAs of the union head (<= SMs in use)
constexpr int kUnionMaxTiles = 8192;            // union rows <= 8192 * 128

__host__ __device__ constexpr int tc_min(int a, int b) { return a < b ? a : b; }

template <int MT> struct TcCfg {
    static constexpr int N = 16 * MT;
    static constexpr int kAtoms = MT >= 8 ? 1 : 2;             // 64-column atoms per stage
    static constexpr int kCols = kAtoms * 64;                  // columns of d per stage
    static constexpr int kABytes = kAtoms * kTcRows * 128;     // W part of a stage
    static constexpr int kBBytes = kAtoms * N * 128;           // H part of a stage
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = tc_min(6, (210 * 1024) / kStageBytes);
    static constexpr int kLook = kStages - 2;                  // stages loaded ahead
    static constexpr int kMeta = kLook + 2;                    // tiles whose row ids are held
    static constexpr int kTmemCols = N <= 32 ? 32 : N <= 64 ? 64 : 128;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 1024 /* align */ +
                                    size_t(kMeta) * 2 * kTcRows * sizeof(int32_t);
    static_assert(kStages >= 3, "the pipeline needs three slots");
};

// Columns of the accumulator a partial tile stores (all N; rows >= R hold zeros).
__host__ __device__ constexpr int union_mt(int rows)
{
    return rows <= 16 ? 1 : rows <= 32 ? 2 : rows <= 48 ? 3 : rows <= 64 ? 4 : rows <= 80 ? 5 : 8;
}

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

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int MT>
__global__ void __launch_bounds__(kTcThreads, 1)
head_union_tc_kernel(UnionArgs a, float *__restrict__ parts, unsigned *__restrict__ tile_cnt)
{
    using C = TcCfg<MT>;
    constexpr int STG = C::kStages, L = C::kLook;
    constexpr int CPR = C::kAtoms * 8;                         // 16-byte chunks per row per stage
    constexpr int RPP = kTcThreads / CPR;                      // rows per pass of all threads
    constexpr int APASS = kTcRows / RPP;                       // W-row passes per stage
    constexpr int BPASS = (C::N + RPP - 1) / RPP;              // head-row passes per stage
    static_assert(kTcRows % RPP == 0, "row passes");
    extern __shared__ __align__(1024) unsigned char tc_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
    int32_t *s_meta = reinterpret_cast<int32_t *>(sm + size_t(STG) * C::kStageBytes);   // [kMeta][v | c][128]
    __shared__ uint64_t mma_done[STG];
    __shared__ int32_t s_hb[C::N];                 // list of head row r (-1: padding)
    __shared__ long long s_hbase[C::N];            // logits index of entry 0 of row r's list
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail, s_cf, s_cl;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.h.d, R = a.R, G = a.G, M = a.M, V = a.h.V;
    const int nU = min(*a.union_count, V);
    const int ntiles = (nU + kTcRows - 1) / kTcRows;
    const int nks = (d + C::kCols - 1) / C::kCols;             // stages per tile
    const long long total = 1LL * ntiles * nks;                // < 2^31: ntiles <= 8192, nks <= 256
    const int grid = gridDim.x, bid = blockIdx.x;
    const int g0 = int(total * bid / grid), g1 = int(total * (bid + 1) / grid);
    if (g0 >= g1) return;                                      // uniform: no stage for this CTA
    constexpr uint32_t idesc = umma_idesc_bf16(kTcRows, C::N);
    // the CTA whose range holds unit i, and the first tile of CTA c
    auto cta_of = [&](long long i) { return int(((i + 1) * grid - 1) / total); };
    auto first_tile = [&](int c) { return int((total * c / grid) / nks); };
    // the owner of the unit after CTA c's range (CTAs with empty ranges own nothing)
    auto next_owner = [&](int c) { return cta_of(total * (c + 1) / grid); };

    if (tid == 0) {
        for (int i = 0; i < STG; ++i) mbar_init(&mma_done[i], 1);
        mbar_fence_init();
        s_fail = 0;
    }
    for (int r = tid; r < C::N; r += kTcThreads) {
        int hb = -1;
        long long base = 0;
        if (r < R) {
            hb = r / G;
            const int gi = r - hb * G, off = a.h.vs_offsets[hb], nb = a.h.vs_offsets[hb + 1] - off;
            base = 1LL * off * G + 1LL * gi * nb;
        }
        s_hb[r] = hb;
        s_hbase[r] = base;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&s_tmem)), "r"(uint32_t(C::kTmemCols)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Every thread copies one fixed 16-byte column chunk `ch` of rows prow + RPP*j.  Its shared-
    // memory destinations are the same in every stage (up to the slot base); its sources move
    // by kCols columns per stage.
    const int ch = tid % CPR, prow = tid / CPR;
    const int coff = (ch >> 3) * 64 + (ch & 7) * 8;            // column of the chunk inside a stage
    const uint32_t dst0 = uint32_t((ch >> 3) * (kTcRows * 128) + prow * 128 + (((ch & 7) ^ (prow & 7)) << 4));
    const uint32_t bdst0 = uint32_t((ch >> 3) * (C::N * 128) + prow * 128 + (((ch & 7) ^ (prow & 7)) << 4));
    static_assert(RPP % 8 == 0, "rows of one thread share their swizzle phase");
    const uint16_t *hsrc[BPASS];
#pragma unroll
    for (int j = 0; j < BPASS; ++j) {
        const int r = prow + RPP * j;
        hsrc[j] = r < R ? a.h.H + size_t(r) * d + coff : nullptr;
    }
    const uint16_t *wsrc[APASS];                               // rows of the tile being filled
    const uint32_t smem0 = smem_u32(sm);

    // Row ids and clusters of tile t into ring slot t % kMeta, and this thread's row pointers
    // for it.  Tiles arrive in increasing order; every thread calls this with the same t.
    int meta_tile = -1;
    auto ensure_meta = [&](int t) {
        if (t == meta_tile) return;
        int32_t *mv = s_meta + (t % C::kMeta) * (2 * kTcRows);
        for (int q = tid; q < kTcRows; q += kTcThreads) {
            const int u = t * kTcRows + q;
            int v = -1, c = -1;
            if (u < nU) {
                v = a.union_ids[u];
                c = a.union_cluster[u];
                if (v < 0 || v >= V || c < 0 || c >= M) { set_status(a.h.status, DS_DEV_BAD_INDEX); v = -1; c = -1; }
            }
            mv[q] = v;
            mv[kTcRows + q] = c;
        }
        meta_tile = t;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < APASS; ++j) {
            const int v = mv[prow + RPP * j];
            wsrc[j] = v >= 0 ? a.h.W + size_t(v) * d + coff : nullptr;
        }
    };
    // cp.async fill of slot `slot` with k-stage ks of the tile ensure_meta last prepared
    auto fill = [&](int slot, int ks) {
        const int k0 = ks * C::kCols;
        const bool kin = k0 + coff < d;
        const uint32_t A = smem0 + uint32_t(slot * C::kStageBytes);
        const uint32_t Bm = A + C::kABytes;
#pragma unroll
        for (int j = 0; j < APASS; ++j) {
            const bool ok = kin && wsrc[j] != nullptr;
            cp_async16(A + dst0 + uint32_t(j * RPP * 128), ok ? wsrc[j] + k0 : a.h.W, ok ? 16 : 0);
        }
#pragma unroll
        for (int j = 0; j < BPASS; ++j) {
            if (prow + RPP * j < C::N) {
                const bool ok = kin && hsrc[j] != nullptr;
                cp_async16(Bm + bdst0 + uint32_t(j * RPP * 128), ok ? hsrc[j] + k0 : a.h.H, ok ? 16 : 0);
            }
        }
    };
    // logits of one W row (v, cluster c, rank rk) against head rows cb .. cb+15
    auto scatter = [&](const float (&x)[16], int cb, int v, int c, int rk) {
        if (v < 0) return;
        int pcs[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int hb = s_hb[cb + e];
            pcs[e] = hb >= 0 ? __ldg(a.cpos + size_t(hb) * M + c) : -1;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if (pcs[e] >= 0) a.h.logits[s_hbase[cb + e] + pcs[e] + rk] = x[e];
    };

    // (tile, k-stage) of the stage being multiplied and of the next stage to load
    int t = g0 / nks, ks = g0 - t * nks;
    int ft = t, fks = ks, fslot = 0;
    // prologue: the first L stages of the range
    for (int p = 0; p < L; ++p) {
        if (g0 + p < g1) {
            ensure_meta(ft);
            fill(fslot, fks);
            if (++fks == nks) { fks = 0; ++ft; }
            if (++fslot == STG) fslot = 0;
        }
        cp_async_commit();
    }
    int issued = 0;                                            // stages whose MMAs were issued
    int slot = 0;                                              // slot of stage li
    for (int i = g0; i < g1; ++i) {
        const int li = i - g0;
        // refill: stage li + L goes into the slot of stage li - 2, whose MMAs were issued two
        // iterations ago
        if (i + L < g1) {
            const int lf = li + L;
            if (lf >= STG && !mbar_wait(&mma_done[fslot], unsigned(lf / STG - 1) & 1u)) {
                s_fail = 1;
                set_status(a.h.status, DS_DEV_TIMEOUT);
            }
            ensure_meta(ft);
            fill(fslot, fks);
            if (++fks == nks) { fks = 0; ++ft; }
            if (++fslot == STG) fslot = 0;
        }
        cp_async_commit();
        cp_async_wait<L>();                                    // stage li has landed (this thread's part)
        proxy_fence_async();                                   // make it visible to the tensor cores
        __syncthreads();
        if (s_fail) break;                                     // uniform: read after the barrier
        const bool first = ks == 0 || i == g0;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t A = smem0 + uint32_t(slot * C::kStageBytes);
            const uint32_t Bm = A + C::kABytes;
#pragma unroll
            for (int at = 0; at < C::kAtoms; ++at) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = umma_desc_sw128(A + at * (kTcRows * 128) + kk * 32);
                    const uint64_t bd = umma_desc_sw128(Bm + at * (C::N * 128) + kk * 32);
                    tc_mma(tmem, ad, bd, idesc, (first && at == 0 && kk == 0) ? 0u : 1u);
                }
            }
            tc_commit(&mma_done[slot]);
        }
        ++issued;
        const int cur_slot = slot;
        if (++slot == STG) slot = 0;
        const bool tile_end = ks == nks - 1 || i == g1 - 1;
        const int tt = t;
        if (++ks == nks) { ks = 0; ++t; }
        if (!tile_end) continue;
        // this CTA's part of tile tt is in the accumulator
        if (!mbar_wait(&mma_done[cur_slot], unsigned(li / STG) & 1u)) {
            s_fail = 1;
            set_status(a.h.status, DS_DEV_TIMEOUT);
        }
        tc_fence_after();
        const int wq = warp & 3;                               // TMEM lane quarter this warp may read
        const int row = wq * 32 + lane;                        // W row of the tile
        const int32_t *mv = s_meta + (tt % C::kMeta) * (2 * kTcRows);
        const int v = mv[row], c = mv[kTcRows + row];
        const int rk = v >= 0 ? __ldg(a.rank + v) : 0;
        const uint32_t taddr = tmem + (uint32_t(wq * 32) << 16);
        const bool whole = 1LL * tt * nks >= g0 && 1LL * (tt + 1) * nks <= g1;
        constexpr int kColStep = 16 * (kTcThreads / 128);      // warps sharing a lane quarter split the columns
        if (whole) {
            for (int cb = (warp >> 2) * 16; cb < C::N; cb += kColStep) {
                uint32_t r16[16];
                tc_ld16(taddr + uint32_t(cb), r16);
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(r16[e]);
                scatter(x, cb, v, c, rk);
            }
        } else {
            // store this part; the last CTA of the tile adds the parts in k (= CTA) order
            const int mine = 2 * bid + (tt == first_tile(bid) ? 0 : 1);
            for (int cb = (warp >> 2) * 16; cb < C::N; cb += kColStep) {
                uint32_t r16[16];
                tc_ld16(taddr + uint32_t(cb), r16);
                float4 *dst = reinterpret_cast<float4 *>(parts + (size_t(mine) * kTcRows + row) * C::N + cb);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    __stcg(dst + e, make_float4(__uint_as_float(r16[4 * e]), __uint_as_float(r16[4 * e + 1]),
                                                __uint_as_float(r16[4 * e + 2]), __uint_as_float(r16[4 * e + 3])));
            }
            __threadfence();
            if (tid == 0) {
                s_cf = cta_of(1LL * tt * nks);
                s_cl = cta_of(1LL * (tt + 1) * nks - 1);
            }
            __syncthreads();
            const int cf = s_cf, cl = s_cl;
            int nparts = 1;                                    // CTAs that own stages of tile tt
            for (int cc = cf; cc != cl; cc = next_owner(cc)) ++nparts;
            if (last_block_done(&tile_cnt[tt], unsigned(nparts))) {
                for (int cb = (warp >> 2) * 16; cb < C::N; cb += kColStep) {
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = 0.f;
                    for (int cc = cf;; cc = next_owner(cc)) {
                        const int pslot = 2 * cc + (tt == first_tile(cc) ? 0 : 1);
                        const float4 *src = reinterpret_cast<const float4 *>(parts + (size_t(pslot) * kTcRows + row) * C::N + cb);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 p = __ldcg(src + e);
                            x[4 * e] += p.x; x[4 * e + 1] += p.y; x[4 * e + 2] += p.z; x[4 * e + 3] += p.w;
                        }
                        if (cc == cl) break;
                    }
                    scatter(x, cb, v, c, rk);
                }
            }
        }
        tc_fence_before();
        __syncthreads();                                       // the accumulator may be overwritten
        if (s_fail) break;
    }
    cp_async_wait<0>();
    // every issued MMA must be complete before the accumulator is released
    if (tid == 0) {
        const long long deadline = clock64() + kWaitBudgetCycles;
        for (int li = max(0, issued - STG); li < issued; ++li)
            (void)mbar_wait_until(&mma_done[li % STG], unsigned(li / STG) & 1u, deadline);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem), "r"(uint32_t(C::kTmemCols)) : "memory");
}

// Softmax statistics and the draft draw of every head row from its stored logits.
// grid (chunks, R): block (x, r) folds elements [x*kRsChunk, ...) of row r; the last block of the
// row combines the partials in a fixed order.
constexpr int kRsPer = 16;
constexpr int kRsChunk = 256 * kRsPer;

__global__ void __launch_bounds__(256)
head_rowstats_kernel(HeadArgs a, int G, Stat *__restrict__ partials, unsigned *__restrict__ counters)
{
    __shared__ Stat ws[8];
    const int r = blockIdx.y, b = r / G, gi = r - b * G;
    const int off = a.vs_offsets[b];
    const int n = a.vs_offsets[b + 1] - off;
    const float *l = a.logits + int64_t(off) * G + int64_t(gi) * n;
    const int32_t *ids = a.vs_ids + off;
    Stat st = stat_empty();
    const int j0 = blockIdx.x * kRsChunk + threadIdx.x * kRsPer;
    for (int e = 0; e < kRsPer; ++e) {
        const int j = j0 + e;
        if (j >= n) break;
        const float lj = l[j];
        const int v = ids[j];
        const float x = lj * a.inv_te;
        const float key = a.T > 0.f ? x + gumbel(a.seed, uint32_t(v), uint32_t(a.pos), uint32_t(r)) : lj;
        stat_add(st, x, key, v, j);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Stat other = shfl_xor_stat(st, o);
        st = (lane & o) ? stat_merge(other, st) : stat_merge(st, other);
    }
    if (lane == 0) ws[warp] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        Stat c = ws[0];
        for (int w = 1; w < 8; ++w) c = stat_merge(c, ws[w]);
        st_stat(&partials[size_t(r) * kGvMaxBlocks + blockIdx.x], c);
    }
    if (!last_block_done(&counters[r], gridDim.x)) return;
    if (warp != 0) return;
    Stat c = stat_empty();
    for (int i = lane; i < int(gridDim.x); i += 32) c = stat_merge(c, ld_stat(&partials[size_t(r) * kGvMaxBlocks + i]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Stat other = shfl_xor_stat(c, o);
        c = (lane & o) ? stat_merge(other, c) : stat_merge(c, other);
    }
    if (lane == 0) write_row(a, r, c);
}

}  // namespace
}  // namespace ds

using namespace ds;

namespace {

constexpr size_t kHeadPartialsPerRow = 1024;   // >= kGvMaxBlocks

// Workspace layout of the head (byte offsets), for `rows` head rows:
//   [row counters | tile counters]  zero before first use; every call leaves them zero
//   [row-statistics partials]       rows x kHeadPartialsPerRow
//   [union parts]                   two 128 x N fp32 partial tiles per union CTA
struct HeadWs {
    size_t row_cnt, tile_cnt, partials, parts, total, counters_bytes;
};

HeadWs head_ws_layout(int rows)
{
    HeadWs w;
    w.row_cnt = 0;
    w.tile_cnt = align256(size_t(rows) * sizeof(unsigned));
    w.partials = w.tile_cnt + align256(size_t(kUnionMaxTiles) * sizeof(unsigned));
    w.counters_bytes = w.partials;
    w.parts = w.partials + align256(size_t(rows) * kHeadPartialsPerRow * sizeof(Stat));
    const size_t n = size_t(16 * union_mt(rows));
    w.total = w.parts + align256(size_t(2) * kUnionMaxGrid * kTcRows * n * sizeof(float));
    return w;
}

template <int MT>
ds_status launch_union(const UnionArgs &ua, float *parts, unsigned *tile_cnt, cudaStream_t stream)
{
    const size_t smem = TcCfg<MT>::kSmem;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(head_union_tc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return DS_ERR_CUDA;
        attr = true;
    }
    const int grid = num_sms() < kUnionMaxGrid ? num_sms() : kUnionMaxGrid;
    head_union_tc_kernel<MT><<<grid, kTcThreads, smem, stream>>>(ua, parts, tile_cnt);
    DS_TRY_LAUNCH();
    return DS_OK;
}

}  // namespace

extern "C" size_t ds_head_workspace_bytes(int rows)
{
    if (rows <= 0) return 0;
    return head_ws_layout(rows).total;
}

extern "C" ds_status ds_gathered_head(const uint16_t *H, int B, int G,
                                      const uint16_t *W, int V, int d,
                                      const int32_t *vs_offsets, const int32_t *vs_ids,
                                      const int32_t *cpos, int M, const int32_t *rank_in_cluster,
                                      const int32_t *union_ids, const int32_t *union_cluster,
                                      const int32_t *union_count,
                                      float T, uint64_t seed, int pos,
                                      float *logits, float *row_max, float *row_sumexp,
                                      int32_t *token, int32_t *token_idx,
                                      void *ws, size_t ws_bytes, int32_t *dev_status,
                                      cudaStream_t stream)
{
    if (!H || !W || !vs_offsets || !vs_ids || !logits || !token || !token_idx) return DS_ERR_INVALID_ARG;
    if (B < 1 || G < 1 || V < 1 || d < 8 || d % 8 || !(T >= 0.f) || pos < 0) return DS_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(W)) return DS_ERR_INVALID_ARG;
    if (d > kGvMaxD) return DS_ERR_UNSUPPORTED;
    const long long rows = 1LL * B * G;
    const int nu = (union_ids != nullptr) + (union_cluster != nullptr) + (union_count != nullptr);
    if (nu != 0 && nu != 3) return DS_ERR_INVALID_ARG;
    if (rows > 65535) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_head_workspace_bytes(int(rows))) return DS_ERR_WORKSPACE;

    const HeadWs lay = head_ws_layout(int(rows));
    char *wsb = static_cast<char *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(wsb + lay.row_cnt);
    Stat *partials = reinterpret_cast<Stat *>(wsb + lay.partials);

    HeadArgs a;
    a.H = H; a.W = W; a.V = V; a.d = d;
    a.vs_offsets = vs_offsets; a.vs_ids = vs_ids;
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.seed = seed; a.pos = pos;
    a.logits = logits; a.row_max = row_max; a.row_sumexp = row_sumexp;
    a.token = token; a.token_idx = token_idx;
    a.status = dev_status;

    if (nu == 0) {
        if (G != 1) return DS_ERR_UNSUPPORTED;
        // One 512-thread block per SM.  At batch 1 a few SMs are left to the side stream, so the
        // next position's router and shortlist build run while this head streams W.
        int gx = B == 1 ? num_sms() - kHeadSideSms : (num_sms() + B - 1) / B;
        if (gx < 1) gx = 1;
        if (gx > kGvMaxBlocks) gx = kGvMaxBlocks;
        const size_t smem = size_t(d) * sizeof(uint16_t);
        static bool attr_set = false;
        if (!attr_set) {
            if (cudaFuncSetAttribute(head_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(kGvMaxD * sizeof(float))) != cudaSuccess)
                return DS_ERR_CUDA;
            attr_set = true;
        }
        head_gemv_kernel<<<dim3(gx, B), kGvWarps * 32, smem, stream>>>(a, partials, counters);
        DS_TRY_LAUNCH();
        return DS_OK;
    }

    if (!cpos || !rank_in_cluster || M < 1) return DS_ERR_INVALID_ARG;
    if (rows > kUnMaxRows) return DS_ERR_UNSUPPORTED;
    if ((V + kRsChunk - 1) / kRsChunk > kGvMaxBlocks) return DS_ERR_UNSUPPORTED;
    if ((V + kTcRows - 1) / kTcRows > kUnionMaxTiles) return DS_ERR_UNSUPPORTED;
    UnionArgs ua;
    ua.h = a; ua.B = B; ua.G = G; ua.R = int(rows); ua.M = M;
    ua.cpos = cpos; ua.rank = rank_in_cluster;
    ua.union_ids = union_ids; ua.union_cluster = union_cluster; ua.union_count = union_count;
    float *parts = reinterpret_cast<float *>(wsb + lay.parts);
    unsigned *tile_cnt = reinterpret_cast<unsigned *>(wsb + lay.tile_cnt);
    ds_status st;
    switch (union_mt(int(rows))) {
    case 1: st = launch_union<1>(ua, parts, tile_cnt, stream); break;
    case 2: st = launch_union<2>(ua, parts, tile_cnt, stream); break;
    case 3: st = launch_union<3>(ua, parts, tile_cnt, stream); break;
    case 4: st = launch_union<4>(ua, parts, tile_cnt, stream); break;
    case 5: st = launch_union<5>(ua, parts, tile_cnt, stream); break;
    default: st = launch_union<8>(ua, parts, tile_cnt, stream); break;
    }
    if (st != DS_OK) return st;
    const int chunks = (V + kRsChunk - 1) / kRsChunk;
    head_rowstats_kernel<<<dim3(chunks, unsigned(rows)), 256, 0, stream>>>(a, G, partials, counters);
    DS_TRY_LAUNCH();
    return DS_OK;
}

// ---------------------------------------------------------------------------------------
// ds_gathered_head_noalloc: the same head for callers that cannot give the library any
// scratch memory.  The cross-block partials and completion counters live in one file-scope
// device array of fixed size instead of a caller workspace.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr int kNoAllocMaxRows = 32;
// head_ws_layout(32), spelled out so the array can be sized at compile time
constexpr size_t kNoAllocCounters = 256 + size_t(kUnionMaxTiles) * sizeof(unsigned);
constexpr size_t kNoAllocBytes = kNoAllocCounters + size_t(kNoAllocMaxRows) * kHeadPartialsPerRow * sizeof(Stat) +
                                 size_t(2) * kUnionMaxGrid * kTcRows * 32 * sizeof(float);
static_assert(256 >= kNoAllocMaxRows * sizeof(unsigned), "counter block");
static_assert(kNoAllocCounters % 256 == 0 && (size_t(kNoAllocMaxRows) * kHeadPartialsPerRow * sizeof(Stat)) % 256 == 0,
              "no padding between the regions");

// Held by every GPU that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_head_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kNoAllocMaxDevices];

// Device address of the scratch array on the current device, looked up once per device.
// (In host code the array's name is only a host-side stand-in, not a device address.)
ds_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return DS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_head_noalloc_scratch) != cudaSuccess || !p) return DS_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return DS_OK;
}

}  // namespace

extern "C" ds_status ds_gathered_head_noalloc(const uint16_t *H, int B, int G,
                                              const uint16_t *W, int V, int d,
                                              const int32_t *vs_offsets, const int32_t *vs_ids,
                                              const int32_t *cpos, int M, const int32_t *rank_in_cluster,
                                              const int32_t *union_ids, const int32_t *union_cluster,
                                              const int32_t *union_count,
                                              float T, uint64_t seed, int pos,
                                              float *logits, float *row_max, float *row_sumexp,
                                              int32_t *token, int32_t *token_idx,
                                              int32_t *dev_status, cudaStream_t stream)
{
    if (B < 1 || G < 1) return DS_ERR_INVALID_ARG;
    if (1LL * B * G > kNoAllocMaxRows) return DS_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const ds_status st = noalloc_scratch(&scratch);
    if (st != DS_OK) return st;
    // The counters must start at zero; the array keeps whatever the previous call left.
    if (cudaMemsetAsync(scratch, 0, kNoAllocCounters, stream) != cudaSuccess) return DS_ERR_CUDA;
    return ds_gathered_head(H, B, G, W, V, d, vs_offsets, vs_ids, cpos, M, rank_in_cluster,
                            union_ids, union_cluster, union_count, T, seed, pos,
                            logits, row_max, row_sumexp, token, token_idx,
                            scratch, kNoAllocBytes, dev_status, stream);
}
