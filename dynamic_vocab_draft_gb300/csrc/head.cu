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
// Union path: W read once over the union of the lists, all head rows on the tensor cores.
//
// Swap-AB tile: the 128 union rows of W are the MMA's M side (8 warps x 16 rows) and the
// R = B*G head rows are its N side (NT tiles of 8, R <= 128), K swept in 64-element (128-
// byte) slabs through a STAGES-deep cp.async ring.  Shared-memory rows are 128 bytes with the
// 16-byte chunks XOR-swizzled by (row & 7), so ldmatrix reads are bank-conflict free.
// ---------------------------------------------------------------------------------------
constexpr int kUnWarps = 8;
constexpr int kUnRows = 128;            // W rows per tile
constexpr int kUnBK = 64;               // K elements per slab
constexpr int kUnStages = 4;
constexpr int kUnMaxRows = 128;         // head rows (N side)

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

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-row swizzled slab
__device__ __forceinline__ uint32_t swz(int r, int ch) { return uint32_t(r * 128 + ((ch ^ (r & 7)) << 4)); }

struct UnionArgs {
    HeadArgs h;
    int B, G, R, M;
    const int32_t *cpos, *rank, *union_ids, *union_cluster, *union_count;
};

template <int NT>
struct UnionSmem {
    static constexpr int kA = kUnRows * 128;          // bytes per A slab
    static constexpr int kB = NT * 8 * 128;           // bytes per B slab
    static constexpr int kStage = kA + kB;
    static constexpr size_t kBytes = size_t(kUnStages) * kStage + sizeof(Stat) * kUnWarps * NT * 8
                                     + 3 * kUnRows * sizeof(int32_t) + 128;
};

template <int NT>
__global__ void __launch_bounds__(kUnWarps * 32, 1)
head_union_kernel(UnionArgs a, Stat *__restrict__ partials)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    using L = UnionSmem<NT>;
    Stat *s_stat = reinterpret_cast<Stat *>(smem + kUnStages * L::kStage);       // [warp][NT*8]
    int32_t *s_uid = reinterpret_cast<int32_t *>(s_stat + kUnWarps * NT * 8);    // [128]
    int32_t *s_ucl = s_uid + kUnRows;
    int32_t *s_rnk = s_ucl + kUnRows;
    const uint32_t s_base = smem_u32(smem);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.h.d, R = a.R, G = a.G, M = a.M;
    const int nU = min(*a.union_count, a.h.V);
    const int ntiles = (nU + kUnRows - 1) / kUnRows;
    const int KT = (d + kUnBK - 1) / kUnBK;

    for (int i = tid; i < kUnWarps * NT * 8; i += blockDim.x) s_stat[i] = stat_empty();

    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        __syncthreads();                    // previous tile's epilogue is done with s_uid
        for (int r = tid; r < kUnRows; r += blockDim.x) {
            const int u = tile * kUnRows + r;
            int v = -1, c = -1, rk = 0;
            if (u < nU) {
                v = a.union_ids[u];
                c = a.union_cluster[u];
                if (v < 0 || v >= a.h.V || c < 0 || c >= M) { set_status(a.h.status, DS_DEV_BAD_INDEX); v = -1; }
                else rk = a.rank[v];
            }
            s_uid[r] = v; s_ucl[r] = c; s_rnk[r] = rk;
        }
        __syncthreads();

        auto load_slab = [&](int stage, int kt) {
            const uint32_t sa = s_base + stage * L::kStage;
            const uint32_t sb = sa + L::kA;
            const int k0 = kt * kUnBK;
            // A: 128 rows x 8 chunks
#pragma unroll
            for (int i = 0; i < (kUnRows * 8) / (kUnWarps * 32); ++i) {
                const int q = tid + i * kUnWarps * 32;
                const int r = q >> 3, ch = q & 7;
                const int k = k0 + ch * 8;
                const int v = s_uid[r];
                const bool ok = v >= 0 && k < d;
                const uint16_t *src = ok ? a.h.W + size_t(v) * d + k : a.h.W;
                cp_async16(sa + swz(r, ch), src, ok ? 16 : 0);
            }
            // B: NT*8 head rows x 8 chunks
            for (int q = tid; q < NT * 8 * 8; q += kUnWarps * 32) {
                const int r = q >> 3, ch = q & 7;
                const int k = k0 + ch * 8;
                const bool ok = r < R && k < d;
                const uint16_t *src = ok ? a.h.H + size_t(r) * d + k : a.h.H;
                cp_async16(sb + swz(r, ch), src, ok ? 16 : 0);
            }
        };

        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

#pragma unroll
        for (int s = 0; s < kUnStages - 1; ++s) {
            if (s < KT) load_slab(s, s);
            cp_async_commit();
        }
        for (int kt = 0; kt < KT; ++kt) {
            cp_async_wait<kUnStages - 2>();
            __syncthreads();
            const int nk = kt + kUnStages - 1;
            if (nk < KT) load_slab(nk % kUnStages, nk);
            cp_async_commit();
            const uint32_t sa = s_base + (kt % kUnStages) * L::kStage;
            const uint32_t sb = sa + L::kA;
#pragma unroll
            for (int ks = 0; ks < kUnBK / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                {
                    const int r = warp * 16 + (lane & 15);
                    const int ch = ks * 2 + (lane >> 4);
                    ldsm_x4(sa + swz(r, ch), a0, a1, a2, a3);
                }
#pragma unroll
                for (int j = 0; j + 1 < NT; j += 2) {
                    uint32_t b0, b1, b2, b3;
                    const int r = (j + (lane >> 4)) * 8 + (lane & 7);
                    const int ch = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x4(sb + swz(r, ch), b0, b1, b2, b3);
                    mma_bf16(acc[j], a0, a1, a2, a3, b0, b1);
                    mma_bf16(acc[j + 1], a0, a1, a2, a3, b2, b3);
                }
                if (NT & 1) {
                    uint32_t b0, b1;
                    const int r = (NT - 1) * 8 + (lane & 7);
                    const int ch = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x2(sb + swz(r, ch), b0, b1);
                    mma_bf16(acc[NT - 1], a0, a1, a2, a3, b0, b1);
                }
            }
        }
        cp_async_wait<0>();

        // Epilogue: keep (W row, head row) pairs whose list selects the row's cluster.
        const int rl0 = warp * 16 + (lane >> 2);
        int vv[2], cc[2], rk[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) { vv[e] = s_uid[rl0 + 8 * e]; cc[e] = s_ucl[rl0 + 8 * e]; rk[e] = s_rnk[rl0 + 8 * e]; }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = j * 8 + (lane & 3) * 2 + q;      // head row
                Stat st = stat_empty();
                if (n < R) {
                    const int b = n / G, gi = n - b * G;
                    const int off = a.h.vs_offsets[b];
                    const int nb = a.h.vs_offsets[b + 1] - off;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (vv[e] < 0) continue;
                        const int p = a.cpos[size_t(b) * M + cc[e]];
                        if (p < 0) continue;
                        const int jj = p + rk[e];
                        const float l = acc[j][2 * e + q];
                        a.h.logits[int64_t(off) * G + int64_t(gi) * nb + jj] = l;
                        const float x = l * a.h.inv_te;
                        const float key = a.h.T > 0.f ? x + gumbel(a.h.seed, uint32_t(vv[e]), uint32_t(a.h.pos), uint32_t(n)) : l;
                        stat_add(st, x, key, vv[e], jj);
                    }
                }
                // combine the 8 lanes that hold this column (lane bits 2..4), in lane order
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    const Stat other = shfl_xor_stat(st, o);
                    st = (lane & o) ? stat_merge(other, st) : stat_merge(st, other);
                }
                if (lane < 4 && n < R) {
                    Stat &dst = s_stat[warp * NT * 8 + n];
                    dst = stat_merge(dst, st);
                }
            }
        }
    }
    __syncthreads();
    for (int n = tid; n < R; n += blockDim.x) {
        Stat c = s_stat[n];
        for (int w = 1; w < kUnWarps; ++w) c = stat_merge(c, s_stat[w * NT * 8 + n]);
        partials[size_t(n) * gridDim.x + blockIdx.x] = c;
    }
}

// One warp per head row: fold the union kernel's per-block partials in a fixed order.
__global__ void head_union_finalize_kernel(HeadArgs a, int R, int nblocks, const Stat *__restrict__ partials)
{
    const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (n >= R) return;
    Stat c = stat_empty();
    for (int i = lane; i < nblocks; i += 32) c = stat_merge(c, partials[size_t(n) * nblocks + i]);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const Stat other = shfl_xor_stat(c, o);
        c = (lane & o) ? stat_merge(other, c) : stat_merge(c, other);
    }
    if (lane == 0) write_row(a, n, c);
}

}  // namespace
}  // namespace ds

using namespace ds;

namespace {

constexpr size_t kHeadPartialsPerRow = 1024;   // >= kGvMaxBlocks and >= any union grid

template <int NT>
ds_status launch_union(const UnionArgs &ua, Stat *partials, cudaStream_t stream, int *grid_out)
{
    const size_t smem = UnionSmem<NT>::kBytes;
    static int occ = -1;
    if (occ < 0) {
        if (cudaFuncSetAttribute(head_union_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return DS_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, head_union_kernel<NT>, kUnWarps * 32, smem) != cudaSuccess)
            return DS_ERR_CUDA;
        occ = o > 0 ? o : 1;
    }
    int grid = num_sms() * occ;
    if (grid > int(kHeadPartialsPerRow)) grid = int(kHeadPartialsPerRow);
    head_union_kernel<NT><<<grid, kUnWarps * 32, smem, stream>>>(ua, partials);
    DS_TRY_LAUNCH();
    *grid_out = grid;
    return DS_OK;
}

}  // namespace

extern "C" size_t ds_head_workspace_bytes(int rows)
{
    if (rows <= 0) return 0;
    return align256(size_t(rows) * sizeof(unsigned)) +
           align256(size_t(rows) * kHeadPartialsPerRow * sizeof(Stat));
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

    unsigned *counters = static_cast<unsigned *>(ws);
    Stat *partials = reinterpret_cast<Stat *>(static_cast<char *>(ws) + align256(size_t(rows) * sizeof(unsigned)));

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
    UnionArgs ua;
    ua.h = a; ua.B = B; ua.G = G; ua.R = int(rows); ua.M = M;
    ua.cpos = cpos; ua.rank = rank_in_cluster;
    ua.union_ids = union_ids; ua.union_cluster = union_cluster; ua.union_count = union_count;
    int grid = 0;
    ds_status st;
    if (rows <= 16) st = launch_union<2>(ua, partials, stream, &grid);
    else if (rows <= 32) st = launch_union<4>(ua, partials, stream, &grid);
    else if (rows <= 64) st = launch_union<8>(ua, partials, stream, &grid);
    else if (rows <= 80) st = launch_union<10>(ua, partials, stream, &grid);
    else st = launch_union<16>(ua, partials, stream, &grid);
    if (st != DS_OK) return st;
    head_union_finalize_kernel<<<(int(rows) + 7) / 8, 256, 0, stream>>>(a, int(rows), grid, partials);
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
constexpr size_t kNoAllocBytes = 256 + size_t(kNoAllocMaxRows) * kHeadPartialsPerRow * sizeof(Stat);
static_assert(256 >= kNoAllocMaxRows * sizeof(unsigned), "counter block");

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
    if (cudaMemsetAsync(scratch, 0, 256, stream) != cudaSuccess) return DS_ERR_CUDA;
    return ds_gathered_head(H, B, G, W, V, d, vs_offsets, vs_ids, cpos, M, rank_in_cluster,
                            union_ids, union_cluster, union_count, T, seed, pos,
                            logits, row_max, row_sumexp, token, token_idx,
                            scratch, kNoAllocBytes, dev_status, stream);
}
