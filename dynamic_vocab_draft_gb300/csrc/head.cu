// Gathered LM head: logits over the shortlist only, fused with the softmax statistics and
// the greedy / Gumbel-max draft draw.
//
// DynaSpec summary, Technical Details > System Modules "Gathered LM Head" (a fused index-
// select + GEMM) and Novel Architectural Elements ("Dynamic Vocabulary Head": the selected rows
// are gathered and multiplied with no intermediate copy in memory); Limitations: the gathered
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
#include "tc_gemm.cuh"

namespace ds {
namespace {

// ---------------------------------------------------------------------------------------
// Per-row gathered GEMV
// ---------------------------------------------------------------------------------------
constexpr int kGvWarps = 16;           // one 512-thread block per SM
constexpr int kHeadSideSms = 8;        // SMs a tensor-core (union) head leaves to the side stream
// SMs the batch-1 head leaves to the side stream.  The router of position t+2 runs there while
// head t+1 streams W (it reads H_{t+1}, which exists only once head t has drawn its token); both
// stream from the same saturated HBM, so the router's share of it follows its share of the SMs,
// and with 8 SMs its 10.5 MB took longer than the later, shorter heads (measured on one GB300:
// step 349.5 us with 8, 325.5 with 12, 318.9 with 16, 319.1 with 24 SMs).
constexpr int kHeadSideSmsB1 = 16;
constexpr int kGvMaxD = 16384;
constexpr int kGvMaxBlocks = 1024;     // per list; bounds the partials in the workspace

// SMs a head launch uses: all but `free_sms` (the caller's choice) or, for free_sms < 0, all but
// the path's default reserve.  At least one.
int head_sms(int sms, int free_sms, int default_free)
{
    const int f = free_sms < 0 ? default_free : free_sms;
    return sms - f < 1 ? 1 : sms - f;
}

struct HeadArgs {
    const uint16_t *H;
    const uint16_t *W;
    int V, d;
    const int32_t *vs_offsets, *vs_ids;
    // batch 1 without copied ids: the list's table (tk selected clusters: {list start, CSR start},
    // then {list size, 0}) and the CSR tokens; used instead of vs_offsets / vs_ids when set
    const int2 *table;
    int tk;
    const int32_t *csr_tok;
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

// A warp takes whole rows: the 16 16-byte loads per lane that cover 4096 columns of its row
// are issued together (8 KB of one row in flight per warp, ~128 KB per SM with 16 warps), then
// multiplied against h, which sits in shared memory as bf16 (one 16-byte load gives the 8
// values a W vector meets).  Rows longer than 4096 columns take several such rounds.
//
// The warp's rows come in batches of 32: lane l loads the id of the batch's row l and computes
// its Gumbel noise up front (all lanes at once), the rows then stream with their ids already in
// registers, lane l keeps row l's logit, and after the batch every lane folds its own row into
// its softmax/draw state -- no lane works alone per row.
//
// grid (gx, B): block (x, b) handles rows j = x*16 + warp, step gx*16, of list b.
constexpr int kGvMaxTable = 8193;      // list-table entries: up to 8192 selected clusters + the end
constexpr int kGvU = 16;               // loads per lane per round (4096 bf16)
constexpr int kGvRound = kGvU * 256;
constexpr int kGvFold = 8;             // block partials a lane of the last block loads at once

__global__ void __launch_bounds__(kGvWarps * 32, 1)
head_gemv_kernel(HeadArgs a, Stat *__restrict__ partials, unsigned *__restrict__ counters)
{
    extern __shared__ uint4 hs[];                 // h as bf16, d / 8 vectors; then the list table
    __shared__ Stat warp_stat[kGvWarps];
    pdl_allow();                                  // a verification launched next may get ready
    const int b = blockIdx.y;
    const int d = a.d;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // h's first 8 * blockDim columns are requested before anything else: the list's offsets,
    // then its ids, then the first W rows form a chain of dependent loads, and h's load (which
    // needs none of them) should not wait behind it
    const uint4 *h = reinterpret_cast<const uint4 *>(a.H + size_t(b) * d);
    const uint4 h0 = int(threadIdx.x) < d / 8 ? h[threadIdx.x] : make_uint4(0, 0, 0, 0);
    int2 *tab = reinterpret_cast<int2 *>(hs + d / 8);
    int base, n;
    if (a.table) {
        // the table takes the place of the offsets in the chain: staged once, then searched
        for (int s = threadIdx.x; s <= a.tk; s += blockDim.x) tab[s] = a.table[s];
        __syncthreads();
        base = 0;
        n = tab[a.tk].x;
    } else {
        base = a.vs_offsets[b];
        n = a.vs_offsets[b + 1] - base;
    }
    const int32_t *ids = a.vs_ids ? a.vs_ids + base : nullptr;
    // token id of list entry j: the copied list, or the CSR slice of the selected cluster whose
    // list start is the last one <= j (binary search over the table)
    auto row_id = [&](int j) -> int {
        if (!a.table) return ids[j];
        int lo = 0, hi = a.tk;                        // tab[lo].x <= j < tab[hi].x
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tab[mid].x <= j) lo = mid; else hi = mid;
        }
        const int q = tab[lo].y + (j - tab[lo].x);
        return unsigned(q) < unsigned(a.V) ? a.csr_tok[q] : -1;    // -1: reported as a bad id
    };
    float *lout = a.logits + base;
    const int stride = gridDim.x * kGvWarps;
    Stat st = stat_empty();

    auto load_round = [&](uint4 (&w)[kGvU], const uint4 *row, int k0) {
#pragma unroll
        for (int u = 0; u < kGvU; ++u) {
            const int k = k0 + (u * 32 + lane) * 8;
            w[u] = k < d ? ld_stream(row + (k >> 3)) : make_uint4(0, 0, 0, 0);
        }
    };
    const int j0 = blockIdx.x * kGvWarps + warp;  // the warp's rows: j0 + i * stride
    // the first batch's ids, and the first row's first round, are requested before h is staged
    int my_v = j0 + lane * stride < n ? row_id(j0 + lane * stride) : -1;
    uint4 w[kGvU];
    bool preloaded = false;
    if (j0 < n) {
        const int v = __shfl_sync(0xFFFFFFFFu, my_v, 0);
        const bool ok = v >= 0 && v < a.V;
        load_round(w, reinterpret_cast<const uint4 *>(a.W + size_t(ok ? v : 0) * d), 0);
        preloaded = true;
    }
    if (int(threadIdx.x) < d / 8) hs[threadIdx.x] = h0;
    for (int k = threadIdx.x + blockDim.x; k < d / 8; k += blockDim.x) hs[k] = h[k];
    __syncthreads();

    for (int jb = j0; jb < n; jb += 32 * stride) {
        // this batch: lane l owns row jb + l * stride
        const int my_j = jb + lane * stride;
        const bool my_ok = my_j < n && my_v >= 0 && my_v < a.V;
        float my_gum = 0.f, my_acc = 0.f;
        if (a.T > 0.f && my_ok) my_gum = gumbel(a.seed, uint32_t(my_j), uint32_t(a.pos), uint32_t(b));
        const int nrows = min(32, (n - jb + stride - 1) / stride);
        // ids of the next batch, one batch ahead
        const int nj = my_j + 32 * stride;
        const int next_v = nj < n ? row_id(nj) : -1;
        for (int k = 0; k < nrows; ++k) {
            const int v = __shfl_sync(0xFFFFFFFFu, my_v, k);
            const bool ok = v >= 0 && v < a.V;
            const uint4 *row = reinterpret_cast<const uint4 *>(a.W + size_t(ok ? v : 0) * d);
            float a0 = 0.f, a1 = 0.f;
            for (int k0 = 0; k0 < d; k0 += kGvRound) {
                if (!preloaded) load_round(w, row, k0);
                preloaded = false;
#pragma unroll
                for (int u = 0; u < kGvU; ++u) {
                    const int kk = k0 + (u * 32 + lane) * 8;
                    if (kk < d) {
                        const uint4 x = hs[kk >> 3];
                        a0 = fmaf(bf16lo(w[u].x), bf16lo(x.x), a0);
                        a1 = fmaf(bf16hi(w[u].x), bf16hi(x.x), a1);
                        a0 = fmaf(bf16lo(w[u].y), bf16lo(x.y), a0);
                        a1 = fmaf(bf16hi(w[u].y), bf16hi(x.y), a1);
                        a0 = fmaf(bf16lo(w[u].z), bf16lo(x.z), a0);
                        a1 = fmaf(bf16hi(w[u].z), bf16hi(x.z), a1);
                        a0 = fmaf(bf16lo(w[u].w), bf16lo(x.w), a0);
                        a1 = fmaf(bf16hi(w[u].w), bf16hi(x.w), a1);
                    }
                }
            }
            const float acc = warp_sum(a0 + a1);
            if (lane == k) my_acc = acc;
        }
        // every lane folds its own row of the batch
        if (my_j < n) {
            if (!my_ok) {
                set_status(a.status, DS_DEV_BAD_INDEX);
                lout[my_j] = 0.f;
            } else {
                lout[my_j] = my_acc;
                const float x = my_acc * a.inv_te;
                stat_add(st, x, a.T > 0.f ? x + my_gum : my_acc, my_v, my_j);
            }
        }
        my_v = next_v;
    }
    // the warp's lanes, then the block's warps, then the blocks (every step's result independent
    // of timing)
    st = stat_reduce_lanes(st);
    if (lane == 0) warp_stat[warp] = st;
    __syncthreads();
    if (warp == 0) {
        const Stat c = stat_reduce_lanes<kGvWarps>(lane < kGvWarps ? warp_stat[lane] : stat_empty());
        if (lane == 0) st_stat(&partials[size_t(b) * kGvMaxBlocks + blockIdx.x], c);
    }
    if (!last_block_done(&counters[b], gridDim.x)) return;
    if (warp != 0) return;
    // Final combine: lane l merges partials l, l+32, ... (their loads issued together, kGvFold
    // at a time), then the lanes.
    const Stat *pb = partials + size_t(b) * kGvMaxBlocks;
    Stat c = stat_empty();
    for (int i0 = lane; i0 < int(gridDim.x); i0 += 32 * kGvFold) {
        Stat q[kGvFold + 1];
        q[0] = c;
#pragma unroll
        for (int f = 0; f < kGvFold; ++f)
            q[f + 1] = i0 + 32 * f < int(gridDim.x) ? ld_stat(pb + i0 + 32 * f) : stat_empty();
        c = stat_merge_n(q);
    }
    c = stat_reduce_lanes(c);
    if (lane == 0) write_row(a, b, c);
}

// ---------------------------------------------------------------------------------------
// Union path: the tensor-core gathered-row GEMM over the union of the lists, every union row
// scored against all B*G head rows; the epilogue keeps the (row, token) pairs whose list
// selects the token's cluster and writes each at its place in that list.
// ---------------------------------------------------------------------------------------
constexpr int kUnMaxRows = 128;                 // head rows
constexpr int kUnionMaxTiles = 8192;            // union rows <= 8192 * 128

struct UnionEp {
    const int32_t *ids, *cluster, *count, *rank, *cpos, *vs_offsets;
    float *logits;
    int V, M, G;
    int32_t *status;

    __device__ int n_rows() const { return min(*count, V); }
    __device__ void pick(int u, int &v, int &c) const
    {
        v = ids[u];
        c = cluster[u];
        if (v < 0 || v >= V || c < 0 || c >= M) { set_status(status, DS_DEV_BAD_INDEX); v = -1; c = -1; }
    }
    // head row r: its list b and the logits index of entry 0 of its part of that list
    __device__ void col_info(int r, int &b, long long &base) const
    {
        b = r / G;
        const int gi = r - b * G, off = vs_offsets[b], nb = vs_offsets[b + 1] - off;
        base = 1LL * off * G + 1LL * gi * nb;
    }
    __device__ int row_aux(int v) const { return v >= 0 ? __ldg(rank + v) : 0; }
    using State = tc::NoState;
    __device__ void finish(State &) const {}
    // logits of union row v (cluster c, rank rk in it) against head rows cb .. cb+15
    __device__ void emit(State &, const float (&x)[16], int cb, int v, int c, int rk,
                         const int32_t *s_b, const long long *s_base) const
    {
        if (v < 0) return;
        int pcs[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int b = s_b[cb + e];
            pcs[e] = b >= 0 ? __ldg(cpos + size_t(b) * M + c) : -1;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if (pcs[e] >= 0) logits[s_base[cb + e] + pcs[e] + rk] = x[e];
    }
};

// Softmax statistics and the draft draw of every head row from its stored logits.
// grid (X, R): block (x, r) folds chunks x, x + X, ... of kRsChunk elements of row r; the last
// block of the row combines the partials in a fixed order.  X is chosen on the host so that the
// grid fills the GPU about once (kRsBlocksPerSm blocks per SM) whatever the number of rows;
// blocks past the end of their row's list leave at once and take no part in the fold (block 0
// stays for an empty list).
constexpr int kRsPer = 4;
constexpr int kRsChunk = 256 * kRsPer;
constexpr int kRsBlocksPerSm = 8;

__global__ void __launch_bounds__(256)
head_rowstats_kernel(HeadArgs a, int G, Stat *__restrict__ partials, unsigned *__restrict__ counters)
{
    __shared__ Stat ws[8];
    pdl_allow();                                  // a verification launched next may get ready
    const int r = blockIdx.y, b = r / G, gi = r - b * G;
    const int off = a.vs_offsets[b];
    const int n = a.vs_offsets[b + 1] - off;
    const int nch = n > 0 ? (n + kRsChunk - 1) / kRsChunk : 1;
    const int nblk = min(nch, int(gridDim.x));
    if (int(blockIdx.x) >= nblk) return;                   // uniform over the block
    const float *l = a.logits + int64_t(off) * G + int64_t(gi) * n;
    const int32_t *ids = a.vs_ids + off;
    static_assert(kRsPer % 4 == 0, "whole noise blocks per thread and chunk");
    // a thread's entries: 16-byte loads of each array where both rows are aligned
    const bool vec = ((reinterpret_cast<uintptr_t>(l) | reinterpret_cast<uintptr_t>(ids)) & 15u) == 0;
    auto load = [&](int ch, float (&lv)[kRsPer], int (&iv)[kRsPer]) {
        const int j0 = ch * kRsChunk + threadIdx.x * kRsPer;
        if (vec && j0 + kRsPer <= n) {
#pragma unroll
            for (int q = 0; q < kRsPer / 4; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(l + j0 + 4 * q);
                const int4 t = *reinterpret_cast<const int4 *>(ids + j0 + 4 * q);
                lv[4 * q] = f.x; lv[4 * q + 1] = f.y; lv[4 * q + 2] = f.z; lv[4 * q + 3] = f.w;
                iv[4 * q] = t.x; iv[4 * q + 1] = t.y; iv[4 * q + 2] = t.z; iv[4 * q + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < kRsPer; ++e) {
                lv[e] = j0 + e < n ? l[j0 + e] : 0.f;
                iv[e] = j0 + e < n ? ids[j0 + e] : 0;
            }
        }
    };
    Stat st = stat_empty();
    // the next chunk's loads are in flight while this one is folded
    float lv[kRsPer];
    int iv[kRsPer];
    load(blockIdx.x, lv, iv);
    for (int ch = blockIdx.x; ch < nch; ch += gridDim.x) {
        float lc[kRsPer];
        int ic[kRsPer];
#pragma unroll
        for (int e = 0; e < kRsPer; ++e) { lc[e] = lv[e]; ic[e] = iv[e]; }
        if (ch + int(gridDim.x) < nch) load(ch + int(gridDim.x), lv, iv);
        const int j0 = ch * kRsChunk + threadIdx.x * kRsPer;   // a multiple of 4
#pragma unroll
        for (int q = 0; q < kRsPer / 4; ++q) {
            // four consecutive entries share one Philox block
            const int jq = j0 + 4 * q;
            uint4 wq = make_uint4(0u, 0u, 0u, 0u);
            if (a.T > 0.f && jq < n) wq = gumbel_block(a.seed, uint32_t(jq) >> 2, uint32_t(a.pos), uint32_t(r));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = jq + e;
                if (j < n) {
                    const float x = lc[4 * q + e] * a.inv_te;
                    const float key = a.T > 0.f ? x + gumbel_from_word(word_of(wq, uint32_t(e))) : lc[4 * q + e];
                    stat_add(st, x, key, ic[4 * q + e], j);
                }
            }
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    st = stat_reduce_lanes(st);
    if (lane == 0) ws[warp] = st;
    __syncthreads();
    if (warp == 0) {
        const Stat c = stat_reduce_lanes<8>(lane < 8 ? ws[lane] : stat_empty());
        if (lane == 0) st_stat(&partials[size_t(r) * kGvMaxBlocks + blockIdx.x], c);
    }
    if (!last_block_done(&counters[r], unsigned(nblk))) return;
    if (warp != 0) return;
    // lane l merges partials l, l+32, ... (their loads issued together, kGvFold at a time)
    const Stat *pr = partials + size_t(r) * kGvMaxBlocks;
    Stat c = stat_empty();
    for (int i0 = lane; i0 < nblk; i0 += 32 * kGvFold) {
        Stat q[kGvFold + 1];
        q[0] = c;
#pragma unroll
        for (int f = 0; f < kGvFold; ++f) q[f + 1] = i0 + 32 * f < nblk ? ld_stat(pr + i0 + 32 * f) : stat_empty();
        c = stat_merge_n(q);
    }
    c = stat_reduce_lanes(c);
    if (lane == 0) write_row(a, r, c);
}

// The per-row head's dynamic shared memory: h (d bf16) and, with a list table, the table.
bool head_smem_limit()
{
    static std::atomic<unsigned long long> smem_set{0};
    return smem_limit_once(head_gemv_kernel, size_t(kGvMaxD) * sizeof(uint16_t) + size_t(kGvMaxTable) * sizeof(int2),
                           smem_set);
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
    w.total = w.parts + align256(tc::parts_bytes(rows, tc::kMaxGrid));
    return w;
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
                                      int32_t *token, int32_t *token_idx, int free_sms,
                                      void *ws, size_t ws_bytes, int32_t *dev_status,
                                      cudaStream_t stream)
{
    ds::NvtxRange range("ds_gathered_head");
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
    a.table = nullptr; a.tk = 0; a.csr_tok = nullptr;
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.seed = seed; a.pos = pos;
    a.logits = logits; a.row_max = row_max; a.row_sumexp = row_sumexp;
    a.token = token; a.token_idx = token_idx;
    a.status = dev_status;

    if (nu == 0) {
        if (G != 1) return DS_ERR_UNSUPPORTED;
        const int sms = sm_count();
        if (sms <= 0) return DS_ERR_CUDA;
        // One 512-thread block per SM.  At batch 1 a few SMs are left to the side stream, so the
        // next position's router and shortlist build run while this head streams W.
        const int use = head_sms(sms, free_sms, B == 1 ? kHeadSideSmsB1 : 0);
        int gx = B == 1 ? use : (use + B - 1) / B;
        if (gx < 1) gx = 1;
        if (gx > kGvMaxBlocks) gx = kGvMaxBlocks;
        const size_t smem = size_t(d) * sizeof(uint16_t);
        if (!head_smem_limit()) return DS_ERR_CUDA;
        head_gemv_kernel<<<dim3(gx, B), kGvWarps * 32, smem, stream>>>(a, partials, counters);
        DS_TRY_LAUNCH();
        return DS_OK;
    }

    if (!cpos || !rank_in_cluster || M < 1) return DS_ERR_INVALID_ARG;
    if (rows > kUnMaxRows) return DS_ERR_UNSUPPORTED;
    if ((V + kRsChunk - 1) / kRsChunk > kGvMaxBlocks) return DS_ERR_UNSUPPORTED;
    if ((V + tc::kRows - 1) / tc::kRows > kUnionMaxTiles) return DS_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    float *parts = reinterpret_cast<float *>(wsb + lay.parts);
    unsigned *tile_cnt = reinterpret_cast<unsigned *>(wsb + lay.tile_cnt);
    UnionEp ep;
    ep.ids = union_ids; ep.cluster = union_cluster; ep.count = union_count;
    ep.rank = rank_in_cluster; ep.cpos = cpos; ep.vs_offsets = vs_offsets;
    ep.logits = logits; ep.V = V; ep.M = M; ep.G = G; ep.status = dev_status;
    // A tensor-core head CTA fills its SM (shared memory and registers); kHeadSideSms SMs are
    // left free so the next position's router and shortlist build run beside it.
    int tc_grid = head_sms(sms, free_sms, kHeadSideSms);
    if (tc_grid > tc::kMaxGrid) tc_grid = tc::kMaxGrid;
    if (tc_grid < 1) tc_grid = 1;
    const tc::Operands op{W, H, d, int(rows), dev_status, wait_budget()};
    const ds_status st = tc::launch_for(op, ep, parts, tile_cnt, tc_grid, stream);
    if (st != DS_OK) return st;
    // about kRsBlocksPerSm blocks per SM in all, spread over the rows (at most one per chunk of
    // the longest possible list)
    const int chunks = (V + kRsChunk - 1) / kRsChunk;
    int gx = int((long long)sms * kRsBlocksPerSm / rows);
    gx = gx < 1 ? 1 : gx > chunks ? chunks : gx;
    if (gx > kGvMaxBlocks) gx = kGvMaxBlocks;             // the partials a row has room for
    head_rowstats_kernel<<<dim3(gx, unsigned(rows)), 256, 0, stream>>>(a, G, partials, counters);
    DS_TRY_LAUNCH();
    return DS_OK;
}

// ---------------------------------------------------------------------------------------
// ds_gathered_head_noalloc: the same head for callers that cannot give the library any
// scratch memory.  The cross-block partials and completion counters live in one file-scope
// device array of fixed size instead of a caller workspace.
// ---------------------------------------------------------------------------------------
#include <mutex>

#include <cuda.h>      // CUcontext / CUresult types only: the two CUDA driver API calls below are
                       // reached through the runtime's entry-point query, so the library does not
                       // link the CUDA driver library

namespace {

constexpr int kNoAllocMaxRows = 32;
// head_ws_layout(32), spelled out so the array can be sized at compile time
constexpr size_t kNoAllocCounters = 256 + size_t(kUnionMaxTiles) * sizeof(unsigned);
constexpr size_t kNoAllocBytes = kNoAllocCounters + size_t(kNoAllocMaxRows) * kHeadPartialsPerRow * sizeof(Stat) +
                                 size_t(2) * tc::kMaxGrid * tc::kRows * 32 * sizeof(float);
static_assert(256 >= kNoAllocMaxRows * sizeof(unsigned), "counter block");
static_assert(kNoAllocCounters % 256 == 0 && (size_t(kNoAllocMaxRows) * kHeadPartialsPerRow * sizeof(Stat)) % 256 == 0,
              "no padding between the regions");

// Held by every GPU that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_head_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kNoAllocMaxDevices];
unsigned long long g_noalloc_ctx[kNoAllocMaxDevices];   // context the address belongs to

// Unique id of the calling thread's current context (the CUDA driver never reuses one within a
// process), or 0 when none is current or the CUDA driver calls cannot be reached.
unsigned long long current_context_id()
{
    typedef CUresult (*GetCurrent)(CUcontext *);
    typedef CUresult (*GetId)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {                                   // under g_noalloc_mutex
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrent>(f1);
            get_id = reinterpret_cast<GetId>(f2);
        }
        (void)cudaGetLastError();
        resolved = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on the current device.  It is looked up once per device
// and context: a reset of the device (cudaDeviceReset) destroys the context and the array with
// it, and the next call looks the address up again in the new context instead of using a stale
// one.  (In host code the array's name is only a host-side stand-in, not a device address.)
ds_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DS_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return DS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_addr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        void *p = nullptr;
        // the lookup also makes the device's primary context current if no context was yet
        if (cudaGetSymbolAddress(&p, g_head_noalloc_scratch) != cudaSuccess || !p) return DS_ERR_CUDA;
        g_noalloc_addr[dev] = p;
        g_noalloc_ctx[dev] = current_context_id();
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
                                              int32_t *token, int32_t *token_idx, int free_sms,
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
                            logits, row_max, row_sumexp, token, token_idx, free_sms,
                            scratch, kNoAllocBytes, dev_status, stream);
}

// ---------------------------------------------------------------------------------------
// ds_prefetch_rows: bring the W rows a list names first into L2 ahead of the head that reads
// them.  A draft position's list is known before the previous position's head has finished (its
// router runs beside that head), and its W rows do not depend on the token that head draws, so
// they can be fetched while that head's last rows stream and HBM has room to spare.  Marked
// evict-last so the rest of the running head's stream does not push them out first; the head's
// own loads, which carry no hint, read them back at normal priority.
// ---------------------------------------------------------------------------------------
namespace ds {
namespace {
__global__ void prefetch_rows_kernel(const uint16_t *__restrict__ W, int V, int d, const int32_t *__restrict__ ids,
                                     const int32_t *__restrict__ offsets, int first)
{
    const int lo = offsets[0];
    const int n = min(offsets[1] - lo, first);
    const int lane = threadIdx.x & 31;
    const int lines = (d * 2 + 127) / 128;                 // 128-byte lines per row
    for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < n; j += gridDim.x * (blockDim.x >> 5)) {
        const int v = ids[lo + j];
        if (v < 0 || v >= V) continue;
        const char *row = reinterpret_cast<const char *>(W + size_t(v) * d);
        for (int l = lane; l < lines; l += 32)
            asm volatile("prefetch.global.L2::evict_last [%0];" :: "l"(row + size_t(l) * 128));
    }
}
}  // namespace
}  // namespace ds

extern "C" ds_status ds_prefetch_rows(const uint16_t *W, int V, int d, const int32_t *ids, const int32_t *offsets,
                                      int first_rows, int blocks, cudaStream_t stream)
{
    ds::NvtxRange range("ds_prefetch_rows");
    if (!W || !ids || !offsets || V < 1 || d < 8 || d % 8 || first_rows < 0 || blocks < 0) return DS_ERR_INVALID_ARG;
    if (first_rows == 0) return DS_OK;
    const int g = blocks > 0 ? blocks : 64;
    prefetch_rows_kernel<<<g, 256, 0, stream>>>(W, V, d, ids, offsets, first_rows);
    DS_TRY_LAUNCH();
    return DS_OK;
}

// Batch 1 with the list's table (ds_router_topk_list_b1) instead of copied ids: the same head,
// each listed token found through the table and the CSR.
extern "C" ds_status ds_gathered_head_b1_table(const uint16_t *H, const uint16_t *W, int V, int d,
                                               const int32_t *list_table, int k, const int32_t *csr_tok,
                                               float T, uint64_t seed, int pos,
                                               float *logits, float *row_max, float *row_sumexp,
                                               int32_t *token, int32_t *token_idx, int free_sms,
                                               void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_gathered_head_b1_table");
    if (!H || !W || !list_table || !csr_tok || !logits || !token || !token_idx) return DS_ERR_INVALID_ARG;
    if (V < 1 || d < 8 || d % 8 || k < 1 || !(T >= 0.f) || pos < 0) return DS_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(W) || (reinterpret_cast<uintptr_t>(list_table) & 7u)) return DS_ERR_INVALID_ARG;
    if (d > kGvMaxD || k + 1 > kGvMaxTable) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_head_workspace_bytes(1)) return DS_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    const HeadWs lay = head_ws_layout(1);
    char *wsb = static_cast<char *>(ws);
    HeadArgs a;
    a.H = H; a.W = W; a.V = V; a.d = d;
    a.vs_offsets = nullptr; a.vs_ids = nullptr;
    a.table = reinterpret_cast<const int2 *>(list_table); a.tk = k; a.csr_tok = csr_tok;
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.seed = seed; a.pos = pos;
    a.logits = logits; a.row_max = row_max; a.row_sumexp = row_sumexp;
    a.token = token; a.token_idx = token_idx;
    a.status = dev_status;
    int gx = head_sms(sms, free_sms, kHeadSideSmsB1);
    if (gx > kGvMaxBlocks) gx = kGvMaxBlocks;
    if (!head_smem_limit()) return DS_ERR_CUDA;
    const size_t smem = size_t(d) * sizeof(uint16_t) + size_t(k + 1) * sizeof(int2);
    head_gemv_kernel<<<dim3(gx, 1), kGvWarps * 32, smem, stream>>>(
        a, reinterpret_cast<Stat *>(wsb + lay.partials), reinterpret_cast<unsigned *>(wsb + lay.row_cnt));
    DS_TRY_LAUNCH();
    return DS_OK;
}
