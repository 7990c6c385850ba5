// Router MLP and position-aware top-k cluster selection.
//
// DynaSpec summary ("DynaSpec: Context-aware Dynamic Speculative Sampling for Large-
// Vocabulary Language Models"), Technical Details > System Modules "Router (Meta-
// Classifier)": a 2-layer MLP scoring vocabulary clusters from the drafter hidden state
// H_{t-1}; Key Hyperparameters: ReLU, and a budget k_c(t) that decays with draft position t;
// abstract: the shortlist is made of the tokens of the best-scoring clusters.
//
// Both layers are GEMV-shaped and HBM-bound at the batch sizes of drafting (one weight row
// feeds at most a few dozen hidden states), so they run on CUDA cores: one warp per weight
// row, 16-byte streaming loads, the hidden states staged once per block in shared memory,
// warp-shuffle reductions.  Top-k is an exact MSB-first radix select on order-preserving
// 32-bit keys followed by two block scans (ties to the lower cluster id, output ascending).
#include "common.cuh"
#include "block_scan.cuh"
#include "tc_gemm.cuh"

namespace ds {
namespace {

constexpr int kGemvWarps = 8;          // rows per block
constexpr int kGemvU = 16;             // 16-byte loads in flight per lane per pass
constexpr int kGemvBT = 4;             // hidden states per block (batched); 1 at batch 1
constexpr int kRouterMaxK = 8192;      // inner dimension the staging buffer allows

__device__ __forceinline__ float act_fn(float x, int act)
{
    if (act == DS_ACT_RELU) return fmaxf(x, 0.f);
    if (act == DS_ACT_GELU) return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
    return x;
}

template <typename XT> __device__ __forceinline__ float load_x(const XT *p);
template <> __device__ __forceinline__ float load_x<uint16_t>(const uint16_t *p) { return bf16_to_f32(*p); }
template <> __device__ __forceinline__ float load_x<float>(const float *p) { return *p; }

// y[b][i] = act(sum_k A[i][k] x[b][k] + bias[i]) for i < N, b < B.
//   grid.x = ceil(N / kGemvWarps), grid.y = ceil(B / BT); dynamic smem = BT*K floats.
__device__ void topk_block(const float *__restrict__ s, int M, int k, int32_t *__restrict__ dst);

// With topk_k > 0 the last block of each batch tile to finish (completion counter per tile)
// also selects the top-k of the tile's finished rows, saving a launch per draft position.
template <typename XT, int BT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_rows_kernel(const uint16_t *__restrict__ A, int N, int K, const XT *__restrict__ x, int B,
                 const uint16_t *__restrict__ bias, int act, float *__restrict__ y,
                 int topk_k, int32_t *__restrict__ topk_ids, unsigned *__restrict__ counters)
{
    extern __shared__ float4 xs4[];
    float *xs = reinterpret_cast<float *>(xs4);
    const int b0 = blockIdx.y * BT;
    const int nb = min(BT, B - b0);
    for (int e = threadIdx.x; e < BT * K; e += blockDim.x) {
        const int bt = e / K, k = e - bt * K;
        xs[e] = bt < nb ? load_x<XT>(x + size_t(b0 + bt) * K + k) : 0.f;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
    if (i < N) {
    const uint4 *row = reinterpret_cast<const uint4 *>(A + size_t(i) * K);
    float acc[BT];
#pragma unroll
    for (int bt = 0; bt < BT; ++bt) acc[bt] = 0.f;

    for (int k0 = 0; k0 < K; k0 += kGemvU * 256) {
        uint4 w[kGemvU];
#pragma unroll
        for (int u = 0; u < kGemvU; ++u) {
            const int k = k0 + u * 256 + lane * 8;
            w[u] = k < K ? ld_stream(row + (k >> 3)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kGemvU; ++u) {
            const int k = k0 + u * 256 + lane * 8;
            if (k < K) {
#pragma unroll
                for (int bt = 0; bt < BT; ++bt) {
                    const float4 *xv = reinterpret_cast<const float4 *>(xs + bt * K + k);
                    acc[bt] = dot8(w[u], xv[0], xv[1], acc[bt]);
                }
            }
        }
    }
#pragma unroll
    for (int bt = 0; bt < BT; ++bt) acc[bt] = warp_sum(acc[bt]);
    if (lane < nb) {
        float a = acc[0];
#pragma unroll
        for (int bt = 1; bt < BT; ++bt) if (lane == bt) a = acc[bt];
        y[size_t(b0 + lane) * N + i] = act_fn(a + bf16_to_f32(bias[i]), act);
    }
    }
    if (topk_k > 0 && last_block_done(&counters[blockIdx.y], gridDim.x)) {
        for (int bt = 0; bt < nb; ++bt)
            topk_block(y + size_t(b0 + bt) * N, N, topk_k, topk_ids + size_t(b0 + bt) * topk_k);
    }
}

// Order-preserving key: a larger float maps to a larger unsigned key; +0 and -0 share a key.
__device__ __forceinline__ uint32_t order_key(float f)
{
    if (f == 0.f) f = 0.f;
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int kTopkThreads = 256;
constexpr int kTopkPerThread = kRouterMaxK / kTopkThreads;

// One block per row: keep the k largest of scores[b][0..M), ties to the lower index, and
// write their indices in ascending order.
// Keep the k largest of s[0..M), ties to the lower index, and write their indices to dst in
// ascending order.  Called by a whole block of kTopkThreads threads; s is read through L2 (other
// blocks may have written it).
__device__ void topk_block(const float *__restrict__ s, int M, int k, int32_t *__restrict__ dst)
{
    __syncthreads();                          // a previous call in this block is done with its state
    __shared__ unsigned hist[256];
    __shared__ int scan_scratch[33];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    // thread t owns the contiguous index range [t*E, t*E + E)
    const int E = (M + kTopkThreads - 1) / kTopkThreads;
    const int lo = threadIdx.x * E;
    uint32_t key[kTopkPerThread];
#pragma unroll
    for (int e = 0; e < kTopkPerThread; ++e)
        key[e] = (e < E && lo + e < M) ? order_key(__ldcg(s + lo + e)) : 0u;

    // MSB-first radix select of the k-th largest key, 8 bits per pass.
    if (threadIdx.x == 0) { s_prefix = 0u; s_need = k; }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (threadIdx.x < 256) hist[threadIdx.x] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        // Scores cluster in a few exponent bytes, so lanes with the same digit are combined
        // first (one shared-memory atomic per distinct digit per warp).
#pragma unroll
        for (int e = 0; e < kTopkPerThread; ++e) {
            if (e >= E) break;                               // E is uniform across the block
            const bool in = lo + e < M && (key[e] & mask) == prefix;
            const unsigned digit = in ? (key[e] >> shift) & 255u : 256u;
            const unsigned same = __match_any_sync(0xFFFFFFFFu, digit);
            if (in && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[digit], unsigned(__popc(same)));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // bins from the top: lane l owns digits 255-8l .. 248-8l
            const int lane = threadIdx.x;
            unsigned c[8], tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) { c[q] = hist[255 - 8 * lane - q]; tot += c[q]; }
            unsigned incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const int need = s_need;
            unsigned before = incl - tot;          // elements in higher digits than my range
            const bool mine = before < unsigned(need) && unsigned(need) <= incl;
            if (mine) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (before + c[q] >= unsigned(need)) {
                        s_prefix = prefix | (uint32_t(255 - 8 * lane - q) << shift);
                        s_need = need - int(before);
                        break;
                    }
                    before += c[q];
                }
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t theta = s_prefix;      // the k-th largest key
    const int need_eq = s_need;           // how many of the keys equal to theta to keep

    // Keep keys above theta, and the first need_eq keys equal to theta in index order.
    int eq = 0;
#pragma unroll
    for (int e = 0; e < kTopkPerThread; ++e)
        if (e < E && lo + e < M && key[e] == theta) ++eq;
    int tot;
    int eq_before = block_exclusive_scan(eq, scan_scratch, &tot);
    bool sel[kTopkPerThread];
    int nsel = 0;
#pragma unroll
    for (int e = 0; e < kTopkPerThread; ++e) {
        const bool valid = e < E && lo + e < M;
        bool keep = false;
        if (valid && key[e] > theta) keep = true;
        if (valid && key[e] == theta) { keep = eq_before < need_eq; ++eq_before; }
        sel[e] = keep;
        nsel += keep;
    }
    int out = block_exclusive_scan(nsel, scan_scratch, &tot);
#pragma unroll
    for (int e = 0; e < kTopkPerThread; ++e)
        if (sel[e] && out < k) dst[out++] = lo + e;
}

static_assert(kGemvWarps * 32 == kTopkThreads, "the GEMV block runs the top-k epilogue");

// The list of one batch-1 draft position without copying its token ids: after the top-k, the
// selected clusters' list starts and CSR starts (list_table[s] = {list start, CSR start} for the
// s-th selected cluster in ascending id, list_table[k] = {list size, 0}), cpos and the list's
// offsets.  The head finds a listed token through the table and the CSR.
struct ListOut {
    const int32_t *csr_off;
    int V;
    int2 *table;
    int32_t *cpos, *vs_offsets;
    int64_t capacity;
    int32_t *status;
};

// Called by the whole block that just wrote ids[0..k) (ascending cluster ids).
__device__ void list_table_block(const ListOut &o, const int32_t *ids, int k, int M)
{
    __shared__ int scratch[33];
    __syncthreads();                                   // this block's ids, to every thread
    for (int c = threadIdx.x; c < M; c += blockDim.x) o.cpos[c] = -1;
    // thread t owns the selected clusters j0 .. j0+E-1, in order
    const int E = (k + blockDim.x - 1) / blockDim.x;
    const int j0 = threadIdx.x * E, j1 = min(k, j0 + E);
    auto slice = [&](int c, int &lo) {
        lo = 0;
        if (c < 0 || c >= M) { set_status(o.status, DS_DEV_BAD_INDEX); return 0; }
        const int l0 = o.csr_off[c], hi = o.csr_off[c + 1];
        if (l0 < 0 || hi < l0 || hi > o.V) { set_status(o.status, DS_DEV_BAD_INDEX); return 0; }
        lo = l0;
        return hi - l0;
    };
    int sum = 0;
    for (int j = j0; j < j1; ++j) { int lo; sum += slice(ids[j], lo); }
    int tot;
    int run = block_exclusive_scan(sum, scratch, &tot);     // its barriers order the -1 pass first
    for (int j = j0; j < j1; ++j) {
        const int c = ids[j];
        int lo;
        const int n = slice(c, lo);
        o.table[j] = make_int2(run, lo);
        if (c >= 0 && c < M) o.cpos[c] = run;
        run += n;
    }
    if (threadIdx.x == 0) {
        // a list longer than the caller's logits is reported and read as empty
        const bool fits = int64_t(tot) <= o.capacity;
        if (!fits) set_status(o.status, DS_DEV_CAPACITY);
        o.table[k] = make_int2(fits ? tot : 0, 0);
        o.vs_offsets[0] = 0;
        o.vs_offsets[1] = fits ? tot : 0;
    }
}

// Batch 1: y[i] = act(A[i] . x + bias[i]).  No staging: every lane loads the slice of x its
// weight vectors meet, next to those weights.  Warps stride over rows, so a small grid covers
// the matrix in one wave -- the router of a later draft position runs on the few SMs the head
// leaves free.  Optional top-k epilogue as in gemv_rows_kernel.
template <typename XT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv1_kernel(const uint16_t *__restrict__ A, int N, int K, const XT *__restrict__ x,
             const uint16_t *__restrict__ bias, int act, float *__restrict__ y,
             int topk_k, int32_t *__restrict__ topk_ids, unsigned *__restrict__ counter, ListOut lout)
{
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * kGemvWarps;
    for (int i = blockIdx.x * kGemvWarps + (threadIdx.x >> 5); i < N; i += nw) {
        const uint4 *row = reinterpret_cast<const uint4 *>(A + size_t(i) * K);
        float a0 = 0.f, a1 = 0.f;
        for (int k0 = 0; k0 < K; k0 += kGemvU * 256) {
            uint4 w[kGemvU];
            float xv[kGemvU][8];
#pragma unroll
            for (int u = 0; u < kGemvU; ++u) {
                const int k = k0 + u * 256 + lane * 8;
                w[u] = k < K ? ld_stream(row + (k >> 3)) : make_uint4(0, 0, 0, 0);
                if (k < K) {
                    if constexpr (sizeof(XT) == 2) {
                        const uint4 q = *reinterpret_cast<const uint4 *>(x + k);
                        xv[u][0] = bf16lo(q.x); xv[u][1] = bf16hi(q.x); xv[u][2] = bf16lo(q.y); xv[u][3] = bf16hi(q.y);
                        xv[u][4] = bf16lo(q.z); xv[u][5] = bf16hi(q.z); xv[u][6] = bf16lo(q.w); xv[u][7] = bf16hi(q.w);
                    } else {
                        const float4 q0 = *reinterpret_cast<const float4 *>(x + k);
                        const float4 q1 = *reinterpret_cast<const float4 *>(x + k + 4);
                        xv[u][0] = q0.x; xv[u][1] = q0.y; xv[u][2] = q0.z; xv[u][3] = q0.w;
                        xv[u][4] = q1.x; xv[u][5] = q1.y; xv[u][6] = q1.z; xv[u][7] = q1.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[u][e] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kGemvU; ++u) {
                a0 = fmaf(bf16lo(w[u].x), xv[u][0], a0);
                a1 = fmaf(bf16hi(w[u].x), xv[u][1], a1);
                a0 = fmaf(bf16lo(w[u].y), xv[u][2], a0);
                a1 = fmaf(bf16hi(w[u].y), xv[u][3], a1);
                a0 = fmaf(bf16lo(w[u].z), xv[u][4], a0);
                a1 = fmaf(bf16hi(w[u].z), xv[u][5], a1);
                a0 = fmaf(bf16lo(w[u].w), xv[u][6], a0);
                a1 = fmaf(bf16hi(w[u].w), xv[u][7], a1);
            }
        }
        const float acc = warp_sum(a0 + a1);
        if (lane == 0) {
            y[i] = act_fn(acc + bf16_to_f32(bias[i]), act);
        }
    }
    if (topk_k > 0 && last_block_done(counter, gridDim.x)) {
        topk_block(y, N, topk_k, topk_ids);
        if (lout.table) list_table_block(lout, topk_ids, topk_k, N);
    }
}

constexpr int kGemv1PerSm = 4;         // a later position's router: four 256-thread blocks on each
constexpr int kGemv1SideSms = 16;      // SM the batch-1 head leaves free (by default 16)

// One block per row: the top-k of scores[b][0..M).
__global__ void __launch_bounds__(kTopkThreads)
topk_rows_kernel(const float *__restrict__ scores, int M, int k, int32_t *__restrict__ ids)
{
    topk_block(scores + size_t(blockIdx.x) * M, M, k, ids + size_t(blockIdx.x) * k);
}

// ---------------------------------------------------------------------------------------
// Batched router (2 <= B <= 64) on the tensor cores, through the gathered-row GEMM with every
// weight row picked in order.  Layer 1 multiplies W1 by the B bf16 hidden states; its
// epilogue adds b1, applies the activation and stores the fp32 result u as a pair of bf16
// values, hi = bf16(u) and lo = bf16(u - hi), which together carry about 16 significant bits
// (the relative error of hi + lo is below 2^-16).  Layer 2 multiplies W2 by the 2B vectors
// (hi_0, lo_0, hi_1, lo_1, ...) and adds each pair of columns, so the scores see u almost as
// the fp32 path does while both layers run as bf16 MMAs with fp32 accumulation.
// ---------------------------------------------------------------------------------------
constexpr int kRouterTcMaxB = 64;                 // 2B vectors fit one 128-column accumulator
constexpr int kRouterMaxTiles = kRouterMaxK / tc::kRows;

struct DenseRows {
    int n;
    using State = tc::NoState;
    __device__ void finish(State &) const {}
    __device__ int n_rows() const { return n; }
    __device__ void pick(int u, int &v, int &c) const { v = u; c = 0; }
    __device__ void col_info(int r, int &i, long long &l) const { i = r; l = 0; }
};

// Layer 1: hid2[(2b) * Hr + i] = hi, hid2[(2b+1) * Hr + i] = lo of act(W1[i] . h_b + b1[i]).
struct Layer1Ep : DenseRows {
    const uint16_t *bias;
    uint16_t *hid2;
    int Hr, act;
    __device__ int row_aux(int v) const { return v >= 0 ? __float_as_int(bf16_to_f32(bias[v])) : 0; }
    __device__ void emit(State &, const float (&x)[16], int cb, int v, int, int aux, const int32_t *s_i,
                         const long long *) const
    {
        if (v < 0) return;
        const float bv = __int_as_float(aux);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int b = s_i[cb + e];
            if (b < 0) continue;
            const float u = act_fn(x[e] + bv, act);
            const uint16_t hi = f32_to_bf16_rne(u);
            const uint16_t lo = f32_to_bf16_rne(u - bf16_to_f32(hi));
            hid2[size_t(2 * b) * Hr + v] = hi;
            hid2[size_t(2 * b + 1) * Hr + v] = lo;
        }
    }
};

// Layer 2: scores[b][c] = (W2[c] . hi_b + W2[c] . lo_b) + b2[c].
struct Layer2Ep : DenseRows {
    const uint16_t *bias;
    float *scores;
    int M, B;
    __device__ int row_aux(int v) const { return v >= 0 ? __float_as_int(bf16_to_f32(bias[v])) : 0; }
    __device__ void emit(State &, const float (&x)[16], int cb, int v, int, int aux, const int32_t *,
                         const long long *) const
    {
        if (v < 0) return;
        const float bv = __int_as_float(aux);
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const int b = (cb + e) >> 1;
            if (b < B) scores[size_t(b) * M + v] = (x[e] + x[e + 1]) + bv;
        }
    }
};

struct RouterTcWs {
    size_t hid2, tile_cnt, parts, total;
};
RouterTcWs router_tc_layout(int B, int Hr)
{
    RouterTcWs w;
    w.hid2 = 0;
    w.tile_cnt = align256(size_t(2) * B * Hr * sizeof(uint16_t));
    w.parts = w.tile_cnt + align256(size_t(kRouterMaxTiles) * sizeof(unsigned));
    w.total = w.parts + align256(tc::parts_bytes(2 * B, tc::kMaxGrid));
    return w;
}

// CTAs of a router GEMM: the first draft position's router runs before any head and may use
// the whole GPU, but a router layer is only a few hundred (tile, k-stage) units, and a tile
// split between many CTAs pays for storing and adding its parts, so each CTA takes at least
// 8 units; a later position's router runs beside the batched head, which leaves kRouterSideSms
// SMs free for it, and must fit there.
constexpr int kRouterSideSms = 8;
constexpr int kRouterMinUnits = 8;
// side: the caller's SM count for the launch (<= 0: the default above)
int router_grid(int pos, int units, int sms, int side)
{
    int g = side > 0 ? side : pos == 1 ? (units + kRouterMinUnits - 1) / kRouterMinUnits : kRouterSideSms;
    if (g > sms) g = sms;
    if (g > tc::kMaxGrid) g = tc::kMaxGrid;
    if (g > units) g = units;
    return g < 1 ? 1 : g;
}

template <typename XT, int BT>
ds_status launch_gemv(const uint16_t *A, int N, int K, const XT *x, int B, const uint16_t *bias, int act,
                      float *y, int topk_k, int32_t *topk_ids, unsigned *counters, cudaStream_t stream)
{
    const size_t smem = size_t(BT) * K * sizeof(float);
    static std::atomic<unsigned long long> smem_set{0};
    if (!smem_limit_once(gemv_rows_kernel<XT, BT>, size_t(BT) * kRouterMaxK * sizeof(float), smem_set))
        return DS_ERR_CUDA;
    dim3 grid((N + kGemvWarps - 1) / kGemvWarps, (B + BT - 1) / BT);
    gemv_rows_kernel<XT, BT><<<grid, kGemvWarps * 32, smem, stream>>>(A, N, K, x, B, bias, act, y,
                                                                       topk_k, topk_ids, counters);
    DS_TRY_LAUNCH();
    return DS_OK;
}

}  // namespace
}  // namespace ds

using namespace ds;

extern "C" size_t ds_router_workspace_bytes(int B, int Hr)
{
    if (B <= 0 || Hr <= 0) return 0;
    if (B >= 2 && B <= kRouterTcMaxB) return router_tc_layout(B, Hr).total;
    // hidden layer u [B, Hr] + one completion counter per batch tile of the second layer
    return align256(size_t(B) * size_t(Hr) * sizeof(float)) + align256(size_t(B) * sizeof(unsigned));
}

namespace {
// ds_router_topk, and at B = 1 optionally the list's table (list_out.table non-null).
ds_status router_topk(const uint16_t *H, int B, int d, const uint16_t *W1, const uint16_t *b1, int Hr,
                      const uint16_t *W2, const uint16_t *b2, int M, int act, const int32_t *budget, int n_budget,
                      int pos, float *scores, int32_t *cluster_ids, int side, void *ws, size_t ws_bytes,
                      int32_t *dev_status, cudaStream_t stream, ListOut list_out)
{
    ds::NvtxRange range("ds_router_topk");
    if (!H || !W1 || !b1 || !W2 || !b2 || !budget || !scores || !cluster_ids)
        return DS_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d < 8 || d % 8 || Hr < 8 || Hr % 8 || M < 1 || M > kRouterMaxK)
        return DS_ERR_INVALID_ARG;
    if (d > kRouterMaxK || Hr > kRouterMaxK) return DS_ERR_UNSUPPORTED;
    if (act != DS_ACT_RELU && act != DS_ACT_GELU) return DS_ERR_INVALID_ARG;
    if (pos < 1 || pos > n_budget) return DS_ERR_INVALID_ARG;
    const int k = budget[pos - 1];
    if (k < 1 || k > M) return DS_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(W1) || !aligned16(W2)) return DS_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ds_router_workspace_bytes(B, Hr)) return DS_ERR_WORKSPACE;

    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    float *u = static_cast<float *>(ws);
    unsigned *counters = reinterpret_cast<unsigned *>(static_cast<char *>(ws) +
                                                      align256(size_t(B) * size_t(Hr) * sizeof(float)));
    if (B == 1) {
        // the first position's router has the GPU to itself: one warp per weight row; a later
        // one runs kGemv1PerSm blocks on each SM the head beside it leaves free
        auto grid1 = [&](int rows) {
            if (side > 0 || pos != 1) {
                const int g = kGemv1PerSm * (side > 0 ? (side < sms ? side : sms) : kGemv1SideSms);
                const int need = (rows + kGemvWarps - 1) / kGemvWarps;
                return g < need ? g : need;
            }
            const int g = (rows + kGemvWarps - 1) / kGemvWarps;
            return g < sms ? g : sms;
        };
        gemv1_kernel<uint16_t><<<grid1(Hr), kGemvWarps * 32, 0, stream>>>(W1, Hr, d, H, b1, act, u, 0,
                                                                         nullptr, nullptr, ListOut{});
        DS_TRY_LAUNCH();
        gemv1_kernel<float><<<grid1(M), kGemvWarps * 32, 0, stream>>>(W2, M, Hr, u, b2, -1, scores, k,
                                                                      cluster_ids, counters, list_out);
        DS_TRY_LAUNCH();
        return DS_OK;
    }
    if (B <= kRouterTcMaxB) {
        const RouterTcWs lay = router_tc_layout(B, Hr);
        char *w = static_cast<char *>(ws);
        uint16_t *hid2 = reinterpret_cast<uint16_t *>(w + lay.hid2);
        unsigned *tile_cnt = reinterpret_cast<unsigned *>(w + lay.tile_cnt);
        float *parts = reinterpret_cast<float *>(w + lay.parts);
        Layer1Ep e1;
        e1.n = Hr; e1.bias = b1; e1.hid2 = hid2; e1.Hr = Hr; e1.act = act;
        const tc::Operands op1{W1, H, d, B, dev_status, wait_budget()};
        const int u1 = ((Hr + tc::kRows - 1) / tc::kRows) * ((d + 127) / 128);
        ds_status st = tc::launch_for(op1, e1, parts, tile_cnt, router_grid(pos, u1, sms, side), stream);
        if (st != DS_OK) return st;
        Layer2Ep e2;
        e2.n = M; e2.bias = b2; e2.scores = scores; e2.M = M; e2.B = B;
        const tc::Operands op2{W2, hid2, Hr, 2 * B, dev_status, wait_budget()};
        const int u2 = ((M + tc::kRows - 1) / tc::kRows) * ((Hr + 127) / 128);
        st = tc::launch_for(op2, e2, parts, tile_cnt, router_grid(pos, u2, sms, side), stream);
        if (st != DS_OK) return st;
        topk_rows_kernel<<<B, kTopkThreads, 0, stream>>>(scores, M, k, cluster_ids);
        DS_TRY_LAUNCH();
        return DS_OK;
    }
    const ds_status s1 = launch_gemv<uint16_t, kGemvBT>(W1, Hr, d, H, B, b1, act, u, 0, nullptr, nullptr, stream);
    if (s1 != DS_OK) return s1;
    const ds_status s2 = launch_gemv<float, kGemvBT>(W2, M, Hr, u, B, b2, -1, scores, k, cluster_ids, counters, stream);
    if (s2 != DS_OK) return s2;
    return DS_OK;
}
}  // namespace

extern "C" ds_status ds_router_topk(const uint16_t *H, int B, int d,
                                    const uint16_t *W1, const uint16_t *b1, int Hr,
                                    const uint16_t *W2, const uint16_t *b2, int M, int act,
                                    const int32_t *budget, int n_budget, int pos,
                                    float *scores, int32_t *cluster_ids, int sms,
                                    void *ws, size_t ws_bytes, int32_t *dev_status,
                                    cudaStream_t stream)
{
    ListOut none{};
    return router_topk(H, B, d, W1, b1, Hr, W2, b2, M, act, budget, n_budget, pos, scores, cluster_ids,
                       sms, ws, ws_bytes, dev_status, stream, none);
}

// ---------------------------------------------------------------------------------------
// Router handle: the weights, sizes, activation and budget table of one router, so that a
// draft position's call names only its hidden states and position.  Host memory only; the
// weights stay the caller's.
// ---------------------------------------------------------------------------------------
#include <new>
#include <vector>

struct ds_router {
    const uint16_t *W1, *b1, *W2, *b2;
    int d, Hr, M, act;
    std::vector<int32_t> budget;
};

extern "C" ds_status ds_router_create(ds_router_t *out, const uint16_t *W1, const uint16_t *b1,
                                      const uint16_t *W2, const uint16_t *b2, int d, int Hr, int M,
                                      int act, const int32_t *budget, int gamma)
{
    if (!out) return DS_ERR_INVALID_ARG;
    *out = nullptr;
    if (!W1 || !b1 || !W2 || !b2 || !budget) return DS_ERR_INVALID_ARG;
    if (d < 8 || d % 8 || Hr < 8 || Hr % 8 || M < 1 || M > kRouterMaxK || gamma < 1) return DS_ERR_INVALID_ARG;
    if (d > kRouterMaxK || Hr > kRouterMaxK) return DS_ERR_UNSUPPORTED;
    if (act != DS_ACT_RELU && act != DS_ACT_GELU) return DS_ERR_INVALID_ARG;
    if (!aligned16(W1) || !aligned16(W2)) return DS_ERR_INVALID_ARG;
    for (int t = 0; t < gamma; ++t)
        if (budget[t] < 1 || budget[t] > M) return DS_ERR_INVALID_ARG;
    ds_router *h = new (std::nothrow) ds_router;
    if (!h) return DS_ERR_UNSUPPORTED;
    h->W1 = W1; h->b1 = b1; h->W2 = W2; h->b2 = b2;
    h->d = d; h->Hr = Hr; h->M = M; h->act = act;
    h->budget.assign(budget, budget + gamma);
    *out = h;
    return DS_OK;
}

extern "C" ds_status ds_router_destroy(ds_router_t r)
{
    delete r;
    return DS_OK;
}

// [the router call's workspace | B x M scores when the caller passes none]
extern "C" size_t ds_router_workspace_bytes_h(ds_router_t r, int B)
{
    if (!r || B <= 0) return 0;
    return align256(ds_router_workspace_bytes(B, r->Hr)) + align256(size_t(B) * size_t(r->M) * sizeof(float));
}

extern "C" ds_status ds_router_topk_h(ds_router_t r, const uint16_t *H, int B, int pos,
                                      float *scores, int32_t *cluster_ids, int sms,
                                      void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    if (!r) return DS_ERR_INVALID_ARG;
    if (B < 1 || B > 4096) return DS_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ds_router_workspace_bytes_h(r, B)) return DS_ERR_WORKSPACE;
    const size_t base = align256(ds_router_workspace_bytes(B, r->Hr));
    if (!scores) scores = reinterpret_cast<float *>(static_cast<char *>(ws) + base);
    return ds_router_topk(H, B, r->d, r->W1, r->b1, r->Hr, r->W2, r->b2, r->M, r->act,
                          r->budget.data(), int(r->budget.size()), pos, scores, cluster_ids, sms,
                          ws, base, dev_status, stream);
}

// Batch 1: the router and top-k of a draft position with the list's table instead of its copied
// ids (see ListOut); one launch fewer than ds_router_topk_h + ds_build_shortlist.
extern "C" ds_status ds_router_topk_list_b1(ds_router_t r, const uint16_t *H, int pos,
                                            const int32_t *csr_off, int V,
                                            float *scores, int32_t *cluster_ids,
                                            int32_t *cpos, int32_t *vs_offsets, int32_t *list_table,
                                            int64_t capacity, int sms,
                                            void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    if (!r || !csr_off || !cpos || !vs_offsets || !list_table || V < 1 || capacity < 0) return DS_ERR_INVALID_ARG;
    if (!scores) return DS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(list_table) & 7u) != 0) return DS_ERR_INVALID_ARG;
    ListOut lo;
    lo.csr_off = csr_off; lo.V = V; lo.table = reinterpret_cast<int2 *>(list_table);
    lo.cpos = cpos; lo.vs_offsets = vs_offsets; lo.capacity = capacity; lo.status = dev_status;
    return router_topk(H, 1, r->d, r->W1, r->b1, r->Hr, r->W2, r->b2, r->M, r->act, r->budget.data(),
                       int(r->budget.size()), pos, scores, cluster_ids, sms, ws, ws_bytes, dev_status, stream, lo);
}
