// Spherical k-means over the LM-head rows: the offline step that forms the vocabulary clusters
// the router scores (DynaSpec summary, Key Novelty and Key Hyperparameters: the LM-head rows are
// clustered by spherical k-means).  The pages give no iteration details; the standard Lloyd
// iteration for the cosine objective is used:
//   assignment  c(v) = argmax_c <W_v, mu_c> (the row's own norm does not change the argmax),
//               ties to the lower c; scored with the centroids rounded to bf16 on the tensor
//               cores (fp32 accumulation);
//   update      mu_c = S_c / |S_c|, S_c = sum of W_v / |W_v| over cluster c's tokens, added in
//               ascending token order (fp32); an empty cluster keeps its centroid;
//   CSR         clusters in ascending id, each cluster's tokens in ascending token id (a stable
//               counting sort), the layout ds_vocab_index and ds_build_shortlist take.
//
// The assignment is a V x M x d contraction (1.1 TFLOP per iteration at V = 128,256, d = 4096,
// M = 1024): it runs on the tcgen05 GEMM of the gathered head with every W row picked in order
// and 128 centroids per launch; the epilogue folds each row's best (score, centroid) pair with
// a 64-bit atomic max of (order-preserving score bits, inverted centroid id), which does not
// depend on the order the parts arrive in.  The update streams W once (HBM-bound).
#include "common.cuh"
#include "block_scan.cuh"
#include "tc_gemm.cuh"

namespace ds {
namespace {

constexpr int kKmMaxM = 4096;            // centroids (the stable scatter keeps 8 x M counts in smem)
constexpr int kKmRowsPerBlock = 256;     // rows per counting-sort block (8 warps)
constexpr int kKmMaxD = 8192;

__device__ __forceinline__ uint32_t order_key(float f)
{
    if (f == 0.f) f = 0.f;
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Scores of every W row against centroids cbase .. cbase + R - 1; keeps the best per row.
struct KmeansEp {
    unsigned long long *best;
    int V, cbase;
    using State = tc::NoState;
    __device__ void finish(State &) const {}
    __device__ int n_rows() const { return V; }
    __device__ void pick(int u, int &v, int &c) const { v = u; c = 0; }
    __device__ void col_info(int r, int &i, long long &l) const { i = r; l = 0; }
    __device__ int row_aux(int) const { return 0; }
    __device__ void emit(State &, const float (&x)[16], int cb, int v, int, int, const int32_t *s_i,
                         const long long *) const
    {
        if (v < 0) return;
        unsigned long long key = 0ull;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            if (s_i[cb + e] < 0) continue;
            const uint32_t c = uint32_t(cbase + s_i[cb + e]);
            const unsigned long long k = (static_cast<unsigned long long>(order_key(x[e])) << 32) | (0xFFFFFFFFu - c);
            key = k > key ? k : key;
        }
        if (key) atomicMax(best + v, key);
    }
};

// inv_norm[v] = 1 / |W_v| (0 for a zero row); a warp per row.
__global__ void km_norms(const uint16_t *__restrict__ W, int V, int d, float *__restrict__ inv_norm)
{
    const int lane = threadIdx.x & 31;
    for (int v = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); v < V; v += gridDim.x * (blockDim.x >> 5)) {
        const uint4 *r = reinterpret_cast<const uint4 *>(W + size_t(v) * d);
        float s = 0.f;
        for (int k = lane * 8; k < d; k += 256) {
            const uint4 w = ld_stream(r + (k >> 3));
            const float a[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(a[e], a[e], s);
        }
        s = warp_sum(s);
        if (lane == 0) inv_norm[v] = s > 0.f ? rsqrtf(s) : 0.f;
    }
}

// cent[c] = W[init[c]] * inv_norm[init[c]]; a block per centroid.
__global__ void km_init(const uint16_t *__restrict__ W, int V, int d, const int32_t *__restrict__ init,
                        const float *__restrict__ inv_norm, float *__restrict__ cent, int32_t *st)
{
    const int c = blockIdx.x;
    int v = init[c];
    if (v < 0 || v >= V) {
        if (threadIdx.x == 0) set_status(st, DS_DEV_BAD_INDEX);
        v = 0;
    }
    const float s = inv_norm[v];
    for (int k = threadIdx.x; k < d; k += blockDim.x) cent[size_t(c) * d + k] = bf16_to_f32(W[size_t(v) * d + k]) * s;
}

// The bf16 operand copy of the centroids, and the per-row best keys cleared.
__global__ void km_prepare(const float *__restrict__ cent, size_t n, uint16_t *__restrict__ cb16,
                           unsigned long long *__restrict__ best, int V)
{
    const size_t i0 = blockIdx.x * size_t(blockDim.x) + threadIdx.x, step = size_t(gridDim.x) * blockDim.x;
    for (size_t i = i0; i < n; i += step) cb16[i] = f32_to_bf16_rne(cent[i]);
    for (size_t i = i0; i < size_t(V); i += step) best[i] = 0ull;
}

// assign[v] from the best keys; per-block cluster counts counts[blk][c] (blk = 256 rows).
__global__ void __launch_bounds__(kKmRowsPerBlock)
km_assign_count(const unsigned long long *__restrict__ best, int V, int M, int32_t *__restrict__ assign,
                int32_t *__restrict__ counts, int32_t *st)
{
    extern __shared__ int hist[];                      // M
    for (int c = threadIdx.x; c < M; c += blockDim.x) hist[c] = 0;
    __syncthreads();
    const int v = blockIdx.x * kKmRowsPerBlock + threadIdx.x;
    if (v < V) {
        int c = int(0xFFFFFFFFu - uint32_t(best[v] & 0xFFFFFFFFull));
        if (best[v] == 0ull || c < 0 || c >= M) { set_status(st, DS_DEV_BAD_INDEX); c = 0; }
        assign[v] = c;
        atomicAdd(&hist[c], 1);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < M; c += blockDim.x) counts[size_t(blockIdx.x) * M + c] = hist[c];
}

// One block: exclusive scan of counts in (cluster, block) order -> start[blk][c] and csr_off.
__global__ void __launch_bounds__(1024)
km_scan(int32_t *__restrict__ counts, int nblk, int M, int32_t *__restrict__ csr_off)
{
    __shared__ int scratch[33];
    const long long total = 1LL * nblk * M;
    const long long per = (total + blockDim.x - 1) / blockDim.x;
    const long long lo = threadIdx.x * per, hi = lo + per < total ? lo + per : total;
    // element i of the (c, blk) order is counts[blk][c] with c = i / nblk, blk = i % nblk
    int sum = 0;
    for (long long i = lo; i < hi; ++i) sum += counts[size_t(i % nblk) * M + size_t(i / nblk)];
    int tot;
    int run = block_exclusive_scan(sum, scratch, &tot);
    for (long long i = lo; i < hi; ++i) {
        const int c = int(i / nblk), b = int(i % nblk);
        const int n = counts[size_t(b) * M + c];
        if (b == 0) csr_off[c] = run;
        counts[size_t(b) * M + c] = run;               // becomes the block's start in cluster c
        run += n;
    }
    if (threadIdx.x == 0) csr_off[M] = tot;
}

// Stable scatter: token v goes to start[blk][c] + (rows of block blk before v with cluster c).
__global__ void __launch_bounds__(kKmRowsPerBlock)
km_scatter(const int32_t *__restrict__ assign, int V, int M, const int32_t *__restrict__ start,
           int32_t *__restrict__ csr_tok)
{
    extern __shared__ int wcnt[];                      // [8 warps][M]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 8 * M; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const int v = blockIdx.x * kKmRowsPerBlock + threadIdx.x;
    const int c = v < V ? assign[v] : -1;
    const unsigned same = __match_any_sync(0xFFFFFFFFu, c);
    const int in_warp = __popc(same & ((1u << lane) - 1u));
    if (c >= 0 && lane == __ffs(same) - 1) wcnt[warp * M + c] = __popc(same);
    __syncthreads();
    if (c >= 0) {
        int before = 0;
        for (int w = 0; w < warp; ++w) before += wcnt[w * M + c];
        csr_tok[start[size_t(blockIdx.x) * M + c] + before + in_warp] = v;
    }
}

// Centroid update: a block per cluster sums the unit rows of its tokens (CSR order, fp32),
// normalises, and writes the centroid; an empty cluster keeps its centroid.
__global__ void __launch_bounds__(256)
km_update(const uint16_t *__restrict__ W, int d, const float *__restrict__ inv_norm,
          const int32_t *__restrict__ csr_off, const int32_t *__restrict__ csr_tok, float *__restrict__ cent)
{
    __shared__ float red[8];
    const int c = blockIdx.x;
    const int lo = csr_off[c], hi = csr_off[c + 1];
    if (hi <= lo) return;                              // uniform over the block
    constexpr int kPer = kKmMaxD / 2048;               // 8-column groups per thread
    float acc[kPer][8];
#pragma unroll
    for (int g = 0; g < kPer; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    for (int r = lo; r < hi; ++r) {
        const int v = csr_tok[r];
        const float s = inv_norm[v];
        const uint4 *row = reinterpret_cast<const uint4 *>(W + size_t(v) * d);
#pragma unroll
        for (int g = 0; g < kPer; ++g) {
            const int k = g * 2048 + threadIdx.x * 8;
            if (k < d) {
                const uint4 w = ld_stream(row + (k >> 3));
                acc[g][0] = fmaf(bf16lo(w.x), s, acc[g][0]); acc[g][1] = fmaf(bf16hi(w.x), s, acc[g][1]);
                acc[g][2] = fmaf(bf16lo(w.y), s, acc[g][2]); acc[g][3] = fmaf(bf16hi(w.y), s, acc[g][3]);
                acc[g][4] = fmaf(bf16lo(w.z), s, acc[g][4]); acc[g][5] = fmaf(bf16hi(w.z), s, acc[g][5]);
                acc[g][6] = fmaf(bf16lo(w.w), s, acc[g][6]); acc[g][7] = fmaf(bf16hi(w.w), s, acc[g][7]);
            }
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int g = 0; g < kPer; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(acc[g][e], acc[g][e], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += red[w];          // the same order in every thread
    const float inv = tot > 0.f ? rsqrtf(tot) : 0.f;
    if (tot <= 0.f) return;                            // a zero sum keeps the centroid (uniform)
#pragma unroll
    for (int g = 0; g < kPer; ++g) {
        const int k = g * 2048 + threadIdx.x * 8;
        if (k < d)
#pragma unroll
            for (int e = 0; e < 8; ++e) cent[size_t(c) * d + k + e] = acc[g][e] * inv;
    }
}

struct KmWs {
    size_t best, cb16, counts, tile_cnt, parts, total;
};
KmWs km_layout(int V, int d, int M)
{
    KmWs w;
    const size_t nblk = size_t((V + kKmRowsPerBlock - 1) / kKmRowsPerBlock);
    w.best = 0;
    w.cb16 = align256(size_t(V) * sizeof(unsigned long long));
    w.counts = w.cb16 + align256(size_t(M) * d * sizeof(uint16_t));
    w.tile_cnt = w.counts + align256(nblk * M * sizeof(int32_t));
    w.parts = w.tile_cnt + align256(size_t((V + tc::kRows - 1) / tc::kRows) * sizeof(unsigned));
    w.total = w.parts + align256(tc::parts_bytes(tc::kRows, tc::kMaxGrid));
    return w;
}

}  // namespace
}  // namespace ds

using namespace ds;

extern "C" size_t ds_kmeans_workspace_bytes(int V, int d, int M)
{
    if (V <= 0 || d <= 0 || M <= 0) return 0;
    return km_layout(V, d, M).total;
}

extern "C" ds_status ds_kmeans_init(const uint16_t *W, int V, int d, const int32_t *init_rows, int M,
                                    float *cent, float *inv_norm, int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_kmeans_init");
    if (!W || !init_rows || !cent || !inv_norm) return DS_ERR_INVALID_ARG;
    if (V < 1 || d < 8 || d % 8 || M < 1 || M > V) return DS_ERR_INVALID_ARG;
    if (d > kKmMaxD || M > kKmMaxM) return DS_ERR_UNSUPPORTED;
    if (!aligned16(W)) return DS_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    km_norms<<<4 * sms, 256, 0, stream>>>(W, V, d, inv_norm);
    DS_TRY_LAUNCH();
    km_init<<<M, 256, 0, stream>>>(W, V, d, init_rows, inv_norm, cent, dev_status);
    DS_TRY_LAUNCH();
    return DS_OK;
}

extern "C" ds_status ds_kmeans_step(const uint16_t *W, int V, int d, int M, const float *inv_norm, float *cent,
                                    int32_t *assign, int32_t *csr_off, int32_t *csr_tok,
                                    void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_kmeans_step");
    if (!W || !inv_norm || !cent || !assign || !csr_off || !csr_tok) return DS_ERR_INVALID_ARG;
    if (V < 1 || d < 8 || d % 8 || M < 1 || M > V) return DS_ERR_INVALID_ARG;
    if (d > kKmMaxD || M > kKmMaxM) return DS_ERR_UNSUPPORTED;
    if ((V + tc::kRows - 1) / tc::kRows > 8192) return DS_ERR_UNSUPPORTED;
    if (!aligned16(W) || !aligned16(cent)) return DS_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ds_kmeans_workspace_bytes(V, d, M)) return DS_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    const KmWs lay = km_layout(V, d, M);
    char *w = static_cast<char *>(ws);
    auto *best = reinterpret_cast<unsigned long long *>(w + lay.best);
    auto *cb16 = reinterpret_cast<uint16_t *>(w + lay.cb16);
    auto *counts = reinterpret_cast<int32_t *>(w + lay.counts);
    auto *tile_cnt = reinterpret_cast<unsigned *>(w + lay.tile_cnt);
    auto *parts = reinterpret_cast<float *>(w + lay.parts);
    const int nblk = (V + kKmRowsPerBlock - 1) / kKmRowsPerBlock;

    km_prepare<<<2 * sms, 256, 0, stream>>>(cent, size_t(M) * d, cb16, best, V);
    DS_TRY_LAUNCH();
    int grid = sms < tc::kMaxGrid ? sms : tc::kMaxGrid;
    for (int c0 = 0; c0 < M; c0 += tc::kRows) {
        const int R = M - c0 < tc::kRows ? M - c0 : tc::kRows;
        KmeansEp ep;
        ep.best = best; ep.V = V; ep.cbase = c0;
        const tc::Operands op{W, cb16 + size_t(c0) * d, d, R, dev_status, wait_budget()};
        const ds_status st = tc::launch_for(op, ep, parts, tile_cnt, grid, stream);
        if (st != DS_OK) return st;
    }
    static std::atomic<unsigned long long> smem_a{0}, smem_s{0};
    if (!smem_limit_once(km_assign_count, size_t(kKmMaxM) * sizeof(int), smem_a)) return DS_ERR_CUDA;
    if (!smem_limit_once(km_scatter, size_t(8) * kKmMaxM * sizeof(int), smem_s)) return DS_ERR_CUDA;
    km_assign_count<<<nblk, kKmRowsPerBlock, size_t(M) * sizeof(int), stream>>>(best, V, M, assign, counts, dev_status);
    DS_TRY_LAUNCH();
    km_scan<<<1, 1024, 0, stream>>>(counts, nblk, M, csr_off);
    DS_TRY_LAUNCH();
    km_scatter<<<nblk, kKmRowsPerBlock, size_t(8) * M * sizeof(int), stream>>>(assign, V, M, counts, csr_tok);
    DS_TRY_LAUNCH();
    km_update<<<M, 256, 0, stream>>>(W, d, inv_norm, csr_off, csr_tok, cent);
    DS_TRY_LAUNCH();
    return DS_OK;
}
