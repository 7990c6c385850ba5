// Shortlist construction: V_S = the union of the selected clusters' tokens.
//
// DynaSpec abstract (the drafter's shortlist is the set of tokens of the best-scoring
// clusters taken together); summary, Technical Details > Problem Definition (the output of
// the step is the shortlist V_S).  The clusters partition the vocabulary, so the union is a concatenation: an
// exclusive scan of the selected clusters' sizes in ascending cluster id gives every
// cluster's place in the list (cpos), and a copy of the CSR slices fills it.  The same
// scan over "selected by any list" gives the batch union the batched / tree heads read W
// through.
#include "common.cuh"
#include "block_scan.cuh"

namespace ds {
namespace {

constexpr int kSlThreads = 1024;
constexpr int kSlMaxM = 8192;
constexpr int kSlMaxPer = kSlMaxM / kSlThreads;

// cluster_of[v] = c and rank_in_cluster[v] = position of v in cluster c's list.
__global__ void vocab_index_kernel(const int32_t *__restrict__ off, const int32_t *__restrict__ tok,
                                   int M, int V, int32_t *__restrict__ cluster_of,
                                   int32_t *__restrict__ rank, int32_t *st)
{
    const int c = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (c >= M) return;
    const int lo = off[c], hi = off[c + 1];
    if (lo < 0 || hi < lo || hi > V) { if ((threadIdx.x & 31) == 0) set_status(st, DS_DEV_BAD_INDEX); return; }
    for (int r = lo + (threadIdx.x & 31); r < hi; r += 32) {
        const int v = tok[r];
        if (v < 0 || v >= V) { set_status(st, DS_DEV_BAD_INDEX); continue; }
        cluster_of[v] = c;
        rank[v] = r - lo;
    }
}

// Single block, once every list's scan is stored: vs_offsets = exclusive scan of the list
// sizes; and, if asked, the batch union (clusters selected by any list) with each cluster's
// start in it (ustart, -1 if out).  Reads what other blocks stored, through L2.
__device__ void offsets_block(const int32_t *__restrict__ off, int M, int B,
                              const int32_t *__restrict__ sizes, const int32_t *__restrict__ cpos,
                              int32_t *__restrict__ vs_offsets, int64_t capacity,
                              int32_t *__restrict__ ustart, int32_t *__restrict__ union_count, int32_t *st)
{
    __shared__ int scratch[33];
    {
        const int E = (B + kSlThreads - 1) / kSlThreads;
        const int lo = threadIdx.x * E;
        int sum = 0;
        for (int e = 0; e < E; ++e) if (lo + e < B) sum += __ldcg(&sizes[lo + e]);
        int tot;
        int run = block_exclusive_scan(sum, scratch, &tot);
        for (int e = 0; e < E; ++e) if (lo + e < B) { vs_offsets[lo + e] = run; run += __ldcg(&sizes[lo + e]); }
        if (threadIdx.x == 0) {
            vs_offsets[B] = tot;
            if (int64_t(tot) > capacity) set_status(st, DS_DEV_CAPACITY);
        }
    }
    if (!ustart) return;
    const int E = (M + kSlThreads - 1) / kSlThreads;
    const int lo = threadIdx.x * E;
    int sz[kSlMaxPer];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        bool any = false;
        if (e < E && c < M) {
            // eight independent loads per round instead of a dependent chain over b
            int b = 0;
            for (; b + 8 <= B && !any; b += 8) {
                int q[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) q[j] = __ldcg(&cpos[size_t(b + j) * M + c]);
#pragma unroll
                for (int j = 0; j < 8; ++j) any |= q[j] >= 0;
            }
            for (; b < B && !any; ++b) any = __ldcg(&cpos[size_t(b) * M + c]) >= 0;
        }
        sz[e] = any ? off[c + 1] - off[c] : 0;
        sum += sz[e];
    }
    int tot;
    int run = block_exclusive_scan(sum, scratch, &tot);
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        if (e < E && c < M) { ustart[c] = sz[e] ? run : -1; run += sz[e]; }
    }
    if (threadIdx.x == 0) *union_count = tot;
}

// One block per list b: cpos[b][c] = exclusive prefix (over ascending c) of the sizes of the
// clusters b selected, or -1; sizes[b] = |S_b|.  The last block to finish (a completion
// counter) then computes the offsets and the union's starts (offsets_block).
__global__ void __launch_bounds__(kSlThreads)
shortlist_scan_kernel(const int32_t *__restrict__ off, int M, const int32_t *__restrict__ ids, int k,
                      int32_t *__restrict__ cpos, int32_t *__restrict__ sizes,
                      int32_t *__restrict__ vs_offsets, int64_t capacity,
                      int32_t *__restrict__ ustart, int32_t *__restrict__ union_count,
                      unsigned *__restrict__ counter, int32_t *st)
{
    __shared__ unsigned char flag[kSlMaxM];
    __shared__ int scratch[33];
    const int b = blockIdx.x;
    for (int c = threadIdx.x; c < M; c += blockDim.x) flag[c] = 0;
    __syncthreads();
    const int32_t *my = ids + size_t(b) * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        const int c = my[j];
        if (c < 0 || c >= M || (j > 0 && my[j - 1] >= c)) { set_status(st, DS_DEV_BAD_INDEX); continue; }
        flag[c] = 1;
    }
    __syncthreads();
    const int E = (M + kSlThreads - 1) / kSlThreads;
    const int lo = threadIdx.x * E;
    int sz[kSlMaxPer];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        sz[e] = (e < E && c < M && flag[c]) ? off[c + 1] - off[c] : 0;
        sum += sz[e];
    }
    int tot;
    int run = block_exclusive_scan(sum, scratch, &tot);
    int32_t *dst = cpos + size_t(b) * M;
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        if (e < E && c < M) { dst[c] = flag[c] ? run : -1; run += sz[e]; }
    }
    if (threadIdx.x == 0) sizes[b] = tot;
    if (!last_block_done(counter, gridDim.x)) return;
    offsets_block(off, M, int(gridDim.x), sizes, cpos, vs_offsets, capacity, ustart, union_count, st);
}

// The copies, one launch: blocks [0, xb * B) take one warp per selected cluster of list
// b = block / xb and copy its CSR slice into the list; the blocks after them (union != null)
// take one warp per cluster of the batch union and copy its slice and cluster id there.
__global__ void shortlist_copy_kernel(const int32_t *__restrict__ off, const int32_t *__restrict__ tok,
                                      int M, int V, const int32_t *__restrict__ ids, int k, int B, int xb,
                                      const int32_t *__restrict__ cpos,
                                      const int32_t *__restrict__ vs_offsets, int32_t *__restrict__ vs_ids,
                                      int64_t capacity, const int32_t *__restrict__ ustart,
                                      int32_t *__restrict__ union_ids, int32_t *__restrict__ union_cluster)
{
    const int wpb = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int nlist = xb * B;
    if (int(blockIdx.x) < nlist) {
        const int b = blockIdx.x / xb;
        const int j = (blockIdx.x - b * xb) * wpb + (threadIdx.x >> 5);
        if (j >= k) return;
        const int c = ids[size_t(b) * k + j];
        if (c < 0 || c >= M) return;                      // flagged by the scan kernel
        const int p = cpos[size_t(b) * M + c];
        if (p < 0) return;                                // duplicate / unsorted ids, flagged
        const int lo = off[c], n = off[c + 1] - lo;
        if (lo < 0 || n < 0 || lo + n > V) return;
        const int64_t base = int64_t(vs_offsets[b]) + p;
        for (int r = lane; r < n; r += 32)
            if (base + r < capacity) vs_ids[base + r] = tok[lo + r];
        return;
    }
    const int c = (int(blockIdx.x) - nlist) * wpb + (threadIdx.x >> 5);
    if (c >= M) return;
    const int u = ustart[c];
    if (u < 0) return;
    const int lo = off[c], n = off[c + 1] - lo;
    if (lo < 0 || n < 0 || lo + n > V || u + n > V) return;
    for (int r = lane; r < n; r += 32) {
        union_ids[u + r] = tok[lo + r];
        union_cluster[u + r] = c;
    }
}

// One list, no union: scan and expansion in one launch.  Every block recomputes the (tiny)
// scan of the selected clusters' sizes in shared memory, then copies its share of the selected
// clusters' CSR slices, one warp per cluster; block 0 also writes cpos and the offsets.
constexpr int kSlCopyWarps = 1;           // selected clusters per copying warp

__global__ void __launch_bounds__(kSlThreads)
shortlist_single_kernel(const int32_t *__restrict__ off, const int32_t *__restrict__ tok, int M, int V,
                        const int32_t *__restrict__ ids, int k, int32_t *__restrict__ cpos,
                        int32_t *__restrict__ vs_offsets, int32_t *__restrict__ vs_ids, int64_t capacity,
                        int32_t *st)
{
    __shared__ unsigned char flag[kSlMaxM];
    __shared__ int spos[kSlMaxM];
    __shared__ int scratch[33];
    for (int c = threadIdx.x; c < M; c += blockDim.x) flag[c] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        const int c = ids[j];
        if (c < 0 || c >= M || (j > 0 && ids[j - 1] >= c)) {
            if (blockIdx.x == 0) set_status(st, DS_DEV_BAD_INDEX);
            continue;
        }
        flag[c] = 1;
    }
    __syncthreads();
    const int E = (M + kSlThreads - 1) / kSlThreads;
    const int lo = threadIdx.x * E;
    int sz[kSlMaxPer];
    int sum = 0;
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        int n = 0;
        if (e < E && c < M && flag[c]) {
            n = off[c + 1] - off[c];
            if (off[c] < 0 || n < 0 || off[c + 1] > V) {
                if (blockIdx.x == 0) set_status(st, DS_DEV_BAD_INDEX);
                n = 0;
            }
        }
        sz[e] = n;
        sum += n;
    }
    int tot;
    int run = block_exclusive_scan(sum, scratch, &tot);
#pragma unroll
    for (int e = 0; e < kSlMaxPer; ++e) {
        const int c = lo + e;
        if (e < E && c < M) {
            const int p = flag[c] ? run : -1;
            spos[c] = p;
            if (blockIdx.x == 0) cpos[c] = p;
            run += sz[e];
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        vs_offsets[0] = 0;
        vs_offsets[1] = tot;
        if (int64_t(tot) > capacity) set_status(st, DS_DEV_CAPACITY);
    }
    __syncthreads();
    // this block's share of the selected clusters, one warp per cluster
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kSlThreads / 32);
    for (int j = blockIdx.x * (kSlThreads / 32) + warp; j < k; j += nwarps) {
        const int c = ids[j];
        if (c < 0 || c >= M) continue;
        const int p = spos[c];
        if (p < 0) continue;
        const int l0 = off[c], n = off[c + 1] - l0;
        if (l0 < 0 || n < 0 || l0 + n > V) continue;
#pragma unroll 4
        for (int r = lane; r < n; r += 32)
            if (int64_t(p) + r < capacity) vs_ids[p + r] = tok[l0 + r];
    }
}

}  // namespace
}  // namespace ds

using namespace ds;

extern "C" ds_status ds_vocab_index(const int32_t *csr_off, const int32_t *csr_tok, int M, int V,
                                    int32_t *cluster_of, int32_t *rank_in_cluster,
                                    int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_vocab_index");
    if (!csr_off || !csr_tok || !cluster_of || !rank_in_cluster) return DS_ERR_INVALID_ARG;
    if (M < 1 || V < 1 || M > V) return DS_ERR_INVALID_ARG;
    vocab_index_kernel<<<(M + 7) / 8, 256, 0, stream>>>(csr_off, csr_tok, M, V, cluster_of,
                                                       rank_in_cluster, dev_status);
    DS_TRY_LAUNCH();
    return DS_OK;
}

extern "C" size_t ds_shortlist_workspace_bytes(int B, int M)
{
    if (B <= 0 || M <= 0) return 0;
    return align256(size_t(B) * sizeof(int32_t)) + align256(size_t(M) * sizeof(int32_t)) + align256(sizeof(unsigned));
}

extern "C" ds_status ds_build_shortlist(const int32_t *csr_off, const int32_t *csr_tok, int M, int V,
                                        const int32_t *cluster_ids, int B, int k,
                                        int32_t *vs_offsets, int32_t *vs_ids, int64_t vs_capacity,
                                        int32_t *cpos,
                                        int32_t *union_ids, int32_t *union_cluster, int32_t *union_count,
                                        void *ws, size_t ws_bytes, int32_t *dev_status,
                                        cudaStream_t stream)
{
    ds::NvtxRange range("ds_build_shortlist");
    if (!csr_off || !csr_tok || !cluster_ids || !vs_offsets || !vs_ids || !cpos)
        return DS_ERR_INVALID_ARG;
    const int nu = (union_ids != nullptr) + (union_cluster != nullptr) + (union_count != nullptr);
    if (nu != 0 && nu != 3) return DS_ERR_INVALID_ARG;
    if (M < 1 || M > kSlMaxM || V < M || B < 1 || B > 4096 || k < 1 || k > M || vs_capacity < 0)
        return DS_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ds_shortlist_workspace_bytes(B, M)) return DS_ERR_WORKSPACE;
    int32_t *sizes = static_cast<int32_t *>(ws);
    int32_t *ustart = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + align256(size_t(B) * 4));
    unsigned *counter = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + align256(size_t(B) * 4) +
                                                     align256(size_t(M) * 4));

    if (B == 1 && nu == 0) {
        const int blocks = (k + kSlCopyWarps * (kSlThreads / 32) - 1) / (kSlCopyWarps * (kSlThreads / 32));
        shortlist_single_kernel<<<blocks, kSlThreads, 0, stream>>>(csr_off, csr_tok, M, V, cluster_ids, k, cpos,
                                                                   vs_offsets, vs_ids, vs_capacity, dev_status);
        DS_TRY_LAUNCH();
        return DS_OK;
    }
    // the scan (its last block also computes the offsets and the union's starts), then the copies
    shortlist_scan_kernel<<<B, kSlThreads, 0, stream>>>(csr_off, M, cluster_ids, k, cpos, sizes, vs_offsets,
                                                        vs_capacity, nu ? ustart : nullptr, union_count, counter,
                                                        dev_status);
    DS_TRY_LAUNCH();
    const int xb = (k + 7) / 8;                   // blocks of 8 warps per list
    const int ub = nu ? (M + 7) / 8 : 0;          // blocks of 8 warps over the union's clusters
    shortlist_copy_kernel<<<xb * B + ub, 256, 0, stream>>>(csr_off, csr_tok, M, V, cluster_ids, k, B, xb, cpos,
                                                          vs_offsets, vs_ids, vs_capacity, ustart, union_ids,
                                                          union_cluster);
    DS_TRY_LAUNCH();
    return DS_OK;
}
