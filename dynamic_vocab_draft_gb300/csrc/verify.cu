// Speculative-sampling verification over the full vocabulary.
//
// DynaSpec abstract ("the target model still verifies over the full vocabulary, preserving
// exactness"); summary, Technical Details > Pipeline Flow ("Rejection Sampling
// Verification") and System Modules "Target Model".  The pages cite Leviathan et al. 2023
// and Chen et al. 2023 for the algorithm without printing it; the kernels follow its
// standard statement (accept x_t iff u_t q_t(x_t) < p_t(x_t); at the first rejection draw
// from norm(max(0, p_t - q_t)); after gamma acceptances draw the bonus from p_{gamma+1}).
//
// The draft distribution q_t lives on the shortlist only; for a full-vocabulary token v it is
// found through the cluster inverse (cluster_of, rank_in_cluster) and the list's cluster
// positions (cpos): j = cpos[cluster_of[v]] + rank_in_cluster[v], or q = 0 when cpos < 0.  So
// no dense copy of q is ever built.
//
// Chain layout of the work (memory-bound; every target row is read once for its softmax
// statistics, and one row per sequence again, from L2, for the residual draw):
//   1. verify_stats_kernel   grid (chunks, B*(gamma+1)): per-chunk max / sum-exp / argmax of
//      each target row and max / sum-exp of each draft row; the last block of a sequence
//      folds them (fixed order) and takes all gamma accept tests in parallel.
//   2. verify_residual_kernel grid (chunks, B): per-chunk mass of the residual (or of p for
//      the bonus draw); the last block of a sequence locates the inverse-CDF crossing chunk
//      and scans it.
#include "common.cuh"
#include "block_scan.cuh"

namespace ds {
namespace {

constexpr int kVThreads = 256;
constexpr int kVPer = 8;                         // elements per thread per chunk
constexpr int kVChunk = kVThreads * kVPer;       // 2048
constexpr int kMaxGamma = 32;
constexpr int kRPer = 4;                         // residual pass: elements per thread
constexpr int kRChunk = kVThreads * kRPer;       // 1024

struct PStat { float m, s, amax; int aid; };   // target-row chunk: max, sum-exp, argmax
struct QStat { float m, s; };

// Reads of partials other blocks published (L2, not the incoherent L1).
__device__ __forceinline__ PStat ldcg(const PStat *p)
{
    const float4 f = __ldcg(reinterpret_cast<const float4 *>(p));
    return PStat{f.x, f.y, f.z, __float_as_int(f.w)};
}
__device__ __forceinline__ QStat ldcg(const QStat *p)
{
    const float2 f = __ldcg(reinterpret_cast<const float2 *>(p));
    return QStat{f.x, f.y};
}

__device__ __forceinline__ PStat pstat_merge(PStat a, const PStat &b)
{
    if (b.m > a.m) { a.s = (a.m == -INFINITY ? 0.f : a.s * __expf(a.m - b.m)) + b.s; a.m = b.m; }
    else if (b.m != -INFINITY) a.s += b.s * __expf(b.m - a.m);
    if (b.aid >= 0 && (a.aid < 0 || b.amax > a.amax || (b.amax == a.amax && b.aid < a.aid))) { a.amax = b.amax; a.aid = b.aid; }
    return a;
}

__device__ __forceinline__ PStat shfl_xor_pstat(const PStat &a, int o)
{
    return PStat{__shfl_xor_sync(0xFFFFFFFFu, a.m, o), __shfl_xor_sync(0xFFFFFFFFu, a.s, o),
                 __shfl_xor_sync(0xFFFFFFFFu, a.amax, o), __shfl_xor_sync(0xFFFFFFFFu, a.aid, o)};
}

__device__ float block_sum(float x, float *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum(x);
    __syncthreads();
    if (lane == 0) scratch[warp] = x;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < int(blockDim.x >> 5); ++w) r += scratch[w];
    __syncthreads();
    return r;
}

// Statistics of one chunk of a row of length n: max and sum-exp of x = value * inv_te, and the
// argmax of the raw values (ties to the lower index).  Two plain block reductions (the max,
// then the sum of exp(x - max)); the result is valid in thread 0.
__device__ PStat chunk_stats(const float *__restrict__ row, int lo, int n, float inv_te, PStat *scratch)
{
    float vals[kVPer];
    const int base = lo + threadIdx.x * kVPer;
    if (base + kVPer <= n && (reinterpret_cast<uintptr_t>(row + base) & 15) == 0) {
#pragma unroll
        for (int i = 0; i < kVPer; i += 4) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(row + base + i));
            vals[i] = f.x; vals[i + 1] = f.y; vals[i + 2] = f.z; vals[i + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kVPer; ++i) vals[i] = base + i < n ? __ldg(row + base + i) : -INFINITY;
    }
    float amax = -INFINITY;
    int aid = -1;
#pragma unroll
    for (int i = 0; i < kVPer; ++i)
        if (vals[i] > amax) { amax = vals[i]; aid = base + i; }     // first max = lowest index
    // block max / argmax of the raw values (x = value * inv_te is monotone in the value)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, aid, o);
        if (oi >= 0 && (aid < 0 || ov > amax || (ov == amax && oi < aid))) { amax = ov; aid = oi; }
    }
    if (lane == 0) { scratch[warp].amax = amax; scratch[warp].aid = aid; }
    __syncthreads();
    float bmax = -INFINITY;
    int bid = -1;
    for (int w = 0; w < nw; ++w) {
        const float ov = scratch[w].amax;
        const int oi = scratch[w].aid;
        if (oi >= 0 && (bid < 0 || ov > bmax || (ov == bmax && oi < bid))) { bmax = ov; bid = oi; }
    }
    const float m = bid >= 0 ? bmax * inv_te : -INFINITY;
    float sl = 0.f;
    if (bid >= 0) {
#pragma unroll
        for (int i = 0; i < kVPer; ++i) sl += __expf(vals[i] * inv_te - m);
    }
    sl = warp_sum(sl);
    __syncthreads();                                   // everyone has read scratch
    if (lane == 0) scratch[warp].s = sl;
    __syncthreads();
    PStat r{m, 0.f, bmax, bid};
    if (threadIdx.x == 0) for (int w = 0; w < nw; ++w) r.s += scratch[w].s;
    __syncthreads();
    return r;
}

struct ChainArgs {
    const float *p_logits;
    int B, gamma, V, nch;
    float T, inv_te;
    const float *q_logits;
    int64_t q_stride;
    const float *q_max, *q_sumexp;     // optional [gamma][B] draft-row statistics
    const int32_t *vs_offsets, *cpos;
    int M;
    const int32_t *cluster_of, *rank;
    const int32_t *draft_ids;
    const float *u;
    int32_t *accepted, *correction;
    int32_t *status;
    // workspace
    unsigned *cnt1, *cnt2;
    PStat *pstat;       // [B][gamma+1][nch]
    QStat *qstat;       // [B][gamma][nch]
    QStat *prow;        // [B][gamma+1] folded target stats
    QStat *qrow;        // [B][gamma]   folded draft stats
    int32_t *decision;  // [B]: -1 done, else the target row to draw from (t* or gamma)
    int nrch;           // residual-pass chunks
    float *rsum, *psum; // [B][nrch]
};

// Index of full-vocabulary token v in list (t, b), or -1.
__device__ __forceinline__ int list_index(const ChainArgs &a, int t, int b, int v)
{
    if (v < 0 || v >= a.V) return -1;
    const int c = a.cluster_of[v];
    const int p = a.cpos[(size_t(t) * a.B + b) * a.M + c];
    return p < 0 ? -1 : p + a.rank[v];
}

__global__ void __launch_bounds__(kVThreads)
verify_stats_kernel(ChainArgs a)
{
    __shared__ PStat scratch[kVThreads / 32];
    __shared__ PStat rows[kMaxGamma + 1];
    __shared__ QStat qrows[kMaxGamma];
    __shared__ int rej[kMaxGamma];
    const int g1 = a.gamma + 1;
    const int b = blockIdx.y / g1, t = blockIdx.y % g1;
    const int c = blockIdx.x;
    const int lo = c * kVChunk;
    {
        const float *row = a.p_logits + (size_t(b) * g1 + t) * a.V;
        const PStat ps = chunk_stats(row, lo, a.V, a.inv_te, scratch);
        if (threadIdx.x == 0) a.pstat[(size_t(b) * g1 + t) * a.nch + c] = ps;
    }
    if (t < a.gamma && a.T > 0.f && !a.q_max) {
        const int *off = a.vs_offsets + size_t(t) * (a.B + 1);
        const int n = off[b + 1] - off[b];
        QStat q{-INFINITY, 0.f};
        if (lo < n) {
            const PStat qs = chunk_stats(a.q_logits + size_t(t) * a.q_stride + off[b], lo, n, a.inv_te, scratch);
            q = QStat{qs.m, qs.s};
        }
        if (threadIdx.x == 0) a.qstat[(size_t(b) * a.gamma + t) * a.nch + c] = q;
    }
    if (!last_block_done(&a.cnt1[b], unsigned(g1) * a.nch)) return;

    // Fold the chunk statistics of this sequence's rows: warp w takes rows w, w+8, ...
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nrows = g1 + (a.T > 0.f && !a.q_max ? a.gamma : 0);
    if (a.T > 0.f && a.q_max && threadIdx.x < a.gamma) {
        const int tt = threadIdx.x;
        const QStat q{a.q_max[size_t(tt) * a.B + b], a.q_sumexp[size_t(tt) * a.B + b]};
        qrows[tt] = q;
        a.qrow[size_t(b) * a.gamma + tt] = q;
    }
    for (int r = warp; r < nrows; r += kVThreads / 32) {
        PStat acc{-INFINITY, 0.f, -INFINITY, -1};
        if (r < g1) {
            for (int i = lane; i < a.nch; i += 32) acc = pstat_merge(acc, ldcg(&a.pstat[(size_t(b) * g1 + r) * a.nch + i]));
        } else {
            for (int i = lane; i < a.nch; i += 32) {
                const QStat q = ldcg(&a.qstat[(size_t(b) * a.gamma + (r - g1)) * a.nch + i]);
                acc = pstat_merge(acc, PStat{q.m, q.s, -INFINITY, -1});
            }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const PStat q = shfl_xor_pstat(acc, o);
            acc = (lane & o) ? pstat_merge(q, acc) : pstat_merge(acc, q);
        }
        if (lane == 0) {
            if (r < g1) { rows[r] = acc; a.prow[size_t(b) * g1 + r] = QStat{acc.m, acc.s}; }
            else { qrows[r - g1] = QStat{acc.m, acc.s}; a.qrow[size_t(b) * a.gamma + (r - g1)] = QStat{acc.m, acc.s}; }
        }
    }
    __syncthreads();
    // All gamma accept tests at once; the first rejection decides.
    if (threadIdx.x < a.gamma) {
        const int tt = threadIdx.x;
        const int x = a.draft_ids[size_t(tt) * a.B + b];
        int reject;
        if (a.T == 0.f) {
            reject = (x != rows[tt].aid);
        } else {
            const int j = list_index(a, tt, b, x);
            if (j < 0) {
                set_status(a.status, DS_DEV_BAD_INDEX);
                reject = 1;
            } else {
                const int *off = a.vs_offsets + size_t(tt) * (a.B + 1);
                const float l = a.q_logits[size_t(tt) * a.q_stride + off[b] + j];
                const float q = __expf(l * a.inv_te - qrows[tt].m) / qrows[tt].s;
                const float z = a.p_logits[(size_t(b) * g1 + tt) * a.V + x];
                const float p = __expf(z * a.inv_te - rows[tt].m) / rows[tt].s;
                reject = !(a.u[size_t(b) * g1 + tt] * q < p);
            }
        }
        rej[tt] = reject;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ts = a.gamma;
        for (int tt = 0; tt < a.gamma; ++tt) if (rej[tt]) { ts = tt; break; }
        a.accepted[b] = ts;
        if (a.T == 0.f) {
            a.correction[b] = rows[ts].aid;
            a.decision[b] = -1;
        } else {
            a.decision[b] = ts;
        }
    }
}

// Residual weight of token v at target row tr: max(0, p - q) at a rejection (tr < gamma),
// p itself for the bonus draw (tr == gamma).
struct ResidualRow {
    const float *z;            // target logits of row tr
    float pm, ps;              // its softmax statistics
    const float *ql;           // draft logits of list (tr, b), or nullptr for the bonus row
    const int32_t *cposb;      // cpos of list (tr, b)
    float qm, qs;
};

__device__ __forceinline__ void residual_weight(const ChainArgs &a, const ResidualRow &rr, int v,
                                                float &r, float &p)
{
    p = __expf(rr.z[v] * a.inv_te - rr.pm) / rr.ps;
    float q = 0.f;
    if (rr.ql) {
        const int pc = rr.cposb[a.cluster_of[v]];
        if (pc >= 0) q = __expf(rr.ql[pc + a.rank[v]] * a.inv_te - rr.qm) / rr.qs;
    }
    r = fmaxf(p - q, 0.f);
}

__device__ ResidualRow residual_row(const ChainArgs &a, int b, int tr)
{
    const int g1 = a.gamma + 1;
    ResidualRow rr;
    rr.z = a.p_logits + (size_t(b) * g1 + tr) * a.V;
    const QStat pr = ldcg(&a.prow[size_t(b) * g1 + tr]);
    rr.pm = pr.m; rr.ps = pr.s;
    rr.ql = nullptr; rr.cposb = nullptr; rr.qm = 0.f; rr.qs = 1.f;
    if (tr < a.gamma) {
        const int *off = a.vs_offsets + size_t(tr) * (a.B + 1);
        rr.ql = a.q_logits + size_t(tr) * a.q_stride + off[b];
        rr.cposb = a.cpos + (size_t(tr) * a.B + b) * a.M;
        const QStat qr = ldcg(&a.qrow[size_t(b) * a.gamma + tr]);
        rr.qm = qr.m; rr.qs = qr.s;
    }
    return rr;
}

__global__ void __launch_bounds__(kVThreads)
verify_residual_kernel(ChainArgs a)
{
    __shared__ float scratch[kVThreads / 32];
    __shared__ float sbuf[kVThreads + 1];
    __shared__ float fscan[33];
    __shared__ int s_chunk, s_use_p, s_hit, s_last;
    __shared__ float s_target;
    const int b = blockIdx.y, c = blockIdx.x;
    const int tr = __ldcg(&a.decision[b]);
    if (tr < 0) return;                              // greedy: decided already (whole group returns)
    const ResidualRow rr = residual_row(a, b, tr);
    const int base = c * kRChunk + threadIdx.x * kRPer;
    float rs = 0.f, psum = 0.f;
#pragma unroll
    for (int i = 0; i < kRPer; ++i) {
        const int v = base + i;
        if (v < a.V) { float r, p; residual_weight(a, rr, v, r, p); rs += r; psum += p; }
    }
    rs = block_sum(rs, scratch);
    psum = block_sum(psum, scratch);
    if (threadIdx.x == 0) { a.rsum[size_t(b) * a.nrch + c] = rs; a.psum[size_t(b) * a.nrch + c] = psum; }
    if (!last_block_done(&a.cnt2[b], unsigned(a.nrch))) return;

    // Locate the chunk where the cumulative mass first exceeds u * total: thread t sums a
    // contiguous run of chunk masses, the runs are scanned in thread order, and the thread
    // whose run crosses walks it.  A residual without mass falls back to p.
    const float u = a.u[size_t(b) * (a.gamma + 1) + a.gamma];
    const int E = (a.nrch + kVThreads - 1) / kVThreads;
    const int c0 = threadIdx.x * E, c1 = min(a.nrch, c0 + E);
    float rrun = 0.f, prun = 0.f;
    for (int i = c0; i < c1; ++i) {
        rrun += __ldcg(&a.rsum[size_t(b) * a.nrch + i]);
        prun += __ldcg(&a.psum[size_t(b) * a.nrch + i]);
    }
    block_cdf_bounds(rrun, sbuf, fscan);
    const float rtot = sbuf[kVThreads];
    const int use_p = !(rtot > 0.f);
    if (use_p) block_cdf_bounds(prun, sbuf, fscan);
    const float *w = use_p ? a.psum : a.rsum;
    const float target = u * sbuf[kVThreads];
    const float lo_b = sbuf[threadIdx.x], hi_b = sbuf[threadIdx.x + 1];
    if (threadIdx.x == 0) { s_hit = 0x7FFFFFFF; s_last = -1; }
    __syncthreads();
    if (lo_b <= target && target < hi_b) atomicMin(&s_hit, threadIdx.x);
    int lastc = -1;
    for (int i = c0; i < c1; ++i) if (__ldcg(&w[size_t(b) * a.nrch + i]) > 0.f) lastc = i;
    if (lastc >= 0) atomicMax(&s_last, lastc);
    __syncthreads();
    if (int(threadIdx.x) == s_hit) {               // the first claimant walks its run of chunks
        float cum = lo_b;
        int ch = -1;
        for (int i = c0; i < c1; ++i) {
            const float wi = __ldcg(&w[size_t(b) * a.nrch + i]);
            if (cum + wi > target) { ch = i; break; }
            cum += wi;
        }
        if (ch < 0) {                               // rounding inside the run: its last chunk with mass
            for (int i = c1 - 1; i >= c0; --i) if (__ldcg(&w[size_t(b) * a.nrch + i]) > 0.f) { ch = i; break; }
            s_target = INFINITY;
        } else {
            s_target = target - cum;
        }
        s_chunk = ch < 0 ? max(s_last, 0) : ch;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (s_hit == 0x7FFFFFFF) { s_chunk = max(s_last, 0); s_target = INFINITY; }   // target beyond total
        s_use_p = use_p;
        s_hit = 0x7FFFFFFF;
        s_last = -1;
    }
    __syncthreads();

    // Scan the chunk: per-thread segment sums, block scan in thread order, then the segment.
    const int lo = s_chunk * kRChunk + threadIdx.x * kRPer;
    float wv[kRPer];
    float seg = 0.f;
#pragma unroll
    for (int i = 0; i < kRPer; ++i) {
        const int v = lo + i;
        float r = 0.f, p = 0.f;
        if (v < a.V) residual_weight(a, rr, v, r, p);
        wv[i] = s_use_p ? p : r;
        seg += wv[i];
    }
    block_cdf_bounds(seg, sbuf, fscan);
    const float tgt = s_target;
    const float lo_s = sbuf[threadIdx.x], hi_s = sbuf[threadIdx.x + 1];
    int last_pos = -1;
#pragma unroll
    for (int i = 0; i < kRPer; ++i) if (wv[i] > 0.f) last_pos = lo + i;
    if (last_pos >= 0) atomicMax(&s_last, last_pos);
    if (lo_s <= tgt && tgt < hi_s) atomicMin(&s_hit, threadIdx.x);
    __syncthreads();
    if (int(threadIdx.x) == s_hit) {
        float cum = lo_s;
        int v = -1;
#pragma unroll
        for (int i = 0; i < kRPer; ++i) {
            cum += wv[i];
            if (v < 0 && cum > tgt) v = lo + i;
        }
        if (v < 0) v = last_pos;                    // rounding inside the segment
        a.correction[b] = v >= 0 ? v : s_last;
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_hit == 0x7FFFFFFF) a.correction[b] = s_last;   // target beyond the chunk
}

// ---------------------------------------------------------------------------------------
// Tree verification.  The pages cite EAGLE-style token trees but state no tree verifier;
// reading: sibling-sequential recursive rejection (the multi-draft form of speculative
// sampling).  All nodes of one depth share their sequence's shortlist, so the residual
// after a rejected sibling differs from the current target only on that shortlist: the walk
// keeps it as (O = target mass off the list, r_j on the list) and never builds a dense row.
// ---------------------------------------------------------------------------------------
constexpr int kWalkThreads = 1024;

struct TreeArgs {
    const float *p_logits;
    int B, D, Wd, N, V, nch;
    float T, inv_te;
    const int32_t *parent;
    const float *q_logits;
    int64_t q_stride;
    const int32_t *vs_offsets, *cpos;
    int M;
    const int32_t *cluster_of, *rank;
    const int32_t *node_tokens;
    const float *u_node, *u_res;
    int32_t *accepted, *correction, *path;
    int32_t *status;
    PStat *tpstat;     // [B][1+N][nch]
    QStat *tqstat;     // [B][N][nch]
    float *rbuf;       // [B][V]
};

// Node n's draft row: logits, length.
__device__ __forceinline__ const float *node_row(const TreeArgs &a, int b, int n, int *len)
{
    const int dep0 = n / a.Wd, i = n - dep0 * a.Wd;
    const int *off = a.vs_offsets + size_t(dep0) * (a.B + 1);
    const int nb = off[b + 1] - off[b];
    *len = nb;
    return a.q_logits + size_t(dep0) * a.q_stride + int64_t(off[b]) * a.Wd + int64_t(i) * nb;
}

__global__ void __launch_bounds__(kVThreads)
tree_stats_kernel(TreeArgs a)
{
    __shared__ PStat scratch[kVThreads / 32];
    const int b = blockIdx.y / (1 + a.N), rr = blockIdx.y % (1 + a.N);
    const int c = blockIdx.x, lo = c * kVChunk;
    const PStat ps = chunk_stats(a.p_logits + (size_t(b) * (1 + a.N) + rr) * a.V, lo, a.V, a.inv_te, scratch);
    if (threadIdx.x == 0) a.tpstat[(size_t(b) * (1 + a.N) + rr) * a.nch + c] = ps;
    if (rr >= 1 && a.T > 0.f) {
        int nb;
        const float *ql = node_row(a, b, rr - 1, &nb);
        QStat q{-INFINITY, 0.f};
        if (lo < nb) { const PStat qs = chunk_stats(ql, lo, nb, a.inv_te, scratch); q = QStat{qs.m, qs.s}; }
        if (threadIdx.x == 0) a.tqstat[(size_t(b) * a.N + (rr - 1)) * a.nch + c] = q;
    }
}

// Warp 0 folds `nch` chunk partials (stride 1) in a fixed order; the result lands in *out.
__device__ void fold_pstats(const PStat *src, int nch, PStat *out)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        PStat acc{-INFINITY, 0.f, -INFINITY, -1};
        for (int i = lane; i < nch; i += 32) acc = pstat_merge(acc, ldcg(&src[i]));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const PStat q = shfl_xor_pstat(acc, o);
            acc = (lane & o) ? pstat_merge(q, acc) : pstat_merge(acc, q);
        }
        if (lane == 0) *out = acc;
    }
    __syncthreads();
}

__device__ void fold_qstats(const QStat *src, int nch, PStat *out)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        PStat acc{-INFINITY, 0.f, -INFINITY, -1};
        for (int i = lane; i < nch; i += 32) { const QStat q = ldcg(&src[i]); acc = pstat_merge(acc, PStat{q.m, q.s, -INFINITY, -1}); }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const PStat q = shfl_xor_pstat(acc, o);
            acc = (lane & o) ? pstat_merge(q, acc) : pstat_merge(acc, q);
        }
        if (lane == 0) *out = acc;
    }
    __syncthreads();
}

// Inverse-CDF draw over weights w(v), v = 0..V-1 ascending: the smallest v whose cumulative
// weight exceeds `target`; if rounding leaves none, the last v with positive weight.  Thread t
// owns a contiguous segment; segment sums are scanned in thread order.
template <typename WF>
__device__ int block_icdf(WF wf, int V, float u, float *sbuf, float *scratch, int *ibuf)
{
    const int E = (V + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * E, hi = min(V, lo + E);
    float seg = 0.f;
    int last = -1;
    for (int v = lo; v < hi; ++v) { const float w = wf(v); seg += w; if (w > 0.f) last = v; }
    block_cdf_bounds(seg, sbuf, scratch);
    const float target = u * sbuf[blockDim.x];
    const float lo_b = sbuf[threadIdx.x], hi_b = sbuf[threadIdx.x + 1];
    if (threadIdx.x == 0) { ibuf[0] = 0x7FFFFFFF; ibuf[1] = -1; ibuf[2] = -1; }
    __syncthreads();
    if (lo_b <= target && target < hi_b) atomicMin(&ibuf[0], threadIdx.x);
    if (last >= 0) atomicMax(&ibuf[1], last);
    __syncthreads();
    if (int(threadIdx.x) == ibuf[0]) {              // the first claimant walks its segment
        float cum = lo_b;
        int hit = -1;
        for (int v = lo; v < hi; ++v) { cum += wf(v); if (cum > target) { hit = v; break; } }
        ibuf[2] = hit >= 0 ? hit : last;            // rounding inside the segment: its last positive
    }
    __syncthreads();
    const int r = ibuf[2] >= 0 ? ibuf[2] : ibuf[1];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kWalkThreads)
tree_walk_kernel(TreeArgs a)
{
    __shared__ PStat s_p, s_q;
    __shared__ float fscr[33];
    __shared__ float sbuf[kWalkThreads + 1];
    __shared__ int ibuf[3];
    __shared__ int s_kids[64];
    __shared__ int s_nkids, s_accept;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    float *r = a.rbuf + size_t(b) * a.V;
    if (tid < a.D) a.path[size_t(b) * a.D + tid] = -1;
    int cur = -1, dep = 0, A = 0, corr = -1;
    for (int guard = 0; guard <= a.D; ++guard) {
        fold_pstats(a.tpstat + (size_t(b) * (1 + a.N) + (cur + 1)) * a.nch, a.nch, &s_p);
        const float *z = a.p_logits + (size_t(b) * (1 + a.N) + (cur + 1)) * a.V;
        const float pm = s_p.m, ps = s_p.s;
        if (tid == 0) {
            int nk = 0;
            if (dep < a.D)
                for (int i = 0; i < a.Wd; ++i) {
                    const int n = dep * a.Wd + i;
                    if (a.parent[n] == cur) s_kids[nk++] = n;
                }
            s_nkids = nk;
        }
        __syncthreads();
        const int nk = s_nkids;
        const int32_t *cposL = a.cpos + (size_t(dep < a.D ? dep : 0) * a.B + b) * a.M;
        if (a.T == 0.f) {
            const int am = s_p.aid;
            int next = -1;
            for (int k = 0; k < nk; ++k) {
                const int n = s_kids[k];
                if (a.node_tokens[size_t(dep) * a.B * a.Wd + size_t(b) * a.Wd + (n - dep * a.Wd)] == am) { next = n; break; }
            }
            if (next < 0) { corr = am; break; }
            if (tid == 0) a.path[size_t(b) * a.D + A] = next;
            ++A; cur = next; ++dep;
            continue;
        }
        auto pval = [&](int v) { return __expf(z[v] * a.inv_te - pm) / ps; };
        if (nk == 0) {
            corr = block_icdf(pval, a.V, a.u_res[size_t(b) * (a.D + 1) + dep], sbuf, fscr, ibuf);
            break;
        }
        // residual state for the children's shared list: O off the list, r_j on it
        float off_mass = 0.f, on_mass = 0.f;
        for (int v = tid; v < a.V; v += blockDim.x) {
            const float p = pval(v);
            const int pc = cposL[a.cluster_of[v]];
            if (pc < 0) off_mass += p;
            else { r[pc + a.rank[v]] = p; on_mass += p; }
        }
        const float O = block_sum(off_mass, fscr);
        float R = O + block_sum(on_mass, fscr);
        int next = -1;
        for (int k = 0; k < nk; ++k) {
            const int n = s_kids[k];
            int nb;
            const float *ql = node_row(a, b, n, &nb);
            fold_qstats(a.tqstat + (size_t(b) * a.N + n) * a.nch, a.nch, &s_q);
            const float qm = s_q.m, qs = s_q.s;
            if (tid == 0) {
                const int x = a.node_tokens[size_t(dep) * a.B * a.Wd + size_t(b) * a.Wd + (n - dep * a.Wd)];
                int j = -1;
                if (x >= 0 && x < a.V) { const int pc = cposL[a.cluster_of[x]]; if (pc >= 0) j = pc + a.rank[x]; }
                int acc = 0;
                if (j < 0) set_status(a.status, DS_DEV_BAD_INDEX);
                else {
                    const float q = __expf(ql[j] * a.inv_te - qm) / qs;
                    acc = a.u_node[size_t(b) * a.N + n] * q < r[j] / R;
                }
                s_accept = acc;
            }
            __syncthreads();
            if (s_accept) { next = n; break; }
            float part = 0.f;
            for (int j = tid; j < nb; j += blockDim.x)
                part += fmaxf(r[j] - R * (__expf(ql[j] * a.inv_te - qm) / qs), 0.f);
            const float Rn = O + block_sum(part, fscr);
            if (Rn > 0.f) {
                for (int j = tid; j < nb; j += blockDim.x)
                    r[j] = fmaxf(r[j] - R * (__expf(ql[j] * a.inv_te - qm) / qs), 0.f);
                R = Rn;
            }
            __syncthreads();
        }
        if (next >= 0) {
            if (tid == 0) a.path[size_t(b) * a.D + A] = next;
            ++A; cur = next; ++dep;
            continue;
        }
        const float u = a.u_res[size_t(b) * (a.D + 1) + dep];
        auto wres = [&](int v) {
            const int pc = cposL[a.cluster_of[v]];
            return pc < 0 ? pval(v) : r[pc + a.rank[v]];
        };
        corr = block_icdf(wres, a.V, u, sbuf, fscr, ibuf);
        break;
    }
    if (tid == 0) { a.accepted[b] = A; a.correction[b] = corr; }
}

}  // namespace
}  // namespace ds

using namespace ds;

static int vchunks(int V) { return (V + kVChunk - 1) / kVChunk; }
static size_t rchunks(int V) { return size_t((V + kRChunk - 1) / kRChunk); }

extern "C" size_t ds_verify_workspace_bytes(int B, int gamma, int V)
{
    if (B <= 0 || gamma <= 0 || V <= 0) return 0;
    const size_t nch = size_t(vchunks(V));
    const size_t g1 = size_t(gamma) + 1;
    return align256(2 * size_t(B) * sizeof(unsigned)) +
           align256(size_t(B) * g1 * nch * sizeof(PStat)) +
           align256(size_t(B) * gamma * nch * sizeof(QStat)) +
           align256(size_t(B) * g1 * sizeof(QStat)) +
           align256(size_t(B) * gamma * sizeof(QStat)) +
           align256(size_t(B) * sizeof(int32_t)) +
           2 * align256(size_t(B) * rchunks(V) * sizeof(float));
}

extern "C" ds_status ds_verify(const float *p_logits, int B, int gamma, int V, float T,
                               const float *q_logits, int64_t q_stride,
                               const float *q_max, const float *q_sumexp,
                               const int32_t *vs_offsets, const int32_t *cpos, int M,
                               const int32_t *cluster_of, const int32_t *rank_in_cluster,
                               const int32_t *draft_ids, const float *uniforms,
                               int32_t *accepted_len, int32_t *correction,
                               void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    if (!p_logits || !q_logits || !vs_offsets || !cpos || !cluster_of || !rank_in_cluster ||
        !draft_ids || !uniforms || !accepted_len || !correction)
        return DS_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > kMaxGamma || V < 1 || V > (1 << 24) || M < 1 || M > 8192 ||
        !(T >= 0.f) || q_stride < 0)
        return DS_ERR_INVALID_ARG;
    if ((q_max == nullptr) != (q_sumexp == nullptr)) return DS_ERR_INVALID_ARG;
    if (B > 65535 / (gamma + 1)) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_verify_workspace_bytes(B, gamma, V)) return DS_ERR_WORKSPACE;
    ChainArgs a;
    a.p_logits = p_logits; a.B = B; a.gamma = gamma; a.V = V; a.nch = vchunks(V);
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.q_logits = q_logits; a.q_stride = q_stride;
    a.q_max = q_max; a.q_sumexp = q_sumexp;
    a.vs_offsets = vs_offsets; a.cpos = cpos; a.M = M;
    a.cluster_of = cluster_of; a.rank = rank_in_cluster;
    a.draft_ids = draft_ids; a.u = uniforms;
    a.accepted = accepted_len; a.correction = correction; a.status = dev_status;
    char *w = static_cast<char *>(ws);
    const size_t nch = size_t(a.nch), g1 = size_t(gamma) + 1;
    a.cnt1 = reinterpret_cast<unsigned *>(w); a.cnt2 = a.cnt1 + B;
    w += align256(2 * size_t(B) * sizeof(unsigned));
    a.pstat = reinterpret_cast<PStat *>(w); w += align256(size_t(B) * g1 * nch * sizeof(PStat));
    a.qstat = reinterpret_cast<QStat *>(w); w += align256(size_t(B) * gamma * nch * sizeof(QStat));
    a.prow = reinterpret_cast<QStat *>(w); w += align256(size_t(B) * g1 * sizeof(QStat));
    a.qrow = reinterpret_cast<QStat *>(w); w += align256(size_t(B) * gamma * sizeof(QStat));
    a.decision = reinterpret_cast<int32_t *>(w); w += align256(size_t(B) * sizeof(int32_t));
    a.nrch = int(rchunks(V));
    a.rsum = reinterpret_cast<float *>(w); w += align256(size_t(B) * rchunks(V) * sizeof(float));
    a.psum = reinterpret_cast<float *>(w);

    verify_stats_kernel<<<dim3(a.nch, B * (gamma + 1)), kVThreads, 0, stream>>>(a);
    DS_TRY_LAUNCH();
    verify_residual_kernel<<<dim3(a.nrch, B), kVThreads, 0, stream>>>(a);
    DS_TRY_LAUNCH();
    return DS_OK;
}

extern "C" size_t ds_verify_tree_workspace_bytes(int B, int D, int Wd, int V)
{
    if (B <= 0 || D <= 0 || Wd <= 0 || V <= 0) return 0;
    const size_t nch = size_t(vchunks(V)), N = size_t(D) * Wd;
    return align256(size_t(B) * (1 + N) * nch * sizeof(PStat)) +
           align256(size_t(B) * N * nch * sizeof(QStat)) +
           align256(size_t(B) * size_t(V) * sizeof(float));
}

extern "C" ds_status ds_verify_tree(const float *p_logits, int B, int D, int Wd, int V, float T,
                                    const int32_t *parent,
                                    const float *q_logits, int64_t q_stride,
                                    const int32_t *vs_offsets, const int32_t *cpos, int M,
                                    const int32_t *cluster_of, const int32_t *rank_in_cluster,
                                    const int32_t *node_tokens, const float *u_node, const float *u_res,
                                    int32_t *accepted_len, int32_t *correction, int32_t *path,
                                    void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    if (!p_logits || !parent || !q_logits || !vs_offsets || !cpos || !cluster_of || !rank_in_cluster ||
        !node_tokens || !u_node || !u_res || !accepted_len || !correction || !path)
        return DS_ERR_INVALID_ARG;
    if (B < 1 || D < 1 || D > kMaxGamma || Wd < 1 || Wd > 64 || V < 1 || V > (1 << 24) || M < 1 ||
        M > 8192 || !(T >= 0.f) || q_stride < 0)
        return DS_ERR_INVALID_ARG;
    const int N = D * Wd;
    if (size_t(B) * (1 + N) > 65535) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_verify_tree_workspace_bytes(B, D, Wd, V)) return DS_ERR_WORKSPACE;
    TreeArgs a;
    a.p_logits = p_logits; a.B = B; a.D = D; a.Wd = Wd; a.N = N; a.V = V; a.nch = vchunks(V);
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.parent = parent; a.q_logits = q_logits; a.q_stride = q_stride;
    a.vs_offsets = vs_offsets; a.cpos = cpos; a.M = M;
    a.cluster_of = cluster_of; a.rank = rank_in_cluster;
    a.node_tokens = node_tokens; a.u_node = u_node; a.u_res = u_res;
    a.accepted = accepted_len; a.correction = correction; a.path = path; a.status = dev_status;
    char *w = static_cast<char *>(ws);
    const size_t nch = size_t(a.nch);
    a.tpstat = reinterpret_cast<PStat *>(w); w += align256(size_t(B) * (1 + N) * nch * sizeof(PStat));
    a.tqstat = reinterpret_cast<QStat *>(w); w += align256(size_t(B) * N * nch * sizeof(QStat));
    a.rbuf = reinterpret_cast<float *>(w);
    tree_stats_kernel<<<dim3(a.nch, B * (1 + N)), kVThreads, 0, stream>>>(a);
    DS_TRY_LAUNCH();
    tree_walk_kernel<<<B, kWalkThreads, 0, stream>>>(a);
    DS_TRY_LAUNCH();
    return DS_OK;
}
