// Speculative-sampling verification over the full vocabulary.
//
// DynaSpec abstract (verification by the target model stays over the whole vocabulary, so
// the output distribution is unchanged); summary, Technical Details > Pipeline Flow ("Rejection Sampling
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
#include <cooperative_groups.h>

#include "common.cuh"
#include "block_scan.cuh"

namespace cg = cooperative_groups;

namespace ds {
namespace {

constexpr int kVThreads = 256;
// Statistics chunks: 8192 elements (32 per thread, 8 float4 loads in flight) when that still
// gives the GPU at least two blocks per SM, else 2048 (few rows: more, smaller blocks).
constexpr int kVPerBig = 32, kVPerSmall = 8;
constexpr int kVChunkMin = kVThreads * kVPerSmall;   // sizes the workspace
constexpr int kMaxGamma = 32;
// Residual chunks: 2048 elements (8 per thread) under the same rule, else 512 (few sequences:
// more, shorter blocks for the dependent lookups of the draw).
constexpr int kRPerBig = 8, kRPerSmall = 2;
constexpr int kRChunkMin = kVThreads * kRPerSmall;

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

// a (earlier in the fixed order) merged with b, without branches (an empty state has m = -inf
// and aid = -1; one of the two scales is exactly 1).
__device__ __forceinline__ PStat pstat_merge(const PStat &a, const PStat &b)
{
    PStat r;
    r.m = fmaxf(a.m, b.m);
    const float ea = a.m == -INFINITY ? 0.f : __expf(a.m - r.m);
    const float eb = b.m == -INFINITY ? 0.f : __expf(b.m - r.m);
    r.s = fmaf(a.s, ea, b.s * eb);
    const bool tb = b.aid >= 0 && (a.aid < 0 || b.amax > a.amax || (b.amax == a.amax && b.aid < a.aid));
    r.amax = tb ? b.amax : a.amax;
    r.aid = tb ? b.aid : a.aid;
    return r;
}

// The warp's states reduced to one, held by every lane: the maximum and the argmax first, then
// the sums scaled once to the common maximum; every step is commutative, so the result does not
// depend on timing (see stat_reduce_lanes).
__device__ __forceinline__ PStat pstat_reduce_lanes(const PStat &mine)
{
    float m = mine.m, amax = mine.amax;
    int aid = mine.aid;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float a2 = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, aid, o);
        m = fmaxf(m, m2);
        const bool take = i2 >= 0 && (aid < 0 || a2 > amax || (a2 == amax && i2 < aid));
        amax = take ? a2 : amax;
        aid = take ? i2 : aid;
    }
    float s = mine.m == -INFINITY ? 0.f : mine.s * __expf(mine.m - m);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    return PStat{m, s, amax, aid};
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
// argmax of the raw values (ties to the lower index).  Each thread reduces its own values (its
// maximum, then its sum of exp(x - that maximum)), then one reduction over the block (the lanes
// in two commutative passes, then the warps); the result is valid in warp 0.
template <int kVPer>
__device__ PStat chunk_stats(const float *__restrict__ row, int lo, int n, float inv_te, PStat *scratch)
{
    // thread t holds the 4-element groups lo + 1024 k + 4 t: every round of loads is one
    // contiguous 4 KB of the row, and all rounds are in flight together
    float vals[kVPer];
    constexpr int kStride = kVThreads * 4;
#pragma unroll
    for (int k = 0; k < kVPer / 4; ++k) {
        const int g = lo + k * kStride + threadIdx.x * 4;
        if (g + 4 <= n && (reinterpret_cast<uintptr_t>(row + g) & 15) == 0) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(row + g));
            vals[4 * k] = f.x; vals[4 * k + 1] = f.y; vals[4 * k + 2] = f.z; vals[4 * k + 3] = f.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) vals[4 * k + e] = g + e < n ? __ldg(row + g + e) : -INFINITY;
        }
    }
    float amax = -INFINITY;
    int aid = -1;
#pragma unroll
    for (int i = 0; i < kVPer; ++i) {                  // indices rise with i: first max = lowest index
        const int idx = lo + (i >> 2) * kStride + threadIdx.x * 4 + (i & 3);
        if (vals[i] > amax) { amax = vals[i]; aid = idx; }
    }
    // x = value * inv_te is monotone in the value: the thread's maximum of x is amax * inv_te
    const float tm = aid >= 0 ? amax * inv_te : -INFINITY;
    float ts = 0.f;
    if (aid >= 0) {
#pragma unroll
        for (int i = 0; i < kVPer; ++i) ts += __expf(vals[i] * inv_te - tm);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const PStat w = pstat_reduce_lanes(PStat{tm, ts, amax, aid});
    if (lane == 0) scratch[warp] = w;
    __syncthreads();
    PStat r{-INFINITY, 0.f, -INFINITY, -1};
    if (warp == 0) r = pstat_reduce_lanes(lane < nw ? scratch[lane] : r);
    __syncthreads();                                   // the caller may reuse scratch
    return r;
}

// What the residual draw of one sequence needs from the decision, in one 32-byte record: the
// target row to draw from (-1: decided already), its softmax statistics, and for a rejection
// the list's offset and the draft row's statistics.
struct Decision {
    int tr, off;
    float pm, ps, qm, qs, pad0, pad1;
};
static_assert(sizeof(Decision) == 32, "two 16-byte loads");

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
    Decision *decision; // [B]
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

// Chunk c of target row t of sequence b: its max / sum-exp / argmax (and, at T > 0 without the
// head's row statistics, those of the draft row's chunk c).  The whole block calls it.
template <int kVPer>
__device__ void stats_unit(const ChainArgs &a, int b, int t, int c, PStat *scratch)
{
    const int g1 = a.gamma + 1;
    const int lo = c * kVThreads * kVPer;
    {
        const float *row = a.p_logits + (size_t(b) * g1 + t) * a.V;
        const PStat ps = chunk_stats<kVPer>(row, lo, a.V, a.inv_te, scratch);
        if (threadIdx.x == 0) a.pstat[(size_t(b) * g1 + t) * a.nch + c] = ps;
    }
    if (t < a.gamma && a.T > 0.f && !a.q_max) {
        const int *off = a.vs_offsets + size_t(t) * (a.B + 1);
        const int n = off[b + 1] - off[b];
        QStat q{-INFINITY, 0.f};
        if (lo < n) {
            const PStat qs = chunk_stats<kVPer>(a.q_logits + size_t(t) * a.q_stride + off[b], lo, n, a.inv_te, scratch);
            q = QStat{qs.m, qs.s};
        }
        if (threadIdx.x == 0) a.qstat[(size_t(b) * a.gamma + t) * a.nch + c] = q;
    }
}

// Sequence b, once every chunk's statistics are stored: fold them (fixed order), take all gamma
// accept tests at once and decide (accepted length; at T = 0 the correction too; else the
// target row to draw the correction from).  The whole block calls it.
__device__ void fold_decide(const ChainArgs &a, int b)
{
    __shared__ PStat rows[kMaxGamma + 1];
    __shared__ QStat qrows[kMaxGamma];
    __shared__ int rej[kMaxGamma];
    const int g1 = a.gamma + 1;
    // warp w folds rows w, w+8, ...
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nrows = g1 + (a.T > 0.f && !a.q_max ? a.gamma : 0);
    // The accept tests' inputs (each draft token, its place in its list, its draft logit, its
    // target logit, the uniform) need none of the row statistics: the last warp, which has the
    // fewest rows to fold, requests them first, so their chain of dependent loads runs while the
    // other warps fold.
    constexpr int kTestWarp = kVThreads / 32 - 1;
    const bool tester = warp == kTestWarp && lane < a.gamma;
    __shared__ int s_off[kMaxGamma];
    int x = -1, j = -1;
    float l = 0.f, z = 0.f, uu = 0.f;
    if (tester) {
        x = a.draft_ids[size_t(lane) * a.B + b];
        if (a.T > 0.f) {
            const int off = a.vs_offsets[size_t(lane) * (a.B + 1) + b];
            s_off[lane] = off;
            j = list_index(a, lane, b, x);
            if (j >= 0) {
                l = a.q_logits[size_t(lane) * a.q_stride + off + j];
                z = a.p_logits[(size_t(b) * g1 + lane) * a.V + x];
            }
            uu = a.u[size_t(b) * g1 + lane];
        }
    }
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
        acc = pstat_reduce_lanes(acc);
        if (lane == 0) {
            if (r < g1) { rows[r] = acc; a.prow[size_t(b) * g1 + r] = QStat{acc.m, acc.s}; }
            else { qrows[r - g1] = QStat{acc.m, acc.s}; a.qrow[size_t(b) * a.gamma + (r - g1)] = QStat{acc.m, acc.s}; }
        }
    }
    __syncthreads();
    // All gamma accept tests at once; the first rejection decides.
    if (tester) {
        const int tt = lane;
        int reject;
        if (a.T == 0.f) {
            reject = (x != rows[tt].aid);
        } else if (j < 0) {
            set_status(a.status, DS_DEV_BAD_INDEX);
            reject = 1;
        } else {
            const float q = __expf(l * a.inv_te - qrows[tt].m) / qrows[tt].s;
            const float p = __expf(z * a.inv_te - rows[tt].m) / rows[tt].s;
            reject = !(uu * q < p);
        }
        rej[tt] = reject;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int ts = a.gamma;
        for (int tt = 0; tt < a.gamma; ++tt) if (rej[tt]) { ts = tt; break; }
        a.accepted[b] = ts;
        Decision dsn{-1, 0, 0.f, 1.f, 0.f, 1.f, 0.f, 0.f};
        if (a.T == 0.f) {
            a.correction[b] = rows[ts].aid;
        } else {
            dsn.tr = ts;
            dsn.pm = rows[ts].m; dsn.ps = rows[ts].s;
            if (ts < a.gamma) { dsn.off = s_off[ts]; dsn.qm = qrows[ts].m; dsn.qs = qrows[ts].s; }
        }
        a.decision[b] = dsn;
    }
    __syncthreads();                                   // the block may call again (shared state)
}

template <int kVPer>
__global__ void __launch_bounds__(kVThreads, 4)
verify_stats_kernel(ChainArgs a)
{
    __shared__ PStat scratch[kVThreads / 32];
    pdl_wait();
    pdl_allow();
    const int g1 = a.gamma + 1;
    const int b = blockIdx.y / g1, t = blockIdx.y % g1;
    stats_unit<kVPer>(a, b, t, blockIdx.x, scratch);
    if (!last_block_done(&a.cnt1[b], unsigned(g1) * a.nch)) return;
    fold_decide(a, b);
}

// What the residual weights of target row tr need: max(0, p - q) at a rejection (tr < gamma),
// p itself for the bonus draw (tr == gamma).
struct ResidualRow {
    const float *z;            // target logits of row tr
    float pm, ps;              // its softmax statistics
    const float *ql;           // draft logits of list (tr, b), or nullptr for the bonus row
    const int32_t *cposb;      // cpos of list (tr, b)
    float qm, qs;
};

__device__ ResidualRow residual_row(const ChainArgs &a, int b, const Decision &dsn)
{
    const int g1 = a.gamma + 1, tr = dsn.tr;
    ResidualRow rr;
    rr.z = a.p_logits + (size_t(b) * g1 + tr) * a.V;
    rr.pm = dsn.pm; rr.ps = dsn.ps;
    rr.ql = nullptr; rr.cposb = nullptr; rr.qm = 0.f; rr.qs = 1.f;
    if (tr < a.gamma) {
        rr.ql = a.q_logits + size_t(tr) * a.q_stride + dsn.off;
        rr.cposb = a.cpos + (size_t(tr) * a.B + b) * a.M;
        rr.qm = dsn.qm; rr.qs = dsn.qs;
    }
    return rr;
}

__device__ __forceinline__ Decision ldcg(const Decision *p)
{
    const float4 f0 = __ldcg(reinterpret_cast<const float4 *>(p));
    const float4 f1 = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    return Decision{__float_as_int(f0.x), __float_as_int(f0.y), f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
}

// Inverse-CDF draw of one sequence over V weights, run by a grid (chunks of kRChunk, B).
// Pass 1 (every block): the chunk's mass of the primary weights r and of the fallback weights
// p.  Pass 2 (the last block of the sequence): locate the chunk where the cumulative mass
// first exceeds u * total -- thread t sums a contiguous run of chunk masses, the runs are
// scanned in thread order and the thread whose run crosses walks it -- then scan that chunk
// the same way.  Weights without mass fall back to p.  The draw is the smallest v whose
// cumulative weight exceeds the target; if rounding leaves none, the last v with weight.
// The policy P gives both weights of token v in two steps: load(v) issues the loads that need
// nothing else (target logit, cluster, rank), weights(raw, r, p) finishes them.  With
// P::kStaged, stage() fills the list's cluster positions into shared memory while the first
// loads are in flight and weights() looks them up there instead of in a third round of global
// loads (fewer dependent round trips, at the price of holding the first loads across a
// barrier: it pays when the grid is small, not on wide batched grids).
// Pass 1 for chunk c: its mass of the primary and the fallback weights, stored at rsum[c], psum[c].
template <int kRPer, class P>
__device__ void icdf_chunk(const P &pol, int V, int c, float *__restrict__ rsum, float *__restrict__ psum)
{
    __shared__ float scratch[kVThreads / 32];
    constexpr int kRChunk = kVThreads * kRPer;
    const int base = c * kRChunk + threadIdx.x * kRPer;
    float rs = 0.f, ps = 0.f;
    if constexpr (P::kStaged) {
        typename P::Raw raw[kRPer];
#pragma unroll
        for (int i = 0; i < kRPer; ++i) {
            const int v = base + i;
            if (v < V) raw[i] = pol.load(v);
        }
        pol.stage();
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kRPer; ++i) {
            const int v = base + i;
            if (v < V) { float r, p; pol.weights(raw[i], r, p); rs += r; ps += p; }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kRPer; ++i) {
            const int v = base + i;
            if (v < V) { float r, p; pol.weights(pol.load(v), r, p); rs += r; ps += p; }
        }
    }
    rs = block_sum(rs, scratch);
    ps = block_sum(ps, scratch);
    if (threadIdx.x == 0) { rsum[c] = rs; psum[c] = ps; }
}

// Pass 2, once every chunk's masses are stored, by the block that ran pass 1 for its own chunk
// (a staged table is still in place): the draw (see icdf_draw).
template <int kRPer, class P>
__device__ void icdf_locate(const P &pol, int V, int nrch, float u, const float *__restrict__ rsum,
                            const float *__restrict__ psum, int32_t *out)
{
    __shared__ float sbuf[kVThreads + 1];
    __shared__ float fscan[33];
    __shared__ int s_chunk, s_use_p, s_hit, s_last;
    __shared__ float s_target;
    constexpr int kRChunk = kVThreads * kRPer;
    // a staged table is still in place: this block staged it for its own chunk (icdf_draw)
    const int E = (nrch + kVThreads - 1) / kVThreads;
    const int c0 = threadIdx.x * E, c1 = min(nrch, c0 + E);
    float rrun = 0.f, prun = 0.f;
    for (int i = c0; i < c1; ++i) { rrun += __ldcg(&rsum[i]); prun += __ldcg(&psum[i]); }
    block_cdf_bounds(rrun, sbuf, fscan);
    const float rtot = sbuf[kVThreads];
    const int use_p = !(rtot > 0.f);
    if (use_p) block_cdf_bounds(prun, sbuf, fscan);
    const float *w = use_p ? psum : rsum;
    const float target = u * sbuf[kVThreads];
    const float lo_b = sbuf[threadIdx.x], hi_b = sbuf[threadIdx.x + 1];
    if (threadIdx.x == 0) { s_hit = 0x7FFFFFFF; s_last = -1; }
    __syncthreads();
    if (lo_b <= target && target < hi_b) atomicMin(&s_hit, threadIdx.x);
    int lastc = -1;
    for (int i = c0; i < c1; ++i) if (__ldcg(&w[i]) > 0.f) lastc = i;
    if (lastc >= 0) atomicMax(&s_last, lastc);
    __syncthreads();
    if (int(threadIdx.x) == s_hit) {               // the first claimant walks its run of chunks
        float cum = lo_b;
        int ch = -1;
        for (int i = c0; i < c1; ++i) {
            const float wi = __ldcg(&w[i]);
            if (cum + wi > target) { ch = i; break; }
            cum += wi;
        }
        if (ch < 0) {                               // rounding inside the run: its last chunk with mass
            for (int i = c1 - 1; i >= c0; --i) if (__ldcg(&w[i]) > 0.f) { ch = i; break; }
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
        if (v < V) pol.weights(pol.load(v), r, p);     // a staged table is still in place
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
        *out = v >= 0 ? v : s_last;
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_hit == 0x7FFFFFFF) *out = s_last;   // target beyond the chunk
    __syncthreads();                                   // the block may call again (shared state)
}

// Both passes in one launch over (chunks, ...): every block stores its chunk's masses, the last
// block of the group draws.
template <int kRPer, class P>
__device__ void icdf_draw(const P &pol, int V, int nrch, float u, float *__restrict__ rsum,
                          float *__restrict__ psum, unsigned *counter, int32_t *out)
{
    icdf_chunk<kRPer>(pol, V, blockIdx.x, rsum, psum);
    if (!last_block_done(counter, unsigned(nrch))) return;
    icdf_locate<kRPer>(pol, V, nrch, u, rsum, psum, out);
}

// The residual weights of row tr of a chain (max(0, p - q), or p for the bonus row); with
// kStage the list's cluster positions are staged in shared memory (dynamic, M ints).
template <bool kStage>
struct ChainResidual {
    static constexpr bool kStaged = kStage;
    const ChainArgs *a;
    ResidualRow rr;
    int *s_cp;
    struct Raw { float z; int c, rk; };
    __device__ Raw load(int v) const
    {
        Raw x;
        x.z = rr.z[v];
        x.c = rr.ql ? a->cluster_of[v] : -1;
        x.rk = rr.ql ? a->rank[v] : 0;
        return x;
    }
    __device__ void stage() const
    {
        if (rr.ql)
            for (int c = threadIdx.x; c < a->M; c += blockDim.x) s_cp[c] = rr.cposb[c];
    }
    __device__ void weights(const Raw &x, float &r, float &p) const
    {
        p = __expf(x.z * a->inv_te - rr.pm) / rr.ps;
        float q = 0.f;
        if (rr.ql && unsigned(x.c) < unsigned(a->M)) {
            const int pc = kStage ? s_cp[x.c] : rr.cposb[x.c];
            if (pc >= 0) q = __expf(rr.ql[pc + x.rk] * a->inv_te - rr.qm) / rr.qs;
        }
        r = fmaxf(p - q, 0.f);
    }
};

template <int kRPer, bool kStage>
__global__ void __launch_bounds__(kVThreads)
verify_residual_kernel(ChainArgs a)
{
    extern __shared__ int s_cp[];                    // M entries when staged
    {
        // the chunk's cluster ids and ranks are fixed inputs: fetch them into L2 while the
        // statistics kernel still runs
        const int v = blockIdx.x * (kVThreads * kRPer) + threadIdx.x * kRPer;
        if (v < a.V && threadIdx.x % (32 / kRPer) == 0) { // one thread per 128-byte line
            prefetch_l2(a.cluster_of + v);
            prefetch_l2(a.rank + v);
        }
    }
    pdl_wait();
    const int b = blockIdx.y;
    const Decision dsn = ldcg(&a.decision[b]);
    if (dsn.tr < 0) return;                          // greedy: decided already (whole group returns)
    const ChainResidual<kStage> pol{&a, residual_row(a, b, dsn), s_cp};
    icdf_draw<kRPer>(pol, a.V, a.nrch, a.u[size_t(b) * (a.gamma + 1) + a.gamma], a.rsum + size_t(b) * a.nrch,
              a.psum + size_t(b) * a.nrch, &a.cnt2[b], &a.correction[b]);
}

// ---------------------------------------------------------------------------------------
// Tree verification.  The pages cite EAGLE-style token trees but state no tree verifier;
// reading: sibling-sequential recursive rejection (the multi-draft form of speculative
// sampling).  All nodes of one depth share their sequence's shortlist, so the residual
// after a rejected sibling differs from the current target only on that shortlist: the walk
// keeps it as (O = target mass off the list, r_j on the list) and never builds a dense row.
//
//   tree_walk_kernel      one cluster of up to 8 CTAs per sequence.  At each visited node one pass
//                         over the target row gives its max, sum-exp, argmax and the mass
//                         off the children's list; r_j = p(S_j) is gathered over the list;
//                         every rejected sibling costs one pass over the list.  Only the
//                         rows on the walked path are read.
//   tree_residual_kernel  grid (chunks, B): the inverse-CDF draw of the correction from the
//                         walk's final state (the residual, or p at a leaf).
// ---------------------------------------------------------------------------------------
constexpr int kWalkThreads = 1024;
constexpr int kWalkMaxM = 8192;
constexpr int kWalkMaxCluster = 8;              // CTAs per sequence (portable cluster size)
constexpr int kWalkU = 6;                       // elements per thread whose loads a pass issues together
// A list of up to kWalkSlots x (CTAs x kWalkThreads) entries keeps the residual in the cluster's
// shared memory (two buffers of kWalkSlots x kWalkThreads floats per CTA): entry j lives in CTA
// (j / kWalkThreads) % CL, slot j / (kWalkThreads * CL), at slot * kWalkThreads + j % kWalkThreads,
// which is the entry a thread's own passes touch.  Longer lists keep it in global memory.
constexpr int kWalkSlots = 16;
constexpr size_t kWalkSmem = size_t(2) * kWalkSlots * kWalkThreads * sizeof(float);

struct WalkState {                 // what the walk leaves for the correction draw
    int mode;                      // 0: decided (greedy); 1: draw from p of `row`; 2: residual
    int row, dep, buf;             // target row (0 = root), list depth, residual buffer
    float m, s;                    // softmax statistics of the target row
    int pad0, pad1;
};

struct TreeArgs {
    const float *p_logits;
    int B, D, Wd, N, V;
    float T, inv_te;
    const int32_t *parent;
    const float *q_logits;
    int64_t q_stride;
    const float *q_max, *q_sumexp;             // optional [D][B*Wd]
    const int32_t *vs_offsets, *vs_ids;
    int64_t vs_stride;
    const int32_t *cpos;
    int M;
    const int32_t *cluster_of, *rank;
    const int32_t *node_tokens;
    const float *u_node, *u_res;
    int32_t *accepted, *correction, *path;
    int32_t *status;
    // workspace
    WalkState *state;                          // [B]
    float *rbuf;                               // [B][2][V]
    int nrch;
    float *rsum, *psum;                        // [B][nrch]
    unsigned *cnt;                             // [B]
};

// Online softmax statistics of x = value * inv_te with the raw argmax (ties to the lower
// index) and the part of the sum-exp over tokens off a list.
struct RowStat { float m, s, o, amax; int aid; };

__device__ __forceinline__ RowStat rowstat_empty() { return RowStat{-INFINITY, 0.f, 0.f, -INFINITY, -1}; }

__device__ __forceinline__ void rowstat_add(RowStat &a, float z, float x, bool off, int v)
{
    if (x > a.m) {
        const float sc = a.m == -INFINITY ? 0.f : __expf(a.m - x);
        a.s = a.s * sc + 1.f;
        a.o = a.o * sc + (off ? 1.f : 0.f);
        a.m = x;
    } else {
        const float e = __expf(x - a.m);
        a.s += e;
        if (off) a.o += e;
    }
    if (z > a.amax || a.aid < 0) { a.amax = z; a.aid = v; }      // v ascending per thread
}

// a (earlier in the fixed order) merged with b, without branches.
__device__ __forceinline__ RowStat rowstat_merge(const RowStat &a, const RowStat &b)
{
    RowStat r;
    r.m = fmaxf(a.m, b.m);
    const float ea = a.m == -INFINITY ? 0.f : __expf(a.m - r.m);
    const float eb = b.m == -INFINITY ? 0.f : __expf(b.m - r.m);
    r.s = fmaf(a.s, ea, b.s * eb);
    r.o = fmaf(a.o, ea, b.o * eb);
    const bool tb = b.aid >= 0 && (a.aid < 0 || b.amax > a.amax || (b.amax == a.amax && b.aid < a.aid));
    r.amax = tb ? b.amax : a.amax;
    r.aid = tb ? b.aid : a.aid;
    return r;
}

__device__ __forceinline__ RowStat shfl_xor_rowstat(const RowStat &a, int o)
{
    return RowStat{__shfl_xor_sync(0xFFFFFFFFu, a.m, o), __shfl_xor_sync(0xFFFFFFFFu, a.s, o),
                   __shfl_xor_sync(0xFFFFFFFFu, a.o, o), __shfl_xor_sync(0xFFFFFFFFu, a.amax, o),
                   __shfl_xor_sync(0xFFFFFFFFu, a.aid, o)};
}

// One butterfly level: both lanes of a pair merge the pair in lane order (the lower lane's
// first), so they hold the same result and the whole tree's order is fixed.
__device__ __forceinline__ RowStat rowstat_butterfly(const RowStat &mine, int lane, int o)
{
    const RowStat other = shfl_xor_rowstat(mine, o);
    const bool hi = (lane & o) != 0;
    const RowStat lo_s{hi ? other.m : mine.m, hi ? other.s : mine.s, hi ? other.o : mine.o,
                       hi ? other.amax : mine.amax, hi ? other.aid : mine.aid};
    const RowStat hi_s{hi ? mine.m : other.m, hi ? mine.s : other.s, hi ? mine.o : other.o,
                       hi ? mine.amax : other.amax, hi ? mine.aid : other.aid};
    return rowstat_merge(lo_s, hi_s);
}

// Cluster-wide reductions, with one CTA barrier and one cluster barrier each.  Every warp
// reduces its lanes (a butterfly, so all lanes hold the same bits); the CTA's first warp
// reduces the warp results the same way and publishes the CTA's result in its shared memory;
// after the cluster barrier every warp of every CTA reads all CTAs' results at once (lane r
// from rank r) and merges them in the same fixed lane tree, so every thread of the cluster
// holds the same bits and takes the same decisions.  Two publication slots alternate: a CTA
// rewrites a slot only after the barrier of the next reduction, which every other CTA reaches
// only once all its warps have read that slot.  The warp results need one buffer: the first
// warp reads them before the cluster barrier, and they are rewritten only after it.
struct ClusterRed {
    RowStat stat[2];
    float sum[2];
    RowStat wstat[32];                           // this CTA's warp results
    float wsum[32];
};

__device__ __forceinline__ RowStat rowstat_tree(RowStat c, int lane, int width)
{
    for (int o = 1; o < width; o <<= 1) c = rowstat_butterfly(c, lane, o);
    return c;
}

__device__ RowStat cluster_rowstat(RowStat st, ClusterRed &cr, int &k)
{
    cg::cluster_group cl = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int slot = k & 1;
    st = rowstat_tree(st, lane, 32);
    if (lane == 0) cr.wstat[warp] = st;
    __syncthreads();
    if (warp == 0) {
        const RowStat c = rowstat_tree(lane < nw ? cr.wstat[lane] : rowstat_empty(), lane, 32);
        if (lane == 0) cr.stat[slot] = c;
    }
    cl.sync();
    const int nb = int(cl.num_blocks());
    RowStat m = lane < nb ? cl.map_shared_rank(&cr, lane)->stat[slot] : rowstat_empty();
    m = rowstat_tree(m, lane, 32);
    ++k;
    return m;
}

__device__ float cluster_sum(float x, ClusterRed &cr, int &k)
{
    cg::cluster_group cl = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int slot = k & 1;
    x = warp_sum(x);
    if (lane == 0) cr.wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const float c = warp_sum(lane < nw ? cr.wsum[lane] : 0.f);
        if (lane == 0) cr.sum[slot] = c;
    }
    cl.sync();
    const int nb = int(cl.num_blocks());
    float t = lane < nb ? cl.map_shared_rank(&cr, lane)->sum[slot] : 0.f;
    ++k;
    return warp_sum(t);
}

// One thread-block cluster per sequence (grid = B clusters of CL CTAs): every pass over the
// target row or the list is split over all CL * 1024 threads of the cluster.
__global__ void __launch_bounds__(kWalkThreads)
tree_walk_kernel(TreeArgs a)
{
    __shared__ int s_cpos[kWalkMaxM];           // cpos of the children's list
    extern __shared__ float s_rbuf[];            // [2][kWalkSlots * kWalkThreads]: the residual
    __shared__ ClusterRed s_cr;
    __shared__ int s_kids[64];
    __shared__ int s_nkids;
    __shared__ int s_cj[64];                     // per child: list index of its token (-1: none)
    __shared__ float s_cu[64], s_cq[64], s_cqm[64], s_cqs[64];   // its uniform, q(x), q's max / sum-exp
    cg::cluster_group cl = cg::this_cluster();
    const int CL = int(cl.num_blocks()), crank = int(cl.block_rank());
    const int b = blockIdx.x / CL;
    const int tid = threadIdx.x;
    const int gt = crank * blockDim.x + tid, GT = CL * blockDim.x;
    const bool lead = crank == 0 && tid == 0;
    int nred = 0;
    if (crank == 0 && tid < a.D) a.path[size_t(b) * a.D + tid] = -1;
    int cur = -1, dep = 0, A = 0, corr = -1;
    WalkState ws{0, 0, 0, 0, 0.f, 1.f, 0, 0};
    int cb = 0;                                  // which residual buffer holds r
    for (int guard = 0; guard <= a.D; ++guard) {
        const int rr = cur + 1;
        const float *z = a.p_logits + (size_t(b) * (1 + a.N) + rr) * a.V;
        const bool has_list = dep < a.D;
        if (tid == 0) {
            int nk = 0;
            if (has_list)
                for (int i = 0; i < a.Wd; ++i) {
                    const int n = dep * a.Wd + i;
                    if (a.parent[n] == cur) s_kids[nk++] = n;
                }
            s_nkids = nk;
        }
        if (has_list) {
            const int32_t *cp = a.cpos + (size_t(dep) * a.B + b) * a.M;
            for (int c = tid; c < a.M; c += blockDim.x) s_cpos[c] = cp[c];
        }
        __syncthreads();
        const int nk = s_nkids;
        // one pass over the target row (kWalkU elements' loads issued together, then folded in
        // ascending v)
        RowStat st = rowstat_empty();
        for (int v0 = gt; v0 < a.V; v0 += kWalkU * GT) {
            float zv[kWalkU];
            int cv[kWalkU];
#pragma unroll
            for (int e = 0; e < kWalkU; ++e) {
                const int v = v0 + e * GT;
                zv[e] = v < a.V ? z[v] : 0.f;
                cv[e] = v < a.V ? a.cluster_of[v] : -1;
            }
#pragma unroll
            for (int e = 0; e < kWalkU; ++e) {
                const int v = v0 + e * GT;
                if (v < a.V) {
                    const int c = cv[e];
                    const bool off = has_list && (unsigned(c) >= unsigned(a.M) || s_cpos[c] < 0);
                    rowstat_add(st, zv[e], zv[e] * a.inv_te, off, v);
                }
            }
        }
        const RowStat row = cluster_rowstat(st, s_cr, nred);
        if (a.T == 0.f) {
            const int am = row.aid;
            int next = -1;
            for (int k = 0; k < nk; ++k) {
                const int n = s_kids[k];
                if (a.node_tokens[size_t(dep) * a.B * a.Wd + size_t(b) * a.Wd + (n - dep * a.Wd)] == am) { next = n; break; }
            }
            if (next < 0) { corr = am; ws.mode = 0; break; }
            if (lead) a.path[size_t(b) * a.D + A] = next;
            ++A; cur = next; ++dep;
            continue;
        }
        ws.row = rr; ws.dep = dep; ws.m = row.m; ws.s = row.s;
        if (nk == 0) { ws.mode = 1; break; }
        // the children's list and r_j = p(S_j) on it
        const int *off = a.vs_offsets + size_t(dep) * (a.B + 1);
        const int lo = off[b];
        int nb = off[b + 1] - lo;
        if (lo < 0 || nb < 0 || nb > a.V) { if (tid == 0) set_status(a.status, DS_DEV_BAD_INDEX); nb = 0; }
        const int32_t *ids = a.vs_ids + size_t(dep) * a.vs_stride + lo;
        // where r lives: the cluster's shared memory when the list fits, else the global buffers
        const bool in_smem = nb <= kWalkSlots * GT;
        auto rbase = [&](int buf) -> float * {
            return in_smem ? s_rbuf + size_t(buf) * kWalkSlots * kWalkThreads : a.rbuf + (size_t(b) * 2 + buf) * a.V;
        };
        // this thread's element j = j0 + e * GT (j0 = gt + it * kWalkU * GT) at index ri of a buffer
        auto rindex = [&](int j, int slot) { return in_smem ? slot * kWalkThreads + tid : j; };
        // r[j] of any entry, after a cluster barrier that followed its write
        auto rread = [&](int buf, int j) -> float {
            if (!in_smem) return __ldcg(rbase(buf) + j);
            const int blk = j / kWalkThreads;
            const float *own = cl.map_shared_rank(rbase(buf), blk % CL);
            return own[(blk / CL) * kWalkThreads + (j - blk * kWalkThreads)];
        };
        cb = 0;
        float *r = rbase(cb);
        float on = 0.f;
        for (int j0 = gt, it = 0; j0 < nb; j0 += kWalkU * GT, ++it) {
            int vv[kWalkU];
            float zv[kWalkU];
#pragma unroll
            for (int e = 0; e < kWalkU; ++e) vv[e] = j0 + e * GT < nb ? ids[j0 + e * GT] : -1;
#pragma unroll
            for (int e = 0; e < kWalkU; ++e) zv[e] = (vv[e] >= 0 && vv[e] < a.V) ? z[vv[e]] : 0.f;
#pragma unroll
            for (int e = 0; e < kWalkU; ++e) {
                const int j = j0 + e * GT;
                if (j < nb) {
                    const float pj = (vv[e] >= 0 && vv[e] < a.V) ? __expf(zv[e] * a.inv_te - row.m) / row.s : 0.f;
                    r[rindex(j, it * kWalkU + e)] = pj;
                    on += pj;
                }
            }
        }
        // r is read across the cluster only after the next cluster barrier (cluster_sum's), whose
        // arrive/wait pair has release/acquire semantics at cluster scope: no fence needed here
        // every child's test inputs at once (one thread per child): the index j of its token
        // in the list, the uniform, and -- when the head's row statistics are given -- q(x)
        // and the statistics the rejection pass needs
        if (tid < nk) {
            const int n = s_kids[tid];
            const int i = n - dep * a.Wd, hr = b * a.Wd + i;
            const int x = a.node_tokens[size_t(dep) * a.B * a.Wd + hr];
            int j = -1;
            if (x >= 0 && x < a.V) {
                const int c = a.cluster_of[x];
                const int pc = unsigned(c) < unsigned(a.M) ? s_cpos[c] : -1;
                if (pc >= 0) j = pc + a.rank[x];
            }
            if (j >= nb) j = -1;
            s_cj[tid] = j;
            s_cu[tid] = a.u_node[size_t(b) * a.N + n];
            if (a.q_max) {
                const float qm = a.q_max[size_t(dep) * a.B * a.Wd + hr];
                const float qs = a.q_sumexp[size_t(dep) * a.B * a.Wd + hr];
                const float *ql = a.q_logits + size_t(dep) * a.q_stride + int64_t(lo) * a.Wd + int64_t(i) * nb;
                s_cqm[tid] = qm;
                s_cqs[tid] = qs;
                s_cq[tid] = j >= 0 ? __expf(ql[j] * a.inv_te - qm) / qs : 0.f;
            }
        }
        // the children's draft rows on this thread's entries, into L2 for the rejection passes
        if ((tid & 31) == 0)
            for (int k = 0; k < nk; ++k) {
                const float *ql = a.q_logits + size_t(dep) * a.q_stride + int64_t(lo) * a.Wd +
                                  int64_t(s_kids[k] - dep * a.Wd) * nb;
                for (int j = gt; j < nb; j += GT) prefetch_l2(ql + j);
            }
        const float O = row.o / row.s;
        float R = O + cluster_sum(on, s_cr, nred);   // (its barriers also publish s_c*)
        int next = -1;
        for (int k = 0; k < nk; ++k) {
            const int n = s_kids[k];
            const int i = n - dep * a.Wd;
            const float *ql = a.q_logits + size_t(dep) * a.q_stride + int64_t(lo) * a.Wd + int64_t(i) * nb;
            float qm, qs;
            if (a.q_max) {
                qm = s_cqm[k];
                qs = s_cqs[k];
            } else {
                RowStat q = rowstat_empty();
                for (int j = gt; j < nb; j += GT) rowstat_add(q, ql[j], ql[j] * a.inv_te, false, j);
                q = cluster_rowstat(q, s_cr, nred);
                qm = q.m; qs = q.s;
            }
            // every thread takes the same test on the same data
            int acc = 0;
            {
                const int j = s_cj[k];
                if (j < 0) {
                    if (tid == 0) set_status(a.status, DS_DEV_BAD_INDEX);
                } else {
                    const float q = a.q_max ? s_cq[k] : __expf(ql[j] * a.inv_te - qm) / qs;
                    acc = s_cu[k] * q < rread(cb, j) / R;
                }
            }
            if (acc) { next = n; break; }
            // rejected: r <- max(r - R q, 0) into the other buffer, kept if it has mass
            float *rn = rbase(cb ^ 1);
            float part = 0.f;
            for (int j0 = gt, it = 0; j0 < nb; j0 += kWalkU * GT, ++it) {
                float rv[kWalkU], lv[kWalkU];
#pragma unroll
                for (int e = 0; e < kWalkU; ++e) {
                    const int j = j0 + e * GT;
                    rv[e] = j < nb ? (in_smem ? r[rindex(j, it * kWalkU + e)] : __ldcg(r + j)) : 0.f;
                    lv[e] = j < nb ? ql[j] : 0.f;
                }
#pragma unroll
                for (int e = 0; e < kWalkU; ++e) {
                    const int j = j0 + e * GT;
                    if (j < nb) {
                        const float w = fmaxf(rv[e] - R * (__expf(lv[e] * a.inv_te - qm) / qs), 0.f);
                        rn[rindex(j, it * kWalkU + e)] = w;
                        part += w;
                    }
                }
            }
            const float Rn = O + cluster_sum(part, s_cr, nred);
            if (Rn > 0.f) { cb ^= 1; r = rn; R = Rn; }
        }
        if (next < 0 && in_smem) {
            // the correction draw reads the residual from the global buffer
            float *g = a.rbuf + size_t(b) * 2 * a.V;
            for (int j0 = gt, it = 0; j0 < nb; j0 += kWalkU * GT, ++it)
#pragma unroll
                for (int e = 0; e < kWalkU; ++e) {
                    const int j = j0 + e * GT;
                    if (j < nb) g[j] = r[rindex(j, it * kWalkU + e)];
                }
            cb = 0;
        }
        if (next >= 0) {
            if (lead) a.path[size_t(b) * a.D + A] = next;
            ++A; cur = next; ++dep;
            continue;
        }
        ws.mode = 2; ws.buf = cb;
        break;
    }
    if (lead) {
        a.accepted[b] = A;
        if (ws.mode == 0) a.correction[b] = corr;
        a.state[b] = ws;
    }
    cl.sync();                                   // no CTA leaves while others may read its slots
}

// The weights of the tree's correction draw: the walk's residual r (on the list; p off it), or
// p of the final row; the list's cluster positions staged in shared memory (dynamic, M ints).
struct TreeResidual {
    static constexpr bool kStaged = true;
    const TreeArgs *a;
    const float *z, *r;
    const int32_t *cp;
    float m, s;
    bool resid;
    int *s_cp;
    struct Raw { float z; int c, rk; };
    __device__ Raw load(int v) const
    {
        Raw x;
        x.z = z[v];
        x.c = resid ? a->cluster_of[v] : -1;
        x.rk = resid ? a->rank[v] : 0;
        return x;
    }
    __device__ void stage() const
    {
        if (resid)
            for (int c = threadIdx.x; c < a->M; c += blockDim.x) s_cp[c] = cp[c];
    }
    __device__ void weights(const Raw &x, float &w, float &p) const
    {
        p = __expf(x.z * a->inv_te - m) / s;
        w = p;
        if (resid) {
            const int pc = unsigned(x.c) < unsigned(a->M) ? s_cp[x.c] : -1;
            if (pc >= 0) { const int j = pc + x.rk; w = unsigned(j) < unsigned(a->V) ? r[j] : 0.f; }
        }
    }
};

template <int kRPer>
__global__ void __launch_bounds__(kVThreads)
tree_residual_kernel(TreeArgs a)
{
    const int b = blockIdx.y;
    const WalkState ws = a.state[b];              // written by the previous launch
    if (ws.mode == 0) return;                     // whole group returns
    extern __shared__ int s_cp[];                 // M entries
    TreeResidual pol;
    pol.a = &a;
    pol.z = a.p_logits + (size_t(b) * (1 + a.N) + ws.row) * a.V;
    pol.r = a.rbuf + (size_t(b) * 2 + ws.buf) * a.V;
    pol.cp = a.cpos + (size_t(ws.dep) * a.B + b) * a.M;
    pol.m = ws.m;
    pol.s = ws.s;
    pol.resid = ws.mode == 2;
    pol.s_cp = s_cp;
    icdf_draw<kRPer>(pol, a.V, a.nrch, a.u_res[size_t(b) * (a.D + 1) + ws.dep], a.rsum + size_t(b) * a.nrch,
              a.psum + size_t(b) * a.nrch, &a.cnt[b], &a.correction[b]);
}

}  // namespace
}  // namespace ds

using namespace ds;

static int vchunks(int V) { return (V + kVChunkMin - 1) / kVChunkMin; }     // the most chunks
static size_t rchunks(int V) { return size_t((V + kRChunkMin - 1) / kRChunkMin); }

// The larger chunks when rows * chunks still covers every SM twice.
static bool big_chunks(long long rows, int V, int chunk, int sms)
{
    return rows * ((V + chunk - 1) / chunk) >= 2LL * sms;
}

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
           align256(size_t(B) * sizeof(Decision)) +
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
    ds::NvtxRange range("ds_verify");
    if (!p_logits || !q_logits || !vs_offsets || !cpos || !cluster_of || !rank_in_cluster ||
        !draft_ids || !uniforms || !accepted_len || !correction)
        return DS_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > kMaxGamma || V < 1 || V > (1 << 24) || M < 1 || M > 8192 ||
        !(T >= 0.f) || q_stride < 0)
        return DS_ERR_INVALID_ARG;
    if ((q_max == nullptr) != (q_sumexp == nullptr)) return DS_ERR_INVALID_ARG;
    if (B > 65535 / (gamma + 1)) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_verify_workspace_bytes(B, gamma, V)) return DS_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    ChainArgs a;
    const bool vbig = big_chunks(1LL * B * (gamma + 1), V, kVThreads * kVPerBig, sms);
    const bool rbig = big_chunks(B, V, kVThreads * kRPerBig, sms);
    a.p_logits = p_logits; a.B = B; a.gamma = gamma; a.V = V;
    a.nch = (V + kVThreads * (vbig ? kVPerBig : kVPerSmall) - 1) / (kVThreads * (vbig ? kVPerBig : kVPerSmall));
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
    a.decision = reinterpret_cast<Decision *>(w); w += align256(size_t(B) * sizeof(Decision));
    a.nrch = (V + kVThreads * (rbig ? kRPerBig : kRPerSmall) - 1) / (kVThreads * (rbig ? kRPerBig : kRPerSmall));
    a.rsum = reinterpret_cast<float *>(w); w += align256(size_t(B) * rchunks(V) * sizeof(float));
    a.psum = reinterpret_cast<float *>(w);

    // both launches may start before the kernel ahead of them ends (their blocks wait for it)
    const dim3 sgrid(a.nch, B * (gamma + 1));
    cudaError_t e = vbig ? launch_pdl(verify_stats_kernel<kVPerBig>, sgrid, dim3(kVThreads), 0, stream, a)
                         : launch_pdl(verify_stats_kernel<kVPerSmall>, sgrid, dim3(kVThreads), 0, stream, a);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return DS_ERR_CUDA; }
    // the small-chunk grid (few sequences) stages the list's cluster positions in shared memory
    const size_t cp_smem = size_t(M) * sizeof(int);   // M <= 8192
    const dim3 rgrid(a.nrch, B);
    e = rbig ? launch_pdl(verify_residual_kernel<kRPerBig, false>, rgrid, dim3(kVThreads), 0, stream, a)
             : launch_pdl(verify_residual_kernel<kRPerSmall, true>, rgrid, dim3(kVThreads), cp_smem, stream, a);
    if (e != cudaSuccess) { (void)cudaGetLastError(); return DS_ERR_CUDA; }
    return DS_OK;
}

extern "C" size_t ds_verify_tree_workspace_bytes(int B, int D, int Wd, int V)
{
    if (B <= 0 || D <= 0 || Wd <= 0 || V <= 0) return 0;
    return align256(size_t(B) * sizeof(WalkState)) +
           align256(size_t(B) * 2 * size_t(V) * sizeof(float)) +
           2 * align256(size_t(B) * rchunks(V) * sizeof(float)) +
           align256(size_t(B) * sizeof(unsigned));
}

extern "C" ds_status ds_verify_tree(const float *p_logits, int B, int D, int Wd, int V, float T,
                                    const int32_t *parent,
                                    const float *q_logits, int64_t q_stride,
                                    const float *q_max, const float *q_sumexp,
                                    const int32_t *vs_offsets, const int32_t *vs_ids, int64_t vs_stride,
                                    const int32_t *cpos, int M,
                                    const int32_t *cluster_of, const int32_t *rank_in_cluster,
                                    const int32_t *node_tokens, const float *u_node, const float *u_res,
                                    int32_t *accepted_len, int32_t *correction, int32_t *path,
                                    void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_verify_tree");
    if (!p_logits || !parent || !q_logits || !vs_offsets || !vs_ids || !cpos || !cluster_of ||
        !rank_in_cluster || !node_tokens || !u_node || !u_res || !accepted_len || !correction || !path)
        return DS_ERR_INVALID_ARG;
    if (B < 1 || D < 1 || D > kMaxGamma || Wd < 1 || Wd > 64 || V < 1 || V > (1 << 24) || M < 1 ||
        M > kWalkMaxM || !(T >= 0.f) || q_stride < 0 || vs_stride < 0)
        return DS_ERR_INVALID_ARG;
    if ((q_max == nullptr) != (q_sumexp == nullptr)) return DS_ERR_INVALID_ARG;
    if (B > 65535) return DS_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ds_verify_tree_workspace_bytes(B, D, Wd, V)) return DS_ERR_WORKSPACE;
    TreeArgs a;
    a.p_logits = p_logits; a.B = B; a.D = D; a.Wd = Wd; a.N = D * Wd; a.V = V;
    a.T = T; a.inv_te = T > 0.f ? 1.f / T : 1.f;
    a.parent = parent; a.q_logits = q_logits; a.q_stride = q_stride;
    a.q_max = q_max; a.q_sumexp = q_sumexp;
    a.vs_offsets = vs_offsets; a.vs_ids = vs_ids; a.vs_stride = vs_stride;
    a.cpos = cpos; a.M = M;
    a.cluster_of = cluster_of; a.rank = rank_in_cluster;
    a.node_tokens = node_tokens; a.u_node = u_node; a.u_res = u_res;
    a.accepted = accepted_len; a.correction = correction; a.path = path; a.status = dev_status;
    char *w = static_cast<char *>(ws);
    a.state = reinterpret_cast<WalkState *>(w); w += align256(size_t(B) * sizeof(WalkState));
    a.rbuf = reinterpret_cast<float *>(w); w += align256(size_t(B) * 2 * size_t(V) * sizeof(float));
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    const bool rbig = big_chunks(B, V, kVThreads * kRPerBig, sms);
    a.nrch = (V + kVThreads * (rbig ? kRPerBig : kRPerSmall) - 1) / (kVThreads * (rbig ? kRPerBig : kRPerSmall));
    a.rsum = reinterpret_cast<float *>(w); w += align256(size_t(B) * rchunks(V) * sizeof(float));
    a.psum = reinterpret_cast<float *>(w); w += align256(size_t(B) * rchunks(V) * sizeof(float));
    a.cnt = reinterpret_cast<unsigned *>(w);
    // one cluster of CL CTAs per sequence, CL = 8, 4, 2 or 1 so that the clusters fit the GPU
    int CL = kWalkMaxCluster;
    while (CL > 1 && long(B) * CL > sms) CL >>= 1;
    static std::atomic<unsigned long long> walk_smem_set{0};
    if (!smem_limit_once(tree_walk_kernel, kWalkSmem, walk_smem_set)) return DS_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B * CL));
    cfg.blockDim = dim3(kWalkThreads);
    cfg.dynamicSmemBytes = kWalkSmem;             // the residual, when the list fits
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tree_walk_kernel, a) != cudaSuccess) { (void)cudaGetLastError(); return DS_ERR_CUDA; }
    const size_t cp_smem = size_t(M) * sizeof(int);   // the list's cluster positions (M <= 8192)
    if (rbig) tree_residual_kernel<kRPerBig><<<dim3(a.nrch, B), kVThreads, cp_smem, stream>>>(a);
    else tree_residual_kernel<kRPerSmall><<<dim3(a.nrch, B), kVThreads, cp_smem, stream>>>(a);
    DS_TRY_LAUNCH();
    return DS_OK;
}
