// Drafter stand-in: the work of one EAGLE-style drafter step, so that the router's overlap with
// the drafter (DynaSpec summary, Pipeline Flow and Novel Architectural Elements: the router runs
// on its own stream beside the drafter's computation) can be measured on a real schedule.  The
// drafter trunk itself is not part of the DynaSpec path and has no trained weights here; this
// kernel chain has the shape and the weight bytes of one such step at batch 1:
//
//   u  = [h_prev ; E[x_prev]]                        previous hidden state and token embedding
//   y1 = Wfc u                     Wfc  [d, 2d]       EAGLE's fusion layer
//   y2 = Wmix y1                   Wmix [d, d]        stands in for the attention projections
//   a_j = silu(Wug[j] y2) * (Wug[F + j] y2)          gated MLP, Wug [2F, d]
//   h_out = bf16(h_base + scale * (Wdn a))            Wdn [d, F]
//
// (at d = 4096, F = 14336: 453 MB of weights per step).  h_out depends on x_prev and h_prev
// through the whole chain, so a step cannot start before the previous token is drawn; with
// scale = 0 it equals h_base bit for bit, which lets a measured step keep the workload's hidden
// states.  GEMV-shaped and HBM-bound: a warp per weight row, 16-byte streaming loads, fp32
// accumulation, the input vector read through L2.
#include "common.cuh"

namespace ds {
namespace {

constexpr int kDsWarps = 8;
constexpr int kDsU = 16;                 // 16-byte loads in flight per lane (4096 columns)
constexpr int kDsSideSms = 8;            // SMs left to the side stream (the router)

__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

// u = [f32(h_prev) ; f32(E[x])]; x out of range sets DS_DEV_BAD_INDEX and reads row 0.
__global__ void standin_gather(const uint16_t *__restrict__ h_prev, const int32_t *__restrict__ x_prev,
                               int V, const uint16_t *__restrict__ E, int d, float *__restrict__ u,
                               int32_t *st)
{
    int x = *x_prev;
    if (x < 0 || x >= V) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_status(st, DS_DEV_BAD_INDEX);
        x = 0;
    }
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < 2 * d; k += gridDim.x * blockDim.x)
        u[k] = k < d ? bf16_to_f32(h_prev[k]) : bf16_to_f32(E[size_t(x) * d + (k - d)]);
}

// Dot product of weight row `row` (K bf16, 16-byte aligned) with fp32 x, summed over the warp.
__device__ __forceinline__ float row_dot(const uint16_t *__restrict__ row, const float *__restrict__ x, int K,
                                         int lane)
{
    const uint4 *r = reinterpret_cast<const uint4 *>(row);
    float acc = 0.f;
    for (int k0 = 0; k0 < K; k0 += kDsU * 256) {
        uint4 w[kDsU];
#pragma unroll
        for (int u = 0; u < kDsU; ++u) {
            const int k = k0 + (u * 32 + lane) * 8;
            w[u] = k < K ? ld_stream(r + (k >> 3)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kDsU; ++u) {
            const int k = k0 + (u * 32 + lane) * 8;
            if (k < K) {
                const float4 x0 = *reinterpret_cast<const float4 *>(x + k);
                const float4 x1 = *reinterpret_cast<const float4 *>(x + k + 4);
                acc = dot8(w[u], x0, x1, acc);
            }
        }
    }
    return warp_sum(acc);
}

// MODE 0: y[i] = A[i] . x.  MODE 1: y[j] = silu(A[j] . x) * (A[N + j] . x).  MODE 2: out[i] =
// bf16(base[i] + scale * (A[i] . x)).  Warps stride over the N outputs.
template <int MODE>
__global__ void __launch_bounds__(kDsWarps * 32)
standin_gemv(const uint16_t *__restrict__ A, int N, int K, const float *__restrict__ x,
             float *__restrict__ y, const uint16_t *__restrict__ base, float scale, uint16_t *__restrict__ out)
{
    const int lane = threadIdx.x & 31;
    for (int i = blockIdx.x * kDsWarps + (threadIdx.x >> 5); i < N; i += gridDim.x * kDsWarps) {
        const float s = row_dot(A + size_t(i) * K, x, K, lane);
        if (MODE == 1) {
            const float g = row_dot(A + size_t(N + i) * K, x, K, lane);
            if (lane == 0) y[i] = silu(s) * g;
        } else if (MODE == 2) {
            if (lane == 0) out[i] = f32_to_bf16_rne(bf16_to_f32(base[i]) + scale * s);
        } else {
            if (lane == 0) y[i] = s;
        }
    }
}

}  // namespace
}  // namespace ds

using namespace ds;

extern "C" size_t ds_drafter_standin_workspace_bytes(int d, int F)
{
    if (d <= 0 || F <= 0) return 0;
    return align256(size_t(2) * d * sizeof(float)) + 2 * align256(size_t(d) * sizeof(float)) +
           align256(size_t(F) * sizeof(float));
}

extern "C" ds_status ds_drafter_standin(const uint16_t *h_prev, const int32_t *x_prev, int V,
                                        const uint16_t *E, const uint16_t *Wfc, const uint16_t *Wmix,
                                        const uint16_t *Wug, const uint16_t *Wdn, int d, int F,
                                        const uint16_t *h_base, float scale, uint16_t *h_out,
                                        void *ws, size_t ws_bytes, int32_t *dev_status, cudaStream_t stream)
{
    ds::NvtxRange range("ds_drafter_standin");
    if (!h_prev || !x_prev || !E || !Wfc || !Wmix || !Wug || !Wdn || !h_base || !h_out) return DS_ERR_INVALID_ARG;
    if (V < 1 || d < 8 || d % 8 || F < 8 || F % 8 || !(scale == scale)) return DS_ERR_INVALID_ARG;
    if (!aligned16(Wfc) || !aligned16(Wmix) || !aligned16(Wug) || !aligned16(Wdn)) return DS_ERR_INVALID_ARG;
    if (!ws || ws_bytes < ds_drafter_standin_workspace_bytes(d, F)) return DS_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return DS_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    float *u = reinterpret_cast<float *>(w);
    w += align256(size_t(2) * d * sizeof(float));
    float *y1 = reinterpret_cast<float *>(w);
    w += align256(size_t(d) * sizeof(float));
    float *y2 = reinterpret_cast<float *>(w);
    w += align256(size_t(d) * sizeof(float));
    float *a = reinterpret_cast<float *>(w);
    int grid = sms - kDsSideSms;
    if (grid < 1) grid = 1;
    standin_gather<<<8, 256, 0, stream>>>(h_prev, x_prev, V, E, d, u, dev_status);
    DS_TRY_LAUNCH();
    standin_gemv<0><<<grid, kDsWarps * 32, 0, stream>>>(Wfc, d, 2 * d, u, y1, nullptr, 0.f, nullptr);
    DS_TRY_LAUNCH();
    standin_gemv<0><<<grid, kDsWarps * 32, 0, stream>>>(Wmix, d, d, y1, y2, nullptr, 0.f, nullptr);
    DS_TRY_LAUNCH();
    standin_gemv<1><<<grid, kDsWarps * 32, 0, stream>>>(Wug, F, d, y2, a, nullptr, 0.f, nullptr);
    DS_TRY_LAUNCH();
    standin_gemv<2><<<grid, kDsWarps * 32, 0, stream>>>(Wdn, d, F, a, nullptr, h_base, scale, h_out);
    DS_TRY_LAUNCH();
    return DS_OK;
}
