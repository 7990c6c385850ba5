// Library-wide entry points: status text, ABI version, and the device Philox4x32-10 exposed
// for checking on its own.
#include "common.cuh"

namespace {

__global__ void philox_kernel(const uint4 *__restrict__ ctr, uint64_t seed, uint4 *__restrict__ out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = ds::philox4x32_10(ctr[i], uint32_t(seed), uint32_t(seed >> 32));
}

// SM-driven copy: 16-byte vectors when both ends allow them, bytes otherwise.
__global__ void copy16_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, size_t n)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

__global__ void copy1_kernel(unsigned char *__restrict__ dst, const unsigned char *__restrict__ src, size_t n)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

constexpr int kCopyThreads = 256;
constexpr size_t kCopyMaxBlocks = 1024;

// The address a kernel on the current device uses for `p`, or nullptr when the device cannot
// reach it: device and managed memory as they are; page-locked host memory through the device
// alias the runtime reports (with unified addressing the same value); pageable or foreign host
// memory is refused, since a kernel reading it would fault on systems without address
// translation services.
void *device_alias(const void *p)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        return const_cast<void *>(p);
    case cudaMemoryTypeHost:
        return at.devicePointer;
    default:
        return nullptr;
    }
}

}  // namespace

extern "C" const char *ds_status_string(ds_status s)
{
    switch (s) {
    case DS_OK: return "ok";
    case DS_ERR_INVALID_ARG: return "invalid argument";
    case DS_ERR_UNSUPPORTED: return "unsupported size";
    case DS_ERR_CUDA: return "CUDA launch or runtime error";
    case DS_ERR_WORKSPACE: return "workspace missing or too small";
    default: break;
    }
    if (s & DS_DEV_BAD_INDEX) return "device: id out of range or token not in its shortlist";
    if (s & DS_DEV_CAPACITY) return "device: shortlist larger than the capacity given";
    if (s & DS_DEV_TIMEOUT) return "device: bounded wait gave up";
    return "unknown status";
}

extern "C" int ds_version(void) { return 4; }

extern "C" size_t ds_workspace_bytes(int op, int B, int V, int M, int gamma, int hidden, int width)
{
    switch (op) {
    case DS_OP_ROUTER: return ds_router_workspace_bytes(B, hidden);
    case DS_OP_SHORTLIST: return ds_shortlist_workspace_bytes(B, M);
    case DS_OP_HEAD:
        if (B <= 0 || width <= 0 || 1LL * B * width > 0x7FFFFFFFLL) return 0;
        return ds_head_workspace_bytes(B * width);
    case DS_OP_VERIFY: return ds_verify_workspace_bytes(B, gamma, V);
    case DS_OP_VERIFY_TREE: return ds_verify_tree_workspace_bytes(B, gamma, width, V);
    default: return 0;
    }
}

extern "C" ds_status ds_set_wait_budget(int64_t cycles)
{
    if (cycles < 0) return DS_ERR_INVALID_ARG;
    ds::wait_budget_cell().store(cycles == 0 ? ds::kWaitBudgetCycles : (long long)cycles,
                                 std::memory_order_relaxed);
    return DS_OK;
}

extern "C" ds_status ds_philox4x32_10(const uint32_t *ctr, uint64_t seed, uint32_t *out, int n,
                                      cudaStream_t stream)
{
    if (!ctr || !out || n < 0) return DS_ERR_INVALID_ARG;
    if (!ds::aligned16(ctr) || !ds::aligned16(out)) return DS_ERR_INVALID_ARG;
    if (n == 0) return DS_OK;
    philox_kernel<<<(n + 255) / 256, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(ctr), seed,
                                                       reinterpret_cast<uint4 *>(out), n);
    DS_TRY_LAUNCH();
    return DS_OK;
}

extern "C" ds_status ds_event_record(cudaEvent_t event, cudaStream_t stream)
{
    if (!event) return DS_ERR_INVALID_ARG;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DS_ERR_CUDA;
    const cudaError_t e = cs == cudaStreamCaptureStatusActive
                              ? cudaEventRecordWithFlags(event, stream, cudaEventRecordExternal)
                              : cudaEventRecord(event, stream);
    return e == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

extern "C" ds_status ds_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream)
{
    ds::NvtxRange range("ds_copy");
    if (bytes == 0) return DS_OK;
    if (!dst || !src) return DS_ERR_INVALID_ARG;
    const char *d0 = static_cast<const char *>(dst), *s0 = static_cast<const char *>(src);
    if (d0 < s0 + bytes && s0 < d0 + bytes) return DS_ERR_INVALID_ARG;     // overlapping ranges
    // both ends must be memory the device can reach (checked before anything is launched)
    dst = device_alias(dst);
    src = device_alias(src);
    if (!dst || !src) return DS_ERR_INVALID_ARG;
    if (ds::aligned16(dst) && ds::aligned16(src) && bytes % 16 == 0) {
        const size_t n = bytes / 16;
        const size_t blocks = (n + kCopyThreads - 1) / kCopyThreads;
        copy16_kernel<<<unsigned(blocks < kCopyMaxBlocks ? blocks : kCopyMaxBlocks), kCopyThreads, 0, stream>>>(
            static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n);
    } else {
        const size_t blocks = (bytes + kCopyThreads - 1) / kCopyThreads;
        copy1_kernel<<<unsigned(blocks < kCopyMaxBlocks ? blocks : kCopyMaxBlocks), kCopyThreads, 0, stream>>>(
            static_cast<unsigned char *>(dst), static_cast<const unsigned char *>(src), bytes);
    }
    DS_TRY_LAUNCH();
    return DS_OK;
}
