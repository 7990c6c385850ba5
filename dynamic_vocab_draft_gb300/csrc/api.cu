// Library-wide entry points: status text, ABI version, and the device Philox4x32-10 exposed
// for checking on its own.
#include "common.cuh"

namespace {

__global__ void philox_kernel(const uint4 *__restrict__ ctr, uint64_t seed, uint4 *__restrict__ out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = ds::philox4x32_10(ctr[i], uint32_t(seed), uint32_t(seed >> 32));
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

extern "C" int ds_version(void) { return 1; }

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
