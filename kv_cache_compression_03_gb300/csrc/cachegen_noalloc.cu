// cg_encode_noalloc: cg_encode without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they need to encode: a
// serving engine that has already reserved nearly all of the GPU for its KV
// cache pool has nothing left for cudaMalloc, and a latency-critical path
// cannot afford cudaMalloc/cudaFree, which may synchronise the whole device.
// For them the encoder's scratch (status word, tile totals and bases, the
// symbol rows and the stream slots) lives in one fixed array in this file,
// which every GPU that loads the library keeps for the life of the process.

#include <cuda_runtime.h>
#include <stdint.h>

#include "cg_internal.h"

namespace {

// The shared scratch. Its size is CG_NOALLOC_SCRATCH_BYTES (cachegen.h).
static __device__ __align__(256) uint8_t g_noalloc_scratch[CG_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch in the current device's context. In host
// code the array's name is only a host-side stand-in, so the address is
// asked for on every call, with the caller's device current: nothing is
// cached, so a context that was torn down and created again (a device
// reset) can never leave a stale address behind. The first call in a
// context also loads this file's device code there.
cudaError_t scratch_address(void **out)
{
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess)
        return err;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" cg_status cg_encode_noalloc(const cg_plan *p, const void *kv, const cg_encoded *out,
                                       void *status_out, cg_stream_t stream)
{
    if (p == nullptr || kv == nullptr || out == nullptr || status_out == nullptr)
        return CG_ERR_INVALID_ARG;
    if (!out->bytestream || !out->lengths || !out->cdf || !out->amax)
        return CG_ERR_INVALID_ARG;
    if (p->ws_bytes > (size_t)CG_NOALLOC_SCRATCH_BYTES)
        return CG_ERR_UNSUPPORTED;  // the plan needs more scratch than the static array holds
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return CG_ERR_CUDA;
    // cg_encode's checks (alignment etc.), with the static array as the workspace;
    // the launch sequence clears the status block itself.
    cg_status st = cg_encode(p, kv, scratch, (size_t)CG_NOALLOC_SCRATCH_BYTES, out, stream);
    if (st != CG_OK)
        return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(status_out, scratch, 16, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return CG_ERR_CUDA;
    return CG_OK;
}
