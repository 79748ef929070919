// Int8 baseline codec: each (K/V, layer, token) row of C bf16 values becomes
// C signed bytes and one fp32 scale. The CacheGen reproduction page
// ("CacheGen复现项目：面向大模型服务的高效KV缓存压缩与流式传输方案",
// §编解码器模块) quantises KV to 8-bit integers with scale factors; the
// formula is the symmetric scaling of "LMCache 中的 KV Cache 压缩：CacheGen
// 编解码原理、配置方式与源码解析" §2 with MAX = 127 and no offset:
//   a = max_c |x_c|, f = 127 / a (0 when a = 0), q = round_half_even(fp32(x * f)),
//   y = bf16_rne(fp32(fp32(q / 127) * a)).
//
// Both kernels are pure streams (2 bytes in, 1 out per value, or the
// reverse), so they are bound by HBM: one warp owns a row, holds it in
// registers (VPL 16-byte vectors per lane), reduces the amax with one
// redux, and writes the row back; a grid of resident blocks strides over
// the rows.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "cg_internal.h"

namespace {

constexpr int kThreads = 256;  // 8 rows in flight per block
constexpr int kMaxDevices = 64;

// SM count of each device, looked up once.
std::mutex g_sms_mutex;
int g_sms[kMaxDevices] = {0};

__device__ __forceinline__ int q8(float x, float f)
{
    return __float2int_rn(__fmul_rn(x, f));
}

// Four bf16 values (two words, low half first) to four signed bytes.
__device__ __forceinline__ uint32_t quantise4(uint32_t w0, uint32_t w1, float f)
{
    const int a = q8(__uint_as_float(w0 << 16), f);
    const int b = q8(__uint_as_float(w0 & 0xFFFF0000u), f);
    const int c = q8(__uint_as_float(w1 << 16), f);
    const int d = q8(__uint_as_float(w1 & 0xFFFF0000u), f);
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

template <int VPL>
__global__ void __launch_bounds__(kThreads)
    k_int8_encode(const uint4 *__restrict__ kv, int64_t rows, int32_t chunks,
                  uint2 *__restrict__ q, float *__restrict__ scales, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const uint4 *src = kv + r * chunks;
        uint4 x[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            x[i] = (j < chunks) ? __ldcs(src + j) : make_uint4(0, 0, 0, 0);
        }
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            m = __vmaxu2(m, x[i].x & 0x7FFF7FFFu);
            m = __vmaxu2(m, x[i].y & 0x7FFF7FFFu);
            m = __vmaxu2(m, x[i].z & 0x7FFF7FFFu);
            m = __vmaxu2(m, x[i].w & 0x7FFF7FFFu);
        }
        m = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        const float a = __uint_as_float(m << 16);
        float f = (m == 0) ? 0.0f : __fdiv_rn(127.0f, a);
        // inf/NaN in the row, or a so small that 127 / a overflows: report
        // it and quantise with f = 0 (NaN converts to 0).
        if (m >= 0x7F80u || isinf(f)) {
            f = 0.0f;
            if (lane == 0)
                *status = CG_ERR_NONFINITE;
        }
        if (lane == 0)
            scales[r] = a;
        uint2 *dst = q + r * chunks;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            if (j < chunks)
                __stcs(dst + j, make_uint2(quantise4(x[i].x, x[i].y, f),
                                           quantise4(x[i].z, x[i].w, f)));
        }
    }
}

// Two bytes of w (selected by shift) to a bf16 pair, low byte first.
__device__ __forceinline__ uint32_t dequant2(const float *tab, uint32_t w, int shift, float a)
{
    const float y0 = __fmul_rn(tab[(w >> shift) & 0xFFu], a);
    const float y1 = __fmul_rn(tab[(w >> (shift + 8)) & 0xFFu], a);
    const __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int VPL>
__global__ void __launch_bounds__(kThreads)
    k_int8_decode(const uint2 *__restrict__ q, const float *__restrict__ scales, int64_t rows,
                  int32_t chunks, uint4 *__restrict__ kv)
{
    // tab[b] = fp32(v / 127) for the byte b holding v = (int8)b; b = 0x80
    // (-128) never comes out of the encoder and decodes like any other byte.
    __shared__ float tab[256];
    tab[threadIdx.x] = __fdiv_rn((float)(int8_t)(uint8_t)threadIdx.x, 127.0f);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const uint2 *src = q + r * chunks;
        const float a = __ldcs(scales + r);
        uint2 x[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            x[i] = (j < chunks) ? __ldcs(src + j) : make_uint2(0, 0);
        }
        uint4 *dst = kv + r * chunks;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int j = lane + 32 * i;
            if (j < chunks)
                __stcs(dst + j, make_uint4(dequant2(tab, x[i].x, 0, a), dequant2(tab, x[i].x, 16, a),
                                           dequant2(tab, x[i].y, 0, a), dequant2(tab, x[i].y, 16, a)));
        }
    }
}

// Smallest vectors-per-lane instantiation that covers chunks = C / 8.
int vpl_for(int32_t chunks)
{
    const int need = (chunks + 31) / 32;
    return need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : need <= 8 ? 8 : 16;
}

template <typename K>
cudaError_t grid_for(K kernel, int64_t rows, int *grid)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_sms_mutex);
        if (g_sms[dev] == 0) {
            err = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev);
            if (err != cudaSuccess)
                return err;
        }
        sms = g_sms[dev];
    }
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (err != cudaSuccess)
        return err;
    const int64_t want = (rows + kThreads / 32 - 1) / (kThreads / 32);
    const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    *grid = (int)(want < resident ? want : resident);
    return cudaSuccess;
}

cg_status check_shape(int64_t rows, int32_t channels)
{
    if (rows < 0 || channels <= 0 || channels % 8 != 0)
        return CG_ERR_INVALID_ARG;
    if (channels > CG_MAX_CHANNELS)
        return CG_ERR_UNSUPPORTED;
    return CG_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

template <int VPL>
cudaError_t launch_encode(const void *kv, int64_t rows, int32_t chunks, void *q, float *scales,
                          uint32_t *status, cudaStream_t s)
{
    int grid = 0;
    cudaError_t err = grid_for(k_int8_encode<VPL>, rows, &grid);
    if (err != cudaSuccess)
        return err;
    k_int8_encode<VPL><<<grid, kThreads, 0, s>>>(static_cast<const uint4 *>(kv), rows, chunks,
                                                  static_cast<uint2 *>(q), scales, status);
    return cudaGetLastError();
}

template <int VPL>
cudaError_t launch_decode(const void *q, const float *scales, int64_t rows, int32_t chunks,
                          void *kv, cudaStream_t s)
{
    int grid = 0;
    cudaError_t err = grid_for(k_int8_decode<VPL>, rows, &grid);
    if (err != cudaSuccess)
        return err;
    k_int8_decode<VPL><<<grid, kThreads, 0, s>>>(static_cast<const uint2 *>(q), scales, rows,
                                                  chunks, static_cast<uint4 *>(kv));
    return cudaGetLastError();
}

}  // namespace

extern "C" cg_status cg_int8_encode(const void *kv, int64_t rows, int32_t channels, void *q_out,
                                    float *scales_out, void *status_out, cg_stream_t stream)
{
    cg_status st = check_shape(rows, channels);
    if (st != CG_OK)
        return st;
    if (status_out == nullptr || !aligned(status_out, 16))
        return CG_ERR_INVALID_ARG;
    if (rows > 0 && (kv == nullptr || q_out == nullptr || scales_out == nullptr ||
                     !aligned(kv, 16) || !aligned(q_out, 8) || !aligned(scales_out, 4)))
        return CG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status_out, 0, 16, s) != cudaSuccess)
        return CG_ERR_CUDA;
    if (rows == 0)
        return CG_OK;
    const int32_t chunks = channels / 8;
    uint32_t *status = static_cast<uint32_t *>(status_out);
    cudaError_t err;
    switch (vpl_for(chunks)) {
    case 1: err = launch_encode<1>(kv, rows, chunks, q_out, scales_out, status, s); break;
    case 2: err = launch_encode<2>(kv, rows, chunks, q_out, scales_out, status, s); break;
    case 4: err = launch_encode<4>(kv, rows, chunks, q_out, scales_out, status, s); break;
    case 8: err = launch_encode<8>(kv, rows, chunks, q_out, scales_out, status, s); break;
    default: err = launch_encode<16>(kv, rows, chunks, q_out, scales_out, status, s); break;
    }
    return err == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}

extern "C" cg_status cg_int8_decode(const void *q, const float *scales, int64_t rows,
                                    int32_t channels, void *kv_out, cg_stream_t stream)
{
    cg_status st = check_shape(rows, channels);
    if (st != CG_OK)
        return st;
    if (rows == 0)
        return CG_OK;
    if (q == nullptr || scales == nullptr || kv_out == nullptr || !aligned(q, 8) ||
        !aligned(scales, 4) || !aligned(kv_out, 16))
        return CG_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int32_t chunks = channels / 8;
    cudaError_t err;
    switch (vpl_for(chunks)) {
    case 1: err = launch_decode<1>(q, scales, rows, chunks, kv_out, s); break;
    case 2: err = launch_decode<2>(q, scales, rows, chunks, kv_out, s); break;
    case 4: err = launch_decode<4>(q, scales, rows, chunks, kv_out, s); break;
    case 8: err = launch_decode<8>(q, scales, rows, chunks, kv_out, s); break;
    default: err = launch_decode<16>(q, scales, rows, chunks, kv_out, s); break;
    }
    return err == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}
