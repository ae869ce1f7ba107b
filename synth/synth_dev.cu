// Seeded synthetic inputs, device side.
//
// Input generation only: the same SplitMix64 stream and Irwin-Hall(4)
// transform as synth_host.c, so a tensor filled here is bit-identical to the
// host copy of the same (key, index range).  Used to create tens of GB of
// weights directly in HBM without a host round trip.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float irwin_hall4(uint64_t u, float scale) {
    int s = (int)(u & 0xFFFF) + (int)((u >> 16) & 0xFFFF) + (int)((u >> 32) & 0xFFFF) + (int)(u >> 48);
    return __fmul_rn((float)(s - 131070), scale);
}

template <typename T>
__device__ __forceinline__ T convert(float f);
template <>
__device__ __forceinline__ float convert<float>(float f) { return f; }
template <>
__device__ __forceinline__ __nv_bfloat16 convert<__nv_bfloat16>(float f) { return __float2bfloat16_rn(f); }

// float -> FP8 E4M3, nearest-even, saturated to +-448 (the host copy's definition)
__device__ __forceinline__ uint8_t f32_to_e4m3_rne(float f) {
    const uint32_t b = __float_as_uint(f);
    const uint32_t sign = (b >> 31) << 7;
    const uint32_t a = b & 0x7FFFFFFFu;
    uint32_t code;
    if (a >= 0x7F800000u) {
        code = 0x7Eu;
    } else if (a >= 0x3C800000u) {
        const uint32_t r = (a + 0x7FFFFu + ((a >> 20) & 1u)) >> 20;
        code = r - (120u << 3);
        if (code > 0x7Eu) code = 0x7Eu;
    } else {
        code = (uint32_t)rintf(__fmul_rn(__uint_as_float(a), 512.0f));
    }
    return (uint8_t)(code | sign);
}
template <>
__device__ __forceinline__ uint8_t convert<uint8_t>(float f) { return f32_to_e4m3_rne(f); }

__global__ void fill_row_scales(uint64_t key, uint64_t start, int64_t n, float* __restrict__ out) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (; i < n; i += stride)
        out[i] = (float)(16 + (int)(sm64_mix(key + (start + (uint64_t)i + 1) * kGamma) & 15u)) * 0x1p-16f;
}

template <typename T>
__global__ void fill_normal(uint64_t key, uint64_t start, int64_t n, float scale, T* __restrict__ out) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (; i < n; i += stride) {
        uint64_t u = sm64_mix(key + (start + (uint64_t)i + 1) * kGamma);
        out[i] = convert<T>(irwin_hall4(u, scale));
    }
}

__global__ void fill_u64(uint64_t key, uint64_t start, int64_t n, uint64_t* __restrict__ out) {
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (; i < n; i += stride) out[i] = sm64_mix(key + (start + (uint64_t)i + 1) * kGamma);
}

int grid_for(int64_t n) {
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (n + 255) / 256;
    int64_t cap = (int64_t)sms * 8;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" {

// Fill out[0..n) with elements start..start+n-1 of the stream `key`.
// dtype 0 = bf16, 1 = fp32, 2 = FP8 E4M3 codes.  Returns a cudaError_t value (0 = success).
int synth_dev_fill_normal(uint64_t key, uint64_t start, int64_t n, float scale, int dtype, void* out,
                          cudaStream_t stream) {
    if (n <= 0) return 0;
    if (out == nullptr) return (int)cudaErrorInvalidValue;
    if (dtype == 0)
        fill_normal<__nv_bfloat16><<<grid_for(n), 256, 0, stream>>>(key, start, n, scale, (__nv_bfloat16*)out);
    else if (dtype == 1)
        fill_normal<float><<<grid_for(n), 256, 0, stream>>>(key, start, n, scale, (float*)out);
    else if (dtype == 2)
        fill_normal<uint8_t><<<grid_for(n), 256, 0, stream>>>(key, start, n, scale, (uint8_t*)out);
    else
        return (int)cudaErrorInvalidValue;
    return (int)cudaGetLastError();
}

// Per-row scales (16 + (u & 15)) * 2^-16 of elements start..start+n-1 of `key`.
int synth_dev_fill_row_scales(uint64_t key, uint64_t start, int64_t n, void* out, cudaStream_t stream) {
    if (n <= 0) return 0;
    if (out == nullptr) return (int)cudaErrorInvalidValue;
    fill_row_scales<<<grid_for(n), 256, 0, stream>>>(key, start, n, (float*)out);
    return (int)cudaGetLastError();
}

int synth_dev_fill_u64(uint64_t key, uint64_t start, int64_t n, void* out, cudaStream_t stream) {
    if (n <= 0) return 0;
    if (out == nullptr) return (int)cudaErrorInvalidValue;
    fill_u64<<<grid_for(n), 256, 0, stream>>>(key, start, n, (uint64_t*)out);
    return (int)cudaGetLastError();
}

}  // extern "C"
