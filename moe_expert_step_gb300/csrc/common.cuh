// Shared device helpers of the moestep library: types, reductions, error word.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moestep.h"

namespace moestep {

using bf16 = __nv_bfloat16;

// Bits of the device error word (kept in the workspace header).
enum : int {
    kErrTimeoutProducer = 1 << 0,
    kErrTimeoutMma = 1 << 1,
    kErrTimeoutEpilogue = 1 << 2,
    kErrBadInput = 1 << 8,
};

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// (value, index) maximum; equal values keep the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
    }
}

// Programmatic dependent launch.  Every kernel of the library is launched so
// that the next kernel in the stream may start early; each kernel first lets
// its own dependents start (trigger), then waits until every preceding kernel
// has completed and its writes are visible (wait) before touching memory.
// Because every kernel waits, completion stays transitive along the stream.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void record_error(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

// Flags between kernels that run concurrently under programmatic dependent launch.
__device__ __forceinline__ uint64_t gtimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int acquire_load_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void release_store_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait until *p >= v (acquire): false if limit_ns passed first.
__device__ __forceinline__ bool wait_at_least(const int* p, int v, uint64_t limit_ns) {
    if (acquire_load_gpu(p) >= v) return true;
    const uint64_t t0 = gtimer_ns();
    for (;;) {
        __nanosleep(64);
        if (acquire_load_gpu(p) >= v) return true;
        if (gtimer_ns() - t0 >= limit_ns) return false;
    }
}

// Merge of softmax partials (m = max logit, a = its lowest index, s = sum exp(l - m)).
struct SoftmaxPartial {
    float m;
    int a;
    float s;
};
__device__ __forceinline__ SoftmaxPartial merge_partial(SoftmaxPartial x, SoftmaxPartial y) {
    if (y.m == -INFINITY) return x;
    if (x.m == -INFINITY) return y;
    SoftmaxPartial r;
    if (y.m > x.m || (y.m == x.m && y.a < x.a)) {
        r.m = y.m;
        r.a = y.a;
    } else {
        r.m = x.m;
        r.a = x.a;
    }
    r.s = x.s * __expf(x.m - r.m) + y.s * __expf(y.m - r.m);
    return r;
}

}  // namespace moestep
