// Combine of the expert outputs into the residual stream and the RMSNorm that
// feeds the next router (shared by the combine kernel and the single-block
// router launch, so both compute bit-identical rows).
#pragma once
#include "common.cuh"

namespace moestep {

constexpr float kRmsEps = 1e-6f;

// Sum over a group of 256 threads (threads 256g .. 256g+255 of the block); every
// thread of the block calls it.  `red` is the group's scratch of 9 floats.
__device__ __forceinline__ float group_sum_256(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, gt = threadIdx.x & 255, warp = gt >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (gt < 8) ? red[gt] : 0.f;
    if (warp == 0) t = warp_sum(t);
    if (gt == 0) red[8] = t;
    __syncthreads();
    return red[8];
}

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void store4<bf16>(bf16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
template <typename T>
__device__ __forceinline__ float4 roundtrip4(float4 v) {
    return v;
}
template <>
__device__ __forceinline__ float4 roundtrip4<bf16>(float4 v) {
    return make_float4(__bfloat162float(__float2bfloat16_rn(v.x)), __bfloat162float(__float2bfloat16_rn(v.y)),
                       __bfloat162float(__float2bfloat16_rn(v.z)), __bfloat162float(__float2bfloat16_rn(v.w)));
}

// Optional extra consumer of the normalised row: called as sink(c, n) for each group
// of four columns c .. c+3 (n: the fp32 values that were rounded into x).
struct NoSink {
    __device__ __forceinline__ void operator()(int, float4) const {}
};

// One token per group of 256 threads (t < 0: the group only joins the barriers;
// every thread of the block calls it).  MODE 0: out = sum_j gate_rr*y[slot_j] +
// y[shared slot].  MODE 1: h += that; x = RMSNorm(h).  MODE 2: h = h_in; x =
// RMSNorm(h).  The routed terms are added in candidate order j = 0..k-1, then the
// shared one.  s_slot / s_g (33 each) and red (9) are the group's scratch.
// The token's slots and gates read into the group's scratch (MODE != 2); combine_row
// does this itself unless its caller already did (slots_loaded).
__device__ __forceinline__ void combine_load_slots(int t, int k, const int32_t* __restrict__ slot_of,
                                                   const int32_t* __restrict__ slot_sh,
                                                   const float* __restrict__ gate_rr, int has_shared, int* s_slot,
                                                   float* s_g) {
    const int gt = threadIdx.x & 255;
    if (t >= 0 && gt < k) {
        s_slot[gt] = __ldcg(&slot_of[t * k + gt]);
        s_g[gt] = __ldcg(&gate_rr[t * k + gt]);
    }
    if (t >= 0 && gt == 32) s_slot[32] = has_shared ? __ldcg(&slot_sh[t]) : -1;
}

template <typename T, int MODE, typename Sink = NoSink>
__device__ void combine_row(int t, int H, int k, const float* __restrict__ y, const int32_t* __restrict__ slot_of,
                            const int32_t* __restrict__ slot_sh, const float* __restrict__ gate_rr, int has_shared,
                            const float* __restrict__ h_in, float* __restrict__ h, T* __restrict__ x,
                            float* __restrict__ x_f32, float* __restrict__ out, int* s_slot, float* s_g, float* red,
                            Sink sink = Sink(), bool slots_loaded = false) {
    const int gt = threadIdx.x & 255;
    const bool on = t >= 0;
    if (MODE != 2 && !slots_loaded) {
        if (on && gt < k) {
            s_slot[gt] = slot_of[t * k + gt];
            s_g[gt] = gate_rr[t * k + gt];
        }
        if (on && gt == 32) s_slot[32] = has_shared ? slot_sh[t] : -1;
        __syncthreads();
    }
    float ss = 0.f;
    const size_t row = static_cast<size_t>(on ? t : 0) * H;
    constexpr int kKeep = 4;  // float4 columns per thread kept in registers (H <= 4096)
    float4 hv[kKeep];
    int i = 0;
    for (int c = gt * 4; on && c < H; c += 1024, ++i) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (MODE != 2) {
            // the shared expert's row is loaded with the first group of routed rows (all in
            // flight together); routed rows in groups of 8, added in candidate order, then the
            // shared one
            const int ssl = s_slot[32];
            const float4 vs = ssl >= 0 ? __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(ssl) * H + c))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < k; j0 += 8) {
                float4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int sl = (j0 + q < k) ? s_slot[j0 + q] : -1;
                    v[q] = sl >= 0 ? __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(sl) * H + c))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (j0 + q < k && s_slot[j0 + q] >= 0) {
                        const float g = s_g[j0 + q];
                        acc.x += g * v[q].x;
                        acc.y += g * v[q].y;
                        acc.z += g * v[q].z;
                        acc.w += g * v[q].w;
                    }
                }
            }
            if (ssl >= 0) {
                acc.x += vs.x;
                acc.y += vs.y;
                acc.z += vs.z;
                acc.w += vs.w;
            }
        }
        if (MODE == 0) {
            *reinterpret_cast<float4*>(out + row + c) = acc;
        } else {
            const float4 base = *reinterpret_cast<const float4*>((MODE == 1 ? h : h_in) + row + c);
            const float4 v = make_float4(base.x + acc.x, base.y + acc.y, base.z + acc.z, base.w + acc.w);
            *reinterpret_cast<float4*>(h + row + c) = v;
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
            for (int q = 0; q < kKeep; ++q)
                if (q == i) hv[q] = v;
        }
    }
    if (MODE == 0) return;
    const float tot = group_sum_256(ss, red);
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(H) + kRmsEps);
    i = 0;
    for (int c = gt * 4; on && c < H; c += 1024, ++i) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < kKeep) {
#pragma unroll
            for (int q = 0; q < kKeep; ++q)
                if (q == i) v = hv[q];
        } else {
            v = *reinterpret_cast<const float4*>(h + row + c);
        }
        const float4 n = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        store4<T>(x + row + c, n);
        sink(c, n);
        if (x_f32 != nullptr) *reinterpret_cast<float4*>(x_f32 + row + c) = roundtrip4<T>(n);
    }
}

// combine_row (MODE 1 or 2) for one token by all 512 threads of the block, H <= 2048:
// thread gt + 256 takes the second 1024-column pass of thread gt, so every load of the
// row is in flight at once.  Each column's arithmetic is combine_row's, and the sum of
// squares is added in its order (thread gt's first-pass terms, then the second pass's,
// then the same 256-thread tree), so the row is bit-identical.  s_slot / s_g / red are
// one group's scratch, shared by both halves; pair holds 256 floats.
template <typename T, int MODE, typename Sink = NoSink>
__device__ void combine_row_pair(int t, int H, int k, const float* __restrict__ y, const int32_t* __restrict__ slot_of,
                                 const int32_t* __restrict__ slot_sh, const float* __restrict__ gate_rr,
                                 int has_shared, const float* __restrict__ h_in, float* __restrict__ h,
                                 T* __restrict__ x, int* s_slot, float* s_g, float* red, float* pair, Sink sink,
                                 bool slots_loaded) {
    static_assert(MODE == 1 || MODE == 2, "residual modes only");
    const int gt = threadIdx.x & 511;
    const bool on = t >= 0;
    if (MODE != 2 && !slots_loaded) {
        if (on && gt < k) {
            s_slot[gt] = slot_of[t * k + gt];
            s_g[gt] = gate_rr[t * k + gt];
        }
        if (on && gt == 32) s_slot[32] = has_shared ? slot_sh[t] : -1;
        __syncthreads();
    }
    const size_t row = static_cast<size_t>(on ? t : 0) * H;
    const int c = (gt & 255) * 4 + 1024 * (gt >> 8);
    const bool mine = on && c < H;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    float ss = 0.f;
    if (mine) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (MODE != 2) {
            const int ssl = s_slot[32];
            const float4 vs = ssl >= 0 ? __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(ssl) * H + c))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j0 = 0; j0 < k; j0 += 8) {
                float4 w[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int sl = (j0 + q < k) ? s_slot[j0 + q] : -1;
                    w[q] = sl >= 0 ? __ldg(reinterpret_cast<const float4*>(y + static_cast<size_t>(sl) * H + c))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (j0 + q < k && s_slot[j0 + q] >= 0) {
                        const float g = s_g[j0 + q];
                        acc.x += g * w[q].x;
                        acc.y += g * w[q].y;
                        acc.z += g * w[q].z;
                        acc.w += g * w[q].w;
                    }
                }
            }
            if (ssl >= 0) {
                acc.x += vs.x;
                acc.y += vs.y;
                acc.z += vs.z;
                acc.w += vs.w;
            }
        }
        const float4 base = *reinterpret_cast<const float4*>((MODE == 1 ? h : h_in) + row + c);
        v = make_float4(base.x + acc.x, base.y + acc.y, base.z + acc.z, base.w + acc.w);
        *reinterpret_cast<float4*>(h + row + c) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (gt >= 256) pair[gt - 256] = ss;
    __syncthreads();
    if (gt < 256) ss += pair[gt];
    // the 256-thread tree of group_sum_256 over threads 0..255 (warps 8..15 take part in
    // the shuffles only; their sums are not read)
    ss = warp_sum(ss);
    const int lane = threadIdx.x & 31, warp = gt >> 5;
    if (lane == 0 && warp < 8) red[warp] = ss;
    __syncthreads();
    float tt = (gt < 8) ? red[gt] : 0.f;
    if (warp == 0) tt = warp_sum(tt);
    if (gt == 0) red[8] = tt;
    __syncthreads();
    const float tot = red[8];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(H) + kRmsEps);
    if (mine) {
        const float4 n = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        store4<T>(x + row + c, n);
        sink(c, n);
    }
}

}  // namespace moestep
