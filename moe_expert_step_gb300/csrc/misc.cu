// Combine + residual + RMSNorm, block embedding, the fp32 FFMA path (router
// aside) for fp32 weights, softmax partials of given logits, and the
// LowConfidence commit.
#include "combine.cuh"
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace moestep {
namespace {

// One CTA (256 threads) per token: see combine_row.
template <typename T, int MODE>
__global__ void __launch_bounds__(256) combine_kernel(int H, int k, const float* __restrict__ y,
                                                      const int32_t* __restrict__ slot_of,
                                                      const int32_t* __restrict__ slot_sh,
                                                      const float* __restrict__ gate_rr, int has_shared,
                                                      const float* __restrict__ h_in, float* __restrict__ h,
                                                      T* __restrict__ x, float* __restrict__ x_f32,
                                                      float* __restrict__ out) {
    __shared__ int s_slot[33];
    __shared__ float s_g[33];
    __shared__ float red[9];
    pdl_trigger();
    pdl_wait();
    combine_row<T, MODE>(blockIdx.x, H, k, y, slot_of, slot_sh, gate_rr, has_shared, h_in, h, x, x_f32, out, s_slot,
                         s_g, red);
}

template <typename T>
__global__ void __launch_bounds__(256) embed_kernel(int H, int P, int V, const int32_t* __restrict__ tokens,
                                                    const uint8_t* __restrict__ masked, const T* __restrict__ emb,
                                                    const T* __restrict__ pos, int mask_id, float* __restrict__ h) {
    const int t = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    const int id = masked[t] ? mask_id : tokens[t];
    if (id < 0 || id >= V) {
        for (int c = threadIdx.x; c < H; c += blockDim.x) h[static_cast<size_t>(t) * H + c] = __int_as_float(0x7fc00000);
        return;
    }
    const T* er = emb + static_cast<size_t>(id) * H;
    const T* pr = pos + static_cast<size_t>(t % P) * H;
    for (int c = threadIdx.x; c < H; c += blockDim.x) h[static_cast<size_t>(t) * H + c] = to_f32(er[c]) + to_f32(pr[c]);
}

// ------------------------------------------------------------------ fp32 FFMA path
__device__ __forceinline__ float dot_f32(const float* __restrict__ a, const float* __restrict__ b, int n) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int i = 0; i < n; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(a + i);
        const float4 w = *reinterpret_cast<const float4*>(b + i);
        s0 = fmaf(x.x, w.x, s0);
        s1 = fmaf(x.y, w.y, s1);
        s2 = fmaf(x.z, w.z, s2);
        s3 = fmaf(x.w, w.w, s3);
    }
    return (s0 + s1) + (s2 + s3);
}

__global__ void __launch_bounds__(256) f32_gateup_kernel(int H, int E, int I, int Is, int Imax, int max_slots,
                                                         const float* __restrict__ xp, const int32_t* __restrict__ slot_exp,
                                                         const int* __restrict__ plan, const float* __restrict__ Wgu,
                                                         const float* __restrict__ Wsgu, float* __restrict__ act,
                                                         int act_ld) {
    pdl_trigger();
    pdl_wait();
    const int n_slots = plan[2];
    const long long total = static_cast<long long>(max_slots) * Imax;
    for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int slot = static_cast<int>(g / Imax);
        const int i = static_cast<int>(g - static_cast<long long>(slot) * Imax);
        if (slot >= n_slots) break;
        const int e = slot_exp[slot];
        const float* grow;
        if (e == E) {
            if (i >= Is) continue;
            grow = Wsgu + static_cast<size_t>(2 * i) * H;
        } else {
            if (i >= I) continue;
            grow = Wgu + (static_cast<size_t>(e) * 2 * I + 2 * i) * H;
        }
        const float* xr = xp + static_cast<size_t>(slot) * H;
        const float gv = dot_f32(grow, xr, H);
        const float uv = dot_f32(grow + H, xr, H);
        act[static_cast<size_t>(slot) * act_ld + i] = gv / (1.0f + expf(-gv)) * uv;
    }
}

__global__ void __launch_bounds__(256) f32_down_kernel(int H, int E, int I, int Is, int max_slots,
                                                       const float* __restrict__ act, int act_ld,
                                                       const int32_t* __restrict__ slot_exp, const int* __restrict__ plan,
                                                       const float* __restrict__ Wd, const float* __restrict__ Wsd,
                                                       float* __restrict__ y) {
    pdl_trigger();
    pdl_wait();
    const int n_slots = plan[2];
    const long long total = static_cast<long long>(max_slots) * H;
    for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int slot = static_cast<int>(g / H);
        const int hh = static_cast<int>(g - static_cast<long long>(slot) * H);
        if (slot >= n_slots) break;
        const int e = slot_exp[slot];
        const float* ar = act + static_cast<size_t>(slot) * act_ld;
        float v;
        if (e == E)
            v = dot_f32(Wsd + static_cast<size_t>(hh) * Is, ar, Is);
        else
            v = dot_f32(Wd + (static_cast<size_t>(e) * H + hh) * I, ar, I);
        y[static_cast<size_t>(slot) * H + hh] = v;
    }
}

__global__ void __launch_bounds__(256) f32_lm_logits_kernel(int T, int H, int V, const float* __restrict__ hidden,
                                                            const float* __restrict__ Wlm, float scale,
                                                            float* __restrict__ logits) {
    pdl_trigger();
    pdl_wait();
    const long long total = static_cast<long long>(T) * V;
    for (long long g = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(g / V);
        const int v = static_cast<int>(g - static_cast<long long>(p) * V);
        logits[g] = scale * dot_f32(Wlm + static_cast<size_t>(v) * H, hidden + static_cast<size_t>(p) * H, H);
    }
}

// ------------------------------------------------------------------ softmax partials of given logits
// grid (ceil(V / kLogitTile), T), 256 threads: (max, lowest argmax, sum exp(l - max)) of one tile.
__global__ void __launch_bounds__(256) partials_kernel(const float* __restrict__ logits, int T, int V,
                                                       float* __restrict__ pmax, int* __restrict__ parg,
                                                       float* __restrict__ psum) {
    __shared__ float sm[8];
    __shared__ int sa[8];
    __shared__ float red[9];
    const int tile = blockIdx.x, p = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const float* row = logits + static_cast<size_t>(p) * V;
    const int v0 = tile * kLogitTile;
    const int v1 = min(V, v0 + kLogitTile);
    float m = -INFINITY;
    int a = 0x7fffffff;
    for (int v = v0 + threadIdx.x; v < v1; v += 256) {
        const float l = row[v];
        if (l > m || a == 0x7fffffff) {
            m = l;
            a = v;
        }
    }
    warp_argmax(m, a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sm[warp] = m;
        sa[warp] = a;
    }
    __syncthreads();
    float M = sm[0];
    int Aidx = sa[0];
    for (int w = 1; w < 8; ++w)
        if (sm[w] > M || (sm[w] == M && sa[w] < Aidx)) {
            M = sm[w];
            Aidx = sa[w];
        }
    float s = 0.f;
    for (int v = v0 + threadIdx.x; v < v1; v += 256) s += __expf(row[v] - M);
    s = group_sum_256(s, red);
    if (threadIdx.x == 0) {
        const size_t o = static_cast<size_t>(tile) * T + p;
        pmax[o] = M;
        parg[o] = Aidx;
        psum[o] = s;
    }
}

// ------------------------------------------------------------------ LowConfidence commit
// grid = T (one CTA of 256 threads per position).  Each CTA merges its
// position's partials (fixed order: per thread by tile, then a fixed tree) into
// conf = 1 / sum exp(l - max) and choice = lowest argmax and writes them out.
// The last CTA of each request (atomic counter, reset by that CTA) then commits:
// every masked position with conf >= threshold, or, if there is none, the
// masked position with the highest conf (lowest position on ties).
__global__ void __launch_bounds__(256) commit_kernel(int P, int T, int n_tiles, const float* __restrict__ pmax,
                                                     const int* __restrict__ parg, const float* __restrict__ psum,
                                                     float thr, int32_t* __restrict__ tokens,
                                                     uint8_t* __restrict__ masked, int32_t* __restrict__ choice,
                                                     float* __restrict__ conf, uint8_t* __restrict__ accept,
                                                     int32_t* __restrict__ n_committed, int* __restrict__ counters) {
    __shared__ SoftmaxPartial wred[8];
    __shared__ int s_last;
    const int pos = blockIdx.x;
    const int r = pos / P;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    SoftmaxPartial acc{-INFINITY, 0x7fffffff, 0.f};
    int tl = threadIdx.x;
    for (; tl + 3 * 256 < n_tiles; tl += 4 * 256) {
        SoftmaxPartial q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t o = static_cast<size_t>(tl + u * 256) * T + pos;
            q[u] = SoftmaxPartial{pmax[o], parg[o], psum[o]};
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) acc = merge_partial(acc, q[u]);
    }
    for (; tl < n_tiles; tl += 256) {
        const size_t o = static_cast<size_t>(tl) * T + pos;
        acc = merge_partial(acc, SoftmaxPartial{pmax[o], parg[o], psum[o]});
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        SoftmaxPartial o;
        o.m = __shfl_xor_sync(0xffffffffu, acc.m, off);
        o.a = __shfl_xor_sync(0xffffffffu, acc.a, off);
        o.s = __shfl_xor_sync(0xffffffffu, acc.s, off);
        acc = merge_partial(acc, o);
    }
    if (lane == 0) wred[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        SoftmaxPartial b = wred[0];
        for (int w = 1; w < 8; ++w) b = merge_partial(b, wred[w]);
        conf[pos] = b.s > 0.f ? 1.0f / b.s : 0.f;
        choice[pos] = b.a;
        __threadfence();
        const int prev = atomicAdd(&counters[r], 1);
        s_last = (prev == P - 1);
        if (s_last) counters[r] = 0;
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    __threadfence();
    int any = 0;
    for (int pp = lane; pp < P; pp += 32)
        if (masked[r * P + pp] && __ldcg(&conf[r * P + pp]) >= thr) any = 1;
    any = __any_sync(0xffffffffu, any);
    int count = 0;
    if (any) {
        for (int pp = lane; pp < P; pp += 32) {
            const int q = r * P + pp;
            const bool ok = masked[q] && __ldcg(&conf[q]) >= thr;
            if (ok) {
                tokens[q] = __ldcg(&choice[q]);
                masked[q] = 0;
                ++count;
            }
            accept[q] = ok ? 1 : 0;
        }
    } else {
        float bv = -INFINITY;
        int bp = 0x7fffffff;
        for (int pp = lane; pp < P; pp += 32) {
            const float c = __ldcg(&conf[r * P + pp]);
            if (masked[r * P + pp] && (c > bv || bp == 0x7fffffff)) {
                bv = c;
                bp = pp;
            }
        }
        warp_argmax(bv, bp);
        for (int pp = lane; pp < P; pp += 32) {
            const int q = r * P + pp;
            const bool ok = (pp == bp);
            if (ok) {
                tokens[q] = __ldcg(&choice[q]);
                masked[q] = 0;
                ++count;
            }
            accept[q] = ok ? 1 : 0;
        }
    }
    count = __reduce_add_sync(0xffffffffu, count);
    if (lane == 0) n_committed[r] = count;
}

int grid_1d(long long work, int per_block = 256) {
    long long g = (work + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > 4096) g = 4096;
    return static_cast<int>(g);
}

// Round-loop condition (one CTA): continue while any position of the block is
// masked and fewer than max_rounds rounds have run.  add = 1 counts the round
// that just ended (inside the loop body); add = 0 starts the count (before it).
__global__ void __launch_bounds__(256) loop_cond_kernel(cudaGraphConditionalHandle h, const uint8_t* __restrict__ masked,
                                                        int T, int32_t* __restrict__ rounds, int max_rounds, int add) {
    int any = 0;
    for (int t = threadIdx.x; t < T; t += blockDim.x) any |= masked[t] != 0;
    any = __syncthreads_or(any);
    if (threadIdx.x == 0) {
        const int r = add ? *rounds + 1 : 0;
        *rounds = r;
        cudaGraphSetConditional(h, (any && r < max_rounds) ? 1u : 0u);
    }
}

}  // namespace

cudaError_t launch_combine(int mode, int dtype, int T, int H, int k, const float* y, const int32_t* slot_of,
                           const int32_t* slot_sh, const float* gate_rr, int has_shared, const float* h_in, float* h,
                           void* x, float* x_f32, float* out, cudaStream_t s) {
#define MOESTEP_COMBINE(TT, MM)                                                                                 \
    launch_pdl(combine_kernel<TT, MM>, dim3(T), dim3(256), 0, s, H, k, y, slot_of, slot_sh, gate_rr, has_shared, \
               h_in, h, static_cast<TT*>(x), x_f32, out)
    if (dtype == MOESTEP_BF16) {
        if (mode == 0) return MOESTEP_COMBINE(bf16, 0);
        if (mode == 1) return MOESTEP_COMBINE(bf16, 1);
        return MOESTEP_COMBINE(bf16, 2);
    }
    if (mode == 0) return MOESTEP_COMBINE(float, 0);
    if (mode == 1) return MOESTEP_COMBINE(float, 1);
    return MOESTEP_COMBINE(float, 2);
#undef MOESTEP_COMBINE
}

cudaError_t launch_embed(int dtype, int T, int H, int P, int V, const int32_t* tokens, const uint8_t* masked,
                         const void* emb, const void* pos, int mask_id, float* h, cudaStream_t s) {
    if (dtype == MOESTEP_BF16)
        return launch_pdl(embed_kernel<bf16>, dim3(T), dim3(256), 0, s, H, P, V, tokens, masked,
                          static_cast<const bf16*>(emb), static_cast<const bf16*>(pos), mask_id, h);
    return launch_pdl(embed_kernel<float>, dim3(T), dim3(256), 0, s, H, P, V, tokens, masked,
                      static_cast<const float*>(emb), static_cast<const float*>(pos), mask_id, h);
}

cudaError_t launch_f32_gateup(int H, int E, int I, int Is, int max_slots, const float* xp, const int32_t* slot_exp,
                              const int* plan, const float* Wgu, const float* Wsgu, float* act, int act_ld,
                              cudaStream_t s) {
    const int Imax = I > Is ? I : Is;
    return launch_pdl(f32_gateup_kernel, dim3(grid_1d(static_cast<long long>(max_slots) * Imax)), dim3(256), 0, s,
                      H, E, I, Is, Imax, max_slots, xp, slot_exp, plan, Wgu, Wsgu, act, act_ld);
}

cudaError_t launch_f32_down(int H, int E, int I, int Is, int max_slots, const float* act, int act_ld,
                            const int32_t* slot_exp, const int* plan, const float* Wd, const float* Wsd, float* y,
                            cudaStream_t s) {
    return launch_pdl(f32_down_kernel, dim3(grid_1d(static_cast<long long>(max_slots) * H)), dim3(256), 0, s, H, E,
                      I, Is, max_slots, act, act_ld, slot_exp, plan, Wd, Wsd, y);
}

cudaError_t launch_f32_lm_logits(int T, int H, int V, const float* hidden, const float* Wlm, float scale,
                                 float* logits, cudaStream_t s) {
    return launch_pdl(f32_lm_logits_kernel, dim3(grid_1d(static_cast<long long>(T) * V)), dim3(256), 0, s, T, H, V,
                      hidden, Wlm, scale, logits);
}

cudaError_t launch_partials_from_logits(const float* logits, int T, int V, float* pmax, int* parg, float* psum,
                                        cudaStream_t s) {
    const dim3 grid((V + kLogitTile - 1) / kLogitTile, T);
    return launch_pdl(partials_kernel, grid, dim3(256), 0, s, logits, T, V, pmax, parg, psum);
}

cudaError_t launch_commit(int R, int P, int n_tiles, const float* pmax, const int* parg, const float* psum,
                          float threshold, int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf,
                          uint8_t* accept, int32_t* n_committed, int* counters, cudaStream_t s) {
    return launch_pdl(commit_kernel, dim3(R * P), dim3(256), 0, s, P, R * P, n_tiles, pmax, parg, psum, threshold,
                      tokens, masked, choice, conf, accept, n_committed, counters);
}

cudaError_t launch_loop_cond(cudaGraphConditionalHandle h, const uint8_t* masked, int T, int32_t* rounds,
                             int max_rounds, int add, cudaStream_t s) {
    loop_cond_kernel<<<1, 256, 0, s>>>(h, masked, T, rounds, max_rounds, add);
    return cudaGetLastError();
}

}  // namespace moestep
