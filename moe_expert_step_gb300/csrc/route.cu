// Router (softmax/top-k per token), block coreset selection and the
// grouped-by-expert work plan, and the activation gather that feeds the
// expert GEMM.
//
// Router [AIT 四]: z = x Wr^T with fp32 accumulation, softmax over the E
// experts, top-k by z (ties to the lower expert id), mass = p at the chosen
// experts, gate = mass renormalised over the k.
// Coreset [GRM "What is the MoE coreset and why does it matter?"]: per request,
// sum candidate masses per expert (exact 2^-54 fixed point), rank experts by
// the sum, keep the shortest prefix that reaches top_p of the total, restrict
// every token to its kept candidates and renormalise its gates.
#include "common.cuh"
#include "kernels.h"

namespace moestep {
namespace {

constexpr int kRouteTokens = 8;    // tokens per router CTA
constexpr int kRouteExperts = 32;  // experts per router CTA (4 per warp)

// Top-k of one token's logits by one warp.  `s` holds the E logits (shared memory).
__device__ void topk_one_token(const float* s, int E, int k, int t, int32_t* idx, float* mass, float* gate) {
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, s[e]);
    m = warp_max(m);
    float sum = 0.f;
    for (int e = lane; e < E; e += 32) sum += expf(s[e] - m);
    sum = warp_sum(sum);
    uint32_t taken = 0;  // bit q: entry lane + 32q already chosen
    float mine = 0.f, gsum = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        int q = 0;
        for (int e = lane; e < E; e += 32, ++q)
            if (!((taken >> q) & 1u) && (s[e] > bv || bi == 0x7fffffff)) {
                bv = s[e];
                bi = e;
            }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        const float mj = expf(bv - m) / sum;
        gsum += mj;
        if (lane == j) mine = mj;
        if (lane == 0) {
            idx[t * k + j] = bi;
            mass[t * k + j] = mj;
        }
    }
    if (lane < k) gate[t * k + lane] = mine / gsum;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* v);
template <>
__device__ __forceinline__ void load8<bf16>(const bf16* p, float* v) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h2[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* v) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// grid (ceil(T/8), ceil(E/32)), 256 threads.  Each CTA computes the logits of
// 8 tokens x 32 experts; the last CTA to finish a token group (counted with an
// atomic, self-resetting) runs the softmax/top-k for those tokens.
template <typename T>
__global__ void __launch_bounds__(256) route_kernel(const T* __restrict__ x, const T* __restrict__ Wr, int ntok, int H,
                                                    int E, int k, float* __restrict__ logits, int32_t* idx,
                                                    float* mass, float* gate, int* counters) {
    extern __shared__ __align__(16) uint8_t route_smem[];
    float* xs = reinterpret_cast<float*>(route_smem);  // [8][H]
    __shared__ int last;
    const int t0 = blockIdx.x * kRouteTokens;
    const int nt = min(kRouteTokens, ntok - t0);
    for (int i = threadIdx.x; i < kRouteTokens * H; i += blockDim.x) {
        const int tt = i / H;
        xs[i] = tt < nt ? to_f32(x[static_cast<size_t>(t0 + tt) * H + (i - tt * H)]) : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ebase = blockIdx.y * kRouteExperts + warp * 4;
    float acc[4][kRouteTokens];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < kRouteTokens; ++b) acc[a][b] = 0.f;
    for (int hb = lane * 8; hb < H; hb += 256) {
        float xv[kRouteTokens][8];
#pragma unroll
        for (int tt = 0; tt < kRouteTokens; ++tt) {
            const float4 a = *reinterpret_cast<const float4*>(&xs[tt * H + hb]);
            const float4 b = *reinterpret_cast<const float4*>(&xs[tt * H + hb + 4]);
            xv[tt][0] = a.x; xv[tt][1] = a.y; xv[tt][2] = a.z; xv[tt][3] = a.w;
            xv[tt][4] = b.x; xv[tt][5] = b.y; xv[tt][6] = b.z; xv[tt][7] = b.w;
        }
#pragma unroll
        for (int ee = 0; ee < 4; ++ee) {
            const int e = ebase + ee;
            if (e < E) {
                float w[8];
                load8<T>(Wr + static_cast<size_t>(e) * H + hb, w);
#pragma unroll
                for (int tt = 0; tt < kRouteTokens; ++tt)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[ee][tt] = fmaf(w[q], xv[tt][q], acc[ee][tt]);
            }
        }
    }
#pragma unroll
    for (int ee = 0; ee < 4; ++ee) {
#pragma unroll
        for (int tt = 0; tt < kRouteTokens; ++tt) {
            const float v = warp_sum(acc[ee][tt]);
            const int e = ebase + ee;
            if (lane == 0 && e < E && tt < nt) logits[static_cast<size_t>(t0 + tt) * E + e] = v;
        }
    }
    // ---- last CTA of this token group does the softmax / top-k
    if (gridDim.y > 1) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int prev = atomicAdd(&counters[blockIdx.x], 1);
            last = (prev == static_cast<int>(gridDim.y) - 1);
            if (last) counters[blockIdx.x] = 0;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
    } else {
        __threadfence();
        __syncthreads();
    }
    float* zs = xs;  // reuse: [8][E]
    __syncthreads();
    for (int i = threadIdx.x; i < nt * E; i += blockDim.x) zs[i] = __ldcg(&logits[static_cast<size_t>(t0) * E + i]);
    __syncthreads();
    if (warp < nt) topk_one_token(zs + warp * E, E, k, t0 + warp, idx, mass, gate);
}

// one warp per token, logits given
__global__ void __launch_bounds__(256) topk_from_logits_kernel(const float* __restrict__ logits, int ntok, int E,
                                                               int k, int32_t* idx, float* mass, float* gate) {
    extern __shared__ __align__(16) uint8_t topk_smem[];
    float* zs = reinterpret_cast<float*>(topk_smem);  // [8][E]
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (t >= ntok) return;
    float* s = zs + warp * E;
    for (int e = threadIdx.x & 31; e < E; e += 32) s[e] = logits[static_cast<size_t>(t) * E + e];
    __syncwarp();
    topk_one_token(s, E, k, t, idx, mass, gate);
}

// ---------------------------------------------------------------------------- coreset
constexpr int kCoresetThreads = 1024;

// Inclusive prefix sum over one value per thread of a 1024-thread block.
template <typename V>
__device__ V block_inclusive_scan(V v, V* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        V w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const V n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += warp_tot[warp - 1];
    __syncthreads();
    return v;
}

// grid R, 1024 threads.  Phase 1 (every CTA): the coreset of request blockIdx.x.
// Phase 2 (the last CTA to finish, or the only one): the grouped-by-expert
// work plan over the union of all requests' kept experts.
__global__ void __launch_bounds__(kCoresetThreads) coreset_kernel(CoresetArgs a) {
    __shared__ long long A[1024];
    __shared__ long long cum[1024];
    __shared__ int cnt[1024];
    __shared__ int order[1024];
    __shared__ int keep[1024];
    __shared__ long long wtot64[32];
    __shared__ int wtot32[32];
    __shared__ int s_last;
    extern __shared__ uint32_t masks[];  // phase 2: [E][ceil(T/32)]

    const int tid = threadIdx.x;
    const int r = blockIdx.x;
    const int E = a.E, k = a.k, P = a.P;
    // ---------------- phase 1
    if (tid < E) {
        A[tid] = 0;
        cnt[tid] = 0;
    }
    __syncthreads();
    for (int c = tid; c < P * k; c += blockDim.x) {
        const int t = r * P + c / k;
        const int j = c - (c / k) * k;
        const int e = a.idx[t * k + j];
        if (e < 0 || e >= E) {
            record_error(a.err, kErrBadInput);
            continue;
        }
        const long long q = __float2ll_rn(a.mass[t * k + j] * 0x1p54f);
        atomicAdd(reinterpret_cast<unsigned long long*>(&A[e]), static_cast<unsigned long long>(q));
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // rank of every candidate expert: (aggregate desc, id asc)
    int my_rank = -1;
    if (tid < E && cnt[tid] > 0) {
        const long long mine = A[tid];
        int rk = 0;
        for (int e2 = 0; e2 < E; ++e2)
            if (cnt[e2] > 0 && (A[e2] > mine || (A[e2] == mine && e2 < tid))) ++rk;
        my_rank = rk;
        order[rk] = tid;
    }
    const int nC = __syncthreads_count(my_rank >= 0);
    long long v = (tid < nC) ? A[order[tid]] : 0;
    v = block_inclusive_scan<long long>(v, wtot64);
    if (tid < nC) cum[tid] = v;
    __syncthreads();
    const long long total = nC > 0 ? cum[nC - 1] : 0;
    const float tp = a.top_p[r];
    int m;
    if (!(tp > 0.0f)) {  // NaN or non-positive fraction: keep everything and flag the input
        if (tid == 0) record_error(a.err, kErrBadInput);
        m = nC;
    } else if (tp >= 1.0f || total == 0) {
        m = nC;
    } else {
        long long target = static_cast<long long>(ceil(__dmul_rn(static_cast<double>(tp), __ll2double_rn(total))));
        target = target < 1 ? 1 : (target > total ? total : target);
        m = 1 + __syncthreads_count(tid < nC && cum[tid] < target);
        m = m > nC ? nC : m;
    }
    if (tid < E) keep[tid] = (my_rank >= 0 && my_rank < m);
    if (tid < m) a.sel[r * E + tid] = order[tid];
    if (tid == 0) a.n_sel[r] = m;
    __syncthreads();
    for (int tt = tid; tt < P; tt += blockDim.x) {
        const int t = r * P + tt;
        float denom = 0.f;
        for (int j = 0; j < k; ++j) {
            const int e = a.idx[t * k + j];
            if (e >= 0 && e < E && keep[e]) denom += a.mass[t * k + j];
        }
        for (int j = 0; j < k; ++j) {
            const int e = a.idx[t * k + j];
            const bool s = e >= 0 && e < E && keep[e];
            a.survive[t * k + j] = s ? 1 : 0;
            a.gate_rr[t * k + j] = (s && denom > 0.f) ? a.mass[t * k + j] / denom : 0.f;
        }
    }
    // ---------------- phase 2 (one CTA)
    if (gridDim.x > 1) {
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int prev = atomicAdd(a.counter, 1);
            s_last = (prev == static_cast<int>(gridDim.x) - 1);
            if (s_last) *a.counter = 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    } else {
        __threadfence();
        __syncthreads();
    }
    const int T = a.T;
    const int TW = (T + 31) >> 5;
    for (int i = tid; i < E * TW; i += blockDim.x) masks[i] = 0u;
    if (tid < E) cnt[tid] = 0;
    __syncthreads();
    for (int c = tid; c < T * k; c += blockDim.x) {
        if (__ldcg(&a.survive[c])) {
            const int e = __ldcg(&a.idx[c]);
            const int t = c / k;
            atomicAdd(&cnt[e], 1);
            atomicOr(&masks[e * TW + (t >> 5)], 1u << (t & 31));
        }
    }
    __syncthreads();
    const int my_cnt = tid < E ? cnt[tid] : 0;
    const int my_nch = (my_cnt + a.nch - 1) / a.nch;
    const int slot_end = block_inclusive_scan<int>(my_cnt, wtot32);
    const int chunk_end = block_inclusive_scan<int>(my_nch, wtot32);
    const int slot_base = slot_end - my_cnt;
    const int chunk_base = chunk_end - my_nch;
    if (tid < E) {
        order[tid] = slot_base;  // reuse: first slot of expert tid
        for (int i = 0; i < my_nch; ++i)
            a.chunks[chunk_base + i] = make_int4(tid, slot_base + i * a.nch, min(a.nch, my_cnt - i * a.nch), 0);
    }
    __shared__ int s_nr, s_nrc;
    if (tid == kCoresetThreads - 1) {
        s_nr = slot_end;
        s_nrc = chunk_end;
    }
    __syncthreads();
    const int NR = s_nr, nrc = s_nrc;
    for (int c = tid; c < T * k; c += blockDim.x) {
        if (__ldcg(&a.survive[c])) {
            const int e = __ldcg(&a.idx[c]);
            const int t = c / k;
            const int w = t >> 5;
            int pos = order[e];
            for (int q = 0; q < w; ++q) pos += __popc(masks[e * TW + q]);
            pos += __popc(masks[e * TW + w] & ((1u << (t & 31)) - 1u));
            a.slot_of[c] = pos;
            a.slot_tok[pos] = t;
            a.slot_exp[pos] = e;
        } else {
            a.slot_of[c] = -1;
        }
    }
    int nsc = 0;
    if (a.has_shared) {
        nsc = (T + a.nch - 1) / a.nch;
        for (int t = tid; t < T; t += blockDim.x) {
            a.slot_sh[t] = NR + t;
            a.slot_tok[NR + t] = t;
            a.slot_exp[NR + t] = E;
        }
        for (int i = tid; i < nsc; i += blockDim.x)
            a.chunks[nrc + i] = make_int4(E, NR + i * a.nch, min(a.nch, T - i * a.nch), 0);
    }
    if (tid == 0) {
        a.plan[0] = nrc;
        a.plan[1] = nsc;
        a.plan[2] = NR + (a.has_shared ? T : 0);
    }
}

// one CTA per slot: xp[slot] = x[slot_tok[slot]]
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, int row_vec,
                                                     const int32_t* __restrict__ slot_tok, const int* __restrict__ plan,
                                                     uint4* __restrict__ xp) {
    const int slot = blockIdx.x;
    if (slot >= plan[2]) return;
    const int t = slot_tok[slot];
    for (int i = threadIdx.x; i < row_vec; i += blockDim.x)
        xp[static_cast<size_t>(slot) * row_vec + i] = x[static_cast<size_t>(t) * row_vec + i];
}

}  // namespace

cudaError_t launch_route(int dtype, const void* x, const void* Wr, int T, int H, int E, int k, float* logits,
                         int32_t* idx, float* mass, float* gate, int* counters, int* err, cudaStream_t s) {
    (void)err;
    const dim3 grid((T + kRouteTokens - 1) / kRouteTokens, (E + kRouteExperts - 1) / kRouteExperts);
    const size_t smem = static_cast<size_t>(kRouteTokens) * (H > E ? H : E) * sizeof(float);
    if (dtype == MOESTEP_BF16) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(route_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        route_kernel<bf16><<<grid, 256, smem, s>>>(static_cast<const bf16*>(x), static_cast<const bf16*>(Wr), T, H,
                                                   E, k, logits, idx, mass, gate, counters);
    } else {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(route_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        route_kernel<float><<<grid, 256, smem, s>>>(static_cast<const float*>(x), static_cast<const float*>(Wr), T,
                                                    H, E, k, logits, idx, mass, gate, counters);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk_from_logits(const float* logits, int T, int E, int k, int32_t* idx, float* mass, float* gate,
                                    cudaStream_t s) {
    const size_t smem = 8ull * E * sizeof(float);
    topk_from_logits_kernel<<<(T + 7) / 8, 256, smem, s>>>(logits, T, E, k, idx, mass, gate);
    return cudaGetLastError();
}

int coreset_smem_bytes(int E, int T) { return E * ((T + 31) / 32) * 4; }

cudaError_t launch_coreset(const CoresetArgs& a, cudaStream_t s) {
    const int smem = coreset_smem_bytes(a.E, a.T);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(coreset_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    coreset_kernel<<<a.R, kCoresetThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather(int dtype, const void* x, int H, const int32_t* slot_tok, const int* plan, int max_slots,
                          void* xp, cudaStream_t s) {
    const int row_vec = H * (dtype == MOESTEP_BF16 ? 2 : 4) / 16;
    gather_kernel<<<max_slots, 256, 0, s>>>(static_cast<const uint4*>(x), row_vec, slot_tok, plan,
                                            static_cast<uint4*>(xp));
    return cudaGetLastError();
}

}  // namespace moestep
