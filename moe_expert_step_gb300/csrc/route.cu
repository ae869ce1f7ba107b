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
#include "launch.cuh"

namespace moestep {
namespace {

constexpr int kRouteTokens = kRouteTokensPerCta;
constexpr int kRouteExperts = 8;  // experts per router CTA (one per warp)

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
struct Vec8;  // 8 consecutive elements loaded with 16-byte accesses
template <>
struct Vec8<bf16> {
    uint4 raw;
    __device__ __forceinline__ void load(const bf16* p) { raw = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ void load_shared(const bf16* p) { raw = *reinterpret_cast<const uint4*>(p); }
    __device__ __forceinline__ void store(bf16* p) const { *reinterpret_cast<uint4*>(p) = raw; }
    __device__ __forceinline__ static void zero(bf16* p) { *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ void to_f32(float* v) const {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h2[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
};
template <>
struct Vec8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void load_shared(const float* p) {
        a = *reinterpret_cast<const float4*>(p);
        b = *(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void store(float* p) const {
        *reinterpret_cast<float4*>(p) = a;
        *(reinterpret_cast<float4*>(p) + 1) = b;
    }
    __device__ __forceinline__ static void zero(float* p) {
        *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
        *(reinterpret_cast<float4*>(p) + 1) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void to_f32(float* v) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// grid (ceil(T/8), ceil(E/8)), 256 threads.  Each CTA stages 8 tokens of x in
// shared memory; each warp computes one expert's logits for those tokens (every
// lane's 16-byte weight loads are issued before any is used).  The last CTA to
// finish a token group (atomic counter, reset by that CTA) runs the softmax and
// top-k of the group's tokens, one warp per token.
template <typename T>
__global__ void __launch_bounds__(256) route_kernel(const T* __restrict__ x, const T* __restrict__ Wr, int ntok, int H,
                                                    int E, int k, float* __restrict__ logits, int32_t* idx,
                                                    float* mass, float* gate, int* counters) {
    extern __shared__ __align__(16) uint8_t route_smem[];
    T* xs = reinterpret_cast<T*>(route_smem);  // [8][H] staged in the input type
    __shared__ int last;
    const int t0 = blockIdx.x * kRouteTokens;
    const int nt = min(kRouteTokens, ntok - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.y * kRouteExperts + warp;
    const int nchunk = (H + 255) >> 8;  // warp-wide passes of 256 elements (8 per lane)
    const T* wrow = Wr + static_cast<size_t>(e < E ? e : 0) * H;
    pdl_trigger();
    pdl_wait();  // nothing is read before every earlier kernel in the stream has finished
    // the first 8 passes' weight loads go out together with the staging loads of x
    Vec8<T> w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int hb = q * 256 + lane * 8;
        if (e < E && hb < H) w[q].load(wrow + hb);
    }
    {
        const int vec = (kRouteTokens * H) >> 3;  // 8-element vectors of the token tile
#pragma unroll 8
        for (int i = threadIdx.x; i < vec; i += blockDim.x) {
            const int tt = (i * 8) / H;
            Vec8<T> xv;
            if (tt < nt) {
                xv.load(x + static_cast<size_t>(t0) * H + static_cast<size_t>(i) * 8);
                xv.store(xs + static_cast<size_t>(i) * 8);
            } else {
                Vec8<T>::zero(xs + static_cast<size_t>(i) * 8);
            }
        }
    }
    __syncthreads();
    if (e < E) {
        float acc[kRouteTokens];
#pragma unroll
        for (int tt = 0; tt < kRouteTokens; ++tt) acc[tt] = 0.f;
        for (int c0 = 0; c0 < nchunk; c0 += 8) {
            if (c0 > 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int hb = (c0 + q) * 256 + lane * 8;
                    if (hb < H) w[q].load(wrow + hb);
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int hb = (c0 + q) * 256 + lane * 8;
                if (hb < H) {
                    float wv[8];
                    w[q].to_f32(wv);
#pragma unroll
                    for (int tt = 0; tt < kRouteTokens; ++tt) {
                        Vec8<T> xv;
                        xv.load_shared(xs + static_cast<size_t>(tt) * H + hb);
                        float xf[8];
                        xv.to_f32(xf);
                        float sacc = acc[tt];
#pragma unroll
                        for (int u = 0; u < 8; ++u) sacc = fmaf(wv[u], xf[u], sacc);
                        acc[tt] = sacc;
                    }
                }
            }
        }
#pragma unroll
        for (int tt = 0; tt < kRouteTokens; ++tt) {
            const float v = warp_sum(acc[tt]);
            if (lane == tt && tt < nt) logits[static_cast<size_t>(t0 + tt) * E + e] = v;
        }
    }
    // ---- last CTA of this token group does the softmax / top-k
    __threadfence();
    __syncthreads();
    if (gridDim.y > 1) {
        if (threadIdx.x == 0) {
            const int prev = atomicAdd(&counters[blockIdx.x], 1);
            last = (prev == static_cast<int>(gridDim.y) - 1);
            if (last) counters[blockIdx.x] = 0;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
    }
    float* zs = reinterpret_cast<float*>(route_smem);  // reuse: [8][E]
    const int n = nt * E;
#pragma unroll 8
    for (int i = threadIdx.x; i < n; i += blockDim.x) zs[i] = __ldcg(&logits[static_cast<size_t>(t0) * E + i]);
    __syncthreads();
    if (warp < nt) topk_one_token(zs + warp * E, E, k, t0 + warp, idx, mass, gate);
}

// one warp per token, logits given
__global__ void __launch_bounds__(256) topk_from_logits_kernel(const float* __restrict__ logits, int ntok, int E,
                                                               int k, int32_t* idx, float* mass, float* gate) {
    extern __shared__ __align__(16) uint8_t topk_smem[];
    float* zs = reinterpret_cast<float*>(topk_smem);  // [8][E]
    pdl_trigger();
    pdl_wait();
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

constexpr int kCandCache = 2048;  // candidates of one request kept in shared memory

// grid R, 1024 threads.  Phase 1 (every CTA): the coreset of request blockIdx.x.
// Phase 2 (the last CTA to finish, or the only one): the grouped-by-expert
// work plan over the union of all requests' kept experts.
__global__ void __launch_bounds__(kCoresetThreads) coreset_kernel(CoresetArgs a) {
    __shared__ long long A[1024];
    __shared__ long long cum[1024];
    __shared__ int cnt[1024];
    __shared__ int order[1024];
    __shared__ int keep[1024];
    __shared__ int cidx[kCandCache];
    __shared__ float cmass[kCandCache];
    __shared__ uint8_t csurv[kCandCache];
    __shared__ long long wtot64[32];
    __shared__ int wtot32[32];
    __shared__ int s_last, s_nr, s_nrc;
    extern __shared__ uint32_t masks[];  // phase 2: [E][ceil(T/32)]

    const int tid = threadIdx.x;
    const int r = blockIdx.x;
    const int E = a.E, k = a.k, P = a.P;
    const int nc = P * k;                    // candidates of this request
    const bool cached = nc <= kCandCache;
    const int base = r * nc;                 // first candidate of this request in idx/mass
    // one request whose candidates all fit in shared memory: the plan reuses phase 1's counts
    const bool local = gridDim.x == 1 && cached;
    const int TWl = (P + 31) >> 5;
    pdl_trigger();
    pdl_wait();
    const float tp = a.top_p[r];
    // ---------------- phase 1
    if (tid < E) {
        A[tid] = 0;
        cnt[tid] = 0;
    }
    if (local)
        for (int i = tid; i < E * TWl; i += blockDim.x) masks[i] = 0u;
    __syncthreads();
    for (int c = tid; c < nc; c += blockDim.x) {
        const int e = a.idx[base + c];
        const float ms = a.mass[base + c];
        if (cached) {
            cidx[c] = e;
            cmass[c] = ms;
        }
        if (e < 0 || e >= E) {
            record_error(a.err, kErrBadInput);
            continue;
        }
        const long long q = __float2ll_rn(ms * 0x1p54f);
        atomicAdd(reinterpret_cast<unsigned long long*>(&A[e]), static_cast<unsigned long long>(q));
        atomicAdd(&cnt[e], 1);
        if (local) {
            const int t = c / k;
            atomicOr(&masks[e * TWl + (t >> 5)], 1u << (t & 31));
        }
    }
    __syncthreads();
    // rank of every candidate expert, (aggregate desc, id asc): `parts` threads share one expert
    int parts = 1;
    while (parts < 32 && parts * 2 * E <= kCoresetThreads) parts *= 2;
    {
        const int e = tid / parts, part = tid % parts;
        int rk = 0;
        const bool mine_valid = e < E && cnt[e] > 0;
        if (mine_valid) {
            const long long mine = A[e];
            const int per = (E + parts - 1) / parts;
            const int lo = part * per, hi = min(E, lo + per);
            for (int e2 = lo; e2 < hi; ++e2)
                if (cnt[e2] > 0 && (A[e2] > mine || (A[e2] == mine && e2 < e))) ++rk;
        }
        for (int o = 1; o < parts; o <<= 1) rk += __shfl_xor_sync(0xffffffffu, rk, o);
        if (mine_valid && part == 0) order[rk] = e;
        if (part == 0 && e < E) keep[e] = mine_valid ? rk : -1;  // rank for now, flag below
    }
    int nC = 0;
    {
        const int e = tid;
        nC = __syncthreads_count(e < E && cnt[e] > 0);
    }
    long long v = (tid < nC) ? A[order[tid]] : 0;
    v = block_inclusive_scan<long long>(v, wtot64);
    if (tid < nC) cum[tid] = v;
    __syncthreads();
    const long long total = nC > 0 ? cum[nC - 1] : 0;
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
    if (tid < E) keep[tid] = (keep[tid] >= 0 && keep[tid] < m);
    if (tid < m) a.sel[r * E + tid] = order[tid];
    if (tid == 0) a.n_sel[r] = m;
    __syncthreads();
    for (int tt = tid; tt < P; tt += blockDim.x) {
        const int c0 = tt * k;
        // candidates in groups of 8; the renormaliser is summed in candidate order
        float denom = 0.f;
        for (int j0 = 0; j0 < k; j0 += 8) {
            int ev[8];
            float mv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + j0 + q;
                const bool in = j0 + q < k;
                ev[q] = in ? (cached ? cidx[c] : a.idx[base + c]) : -1;
                mv[q] = in ? (cached ? cmass[c] : a.mass[base + c]) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (ev[q] >= 0 && ev[q] < E && keep[ev[q]]) denom += mv[q];
        }
        for (int j0 = 0; j0 < k; j0 += 8) {
            int ev[8];
            float mv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + j0 + q;
                const bool in = j0 + q < k;
                ev[q] = in ? (cached ? cidx[c] : a.idx[base + c]) : -1;
                mv[q] = in ? (cached ? cmass[c] : a.mass[base + c]) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = c0 + j0 + q;
                if (j0 + q < k) {
                    const bool sv = ev[q] >= 0 && ev[q] < E && keep[ev[q]];
                    a.survive[base + c] = sv ? 1 : 0;
                    a.gate_rr[base + c] = (sv && denom > 0.f) ? mv[q] / denom : 0.f;
                    if (cached) csurv[c] = sv ? 1 : 0;
                }
            }
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
    if (!local) {  // count survivors per expert over every request
        for (int i = tid; i < E * TW; i += blockDim.x) masks[i] = 0u;
        if (tid < E) cnt[tid] = 0;
        __syncthreads();
        for (int c = tid; c < T * k; c += blockDim.x) {
            if (__ldcg(&a.survive[c]) != 0) {
                const int e = __ldcg(&a.idx[c]);
                const int t = c / k;
                atomicAdd(&cnt[e], 1);
                atomicOr(&masks[e * TW + (t >> 5)], 1u << (t & 31));
            }
        }
        __syncthreads();
    }
    // one request: every candidate of a kept expert survives, so phase 1's counts and masks hold
    const int my_cnt = tid < E ? ((local && !keep[tid]) ? 0 : cnt[tid]) : 0;
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
    if (tid == kCoresetThreads - 1) {
        s_nr = slot_end;
        s_nrc = chunk_end;
    }
    __syncthreads();
    const int NR = s_nr, nrc = s_nrc;
    for (int c = tid; c < T * k; c += blockDim.x) {
        const bool sv = local ? csurv[c] != 0 : __ldcg(&a.survive[c]) != 0;
        if (sv) {
            const int e = local ? cidx[c] : __ldcg(&a.idx[c]);
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

// One CTA per slot: xp[slot] = x[slot_tok[slot]].  Then, while HBM would
// otherwise idle until the expert GEMM starts streaming, every thread hints a
// few 128-byte lines of the gate/up weights of the first chunks in the plan
// (the experts the GEMM processes first) into L2.  The hints are
// fire-and-forget: nothing waits for them.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, int row_vec,
                                                     const int32_t* __restrict__ slot_tok, const int* __restrict__ plan,
                                                     uint4* __restrict__ xp, const int4* __restrict__ chunks,
                                                     const char* __restrict__ pf_base, long long pf_stride,
                                                     int pf_chunks, int* __restrict__ done, int n_done) {
    const int slot = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (done != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_done; i += blockDim.x) done[i] = 0;
    if (slot < plan[2]) {
        const int t = slot_tok[slot];
        for (int i = threadIdx.x; i < row_vec; i += blockDim.x)
            xp[static_cast<size_t>(slot) * row_vec + i] = x[static_cast<size_t>(t) * row_vec + i];
    }
    if (pf_base != nullptr) {
        const int nc = min(pf_chunks, plan[0]);
        const long long lines_per = pf_stride >> 7;
        const long long total = lines_per * nc;
        const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
        for (long long l = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; l < total; l += nthreads) {
            const int c = static_cast<int>(l / lines_per);
            const long long off = (l - c * lines_per) << 7;
            const char* p = pf_base + static_cast<long long>(chunks[c].x) * pf_stride + off;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
        }
    }
}

}  // namespace

cudaError_t launch_route(int dtype, const void* x, const void* Wr, int T, int H, int E, int k, float* logits,
                         int32_t* idx, float* mass, float* gate, int* counters, int* err, cudaStream_t s) {
    (void)err;
    const dim3 grid((T + kRouteTokens - 1) / kRouteTokens, (E + kRouteExperts - 1) / kRouteExperts);
    const size_t esz = dtype == MOESTEP_BF16 ? 2 : 4;
    const size_t xs_bytes = static_cast<size_t>(kRouteTokens) * H * esz;
    const size_t zs_bytes = static_cast<size_t>(kRouteTokens) * E * sizeof(float);
    const size_t smem = xs_bytes > zs_bytes ? xs_bytes : zs_bytes;
    cudaError_t e;
    static int done_bf16[64] = {}, done_f32[64] = {};
    if (dtype == MOESTEP_BF16) {
        if ((e = ensure_smem(route_kernel<bf16>, smem, done_bf16)) != cudaSuccess) return e;
        return launch_pdl(route_kernel<bf16>, grid, dim3(256), smem, s, static_cast<const bf16*>(x),
                          static_cast<const bf16*>(Wr), T, H, E, k, logits, idx, mass, gate, counters);
    }
    if ((e = ensure_smem(route_kernel<float>, smem, done_f32)) != cudaSuccess) return e;
    return launch_pdl(route_kernel<float>, grid, dim3(256), smem, s, static_cast<const float*>(x),
                      static_cast<const float*>(Wr), T, H, E, k, logits, idx, mass, gate, counters);
}

cudaError_t launch_topk_from_logits(const float* logits, int T, int E, int k, int32_t* idx, float* mass, float* gate,
                                    cudaStream_t s) {
    const size_t smem = 8ull * E * sizeof(float);
    static int done[64] = {};
    cudaError_t e = ensure_smem(topk_from_logits_kernel, smem, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_from_logits_kernel, dim3((T + 7) / 8), dim3(256), smem, s, logits, T, E, k, idx, mass,
                      gate);
}

int coreset_smem_bytes(int E, int T) { return E * ((T + 31) / 32) * 4; }

cudaError_t launch_coreset(const CoresetArgs& a, cudaStream_t s) {
    const size_t smem = coreset_smem_bytes(a.E, a.T);
    static int done[64] = {};
    cudaError_t e = ensure_smem(coreset_kernel, smem, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(coreset_kernel, dim3(a.R), dim3(kCoresetThreads), smem, s, a);
}

cudaError_t launch_gather(int dtype, const void* x, int H, const int32_t* slot_tok, const int* plan, int max_slots,
                          void* xp, const int4* chunks, const void* pf_wgu, long long pf_stride, int pf_chunks,
                          int* done, int n_done, cudaStream_t s) {
    const int row_vec = H * (dtype == MOESTEP_BF16 ? 2 : 4) / 16;
    return launch_pdl(gather_kernel, dim3(max_slots), dim3(256), 0, s, static_cast<const uint4*>(x), row_vec,
                      slot_tok, plan, static_cast<uint4*>(xp), chunks, static_cast<const char*>(pf_wgu), pf_stride,
                      pf_chunks, done, n_done);
}

}  // namespace moestep
