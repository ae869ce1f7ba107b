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
#include <cooperative_groups.h>

#include "combine.cuh"
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "target.h"

namespace moestep {
namespace {

constexpr int kRouteTokens = kRouteTokensPerCta;
constexpr int kRouteExperts = 8;  // experts per router CTA (one per warp)

// Order-preserving unsigned key of a float (a larger float has a larger key; -0
// is taken as +0) and its inverse.
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t b = __float_as_uint(f + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token's logits by one warp.  `s` holds the E logits (shared
// memory, E <= 1024); lane l keeps the keys of entries l, l+32, ... in
// registers.  Each pick is an exact warp maximum of the keys (redux.sync) and,
// among equal values, the lowest expert id.  mass_j = exp(z_j - max) / sum of
// exp over all E (the sum per lane in entry order, then across lanes);
// gate_j = mass_j / (mass_0 + ... + mass_{k-1}), summed in pick order.
template <int kMaxPerLane>
__device__ void topk_regs(const float* s, int E, int k, int t, int32_t* idx, float* mass, float* gate,
                          int32_t* idx2, float* mass2) {
    const int lane = threadIdx.x & 31;
    const int nv = (E - lane + 31) >> 5;  // entries of this lane
    uint32_t key[kMaxPerLane];
    uint32_t km = 0u;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
        key[q] = q < nv ? fkey(s[lane + 32 * q]) : 0u;
        km = max(km, key[q]);
    }
    const float m = fkey_inv(__reduce_max_sync(0xffffffffu, km));
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q)
        if (q < nv) sum += expf(fkey_inv(key[q]) - m);
    sum = warp_sum(sum);
    uint32_t taken = 0;  // bit q: entry lane + 32q already chosen
    uint32_t bk = 0u;    // best key of this lane among the entries not taken, and its slot
    int bq = -1;
    auto local_best = [&]() {
        bk = 0u;
        bq = -1;
#pragma unroll
        for (int q = 0; q < kMaxPerLane; ++q)
            if (q < nv && !((taken >> q) & 1u) && (bq < 0 || key[q] > bk)) {
                bk = key[q];
                bq = q;
            }
    };
    local_best();
    uint32_t my_key = 0u;  // lane j: key and expert of pick j
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t kb = __reduce_max_sync(0xffffffffu, bq >= 0 ? bk : 0u);
        const int cand = (bq >= 0 && bk == kb) ? lane + 32 * bq : 0x7fffffff;
        const int bi = __reduce_min_sync(0xffffffffu, cand);
        if (lane == j) {
            my_key = kb;
            my_e = bi;
        }
        if ((bi & 31) == lane) {
            taken |= 1u << (bi >> 5);
            local_best();
        }
    }
    const float mj = lane < k ? expf(fkey_inv(my_key) - m) / sum : 0.f;
    float gsum = 0.f;
    for (int j = 0; j < k; ++j) gsum += __shfl_sync(0xffffffffu, mj, j);
    if (lane < k) {
        idx[t * k + lane] = my_e;
        mass[t * k + lane] = mj;
        gate[t * k + lane] = mj / gsum;
        if (idx2 != nullptr) {
            idx2[t * k + lane] = my_e;
            mass2[t * k + lane] = mj;
        }
    }
}

// idx2 / mass2 (may be NULL): a second copy of idx / mass
__device__ void topk_one_token(const float* s, int E, int k, int t, int32_t* idx, float* mass, float* gate,
                               int32_t* idx2 = nullptr, float* mass2 = nullptr) {
    if (E <= 256)
        topk_regs<8>(s, E, k, t, idx, mass, gate, idx2, mass2);
    else if (E <= 512)
        topk_regs<16>(s, E, k, t, idx, mass, gate, idx2, mass2);
    else
        topk_regs<32>(s, E, k, t, idx, mass, gate, idx2, mass2);
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

// grid (ceil(T/4), ceil(E/8)), 256 threads.  Each CTA stages 4 tokens of x in
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

// The block coreset and work plan, executed by one 1024-thread CTA for request
// r of nreq.  Phase 1: the coreset of request r.  Phase 2 (done by the last
// request's CTA to finish, or directly when nreq == 1): the grouped-by-expert
// work plan over the union of all requests' kept experts.  `masks` (each
// expert's token bitmask, word-major: word w of every expert side by side,
// ceil(T/32) x E words) and `sc` are shared-memory scratch.  Used by the
// coreset kernel (one CTA per request).
struct CoresetScratch {  // shared memory of one coreset CTA
    long long A[1024];
    long long cum[1024];
    int cnt[1024];
    int order[1024];
    int keep[1024];
    int cidx[kCandCache];
    float cmass[kCandCache];
    uint32_t khi[1024 + 32];  // candidates' aggregates, compacted: high words (zero padded) ...
    int ce[1024];             // ... and expert ids; the full aggregates go to cum
    long long wtot64[32];
    long long s_target;
    int s_last, s_nr, s_nrc;
    uint8_t csurv[kCandCache];
};

// Slots of the work plan staged in shared memory (token and expert of each slot)
// by the coreset launch's plan step when several requests share it, so the plan
// goes out as coalesced stores: up to kSlotStage slots, within the CTA's limit.
constexpr int kSlotStage = 8192;
__host__ __device__ inline size_t coreset_masks_bytes(int E, int T) {
    return (static_cast<size_t>(E) * ((T + 31) / 32) * 4 + 15) / 16 * 16;
}
__host__ __device__ inline int coreset_stage_slots(int E, int T, int k) {
    const size_t slots = static_cast<size_t>(T) * (k + 1);
    const size_t bytes = sizeof(CoresetScratch) + coreset_masks_bytes(E, T) + slots * 8;
    // 1 KiB left for the kernel's static shared memory
    return (slots <= kSlotStage && bytes <= 226 * 1024) ? static_cast<int>(slots) : 0;
}

// stage: shared memory for coreset_stage_slots(E, T, k) slots (2 ints each), or NULL
__device__ void coreset_body(const CoresetArgs& a, int r, int nreq, uint32_t* masks, CoresetScratch& sc,
                             int* stage = nullptr, int nstage = 0) {
    long long* A = sc.A;
    long long* cum = sc.cum;
    int* cnt = sc.cnt;
    int* order = sc.order;
    int* keep = sc.keep;
    int* cidx = sc.cidx;
    float* cmass = sc.cmass;
    uint8_t* csurv = sc.csurv;
    int& s_last = sc.s_last;
    int& s_nr = sc.s_nr;
    int& s_nrc = sc.s_nrc;

    const int tid = threadIdx.x;
    const int E = a.E, k = a.k, P = a.P;
    const int nc = P * k;                    // candidates of this request
    const bool cached = nc <= kCandCache;
    const int base = r * nc;                 // first candidate of this request in idx/mass
    // one request whose candidates all fit in shared memory: the plan reuses phase 1's counts
    const bool local = nreq == 1 && cached;
    const int TWl = (P + 31) >> 5;
    const float tp = a.top_p[r];
    // ---------------- phase 1
    if (tid < E) {
        A[tid] = 0;
        cnt[tid] = 0;
        keep[tid] = -1;
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
            atomicOr(&masks[(t >> 5) * E + e], 1u << (t & 31));
        }
    }
    __syncthreads();
    // compact the candidate experts in id order: cum[p] = aggregate, khi[p] = its high
    // word, ce[p] = expert id
    const int flag = (tid < E && cnt[tid] > 0) ? 1 : 0;
    const int incl = block_inclusive_scan<int>(flag, reinterpret_cast<int*>(sc.wtot64));
    const int nC = reinterpret_cast<int*>(sc.wtot64)[31];
    if (flag) {
        cum[incl - 1] = A[tid];
        sc.khi[incl - 1] = static_cast<uint32_t>(static_cast<unsigned long long>(A[tid]) >> 32);
        sc.ce[incl - 1] = tid;
    }
    if (tid < 32) sc.khi[nC + tid] = 0u;  // padding of the last 4-key block
    __syncthreads();
    // rank of every candidate, (aggregate desc, id asc): `parts` threads share one
    // candidate and take every parts-th block of 4 rivals.  The high words settle
    // every rival whose high word differs; a tie on the high word (rare) is settled
    // on the full aggregate and the id.  All sums are >= 0.
    {
        int parts = 1;
        while (parts < 32 && parts * 2 * nC <= kCoresetThreads) parts *= 2;
        const int p = tid / parts, part = tid % parts;
        const bool mine_ok = p < nC;
        const uint32_t mh = mine_ok ? sc.khi[p] : 0u;
        int gt = 0, eq = 0;
        if (mine_ok) {
            const int nblk = (nC + 3) >> 2;
#pragma unroll 4
            for (int b = part; b < nblk; b += parts) {
                const uint4 h = *reinterpret_cast<const uint4*>(&sc.khi[4 * b]);
                gt += (h.x > mh) + (h.y > mh) + (h.z > mh) + (h.w > mh);
                eq += (h.x == mh) + (h.y == mh) + (h.z == mh) + (h.w == mh);
            }
        }
        const int lane = tid & 31;
        const unsigned gmask = parts == 32 ? 0xffffffffu : (((1u << parts) - 1u) << (lane & ~(parts - 1)));
        for (int o = 1; o < parts; o <<= 1) {
            gt += __shfl_xor_sync(gmask, gt, o);
            eq += __shfl_xor_sync(gmask, eq, o);
        }
        if (mine_ok && eq > 1) {  // uniform within the group of `parts` lanes
            const long long mine = cum[p];
            int add = 0;
            for (int p2 = part; p2 < nC; p2 += parts)
                if (p2 != p && sc.khi[p2] == mh) {
                    const long long o = cum[p2];
                    add += (o > mine || (o == mine && p2 < p)) ? 1 : 0;
                }
            for (int o = 1; o < parts; o <<= 1) add += __shfl_xor_sync(gmask, add, o);
            gt += add;
        }
        if (mine_ok && part == 0) {
            order[gt] = sc.ce[p];
            keep[sc.ce[p]] = gt;  // rank for now, flag below
        }
    }
    __syncthreads();
    // the cut: m = smallest prefix of the ranked candidates whose aggregate reaches
    // ceil(top_p * total) (exact integer sums; one thread takes the target)
    long long v = (tid < nC) ? A[order[tid]] : 0;
    v = block_inclusive_scan<long long>(v, sc.wtot64);
    const long long total = sc.wtot64[31];
    int m = nC;
    if (!(tp > 0.0f)) {  // NaN or non-positive fraction: keep everything and flag the input
        if (tid == 0) record_error(a.err, kErrBadInput);
    } else if (tp < 1.0f && total != 0) {
        if (tid == 0) sc.s_target = coreset_target(tp, total);
        __syncthreads();
        m = 1 + __syncthreads_count(tid < nC && v < sc.s_target);
        m = m > nC ? nC : m;
    }
    if (tid == 0) a.n_sel[r] = m;
    if (tid < E) keep[tid] = (keep[tid] >= 0 && keep[tid] < m);
    if (tid < m) a.sel[r * E + tid] = order[tid];
    __syncthreads();
    if (cached && nc <= static_cast<int>(blockDim.x) && (32 % k) == 0) {
        // one thread per candidate; a token's k candidates are k adjacent lanes, and
        // each lane sums the kept masses of its token in candidate order
        const int c = tid;
        const bool valid = c < nc;
        const int e = valid ? cidx[c] : -1;
        const float ms = valid ? cmass[c] : 0.f;
        const bool sv = e >= 0 && e < E && keep[e];
        const float mv = sv ? ms : 0.f;
        const int g0 = (threadIdx.x & 31) / k * k;
        float denom = 0.f;
        for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, mv, g0 + j);
        if (valid) {
            a.survive[base + c] = sv ? 1 : 0;
            a.gate_rr[base + c] = (sv && denom > 0.f) ? ms / denom : 0.f;
            csurv[c] = sv ? 1 : 0;
        }
    } else {
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
    }
    // ---------------- phase 2 (one CTA)
    if (nreq > 1) {
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int prev = atomicAdd(a.counter, 1);
            s_last = (prev == nreq - 1);
            if (s_last) *a.counter = 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    } else {
        if (!local) __threadfence();
        __syncthreads();
    }
    const int T = a.T;
    const int TW = (T + 31) >> 5;
    const int nck = T * k;
    // Every request's candidates: expert id, or -1 if pruned.  Staged in shared memory
    // (int16 over the dead aggregates) when they fit, with all of a thread's loads in
    // flight at once; otherwise read from global memory where used.
    int16_t* pk = reinterpret_cast<int16_t*>(A);
    const bool staged = !local && nck <= static_cast<int>(sizeof(sc.A) / sizeof(int16_t));
    if (!local) {  // survivors per expert over every request: a token bitmask per expert
        for (int i = tid; i < E * TW; i += blockDim.x) masks[i] = 0u;
        if (staged) {
            const int nth = blockDim.x;
            for (int c0 = tid; c0 < nck; c0 += 4 * nth) {
                int e4[4];
                uint8_t s4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * nth;
                    e4[u] = c < nck ? __ldcg(&a.idx[c]) : 0;
                    s4[u] = c < nck ? __ldcg(&a.survive[c]) : 0;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u * nth;
                    if (c < nck) pk[c] = static_cast<int16_t>(s4[u] != 0 ? e4[u] : -1);
                }
            }
        }
        __syncthreads();
        for (int c = tid; c < nck; c += blockDim.x) {
            const int e = staged ? pk[c] : (__ldcg(&a.survive[c]) != 0 ? __ldcg(&a.idx[c]) : -1);
            if (e >= 0) {
                const int t = c / k;
                atomicOr(&masks[(t >> 5) * E + e], 1u << (t & 31));
            }
        }
        __syncthreads();
    }
    // one request: every candidate of a kept expert survives, so phase 1's counts and masks
    // hold; several: an expert's survivors are the bits of its mask
    int my_cnt = 0;
    if (tid < E) {
        if (local) {
            my_cnt = keep[tid] ? cnt[tid] : 0;
        } else {
            for (int w = 0; w < TW; ++w) my_cnt += __popc(masks[w * E + tid]);
        }
    }
    const int my_nch = (my_cnt + a.nch - 1) / a.nch;
    // one scan of (chunks << 32 | slots)
    const long long both = block_inclusive_scan<long long>(
        (static_cast<long long>(my_nch) << 32) | static_cast<long long>(my_cnt), sc.wtot64);
    const int slot_end = static_cast<int>(both & 0xffffffffll);
    const int chunk_end = static_cast<int>(both >> 32);
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
    for (int c = tid; c < nck; c += blockDim.x) {
        int e;
        if (local)
            e = csurv[c] != 0 ? cidx[c] : -1;
        else if (staged)
            e = pk[c];
        else
            e = __ldcg(&a.survive[c]) != 0 ? __ldcg(&a.idx[c]) : -1;
        if (e >= 0) {
            const int t = c / k;
            const int w = t >> 5;
            int pos = order[e];
            for (int q = 0; q < w; ++q) pos += __popc(masks[q * E + e]);
            pos += __popc(masks[w * E + e] & ((1u << (t & 31)) - 1u));
            a.slot_of[c] = pos;
            if (stage != nullptr) {
                stage[pos] = t;
                stage[nstage + pos] = e;
            } else {
                a.slot_tok[pos] = t;
                a.slot_exp[pos] = e;
            }
        } else {
            a.slot_of[c] = -1;
        }
    }
    int nsc = 0;
    if (a.has_shared) {
        nsc = (T + a.nch - 1) / a.nch;
        for (int t = tid; t < T; t += blockDim.x) {
            a.slot_sh[t] = NR + t;
            if (stage != nullptr) {
                stage[NR + t] = t;
                stage[nstage + NR + t] = E;
            } else {
                a.slot_tok[NR + t] = t;
                a.slot_exp[NR + t] = E;
            }
        }
        for (int i = tid; i < nsc; i += blockDim.x)
            a.chunks[nrc + i] = make_int4(E, NR + i * a.nch, min(a.nch, T - i * a.nch), 0);
    }
    if (tid == 0) {
        a.plan[0] = nrc;
        a.plan[1] = nsc;
        a.plan[2] = NR + (a.has_shared ? T : 0);
    }
    if (stage != nullptr) {  // the staged slots, in order
        __syncthreads();
        const int ns = NR + (a.has_shared ? T : 0);
        for (int i = tid; i < ns; i += blockDim.x) {
            a.slot_tok[i] = stage[i];
            a.slot_exp[i] = stage[nstage + i];
        }
    }
}

// L2 hints by the extra CTAs of the coreset launch: the union of the experts the
// router picked, then the gate/up weights of its pf_experts lowest ids (the
// expert launch takes the kept experts in id order, so these are the first it
// streams; most candidates are kept).  Hints only: nothing is written.
constexpr int kMaxPrefetchExperts = 64;
__device__ void coreset_prefetch(const CoresetArgs& a, uint32_t* bits) {
    __shared__ int s_pe[kMaxPrefetchExperts];
    __shared__ int s_npe;
    const int tid = threadIdx.x;
    const int E = a.E, nw = (E + 31) >> 5;
    const int npf = min(a.pf_experts, kMaxPrefetchExperts);
    for (int i = tid; i < nw; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int c = tid; c < a.T * a.k; c += blockDim.x) {
        const int e = __ldg(&a.idx[c]);
        if (e >= 0 && e < E) atomicOr(&bits[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (tid < 32) {  // the first npf set bits in id order
        int found = 0;
        for (int w0 = 0; w0 < nw && found < npf; w0 += 32) {
            uint32_t word = w0 + tid < nw ? bits[w0 + tid] : 0u;
            int incl = __popc(word);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += n;
            }
            int pos = found + incl - __popc(word);
            while (word != 0u && pos < npf) {
                const int b = __ffs(word) - 1;
                s_pe[pos++] = (w0 + tid) * 32 + b;
                word &= word - 1u;
            }
            found = min(npf, found + __shfl_sync(0xffffffffu, incl, 31));
        }
        if (tid == 0) s_npe = found;
    }
    __syncthreads();
    const long long lines_per = a.pf_stride >> 7;
    const long long total = lines_per * s_npe;
    const long long stride = static_cast<long long>(gridDim.x - a.R) * blockDim.x;
    const long long g = static_cast<long long>(blockIdx.x - a.R) * blockDim.x + tid;
    for (long long l = g; l < total; l += stride) {
        const int j = static_cast<int>(l / lines_per);
        const char* p = a.pf_base + static_cast<long long>(s_pe[j]) * a.pf_stride + ((l - j * lines_per) << 7);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
    if (a.pf_next != nullptr)
        for (long long l = g; l < (a.pf_next_bytes >> 7); l += stride)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.pf_next + (l << 7)));
}

// grid R (+ pf_ctas hint CTAs), 1024 threads: one CTA per request (see coreset_body).
__global__ void __launch_bounds__(kCoresetThreads) coreset_kernel(CoresetArgs a) {
    extern __shared__ __align__(16) uint8_t coreset_smem[];  // scratch, masks [ceil(T/32)][E], slot staging
    pdl_trigger();
    pdl_wait();
    if (static_cast<int>(blockIdx.x) >= a.R) {
        coreset_prefetch(a, reinterpret_cast<uint32_t*>(coreset_smem));
        return;
    }
    // slot staging only pays when several requests share the plan step
    const int nstage = a.R > 1 ? coreset_stage_slots(a.E, a.T, a.k) : 0;
    int* stage = nstage > 0 ? reinterpret_cast<int*>(coreset_smem + sizeof(CoresetScratch) +
                                                     coreset_masks_bytes(a.E, a.T))
                            : nullptr;
    coreset_body(a, blockIdx.x, a.R, reinterpret_cast<uint32_t*>(coreset_smem + sizeof(CoresetScratch)),
                 *reinterpret_cast<CoresetScratch*>(coreset_smem), stage, nstage);
}

// ---------------------------------------------------------------------------- tensor-core router
namespace cg = cooperative_groups;

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// word i (0..7) of a pair of 16-byte vectors holding 16 bf16
__device__ __forceinline__ uint32_t word8(const uint4& lo, const uint4& hi, int i) {
    const uint4& v = i < 4 ? lo : hi;
    const int j = i & 3;
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// Tensor-core router for bf16 (E % 32 == 0, H % 512 == 0): grid (ceil(T / (8 NT)),
// E / 32), 512 threads.  A CTA computes the logits of 32 experts for 8*NT tokens
// with mma.sync m16n8k16 (bf16 in, fp32 accumulation): warp w takes the 16-expert
// half w & 1 and the K eighth w >> 1, reads its weight rows and token rows straight
// from global memory (16-byte loads; each thread's four K positions per MMA are
// four consecutive elements, the same permutation for both operands, so its
// fragments are plain 16-byte loads), and the eight K partial sums of every logit
// are added in K order through shared memory.  The last CTA of a token tile (self-resetting counter) runs the
// softmax and top-k of the tile's tokens.
constexpr int kRouteTcThreads = 512;
constexpr int kRouteTcExperts = 32;

__host__ __device__ inline size_t route_tc_smem_bytes(int nt, int E) {
    const size_t part = static_cast<size_t>(kRouteTcThreads / 32) * nt * 32 * 4 * sizeof(float);
    const size_t zs = static_cast<size_t>(8) * nt * E * sizeof(float);
    return part > zs ? part : zs;
}

template <int NT>
__global__ void __launch_bounds__(kRouteTcThreads, 1)
    route_tc_kernel(const bf16* __restrict__ x, const bf16* __restrict__ Wr, int ntok, int H, int E, int k,
                    float* __restrict__ logits, int32_t* idx, float* mass, float* gate, int* counters) {
    extern __shared__ __align__(16) uint8_t rtc_smem[];
    float* part = reinterpret_cast<float*>(rtc_smem);  // [16 warps][NT][32 lanes][4]
    __shared__ int last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int eh = warp & 1, q = warp >> 1;
    const int t0 = blockIdx.x * 8 * NT;
    const int e0 = blockIdx.y * kRouteTcExperts;
    const int kspan = H >> 3;
    {  // router weights are never written: hint this CTA's rows before waiting
        const char* w = reinterpret_cast<const char*>(Wr + static_cast<size_t>(e0) * H);
        const int lines = kRouteTcExperts * H * 2 / 128;
        for (int l = threadIdx.x; l < lines; l += kRouteTcThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(w + 128ll * l));
    }
    pdl_trigger();
    pdl_wait();
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) d[nt][r] = 0.f;
    const bf16* w0 = Wr + static_cast<size_t>(e0 + eh * 16 + g) * H;
    const bf16* w1 = w0 + static_cast<size_t>(8) * H;
    const bf16* xr[NT];
    bool ok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int t = t0 + nt * 8 + g;
        ok[nt] = t < ntok;
        xr[nt] = x + static_cast<size_t>(ok[nt] ? t : 0) * H;
    }
#pragma unroll 2
    for (int h0 = q * kspan; h0 < (q + 1) * kspan; h0 += 64) {
        const int hb = h0 + 16 * tig;
        const uint4 a00 = __ldg(reinterpret_cast<const uint4*>(w0 + hb));
        const uint4 a01 = __ldg(reinterpret_cast<const uint4*>(w0 + hb + 8));
        const uint4 a10 = __ldg(reinterpret_cast<const uint4*>(w1 + hb));
        const uint4 a11 = __ldg(reinterpret_cast<const uint4*>(w1 + hb + 8));
        uint4 b0[NT], b1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            b0[nt] = ok[nt] ? __ldcg(reinterpret_cast<const uint4*>(xr[nt] + hb)) : make_uint4(0, 0, 0, 0);
            b1[nt] = ok[nt] ? __ldcg(reinterpret_cast<const uint4*>(xr[nt] + hb + 8)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mma_16816(d[nt], word8(a00, a01, 2 * j), word8(a10, a11, 2 * j), word8(a00, a01, 2 * j + 1),
                          word8(a10, a11, 2 * j + 1), word8(b0[nt], b1[nt], 2 * j), word8(b0[nt], b1[nt], 2 * j + 1));
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4*>(part + ((warp * NT + nt) * 32 + lane) * 4) =
            make_float4(d[nt][0], d[nt][1], d[nt][2], d[nt][3]);
    __syncthreads();
    // element r of lane ln in an MMA tile: expert g + 8*(r >= 2), token 2*tig + (r & 1)
    for (int i = threadIdx.x; i < 2 * NT * 128; i += kRouteTcThreads) {
        const int tile = i >> 7, ln = (i >> 2) & 31, r = i & 3;
        const int h = tile / NT, nt = tile % NT;
        float v = 0.f;
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) v += part[(((qq * 2 + h) * NT + nt) * 32 + ln) * 4 + r];
        const int e = e0 + h * 16 + (ln >> 2) + (r >= 2 ? 8 : 0);
        const int t = t0 + nt * 8 + 2 * (ln & 3) + (r & 1);
        if (t < ntok) logits[static_cast<size_t>(t) * E + e] = v;
    }
    // ---- last CTA of this token tile does the softmax / top-k
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
    const int nt_tok = min(8 * NT, ntok - t0);
    float* zs = reinterpret_cast<float*>(rtc_smem);  // reuse: [8 NT][E]
    const int n = nt_tok * E;
#pragma unroll 4
    for (int i = threadIdx.x; i < n; i += kRouteTcThreads) zs[i] = __ldcg(&logits[static_cast<size_t>(t0) * E + i]);
    __syncthreads();
    for (int tt = warp; tt < nt_tok; tt += kRouteTcThreads / 32)
        topk_one_token(zs + tt * E, E, k, t0 + tt, idx, mass, gate);
}

// The previous layer's combine + RMSNorm and the tensor-core router in one
// cluster launch (bf16 activations, E % 32 == 0, E <= 256, H % 512 == 0, H <= 2560):
// grid (E / 32, ceil(T / 8)), one cluster of E / 32 CTAs per 8-token tile.
// Before waiting for the previous kernel, CTA c copies the router rows of its
// experts 32c .. 32c + 31 into shared memory (cp.async; the weights are never
// written).  It then runs the combine of tokens c, c + CL, ... of the tile (the
// combine kernel's arithmetic, so both write bit-identical rows) and copies each
// normalised row into the shared memory of every CTA of the cluster (distributed
// shared memory); after the cluster barrier it computes the logits of its 32
// experts for the tile from shared memory with route_tc_kernel's fragments and
// K order, and sends each logit to the CTA that takes the token's softmax and
// top-k (token j of the tile: CTA j mod CL).
struct RouteCombineSmem {
    static constexpr int kPart = (kRouteTcThreads / 32) * 32 * 4;  // K partial sums [16 warps][32][4]
    // staged rows: H + 8 elements, so the 8 rows an MMA fragment reads start in distinct banks
    __host__ __device__ static int ld(int H) { return H + 8; }
    __host__ __device__ static int tokens_per_cta(int CL) { return (8 + CL - 1) / CL; }
    __host__ __device__ static size_t w_off() { return 0; }
    __host__ __device__ static size_t x_off(int H) { return static_cast<size_t>(kRouteTcExperts) * ld(H) * 2; }
    __host__ __device__ static size_t part_off(int H) { return x_off(H) + static_cast<size_t>(8) * ld(H) * 2; }
    __host__ __device__ static size_t bytes(int CL, int E, int H) {
        return part_off(H) + sizeof(float) * (kPart + static_cast<size_t>(tokens_per_cta(CL)) * E) +
               sizeof(int) * 2 * 33 + sizeof(float) * (2 * 33 + 2 * 9);
    }
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

// Writes each normalised 4-column group of token row j of the tile into the staged x
// tile of every CTA of the cluster.
struct ClusterRowSink {
    bf16* xs;  // this CTA's staged tile [8][ld]
    int row_off;
    int CL;
    __device__ __forceinline__ void operator()(int c, float4 n) const {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(n.x, n.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(n.z, n.w);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        cg::cluster_group cluster = cg::this_cluster();
        for (int r = 0; r < CL; ++r)
            *reinterpret_cast<uint2*>(cluster.map_shared_rank(xs, r) + row_off + c) = u;
    }
};

__global__ void __launch_bounds__(kRouteTcThreads, 1) route_combine_kernel(RouteCombineArgs a) {
    extern __shared__ __align__(16) uint8_t rc_smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int CL = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int eh = warp & 1, q = warp >> 1;
    const int T = a.T, H = a.H, E = a.E, k = a.k;
    const int LD = RouteCombineSmem::ld(H);
    const int t0 = blockIdx.y * 8;
    const int e0 = rank * kRouteTcExperts;
    const int kspan = H >> 3;
    const int TPC = RouteCombineSmem::tokens_per_cta(CL);
    const int grp = threadIdx.x >> 8;  // combine: two groups of 256 threads
    bf16* ws = reinterpret_cast<bf16*>(rc_smem + RouteCombineSmem::w_off());   // [32][LD] router rows
    bf16* xs = reinterpret_cast<bf16*>(rc_smem + RouteCombineSmem::x_off(H));  // [8][LD] the tile's x rows
    float* part = reinterpret_cast<float*>(rc_smem + RouteCombineSmem::part_off(H));
    float* zs = part + RouteCombineSmem::kPart;  // [TPC][E] logits of this CTA's tokens
    int* c_slot = reinterpret_cast<int*>(zs + static_cast<size_t>(TPC) * E) + 33 * grp;
    float* c_g = reinterpret_cast<float*>(reinterpret_cast<int*>(zs + static_cast<size_t>(TPC) * E) + 66) + 33 * grp;
    float* c_red = reinterpret_cast<float*>(reinterpret_cast<int*>(zs + static_cast<size_t>(TPC) * E) + 66) + 66 +
                   9 * grp;
    {  // router weights are never written: stage this CTA's rows before waiting
        const int vec = H >> 3;  // 16-byte pieces per row
        const bf16* w = a.Wr + static_cast<size_t>(e0) * H;
        for (int i = threadIdx.x; i < kRouteTcExperts * vec; i += kRouteTcThreads) {
            const int r = i / vec, c = (i - r * vec) << 3;
            cp_async16(ws + r * LD + c, w + static_cast<size_t>(r) * H + c);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    pdl_trigger();
    // One pass of the combine loop per group (E >= 128): its token's slots and gates, final once
    // the previous layer's coreset set its flag, are read while the previous kernel still runs.
    bool pre = false;
    if (a.mode == 1 && a.plan_flag != nullptr && 2 * CL >= 8) {
        __shared__ int s_pre;
        if (threadIdx.x == 0) s_pre = wait_at_least(a.plan_flag, a.plan_value, a.timeout_ns);
        __syncthreads();
        pre = s_pre != 0;
        if (pre) {
            const int j = rank + CL * grp;
            combine_load_slots((j < 8 && t0 + j < T) ? t0 + j : -1, k, a.slot_of, a.slot_sh, a.gate_rr_prev,
                               a.has_shared, c_slot, c_g);
        }
    }
    cluster.sync();  // every CTA of the cluster runs before any writes into another's shared memory
    pdl_wait();
    // 1. combine of this CTA's tokens of the tile; each normalised row also goes to the
    //    x tile of every CTA of the cluster (rows past the block's last token are zero)
    if (CL >= 8 && H <= 2048) {
        // one token per CTA: both groups of 256 threads take its row (all loads in flight at once)
        const int t = t0 + rank < T ? t0 + rank : -1;
        const ClusterRowSink sink{xs, rank * LD, CL};
        int* s0 = c_slot - 33 * grp;  // group 0's scratch (the preload filled it)
        float* g0 = c_g - 33 * grp;
        float* r0 = c_red - 9 * grp;
        if (a.mode == 1)
            combine_row_pair<bf16, 1>(t, H, k, a.y, a.slot_of, a.slot_sh, a.gate_rr_prev, a.has_shared, nullptr,
                                      a.hres, a.x, s0, g0, r0, part, sink, pre);
        else
            combine_row_pair<bf16, 2>(t, H, k, nullptr, nullptr, nullptr, nullptr, 0, a.h_in, a.hres, a.x, s0, g0, r0,
                                      part, sink, false);
        if (t < 0)
            for (int c = threadIdx.x * 4; c < H; c += 4 * kRouteTcThreads) sink(c, make_float4(0.f, 0.f, 0.f, 0.f));
    } else {
    for (int j0 = 0; j0 < 8; j0 += 2 * CL) {
        const int j = j0 + rank + CL * grp;
        const int t = (j < 8 && t0 + j < T) ? t0 + j : -1;
        const ClusterRowSink sink{xs, j * LD, CL};
        if (a.mode == 1)
            combine_row<bf16, 1>(t, H, k, a.y, a.slot_of, a.slot_sh, a.gate_rr_prev, a.has_shared, nullptr, a.hres,
                                 a.x, nullptr, nullptr, c_slot, c_g, c_red, sink, pre);
        else
            combine_row<bf16, 2>(t, H, k, nullptr, nullptr, nullptr, nullptr, 0, a.h_in, a.hres, a.x, nullptr,
                                 nullptr, c_slot, c_g, c_red, sink);
        if (j < 8 && t < 0)
            for (int c = (threadIdx.x & 255) * 4; c < H; c += 1024) sink(c, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    cluster.sync();  // the tile's x rows and this CTA's router rows are in shared memory
    // 2. logits of experts e0 .. e0 + 31 for the tile (route_tc_kernel's fragments and K order)
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const bf16* w0 = ws + (eh * 16 + g) * LD;
    const bf16* w1 = w0 + 8 * LD;
    const bf16* xr = xs + g * LD;
#pragma unroll 4
    for (int h0 = q * kspan; h0 < (q + 1) * kspan; h0 += 64) {
        const int hb = h0 + 16 * tig;
        const uint4 a00 = *reinterpret_cast<const uint4*>(w0 + hb);
        const uint4 a01 = *reinterpret_cast<const uint4*>(w0 + hb + 8);
        const uint4 a10 = *reinterpret_cast<const uint4*>(w1 + hb);
        const uint4 a11 = *reinterpret_cast<const uint4*>(w1 + hb + 8);
        const uint4 b0 = *reinterpret_cast<const uint4*>(xr + hb);
        const uint4 b1 = *reinterpret_cast<const uint4*>(xr + hb + 8);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            mma_16816(d, word8(a00, a01, 2 * jj), word8(a10, a11, 2 * jj), word8(a00, a01, 2 * jj + 1),
                      word8(a10, a11, 2 * jj + 1), word8(b0, b1, 2 * jj), word8(b0, b1, 2 * jj + 1));
    }
    *reinterpret_cast<float4*>(part + (warp * 32 + lane) * 4) = make_float4(d[0], d[1], d[2], d[3]);
    __syncthreads();
    // 3. the eight K splits added in K order; each logit to the CTA that takes its token
    for (int i = threadIdx.x; i < 2 * 128; i += kRouteTcThreads) {
        const int h = i >> 7, ln = (i >> 2) & 31, r = i & 3;
        float v = 0.f;
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) v += part[((qq * 2 + h) * 32 + ln) * 4 + r];
        const int e = e0 + h * 16 + (ln >> 2) + (r >= 2 ? 8 : 0);
        const int j = 2 * (ln & 3) + (r & 1);
        if (t0 + j < T) {
            if (a.logits != nullptr) a.logits[static_cast<size_t>(t0 + j) * E + e] = v;
            cluster.map_shared_rank(zs, j % CL)[(j / CL) * E + e] = v;
        }
    }
    cluster.sync();  // every logit of this CTA's tokens has arrived
    // 4. softmax and top-k, one warp per token
    for (int jj = warp; jj < TPC; jj += kRouteTcThreads / 32) {
        const int j = rank + CL * jj;
        if (j < 8 && t0 + j < T) topk_one_token(zs + static_cast<size_t>(jj) * E, E, k, t0 + j, a.idx, a.mass, a.gate);
    }
}

// 8 bf16 -> 8 f16 (round to nearest even; exact unless below f16's normal range)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        const __half2 h = __floats2half2_rn(f.x, f.y);
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// One CTA per slot: xp[slot] = x[slot_tok[slot]] (TO_F16: bf16 rows stored as f16,
// the activation type of the FP8 expert launch); CTA 0 also zeroes the expert
// launch's chunk counters and, if given, release-stores flag_value into *flag
// (the coreset before it has completed: its plan, slots and gates are final).
template <bool TO_F16>
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ x, int row_vec,
                                                     const int32_t* __restrict__ slot_tok, const int* __restrict__ plan,
                                                     uint4* __restrict__ xp, int* __restrict__ done, int n_done,
                                                     int* __restrict__ flag, int flag_value) {
    const int slot = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (flag != nullptr && blockIdx.x == 0 && threadIdx.x == 0) release_store_gpu(flag, flag_value);
    if (done != nullptr && blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_done; i += blockDim.x) done[i] = 0;
    if (slot < plan[2]) {
        const int t = slot_tok[slot];
        for (int i = threadIdx.x; i < row_vec; i += blockDim.x) {
            const uint4 v = x[static_cast<size_t>(t) * row_vec + i];
            xp[static_cast<size_t>(slot) * row_vec + i] = TO_F16 ? bf16x8_to_f16x8(v) : v;
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
    static int done_bf16[64] = {}, done_f32[64] = {}, done_tc[2][64] = {};
    if (dtype == MOESTEP_BF16 && E % kRouteTcExperts == 0 && H % 512 == 0 && E <= 1024) {
        // 8*NT tokens per CTA: 16 above 256 tokens (measured faster at 512 tokens than 8 or 32), else 8
        const int nt = T > 256 ? 2 : 1;
        const dim3 g((T + 8 * nt - 1) / (8 * nt), E / kRouteTcExperts);
        const size_t sm = route_tc_smem_bytes(nt, E);
        const bf16* xb = static_cast<const bf16*>(x);
        const bf16* wb = static_cast<const bf16*>(Wr);
        if (nt == 2) {
            if ((e = ensure_smem(route_tc_kernel<2>, sm, done_tc[1])) != cudaSuccess) return e;
            return launch_pdl(route_tc_kernel<2>, g, dim3(kRouteTcThreads), sm, s, xb, wb, T, H, E, k, logits, idx,
                              mass, gate, counters);
        }
        if ((e = ensure_smem(route_tc_kernel<1>, sm, done_tc[0])) != cudaSuccess) return e;
        return launch_pdl(route_tc_kernel<1>, g, dim3(kRouteTcThreads), sm, s, xb, wb, T, H, E, k, logits, idx, mass,
                          gate, counters);
    }
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

int coreset_smem_bytes(int E, int T) { return static_cast<int>(sizeof(CoresetScratch) + coreset_masks_bytes(E, T)); }

cudaError_t launch_coreset(const CoresetArgs& a, cudaStream_t s) {
    const size_t smem = coreset_smem_bytes(a.E, a.T) +
                        (a.R > 1 ? static_cast<size_t>(coreset_stage_slots(a.E, a.T, a.k)) * 8 : 0);
    static int done[64] = {};
    cudaError_t e = ensure_smem(coreset_kernel, smem, done);
    if (e != cudaSuccess) return e;
    const int helpers = (a.pf_base != nullptr && a.pf_experts > 0) ? a.pf_ctas : 0;
    return launch_pdl(coreset_kernel, dim3(a.R + helpers), dim3(kCoresetThreads), smem, s, a);
}

cudaError_t launch_gather(int dtype, const void* x, int H, const int32_t* slot_tok, const int* plan, int max_slots,
                          void* xp, int* done, int n_done, int* flag, int flag_value, cudaStream_t s) {
    const int row_vec = H * (dtype == MOESTEP_F32 ? 4 : 2) / 16;
    if (dtype == MOESTEP_FP8)
        return launch_pdl(gather_kernel<true>, dim3(max_slots), dim3(256), 0, s, static_cast<const uint4*>(x),
                          row_vec, slot_tok, plan, static_cast<uint4*>(xp), done, n_done, flag, flag_value);
    return launch_pdl(gather_kernel<false>, dim3(max_slots), dim3(256), 0, s, static_cast<const uint4*>(x), row_vec,
                      slot_tok, plan, static_cast<uint4*>(xp), done, n_done, flag, flag_value);
}

int route_combine_eligible(int act_dtype, int T, int H, int E, int k) {
    if (act_dtype != MOESTEP_BF16 || T < 1 || T > 256 || k < 1 || k > 32) return 0;
    if (E % kRouteTcExperts != 0 || E > 8 * kRouteTcExperts || H % 512 != 0) return 0;
    return RouteCombineSmem::bytes(E / kRouteTcExperts, E, H) <= 225 * 1024 ? 1 : 0;
}

cudaError_t launch_route_combine(const RouteCombineArgs& a, cudaStream_t s) {
    const int CL = a.E / kRouteTcExperts;
    const size_t smem = RouteCombineSmem::bytes(CL, a.E, a.H);
    static int done[64] = {};
    cudaError_t e = ensure_smem(route_combine_kernel, smem, done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(CL, (a.T + 7) / 8);
    cfg.blockDim = dim3(kRouteTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_launch_pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, route_combine_kernel, a);
}

}  // namespace moestep
