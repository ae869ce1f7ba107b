// Grouped expert GEMM on tcgen05 tensor cores, weights streamed by TMA.
//
// One persistent CTA per SM walks a list of work units.  A unit is one
// 128-row tile of one weight matrix (an expert's gate/up pair, an expert's
// down projection, or a block of LM-head vocabulary rows) applied to the
// tokens that use it.  The expert launch holds the whole routed + shared FFN:
// every gate/up unit first, then every down unit; a down unit's producer
// waits (bounded) on a per-chunk counter that the chunk's gate/up epilogues
// raise after their SwiGLU rows are stored, so the gate/up tail overlaps the
// first down units instead of idling before a second launch.  Each CTA issues
// all of its gate/up units before any down unit, and its epilogue drains them
// without waiting on the producer, so the counters always complete.  The
// operands are swapped so the weight rows are the MMA's
// M = 128 and the block tokens are its N (16..NCH), because a 32-token block
// gives every expert only a handful of tokens.  Each weight element is read
// from HBM exactly once per block ([AIT 五]: the block's speed-up comes from
// reusing every loaded weight for all of its tokens).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: fills a ring of STAGES shared-memory stages
//               (A: two 64x64 bf16 boxes = 16 KiB, B: N rows x 64 bf16),
//               all in the 128-byte swizzled layout.
//   warp 1      MMA issuer: 4 x tcgen05.mma (K = 16 each) per stage into a
//               TMEM accumulator; double-buffered accumulators let the
//               epilogue of one unit overlap the main loop of the next.
//   warps 2-5   epilogue: tcgen05.ld of the 128 x N fp32 accumulator, then
//                 gate/up: act = silu(gate) * up, stored as bf16 (gate and up
//                          rows of one intermediate index are adjacent in the
//                          weight layout, so the pair meets in one shuffle)
//                 down:    y (fp32) per token slot
//                 LM head: per position and 32-row slice: (max, argmax, sum exp)
// The epilogue warps never wait on each other, and every wait is bounded
// (timeout -> error word, orderly teardown), so no wait can hang the GPU.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

namespace moestep {
namespace {

constexpr int kThreads = 192;
constexpr uint64_t kTeardownNs = 1000000000ull;  // fixed limit for draining in-flight copies/MMAs
constexpr int kABytes = 16384;            // 128 rows x 64 bf16
constexpr int kBoxBBytes = 16 * 128;      // 16 rows x 64 bf16
constexpr int kSmemBudget = 232448 - 1024 - 512;

__host__ __device__ constexpr int stage_bytes(int nch) { return kABytes + nch * 128; }
__host__ __device__ constexpr int num_stages(int nch) {
    return (kSmemBudget / stage_bytes(nch)) > 10 ? 10 : (kSmemBudget / stage_bytes(nch));
}
__host__ __device__ constexpr int smem_bytes(int nch) { return num_stages(nch) * stage_bytes(nch) + 512 + 1024; }

struct Unit {
    int kb, rowA0, rowA1, slot0, n, mt, c;
    bool shared, dn;
};

template <int MODE, int NCH>
__device__ __forceinline__ Unit decode_unit(int u, const GemmParams& p, int nrc, int nsc) {
    Unit w;
    if (MODE == kLmHead) {
        const int mt = u / p.lm_chunks;
        const int c = u - mt * p.lm_chunks;
        w.mt = mt;
        w.rowA0 = mt * 128;
        w.rowA1 = w.rowA0 + 64;
        w.kb = p.routed_kb;
        w.shared = false;
        w.dn = false;
        w.c = c;
        w.slot0 = c * NCH;
        w.n = min(NCH, p.n_pos - w.slot0);
        return w;
    }
    int rt = p.routed_tiles, st = p.shared_tiles, rkb = p.routed_kb, skb = p.shared_kb, rpe = p.rows_per_expert;
    bool dn = MODE == kDown;
    if (MODE == kExperts) {
        const int n_gu = nrc * p.routed_tiles + nsc * p.shared_tiles;
        if (u >= n_gu) {  // second half of the unit list: down projections
            u -= n_gu;
            dn = true;
            rt = p.dn_routed_tiles;
            st = p.dn_shared_tiles;
            rkb = p.dn_routed_kb;
            skb = p.dn_shared_kb;
            rpe = p.dn_rows_per_expert;
        }
    }
    const int routed_units = nrc * rt;
    int c, mt;
    if (u < routed_units) {
        c = u / rt;
        mt = u - c * rt;
        w.shared = false;
    } else {
        const int v = u - routed_units;
        const int cs = v / st;
        mt = v - cs * st;
        c = nrc + cs;
        w.shared = true;
    }
    const int4 ch = p.chunks[c];
    w.slot0 = ch.y;
    w.n = ch.z;
    w.mt = mt;
    w.c = c;
    w.dn = dn;
    const int base = (w.shared ? 0 : ch.x * rpe) + mt * p.tile_rows;
    w.rowA0 = base;
    w.rowA1 = base + 64;
    w.kb = w.shared ? skb : rkb;
    return w;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Wait (bounded, like the mbarrier waits) until *ctr >= need; then order this
// thread's later TMA (async-proxy) reads after what the counter published.
__device__ __forceinline__ bool wait_count(const int* ctr, int need, volatile int* abort, uint64_t limit_ns) {
    if (ld_acquire_gpu(ctr) < need) {
        const uint64_t t0 = tc::globaltimer_ns();
        for (;;) {
            if (*abort) return false;
            if (tc::globaltimer_ns() - t0 >= limit_ns) return false;
            __nanosleep(100);
            if (ld_acquire_gpu(ctr) >= need) break;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

// Where a bounded wait gave up: the first CTA to time out writes
// {role, block, unit, k-block, stage, phase, units, tokens} after the error word.
__device__ __forceinline__ void record_timeout(int* err, int role, int u, int kb, int stage, uint32_t phase,
                                               int n_units, int n) {
    if (err == nullptr) return;
    if (atomicCAS(err + 8, 0, role) == 0) {
        err[9] = blockIdx.x;
        err[10] = u;
        err[11] = kb;
        err[12] = stage;
        err[13] = static_cast<int>(phase);
        err[14] = n_units;
        err[15] = n;
    }
}

template <int MODE, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TensorMaps maps, const GemmParams p) {
    constexpr int STAGES = num_stages(NCH);
    constexpr int SB = stage_bytes(NCH);
    constexpr uint32_t TMEM_COLS = (2 * NCH < 32) ? 32u : static_cast<uint32_t>(2 * NCH);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * SB);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* fin = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(fin + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int* zero_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(fin, 1);
        *abort_flag = 0;
        *zero_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&maps.a[0]);
        tc::prefetch_tmap(&maps.b[0]);
        if (MODE != kLmHead) {
            tc::prefetch_tmap(&maps.a[1]);
            if (MODE == kExperts) {
                tc::prefetch_tmap(&maps.a[2]);
                tc::prefetch_tmap(&maps.a[3]);
                tc::prefetch_tmap(&maps.b[1]);
            }
        }
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // prologue done: let the next kernel start, then wait for the work plan / inputs
    pdl_trigger();
    pdl_wait();
    int nrc = 0, nsc = 0, n_units;
    if (MODE == kLmHead) {
        n_units = p.lm_chunks * p.lm_tiles;
    } else {
        nrc = p.plan[0];
        nsc = p.plan[1];
        n_units = nrc * p.routed_tiles + nsc * p.shared_tiles;
        if (MODE == kExperts) n_units += nrc * p.dn_routed_tiles + nsc * p.dn_shared_tiles;
    }
    volatile int* abortv = abort_flag;
    const uint64_t tmo = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol = tc::policy_evict_first();
        uint32_t issued = 0, issued_parity = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int nb = (w.n + 15) >> 4;
            const CUtensorMap* mA = &maps.a[(w.dn && MODE == kExperts ? 2 : 0) + (w.shared ? 1 : 0)];
            const CUtensorMap* mB = &maps.b[w.dn && MODE == kExperts ? 1 : 0];
            if (MODE == kExperts && w.dn) {
                // the SwiGLU rows of this chunk come from gate/up units of other CTAs
                int good = 1;
                if (lane == 0)
                    good = wait_count(&p.done[w.c], 4 * (w.shared ? p.shared_tiles : p.routed_tiles), abortv, tmo);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 6, u, -1, -1, 0, n_units, w.n);
                    break;
                }
            }
            for (int kb = 0; kb < w.kb; ++kb) {
                int good = 1;
                if (lane == 0) {
                    good = tc::mbar_wait(&empty[stage], phase ^ 1u, abortv, tmo);
                    if (good) {
                        uint8_t* sa = smem + stage * SB;
                        tc::mbar_arrive_expect_tx(&full[stage], kABytes + nb * kBoxBBytes);
                        tc::tma_load_2d_hint(sa, mA, &full[stage], kb * 64, w.rowA0, pol);
                        tc::tma_load_2d_hint(sa + kABytes / 2, mA, &full[stage], kb * 64, w.rowA1, pol);
                        for (int b = 0; b < nb; ++b)
                            tc::tma_load_2d(sa + kABytes + b * kBoxBBytes, mB, &full[stage], kb * 64,
                                            w.slot0 + 16 * b);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                }
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 1, u, kb, stage, phase, n_units, w.n);
                    break;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) {
            if (!ok) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeoutProducer);
            }
            // let every copy this CTA issued land before shared memory is released
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) tc::mbar_wait(&full[s], (issued_parity >> s) & 1u, zero_flag, kTeardownNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int it = 0;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++it) {
            const Unit w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int buf = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            const int N = ((w.n + 15) >> 4) << 4;
            const uint32_t idesc = tc::idesc_bf16(128, N);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * NCH);
            int good = 1;
            if (lane == 0) good = tc::mbar_wait(&tempty[buf], aph ^ 1u, abortv, tmo);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                ok = false;
                if (lane == 0) record_timeout(p.err, 2, u, -1, buf, aph, n_units, w.n);
                break;
            }
            tc::fence_after_sync();
            for (int kb = 0; kb < w.kb; ++kb) {
                good = 1;
                if (lane == 0) {
                    good = tc::mbar_wait(&full[stage], phase, abortv, tmo);
                    if (good) {
                        tc::fence_after_sync();
                        const uint32_t sa = tc::smem_addr(smem + stage * SB);
                        const uint32_t sb = sa + kABytes;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc::mma_bf16(d_tmem, tc::sdesc_k_sw128(sa + 32 * k), tc::sdesc_k_sw128(sb + 32 * k),
                                         idesc, (kb | k) != 0);
                        tc::mma_commit(&empty[stage]);
                    }
                }
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 3, u, kb, stage, phase, n_units, w.n);
                    break;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (lane == 0) tc::mma_commit(&tfull[buf]);
            __syncwarp();
        }
        if (lane == 0) {
            if (!ok) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeoutMma);
            }
            // every MMA issued here has finished before TMEM and shared memory are released
            tc::mma_commit(fin);
            tc::mbar_wait(fin, 0, zero_flag, kTeardownNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int sp = warp & 3;  // TMEM sub-partition this warp may access: lanes 32*sp .. 32*sp+31
        int it = 0;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
            const Unit w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int buf = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            int good = tc::mbar_wait(&tfull[buf], aph, abortv, tmo);
            good = __all_sync(0xffffffffu, good);
            if (!good) {
                if (lane == 0) {
                    *abort_flag = 1;
                    record_error(p.err, kErrTimeoutEpilogue);
                    record_timeout(p.err, 4 + sp, u, -1, buf, aph, n_units, w.n);
                }
                break;
            }
            tc::fence_after_sync();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(32 * sp) << 16) + static_cast<uint32_t>(buf * NCH);
            const int L = 32 * sp + lane;  // accumulator row held by this thread
            for (int c0 = 0; c0 < w.n; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tb + c0, v);
                const int cnt = min(32, w.n - c0);
                if (MODE == kGateUp || (MODE == kExperts && !w.dn)) {
                    // rows alternate gate / up of one intermediate index: partner lane holds the other half
                    bf16* act = static_cast<bf16*>(p.out);
                    const int i = w.mt * 64 + (L >> 1);
                    const bool is_gate = (lane & 1) == 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float o = __shfl_xor_sync(0xffffffffu, v[j], 1);
                        if (j < cnt && (j & 1) == (lane & 1)) {
                            const float g = is_gate ? v[j] : o;
                            const float up = is_gate ? o : v[j];
                            act[static_cast<size_t>(w.slot0 + c0 + j) * p.out_ld + i] =
                                __float2bfloat16_rn(silu_f(g) * up);
                        }
                    }
                } else if (MODE == kDown || MODE == kExperts) {
                    float* y = static_cast<float*>(MODE == kExperts ? p.out2 : p.out);
                    const int ld = MODE == kExperts ? p.out2_ld : p.out_ld;
                    const int h = w.mt * 128 + L;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < cnt) y[static_cast<size_t>(w.slot0 + c0 + j) * ld + h] = v[j];
                } else {
                    // per (position, 32-row slice): max logit, its lowest row, sum of exp(l - max)
                    const int row = w.mt * 128 + L;
                    const bool valid = row < p.V;
                    float mm = -INFINITY, ss = 0.f;
                    int aa = 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j < cnt) {
                            const float l = valid ? v[j] * p.scale : -INFINITY;
                            if (p.logits != nullptr && valid)
                                p.logits[static_cast<size_t>(w.slot0 + c0 + j) * p.V + row] = l;
                            float m = l;
                            int a = row;
                            warp_argmax(m, a);
                            const float s = (m == -INFINITY) ? 0.f : warp_sum(valid ? __expf(l - m) : 0.f);
                            if (lane == j) {
                                mm = m;
                                aa = a;
                                ss = s;
                            }
                        }
                    }
                    if (lane < cnt) {
                        const size_t o = static_cast<size_t>(w.mt * 4 + sp) * p.n_pos + (w.slot0 + c0 + lane);
                        p.pmax[o] = mm;
                        p.parg[o] = aa;
                        p.psum[o] = ss;
                    }
                }
            }
            if (MODE == kExperts && !w.dn) {
                // publish this warp's SwiGLU rows to the down units of the chunk (any CTA)
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(&p.done[w.c], 1);
            }
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[buf]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int MODE, int NCH>
cudaError_t launch_one(const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s) {
    constexpr int bytes = smem_bytes(NCH);
    static int done[64] = {};
    cudaError_t e = ensure_smem(tc_gemm_kernel<MODE, NCH>, bytes, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_gemm_kernel<MODE, NCH>, dim3(grid), dim3(kThreads), bytes, s, maps, p);
}

template <int MODE>
cudaError_t launch_mode(int nch, const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s) {
    switch (nch) {
        case 32: return launch_one<MODE, 32>(maps, p, grid, s);
        case 64: return launch_one<MODE, 64>(maps, p, grid, s);
        case 128: return launch_one<MODE, 128>(maps, p, grid, s);
        case 256: return launch_one<MODE, 256>(maps, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int tc_gemm_smem_bytes(int nch) { return smem_bytes(nch); }

cudaError_t launch_tc_gemm(int mode, int nch, const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s) {
    switch (mode) {
        case kExperts: return launch_mode<kExperts>(nch, maps, p, grid, s);
        case kLmHead: return launch_mode<kLmHead>(nch, maps, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moestep
