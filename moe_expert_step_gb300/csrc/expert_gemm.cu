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
//
// FP8 E4M3 weights (kExpertsF8, 512 threads), K blocks of 128:
//   warp 0      TMA producer of the A ring: 128 x 128-byte FP8 weight tiles
//               (128-byte swizzle), one per K block; a slot is free again as
//               soon as its converters have read it into registers.
//   warp 15     TMA producer of the B ring: each K block's token rows (f16) in
//               an entry of 1, 2 or 4 consecutive 4 KiB granules of 16 tokens
//               (one copy per K half), so one MMA covers all of a unit's tokens;
//               a ring of 12 granules (24 at 64-token chunks), so the rows land
//               well before their stage comes round; an entry is free again at
//               its MMAs' commit.
//   warps 6-13  converters, two groups of four on alternate K blocks: each
//               warp turns the 32 tile rows of its TMEM lane quarter into f16
//               (exact, one conversion instruction per pair) and stores them with tcgen05.st
//               as the MMA's A operand in tensor memory.
//   warps 1, 14 MMA issuers on one lane each, the even and the odd K blocks of
//               every unit (eight MMAs per wait and commit) into their own
//               accumulators (the issue cost is per issuing thread).
//   warps 2-5   epilogue as above, adding the two accumulators and applying
//               each weight row's scale; SwiGLU rows stored as f16.
// The epilogue warps never wait on each other, and every wait is bounded
// (timeout -> error word, orderly teardown), so no wait can hang the GPU.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

#include <type_traits>

namespace moestep {
namespace {

constexpr int kThreads = 192;
constexpr int kThreadsF8 = 512;  // + eight converter warps (two groups of four), a second MMA warp and a
                                 // second TMA warp
constexpr int kMmaWarp2 = 14;    // FP8: issues each unit's odd K blocks into its own accumulator
constexpr int kTmaWarp2 = 15;    // FP8: loads the token rows (B ring); warp 0 loads the weight tiles
constexpr uint64_t kTeardownNs = 1000000000ull;  // fixed limit for draining in-flight copies/MMAs
constexpr int kABytes = 16384;            // 128 rows x 64 bf16
constexpr int kBoxBBytes = 16 * 128;      // 16 rows x 64 bf16
constexpr int kSmemBudget = 232448 - 1024 - 512;

__host__ __device__ constexpr int stage_bytes(int nch) { return kABytes + nch * 128; }
__host__ __device__ constexpr int num_stages(int nch) {
    return (kSmemBudget / stage_bytes(nch)) > 11 ? 11 : (kSmemBudget / stage_bytes(nch));
}
__host__ __device__ constexpr int smem_bytes(int nch) { return num_stages(nch) * stage_bytes(nch) + 512 + 1024; }

// FP8 weights: shared memory holds two rings that two TMA warps fill far ahead.  The
// A ring holds 128 x 128 E4M3 weight tiles (a K block of 128); a tile's slot is
// released as soon as its converters hold it in registers, so the weight stream does
// not wait out the MMAs.  The converted f16 A operands live in tensor memory
// (f8_a_stages stages of 64 columns from column f8_a_column), so the conversion adds no
// shared-memory traffic beyond reading the FP8 tile once.  The B ring holds the K blocks'
// token rows (the MMA's B operand, read in place) far enough ahead that a stage's round
// trip (freed, converted, multiplied, committed) does not include a load of its token
// rows; a stage's converters arrive only once its token rows have landed, so an MMA warp
// waits once per K block it takes (eight MMAs).  The ring is sized in 16-token granules,
// so a unit with few tokens (the usual case: a handful per expert) takes one granule per
// K block and the shared memory left over holds more weight tiles in flight.
constexpr int kF8Tile = 16384;    // 128 rows x 128 E4M3 bytes
// f16 A operands in TMEM after the accumulators (two MMA warps x two buffers x NCH columns):
// as many 64-column stages as the 512 columns leave, an even number (each converter group owns
// every other stage)
__host__ __device__ constexpr int f8_a_column(int nch) { return 4 * nch; }
__host__ __device__ constexpr int f8_a_stages(int nch) { return ((512 - 4 * nch) / 64) & ~1; }
// A granule: 16 token rows of one K block of 128, in two halves of 2 KiB (K 0..63 and
// K 64..127, 128-byte swizzle) kept in two half-rings, so that n consecutive granules form
// one B operand of 16 n rows per half.
constexpr int kGranule = 4096;
constexpr int kGranuleHalf = kGranule / 2;
__host__ __device__ constexpr int f8_b_granules(int nch) { return nch <= 32 ? 12 : 24; }
static_assert(f8_b_granules(32) % 4 == 0 && f8_b_granules(64) % 4 == 0, "whole entries of up to 4 granules");
// The rest of shared memory, an even number of slots (so that each A slot is always read by the
// same converter group).  At 64-token chunks the token-row ring takes 24 granules (eight K blocks
// of 48-64 tokens ahead) and leaves 8 weight slots.
__host__ __device__ constexpr int f8_a_slots(int nch) {
    return ((kSmemBudget - 1024 - f8_b_granules(nch) * kGranule) / kF8Tile) & ~1;
}
constexpr int kF8BarrierBytes = 2048;  // the FP8 launch's barriers and unit ring
static_assert(f8_a_slots(32) == 10 && f8_a_slots(64) == 8, "FP8 weight-tile ring");
static_assert(f8_a_stages(32) == 6 && f8_a_stages(64) == 4, "FP8 A stages in tensor memory");
__host__ __device__ constexpr int smem_bytes_f8(int nch) {
    return f8_a_slots(nch) * kF8Tile + f8_b_granules(nch) * kGranule + kF8BarrierBytes + 1024;
}
static_assert(smem_bytes_f8(32) <= 232448 && smem_bytes_f8(64) <= 232448, "FP8 shared memory");

struct Unit {
    int kb, rowA0, rowA1, slot0, n, mt, c;
    bool shared, dn;
};

// Token-row entries of the FP8 launch.  Every role that touches the granule ring walks the
// same K blocks in the same order and places them alike: each K block of a unit with n tokens
// takes an entry of granules_for(n) granules (a power of two; one copy per half-ring of that
// many 16-row granules), a unit's first entry starts at the ring position rounded up to a
// multiple of that (the ring's size is a multiple of 4, so no entry runs past its end) and the
// unit's later entries follow one another around the ring.  An entry's copies complete on its
// first granule's full barrier; the MMAs that read it release every granule of it.  Granules
// that an entry skips sit out that lap; the roles that wait on the ring's barriers keep the use
// counts mod 2 (per granule for the empty barriers, per first granule for the full ones).
__device__ __forceinline__ int granules_for(int n) {
    const int q = (n + 15) >> 4;
    return q <= 1 ? 1 : q <= 2 ? 2 : 4;
}
template <int G>
__device__ __forceinline__ int granule_start(int pos, int nbp) {
    const int p = (pos + nbp - 1) & ~(nbp - 1);
    return p >= G ? 0 : p;
}

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
    if (MODE == kExperts || MODE == kExpertsF8) {
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
    // Within each half the routed units come first, except in the FP8 launch: there the shared
    // expert's units (all of the block's tokens, so the widest token-row entries) come first, so
    // that they run alongside routed units rather than at the end of the launch.
    constexpr bool kSharedFirst = MODE == kExpertsF8;
    const int routed_units = nrc * rt;
    const int shared_units = nsc * st;
    int c, mt;
    const bool shared = kSharedFirst ? u < shared_units : u >= routed_units;
    if (!shared) {
        const int v = kSharedFirst ? u - shared_units : u;
        c = v / rt;
        mt = v - c * rt;
        w.shared = false;
    } else {
        const int v = kSharedFirst ? u : u - routed_units;
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

// Units of the expert launches are handed out at run time: a CTA's first unit is its block
// index (no counter round trip at the launch's start); the (weight) producer warp takes
// each later unit index from a global counter (so CTAs that stream faster take more units and
// the launch ends together) and publishes it in a ring of kUnitQ shared-memory entries that
// every other role's warps read in the same order (bf16: the MMA warp and the four epilogue
// warps; FP8 also the token-row producer, the second MMA warp and the eight converters).  Gate/up units have the lower
// indices, so every gate/up unit is taken before any down unit, as with the static order.
constexpr int kUnitQ = 8;
constexpr int kUnitReaders = 5;     // bf16: MMA + 4 epilogue warps
constexpr int kUnitReadersF8 = 15;  // FP8: B producer, 2 MMA, 4 epilogue and 8 converter warps
struct UnitRing {
    uint64_t* full;   // [kUnitQ] the producer wrote the entry (count 1)
    uint64_t* empty;  // [kUnitQ] every reader warp read it (count kUnitReaders / kUnitReadersF8)
    int* idx;         // [kUnitQ] unit index, or -1: no more units
    int4* ent;        // FP8 [kUnitQ][2]: the unit decoded, {u, kb, rowA0, slot0}, {n, mt, c, shared | dn << 1}
};

// Producer warp: the next unit (or -1), taken from *ctr by lane 0 and published in the ring;
// false if the wait for a free entry gave up.
__device__ __forceinline__ bool take_unit(const UnitRing& r, int* ctr, int n_units, int& qi, int& u,
                                          volatile int* abort, uint64_t tmo) {
    int good = 1, v = -1;
    if ((threadIdx.x & 31) == 0) {
        const int e = qi % kUnitQ;
        good = tc::mbar_wait(&r.empty[e], ((qi / kUnitQ) & 1) ^ 1u, abort, tmo);
        if (good) {
            // a CTA's first unit is its own index, the rest come from the counter
            v = qi == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(ctr, 1);
            if (v >= n_units) v = -1;
            r.idx[e] = v;
            tc::mbar_arrive(&r.full[e]);
        }
    }
    ++qi;
    u = __shfl_sync(0xffffffffu, v, 0);
    return __shfl_sync(0xffffffffu, good, 0) != 0;
}

// MMA or epilogue warp: the next published unit (or -1); false if the wait gave up.
__device__ __forceinline__ bool read_unit(const UnitRing& r, int& qi, int& u, volatile int* abort, uint64_t tmo) {
    int good = 1, v = -1;
    if ((threadIdx.x & 31) == 0) {
        const int e = qi % kUnitQ;
        good = tc::mbar_wait(&r.full[e], (qi / kUnitQ) & 1, abort, tmo);
        if (good) {
            v = r.idx[e];
            tc::mbar_arrive(&r.empty[e]);
        }
    }
    ++qi;
    u = __shfl_sync(0xffffffffu, v, 0);
    return __shfl_sync(0xffffffffu, good, 0) != 0;
}

// FP8 reader warp: the next unit, decoded (u = -1: none left); false if the wait gave up.
__device__ __forceinline__ bool read_unit_f8(const UnitRing& r, int& qi, int& u, Unit& w, volatile int* abort,
                                             uint64_t tmo) {
    const int e = qi % kUnitQ;
    int good = 1;
    if ((threadIdx.x & 31) == 0) good = tc::mbar_wait(&r.full[e], (qi / kUnitQ) & 1, abort, tmo);
    good = __shfl_sync(0xffffffffu, good, 0);
    ++qi;
    if (!good) return false;
    const int4 a = r.ent[2 * e], b = r.ent[2 * e + 1];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&r.empty[e]);
    u = a.x;
    w = Unit{a.y, a.z, a.z + 64, a.w, b.x, b.y, b.z, (b.w & 1) != 0, (b.w & 2) != 0};
    return true;
}

template <int MODE, int NCH>
__global__ void __launch_bounds__(MODE == kExpertsF8 ? kThreadsF8 : kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ TensorMaps maps, const GemmParams p) {
    constexpr bool EXP = MODE == kExperts || MODE == kExpertsF8;  // whole routed + shared FFN
    constexpr bool F8 = MODE == kExpertsF8;                       // FP8 weights, converted in shared memory
    constexpr int STAGES = F8 ? f8_a_stages(NCH) : num_stages(NCH);  // F8: A stages in TMEM
    constexpr int SB = F8 ? 0 : stage_bytes(NCH);
    constexpr int SA = F8 ? f8_a_slots(NCH) : 0;          // F8: weight-tile slots
    constexpr int GB = F8 ? f8_b_granules(NCH) : 0;       // F8: token-row granules
    constexpr uint32_t TMEM_COLS = F8 ? 512u : ((2 * NCH < 32) ? 32u : static_cast<uint32_t>(2 * NCH));

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* aring = smem + STAGES * SB;  // F8: SA weight tiles of kF8Tile bytes
    uint8_t* bring = aring + SA * kF8Tile;  // F8: GB token-row granules (two half-rings)
    uint64_t* bars = reinterpret_cast<uint64_t*>(bring + GB * kGranule);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* fin = tempty + 2;
    uint64_t* conv = fin + 1;            // F8: the stage's weight tile is converted (count 1)
    uint64_t* fullA = conv + STAGES;     // F8: the weight tile landed (TMA bytes)
    uint64_t* emptyA = fullA + SA;       // F8: its four converter warps read it (count 4)
    uint64_t* fullB = emptyA + SA;       // F8: a granule's token rows landed (TMA bytes)
    uint64_t* emptyB = fullB + GB;       // F8: the MMAs that read them completed (commit)
    uint64_t* rend = emptyB + GB;
    constexpr bool DYN = EXP;  // units handed out at run time (UnitRing)
    int* ring_idx = reinterpret_cast<int*>(rend + 2 * kUnitQ);
    // F8: the decoded entries after the indices, 16-byte aligned (within the barrier area)
    int4* ring_ent = F8 ? reinterpret_cast<int4*>((reinterpret_cast<uintptr_t>(ring_idx + kUnitQ) + 15) & ~uintptr_t(15))
                        : nullptr;
    static_assert(!F8 || (3 * STAGES + 5 + 2 * SA + 2 * GB + 2 * kUnitQ) * 8 + 4 * kUnitQ + 16 + 2 * kUnitQ * 16 + 16 <=
                             kF8BarrierBytes,
                  "FP8 barrier area");
    const UnitRing ring{rend, rend + kUnitQ, ring_idx, ring_ent};
    uint32_t* tmem_holder =
        F8 ? reinterpret_cast<uint32_t*>(ring_ent + 2 * kUnitQ) : reinterpret_cast<uint32_t*>(ring.idx + kUnitQ);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int* zero_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);  // the MMA warp that used the stage releases it
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], F8 ? 2 : 1);  // F8: both MMA warps commit
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(fin, F8 ? 2 : 1);
        if (DYN)
            for (int q = 0; q < kUnitQ; ++q) {
                tc::mbar_init(&ring.full[q], 1);
                tc::mbar_init(&ring.empty[q], F8 ? kUnitReadersF8 : kUnitReaders);
            }
        if (F8) {
            for (int s = 0; s < STAGES; ++s) tc::mbar_init(&conv[s], 4);  // one arrival per warp of a group
            for (int s = 0; s < SA; ++s) {
                tc::mbar_init(&fullA[s], 1);
                tc::mbar_init(&emptyA[s], 4);
            }
            for (int s = 0; s < GB; ++s) {
                tc::mbar_init(&fullB[s], 1);
                tc::mbar_init(&emptyB[s], 1);  // the MMA warp that read the granule releases it
            }
        }
        *abort_flag = 0;
        *zero_flag = 0;
        tc::fence_mbar_init();
        tc::prefetch_tmap(&maps.a[0]);
        tc::prefetch_tmap(&maps.b[0]);
        if (F8)
            for (int i = 2; i < 6; ++i) tc::prefetch_tmap(&maps.b[i]);
        if (MODE != kLmHead) {
            tc::prefetch_tmap(&maps.a[1]);
            if (EXP) {
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
        if (EXP) n_units += nrc * p.dn_routed_tiles + nsc * p.dn_shared_tiles;
    }
    volatile int* abortv = abort_flag;
    const uint64_t tmo = p.timeout_ns;

    if (F8 && warp == 0) {
        // ------------------------------------------------------------ FP8 weight-tile producer
        // Fills the A ring in unit / K-block order; needs nothing from other CTAs, so a down
        // unit's tiles stream in while its chunk's SwiGLU rows are still being written.  Lane 0
        // alone runs the role: it takes each unit (a CTA's first unit is its block index, the
        // rest come from the global counter), decodes it and publishes it decoded in the unit
        // ring for the other roles.
        if (lane == 0) {
            const uint64_t pol = tc::policy_evict_first();
            uint32_t issued = 0, issued_parity = 0;
            constexpr int SAd = SA > 0 ? SA : 1;
            int seq = 0;
            bool ok = true;
            for (int qi = 0; ok; ++qi) {
                const int e = qi % kUnitQ;
                if (!tc::mbar_wait(&ring.empty[e], ((qi / kUnitQ) & 1) ^ 1u, abortv, tmo)) {
                    ok = false;
                    record_timeout(p.err, 7, -1, -1, -1, 0, n_units, 0);
                    break;
                }
                int u = qi == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(p.unit_ctr, 1);
                if (u >= n_units) u = -1;
                Unit w{};
                if (u >= 0) w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
                ring.ent[2 * e] = make_int4(u, w.kb, w.rowA0, w.slot0);
                ring.ent[2 * e + 1] = make_int4(w.n, w.mt, w.c, (w.shared ? 1 : 0) | (w.dn ? 2 : 0));
                tc::mbar_arrive(&ring.full[e]);
                if (u < 0) break;
                const CUtensorMap* mA = &maps.a[(w.dn ? 2 : 0) + (w.shared ? 1 : 0)];
                for (int kb = 0; kb < w.kb; ++kb, ++seq) {
                    const int slot = seq % SAd;
                    const uint32_t ph = (seq / SAd) & 1u;
                    if (!tc::mbar_wait(&emptyA[slot], ph ^ 1u, abortv, tmo)) {
                        ok = false;
                        record_timeout(p.err, 1, u, kb, slot, ph, n_units, w.n);
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&fullA[slot], kF8Tile);
                    tc::tma_load_2d_hint(aring + slot * kF8Tile, mA, &fullA[slot], kb * 128, w.rowA0, pol);
                    issued |= 1u << slot;
                    issued_parity = (issued_parity & ~(1u << slot)) | (ph << slot);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeoutProducer);
            }
            for (int s = 0; s < SA; ++s)
                if (issued & (1u << s)) tc::mbar_wait(&fullA[s], (issued_parity >> s) & 1u, zero_flag, kTeardownNs);
        }
        __syncwarp();
    } else if (F8 && warp == kTmaWarp2) {
        // ------------------------------------------------------------ FP8 token-row producer
        // Fills the B ring in the same order, a granule once the MMAs that read it completed; a
        // down unit's SwiGLU rows once its chunk's gate/up epilogues (any CTA) counted them stored.
        // One copy of 16, 32 or 64 rows per half-ring and K block.  Lane 0 alone runs the role,
        // unit reads included (no warp-wide step per K block: its loop paces the token rows).
        if (lane == 0) {
            uint32_t issued = 0, issued_parity = 0;
            uint32_t epar = 0, fpar = 0;  // use counts mod 2: per granule, per first granule of an entry
            int gpos = 0;
            bool ok = true;
            for (int qi = 0;;) {
                const int e = qi % kUnitQ;
                if (!tc::mbar_wait(&ring.full[e], (qi / kUnitQ) & 1, abortv, tmo)) {
                    ok = false;
                    break;
                }
                ++qi;
                const int4 ea = ring.ent[2 * e], eb = ring.ent[2 * e + 1];
                tc::mbar_arrive(&ring.empty[e]);
                const int u = ea.x;
                if (u < 0) break;
                const Unit w{ea.y, ea.z, ea.z + 64, ea.w, eb.x, eb.y, eb.z, (eb.w & 1) != 0, (eb.w & 2) != 0};
                const int nbp = granules_for(w.n);
                int g0 = granule_start<GB>(gpos, nbp);
                const CUtensorMap* mB = &maps.b[(w.dn ? 1 : 0) + (nbp & 6)];  // boxes of 16 nbp rows
                if (w.dn && !wait_count(&p.done[w.c], 4 * (w.shared ? p.shared_tiles : p.routed_tiles), abortv, tmo)) {
                    ok = false;
                    record_timeout(p.err, 6, u, -1, -1, 0, n_units, w.n);
                    break;
                }
                // the unit's K blocks with the entry size a constant (one granule nearly always)
                auto kblocks = [&](auto nbp_c) -> bool {
                    constexpr int NBP = decltype(nbp_c)::value;
                    for (int kb = 0; kb < w.kb; ++kb) {
#pragma unroll
                        for (int j = 0; j < NBP; ++j) {
                            const int g = g0 + j;
                            if (!tc::mbar_wait(&emptyB[g], ((epar >> g) & 1u) ^ 1u, abortv, tmo)) {
                                record_timeout(p.err, 1, u, kb, g, 0, n_units, w.n);
                                return false;
                            }
                        }
                        const uint32_t ph = (fpar >> g0) & 1u;
                        tc::mbar_arrive_expect_tx(&fullB[g0], NBP * kGranule);
                        tc::tma_load_2d(bring + g0 * kGranuleHalf, mB, &fullB[g0], kb * 128, w.slot0);
                        tc::tma_load_2d(bring + (GB + g0) * kGranuleHalf, mB, &fullB[g0], kb * 128 + 64, w.slot0);
                        issued |= 1u << g0;
                        issued_parity = (issued_parity & ~(1u << g0)) | (ph << g0);
                        epar ^= ((1u << NBP) - 1u) << g0;
                        fpar ^= 1u << g0;
                        g0 += NBP;
                        if (g0 == GB) g0 = 0;
                    }
                    return true;
                };
                // (entries of 4 granules only at 64-token chunks)
                const bool kok = nbp == 1                 ? kblocks(std::integral_constant<int, 1>{})
                                 : (NCH <= 32 || nbp == 2) ? kblocks(std::integral_constant<int, 2>{})
                                                           : kblocks(std::integral_constant<int, NCH <= 32 ? 2 : 4>{});
                if (!kok) {
                    ok = false;
                    break;
                }
                gpos = g0;
            }
            if (!ok) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeoutProducer);
            }
            for (int s = 0; s < GB; ++s)
                if (issued & (1u << s)) tc::mbar_wait(&fullB[s], (issued_parity >> s) & 1u, zero_flag, kTeardownNs);
        }
        __syncwarp();
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol = tc::policy_evict_first();
        uint32_t issued = 0, issued_parity = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int qi = 0;
        for (int u = blockIdx.x; ok; u += gridDim.x) {
            if (DYN) {
                if (!take_unit(ring, p.unit_ctr, n_units, qi, u, abortv, tmo)) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 7, u, -1, -1, 0, n_units, 0);
                    break;
                }
                if (u < 0) break;
            } else if (u >= n_units) {
                break;
            }
            const Unit w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int nb = (w.n + 15) >> 4;
            const CUtensorMap* mA = &maps.a[(w.dn && EXP ? 2 : 0) + (w.shared ? 1 : 0)];
            const CUtensorMap* mB = &maps.b[w.dn && EXP ? 1 : 0];
            if (EXP && w.dn) {
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
                        if (F8) {
                            // 128 x 64 FP8 bytes into the upper half of the A area (row r at 64 r);
                            // the converter warps rewrite the whole area as swizzled f16
                            tc::mbar_arrive_expect_tx(&full[stage], kABytes / 2 + nb * kBoxBBytes);
                            tc::tma_load_2d_hint(sa + kABytes / 2, mA, &full[stage], kb * 64, w.rowA0, pol);
                            tc::tma_load_2d_hint(sa + kABytes / 2 + kABytes / 4, mA, &full[stage], kb * 64,
                                                 w.rowA1, pol);
                        } else {
                            tc::mbar_arrive_expect_tx(&full[stage], kABytes + nb * kBoxBBytes);
                            tc::tma_load_2d_hint(sa, mA, &full[stage], kb * 64, w.rowA0, pol);
                            tc::tma_load_2d_hint(sa + kABytes / 2, mA, &full[stage], kb * 64, w.rowA1, pol);
                        }
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
    } else if (F8 && (warp == 1 || warp == kMmaWarp2)) {
        // ------------------------------------------------------------ FP8 MMA issuers
        // Lane 0 alone runs the role, unit reads included (no warp-wide step per unit: these
        // two warps bound the FP8 launch); the other lanes wait at the end.  Warp 1 issues the
        // eight MMAs of a unit's even K blocks into accumulator 0, warp kMmaWarp2 those of its
        // odd K blocks into accumulator 1 (TMEM columns 2 NCH ..), each with one wait and one
        // commit per K block; the epilogue adds the two.
        const int mh = warp == kMmaWarp2 ? 1 : 0;
        if (lane == 0) {
            bool ok = true;
            int qi = 0;
            int seq0 = 0;  // K blocks of the earlier units (the converters' stage sequence)
            int gpos = 0;  // the token-row ring position after the earlier units
            for (int it = 0;; ++it) {
                int u;
                Unit w;
                const int e = qi % kUnitQ;
                if (!tc::mbar_wait(&ring.full[e], (qi / kUnitQ) & 1, abortv, tmo)) {
                    ok = false;
                    break;
                }
                ++qi;
                const int4 a = ring.ent[2 * e], b = ring.ent[2 * e + 1];
                tc::mbar_arrive(&ring.empty[e]);
                u = a.x;
                if (u < 0) break;
                w = Unit{a.y, a.z, a.z + 64, a.w, b.x, b.y, b.z, (b.w & 1) != 0, (b.w & 2) != 0};
                const int buf = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                const int N = ((w.n + 15) >> 4) << 4;
                const uint32_t idesc = tc::idesc_f16(128, N);
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(mh * 2 * NCH + buf * NCH);
                bool good = tc::mbar_wait(&tempty[buf], aph ^ 1u, abortv, tmo);
                if (!good) record_timeout(p.err, 2, u, -1, buf, aph, n_units, w.n);
                tc::fence_after_sync();
                const int nbp = granules_for(w.n);  // token-row granules per K block
                const int p0 = granule_start<GB>(gpos, nbp);
                // this warp's K blocks with the entry size a constant (one granule nearly always)
                auto kblocks = [&](auto nbp_c) {
                    constexpr int NBP = decltype(nbp_c)::value;
                    int g0 = p0 + mh * NBP;  // this warp's first K block's entry
                    if (g0 >= GB) g0 -= GB;
                    for (int kb = mh; kb < w.kb && good; kb += 2) {
                        const int seq = seq0 + kb;
                        const int stage = seq % STAGES;
                        const uint32_t phase = (seq / STAGES) & 1u;
                        // the converted A operand (its converters saw the token rows land)
                        good = tc::mbar_wait(&conv[stage], phase, abortv, tmo);
                        if (!good) {
                            record_timeout(p.err, 3, u, kb, stage, phase, n_units, w.n);
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t at = tmem_base + static_cast<uint32_t>(f8_a_column(NCH) + 64 * stage);
                        const uint32_t sb = tc::smem_addr(bring + g0 * kGranuleHalf);
                        uint64_t bd[8];  // K = 16 steps 0..7: half-ring k >> 2, 32 bytes per step
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            bd[k] = tc::sdesc_k_sw128(sb + (k >> 2) * GB * kGranuleHalf + 32 * (k & 3));
                        tc::mma8_f16_tmem_a(d_tmem, at, bd, idesc, kb != mh);
                        tc::mma_commit(&empty[stage]);
#pragma unroll
                        for (int j = 0; j < NBP; ++j) tc::mma_commit(&emptyB[g0 + j]);
                        g0 += 2 * NBP;
                        if (g0 >= GB) g0 -= GB;
                    }
                };
                if (nbp == 1)
                    kblocks(std::integral_constant<int, 1>{});
                else if (NCH <= 32 || nbp == 2)  // (entries of 4 granules only at 64-token chunks)
                    kblocks(std::integral_constant<int, 2>{});
                else
                    kblocks(std::integral_constant<int, NCH <= 32 ? 2 : 4>{});
                if (!good) {
                    ok = false;
                    break;
                }
                tc::mma_commit(&tfull[buf]);
                seq0 += w.kb;
                gpos = (p0 + w.kb * nbp) % (GB > 0 ? GB : 4);
            }
            if (!ok) {
                *abort_flag = 1;
                record_error(p.err, kErrTimeoutMma);
            }
            // every MMA issued here has finished before TMEM and shared memory are released
            tc::mma_commit(fin);
            tc::mbar_wait(fin, 0, zero_flag, kTeardownNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (bf16)
        // Lane 0 alone walks a unit's K blocks (no warp-wide step per block); the warp
        // agrees on success once per unit.
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int it = 0;
        int qi = 0;
        for (int u = blockIdx.x; ok; u += gridDim.x, ++it) {
            if (DYN) {
                if (!read_unit(ring, qi, u, abortv, tmo)) {
                    ok = false;
                    break;
                }
                if (u < 0) break;
            } else if (u >= n_units) {
                break;
            }
            const Unit w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int buf = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            const int N = ((w.n + 15) >> 4) << 4;
            const uint32_t idesc = tc::idesc_bf16(128, N);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * NCH);
            int good = 1;
            if (lane == 0) {
                good = tc::mbar_wait(&tempty[buf], aph ^ 1u, abortv, tmo);
                if (!good) record_timeout(p.err, 2, u, -1, buf, aph, n_units, w.n);
                tc::fence_after_sync();
                for (int kb = 0; kb < w.kb && good; ++kb) {
                    good = tc::mbar_wait(&full[stage], phase, abortv, tmo);
                    if (!good) {
                        record_timeout(p.err, 3, u, kb, stage, phase, n_units, w.n);
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t sa = tc::smem_addr(smem + stage * SB);
                    const uint32_t sb = sa + kABytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc::mma_bf16(d_tmem, tc::sdesc_k_sw128(sa + 32 * k), tc::sdesc_k_sw128(sb + 32 * k), idesc,
                                     (kb | k) != 0);
                    tc::mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (good) tc::mma_commit(&tfull[buf]);
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) ok = false;
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
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int sp = warp & 3;  // TMEM sub-partition this warp may access: lanes 32*sp .. 32*sp+31
        int it = 0;
        int qi = 0;
        for (int u = blockIdx.x;; u += gridDim.x, ++it) {
            Unit w;
            if (DYN) {
                if (!(F8 ? read_unit_f8(ring, qi, u, w, abortv, tmo) : read_unit(ring, qi, u, abortv, tmo))) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        record_error(p.err, kErrTimeoutEpilogue);
                    }
                    break;
                }
                if (u < 0) break;
            } else if (u >= n_units) {
                break;
            }
            if (!F8) w = decode_unit<MODE, NCH>(u, p, nrc, nsc);
            const int L = 32 * sp + lane;  // accumulator row held by this thread
            // F8: the scale of weight row L of this tile, loaded while the unit's MMAs run
            const float rs = F8 ? __ldg(&p.sc[(w.dn ? 2 : 0) + (w.shared ? 1 : 0)][w.rowA0 + L]) : 1.0f;
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
            for (int c0 = 0; c0 < w.n; c0 += 32) {
                float v[32];
                tc::tmem_ld32(tb + c0, v);
                const int cnt = min(32, w.n - c0);
                if (F8) {
                    if (w.kb > 1) {  // the second MMA warp's K blocks (none in a one-block unit)
                        float v2[32];
                        tc::tmem_ld32(tb + 2 * NCH + c0, v2);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += v2[j];
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= rs;
                }
                if (MODE == kGateUp || (EXP && !w.dn)) {
                    // rows alternate gate / up of one intermediate index: partner lane holds the other half
                    const int i = w.mt * 64 + (L >> 1);
                    const bool is_gate = (lane & 1) == 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float o = __shfl_xor_sync(0xffffffffu, v[j], 1);
                        if (j < cnt && (j & 1) == (lane & 1)) {
                            const float g = is_gate ? v[j] : o;
                            const float up = is_gate ? o : v[j];
                            const size_t at = static_cast<size_t>(w.slot0 + c0 + j) * p.out_ld + i;
                            if (F8)
                                static_cast<__half*>(p.out)[at] = __float2half_rn(silu_f(g) * up);
                            else
                                static_cast<bf16*>(p.out)[at] = __float2bfloat16_rn(silu_f(g) * up);
                        }
                    }
                } else if (MODE == kDown || EXP) {
                    float* y = static_cast<float*>(EXP ? p.out2 : p.out);
                    const int ld = EXP ? p.out2_ld : p.out_ld;
                    const int h = w.mt * 128 + L;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < cnt) y[static_cast<size_t>(w.slot0 + c0 + j) * ld + h] = v[j];
                } else {
                    // per (position, 32-row slice): max logit, its lowest row, sum of exp(l - max).
                    // Transposed butterfly over the warp: at offset o each lane keeps the half of
                    // its columns whose bit o matches its own and takes its partner's partial of
                    // them, so after five steps lane j holds column j reduced over the 32 rows
                    // (31 shuffles per quantity instead of 10 per column).
                    const int row = w.mt * 128 + L;
                    const bool valid = row < p.V;
                    float lg[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        lg[j] = (valid && j < cnt) ? v[j] * p.scale : -INFINITY;
                        if (p.logits != nullptr && valid && j < cnt)
                            p.logits[static_cast<size_t>(w.slot0 + c0 + j) * p.V + row] = lg[j];
                    }
                    float m[32];
                    int ar[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        m[j] = lg[j];
                        ar[j] = row;
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        const bool up = (lane & o) != 0;
#pragma unroll
                        for (int i = 0; i < o; ++i) {
                            const float give_m = up ? m[i] : m[i + o];
                            const int give_a = up ? ar[i] : ar[i + o];
                            const float km = up ? m[i + o] : m[i];
                            const int ka = up ? ar[i + o] : ar[i];
                            const float rm = __shfl_xor_sync(0xffffffffu, give_m, o);
                            const int ra = __shfl_xor_sync(0xffffffffu, give_a, o);
                            const bool take = rm > km || (rm == km && ra < ka);
                            m[i] = take ? rm : km;
                            ar[i] = take ? ra : ka;
                        }
                    }
                    const float mm = m[0];  // column `lane`
                    const int aa = ar[0];
                    float e[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float mj = __shfl_sync(0xffffffffu, mm, j);
                        e[j] = (mj == -INFINITY || lg[j] == -INFINITY) ? 0.f : __expf(lg[j] - mj);
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        const bool up = (lane & o) != 0;
#pragma unroll
                        for (int i = 0; i < o; ++i) {
                            const float give = up ? e[i] : e[i + o];
                            const float keep = up ? e[i + o] : e[i];
                            e[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
                        }
                    }
                    const float ss = e[0];
                    if (lane < cnt) {
                        const size_t o = static_cast<size_t>(w.mt * 4 + sp) * p.n_pos + (w.slot0 + c0 + lane);
                        p.pmax[o] = mm;
                        p.parg[o] = aa;
                        p.psum[o] = ss;
                    }
                }
            }
            if (EXP && !w.dn) {
                // publish this warp's SwiGLU rows to the down units of the chunk (any CTA)
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(&p.done[w.c], 1);
            }
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[buf]);
        }
    } else if (F8 && warp < kMmaWarp2) {
        // ------------------------------------------------------------ FP8 -> f16 converters (warps 6..13)
        // Two groups of four warps take alternate K blocks.  Within a group each warp takes
        // the 32 weight rows of its TMEM lane quarter; thread i reads row 32q + i of the
        // FP8 tile (128 bytes, 16-byte chunk j of row r at chunk j ^ (r & 7): the TMA's
        // 128-byte swizzle, so a warp's reads hit distinct banks) and releases the A slot,
        // then, once the TMEM stage is free, converts the row into 64 f16x2 words (exactly)
        // and stores them as TMEM lane 32q + i, columns
        // f8_a_column(NCH) + 64 stage ..: A row i in lane i, elements 2c, 2c+1 in column c.
        const int q = warp & 3;
        const int grp = (warp - 6) >> 2;
        const int row = 32 * q + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        constexpr int SAd = SA > 0 ? SA : 1;
        bool ok = true;
        int seq = 0;
        int qi = 0;
        uint32_t fpar = 0;  // use count mod 2 of each granule as an entry's first
        int gpos = 0;
        for (int u = blockIdx.x; ok; u += gridDim.x) {
            Unit w;
            if (!read_unit_f8(ring, qi, u, w, abortv, tmo)) {
                ok = false;
                break;
            }
            if (u < 0) break;
            const int nbp = granules_for(w.n);
            int gn = granule_start<GB>(gpos, nbp);
            for (int kb = 0; kb < w.kb; ++kb, ++seq) {
                // every K block's entry, the other group's too, to keep the parities
                const int g0 = gn;
                const uint32_t phb = (fpar >> g0) & 1u;
                fpar ^= 1u << g0;
                gn += nbp;
                if (gn == GB) gn = 0;
                if ((seq & 1) != grp) continue;
                const int stage = seq % STAGES;
                const uint32_t phase = (seq / STAGES) & 1u;
                const int slot = seq % SAd;
                const uint32_t pha = (seq / SAd) & 1u;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&fullA[slot], pha, abortv, tmo))) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 8, u, kb, slot, pha, n_units, w.n);
                    break;
                }
                const uint4* src = reinterpret_cast<const uint4*>(aring + slot * kF8Tile + 128 * row);
                uint4 raw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) raw[i] = src[i ^ (row & 7)];
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&emptyA[slot]);  // the tile is in registers
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&empty[stage], phase ^ 1u, abortv, tmo))) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 9, u, kb, stage, phase, n_units, w.n);
                    break;
                }
                tc::fence_after_sync();
                uint32_t h[64];  // the row's 128 codes as 64 f16x2 words, stored with one instruction
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = raw[i];
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        h[8 * i + 2 * j] = tc::e4m3x2_to_f16x2(wv[j], 0);
                        h[8 * i + 2 * j + 1] = tc::e4m3x2_to_f16x2(wv[j], 2);
                    }
                }
                tc::tmem_st64(lane_base + static_cast<uint32_t>(f8_a_column(NCH) + 64 * stage), h);
                tc::fence_before_sync();
                // the K block's token rows have landed before the MMA warps may read them
                if (!__all_sync(0xffffffffu, lane != 0 || tc::mbar_wait(&fullB[g0], phb, abortv, tmo))) {
                    ok = false;
                    if (lane == 0) record_timeout(p.err, 10, u, kb, g0, 0, n_units, w.n);
                    break;
                }
                if (lane == 0) tc::mbar_arrive(&conv[stage]);
            }
            gpos = gn;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            record_error(p.err, kErrTimeoutProducer);
        }
        __syncwarp();
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
    constexpr int bytes = MODE == kExpertsF8 ? smem_bytes_f8(NCH) : smem_bytes(NCH);
    static int done[64] = {};
    cudaError_t e = ensure_smem(tc_gemm_kernel<MODE, NCH>, bytes, done);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc_gemm_kernel<MODE, NCH>, dim3(grid), dim3(MODE == kExpertsF8 ? kThreadsF8 : kThreads), bytes,
                      s, maps, p);
}

template <int MODE>
cudaError_t launch_mode(int nch, const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s) {
    if constexpr (MODE == kExpertsF8) {  // token chunks of at most 64 (accumulators and A stages share the TMEM)
        if (nch == 32) return launch_one<MODE, 32>(maps, p, grid, s);
        if (nch == 64) return launch_one<MODE, 64>(maps, p, grid, s);
        return cudaErrorInvalidValue;
    } else {
        switch (nch) {
            case 32: return launch_one<MODE, 32>(maps, p, grid, s);
            case 64: return launch_one<MODE, 64>(maps, p, grid, s);
            case 128: return launch_one<MODE, 128>(maps, p, grid, s);
            case 256: return launch_one<MODE, 256>(maps, p, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
}

}  // namespace

int tc_gemm_smem_bytes(int nch) { return smem_bytes(nch); }

cudaError_t launch_tc_gemm(int mode, int nch, const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s) {
    switch (mode) {
        case kExperts: return launch_mode<kExperts>(nch, maps, p, grid, s);
        case kExpertsF8: return launch_mode<kExpertsF8>(nch, maps, p, grid, s);
        case kLmHead: return launch_mode<kLmHead>(nch, maps, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moestep
