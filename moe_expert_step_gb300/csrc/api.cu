// C ABI of the moestep library: argument validation, workspace layout, TMA
// tensor maps, kernel sequencing and the optional event-based kernel timing.
// Every check happens before the first launch of a call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "moestep.h"

namespace moestep {

bool g_launch_pdl = true;

namespace {

thread_local int g_last_cuda = 0;
unsigned long long g_timeout_ns = 2000000000ull;  // bounded waits inside the tcgen05 kernels
// What runs between two expert launches of block_decode_step: 0 separate combine /
// router / coreset / gather launches; 2 the combine fused into the router's
// cluster launch
int g_layer_head = 2;

#define MOESTEP_CK(expr)                             \
    do {                                             \
        cudaError_t e_ = (expr);                     \
        if (e_ != cudaSuccess) {                     \
            g_last_cuda = static_cast<int>(e_);      \
            return MOESTEP_ECUDA;                    \
        }                                            \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// element type of everything but the expert weights (router, activations, LM head)
int act_dtype(int dtype) { return dtype == MOESTEP_FP8 ? MOESTEP_BF16 : dtype; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Token chunk of a unit (the MMA's N is at most this).  The expert GEMM caps it
// at 64 so the shared-memory ring keeps >= 8 stages (more weight bytes in
// flight); an expert with more tokens is split into chunks whose weight tiles
// are re-read from L2.  The LM head streams one tile per position chunk, so it
// keeps wide chunks.
int nch_for(int T) { return T <= 32 ? 32 : 64; }
int lm_nch_for(int T) { return T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }

// ---------------------------------------------------------------------------- workspace
struct Layout {
    int T, max_slots, max_chunks, act_ld, n_ptiles, nch, lm_nch, route_groups;
    size_t hdr, counters, counters_bytes, logits, idx, mass, gate, nsel, sel, survive, gaterr, slot_of, slot_sh,
        slot_tok, slot_exp, chunks, done, xp, act, y, hres, x, pmax, parg, psum, lmlogits, loop_h, loop_choice,
        loop_conf, loop_accept, loop_ncomm, total;
};

Layout make_layout(const moestep_dims& d, int R) {
    Layout L{};
    const int T = R * d.P;
    const size_t esz = d.dtype == MOESTEP_F32 ? 4 : 2;
    L.T = T;
    L.max_slots = T * d.k + T;
    L.max_chunks = T * d.k + d.E + T + 1;
    L.act_ld = d.I > d.Is ? d.I : d.Is;
    L.nch = nch_for(T);
    L.lm_nch = lm_nch_for(T);
    L.route_groups = (T + kRouteTokensPerCta - 1) / kRouteTokensPerCta;
    const int tiles_tc = (d.V + 127) / 128 * 4;
    const int tiles_logit = (d.V + kLogitTile - 1) / kLogitTile;
    L.n_ptiles = tiles_tc > tiles_logit ? tiles_tc : tiles_logit;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + (bytes ? bytes : 1), 256);
        return at;
    };
    L.hdr = take(256);  // int[0]: error word, int[8..15]: where a wait timed out, int[32..34]: expert work plan
    // router groups, coreset, commit per request, plan flag (zeroed at the start of every call)
    L.counters_bytes = sizeof(int) * (L.route_groups + 1 + R + 1);
    L.counters = take(L.counters_bytes);
    L.logits = take(sizeof(float) * T * d.E);
    L.idx = take(sizeof(int32_t) * T * d.k);
    L.mass = take(sizeof(float) * T * d.k);
    L.gate = take(sizeof(float) * T * d.k);
    L.nsel = take(sizeof(int32_t) * R);
    L.sel = take(sizeof(int32_t) * R * d.E);
    L.survive = take(static_cast<size_t>(T) * d.k);
    L.gaterr = take(sizeof(float) * T * d.k);
    L.slot_of = take(sizeof(int32_t) * T * d.k);
    L.slot_sh = take(sizeof(int32_t) * T);
    L.slot_tok = take(sizeof(int32_t) * L.max_slots);
    L.slot_exp = take(sizeof(int32_t) * L.max_slots);
    L.chunks = take(sizeof(int4) * L.max_chunks);
    L.done = take(sizeof(int) * (L.max_chunks + 1));  // chunk counters, then the expert launch's unit counter
    L.xp = take(esz * L.max_slots * d.H);
    L.act = take(esz * L.max_slots * L.act_ld);
    L.y = take(sizeof(float) * L.max_slots * d.H);
    L.hres = take(sizeof(float) * T * d.H);
    L.x = take(esz * T * d.H);
    L.pmax = take(sizeof(float) * L.n_ptiles * T);
    L.parg = take(sizeof(int) * L.n_ptiles * T);
    L.psum = take(sizeof(float) * L.n_ptiles * T);
    L.lmlogits = take(d.dtype == MOESTEP_F32 ? sizeof(float) * T * static_cast<size_t>(d.V) : 0);
    // device-resident round loop: embedded block and the per-round commit outputs
    L.loop_h = take(sizeof(float) * T * d.H);
    L.loop_choice = take(sizeof(int32_t) * T);
    L.loop_conf = take(sizeof(float) * T);
    L.loop_accept = take(static_cast<size_t>(T));
    L.loop_ncomm = take(sizeof(int32_t) * R);
    L.total = o;
    return L;
}

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------------------- validation
int check_dims(const moestep_dims* d) {
    if (d == nullptr) return MOESTEP_EINVAL;
    if (d->H <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0 || d->Is < 0 || d->P <= 0 || d->V <= 0) return MOESTEP_EINVAL;
    if (d->dtype != MOESTEP_BF16 && d->dtype != MOESTEP_F32 && d->dtype != MOESTEP_FP8) return MOESTEP_EINVAL;
    if (d->k > d->E || d->k > 32 || d->E > 1024 || d->P > 1024) return MOESTEP_EUNSUPPORTED;
    if (d->H % 8 || d->I % 4 || d->Is % 4) return MOESTEP_EUNSUPPORTED;
    if (8ll * (d->H > d->E ? d->H : d->E) * 4 > 200 * 1024) return MOESTEP_EUNSUPPORTED;  // router staging
    if (d->dtype != MOESTEP_F32 && (d->H % 128 || d->I % 64 || d->Is % 64)) return MOESTEP_EUNSUPPORTED;
    return MOESTEP_OK;
}

int check_ws(const moestep_dims* d, int R, const void* ws, size_t ws_bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOESTEP_EWORKSPACE;
    if (ws_bytes < make_layout(*d, R).total) return MOESTEP_EWORKSPACE;
    return MOESTEP_OK;
}

int check_R(const moestep_dims* d, int R) {
    if (R <= 0) return MOESTEP_EINVAL;
    const long long T = 1ll * R * d->P;
    if (T > 8192) return MOESTEP_EUNSUPPORTED;
    if (1ll * d->E * ((T + 31) / 32) * 4 > 160 * 1024) return MOESTEP_EUNSUPPORTED;  // coreset plan masks
    return MOESTEP_OK;
}

struct DeviceInfo {
    int ok = -1;
    int sms = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int device_check(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda = static_cast<int>(e);
        return MOESTEP_ECUDA;
    }
    if (dev < 0 || dev >= 64) return MOESTEP_EDEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& di = g_dev[dev];
    if (di.ok < 0) {
        int major = 0, minor = 0;
        MOESTEP_CK(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
        MOESTEP_CK(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
        MOESTEP_CK(cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev));
        di.ok = (major == 10 && minor == 3) ? 1 : 0;
    }
    if (!di.ok) return MOESTEP_EDEVICE;
    if (sms) *sms = di.sms;
    return MOESTEP_OK;
}

// ---------------------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? MOESTEP_OK : MOESTEP_ECUDA;
}

// 2D bf16 tensor [rows][cols] (cols contiguous), boxes of 64 columns x box_rows
// rows in the 128-byte swizzled shared-memory layout; out-of-range rows read as 0.
// FP8 E4M3 weights: boxes of 128 rows x 128 bytes (a K block of 128) in the 128-byte
// swizzled layout, so the converter threads' row reads hit distinct banks (the expert launch's
// converter warps write the swizzled f16 operand themselves)
int make_map_fp8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda = static_cast<int>(r);
        return MOESTEP_ECUDA;
    }
    return MOESTEP_OK;
}

int make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda = static_cast<int>(r);
        return MOESTEP_ECUDA;
    }
    return MOESTEP_OK;
}

// ---------------------------------------------------------------------------- timing
std::atomic<long long> g_launches{0};

struct Prof {
    int mask = 0;
    std::vector<cudaEvent_t> pool;
    size_t next = 0;
    cudaEvent_t pending[MOESTEP_PROF_KERNELS] = {};
    std::vector<int> kid;
    std::vector<cudaEvent_t> start, stop;
} g_prof;

cudaEvent_t prof_event() {
    if (g_prof.next == g_prof.pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_prof.pool.push_back(e);
    }
    return g_prof.pool[g_prof.next++];
}

// ---------------------------------------------------------------------------- pieces
struct Ctx {
    const moestep_dims* d;
    Layout L;
    void* ws;
    cudaStream_t s;
    int sms;
};

#define MOESTEP_LAUNCH(kid, call)               \
    do {                                        \
        prof_begin((kid), c.s);                 \
        cudaError_t e_ = (call);                \
        prof_end((kid), c.s);                   \
        if (e_ != cudaSuccess) {                \
            g_last_cuda = static_cast<int>(e_); \
            return MOESTEP_ECUDA;               \
        }                                       \
        g_launches.fetch_add(1);                \
    } while (0)

int run_route(const Ctx& c, int T, const void* x, const void* Wr, int32_t* idx, float* mass, float* gate,
              float* logits) {
    const moestep_dims* d = c.d;
    float* lg = logits ? logits : at<float>(c.ws, c.L.logits);
    MOESTEP_LAUNCH(0, launch_route(act_dtype(d->dtype), x, Wr, T, d->H, d->E, d->k, lg, idx, mass, gate,
                                   at<int>(c.ws, c.L.counters), at<int>(c.ws, c.L.hdr), c.s));
    return MOESTEP_OK;
}

CoresetArgs coreset_args(const Ctx& c, int R, const float* top_p, const int32_t* idx, const float* mass,
                         int32_t* n_sel, int32_t* sel, uint8_t* survive, float* gate_rr) {
    const moestep_dims* d = c.d;
    CoresetArgs a{};
    a.R = R;
    a.P = d->P;
    a.k = d->k;
    a.E = d->E;
    a.T = R * d->P;
    a.top_p = top_p;
    a.idx = idx;
    a.mass = mass;
    a.n_sel = n_sel;
    a.sel = sel;
    a.survive = survive;
    a.gate_rr = gate_rr;
    a.slot_of = at<int32_t>(c.ws, c.L.slot_of);
    a.slot_sh = at<int32_t>(c.ws, c.L.slot_sh);
    a.slot_tok = at<int32_t>(c.ws, c.L.slot_tok);
    a.slot_exp = at<int32_t>(c.ws, c.L.slot_exp);
    a.chunks = at<int4>(c.ws, c.L.chunks);
    a.plan = at<int>(c.ws, c.L.hdr) + 32;
    a.counter = at<int>(c.ws, c.L.counters) + c.L.route_groups;
    a.nch = c.L.nch;
    a.has_shared = d->Is > 0;
    a.err = at<int>(c.ws, c.L.hdr);
    return a;
}

// set to l + 1 by layer l's gather launch once the coreset has completed; zeroed with the counters
int* plan_flag(const Ctx& c, int R) { return at<int>(c.ws, c.L.counters) + c.L.route_groups + 1 + R; }

// Wgu (may be NULL): the layer's gate/up weights, hinted into L2 for the first candidates
// Wr_next (may be NULL): the next layer's router weights, hinted too
int run_coreset(const Ctx& c, int R, const float* top_p, const int32_t* idx, const float* mass, int32_t* n_sel,
                int32_t* sel, uint8_t* survive, float* gate_rr, const void* Wgu = nullptr,
                const void* Wr_next = nullptr) {
    CoresetArgs a = coreset_args(c, R, top_p, idx, mass, n_sel, sel, survive, gate_rr);
    if (Wgu != nullptr && c.d->dtype != MOESTEP_F32 && c.sms > R) {
        a.pf_base = static_cast<const char*>(Wgu);
        a.pf_stride = 2ll * c.d->I * c.d->H * (c.d->dtype == MOESTEP_FP8 ? 1 : 2);
        a.pf_experts = c.d->dtype == MOESTEP_FP8 ? kCoresetPrefetchExpertsF8 : kCoresetPrefetchExperts;
        a.pf_ctas = c.sms - R;
        a.pf_next = static_cast<const char*>(Wr_next);
        a.pf_next_bytes = 2ll * c.d->E * c.d->H;
    }
    MOESTEP_LAUNCH(1, launch_coreset(a, c.s));
    return MOESTEP_OK;
}

// the previous layer's combine (mode 1) or the input norm (mode 2), then the router
int run_route_combine(const Ctx& c, int mode, const float* h_in, const void* Wr, int32_t* idx, int layer = 0) {
    const moestep_dims* d = c.d;
    const Layout& L = c.L;
    RouteCombineArgs a{};
    a.mode = mode;
    a.y = at<float>(c.ws, L.y);
    a.slot_of = at<int32_t>(c.ws, L.slot_of);
    a.slot_sh = at<int32_t>(c.ws, L.slot_sh);
    a.gate_rr_prev = at<float>(c.ws, L.gaterr);
    a.has_shared = d->Is > 0;
    a.h_in = h_in;
    a.hres = at<float>(c.ws, L.hres);
    a.x = at<__nv_bfloat16>(c.ws, L.x);
    a.Wr = static_cast<const __nv_bfloat16*>(Wr);
    a.T = L.T;
    a.H = d->H;
    a.E = d->E;
    a.k = d->k;
    a.logits = nullptr;
    a.idx = idx;
    a.mass = at<float>(c.ws, L.mass);
    a.gate = at<float>(c.ws, L.gate);
    a.plan_flag = plan_flag(c, L.T / d->P);
    a.plan_value = layer;  // layer - 1's gather stored layer
    a.timeout_ns = g_timeout_ns;
    MOESTEP_LAUNCH(0, launch_route_combine(a, c.s));
    return MOESTEP_OK;
}

// gather + experts (fp32: FFMA; bf16: tcgen05 gate/up then down); leaves y
// (per slot) in the workspace.  layer >= 0 (block_decode_step): the gather sets the plan flag
// to layer + 1 for the next layer's router launch.
int run_experts(const Ctx& c, int R, const void* x, const moestep_layer* layer, int layer_index = -1) {
    const moestep_dims* d = c.d;
    const Layout& L = c.L;
    const int* plan = at<int>(c.ws, L.hdr) + 32;
    const bool tc = d->dtype != MOESTEP_F32;
    MOESTEP_LAUNCH(2, launch_gather(d->dtype, x, d->H, at<int32_t>(c.ws, L.slot_tok), plan, L.max_slots,
                                    at<void>(c.ws, L.xp), tc ? at<int>(c.ws, L.done) : nullptr, L.max_chunks + 1,
                                    layer_index >= 0 ? plan_flag(c, R) : nullptr, layer_index + 1, c.s));
    if (d->dtype == MOESTEP_F32) {
        MOESTEP_LAUNCH(3, launch_f32_gateup(d->H, d->E, d->I, d->Is, L.max_slots, at<float>(c.ws, L.xp),
                                            at<int32_t>(c.ws, L.slot_exp), plan, static_cast<const float*>(layer->Wgu),
                                            static_cast<const float*>(layer->Wsgu), at<float>(c.ws, L.act), L.act_ld,
                                            c.s));
        MOESTEP_LAUNCH(4, launch_f32_down(d->H, d->E, d->I, d->Is, L.max_slots, at<float>(c.ws, L.act), L.act_ld,
                                          at<int32_t>(c.ws, L.slot_exp), plan, static_cast<const float*>(layer->Wd),
                                          static_cast<const float*>(layer->Wsd), at<float>(c.ws, L.y), c.s));
        return MOESTEP_OK;
    }
    if (get_encode() != MOESTEP_OK) return MOESTEP_ECUDA;
    const bool sh = d->Is > 0;
    const bool f8 = d->dtype == MOESTEP_FP8;
    TensorMaps m{};
    int rc;
    if (f8) {
        if ((rc = make_map_fp8(&m.a[0], layer->Wgu, d->H, 2ull * d->E * d->I))) return rc;
        if ((rc = make_map_fp8(&m.a[1], sh ? layer->Wsgu : layer->Wgu, d->H, sh ? 2ull * d->Is : 128))) return rc;
        if ((rc = make_map_fp8(&m.a[2], layer->Wd, d->I, 1ull * d->E * d->H))) return rc;
        if ((rc = make_map_fp8(&m.a[3], sh ? layer->Wsd : layer->Wd, sh ? d->Is : d->I, d->H))) return rc;
    } else {
        if ((rc = make_map(&m.a[0], layer->Wgu, d->H, 2ull * d->E * d->I, 64))) return rc;
        if ((rc = make_map(&m.a[1], sh ? layer->Wsgu : layer->Wgu, d->H, sh ? 2ull * d->Is : 128, 64))) return rc;
        if ((rc = make_map(&m.a[2], layer->Wd, d->I, 1ull * d->E * d->H, 64))) return rc;
        if ((rc = make_map(&m.a[3], sh ? layer->Wsd : layer->Wd, sh ? d->Is : d->I, d->H, 64))) return rc;
    }
    if ((rc = make_map(&m.b[0], at<void>(c.ws, L.xp), d->H, L.max_slots, 16))) return rc;
    if ((rc = make_map(&m.b[1], at<void>(c.ws, L.act), L.act_ld, L.max_slots, 16))) return rc;
    for (int i = 1; f8 && i <= 2; ++i) {  // 32- and 64-row boxes: a K block's token rows in one copy
        if ((rc = make_map(&m.b[2 * i], at<void>(c.ws, L.xp), d->H, L.max_slots, 16u << i))) return rc;
        if ((rc = make_map(&m.b[2 * i + 1], at<void>(c.ws, L.act), L.act_ld, L.max_slots, 16u << i))) return rc;
    }
    GemmParams g{};
    g.plan = plan;
    g.chunks = at<int4>(c.ws, L.chunks);
    g.err = at<int>(c.ws, L.hdr);
    g.timeout_ns = g_timeout_ns;
    g.tile_rows = 128;
    // gate/up: 128-row tiles of interleaved gate/up rows = 64 intermediate indices
    g.routed_tiles = 2 * d->I / 128;
    g.shared_tiles = 2 * d->Is / 128;
    const int kbw = f8 ? 128 : 64;  // K per block: FP8 tiles are 128 bytes wide
    g.routed_kb = d->H / kbw;
    g.shared_kb = d->H / kbw;
    g.rows_per_expert = 2 * d->I;
    g.out = at<void>(c.ws, L.act);
    g.out_ld = L.act_ld;
    // down: 128-row tiles of the hidden dimension
    g.dn_routed_tiles = d->H / 128;
    g.dn_shared_tiles = d->H / 128;
    g.dn_routed_kb = d->I / kbw;
    g.dn_shared_kb = d->Is / kbw;
    g.dn_rows_per_expert = d->H;
    g.out2 = at<void>(c.ws, L.y);
    g.out2_ld = d->H;
    g.done = at<int>(c.ws, L.done);
    g.unit_ctr = at<int>(c.ws, L.done) + L.max_chunks;
    g.sc[0] = layer->Sgu;
    g.sc[1] = sh ? layer->Ssgu : layer->Sgu;
    g.sc[2] = layer->Sd;
    g.sc[3] = sh ? layer->Ssd : layer->Sd;
    MOESTEP_LAUNCH(3, launch_tc_gemm(f8 ? kExpertsF8 : kExperts, L.nch, m, g, c.sms, c.s));
    return MOESTEP_OK;
}

int run_lm_commit(const Ctx& c, int R, const void* hidden, const void* Wlm, float scale, float thr, int32_t* tokens,
                  uint8_t* masked, int32_t* choice, float* conf, uint8_t* accept, int32_t* n_committed,
                  float* logits) {
    const moestep_dims* d = c.d;
    const Layout& L = c.L;
    const int T = R * d->P;
    int n_tiles;
    if (d->dtype != MOESTEP_F32) {
        if (get_encode() != MOESTEP_OK) return MOESTEP_ECUDA;
        TensorMaps m{};
        int rc;
        if ((rc = make_map(&m.a[0], Wlm, d->H, d->V, 64))) return rc;
        if ((rc = make_map(&m.b[0], hidden, d->H, T, 16))) return rc;
        m.a[1] = m.a[2] = m.a[3] = m.a[0];
        m.b[1] = m.b[0];
        GemmParams g{};
        g.routed_kb = d->H / 64;
        g.lm_chunks = (T + L.lm_nch - 1) / L.lm_nch;
        g.lm_tiles = (d->V + 127) / 128;
        g.n_pos = T;
        g.V = d->V;
        g.scale = scale;
        g.pmax = at<float>(c.ws, L.pmax);
        g.parg = at<int>(c.ws, L.parg);
        g.psum = at<float>(c.ws, L.psum);
        g.logits = logits;
        g.err = at<int>(c.ws, L.hdr);
        g.timeout_ns = g_timeout_ns;
        const int units = g.lm_chunks * g.lm_tiles;
        MOESTEP_LAUNCH(6, launch_tc_gemm(kLmHead, L.lm_nch, m, g, units < c.sms ? units : c.sms, c.s));
        n_tiles = g.lm_tiles * 4;
    } else {
        float* lg = logits ? logits : at<float>(c.ws, L.lmlogits);
        MOESTEP_LAUNCH(6, launch_f32_lm_logits(T, d->H, d->V, static_cast<const float*>(hidden),
                                               static_cast<const float*>(Wlm), scale, lg, c.s));
        MOESTEP_LAUNCH(8, launch_partials_from_logits(lg, T, d->V, at<float>(c.ws, L.pmax), at<int>(c.ws, L.parg),
                                                      at<float>(c.ws, L.psum), c.s));
        n_tiles = (d->V + kLogitTile - 1) / kLogitTile;
    }
    MOESTEP_LAUNCH(7, launch_commit(R, d->P, n_tiles, at<float>(c.ws, L.pmax), at<int>(c.ws, L.parg),
                                    at<float>(c.ws, L.psum), thr, tokens, masked, choice, conf, accept, n_committed,
                                    at<int>(c.ws, L.counters) + L.route_groups + 1, c.s));
    return MOESTEP_OK;
}

int layer_ok(const moestep_dims* d, const moestep_layer* l) {
    if (l == nullptr || !l->Wr || !l->Wgu || !l->Wd) return MOESTEP_EINVAL;
    if (d->Is > 0 && (!l->Wsgu || !l->Wsd)) return MOESTEP_EINVAL;
    if (!aligned16(l->Wr) || !aligned16(l->Wgu) || !aligned16(l->Wd)) return MOESTEP_EALIGN;
    if (d->Is > 0 && (!aligned16(l->Wsgu) || !aligned16(l->Wsd))) return MOESTEP_EALIGN;
    if (d->dtype == MOESTEP_FP8) {
        if (!l->Sgu || !l->Sd || (d->Is > 0 && (!l->Ssgu || !l->Ssd))) return MOESTEP_EINVAL;
        if (d->H % 128 || d->I % 128 || d->Is % 128) return MOESTEP_EUNSUPPORTED;  // K blocks of 128
    }
    return MOESTEP_OK;
}

bool thr_ok(float t) { return t > 0.f && t <= 1.f; }

}  // namespace

int validate_dims(const moestep_dims* d) { return check_dims(d); }
int device_ok(int* sms) { return device_check(sms); }
void set_last_cuda(int err) { g_last_cuda = err; }
void count_launch() { g_launches.fetch_add(1); }

void prof_begin(int kid, cudaStream_t s) {
    if (kid < 0 || kid >= MOESTEP_PROF_KERNELS || !((g_prof.mask >> kid) & 1)) return;
    cudaEvent_t e = prof_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess) g_prof.pending[kid] = e;
}

void prof_end(int kid, cudaStream_t s) {
    if (kid < 0 || kid >= MOESTEP_PROF_KERNELS || !((g_prof.mask >> kid) & 1) || !g_prof.pending[kid]) return;
    cudaEvent_t e = prof_event();
    if (e && cudaEventRecord(e, s) == cudaSuccess) {
        g_prof.kid.push_back(kid);
        g_prof.start.push_back(g_prof.pending[kid]);
        g_prof.stop.push_back(e);
    }
    g_prof.pending[kid] = nullptr;
}

}  // namespace moestep

using namespace moestep;

#define MOESTEP_TRY(expr)        \
    do {                         \
        int rc_ = (expr);        \
        if (rc_ != MOESTEP_OK) return rc_; \
    } while (0)

namespace {

// ---------------------------------------------------------------------------- device-resident round loop
// One cached executable graph: [condition kernel (rounds = 0)] -> while node
// { block_embed, block_decode_step, condition kernel (rounds += 1) }.
struct LoopGraph {
    std::vector<unsigned char> key;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};
std::mutex g_loop_mu;
LoopGraph g_loop;
cudaStream_t g_capture_stream[64] = {};

template <typename V>
void key_add(std::vector<unsigned char>& k, const V& v) {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(&v);
    k.insert(k.end(), p, p + sizeof(V));
}

void loop_release() {
    if (g_loop.exec) cudaGraphExecDestroy(g_loop.exec);
    if (g_loop.graph) cudaGraphDestroy(g_loop.graph);
    g_loop = LoopGraph{};
}

}  // namespace

namespace {

// Builds [condition (rounds = 0)] -> while { embed, step, condition (rounds += 1) } by
// capture on `cs`.  Returns a MOESTEP_E* code for invalid arguments, else OK with the
// CUDA status in *err (graph and exec set on success; nothing kept on failure).
int build_loop_graph(const moestep_dims* dims, int R, int n_layers, const moestep_layer* layers, const void* Wlm,
                     const void* emb, const void* pos, int mask_id, const float* top_p, float logit_scale,
                     float threshold, int max_rounds, int32_t* tokens, uint8_t* masked, int32_t* rounds, void* ws,
                     size_t ws_bytes, const Layout& L, cudaStream_t cs, cudaGraph_t* g_out, cudaGraphExec_t* ex_out,
                     cudaError_t* err) {
    cudaGraph_t g = nullptr;
    cudaGraphConditionalHandle h = 0;
    int rc = MOESTEP_OK;
    cudaError_t e = cudaGraphCreate(&g, 0);
    if (e == cudaSuccess) e = cudaGraphConditionalHandleCreate(&h, g, 0, 0);
    if (e == cudaSuccess) e = cudaStreamBeginCaptureToGraph(cs, g, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed);
    if (e == cudaSuccess) {
        const cudaError_t le = launch_loop_cond(h, masked, L.T, rounds, max_rounds, 0, cs);
        cudaGraph_t got = nullptr;
        e = cudaStreamEndCapture(cs, &got);
        if (e == cudaSuccess) e = le;
    }
    cudaGraphNode_t first = nullptr;
    size_t n_nodes = 1;
    if (e == cudaSuccess) e = cudaGraphGetNodes(g, &first, &n_nodes);
    cudaGraphNodeParams cp{};
    cp.type = cudaGraphNodeTypeConditional;
    cp.conditional.handle = h;
    cp.conditional.type = cudaGraphCondTypeWhile;
    cp.conditional.size = 1;
    cudaGraphNode_t wnode = nullptr;
    if (e == cudaSuccess) e = cudaGraphAddNode(&wnode, g, &first, nullptr, 1, &cp);
    if (e == cudaSuccess)
        e = cudaStreamBeginCaptureToGraph(cs, cp.conditional.phGraph_out[0], nullptr, nullptr, 0,
                                          cudaStreamCaptureModeRelaxed);
    if (e == cudaSuccess) {
        float* hb = at<float>(ws, L.loop_h);
        rc = block_embed(dims, R, tokens, masked, emb, pos, mask_id, hb, cs);
        if (rc == MOESTEP_OK)
            rc = block_decode_step(dims, R, n_layers, layers, Wlm, top_p, logit_scale, threshold, hb, nullptr,
                                        tokens, masked, at<int32_t>(ws, L.loop_choice), at<float>(ws, L.loop_conf),
                                        at<uint8_t>(ws, L.loop_accept), at<int32_t>(ws, L.loop_ncomm), nullptr, ws,
                                        ws_bytes, cs);
        cudaError_t le = cudaSuccess;
        if (rc == MOESTEP_OK) le = launch_loop_cond(h, masked, L.T, rounds, max_rounds, 1, cs);
        cudaGraph_t got = nullptr;
        e = cudaStreamEndCapture(cs, &got);
        if (e == cudaSuccess) e = le;
    }
    cudaGraphExec_t ex = nullptr;
    if (e == cudaSuccess && rc == MOESTEP_OK) e = cudaGraphInstantiate(&ex, g, 0);
    if (e != cudaSuccess || rc != MOESTEP_OK) {
        if (g) cudaGraphDestroy(g);
        *err = e;
        return rc;
    }
    *g_out = g;
    *ex_out = ex;
    *err = cudaSuccess;
    return MOESTEP_OK;
}

}  // namespace

extern "C" {

int moestep_workspace_size(const moestep_dims* dims, int R, size_t* bytes) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (bytes == nullptr) return MOESTEP_EINVAL;
    *bytes = make_layout(*dims, R).total;
    return MOESTEP_OK;
}

int moestep_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 512) return MOESTEP_EWORKSPACE;
    MOESTEP_CK(cudaMemsetAsync(ws, 0, 512, static_cast<cudaStream_t>(stream)));
    return MOESTEP_OK;
}

int moe_block_route(const moestep_dims* dims, int T, const void* x, const void* Wr, int32_t* idx, float* mass,
                    float* gate, float* logits, void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    if (T <= 0) return MOESTEP_EINVAL;
    const int R = (T + dims->P - 1) / dims->P;
    MOESTEP_TRY(check_R(dims, R));
    if (!x || !Wr || !idx || !mass || !gate) return MOESTEP_EINVAL;
    if (!aligned16(x) || !aligned16(Wr)) return MOESTEP_EALIGN;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    MOESTEP_CK(cudaMemsetAsync(at<char>(ws, c.L.counters), 0, c.L.counters_bytes, c.s));
    return run_route(c, T, x, Wr, idx, mass, gate, logits);
}

int moe_route_from_logits(const moestep_dims* dims, int T, const float* logits, int32_t* idx, float* mass, float* gate,
                          void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    if (T <= 0) return MOESTEP_EINVAL;
    const int R = (T + dims->P - 1) / dims->P;
    MOESTEP_TRY(check_R(dims, R));
    if (!logits || !idx || !mass || !gate) return MOESTEP_EINVAL;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    MOESTEP_TRY(device_check(nullptr));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_begin(0, s);
    cudaError_t e = launch_topk_from_logits(logits, T, dims->E, dims->k, idx, mass, gate, s);
    prof_end(0, s);
    MOESTEP_CK(e);
    g_launches.fetch_add(1);
    return MOESTEP_OK;
}

int coreset_select(const moestep_dims* dims, int R, const float* top_p, const int32_t* idx, const float* mass,
                   int32_t* n_sel, int32_t* sel, uint8_t* survive, float* gate_rr, void* ws, size_t ws_bytes,
                   void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (!top_p || !idx || !mass || !n_sel || !sel || !survive || !gate_rr) return MOESTEP_EINVAL;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    MOESTEP_CK(cudaMemsetAsync(at<char>(ws, c.L.counters), 0, c.L.counters_bytes, c.s));
    return run_coreset(c, R, top_p, idx, mass, n_sel, sel, survive, gate_rr);
}

int moe_block_ffn(const moestep_dims* dims, int R, const void* x, const moestep_layer* layer, const float* gate_rr,
                  float* out, void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (!x || !gate_rr || !out) return MOESTEP_EINVAL;
    MOESTEP_TRY(layer_ok(dims, layer));
    if (!aligned16(x) || !aligned16(out)) return MOESTEP_EALIGN;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    MOESTEP_TRY(run_experts(c, R, x, layer));
    MOESTEP_LAUNCH(5, launch_combine(0, act_dtype(dims->dtype), c.L.T, dims->H, dims->k, at<float>(ws, c.L.y),
                                     at<int32_t>(ws, c.L.slot_of), at<int32_t>(ws, c.L.slot_sh), gate_rr,
                                     dims->Is > 0, nullptr, nullptr, nullptr, nullptr, out, c.s));
    return MOESTEP_OK;
}

int lm_head_commit(const moestep_dims* dims, int R, const void* hidden, const void* Wlm, float logit_scale,
                   float threshold, int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf, uint8_t* accept,
                   int32_t* n_committed, float* logits, void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (!hidden || !Wlm || !tokens || !masked || !choice || !conf || !accept || !n_committed) return MOESTEP_EINVAL;
    if (!thr_ok(threshold) || !std::isfinite(logit_scale)) return MOESTEP_EINVAL;
    if (!aligned16(hidden) || !aligned16(Wlm)) return MOESTEP_EALIGN;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    MOESTEP_CK(cudaMemsetAsync(at<char>(ws, c.L.counters), 0, c.L.counters_bytes, c.s));
    return run_lm_commit(c, R, hidden, Wlm, logit_scale, threshold, tokens, masked, choice, conf, accept,
                         n_committed, logits);
}

int lm_commit_from_logits(const moestep_dims* dims, int R, const float* logits, float threshold, int32_t* tokens,
                          uint8_t* masked, int32_t* choice, float* conf, uint8_t* accept, int32_t* n_committed,
                          void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (!logits || !tokens || !masked || !choice || !conf || !accept || !n_committed) return MOESTEP_EINVAL;
    if (!thr_ok(threshold)) return MOESTEP_EINVAL;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    const int T = R * dims->P;
    MOESTEP_CK(cudaMemsetAsync(at<char>(ws, c.L.counters), 0, c.L.counters_bytes, c.s));
    MOESTEP_LAUNCH(8, launch_partials_from_logits(logits, T, dims->V, at<float>(ws, c.L.pmax), at<int>(ws, c.L.parg),
                                                  at<float>(ws, c.L.psum), c.s));
    MOESTEP_LAUNCH(7, launch_commit(R, dims->P, (dims->V + kLogitTile - 1) / kLogitTile, at<float>(ws, c.L.pmax),
                                    at<int>(ws, c.L.parg), at<float>(ws, c.L.psum), threshold, tokens, masked, choice,
                                    conf, accept, n_committed, at<int>(ws, c.L.counters) + c.L.route_groups + 1,
                                    c.s));
    return MOESTEP_OK;
}

int block_embed(const moestep_dims* dims, int R, const int32_t* tokens, const uint8_t* masked, const void* emb,
                const void* pos, int mask_id, float* h, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (!tokens || !masked || !emb || !pos || !h) return MOESTEP_EINVAL;
    if (mask_id < 0 || mask_id >= dims->V) return MOESTEP_EINVAL;
    MOESTEP_TRY(device_check(nullptr));
    Ctx c{dims, Layout{}, nullptr, static_cast<cudaStream_t>(stream), 0};
    MOESTEP_LAUNCH(8, launch_embed(act_dtype(dims->dtype), R * dims->P, dims->H, dims->P, dims->V, tokens, masked, emb, pos,
                                   mask_id, h, c.s));
    return MOESTEP_OK;
}

int block_decode_step(const moestep_dims* dims, int R, int n_layers, const moestep_layer* layers, const void* Wlm,
                      const float* top_p, float logit_scale, float threshold, const float* h_in, float* h_out,
                      int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf, uint8_t* accept,
                      int32_t* n_committed, const moestep_trace* trace, void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (n_layers < 0 || (n_layers > 0 && !layers)) return MOESTEP_EINVAL;
    if (!Wlm || !top_p || !h_in || !tokens || !masked || !choice || !conf || !accept || !n_committed)
        return MOESTEP_EINVAL;
    if (!thr_ok(threshold) || !std::isfinite(logit_scale)) return MOESTEP_EINVAL;
    if (!aligned16(h_in) || !aligned16(Wlm) || (h_out && !aligned16(h_out))) return MOESTEP_EALIGN;
    for (int l = 0; l < n_layers; ++l) MOESTEP_TRY(layer_ok(dims, &layers[l]));
    if (trace && trace->hidden && !aligned16(trace->hidden)) return MOESTEP_EALIGN;
    if (trace && ((trace->x && !aligned16(trace->x)) || (trace->h && !aligned16(trace->h)))) return MOESTEP_EALIGN;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    int sms = 0;
    MOESTEP_TRY(device_check(&sms));
    Ctx c{dims, make_layout(*dims, R), ws, static_cast<cudaStream_t>(stream), sms};
    const Layout& L = c.L;
    const int T = L.T, k = dims->k;
    float* hres = at<float>(ws, L.hres);
    void* x = at<void>(ws, L.x);
    MOESTEP_CK(cudaMemsetAsync(at<char>(ws, L.counters), 0, L.counters_bytes, c.s));
    float* hid_trace = trace ? trace->hidden : nullptr;
    const bool fused_head = g_layer_head == 2 && n_layers > 0 &&
                            route_combine_eligible(act_dtype(dims->dtype), T, dims->H, dims->E, k);
    if (!fused_head)
        MOESTEP_LAUNCH(5, launch_combine(2, act_dtype(dims->dtype), T, dims->H, k, nullptr, nullptr, nullptr, nullptr, 0, h_in,
                                         hres, x, n_layers == 0 ? hid_trace : nullptr, nullptr, c.s));
    const size_t act_row = static_cast<size_t>(dims->H) * (dims->dtype == MOESTEP_F32 ? 4 : 2);
    for (int l = 0; l < n_layers; ++l) {
        int32_t* idx = (trace && trace->idx) ? trace->idx + static_cast<size_t>(l) * T * k : at<int32_t>(ws, L.idx);
        int32_t* nsel = (trace && trace->n_sel) ? trace->n_sel + static_cast<size_t>(l) * R : at<int32_t>(ws, L.nsel);
        int32_t* sel = (trace && trace->sel) ? trace->sel + static_cast<size_t>(l) * R * dims->E : at<int32_t>(ws, L.sel);
        const bool last = l == n_layers - 1;
        if (fused_head) {
            // the combine of layer l-1 (or the input norm) runs inside the layer-l router launch
            MOESTEP_TRY(run_route_combine(c, l == 0 ? 2 : 1, h_in, layers[l].Wr, idx, l));
        } else {
            MOESTEP_TRY(run_route(c, T, x, layers[l].Wr, idx, at<float>(ws, L.mass), at<float>(ws, L.gate), nullptr));
        }
        // layer l's input and residual stream are complete once its router has run
        if (trace && trace->x)
            MOESTEP_CK(cudaMemcpyAsync(static_cast<char*>(trace->x) + l * T * act_row, x, T * act_row,
                                       cudaMemcpyDeviceToDevice, c.s));
        if (trace && trace->h)
            MOESTEP_CK(cudaMemcpyAsync(trace->h + static_cast<size_t>(l) * T * dims->H, hres,
                                       sizeof(float) * T * dims->H, cudaMemcpyDeviceToDevice, c.s));
        MOESTEP_TRY(run_coreset(c, R, top_p, idx, at<float>(ws, L.mass), nsel, sel,
                                at<uint8_t>(ws, L.survive), at<float>(ws, L.gaterr), layers[l].Wgu,
                                last ? nullptr : layers[l + 1].Wr));
        MOESTEP_TRY(run_experts(c, R, x, &layers[l], l));
        if (!fused_head || last)
            MOESTEP_LAUNCH(5, launch_combine(1, act_dtype(dims->dtype), T, dims->H, k, at<float>(ws, L.y),
                                             at<int32_t>(ws, L.slot_of), at<int32_t>(ws, L.slot_sh),
                                             at<float>(ws, L.gaterr), dims->Is > 0, nullptr, hres, x,
                                             last ? hid_trace : nullptr, nullptr, c.s));
    }
    MOESTEP_TRY(run_lm_commit(c, R, x, Wlm, logit_scale, threshold, tokens, masked, choice, conf, accept, n_committed,
                              nullptr));
    if (h_out) MOESTEP_CK(cudaMemcpyAsync(h_out, hres, sizeof(float) * T * dims->H, cudaMemcpyDeviceToDevice, c.s));
    return MOESTEP_OK;
}

int block_decode_loop(const moestep_dims* dims, int R, int n_layers, const moestep_layer* layers, const void* Wlm,
                      const void* emb, const void* pos, int mask_id, const float* top_p, float logit_scale,
                      float threshold, int max_rounds, int32_t* tokens, uint8_t* masked, int32_t* rounds,
                      void* ws, size_t ws_bytes, void* stream) {
    MOESTEP_TRY(check_dims(dims));
    MOESTEP_TRY(check_R(dims, R));
    if (max_rounds < 0 || !rounds || !emb || !pos || !tokens || !masked) return MOESTEP_EINVAL;
    if (n_layers < 0 || (n_layers > 0 && !layers)) return MOESTEP_EINVAL;
    MOESTEP_TRY(check_ws(dims, R, ws, ws_bytes));
    MOESTEP_TRY(device_check(nullptr));
    int dev = 0;
    MOESTEP_CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOESTEP_EDEVICE;
    const Layout L = make_layout(*dims, R);
    std::vector<unsigned char> key;
    key_add(key, dev);
    key_add(key, *dims);
    key_add(key, R);
    key_add(key, n_layers);
    for (int l = 0; l < n_layers; ++l) key_add(key, layers[l]);
    const void* ptrs[] = {Wlm, emb, pos, top_p, tokens, masked, rounds, ws};
    for (const void* q : ptrs) key_add(key, q);
    key_add(key, ws_bytes);
    key_add(key, mask_id);
    key_add(key, logit_scale);
    key_add(key, threshold);
    key_add(key, max_rounds);
    key_add(key, g_layer_head);
    key_add(key, g_timeout_ns);
    std::lock_guard<std::mutex> lock(g_loop_mu);
    if (g_loop.exec == nullptr || g_loop.key != key) {
        loop_release();
        if (g_capture_stream[dev] == nullptr)
            MOESTEP_CK(cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking));
        cudaStream_t cs = g_capture_stream[dev];
        const int prof_mask = g_prof.mask;  // event records are not allowed in a loop body
        g_prof.mask = 0;
        cudaGraph_t g = nullptr;
        cudaGraphExec_t ex = nullptr;
        int rc = MOESTEP_OK;
        cudaError_t e = cudaSuccess;
        // with programmatic edges between the round's kernels; without, if the graph refuses them
        for (int attempt = 0; attempt < 2; ++attempt) {
            g_launch_pdl = attempt == 0;
            rc = build_loop_graph(dims, R, n_layers, layers, Wlm, emb, pos, mask_id, top_p, logit_scale, threshold,
                                  max_rounds, tokens, masked, rounds, ws, ws_bytes, L, cs, &g, &ex, &e);
            if (rc != MOESTEP_OK || e == cudaSuccess) break;
            cudaGetLastError();
        }
        g_launch_pdl = true;
        g_prof.mask = prof_mask;
        if (rc != MOESTEP_OK) return rc;
        if (e != cudaSuccess) {
            g_last_cuda = static_cast<int>(e);
            return MOESTEP_ECUDA;
        }
        g_loop.key = std::move(key);
        g_loop.graph = g;
        g_loop.exec = ex;
    }
    MOESTEP_CK(cudaGraphLaunch(g_loop.exec, static_cast<cudaStream_t>(stream)));
    return MOESTEP_OK;
}

int moestep_read_device_error(void* ws, size_t ws_bytes, void* stream, int* word) {
    if (!ws || ws_bytes < 256 || !word) return MOESTEP_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int bits = 0;
    MOESTEP_CK(cudaMemcpyAsync(&bits, ws, sizeof(int), cudaMemcpyDeviceToHost, s));
    MOESTEP_CK(cudaStreamSynchronize(s));
    MOESTEP_CK(cudaMemsetAsync(ws, 0, 16 * sizeof(int), s));
    *word = (bits & 0xff) ? MOESTEP_ETIMEOUT : (bits ? MOESTEP_EDEVINPUT : MOESTEP_OK);
    return MOESTEP_OK;
}

const char* moestep_error_string(int code) {
    switch (code) {
        case MOESTEP_OK: return "ok";
        case MOESTEP_EINVAL: return "invalid argument";
        case MOESTEP_EWORKSPACE: return "workspace missing, misaligned or too small";
        case MOESTEP_EALIGN: return "tensor not 16-byte aligned";
        case MOESTEP_ECUDA: return "CUDA call failed";
        case MOESTEP_EDEVICE: return "device is not an sm_103 GPU";
        case MOESTEP_EUNSUPPORTED: return "shape not supported";
        case MOESTEP_ETIMEOUT: return "a bounded wait inside a kernel timed out";
        case MOESTEP_EDEVINPUT: return "device input held an out-of-range value";
        default: return "unknown error";
    }
}

int moestep_last_cuda_error(void) { return g_last_cuda; }

long long moestep_launch_count(void) { return g_launches.load(); }

int moestep_prof_enable(int kernel_mask) {
    g_prof.mask = kernel_mask & ((1 << MOESTEP_PROF_KERNELS) - 1);
    if (g_prof.mask) {
        g_prof.next = 0;
        g_prof.kid.clear();
        g_prof.start.clear();
        g_prof.stop.clear();
        for (auto& p : g_prof.pending) p = nullptr;
    }
    return MOESTEP_OK;
}

int moestep_prof_read(int kernel_id, int* launches, double* total_ms) {
    if (kernel_id < 0 || kernel_id >= MOESTEP_PROF_KERNELS || !launches || !total_ms) return MOESTEP_EINVAL;
    int n = 0;
    double ms = 0.0;
    for (size_t i = 0; i < g_prof.kid.size(); ++i) {
        if (g_prof.kid[i] != kernel_id) continue;
        MOESTEP_CK(cudaEventSynchronize(g_prof.stop[i]));
        float t = 0.f;
        MOESTEP_CK(cudaEventElapsedTime(&t, g_prof.start[i], g_prof.stop[i]));
        ms += t;
        ++n;
    }
    *launches = n;
    *total_ms = ms;
    return MOESTEP_OK;
}

int moestep_set_route_fusion(int mode) {
    if (mode != 0 && mode != 2) return MOESTEP_EINVAL;
    g_layer_head = mode;
    return MOESTEP_OK;
}

int moestep_route_fusion(void) { return g_layer_head; }

// Test hook: limit of every bounded wait in the tensor-core kernels (ns).
int moestep_set_wait_timeout_ns(unsigned long long ns) {
    g_timeout_ns = ns;
    return MOESTEP_OK;
}

}  // extern "C"
