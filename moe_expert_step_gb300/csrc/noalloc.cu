// Router entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a scratch buffer: plugins
// inside a host application that owns every device allocation, or embedded
// runtimes whose device-memory budget is fixed up front.  For them,
// moe_block_route_noalloc needs no workspace:
// its scratch (the router logits and the per-token-group completion counters)
// lives in one fixed-size array in this file, which every GPU that loads the
// library holds until the process exits.  The caller still passes x, Wr and
// the outputs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "moestep.h"

namespace {

constexpr int kMaxLogits = 131072;  // T * E of one call (512 KiB of fp32 logits)
constexpr int kMaxGroups = 2048;    // completion counters, one per kRouteTokensPerCta tokens

struct RouteScratch {
    float logits[kMaxLogits];
    int counters[kMaxGroups];
};

// One copy per CUDA context.  In host code this name is only a stand-in: host
// code uses the device address looked up below, never the symbol itself.
static __device__ __align__(256) RouteScratch g_route_scratch;

// The array's device address belongs to the CUDA context that loaded this
// module, not to the device number: a context the caller makes current
// itself, or the primary context re-created after cudaDeviceReset, holds its
// own copy at another address.  So the address is cached per context, under
// the context's process-unique id (cuCtxGetId; ids are never reused, unlike
// context handles), and looked up again for a context not seen before.
struct CachedAddress {
    unsigned long long ctx_id;
    RouteScratch* addr;
};
constexpr int kCacheSlots = 64;
std::mutex g_mu;
CachedAddress g_cache[kCacheSlots] = {};
int g_cache_used = 0, g_cache_next = 0;

PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_id_once;

// Id of the calling thread's current context; false if there is none (or the
// driver call is unavailable).
bool current_context_id(unsigned long long* id) {
    std::call_once(g_ctx_id_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    return g_ctx_id != nullptr && g_ctx_id(nullptr, id) == CUDA_SUCCESS;
}

int lookup(RouteScratch** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || p == nullptr) {
        moestep::set_last_cuda(static_cast<int>(e != cudaSuccess ? e : cudaErrorInvalidSymbol));
        return MOESTEP_ECUDA;
    }
    *out = static_cast<RouteScratch*>(p);
    return MOESTEP_OK;
}

// The array's device address in the current context (looked up once per context).
int scratch_address(RouteScratch** out) {
    unsigned long long id = 0;
    if (!current_context_id(&id)) {
        // no current context yet: the symbol lookup makes the current device's
        // primary context current, then its id can be read
        RouteScratch* a = nullptr;
        const int rc = lookup(&a);
        if (rc != MOESTEP_OK) return rc;
        if (!current_context_id(&id)) {
            moestep::set_last_cuda(static_cast<int>(cudaErrorDeviceUninitialized));
            return MOESTEP_ECUDA;
        }
    }
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_cache_used; ++i)
        if (g_cache[i].ctx_id == id) {
            *out = g_cache[i].addr;
            return MOESTEP_OK;
        }
    RouteScratch* a = nullptr;
    const int rc = lookup(&a);
    if (rc != MOESTEP_OK) return rc;
    const int slot = g_cache_used < kCacheSlots ? g_cache_used++ : (g_cache_next++ % kCacheSlots);
    g_cache[slot] = CachedAddress{id, a};
    *out = a;
    return MOESTEP_OK;
}

}  // namespace

extern "C" int moe_block_route_noalloc(const moestep_dims* dims, int T, const void* x, const void* Wr, int32_t* idx,
                                       float* mass, float* gate, float* logits, void* stream) {
    int rc = moestep::validate_dims(dims);
    if (rc != MOESTEP_OK) return rc;
    if (T <= 0 || !x || !Wr || !idx || !mass || !gate) return MOESTEP_EINVAL;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(Wr)) & 15u) return MOESTEP_EALIGN;
    const int groups = (T + moestep::kRouteTokensPerCta - 1) / moestep::kRouteTokensPerCta;
    if (static_cast<long long>(T) * dims->E > kMaxLogits || groups > kMaxGroups) return MOESTEP_EUNSUPPORTED;
    if ((rc = moestep::device_ok(nullptr)) != MOESTEP_OK) return rc;
    RouteScratch* s = nullptr;
    if ((rc = scratch_address(&s)) != MOESTEP_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the completion counters must start at zero; the logits are fully written before they are read
    cudaError_t e = cudaMemsetAsync(s->counters, 0, sizeof(int) * groups, st);
    if (e != cudaSuccess) {
        moestep::set_last_cuda(static_cast<int>(e));
        return MOESTEP_ECUDA;
    }
    float* lg = logits ? logits : s->logits;
    moestep::prof_begin(0, st);  // kernel id 0 (route), as for moe_block_route
    e = moestep::launch_route(dims->dtype == MOESTEP_FP8 ? MOESTEP_BF16 : dims->dtype, x, Wr, T, dims->H, dims->E,
                              dims->k, lg, idx, mass, gate, s->counters, nullptr, st);
    moestep::prof_end(0, st);
    if (e != cudaSuccess) {
        moestep::set_last_cuda(static_cast<int>(e));
        return MOESTEP_ECUDA;
    }
    moestep::count_launch();
    return MOESTEP_OK;
}
