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

// One copy per device.  In host code this name is only a stand-in: host code
// uses the device address looked up below, never the symbol itself.
static __device__ __align__(256) RouteScratch g_route_scratch;

std::mutex g_mu;
RouteScratch* g_addr[64] = {};  // device address of g_route_scratch, per device

// Looks up the array's device address on the current device (once per device).
int scratch_address(RouteScratch** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOESTEP_ECUDA;
    if (dev < 0 || dev >= 64) return MOESTEP_EDEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOESTEP_ECUDA;
        g_addr[dev] = static_cast<RouteScratch*>(p);
    }
    *out = g_addr[dev];
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
    if (cudaMemsetAsync(s->counters, 0, sizeof(int) * groups, st) != cudaSuccess) return MOESTEP_ECUDA;
    float* lg = logits ? logits : s->logits;
    if (moestep::launch_route(dims->dtype == MOESTEP_FP8 ? MOESTEP_BF16 : dims->dtype, x, Wr, T, dims->H, dims->E, dims->k, lg, idx, mass, gate, s->counters,
                              nullptr, st) != cudaSuccess)
        return MOESTEP_ECUDA;
    return MOESTEP_OK;
}
