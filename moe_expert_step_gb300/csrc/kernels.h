// Host-side launch functions of the moestep kernels (one translation unit per
// kernel family; api.cu validates arguments and calls these).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moestep.h"

namespace moestep {

// ------------------------------------------------------------------ grouped tcgen05 GEMM
enum GemmMode { kGateUp = 0, kDown = 1, kLmHead = 2, kExperts = 3, kExpertsF8 = 4 };

// kExperts: one persistent launch runs every gate/up unit (a[0] routed / a[1]
// shared weights, b[0] gathered activations), then every down unit (a[2] / a[3],
// b[1] = SwiGLU output); a down unit of a chunk starts once all of that
// chunk's gate/up units have signalled completion.  kLmHead uses a[0] and b[0].
// kExpertsF8: as kExperts with FP8 E4M3 weight maps (a[0..3], boxes of 128 rows x
// 128 bytes, 128-byte swizzle; K blocks of 128), f16 activations in b[0..1], per-row
// scales sc[0..3] (same order as a[0..3]) applied to the accumulators, and the
// SwiGLU output stored as f16.
struct TensorMaps {
    CUtensorMap a[4];
    // token rows: [0] gathered rows, [1] SwiGLU rows, in 16-row boxes; the FP8 expert launch
    // also [2], [3] in 32-row and [4], [5] in 64-row boxes
    CUtensorMap b[6];
};

struct GemmParams {
    // expert modes: work plan written by the coreset kernel
    const int* plan;       // [0] routed chunks, [1] shared chunks, [2] slots
    const int4* chunks;    // {expert, first slot, slots, 0}; routed chunks first, then shared
    int routed_tiles;      // M tiles per routed chunk
    int shared_tiles;      // M tiles per shared chunk
    int routed_kb;         // 64-wide K blocks per routed unit (LM head: per unit)
    int shared_kb;         // 64-wide K blocks per shared unit
    int rows_per_expert;   // rows of one routed expert in the A tensor
    int tile_rows;         // row step between M tiles (128)
    // LM head
    int lm_chunks;         // position chunks
    int lm_tiles;          // vocabulary tiles of 128 rows
    int n_pos;             // positions (rows of B)
    int V;
    float scale;
    float* pmax;           // [lm_tiles * 4][n_pos]: one partial per 32-row slice
    int* parg;
    float* psum;
    float* logits;         // optional [n_pos][V]
    // outputs of expert modes: act (bf16, gate/up) or y (fp32, down)
    void* out;
    int out_ld;
    // kExperts: the down half (tiles / K blocks / rows per expert / output y) and the per-chunk
    // completion counters of the gate/up half (zeroed by the gather kernel before the launch)
    int dn_routed_tiles, dn_shared_tiles, dn_routed_kb, dn_shared_kb, dn_rows_per_expert;
    void* out2;
    int out2_ld;
    int* done;
    int* err;
    unsigned long long timeout_ns;
    const float* sc[4];    // kExpertsF8: row scales of the weights of a[0..3]
    int* unit_ctr;         // kExperts: next unit to hand out (zeroed with the chunk counters)
};

cudaError_t launch_tc_gemm(int mode, int nch, const TensorMaps& maps, const GemmParams& p, int grid, cudaStream_t s);
int tc_gemm_smem_bytes(int nch);

// ------------------------------------------------------------------ routing / coreset / plan
constexpr int kRouteTokensPerCta = 4;  // tokens per router CTA = tokens per completion counter
struct CoresetArgs {
    int R, P, k, E, T;
    const float* top_p;
    const int32_t* idx;
    const float* mass;
    int32_t* n_sel;
    int32_t* sel;
    uint8_t* survive;
    float* gate_rr;
    int32_t* slot_of;   // [T][k]
    int32_t* slot_sh;   // [T]
    int32_t* slot_tok;  // [max slots]
    int32_t* slot_exp;  // [max slots]
    int4* chunks;
    int* plan;
    int* counter;
    int nch;
    int has_shared;
    int* err;
    // optional L2 hints: CTAs R .. R+pf_ctas-1 of the coreset launch hint the
    // weights (pf_stride bytes from pf_base + e * pf_stride) of the pf_experts
    // lowest-id experts that any token picked, while CTAs 0 .. R-1 run the coreset
    const char* pf_base;
    long long pf_stride;
    int pf_experts;
    int pf_ctas;
    const char* pf_next;      // also hinted by those CTAs: pf_next_bytes from here (the next layer's router)
    long long pf_next_bytes;
};

cudaError_t launch_route(int dtype, const void* x, const void* Wr, int T, int H, int E, int k, float* logits,
                         int32_t* idx, float* mass, float* gate, int* counters, int* err, cudaStream_t s);
cudaError_t launch_topk_from_logits(const float* logits, int T, int E, int k, int32_t* idx, float* mass,
                                    float* gate, cudaStream_t s);
// experts whose gate/up weights the coreset launch hints into L2 in the block step
// (measured best: 32 of 4 MiB bf16 gate/up pairs, 48 of 2 MiB FP8 ones; more evicts them again)
constexpr int kCoresetPrefetchExperts = 32;
constexpr int kCoresetPrefetchExpertsF8 = 48;
cudaError_t launch_coreset(const CoresetArgs& a, cudaStream_t s);
int coreset_smem_bytes(int E, int T);
// The previous layer's combine + RMSNorm and the router (logits, softmax, top-k) in
// one cluster launch over 8-token tiles (bf16 activations).
struct RouteCombineArgs {
    int mode;                       // 1: h += experts' outputs, x = RMSNorm(h); 2: h = h_in, x = RMSNorm(h)
    const float* y;
    const int32_t* slot_of;
    const int32_t* slot_sh;
    const float* gate_rr_prev;
    int has_shared;
    const float* h_in;
    float* hres;
    __nv_bfloat16* x;
    const __nv_bfloat16* Wr;
    int T, H, E, k;
    float* logits;                  // optional [T][E]
    int32_t* idx;
    float* mass;
    float* gate;
    // mode 1, optional: once *plan_flag >= plan_value (set by the previous layer's gather launch:
    // its coreset completed, so slot_of / slot_sh / gate_rr_prev are final) they are read before
    // waiting for the previous kernel; without the flag, or if the bounded wait runs out, after it
    const int* plan_flag;
    int plan_value;
    unsigned long long timeout_ns;
};
int route_combine_eligible(int act_dtype, int T, int H, int E, int k);
cudaError_t launch_route_combine(const RouteCombineArgs& a, cudaStream_t s);

// xp[slot] = x[slot_tok[slot]] for the plan's slots; zeroes done[0..n_done)
// (the fused expert launch's counters; NULL: none); release-stores flag_value into *flag
// (NULL: none) once the preceding coreset launch has completed
cudaError_t launch_gather(int dtype, const void* x, int H, const int32_t* slot_tok, const int* plan,
                          int max_slots, void* xp, int* done, int n_done, int* flag, int flag_value,
                          cudaStream_t s);

// ------------------------------------------------------------------ combine / norm / embed
// mode 0: out = routed + shared; mode 1: h += routed + shared, x = RMSNorm(h); mode 2: h = h_in, x = RMSNorm(h)
cudaError_t launch_combine(int mode, int dtype, int T, int H, int k, const float* y, const int32_t* slot_of,
                           const int32_t* slot_sh, const float* gate_rr, int has_shared, const float* h_in,
                           float* h, void* x, float* x_f32, float* out, cudaStream_t s);
cudaError_t launch_embed(int dtype, int T, int H, int P, int V, const int32_t* tokens, const uint8_t* masked,
                         const void* emb, const void* pos, int mask_id, float* h, cudaStream_t s);

// ------------------------------------------------------------------ fp32 FFMA path
// act[slot][i] = silu(gate_i . xp[slot]) * (up_i . xp[slot]) for the slot's expert (interleaved gate/up rows)
cudaError_t launch_f32_gateup(int H, int E, int I, int Is, int max_slots, const float* xp, const int32_t* slot_exp,
                              const int* plan, const float* Wgu, const float* Wsgu, float* act, int act_ld,
                              cudaStream_t s);
// y[slot][h] = Wd_e[h] . act[slot]
cudaError_t launch_f32_down(int H, int E, int I, int Is, int max_slots, const float* act, int act_ld,
                            const int32_t* slot_exp, const int* plan, const float* Wd, const float* Wsd, float* y,
                            cudaStream_t s);
cudaError_t launch_f32_lm_logits(int T, int H, int V, const float* hidden, const float* Wlm, float scale,
                                 float* logits, cudaStream_t s);

// ------------------------------------------------------------------ softmax partials / commit
constexpr int kLogitTile = 2048;  // vocabulary entries per partial when reducing given logits
cudaError_t launch_partials_from_logits(const float* logits, int T, int V, float* pmax, int* parg, float* psum,
                                        cudaStream_t s);
cudaError_t launch_commit(int R, int P, int n_tiles, const float* pmax, const int* parg, const float* psum,
                          float threshold, int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf,
                          uint8_t* accept, int32_t* n_committed, int* counters, cudaStream_t s);

// ------------------------------------------------------------------ shared host checks (api.cu)
int validate_dims(const moestep_dims* d);  // MOESTEP_OK or the code every entry point returns
int device_ok(int* sms);                   // current device is sm_103; *sms = its SM count

// ------------------------------------------------------------------ profiling hooks (api.cu)
void prof_begin(int kid, cudaStream_t s);
void prof_end(int kid, cudaStream_t s);
// Bookkeeping shared by every entry point: the cudaError_t that moestep_last_cuda_error()
// reports (this host thread), and the count that moestep_launch_count() reports.
void set_last_cuda(int err);
void count_launch();

// Round loop: sets the while-node condition h to (any masked && rounds < max_rounds);
// add = 1 increments *rounds first, add = 0 sets it to 0.
cudaError_t launch_loop_cond(cudaGraphConditionalHandle h, const uint8_t* masked, int T, int32_t* rounds,
                             int max_rounds, int add, cudaStream_t s);

}  // namespace moestep
