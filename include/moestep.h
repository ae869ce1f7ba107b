/*
 * moestep.h - C ABI of the block-diffusion MoE denoising step for GB300 (sm_103a).
 *
 * One denoising round over a block of P masked positions per request: router
 * softmax/top-k, block coreset expert selection, routed + shared SwiGLU
 * experts (each selected expert's weights streamed from HBM once per block),
 * residual + RMSNorm between layers, LM head, and the LowConfidence commit.
 *
 * Sources (cited by page title and section):
 *   [AIT] aitujian.cn engineering analysis of Clover-35B-A3B-Preview:
 *         section 二 (block diffusion), 三 (LowConfidence decode loop),
 *         四 (40 layers, 256 routed experts, top-8, one shared expert),
 *         五 (a block touches the union of its tokens' experts).
 *   [GRM] "What Is Clover-35B-A3B? Block Diffusion on a Qwen3.6 MoE":
 *         "How does confidence-threshold block decoding work?",
 *         "What is the MoE coreset and why does it matter?".
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer unless marked "host".
 *   - The caller owns all memory.  The library allocates no device memory;
 *     scratch lives in a caller-provided workspace of at least
 *     moestep_workspace_size() bytes, 256-byte aligned.  A workspace must not
 *     be used by two calls that may run concurrently.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Arguments are validated on the host before anything
 *     is launched; on a non-zero return nothing was launched.
 *   - Tensors are dense row-major ("[A][B]" = B contiguous).  bf16 tensors
 *     used as tensor-core operands must be 16-byte aligned (TMA rule).
 *   - Returns MOESTEP_OK (0) or a negative MOESTEP_E* code.  Faults found on
 *     the device (an out-of-range index in fed input, a bounded wait that ran
 *     out) are recorded in the workspace's error word: read it with
 *     moestep_read_device_error().  A new workspace is zeroed once with
 *     moestep_workspace_init() before its first use.
 *   - Decisions taken on floating point are deterministic: top-k, expert
 *     ranking, argmax and the commit fallback break ties toward the lower
 *     index; coreset sums are exact integers.
 */
#ifndef MOESTEP_H
#define MOESTEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOESTEP_OK 0
#define MOESTEP_EINVAL (-1)       /* bad argument (null pointer, size out of range, bad top_p/threshold) */
#define MOESTEP_EWORKSPACE (-2)   /* workspace NULL, misaligned or smaller than moestep_workspace_size() */
#define MOESTEP_EALIGN (-3)       /* a tensor-core operand is not 16-byte aligned */
#define MOESTEP_ECUDA (-4)        /* a CUDA runtime/driver call failed (moestep_last_cuda_error()) */
#define MOESTEP_EDEVICE (-5)      /* current device is not an sm_103 GPU with tcgen05 */
#define MOESTEP_EUNSUPPORTED (-6) /* shape outside what the kernels support (see each call) */
#define MOESTEP_ETIMEOUT (-7)     /* device error word: a bounded wait inside a kernel gave up */
#define MOESTEP_EDEVINPUT (-8)    /* device error word: fed input held an out-of-range index */

/* Element type of weights and MoE activations. */
#define MOESTEP_BF16 0 /* bf16 storage, fp32 accumulation on tcgen05 tensor cores */
#define MOESTEP_F32 1  /* fp32 storage and fp32 FFMA arithmetic (accuracy path) */
/* FP8 E4M3 expert weights (routed and shared; one fp32 scale per weight row),
 * everything else as MOESTEP_BF16: the expert launch converts each weight tile
 * to f16 in shared memory (exact), multiplies by f16 token rows on tcgen05
 * with fp32 accumulation and applies the row scales in its epilogue. */
#define MOESTEP_FP8 2

/* Model dimensions.  Supported: 1 <= k <= min(E, 32), E <= 1024, P <= 1024.
 * bf16 and fp8 paths additionally: H % 128 == 0, I % 64 == 0, Is % 64 == 0;
 * fp8 (calls that take expert weights): I % 128 == 0, Is % 128 == 0.
 * Is == 0 means no shared expert. */
typedef struct {
    int H;     /* hidden size */
    int E;     /* routed experts per layer */
    int k;     /* experts per token (top-k) */
    int I;     /* routed-expert SwiGLU intermediate size */
    int Is;    /* shared-expert intermediate size (0 = none) */
    int V;     /* vocabulary size of the LM head */
    int P;     /* block size: positions per request (32 by default in [AIT 三]) */
    int dtype; /* MOESTEP_BF16, MOESTEP_F32 or MOESTEP_FP8 */
} moestep_dims;

/* Device weights of one MoE layer (element type = dims.dtype; with
 * MOESTEP_FP8 the router is bf16 and the four expert tensors are E4M3 bytes).
 *   Wr   [E][H]        router
 *   Wgu  [E][I][2][H]  per expert, gate and up projections interleaved by row:
 *                      row 2i is gate row i, row 2i+1 is up row i
 *   Wd   [E][H][I]     per expert down projection
 *   Wsgu [Is][2][H]    shared expert gate/up, same interleaving (NULL iff Is == 0)
 *   Wsd  [H][Is]       shared expert down (NULL iff Is == 0)
 *   Sgu  [E][2I], Sd [E][H], Ssgu [2Is], Ssd [H]: fp32 scale of each weight
 *                      row (MOESTEP_FP8 only, NULL otherwise): a weight is
 *                      its E4M3 value times its row's scale
 * The interleaving puts the two halves of each SwiGLU pair into neighbouring
 * accumulator rows, so the tensor-core epilogue combines them with one shuffle. */
typedef struct {
    const void* Wr;
    const void* Wgu;
    const void* Wd;
    const void* Wsgu;
    const void* Wsd;
    const float* Sgu;
    const float* Sd;
    const float* Ssgu;
    const float* Ssd;
} moestep_layer;

/* Optional per-layer records written by block_decode_step (any field may be NULL;
 * x and h must be 16-byte aligned). */
typedef struct {
    int32_t* n_sel;  /* [n_layers][R]     experts kept by each request's coreset */
    int32_t* idx;    /* [n_layers][T][k]  router top-k */
    float* hidden;   /* [T][H]            fp32 LM-head input (final RMSNorm output) */
    int32_t* sel;    /* [n_layers][R][E]  kept experts in ranking order (first n_sel entries) */
    void* x;         /* [n_layers][T][H]  each layer's MoE input RMSNorm(h_l) (bf16, or fp32 in
                      *                   MOESTEP_F32 models), exactly as its router and experts read it */
    float* h;        /* [n_layers][T][H]  fp32 residual stream h_l entering each layer (h_0 = h_in;
                      *                   the layer's MoE output is h_{l+1} - h_l, h_L is h_out) */
} moestep_trace;

/* Bytes of workspace needed by every entry point below for R requests
 * (T = R * P tokens).  *bytes (host) receives the size. */
int moestep_workspace_size(const moestep_dims* dims, int R, size_t* bytes);

/* Zero the workspace's header (device error word and counters), asynchronously
 * on `stream`.  Call once on a new workspace before its first use; afterwards
 * the error word is sticky until moestep_read_device_error() clears it. */
int moestep_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* (a1) Router [AIT 四]; [GRM coreset section: each token picks its own top-k].
 * z = x Wr^T (fp32 accumulation), p = softmax(z) over E, idx = the k largest z
 * (ties: lower expert id), mass[t][j] = p[t][idx[t][j]], gate = mass / sum_j mass.
 *   x [T][H] (dims.dtype), Wr [E][H] (dims.dtype)
 *   idx [T][k] int32, mass [T][k] fp32, gate [T][k] fp32 (outputs)
 *   logits [T][E] fp32: optional copy of z (may be NULL)
 * T <= R*P of the workspace's sizing. */
int moe_block_route(const moestep_dims* dims, int T, const void* x, const void* Wr, int32_t* idx,
                    float* mass, float* gate, float* logits, void* ws, size_t ws_bytes, void* stream);

/* The router of moe_block_route for callers that cannot allocate device memory
 * (no workspace argument).  The pages have no counterpart: this is an
 * interface for hosts whose device memory is owned elsewhere (an application
 * allocator, a fixed embedded budget) and that therefore cannot call
 * cudaMalloc or hand over a scratch buffer.
 * Scratch (router logits when `logits` is NULL, and the completion counters)
 * lives in one fixed array inside the library, 520 KiB per CUDA context (one
 * per device for the runtime's primary contexts), held by every GPU that loads
 * the library until the process exits.  Limits:
 * T * E <= 131072 and T <= 8192; larger calls return MOESTEP_EUNSUPPORTED.
 * Arguments as in moe_block_route; x, Wr, the outputs and `stream` belong to
 * the calling thread's current CUDA context.  The array has one copy per
 * context, so its device address is looked up (cudaGetSymbolAddress) on the
 * first call in each context: the primary context of a device, a context the
 * caller created and made current, or a primary context re-created after
 * cudaDeviceReset.  Make that first call before any stream capture.  The
 * call allocates nothing and clears the counters it needs on `stream`; all
 * calls in one context share the one array, so calls whose executions overlap
 * on the GPU (other streams, other threads) race and must be serialised by the
 * caller.  Failures return MOESTEP_ECUDA with the cudaError_t in
 * moestep_last_cuda_error(). */
int moe_block_route_noalloc(const moestep_dims* dims, int T, const void* x, const void* Wr, int32_t* idx,
                            float* mass, float* gate, float* logits, void* stream);

/* Top-k, masses and gates from given router logits [T][E] fp32 (same rules as
 * moe_block_route).  Lets integer outputs be compared on identical inputs. */
int moe_route_from_logits(const moestep_dims* dims, int T, const float* logits, int32_t* idx,
                          float* mass, float* gate, void* ws, size_t ws_bytes, void* stream);

/* (a2) Block coreset [GRM "What is the MoE coreset and why does it matter?"].
 * For each request r (tokens r*P .. r*P+P-1): sum each candidate's mass per
 * expert as exact integers rne(mass * 2^54); rank experts by the sum
 * (descending, ties to the lower id); keep the shortest prefix whose sum
 * reaches ceil(top_p[r] * total) (clamped to [1, total]; top_p >= 1 keeps every
 * candidate); a token keeps the candidates inside the kept set, with gates
 * renormalised over them (zero if none survive).
 *   top_p [R] fp32 in (0, inf); idx, mass [R*P][k] as produced by the router
 *   n_sel [R] int32, sel [R][E] int32 (kept experts in ranking order; entries
 *   past n_sel[r] are unspecified), survive [R*P][k] uint8, gate_rr [R*P][k] fp32
 * Also leaves, inside the workspace, the grouped-by-expert work plan that
 * moe_block_ffn consumes; call moe_block_ffn with the same workspace next. */
int coreset_select(const moestep_dims* dims, int R, const float* top_p, const int32_t* idx,
                   const float* mass, int32_t* n_sel, int32_t* sel, uint8_t* survive, float* gate_rr,
                   void* ws, size_t ws_bytes, void* stream);

/* (a3-a5) Routed + shared SwiGLU experts over the block [AIT 四, 五].
 * out[t] = sum_j gate_rr[t][j] * Wd_e (silu(Wg_e x_t) * (Wu_e x_t)) over t's
 * surviving candidates e = idx[t][j], plus the shared expert with weight 1.
 * Each selected expert's weights are read once for all of its tokens
 * (bf16: TMA + tcgen05 grouped GEMM, expert rows as M, tokens as N).
 *   x [R*P][H] (dims.dtype; must be the router's input), layer (host struct of
 *   device pointers), gate_rr [R*P][k] from coreset_select, out [R*P][H] fp32.
 * Requires the plan left in `ws` by the coreset_select call of this layer. */
int moe_block_ffn(const moestep_dims* dims, int R, const void* x, const moestep_layer* layer,
                  const float* gate_rr, float* out, void* ws, size_t ws_bytes, void* stream);

/* (a7-a8) LM head + LowConfidence commit [AIT 三]; [GRM decoding loop].
 * logits = logit_scale * hidden Wlm^T, streamed by 128-row vocabulary tiles
 * with a per-tile online softmax (never stored unless `logits` is given);
 * conf = max softmax probability, choice = lowest argmax.  Per request: every
 * masked position with conf >= threshold is committed; if none is, the
 * masked position with the highest conf (lowest position on ties) is.
 * Committed positions are never written again.
 *   hidden [R*P][H] (dims.dtype), Wlm [V][H] (dims.dtype)
 *   tokens [R*P] int32, masked [R*P] uint8 (in/out; 1 = still masked)
 *   choice [R*P] int32, conf [R*P] fp32, accept [R*P] uint8 (1 = committed
 *   this round), n_committed [R] int32 (outputs)
 *   logits [R*P][V] fp32 optional debug copy (may be NULL)
 * threshold in (0, 1]. */
int lm_head_commit(const moestep_dims* dims, int R, const void* hidden, const void* Wlm, float logit_scale,
                   float threshold, int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf,
                   uint8_t* accept, int32_t* n_committed, float* logits, void* ws, size_t ws_bytes,
                   void* stream);

/* The confidence/argmax and commit of lm_head_commit applied to given logits
 * [R*P][V] fp32, so integer outputs can be compared on identical inputs. */
int lm_commit_from_logits(const moestep_dims* dims, int R, const float* logits, float threshold,
                          int32_t* tokens, uint8_t* masked, int32_t* choice, float* conf, uint8_t* accept,
                          int32_t* n_committed, void* ws, size_t ws_bytes, void* stream);

/* Input of the round-loop model: h[t] = emb[masked[t] ? mask_id : tokens[t]] + pos[t % P].
 * emb [V][H], pos [P][H] (dims.dtype), h [R*P][H] fp32 (output). */
int block_embed(const moestep_dims* dims, int R, const int32_t* tokens, const uint8_t* masked,
                const void* emb, const void* pos, int mask_id, float* h, void* stream);

/* One full denoising round: n_layers x [x = RMSNorm(h) -> router -> coreset ->
 * experts -> h += out], then RMSNorm -> LM head -> commit ([AIT 三] loop body
 * with the token mixers omitted).  RMSNorm has gamma = 1 and eps = 1e-6; in
 * the bf16 path the normalised activations are rounded to bf16.
 *   layers: HOST array [n_layers] of device-pointer structs
 *   top_p [R] fp32 (device), h_in [R*P][H] fp32 (not modified),
 *   h_out [R*P][H] fp32 final residual (may be NULL),
 *   tokens/masked/choice/conf/accept/n_committed as in lm_head_commit,
 *   trace: HOST pointer to optional records (may be NULL). */
int block_decode_step(const moestep_dims* dims, int R, int n_layers, const moestep_layer* layers,
                      const void* Wlm, const float* top_p, float logit_scale, float threshold,
                      const float* h_in, float* h_out, int32_t* tokens, uint8_t* masked, int32_t* choice,
                      float* conf, uint8_t* accept, int32_t* n_committed, const moestep_trace* trace,
                      void* ws, size_t ws_bytes, void* stream);

/* The whole LowConfidence loop of one block on the device ([AIT 三] block
 * decoding loop; [GRM] "How does confidence-threshold block decoding
 * work?"): while any position of the R requests is masked and fewer than
 * max_rounds rounds have run, h = block_embed(tokens, masked) and one
 * block_decode_step (no h_out, no trace).  The rounds run as the body of a
 * CUDA-graph while node whose condition a device kernel sets after each
 * commit, so no round returns to the host.
 *   emb, pos, mask_id as in block_embed; the model and top_p, logit_scale,
 *   threshold as in block_decode_step; tokens/masked [R*P] in/out;
 *   rounds [1] int32 (device, output): the rounds that ran.
 * The executable graph is cached and reused while every argument (pointers,
 * sizes, scalars, the layer array's contents) is unchanged, and rebuilt
 * otherwise.  Kernel timing (moestep_prof_enable) does not apply inside the
 * loop.  max_rounds >= 0; 0 runs nothing.  Not thread-safe. */
int block_decode_loop(const moestep_dims* dims, int R, int n_layers, const moestep_layer* layers, const void* Wlm,
                      const void* emb, const void* pos, int mask_id, const float* top_p, float logit_scale,
                      float threshold, int max_rounds, int32_t* tokens, uint8_t* masked, int32_t* rounds,
                      void* ws, size_t ws_bytes, void* stream);

/* Synchronously reads and clears the workspace's device error word (host *word:
 * 0 or a MOESTEP_E* code).  Waits for `stream`. */
int moestep_read_device_error(void* ws, size_t ws_bytes, void* stream, int* word);

/* Error text for a return code (static string). */
const char* moestep_error_string(int code);
/* The last cudaError_t seen by the library on this host thread. */
int moestep_last_cuda_error(void);
/* Number of kernels this library has launched in this process. */
long long moestep_launch_count(void);

/* Kernel timing with CUDA events on the launching stream (host-side tool for
 * the benchmark).  Bit i of kernel_mask brackets every launch of kernel id i
 * with events (0 turns timing off; enabling clears earlier records);
 * moestep_prof_read() synchronises and returns, per kernel id, the number of
 * timed launches and their summed duration in ms.  Kernel ids: 0 route
 * (with moestep_set_route_fusion(2): the cluster launch that holds the
 * router),
 * 1 coreset, 2 gather, 3 expert FFN (bf16: gate/up + SwiGLU + down in one
 * launch; fp32: gate/up), 4 fp32 expert down, 5 combine/norm, 6 LM head,
 * 7 commit, 8 other.  Not thread-safe. */
int moestep_prof_enable(int kernel_mask);
int moestep_prof_read(int kernel_id, int* launches, double* total_ms);
#define MOESTEP_PROF_KERNELS 9

/* Limit (ns) of every bounded wait inside the tensor-core kernels; default
 * 2e9.  When a wait runs out the kernel stops issuing work, lets the copies
 * and MMAs it already issued finish, frees its tensor memory, sets the
 * workspace error word (MOESTEP_ETIMEOUT) and returns.  Lowering it is a test
 * hook for that path. */
int moestep_set_wait_timeout_ns(unsigned long long ns);

/* What block_decode_step runs between two expert launches (the previous
 * layer's combine and RMSNorm, router, top-k, coreset, work plan and token
 * gather):
 *   0  separate launches: combine, router, coreset, gather;
 *   2  (the default) the combine and RMSNorm inside the router's launch (a
 *      cluster of E / 32 CTAs per 8 tokens), then coreset and gather: bf16
 *      activations, at most 256 block tokens, E a multiple of 32 up to 256 and
 *      H a multiple of 512.
 * Shapes mode 2 does not cover take the separate launches.  Both modes
 * compute bit-identical results.  Returns MOESTEP_EINVAL for another mode.
 * Process-wide; not thread-safe. */
int moestep_set_route_fusion(int mode);
/* The mode set by moestep_set_route_fusion. */
int moestep_route_fusion(void);

#ifdef __cplusplus
}
#endif
#endif /* MOESTEP_H */
