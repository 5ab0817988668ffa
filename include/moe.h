/*
 * moe.h -- C ABI of the GB300 (sm_103a) Mixture-of-Experts decode-layer forward.
 *
 * One library, libmoe_gb300.so, computes the MoE layer of a decoder for a
 * decode-sized batch of N tokens (N = 1..256 and beyond), on one GPU:
 *
 *   router   logits[t,e] = sum_h x[t,h] * Wr[e,h]                 (fp32)
 *   top-k    softmax: rank logits, p = softmax over all E logits;
 *            sigmoid+bias: rank sigmoid(l)+bias, p = sigmoid(l);
 *            w = p / sum_topk p if norm_topk_prob; w *= routed_scaling_factor
 *   experts  per (token t, slot j), e = idx[t,j]:
 *            d = Wd[e] (SiLU(Wg[e] x_t) * (Wu[e] x_t)),  SiLU(g) = g/(1+exp(-g))
 *   shared   ds = the same SwiGLU with the shared expert's three matrices
 *   blend    out[t] = sum_j w[t,j] d[t,j] + g_s ds,
 *            g_s = sigmoid(x_t . shared_gate_w), or 1 without a gate weight
 *
 * The operation is the one the pages "metrale_model_layers/layers/moe/forward.rs"
 * (MoeLayer::forward: gate, topk, exp_gate_up, exp_silu_down and wsum_blend
 * steps), "spark_model/layers/moe/forward_token_major.rs"
 * (forward_token_major_decode: gate GEMM, batched top-k, gate+up, silu+down,
 * weighted sum and blend for N tokens) and
 * "metrale_model_layers/layers/moe/forward_fp8_grouped_router.rs"
 * (grouped_route: router logits and top-k written as [m*top_k] indices and
 * fp32 weights) describe.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer marked "device" is a CUDA device (or managed) address on the
 *    current device; the caller owns every buffer (weights, input, outputs,
 *    workspace).  The library never allocates, frees or synchronises: each call
 *    only enqueues kernels on `stream` and returns.
 *  - The layer input x (moe_route, moe_experts, moe_forward) and output out
 *    (moe_experts, moe_forward) may instead be pinned (page-locked) host
 *    memory mapped into the device's address space (cudaHostAlloc, or any
 *    pinned allocation under unified addressing).  The kernels then reach x
 *    and out over the host link (NVLink-C2C on Grace systems) and no copy is
 *    needed before or after the call: one token's kernel reads x directly;
 *    for more tokens the call first copies x into the workspace with a kernel
 *    of its own, so that its other kernels read it from device memory.  Host
 *    memory that is not pinned is refused (MOE_ERR_HOST_MEMORY).  idx, w,
 *    logits, the weights and the workspace stay in device memory.
 *  - Device pointers must be 16-byte aligned (MOE_ERR_ALIGNMENT otherwise),
 *    except the scale and scale2 arrays of moe_qmat_t, which need 4 bytes (so
 *    that one rank's slice of a stacked scale array can be passed as it is).
 *  - All arguments are validated on the host before anything is enqueued; an
 *    error status means nothing was launched.  There is no fallback path: a
 *    configuration the kernels do not cover is refused by name
 *    (MOE_ERR_UNSUPPORTED), never computed some other way.
 *  - Asynchronous device faults are not reported by the call that enqueued
 *    the work; they surface from the next CUDA call as usual.
 *  - n == 0 is a valid no-op (MOE_OK, nothing launched).
 *  - The workspace is scratch the layer reuses across its steps.  Its first 256
 *    bytes are a control block that must be zero before the first call (for
 *    example cudaMemsetAsync(ws, 0, 256, stream) after allocating it); every
 *    call leaves it valid for the next one.  The rest is not meaningful between
 *    calls.  Two
 *    calls that run at the same time on the GPU must not share a workspace.
 *  - Device-side failures that the kernels detect themselves (a bounded wait
 *    that gave up after 2 s, or a control block that was not zeroed) end the
 *    kernel early and set an error word in the workspace: read it with
 *    moe_workspace_check().  The output of such a call is not valid.
 *
 * Tensor layouts (row-major, C order)
 * -----------------------------------
 *  x            BF16  [N, H]
 *  router_w     BF16  [E, H]  (each expert's router row contiguous)
 *  routed gate, up:   [E, I, H];  routed down: [E, H, I]
 *  shared gate, up:   [1, S, H];  shared down: [1, H, S]
 *  For a stacked [E, out, in] matrix the formats are
 *   MOE_W_BF16      w: BF16 [E, out, in]; scale, scale2 unused (NULL)
 *   MOE_W_FP8_B128  w: FP8 E4M3 bytes [E, out, in];
 *                   scale: fp32 [E, ceil(out/128), ceil(in/128)];
 *                   value = e4m3(w) * scale[o/128][i/128]
 *   MOE_W_NVFP4     w: bytes [E, out, in/2], two E2M1 codes per byte, the
 *                   element with even `in` index in the low nibble;
 *                   scale: FP8 E4M3 bytes [E, out, in/16] (one per 16 elements);
 *                   scale2: fp32 [E];
 *                   value = e2m1(code) * e4m3(scale[o][i/16]) * scale2[e]
 *  idx          int32 [N, k], slots in descending selection score
 *  w            fp32  [N, k]
 *  logits       fp32  [N, E]
 *  out          BF16  [N, H] (round to nearest even from fp32)
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

/* A CUDA stream handle (the same object as cudaStream_t; NULL = legacy default stream). */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_NULL = 1,            /* a required pointer is NULL                              */
    MOE_ERR_INVALID_CONFIG = 2,  /* a size, enum or flag is out of range or inconsistent    */
    MOE_ERR_UNSUPPORTED = 3,     /* valid, but outside what the kernels cover (named refusal)*/
    MOE_ERR_WORKSPACE = 4,       /* workspace missing or smaller than moe_workspace_bytes()  */
    MOE_ERR_CUDA = 5,            /* a CUDA call failed while enqueueing (cudaGetLastError)   */
    MOE_ERR_ALIGNMENT = 6,       /* a device pointer is not aligned (16 bytes; 4 for scales) */
    MOE_ERR_ALIAS = 7,           /* `out` overlaps `x`                                       */
    MOE_ERR_HOST_MEMORY = 8      /* `x` or `out` is host memory that is not pinned (page-locked) */
} moe_status_t;

typedef enum { MOE_ROUTE_SOFTMAX = 0, MOE_ROUTE_SIGMOID_BIAS = 1 } moe_routing_t;
typedef enum { MOE_W_BF16 = 0, MOE_W_FP8_B128 = 1, MOE_W_NVFP4 = 2 } moe_wfmt_t;
/* Expert-stage algorithm.  AUTO: one token runs the single-token kernel,
 * 2-3 tokens the token-major kernels, 4 or more the expert-grouped
 * tensor-core GEMM.  The two explicit values force one (tests); TOKEN_MAJOR
 * with one token still runs the single-token kernel (same arithmetic). */
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_TOKEN_MAJOR = 1, MOE_PATH_GROUPED = 2 } moe_path_t;

/* Pre-expert RMSNorm (the pre_expert_norm step of MoeLayer::forward, page
 * "metrale_model_layers/layers/moe/forward.rs"): with a norm weight, the routed
 * and shared experts take xe = BF16(x / sqrt(mean(x^2) + eps) * w); the router
 * and the shared-expert gate keep x.
 *
 * Expert parallelism (the EP branch of MoeLayer::forward and
 * forward_token_major_decode): a call with [expert_begin, expert_end) holds
 * only those experts -- the routed weight stacks have expert_end - expert_begin
 * entries, indexed from expert_begin -- and routes to other experts contribute
 * nothing; routing is still computed over all E.  With exclude_shared = 1 the
 * output is one rank's partial: the caller sums the partials over ranks (an
 * all-reduce) and adds the shared expert once, with a call that holds no
 * experts (expert_begin = expert_end = E) and accumulate = 1: it adds the
 * (gated) shared expert into the summed output, as the pages' residual_add /
 * moe_batched_blend after the all-reduce do.  A call that holds no experts and
 * is given neither idx nor w skips routing (it computes only the shared-gate
 * logit); on one token it still routes.
 *
 * accumulate = 1: every output element is BF16(out + result), with out read
 * on entry (rounded once, in fp32); out must then hold n x H valid values.
 *
 * NVFP4 router (the gate_nvfp4 / w4a16_gemm branch of the router step on the
 * same page): router_fmt = MOE_W_NVFP4 takes the router from router_q, an
 * NVFP4 matrix [E, H] in the expert layout below with one expert (w: bytes
 * [E, H/2]; scale: E4M3 [E, H/16]; scale2: one fp32), multiplying the BF16
 * activations; router_w is then unused (may be NULL).  One token then runs the
 * token-major kernels (the single-token kernel reads a BF16 router).  On the
 * expert-grouped path the router is expanded to BF16 in the workspace (each
 * code times its block scale, exact) for the tensor-core router, which applies
 * scale2 to its partial logits; the workspace then holds E x H BF16 more.
 *
 * Layer configuration (the config fields hidden_size, num_experts,
 * num_experts_per_tok, moe_intermediate_size, shared_expert_intermediate_size,
 * norm_topk_prob and routed_scaling_factor of the pages' layer).
 * Limits: 1 <= num_experts <= 1024; 1 <= top_k <= min(num_experts, 32);
 * hidden, inter > 0 and multiples of 32; shared_inter >= 0 and a multiple of 32
 * (0 = no shared expert); routed_scaling_factor finite. */
typedef struct {
    int32_t hidden;                 /* H */
    int32_t num_experts;            /* E */
    int32_t top_k;                  /* k */
    int32_t inter;                  /* I  (routed expert intermediate size) */
    int32_t shared_inter;           /* S  (shared expert intermediate size; 0 = none) */
    int32_t routing;                /* moe_routing_t */
    int32_t norm_topk_prob;         /* 0 or 1 */
    float   routed_scaling_factor;
    int32_t expert_fmt;             /* moe_wfmt_t: routed and shared experts alike */
    int32_t path;                   /* moe_path_t */
    /* ABI version 2 (a zero-filled tail keeps the version-1 behaviour): */
    float   rms_norm_eps;           /* epsilon of the pre-expert RMSNorm (when a norm weight is given) */
    int32_t expert_begin;           /* expert parallelism: this call holds experts   */
    int32_t expert_end;             /*   [expert_begin, expert_end); 0 and 0 = all E  */
    int32_t exclude_shared;         /* 1: leave the shared expert out of the output  */
    int32_t accumulate;             /* 1: out = BF16(out + layer output)             */
    int32_t router_fmt;             /* MOE_W_BF16 (router_w) or MOE_W_NVFP4 (router_q) */
} moe_config_t;

/* One stacked expert matrix (device pointers; see the layouts above). */
typedef struct {
    const void*  w;
    const void*  scale;    /* FP8: fp32 block scales; NVFP4: E4M3 bytes; BF16: NULL */
    const float* scale2;   /* NVFP4 only: fp32 [E]; else NULL */
} moe_qmat_t;

/* All weights of one layer (device pointers).  The shared-expert matrices are
 * ignored (may be NULL) when shared_inter == 0. */
typedef struct {
    const void*  router_w;          /* BF16 [E, H] */
    const float* correction_bias;   /* fp32 [E]; required for SIGMOID_BIAS, must be NULL for SOFTMAX */
    moe_qmat_t   gate, up, down;    /* routed experts */
    moe_qmat_t   sh_gate, sh_up, sh_down;   /* shared expert (E = 1) */
    const void*  shared_gate_w;     /* BF16 [H] or NULL (then the shared gate is 1) */
    /* ABI version 2: */
    const void*  pre_expert_norm_w; /* BF16 [H] or NULL: RMSNorm of the experts' input */
    moe_qmat_t   router_q;          /* NVFP4 router [E, H] when router_fmt = MOE_W_NVFP4 */
} moe_weights_t;

/* Bytes of workspace a call with up to `max_tokens` tokens needs (a multiple
 * of 256).  Returns 0 if `cfg` is NULL or invalid, or max_tokens < 0. */
size_t moe_workspace_bytes(const moe_config_t* cfg, int32_t max_tokens);

/* Router and top-k for n tokens (the pages' gate and topk steps, grouped_route).
 * The router runs where moe_forward's would for the same cfg and n: a BF16
 * router on the grouped path (cfg->path, or n > 3 under MOE_PATH_AUTO) on the
 * tensor cores (fp32 accumulation per K range, the ranges summed in a fixed
 * order), otherwise on the CUDA cores; so moe_route + moe_experts is
 * moe_forward bit for bit.
 *   x       device BF16 [n, H]
 *   idx     device int32 [n, k]   (out) selected experts, descending score
 *   w       device fp32  [n, k]   (out) routing weights
 *   logits  device fp32  [n, E]   (out, optional: NULL = not returned)
 *   ws      device workspace of at least moe_workspace_bytes(cfg, n) bytes
 * Errors: MOE_ERR_NULL, MOE_ERR_INVALID_CONFIG, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_WORKSPACE, MOE_ERR_ALIGNMENT, MOE_ERR_HOST_MEMORY, MOE_ERR_CUDA. */
moe_status_t moe_route(const moe_config_t* cfg, const moe_weights_t* wts,
                       const void* x, int32_t n,
                       int32_t* idx, float* w, float* logits,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* Routed experts, shared expert and blend for n tokens given their routing
 * (the pages' exp_gate_up, exp_silu_down and wsum_blend steps).
 *   x     device BF16 [n, H] (the layer input: with a pre-expert norm weight
 *         the experts take its RMSNorm, and the shared gate takes x itself)
 *   idx   device int32 [n, k]; an entry outside [expert_begin, expert_end)
 *         (all of [0, E) by default) is dropped (that slot contributes
 *         nothing), so a bad index never reads outside the weights
 *   w     device fp32  [n, k]
 *   out   device BF16 [n, H] (out); must not overlap x
 * Errors: as moe_route, plus MOE_ERR_ALIAS. */
moe_status_t moe_experts(const moe_config_t* cfg, const moe_weights_t* wts,
                         const void* x, int32_t n,
                         const int32_t* idx, const float* w,
                         void* out, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer: moe_route then moe_experts on one stream.
 *   idx, w  optional device outputs ([n, k] int32 / fp32); NULL = kept in the
 *           workspace only. */
moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* wts,
                         const void* x, int32_t n, void* out,
                         int32_t* idx, float* w,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_forward with stage markers, for profiling (the per-stage timing the
 * pages' `prof!` macro in MoeLayer::forward takes with a stream sync, done here
 * with device events and no sync).
 *   events    array of n_events cudaEvent_t handles (cast to void*) created by
 *             the caller on the current device; marker i is recorded with
 *             cudaEventRecord(events[i], stream) for i < n_events
 *   n_marks   (out, optional) markers the call reached
 * Markers: 0 before the first kernel, then one after each stage, in launch
 * order.  One token on the single-token kernel: 2 markers (before, after).
 * Token-major kernels: 5 (router, top-k + grouping, gate+up, down+blend).
 * Grouped tensor-core path: 7 (router, top-k + grouping, gather, gate+up, down,
 * combine).  The pre-expert RMSNorm, when present, runs at the start of the
 * stage after top-k + grouping.
 * Errors: as moe_forward, plus MOE_ERR_NULL for events == NULL with n_events > 0. */
moe_status_t moe_forward_timed(const moe_config_t* cfg, const moe_weights_t* wts,
                               const void* x, int32_t n, void* out,
                               int32_t* idx, float* w,
                               void* ws, size_t ws_bytes, moe_stream_t stream,
                               void* const* events, int32_t n_events, int32_t* n_marks);

/* Bytes of the static device workspace of moe_forward_static_ws. */
#define MOE_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

/* moe_forward for callers that cannot allocate device memory (no counterpart
 * in the pages: an addition of this library).  A plugin whose host owns every
 * allocation, or code that is recording a CUDA graph (where cudaMalloc is not
 * allowed), may have input and output buffers but no way to get a workspace.
 * This call takes none: its scratch is one file-scope device array of
 * MOE_STATIC_WORKSPACE_BYTES that every GPU which loads the library keeps until
 * the process exits.  It allocates nothing and calls no allocating routine.
 *   Arguments, outputs and errors: as moe_forward, without ws / ws_bytes.
 *   A call that would need more than MOE_STATIC_WORKSPACE_BYTES of workspace
 *   (moe_workspace_bytes(cfg, n)) returns MOE_ERR_WORKSPACE and launches nothing.
 *   The first call on each device looks up the array's device address and
 *   clears its control block on `stream`, then synchronises `stream`; make
 *   that first call before any stream capture (a first call on a stream that
 *   is being captured returns MOE_ERR_UNSUPPORTED and launches nothing).
 *   Every call shares the one array: calls whose work overlaps on the GPU
 *   (other streams, other host threads) race on it and must be serialised by
 *   the caller.
 *   Device-side failures (a bounded wait that gave up; a control block left
 *   dirty by such a call, which makes every later one-token call refuse and
 *   leave `out` unwritten) are recorded in the array's control block and are
 *   not returned by this call: read and clear them with
 *   moe_static_workspace_check(). */
moe_status_t moe_forward_static_ws(const moe_config_t* cfg, const moe_weights_t* wts,
                                   const void* x, int32_t n, void* out,
                                   int32_t* idx, float* w, moe_stream_t stream);

/* moe_workspace_check for the static workspace of moe_forward_static_ws on the
 * current device (no counterpart in the pages: an addition of this library).
 * Reads, then clears, the array's device error word and resets its
 * single-token barrier word, so the next static call runs; synchronises
 * `stream`.
 *   device_error (out)  as moe_workspace_check: 0, 11-17, 1-8 or 20.
 *   workspace    (out, optional) the array's device address on this device
 *                (NULL = not returned); the library owns it.
 * The first use on a device runs the set-up of moe_forward_static_ws.
 * Errors: MOE_ERR_NULL (device_error NULL), MOE_ERR_UNSUPPORTED (`stream` is
 * being captured into a graph), MOE_ERR_CUDA. */
moe_status_t moe_static_workspace_check(int32_t* device_error, void** workspace, moe_stream_t stream);

/* Reads, then clears, the device error word of a workspace, and resets the
 * single-token kernel's and the grouped down kernel's barrier words (which a
 * call that ended early leaves non-zero) and the routed-token count, so the
 * workspace serves the next call.  Synchronises `stream` (the only entry
 * point that does).
 *   device_error (out)  0: no failure since the last check; 11-17: a bounded
 *                       wait of the single-token kernel gave up; 1-5: a bounded
 *                       wait of the grouped tensor-core kernels gave up (8: the
 *                       down kernel's grid barrier before its combine); 6-7:
 *                       one of the tensor-core router's; 20: the workspace
 *                       control block was not zeroed before use.  An FP8
 *                       call on the grouped path made while an error is
 *                       pending does not write out (its down kernel, which
 *                       also combines, skips the combine); check (and so
 *                       clear) after a failure.
 * Errors: MOE_ERR_NULL, MOE_ERR_ALIGNMENT, MOE_ERR_WORKSPACE (ws_bytes < 256),
 * MOE_ERR_CUDA. */
moe_status_t moe_workspace_check(void* ws, size_t ws_bytes, int32_t* device_error,
                                 moe_stream_t stream);

/* Static description of a status code (never NULL). */
const char* moe_status_string(moe_status_t status);

/* MOE_ABI_VERSION of the built library. */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_MOE_H */
