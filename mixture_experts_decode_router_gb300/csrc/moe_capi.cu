// moe_capi.cu -- the C ABI of libmoe_gb300 (declared in include/moe.h):
// host-side validation, workspace carving and the launch sequence.
//
// Validation refuses by name before anything is enqueued, in the manner of the
// pages' named refusals ("spark_model/layers/moe/forward_token_major.rs":
// forward_token_major_decode refuses zero-expert routing rather than compute
// it wrongly; "metrale_model_layers/layers/moe/forward.rs": reject_decode_lora,
// refuse_lean_layout).
#include <mutex>

#include "moe_launch.cuh"

namespace moe {

static int device_sm_count() {
    static std::mutex mu;
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cache[dev] = v;
    }
    return cache[dev];
}

// Optional stage markers: records events[i] on the stream at stage boundaries
// (the pages' per-stage `prof!` timing, done with device events, no sync).
struct Marks {
    cudaEvent_t* ev = nullptr;
    int n = 0, next = 0;
    void mark(cudaStream_t st) {
        if (next < n) cudaEventRecord(ev[next], st);
        ++next;
    }
};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Where a caller's x or out lives: 0 device (or managed) memory, 1 pinned host
// memory the device addresses at the same pointer, -1 anything else (host memory
// that is not pinned, or a pointer CUDA does not know).
static int residency(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return 0;
    if (a.type == cudaMemoryTypeHost && a.devicePointer == p) return 1;
    return -1;
}
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static moe_status_t check_config(const moe_config_t* c) {
    if (!c) return MOE_ERR_NULL;
    if (c->num_experts < 1 || c->num_experts > kMaxExperts) return MOE_ERR_INVALID_CONFIG;
    if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > kMaxTopK) return MOE_ERR_INVALID_CONFIG;
    if (c->hidden <= 0 || c->hidden % 32) return MOE_ERR_INVALID_CONFIG;
    if (c->inter <= 0 || c->inter % 32) return MOE_ERR_INVALID_CONFIG;
    if (c->shared_inter < 0 || c->shared_inter % 32) return MOE_ERR_INVALID_CONFIG;
    if (c->routing != MOE_ROUTE_SOFTMAX && c->routing != MOE_ROUTE_SIGMOID_BIAS)
        return MOE_ERR_INVALID_CONFIG;
    if (c->norm_topk_prob != 0 && c->norm_topk_prob != 1) return MOE_ERR_INVALID_CONFIG;
    if (!(c->routed_scaling_factor == c->routed_scaling_factor) ||
        c->routed_scaling_factor > 3.0e38f || c->routed_scaling_factor < -3.0e38f)
        return MOE_ERR_INVALID_CONFIG;
    if (c->expert_fmt != MOE_W_BF16 && c->expert_fmt != MOE_W_FP8_B128 && c->expert_fmt != MOE_W_NVFP4)
        return MOE_ERR_INVALID_CONFIG;
    if (c->path != MOE_PATH_AUTO && c->path != MOE_PATH_TOKEN_MAJOR && c->path != MOE_PATH_GROUPED)
        return MOE_ERR_INVALID_CONFIG;
    // Sizes that keep every index below 2^31.
    const int64_t big = (int64_t)c->num_experts * c->inter * c->hidden;
    if (big > (int64_t)1 << 40) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// The configuration a call runs: the expert range resolved ((0, 0) = all E)
// and the shared expert dropped when the call leaves it out.
static moe_status_t effective_config(const moe_config_t* c, moe_config_t* out) {
    moe_status_t s = check_config(c);
    if (s != MOE_OK) return s;
    *out = *c;
    if (c->expert_begin == 0 && c->expert_end == 0) out->expert_end = c->num_experts;
    if (out->expert_begin < 0 || out->expert_begin > out->expert_end || out->expert_end > c->num_experts)
        return MOE_ERR_INVALID_CONFIG;
    if (c->exclude_shared != 0 && c->exclude_shared != 1) return MOE_ERR_INVALID_CONFIG;
    if (c->accumulate != 0 && c->accumulate != 1) return MOE_ERR_INVALID_CONFIG;
    if (c->router_fmt != MOE_W_BF16 && c->router_fmt != MOE_W_NVFP4) return MOE_ERR_INVALID_CONFIG;
    if (!(c->rms_norm_eps >= 0.0f && c->rms_norm_eps <= 3.0e38f)) return MOE_ERR_INVALID_CONFIG;
    if (c->exclude_shared) out->shared_inter = 0;
    return MOE_OK;
}

static int local_experts(const moe_config_t* c) { return c->expert_end - c->expert_begin; }

static moe_status_t check_qmat(int fmt, const moe_qmat_t& q) {
    if (!q.w) return MOE_ERR_NULL;
    if (!aligned16(q.w)) return MOE_ERR_ALIGNMENT;
    // Scales are read 4 bytes at a time at most.
    if (fmt == MOE_W_FP8_B128 || fmt == MOE_W_NVFP4) {
        if (!q.scale) return MOE_ERR_NULL;
        if (!aligned4(q.scale)) return MOE_ERR_ALIGNMENT;
    }
    if (fmt == MOE_W_NVFP4) {
        if (!q.scale2) return MOE_ERR_NULL;
        if (!aligned4(q.scale2)) return MOE_ERR_ALIGNMENT;
    }
    return MOE_OK;
}

static moe_status_t check_router_weights(const moe_config_t* c, const moe_weights_t* w) {
    if (!w) return MOE_ERR_NULL;
    if (c->router_fmt == MOE_W_NVFP4) {
        const moe_status_t s = check_qmat(MOE_W_NVFP4, w->router_q);
        if (s != MOE_OK) return s;
    } else {
        if (!w->router_w) return MOE_ERR_NULL;
        if (!aligned16(w->router_w)) return MOE_ERR_ALIGNMENT;
    }
    if (c->routing == MOE_ROUTE_SIGMOID_BIAS) {
        if (!w->correction_bias) return MOE_ERR_NULL;
        if (!aligned16(w->correction_bias)) return MOE_ERR_ALIGNMENT;
    } else if (w->correction_bias) {
        return MOE_ERR_INVALID_CONFIG;   // a bias has no meaning under softmax routing
    }
    return MOE_OK;
}

static moe_status_t check_expert_weights(const moe_config_t* c, const moe_weights_t* w) {
    if (!w) return MOE_ERR_NULL;
    moe_status_t s;
    if (local_experts(c) > 0) {   // routed stacks, unless the call holds no expert
        if ((s = check_qmat(c->expert_fmt, w->gate)) != MOE_OK) return s;
        if ((s = check_qmat(c->expert_fmt, w->up)) != MOE_OK) return s;
        if ((s = check_qmat(c->expert_fmt, w->down)) != MOE_OK) return s;
    }
    if (c->shared_inter > 0) {
        if ((s = check_qmat(c->expert_fmt, w->sh_gate)) != MOE_OK) return s;
        if ((s = check_qmat(c->expert_fmt, w->sh_up)) != MOE_OK) return s;
        if ((s = check_qmat(c->expert_fmt, w->sh_down)) != MOE_OK) return s;
    }
    if (w->shared_gate_w && !aligned16(w->shared_gate_w)) return MOE_ERR_ALIGNMENT;
    if (w->pre_expert_norm_w && !aligned16(w->pre_expert_norm_w)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

static moe_status_t check_ws(const moe_config_t* c, int32_t n, const void* ws, size_t ws_bytes,
                             WsLayout* L) {
    *L = ws_layout(*c, n);
    if (!ws) return MOE_ERR_WORKSPACE;
    if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

template <typename T> static T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// e_base: global index of the stack's first expert (0 for the shared expert).
static QMatDev qdev(const moe_qmat_t& q, int out_dim, int in_dim, int e_base) {
    QMatDev d;
    d.w = static_cast<const uint8_t*>(q.w);
    d.scale = q.scale;
    d.scale2 = q.scale2;
    d.out_dim = out_dim;
    d.in_dim = in_dim;
    d.e_base = e_base;
    return d;
}

// Copy a pinned-host-resident x ([n, H] BF16) into the workspace; `x` then
// points there.
static moe_status_t stage_x(const moe_config_t* c, const void*& x, int32_t n, void* ws, const WsLayout& L,
                            cudaStream_t st) {
    void* xd = at<uint16_t>(ws, L.xd);
    if (launch_copy16(x, xd, (size_t)n * c->hidden * 2, device_sm_count(), st) != cudaSuccess) return MOE_ERR_CUDA;
    x = xd;
    return MOE_OK;
}

// Token counts up to this use the token-major CUDA-core kernels under AUTO
// (one token: the single-token kernel); above it the grouped tensor-core path.
// Measured on GB300 at H=2048, E=256, k=8, BF16: grouped is faster from 4
// tokens on (4: 90 vs 95 us, 8: 128 vs 177 us, 16: 160 vs 279 us), token-major
// at 2 (63 vs 74 us).
constexpr int kTokenMajorMaxN = 3;

// Whether the small kernels of a grouped call of n tokens signal their
// dependent launch right after their own wait (pdl_trigger), so that the next
// kernel's launch and prologue overlap them.  Measured on GB300: decode_n16
// 129.9 -> 126.2 us, fp8_n64 984 -> 979 us; at 256 tokens slower (198.7 ->
// 205.5 us), where the top-k kernel needs two 1024-thread CTAs on every SM
// and a router CTA still on an SM leaves room for one.
static bool early_dependents(int32_t n, int sms) { return n <= sms; }

// The multi-kernel path a call of n tokens takes.
static int effective_path(const moe_config_t* c, int32_t n) {
    return c->path == MOE_PATH_AUTO ? (n <= kTokenMajorMaxN ? MOE_PATH_TOKEN_MAJOR : MOE_PATH_GROUPED) : c->path;
}

// Enqueue router + top-k.  Arguments already validated.  `with_group`: the
// top-k launch also groups the routes by expert (the fused top-k + grouping
// kernel), so the expert stage that follows skips its grouping launch.
// `x_dev`: x is in device memory.  A BF16 or NVFP4 router on the grouped path
// runs on the tensor cores (partial logits per K split, summed in order by the
// top-k kernel; an NVFP4 router expanded to BF16 first; the shared-gate row
// keeps the CUDA-core kernel); the token-major path keeps the CUDA-core
// routers, whose arithmetic the single-token kernel repeats, so that a token
// alone and in a batch route alike.
static moe_status_t enqueue_route(const moe_config_t* c, const moe_weights_t* w, const void* x,
                                  int32_t n, int32_t* idx, float* wt, float* logits, void* ws,
                                  const WsLayout& L, bool with_group, bool x_dev, cudaStream_t st, Marks& mk) {
    const int sms = device_sm_count();
    float* lg = logits ? logits : at<float>(ws, L.logits);
    const float* lin = lg;   // what the top-k kernel reads: logits, or the partials
    float* lsum = nullptr;   // where it writes summed logits (moe_route's output)
    int ns = 1;
    cudaError_t e;
    // The shared-gate row beside the tensor-core router: formed by the top-k +
    // grouping kernel when it runs and has room, else launched on its own.
    const uint16_t* gate_in_topk = nullptr;
    if ((c->router_fmt == MOE_W_BF16 || c->router_fmt == MOE_W_NVFP4) && x_dev &&
        effective_path(c, n) == MOE_PATH_GROUPED && router_tc_fits(n, c->num_experts, c->hidden)) {
        // An NVFP4 router is first expanded to BF16 (exactly); its scale2
        // multiplies the partials.
        float* part = at<float>(ws, L.lgp);
        const uint16_t* wr = static_cast<const uint16_t*>(w->router_w);
        const float* rsc = nullptr;
        e = cudaSuccess;
        if (c->router_fmt == MOE_W_NVFP4) {
            uint16_t* rq = at<uint16_t>(ws, L.rq);
            e = launch_router_nvfp4_expand(qdev(w->router_q, c->num_experts, c->hidden, 0), c->num_experts,
                                           c->hidden, rq, early_dependents(n, sms), sms, st);
            wr = rq;
            rsc = w->router_q.scale2;
        }
        if (e == cudaSuccess)
            e = launch_router_tc(static_cast<const uint16_t*>(x), n, c->hidden, wr, c->num_experts, part,
                                 &at<Ctrl>(ws, L.ctrl)->err, rsc, early_dependents(n, sms), st);
        if (w->shared_gate_w && with_group && topk_group_gate_fits(c->num_experts, c->hidden))
            gate_in_topk = static_cast<const uint16_t*>(w->shared_gate_w);
        else if (e == cudaSuccess && w->shared_gate_w)
            e = launch_router(static_cast<const uint16_t*>(x), n, c->hidden, nullptr, 0,
                              static_cast<const uint16_t*>(w->shared_gate_w), nullptr,
                              at<float>(ws, L.sg_logit), sms, st);
        lin = part;
        ns = router_tc_split(c->hidden).splits;
        lsum = logits;
    } else if (c->router_fmt == MOE_W_NVFP4) {
        e = launch_router_nvfp4(static_cast<const uint16_t*>(x), n, c->hidden,
                                qdev(w->router_q, c->num_experts, c->hidden, 0), c->num_experts, lg, st);
        if (e == cudaSuccess && w->shared_gate_w)   // the BF16 shared-gate row on its own
            e = launch_router(static_cast<const uint16_t*>(x), n, c->hidden, nullptr, 0,
                              static_cast<const uint16_t*>(w->shared_gate_w), nullptr,
                              at<float>(ws, L.sg_logit), sms, st);
    } else {
        e = launch_router(static_cast<const uint16_t*>(x), n, c->hidden,
                          static_cast<const uint16_t*>(w->router_w), c->num_experts,
                          static_cast<const uint16_t*>(w->shared_gate_w), lg,
                          at<float>(ws, L.sg_logit), sms, st);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);
    if (with_group)
        e = launch_topk_group(lin, ns, n, c->num_experts, c->top_k, c->routing, w->correction_bias, c->norm_topk_prob,
                              c->routed_scaling_factor, idx, wt, c->expert_begin, c->expert_end,
                              at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.perm),
                              at<int32_t>(ws, L.inv), at<int32_t>(ws, L.active), at<int32_t>(ws, L.segs),
                              at<Ctrl>(ws, L.ctrl), static_cast<const uint16_t*>(x), gate_in_topk,
                              at<float>(ws, L.sg_logit), c->hidden, early_dependents(n, sms), sms, st);
    else
        e = launch_topk(lin, ns, lsum, n, c->num_experts, c->top_k, c->routing, w->correction_bias,
                        c->norm_topk_prob, c->routed_scaling_factor, idx, wt, st);
    mk.mark(st);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}


// The grouped tensor-core expert stage (after the grouping kernel).
// x: the layer input; the gather applies the pre-expert RMSNorm, if any.
static moe_status_t enqueue_grouped(const moe_config_t* c, const moe_weights_t* w, const void* x,
                                    int32_t n, const float* wt, void* out, void* ws, const WsLayout& L,
                                    float* sg_logit, cudaStream_t st, Marks& mk) {
    const int sms = device_sm_count();
    const int fmt = c->expert_fmt;
    const int H = c->hidden, I = c->inter, S = c->shared_inter, k = c->top_k, E = c->num_experts;
    const int E_loc = local_experts(c);
    uint16_t* xs = at<uint16_t>(ws, L.xs);
    uint16_t* xh = at<uint16_t>(ws, L.xh);
    cudaError_t e = launch_gather(fmt, static_cast<const uint16_t*>(x), n, H, k, at<int32_t>(ws, L.perm),
                                  at<int32_t>(ws, L.offsets), E, xs, xh,
                                  static_cast<const uint16_t*>(w->pre_expert_norm_w), c->rms_norm_eps,
                                  early_dependents(n, sms), sms, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);

    TcParams p{};
    p.n = n;
    p.k = k;
    p.e_base = c->expert_begin;
    p.segs = at<int32_t>(ws, L.segs);
    p.ctrl = at<Ctrl>(ws, L.ctrl);
    p.err = &at<Ctrl>(ws, L.ctrl)->err;
    p.zero4 = &at<Ctrl>(ws, L.ctrl)->pad[0];   // never written: zero
    p.perm = at<int32_t>(ws, L.perm);
    p.route_w = wt;
    p.sg_logit = w->shared_gate_w ? sg_logit : nullptr;
    p.act_out = at<uint16_t>(ws, L.as);
    p.act_sh_out = at<uint16_t>(ws, L.ash);
    p.y = at<float>(ws, L.y);
    p.y_sh = at<float>(ws, L.ysh);

    const bool tiles = E_loc > 0 || S > 0;   // otherwise the output is zero: combine alone
    // gate + up
    TcMaps maps;
    if (tiles && !build_tc_maps(fmt, true, w, E_loc, H, I, S, n, n * k, xs, xh, &maps))
        return MOE_ERR_CUDA;
    p.out_dim = I; p.in_dim = H; p.sh_out = S; p.sh_in = H;
    p.scale[0] = w->gate.scale; p.scale[1] = w->up.scale;
    p.sh_scale[0] = w->sh_gate.scale; p.sh_scale[1] = w->sh_up.scale;
    p.scale2[0] = w->gate.scale2; p.scale2[1] = w->up.scale2;
    p.sh_scale2[0] = w->sh_gate.scale2; p.sh_scale2[1] = w->sh_up.scale2;
    if (tiles && (e = launch_grouped_tc(fmt, true, maps, p, sms, st)) != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);

    // down (+ routing weight / shared gate)
    if (tiles && !build_tc_maps(fmt, false, w, E_loc, H, I, S, n, n * k, p.act_out, p.act_sh_out, &maps))
        return MOE_ERR_CUDA;
    p.out_dim = H; p.in_dim = I; p.sh_out = S > 0 ? H : 0; p.sh_in = S;
    p.scale[0] = p.scale[1] = w->down.scale;
    p.sh_scale[0] = p.sh_scale[1] = w->sh_down.scale;
    p.scale2[0] = p.scale2[1] = w->down.scale2;
    p.sh_scale2[0] = p.sh_scale2[1] = w->sh_down.scale2;
    // The FP8 down kernel also runs the combine, after a grid barrier on its
    // persistent blocks (fp8_n64 992 -> 983 us on GB300).  The BF16 and NVFP4
    // down kernels have 192 and 480 threads a block against FP8's 736, too
    // few for the latency-bound combine (decode_n16 128.7 -> 131.3 us,
    // nvfp4_n256 196.8 -> 198.2 us with it), so theirs runs on its own, as
    // it does when there are no tiles.
    p.combine = (tiles && fmt == MOE_W_FP8_B128) ? 1 : 0;
    p.inv = at<int32_t>(ws, L.inv);
    p.out = static_cast<uint16_t*>(out);
    p.has_shared = S > 0 ? 1 : 0;
    p.accumulate = c->accumulate;
    p.tc_count = &at<Ctrl>(ws, L.ctrl)->tc_count;
    p.tc_gen = &at<Ctrl>(ws, L.ctrl)->tc_gen;
    if (tiles && (e = launch_grouped_tc(fmt, false, maps, p, sms, st)) != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);

    if (!p.combine) {
        e = launch_combine(p.y, p.y_sh, p.inv, n, H, k, S > 0 ? 1 : 0, c->accumulate, static_cast<uint16_t*>(out),
                           early_dependents(n, sms), sms, st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        mk.mark(st);
    }
    return MOE_OK;
}

// Enqueue grouping + experts + blend.  `sg_from_ws`: the shared-gate logit was
// written to the workspace by enqueue_route of the same call.  `grouped`: so
// were the routes' grouping by expert (enqueue_route with_group).
static moe_status_t enqueue_experts(const moe_config_t* c, const moe_weights_t* w, const void* x,
                                    int32_t n, const int32_t* idx, const float* wt, void* out,
                                    void* ws, const WsLayout& L, bool sg_from_ws, bool grouped,
                                    cudaStream_t st, Marks& mk) {
    const int sms = device_sm_count();
    const int H = c->hidden, I = c->inter, S = c->shared_inter, k = c->top_k, E = c->num_experts;
    float* sg_logit = at<float>(ws, L.sg_logit);
    cudaError_t e;
    if (w->shared_gate_w && !sg_from_ws) {
        // moe_experts called on its own: the shared gate logit x . gw is the
        // router kernel's extra row, run with no expert rows.
        e = launch_router(static_cast<const uint16_t*>(x), n, H,
                          static_cast<const uint16_t*>(w->router_w), 0,
                          static_cast<const uint16_t*>(w->shared_gate_w), nullptr, sg_logit, sms, st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    // The experts' input: x, or its pre-expert RMSNorm (the router and the
    // shared gate keep x); the grouped path's gather applies the norm itself.
    const int path = effective_path(c, n);
    const void* xin = x;
    if (w->pre_expert_norm_w && path != MOE_PATH_GROUPED) {
        uint16_t* xe = at<uint16_t>(ws, L.xe);
        e = launch_rmsnorm(static_cast<const uint16_t*>(x), n, H,
                           static_cast<const uint16_t*>(w->pre_expert_norm_w), c->rms_norm_eps, xe, st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        xin = xe;
    }
    if (!grouped) {
        e = launch_group(idx, n * k, E, c->expert_begin, c->expert_end, at<int32_t>(ws, L.counts),
                         at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.perm), at<int32_t>(ws, L.inv),
                         at<int32_t>(ws, L.active), at<int32_t>(ws, L.segs), at<Ctrl>(ws, L.ctrl), st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        mk.mark(st);
    }

    if (path == MOE_PATH_GROUPED)
        return enqueue_grouped(c, w, x, n, wt, out, ws, L, sg_logit, st, mk);

    const int eb = c->expert_begin;
    GateUpParams gu{};
    gu.x = static_cast<const uint16_t*>(xin);
    gu.n = n; gu.H = H; gu.I = I; gu.S = S; gu.k = k;
    gu.gate = qdev(w->gate, I, H, eb);
    gu.up = qdev(w->up, I, H, eb);
    if (S > 0) {
        gu.sh_gate = qdev(w->sh_gate, S, H, 0);
        gu.sh_up = qdev(w->sh_up, S, H, 0);
    }
    gu.counts = at<int32_t>(ws, L.counts);
    gu.offsets = at<int32_t>(ws, L.offsets);
    gu.perm = at<int32_t>(ws, L.perm);
    gu.active = at<int32_t>(ws, L.active);
    gu.ctrl = at<Ctrl>(ws, L.ctrl);
    gu.act = at<float>(ws, L.act);
    gu.act_sh = at<float>(ws, L.act_sh);

    DownParams dn{};
    dn.n = n; dn.H = H; dn.I = I; dn.S = S; dn.k = k; dn.E = E;
    dn.e_begin = c->expert_begin; dn.e_end = c->expert_end;
    dn.accumulate = c->accumulate;
    dn.down = qdev(w->down, H, I, eb);
    if (S > 0) dn.sh_down = qdev(w->sh_down, H, S, 0);
    dn.idx = idx;
    dn.w = wt;
    dn.act = gu.act;
    dn.act_sh = gu.act_sh;
    dn.sg_logit = w->shared_gate_w ? sg_logit : nullptr;
    dn.out = static_cast<uint16_t*>(out);

    e = launch_gate_up_tm(c->expert_fmt, gu, sms, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);
    e = launch_down_blend_tm(c->expert_fmt, dn, sms, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    mk.mark(st);
    return MOE_OK;
}

static bool overlaps(const void* a, const void* b, size_t bytes) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + bytes && pb < pa + bytes;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_config_t* cfg_in, int32_t max_tokens) {
    moe_config_t c;
    if (effective_config(cfg_in, &c) != MOE_OK || max_tokens < 0) return 0;
    return ws_layout(c, max_tokens).total;
}

moe_status_t moe_route(const moe_config_t* cfg_in, const moe_weights_t* wts, const void* x, int32_t n,
                       int32_t* idx, float* w, float* logits, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
    moe_config_t c;
    const moe_config_t* cfg = &c;
    moe_status_t s = effective_config(cfg_in, &c);
    if (s != MOE_OK) return s;
    if (n < 0) return MOE_ERR_INVALID_CONFIG;
    if ((s = check_router_weights(cfg, wts)) != MOE_OK) return s;
    if (n == 0) return MOE_OK;
    if (!x || !idx || !w) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(idx) || !aligned16(w) || (logits && !aligned16(logits)))
        return MOE_ERR_ALIGNMENT;
    if (wts->shared_gate_w && !aligned16(wts->shared_gate_w)) return MOE_ERR_ALIGNMENT;
    WsLayout L;
    if ((s = check_ws(cfg, n, ws, ws_bytes, &L)) != MOE_OK) return s;
    const int x_res = residency(x);
    if (x_res < 0) return MOE_ERR_HOST_MEMORY;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (x_res == 1 && n > 1 && (s = stage_x(cfg, x, n, ws, L, st)) != MOE_OK) return s;
    Marks mk;
    return enqueue_route(cfg, wts, x, n, idx, w, logits, ws, L, false, x_res == 0 || n > 1, st, mk);
}

moe_status_t moe_experts(const moe_config_t* cfg_in, const moe_weights_t* wts, const void* x, int32_t n,
                         const int32_t* idx, const float* w, void* out, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
    moe_config_t c;
    const moe_config_t* cfg = &c;
    moe_status_t s = effective_config(cfg_in, &c);
    if (s != MOE_OK) return s;
    if (n < 0) return MOE_ERR_INVALID_CONFIG;
    if ((s = check_expert_weights(cfg, wts)) != MOE_OK) return s;
    if (n == 0) return MOE_OK;
    if (!x || !idx || !w || !out) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(idx) || !aligned16(w) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
    if (overlaps(x, out, (size_t)n * cfg->hidden * 2)) return MOE_ERR_ALIAS;
    WsLayout L;
    if ((s = check_ws(cfg, n, ws, ws_bytes, &L)) != MOE_OK) return s;
    const int x_res = residency(x);
    if (x_res < 0 || residency(out) < 0) return MOE_ERR_HOST_MEMORY;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (x_res == 1 && n > 1 && (s = stage_x(cfg, x, n, ws, L, st)) != MOE_OK) return s;
    Marks mk;
    return enqueue_experts(cfg, wts, x, n, idx, w, out, ws, L, false, false, st, mk);
}

static moe_status_t forward_impl(const moe_config_t* cfg_in, const moe_weights_t* wts, const void* x,
                                 int32_t n, void* out, int32_t* idx, float* w, void* ws,
                                 size_t ws_bytes, moe_stream_t stream, Marks& mk) {
    moe_config_t c;
    const moe_config_t* cfg = &c;
    moe_status_t s = effective_config(cfg_in, &c);
    if (s != MOE_OK) return s;
    if (n < 0) return MOE_ERR_INVALID_CONFIG;
    if ((s = check_router_weights(cfg, wts)) != MOE_OK) return s;
    if ((s = check_expert_weights(cfg, wts)) != MOE_OK) return s;
    if (n == 0) return MOE_OK;
    if (!x || !out) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(out) || (idx && !aligned16(idx)) || (w && !aligned16(w)))
        return MOE_ERR_ALIGNMENT;
    if (overlaps(x, out, (size_t)n * cfg->hidden * 2)) return MOE_ERR_ALIAS;
    WsLayout L;
    if ((s = check_ws(cfg, n, ws, ws_bytes, &L)) != MOE_OK) return s;
    const int x_res = residency(x);
    if (x_res < 0 || residency(out) < 0) return MOE_ERR_HOST_MEMORY;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t* idx_p = idx ? idx : at<int32_t>(ws, L.idx);
    float* w_p = w ? w : at<float>(ws, L.w);
    mk.mark(st);
    if (n == 1 && cfg->path != MOE_PATH_GROUPED && cfg->router_fmt == MOE_W_BF16) {
        // One token: the whole layer in one cooperative launch when its
        // shared-memory plan fits (same arithmetic as the kernels below).
        const int sms = device_sm_count();
        FusedParams fp{};
        if (fused_plan(cfg, sms, &fp)) {
            const int H = cfg->hidden, I = cfg->inter, S = cfg->shared_inter;
            fp.x = static_cast<const uint16_t*>(x);
            fp.H = H; fp.E = cfg->num_experts; fp.k = cfg->top_k; fp.I = I; fp.S = S;
            fp.routing = cfg->routing; fp.norm = cfg->norm_topk_prob; fp.scale = cfg->routed_scaling_factor;
            fp.e_begin = cfg->expert_begin; fp.e_end = cfg->expert_end;
            fp.accumulate = cfg->accumulate;
            fp.norm_w = static_cast<const uint16_t*>(wts->pre_expert_norm_w);
            fp.eps = cfg->rms_norm_eps;
            fp.router = static_cast<const uint16_t*>(wts->router_w);
            fp.gw = static_cast<const uint16_t*>(wts->shared_gate_w);
            fp.bias = wts->correction_bias;
            const int eb = cfg->expert_begin;
            fp.gate = qdev(wts->gate, I, H, eb);
            fp.up = qdev(wts->up, I, H, eb);
            fp.down = qdev(wts->down, H, I, eb);
            if (S > 0) {
                fp.sh_gate = qdev(wts->sh_gate, S, H, 0);
                fp.sh_up = qdev(wts->sh_up, S, H, 0);
                fp.sh_down = qdev(wts->sh_down, H, S, 0);
            }
            fp.logits = at<float>(ws, L.logits);
            fp.sg_logit = at<float>(ws, L.sg_logit);
            fp.act = at<float>(ws, L.act);
            fp.act_sh = at<float>(ws, L.act_sh);
            fp.idx_out = idx_p;
            fp.w_out = w_p;
            fp.out = static_cast<uint16_t*>(out);
            fp.ctrl = at<Ctrl>(ws, L.ctrl);
            if (launch_fused_n1(cfg->expert_fmt, fp, sms, st) == cudaSuccess) {
                mk.mark(st);
                return MOE_OK;
            }
            (void)cudaGetLastError();   // not launchable here: the multi-kernel path below
        }
    }
    // More than one token: a host-resident x is copied into the workspace
    // once, rather than read across the host link by every kernel and block.
    if (x_res == 1 && (s = stage_x(cfg, x, n, ws, L, st)) != MOE_OK) return s;
    if (local_experts(cfg) == 0 && !idx && !w) {
        // No expert held here and no routing asked for (the shared-expert call
        // of expert parallelism): only the shared-gate logit is needed.
        if (wts->shared_gate_w) {
            const cudaError_t e = launch_router(static_cast<const uint16_t*>(x), n, cfg->hidden,
                                                static_cast<const uint16_t*>(wts->router_w), 0,
                                                static_cast<const uint16_t*>(wts->shared_gate_w), nullptr,
                                                at<float>(ws, L.sg_logit), device_sm_count(), st);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
        }
        mk.mark(st);
        return enqueue_experts(cfg, wts, x, n, idx_p, w_p, out, ws, L, true, false, st, mk);
    }
    if ((s = enqueue_route(cfg, wts, x, n, idx_p, w_p, nullptr, ws, L, true, true, st, mk)) != MOE_OK) return s;
    return enqueue_experts(cfg, wts, x, n, idx_p, w_p, out, ws, L, true, true, st, mk);
}

moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* wts, const void* x, int32_t n,
                         void* out, int32_t* idx, float* w, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
    Marks mk;
    return forward_impl(cfg, wts, x, n, out, idx, w, ws, ws_bytes, stream, mk);
}

moe_status_t moe_forward_timed(const moe_config_t* cfg, const moe_weights_t* wts, const void* x,
                               int32_t n, void* out, int32_t* idx, float* w, void* ws,
                               size_t ws_bytes, moe_stream_t stream, void* const* events,
                               int32_t n_events, int32_t* n_marks) {
    if (n_events < 0 || (n_events > 0 && !events)) return MOE_ERR_NULL;
    Marks mk;
    mk.ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
    mk.n = n_events;
    const moe_status_t s = forward_impl(cfg, wts, x, n, out, idx, w, ws, ws_bytes, stream, mk);
    if (n_marks) *n_marks = mk.next;
    return s;
}

moe_status_t moe_workspace_check(void* ws, size_t ws_bytes, int32_t* device_error, moe_stream_t stream) {
    if (!ws || !device_error) return MOE_ERR_NULL;
    if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
    if (ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Ctrl* c = static_cast<Ctrl*>(ws);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, &c->err, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    // Clear the error word and the single-token kernel's barrier word (left
    // non-zero when a call ends early), so the workspace serves the next call.
    // err, gbar, routed and tc_count (adjacent): zero between calls.
    if (cudaMemsetAsync(&c->err, 0, 4 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *device_error = v;
    return MOE_OK;
}

const char* moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK: success";
        case MOE_ERR_NULL: return "MOE_ERR_NULL: a required pointer is NULL";
        case MOE_ERR_INVALID_CONFIG: return "MOE_ERR_INVALID_CONFIG: a size, enum or flag is out of range";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: configuration outside what the kernels cover";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA launch failed";
        case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT: a device pointer is not aligned (16 bytes; scales 4)";
        case MOE_ERR_ALIAS: return "MOE_ERR_ALIAS: out overlaps x";
        case MOE_ERR_HOST_MEMORY: return "MOE_ERR_HOST_MEMORY: x or out is host memory that is not pinned";
        default: return "unknown moe_status_t";
    }
}

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

}  // extern "C"

namespace moe {
// moe_forward with a workspace the caller of this function chose (used by the
// static-workspace entry point in moe_noalloc.cu).
moe_status_t forward_with_workspace(const moe_config_t* cfg, const moe_weights_t* wts, const void* x,
                                    int32_t n, void* out, int32_t* idx, float* w, void* ws,
                                    size_t ws_bytes, moe_stream_t stream) {
    Marks mk;
    return forward_impl(cfg, wts, x, n, out, idx, w, ws, ws_bytes, stream, mk);
}
}  // namespace moe
