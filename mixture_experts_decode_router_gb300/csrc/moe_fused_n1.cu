// moe_fused_n1.cu -- the whole layer for one decode token in one launch (sm_103a).
//
// MoeLayer::forward (page "metrale_model_layers/layers/moe/forward.rs") runs
// gate, topk, exp_gate_up, exp_silu_down and wsum_blend as separate launches
// for one token.  At one token every step is a short weight stream, so the
// launch and drain gaps between them cost more than the streams.  This kernel
// does all of it in one cooperative, persistent launch (one CTA per SM), with
// two grid barriers:
//
//  phase 0  every CTA computes its router rows (and the shared-gate row) and
//           starts streaming the routing-independent work: its share of the
//           shared expert's gate/up rows and its slice of the shared down rows.
//           Grid barrier 1: all logits are written.
//  phase 1  every CTA ranks the logits itself (block-wide, by counting) and
//           streams its share of the routed experts' gate/up rows straight
//           into registers (15 warps, ~120 KB of loads in flight per SM),
//           while the TMA bulk-copy engine prefetches its slice of the routed
//           down rows into shared memory.
//           Grid barrier 2: all SiLU(g)*u values are written.
//  phase 2  every CTA computes its output columns from the down rows already
//           in shared memory: first each lane's partial dot product of every
//           (expert slot, row) pair -- the pairs split evenly over the warps in
//           slot-major order, a warp's activation chunk held in registers across
//           its rows of a slot -- then per row the partials
//           weighted in slot order, the gated shared expert, the butterfly
//           and the BF16 write.
//
// The arithmetic of every dot product, the top-k weights and the blend is the
// same, operation for operation, as the token-major kernels' for one token,
// so a token's output bits do not depend on which path or batch computed it.
//
// Warp 15 (one lane) issues the bulk copies; warps 0-14 compute.  Every wait is
// bounded (2 s), records an error code in the workspace and ends the kernel.
#include <mutex>

#include "moe_launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kFThreads = 512;
constexpr int kFComputeWarps = 15;
constexpr int kFCompute = kFComputeWarps * 32;
constexpr int kSeg = 8;   // row chunks per lane loaded before they are used

template <int FMT>
__device__ __forceinline__ void decode_at(const uint8_t* row, int c, float (&v)[8]) {
    WChunk<FMT> ch;
    if constexpr (FMT == MOE_W_BF16) ch.raw = *reinterpret_cast<const uint4*>(row + c * 16);
    else if constexpr (FMT == MOE_W_FP8_B128) ch.raw = *reinterpret_cast<const uint2*>(row + c * 8);
    else ch.raw = *reinterpret_cast<const uint32_t*>(row + c * 4);
    ch.decode(v);
}

__device__ __forceinline__ size_t row_bytes_of(int fmt, int in_dim) {
    return fmt == MOE_W_BF16 ? (size_t)in_dim * 2 : (fmt == MOE_W_FP8_B128 ? (size_t)in_dim : (size_t)in_dim / 2);
}

template <int FMT>
__device__ __forceinline__ const uint8_t* row_ptr(const QMatDev& m, int e, int row) {
    return m.w + ((size_t)(e - m.e_base) * m.out_dim + row) * row_bytes_of(FMT, m.in_dim);
}

template <int FMT>
__global__ void __launch_bounds__(kFThreads, 1) fused_n1_kernel(const FusedParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int H = p.H, E = p.E, k = p.k, I = p.I, S = p.S;

    uint16_t* sx = reinterpret_cast<uint16_t*>(sm + p.off_x);
    float* slg = reinterpret_cast<float*>(sm + p.off_lg);
    unsigned long long* skey = reinterpret_cast<unsigned long long*>(sm + p.off_sc);   // [E + 32]
    int* ssel = reinterpret_cast<int*>(sm + p.off_sel);
    float* sselw = reinterpret_cast<float*>(sm + p.off_sel + 128);
    uint8_t* sdown = sm + p.off_down;
    float* sact = reinterpret_cast<float*>(sm + p.off_act);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
    uint64_t* dfull = bars;
    uint64_t* dshfull = bars + 1;
    uint64_t* sel_ready = bars + 2;
    uint64_t* shgu_full = bars + 3;
    volatile int* abort_f = reinterpret_cast<volatile int*>(bars + 4);
    volatile int* s_go = abort_f + 1;   // phase decision, written by tid 0 before a barrier
    Ctrl* ctrl = p.ctrl;
    int32_t* err = &ctrl->err;

    // The barrier word must be below G at the start of a call (zeroed once,
    // returned to zero by every call); anything else is a workspace that was
    // not initialised (or a call that failed): refuse before writing anything.
    // The word is read early and tested after x is staged, so its latency and
    // x's overlap.
    uint32_t gbar0 = 0;
    if (tid == 0) {
        gbar0 = ptx::ld_relaxed_gpu(&ctrl->gbar);
        ptx::mbar_init(dfull, 1);
        ptx::mbar_init(dshfull, 1);
        ptx::mbar_init(sel_ready, 1);
        ptx::mbar_init(shgu_full, 1);
        ptx::fence_mbar_init();
    }
    // Router row of this warp (r == E: the shared-gate row): its first chunks
    // are requested before x is staged, so the two loads overlap.
    const int C = H >> 3;
    const int r_row = cta + G * warp;
    const bool has_row = warp < kFComputeWarps && r_row < E + (p.gw ? 1 : 0);
    const uint16_t* wrow = has_row ? ((r_row < E) ? p.router + (size_t)r_row * H : p.gw) : nullptr;
    uint4 rw[kSeg];
    if (has_row) {
#pragma unroll
        for (int i = 0; i < kSeg; ++i) {
            const int c = lane + 32 * i;
            if (c < C) rw[i] = __ldg(reinterpret_cast<const uint4*>(wrow) + c);
        }
    }
    for (int i = tid; i < H / 8; i += kFThreads)
        reinterpret_cast<uint4*>(sx)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
    if (tid == 0) {
        const bool clean = gbar0 < (uint32_t)G;
        if (!clean) atomicExch(err, 20);
        *abort_f = clean ? 0 : 2;
    }
    __syncthreads();
    const bool refused = *abort_f == 2;
    // The experts' input: x, or its pre-expert RMSNorm (the norm kernel's
    // arithmetic); the router keeps x.
    const uint16_t* sxe = sx;
    if (p.norm_w) {
        uint16_t* sxn = reinterpret_cast<uint16_t*>(sm + p.off_xe);
        float* s_inv = reinterpret_cast<float*>(sm + p.off_sel + 256);
        if (warp == 0) {
            const float inv = rms_inv_warp(sx, H, p.eps, lane);
            if (lane == 0) *s_inv = inv;
        }
        __syncthreads();
        const float inv = *s_inv;
        for (int c = tid; c < H / 8; c += kFThreads)
            reinterpret_cast<uint4*>(sxn)[c] = rms_apply8(reinterpret_cast<const uint4*>(sx)[c],
                                                          __ldg(reinterpret_cast<const uint4*>(p.norm_w) + c), inv);
        __syncthreads();
        sxe = sxn;
    }
    auto local = [&](int e) { return e >= p.e_begin && e < p.e_end; };

    // Work of this CTA.
    const int rpc = p.rpc;
    const int h0 = cta * rpc, h1 = min(H, h0 + rpc), nrows = max(0, h1 - h0);
    const int sh_b = (int)((int64_t)S * cta / G), sh_e = (int)((int64_t)S * (cta + 1) / G);
    const int64_t Q = (int64_t)k * I;
    const int r_b = (int)(Q * cta / G), r_e = (int)(Q * (cta + 1) / G);
    const int n_sh = sh_e - sh_b, n_r = r_e - r_b;

    if (refused) {
        // nothing: the error word says why
    } else if (warp == kFComputeWarps) {
        // ------------------------------------------------------------ copy producer
        if (lane == 0) {
            bool ok = true;
            // The CTA's shared gate/up rows (needed first), the shared down
            // slice (routing-independent), then the routed down slices.
            uint8_t* sshgu = sm + p.off_shgu;
            if (S > 0 && n_sh > 0) {
                const uint32_t bytes = (uint32_t)n_sh * p.row_bytes;
                ptx::mbar_arrive_expect_tx(shgu_full, 2 * bytes);
                ptx::bulk_load(sshgu, row_ptr<FMT>(p.sh_gate, 0, sh_b), bytes, shgu_full);
                ptx::bulk_load(sshgu + bytes, row_ptr<FMT>(p.sh_up, 0, sh_b), bytes, shgu_full);
            } else {
                ptx::mbar_arrive(shgu_full);
            }
            if (S > 0 && nrows > 0) {
                ptx::mbar_arrive_expect_tx(dshfull, nrows * p.dsh_row_bytes);
                ptx::bulk_load(sdown + (size_t)k * rpc * p.drow_bytes, row_ptr<FMT>(p.sh_down, 0, h0),
                               nrows * p.dsh_row_bytes, dshfull);
            } else {
                ptx::mbar_arrive(dshfull);
            }
            ok = ptx::mbar_wait(sel_ready, 0, abort_f, err, 12);
            int n_local = 0;
            if (ok)
                for (int j = 0; j < k; ++j) n_local += local(ssel[j]) ? 1 : 0;
            if (ok && nrows > 0 && n_local > 0) {
                ptx::mbar_arrive_expect_tx(dfull, (uint32_t)(n_local * nrows * p.drow_bytes));
                for (int j = 0; j < k; ++j)
                    if (local(ssel[j]))
                        ptx::bulk_load(sdown + (size_t)j * rpc * p.drow_bytes, row_ptr<FMT>(p.down, ssel[j], h0),
                                       nrows * p.drow_bytes, dfull);
            } else if (ok) {
                ptx::mbar_arrive(dfull);
            } else {
                // Let the copies issued land before the CTA exits.
                ptx::mbar_wait_quiet(shgu_full, 0, 100000000ull);
                ptx::mbar_wait_quiet(dshfull, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ compute warps
        // Phase 0a: the router row of this warp, with the router kernel's chunk order.
        if (has_row) {
            float acc = 0.f;
            for (int c0 = 0; c0 < C; c0 += 32 * kSeg) {
#pragma unroll
                for (int i = 0; i < kSeg; ++i) {
                    const int c = c0 + lane + 32 * i;
                    if (c < C) {
                        const uint4 raw = (c0 == 0) ? rw[i] : __ldg(reinterpret_cast<const uint4*>(wrow) + c);
                        float wv[8], xv[8];
                        bf16x8_to_float(raw, wv);
                        bf16x8_to_float(reinterpret_cast<const uint4*>(sx)[c], xv);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc = fmaf(wv[q], xv[q], acc);
                    }
                }
            }
            const float s = warp_sum(acc);
            if (lane == 0) {
                if (r_row < E) p.logits[r_row] = s;
                else *p.sg_logit = s;
            }
        }
        ptx::named_bar(1, kFCompute);
        if (tid == 0) ptx::red_add_release_gpu(&ctrl->gbar, 1u);   // barrier 1 arrival

        // One gate/up row pair: SiLU(g) * u of weight row `row`, written to dst,
        // with the token-major gate_up kernel's arithmetic.  Each segment's
        // loads are all issued before any is used.
        auto consume = [&](const QMatDev& Gm, const QMatDev& Um, int e, int row, float msg, float msu,
                           float* dst) {
            float ag = 0.f, au = 0.f;
            for (int c0 = lane; c0 < C; c0 += 32 * kSeg) {
                WChunk<FMT> cg[kSeg], cu[kSeg];
#pragma unroll
                for (int i = 0; i < kSeg; ++i) {
                    const int c = c0 + 32 * i;
                    if (c < C) {
                        cg[i].load(Gm, e, row, c);
                        cu[i].load(Um, e, row, c);
                    }
                }
#pragma unroll
                for (int i = 0; i < kSeg; ++i) {
                    const int c = c0 + 32 * i;
                    if (c < C) {
                        float wg[8], wu[8], xv[8];
                        cg[i].decode(wg);
                        cu[i].decode(wu);
                        const float sg = cg[i].scale(Gm, e, row, c), su = cu[i].scale(Um, e, row, c);
                        bf16x8_to_float(reinterpret_cast<const uint4*>(sxe)[c], xv);
                        ag = fmaf(dot8(wg, xv), sg, ag);
                        au = fmaf(dot8(wu, xv), su, au);
                    }
                }
            }
            const float g = warp_sum(ag) * msg;
            const float u = warp_sum(au) * msu;
            if (lane == 0) *dst = silu(g) * u;
        };

        // Phase 0b: the shared expert's gate/up rows of this CTA, from the copy
        // the producer started at kernel entry (the same arithmetic as consume).
        const float msg_sh = S > 0 ? matrix_scale<FMT>(p.sh_gate, 0) : 1.f;
        const float msu_sh = S > 0 ? matrix_scale<FMT>(p.sh_up, 0) : 1.f;
        if (warp < n_sh && ptx::mbar_wait_warp(shgu_full, 0, abort_f, err, 17)) {
            const uint8_t* sshgu = sm + p.off_shgu;
            for (int s = warp; s < n_sh; s += kFComputeWarps) {
                const uint8_t* grow = sshgu + (size_t)s * p.row_bytes;
                const uint8_t* urow = sshgu + (size_t)(n_sh + s) * p.row_bytes;
                const int row = sh_b + s;
                float ag = 0.f, au = 0.f;
                for (int c0 = lane; c0 < C; c0 += 32 * kSeg) {
#pragma unroll
                    for (int i = 0; i < kSeg; ++i) {
                        const int c = c0 + 32 * i;
                        if (c < C) {
                            float wg[8], wu[8], xv[8];
                            decode_at<FMT>(grow, c, wg);
                            decode_at<FMT>(urow, c, wu);
                            WChunk<FMT> sch;
                            const float sg = sch.scale(p.sh_gate, 0, row, c), su = sch.scale(p.sh_up, 0, row, c);
                            bf16x8_to_float(reinterpret_cast<const uint4*>(sxe)[c], xv);
                            ag = fmaf(dot8(wg, xv), sg, ag);
                            au = fmaf(dot8(wu, xv), su, au);
                        }
                    }
                }
                const float g = warp_sum(ag) * msg_sh;
                const float u = warp_sum(au) * msu_sh;
                if (lane == 0) p.act_sh[row] = silu(g) * u;
            }
        }

        // Grid barrier 1: every logit is written.
        ptx::named_bar(1, kFCompute);
        if (tid == 0) {
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::ld_acquire_gpu(&ctrl->gbar) < (uint32_t)G) {
                if (*abort_f) break;
                if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                    atomicExch(err, 14);
                    *abort_f = 1;
                    break;
                }
            }
            *s_go = *abort_f ? 0 : 1;
        }
        ptx::named_bar(1, kFCompute);
        const bool go1 = *s_go != 0;    // the same value for every compute thread

        if (go1) {
            // Phase 1a: routing, computed by every CTA for itself.
            for (int e = tid; e < E + 32; e += kFCompute) {
                if (e < E) {
                    const float l = __ldcg(p.logits + e);
                    float sc;
                    if (p.routing == MOE_ROUTE_SOFTMAX) sc = l;
                    else sc = 1.0f / (1.0f + expf(-l)) + p.bias[e];
                    if (sc != sc) sc = -INFINITY;
                    slg[e] = l;
                    skey[e] = route_key(sc, e);
                } else {
                    skey[e] = 0ull;
                }
            }
            ptx::named_bar(1, kFCompute);
            // Selection, with the top-k kernel's arithmetic; the copy producer
            // starts on the routed down rows as soon as it is known.  The
            // weights are formed later, while grid barrier 2 fills.
            unsigned long long* cand_k = reinterpret_cast<unsigned long long*>(sm + p.off_cand);
            float* gmax = reinterpret_cast<float*>(cand_k + p.n_cand);
            route_select_block(slg, skey, E, k, p.routing, tid, kFCompute, cand_k, gmax, ssel,
                               [] { ptx::named_bar(1, kFCompute); });
            if (tid == 0) ptx::mbar_arrive(sel_ready);

            // Phase 1b: the routed gate/up rows of this CTA.
            // Items continue the shared ones' warp rotation, so the CTA's warps
            // stay evenly loaded.
            for (int s = warp; s < n_sh + n_r; s += kFComputeWarps) {
                if (s < n_sh) continue;
                const int q = r_b + (s - n_sh);
                const int j = q / I, i = q - j * I, e = ssel[j];
                if (!local(e)) continue;   // held by another call (expert parallelism)
                consume(p.gate, p.up, e, i, matrix_scale<FMT>(p.gate, e), matrix_scale<FMT>(p.up, e),
                        p.act + (size_t)j * I + i);
            }
        }

        // Grid barrier 2: every SiLU(g) * u is written.  The routing weights
        // (needed from phase 2 on) are formed between the arrival and the wait.
        ptx::named_bar(1, kFCompute);
        uint32_t old2 = 0;
        const bool arrived2 = tid == 0 && !*abort_f;
        if (arrived2) old2 = ptx::atom_add_acq_rel_gpu(&ctrl->gbar, 1u);
        if (go1) {
            float* gmax = reinterpret_cast<float*>(reinterpret_cast<unsigned long long*>(sm + p.off_cand) + p.n_cand);
            route_weights_block(slg, E, k, p.routing, p.norm, p.scale, tid, kFCompute, gmax, gmax + 32, ssel,
                                sselw, [] { ptx::named_bar(1, kFCompute); });
            if (cta == 0 && tid < k) {
                p.idx_out[tid] = ssel[tid];
                p.w_out[tid] = sselw[tid];
            }
        }
        if (tid == 0) {
            if (arrived2) {
                // The last CTA to arrive returns the word to zero for the next
                // call; the others stop waiting at 2G or at that zero (the word
                // cannot be zero again before this call ends).
                const uint32_t old = old2;
                if (old == 2u * G - 1) {
                    ptx::st_relaxed_gpu(&ctrl->gbar, 0u);
                } else {
                    const uint64_t t0 = ptx::globaltimer();
                    for (;;) {
                        const uint32_t v = ptx::ld_acquire_gpu(&ctrl->gbar);
                        if (v >= 2u * G || v == 0) break;
                        if (*abort_f) break;
                        if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                            atomicExch(err, 15);
                            *abort_f = 1;
                            break;
                        }
                    }
                }
            }
            *s_go = *abort_f ? 0 : 1;
        }
        ptx::named_bar(1, kFCompute);
        const bool go2 = *s_go != 0;

        if (go2 && nrows > 0) {
            // Phase 2: down rows [h0, h1) from shared memory.
            // SiLU(g) * u of every route, then of the shared expert, contiguous in
            // shared memory; each thread issues its loads before storing any.
            {
                const int n4 = (k * I) >> 2, t4 = n4 + (S >> 2);
                const float4* a4 = reinterpret_cast<const float4*>(p.act);
                const float4* s4 = reinterpret_cast<const float4*>(p.act_sh);
                constexpr int kB = 4;
                for (int i0 = tid; i0 < t4; i0 += kB * kFCompute) {
                    float4 v[kB];
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int i = i0 + b * kFCompute;
                        if (i < t4) v[b] = __ldcg(i < n4 ? a4 + i : s4 + (i - n4));
                    }
#pragma unroll
                    for (int b = 0; b < kB; ++b) {
                        const int i = i0 + b * kFCompute;
                        if (i < t4) reinterpret_cast<float4*>(sact)[i] = v[b];
                    }
                }
            }
            ptx::named_bar(1, kFCompute);
            const bool ok_w = ptx::mbar_wait_warp(dfull, 0, abort_f, err, 16) &&
                              ptx::mbar_wait_warp(dshfull, 0, abort_f, err, 16);
            if (!ok_w) *s_go = 0;              // one decision for every compute warp
            ptx::named_bar(1, kFCompute);
            if (*s_go != 0) {
                // Phase 2a: each lane's partial dot product of every (slot, row) of
                // this CTA -- slot j < k a routed expert, slot k the shared one --
                // with the token-major kernel's chunk order.  The (slot, row) pairs
                // are split evenly over the warps in slot-major order; a warp walks
                // exactly its rows.
                float* spart = reinterpret_cast<float*>(sm + p.off_part);   // [J][rpc][32]
                const int J = k + (S > 0 ? 1 : 0);
                const int P = J * nrows;
                const int q1 = (int)((int64_t)P * (warp + 1) / kFComputeWarps);
                for (int q = (int)((int64_t)P * warp / kFComputeWarps); q < q1;) {
                    const int j = q / nrows, rb0 = q - j * nrows;
                    const int nr = min(q1 - q, nrows - rb0);   // this warp's rows of slot j
                    q += nr;
                    const bool shj = S > 0 && j == k;
                    const int e = shj ? 0 : ssel[j];
                    if (!shj && !local(e)) continue;
                    const QMatDev& M = shj ? p.sh_down : p.down;
                    const int K = shj ? S : I;
                    const float* a = sact + (size_t)j * I;
                    const uint8_t* base = sdown + (size_t)j * rpc * p.drow_bytes;
                    const uint32_t rb = shj ? p.dsh_row_bytes : p.drow_bytes;
                    const int C8 = K >> 3;
                    auto load_act = [&](int c, float (&av)[8]) {
                        const float4 a0 = reinterpret_cast<const float4*>(a)[2 * c];
                        const float4 a1 = reinterpret_cast<const float4*>(a)[2 * c + 1];
                        av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
                        av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
                    };
                    auto term = [&](int r, int c, const float (&av)[8], float acc) {
                        float wv[8];
                        decode_at<FMT>(base + (size_t)r * rb, c, wv);
                        WChunk<FMT> sch;
                        return fmaf(dot8(wv, av), sch.scale(M, e, h0 + r, c), acc);
                    };
                    if (C8 <= 64) {
                        // At most two chunks a lane (c = lane, lane + 32): the slot's
                        // activation chunks stay in registers across its rows, and
                        // rows go two at a time (independent chains).
                        const bool two = lane + 32 < C8, one = lane < C8;
                        float av0[8], av1[8];
                        if (one) load_act(lane, av0);
                        if (two) load_act(lane + 32, av1);
                        int r = rb0;
                        for (; r + 1 < rb0 + nr; r += 2) {
                            float p0 = 0.f, p1 = 0.f;
                            if (one) { p0 = term(r, lane, av0, p0); p1 = term(r + 1, lane, av0, p1); }
                            if (two) { p0 = term(r, lane + 32, av1, p0); p1 = term(r + 1, lane + 32, av1, p1); }
                            spart[((size_t)j * rpc + r) * 32 + lane] = p0;
                            spart[((size_t)j * rpc + r + 1) * 32 + lane] = p1;
                        }
                        if (r < rb0 + nr) {
                            float p0 = 0.f;
                            if (one) p0 = term(r, lane, av0, p0);
                            if (two) p0 = term(r, lane + 32, av1, p0);
                            spart[((size_t)j * rpc + r) * 32 + lane] = p0;
                        }
                    } else {
                        for (int r = rb0; r < rb0 + nr; ++r) {
                            float part = 0.f;
                            for (int c = lane; c < C8; c += 32) {
                                float av[8];
                                load_act(c, av);
                                part = term(r, c, av, part);
                            }
                            spart[((size_t)j * rpc + r) * 32 + lane] = part;
                        }
                    }
                }
                ptx::named_bar(1, kFCompute);
                // Phase 2b: per output row, the slots' partials weighted in slot
                // order, the gated shared expert last, then the butterfly.
                float gs = 1.0f;
                if (p.gw) gs = 1.0f / (1.0f + expf(-__ldcg(p.sg_logit)));
                if (S > 0) gs *= matrix_scale<FMT>(p.sh_down, 0);
                for (int h = h0 + warp; h < h1; h += kFComputeWarps) {
                    const int r = h - h0;
                    float acc = 0.f;
                    for (int j0 = 0; j0 < k; j0 += 8) {
                        // Eight slots' loads first, then their terms in slot order.
                        float pv[8], wv[8];
                        bool lv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int j = j0 + u;
                            const int e = j < k ? ssel[j] : -1;
                            lv[u] = j < k && local(e);
                            pv[u] = lv[u] ? spart[((size_t)j * rpc + r) * 32 + lane] : 0.f;
                            wv[u] = lv[u] ? sselw[j] * matrix_scale<FMT>(p.down, e) : 0.f;
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (lv[u]) acc = fmaf(pv[u], wv[u], acc);
                    }
                    if (S > 0) acc = fmaf(spart[((size_t)k * rpc + r) * 32 + lane], gs, acc);
                    float s = warp_sum(acc);
                    if (lane == 0) {
                        if (p.accumulate) s += __uint_as_float((uint32_t)p.out[h] << 16);
                        const __nv_bfloat16 b = __float2bfloat16_rn(s);
                        p.out[h] = *reinterpret_cast<const uint16_t*>(&b);
                    }
                }
            }
        }
    }

    __syncthreads();
}

}  // namespace

// Shared-memory plan of the fused kernel; returns false if it does not fit.
bool fused_plan(const moe_config_t* c, int num_sms, FusedParams* p) {
    const int H = c->hidden, E = c->num_experts, k = c->top_k, I = c->inter, S = c->shared_inter;
    auto rb = [&](int in_dim) -> uint32_t {
        return c->expert_fmt == MOE_W_BF16 ? in_dim * 2 : (c->expert_fmt == MOE_W_FP8_B128 ? in_dim : in_dim / 2);
    };
    p->rpc = (H + num_sms - 1) / num_sms;
    p->row_bytes = rb(H);
    p->drow_bytes = rb(I);
    p->dsh_row_bytes = rb(S > 0 ? S : 32);
    if (S > 0 && p->dsh_row_bytes > p->drow_bytes) return false;   // the shared slice uses the routed slot size
    if (E + 1 > kFComputeWarps * num_sms) return false;              // one router row per compute warp
    size_t off = 0;
    auto take = [&](size_t b, size_t al) { off = (off + al - 1) / al * al; size_t o = off; off += b; return (uint32_t)o; };
    p->off_x = take((size_t)H * 2, 128);
    p->off_xe = take((size_t)H * 2, 128);
    p->off_lg = take((size_t)E * 4, 16);
    p->off_sc = take((size_t)(E + 32) * 8, 16);   // selection keys, zero-padded
    p->off_sel = take(256 + 16, 16);   // 32 experts, 32 weights, the inverse RMS
    p->n_cand = (E + 31) / 32 * k;     // top-k candidate keys, group maxima and sums
    p->off_cand = take((size_t)p->n_cand * 8 + 2 * 32 * 4, 16);
    p->off_down = take((size_t)(k + 1) * p->rpc * p->drow_bytes, 128);
    p->off_act = take(((size_t)k * I + (S > 0 ? S : 0)) * 4, 16);
    p->off_part = take((size_t)(k + (S > 0 ? 1 : 0)) * p->rpc * 32 * 4, 16);   // phase-2 lane partials
    // The CTA's shared gate and up rows: at most ceil(S / #SM) of each.
    p->off_shgu = take((size_t)2 * ((S + num_sms - 1) / num_sms) * p->row_bytes, 128);
    // dfull, dshfull, sel_ready, shgu_full, abort + phase flags
    p->off_bar = take(4 * 8 + 16, 8);
    p->smem_bytes = (uint32_t)off;
    return off <= 227 * 1024 && k <= 32 && (size_t)k * p->rpc * p->drow_bytes < (1u << 20);
}

cudaError_t launch_fused_n1(int fmt, const FusedParams& p, int num_sms, cudaStream_t st) {
    const void* fn = nullptr;
    switch (fmt) {
        case MOE_W_BF16: fn = reinterpret_cast<const void*>(fused_n1_kernel<MOE_W_BF16>); break;
        case MOE_W_FP8_B128: fn = reinterpret_cast<const void*>(fused_n1_kernel<MOE_W_FP8_B128>); break;
        case MOE_W_NVFP4: fn = reinterpret_cast<const void*>(fused_n1_kernel<MOE_W_NVFP4>); break;
        default: return cudaErrorInvalidValue;
    }
    // Per device and format: the largest dynamic shared memory configured so
    // far (set once, re-set only when a larger plan arrives).
    static std::mutex mu;
    static uint32_t configured[128][3] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev][fmt] < p.smem_bytes) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)p.smem_bytes);
            if (e != cudaSuccess) return e;
            int per_sm = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kFThreads, p.smem_bytes);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
            configured[dev][fmt] = p.smem_bytes;
        }
    }
    FusedParams pc = p;
    void* args[] = {&pc};
    return cudaLaunchCooperativeKernel(fn, dim3(num_sms), dim3(kFThreads), args, p.smem_bytes, st);
}

}  // namespace moe
