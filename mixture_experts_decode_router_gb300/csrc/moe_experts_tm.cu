// moe_experts_tm.cu -- token-major expert stage for small batches (sm_103a).
//
// The expert steps of MoeLayer::forward (page "metrale_model_layers/layers/moe/
// forward.rs": exp_gate_up, exp_silu_down and wsum_blend, routed experts and
// the always-on shared expert together) and of forward_token_major_decode
// (page "spark_model/layers/moe/forward_token_major.rs": gate+up, silu+down,
// weighted sum and blend over all (token, expert-slot) routes).
//
// Two kernels on CUDA cores (the decode batch is too thin for a tensor-core
// tile to pay):
//  * gate_up: one warp per (unit, row i) pair, where a unit is an expert that
//    at least one token chose (read from the device-built expert grouping, so
//    an expert that two tokens chose is streamed once) or the shared expert.
//    The warp streams row i of the unit's gate and up matrices once, with
//    128-bit (BF16), 64-bit (FP8) or 32-bit (NVFP4) coalesced loads that skip
//    L1, dequantises in registers, and dots them with every token of the unit:
//    act[route, i] = SiLU(g) * u in fp32.
//  * down_blend: one warp per output column h.  For each token it sums, over
//    the token's slots in order, w * (Wd[e][h, :] . act[route, :]), adds the
//    gated shared expert and writes the BF16 output: down projection,
//    weighted sum and blend in one pass, with no atomics.
// Every dot product has a fixed lane order and butterfly, independent of the
// batch, so a token's output does not depend on which tokens share the call.
#include "moe_launch.cuh"

namespace moe {

template <int FMT, int TB>
__global__ void __launch_bounds__(256, 2)
gate_up_tm_kernel(const GateUpParams p) {
    const int lane = threadIdx.x & 31;
    const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    pdl_wait();
    const int n_active = p.ctrl->n_active;
    const int64_t routed_rows = (int64_t)n_active * p.I;
    const int64_t R = routed_rows + (p.S > 0 ? p.S : 0);
    const int C = p.H >> 3;

    for (int64_t q = gwarp; q < R; q += nwarps) {
        const bool shared = q >= routed_rows;
        int e = 0, row, first = 0, cnt, Iu;
        if (!shared) {
            const int u = (int)(q / p.I);
            row = (int)(q - (int64_t)u * p.I);
            e = p.active[u];
            first = p.offsets[e];
            cnt = p.counts[e];
            Iu = p.I;
        } else {
            row = (int)(q - routed_rows);
            cnt = p.n;
            Iu = p.S;
        }
        const QMatDev& G = shared ? p.sh_gate : p.gate;
        const QMatDev& U = shared ? p.sh_up : p.up;
        const float msg = matrix_scale<FMT>(G, e), msu = matrix_scale<FMT>(U, e);

        for (int tb0 = 0; tb0 < cnt; tb0 += TB) {
            int tok[TB], route[TB];
#pragma unroll
            for (int q2 = 0; q2 < TB; ++q2) {
                const int j = tb0 + q2;
                if (j < cnt) {
                    const int r = shared ? j : p.perm[first + j];
                    route[q2] = r;
                    tok[q2] = shared ? j : r / p.k;
                } else {
                    route[q2] = -1;
                    tok[q2] = 0;
                }
            }
            float ag[TB], au[TB];
#pragma unroll
            for (int q2 = 0; q2 < TB; ++q2) { ag[q2] = 0.f; au[q2] = 0.f; }

            // The lane's chunks c = lane, lane+32, ... in order; each segment's
            // weight loads are all issued before any of them is used.
            constexpr int SEG = (FMT == MOE_W_BF16 && TB >= 8) ? 4 : 8;
            for (int c0 = lane; c0 < C; c0 += 32 * SEG) {
                WChunk<FMT> cg[SEG], cu[SEG];
#pragma unroll
                for (int i = 0; i < SEG; ++i) {
                    const int c = c0 + 32 * i;
                    if (c < C) {
                        cg[i].load(G, e, row, c);
                        cu[i].load(U, e, row, c);
                    }
                }
#pragma unroll
                for (int i = 0; i < SEG; ++i) {
                    const int c = c0 + 32 * i;
                    if (c < C) {
                        const float sg = cg[i].scale(G, e, row, c), su = cu[i].scale(U, e, row, c);
                        float wg[8], wu[8];
                        cg[i].decode(wg);
                        cu[i].decode(wu);
#pragma unroll
                        for (int q2 = 0; q2 < TB; ++q2) {
                            if (route[q2] >= 0) {
                                float xv[8];
                                bf16x8_to_float(
                                    __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)tok[q2] * p.H) + c), xv);
                                ag[q2] = fmaf(dot8(wg, xv), sg, ag[q2]);
                                au[q2] = fmaf(dot8(wu, xv), su, au[q2]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int q2 = 0; q2 < TB; ++q2) {
                const float g = warp_sum(ag[q2]) * msg;
                const float u = warp_sum(au[q2]) * msu;
                if (lane == 0 && route[q2] >= 0) {
                    float* dst = shared ? p.act_sh : p.act;
                    dst[(size_t)route[q2] * Iu + row] = silu(g) * u;
                }
            }
        }
    }
    pdl_trigger();
}

template <int FMT>
__device__ __forceinline__ float row_dot_act(const QMatDev& M, int e, int h, const float* a, int K,
                                             int lane) {
    float acc = 0.f;
    const int C = K >> 3;
#pragma unroll 2
    for (int c = lane; c < C; c += 32) {
        WChunk<FMT> ch;
        ch.load(M, e, h, c);
        const float cs = ch.scale(M, e, h, c);
        float wv[8], av[8];
        ch.decode(wv);
        const float4 a0 = __ldg(reinterpret_cast<const float4*>(a) + 2 * c);
        const float4 a1 = __ldg(reinterpret_cast<const float4*>(a) + 2 * c + 1);
        av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
        av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
        acc = fmaf(dot8(wv, av), cs, acc);
    }
    return acc;
}

template <int FMT>
__global__ void __launch_bounds__(256, 2)
down_blend_tm_kernel(const DownParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;

    for (int h = gwarp; h < p.H; h += nwarps) {
        for (int t = 0; t < p.n; ++t) {
            float acc = 0.f;
            for (int j = 0; j < p.k; ++j) {
                const int r = t * p.k + j;
                const int e = __ldg(p.idx + r);
                if (e < p.e_begin || e >= p.e_end) continue;   // dropped route (see the grouping)
                const float wt = __ldg(p.w + r) * matrix_scale<FMT>(p.down, e);
                acc = fmaf(row_dot_act<FMT>(p.down, e, h, p.act + (size_t)r * p.I, p.I, lane), wt, acc);
            }
            if (p.S > 0) {
                float gs = 1.0f;
                if (p.sg_logit) gs = 1.0f / (1.0f + expf(-__ldg(p.sg_logit + t)));
                gs *= matrix_scale<FMT>(p.sh_down, 0);
                acc = fmaf(row_dot_act<FMT>(p.sh_down, 0, h, p.act_sh + (size_t)t * p.S, p.S, lane), gs,
                           acc);
            }
            float s = warp_sum(acc);
            if (lane == 0) {
                uint16_t* o = p.out + (size_t)t * p.H + h;
                if (p.accumulate) s += __uint_as_float((uint32_t)*o << 16);
                const __nv_bfloat16 b = __float2bfloat16_rn(s);
                *o = *reinterpret_cast<const uint16_t*>(&b);
            }
        }
    }
    pdl_trigger();
}

template <int FMT>
static cudaError_t launch_gate_up_fmt(const GateUpParams& gu, int num_sms, cudaStream_t st) {
    const dim3 grid(2 * num_sms), block(256);
    // Tokens per pass over a weight row: as many as a unit can have, up to 8
    // (BF16) or 4 (FP8 / NVFP4, whose dequantisation needs more registers).
    constexpr int kMaxTB = (FMT == MOE_W_BF16) ? 8 : 4;
    const int tb = gu.n >= kMaxTB ? kMaxTB : (gu.n >= 4 ? 4 : (gu.n >= 2 ? 2 : 1));
    if (tb == 1) launch_pdl(gate_up_tm_kernel<FMT, 1>, grid, block, 0, st, gu);
    else if (tb == 2) launch_pdl(gate_up_tm_kernel<FMT, 2>, grid, block, 0, st, gu);
    else if (tb == 4) launch_pdl(gate_up_tm_kernel<FMT, 4>, grid, block, 0, st, gu);
    else launch_pdl(gate_up_tm_kernel<FMT, kMaxTB>, grid, block, 0, st, gu);
    return cudaGetLastError();
}

cudaError_t launch_gate_up_tm(int fmt, const GateUpParams& gu, int num_sms, cudaStream_t st) {
    switch (fmt) {
        case MOE_W_BF16: return launch_gate_up_fmt<MOE_W_BF16>(gu, num_sms, st);
        case MOE_W_FP8_B128: return launch_gate_up_fmt<MOE_W_FP8_B128>(gu, num_sms, st);
        case MOE_W_NVFP4: return launch_gate_up_fmt<MOE_W_NVFP4>(gu, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_down_blend_tm(int fmt, const DownParams& dn, int num_sms, cudaStream_t st) {
    const dim3 grid(2 * num_sms), block(256);
    switch (fmt) {
        case MOE_W_BF16: launch_pdl(down_blend_tm_kernel<MOE_W_BF16>, grid, block, 0, st, dn); break;
        case MOE_W_FP8_B128: launch_pdl(down_blend_tm_kernel<MOE_W_FP8_B128>, grid, block, 0, st, dn); break;
        case MOE_W_NVFP4: launch_pdl(down_blend_tm_kernel<MOE_W_NVFP4>, grid, block, 0, st, dn); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace moe
