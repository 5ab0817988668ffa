// moe_route.cu -- router logits and top-k routing (sm_103a).
//
// Router: the "gate" step of MoeLayer::forward (page
// "metrale_model_layers/layers/moe/forward.rs") and the gate GEMM of
// forward_token_major_decode (page "spark_model/layers/moe/forward_token_major.rs"):
// logits[t, e] = sum_h x[t, h] * Wr[e, h] in fp32.  The page
// "metrale_model_layers/layers/moe/forward_fp8_grouped_router.rs" (router_block_rows)
// shows a row-grouped router GEMV in which every block row re-reads the whole
// router; here each warp owns one router row and walks every token row of the
// call against it, so the router crosses HBM once per launch and the other rows
// hit L1/L2.
//
// Top-k: the "topk" step (moe_topk_softmax_batched / moe_topk_sigmoid_batched
// on the same pages): one warp per token row.
#include "moe_launch.cuh"

namespace moe {

// Each warp: one router row r (r < E: expert r; r == E: the shared-expert gate
// weight, written to sg_logit).  blockIdx.y selects a contiguous range of token
// rows.  The arithmetic of one (row, expert) dot product -- lane l accumulates
// chunks l, l+32, ... of 8 elements in order, then a fixed butterfly -- is the
// same for every n and every grid, so a row's logits never depend on which
// other rows share the launch.
__global__ void __launch_bounds__(128)
router_kernel(const uint16_t* __restrict__ x, int n, int H,
              const uint16_t* __restrict__ wr, int E,
              const uint16_t* __restrict__ gw,
              float* __restrict__ logits, float* __restrict__ sg_logit,
              int rows_per_block) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + warp;
    const int n_rows_router = E + (gw ? 1 : 0);
    if (r >= n_rows_router) return;
    const uint16_t* wrow = (r < E) ? wr + (size_t)r * H : gw;
    const int t_begin = blockIdx.y * rows_per_block;
    const int t_end = min(n, t_begin + rows_per_block);
    const int C = H >> 3;   // 8-element chunks per row

    for (int t0 = t_begin; t0 < t_end; t0 += 4) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c = lane; c < C; c += 32) {
            float wv[8];
            bf16x8_to_float(__ldg(reinterpret_cast<const uint4*>(wrow) + c), wv);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (t0 + q < t_end) {
                    float xv[8];
                    bf16x8_to_float(
                        __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + q) * H) + c), xv);
                    // Fixed order within the chunk.
                    float a = acc[q];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a = fmaf(wv[i], xv[i], a);
                    acc[q] = a;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float s = warp_sum(acc[q]);
            if (lane == 0 && t0 + q < t_end) {
                if (r < E) logits[(size_t)(t0 + q) * E + r] = s;
                else sg_logit[t0 + q] = s;
            }
        }
    }
}

// One warp per token row; lane l holds experts l, l+32, ..., (VPL per lane).
// Selection ranks the fp32 score (softmax: the logit; sigmoid: sigmoid(l) +
// bias); equal scores go to the lower expert index; slots are written in
// descending score.  Weights: softmax p = exp(l - max) / sum over all experts,
// sigmoid p = sigmoid(l) (the bias only selects); renormalised over the k
// selected when norm != 0; then multiplied by `scale`.
template <int VPL>
__global__ void __launch_bounds__(256)
topk_kernel(const float* __restrict__ logits, int n, int E, int k, int routing,
            const float* __restrict__ bias, int norm, float scale,
            int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= n) return;
    const float* lrow = logits + (size_t)t * E;

    float lg[VPL], sc[VPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            lg[i] = lrow[e];
            if (routing == MOE_ROUTE_SOFTMAX) {
                sc[i] = lg[i];
            } else {
                const float s = 1.0f / (1.0f + expf(-lg[i]));
                sc[i] = s + bias[e];
            }
            // A NaN score ranks last (as -inf), so every slot still names a
            // valid expert and nothing downstream reads outside the weights.
            if (sc[i] != sc[i]) sc[i] = -INFINITY;
        } else {
            lg[i] = -INFINITY;
            sc[i] = -INFINITY;
            taken |= 1u << i;   // never selectable
        }
    }

    int sel_e = -1;          // lane j keeps slot j
    float sel_l = 0.f;
    for (int j = 0; j < k; ++j) {
        // Local best: strictly greater wins, so the lowest index keeps a tie.
        float bv = -INFINITY; int be = 0x7fffffff; float bl = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const bool free_i = !((taken >> i) & 1u);
            const int e = lane + 32 * i;
            if (free_i && (sc[i] > bv || (sc[i] == bv && e < be))) { bv = sc[i]; be = e; bl = lg[i]; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; bl = ol; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == j) { sel_e = be; sel_l = bl; }
    }

    float p = 0.f;
    if (routing == MOE_ROUTE_SOFTMAX) {
        // max logit = the first selected score.
        const float mx = __shfl_sync(0xffffffffu, sel_l, 0);
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (lane + 32 * i < E) z += expf(lg[i] - mx);
        z = warp_sum(z);
        p = (lane < k) ? expf(sel_l - mx) / z : 0.f;
    } else {
        p = (lane < k) ? 1.0f / (1.0f + expf(-sel_l)) : 0.f;
    }
    if (norm) {
        const float tot = warp_sum(p);
        p = p / tot;
    }
    if (lane < k) {
        idx_out[(size_t)t * k + lane] = sel_e;
        w_out[(size_t)t * k + lane] = p * scale;
    }
}

cudaError_t launch_router(const uint16_t* x, int n, int H, const uint16_t* wr, int E,
                          const uint16_t* gw, float* logits, float* sg_logit, int num_sms,
                          cudaStream_t st) {
    const int warps = 4;
    const int rows = E + (gw ? 1 : 0);
    dim3 grid((rows + warps - 1) / warps, 1);
    int gy = (2 * num_sms + (int)grid.x - 1) / (int)grid.x;
    gy = max(1, min(gy, (n + 3) / 4));
    int rpb = (n + gy - 1) / gy;
    rpb = (rpb + 3) / 4 * 4;
    gy = (n + rpb - 1) / rpb;
    grid.y = gy;
    router_kernel<<<grid, warps * 32, 0, st>>>(x, n, H, wr, E, gw, logits, sg_logit, rpb);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int n, int E, int k, int routing, const float* bias,
                        int norm, float scale, int32_t* idx, float* w, cudaStream_t st) {
    const int warps = 8;
    dim3 grid((n + warps - 1) / warps);
    const int vpl = (E + 31) / 32;
#define MOE_TOPK_CASE(V)                                                                   \
    if (vpl <= V) {                                                                        \
        topk_kernel<V><<<grid, warps * 32, 0, st>>>(logits, n, E, k, routing, bias, norm,  \
                                                    scale, idx, w);                        \
        return cudaGetLastError();                                                         \
    }
    MOE_TOPK_CASE(1) MOE_TOPK_CASE(2) MOE_TOPK_CASE(4) MOE_TOPK_CASE(8) MOE_TOPK_CASE(16)
    MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
    return cudaErrorInvalidValue;
}

}  // namespace moe
