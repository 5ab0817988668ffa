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
// on the same pages): one CTA per token row.
#include <mutex>

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
    pdl_wait();
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
    pdl_trigger();
}

// Register-tiled router: each warp computes RE router rows x RT token rows.
// For every (token, expert) pair the arithmetic is the one above -- lane l
// chains fmaf over its chunks l, l+32, ... in order, then the same butterfly
// -- so tiling changes nothing but how often each chunk is loaded.
// XS: the block first copies its RT token rows into shared memory (every
// thread's loads issued together: one round of latency instead of one per
// chunk step); otherwise each warp reads them from L1/L2 as it goes.
template <int RE, int RT, bool XS>
__global__ void __launch_bounds__(256)
router_tiled_kernel(const uint16_t* __restrict__ x, int n, int H,
                    const uint16_t* __restrict__ wr, int E,
                    const uint16_t* __restrict__ gw,
                    float* __restrict__ logits, float* __restrict__ sg_logit) {
    extern __shared__ uint4 sxt[];   // XS: [RT][H / 8] chunks of the block's token rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = E + (gw ? 1 : 0);
    const int r0 = (blockIdx.x * (blockDim.x >> 5) + warp) * RE;
    if (!XS && r0 >= rows) return;
    pdl_wait();
    const int t0 = blockIdx.y * RT;
    const int C = H >> 3;
    if constexpr (XS) {
        // Eight chunks a thread loaded before any is stored: one round of load
        // latency for (up to) 8 x 256 chunks, not one per chunk.
        constexpr int kU = 8;
        for (int i0 = threadIdx.x; i0 < RT * C; i0 += kU * blockDim.x) {
            uint4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + u * blockDim.x;
                if (i < RT * C) {
                    const int b = i / C, c = i - b * C;
                    v[u] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)min(t0 + b, n - 1) * H) + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = i0 + u * blockDim.x;
                if (i < RT * C) sxt[i] = v[u];
            }
        }
        __syncthreads();
        if (r0 >= rows) {
            pdl_trigger();
            return;
        }
    }
    const uint16_t* wrow[RE];
#pragma unroll
    for (int a = 0; a < RE; ++a) {
        const int r = min(r0 + a, rows - 1);
        wrow[a] = (r < E) ? wr + (size_t)r * H : gw;
    }
    float acc[RE][RT];
#pragma unroll
    for (int a = 0; a < RE; ++a)
#pragma unroll
        for (int b = 0; b < RT; ++b) acc[a][b] = 0.f;
    // The router chunks of KB consecutive steps (lane, lane+32, ...) are all
    // requested before any is used, so a warp has RE*KB 16-byte loads of its
    // rows in flight; the token rows come from L1/L2.
    constexpr int KB = RE >= 4 ? 2 : 8 / RE;
    for (int c0 = lane; c0 < C; c0 += 32 * KB) {
        uint4 wv4[RE][KB];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
            const int c = c0 + 32 * q;
#pragma unroll
            for (int a = 0; a < RE; ++a)
                wv4[a][q] = c < C ? __ldg(reinterpret_cast<const uint4*>(wrow[a]) + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < KB; ++q) {
            const int c = c0 + 32 * q;
            if (c >= C) break;
            uint4 xv4[RT];
#pragma unroll
            for (int b = 0; b < RT; ++b)
                xv4[b] = XS ? sxt[b * C + c]
                            : __ldg(reinterpret_cast<const uint4*>(x + (size_t)min(t0 + b, n - 1) * H) + c);
#pragma unroll
            for (int b = 0; b < RT; ++b) {
                float xv[8];
                bf16x8_to_float(xv4[b], xv);
#pragma unroll
                for (int a = 0; a < RE; ++a) {
                    float wv[8];
                    bf16x8_to_float(wv4[a][q], wv);
                    float s = acc[a][b];
#pragma unroll
                    for (int i = 0; i < 8; ++i) s = fmaf(wv[i], xv[i], s);
                    acc[a][b] = s;
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < RE; ++a)
#pragma unroll
        for (int b = 0; b < RT; ++b) {
            const float v = warp_sum(acc[a][b]);
            const int r = r0 + a, t = t0 + b;
            if (lane == 0 && r < rows && t < n) {
                if (r < E) logits[(size_t)t * E + r] = v;
                else sg_logit[t] = v;
            }
        }
    pdl_trigger();
}

// NVFP4 router (the gate_nvfp4 / w4a16_gemm branch of the router step on the
// page "metrale_model_layers/layers/moe/forward.rs"): the router matrix
// [E, H] is stored as E2M1 codes with one E4M3 scale per 16 elements and one
// fp32 scale2, and multiplies BF16 activations.  One warp per router row and
// RT token rows per blockIdx.y; lane l takes the 8-element chunks l, l+32, ...
// in order, each chunk's dot product times its block scale chained with fmaf,
// then the butterfly, then scale2 -- the expert kernels' NVFP4 row arithmetic,
// identical for every n and grid.
template <int RT>
__global__ void __launch_bounds__(256)
router_nvfp4_kernel(const uint16_t* __restrict__ x, int n, int H, const QMatDev wq, int E,
                    float* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + warp;
    if (r >= E) return;
    pdl_wait();
    const int t0 = blockIdx.y * RT;
    const int C = H >> 3;
    float acc[RT];
#pragma unroll
    for (int b = 0; b < RT; ++b) acc[b] = 0.f;
#pragma unroll 2
    for (int c = lane; c < C; c += 32) {
        WChunk<MOE_W_NVFP4> ch;
        ch.load(wq, 0, r, c);
        const float cs = ch.scale(wq, 0, r, c);
        float wv[8];
        ch.decode(wv);
#pragma unroll
        for (int b = 0; b < RT; ++b) {
            float xv[8];
            bf16x8_to_float(__ldg(reinterpret_cast<const uint4*>(x + (size_t)min(t0 + b, n - 1) * H) + c), xv);
            acc[b] = fmaf(dot8(wv, xv), cs, acc[b]);
        }
    }
    const float s2 = matrix_scale<MOE_W_NVFP4>(wq, 0);
#pragma unroll
    for (int b = 0; b < RT; ++b) {
        const float v = warp_sum(acc[b]) * s2;
        if (lane == 0 && t0 + b < n) logits[(size_t)(t0 + b) * E + r] = v;
    }
    pdl_trigger();
}

cudaError_t launch_router_nvfp4(const uint16_t* x, int n, int H, const QMatDev& wq, int E, float* logits,
                                cudaStream_t st) {
    const int rt = n >= 8 ? 8 : (n >= 4 ? 4 : 1);
    const dim3 grid((E + 7) / 8, (n + rt - 1) / rt);
    if (rt == 8) launch_pdl(router_nvfp4_kernel<8>, grid, 256, 0, st, x, n, H, wq, E, logits);
    else if (rt == 4) launch_pdl(router_nvfp4_kernel<4>, grid, 256, 0, st, x, n, H, wq, E, logits);
    else launch_pdl(router_nvfp4_kernel<1>, grid, 256, 0, st, x, n, H, wq, E, logits);
    return cudaGetLastError();
}

// One CTA per token row: selection and weights by route_select_block and
// route_weights_block (exact ranks, fixed-order softmax normaliser), which the
// single-token kernel also uses.
__global__ void __launch_bounds__(256)
topk_block_kernel(const float* __restrict__ logits, int ns, float* __restrict__ lsum, int n, int E, int k,
                  int routing, const float* __restrict__ bias, int norm, float scale,
                  int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
    extern __shared__ float smf[];
    float* slg = smf;                                                    // [E]
    unsigned long long* skey =
        reinterpret_cast<unsigned long long*>(smf + ((E + 3) & ~3));     // [E + 32], 16-byte aligned
    __shared__ int ssel[kMaxTopK];
    __shared__ float sselw[kMaxTopK];
    __shared__ __align__(16) unsigned long long cand_k[kMaxExperts / 32 * kMaxTopK];
    __shared__ float gmax[kMaxExperts / 32], zg[kMaxExperts / 32];
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    route_token_block(logits + (size_t)t * E, ns, (size_t)n * E, lsum ? lsum + (size_t)t * E : nullptr, E, k,
                      routing, bias, norm, scale, slg, skey, cand_k, gmax, zg, ssel, sselw);
    if (tid < k) {
        idx_out[(size_t)t * k + tid] = ssel[tid];
        w_out[(size_t)t * k + tid] = sselw[tid];
    }
    pdl_trigger();
}

// The pre-expert RMSNorm ("pre_expert_norm" of MoeLayer::forward, page
// "metrale_model_layers/layers/moe/forward.rs": it normalises the experts'
// input, leaving the router's and the shared gate's input unchanged):
// xe = BF16(x / sqrt(mean(x^2) + eps) * w), one warp per token row.
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const uint16_t* __restrict__ x, int n, int H, const uint16_t* __restrict__ w, float eps,
               uint16_t* __restrict__ xe) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t < n) {
        const uint16_t* xr = x + (size_t)t * H;
        const float inv = rms_inv_warp(xr, H, eps, lane);
        for (int c = lane; c < (H >> 3); c += 32)
            reinterpret_cast<uint4*>(xe + (size_t)t * H)[c] =
                rms_apply8(reinterpret_cast<const uint4*>(xr)[c], __ldg(reinterpret_cast<const uint4*>(w) + c), inv);
    }
    pdl_trigger();
}

cudaError_t launch_rmsnorm(const uint16_t* x, int n, int H, const uint16_t* w, float eps, uint16_t* xe,
                           cudaStream_t st) {
    launch_pdl(rmsnorm_kernel, dim3((n + 7) / 8), dim3(256), 0, st, x, n, H, w, eps, xe);
    return cudaGetLastError();
}

cudaError_t launch_router(const uint16_t* x, int n, int H, const uint16_t* wr, int E,
                          const uint16_t* gw, float* logits, float* sg_logit, int num_sms,
                          cudaStream_t st) {
    const int rows = E + (gw ? 1 : 0);
    if (n <= 2) {
        // Few tokens: one router row per warp, all tokens in the warp's loop.
        const int warps = 4;
        dim3 grid((rows + warps - 1) / warps, 1);
        launch_pdl(router_kernel, grid, warps * 32, 0, st, x, n, H, wr, E, gw, logits, sg_logit, 4);
        return cudaGetLastError();
    }
    // RT tokens x RE router rows per warp, 8 warps per CTA; RE as large as keeps
    // at least one CTA per SM.  The token rows are staged in shared memory when
    // RT of them fit in kRouterXsMax bytes (8 tokens, else 4).
    constexpr size_t kRouterXsMax = 64 * 1024;
    int rt = n >= 8 ? 8 : 4;
    if (rt == 8 && (size_t)8 * H * 2 > kRouterXsMax) rt = 4;
    const size_t xs_bytes = (size_t)rt * H * 2;
    const bool xs = xs_bytes <= kRouterXsMax;
    const int gy = (n + rt - 1) / rt;
    int re = 4;
    while (re > 1 && (long)((rows + 8 * re - 1) / (8 * re)) * gy < num_sms) re >>= 1;
    dim3 grid((rows + 8 * re - 1) / (8 * re), gy);
    static std::mutex mu;
    static bool configured[128][6] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
#define MOE_ROUTER_CASE(RE_, RT_, SLOT_)                                                             \
    if (re == RE_ && rt == RT_) {                                                                    \
        if (xs) {                                                                                    \
            {                                                                                        \
                std::lock_guard<std::mutex> lock(mu);                                                \
                if (!configured[dev][SLOT_]) {                                                       \
                    const cudaError_t e = cudaFuncSetAttribute(router_tiled_kernel<RE_, RT_, true>,  \
                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRouterXsMax);             \
                    if (e != cudaSuccess) return e;                                                  \
                    configured[dev][SLOT_] = true;                                                   \
                }                                                                                    \
            }                                                                                        \
            launch_pdl(router_tiled_kernel<RE_, RT_, true>, grid, 256, xs_bytes, st, x, n, H, wr, E, gw, \
                       logits, sg_logit);                                                            \
        } else {                                                                                     \
            launch_pdl(router_tiled_kernel<RE_, RT_, false>, grid, 256, 0, st, x, n, H, wr, E, gw,  \
                       logits, sg_logit);                                                            \
        }                                                                                            \
        return cudaGetLastError();                                                                   \
    }
    MOE_ROUTER_CASE(4, 8, 0) MOE_ROUTER_CASE(2, 8, 1) MOE_ROUTER_CASE(1, 8, 2)
    MOE_ROUTER_CASE(4, 4, 3) MOE_ROUTER_CASE(2, 4, 4) MOE_ROUTER_CASE(1, 4, 5)
#undef MOE_ROUTER_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const float* logits, int ns, float* lsum, int n, int E, int k, int routing,
                        const float* bias, int norm, float scale, int32_t* idx, float* w, cudaStream_t st) {
    // Logits and keys: ~12 E + 272 bytes of shared memory (<= 13 KB for E <= 1024).
    const size_t smem = (size_t)((E + 3) & ~3) * sizeof(float) + (size_t)(E + 32) * sizeof(unsigned long long);
    launch_pdl(topk_block_kernel, n, 256, smem, st, logits, ns, lsum, n, E, k, routing, bias, norm, scale, idx, w);
    return cudaGetLastError();
}

}  // namespace moe
