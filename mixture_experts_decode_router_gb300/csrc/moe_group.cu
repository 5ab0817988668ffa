// moe_group.cu -- group the routes of a call by expert (sm_103a).
//
// The pages' grouped decode ("metrale_model_layers/layers/moe/forward.rs",
// forward_nvfp4_grouped_decode; "metrale_model_layers/layers/moe/
// forward_fp8_grouped_router.rs", module header) runs the experts sorted by
// expert, so that every expert's weights are streamed once for all the tokens
// that chose it.  This kernel builds that order on the device (no host
// read-back, so the call can be captured in a CUDA graph):
//   counts[e]   routes of expert e
//   offsets[e]  exclusive prefix sum of counts (offsets[E] = routes kept)
//   perm[p]     route ids r = t*k + j, grouped by expert, ascending r within an
//               expert (a stable order, independent of thread timing); a route
//               whose expert lies outside [e_begin, e_end) -- not held by this
//               call, or not an expert at all -- is dropped
//   inv[r]      sorted position of route r (-1 for a dropped route)
//   active[u]   experts with counts > 0, ascending; ctrl->n_active of them
//   segs[s]     (expert, first sorted position, routes) for runs of at most
//               kTcTokensPerTile routes of one expert, ascending expert;
//               ctrl->n_rsegs of them (the tiles of the grouped path)
#include <algorithm>
#include <mutex>

#include "moe_launch.cuh"

namespace moe {

constexpr int kGroupThreads = 1024;
constexpr int kIdxBatch = 8;   // rounds of 32 routes a segment warp loads before using them

// Warps that own contiguous route segments: 8, or one per 64 routes (two
// rounds of 32 each) above 512 routes, at most as many as keep the per-warp
// counts, (warps + 1) * E ints, within 36 KB -- 32 for E <= 256, 16 for
// E <= 512, 8 for E <= 1024.  (Measured on GB300: 2048 routes group faster
// with 32 warps; 128 routes slower with 2 or 32 than with 8.)
inline int seg_warps(int E, int nk) {
    const int cap = E <= 256 ? 32 : (E <= 512 ? 16 : 8);
    return std::min(cap, std::max(8, nk / 64));
}

// From tot[e] = routes of expert e (e < E <= blockDim.x): counts, offsets,
// active, segs and the control block's totals; tot[e] becomes the first sorted
// position of expert e.  Called by every thread of the block; ends with a
// barrier.
__device__ __forceinline__ void group_scan_experts(int32_t* tot, int E, int32_t* __restrict__ counts,
                                                   int32_t* __restrict__ offsets, int32_t* __restrict__ active,
                                                   int32_t* __restrict__ segs, Ctrl* __restrict__ ctrl) {
    __shared__ int32_t warp_sums[3][32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Exclusive scans over experts (one element per thread):
    // offsets (of counts), active positions (of counts > 0) and segment starts
    // (of ceil(counts / kTcTokensPerTile)).
    const int c = (tid < E) ? tot[tid] : 0;
    const int a = (tid < E && c > 0) ? 1 : 0;
    const int g = (c + kTcTokensPerTile - 1) / kTcTokensPerTile;
    int sc = c, sa = a, sg = g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xffffffffu, sc, o);
        const int ya = __shfl_up_sync(0xffffffffu, sa, o);
        const int yg = __shfl_up_sync(0xffffffffu, sg, o);
        if (lane >= o) { sc += yc; sa += ya; sg += yg; }
    }
    if (lane == 31) { warp_sums[0][warp] = sc; warp_sums[1][warp] = sa; warp_sums[2][warp] = sg; }
    __syncthreads();
    if (warp == 0) {
        int vc = warp_sums[0][lane], va = warp_sums[1][lane], vg = warp_sums[2][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yc = __shfl_up_sync(0xffffffffu, vc, o);
            const int ya = __shfl_up_sync(0xffffffffu, va, o);
            const int yg = __shfl_up_sync(0xffffffffu, vg, o);
            if (lane >= o) { vc += yc; va += ya; vg += yg; }
        }
        warp_sums[0][lane] = vc;   // inclusive over warps
        warp_sums[1][lane] = va;
        warp_sums[2][lane] = vg;
    }
    __syncthreads();
    const int base_c = (warp > 0 ? warp_sums[0][warp - 1] : 0);
    const int base_a = (warp > 0 ? warp_sums[1][warp - 1] : 0);
    const int base_g = (warp > 0 ? warp_sums[2][warp - 1] : 0);
    const int excl_c = base_c + sc - c;
    const int excl_a = base_a + sa - a;
    const int excl_g = base_g + sg - g;
    if (tid < E) {
        counts[tid] = c;
        offsets[tid] = excl_c;
        tot[tid] = excl_c;                 // reuse: start of expert tid
        if (a) active[excl_a] = tid;
        for (int b = 0; b < g; ++b) {
            int32_t* sgp = segs + 3 * (excl_g + b);
            sgp[0] = tid;
            sgp[1] = excl_c + b * kTcTokensPerTile;
            sgp[2] = min(kTcTokensPerTile, c - b * kTcTokensPerTile);
        }
    }
    if (tid == 0) {
        offsets[E] = warp_sums[0][31];     // routes kept (n*k minus dropped ones)
        ctrl->n_active = warp_sums[1][31];
        ctrl->n_rsegs = warp_sums[2][31];
    }
    __syncthreads();
}

// The grouping of all n*k routes by one block of kGroupThreads threads, sw of
// whose warps own route segments.  sm: (sw + 1) * E ints of shared memory.
__device__ __forceinline__ void group_block(const int32_t* __restrict__ idx, int nk, int E, int e_begin, int e_end,
                                            int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                            int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                            int32_t* __restrict__ active, int32_t* __restrict__ segs,
                                            Ctrl* __restrict__ ctrl, int32_t* sm, int sw) {
    int32_t* cnt = sm;                           // [sw][E]
    int32_t* tot = sm + sw * E;                  // [E]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < sw * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();

    const int seg = (nk + sw - 1) / sw;
    if (warp < sw) {
        const int b = warp * seg, e_ = min(nk, b + seg);
        for (int r0 = b; r0 < e_; r0 += 32 * kIdxBatch) {
            int ev[kIdxBatch];   // L2 (__ldcg): the fused kernel's other blocks wrote idx
#pragma unroll
            for (int u = 0; u < kIdxBatch; ++u) {
                const int r = r0 + 32 * u + lane;
                ev[u] = r < e_ ? __ldcg(idx + r) : -1;
            }
#pragma unroll
            for (int u = 0; u < kIdxBatch; ++u)
                if (r0 + 32 * u + lane < e_ && ev[u] >= e_begin && ev[u] < e_end)
                    atomicAdd(&cnt[warp * E + ev[u]], 1);   // not held here: dropped
        }
    }
    __syncthreads();

    // Per expert: exclusive scan over the segment warps, and the total.
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < sw; ++w) {
            const int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        tot[e] = run;
    }
    __syncthreads();

    group_scan_experts(tot, E, counts, offsets, active, segs, ctrl);

    // Stable scatter: each segment warp walks its routes in order (loaded
    // kIdxBatch rounds of 32 at a time).
    if (warp < sw) {
        const int b = warp * seg, e_ = min(nk, b + seg);
        for (int r1 = b; r1 < e_; r1 += 32 * kIdxBatch) {
            int ev[kIdxBatch];
#pragma unroll
            for (int u = 0; u < kIdxBatch; ++u) {
                const int r = r1 + 32 * u + lane;
                ev[u] = r < e_ ? __ldcg(idx + r) : -1;
            }
#pragma unroll
            for (int u = 0; u < kIdxBatch; ++u) {
                const int r0 = r1 + 32 * u;
                if (r0 >= e_) break;   // warp-uniform
                const int r = r0 + lane;
                const bool valid = r < e_;
                const int e = ev[u];
                const bool in_range = valid && e >= e_begin && e < e_end;
                if (valid && !in_range) inv[r] = -1;
                const unsigned vmask = __ballot_sync(0xffffffffu, in_range);
                if (in_range) {
                    const unsigned peers = __match_any_sync(vmask, e);
                    const int rank = __popc(peers & ((1u << lane) - 1u));
                    const int pos = tot[e] + cnt[warp * E + e] + rank;
                    perm[pos] = r;
                    inv[r] = pos;
                    __syncwarp(vmask);
                    if (rank == 0) cnt[warp * E + e] += __popc(peers);
                }
                __syncwarp();
            }
        }
    }
}

// The grouping of the routes of n tokens with k distinct experts each (the
// top-k kernel's routes), by one block.  Within one expert the routes then
// come from distinct tokens, so the stable position of route r = t*k + j of
// expert e among e's routes is the number of earlier tokens that chose e:
// bits[e][w] holds bit t & 31 of word w = t >> 5 for each token t that chose
// e, and pre[e][w] the tokens of e's words before w.  No per-warp counts and
// no match over a warp's routes; the same outputs as group_block.
// sm: 2 * E * W + E ints, W = ceil(n / 32); n * k <= kBitsRoutes.
constexpr int kBitsRoutes = 8 * kGroupThreads;   // routes a thread holds in registers: 8
constexpr int kBitsWords = 8192;                 // E * W words of bitmap at most (32 KB)

__device__ __forceinline__ void group_block_bits(const int32_t* __restrict__ idx, int n, int k, int E, int e_begin,
                                                 int e_end, int32_t* __restrict__ counts,
                                                 int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                 int32_t* __restrict__ inv, int32_t* __restrict__ active,
                                                 int32_t* __restrict__ segs, Ctrl* __restrict__ ctrl, int32_t* sm) {
    const int W = (n + 31) >> 5, nk = n * k, tid = threadIdx.x, nt = blockDim.x;
    uint32_t* bits = reinterpret_cast<uint32_t*>(sm);   // [E][W]
    int32_t* pre = sm + E * W;                           // [E][W]
    int32_t* tot = pre + E * W;                          // [E]
    // This thread's routes r = tid + nt * u, loaded together (L2: other blocks
    // of the kernel wrote idx), then the bitmap.
    int ev[kBitsRoutes / kGroupThreads];
#pragma unroll
    for (int u = 0; u < kBitsRoutes / kGroupThreads; ++u) {
        const int r = tid + nt * u;
        ev[u] = r < nk ? __ldcg(idx + r) : -1;
    }
    for (int i = tid; i < E * W; i += nt) bits[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kBitsRoutes / kGroupThreads; ++u) {
        const int r = tid + nt * u;
        if (r < nk && ev[u] >= e_begin && ev[u] < e_end) {   // not held here: dropped
            const int t = r / k;
            atomicOr(&bits[ev[u] * W + (t >> 5)], 1u << (t & 31));
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            pre[e * W + w] = run;
            run += __popc(bits[e * W + w]);
        }
        tot[e] = run;
    }
    __syncthreads();
    group_scan_experts(tot, E, counts, offsets, active, segs, ctrl);
#pragma unroll
    for (int u = 0; u < kBitsRoutes / kGroupThreads; ++u) {
        const int r = tid + nt * u;
        if (r >= nk) break;
        const int e = ev[u];
        if (e >= e_begin && e < e_end) {
            const int t = r / k, w = t >> 5;
            const int pos = tot[e] + pre[e * W + w] + __popc(bits[e * W + w] & ((1u << (t & 31)) - 1u));
            perm[pos] = r;
            inv[r] = pos;
        } else {
            inv[r] = -1;
        }
    }
}

inline bool group_bits_fits(int n, int k, int E) {
    return n * k <= kBitsRoutes && (size_t)E * ((n + 31) / 32) <= (size_t)kBitsWords;
}

__global__ void __launch_bounds__(kGroupThreads)
group_kernel(const int32_t* __restrict__ idx, int nk, int E, int e_begin, int e_end,
             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
             int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ active,
             int32_t* __restrict__ segs, Ctrl* __restrict__ ctrl, int sw) {
    extern __shared__ int32_t sm[];
    pdl_wait();
    group_block(idx, nk, E, e_begin, e_end, counts, offsets, perm, inv, active, segs, ctrl, sm, sw);
    pdl_trigger();
}

// Top-k routing of every token (one CTA per token, the top-k kernel's
// arithmetic) and then, in the CTA that finishes last, the grouping of all
// routes (group_block_bits when its bitmap fits, else group_block): one
// launch instead of two.  The last CTA is found with a counter in
// the control block (release fence before the increment, acquire fence after
// it), which that CTA returns to zero.  kMinBlocks = 2 (at most 32 registers
// a thread) when there are more tokens than SMs, so that up to two SMs' worth
// route in one wave; 1 otherwise (no register cap).
template <int kMinBlocks>
__global__ void __launch_bounds__(kGroupThreads, kMinBlocks)
topk_group_kernel(const float* __restrict__ logits, int ns, int n, int E, int k, int routing,
                  const float* __restrict__ bias, int norm, float scale, int32_t* idx_out,
                  float* __restrict__ w_out, int e_begin, int e_end, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                  int32_t* __restrict__ active, int32_t* __restrict__ segs, Ctrl* __restrict__ ctrl, int sw,
                  int bits, const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw,
                  float* __restrict__ sg_logit, int H, int sgx_off, int early) {
    extern __shared__ __align__(16) float smf[];
    float* slg = smf;                                                    // [E]
    unsigned long long* skey =
        reinterpret_cast<unsigned long long*>(smf + ((E + 3) & ~3));     // [E + 32]
    int32_t* gsm = reinterpret_cast<int32_t*>(skey + E + 32);           // grouping scratch
    __shared__ int ssel[kMaxTopK];
    __shared__ float sselw[kMaxTopK];
    __shared__ __align__(16) unsigned long long cand_k[kMaxExperts / 32 * kMaxTopK];
    __shared__ float gmax[kMaxExperts / 32], zg[kMaxExperts / 32];
    __shared__ int s_last;
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    if (early) pdl_trigger();
    // The shared gate's logit of token t, when the layer has one and the router
    // ran on the tensor cores (which leaves that row to this kernel): the
    // threads past the key phase's E + 32 entries (at least the last warp)
    // stage x[t] and the gate row in shared memory while the routing loads its
    // logits; warp 0 forms the dot product after the routing, with the
    // CUDA-core router's arithmetic for a row (lane l chains its chunks l,
    // l + 32, ... in order, then the butterfly), so its bits are that kernel's.
    const int C = H >> 3;
    uint4* sgx = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(smf) + sgx_off);   // [x[t] | gw], C each
    if (gw) {
        const int s0 = min(E + 32, (int)blockDim.x - 32), nst = (int)blockDim.x - s0;
        if (tid >= s0) {
            constexpr int kU = 4;
            for (int i0 = tid - s0; i0 < 2 * C; i0 += kU * nst) {
                uint4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = i0 + u * nst;
                    if (i < 2 * C)
                        v[u] = __ldg(i < C ? reinterpret_cast<const uint4*>(x + (size_t)t * H) + i
                                           : reinterpret_cast<const uint4*>(gw) + (i - C));
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int i = i0 + u * nst;
                    if (i < 2 * C) sgx[i] = v[u];
                }
            }
        }
    }
    route_token_block(logits + (size_t)t * E, ns, (size_t)n * E, nullptr, E, k, routing, bias, norm, scale, slg, skey,
                      cand_k, gmax, zg, ssel, sselw);   // (its barriers order the staging before the use below)
    if (gw && tid < 32) {
        float acc = 0.f;
        for (int c = tid; c < C; c += 32) {
            float wv[8], xv[8];
            bf16x8_to_float(sgx[C + c], wv);
            bf16x8_to_float(sgx[c], xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(wv[i], xv[i], acc);
        }
        const float v = warp_sum(acc);
        if (tid == 0) sg_logit[t] = v;
    }
    if (tid < k) {
        idx_out[(size_t)t * k + tid] = ssel[tid];
        w_out[(size_t)t * k + tid] = sselw[tid];
    }
    // Release: the barrier orders the block's writes before thread 0's fence,
    // which is cumulative over them, then the count.  The block that counts
    // last takes an acquire fence before it reads every block's routes.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const int done = atomicAdd(&ctrl->routed, 1);
        s_last = done == n - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (s_last) {
        if (bits)
            group_block_bits(idx_out, n, k, E, e_begin, e_end, counts, offsets, perm, inv, active, segs, ctrl, gsm);
        else
            group_block(idx_out, n * k, E, e_begin, e_end, counts, offsets, perm, inv, active, segs, ctrl, gsm, sw);
        if (tid == 0) ctrl->routed = 0;
    }
    pdl_trigger();
}

cudaError_t launch_group(const int32_t* idx, int nk, int E, int e_begin, int e_end, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active, int32_t* segs,
                         Ctrl* ctrl, cudaStream_t st) {
    const int sw = seg_warps(E, nk);
    const size_t smem = sizeof(int32_t) * (size_t)(sw + 1) * E;
    // (sw + 1) * E ints <= 36 KB for E <= 1024: under the 48 KB default.
    launch_pdl(group_kernel, 1, kGroupThreads, smem, st, idx, nk, E, e_begin, e_end, counts, offsets, perm, inv,
               active, segs, ctrl, sw);
    return cudaGetLastError();
}

bool topk_group_gate_fits(int E, int H) {
    // The stagers (threads past E + 32, at least one warp) hold both rows' chunks
    // at kU = 4 loads each.
    const int nst = kGroupThreads - std::min(E + 32, kGroupThreads - 32);
    return H % 8 == 0 && 2 * (H / 8) <= 4 * nst;
}

cudaError_t launch_topk_group(const float* logits, int ns, int n, int E, int k, int routing, const float* bias, int norm,
                              float scale, int32_t* idx, float* w, int e_begin, int e_end, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active, int32_t* segs,
                              Ctrl* ctrl, const uint16_t* x, const uint16_t* gw, float* sg_logit, int H, bool early,
                              int num_sms, cudaStream_t st) {
    const int sw = seg_warps(E, n * k);
    // The routes of one top-k call have distinct experts per token: the bitmap
    // grouping when its bitmap fits.
    const bool bits = group_bits_fits(n, k, E);
    const size_t gwords = bits ? (size_t)(2 * ((n + 31) / 32) + 1) * E : (size_t)(sw + 1) * E;
    size_t smem = (size_t)((E + 3) & ~3) * sizeof(float) + (size_t)(E + 32) * sizeof(unsigned long long) +
                  sizeof(int32_t) * gwords;
    smem = (smem + 15) / 16 * 16;
    const int sgx_off = (int)smem;
    if (gw) smem += (size_t)2 * H * sizeof(uint16_t);   // x[t] and the gate row
    static std::mutex mu;
    static size_t configured[128][2] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    const bool two = n > num_sms;
    auto kern = two ? topk_group_kernel<2> : topk_group_kernel<1>;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev][two] < smem) {
            const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            configured[dev][two] = smem;
        }
    }
    launch_pdl(kern, n, kGroupThreads, smem, st, logits, ns, n, E, k, routing, bias, norm, scale, idx, w,
               e_begin, e_end, counts, offsets, perm, inv, active, segs, ctrl, sw, bits ? 1 : 0, x, gw, sg_logit, H,
               sgx_off, early ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace moe
