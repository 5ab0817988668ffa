// moe_gather.cu -- the grouped path's small memory-bound kernels around the
// tensor-core GEMMs (sm_103a): gathering the token rows into expert order
// before them, and combining the weighted expert rows after them.
#include <algorithm>

#include "moe_launch.cuh"

namespace moe {

namespace {

// xs[p, :] = x[perm[p] / k, :] for the grouped routes, and xh = x (the shared
// expert's operand); 16-bit values as the tiles take them (F16: f16 for the FP8
// and NVFP4 tiles, else bf16).  The tensor-core kernels' TMA copies therefore
// read only workspace buffers: x itself is read here with plain loads, so it
// may also live in pinned host memory.
template <bool F16>
__device__ __forceinline__ uint4 to_tile16(uint4 v) {
    if constexpr (F16) {
        uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xffff0000u);
            const __half2 h = __floats2half2_rn(fminf(fmaxf(lo, -65504.f), 65504.f),
                                                fminf(fmaxf(hi, -65504.f), 65504.f));
            w4[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    return v;
}

// One warp per destination row (the row's source index read once), its lanes
// taking 16-byte chunks lane, lane + 32, ...: kU chunks per lane loaded before
// any is stored, so a row costs one round of load latency, not one per chunk.
// With a pre-expert RMSNorm weight nw, the rows copied are the normalised ones,
// with the norm kernel's arithmetic (rms_inv_warp, then rms_apply8): a first
// pass over the row sums its squares in the same chunk order (lane l's chunks
// l, l + 32, ... in order, then the butterfly), so the values are that
// kernel's, bit for bit.  (NORM: whether nw is given -- its own instance, so
// that the plain copy keeps its small register count.)
template <bool F16, bool NORM>
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int n, int H, int k,
                                                     const int32_t* __restrict__ perm,
                                                     const int32_t* __restrict__ offsets, int E,
                                                     uint16_t* __restrict__ xs, uint16_t* __restrict__ xh,
                                                     const uint16_t* __restrict__ nw, float eps, int early) {
    constexpr int kU = 8;
    pdl_wait();
    if (early) pdl_trigger();
    const int n_routes = offsets[E];
    const int rows = n_routes + n;
    const int C8 = H >> 3;
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const bool routed = r < n_routes;
        const int t = routed ? perm[r] / k : r - n_routes;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
        uint4* dst = reinterpret_cast<uint4*>(routed ? xs + (size_t)r * H : xh + (size_t)(r - n_routes) * H);
        if (NORM && C8 <= 32 * kU) {
            // The whole row in one round: the lane's chunks and their norm
            // weights loaded together, then the sum of squares, then the stores.
            uint4 v[kU], wv[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = lane + 32 * u;
                if (c < C8) {
                    v[u] = __ldg(src + c);
                    wv[u] = __ldg(reinterpret_cast<const uint4*>(nw) + c);
                }
            }
            float ss = 0.f;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (lane + 32 * u < C8) {
                    float f[8];
                    bf16x8_to_float(v[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
                }
            }
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss / (float)H + eps);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = lane + 32 * u;
                if (c < C8) dst[c] = to_tile16<F16>(rms_apply8(v[u], wv[u], inv));
            }
            continue;
        }
        float inv = 0.f;
        if (NORM) {   // a longer row: its sum of squares first, then the copy below
            float ss = 0.f;
            for (int c0 = lane; c0 < C8; c0 += 32 * kU) {
                uint4 v[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < C8) v[u] = __ldg(src + c);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (c0 + 32 * u < C8) {
                        float f[8];
                        bf16x8_to_float(v[u], f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
                    }
                }
            }
            ss = warp_sum(ss);
            inv = rsqrtf(ss / (float)H + eps);
        }
        for (int c0 = lane; c0 < C8; c0 += 32 * kU) {
            uint4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = c0 + 32 * u;
                if (c < C8) {
                    v[u] = __ldg(src + c);
                    if (NORM) v[u] = rms_apply8(v[u], __ldg(reinterpret_cast<const uint4*>(nw) + c), inv);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = c0 + 32 * u;
                if (c < C8) dst[c] = to_tile16<F16>(v[u]);
            }
        }
    }
    pdl_trigger();
}

// out[t, h] = bf16( sum_j y[inv[t*k + j], h] (slot order) + y_sh[t, h] ), for
// calls whose down kernel does not run the combine itself.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const float* __restrict__ ysh,
                                                      const int32_t* __restrict__ inv, int n, int H, int k,
                                                      int has_shared, int accumulate, uint16_t* __restrict__ out,
                                                      int early) {
    pdl_wait();
    if (early) pdl_trigger();
    combine_range<false>(y, ysh, inv, n, H, k, has_shared, accumulate, out,
                         blockIdx.x * (int64_t)blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
    pdl_trigger();
}

// dst = src, n16 16-byte words (x staged from pinned host memory).
__global__ void __launch_bounds__(256) copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                     size_t n16) {
    pdl_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
    pdl_trigger();
}

}  // namespace

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st) {
    const size_t n16 = bytes / 16;
    const int grid = (int)std::min<size_t>((size_t)num_sms, (n16 + 255) / 256);
    launch_pdl(copy16_kernel, grid > 0 ? grid : 1, 256, 0, st, static_cast<const uint4*>(src),
               static_cast<uint4*>(dst), n16);
    return cudaGetLastError();
}

cudaError_t launch_gather(int fmt, const uint16_t* x, int n, int H, int k, const int32_t* perm,
                          const int32_t* offsets, int E, uint16_t* xs, uint16_t* xh, const uint16_t* norm_w,
                          float eps, bool early, int num_sms, cudaStream_t st) {
    const int grid = 2 * num_sms;
    auto kern = fmt != MOE_W_BF16 ? (norm_w ? gather_kernel<true, true> : gather_kernel<true, false>)
                                  : (norm_w ? gather_kernel<false, true> : gather_kernel<false, false>);
    launch_pdl(kern, grid, 256, 0, st, x, n, H, k, perm, offsets, E, xs, xh, norm_w, eps, early ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* y, const float* ysh, const int32_t* inv, int n, int H, int k,
                           int has_shared, int accumulate, uint16_t* out, bool early, int num_sms, cudaStream_t st) {
    launch_pdl(combine_kernel, 2 * num_sms, 256, 0, st, y, ysh, inv, n, H, k, has_shared, accumulate, out,
               early ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace moe
