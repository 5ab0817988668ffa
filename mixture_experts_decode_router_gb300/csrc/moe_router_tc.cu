// moe_router_tc.cu -- the router GEMM on the tensor cores (sm_103a), for the
// expert-grouped path: partial logits p[s, t, e] = sum over the K range of
// split s of x[t, k] * Wr[e, k], BF16 operands, fp32 accumulation in tensor
// memory.  The router step of the pages' grouped decode ("metrale_model_layers/
// layers/moe/forward_fp8_grouped_router.rs", grouped_route: the gate GEMM of
// all tokens against the [E, H] router matrix, fp32 logits).
//
// One CTA per (128-expert tile, K split, token tile of at most 128 rows): a
// thread of warp 0 copies the split's router rows and token rows by TMA
// (128-byte-swizzled 64-element boxes, out-of-range rows and columns read as
// zero), one elected lane of warp 1 issues the MMAs (M = 128 experts, N = the
// token tile, K = 16 per instruction, the split's K steps in order), and the
// four warps write their TMEM lane quarter of the accumulator to the partials.
// The K splits depend on H only, so a token's partials, and the fixed-order
// sum of them that the top-k kernels form, do not depend on which or how many
// tokens share the call.
#include <algorithm>
#include <mutex>

#include "moe_launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kRM = 128;        // experts per tile (MMA M)
constexpr int kRBox = 64;       // K elements per 128-byte box
constexpr int kRThreads = 128;  // four warps: TMEM lane quarters 0..3

struct RouterTcParams {
    int n, E, H;
    int kc;          // K elements per split (a multiple of 64)
    int nt;          // tokens per tile (a multiple of 16, <= kRouterTcMaxTile)
    int tmem_cols;   // accumulator columns allocated (a power of two >= 32, >= nt)
    float* part;     // [splits][n][E]
    int32_t* err;
    const float* scale;   // a multiplier of every partial (an NVFP4 router's scale2), or null
    int early;            // signal the dependent launch right after the wait (see pdl_trigger)
};

__global__ void __launch_bounds__(kRThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                 const RouterTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nsteps = p.kc / kRBox;
    uint8_t* sA = smem;                                  // nsteps x [128 rows x 128 B]
    uint8_t* sB = smem + (size_t)nsteps * kRM * 128;     // nsteps x [nt rows x 128 B]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)nsteps * p.nt * 128);   // loaded, mma done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kRM, s = blockIdx.y, t0 = blockIdx.z * p.nt, k0 = s * p.kc;

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bars[0], 1);
        ptx::mbar_init(&bars[1], 1);
        *s_abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(s_tmem, p.tmem_cols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    if (p.early) pdl_trigger();

    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(&bars[0], nsteps * (kRM + p.nt) * 128);
        for (int j = 0; j < nsteps; ++j) {
            ptx::tma_load_2d(sA + (size_t)j * kRM * 128, &wmap, k0 + j * kRBox, m0, &bars[0]);
            for (int b = 0; b < p.nt / 16; ++b)
                ptx::tma_load_2d(sB + (size_t)j * p.nt * 128 + b * 2048, &xmap, k0 + j * kRBox, t0 + 16 * b,
                                 &bars[0]);
        }
    }
    if (warp == 1) {
        if (ptx::mbar_wait_warp(&bars[0], 0, s_abort, p.err, 6)) {
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
                const uint32_t idesc = ptx::idesc_f16(kRM, p.nt, true);
                for (int j = 0; j < nsteps; ++j) {
                    const uint64_t a_desc = ptx::sw128_desc(ptx::smem_u32(sA + (size_t)j * kRM * 128));
                    const uint64_t b_desc = ptx::sw128_desc(ptx::smem_u32(sB + (size_t)j * p.nt * 128));
#pragma unroll
                    for (int kk = 0; kk < kRBox / 16; ++kk)   // K step kk: 32 bytes into the box
                        ptx::mma_f16(tmem, a_desc + (uint64_t)((kk * 32) >> 4), b_desc + (uint64_t)((kk * 32) >> 4),
                                     idesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
                ptx::mma_commit(&bars[1]);
            }
            __syncwarp();
        }
    }
    // Epilogue: warp q holds experts m0 + 32 q + lane (TMEM lanes of its quarter);
    // for each token the warp's 32 lanes write 32 consecutive experts.
    if (ptx::mbar_wait_warp(&bars[1], 0, s_abort, p.err, 7)) {
        ptx::tc_fence_after();
        const float sc = p.scale ? __ldg(p.scale) : 1.0f;
        const int e = m0 + 32 * warp + lane;
        const uint32_t tb = tmem + ((uint32_t)(32 * warp) << 16);
        float* dst = p.part + (size_t)s * p.n * p.E;
        for (int j0 = 0; j0 < p.nt; j0 += 16) {
            float d[16];
            ptx::tmem_ld16(tb + j0, d);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int t = t0 + j0 + jj;
                if (t < p.n && e < p.E) dst[(size_t)t * p.E + e] = p.scale ? d[jj] * sc : d[jj];
            }
        }
    }
    pdl_trigger();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, p.tmem_cols);
    }
}

// The NVFP4 router matrix [E, H] expanded to BF16 for the tensor-core router:
// each 16-element block's E2M1 codes times its E4M3 scale, a value of at most
// 6 significant bits and so exact in BF16; scale2 multiplies the partials.
// One 8-element chunk a thread.
__global__ void __launch_bounds__(256)
router_nvfp4_expand_kernel(const QMatDev wq, int E, int H, uint16_t* __restrict__ out, int early) {
    pdl_wait();
    if (early) pdl_trigger();
    const int C = H >> 3;
    const int64_t total = (int64_t)E * C;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / C), c = (int)(i - (int64_t)r * C);
        WChunk<MOE_W_NVFP4> ch;
        ch.load(wq, 0, r, c);
        float v[8];
        ch.decode(v);
        const float s = ch.scale(wq, 0, r, c);
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q] * s));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q + 1] * s));
            o[q] = lo | (hi << 16);
        }
        reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    pdl_trigger();
}

}  // namespace

cudaError_t launch_router_nvfp4_expand(const QMatDev& wq, int E, int H, uint16_t* out, bool early, int num_sms,
                                       cudaStream_t st) {
    const int64_t chunks = (int64_t)E * (H / 8);
    const int blocks = (int)std::min<int64_t>((chunks + 255) / 256, (int64_t)num_sms * 8);
    launch_pdl(router_nvfp4_expand_kernel, blocks, 256, 0, st, wq, E, H, out, early ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_router_tc(const uint16_t* x, int n, int H, const uint16_t* wr, int E, float* part,
                             int32_t* err, const float* scale, bool early, cudaStream_t st) {
    const RouterTcSplit sp = router_tc_split(H);
    const int nt = router_tc_tile(n);
    CUtensorMap wmap, xmap;
    // Router rows: boxes of 64 K x 128 rows; token rows: boxes of 64 K x 16 rows.
    if (!make_map(&wmap, wr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)H, (uint64_t)E, kRBox, kRM,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&xmap, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)H, (uint64_t)n, kRBox, 16,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    RouterTcParams p;
    p.n = n; p.E = E; p.H = H; p.kc = sp.kc; p.nt = nt;
    p.tmem_cols = nt <= 32 ? 32 : (nt <= 64 ? 64 : 128);
    p.part = part;
    p.err = err;
    p.scale = scale;
    p.early = early ? 1 : 0;
    const size_t smem = router_tc_smem(H, n);
    static std::mutex mu;
    static size_t configured[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            const cudaError_t e =
                cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            configured[dev] = smem;
        }
    }
    const dim3 grid((E + kRM - 1) / kRM, sp.splits, (n + nt - 1) / nt);
    launch_pdl(router_tc_kernel, grid, kRThreads, smem, st, wmap, xmap, p);
    return cudaGetLastError();
}

}  // namespace moe
