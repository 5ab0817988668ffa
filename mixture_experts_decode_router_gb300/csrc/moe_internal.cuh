// moe_internal.cuh -- device helpers and host/device structures shared by the
// kernels of libmoe_gb300 (sm_103a).  Nothing here is part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kWarp = 32;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

// ----------------------------------------------------------------------------
// Workspace layout.  The control block sits at offset 0 for every n; the other
// regions follow, each 256-byte aligned, sized for the call's n.
// ----------------------------------------------------------------------------
struct Ctrl {
    int32_t n_active;      // experts with at least one route (written by the group kernel)
    int32_t n_rsegs;       // routed token segments of <= kTcTokensPerTile (group kernel)
    int32_t err;           // sticky device error code (bounded waits that gave up); 0 = none
    uint32_t gbar;         // grid-barrier arrivals of the single-token kernel (0 between calls)
    int32_t routed;        // tokens routed so far by the fused top-k + grouping kernel (0 between calls)
    uint32_t tc_count;     // grid-barrier arrivals of the grouped down kernel before its combine (0 between calls)
    uint32_t tc_gen;       // that barrier's generation (advanced by the last arrival)
    int32_t pad[57];
};

// Tokens per tile of the grouped tensor-core path (its MMA N is at most this).
constexpr int kTcTokensPerTile = 64;

// Tensor-core router (grouped path): K splits fixed by H alone -- at most
// kRouterTcMaxSplits splits of a multiple of 64 elements -- so that a token's
// partial logits do not depend on the batch; token tiles of at most
// kRouterTcMaxTile rows; partials [splits][n][E] fp32, used while they fit in
// kRouterTcMaxPartialBytes (larger calls take the CUDA-core router).
constexpr int kRouterTcMaxSplits = 16;
constexpr int kRouterTcMaxTile = 128;
constexpr int64_t kRouterTcMaxPartialBytes = 8ll << 20;

struct RouterTcSplit {
    int splits;   // K splits
    int kc;       // K elements per split (a multiple of 64)
};

inline RouterTcSplit router_tc_split(int H) {
    RouterTcSplit r;
    const int boxes = (H + 63) / 64;
    r.splits = boxes < kRouterTcMaxSplits ? (boxes > 0 ? boxes : 1) : kRouterTcMaxSplits;
    r.kc = 64 * ((boxes + r.splits - 1) / r.splits);
    r.splits = (H + r.kc - 1) / r.kc;
    if (r.splits < 1) r.splits = 1;
    return r;
}

// Token tile of a call with n tokens, and the kernel's shared memory for it.
inline int router_tc_tile(int64_t n) { return n >= kRouterTcMaxTile ? kRouterTcMaxTile : (int)((n + 15) / 16) * 16; }
inline size_t router_tc_smem(int H, int64_t n) {
    return (size_t)(router_tc_split(H).kc / 64) * (128 + router_tc_tile(n)) * 128 + 64 + 1024;
}

// Bytes reserved for the partials (monotone in n, so a workspace sized for
// max_tokens serves every smaller call).
inline size_t router_tc_partials_bytes(int64_t n, int64_t E, int H) {
    const int64_t b = (int64_t)router_tc_split(H).splits * n * E * (int64_t)sizeof(float);
    return (size_t)(b < kRouterTcMaxPartialBytes ? b : kRouterTcMaxPartialBytes);
}

// Whether a call of n tokens can take the tensor-core router.
inline bool router_tc_fits(int64_t n, int64_t E, int H) {
    const int64_t b = (int64_t)router_tc_split(H).splits * n * E * (int64_t)sizeof(float);
    return n >= 1 && E >= 1 && H % 8 == 0 && b <= kRouterTcMaxPartialBytes && router_tc_smem(H, n) <= 232448;
}

struct WsLayout {
    size_t ctrl, logits, sg_logit, idx, w, counts, offsets, perm, active, act, act_sh,
        inv, segs, xs, xh, as, ash, y, ysh, xe, xd, lgp, rq, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Upper bound of the routed segments (<= kTcTokensPerTile routes of one expert):
// sum_e ceil(c_e / T) <= (n*k)/T + min(E, n*k).
inline int64_t grouped_segs_bound(int64_t n, int64_t k, int64_t E) {
    const int64_t nk = n * k;
    return nk / kTcTokensPerTile + (nk < E ? nk : E) + 1;
}

inline WsLayout ws_layout(const moe_config_t& c, int64_t n) {
    WsLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const int64_t E = c.num_experts, k = c.top_k, H = c.hidden, I = c.inter, S = c.shared_inter;
    L.ctrl = take(sizeof(Ctrl));
    L.logits = take(sizeof(float) * n * E);
    L.sg_logit = take(sizeof(float) * n);
    L.idx = take(sizeof(int32_t) * n * k);
    L.w = take(sizeof(float) * n * k);
    L.counts = take(sizeof(int32_t) * E);
    L.offsets = take(sizeof(int32_t) * (E + 1));
    L.perm = take(sizeof(int32_t) * n * k);
    L.active = take(sizeof(int32_t) * E);
    L.act = take(sizeof(float) * n * k * I);
    L.act_sh = take(sizeof(float) * n * (S > 0 ? S : 1));
    // Grouped tensor-core path.
    L.inv = take(sizeof(int32_t) * n * k);                       // route -> sorted position
    L.segs = take(sizeof(int32_t) * 3 * grouped_segs_bound(n, k, E));
    L.xs = take(sizeof(uint16_t) * n * k * H);                   // expert-sorted activations
    L.xh = take(sizeof(uint16_t) * n * H);                       // copy of x for the shared expert (f16 / bf16)
    L.as = take(sizeof(uint16_t) * n * k * I);                   // SiLU(g)*u, sorted rows
    L.ash = take(sizeof(uint16_t) * n * (S > 0 ? S : 1));
    L.y = take(sizeof(float) * n * k * H);                       // weighted down rows
    L.ysh = take(sizeof(float) * n * H);
    L.xe = take(sizeof(uint16_t) * n * H);                       // pre-expert RMSNorm of x
    L.xd = take(sizeof(uint16_t) * n * H);                       // x staged from pinned host memory
    L.lgp = take(router_tc_partials_bytes(n, E, (int)H));        // tensor-core router partials
    L.rq = take(c.router_fmt == MOE_W_NVFP4 ? sizeof(uint16_t) * E * H : 0);   // an NVFP4 router as BF16
    L.total = off;
    return L;
}

// ----------------------------------------------------------------------------
// Device-side views of the weights.
// ----------------------------------------------------------------------------
struct QMatDev {
    const uint8_t* w;       // base of the stacked matrix (bytes)
    const void* scale;      // FP8: float blocks; NVFP4: E4M3 bytes
    const float* scale2;    // NVFP4 per-expert
    int out_dim, in_dim;
    int e_base;             // global index of the stack's first expert (expert parallelism)
};

// ----------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of a multi-kernel sequence is
// launched with programmatic stream serialisation, so its launch and prologue
// overlap the tail of the kernel before it.  Each kernel calls pdl_wait()
// before its first global-memory access (it returns once every earlier kernel
// on the stream has completed and its writes are visible), and pdl_trigger()
// once its own main work is done.  A dependent grid launches only after every
// CTA of this grid has signalled or exited, so every CTA has started by then;
// the small kernels of a grouped call with at most one token per SM signal
// right after pdl_wait(), so that the next kernel's launch and prologue
// overlap them (it still waits for their completion before reading).
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------
// Small device helpers.
// ----------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// 16-byte streaming load that does not allocate in L1 (each weight byte is used once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// Two FP8 E4M3 codes (low byte = first element) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(two_codes));
    __half2_raw raw;
    raw.x = (unsigned short)(h2 & 0xffffu);
    raw.y = (unsigned short)(h2 >> 16);
    return __half22float2(__half2(raw));
}

// Two E2M1 codes in one byte (low nibble = first element) -> two floats, exactly.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
    __half2_raw raw;
    raw.x = (unsigned short)(h2 & 0xffffu);
    raw.y = (unsigned short)(h2 >> 16);
    return __half22float2(__half2(raw));
}

// One E4M3 code -> float (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
    return e4m3x2_to_float2(code & 0xffu).x;
}

// ----------------------------------------------------------------------------
// Weight chunks: 8 consecutive elements of one row (along `in`), decoded to
// fp32, plus the multiplier that applies to the whole chunk.  Every format's
// chunk lies inside one scale block (FP8: 128 columns; NVFP4: 16 columns),
// because chunks start at multiples of 8.
// ----------------------------------------------------------------------------
template <int FMT> struct WChunk;

template <> struct WChunk<MOE_W_BF16> {
    uint4 raw;
    __device__ __forceinline__ void load(const QMatDev& m, int e, int row, int c) {
        const uint16_t* base = reinterpret_cast<const uint16_t*>(m.w) +
                               ((size_t)(e - m.e_base) * m.out_dim + row) * m.in_dim + (size_t)c * 8;
        raw = ld_stream_v4(base);
    }
    __device__ __forceinline__ float scale(const QMatDev&, int, int, int) const { return 1.0f; }
    __device__ __forceinline__ void decode(float (&v)[8]) const {
        v[0] = bf16_lo(raw.x); v[1] = bf16_hi(raw.x); v[2] = bf16_lo(raw.y); v[3] = bf16_hi(raw.y);
        v[4] = bf16_lo(raw.z); v[5] = bf16_hi(raw.z); v[6] = bf16_lo(raw.w); v[7] = bf16_hi(raw.w);
    }
};

template <> struct WChunk<MOE_W_FP8_B128> {
    uint2 raw;
    __device__ __forceinline__ void load(const QMatDev& m, int e, int row, int c) {
        const uint8_t* base = m.w + ((size_t)(e - m.e_base) * m.out_dim + row) * m.in_dim + (size_t)c * 8;
        raw = ld_stream_v2(base);
    }
    __device__ __forceinline__ float scale(const QMatDev& m, int e, int row, int c) const {
        const int ob = (m.out_dim + 127) >> 7, ib = (m.in_dim + 127) >> 7;
        const float* s = reinterpret_cast<const float*>(m.scale) + (size_t)(e - m.e_base) * ob * ib;
        return __ldg(s + (row >> 7) * ib + ((c * 8) >> 7));
    }
    __device__ __forceinline__ void decode(float (&v)[8]) const {
        float2 a = e4m3x2_to_float2(raw.x & 0xffffu), b = e4m3x2_to_float2(raw.x >> 16);
        float2 c2 = e4m3x2_to_float2(raw.y & 0xffffu), d = e4m3x2_to_float2(raw.y >> 16);
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c2.x; v[5] = c2.y; v[6] = d.x; v[7] = d.y;
    }
};

template <> struct WChunk<MOE_W_NVFP4> {
    uint32_t raw;
    __device__ __forceinline__ void load(const QMatDev& m, int e, int row, int c) {
        const uint8_t* base = m.w + ((size_t)(e - m.e_base) * m.out_dim + row) * (m.in_dim / 2) + (size_t)c * 4;
        raw = ld_stream_u32(base);
    }
    __device__ __forceinline__ float scale(const QMatDev& m, int e, int row, int c) const {
        const uint8_t* s = reinterpret_cast<const uint8_t*>(m.scale) +
                           ((size_t)(e - m.e_base) * m.out_dim + row) * (m.in_dim / 16);
        return e4m3_to_float(__ldg(s + (c >> 1)));
    }
    __device__ __forceinline__ void decode(float (&v)[8]) const {
        float2 a = e2m1x2_to_float2(raw & 0xffu), b = e2m1x2_to_float2((raw >> 8) & 0xffu);
        float2 c2 = e2m1x2_to_float2((raw >> 16) & 0xffu), d = e2m1x2_to_float2(raw >> 24);
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c2.x; v[5] = c2.y; v[6] = d.x; v[7] = d.y;
    }
};

// Per-matrix multiplier applied after the row's dot product (NVFP4 scale2).
template <int FMT>
__device__ __forceinline__ float matrix_scale(const QMatDev& m, int e) {
    if constexpr (FMT == MOE_W_NVFP4) return __ldg(m.scale2 + (e - m.e_base));
    else return 1.0f;
}

// 8 BF16 activations (16 bytes) -> floats.
__device__ __forceinline__ void bf16x8_to_float(uint4 r, float (&v)[8]) {
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
}

__device__ __forceinline__ float dot8(const float (&a)[8], const float (&b)[8]) {
    float s = a[0] * b[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) s = fmaf(a[i], b[i], s);
    return s;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Routing of one token by one thread block, in two calls: route_select_block
// (the top-k experts) and route_weights_block (their weights).
//
// Selection ranks the score s[e] (softmax: the logit; sigmoid: sigmoid(l) +
// bias, the bias only selects): the rank of e is the number of experts ahead
// of it in (score descending, index ascending) order, and ssel[j] is the
// expert of rank j < k.  Each expert carries that order as one 64-bit key
// (route_key: the score's bits made order-preserving above the complemented
// index), so "ahead" is one integer comparison.  The ranks are exact, in two
// levels: each group of 32 consecutive experts ranks its members and keeps
// its first k as candidates; then each candidate is ranked among all
// candidates (eight threads per candidate, their counts summed by shuffles).
// An expert of global rank < k is among its group's first k, and so is every
// expert ahead of it, so its rank among the candidates is its global rank;
// any other candidate has the k true top experts ahead of it.
//
// Weights: softmax p = exp(l - m) / z with m the largest logit and z the sum
// of exp(l - m) over all E experts, taken as a fixed butterfly within each
// group of 32 and then over the groups in order; sigmoid p = sigmoid(l).
// Renormalised over the k selected when norm != 0 (a fixed butterfly), then
// multiplied by `scale`: sselw[j] is the weight of ssel[j].
//
// The results depend on E, k and the logits only (not on the thread count),
// so every kernel that routes with these functions routes alike.  All nthr
// threads of the block call each function; `sync` is the block's barrier.
//   slg            logits [E] (shared memory)
//   skey           keys [E + 32] (shared memory, 16-byte aligned; entries E..E+31 zero)
//   cand_k         ceil(E/32) * k slots (shared memory, 16-byte aligned)
//   gmax, zg       ceil(E/32) floats each (shared memory)

// The selection key of expert e with score s (NaN already replaced by -inf):
// larger key = ahead.  -0 counts as +0, as equal scores must tie.
__device__ __forceinline__ unsigned long long route_key(float s, int e) {
    uint32_t b = __float_as_uint(s + 0.0f);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (uint32_t)~(uint32_t)e;
}

template <typename Sync>
__device__ __forceinline__ void route_select_block(const float* slg, const unsigned long long* skey, int E, int k,
                                                   int routing, int tid, int nthr, unsigned long long* cand_k,
                                                   float* gmax, int* ssel, Sync sync) {
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int ngroups = (E + 31) >> 5;
    // Level 1, and (softmax) each group's largest logit.  Every real key is
    // above zero, the padding's.
    for (int g = warp; g < ngroups; g += nwarps) {
        const int e = 32 * g + lane;
        const unsigned long long kv = skey[e];
        const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(skey + 32 * g);
        int rank = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const ulonglong2 u = k2[q];
            rank += (u.x > kv ? 1 : 0) + (u.y > kv ? 1 : 0);
        }
        const bool valid = e < E;
        if (valid && rank < k) cand_k[g * k + rank] = kv;
        const int nvalid = min(32, E - 32 * g);
        if (lane < k && lane >= nvalid) cand_k[g * k + lane] = 0ull;   // slots no member fills
        if (routing == MOE_ROUTE_SOFTMAX) {
            float m = valid ? slg[e] : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) gmax[g] = m;
        }
    }
    sync();
    // Level 2: 4 candidates per warp per pass, 8 lanes each.
    const int nc = ngroups * k;
    for (int q0 = warp * 4; q0 < nc; q0 += nwarps * 4) {
        const int c = q0 + (lane >> 3), part = lane & 7;
        const unsigned long long kv = c < nc ? cand_k[c] : 0ull;
        int cnt = 0;
        if (kv != 0ull) {
#pragma unroll 4
            for (int c2 = part; c2 < nc; c2 += 8) cnt += cand_k[c2] > kv ? 1 : 0;
        }
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 4);
        if (kv != 0ull && part == 0 && cnt < k) ssel[cnt] = (int)~(uint32_t)kv;
    }
    sync();
}

template <typename Sync>
__device__ __forceinline__ void route_weights_block(const float* slg, int E, int k, int routing, int norm,
                                                    float scale, int tid, int nthr, const float* gmax, float* zg,
                                                    const int* ssel, float* sselw, Sync sync) {
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int ngroups = (E + 31) >> 5;
    const bool softmax = routing == MOE_ROUTE_SOFTMAX;
    float mx = 0.f;
    if (softmax) {
        mx = lane < ngroups ? gmax[lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        for (int g = warp; g < ngroups; g += nwarps) {
            const int e = 32 * g + lane;
            float z = e < E ? expf(slg[e] - mx) : 0.f;
            z = warp_sum(z);
            if (lane == 0) zg[g] = z;
        }
        sync();
    }
    if (warp == 0) {
        const int sel_e = lane < k ? ssel[lane] : -1;
        const float sel_l = lane < k ? slg[sel_e] : 0.f;
        float p;
        if (softmax) {
            float z = 0.f;
            for (int g = 0; g < ngroups; ++g) z += zg[g];
            p = lane < k ? expf(sel_l - mx) / z : 0.f;
        } else {
            p = lane < k ? 1.0f / (1.0f + expf(-sel_l)) : 0.f;
        }
        if (norm) {
            const float tot = warp_sum(p);
            p = p / tot;
        }
        if (lane < k) sselw[lane] = p * scale;
    }
    sync();
}

// One token's routing by one thread block from its logit row: the selection
// keys (sigmoid routing: sigmoid(l) + bias selects; NaN scores rank last),
// then route_select_block and route_weights_block.  ssel / sselw receive the
// k experts and weights.  slg [E] and skey [E + 32] as above.
// lrow holds ns partial rows sstride floats apart (the tensor-core router's
// K splits; ns = 1 for the other routers): the logit is their sum in split
// order, written to lsum (when not null).
__device__ __forceinline__ void route_token_block(const float* __restrict__ lrow, int ns, size_t sstride,
                                                  float* __restrict__ lsum, int E, int k, int routing,
                                                  const float* __restrict__ bias, int norm, float scale,
                                                  float* slg, unsigned long long* skey,
                                                  unsigned long long* cand_k, float* gmax, float* zg, int* ssel,
                                                  float* sselw) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    for (int e = tid; e < E + 32; e += nthr) {
        if (e < E) {
            float l;
            if (ns == 1) {
                l = lrow[e];
            } else {   // all partials (ns <= kRouterTcMaxSplits) in flight, added in order
                float v[kRouterTcMaxSplits];
#pragma unroll
                for (int u = 0; u < kRouterTcMaxSplits; ++u) v[u] = u < ns ? lrow[(size_t)u * sstride + e] : 0.f;
                l = v[0];
#pragma unroll
                for (int u = 1; u < kRouterTcMaxSplits; ++u)
                    if (u < ns) l += v[u];
            }
            if (lsum) lsum[e] = l;
            float sc;
            if (routing == MOE_ROUTE_SOFTMAX) sc = l;
            else sc = 1.0f / (1.0f + expf(-l)) + bias[e];
            if (sc != sc) sc = -INFINITY;
            slg[e] = l;
            skey[e] = route_key(sc, e);
        } else {
            skey[e] = 0ull;
        }
    }
    __syncthreads();
    route_select_block(slg, skey, E, k, routing, tid, nthr, cand_k, gmax, ssel, [] { __syncthreads(); });
    route_weights_block(slg, E, k, routing, norm, scale, tid, nthr, gmax, zg, ssel, sselw,
                        [] { __syncthreads(); });
}

// The combine (the blend step), elements [i0, n*H/4) in steps of `step`
// float4s: out[t, h] = BF16(sum_j y[inv[t*k + j], h] in slot order, then
// + y_sh[t, h], then + out[t, h] when accumulating).  kL2: y and y_sh were
// written by other blocks of the same kernel, so they are read through L2,
// not the read-only path.
template <bool kL2>
__device__ __forceinline__ void combine_range(const float* __restrict__ y, const float* __restrict__ ysh,
                                              const int32_t* __restrict__ inv, int n, int H, int k,
                                              int has_shared, int accumulate, uint16_t* __restrict__ out,
                                              int64_t i0, int64_t step) {
    constexpr int kU = 8;
    auto ld4 = [](const float* p) -> float4 {
        if constexpr (kL2) return __ldcg(reinterpret_cast<const float4*>(p));
        else return __ldg(reinterpret_cast<const float4*>(p));
    };
    const int C4 = H >> 2;
    for (int64_t i = i0; i < (int64_t)n * C4; i += step) {
        const int t = (int)(i / C4), c = (int)(i - (int64_t)t * C4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < k; j0 += kU) {
            int pos[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) pos[u] = (j0 + u < k) ? __ldg(inv + t * k + j0 + u) : -1;
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (pos[u] >= 0) v[u] = ld4(y + (size_t)pos[u] * H + 4 * c);
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (pos[u] >= 0) { acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w; }
        }
        if (has_shared) {
            const float4 v = ld4(ysh + (size_t)t * H + 4 * c);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (accumulate) {
            const uint2 o = reinterpret_cast<const uint2*>(out + (size_t)t * H)[c];
            acc.x += __uint_as_float(o.x << 16); acc.y += __uint_as_float(o.x & 0xffff0000u);
            acc.z += __uint_as_float(o.y << 16); acc.w += __uint_as_float(o.y & 0xffff0000u);
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        reinterpret_cast<uint2*>(out + (size_t)t * H)[c] =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
}

// 1 / sqrt(mean(x^2) + eps) of one BF16 row of H elements, by one warp: lane l
// chains fmaf over its chunks l, l+32, ... in order, then a fixed butterfly.
// (Generic pointer: the row may be in global or shared memory.)
__device__ __forceinline__ float rms_inv_warp(const uint16_t* row, int H, float eps, int lane) {
    float ss = 0.f;
    for (int c = lane; c < (H >> 3); c += 32) {
        float v[8];
        bf16x8_to_float(reinterpret_cast<const uint4*>(row)[c], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
    ss = warp_sum(ss);
    return rsqrtf(ss / (float)H + eps);
}

// One 8-element chunk of the normalised row: BF16(x * inv * w), element-wise.
__device__ __forceinline__ uint4 rms_apply8(uint4 xr, uint4 wr, float inv) {
    float x[8], w[8];
    bf16x8_to_float(xr, x);
    bf16x8_to_float(wr, w);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn((x[2 * i] * inv) * w[2 * i], (x[2 * i + 1] * inv) * w[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moe
