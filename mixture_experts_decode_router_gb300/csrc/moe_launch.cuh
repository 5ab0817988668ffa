// moe_launch.cuh -- kernel parameter blocks and launch entry points used by
// the C ABI layer (moe_capi.cu).  Internal to libmoe_gb300.
#pragma once

#include <cuda.h>

#include "moe_internal.cuh"

namespace moe {

struct GateUpParams {
    const uint16_t* x;
    int n, H, I, S, k;
    QMatDev gate, up, sh_gate, sh_up;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* active;
    const Ctrl* ctrl;
    float* act;      // [n*k, I], row = route id t*k + j
    float* act_sh;   // [n, S]
};

struct DownParams {
    int n, H, I, S, k, E;
    int e_begin, e_end;      // routes to experts outside [e_begin, e_end) contribute nothing
    int accumulate;          // out = BF16(out + result)
    QMatDev down, sh_down;
    const int32_t* idx;
    const float* w;
    const float* act;
    const float* act_sh;
    const float* sg_logit;   // NULL = shared gate 1
    uint16_t* out;
};

// Grouped tensor-core path (moe_grouped_tc.cu).
struct TcMaps {
    CUtensorMap w[2];    // routed weights: (gate, up) or (down)
    CUtensorMap ws[2];   // shared-expert weights
    CUtensorMap b;       // routed activations (expert-sorted rows)
    CUtensorMap bs;      // shared-expert activations (token rows)
};

struct TcParams {
    int out_dim, in_dim;     // routed matrix [out, in] per expert
    int sh_out, sh_in;       // shared matrix (sh_out == 0: no shared expert)
    int n, k;
    int e_base;              // global index of the weight stacks' first expert
    const int32_t* segs;     // [n_rsegs][3] = (expert, first sorted row, tokens)
    const Ctrl* ctrl;
    const void* scale[2];    // routed scales (FP8 fp32 blocks / NVFP4 E4M3 bytes)
    const void* sh_scale[2];
    const float* scale2[2];  // NVFP4 per-expert fp32
    const float* sh_scale2[2];
    void* act_out;           // gate_up: sorted SiLU(g)*u rows [n*k, I] (bf16 / f16)
    void* act_sh_out;        // gate_up: shared [n, S]
    float* y;                // down: weighted rows [n*k, H]
    float* y_sh;             // down: gated shared rows [n, H]
    const float* route_w;    // [n*k] routing weights (by route id)
    const int32_t* perm;     // sorted position -> route id
    const float* sg_logit;   // shared gate logits or NULL
    int32_t* err;            // Ctrl::err
    const void* zero4;       // 4 zero bytes (stand-in scale source past the last row)
    // Down kernel only: after every tile, a grid barrier and the combine
    // (out = BF16(sum_j y[inv[t*k + j]] in slot order + y_sh[t] (+ out))).
    int combine;             // 0: the combine runs as a kernel of its own
    const int32_t* inv;      // route id -> sorted position (-1: dropped)
    uint16_t* out;           // [n, H] BF16 (device or mapped pinned host memory)
    int has_shared, accumulate;
    uint32_t* tc_count;      // Ctrl::tc_count
    uint32_t* tc_gen;        // Ctrl::tc_gen
};

bool build_tc_maps(int fmt, bool gate_up, const moe_weights_t* w, int E, int H, int I, int S, int n,
                   int n_routes_max, const void* act_routed, const void* act_shared, TcMaps* maps);
cudaError_t launch_grouped_tc(int fmt, bool gate_up, const TcMaps& maps, const TcParams& p, int num_sms,
                              cudaStream_t st);
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t st);
// norm_w (may be null): the pre-expert RMSNorm weight; the rows gathered are
// then the normalised ones (the norm kernel's values).
cudaError_t launch_gather(int fmt, const uint16_t* x, int n, int H, int k, const int32_t* perm,
                          const int32_t* offsets, int E, uint16_t* xs, uint16_t* xh, const uint16_t* norm_w,
                          float eps, bool early, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const float* y, const float* ysh, const int32_t* inv, int n, int H, int k,
                           int has_shared, int accumulate, uint16_t* out, bool early, int num_sms, cudaStream_t st);

// Fused single-token kernel (moe_fused_n1.cu).
struct FusedParams {
    const uint16_t* x;
    int H, E, k, I, S, routing, norm;
    float scale;
    int e_begin, e_end;       // local experts (expert parallelism)
    int accumulate;           // out = BF16(out + result)
    const uint16_t* norm_w;   // pre-expert RMSNorm weight or NULL
    float eps;
    const uint16_t* router;
    const uint16_t* gw;       // shared-gate weight or NULL
    const float* bias;
    QMatDev gate, up, down, sh_gate, sh_up, sh_down;
    float* logits;            // [E]
    float* sg_logit;          // [1]
    float* act;               // [k * I]
    float* act_sh;            // [S]
    int32_t* idx_out;         // [k]
    float* w_out;             // [k]
    uint16_t* out;            // [H]
    Ctrl* ctrl;
    int rpc;                  // output columns per CTA
    uint32_t row_bytes, drow_bytes, dsh_row_bytes;
    uint32_t off_x, off_xe, off_lg, off_sc, off_sel, off_cand, off_down, off_act, off_part, off_shgu, off_bar,
        smem_bytes;
    int n_cand;
};

bool fused_plan(const moe_config_t* c, int num_sms, FusedParams* p);
cudaError_t launch_fused_n1(int fmt, const FusedParams& p, int num_sms, cudaStream_t st);

cudaError_t launch_router(const uint16_t* x, int n, int H, const uint16_t* wr, int E,
                          const uint16_t* gw, float* logits, float* sg_logit, int num_sms,
                          cudaStream_t st);
// Tensor-core router (moe_router_tc.cu): partial logits [splits][n][E] of the
// BF16 router (rows E) for device-resident x, each multiplied by *scale when
// scale is not null; the caller checked router_tc_fits.
cudaError_t launch_router_tc(const uint16_t* x, int n, int H, const uint16_t* wr, int E, float* part,
                             int32_t* err, const float* scale, bool early, cudaStream_t st);
// The NVFP4 router [E, H] as BF16 (exact: E2M1 code times E4M3 block scale),
// for the tensor-core router, which multiplies its partials by scale2.
cudaError_t launch_router_nvfp4_expand(const QMatDev& wq, int E, int H, uint16_t* out, bool early, int num_sms,
                                       cudaStream_t st);
// 2-D TMA map over a row-major [rows, cols] matrix of `esize`-byte elements (moe_grouped_tc.cu).
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);
cudaError_t launch_router_nvfp4(const uint16_t* x, int n, int H, const QMatDev& wq, int E, float* logits,
                                cudaStream_t st);
// logits: ns partial rows per token ([ns][n][E], ns = 1 for a plain logit
// matrix), summed in order; lsum (may be null) receives the sums.
cudaError_t launch_topk(const float* logits, int ns, float* lsum, int n, int E, int k, int routing, const float* bias,
                        int norm, float scale, int32_t* idx, float* w, cudaStream_t st);
cudaError_t launch_group(const int32_t* idx, int nk, int E, int e_begin, int e_end, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active, int32_t* segs,
                         Ctrl* ctrl, cudaStream_t st);
cudaError_t launch_topk_group(const float* logits, int ns, int n, int E, int k, int routing, const float* bias,
                              int norm, float scale, int32_t* idx, float* w, int e_begin, int e_end, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active, int32_t* segs,
                              Ctrl* ctrl, const uint16_t* x, const uint16_t* gw, float* sg_logit, int H, bool early,
                              int num_sms, cudaStream_t st);
// Whether launch_topk_group can form the shared gate's logit (gw != null) for
// E experts and hidden size H.
bool topk_group_gate_fits(int E, int H);
cudaError_t launch_rmsnorm(const uint16_t* x, int n, int H, const uint16_t* w, float eps, uint16_t* xe,
                           cudaStream_t st);
cudaError_t launch_gate_up_tm(int fmt, const GateUpParams& gu, int num_sms, cudaStream_t st);
cudaError_t launch_down_blend_tm(int fmt, const DownParams& dn, int num_sms, cudaStream_t st);

}  // namespace moe
