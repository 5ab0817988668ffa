// moe_grouped_tc.cu -- expert-grouped tensor-core path for batched decode (sm_103a).
//
// The grouped decode of the pages ("metrale_model_layers/layers/moe/forward.rs":
// forward_nvfp4_grouped_decode, "rows do not depend on how many share the
// call"; "metrale_model_layers/layers/moe/forward_fp8_grouped_router.rs":
// grouped FP8 expert kernels fed by grouped_route): routes are grouped by
// expert, and each expert's matrices are streamed once for all of its tokens
// as a dense GEMM on the 5th-generation tensor cores.
//
//   gather     xs[p, :] = x[token(perm[p]), :]   (expert-sorted activations;
//              moe_gather.cu)
//   gate_up    per (expert, 128 rows of I, <=64 tokens) tile:
//              G = Wg x^T, U = Wu x^T on tcgen05 (TMEM accumulators),
//              a = SiLU(G) * U  -> as[p, i]
//   down       per (expert, 128 rows of H, <=64 tokens) tile:
//              D = Wd a^T;  y[p, h] = w(route p) * D      (fp32)
//   combine    out[t, h] = sum over t's slots, in slot order, of y[., h]
//              + the gated shared expert; BF16 (moe_gather.cu).  No atomics,
//              so every row's bits are independent of the rest of the batch.
//
// The tile's M dimension is 128 weight rows and its N dimension the expert's
// tokens (padded to a multiple of 16), so a thin token set still fills the
// MMA.  Weights: BF16 arrive by TMA straight in the 128-byte swizzled K-major
// layout the MMA reads from shared memory.  FP8 and NVFP4 arrive raw by TMA
// and dequant warps (8; 16 in two sets for FP8 gate/up) write them as f16 into tensor
// memory, where tcgen05.mma reads its A operand (FP8: RNE_f16(e4m3 * block
// scale), one rounding with an 11-bit significand; NVFP4: e2m1 * e4m3 scale,
// exact in f16, with the fp32 scale2 applied to the accumulator).  Those tiles
// run the f16 MMA with f16 activations (exact for BF16 inputs in f16's normal
// range, saturated at +-65504).  A pipeline stage covers 64 K (128 K in the
// FP8 and NVFP4 down kernels).  Warp roles: 0 TMA producer of the weight
// codes (and FP8/NVFP4 block scales), 1 MMA issuer (one thread) and TMEM
// owner, 2-5 epilogue (TMEM -> registers -> global), then the dequant warps,
// then (dequantised formats) the TMA producer of the token tiles.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "moe_launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;   // weight rows per tile (MMA M)
constexpr int BK = 64;    // K elements of one 128-byte-swizzled token-tile box (and a BF16 / FP8 stage)
constexpr int NT = kTcTokensPerTile;   // tokens per tile (max MMA N)

template <int FMT, bool GU>
struct TcCfg {
    static constexpr bool kDeq = FMT != MOE_W_BF16;
    static constexpr bool kF16 = FMT != MOE_W_BF16;   // FP8 and NVFP4 tiles: f16 operands
    static constexpr int kMats = GU ? 2 : 1;
    // K elements per pipeline stage: 64, or 128 for the dequantised down
    // kernels, whose one matrix gives a 64-K stage half the codes of gate/up's
    // for the same handshakes (measured on GB300: NVFP4 down 103.7 -> 78.8 us
    // at nvfp4_n256, fp8_n64 1076 -> 1009 us; gate/up at 128 K, three TMEM
    // operand stages, was slower: NVFP4 128.2 -> 136.2 us).
    static constexpr int kBK = (kDeq && !GU) ? 128 : BK;
    static constexpr int kAMat = BM * kBK * 2;
    static constexpr int kAStage = kMats * kAMat;
    // Token tiles: kBK / BK boxes of BK columns (one 128-byte swizzle atom each),
    // kBAtom bytes apart.
    static constexpr int kBAtom = NT * BK * 2;
    static constexpr int kBStage = (kBK / BK) * kBAtom;
    static constexpr int kRawRow = FMT == MOE_W_FP8_B128 ? kBK : (FMT == MOE_W_NVFP4 ? kBK / 2 : 0);
    static constexpr int kRawMat = BM * kRawRow;
    static constexpr int kRawStage = kMats * kRawMat;
    // BF16 tiles: operand stages in shared memory (TMA, 128-byte swizzle).
    // FP8 / NVFP4 tiles: the dequant warps write the f16 operand stages into
    // tensor memory (tcgen05.st), where tcgen05.mma reads A; shared memory
    // holds only the raw codes and the token tiles, so the raw ring is deep.
    // Tensor memory: kAccBufs accumulators of kMats x NT fp32 columns (two, so
    // a tile's epilogue overlaps the next tile's MMAs; one for dequantised
    // gate/up, so that the operand ring gets the columns -- its thin tiles
    // still alternate between the accumulator's halves, see AccSlots), then
    // (dequantised tiles) the operand
    // stages, kMats x kBK/2 columns each (two f16 per 32-bit column, row i of
    // the tile in lane i).
    static constexpr int kAccBufs = (kDeq && GU) ? 1 : 2;
    static constexpr int kAccCols = kMats * NT;
    static constexpr int kACols = kMats * kBK / 2;
    static constexpr int kAColBase = kAccBufs * kAccCols;
    static constexpr int kTmemCols = kDeq ? 512 : kAccBufs * kAccCols;
    static constexpr int kAStages = kDeq ? (512 - kAColBase) / kACols : (GU ? 5 : 8);
    static constexpr int kASmemStages = kDeq ? 0 : kAStages;
    // Dequantised tiles hand operand stages to the MMA warp in groups (one
    // barrier round trip per group instead of per stage), sizes measured on
    // GB300: NVFP4 gate/up three of its six 64-K stages, FP8 gate/up two of
    // six (fp8_n64 1129 -> 1113 us against three), both down kernels pairs of
    // their six 128-K stages (FP8 triples: 1065 against 1009 us; NVFP4
    // gate/up pairs were slower, 214 -> 219 us at nvfp4_n256).
    static constexpr int kGrp = !kDeq ? 1 : ((FMT == MOE_W_NVFP4 && GU) ? 3 : 2);
    static constexpr int kAGroups = kAStages / kGrp;
    // Dequantised tiles: the token (B) tiles have a ring of their own, so they
    // are fetched ahead instead of after the MMA frees an A slot.  It holds
    // kBGroups groups of kGrp stages with one full / empty barrier pair per
    // group, so the MMA warp waits and commits once per group, not per stage.
    static constexpr int kBGroups = kDeq ? 2 : 1;   // (BF16: no token ring of its own)
    static constexpr int kBStages = kDeq ? kBGroups * kGrp : kAStages;
    // Raw stages: FP8 gate/up 10 of 16 KB (64 K), FP8 down 8 of 16 KB (128 K),
    // NVFP4 gate/up 16 of 8 KB (64 K), NVFP4 down 12 of 8 KB (128 K).
    static constexpr int kRawStages = !kDeq ? 0 : (GU ? (FMT == MOE_W_FP8_B128 ? 10 : 16) : (FMT == MOE_W_FP8_B128 ? 8 : 12));
    // Dequant warps: kDeqSets sets of 8 (two per TMEM lane quarter); set s
    // converts the stages with stage counter = s (mod kDeqSets), so a set's
    // warps overlap their per-stage chains with the other set's while every
    // stage still has 8 handshakes.  Measured on GB300: FP8 two sets (gate/up
    // 668 -> 638 us at fp8_n64; the down kernel at 128-K stages 1009.7 ->
    // 992.7 us for the layer), NVFP4 one (two: nvfp4_n256 207.4 -> 211.3 us
    // for both kernels, no change for down alone; 16 warps each converting a
    // quarter of every stage: 213.7 -> 219.5).
    static constexpr int kDeqSets = !kDeq ? 0 : (FMT == MOE_W_FP8_B128 ? 2 : 1);
    static constexpr int kSetWarps = 8;
    static constexpr int kDeqWarps = kDeqSets * kSetWarps;
    // Dequant work split: warp 6 + dw serves TMEM lane quarter (6 + dw) & 3 (the
    // quarter a warp may access), set dw / 8 and part (dw % 8) >> 2 of each row's
    // kMats x kBK codes.
    static constexpr int kParts = kSetWarps / 4;
    static constexpr int kPartElems = kDeq ? kMats * kBK / kParts : 0;
    // Dequantised tiles: a second producer warp for the token (B) tiles, after
    // the dequant warps, so a full B ring never holds up the weight copies.
    static constexpr int kBWarp = 6 + kDeqWarps;
    static constexpr int kThreads = (6 + kDeqWarps + (kDeq ? 1 : 0)) * 32;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kASmemStages * kAStage;
    static constexpr int kOffRaw = kOffB + kBStages * kBStage;
    // Block scales of each raw stage, fetched by the producer warp with the
    // raw codes: FP8 one fp32 per matrix; NVFP4 kBK / 16 E4M3 bytes per row per matrix.
    static constexpr int kScaleRow = FMT == MOE_W_NVFP4 ? kBK / 16 : 0;
    static constexpr int kScaleStage = FMT == MOE_W_FP8_B128 ? 16 : (FMT == MOE_W_NVFP4 ? kMats * BM * kScaleRow : 0);
    static constexpr int kOffScale = kOffRaw + kRawStages * kRawStage;
    static constexpr int kOffBar = kOffScale + kRawStages * kScaleStage;
    // a_full, a_empty per A stage; b_full, b_empty per B stage; raw_full,
    // raw_empty per raw stage; acc_full[2], acc_empty[2], drain.
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kRawStages + 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;   // + alignment slack
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kTmemCols <= 512, "TMEM budget");
    static_assert(!kDeq || kAColBase + kAStages * kACols <= kTmemCols, "TMEM operand stages");
    static_assert(kAStages % kGrp == 0, "operand stages come in whole groups");
    static_assert(kOffRaw % 1024 == 0 && kRawMat % 1024 == 0, "swizzled raw stages sit on 1024-byte boundaries");
    static_assert(!kDeq || (kPartElems % 16 == 0 && kBK % (kDeq ? kPartElems : 1) == 0),
                  "a dequant part is whole 16-code blocks of one matrix");
    static_assert(kBK % BK == 0 && kBStage % 1024 == 0, "token-tile boxes on swizzle-atom boundaries");
};

// Accumulator slots of the tiles, chosen alike by the MMA warp and the
// epilogue (both walk the same tile sequence).  Two accumulators (kAccBufs
// == 2): tile i takes buffer i % 2.  One accumulator: it is two slots of NT/2
// tokens; a tile of at most NT/2 tokens takes one slot, the thin tiles
// alternating, and a wider tile takes both.  So consecutive thin tiles are
// double-buffered: one's epilogue overlaps the next one's MMAs.  Each slot has
// its own full/empty barriers, and each role counts its uses of each slot for
// the barrier parity.
template <int kAccBufs, int kAccCols>
struct AccSlots {
    uint32_t use[2] = {0u, 0u};
    uint32_t seq = 0;   // tiles (two accumulators) or thin tiles (one)
    // mask: bit s = slot s used; col: first accumulator column of the tile.
    __device__ __forceinline__ void pick(int nmma, int& mask, int& col) {
        if constexpr (kAccBufs == 2) {
            const int s = (int)(seq++ & 1u);
            mask = 1 << s;
            col = s * kAccCols;
        } else if (nmma <= NT / 2) {
            const int s = (int)(seq++ & 1u);
            mask = 1 << s;
            col = s * (NT / 2);
        } else {
            mask = 3;
            col = 0;
        }
    }
    __device__ __forceinline__ void done(int mask) {
        use[0] += mask & 1;
        use[1] += (mask >> 1) & 1;
    }
};

struct Tile {
    int e;        // expert (routed) or -1 (shared)
    int le;       // the expert's index in the weight stacks (0 for the shared expert)
    int pos0;     // first row of this tile's tokens in the activation matrix
    int ntok;     // tokens in the tile (1..NT)
    int m0;       // first weight row
    int out;      // weight rows of this matrix
    int K;        // reduction length
};

// Tiles in order: the shared expert's (token segments of sh_seg rows x its
// BM-row blocks), then each routed segment's row blocks.
__device__ __forceinline__ Tile decode_tile(int tau, const TcParams& p, int n_ssegs, int sh_seg) {
    Tile t;
    const int mbs = (p.sh_out + BM - 1) / BM;
    const int mbr = (p.out_dim + BM - 1) / BM;
    if (tau < n_ssegs * mbs) {
        const int s = tau / mbs, mb = tau - s * mbs;
        t.e = -1;
        t.le = 0;
        t.pos0 = s * sh_seg;
        t.ntok = min(sh_seg, p.n - t.pos0);
        t.m0 = mb * BM;
        t.out = p.sh_out;
        t.K = p.sh_in;
    } else {
        const int t2 = tau - n_ssegs * mbs;
        const int s = t2 / mbr, mb = t2 - s * mbr;
        const int32_t* sg = p.segs + 3 * s;
        t.e = sg[0];
        t.le = sg[0] - p.e_base;
        t.pos0 = sg[1];
        t.ntok = sg[2];
        t.m0 = mb * BM;
        t.out = p.out_dim;
        t.K = p.in_dim;
    }
    return t;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t h2;
    asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(two));
    return h2;
}

// The four bytes of w, each a pair of E2M1 codes (the even element in the low
// nibble), as four f16x2: byte b -> h[b], exact.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// The two 16-bit halves of w, each a pair of E4M3 codes, as two f16x2.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t (&h)[2]) {
    asm("{ .reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi; }"
        : "=r"(h[0]), "=r"(h[1])
        : "r"(w));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t h2) {
    __half2_raw raw;
    raw.x = (unsigned short)(h2 & 0xffffu);
    raw.y = (unsigned short)(h2 >> 16);
    return __half22float2(__half2(raw));
}

// Byte offset of 16-byte chunk c of row r in a raw stage of kRawRow-byte rows.
// The TMA writes the raw codes swizzled, the row's chunk index XORed with
// address bits 7 and up: 128-byte rows (the FP8 down kernel's 128 codes) with
// the 128-byte swizzle, c ^ (r & 7); 64-byte rows (FP8 gate/up's 64 codes,
// the NVFP4 down kernel's 128) with the 64-byte swizzle, c ^ ((r >> 1) & 3);
// NVFP4 gate/up's 32-byte rows with the 32-byte swizzle, c ^ ((r >> 2) & 1).
// So each 8-lane phase of 32 lanes reading one chunk of 32 consecutive rows
// touches 8 distinct 16-byte bank groups.
template <int kRawRow>
__device__ __forceinline__ int raw_chunk(int r, int c) {
    if constexpr (kRawRow == 128) return r * 128 + ((c ^ (r & 7)) << 4);
    else if constexpr (kRawRow == 64) return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
    else return r * 32 + ((c ^ ((r >> 2) & 1)) << 4);
}

template <int FMT, bool GU>
__global__ void __launch_bounds__(TcCfg<FMT, GU>::kThreads, 1)
grouped_tc_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
    using C = TcCfg<FMT, GU>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    uint8_t* sRaw = smem + C::kOffRaw;
    uint8_t* sScale = smem + C::kOffScale;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* a_full = bars;
    uint64_t* a_empty = bars + C::kAStages;
    uint64_t* b_full = bars + 2 * C::kAStages;
    uint64_t* b_empty = b_full + C::kBStages;
    uint64_t* raw_full = b_empty + C::kBStages;
    uint64_t* raw_empty = raw_full + C::kRawStages;
    uint64_t* acc_full = raw_empty + C::kRawStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kAGroups; ++s) {
            ptx::mbar_init(&a_full[s], C::kDeq ? C::kDeqWarps : 1);
            ptx::mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < C::kBStages; ++s) {
            ptx::mbar_init(&b_full[s], 1);
            ptx::mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < C::kRawStages; ++s) {
            ptx::mbar_init(&raw_full[s], 1 + 32);   // TMA expect_tx + the producer warp's scale copies
            ptx::mbar_init(&raw_empty[s], C::kSetWarps);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 4);
        }
        ptx::mbar_init(drain, 1);
        *s_abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) ptx::tmem_alloc(s_tmem, C::kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    // Down kernel with the combine: whether this block takes part (no device
    // error pending from an earlier call), and the generation of the grid
    // barrier before the combine, read before this block arrives (it advances
    // only after every block's arrival, this one's included).
    volatile int* s_comb = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile uint32_t* s_gen = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 12);
    if (!GU && threadIdx.x == 0 && p.combine) {
        *s_comb = ptx::ld_relaxed_gpu(reinterpret_cast<const uint32_t*>(p.err)) == 0u ? 1 : 0;
        *s_gen = ptx::ld_relaxed_gpu(p.tc_gen);
    }

    const int n_rsegs = p.ctrl->n_rsegs;
    // The shared expert's token segments: NT rows, or NT / 2 with one
    // accumulator, so that its tiles alternate between the accumulator's two
    // slots like the routed ones (a wide tile would hold both and stall the
    // next tile's MMAs for its whole epilogue).
    constexpr int kShSeg = C::kAccBufs == 1 ? NT / 2 : NT;
    const int n_ssegs = (p.sh_out > 0) ? (p.n + kShSeg - 1) / kShSeg : 0;
    const int n_tiles = n_ssegs * ((p.sh_out + BM - 1) / BM) + n_rsegs * ((p.out_dim + BM - 1) / BM);
    int32_t* err = p.err;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop: lane 0 issues the TMA copies; for FP8 /
        // NVFP4 every lane also copies its share of the stage's block scales
        // into shared memory (cp.async), completing on the raw stage's barrier.
        uint32_t it = 0;
        bool stop = false;
        for (int tau = blockIdx.x; tau < n_tiles && !stop && !ptx::aborted_warp(s_abort); tau += gridDim.x) {
            const Tile t = decode_tile(tau, p, n_ssegs, kShSeg);
            const bool sh = t.e < 0;
            const int wrow = sh ? t.m0 : t.le * t.out + t.m0;
            const int nbox = (t.ntok + 15) >> 4;
            const CUtensorMap* bmap = sh ? &maps.bs : &maps.b;
            const int KB = (t.K + C::kBK - 1) / C::kBK;
            const bool nv_smem_scales = (FMT == MOE_W_NVFP4) && (t.K % C::kBK == 0);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int k0 = kb * C::kBK;
                if constexpr (C::kDeq) {
                    const int rs = it % C::kRawStages;
                    if (!ptx::mbar_wait_warp(&raw_empty[rs], ((it / C::kRawStages) & 1) ^ 1, s_abort, err, 1)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&raw_full[rs], C::kRawStage);
                        const int xr = (FMT == MOE_W_FP8_B128) ? k0 : k0 / 2;
                        for (int m = 0; m < C::kMats; ++m)
                            ptx::tma_load_2d(sRaw + rs * C::kRawStage + m * C::kRawMat,
                                             sh ? &maps.ws[m] : &maps.w[m], xr, wrow, &raw_full[rs]);
                    }
                    uint8_t* ssc = sScale + rs * C::kScaleStage;
                    if constexpr (FMT == MOE_W_FP8_B128) {
                        if (lane < C::kMats) {
                            const int ob = (t.out + 127) >> 7, ib = (t.K + 127) >> 7;
                            const float* sp = reinterpret_cast<const float*>(sh ? p.sh_scale[lane] : p.scale[lane]);
                            ptx::cp_async4(ssc + 4 * lane,
                                           sp + (size_t)t.le * ob * ib + (t.m0 >> 7) * ib + (k0 >> 7));
                        }
                    } else if (nv_smem_scales) {
                        // Row r's kScaleRow scale bytes of this stage: columns [k0, k0 + kBK),
                        // four bytes per copy (the scale arrays are 4-byte aligned).
                        for (int m = 0; m < C::kMats; ++m) {
                            const uint8_t* sp = reinterpret_cast<const uint8_t*>(sh ? p.sh_scale[m] : p.scale[m]);
#pragma unroll
                            for (int q = 0; q < BM / 32; ++q) {
                                const int r = lane + 32 * q, mrow = t.m0 + r;
#pragma unroll
                                for (int h = 0; h < C::kScaleRow / 4; ++h) {
                                    const uint8_t* src = (mrow < t.out)
                                        ? sp + ((size_t)t.le * t.out + mrow) * (t.K / 16) + k0 / 16 + 4 * h
                                        : reinterpret_cast<const uint8_t*>(p.zero4);
                                    ptx::cp_async4(ssc + (m * BM + r) * C::kScaleRow + 4 * h, src);
                                }
                            }
                        }
                    }
                    ptx::cp_async_mbar_arrive(&raw_full[rs]);
                } else {
                    const int as = it % C::kAStages;   // kGrp == 1: a group is a stage
                    if (!ptx::mbar_wait_warp(&a_empty[as], ((it / C::kAStages) & 1) ^ 1, s_abort, err, 1)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(&a_full[as], C::kAStage + nbox * 2048 * (C::kBK / BK));
                        for (int m = 0; m < C::kMats; ++m)
                            ptx::tma_load_2d(sA + as * C::kAStage + m * C::kAMat,
                                             sh ? &maps.ws[m] : &maps.w[m], k0, wrow, &a_full[as]);
                        for (int a = 0; a < C::kBK / BK; ++a)
                            for (int j = 0; j < nbox; ++j)
                                ptx::tma_load_2d(sB + as * C::kBStage + a * C::kBAtom + j * 2048, bmap, k0 + a * BK,
                                                 t.pos0 + 16 * j, &a_full[as]);
                    }
                }
            }
        }
        if constexpr (C::kDeq) asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0 && *s_abort) {
            // Let every copy this warp issued land before the CTA exits:
            // wait (bounded) on the last phase of each ring stage it used.
            constexpr uint32_t kRing = C::kDeq ? C::kRawStages : C::kAStages;
            const uint32_t na = it < kRing ? it : kRing;
            for (uint32_t q = 0; q < na; ++q) {
                const uint32_t i2 = it - 1 - q, s2 = i2 % kRing;
                ptx::mbar_wait_quiet(C::kDeq ? &raw_full[s2] : &a_full[s2], (i2 / kRing) & 1, 100000000ull);
            }
        }
    } else if (C::kDeq && warp == C::kBWarp) {
        // ------------------------------------------------------------ token-tile producer
        // Group by group, as the MMA warp consumes them: group gb (of the MMA
        // warp's group sequence) fills B group gb % kBGroups, its stages' token
        // tiles completing on that group's barrier.
        if (lane == 0) {
            uint32_t gb = 0;
            bool stop = false;
            for (int tau = blockIdx.x; tau < n_tiles && !stop && !*s_abort; tau += gridDim.x) {
                const Tile t = decode_tile(tau, p, n_ssegs, kShSeg);
                const int nbox = (t.ntok + 15) >> 4;
                const CUtensorMap* bmap = t.e < 0 ? &maps.bs : &maps.b;
                const int KB = (t.K + C::kBK - 1) / C::kBK;
                for (int kb = 0; kb < KB; ++gb) {
                    const int bg = gb % C::kBGroups;
                    const int n = min(C::kGrp, KB - kb);
                    if (!ptx::mbar_wait(&b_empty[bg], ((gb / C::kBGroups) & 1) ^ 1, s_abort, err, 5)) {
                        stop = true;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&b_full[bg], n * nbox * 2048 * (C::kBK / BK));
                    for (int u = 0; u < n; ++u, ++kb)
                        for (int a = 0; a < C::kBK / BK; ++a)
                            for (int j = 0; j < nbox; ++j)
                                ptx::tma_load_2d(sB + (bg * C::kGrp + u) * C::kBStage + a * C::kBAtom + j * 2048,
                                                 bmap, kb * C::kBK + a * BK, t.pos0 + 16 * j, &b_full[bg]);
                }
            }
            if (*s_abort) {
                const uint32_t nb = gb < (uint32_t)C::kBGroups ? gb : C::kBGroups;
                for (uint32_t q = 0; q < nb; ++q) {
                    const uint32_t i2 = gb - 1 - q, s2 = i2 % C::kBGroups;
                    ptx::mbar_wait_quiet(&b_full[s2], (i2 / C::kBGroups) & 1, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop, so the operand descriptors are
        // warp-uniform values; one elected lane issues the MMAs and commits.
        uint32_t git = 0;
        AccSlots<C::kAccBufs, C::kAccCols> slots;
        for (int tau = blockIdx.x; tau < n_tiles && !ptx::aborted_warp(s_abort); tau += gridDim.x) {
            const Tile t = decode_tile(tau, p, n_ssegs, kShSeg);
            const int nmma = ((t.ntok + 15) >> 4) << 4;
            int amask, acol;
            slots.pick(nmma, amask, acol);
            bool free_ok = true;
            for (int sl = 0; sl < 2 && free_ok; ++sl)
                if ((amask >> sl) & 1)
                    free_ok = ptx::mbar_wait_warp(&acc_empty[sl], (slots.use[sl] & 1) ^ 1, s_abort, err, 2);
            if (!free_ok) break;
            ptx::tc_fence_after();
            const uint32_t idesc = ptx::idesc_f16(BM, nmma, !C::kF16);
            const uint32_t d0 = tmem + acol;
            const int KB = (t.K + C::kBK - 1) / C::kBK;
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++git) {
                // One group of operand stages: one a_full wait, one a_empty commit.
                const int g = git % C::kAGroups;
                const int bg = C::kDeq ? (int)(git % C::kBGroups) : 0;
                if (!ptx::mbar_wait_warp(&a_full[g], (git / C::kAGroups) & 1, s_abort, err, 2)) { ok = false; break; }
                if constexpr (C::kDeq)
                    if (!ptx::mbar_wait_warp(&b_full[bg], (git / C::kBGroups) & 1, s_abort, err, 2)) {
                        ok = false;
                        break;
                    }
                ptx::tc_fence_after();
                const int n = min(C::kGrp, KB - kb);
                // The group's MMAs and its commits from one elected lane (one
                // divergent region per group, not per stage).
                if (ptx::elect_one()) {
                    for (int u = 0; u < n; ++u) {
                        const int as = g * C::kGrp + u;
                        const int bs = C::kDeq ? bg * C::kGrp + u : as;
                        const bool first = kb + u == 0;   // the tile's first stage starts the accumulator
                        // Descriptors of the stage's first K step; a later step (or the
                        // second matrix) only moves the start address field (16-byte units):
                        // K step kk of the token tile is 32 bytes into swizzle atom kk / 4.
                        const uint64_t b_desc = ptx::sw128_desc(ptx::smem_u32(sB + bs * C::kBStage));
                        if constexpr (C::kDeq) {
                            // A in tensor memory: K step kk of matrix m is 8 columns on.
                            const uint32_t a_t = tmem + C::kAColBase + as * C::kACols;
    #pragma unroll
                            for (int m = 0; m < C::kMats; ++m)
    #pragma unroll
                                for (int kk = 0; kk < C::kBK / 16; ++kk)
                                    ptx::mma_f16_ts(d0 + m * NT, a_t + m * (C::kBK / 2) + kk * 8,
                                                    b_desc + (uint64_t)(((kk >> 2) * C::kBAtom + (kk & 3) * 32) >> 4),
                                                    idesc, (!first || kk > 0) ? 1u : 0u);
                        } else {
                            const uint64_t a_desc = ptx::sw128_desc(ptx::smem_u32(sA + as * C::kAStage));
    #pragma unroll
                            for (int m = 0; m < C::kMats; ++m)
    #pragma unroll
                                for (int kk = 0; kk < C::kBK / 16; ++kk)   // BF16: kBK == BK, one atom
                                    ptx::mma_f16(d0 + m * NT, a_desc + (uint64_t)((m * C::kAMat + kk * 32) >> 4),
                                                 b_desc + (uint64_t)((kk * 32) >> 4), idesc,
                                                 (!first || kk > 0) ? 1u : 0u);
                        }
                    }
                    ptx::mma_commit(&a_empty[g]);   // after the group's MMAs
                    if constexpr (C::kDeq) ptx::mma_commit(&b_empty[bg]);
                }
                __syncwarp();
                kb += n;
            }
            if (!ok) break;
            if (ptx::elect_one())
                for (int sl = 0; sl < 2; ++sl)
                    if ((amask >> sl) & 1) ptx::mma_commit(&acc_full[sl]);
            __syncwarp();
            slots.done(amask);
        }
        // Every MMA issued has completed before TMEM is released.
        if (ptx::elect_one()) {
            ptx::mma_commit(drain);
            ptx::mbar_wait_quiet(drain, 0, 100000000ull);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        // The tile's global operands (NVFP4 scale2; per token the routing
        // weight or the shared-expert gate) are loaded before the accumulator
        // wait, lane l holding token l and l + 32, and broadcast by shuffles.
        const int q = warp & 3;                     // TMEM lane quarter of this warp
        const int row = 32 * q + lane;
        AccSlots<C::kAccBufs, C::kAccCols> slots;
        for (int tau = blockIdx.x; tau < n_tiles && !ptx::aborted_warp(s_abort); tau += gridDim.x) {
            const Tile t = decode_tile(tau, p, n_ssegs, kShSeg);
            int amask, acol;
            slots.pick(((t.ntok + 15) >> 4) << 4, amask, acol);
            const int m = t.m0 + row;
            const bool valid = m < t.out;
            const bool sh = t.e < 0;
            float s2g = 1.f, s2u = 1.f;
            if constexpr (FMT == MOE_W_NVFP4) {
                s2g = sh ? p.sh_scale2[0][0] : p.scale2[0][t.le];
                if constexpr (GU) s2u = sh ? p.sh_scale2[1][0] : p.scale2[1][t.le];
            }
            float tw[2] = {0.f, 0.f};   // down: weight of token lane, lane + 32 (times scale2)
            if constexpr (!GU) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    if (j < t.ntok) {
                        float wgt;
                        if (sh) wgt = p.sg_logit ? 1.0f / (1.0f + expf(-p.sg_logit[t.pos0 + j])) : 1.0f;
                        else wgt = p.route_w[p.perm[t.pos0 + j]];
                        tw[h] = wgt * s2g;
                    }
                }
            }
            bool full_ok = true;
            for (int sl = 0; sl < 2 && full_ok; ++sl)
                if ((amask >> sl) & 1)
                    full_ok = ptx::mbar_wait_warp(&acc_full[sl], slots.use[sl] & 1, s_abort, err, 3);
            if (!full_ok) break;
            ptx::tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + acol;
            if constexpr (GU) {
                uint16_t* dst = reinterpret_cast<uint16_t*>(sh ? p.act_sh_out : p.act_out);
                for (int j0 = 0; j0 < t.ntok; j0 += 16) {
                    float g[16], u[16];
                    ptx::tmem_ld16(tb + j0, g);
                    ptx::tmem_ld16(tb + NT + j0, u);
                    if (valid) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j < t.ntok) {
                                const float gv = g[jj] * s2g, uv = u[jj] * s2u;
                                const float a = gv / (1.0f + expf(-gv)) * uv;
                                uint16_t bits;
                                if constexpr (C::kF16) {
                                    const __half h = __float2half_rn(fminf(fmaxf(a, -65504.f), 65504.f));
                                    bits = *reinterpret_cast<const uint16_t*>(&h);
                                } else {
                                    const __nv_bfloat16 b = __float2bfloat16_rn(a);
                                    bits = *reinterpret_cast<const uint16_t*>(&b);
                                }
                                dst[(size_t)(t.pos0 + j) * t.out + m] = bits;
                            }
                        }
                    }
                }
            } else {
                float* dst = sh ? p.y_sh : p.y;
                for (int j0 = 0; j0 < t.ntok; j0 += 16) {
                    float d[16];
                    ptx::tmem_ld16(tb + j0, d);
                    float wj[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        wj[jj] = __shfl_sync(0xffffffffu, j < 32 ? tw[0] : tw[1], j & 31);
                    }
                    if (valid) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j < t.ntok) dst[(size_t)(t.pos0 + j) * t.out + m] = d[jj] * wj[jj];
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            for (int sl = 0; sl < 2; ++sl)
                if ((amask >> sl) & 1) ptx::mbar_arrive_elect(&acc_empty[sl]);
            slots.done(amask);
        }
    } else if constexpr (C::kDeq) {
        // ------------------------------------------------------------ dequant
        // Thread `lane` of a dequant warp converts row r = 32 qd + lane of its
        // part of every stage: kPartElems codes of matrix pm from column pk0 of
        // the stage, kPartElems / 2 f16x2 words written to that row's lane of
        // the stage's TMEM operand columns.
        constexpr int PE = C::kPartElems, NC = PE / 2;
        const int dset = (warp - 6) / C::kSetWarps;
        const int qd = warp & 3, part = ((warp - 6) % C::kSetWarps) >> 2;
        const int r = 32 * qd + lane;
        const int pm = (part * PE) / C::kBK, pk0 = (part * PE) % C::kBK;
        const uint32_t t_row = tmem + ((uint32_t)(32 * qd) << 16) + C::kAColBase + pm * (C::kBK / 2) + pk0 / 2;
        uint32_t it = 0, git = 0;
        for (int tau = blockIdx.x; tau < n_tiles && !ptx::aborted_warp(s_abort); tau += gridDim.x) {
            const Tile t = decode_tile(tau, p, n_ssegs, kShSeg);
            const bool sh = t.e < 0;
            const int KB = (t.K + C::kBK - 1) / C::kBK;
            const int mrow = t.m0 + r;
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++git) {
                // A group of kGrp operand stages (fewer at the end of the tile).
                const int g = git % C::kAGroups;
                if (!ptx::mbar_wait_warp(&a_empty[g], ((git / C::kAGroups) & 1) ^ 1, s_abort, err, 4)) { ok = false; break; }
                ptx::tc_fence_after();   // the MMAs that read these columns are complete
                const int n = min(C::kGrp, KB - kb);
                for (int u = 0; u < n; ++u, ++kb, ++it) {
                    if (C::kDeqSets > 1 && (int)(it % C::kDeqSets) != dset) continue;   // the other set's stage
                    const int rs = it % C::kRawStages, as = g * C::kGrp + u;
                    if (!ptx::mbar_wait_warp(&raw_full[rs], (it / C::kRawStages) & 1, s_abort, err, 4)) { ok = false; break; }
                    const int k0 = kb * C::kBK;
                    const uint8_t* raw = sRaw + rs * C::kRawStage + pm * C::kRawMat;
                    uint32_t o[NC];
                    if constexpr (FMT == MOE_W_FP8_B128) {
                        // One fp32 scale per 128x128 block: uniform over this stage
                        // (fetched into shared memory with the codes).
                        const float s = reinterpret_cast<const float*>(sScale + rs * C::kScaleStage)[pm];
                        // In f16's normal range the product is formed in f16x2 (the
                        // scale and the product each rounded once to f16); else in fp32.
                        const bool f16_scale = s >= 6.2e-5f && s <= 128.0f;
                        const __half2 s2 = __float2half2_rn(s);
                        const uint32_t s2u = *reinterpret_cast<const uint32_t*>(&s2);
    #pragma unroll
                        for (int c = 0; c < PE / 16; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4*>(raw + raw_chunk<C::kRawRow>(r, pk0 / 16 + c));
                            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                            if (f16_scale) {
    #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    uint32_t h[2];
                                    e4m3x4_to_f16x2x2(w4[i], h);
                                    o[8 * c + 2 * i] = f16x2_mul(h[0], s2u);
                                    o[8 * c + 2 * i + 1] = f16x2_mul(h[1], s2u);
                                }
                            } else {
    #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float2 lo = f16x2_to_float2(e4m3x2_to_f16x2(w4[i] & 0xffffu));
                                    const float2 hi = f16x2_to_float2(e4m3x2_to_f16x2(w4[i] >> 16));
                                    o[8 * c + 2 * i] = pack_f16(lo.x * s, lo.y * s);
                                    o[8 * c + 2 * i + 1] = pack_f16(hi.x * s, hi.y * s);
                                }
                            }
                        }
                    } else {
                        // NVFP4: 16 codes (8 bytes) per E4M3 block scale.  A part is whole
                        // pairs of blocks, one 16-byte chunk of the raw row each (a
                        // conflict-free shared load under either swizzle).
                        static_assert(PE % 32 == 0, "NVFP4 dequant parts are pairs of scale blocks");
    #pragma unroll
                        for (int b = 0; b < PE / 16; b += 2) {
                            const int qb = pk0 / 16 + b;   // even scale block of the stage
                            const uint4 v = *reinterpret_cast<const uint4*>(raw + raw_chunk<C::kRawRow>(r, qb >> 1));
                            uint32_t sc[2] = {0u, 0u};   // f16x2 of the two block scales (0 outside the matrix)
                            if (t.K % C::kBK == 0) {
                                // Fetched into shared memory with the codes (0 past the last row):
                                // bytes qb and qb + 1 of the row's scales, in one 4-byte word.
                                const uint32_t w = reinterpret_cast<const uint32_t*>(
                                    sScale + rs * C::kScaleStage + (pm * BM + r) * C::kScaleRow)[qb >> 2];
                                const uint32_t s2 = e4m3x2_to_f16x2((w >> (8 * (qb & 3))) & 0xffffu);
                                sc[0] = __byte_perm(s2, 0u, 0x1010);
                                sc[1] = __byte_perm(s2, 0u, 0x3232);
                            } else {
    #pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int kc = k0 + 16 * (qb + h);
                                    if (mrow < t.out && kc < t.K) {
                                        const uint8_t* sp = reinterpret_cast<const uint8_t*>(sh ? p.sh_scale[pm] : p.scale[pm]) +
                                                            ((size_t)t.le * t.out + mrow) * (t.K / 16) + kc / 16;
                                        const uint32_t bb = __ldg(sp);
                                        sc[h] = e4m3x2_to_f16x2(bb | (bb << 8));
                                    }
                                }
                            }
                            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t lo[4], hi[4];
                                e2m1x8_to_f16x2x4(w4[2 * h], lo);
                                e2m1x8_to_f16x2x4(w4[2 * h + 1], hi);
    #pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    o[8 * (b + h) + i] = f16x2_mul(lo[i], sc[h]);
                                    o[8 * (b + h) + 4 + i] = f16x2_mul(hi[i], sc[h]);
                                }
                            }
                        }
                    }
                    const uint32_t ta = t_row + as * C::kACols;
                    if constexpr (NC == 8) ptx::tmem_st8(ta, o);
                    else if constexpr (NC == 16) ptx::tmem_st16(ta, o);
                    else ptx::tmem_st32(ta, o);
                    // The codes are in registers: the raw stage may be refilled.
                    __syncwarp();
                    ptx::mbar_arrive_elect(&raw_empty[rs]);
                }
                if (!ok) break;
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                ptx::mbar_arrive_elect(&a_full[g]);
            }
            if (!ok) break;
        }
    }

    if constexpr (!GU) {
        if (p.combine) {
            // Grid barrier: every block's y / y_sh rows are written before any
            // block combines.  The block's writes are ordered before thread 0's
            // fence by the barrier; the last arrival zeroes the count for the
            // next call and publishes the next generation; the others wait
            // (bounded) for it.
            __syncthreads();
            if (threadIdx.x == 0 && *s_comb) {
                __threadfence();
                const uint32_t g0 = *s_gen;
                if (atomicAdd(p.tc_count, 1u) == gridDim.x - 1) {
                    atomicExch(p.tc_count, 0u);
                    __threadfence();
                    ptx::st_release_gpu(p.tc_gen, g0 + 1u);
                } else {
                    const uint64_t t0 = ptx::globaltimer();
                    while (ptx::ld_acquire_gpu(p.tc_gen) == g0) {
                        if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
                            atomicExch(p.err, 8);
                            *s_comb = 0;
                            break;
                        }
                    }
                }
                __threadfence();
            }
            __syncthreads();
            if (*s_comb)
                combine_range<true>(p.y, p.y_sh, p.inv, p.n, p.out_dim, p.k, p.has_shared, p.accumulate, p.out,
                                    blockIdx.x * (int64_t)blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
        }
    }
    pdl_trigger();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

// Weight map: BF16 (128-byte swizzle, the MMA operand layout) or raw codes
// (FP8: 64-byte rows, 64-byte swizzle; NVFP4: 32-byte rows and the 32-byte
// swizzle for gate/up, 64-byte rows and the 64-byte swizzle for down; the
// layout raw_chunk reads).
bool weight_map(CUtensorMap* m, int fmt, const void* w, int rows_total, int in_dim, bool gate_up) {
    if (fmt == MOE_W_BF16)
        return make_map(m, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, in_dim, rows_total, BK, BM,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (fmt == MOE_W_FP8_B128)
        return gate_up ? make_map(m, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, in_dim, rows_total,
                                  TcCfg<MOE_W_FP8_B128, true>::kBK, BM, CU_TENSOR_MAP_SWIZZLE_64B)
                       : make_map(m, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, in_dim, rows_total,
                                  TcCfg<MOE_W_FP8_B128, false>::kBK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (gate_up)
        return make_map(m, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, in_dim / 2, rows_total,
                        TcCfg<MOE_W_NVFP4, true>::kBK / 2, BM, CU_TENSOR_MAP_SWIZZLE_32B);
    return make_map(m, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, in_dim / 2, rows_total,
                    TcCfg<MOE_W_NVFP4, false>::kBK / 2, BM, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool act_map(CUtensorMap* m, int fmt, const void* a, int rows, int cols) {
    return make_map(m, a, fmt != MOE_W_BF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    2, cols, rows > 0 ? rows : 1, BK, 16, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int FMT, bool GU>
cudaError_t launch_tc(const TcMaps& maps, const TcParams& p, int num_sms, cudaStream_t st) {
    using C = TcCfg<FMT, GU>;
    auto kern = grouped_tc_kernel<FMT, GU>;
    static std::mutex mu;
    static bool configured[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    launch_pdl(kern, num_sms, C::kThreads, C::kSmem, st, maps, p);
    return cudaGetLastError();
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// 2-D map over a row-major [rows, cols] matrix of `esize`-byte elements.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool build_tc_maps(int fmt, bool gate_up, const moe_weights_t* w, int E, int H, int I, int S, int n,
                   int n_routes_max, const void* act_routed, const void* act_shared, TcMaps* maps) {
    // gate_up: routed weights [E*I, H], shared [S, H], B = xs [rows, H] / x(or xh) [n, H]
    // down:    routed weights [E*H, I], shared [H, S], B = as [rows, I] / ash [n, S]
    // E is the experts the weight stacks hold.  With none (a call that holds
    // only the shared expert, S > 0) the routed maps repeat the shared ones:
    // no routed tile exists to use them.
    bool ok = true;
    if (E == 0 && S == 0) return false;
    if (gate_up) {
        if (E > 0) {
            ok &= weight_map(&maps->w[0], fmt, w->gate.w, E * I, H, true);
            ok &= weight_map(&maps->w[1], fmt, w->up.w, E * I, H, true);
        } else {
            ok &= weight_map(&maps->w[0], fmt, w->sh_gate.w, S, H, true);
            ok &= weight_map(&maps->w[1], fmt, w->sh_up.w, S, H, true);
        }
        if (S > 0) {
            ok &= weight_map(&maps->ws[0], fmt, w->sh_gate.w, S, H, true);
            ok &= weight_map(&maps->ws[1], fmt, w->sh_up.w, S, H, true);
            ok &= act_map(&maps->bs, fmt, act_shared, n, H);
        } else {
            maps->ws[0] = maps->w[0];
            maps->ws[1] = maps->w[1];
            maps->bs = maps->w[0];
        }
        ok &= act_map(&maps->b, fmt, act_routed, n_routes_max, H);
    } else {
        ok &= (E > 0) ? weight_map(&maps->w[0], fmt, w->down.w, E * H, I, false)
                      : weight_map(&maps->w[0], fmt, w->sh_down.w, H, S, false);
        maps->w[1] = maps->w[0];
        if (S > 0) {
            ok &= weight_map(&maps->ws[0], fmt, w->sh_down.w, H, S, false);
            ok &= act_map(&maps->bs, fmt, act_shared, n, S);
        } else {
            maps->ws[0] = maps->w[0];
            maps->bs = maps->w[0];
        }
        maps->ws[1] = maps->ws[0];
        ok &= act_map(&maps->b, fmt, act_routed, n_routes_max, I);
    }
    return ok;
}

cudaError_t launch_grouped_tc(int fmt, bool gate_up, const TcMaps& maps, const TcParams& p, int num_sms,
                              cudaStream_t st) {
    if (gate_up) {
        switch (fmt) {
            case MOE_W_BF16: return launch_tc<MOE_W_BF16, true>(maps, p, num_sms, st);
            case MOE_W_FP8_B128: return launch_tc<MOE_W_FP8_B128, true>(maps, p, num_sms, st);
            case MOE_W_NVFP4: return launch_tc<MOE_W_NVFP4, true>(maps, p, num_sms, st);
        }
    } else {
        switch (fmt) {
            case MOE_W_BF16: return launch_tc<MOE_W_BF16, false>(maps, p, num_sms, st);
            case MOE_W_FP8_B128: return launch_tc<MOE_W_FP8_B128, false>(maps, p, num_sms, st);
            case MOE_W_NVFP4: return launch_tc<MOE_W_NVFP4, false>(maps, p, num_sms, st);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
