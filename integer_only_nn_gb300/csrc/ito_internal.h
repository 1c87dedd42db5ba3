// Host-side internals shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ito.h"

namespace ito {

// Launches a kernel of this library with programmatic stream serialisation:
// it may be scheduled while the previous kernel in the stream finishes (its
// launch and CTA dispatch overlap that kernel's tail). Each kernel waits for its
// predecessor (griddep_wait) before it touches global memory, so the stream
// order of every memory access is the same as with a plain launch.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Records an error text for ito_last_error_string() and returns `code`.
int set_error(int code, const char* fmt, ...);

// Number of K terms per exactly-accumulated tensor-core chunk: products of
// two int8 values are at most 2^14 in magnitude, so 1024 of them sum to at
// most 2^24, the largest range in which fp32 holds every integer.
constexpr int kExactChunk = 1024;
// uint8 x int8 products reach 255 * 128 < 2^15: 512 terms stay within 2^24.
constexpr int kExactChunkU8 = 512;

inline int64_t pad8(int64_t n) { return (n + 7) & ~int64_t(7); }

// A row-major bf16 tensor [rows][cols] with `pitch` elements per row
// (pitch * 2 bytes must be a multiple of 16 for TMA).
struct Bf16View {
    const uint16_t* ptr;
    int64_t rows, cols, pitch;
};

// A prepared tensor-core contraction C[M][N] = sum_k A(m,k) B(n,k):
// A is [M][K] (K-major) or [K][M] (a_mn); B is [N][K] or [K][N] (b_mn).
struct GemmPlan {
    CUtensorMap mapA, mapB, mapC;
    CUtensorMap mapP;             // pair kernel: partial tiles of the split last wave (in split_ws)
    int use_tma_store;
    int pair;   // CTA-pair (cta_group::2) kernel
    int group;  // row tiles per raster group (L2 reuse)
    int tail_full, tail_parts;    // pair kernel: whole tiles, K pieces per remaining tile (1: no split)
    // pair kernel: speculative requantisation in the epilogue (rq_pred != nullptr); rq_redo
    // set: the re-launch that checks the prediction and recomputes on a miss (see FusedRq)
    CUtensorMap mapO8, mapOB;
    const int32_t* rq_pred;
    const int8_t* rq_gate;
    int64_t rq_ldg;
    int rq_relu;
    int32_t* rq_redo;
    int32_t* rq_d_shift;
    int32_t* rq_s_last;
    int rq_target_bits;
    int M, N, K, bn, chunk_kb;
    int splits, kb_per_split;     // split-K: slices of kb_per_split K blocks (splits == 1: none)
    int32_t* split_ws;            // [splits][M][ldc] int32 partials
    CUtensorMap mapS;             // split-K: the partials as a 3-D tensor [splits][M][N] (TMA stores)
    int split_tma;
    int64_t split_stride;
    bool a_mn, b_mn;
    int32_t* C;
    int64_t ldc;
    uint32_t* d_max;
    int* err;
};

// Device address of this library's error word on the current device.
int* device_error_word();
// One CTA whose bounded mbarrier wait runs out (records ITO_ERR_TIMEOUT).
int launch_wait_timeout_selftest(cudaStream_t s);

// cuTensorMapEncodeTiled through the runtime's driver entry point (nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 get_encode();
// SM count of the current device.
int num_sms();
// Tensor map over a bf16 view: box of 64 columns (128 bytes) x box_rows rows,
// 128-byte swizzle, zero fill outside the view.
int make_map_bf16(CUtensorMap* map, const Bf16View& v, int box_rows);

// ---- stride-2 convolution delta propagation by parity phases (ito_conv_dgrad.cu)

// Geometry of the phase kernel: output grid B x OH x OW (input H = 2 OH, W = 2 OW),
// IC input channels in tiles of 64, OC delta channels in blocks of 64; a row tile is
// ba images x oha output rows x OW columns (128 positions), n_iblk tiles per image column.
struct S2Geom {
    int B, OH, OW, IC;
    int oc_blocks, n_tiles;
    int oha, ba, n_iblk, m_tiles;
};

struct ConvS2Plan {
    CUtensorMap mapE;       // delta's bf16 copy [B][OH][OW][OC], 4-D
    CUtensorMap mapW;       // weights' bf16 copy [OC][9 IC], MN-major boxes
    CUtensorMap mapD[4];    // phase (py, px) = (i >> 1, i & 1) of the int32 delta D [B][H][W][IC]
    S2Geom g;
    int bn;                 // tile width (128 where IC is a multiple of 128, else 64)
    uint32_t* d_max;
    int* err;
};

// true when the phase kernel takes this convolution: stride 2, even H and W, OW in
// {8, 16, 32}, OH a power of two with OH * OW >= 32, IC and OC multiples of 64
bool conv_dgrad_s2_eligible(int B, int H, int W, int IC, int OC, int stride);
// D[b][y][x][ic] = sum over the taps reaching (y, x) of E[b][oh][ow][oc] W[oc][kh][kw][ic]
// for a 3x3, pad-1, stride-2 convolution; E: [B*OH*OW][lde] bf16, W: [OC][ldw] bf16
// (9 IC used); max |D| folded into *d_max (atomicMax; the caller zeroes it)
int conv_dgrad_s2_plan(ConvS2Plan* p, const uint16_t* eb, int64_t lde, const uint16_t* Wb, int64_t ldw, int B,
                       int H, int W, int IC, int OC, int32_t* D, uint32_t* d_max);
int conv_dgrad_s2_run(const ConvS2Plan& p, cudaStream_t s);

// Forward and weight gradient of the same convolutions on the four parity planes of the
// bf16 NHWC input X [B][H][W][ldx] (no patches; see k_conv_igemm).
enum { CONV_FWD = 0, CONV_WGRAD = 1 };
struct IgGeom {
    int B, OH, OW, IC, ic_blocks;
    int oha, ba, n_iblk;          // forward row tiles: ba images x oha rows x OW (128 positions)
    int ohb, bb, n_iblk_w;        // weight-gradient position blocks: bb images x ohb rows x OW (64)
    int m_tiles, n_tiles, num_kb, splits, kb_per_split, rows;
};
struct ConvIgPlan {
    int mode;
    int bn;                       // tile width: 128 where the result's columns allow, else 64
    CUtensorMap mapX[4];          // parity planes (py, px) = (i >> 1, i & 1)
    CUtensorMap mapOp;            // forward: W [OC][9 IC] K-major; weight gradient: E [positions][OC] MN-major
    CUtensorMap mapOut;           // Y [positions][OC], G [OC][9 IC], or G's K-slice partials
    IgGeom g;
    int32_t* G;                   // weight gradient with K slices: the result the reduction writes
    int32_t* ws;
    int OC, K9;
    uint32_t* d_max;
    int* err;
};
// Y[(b,oh,ow)][oc] (rows of OC) = the convolution; max |Y| into *d_max (the caller zeroes it)
int conv_fwd_s2_plan(ConvIgPlan* p, const uint16_t* xb, int64_t ldx, const uint16_t* Wb, int64_t ldw, int B, int H,
                     int W, int IC, int OC, int32_t* Y, uint32_t* d_max);
// G[oc][(kh,kw,ic)] (rows of 9 IC) = sum over positions of E x X; max |G| into *d_max; K slices
// over the positions when ws holds conv_wgrad_s2_ws_bytes
int conv_wgrad_s2_plan(ConvIgPlan* p, const uint16_t* eb, int64_t lde, const uint16_t* xb, int64_t ldx, int B,
                       int H, int W, int IC, int OC, int32_t* G, uint32_t* d_max, int32_t* ws, size_t ws_bytes);
size_t conv_wgrad_s2_ws_bytes(int B, int H, int W, int IC, int OC);
int conv_igemm_run(const ConvIgPlan& p, cudaStream_t s);

// ---- DFP16 limb contraction (ito_dfp.cu)

// P[M][N] (int64, exact) = sum_k A(m,k) B(n,k) for int16 operands given as two
// bf16 limb planes each (value = 256 * hi + lo).
struct DfpGemmPlan {
    CUtensorMap mapAh, mapAl, mapBh, mapBl, mapC;
    int use_tma_store;
    CUtensorMap mapC8;            // the wide-tile kernel's result boxes (32 rows x 8 int64)
    int use_tma_store8;
    int M, N, K;
    int chunk_kb;                 // K blocks of 64 per exact chunk
    int pair;                     // CTA-pair kernel (256 x 64 tiles)
    int stacked;                  // wide-tile CTA-pair kernel (256 x bn4 tiles; see k_gemm_dfp4)
    int bn4;                      // its tile width: 128 or 112
    CUtensorMap mapBh3, mapBl3;   // its B maps (128-row boxes when B is K-major)
    int tail_full, tail_parts;    // pair kernel: whole tiles, K pieces per remaining tile (1: no split)
    int64_t* tail_ws;             // [pieces][256][64] int64 partials of the split tiles
    bool a_mn, b_mn;
    int64_t* C;
    int64_t ldc;
    unsigned long long* d_max;
    int* err;
    // FP32-output forward: blocked = 1 for Blocked-DFP (one exponent per chunk-long
    // block of K), 2 for the chained FP32 partial accumulation (one chain per chunk)
    int blocked;
    const int8_t* ex;             // [M][nb]
    const int8_t* ew;             // [N][nb]
    int nb;
    const int32_t* d_ex;          // chained: device exponents of the input and the weights
    const int32_t* d_ew;
    int shift;                    // chained: inputs shifted right by one bit
    float* Y;                     // [M][ldy] float output
    int64_t ldy;
};

// tail_ws (optional): room for the int64 partial tiles of a split last wave
// (dfp_split_ws_bytes); without it the pair kernel runs every tile whole.
// fill_waves: the wide-tile kernel may narrow its tiles to 112 columns so that they fill
// the last wave; false keeps 128 (a contraction with work of another stream beside it
// leaves that work the SMs of its partial last wave).
int dfp_gemm_plan(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, bool a_mn, const Bf16View& Bh,
                  const Bf16View& Bl, bool b_mn, int M, int N, int K, int64_t* C, int64_t ldc,
                  unsigned long long* d_max, int64_t* tail_ws = nullptr, size_t tail_ws_bytes = 0,
                  bool fill_waves = true);
size_t dfp_split_ws_bytes(int M, int N, int K);
// Chained FP32 partial accumulation (forward, both operands K-major): chains of `chain` K
// terms (64..512, a multiple of 64), each wrapped to int32, converted to float, scaled by
// 2^(*d_ex + shift + *d_ew) and added to Y in chain order; the A limb planes must hold the
// inputs already shifted when shift = 1
int dfp_gemm_plan_chained(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, const Bf16View& Bh,
                          const Bf16View& Bl, int M, int N, int K, int chain, const int32_t* d_ex,
                          const int32_t* d_ew, int shift, float* Y, int64_t ldy);
// Blocked-DFP forward: Y[m][n] = float(sum over K blocks j, in order, in double, of
// P_j * 2^(ex[m][j] + ew[n][j])), P_j the exact int64 sum over block j (block: 64..512, multiple of 64)
int dfp_gemm_plan_blocked(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, const Bf16View& Bh,
                          const Bf16View& Bl, int M, int N, int K, int block, const int8_t* ex, const int8_t* ew,
                          float* Y, int64_t ldy);
int dfp_gemm_run(const DfpGemmPlan& p, cudaStream_t s);

// int16 [rows][cols] -> bf16 limb planes hi/lo [rows][ldl]
int launch_i16_to_limbs(const int16_t* src, int64_t rows, int64_t cols, uint16_t* hi, uint16_t* lo, int64_t ldl,
                        cudaStream_t s, int shift = 0);
// DFP down-conversion of P with exponent *d_ea + *d_eb: Rs from *d_max,
// out16 = sat16(rhu(P, Rs)) (+ limb planes if hi != null), *d_exp_out = Ea + Eb + Rs,
// *d_rs = Rs; an exponent outside int8 raises ITO_ERR_EXPONENT in the error word.
// d_abs_sum (optional): sum of |out16| is added to it (exact).
int launch_dfp_down(const int64_t* P, int64_t rows, int64_t cols, const unsigned long long* d_max, const int32_t* d_ea,
                    const int32_t* d_eb, int16_t* out16, uint16_t* hi, uint16_t* lo, int64_t ldl, int32_t* d_exp_out,
                    int32_t* d_rs, cudaStream_t s, unsigned long long* d_abs_sum = nullptr,
                    int32_t* d_exp_out2 = nullptr);   // a second copy of the exponent
// float -> DFP16 (exponent from max |f|; d_bits: device scratch for the max's bits),
// DFP16 -> float, and float(P) * 2^(Ea + Eb)
int launch_dfp_from_float(const float* f, int64_t n, unsigned int* d_bits, int16_t* out, int32_t* d_exp,
                          cudaStream_t s);
int launch_dfp_to_float(const int16_t* m, int64_t n, const int32_t* d_exp, float* out, cudaStream_t s);
// Blocked-DFP conversions: blocks of `block` consecutive elements per row, int8 exponents [rows][nb]
int launch_bdfp_from_float(const float* f, int64_t rows, int64_t cols, int block, int16_t* out, int8_t* exps,
                           cudaStream_t s);
int launch_bdfp_to_float(const int16_t* m, const int8_t* exps, int64_t rows, int64_t cols, int block, float* out,
                         cudaStream_t s);
int launch_p64_to_float(const int64_t* P, int64_t n, const int32_t* d_ea, const int32_t* d_eb, float* out,
                        cudaStream_t s);
// W <- sat_bits(W - dW), dW = rhu(G, k) (k >= 0) or G * 2^-k (k < 0), k = exp_w + eta - *d_exp_g;
// sat_bits clamps to +-(2^(bits-1) - 1) (bits = 16: sat16)
int launch_dfp_update(int16_t* W, uint16_t* hi, uint16_t* lo, int64_t ldl, const int16_t* G, int64_t rows,
                      int64_t cols, const int32_t* d_exp_g, int32_t exp_w, int32_t eta, int32_t* d_k,
                      uint32_t* d_nonzero, cudaStream_t s, int bits = 16);
// weight precision change bits_old -> bits_new (W * 2^d, or rhu + saturation), limbs rewritten
int launch_dfp_set_bits(int16_t* W, uint16_t* hi, uint16_t* lo, int64_t ldl, int64_t rows, int64_t cols,
                        int bits_old, int bits_new, cudaStream_t s);

// split_ws (optional): room for split-K partials; without it (or when too
// small) the contraction is not split.
// chunk_terms: K terms per exact fp32 chunk (a multiple of 64, at most kExactChunk).
// min_pair_tiles: the CTA-pair kernel only when the output has at least this many 256 x 256
// tiles (below that the single-CTA kernel, with more CTAs and no cluster launch, is faster).
int gemm_plan(GemmPlan* p, const Bf16View& A, bool a_mn, const Bf16View& B, bool b_mn, int M, int N, int K,
              int32_t* C, int64_t ldc, uint32_t* d_max, int32_t* split_ws = nullptr, size_t split_ws_bytes = 0,
              int chunk_terms = kExactChunk, int min_pair_tiles = 1);
// bytes of split-K partials gemm_plan would use for this contraction (0: no split)
size_t gemm_split_ws_bytes(int M, int N, int K, int64_t ldc);
// Turns on the speculative requantisation of a planned pair-kernel contraction:
// out8 [M][ld8] int8 and outb [M][ldb] bf16 receive sat8(rhu(C, *pred)), ReLU'd if
// relu, zeroed where gate [M][ldg] <= 0 (gate may be null). Leaves the plan
// unfused (no error) when the contraction does not qualify (not the pair kernel,
// a split last wave, N or pitches not multiples of 16 bytes).
int gemm_plan_fuse_requant(GemmPlan* p, const int32_t* pred, int relu, const int8_t* gate, int64_t ldg,
                           int8_t* out8, int64_t ld8, uint16_t* outb, int64_t ldb);
int gemm_run(const GemmPlan& p, cudaStream_t s);
// C[m][n] = sum over s < splits of P[s * stride + m * ldc + n] (exact), max |C| into *d_max
int launch_splitk_reduce(const int32_t* P, int splits, int64_t stride, int M, int N, int64_t ldc, int32_t* C,
                         uint32_t* d_max, cudaStream_t s);

// ---- bandwidth kernels (ito_elementwise.cu)

// dst[r][c] (pitch dst_pitch) = bf16(src[r][c]) for a row-major int8 tensor.
int launch_i8_to_bf16(const int8_t* src, int64_t rows, int64_t cols, uint16_t* dst, int64_t dst_pitch,
                      cudaStream_t s);

// NITI Steps 1-3 on an int32 tensor Y [rows][cols] whose max |Y| is *d_max:
// out8 = sat8(rhu(Y, s)) (ReLU'd if relu), plus the bf16 copy outb (pitch
// ldb, may be null) and *d_shift = s (may be null). If gate is non-null the
// result is zeroed where gate <= 0 (delta propagation through a ReLU).
// gate_bits / mask_out (optional, cols % 8 == 0): bit-packed ReLU masks, one
// byte per 8 elements: read in place of the int8 gate / written from the result.
// s_last (optional) receives the shift as well (the next step's prediction of a speculating model)
// The top error computed beside a requantisation of the logits (labels != nullptr):
// e8 = sat_int8(q - target_mag * onehot(label)) for the requantised logits q, and its bf16
// copy eb (pitch lde) when given; a label outside [0, cols) records ITO_ERR_ARG.
struct TopErr {
    const int32_t* labels;
    int target_mag;
    int8_t* e8;
    uint16_t* eb;
    int64_t lde;
    int* err;   // set by launch_requant
};
int launch_requant(const int32_t* Y, int64_t rows, int64_t cols, const uint32_t* d_max, int target_bits, int relu,
                   const int8_t* gate, int8_t* out8, uint16_t* outb, int64_t ldb, int32_t* d_shift, cudaStream_t s,
                   const uint8_t* gate_bits = nullptr, uint8_t* mask_out = nullptr, int32_t* s_last = nullptr,
                   const TopErr* top = nullptr);
// a step's start in one kernel: stats[0..n_stats) = 0, the predictions rolled (n_pred > 0:
// the last step's scored into count[0] held / count[1] missed over the used slots, then
// pred[i] = (on && used[i]) ? last[i] : -1), and x (int8, or uint8 when x_u8) [rows][cols]
// converted to bf16 xb (pitch ldx) unless x is null
int launch_step_begin(int32_t* stats, int n_stats, int32_t* pred, const int32_t* last, const int32_t* used,
                      int64_t* count, int n_pred, int on, const void* x, int x_u8, int64_t rows, int64_t cols,
                      uint16_t* xb, int64_t ldx, cudaStream_t s);
// static per-channel requantisation: clip(floor((Y + off[c]) * mult[c] / 2^k[c]), relu ? 0 : -128, 127)
int launch_requant_static(const int32_t* Y, int64_t rows, int64_t cols, const int32_t* off, const int32_t* mult,
                          const int32_t* ksh, int relu, int8_t* out8, uint16_t* outb, int64_t ldb, uint8_t* mask_out,
                          cudaStream_t s);
// offset gradient g[c] = sum_r delta[r][c] (max |g| into *d_max), then the NITI update of the INT32 offsets
int launch_offset_grad_update(const int8_t* delta, int64_t rows, int64_t cols, int32_t* g, uint32_t* d_max,
                              int32_t* off, int target_bits, int mu_weight, int32_t* d_shift, int32_t* d_wshift,
                              uint32_t* d_nonzero, cudaStream_t s);

// NITI Steps 2-5 in place on W [rows][cols] (int8) with gradient G (int32),
// refreshing the bf16 copy Wb (pitch ldb, may be null).
int launch_niti_update(int8_t* W, uint16_t* Wb, int64_t ldb, const int32_t* G, int64_t rows, int64_t cols,
                       const uint32_t* d_max, int target_bits, int mu_weight, int32_t* d_shift, int32_t* d_wshift,
                       uint32_t* d_nonzero, cudaStream_t s);

// delta = sat8(logits - target_mag * onehot(labels)), plus bf16 copy.
int launch_top_error(const int8_t* logits, const int32_t* labels, int B, int C, int target_mag, int8_t* delta,
                     uint16_t* deltab, int64_t ldb, cudaStream_t s);

int launch_grid_blocks(int64_t work_items, int threads);

}  // namespace ito
