// Tensor-core kernels of a 3x3, stride-2, pad-1 convolution over NHWC tensors with
// even H and W ("Integer On-Device Training: Overview", section 7, Conv2D layers:
// the forward convolution, the error propagated to the input as the transposed
// convolution with the same weights, and the weight gradient as the correlation of
// the input with the output error), without materialised patches.
//
// Input row y and output row oh meet through kernel row kh exactly when
// y = 2 oh + kh - 1, and so for columns. Split the input into its four parity
// planes X_(py,px)[b][i][j] = x[b][2i+py][2j+px] (i < OH = H/2, j < OW = W/2):
// kernel row kh reads plane row py = (kh + 1) mod 2 at i = oh - 1 (kh = 0) or
// i = oh (kh = 1, 2); columns alike. A 4-D tensor map over one plane of the bf16
// NHWC activation (base offset by the plane, strides of two rows and two columns)
// then gives every tap's operand tile as one TMA box at a shift of -1 or 0, the
// part outside the plane read as 0: the forward and weight-gradient contractions
// take their patch operand straight from the activation (k_conv_igemm).
//
// For the propagated error the same relation read the other way: write
// y = 2 i + py; then
//   py = 0: kh = 1 with oh = i;
//   py = 1: kh = 0 with oh = i + 1, and kh = 2 with oh = i;
// and the same for columns (x = 2 j + px, kernel column kw, output column ow).
// So each of the four phases (py, px) of the input-space delta is a plain
// contraction over the output positions (b, i, j):
//   D[b][2i+py][2j+px][ic] = sum over the phase's taps (dh, kh) x (dw, kw) and oc of
//                            E[b][i+dh][j+dw][oc] * W[oc][kh][kw][ic]
// (E outside the output grid is 0), with 1, 2, 2 or 4 taps. The A operand is a 4-D
// TMA box of the delta's bf16 copy E [B][OH][OW][OC] at the tap's shift (the box
// reads 0 past the edge); the B operand is the weights' bf16 copy [OC][3][3][IC]
// read MN-major at the tap's columns; the int32 result goes straight to D through a
// 4-D tensor map over the phase's rows and columns of D (every other row and column,
// base offset by the phase), so no patch-space delta is formed and no gather pass
// follows (k_conv_dgrad_s2).
//
// All three contractions are exact as in the GEMM kernels (bf16 operands holding
// int8 values, fp32 tensor-memory accumulators drained into int32 every 1024
// terms), and fold max |result| into the NITI max word.
#include <cstdio>

#include <cudaTypedefs.h>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

#define IG_TRY(x)                    \
    do {                             \
        int _r = (x);                \
        if (_r != ITO_OK) return _r; \
    } while (0)

// Tiles of all three kernels: 128 rows x BN (64 or 128) columns of the result, K blocks of
// 64 terms. These contractions are paced by their operand loads (a few K blocks of 4-D
// boxes per tile), so where the result has a multiple of 128 columns the wider tile, which
// loads each A tile once for twice the columns, is taken.
template <int BN_>
struct S2Cfg {
    static constexpr int BM = 128, BN = BN_, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;       // 16 KB: 128 rows x 64 K terms (bf16)
    static constexpr int B_BYTES = BN * BK * 2;       // 8 or 16 KB: BN columns x 64 K terms
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 6;
    static constexpr int EPI_WARPS = 8;               // 4 lane quarters x 2 column halves of BN / 2
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int TMEM_COLS = 2 * BN;          // two accumulators
    static constexpr int CHUNK_KB = 1024 / BK;        // exact chunk: 1024 terms
    static constexpr int STAGING_BYTES = EPI_WARPS * 4096;   // one 32 x 32 int32 box per epilogue warp
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
};
static_assert(S2Cfg<64>::SMEM_BYTES <= 227 * 1024 && S2Cfg<128>::SMEM_BYTES <= 227 * 1024,
              "conv kernels: shared memory above the per-CTA limit");

// The phases in the order their tiles are handed out (most taps first): (py, px).
__device__ __forceinline__ void s2_phase(int po, int& py, int& px)
{
    py = po == 3 ? 0 : (po == 2 ? 0 : 1);
    px = po == 3 ? 0 : (po == 1 ? 0 : 1);
}

// Tap t of a phase: the shift (dh, dw) of the delta and the kernel position (kh, kw).
// Rows of phase py: py = 0 -> {(0, 1)}; py = 1 -> {(1, 0), (0, 2)}; columns alike.
__device__ __forceinline__ void s2_tap(int py, int px, int t, int& dh, int& kh, int& dw, int& kw)
{
    const int nx = px ? 2 : 1;
    const int ty = t / nx, tx = t - ty * nx;
    dh = py ? (ty == 0 ? 1 : 0) : 0;
    kh = py ? (ty == 0 ? 0 : 2) : 1;
    dw = px ? (tx == 0 ? 1 : 0) : 0;
    kw = px ? (tx == 0 ? 0 : 2) : 1;
}

template <int BN_>
__global__ void __launch_bounds__(S2Cfg<BN_>::THREADS, 1)
    k_conv_dgrad_s2(const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmD0, const __grid_constant__ CUtensorMap tmD1,
                    const __grid_constant__ CUtensorMap tmD2, const __grid_constant__ CUtensorMap tmD3, S2Geom g,
                    uint32_t* __restrict__ d_max, int* __restrict__ err)
{
    using Cfg = S2Cfg<BN_>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;   // [2]
    uint64_t* acce_bar = accf_bar + 2;         // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int per_phase = g.m_tiles * g.n_tiles;
    const int num_items = 4 * per_phase;
    // item w: phase po, row tile mt (a block of ba images x oha output rows, all columns), column tile nt
    auto item = [&](int w, int& py, int& px, int& b0, int& i0, int& nt) {
        const int po = w / per_phase;
        const int r = w - po * per_phase;
        const int mt = r / g.n_tiles;
        nt = r - mt * g.n_tiles;
        s2_phase(po, py, px);
        const int ib = mt % g.n_iblk;
        b0 = (mt / g.n_iblk) * g.ba;
        i0 = ib * g.oha;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], Cfg::EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmE);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // on-chip setup above overlaps the previous kernel; global memory only from here on
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
                int py, px, b0, i0, nt;
                item(w, py, px, b0, i0, nt);
                const int ntaps = (py ? 2 : 1) * (px ? 2 : 1);
                for (int kb = 0; kb < ntaps * g.oc_blocks; ++kb) {
                    const int t = kb / g.oc_blocks, ocb = kb - t * g.oc_blocks;
                    int dh, kh, dw, kw;
                    s2_tap(py, px, t, dh, kh, dw, kw);
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
                    uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sB = sA + Cfg::A_BYTES;
                    // E[b0.., i0 + dh.., dw.., ocb * 64..]: 128 rows of 128 bytes (0 past the grid)
                    tma_load_4d(&tmE, &full_bar[stage], sA, ocb * 64, dw, i0 + dh, b0);
                    // W[oc][kh][kw][ic] as [OC][9 IC], MN-major: rows ocb * 64.., columns tap * IC + nt * BN..
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(&tmW, &full_bar[stage], sB + j * 8192, (kh * 3 + kw) * g.IC + nt * BN + j * 64,
                                    ocb * 64);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
                int py, px, b0, i0, nt;
                item(w, py, px, b0, i0, nt);
                const int nkb = (py ? 2 : 1) * (px ? 2 : 1) * g.oc_blocks;
                for (int kb0 = 0; ok && kb0 < nkb; kb0 += Cfg::CHUNK_KB) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb1 = min(nkb, kb0 + Cfg::CHUNK_KB);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t b0s = a0 + Cfg::A_BYTES;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ad = smem_desc_sw128(a0 + k * 32, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(b0s + k * 2048, 8192, 1024);
                            tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        tc_commit(&empty_bar[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit(&accf_bar[buf]);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
        }
    } else {
        // ---------------- epilogue: drain into int32, max, store through the phase's map
        const int e = warp - 2;
        const int quad = warp & 3;               // TMEM lanes this warp may access
        const int half = e >> 2;                 // which half (BN / 2 columns) of the tile
        uint8_t* stg = staging + e * 4096;       // this warp's 32 x 32 int32 store box
        const uint32_t stg_row = smem_u32(stg) + lane * 128;
        // this warp's 32 rows of the tile: (32 / OW) output rows of one image
        const int r0 = quad * 32;
        const int b_off = r0 / (g.oha * g.OW);
        const int i_off = (r0 - b_off * g.oha * g.OW) / g.OW;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
            int py, px, b0, i0, nt;
            item(w, py, px, b0, i0, nt);
            const int nkb = (py ? 2 : 1) * (px ? 2 : 1) * g.oc_blocks;
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int kb0 = 0; kb0 < nkb; kb0 += Cfg::CHUNK_KB) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + half * HALF);
#pragma unroll
                for (int j = 0; j < HALF / 16; ++j) {
                    uint32_t r[16];
                    tmem_ld16(taddr + j * 16, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[j * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce_bar[buf]);
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            // rows past the batch read zero-filled operands and hold 0
            uint32_t mx = 0;
#pragma unroll
            for (int i = 0; i < HALF; ++i) mx = max(mx, abs_u32(acc[i]));
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            const int b = b0 + b_off;
            if (b >= g.B) continue;
            // 32 x 32 boxes (128-byte swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8))
#pragma unroll
            for (int gq = 0; gq < HALF / 32; ++gq) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), acc[gq * 32 + 4 * j], acc[gq * 32 + 4 * j + 1],
                                 acc[gq * 32 + 4 * j + 2], acc[gq * 32 + 4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const CUtensorMap* tmD = py ? (px ? &tmD3 : &tmD2) : (px ? &tmD1 : &tmD0);
                    tma_store_4d(tmD, stg, nt * BN + half * HALF + gq * 32, 0, i0 + i_off, b);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

bool conv_dgrad_s2_eligible(int B, int H, int W, int IC, int OC, int stride)
{
    if (stride != 2 || H % 2 || W % 2 || B < 1) return false;
    const int OH = H / 2, OW = W / 2;
    auto pow2 = [](int v) { return v > 0 && (v & (v - 1)) == 0; };
    // a warp's 32 rows are whole output rows of one image; a tile's 128 rows whole rows of
    // whole images or of one image
    return (OW == 8 || OW == 16 || OW == 32) && pow2(OH) && OH * OW >= 32 && IC % 64 == 0 && OC % 64 == 0 &&
           OC <= (1 << 16);
}

int conv_dgrad_s2_plan(ConvS2Plan* p, const uint16_t* eb, int64_t lde, const uint16_t* Wb, int64_t ldw, int B,
                       int H, int W, int IC, int OC, int32_t* D, uint32_t* d_max)
{
    if (!conv_dgrad_s2_eligible(B, H, W, IC, OC, 2))
        return set_error(ITO_ERR_UNSUPPORTED, "stride-2 phase delta propagation: unsupported shape");
    if ((reinterpret_cast<uintptr_t>(eb) & 15) || (reinterpret_cast<uintptr_t>(Wb) & 15) ||
        (reinterpret_cast<uintptr_t>(D) & 15) || (lde * 2) % 16 || (ldw * 2) % 16)
        return set_error(ITO_ERR_ARG, "stride-2 phase delta propagation: operands not 16-byte aligned");
    auto enc = get_encode();
    if (!enc) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    *p = ConvS2Plan{};
    S2Geom& g = p->g;
    g.B = B;
    g.OH = H / 2;
    g.OW = W / 2;
    g.IC = IC;
    g.oc_blocks = OC / 64;
    p->bn = IC % 128 == 0 ? 128 : 64;
    g.n_tiles = IC / p->bn;
    g.oha = g.OH < 128 / g.OW ? g.OH : 128 / g.OW;
    g.ba = 128 / (g.OW * g.oha);
    g.n_iblk = g.OH / g.oha;
    g.m_tiles = ((B + g.ba - 1) / g.ba) * g.n_iblk;
    p->d_max = d_max;
    p->err = device_error_word();
    if (!p->err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    cuuint32_t estr[4] = {1, 1, 1, 1};
    {
        // E [B][OH][OW][OC] (rows of lde): boxes of 64 channels x OW x oha x ba
        cuuint64_t dims[4] = {(cuuint64_t)OC, (cuuint64_t)g.OW, (cuuint64_t)g.OH, (cuuint64_t)B};
        cuuint64_t strides[3] = {(cuuint64_t)lde * 2, (cuuint64_t)g.OW * lde * 2, (cuuint64_t)g.OH * g.OW * lde * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)g.OW, (cuuint32_t)g.oha, (cuuint32_t)g.ba};
        CUresult r = enc(&p->mapE, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(eb), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (delta, 4-D) failed (%d)", (int)r);
    }
    // W [OC][9 IC] read MN-major (64 x 64 boxes)
    int r = make_map_bf16(&p->mapW, Bf16View{Wb, OC, 9 * (int64_t)IC, ldw}, 64);
    if (r) return r;
    for (int ph = 0; ph < 4; ++ph) {
        // phase (py, px) = (ph >> 1, ph & 1) of D [B][H][W][IC]: rows 2i + py, columns 2j + px
        const int py = ph >> 1, px = ph & 1;
        int32_t* base = D + ((int64_t)py * W + px) * IC;
        cuuint64_t dims[4] = {(cuuint64_t)IC, (cuuint64_t)g.OW, (cuuint64_t)g.OH, (cuuint64_t)B};
        cuuint64_t strides[3] = {(cuuint64_t)2 * IC * 4, (cuuint64_t)2 * W * IC * 4, (cuuint64_t)H * W * IC * 4};
        cuuint32_t box[4] = {32, (cuuint32_t)g.OW, (cuuint32_t)(32 / g.OW), 1};
        CUresult cr = enc(&p->mapD[ph], CU_TENSOR_MAP_DATA_TYPE_INT32, 4, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS)
            return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (delta phase %d) failed (%d)", ph, (int)cr);
    }
    return ITO_OK;
}

template <int BN>
static int launch_dgrad_s2(const ConvS2Plan& p, cudaStream_t s)
{
    using Cfg = S2Cfg<BN>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(k_conv_dgrad_s2<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
            cudaSuccess)
            return set_error(ITO_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(cudaGetLastError()));
        attr_set = true;
    }
    const int items = 4 * p.g.m_tiles * p.g.n_tiles;
    const int grid = items < num_sms() ? items : num_sms();
    launch_pdl(k_conv_dgrad_s2<BN>, grid, Cfg::THREADS, Cfg::SMEM_BYTES, s, p.mapE, p.mapW, p.mapD[0], p.mapD[1],
               p.mapD[2], p.mapD[3], p.g, p.d_max, p.err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK
                            : set_error(ITO_ERR_CUDA, "stride-2 delta propagation launch: %s", cudaGetErrorString(e));
}

int conv_dgrad_s2_run(const ConvS2Plan& p, cudaStream_t s)
{
    return p.bn == 128 ? launch_dgrad_s2<128>(p, s) : launch_dgrad_s2<64>(p, s);
}

// ------------------------------------------------ forward and weight gradient

// Tap (kh, kw) of the forward reads parity plane (py, px) at shift (sh, sw).
__device__ __forceinline__ void ig_tap(int tap, int& plane, int& sh, int& sw)
{
    const int kh = tap / 3, kw = tap - kh * 3;
    plane = ((kh + 1) & 1) * 2 + ((kw + 1) & 1);
    sh = kh == 0 ? -1 : 0;
    sw = kw == 0 ? -1 : 0;
}

// FWD: Y[(b,oh,ow)][oc] = sum over taps and ic of X[b][2oh+kh-1][2ow+kw-1][ic] W[oc][kh][kw][ic].
//   Items: row tiles of 128 output positions x BN output channels; K = 9 taps x IC.
//   A: the tap's plane box {64 ic, OW, oha, ba}; B: W [OC][9 IC] K-major (BN rows); out: 2-D
//   map over Y.
// WGRAD: G[oc][(kh,kw,ic)] = sum over positions (b,oh,ow) of E[(b,oh,ow)][oc] X[b][2oh+kh-1][2ow+kw-1][ic].
//   Items: tiles of 128 output channels x BN columns (a tap's input channels, 64 or 128) x K slice;
//   K = positions in blocks of 64 (bb images x ohb rows x OW). A: E [positions][OC] MN-major;
//   B: per 64 columns the tap's plane box {64 ic, OW, ohb, bb} (MN-major: 64 positions of 128
//   bytes); out: G,
//   or with several slices their int32 partials [slice][OC][9 IC] (3-D map, no max) for
//   launch_splitk_reduce.
template <int MODE, int BN_>
__global__ void __launch_bounds__(S2Cfg<BN_>::THREADS, 1)
    k_conv_igemm(const __grid_constant__ CUtensorMap tmX0, const __grid_constant__ CUtensorMap tmX1,
                 const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmX3,
                 const __grid_constant__ CUtensorMap tmOp, const __grid_constant__ CUtensorMap tmOut, IgGeom g,
                 uint32_t* __restrict__ d_max, int* __restrict__ err)
{
    using Cfg = S2Cfg<BN_>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;
    constexpr bool W_ = MODE == CONV_WGRAD;
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, W_, W_);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;   // [2]
    uint64_t* acce_bar = accf_bar + 2;         // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_items = W_ ? g.m_tiles * g.n_tiles * g.splits : g.m_tiles * g.n_tiles;
    // item w: output tile (mt, nt) and, for the weight gradient, K blocks [kb_lo, kb_hi)
    auto item = [&](int w, int& mt, int& nt, int& kb_lo, int& kb_hi) {
        int t = w;
        int sl = 0;
        if (W_) {
            sl = w % g.splits;
            t = w / g.splits;
        }
        mt = t / g.n_tiles;
        nt = t - mt * g.n_tiles;
        kb_lo = W_ ? sl * g.kb_per_split : 0;
        kb_hi = W_ ? min(g.num_kb, kb_lo + g.kb_per_split) : g.num_kb;
    };
    auto plane_map = [&](int plane) -> const CUtensorMap* {
        return plane == 0 ? &tmX0 : (plane == 1 ? &tmX1 : (plane == 2 ? &tmX2 : &tmX3));
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], Cfg::EPI_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmOp);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // on-chip setup above overlaps the previous kernel; global memory only from here on
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
                int mt, nt, kb_lo, kb_hi;
                item(w, mt, nt, kb_lo, kb_hi);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
                    uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sB = sA + Cfg::A_BYTES;
                    int plane, sh, sw;
                    if (!W_) {
                        // A: the tap's plane at the row tile; B: W rows nt * BN.., K columns tap * IC + icb * 64
                        const int tap = kb / g.ic_blocks, icb = kb - tap * g.ic_blocks;
                        ig_tap(tap, plane, sh, sw);
                        const int b0 = (mt / g.n_iblk) * g.ba, i0 = (mt % g.n_iblk) * g.oha;
                        tma_load_4d(plane_map(plane), &full_bar[stage], sA, icb * 64, sw, i0 + sh, b0);
                        tma_load_2d(&tmOp, &full_bar[stage], sB, tap * g.IC + icb * 64, nt * BN);
                    } else {
                        // A: E positions kb * 64.., channels mt * 128..; B: for each 64 of the tile's
                        // columns (a tap's input channels), that tap's plane at position block kb
                        const int b0 = (kb / g.n_iblk_w) * g.bb, i0 = (kb % g.n_iblk_w) * g.ohb;
                        tma_load_2d(&tmOp, &full_bar[stage], sA, mt * BM, kb * 64);
                        tma_load_2d(&tmOp, &full_bar[stage], sA + 8192, mt * BM + 64, kb * 64);
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j) {
                            const int c = nt * BN + j * 64;
                            const int tap = c / g.IC, icb = (c - tap * g.IC) / 64;
                            ig_tap(tap, plane, sh, sw);
                            tma_load_4d(plane_map(plane), &full_bar[stage], sB + j * 8192, icb * 64, sw, i0 + sh, b0);
                        }
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
                int mt, nt, kb_lo, kb_hi;
                item(w, mt, nt, kb_lo, kb_hi);
                for (int kb0 = kb_lo; ok && kb0 < kb_hi; kb0 += Cfg::CHUNK_KB) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb1 = min(kb_hi, kb0 + Cfg::CHUNK_KB);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t b0s = a0 + Cfg::A_BYTES;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // K-major: the 16-element K step is 32 bytes inside the swizzled row;
                            // MN-major: it is 16 rows of 128 bytes
                            const uint64_t ad = W_ ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                                   : smem_desc_sw128(a0 + k * 32, 16, 1024);
                            const uint64_t bd = W_ ? smem_desc_sw128(b0s + k * 2048, 8192, 1024)
                                                   : smem_desc_sw128(b0s + k * 32, 16, 1024);
                            tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        tc_commit(&empty_bar[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit(&accf_bar[buf]);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
        }
    } else {
        // ---------------- epilogue: drain into int32, max, one 32 x 32 box through TMA
        const int e = warp - 2;
        const int quad = warp & 3;               // TMEM lanes this warp may access
        const int half = e >> 2;                 // which half (BN / 2 columns) of the tile
        uint8_t* stg = staging + e * 4096;
        const uint32_t stg_row = smem_u32(stg) + lane * 128;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
            int mt, nt, kb_lo, kb_hi;
            item(w, mt, nt, kb_lo, kb_hi);
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int kb0 = kb_lo; kb0 < kb_hi; kb0 += Cfg::CHUNK_KB) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + half * HALF);
#pragma unroll
                for (int j = 0; j < HALF / 16; ++j) {
                    uint32_t r[16];
                    tmem_ld16(taddr + j * 16, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[j * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce_bar[buf]);
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            // rows and columns outside the result read zero-filled operands and hold 0
            const bool partial = W_ && g.splits > 1;
            if (!partial) {
                uint32_t mx = 0;
#pragma unroll
                for (int i = 0; i < HALF; ++i) mx = max(mx, abs_u32(acc[i]));
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            }
            // forward: rows are positions (the row tile's 128 are consecutive), columns output
            // channels; weight gradient: rows output channels, columns tap * IC + input channel
            const int row = W_ ? mt * BM + quad * 32 : ((mt / g.n_iblk) * g.ba * g.OH + (mt % g.n_iblk) * g.oha) * g.OW + quad * 32;
            const int col = nt * BN + half * HALF;
            if (row >= g.rows) continue;
#pragma unroll
            for (int gq = 0; gq < HALF / 32; ++gq) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), acc[gq * 32 + 4 * j], acc[gq * 32 + 4 * j + 1],
                                 acc[gq * 32 + 4 * j + 2], acc[gq * 32 + 4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (partial)
                        tma_store_3d(&tmOut, stg, col + gq * 32, row, w % g.splits);
                    else
                        tma_store_2d(&tmOut, stg, col + gq * 32, row);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// The four parity-plane maps of a bf16 NHWC activation X [B][H][W][ldx] (IC used), boxes of
// 64 channels x OW x rows x images.
static int plane_maps(CUtensorMap* maps, const uint16_t* xb, int64_t ldx, int B, int H, int W, int IC, int rows,
                      int imgs)
{
    auto enc = get_encode();
    if (!enc) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const int OH = H / 2, OW = W / 2;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    for (int pl = 0; pl < 4; ++pl) {
        const int py = pl >> 1, px = pl & 1;
        const uint16_t* base = xb + ((int64_t)py * W + px) * ldx;
        cuuint64_t dims[4] = {(cuuint64_t)IC, (cuuint64_t)OW, (cuuint64_t)OH, (cuuint64_t)B};
        cuuint64_t strides[3] = {(cuuint64_t)2 * ldx * 2, (cuuint64_t)2 * W * ldx * 2, (cuuint64_t)H * W * ldx * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)OW, (cuuint32_t)rows, (cuuint32_t)imgs};
        CUresult r = enc(&maps[pl], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(base), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (activation plane %d) failed (%d)", pl, (int)r);
    }
    return ITO_OK;
}

static int int32_out_map(CUtensorMap* map, int32_t* C, int rows, int cols, int64_t ldc)
{
    auto enc = get_encode();
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ldc * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, C, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ITO_OK : set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (int32 out) failed (%d)", (int)r);
}

static int ig_check(const uint16_t* xb, int64_t ldx, int B, int H, int W, int IC, int OC)
{
    if (!conv_dgrad_s2_eligible(B, H, W, IC, OC, 2))
        return set_error(ITO_ERR_UNSUPPORTED, "stride-2 conv on parity planes: unsupported shape");
    if ((reinterpret_cast<uintptr_t>(xb) & 15) || (ldx * 2) % 16 || ldx < IC)
        return set_error(ITO_ERR_ARG, "stride-2 conv on parity planes: activation not 16-byte aligned");
    return ITO_OK;
}

static void ig_geom(IgGeom& g, int B, int H, int W, int IC)
{
    g.B = B;
    g.OH = H / 2;
    g.OW = W / 2;
    g.IC = IC;
    g.ic_blocks = IC / 64;
    g.oha = g.OH < 128 / g.OW ? g.OH : 128 / g.OW;
    g.ba = 128 / (g.OW * g.oha);
    g.n_iblk = g.OH / g.oha;
    g.ohb = g.OH < 64 / g.OW ? g.OH : 64 / g.OW;
    g.bb = 64 / (g.OW * g.ohb);
    g.n_iblk_w = g.OH / g.ohb;
}

int conv_fwd_s2_plan(ConvIgPlan* p, const uint16_t* xb, int64_t ldx, const uint16_t* Wb, int64_t ldw, int B, int H,
                     int W, int IC, int OC, int32_t* Y, uint32_t* d_max)
{
    IG_TRY(ig_check(xb, ldx, B, H, W, IC, OC));
    if ((reinterpret_cast<uintptr_t>(Wb) & 15) || (ldw * 2) % 16 || (reinterpret_cast<uintptr_t>(Y) & 15) || OC % 4)
        return set_error(ITO_ERR_ARG, "stride-2 conv forward: operands not 16-byte aligned");
    *p = ConvIgPlan{};
    p->mode = CONV_FWD;
    IgGeom& g = p->g;
    ig_geom(g, B, H, W, IC);
    g.m_tiles = ((B + g.ba - 1) / g.ba) * g.n_iblk;
    p->bn = OC % 128 == 0 ? 128 : 64;
    g.n_tiles = OC / p->bn;
    g.num_kb = 9 * g.ic_blocks;
    g.splits = 1;
    g.kb_per_split = g.num_kb;
    g.rows = B * g.OH * g.OW;
    p->d_max = d_max;
    p->err = device_error_word();
    if (!p->err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    IG_TRY(plane_maps(p->mapX, xb, ldx, B, H, W, IC, g.oha, g.ba));
    IG_TRY(make_map_bf16(&p->mapOp, Bf16View{Wb, OC, 9 * (int64_t)IC, ldw}, p->bn));
    return int32_out_map(&p->mapOut, Y, g.rows, OC, OC);
}

size_t conv_wgrad_s2_ws_bytes(int B, int H, int W, int IC, int OC)
{
    if (!conv_dgrad_s2_eligible(B, H, W, IC, OC, 2)) return 0;
    IgGeom g;
    ig_geom(g, B, H, W, IC);
    const int tiles = ((OC + 127) / 128) * (9 * IC / (IC % 128 == 0 ? 128 : 64));
    const int num_kb = (B + g.bb - 1) / g.bb * g.n_iblk_w;
    int splits = num_sms() / tiles;
    if (splits > num_kb) splits = num_kb;
    if (splits < 2) return 0;
    return (size_t)splits * OC * 9 * IC * sizeof(int32_t);
}

int conv_wgrad_s2_plan(ConvIgPlan* p, const uint16_t* eb, int64_t lde, const uint16_t* xb, int64_t ldx, int B,
                       int H, int W, int IC, int OC, int32_t* G, uint32_t* d_max, int32_t* ws, size_t ws_bytes)
{
    IG_TRY(ig_check(xb, ldx, B, H, W, IC, OC));
    if ((reinterpret_cast<uintptr_t>(eb) & 15) || (lde * 2) % 16 || (reinterpret_cast<uintptr_t>(G) & 15))
        return set_error(ITO_ERR_ARG, "stride-2 conv weight gradient: operands not 16-byte aligned");
    *p = ConvIgPlan{};
    p->mode = CONV_WGRAD;
    IgGeom& g = p->g;
    ig_geom(g, B, H, W, IC);
    const int K9 = 9 * IC;
    g.m_tiles = (OC + 127) / 128;
    p->bn = IC % 128 == 0 ? 128 : 64;   // a 128-column tile: one tap's 128 input channels
    g.n_tiles = K9 / p->bn;
    // position blocks of 64 (whole rows of one image, or whole images), in flat position order
    g.num_kb = (B + g.bb - 1) / g.bb * g.n_iblk_w;
    g.rows = OC;
    // K slices: enough work items to cover the SMs when the workspace holds their partials
    int splits = num_sms() / (g.m_tiles * g.n_tiles);
    if (splits > g.num_kb) splits = g.num_kb;
    if (splits < 2 || !ws || ws_bytes < (size_t)splits * OC * K9 * sizeof(int32_t)) splits = 1;
    g.kb_per_split = (g.num_kb + splits - 1) / splits;
    g.splits = (g.num_kb + g.kb_per_split - 1) / g.kb_per_split;
    p->d_max = d_max;
    p->err = device_error_word();
    if (!p->err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    p->G = G;
    p->ws = ws;
    p->OC = OC;
    p->K9 = K9;
    IG_TRY(plane_maps(p->mapX, xb, ldx, B, H, W, IC, g.ohb, g.bb));
    // E [positions][OC] read MN-major: boxes of 64 channels x 64 positions
    IG_TRY(make_map_bf16(&p->mapOp, Bf16View{eb, (int64_t)B * g.OH * g.OW, OC, lde}, 64));
    if (g.splits == 1) return int32_out_map(&p->mapOut, G, OC, K9, K9);
    auto enc = get_encode();
    cuuint64_t dims[3] = {(cuuint64_t)K9, (cuuint64_t)OC, (cuuint64_t)g.splits};
    cuuint64_t strides[2] = {(cuuint64_t)K9 * 4, (cuuint64_t)OC * K9 * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&p->mapOut, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, ws, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ITO_OK : set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (partials) failed (%d)", (int)r);
}

template <int MODE, int BN>
static int launch_igemm(const ConvIgPlan& p, cudaStream_t s)
{
    using Cfg = S2Cfg<BN>;
    auto kern = k_conv_igemm<MODE, BN>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(cudaGetLastError()));
        attr_set = true;
    }
    const int items = p.g.m_tiles * p.g.n_tiles * p.g.splits;
    const int grid = items < num_sms() ? items : num_sms();
    const bool partial = MODE == CONV_WGRAD && p.g.splits > 1;
    launch_pdl(kern, grid, Cfg::THREADS, Cfg::SMEM_BYTES, s, p.mapX[0], p.mapX[1], p.mapX[2], p.mapX[3], p.mapOp,
               p.mapOut, p.g, partial ? nullptr : p.d_max, p.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "stride-2 conv launch: %s", cudaGetErrorString(e));
    if (partial)
        return launch_splitk_reduce(p.ws, p.g.splits, (int64_t)p.OC * p.K9, p.OC, p.K9, p.K9, p.G, p.d_max, s);
    return ITO_OK;
}

int conv_igemm_run(const ConvIgPlan& p, cudaStream_t s)
{
    if (p.mode == CONV_WGRAD)
        return p.bn == 128 ? launch_igemm<CONV_WGRAD, 128>(p, s) : launch_igemm<CONV_WGRAD, 64>(p, s);
    return p.bn == 128 ? launch_igemm<CONV_FWD, 128>(p, s) : launch_igemm<CONV_FWD, 64>(p, s);
}

}  // namespace ito
