// DFP16 (dynamic fixed point, one shared exponent per tensor) linear path
// ("Mixed Precision Training of Convolutional Neural Networks using Integer
// Operations", section 3 "The Dynamic Fixed Point Format" and 3.1 "DFP
// Tensor Primitives": a tensor is an int16 mantissa tensor i with one shared
// signed 8-bit exponent E, value i * 2^E; a product tensor carries exponent
// Ea + Eb and its accumulation chain shares it; down-conversion right-shifts
// the wide result by Rs and adds Rs to the exponent).
//
// Contraction: int16 x int16 products summed exactly in int64. Each int16 v is
// split into balanced limbs v = 256 * h + l with l in [-128, 127] and h in
// [-128, 128]; both are exact in bf16. Then
//   sum v*w = 65536 * sum(h_v h_w) + 256 * sum(h_v l_w + l_v h_w) + sum(l_v l_w),
// four limb products into three fp32 accumulators (hh, mid, ll) laid side by
// side in tensor memory, issued as two tensor-core MMAs of twice the tile
// width: h_v x [h_w | l_w] into [hh | mid] and l_v x [h_w | l_w] into [mid | ll].
// Every limb product is at most 2^14 in magnitude, so over a chunk of 512 K
// terms each accumulator stays within 2^24 (the middle one gets two products
// per term) and holds an exact integer. After each chunk the epilogue combines
// the three into an exact int64 partial sum in registers; the tile's int64
// result and its max |P| (atomicMax) go to global memory.
#include <cstdlib>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

struct DfpCfg {
    static constexpr int BM = 128, BN = 64, BK = 64;
    static constexpr int A_PLANE = BM * BK * 2;             // 16 KB per limb plane
    static constexpr int B_PLANE = BN * BK * 2;             // 8 KB per limb plane
    static constexpr int STAGE_BYTES = 2 * A_PLANE + 2 * B_PLANE;
    static constexpr int STAGES = 4;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int BUF_COLS = 256;                    // per accumulator buffer: hh, mid, ll at +0, +64, +128
    static constexpr int TMEM_COLS = 512;
    static constexpr int CHUNK_KB = 512 / BK;               // exact chunk: 512 K terms
    static constexpr int STAGING_BYTES = EPI_WARPS * 4096;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
};

__device__ __forceinline__ void limb_split(int32_t v, int32_t& h, int32_t& l)
{
    l = ((v + 128) & 255) - 128;
    h = (v - l) >> 8;   // v - l is a multiple of 256
}

// 2^k as a double (k in [-1022, 1023]): scaling by it is exact, so converting the
// product to float or int rounds once, like ldexpf
__device__ __forceinline__ double pow2d(int k) { return __longlong_as_double((long long)(k + 1023) << 52); }

// Drain modes of the limb kernel. DFP_EXACT: the tile's exact int64 sums go to C.
// The two FP32-output modes write the tile as float (Y) instead:
// DFP_BLOCKED (Blocked-DFP operands): the exact chunk is one exponent block of
//   the contraction; after each chunk the epilogue scales its exact int64
//   partial by 2^(ex[row][chunk] + ew[col][chunk]) and adds it in double.
// DFP_CHAINED (the FP32 partial accumulation of "Mixed Precision Training...",
//   section 4, "Handling overflows"): the exact chunk is one accumulation chain;
//   its sum is taken modulo 2^32 as an INT32 accumulator would hold it, converted
//   to float, scaled by 2^(*d_ex + shift + *d_ew) (exact in double, rounded once
//   to float) and added to the float output in chain order.
enum DfpDrain { DFP_EXACT = 0, DFP_BLOCKED = 1, DFP_CHAINED = 2 };

struct DfpF32Out {
    const int8_t* ex;     // DFP_BLOCKED: [M][nb]
    const int8_t* ew;     // DFP_BLOCKED: [N][nb]
    int nb;
    const int32_t* d_ex;  // DFP_CHAINED: input and weight exponents (device scalars)
    const int32_t* d_ew;
    int shift;            // DFP_CHAINED: 1 when the inputs were shifted right by one bit
    float* Y;             // [M][ldy]
    int64_t ldy;
};

template <bool A_MN, bool B_MN, int MODE>
__global__ void __launch_bounds__(DfpCfg::THREADS, 1)
    k_gemm_dfp(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
               const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
               const __grid_constant__ CUtensorMap tmC, int use_tma_store, int M, int N, int K, int chunk_kb,
               int64_t* __restrict__ C, int64_t ldc, unsigned long long* __restrict__ d_max, DfpF32Out bk,
               int* __restrict__ err)
{
    using Cfg = DfpCfg;
    constexpr bool F32OUT = MODE != DFP_EXACT;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;                        // 32 columns per epilogue warp
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
    // the two B limb planes are adjacent in shared memory, so [B_hi | B_lo] is one N = 2 * BN operand
    constexpr uint32_t IDESC2 = idesc_bf16_f32(BM, 2 * BN, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;
    uint64_t* acce_bar = accf_bar + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    const int num_kb = (K + BK - 1) / BK;
    const int num_chunks = (num_kb + chunk_kb - 1) / chunk_kb;

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

    // tiles in row-major order over (m, n): consecutive CTAs share the A band
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                const int tm = t / num_n, tn = t % num_n;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
                    uint8_t* sAh = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sAl = sAh + Cfg::A_PLANE;
                    uint8_t* sBh = sAl + Cfg::A_PLANE;
                    uint8_t* sBl = sBh + Cfg::B_PLANE;
                    if (!A_MN) {
                        tma_load_2d(&tmAh, &full_bar[stage], sAh, kb * BK, tm * BM);
                        tma_load_2d(&tmAl, &full_bar[stage], sAl, kb * BK, tm * BM);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j) {
                            tma_load_2d(&tmAh, &full_bar[stage], sAh + j * 8192, tm * BM + j * 64, kb * BK);
                            tma_load_2d(&tmAl, &full_bar[stage], sAl + j * 8192, tm * BM + j * 64, kb * BK);
                        }
                    }
                    if (!B_MN) {
                        tma_load_2d(&tmBh, &full_bar[stage], sBh, kb * BK, tn * BN);
                        tma_load_2d(&tmBl, &full_bar[stage], sBl, kb * BK, tn * BN);
                    } else {
                        tma_load_2d(&tmBh, &full_bar[stage], sBh, tn * BN, kb * BK);
                        tma_load_2d(&tmBl, &full_bar[stage], sBl, tn * BN, kb * BK);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                for (int c = 0; ok && c < num_chunks; ++c) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_hh = tmem_base + (uint32_t)(buf * Cfg::BUF_COLS);
                    const uint32_t d_mid = d_hh + 64, d_ll = d_hh + 128;
                    const int kb0 = c * chunk_kb;
                    const int kb1 = min(num_kb, kb0 + chunk_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ah0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t al0 = ah0 + Cfg::A_PLANE;
                        const uint32_t bh0 = al0 + Cfg::A_PLANE;
                        const uint32_t bl0 = bh0 + Cfg::B_PLANE;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint32_t ao = A_MN ? k * 2048 : k * 32;
                            const uint32_t bo = B_MN ? k * 2048 : k * 32;
                            const uint32_t albo = A_MN ? 8192 : 16, blbo = B_MN ? 8192 : 16;
                            const uint64_t ah = smem_desc_sw128(ah0 + ao, albo, 1024);
                            const uint64_t al = smem_desc_sw128(al0 + ao, albo, 1024);
                            const uint64_t bh = smem_desc_sw128(bh0 + bo, blbo, 1024);
                            const uint64_t bl = smem_desc_sw128(bl0 + bo, blbo, 1024);
                            // A_hi x [B_hi | B_lo] accumulates into columns [hh | mid] and
                            // A_lo x [B_hi | B_lo] into [mid | ll]: the middle accumulator gets
                            // both cross products. The first step of a chunk starts ll on its own
                            // so that it does not overwrite mid.
                            if (kb > kb0 || k > 0) {
                                tc_mma_bf16(d_hh, ah, bh, IDESC2, 1u);
                                tc_mma_bf16(d_mid, al, bh, IDESC2, 1u);
                            } else {
                                tc_mma_bf16(d_hh, ah, bh, IDESC2, 0u);
                                tc_mma_bf16(d_ll, al, bl, IDESC, 0u);
                                tc_mma_bf16(d_mid, al, bh, IDESC, 1u);
                            }
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
        const int e = warp - 2;
        const int quad = warp & 3;
        const int half = e >> 2;
        uint8_t* stg = staging + e * 4096;
        const uint32_t stg_row = smem_u32(stg) + lane * 128;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
            const int tm = t / num_n, tn = t % num_n;
            // FP32 outputs: the double (BLOCKED) or float (CHAINED) sums live in the same
            // registers as the int64 ones; both start at +0
            int64_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            const int brow = tm * BM + quad * 32 + lane;                  // this thread's row (FP32 outputs)
            int e_chain = 0;                                              // CHAINED: 2^e scales every chain
            if (MODE == DFP_CHAINED) {
                const int ex = *bk.d_ex, ew = *bk.d_ew;
                if (ex < -128 || ex > 127 || ew < -128 || ew > 127) raise_device_error(err, ITO_ERR_EXPONENT);
                e_chain = max(-300, min(300, ex + bk.shift + ew));
            }
            for (int c = 0; c < num_chunks; ++c) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)(buf * Cfg::BUF_COLS + half * HALF);
                if (MODE == DFP_EXACT) {
                    // one accumulator at a time keeps 16 staging registers live
#pragma unroll
                    for (int j = 0; j < HALF / 16; ++j) {
#pragma unroll 1
                        for (int part = 0; part < 3; ++part) {
                            uint32_t r[16];
                            tmem_ld16(taddr + part * 64 + j * 16, r);
                            tmem_ld_wait();
                            const int sh = part == 0 ? 16 : (part == 1 ? 8 : 0);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                acc[j * 16 + i] += (int64_t)__float2int_rn(__uint_as_float(r[i])) << sh;
                        }
                    }
                } else {
                    const int exr = MODE == DFP_BLOCKED && brow < M ? bk.ex[(int64_t)brow * bk.nb + c] : 0;
#pragma unroll
                    for (int j = 0; j < HALF / 16; ++j) {
                        int64_t pj[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) pj[i] = 0;
#pragma unroll 1
                        for (int part = 0; part < 3; ++part) {
                            uint32_t r[16];
                            tmem_ld16(taddr + part * 64 + j * 16, r);
                            tmem_ld_wait();
                            const int sh = part == 0 ? 16 : (part == 1 ? 8 : 0);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pj[i] += (int64_t)__float2int_rn(__uint_as_float(r[i])) << sh;
                        }
                        if (MODE == DFP_BLOCKED) {
                            // the chunk's exact partial (below 2^53) times a power of two: exact
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int col = tn * BN + half * HALF + j * 16 + i;
                                const int e = exr + (col < N ? bk.ew[(int64_t)col * bk.nb + c] : 0);
                                acc[j * 16 + i] = __double_as_longlong(__longlong_as_double(acc[j * 16 + i]) +
                                                                       (double)pj[i] * pow2d(e));
                            }
                        } else {
                            // the chain as an INT32 accumulator holds it (two's complement, modulo
                            // 2^32), to float, scaled exactly in double and rounded once, then one
                            // float addition per chain in chain order
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int32_t p32 = (int32_t)(uint32_t)(unsigned long long)pj[i];
                                const float term =
                                    __double2float_rn(__dmul_rn((double)__int2float_rn(p32), pow2d(e_chain)));
                                acc[j * 16 + i] =
                                    (uint32_t)__float_as_uint(__fadd_rn(__uint_as_float((uint32_t)acc[j * 16 + i]),
                                                                        term));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce_bar[buf]);
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            if (F32OUT) {
                const int col0 = tn * BN + half * HALF;
                if (brow < M) {
                    float* dst = bk.Y + (int64_t)brow * bk.ldy + col0;
#pragma unroll
                    for (int i = 0; i < HALF; ++i)
                        if (col0 + i < N)
                            dst[i] = MODE == DFP_BLOCKED ? __double2float_rn(__longlong_as_double(acc[i]))
                                                         : __uint_as_float((uint32_t)acc[i]);
                }
                continue;
            }
            unsigned long long mx = 0;
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
                const unsigned long long a = (unsigned long long)(acc[i] < 0 ? -acc[i] : acc[i]);
                mx = a > mx ? a : mx;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long v = __shfl_xor_sync(0xffffffffu, mx, o);
                mx = v > mx ? v : mx;
            }
            if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            const int row0 = tm * BM + quad * 32;
            const int col0 = tn * BN + half * HALF;
            if (use_tma_store) {
                // two 16-column int64 boxes (128 bytes per row, 128-byte swizzle)
#pragma unroll
                for (int g = 0; g < HALF / 16; ++g) {
                    if (row0 >= M || col0 + g * 16 >= N) continue;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int64_t a0 = acc[g * 16 + 2 * j], a1 = acc[g * 16 + 2 * j + 1];
                        st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), (int32_t)(a0 & 0xffffffff),
                                     (int32_t)(a0 >> 32), (int32_t)(a1 & 0xffffffff), (int32_t)(a1 >> 32));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, stg, col0 + g * 16, row0);
                        bulk_commit();
                    }
                }
            } else {
                const int row = row0 + lane;
                if (row < M) {
                    int64_t* dst = C + (int64_t)row * ldc + col0;
#pragma unroll
                    for (int i = 0; i < HALF; ++i)
                        if (col0 + i < N) dst[i] = acc[i];
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

// ------------------------------------------------- CTA-pair limb kernel
//
// The same exact contraction on a CTA pair (tcgen05 cta_group::2): the pair
// computes a 256 x 64 tile. Each CTA loads both limb planes of its 128 rows of
// A and ONE limb plane of B -- the leader the high plane, the other CTA the low
// plane -- so the pair's B operand [B_hi | B_lo] (N = 128) is split between the
// two CTAs exactly as an M = 256 MMA reads it. Per CTA that is 40 KB per K
// block instead of 48 KB for the same products. Two MMAs per k-step:
// A_hi x [B_hi | B_lo] into [hh | mid1] and A_lo x [B_hi | B_lo] into
// [mid2 | ll], four 64-column fp32 accumulators per buffer (two buffers fill
// the 512 tensor-memory columns). Each accumulator gets one limb product per
// K term (at most 2^14), so an exact chunk is 1024 terms. After a chunk the
// epilogue forms 65536 hh + 256 (mid1 + mid2) + ll in int64.

// Work list of the pair kernel: `full` whole tiles, then each remaining tile of
// the last, partial wave cut into `parts` chunk-aligned K pieces (slot = piece
// index; -1 for a whole tile).
struct DfpWork {
    int tile, c0, c1, slot;
};

__device__ __forceinline__ DfpWork dfp_work(int w, int full, int parts, int num_chunks)
{
    if (w < full) return DfpWork{w, 0, num_chunks, -1};
    const int u = w - full;
    const int ti = u / parts, part = u - ti * parts;
    return DfpWork{full + ti, part * num_chunks / parts, (part + 1) * num_chunks / parts, u};
}

// C = the sum of the K pieces of each split tile (exact int64), inside the M x N
// bounds; max |C| folded into *d_max. P: [tail tiles][parts][256][64] int64.
__global__ void k_tail_reduce64(const int64_t* __restrict__ P, int tail_tiles, int parts, int full_tiles, int num_n,
                                int M, int N, int64_t ldc, int64_t* __restrict__ C,
                                unsigned long long* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int TR = 256, TC = 64;
    const int64_t n = (int64_t)tail_tiles * TR * (TC / 2);
    unsigned long long mx = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int ti = (int)(i / (TR * (TC / 2)));
        const int rem = (int)(i - (int64_t)ti * (TR * (TC / 2)));
        const int r = rem / (TC / 2), c = (rem % (TC / 2)) * 2;
        int64_t a0 = 0, a1 = 0;
        for (int q = 0; q < parts; ++q) {
            const longlong2 v =
                __ldcs(reinterpret_cast<const longlong2*>(P + (((int64_t)ti * parts + q) * TR + r) * TC + c));
            a0 += v.x;
            a1 += v.y;
        }
        const int tile = full_tiles + ti;
        const int gr = (tile / num_n) * TR + r, gc = (tile % num_n) * TC + c;
        if (gr < M) {
            if (gc < N) {
                C[(int64_t)gr * ldc + gc] = a0;
                const unsigned long long u = (unsigned long long)(a0 < 0 ? -a0 : a0);
                mx = u > mx ? u : mx;
            }
            if (gc + 1 < N) {
                C[(int64_t)gr * ldc + gc + 1] = a1;
                const unsigned long long u = (unsigned long long)(a1 < 0 ? -a1 : a1);
                mx = u > mx ? u : mx;
            }
        }
    }
    block_atomic_max(d_max, mx);
}

struct Dfp2Cfg {
    static constexpr int BM = 128, BN = 64, BK = 64;       // BM rows per CTA (256 per pair)
    static constexpr int A_PLANE = BM * BK * 2;             // 16 KB
    static constexpr int B_PLANE = BN * BK * 2;             // 8 KB: one limb plane of the tile's B
    static constexpr int STAGE_BYTES = 2 * A_PLANE + B_PLANE;
    static constexpr int STAGES = 5;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int BUF_COLS = 256;                    // hh, mid1, mid2, ll at +0, +64, +128, +192
    static constexpr int TMEM_COLS = 512;
    static constexpr int CHUNK_KB = 1024 / BK;              // exact chunk: 1024 K terms
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
};

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(Dfp2Cfg::THREADS, 1)
    k_gemm_dfp2(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl, int M, int N,
                int K, int full_tiles, int parts, int64_t* __restrict__ C, int64_t ldc,
                int64_t* __restrict__ tail_ws, unsigned long long* __restrict__ d_max, int* __restrict__ err)
{
    using Cfg = Dfp2Cfg;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;                         // 32 columns per epilogue warp
    constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, 2 * BN, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;
    uint64_t* acce_bar = accf_bar + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int num_m = (M + 2 * BM - 1) / (2 * BM), num_n = (N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    const int num_kb = (K + BK - 1) / BK;
    const int num_chunks = (num_kb + Cfg::CHUNK_KB - 1) / Cfg::CHUNK_KB;
    // the last partial wave's tiles may be cut into `parts` K pieces (see work_item)
    const int total_work = full_tiles + (num_tiles - full_tiles) * parts;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], 2 * Cfg::EPI_WARPS);   // epilogue warps of both CTAs
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // on-chip setup above overlaps the previous kernel; global memory only from here on
    griddep_wait();
    griddep_launch_dependents();

    // tiles in row-major order over (m, n): consecutive clusters share the A band
    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap* tmB = leader ? &tmBh : &tmBl;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = cluster; ok && w < total_work; w += nclusters) {
                const DfpWork wi = dfp_work(w, full_tiles, parts, num_chunks);
                const int tm = wi.tile / num_n, tn = wi.tile % num_n;
                const int rowA = tm * 2 * BM + (int)rank * BM;
                const int kb_end = min(num_kb, wi.c1 * Cfg::CHUNK_KB);
                for (int kb = wi.c0 * Cfg::CHUNK_KB; kb < kb_end; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
                    uint8_t* sAh = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sAl = sAh + Cfg::A_PLANE;
                    uint8_t* sB = sAl + Cfg::A_PLANE;
                    if (!A_MN) {
                        tma_load_2d_pair(&tmAh, fb, sAh, kb * BK, rowA);
                        tma_load_2d_pair(&tmAl, fb, sAl, kb * BK, rowA);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j) {
                            tma_load_2d_pair(&tmAh, fb, sAh + j * 8192, rowA + j * 64, kb * BK);
                            tma_load_2d_pair(&tmAl, fb, sAl + j * 8192, rowA + j * 64, kb * BK);
                        }
                    }
                    if (!B_MN)
                        tma_load_2d_pair(tmB, fb, sB, kb * BK, tn * BN);
                    else
                        tma_load_2d_pair(tmB, fb, sB, tn * BN, kb * BK);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int w = cluster; ok && w < total_work; w += nclusters) {
                const DfpWork wi = dfp_work(w, full_tiles, parts, num_chunks);
                for (int c = wi.c0; ok && c < wi.c1; ++c) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_hi = tmem_base + (uint32_t)(buf * Cfg::BUF_COLS);   // [hh | mid1]
                    const uint32_t d_lo = d_hi + 2 * BN;                                  // [mid2 | ll]
                    const int kb0 = c * Cfg::CHUNK_KB;
                    const int kb1 = min(num_kb, kb0 + Cfg::CHUNK_KB);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ah0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t al0 = ah0 + Cfg::A_PLANE;
                        const uint32_t b0 = al0 + Cfg::A_PLANE;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint32_t ao = A_MN ? k * 2048 : k * 32;
                            const uint32_t bo = B_MN ? k * 2048 : k * 32;
                            const uint32_t albo = A_MN ? 8192 : 16, blbo = B_MN ? 8192 : 16;
                            const uint64_t ah = smem_desc_sw128(ah0 + ao, albo, 1024);
                            const uint64_t al = smem_desc_sw128(al0 + ao, albo, 1024);
                            const uint64_t bd = smem_desc_sw128(b0 + bo, blbo, 1024);
                            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
                            tc_mma_bf16_pair(d_hi, ah, bd, IDESC, acc);
                            tc_mma_bf16_pair(d_lo, al, bd, IDESC, acc);
                        }
                        tc_commit_pair_mc(&empty_bar[stage], 0x3);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(&accf_bar[buf], 0x3);
                    if (++buf == 2) { buf = 0; buf_phase ^= 1; }
                }
            }
        }
    } else {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the pair tile
        const int e = warp - 2;
        const int quad = warp & 3;
        const int half = e >> 2;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int w = cluster; ok && w < total_work; w += nclusters) {
            const DfpWork wi = dfp_work(w, full_tiles, parts, num_chunks);
            const int tm = wi.tile / num_n, tn = wi.tile % num_n;
            int64_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int c = wi.c0; c < wi.c1; ++c) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)(buf * Cfg::BUF_COLS + half * HALF);
#pragma unroll
                for (int j = 0; j < HALF / 16; ++j) {
#pragma unroll 1
                    for (int part = 0; part < 4; ++part) {
                        uint32_t r[16];
                        tmem_ld16(taddr + part * BN + j * 16, r);
                        tmem_ld_wait();
                        const int sh = part == 0 ? 16 : (part == 3 ? 0 : 8);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[j * 16 + i] += (int64_t)__float2int_rn(__uint_as_float(r[i])) << sh;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acce_bar[buf]), 0));
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            if (wi.slot >= 0) {
                // a K piece of a split tile: its exact partial goes to workspace slot wi.slot
                // ([slot][256 rows][64 cols] int64); k_tail_reduce64 finishes the tile
                int64_t* dst = tail_ws + ((int64_t)wi.slot * 2 * BM + (int)rank * BM + quad * 32 + lane) * BN +
                               half * HALF;
#pragma unroll
                for (int i = 0; i < HALF; i += 2)
                    *reinterpret_cast<longlong2*>(dst + i) = make_longlong2(acc[i], acc[i + 1]);
                continue;
            }
            unsigned long long mx = 0;
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
                const unsigned long long a = (unsigned long long)(acc[i] < 0 ? -acc[i] : acc[i]);
                mx = a > mx ? a : mx;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long v = __shfl_xor_sync(0xffffffffu, mx, o);
                mx = v > mx ? v : mx;
            }
            if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            // the int64 result from registers: 32 consecutive values per row
            const int row = tm * 2 * BM + (int)rank * BM + quad * 32 + lane;
            const int col0 = tn * BN + half * HALF;
            if (row < M) {
                int64_t* dst = C + (int64_t)row * ldc + col0;
                if (col0 + HALF <= N && (ldc & 1) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0) {
#pragma unroll
                    for (int i = 0; i < HALF; i += 2)
                        *reinterpret_cast<longlong2*>(dst + i) = make_longlong2(acc[i], acc[i + 1]);
                } else {
#pragma unroll
                    for (int i = 0; i < HALF; ++i)
                        if (col0 + i < N) dst[i] = acc[i];
                }
            }
        }
    }

    tc_fence_before();
    cluster_sync();   // the pair's MMAs and drains are complete in both CTAs
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// ------------------------------------------- wide-tile CTA-pair kernel
//
// The exact contraction on a CTA pair with 256 x bn output tiles (bn = 128, or
// 112 where that fills the last wave better): each CTA loads both limb planes of
// its 128 rows of A and ONE limb plane of the tile's bn columns of B (the leader
// the high plane, the other CTA the low plane), so the pair's B operand
// [B_hi | B_lo] (N = 2 bn) is split between the two CTAs as an M = 256 MMA reads
// it. Two MMAs per 16-term K step: A_hi x [B_hi | B_lo] into [hh | hl] at tensor-
// memory column 0 and A_lo x [B_hi | B_lo] into [lh | ll] at column 256, four
// bn-column fp32 accumulators in the 512 tensor-memory columns (one buffer: the
// MMAs of the next chunk wait for the drain). Against the 64-column tile this
// halves the A bytes per operation moved into and read from shared memory. Each
// accumulator gets one limb product (at most 2^14) per K term, so an exact chunk
// is 1024 terms; after a chunk the epilogue adds 65536 hh + 256 (hl + lh) + ll
// into the tile's int64 sums in registers.
struct Dfp4Cfg {
    static constexpr int BM = 128, BN = 128, BK = 64;      // BM rows per CTA (256 per pair), BN columns at most
    static constexpr int A_PLANE = BM * BK * 2;             // 16 KB
    static constexpr int B_PLANE = BN * BK * 2;             // 16 KB: one limb plane of B (BN columns loaded)
    static constexpr int STAGE_BYTES = 2 * A_PLANE + B_PLANE;
    static constexpr int STAGES = 4;
    // 16 epilogue warps, each 32 TMEM lanes x 32 columns of the four accumulators: the
    // drain, which the next chunk's MMAs wait for, is spread over twice the warps
    static constexpr int EPI_WARPS = 16;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int TMEM_COLS = 512;                   // hh, hl, lh, ll at +0, +bn, +256, +256 + bn
    static constexpr int CHUNK_KB = 1024 / BK;              // exact chunk: 1024 K terms
    // one 32-row x 8-column int64 store box per epilogue warp: the result leaves by TMA
    static constexpr int STAGING_BYTES = EPI_WARPS * 32 * 8 * 8;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
};
static_assert(Dfp4Cfg::SMEM_BYTES <= 227 * 1024, "wide-tile kernel: shared memory above the per-CTA limit");
// a CTA's last tile stages each warp's whole 32 x 32 block in the (then idle) pipeline stages
static_assert(Dfp4Cfg::EPI_WARPS * 32 * 32 * 8 <= Dfp4Cfg::STAGES * Dfp4Cfg::STAGE_BYTES, "stages too small");

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(Dfp4Cfg::THREADS, 1)
    k_gemm_dfp4(const __grid_constant__ CUtensorMap tmAh, const __grid_constant__ CUtensorMap tmAl,
                const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmBl,
                const __grid_constant__ CUtensorMap tmC, int use_tma_store, int bn, int M, int N, int K,
                int64_t* __restrict__ C, int64_t ldc, unsigned long long* __restrict__ d_max, int* __restrict__ err)
{
    using Cfg = Dfp4Cfg;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int COLS = BN / (Cfg::EPI_WARPS / 4);       // 32 output columns per epilogue warp (fewer past bn)
    const uint32_t idesc = idesc_bf16_f32(2 * BM, 2 * bn, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;     // 1024-aligned
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;   // the chunk's accumulators are complete
    uint64_t* acce_bar = accf_bar + 1;         // they have been drained (both CTAs)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int num_m = (M + 2 * BM - 1) / (2 * BM), num_n = (N + bn - 1) / bn;
    const int num_tiles = num_m * num_n;
    const int num_kb = (K + BK - 1) / BK;
    const int num_chunks = (num_kb + Cfg::CHUNK_KB - 1) / Cfg::CHUNK_KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(accf_bar, 1);
        mbar_init(acce_bar, 2 * Cfg::EPI_WARPS);   // epilogue warps of both CTAs
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmAh);
        prefetch_tensormap(&tmAl);
        prefetch_tensormap(leader ? &tmBh : &tmBl);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // on-chip setup above overlaps the previous kernel; global memory only from here on
    griddep_wait();
    griddep_launch_dependents();

    // tiles in row-major order over (m, n): consecutive clusters share the A band
    if (warp == 0) {
        // ---------------- TMA producer (both CTAs): loads complete on the leader's barrier
        if (lane == 0) {
            const CUtensorMap* tmB = leader ? &tmBh : &tmBl;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = cluster; ok && t < num_tiles; t += nclusters) {
                const int rowA = (t / num_n) * 2 * BM + (int)rank * BM, colB = (t % num_n) * bn;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
                    uint8_t* sAh = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sAl = sAh + Cfg::A_PLANE;
                    uint8_t* sB = sAl + Cfg::A_PLANE;
                    if (!A_MN) {
                        tma_load_2d_pair(&tmAh, fb, sAh, kb * BK, rowA);
                        tma_load_2d_pair(&tmAl, fb, sAl, kb * BK, rowA);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j) {
                            tma_load_2d_pair(&tmAh, fb, sAh + j * 8192, rowA + j * 64, kb * BK);
                            tma_load_2d_pair(&tmAl, fb, sAl + j * 8192, rowA + j * 64, kb * BK);
                        }
                    }
                    if (!B_MN) {
                        tma_load_2d_pair(tmB, fb, sB, kb * BK, colB);
                    } else {
                        tma_load_2d_pair(tmB, fb, sB, colB, kb * BK);
                        tma_load_2d_pair(tmB, fb, sB + 8192, colB + 64, kb * BK);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread of the leader CTA
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            const uint32_t d_hi = tmem_base;               // [hh | hl]
            const uint32_t d_lo = tmem_base + 256;         // [lh | ll]
            for (int t = cluster; ok && t < num_tiles; t += nclusters) {
                for (int c = 0; ok && c < num_chunks; ++c) {
                    if (!mbar_wait(acce_bar, acc_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const int kb0 = c * Cfg::CHUNK_KB;
                    const int kb1 = min(num_kb, kb0 + Cfg::CHUNK_KB);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t ah0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t al0 = ah0 + Cfg::A_PLANE;
                        const uint32_t b0 = al0 + Cfg::A_PLANE;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint32_t ao = A_MN ? k * 2048 : k * 32;
                            const uint32_t albo = A_MN ? 8192 : 16;
                            const uint64_t ah = smem_desc_sw128(ah0 + ao, albo, 1024);
                            const uint64_t al = smem_desc_sw128(al0 + ao, albo, 1024);
                            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                                     : smem_desc_sw128(b0 + k * 32, 16, 1024);
                            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
                            tc_mma_bf16_pair(d_hi, ah, bd, idesc, acc);
                            tc_mma_bf16_pair(d_lo, al, bd, idesc, acc);
                        }
                        tc_commit_pair_mc(&empty_bar[stage], 0x3);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    tc_commit_pair_mc(accf_bar, 0x3);
                    acc_phase ^= 1;
                }
            }
        }
    } else {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of the pair tile
        const int e = warp - 2;
        const int quad = warp & 3;            // TMEM lanes this warp may access
        const int cg = e >> 2;                // which 32-column group of the tile
        const int valid = min(COLS, bn - cg * COLS);   // its columns inside the tile (16 or 32)
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int t = cluster; ok && t < num_tiles; t += nclusters) {
            int64_t acc[COLS];
#pragma unroll
            for (int i = 0; i < COLS; ++i) acc[i] = 0;
            const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cg * COLS);
            for (int c = 0; c < num_chunks; ++c) {
                if (!mbar_wait(accf_bar, acc_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                // 65536 hh + 256 hl + 256 lh + ll, one accumulator at a time
#pragma unroll 1
                for (int part = 0; part < 4; ++part) {
                    const int32_t scale = part == 0 ? 65536 : (part == 3 ? 1 : 256);
                    const uint32_t poff = (uint32_t)((part & 1) * bn + (part >> 1) * 256);
#pragma unroll
                    for (int j = 0; j < COLS / 16; ++j) {
                        // past the tile's bn columns this reads unused accumulator columns;
                        // those sums are neither stored nor counted in the max
                        uint32_t r[16];
                        tmem_ld16(taddr + poff + j * 16, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[j * 16 + i] += (int64_t)__float2int_rn(__uint_as_float(r[i])) * scale;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(acce_bar), 0));
                acc_phase ^= 1;
            }
            if (!ok) break;
            // the int64 result from registers: 32 consecutive values per row (the last 16
            // outside the tile when the warp's group has only 16 columns)
            const int row0 = (t / num_n) * 2 * BM + (int)rank * BM + quad * 32;
            const int row = row0 + lane;
            const int col0 = (t % num_n) * bn + cg * COLS;
            const int ncols = min(valid, N - col0);   // columns of this warp's block inside C (may be <= 0)
            unsigned long long mx = 0;
#pragma unroll
            for (int i = 0; i < COLS; ++i) {
                const unsigned long long a = (unsigned long long)(acc[i] < 0 ? -acc[i] : acc[i]);
                if (i < 16 || valid == COLS) mx = a > mx ? a : mx;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long v = __shfl_xor_sync(0xffffffffu, mx, o);
                mx = v > mx ? v : mx;
            }
            if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            if (use_tma_store) {
                // 32 x 8 boxes (row-major, 64 bytes a row) written out by TMA, the edges clipped.
                // Before the CTA's last tile they go one at a time through this warp's 2 KB
                // slot; for the last tile (every MMA done, no load left) the warp stages its
                // whole block in the pipeline stages and issues the four stores at once.
                const bool last = t + nclusters >= num_tiles;
                uint8_t* stg = last ? smem + e * (32 * COLS * 8) : staging + e * (32 * 8 * 8);
#pragma unroll
                for (int g = 0; g < COLS / 8; ++g) {
                    uint8_t* box = last ? stg + g * (32 * 8 * 8) : stg;
                    if (!last) {
                        if (lane == 0) bulk_wait_read_all();   // the slot's previous box has been read
                        __syncwarp();
                    }
                    const uint32_t srow = smem_u32(box) + lane * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t v0 = acc[g * 8 + 2 * j], v1 = acc[g * 8 + 2 * j + 1];
                        st_shared_v4(srow + j * 16, (int32_t)v0, (int32_t)(v0 >> 32), (int32_t)v1,
                                     (int32_t)(v1 >> 32));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (row0 < M && g * 8 < ncols) tma_store_2d(&tmC, box, col0 + g * 8, row0);
                        if (!last) bulk_commit();
                    }
                }
                if (last && lane == 0) bulk_commit();
            } else if (row < M) {
                int64_t* dst = C + (int64_t)row * ldc + col0;
                if (ncols == COLS && (ldc & 1) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0) {
#pragma unroll
                    for (int i = 0; i < COLS; i += 2)
                        *reinterpret_cast<longlong2*>(dst + i) = make_longlong2(acc[i], acc[i + 1]);
                } else {
#pragma unroll
                    for (int i = 0; i < COLS; ++i)
                        if (i < ncols) dst[i] = acc[i];
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    cluster_sync();   // the pair's MMAs and drains are complete in both CTAs
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// CTA pairs of k_gemm_dfp4 resident at once (all operand layouts share one occupancy);
// the first call also raises every instance's shared-memory limit. 0 on failure.
static int dfp4_clusters()
{
    using Cfg = Dfp4Cfg;
    static int n = 0;
    if (!n) {
        void (*kerns[4])(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, int, int, int, int, int,
                         int64_t*, int64_t, unsigned long long*, int*) = {
            k_gemm_dfp4<false, false>, k_gemm_dfp4<false, true>, k_gemm_dfp4<true, false>, k_gemm_dfp4<true, true>};
        for (auto k : kerns)
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
                return 0;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * num_sms());
        q.blockDim = dim3(Cfg::THREADS);
        q.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, k_gemm_dfp4<false, false>, &q) != cudaSuccess || c < 1) return 0;
        n = c;
    }
    return n;
}

// Tile width of the wide-tile kernel: 112 columns instead of 128 when the tiles then
// fill their waves enough better (waves x width at least 5% smaller; e.g. a 2048 x 2048
// output on 76 pairs: 152 tiles of 112 columns in two full waves, against 128 tiles of
// 128 columns whose second wave leaves 24 pairs idle).
static int dfp4_width(int M, int N, int clusters)
{
    if (clusters < 1) return 128;
    const int num_m = (M + 255) / 256;
    auto cost = [&](int bn) { return (double)((num_m * ((N + bn - 1) / bn) + clusters - 1) / clusters) * bn; };
    return cost(112) < 0.95 * cost(128) ? 112 : 128;
}

template <bool A_MN, bool B_MN>
static int launch_dfp4(const DfpGemmPlan& p, cudaStream_t s)
{
    using Cfg = Dfp4Cfg;
    auto kern = k_gemm_dfp4<A_MN, B_MN>;
    const int max_clusters = dfp4_clusters();
    if (max_clusters < 1) return set_error(ITO_ERR_CUDA, "no CTA pair of the wide-tile kernel fits on this device");
    const int tiles = ((p.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((p.N + p.bn4 - 1) / p.bn4);
    const int clusters = tiles < max_clusters ? tiles : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p.mapAh, p.mapAl, p.mapBh3, p.mapBl3, p.mapC8, p.use_tma_store8,
                                       p.bn4, p.M, p.N, p.K, p.C, p.ldc, p.d_max, p.err);
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp wide gemm launch: %s", cudaGetErrorString(e));
}

template <bool A_MN, bool B_MN>
static int launch_dfp2(const DfpGemmPlan& p, cudaStream_t s)
{
    using Cfg = Dfp2Cfg;
    auto kern = k_gemm_dfp2<A_MN, B_MN>;
    static int max_clusters = 0;
    if (!max_clusters) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(cudaGetLastError()));
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * num_sms());
        q.blockDim = dim3(Cfg::THREADS);
        q.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1)
            return set_error(ITO_ERR_CUDA, "no CTA pair fits on this device");
        max_clusters = n;
    }
    const int num_n = (p.N + Cfg::BN - 1) / Cfg::BN;
    const int tiles = ((p.M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * num_n;
    const int work = p.tail_full + (tiles - p.tail_full) * p.tail_parts;
    const int clusters = work < max_clusters ? work : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p.mapAh, p.mapAl, p.mapBh, p.mapBl, p.M, p.N, p.K, p.tail_full,
                                       p.tail_parts, p.C, p.ldc, p.tail_ws, p.d_max, p.err);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "dfp pair gemm launch: %s", cudaGetErrorString(e));
    if (p.tail_parts > 1) {
        const int tail = tiles - p.tail_full;
        launch_pdl(k_tail_reduce64, launch_grid_blocks((int64_t)tail * 256 * 32, 256), 256, 0, s, 
            p.tail_ws, tail, p.tail_parts, p.tail_full, num_n, p.M, p.N, p.ldc, p.C, p.d_max);
        e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "dfp tail reduce launch: %s", cudaGetErrorString(e));
    }
    return ITO_OK;
}

// CTA pairs of k_gemm_dfp2 resident at once (all operand layouts share one occupancy).
static int dfp2_clusters()
{
    using Cfg = Dfp2Cfg;
    static int n = 0;
    if (!n) {
        auto kern = k_gemm_dfp2<false, false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(2 * num_sms());
        q.blockDim = dim3(Cfg::THREADS);
        q.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, kern, &q) != cudaSuccess || c < 1) return 0;
        n = c;
    }
    return n;
}

// Last-wave split of a pair-kernel limb contraction (whole tiles, K pieces per
// remaining tile); estimated time = waves of whole tiles + rounds of pieces, plus
// the reduction pass (pieces written and read once at about 5 TB/s, one launch).
// A 256 x 64 tile takes 4 limb products of 2 * 256 * 64 * K operations at about
// 13 TFLOP/s per pair (the measured pair-kernel rate).
static void dfp_tail_split(int M, int N, int K, int* full, int* parts)
{
    using Cfg = Dfp2Cfg;
    const int tiles = ((M + 2 * Cfg::BM - 1) / (2 * Cfg::BM)) * ((N + Cfg::BN - 1) / Cfg::BN);
    *full = tiles;
    *parts = 1;
    const int clusters = dfp2_clusters();
    const int num_chunks = ((K + Cfg::BK - 1) / Cfg::BK + Cfg::CHUNK_KB - 1) / Cfg::CHUNK_KB;
    if (clusters < 1 || tiles % clusters == 0) return;
    const int waves = tiles / clusters, r = tiles % clusters;
    const double tile_us = 4.0 * 2 * 256 * 64 * (double)K / 13.0e6;
    double best = (waves + 1.0) * tile_us;
    for (int q = 2; q <= 4 && q <= num_chunks; ++q) {
        const double red_us = 3.0 + 2.0 * r * q * 256.0 * 64 * 8 / 5.0e6;
        const double t = (waves + (double)((r * q + clusters - 1) / clusters) / q) * tile_us + red_us;
        if (t < best) {
            best = t;
            *full = tiles - r;
            *parts = q;
        }
    }
}

size_t dfp_split_ws_bytes(int M, int N, int K)
{
    if (M < 256) return 0;
    int full, parts;
    dfp_tail_split(M, N, K, &full, &parts);
    const int tiles = ((M + 255) / 256) * ((N + 63) / 64);
    return parts > 1 ? (size_t)(tiles - full) * parts * 256 * 64 * sizeof(int64_t) : 0;
}

template <bool A_MN, bool B_MN, int MODE = DFP_EXACT>
static int launch_dfp(const DfpGemmPlan& p, cudaStream_t s)
{
    auto kern = k_gemm_dfp<A_MN, B_MN, MODE>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DfpCfg::SMEM_BYTES) !=
            cudaSuccess)
            return set_error(ITO_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(cudaGetLastError()));
        attr_set = true;
    }
    const int tiles = ((p.M + DfpCfg::BM - 1) / DfpCfg::BM) * ((p.N + DfpCfg::BN - 1) / DfpCfg::BN);
    const int grid = tiles < num_sms() ? tiles : num_sms();
    const DfpF32Out bk{p.ex, p.ew, p.nb, p.d_ex, p.d_ew, p.shift, p.Y, p.ldy};
    launch_pdl(kern, grid, DfpCfg::THREADS, DfpCfg::SMEM_BYTES, s, p.mapAh, p.mapAl, p.mapBh, p.mapBl, p.mapC,
                                                           p.use_tma_store, p.M, p.N, p.K, p.chunk_kb, p.C, p.ldc,
                                                           p.d_max, bk, p.err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp gemm launch: %s", cudaGetErrorString(e));
}

int dfp_gemm_plan(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, bool a_mn, const Bf16View& Bh,
                  const Bf16View& Bl, bool b_mn, int M, int N, int K, int64_t* C, int64_t ldc,
                  unsigned long long* d_max, int64_t* tail_ws, size_t tail_ws_bytes, bool fill_waves)
{
    if (M < 1 || N < 1 || K < 1) return set_error(ITO_ERR_SHAPE, "dfp gemm: empty contraction");
    if (K > (1 << 20)) return set_error(ITO_ERR_SHAPE, "dfp gemm: contraction longer than 2^20");
    if (a_mn ? (Ah.rows != K || Ah.cols != M) : (Ah.rows != M || Ah.cols != K))
        return set_error(ITO_ERR_SHAPE, "dfp gemm: A view does not match M x K");
    if (b_mn ? (Bh.rows != K || Bh.cols != N) : (Bh.rows != N || Bh.cols != K))
        return set_error(ITO_ERR_SHAPE, "dfp gemm: B view does not match N x K");
    *p = DfpGemmPlan{};
    p->chunk_kb = DfpCfg::CHUNK_KB;
    p->M = M;
    p->N = N;
    p->K = K;
    p->a_mn = a_mn;
    p->b_mn = b_mn;
    p->C = C;
    p->ldc = ldc;
    p->d_max = d_max;
    p->err = device_error_word();
    if (!p->err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    int r;
    if ((r = make_map_bf16(&p->mapAh, Ah, a_mn ? 64 : 128)) || (r = make_map_bf16(&p->mapAl, Al, a_mn ? 64 : 128)) ||
        (r = make_map_bf16(&p->mapBh, Bh, 64)) || (r = make_map_bf16(&p->mapBl, Bl, 64)))
        return r;
    // CTA-pair kernels when there are at least 256 rows: the wide-tile one (256 x 128 tiles,
    // B tensor maps of 128-row boxes when B is K-major) when the output has 128 columns or more,
    // else the 256 x 64 one (which splits a partial last wave along K when given room)
    p->pair = M >= 256 && C != nullptr;
    p->stacked = p->pair && N >= 128;
    p->bn4 = p->stacked && fill_waves ? dfp4_width(M, N, dfp4_clusters()) : 128;
    if (p->stacked &&
        ((r = make_map_bf16(&p->mapBh3, Bh, b_mn ? 64 : 128)) || (r = make_map_bf16(&p->mapBl3, Bl, b_mn ? 64 : 128))))
        return r;
    p->tail_full = ((M + 255) / 256) * ((N + 63) / 64);
    p->tail_parts = 1;
    if (p->pair && !p->stacked && tail_ws) {
        int full, parts;
        dfp_tail_split(M, N, K, &full, &parts);
        const size_t need = parts > 1 ? (size_t)(p->tail_full - full) * parts * 256 * 64 * sizeof(int64_t) : 0;
        if (parts > 1 && need <= tail_ws_bytes) {
            p->tail_full = full;
            p->tail_parts = parts;
            p->tail_ws = tail_ws;
        }
    }
    p->use_tma_store = 0;
    if (C && (reinterpret_cast<uintptr_t>(C) & 15) == 0 && (ldc & 1) == 0) {
        auto enc = get_encode();
        cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)ldc * 8};
        cuuint32_t box[2] = {16, 32};
        cuuint32_t estr[2] = {1, 1};
        CUresult cr = enc(&p->mapC, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (P) failed (%d)", (int)cr);
        p->use_tma_store = 1;
        // the wide-tile kernel's 32 x 8 boxes, unswizzled
        cuuint32_t box8[2] = {8, 32};
        cr = enc(&p->mapC8, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, C, dims, strides, box8, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (P, 8) failed (%d)", (int)cr);
        p->use_tma_store8 = 1;
    }
    return ITO_OK;
}

int dfp_gemm_plan_blocked(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, const Bf16View& Bh,
                          const Bf16View& Bl, int M, int N, int K, int block, const int8_t* ex, const int8_t* ew,
                          float* Y, int64_t ldy)
{
    if (block < 64 || block > 512 || block % 64)
        return set_error(ITO_ERR_ARG, "blocked DFP: block must be a multiple of 64 in [64, 512]");
    if (!ex || !ew || !Y) return set_error(ITO_ERR_ARG, "blocked DFP: NULL exponent or output pointer");
    // the int64 result and its max are not produced; C = nullptr keeps the int64 store map unused
    int r = dfp_gemm_plan(p, Ah, Al, false, Bh, Bl, false, M, N, K, nullptr, 0, nullptr, nullptr, 0);
    if (r) return r;
    p->chunk_kb = block / 64;
    p->blocked = 1;
    p->ex = ex;
    p->ew = ew;
    p->nb = (K + block - 1) / block;
    p->Y = Y;
    p->ldy = ldy;
    return ITO_OK;
}

int dfp_gemm_plan_chained(DfpGemmPlan* p, const Bf16View& Ah, const Bf16View& Al, const Bf16View& Bh,
                          const Bf16View& Bl, int M, int N, int K, int chain, const int32_t* d_ex,
                          const int32_t* d_ew, int shift, float* Y, int64_t ldy)
{
    if (chain < 64 || chain > 512 || chain % 64)
        return set_error(ITO_ERR_ARG, "chained DFP: chain must be a multiple of 64 in [64, 512]");
    if (!d_ex || !d_ew || !Y) return set_error(ITO_ERR_ARG, "chained DFP: NULL exponent or output pointer");
    // single-CTA kernel, every tile whole: the chains of an output are added in order by one thread
    int r = dfp_gemm_plan(p, Ah, Al, false, Bh, Bl, false, M, N, K, nullptr, 0, nullptr, nullptr, 0);
    if (r) return r;
    p->chunk_kb = chain / 64;
    p->blocked = 2;
    p->d_ex = d_ex;
    p->d_ew = d_ew;
    p->shift = shift ? 1 : 0;
    p->Y = Y;
    p->ldy = ldy;
    return ITO_OK;
}

int dfp_gemm_run(const DfpGemmPlan& p, cudaStream_t s)
{
    if (p.blocked == 1) return launch_dfp<false, false, DFP_BLOCKED>(p, s);
    if (p.blocked == 2) return launch_dfp<false, false, DFP_CHAINED>(p, s);
    if (p.stacked) {
        if (!p.a_mn && !p.b_mn) return launch_dfp4<false, false>(p, s);
        if (!p.a_mn && p.b_mn) return launch_dfp4<false, true>(p, s);
        if (p.a_mn && p.b_mn) return launch_dfp4<true, true>(p, s);
        return launch_dfp4<true, false>(p, s);
    }
    if (p.pair) {
        if (!p.a_mn && !p.b_mn) return launch_dfp2<false, false>(p, s);
        if (!p.a_mn && p.b_mn) return launch_dfp2<false, true>(p, s);
        if (p.a_mn && p.b_mn) return launch_dfp2<true, true>(p, s);
        return launch_dfp2<true, false>(p, s);
    }
    if (!p.a_mn && !p.b_mn) return launch_dfp<false, false>(p, s);
    if (!p.a_mn && p.b_mn) return launch_dfp<false, true>(p, s);
    if (p.a_mn && p.b_mn) return launch_dfp<true, true>(p, s);
    return launch_dfp<true, false>(p, s);
}

// ---------------------------------------------------------- limb planes

// shift = 1: the mantissas are first shifted right by one bit, rounding half up
// (the input shift of the FP32 partial accumulation)
__global__ void k_i16_to_limbs(const int16_t* __restrict__ src, int64_t rows, int64_t cols,
                               uint16_t* __restrict__ hi, uint16_t* __restrict__ lo, int64_t ldl, int shift)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        int32_t h, l;
        const int32_t v = src[i];
        limb_split(shift ? (v + 1) >> 1 : v, h, l);
        hi[r * ldl + c] = int_to_bf16_bits(h);
        lo[r * ldl + c] = int_to_bf16_bits(l);
    }
}

int launch_i16_to_limbs(const int16_t* src, int64_t rows, int64_t cols, uint16_t* hi, uint16_t* lo, int64_t ldl,
                        cudaStream_t s, int shift)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    launch_pdl(k_i16_to_limbs, launch_grid_blocks(rows * cols, 256), 256, 0, s, src, rows, cols, hi, lo, ldl, shift);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "limb launch: %s", cudaGetErrorString(e));
}

// ------------------------------------------------------- down-conversion

// adds the block's partial sums of |mantissa| to *d_abs_sum (exact: integer atomics)
__device__ __forceinline__ void add_abs_sum(unsigned long long* d_abs_sum, unsigned long long v)
{
    block_atomic_add(d_abs_sum, v);
}

__global__ void k_dfp_down(const int64_t* __restrict__ P, int64_t rows, int64_t cols,
                           const unsigned long long* __restrict__ d_max, const int32_t* __restrict__ d_ea,
                           const int32_t* __restrict__ d_eb, int16_t* __restrict__ out16, uint16_t* __restrict__ hi,
                           uint16_t* __restrict__ lo, int64_t ldl, int32_t* __restrict__ d_exp_out,
                           int32_t* __restrict__ d_exp_out2, int32_t* __restrict__ d_rs,
                           unsigned long long* __restrict__ d_abs_sum,
                           int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    // section 3.1: Rs brings max |P| within 15 magnitude bits; the new exponent is Ea + Eb + Rs
    const unsigned long long m = *d_max;
    const int bl = m ? 64 - __clzll((long long)m) : 0;
    const int rs = bl > 15 ? bl - 15 : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int e = *d_ea + (d_eb ? *d_eb : 0) + rs;
        if (d_exp_out) *d_exp_out = e;
        if (d_exp_out2) *d_exp_out2 = e;
        if (d_rs) *d_rs = rs;
        if (e < -128 || e > 127) raise_device_error(err, ITO_ERR_EXPONENT);
    }
    const int64_t n = rows * cols;
    unsigned long long asum = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t v = (int32_t)sat16s(rhu64(__ldcs(P + i), rs));
        out16[i] = (int16_t)v;
        asum += (unsigned long long)(v < 0 ? -v : v);
        if (hi) {
            const int64_t r = i / cols, c = i - r * cols;
            int32_t h, l;
            limb_split(v, h, l);
            hi[r * ldl + c] = int_to_bf16_bits(h);
            lo[r * ldl + c] = int_to_bf16_bits(l);
        }
    }
    if (d_abs_sum) add_abs_sum(d_abs_sum, asum);
}

// four elements per thread step: 32 bytes of P in, 8 bytes of mantissas and
// 8 + 8 bytes of limbs out; cols % 4 == 0 and rows * cols < 2^31
__global__ void k_dfp_down_v4(const int64_t* __restrict__ P, int rows, int cols,
                              const unsigned long long* __restrict__ d_max, const int32_t* __restrict__ d_ea,
                              const int32_t* __restrict__ d_eb, int16_t* __restrict__ out16,
                              uint16_t* __restrict__ hi, uint16_t* __restrict__ lo, int ldl,
                              int32_t* __restrict__ d_exp_out, int32_t* __restrict__ d_exp_out2, int32_t* __restrict__ d_rs,
                              unsigned long long* __restrict__ d_abs_sum, int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    const unsigned long long m = *d_max;
    const int bl = m ? 64 - __clzll((long long)m) : 0;
    const int rs = bl > 15 ? bl - 15 : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int e = *d_ea + (d_eb ? *d_eb : 0) + rs;
        if (d_exp_out) *d_exp_out = e;
        if (d_exp_out2) *d_exp_out2 = e;
        if (d_rs) *d_rs = rs;
        if (e < -128 || e > 127) raise_device_error(err, ITO_ERR_EXPONENT);
    }
    const int groups = rows * (cols >> 2);
    const int gpr = cols >> 2;
    unsigned long long asum = 0;
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += gridDim.x * blockDim.x) {
        const int r = g / gpr, c = (g - r * gpr) << 2;
        const int64_t i0 = (int64_t)r * cols + c;
        const longlong2 p0 = __ldcs(reinterpret_cast<const longlong2*>(P + i0));
        const longlong2 p1 = __ldcs(reinterpret_cast<const longlong2*>(P + i0 + 2));
        const int64_t pv[4] = {p0.x, p0.y, p1.x, p1.y};
        int16_t v[4];
        uint16_t h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int32_t q = (int32_t)sat16s(rhu64(pv[k], rs));
            int32_t hh, ll;
            limb_split(q, hh, ll);
            asum += (unsigned long long)(q < 0 ? -q : q);
            v[k] = (int16_t)q;
            h[k] = int_to_bf16_bits(hh);
            l[k] = int_to_bf16_bits(ll);
        }
        *reinterpret_cast<uint2*>(out16 + i0) = *reinterpret_cast<const uint2*>(v);
        if (hi) {
            const int64_t o = (int64_t)r * ldl + c;
            *reinterpret_cast<uint2*>(hi + o) = *reinterpret_cast<const uint2*>(h);
            *reinterpret_cast<uint2*>(lo + o) = *reinterpret_cast<const uint2*>(l);
        }
    }
    if (d_abs_sum) add_abs_sum(d_abs_sum, asum);
}

static inline bool al(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int launch_dfp_down(const int64_t* P, int64_t rows, int64_t cols, const unsigned long long* d_max, const int32_t* d_ea,
                    const int32_t* d_eb, int16_t* out16, uint16_t* hi, uint16_t* lo, int64_t ldl, int32_t* d_exp_out,
                    int32_t* d_rs, cudaStream_t s, unsigned long long* d_abs_sum, int32_t* d_exp_out2)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    int* err = device_error_word();
    if (!err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    if (cols % 4 == 0 && rows * cols < (1LL << 31) && ldl % 4 == 0 && al(P, 16) && al(out16, 8) &&
        (!hi || (al(hi, 8) && al(lo, 8))))
        launch_pdl(k_dfp_down_v4, launch_grid_blocks(rows * cols / 4, 256), 256, 0, s, 
            P, (int)rows, (int)cols, d_max, d_ea, d_eb, out16, hi, lo, (int)ldl, d_exp_out, d_exp_out2, d_rs, d_abs_sum,
            err);
    else
        launch_pdl(k_dfp_down, launch_grid_blocks(rows * cols, 256), 256, 0, s, P, rows, cols, d_max, d_ea, d_eb, out16, hi,
                   lo, ldl, d_exp_out, d_exp_out2, d_rs, d_abs_sum, err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp down launch: %s", cudaGetErrorString(e));
}

// --------------------------------------------------- float <-> DFP16

// max |f| as float bits (non-negative floats order like their bit patterns)
__global__ void k_absmax_f32(const float* __restrict__ f, int64_t n, unsigned int* __restrict__ d_bits)
{
    griddep_wait();
    griddep_launch_dependents();
    uint32_t mx = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        mx = max(mx, __float_as_uint(f[i]) & 0x7fffffffu);
    block_atomic_max(d_bits, mx);
}

// frexp exponent e of a positive finite float given by its bits: m = frac * 2^e, frac in [0.5, 1)
__device__ __forceinline__ int frexp_exponent(uint32_t bits)
{
    const int ef = (int)(bits >> 23);
    if (ef != 0) return ef - 126;
    const uint32_t mant = bits & 0x7fffffu;             // subnormal: mant * 2^-149
    return (32 - __clz(mant)) - 149;
}

// section 3.1: the shared exponent comes from the absolute maximum's exponent:
// E = e - 15 so that |f| * 2^-E < 2^15; mantissas round to nearest even, saturate
__global__ void k_dfp_from_float(const float* __restrict__ f, int64_t n, const unsigned int* __restrict__ d_bits,
                                 int16_t* __restrict__ out, int32_t* __restrict__ d_exp, int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t bits = *d_bits;
    const int E = bits ? frexp_exponent(bits) - 15 : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *d_exp = E;
        if (bits >= 0x7f800000u) raise_device_error(err, ITO_ERR_ARG);      // inf or nan in the input
        if (E < -128 || E > 127) raise_device_error(err, ITO_ERR_EXPONENT);
    }
    const double sc = pow2d(-E);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int q = __double2int_rn((double)f[i] * sc);
        q = q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
        out[i] = (int16_t)q;
    }
}

__global__ void k_dfp_to_float(const int16_t* __restrict__ m, int64_t n, const int32_t* __restrict__ d_exp,
                               float* __restrict__ out)
{
    griddep_wait();
    griddep_launch_dependents();
    const double sc = pow2d(*d_exp);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __double2float_rn((double)m[i] * sc);
}

// float(P) (round to nearest even) times 2^(Ea + Eb), one more rounding at most
__global__ void k_p64_to_float(const int64_t* __restrict__ P, int64_t n, const int32_t* __restrict__ d_ea,
                               const int32_t* __restrict__ d_eb, float* __restrict__ out)
{
    griddep_wait();
    griddep_launch_dependents();
    const double sc = pow2d(*d_ea + *d_eb);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __double2float_rn((double)__ll2float_rn(P[i]) * sc);
}

int launch_dfp_from_float(const float* f, int64_t n, unsigned int* d_bits, int16_t* out, int32_t* d_exp, cudaStream_t s)
{
    if (n < 1) return ITO_OK;
    int* err = device_error_word();
    if (!err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    if (cudaMemsetAsync(d_bits, 0, sizeof(unsigned int), s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset");
    launch_pdl(k_absmax_f32, launch_grid_blocks(n, 256), 256, 0, s, f, n, d_bits);
    launch_pdl(k_dfp_from_float, launch_grid_blocks(n, 256), 256, 0, s, f, n, d_bits, out, d_exp, err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "float->dfp launch: %s", cudaGetErrorString(e));
}

// Blocked-DFP ("Mixed Precision Training...", section 3: several fine-grained
// exponents per tensor): every run of `block` consecutive elements of a row
// (the last one shorter when block does not divide cols) is converted like a
// DFP-16 tensor of its own. One warp per block: max |f| by a warp reduction,
// then E = e - 15 and round-to-nearest-even mantissas, saturated.
__global__ void k_bdfp_from_float(const float* __restrict__ f, int64_t rows, int64_t cols, int block,
                                  int16_t* __restrict__ out, int8_t* __restrict__ exps, int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t nb = (cols + block - 1) / block;
    const int64_t nblocks = rows * nb;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < nblocks; w += nwarps) {
        const int64_t r = w / nb, j = w - r * nb;
        const int64_t c0 = j * block;
        const int len = (int)(cols - c0 < block ? cols - c0 : block);
        const float* src = f + r * cols + c0;
        uint32_t mx = 0;
        for (int i = lane; i < len; i += 32) mx = max(mx, __float_as_uint(src[i]) & 0x7fffffffu);
        mx = __reduce_max_sync(0xffffffffu, mx);
        const int E = mx ? frexp_exponent(mx) - 15 : 0;
        if (lane == 0) {
            exps[w] = (int8_t)(E < -128 ? -128 : (E > 127 ? 127 : E));
            if (mx >= 0x7f800000u) raise_device_error(err, ITO_ERR_ARG);    // inf or nan in the input
            if (E < -128 || E > 127) raise_device_error(err, ITO_ERR_EXPONENT);
        }
        const double sc = pow2d(-E);
        int16_t* dst = out + r * cols + c0;
        for (int i = lane; i < len; i += 32) {
            int q = __double2int_rn((double)src[i] * sc);
            q = q > 32767 ? 32767 : (q < -32767 ? -32767 : q);
            dst[i] = (int16_t)q;
        }
    }
}

__global__ void k_bdfp_to_float(const int16_t* __restrict__ m, const int8_t* __restrict__ exps, int64_t rows,
                                int64_t cols, int block, float* __restrict__ out)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t nb = (cols + block - 1) / block;
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        out[i] = __double2float_rn((double)m[i] * pow2d(exps[r * nb + c / block]));
    }
}

int launch_bdfp_from_float(const float* f, int64_t rows, int64_t cols, int block, int16_t* out, int8_t* exps,
                           cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    int* err = device_error_word();
    if (!err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    const int64_t nblocks = rows * ((cols + block - 1) / block);
    launch_pdl(k_bdfp_from_float, launch_grid_blocks(nblocks * 32, 256), 256, 0, s, f, rows, cols, block, out, exps, err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "float->bdfp launch: %s", cudaGetErrorString(e));
}

int launch_bdfp_to_float(const int16_t* m, const int8_t* exps, int64_t rows, int64_t cols, int block, float* out,
                         cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    launch_pdl(k_bdfp_to_float, launch_grid_blocks(rows * cols, 256), 256, 0, s, m, exps, rows, cols, block, out);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "bdfp->float launch: %s", cudaGetErrorString(e));
}

int launch_dfp_to_float(const int16_t* m, int64_t n, const int32_t* d_exp, float* out, cudaStream_t s)
{
    if (n < 1) return ITO_OK;
    launch_pdl(k_dfp_to_float, launch_grid_blocks(n, 256), 256, 0, s, m, n, d_exp, out);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp->float launch: %s", cudaGetErrorString(e));
}

int launch_p64_to_float(const int64_t* P, int64_t n, const int32_t* d_ea, const int32_t* d_eb, float* out,
                        cudaStream_t s)
{
    if (n < 1) return ITO_OK;
    launch_pdl(k_p64_to_float, launch_grid_blocks(n, 256), 256, 0, s, P, n, d_ea, d_eb, out);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "p64->float launch: %s", cudaGetErrorString(e));
}

// ----------------------------------------------------------------- update

__global__ void k_dfp_update(int16_t* __restrict__ W, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                             int64_t ldl, const int16_t* __restrict__ G, int64_t rows, int64_t cols,
                             const int32_t* __restrict__ d_exp_g, int32_t exp_w, int32_t eta, int32_t lim,
                             int32_t* __restrict__ d_k, uint32_t* __restrict__ d_nonzero)
{
    griddep_wait();
    griddep_launch_dependents();
    // W * 2^Ew <- W * 2^Ew - G * 2^Eg * 2^-eta  =>  dW = G * 2^-(Ew + eta - Eg); W saturates to +-lim
    const int k = exp_w + eta - *d_exp_g;
    if (d_k && blockIdx.x == 0 && threadIdx.x == 0) *d_k = k;
    uint32_t cnt = 0;
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = G[i];
        // a left shift past 17 bits already saturates every difference
        const int64_t dw = k >= 0 ? rhu64(g, k) : g * ((int64_t)1 << (-k > 17 ? 17 : -k));
        cnt += dw != 0;
        const int64_t d = (int64_t)W[i] - dw;
        const int32_t w = (int32_t)(d > lim ? lim : (d < -lim ? -lim : d));
        W[i] = (int16_t)w;
        if (hi) {
            const int64_t r = i / cols, c = i - r * cols;
            int32_t h, l;
            limb_split(w, h, l);
            hi[r * ldl + c] = int_to_bf16_bits(h);
            lo[r * ldl + c] = int_to_bf16_bits(l);
        }
    }
    if (d_nonzero) block_atomic_add(d_nonzero, cnt);
}

// four weights per thread step; cols % 4 == 0 and rows * cols < 2^31
__global__ void k_dfp_update_v4(int16_t* __restrict__ W, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                                int ldl, const int16_t* __restrict__ G, int rows, int cols,
                                const int32_t* __restrict__ d_exp_g, int32_t exp_w, int32_t eta, int32_t lim,
                                int32_t* __restrict__ d_k, uint32_t* __restrict__ d_nonzero)
{
    griddep_wait();
    griddep_launch_dependents();
    const int k = exp_w + eta - *d_exp_g;
    if (d_k && blockIdx.x == 0 && threadIdx.x == 0) *d_k = k;
    const int kl = -k > 17 ? 17 : -k;     // a left shift past 17 bits saturates every difference anyway
    uint32_t cnt = 0;
    const int gpr = cols >> 2;
    const int groups = rows * gpr;
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += gridDim.x * blockDim.x) {
        const int r = g / gpr, c = (g - r * gpr) << 2;
        const int64_t i0 = (int64_t)r * cols + c;
        int16_t w[4], gv[4];
        *reinterpret_cast<uint2*>(w) = *reinterpret_cast<const uint2*>(W + i0);
        *reinterpret_cast<uint2*>(gv) = __ldcs(reinterpret_cast<const uint2*>(G + i0));
        uint16_t h[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t dw = k >= 0 ? rhu64(gv[j], k) : (int64_t)gv[j] * ((int64_t)1 << kl);
            cnt += dw != 0;
            const int64_t d = (int64_t)w[j] - dw;
            const int32_t nw = (int32_t)(d > lim ? lim : (d < -lim ? -lim : d));
            int32_t hh, ll;
            limb_split(nw, hh, ll);
            w[j] = (int16_t)nw;
            h[j] = int_to_bf16_bits(hh);
            l[j] = int_to_bf16_bits(ll);
        }
        *reinterpret_cast<uint2*>(W + i0) = *reinterpret_cast<const uint2*>(w);
        if (hi) {
            const int64_t o = (int64_t)r * ldl + c;
            *reinterpret_cast<uint2*>(hi + o) = *reinterpret_cast<const uint2*>(h);
            *reinterpret_cast<uint2*>(lo + o) = *reinterpret_cast<const uint2*>(l);
        }
    }
    if (d_nonzero) block_atomic_add(d_nonzero, cnt);
}

int launch_dfp_update(int16_t* W, uint16_t* hi, uint16_t* lo, int64_t ldl, const int16_t* G, int64_t rows,
                      int64_t cols, const int32_t* d_exp_g, int32_t exp_w, int32_t eta, int32_t* d_k,
                      uint32_t* d_nonzero, cudaStream_t s, int bits)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    if (bits < 2 || bits > 16) return set_error(ITO_ERR_ARG, "weight precision must be 2 .. 16 bits");
    const int32_t lim = (1 << (bits - 1)) - 1;
    if (cols % 4 == 0 && rows * cols < (1LL << 31) && ldl % 4 == 0 && al(W, 8) && al(G, 8) &&
        (!hi || (al(hi, 8) && al(lo, 8))))
        launch_pdl(k_dfp_update_v4, launch_grid_blocks(rows * cols / 4, 256), 256, 0, s, 
            W, hi, lo, (int)ldl, G, (int)rows, (int)cols, d_exp_g, exp_w, eta, lim, d_k, d_nonzero);
    else
        launch_pdl(k_dfp_update, launch_grid_blocks(rows * cols, 256), 256, 0, s, W, hi, lo, ldl, G, rows, cols, d_exp_g,
                                                                           exp_w, eta, lim, d_k, d_nonzero);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp update launch: %s", cudaGetErrorString(e));
}

// ------------------------------------------------------ precision change
//
// "Adaptive Precision Training for Resource Constrained Devices", Algorithm 1
// changes a layer's weight precision by one bit at a time. With the weights
// held as bits-bit mantissas and one shared exponent, a change by d bits is
// W * 2^d (d > 0, every value kept exactly; the exponent drops by d) or
// round-half-up of W / 2^-d saturated to the new range (d < 0; the exponent
// rises by -d). The bf16 limb planes are rewritten too.
__global__ void k_dfp_set_bits(int16_t* __restrict__ W, uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                               int64_t ldl, int64_t rows, int64_t cols, int d, int32_t lim)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t v = d >= 0 ? (int64_t)W[i] * ((int64_t)1 << d) : rhu64(W[i], -d);
        const int32_t w = (int32_t)(v > lim ? lim : (v < -lim ? -lim : v));
        W[i] = (int16_t)w;
        if (hi) {
            const int64_t r = i / cols, c = i - r * cols;
            int32_t h, l;
            limb_split(w, h, l);
            hi[r * ldl + c] = int_to_bf16_bits(h);
            lo[r * ldl + c] = int_to_bf16_bits(l);
        }
    }
}

int launch_dfp_set_bits(int16_t* W, uint16_t* hi, uint16_t* lo, int64_t ldl, int64_t rows, int64_t cols,
                        int bits_old, int bits_new, cudaStream_t s)
{
    if (bits_old < 2 || bits_old > 16 || bits_new < 2 || bits_new > 16)
        return set_error(ITO_ERR_ARG, "weight precision must be 2 .. 16 bits");
    if (rows < 1 || cols < 1 || bits_old == bits_new) return ITO_OK;
    launch_pdl(k_dfp_set_bits, launch_grid_blocks(rows * cols, 256), 256, 0, s, W, hi, lo, ldl, rows, cols,
                                                                       bits_new - bits_old, (1 << (bits_new - 1)) - 1);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "precision change launch: %s", cudaGetErrorString(e));
}

}  // namespace ito
