// Exact integer contractions C[M][N] = sum_k A(m,k) * B(n,k) for int8 data
// ("Integer On-Device Training: Overview", section 2.1: the training pass is
// dominated by multiply-accumulates across weight matrices; section 3: each
// contraction result G is an int32 tensor whose max |G| drives the shift).
//
// Tensor-core path (k_gemm_tc): sm_103a has no integer tcgen05 MMA kind, so the
// operands are bf16 tensors holding int8 values (every integer of magnitude
// <= 256 is exact in bf16) and the MMA accumulates in fp32 in tensor memory.
// Each product is at most 2^14 in magnitude, so a chunk of up to 1024
// products sums to at most 2^24: every partial sum is an integer that fp32
// represents exactly, whatever the order of additions. The K loop is cut
// into such chunks; after each chunk the epilogue warps read the fp32
// accumulator from tensor memory, convert it to int32 and add it into int32
// registers, while the MMA warp fills the other of two accumulator buffers.
// The epilogue of a tile writes the int32 tile and folds its max |C| into a
// global atomicMax (the first half of the grid-wide max of NITI Step 1).
//
// Operands are loaded by TMA with 128-byte swizzle, either K-major
// ([rows][K], K contiguous) or MN-major ([K][rows], rows contiguous), so the
// forward (x.W^T), delta-propagation (delta.W) and weight-gradient
// (delta^T.a) contractions read the same row-major tensors without any
// transpose pass.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cudaTypedefs.h>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

// The device error word of this library (one per device).
__device__ int g_device_error = 0;

int* device_error_word()
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

// ------------------------------------------------------------ tile schedule

struct TileSched {
    int num_m, num_n, group;
    __device__ __forceinline__ void coords(int t, int& tm, int& tn) const
    {
        // groups of `group` m-tiles sweep all n-tiles, so consecutive CTAs
        // share B tiles and a band of A tiles in L2
        const int per_group = group * num_n;
        const int g = t / per_group;
        const int first_m = g * group;
        const int gm = min(group, num_m - first_m);
        const int r = t - g * per_group;
        tm = first_m + r % gm;
        tn = r / gm;
    }
};

// Work list of the CTA-pair kernel: the first `full` tiles whole, then each of
// the remaining tiles (the last, partial wave) split along K into `parts`
// chunk-aligned pieces, so that the partial wave keeps more SMs busy. A piece
// writes its int32 partial tile to workspace slot `slot`; k_tail_reduce adds
// the pieces exactly afterwards.
struct WorkItem {
    int tile, c0, c1, slot;   // chunks [c0, c1); slot -1: a whole tile written to C
};

__device__ __forceinline__ WorkItem work_item(int w, int full, int parts, int num_chunks)
{
    if (w < full) return WorkItem{w, 0, num_chunks, -1};
    const int u = w - full;
    const int ti = u / parts, part = u - ti * parts;
    return WorkItem{full + ti, part * num_chunks / parts, (part + 1) * num_chunks / parts, u};
}

// ----------------------------------------------------- tensor-core kernel

template <int BN>
struct TcCfg {
    static constexpr int BM = 128;
    static constexpr int BK = 64;                          // 64 bf16 = one 128-byte swizzle row
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (192 * 1024) / STAGE_BYTES > 8 ? 8 : (192 * 1024) / STAGE_BYTES;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;    // producer warp, MMA warp, 8 epilogue warps
    static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
    static constexpr int STAGING_BYTES = EPI_WARPS * 4096;   // one 32x32 int32 store box per epilogue warp
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(TcCfg<BN>::THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS, int use_tma_store,
              int split_tma, int M, int N, int K, int chunk_kb,
              int splits, int kb_per_split, int64_t split_stride, int32_t* __restrict__ C, int64_t ldc,
              uint32_t* __restrict__ d_max, int* __restrict__ err)
{
    // Work item w covers output tile w / splits and the K slice w % splits; with
    // splits > 1 each slice writes an int32 partial tile at C + slice * split_stride
    // (no max; by TMA through tmS, the partials as [splits][M][N], when split_tma) and a
    // reduction kernel adds the slices.
    using Cfg = TcCfg<BN>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;                             // columns per epilogue warp
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem + STAGES * Cfg::STAGE_BYTES;     // 1024-aligned, for the swizzled store boxes
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* accf_bar = empty_bar + STAGES;   // [2] accumulator buffer filled
    uint64_t* acce_bar = accf_bar + 2;         // [2] accumulator buffer drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const TileSched sched{(M + BM - 1) / BM, (N + BN - 1) / BN, 16};
    const int num_items = sched.num_m * sched.num_n * splits;
    const int num_kb = (K + BK - 1) / BK;
    // K-block range and chunk count of work item w
    auto kb_range = [&](int w, int& lo, int& hi) {
        lo = (w % splits) * kb_per_split;
        hi = min(num_kb, lo + kb_per_split);
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
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
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
                int tm, tn, kb_lo, kb_hi;
                sched.coords(w / splits, tm, tn);
                kb_range(w, kb_lo, kb_hi);
                for (int kb = kb_lo; kb < kb_hi; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
                    uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sB = sA + Cfg::A_BYTES;
                    if (!A_MN) {
                        tma_load_2d(&tmA, &full_bar[stage], sA, kb * BK, tm * BM);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d(&tmA, &full_bar[stage], sA + j * 8192, tm * BM + j * 64, kb * BK);
                    }
                    if (!B_MN) {
                        tma_load_2d(&tmB, &full_bar[stage], sB, kb * BK, tn * BN);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(&tmB, &full_bar[stage], sB + j * 8192, tn * BN + j * 64, kb * BK);
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
                int kb_lo, kb_hi;
                kb_range(w, kb_lo, kb_hi);
                const int num_chunks = (kb_hi - kb_lo + chunk_kb - 1) / chunk_kb;
                for (int c = 0; ok && c < num_chunks; ++c) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb0 = kb_lo + c * chunk_kb;
                    const int kb1 = min(kb_hi, kb0 + chunk_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t b0 = a0 + Cfg::A_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            // K-major: the 16-element K step is 32 bytes inside the swizzled row;
                            // MN-major: it is 16 rows of 128 bytes
                            const uint64_t ad = A_MN ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                                     : smem_desc_sw128(a0 + k * 32, 16, 1024);
                            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                                     : smem_desc_sw128(b0 + k * 32, 16, 1024);
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
        // ---------------- epilogue: drain chunks into int32, then max + store
        const int e = warp - 2;
        const int quad = warp & 3;               // TMEM lanes this warp may access
        const int half = e >> 2;                 // which half of the tile's columns
        uint8_t* stg = staging + e * 4096;       // this warp's 32 x 32 int32 store box
        const uint32_t stg_row = smem_u32(stg) + lane * 128;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int w = blockIdx.x; ok && w < num_items; w += gridDim.x) {
            int tm, tn, kb_lo, kb_hi;
            sched.coords(w / splits, tm, tn);
            kb_range(w, kb_lo, kb_hi);
            const int num_chunks = (kb_hi - kb_lo + chunk_kb - 1) / chunk_kb;
            int32_t* Cw = C + (int64_t)(w % splits) * split_stride;
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int c = 0; c < num_chunks; ++c) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + half * HALF);
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
            // out-of-range rows and columns read zero-filled operands, so they hold 0
            uint32_t mx = 0;
#pragma unroll
            for (int i = 0; i < HALF; ++i) mx = max(mx, abs_u32(acc[i]));
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0 && mx != 0 && d_max) atomicMax(d_max, mx);
            const int row0 = tm * BM + quad * 32;
            const int col0 = tn * BN + half * HALF;
            if (use_tma_store || split_tma) {
                // 32 x 32 boxes through shared memory (128-byte swizzle: 16-byte chunk j of
                // row r sits at chunk j ^ (r % 8)), written out by TMA; the edges are clipped
#pragma unroll
                for (int g = 0; g < HALF / 32; ++g) {
                    if (row0 >= M || col0 + g * 32 >= N) continue;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), acc[g * 32 + 4 * j], acc[g * 32 + 4 * j + 1],
                                     acc[g * 32 + 4 * j + 2], acc[g * 32 + 4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (split_tma)
                            tma_store_3d(&tmS, stg, col0 + g * 32, row0, w % splits);
                        else
                            tma_store_2d(&tmC, stg, col0 + g * 32, row0);
                        bulk_commit();
                    }
                }
            } else {
                const int row = row0 + lane;
                if (row < M) {
                    int32_t* dst = Cw + (int64_t)row * ldc + col0;
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


// --------------------------------------------- CTA-pair tensor-core kernel
//
// A cluster of two CTAs on one TPC computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2: each CTA loads its 128 rows of A and its half (128
// rows) of the B tile, both halves' TMA loads complete on the leader CTA's
// barrier, the leader's single MMA thread issues the M = 256 MMAs, and each
// CTA's tensor memory receives its 128 rows of the accumulator. Per SM this
// halves the B bytes moved from L2 and stored in shared memory, so six 32 KB
// stages hold twice the MMA work of the single-CTA kernel's four 48 KB stages.
// Exactness and the epilogue are as in k_gemm_tc; both CTAs' epilogue warps
// release an accumulator buffer on the leader's barrier.

// Speculative requantisation in the pair kernel's epilogue (FusedRq.pred set).
// The first launch folds max|y| into d_max and writes no int32 result. When
// *pred >= 0 (the shift the same tensor had in the previous step) its epilogue
// writes q = sat8(rhu(y, *pred)) (ReLU'd, or zeroed where gate <= 0) as int8 and
// as bf16; when *pred < 0 (no prediction yet) it writes nothing else. A second
// launch of the same plan with FusedRq.redo set computes, in its prologue, the
// true shift s = max(0, bitlen(*d_max) - target_bits), records it (d_shift,
// s_last, and *redo = 0 when the prediction held, else s + 1), and returns at once
// when *pred == s; otherwise it recomputes the contraction and writes q with
// shift s (no max, no int32 result).
struct FusedRq {
    const int32_t* pred;   // predicted shift (device word; < 0: none this step); nullptr: off
    const int8_t* gate;    // [M][ldg] int8 ReLU gate, or nullptr
    int64_t ldg;
    int relu;
    // the re-launch (redo != nullptr): its record of this step's shift
    int32_t* redo;         // 0 = the prediction held, else the shift + 1
    int32_t* d_shift;      // the step's shift (statistics), may be null
    int32_t* s_last;       // the step's shift (the next step's prediction), may be null
    int target_bits;
};

struct Tc2Cfg {
    static constexpr int BM = 128;                          // rows of A per CTA (256 per pair)
    static constexpr int BN = 256;                          // columns per pair tile
    static constexpr int BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (BN / 2) * BK * 2;       // this CTA's half of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = 6;
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + EPI_WARPS * 32;
    static constexpr int TMEM_COLS = 512;                   // two 256-column fp32 accumulators
    static constexpr int STAGING_BYTES = EPI_WARPS * 4096;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
};

// Ten warps a CTA: three share one SM sub-partition's 16,384 registers, so a thread gets 168
template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(Tc2Cfg::THREADS, 1)
    k_gemm_tc2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
               const __grid_constant__ CUtensorMap tmO8, const __grid_constant__ CUtensorMap tmOB, FusedRq fz,
               int use_tma_store, int M, int N, int K, int chunk_kb, int group, int full_tiles, int parts,
               int32_t* __restrict__ C, int64_t ldc, uint32_t* __restrict__ d_max, int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    using Cfg = Tc2Cfg;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int HALF = BN / 2;
    constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, A_MN, B_MN);

    // the shift of a speculative requantisation (< 0: none). A re-launch first checks the
    // first launch's prediction against the step's max and returns, in every CTA alike,
    // when it held
    int sp = -1;
    if (fz.redo) {
        const int s_true = shift_for(*d_max, fz.target_bits);
        const int p = *fz.pred;
        const bool held = p >= 0 && p == s_true;
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            *fz.redo = held ? 0 : s_true + 1;
            if (fz.d_shift) *fz.d_shift = s_true;
            if (fz.s_last) *fz.s_last = s_true;
        }
        if (held) return;
        sp = s_true;
    } else if (fz.pred) {
        sp = *fz.pred;
    }

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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    const TileSched sched{(M + 2 * BM - 1) / (2 * BM), (N + BN - 1) / BN, group};
    const int num_tiles = sched.num_m * sched.num_n;
    const int num_kb = (K + BK - 1) / BK;
    const int num_chunks = (num_kb + chunk_kb - 1) / chunk_kb;
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
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs): loads complete on the leader's barrier
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = cluster; ok && w < total_work; w += nclusters) {
                const WorkItem wi = work_item(w, full_tiles, parts, num_chunks);
                int tm, tn;
                sched.coords(wi.tile, tm, tn);
                const int rowA = tm * 2 * BM + rank * BM;
                const int rowB = tn * BN + rank * (BN / 2);
                const int kb_end = min(num_kb, wi.c1 * chunk_kb);
                for (int kb = wi.c0 * chunk_kb; kb < kb_end; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag, err)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * Cfg::STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
                    uint8_t* sA = smem + stage * Cfg::STAGE_BYTES;
                    uint8_t* sB = sA + Cfg::A_BYTES;
                    if (!A_MN) {
                        tma_load_2d_pair(&tmA, fb, sA, kb * BK, rowA);
                    } else {
                        tma_load_2d_pair(&tmA, fb, sA, rowA, kb * BK);
                        tma_load_2d_pair(&tmA, fb, sA + 8192, rowA + 64, kb * BK);
                    }
                    if (!B_MN) {
                        tma_load_2d_pair(&tmB, fb, sB, kb * BK, rowB);
                    } else {
                        tma_load_2d_pair(&tmB, fb, sB, rowB, kb * BK);
                        tma_load_2d_pair(&tmB, fb, sB + 8192, rowB + 64, kb * BK);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: one thread of the leader CTA
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t buf_phase = 0;
            bool ok = true;
            for (int w = cluster; ok && w < total_work; w += nclusters) {
                const WorkItem wi = work_item(w, full_tiles, parts, num_chunks);
                for (int c = wi.c0; ok && c < wi.c1; ++c) {
                    if (!mbar_wait(&acce_bar[buf], buf_phase ^ 1, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                    const int kb0 = c * chunk_kb;
                    const int kb1 = min(num_kb, kb0 + chunk_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full_bar[stage], phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(smem + stage * Cfg::STAGE_BYTES);
                        const uint32_t b0 = a0 + Cfg::A_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint64_t ad = A_MN ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                                     : smem_desc_sw128(a0 + k * 32, 16, 1024);
                            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                                     : smem_desc_sw128(b0 + k * 32, 16, 1024);
                            tc_mma_bf16_pair(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
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
        uint8_t* stg = staging + e * 4096;
        const uint32_t stg_row = smem_u32(stg) + lane * 128;
        int buf = 0;
        uint32_t buf_phase = 0;
        bool ok = true;
        for (int w = cluster; ok && w < total_work; w += nclusters) {
            const WorkItem wi = work_item(w, full_tiles, parts, num_chunks);
            int tm, tn;
            sched.coords(wi.tile, tm, tn);
            const int row0 = tm * 2 * BM + (int)rank * BM + quad * 32;
            const int col0 = tn * BN + half * HALF;
            const bool fused = sp >= 0 && wi.slot < 0 && use_tma_store && row0 < M && col0 < N;
            if (fused && fz.gate) {
                // the gate tile (this warp's 32 rows x 128 int8 columns) into the staging buffer
                // while the accumulator is still being computed, in the swizzled layout the
                // stores use: coalesced 16-byte loads (lane L takes chunk L % 8 of rows
                // 4 i + L / 8); outside the tensor the gate reads 0
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
                const int cc = lane & 7, rr = lane >> 3;
                const bool col_in = col0 + cc * 16 < N;
                const int8_t* gsrc = fz.gate + (int64_t)(row0 + rr) * fz.ldg + col0 + cc * 16;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int4 gv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (h * 4 + i) * 4 + rr;
                        gv[i] = (col_in && row0 + r < M)
                                    ? __ldg(reinterpret_cast<const int4*>(gsrc + (int64_t)(r - rr) * fz.ldg))
                                    : make_int4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (h * 4 + i) * 4 + rr;
                        st_shared_v4(smem_u32(stg) + r * 128 + ((cc ^ (r & 7)) << 4), gv[i].x, gv[i].y, gv[i].z,
                                     gv[i].w);
                    }
                }
                __syncwarp();
            }
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int c = wi.c0; c < wi.c1; ++c) {
                if (!mbar_wait(&accf_bar[buf], buf_phase, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN + half * HALF);
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
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acce_bar[buf]), 0));
                if (++buf == 2) { buf = 0; buf_phase ^= 1; }
            }
            if (!ok) break;
            if (wi.slot >= 0) {
                // a piece of a split tile: its partial sum goes to workspace slot wi.slot
                // (rows slot * 256 .. +255 of the partials map); k_tail_reduce finishes it
                const int prow = wi.slot * 2 * BM + (int)rank * BM + quad * 32;
#pragma unroll
                for (int g = 0; g < HALF / 32; ++g) {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), acc[g * 32 + 4 * j], acc[g * 32 + 4 * j + 1],
                                     acc[g * 32 + 4 * j + 2], acc[g * 32 + 4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmP, stg, half * HALF + g * 32, prow);
                        bulk_commit();
                    }
                }
                continue;
            }
            if (!fz.redo) {
                uint32_t mx = 0;
#pragma unroll
                for (int i = 0; i < HALF; ++i) mx = max(mx, abs_u32(acc[i]));
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0 && mx != 0) atomicMax(d_max, mx);
            }
            if (fused) {
                // speculative requantisation: q = sat8(rhu(y, sp)), ReLU'd or zeroed where the
                // gate is closed, written over the staged gate tile (each lane reads and
                // rewrites only its own row's 16-byte chunks), then stored as one 32 x 128 int8
                // box and two 32 x 64 bf16 boxes; no int32 result
                // round half up as ((y >> (s - 1)) + 1) >> 1 (= floor((y + 2^(s-1)) / 2^s), and no
                // addition that could overflow), the identity for s = 0; then the int8 (or ReLU)
                // range; four results to a word
                const int sh1 = sp > 0 ? sp - 1 : 0, rnd = sp > 0 ? 1 : 0;
                const int qlo = fz.relu ? 0 : -128;
                uint32_t q8w[HALF / 4];      // the 128 int8 results, packed four to a word
#pragma unroll
                for (int k = 0; k < HALF / 4; ++k) {
                    int32_t q[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b) q[b] = min(max(((acc[4 * k + b] >> sh1) + rnd) >> rnd, qlo), 127);
                    q8w[k] = __byte_perm(__byte_perm((uint32_t)q[0], (uint32_t)q[1], 0x0040),
                                         __byte_perm((uint32_t)q[2], (uint32_t)q[3], 0x0040), 0x5410);
                }
                if (fz.gate) {
                    // zero where the staged gate byte is not positive
#pragma unroll
                    for (int j = 0; j < HALF / 16; ++j) {
                        const uint4 gv = ld_shared_v4(stg_row + ((j ^ (lane & 7)) << 4));
                        q8w[4 * j] &= bytes_positive_mask(gv.x);
                        q8w[4 * j + 1] &= bytes_positive_mask(gv.y);
                        q8w[4 * j + 2] &= bytes_positive_mask(gv.z);
                        q8w[4 * j + 3] &= bytes_positive_mask(gv.w);
                    }
                } else {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                }
#pragma unroll
                for (int j = 0; j < HALF / 16; ++j)
                    st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), (int32_t)q8w[4 * j], (int32_t)q8w[4 * j + 1],
                                 (int32_t)q8w[4 * j + 2], (int32_t)q8w[4 * j + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmO8, stg, col0, row0);
                    bulk_commit();
                }
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    if (col0 + g * 64 >= N) continue;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t wv[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int i = g * 64 + j * 8 + 2 * h;
                            const int8_t lo = (int8_t)(q8w[i >> 2] >> (8 * (i & 3)));
                            const int8_t hi = (int8_t)(q8w[(i + 1) >> 2] >> (8 * ((i + 1) & 3)));
                            wv[h] = int_pair_to_bf16x2(lo, hi);
                        }
                        st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), (int32_t)wv[0], (int32_t)wv[1],
                                     (int32_t)wv[2], (int32_t)wv[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOB, stg, col0 + g * 64, row0);
                        bulk_commit();
                    }
                }
            } else if (fz.pred) {
                // a speculating launch with no prediction yet: the max only (above); the
                // re-launch writes the outputs
            } else if (use_tma_store) {
                // the int32 result through the staging buffer, 32 x 32 boxes
#pragma unroll
                for (int g = 0; g < HALF / 32; ++g) {
                    if (row0 >= M || col0 + g * 32 >= N) continue;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stg_row + ((j ^ (lane & 7)) << 4), acc[g * 32 + 4 * j], acc[g * 32 + 4 * j + 1],
                                     acc[g * 32 + 4 * j + 2], acc[g * 32 + 4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, stg, col0 + g * 32, row0);
                        bulk_commit();
                    }
                }
            } else {
                const int row = row0 + lane;
                if (row < M) {
                    int32_t* dst = C + (int64_t)row * ldc + col0;
#pragma unroll
                    for (int i = 0; i < HALF; ++i)
                        if (col0 + i < N) dst[i] = acc[i];
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

// ------------------------------------------------------ failure self-test

// One CTA waits on an mbarrier that nothing completes: the bounded wait gives
// up after its time limit, records ITO_ERR_TIMEOUT in the error word and the
// kernel returns (the wait every pipeline barrier of the contractions uses).
__global__ void k_wait_timeout_selftest(int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err);
}

int launch_wait_timeout_selftest(cudaStream_t s)
{
    int* err = device_error_word();
    if (!err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    launch_pdl(k_wait_timeout_selftest, 1, 32, 0, s, err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
}

// ----------------------------------------------------------- host launchers

PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// rows x cols row-major bf16 tensor with `pitch` elements per row; box of
// box_cols (inner, 64 = 128 bytes) x box_rows, 128-byte swizzle, zero fill.
int make_map_bf16(CUtensorMap* map, const Bf16View& v, int box_rows)
{
    auto enc = get_encode();
    if (!enc) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    if ((reinterpret_cast<uintptr_t>(v.ptr) & 15) || ((v.pitch * 2) & 15))
        return set_error(ITO_ERR_ARG, "bf16 operand not 16-byte aligned");
    cuuint64_t dims[2] = {(cuuint64_t)v.cols, (cuuint64_t)v.rows};
    cuuint64_t strides[1] = {(cuuint64_t)v.pitch * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(v.ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ITO_OK;
}

int num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = kNumSMsHint;
    }
    return n;
}

// C[r][c] = sum over slices of P[s][r][c]; max |C| folded into *d_max. Integer
// addition wraps modulo 2^32, so the slice order cannot change a result that fits int32.
// C = the sum of the `splits` partial results (exact: integer addition modulo 2^32);
// max |C| folded into *d_max. A warp per group of outputs (four consecutive columns
// when the rows allow 16-byte loads, else one): its lanes load different slices, so
// every load of a group is in flight at once, and a shuffle tree adds the lanes'
// sums. Contractions split many ways over few outputs (a conv weight gradient: 147
// slices of 64 x 27 outputs) keep the whole grid busy this way.
__global__ void k_splitk_reduce(const int32_t* __restrict__ P, int splits, int64_t stride, int M, int N, int64_t ldc,
                                int32_t* __restrict__ C, uint32_t* __restrict__ d_max, int vec)
{
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int gpr = vec ? N >> 2 : N;   // groups per row
    const int64_t groups = (int64_t)M * gpr;
    uint32_t mx = 0;
    for (int64_t g = warp0; g < groups; g += nwarps) {
        const int64_t r = g / gpr;
        const int64_t off = r * ldc + (g - r * gpr) * (vec ? 4 : 1);
        if (vec) {
            int4 acc = make_int4(0, 0, 0, 0);
            for (int sl = lane; sl < splits; sl += 32) {
                const int4 v = __ldcs(reinterpret_cast<const int4*>(P + sl * stride + off));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
                acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
                acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
                acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
            }
            if (lane == 0) {
                *reinterpret_cast<int4*>(C + off) = acc;
                mx = max(max(max(mx, abs_u32(acc.x)), abs_u32(acc.y)), max(abs_u32(acc.z), abs_u32(acc.w)));
            }
        } else {
            int32_t acc = 0;
            for (int sl = lane; sl < splits; sl += 32) acc += __ldcs(P + sl * stride + off);
            acc = __reduce_add_sync(0xffffffffu, acc);
            if (lane == 0) {
                C[off] = acc;
                mx = max(mx, abs_u32(acc));
            }
        }
    }
    block_atomic_max(d_max, mx);
}

// The split tiles of the pair kernel's last wave: C = the sum of each tile's
// `parts` partial tiles (exact integer sums), written inside the M x N bounds;
// max |C| folded into *d_max. P holds [tail tiles][parts][256][256] int32.
__global__ void k_tail_reduce(const int32_t* __restrict__ P, int tail_tiles, int parts, int full_tiles,
                              TileSched sched, int M, int N, int64_t ldc, int32_t* __restrict__ C,
                              uint32_t* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    constexpr int T = 256;
    const int64_t n = (int64_t)tail_tiles * T * (T / 4);
    uint32_t mx = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int ti = (int)(i / (T * (T / 4)));
        const int rem = (int)(i - (int64_t)ti * (T * (T / 4)));
        const int r = rem / (T / 4), c = (rem % (T / 4)) * 4;
        int4 acc = make_int4(0, 0, 0, 0);
        for (int q = 0; q < parts; ++q) {
            const int4 v = __ldcs(reinterpret_cast<const int4*>(P + (((int64_t)ti * parts + q) * T + r) * T + c));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        int tm, tn;
        sched.coords(full_tiles + ti, tm, tn);
        const int gr = tm * T + r, gc = tn * T + c;
        if (gr < M) {
            const int32_t a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (gc + j < N) {
                    C[(int64_t)gr * ldc + gc + j] = a[j];
                    mx = max(mx, abs_u32(a[j]));
                }
        }
    }
    block_atomic_max(d_max, mx);
}

template <int BN, bool A_MN, bool B_MN>
static int launch_tc(const GemmPlan& p, cudaStream_t s)
{
    using Cfg = TcCfg<BN>;
    auto kern = k_gemm_tc<BN, A_MN, B_MN>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(cudaGetLastError()));
        attr_set = true;
    }
    const int items = ((p.M + Cfg::BM - 1) / Cfg::BM) * ((p.N + BN - 1) / BN) * p.splits;
    const int grid = items < num_sms() ? items : num_sms();
    const bool split = p.splits > 1;
    launch_pdl(kern, grid, Cfg::THREADS, Cfg::SMEM_BYTES, s, p.mapA, p.mapB, p.mapC, p.mapS,
               split ? 0 : p.use_tma_store, split ? p.split_tma : 0, p.M, p.N, p.K, p.chunk_kb, p.splits,
               p.kb_per_split, p.split_stride, split ? p.split_ws : p.C, p.ldc, split ? nullptr : p.d_max, p.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
    if (split) return launch_splitk_reduce(p.split_ws, p.splits, p.split_stride, p.M, p.N, p.ldc, p.C, p.d_max, s);
    return ITO_OK;
}

int launch_splitk_reduce(const int32_t* P, int splits, int64_t stride, int M, int N, int64_t ldc, int32_t* C,
                         uint32_t* d_max, cudaStream_t s)
{
    const int vec = N % 4 == 0 && ldc % 4 == 0 && stride % 4 == 0 && (reinterpret_cast<uintptr_t>(P) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    launch_pdl(k_splitk_reduce, launch_grid_blocks((int64_t)M * N / (vec ? 4 : 1) * 32, 256), 256, 0, s, P, splits,
               stride, M, N, ldc, C, d_max, vec);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "split-K reduce launch: %s", cudaGetErrorString(e));
}

// CTA pairs of k_gemm_tc2<A_MN, B_MN> that fit on the device at once (its
// persistent grid); sets the kernel's shared-memory limit on first use.
template <bool A_MN, bool B_MN>
static int pair_clusters()
{
    using Cfg = Tc2Cfg;
    auto kern = k_gemm_tc2<A_MN, B_MN>;
    static int max_clusters = 0;
    if (!max_clusters) {
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
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) return 0;
        max_clusters = n;
    }
    return max_clusters;
}

static int pair_clusters_for(bool a_mn, bool b_mn)
{
    if (!a_mn && !b_mn) return pair_clusters<false, false>();
    if (!a_mn && b_mn) return pair_clusters<false, true>();
    if (a_mn && b_mn) return pair_clusters<true, true>();
    return pair_clusters<true, false>();
}

// Tail split of a pair-kernel contraction: how many of the tiles run whole and
// into how many K pieces each remaining tile of the last, partial wave is cut.
// Estimated time: waves of whole tiles + rounds of pieces (each 1/parts of a
// tile), plus the reduction pass (the pieces written and read back once, at
// about 5 TB/s, and one launch). A tile takes 2 * 256 * 256 * K operations at
// about 23 TFLOP/s per CTA pair (the measured pair-kernel rate).
struct TailSplit {
    int full, parts;
};

static TailSplit tail_split(int tiles, int clusters, int num_chunks, int K)
{
    TailSplit best{tiles, 1};
    if (clusters < 1 || tiles % clusters == 0) return best;
    const int waves = tiles / clusters, r = tiles % clusters;
    const double tile_us = 2.0 * 256 * 256 * K / 23.0e6;
    double best_t = (waves + 1.0) * tile_us;
    for (int parts = 2; parts <= 4 && parts <= num_chunks; ++parts) {
        const double reduce_us = 3.0 + 2.0 * r * parts * 256.0 * 256 * 4 / 5.0e6;
        const double t = (waves + (double)((r * parts + clusters - 1) / clusters) / parts) * tile_us + reduce_us;
        if (t < best_t) {
            best_t = t;
            best = TailSplit{tiles - r, parts};
        }
    }
    return best;
}

static size_t tail_ws_bytes(const TailSplit& ts, int tiles)
{
    return ts.parts > 1 ? (size_t)(tiles - ts.full) * ts.parts * 256 * 256 * sizeof(int32_t) : 0;
}

template <bool A_MN, bool B_MN>
static int launch_tc2(const GemmPlan& p, cudaStream_t s)
{
    using Cfg = Tc2Cfg;
    auto kern = k_gemm_tc2<A_MN, B_MN>;
    const int max_clusters = pair_clusters<A_MN, B_MN>();
    if (!max_clusters) return set_error(ITO_ERR_CUDA, "no CTA pair fits on this device");
    const int tiles = ((p.M + 255) / 256) * ((p.N + 255) / 256);
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
    const FusedRq fz{p.rq_pred, p.rq_gate, p.rq_ldg, p.rq_relu, p.rq_redo, p.rq_d_shift, p.rq_s_last, p.rq_target_bits};
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p.mapA, p.mapB, p.mapC, p.mapP, p.mapO8, p.mapOB, fz,
                                       p.use_tma_store, p.M, p.N, p.K, p.chunk_kb, p.group, p.tail_full, p.tail_parts,
                                       p.C, p.ldc, p.d_max, p.err);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "pair gemm launch: %s", cudaGetErrorString(e));
    if (p.tail_parts > 1) {
        const TileSched sched{(p.M + 255) / 256, (p.N + 255) / 256, p.group};
        const int tail = tiles - p.tail_full;
        launch_pdl(k_tail_reduce, launch_grid_blocks((int64_t)tail * 256 * 64, 256), 256, 0, s, 
            p.split_ws, tail, p.tail_parts, p.tail_full, sched, p.M, p.N, p.ldc, p.C, p.d_max);
        e = cudaGetLastError();
        if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "tail reduce launch: %s", cudaGetErrorString(e));
    }
    return ITO_OK;
}

// Tile width of the single-CTA kernel for N output columns: the fewest computed
// columns, a 64-column tile counted one and a half times (its B tile is too
// narrow to keep the MMA fed from shared memory); ties go to the wider tile.
// N = 576 takes 128 (640 columns computed, against 768 at 256).
static int choose_bn(int N)
{
    int best = 256;
    int64_t best_cost = INT64_MAX;
    for (int bn = 256; bn >= 64; bn /= 2) {
        const int64_t cols = (int64_t)((N + bn - 1) / bn) * bn;
        const int64_t cost = bn == 64 ? 3 * cols : 2 * cols;
        if (cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// K slices for a contraction with few output tiles and a long K on the
// single-CTA kernel (1 = no split): enough work items to cover the SMs, each
// slice at least one K block.
static int split_count(int M, int N, int K)
{
    const int bn = choose_bn(N);
    const int tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
    const int num_kb = (K + 63) / 64;
    if (num_kb < 32 || 2 * tiles > num_sms()) return 1;
    int splits = num_sms() / tiles;
    if (splits > num_kb) splits = num_kb;
    const int per = (num_kb + splits - 1) / splits;
    return (num_kb + per - 1) / per;
}

static bool pair_eligible(int M, int N, int splits, int min_pair_tiles = 1)
{
    const int pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    return M >= 256 && N >= 256 && splits == 1 && pair_tiles >= min_pair_tiles;
}

size_t gemm_split_ws_bytes(int M, int N, int K, int64_t ldc)
{
    const int s = split_count(M, N, K);
    if (s > 1) return (size_t)s * M * ldc * sizeof(int32_t);
    if (!pair_eligible(M, N, s)) return 0;
    // pair kernel: partial tiles of the split last wave (operand layouts share one occupancy)
    const int tiles = ((M + 255) / 256) * ((N + 255) / 256);
    const int num_chunks = ((K + 63) / 64 + kExactChunk / 64 - 1) / (kExactChunk / 64);
    return tail_ws_bytes(tail_split(tiles, pair_clusters_for(false, false), num_chunks, K), tiles);
}

int gemm_plan(GemmPlan* p, const Bf16View& A, bool a_mn, const Bf16View& B, bool b_mn, int M, int N, int K,
              int32_t* C, int64_t ldc, uint32_t* d_max, int32_t* split_ws, size_t split_ws_bytes, int chunk_terms,
              int min_pair_tiles)
{
    if (chunk_terms < 64 || chunk_terms > kExactChunk || chunk_terms % 64)
        return set_error(ITO_ERR_ARG, "gemm: exact chunk must be a multiple of 64 up to %d", kExactChunk);
    if (M < 1 || N < 1 || K < 1) return set_error(ITO_ERR_SHAPE, "gemm: empty contraction");
    if (K > (1 << 20)) return set_error(ITO_ERR_SHAPE, "gemm: contraction longer than 2^20");
    // operand extents must match the problem
    if (a_mn ? (A.rows != K || A.cols != M) : (A.rows != M || A.cols != K))
        return set_error(ITO_ERR_SHAPE, "gemm: A view does not match M x K");
    if (b_mn ? (B.rows != K || B.cols != N) : (B.rows != N || B.cols != K))
        return set_error(ITO_ERR_SHAPE, "gemm: B view does not match N x K");
    memset(p, 0, sizeof(*p));
    p->M = M;
    p->N = N;
    p->K = K;
    p->a_mn = a_mn;
    p->b_mn = b_mn;
    p->C = C;
    p->ldc = ldc;
    p->d_max = d_max;
    p->chunk_kb = chunk_terms / 64;
    p->err = device_error_word();
    if (!p->err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    p->bn = choose_bn(N);
    // CTA-pair kernel for large tiles
    p->splits = 1;
    p->kb_per_split = (K + 63) / 64;
    const int splits = split_count(M, N, K);
    if (splits > 1 && split_ws && split_ws_bytes >= (size_t)splits * M * ldc * sizeof(int32_t)) {
        const int num_kb = (K + 63) / 64;
        p->splits = splits;
        p->kb_per_split = (num_kb + splits - 1) / splits;
        p->split_ws = split_ws;
        p->split_stride = (int64_t)M * ldc;
    }
    p->pair = pair_eligible(M, N, p->splits, min_pair_tiles);
    // few output tiles on the single-CTA kernel: narrower tiles (down to 64 columns) while
    // they still fit in one wave put more SMs to work on the same contraction
    if (!p->pair && p->splits == 1)
        while (p->bn > 64 && ((M + 127) / 128) * ((N + p->bn / 2 - 1) / (p->bn / 2)) <= num_sms()) p->bn /= 2;
    // tiles are rastered in groups of 16 row tiles
    p->group = 16;
    // pair kernel: split the last partial wave along K when the workspace holds the partial tiles
    p->tail_full = ((M + 255) / 256) * ((N + 255) / 256);
    p->tail_parts = 1;
    if (p->pair && split_ws) {
        const int tiles = p->tail_full;
        const int num_chunks = ((K + 63) / 64 + p->chunk_kb - 1) / p->chunk_kb;
        const int clusters = pair_clusters_for(a_mn, b_mn);
        if (!clusters) return set_error(ITO_ERR_CUDA, "no CTA pair fits on this device");
        const TailSplit ts = tail_split(tiles, clusters, num_chunks, K);
        const size_t need = tail_ws_bytes(ts, tiles);
        if (ts.parts > 1 && need <= split_ws_bytes) {
            p->tail_full = ts.full;
            p->tail_parts = ts.parts;
            p->split_ws = split_ws;
            auto enc = get_encode();
            cuuint64_t dims[2] = {256, (cuuint64_t)(tiles - ts.full) * ts.parts * 256};
            cuuint64_t strides[1] = {256 * 4};
            cuuint32_t box[2] = {32, 32};
            cuuint32_t estr[2] = {1, 1};
            CUresult cr = enc(&p->mapP, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, split_ws, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (cr != CUDA_SUCCESS)
                return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (partials) failed (%d)", (int)cr);
        }
    }
    int r = make_map_bf16(&p->mapA, A, a_mn ? 64 : 128);
    if (r) return r;
    // the pair kernel loads half of a 256-wide B tile per CTA
    r = make_map_bf16(&p->mapB, B, b_mn ? 64 : (p->pair ? 128 : p->bn));
    if (r) return r;
    // int32 output through TMA stores when its rows are 16-byte aligned; plain stores otherwise
    if (p->splits > 1 && (reinterpret_cast<uintptr_t>(p->split_ws) & 15) == 0 && (ldc & 3) == 0) {
        // the split partials [splits][M][N] (pitch ldc): a slice's 32-row boxes clip at its own M
        auto enc = get_encode();
        cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)p->splits};
        cuuint64_t strides[2] = {(cuuint64_t)ldc * 4, (cuuint64_t)p->split_stride * 4};
        cuuint32_t box[3] = {32, 32, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult cr = enc(&p->mapS, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, p->split_ws, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (partials) failed (%d)", (int)cr);
        p->split_tma = 1;
    }
    p->use_tma_store = 0;
    if ((reinterpret_cast<uintptr_t>(C) & 15) == 0 && (ldc & 3) == 0) {
        auto enc = get_encode();
        cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)ldc * 4};
        cuuint32_t box[2] = {32, 32};
        cuuint32_t estr[2] = {1, 1};
        CUresult cr = enc(&p->mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, C, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (C) failed (%d)", (int)cr);
        p->use_tma_store = 1;
    }
    return ITO_OK;
}

int gemm_plan_fuse_requant(GemmPlan* p, const int32_t* pred, int relu, const int8_t* gate, int64_t ldg,
                           int8_t* out8, int64_t ld8, uint16_t* outb, int64_t ldb)
{
    p->rq_pred = nullptr;
    // the pair kernel's TMA-store epilogue over whole tiles; int8 rows must be 16-byte multiples
    if (!p->pair || !p->use_tma_store || p->tail_parts != 1 || !pred || !out8 || !outb) return ITO_OK;
    if (p->N % 16 || ld8 % 16 || ldb % 8 || (reinterpret_cast<uintptr_t>(out8) & 15) ||
        (reinterpret_cast<uintptr_t>(outb) & 15))
        return ITO_OK;
    if (gate && (ldg % 16 || (reinterpret_cast<uintptr_t>(gate) & 15))) return ITO_OK;
    auto enc = get_encode();
    if (!enc) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint32_t estr[2] = {1, 1};
    {
        cuuint64_t dims[2] = {(cuuint64_t)p->N, (cuuint64_t)p->M};
        cuuint64_t strides[1] = {(cuuint64_t)ld8};
        cuuint32_t box[2] = {128, 32};
        CUresult cr = enc(&p->mapO8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, out8, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (int8 out) failed (%d)", (int)cr);
    }
    {
        cuuint64_t dims[2] = {(cuuint64_t)p->N, (cuuint64_t)p->M};
        cuuint64_t strides[1] = {(cuuint64_t)ldb * 2};
        cuuint32_t box[2] = {64, 32};
        CUresult cr = enc(&p->mapOB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, outb, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return set_error(ITO_ERR_CUDA, "cuTensorMapEncodeTiled (bf16 out) failed (%d)", (int)cr);
    }
    p->rq_pred = pred;
    p->rq_gate = gate;
    p->rq_ldg = ldg;
    p->rq_relu = relu;
    return ITO_OK;
}

int gemm_run(const GemmPlan& p, cudaStream_t s)
{
    if (p.pair) {
        if (!p.a_mn && !p.b_mn) return launch_tc2<false, false>(p, s);
        if (!p.a_mn && p.b_mn) return launch_tc2<false, true>(p, s);
        if (p.a_mn && p.b_mn) return launch_tc2<true, true>(p, s);
        return launch_tc2<true, false>(p, s);
    }
#define ITO_TC_CASE(BN)                                                            \
    if (p.bn == BN) {                                                              \
        if (!p.a_mn && !p.b_mn) return launch_tc<BN, false, false>(p, s);          \
        if (!p.a_mn && p.b_mn) return launch_tc<BN, false, true>(p, s);            \
        if (p.a_mn && p.b_mn) return launch_tc<BN, true, true>(p, s);              \
        return launch_tc<BN, true, false>(p, s);                                   \
    }
    ITO_TC_CASE(256)
    ITO_TC_CASE(128)
    ITO_TC_CASE(64)
#undef ITO_TC_CASE
    return set_error(ITO_ERR_ARG, "gemm: bad tile width");
}

}  // namespace ito
