// Conv2D and global pooling support kernels for the integer CNN step
// ("Integer On-Device Training: Overview", section 7: Conv2D and Conv2D+ReLU
// layers, dense, groups = 1, dilation = 1). Activations are NHWC and conv
// weights [OC][3][3][IC] (TiGrIS "Compilation Pipeline", emission stage
// "Layout transpose"), so a 3x3 conv is a Linear layer over im2col patches
// with K = 9 * IC in (kh, kw, ic) order, padding 1.
//
//  im2col:  int8 NHWC input -> bf16 patch matrix [B*OH*OW][9*IC] (the
//           tensor-core operand; padding taps are 0)
//  col2im:  int32 patch-space delta [B*OH*OW][9*IC] -> int32 input-space delta
//           [B*H*W][IC], gathering the (at most 9) patch entries that came
//           from each input position; folds max |D| into an atomicMax. Integer
//           addition wraps modulo 2^32, so the gather order cannot change a
//           result that fits int32.
//  gap:     integer sum over the spatial positions (no division: the NITI
//           shift that follows rescales), with max |P|; backward broadcasts
//           the pooled delta to every position where the ReLU was open.
#include "ito_device.cuh"
#include "ito_internal.h"
#include "ito_conv.h"

namespace ito {

static inline bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static int launched(const char* what)
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- im2col

// one thread per (output pixel, tap, 8 channels); IC % 8 == 0
__global__ void k_im2col_v8(const int8_t* __restrict__ x, int B, int H, int W, int IC, int OH, int OW, int stride,
                            uint16_t* __restrict__ P, int64_t ldp)
{
    griddep_wait();
    griddep_launch_dependents();
    const int cg = IC >> 3;
    const int64_t n = (int64_t)B * OH * OW * 9 * cg;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(i % cg);
        const int64_t t = i / cg;
        const int tap = (int)(t % 9);
        const int64_t m = t / 9;
        const int ow = (int)(m % OW);
        const int oh = (int)((m / OW) % OH);
        const int b = (int)(m / ((int64_t)OW * OH));
        const int ih = oh * stride - 1 + tap / 3, iw = ow * stride - 1 + tap % 3;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (ih >= 0 && ih < H && iw >= 0 && iw < W) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + (((int64_t)b * H + ih) * W + iw) * IC + c8 * 8));
            const int8_t* q = reinterpret_cast<const int8_t*>(&v);
            o.x = (uint32_t)int_to_bf16_bits(q[0]) | ((uint32_t)int_to_bf16_bits(q[1]) << 16);
            o.y = (uint32_t)int_to_bf16_bits(q[2]) | ((uint32_t)int_to_bf16_bits(q[3]) << 16);
            o.z = (uint32_t)int_to_bf16_bits(q[4]) | ((uint32_t)int_to_bf16_bits(q[5]) << 16);
            o.w = (uint32_t)int_to_bf16_bits(q[6]) | ((uint32_t)int_to_bf16_bits(q[7]) << 16);
        }
        *reinterpret_cast<uint4*>(P + m * ldp + tap * IC + c8 * 8) = o;
    }
}

// one thread per patch-matrix element, including the pitch padding (written 0)
// one thread per patch row (output pixel) when IC % 8 != 0: its 9 * IC taps in (kh, kw, ic)
// order and the zero padding up to ldp, eight bf16 values per 16-byte store, the (tap, ic)
// position advanced by counting instead of dividing; ldp % 8 == 0 and P 16-byte aligned
__global__ void k_im2col_rows(const int8_t* __restrict__ x, int B, int H, int W, int IC, int OH, int OW, int stride,
                              uint16_t* __restrict__ P, int64_t ldp)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t rows = (int64_t)B * OH * OW;
    const int K = 9 * IC;
    for (int64_t m = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; m < rows; m += (int64_t)gridDim.x * blockDim.x) {
        const int ow = (int)(m % OW);
        const int64_t t = m / OW;
        const int oh = (int)(t % OH);
        const int b = (int)(t / OH);
        uint16_t* dst = P + m * ldp;
        int tap = 0, ic = 0;
        for (int k0 = 0; k0 < ldp; k0 += 8) {
            int v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                int val = 0;
                if (k0 + q < K) {
                    const int ih = oh * stride - 1 + tap / 3, iw = ow * stride - 1 + tap % 3;
                    if (ih >= 0 && ih < H && iw >= 0 && iw < W) val = x[(((int64_t)b * H + ih) * W + iw) * IC + ic];
                    if (++ic == IC) {
                        ic = 0;
                        ++tap;
                    }
                }
                v[q] = val;
            }
            *reinterpret_cast<uint4*>(dst + k0) = make_uint4(int_pair_to_bf16x2(v[0], v[1]), int_pair_to_bf16x2(v[2], v[3]),
                                                             int_pair_to_bf16x2(v[4], v[5]), int_pair_to_bf16x2(v[6], v[7]));
        }
    }
}

// one thread per patch element (any ldp or alignment)
__global__ void k_im2col_1(const int8_t* __restrict__ x, int B, int H, int W, int IC, int OH, int OW, int stride,
                           uint16_t* __restrict__ P, int64_t ldp)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t K = 9 * (int64_t)IC;
    const int64_t n = (int64_t)B * OH * OW * ldp;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k = i % ldp, m = i / ldp;
        int v = 0;
        if (k < K) {
            const int tap = (int)(k / IC), ic = (int)(k % IC);
            const int ow = (int)(m % OW);
            const int oh = (int)((m / OW) % OH);
            const int b = (int)(m / ((int64_t)OW * OH));
            const int ih = oh * stride - 1 + tap / 3, iw = ow * stride - 1 + tap % 3;
            if (ih >= 0 && ih < H && iw >= 0 && iw < W) v = x[(((int64_t)b * H + ih) * W + iw) * IC + ic];
        }
        P[i] = int_to_bf16_bits(v);
    }
}

int launch_im2col(const int8_t* x, int B, int H, int W, int IC, int OH, int OW, int stride, uint16_t* P, int64_t ldp,
                  cudaStream_t s)
{
    if (IC % 8 == 0 && ldp % 8 == 0 && aligned(x, 8) && aligned(P, 16)) {
        const int64_t n = (int64_t)B * OH * OW * 9 * (IC / 8);
        launch_pdl(k_im2col_v8, launch_grid_blocks(n, 256), 256, 0, s, x, B, H, W, IC, OH, OW, stride, P, ldp);
    } else if (ldp % 8 == 0 && aligned(P, 16)) {
        launch_pdl(k_im2col_rows, launch_grid_blocks((int64_t)B * OH * OW, 128), 128, 0, s, x, B, H, W, IC, OH, OW, stride, P,
                                                                                  ldp);
    } else {
        const int64_t n = (int64_t)B * OH * OW * ldp;
        launch_pdl(k_im2col_1, launch_grid_blocks(n, 256), 256, 0, s, x, B, H, W, IC, OH, OW, stride, P, ldp);
    }
    return launched("im2col");
}

// ---------------------------------------------------------------- col2im

// one thread per (input pixel, 8 channels); IC % 8 == 0, Dcol pitch 9*IC
__global__ void k_col2im_v8(const int32_t* __restrict__ Dcol, int B, int H, int W, int IC, int OH, int OW,
                            int stride, int32_t* __restrict__ D, uint32_t* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    const int cg = IC >> 3;
    const int64_t ldc = 9 * (int64_t)IC;
    const int64_t n = (int64_t)B * H * W * cg;
    uint32_t mx = 0;
    const bool narrow = n <= 0x7fffffff;   // 32-bit index arithmetic (the same for every thread)
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        int c8, iw, ih, b;
        int64_t pix;
        if (narrow) {
            const uint32_t u = (uint32_t)i, px = u / (uint32_t)cg, t = px / (uint32_t)W;
            c8 = (int)(u - px * (uint32_t)cg);
            iw = (int)(px - t * (uint32_t)W);
            ih = (int)(t % (uint32_t)H);
            b = (int)(t / (uint32_t)H);
            pix = px;
        } else {
            c8 = (int)(i % cg);
            pix = i / cg;
            iw = (int)(pix % W);
            ih = (int)((pix / W) % H);
            b = (int)(pix / ((int64_t)W * H));
        }
        int32_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int kh = 0; kh < 3; ++kh) {
            const int th = ih + 1 - kh;              // = oh * stride
            if (th < 0 || th % stride) continue;
            const int oh = th / stride;
            if (oh >= OH) continue;
#pragma unroll
            for (int kw = 0; kw < 3; ++kw) {
                const int tw = iw + 1 - kw;
                if (tw < 0 || tw % stride) continue;
                const int ow = tw / stride;
                if (ow >= OW) continue;
                const int32_t* src = Dcol + (((int64_t)b * OH + oh) * OW + ow) * ldc + (kh * 3 + kw) * IC + c8 * 8;
                const int4 v0 = __ldg(reinterpret_cast<const int4*>(src));
                const int4 v1 = __ldg(reinterpret_cast<const int4*>(src + 4));
                acc[0] += v0.x; acc[1] += v0.y; acc[2] += v0.z; acc[3] += v0.w;
                acc[4] += v1.x; acc[5] += v1.y; acc[6] += v1.z; acc[7] += v1.w;
            }
        }
        int32_t* dst = D + pix * IC + c8 * 8;
        *reinterpret_cast<int4*>(dst) = make_int4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<int4*>(dst + 4) = make_int4(acc[4], acc[5], acc[6], acc[7]);
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = max(mx, abs_u32(acc[j]));
    }
    block_atomic_max(d_max, mx);
}

// one thread per input-space element (any IC)
__global__ void k_col2im_1(const int32_t* __restrict__ Dcol, int B, int H, int W, int IC, int OH, int OW,
                           int stride, int32_t* __restrict__ D, uint32_t* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t ldc = 9 * (int64_t)IC;
    const int64_t n = (int64_t)B * H * W * IC;
    uint32_t mx = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int ic = (int)(i % IC);
        const int64_t pix = i / IC;
        const int iw = (int)(pix % W);
        const int ih = (int)((pix / W) % H);
        const int b = (int)(pix / ((int64_t)W * H));
        int32_t acc = 0;
        for (int kh = 0; kh < 3; ++kh) {
            const int th = ih + 1 - kh;
            if (th < 0 || th % stride) continue;
            const int oh = th / stride;
            if (oh >= OH) continue;
            for (int kw = 0; kw < 3; ++kw) {
                const int tw = iw + 1 - kw;
                if (tw < 0 || tw % stride) continue;
                const int ow = tw / stride;
                if (ow >= OW) continue;
                acc += __ldg(Dcol + (((int64_t)b * OH + oh) * OW + ow) * ldc + (kh * 3 + kw) * IC + ic);
            }
        }
        D[i] = acc;
        mx = max(mx, abs_u32(acc));
    }
    block_atomic_max(d_max, mx);
}

int launch_col2im(const int32_t* Dcol, int B, int H, int W, int IC, int OH, int OW, int stride, int32_t* D,
                  uint32_t* d_max, cudaStream_t s)
{
    if (IC % 8 == 0 && aligned(Dcol, 16) && aligned(D, 16)) {
        const int64_t n = (int64_t)B * H * W * (IC / 8);
        launch_pdl(k_col2im_v8, launch_grid_blocks(n, 256), 256, 0, s, Dcol, B, H, W, IC, OH, OW, stride, D, d_max);
    } else {
        const int64_t n = (int64_t)B * H * W * IC;
        launch_pdl(k_col2im_1, launch_grid_blocks(n, 256), 256, 0, s, Dcol, B, H, W, IC, OH, OW, stride, D, d_max);
    }
    return launched("col2im");
}

// ------------------------------------------------------------------ pooling

// P[b][c] = sum over HW positions of A[b][pos][c]; max |P|
__global__ void k_gap_fwd(const int8_t* __restrict__ A, int B, int HW, int C, int32_t* __restrict__ P,
                          uint32_t* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = (int64_t)B * C;
    uint32_t mx = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % C);
        const int64_t b = i / C;
        const int8_t* src = A + b * HW * C + c;
        // eight independent partial sums, so that eight loads are in flight per thread
        int32_t part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int p = 0;
        for (; p + 8 <= HW; p += 8) {
#pragma unroll
            for (int u = 0; u < 8; ++u) part[u] += src[(int64_t)(p + u) * C];
        }
        for (; p < HW; ++p) part[0] += src[(int64_t)p * C];
        int32_t acc = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += part[u];
        P[i] = acc;
        mx = max(mx, abs_u32(acc));
    }
    block_atomic_max(d_max, mx);
}

int launch_gap_fwd(const int8_t* A, int B, int HW, int C, int32_t* P, uint32_t* d_max, cudaStream_t s)
{
    launch_pdl(k_gap_fwd, launch_grid_blocks((int64_t)B * C, 256), 256, 0, s, A, B, HW, C, P, d_max);
    return launched("gap fwd");
}

// E[b][pos][c] = (A[b][pos][c] > 0) ? dP[b][c] : 0, plus bf16 copy (pitch C)
// C % 8 == 0, E 8-byte and Eb 16-byte aligned: eight channels of one position per thread
__global__ void k_gap_bwd_v8(const int8_t* __restrict__ dP, const int8_t* __restrict__ A, int B, int HW, int C,
                             int8_t* __restrict__ E, uint16_t* __restrict__ Eb)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t groups = (int64_t)B * HW * (C >> 3);
    const int cg = C >> 3;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups; g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = g / cg;                       // b * HW + p
        const int c0 = (int)(g - pos * cg) * 8;
        const int64_t b = pos / HW;
        const int64_t i0 = pos * C + c0;
        int8_t a[8], d[8], e[8];
        *reinterpret_cast<uint2*>(a) = __ldg(reinterpret_cast<const uint2*>(A + i0));
        *reinterpret_cast<uint2*>(d) = __ldg(reinterpret_cast<const uint2*>(dP + b * C + c0));
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = a[j] > 0 ? d[j] : (int8_t)0;
        *reinterpret_cast<uint2*>(E + i0) = *reinterpret_cast<const uint2*>(e);
        if (Eb)
            *reinterpret_cast<uint4*>(Eb + i0) = make_uint4(int_pair_to_bf16x2(e[0], e[1]), int_pair_to_bf16x2(e[2], e[3]),
                                                            int_pair_to_bf16x2(e[4], e[5]), int_pair_to_bf16x2(e[6], e[7]));
    }
}

__global__ void k_gap_bwd(const int8_t* __restrict__ dP, const int8_t* __restrict__ A, int B, int HW, int C,
                          int8_t* __restrict__ E, uint16_t* __restrict__ Eb)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = (int64_t)B * HW * C;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % C);
        const int64_t b = i / ((int64_t)HW * C);
        const int32_t v = A[i] > 0 ? dP[b * C + c] : 0;
        E[i] = (int8_t)v;
        if (Eb) Eb[i] = int_to_bf16_bits(v);
    }
}

int launch_gap_bwd(const int8_t* dP, const int8_t* A, int B, int HW, int C, int8_t* E, uint16_t* Eb, cudaStream_t s)
{
    if (C % 8 == 0 && aligned(A, 8) && aligned(dP, 8) && aligned(E, 8) && (!Eb || aligned(Eb, 16)))
        launch_pdl(k_gap_bwd_v8, launch_grid_blocks((int64_t)B * HW * C / 8, 256), 256, 0, s, dP, A, B, HW, C, E, Eb);
    else
        launch_pdl(k_gap_bwd, launch_grid_blocks((int64_t)B * HW * C, 256), 256, 0, s, dP, A, B, HW, C, E, Eb);
    return launched("gap bwd");
}

}  // namespace ito
