// Bandwidth-bound kernels of the NITI step: requantisation of the int32
// contraction results (with ReLU or a ReLU gate), the NITI weight update, the
// top error, and int8 -> bf16 operand conversion. Each reads the per-tensor
// max written by the contraction epilogue (the grid-wide dependency of NITI
// Step 1 is the kernel boundary between them) and streams its tensor once,
// eight elements per thread step with 16-byte accesses where the row length
// allows.
//
// Rules: "Integer On-Device Training: Overview", section 3 "The NITI
// Algorithm", Steps 1-5 (per-tensor max, bits_needed, shift, round-half-up,
// weight_shift = shift - mu_weight, sat_int8 update) and the delta
// propagation note (target_bits = 7).
#include <cstdarg>
#include <cstdio>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

int launch_grid_blocks(int64_t work_items, int threads)
{
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = kNumSMsHint;
    }
    int64_t b = (work_items + threads - 1) / threads;
    int64_t cap = (int64_t)sms * 8;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (int)b;
}

static inline bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Offset of element i of a [rows][cols] tensor in a copy with row pitch ld; no division when
// the copy is unpadded (ld == cols, the same for every thread of a launch).
__device__ __forceinline__ int64_t pitched(int64_t i, int64_t cols, int64_t ld)
{
    if (ld == cols) return i;
    const int64_t r = i / cols;
    return r * ld + (i - r * cols);
}

// ------------------------------------------------------------- conversion

__global__ void k_i8_to_bf16_v8(const int8_t* __restrict__ src, int64_t rows, int64_t cols,
                                uint16_t* __restrict__ dst, int64_t ldd)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t groups = rows * (cols >> 3);
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = g << 3;
        const int64_t off = pitched(i0, cols, ldd);
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(src + i0));
        const int8_t* b = reinterpret_cast<const int8_t*>(&v);
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            ow[i] = int_pair_to_bf16x2(b[2 * i], b[2 * i + 1]);
        *reinterpret_cast<uint4*>(dst + off) = o;
    }
}

__global__ void k_i8_to_bf16_1(const int8_t* __restrict__ src, int64_t rows, int64_t cols, uint16_t* __restrict__ dst,
                               int64_t ldd)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        dst[pitched(i, cols, ldd)] = int_to_bf16_bits(src[i]);
    }
}

int launch_i8_to_bf16(const int8_t* src, int64_t rows, int64_t cols, uint16_t* dst, int64_t ldd, cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    if (cols % 8 == 0 && ldd % 8 == 0 && aligned(src, 8) && aligned(dst, 16))
        launch_pdl(k_i8_to_bf16_v8, launch_grid_blocks(rows * cols / 8, 256), 256, 0, s, src, rows, cols, dst, ldd);
    else
        launch_pdl(k_i8_to_bf16_1, launch_grid_blocks(rows * cols, 256), 256, 0, s, src, rows, cols, dst, ldd);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "convert launch: %s", cudaGetErrorString(e));
}

// --------------------------------------------------------------- requant

// q = sat8(rhu(y, s)); ReLU; gate
__device__ __forceinline__ int32_t requant_one(int32_t y, int s, int relu, int gate_ok)
{
    int32_t q = sat8(rhu32(y, s));
    if (relu && q < 0) q = 0;
    return gate_ok ? q : 0;
}

// The optional bit-packed ReLU masks hold one byte per eight elements of a
// row (cols / 8 bytes per row; bit j is element j of the group): mask_out
// receives (q > 0) of the result, gate_bits replaces the int8 gate.
// s_last (optional) receives the shift (a model's prediction of the same tensor's
// shift in the next step, for the speculative requantisation of FusedRq).
__global__ void k_requant_v8(const int32_t* __restrict__ Y, int64_t rows, int64_t cols,
                             const uint32_t* __restrict__ d_max, int target_bits, int relu,
                             const int8_t* __restrict__ gate, int8_t* __restrict__ out8, uint16_t* __restrict__ outb,
                             int64_t ldb, int32_t* __restrict__ d_shift, const uint8_t* __restrict__ gate_bits,
                             uint8_t* __restrict__ mask_out, int32_t* __restrict__ s_last, TopErr te)
{
    griddep_wait();
    griddep_launch_dependents();
    const int s = shift_for(*d_max, target_bits);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (d_shift) *d_shift = s;
        if (s_last) *s_last = s;
    }
    const int64_t groups = rows * (cols >> 3);
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = g << 3;
        const int4 y0 = __ldcs(reinterpret_cast<const int4*>(Y + i0));
        const int4 y1 = __ldcs(reinterpret_cast<const int4*>(Y + i0 + 4));
        const int32_t y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        int8_t gv[8] = {1, 1, 1, 1, 1, 1, 1, 1};
        if (gate) *reinterpret_cast<uint2*>(gv) = __ldg(reinterpret_cast<const uint2*>(gate + i0));
        if (gate_bits) {
            const uint32_t bits = __ldg(gate_bits + g);
#pragma unroll
            for (int i = 0; i < 8; ++i) gv[i] = (bits >> i) & 1;
        }
        int8_t q8[8];
        uint32_t qb[4];
        uint32_t mbits = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q8[i] = (int8_t)requant_one(y[i], s, relu, gv[i] > 0);
            mbits |= (q8[i] > 0 ? 1u : 0u) << i;
        }
        if (mask_out) mask_out[g] = (uint8_t)mbits;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            qb[i] = int_pair_to_bf16x2(q8[2 * i], q8[2 * i + 1]);
        *reinterpret_cast<uint2*>(out8 + i0) = *reinterpret_cast<const uint2*>(q8);
        if (outb) {
            *reinterpret_cast<uint4*>(outb + pitched(i0, cols, ldb)) = make_uint4(qb[0], qb[1], qb[2], qb[3]);
        }
        if (te.labels) {
            // the top error of these eight logits (as k_top_error_v8)
            const int64_t row = i0 / cols;
            const int64_t c0 = i0 - row * cols;
            const int label = te.labels[row];
            if (c0 == 0 && (label < 0 || label >= cols)) raise_device_error(te.err, ITO_ERR_ARG);
            int8_t d[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) d[i] = (int8_t)sat8((int32_t)q8[i] - (c0 + i == label ? te.target_mag : 0));
            *reinterpret_cast<uint2*>(te.e8 + i0) = *reinterpret_cast<const uint2*>(d);
            if (te.eb)
                *reinterpret_cast<uint4*>(te.eb + pitched(i0, cols, te.lde)) =
                    make_uint4(int_pair_to_bf16x2(d[0], d[1]), int_pair_to_bf16x2(d[2], d[3]),
                               int_pair_to_bf16x2(d[4], d[5]), int_pair_to_bf16x2(d[6], d[7]));
        }
    }
}

__global__ void k_requant_1(const int32_t* __restrict__ Y, int64_t rows, int64_t cols,
                            const uint32_t* __restrict__ d_max, int target_bits, int relu,
                            const int8_t* __restrict__ gate, int8_t* __restrict__ out8, uint16_t* __restrict__ outb,
                            int64_t ldb, int32_t* __restrict__ d_shift, int32_t* __restrict__ s_last, TopErr te)
{
    griddep_wait();
    griddep_launch_dependents();
    const int s = shift_for(*d_max, target_bits);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (d_shift) *d_shift = s;
        if (s_last) *s_last = s;
    }
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t q = requant_one(Y[i], s, relu, gate ? gate[i] > 0 : 1);
        out8[i] = (int8_t)q;
        if (outb) {
            outb[pitched(i, cols, ldb)] = int_to_bf16_bits(q);
        }
        if (te.labels) {
            // the top error of this logit (as k_top_error)
            const int64_t row = i / cols, c = i - row * cols;
            const int label = te.labels[row];
            if (c == 0 && (label < 0 || label >= cols)) raise_device_error(te.err, ITO_ERR_ARG);
            const int32_t d = sat8(q - (c == label ? te.target_mag : 0));
            te.e8[i] = (int8_t)d;
            if (te.eb) te.eb[pitched(i, cols, te.lde)] = int_to_bf16_bits(d);
        }
    }
}

int launch_requant(const int32_t* Y, int64_t rows, int64_t cols, const uint32_t* d_max, int target_bits, int relu,
                   const int8_t* gate, int8_t* out8, uint16_t* outb, int64_t ldb, int32_t* d_shift, cudaStream_t s,
                   const uint8_t* gate_bits, uint8_t* mask_out, int32_t* s_last, const TopErr* top)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    TopErr te{};
    if (top) {
        te = *top;
        te.err = device_error_word();
        if (!te.err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    }
    const bool vec = cols % 8 == 0 && aligned(Y, 16) && aligned(out8, 8) && (!gate || aligned(gate, 8)) &&
                     (!outb || (aligned(outb, 16) && ldb % 8 == 0)) &&
                     (!top || (aligned(te.e8, 8) && (!te.eb || (aligned(te.eb, 16) && te.lde % 8 == 0))));
    if ((gate_bits || mask_out) && !vec)
        return set_error(ITO_ERR_UNSUPPORTED, "bit-packed masks need rows of a multiple of 8 elements");
    if (vec)
        launch_pdl(k_requant_v8, launch_grid_blocks(rows * cols / 8, 256), 256, 0, s, Y, rows, cols, d_max,
                   target_bits, relu, gate, out8, outb, ldb, d_shift, gate_bits, mask_out, s_last, te);
    else
        launch_pdl(k_requant_1, launch_grid_blocks(rows * cols, 256), 256, 0, s, Y, rows, cols, d_max, target_bits,
                   relu, gate, out8, outb, ldb, d_shift, s_last, te);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "requant launch: %s", cudaGetErrorString(e));
}

// --------------------------------------------- start of a step

// The start of a training (or inference) step in one launch: the step's statistics block
// zeroed and, for n_pred > 0, the shift predictions rolled by block 0, and a Linear first
// layer's int8 or uint8 (a partial model's input from a frozen prefix; 0..255, exact in
// bf16) input converted to its bf16 copy by all blocks (x == nullptr: none). Rolling the
// predictions first scores the previous step's speculation: over the slots a contraction
// epilogue speculated on (used[i] != 0, pred[i] >= 0), count[0] += the predictions that
// held (pred[i] == last[i], the shift that step computed) and count[1] += the ones that did
// not (both int64); then pred[i] = last[i] where used and on, else -1 (no speculation).
__global__ void k_step_begin(int32_t* __restrict__ stats, int n_stats, int32_t* __restrict__ pred,
                             const int32_t* __restrict__ last, const int32_t* __restrict__ used,
                             unsigned long long* __restrict__ count, int n_pred, int on, const void* __restrict__ x,
                             int x_u8, int64_t rows, int64_t cols, uint16_t* __restrict__ xb, int64_t ldx, int vec)
{
    griddep_wait();
    griddep_launch_dependents();
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < n_stats; i += blockDim.x) stats[i] = 0;
        if (threadIdx.x < 32 && n_pred > 0) {
            unsigned hits = 0, misses = 0;
            for (int i = threadIdx.x; i < n_pred; i += 32) {
                const int32_t p = pred[i], l = last[i];
                const bool u = used[i] != 0;
                if (u && p >= 0) {
                    hits += p == l;
                    misses += p != l;
                }
                pred[i] = (on && u) ? l : -1;
            }
            hits = __reduce_add_sync(0xffffffffu, hits);
            misses = __reduce_add_sync(0xffffffffu, misses);
            if (threadIdx.x == 0) {
                count[0] += hits;
                count[1] += misses;
            }
        }
    }
    if (!x) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (vec) {
        const int64_t groups = rows * (cols >> 3);
        for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups; g += stride) {
            const int64_t i0 = g << 3;
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(x) + i0));
            const uint8_t* b = reinterpret_cast<const uint8_t*>(&v);
            int32_t t[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = x_u8 ? (int32_t)b[k] : (int32_t)(int8_t)b[k];
            *reinterpret_cast<uint4*>(xb + pitched(i0, cols, ldx)) =
                make_uint4(int_pair_to_bf16x2(t[0], t[1]), int_pair_to_bf16x2(t[2], t[3]),
                           int_pair_to_bf16x2(t[4], t[5]), int_pair_to_bf16x2(t[6], t[7]));
        }
    } else {
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < rows * cols; i += stride) {
            const uint8_t b = static_cast<const uint8_t*>(x)[i];
            xb[pitched(i, cols, ldx)] = int_to_bf16_bits(x_u8 ? (int32_t)b : (int32_t)(int8_t)b);
        }
    }
}

int launch_step_begin(int32_t* stats, int n_stats, int32_t* pred, const int32_t* last, const int32_t* used,
                      int64_t* count, int n_pred, int on, const void* x, int x_u8, int64_t rows, int64_t cols,
                      uint16_t* xb, int64_t ldx, cudaStream_t s)
{
    const bool vec = x && cols % 8 == 0 && ldx % 8 == 0 && aligned(x, 8) && aligned(xb, 16);
    const int blocks = x ? launch_grid_blocks(vec ? rows * cols / 8 : rows * cols, 256) : 1;
    launch_pdl(k_step_begin, blocks, 256, 0, s, stats, n_stats, pred, last, used,
               reinterpret_cast<unsigned long long*>(count), n_pred, on, x, x_u8, rows, cols, xb, ldx, vec ? 1 : 0);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "step start launch: %s", cudaGetErrorString(e));
}

// ------------------------------------------- static requantisation + offsets

// out = clip(floor((Y + offset[c]) * mult[c] / 2^k[c]), relu ? 0 : -128, 127)
// ("Integer On-Device Training: Overview", section 4: INT32 offsets and const
// k / mult arrays; the exported chain Add(offset) -> Mul -> Mul -> Floor -> Clip)
__device__ __forceinline__ int32_t static_one(int32_t y, int32_t off, int32_t mult, int32_t k, int32_t lo)
{
    const int64_t v = ((int64_t)y + off) * (int64_t)mult;
    int64_t q = v >> k;                   // arithmetic shift = floor division by 2^k
    q = q < lo ? lo : (q > 127 ? 127 : q);
    return (int32_t)q;
}

__global__ void k_requant_static_v8(const int32_t* __restrict__ Y, int64_t rows, int64_t cols,
                                    const int32_t* __restrict__ off, const int32_t* __restrict__ mult,
                                    const int32_t* __restrict__ ksh, int relu, int8_t* __restrict__ out8,
                                    uint16_t* __restrict__ outb, int64_t ldb, uint8_t* __restrict__ mask_out)
{
    griddep_wait();
    griddep_launch_dependents();
    const int32_t lo = relu ? 0 : -128;
    const int64_t groups = rows * (cols >> 3);
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = g << 3;
        const int64_t r = i0 / cols, c = i0 - r * cols;
        const int4 y0 = __ldcs(reinterpret_cast<const int4*>(Y + i0));
        const int4 y1 = __ldcs(reinterpret_cast<const int4*>(Y + i0 + 4));
        const int32_t y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        int8_t q8[8];
        uint32_t qb[4], mbits = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            q8[i] = (int8_t)static_one(y[i], __ldg(off + c + i), __ldg(mult + c + i), __ldg(ksh + c + i), lo);
            mbits |= (q8[i] > 0 ? 1u : 0u) << i;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            qb[i] = int_pair_to_bf16x2(q8[2 * i], q8[2 * i + 1]);
        *reinterpret_cast<uint2*>(out8 + i0) = *reinterpret_cast<const uint2*>(q8);
        if (outb) *reinterpret_cast<uint4*>(outb + r * ldb + c) = make_uint4(qb[0], qb[1], qb[2], qb[3]);
        if (mask_out) mask_out[g] = (uint8_t)mbits;
    }
}

__global__ void k_requant_static_1(const int32_t* __restrict__ Y, int64_t rows, int64_t cols,
                                   const int32_t* __restrict__ off, const int32_t* __restrict__ mult,
                                   const int32_t* __restrict__ ksh, int relu, int8_t* __restrict__ out8,
                                   uint16_t* __restrict__ outb, int64_t ldb)
{
    griddep_wait();
    griddep_launch_dependents();
    const int32_t lo = relu ? 0 : -128;
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        const int32_t q = static_one(Y[i], off[c], mult[c], ksh[c], lo);
        out8[i] = (int8_t)q;
        if (outb) outb[r * ldb + c] = int_to_bf16_bits(q);
    }
}

int launch_requant_static(const int32_t* Y, int64_t rows, int64_t cols, const int32_t* off, const int32_t* mult,
                          const int32_t* ksh, int relu, int8_t* out8, uint16_t* outb, int64_t ldb, uint8_t* mask_out,
                          cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    const bool vec = cols % 8 == 0 && aligned(Y, 16) && aligned(out8, 8) && (!outb || (aligned(outb, 16) && ldb % 8 == 0));
    if (mask_out && !vec) return set_error(ITO_ERR_UNSUPPORTED, "bit-packed masks need rows of a multiple of 8");
    if (vec)
        launch_pdl(k_requant_static_v8, launch_grid_blocks(rows * cols / 8, 256), 256, 0, s, Y, rows, cols, off, mult, ksh,
                                                                                      relu, out8, outb, ldb, mask_out);
    else
        launch_pdl(k_requant_static_1, launch_grid_blocks(rows * cols, 256), 256, 0, s, Y, rows, cols, off, mult, ksh, relu,
                                                                                 out8, outb, ldb);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "static requant launch: %s", cudaGetErrorString(e));
}

// g[c] = sum over rows of delta[r][c] (the offsets' gradient); max |g| into *d_max
__global__ void k_offset_grad(const int8_t* __restrict__ delta, int64_t rows, int64_t cols, int32_t* __restrict__ g,
                              uint32_t* __restrict__ d_max)
{
    griddep_wait();
    griddep_launch_dependents();
    uint32_t mx = 0;
    for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < cols; c += (int64_t)gridDim.x * blockDim.x) {
        int32_t acc = 0;
        for (int64_t r = 0; r < rows; ++r) acc += delta[r * cols + c];
        g[c] = acc;
        mx = max(mx, abs_u32(acc));
    }
    block_atomic_max(d_max, mx);
}

// NITI Steps 2-5 on INT32 offsets, saturating to int32
__global__ void k_offset_update(int32_t* __restrict__ off, const int32_t* __restrict__ g, int64_t n,
                                const uint32_t* __restrict__ d_max, int target_bits, int mu_weight,
                                int32_t* __restrict__ d_shift, int32_t* __restrict__ d_wshift,
                                uint32_t* __restrict__ d_nonzero)
{
    griddep_wait();
    griddep_launch_dependents();
    const int s = shift_for(*d_max, target_bits);
    const int ws = s - mu_weight > 0 ? s - mu_weight : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (d_shift) *d_shift = s;
        if (d_wshift) *d_wshift = ws;
    }
    uint32_t cnt = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t d = rhu32(sat8(rhu32(g[i], s)), ws);
        cnt += d != 0;
        int64_t v = (int64_t)off[i] - d;
        v = v < INT32_MIN ? INT32_MIN : (v > INT32_MAX ? INT32_MAX : v);
        off[i] = (int32_t)v;
    }
    if (d_nonzero) block_atomic_add(d_nonzero, cnt);
}

int launch_offset_grad_update(const int8_t* delta, int64_t rows, int64_t cols, int32_t* g, uint32_t* d_max,
                              int32_t* off, int target_bits, int mu_weight, int32_t* d_shift, int32_t* d_wshift,
                              uint32_t* d_nonzero, cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    launch_pdl(k_offset_grad, launch_grid_blocks(cols, 256), 256, 0, s, delta, rows, cols, g, d_max);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "offset grad launch: %s", cudaGetErrorString(e));
    launch_pdl(k_offset_update, launch_grid_blocks(cols, 256), 256, 0, s, off, g, cols, d_max, target_bits, mu_weight, d_shift,
                                                                  d_wshift, d_nonzero);
    e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "offset update launch: %s", cudaGetErrorString(e));
}

// ------------------------------------------------------------ NITI update

// weight_delta of Steps 3-4: round(sat8(round(G >> s)) >> ws); the operand
// of the second shift is G_quantized, as the step is written.
__device__ __forceinline__ int32_t niti_step_delta(int32_t g, int s, int ws)
{
    const int32_t gq = sat8(rhu32(g, s));     // Step 3
    return rhu32(gq, ws);                     // Step 4
}

__device__ __forceinline__ void count_nonzero(uint32_t cnt, uint32_t* d_nonzero)
{
    block_atomic_add(d_nonzero, cnt);
}

// Steps 3-5 for eight consecutive weights from their loaded gradients and weights:
// stores the new weights and their bf16 copy, returns how many moved.
__device__ __forceinline__ uint32_t niti_update_group(int8_t* __restrict__ W, uint16_t* __restrict__ Wb, int64_t ldb,
                                                      int64_t cols, int64_t i0, int4 g0, int4 g1, uint2 wold, int s,
                                                      int ws)
{
    const int32_t gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    int8_t w8[8];
    *reinterpret_cast<uint2*>(w8) = wold;
    uint32_t cnt = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int32_t dw = niti_step_delta(gv[i], s, ws);
        cnt += dw != 0;
        w8[i] = (int8_t)sat8(w8[i] - dw);          // Step 5
    }
    *reinterpret_cast<uint2*>(W + i0) = *reinterpret_cast<const uint2*>(w8);
    if (Wb) {
        uint32_t wb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wb[i] = int_pair_to_bf16x2(w8[2 * i], w8[2 * i + 1]);
        *reinterpret_cast<uint4*>(Wb + pitched(i0, cols, ldb)) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
    return cnt;
}

// Two groups of eight per thread and iteration: both groups' loads are issued before either
// is computed, so that more bytes are in flight per thread.
__global__ void k_niti_update_v8(int8_t* __restrict__ W, uint16_t* __restrict__ Wb, int64_t ldb,
                                 const int32_t* __restrict__ G, int64_t rows, int64_t cols,
                                 const uint32_t* __restrict__ d_max, int target_bits, int mu_weight,
                                 int32_t* __restrict__ d_shift, int32_t* __restrict__ d_wshift,
                                 uint32_t* __restrict__ d_nonzero)
{
    griddep_wait();
    griddep_launch_dependents();
    const int s = shift_for(*d_max, target_bits);
    const int ws = s - mu_weight > 0 ? s - mu_weight : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (d_shift) *d_shift = s;
        if (d_wshift) *d_wshift = ws;
    }
    uint32_t cnt = 0;
    const int64_t groups = rows * (cols >> 3);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < groups; g += 2 * stride) {
        const int64_t gb = g + stride;
        const int64_t ia = g << 3, ib = gb << 3;
        const int4 a0 = __ldcs(reinterpret_cast<const int4*>(G + ia));
        const int4 a1 = __ldcs(reinterpret_cast<const int4*>(G + ia + 4));
        const uint2 wa = *reinterpret_cast<const uint2*>(W + ia);
        int4 b0 = make_int4(0, 0, 0, 0), b1 = b0;
        uint2 wb = make_uint2(0, 0);
        if (gb < groups) {
            b0 = __ldcs(reinterpret_cast<const int4*>(G + ib));
            b1 = __ldcs(reinterpret_cast<const int4*>(G + ib + 4));
            wb = *reinterpret_cast<const uint2*>(W + ib);
        }
        cnt += niti_update_group(W, Wb, ldb, cols, ia, a0, a1, wa, s, ws);
        if (gb < groups) cnt += niti_update_group(W, Wb, ldb, cols, ib, b0, b1, wb, s, ws);
    }
    if (d_nonzero) count_nonzero(cnt, d_nonzero);
}

__global__ void k_niti_update_1(int8_t* __restrict__ W, uint16_t* __restrict__ Wb, int64_t ldb,
                                const int32_t* __restrict__ G, int64_t rows, int64_t cols,
                                const uint32_t* __restrict__ d_max, int target_bits, int mu_weight,
                                int32_t* __restrict__ d_shift, int32_t* __restrict__ d_wshift,
                                uint32_t* __restrict__ d_nonzero)
{
    griddep_wait();
    griddep_launch_dependents();
    const int s = shift_for(*d_max, target_bits);
    const int ws = s - mu_weight > 0 ? s - mu_weight : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (d_shift) *d_shift = s;
        if (d_wshift) *d_wshift = ws;
    }
    uint32_t cnt = 0;
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t dw = niti_step_delta(G[i], s, ws);
        cnt += dw != 0;
        const int8_t nw = (int8_t)sat8(W[i] - dw);
        W[i] = nw;
        if (Wb) {
            Wb[pitched(i, cols, ldb)] = int_to_bf16_bits(nw);
        }
    }
    if (d_nonzero) count_nonzero(cnt, d_nonzero);
}

int launch_niti_update(int8_t* W, uint16_t* Wb, int64_t ldb, const int32_t* G, int64_t rows, int64_t cols,
                       const uint32_t* d_max, int target_bits, int mu_weight, int32_t* d_shift, int32_t* d_wshift,
                       uint32_t* d_nonzero, cudaStream_t s)
{
    if (rows < 1 || cols < 1) return ITO_OK;
    const bool vec = cols % 8 == 0 && aligned(W, 8) && aligned(G, 16) && (!Wb || (aligned(Wb, 16) && ldb % 8 == 0));
    if (vec)
        launch_pdl(k_niti_update_v8, launch_grid_blocks(rows * cols / 8, 256), 256, 0, s, 
            W, Wb, ldb, G, rows, cols, d_max, target_bits, mu_weight, d_shift, d_wshift, d_nonzero);
    else
        launch_pdl(k_niti_update_1, launch_grid_blocks(rows * cols, 256), 256, 0, s, 
            W, Wb, ldb, G, rows, cols, d_max, target_bits, mu_weight, d_shift, d_wshift, d_nonzero);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "update launch: %s", cudaGetErrorString(e));
}

// -------------------------------------------------------------- top error

// A label outside [0, C) has no class to take the target: the row is copied and
// ITO_ERR_ARG is recorded in the device error word (once per row, by the thread
// that handles the row's first class).
__global__ void k_top_error(const int8_t* __restrict__ logits, const int32_t* __restrict__ labels, int B, int C,
                            int target_mag, int8_t* __restrict__ delta, uint16_t* __restrict__ deltab, int64_t ldb,
                            int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t n = (int64_t)B * C;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i / C), j = (int)(i - (int64_t)b * C);
        if (j == 0 && (labels[b] < 0 || labels[b] >= C)) raise_device_error(err, ITO_ERR_ARG);
        const int32_t t = (labels[b] == j) ? target_mag : 0;
        const int32_t d = sat8((int32_t)logits[i] - t);
        delta[i] = (int8_t)d;
        if (deltab) deltab[(int64_t)b * ldb + j] = int_to_bf16_bits(d);
    }
}

// Rows of a multiple of 8 classes: a thread takes 8 consecutive logits of one row (one
// 8-byte load, one 8-byte and one 16-byte store); rows over blockIdx.y (strided past 65535).
__global__ void k_top_error_v8(const int8_t* __restrict__ logits, const int32_t* __restrict__ labels, int B, int C,
                               int target_mag, int8_t* __restrict__ delta, uint16_t* __restrict__ deltab, int64_t ldb,
                               int* __restrict__ err)
{
    griddep_wait();
    griddep_launch_dependents();
    const int groups = C >> 3;
    for (int b = blockIdx.y; b < B; b += gridDim.y) {
        const int label = labels[b];
        if (blockIdx.x == 0 && threadIdx.x == 0 && (label < 0 || label >= C)) raise_device_error(err, ITO_ERR_ARG);
        for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += gridDim.x * blockDim.x) {
            const int64_t i0 = (int64_t)b * C + 8 * g;
            int8_t v[8];
            *reinterpret_cast<uint2*>(v) = *reinterpret_cast<const uint2*>(logits + i0);
            int8_t d[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                d[k] = (int8_t)sat8((int32_t)v[k] - (8 * g + k == label ? target_mag : 0));
            *reinterpret_cast<uint2*>(delta + i0) = *reinterpret_cast<const uint2*>(d);
            if (deltab)
                *reinterpret_cast<uint4*>(deltab + (int64_t)b * ldb + 8 * g) =
                    make_uint4(int_pair_to_bf16x2(d[0], d[1]), int_pair_to_bf16x2(d[2], d[3]),
                               int_pair_to_bf16x2(d[4], d[5]), int_pair_to_bf16x2(d[6], d[7]));
        }
    }
}

int launch_top_error(const int8_t* logits, const int32_t* labels, int B, int C, int target_mag, int8_t* delta,
                     uint16_t* deltab, int64_t ldb, cudaStream_t s)
{
    if (B < 1 || C < 1) return ITO_OK;
    int* err = device_error_word();
    if (!err) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    const bool vec = C % 8 == 0 && aligned(logits, 8) && aligned(delta, 8) &&
                     (!deltab || (aligned(deltab, 16) && ldb % 8 == 0));
    if (vec) {
        const int groups = C / 8;
        const dim3 grid((groups + 127) / 128, B < 65535 ? B : 65535);
        launch_pdl(k_top_error_v8, grid, 128, 0, s, logits, labels, B, C, target_mag, delta, deltab, ldb, err);
    } else {
        launch_pdl(k_top_error, launch_grid_blocks((int64_t)B * C, 256), 256, 0, s, logits, labels, B, C, target_mag, delta,
                                                                             deltab, ldb, err);
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "top error launch: %s", cudaGetErrorString(e));
}

}  // namespace ito
