// DFP16 single-layer entry points and the DFP16 model: a stack of Linear
// layers over dynamic-fixed-point tensors (int16 mantissas, one shared
// exponent per tensor) trained with integer-only arithmetic ("Mixed
// Precision Training of Convolutional Neural Networks using Integer
// Operations", sections 3 and 3.1; section 4 names the forward, backward and
// weight-gradient kernels, each of whose wide outputs is quantised for the
// next operation).
//
// Step (one reading, since the page fixes no loss or update rule): forward
// through all layers (no ReLU), each contraction down-converted to DFP16;
// top error = the output itself (an MSE error against a zero target);
// for each layer from the top down: delta propagation with the pre-update
// weights (not for the first layer), weight gradient, then integer SGD with
// rate 2^-eta on the mantissas: W <- sat16(W - G * 2^(Eg - eta - Ew)), with
// the weight exponent Ew held fixed.
//
// Exponents live on the device (int32 scalars) and are updated by the kernels
// that produce each tensor, so a step needs no host synchronisation.
//
// Adaptive precision ("Adaptive Precision Training for Resource Constrained
// Devices", section III): every layer's weights are bits-bit mantissas
// (2 <= bits <= 16) with their own exponent E_W; the update saturates to the
// layer's precision. With APT enabled, the weight-gradient down-conversion also
// sums |g| exactly, each evaluated step logs (sum|g|, E_G) per layer on the
// device, and ito_dfp16_model_apt_epoch_end applies Algorithm 1 to the mean
// Gavg of the epoch's evaluations (Algorithm 2: adjustment between epochs).
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

__global__ void k_set_i32(int32_t* p, int32_t v) {
    griddep_wait();
    griddep_launch_dependents(); *p = v; }
// The start of a DFP16 step: its statistics blocks zeroed and the input exponent set.
__global__ void k_dfp_step_begin(int32_t* __restrict__ s32, int n32, unsigned long long* __restrict__ s64, int n64,
                                 int32_t* __restrict__ ex, int32_t exp_x)
{
    griddep_wait();
    griddep_launch_dependents();
    for (int i = threadIdx.x; i < n32; i += blockDim.x) s32[i] = 0;
    for (int i = threadIdx.x; i < n64; i += blockDim.x) s64[i] = 0;
    if (threadIdx.x == 0) *ex = exp_x;
}

enum { D_EY = 0, D_EE, D_RS, D_RSD, D_RSG, D_EG, D_K, D_NZ, D_N32 };
enum { D_PMAX = 0, D_PDMAX, D_PGMAX, D_GABS, D_N64 };
constexpr int kAptMaxEvals = 256;   // logged Gavg evaluations per epoch

// copies this step's (sum |g|, E_G) of every layer into one log slot
__global__ void k_apt_log(const unsigned long long* __restrict__ s64, const int32_t* __restrict__ s32, int nl,
                          unsigned long long* __restrict__ log_abs, int32_t* __restrict__ log_eg)
{
    griddep_wait();
    griddep_launch_dependents();
    const int l = threadIdx.x;
    if (l < nl) {
        log_abs[l] = s64[l * D_N64 + D_GABS];
        log_eg[l] = s32[l * D_N32 + D_EG];
    }
}

struct DLayer {
    int IC, OC;
    int16_t* W = nullptr;
    uint16_t *Wh = nullptr, *Wl = nullptr;
    int64_t ldw = 0;
    int64_t* p64 = nullptr;
    int16_t* y16 = nullptr;
    uint16_t *yh = nullptr, *yl = nullptr;
    int64_t ldy = 0;
    int16_t* e16 = nullptr;     // delta at the output (the output itself for the top layer)
    uint16_t *eh = nullptr, *el = nullptr;
    int64_t* pd64 = nullptr;    // [B][IC]
    int64_t* pg64 = nullptr;    // [OC][IC]
    int16_t* g16 = nullptr;
    DfpGemmPlan pf{}, pd{}, pg{};
};

}  // namespace ito

struct ito_dfp16_model {
    int batch = 0, exp_w = 0, eta = 0;
    std::vector<ito::DLayer> L;
    std::vector<int32_t> wexp, wbits;  // per-layer weight exponent and precision (host copies)
    int32_t* wexp_d = nullptr;         // device copy of wexp
    bool apt = false;
    ito_apt_params ap{};
    int apt_step = 0, apt_nlog = 0;     // steps since the last epoch end; logged evaluations
    unsigned long long* log_abs = nullptr;
    int32_t* log_eg = nullptr;
    int64_t* tail_ws = nullptr;        // partial tiles of split last waves (shared by the step's contractions)
    size_t tail_ws_bytes = 0;
    // backward overlap: down-conversions of the propagated delta and of the weight gradient,
    // and the update, run on a second stream beside the next contraction
    bool overlap = true;
    cudaStream_t side = nullptr;
    std::vector<cudaEvent_t> sync_ev;  // [0] fork, [1] join, per layer: delta propagated, delta ready, wgrad done
    int16_t* x16 = nullptr;
    // pipelined host-path steps (ito_dfp16_train_step_host_async): a second input buffer, the
    // copy stream, per buffer "copied" / "read by its step" events, the statistics packed as
    // ito_dfp16_model_read_stats lays them out
    int16_t* x16b = nullptr;
    int64_t* stats_packed = nullptr;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_copied[2] = {nullptr, nullptr}, ev_consumed[2] = {nullptr, nullptr};
    int64_t async_steps = 0;
    uint16_t *xh = nullptr, *xl = nullptr;
    int64_t ldx = 0;
    int32_t* s32 = nullptr;            // [layers][D_N32] + [ex, ew]
    unsigned long long* s64 = nullptr; // [layers][D_N64]
    std::vector<void*> allocs;
    // per-kernel timing (ito_dfp16_model_profile): an event pair around every launch, on the
    // launch's stream; classes as ito_prof_class (the down-conversions count as requantisation)
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;
    std::vector<int> prof_cls;
    std::vector<double> prof_work;
    int prof_n = 0;
    int launches = 0;                  // kernels launched by the last step

    void mark_begin(cudaStream_t st)
    {
        ++launches;
        if (!prof_on) return;
        while (prof_ev.size() < (size_t)(2 * prof_n + 2)) {
            cudaEvent_t e;
            cudaEventCreate(&e);
            prof_ev.push_back(e);
        }
        cudaEventRecord(prof_ev[2 * prof_n], st);
    }
    void mark_end(cudaStream_t st, int cls, double work)
    {
        if (!prof_on) return;
        cudaEventRecord(prof_ev[2 * prof_n + 1], st);
        prof_cls.push_back(cls);
        prof_work.push_back(work);
        ++prof_n;
    }

    template <class T>
    int alloc(T** out, size_t count)
    {
        void* p = nullptr;
        if (count == 0) count = 1;
        cudaError_t e = cudaMalloc(&p, count * sizeof(T));
        if (e != cudaSuccess) return ito::set_error(ITO_ERR_CUDA, "cudaMalloc: %s", cudaGetErrorString(e));
        cudaMemset(p, 0, count * sizeof(T));
        allocs.push_back(p);
        *out = static_cast<T*>(p);
        return ITO_OK;
    }
    int32_t* i32(int l, int k) { return s32 + l * ito::D_N32 + k; }
    unsigned long long* u64(int l, int k) { return s64 + l * ito::D_N64 + k; }
    int32_t* ex() { return s32 + (int)L.size() * ito::D_N32; }
    int32_t* ew() { return s32 + (int)L.size() * ito::D_N32 + 1; }
};

using namespace ito;

#define ITO_TRY(x)                   \
    do {                             \
        int _r = (x);                \
        if (_r != ITO_OK) return _r; \
    } while (0)

// a model launch, bracketed by the profiling events when they are on
#define ITO_DLAUNCH(m, st, cls, work, call)      \
    do {                                         \
        (m)->mark_begin(st);                     \
        int _r = (call);                         \
        (m)->mark_end(st, cls, (double)(work));  \
        if (_r != ITO_OK) return _r;             \
    } while (0)

// executed bf16 operations of a limb contraction: four limb products per int16 multiply-add
static double dfp_gemm_ops(const DfpGemmPlan& g) { return 8.0 * g.M * (double)g.N * g.K; }

// kernels one dfp_gemm_run launches: the contraction, and the reduction of a split last wave
static int dfp_gemm_kernels(const DfpGemmPlan& g) { return 1 + ((g.pair && g.tail_parts > 1) ? 1 : 0); }

static inline size_t al256(size_t n) { return (n + 255) & ~size_t(255); }

// standalone workspace: limb planes of operand A (x or delta) and operand B (W or x)
static size_t dws_a(int B, int IC, int OC) { return al256((size_t)2 * 2 * B * pad8(IC > OC ? IC : OC)); }
static size_t dws_b(int B, int IC, int OC) { return al256((size_t)2 * 2 * (OC > B ? OC : B) * pad8(IC)); }
// partial tiles of a split last wave, for whichever of the three contractions needs most
static size_t dws_c(int B, int IC, int OC)
{
    const size_t a = dfp_split_ws_bytes(B, OC, IC), b = dfp_split_ws_bytes(B, IC, OC),
                 c = dfp_split_ws_bytes(OC, IC, B);
    return al256(a > b ? (a > c ? a : c) : (b > c ? b : c));
}
static int64_t* dws_tail(void* ws, int B, int IC, int OC)
{
    return reinterpret_cast<int64_t*>(static_cast<char*>(ws) + dws_a(B, IC, OC) + dws_b(B, IC, OC));
}

struct Planes {
    uint16_t *h, *l;
};

static Planes planes_at(void* base, size_t plane_elems)
{
    uint16_t* h = static_cast<uint16_t*>(base);
    return Planes{h, h + plane_elems};
}

static int dfp_check(const void* a, const void* b, const void* c, const void* d, int B, int IC, int OC, void* ws,
                     size_t ws_bytes)
{
    if (!a || !b || !c || !d) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (B < 1 || IC < 1 || OC < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    if (B > (1 << 20) || IC > (1 << 20) || OC > (1 << 20)) return set_error(ITO_ERR_SHAPE, "size above 2^20");
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return set_error(ITO_ERR_ARG, "workspace NULL or misaligned");
    if (ws_bytes < ito_dfp16_workspace_size(B, IC, OC)) return set_error(ITO_ERR_ARG, "workspace too small");
    return ITO_OK;
}

extern "C" {

size_t ito_dfp16_workspace_size(int B, int IC, int OC)
{
    if (B < 1 || IC < 1 || OC < 1) return 0;
    return dws_a(B, IC, OC) + dws_b(B, IC, OC) + dws_c(B, IC, OC);
}

int ito_dfp16_linear_fwd(const int16_t* x, const int32_t* d_exp_x, const int16_t* W, const int32_t* d_exp_w, int B,
                         int IC, int OC, void* workspace, size_t workspace_bytes, int64_t* p64, uint64_t* d_max,
                         int16_t* y, int32_t* d_exp_y, int32_t* d_rs, void* stream)
{
    ITO_TRY(dfp_check(x, W, p64, y, B, IC, OC, workspace, workspace_bytes));
    if (!d_exp_x || !d_exp_w || !d_max || !d_exp_y) return set_error(ITO_ERR_ARG, "NULL scalar pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t ld = pad8(IC);
    Planes xa = planes_at(workspace, (size_t)B * ld);
    Planes wb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)OC * ld);
    ITO_TRY(launch_i16_to_limbs(x, B, IC, xa.h, xa.l, ld, s));
    ITO_TRY(launch_i16_to_limbs(W, OC, IC, wb.h, wb.l, ld, s));
    if (cudaMemsetAsync(d_max, 0, 8, s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset");
    DfpGemmPlan g;
    ITO_TRY(dfp_gemm_plan(&g, Bf16View{xa.h, B, IC, ld}, Bf16View{xa.l, B, IC, ld}, false, Bf16View{wb.h, OC, IC, ld},
                          Bf16View{wb.l, OC, IC, ld}, false, B, OC, IC, p64, OC,
                          reinterpret_cast<unsigned long long*>(d_max), dws_tail(workspace, B, IC, OC),
                          dws_c(B, IC, OC)));
    ITO_TRY(dfp_gemm_run(g, s));
    return launch_dfp_down(p64, B, OC, reinterpret_cast<unsigned long long*>(d_max), d_exp_x, d_exp_w, y, nullptr,
                           nullptr, 0, d_exp_y, d_rs, s);
}

int ito_dfp16_linear_bwd_delta(const int16_t* delta, const int32_t* d_exp_delta, const int16_t* W,
                               const int32_t* d_exp_w, int B, int IC, int OC, void* workspace, size_t workspace_bytes,
                               int64_t* p64, uint64_t* d_max, int16_t* delta_prev, int32_t* d_exp_prev,
                               int32_t* d_rs, void* stream)
{
    ITO_TRY(dfp_check(delta, W, p64, delta_prev, B, IC, OC, workspace, workspace_bytes));
    if (!d_exp_delta || !d_exp_w || !d_max || !d_exp_prev) return set_error(ITO_ERR_ARG, "NULL scalar pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t lde = pad8(OC), ldw = pad8(IC);
    Planes ea = planes_at(workspace, (size_t)B * lde);
    Planes wb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)OC * ldw);
    ITO_TRY(launch_i16_to_limbs(delta, B, OC, ea.h, ea.l, lde, s));
    ITO_TRY(launch_i16_to_limbs(W, OC, IC, wb.h, wb.l, ldw, s));
    if (cudaMemsetAsync(d_max, 0, 8, s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset");
    DfpGemmPlan g;
    ITO_TRY(dfp_gemm_plan(&g, Bf16View{ea.h, B, OC, lde}, Bf16View{ea.l, B, OC, lde}, false,
                          Bf16View{wb.h, OC, IC, ldw}, Bf16View{wb.l, OC, IC, ldw}, true, B, IC, OC, p64, IC,
                          reinterpret_cast<unsigned long long*>(d_max), dws_tail(workspace, B, IC, OC),
                          dws_c(B, IC, OC)));
    ITO_TRY(dfp_gemm_run(g, s));
    return launch_dfp_down(p64, B, IC, reinterpret_cast<unsigned long long*>(d_max), d_exp_delta, d_exp_w, delta_prev,
                           nullptr, nullptr, 0, d_exp_prev, d_rs, s);
}

int ito_dfp16_linear_wgrad(const int16_t* delta, const int32_t* d_exp_delta, const int16_t* x, const int32_t* d_exp_x,
                           int B, int IC, int OC, void* workspace, size_t workspace_bytes, int64_t* p64,
                           uint64_t* d_max, int16_t* g, int32_t* d_exp_g, int32_t* d_rs, void* stream)
{
    ITO_TRY(dfp_check(delta, x, p64, g, B, IC, OC, workspace, workspace_bytes));
    if (!d_exp_delta || !d_exp_x || !d_max || !d_exp_g) return set_error(ITO_ERR_ARG, "NULL scalar pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t lde = pad8(OC), ldx = pad8(IC);
    Planes ea = planes_at(workspace, (size_t)B * lde);
    Planes xb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)B * ldx);
    ITO_TRY(launch_i16_to_limbs(delta, B, OC, ea.h, ea.l, lde, s));
    ITO_TRY(launch_i16_to_limbs(x, B, IC, xb.h, xb.l, ldx, s));
    if (cudaMemsetAsync(d_max, 0, 8, s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset");
    DfpGemmPlan gp;
    ITO_TRY(dfp_gemm_plan(&gp, Bf16View{ea.h, B, OC, lde}, Bf16View{ea.l, B, OC, lde}, true,
                          Bf16View{xb.h, B, IC, ldx}, Bf16View{xb.l, B, IC, ldx}, true, OC, IC, B, p64, IC,
                          reinterpret_cast<unsigned long long*>(d_max), dws_tail(workspace, B, IC, OC),
                          dws_c(B, IC, OC)));
    ITO_TRY(dfp_gemm_run(gp, s));
    return launch_dfp_down(p64, OC, IC, reinterpret_cast<unsigned long long*>(d_max), d_exp_delta, d_exp_x, g, nullptr,
                           nullptr, 0, d_exp_g, d_rs, s);
}

int ito_dfp16_from_float(const float* f, int64_t n, uint32_t* d_max_bits, int16_t* mant, int32_t* d_exp,
                         void* stream)
{
    if (!f || !d_max_bits || !mant || !d_exp) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    return launch_dfp_from_float(f, n, d_max_bits, mant, d_exp, static_cast<cudaStream_t>(stream));
}

int ito_dfp16_to_float(const int16_t* mant, const int32_t* d_exp, int64_t n, float* f, void* stream)
{
    if (!f || !mant || !d_exp) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    return launch_dfp_to_float(mant, n, d_exp, f, static_cast<cudaStream_t>(stream));
}

int ito_dfp16_linear_fwd_f32(const int16_t* x, const int32_t* d_exp_x, const int16_t* W, const int32_t* d_exp_w,
                             int B, int IC, int OC, void* workspace, size_t workspace_bytes, int64_t* p64,
                             uint64_t* d_max, float* y, void* stream)
{
    ITO_TRY(dfp_check(x, W, p64, y, B, IC, OC, workspace, workspace_bytes));
    if (!d_exp_x || !d_exp_w || !d_max) return set_error(ITO_ERR_ARG, "NULL scalar pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t ld = pad8(IC);
    Planes xa = planes_at(workspace, (size_t)B * ld);
    Planes wb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)OC * ld);
    ITO_TRY(launch_i16_to_limbs(x, B, IC, xa.h, xa.l, ld, s));
    ITO_TRY(launch_i16_to_limbs(W, OC, IC, wb.h, wb.l, ld, s));
    if (cudaMemsetAsync(d_max, 0, 8, s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset");
    DfpGemmPlan g;
    ITO_TRY(dfp_gemm_plan(&g, Bf16View{xa.h, B, IC, ld}, Bf16View{xa.l, B, IC, ld}, false, Bf16View{wb.h, OC, IC, ld},
                          Bf16View{wb.l, OC, IC, ld}, false, B, OC, IC, p64, OC,
                          reinterpret_cast<unsigned long long*>(d_max), dws_tail(workspace, B, IC, OC),
                          dws_c(B, IC, OC)));
    ITO_TRY(dfp_gemm_run(g, s));
    return launch_p64_to_float(p64, (int64_t)B * OC, d_exp_x, d_exp_w, y, s);
}

int ito_dfp16_linear_fwd_f32_chained(const int16_t* x, const int32_t* d_exp_x, const int16_t* W,
                                     const int32_t* d_exp_w, int B, int IC, int OC, int32_t chain, int32_t input_shift,
                                     void* workspace, size_t workspace_bytes, float* y, void* stream)
{
    ITO_TRY(dfp_check(x, W, y, y, B, IC, OC, workspace, workspace_bytes));
    if (!d_exp_x || !d_exp_w) return set_error(ITO_ERR_ARG, "NULL scalar pointer");
    if (input_shift != 0 && input_shift != 1) return set_error(ITO_ERR_ARG, "input_shift must be 0 or 1");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t ld = pad8(IC);
    Planes xa = planes_at(workspace, (size_t)B * ld);
    Planes wb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)OC * ld);
    DfpGemmPlan g;
    ITO_TRY(dfp_gemm_plan_chained(&g, Bf16View{xa.h, B, IC, ld}, Bf16View{xa.l, B, IC, ld},
                                  Bf16View{wb.h, OC, IC, ld}, Bf16View{wb.l, OC, IC, ld}, B, OC, IC, chain, d_exp_x,
                                  d_exp_w, input_shift, y, OC));
    ITO_TRY(launch_i16_to_limbs(x, B, IC, xa.h, xa.l, ld, s, input_shift));
    ITO_TRY(launch_i16_to_limbs(W, OC, IC, wb.h, wb.l, ld, s));
    return dfp_gemm_run(g, s);
}

int ito_bdfp16_from_float(const float* f, int64_t rows, int64_t cols, int32_t block, int16_t* mant, int8_t* exps,
                          void* stream)
{
    if (!f || !mant || !exps) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (rows < 1 || cols < 1 || block < 1) return set_error(ITO_ERR_SHAPE, "rows, cols and block must be >= 1");
    return launch_bdfp_from_float(f, rows, cols, block, mant, exps, static_cast<cudaStream_t>(stream));
}

int ito_bdfp16_to_float(const int16_t* mant, const int8_t* exps, int64_t rows, int64_t cols, int32_t block, float* f,
                        void* stream)
{
    if (!f || !mant || !exps) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (rows < 1 || cols < 1 || block < 1) return set_error(ITO_ERR_SHAPE, "rows, cols and block must be >= 1");
    return launch_bdfp_to_float(mant, exps, rows, cols, block, f, static_cast<cudaStream_t>(stream));
}

int ito_bdfp16_linear_fwd_f32(const int16_t* x, const int8_t* ex, const int16_t* W, const int8_t* ew, int B, int IC,
                              int OC, int32_t block, void* workspace, size_t workspace_bytes, float* y, void* stream)
{
    ITO_TRY(dfp_check(x, W, ex, y, B, IC, OC, workspace, workspace_bytes));
    if (!ew) return set_error(ITO_ERR_ARG, "NULL pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t ld = pad8(IC);
    Planes xa = planes_at(workspace, (size_t)B * ld);
    Planes wb = planes_at(static_cast<char*>(workspace) + dws_a(B, IC, OC), (size_t)OC * ld);
    ITO_TRY(launch_i16_to_limbs(x, B, IC, xa.h, xa.l, ld, s));
    ITO_TRY(launch_i16_to_limbs(W, OC, IC, wb.h, wb.l, ld, s));
    DfpGemmPlan g;
    ITO_TRY(dfp_gemm_plan_blocked(&g, Bf16View{xa.h, B, IC, ld}, Bf16View{xa.l, B, IC, ld},
                                  Bf16View{wb.h, OC, IC, ld}, Bf16View{wb.l, OC, IC, ld}, B, OC, IC, block, ex, ew,
                                  y, OC));
    return dfp_gemm_run(g, s);
}

int ito_dfp16_update(int16_t* W, const int16_t* g, const int32_t* d_exp_g, int64_t n, int32_t exp_w, int32_t eta,
                     int32_t* d_k, uint32_t* d_nonzero, void* stream)
{
    if (!W || !g || !d_exp_g) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    return launch_dfp_update(W, nullptr, nullptr, 0, g, 1, n, d_exp_g, exp_w, eta, d_k, d_nonzero,
                             static_cast<cudaStream_t>(stream));
}

int ito_dfp16_update_bits(int16_t* W, const int16_t* g, const int32_t* d_exp_g, int64_t n, int32_t exp_w, int32_t eta,
                          int32_t bits, int32_t* d_k, uint32_t* d_nonzero, void* stream)
{
    if (!W || !g || !d_exp_g) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    return launch_dfp_update(W, nullptr, nullptr, 0, g, 1, n, d_exp_g, exp_w, eta, d_k, d_nonzero,
                             static_cast<cudaStream_t>(stream), bits);
}

int ito_dfp_set_bits(int16_t* W, int64_t n, int32_t bits_old, int32_t bits_new, void* stream)
{
    if (!W) return set_error(ITO_ERR_ARG, "NULL pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    return launch_dfp_set_bits(W, nullptr, nullptr, 0, 1, n, bits_old, bits_new, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ model

int ito_dfp16_model_destroy(ito_dfp16_model* m)
{
    if (!m) return ITO_OK;
    cudaDeviceSynchronize();
    for (cudaEvent_t e : m->sync_ev) cudaEventDestroy(e);
    for (cudaEvent_t e : m->prof_ev) cudaEventDestroy(e);
    for (int i = 0; i < 2; ++i) {
        if (m->ev_copied[i]) cudaEventDestroy(m->ev_copied[i]);
        if (m->ev_consumed[i]) cudaEventDestroy(m->ev_consumed[i]);
    }
    if (m->side) cudaStreamDestroy(m->side);
    if (m->copy_stream) cudaStreamDestroy(m->copy_stream);
    for (void* p : m->allocs) cudaFree(p);
    delete m;
    return ITO_OK;
}

static int dfp_build(ito_dfp16_model* m, const int32_t* dims, int nl)
{
    const int B = m->batch;
    for (int l = 0; l < nl; ++l) {
        if (dims[l] < 1 || dims[l + 1] < 1) return set_error(ITO_ERR_SHAPE, "layer %d size", l);
        DLayer L;
        L.IC = dims[l];
        L.OC = dims[l + 1];
        m->L.push_back(L);
    }
    ITO_TRY(m->alloc(&m->s32, (size_t)nl * D_N32 + 2));
    ITO_TRY(m->alloc(&m->s64, (size_t)nl * D_N64));
    ITO_TRY(m->alloc(&m->wexp_d, (size_t)nl));
    ITO_TRY(m->alloc(&m->log_abs, (size_t)kAptMaxEvals * nl));
    ITO_TRY(m->alloc(&m->log_eg, (size_t)kAptMaxEvals * nl));
    m->wexp.assign(nl, m->exp_w);
    m->wbits.assign(nl, 16);
    m->ldx = pad8(dims[0]);
    ITO_TRY(m->alloc(&m->x16, (size_t)B * dims[0]));
    ITO_TRY(m->alloc(&m->x16b, (size_t)B * dims[0]));
    ITO_TRY(m->alloc(&m->stats_packed, (size_t)nl * (D_N32 + D_N64)));
    ITO_TRY(m->alloc(&m->xh, (size_t)B * m->ldx));
    ITO_TRY(m->alloc(&m->xl, (size_t)B * m->ldx));
    for (int l = 0; l < nl; ++l) {
        DLayer& L = m->L[l];
        L.ldw = pad8(L.IC);
        L.ldy = pad8(L.OC);
        ITO_TRY(m->alloc(&L.W, (size_t)L.OC * L.IC));
        ITO_TRY(m->alloc(&L.Wh, (size_t)L.OC * L.ldw));
        ITO_TRY(m->alloc(&L.Wl, (size_t)L.OC * L.ldw));
        ITO_TRY(m->alloc(&L.p64, (size_t)B * L.OC));
        ITO_TRY(m->alloc(&L.y16, (size_t)B * L.OC));
        ITO_TRY(m->alloc(&L.yh, (size_t)B * L.ldy));
        ITO_TRY(m->alloc(&L.yl, (size_t)B * L.ldy));
        if (l == nl - 1) {
            L.e16 = L.y16;   // the top error is the output itself
            L.eh = L.yh;
            L.el = L.yl;
        } else {
            ITO_TRY(m->alloc(&L.e16, (size_t)B * L.OC));
            ITO_TRY(m->alloc(&L.eh, (size_t)B * L.ldy));
            ITO_TRY(m->alloc(&L.el, (size_t)B * L.ldy));
        }
        if (l > 0) ITO_TRY(m->alloc(&L.pd64, (size_t)B * L.IC));
        ITO_TRY(m->alloc(&L.pg64, (size_t)L.OC * L.IC));
        ITO_TRY(m->alloc(&L.g16, (size_t)L.OC * L.IC));
    }
    // partial tiles of split last waves: one buffer for the largest need (the step runs in order)
    for (int l = 0; l < nl; ++l) {
        const DLayer& L = m->L[l];
        m->tail_ws_bytes = std::max(m->tail_ws_bytes, dfp_split_ws_bytes(B, L.OC, L.IC));
        if (l > 0) m->tail_ws_bytes = std::max(m->tail_ws_bytes, dfp_split_ws_bytes(B, L.IC, L.OC));
        m->tail_ws_bytes = std::max(m->tail_ws_bytes, dfp_split_ws_bytes(L.OC, L.IC, B));
    }
    if (m->tail_ws_bytes) ITO_TRY(m->alloc(&m->tail_ws, m->tail_ws_bytes / sizeof(int64_t)));
    for (int l = 0; l < nl; ++l) {
        DLayer& L = m->L[l];
        const Bf16View wh{L.Wh, L.OC, L.IC, L.ldw}, wl{L.Wl, L.OC, L.IC, L.ldw};
        const Bf16View eh{L.eh, B, L.OC, L.ldy}, el{L.el, B, L.OC, L.ldy};
        Bf16View ih, il;
        if (l == 0) {
            ih = Bf16View{m->xh, B, L.IC, m->ldx};
            il = Bf16View{m->xl, B, L.IC, m->ldx};
        } else {
            ih = Bf16View{m->L[l - 1].yh, B, L.IC, m->L[l - 1].ldy};
            il = Bf16View{m->L[l - 1].yl, B, L.IC, m->L[l - 1].ldy};
        }
        ITO_TRY(dfp_gemm_plan(&L.pf, ih, il, false, wh, wl, false, B, L.OC, L.IC, L.p64, L.OC, m->u64(l, D_PMAX),
                              m->tail_ws, m->tail_ws_bytes));
        // the backward contractions run beside down-conversions and updates on the side
        // stream (when the overlap is on), which take the SMs of a partial last wave
        const bool fill = !m->overlap;
        if (l > 0)
            ITO_TRY(dfp_gemm_plan(&L.pd, eh, el, false, wh, wl, true, B, L.IC, L.OC, L.pd64, L.IC, m->u64(l, D_PDMAX),
                                  m->tail_ws, m->tail_ws_bytes, fill));
        ITO_TRY(dfp_gemm_plan(&L.pg, eh, el, true, ih, il, true, L.OC, L.IC, B, L.pg64, L.IC, m->u64(l, D_PGMAX),
                              m->tail_ws, m->tail_ws_bytes, fill));
    }
    launch_pdl(k_set_i32, 1, 1, 0, 0, m->ew(), m->exp_w);
    if (cudaMemcpy(m->wexp_d, m->wexp.data(), sizeof(int32_t) * nl, cudaMemcpyHostToDevice) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "weight exponent copy");
    m->overlap = true;
    if (cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&m->copy_stream, cudaStreamNonBlocking) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "stream creation failed");
    for (int i = 0; i < 2; ++i)
        if (cudaEventCreateWithFlags(&m->ev_copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&m->ev_consumed[i], cudaEventDisableTiming) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "event creation failed");
    for (int i = 0; i < 2 + 3 * nl; ++i) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "event creation failed");
        m->sync_ev.push_back(e);
    }
    return cudaDeviceSynchronize() == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp model init");
}

int ito_dfp16_model_create(const int32_t* dims, int n_layers, int batch, int32_t exp_w, int32_t eta,
                           ito_dfp16_model** out)
{
    if (!dims || !out || n_layers < 1) return set_error(ITO_ERR_ARG, "NULL dims/out or no layers");
    if (batch < 1 || batch > (1 << 20)) return set_error(ITO_ERR_SHAPE, "batch");
    if (exp_w < -128 || exp_w > 127 || eta < 0 || eta > 62) return set_error(ITO_ERR_ARG, "exponent or eta");
    *out = nullptr;
    ito_dfp16_model* m = new ito_dfp16_model();
    m->batch = batch;
    m->exp_w = exp_w;
    m->eta = eta;
    int r = dfp_build(m, dims, n_layers);
    if (r != ITO_OK) {
        ito_dfp16_model_destroy(m);
        return r;
    }
    *out = m;
    return ITO_OK;
}

int ito_dfp16_model_set_weights(ito_dfp16_model* m, int layer, const int16_t* W, int on_host, void* stream)
{
    if (!m || !W || layer < 0 || layer >= (int)m->L.size()) return set_error(ITO_ERR_ARG, "bad model, layer or W");
    DLayer& L = m->L[layer];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(L.W, W, sizeof(int16_t) * L.OC * L.IC,
                                    on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "weight copy: %s", cudaGetErrorString(e));
    ITO_TRY(launch_i16_to_limbs(L.W, L.OC, L.IC, L.Wh, L.Wl, L.ldw, s));
    if (on_host && cudaStreamSynchronize(s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    return ITO_OK;
}

int ito_dfp16_model_tensor(const ito_dfp16_model* m, const char* name, void** dev_ptr, int* elem_bytes,
                           int64_t* numel)
{
    if (!m || !name || !dev_ptr || !elem_bytes || !numel) return set_error(ITO_ERR_ARG, "NULL argument");
    const int B = m->batch;
    auto put = [&](const void* p, int eb, int64_t n) {
        *dev_ptr = const_cast<void*>(p);
        *elem_bytes = eb;
        *numel = n;
        return p ? ITO_OK : set_error(ITO_ERR_ARG, "tensor %s does not exist in this model", name);
    };
    const std::string s(name);
    if (s == "x") return put(m->x16, 2, (int64_t)B * m->L[0].IC);
    size_t pos = 0;
    while (pos < s.size() && (s[pos] < '0' || s[pos] > '9')) ++pos;
    if (pos == 0 || pos == s.size()) return set_error(ITO_ERR_ARG, "unknown tensor name %s", name);
    const std::string key = s.substr(0, pos);
    char* end = nullptr;
    const long l = strtol(s.c_str() + pos, &end, 10);
    if (!end || *end || l < 0 || l >= (long)m->L.size()) return set_error(ITO_ERR_ARG, "unknown tensor %s", name);
    const DLayer& L = m->L[l];
    if (key == "w") return put(L.W, 2, (int64_t)L.OC * L.IC);
    if (key == "p") return put(L.p64, 8, (int64_t)B * L.OC);
    if (key == "y") return put(L.y16, 2, (int64_t)B * L.OC);
    if (key == "e") return put(L.e16, 2, (int64_t)B * L.OC);
    if (key == "pd") return put(L.pd64, 8, (int64_t)B * L.IC);
    if (key == "pg") return put(L.pg64, 8, (int64_t)L.OC * L.IC);
    if (key == "g") return put(L.g16, 2, (int64_t)L.OC * L.IC);
    return set_error(ITO_ERR_ARG, "unknown tensor name %s", name);
}

static const char* kD32[D_N32] = {"ey", "ee", "rs", "rsd", "rsg", "eg", "k", "nz"};
static const char* kD64[D_N64] = {"pmax", "pdmax", "pgmax", "gabs"};

int ito_dfp16_model_num_stats(const ito_dfp16_model* m)
{
    return m ? (int)m->L.size() * (D_N32 + D_N64) : 0;
}

int ito_dfp16_model_stat_index(const ito_dfp16_model* m, const char* name)
{
    if (!m || !name) return -1;
    const int nl = (int)m->L.size();
    for (int l = 0; l < nl; ++l) {
        for (int k = 0; k < D_N32; ++k)
            if (std::string(kD32[k]) + std::to_string(l) == name) return l * (D_N32 + D_N64) + k;
        for (int k = 0; k < D_N64; ++k)
            if (std::string(kD64[k]) + std::to_string(l) == name) return l * (D_N32 + D_N64) + D_N32 + k;
    }
    return -1;
}

int ito_dfp16_model_read_stats(const ito_dfp16_model* m, int64_t* host_out, int n)
{
    if (!m || !host_out || n < ito_dfp16_model_num_stats(m)) return set_error(ITO_ERR_ARG, "bad arguments");
    const int nl = (int)m->L.size();
    std::vector<int32_t> a((size_t)nl * D_N32);
    std::vector<unsigned long long> b((size_t)nl * D_N64);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(a.data(), m->s32, a.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(b.data(), m->s64, b.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "stats read failed");
    for (int l = 0; l < nl; ++l) {
        for (int k = 0; k < D_N32; ++k) host_out[l * (D_N32 + D_N64) + k] = a[l * D_N32 + k];
        for (int k = 0; k < D_N64; ++k) host_out[l * (D_N32 + D_N64) + D_N32 + k] = (int64_t)b[l * D_N64 + k];
    }
    return ITO_OK;
}

// The statistics in the layout of ito_dfp16_model_read_stats: per layer its D_N32 int32 words
// (sign-extended), then its D_N64 words.
__global__ void k_dfp_pack_stats(const int32_t* __restrict__ s32, const unsigned long long* __restrict__ s64, int nl,
                                 int64_t* __restrict__ out)
{
    griddep_wait();
    griddep_launch_dependents();
    for (int i = threadIdx.x; i < nl * (D_N32 + D_N64); i += blockDim.x) {
        const int l = i / (D_N32 + D_N64), k = i - l * (D_N32 + D_N64);
        out[i] = k < D_N32 ? (int64_t)s32[l * D_N32 + k] : (int64_t)s64[l * D_N64 + (k - D_N32)];
    }
}

int ito_dfp16_train_step_host_async(ito_dfp16_model* m, const int16_t* x_host, int32_t exp_x, int64_t* stats_host,
                                    void* stream)
{
    if (!m || !x_host) return set_error(ITO_ERR_ARG, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int i = (int)(m->async_steps & 1);
    int16_t* xd = i ? m->x16b : m->x16;
    const int nl = (int)m->L.size();
    // the copy waits for the step that last read this buffer, and the step for the copy
    cudaError_t e = cudaStreamWaitEvent(m->copy_stream, m->ev_consumed[i], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(xd, x_host, sizeof(int16_t) * m->batch * m->L[0].IC, cudaMemcpyHostToDevice,
                            m->copy_stream);
    if (e == cudaSuccess) e = cudaEventRecord(m->ev_copied[i], m->copy_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, m->ev_copied[i], 0);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "input copy: %s", cudaGetErrorString(e));
    ITO_TRY(ito_dfp16_train_step(m, xd, exp_x, stream));
    if (stats_host) {
        launch_pdl(k_dfp_pack_stats, 1, 128, 0, s, m->s32, m->s64, nl, m->stats_packed);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(stats_host, m->stats_packed, sizeof(int64_t) * nl * (D_N32 + D_N64),
                                cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "stats copy: %s", cudaGetErrorString(e));
    }
    e = cudaEventRecord(m->ev_consumed[i], s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "event: %s", cudaGetErrorString(e));
    ++m->async_steps;
    return ITO_OK;
}

int ito_dfp16_model_profile(ito_dfp16_model* m, int enable)
{
    if (!m) return set_error(ITO_ERR_ARG, "NULL model");
    if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    m->prof_on = enable != 0;
    m->prof_n = 0;
    m->prof_cls.clear();
    m->prof_work.clear();
    return ITO_OK;
}

int ito_dfp16_model_profile_read(ito_dfp16_model* m, double* ms, double* work, int64_t* launches)
{
    if (!m || !ms || !work || !launches) return set_error(ITO_ERR_ARG, "NULL argument");
    for (int c = 0; c < ITO_PROF_NCLASS; ++c) {
        ms[c] = work[c] = 0.0;
        launches[c] = 0;
    }
    for (int i = 0; i < m->prof_n; ++i) {
        float t = 0.f;
        if (cudaEventSynchronize(m->prof_ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "profile event read failed");
        ms[m->prof_cls[i]] += t;
        work[m->prof_cls[i]] += m->prof_work[i];
        launches[m->prof_cls[i]] += 1;
    }
    m->prof_n = 0;
    m->prof_cls.clear();
    m->prof_work.clear();
    return ITO_OK;
}

int ito_dfp16_model_kernels_per_step(const ito_dfp16_model* m) { return m ? m->launches : 0; }

int ito_dfp16_train_step(ito_dfp16_model* m, const int16_t* x, int32_t exp_x, void* stream)
{
    if (!m || !x) return set_error(ITO_ERR_ARG, "NULL argument");
    if (exp_x < -128 || exp_x > 127) return set_error(ITO_ERR_EXPONENT, "input exponent outside int8");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int B = m->batch;
    const int nl = (int)m->L.size();
    m->launches = 0;
    // statistics zeroed and the input exponent set in one launch (no memset nodes, which would
    // break the programmatic launch chain)
    ITO_DLAUNCH(m, s, ITO_PROF_OTHER, 0.0,
                (launch_pdl(k_dfp_step_begin, 1, 256, 0, s, m->s32, nl * D_N32, m->s64, nl * D_N64, m->ex(), exp_x),
                 ITO_OK));
    ITO_DLAUNCH(m, s, ITO_PROF_OTHER, 6.0 * B * m->L[0].IC,
                launch_i16_to_limbs(x, B, m->L[0].IC, m->xh, m->xl, m->ldx, s));
    for (int l = 0; l < nl; ++l) {
        DLayer& L = m->L[l];
        const int32_t* e_in = l == 0 ? m->ex() : m->i32(l - 1, D_EY);
        ITO_DLAUNCH(m, s, ITO_PROF_GEMM, dfp_gemm_ops(L.pf), dfp_gemm_run(L.pf, s));
        m->launches += dfp_gemm_kernels(L.pf) - 1;
        // the top layer's output exponent is also its delta's (the backward's first D_EE)
        ITO_DLAUNCH(m, s, ITO_PROF_REQUANT, 14.0 * B * L.OC,
                    launch_dfp_down(L.p64, B, L.OC, m->u64(l, D_PMAX), e_in, m->wexp_d + l, L.y16, L.yh, L.yl, L.ldy,
                                    m->i32(l, D_EY), m->i32(l, D_RS), s, nullptr,
                                    l == nl - 1 ? m->i32(nl - 1, D_EE) : nullptr));
    }
    // backward, top-down; with the overlap on, the contractions stay on s and the
    // down-conversions and the update go to the side stream b: the propagated delta's
    // down-conversion runs beside the weight gradient, the gradient's down-conversion
    // and the update beside the next layer's delta propagation
    cudaStream_t b = m->overlap ? m->side : s;
    auto ev = [&](int l, int k) { return m->sync_ev[2 + 3 * l + k]; };   // k: 0 propagated, 1 ready, 2 wgrad
    auto sync = [&](cudaEvent_t e, cudaStream_t from, cudaStream_t to) -> int {
        if (from == to) return ITO_OK;
        if (cudaEventRecord(e, from) != cudaSuccess || cudaStreamWaitEvent(to, e, 0) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        return ITO_OK;
    };
    ITO_TRY(sync(m->sync_ev[0], s, b));
    for (int l = nl - 1; l >= 0; --l) {
        DLayer& L = m->L[l];
        const int32_t* e_in = l == 0 ? m->ex() : m->i32(l - 1, D_EY);
        if (l < nl - 1 && b != s && cudaStreamWaitEvent(s, ev(l + 1, 1), 0) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        if (l > 0) {
            DLayer& P = m->L[l - 1];
            ITO_DLAUNCH(m, s, ITO_PROF_GEMM, dfp_gemm_ops(L.pd), dfp_gemm_run(L.pd, s));
        m->launches += dfp_gemm_kernels(L.pd) - 1;
            ITO_TRY(sync(ev(l, 0), s, b));
            ITO_DLAUNCH(m, b, ITO_PROF_REQUANT, 14.0 * B * L.IC,
                        launch_dfp_down(L.pd64, B, L.IC, m->u64(l, D_PDMAX), m->i32(l, D_EE), m->wexp_d + l, P.e16,
                                        P.eh, P.el, P.ldy, m->i32(l - 1, D_EE), m->i32(l, D_RSD), b));
            if (b != s && cudaEventRecord(ev(l, 1), b) != cudaSuccess)
                return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        }
        ITO_DLAUNCH(m, s, ITO_PROF_GEMM, dfp_gemm_ops(L.pg), dfp_gemm_run(L.pg, s));
        m->launches += dfp_gemm_kernels(L.pg) - 1;
        ITO_TRY(sync(ev(l, 2), s, b));
        ITO_DLAUNCH(m, b, ITO_PROF_REQUANT, 10.0 * L.OC * L.IC,
                    launch_dfp_down(L.pg64, L.OC, L.IC, m->u64(l, D_PGMAX), m->i32(l, D_EE), e_in, L.g16, nullptr,
                                    nullptr, 0, m->i32(l, D_EG), m->i32(l, D_RSG), b, m->u64(l, D_GABS)));
        ITO_DLAUNCH(m, b, ITO_PROF_UPDATE, 10.0 * L.OC * L.IC,
                    launch_dfp_update(L.W, L.Wh, L.Wl, L.ldw, L.g16, L.OC, L.IC, m->i32(l, D_EG), m->wexp[l], m->eta,
                                      m->i32(l, D_K), reinterpret_cast<uint32_t*>(m->i32(l, D_NZ)), b,
                                      m->wbits[l]));
    }
    ITO_TRY(sync(m->sync_ev[1], b, s));
    if (m->apt) {
        // Algorithm 2: Gavg is evaluated at every eval_every-th step of the epoch
        if (m->apt_step % m->ap.eval_every == 0) {
            if (m->apt_nlog >= kAptMaxEvals)
                return set_error(ITO_ERR_ARG, "more than %d Gavg evaluations in one epoch", kAptMaxEvals);
            ITO_DLAUNCH(m, s, ITO_PROF_OTHER, 0.0,
                        (launch_pdl(k_apt_log, 1, 32 * ((nl + 31) / 32), 0, s, m->s64, m->s32, nl,
                                                                       m->log_abs + (size_t)m->apt_nlog * nl,
                                                                       m->log_eg + (size_t)m->apt_nlog * nl),
                         ITO_OK));
            ++m->apt_nlog;
        }
        ++m->apt_step;
    }
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "dfp step: %s", cudaGetErrorString(e));
}

int ito_dfp16_model_get_precision(const ito_dfp16_model* m, int layer, int32_t* bits, int32_t* exp_w)
{
    if (!m || layer < 0 || layer >= (int)m->L.size()) return set_error(ITO_ERR_ARG, "bad model or layer");
    if (bits) *bits = m->wbits[layer];
    if (exp_w) *exp_w = m->wexp[layer];
    return ITO_OK;
}

int ito_dfp16_model_set_precision(ito_dfp16_model* m, int layer, int32_t bits, void* stream)
{
    if (!m || layer < 0 || layer >= (int)m->L.size()) return set_error(ITO_ERR_ARG, "bad model or layer");
    if (bits < 2 || bits > 16) return set_error(ITO_ERR_ARG, "weight precision must be 2 .. 16 bits");
    const int d = bits - m->wbits[layer];
    if (d == 0) return ITO_OK;
    const int e = m->wexp[layer] - d;
    if (e < -128 || e > 127) return set_error(ITO_ERR_EXPONENT, "weight exponent %d outside int8", e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DLayer& L = m->L[layer];
    ITO_TRY(launch_dfp_set_bits(L.W, L.Wh, L.Wl, L.ldw, L.OC, L.IC, m->wbits[layer], bits, s));
    launch_pdl(k_set_i32, 1, 1, 0, s, m->wexp_d + layer, e);
    m->wbits[layer] = bits;
    m->wexp[layer] = e;
    cudaError_t ce = cudaGetLastError();
    return ce == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "precision change: %s", cudaGetErrorString(ce));
}

int ito_dfp16_model_apt_enable(ito_dfp16_model* m, const ito_apt_params* p, void* stream)
{
    if (!m || !p) return set_error(ITO_ERR_ARG, "NULL argument");
    if (!(2 <= p->k_min && p->k_min <= p->k_init && p->k_init <= p->k_max && p->k_max <= 16))
        return set_error(ITO_ERR_ARG, "need 2 <= k_min <= k_init <= k_max <= 16");
    if (p->eval_every < 1) return set_error(ITO_ERR_ARG, "eval_every must be >= 1");
    if (!(p->t_min <= p->t_max)) return set_error(ITO_ERR_ARG, "need t_min <= t_max");
    if (m->L.size() > 1024) return set_error(ITO_ERR_UNSUPPORTED, "APT supports at most 1024 layers");
    for (int l = 0; l < (int)m->L.size(); ++l) ITO_TRY(ito_dfp16_model_set_precision(m, l, p->k_init, stream));
    m->ap = *p;
    m->apt = true;
    m->apt_step = 0;
    m->apt_nlog = 0;
    return ITO_OK;
}

int ito_dfp16_model_apt_epoch_end(ito_dfp16_model* m, double* gavg_out, int32_t* bits_out, void* stream)
{
    if (!m || !m->apt) return set_error(ITO_ERR_ARG, "APT is not enabled on this model");
    if (m->apt_nlog < 1) return set_error(ITO_ERR_ARG, "no Gavg evaluation since the last epoch end");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int nl = (int)m->L.size();
    const size_t cnt = (size_t)m->apt_nlog * nl;
    std::vector<unsigned long long> ab(cnt);
    std::vector<int32_t> eg(cnt);
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(ab.data(), m->log_abs, cnt * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(eg.data(), m->log_eg, cnt * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "reading the Gavg log failed");
    for (int l = 0; l < nl; ++l) {
        // Equation 4 per evaluation: Gavg = sum|G| * 2^(E_G - E_W) / (N * B), the gradient taken
        // as the batch mean; the epoch's value is the mean over its evaluations, in order
        const double nb = (double)((int64_t)m->L[l].OC * m->L[l].IC * (int64_t)m->batch);
        double acc = 0.0;
        for (int i = 0; i < m->apt_nlog; ++i) {
            const size_t j = (size_t)i * nl + l;
            acc += ldexp((double)ab[j], eg[j] - m->wexp[l]) / nb;
        }
        const double g = acc / (double)m->apt_nlog;
        // Algorithm 1
        int k = m->wbits[l];
        if (g < m->ap.t_min && k < m->ap.k_max)
            ++k;
        else if (g > m->ap.t_max && k > m->ap.k_min)
            --k;
        ITO_TRY(ito_dfp16_model_set_precision(m, l, k, stream));
        if (gavg_out) gavg_out[l] = g;
        if (bits_out) bits_out[l] = k;
    }
    m->apt_step = 0;
    m->apt_nlog = 0;
    return ITO_OK;
}

}  // extern "C"
