// extern "C" entry points of libito.so: argument checking, workspace layout
// and launch order of the single-layer operations. The model (INT_LAYERS-like
// stack and the whole training step) is in ito_model.cu.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <algorithm>

#include "ito_conv.h"
#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

static thread_local char g_err_text[512] = "";

int set_error(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err_text, sizeof(g_err_text), fmt, ap);
    va_end(ap);
    return code;
}

static inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Workspace: slot 0 holds the bf16 copy of the [B][*] operand (x or delta),
// slot 1 the bf16 copy of the weight or of the layer input.
static size_t ws_slot0(int B, int IC, int OC) { return align256((size_t)2 * B * pad8(IC > OC ? IC : OC)); }
static size_t ws_slot1(int B, int IC, int OC) { return align256((size_t)2 * (OC > B ? OC : B) * pad8(IC)); }
// slot 2: split-K partials of whichever of the three contractions needs most
static size_t ws_slot2(int B, int IC, int OC)
{
    size_t a = gemm_split_ws_bytes(B, OC, IC, OC), b = gemm_split_ws_bytes(B, IC, OC, IC),
           c = gemm_split_ws_bytes(OC, IC, B, IC);
    return align256(a > b ? (a > c ? a : c) : (b > c ? b : c));
}
static int32_t* ws_split(void* ws, int B, int IC, int OC)
{
    return reinterpret_cast<int32_t*>(static_cast<char*>(ws) + ws_slot0(B, IC, OC) + ws_slot1(B, IC, OC));
}

static int check_sizes(int B, int IC, int OC)
{
    if (B < 1 || IC < 1 || OC < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    if (B > (1 << 20) || IC > (1 << 20) || OC > (1 << 20))
        return set_error(ITO_ERR_SHAPE, "a contraction length above 2^20");
    return ITO_OK;
}

static int check_ws(void* ws, size_t bytes, int B, int IC, int OC)
{
    if (!ws) return set_error(ITO_ERR_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return set_error(ITO_ERR_ARG, "workspace not 256-byte aligned");
    if (bytes < ito_linear_workspace_size(B, IC, OC)) return set_error(ITO_ERR_ARG, "workspace too small");
    return ITO_OK;
}

static int cuda_ok(cudaError_t e, const char* what)
{
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------- conv 3x3

// Geometry of a 3x3, pad-1 conv over NHWC input [B][H][W][IC] with weights
// [OC][3][3][IC]: a Linear layer over the im2col patch matrix [rows_out][K].
struct ConvGeom {
    int B, H, W, IC, stride;
    int OH, OW;
    int64_t rows_in, rows_out, K, ldp, lde;
    bool s2;   // stride 2 on parity planes (no patches; see ito_conv_tc.cu)
};

static ConvGeom conv_geom(int B, int H, int W, int IC, int OC, int stride)
{
    ConvGeom g;
    g.B = B;
    g.H = H;
    g.W = W;
    g.IC = IC;
    g.stride = stride;
    g.s2 = conv_dgrad_s2_eligible(B, H, W, IC, OC, stride);
    g.OH = (H - 1) / stride + 1;
    g.OW = (W - 1) / stride + 1;
    g.rows_in = (int64_t)B * H * W;
    g.rows_out = (int64_t)B * g.OH * g.OW;
    g.K = 9 * (int64_t)IC;
    g.ldp = pad8(g.K);
    g.lde = pad8(OC);
    return g;
}

// Workspace slots: 0 bf16 patches [rows_out][ldp] (for a stride-2 conv on parity planes
// the bf16 copy of the input [rows_in][IC], which is smaller); 1 bf16 weights [OC][ldp];
// 2 bf16 delta [rows_out][lde]; 3 int32 patch-space delta [rows_out][K];
// 4 split-K partials of the largest of the three contractions; 5 one uint32
// receiving the (unused) max of the patch-space delta.
static void conv_slots(const ConvGeom& g, int OC, size_t sz[6])
{
    const int M = (int)g.rows_out, K = (int)g.K;
    sz[0] = align256((size_t)2 * g.rows_out * g.ldp);
    sz[1] = align256((size_t)2 * OC * g.ldp);
    sz[2] = align256((size_t)2 * g.rows_out * g.lde);
    sz[3] = align256((size_t)4 * g.rows_out * g.K);
    size_t a = gemm_split_ws_bytes(M, OC, K, OC), b = gemm_split_ws_bytes(M, K, OC, K),
           c = gemm_split_ws_bytes(OC, K, M, K);
    const size_t d = conv_wgrad_s2_ws_bytes(g.B, g.H, g.W, g.IC, OC);
    sz[4] = align256(std::max(std::max(a, d), std::max(b, c)));
    sz[5] = 256;
}

static char* conv_slot(void* ws, const size_t sz[6], int i)
{
    char* p = static_cast<char*>(ws);
    for (int j = 0; j < i; ++j) p += sz[j];
    return p;
}

static int check_conv(int B, int H, int W, int IC, int OC, int stride)
{
    if (B < 1 || H < 1 || W < 1 || IC < 1 || OC < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    if (stride < 1 || stride > 4) return set_error(ITO_ERR_SHAPE, "stride must be 1 .. 4");
    if (IC > (1 << 16) || OC > (1 << 20)) return set_error(ITO_ERR_SHAPE, "IC above 2^16 or OC above 2^20");
    const ConvGeom g = conv_geom(B, H, W, IC, OC, stride);
    if (g.rows_in > (1 << 20) * 64LL || g.rows_out > (1 << 20))
        return set_error(ITO_ERR_SHAPE, "B*OH*OW above 2^20 (the weight-gradient contraction length)");
    return ITO_OK;
}

static int check_conv_ws(void* ws, size_t bytes, int B, int H, int W, int IC, int OC, int stride);

}  // namespace ito

using namespace ito;

#define ITO_TRY(x)                 \
    do {                           \
        int _r = (x);              \
        if (_r != ITO_OK) return _r; \
    } while (0)

extern "C" {

int ito_version(void) { return 1; }

const char* ito_last_error_string(void) { return g_err_text; }

int ito_get_error(void)
{
    int v = 0, zero = 0;
    int* w = device_error_word();
    if (!w) return set_error(ITO_ERR_CUDA, "device error word unavailable");
    if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "device sync failed");
    if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "reading the device error word failed");
    if (v != 0) cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return v;
}

int ito_selftest_wait_timeout(void* stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ITO_TRY(launch_wait_timeout_selftest(s));
    return cuda_ok(cudaStreamSynchronize(s), "self-test");
}

size_t ito_linear_workspace_size(int B, int IC, int OC)
{
    if (B < 1 || IC < 1 || OC < 1) return 0;
    return ws_slot0(B, IC, OC) + ws_slot1(B, IC, OC) + ws_slot2(B, IC, OC);
}

int ito_linear_fwd(const int8_t* x, const int8_t* W, int B, int IC, int OC, int relu, ito_niti_params p,
                   void* workspace, size_t workspace_bytes, int32_t* y32, uint32_t* d_max, int32_t* d_shift,
                   int8_t* y, void* stream)
{
    if (!x || !W || !y32 || !d_max || !y) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_sizes(B, IC, OC));
    ITO_TRY(check_ws(workspace, workspace_bytes, B, IC, OC));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* xb = static_cast<uint16_t*>(workspace);
    uint16_t* Wb = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + ws_slot0(B, IC, OC));
    const int64_t ld = pad8(IC);
    ITO_TRY(launch_i8_to_bf16(x, B, IC, xb, ld, s));
    ITO_TRY(launch_i8_to_bf16(W, OC, IC, Wb, ld, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    GemmPlan g;
    ITO_TRY(gemm_plan(&g, Bf16View{xb, B, IC, ld}, false, Bf16View{Wb, OC, IC, ld}, false, B, OC, IC, y32, OC,
                      d_max, ws_split(workspace, B, IC, OC), ws_slot2(B, IC, OC)));
    ITO_TRY(gemm_run(g, s));
    return launch_requant(y32, B, OC, d_max, p.target_bits, relu, nullptr, y, nullptr, 0, d_shift, s);
}

int ito_linear_bwd_delta(const int8_t* delta, const int8_t* W, const int8_t* a_prev, int B, int IC, int OC,
                         ito_niti_params p, void* workspace, size_t workspace_bytes, int32_t* d32, uint32_t* d_max,
                         int32_t* d_shift, int8_t* delta_prev, void* stream)
{
    if (!delta || !W || !d32 || !d_max || !delta_prev) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_sizes(B, IC, OC));
    ITO_TRY(check_ws(workspace, workspace_bytes, B, IC, OC));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* eb = static_cast<uint16_t*>(workspace);
    uint16_t* Wb = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + ws_slot0(B, IC, OC));
    const int64_t lde = pad8(OC), ldw = pad8(IC);
    ITO_TRY(launch_i8_to_bf16(delta, B, OC, eb, lde, s));
    ITO_TRY(launch_i8_to_bf16(W, OC, IC, Wb, ldw, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    GemmPlan g;
    // D[b][ic] = sum_oc delta[b][oc] W[oc][ic]: A = delta (K-major), B = W read as [K=OC][N=IC] (MN-major)
    ITO_TRY(gemm_plan(&g, Bf16View{eb, B, OC, lde}, false, Bf16View{Wb, OC, IC, ldw}, true, B, IC, OC, d32, IC,
                      d_max, ws_split(workspace, B, IC, OC), ws_slot2(B, IC, OC)));
    ITO_TRY(gemm_run(g, s));
    return launch_requant(d32, B, IC, d_max, p.target_bits, 0, a_prev, delta_prev, nullptr, 0, d_shift, s);
}

int ito_linear_wgrad(const int8_t* delta, const int8_t* a_prev, int B, int IC, int OC, void* workspace,
                     size_t workspace_bytes, int32_t* G, uint32_t* d_max, void* stream)
{
    if (!delta || !a_prev || !G || !d_max) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_sizes(B, IC, OC));
    ITO_TRY(check_ws(workspace, workspace_bytes, B, IC, OC));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* eb = static_cast<uint16_t*>(workspace);
    uint16_t* ab = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + ws_slot0(B, IC, OC));
    const int64_t lde = pad8(OC), lda = pad8(IC);
    ITO_TRY(launch_i8_to_bf16(delta, B, OC, eb, lde, s));
    ITO_TRY(launch_i8_to_bf16(a_prev, B, IC, ab, lda, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    GemmPlan g;
    // G[oc][ic] = sum_b delta[b][oc] a[b][ic]: A = delta read as [K=B][M=OC], B = a read as [K=B][N=IC]
    ITO_TRY(gemm_plan(&g, Bf16View{eb, B, OC, lde}, true, Bf16View{ab, B, IC, lda}, true, OC, IC, B, G, IC, d_max,
                      ws_split(workspace, B, IC, OC), ws_slot2(B, IC, OC)));
    return gemm_run(g, s);
}

int ito_niti_update(int8_t* W, const int32_t* G, int64_t n, const uint32_t* d_max, ito_niti_params p,
                    int32_t* d_shift, int32_t* d_wshift, uint32_t* d_nonzero, void* stream)
{
    if (!W || !G || !d_max) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    if (n < 1) return set_error(ITO_ERR_SHAPE, "n must be >= 1");
    // viewed as one row of n elements when n is a multiple of 8 (vector path), else n rows of 1
    const int64_t cols = (n % 8 == 0) ? n : 1;
    return launch_niti_update(W, nullptr, 0, G, n / cols, cols, d_max, p.target_bits, p.mu_weight, d_shift,
                              d_wshift, d_nonzero, static_cast<cudaStream_t>(stream));
}

int ito_top_error(const int8_t* logits, const int32_t* labels, int B, int C, int32_t target_mag, int8_t* delta,
                  void* stream)
{
    if (!logits || !labels || !delta) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    if (B < 1 || C < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    return launch_top_error(logits, labels, B, C, target_mag, delta, nullptr, 0, static_cast<cudaStream_t>(stream));
}

size_t ito_conv2d_workspace_size(int B, int H, int W, int IC, int OC, int stride)
{
    if (B < 1 || H < 1 || W < 1 || IC < 1 || OC < 1 || stride < 1 || stride > 4) return 0;
    size_t sz[6];
    conv_slots(conv_geom(B, H, W, IC, OC, stride), OC, sz);
    return sz[0] + sz[1] + sz[2] + sz[3] + sz[4] + sz[5];
}

int ito_conv2d_fwd(const int8_t* x, const int8_t* Wt, int B, int H, int W, int IC, int OC, int stride, int relu,
                   ito_niti_params p, void* workspace, size_t workspace_bytes, int32_t* y32, uint32_t* d_max,
                   int32_t* d_shift, int8_t* y, void* stream)
{
    if (!x || !Wt || !y32 || !d_max || !y) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_conv(B, H, W, IC, OC, stride));
    ITO_TRY(check_conv_ws(workspace, workspace_bytes, B, H, W, IC, OC, stride));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ConvGeom g = conv_geom(B, H, W, IC, OC, stride);
    size_t sz[6];
    conv_slots(g, OC, sz);
    uint16_t* Pb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 0));
    uint16_t* Wb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 1));
    if (g.s2) {
        // the input's bf16 copy, read through its parity planes
        ITO_TRY(launch_i8_to_bf16(x, g.rows_in, IC, Pb, IC, s));
        ITO_TRY(launch_i8_to_bf16(Wt, OC, g.K, Wb, g.ldp, s));
        ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
        ConvIgPlan ip;
        ITO_TRY(conv_fwd_s2_plan(&ip, Pb, IC, Wb, g.ldp, B, H, W, IC, OC, y32, d_max));
        ITO_TRY(conv_igemm_run(ip, s));
        return launch_requant(y32, g.rows_out, OC, d_max, p.target_bits, relu, nullptr, y, nullptr, 0, d_shift, s);
    }
    ITO_TRY(launch_im2col(x, B, H, W, IC, g.OH, g.OW, stride, Pb, g.ldp, s));
    ITO_TRY(launch_i8_to_bf16(Wt, OC, g.K, Wb, g.ldp, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    GemmPlan gp;
    // Y[(b,oh,ow)][oc] = sum_k P[(b,oh,ow)][k] W[oc][k]
    ITO_TRY(gemm_plan(&gp, Bf16View{Pb, g.rows_out, g.K, g.ldp}, false, Bf16View{Wb, OC, g.K, g.ldp}, false,
                      (int)g.rows_out, OC, (int)g.K, y32, OC, d_max,
                      reinterpret_cast<int32_t*>(conv_slot(workspace, sz, 4)), sz[4]));
    ITO_TRY(gemm_run(gp, s));
    return launch_requant(y32, g.rows_out, OC, d_max, p.target_bits, relu, nullptr, y, nullptr, 0, d_shift, s);
}

int ito_conv2d_bwd_delta(const int8_t* delta, const int8_t* Wt, const int8_t* a_prev, int B, int H, int W, int IC,
                         int OC, int stride, ito_niti_params p, void* workspace, size_t workspace_bytes, int32_t* d32,
                         uint32_t* d_max, int32_t* d_shift, int8_t* delta_prev, void* stream)
{
    if (!delta || !Wt || !d32 || !d_max || !delta_prev) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_conv(B, H, W, IC, OC, stride));
    ITO_TRY(check_conv_ws(workspace, workspace_bytes, B, H, W, IC, OC, stride));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ConvGeom g = conv_geom(B, H, W, IC, OC, stride);
    size_t sz[6];
    conv_slots(g, OC, sz);
    uint16_t* Wb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 1));
    uint16_t* eb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 2));
    int32_t* dcol = reinterpret_cast<int32_t*>(conv_slot(workspace, sz, 3));
    ITO_TRY(launch_i8_to_bf16(delta, g.rows_out, OC, eb, g.lde, s));
    ITO_TRY(launch_i8_to_bf16(Wt, OC, g.K, Wb, g.ldp, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    if (g.s2) {
        // stride 2: each parity phase of the input-space delta is its own contraction, written
        // straight into d32 with its max
        ConvS2Plan sp;
        ITO_TRY(conv_dgrad_s2_plan(&sp, eb, g.lde, Wb, g.ldp, B, H, W, IC, OC, d32, d_max));
        ITO_TRY(conv_dgrad_s2_run(sp, s));
        return launch_requant(d32, g.rows_in, IC, d_max, p.target_bits, 0, a_prev, delta_prev, nullptr, 0, d_shift,
                              s);
    }
    // patch-space delta Dcol[(b,oh,ow)][k] = sum_oc delta[(b,oh,ow)][oc] W[oc][k]; its max is not
    // the NITI max (col2im takes that), so the contraction folds it into a scratch word
    uint32_t* discard = reinterpret_cast<uint32_t*>(conv_slot(workspace, sz, 5));
    GemmPlan gp;
    ITO_TRY(gemm_plan(&gp, Bf16View{eb, g.rows_out, OC, g.lde}, false, Bf16View{Wb, OC, g.K, g.ldp}, true,
                      (int)g.rows_out, (int)g.K, OC, dcol, g.K, discard,
                      reinterpret_cast<int32_t*>(conv_slot(workspace, sz, 4)), sz[4]));
    ITO_TRY(gemm_run(gp, s));
    // input-space delta (gather of the <= 9 patch entries per input position) and its max
    ITO_TRY(launch_col2im(dcol, B, H, W, IC, g.OH, g.OW, stride, d32, d_max, s));
    return launch_requant(d32, g.rows_in, IC, d_max, p.target_bits, 0, a_prev, delta_prev, nullptr, 0, d_shift, s);
}

int ito_conv2d_wgrad(const int8_t* delta, const int8_t* x, int B, int H, int W, int IC, int OC, int stride,
                     void* workspace, size_t workspace_bytes, int32_t* G, uint32_t* d_max, void* stream)
{
    if (!delta || !x || !G || !d_max) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    ITO_TRY(check_conv(B, H, W, IC, OC, stride));
    ITO_TRY(check_conv_ws(workspace, workspace_bytes, B, H, W, IC, OC, stride));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ConvGeom g = conv_geom(B, H, W, IC, OC, stride);
    size_t sz[6];
    conv_slots(g, OC, sz);
    uint16_t* Pb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 0));
    uint16_t* eb = reinterpret_cast<uint16_t*>(conv_slot(workspace, sz, 2));
    if (g.s2) {
        ITO_TRY(launch_i8_to_bf16(x, g.rows_in, IC, Pb, IC, s));
        ITO_TRY(launch_i8_to_bf16(delta, g.rows_out, OC, eb, g.lde, s));
        ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
        ConvIgPlan ip;
        ITO_TRY(conv_wgrad_s2_plan(&ip, eb, g.lde, Pb, IC, B, H, W, IC, OC, G, d_max,
                                   reinterpret_cast<int32_t*>(conv_slot(workspace, sz, 4)), sz[4]));
        return conv_igemm_run(ip, s);
    }
    ITO_TRY(launch_im2col(x, B, H, W, IC, g.OH, g.OW, stride, Pb, g.ldp, s));
    ITO_TRY(launch_i8_to_bf16(delta, g.rows_out, OC, eb, g.lde, s));
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    GemmPlan gp;
    // G[oc][k] = sum_(b,oh,ow) delta[(b,oh,ow)][oc] P[(b,oh,ow)][k]
    ITO_TRY(gemm_plan(&gp, Bf16View{eb, g.rows_out, OC, g.lde}, true, Bf16View{Pb, g.rows_out, g.K, g.ldp}, true,
                      OC, (int)g.K, (int)g.rows_out, G, g.K, d_max,
                      reinterpret_cast<int32_t*>(conv_slot(workspace, sz, 4)), sz[4]));
    return gemm_run(gp, s);
}

int ito_gap_fwd(const int8_t* a, int B, int HW, int C, ito_niti_params p, int32_t* P32, uint32_t* d_max,
                int32_t* d_shift, int8_t* pa, void* stream)
{
    if (!a || !P32 || !d_max || !pa) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    if (B < 1 || HW < 1 || C < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    if (HW > (1 << 24)) return set_error(ITO_ERR_SHAPE, "HW above 2^24 (the int32 sum could overflow)");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ITO_TRY(cuda_ok(cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s), "memset"));
    ITO_TRY(launch_gap_fwd(a, B, HW, C, P32, d_max, s));
    return launch_requant(P32, B, C, d_max, p.target_bits, 0, nullptr, pa, nullptr, 0, d_shift, s);
}

int ito_gap_bwd(const int8_t* dP, const int8_t* a, int B, int HW, int C, int8_t* delta, void* stream)
{
    if (!dP || !a || !delta) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    if (B < 1 || HW < 1 || C < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    return launch_gap_bwd(dP, a, B, HW, C, delta, nullptr, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace ito {
static int check_conv_ws(void* ws, size_t bytes, int B, int H, int W, int IC, int OC, int stride)
{
    if (!ws) return set_error(ITO_ERR_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return set_error(ITO_ERR_ARG, "workspace not 256-byte aligned");
    if (bytes < ito_conv2d_workspace_size(B, H, W, IC, OC, stride))
        return set_error(ITO_ERR_ARG, "workspace too small");
    return ITO_OK;
}
}  // namespace ito
