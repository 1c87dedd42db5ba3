// extern "C" entry points of libito.so: argument checking, workspace layout
// and launch order of the single-layer operations. The model (INT_LAYERS-like
// stack and the whole training step) is in ito_model.cu.
#include <cstdarg>
#include <cstdio>
#include <cstring>

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

}  // extern "C"
