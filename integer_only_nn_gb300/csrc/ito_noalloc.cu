// ito_linear_fwd_noalloc: the forward Linear layer of ito_linear_fwd for
// callers that cannot allocate device memory while they run. Its scratch (the
// bf16 operand copies that ito_linear_fwd keeps in a caller workspace) is a
// fixed array in the library's own device image instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds ITO_NOALLOC_SCRATCH_BYTES of it until the process exits. Host
// code must not hand the array's name to a kernel: on the host that name is a
// stand-in symbol, not a device address. Its device address is looked up with
// the device current, by the first call in each context of that device: the
// cache is keyed on the driver's process-unique context id, so a
// cudaDeviceReset (which destroys the primary context and with it the array's
// old address) makes the next call look the address up again.
//
// All calls share the one array and it keeps the previous call's contents.
// Each call overwrites every scratch byte the contraction reads, so nothing has
// to start at zero; two calls whose work overlaps on the GPU (different
// streams, no ordering between them) race on the array.
#include <mutex>

#include <cudaTypedefs.h>

#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

static_assert(ITO_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[ITO_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    unsigned long long ctx_id;   // context the address belongs to (0: none yet)
    void* addr;
};
ScratchSlot g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

inline size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Process-unique id of the calling thread's current context, 0 when there is
// none yet or the driver entry points are unavailable (then the address is
// looked up again).
unsigned long long current_context_id()
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current context of the current
// device (looked up by the first call in each context).
int scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return set_error(ITO_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot& slot = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (!slot.addr || id == 0 || slot.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return set_error(ITO_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        slot.addr = p;
        slot.ctx_id = current_context_id();   // the lookup may have created the primary context
    }
    *out = slot.addr;
    return ITO_OK;
}

}  // namespace
}  // namespace ito

using namespace ito;

extern "C" int ito_linear_fwd_noalloc(const int8_t* x, const int8_t* W, int B, int IC, int OC, int relu,
                                      ito_niti_params p, int32_t* y32, uint32_t* d_max, int32_t* d_shift,
                                      int8_t* y, void* stream)
{
    if (!x || !W || !y32 || !d_max || !y) return set_error(ITO_ERR_ARG, "NULL tensor pointer");
    if (B < 1 || IC < 1 || OC < 1) return set_error(ITO_ERR_SHAPE, "sizes must be >= 1");
    if (B > (1 << 20) || IC > (1 << 20) || OC > (1 << 20))
        return set_error(ITO_ERR_SHAPE, "a contraction length above 2^20");
    // bf16 copies of x [B][IC] and W [OC][IC], rows padded to 8 elements
    const int64_t ld = pad8(IC);
    const size_t x_bytes = round256((size_t)2 * B * ld);
    const size_t need = x_bytes + round256((size_t)2 * OC * ld);
    if (need > (size_t)ITO_NOALLOC_SCRATCH_BYTES)
        return set_error(ITO_ERR_SHAPE,
                         "B=%d IC=%d OC=%d needs %zu bytes of scratch; the built-in scratch holds %zu "
                         "(use ito_linear_fwd with a workspace)",
                         B, IC, OC, need, (size_t)ITO_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    int r = scratch_address(&scratch);
    if (r != ITO_OK) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint16_t* xb = static_cast<uint16_t*>(scratch);
    uint16_t* Wb = reinterpret_cast<uint16_t*>(static_cast<char*>(scratch) + x_bytes);
    if ((r = launch_i8_to_bf16(x, B, IC, xb, ld, s)) != ITO_OK) return r;
    if ((r = launch_i8_to_bf16(W, OC, IC, Wb, ld, s)) != ITO_OK) return r;
    cudaError_t e = cudaMemsetAsync(d_max, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
    GemmPlan g;
    if ((r = gemm_plan(&g, Bf16View{xb, B, IC, ld}, false, Bf16View{Wb, OC, IC, ld}, false, B, OC, IC, y32, OC,
                       d_max)) != ITO_OK)
        return r;
    if ((r = gemm_run(g, s)) != ITO_OK) return r;
    return launch_requant(y32, B, OC, d_max, p.target_bits, relu, nullptr, y, nullptr, 0, d_shift, s);
}
