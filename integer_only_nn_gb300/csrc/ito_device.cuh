// Device-side building blocks for the integer training library: the NITI
// scalar rules in integer arithmetic, and thin inline-PTX wrappers for the
// Blackwell (sm_103a) features the contraction kernels use (mbarrier, TMA,
// tcgen05 / TMEM).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ito.h"

namespace ito {

// ------------------------------------------------------------------ limits

constexpr int kNumSMsHint = 152;
// Every bounded wait gives up after this long (ns of %globaltimer) and raises
// ITO_ERR_TIMEOUT in the device error word instead of spinning forever.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Kernels that can fail report into a per-device error word (the first
// failure code wins), passed to them as a pointer; ito_get_error() reads and
// clears it.
__device__ __forceinline__ void raise_device_error(int* err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------- NITI integer rules

// bits_needed = ceil(log2(m + 1)) = number of binary digits of m
// ("Integer On-Device Training: Overview", section 3, NITI Step 2).
__device__ __forceinline__ int bitlen_u32(uint32_t m) { return 32 - __clz(m); }
__device__ __forceinline__ int bitlen_u64(uint64_t m) { return 64 - __clzll(m); }

__device__ __forceinline__ int shift_for(uint32_t max_abs, int target_bits)
{
    int s = bitlen_u32(max_abs) - target_bits;
    return s > 0 ? s : 0;
}

// Round-half-up arithmetic shift (NITI Step 3): floor(y / 2^s + 1/2).
// With y = q * 2^s + r (0 <= r < 2^s, q = y >> s arithmetic), the rounded value
// is q + [r >= 2^(s-1)], and that bracket is bit s-1 of y. No addition that
// could overflow is needed.
__device__ __forceinline__ int32_t rhu32(int32_t y, int s)
{
    if (s == 0) return y;
    return (y >> s) + ((y >> (s - 1)) & 1);
}

__device__ __forceinline__ int64_t rhu64(int64_t y, int s)
{
    if (s == 0) return y;
    if (s >= 63) return 0;   // callers keep |y| < 2^62: floor(y/2^s + 1/2) = 0
    return (y >> s) + ((y >> (s - 1)) & 1);
}

__device__ __forceinline__ int32_t sat8(int32_t v) { return v < -128 ? -128 : (v > 127 ? 127 : v); }
__device__ __forceinline__ int64_t sat16s(int64_t v) { return v < -32767 ? -32767 : (v > 32767 ? 32767 : v); }

__device__ __forceinline__ uint32_t abs_u32(int32_t v)
{
    return v < 0 ? (uint32_t)0 - (uint32_t)v : (uint32_t)v;
}

// Small integers (|v| <= 256) are exact in bf16; this builds the bit pattern
// through an exact float conversion.
__device__ __forceinline__ uint16_t int_to_bf16_bits(int32_t v)
{
    __nv_bfloat16 b = __float2bfloat16_rn((float)v);
    return *reinterpret_cast<uint16_t*>(&b);
}

// Two small integers (|v| <= 256) as one bf16x2 word, lo in the low half, on the
// integer and FP32 add pipes instead of the conversion units. The float with bit
// pattern 0x4B400000 + v is 1.5 * 2^23 + v (its unit in the last place is 1, and
// the mantissa field has room for any |v| < 2^22), so subtracting 1.5 * 2^23 gives
// float(v) exactly. An integer of at most 8 significant bits has a float whose low
// 16 bits are zero, so its bf16 is the float's high half.
__device__ __forceinline__ uint32_t int_pair_to_bf16x2(int32_t lo, int32_t hi)
{
    const float flo = __fsub_rn(__int_as_float(0x4B400000 + lo), 12582912.0f);
    const float fhi = __fsub_rn(__int_as_float(0x4B400000 + hi), 12582912.0f);
    return __byte_perm(__float_as_uint(flo), __float_as_uint(fhi), 0x7632);
}

// 0xff in each byte of g that is positive as a signed int8, 0x00 in the others. Bit 7
// of ((g & 0x7f7f7f7f) + 0x7f7f7f7f) is set in a byte exactly when its low seven bits
// are not all zero (0x7f + 0x7f = 0xfe: no carry reaches the next byte); a positive
// byte is one of those with its sign bit clear.
__device__ __forceinline__ uint32_t bytes_positive_mask(uint32_t g)
{
    const uint32_t pos = ((g & 0x7f7f7f7fu) + 0x7f7f7f7fu) & ~g & 0x80808080u;
    return (pos >> 7) * 0xffu;
}

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up (returns
// false) when *abort is set by another warp of the CTA, or after
// kWaitTimeoutNs, in which case it sets *abort and raises ITO_ERR_TIMEOUT in
// the error word; the caller then unwinds.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                *abort = 1;
                raise_device_error(err, ITO_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Programmatic dependent launch. Every kernel of this library starts with
// griddep_wait(): when it was launched with programmatic stream serialisation
// (launch_pdl) it may already be resident while the previous kernel in the
// stream finishes, and the wait returns once that kernel has completed and its
// memory operations are visible; for a plain launch it returns at once. Only
// then does the kernel touch global memory, and it allows the next kernel to be
// scheduled (griddep_launch_dependents), which waits the same way.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 4-D tiled TMA load (coordinates x innermost); parts of the box outside the tensor read zero.
__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y, int z,
                                            int w)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// --- tcgen05 (5th-generation tensor core, accumulators in tensor memory)

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Load 32 consecutive 32-bit columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Load 16 consecutive 32-bit columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// --- bulk (TMA) stores from shared memory

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, int32_t a, int32_t b, int32_t c, int32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t saddr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr)
                 : "memory");
    return v;
}

// make this thread's generic-proxy shared-memory writes visible to the async (TMA) proxy
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}

// 3-D tiled TMA store from shared memory (coordinates x innermost).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// 4-D tiled TMA store from shared memory (coordinates x innermost; the box is clipped at the
// tensor's edges).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// An L2 cache policy that marks the lines it touches for early eviction: for outputs no
// later kernel of the same pass reads back soon, so that they do not displace operands.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_store_2d with an L2 cache policy
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* src, int x, int y,
                                                  uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::
                     "l"(reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the shared-memory sources of all committed bulk stores have been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until all committed bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// --- thread-block clusters and CTA pairs (cta_group::2)

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// all threads of all CTAs of the cluster
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory that completes on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t mbar_cluster_addr, void* dst, int x,
                                                 int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster_addr), "r"(x), "r"(y)
        : "memory");
}

// TMEM allocation shared by a CTA pair: one warp of each CTA executes these together
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (M = 256 over the pair) (+)= A * B, issued by one thread of the leader CTA
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on the mbarrier at this shared-memory offset in every CTA of `cta_mask`
// once the pair's previously issued MMAs completed
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------ block-wide reductions
//
// Grid-stride kernels fold a per-thread value into one global word. One atomic
// per warp puts thousands of atomics on a single address at the end of such a
// kernel; these reduce over the block first (every thread of the block must
// call them, after its loop) and issue one atomic per block.

template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op)
{
    __shared__ T red[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();                       // red[] may still be read by an earlier call
    if (l == 0) red[w] = v;
    __syncthreads();
    const int nw = (blockDim.x + 31) >> 5;
    v = l < nw ? red[l] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;                              // every thread holds the block's result
}

struct MaxOp {
    template <typename T>
    __device__ __forceinline__ T operator()(T a, T b) const { return a > b ? a : b; }
};
struct AddOp {
    template <typename T>
    __device__ __forceinline__ T operator()(T a, T b) const { return a + b; }
};

__device__ __forceinline__ void block_atomic_max(uint32_t* dst, uint32_t v)
{
    v = block_reduce(v, MaxOp());
    if (threadIdx.x == 0 && v) atomicMax(dst, v);
}

__device__ __forceinline__ void block_atomic_max(unsigned long long* dst, unsigned long long v)
{
    v = block_reduce(v, MaxOp());
    if (threadIdx.x == 0 && v) atomicMax(dst, v);
}

__device__ __forceinline__ void block_atomic_add(uint32_t* dst, uint32_t v)
{
    v = block_reduce(v, AddOp());
    if (threadIdx.x == 0 && v) atomicAdd(dst, v);
}

__device__ __forceinline__ void block_atomic_add(unsigned long long* dst, unsigned long long v)
{
    v = block_reduce(v, AddOp());
    if (threadIdx.x == 0 && v) atomicAdd(dst, v);
}

// Shared-memory matrix descriptor for tcgen05.mma (128-byte swizzle).
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and an fp32 accumulator.
//   bits 4-5 D format (1 = f32)   bits 7-9 A format (1 = bf16)  bits 10-12 B format (1 = bf16)
//   bit 15 A major (1 = MN)        bit 16 B major (1 = MN)
//   bits 17-22 N >> 3              bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace ito
