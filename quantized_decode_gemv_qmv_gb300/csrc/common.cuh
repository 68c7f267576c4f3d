// Device-side building blocks shared by the libqmv kernels: block-format
// constants, the PTX wrappers for mbarriers, bulk asynchronous copies and
// programmatic dependent launch, and bounded waits.
//
// Block formats (GGUF, as described on "llama.cpp 源码完全拆解(十四)：
// mul_mat_vec_q", section "权重的排法", and "GGUF 量化内幕 第16章", 16.1.2):
//   q4_0: half d @0, qs[16] @2                         18 B / 32 weights
//   q4_K: half d @0, half dmin @2, scales[12] @4,
//         qs[128] @16                                  144 B / 256 weights
//   q6_K: ql[128] @0, qh[64] @128, int8 scales[16] @192,
//         half d @208                                  210 B / 256 weights
//   q8_1: half d @0, half s @2, int8 qs[32] @4         36 B / 32 values
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmv {

constexpr int QK4_0 = 32;
constexpr int QK_K = 256;
constexpr int QK8_1 = 32;
constexpr int Q4_0_BYTES = 18;
constexpr int Q4_K_BYTES = 144;
constexpr int Q6_K_BYTES = 210;
constexpr int Q8_1_BYTES = 36;
constexpr int ROW_PAD = 512;  // activation rows are padded to a multiple of this

static_assert(2 + QK4_0 / 2 == Q4_0_BYTES, "q4_0 block size");
static_assert(4 + 12 + QK_K / 2 == Q4_K_BYTES, "q4_K block size");
static_assert(QK_K / 2 + QK_K / 4 + QK_K / 16 + 2 == Q6_K_BYTES, "q6_K block size");
static_assert(4 + QK8_1 == Q8_1_BYTES, "q8_1 block size");

enum Fmt { FMT_Q4_0 = 2, FMT_Q4_K = 12, FMT_Q6_K = 14 };

// Fault codes written to the sticky device word when a bounded wait runs out.
enum FaultCode : unsigned int {
    FAULT_NONE = 0,
    FAULT_WAIT_TIMEOUT = 1,     // a pipeline slot never completed
    FAULT_CLUSTER_STAGING = 2,  // a cluster partner's share of the staged activations never arrived
};

// How long a kernel waits on one mbarrier phase before giving up (ns).  A
// healthy copy completes in microseconds.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

// ---- small helpers ---------------------------------------------------------

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xffffu)));
}

__device__ __forceinline__ int dp4a(int a, int b, int c)
{
    return __dp4a(a, b, c);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Shared-memory loads by 32-bit shared-window address.
__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t a)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ int lds_s8(uint32_t a)
{
    int v;
    asm volatile("ld.shared.s8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// 16 bytes starting at a 2-byte aligned shared address, assembled from five
// aligned 32-bit loads and funnel shifts.
__device__ __forceinline__ void lds16_unaligned2(uint32_t a, uint32_t out[4])
{
    const uint32_t base = a & ~3u;
    const uint32_t sh = (a & 3u) * 8u;  // 0 or 16
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = lds32(base + 4u * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// ---- mbarrier + bulk copy (Blackwell TMA engine) ---------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared accesses before later
// async-proxy (bulk copy) accesses to the same shared memory.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; returns false if
// limit_ns passes first.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Global -> shared bulk copy completing on an mbarrier (both addresses and
// the size multiples of 16 bytes).  The L2 policy marks the weight stream
// evict-first: it is read once per call.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- loads of inputs written by the previous grid ---------------------------
// Activations (and ids) may be produced by the kernel this one overlaps under
// programmatic dependent launch, so they are read after the dependency wait
// through L2 (ld.global.cg), never through the read-only path that assumes the
// data is constant for the kernel's lifetime.

__device__ __forceinline__ uint4 ld_cg_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_cg_f4(const float *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_cg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Read-only (non-coherent) load of a value that nothing writes while this
// kernel runs (biases, read after the dependency wait).
__device__ __forceinline__ float ld_nc_f32(const float *p)
{
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int ld_cg_s32(const int32_t *p)
{
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---- per-thread asynchronous copies (cp.async, 16 bytes) --------------------

// 16-byte global -> shared copy that bypasses registers and L1 (.cg); both
// addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// The same at a constant byte offset from both addresses (an immediate).
template <int OFF>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%2], 16;" ::"r"(dst), "l"(src), "n"(OFF) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most n of this thread's committed copy groups are pending
// (hardware completion of in-flight loads; n is clamped to 0..7).
__device__ __forceinline__ void cp_async_wait(int n)
{
    switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// ---- programmatic dependent launch ------------------------------------------

// Blocks until the grids this grid depends on have completed and their memory
// is visible (a no-op when the launch was not programmatic).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next programmatic launch on the stream begin scheduling its CTAs.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---- thread-block clusters --------------------------------------------------
// A launch without a cluster dimension is a cluster of one CTA: rank 0 of 1,
// and the barriers below complete at once.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the variable at shared::cta address a in the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_v2(uint32_t a, uint32_t v0, uint32_t v1)
{
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(v0), "r"(v1) : "memory");
}

// Stores into another CTA's shared memory (cluster address a) whose byte count
// completes on that CTA's mbarrier (cluster address bar): the receiver waits
// for the bytes it expects instead of a cluster-wide barrier.
__device__ __forceinline__ void st_async_u32(uint32_t a, uint32_t v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(a), "r"(v),
                 "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void st_async_v2(uint32_t a, uint32_t v0, uint32_t v1, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(a),
                 "r"(v0), "r"(v1), "r"(bar)
                 : "memory");
}

// Split cluster barrier (every thread of every CTA of the cluster arrives, then
// waits; a hardware barrier over co-scheduled CTAs, not a spin loop).  The
// relaxed arrive orders nothing (used to know that every CTA has started);
// arrive (release) + wait (acquire) make every thread's earlier shared-memory
// writes, local and remote, visible to the whole cluster.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace qmv
