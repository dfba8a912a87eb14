// common.cuh -- device helpers shared by the decode-step kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gd {

// device error word bits (mirrors DEC_FAULT_* of graphdec.h)
constexpr unsigned FAULT_TOKEN = 0x1u;
constexpr unsigned FAULT_POS = 0x2u;
constexpr unsigned FAULT_WRITE_MAP = 0x4u;
constexpr unsigned FAULT_SLOT_MAP = 0x8u;
constexpr unsigned FAULT_WAIT = 0x10u;   // an in-kernel wait gave up (bounded spin)

// ---- programmatic dependent launch (griddepcontrol) ----
// wait: block until the preceding kernel in the stream/graph has completed and
// its writes are visible (no-op when the launch carried no programmatic edge).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// trigger: allow the dependent kernel to start launching its CTAs.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- in-graph trace (profiling) ----
// A trace buffer holds an enable word followed by 4 stamps per recorded
// kernel: [earliest CTA entry, latest CTA past the dependency wait, earliest
// CTA exit, latest CTA exit], in %globaltimer nanoseconds.
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// The trace buffer if this launch records a trace, else null: one global load
// of the enable word per thread that stamps, so a disabled trace costs no
// further round trips.
__device__ __forceinline__ unsigned long long* trace_if_on(unsigned long long* tr) {
    return (tr && *reinterpret_cast<volatile unsigned long long*>(tr)) ? tr : nullptr;
}
// stamp into a buffer that trace_if_on returned (nothing on null)
__device__ __forceinline__ void trace_mark(unsigned long long* on, int id, int slot) {
    if (on) {
        unsigned long long* w = on + 1 + 4 * id + slot;
        const unsigned long long t = gtimer();
        if (slot == 0 || slot == 2) atomicMin(w, t);
        else atomicMax(w, t);
    }
}

// ---- loads ----
// 16-byte streaming load of data read once per step (weights, KV): read-only
// path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16)
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- shared-memory barriers and bulk copies (TMA engine, no tensor map) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make barrier initialisation visible to the async (bulk-copy) proxy
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity to complete: false after
// MBAR_POLLS polls (each poll may suspend briefly), never an endless spin.
constexpr uint32_t MBAR_POLLS = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < MBAR_POLLS; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// named barrier over `threads` threads (a multiple of 32)
__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- bf16 unpacking (exact widening) ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// element type traits: how many elements one 16-byte vector holds and how to
// widen them to fp32
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int VEC = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float load1(const float* p) { return *p; }
    __device__ __forceinline__ static float round_store(float v, float* p) { *p = v; return v; }
    __device__ __forceinline__ static float round(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[8]) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    __device__ __forceinline__ static float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    // round to nearest even, store, and return the stored value widened
    __device__ __forceinline__ static float round_store(float v, __nv_bfloat16* p) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        *p = b;
        return __bfloat162float(b);
    }
    __device__ __forceinline__ static float round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
};

// ---- reductions ----
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// key that orders (value, index) pairs: larger value wins, then lower index
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    unsigned u = __float_as_uint(v);
    unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

}  // namespace gd
