// prefill.cu -- multi-token prefill of one sequence ("Models, Registry and the
// Driver", "The Model": a step shape is rows x new tokens, positions are
// absolute, so a prefill is a step continuing from a position).
//
// The prompt runs in passes of up to PF_PASS tokens (blocks of PF_T = 128 for
// the tensor cores), layer by layer, so each pass reads every weight once.
// Per pass and layer:
//   RMSNorm -> QKV projection (tensor cores, pf_gemm.cuh) -> RoPE, K/V written
//   into the sequence's store -> causal attention over every position up to
//   each token (flash-style online softmax) -> O projection + residual ->
//   RMSNorm -> gate/up projection with SwiGLU in its epilogue -> down
//   projection + residual.
// After the last pass the final token's hidden state goes through the
// decoder's own head (final RMSNorm, LM head, greedy argmax).  A projection
// splits K over CTAs only when its tiles x token blocks do not fill the GPU;
// the kernel that consumes a projection adds its splits in split order, so
// results do not depend on scheduling.  Unsplit O and down projections add
// into the residual rows in their own epilogue.
//
// Activations enter the tensor cores as bf16 hi + lo rows (about 16
// significant bits, fp32 accumulation); everything else is fp32, and K/V are
// rounded to the KV dtype (bf16) when stored, as in a decode step.
#include <cuda.h>
#include <math.h>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "mma_helpers.cuh"
#include "pf_gemm.cuh"

namespace gd {

namespace {

constexpr int PF_NB = 8;                 // token blocks per pass
constexpr int PF_PASS = PF_NB * PF_T;    // tokens per pass
constexpr int PF_NT = 256;               // threads of the per-token kernels

// hi / lo bf16 rows of one activation value: token t of the pass is row t % PF_T
// of block t / PF_T, whose PF_BN rows are the block's hi rows, then its lo rows
__device__ __forceinline__ size_t hilo_row(int t) { return (size_t)(t / PF_T) * PF_BN + (t % PF_T); }
__device__ __forceinline__ void put_hilo(__nv_bfloat16* hb, int K, int t, int k, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const size_t r = hilo_row(t);
    hb[r * K + k] = hi;
    hb[(r + PF_T) * K + k] = __float2bfloat16_rn(v - __bfloat162float(hi));
}
// four consecutive values (k a multiple of 4)
__device__ __forceinline__ void put_hilo4(__nv_bfloat16* hb, int K, int t, int k, float4 v) {
    const float a[4] = {v.x, v.y, v.z, v.w};
    float h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = bf16_round_f(a[i]);
        l[i] = a[i] - h[i];
    }
    const size_t r = hilo_row(t);
    *reinterpret_cast<uint2*>(hb + r * K + k) = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
    *reinterpret_cast<uint2*>(hb + (r + PF_T) * K + k) = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
}

__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];   // fixed order
    __syncthreads();
    return t;
}

// two bf16 values (low half first) widened exactly to fp32
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// x[t] = E[tok[t]] (fp32) for the pass's tokens; rows past nt are zero.  One
// CTA per token row, 8 values per thread and step.
__global__ void k_pf_embed(const __nv_bfloat16* E, const int* tok, int nt, int d, float* x) {
    const int t = blockIdx.x;
    for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < nt) Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(E + (size_t)tok[t] * d + i), f);
        float4* o = reinterpret_cast<float4*>(x + (size_t)t * d + i);
        o[0] = make_float4(f[0], f[1], f[2], f[3]);
        o[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// x[t] += sum over splits of part[s][t] (when part is given; ntp token rows per
// split); then, when gain is given, hb = hi/lo of x[t] / sqrt(mean(x[t]^2) +
// eps) * gain.  Rows past nt give zero hb rows.  One CTA per token row; the
// row stays in registers between the two passes (d <= 4 PF_NT PF_RN).
constexpr int PF_RN = 8;   // float4 groups per thread
__global__ void k_pf_resid_norm(float* x, const float* part, int splits, int ntp, int d, const __nv_bfloat16* gain,
                                float eps, int nt, __nv_bfloat16* hb) {
    __shared__ float red[PF_NT / 32];
    const int t = blockIdx.x;
    float* xr = x + (size_t)t * d;
    float4 v[PF_RN];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < PF_RN; ++j) {
        const int i = (threadIdx.x + j * PF_NT) * 4;
        if (i < d) {
            v[j] = *reinterpret_cast<const float4*>(xr + i);
            if (part && t < nt)
                for (int s = 0; s < splits; ++s)
                    v[j] = f4add(v[j], __ldg(reinterpret_cast<const float4*>(part + ((size_t)s * ntp + t) * d + i)));
        }
    }
#pragma unroll
    for (int j = 0; j < PF_RN; ++j) {
        const int i = (threadIdx.x + j * PF_NT) * 4;
        if (i < d) {
            if (part && t < nt) *reinterpret_cast<float4*>(xr + i) = v[j];
            ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
        }
    }
    if (!gain) return;
    const float tot = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
#pragma unroll
    for (int j = 0; j < PF_RN; ++j) {
        const int i = (threadIdx.x + j * PF_NT) * 4;
        if (i < d) {
            const uint2 gr = __ldg(reinterpret_cast<const uint2*>(gain + i));
            const float2 g01 = bf16x2_to_f2(gr.x), g23 = bf16x2_to_f2(gr.y);
            const float4 o = t < nt ? make_float4(v[j].x * inv * g01.x, v[j].y * inv * g01.y, v[j].z * inv * g23.x,
                                                  v[j].w * inv * g23.y)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            put_hilo4(hb, d, t, i, o);
        }
    }
}

// the QKV splits of each token: RoPE of q and k at the token's position; q to
// qout (fp32, for attention), k and v rounded to bf16 into the K/V store
struct PfKv {
    __nv_bfloat16* K;
    __nv_bfloat16* V;
    const int* pages;   // paged: the sequence's page table, else null
    int row, Hkv, hd, cap, page;
};
__device__ __forceinline__ size_t kv_off(const PfKv& kv, int g, int pos) {
    if (kv.pages) {
        const int pg = __ldg(kv.pages + pos / kv.page), o = pos % kv.page;
        return (((size_t)pg * kv.Hkv + g) * kv.page + o) * kv.hd;
    }
    return (((size_t)kv.row * kv.Hkv + g) * kv.cap + pos) * kv.hd;
}
// Four consecutive dims per thread and step (16-byte loads), every load of a
// step issued before its arithmetic; the partial sums, the RoPE table and the
// page table are read-only here (non-coherent loads).
__global__ void k_pf_qkv(const float* part, int splits, int ntp, int Hq, int nt, int pos0, const float2* rope,
                         float* qout, PfKv kv) {
    const int t = blockIdx.x;
    if (t >= nt) return;
    const int hd = kv.hd, h2 = hd / 2, qd = Hq * hd, kvd = kv.Hkv * hd, N = qd + 2 * kvd;
    const int pos = pos0 + t;
    const float2* rt = rope + (size_t)pos * h2;
    const int q4 = h2 / 4;                          // 4-dim groups per half head
    const int npair = (Hq + kv.Hkv) * q4;           // q and k: (head, group) pairs
    const int nv = kvd / 4;                         // v: 4-dim groups
    for (int i = threadIdx.x; i < npair + nv; i += blockDim.x) {
        const float* pp = part + (size_t)t * N;
        if (i < npair) {
            const int hh = i / q4, e = (i % q4) * 4;
            const bool is_q = hh < Hq;
            const int base = is_q ? hh * hd : qd + (hh - Hq) * hd;
            float4 a = __ldg(reinterpret_cast<const float4*>(pp + base + e));
            float4 b = __ldg(reinterpret_cast<const float4*>(pp + base + e + h2));
            for (int s = 1; s < splits; ++s) {
                const float* ps = pp + (size_t)s * ntp * N;
                a = f4add(a, __ldg(reinterpret_cast<const float4*>(ps + base + e)));
                b = f4add(b, __ldg(reinterpret_cast<const float4*>(ps + base + e + h2)));
            }
            const float4 c01 = __ldg(reinterpret_cast<const float4*>(rt + e));       // (cos, sin) of e, e + 1
            const float4 c23 = __ldg(reinterpret_cast<const float4*>(rt + e + 2));   // ... of e + 2, e + 3
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
            const float cs[4] = {c01.x, c01.z, c23.x, c23.z}, sn[4] = {c01.y, c01.w, c23.y, c23.w};
            float r0[4], r1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                r0[j] = av[j] * cs[j] - bv[j] * sn[j];
                r1[j] = av[j] * sn[j] + bv[j] * cs[j];
            }
            if (is_q) {
                float* qo = qout + (size_t)t * qd + hh * hd + e;
                *reinterpret_cast<float4*>(qo) = make_float4(r0[0], r0[1], r0[2], r0[3]);
                *reinterpret_cast<float4*>(qo + h2) = make_float4(r1[0], r1[1], r1[2], r1[3]);
            } else {
                __nv_bfloat16* ko = kv.K + kv_off(kv, hh - Hq, pos) + e;
                *reinterpret_cast<uint2*>(ko) = make_uint2(pack_bf16x2(r0[0], r0[1]), pack_bf16x2(r0[2], r0[3]));
                *reinterpret_cast<uint2*>(ko + h2) = make_uint2(pack_bf16x2(r1[0], r1[1]), pack_bf16x2(r1[2], r1[3]));
            }
        } else {
            const int j = (i - npair) * 4, g = j / hd, e = j % hd;
            float4 v = __ldg(reinterpret_cast<const float4*>(pp + qd + kvd + j));
            for (int s = 1; s < splits; ++s)
                v = f4add(v, __ldg(reinterpret_cast<const float4*>(pp + (size_t)s * ntp * N + qd + kvd + j)));
            *reinterpret_cast<uint2*>(kv.V + kv_off(kv, g, pos) + e) =
                make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        }
    }
}

// ---- causal attention on the 5th-generation tensor cores ----
// A CTA takes 128 query rows (the TMEM lanes): 128 / G tokens x the G query
// heads of kv head g, row r = token * G + head.  Per 64-key tile:
//   S = Q K^T        tcgen05.mma, A = Q (bf16 hi rows, then lo rows: two MMAs
//                    into one accumulator), B = the K tile, D in TMEM (two S
//                    buffers, so the next tile's S is computed while this one
//                    is in softmax).  Q carries 1 / sqrt(hd) * log2(e), so
//                    the softmax works in powers of two
//   softmax          four threads per row (warps w, w + 4, w + 8, w + 12 share
//                    TMEM lanes), 16 keys each: the row's tile max through shared memory,
//                    p = 2^(s - m) against the row's reference max m, the sum;
//                    P as bf16 hi + lo rows in shared memory.  The accumulated
//                    O and l are rescaled (O in TMEM, each thread its half of
//                    the columns) only when the row max grows by more than
//                    PA_RESCALE, since O / l is the same for any reference
//   O += P V         tcgen05.mma, A = P (hi, then lo), B = the V tile read
//                    MN-major (V is stored key-major), D = O in TMEM
// K/V tiles arrive by TMA (128-byte swizzle: the layout the MMAs read; one box
// per 64 keys x 64 dims, or per page x 64 dims) in a ring of stages; the
// loader warp then zeroes the V rows past the CTA's last position (they may
// hold any bits, and P = 0 does not clear a NaN).  Warp 16 issues the MMAs.
// All waits are bounded; one that gives up sets FAULT_WAIT and every role
// skips the rest.
constexpr int PA_ROWS = 128;
constexpr int PA_KT = 64;
constexpr int PA_PARTS = 4;                // softmax threads per row
constexpr int PA_SMX = 128 * PA_PARTS;     // softmax threads: warps 0-15
constexpr int PA_THREADS = PA_SMX + 64;    // + warp 16 (MMA) + warp 17 (K/V loads)
constexpr int PA_MMA_WARP = PA_SMX / 32, PA_LOAD_WARP = PA_MMA_WARP + 1;
constexpr int PA_LOAD_T = 32;
constexpr float PA_RESCALE = 8.0f;         // log2 units: p <= 2^8 between rescales
constexpr float PA_LOG2E = 1.4426950408889634f;

// K/V ring stages: as many as fit next to Q and P (3 at head_dim 128, 4 at 64)
__host__ __device__ constexpr int pa_kv_stages(int hd) { return hd >= 128 ? 3 : 4; }
template <int HD>
struct PaLayout {
    static constexpr int NS = pa_kv_stages(HD);
    static constexpr int QB = PA_ROWS * HD * 2;   // Q hi (or lo): HD / 64 atoms of [128 rows x 128 B]
    static constexpr int TB = PA_KT * HD * 2;     // a K (or V) tile: HD / 64 atoms of [64 keys x 128 B]
    static constexpr int PB = PA_ROWS * PA_KT * 2;   // P hi (or lo): one atom of [128 rows x 128 B]
    static constexpr int Q_HI = 0, Q_LO = QB, KV = 2 * QB;   // stage b: K at KV + 2 b TB, V at KV + (2 b + 1) TB
    static constexpr int P_HI = KV + 2 * NS * TB, P_LO = P_HI + PB;
    static constexpr int BYTES = P_LO + PB;
};
__host__ __device__ constexpr int pf_attn_tc_smem(int hd) {
    return 2 * PA_ROWS * hd * 2 + 2 * pa_kv_stages(hd) * PA_KT * hd * 2 + 2 * PA_ROWS * PA_KT * 2 + 1024;
}
// byte offset of 16-byte chunk c (8 bf16) of row r in a [rows x 64] bf16 atom, 128-byte swizzle
__device__ __forceinline__ uint32_t pa_sw(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint64_t pa_desc(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// 2^x by the hardware's base-2 exponential (ex2.approx.ftz; relative error about 2^-22)
__device__ __forceinline__ float pa_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// the softmax warps of a TMEM lane quarter (w, w + 4, ...) meet at barrier 1 + w
__device__ __forceinline__ void pa_part_sync(int quarter) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + quarter), "n"(32 * PA_PARTS) : "memory");
}
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 16) tmem_ld_x16(taddr, r);
    else tmem_ld_x32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
    if constexpr (N == 16) tmem_st_x16(taddr, r);
    else tmem_st_x32(taddr, r);
}

// kvm: this layer's K and V tensor maps (contiguous: rows (row Hkv + g) cap + pos,
// box 64 x 64; paged: rows (page Hkv + g) page + o, box 64 x page)
template <int HD, int G>
__global__ void __launch_bounds__(PA_THREADS, 1) k_pf_attn_tc(const float* q, int Hq, int nt, int pos0, float scale,
                                                              PfKv kv, const CUtensorMap* kvm, unsigned* err,
                                                              __nv_bfloat16* hb) {
    using LY = PaLayout<HD>;
    constexpr int TPC = PA_ROWS / G;   // tokens per CTA
    constexpr int NA = HD / 64;        // 64-column atoms along head_dim
    constexpr int NS = LY::NS;         // K/V ring stages
    extern __shared__ __align__(1024) unsigned char pa_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(pa_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t kv_tma[LY::NS], kv_full[LY::NS], kv_empty[LY::NS], s_full[2], s_free[2], p_full,
        p_free, mma_done;
    __shared__ float pmax[2][PA_PARTS][PA_ROWS];   // [tile parity][part][row]: the parts' tile maxima
    __shared__ float psum[PA_PARTS][PA_ROWS];      // [part][row]: the parts' sums at the end
    __shared__ uint32_t tmem;
    __shared__ int aborted;
    // grid (kv heads, token blocks): CTAs start in x-fastest order, so the token
    // blocks with the most keys (the last ones) come first for every head
    const int g = blockIdx.x, t0 = (gridDim.y - 1 - blockIdx.y) * TPC, tid = threadIdx.x, warp = tid >> 5,
              lane = tid & 31;
    const int qd = Hq * HD;
    const int last = pos0 + min(t0 + TPC, nt) - 1;   // the last key any row of the CTA sees
    const int ntiles = last / PA_KT + 1;
    const float qscale = scale * PA_LOG2E;

    // Q of the CTA's rows as bf16 hi and lo A tiles (scaled by log2(e) / sqrt(hd));
    // every thread's loads are issued before any is used
    {
        constexpr int NQ = (PA_ROWS * (HD / 8) + PA_THREADS - 1) / PA_THREADS;   // 8-column chunks per thread
        float4 qa[NQ][2];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int i = tid + u * PA_THREADS, r = i / (HD / 8), c = i % (HD / 8), tk = t0 + r / G;
            if (i < PA_ROWS * (HD / 8) && tk < nt) {
                const float4* src = reinterpret_cast<const float4*>(q + (size_t)tk * qd + (g * G + r % G) * HD + c * 8);
                qa[u][0] = __ldg(src);
                qa[u][1] = __ldg(src + 1);
            } else {
                qa[u][0] = qa[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int i = tid + u * PA_THREADS, r = i / (HD / 8), c = i % (HD / 8);
            if (i >= PA_ROWS * (HD / 8)) continue;
            const float v[8] = {qa[u][0].x, qa[u][0].y, qa[u][0].z, qa[u][0].w,
                                qa[u][1].x, qa[u][1].y, qa[u][1].z, qa[u][1].w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = v[2 * e] * qscale, x1 = v[2 * e + 1] * qscale;
                const float h0 = bf16_round_f(x0), h1 = bf16_round_f(x1);
                hi[e] = pack_bf16x2(h0, h1);
                lo[e] = pack_bf16x2(x0 - h0, x1 - h1);
            }
            const uint32_t off = (uint32_t)(c / 8) * (PA_ROWS * 128) + pa_sw(r, c % 8);
            *reinterpret_cast<uint4*>(sm + LY::Q_HI + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + LY::Q_LO + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&tmem))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int b = 0; b < NS; ++b) {
            mbar_init(&kv_tma[b], 1);
            mbar_init(&kv_full[b], PA_LOAD_T);
            mbar_init(&kv_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], PA_SMX);
        }
        mbar_init(&p_full, PA_SMX);
        mbar_init(&p_free, 1);
        mbar_init(&mma_done, 1);
        aborted = 0;
        mbar_fence_init();
    }
    fence_proxy_async_smem();   // Q's generic writes before the tensor core reads them
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t dt = tmem;           // S buffers at columns 0 and 64, O at 128
    volatile int* ab = &aborted;
    auto give_up = [&]() {
        *ab = 1;
        atomicOr(err, FAULT_WAIT);
    };

    if (warp == PA_LOAD_WARP) {
        // ---- K/V loader warp: lane 0 issues the TMA boxes, the warp zeroes late V rows ----
        for (int j = 0; j < ntiles; ++j) {
            const int b = j % NS, j0 = j * PA_KT;
            unsigned char* kd = sm + LY::KV + 2 * b * LY::TB;
            unsigned char* vd = kd + LY::TB;
            if (lane == 0) {
                if (j >= NS && !(*ab) && !mbar_wait(&kv_empty[b], (uint32_t)((j / NS) - 1) & 1u)) give_up();
                if (!*ab) {
                    if (kv.pages) {
                        const int np = (min(j0 + PA_KT - 1, last) - j0) / kv.page + 1;   // pages holding keys <= last
                        mbar_arrive_expect_tx(&kv_tma[b], (uint32_t)(np * 2 * NA * kv.page * 128));
                        for (int pi = 0; pi < np; ++pi) {
                            const int key = j0 + pi * kv.page;
                            const int y = (kv.pages[key / kv.page] * kv.Hkv + g) * kv.page;
#pragma unroll
                            for (int a = 0; a < NA; ++a) {
                                const uint32_t o = (uint32_t)a * (PA_KT * 128) + (uint32_t)(pi * kv.page * 128);
                                tma_load_2d(kd + o, kvm, a * 64, y, &kv_tma[b]);
                                tma_load_2d(vd + o, kvm + 1, a * 64, y, &kv_tma[b]);
                            }
                        }
                    } else {
                        const int y = (kv.row * kv.Hkv + g) * kv.cap + j0;
                        mbar_arrive_expect_tx(&kv_tma[b], (uint32_t)(2 * NA * PA_KT * 128));
#pragma unroll
                        for (int a = 0; a < NA; ++a) {
                            tma_load_2d(kd + a * (PA_KT * 128), kvm, a * 64, y, &kv_tma[b]);
                            tma_load_2d(vd + a * (PA_KT * 128), kvm + 1, a * 64, y, &kv_tma[b]);
                        }
                    }
                }
            }
            __syncwarp();
            if (!*ab && !mbar_wait(&kv_tma[b], (uint32_t)(j / NS) & 1u)) give_up();
            // V rows of keys past `last` become zero
            const int k1 = last - j0 + 1;   // keys of the tile that are <= last
            if (!*ab && k1 < PA_KT)
                for (int i = lane; i < (PA_KT - k1) * (HD / 8); i += PA_LOAD_T) {
                    const int kk = k1 + i / (HD / 8), c = i % (HD / 8);
                    *reinterpret_cast<uint4*>(vd + (c / 8) * (PA_KT * 128) + pa_sw(kk, c % 8)) = make_uint4(0u, 0u, 0u, 0u);
                }
            fence_proxy_async_smem();   // the zeroes (generic proxy) before the tensor core reads the tile
            mbar_arrive(&kv_full[b]);
        }
    } else if (warp == PA_MMA_WARP) {
        // ---- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t id_s = pf_idesc(128, PA_KT);
            constexpr uint32_t id_o = pf_idesc(128, HD) | (1u << 16);   // B (V) MN-major
            const uint32_t qhi = smem_u32(sm + LY::Q_HI), qlo = smem_u32(sm + LY::Q_LO);
            const uint32_t phi = smem_u32(sm + LY::P_HI), plo = smem_u32(sm + LY::P_LO);
            auto pv = [&](int jj) {   // O += P V of tile jj (after its P is written)
                if (*ab || !mbar_wait(&p_full, (uint32_t)jj & 1u)) {
                    give_up();
                    return;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t vt = smem_u32(sm + LY::KV + (2 * (jj % NS) + 1) * LY::TB);
#pragma unroll
                for (int kk = 0; kk < PA_KT / 16; ++kk) {
                    const uint64_t bv = pa_desc(vt + 2048u * kk, PA_KT * 128);
                    umma_bf16(dt + 128, pa_desc(phi + 32u * kk, 16), bv, id_o, (jj > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16(dt + 128, pa_desc(plo + 32u * kk, 16), bv, id_o, 1u);
                }
                umma_commit(&kv_empty[jj % NS]);   // the tile's K/V stage is free
                umma_commit(&p_free);              // P may be rewritten, O is settled
            };
            for (int j = 0; j < ntiles && !*ab; ++j) {
                const int b = j & 1, kb = j % NS;   // S buffer, K/V stage
                if (!mbar_wait(&kv_full[kb], (uint32_t)(j / NS) & 1u) ||
                    (j >= 2 && !mbar_wait(&s_free[b], (uint32_t)((j >> 1) - 1) & 1u))) {
                    give_up();
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t kt = smem_u32(sm + LY::KV + 2 * kb * LY::TB);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t ko = (uint32_t)(kk / 4) * (PA_KT * 128) + 32u * (kk % 4);
                    const uint32_t qo = (uint32_t)(kk / 4) * (PA_ROWS * 128) + 32u * (kk % 4);
                    const uint64_t bk = pa_desc(kt + ko, 16);
                    umma_bf16(dt + (uint32_t)(b * PA_KT), pa_desc(qhi + qo, 16), bk, id_s, kk > 0 ? 1u : 0u);
                    umma_bf16(dt + (uint32_t)(b * PA_KT), pa_desc(qlo + qo, 16), bk, id_s, 1u);
                }
                umma_commit(&s_full[b]);
                if (j >= 1) pv(j - 1);
            }
            if (!*ab) pv(ntiles - 1);
            // every MMA issued has finished before TMEM is released (also after a give-up)
            umma_commit(&mma_done);
            if (!mbar_wait(&mma_done, 0u)) give_up();
        }
        __syncwarp();
    } else {
        // ---- softmax warps: warp w reads TMEM lanes 32 (w % 4) + lane, i.e. row
        // r = 32 (w % 4) + lane; part = w / 4 takes keys KPT part .. + KPT - 1 of
        // each tile and O columns OC part .. + OC - 1 ----
        constexpr int KPT = PA_KT / PA_PARTS, OC = HD / PA_PARTS;
        const int quarter = warp & 3, part = warp >> 2, r = quarter * 32 + lane;
        const int tk = t0 + r / G, qpos = pos0 + tk;
        const bool live = tk < nt;
        const uint32_t lrow = dt + ((uint32_t)(quarter * 32) << 16);
        const uint32_t ocol = 128u + (uint32_t)(part * OC);   // this thread's O columns in TMEM
        const int diag0 = pos0 + t0;   // the smallest position of the CTA's rows: earlier keys are seen by every row
        float m_ref = -INFINITY, l = 0.f;
        // tcgen05.ld / st are warp-wide: every condition around them is made warp-uniform
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1, j0 = j * PA_KT + KPT * part;   // this thread's first key of the tile
            bool ok = __all_sync(0xffffffffu, !*ab && mbar_wait(&s_full[b], (uint32_t)(j >> 1) & 1u));
            if (!ok) give_up();
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t sv[KPT];
            if (ok) {
                tmem_ld_n<KPT>(lrow + (uint32_t)(b * PA_KT + KPT * part), sv);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&s_free[b]);
            const bool all_seen = j * PA_KT + PA_KT - 1 <= diag0;   // CTA-uniform: no key of the tile is masked
            // this part's max over the visible keys (masked keys by select), then the row's
            float mt = -INFINITY;
#pragma unroll
            for (int t = 0; t < KPT; ++t)
                if (all_seen || j0 + t <= qpos) mt = fmaxf(mt, __uint_as_float(sv[t]));
            pmax[b][part][r] = mt;
            pa_part_sync(quarter);
#pragma unroll
            for (int o = 0; o < PA_PARTS; ++o) mt = fmaxf(mt, pmax[b][o][r]);
            // a new reference max when the row's max grows by more than PA_RESCALE
            const bool need = mt > m_ref + PA_RESCALE || m_ref == -INFINITY;
            const float mn = need ? fmaxf(mt, m_ref) : m_ref;
            const float alpha = (need && m_ref != -INFINITY && mn != -INFINITY) ? pa_exp2(m_ref - mn) : 1.f;
            l *= alpha;
            m_ref = mn;
            // P = 2^(s - m_ref) as bf16 hi and lo rows, in registers while P V of tile j - 1 runs
            float ps = 0.f;
            uint4 ph[KPT / 8], pl[KPT / 8];
#pragma unroll
            for (int c = 0; c < KPT / 8; ++c) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float pv2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = 8 * c + 2 * e + u;
                        const float sc = __uint_as_float(sv[col]);
                        pv2[u] = ((all_seen || j0 + col <= qpos) && m_ref != -INFINITY) ? pa_exp2(sc - m_ref) : 0.f;
                        ps += pv2[u];
                    }
                    const float h0 = bf16_round_f(pv2[0]), h1 = bf16_round_f(pv2[1]);
                    hi[e] = pack_bf16x2(h0, h1);
                    lo[e] = pack_bf16x2(pv2[0] - h0, pv2[1] - h1);
                }
                ph[c] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                pl[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            l += ps;
            // P(j - 1) has been consumed (and O settled) before P or O is touched
            if (j >= 1 && ok) {
                ok = __all_sync(0xffffffffu, !*ab && mbar_wait(&p_free, (uint32_t)(j - 1) & 1u));
                if (!ok) give_up();
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            }
            if (ok && j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {   // O holds tiles 0 .. j - 1
                uint32_t ov[OC];
                tmem_ld_n<OC>(lrow + ocol, ov);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int t = 0; t < OC; ++t) ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
                tmem_st_n<OC>(lrow + ocol, ov);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
#pragma unroll
            for (int c = 0; c < KPT / 8; ++c) {
                *reinterpret_cast<uint4*>(sm + LY::P_HI + pa_sw(r, (KPT / 8) * part + c)) = ph[c];
                *reinterpret_cast<uint4*>(sm + LY::P_LO + pa_sw(r, (KPT / 8) * part + c)) = pl[c];
            }
            fence_proxy_async_smem();   // P's generic writes before the tensor core reads them
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&p_full);
        }
        // O / l after the last P V (the row's own position is always visible: l > 0)
        psum[part][r] = l;
        pa_part_sync(quarter);
        float lt = 0.f;
#pragma unroll
        for (int o = 0; o < PA_PARTS; ++o) lt += psum[o][r];
        const float inv = 1.0f / lt;
        const bool ok = __all_sync(0xffffffffu, !*ab && mbar_wait(&p_free, (uint32_t)(ntiles - 1) & 1u));
        if (!ok) give_up();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        uint32_t ov[OC];
        tmem_ld_n<OC>(lrow + ocol, ov);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (ok && live) {
            const int head = g * G + r % G;
#pragma unroll
            for (int t = 0; t < OC; t += 4)
                put_hilo4(hb, qd, tk, head * HD + part * OC + t,
                          make_float4(__uint_as_float(ov[t]) * inv, __uint_as_float(ov[t + 1]) * inv,
                                      __uint_as_float(ov[t + 2]) * inv, __uint_as_float(ov[t + 3]) * inv));
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(dt) : "memory");
    }
}

// rows of zeros for the hi/lo activation rows past the pass's tokens (the
// attention kernel writes only live rows)
__global__ void k_pf_zero_rows(__nv_bfloat16* hb, int K, int nt) {
    const int t = nt + blockIdx.x;
    for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) put_hilo4(hb, K, t, k, make_float4(0.f, 0.f, 0.f, 0.f));
}

typedef CUresult (*PfEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PfEncodeFn pf_encoder() {
    static PfEncodeFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PfEncodeFn>(f);
    }
    return fn;
}

// a [rows, cols] bf16 row-major matrix as TMA tiles of [box_rows, 64] (128-byte swizzle)
bool pf_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    PfEncodeFn fn = pf_encoder();
    if (!fn || ((uintptr_t)base & 15) || (cols * 2) % 16) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)PF_BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K splits (a divisor of the K steps, at most 16, at least 4 K steps each)
// with the shortest modelled time: waves of the GPU's CTA slots x (K steps per
// split + PF_CTA_COST, a CTA's fixed cost of pipeline fill and epilogue in K
// steps).  More splits must win by a tenth: each adds a pass of partial sums
// for the consuming kernel to read.
constexpr int PF_CTA_COST = 6;
int pf_splits(int tiles, int ksteps, int num_sms) {
    const int slots = num_sms * PF_CTAS_PER_SM;
    int best = 1;
    long long best_t = -1;
    for (int s = 1; s <= 16; ++s) {
        if (ksteps % s || (s > 1 && ksteps / s < 4)) continue;
        const long long waves = ((long long)tiles * s + slots - 1) / slots;
        const long long t = waves * (ksteps / s + PF_CTA_COST);
        if (best_t < 0 || 10 * t < 9 * best_t) {
            best_t = t;
            best = s;
        }
    }
    return best;
}

}  // namespace

// one projection: up to three stacked weight segments
struct PfProj {
    PfGemmParams p{};
    int tiles = 0, K = 0;
    bool add = false;      // O / down: unsplit launches add into the residual rows
    bool swiglu = false;   // gate/up: never split, SwiGLU epilogue
};

struct PrefillState {
    PrefillArgs a;
    int num_sms = 0;
    float *x = nullptr, *part = nullptr, *q = nullptr;
    __nv_bfloat16* hb = nullptr;    // hi/lo rows of the projections with K = d or Hq hd
    __nv_bfloat16* hb2 = nullptr;   // hi/lo rows of the down projection (K = F)
    int* tok = nullptr;
    int* pages = nullptr;
    std::vector<PfProj> proj;   // per layer: qkv, o, gate/up, down
    size_t part_floats = 0;
    CUtensorMap* kvmaps = nullptr;   // device [L][K, V]: the attention's TMA maps of the K/V stores
};

// the partial-sum buffer: the largest splits x token rows x N over the
// projections and the pass sizes (1..PF_NB blocks)
size_t prefill_part_floats(const PrefillArgs& a, int num_sms) {
    const int qd = a.Hq * a.hd, kvd = a.Hkv * a.hd;
    size_t most = 0;
    auto need = [&](int N, int K) {
        const int tiles = (N + 127) / 128;
        for (int nb = 1; nb <= PF_NB; ++nb) {
            const int s = pf_splits(tiles * nb, K / PF_BK, num_sms);
            const size_t v = (size_t)s * nb * PF_T * N;
            if (v > most) most = v;
        }
    };
    need(qd + 2 * kvd, a.d);
    need(a.d, qd);
    need(a.d, a.F);
    return most;
}

bool prefill_supported(const PrefillArgs& a) {
    const int qd = a.Hq * a.hd;
    if (a.hd != 64 && a.hd != 128) return false;
    const int G = a.Hq / a.Hkv;
    if (G != 2 && G != 4) return false;
    if (a.d % PF_BK || qd % PF_BK || a.F % PF_BK) return false;
    if (a.d > 4 * PF_NT * PF_RN) return false;   // the norm kernel's row in registers
    if (a.paged && (a.page < 8 || 64 % a.page)) return false;   // whole 8-row swizzle atoms per page box
    return true;
}

void prefill_free(PrefillState* s) {
    if (!s) return;
    cudaFree(s->x);
    cudaFree(s->part);
    cudaFree(s->q);
    cudaFree(s->hb);
    cudaFree(s->hb2);
    cudaFree(s->tok);
    cudaFree(s->pages);
    cudaFree(s->kvmaps);
    delete s;
}

static const void* pf_attn_fn(int hd, int G) {
    if (hd == 128) {
        if (G == 4) return (const void*)&k_pf_attn_tc<128, 4>;
        if (G == 2) return (const void*)&k_pf_attn_tc<128, 2>;
    } else if (hd == 64) {
        if (G == 4) return (const void*)&k_pf_attn_tc<64, 4>;
        if (G == 2) return (const void*)&k_pf_attn_tc<64, 2>;
    }
    return nullptr;
}

cudaError_t prefill_create(const PrefillArgs& a, int num_sms, PrefillState** out) {
    *out = nullptr;
    PrefillState* s = new PrefillState();
    s->a = a;
    s->num_sms = num_sms;
    const int qd = a.Hq * a.hd, kvd = a.Hkv * a.hd;
    const int kmax = a.d > qd ? a.d : qd;
    s->part_floats = prefill_part_floats(a, num_sms);
    const long long hrows = (long long)PF_NB * PF_BN;   // hi/lo activation rows of a pass
    cudaError_t e;
    if ((e = cudaMalloc(&s->x, sizeof(float) * PF_PASS * a.d)) != cudaSuccess ||
        (e = cudaMalloc(&s->part, sizeof(float) * s->part_floats)) != cudaSuccess ||
        (e = cudaMalloc(&s->q, sizeof(float) * PF_PASS * qd)) != cudaSuccess ||
        (e = cudaMalloc(&s->hb, sizeof(__nv_bfloat16) * hrows * kmax)) != cudaSuccess ||
        (e = cudaMalloc(&s->hb2, sizeof(__nv_bfloat16) * hrows * a.F)) != cudaSuccess ||
        (e = cudaMalloc(&s->tok, sizeof(int) * a.cap)) != cudaSuccess ||
        (e = cudaMalloc(&s->pages, sizeof(int) * (a.paged ? a.ppr : 1))) != cudaSuccess ||
        (e = cudaMalloc(&s->kvmaps, sizeof(CUtensorMap) * 2 * a.L)) != cudaSuccess) {
        cudaGetLastError();
        prefill_free(s);
        return e;
    }
    // tensor maps: every layer's weights, and the hi/lo activation rows for K = d, qd, F
    CUtensorMap hd_map, hq_map, hf_map;
    if (!pf_map(&hd_map, s->hb, hrows, a.d, PF_BN) || !pf_map(&hq_map, s->hb, hrows, qd, PF_BN) ||
        !pf_map(&hf_map, s->hb2, hrows, a.F, PF_BN)) {
        prefill_free(s);
        return cudaErrorInvalidValue;
    }
    auto proj = [&](const void* w0, int n0, const void* w1, int n1, const void* w2, int n2, int K,
                    const CUtensorMap& hm, PfProj& pr) {
        const void* w[3] = {w0, w1, w2};
        const int n[3] = {n0, n1, n2};
        PfGemmParams& p = pr.p;
        p.nseg = 0;
        int tiles = 0, rows = 0;
        for (int k = 0; k < 3; ++k) {
            if (!w[k] || !n[k]) continue;
            if (!pf_map(&p.map_w[p.nseg], w[k], n[k], K, 128)) return false;
            p.tile0[p.nseg] = tiles;
            p.row0[p.nseg] = rows;
            p.rows[p.nseg] = n[k];
            tiles += (n[k] + 127) / 128;
            rows += n[k];
            ++p.nseg;
        }
        p.tile0[p.nseg] = tiles;
        p.map_h = hm;
        p.N = rows;
        p.part = s->part;
        p.x = s->x;
        p.err = a.err;
        pr.tiles = tiles;
        pr.K = K;
        return true;
    };
    // gate/up: tile i = gate rows [64 i, 64 i + 64) over the same up rows, written
    // as silu(gate) * up into the down projection's hi/lo rows
    auto proj_gu = [&](const void* wg, const void* wu, PfProj& pr) {
        PfGemmParams& p = pr.p;
        if (!pf_map(&p.map_w[0], wg, a.F, a.d, 64) || !pf_map(&p.map_w[1], wu, a.F, a.d, 64)) return false;
        p.nseg = 1;
        p.tile0[0] = 0;
        p.tile0[1] = a.F / 64;
        p.row0[0] = 0;
        p.rows[0] = a.F;
        p.map_h = hd_map;
        p.N = a.F;
        p.mode = PF_EPI_SWIGLU;
        p.hb_out = s->hb2;
        p.err = a.err;
        pr.tiles = a.F / 64;
        pr.K = a.d;
        pr.swiglu = true;
        return true;
    };
    s->proj.resize((size_t)a.L * 4);
    for (int l = 0; l < a.L; ++l) {
        const void* const* w = a.lw + (size_t)l * 9;   // attn_norm, q, k, v, o, ffn_norm, gate, up, down
        if (!proj(w[1], qd, w[2], kvd, w[3], kvd, a.d, hd_map, s->proj[4 * l + 0]) ||
            !proj(w[4], a.d, nullptr, 0, nullptr, 0, qd, hq_map, s->proj[4 * l + 1]) ||
            !proj_gu(w[6], w[7], s->proj[4 * l + 2]) ||
            !proj(w[8], a.d, nullptr, 0, nullptr, 0, a.F, hf_map, s->proj[4 * l + 3])) {
            prefill_free(s);
            return cudaErrorInvalidValue;
        }
        s->proj[4 * l + 1].add = true;
        s->proj[4 * l + 3].add = true;
    }
    // the attention's K/V tensor maps, one pair per layer
    {
        std::vector<CUtensorMap> km((size_t)2 * a.L);
        const long long kvrows = a.paged ? (long long)a.num_pages * a.Hkv * a.page : (long long)a.rows * a.Hkv * a.cap;
        const int box = a.paged ? a.page : PA_KT;
        for (int l = 0; l < a.L; ++l)
            if (!pf_map(&km[2 * l], a.K[l], kvrows, a.hd, box) || !pf_map(&km[2 * l + 1], a.V[l], kvrows, a.hd, box)) {
                prefill_free(s);
                return cudaErrorInvalidValue;
            }
        if ((e = cudaMemcpy(s->kvmaps, km.data(), km.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice)) !=
            cudaSuccess) {
            prefill_free(s);
            return e;
        }
    }
    if ((e = cudaFuncSetAttribute(k_pf_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(pf_attn_fn(a.hd, a.Hq / a.Hkv), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pf_attn_tc_smem(a.hd))) != cudaSuccess) {
        prefill_free(s);
        return e;
    }
    *out = s;
    return cudaSuccess;
}

// one projection over nb token blocks; *splits gets its K splits (0: the
// epilogue added into the residual rows or wrote SwiGLU, nothing to add up)
static cudaError_t pf_gemm_launch(const PrefillState* s, const PfProj& pr, int nb, int* splits, cudaStream_t st) {
    const int ks = pr.K / PF_BK;
    const int sp = pr.swiglu ? 1 : pf_splits(pr.tiles * nb, ks, s->num_sms);
    PfGemmParams p = pr.p;
    p.ksteps = ks / sp;
    p.ntp = nb * PF_T;
    if (!pr.swiglu) p.mode = (pr.add && sp == 1) ? PF_EPI_ADD : PF_EPI_PART;
    if (p.mode == PF_EPI_PART && (size_t)sp * p.ntp * p.N > s->part_floats) return cudaErrorInvalidValue;
    *splits = p.mode == PF_EPI_PART ? sp : 0;
    k_pf_gemm<<<dim3(nb, pr.tiles, sp), PF_THREADS, PF_SMEM, st>>>(p);
    return cudaGetLastError();
}

cudaError_t prefill_run(PrefillState* s, const int* tokens, int n, int pos0, int row, const int* pages,
                        float* x_last, cudaStream_t st) {
    const PrefillArgs& a = s->a;
    const int qd = a.Hq * a.hd, G = a.Hq / a.Hkv;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(s->tok, tokens, sizeof(int) * n, cudaMemcpyHostToDevice, st)) != cudaSuccess) return e;
    if (a.paged &&
        (e = cudaMemcpyAsync(s->pages, pages, sizeof(int) * a.ppr, cudaMemcpyHostToDevice, st)) != cudaSuccess)
        return e;
    const void* attn = pf_attn_fn(a.hd, G);
    if (!attn) return cudaErrorInvalidValue;
    const float scale = (float)(1.0 / sqrt((double)a.hd));
    for (int c0 = 0; c0 < n; c0 += PF_PASS) {
        int nt = n - c0 < PF_PASS ? n - c0 : PF_PASS;
        const int nb = (nt + PF_T - 1) / PF_T, ntp = nb * PF_T;
        int p0 = pos0 + c0;
        k_pf_embed<<<ntp, PF_NT, 0, st>>>(static_cast<const __nv_bfloat16*>(a.embed), s->tok + c0, nt, a.d, s->x);
        k_pf_resid_norm<<<ntp, PF_NT, 0, st>>>(s->x, nullptr, 0, ntp, a.d,
                                               static_cast<const __nv_bfloat16*>(a.lw[0]), a.eps, nt, s->hb);
        for (int l = 0; l < a.L; ++l) {
            const void* const* w = a.lw + (size_t)l * 9;
            PfKv kv{static_cast<__nv_bfloat16*>(a.K[l]), static_cast<__nv_bfloat16*>(a.V[l]),
                    a.paged ? s->pages : nullptr, row, a.Hkv, a.hd, a.cap, a.page};
            int sp = 1;
            if ((e = pf_gemm_launch(s, s->proj[4 * l + 0], nb, &sp, st)) != cudaSuccess) return e;
            k_pf_qkv<<<nt, PF_NT, 0, st>>>(s->part, sp, ntp, a.Hq, nt, p0, a.rope, s->q, kv);
            if (nt < ntp) k_pf_zero_rows<<<ntp - nt, PF_NT, 0, st>>>(s->hb, qd, nt);
            {
                unsigned* errp = a.err;
                const CUtensorMap* kvm = s->kvmaps + 2 * l;
                void* args[] = {&s->q,   const_cast<int*>(&a.Hq), &nt,   &p0, const_cast<float*>(&scale),
                                &kv,     &kvm,                    &errp, &s->hb};
                const int tpc = PA_ROWS / G;   // tokens per attention CTA
                if ((e = cudaLaunchKernel(attn, dim3(a.Hkv, (nt + tpc - 1) / tpc), dim3(PA_THREADS), args,
                                          pf_attn_tc_smem(a.hd), st)) != cudaSuccess)
                    return e;
            }
            if ((e = pf_gemm_launch(s, s->proj[4 * l + 1], nb, &sp, st)) != cudaSuccess) return e;
            k_pf_resid_norm<<<ntp, PF_NT, 0, st>>>(s->x, sp ? s->part : nullptr, sp, ntp, a.d,
                                                   static_cast<const __nv_bfloat16*>(w[5]), a.eps, nt, s->hb);
            if ((e = pf_gemm_launch(s, s->proj[4 * l + 2], nb, &sp, st)) != cudaSuccess) return e;
            if ((e = pf_gemm_launch(s, s->proj[4 * l + 3], nb, &sp, st)) != cudaSuccess) return e;
            const __nv_bfloat16* next_gain =
                l + 1 < a.L ? static_cast<const __nv_bfloat16*>(a.lw[(size_t)(l + 1) * 9 + 0]) : nullptr;
            if (sp || next_gain)
                k_pf_resid_norm<<<ntp, PF_NT, 0, st>>>(s->x, sp ? s->part : nullptr, sp, ntp, a.d, next_gain, a.eps,
                                                       nt, s->hb);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        if (c0 + PF_PASS >= n &&
            (e = cudaMemcpyAsync(x_last, s->x + (size_t)(nt - 1) * a.d, sizeof(float) * a.d, cudaMemcpyDeviceToDevice,
                                 st)) != cudaSuccess)
            return e;
    }
    return cudaGetLastError();
}

}  // namespace gd
