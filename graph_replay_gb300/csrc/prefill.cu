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

// 16-byte asynchronous copy global -> shared; zero bytes read (the 16 bytes
// zero-filled) when !valid
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every copy group of this thread but the newest has landed
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Causal attention on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate), flash-style.  A CTA takes 64 query rows -- PF_QR / G tokens x
// the G query heads of kv head g, row r = token * G + head -- and sweeps the
// keys [0, last position of its tokens] in tiles of PF_KT2 keys, double
// buffered: the next tile's asynchronous copies are in flight while the
// current one is computed.  The CTAs with the most keys start first.  Q lives
// in shared memory (read by ldmatrix at every k-step), so a thread stays under
// 128 registers and two CTAs share an SM.  Warp w owns
// query rows 8w..8w+7: the MMA's 16 A rows hold their bf16 parts (rows 0-7) and
// remainders (rows 8-15), so q keeps about 16 significant bits; S = Q K^T comes
// out as hi + lo row pairs, and P (online softmax, fp32) goes back into the
// next MMA's A fragments the same way, straight from the registers.  K and V
// tiles are staged in shared memory (rows padded by 16 bytes: conflict-free
// ldmatrix); V is read transposed.  The output goes to hb as the O projection's
// hi/lo activation rows.
constexpr int PF_QR = 64;          // query rows per CTA
constexpr int PF_KT2 = 32;         // keys per tile
// dynamic shared memory of the attention kernel: two K and two V tiles, and the
// CTA's Q as 8 warps x 16 rows (bf16 parts, then remainders)
__host__ __device__ constexpr int pf_attn_smem(int hd) { return (4 * PF_KT2 + 128) * (hd + 8) * 2; }
// 2 CTAs per SM: Q in shared memory and 32-key tiles keep a thread under 128 registers
template <int HD, int G>
__global__ void __launch_bounds__(256, 2) k_pf_attn_mma(const float* q, int Hq, int nt, int pos0, float scale, PfKv kv,
                                                        __nv_bfloat16* hb) {
    constexpr int KS = HD / 16;            // k-steps of S = Q K^T
    constexpr int DT = HD / 8;             // n-tiles of O
    constexpr int NT = PF_KT2 / 8;         // n-tiles of S
    constexpr int RS = HD + 8;             // shared row stride (bf16)
    constexpr int TPC = PF_QR / G;         // tokens per CTA
    constexpr int TILE = PF_KT2 * RS;      // elements of one K (or V) tile
    extern __shared__ __align__(16) __nv_bfloat16 pf_kv_smem[];   // K0, K1, V0, V1, Q
    const int g = blockIdx.y, t0 = (gridDim.x - 1 - blockIdx.x) * TPC, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int qd = Hq * HD;
    // this lane's query row (warp row gq) and its position
    const int r = warp * 8 + gq, tok = t0 + r / G, head = g * G + r % G;
    const bool live = tok < nt;
    const int qpos = pos0 + tok;
    // this warp's Q as the MMA's A tile: rows 0-7 bf16(q * scale) of its 8 query
    // rows, rows 8-15 the remainders (read back by ldmatrix at every tile)
    __nv_bfloat16* q_s = pf_kv_smem + 4 * TILE + warp * 16 * RS;
    for (int i = lane; i < 8 * HD; i += 32) {
        const int qr = i / HD, c = i % HD, rw = warp * 8 + qr, tk = t0 + rw / G;
        const float v = tk < nt ? q[(size_t)tk * qd + (g * G + rw % G) * HD + c] * scale : 0.f;
        const float hi = bf16_round_f(v);
        q_s[qr * RS + c] = __float2bfloat16_rn(hi);
        q_s[(8 + qr) * RS + c] = __float2bfloat16_rn(v - hi);
    }
    __syncwarp();
    float o[DT][4];
#pragma unroll
    for (int n = 0; n < DT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const int last = pos0 + min(t0 + TPC, nt) - 1;               // the last key any row of the CTA sees
    const int wlast = pos0 + min(t0 + (warp * 8 + 7) / G + 1, nt) - 1;   // ... any row of this warp
    // copies of the tile at key j0 into buffer b (keys past `last` zero-filled)
    auto load_tile = [&](int j0, int b) {
        __nv_bfloat16* kd = pf_kv_smem + b * TILE;
        __nv_bfloat16* vd = pf_kv_smem + (2 + b) * TILE;
        for (int i = tid; i < PF_KT2 * (HD / 8); i += 256) {   // 16-byte vectors of K and V
            const int kk = i / (HD / 8), c = i % (HD / 8), j = j0 + kk;
            const bool in = j <= last;
            const size_t off = in ? kv_off(kv, g, j) + (size_t)c * 8 : 0;
            cp_async16(kd + kk * RS + c * 8, kv.K + off, in);
            cp_async16(vd + kk * RS + c * 8, kv.V + off, in);
        }
        cp_async_commit();
    };
    load_tile(0, 0);
    int it = 0;
    for (int j0 = 0; j0 <= last; j0 += PF_KT2, ++it) {
        if (j0 + PF_KT2 <= last) {
            load_tile(j0 + PF_KT2, (it + 1) & 1);
        } else {
            cp_async_commit();   // an empty group: the wait below still means "this tile has landed"
        }
        cp_async_wait_prev();
        __syncthreads();   // every thread's copies of this tile are visible
        const __nv_bfloat16* ks = pf_kv_smem + (it & 1) * TILE;
        const __nv_bfloat16* vs = pf_kv_smem + (2 + (it & 1)) * TILE;
        if (j0 > wlast) {   // every row of this warp is past these keys (masked)
            __syncthreads();
            continue;
        }
        // S = Q K^T: 16 rows x PF_KT2 keys
        float sacc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t qa[4];   // A: (rows 0-7 | 8-15) x (k 0-7 | 8-15) of this k-step
            ldsm_x4(smem_u32(q_s + (rr + ((mi & 1) << 3)) * RS + 16 * k + ((mi >> 1) << 3)), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
            for (int n2 = 0; n2 < NT / 2; ++n2) {   // two n-tiles (16 keys) per ldmatrix
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(ks + (16 * n2 + rr + ((mi >> 1) << 3)) * RS + 16 * k + ((mi & 1) << 3)), b0, b1, b2, b3);
                mma_bf16(sacc[2 * n2], qa, b0, b1);
                mma_bf16(sacc[2 * n2 + 1], qa, b2, b3);
            }
        }
        // scores of row gq (hi + lo rows), keys 8n + 2tq + e; online softmax over the tile
        float sc[NT][2];
        float mx = -INFINITY;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = j0 + 8 * n + 2 * tq + e;
                const float v = sacc[n][e] + sacc[n][2 + e];
                sc[n][e] = (live && j <= qpos) ? v : -INFINITY;
                mx = fmaxf(mx, sc[n][e]);
            }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : expf(m_run - mn);
        float ps = 0.f;
        // P as A fragments: per 16 keys (n-tiles 2kk, 2kk+1), rows 0-7 bf16(p), rows 8-15 remainders
        uint32_t pa[NT / 2][4];
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk) {
            float p[4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float s_ = sc[2 * kk + h][e];
                    const float pv = s_ == -INFINITY ? 0.f : expf(s_ - mn);
                    p[2 * h + e] = pv;
                    ps += pv;
                }
            const float h0 = bf16_round_f(p[0]), h1 = bf16_round_f(p[1]), h2 = bf16_round_f(p[2]), h3 = bf16_round_f(p[3]);
            pa[kk][0] = pack_bf16x2(h0, h1);
            pa[kk][1] = pack_bf16x2(p[0] - h0, p[1] - h1);
            pa[kk][2] = pack_bf16x2(h2, h3);
            pa[kk][3] = pack_bf16x2(p[2] - h2, p[3] - h3);
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l_run = l_run * alpha + ps;
        m_run = mn;
#pragma unroll
        for (int n = 0; n < DT; ++n) {
            o[n][0] *= alpha; o[n][1] *= alpha; o[n][2] *= alpha; o[n][3] *= alpha;
        }
        // O += P V: V tiles read transposed (k = keys, n = dims)
#pragma unroll
        for (int kk = 0; kk < NT / 2; ++kk)
#pragma unroll
            for (int d2 = 0; d2 < DT / 2; ++d2) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(smem_u32(vs + (16 * kk + rr + ((mi & 1) << 3)) * RS + 16 * d2 + ((mi >> 1) << 3)), v0, v1, v2,
                          v3);
                mma_bf16(o[2 * d2], pa[kk], v0, v1);
                mma_bf16(o[2 * d2 + 1], pa[kk], v2, v3);
            }
        __syncthreads();   // this buffer is refilled by the next iteration's copies
    }
    if (!live) return;
    // O of row gq = its bf16-part row + its remainder row
    const float inv = 1.0f / l_run;   // the row's own position is always visible: l_run > 0
#pragma unroll
    for (int n = 0; n < DT; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) put_hilo(hb, qd, tok, head * HD + 8 * n + 2 * tq + e, (o[n][e] + o[n][2 + e]) * inv);
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
    delete s;
}

static const void* pf_attn_fn(int hd, int G) {
    if (hd == 128) {
        if (G == 4) return (const void*)&k_pf_attn_mma<128, 4>;
        if (G == 2) return (const void*)&k_pf_attn_mma<128, 2>;
    } else if (hd == 64) {
        if (G == 4) return (const void*)&k_pf_attn_mma<64, 4>;
        if (G == 2) return (const void*)&k_pf_attn_mma<64, 2>;
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
        (e = cudaMalloc(&s->pages, sizeof(int) * (a.paged ? a.ppr : 1))) != cudaSuccess) {
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
    if ((e = cudaFuncSetAttribute(k_pf_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(pf_attn_fn(a.hd, a.Hq / a.Hkv), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  pf_attn_smem(a.hd))) != cudaSuccess) {
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
                void* args[] = {&s->q, const_cast<int*>(&a.Hq), &nt, &p0, const_cast<float*>(&scale), &kv, &s->hb};
                const int tpc = PF_QR / G;   // tokens per attention CTA
                if ((e = cudaLaunchKernel(attn, dim3((nt + tpc - 1) / tpc, a.Hkv), dim3(256), args,
                                          pf_attn_smem(a.hd), st)) != cudaSuccess)
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
