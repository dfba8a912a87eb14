// prefill.cu -- multi-token prefill of one sequence ("Models, Registry and the
// Driver", "The Model": a step shape is rows x new tokens, positions are
// absolute, so a prefill is a step continuing from a position).
//
// The prompt runs in blocks of PF_T = 128 tokens.  Per block and layer:
//   RMSNorm -> QKV projection (tensor cores, pf_gemm.cuh) -> RoPE, K/V written
//   into the sequence's store -> causal attention over every position up to
//   each token (flash-style online softmax) -> O projection + residual ->
//   RMSNorm -> gate/up projection -> SwiGLU -> down projection + residual.
// After the last block the final token's hidden state goes through the
// decoder's own head (final RMSNorm, LM head, greedy argmax).  Projections
// split K over CTAs; the kernel that consumes a projection adds its splits in
// split order, so results do not depend on scheduling.
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

constexpr int PF_NT = 1024;        // threads of the per-token kernels

// hi / lo bf16 rows of one activation value (row t of the block and row PF_T + t)
__device__ __forceinline__ void put_hilo(__nv_bfloat16* hb, int K, int t, int k, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    hb[(size_t)t * K + k] = hi;
    hb[(size_t)(PF_T + t) * K + k] = __float2bfloat16_rn(v - __bfloat162float(hi));
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

// x[t] = E[tok[t]] (fp32) for the block's tokens; rows past nt are zero
__global__ void k_pf_embed(const __nv_bfloat16* E, const int* tok, int nt, int d, float* x) {
    const int t = blockIdx.x;
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        x[(size_t)t * d + i] = t < nt ? __bfloat162float(E[(size_t)tok[t] * d + i]) : 0.f;
}

// x[t] += sum over splits of part[s][t] (when part is given); then, when gain
// is given, hb = hi/lo of x[t] / sqrt(mean(x[t]^2) + eps) * gain.  Rows past nt
// give zero hb rows.  One CTA per token row of the block.
__global__ void k_pf_resid_norm(float* x, const float* part, int splits, int d, const __nv_bfloat16* gain, float eps,
                                int nt, __nv_bfloat16* hb) {
    __shared__ float red[PF_NT / 32];
    const int t = blockIdx.x;
    float* xr = x + (size_t)t * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        float v = xr[i];
        if (part && t < nt) {
#pragma unroll 4
            for (int s = 0; s < splits; ++s) v += part[((size_t)s * PF_T + t) * d + i];
            xr[i] = v;
        }
        ss = fmaf(v, v, ss);
    }
    if (!gain) return;
    const float tot = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        put_hilo(hb, d, t, i, t < nt ? xr[i] * inv * __bfloat162float(gain[i]) : 0.f);
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
        const int pg = kv.pages[pos / kv.page], o = pos % kv.page;
        return (((size_t)pg * kv.Hkv + g) * kv.page + o) * kv.hd;
    }
    return (((size_t)kv.row * kv.Hkv + g) * kv.cap + pos) * kv.hd;
}
__global__ void k_pf_qkv(const float* part, int splits, int Hq, int nt, int pos0, const float2* rope, float* qout,
                         PfKv kv) {
    const int t = blockIdx.x;
    if (t >= nt) return;
    const int hd = kv.hd, h2 = hd / 2, qd = Hq * hd, kvd = kv.Hkv * hd, N = qd + 2 * kvd;
    const int pos = pos0 + t;
    const float2* rt = rope + (size_t)pos * h2;
    auto val = [&](int n) {
        float v = 0.f;
#pragma unroll 4
        for (int s = 0; s < splits; ++s) v += part[((size_t)s * PF_T + t) * N + n];
        return v;
    };
    for (int i = threadIdx.x; i < (Hq + kv.Hkv) * h2; i += blockDim.x) {   // q and k pairs
        const int hh = i / h2, e = i % h2;
        const bool is_q = hh < Hq;
        const int base = is_q ? hh * hd : qd + (hh - Hq) * hd;
        const float a = val(base + e), b = val(base + e + h2);
        const float2 cs = rt[e];
        const float r0 = a * cs.x - b * cs.y, r1 = a * cs.y + b * cs.x;
        if (is_q) {
            qout[(size_t)t * qd + hh * hd + e] = r0;
            qout[(size_t)t * qd + hh * hd + e + h2] = r1;
        } else {
            const size_t o = kv_off(kv, hh - Hq, pos);
            kv.K[o + e] = __float2bfloat16_rn(r0);
            kv.K[o + e + h2] = __float2bfloat16_rn(r1);
        }
    }
    for (int i = threadIdx.x; i < kvd; i += blockDim.x) {   // v
        const int g = i / hd, e = i % hd;
        kv.V[kv_off(kv, g, pos) + e] = __float2bfloat16_rn(val(qd + kvd + i));
    }
}

// Causal attention on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate), flash-style.  A CTA takes 64 query rows -- PF_QR / G tokens x
// the G query heads of kv head g, row r = token * G + head -- and sweeps the
// keys [0, last position of its tokens] in tiles of PF_KT2 keys.  Warp w owns
// query rows 8w..8w+7: the MMA's 16 A rows hold their bf16 parts (rows 0-7) and
// remainders (rows 8-15), so q keeps about 16 significant bits; S = Q K^T comes
// out as hi + lo row pairs, and P (online softmax, fp32) goes back into the
// next MMA's A fragments the same way, straight from the registers.  K and V
// tiles are staged in shared memory (rows padded by 16 bytes: conflict-free
// ldmatrix); V is read transposed.  The output goes to hb as the O projection's
// hi/lo activation rows.
constexpr int PF_QR = 64;          // query rows per CTA
constexpr int PF_KT2 = 64;         // keys per tile
template <int HD, int G>
__global__ void __launch_bounds__(256) k_pf_attn_mma(const float* q, int Hq, int nt, int pos0, float scale, PfKv kv,
                                                     __nv_bfloat16* hb) {
    constexpr int KS = HD / 16;            // k-steps of S = Q K^T
    constexpr int DT = HD / 8;             // n-tiles of O
    constexpr int NT = PF_KT2 / 8;         // n-tiles of S
    constexpr int RS = HD + 8;             // shared row stride (bf16)
    constexpr int TPC = PF_QR / G;         // tokens per CTA
    __shared__ __align__(16) __nv_bfloat16 ks[PF_KT2 * RS];
    __shared__ __align__(16) __nv_bfloat16 vs[PF_KT2 * RS];
    const int g = blockIdx.y, t0 = blockIdx.x * TPC, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
    const int qd = Hq * HD;
    // this lane's query row (warp row gq) and its position
    const int r = warp * 8 + gq, tok = t0 + r / G, head = g * G + r % G;
    const bool live = tok < nt;
    const int qpos = pos0 + tok;
    // Q fragments: rows 0-7 bf16(q * scale), rows 8-15 the remainders
    uint32_t qa[KS][4];
    {
        const float* qr = q + (size_t)tok * qd + head * HD;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            float v[4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) v[2 * h + e] = live ? qr[16 * k + 8 * h + 2 * tq + e] * scale : 0.f;
            const float h0 = bf16_round_f(v[0]), h1 = bf16_round_f(v[1]), h2 = bf16_round_f(v[2]), h3 = bf16_round_f(v[3]);
            qa[k][0] = pack_bf16x2(h0, h1);
            qa[k][1] = pack_bf16x2(v[0] - h0, v[1] - h1);
            qa[k][2] = pack_bf16x2(h2, h3);
            qa[k][3] = pack_bf16x2(v[2] - h2, v[3] - h3);
        }
    }
    float o[DT][4];
#pragma unroll
    for (int n = 0; n < DT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const int last = pos0 + min(t0 + TPC, nt) - 1;               // the last key any row of the CTA sees
    const int wlast = pos0 + min(t0 + (warp * 8 + 7) / G + 1, nt) - 1;   // ... any row of this warp
    for (int j0 = 0; j0 <= last; j0 += PF_KT2) {
        __syncthreads();
        for (int i = tid; i < PF_KT2 * (HD / 8); i += 256) {     // 16-byte vectors of K and V
            const int kk = i / (HD / 8), c = i % (HD / 8), j = j0 + kk;
            uint4 kv4 = make_uint4(0u, 0u, 0u, 0u), vv4 = make_uint4(0u, 0u, 0u, 0u);
            if (j <= last) {
                const size_t off = kv_off(kv, g, j) + (size_t)c * 8;
                kv4 = *reinterpret_cast<const uint4*>(kv.K + off);
                vv4 = *reinterpret_cast<const uint4*>(kv.V + off);
            }
            *reinterpret_cast<uint4*>(ks + kk * RS + c * 8) = kv4;
            *reinterpret_cast<uint4*>(vs + kk * RS + c * 8) = vv4;
        }
        __syncthreads();
        if (j0 > wlast) continue;   // every row of this warp is past these keys (masked)
        // S = Q K^T: 16 rows x PF_KT2 keys
        float sacc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int k = 0; k < KS; ++k)
#pragma unroll
            for (int n2 = 0; n2 < NT / 2; ++n2) {   // two n-tiles (16 keys) per ldmatrix
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(ks + (16 * n2 + rr + ((mi >> 1) << 3)) * RS + 16 * k + ((mi & 1) << 3)), b0, b1, b2, b3);
                mma_bf16(sacc[2 * n2], qa[k], b0, b1);
                mma_bf16(sacc[2 * n2 + 1], qa[k], b2, b3);
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
    }
    if (!live) return;
    // O of row gq = its bf16-part row + its remainder row
    const float inv = 1.0f / l_run;   // the row's own position is always visible: l_run > 0
#pragma unroll
    for (int n = 0; n < DT; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) put_hilo(hb, qd, tok, head * HD + 8 * n + 2 * tq + e, (o[n][e] + o[n][2 + e]) * inv);
}

// SwiGLU of the gate/up splits: a = silu(gate) * up, as the down projection's hi/lo rows
__global__ void k_pf_swiglu(const float* part, int splits, int F, int nt, __nv_bfloat16* hb) {
    const int t = blockIdx.x;
    for (int f = threadIdx.x; f < F; f += blockDim.x) {
        float a = 0.f;
        if (t < nt) {
            float gs = 0.f, us = 0.f;
#pragma unroll 4
            for (int s = 0; s < splits; ++s) {
                const float* pr = part + ((size_t)s * PF_T + t) * 2 * F;
                gs += pr[f];
                us += pr[F + f];
            }
            a = gs / (1.0f + expf(-gs)) * us;
        }
        put_hilo(hb, F, t, f, a);
    }
}

// rows of zeros for the hi/lo activation rows past the block's tokens (the
// attention kernel writes only live rows)
__global__ void k_pf_zero_rows(__nv_bfloat16* hb, int K, int nt) {
    const int t = nt + blockIdx.x;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        hb[(size_t)t * K + k] = __float2bfloat16_rn(0.f);
        hb[(size_t)(PF_T + t) * K + k] = __float2bfloat16_rn(0.f);
    }
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

// the fewest K splits (a divisor of the K steps, at most 16) that give at least
// one CTA per SM
int pf_splits(int tiles, int ksteps, int num_sms) {
    for (int s = 1; s <= 16; ++s)
        if (ksteps % s == 0 && tiles * s >= num_sms) return s;
    for (int s = 16; s >= 1; --s)
        if (ksteps % s == 0) return s;
    return 1;
}

}  // namespace

// one projection of the block: up to three stacked weight segments
struct PfProj {
    PfGemmParams p{};
    int tiles = 0, splits = 1;
};

struct PrefillState {
    PrefillArgs a;
    float *x = nullptr, *part = nullptr, *q = nullptr;
    __nv_bfloat16* hb = nullptr;
    int* tok = nullptr;
    int* pages = nullptr;
    std::vector<PfProj> proj;   // per layer: qkv, o, gate/up, down
    size_t part_floats = 0;
};

size_t prefill_part_floats(const PrefillArgs& a, int num_sms) {
    const int qd = a.Hq * a.hd, kvd = a.Hkv * a.hd;
    size_t most = 0;
    auto need = [&](int N, int K) {
        const int tiles = (N + 127) / 128;
        const int s = pf_splits(tiles, K / PF_BK, num_sms);
        const size_t v = (size_t)s * PF_T * N;
        if (v > most) most = v;
    };
    need(qd + 2 * kvd, a.d);
    need(a.d, qd);
    need(2 * a.F, a.d);
    need(a.d, a.F);
    return most;
}

bool prefill_supported(const PrefillArgs& a) {
    const int qd = a.Hq * a.hd;
    if (a.hd != 64 && a.hd != 128) return false;
    const int G = a.Hq / a.Hkv;
    if (G != 2 && G != 4) return false;
    if (a.d % PF_BK || qd % PF_BK || a.F % PF_BK) return false;
    return true;
}

void prefill_free(PrefillState* s) {
    if (!s) return;
    cudaFree(s->x);
    cudaFree(s->part);
    cudaFree(s->q);
    cudaFree(s->hb);
    cudaFree(s->tok);
    cudaFree(s->pages);
    delete s;
}

cudaError_t prefill_create(const PrefillArgs& a, int num_sms, PrefillState** out) {
    *out = nullptr;
    PrefillState* s = new PrefillState();
    s->a = a;
    const int qd = a.Hq * a.hd, kvd = a.Hkv * a.hd;
    const int kmax = a.d > qd ? (a.d > a.F ? a.d : a.F) : (qd > a.F ? qd : a.F);
    s->part_floats = prefill_part_floats(a, num_sms);
    cudaError_t e;
    if ((e = cudaMalloc(&s->x, sizeof(float) * PF_T * a.d)) != cudaSuccess ||
        (e = cudaMalloc(&s->part, sizeof(float) * s->part_floats)) != cudaSuccess ||
        (e = cudaMalloc(&s->q, sizeof(float) * PF_T * qd)) != cudaSuccess ||
        (e = cudaMalloc(&s->hb, sizeof(__nv_bfloat16) * PF_BN * kmax)) != cudaSuccess ||
        (e = cudaMalloc(&s->tok, sizeof(int) * a.cap)) != cudaSuccess ||
        (e = cudaMalloc(&s->pages, sizeof(int) * (a.paged ? a.ppr : 1))) != cudaSuccess) {
        cudaGetLastError();
        prefill_free(s);
        return e;
    }
    // tensor maps: every layer's weights, and the hi/lo activation rows for K = d, qd, F
    CUtensorMap hd_map, hq_map, hf_map;
    if (!pf_map(&hd_map, s->hb, PF_BN, a.d, PF_BN) || !pf_map(&hq_map, s->hb, PF_BN, qd, PF_BN) ||
        !pf_map(&hf_map, s->hb, PF_BN, a.F, PF_BN)) {
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
        pr.tiles = tiles;
        pr.splits = pf_splits(tiles, K / PF_BK, num_sms);
        p.ksteps = K / PF_BK / pr.splits;
        p.part = s->part;
        p.err = a.err;
        return (size_t)pr.splits * PF_T * rows <= s->part_floats;
    };
    s->proj.resize((size_t)a.L * 4);
    for (int l = 0; l < a.L; ++l) {
        const void* const* w = a.lw + (size_t)l * 9;   // attn_norm, q, k, v, o, ffn_norm, gate, up, down
        if (!proj(w[1], qd, w[2], kvd, w[3], kvd, a.d, hd_map, s->proj[4 * l + 0]) ||
            !proj(w[4], a.d, nullptr, 0, nullptr, 0, qd, hq_map, s->proj[4 * l + 1]) ||
            !proj(w[6], a.F, w[7], a.F, nullptr, 0, a.d, hd_map, s->proj[4 * l + 2]) ||
            !proj(w[8], a.d, nullptr, 0, nullptr, 0, a.F, hf_map, s->proj[4 * l + 3])) {
            prefill_free(s);
            return cudaErrorInvalidValue;
        }
    }
    if ((e = cudaFuncSetAttribute(k_pf_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM)) != cudaSuccess) {
        prefill_free(s);
        return e;
    }
    *out = s;
    return cudaSuccess;
}

static cudaError_t pf_gemm_launch(const PfProj& pr, cudaStream_t st) {
    k_pf_gemm<<<dim3(pr.tiles, pr.splits), PF_THREADS, PF_SMEM, st>>>(pr.p);
    return cudaGetLastError();
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
    for (int c0 = 0; c0 < n; c0 += PF_T) {
        const int nt = n - c0 < PF_T ? n - c0 : PF_T;
        const int p0 = pos0 + c0;
        k_pf_embed<<<PF_T, PF_NT, 0, st>>>(static_cast<const __nv_bfloat16*>(a.embed), s->tok + c0, nt, a.d, s->x);
        k_pf_resid_norm<<<PF_T, PF_NT, 0, st>>>(s->x, nullptr, 0, a.d,
                                                static_cast<const __nv_bfloat16*>(a.lw[0]), a.eps, nt, s->hb);
        for (int l = 0; l < a.L; ++l) {
            const void* const* w = a.lw + (size_t)l * 9;
            PfKv kv{static_cast<__nv_bfloat16*>(a.K[l]), static_cast<__nv_bfloat16*>(a.V[l]),
                    a.paged ? s->pages : nullptr, row, a.Hkv, a.hd, a.cap, a.page};
            const PfProj& pq = s->proj[4 * l + 0];
            if ((e = pf_gemm_launch(pq, st)) != cudaSuccess) return e;
            k_pf_qkv<<<PF_T, PF_NT, 0, st>>>(s->part, pq.splits, a.Hq, nt, p0, a.rope, s->q, kv);
            if (nt < PF_T) k_pf_zero_rows<<<PF_T - nt, PF_NT, 0, st>>>(s->hb, qd, nt);
            {
                void* args[] = {&s->q, const_cast<int*>(&a.Hq), const_cast<int*>(&nt), const_cast<int*>(&p0),
                                const_cast<float*>(&scale), &kv, &s->hb};
                const int tpc = PF_QR / G;   // tokens per attention CTA
                if ((e = cudaLaunchKernel(attn, dim3((nt + tpc - 1) / tpc, a.Hkv), dim3(256), args, 0, st)) !=
                    cudaSuccess)
                    return e;
            }
            const PfProj& po = s->proj[4 * l + 1];
            if ((e = pf_gemm_launch(po, st)) != cudaSuccess) return e;
            k_pf_resid_norm<<<PF_T, PF_NT, 0, st>>>(s->x, s->part, po.splits, a.d,
                                                    static_cast<const __nv_bfloat16*>(w[5]), a.eps, nt, s->hb);
            const PfProj& pg = s->proj[4 * l + 2];
            if ((e = pf_gemm_launch(pg, st)) != cudaSuccess) return e;
            k_pf_swiglu<<<PF_T, PF_NT, 0, st>>>(s->part, pg.splits, a.F, nt, s->hb);
            const PfProj& pd = s->proj[4 * l + 3];
            if ((e = pf_gemm_launch(pd, st)) != cudaSuccess) return e;
            const __nv_bfloat16* next_gain =
                l + 1 < a.L ? static_cast<const __nv_bfloat16*>(a.lw[(size_t)(l + 1) * 9 + 0]) : nullptr;
            k_pf_resid_norm<<<PF_T, PF_NT, 0, st>>>(s->x, s->part, pd.splits, a.d, next_gain, a.eps, nt, s->hb);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        if (c0 + PF_T >= n &&
            (e = cudaMemcpyAsync(x_last, s->x + (size_t)(nt - 1) * a.d, sizeof(float) * a.d, cudaMemcpyDeviceToDevice,
                                 st)) != cudaSuccess)
            return e;
    }
    return cudaGetLastError();
}

}  // namespace gd
