// attn.cu -- masked split-KV decode attention over the fixed capacity, with
// the step's RoPE and K/V write fused in (sm_103a, CUDA cores, fp32 math).
//
// What it computes ("Execution", section "A constant-shape decode graph"):
// each step writes the new K/V at pos (DynamicUpdateSlice, or a ScatterUpdate
// through Slot::WriteMap for paged KV); attention always sweeps [0, cap); a
// mask computed from Slot::Pos against an iota hides every position after
// pos.  Masked positions are read (the sweep is constant-shape) but excluded
// by select, never by multiplying with zero, so garbage there (NaN, Inf)
// cannot reach the result.
//
// Work decomposition: one CTA per (KV split, kv head, row).  The CTA owns a
// contiguous range of positions; it loads each K/V vector once and uses it for
// all G = Hq/Hkv query heads of the group (GQA sharing).  Pass 1 computes the
// masked scores of the range into shared memory, pass 2 accumulates
// p_j * v_j; the split's (max, sum, o) partial goes to global memory and the
// last CTA of the (row, kv head) -- found with an atomic completion counter --
// merges the splits in fixed split order (log-sum-exp), so results do not
// depend on CTA scheduling.  The CTA whose range holds pos rotates and rounds
// the new k, v, writes them to the store, and uses the rounded values for
// position pos directly.  Paged addressing ("Execution", section "Slot
// buffers": SlotMap and WriteMap are slots): logical position j of row r is
// slot SlotMap[r][j / page] * page + j % page.
#include <math.h>
#include "common.cuh"
#include "internal.h"

namespace gd {

constexpr int ATTN_THREADS = 256;
constexpr int ATTN_WARPS = ATTN_THREADS / 32;
constexpr int ATTN_U = 4;
constexpr int ATTN_MAX_SPLIT = 1024;

size_t attn_part_floats(int R, int Hq, int hd, int nsplit) {
    return (size_t)R * Hq * nsplit * (hd + 2);
}

template <int HD, int G>
struct AttnSmem {
    // float offsets into dynamic shared memory
    static constexpr int q = 0;                          // [G][HD]
    static constexpr int kn = q + G * HD;                // [HD]
    static constexpr int vn = kn + HD;                   // [HD]
    static constexpr int red = vn + HD;                  // [WARPS][G][HD]
    static constexpr int sc = red + ATTN_WARPS * G * HD; // [G][split_len] scores / weights
};

template <typename KT, int HD, int G, bool PAGED>
__global__ void __launch_bounds__(ATTN_THREADS) k_attn(const AttnParams p) {
    constexpr int DPL = Elem<KT>::VEC;   // elements per lane per 16-byte vector
    constexpr int LPP = HD / DPL;        // lanes per position
    constexpr int PPW = 32 / LPP;        // positions per warp per load
    constexpr int PPI = ATTN_WARPS * PPW;
    static_assert(HD % DPL == 0 && LPP >= 1 && LPP <= 32 && (32 % LPP) == 0, "head_dim");
    using SM = AttnSmem<HD, G>;

    extern __shared__ float4 smem_f4[];
    float* smem = reinterpret_cast<float*>(smem_f4);
    float* q_s = smem + SM::q;
    float* kn_s = smem + SM::kn;
    float* vn_s = smem + SM::vn;
    float* red_s = smem + SM::red;
    float* sc_s = smem + SM::sc;
    const int L = p.split_len;
    float* cm_s = sc_s + G * L;          // [G][nsplit] split maxima (combine)
    float* cw_s = cm_s + G * p.nsplit;   // [G][nsplit] split weights (combine)
    int* page_s = reinterpret_cast<int*>(cw_s + G * p.nsplit);
    __shared__ float wred[ATTN_WARPS][G];
    __shared__ float m_s[G], l_s[G];
    __shared__ int last_s;

    const int s = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j0 = s * L;
    const int j1 = min(j0 + L, p.cap);
    const int P = p.page_size;

    pdl_wait();

    int pos = p.pos[r];
    pos = min(max(pos, 0), p.cap - 1);   // out-of-range pos was flagged by the embedding kernel

    // ---- q of the G heads of this group: RoPE at pos, scaled by 1/sqrt(hd) ----
    const float* qrow = p.qkv + (size_t)r * p.qkv_stride;
    const float2* rt = p.rope + (size_t)pos * (HD / 2);
    for (int i = tid; i < G * (HD / 2); i += ATTN_THREADS) {
        const int h = i / (HD / 2), d = i % (HD / 2);
        const float* qh = qrow + (size_t)(g * G + h) * HD;
        const float a = qh[d], b = qh[d + HD / 2];
        const float2 cs = rt[d];
        q_s[h * HD + d] = (a * cs.x - b * cs.y) * p.scale;
        q_s[h * HD + d + HD / 2] = (a * cs.y + b * cs.x) * p.scale;
    }

    // ---- paged: page ids of this split's positions ----
    if (PAGED) {
        const int pg0 = j0 / P, npg = (j1 - j0 + P - 1) / P;
        for (int i = tid; i < npg; i += ATTN_THREADS) {
            int pg = p.slot_map[(size_t)r * p.pages_per_row + pg0 + i];
            if (pg < 0 || pg >= p.num_pages) {
                atomicOr(p.err, FAULT_SLOT_MAP);
                pg = 0;
            }
            page_s[i] = pg;
        }
    }

    // ---- the new k, v: RoPE, storage rounding, write at pos (owner CTA only) ----
    const bool owner = pos >= j0 && pos < j1;
    KT* Kc = reinterpret_cast<KT*>(p.Kc);
    KT* Vc = reinterpret_cast<KT*>(p.Vc);
    if (owner) {
        const float* kh = qrow + (size_t)p.Hq * HD + (size_t)g * HD;
        const float* vh = kh + (size_t)p.Hkv * HD;
        size_t off;
        bool ok = true;
        if (PAGED) {
            const int slot = p.write_map[r];
            if (slot < 0 || slot >= p.num_pages * P) {
                ok = false;
                if (tid == 0) atomicOr(p.err, FAULT_WRITE_MAP);
            }
            const int pg = ok ? slot / P : 0, o = ok ? slot % P : 0;
            off = (((size_t)pg * p.Hkv + g) * P + o) * HD;
        } else {
            off = (((size_t)r * p.Hkv + g) * p.cap + pos) * HD;
        }
        for (int d = tid; d < HD / 2; d += ATTN_THREADS) {
            const float a = kh[d], b = kh[d + HD / 2];
            const float2 cs = rt[d];
            const float k0 = a * cs.x - b * cs.y, k1 = a * cs.y + b * cs.x;
            if (ok) {
                kn_s[d] = Elem<KT>::round_store(k0, Kc + off + d);
                kn_s[d + HD / 2] = Elem<KT>::round_store(k1, Kc + off + d + HD / 2);
            } else {
                kn_s[d] = Elem<KT>::round(k0);
                kn_s[d + HD / 2] = Elem<KT>::round(k1);
            }
        }
        for (int d = tid; d < HD; d += ATTN_THREADS)
            vn_s[d] = ok ? Elem<KT>::round_store(vh[d], Vc + off + d) : Elem<KT>::round(vh[d]);
    }
    __syncthreads();
    pdl_trigger();

    // address of the K (or V) vector slice [sub*DPL, +DPL) of logical position j
    const int sub = lane % LPP, pw = lane / LPP;
    auto vec_off = [&](int j) -> size_t {
        if (PAGED) {
            const int pg = page_s[(j - (j0 / P) * P) / P];
            return (((size_t)pg * p.Hkv + g) * P + (j % P)) * HD + sub * DPL;
        }
        return (((size_t)r * p.Hkv + g) * p.cap + j) * HD + sub * DPL;
    };

    // ---- pass 1: masked scores s[h][j] for j in [j0, j1) ----
    float qr[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) qr[h][e] = q_s[h * HD + sub * DPL + e];

    // the loop base is warp-uniform so every lane reaches the shuffles
    for (int jw = j0 + warp * PPW; jw < j1; jw += PPI * ATTN_U) {
        const int jb = jw + pw;
        uint4 kv[ATTN_U];
#pragma unroll
        for (int u = 0; u < ATTN_U; ++u) {
            const int j = jb + u * PPI;
            kv[u] = j < j1 ? ld_stream16(Kc + vec_off(j)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < ATTN_U; ++u) {
            const int j = jb + u * PPI;
            float kf[DPL];
            Elem<KT>::unpack(kv[u], kf);
            if (j == pos) {
#pragma unroll
                for (int e = 0; e < DPL; ++e) kf[e] = kn_s[sub * DPL + e];
            }
            float part[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) a = fmaf(qr[h][e], kf[e], a);
                part[h] = a;
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int o = LPP / 2; o > 0; o >>= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
            if (sub == 0 && j < j1) {
#pragma unroll
                for (int h = 0; h < G; ++h) sc_s[h * L + (j - j0)] = (j <= pos) ? part[h] : -INFINITY;
            }
        }
    }
    __syncthreads();

    // ---- split max and exp-sum per head ----
    const int len = j1 - j0;
    {
        float mx[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mx[h] = -INFINITY;
            for (int i = tid; i < len; i += ATTN_THREADS) mx[h] = fmaxf(mx[h], sc_s[h * L + i]);
            mx[h] = warp_max(mx[h]);
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) wred[warp][h] = mx[h];
        }
        __syncthreads();
        if (tid < G) {
            float m = -INFINITY;
#pragma unroll
            for (int w = 0; w < ATTN_WARPS; ++w) m = fmaxf(m, wred[w][tid]);
            m_s[tid] = m;
        }
        __syncthreads();
        float sm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float m = m_s[h];
            sm[h] = 0.f;
            for (int i = tid; i < len; i += ATTN_THREADS) {
                const float sv = sc_s[h * L + i];
                const float e = (m == -INFINITY) ? 0.f : expf(sv - m);
                sc_s[h * L + i] = e;
                sm[h] += e;
            }
            sm[h] = warp_sum(sm[h]);
        }
        __syncthreads();
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) wred[warp][h] = sm[h];
        }
        __syncthreads();
        if (tid < G) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < ATTN_WARPS; ++w) t += wred[w][tid];
            l_s[tid] = t;
        }
    }

    // ---- pass 2: o[h] = sum_j e[h][j] * v_j over unmasked j ----
    float o[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
    for (int jw = j0 + warp * PPW; jw < j1; jw += PPI * ATTN_U) {
        const int jb = jw + pw;
        uint4 vv[ATTN_U];
#pragma unroll
        for (int u = 0; u < ATTN_U; ++u) {
            const int j = jb + u * PPI;
            vv[u] = j < j1 ? ld_stream16(Vc + vec_off(j)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < ATTN_U; ++u) {
            const int j = jb + u * PPI;
            float vf[DPL];
            Elem<KT>::unpack(vv[u], vf);
            if (j == pos) {
#pragma unroll
                for (int e = 0; e < DPL; ++e) vf[e] = vn_s[sub * DPL + e];
            }
            const bool valid = j <= pos && j < j1;
            const int jj = valid ? j - j0 : 0;   // keeps the shared-memory index in range
#pragma unroll
            for (int e = 0; e < DPL; ++e) vf[e] = valid ? vf[e] : 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pj = valid ? sc_s[h * L + jj] : 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pj, vf[e], o[h][e]);
            }
        }
    }
    // reduce over the positions of a warp, then over warps
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
#pragma unroll
            for (int off = 16; off >= LPP; off >>= 1) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], off);
    if (pw == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL; ++e) red_s[(warp * G + h) * HD + sub * DPL + e] = o[h][e];
    }
    __syncthreads();

    // ---- write this split's partial (m, l, o) ----
    for (int i = tid; i < G * HD; i += ATTN_THREADS) {
        const int h = i / HD, d = i % HD;
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < ATTN_WARPS; ++w) t += red_s[(w * G + h) * HD + d];
        float* pp = p.part + (((size_t)r * p.Hq + g * G + h) * p.nsplit + s) * (HD + 2);
        pp[2 + d] = t;
        if (d == 0) {
            pp[0] = m_s[h];
            pp[1] = l_s[h];
        }
    }

    // ---- the last split of this (row, kv head) merges all splits ----
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(p.counters + r * p.Hkv + g, 1u);
        last_s = (prev == (unsigned)p.nsplit - 1u);
    }
    __syncthreads();
    if (!last_s) return;
    __threadfence();
    if (tid == 0) p.counters[r * p.Hkv + g] = 0u;   // ready for the next step

    const int NS = p.nsplit;
    for (int i = tid; i < G * NS; i += ATTN_THREADS) {
        const int h = i / NS, ss = i % NS;
        const float* pp = p.part + (((size_t)r * p.Hq + g * G + h) * NS + ss) * (HD + 2);
        cm_s[h * NS + ss] = __ldcg(pp);
        cw_s[h * NS + ss] = __ldcg(pp + 1);
    }
    __syncthreads();
    if (warp < G) {
        const int h = warp;
        float M = -INFINITY;
        for (int ss = lane; ss < NS; ss += 32) M = fmaxf(M, cm_s[h * NS + ss]);
        M = warp_max(M);
        float Lsum = 0.f;
        for (int ss = lane; ss < NS; ss += 32) {
            const float m = cm_s[h * NS + ss];
            Lsum += (m == -INFINITY) ? 0.f : expf(m - M) * cw_s[h * NS + ss];
        }
        Lsum = warp_sum(Lsum);
        __syncwarp();
        for (int ss = lane; ss < NS; ss += 32) {
            const float m = cm_s[h * NS + ss];
            cw_s[h * NS + ss] = (m == -INFINITY) ? 0.f : expf(m - M) / Lsum;
        }
    }
    __syncthreads();
    for (int i = tid; i < G * HD; i += ATTN_THREADS) {
        const int h = i / HD, d = i % HD;
        float acc = 0.f;
        for (int ss = 0; ss < NS; ++ss) {
            const float w = cw_s[h * NS + ss];
            const float* pp = p.part + (((size_t)r * p.Hq + g * G + h) * NS + ss) * (HD + 2);
            acc = fmaf(w, __ldcg(pp + 2 + d), acc);
        }
        p.out[(size_t)r * p.Hq * HD + (size_t)(g * G + h) * HD + d] = acc;
    }
}

// ---------------- host side ----------------

template <typename KT, int HD, int G, bool PAGED>
static const void* kptr() {
    return reinterpret_cast<const void*>(&k_attn<KT, HD, G, PAGED>);
}

template <typename KT, int HD, int G>
static const void* pick_paged(bool paged) {
    return paged ? kptr<KT, HD, G, true>() : kptr<KT, HD, G, false>();
}

template <typename KT, int HD>
static const void* pick_group(int G, bool paged) {
    switch (G) {
        case 1: return pick_paged<KT, HD, 1>(paged);
        case 2: return pick_paged<KT, HD, 2>(paged);
        case 4: return pick_paged<KT, HD, 4>(paged);
        case 8: return pick_paged<KT, HD, 8>(paged);
    }
    return nullptr;
}

template <typename KT>
static const void* pick_hd(int hd, int G, bool paged) {
    switch (hd) {
        case 16: return pick_group<KT, 16>(G, paged);
        case 32: return pick_group<KT, 32>(G, paged);
        case 64: return pick_group<KT, 64>(G, paged);
        case 128: return pick_group<KT, 128>(G, paged);
    }
    return nullptr;
}

static const void* pick(int kvtype, int hd, int G, bool paged) {
    return kvtype == W_BF16 ? pick_hd<__nv_bfloat16>(hd, G, paged) : pick_hd<float>(hd, G, paged);
}

// dynamic shared memory: the float regions of AttnSmem, the two combine
// arrays, and (paged) the page ids of one split
static size_t smem_bytes(int hd, int G, int L, int ns, bool paged, int page) {
    size_t f = (size_t)G * hd + 2 * (size_t)hd + (size_t)ATTN_WARPS * G * hd + (size_t)G * L + 2 * (size_t)G * ns;
    size_t b = f * sizeof(float);
    if (paged) b += (size_t)(L + page - 1) / page * sizeof(int);
    return b;
}

cudaError_t attn_plan(AttnPlan* plan, int num_sms) {
    AttnParams& p = plan->p;
    if (p.Hkv <= 0 || p.Hq % p.Hkv) return cudaErrorInvalidValue;
    plan->group = p.Hq / p.Hkv;
    const void* fn = pick(plan->kvtype, p.hd, plan->group, plan->paged);
    if (!fn) return cudaErrorInvalidValue;
    // aim at ~4 CTAs per SM over all (row, kv head) units; splits are whole
    // multiples of 64 positions (and of the page size), at most ATTN_MAX_SPLIT
    const int units = p.R * p.Hkv;
    const int want = (4 * num_sms + units - 1) / units;
    int L = (p.cap + want - 1) / want;
    int q = 64;
    if (plan->paged && p.page_size > q) q = p.page_size;
    if (plan->paged && (p.page_size < 1 || q % p.page_size)) return cudaErrorInvalidValue;
    L = (L + q - 1) / q * q;
    if (L > ATTN_MAX_SPLIT) L = ATTN_MAX_SPLIT;
    if (L < q) L = q;
    if (plan->paged && (L % p.page_size)) return cudaErrorInvalidValue;
    p.split_len = L;
    p.nsplit = (p.cap + L - 1) / L;
    plan->block = ATTN_THREADS;
    plan->grid = dim3(p.nsplit, p.Hkv, p.R);
    plan->smem = smem_bytes(p.hd, plan->group, L, p.nsplit, plan->paged, plan->paged ? p.page_size : 1);
    if (plan->smem > 200 * 1024) return cudaErrorInvalidValue;
    return raise_smem_cap(fn);
}

cudaError_t attn_launch(const AttnPlan& plan, cudaStream_t s, bool pdl) {
    const void* fn = pick(plan.kvtype, plan.p.hd, plan.group, plan.paged);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = plan.grid;
    cfg.blockDim = dim3(plan.block);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {const_cast<AttnParams*>(&plan.p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gd
