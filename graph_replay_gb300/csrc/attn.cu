// attn.cu -- masked split-KV decode attention over the fixed capacity, with
// the step's RoPE and K/V write fused in (sm_103a, fp32 math).
//
// What it computes ("Execution", section "A constant-shape decode graph"):
// each step writes the new K/V at pos (DynamicUpdateSlice, or a ScatterUpdate
// through Slot::WriteMap for paged KV); attention always sweeps [0, cap); a
// mask computed from Slot::Pos against an iota hides every position after
// pos.  Masked positions are read (the sweep is constant-shape) but excluded
// by select, never by multiplying with zero, so garbage there (NaN, Inf)
// cannot reach the result.
//
// Work decomposition: one CTA per (KV split, kv head, row); the split count
// is chosen so the CTAs cover the SMs evenly.  A producer warp streams the
// split's K and V through a shared-memory ring with bulk asynchronous copies
// (one copy per contiguous run: a whole stage for contiguous KV, one per page
// for paged KV); it starts before the programmatic-launch wait because the
// stored K/V and the slot buffers do not depend on the previous kernel.  Eight
// consumer warps each take a fixed slice of every stage's positions and keep
// a warp-local online softmax (running max, sum and output) for the G query
// heads that share the kv head (GQA: each K/V vector is loaded once for all G
// heads).  At the end the warps' states are merged in fixed order, the split's
// (max, sum, o) partial goes to global memory, and the last CTA of the (row,
// kv head) -- found with an atomic completion counter -- merges the splits in
// split order (log-sum-exp), so results do not depend on scheduling.
// The CTA whose range holds pos rotates and rounds the new k, v, writes them to
// the store, and uses the rounded values for position pos directly.  Paged
// addressing ("Execution", section "Slot buffers": SlotMap and WriteMap are
// slots): logical position j of row r is slot SlotMap[r][j/page]*page + j%page.
// Every mbarrier wait is bounded (FAULT_WAIT on give-up).
#include <math.h>
#include "common.cuh"
#include "internal.h"

namespace gd {

constexpr int AT_CW = 8;                 // consumer warps
constexpr int AT_CT = AT_CW * 32;
constexpr int AT_THREADS = AT_CT + 32;   // + producer warp
constexpr int AT_STAGE = 32768;          // bytes per stage (K and V tiles)
constexpr int AT_MAX_S = 4;

// partial record of one (row, head, split): m, l, pad, pad, o[hd] -- padded so
// every record starts on a 16-byte boundary
size_t attn_part_floats(int R, int Hq, int hd, int nsplit) {
    return (size_t)R * Hq * nsplit * (hd + 4);
}

template <typename KT, int HD>
struct AttnShape {
    static constexpr int ES = (int)sizeof(KT);
    static constexpr int DPL = Elem<KT>::VEC;            // elements per lane per 16-byte vector
    static constexpr int LPP = HD / DPL;                 // lanes per position
    static constexpr int PPI = 32 / LPP;                 // positions per warp per iteration
    static constexpr int PPS = AT_STAGE / (2 * HD * ES); // positions per stage
    static constexpr int ITER = PPS / (AT_CW * PPI);     // iterations per warp per stage
    static_assert(HD % DPL == 0 && LPP >= 1 && LPP <= 32 && 32 % LPP == 0, "head_dim");
    static_assert(PPS % (AT_CW * PPI) == 0 && ITER >= 1, "stage shape");
};

template <typename KT, int HD, int G, bool PAGED>
__global__ void __launch_bounds__(AT_THREADS) k_attn(const AttnParams p) {
    using SH = AttnShape<KT, HD>;
    constexpr int ES = SH::ES, DPL = SH::DPL, LPP = SH::LPP, PPI = SH::PPI, PPS = SH::PPS, ITER = SH::ITER;
    constexpr int TILE = PPS * HD * ES;   // bytes of the K (or V) half of a stage

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem;                                                  // [S][K tile | V tile]
    float* q_s = reinterpret_cast<float*>(smem + (size_t)p.stages * AT_STAGE);   // [G][HD]
    float* kn_s = q_s + G * HD;                                                  // [HD]
    float* vn_s = kn_s + HD;                                                     // [HD]
    float* cm_s = vn_s + HD;                                                     // [G][nsplit]
    float* cw_s = cm_s + G * p.nsplit;                                           // [G][nsplit]
    __shared__ __align__(8) uint64_t full_bar[AT_MAX_S];
    __shared__ __align__(8) uint64_t empty_bar[AT_MAX_S];
    __shared__ float wm_s[AT_CW][G], wl_s[AT_CW][G];
    __shared__ int abort_s, last_s;
    volatile int* abort_v = &abort_s;

    const int s = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = p.split_len;
    const int j0 = s * L;
    const int j1 = min(j0 + L, p.cap);
    const int nst = (j1 - j0 + PPS - 1) / PPS;
    const int S = p.stages;
    const int P = p.page_size;
    KT* Kc = reinterpret_cast<KT*>(p.Kc);
    KT* Vc = reinterpret_cast<KT*>(p.Vc);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], AT_CW);
        }
        abort_s = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == AT_CW) {
        // ---------------- producer: K and V tiles of this split ----------------
        if (lane == 1) trace_mark(trace_if_on(p.trace), p.trace_id, 0);
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < nst; ++t) {
                const int slot = t % S;
                if (t >= S && !*abort_v && !mbar_wait(&empty_bar[slot], ((t / S) - 1) & 1)) {
                    *abort_v = 1;
                    atomicOr(p.err, FAULT_WAIT);
                }
                if (*abort_v) break;
                const int p0 = j0 + t * PPS, p1 = min(p0 + PPS, j1);
                mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(2 * (p1 - p0) * HD * ES));
                unsigned char* kd = ring + (size_t)slot * AT_STAGE;
                unsigned char* vd = kd + TILE;
                if (PAGED) {
                    int q = p0;
                    while (q < p1) {
                        int pg = p.slot_map[(size_t)r * p.pages_per_row + q / P];
                        if (pg < 0 || pg >= p.num_pages) {
                            atomicOr(p.err, FAULT_SLOT_MAP);
                            pg = 0;
                        }
                        const int off = q % P, cnt = min(P - off, p1 - q);
                        const size_t src = (((size_t)pg * p.Hkv + g) * P + off) * HD;
                        const uint32_t bytes = (uint32_t)(cnt * HD * ES);
                        bulk_g2s(kd + (size_t)(q - p0) * HD * ES, Kc + src, bytes, &full_bar[slot]);
                        bulk_g2s(vd + (size_t)(q - p0) * HD * ES, Vc + src, bytes, &full_bar[slot]);
                        q += cnt;
                    }
                } else {
                    const size_t src = (((size_t)r * p.Hkv + g) * p.cap + p0) * HD;
                    const uint32_t bytes = (uint32_t)((p1 - p0) * HD * ES);
                    bulk_g2s(kd, Kc + src, bytes, &full_bar[slot]);
                    bulk_g2s(vd, Vc + src, bytes, &full_bar[slot]);
                }
                issued = t + 1;
            }
            for (int t = max(0, issued - S); t < issued; ++t)
                if (!mbar_wait(&full_bar[t % S], (t / S) & 1)) atomicOr(p.err, FAULT_WAIT);
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
    unsigned long long* tr = nullptr;   // trace buffer if tracing is on (thread 0)
    if (tid == 0) {
        tr = trace_if_on(p.trace);
        trace_mark(tr, p.trace_id, 1);
    }
    int pos = p.pos[r];
    pos = min(max(pos, 0), p.cap - 1);   // an out-of-range pos was flagged by the embedding kernel
    const float* qrow = p.qkv + (size_t)r * p.qkv_stride;
    const float2* rt = p.rope + (size_t)pos * (HD / 2);
    for (int i = tid; i < G * (HD / 2); i += AT_CT) {
        const int h = i / (HD / 2), d = i % (HD / 2);
        const float* qh = qrow + (size_t)(g * G + h) * HD;
        const float a = qh[d], b = qh[d + HD / 2];
        const float2 cs = rt[d];
        q_s[h * HD + d] = (a * cs.x - b * cs.y) * p.scale;
        q_s[h * HD + d + HD / 2] = (a * cs.y + b * cs.x) * p.scale;
    }
    if (pos >= j0 && pos < j1) {
        // the new k, v: RoPE, storage rounding, write at pos
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
        for (int d = tid; d < HD / 2; d += AT_CT) {
            const float a = kh[d], b = kh[d + HD / 2];
            const float2 cs = rt[d];
            const float k0 = a * cs.x - b * cs.y, k1 = a * cs.y + b * cs.x;
            kn_s[d] = ok ? Elem<KT>::round_store(k0, Kc + off + d) : Elem<KT>::round(k0);
            kn_s[d + HD / 2] = ok ? Elem<KT>::round_store(k1, Kc + off + d + HD / 2) : Elem<KT>::round(k1);
        }
        for (int d = tid; d < HD; d += AT_CT)
            vn_s[d] = ok ? Elem<KT>::round_store(vh[d], Vc + off + d) : Elem<KT>::round(vh[d]);
    }
    named_sync(1, AT_CT);
    pdl_trigger();

    const int sub = lane % LPP, pw = lane / LPP;
    float qr[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) qr[h][e] = q_s[h * HD + sub * DPL + e];

    // warp-local online softmax state
    float m[G], l[G], o[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
    }

    for (int t = 0; t < nst; ++t) {
        const int slot = t % S;
        if (!*abort_v && !mbar_wait(&full_bar[slot], (t / S) & 1)) {
            *abort_v = 1;
            atomicOr(p.err, FAULT_WAIT);
        }
        const bool live = !*abort_v;
        const unsigned char* kt = ring + (size_t)slot * AT_STAGE;
        const unsigned char* vt = kt + TILE;
        const int p0 = j0 + t * PPS;
        if (live) {
            // scores of this warp's positions: ITER iterations of PPI positions
            float sc[ITER][G];
            int jpos[ITER];
#pragma unroll
            for (int it = 0; it < ITER; ++it) {
                const int jl = warp * (ITER * PPI) + it * PPI + pw;   // position within the stage
                const int j = p0 + jl;
                jpos[it] = j;
                const uint4 kv = *reinterpret_cast<const uint4*>(kt + ((size_t)jl * HD + sub * DPL) * ES);
                float kf[DPL];
                Elem<KT>::unpack(kv, kf);
                if (j == pos) {
#pragma unroll
                    for (int e = 0; e < DPL; ++e) kf[e] = kn_s[sub * DPL + e];
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) a = fmaf(qr[h][e], kf[e], a);
                    sc[it][h] = a;
                }
            }
#pragma unroll
            for (int it = 0; it < ITER; ++it)
#pragma unroll
                for (int h = 0; h < G; ++h) {
#pragma unroll
                    for (int off = LPP / 2; off > 0; off >>= 1) sc[it][h] += __shfl_xor_sync(0xffffffffu, sc[it][h], off);
                    const bool valid = jpos[it] <= pos && jpos[it] < j1;
                    sc[it][h] = valid ? sc[it][h] : -INFINITY;
                }
            // new running max per head over the warp's positions
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mx = sc[0][h];
#pragma unroll
                for (int it = 1; it < ITER; ++it) mx = fmaxf(mx, sc[it][h]);
#pragma unroll
                for (int off = 16; off >= LPP; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float mn = fmaxf(m[h], mx);
                const float alpha = (m[h] == -INFINITY) ? 0.f : expf(m[h] - mn);
                float psum = 0.f;
#pragma unroll
                for (int it = 0; it < ITER; ++it) {
                    const float pj = (sc[it][h] == -INFINITY) ? 0.f : expf(sc[it][h] - mn);
                    sc[it][h] = pj;
                    psum += pj;
                }
#pragma unroll
                for (int off = 16; off >= LPP; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
                l[h] = l[h] * alpha + psum;
                m[h] = mn;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[h][e] *= alpha;
            }
            // o += p_j * v_j over the valid positions (masked v replaced by 0 by select)
#pragma unroll
            for (int it = 0; it < ITER; ++it) {
                const int jl = warp * (ITER * PPI) + it * PPI + pw;
                float vf[DPL];
                Elem<KT>::unpack(*reinterpret_cast<const uint4*>(vt + ((size_t)jl * HD + sub * DPL) * ES), vf);
                const int j = jpos[it];
                if (j == pos) {
#pragma unroll
                    for (int e = 0; e < DPL; ++e) vf[e] = vn_s[sub * DPL + e];
                }
                const bool valid = j <= pos && j < j1;
#pragma unroll
                for (int e = 0; e < DPL; ++e) vf[e] = valid ? vf[e] : 0.f;
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(sc[it][h], vf[e], o[h][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ---- merge the warps' states (fixed order), write the split partial ----
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
#pragma unroll
            for (int off = 16; off >= LPP; off >>= 1) o[h][e] += __shfl_xor_sync(0xffffffffu, o[h][e], off);
    named_sync(1, AT_CT);   // every warp is done with the ring: reuse it for the merge
    float* wo_s = reinterpret_cast<float*>(ring);   // [AT_CW][G][HD]
    if (pw == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL; ++e) wo_s[(warp * G + h) * HD + sub * DPL + e] = o[h][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            wm_s[warp][h] = m[h];
            wl_s[warp][h] = l[h];
        }
    }
    named_sync(1, AT_CT);
    for (int i = tid; i < G * HD; i += AT_CT) {
        const int h = i / HD, d = i % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AT_CW; ++w) M = fmaxf(M, wm_s[w][h]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < AT_CW; ++w) {
            const float f = (wm_s[w][h] == -INFINITY) ? 0.f : expf(wm_s[w][h] - M);
            Ls = fmaf(f, wl_s[w][h], Ls);
            Os = fmaf(f, wo_s[(w * G + h) * HD + d], Os);
        }
        float* pp = p.part + (((size_t)r * p.Hq + g * G + h) * p.nsplit + s) * (HD + 4);
        pp[4 + d] = Os;
        if (d == 0) {
            pp[0] = M;
            pp[1] = Ls;
        }
    }

    // ---- the last split of this (row, kv head) merges all splits ----
    __threadfence();
    named_sync(1, AT_CT);
    if (tid == 0) {
        const unsigned prev = atomicAdd(p.counters + r * p.Hkv + g, 1u);
        last_s = (prev == (unsigned)p.nsplit - 1u);
    }
    named_sync(1, AT_CT);
    if (tid == 0) trace_mark(tr, p.trace_id, 2);
    if (!last_s) return;
    __threadfence();
    if (tid == 0) p.counters[r * p.Hkv + g] = 0u;   // ready for the next step

    const int NS = p.nsplit;
    // this (row, kv head)'s partials are one contiguous block [G][NS][HD + 4]:
    // stage it in shared memory (the ring is free) with coalesced 16-byte loads
    float* pb = reinterpret_cast<float*>(ring);
    {
        const float4* src = reinterpret_cast<const float4*>(p.part + ((size_t)r * p.Hq + g * G) * NS * (HD + 4));
        const int n4 = G * NS * (HD + 4) / 4;
        for (int i = tid; i < n4; i += AT_CT) reinterpret_cast<float4*>(pb)[i] = __ldcg(src + i);
    }
    named_sync(1, AT_CT);
    for (int i = tid; i < G * NS; i += AT_CT) {
        const int h = i / NS, ss = i % NS;
        cm_s[h * NS + ss] = pb[(h * NS + ss) * (HD + 4)];
        cw_s[h * NS + ss] = pb[(h * NS + ss) * (HD + 4) + 1];
    }
    named_sync(1, AT_CT);
    for (int h = warp; h < G; h += AT_CW) {
        float M = -INFINITY;
        for (int ss = lane; ss < NS; ss += 32) M = fmaxf(M, cm_s[h * NS + ss]);
        M = warp_max(M);
        float Lsum = 0.f;
        for (int ss = lane; ss < NS; ss += 32) {
            const float mm = cm_s[h * NS + ss];
            Lsum += (mm == -INFINITY) ? 0.f : expf(mm - M) * cw_s[h * NS + ss];
        }
        Lsum = warp_sum(Lsum);
        for (int ss = lane; ss < NS; ss += 32) {
            const float mm = cm_s[h * NS + ss];
            cw_s[h * NS + ss] = (mm == -INFINITY) ? 0.f : expf(mm - M) / Lsum;
        }
    }
    named_sync(1, AT_CT);
    for (int i = tid; i < G * HD; i += AT_CT) {
        const int h = i / HD, d = i % HD;
        float acc = 0.f;
        for (int ss = 0; ss < NS; ++ss) acc = fmaf(cw_s[h * NS + ss], pb[(h * NS + ss) * (HD + 4) + 4 + d], acc);
        p.out[(size_t)r * p.Hq * HD + (size_t)(g * G + h) * HD + d] = acc;
    }
    named_sync(1, AT_CT);
    if (tid == 0) trace_mark(tr, p.trace_id, 3);
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
static const void* pick(int kvtype, int hd, int G, bool paged) {
    if (kvtype == W_BF16) {
        switch (hd) {
            case 16: return pick_group<__nv_bfloat16, 16>(G, paged);
            case 32: return pick_group<__nv_bfloat16, 32>(G, paged);
            case 64: return pick_group<__nv_bfloat16, 64>(G, paged);
            case 128: return pick_group<__nv_bfloat16, 128>(G, paged);
        }
    } else {
        switch (hd) {
            case 16: return pick_group<float, 16>(G, paged);
            case 32: return pick_group<float, 32>(G, paged);
            case 64: return pick_group<float, 64>(G, paged);
            case 128: return pick_group<float, 128>(G, paged);
        }
    }
    return nullptr;
}

cudaError_t attn_plan(AttnPlan* plan, int num_sms) {
    AttnParams& p = plan->p;
    if (p.Hkv <= 0 || p.Hq % p.Hkv) return cudaErrorInvalidValue;
    plan->group = p.Hq / p.Hkv;
    const void* fn = pick(plan->kvtype, p.hd, plan->group, plan->paged);
    if (!fn) return cudaErrorInvalidValue;
    const int es = plan->kvtype == W_BF16 ? 2 : 4;
    const int pps = AT_STAGE / (2 * p.hd * es);   // positions per stage
    if (plan->paged && (p.page_size < 1 || pps % p.page_size)) return cudaErrorInvalidValue;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    // Resident CTAs per SM that a ring of >= 2 stages allows (shared memory and
    // registers), for 1..3 co-resident CTAs.
    const int units = p.R * p.Hkv;
    const int max_ns = (p.cap + pps - 1) / pps;
    auto ring_stages = [&](int k, int ns) -> int {
        const size_t extra =
            ((size_t)plan->group * p.hd + 2 * (size_t)p.hd + 2 * (size_t)plan->group * ns) * sizeof(float);
        // per-SM shared memory is the per-block opt-in limit plus 1 KB reserved per block
        const long long per_cta = ((long long)optin + 1024) / k - 1024 - (long long)fa.sharedSizeBytes;
        int S = AT_MAX_S;
        while (S > 2 && (long long)((size_t)S * AT_STAGE + extra) > per_cta) --S;
        if ((long long)((size_t)S * AT_STAGE + extra) > per_cta) return 0;
        return S;
    };
    // the occupancy queries below see the dynamic shared-memory cap: raise it first
    if (cudaError_t e0 = raise_smem_cap(fn)) return e0;
    int kmax = 1;
    for (int k = 2; k <= 3; ++k) {
        const int S = ring_stages(k, max_ns);
        if (!S) break;
        int occ = 0;
        const size_t sm = (size_t)S * AT_STAGE +
                          ((size_t)plan->group * p.hd + 2 * (size_t)p.hd + 2 * (size_t)plan->group * max_ns) * 4;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, AT_THREADS, sm) != cudaSuccess || occ < k) break;
        kmax = k;
    }
    // Split choice: splits are whole stages; minimise the busiest SM's share
    // ceil(CTAs / SMs) * split_len with at most kmax co-resident CTAs per SM;
    // ties go to fewer splits.
    long long best_cost = -1;
    int best_L = 0, best_ns = 0;
    for (int want = 1; want <= max_ns; ++want) {
        int L = (p.cap + want - 1) / want;
        L = (L + pps - 1) / pps * pps;
        const int ns = (p.cap + L - 1) / L;
        const long long ctas = (long long)units * ns;
        const long long per_sm = (ctas + num_sms - 1) / num_sms;
        if (per_sm > kmax && want > 1) continue;
        // the final merge stages [G][ns][hd + 4] floats in a ring of >= 2 stages
        if ((size_t)plan->group * ns * (p.hd + 4) * sizeof(float) > 2 * (size_t)AT_STAGE && want > 1) continue;
        const long long cost = per_sm * L;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_L = L;
            best_ns = ns;
        }
    }
    p.split_len = best_L;
    p.nsplit = best_ns;
    const long long ctas = (long long)units * best_ns;
    int per_sm = (int)((ctas + num_sms - 1) / num_sms);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > kmax) per_sm = kmax;
    const int S = ring_stages(per_sm, best_ns);
    if (!S) return cudaErrorInvalidValue;
    // the final merge reuses the ring: [warps][G][hd] floats must fit
    if ((size_t)AT_CW * plan->group * p.hd * sizeof(float) > (size_t)S * AT_STAGE) return cudaErrorInvalidValue;
    p.stages = S;
    plan->smem = (size_t)S * AT_STAGE +
                 ((size_t)plan->group * p.hd + 2 * (size_t)p.hd + 2 * (size_t)plan->group * best_ns) * sizeof(float);
    if (plan->smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
    plan->block = AT_THREADS;
    plan->grid = dim3(p.nsplit, p.Hkv, p.R);
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
