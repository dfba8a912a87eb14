// attn_mma.cu -- masked split-KV decode attention over the fixed capacity for
// bf16 K/V, contractions on the tensor cores (sm_103a, mma.sync m16n8k16).
//
// What it computes is the same as attn.cu ("Execution", section "A
// constant-shape decode graph": the step writes K/V at pos, attention sweeps
// [0, cap), a mask from Slot::Pos against an iota hides every position after
// pos).  For a GQA group the step is a small dense contraction: the G query
// heads that share a kv head form Q [G x hd], scores S = Q K^T over the keys,
// then O = P V.  Here both run as m16n8k16 bf16 MMAs with fp32 accumulation:
//   * Q rows 0..7 hold bf16(q) of head g, rows 8..15 hold bf16(q - bf16(q)),
//     so S = C[g] + C[g + 8] carries ~16 mantissa bits of q (K is exact bf16);
//   * P is split the same way (rows g and g + 8) for P V;
//   * K/V tiles are staged by TMA tensor copies (128-byte swizzle) issued by
//     thread 0 -- the first ring fill before the programmatic-launch wait --
//     and read with ldmatrix (V transposed), conflict-free.
// Masking: scores of positions after pos (or past the split) are replaced by
// -inf by select; in the 16-key block that holds pos, the V fragments of
// masked keys are replaced by zero by select before the MMA, and blocks with
// no visible key skip the arithmetic (the TMA sweep still reads them), so
// garbage (NaN, Inf) in masked positions never reaches an arithmetic op.
// Each of the four warps keeps an online softmax over its keys; warps merge
// in fixed order, splits merge in split order in the last CTA of the (row, kv
// head) -- as in attn.cu.  The CTA holding pos writes the rotated, rounded
// new k, v to the store and into its staged tile before any read of it.
#include <cuda.h>
#include <math.h>
#include "common.cuh"
#include "internal.h"
#include "mma_helpers.cuh"

namespace gd {

constexpr int AM_WARPS = 4;
constexpr int AM_THREADS = AM_WARPS * 32;
constexpr int AM_STAGE = 32768;   // K tile + V tile
constexpr int AM_MAX_S = 3;   // ~96 KB ring: the next kernel's CTA can share the SM

template <int HD>
struct AmShape {
    static constexpr int PPS = AM_STAGE / (2 * HD * 2);     // keys per stage (64 for hd 128, 128 for hd 64)
    static constexpr int KPW = PPS / AM_WARPS;              // keys per warp per stage
    static constexpr int BLK = KPW / 16;                    // 16-key blocks per warp per stage
    static constexpr int SUB = HD / 64;                     // 64-column (128-byte) sub-tiles per row
    static constexpr int TILE = PPS * HD * 2;               // bytes of the K (or V) tile
    static constexpr int KSTEP = HD / 16;                   // k-steps of the QK contraction
    static constexpr int NT = HD / 8;                       // 8-column output tiles of P V
    static_assert(KPW % 16 == 0 && BLK >= 1, "stage shape");
};

struct AttnMmaParams {   // 64-byte aligned through its CUtensorMap members
    CUtensorMap kmap;
    CUtensorMap vmap;
    AttnParams a;
};

template <int HD, int G, bool PAGED>
__global__ void __launch_bounds__(AM_THREADS, 2) k_attn_mma(const __grid_constant__ AttnMmaParams prm) {
    using SH = AmShape<HD>;
    constexpr int PPS = SH::PPS, KPW = SH::KPW, BLK = SH::BLK, SUB = SH::SUB, TILE = SH::TILE;
    constexpr int KSTEP = SH::KSTEP, NT = SH::NT;
    static_assert(G >= 1 && G <= 8, "group");
    const AttnParams& p = prm.a;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1 KB alignment for the swizzled tiles
    unsigned char* ring =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    float* q_s = reinterpret_cast<float*>(ring + (size_t)p.stages * AM_STAGE);   // [G][HD]
    float* kn_s = q_s + G * HD;                                                  // [HD]
    float* vn_s = kn_s + HD;                                                     // [HD]
    float* cm_s = vn_s + HD;                                                     // [G][nsplit]
    float* cw_s = cm_s + G * p.nsplit;                                           // [G][nsplit]
    __shared__ __align__(8) uint64_t full_bar[AM_MAX_S];
    __shared__ float wm_s[AM_WARPS][8], wl_s[AM_WARPS][8];
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
    __nv_bfloat16* Kc = reinterpret_cast<__nv_bfloat16*>(p.Kc);
    __nv_bfloat16* Vc = reinterpret_cast<__nv_bfloat16*>(p.Vc);

    auto issue = [&](int t) {
        const int slot = t % S;
        const int p0 = j0 + t * PPS, p1 = min(p0 + PPS, j1);
        unsigned char* kd = ring + (size_t)slot * AM_STAGE;
        unsigned char* vd = kd + TILE;
        if (PAGED) {
            // whole pages: a split is a multiple of the stage, a stage a multiple of the page
            const int npg = (p1 - p0 + P - 1) / P;
            mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(2 * npg * P * HD * 2));
            for (int i = 0; i < npg; ++i) {
                const int q = p0 + i * P;
                int pg = p.slot_map[(size_t)r * p.pages_per_row + q / P];
                if (pg < 0 || pg >= p.num_pages) {
                    atomicOr(p.err, FAULT_SLOT_MAP);
                    pg = 0;
                }
                const int y = (pg * p.Hkv + g) * P;
#pragma unroll
                for (int sb = 0; sb < SUB; ++sb) {
                    tma_load_2d(kd + sb * PPS * 128 + i * P * 128, &prm.kmap, sb * 64, y, &full_bar[slot]);
                    tma_load_2d(vd + sb * PPS * 128 + i * P * 128, &prm.vmap, sb * 64, y, &full_bar[slot]);
                }
            }
        } else {
            // one box of PPS rows per 64-column sub-tile; rows past the tensor read as zero
            mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(2 * PPS * HD * 2));
            const int y = (r * p.Hkv + g) * p.cap + p0;
#pragma unroll
            for (int sb = 0; sb < SUB; ++sb) {
                tma_load_2d(kd + sb * PPS * 128, &prm.kmap, sb * 64, y, &full_bar[slot]);
                tma_load_2d(vd + sb * PPS * 128, &prm.vmap, sb * 64, y, &full_bar[slot]);
            }
        }
    };
    int issued = 0;
    unsigned long long* tr = nullptr;   // trace buffer if tracing is on (thread 0)
    if (tid == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&full_bar[i], 1);
        abort_s = 0;
        mbar_fence_init();
        // the first ring fill does not depend on the previous kernel -- unless
        // that kernel wrote this step's keys (rows may share pages), or the
        // fill is bounded by pos (read after the wait)
        if (!p.kv_prewritten && !p.pos_bound)
            for (; issued < min(S, nst); ++issued) issue(issued);
        tr = trace_if_on(p.trace);   // after the copies: the enable word is a global load
        trace_mark(tr, p.trace_id, 0);
    }
    __syncthreads();

    pdl_wait();
    int pos = p.pos[r];
    pos = min(max(pos, 0), p.cap - 1);   // an out-of-range pos was flagged by the embedding kernel
    // stages this split loads: all of them, or (pos-bounded sweep) those up to
    // the one holding pos; the stages left out hold no visible key, so no
    // arithmetic would have touched them
    const int nld = !p.pos_bound ? nst : (pos < j0 ? 0 : min(nst, (pos - j0) / PPS + 1));
    if (tid == 0) {
        for (; issued < min(S, nld); ++issued) issue(issued);
        trace_mark(tr, p.trace_id, 1);
    }
    const float* qrow = p.qkv + (size_t)r * p.qkv_stride;
    const float2* rt = p.rope + (size_t)pos * (HD / 2);
    for (int i = tid; i < G * (HD / 2); i += AM_THREADS) {
        const int h = i / (HD / 2), d = i % (HD / 2);
        const float* qh = qrow + (size_t)(g * G + h) * HD;
        const float a = qh[d], b = qh[d + HD / 2];
        const float2 cs = rt[d];
        q_s[h * HD + d] = (a * cs.x - b * cs.y) * p.scale;
        q_s[h * HD + d + HD / 2] = (a * cs.y + b * cs.x) * p.scale;
    }
    const bool owner = !p.kv_prewritten && pos >= j0 && pos < j1;
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
        for (int d = tid; d < HD / 2; d += AM_THREADS) {
            const float a = kh[d], b = kh[d + HD / 2];
            const float2 cs = rt[d];
            const float k0 = a * cs.x - b * cs.y, k1 = a * cs.y + b * cs.x;
            kn_s[d] = ok ? Elem<__nv_bfloat16>::round_store(k0, Kc + off + d) : bf16_round_f(k0);
            kn_s[d + HD / 2] = ok ? Elem<__nv_bfloat16>::round_store(k1, Kc + off + d + HD / 2) : bf16_round_f(k1);
        }
        for (int d = tid; d < HD; d += AM_THREADS)
            vn_s[d] = ok ? Elem<__nv_bfloat16>::round_store(vh[d], Vc + off + d) : bf16_round_f(vh[d]);
    }
    __syncthreads();
    pdl_trigger();

    // ---- Q fragments: rows g = head (bf16 of q), rows g + 8 = the bf16 remainder ----
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t qa[KSTEP][4];
#pragma unroll
    for (int ks = 0; ks < KSTEP; ++ks) {
        float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
        if (gq < G) {
            const float* qh = q_s + gq * HD + ks * 16 + 2 * tq;
            v0 = qh[0]; v1 = qh[1]; v2 = qh[8]; v3 = qh[9];
        }
        const float h0 = bf16_round_f(v0), h1 = bf16_round_f(v1), h2 = bf16_round_f(v2), h3 = bf16_round_f(v3);
        qa[ks][0] = pack_bf16x2(h0, h1);
        qa[ks][1] = pack_bf16x2(v0 - h0, v1 - h1);
        qa[ks][2] = pack_bf16x2(h2, h3);
        qa[ks][3] = pack_bf16x2(v2 - h2, v3 - h3);
    }

    // online softmax state of head gq over this warp's keys (replicated over tq)
    float m_run = -INFINITY, l_run = 0.f;
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    for (int t = 0; t < nld; ++t) {
        const int slot = t % S;
        if (!*abort_v && !mbar_wait(&full_bar[slot], (t / S) & 1)) {
            *abort_v = 1;
            atomicOr(p.err, FAULT_WAIT);
        }
        const bool live = !*abort_v;
        unsigned char* kt = ring + (size_t)slot * AM_STAGE;
        unsigned char* vt = kt + TILE;
        const int p0 = j0 + t * PPS;
        if (owner && pos >= p0 && pos < p0 + PPS) {   // CTA-uniform (no abort test: it guards a barrier)
            // the new k, v replace the staged row of position pos
            const int row = pos - p0;
            for (int i = tid; i < 2 * (HD / 8); i += AM_THREADS) {
                const int c = i % (HD / 8);
                const float* src = (i < HD / 8 ? kn_s : vn_s) + c * 8;
                uint4 v;
                v.x = pack_bf16x2(src[0], src[1]);
                v.y = pack_bf16x2(src[2], src[3]);
                v.z = pack_bf16x2(src[4], src[5]);
                v.w = pack_bf16x2(src[6], src[7]);
                *reinterpret_cast<uint4*>((i < HD / 8 ? kt : vt) + swz<HD, PPS>(row, c)) = v;
            }
            __syncthreads();
        }
        if (live) {
#pragma unroll
            for (int b = 0; b < BLK; ++b) {
                const int kb = warp * KPW + b * 16;   // first key of this 16-key block (within the stage)
                const int key0 = p0 + kb;
                if (key0 > pos || key0 >= j1) continue;   // no visible key in the block (warp-uniform)
                // S = Q K^T for 16 keys: two 8-key tiles
                float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KSTEP; ++ks) {
                    // matrices: (keys 0-7, dims 0-7), (keys 0-7, dims 8-15), (keys 8-15, dims 0-7), (keys 8-15, dims 8-15)
                    const int mi = lane >> 3, rr = lane & 7;
                    const int krow = kb + rr + ((mi >> 1) << 3);
                    const int chunk = ks * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(kt + swz<HD, PPS>(krow, chunk)), b0, b1, b2, b3);
                    mma_bf16(sacc[0], qa[ks], b0, b1);
                    mma_bf16(sacc[1], qa[ks], b2, b3);
                }
                // scores of this lane's keys (head gq): tile n, key kb + 8n + 2tq + {0,1}
                float sc[4];
                bool vis[4];
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = key0 + 8 * n + 2 * tq + e;
                        vis[2 * n + e] = key <= pos && key < j1;
                        const float v = sacc[n][e] + sacc[n][2 + e];
                        sc[2 * n + e] = vis[2 * n + e] ? v : -INFINITY;
                    }
                float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m_run, mx);   // finite: the block has a visible key
                const float alpha = (m_run == -INFINITY) ? 0.f : expf(m_run - mn);
                float pr[4];
                float ps = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pr[i] = vis[i] ? expf(sc[i] - mn) : 0.f;
                    ps += pr[i];
                }
                l_run = l_run * alpha + ps;
                m_run = mn;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    o[n][0] *= alpha; o[n][1] *= alpha; o[n][2] *= alpha; o[n][3] *= alpha;
                }
                // P fragments: rows gq = bf16(p), rows gq + 8 = remainder; keys of tile 0 then tile 1
                uint32_t pa[4];
                {
                    const float h0 = bf16_round_f(pr[0]), h1 = bf16_round_f(pr[1]);
                    const float h2 = bf16_round_f(pr[2]), h3 = bf16_round_f(pr[3]);
                    pa[0] = pack_bf16x2(h0, h1);
                    pa[1] = pack_bf16x2(pr[0] - h0, pr[1] - h1);
                    pa[2] = pack_bf16x2(h2, h3);
                    pa[3] = pack_bf16x2(pr[2] - h2, pr[3] - h3);
                }
                // V fragments of masked keys become zero by select (block holding pos only)
                const bool partial = key0 + 15 > pos || key0 + 15 >= j1;
                // a B register holds keys (2tq, 2tq+1) [b0] or (8+2tq, 8+2tq+1) [b1] of one dim column
                const uint32_t keep0 = (vis[0] ? 0x0000FFFFu : 0u) | (vis[1] ? 0xFFFF0000u : 0u);
                const uint32_t keep1 = (vis[2] ? 0x0000FFFFu : 0u) | (vis[3] ? 0xFFFF0000u : 0u);
                // O += P V: output tiles of 8 dims, two per ldmatrix.x4.trans
#pragma unroll
                for (int n2 = 0; n2 < NT / 2; ++n2) {
                    // matrices: (keys 0-7, dims 16n2..+7), (keys 8-15, same), (keys 0-7, dims +8..), (keys 8-15, +8..)
                    const int mi = lane >> 3, rr = lane & 7;
                    const int vrow = kb + rr + ((mi & 1) << 3);
                    const int chunk = n2 * 2 + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(vt + swz<HD, PPS>(vrow, chunk)), b0, b1, b2, b3);
                    if (partial) {
                        // after the transpose, lane (gq, tq) holds keys 2tq, 2tq+1 (b0/b2) and
                        // 8+2tq, 9+2tq (b1/b3): the same keys as its scores
                        b0 &= keep0;
                        b2 &= keep0;
                        b1 &= keep1;
                        b3 &= keep1;
                    }
                    mma_bf16(o[2 * n2], pa, b0, b1);
                    mma_bf16(o[2 * n2 + 1], pa, b2, b3);
                }
            }
        }
        __syncthreads();   // every warp is done with slot `slot`
        if (tid == 0 && !*abort_v && issued < nld) {
            fence_proxy_async_smem();   // generic writes to the slot (pos row) before the async refill
            issue(issued++);
        }
    }
    if (tid == 0) {
        for (int t = max(0, issued - S); t < issued; ++t)
            if (!mbar_wait(&full_bar[t % S], (t / S) & 1)) atomicOr(p.err, FAULT_WAIT);
    }

    // ---- merge the warps (fixed order), write the split partial ----
    // sum the remainder rows into the head rows, and l over the four lanes of a head
    float lsum = l_run;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    __syncthreads();
    float* wo_s = reinterpret_cast<float*>(ring);   // [AM_WARPS][8][HD], ring is free now
    if (gq < G) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            wo_s[(warp * 8 + gq) * HD + n * 8 + 2 * tq] = o[n][0] + o[n][2];
            wo_s[(warp * 8 + gq) * HD + n * 8 + 2 * tq + 1] = o[n][1] + o[n][3];
        }
        if (tq == 0) {
            wm_s[warp][gq] = m_run;
            wl_s[warp][gq] = lsum;
        }
    }
    __syncthreads();
    for (int i = tid; i < G * HD; i += AM_THREADS) {
        const int h = i / HD, d = i % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AM_WARPS; ++w) M = fmaxf(M, wm_s[w][h]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < AM_WARPS; ++w) {
            const float f = (wm_s[w][h] == -INFINITY) ? 0.f : expf(wm_s[w][h] - M);
            Ls = fmaf(f, wl_s[w][h], Ls);
            Os = fmaf(f, wo_s[(w * 8 + h) * HD + d], Os);
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
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(p.counters + r * p.Hkv + g, 1u);
        last_s = (prev == (unsigned)p.nsplit - 1u);
        trace_mark(tr, p.trace_id, 2);
    }
    __syncthreads();
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
        for (int i = tid; i < n4; i += AM_THREADS) reinterpret_cast<float4*>(pb)[i] = __ldcg(src + i);
    }
    __syncthreads();
    for (int i = tid; i < G * NS; i += AM_THREADS) {
        const int h = i / NS, ss = i % NS;
        cm_s[h * NS + ss] = pb[(h * NS + ss) * (HD + 4)];
        cw_s[h * NS + ss] = pb[(h * NS + ss) * (HD + 4) + 1];
    }
    __syncthreads();
    for (int h = warp; h < G; h += AM_WARPS) {
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
    __syncthreads();
    for (int i = tid; i < G * HD; i += AM_THREADS) {
        const int h = i / HD, d = i % HD;
        float acc = 0.f;
        for (int ss = 0; ss < NS; ++ss) acc = fmaf(cw_s[h * NS + ss], pb[(h * NS + ss) * (HD + 4) + 4 + d], acc);
        p.out[(size_t)r * p.Hq * HD + (size_t)(g * G + h) * HD + d] = acc;
    }
    __syncthreads();
    if (tid == 0) trace_mark(tr, p.trace_id, 3);
}

// ---------------- host side ----------------

// The K/V write of every row as its own kernel, so that rows which share
// pages (the chunk of a multi-token prefill: row t is position pos0 + t of one
// sequence) all see each other's new keys.  One CTA per (kv head, row);
// arithmetic identical to the in-kernel write of k_attn_mma.
__global__ void __launch_bounds__(128) k_kv_write(const AttnParams p) {
    const int g = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const int HD = p.hd;
    pdl_wait();
    int pos = p.pos[r];
    pos = min(max(pos, 0), p.cap - 1);   // an out-of-range pos was flagged by the embedding kernel
    const float* kh = p.qkv + (size_t)r * p.qkv_stride + (size_t)p.Hq * HD + (size_t)g * HD;
    const float* vh = kh + (size_t)p.Hkv * HD;
    const float2* rt = p.rope + (size_t)pos * (HD / 2);
    size_t off;
    if (p.page_size > 0 && p.write_map && p.slot_map) {
        const int P = p.page_size;
        const int slot = p.write_map[r];
        if (slot < 0 || slot >= p.num_pages * P) {
            if (tid == 0) atomicOr(p.err, FAULT_WRITE_MAP);
            pdl_trigger();
            return;
        }
        off = (((size_t)(slot / P) * p.Hkv + g) * P + slot % P) * HD;
    } else {
        off = (((size_t)r * p.Hkv + g) * p.cap + pos) * HD;
    }
    __nv_bfloat16* Kc = reinterpret_cast<__nv_bfloat16*>(p.Kc);
    __nv_bfloat16* Vc = reinterpret_cast<__nv_bfloat16*>(p.Vc);
    for (int d = tid; d < HD / 2; d += blockDim.x) {
        const float a = kh[d], b = kh[d + HD / 2];
        const float2 cs = rt[d];
        Elem<__nv_bfloat16>::round_store(a * cs.x - b * cs.y, Kc + off + d);
        Elem<__nv_bfloat16>::round_store(a * cs.y + b * cs.x, Kc + off + d + HD / 2);
    }
    for (int d = tid; d < HD; d += blockDim.x) Elem<__nv_bfloat16>::round_store(vh[d], Vc + off + d);
    pdl_trigger();
}

cudaError_t kv_write_launch(const AttnPlan& plan, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.p.Hkv, plan.p.R);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    AttnParams p = plan.p;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, (const void*)&k_kv_write, args);
}

template <int HD, int G>
static const void* am_pick_paged(bool paged) {
    return paged ? (const void*)&k_attn_mma<HD, G, true> : (const void*)&k_attn_mma<HD, G, false>;
}
template <int HD>
static const void* am_pick_group(int G, bool paged) {
    switch (G) {
        case 1: return am_pick_paged<HD, 1>(paged);
        case 2: return am_pick_paged<HD, 2>(paged);
        case 4: return am_pick_paged<HD, 4>(paged);
        case 8: return am_pick_paged<HD, 8>(paged);
    }
    return nullptr;
}
static const void* am_pick(int hd, int G, bool paged) {
    if (hd == 64) return am_pick_group<64>(G, paged);
    if (hd == 128) return am_pick_group<128>(G, paged);
    return nullptr;
}

bool attn_mma_supported(int kvtype, int hd, int G, bool paged, int page_size) {
    if (kvtype != W_BF16 || (hd != 64 && hd != 128) || !am_pick(hd, G, paged)) return false;
    const int pps = AM_STAGE / (2 * hd * 2);
    if (paged && (page_size < 8 || page_size % 8 || pps % page_size)) return false;
    return true;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D bf16 view [rows, hd] of a K or V store, boxes of [64 columns x box_rows]
static cudaError_t make_map(CUtensorMap* map, void* base, long long rows, int hd, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t attn_mma_plan(AttnPlan* plan, int num_sms) {
    AttnParams& p = plan->p;
    plan->group = p.Hq / p.Hkv;
    const void* fn = am_pick(p.hd, plan->group, plan->paged);
    if (!fn) return cudaErrorInvalidValue;
    const int pps = AM_STAGE / (2 * p.hd * 2);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    // the occupancy queries below see the dynamic shared-memory cap: raise it first
    if ((e = raise_smem_cap(fn)) != cudaSuccess) return e;
    const int units = p.R * p.Hkv;
    const int max_ns = (p.cap + pps - 1) / pps;
    auto extra = [&](int ns) {
        return ((size_t)plan->group * p.hd + 2 * (size_t)p.hd + 2 * (size_t)plan->group * ns) * sizeof(float) + 1024;
    };
    auto stages_for = [&](int k, int ns) -> int {
        const long long per_cta = ((long long)optin + 1024) / k - 1024 - (long long)fa.sharedSizeBytes;
        for (int S = AM_MAX_S; S >= 2; --S)
            if ((long long)((size_t)S * AM_STAGE + extra(ns)) <= per_cta) return S;
        return 0;
    };
    int kmax = 1;
    for (int k = 2; k <= 4; ++k) {
        const int S = stages_for(k, max_ns);
        if (!S) break;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, AM_THREADS, (size_t)S * AM_STAGE + extra(max_ns)) !=
                cudaSuccess ||
            occ < k)
            break;
        kmax = k;
    }
    // split choice as in attn.cu: whole stages per split, minimise the busiest
    // SM's share with at most kmax co-resident CTAs per SM
    long long best_cost = -1;
    int best_L = 0, best_ns = 0;
    for (int want = 1; want <= max_ns; ++want) {
        int Ls = (p.cap + want - 1) / want;
        Ls = (Ls + pps - 1) / pps * pps;
        const int ns = (p.cap + Ls - 1) / Ls;
        const long long ctas = (long long)units * ns;
        const long long per_sm = (ctas + num_sms - 1) / num_sms;
        if (per_sm > kmax && want > 1) continue;
        // the final merge stages [G][ns][hd + 4] floats in a ring of >= 2 stages
        if ((size_t)plan->group * ns * (p.hd + 4) * sizeof(float) > 2 * (size_t)AM_STAGE && want > 1) continue;
        // one CTA streams well below an SM's share of HBM bandwidth, so CTAs
        // sharing an SM run side by side: the time is the split length
        // (+ a small per-split merge cost)
        const long long cost = Ls + 64;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_L = Ls;
            best_ns = ns;
        }
    }
    p.split_len = best_L;
    p.nsplit = best_ns;
    int per_sm = (int)(((long long)units * best_ns + num_sms - 1) / num_sms);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > kmax) per_sm = kmax;
    const int S = stages_for(per_sm, best_ns);
    if (!S) return cudaErrorInvalidValue;
    // the warp merge reuses the ring: [warps][8][hd] floats
    if ((size_t)AM_WARPS * 8 * p.hd * sizeof(float) > (size_t)S * AM_STAGE) return cudaErrorInvalidValue;
    p.stages = S;
    plan->smem = (size_t)S * AM_STAGE + extra(best_ns);
    if (plan->smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidValue;
    plan->block = AM_THREADS;
    plan->grid = dim3(p.nsplit, p.Hkv, p.R);
    plan->mma = true;
    // tensor maps over this layer's K and V stores
    const long long rows = plan->paged ? (long long)p.num_pages * p.Hkv * p.page_size : (long long)p.R * p.Hkv * p.cap;
    const int box_rows = plan->paged ? p.page_size : pps;
    AttnMmaParams* mp = new AttnMmaParams();
    if ((e = make_map(&mp->kmap, p.Kc, rows, p.hd, box_rows)) != cudaSuccess ||
        (e = make_map(&mp->vmap, p.Vc, rows, p.hd, box_rows)) != cudaSuccess) {
        delete mp;
        return e;
    }
    plan->mma_params = mp;
    return raise_smem_cap(fn);
}

cudaError_t attn_mma_launch(const AttnPlan& plan, cudaStream_t s, bool pdl) {
    const void* fn = am_pick(plan.p.hd, plan.group, plan.paged);
    if (!fn || !plan.mma_params) return cudaErrorInvalidValue;
    AttnMmaParams* mp = reinterpret_cast<AttnMmaParams*>(plan.mma_params);
    mp->a = plan.p;
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
    void* args[] = {mp};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

void attn_mma_release(AttnPlan& plan) {
    delete reinterpret_cast<AttnMmaParams*>(plan.mma_params);
    plan.mma_params = nullptr;
}

}  // namespace gd
