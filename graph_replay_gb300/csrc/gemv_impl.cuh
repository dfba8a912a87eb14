// gemv_impl.cuh -- fused (RMSNorm | SwiGLU) + GEMV + (store | residual add |
// logits + greedy argmax) for small-batch decode on sm_103a.
//
// Decode at 1..8 rows multiplies every weight matrix by a few activation
// vectors: each weight byte is read once per step, so the kernel is bound by
// HBM bandwidth and its job is to keep enough bytes in flight on every SM.
// Design (one persistent CTA per SM):
//   * the CTA owns a contiguous, balanced range of output rows -- a contiguous
//     byte range of each weight segment (e.g. Wq;Wk;Wv stacked);
//   * thread 0 streams that range through a ring of shared-memory stages (up
//     to 64 KB, whole rows) with bulk asynchronous copies (cp.async.bulk,
//     mbarrier completion), ~128-192 KB in flight per SM; a stage's slot is
//     refilled right after the barrier that ends its consumption;
//   * the first ring fill is issued before the programmatic-launch wait: the
//     weights do not depend on the previous kernel, so the ring fills while
//     that kernel's tail is still running;
//   * sixteen consumer warps: eight K-slices x two row groups (even / odd rows
//     of each stage); a lane's activation values for its columns are built
//     once by the prologue (RMSNorm with gain, SwiGLU, or a copy) and kept in
//     registers, so shared memory only carries the weights;
//   * per stage: warp-shuffle reduction of each row's slice partial, a named
//     barrier, and a fixed-order sum of the eight slice partials by warp 0,
//     which applies the epilogue -- results do not depend on scheduling.
// Every mbarrier wait is bounded; a wait that gives up sets FAULT_WAIT in the
// error word, the CTA stops consuming and issuing, and thread 0 waits (bounded)
// for the copies in flight before the CTA exits.
//
// The pages' composition: "Models, Registry and the Driver", section "Shared
// components" (x += mixer(norm(x)); x += ffn(norm(x)); final norm and head);
// "Architecture Overview", section "Automatic fusion" (RMSNorm and SwiGLU as
// fusable regions).  The greedy pick is the sampling suffix ("Models, Registry
// and the Driver", section "The Driver": the host reads back a token id and a
// non-finite flag).
#pragma once
#include "common.cuh"
#include "internal.h"

namespace gd {

constexpr int GV_SL = 8;                 // K-slices
constexpr int GV_GR = 1;                 // row groups (a stage's rows alternate between them)
constexpr int GV_CW = GV_SL * GV_GR;     // consumer warps
constexpr int GV_CT = GV_CW * 32;        // consumer threads
constexpr int GV_THREADS = GV_CT;        // thread 0 also issues the bulk copies
constexpr int GV_MAX_S = 6;              // ring stages at most
constexpr int GV_MAX_RPS = 32;           // rows per stage at most
constexpr int GV_MAX_RES = 64;           // residual rows a CTA keeps in shared memory (EPI_ADD)

// weight segment holding output row `row`: its pointer, first row and row count
// (selects without indexing the parameter arrays, which would force a local copy)
__device__ __forceinline__ const void* segment_of(const GemvParams& p, int row, int& base, int& nrows) {
    const int e0 = p.seg_rows[0], e1 = e0 + p.seg_rows[1];
    if (row < e0) { base = 0; nrows = p.seg_rows[0]; return p.w[0]; }
    if (row < e1) { base = e0; nrows = p.seg_rows[1]; return p.w[1]; }
    base = e1;
    nrows = p.seg_rows[2];
    return p.w[2];
}

// rows whose slice products are loaded together (register budget ~32 words)
template <int CPL> struct RowUnroll { static constexpr int value = CPL == 0 ? 2 : (8 / CPL > 0 ? 8 / CPL : 1); };

template <typename WT, int NR, int PRO, int EPI, int CPL>
__global__ void __launch_bounds__(GV_THREADS, 2) k_gemv(const GemvParams p) {
    constexpr int VEC = Elem<WT>::VEC;
    constexpr int ES = (int)sizeof(WT);
    constexpr int RU = RowUnroll<CPL>::value;
    constexpr int CA = CPL > 0 ? CPL : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[GV_MAX_S];
    __shared__ float red_s[2][GV_MAX_RPS][GV_SL][NR];
    __shared__ float nrm_s[GV_CW][NR];
    __shared__ float res_s[EPI == EPI_ADD ? GV_MAX_RES : 1][NR];   // this CTA's residual rows
    __shared__ int abort_s;
    volatile int* abort_v = &abort_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K;
    const int row0 = (int)(((long long)blockIdx.x * p.N) / gridDim.x);
    const int row1 = (int)(((long long)(blockIdx.x + 1) * p.N) / gridDim.x);
    const int rps = p.rps;
    const int nst = (row1 - row0 + rps - 1) / rps;
    const int S = p.stages;
    const size_t row_bytes = (size_t)K * ES;
    const size_t stage_bytes = (size_t)rps * row_bytes;
    unsigned char* ring = smem;
    float* act_s = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);   // [NR][K], CPL == 0 only

    // stage k: rows [row0 + k*rps, ...) into slot k % S, completing on full_bar
    auto issue = [&](int k) {
        const int slot = k % S;
        const int a = row0 + k * rps, b = min(a + rps, row1);
        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)((size_t)(b - a) * row_bytes));
        unsigned char* dst = ring + (size_t)slot * stage_bytes;
        int r = a;
        while (r < b) {
            int base, nseg;
            const void* w = segment_of(p, r, base, nseg);
            const int e = min(b, base + nseg);
            const uint32_t bytes = (uint32_t)((size_t)(e - r) * row_bytes);
            bulk_g2s(dst, reinterpret_cast<const unsigned char*>(w) + (size_t)(r - base) * row_bytes, bytes,
                     &full_bar[slot]);
            dst += bytes;
            r = e;
        }
    };
    int issued = 0;                  // meaningful in thread 0
    unsigned long long* tr = nullptr;   // trace buffer if tracing is on (thread 0)
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full_bar[s], 1);
        abort_s = 0;
        mbar_fence_init();
        // the first ring fill does not depend on the previous kernel
        for (; issued < min(S, nst); ++issued) issue(issued);
        tr = trace_if_on(p.trace);   // after the copies: the enable word is a global load
        trace_mark(tr, p.trace_id, 0);
    }
    __syncthreads();

    // ---------------- consumers ----------------
    pdl_wait();
    if (tid == 0) trace_mark(tr, p.trace_id, 1);
    const int SWV = K / (GV_SL * VEC);   // 16-byte vectors in one warp's K-slice
    const int slice = warp % GV_SL, grp = warp / GV_SL;
    const int vbase = slice * SWV;
    const bool exact = SWV == 32 * CA;   // every lane owns exactly CA vectors of the slice

    float inv[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) inv[r] = 1.f;
    if (PRO == PRO_RMSNORM) {
        float ss[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            ss[r] = 0.f;
            if (r < p.R) {
                const float* a = p.act + (size_t)r * p.act_stride;
                for (int k = tid * 4; k < K; k += GV_CT * 4) {
                    const float4 x = *reinterpret_cast<const float4*>(a + k);
                    ss[r] = fmaf(x.x, x.x, ss[r]);
                    ss[r] = fmaf(x.y, x.y, ss[r]);
                    ss[r] = fmaf(x.z, x.z, ss[r]);
                    ss[r] = fmaf(x.w, x.w, ss[r]);
                }
            }
            ss[r] = warp_sum(ss[r]);
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) nrm_s[warp][r] = ss[r];
        }
        named_sync(1, GV_CT);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < GV_CW; ++w) t += nrm_s[w][r];
            inv[r] = 1.0f / sqrtf(t / (float)K + p.eps);
        }
    }
    const WT* gain = reinterpret_cast<const WT*>(p.gain);
    // the prologue's activation values for columns [c, c + VEC) of row r
    auto act_vec = [&](int r, int c, float (&o)[VEC]) {
        if (r >= p.R) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = 0.f;
            return;
        }
        const float* a = p.act + (size_t)r * p.act_stride + c;
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
            const float4 x = *reinterpret_cast<const float4*>(a + e);
            o[e] = x.x; o[e + 1] = x.y; o[e + 2] = x.z; o[e + 3] = x.w;
        }
        if (PRO == PRO_RMSNORM) {
            float g[VEC];
            Elem<WT>::unpack(*reinterpret_cast<const uint4*>(gain + c), g);
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = o[e] * inv[r] * g[e];
        } else if (PRO == PRO_SWIGLU) {
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
                const float4 u = *reinterpret_cast<const float4*>(a + K + e);
                const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) o[e + q] = o[e + q] / (1.0f + expf(-o[e + q])) * uu[q];
            }
        }
    };

    float areg[NR][CA][VEC];
    if (CPL > 0) {
#pragma unroll
        for (int j = 0; j < CA; ++j) {
            const int v = vbase + lane + 32 * j;
            const bool in = v < vbase + SWV;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (in) {
                    act_vec(r, v * VEC, areg[r][j]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) areg[r][j][e] = 0.f;
                }
            }
        }
    } else {
        for (int i = tid; i < NR * (K / VEC); i += GV_CT) {
            const int r = i / (K / VEC), c = (i % (K / VEC)) * VEC;
            float o[VEC];
            act_vec(r, c, o);
#pragma unroll
            for (int e = 0; e < VEC; ++e) act_s[(size_t)r * K + c + e] = o[e];
        }
    }
    // residual rows of this CTA, read once (the epilogue then adds without a global read)
    const bool res_local = EPI == EPI_ADD && (row1 - row0) <= GV_MAX_RES;
    if (EPI == EPI_ADD && res_local) {
        for (int i = tid; i < (row1 - row0) * NR; i += GV_CT) {
            const int rr = i / NR, r = i % NR;
            res_s[rr][r] = r < p.R ? p.out[(size_t)r * p.out_stride + row0 + rr] : 0.f;
        }
    }
    if (CPL == 0 || EPI == EPI_ADD) named_sync(1, GV_CT);
    pdl_trigger();

    unsigned long long best[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) best[r] = 0ull;
    bool nonfin = false;

    for (int k = 0; k < nst; ++k) {
        const int slot = k % S;
        const int a = row0 + k * rps;
        const int nr = min(rps, row1 - a);
        if (!*abort_v && !mbar_wait(&full_bar[slot], (k / S) & 1)) {
            *abort_v = 1;
            atomicOr(p.err, FAULT_WAIT);
        }
        const bool live = !*abort_v;
        const unsigned char* st = ring + (size_t)slot * stage_bytes;
        // this warp's rows of the stage: grp, grp + GV_GR, ...
        const int nmine = nr > grp ? (nr - grp + GV_GR - 1) / GV_GR : 0;
        for (int m0 = 0; m0 < nmine; m0 += RU) {
            float acc[RU][NR];
#pragma unroll
            for (int u = 0; u < RU; ++u)
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[u][r] = 0.f;
            if (live) {
                if (CPL > 0) {
                    uint4 wv[RU][CA];
                    if (exact && m0 + RU <= nmine) {
#pragma unroll
                        for (int u = 0; u < RU; ++u) {
                            const uint4* wr = reinterpret_cast<const uint4*>(st + (size_t)(grp + GV_GR * (m0 + u)) * row_bytes);
#pragma unroll
                            for (int j = 0; j < CA; ++j) wv[u][j] = wr[vbase + lane + 32 * j];
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < RU; ++u) {
                            // rows past this warp's last read its last row (in bounds) and are zeroed
                            const int iu = grp + GV_GR * min(m0 + u, nmine - 1);
                            const uint4* wr = reinterpret_cast<const uint4*>(st + (size_t)iu * row_bytes);
#pragma unroll
                            for (int j = 0; j < CA; ++j) {
                                const int v = min(vbase + lane + 32 * j, vbase + SWV - 1);
                                const uint4 t = wr[v];
                                wv[u][j] = (m0 + u < nmine && vbase + lane + 32 * j < vbase + SWV) ? t
                                                                                                     : make_uint4(0u, 0u, 0u, 0u);
                            }
                        }
                    }
                    float acc2[RU][NR];   // second chain: shorter dependency chains
#pragma unroll
                    for (int u = 0; u < RU; ++u)
#pragma unroll
                        for (int r = 0; r < NR; ++r) acc2[u][r] = 0.f;
#pragma unroll
                    for (int u = 0; u < RU; ++u)
#pragma unroll
                        for (int j = 0; j < CA; ++j) {
                            float wf[VEC];
                            Elem<WT>::unpack(wv[u][j], wf);
#pragma unroll
                            for (int r = 0; r < NR; ++r)
#pragma unroll
                                for (int e = 0; e < VEC; e += 2) {
                                    acc[u][r] = fmaf(wf[e], areg[r][j][e], acc[u][r]);
                                    acc2[u][r] = fmaf(wf[e + 1], areg[r][j][e + 1], acc2[u][r]);
                                }
                        }
#pragma unroll
                    for (int u = 0; u < RU; ++u)
#pragma unroll
                        for (int r = 0; r < NR; ++r) acc[u][r] += acc2[u][r];
                } else {
#pragma unroll
                    for (int u = 0; u < RU; ++u) {
                        if (m0 + u >= nmine) continue;
                        const uint4* wr = reinterpret_cast<const uint4*>(st + (size_t)(grp + GV_GR * (m0 + u)) * row_bytes);
                        for (int v = vbase + lane; v < vbase + SWV; v += 32) {
                            float wf[VEC];
                            Elem<WT>::unpack(wr[v], wf);
#pragma unroll
                            for (int r = 0; r < NR; ++r) {
                                const float* ar = act_s + (size_t)r * K + v * VEC;
#pragma unroll
                                for (int e = 0; e < VEC; ++e) acc[u][r] = fmaf(wf[e], ar[e], acc[u][r]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < RU; ++u) {
#pragma unroll
                for (int r = 0; r < NR; ++r) acc[u][r] = warp_sum(acc[u][r]);
                if (lane == 0 && m0 + u < nmine) {
#pragma unroll
                    for (int r = 0; r < NR; ++r) red_s[k & 1][grp + GV_GR * (m0 + u)][slice][r] = acc[u][r];
                }
            }
        }
        named_sync(1, GV_CT);   // every warp is done reading slot `slot`
        if (tid == 0 && !*abort_v && issued < nst) issue(issued++);
        if (warp == 0 && lane < nr && live) {
            const int row = a + lane;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= p.R) continue;
                float t = 0.f;
#pragma unroll
                for (int w = 0; w < GV_SL; ++w) t += red_s[k & 1][lane][w][r];
                float* o = p.out + (size_t)r * p.out_stride + row;
                if (EPI == EPI_ADD) {
                    *o = (res_local ? res_s[row - row0][r] : *o) + t;
                } else {
                    *o = t;
                }
                if (EPI == EPI_LOGITS) {
                    if (!isfinite(t)) nonfin = true;
                    const unsigned long long key = argmax_key(t, row);
                    best[r] = key > best[r] ? key : best[r];
                }
            }
        }
    }

    if (tid == 0) {
        // no copy may still be landing when the CTA exits (only after an abort
        // can an issued stage be unconsumed)
        for (int k = max(0, issued - S); k < issued; ++k)
            if (!mbar_wait(&full_bar[k % S], (k / S) & 1)) atomicOr(p.err, FAULT_WAIT);
        trace_mark(tr, p.trace_id, 2);
        trace_mark(tr, p.trace_id, 3);
    }
    if (EPI == EPI_LOGITS && warp == 0) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, best[r], o);
                best[r] = other > best[r] ? other : best[r];
            }
        }
        const bool any_nf = __any_sync(0xffffffffu, nonfin);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= p.R) continue;
                if (best[r]) atomicMax(p.amax + r, best[r]);
                if (any_nf) atomicOr(p.nonfinite + r, 1u);
            }
        }
    }
}

// ---------------- host side ----------------

template <typename WT, int NR, int CPL>
inline const void* gemv_pick_epi(int pro, int epi) {
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return (const void*)&k_gemv<WT, NR, PRO_RMSNORM, EPI_STORE, CPL>;
    if (pro == PRO_RMSNORM && epi == EPI_LOGITS) return (const void*)&k_gemv<WT, NR, PRO_RMSNORM, EPI_LOGITS, CPL>;
    if (pro == PRO_PLAIN && epi == EPI_ADD) return (const void*)&k_gemv<WT, NR, PRO_PLAIN, EPI_ADD, CPL>;
    if (pro == PRO_SWIGLU && epi == EPI_ADD) return (const void*)&k_gemv<WT, NR, PRO_SWIGLU, EPI_ADD, CPL>;
    return nullptr;
}

}  // namespace gd
