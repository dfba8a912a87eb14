// gemv_tma.cu -- box-streamed tensor-core GEMV for 2..8 decode rows on sm_103a.
//
// Same contraction and operand arrangement as gemv_tc.cu (mma.sync m16n8k16;
// A = the decode rows' bf16 hi parts in rows 0..7 and bf16 remainders in rows
// 8..15, B = 8 weight rows; lane (g, t) supplies columns 8t..8t+7 and
// 32+8t..32+8t+7 of every 64-column box for both), with the weights moved by
// TMA tensor copies instead of one bulk copy per weight row:
//   * a stage is one 64-column x BH-row box of the CTA's weight rows (BH <=
//     256, up to 32 KB; gate/up: one box of each), copied by ONE
//     cp.async.bulk.tensor instruction with a 128-byte swizzle.  The copy
//     engine takes about 8 copy instructions per microsecond per SM; with
//     4 KB per instruction that capped the row-copy design near 30 GB/s per
//     SM, while 8-32 KB boxes stream at the HBM rate (a probe of this stream
//     alone: 5.5-6.3 TB/s);
//   * each of 16 compute warps owns up to 2 whole 8-row tiles of the group
//     for the CTA's whole K range, so the K sum of a tile never leaves the
//     warp: no cross-warp reduction and no CTA barrier per group; the
//     epilogue runs from registers;
//   * K is split over ks CTAs (each keeps the activations of its K range
//     resident, <= 64 KB) so that every CTA's row range fills a box; the
//     last CTA of a row range adds the splits in order (as in gemv_tc.cu);
//   * the activations arrive with one bulk copy per row and are converted in
//     place to hi/lo fragment order (RMSNorm gain applied, the 1/rms scale in
//     the epilogue), as in gemv_tc.cu.
// The weight reads of a tile row: chunk c of row r sits at 16-byte position
// c ^ (r & 7) of the row's 128 bytes; even rows read their chunk t first and
// odd rows chunk 4+t first, so a warp's 8-lane phases hit distinct banks.
// Every mbarrier wait is bounded; a wait that gives up sets FAULT_WAIT.
//
// The pages' composition: "Models, Registry and the Driver", section "Shared
// components"; "Architecture Overview", section "Automatic fusion";
// "Backends", section "PTX (NVIDIA)" (tensor-core matmul).
#include <cuda.h>
#include <stdlib.h>
#include "common.cuh"
#include "internal.h"
#include "mma_helpers.cuh"

namespace gd {

namespace {
constexpr int BX_CW = 16;                        // compute warps
constexpr int BX_CT = BX_CW * 32;
constexpr int BX_THREADS = BX_CT + 32;           // + the producer warp
constexpr int BX_TPW = 2;                        // tiles per warp per row group
constexpr int BX_MAX_BH = BX_CW * BX_TPW * 8;    // rows per box at most (256)
constexpr int BX_MAX_S = 12;                     // ring stages at most
constexpr int BX_PAD = 64;                       // bytes after every activation row
constexpr int BX_ACT_BUDGET = 64 * 1024;         // resident activations per CTA

struct BoxArgs {
    CUtensorMap map[3];   // per weight segment: bf16 [rows, K], boxes [64 columns x BH rows], 128-byte swizzle
    GemvParams p;
};

__device__ __forceinline__ uint4 lds_u4(const void* q) { return *reinterpret_cast<const uint4*>(q); }
__device__ __forceinline__ uint4 selu4(bool c, const uint4& x, const uint4& y) {
    return make_uint4(c ? x.x : y.x, c ? x.y : y.y, c ? x.z : y.z, c ? x.w : y.w);
}
__device__ __forceinline__ float ld_part(const float* q) { return __ldcg(q); }
}  // namespace

template <int PRO, int EPI>
__global__ void __launch_bounds__(BX_THREADS, 1) k_gemv_box(const __grid_constant__ BoxArgs args) {
    constexpr bool PAIRED = EPI == EPI_SWIGLU;
    constexpr bool RMS = PRO == PRO_RMSNORM;
    const GemvParams& p = args.p;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full_bar[BX_MAX_S];
    __shared__ __align__(8) uint64_t empty_bar[BX_MAX_S];
    __shared__ __align__(8) uint64_t act_bar;
    __shared__ float ss_s[BX_CW][8];
    __shared__ float inv_s[8];
    __shared__ unsigned long long best_s[8];
    __shared__ unsigned nonfin_s;
    __shared__ int abort_s, last_s;
    volatile int* abort_v = &abort_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, S = p.stages, KS = p.tc_ks, BH = p.tc_bh;
    const int q = blockIdx.x % KS, ri = blockIdx.x / KS, nrr = gridDim.x / KS;
    const int KQ = p.K / KS, kq0 = q * KQ, nkb = KQ / 64;
    // this CTA's row range: segment `seg` (gate rows when paired), range li of it
    int seg = 0, li = ri;
    if (!PAIRED) {
        while (seg < 2 && li >= p.tc_seg_ranges[seg]) {
            li -= p.tc_seg_ranges[seg];
            ++seg;
        }
    }
    const int nsr = PAIRED ? nrr : p.tc_seg_ranges[seg];
    const int Ns = p.seg_rows[seg];
    int seg_base = 0;
    if (!PAIRED)
        for (int i = 0; i < seg; ++i) seg_base += p.seg_rows[i];
    const int ra = (int)(((long long)li * Ns) / nsr), rb = (int)(((long long)(li + 1) * Ns) / nsr);
    const int ngroups = (rb - ra + BH - 1) / BH;
    const int nst = ngroups * nkb;
    const size_t box_bytes = (size_t)BH * 128;
    const size_t slot_bytes = box_bytes * (PAIRED ? 2 : 1);
    const size_t arow = (size_t)KQ * 4 + BX_PAD;
    unsigned char* ring = smem;
    unsigned char* act_s = ring + (size_t)S * slot_bytes;                                      // [R][arow]
    __nv_bfloat16* gain_s = reinterpret_cast<__nv_bfloat16*>(act_s + (size_t)R * arow);      // [KQ] (RMSNorm)

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], BX_CW);
        }
        mbar_init(&act_bar, 1);
        abort_s = 0;
        nonfin_s = 0u;
        mbar_fence_init();
    }
    if (tid < 8) best_s[tid] = 0ull;
    __syncthreads();

    // ---------------- producer (one lane) ----------------
    if (warp == BX_CW) {
        if (lane == 0) {
            const CUtensorMap* m0 = &args.map[PAIRED ? 0 : seg];
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                if (*abort_v) break;
                if (s >= S && !mbar_wait(&empty_bar[s % S], ((s / S) - 1) & 1)) {
                    *abort_v = 1;
                    atomicOr(p.err, FAULT_WAIT);
                    break;
                }
                const int y = ra + (s / nkb) * BH, x = kq0 + (s % nkb) * 64;
                unsigned char* dst = ring + (size_t)(s % S) * slot_bytes;
                mbar_arrive_expect_tx(&full_bar[s % S], (uint32_t)slot_bytes);
                tma_load_2d(dst, m0, x, y, &full_bar[s % S]);
                if (PAIRED) tma_load_2d(dst + box_bytes, &args.map[1], x, y, &full_bar[s % S]);
                issued = s + 1;
                if (s == 0) {
                    // the activations come from the previous kernel: after its completion
                    pdl_wait();
                    mbar_arrive_expect_tx(&act_bar, (uint32_t)((size_t)R * KQ * 4 + (RMS ? (size_t)KQ * 2 : 0)));
                    for (int r = 0; r < R; ++r)
                        bulk_g2s(act_s + (size_t)r * arow, p.act + (size_t)r * p.act_stride + kq0, (uint32_t)(KQ * 4),
                                 &act_bar);
                    if (RMS)
                        bulk_g2s(gain_s, reinterpret_cast<const __nv_bfloat16*>(p.gain) + kq0, (uint32_t)(KQ * 2),
                                 &act_bar);
                }
            }
            // no copy may still be landing when the CTA exits
            for (int s = max(0, issued - S); s < issued; ++s)
                if (!mbar_wait(&full_bar[s % S], (s / S) & 1)) atomicOr(p.err, FAULT_WAIT);
            if (issued > 0 && !mbar_wait(&act_bar, 0)) atomicOr(p.err, FAULT_WAIT);
        }
        return;
    }

    // ---------------- compute warps ----------------
    unsigned long long* tr = nullptr;
    if (tid == 0) {
        tr = trace_if_on(p.trace);
        trace_mark(tr, p.trace_id, 0);
    }
    pdl_wait();
    if (tid == 0) trace_mark(tr, p.trace_id, 1);
    pdl_trigger();
    const int g = lane >> 2, t = lane & 3;
    const bool odd = (g & 1) != 0;

    // resident activations, converted in place (as in gemv_tc.cu)
    if (!*abort_v && !mbar_wait(&act_bar, 0)) {
        *abort_v = 1;
        atomicOr(p.err, FAULT_WAIT);
    }
    {
        const int nbx = KQ / 64;
        const int c = 2 * lane, ch = c >> 3, e = c & 7;
        const int qoff = (ch >> 2) * 64 + (ch & 3) * 16 + e * 2;
        float ss[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            ss[r] = 0.f;
            if (r < R) {
                for (int b = warp; b < nbx; b += BX_CW) {
                    unsigned char* box = act_s + (size_t)r * arow + (size_t)b * 256;
                    const float2 x = *reinterpret_cast<const float2*>(box + c * 4);
                    ss[r] = fmaf(x.x, x.x, ss[r]);
                    ss[r] = fmaf(x.y, x.y, ss[r]);
                    float v0 = x.x, v1 = x.y;
                    if (RMS) {
                        const uint32_t gw = *reinterpret_cast<const uint32_t*>(gain_s + b * 64 + c);
                        v0 *= bf16_lo(gw);
                        v1 *= bf16_hi(gw);
                    }
                    const uint32_t hi = pack_bf16x2(v0, v1);
                    const uint32_t lo = pack_bf16x2(v0 - bf16_lo(hi), v1 - bf16_hi(hi));
                    __syncwarp();
                    *reinterpret_cast<uint32_t*>(box + qoff) = hi;
                    *reinterpret_cast<uint32_t*>(box + 128 + qoff) = lo;
                    __syncwarp();
                }
            }
            ss[r] = warp_sum(ss[r]);
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < 8; ++r) ss_s[warp][r] = ss[r];
        }
        named_sync(1, BX_CT);
        if (tid < 8) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < BX_CW; ++w) tot += ss_s[w][tid];
            inv_s[tid] = RMS ? 1.0f / sqrtf(tot / (float)p.K + p.eps) : 1.f;
            if (KS > 1 && RMS) p.tc_part[(size_t)KS * R * (PAIRED ? 2 * Ns : p.N) + ((size_t)q * nrr + ri) * 8 + tid] = tot;
        }
        named_sync(1, BX_CT);
    }

    const size_t np_stride = (size_t)(PAIRED ? 2 * Ns : p.N);
    unsigned long long best = 0ull;   // EPI_LOGITS: this lane's activation row is g
    bool nonfin = false;
    auto finish = [&](int r, int n, float v, float u, float iv) {
        float* o = p.out + (size_t)r * p.out_stride + n;
        v *= iv;
        if (PAIRED) {
            u *= iv;
            *o = v / (1.0f + expf(-v)) * u;
        } else if (EPI == EPI_ADD) {
            *o += v;
        } else {
            *o = v;
        }
        if (EPI == EPI_LOGITS) {
            if (!isfinite(v)) nonfin = true;
            const unsigned long long key = argmax_key(v, n);
            best = key > best ? key : best;
        }
    };

    const unsigned char* abase = act_s + (size_t)(g < R ? g : 0) * arow + t * 16;
    // byte offsets of chunk t and chunk 4+t in a swizzled 128-byte row of residue g
    const int cpos_t = ((t ^ g) & 7) * 16, cpos_4t = (((4 + t) ^ g) & 7) * 16;
    const int first = odd ? cpos_4t : cpos_t, second = odd ? cpos_t : cpos_4t;
    int s = 0;
    for (int gi = 0; gi < ngroups; ++gi) {
        const int ga = ra + gi * BH, nr = min(BH, rb - ga);
        const int T = (nr + 7) >> 3;
        float acc[BX_TPW][4], accu[BX_TPW][4];
#pragma unroll
        for (int i = 0; i < BX_TPW; ++i)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[i][x] = accu[i][x] = 0.f;
        for (int kb = 0; kb < nkb; ++kb, ++s) {
            const int slot = s % S;
            if (!*abort_v && !mbar_wait(&full_bar[slot], (s / S) & 1)) {
                *abort_v = 1;
                atomicOr(p.err, FAULT_WAIT);
            }
            if (!*abort_v && warp < T) {
                const unsigned char* ab = abase + (size_t)kb * 256;
                uint4 q0 = lds_u4(ab), q1 = lds_u4(ab + 64), q2 = lds_u4(ab + 128), q3 = lds_u4(ab + 192);
                if (g >= R) q0 = q1 = q2 = q3 = make_uint4(0u, 0u, 0u, 0u);
                const uint32_t a0[4] = {q0.x, q2.x, q0.y, q2.y};
                const uint32_t a1[4] = {q0.z, q2.z, q0.w, q2.w};
                const uint32_t a2[4] = {q1.x, q3.x, q1.y, q3.y};
                const uint32_t a3[4] = {q1.z, q3.z, q1.w, q3.w};
                const unsigned char* box = ring + (size_t)slot * slot_bytes;
#pragma unroll
                for (int i = 0; i < BX_TPW; ++i) {
                    const int tile = warp + BX_CW * i;
                    if (tile < T) {
                        const unsigned char* rowp = box + (size_t)(8 * tile + g) * 128;
                        const uint4 u0 = lds_u4(rowp + first), u1 = lds_u4(rowp + second);
                        const uint4 w0 = selu4(odd, u1, u0), w1 = selu4(odd, u0, u1);   // chunk t, chunk 4+t
                        mma_bf16(acc[i], a0, w0.x, w0.y);
                        mma_bf16(acc[i], a1, w0.z, w0.w);
                        mma_bf16(acc[i], a2, w1.x, w1.y);
                        mma_bf16(acc[i], a3, w1.z, w1.w);
                        if (PAIRED) {
                            const unsigned char* rowu = rowp + box_bytes;
                            const uint4 v0 = lds_u4(rowu + first), v1 = lds_u4(rowu + second);
                            const uint4 x0 = selu4(odd, v1, v0), x1 = selu4(odd, v0, v1);
                            mma_bf16(accu[i], a0, x0.x, x0.y);
                            mma_bf16(accu[i], a1, x0.z, x0.w);
                            mma_bf16(accu[i], a2, x1.x, x1.y);
                            mma_bf16(accu[i], a3, x1.z, x1.w);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
        }
        // the group's tiles are complete in this warp's registers
        if (!*abort_v && g < R) {
#pragma unroll
            for (int i = 0; i < BX_TPW; ++i) {
                const int tile = warp + BX_CW * i;
                if (tile >= T) continue;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int nl = ga + 8 * tile + 2 * t + c;   // row within the segment
                    if (nl >= rb) continue;
                    const float v = acc[i][c] + acc[i][c + 2];
                    const float u = PAIRED ? accu[i][c] + accu[i][c + 2] : 0.f;
                    if (KS == 1) {
                        finish(g, seg_base + nl, v, u, inv_s[g]);
                    } else {
                        float* pp = p.tc_part + ((size_t)q * R + g) * np_stride;
                        pp[seg_base + nl] = v;
                        if (PAIRED) pp[Ns + nl] = u;
                    }
                }
            }
        }
    }

    // split K: the last CTA of the row range adds the splits in order
    if (KS > 1) {
        __threadfence();
        named_sync(1, BX_CT);
        if (tid == 0) last_s = atomicAdd(p.tc_cnt + ri, 1u) == (unsigned)(KS - 1) ? 1 : 0;
        named_sync(1, BX_CT);
        if (last_s && !*abort_v) {
            __threadfence();
            if (tid < 8) {
                float tot = 0.f;
                for (int x = 0; x < KS; ++x)
                    tot += ld_part(p.tc_part + (size_t)KS * R * np_stride + ((size_t)x * nrr + ri) * 8 + tid);
                inv_s[tid] = RMS ? 1.0f / sqrtf(tot / (float)p.K + p.eps) : 1.f;
            }
            named_sync(1, BX_CT);
            const int r = tid & 7;
            for (int idx = tid; idx < (rb - ra) * 8; idx += BX_CT) {
                const int nl = ra + (idx >> 3);
                if (r >= R) continue;
                float v = 0.f, u = 0.f;
                for (int x = 0; x < KS; ++x) {
                    const float* pp = p.tc_part + ((size_t)x * R + r) * np_stride;
                    v += ld_part(pp + seg_base + nl);
                    if (PAIRED) u += ld_part(pp + Ns + nl);
                }
                // LOGITS keys of the final pass are per thread row r
                float* o = p.out + (size_t)r * p.out_stride + seg_base + nl;
                const float iv = inv_s[r];
                const float vv = v * iv;
                if (PAIRED) {
                    *o = vv / (1.0f + expf(-vv)) * (u * iv);
                } else if (EPI == EPI_ADD) {
                    *o += vv;
                } else {
                    *o = vv;
                }
                if (EPI == EPI_LOGITS) {
                    if (!isfinite(vv)) atomicOr(&nonfin_s, 1u << r);
                    atomicMax(&best_s[r], argmax_key(vv, seg_base + nl));
                }
            }
            if (tid == 0) p.tc_cnt[ri] = 0u;   // ready for the next launch
        }
    }

    if (EPI == EPI_LOGITS) {
        if (g < R) {
            if (best) atomicMax(&best_s[g], best);
            if (nonfin) atomicOr(&nonfin_s, 1u << g);
        }
        named_sync(1, BX_CT);
        if (tid < R) {
            if (best_s[tid]) atomicMax(p.amax + tid, best_s[tid]);
            if ((nonfin_s >> tid) & 1u) atomicOr(p.nonfinite + tid, 1u);
        }
    }
    if (tid == 0) {
        trace_mark(tr, p.trace_id, 2);
        trace_mark(tr, p.trace_id, 3);
    }
}

// ---------------- host side ----------------

namespace {
const void* box_kernel(int pro, int epi) {
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return (const void*)&k_gemv_box<PRO_RMSNORM, EPI_STORE>;
    if (pro == PRO_RMSNORM && epi == EPI_LOGITS) return (const void*)&k_gemv_box<PRO_RMSNORM, EPI_LOGITS>;
    if (pro == PRO_RMSNORM && epi == EPI_SWIGLU) return (const void*)&k_gemv_box<PRO_RMSNORM, EPI_SWIGLU>;
    if (pro == PRO_PLAIN && epi == EPI_ADD) return (const void*)&k_gemv_box<PRO_PLAIN, EPI_ADD>;
    if (pro == PRO_PLAIN && epi == EPI_STORE) return (const void*)&k_gemv_box<PRO_PLAIN, EPI_STORE>;
    return nullptr;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}
}  // namespace

// the kernel of a box-streamed plan (nullptr: none for this prologue/epilogue)
const void* gemv_box_kernel(int pro, int epi) { return box_kernel(pro, epi); }

constexpr int BX_MAX_KS = 16;

// scratch for the split partials: room for every split count up to 16 MiB,
// and at least for two splits (the planner skips counts that do not fit)
size_t gemv_box_part_floats(int R, int K, int N) {
    constexpr size_t CAP = (size_t)4 << 20;   // floats
    size_t most = 0, two = 0;
    for (int ks = 2; ks <= BX_MAX_KS; ++ks) {
        if (K % ks || (K / ks) % 64) continue;
        const size_t need = (size_t)ks * R * (size_t)N + (size_t)ks * GEMV_TC_CNT_WORDS * 8;
        if (!two) two = need;
        if (need <= CAP && need > most) most = need;
    }
    return most > two ? most : two;
}

cudaError_t gemv_box_plan(GemvPlan* plan, int num_sms) {
    GemvParams& p = plan->p;
    const bool paired = plan->epi == EPI_SWIGLU;
    if (plan->wtype != W_BF16) return cudaErrorInvalidValue;
    if (p.R < 1 || p.R > 8 || p.K <= 0 || p.K % 64 != 0 || p.N <= 0) return cudaErrorInvalidValue;
    if (paired && (p.seg_rows[0] != p.seg_rows[1] || p.seg_rows[2] != 0)) return cudaErrorInvalidValue;
    if (p.act_stride % 4 != 0 || (reinterpret_cast<uintptr_t>(p.act) & 15u) != 0) return cudaErrorInvalidValue;
    for (int i = 0; i < 3; ++i)
        if (p.seg_rows[i] > 0 && (reinterpret_cast<uintptr_t>(p.w[i]) & 15u) != 0) return cudaErrorInvalidValue;
    if (plan->pro == PRO_RMSNORM && (!p.gain || (reinterpret_cast<uintptr_t>(p.gain) & 15u) != 0))
        return cudaErrorInvalidValue;
    const void* fn = box_kernel(plan->pro, plan->epi);
    EncodeTiledFn enc = encode_fn();
    if (!fn || !enc) return cudaErrorInvalidValue;
    const int nseg = paired ? 1 : (p.seg_rows[2] > 0 ? 3 : (p.seg_rows[1] > 0 ? 2 : 1));
    const int NU = paired ? p.seg_rows[0] : p.N;

    // K splits and row ranges: the fewest weight elements per CTA (box rows incl.
    // the over-fetch of the last box x the K range) plus a start-up cost
    int best_ks = 0, best_bh = 0, best_ranges[3] = {0, 0, 0};
    double best_cost = 0.0;
    for (int ks = 1; ks <= BX_MAX_KS; ++ks) {
        if (p.K % ks || (p.K / ks) % 64) continue;
        const int kq = p.K / ks;
        if ((size_t)p.R * kq * 4 > (size_t)BX_ACT_BUDGET) continue;
        const int nrr = num_sms / ks;
        if (nrr < nseg || (ks > 1 && nrr > (int)GEMV_TC_CNT_WORDS)) continue;
        // the split partials and sums of squares must fit the scratch
        if (ks > 1 && (size_t)ks * p.R * (size_t)p.N + (size_t)ks * nrr * 8 > p.tc_part_cap) continue;
        int ranges[3] = {0, 0, 0};
        if (paired) {
            ranges[0] = nrr < NU ? nrr : NU;
        } else {
            // ranges per segment in proportion to its rows, at least one each
            int used = 0;
            for (int i = 0; i < nseg; ++i) {
                ranges[i] = (int)((long long)nrr * p.seg_rows[i] / p.N);
                if (ranges[i] < 1) ranges[i] = 1;
                if (ranges[i] > p.seg_rows[i]) ranges[i] = p.seg_rows[i];
                used += ranges[i];
            }
            while (used > nrr) {   // give back from the segment with the fewest rows per range
                int j = -1;
                for (int i = 0; i < nseg; ++i)
                    if (ranges[i] > 1 && (j < 0 || (double)p.seg_rows[i] / ranges[i] < (double)p.seg_rows[j] / ranges[j]))
                        j = i;
                if (j < 0) break;
                --ranges[j];
                --used;
            }
            while (used < nrr) {   // add to the segment with the most rows per range
                int j = 0;
                for (int i = 1; i < nseg; ++i)
                    if ((double)p.seg_rows[i] / ranges[i] > (double)p.seg_rows[j] / ranges[j]) j = i;
                if (ranges[j] >= p.seg_rows[j]) break;
                ++ranges[j];
                ++used;
            }
        }
        int maxrows = 0;
        for (int i = 0; i < nseg; ++i)
            if (ranges[i] > 0) {
                const int rr = (p.seg_rows[i] + ranges[i] - 1) / ranges[i];
                maxrows = rr > maxrows ? rr : maxrows;
            }
        const int groups = (maxrows + BX_MAX_BH - 1) / BX_MAX_BH;
        const int bh = ((maxrows + groups - 1) / groups + 7) / 8 * 8;
        // bytes-equivalent time of one CTA: every stage costs at least ~6 KB (the
        // copy engine's instruction rate), the last CTA of a row range reads the
        // splits' partial sums, and a fixed start-up (activation copy, ring fill)
        const double stage = (double)bh * 128 * (paired ? 2 : 1);
        const double cost = (double)groups * (kq / 64) * (stage > 6144.0 ? stage : 6144.0) +
                            (ks > 1 ? (double)ks * p.R * maxrows * 4 * (paired ? 2 : 1) : 0.0) + 65536.0;
        if (best_ks == 0 || cost < best_cost) {
            best_cost = cost;
            best_ks = ks;
            best_bh = bh;
            for (int i = 0; i < 3; ++i) best_ranges[i] = ranges[i];
        }
    }
    if (!best_ks) return cudaErrorInvalidValue;
    const int ks = best_ks, kq = p.K / ks, bh = best_bh;
    int nrr = 0;
    for (int i = 0; i < 3; ++i) nrr += best_ranges[i];
    if (ks > 1 && (!p.tc_part || !p.tc_cnt)) return cudaErrorInvalidValue;

    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    const size_t avail = (size_t)optin - fa.sharedSizeBytes;
    const size_t fixed = (size_t)p.R * ((size_t)kq * 4 + BX_PAD) + (plan->pro == PRO_RMSNORM ? (size_t)kq * 2 : 0) +
                         1024;   // + the 1 KB alignment of the swizzled boxes
    const size_t slot = (size_t)bh * 128 * (paired ? 2 : 1);
    if (fixed >= avail) return cudaErrorInvalidValue;
    int S = (int)((avail - fixed) / slot);
    if (S > BX_MAX_S) S = BX_MAX_S;
    if (S < 2) return cudaErrorInvalidValue;

    // one tensor map per weight segment: [rows, K] bf16, boxes of 64 columns x bh rows
    CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(plan->tma_maps);
    const int nmaps = paired ? 2 : nseg;
    for (int i = 0; i < nmaps; ++i) {
        cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)p.seg_rows[i]};
        cuuint64_t strides[1] = {(cuuint64_t)p.K * 2};
        cuuint32_t box[2] = {64u, (cuuint32_t)bh};
        cuuint32_t estr[2] = {1u, 1u};
        if (enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.w[i]), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    p.stages = S;
    p.tc_ks = ks;
    p.tc_bh = bh;
    for (int i = 0; i < 3; ++i) p.tc_seg_ranges[i] = best_ranges[i];
    plan->grid = nrr * ks;
    plan->block = BX_THREADS;
    plan->smem = (size_t)S * slot + fixed;
    plan->nr = 8;
    plan->cpl = 0;
    return raise_smem_cap(fn);
}

cudaError_t gemv_box_launch(const GemvPlan& plan, cudaStream_t s, bool pdl) {
    const void* fn = box_kernel(plan.pro, plan.epi);
    if (!fn) return cudaErrorInvalidValue;
    alignas(64) BoxArgs a;
    memcpy(a.map, plan.tma_maps, sizeof(a.map));
    a.p = plan.p;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.block);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* kargs[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, kargs);
}

}  // namespace gd
