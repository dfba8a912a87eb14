// gemv_tc.cu -- tensor-core GEMV for 2..8 decode rows on sm_103a.
//
// With several decode rows every projection is a small dense contraction
// out[r, n] = sum_k W[n, k] a[r, k] over r < R <= 8.  A CUDA-core GEMV would
// have to keep R activation values per weight column on chip in fp32 and
// spend R FMAs per weight element; here the contraction runs on the tensor
// cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with the operands
// arranged so that no tensor-core row is wasted:
//   A (16 x 16) = the activations: rows 0..7 are the bf16 "hi" parts of the
//                 R decode rows, rows 8..15 the bf16 remainders a - hi ("lo"),
//                 so the products keep ~16 significant bits of the fp32
//                 activations (rows >= R are zero);
//   B (16 x 8)  = 8 weight rows x 16 columns, bf16 as stored;
//   D (16 x 8)  = fp32, out[r, n] = D[r, n] + D[r + 8, n].
// The reduction order inside a 16-column step is free, so a lane's A and B
// fragments use one and the same permutation of the columns: lane (g, t)
// supplies columns 8t..8t+7 and 32+8t..32+8t+7 of every 64-column box, which
// it reads as whole 16-byte vectors (no ldmatrix, no swizzled layout).
//
// Data movement (one CTA per SM, balanced contiguous row ranges):
//   * each CTA owns one row range and one range of K (K is split over
//     several CTAs only when the activations of the whole K do not fit in
//     shared memory); its activation rows arrive with one bulk copy per row
//     and stay resident; the compute warps convert them in place into bf16
//     hi/lo pairs in fragment order (gain applied) and take the sum of
//     squares in the same pass -- the RMSNorm scale 1/rms(x) is a per-row
//     factor and is applied to the dot products in the epilogue;
//   * the weights stream through a ring of stages of one 8-row tile x up to
//     2048 columns: a producer warp issues one bulk asynchronous copy
//     (cp.async.bulk, mbarrier completion) per weight row -- whole 2-4 KB row
//     pieces keep the copy engine's per-copy cost small -- and refills a slot
//     once the eight compute warps that took it have released it (one
//     "empty" mbarrier per slot); the weights do not depend on the previous
//     kernel, so the first stage is issued before the programmatic-launch
//     wait, the activations right after it;
//   * sixteen compute warps in two sets take alternate tiles; warp w of a set
//     takes the 64-column boxes w, w+8, ... of its stages and accumulates its
//     tiles of a row group (up to 8 tiles) in registers; at the end of the
//     group the eight box warps' partial tiles are added in warp order in
//     shared memory, followed by the epilogue (store, residual add, logits +
//     greedy argmax key, or SwiGLU of a gate/up pair);
//   * every shared-memory row (weight stage rows, activation rows) is padded
//     by 64 bytes, so even and odd rows start 16 banks apart and a warp's
//     16-byte fragment reads are conflict-free;
//   * with K split over ks CTAs, each writes its partial sums (and its part of
//     the sum of squares) to global scratch; the last of the ks CTAs to
//     arrive at the row range's counter adds them in split order and applies
//     the epilogue, then clears the counter for the next launch.
// Results do not depend on scheduling: every sum has a fixed order.
// Every mbarrier wait is bounded; a wait that gives up sets FAULT_WAIT in the
// error word, the CTA stops consuming and issuing, and the producer waits
// (bounded) for the copies in flight before it exits.
//
// The pages' composition: "Models, Registry and the Driver", section "Shared
// components" (x += mixer(norm(x)); x += ffn(norm(x)); final norm and head);
// "Architecture Overview", section "Automatic fusion" (RMSNorm and SwiGLU as
// fusable regions); "Backends", section "PTX (NVIDIA)" (tensor-core matmul
// through the mma instructions).
#include <stdlib.h>
#include "common.cuh"
#include "internal.h"
#include "mma_helpers.cuh"

namespace gd {

namespace {
constexpr int TC_BW = 8;                      // box warps: warp w takes boxes (w & 7) + 8i of a stage
constexpr int TC_CW = 2 * TC_BW;              // compute warps: two sets take alternate tiles
constexpr int TC_CT = TC_CW * 32;             // compute threads
constexpr int TC_THREADS = TC_CT + 32;        // + the producer warp
constexpr int TC_GT = 8;                      // tiles (8 weight rows each) per row group
constexpr int TC_PAD = 64;                    // bytes after every shared-memory row: even and odd
                                              // rows start 16 banks apart, so the fragment reads
                                              // of a warp never collide
constexpr int TC_MAX_S = 12;                  // ring stages at most
constexpr int TC_WS_MAX = 2048;               // weight columns per stage at most
constexpr int TC_WS_MIN = 1024;               // ... at least
constexpr int TC_ACT_BUDGET_DEFAULT = 64 * 1024;    // shared memory for the resident activations (leaves
                                                    // ~130 KB of ring; measured best of 32/64/128 KB)

// source of weight row n (an index into the stacked segments) at column k0
__device__ __forceinline__ const unsigned char* tc_row_src(const GemvParams& p, int n, int k0) {
    const int e0 = p.seg_rows[0], e1 = e0 + p.seg_rows[1];
    const void* w;
    int base;
    if (n < e0) { w = p.w[0]; base = 0; }
    else if (n < e1) { w = p.w[1]; base = e0; }
    else { w = p.w[2]; base = e1; }
    return reinterpret_cast<const unsigned char*>(w) + ((size_t)(n - base) * p.K + k0) * 2;
}

__device__ __forceinline__ uint4 lds_u4(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// acquire-ordered read of another CTA's partial sum (bypasses L1)
__device__ __forceinline__ float ld_part(const float* p) { return __ldcg(p); }
}  // namespace

// EPI_SWIGLU (paired mode): segments 0 and 1 are the gate and up matrices with
// the same row count F; out[r, n] = silu(gate_n . a_r) * (up_n . a_r), n < F.
template <int PRO, int EPI, int NBW>
__global__ void __launch_bounds__(TC_THREADS, 1) k_gemv_tc(const GemvParams p) {
    constexpr bool PAIRED = EPI == EPI_SWIGLU;
    constexpr bool RMS = PRO == PRO_RMSNORM;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[TC_MAX_S];
    __shared__ __align__(8) uint64_t empty_bar[TC_MAX_S];
    __shared__ __align__(8) uint64_t act_bar;
    __shared__ float ss_s[TC_CW][8];
    __shared__ float inv_s[8];
    __shared__ unsigned long long best_s[8];
    __shared__ unsigned nonfin_s;
    __shared__ int abort_s, last_s;
    volatile int* abort_v = &abort_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int WS = NBW * 64 * TC_BW;                   // weight columns per stage
    constexpr int WROW = WS * 2 + TC_PAD;                  // shared-memory pitch of a stage row
    const int R = p.R, S = p.stages, KS = p.tc_ks;
    const int TPG = PAIRED ? TC_GT / 2 : TC_GT;           // row tiles per group
    const int GRW = TPG * 8;                               // rows per group
    const int NU = PAIRED ? p.seg_rows[0] : p.N;          // rows the row ranges divide
    const int q = blockIdx.x % KS, ri = blockIdx.x / KS, nrr = gridDim.x / KS;
    const int KQ = p.K / KS, kq0 = q * KQ;                 // this CTA's K range
    const int row0 = (int)(((long long)ri * NU) / nrr);
    const int row1 = (int)(((long long)(ri + 1) * NU) / nrr);
    const int ngroups = (row1 - row0 + GRW - 1) / GRW;
    const int nwin = KQ / WS;
    const int nbx = KQ / 64;                               // 64-column boxes of the K range
    const size_t slot_bytes = (size_t)8 * WROW;
    const size_t arow = (size_t)KQ * 4 + TC_PAD;                            // pitch of an activation row
    unsigned char* ring = smem;
    unsigned char* act_s = smem + (size_t)S * slot_bytes;                   // [R][nbx][256 B] + pad per row
    float* red = reinterpret_cast<float*>(act_s + (size_t)R * arow);       // [8 box warps][TC_GT * 8][8]
    __nv_bfloat16* gain_s = reinterpret_cast<__nv_bfloat16*>(red + TC_BW * TC_GT * 8 * 8);   // [KQ] (RMSNorm)

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], TC_BW);   // the eight warps of the set that takes the stage
        }
        mbar_init(&act_bar, 1);
        abort_s = 0;
        nonfin_s = 0u;
        mbar_fence_init();
    }
    if (tid < 8) best_s[tid] = 0ull;
    __syncthreads();

    // ---------------- producer warp ----------------
    if (warp == TC_CW) {
        // stage s = (group, window, tile); the compute warps walk the same sequence
        auto issue = [&](int s, int& issued) -> bool {
                    int rem = s, gi = 0, ga = 0, nr = 0, nth = 0, ntl = 0;
            for (gi = 0; gi < ngroups; ++gi) {
                ga = row0 + gi * GRW;
                nr = min(GRW, row1 - ga);
                nth = (nr + 7) >> 3;
                ntl = PAIRED ? 2 * nth : nth;
                if (rem < nwin * ntl) break;
                rem -= nwin * ntl;
            }
            const int w = rem / ntl, jj = rem % ntl;
            const int half = (PAIRED && jj >= nth) ? 1 : 0;
            const int ta = ga + 8 * (jj - half * nth);    // first row of the tile
            const int tv = min(8, ga + nr - ta);           // valid rows of the tile
            const int k0 = kq0 + w * WS;
            int ok = 1;
            if (lane == 0) {
                if (*abort_v) {
                    ok = 0;
                } else if (s >= S && !mbar_wait(&empty_bar[s % S], ((s / S) - 1) & 1)) {
                    ok = 0;
                    *abort_v = 1;
                    atomicOr(p.err, FAULT_WAIT);
                } else {
                    mbar_arrive_expect_tx(&full_bar[s % S], (uint32_t)(tv * WS * 2));
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
            if (lane < tv) {
                const unsigned char* src =
                    PAIRED ? reinterpret_cast<const unsigned char*>(p.w[half]) + ((size_t)(ta + lane) * p.K + k0) * 2
                           : tc_row_src(p, ta + lane, k0);
                bulk_g2s(ring + (size_t)(s % S) * slot_bytes + (size_t)lane * WROW, src, (uint32_t)(WS * 2),
                         &full_bar[s % S]);
            }
            issued = s + 1;
            return true;
        };
        int nst = 0;
        for (int gi = 0; gi < ngroups; ++gi) {
            const int nr = min(GRW, row1 - (row0 + gi * GRW));
            nst += nwin * (PAIRED ? 2 : 1) * ((nr + 7) >> 3);
        }
        int issued = 0;
        bool go = true;
        // the first weight stage, then the activations (they come from the
        // previous kernel and gate every MMA), then the rest of the ring
        if (nst > 0) go = issue(0, issued);
        pdl_wait();
        if (lane == 0)
            mbar_arrive_expect_tx(&act_bar, (uint32_t)((size_t)R * KQ * 4 + (RMS ? (size_t)KQ * 2 : 0)));
        __syncwarp();
        if (lane < R)
            bulk_g2s(act_s + (size_t)lane * arow, p.act + (size_t)lane * p.act_stride + kq0, (uint32_t)(KQ * 4),
                     &act_bar);
        if (RMS && lane == 31)
            bulk_g2s(gain_s, reinterpret_cast<const __nv_bfloat16*>(p.gain) + kq0, (uint32_t)(KQ * 2), &act_bar);
        for (int s = 1; s < nst && go; ++s) go = issue(s, issued);
        // no copy may still be landing when the CTA exits (only after an abort
        // can an issued stage be unconsumed)
        if (lane == 0) {
            for (int s = max(0, issued - S); s < issued; ++s)
                if (!mbar_wait(&full_bar[s % S], (s / S) & 1)) atomicOr(p.err, FAULT_WAIT);
            if (!mbar_wait(&act_bar, 0)) atomicOr(p.err, FAULT_WAIT);
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
    const int g = lane >> 2, t = lane & 3;   // mma group (activation row / tile row), thread in group
    const int bw = warp & (TC_BW - 1), par = warp / TC_BW;   // box warp, tile parity

    // resident activations: box (r, b) holds 64 fp32 values as copied and is
    // rewritten in place as four 64-byte quads [hi cols 8t.. | hi cols 32+8t.. |
    // lo cols 8t.. | lo cols 32+8t..], each [t][8 x bf16]; lane l converts
    // columns 2l, 2l+1 of the box (conflict-free 8-byte reads, 4-byte writes)
    if (!*abort_v && !mbar_wait(&act_bar, 0)) {
        *abort_v = 1;
        atomicOr(p.err, FAULT_WAIT);
    }
    {
        const int c = 2 * lane, ch = c >> 3, e = c & 7;
        const int qoff = (ch >> 2) * 64 + (ch & 3) * 16 + e * 2;    // hi position; lo at +128
        float ss[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            ss[r] = 0.f;
            if (r < R) {   // warp-uniform (after a timeout the stale bytes are converted harmlessly)
                for (int b = warp; b < nbx; b += TC_CW) {
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
                    __syncwarp();   // the whole box is read before it is rewritten
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
        named_sync(1, TC_CT);
        if (tid < 8) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < TC_CW; ++w) tot += ss_s[w][tid];
            // the CTA's own sum of squares; with split K the last arriver adds the splits'
            inv_s[tid] = RMS ? 1.0f / sqrtf(tot / (float)p.K + p.eps) : 1.f;
            if (KS > 1 && RMS) p.tc_part[(size_t)KS * R * (PAIRED ? 2 * NU : NU) + ((size_t)q * nrr + ri) * 8 + tid] = tot;
        }
    }

    float acc[TC_GT / 2][4];   // the tiles of this warp's parity
#pragma unroll
    for (int j = 0; j < TC_GT / 2; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[j][x] = 0.f;
    unsigned long long best = 0ull;   // EPI_LOGITS: this thread's activation row is tid & 7
    bool nonfin = false;
    // per-lane bases: activation row g (zero rows past R), stage row g, thread-in-group column offset
    const unsigned char* abase = act_s + (size_t)(g < R ? g : 0) * arow + t * 16;
    const size_t wofs = (size_t)g * WROW + t * 16;
    const size_t np_stride = (size_t)(PAIRED ? 2 * NU : NU);   // partial sums per (split, activation row)

    // the epilogue of one output: v (and the up projection u when paired), unscaled
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

    int s = 0;
    for (int gi = 0; gi < ngroups; ++gi) {
        const int ga = row0 + gi * GRW, nr = min(GRW, row1 - ga);
        const int nth = (nr + 7) >> 3;
        const int ntl = PAIRED ? 2 * nth : nth;
        for (int w = 0; w < nwin; ++w) {
            const int bw0 = w * (WS / 64);   // first box of this window within the K range
#pragma unroll
            for (int jj = 0; jj < TC_GT; ++jj) {
                if (jj < ntl) {
                    const int slot = s % S;
                    if ((jj & 1) == par) {
                        if (!*abort_v && !mbar_wait(&full_bar[slot], (s / S) & 1)) {
                            *abort_v = 1;
                            atomicOr(p.err, FAULT_WAIT);
                        }
                        if (!*abort_v) {
                            const unsigned char* st = ring + (size_t)slot * slot_bytes + wofs;
#pragma unroll
                            for (int i = 0; i < NBW; ++i) {
                                const int bs = bw + TC_BW * i;   // box within the stage
                                const unsigned char* ab = abase + (size_t)(bw0 + bs) * 256;
                                uint4 q0 = lds_u4(ab), q1 = lds_u4(ab + 64), q2 = lds_u4(ab + 128), q3 = lds_u4(ab + 192);
                                if (g >= R) q0 = q1 = q2 = q3 = make_uint4(0u, 0u, 0u, 0u);
                                const uint4 w0 = lds_u4(st + bs * 128), w1 = lds_u4(st + bs * 128 + 64);
                                // q0/q1: hi of columns 8t.. / 32+8t..; q2/q3: lo of the same
                                const uint32_t a0[4] = {q0.x, q2.x, q0.y, q2.y};
                                const uint32_t a1[4] = {q0.z, q2.z, q0.w, q2.w};
                                const uint32_t a2[4] = {q1.x, q3.x, q1.y, q3.y};
                                const uint32_t a3[4] = {q1.z, q3.z, q1.w, q3.w};
                                mma_bf16(acc[jj >> 1], a0, w0.x, w0.y);
                                mma_bf16(acc[jj >> 1], a1, w0.z, w0.w);
                                mma_bf16(acc[jj >> 1], a2, w1.x, w1.y);
                                mma_bf16(acc[jj >> 1], a3, w1.z, w1.w);
                            }
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty_bar[slot]);   // this warp is done with the slot
                    }
                    ++s;
                }
            }
        }

        // row group done: the eight warps' partial tiles, added in warp order
        const bool live = !*abort_v;
        if (live) {
#pragma unroll
            for (int j2 = 0; j2 < TC_GT / 2; ++j2) {
                const int jj = 2 * j2 + par;
                if (jj < ntl) {
                    const int n0 = 8 * jj + 2 * t;
                    red[((size_t)bw * TC_GT * 8 + n0) * 8 + g] = acc[j2][0] + acc[j2][2];
                    red[((size_t)bw * TC_GT * 8 + n0 + 1) * 8 + g] = acc[j2][1] + acc[j2][3];
                }
            }
        }
#pragma unroll
        for (int j2 = 0; j2 < TC_GT / 2; ++j2)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[j2][x] = 0.f;
        named_sync(1, TC_CT);
        if (live) {
            const int r = tid & 7;
            for (int idx = tid; idx < nr * 8; idx += TC_CT) {
                const int n = idx >> 3;
                if (r >= R) continue;
                float v = 0.f, u = 0.f;
#pragma unroll
                for (int w = 0; w < TC_BW; ++w) v += red[((size_t)w * TC_GT * 8 + n) * 8 + r];
                if (PAIRED) {
#pragma unroll
                    for (int w = 0; w < TC_BW; ++w) u += red[((size_t)w * TC_GT * 8 + 8 * nth + n) * 8 + r];
                }
                if (KS == 1) {
                    finish(r, ga + n, v, u, inv_s[r]);
                } else {
                    float* pp = p.tc_part + ((size_t)q * R + r) * np_stride;
                    pp[ga + n] = v;
                    if (PAIRED) pp[NU + ga + n] = u;
                }
            }
        }
        named_sync(1, TC_CT);   // `red` is rewritten by the next group
    }

    // split K: the last CTA of the row range adds the splits in order
    if (KS > 1) {
        __threadfence();
        named_sync(1, TC_CT);
        if (tid == 0) last_s = atomicAdd(p.tc_cnt + ri, 1u) == (unsigned)(KS - 1) ? 1 : 0;
        named_sync(1, TC_CT);
        if (last_s && !*abort_v) {
            __threadfence();
            if (tid < 8) {
                float tot = 0.f;
                for (int x = 0; x < KS; ++x) tot += ld_part(p.tc_part + (size_t)KS * R * np_stride + ((size_t)x * nrr + ri) * 8 + tid);
                inv_s[tid] = RMS ? 1.0f / sqrtf(tot / (float)p.K + p.eps) : 1.f;
            }
            named_sync(1, TC_CT);
            const int r = tid & 7;
            for (int idx = tid; idx < (row1 - row0) * 8; idx += TC_CT) {
                const int n = row0 + (idx >> 3);
                if (r >= R) continue;
                float v = 0.f, u = 0.f;
                for (int x = 0; x < KS; ++x) {
                    const float* pp = p.tc_part + ((size_t)x * R + r) * np_stride;
                    v += ld_part(pp + n);
                    if (PAIRED) u += ld_part(pp + NU + n);
                }
                finish(r, n, v, u, inv_s[r]);
            }
            if (tid == 0) p.tc_cnt[ri] = 0u;   // ready for the next launch
        }
    }

    if (EPI == EPI_LOGITS) {
        const int r = tid & 7;
        if (r < R) {
            if (best) atomicMax(&best_s[r], best);
            if (nonfin) atomicOr(&nonfin_s, 1u << r);
        }
        named_sync(1, TC_CT);
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

template <int NBW>
const void* gemv_tc_pick(int pro, int epi) {
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_STORE, NBW>;
    if (pro == PRO_RMSNORM && epi == EPI_LOGITS) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_LOGITS, NBW>;
    if (pro == PRO_RMSNORM && epi == EPI_SWIGLU) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_SWIGLU, NBW>;
    if (pro == PRO_PLAIN && epi == EPI_ADD) return (const void*)&k_gemv_tc<PRO_PLAIN, EPI_ADD, NBW>;
    if (pro == PRO_PLAIN && epi == EPI_STORE) return (const void*)&k_gemv_tc<PRO_PLAIN, EPI_STORE, NBW>;
    return nullptr;
}

// the kernel for a plan: stage width 1024 (2 boxes per warp) or 2048 (4)
const void* gemv_tc_kernel(int pro, int epi, int ws) {
    return ws == 2048 ? gemv_tc_pick<4>(pro, epi) : ws == 1024 ? gemv_tc_pick<2>(pro, epi) : nullptr;
}

namespace {
// K splits: the fewest whose K range is a multiple of the stage width
// (>= 1024 columns) and whose activations fit the budget; 0 if none
int tc_splits(int R, int K, int budget) {
    for (int ks = 1; ks <= 64; ++ks) {
        if (K % ks) continue;
        const int kq = K / ks;
        if (kq % TC_WS_MIN) continue;
        if ((size_t)R * kq * 4 <= (size_t)budget) return ks;
    }
    return 0;
}
}  // namespace

size_t gemv_tc_part_floats(int R, int K, int N, bool paired) {
    // the need at the plan's resident activation budget
    const int ks = tc_splits(R, K, TC_ACT_BUDGET_DEFAULT);
    (void)paired;   // N already counts both halves of a gate/up pair
    return ks > 1 ? (size_t)ks * R * (size_t)N + (size_t)ks * GEMV_TC_CNT_WORDS * 8 : 0;
}

cudaError_t gemv_tc_plan(GemvPlan* plan, int num_sms) {
    GemvParams& p = plan->p;
    const bool paired = plan->epi == EPI_SWIGLU;
    if (plan->wtype != W_BF16) return cudaErrorInvalidValue;
    if (p.R < 1 || p.R > 8 || p.K <= 0 || p.K % TC_WS_MIN != 0 || p.N <= 0) return cudaErrorInvalidValue;
    if (paired && (p.seg_rows[0] != p.seg_rows[1] || p.seg_rows[2] != 0)) return cudaErrorInvalidValue;
    // 16-byte aligned sources: weight rows (K % 1024 == 0), activation rows, gains, segment bases
    if (p.act_stride % 4 != 0 || (reinterpret_cast<uintptr_t>(p.act) & 15u) != 0) return cudaErrorInvalidValue;
    for (int i = 0; i < 3; ++i)
        if (p.seg_rows[i] > 0 && (reinterpret_cast<uintptr_t>(p.w[i]) & 15u) != 0) return cudaErrorInvalidValue;
    if (plan->pro == PRO_RMSNORM && (!p.gain || (reinterpret_cast<uintptr_t>(p.gain) & 15u) != 0))
        return cudaErrorInvalidValue;
    const void* fn = gemv_tc_kernel(plan->pro, plan->epi, TC_WS_MAX);
    if (!fn) return cudaErrorInvalidValue;
    const int ks = tc_splits(p.R, p.K, TC_ACT_BUDGET_DEFAULT);
    if (ks < 1) return cudaErrorInvalidValue;
    const int kq = p.K / ks;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    const size_t avail = (size_t)optin - fa.sharedSizeBytes;
    const size_t fixed = (size_t)p.R * ((size_t)kq * 4 + TC_PAD) + (size_t)TC_BW * TC_GT * 8 * 8 * sizeof(float) +
                         (plan->pro == PRO_RMSNORM ? (size_t)kq * 2 : 0);
    if (fixed >= avail) return cudaErrorInvalidValue;
    // stage width: 2048 columns when at least 3 such stages fit, else 1024
    int ws = (kq % TC_WS_MAX == 0) ? TC_WS_MAX : TC_WS_MIN;
    auto slot_of = [](int w) { return (size_t)8 * ((size_t)w * 2 + TC_PAD); };
    int S = (int)((avail - fixed) / slot_of(ws));
    if (S < 3 && ws > TC_WS_MIN) {
        ws = TC_WS_MIN;
        S = (int)((avail - fixed) / slot_of(ws));
    }
    if (S > TC_MAX_S) S = TC_MAX_S;
    if (S < 2) return cudaErrorInvalidValue;
    const int nu = paired ? p.seg_rows[0] : p.N;
    int nrr = num_sms / ks;                      // row ranges
    if (nrr > nu) nrr = nu;
    if (nrr < 1 || (ks > 1 && nrr > (int)GEMV_TC_CNT_WORDS)) return cudaErrorInvalidValue;
    if (ks > 1 && (!p.tc_part || !p.tc_cnt ||
                   (size_t)ks * p.R * (size_t)p.N + (size_t)ks * nrr * 8 > p.tc_part_cap))
        return cudaErrorInvalidValue;
    fn = gemv_tc_kernel(plan->pro, plan->epi, ws);   // same static shared memory at either width
    p.rps = TC_GT;
    p.stages = S;
    p.tc_ws = ws;
    p.tc_ks = ks;
    plan->grid = nrr * ks;
    plan->block = TC_THREADS;
    plan->smem = (size_t)S * slot_of(ws) + fixed;
    plan->nr = 8;
    plan->cpl = 0;
    return raise_smem_cap(fn);
}

}  // namespace gd
