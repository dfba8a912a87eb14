// gemv_tc.cu -- tensor-core GEMV for 2..8 decode rows on sm_103a.
//
// With several decode rows every projection is a small dense contraction
// out[r, n] = sum_k W[n, k] a[r, k] over r < R <= 8.  A CUDA-core GEMV would
// have to keep R activation values per weight column on chip (R x K fp32:
// 458 KB for the 8B-shape down projection at R = 8), so this kernel runs the
// contraction on the tensor cores instead (mma.sync m16n8k16, bf16 in, fp32
// accumulate) with the operands arranged so that nothing is wasted:
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
//   * a stage is (up to 64 weight rows) x 256 columns plus the matching 256
//     columns of the R activation rows; a producer warp fills a ring of stages
//     with bulk asynchronous copies (cp.async.bulk, one 512-byte piece per
//     weight row, mbarrier completion), and refills a slot once all eight
//     compute warps have released it (one "empty" mbarrier per slot);
//   * the weight copies of the first ring fill are issued before the
//     programmatic-launch wait (weights do not depend on the previous kernel);
//     the activation copies after it;
//   * compute warp w takes the 64-column box (w & 3) of every stage for the
//     tiles of parity (w >> 2); it builds its A fragments once per stage
//     (RMSNorm scale and gain applied in registers) and reuses them for every
//     tile;
//   * the four boxes' partial tiles are added in fixed order in shared memory
//     at the end of each row group, followed by the epilogue (store, residual
//     add, logits + greedy argmax key, or SwiGLU of a gate/up pair).
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
constexpr int TC_WK = 256;                    // weight columns per stage
constexpr int TC_ROWB = TC_WK * 2;            // bytes of one weight-row piece
constexpr int TC_ACTB = TC_WK * 4;            // bytes of one activation-row piece
constexpr int TC_ACT_SLOT = 8 * TC_ACTB;      // activation bytes per slot (8 rows reserved)
constexpr int TC_CW = 8;                      // compute warps: 4 boxes x 2 tile parities
constexpr int TC_CT = TC_CW * 32;             // compute threads
constexpr int TC_THREADS = TC_CT + 32;        // + the producer warp
constexpr int TC_MAX_SR = 64;                 // weight rows per stage at most
constexpr int TC_MAX_TW = TC_MAX_SR / 8 / 2;  // tiles per compute warp per stage at most
constexpr int TC_MAX_S = 8;                   // ring stages at most
constexpr int TC_RING_DEFAULT = 96 * 1024;    // ring bytes (leaves room for the next kernel's CTA)

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

__device__ __forceinline__ float4 lds_f4(const void* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ uint4 lds_u4(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ float4 sel4(bool c, const float4& a, const float4& b) {
    return make_float4(c ? a.x : b.x, c ? a.y : b.y, c ? a.z : b.z, c ? a.w : b.w);
}
__device__ __forceinline__ uint4 selu4(bool c, const uint4& a, const uint4& b) {
    return make_uint4(c ? a.x : b.x, c ? a.y : b.y, c ? a.z : b.z, c ? a.w : b.w);
}
}  // namespace

// EPI_SWIGLU (paired mode): segments 0 and 1 are the gate and up matrices with
// the same row count F; out[r, n] = silu(gate_n . a_r) * (up_n . a_r), n < F.
template <int PRO, int EPI>
__global__ void __launch_bounds__(TC_THREADS, 2) k_gemv_tc(const GemvParams p) {
    constexpr bool PAIRED = EPI == EPI_SWIGLU;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[TC_MAX_S];
    __shared__ __align__(8) uint64_t empty_bar[TC_MAX_S];
    __shared__ float nrm_s[TC_CW][8];
    __shared__ unsigned long long best_s[8];
    __shared__ unsigned nonfin_s;
    __shared__ int abort_s;
    volatile int* abort_v = &abort_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, R = p.R, S = p.stages, GRW = p.rps;
    const int SR = PAIRED ? 2 * GRW : GRW;              // weight rows of a full stage
    const int NU = PAIRED ? p.seg_rows[0] : p.N;        // rows the CTAs divide
    const int row0 = (int)(((long long)blockIdx.x * NU) / gridDim.x);
    const int row1 = (int)(((long long)(blockIdx.x + 1) * NU) / gridDim.x);
    const int NW = K / TC_WK;
    const int ngroups = (row1 - row0 + GRW - 1) / GRW;
    const int nst = ngroups * NW;
    const size_t slot_bytes = (size_t)SR * TC_ROWB + TC_ACT_SLOT;
    unsigned char* ring = smem;
    float* red = reinterpret_cast<float*>(smem + (size_t)S * slot_bytes);   // [4 boxes][SR][8]

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], TC_CW);
        }
        abort_s = 0;
        nonfin_s = 0u;
        mbar_fence_init();
    }
    if (tid < 8) best_s[tid] = 0ull;
    __syncthreads();

    // ---------------- producer warp ----------------
    if (warp == TC_CW) {
        auto stage_of = [&](int s, int& ga, int& nr, int& k0) {
            ga = row0 + (s / NW) * GRW;
            nr = min(GRW, row1 - ga);
            k0 = (s % NW) * TC_WK;
        };
        auto expect = [&](int s) {
            int ga, nr, k0;
            stage_of(s, ga, nr, k0);
            const uint32_t bytes = (uint32_t)((PAIRED ? 2 : 1) * nr * TC_ROWB + R * TC_ACTB);
            if (lane == 0) mbar_arrive_expect_tx(&full_bar[s % S], bytes);
            __syncwarp();
        };
        auto copy_w = [&](int s) {
            int ga, nr, k0;
            stage_of(s, ga, nr, k0);
            unsigned char* dst = ring + (size_t)(s % S) * slot_bytes;
            const int total = (PAIRED ? 2 : 1) * nr;
            for (int i = lane; i < total; i += 32) {
                const int half = (PAIRED && i >= nr) ? 1 : 0;
                const int rr = i - half * nr;
                const unsigned char* src =
                    PAIRED ? reinterpret_cast<const unsigned char*>(p.w[half]) + ((size_t)(ga + rr) * K + k0) * 2
                           : tc_row_src(p, ga + rr, k0);
                bulk_g2s(dst + (size_t)(half * GRW + rr) * TC_ROWB, src, TC_ROWB, &full_bar[s % S]);
            }
        };
        auto copy_a = [&](int s) {
            int ga, nr, k0;
            stage_of(s, ga, nr, k0);
            unsigned char* dst = ring + (size_t)(s % S) * slot_bytes + (size_t)SR * TC_ROWB;
            for (int r = lane; r < R; r += 32)
                bulk_g2s(dst + r * TC_ACTB, p.act + (size_t)r * p.act_stride + k0, TC_ACTB, &full_bar[s % S]);
        };
        const int pre = min(S, nst);
        for (int s = 0; s < pre; ++s) {
            expect(s);
            copy_w(s);
        }
        pdl_wait();   // the activations come from the previous kernel
        for (int s = 0; s < pre; ++s) copy_a(s);
        int issued = pre;
        for (int s = pre; s < nst; ++s) {
            int ok = 1;
            if (lane == 0) {
                if (*abort_v) {
                    ok = 0;
                } else if (!mbar_wait(&empty_bar[s % S], ((s / S) - 1) & 1)) {
                    ok = 0;
                    *abort_v = 1;
                    atomicOr(p.err, FAULT_WAIT);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            expect(s);
            copy_w(s);
            copy_a(s);
            issued = s + 1;
        }
        // no copy may still be landing when the CTA exits (only after an abort
        // can an issued stage be unconsumed)
        if (lane == 0)
            for (int s = max(0, issued - S); s < issued; ++s)
                if (!mbar_wait(&full_bar[s % S], (s / S) & 1)) atomicOr(p.err, FAULT_WAIT);
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
    const int g = lane >> 2, t = lane & 3;   // mma group (activation row / weight row of a tile), thread in group
    const int box = warp & 3, par = warp >> 2;
    const bool odd = (g & 1) != 0;           // odd rows take their two 16-byte halves in the other order

    float inv = 1.f;   // RMSNorm scale of activation row g
    if (PRO == PRO_RMSNORM) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float ss = 0.f;
            if (r < R) {
                const float* a = p.act + (size_t)r * p.act_stride;
                for (int k = tid * 4; k < K; k += TC_CT * 4) {
                    const float4 x = *reinterpret_cast<const float4*>(a + k);
                    ss = fmaf(x.x, x.x, ss);
                    ss = fmaf(x.y, x.y, ss);
                    ss = fmaf(x.z, x.z, ss);
                    ss = fmaf(x.w, x.w, ss);
                }
            }
            ss = warp_sum(ss);
            if (lane == 0) nrm_s[warp][r] = ss;
        }
        named_sync(1, TC_CT);
        if (g < R) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < TC_CW; ++w) tot += nrm_s[w][g];
            inv = 1.0f / sqrtf(tot / (float)K + p.eps);
        }
    }
    pdl_trigger();

    const __nv_bfloat16* gain = reinterpret_cast<const __nv_bfloat16*>(p.gain);
    float acc[TC_MAX_TW][4];
#pragma unroll
    for (int j = 0; j < TC_MAX_TW; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
    unsigned long long best = 0ull;   // EPI_LOGITS: this thread's activation row is tid & 7
    bool nonfin = false;

    for (int s = 0; s < nst; ++s) {
        const int slot = s % S;
        const int grp = s / NW, win = s % NW;
        const int ga = row0 + grp * GRW, nr = min(GRW, row1 - ga);
        const int nt = (nr + 7) >> 3;                  // tiles per half
        const int ntile = PAIRED ? 2 * nt : nt;
        if (!*abort_v && !mbar_wait(&full_bar[slot], (s / S) & 1)) {
            *abort_v = 1;
            atomicOr(p.err, FAULT_WAIT);
        }
        const bool live = !*abort_v;
        const unsigned char* st = ring + (size_t)slot * slot_bytes;
        if (live) {
            // A fragments of this warp's box: activation row g, chunks t and 4+t
            // (columns 8t..8t+7 and 32+8t..32+8t+7 of the box)
            float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0, q2 = q0, q3 = q0;
            if (g < R) {
                const unsigned char* ar = st + (size_t)SR * TC_ROWB + g * TC_ACTB + box * 256 + t * 32;
                // even rows: (t, lo half), (t, hi half), (4+t, lo), (4+t, hi); odd rows the reverse
                const float4 v0 = lds_f4(ar + (odd ? 144 : 0));
                const float4 v1 = lds_f4(ar + (odd ? 128 : 16));
                const float4 v2 = lds_f4(ar + (odd ? 16 : 128));
                const float4 v3 = lds_f4(ar + (odd ? 0 : 144));
                q0 = sel4(odd, v3, v0);
                q1 = sel4(odd, v2, v1);
                q2 = sel4(odd, v1, v2);
                q3 = sel4(odd, v0, v3);
                if (PRO == PRO_RMSNORM) {
                    const int kb = win * TC_WK + box * 64 + t * 8;
                    float gl[8], gh[8];
                    Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4*>(gain + kb)), gl);
                    Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4*>(gain + kb + 32)), gh);
                    q0 = make_float4(q0.x * inv * gl[0], q0.y * inv * gl[1], q0.z * inv * gl[2], q0.w * inv * gl[3]);
                    q1 = make_float4(q1.x * inv * gl[4], q1.y * inv * gl[5], q1.z * inv * gl[6], q1.w * inv * gl[7]);
                    q2 = make_float4(q2.x * inv * gh[0], q2.y * inv * gh[1], q2.z * inv * gh[2], q2.w * inv * gh[3]);
                    q3 = make_float4(q3.x * inv * gh[4], q3.y * inv * gh[5], q3.z * inv * gh[6], q3.w * inv * gh[7]);
                }
            }
            // k-step ks uses 4 consecutive values: ks 0 -> q0, 1 -> q1, 2 -> q2, 3 -> q3
            uint32_t a[4][4];
            auto frag = [&](const float4& v, uint32_t (&f)[4]) {
                const uint32_t h01 = pack_bf16x2(v.x, v.y), h23 = pack_bf16x2(v.z, v.w);
                f[0] = h01;
                f[2] = h23;
                f[1] = pack_bf16x2(v.x - bf16_lo(h01), v.y - bf16_hi(h01));
                f[3] = pack_bf16x2(v.z - bf16_lo(h23), v.w - bf16_hi(h23));
            };
            frag(q0, a[0]);
            frag(q1, a[1]);
            frag(q2, a[2]);
            frag(q3, a[3]);
#pragma unroll
            for (int jj = 0; jj < TC_MAX_TW; ++jj) {
                const int j = par + 2 * jj;
                if (j < ntile) {
                    const int srow = (PAIRED && j >= nt) ? GRW + 8 * (j - nt) + g : 8 * j + g;
                    const unsigned char* wr = st + (size_t)srow * TC_ROWB + box * 128 + t * 16;
                    const uint4 u0 = lds_u4(wr + (odd ? 64 : 0));
                    const uint4 u1 = lds_u4(wr + (odd ? 0 : 64));
                    const uint4 w0 = selu4(odd, u1, u0), w1 = selu4(odd, u0, u1);   // chunk t, chunk 4+t
                    mma_bf16(acc[jj], a[0], w0.x, w0.y);
                    mma_bf16(acc[jj], a[1], w0.z, w0.w);
                    mma_bf16(acc[jj], a[2], w1.x, w1.y);
                    mma_bf16(acc[jj], a[3], w1.z, w1.w);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);   // this warp is done with the slot

        if (win == NW - 1) {
            // row group done: the four boxes' partial tiles, added in box order
            if (live) {
#pragma unroll
                for (int jj = 0; jj < TC_MAX_TW; ++jj) {
                    const int j = par + 2 * jj;
                    if (j < ntile) {
                        const int n0 = ((PAIRED && j >= nt) ? GRW + 8 * (j - nt) : 8 * j) + 2 * t;
                        red[((size_t)box * SR + n0) * 8 + g] = acc[jj][0] + acc[jj][2];
                        red[((size_t)box * SR + n0 + 1) * 8 + g] = acc[jj][1] + acc[jj][3];
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < TC_MAX_TW; ++jj)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[jj][q] = 0.f;
            named_sync(1, TC_CT);
            if (live) {
                const int r = tid & 7;
                for (int idx = tid; idx < nr * 8; idx += TC_CT) {
                    const int n = idx >> 3;
                    if (r >= R) continue;
                    float v = red[((size_t)0 * SR + n) * 8 + r];
                    v += red[((size_t)1 * SR + n) * 8 + r];
                    v += red[((size_t)2 * SR + n) * 8 + r];
                    v += red[((size_t)3 * SR + n) * 8 + r];
                    float* o = p.out + (size_t)r * p.out_stride + ga + n;
                    if (PAIRED) {
                        float u = red[((size_t)0 * SR + GRW + n) * 8 + r];
                        u += red[((size_t)1 * SR + GRW + n) * 8 + r];
                        u += red[((size_t)2 * SR + GRW + n) * 8 + r];
                        u += red[((size_t)3 * SR + GRW + n) * 8 + r];
                        *o = v / (1.0f + expf(-v)) * u;
                    } else if (EPI == EPI_ADD) {
                        *o += v;
                    } else {
                        *o = v;
                    }
                    if (EPI == EPI_LOGITS) {
                        if (!isfinite(v)) nonfin = true;
                        const unsigned long long key = argmax_key(v, ga + n);
                        best = key > best ? key : best;
                    }
                }
            }
            named_sync(1, TC_CT);   // `red` is rewritten by the next group
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

const void* gemv_tc_kernel(int pro, int epi) {
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_STORE>;
    if (pro == PRO_RMSNORM && epi == EPI_LOGITS) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_LOGITS>;
    if (pro == PRO_RMSNORM && epi == EPI_SWIGLU) return (const void*)&k_gemv_tc<PRO_RMSNORM, EPI_SWIGLU>;
    if (pro == PRO_PLAIN && epi == EPI_ADD) return (const void*)&k_gemv_tc<PRO_PLAIN, EPI_ADD>;
    if (pro == PRO_PLAIN && epi == EPI_STORE) return (const void*)&k_gemv_tc<PRO_PLAIN, EPI_STORE>;
    return nullptr;
}

cudaError_t gemv_tc_plan(GemvPlan* plan, int num_sms) {
    GemvParams& p = plan->p;
    const bool paired = plan->epi == EPI_SWIGLU;
    if (plan->wtype != W_BF16) return cudaErrorInvalidValue;
    if (p.R < 1 || p.R > 8 || p.K <= 0 || p.K % TC_WK != 0 || p.N <= 0) return cudaErrorInvalidValue;
    if (paired && (p.seg_rows[0] != p.seg_rows[1] || p.seg_rows[2] != 0)) return cudaErrorInvalidValue;
    // 16-byte aligned sources for every bulk copy: weight rows (K % 256 == 0),
    // activation rows, and the segment bases
    if (p.act_stride % 4 != 0 || (reinterpret_cast<uintptr_t>(p.act) & 15u) != 0) return cudaErrorInvalidValue;
    for (int i = 0; i < 3; ++i)
        if (p.seg_rows[i] > 0 && (reinterpret_cast<uintptr_t>(p.w[i]) & 15u) != 0) return cudaErrorInvalidValue;
    if (p.gain && (reinterpret_cast<uintptr_t>(p.gain) & 15u) != 0) return cudaErrorInvalidValue;
    const void* fn = gemv_tc_kernel(plan->pro, plan->epi);
    if (!fn) return cudaErrorInvalidValue;
    const int nu = paired ? p.seg_rows[0] : p.N;
    const int grid = nu < num_sms ? nu : num_sms;
    const int per_cta = (nu + grid - 1) / grid;
    const int max_grw = paired ? TC_MAX_SR / 2 : TC_MAX_SR;
    int grw = (per_cta + 7) / 8 * 8;
    if (grw > max_grw) grw = max_grw;
    const int sr = paired ? 2 * grw : grw;
    const size_t slot = (size_t)sr * TC_ROWB + TC_ACT_SLOT;
    size_t ring = TC_RING_DEFAULT;
    if (const char* env = getenv("GRAPHDEC_TC_RING")) {   // ring bytes per CTA (tuning)
        const long v = atol(env);
        if (v >= 32768 && v <= 220 * 1024) ring = (size_t)v;
    }
    int S = (int)(ring / slot);
    if (S > TC_MAX_S) S = TC_MAX_S;
    if (S < 2) S = 2;
    const size_t red = (size_t)4 * sr * 8 * sizeof(float);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    while (S > 2 && (size_t)S * slot + red > (size_t)optin - fa.sharedSizeBytes) --S;
    if ((size_t)S * slot + red > (size_t)optin - fa.sharedSizeBytes) return cudaErrorInvalidValue;
    p.rps = grw;
    p.stages = S;
    plan->grid = grid;
    plan->block = TC_THREADS;
    plan->smem = (size_t)S * slot + red;
    plan->nr = 8;
    plan->cpl = 0;
    return raise_smem_cap(fn);
}

}  // namespace gd
