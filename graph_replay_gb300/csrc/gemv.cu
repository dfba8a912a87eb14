// gemv.cu -- fused (RMSNorm | SwiGLU) + GEMV + (store | residual add | logits
// + greedy argmax) for small-batch decode on sm_103a, CUDA cores.
//
// Decode at 1..4 rows is a matrix-vector product per weight matrix: every
// weight byte is read once per step and used for R multiply-adds, so the
// kernel is bound by HBM bandwidth.  Design:
//   * each CTA owns a contiguous range of output rows (a contiguous byte range
//     of each weight segment); the grid is sized to the GPU's resident CTA
//     slots so every SM streams;
//   * the activation rows are built once per CTA in shared memory by the
//     prologue (RMSNorm with gain, SwiGLU, or a plain copy) -- the norm of the
//     residual is recomputed per CTA from L2 instead of taking a kernel;
//   * one warp per output row; each lane streams 16-byte vectors with
//     no-L1-allocate loads, U vectors in flight, fp32 FMA, then a warp
//     shuffle reduction;
//   * before waiting on the producing kernel (programmatic dependent launch)
//     each CTA bulk-prefetches the start of its weight range into L2, since
//     the weights do not depend on the previous kernel.
// The pages' composition: "Models, Registry and the Driver", section "Shared
// components" (x += mixer(norm(x)); x += ffn(norm(x)); final norm and head);
// "Architecture Overview", section "Automatic fusion" (RMSNorm and SwiGLU as
// fusable regions).  The greedy pick is the sampling suffix of "Execution"
// and "Models, Registry and the Driver" (section "The Driver": the host reads
// back a token id and a non-finite flag).
#include "common.cuh"
#include "internal.h"

namespace gd {

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;
constexpr int GEMV_U = 8;          // 16-byte vectors in flight per lane
constexpr unsigned PREFETCH_BYTES = 32768;

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

template <typename WT, int NR, int PRO, int EPI>
__global__ void __launch_bounds__(GEMV_THREADS) k_gemv(const GemvParams p) {
    extern __shared__ float4 smem_f4[];
    float* act_s = reinterpret_cast<float*>(smem_f4);   // [NR][K]
    __shared__ float red_s[GEMV_WARPS][NR];
    __shared__ float inv_s[NR];
    __shared__ unsigned long long key_s[GEMV_WARPS][NR];
    __shared__ unsigned nf_s;

    constexpr int VEC = Elem<WT>::VEC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K;
    const int row0 = blockIdx.x * p.rows_per_cta;
    const int row1 = min(row0 + p.rows_per_cta, p.N);

    // locate the weight bytes of this CTA's first rows and prefetch them into L2
    if (tid == 0 && row0 < row1) {
        int base, nseg;
        const void* wseg = segment_of(p, row0, base, nseg);
        const char* w = reinterpret_cast<const char*>(wseg) + (size_t)(row0 - base) * K * sizeof(WT);
        size_t seg_left = (size_t)(base + nseg - row0) * K * sizeof(WT);
        size_t want = (size_t)(row1 - row0) * K * sizeof(WT);
        size_t bytes = min(min(seg_left, want), (size_t)PREFETCH_BYTES);
        bytes &= ~(size_t)15;
        if (bytes) prefetch_l2_bulk(w, (unsigned)bytes);
    }
    if (tid == 0) nf_s = 0u;

    pdl_wait();

    // ---------------- prologue: activation rows in shared memory ----------------
    if (PRO == PRO_RMSNORM) {
        float ss[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            ss[r] = 0.f;
            if (r < p.R) {
                const float* a = p.act + (size_t)r * p.act_stride;
                for (int k = tid; k < K; k += GEMV_THREADS) ss[r] = fmaf(a[k], a[k], ss[r]);
            }
            ss[r] = warp_sum(ss[r]);
        }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) red_s[warp][r] = ss[r];
        }
        __syncthreads();
        if (tid < NR) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < GEMV_WARPS; ++w) t += red_s[w][tid];
            inv_s[tid] = 1.0f / sqrtf(t / (float)K + p.eps);
        }
        __syncthreads();
        const WT* g = reinterpret_cast<const WT*>(p.gain);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float* a = p.act + (size_t)r * p.act_stride;
            const float inv = inv_s[r];
            for (int k = tid; k < K; k += GEMV_THREADS)
                act_s[r * K + k] = (r < p.R) ? a[k] * inv * Elem<WT>::load1(g + k) : 0.f;
        }
    } else if (PRO == PRO_SWIGLU) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float* a = p.act + (size_t)r * p.act_stride;
            for (int k = tid; k < K; k += GEMV_THREADS) {
                float v = 0.f;
                if (r < p.R) {
                    float gt = a[k], up = a[K + k];
                    v = gt / (1.0f + expf(-gt)) * up;
                }
                act_s[r * K + k] = v;
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float* a = p.act + (size_t)r * p.act_stride;
            for (int k = tid; k < K; k += GEMV_THREADS) act_s[r * K + k] = (r < p.R) ? a[k] : 0.f;
        }
    }
    __syncthreads();
    pdl_trigger();

    // ---------------- main loop: one warp per output row ----------------
    unsigned long long best[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) best[r] = 0ull;
    bool nonfinite = false;

    const int KV = K / VEC;   // 16-byte vectors per row
    for (int row = row0 + warp; row < row1; row += GEMV_WARPS) {
        int base, nseg;
        const void* wseg = segment_of(p, row, base, nseg);
        const uint4* wv = reinterpret_cast<const uint4*>(reinterpret_cast<const WT*>(wseg) + (size_t)(row - base) * K);
        float acc[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = 0.f;

        for (int vb = 0; vb < KV; vb += 32 * GEMV_U) {
            uint4 w[GEMV_U];
#pragma unroll
            for (int u = 0; u < GEMV_U; ++u) {
                const int idx = vb + u * 32 + lane;
                w[u] = idx < KV ? ld_stream16(wv + idx) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < GEMV_U; ++u) {
                const int idx = vb + u * 32 + lane;
                if (idx < KV) {
                    float wf[VEC];
                    Elem<WT>::unpack(w[u], wf);
                    const float* a = act_s + idx * VEC;
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
#pragma unroll
                        for (int e = 0; e < VEC; e += 4) {
                            const float4 av = *reinterpret_cast<const float4*>(a + r * K + e);
                            acc[r] = fmaf(wf[e + 0], av.x, acc[r]);
                            acc[r] = fmaf(wf[e + 1], av.y, acc[r]);
                            acc[r] = fmaf(wf[e + 2], av.z, acc[r]);
                            acc[r] = fmaf(wf[e + 3], av.w, acc[r]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = warp_sum(acc[r]);

        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= p.R) continue;
                float* o = p.out + (size_t)r * p.out_stride + row;
                if (EPI == EPI_ADD) {
                    *o += acc[r];
                } else {
                    *o = acc[r];
                }
                if (EPI == EPI_LOGITS) {
                    if (!isfinite(acc[r])) nonfinite = true;
                    const unsigned long long k = argmax_key(acc[r], row);
                    if (k > best[r]) best[r] = k;
                }
            }
        }
    }

    if (EPI == EPI_LOGITS) {
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r) key_s[warp][r] = best[r];
            if (nonfinite) atomicOr(&nf_s, 1u);
        }
        __syncthreads();
        if (tid < NR && tid < p.R) {
            unsigned long long b = 0ull;
#pragma unroll
            for (int w = 0; w < GEMV_WARPS; ++w) b = key_s[w][tid] > b ? key_s[w][tid] : b;
            if (b) atomicMax(p.amax + tid, b);
            if (nf_s) atomicOr(p.nonfinite + tid, 1u);
        }
    }
}

// ---------------- host side ----------------

template <typename WT, int NR, int PRO, int EPI>
static const void* kernel_ptr() {
    return reinterpret_cast<const void*>(&k_gemv<WT, NR, PRO, EPI>);
}

template <typename WT, int NR>
static const void* pick_epi(int pro, int epi) {
    if (pro == PRO_RMSNORM && epi == EPI_STORE) return kernel_ptr<WT, NR, PRO_RMSNORM, EPI_STORE>();
    if (pro == PRO_RMSNORM && epi == EPI_LOGITS) return kernel_ptr<WT, NR, PRO_RMSNORM, EPI_LOGITS>();
    if (pro == PRO_PLAIN && epi == EPI_ADD) return kernel_ptr<WT, NR, PRO_PLAIN, EPI_ADD>();
    if (pro == PRO_SWIGLU && epi == EPI_ADD) return kernel_ptr<WT, NR, PRO_SWIGLU, EPI_ADD>();
    if (pro == PRO_PLAIN && epi == EPI_STORE) return kernel_ptr<WT, NR, PRO_PLAIN, EPI_STORE>();
    return nullptr;
}

static const void* pick(int wtype, int nr, int pro, int epi) {
    if (wtype == W_BF16) {
        if (nr == 1) return pick_epi<__nv_bfloat16, 1>(pro, epi);
        if (nr == 4) return pick_epi<__nv_bfloat16, 4>(pro, epi);
        if (nr == 8) return pick_epi<__nv_bfloat16, 8>(pro, epi);
    } else {
        if (nr == 1) return pick_epi<float, 1>(pro, epi);
        if (nr == 4) return pick_epi<float, 4>(pro, epi);
        if (nr == 8) return pick_epi<float, 8>(pro, epi);
    }
    return nullptr;
}

cudaError_t gemv_plan(GemvPlan* plan, int num_sms) {
    GemvParams& p = plan->p;
    const int vec = plan->wtype == W_BF16 ? 8 : 4;
    if (p.K <= 0 || p.N <= 0 || p.K % vec != 0 || p.R < 1 || p.R > 8) return cudaErrorInvalidValue;
    plan->nr = p.R == 1 ? 1 : (p.R <= 4 ? 4 : 8);
    const void* fn = pick(plan->wtype, plan->nr, plan->pro, plan->epi);
    if (!fn) return cudaErrorInvalidValue;
    plan->block = GEMV_THREADS;
    plan->smem = (size_t)plan->nr * p.K * sizeof(float);
    if (plan->smem > 220 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = raise_smem_cap(fn);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, GEMV_THREADS, plan->smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > 4) per_sm = 4;
    const int slots = per_sm * num_sms;
    int rpc = (p.N + slots - 1) / slots;
    if (rpc < 1) rpc = 1;
    p.rows_per_cta = rpc;
    plan->grid = (p.N + rpc - 1) / rpc;
    return cudaSuccess;
}

cudaError_t gemv_launch(const GemvPlan& plan, cudaStream_t s, bool pdl) {
    const void* fn = pick(plan.wtype, plan.nr, plan.pro, plan.epi);
    if (!fn) return cudaErrorInvalidValue;
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
    void* args[] = {const_cast<GemvParams*>(&plan.p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gd
