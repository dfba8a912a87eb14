// sample.cu -- the sampling suffix of the step beyond greedy: temperature,
// top-k, top-p, min-p with a counter-based uniform, and top-n logprobs
// ("Models, Registry and the Driver", section "The Driver": Head::Sample
// appends sampling to the decode graph -- greedy or temperature / top-k /
// top-p / min-p -- and can return top-n logprobs; "Execution", section "Per
// backend": the host reads back the token id).
//
// For row r (one CTA of 1024 threads per row), with l the row's logits:
//   1. candidates: the k tokens of largest logit, ties to the lower index
//      (k = top_k, raised to n_logprobs when more are asked for);
//      the k-th largest 32-bit order key is found by a 4-pass radix select
//      (8-bit histograms), the candidates are collected and sorted by
//      (logit desc, index asc) -- a bitonic sort of 1024 keys;
//   2. q_j = exp((l_j - l_max) / T) over the sorted candidates, S_j their
//      inclusive prefix sums (fixed-order block scan);
//   3. kept: the shortest prefix with S_j >= top_p * S_k, cut further to the
//      candidates with q_j >= min_p (q_1 = 1, so min_p is relative to the
//      largest probability);
//   4. u = the counter-based uniform of (seed, row, Pos[r]) (splitmix64 at
//      counter (row << 32 | pos), top 53 bits); the pick is the first kept
//      candidate with S_j > u * S_last (in double);
//   5. logprobs: l_j - l_max - log(sum over the whole vocabulary of
//      exp(l - l_max)) for the first n candidates.
// T = 0 picks the greedy id (the head's argmax key).  Every reduction has a
// fixed order, so a replay repeats the same pick.
#include <math.h>
#include "common.cuh"
#include "internal.h"

namespace gd {

namespace {
constexpr int SM_THREADS = 1024;
constexpr int SM_MAXK = 1024;

__device__ __forceinline__ unsigned order_key(float v) {
    const unsigned u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned ord) {
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
// splitmix64 output for stream position c of `seed` (Steele, Lea, Flood:
// state seed + (c + 1) * golden gamma, then the variant-13 finalizer)
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed, unsigned long long c) {
    unsigned long long z = seed + (c + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
// inclusive block scan of one float per thread, fixed order
__device__ float block_scan(float v, float* warp_s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_s[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = warp_s[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_s[lane] = w;
    }
    __syncthreads();
    const float before = warp > 0 ? warp_s[warp - 1] : 0.f;
    __syncthreads();
    return v + before;
}
__device__ int block_scan_int(int v, int* warp_s) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_s[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_s[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_s[lane] = w;
    }
    __syncthreads();
    const int before = warp > 0 ? warp_s[warp - 1] : 0;
    __syncthreads();
    return v + before;
}
}  // namespace

__global__ void __launch_bounds__(SM_THREADS) k_sample(const SampleParams p) {
    __shared__ unsigned hist[256];
    __shared__ unsigned long long cand[SM_MAXK];
    __shared__ float scan_s[32];
    __shared__ int iscan_s[32];
    __shared__ unsigned sel_s[3];      // prefix, keys above it, next free candidate slot
    __shared__ int pick_s[3];          // top-p cut, min-p cut
    __shared__ float red_s[32];
    const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const SamplerSlot cfg = *p.cfg;
    const float* l = p.logits + (size_t)r * p.V;
    const unsigned long long gkey = p.amax[r];
    const int greedy = gkey ? (int)(0xFFFFFFFFu - (unsigned)(gkey & 0xFFFFFFFFull)) : 0;
    const float lmax = key_value((unsigned)(gkey >> 32));
    const int nlp = min(max(cfg.n_logprobs, 0), DEC_LOGPROBS_MAX);
    const bool sampling = cfg.temperature > 0.f;
    if (!sampling && nlp == 0) {
        if (tid == 0) p.sampled[r] = greedy;
        return;
    }
    int k = sampling ? cfg.top_k : 1;
    k = max(k, nlp);
    k = min(max(k, 1), min(SM_MAXK, p.V));

    // ---- 1. the k-th largest order key: 4 radix passes of 8 bits ----
    unsigned prefix = 0u, mask = 0u;
    int need = k;           // candidates still to find at or below the prefix
    unsigned above = 0u;    // keys strictly above the final prefix
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += SM_THREADS) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < p.V; i += SM_THREADS) {
            const unsigned key = order_key(l[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0, b = 255;
            for (; b > 0; --b) {
                if (acc + (int)hist[b] >= need) break;
                acc += (int)hist[b];
            }
            sel_s[0] = prefix | ((unsigned)b << shift);
            sel_s[1] = (unsigned)acc;
        }
        __syncthreads();
        prefix = sel_s[0];
        need -= (int)sel_s[1];
        above += sel_s[1];
        mask |= 255u << shift;
        __syncthreads();
    }
    // `prefix` is the k-th largest key; `above` keys exceed it; take the first
    // `need` (>= 1) keys equal to it, in index order
    const unsigned tau = prefix;
    const int chunk = (p.V + SM_THREADS - 1) / SM_THREADS;
    const int c0 = min(tid * chunk, p.V), c1 = min(c0 + chunk, p.V);
    int eq = 0;
    for (int i = c0; i < c1; ++i) eq += order_key(l[i]) == tau;
    const int eq_before = block_scan_int(eq, iscan_s) - eq;
    for (int i = tid; i < SM_MAXK; i += SM_THREADS) cand[i] = 0ull;
    if (tid == 0) sel_s[2] = 0u;
    __syncthreads();
    int rank = eq_before;
    for (int i = c0; i < c1; ++i) {
        const unsigned key = order_key(l[i]);
        bool take = key > tau;
        if (key == tau) {
            take = rank < need;
            ++rank;
        }
        if (take) {
            const unsigned slot = atomicAdd(&sel_s[2], 1u);
            if (slot < (unsigned)SM_MAXK)
                cand[slot] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)i);
        }
    }
    __syncthreads();
    // bitonic sort, descending: (logit desc, index asc); empty slots (0) sink
    for (int size = 2; size <= SM_MAXK; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int i = tid, j = i ^ stride;
            if (j > i) {
                const bool desc = (i & size) == 0;
                const unsigned long long a = cand[i], b = cand[j];
                if (desc ? (a < b) : (a > b)) {
                    cand[i] = b;
                    cand[j] = a;
                }
            }
            __syncthreads();
        }
    }

    // ---- 2-4. weights, cuts, the pick ----
    const bool mine = tid < k;
    const int idx = mine ? (int)(0xFFFFFFFFu - (unsigned)(cand[tid] & 0xFFFFFFFFull)) : 0;
    const float lv = mine ? l[idx] : 0.f;
    int pick = greedy;
    if (sampling) {
        const float q = mine ? expf((lv - lmax) / cfg.temperature) : 0.f;
        const float S = block_scan(q, scan_s);
        __shared__ float S_s[SM_MAXK];
        S_s[tid] = S;
        if (tid == 0) {
            pick_s[0] = k - 1;
            pick_s[1] = 0;
        }
        __syncthreads();
        const float total = S_s[k - 1];
        const float target_p = (cfg.top_p < 1.f ? cfg.top_p : 1.f) * total;
        if (mine && S >= target_p && (tid == 0 || S_s[tid - 1] < target_p)) pick_s[0] = tid;
        const int nmin = __syncthreads_count(mine && q >= cfg.min_p);
        const int last = min(pick_s[0], max(nmin, 1) - 1);
        const unsigned long long z =
            splitmix64_at(cfg.seed, ((unsigned long long)r << 32) | (unsigned)p.pos[r]);
        const double u = (double)(z >> 11) * (1.0 / 9007199254740992.0);
        const double target = u * (double)S_s[last];
        if (tid == 0) pick_s[2] = last;
        __syncthreads();
        if (tid <= last && (double)S_s[tid] > target && (tid == 0 || (double)S_s[tid - 1] <= target)) pick_s[2] = tid;
        __syncthreads();
        pick = (int)(0xFFFFFFFFu - (unsigned)(cand[pick_s[2]] & 0xFFFFFFFFull));
    }
    if (tid == 0) p.sampled[r] = pick;

    // ---- 5. top-n logprobs of the whole distribution ----
    if (nlp > 0) {
        float z = 0.f;
        for (int i = tid; i < p.V; i += SM_THREADS) z += expf(l[i] - lmax);
        z = warp_sum(z);
        if (lane == 0) red_s[warp] = z;
        __syncthreads();
        if (warp == 0) {
            float t = red_s[lane];
            t = warp_sum(t);
            if (lane == 0) red_s[0] = logf(t);
        }
        __syncthreads();
        if (tid < nlp) {
            p.lp_ids[r * DEC_LOGPROBS_MAX + tid] = idx;
            p.lp_vals[r * DEC_LOGPROBS_MAX + tid] = (lv - lmax) - red_s[0];
        }
    }
}

cudaError_t sample_launch(const SampleParams& p, cudaStream_t s) {
    k_sample<<<p.R, SM_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gd
