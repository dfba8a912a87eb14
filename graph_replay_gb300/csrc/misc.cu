// misc.cu -- the step's first kernel (slot checks, per-step resets, embedding
// gather) and a self-limiting busy kernel used to exercise the bounded wait.
#include "common.cuh"
#include "internal.h"

namespace gd {

// First kernel of every step.  One CTA, so the resets it makes are ordered
// before its own checks, and every later kernel of the step runs after it.
//   * clears the error word, the argmax keys and the non-finite flags;
//   * checks Token[r] in [0, V) and Pos[r] in [0, cap), setting error bits
//     ("Execution", section "Failure handling": a failing kernel check sets a
//     bit in a reserved error word and the dispatch continues; the step's
//     result is then discarded) -- an out-of-range token reads row 0 instead;
//   * x[r, :] = E[Token[r], :] widened to fp32.
template <typename WT>
__global__ void __launch_bounds__(256) k_embed(const EmbedParams p) {
    const int tid = threadIdx.x;
    unsigned long long* tr = nullptr;   // trace buffer if tracing is on (thread 0)
    if (tid == 0) {
        tr = trace_if_on(p.trace);
        trace_mark(tr, p.trace_id, 0);
    }
    if (tid == 0) *p.err = 0u;
    if (tid < p.R) {
        p.amax[tid] = 0ull;
        p.nonfinite[tid] = 0u;
    }
    __syncthreads();
    const WT* E = reinterpret_cast<const WT*>(p.E);
    for (int r = 0; r < p.R; ++r) {
        int tok = p.tok[r];
        const int pos = p.pos[r];
        if (tok < 0 || tok >= p.V) {
            if (tid == 0) atomicOr(p.err, FAULT_TOKEN);
            tok = 0;
        }
        if ((pos < 0 || pos >= p.cap) && tid == 0) atomicOr(p.err, FAULT_POS);
        const WT* e = E + (size_t)tok * p.d;
        float* x = p.x + (size_t)r * p.d;
        // 16-byte loads, all in flight at once (d is a multiple of the vector width)
        constexpr int VEC = Elem<WT>::VEC;
        for (int i = tid * VEC; i < p.d; i += blockDim.x * VEC) {
            float f[VEC];
            Elem<WT>::unpack(*reinterpret_cast<const uint4*>(e + i), f);
#pragma unroll
            for (int q = 0; q < VEC; q += 4)
                *reinterpret_cast<float4*>(x + i + q) = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
        }
    }
    __syncthreads();
    if (tid == 0) {
        trace_mark(tr, p.trace_id, 1);
        trace_mark(tr, p.trace_id, 2);
        trace_mark(tr, p.trace_id, 3);
    }
}

cudaError_t embed_launch(int wtype, const EmbedParams& p, cudaStream_t s) {
    if (wtype == W_BF16)
        k_embed<__nv_bfloat16><<<1, 256, 0, s>>>(p);
    else
        k_embed<float><<<1, 256, 0, s>>>(p);
    return cudaGetLastError();
}

// Between two steps of a chain ("Models, Registry and the Driver", section
// "The Driver": RowWork::Chain -- with no guided row, the device feeds each
// pick to the next step and the host waits once).  One CTA of 32 threads,
// thread r < R for row r:
//   * keeps the step's error word in the chain's sticky word (the next step's
//     first kernel clears the error word);
//   * decodes the greedy key into the token id, records it and the non-finite
//     flag in the history at the chain's step counter;
//   * writes the slots of the next step: Token = the id, Pos += 1, and for
//     paged KV the WriteMap slot of the new position from the SlotMap (only
//     while Pos < cap; the host checks the chain stays below cap).
__global__ void __launch_bounds__(32) k_chain_advance(const ChainParams p) {
    const int r = threadIdx.x;
    const int i = *p.counter;
    if (r == 0) {
        const unsigned e = *p.err;
        if (e) atomicOr(p.chain_err, e);
    }
    if (r < p.R && i < p.max_steps) {
        const unsigned long long k = p.amax[r];
        int id = p.sampled ? p.sampled[r] : (k ? (int)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull)) : -1);
        if (id < 0 || id >= p.V) {
            atomicOr(p.chain_err, FAULT_TOKEN);
            id = 0;
        }
        p.ids[(size_t)i * p.R + r] = id;
        p.nf[(size_t)i * p.R + r] = p.nonfinite[r] ? 1 : 0;
        p.tok[r] = id;
        const int np = p.pos[r] + 1;
        p.pos[r] = np;
        if (p.slot_map && np < p.cap) p.wm[r] = p.slot_map[(size_t)r * p.ppr + np / p.page] * p.page + np % p.page;
    }
    __syncwarp();
    if (r == 0) *p.counter = i + 1;
}

cudaError_t chain_advance_launch(const ChainParams& p, cudaStream_t s) {
    k_chain_advance<<<1, 32, 0, s>>>(p);
    return cudaGetLastError();
}

// Spins on the global nanosecond timer for `ns`, with an iteration cap as a
// second bound, then returns: a kernel that is slow on purpose but always ends.
__global__ void k_busy(long long ns) {
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (long long it = 0; it < (1ll << 26); ++it) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if ((long long)(t - t0) >= ns) break;
        __nanosleep(1000);
    }
}

cudaError_t busy_launch(long long ns, cudaStream_t s) {
    k_busy<<<1, 32, 0, s>>>(ns);
    return cudaGetLastError();
}

}  // namespace gd
