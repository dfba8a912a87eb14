// pf_gemm.cuh -- the prefill projections on the 5th-generation tensor cores
// (tcgen05.mma, sm_103a): out[t, n] = sum_k W[n, k] * h[t, k] for the tokens
// of a pass (blocks of PF_T), W bf16 row-major [N, K] (nn.Linear layout), h fp32.
//
// A prefill step is a dense contraction: at 128 tokens every weight byte feeds
// 256 multiply-adds ("Models, Registry and the Driver", "The Model": a step
// shape is rows x new tokens).  The activations enter as two bf16 rows per
// token, hi = bf16(h) and lo = bf16(h - hi), so the product keeps about 16
// significant bits of h with fp32 accumulation; the weights are exact in bf16.
//
// One CTA computes a 128-row tile of W against one block of PF_T tokens over
// one K split (up to three weight segments, e.g. Wq | Wk | Wv, share one launch
// and one output row space).  The token blocks are the grid's fastest index, so
// the CTAs that share a weight tile run together and read it from HBM once.
// A = the W tile [128 x 64] and B = the block's activations [2 PF_T x 64] (hi
// rows, then lo rows) are staged by TMA (128-byte swizzle) in a ring of
// PF_STAGES; one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32)
// into a TMEM accumulator of 128 lanes x 2 PF_T columns; each MMA group's
// commit frees its ring stage.  The epilogue (all four warps, warp w reads TMEM
// lanes 32w..32w+31) adds the hi and lo columns and, by the launch's mode,
// stores the split's partial sums part[split][t][n] (the caller adds the
// splits in split order), adds the sums to the residual rows x[t][n] (one
// split), or -- for a gate/up tile of 64 gate rows and the same 64 up rows --
// writes silu(gate) * up as the down projection's hi/lo activation rows.
#pragma once
#include <cuda.h>
#include "common.cuh"
#include "mma_helpers.cuh"

namespace gd {

constexpr int PF_T = 128;                        // tokens per block
constexpr int PF_BN = 2 * PF_T;                  // MMA N: hi rows, then lo rows
constexpr int PF_BK = 64;                        // K per stage: one 128-byte swizzle atom of bf16
constexpr int PF_STAGES = 2;                     // two CTAs per SM: one's epilogue overlaps the other's MMAs
constexpr int PF_A_BYTES = 128 * PF_BK * 2;      // W tile
constexpr int PF_B_BYTES = PF_BN * PF_BK * 2;    // activation tile
constexpr int PF_STAGE = PF_A_BYTES + PF_B_BYTES;
constexpr int PF_THREADS = 128;
constexpr int PF_SMEM = PF_STAGES * PF_STAGE + 1024;
constexpr int PF_CTAS_PER_SM = 2;                // TMEM: 2 x PF_BN = 512 columns

enum { PF_EPI_PART = 0, PF_EPI_ADD = 1, PF_EPI_SWIGLU = 2 };

struct PfGemmParams {
    CUtensorMap map_w[3];   // segment s: [rows_s, K] bf16, box [PF_BK, 128], 128-byte swizzle
    CUtensorMap map_h;      // [blocks * PF_BN, K] bf16, box [PF_BK, PF_BN], 128-byte swizzle
    int tile0[4];           // first 128-row tile of each segment; tile0[nseg] = all tiles
    int row0[3];            // first output row of each segment
    int rows[3];            // rows of each segment
    int nseg;
    float* part;            // [splits][ntp][N] fp32
    int N;                  // output rows of all segments
    int ksteps;             // K steps of PF_BK per split
    int ntp;                // token rows of a split's partial (blocks * PF_T)
    int mode;               // PF_EPI_*
    float* x;               // PF_EPI_ADD: residual rows [ntp][N] (one split)
    __nv_bfloat16* hb_out;  // PF_EPI_SWIGLU: hi/lo rows [blocks * PF_BN][N]; map_w[0] gate, map_w[1] up (64-row boxes)
    unsigned* err;          // FAULT_WAIT if a bounded wait gives up
};

// shared-memory matrix descriptor of a K-major tile with 128-byte swizzle
// (8-row atoms of 1024 bytes), version 1
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D, M x N
__host__ __device__ constexpr uint32_t pf_idesc(int M, int N) {
    return (1u << 4)              // D fp32
           | (1u << 7)            // A bf16
           | (1u << 10)           // B bf16
           | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// the mbarrier receives one arrival when every earlier tcgen05 operation of this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t dt, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dt),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// grid (token blocks, tile0[nseg], splits), PF_THREADS threads, PF_SMEM dynamic shared memory
__global__ void __launch_bounds__(PF_THREADS, PF_CTAS_PER_SM) k_pf_gemm(const __grid_constant__ PfGemmParams p) {
    extern __shared__ __align__(1024) unsigned char pf_raw[];
    unsigned char* ring =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(pf_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t full[PF_STAGES], empty[PF_STAGES], accb;
    __shared__ uint32_t tmem;
    __shared__ int aborted;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int blk = blockIdx.x, tile = blockIdx.y, split = blockIdx.z;
    // the weight segment of this tile
    int sg = 0;
    while (sg + 1 < p.nseg && tile >= p.tile0[sg + 1]) ++sg;
    const int mt = tile - p.tile0[sg];   // tile within the segment
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem)),
                     "n"(PF_BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int s = 0; s < PF_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&accb, 1);
        aborted = 0;
        mbar_fence_init();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t dt = tmem;
    volatile int* ab = &aborted;
    int issued = 0;   // TMA stages issued (producer thread)

    if (warp == 0) {
        if (lane == 0) {   // TMA producer
            for (int ks = 0; ks < p.ksteps; ++ks) {
                const int s = ks % PF_STAGES;
                if (ks >= PF_STAGES && !mbar_wait(&empty[s], (uint32_t)((ks / PF_STAGES) - 1) & 1u)) {
                    *ab = 1;
                    atomicOr(p.err, FAULT_WAIT);
                    break;
                }
                if (*ab) break;
                unsigned char* a = ring + (size_t)s * PF_STAGE;
                const int k0 = (split * p.ksteps + ks) * PF_BK;
                mbar_arrive_expect_tx(&full[s], PF_STAGE);
                if (p.mode == PF_EPI_SWIGLU) {   // A rows 0-63: gate rows of the tile, 64-127: the same up rows
                    tma_load_2d(a, &p.map_w[0], k0, tile * 64, &full[s]);
                    tma_load_2d(a + PF_A_BYTES / 2, &p.map_w[1], k0, tile * 64, &full[s]);
                } else {
                    tma_load_2d(a, &p.map_w[sg], k0, mt * 128, &full[s]);
                }
                tma_load_2d(a + PF_A_BYTES, &p.map_h, k0, blk * PF_BN, &full[s]);
                issued = ks + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            constexpr uint32_t idesc = pf_idesc(128, PF_BN);
            for (int ks = 0; ks < p.ksteps; ++ks) {
                const int s = ks % PF_STAGES;
                if (*ab || !mbar_wait(&full[s], (uint32_t)(ks / PF_STAGES) & 1u)) {
                    *ab = 1;
                    atomicOr(p.err, FAULT_WAIT);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a = smem_u32(ring + (size_t)s * PF_STAGE);
#pragma unroll
                for (int kk = 0; kk < PF_BK / 16; ++kk)   // 16 K per MMA: 32 bytes along the swizzled row
                    umma_bf16(dt, smem_desc_sw128(a + 32u * kk), smem_desc_sw128(a + PF_A_BYTES + 32u * kk), idesc,
                              (ks > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);   // the stage is free once these MMAs have read it
            }
            umma_commit(&accb);   // the accumulator is complete once every MMA issued has finished
        }
        __syncwarp();
    }

    // epilogue: thread (warp w, lane l) owns segment row 128 mt + 32 w + l (TMEM lane 32 w + l)
    const bool ok = mbar_wait(&accb, 0u);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!ok) atomicOr(p.err, FAULT_WAIT);
    const int rs = mt * 128 + warp * 32 + lane;
    const int n = p.row0[sg] + rs;
    const uint32_t lanebase = dt + ((uint32_t)(warp * 32) << 16);
    if (p.mode == PF_EPI_SWIGLU) {
        // the gate rows' sums (TMEM lanes 0-63) and the up rows' sums (lanes
        // 64-127) meet in shared memory -- the ring: every copy has landed and
        // every MMA has read it -- and all four warps write silu(gate) * up
        constexpr int US = PF_T + 1;   // padded row: the lanes of a column hit distinct banks
        float* gu_s = reinterpret_cast<float*>(ring);   // [128 rows][US]
        const bool live = ok && !*ab;
        fence_proxy_async_smem();
        if (live) {
            for (int c = 0; c < PF_T; c += 32) {
                uint32_t hi[32], lo[32];
                tmem_ld_x32(lanebase + (uint32_t)c, hi);
                tmem_ld_x32(lanebase + (uint32_t)(PF_T + c), lo);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    gu_s[(warp * 32 + lane) * US + c + t] = __uint_as_float(hi[t]) + __uint_as_float(lo[t]);
            }
        }
        __syncthreads();
        if (live) {
            // thread: row f = tid % 64 of the tile, tokens tid / 64 + 2 j
            const int fr = tid & 63, t0 = tid >> 6;
            __nv_bfloat16* hrow = p.hb_out + (size_t)blk * PF_BN * p.N + (size_t)tile * 64 + fr;
#pragma unroll 4
            for (int j = 0; j < PF_T / 2; ++j) {
                const int t = t0 + 2 * j;
                const float gs = gu_s[fr * US + t], us = gu_s[(64 + fr) * US + t];
                const float a = gs / (1.0f + expf(-gs)) * us;
                const __nv_bfloat16 ah = __float2bfloat16_rn(a);
                hrow[(size_t)t * p.N] = ah;
                hrow[(size_t)(PF_T + t) * p.N] = __float2bfloat16_rn(a - __bfloat162float(ah));
            }
        }
    } else if (ok && !*ab) {
        const bool add = p.mode == PF_EPI_ADD;
        float* out = add ? p.x + (size_t)blk * PF_T * p.N : p.part + ((size_t)split * p.ntp + (size_t)blk * PF_T) * p.N;
        for (int c = 0; c < PF_T; c += 32) {
            uint32_t hi[32], lo[32];
            tmem_ld_x32(lanebase + (uint32_t)c, hi);
            tmem_ld_x32(lanebase + (uint32_t)(PF_T + c), lo);
            const bool inrow = rs < p.rows[sg];
            float xv[32];   // the residual values: every load in flight before any store
#pragma unroll
            for (int t = 0; t < 32; ++t) xv[t] = (add && inrow) ? out[(size_t)(c + t) * p.N + n] : 0.f;
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (inrow) {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    asm volatile("" : "+r"(hi[t]), "+r"(lo[t]));
                    out[(size_t)(c + t) * p.N + n] = xv[t] + (__uint_as_float(hi[t]) + __uint_as_float(lo[t]));
                }
            }
        }
    }
    // no copy may still be landing in the ring when the CTA exits
    if (tid == 0)
        for (int ks = (issued > PF_STAGES ? issued - PF_STAGES : 0); ks < issued; ++ks)
            if (!mbar_wait(&full[ks % PF_STAGES], (uint32_t)(ks / PF_STAGES) & 1u)) atomicOr(p.err, FAULT_WAIT);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(dt), "n"(PF_BN) : "memory");
    }
}

}  // namespace gd
