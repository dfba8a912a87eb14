// persist.cu -- the whole decode step as one persistent kernel (sm_103a).
//
// The pages' own strategy records the step's dispatch sequence and replays it
// ("Execution", "A constant-shape decode graph"; "Backends", "PTX (NVIDIA)");
// they name a megakernel as a possible future strategy ("Architecture
// Overview", "Current state").  This file is that alternative: one cooperative
// kernel (one CTA per SM) runs every phase of the step -- embedding; per layer
// RMSNorm+QKV, attention, O-proj, RMSNorm+gate/up+SwiGLU, down; final norm +
// head + argmax -- and is captured as the graph's single node, replayed per
// token exactly like the multi-kernel graph.
//
// Why it is faster on this GPU: a phase moves 32-235 MB, so each kernel
// boundary of the multi-kernel graph costs a ramp-up and a tail of several
// microseconds with HBM partly idle.  Here a producer warp of each CTA (one
// lane) streams the CTA's whole step -- every phase's weight rows and K/V
// tiles, in phase order -- through one ring of shared-memory stages (64 KB,
// bulk and TMA-tensor copies), while eight compute warps consume it.  The data
// of the next phase is already landing while the compute warps wait for the
// phase's grid-wide dependency, so the memory stream never stops.
//
// Phase dependencies are grid-wide counters: a CTA adds 1 to its phase's
// counter after writing the phase's outputs (release reduction), and waits
// until a phase's counter reaches the grid size before reading that phase's
// outputs (acquire load, bounded poll).  Data written by other CTAs is read
// through L2 (ld.global.cg).  The cooperative launch guarantees that every CTA
// is resident, so the waits always end; every wait is still bounded and sets
// FAULT_WAIT (plus a grid-wide abort word) if it gives up, after which every
// other wait returns at once.  The last CTA to finish resets the counters for
// the next replay.
//
// Every phase but the last gives each CTA a fixed contiguous range of weight
// rows, so that a CTA that finishes early streams the next phase's first
// stages during the tail.  The last phase (final norm, LM head, argmax) has no
// next phase to prefetch: its producers instead take 64 KB blocks of head rows
// from a grid-wide counter, one take ahead, so that no SM idles while others
// still stream.  Each row is still reduced by one CTA in slice order, so the
// logits do not depend on which CTA took the block.
//
// The arithmetic of each phase is the multi-kernel graph's (gemv_impl.cuh and
// attn_mma.cu): fixed-order reductions, no floating-point atomics, so the
// results do not depend on scheduling.
#include <cuda.h>
#include <math.h>
#include "common.cuh"
#include "internal.h"
#include "mma_helpers.cuh"

namespace gd {

constexpr int PS_CW = 8;                   // compute warps
constexpr int PS_CT = PS_CW * 32;          // compute threads
constexpr int PS_THREADS = PS_CT + 32;     // + one producer warp
constexpr int PS_SL = PS_CW;               // K-slices of a GEMV stage, one per compute warp
constexpr int PS_CBAR = 1;                 // named barrier of the compute warps
constexpr int PS_SLOT = 64 * 1024;         // bytes per ring slot
constexpr int PS_S = 196608 / PS_SLOT;      // ring slots (192 KB of shared memory)
constexpr int PS_MAX_RPS = 32;
constexpr int PS_MAX_RES = 64;
constexpr int PS_RED_ROWS = 192;          // rows whose slice partials wait in shared memory
constexpr int PS_AW = PS_CW;               // warps that compute attention
constexpr int PS_MAX_NS = 64;              // attention splits per (row, kv head)
constexpr uint32_t PS_SPIN = 1u << 22;     // default polls of a grid-wide wait (each an L2 round trip)

enum { PK_EMBED = 0, PK_QKV = 1, PK_ATTN = 2, PK_O = 3, PK_GU = 4, PK_DOWN = 5, PK_HEAD = 6 };
// gate/up phase: a CTA owns gate rows [a, b) and up rows [a, b) and writes silu(gate) * up
constexpr int EPI_SWIGLU_PAIR = 3;

// Bounded wait on a ring barrier: false after `polls` polls of try_wait (each
// may suspend for a hardware-chosen time), never an endless spin.
__device__ __forceinline__ bool ps_wait(uint64_t* bar, uint32_t parity, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }
// release add: this thread's prior writes, and those it has observed through a
// CTA barrier, are visible at gpu scope before the count is
__device__ __forceinline__ void red_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The producer's position in the CTA's whole-step stream of ring stages (in
// the producer thread's registers).  GEMV phases: the CTA's rows are up to
// three byte runs, one per stacked weight segment; a stage takes the next
// stage_bytes of them.
struct PsCursor {
    int p, loc, nst;           // phase, stage within the phase, stages of the phase (-1: not set up)
    int kind, layer;
    const unsigned char* src;  // next byte of the current run
    uint32_t run_left, stage_bytes, phase_left;
    int run, nruns;
    const unsigned char *rs0, *rs1, *rs2;
    uint32_t rb0, rb1, rb2;
    int u, uloc, ust;          // attention: unit, stage within the unit, the unit's stages
    int nextb;                 // head: the block taken for the next stage
};

// One stage, resolved before its ring slot is free: a GEMV stage is up to three
// bulk copies; an attention stage is issued from (layer, unit, stage in unit).
struct PsStage {
    int kind;
    int layer, u, uloc;
    int blk;                   // head: block of head rows, -1 for the stream's end marker
    const unsigned char *s0, *s1, *s2;
    uint32_t b0, b1, b2;
};

// shared memory besides the ring; the GEMV and attention phases never overlap,
// so their scratch shares one union
// poll until *p >= target (acquire), giving up after `polls` polls or when the
// grid-wide abort word is set; false if it gave up
__device__ __forceinline__ bool ps_poll_ge(const unsigned* p, unsigned target, const volatile unsigned* abort_word,
                                           uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i) {
        if (ld_acquire(p) >= target) return true;
        if ((i & 63u) == 63u && *abort_word) return false;
    }
    return false;
}

template <int HD, int G, int R>
struct PsShared {
    uint64_t full_bar[PS_S];   // a ring slot's copy landed (producer's expect_tx + the copy bytes)
    uint64_t empty_bar[PS_S];  // every compute warp is done with the slot
    int blk[PS_S];             // head phase: the block of head rows in the slot (-1: end of the stream)
    int abort;
    int head_end;              // head phase: a compute warp met the end of the stream
    // wait bounds of this launch (the defaults unless a test shortened them) and
    // the test hooks: a phase whose grid-wait target is one above the grid size,
    // and a stage that CTA 0's producer never issues (-1: none)
    uint32_t spin, ring_polls;
    int hold_phase, drop_stage;
    float nrm[PS_CW * R];   // per (compute warp, decode row): sum of squares of the warp's K-slice
    float wm[PS_AW][8], wl[PS_AW][8], wf[PS_AW][8];   // per (attention warp, head): max, sum, merge factor
    float hm[8], hl[8];                               // per head: the split's max and sum
    union {
        struct {
            float red[PS_RED_ROWS * R][PS_SL];   // slice partial sums of pending (weight row, decode row) pairs
            float res[PS_MAX_RES];           // residual rows (EPI_ADD)
            int cblk[PS_RED_ROWS];           // head phase: the block of each pending stage
        } gv;
        struct {
            float q[G * HD];                 // rotated, scaled query heads of the group
            float kn[HD], vn[HD];            // the new K / V row (owner of pos)
            float wo[PS_AW * G * HD];        // per-warp outputs to merge
            __align__(16) __nv_bfloat16 qt[16 * (HD + 8)];   // Q as the MMA's A tile
        } at;
    } sc;
};

// geometry of a GEMV phase: up to three stacked weight segments
struct GvGeom {
    const void* w[3];
    int n[3];
    int N, K, rps;
};

template <int HD, int G, bool PAGED, int R>
struct PsState {
    static constexpr int NR = R;   // decode rows of the step
    const PersistParams& P;
    PsShared<HD, G, R>& sh;
    unsigned char* ring;
    int cta, nc, np, tid;
    int cons;   // stages consumed (uniform over the CTA)
    // the trace buffer if tracing is on for this launch, else null: the enable
    // word is read once, so a disabled trace costs no L2 round trips per phase
    unsigned long long* trace;

    static constexpr int PPS = PS_SLOT / (2 * HD * 2);   // keys per full attention stage
    static constexpr int TILE = PPS * HD * 2;            // bytes of the K (or V) tile
    static constexpr int SUB = HD / 64;

    __device__ PsState(const PersistParams& p, PsShared<HD, G, R>& s, unsigned char* r, bool trace_on)
        : P(p), sh(s), ring(r), cta(blockIdx.x), nc(gridDim.x), np(5 * p.L + 2), tid(threadIdx.x), cons(0),
          trace(trace_on ? p.trace : nullptr) {}

    __device__ int kind(int p) const { return p == 0 ? PK_EMBED : (p == np - 1 ? PK_HEAD : 1 + (p - 1) % 5); }
    __device__ int layer(int p) const { return (p - 1) / 5; }
    __device__ void rows_of(int N, int& r0, int& r1) const {
        r0 = (int)(((long long)cta * N) / nc);
        r1 = (int)(((long long)(cta + 1) * N) / nc);
    }
    __device__ void geom(int k, int l, GvGeom& g) const {
        const void* const* w = P.lw + l * 9;   // attn_norm, q, k, v, o, ffn_norm, gate, up, down
        const int qd = P.Hq * HD, kvd = P.Hkv * HD;
        g.w[1] = g.w[2] = nullptr;
        g.n[1] = g.n[2] = 0;
        switch (k) {
            case PK_QKV: g.w[0] = w[1]; g.n[0] = qd; g.w[1] = w[2]; g.n[1] = kvd; g.w[2] = w[3]; g.n[2] = kvd;
                         g.K = P.d; g.rps = P.rps_d; break;
            case PK_O:   g.w[0] = w[4]; g.n[0] = P.d; g.K = qd; g.rps = P.rps_d; break;
            case PK_GU:  g.w[0] = w[6]; g.n[0] = P.F; g.w[1] = w[7]; g.n[1] = P.F; g.K = P.d; g.rps = P.rps_d; break;
            case PK_DOWN: g.w[0] = w[8]; g.n[0] = P.d; g.K = P.F; g.rps = P.rps_f; break;
            default:     g.w[0] = P.lm_head; g.n[0] = P.V; g.K = P.d; g.rps = P.rps_d; break;
        }
        g.N = g.n[0] + g.n[1] + g.n[2];
    }
    __device__ int units() const { return P.R * P.Hkv * P.nsplit; }
    __device__ int unit_stages(int u) const {
        const int j0 = (u % P.nsplit) * P.split_len;
        return (min(j0 + P.split_len, P.cap) - j0 + PPS - 1) / PPS;
    }

    // the head phase's block counter (after the phase arrivals, the exit counter
    // and the abort word; reset with them by the last CTA out)
    __device__ unsigned* head_ctr() const { return P.bar + np + 2; }
    __device__ int head_blocks() const { return (P.V + P.rps_d - 1) / P.rps_d; }

    __device__ const CUtensorMap* tmap(int l, int which, int box) const {
        return reinterpret_cast<const CUtensorMap*>(P.tmaps) + (l * 2 + which) * 2 + box;
    }

    // ---- the stream of stages (producer warp, lane 0) ----
    __device__ void setup(PsCursor& c) const {
        c.kind = kind(c.p);
        c.layer = (c.kind == PK_EMBED || c.kind == PK_HEAD) ? 0 : layer(c.p);
        if (c.kind == PK_EMBED) {
            c.nst = 0;
        } else if (c.kind == PK_ATTN) {
            int n = 0;
            for (int u = cta; u < units(); u += nc) n += unit_stages(u);
            c.nst = n;
            c.u = cta;
            c.uloc = 0;
            c.ust = cta < units() ? unit_stages(cta) : 0;
        } else if (c.kind == PK_HEAD) {
            // blocks of rps_d rows taken from the grid-wide counter until it passes
            // the last block; the stage after that is the end marker
            c.nst = 0x7fffffff;
            c.nextb = (int)atomicAdd(head_ctr(), 1u);
        } else {
            GvGeom g;
            geom(c.kind, c.layer, g);
            const uint32_t rb = (uint32_t)g.K * 2u;
            if (c.kind == PK_GU) {   // gate rows [a, b), then up rows [a, b)
                int a, b;
                rows_of(g.n[0], a, b);
                c.rs0 = static_cast<const unsigned char*>(g.w[0]) + (size_t)a * rb;
                c.rs1 = static_cast<const unsigned char*>(g.w[1]) + (size_t)a * rb;
                c.rs2 = c.rs1;
                c.rb0 = c.rb1 = (uint32_t)(b - a) * rb;
                c.rb2 = 0u;
                c.nruns = b > a ? 2 : 0;
                c.run = 0;
                c.src = c.rs0;
                c.run_left = c.nruns ? c.rb0 : 0u;
                c.stage_bytes = (uint32_t)g.rps * rb;
                c.phase_left = 2u * (uint32_t)(b - a) * rb;
                c.nst = (2 * (b - a) + g.rps - 1) / g.rps;
                return;
            }
            int r0, r1;
            rows_of(g.N, r0, r1);
            // the CTA's rows [r0, r1) cut by the segments [0, n0), [n0, n0 + n1), [n0 + n1, N)
            const int e0 = g.n[0], e1 = g.n[0] + g.n[1];
            const int a0 = r0, z0 = min(r1, e0);
            const int a1 = max(r0, e0), z1 = min(r1, e1);
            const int a2 = max(r0, e1), z2 = r1;
            const unsigned char* w0 = static_cast<const unsigned char*>(g.w[0]);
            const unsigned char* w1 = static_cast<const unsigned char*>(g.w[1]);
            const unsigned char* w2 = static_cast<const unsigned char*>(g.w[2]);
            const unsigned char* q0 = w0 + (size_t)a0 * rb;
            const unsigned char* q1 = w1 + (size_t)(a1 - e0) * rb;
            const unsigned char* q2 = w2 + (size_t)(a2 - e1) * rb;
            const uint32_t n0 = z0 > a0 ? (uint32_t)(z0 - a0) * rb : 0u;
            const uint32_t n1 = z1 > a1 ? (uint32_t)(z1 - a1) * rb : 0u;
            const uint32_t n2 = z2 > a2 ? (uint32_t)(z2 - a2) * rb : 0u;
            // non-empty runs, in order
            c.rs0 = n0 ? q0 : (n1 ? q1 : q2);
            c.rb0 = n0 ? n0 : (n1 ? n1 : n2);
            c.rs1 = n0 ? (n1 ? q1 : q2) : q2;
            c.rb1 = n0 ? (n1 ? n1 : n2) : (n1 ? n2 : 0u);
            c.rs2 = q2;
            c.rb2 = (n0 && n1) ? n2 : 0u;
            c.nruns = (n0 != 0u) + (n1 != 0u) + (n2 != 0u);
            c.run = 0;
            c.src = c.rs0;
            c.run_left = c.rb0;
            c.stage_bytes = (uint32_t)g.rps * rb;
            c.phase_left = (uint32_t)(r1 - r0) * rb;
            c.nst = (r1 - r0 + g.rps - 1) / g.rps;
        }
    }
    // take up to `want` bytes from the runs (the current one, then the next)
    __device__ static uint32_t take(PsCursor& c, uint32_t want, const unsigned char*& src) {
        if (c.run_left == 0u && c.run + 1 < c.nruns) {
            ++c.run;
            c.src = c.run == 1 ? c.rs1 : c.rs2;
            c.run_left = c.run == 1 ? c.rb1 : c.rb2;
        }
        const uint32_t n = min(want, c.run_left);
        src = c.src;
        c.src += n;
        c.run_left -= n;
        return n;
    }
    // resolve the next stage of the stream into s and step past it; false at the end
    __device__ bool next(PsCursor& c, PsStage& s) const {
        for (;;) {
            if (c.p >= np) return false;
            if (c.nst < 0) setup(c);
            if (c.loc < c.nst) break;
            ++c.p;
            c.loc = 0;
            c.nst = -1;
        }
        s.kind = c.kind;
        if (c.kind == PK_HEAD) {
            const int b = c.nextb;
            if (b >= 0 && b < head_blocks()) {
                const uint32_t rb = (uint32_t)P.d * 2u;
                const int nr = min(P.rps_d, P.V - b * P.rps_d);
                s.blk = b;
                s.s0 = static_cast<const unsigned char*>(P.lm_head) + (size_t)b * P.rps_d * rb;
                s.b0 = (uint32_t)nr * rb;
                // the next take: its result is first used after this stage's slot wait
                c.nextb = (int)atomicAdd(head_ctr(), 1u);
            } else {
                s.blk = -1;   // the end marker is the stream's last stage
                c.p = np;
            }
            ++c.loc;
            return true;
        }
        if (c.kind == PK_ATTN) {
            s.layer = c.layer;
            s.u = c.u;
            s.uloc = c.uloc;
            if (++c.uloc == c.ust) {
                c.u += nc;
                c.uloc = 0;
                c.ust = c.u < units() ? unit_stages(c.u) : 0;
            }
        } else {
            const uint32_t total = min(c.stage_bytes, c.phase_left);
            s.b0 = take(c, total, s.s0);
            s.b1 = take(c, total - s.b0, s.s1);
            s.b2 = take(c, total - s.b0 - s.b1, s.s2);
            c.phase_left -= total;
        }
        ++c.loc;
        return true;
    }
    // copy stage s into ring slot `slot`
    __device__ void issue(const PsStage& s, int slot) const {
        unsigned char* dst = ring + (size_t)slot * PS_SLOT;
        uint64_t* bar = &sh.full_bar[slot];
        if (s.kind == PK_HEAD) {
            // the header before the arrival that releases it to the consumers
            sh.blk[slot] = s.blk;
            if (s.blk < 0) {
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, s.b0);
                bulk_g2s(dst, s.s0, s.b0, bar);
            }
            return;
        }
        if (s.kind != PK_ATTN) {
            mbar_arrive_expect_tx(bar, s.b0 + s.b1 + s.b2);
            if (s.b0) bulk_g2s(dst, s.s0, s.b0, bar);
            if (s.b1) bulk_g2s(dst + s.b0, s.s1, s.b1, bar);
            if (s.b2) bulk_g2s(dst + s.b0 + s.b1, s.s2, s.b2, bar);
            return;
        }
        const int l = s.layer, u = s.u;
        const int sp = u % P.nsplit, g = (u / P.nsplit) % P.Hkv, r = u / (P.nsplit * P.Hkv);
        const int j0 = sp * P.split_len;
        const int j1 = min(j0 + P.split_len, P.cap);
        const int p0 = j0 + s.uloc * PPS, p1 = min(p0 + PPS, j1);
        const int n = p1 - p0;
        unsigned char* kd = dst;
        unsigned char* vd = dst + TILE;
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * n * HD * 2));
        if (PAGED) {
            const int pg_size = P.page;
            for (int q = p0; q < p1; q += pg_size) {
                int pg = P.slot_map[(size_t)r * P.pages_per_row + q / pg_size];
                if (pg < 0 || pg >= P.num_pages) pg = 0;   // flagged by the consumers
                const int y = (pg * P.Hkv + g) * pg_size;
#pragma unroll
                for (int sb = 0; sb < SUB; ++sb) {
                    tma_load_2d(kd + sb * PPS * 128 + (q - p0) * 128, tmap(l, 0, 0), sb * 64, y, bar);
                    tma_load_2d(vd + sb * PPS * 128 + (q - p0) * 128, tmap(l, 1, 0), sb * 64, y, bar);
                }
            }
        } else {
            const int y = (r * P.Hkv + g) * P.cap + p0;
            const int box = n == PPS ? 0 : 1;   // full stage, or the half stage that ends a split
#pragma unroll
            for (int sb = 0; sb < SUB; ++sb) {
                tma_load_2d(kd + sb * PPS * 128, tmap(l, 0, box), sb * 64, y, bar);
                tma_load_2d(vd + sb * PPS * 128, tmap(l, 1, box), sb * 64, y, bar);
            }
        }
    }

    // consumer side of one stage: wait for it (skipped after an abort)
    __device__ const unsigned char* stage_wait() {
        const int slot = cons % PS_S;
        volatile int* ab = &sh.abort;
        if (!*ab && !ps_wait(&sh.full_bar[slot], (cons / PS_S) & 1, sh.ring_polls)) {
            *ab = 1;
            atomicOr(P.err, FAULT_WAIT);
        }
        return ring + (size_t)slot * PS_SLOT;
    }
    // this warp is done reading the stage (every compute warp calls it once per stage)
    __device__ void stage_release() {
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&sh.empty_bar[cons % PS_S]);
        ++cons;
    }
    __device__ static void csync() { named_sync(PS_CBAR, PS_CT); }

    // producer warp, lane 0: stream every stage of the CTA's step through the
    // ring; each stage is resolved while its slot is still in use, so a freed
    // slot is refilled by the copy instructions alone.  After an abort it issues
    // nothing more and waits (bounded) for the copies it has in flight.
    __device__ void produce() {
        PsCursor c;
        c.p = 0;
        c.loc = 0;
        c.nst = -1;
        PsStage s;
        volatile int* ab = &sh.abort;
        const int dropped = cta == 0 ? sh.drop_stage : -1;   // test hook: a copy that never lands
        bool have = next(c, s);
        int i = 0;
        for (; have && !*ab; ++i) {
            const int slot = i % PS_S;
            if (i >= PS_S) {
                if (!ps_wait(&sh.empty_bar[slot], ((i / PS_S) - 1) & 1, sh.ring_polls)) {
                    *ab = 1;
                    atomicOr(P.err, FAULT_WAIT);
                    break;
                }
                if (*ab) break;
            }
            if (i != dropped) issue(s, slot);
            have = next(c, s);
        }
        // no copy may still be landing when the CTA exits (after an abort some were never consumed)
        for (int j = max(0, i - PS_S); j < i; ++j)
            if (j != dropped && !ps_wait(&sh.full_bar[j % PS_S], (j / PS_S) & 1, sh.ring_polls))
                atomicOr(P.err, FAULT_WAIT);
    }

    __device__ void grid_arrive(int p) {
        csync();
        if (tid == 0) red_release(P.bar + p, 1u);
    }
    __device__ void grid_wait(int p) {
        if (tid == 0) {
            volatile unsigned* gab = P.bar + np + 1;
            const unsigned target = (unsigned)nc + (p == sh.hold_phase ? 1u : 0u);
            if (!ps_poll_ge(P.bar + p, target, gab, sh.spin)) {
                sh.abort = 1;
                atomicOr(P.err, FAULT_WAIT);
                atomicExch(const_cast<unsigned*>(gab), 1u);
            }
        }
        csync();
    }
};

// ---------------- GEMV phase ----------------
// Sum RU values over the warp with RU/2 + RU/4 + ... + 5 - log2(RU) shuffles
// (each level halves the rows a lane carries); returns the total of row `row`,
// held by the lanes whose low 5 - log2(RU) bits are zero.
template <int RU>
__device__ __forceinline__ float rows_reduce(float (&v)[RU], int lane, int& row) {
    row = 0;
    int off = 16;
#pragma unroll
    for (int h = RU / 2; h >= 1; h /= 2) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int u = 0; u < h; ++u) {
            const float send = up ? v[u] : v[u + h];
            const float keep = up ? v[u + h] : v[u];
            v[u] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        if (up) row += h;
        off >>= 1;
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 / RU; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// One GEMV phase over this CTA's rows: warp w owns K-slice w of every row, with
// the slice's activations of each decode row in registers; each lane's partial
// sums are reduced over the warp, the slices' sums wait in shared memory and
// are added in slice order (fixed order: no atomics) when a chunk of
// PS_RED_ROWS weight rows is complete.  Stages carry no CTA-wide barrier: a
// warp releases a stage when it is done.  Decode row r of the activations and
// of the output sits at r * K and r * N (r * n[0] for the SwiGLU pair).
template <int CPL, int PRO, int EPI, int HD, int G, bool PAGED, int R>
__device__ __forceinline__ void ps_gemv(PsState<HD, G, PAGED, R>& st, const GvGeom& g, const float* act,
                                        const __nv_bfloat16* gain, float* out, int phase) {
    using ST = PsState<HD, G, PAGED, R>;
    constexpr int VEC = 8;
    // weight rows per pass: a slot holds PS_SLOT / (4096 CPL) rows of K = 2048 CPL (rounded to a
    // power of two), divided among the decode rows so that a lane keeps at most 16 sums
    constexpr int RU0 = PS_SLOT / (4096 * CPL) > 0 ? PS_SLOT / (4096 * CPL) : 1;
    constexpr int RU1 = RU0 >= 16 ? 16 : (RU0 >= 8 ? 8 : (RU0 >= 4 ? 4 : (RU0 >= 2 ? 2 : 1)));
    constexpr int RU = RU1 / R >= 1 ? RU1 / R : 1;
    constexpr int RS = RU * R;   // sums per lane and pass
    constexpr bool TWO = R == 1 || RS < 4;   // two FMA chains per sum, unless several rows give the ILP
    static_assert((RU & (RU - 1)) == 0 && (R & (R - 1)) == 0 && RS <= 16, "rows per pass must be a power of two");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = g.K;
    const int SWV = K / (PS_SL * VEC);
    const int slice = warp;
    const int vbase = slice * SWV;
    int row0, row1;   // the CTA's rows; for the gate/up pair, 2 (b - a) logical rows from row0 = a
    if (EPI == EPI_SWIGLU_PAIR) {
        st.rows_of(g.n[0], row0, row1);
        row1 = row0 + 2 * (row1 - row0);
    } else {
        st.rows_of(g.N, row0, row1);
    }
    const int rps = g.rps;
    const int nst = (row1 - row0 + rps - 1) / rps;
    const int chunk = (PS_RED_ROWS / rps) * rps;   // weight rows per flush, whole stages
    const size_t row_bytes = (size_t)K * 2;
    const int ostride = EPI == EPI_SWIGLU_PAIR ? g.n[0] : g.N;   // output row stride per decode row
    auto& sh = st.sh;

    // the norm gains do not depend on the previous phase: load them before its wait
    uint4 graw[PRO == PRO_RMSNORM ? CPL : 1];
    if (PRO == PRO_RMSNORM) {
#pragma unroll
        for (int j = 0; j < CPL; ++j) graw[j] = *reinterpret_cast<const uint4*>(gain + (vbase + lane + 32 * j) * VEC);
    }
    st.grid_wait(phase - 1);
    if (tid == 0 && st.trace) trace_mark(st.trace, phase, 1);

    // prologue: this lane's activations (its slice columns) of every decode row,
    // in registers; the slices of the compute warps cover K exactly, so they
    // also give the norms
    float areg[R][CPL][VEC];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = (vbase + lane + 32 * j) * VEC;
            const float4 x0 = ldcg4(act + (size_t)r * K + c), x1 = ldcg4(act + (size_t)r * K + c + 4);
            areg[r][j][0] = x0.x; areg[r][j][1] = x0.y; areg[r][j][2] = x0.z; areg[r][j][3] = x0.w;
            areg[r][j][4] = x1.x; areg[r][j][5] = x1.y; areg[r][j][6] = x1.z; areg[r][j][7] = x1.w;
        }
    if (PRO == PRO_RMSNORM) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int e = 0; e < VEC; ++e) ss = fmaf(areg[r][j][e], areg[r][j][e], ss);
            ss = warp_sum(ss);
            if (lane == 0) sh.nrm[warp * R + r] = ss;
        }
        ST::csync();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < PS_CW; ++w) t += sh.nrm[w * R + r];
            const float inv = 1.0f / sqrtf(t / (float)K + st.P.eps);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                float gf[VEC];
                Elem<__nv_bfloat16>::unpack(graw[j], gf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) areg[r][j][e] = areg[r][j][e] * inv * gf[e];
            }
        }
    }
    const bool res_local = R == 1 && EPI == EPI_ADD && (row1 - row0) <= PS_MAX_RES;
    if (EPI == EPI_ADD && res_local)   // read before this phase writes any row; used after a barrier
        for (int i = tid; i < row1 - row0; i += PS_CT) sh.sc.gv.res[i] = __ldcg(out + row0 + i);

    unsigned long long best[R];
    bool nonfin[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        best[r] = 0ull;
        nonfin[r] = false;
    }
    bool live_all = true;
    // one landed stage of nr weight rows: the slice partial of each (row, decode
    // row) pair goes to the pending rows from `base` on
    auto consume = [&](const unsigned char* stg, int nr, int base, bool live) {
        for (int m0 = 0; m0 < nr; m0 += RU) {
            float acc[RS], acc2[RS];   // sum u * R + r: weight row m0 + u, decode row r
#pragma unroll
            for (int u = 0; u < RS; ++u) acc[u] = acc2[u] = 0.f;
            // slices are exactly 32 * CPL vectors wide (the plan admits no other K);
            // rows of the last pass beyond nr re-read row nr - 1, results dropped
            if (live) {
                // the pass's weight vectors: all loaded up front while the activations leave
                // room in the registers, else each just before its use
                constexpr bool PRE = R * CPL * VEC <= 64;
                uint4 wv[RU][CPL];
                if (PRE) {
#pragma unroll
                    for (int u = 0; u < RU; ++u) {
                        const int iu = min(m0 + u, nr - 1);
                        const uint4* wr = reinterpret_cast<const uint4*>(stg + (size_t)iu * row_bytes);
#pragma unroll
                        for (int j = 0; j < CPL; ++j) wv[u][j] = wr[vbase + lane + 32 * j];
                    }
                }
#pragma unroll
                for (int u = 0; u < RU; ++u)
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        float wf[VEC];
                        if (PRE) {
                            Elem<__nv_bfloat16>::unpack(wv[u][j], wf);
                        } else {
                            const uint4* wr =
                                reinterpret_cast<const uint4*>(stg + (size_t)min(m0 + u, nr - 1) * row_bytes);
                            Elem<__nv_bfloat16>::unpack(wr[vbase + lane + 32 * j], wf);
                        }
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int e = 0; e < VEC; e += 2) {
                                acc[u * R + r] = fmaf(wf[e], areg[r][j][e], acc[u * R + r]);
                                if (TWO)
                                    acc2[u * R + r] = fmaf(wf[e + 1], areg[r][j][e + 1], acc2[u * R + r]);
                                else
                                    acc[u * R + r] = fmaf(wf[e + 1], areg[r][j][e + 1], acc[u * R + r]);
                            }
                    }
            }
            if (TWO) {
#pragma unroll
                for (int u = 0; u < RS; ++u) acc[u] += acc2[u];
            }
            int ru;
            const float t = rows_reduce<RS>(acc, lane, ru);   // ru = u * R + r
            if ((lane & (32 / RS - 1)) == 0 && m0 + ru / R < nr)
                sh.sc.gv.red[(base + m0) * R + ru][slice] = t;
        }
    };
    // the argmax key and non-finite flag of a head row's logit
    auto pick = [&](float t, int row, int r) {
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (q == r) {
                if (!isfinite(t)) nonfin[q] = true;
                const unsigned long long key = argmax_key(t, row);
                best[q] = key > best[q] ? key : best[q];
            }
    };

    if (EPI == EPI_LOGITS) {
        // blocks of rps rows in the order the producer took them; a chunk of
        // stages is flushed when full or at the end of the stream.  The compute
        // warps see the same headers, so they agree on every chunk; a warp that
        // stops on an abort sets head_end, which every warp reads between the
        // chunk's two barriers, so all leave after the same chunk.
        const int spc = PS_RED_ROWS / rps;   // stages per chunk
        for (;;) {
            int n = 0;
            bool end = false;
            for (; n < spc; ++n) {
                const int slot = st.cons % PS_S;
                const unsigned char* stg = st.stage_wait();
                const bool live = !*reinterpret_cast<volatile int*>(&sh.abort);
                live_all = live_all && live;
                const int blk = live ? *reinterpret_cast<volatile int*>(&sh.blk[slot]) : -1;
                if (blk < 0) {
                    end = true;
                    break;
                }
                if (tid == 0) sh.sc.gv.cblk[n] = blk;
                consume(stg, min(rps, g.N - blk * rps), n * rps, true);
                st.stage_release();
            }
            if (end && lane == 0) *reinterpret_cast<volatile int*>(&sh.head_end) = 1;
            ST::csync();
            const bool stop = *reinterpret_cast<volatile int*>(&sh.head_end) != 0;
            if (live_all) {
                for (int ir = tid; ir < n * rps * R; ir += PS_CT) {
                    const int i = ir / R, r = ir % R;
                    const int row = sh.sc.gv.cblk[i / rps] * rps + i % rps;
                    if (row >= g.N) continue;
                    float t = 0.f;
#pragma unroll
                    for (int w = 0; w < PS_SL; ++w) t += sh.sc.gv.red[i * R + r][w];
                    out[(size_t)r * ostride + row] = t;
                    pick(t, row, r);
                }
            }
            ST::csync();
            if (stop) break;
        }
    }

    int c0 = 0;   // first row (within the CTA's rows) of the pending chunk
    for (int k = 0; EPI != EPI_LOGITS && k < nst; ++k) {
        const int a = k * rps;   // first row of the stage, within the CTA's rows
        const int nr = min(rps, row1 - row0 - a);
        const unsigned char* stg = st.stage_wait();
        const bool live = !*reinterpret_cast<volatile int*>(&sh.abort);
        live_all = live_all && live;
        consume(stg, nr, a - c0, live);
        st.stage_release();
        // a full chunk (or the phase's last rows): add the slices, write the rows
        const int done = a + nr;
        if (done - c0 == chunk || k == nst - 1) {
            ST::csync();
            if (EPI == EPI_SWIGLU_PAIR && live_all) {   // one flush holds both halves (the plan checks it)
                const int n = (row1 - row0) / 2;
                for (int ir = tid; ir < n * R; ir += PS_CT) {
                    const int i = ir / R, r = ir % R;
                    float gs = 0.f, us = 0.f;
#pragma unroll
                    for (int w = 0; w < PS_SL; ++w) {
                        gs += sh.sc.gv.red[i * R + r][w];
                        us += sh.sc.gv.red[(n + i) * R + r][w];
                    }
                    out[(size_t)r * ostride + row0 + i] = gs / (1.0f + expf(-gs)) * us;
                }
            } else if (live_all) {
                for (int ir = tid; ir < (done - c0) * R; ir += PS_CT) {
                    const int i = ir / R, r = ir % R;
                    const int row = row0 + c0 + i;
                    float t = 0.f;
#pragma unroll
                    for (int w = 0; w < PS_SL; ++w) t += sh.sc.gv.red[i * R + r][w];
                    float* o = out + (size_t)r * ostride + row;
                    if (EPI == EPI_ADD) {
                        *o = (res_local ? sh.sc.gv.res[row - row0] : __ldcg(o)) + t;
                    } else {
                        *o = t;
                    }
                }
            }
            ST::csync();
            c0 = done;
        }
    }
    if (EPI == EPI_LOGITS) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, best[r], o);
                best[r] = other > best[r] ? other : best[r];
            }
            const bool any_nf = __any_sync(0xffffffffu, nonfin[r]);
            if (lane == 0) {
                if (best[r]) atomicMax(st.P.amax + r, best[r]);
                if (any_nf) atomicOr(st.P.nonfinite + r, 1u);
            }
        }
    }
}

// ---------------- attention phase (tensor cores, as attn_mma.cu) ----------------
template <int HD, int G, bool PAGED, int R>
__device__ __forceinline__ void ps_attention(PsState<HD, G, PAGED, R>& st, int l) {
    using ST = PsState<HD, G, PAGED, R>;
    constexpr int PPS = ST::PPS, TILE = ST::TILE;
    constexpr int KPW = PPS / PS_AW, BLK = KPW / 16, KSTEP = HD / 16, DT = HD / 16;
    static_assert(G <= 4, "P^T columns hold G heads' bf16 parts and G remainders");
    static_assert(KPW >= 16 && KPW % 16 == 0, "each attention warp takes whole 16-key blocks of a stage");
    const PersistParams& P = st.P;
    auto& sh = st.sh;
    float* q_s = sh.sc.at.q;
    float* kn_s = sh.sc.at.kn;
    float* vn_s = sh.sc.at.vn;
    float* wo_s = sh.sc.at.wo;
    __nv_bfloat16* qt_s = sh.sc.at.qt;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    __nv_bfloat16* Kc = reinterpret_cast<__nv_bfloat16*>(P.kv[2 * l]);
    __nv_bfloat16* Vc = reinterpret_cast<__nv_bfloat16*>(P.kv[2 * l + 1]);
    const int Pg = P.page;

    for (int u = st.cta; u < st.units(); u += st.nc) {
        const int s = u % P.nsplit, g = (u / P.nsplit) % P.Hkv, r = u / (P.nsplit * P.Hkv);
        const int j0 = s * P.split_len;
        const int j1 = min(j0 + P.split_len, P.cap);
        const int nst = (j1 - j0 + PPS - 1) / PPS;
        int pos = P.slots[P.R + r];
        pos = min(max(pos, 0), P.cap - 1);
        const float* qrow = P.qkv + (size_t)r * (P.Hq + 2 * P.Hkv) * HD;
        const float2* rt = P.rope + (size_t)pos * (HD / 2);
        if (PAGED) {   // page ids this unit's producer read
            for (int q = j0 + tid * Pg; q < j1; q += PS_CT * Pg) {
                const int pg = P.slot_map[(size_t)r * P.pages_per_row + q / Pg];
                if (pg < 0 || pg >= P.num_pages) atomicOr(P.err, FAULT_SLOT_MAP);
            }
        }
        for (int i = tid; i < G * (HD / 2); i += PS_CT) {
            const int h = i / (HD / 2), d = i % (HD / 2);
            const float* qh = qrow + (size_t)(g * G + h) * HD;
            const float a = __ldcg(qh + d), b = __ldcg(qh + d + HD / 2);
            const float2 cs = rt[d];
            q_s[h * HD + d] = (a * cs.x - b * cs.y) * P.scale;
            q_s[h * HD + d + HD / 2] = (a * cs.y + b * cs.x) * P.scale;
        }
        const bool owner = pos >= j0 && pos < j1;
        if (owner) {
            const float* kh = qrow + (size_t)P.Hq * HD + (size_t)g * HD;
            const float* vh = kh + (size_t)P.Hkv * HD;
            size_t off;
            bool ok = true;
            if (PAGED) {
                const int slot = P.slots[2 * P.R + r];
                if (slot < 0 || slot >= P.num_pages * Pg) {
                    ok = false;
                    if (tid == 0) atomicOr(P.err, FAULT_WRITE_MAP);
                }
                const int pg = ok ? slot / Pg : 0, o = ok ? slot % Pg : 0;
                off = (((size_t)pg * P.Hkv + g) * Pg + o) * HD;
            } else {
                off = (((size_t)r * P.Hkv + g) * P.cap + pos) * HD;
            }
            for (int d = tid; d < HD / 2; d += PS_CT) {
                const float a = __ldcg(kh + d), b = __ldcg(kh + d + HD / 2);
                const float2 cs = rt[d];
                const float k0 = a * cs.x - b * cs.y, k1 = a * cs.y + b * cs.x;
                kn_s[d] = ok ? Elem<__nv_bfloat16>::round_store(k0, Kc + off + d) : bf16_round_f(k0);
                kn_s[d + HD / 2] = ok ? Elem<__nv_bfloat16>::round_store(k1, Kc + off + d + HD / 2) : bf16_round_f(k1);
            }
            for (int d = tid; d < HD; d += PS_CT) {
                const float vv = __ldcg(vh + d);
                vn_s[d] = ok ? Elem<__nv_bfloat16>::round_store(vv, Vc + off + d) : bf16_round_f(vv);
            }
        }
        ST::csync();
        // Q as the MMA's A operand, a padded bf16 tile [16][HD + 8]: rows g < G hold
        // bf16(q) of head g, rows 8 + g the remainder q - bf16(q), the rest zero
        for (int i = tid; i < 16 * HD; i += PS_CT) {
            const int row = i / HD, col = i % HD, h = row & 7;
            const float v = h < G ? q_s[h * HD + col] : 0.f;
            const float hi = bf16_round_f(v);
            qt_s[row * (HD + 8) + col] = __float2bfloat16_rn(row < 8 ? hi : v - hi);
        }
        ST::csync();

        // O^T accumulators: tile dt covers dims 16dt..16dt+15 (rows g, g + 8) x
        // columns 2tq, 2tq+1 (columns 0..3: heads' bf16 parts, 4..7: remainders)
        float m_run = -INFINITY, l_run = 0.f;
        float o[DT][4];
        if (warp < PS_AW) {
#pragma unroll
            for (int n = 0; n < DT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        }
        const int h0 = (2 * tq) & 3, h1 = (2 * tq + 1) & 3;   // heads of this lane's two columns

        for (int t = 0; t < nst; ++t) {
            unsigned char* kt = const_cast<unsigned char*>(st.stage_wait());
            unsigned char* vt = kt + TILE;
            const bool live = !*reinterpret_cast<volatile int*>(&sh.abort);
            const int p0 = j0 + t * PPS;
            if (owner && pos >= p0 && pos < p0 + PPS) {   // CTA-uniform
                const int row = pos - p0;
                for (int i = tid; i < 2 * (HD / 8); i += PS_CT) {
                    const int c = i % (HD / 8);
                    const float* src = (i < HD / 8 ? kn_s : vn_s) + c * 8;
                    uint4 v;
                    v.x = pack_bf16x2(src[0], src[1]);
                    v.y = pack_bf16x2(src[2], src[3]);
                    v.z = pack_bf16x2(src[4], src[5]);
                    v.w = pack_bf16x2(src[6], src[7]);
                    *reinterpret_cast<uint4*>((i < HD / 8 ? kt : vt) + swz<HD, PPS>(row, c)) = v;
                }
                fence_proxy_async_smem();   // these generic writes before the slot's next async refill
                ST::csync();
            }
            if (live && warp < PS_AW) {
#pragma unroll
                for (int b = 0; b < BLK; ++b) {
                    const int kb = warp * KPW + b * 16;
                    const int key0 = p0 + kb;
                    if (key0 > pos || key0 >= j1) continue;
                    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                    for (int ks = 0; ks < KSTEP; ++ks) {
                        const int mi = lane >> 3, rr = lane & 7;
                        // A fragments: (rows 0-7 | 8-15) x (cols 16ks..+7 | +8..+15)
                        uint32_t qa[4];
                        ldsm_x4(smem_u32(qt_s + (rr + ((mi & 1) << 3)) * (HD + 8) + ks * 16 + ((mi >> 1) << 3)), qa[0],
                                qa[1], qa[2], qa[3]);
                        const int krow = kb + rr + ((mi >> 1) << 3);
                        const int chunk = ks * 2 + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(smem_u32(kt + swz<HD, PPS>(krow, chunk)), b0, b1, b2, b3);
                        mma_bf16(sacc[0], qa, b0, b1);
                        mma_bf16(sacc[1], qa, b2, b3);
                    }
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
                    const float mn = fmaxf(m_run, mx);
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
                    // rescale: the lane's columns belong to heads h0, h1 (alpha of head h sits in lanes 4h..4h+3)
                    const float a0 = __shfl_sync(0xffffffffu, alpha, 4 * h0);
                    const float a1 = __shfl_sync(0xffffffffu, alpha, 4 * h1);
#pragma unroll
                    for (int n = 0; n < DT; ++n) {
                        o[n][0] *= a0; o[n][1] *= a1; o[n][2] *= a0; o[n][3] *= a1;
                    }
                    // P^T as the B operand: column gq < 4 is head gq's bf16(p), column 4 + h
                    // the remainder p - bf16(p) of head h (taken from lane - 16)
                    uint32_t pb0, pb1;
                    {
                        float pv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float other = __shfl_xor_sync(0xffffffffu, pr[i], 16);
                            const int h = gq & 3;
                            const float v = (gq < 4) ? pr[i] : other;
                            const float vv = h < G ? v : 0.f;
                            const float hi = bf16_round_f(vv);
                            pv[i] = gq < 4 ? hi : vv - hi;
                        }
                        pb0 = pack_bf16x2(pv[0], pv[1]);   // keys 2tq, 2tq+1 of the block
                        pb1 = pack_bf16x2(pv[2], pv[3]);   // keys 8+2tq, 9+2tq
                    }
                    const bool partial = key0 + 15 > pos || key0 + 15 >= j1;
                    const uint32_t keep0 = (vis[0] ? 0x0000FFFFu : 0u) | (vis[1] ? 0xFFFF0000u : 0u);
                    const uint32_t keep1 = (vis[2] ? 0x0000FFFFu : 0u) | (vis[3] ? 0xFFFF0000u : 0u);
                    // O^T += V^T P^T: V^T fragments by transposed ldmatrix (rows = dims, k = keys)
#pragma unroll
                    for (int dt = 0; dt < DT; ++dt) {
                        // matrices: (keys 0-7, dims 0-7) a0, (keys 0-7, dims 8-15) a1,
                        //           (keys 8-15, dims 0-7) a2, (keys 8-15, dims 8-15) a3
                        const int mi = lane >> 3, rr = lane & 7;
                        const int vrow = kb + rr + ((mi >> 1) << 3);
                        const int chunk = dt * 2 + (mi & 1);
                        uint32_t va[4];
                        ldsm_x4_t(smem_u32(vt + swz<HD, PPS>(vrow, chunk)), va[0], va[1], va[2], va[3]);
                        if (partial) {   // masked keys' V become zero by select (this lane's keys = its scores' keys)
                            va[0] &= keep0;
                            va[1] &= keep0;
                            va[2] &= keep1;
                            va[3] &= keep1;
                        }
                        mma_bf16(o[dt], va, pb0, pb1);
                    }
                }
            }
            st.stage_release();
        }

        // merge the attention warps (fixed order), write this split's partial
        if (warp < PS_AW) {
            float lsum = l_run;
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
            // add the remainder columns (lane + 2 within the quad) to the heads' columns
#pragma unroll
            for (int n = 0; n < DT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] += __shfl_xor_sync(0xffffffffu, o[n][e], 2);
            if (tq < 2) {
#pragma unroll
                for (int n = 0; n < DT; ++n) {
                    if (h0 < G) {
                        wo_s[(warp * G + h0) * HD + n * 16 + gq] = o[n][0];
                        wo_s[(warp * G + h0) * HD + n * 16 + gq + 8] = o[n][2];
                    }
                    if (h1 < G) {
                        wo_s[(warp * G + h1) * HD + n * 16 + gq] = o[n][1];
                        wo_s[(warp * G + h1) * HD + n * 16 + gq + 8] = o[n][3];
                    }
                }
            }
            if (gq < G && tq == 0) {
                sh.wm[warp][gq] = m_run;
                sh.wl[warp][gq] = lsum;
            }
        }
        ST::csync();
        // per (warp, head) merge factors and the split's (max, sum) per head
        if (tid < G) {
            const int h = tid;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < PS_AW; ++w) M = fmaxf(M, sh.wm[w][h]);
            float Ls = 0.f;
#pragma unroll
            for (int w = 0; w < PS_AW; ++w) {
                const float f = (sh.wm[w][h] == -INFINITY) ? 0.f : expf(sh.wm[w][h] - M);
                sh.wf[w][h] = f;
                Ls = fmaf(f, sh.wl[w][h], Ls);
            }
            sh.hm[h] = M;
            sh.hl[h] = Ls;
        }
        ST::csync();
        for (int i = tid; i < G * HD; i += PS_CT) {
            const int h = i / HD, d = i % HD;
            float Os = 0.f;
#pragma unroll
            for (int w = 0; w < PS_AW; ++w) Os = fmaf(sh.wf[w][h], wo_s[(w * G + h) * HD + d], Os);
            float* pp = P.part + (((size_t)r * P.Hq + g * G + h) * P.nsplit + s) * (HD + 4);
            pp[4 + d] = Os;
            if (d == 0) {
                pp[0] = sh.hm[h];
                pp[1] = sh.hl[h];
            }
        }
        ST::csync();
        // publish the partial; wait until every split of this (row, kv head) has
        // published (the group's counter grows by nsplit per layer; all CTAs are
        // resident, and the wait is bounded)
        if (tid == 0) {
            unsigned* cnt = P.counters + r * P.Hkv + g;
            red_release(cnt, 1u);
            const unsigned target = (unsigned)P.nsplit * (unsigned)(l + 1);
            volatile unsigned* gab = P.bar + st.np + 1;
            if (!ps_poll_ge(cnt, target, gab, sh.spin)) {
                sh.abort = 1;
                atomicOr(P.err, FAULT_WAIT);
                atomicExch(const_cast<unsigned*>(gab), 1u);
            }
        }
        ST::csync();
        // this split's share of the group's G * HD outputs: every split's
        // (max, sum, value) requested before any is used
        {
            const int NS = P.nsplit, E = G * HD;
            const int e0 = (int)(((long long)s * E) / NS), e1 = (int)(((long long)(s + 1) * E) / NS);
            constexpr int CH = 24;   // splits per batch of loads
            for (int e = e0 + tid; e < e1; e += PS_CT) {
                const int h = e / HD, d = e % HD;
                const float* base = P.part + (((size_t)r * P.Hq + g * G + h) * NS) * (HD + 4);
                float M = -INFINITY, Lsum = 0.f, acc = 0.f;
                for (int s0 = 0; s0 < NS; s0 += CH) {
                    float mv[CH], lv[CH], ov[CH];
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const bool in = s0 + j < NS;
                        const float* pj = base + (size_t)(in ? s0 + j : 0) * (HD + 4);
                        mv[j] = in ? __ldcg(pj) : -INFINITY;
                        lv[j] = in ? __ldcg(pj + 1) : 0.f;
                        ov[j] = in ? __ldcg(pj + 4 + d) : 0.f;
                    }
                    float Mc = M;
#pragma unroll
                    for (int j = 0; j < CH; ++j) Mc = fmaxf(Mc, mv[j]);
                    const float resc = (M == -INFINITY) ? 0.f : expf(M - Mc);
                    Lsum *= resc;
                    acc *= resc;
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const float f = (mv[j] == -INFINITY) ? 0.f : expf(mv[j] - Mc);
                        Lsum = fmaf(f, lv[j], Lsum);
                        acc = fmaf(f, ov[j], acc);
                    }
                    M = Mc;
                }
                P.attn[(size_t)r * P.Hq * HD + (size_t)(g * G + h) * HD + d] = acc / Lsum;
            }
        }
        ST::csync();
    }
}

template <int CPL_D, int CPL_F, int HD, int G, bool PAGED, int R>
__global__ void __launch_bounds__(PS_THREADS, 1) k_persist(const __grid_constant__ PersistParams P) {
    extern __shared__ __align__(1024) unsigned char ps_raw[];
    unsigned char* ring =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(ps_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ PsShared<HD, G, R> sh;
    using ST = PsState<HD, G, PAGED, R>;
    const int tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < PS_S; ++s) {
            mbar_init(&sh.full_bar[s], 1);
            mbar_init(&sh.empty_bar[s], PS_CW);
        }
        sh.abort = 0;
        sh.head_end = 0;
        // the wait bounds and test hooks of this launch (all zero: defaults, no hooks)
        const uint4 dbg = __ldcg(reinterpret_cast<const uint4*>(P.dbg));
        sh.spin = dbg.x ? dbg.x : PS_SPIN;
        sh.ring_polls = dbg.y ? dbg.y : MBAR_POLLS;
        sh.hold_phase = (int)dbg.z - 1;
        sh.drop_stage = (int)dbg.w - 1;
        mbar_fence_init();
    }
    __syncthreads();
    ST st(P, sh, ring, trace_if_on(P.trace) != nullptr);
    const int np = st.np;

    if (tid >= PS_CT) {
        // producer warp: the CTA's whole weight / KV stream, independent of the
        // phases' grid-wide dependencies (it only waits for free ring slots)
        if (tid == PS_CT) st.produce();
        __syncwarp();
    } else {
        for (int p = 0; p < np; ++p) {
            const int k = st.kind(p);
            if (tid == 0 && st.trace) trace_mark(st.trace, p, 0);
            const bool gemv = k != PK_EMBED && k != PK_ATTN;   // GEMV phases wait inside (after their gain loads)
            if (!gemv) {
                if (p > 0) st.grid_wait(p - 1);
                if (tid == 0 && st.trace) trace_mark(st.trace, p, 1);
            }
            if (k == PK_EMBED) {
                if (st.cta == 0) {
                    // the step's first phase: resets, checks, gather (as k_embed)
                    if (tid == 0) *P.err = 0u;
                    if (tid < P.R) {
                        P.amax[tid] = 0ull;
                        P.nonfinite[tid] = 0u;
                    }
                    ST::csync();
                    for (int r = 0; r < P.R; ++r) {
                        int tok = P.slots[r];
                        const int pos = P.slots[P.R + r];
                        if (tok < 0 || tok >= P.V) {
                            if (tid == 0) atomicOr(P.err, FAULT_TOKEN);
                            tok = 0;
                        }
                        if ((pos < 0 || pos >= P.cap) && tid == 0) atomicOr(P.err, FAULT_POS);
                        const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(P.embed) + (size_t)tok * P.d;
                        for (int i = tid * 8; i < P.d; i += PS_CT * 8) {
                            float f[8];
                            Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(e + i), f);
                            *reinterpret_cast<float4*>(P.x + i + (size_t)r * P.d) = make_float4(f[0], f[1], f[2], f[3]);
                            *reinterpret_cast<float4*>(P.x + i + 4 + (size_t)r * P.d) =
                                make_float4(f[4], f[5], f[6], f[7]);
                        }
                    }
                }
            } else if (k == PK_ATTN) {
                ps_attention<HD, G, PAGED, R>(st, st.layer(p));
            } else {
                GvGeom g;
                const int l = k == PK_HEAD ? 0 : st.layer(p);
                st.geom(k, l, g);
                const __nv_bfloat16* w9 = nullptr;
                switch (k) {
                    case PK_QKV:
                        ps_gemv<CPL_D, PRO_RMSNORM, EPI_STORE>(st, g, P.x,
                            reinterpret_cast<const __nv_bfloat16*>(P.lw[l * 9 + 0]), P.qkv, p);
                        break;
                    case PK_O:
                        ps_gemv<CPL_D, PRO_PLAIN, EPI_ADD>(st, g, P.attn, w9, P.x, p);
                        break;
                    case PK_GU:
                        ps_gemv<CPL_D, PRO_RMSNORM, EPI_SWIGLU_PAIR>(st, g, P.x,
                            reinterpret_cast<const __nv_bfloat16*>(P.lw[l * 9 + 5]), P.gu, p);
                        break;
                    case PK_DOWN:
                        ps_gemv<CPL_F, PRO_PLAIN, EPI_ADD>(st, g, P.gu, w9, P.x, p);
                        break;
                    default:
                        ps_gemv<CPL_D, PRO_RMSNORM, EPI_LOGITS>(st, g, P.x,
                            reinterpret_cast<const __nv_bfloat16*>(P.final_norm), P.logits, p);
                        break;
                }
            }
            st.grid_arrive(p);
            if (tid == 0 && st.trace) {
                trace_mark(st.trace, p, 2);
                trace_mark(st.trace, p, 3);
            }
        }
    }
    __syncthreads();   // the producer has seen its last copy land
    // the last CTA out resets the grid counters for the next replay
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(P.bar + np, 1u);
        if (prev == (unsigned)gridDim.x - 1u) {
            for (int p = 0; p <= np + 2; ++p) P.bar[p] = 0u;
            for (int i = 0; i < P.R * P.Hkv; ++i) P.counters[i] = 0u;
            __threadfence();
        }
    }
}

// ---------------- host side ----------------

template <int CPL_D, int CPL_F, int HD, int G>
static const void* ps_pick_paged(bool paged) {
    return paged ? (const void*)&k_persist<CPL_D, CPL_F, HD, G, true, 1>
                 : (const void*)&k_persist<CPL_D, CPL_F, HD, G, false, 1>;
}
// instantiated shapes: (d, F, hd, G) of the 8B-shape and 1B-class decoders at
// one row; the 1B-class decoder with contiguous K/V also at 2 and 4 rows (its
// down projection's K-slice of 4 rows is 128 activations per thread, the
// most the register file holds next to the rest)
static const void* ps_pick(int cpl_d, int cpl_f, int hd, int G, bool paged, int R) {
    if (R == 1) {
        if (cpl_d == 2 && cpl_f == 7 && hd == 128 && G == 4) return ps_pick_paged<2, 7, 128, 4>(paged);
        if (cpl_d == 1 && cpl_f == 4 && hd == 64 && G == 4) return ps_pick_paged<1, 4, 64, 4>(paged);
        return nullptr;
    }
    if (!paged && cpl_d == 1 && cpl_f == 4 && hd == 64 && G == 4) {
        if (R == 2) return (const void*)&k_persist<1, 4, 64, 4, false, 2>;
        if (R == 4) return (const void*)&k_persist<1, 4, 64, 4, false, 4>;
    }
    return nullptr;
}

static int cpl_of(int K) { return (K / (PS_SL * 8) + 31) / 32; }

cudaError_t persist_plan(PersistPlan* plan, int num_sms) {
    PersistParams& p = plan->p;
    if (p.Hq * p.hd != p.d) return cudaErrorNotSupported;   // O-proj uses the d-column variant
    if (p.d % (PS_SL * 8 * 32) || p.F % (PS_SL * 8 * 32)) return cudaErrorNotSupported;
    const int cd = cpl_of(p.d), cf = cpl_of(p.F);
    if (p.d / (PS_SL * 8) != 32 * cd || p.F / (PS_SL * 8) != 32 * cf) return cudaErrorNotSupported;
    const int G = p.Hq / p.Hkv;
    const void* fn = ps_pick(cd, cf, p.hd, G, p.paged != 0, p.R);
    if (!fn) return cudaErrorNotSupported;
    // rows per 64 KB stage (whole rows, a multiple of the row groups' loads)
    auto rps_for = [&](int K, int cpl) {
        int r = PS_SLOT / (K * 2);
        if (r > PS_MAX_RPS) r = PS_MAX_RPS;
        int ru0 = PS_SLOT / (4096 * cpl), ru = 1;   // the kernel's rows per pass
        while (ru * 2 <= ru0 && ru < 16) ru *= 2;
        if (r >= ru) r -= r % ru;
        return r;
    };
    p.rps_d = rps_for(p.d, cd);
    p.rps_f = rps_for(p.F, cf);
    if (p.rps_d < 1 || p.rps_f < 1) return cudaErrorNotSupported;
    // gate/up: a CTA's gate and up rows are added in one flush
    if (2 * ((p.F + num_sms - 1) / num_sms) > (PS_RED_ROWS / p.rps_d) * p.rps_d) return cudaErrorNotSupported;
    // attention splits: whole half-stages; units spread over the grid
    const int pps = PS_SLOT / (2 * p.hd * 2), half = pps / 2;
    if (p.paged ? (pps % p.page != 0 || p.cap % p.page != 0) : (p.cap % half != 0)) return cudaErrorNotSupported;
    const int units0 = p.R * p.Hkv;
    long long best = -1;
    int bl = 0, bn = 0;
    for (int want = 1; want <= PS_MAX_NS; ++want) {
        int L = (p.cap + want - 1) / want;
        L = (L + half - 1) / half * half;
        if (p.paged) L = (L + p.page - 1) / p.page * p.page;
        const int ns = (p.cap + L - 1) / L;
        // one unit per CTA at most: the splits of a group wait for each other
        if (ns > PS_MAX_NS || (long long)units0 * ns > num_sms) continue;
        const long long cost = (long long)L + 16LL * ns;
        if (best < 0 || cost < best) {
            best = cost;
            bl = L;
            bn = ns;
        }
    }
    if (bn == 0) return cudaErrorNotSupported;
    p.split_len = bl;
    p.nsplit = bn;
    plan->grid = num_sms;
    plan->block = PS_THREADS;
    plan->smem = (size_t)PS_S * PS_SLOT + 1024;
    plan->fn = fn;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    if (plan->smem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorNotSupported;
    if ((e = raise_smem_cap(fn)) != cudaSuccess) return e;
    int occ = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, PS_THREADS, plan->smem)) != cudaSuccess) return e;
    if (occ < 1) return cudaErrorNotSupported;
    return cudaSuccess;
}

size_t persist_tmap_bytes(int n_layers) { return (size_t)n_layers * 4 * sizeof(CUtensorMap); }

typedef CUresult (*PsEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// host images of the tensor maps [layer][K|V][full box | half box (or page box)]
cudaError_t persist_tmaps(const PersistParams& p, void* const* kv, void* host_out) {
    void* fptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return cudaErrorNotSupported;
    PsEncodeFn fn = reinterpret_cast<PsEncodeFn>(fptr);
    CUtensorMap* out = static_cast<CUtensorMap*>(host_out);
    const int pps = PS_SLOT / (2 * p.hd * 2);
    const long long rows = p.paged ? (long long)p.num_pages * p.Hkv * p.page : (long long)p.R * p.Hkv * p.cap;
    for (int l = 0; l < p.L; ++l)
        for (int w = 0; w < 2; ++w)
            for (int b = 0; b < 2; ++b) {
                const int box_rows = p.paged ? p.page : (b == 0 ? pps : pps / 2);
                cuuint64_t dims[2] = {(cuuint64_t)p.hd, (cuuint64_t)rows};
                cuuint64_t strides[1] = {(cuuint64_t)p.hd * 2};
                cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
                cuuint32_t estr[2] = {1u, 1u};
                CUresult r = fn(&out[(l * 2 + w) * 2 + b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv[2 * l + w], dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
            }
    return cudaSuccess;
}

cudaError_t persist_launch(const PersistPlan& plan, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.block);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: grid-wide waits always end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<PersistParams*>(&plan.p)};
    return cudaLaunchKernelExC(&cfg, plan.fn, args);
}

}  // namespace gd
