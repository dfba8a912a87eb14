// internal.h -- launch interface between the engine (engine.cu) and the
// kernel translation units.  Host-side only; no torch types anywhere.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include "graphdec.h"

namespace gd {

// Raise a kernel's dynamic shared-memory cap to the device's opt-in limit
// minus its static shared memory.  The cap is per function and shared by every
// handle in the process, so it is raised once to the limit rather than set to
// one plan's size (a smaller later value would break an earlier plan).
inline cudaError_t raise_smem_cap(const void* fn) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    int dev = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
}

enum WType { W_F32 = 0, W_BF16 = 1 };

// ---------------- fused norm + GEMV ----------------
// out[r, n] (=|+=) sum_k W[n, k] * a[r, k] for the rows n of up to three
// weight segments stacked in one output index space (e.g. Wq;Wk;Wv).
// The activation a is built in shared memory by the prologue:
//   PRO_PLAIN   a = act
//   PRO_RMSNORM a = act / sqrt(mean(act^2) + eps) * gain
//   PRO_SWIGLU  a = silu(act[:, :K]) * act[:, K:2K]
enum Prologue { PRO_PLAIN = 0, PRO_RMSNORM = 1, PRO_SWIGLU = 2 };
// Epilogue: store, add into out (residual), or store logits + greedy argmax.
// EPI_SWIGLU (tensor-core GEMV only): segments 0 and 1 are gate and up with the
// same row count F, and out[r, n] = silu(gate_n . a_r) * (up_n . a_r), n < F.
enum Epilogue { EPI_STORE = 0, EPI_ADD = 1, EPI_LOGITS = 2, EPI_SWIGLU = 3 };

struct GemvParams {
    const void* w[3];
    int seg_rows[3];
    int N;                 // total output rows
    int K;                 // reduction length
    int R;                 // activation rows in use (<= the kernel's NR)
    const float* act;      // [R, act_stride] fp32
    int act_stride;
    const void* gain;      // [K] in the weight dtype (PRO_RMSNORM)
    float eps;
    float* out;            // [R, out_stride] fp32
    int out_stride;
    unsigned long long* amax;  // [R] argmax keys (EPI_LOGITS)
    unsigned* nonfinite;       // [R] flags (EPI_LOGITS)
    unsigned* err;             // error word (FAULT_WAIT)
    int rps;                   // weight rows per ring stage (tensor-core GEMV: tiles per row group)
    int stages;                // ring stages
    int tc_bh;                 // box-streamed tensor-core GEMV: rows per box (row group)
    int tc_seg_ranges[3];      // box-streamed tensor-core GEMV: row ranges per segment
    int tc_ws;                 // tensor-core GEMV: weight columns per stage
    int tc_ks;                 // tensor-core GEMV: K splits (CTAs per row range)
    float* tc_part;            // tensor-core GEMV, tc_ks > 1: partial sums [ks][R][N or 2F] + [ks][ranges][8] sums of squares
    size_t tc_part_cap;        // floats available at tc_part
    unsigned* tc_cnt;          // tensor-core GEMV, tc_ks > 1: arrivals per row range (zero between launches)
    unsigned long long* trace; // trace buffer or null
    int trace_id;
};

struct GemvPlan {
    int wtype, pro, epi, nr, cpl;
    int tc;                // 1: tensor-core GEMV (gemv_tc.cu), 2: box-streamed tensor-core GEMV (gemv_tma.cu)
    alignas(64) unsigned char tma_maps[3 * 128];   // tc == 2: one TMA tensor map per weight segment
    int grid, block;
    size_t smem;
    GemvParams p;
};

// Fill plan->grid/block/smem/nr/cpl and p.rps/p.stages for the given shape.
cudaError_t gemv_plan(GemvPlan* plan, int num_sms);
// Scratch of the tensor-core GEMV for rows x (K -> N) (paired: N = 2F): floats
// of split partials, and the arrival counters (words), for any device.
size_t gemv_tc_part_floats(int R, int K, int N, bool paired);
// the same for the box-streamed tensor-core GEMV (it splits K up to 16 ways)
size_t gemv_box_part_floats(int R, int K, int N);
constexpr size_t GEMV_TC_CNT_WORDS = 1024;
cudaError_t gemv_launch(const GemvPlan& plan, cudaStream_t s, bool pdl);

// ---------------- split-KV masked decode attention ----------------
struct AttnParams {
    const float* qkv;      // [R, qkv_stride]: q [Hq*hd], k [Hkv*hd], v [Hkv*hd] (fp32, pre-RoPE)
    int qkv_stride;
    void* Kc;              // this layer's K store (layout per `paged`)
    void* Vc;
    const int* pos;        // [R] slot
    const int* slot_map;   // [R, pages_per_row] slot (paged)
    const int* write_map;  // [R] slot (paged)
    const float2* rope;    // [cap, hd/2] (cos, sin)
    int cap, R, Hq, Hkv, hd;
    int split_len, nsplit;
    int stages;            // ring stages
    int page_size, pages_per_row, num_pages;
    float* part;           // [R, Hq, nsplit, hd + 2] partial (m, l, o)
    unsigned* counters;    // [R, Hkv] split-completion counters (zero between steps)
    float* out;            // [R, Hq * hd]
    unsigned* err;
    int kv_prewritten;     // 1: every row's new k, v are already in the store (k_kv_write ran)
    int pos_bound;         // 1: a split loads no K/V tile after the one holding pos (DEC_SWEEP_POS)
    float scale;
    unsigned long long* trace;
    int trace_id;
};

struct AttnPlan {
    int kvtype;   // W_F32 / W_BF16
    bool paged;
    int group;    // Hq / Hkv
    dim3 grid;
    int block;
    size_t smem;
    AttnParams p;
    bool mma = false;              // tensor-core kernel (attn_mma.cu)
    void* mma_params = nullptr;    // its parameter block (tensor maps + p), owned by the plan
    bool prewrite = false;         // launch k_kv_write before the attention (p.kv_prewritten = 1)
};

// RoPE of every row's k at Pos, rounding and store of k, v (bf16 store) at the
// row's position or WriteMap slot, before the attention of any row reads them
cudaError_t kv_write_launch(const AttnPlan& plan, cudaStream_t s, bool pdl);

// choose split_len / nsplit; returns cudaErrorInvalidValue for unsupported head_dim / group
cudaError_t attn_plan(AttnPlan* plan, int num_sms);
cudaError_t attn_launch(const AttnPlan& plan, cudaStream_t s, bool pdl);
size_t attn_part_floats(int R, int Hq, int hd, int nsplit);

// tensor-core variant for bf16 K/V (head_dim 64 or 128)
bool attn_mma_supported(int kvtype, int hd, int G, bool paged, int page_size);
cudaError_t attn_mma_plan(AttnPlan* plan, int num_sms);
cudaError_t attn_mma_launch(const AttnPlan& plan, cudaStream_t s, bool pdl);
void attn_mma_release(AttnPlan& plan);

// ---------------- embedding gather + per-step resets ----------------
struct EmbedParams {
    const void* E;         // [V, d] weight dtype
    const int* tok;        // [R]
    const int* pos;        // [R]
    int R, V, d, cap;
    float* x;              // [R, d]
    unsigned* err;
    unsigned long long* amax;
    unsigned* nonfinite;
    unsigned long long* trace;
    int trace_id;
};
cudaError_t embed_launch(int wtype, const EmbedParams& p, cudaStream_t s);

// ---------------- sampling suffix ----------------
struct SamplerSlot {                 // device copy of dec_sampler (same field order)
    float temperature;
    int top_k;
    float top_p;
    float min_p;
    unsigned long long seed;
    int n_logprobs;
    int reserved;
};
struct SampleParams {
    const float* logits;             // [R, V]
    int V, R;
    const unsigned long long* amax;  // [R] greedy keys
    const int* pos;                  // [R] Pos slot (the uniform's counter)
    const SamplerSlot* cfg;          // parameter slot
    int* sampled;                    // [R] picks
    int* lp_ids;                     // [R, DEC_LOGPROBS_MAX]
    float* lp_vals;                  // [R, DEC_LOGPROBS_MAX]
};
cudaError_t sample_launch(const SampleParams& p, cudaStream_t s);

// ---------------- chained greedy steps ----------------
struct ChainParams {
    int* tok;                        // [R] Token slot
    int* pos;                        // [R] Pos slot
    int* wm;                         // [R] WriteMap slot (paged)
    const int* slot_map;             // [R, ppr] SlotMap (paged) or null
    int R, V, cap, ppr, page;
    const unsigned long long* amax;  // [R] greedy keys of the step just run
    const unsigned* nonfinite;       // [R]
    unsigned* err;                   // the step's error word
    unsigned* chain_err;             // sticky over the chain
    const int* sampled;              // [R] sampled ids, or null: greedy keys
    int* counter;                    // steps recorded so far
    int* ids;                        // [max_steps, R] history
    int* nf;                         // [max_steps, R] history
    int max_steps;
};
cudaError_t chain_advance_launch(const ChainParams& p, cudaStream_t s);

// a kernel that spins for about `ns` nanoseconds on one SM, then returns
cudaError_t busy_launch(long long ns, cudaStream_t s);

// ---------------- the whole step as one persistent kernel ----------------
struct PersistParams {
    int L, d, F, V, Hq, Hkv, hd, R, cap;
    int paged, page, pages_per_row, num_pages;
    float eps, scale;
    const void* const* lw;     // [L * 9] device table: attn_norm, q, k, v, o, ffn_norm, gate, up, down
    const void* embed;
    const void* final_norm;
    const void* lm_head;
    float* x;
    float* qkv;
    float* attn;
    float* gu;
    float* logits;
    float* part;
    unsigned* counters;        // [R * Hkv] split completion
    const int* slots;          // tokens [R], pos [R], write map [R]
    const int* slot_map;
    const float2* rope;
    void* const* kv;           // [L * 2] device table: K, V store of each layer
    const void* tmaps;         // [L][K|V][2] tensor maps in device memory (64-byte aligned)
    unsigned* err;
    unsigned long long* amax;
    unsigned* nonfinite;
    unsigned* bar;             // [5L + 5]: per-phase arrivals, exit counter, abort word, head block counter
    unsigned long long* trace;
    int split_len, nsplit;
    int rps_d, rps_f;          // weight rows per ring stage for K = d and K = F
    const unsigned* dbg;       // [4] wait bounds and test hooks: grid-wait polls, ring-wait polls (0: defaults),
                               // phase whose grid-wait target is raised by one + 1, stage CTA 0 never issues + 1
                               // (0: none); 16-byte aligned
};

struct PersistPlan {
    PersistParams p;
    int grid = 0, block = 0;
    size_t smem = 0;
    const void* fn = nullptr;
};

// fills split_len / nsplit / rps_* and the launch shape; cudaErrorNotSupported
// when this shape has no persistent kernel
cudaError_t persist_plan(PersistPlan* plan, int num_sms);
size_t persist_tmap_bytes(int n_layers);
// host images of the layer tensor maps (written to the device table by the caller)
cudaError_t persist_tmaps(const PersistParams& p, void* const* kv, void* host_out);
cudaError_t persist_launch(const PersistPlan& plan, cudaStream_t s);

// ---------------- multi-token prefill of one sequence (prefill.cu) ----------------
struct PrefillArgs {
    int L, d, Hq, Hkv, hd, F, cap;
    float eps;
    const void* embed;          // [V, d] bf16
    const void* const* lw;      // host array [L * 9] of device pointers: attn_norm, q, k, v, o, ffn_norm, gate, up, down
    void* const* K;             // host array [L] of device pointers: K store of each layer
    void* const* V;             // host array [L]: V store
    bool paged;
    int page, ppr;              // paged: tokens per page, pages per sequence
    int rows, num_pages;        // contiguous: the capture's rows; paged: the pool's pages
    const float2* rope;         // device [cap, hd / 2]
    unsigned* err;              // device error word
};
struct PrefillState;
// whether this shape has a block prefill (bf16 weights and K/V are the caller's check)
bool prefill_supported(const PrefillArgs& a);
// device buffers and tensor maps of the block prefill (cudaMalloc; freed by prefill_free)
cudaError_t prefill_create(const PrefillArgs& a, int num_sms, PrefillState** out);
void prefill_free(PrefillState* s);
// n tokens (host) at positions pos0 .. pos0 + n - 1 of sequence `row` (contiguous
// K/V) or of the sequence on `pages` (host, paged K/V): every layer's K/V of those
// positions written; the last token's hidden state (fp32 [d]) to x_last (device)
cudaError_t prefill_run(PrefillState* s, const int* tokens, int n, int pos0, int row, const int* pages, float* x_last,
                        cudaStream_t st);

}  // namespace gd

struct dec_handle;
namespace gd {
// engine services for other translation units of the library
int engine_run_attention(dec_handle* h, int32_t layer, const float* qkv, const int32_t* pos, float* out, float* part,
                         unsigned* counters);
void engine_attention_scratch(const dec_handle* h, size_t* part_floats, size_t* counters);
int engine_gate(dec_handle* h);
int engine_fail(dec_handle* h, int code, const char* msg);
int engine_device(const dec_handle* h);

}  // namespace gd
