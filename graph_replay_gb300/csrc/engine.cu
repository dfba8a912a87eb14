// engine.cu -- the C ABI of graphdec.h: configuration checks, weight binding
// by role, step buffers, capture into one CUDA graph, per-token replay with
// slot writes and bounded waits, and the failure states.
//
// The executor contract follows "Execution" (sections "Slot buffers",
// "Per backend" -- PTX row: cuStreamBeginCapture, launch every plan,
// instantiate; per token: write slots, graph launch, copy results, sync --
// and "Failure handling"), and "Backends", section "PTX (NVIDIA)" (kernel
// arguments point at stable slot buffers that the host rewrites in place).
// Kernels receive only pointers to slots, never a position by value, so one
// recorded graph serves every position ("Execution", section "Slot buffers":
// a scalar that depends on a slot is bound to the slot buffer).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <array>
#include <chrono>
#include <cmath>
#include <string>
#include <thread>
#include <vector>

#include "graphdec.h"
#include "internal.h"

using namespace gd;

namespace {

thread_local std::string g_init_msg;   // message of the last failed dec_init on this thread

constexpr int ST_READY = 0, ST_NEEDS_RESET = 1, ST_POISONED = 2;
constexpr int MAX_ROWS = 8;
constexpr int CHAIN_MAX = DEC_CHAIN_MAX_STEPS;   // steps one dec_chain call records
constexpr size_t ALIGN = 256;

// per-step status block read back after every step (one copy)
static_assert(sizeof(dec_sampler) == sizeof(SamplerSlot), "the sampler slot mirrors dec_sampler");
static_assert(offsetof(dec_sampler, seed) == offsetof(SamplerSlot, seed), "the sampler slot mirrors dec_sampler");
static_assert(offsetof(dec_sampler, n_logprobs) == offsetof(SamplerSlot, n_logprobs), "the sampler slot mirrors dec_sampler");

struct StatusBlock {
    unsigned err;
    unsigned pad;
    unsigned long long amax[MAX_ROWS];
    unsigned nonfinite[MAX_ROWS];
    int sampled[MAX_ROWS];                        // sampling suffix: the picks
    int lp_ids[MAX_ROWS * DEC_LOGPROBS_MAX];      // top-n logprob ids
    float lp_vals[MAX_ROWS * DEC_LOGPROBS_MAX];   // and values
};

size_t align_up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }

int es_of(int dtype) { return dtype == DEC_DTYPE_BF16 ? 2 : 4; }

// Offsets of every buffer of a capture inside one workspace.
struct WsLayout {
    size_t status, slots, slot_map, counters, trace, ptabs, tmaps, gbar, dbg, x, qkv, attn, gu, logits, part, gpart,
        gcnt, chain, sampler, rope, kv, kv_layer, total;
};

// kernels recorded per step: embedding, 5 per layer, head
int kernels_per_step(int n_layers) { return 2 + 5 * n_layers; }

bool compute_layout(const dec_config& c, int cap, int R, int layout, int page, int npages, WsLayout* L) {
    const size_t hd = (size_t)c.head_dim, Hq = (size_t)c.n_heads, Hkv = (size_t)c.n_kv_heads;
    const size_t d = (size_t)c.d_model, F = (size_t)c.ffn_hidden, V = (size_t)c.vocab;
    const size_t max_splits = ((size_t)cap + 63) / 64;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    L->status = take(sizeof(StatusBlock));
    L->slots = take(3 * (size_t)R * sizeof(int32_t));
    L->slot_map = take(layout == DEC_KV_PAGED ? (size_t)R * (cap / page) * sizeof(int32_t) : 0);
    L->counters = take((size_t)R * Hkv * sizeof(unsigned));
    L->trace = take((1 + 4 * (size_t)kernels_per_step(c.n_layers)) * sizeof(unsigned long long));
    // persistent-kernel tables: weight and KV pointers, tensor maps, grid counters
    L->ptabs = take((size_t)c.n_layers * 11 * sizeof(void*));
    L->tmaps = take(persist_tmap_bytes(c.n_layers));
    L->gbar = take(((size_t)kernels_per_step(c.n_layers) + 3) * sizeof(unsigned));
    L->dbg = take(4 * sizeof(unsigned));   // persistent kernel: wait bounds and test hooks (zero: defaults)
    L->x = take((size_t)R * d * 4);
    L->qkv = take((size_t)R * (Hq + 2 * Hkv) * hd * 4);
    L->attn = take((size_t)R * Hq * hd * 4);
    L->gu = take((size_t)R * 2 * F * 4);
    L->logits = take((size_t)R * V * 4);
    L->part = take(attn_part_floats(R, (int)Hq, (int)hd, (int)max_splits) * 4);
    // split-K partial sums of the tensor-core GEMV (bf16, 2..8 rows): the largest projection's need
    size_t gp = 0;
    if (c.weight_dtype == DEC_DTYPE_BF16 && R >= 2) {
        const int qkv_n = (int)((Hq + 2 * Hkv) * hd);
        for (size_t need : {gemv_tc_part_floats(R, (int)d, qkv_n, false), gemv_tc_part_floats(R, (int)(Hq * hd), (int)d, false),
                            gemv_tc_part_floats(R, (int)d, (int)(2 * F), true), gemv_tc_part_floats(R, (int)F, (int)d, false),
                            gemv_tc_part_floats(R, (int)d, (int)V, false), gemv_box_part_floats(R, (int)d, qkv_n),
                            gemv_box_part_floats(R, (int)(Hq * hd), (int)d), gemv_box_part_floats(R, (int)d, (int)(2 * F)),
                            gemv_box_part_floats(R, (int)F, (int)d), gemv_box_part_floats(R, (int)d, (int)V)})
            gp = need > gp ? need : gp;
    }
    L->gpart = take(gp * 4);
    L->gcnt = take(gp ? GEMV_TC_CNT_WORDS * sizeof(unsigned) : 0);
    // chained steps: counter, sticky error word, id and flag histories
    L->chain = take(2 * sizeof(int) + 2 * (size_t)CHAIN_MAX * R * sizeof(int));
    L->sampler = take(sizeof(SamplerSlot));
    L->rope = take((size_t)cap * (hd / 2) * sizeof(float2));
    const size_t es = (size_t)es_of(c.kv_dtype);
    if (layout == DEC_KV_PAGED)
        L->kv_layer = align_up((size_t)npages * Hkv * page * hd * es);
    else
        L->kv_layer = align_up((size_t)R * Hkv * cap * hd * es);
    L->kv = take(0);
    o += 2 * (size_t)c.n_layers * L->kv_layer;
    L->total = o;
    return true;
}

}  // namespace

struct dec_handle {
    dec_config cfg{};
    std::string msg;
    int state = ST_READY;
    uint32_t last_fault = 0;
    int num_sms = 0;
    bool pdl = true;
    bool eager = false;
    int strategy = DEC_STRATEGY_GRAPH;
    int kv_sweep = DEC_SWEEP_CAP;
    PersistPlan persist;

    // weights by role
    const void* embed = nullptr;
    const void* final_norm = nullptr;
    const void* lm_head = nullptr;
    std::vector<std::array<const void*, 9>> lw;   // roles DEC_W_ATTN_NORM .. DEC_W_DOWN

    // capture
    bool captured = false;
    int cap = 0, rows = 0, layout = 0, page = 0, npages = 0, ppr = 0;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    char* ws = nullptr;
    bool own_ws = false;
    int extra_kernels = 0;         // recorded kernels without a trace slot (K/V writes, sampling)
    bool sampler_on = false;       // the sampling kernel is (to be) recorded after the head
    dec_sampler sampler{};         // its parameters
    WsLayout lay{};
    StatusBlock* d_status = nullptr;
    int32_t* d_slots = nullptr;
    int32_t* d_slot_map = nullptr;
    unsigned* d_counters = nullptr;
    unsigned long long* d_trace = nullptr;
    float *d_x = nullptr, *d_qkv = nullptr, *d_attn = nullptr, *d_gu = nullptr, *d_logits = nullptr;
    float* d_part = nullptr;
    float2* d_rope = nullptr;
    std::vector<void*> K, V;

    // pinned host staging
    int32_t* h_slots = nullptr;
    StatusBlock* h_status = nullptr;
    float* h_logits = nullptr;
    int* h_chain = nullptr;        // pinned: [2 + 2 * CHAIN_MAX * rows] chain read-back
    std::vector<int32_t> slot_map_host;

    // recorded launches
    EmbedParams embed_p{};
    std::vector<GemvPlan> gemv;   // 4 per layer (qkv, o, gate/up, down) + head
    std::vector<AttnPlan> attn;   // 1 per layer
    int kernels = 0;

    PrefillState* pf = nullptr;    // block prefill buffers (created by the first dec_prefill_block)

    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    size_t nodes = 0;
    cudaEvent_t ev = nullptr;

    int64_t steps = 0, replays = 0, eager_steps = 0;
    double last_step_us = 0.0;
};

namespace {

int fail(dec_handle* h, int code, const char* fmt, ...) {
    if (h) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        h->msg = buf;
    }
    return code;
}

// A CUDA runtime error is treated as sticky: the handle is poisoned and every
// later call is refused without touching the device ("Execution", section
// "Failure handling": on PTX a fault is a sticky CUDA error).
int cuda_fail(dec_handle* h, cudaError_t e, const char* what) {
    h->state = ST_POISONED;
    return fail(h, DEC_E_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int gate(dec_handle* h, bool need_capture) {
    if (!h) return DEC_E_INVALID;
    if (h->state == ST_POISONED) return fail(h, DEC_E_POISONED, "handle is poisoned by an earlier device error or timeout");
    if (need_capture && !h->captured) return fail(h, DEC_E_STATE, "dec_capture has not run");
    return DEC_OK;
}

// Every wait on the device is bounded ("Execution", section "Failure
// handling": a wait that outlasts the configured timeout fails with a typed
// timeout error and poisons the context).
int bounded_wait(dec_handle* h) {
    cudaError_t e = cudaEventRecord(h->ev, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventRecord");
    const auto t0 = std::chrono::steady_clock::now();
    for (uint64_t it = 0;; ++it) {
        e = cudaEventQuery(h->ev);
        if (e == cudaSuccess) return DEC_OK;
        if (e != cudaErrorNotReady) return cuda_fail(h, e, "device wait");
        if ((it & 31) == 0) {
            const double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
            if (ms > (double)h->cfg.wait_timeout_ms) {
                h->state = ST_POISONED;
                return fail(h, DEC_E_TIMEOUT, "device wait exceeded %lld ms; handle poisoned",
                            (long long)h->cfg.wait_timeout_ms);
            }
            // a step takes milliseconds: poll (yielding the core) for the first 50 ms,
            // since a sleep wakes tens of microseconds late; sleep after that
            if (ms > 50.0)
                std::this_thread::sleep_for(std::chrono::microseconds(20));
            else
                std::this_thread::yield();
        }
    }
}

// Host -> device copy ordered on the handle's stream, waited for (bounded): the
// source may change as soon as this returns, and the handle's non-blocking
// stream does not order itself after a legacy-stream cudaMemcpy.
int h2d_wait(dec_handle* h, void* dst, const void* src, size_t bytes, const char* what) {
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, what);
    return bounded_wait(h);
}

int validate_config(const dec_config* c, dec_handle* h) {
    if (!c) return fail(h, DEC_E_INVALID, "config is NULL");
    if (c->n_layers < 1) return fail(h, DEC_E_INVALID, "n_layers must be >= 1");
    if (c->d_model < 1) return fail(h, DEC_E_INVALID, "d_model must be >= 1");
    if (c->n_heads < 1 || c->n_kv_heads < 1) return fail(h, DEC_E_INVALID, "n_heads and n_kv_heads must be >= 1");
    if (c->n_heads % c->n_kv_heads) return fail(h, DEC_E_INVALID, "n_kv_heads must divide n_heads");
    if (c->head_dim < 2 || (c->head_dim & 1)) return fail(h, DEC_E_INVALID, "head_dim must be even and >= 2");
    if (c->ffn_hidden < 1) return fail(h, DEC_E_INVALID, "ffn_hidden must be >= 1");
    if (c->vocab < 1) return fail(h, DEC_E_INVALID, "vocab must be >= 1");
    if (c->weight_dtype != DEC_DTYPE_F32 && c->weight_dtype != DEC_DTYPE_BF16)
        return fail(h, DEC_E_INVALID, "weight_dtype must be DEC_DTYPE_F32 or DEC_DTYPE_BF16");
    if (c->kv_dtype != DEC_DTYPE_F32 && c->kv_dtype != DEC_DTYPE_BF16)
        return fail(h, DEC_E_INVALID, "kv_dtype must be DEC_DTYPE_F32 or DEC_DTYPE_BF16");
    if (!(c->rms_eps >= 0.0) || !std::isfinite(c->rms_eps)) return fail(h, DEC_E_INVALID, "rms_eps must be finite and >= 0");
    if (!(c->rope_theta > 0.0) || !std::isfinite(c->rope_theta)) return fail(h, DEC_E_INVALID, "rope_theta must be finite and > 0");
    if (c->device < 0) return fail(h, DEC_E_INVALID, "device must be >= 0");
    // what the kernels of this library can run
    const int hd = c->head_dim;
    if (hd != 16 && hd != 32 && hd != 64 && hd != 128)
        return fail(h, DEC_E_UNSUPPORTED, "head_dim %d unsupported (16, 32, 64 or 128)", hd);
    const int G = c->n_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(h, DEC_E_UNSUPPORTED, "n_heads / n_kv_heads = %d unsupported (1, 2, 4 or 8)", G);
    const int vec = c->weight_dtype == DEC_DTYPE_BF16 ? 8 : 4;
    if (c->d_model % vec) return fail(h, DEC_E_UNSUPPORTED, "d_model must be a multiple of %d", vec);
    if (c->ffn_hidden % vec) return fail(h, DEC_E_UNSUPPORTED, "ffn_hidden must be a multiple of %d", vec);
    if ((c->n_heads * hd) % vec) return fail(h, DEC_E_UNSUPPORTED, "n_heads * head_dim must be a multiple of %d", vec);
    return DEC_OK;
}

bool shape_ok(const dec_config& c, int role, int64_t rows, int64_t cols) {
    const int64_t d = c.d_model, F = c.ffn_hidden, V = c.vocab;
    const int64_t qd = (int64_t)c.n_heads * c.head_dim, kvd = (int64_t)c.n_kv_heads * c.head_dim;
    auto vec = [&](int64_t n) { return (rows == n && cols == 1) || (rows == 1 && cols == n); };
    switch (role) {
        case DEC_W_EMBED: case DEC_W_LM_HEAD: return rows == V && cols == d;
        case DEC_W_ATTN_NORM: case DEC_W_FFN_NORM: case DEC_W_FINAL_NORM: return vec(d);
        case DEC_W_Q: return rows == qd && cols == d;
        case DEC_W_K: case DEC_W_V: return rows == kvd && cols == d;
        case DEC_W_O: return rows == d && cols == qd;
        case DEC_W_GATE: case DEC_W_UP: return rows == F && cols == d;
        case DEC_W_DOWN: return rows == d && cols == F;
    }
    return false;
}

const char* role_name(int role) {
    static const char* names[] = {"EMBED", "ATTN_NORM", "Q", "K", "V", "O", "FFN_NORM",
                                  "GATE", "UP", "DOWN", "FINAL_NORM", "LM_HEAD"};
    return (role >= 0 && role < DEC_W_NROLES) ? names[role] : "?";
}

// RoPE table [cap, hd/2] of (cos, sin)(pos * theta^(-2i/hd)), built in fp64
// and rounded to fp32 (avoids large-argument fp32 trigonometry on the device).
std::vector<float2> rope_table(int cap, int hd, double theta) {
    std::vector<float2> t((size_t)cap * (hd / 2));
    for (int i = 0; i < hd / 2; ++i) {
        const double w = std::pow(theta, -2.0 * i / hd);
        for (int p = 0; p < cap; ++p) {
            const double a = (double)p * w;
            t[(size_t)p * (hd / 2) + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
    }
    return t;
}

cudaError_t launch_attn(const AttnPlan& a, cudaStream_t s, bool pdl) {
    if (a.prewrite) {
        cudaError_t e = kv_write_launch(a, s, pdl);
        if (e != cudaSuccess) return e;
    }
    return a.mma ? attn_mma_launch(a, s, pdl) : attn_launch(a, s, pdl);
}

// launch the whole step (the sequence the graph records)
cudaError_t enqueue_step(dec_handle* h) {
    cudaError_t e;
    if (h->strategy == DEC_STRATEGY_PERSISTENT) {
        if ((e = persist_launch(h->persist, h->stream)) != cudaSuccess) return e;
    } else {
        if ((e = embed_launch(h->cfg.weight_dtype == DEC_DTYPE_BF16 ? W_BF16 : W_F32, h->embed_p, h->stream)) !=
            cudaSuccess)
            return e;
        for (int l = 0; l < h->cfg.n_layers; ++l) {
            if ((e = gemv_launch(h->gemv[4 * l + 0], h->stream, h->pdl)) != cudaSuccess) return e;
            if ((e = launch_attn(h->attn[l], h->stream, h->pdl)) != cudaSuccess) return e;
            if ((e = gemv_launch(h->gemv[4 * l + 1], h->stream, h->pdl)) != cudaSuccess) return e;
            if ((e = gemv_launch(h->gemv[4 * l + 2], h->stream, h->pdl)) != cudaSuccess) return e;
            if ((e = gemv_launch(h->gemv[4 * l + 3], h->stream, h->pdl)) != cudaSuccess) return e;
        }
        if ((e = gemv_launch(h->gemv.back(), h->stream, h->pdl)) != cudaSuccess) return e;
    }
    if (h->sampler_on) {
        SampleParams sp{};
        sp.logits = h->d_logits;
        sp.V = h->cfg.vocab;
        sp.R = h->rows;
        sp.amax = h->d_status->amax;
        sp.pos = h->d_slots + h->rows;
        sp.cfg = reinterpret_cast<const SamplerSlot*>(h->ws + h->lay.sampler);
        sp.sampled = h->d_status->sampled;
        sp.lp_ids = h->d_status->lp_ids;
        sp.lp_vals = h->d_status->lp_vals;
        if ((e = sample_launch(sp, h->stream)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t zero_state(dec_handle* h) {
    cudaError_t e;
    for (int l = 0; l < h->cfg.n_layers; ++l) {
        if ((e = cudaMemsetAsync(h->K[l], 0, h->lay.kv_layer, h->stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(h->V[l], 0, h->lay.kv_layer, h->stream)) != cudaSuccess) return e;
    }
    if ((e = cudaMemsetAsync(h->d_status, 0, sizeof(StatusBlock), h->stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(h->ws + h->lay.gbar, 0, ((size_t)h->kernels + 3) * sizeof(unsigned), h->stream)) !=
        cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(h->d_slots, 0, 3 * sizeof(int32_t) * h->rows, h->stream)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(h->d_counters, 0, sizeof(unsigned) * h->rows * h->cfg.n_kv_heads, h->stream)) != cudaSuccess)
        return e;
    if (h->lay.gcnt != h->lay.gpart &&
        (e = cudaMemsetAsync(h->ws + h->lay.gcnt, 0, GEMV_TC_CNT_WORDS * sizeof(unsigned), h->stream)) != cudaSuccess)
        return e;
    return cudaMemsetAsync(h->d_x, 0, sizeof(float) * h->rows * h->cfg.d_model, h->stream);
}

// launch one step (graph replay or the same kernels eagerly)
int launch_step(dec_handle* h) {
    cudaError_t e;
    if (h->eager) {
        e = enqueue_step(h);
        if (e != cudaSuccess) return cuda_fail(h, e, "eager step launch");
        ++h->eager_steps;
    } else {
        e = cudaGraphLaunch(h->exec, h->stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaGraphLaunch");
        ++h->replays;
    }
    return DEC_OK;
}

// copy back the status block (and logits), wait, and check the error word
int finish_step(dec_handle* h, float* logits_out, int32_t* ids_out, uint8_t* nonfinite_out) {
    cudaError_t e = cudaMemcpyAsync(h->h_status, h->d_status, sizeof(StatusBlock), cudaMemcpyDeviceToHost, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "status readback");
    const size_t lbytes = (size_t)h->rows * h->cfg.vocab * sizeof(float);
    if (logits_out) {
        e = cudaMemcpyAsync(h->h_logits, h->d_logits, lbytes, cudaMemcpyDeviceToHost, h->stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "logits readback");
    }
    int rc = bounded_wait(h);
    if (rc != DEC_OK) return rc;
    ++h->steps;
    if (h->h_status->err) {
        h->last_fault = h->h_status->err;
        h->state = ST_NEEDS_RESET;
        return fail(h, DEC_E_DEVICE_FAULT, "device check failed (error word 0x%x); results discarded, reset needed",
                    h->h_status->err);
    }
    if (logits_out) memcpy(logits_out, h->h_logits, lbytes);
    for (int r = 0; r < h->rows; ++r) {
        if (ids_out) {
            const unsigned long long k = h->h_status->amax[r];
            ids_out[r] = h->sampler_on ? h->h_status->sampled[r]
                                       : (k ? (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull)) : -1);
        }
        if (nonfinite_out) nonfinite_out[r] = h->h_status->nonfinite[r] ? 1 : 0;
    }
    return DEC_OK;
}

}  // namespace

extern "C" {

int dec_init(const dec_config* cfg, dec_handle** out) {
    if (!out) return DEC_E_INVALID;
    *out = nullptr;
    dec_handle tmp;
    int rc = validate_config(cfg, &tmp);
    if (rc != DEC_OK) {
        g_init_msg = tmp.msg;
        return rc;
    }
    dec_handle* h = new dec_handle();
    h->cfg = *cfg;
    if (h->cfg.wait_timeout_ms <= 0) h->cfg.wait_timeout_ms = 600000;
    h->lw.assign(cfg->n_layers, std::array<const void*, 9>{});
    cudaError_t e = cudaSetDevice(cfg->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
    if (e != cudaSuccess) {
        g_init_msg = std::string("device ") + std::to_string(cfg->device) + ": " + cudaGetErrorString(e);
        delete h;
        return DEC_E_CUDA;
    }
    *out = h;
    return DEC_OK;
}

int dec_load_weights(dec_handle* h, const dec_weight* w, size_t n) {
    int rc = gate(h, false);
    if (rc) return rc;
    if (h->captured) return fail(h, DEC_E_STATE, "weights are bound before dec_capture");
    if (!w && n) return fail(h, DEC_E_INVALID, "binding array is NULL");
    for (size_t i = 0; i < n; ++i) {
        const dec_weight& b = w[i];
        if (b.role < 0 || b.role >= DEC_W_NROLES) return fail(h, DEC_E_INVALID, "binding %zu: unknown role %d", i, b.role);
        const bool global = b.role == DEC_W_EMBED || b.role == DEC_W_FINAL_NORM || b.role == DEC_W_LM_HEAD;
        if (global ? b.layer != -1 : (b.layer < 0 || b.layer >= h->cfg.n_layers))
            return fail(h, DEC_E_INVALID, "binding %zu (%s): bad layer %d", i, role_name(b.role), b.layer);
        if (b.dtype != h->cfg.weight_dtype)
            return fail(h, DEC_E_INVALID, "binding %zu (%s): dtype %d differs from weight_dtype", i, role_name(b.role), b.dtype);
        if (!shape_ok(h->cfg, b.role, b.rows, b.cols))
            return fail(h, DEC_E_INVALID, "binding %zu (%s, layer %d): shape [%lld, %lld] does not match the config", i,
                        role_name(b.role), b.layer, (long long)b.rows, (long long)b.cols);
        if (!b.data || ((uintptr_t)b.data & 15))
            return fail(h, DEC_E_INVALID, "binding %zu (%s): data must be a non-NULL 16-byte aligned device pointer", i,
                        role_name(b.role));
    }
    for (size_t i = 0; i < n; ++i) {
        const dec_weight& b = w[i];
        switch (b.role) {
            case DEC_W_EMBED: h->embed = b.data; break;
            case DEC_W_FINAL_NORM: h->final_norm = b.data; break;
            case DEC_W_LM_HEAD: h->lm_head = b.data; break;
            default: h->lw[b.layer][b.role - DEC_W_ATTN_NORM] = b.data;
        }
    }
    return DEC_OK;
}

int dec_workspace_size(const dec_config* cfg, int32_t cap, int32_t rows, int32_t kv_layout, int32_t page_size,
                       int32_t num_pages, size_t* bytes) {
    if (!bytes) return DEC_E_INVALID;
    if (validate_config(cfg, nullptr) != DEC_OK) return DEC_E_INVALID;
    if (cap < 1 || rows < 1 || rows > MAX_ROWS) return DEC_E_INVALID;
    if (kv_layout == DEC_KV_PAGED && (page_size < 1 || cap % page_size || num_pages < 1)) return DEC_E_INVALID;
    WsLayout L;
    compute_layout(*cfg, cap, rows, kv_layout, page_size, num_pages, &L);
    *bytes = L.total;
    return DEC_OK;
}

int dec_capture(dec_handle* h, int32_t cap, int32_t rows, int32_t kv_layout, int32_t page_size, int32_t num_pages,
                void* workspace, size_t workspace_bytes, void* stream) {
    int rc = gate(h, false);
    if (rc) return rc;
    if (h->captured) return fail(h, DEC_E_STATE, "this handle is already captured (one entry per handle)");
    const dec_config& c = h->cfg;
    if (cap < 1) return fail(h, DEC_E_INVALID, "cap must be >= 1");
    if (rows < 1 || rows > MAX_ROWS) return fail(h, DEC_E_UNSUPPORTED, "rows must be in [1, %d]", MAX_ROWS);
    if (kv_layout != DEC_KV_CONTIGUOUS && kv_layout != DEC_KV_PAGED) return fail(h, DEC_E_INVALID, "unknown kv_layout");
    if (kv_layout == DEC_KV_PAGED) {
        if (page_size < 1 || 64 % page_size) return fail(h, DEC_E_UNSUPPORTED, "page_size must divide 64");
        if (cap % page_size) return fail(h, DEC_E_INVALID, "cap must be a multiple of page_size");
        if (num_pages < rows * (cap / page_size))
            return fail(h, DEC_E_INVALID, "num_pages must hold rows * cap / page_size pages");
        if ((int64_t)num_pages * page_size > INT32_MAX) return fail(h, DEC_E_UNSUPPORTED, "pool too large");
    }
    if ((int64_t)cap * c.head_dim > INT32_MAX) return fail(h, DEC_E_UNSUPPORTED, "cap too large");
    if (!h->embed) return fail(h, DEC_E_INVALID, "weight EMBED is unbound");
    if (!h->final_norm) return fail(h, DEC_E_INVALID, "weight FINAL_NORM is unbound");
    if (!h->lm_head) return fail(h, DEC_E_INVALID, "weight LM_HEAD is unbound");
    for (int l = 0; l < c.n_layers; ++l)
        for (int k = 0; k < 9; ++k)
            if (!h->lw[l][k]) return fail(h, DEC_E_INVALID, "weight %s of layer %d is unbound", role_name(k + 1), l);

    cudaError_t e = cudaSetDevice(c.device);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaSetDevice");
    if (stream) {
        h->stream = (cudaStream_t)stream;
        h->own_stream = false;
    } else {
        if ((e = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(h, e, "cudaStreamCreate");
        h->own_stream = true;
    }
    if ((e = cudaEventCreateWithFlags(&h->ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(h, e, "cudaEventCreate");

    h->cap = cap;
    h->rows = rows;
    h->layout = kv_layout;
    h->page = kv_layout == DEC_KV_PAGED ? page_size : 0;
    h->npages = kv_layout == DEC_KV_PAGED ? num_pages : 0;
    h->ppr = kv_layout == DEC_KV_PAGED ? cap / page_size : 0;
    compute_layout(c, cap, rows, kv_layout, page_size, num_pages, &h->lay);
    if (workspace) {
        if (workspace_bytes < h->lay.total)
            return fail(h, DEC_E_OOM, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, h->lay.total);
        if ((uintptr_t)workspace % ALIGN) return fail(h, DEC_E_INVALID, "workspace must be 256-byte aligned");
        h->ws = (char*)workspace;
        h->own_ws = false;
    } else {
        e = cudaMalloc((void**)&h->ws, h->lay.total);
        if (e != cudaSuccess) {
            cudaGetLastError();
            h->ws = nullptr;
            return fail(h, DEC_E_OOM, "cudaMalloc of %zu bytes failed", h->lay.total);
        }
        h->own_ws = true;
    }
    const WsLayout& L = h->lay;
    h->d_status = (StatusBlock*)(h->ws + L.status);
    h->d_slots = (int32_t*)(h->ws + L.slots);
    h->d_slot_map = kv_layout == DEC_KV_PAGED ? (int32_t*)(h->ws + L.slot_map) : nullptr;
    h->d_counters = (unsigned*)(h->ws + L.counters);
    h->d_trace = (unsigned long long*)(h->ws + L.trace);
    h->d_x = (float*)(h->ws + L.x);
    h->d_qkv = (float*)(h->ws + L.qkv);
    h->d_attn = (float*)(h->ws + L.attn);
    h->d_gu = (float*)(h->ws + L.gu);
    h->d_logits = (float*)(h->ws + L.logits);
    h->d_part = (float*)(h->ws + L.part);
    h->d_rope = (float2*)(h->ws + L.rope);
    h->K.resize(c.n_layers);
    h->V.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        h->K[l] = h->ws + L.kv + (size_t)(2 * l) * L.kv_layer;
        h->V[l] = h->ws + L.kv + (size_t)(2 * l + 1) * L.kv_layer;
    }

    if ((e = cudaHostAlloc((void**)&h->h_slots, 3 * sizeof(int32_t) * rows, cudaHostAllocDefault)) != cudaSuccess)
        return cuda_fail(h, e, "cudaHostAlloc");
    if ((e = cudaHostAlloc((void**)&h->h_status, sizeof(StatusBlock), cudaHostAllocDefault)) != cudaSuccess)
        return cuda_fail(h, e, "cudaHostAlloc");
    if ((e = cudaHostAlloc((void**)&h->h_chain, (2 + 2 * (size_t)CHAIN_MAX * rows) * sizeof(int),
                           cudaHostAllocDefault)) != cudaSuccess)
        return cuda_fail(h, e, "cudaHostAlloc");
    if ((e = cudaHostAlloc((void**)&h->h_logits, sizeof(float) * rows * (size_t)c.vocab, cudaHostAllocDefault)) !=
        cudaSuccess)
        return cuda_fail(h, e, "cudaHostAlloc");

    // RoPE table and the default page table (row r owns pages r*ppr .. r*ppr+ppr-1)
    {
        std::vector<float2> t = rope_table(cap, c.head_dim, c.rope_theta);
        if ((rc = h2d_wait(h, h->d_rope, t.data(), t.size() * sizeof(float2), "RoPE table upload")) != DEC_OK)
            return rc;
        if (kv_layout == DEC_KV_PAGED) {
            h->slot_map_host.resize((size_t)rows * h->ppr);
            for (size_t i = 0; i < h->slot_map_host.size(); ++i) h->slot_map_host[i] = (int32_t)i;
            if ((rc = h2d_wait(h, h->d_slot_map, h->slot_map_host.data(), h->slot_map_host.size() * sizeof(int32_t),
                               "slot map upload")) != DEC_OK)
                return rc;
        }
    }

    // ---- the recorded launches ----
    const int wt = c.weight_dtype == DEC_DTYPE_BF16 ? W_BF16 : W_F32;
    const int hd = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads, d = c.d_model, F = c.ffn_hidden;
    const int qkv_stride = (Hq + 2 * Hkv) * hd;
    h->embed_p = EmbedParams{h->embed, h->d_slots, h->d_slots + rows, rows, c.vocab, d, cap, h->d_x,
                             &h->d_status->err, h->d_status->amax, h->d_status->nonfinite, h->d_trace, 0};
    h->gemv.clear();
    h->attn.clear();
    // Projections of 2..8 bf16 rows are dense contractions: tensor-core GEMV
    // (GRAPHDEC_GEMV=simd keeps the CUDA-core GEMV at every row count).  Its
    // gate/up kernel applies SwiGLU in the epilogue, so the down projection
    // reads silu(gate) * up from the first F columns of the gate/up buffer.
    const char* gemv_env = getenv("GRAPHDEC_GEMV");
    const bool tc = wt == W_BF16 && rows >= 2 && !(gemv_env && strcmp(gemv_env, "simd") == 0);
    // Which tensor-core GEMV streams a projection: whole-box TMA copies for large
    // matrices (>= 96 MB of weights), one bulk copy per weight row below that,
    // where its shorter start-up wins (measured: 8B qkv / o-proj 20.7 / 14.6 us
    // row-copy vs 25.2 / 22.8 us box; gate/up / down / head 67.7 / 40.8 / 355 us
    // row-copy vs 52.3 / 35.4 / 200 us box).  GRAPHDEC_GEMV=rowcopy or =box forces one.
    const bool force_row = gemv_env && strcmp(gemv_env, "rowcopy") == 0;
    const bool force_box = gemv_env && strcmp(gemv_env, "box") == 0;
    auto tc_kind_for = [&](long long n, long long k) {
        if (!tc) return 0;
        if (force_row) return 1;
        if (force_box) return 2;
        return n * k * 2 >= (96ll << 20) ? 2 : 1;
    };
    auto mk = [&](int pro, int epi, const void* w0, int n0, const void* w1, int n1, const void* w2, int n2, int K,
                  const float* act, int act_stride, const void* gain, float* out, int out_stride) {
        GemvPlan pl{};
        pl.wtype = wt;
        pl.tc = tc_kind_for(n0 + n1 + n2, K);
        pl.pro = pro;
        pl.epi = epi;
        GemvParams& p = pl.p;
        p.w[0] = w0; p.w[1] = w1; p.w[2] = w2;
        p.seg_rows[0] = n0; p.seg_rows[1] = n1; p.seg_rows[2] = n2;
        p.N = n0 + n1 + n2;
        p.K = K;
        p.R = rows;
        p.act = act;
        p.act_stride = act_stride;
        p.gain = gain;
        p.eps = (float)c.rms_eps;
        p.out = out;
        p.out_stride = out_stride;
        p.amax = h->d_status->amax;
        p.nonfinite = h->d_status->nonfinite;
        p.err = &h->d_status->err;
        p.trace = h->d_trace;
        p.tc_part = (float*)(h->ws + h->lay.gpart);
        p.tc_part_cap = (h->lay.gcnt - h->lay.gpart) / sizeof(float);
        p.tc_cnt = (unsigned*)(h->ws + h->lay.gcnt);
        return pl;
    };
    for (int l = 0; l < c.n_layers; ++l) {
        const auto& w = h->lw[l];   // attn_norm, q, k, v, o, ffn_norm, gate, up, down
        h->gemv.push_back(mk(PRO_RMSNORM, EPI_STORE, w[1], Hq * hd, w[2], Hkv * hd, w[3], Hkv * hd, d, h->d_x, d, w[0],
                             h->d_qkv, qkv_stride));
        h->gemv.push_back(mk(PRO_PLAIN, EPI_ADD, w[4], d, nullptr, 0, nullptr, 0, Hq * hd, h->d_attn, Hq * hd, nullptr,
                             h->d_x, d));
        if (tc) {
            h->gemv.push_back(mk(PRO_RMSNORM, EPI_SWIGLU, w[6], F, w[7], F, nullptr, 0, d, h->d_x, d, w[5], h->d_gu,
                                 2 * F));
            h->gemv.push_back(mk(PRO_PLAIN, EPI_ADD, w[8], d, nullptr, 0, nullptr, 0, F, h->d_gu, 2 * F, nullptr,
                                 h->d_x, d));
        } else {
            h->gemv.push_back(mk(PRO_RMSNORM, EPI_STORE, w[6], F, w[7], F, nullptr, 0, d, h->d_x, d, w[5], h->d_gu,
                                 2 * F));
            h->gemv.push_back(mk(PRO_SWIGLU, EPI_ADD, w[8], d, nullptr, 0, nullptr, 0, F, h->d_gu, 2 * F, nullptr,
                                 h->d_x, d));
        }
        AttnPlan ap{};
        ap.kvtype = c.kv_dtype == DEC_DTYPE_BF16 ? W_BF16 : W_F32;
        ap.paged = kv_layout == DEC_KV_PAGED;
        AttnParams& p = ap.p;
        p.qkv = h->d_qkv;
        p.qkv_stride = qkv_stride;
        p.Kc = h->K[l];
        p.Vc = h->V[l];
        p.pos = h->d_slots + rows;
        p.slot_map = h->d_slot_map;
        p.write_map = h->d_slots + 2 * rows;
        p.rope = h->d_rope;
        p.cap = cap;
        p.R = rows;
        p.Hq = Hq;
        p.Hkv = Hkv;
        p.hd = hd;
        p.page_size = h->page > 0 ? h->page : 1;
        p.pages_per_row = h->ppr;
        p.num_pages = h->npages;
        p.part = h->d_part;
        p.counters = h->d_counters;
        p.out = h->d_attn;
        p.err = &h->d_status->err;
        p.scale = (float)(1.0 / std::sqrt((double)hd));
        p.trace = h->d_trace;
        p.trace_id = 2 + 5 * l;
        h->attn.push_back(ap);
    }
    h->gemv.push_back(mk(PRO_RMSNORM, EPI_LOGITS, h->lm_head, c.vocab, nullptr, 0, nullptr, 0, d, h->d_x, d,
                         h->final_norm, h->d_logits, c.vocab));
    for (int l = 0; l < c.n_layers; ++l) {
        h->gemv[4 * l + 0].p.trace_id = 1 + 5 * l;
        h->gemv[4 * l + 1].p.trace_id = 3 + 5 * l;
        h->gemv[4 * l + 2].p.trace_id = 4 + 5 * l;
        h->gemv[4 * l + 3].p.trace_id = 5 + 5 * l;
    }
    h->gemv.back().p.trace_id = 5 * c.n_layers + 1;
    for (auto& pl : h->gemv) {
        if ((e = gemv_plan(&pl, h->num_sms)) != cudaSuccess)
            return fail(h, DEC_E_UNSUPPORTED, "no GEMV kernel for rows=%d K=%d N=%d (%s)", rows, pl.p.K, pl.p.N,
                        cudaGetErrorString(e));
    }
    const char* att_env = getenv("GRAPHDEC_ATTN");   // "simd" selects the CUDA-core attention kernel
    const bool allow_mma = !(att_env && strcmp(att_env, "simd") == 0);
    for (auto& ap : h->attn) {
        if (allow_mma && attn_mma_supported(ap.kvtype, hd, Hq / Hkv, ap.paged, ap.p.page_size)) {
            if ((e = attn_mma_plan(&ap, h->num_sms)) != cudaSuccess)
                return fail(h, DEC_E_UNSUPPORTED, "no attention kernel for head_dim=%d group=%d cap=%d (%s)", hd,
                            Hq / Hkv, cap, cudaGetErrorString(e));
            // several rows: every row's K/V lands before any row's attention, so
            // rows may share pages (a multi-token prefill chunk of one sequence)
            if (rows >= 2) {
                ap.prewrite = true;
                ap.p.kv_prewritten = 1;
            }
            ap.p.pos_bound = h->kv_sweep == DEC_SWEEP_POS ? 1 : 0;
            continue;
        }
        if (h->kv_sweep == DEC_SWEEP_POS)
            return fail(h, DEC_E_UNSUPPORTED,
                        "DEC_SWEEP_POS needs the tensor-core attention kernel (bf16 K/V, head_dim 64 or 128)");
        if ((e = attn_plan(&ap, h->num_sms)) != cudaSuccess)
            return fail(h, DEC_E_UNSUPPORTED, "no attention kernel for head_dim=%d group=%d cap=%d (%s)", hd,
                        Hq / Hkv, cap, cudaGetErrorString(e));
    }
    h->kernels = kernels_per_step(c.n_layers);
    h->extra_kernels = ((!h->attn.empty() && h->attn[0].prewrite) ? c.n_layers : 0) + (h->sampler_on ? 1 : 0);
    if ((e = cudaMemsetAsync(h->d_trace, 0, sizeof(unsigned long long), h->stream)) != cudaSuccess)
        return cuda_fail(h, e, "trace clear");
    if (h->strategy == DEC_STRATEGY_PERSISTENT) {
        if (h->kv_sweep == DEC_SWEEP_POS)
            return fail(h, DEC_E_UNSUPPORTED, "DEC_SWEEP_POS is available with DEC_STRATEGY_GRAPH only");
        if (c.weight_dtype != DEC_DTYPE_BF16 || c.kv_dtype != DEC_DTYPE_BF16)
            return fail(h, DEC_E_UNSUPPORTED, "the persistent strategy needs bf16 weights and KV");
        PersistParams& pp = h->persist.p;
        pp = PersistParams{};
        pp.L = c.n_layers; pp.d = d; pp.F = F; pp.V = c.vocab; pp.Hq = Hq; pp.Hkv = Hkv; pp.hd = hd;
        pp.R = rows; pp.cap = cap;
        pp.paged = kv_layout == DEC_KV_PAGED; pp.page = h->page > 0 ? h->page : 1;
        pp.pages_per_row = h->ppr; pp.num_pages = h->npages;
        pp.eps = (float)c.rms_eps; pp.scale = (float)(1.0 / std::sqrt((double)hd));
        void** ptab = (void**)(h->ws + L.ptabs);
        pp.lw = (const void* const*)ptab;
        pp.kv = (void* const*)(ptab + 9 * (size_t)c.n_layers);
        pp.embed = h->embed; pp.final_norm = h->final_norm; pp.lm_head = h->lm_head;
        pp.x = h->d_x; pp.qkv = h->d_qkv; pp.attn = h->d_attn; pp.gu = h->d_gu; pp.logits = h->d_logits;
        pp.part = h->d_part; pp.counters = h->d_counters; pp.slots = h->d_slots; pp.slot_map = h->d_slot_map;
        pp.rope = h->d_rope; pp.tmaps = h->ws + L.tmaps;
        pp.err = &h->d_status->err; pp.amax = h->d_status->amax; pp.nonfinite = h->d_status->nonfinite;
        pp.bar = (unsigned*)(h->ws + L.gbar); pp.trace = h->d_trace;
        pp.dbg = (const unsigned*)(h->ws + L.dbg);
        if ((e = cudaMemsetAsync(h->ws + L.dbg, 0, 4 * sizeof(unsigned), h->stream)) != cudaSuccess)
            return cuda_fail(h, e, "wait bound clear");
        if ((e = persist_plan(&h->persist, h->num_sms)) != cudaSuccess)
            return fail(h, DEC_E_UNSUPPORTED, "no persistent step kernel for this shape (%s)", cudaGetErrorString(e));
        std::vector<const void*> host_tab((size_t)c.n_layers * 11);
        for (int l = 0; l < c.n_layers; ++l) {
            for (int k = 0; k < 9; ++k) host_tab[(size_t)l * 9 + k] = h->lw[l][k];
            host_tab[9 * (size_t)c.n_layers + 2 * l] = h->K[l];
            host_tab[9 * (size_t)c.n_layers + 2 * l + 1] = h->V[l];
        }
        if ((rc = h2d_wait(h, ptab, host_tab.data(), host_tab.size() * sizeof(void*), "persistent table upload")) !=
            DEC_OK)
            return rc;
        std::vector<unsigned char> tm(persist_tmap_bytes(c.n_layers));
        std::vector<void*> kvp(2 * (size_t)c.n_layers);
        for (int l = 0; l < c.n_layers; ++l) {
            kvp[2 * l] = h->K[l];
            kvp[2 * l + 1] = h->V[l];
        }
        if ((e = persist_tmaps(pp, kvp.data(), tm.data())) != cudaSuccess)
            return fail(h, DEC_E_UNSUPPORTED, "tensor maps for the persistent kernel (%s)", cudaGetErrorString(e));
        if ((rc = h2d_wait(h, h->ws + L.tmaps, tm.data(), tm.size(), "tensor map upload")) != DEC_OK) return rc;
    }

    // the sampler's parameter slot (read by the recorded sampling kernel)
    if (h->sampler_on && (rc = h2d_wait(h, h->ws + L.sampler, &h->sampler, sizeof(SamplerSlot), "sampler upload")) != DEC_OK)
        return rc;

    // ---- one eager step (launch checks), then a clean state ----
    if ((e = zero_state(h)) != cudaSuccess) return cuda_fail(h, e, "state clear");
    for (int r = 0; r < rows; ++r) {
        h->h_slots[r] = 0;
        h->h_slots[rows + r] = 0;
        h->h_slots[2 * rows + r] = kv_layout == DEC_KV_PAGED ? h->slot_map_host[(size_t)r * h->ppr] * page_size : 0;
    }
    if ((e = cudaMemcpyAsync(h->d_slots, h->h_slots, 3 * sizeof(int32_t) * rows, cudaMemcpyHostToDevice, h->stream)) !=
        cudaSuccess)
        return cuda_fail(h, e, "slot write");
    if ((e = enqueue_step(h)) != cudaSuccess) return cuda_fail(h, e, "eager check step");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(h, e, "eager check step");
    if ((e = zero_state(h)) != cudaSuccess) return cuda_fail(h, e, "state clear");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;

    // ---- capture ----
    if ((e = cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
        return cuda_fail(h, e, "cudaStreamBeginCapture");
    cudaError_t le = enqueue_step(h);
    e = cudaStreamEndCapture(h->stream, &h->graph);
    if (le != cudaSuccess) return cuda_fail(h, le, "launch during capture");
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamEndCapture");
    if ((e = cudaGraphInstantiate(&h->exec, h->graph, 0)) != cudaSuccess) return cuda_fail(h, e, "cudaGraphInstantiate");
    if ((e = cudaGraphGetNodes(h->graph, nullptr, &h->nodes)) != cudaSuccess) return cuda_fail(h, e, "cudaGraphGetNodes");
    if ((e = cudaGraphUpload(h->exec, h->stream)) != cudaSuccess) return cuda_fail(h, e, "cudaGraphUpload");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    h->captured = true;
    return DEC_OK;
}

int dec_set_slot_map(dec_handle* h, const int32_t* map) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->layout != DEC_KV_PAGED) return fail(h, DEC_E_STATE, "the capture uses contiguous KV");
    if (!map) return fail(h, DEC_E_INVALID, "map is NULL");
    const size_t n = (size_t)h->rows * h->ppr;
    for (size_t i = 0; i < n; ++i)
        if (map[i] < 0 || map[i] >= h->npages)
            return fail(h, DEC_E_RANGE, "slot map entry %zu = %d outside [0, %d)", i, map[i], h->npages);
    // wait for in-flight steps before rewriting the slot buffer
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    h->slot_map_host.assign(map, map + n);
    return h2d_wait(h, h->d_slot_map, h->slot_map_host.data(), n * sizeof(int32_t), "slot map upload");
}

int dec_step(dec_handle* h, const int32_t* tokens, const int32_t* pos, const int32_t* write_map, float* logits_out,
             int32_t* ids_out, uint8_t* nonfinite_out) {
    const auto t0 = std::chrono::steady_clock::now();
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    if (!tokens || !pos) return fail(h, DEC_E_INVALID, "tokens and pos are required");
    const int R = h->rows;
    for (int r = 0; r < R; ++r) {
        if (tokens[r] < 0 || tokens[r] >= h->cfg.vocab)
            return fail(h, DEC_E_RANGE, "token[%d] = %d outside [0, %d)", r, tokens[r], h->cfg.vocab);
        if (pos[r] < 0 || pos[r] >= h->cap) return fail(h, DEC_E_RANGE, "pos[%d] = %d outside [0, %d)", r, pos[r], h->cap);
    }
    for (int r = 0; r < R; ++r) {
        h->h_slots[r] = tokens[r];
        h->h_slots[R + r] = pos[r];
        int32_t wm = 0;
        if (h->layout == DEC_KV_PAGED) {
            if (write_map) {
                wm = write_map[r];
                if (wm < 0 || (int64_t)wm >= (int64_t)h->npages * h->page)
                    return fail(h, DEC_E_RANGE, "write_map[%d] = %d outside the pool", r, wm);
            } else {
                wm = h->slot_map_host[(size_t)r * h->ppr + pos[r] / h->page] * h->page + pos[r] % h->page;
            }
        }
        h->h_slots[2 * R + r] = wm;
    }
    cudaError_t e = cudaMemcpyAsync(h->d_slots, h->h_slots, 3 * sizeof(int32_t) * R, cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "slot write");
    if ((rc = launch_step(h)) != DEC_OK) return rc;
    rc = finish_step(h, logits_out, ids_out, nonfinite_out);
    h->last_step_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    return rc;
}

int dec_launch(dec_handle* h, const int32_t* dev_slots) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    if (dev_slots) {
        cudaError_t e = cudaMemcpyAsync(h->d_slots, dev_slots, 3 * sizeof(int32_t) * h->rows, cudaMemcpyDeviceToDevice,
                                        h->stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "slot copy");
    }
    return launch_step(h);
}

int dec_wait(dec_handle* h, float* logits_out, int32_t* ids_out, uint8_t* nonfinite_out) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    return finish_step(h, logits_out, ids_out, nonfinite_out);
}

int dec_chain(dec_handle* h, int32_t n_steps, const int32_t* tokens, const int32_t* pos, int32_t* ids_out,
              uint8_t* nonfinite_out) {
    const auto t0 = std::chrono::steady_clock::now();
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    if (!tokens || !pos || !ids_out) return fail(h, DEC_E_INVALID, "tokens, pos and ids_out are required");
    if (n_steps < 1 || n_steps > CHAIN_MAX)
        return fail(h, DEC_E_RANGE, "n_steps = %d outside [1, %d]", n_steps, CHAIN_MAX);
    const int R = h->rows;
    for (int r = 0; r < R; ++r) {
        if (tokens[r] < 0 || tokens[r] >= h->cfg.vocab)
            return fail(h, DEC_E_RANGE, "token[%d] = %d outside [0, %d)", r, tokens[r], h->cfg.vocab);
        if (pos[r] < 0 || (int64_t)pos[r] + n_steps > h->cap)
            return fail(h, DEC_E_RANGE, "pos[%d] = %d: a chain of %d steps leaves [0, %d)", r, pos[r], n_steps, h->cap);
    }
    for (int r = 0; r < R; ++r) {
        h->h_slots[r] = tokens[r];
        h->h_slots[R + r] = pos[r];
        h->h_slots[2 * R + r] =
            h->layout == DEC_KV_PAGED ? h->slot_map_host[(size_t)r * h->ppr + pos[r] / h->page] * h->page + pos[r] % h->page
                                      : 0;
    }
    int* d_chain = (int*)(h->ws + h->lay.chain);
    cudaError_t e = cudaMemcpyAsync(h->d_slots, h->h_slots, 3 * sizeof(int32_t) * R, cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "slot write");
    if ((e = cudaMemsetAsync(d_chain, 0, 2 * sizeof(int), h->stream)) != cudaSuccess) return cuda_fail(h, e, "chain clear");
    ChainParams cp{};
    cp.tok = h->d_slots;
    cp.pos = h->d_slots + R;
    cp.wm = h->d_slots + 2 * R;
    cp.slot_map = h->layout == DEC_KV_PAGED ? h->d_slot_map : nullptr;
    cp.R = R;
    cp.V = h->cfg.vocab;
    cp.cap = h->cap;
    cp.ppr = h->ppr;
    cp.page = h->page > 0 ? h->page : 1;
    cp.amax = h->d_status->amax;
    cp.nonfinite = h->d_status->nonfinite;
    cp.err = &h->d_status->err;
    cp.sampled = h->sampler_on ? h->d_status->sampled : nullptr;
    cp.counter = d_chain;
    cp.chain_err = reinterpret_cast<unsigned*>(d_chain + 1);
    cp.ids = d_chain + 2;
    cp.nf = d_chain + 2 + (size_t)CHAIN_MAX * R;
    cp.max_steps = CHAIN_MAX;
    for (int i = 0; i < n_steps; ++i) {
        if ((rc = launch_step(h)) != DEC_OK) return rc;
        if ((e = chain_advance_launch(cp, h->stream)) != cudaSuccess) return cuda_fail(h, e, "chain advance");
    }
    // one read-back: counter, sticky error, then the two histories
    const size_t hist = (size_t)n_steps * R * sizeof(int);
    if ((e = cudaMemcpyAsync(h->h_chain, d_chain, 2 * sizeof(int) + hist, cudaMemcpyDeviceToHost, h->stream)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(h->h_chain + 2 + (size_t)CHAIN_MAX * R, cp.nf, hist, cudaMemcpyDeviceToHost, h->stream)) !=
            cudaSuccess)
        return cuda_fail(h, e, "chain readback");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    h->steps += n_steps;
    const unsigned err = (unsigned)h->h_chain[1];
    if (err || h->h_chain[0] != n_steps) {
        h->last_fault = err;
        h->state = ST_NEEDS_RESET;
        return fail(h, DEC_E_DEVICE_FAULT, "device check failed in a chained step (error word 0x%x); results "
                    "discarded, reset needed", err);
    }
    memcpy(ids_out, h->h_chain + 2, hist);
    if (nonfinite_out)
        for (size_t k = 0; k < (size_t)n_steps * R; ++k) nonfinite_out[k] = h->h_chain[2 + (size_t)CHAIN_MAX * R + k] ? 1 : 0;
    h->last_step_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count() / n_steps;
    return DEC_OK;
}

int dec_prefill(dec_handle* h, const int32_t* pages, const int32_t* tokens, int32_t n, int32_t pos0, float* logits_out,
                int32_t* id_out) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    if (h->layout != DEC_KV_PAGED || h->rows < 2 || h->strategy != DEC_STRATEGY_GRAPH || h->attn.empty() ||
        !h->attn[0].prewrite)
        return fail(h, DEC_E_UNSUPPORTED, "multi-token prefill needs a paged graph capture of 2..8 rows with bf16 K/V");
    if (!pages || !tokens) return fail(h, DEC_E_INVALID, "pages and tokens are required");
    if (n < 1 || pos0 < 0 || (int64_t)pos0 + n > h->cap)
        return fail(h, DEC_E_RANGE, "positions [%d, %d) outside [0, %d)", pos0, pos0 + n, h->cap);
    for (int i = 0; i < h->ppr; ++i)
        if (pages[i] < 0 || pages[i] >= h->npages)
            return fail(h, DEC_E_RANGE, "pages[%d] = %d outside [0, %d)", i, pages[i], h->npages);
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab)
            return fail(h, DEC_E_RANGE, "tokens[%d] = %d outside [0, %d)", i, tokens[i], h->cfg.vocab);
    const int R = h->rows;
    // every row reads and writes this sequence's pages for the duration of the prefill
    std::vector<int32_t> shared((size_t)R * h->ppr);
    for (int r = 0; r < R; ++r) memcpy(shared.data() + (size_t)r * h->ppr, pages, sizeof(int32_t) * h->ppr);
    cudaError_t e = cudaMemcpyAsync(h->d_slot_map, shared.data(), shared.size() * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "slot map write");
    std::vector<float> last;
    int32_t ids[MAX_ROWS];
    int last_row = 0;
    for (int c = 0; c < n && rc == DEC_OK; c += R) {
        const int m = std::min(R, n - c);
        // rows past the chunk repeat its last token: same position, same bytes written
        for (int r = 0; r < R; ++r) {
            const int t = c + std::min(r, m - 1), p = pos0 + t;
            h->h_slots[r] = tokens[t];
            h->h_slots[R + r] = p;
            h->h_slots[2 * R + r] = pages[p / h->page] * h->page + p % h->page;
        }
        if ((e = cudaMemcpyAsync(h->d_slots, h->h_slots, 3 * sizeof(int32_t) * R, cudaMemcpyHostToDevice, h->stream)) !=
            cudaSuccess)
            return cuda_fail(h, e, "slot write");
        if ((rc = launch_step(h)) != DEC_OK) return rc;
        const bool final_chunk = c + R >= n;
        if (final_chunk && logits_out) last.resize((size_t)R * h->cfg.vocab);
        rc = finish_step(h, final_chunk && logits_out ? last.data() : nullptr, ids, nullptr);
        last_row = m - 1;
    }
    // the caller's page table again
    e = cudaMemcpyAsync(h->d_slot_map, h->slot_map_host.data(), h->slot_map_host.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "slot map restore");
    if (rc != DEC_OK) return rc;
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    if (logits_out) memcpy(logits_out, last.data() + (size_t)last_row * h->cfg.vocab, sizeof(float) * h->cfg.vocab);
    if (id_out) *id_out = ids[last_row];
    return DEC_OK;
}

int dec_prefill_block(dec_handle* h, int32_t row, const int32_t* pages, const int32_t* tokens, int32_t n, int32_t pos0,
                      float* logits_out, int32_t* id_out) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    const dec_config& c = h->cfg;
    if (c.weight_dtype != DEC_DTYPE_BF16 || c.kv_dtype != DEC_DTYPE_BF16)
        return fail(h, DEC_E_UNSUPPORTED, "the block prefill needs bf16 weights and K/V");
    PrefillArgs a{};
    a.L = c.n_layers; a.d = c.d_model; a.Hq = c.n_heads; a.Hkv = c.n_kv_heads; a.hd = c.head_dim;
    a.F = c.ffn_hidden; a.cap = h->cap; a.eps = (float)c.rms_eps;
    a.embed = h->embed;
    a.lw = reinterpret_cast<const void* const*>(h->lw.data());
    a.K = h->K.data();
    a.V = h->V.data();
    a.paged = h->layout == DEC_KV_PAGED;
    a.page = h->page;
    a.ppr = h->ppr;
    a.rows = h->rows;
    a.num_pages = h->npages;
    a.rope = h->d_rope;
    a.err = &h->d_status->err;
    if (!prefill_supported(a))
        return fail(h, DEC_E_UNSUPPORTED, "no block prefill for this shape (head_dim 64 or 128, n_heads / n_kv_heads "
                    "2 or 4, d_model, n_heads * head_dim and ffn_hidden multiples of 64, d_model <= 8192, pages of "
                    "at least 8 tokens)");
    if (!tokens || (a.paged && !pages)) return fail(h, DEC_E_INVALID, "tokens (and for paged K/V the pages) are required");
    if (!a.paged && (row < 0 || row >= h->rows)) return fail(h, DEC_E_RANGE, "row %d outside [0, %d)", row, h->rows);
    if (n < 1 || pos0 < 0 || (int64_t)pos0 + n > h->cap)
        return fail(h, DEC_E_RANGE, "positions [%d, %d) outside [0, %d)", pos0, pos0 + n, h->cap);
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= c.vocab)
            return fail(h, DEC_E_RANGE, "tokens[%d] = %d outside [0, %d)", i, tokens[i], c.vocab);
    if (a.paged)
        for (int i = 0; i < h->ppr; ++i)
            if (pages[i] < 0 || pages[i] >= h->npages)
                return fail(h, DEC_E_RANGE, "pages[%d] = %d outside [0, %d)", i, pages[i], h->npages);
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;   // no step in flight
    cudaError_t e;
    if (!h->pf) {
        e = prefill_create(a, h->num_sms, &h->pf);
        if (e == cudaErrorMemoryAllocation) return fail(h, DEC_E_OOM, "block prefill buffers: device allocation failed");
        if (e != cudaSuccess) return cuda_fail(h, e, "block prefill setup");
    }
    // the last token's hidden state goes through the step's own head as row 0
    if ((e = cudaMemsetAsync(h->d_status, 0, sizeof(StatusBlock), h->stream)) != cudaSuccess)
        return cuda_fail(h, e, "status clear");
    if ((e = prefill_run(h->pf, tokens, n, pos0, row, pages, h->d_x, h->stream)) != cudaSuccess)
        return cuda_fail(h, e, "block prefill");
    if ((e = gemv_launch(h->gemv.back(), h->stream, false)) != cudaSuccess) return cuda_fail(h, e, "prefill head");
    if ((e = cudaMemcpyAsync(h->h_status, h->d_status, sizeof(StatusBlock), cudaMemcpyDeviceToHost, h->stream)) !=
        cudaSuccess)
        return cuda_fail(h, e, "status readback");
    if (logits_out && (e = cudaMemcpyAsync(h->h_logits, h->d_logits, sizeof(float) * c.vocab, cudaMemcpyDeviceToHost,
                                           h->stream)) != cudaSuccess)
        return cuda_fail(h, e, "logits readback");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    if (h->h_status->err) {
        h->last_fault = h->h_status->err;
        h->state = ST_NEEDS_RESET;
        return fail(h, DEC_E_DEVICE_FAULT, "device check failed in the prefill (error word 0x%x)", h->h_status->err);
    }
    if (logits_out) memcpy(logits_out, h->h_logits, sizeof(float) * c.vocab);
    if (id_out) {
        const unsigned long long k = h->h_status->amax[0];
        *id_out = k ? (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull)) : -1;
    }
    return DEC_OK;
}

int dec_set_sampler(dec_handle* h, const dec_sampler* sp) {
    int rc = gate(h, false);
    if (rc) return rc;
    if (sp) {
        if (!(sp->temperature >= 0.f) || !std::isfinite(sp->temperature))
            return fail(h, DEC_E_INVALID, "temperature must be finite and >= 0");
        if (sp->temperature > 0.f && (sp->top_k < 1 || sp->top_k > DEC_SAMPLER_MAX_TOP_K))
            return fail(h, DEC_E_INVALID, "top_k must be in [1, %d] when sampling", DEC_SAMPLER_MAX_TOP_K);
        if (!(sp->top_p > 0.f && sp->top_p <= 1.f)) return fail(h, DEC_E_INVALID, "top_p must be in (0, 1]");
        if (!(sp->min_p >= 0.f && sp->min_p < 1.f)) return fail(h, DEC_E_INVALID, "min_p must be in [0, 1)");
        if (sp->n_logprobs < 0 || sp->n_logprobs > DEC_LOGPROBS_MAX)
            return fail(h, DEC_E_INVALID, "n_logprobs must be in [0, %d]", DEC_LOGPROBS_MAX);
    }
    if (!h->captured) {
        h->sampler_on = sp != nullptr;
        if (sp) h->sampler = *sp;
        return DEC_OK;
    }
    if (!h->sampler_on) return fail(h, DEC_E_STATE, "no sampler was recorded: set one before dec_capture");
    if (h->state == ST_POISONED) return fail(h, DEC_E_POISONED, "handle is poisoned");
    dec_sampler v{};
    v.top_k = 1;
    v.top_p = 1.f;
    if (sp) v = *sp;
    h->sampler = v;
    cudaError_t e = cudaMemcpyAsync(h->ws + h->lay.sampler, &h->sampler, sizeof(SamplerSlot), cudaMemcpyHostToDevice,
                                    h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "sampler write");
    return bounded_wait(h);   // the host copy may change as soon as this returns
}

int dec_logprobs(dec_handle* h, int32_t n, int32_t* ids_out, float* logprobs_out) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (!h->sampler_on || n < 1 || n > h->sampler.n_logprobs || !ids_out || !logprobs_out)
        return fail(h, DEC_E_INVALID, "n = %d: at most the sampler's n_logprobs (%d)", n,
                    h->sampler_on ? h->sampler.n_logprobs : 0);
    for (int r = 0; r < h->rows; ++r)
        for (int j = 0; j < n; ++j) {
            ids_out[r * n + j] = h->h_status->lp_ids[r * DEC_LOGPROBS_MAX + j];
            logprobs_out[r * n + j] = h->h_status->lp_vals[r * DEC_LOGPROBS_MAX + j];
        }
    return DEC_OK;
}

int dec_set_strategy(dec_handle* h, int32_t strategy) {
    int rc = gate(h, false);
    if (rc) return rc;
    if (h->captured) return fail(h, DEC_E_STATE, "the strategy is chosen before dec_capture");
    if (strategy != DEC_STRATEGY_GRAPH && strategy != DEC_STRATEGY_PERSISTENT)
        return fail(h, DEC_E_INVALID, "unknown strategy %d", strategy);
    h->strategy = strategy;
    return DEC_OK;
}

int dec_set_kv_sweep(dec_handle* h, int32_t sweep) {
    int rc = gate(h, false);
    if (rc) return rc;
    if (h->captured) return fail(h, DEC_E_STATE, "the K/V sweep is chosen before dec_capture");
    if (sweep != DEC_SWEEP_CAP && sweep != DEC_SWEEP_POS) return fail(h, DEC_E_INVALID, "unknown K/V sweep %d", sweep);
    h->kv_sweep = sweep;
    return DEC_OK;
}

int dec_set_eager(dec_handle* h, int32_t eager) {
    int rc = gate(h, false);
    if (rc) return rc;
    h->eager = eager != 0;
    return DEC_OK;
}

int dec_reset_state(dec_handle* h) {
    int rc = gate(h, true);
    if (rc) return rc;
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    cudaError_t e = zero_state(h);
    if (e != cudaSuccess) return cuda_fail(h, e, "state clear");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    h->state = ST_READY;
    h->last_fault = 0;
    return DEC_OK;
}

int dec_kv_ptr(dec_handle* h, int32_t layer, int32_t which, void** ptr, size_t* bytes) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (layer < 0 || layer >= h->cfg.n_layers || (which != 0 && which != 1) || !ptr)
        return fail(h, DEC_E_INVALID, "dec_kv_ptr: bad layer/which/ptr");
    *ptr = which ? h->V[layer] : h->K[layer];
    if (bytes) {
        const size_t es = (size_t)es_of(h->cfg.kv_dtype), hd = h->cfg.head_dim, Hkv = h->cfg.n_kv_heads;
        *bytes = h->layout == DEC_KV_PAGED ? (size_t)h->npages * Hkv * h->page * hd * es
                                          : (size_t)h->rows * Hkv * h->cap * hd * es;
    }
    return DEC_OK;
}

int dec_logits_ptr(dec_handle* h, float** ptr) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (!ptr) return fail(h, DEC_E_INVALID, "ptr is NULL");
    *ptr = h->d_logits;
    return DEC_OK;
}

int dec_stream(dec_handle* h, void** stream) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (!stream) return fail(h, DEC_E_INVALID, "stream is NULL");
    *stream = (void*)h->stream;
    return DEC_OK;
}

int dec_stats_get(const dec_handle* h, dec_stats* out) {
    if (!h || !out) return DEC_E_INVALID;
    memset(out, 0, sizeof *out);
    out->steps = h->steps;
    out->replays = h->replays;
    out->eager_steps = h->eager_steps;
    out->kernels_per_step =
        h->strategy == DEC_STRATEGY_PERSISTENT ? 1 + (h->sampler_on ? 1 : 0) : h->kernels + h->extra_kernels;
    out->graph_nodes = (int32_t)h->nodes;
    out->attn_splits = h->strategy == DEC_STRATEGY_PERSISTENT ? h->persist.p.nsplit
                                                              : (h->attn.empty() ? 0 : h->attn[0].p.nsplit);
    out->attn_split_len = h->strategy == DEC_STRATEGY_PERSISTENT ? h->persist.p.split_len
                                                                 : (h->attn.empty() ? 0 : h->attn[0].p.split_len);
    out->strategy = h->strategy;
    out->last_fault = h->last_fault;
    out->state = h->state;
    out->captured = h->captured ? 1 : 0;
    out->rows = h->rows;
    out->cap = h->cap;
    out->kv_layout = h->layout;
    out->last_step_us = h->last_step_us;
    out->workspace_bytes = (int64_t)h->lay.total;
    out->kv_bytes = (int64_t)(2 * (size_t)h->cfg.n_layers * h->lay.kv_layer);
    return DEC_OK;
}

int dec_slot_map_ptr(dec_handle* h, int32_t** ptr) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->layout != DEC_KV_PAGED) return fail(h, DEC_E_STATE, "the capture uses contiguous KV");
    if (!ptr) return fail(h, DEC_E_INVALID, "ptr is NULL");
    *ptr = h->d_slot_map;
    return DEC_OK;
}

int dec_debug_wait(dec_handle* h, uint32_t grid_polls, uint32_t ring_polls, int32_t hold_phase, int32_t drop_stage) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (h->strategy != DEC_STRATEGY_PERSISTENT)
        return fail(h, DEC_E_STATE, "the wait hooks belong to the persistent strategy");
    if (hold_phase < -1 || drop_stage < -1) return fail(h, DEC_E_INVALID, "hold_phase and drop_stage must be >= -1");
    // the kernel reads the block at its start: write it between launches
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    const unsigned v[4] = {grid_polls, ring_polls, (unsigned)(hold_phase + 1), (unsigned)(drop_stage + 1)};
    return h2d_wait(h, h->ws + h->lay.dbg, v, sizeof v, "wait bound write");
}

int dec_launch_kernel(dec_handle* h, int32_t index, int32_t pdl, int64_t* bytes) {
    int rc = gate(h, true);
    if (rc) return rc;
    const int L = h->cfg.n_layers;
    if (h->strategy == DEC_STRATEGY_PERSISTENT) {
        if (index != 0) return fail(h, DEC_E_INVALID, "the persistent strategy records one kernel (index 0)");
        cudaError_t e = persist_launch(h->persist, h->stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
        if (bytes) {
            const dec_config& c = h->cfg;
            *bytes = (int64_t)(h->lay.kv_layer * 0);
            const int64_t wes = 2, R = h->rows;
            const int64_t d = c.d_model, F = c.ffn_hidden, V = c.vocab, qd = (int64_t)c.n_heads * c.head_dim,
                          kvd = (int64_t)c.n_kv_heads * c.head_dim;
            const int64_t per_layer = (qd + 2 * kvd) * d + d * qd + 3 * F * d + 2 * d;
            *bytes = wes * (L * per_layer + V * d + d + R * d) + R * L * 2 * (int64_t)h->cap * kvd * 2;
        }
        return DEC_OK;
    }
    if (index < 0 || index > 5 * L + 1) return fail(h, DEC_E_INVALID, "kernel index %d outside [0, %d]", index, 5 * L + 1);
    const dec_config& c = h->cfg;
    const int64_t wes = es_of(c.weight_dtype), kes = es_of(c.kv_dtype), R = h->rows;
    cudaError_t e;
    int64_t b = 0;
    if (index == 0) {
        e = embed_launch(c.weight_dtype == DEC_DTYPE_BF16 ? W_BF16 : W_F32, h->embed_p, h->stream);
        b = R * c.d_model * (wes + 4);
    } else if (index == 5 * L + 1) {
        const GemvPlan& g = h->gemv.back();
        e = gemv_launch(g, h->stream, pdl != 0);
        b = (int64_t)g.p.N * g.p.K * wes + R * g.p.K * 4 + R * (int64_t)g.p.N * 4;
    } else {
        const int l = (index - 1) / 5, k = (index - 1) % 5;
        if (k == 1) {
            const AttnPlan& a = h->attn[l];
            e = launch_attn(a, h->stream, pdl != 0);
            b = R * 2 * (int64_t)h->cap * c.n_kv_heads * c.head_dim * kes +
                R * (int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim * 4 + R * (int64_t)c.n_heads * c.head_dim * 4;
        } else {
            const GemvPlan& g = h->gemv[4 * l + (k == 0 ? 0 : k - 1)];
            e = gemv_launch(g, h->stream, pdl != 0);
            const int64_t act_in = g.pro == PRO_SWIGLU ? 2 * g.p.K : g.p.K;
            const int64_t out_rw = g.epi == EPI_ADD ? 8 : 4;
            const int64_t n_out = g.epi == EPI_SWIGLU ? g.p.N / 2 : g.p.N;
            b = (int64_t)g.p.N * g.p.K * wes + R * act_in * 4 + R * n_out * out_rw +
                (g.pro == PRO_RMSNORM ? g.p.K * wes : 0);
        }
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
    if (bytes) *bytes = b;
    return DEC_OK;
}

int dec_trace(dec_handle* h, int32_t enable) {
    int rc = gate(h, true);
    if (rc) return rc;
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    const size_t n = 1 + 4 * (size_t)h->kernels;
    std::vector<unsigned long long> init(n, 0ull);
    init[0] = enable ? 1ull : 0ull;
    for (int k = 0; k < h->kernels; ++k) {
        init[1 + 4 * k + 0] = ~0ull;   // minima start high
        init[1 + 4 * k + 2] = ~0ull;
    }
    return h2d_wait(h, h->d_trace, init.data(), n * sizeof(unsigned long long), "trace reset");
}

int dec_trace_read(dec_handle* h, uint64_t* out, size_t n_kernels) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (!out || n_kernels > (size_t)h->kernels) return fail(h, DEC_E_INVALID, "dec_trace_read: bad buffer");
    if ((rc = bounded_wait(h)) != DEC_OK) return rc;
    cudaError_t e = cudaMemcpyAsync(out, h->d_trace + 1, 4 * n_kernels * sizeof(unsigned long long),
                                    cudaMemcpyDeviceToHost, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "trace read");
    return bounded_wait(h);
}

}  // extern "C"

namespace gd {

// One layer's attention on caller buffers: the recorded plan with its q/k/v
// input, position slot, output and split scratch replaced.  Synchronous.
int engine_run_attention(dec_handle* h, int32_t layer, const float* qkv, const int32_t* pos, float* out, float* part,
                         unsigned* counters) {
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(h, DEC_E_INVALID, "layer %d out of range", layer);
    if (!qkv || !pos || !out) return fail(h, DEC_E_INVALID, "qkv, pos and out are required");
    if (h->state == ST_NEEDS_RESET) return fail(h, DEC_E_NEEDS_RESET, "an earlier step failed; call dec_reset_state");
    AttnPlan a = h->attn[layer];
    a.p.qkv = qkv;
    a.p.qkv_stride = (h->cfg.n_heads + 2 * h->cfg.n_kv_heads) * h->cfg.head_dim;
    a.p.pos = pos;
    a.p.out = out;
    a.p.part = part;
    a.p.counters = counters;
    a.p.trace = nullptr;
    cudaError_t e = cudaMemsetAsync(&h->d_status->err, 0, sizeof(unsigned), h->stream);
    if (e == cudaSuccess) e = launch_attn(a, h->stream, false);
    if (e != cudaSuccess) return cuda_fail(h, e, "attention launch");
    if ((e = cudaMemcpyAsync(&h->h_status->err, &h->d_status->err, sizeof(unsigned), cudaMemcpyDeviceToHost,
                             h->stream)) != cudaSuccess)
        return cuda_fail(h, e, "status readback");
    int rc = bounded_wait(h);
    if (rc != DEC_OK) return rc;
    if (h->h_status->err) {
        h->last_fault = h->h_status->err;
        h->state = ST_NEEDS_RESET;
        return fail(h, DEC_E_DEVICE_FAULT, "device check failed (error word 0x%x)", h->h_status->err);
    }
    return DEC_OK;
}

// split scratch one layer's attention needs: partial floats and counters
void engine_attention_scratch(const dec_handle* h, size_t* part_floats, size_t* counters) {
    *part_floats = attn_part_floats(h->rows, h->cfg.n_heads, h->cfg.head_dim, h->attn.empty() ? 0 : h->attn[0].p.nsplit);
    *counters = (size_t)h->rows * h->cfg.n_kv_heads;
}

int engine_gate(dec_handle* h) { return gate(h, true); }
int engine_fail(dec_handle* h, int code, const char* msg) {
    if (code == DEC_E_CUDA) h->state = ST_POISONED;   // CUDA errors are sticky, as everywhere in the ABI
    return fail(h, code, "%s", msg);
}
int engine_device(const dec_handle* h) { return h->cfg.device; }

}  // namespace gd

extern "C" {

int dec_attention(dec_handle* h, int32_t layer, const float* qkv, const int32_t* pos, float* out) {
    int rc = gate(h, true);
    if (rc) return rc;
    return engine_run_attention(h, layer, qkv, pos, out, h->d_part, h->d_counters);
}

int dec_debug_busy(dec_handle* h, int64_t microseconds) {
    int rc = gate(h, true);
    if (rc) return rc;
    if (microseconds < 0) microseconds = 0;
    if (microseconds > 2000000) microseconds = 2000000;
    cudaError_t e = busy_launch((long long)microseconds * 1000ll, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "busy kernel");
    return DEC_OK;
}

int dec_set_timeout(dec_handle* h, int64_t wait_timeout_ms) {
    if (!h) return DEC_E_INVALID;
    if (wait_timeout_ms <= 0) return fail(h, DEC_E_INVALID, "timeout must be > 0");
    h->cfg.wait_timeout_ms = wait_timeout_ms;
    return DEC_OK;
}

// With a NULL handle: the message of the last failed dec_init on this thread.
const char* dec_last_error(const dec_handle* h) { return h ? h->msg.c_str() : g_init_msg.c_str(); }

const char* dec_status_str(int s) {
    switch (s) {
        case DEC_OK: return "DEC_OK";
        case DEC_E_INVALID: return "DEC_E_INVALID";
        case DEC_E_UNSUPPORTED: return "DEC_E_UNSUPPORTED";
        case DEC_E_RANGE: return "DEC_E_RANGE";
        case DEC_E_STATE: return "DEC_E_STATE";
        case DEC_E_CUDA: return "DEC_E_CUDA";
        case DEC_E_OOM: return "DEC_E_OOM";
        case DEC_E_DEVICE_FAULT: return "DEC_E_DEVICE_FAULT";
        case DEC_E_NEEDS_RESET: return "DEC_E_NEEDS_RESET";
        case DEC_E_POISONED: return "DEC_E_POISONED";
        case DEC_E_TIMEOUT: return "DEC_E_TIMEOUT";
    }
    return "DEC_E_UNKNOWN";
}

int dec_destroy(dec_handle* h) {
    if (!h) return DEC_E_INVALID;
    bool device_idle = true;
    if (h->stream && h->ev && h->state != ST_POISONED) device_idle = bounded_wait(h) == DEC_OK;
    if (h->state == ST_POISONED) device_idle = false;
    if (device_idle) {
        // work that could still reference these buffers has finished
        if (h->exec) cudaGraphExecDestroy(h->exec);
        if (h->graph) cudaGraphDestroy(h->graph);
        if (h->own_ws && h->ws) cudaFree(h->ws);
        if (h->h_slots) cudaFreeHost(h->h_slots);
        if (h->h_status) cudaFreeHost(h->h_status);
        if (h->h_logits) cudaFreeHost(h->h_logits);
        if (h->h_chain) cudaFreeHost(h->h_chain);
        if (h->ev) cudaEventDestroy(h->ev);
        if (h->own_stream && h->stream) cudaStreamDestroy(h->stream);
    }
    // a poisoned handle leaks what the pending work could reference
    if (device_idle) prefill_free(h->pf);
    for (auto& a : h->attn) attn_mma_release(a);
    delete h;
    return DEC_OK;
}

}  // extern "C"
