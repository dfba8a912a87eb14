/*
 * graphdec.h -- C ABI of the captured, constant-shape decode step on one GPU.
 *
 * What the library does.  A Llama-style pre-norm decoder step (embedding;
 * per layer RMSNorm, QKV projection, RoPE, K/V write at the slot position,
 * attention that sweeps the fixed KV capacity `cap` under an iota-vs-pos mask,
 * output projection, RMSNorm, SwiGLU MLP; final RMSNorm, LM head, greedy
 * argmax) is recorded once into a CUDA graph and replayed per token.  Between
 * replays the host only rewrites the slot buffers (Token, Pos, and for paged
 * KV the SlotMap page table and the WriteMap target slot).  Sources on the
 * pages: "Execution" (sections "Why capture", "A constant-shape decode graph",
 * "Slot buffers", "Per backend" -- PTX row, "Failure handling"),
 * "Backends" (section "PTX (NVIDIA)"), "Models, Registry and the Driver"
 * (sections "The Model" -- StepShape, "Shared components" -- standard_stack).
 *
 * Conventions shared by every call.
 *   - Every call returns an int status (dec_status); DEC_OK == 0.  After a
 *     failure, dec_last_error() returns a NUL-terminated message owned by the
 *     handle (valid until the next call on that handle); dec_last_error(NULL)
 *     gives the message of the last failed dec_init on the calling thread.
 *   - Pointers marked "device" are CUDA device addresses on the handle's GPU;
 *     "host" pointers are ordinary (pageable or pinned) host memory.  The
 *     library never frees memory it did not allocate.
 *   - A handle is thread-compatible, not thread-safe: one thread at a time.
 *     All device work of a handle runs on one CUDA stream.
 *   - Row-major everywhere.  Matrices use the nn.Linear layout [out, in].
 *   - Failure states ("Execution", section "Failure handling"): a device-side
 *     check that fails (token, position or map value out of range) sets a bit
 *     in the step's error word; the step's results are discarded, the call
 *     returns DEC_E_DEVICE_FAULT and the handle needs dec_reset_state() before
 *     it steps again (DEC_E_NEEDS_RESET until then).  A CUDA error or a wait
 *     that outlasts the configured timeout poisons the handle: every later
 *     call except dec_last_error / dec_stats / dec_destroy returns
 *     DEC_E_POISONED without touching the device.
 */
#ifndef GRAPHDEC_H
#define GRAPHDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DEC_ABI_VERSION 1

typedef struct dec_handle dec_handle;

typedef enum dec_status {
    DEC_OK = 0,
    DEC_E_INVALID = 1,       /* malformed argument or configuration */
    DEC_E_UNSUPPORTED = 2,   /* well-formed, but this library cannot run it (message names the field) */
    DEC_E_RANGE = 3,         /* a token, position or map entry outside its range (host check) */
    DEC_E_STATE = 4,         /* call out of order (e.g. dec_step before dec_capture) */
    DEC_E_CUDA = 5,          /* CUDA runtime error; the handle is poisoned */
    DEC_E_OOM = 6,           /* device allocation failed or workspace too small */
    DEC_E_DEVICE_FAULT = 7,  /* a device-side check failed; see dec_stats.last_fault */
    DEC_E_NEEDS_RESET = 8,   /* an earlier step failed; call dec_reset_state */
    DEC_E_POISONED = 9,      /* the handle saw a CUDA error or a timeout; only dec_destroy helps */
    DEC_E_TIMEOUT = 10       /* a device wait outlasted wait_timeout_ms; the handle is poisoned */
} dec_status;

/* bits of the device error word (dec_stats.last_fault) */
#define DEC_FAULT_TOKEN     0x1u  /* Token[r] outside [0, vocab) */
#define DEC_FAULT_POS       0x2u  /* Pos[r] outside [0, cap) */
#define DEC_FAULT_WRITE_MAP 0x4u  /* WriteMap[r] outside [0, num_pages * page_size) */
#define DEC_FAULT_SLOT_MAP  0x8u  /* a SlotMap entry outside [0, num_pages) */
#define DEC_FAULT_WAIT      0x10u /* an in-kernel wait on another CTA or on a copy gave up (bounded poll) */

typedef enum dec_dtype { DEC_DTYPE_F32 = 0, DEC_DTYPE_BF16 = 1 } dec_dtype;

/* KV layouts ("Execution", section "A constant-shape decode graph"):
 *   CONTIGUOUS: per layer K and V of shape [rows, n_kv_heads, cap, head_dim];
 *               the step writes position Pos[r] (a DynamicUpdateSlice).
 *   PAGED:      per layer a pool [num_pages, n_kv_heads, page_size, head_dim]
 *               for K and one for V; logical position j of row r lives in
 *               slot SlotMap[r][j / page_size] * page_size + j % page_size, and
 *               the step scatters the new K/V to slot WriteMap[r]
 *               (a ScatterUpdate through Slot::WriteMap). */
typedef enum dec_kv_layout { DEC_KV_CONTIGUOUS = 0, DEC_KV_PAGED = 1 } dec_kv_layout;

/* How the captured step executes (chosen before dec_capture):
 *   GRAPH       the pages' strategy: the step's dispatch sequence (embedding,
 *               5 fused kernels per layer, head) recorded into one CUDA graph
 *               with programmatic dependent launches ("Execution", "Per
 *               backend", PTX row);
 *   PERSISTENT  the step as one cooperative kernel captured as the graph's
 *               single node; phases separated by grid-wide dependency counters
 *               and one continuous weight/KV stream per SM (the pages' possible
 *               future megakernel strategy).  Same arithmetic, other fp32
 *               summation order: results agree with GRAPH within the parity
 *               tolerances, not bit for bit; replay and eager runs of one
 *               strategy are bit-identical.  Available for bf16 weights and
 *               KV with the 8B-shape or 1B-class layer shapes at rows = 1
 *               (contiguous or paged K/V), and with the 1B-class shape at
 *               rows = 2 or 4 with contiguous K/V (DEC_E_UNSUPPORTED at
 *               capture otherwise). */
typedef enum dec_strategy { DEC_STRATEGY_GRAPH = 0, DEC_STRATEGY_PERSISTENT = 1 } dec_strategy;

/* Which K/V positions the attention of the captured step reads:
 *   CAP  the method's constant-shape sweep of [0, cap) with the position mask
 *        ("Execution", "A constant-shape decode graph": attention always
 *        sweeps [cap]; a mask computed from Slot::Pos against an iota hides
 *        the positions after pos) -- the default;
 *   POS  the same captured graph and grid, but each split stops loading K/V
 *        tiles after the one holding pos (a split that starts after pos loads
 *        none).  The tiles it skips are fully masked, and the kernel already
 *        does no arithmetic on a 16-key block without a visible key, so the
 *        results are bit-identical to CAP; only the bytes read shrink from the
 *        capacity to the positions up to pos. */
typedef enum dec_kv_sweep { DEC_SWEEP_CAP = 0, DEC_SWEEP_POS = 1 } dec_kv_sweep;

/* Model configuration.  RMSNorm is x / sqrt(mean(x^2) + rms_eps) * g; RoPE is
 * the half-split rotation of pairs (i, i + head_dim/2) by pos * rope_theta^(-2i/head_dim);
 * attention scale is 1/sqrt(head_dim); q head i reads kv head i / (n_heads / n_kv_heads). */
typedef struct dec_config {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_heads;        /* query heads */
    int32_t n_kv_heads;     /* key/value heads; must divide n_heads */
    int32_t head_dim;       /* even */
    int32_t ffn_hidden;     /* SwiGLU hidden width */
    int32_t vocab;
    int32_t weight_dtype;   /* dec_dtype of every weight (matrices, embeddings, norm gains) */
    int32_t kv_dtype;       /* dec_dtype of the stored K/V */
    int32_t device;         /* CUDA device ordinal */
    double rms_eps;
    double rope_theta;
    int64_t wait_timeout_ms;  /* bound on every device wait; <= 0 means 600000 (600 s) */
} dec_config;

/* Weight roles ("Execution": load_weights binds each weight by its typed role;
 * a weight no binding names stays unbound and dec_capture refuses to run). */
typedef enum dec_role {
    DEC_W_EMBED = 0,       /* [vocab, d_model]                     global (layer = -1) */
    DEC_W_ATTN_NORM = 1,   /* [d_model]                            per layer */
    DEC_W_Q = 2,           /* [n_heads * head_dim, d_model]        per layer */
    DEC_W_K = 3,           /* [n_kv_heads * head_dim, d_model]     per layer */
    DEC_W_V = 4,           /* [n_kv_heads * head_dim, d_model]     per layer */
    DEC_W_O = 5,           /* [d_model, n_heads * head_dim]        per layer */
    DEC_W_FFN_NORM = 6,    /* [d_model]                            per layer */
    DEC_W_GATE = 7,        /* [ffn_hidden, d_model]                per layer */
    DEC_W_UP = 8,          /* [ffn_hidden, d_model]                per layer */
    DEC_W_DOWN = 9,        /* [d_model, ffn_hidden]                per layer */
    DEC_W_FINAL_NORM = 10, /* [d_model]                            global */
    DEC_W_LM_HEAD = 11,    /* [vocab, d_model]                     global */
    DEC_W_NROLES = 12
} dec_role;

typedef struct dec_weight {
    int32_t role;      /* dec_role */
    int32_t layer;     /* 0 .. n_layers-1 for per-layer roles, -1 for global roles */
    int32_t dtype;     /* must equal dec_config.weight_dtype */
    int32_t reserved;  /* 0 */
    int64_t rows;      /* shape [rows, cols]; a gain vector of length n is [n, 1] */
    int64_t cols;
    const void *data;  /* device, 16-byte aligned, borrowed: must outlive the handle */
} dec_weight;

typedef struct dec_stats {
    int64_t steps;            /* completed dec_step / dec_wait calls */
    int64_t replays;          /* graph launches */
    int64_t eager_steps;      /* kernel sequences launched without the graph */
    int32_t kernels_per_step; /* kernel launches recorded per step */
    int32_t graph_nodes;      /* nodes of the instantiated graph */
    int32_t attn_splits;      /* KV splits per (row, kv head) */
    int32_t attn_split_len;   /* positions per split */
    uint32_t last_fault;      /* error word of the last failed step (DEC_FAULT_* bits) */
    int32_t state;            /* 0 ready, 1 needs reset, 2 poisoned */
    int32_t captured;         /* 1 after dec_capture */
    int32_t rows;
    int32_t cap;
    int32_t kv_layout;
    int32_t strategy;         /* dec_strategy of the capture */
    int32_t reserved;
    double last_step_us;      /* host wall time of the last dec_step */
    int64_t workspace_bytes;  /* device bytes the capture uses (KV included) */
    int64_t kv_bytes;         /* device bytes of K and V over all layers */
} dec_stats;

/* Create a handle for `cfg` on cfg->device ("Execution", executor contract:
 * one engine per target, set up before any weight is bound; the handle plays
 * the executor object and every later call goes through it).  Validates the
 * configuration (DEC_E_INVALID / DEC_E_UNSUPPORTED naming the field, like the
 * planner's refusals) before touching the GPU; DEC_E_CUDA if the device cannot
 * be selected.  *out receives the handle, or NULL on failure; the caller owns
 * it and releases it with dec_destroy. */
int dec_init(const dec_config *cfg, dec_handle **out);

/* Bind `n` weights by role ("Execution": load_weights(store, map)).  May be
 * called several times before dec_capture; a later binding of the same
 * (role, layer) replaces the earlier one.  Shapes and dtypes are checked
 * against the configuration (DEC_E_INVALID).  The library reads the weights in
 * place: nothing is copied. */
int dec_load_weights(dec_handle *h, const dec_weight *w, size_t n);

/* Device bytes that dec_capture needs for this shape (KV store, slots,
 * activations, attention partials, RoPE table): the preallocated Storage::State
 * buffers of capacity cap per layer plus the step's intermediates ("Execution",
 * section "A constant-shape decode graph": K and V are preallocated to cap).
 * Host-only (no device call).  *bytes (host) receives the size; DEC_E_INVALID
 * for a configuration dec_init would refuse or a shape dec_capture would refuse. */
int dec_workspace_size(const dec_config *cfg, int32_t cap, int32_t rows, int32_t kv_layout,
                       int32_t page_size, int32_t num_pages, size_t *bytes);

/* Allocate the step's buffers, run the kernel sequence once eagerly (checks),
 * clear the state, and record the sequence into one CUDA graph that serves
 * every position 0 <= pos < cap ("Execution", section "A constant-shape decode
 * graph": grids and buffer addresses stay constant, so one capture serves
 * every position up to cap).  One capture per handle ("Models, Registry and
 * the Driver": one entry per step shape; capacity is part of the shape).
 *   cap        KV capacity (positions per row), >= 1
 *   rows       sequences stepped together, 1 .. 8
 *   kv_layout  dec_kv_layout
 *   page_size, num_pages  paged layout only (cap % page_size == 0,
 *              rows * cap / page_size <= num_pages); ignored for contiguous
 *   workspace  device buffer of >= dec_workspace_size bytes, 256-byte aligned,
 *              owned by the caller and kept until dec_destroy; NULL: the library
 *              allocates (and frees at dec_destroy)
 *   stream     cudaStream_t to run on; NULL: the library creates its own.
 *              The legacy default stream cannot be captured and is refused.
 * All bound weights must be present (DEC_E_INVALID names the first missing). */
int dec_capture(dec_handle *h, int32_t cap, int32_t rows, int32_t kv_layout, int32_t page_size,
                int32_t num_pages, void *workspace, size_t workspace_bytes, void *stream);

/* Rewrite the paged read map ("Execution", section "Slot buffers":
 * Slot::SlotMap).  map: host, [rows, cap / page_size] int32 page ids, each in
 * [0, num_pages) (DEC_E_RANGE otherwise).  Takes effect from the next step.
 * DEC_E_STATE for a contiguous capture. */
int dec_set_slot_map(dec_handle *h, const int32_t *map);

/* One decode step of every row ("Execution", section "Per backend", PTX row:
 * write slots, launch the graph, copy results back, wait).
 *   tokens     host [rows], each in [0, vocab)
 *   pos        host [rows], each in [0, cap): the absolute position of the token
 *   write_map  host [rows] target slot for paged KV, or NULL to derive it from
 *              the slot map as SlotMap[r][pos/page]*page + pos%page; ignored
 *              for contiguous KV
 *   logits_out host [rows, vocab] fp32, or NULL
 *   ids_out    host [rows] greedy token ids (largest logit, lowest index on
 *              ties), or NULL
 *   nonfinite_out host [rows], 1 if any logit of the row is NaN or Inf, or NULL
 * Host-side range checks return DEC_E_RANGE before anything is launched. */
int dec_step(dec_handle *h, const int32_t *tokens, const int32_t *pos, const int32_t *write_map,
             float *logits_out, int32_t *ids_out, uint8_t *nonfinite_out);

/* Asynchronous half of a step: copy the slot record (device, [3 * rows]
 * int32: tokens, then positions, then write map) into the slot buffers and
 * launch the step, without waiting and without host-side range checks (the
 * device checks still run).  Results stay on the device until dec_wait. */
int dec_launch(dec_handle *h, const int32_t *dev_slots);

/* Wait (bounded by wait_timeout_ms) for the launched steps and copy the last
 * step's results back; any pointer may be NULL.  Returns DEC_E_DEVICE_FAULT if
 * the last step's error word is non-zero. */
int dec_wait(dec_handle *h, float *logits_out, int32_t *ids_out, uint8_t *nonfinite_out);

/* Chained greedy steps ("Models, Registry and the Driver", section "The
 * Driver": RowWork::Chain -- with no guided row, several decode steps run back
 * to back, the device feeds each step's pick to the next and the host waits
 * once).  Step 0 runs tokens at pos; step i > 0 runs, for every row, the
 * greedy id of step i - 1 at pos + i.  Each step is one replay of the recorded
 * step followed by a one-CTA kernel that records the ids and writes the next
 * step's Token, Pos and (paged) WriteMap slots from the device; the host
 * copies the histories back once and waits once.
 *   n_steps       1 .. DEC_CHAIN_MAX_STEPS
 *   tokens, pos   host [rows], as for dec_step; pos[r] + n_steps <= cap
 *                 (DEC_E_RANGE otherwise, before anything is launched)
 *   ids_out       host [n_steps, rows]: the greedy id of each step (required)
 *   nonfinite_out host [n_steps, rows] non-finite flags, or NULL
 * Paged KV takes every WriteMap from the current slot map.  A device check
 * that fails in any step of the chain returns DEC_E_DEVICE_FAULT (results
 * discarded, reset needed).  The logits of the last step stay on the device
 * (dec_logits_ptr). */
#define DEC_CHAIN_MAX_STEPS 4096
int dec_chain(dec_handle *h, int32_t n_steps, const int32_t *tokens, const int32_t *pos, int32_t *ids_out,
              uint8_t *nonfinite_out);

/* Multi-token prefill of ONE sequence ("Models, Registry and the Driver",
 * section "The Model": a step shape is rows x new tokens; positions are
 * absolute, so a prefill is a step continuing from a position).  The n tokens
 * at positions pos0 .. pos0 + n - 1 run through the recorded paged step in
 * chunks of `rows` tokens: in each chunk row t is position pos0 + c + t of the
 * sequence, every row reads and writes the sequence's pages, and every row's
 * K/V is stored before any row's attention reads the pages.  Afterwards the
 * sequence's K/V for those positions is in its pages, and the caller's slot
 * map is in place again.
 *   pages       host [cap / page_size] page ids of the sequence, each in
 *               [0, num_pages)
 *   tokens      host [n], each in [0, vocab)
 *   pos0        first position; pos0 + n <= cap (DEC_E_RANGE otherwise)
 *   logits_out  host [vocab] fp32 logits after the last token, or NULL
 *   id_out      host, the greedy id after the last token, or NULL
 * Needs a paged graph capture of 2..8 rows with bf16 K/V (DEC_E_UNSUPPORTED
 * otherwise).  Per token the arithmetic equals a decode step of that token, so
 * the chunking does not change any result. */
int dec_prefill(dec_handle *h, const int32_t *pages, const int32_t *tokens, int32_t n, int32_t pos0,
                float *logits_out, int32_t *id_out);

/* Multi-token prefill of ONE sequence as a block step ("Models, Registry and
 * the Driver", section "The Model": a step shape is rows x new tokens;
 * positions are absolute, so a prefill is a step continuing from a position).
 * The n tokens at positions pos0 .. pos0 + n - 1 run layer by layer in passes
 * of up to 1024 tokens (blocks of 128 for the tensor cores): per layer the
 * projections are dense contractions on the tensor cores
 * (tcgen05.mma, bf16 weights, activations as bf16 hi + lo parts, fp32
 * accumulation), attention is causal over every position up to each token
 * (online softmax, fp32), and every layer's K/V of the n positions is written
 * into the sequence's store (rounded to bf16).  The last token's hidden state
 * then goes through the captured step's final RMSNorm, LM head and argmax.
 *   row         contiguous K/V: the capture row whose store holds the
 *               sequence (0 .. rows-1); ignored for paged K/V
 *   pages       paged K/V: host [cap / page_size] page ids of the sequence, each
 *               in [0, num_pages); NULL for contiguous K/V
 *   tokens      host [n], each in [0, vocab)
 *   pos0        first position; pos0 + n <= cap (DEC_E_RANGE otherwise)
 *   logits_out  host [vocab] fp32 logits after the last token, or NULL
 *   id_out      host, the greedy id after the last token, or NULL
 * Positions before pos0 must already hold the sequence's K/V (from steps or an
 * earlier prefill).  Any capture with bf16 weights and K/V whose shape has
 * head_dim 64 or 128, n_heads / n_kv_heads of 2 or 4, d_model, n_heads *
 * head_dim and ffn_hidden multiples of 64, d_model <= 8192 and (paged
 * K/V) pages of at least 8 tokens (DEC_E_UNSUPPORTED otherwise).  The
 * first call allocates the block's device buffers (cudaMalloc, kept until
 * dec_destroy); the call is synchronous (bounded wait) and must not be
 * captured.  Results agree with stepping the tokens one at a time within the
 * parity tolerances, not bit for bit (other arithmetic, other summation
 * order).  The captured step's slot buffers are untouched; its logits buffer
 * holds this call's logits afterwards. */
int dec_prefill_block(dec_handle *h, int32_t row, const int32_t *pages, const int32_t *tokens, int32_t n,
                      int32_t pos0, float *logits_out, int32_t *id_out);

/* Sampling suffix beyond greedy ("Models, Registry and the Driver", section
 * "The Driver": Head::Sample -- greedy or temperature / top-k / top-p /
 * min-p, optional top-n logprobs).  For each row of a step:
 *   candidates  the top_k tokens of largest logit (ties: lower index);
 *   weights     q = exp((logit - max logit) / temperature);
 *   kept        the shortest prefix of the candidates, by logit, whose weight
 *               reaches top_p of the candidates' total, and only candidates
 *               with q >= min_p (relative to the largest probability);
 *   pick        inverse CDF over the kept prefix at u = the top 53 bits of
 *               splitmix64 at counter (row << 32 | Pos[row]) of `seed`,
 *               i.e. mix64(seed + (counter + 1) * 0x9E3779B97F4A7C15);
 *   logprobs    logit - max - log(sum over the vocabulary of exp(logit - max))
 *               of the n_logprobs tokens of largest logit.
 * temperature = 0 picks the greedy id. */
#define DEC_SAMPLER_MAX_TOP_K 1024
#define DEC_LOGPROBS_MAX 8
typedef struct dec_sampler {
    float temperature;   /* >= 0; 0: greedy */
    int32_t top_k;       /* 1 .. DEC_SAMPLER_MAX_TOP_K when temperature > 0 */
    float top_p;         /* (0, 1]; 1: no top-p cut */
    float min_p;         /* [0, 1); 0: no min-p cut */
    uint64_t seed;
    int32_t n_logprobs;  /* 0 .. DEC_LOGPROBS_MAX */
    int32_t reserved;
} dec_sampler;

/* Before dec_capture: a non-NULL sampler records the sampling kernel after the
 * head in the step (NULL: greedy only, nothing recorded).  After dec_capture:
 * rewrites the sampler's parameters in place for the coming steps (a slot
 * buffer, no re-capture); DEC_E_STATE if no sampler was recorded.  With a
 * sampler recorded, the ids returned by dec_step / dec_wait and fed forward by
 * dec_chain are the sampled ids.  DEC_E_INVALID for parameters out of range. */
int dec_set_sampler(dec_handle *h, const dec_sampler *s);

/* Top-n logprobs of the last completed step: ids_out and logprobs_out host
 * [rows, n], n <= the sampler's n_logprobs (DEC_E_INVALID otherwise). */
int dec_logprobs(dec_handle *h, int32_t n, int32_t *ids_out, float *logprobs_out);

/* Choose the execution strategy (dec_strategy) for the coming dec_capture;
 * DEC_E_STATE after capture.  Default DEC_STRATEGY_GRAPH. */
int dec_set_strategy(dec_handle *h, int32_t strategy);

/* Choose the K/V sweep (dec_kv_sweep) of the coming dec_capture; DEC_E_STATE
 * after capture, DEC_E_INVALID for an unknown value.  Default DEC_SWEEP_CAP.
 * DEC_SWEEP_POS needs the GRAPH strategy and the tensor-core attention kernel
 * (bf16 K/V, head_dim 64 or 128): dec_capture returns DEC_E_UNSUPPORTED
 * otherwise.  It also applies to dec_attention on the same handle. */
int dec_set_kv_sweep(dec_handle *h, int32_t sweep);

/* 1: later steps launch the recorded kernel sequence directly on the stream
 * instead of replaying the graph (same kernels, same arguments); 0: replay. */
int dec_set_eager(dec_handle *h, int32_t eager);

/* Zero the KV store, the slot buffers and the error word, and clear the
 * needs-reset state ("Execution", section "Failure handling": step refuses
 * until reset_state clears it).  A poisoned handle stays poisoned. */
int dec_reset_state(dec_handle *h);

/* Device address and byte size of one layer's K (which = 0) or V (which = 1)
 * store, in the layout of the capture's dec_kv_layout: the carried state that
 * the pages' reference evaluation returns beside the primary output and that
 * parity covers element by element ("Execution", section "Verification", tier
 * 2: every output and carried state).  For tests that pre-fill or inspect it.
 * *ptr (host) receives a device pointer owned by the handle (valid until
 * dec_destroy); *bytes (host, optional) its size.  DEC_E_STATE before
 * dec_capture, DEC_E_INVALID for a bad layer or which. */
int dec_kv_ptr(dec_handle *h, int32_t layer, int32_t which, void **ptr, size_t *bytes);

/* One layer's decode attention as a standalone operation, on the caller's
 * buffers ("Execution", section "A constant-shape decode graph"): rotates q and
 * k by RoPE at pos[r], writes the rotated k and v (rounded to the KV dtype)
 * into this layer's KV store at pos[r] (paged: at the slot of the current
 * write map), and attends over the full capacity with positions after pos[r]
 * masked.  Runs on the handle's stream and waits (bounded).
 *   layer  0 .. n_layers-1
 *   qkv    device fp32 [rows, (n_heads + 2 * n_kv_heads) * head_dim]: q, then k,
 *          then v of every row, before RoPE
 *   pos    device int32 [rows], each in [0, cap)
 *   out    device fp32 [rows, n_heads * head_dim]
 * The split partials use the handle's workspace.  DEC_E_DEVICE_FAULT if a
 * device check fails (the handle then needs dec_reset_state). */
int dec_attention(dec_handle *h, int32_t layer, const float *qkv, const int32_t *pos, float *out);

/* dec_attention without any allocation.  Same operation, arguments and
 * results as dec_attention; the split scratch (partials and completion
 * counters) lives in a fixed device array inside the library instead of the
 * handle's workspace, so this call allocates nothing.  It is for callers that
 * cannot allocate device memory where they run attention: a serving process
 * that reserved its whole device-memory budget up front (weights and KV cache
 * sized to fill the GPU) and has nothing left to hand out per call, and code
 * whose latency cannot absorb cudaMalloc / cudaFree, which may synchronise the
 * whole device.  Like dec_attention it runs on the handle's stream and waits
 * (bounded) for its result before returning.  The pages have no counterpart of
 * this entry point.
 * Limits: the array holds 2^19 fp32 partials and 1024 counters (about 2 MiB); a
 * shape that needs more (rows * n_heads * splits * (head_dim + 4) floats)
 * returns DEC_E_UNSUPPORTED and leaves the handle usable.  Every GPU that loads
 * the library keeps the array until the process exits.  All calls on a device
 * share the array (it keeps the last call's contents; the counters are cleared
 * on entry), so calls that overlap on the GPU race: serialise them.  The first
 * call on a device looks up the array's device address (once per device, kept
 * for the life of the process; a cudaDeviceReset invalidates it together with
 * every handle); make that first call before any stream capture. */
int dec_attention_static(dec_handle *h, int32_t layer, const float *qkv, const int32_t *pos, float *out);

/* Device address of the logits [rows, vocab] fp32 of the last step. */
int dec_logits_ptr(dec_handle *h, float **ptr);

/* The CUDA stream the handle runs on (as a cudaStream_t). */
int dec_stream(dec_handle *h, void **stream);

/* Counters and state of the handle ("Execution", executor contract: stats).
 * Copies a dec_stats snapshot into *out (host); touches no device and works on
 * a poisoned handle.  DEC_E_INVALID for a NULL argument. */
int dec_stats_get(const dec_handle *h, dec_stats *out);

/* Device address of the paged read map [rows, cap / page_size] int32 (the
 * Slot::SlotMap buffer that the recorded kernels read, "Execution", section
 * "Slot buffers").  Introspection for tests: writing it directly bypasses
 * dec_set_slot_map's host range check, so the kernels' own check
 * (DEC_FAULT_SLOT_MAP) can be exercised.  Owned by the handle.  DEC_E_STATE
 * for a contiguous capture or before dec_capture. */
int dec_slot_map_ptr(dec_handle *h, int32_t **ptr);

/* Profiling hook: launch kernel `index` of the recorded step sequence alone,
 * eagerly, on the handle's stream (no slot write, no wait).  Order: 0 embedding;
 * per layer l: 1+5l RMSNorm+QKV, 2+5l attention (RoPE, K/V write, combine),
 * 3+5l output projection + residual, 4+5l RMSNorm+gate/up, 5+5l SwiGLU+down +
 * residual; last (5L+1) final RMSNorm + LM head + argmax.  The kernel reads and
 * writes the step's buffers as in a step (it changes the state).
 * pdl: 1 launches with the programmatic-serialization attribute as in the
 * graph, 0 with plain stream order.  *bytes (optional) receives the
 * algorithmic bytes one launch moves (weights read once + activations, or the
 * cap-swept K/V + q + partials for attention). */
int dec_launch_kernel(dec_handle *h, int32_t index, int32_t pdl, int64_t *bytes);

/* In-graph trace (profiling).  enable = 1 clears the stamps and makes every
 * recorded kernel stamp the device's global nanosecond timer at: its earliest
 * CTA entry, the latest CTA to pass the wait on the previous kernel, its
 * earliest CTA exit and its latest CTA exit; enable = 0 stops recording.
 * Stamps accumulate (min / max) over the steps run while enabled. */
int dec_trace(dec_handle *h, int32_t enable);

/* Copy 4 stamps per kernel for the first n_kernels kernels of the step
 * (order as in dec_launch_kernel) into out[4 * n_kernels] (host). */
int dec_trace_read(dec_handle *h, uint64_t *out, size_t n_kernels);

/* Test hook for the bounded wait: enqueue a kernel that busies one SM for
 * about `microseconds` (clamped to [0, 2000000]) and then ends by itself. */
int dec_debug_busy(dec_handle *h, int64_t microseconds);

/* Test hook: change the wait bound of an existing handle (ms, > 0). */
int dec_set_timeout(dec_handle *h, int64_t wait_timeout_ms);

/* Test hook for the in-kernel bounded waits of the persistent step ("Execution",
 * section "Failure handling": every wait is bounded, and a wait that gives up
 * is a typed error rather than a hang).  Takes effect from the next launch:
 *   grid_polls  polls of a wait on other CTAs (phase counters, attention split
 *               groups) before it gives up; 0: the default (2^22)
 *   ring_polls  polls of a wait on a shared-memory ring stage (a copy landing,
 *               a slot freed) before it gives up; 0: the default (2^22)
 *   hold_phase  phase index whose grid-wide wait target is raised by one, so
 *               that wait cannot complete and gives up after grid_polls
 *               (phases: 0 embedding, 1 + 5l + {0 QKV, 1 attention, 2 O-proj,
 *               3 gate/up, 4 down} of layer l, 5L + 1 head); -1: none
 *   drop_stage  ring stage index (counted over the whole step) that CTA 0's
 *               producer never issues, so its consumers give up after
 *               ring_polls; -1: none
 * A wait that gives up sets DEC_FAULT_WAIT in the error word; the kernel then
 * skips the remaining work, waits (bounded) for its own copies in flight and
 * exits; the step returns DEC_E_DEVICE_FAULT and the handle needs
 * dec_reset_state.  (0, 0, -1, -1) restores the defaults.  DEC_E_STATE unless
 * the capture uses DEC_STRATEGY_PERSISTENT; DEC_E_INVALID for hold_phase or
 * drop_stage below -1. */
int dec_debug_wait(dec_handle *h, uint32_t grid_polls, uint32_t ring_polls, int32_t hold_phase, int32_t drop_stage);

const char *dec_last_error(const dec_handle *h);
const char *dec_status_str(int status);

/* Release the handle ("Execution", executor contract: unload): after a
 * bounded wait for its stream, free everything the library allocated (graph,
 * library-owned workspace, pinned staging, stream and event).  Borrowed
 * weights and a caller workspace are not touched.  A poisoned handle frees
 * only host state and leaks the device memory that pending work could
 * reference ("Execution", section "Failure handling").  DEC_E_INVALID for
 * NULL; the handle is invalid afterwards whatever the status. */
int dec_destroy(dec_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* GRAPHDEC_H */
