/*
 * mk.h -- C ABI of the GB300 persistent MoE decode-layer library (libmk.so).
 *
 * One call runs the batch-1 speculative-verify decode step (T <= 16 tokens) of
 * one decoder layer as ONE persistent kernel launch; a stack call chains one
 * launch per layer with programmatic dependent launch.
 *
 * What a launch computes (page "Muse Spark Open: 1,109 Tokens a Second Is a
 * Kernel Change, Not a Model Change", section "Where the kernel boundary sits,
 * and why it stops there"): a layer's attention through the next layer's qkv
 * projection and KV write -- GQA attention over a bf16 KV cache (sliding window
 * of 2,048 tokens or global), o-proj + residual, RMSNorm, router (top-k of E
 * experts), the pooler projection, NVFP4 expert gate/up/down with SiLU, the
 * weighted combine (section "What the 5.9 ms is still spent on"), the
 * unpooler + residual, and optionally the next layer's RMSNorm + QKV
 * projection + KV write.  The first layer of a chain runs its own RMSNorm +
 * QKV + KV write first ("The first and last layers have slightly different
 * operations", same section).  The dense variant (page "LMSYS Details SGLang
 * Megakernel ...", "Key Takeaways": the draft's dense layers, one launch each)
 * replaces router..unpooler with a bf16 SwiGLU MLP.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the device that was current
 *     when the layer was created.  Layouts are row-major, "out x in" for
 *     weights (the input dimension is contiguous), element types as stated.
 *   - Ownership: the caller owns every weight, KV cache, activation and output
 *     buffer and keeps them alive while a layer that uses them exists or a
 *     step is in flight.  Weights are borrowed and never written.  The library
 *     owns and frees its own scratch, counters, repacked scale factors and
 *     status word.
 *   - Errors: every call returns an mk_status; no call aborts, throws or
 *     prints (unless MK_LOG=1 in the environment, at create time).  Argument
 *     and shape errors are reported before anything is launched.  Launch
 *     failures return MK_ERR_CUDA.  Device-side timeouts are reported by
 *     mk_layer_status / mk_stack_status after the caller synchronises.
 *   - Steps are asynchronous on the caller's stream; the library never
 *     synchronises a stream.  One step may be in flight per layer / stack
 *     object at a time.
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer        */
  MK_ERR_UNSUPPORTED = 2,   /* shape/flag combination not built, wrong GPU arch */
  MK_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed      */
  MK_ERR_OOM = 4,           /* library-owned allocation failed                  */
  MK_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired               */
  MK_ERR_DEVICE_FAULT = 6   /* device reported an inconsistent state            */
} mk_status;

typedef enum {
  MK_FFN_MOE_NVFP4 = 0,           /* router + pooler + NVFP4 experts + unpooler */
  MK_FFN_DENSE_SWIGLU_BF16 = 1    /* bf16 SwiGLU MLP                            */
} mk_ffn_kind;

/* mk_layer_config.flags */
#define MK_FIRST_LAYER   0x1u  /* run RMSNorm + QKV + KV write on x_in first     */
#define MK_FUSE_NEXT_QKV 0x2u  /* end with the next layer's RMSNorm+QKV+KV write;
                                  it projects bf16(x_out * gain) and multiplies
                                  the sum by the RMS factor, so that it can start
                                  per 128-column tile of x_out: the same map as
                                  RMSNorm-then-QKV, with the bf16 rounding of the
                                  normalised input moved                          */
#define MK_TOPK_RENORM   0x4u  /* combine weights renormalised over the top-k    */
#define MK_PREFETCH_NEXT_KV 0x8u /* in a stack (mk_stack_step), fetch the next
                                    layer's old KV rows -- those its verify tokens
                                    will see, when K and V together are at most
                                    16 MB -- into L2 while this layer runs its
                                    last weight phases (page "Muse Spark Open:
                                    1,109 Tokens a Second ...", section "What the
                                    5.9 ms is still spent on": the next layer's
                                    old KV is prefetched into L2 before its launch
                                    lands); ignored by mk_decode_step           */

typedef struct mk_layer_config {
  int32_t hidden;         /* H, a multiple of 256                                */
  int32_t n_q_heads;      /* Hq; must equal 4 * n_kv_heads                        */
  int32_t n_kv_heads;     /* Hkv                                                 */
  int32_t head_dim;       /* d: 64 or 128                                        */
  int32_t window;         /* 0 = global; else key j visible to the query at
                             position p iff j <= p and p - j < window            */
  int32_t ffn_kind;       /* mk_ffn_kind                                         */
  int32_t n_experts;      /* E (MoE), <= 256                                     */
  int32_t top_k;          /* k (MoE), <= 8                                       */
  int32_t pooled_dim;     /* P (MoE): pooler output / expert input, % 128 == 0   */
  int32_t expert_inter;   /* I (MoE): expert intermediate, % 128 == 0            */
  int32_t dense_inter;    /* F (dense): SwiGLU intermediate, % 128 == 0          */
  int32_t max_tokens;     /* <= 16                                               */
  int32_t max_ctx;        /* KV capacity in positions (rows of each cache)       */
  float rms_eps;          /* RMSNorm epsilon; 0 selects 1e-6                      */
  uint32_t flags;         /* MK_FIRST_LAYER | MK_FUSE_NEXT_QKV | MK_TOPK_RENORM
                             | MK_PREFETCH_NEXT_KV                               */
  int32_t prefetch_experts; /* MoE, 0..16: while the router picks this step's
                               experts, the weights of the previous step's N
                               most-used experts are fetched into L2 (page
                               "Muse Spark Open: 1,109 Tokens a Second ...",
                               section "Three bills a kernel this big has to
                               pay": the 14 most-used experts); 0 = off       */
  uint64_t wait_timeout_ns; /* bound on every device-side wait; 0 -> 200 ms      */
} mk_layer_config;

/* Weights: borrowed device pointers, never written.  bf16 unless stated.
 * hidden must be a multiple of 64; Hq*d and every "in" size of a bf16 matrix a
 * multiple of 64; NVFP4 "in" sizes a multiple of 64.                          */
typedef struct mk_layer_weights {
  const void* attn_norm_w;  /* [H]            (MK_FIRST_LAYER only)             */
  const void* w_qkv;        /* [Hq*d + 2*Hkv*d, H] q heads, k heads, v heads     */
  const void* w_o;          /* [H, Hq*d]                                         */
  const void* ffn_norm_w;   /* [H]                                               */
  /* MoE */
  const void* w_router;     /* [E, H]                                            */
  const void* w_pool;       /* [P, H]                                            */
  const void* w_unpool;     /* [H, P]                                            */
  const void* exp_gate_q;   /* uint8 [E, I, P/2]: E2M1 codes, element 2i in the
                               low nibble of byte i, bit 3 = sign               */
  const void* exp_gate_s;   /* uint8 [E, I, P/16]: E4M3 scale per 16 inputs      */
  const float* exp_gate_ts; /* float [E]: tensor scale per expert matrix         */
  const void* exp_up_q;     /* uint8 [E, I, P/2]                                 */
  const void* exp_up_s;     /* uint8 [E, I, P/16]                                */
  const float* exp_up_ts;   /* float [E]                                         */
  const void* exp_down_q;   /* uint8 [E, P, I/2]                                 */
  const void* exp_down_s;   /* uint8 [E, P, I/16]                                */
  const float* exp_down_ts; /* float [E]                                         */
  /* dense */
  const void* w_gate;       /* [F, H]                                            */
  const void* w_up;         /* [F, H]                                            */
  const void* w_down;       /* [H, F]                                            */
  /* MK_FUSE_NEXT_QKV: the next layer's norm gain and QKV weight */
  const void* next_attn_norm_w; /* [H]                                           */
  const void* next_w_qkv;       /* [Hq*d + 2*Hkv*d, H]                           */
} mk_layer_weights;

/* Per-step buffers of a single-layer step (all device pointers). */
typedef struct mk_step_io {
  int32_t n_tokens;       /* T, 1..max_tokens; verify token i sits at ctx + i   */
  int32_t ctx_len;        /* positions [0, ctx) of the caches are valid          */
  const void* x_in;       /* bf16 [T, H]                                         */
  void* x_out;            /* bf16 [T, H] (must not alias x_in)                   */
  const void* q_in;       /* bf16 [T, Hq*d]; required iff !MK_FIRST_LAYER, and
                             then rows ctx..ctx+T-1 of the caches must be written */
  void* k_cache;          /* bf16 [max_ctx, Hkv, d], this layer                  */
  void* v_cache;          /* bf16 [max_ctx, Hkv, d]                              */
  void* next_k_cache;     /* MK_FUSE_NEXT_QKV: next layer's caches; rows
                             ctx..ctx+T-1 are written                            */
  void* next_v_cache;
  void* q_out;            /* MK_FUSE_NEXT_QKV: bf16 [T, Hq*d] next layer's q     */
  int32_t* topk_idx_out;  /* optional (may be NULL), MoE: int32 [T, k]           */
  float* topk_w_out;      /* optional (may be NULL), MoE: float [T, k]           */
  const uint16_t* tree_mask; /* optional HOST pointer to T uint16, read during the
                             call: token-tree verification (page "sgl-muse-mega:
                             Meta's Megakernel ...", section "What the README says
                             the kernels do": the draft's candidates form a
                             tree).  Bit j of tree_mask[i] is set iff verify
                             token j is token i itself or an ancestor of i;
                             tokens in topological order, so every mask holds
                             bit i and no bit above i, and the ancestors of an
                             ancestor are in the mask too (MK_ERR_INVALID_ARG
                             otherwise).  Token i sits at sequence position
                             ctx + depth_i (depth = its ancestors' count) and
                             keeps its K/V row at ctx + i; it sees the prefix
                             positions j < ctx with ctx + depth_i - j < window
                             and its ancestors-or-self a with depth_i - depth_a
                             < window (window 0: no limit).  NULL = the causal
                             chain (token i's ancestors are 0 .. i-1).           */
} mk_step_io;

typedef struct mk_layer mk_layer;
typedef struct mk_stack mk_stack;

/* Create a layer: validates the configuration, checks the current device is a
 * compute-capability 10.3 GPU, allocates library-owned scratch, repacks the
 * NVFP4 block scales into the tensor-core layout (library-owned copy) and
 * encodes the TMA descriptors of the weights.  Synchronous.  *out is NULL on
 * error. */
mk_status mk_layer_create(const mk_layer_config* cfg, const mk_layer_weights* w,
                          mk_layer** out);

/* Run one decode step of one layer as one persistent launch on `stream`
 * (a cudaStream_t; NULL = legacy default stream).  Asynchronous. */
mk_status mk_decode_step(mk_layer* layer, const mk_step_io* io, void* stream);

/* Device status of the layer's last step(s): MK_OK, or MK_ERR_TIMEOUT if a
 * bounded wait expired (the step's outputs are then undefined).  Reads a
 * device word synchronously; call after synchronising the step's stream.
 * The status is sticky until mk_layer_clear_status. */
mk_status mk_layer_status(mk_layer* layer);
mk_status mk_layer_clear_status(mk_layer* layer);

/* Frees library-owned memory only.  NULL is ignored. */
void mk_layer_destroy(mk_layer* layer);

/* Stacks: layers[0] must have MK_FIRST_LAYER; layers[0..n-2] must have
 * MK_FUSE_NEXT_QKV with next_w_qkv == layers[l+1]'s w_qkv and
 * next_attn_norm_w == layers[l+1]'s attn_norm_w; layers[n-1] must not fuse.
 * All layers share shapes except the window.  The stack borrows the layers
 * (destroy the stack before them). */
mk_status mk_stack_create(mk_layer* const* layers, int32_t n_layers, mk_stack** out);

typedef struct mk_stack_io {
  int32_t n_tokens;
  int32_t ctx_len;
  const void* x_in;           /* bf16 [T, H]                                   */
  void* x_out;                /* bf16 [T, H]                                   */
  void* const* k_caches;      /* host array of n_layers device pointers        */
  void* const* v_caches;      /* host array of n_layers device pointers        */
  int32_t* topk_idx_out;      /* optional: int32 [n_layers, T, k]              */
  float* topk_w_out;          /* optional: float [n_layers, T, k]              */
  const uint16_t* tree_mask;  /* optional HOST [T]: as mk_step_io.tree_mask, for
                                 every layer                                   */
} mk_stack_io;

/* One decode step through every layer: one launch per layer on `stream`,
 * chained with programmatic dependent launch.  Asynchronous. */
mk_status mk_stack_step(mk_stack* stack, const mk_stack_io* io, void* stream);
mk_status mk_stack_status(mk_stack* stack);
void mk_stack_destroy(mk_stack* stack);

/* Expert-prefetch statistics of a layer (MoE, prefetch_experts > 0), summed
 * over its steps since creation: `predicted` experts prefetched, `active`
 * experts the steps routed to, `hits` prefetched experts that were active.
 * hits / active is the share of expert weights that the prefetch covered.
 * Reads device counters synchronously: call after synchronising. */
typedef struct mk_prefetch_stats {
  uint64_t steps;
  uint64_t predicted;
  uint64_t active;
  uint64_t hits;
} mk_prefetch_stats;
mk_status mk_layer_prefetch_stats(mk_layer* layer, mk_prefetch_stats* out);
/* The same summed over the stack's layers. */
mk_status mk_stack_prefetch_stats(mk_stack* stack, mk_prefetch_stats* out);

/* Human-readable name of a status code (static storage). */
const char* mk_status_string(mk_status s);

/* Launch geometry chosen at create time (for reporting). */
typedef struct mk_layer_info {
  int32_t grid;            /* CTAs (one per SM)                                */
  int32_t threads;         /* threads per CTA                                  */
  int32_t smem_bytes;      /* dynamic shared memory per CTA                    */
  int32_t tmem_cols;       /* tensor-memory columns per CTA                    */
  int64_t scratch_bytes;   /* library-owned device bytes                       */
} mk_layer_info;
mk_status mk_layer_get_info(mk_layer* layer, mk_layer_info* info);

/* Self-timing (page "Muse Spark Open: 1,109 Tokens a Second ...", section
 * "What the 5.9 ms is still spent on": the kernel times itself with
 * %globaltimer stamps written by one lane per block).  Enabled for layers
 * created while the environment holds MK_TIMESTAMPS=1 (else this returns
 * MK_ERR_UNSUPPORTED).  Copies min(n, grid * 160) u64 of the layer's last
 * step to host memory: per CTA, 10 rows of 16 -- rows 0..8 are the phases
 * (QKV, attention, merge, o-proj, router+pool, expert gate/up, expert down,
 * unpool, next QKV) with %globaltimer stamps (epilogue start, epilogue end,
 * last MMA issued, last weight tile issued) followed by nanoseconds spent
 * (producer waiting for a free stage, MMA waiting for weights, for the token
 * operand, for a free accumulator, stager waiting for a free operand buffer,
 * stager working, epilogue waiting for an accumulator, epilogue working,
 * MMA issuing) and three more stamps (MMA starts the phase's units, stagers'
 * input dependency met, epilogue starts the phase's units);
 * row 9 starts with (kernel start, inputs ready, kernel end, this CTA's
 * router top-k start and its routing arrival -- CTAs 0..T-1 select one token
 * each --, router logits complete (in the CTA that finished the last router
 * tile), p complete seen by this CTA's stagers, its share of the p image
 * written).  All values are of the last step; stamps of
 * unused phases read 0.  Each CTA keeps them in shared memory and writes them
 * out when it exits, so that timing costs little.  Synchronous. */
mk_status mk_get_timestamps(mk_layer* layer, uint64_t* host_buf, size_t n);

/* One decode step of one layer, like mk_layer_create + mk_decode_step, but
 * allocating nothing: for callers that cannot call cudaMalloc -- code that
 * runs where device allocation is not allowed or not wanted, such as a
 * process whose device memory is handed out by another allocator or pool, or
 * one that must not grow its footprint after start-up.  (The pages describe
 * no counterpart; this is an addition of this library.)
 *
 * Every library-owned buffer of the step -- split-K and attention partials,
 * intermediates, counters, the repacked NVFP4 scale factors -- is carved out
 * of one static device array of 16 MiB that every GPU loading the library
 * holds until the process exits.  The caller still passes the weights, KV
 * caches, inputs and outputs, exactly as for mk_layer_create/mk_decode_step.
 * Layers whose buffers do not fit (roughly: small shapes such as hidden 256
 * with 16 small experts fit; the 4096-hidden, 256-expert shapes do not) are
 * rejected with MK_ERR_UNSUPPORTED before anything is launched (with
 * MK_LOG=1 a line on stderr says why); the attention split uses at most 32
 * chunks per KV head.  cfg->prefetch_experts is ignored: the shared array
 * keeps no routing history from one call to the next.
 *
 * The first call on a device performs a one-time set-up with that device
 * current (it looks up the array's device address); make that first call
 * before any stream capture.  The call is asynchronous on `stream`; every
 * call re-zeroes the counters it needs and re-derives the scale factors, and
 * all calls share the one array, so calls whose work overlaps on the GPU
 * (other streams, other threads) race and give undefined results.  A
 * device-side wait timeout leaves the outputs undefined and is not reported
 * by this call.  Same argument rules and errors as mk_layer_create and
 * mk_decode_step. */
mk_status mk_decode_step_noalloc(const mk_layer_config* cfg, const mk_layer_weights* w,
                                 const mk_step_io* io, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_H_ */
