// layer.h -- parameters of the persistent decode-layer kernel, shared by the
// host launcher (api.cu) and the kernel (layer.cu).
#pragma once
#include <cuda.h>
#include <cstdint>
#include <cuda_bf16.h>

namespace mk {

constexpr int kThreads = 384;     // 12 warps: TMA, 4 MMA issuers, 2 stagers, spare, 4 epilogue/math
constexpr int kStages = 7;        // weight ring depth (16 KB tile + 2 KB scales)
constexpr int kKC = 512;          // K elements per split-K unit (bf16 phases)
constexpr int kMaxT = 16;         // verify tokens per step (MMA N)
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;          // top-k
constexpr int kTmemCols = 512;
constexpr int kNumCounters = 16;  // grid-wide dependency counters
constexpr int kMaxPf = 16;        // experts prefetched from the previous step, at most
constexpr int kMaxGroups = 16;    // KV heads (GQA groups), at most

// Phases of one launch, in order.
enum PhaseId : int {
  PH_QKV = 0,      // first layer: RMSNorm(x_in) -> QKV, K/V rows written
  PH_ATTN = 1,     // split-KV GQA attention partials
  PH_MERGE = 2,    // merge of the attention partials -> o
  PH_O = 3,        // o-proj + residual -> x_mid
  PH_RP = 4,       // router (+ top-k) and pooler (MoE) | dense gate/up
  PH_GU = 5,       // expert gate/up (MoE)
  PH_DOWN = 6,     // expert down + combine (MoE) | dense down + residual
  PH_UNPOOL = 7,   // unpooler + residual (MoE)
  PH_NQKV = 8,     // fused next-layer RMSNorm -> QKV, next K/V rows written
  PH_COUNT = 9
};

// Grid dependency counters.  Each CTA arrives once per launch on every
// counter its layer uses; a waiter waits for (epoch + 1) * grid arrivals.
// QKV, ATTN, MERGE and GU only mark completion: the stages after them wait per
// head group (grp_sync) or per expert (exp_sync) instead.
enum BarrierId : int {
  BAR_QKV = 0,    // q and the new K/V rows written
  BAR_ATTN = 1,   // attention partials written
  BAR_MERGE = 2,  // o written
  BAR_O = 3,      // x_mid and its sum-of-squares partials written
  BAR_RP = 4,     // logits, top-k, p (MoE) | dense SwiGLU output (dense)
  BAR_GU = 5,     // expert SwiGLU rows and their amax partials written
  BAR_DOWN = 6,   // z slots and the combined y written
  BAR_X = 7,      // x_out and its sum-of-squares partials written
  BAR_END = 8,    // next layer's q and K/V rows written
  BAR_ROUTE = 9,  // router top-k written (one CTA adds grid)
  BAR_PQ = 10     // MoE: each CTA's share of the p image written
};

struct LayerParams {
  // tensor maps (weights; 128-row x 128-byte boxes, 128-byte swizzle)
  CUtensorMap tm_qkv, tm_o, tm_router, tm_pool, tm_unpool, tm_nqkv, tm_gate, tm_up, tm_down;

  // shapes
  int H, Hq, Hkv, d, window, E, topk, P, I, F, moe, first_layer, fuse_next, renorm;
  int Nqkv;                 // Hq*d + 2*Hkv*d
  float eps;
  uint64_t timeout_ns;
  int grid;

  // per-step
  int T, ctx;
  const __nv_bfloat16* x_in;
  __nv_bfloat16* x_out;
  const __nv_bfloat16* q_in;      // !first_layer
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  __nv_bfloat16* nk_cache;
  __nv_bfloat16* nv_cache;
  __nv_bfloat16* q_out;
  int32_t* topk_idx_out;
  float* topk_w_out;
  // attention visibility of the verify tokens (token tree or causal chain):
  // token t sits at position ctx + tree_depth[t]; bit j of tree_vis[t] =
  // verify token j is visible to t (ancestor-or-self within the window);
  // rows t >= T: 0
  uint16_t tree_vis[kMaxT];
  uint8_t tree_depth[kMaxT];
  int tree;                 // 1: a token tree was given (else the causal chain)
  // stacks (MK_PREFETCH_NEXT_KV): the next layer's old K and V rows, each
  // one contiguous range of nkv_bytes from nkv[0] / nkv[1] (0: none)
  const uint8_t* nkv[2];
  uint64_t nkv_bytes;

  // weights used outside TMA
  const __nv_bfloat16* attn_norm_w;
  const __nv_bfloat16* ffn_norm_w;
  const __nv_bfloat16* next_attn_norm_w;
  const float* ts_gate;
  const float* ts_up;
  const float* ts_down;
  const uint8_t* sf_gate;   // repacked scale factors (library-owned)
  const uint8_t* sf_up;
  const uint8_t* sf_down;

  // attention split
  int attn_chunks;          // chunks per KV head
  int attn_chunk_len;       // positions per chunk (multiple of 64)
  int attn_lo;              // first key position any verify token sees

  // split-K geometry of the bf16 phases: tiles of 128 rows x ksplit
  int ks_qkv, ks_o, ks_rp, ks_dgu, ks_ddown, ks_unpool;
  int tiles_qkv, tiles_o, tiles_router, tiles_pool, tiles_dgu, tiles_ddown, tiles_unpool;

  // library-owned scratch
  __nv_bfloat16* q_buf;     // [16][Hq*d]  (first layer)
  __nv_bfloat16* o_buf;     // [16][Hq*d]
  __nv_bfloat16* xmid;      // [16][H]
  __nv_bfloat16* p_buf;     // [16][P]
  __nv_bfloat16* a_buf;     // MoE [16*k][I]; dense [16][F]
  __nv_bfloat16* z_buf;     // [16*k][P]
  __nv_bfloat16* y_buf;     // [16][P]
  float* logits;            // [16][E]
  int32_t* idx;             // [16][k]
  float* wts;               // [16][k]
  float* ssq_mid;           // [H/128][16]
  float* ssq_out;           // [H/128][16]
  float* pamax;             // [P/128][16]
  float* aamax;             // [16*k][I/128]
  float* part;              // split-K partials (sized for the largest phase)
  float* attn_part;         // [Hkv*chunks][64][d + 2]
  uint32_t* fix_ctr;        // fixup counters per (phase, tile)  [PH_COUNT][256]
  uint32_t* comb_ctr;       // combine counters [16][P/128]
  uint32_t* exp_sync;       // MoE: [0, 256) finished gate/up tiles per expert (reset
                            // by CTA 0 at the end of a launch), [256, 512) expert's
                            // SwiGLU image and row scales ready (epoch + 1)
  float* srow_a;            // MoE: NVFP4 row scales of the SwiGLU rows [16*k]
  // MoE: the expert MMAs' token operands, NVFP4-quantised once per launch in
  // the layout of a shared-memory operand buffer (image_bytes(K) each: codes
  // in K-blocks of 2048 B -- 16 rows x 128 B, 128-byte swizzle -- then the
  // 512-byte scale chunks).  pq_img: p of all T tokens (row t = token t),
  // quantised in shares by the CTAs without a top-k token once p is complete;
  // aq_img [E]: the SwiGLU rows of expert e in slot order, by warp 7 of CTA
  // (e's active index) mod grid once all of e's gate/up tiles are in.
  uint8_t* pq_img;
  uint8_t* aq_img;
  // Fused next-layer QKV: its token operand bf16(x_out * gain) (the RMS
  // factor is applied after the projection) as a bf16 operand image (H/64
  // K-blocks of 2048 B: 16 rows x 128 B, 128-byte swizzle), written by the
  // final step of each 128-column tile of x_out; xt_flag [H/128]: that tile's
  // image columns and sum-of-squares partial written (epoch + 1).
  uint8_t* xn_img;
  uint32_t* xt_flag;
  uint32_t* misc_ctr;       // [0]: router tiles done, [1]: pooler tiles done,
                            // [2]: p and its amax partials complete (epoch + 1),
                            // [3]: router logits complete (epoch + 1)
  uint32_t* sched;          // [PH_COUNT] next unclaimed unit of each phase (reset by CTA 0 at the end)
  int pf_n;                 // MoE: experts prefetched from the previous step (0: off)
  int32_t* pf_list;         // [2][kMaxPf] predicted experts by launch parity, -1 ends a list
  unsigned long long* pf_stats;  // [4] steps, predicted, active, hits
  uint32_t* bar_ctr;        // [kNumCounters] grid dependency counters
  uint32_t* epoch;          // launches of this layer so far
  uint32_t* status;         // sticky error word
  // self-timing (optional, nullptr when off): %globaltimer stamps per CTA of
  // the last launch (kept in shared memory, written out at CTA exit),
  // [grid][PH_COUNT + 1][kTsSlots]: per phase 0 epilogue start, 1 epilogue
  // end, 2 last MMA issued, 3 last weight tile issued, then nanoseconds spent
  // 4 producer waiting for a free stage, 5 MMA waiting for weights, 6 MMA
  // waiting for the token operand, 7 MMA waiting for a free accumulator,
  // 8 stager waiting for a free operand buffer, 9 stager working, 10 epilogue
  // waiting for an accumulator, 11 epilogue working; 12 MMA issuing (weights
  // ready to commit); 13 MMA starts the phase's units, 14 stagers' input
  // dependency met, 15 epilogue starts the phase's units.  Last row: kernel
  // start, inputs ready, kernel end, router top-k start and release.
  uint64_t* ts;
  // per KV-head group dataflow QKV -> attention -> merge -> o-proj:
  // [0..2][kMaxGroups] counters: finished QKV tiles (growing by the group's
  // tile count per launch), attention chunks and merge items (reset by CTA 0
  // at the end of a launch)
  uint32_t* grp_sync;
  uint8_t qkv_order[64];           // QKV tile taken in claim position i (< 64): group by group
  uint8_t grp_tiles[kMaxGroups];   // QKV tiles holding rows of group g
  float* part_o;            // split-K partials of the o-proj (it overlaps the QKV phase)
  float* part_n;            // split-K partials of the fused next-layer QKV (it overlaps
                            // the fix-ups of the phase that writes x_out)
};
constexpr int kTsSlots = 16;

// Bytes of an NVFP4 operand image of K inputs (K-blocks of 256 inputs: 2 KB of
// codes and 2 KB of scale chunks each).
__host__ __device__ constexpr uint32_t image_bytes(int K) {
  return static_cast<uint32_t>((K + 255) / 256) * 4096u;
}
constexpr int kTsPerCta = (PH_COUNT + 1) * kTsSlots;

}  // namespace mk
