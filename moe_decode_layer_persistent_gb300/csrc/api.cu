// api.cu -- the mk_* C ABI: argument validation, library-owned memory, TMA
// descriptors and the launches of the persistent layer kernel (one launch per
// layer; a stack chains them with programmatic dependent launch).
#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <cstring>
#include <new>
#include <vector>

#include "host_util.h"
#include "layer.h"

namespace mk {
const void* layer_kernel_ptr();
uint32_t layer_smem_bytes();
mk_status launch_sf_repack(const void* in, void* out, int G, int N, int K, cudaStream_t s);
size_t sf_repacked_bytes(int G, int N, int K);
}  // namespace mk

using namespace mk;

struct mk_layer {
  mk_layer_config cfg;
  mk_layer_weights w;
  int device = -1;
  int sm_count = 0;
  LayerParams tmpl;                 // everything but the per-step fields
  std::vector<void*> allocs;        // library-owned device memory
  int64_t scratch_bytes = 0;
  int attn_max_chunks = 1;
};

struct mk_stack {
  std::vector<mk_layer*> layers;
  __nv_bfloat16* xbuf[2] = {nullptr, nullptr};
  __nv_bfloat16* qbuf[2] = {nullptr, nullptr};
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Split of a bf16 contraction over K into units of at most max_kb K-blocks
// (64 inputs each) that divide K evenly.  Units whose token operand is staged
// through the landing area hold at most 8 K-blocks; units that copy an operand
// image straight into the 40 KB operand buffer hold up to 16.
constexpr int kImageMaxKb = 16;
int choose_ksplit(int K, int max_kb = 8) {
  const int nkb = K / 64;
  for (int ks = 1; ks <= nkb; ++ks)
    if (nkb % ks == 0 && nkb / ks <= max_kb) return ks;
  return nkb;
}

// QKV output rows of KV-head group g: its 4 q heads, its k head, its v head.
bool tile_holds_group(const LayerParams& P, int tile, int g) {
  const int a = tile * 128, b = a + 128;
  auto hit = [&](int lo, int n) { return lo < b && lo + n > a; };
  return hit(g * 4 * P.d, 4 * P.d) || hit(P.Hq * P.d + g * P.d, P.d) ||
         hit(P.Hq * P.d + P.Hkv * P.d + g * P.d, P.d);
}

// QKV tiles in claim order, group by group (so that each group's q, k and v
// rows are finished early and its attention can start), and the number of
// tiles each group waits for.
void qkv_group_order(LayerParams& P) {
  for (int i = 0; i < 64; ++i) P.qkv_order[i] = static_cast<uint8_t>(i);
  for (int g = 0; g < kMaxGroups; ++g) P.grp_tiles[g] = 0;
  if (P.tiles_qkv > 256) return;  // rejected by the shape checks
  bool taken[256] = {};
  int order[256];
  int n = 0;
  for (int g = 0; g < P.Hkv; ++g) {
    P.grp_tiles[g] = 0;
    for (int t = 0; t < P.tiles_qkv; ++t) {
      if (!tile_holds_group(P, t, g)) continue;
      ++P.grp_tiles[g];
      if (!taken[t]) {
        taken[t] = true;
        order[n++] = t;
      }
    }
  }
  for (int t = 0; t < P.tiles_qkv; ++t)
    if (!taken[t]) order[n++] = t;
  // the kernel reorders the first 64 tiles (wider QKV projections keep their
  // order: readiness is counted per tile either way)
  if (P.tiles_qkv <= 64)
    for (int i = 0; i < P.tiles_qkv; ++i) P.qkv_order[i] = static_cast<uint8_t>(order[i]);
}

mk_status validate_config(const mk_layer_config* c, const mk_layer_weights* w) {
  if (!c || !w) return MK_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->hidden % 256) return MK_ERR_UNSUPPORTED;
  if (c->n_kv_heads <= 0 || c->n_q_heads != 4 * c->n_kv_heads) return MK_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return MK_ERR_UNSUPPORTED;
  if (c->window < 0) return MK_ERR_INVALID_ARG;
  if (c->max_tokens < 1 || c->max_tokens > kMaxT) return MK_ERR_UNSUPPORTED;
  if (c->max_ctx < 1) return MK_ERR_INVALID_ARG;
  if (c->flags & ~(MK_FIRST_LAYER | MK_FUSE_NEXT_QKV | MK_TOPK_RENORM | MK_PREFETCH_NEXT_KV))
    return MK_ERR_INVALID_ARG;
  if (c->prefetch_experts < 0 || c->prefetch_experts > kMaxPf) return MK_ERR_INVALID_ARG;
  if (c->n_kv_heads > kMaxGroups) return MK_ERR_UNSUPPORTED;
  if (!w->w_qkv && (c->flags & MK_FIRST_LAYER)) return MK_ERR_INVALID_ARG;
  if ((c->flags & MK_FIRST_LAYER) && !w->attn_norm_w) return MK_ERR_INVALID_ARG;
  if (!w->w_o || !w->ffn_norm_w) return MK_ERR_INVALID_ARG;
  if ((c->flags & MK_FUSE_NEXT_QKV) && (!w->next_w_qkv || !w->next_attn_norm_w))
    return MK_ERR_INVALID_ARG;
  if (c->ffn_kind == MK_FFN_MOE_NVFP4) {
    if (c->n_experts < 1 || c->n_experts > kMaxE) return MK_ERR_UNSUPPORTED;
    if (c->top_k < 1 || c->top_k > kMaxK || c->top_k > c->n_experts) return MK_ERR_UNSUPPORTED;
    if (c->pooled_dim < 128 || c->pooled_dim % 128 || c->pooled_dim > 2048) return MK_ERR_UNSUPPORTED;
    if (c->expert_inter < 128 || c->expert_inter % 128 || c->expert_inter > 2048)
      return MK_ERR_UNSUPPORTED;
    if (!w->w_router || !w->w_pool || !w->w_unpool || !w->exp_gate_q || !w->exp_gate_s ||
        !w->exp_gate_ts || !w->exp_up_q || !w->exp_up_s || !w->exp_up_ts || !w->exp_down_q ||
        !w->exp_down_s || !w->exp_down_ts)
      return MK_ERR_INVALID_ARG;
  } else if (c->ffn_kind == MK_FFN_DENSE_SWIGLU_BF16) {
    if (c->dense_inter < 128 || c->dense_inter % 128) return MK_ERR_UNSUPPORTED;
    if (!w->w_gate || !w->w_up || !w->w_down) return MK_ERR_INVALID_ARG;
  } else {
    return MK_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {w->attn_norm_w, w->w_qkv, w->w_o, w->ffn_norm_w, w->w_router, w->w_pool,
                        w->w_unpool, w->exp_gate_q, w->exp_up_q, w->exp_down_q, w->w_gate,
                        w->w_up, w->w_down, w->next_attn_norm_w, w->next_w_qkv};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MK_ERR_INVALID_ARG;
  return MK_OK;
}

template <class T>
mk_status dalloc(mk_layer* L, T** p, size_t count) {
  void* q = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_OOM;
  }
  if (cudaMemset(q, 0, bytes) != cudaSuccess) {
    cudaFree(q);
    return MK_ERR_CUDA;
  }
  L->allocs.push_back(q);
  L->scratch_bytes += static_cast<int64_t>(bytes);
  *p = static_cast<T*>(q);
  return MK_OK;
}

void free_layer(mk_layer* L) {
  if (!L) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (L->device >= 0) cudaSetDevice(L->device);
  for (void* p : L->allocs) cudaFree(p);
  if (cur >= 0) cudaSetDevice(cur);
  delete L;
}

#define MK_TRY(expr)                  \
  do {                                \
    mk_status _s = (expr);            \
    if (_s != MK_OK) {                \
      free_layer(L);                  \
      return _s;                      \
    }                                 \
  } while (0)

mk_status fill_step(const mk_layer* L, const mk_step_io* io, LayerParams& P) {
  const mk_layer_config& c = L->cfg;
  if (!io) return MK_ERR_INVALID_ARG;
  if (io->n_tokens < 1 || io->n_tokens > c.max_tokens) return MK_ERR_INVALID_ARG;
  if (io->ctx_len < 0 || static_cast<int64_t>(io->ctx_len) + io->n_tokens > c.max_ctx)
    return MK_ERR_INVALID_ARG;
  if (!io->x_in || !io->x_out || !io->k_cache || !io->v_cache) return MK_ERR_INVALID_ARG;
  if (io->x_in == io->x_out) return MK_ERR_INVALID_ARG;
  if (!(c.flags & MK_FIRST_LAYER) && !io->q_in) return MK_ERR_INVALID_ARG;
  if ((c.flags & MK_FUSE_NEXT_QKV) && (!io->next_k_cache || !io->next_v_cache || !io->q_out))
    return MK_ERR_INVALID_ARG;
  const void* ptrs[] = {io->x_in, io->x_out, io->q_in, io->k_cache, io->v_cache,
                        io->next_k_cache, io->next_v_cache, io->q_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return MK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(io->topk_idx_out) | reinterpret_cast<uintptr_t>(io->topk_w_out)) & 3u)
    return MK_ERR_INVALID_ARG;
  P = L->tmpl;
  P.T = io->n_tokens;
  P.ctx = io->ctx_len;
  P.x_in = static_cast<const __nv_bfloat16*>(io->x_in);
  P.x_out = static_cast<__nv_bfloat16*>(io->x_out);
  P.q_in = static_cast<const __nv_bfloat16*>(io->q_in);
  P.k_cache = static_cast<__nv_bfloat16*>(io->k_cache);
  P.v_cache = static_cast<__nv_bfloat16*>(io->v_cache);
  P.nk_cache = static_cast<__nv_bfloat16*>(io->next_k_cache);
  P.nv_cache = static_cast<__nv_bfloat16*>(io->next_v_cache);
  P.q_out = static_cast<__nv_bfloat16*>(io->q_out);
  P.topk_idx_out = io->topk_idx_out;
  P.topk_w_out = io->topk_w_out;
  // verify-token visibility: the tree's ancestor-or-self masks (validated),
  // or the causal chain
  int depth[kMaxT];
  P.tree = io->tree_mask != nullptr;
  for (int i = 0; i < kMaxT; ++i) {
    P.tree_vis[i] = 0;
    P.tree_depth[i] = 0;
  }
  for (int i = 0; i < io->n_tokens; ++i) {
    const uint32_t m = io->tree_mask ? io->tree_mask[i] : (2u << i) - 1u;
    if (!((m >> i) & 1u) || (m >> (i + 1)) != 0) return MK_ERR_INVALID_ARG;
    if (io->tree_mask)  // the ancestors of an ancestor are ancestors
      for (int j = 0; j < i; ++j)
        if (((m >> j) & 1u) && (io->tree_mask[j] & ~m) != 0) return MK_ERR_INVALID_ARG;
    depth[i] = __builtin_popcount(m) - 1;
    uint32_t vis = 0;
    for (int j = 0; j <= i; ++j)
      if (((m >> j) & 1u) && (c.window == 0 || depth[i] - depth[j] < c.window)) vis |= 1u << j;
    P.tree_vis[i] = static_cast<uint16_t>(vis);
    P.tree_depth[i] = static_cast<uint8_t>(depth[i]);
  }
  // split-KV attention: the key range every verify token may see, cut into
  // chunks of a multiple of 64 positions, about one unit per SM
  const int lo = c.window ? std::max(0, io->ctx_len - c.window + 1) : 0;
  const int n = io->ctx_len + io->n_tokens - lo;
  const int target = std::max(1, L->sm_count / c.n_kv_heads);
  int len = (n + target - 1) / target;
  len = std::max(64, (len + 63) / 64 * 64);
  P.attn_lo = lo;
  P.attn_chunk_len = len;
  P.attn_chunks = (n + len - 1) / len;
  if (P.attn_chunks > L->attn_max_chunks) return MK_ERR_UNSUPPORTED;
  return MK_OK;
}

mk_status launch(const mk_layer* L, const LayerParams& P, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(L->tmpl.grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = layer_smem_bytes();
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  lc.attrs = attr;
  lc.numAttrs = 1;
  void* args[] = {const_cast<LayerParams*>(&P)};
  MK_CUDA_TRY(cudaLaunchKernelExC(&lc, layer_kernel_ptr(), args));
  return MK_OK;
}

}  // namespace

extern "C" {

const char* mk_status_string(mk_status s) {
  switch (s) {
    case MK_OK: return "MK_OK";
    case MK_ERR_INVALID_ARG: return "MK_ERR_INVALID_ARG";
    case MK_ERR_UNSUPPORTED: return "MK_ERR_UNSUPPORTED";
    case MK_ERR_CUDA: return "MK_ERR_CUDA";
    case MK_ERR_OOM: return "MK_ERR_OOM";
    case MK_ERR_TIMEOUT: return "MK_ERR_TIMEOUT";
    case MK_ERR_DEVICE_FAULT: return "MK_ERR_DEVICE_FAULT";
  }
  return "MK_ERR_UNKNOWN";
}

mk_status mk_layer_create(const mk_layer_config* cfg, const mk_layer_weights* w, mk_layer** out) {
  if (!out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  mk_status st = validate_config(cfg, w);
  if (st != MK_OK) return st;

  int dev = -1;
  MK_CUDA_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  MK_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return MK_ERR_UNSUPPORTED;
  const void* kern = layer_kernel_ptr();
  const uint32_t smem = layer_smem_bytes();
  if (smem > prop.sharedMemPerBlockOptin) return MK_ERR_UNSUPPORTED;
  MK_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  int per_sm = 0;
  MK_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem));
  if (per_sm < 1) return MK_ERR_UNSUPPORTED;

  mk_layer* L = new (std::nothrow) mk_layer();
  if (!L) return MK_ERR_OOM;
  L->cfg = *cfg;
  L->w = *w;
  L->device = dev;
  L->sm_count = prop.multiProcessorCount;
  if (L->cfg.rms_eps == 0.f) L->cfg.rms_eps = 1e-6f;
  if (L->cfg.wait_timeout_ns == 0) L->cfg.wait_timeout_ns = 200ull * 1000 * 1000;
  const mk_layer_config& c = L->cfg;

  LayerParams& P = L->tmpl;
  std::memset(&P, 0, sizeof(P));
  P.H = c.hidden;
  P.Hq = c.n_q_heads;
  P.Hkv = c.n_kv_heads;
  P.d = c.head_dim;
  P.window = c.window;
  P.moe = c.ffn_kind == MK_FFN_MOE_NVFP4;
  P.E = P.moe ? c.n_experts : 0;
  P.topk = P.moe ? c.top_k : 0;
  P.P = P.moe ? c.pooled_dim : 0;
  P.I = P.moe ? c.expert_inter : 0;
  P.F = P.moe ? 0 : c.dense_inter;
  P.first_layer = (c.flags & MK_FIRST_LAYER) != 0;
  P.fuse_next = (c.flags & MK_FUSE_NEXT_QKV) != 0;
  P.renorm = (c.flags & MK_TOPK_RENORM) != 0;
  P.Nqkv = P.Hq * P.d + 2 * P.Hkv * P.d;
  P.eps = c.rms_eps;
  P.timeout_ns = c.wait_timeout_ns;
  P.grid = L->sm_count;
  P.pf_n = P.moe ? std::min(c.prefetch_experts, P.E) : 0;
  P.attn_norm_w = static_cast<const __nv_bfloat16*>(w->attn_norm_w);
  P.ffn_norm_w = static_cast<const __nv_bfloat16*>(w->ffn_norm_w);
  P.next_attn_norm_w = static_cast<const __nv_bfloat16*>(w->next_attn_norm_w);

  // split-K geometry
  P.ks_qkv = choose_ksplit(P.H);
  P.tiles_qkv = (P.Nqkv + 127) / 128;
  qkv_group_order(P);
  P.ks_o = choose_ksplit(P.Hq * P.d, kImageMaxKb);
  P.tiles_o = P.H / 128;
  P.ks_rp = choose_ksplit(P.H);
  if (P.moe) {
    P.tiles_router = (P.E + 127) / 128;
    P.tiles_pool = P.P / 128;
    P.ks_unpool = choose_ksplit(P.P);
    P.tiles_unpool = P.H / 128;
  } else {
    P.ks_dgu = choose_ksplit(P.H);
    P.tiles_dgu = P.F / 128;
    P.ks_ddown = choose_ksplit(P.F);
    P.tiles_ddown = P.H / 128;
  }
  if (P.tiles_qkv > 256 || P.tiles_o > 256 || P.tiles_dgu > 256 ||
      P.tiles_router + P.tiles_pool > 256)
    MK_TRY(MK_ERR_UNSUPPORTED);

  // tensor maps
  const int qd = P.Hq * P.d;
  if (P.first_layer) MK_TRY(encode_tmap_2d(&P.tm_qkv, w->w_qkv, 2, P.H, P.Nqkv, 64, 128));
  MK_TRY(encode_tmap_2d(&P.tm_o, w->w_o, 2, qd, P.H, 64, 128));
  if (P.fuse_next) MK_TRY(encode_tmap_2d(&P.tm_nqkv, w->next_w_qkv, 2, P.H, P.Nqkv, 64, 128));
  if (P.moe) {
    MK_TRY(encode_tmap_2d(&P.tm_router, w->w_router, 2, P.H, P.E, 64, 128));
    MK_TRY(encode_tmap_2d(&P.tm_pool, w->w_pool, 2, P.H, P.P, 64, 128));
    MK_TRY(encode_tmap_2d(&P.tm_unpool, w->w_unpool, 2, P.P, P.H, 64, 128));
    MK_TRY(encode_tmap_2d(&P.tm_gate, w->exp_gate_q, 1, P.P / 2,
                          static_cast<uint64_t>(P.E) * P.I, 128, 128));
    MK_TRY(encode_tmap_2d(&P.tm_up, w->exp_up_q, 1, P.P / 2,
                          static_cast<uint64_t>(P.E) * P.I, 128, 128));
    MK_TRY(encode_tmap_2d(&P.tm_down, w->exp_down_q, 1, P.I / 2,
                          static_cast<uint64_t>(P.E) * P.P, 128, 128));
    P.ts_gate = w->exp_gate_ts;
    P.ts_up = w->exp_up_ts;
    P.ts_down = w->exp_down_ts;
  } else {
    MK_TRY(encode_tmap_2d(&P.tm_gate, w->w_gate, 2, P.H, P.F, 64, 128));
    MK_TRY(encode_tmap_2d(&P.tm_up, w->w_up, 2, P.H, P.F, 64, 128));
    MK_TRY(encode_tmap_2d(&P.tm_down, w->w_down, 2, P.F, P.H, 64, 128));
  }

  // library-owned memory
  const size_t T = kMaxT;
  MK_TRY(dalloc(L, &P.q_buf, T * qd));
  MK_TRY(dalloc(L, &P.o_buf, T * qd));
  MK_TRY(dalloc(L, &P.xmid, T * P.H));
  MK_TRY(dalloc(L, &P.ssq_mid, T * (P.H / 128)));
  MK_TRY(dalloc(L, &P.ssq_out, T * (P.H / 128)));
  if (P.fuse_next) {
    MK_TRY(dalloc(L, &P.xn_img, T * P.H * 2));
    MK_TRY(dalloc(L, &P.xt_flag, P.H / 128));
  }
  size_t part = static_cast<size_t>(P.ks_qkv) * T * P.tiles_qkv * 128;
  part = std::max(part, static_cast<size_t>(P.ks_o) * T * P.tiles_o * 128);
  if (P.moe) {
    MK_TRY(dalloc(L, &P.p_buf, T * P.P));
    MK_TRY(dalloc(L, &P.a_buf, T * P.topk * P.I));
    MK_TRY(dalloc(L, &P.z_buf, T * P.topk * P.P));
    MK_TRY(dalloc(L, &P.y_buf, T * P.P));
    MK_TRY(dalloc(L, &P.logits, T * kMaxE));
    MK_TRY(dalloc(L, &P.idx, T * kMaxK));
    MK_TRY(dalloc(L, &P.wts, T * kMaxK));
    MK_TRY(dalloc(L, &P.pamax, T * (P.P / 128)));
    MK_TRY(dalloc(L, &P.aamax, T * P.topk * (P.I / 128)));
    MK_TRY(dalloc(L, &P.comb_ctr, T * (P.P / 128)));
    MK_TRY(dalloc(L, &P.exp_sync, 2 * kMaxE));
    MK_TRY(dalloc(L, &P.srow_a, T * kMaxK));
    // operand images: zero-filled here, so that inputs past K in the last
    // K-block read as zero codes and zero scales in every later step
    MK_TRY(dalloc(L, &P.pq_img, image_bytes(P.P)));
    MK_TRY(dalloc(L, &P.aq_img, static_cast<size_t>(P.E) * image_bytes(P.I)));
    MK_TRY(dalloc(L, &P.pf_list, 2 * kMaxPf));
    MK_CUDA_TRY(cudaMemset(P.pf_list, 0xFF, 2 * kMaxPf * sizeof(int32_t)));  // empty lists
    MK_TRY(dalloc(L, &P.pf_stats, 4));
    part = std::max(part, static_cast<size_t>(P.ks_rp) * T * (P.tiles_router + P.tiles_pool) * 128);
    part = std::max(part, static_cast<size_t>(P.ks_unpool) * T * P.tiles_unpool * 128);
    uint8_t* sf = nullptr;
    const size_t gu = sf_repacked_bytes(P.E, P.I, P.P), dn = sf_repacked_bytes(P.E, P.P, P.I);
    MK_TRY(dalloc(L, &sf, 2 * gu + dn));
    P.sf_gate = sf;
    P.sf_up = sf + gu;
    P.sf_down = sf + 2 * gu;
    MK_TRY(launch_sf_repack(w->exp_gate_s, sf, P.E, P.I, P.P, 0));
    MK_TRY(launch_sf_repack(w->exp_up_s, sf + gu, P.E, P.I, P.P, 0));
    MK_TRY(launch_sf_repack(w->exp_down_s, sf + 2 * gu, P.E, P.P, P.I, 0));
    if (cudaDeviceSynchronize() != cudaSuccess) MK_TRY(MK_ERR_CUDA);
  } else {
    MK_TRY(dalloc(L, &P.a_buf, T * P.F));
    part = std::max(part, static_cast<size_t>(P.ks_dgu) * 2 * T * P.tiles_dgu * 128);
    part = std::max(part, static_cast<size_t>(P.ks_ddown) * T * P.tiles_ddown * 128);
  }
  MK_TRY(dalloc(L, &P.part, part));
  MK_TRY(dalloc(L, &P.part_o, static_cast<size_t>(P.ks_o) * T * P.tiles_o * 128));
  if (P.fuse_next) MK_TRY(dalloc(L, &P.part_n, static_cast<size_t>(P.ks_qkv) * T * P.tiles_qkv * 128));
  L->attn_max_chunks = std::max(1, L->sm_count / P.Hkv);
  MK_TRY(dalloc(L, &P.attn_part,
                static_cast<size_t>(P.Hkv) * L->attn_max_chunks * 64 * (P.d + 2)));
  MK_TRY(dalloc(L, &P.fix_ctr, static_cast<size_t>(PH_COUNT) * 256));
  MK_TRY(dalloc(L, &P.misc_ctr, 4));
  MK_TRY(dalloc(L, &P.sched, PH_COUNT));
  MK_TRY(dalloc(L, &P.grp_sync, 3 * kMaxGroups));
  MK_TRY(dalloc(L, &P.bar_ctr, kNumCounters));
  MK_TRY(dalloc(L, &P.epoch, 1));
  MK_TRY(dalloc(L, &P.status, 1));
  {
    const char* e = std::getenv("MK_TIMESTAMPS");
    if (e && e[0] == '1') MK_TRY(dalloc(L, &P.ts, static_cast<size_t>(P.grid) * kTsPerCta));
  }
  if (log_enabled())
    std::fprintf(stderr,
                 "mk: layer grid=%d threads=%d smem=%u tmem=%d scratch=%lld B ffn=%s flags=%u\n",
                 P.grid, kThreads, smem, kTmemCols, static_cast<long long>(L->scratch_bytes),
                 P.moe ? "moe-nvfp4" : "dense-bf16", c.flags);
  *out = L;
  return MK_OK;
}

mk_status mk_decode_step(mk_layer* layer, const mk_step_io* io, void* stream) {
  if (!layer) return MK_ERR_INVALID_ARG;
  LayerParams P;
  mk_status st = fill_step(layer, io, P);
  if (st != MK_OK) return st;
  return launch(layer, P, static_cast<cudaStream_t>(stream), false);
}

mk_status mk_layer_status(mk_layer* layer) {
  if (!layer) return MK_ERR_INVALID_ARG;
  uint32_t s = 0;
  MK_CUDA_TRY(cudaMemcpy(&s, layer->tmpl.status, sizeof(s), cudaMemcpyDeviceToHost));
  return s == 0 ? MK_OK : MK_ERR_TIMEOUT;
}

mk_status mk_layer_clear_status(mk_layer* layer) {
  if (!layer) return MK_ERR_INVALID_ARG;
  const LayerParams& P = layer->tmpl;
  MK_CUDA_TRY(cudaDeviceSynchronize());
  MK_CUDA_TRY(cudaMemset(P.status, 0, sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.epoch, 0, sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.bar_ctr, 0, kNumCounters * sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.fix_ctr, 0, PH_COUNT * 256 * sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.misc_ctr, 0, 4 * sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.sched, 0, PH_COUNT * sizeof(uint32_t)));
  MK_CUDA_TRY(cudaMemset(P.grp_sync, 0, 3 * kMaxGroups * sizeof(uint32_t)));
  if (P.comb_ctr)
    MK_CUDA_TRY(cudaMemset(P.comb_ctr, 0, kMaxT * (P.P / 128) * sizeof(uint32_t)));
  if (P.exp_sync) MK_CUDA_TRY(cudaMemset(P.exp_sync, 0, 2 * kMaxE * sizeof(uint32_t)));
  if (P.xt_flag) MK_CUDA_TRY(cudaMemset(P.xt_flag, 0, (P.H / 128) * sizeof(uint32_t)));
  return MK_OK;
}

void mk_layer_destroy(mk_layer* layer) { free_layer(layer); }

mk_status mk_layer_get_info(mk_layer* layer, mk_layer_info* info) {
  if (!layer || !info) return MK_ERR_INVALID_ARG;
  info->grid = layer->tmpl.grid;
  info->threads = kThreads;
  info->smem_bytes = static_cast<int32_t>(layer_smem_bytes());
  info->tmem_cols = kTmemCols;
  info->scratch_bytes = layer->scratch_bytes;
  return MK_OK;
}

mk_status mk_stack_create(mk_layer* const* layers, int32_t n, mk_stack** out) {
  if (!out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  if (!layers || n < 1) return MK_ERR_INVALID_ARG;
  for (int l = 0; l < n; ++l) {
    const mk_layer* L = layers[l];
    if (!L) return MK_ERR_INVALID_ARG;
    const mk_layer_config& c = L->cfg;
    const mk_layer_config& c0 = layers[0]->cfg;
    if (c.hidden != c0.hidden || c.n_q_heads != c0.n_q_heads || c.n_kv_heads != c0.n_kv_heads ||
        c.head_dim != c0.head_dim || L->device != layers[0]->device)
      return MK_ERR_INVALID_ARG;
    const bool first = (c.flags & MK_FIRST_LAYER) != 0, fuse = (c.flags & MK_FUSE_NEXT_QKV) != 0;
    if (first != (l == 0) || fuse != (l + 1 < n)) return MK_ERR_INVALID_ARG;
    if (fuse && (L->w.next_w_qkv != layers[l + 1]->w.w_qkv ||
                 L->w.next_attn_norm_w != layers[l + 1]->w.attn_norm_w))
      return MK_ERR_INVALID_ARG;
  }
  mk_stack* S = new (std::nothrow) mk_stack();
  if (!S) return MK_ERR_OOM;
  S->layers.assign(layers, layers + n);
  const mk_layer_config& c = layers[0]->cfg;
  const size_t xe = static_cast<size_t>(kMaxT) * c.hidden;
  const size_t qe = static_cast<size_t>(kMaxT) * c.n_q_heads * c.head_dim;
  bool ok = true;
  for (int i = 0; i < 2 && ok; ++i) {
    ok = cudaMalloc(&S->xbuf[i], xe * 2) == cudaSuccess && cudaMalloc(&S->qbuf[i], qe * 2) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    mk_stack_destroy(S);
    return MK_ERR_OOM;
  }
  *out = S;
  return MK_OK;
}

mk_status mk_stack_step(mk_stack* S, const mk_stack_io* io, void* stream) {
  if (!S || !io || !io->k_caches || !io->v_caches) return MK_ERR_INVALID_ARG;
  if (io->n_tokens < 1 || io->n_tokens > kMaxT) return MK_ERR_INVALID_ARG;  // before offsets use it
  const int n = static_cast<int>(S->layers.size());
  std::vector<LayerParams> params(n);
  for (int l = 0; l < n; ++l) {
    const mk_layer* L = S->layers[l];
    mk_step_io s;
    std::memset(&s, 0, sizeof(s));
    s.n_tokens = io->n_tokens;
    s.ctx_len = io->ctx_len;
    s.x_in = l == 0 ? io->x_in : S->xbuf[(l - 1) & 1];
    s.x_out = l == n - 1 ? io->x_out : S->xbuf[l & 1];
    s.q_in = l == 0 ? nullptr : S->qbuf[(l - 1) & 1];
    s.k_cache = io->k_caches[l];
    s.v_cache = io->v_caches[l];
    if (l + 1 < n) {
      s.next_k_cache = io->k_caches[l + 1];
      s.next_v_cache = io->v_caches[l + 1];
      s.q_out = S->qbuf[l & 1];
    }
    s.tree_mask = io->tree_mask;
    const int k = L->cfg.ffn_kind == MK_FFN_MOE_NVFP4 ? L->cfg.top_k : 0;
    if (io->topk_idx_out && k)
      s.topk_idx_out = io->topk_idx_out + static_cast<size_t>(l) * io->n_tokens * k;
    if (io->topk_w_out && k) s.topk_w_out = io->topk_w_out + static_cast<size_t>(l) * io->n_tokens * k;
    mk_status st = fill_step(L, &s, params[l]);
    if (st != MK_OK) return st;
    if ((L->cfg.flags & MK_PREFETCH_NEXT_KV) && l + 1 < n) {
      // the rows [lo, ctx) the next layer's verify tokens will see, when K and
      // V together stay within kNextKvMax (a sliding-window layer's 2 x 4 MB;
      // a long global context would crowd the L2 that holds this layer's
      // prefetched unpooler and next-QKV weights)
      constexpr int64_t kNextKvMax = 16ll << 20;
      const mk_layer_config& nc = S->layers[l + 1]->cfg;
      const int64_t lo = nc.window ? std::max(0, io->ctx_len - nc.window + 1) : 0;
      const int64_t row = static_cast<int64_t>(nc.n_kv_heads) * nc.head_dim * 2;
      const int64_t bytes = (io->ctx_len - lo) * row;
      if (2 * bytes <= kNextKvMax) {
        params[l].nkv[0] = static_cast<const uint8_t*>(io->k_caches[l + 1]) + lo * row;
        params[l].nkv[1] = static_cast<const uint8_t*>(io->v_caches[l + 1]) + lo * row;
        params[l].nkv_bytes = static_cast<uint64_t>(bytes);
      }
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int l = 0; l < n; ++l) {
    mk_status r = launch(S->layers[l], params[l], st, true);
    if (r != MK_OK) return r;
  }
  return MK_OK;
}

mk_status mk_stack_status(mk_stack* S) {
  if (!S) return MK_ERR_INVALID_ARG;
  for (mk_layer* L : S->layers) {
    mk_status s = mk_layer_status(L);
    if (s != MK_OK) return s;
  }
  return MK_OK;
}

mk_status mk_layer_prefetch_stats(mk_layer* layer, mk_prefetch_stats* out) {
  if (!layer || !out) return MK_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  const LayerParams& P = layer->tmpl;
  if (!P.pf_stats) return MK_OK;
  unsigned long long v[4];
  MK_CUDA_TRY(cudaMemcpy(v, P.pf_stats, sizeof(v), cudaMemcpyDeviceToHost));
  out->steps = v[0];
  out->predicted = v[1];
  out->active = v[2];
  out->hits = v[3];
  return MK_OK;
}

mk_status mk_stack_prefetch_stats(mk_stack* S, mk_prefetch_stats* out) {
  if (!S || !out) return MK_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  for (mk_layer* L : S->layers) {
    mk_prefetch_stats s;
    mk_status st = mk_layer_prefetch_stats(L, &s);
    if (st != MK_OK) return st;
    out->steps += s.steps;
    out->predicted += s.predicted;
    out->active += s.active;
    out->hits += s.hits;
  }
  return MK_OK;
}

mk_status mk_get_timestamps(mk_layer* layer, uint64_t* host_buf, size_t n) {
  if (!layer || !host_buf) return MK_ERR_INVALID_ARG;
  const LayerParams& P = layer->tmpl;
  if (!P.ts) return MK_ERR_UNSUPPORTED;
  const size_t cap = static_cast<size_t>(P.grid) * kTsPerCta;
  MK_CUDA_TRY(cudaMemcpy(host_buf, P.ts, std::min(n, cap) * sizeof(uint64_t), cudaMemcpyDeviceToHost));
  return MK_OK;
}

void mk_stack_destroy(mk_stack* S) {
  if (!S) return;
  for (int i = 0; i < 2; ++i) {
    if (S->xbuf[i]) cudaFree(S->xbuf[i]);
    if (S->qbuf[i]) cudaFree(S->qbuf[i]);
  }
  delete S;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// mk_decode_step_noalloc: one decode step of a small layer for callers that
// may not allocate device memory at all -- code that runs where cudaMalloc is
// not allowed or not wanted (for example a host whose device memory is owned
// by another allocator or pool, or a process that has finished its start-up
// allocations).  Every library-owned buffer of the step (split-K partials,
// attention partials, intermediates, counters, the repacked NVFP4 scale
// factors) comes from the one fixed-size device array below, which every GPU
// that loads the library holds until the process exits.
namespace {

constexpr size_t kNoAllocBytes = 16u << 20;   // 16 MiB
constexpr int kNoAllocMaxChunks = 32;         // attention chunks per KV head

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  bool ready = false;
  uint8_t* base = nullptr;  // device address of g_noalloc_scratch on this device
  int sm_count = 0;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// Carves 256-byte-aligned pieces out of the scratch array (no allocation).
struct Carve {
  uint8_t* base;
  size_t used = 0;
  bool overflow = false;
  template <class T>
  T* take(size_t count) {
    const size_t bytes = (std::max<size_t>(count * sizeof(T), 16) + 255) & ~static_cast<size_t>(255);
    if (used + bytes > kNoAllocBytes) {
      overflow = true;
      return nullptr;
    }
    T* p = reinterpret_cast<T*>(base + used);
    used += bytes;
    return p;
  }
};

}  // namespace

extern "C" mk_status mk_decode_step_noalloc(const mk_layer_config* cfg, const mk_layer_weights* w,
                                            const mk_step_io* io, void* stream) {
  mk_status st = validate_config(cfg, w);
  if (st != MK_OK) return st;
  if (!io) return MK_ERR_INVALID_ARG;
  int dev = -1;
  MK_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MK_ERR_UNSUPPORTED;
  NoAllocDevice& D = g_noalloc_dev[dev];
  {
    // set-up, once per device, with that device current
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!D.ready) {
      cudaDeviceProp prop;
      MK_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
      if (prop.major != 10 || prop.minor != 3) return MK_ERR_UNSUPPORTED;
      // the same launch checks as mk_layer_create: the kernel's shared memory
      // fits and one CTA per SM can be resident
      if (layer_smem_bytes() > prop.sharedMemPerBlockOptin) return MK_ERR_UNSUPPORTED;
      void* p = nullptr;
      MK_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
      MK_CUDA_TRY(cudaFuncSetAttribute(layer_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       layer_smem_bytes()));
      int per_sm = 0;
      MK_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, layer_kernel_ptr(), kThreads,
                                                                layer_smem_bytes()));
      if (per_sm < 1) return MK_ERR_UNSUPPORTED;
      D.base = static_cast<uint8_t*>(p);
      D.sm_count = prop.multiProcessorCount;
      D.ready = true;
    }
  }
  // the layer object of mk_layer_create, assembled on the stack
  mk_layer L;
  L.cfg = *cfg;
  L.w = *w;
  L.device = dev;
  // the attention split targets sm_count / Hkv chunks per KV head; capping it
  // keeps the chunk partials inside the fixed scratch (the grid stays one CTA
  // per SM: P.grid below)
  L.sm_count = std::min(D.sm_count, kNoAllocMaxChunks * std::max(1, cfg->n_kv_heads));
  if (L.cfg.rms_eps == 0.f) L.cfg.rms_eps = 1e-6f;
  if (L.cfg.wait_timeout_ns == 0) L.cfg.wait_timeout_ns = 200ull * 1000 * 1000;
  const mk_layer_config& c = L.cfg;
  LayerParams& P = L.tmpl;
  std::memset(&P, 0, sizeof(P));
  P.H = c.hidden;
  P.Hq = c.n_q_heads;
  P.Hkv = c.n_kv_heads;
  P.d = c.head_dim;
  P.window = c.window;
  P.moe = c.ffn_kind == MK_FFN_MOE_NVFP4;
  P.E = P.moe ? c.n_experts : 0;
  P.topk = P.moe ? c.top_k : 0;
  P.P = P.moe ? c.pooled_dim : 0;
  P.I = P.moe ? c.expert_inter : 0;
  P.F = P.moe ? 0 : c.dense_inter;
  P.first_layer = (c.flags & MK_FIRST_LAYER) != 0;
  P.fuse_next = (c.flags & MK_FUSE_NEXT_QKV) != 0;
  P.renorm = (c.flags & MK_TOPK_RENORM) != 0;
  P.Nqkv = P.Hq * P.d + 2 * P.Hkv * P.d;
  P.eps = c.rms_eps;
  P.timeout_ns = c.wait_timeout_ns;
  P.grid = D.sm_count;
  P.pf_n = 0;  // the shared scratch keeps no routing history between calls
  P.attn_norm_w = static_cast<const __nv_bfloat16*>(w->attn_norm_w);
  P.ffn_norm_w = static_cast<const __nv_bfloat16*>(w->ffn_norm_w);
  P.next_attn_norm_w = static_cast<const __nv_bfloat16*>(w->next_attn_norm_w);
  P.ks_qkv = choose_ksplit(P.H);
  P.tiles_qkv = (P.Nqkv + 127) / 128;
  qkv_group_order(P);
  P.ks_o = choose_ksplit(P.Hq * P.d, kImageMaxKb);
  P.tiles_o = P.H / 128;
  P.ks_rp = choose_ksplit(P.H);
  if (P.moe) {
    P.tiles_router = (P.E + 127) / 128;
    P.tiles_pool = P.P / 128;
    P.ks_unpool = choose_ksplit(P.P);
    P.tiles_unpool = P.H / 128;
  } else {
    P.ks_dgu = choose_ksplit(P.H);
    P.tiles_dgu = P.F / 128;
    P.ks_ddown = choose_ksplit(P.F);
    P.tiles_ddown = P.H / 128;
  }
  if (P.tiles_qkv > 256 || P.tiles_o > 256 || P.tiles_dgu > 256 ||
      P.tiles_router + P.tiles_pool > 256)
    return MK_ERR_UNSUPPORTED;
  const int qd = P.Hq * P.d;
  if (P.first_layer) {
    st = encode_tmap_2d(&P.tm_qkv, w->w_qkv, 2, P.H, P.Nqkv, 64, 128);
    if (st != MK_OK) return st;
  }
  st = encode_tmap_2d(&P.tm_o, w->w_o, 2, qd, P.H, 64, 128);
  if (st == MK_OK && P.fuse_next) st = encode_tmap_2d(&P.tm_nqkv, w->next_w_qkv, 2, P.H, P.Nqkv, 64, 128);
  if (st == MK_OK && P.moe) {
    st = encode_tmap_2d(&P.tm_router, w->w_router, 2, P.H, P.E, 64, 128);
    if (st == MK_OK) st = encode_tmap_2d(&P.tm_pool, w->w_pool, 2, P.H, P.P, 64, 128);
    if (st == MK_OK) st = encode_tmap_2d(&P.tm_unpool, w->w_unpool, 2, P.P, P.H, 64, 128);
    if (st == MK_OK)
      st = encode_tmap_2d(&P.tm_gate, w->exp_gate_q, 1, P.P / 2, static_cast<uint64_t>(P.E) * P.I, 128, 128);
    if (st == MK_OK)
      st = encode_tmap_2d(&P.tm_up, w->exp_up_q, 1, P.P / 2, static_cast<uint64_t>(P.E) * P.I, 128, 128);
    if (st == MK_OK)
      st = encode_tmap_2d(&P.tm_down, w->exp_down_q, 1, P.I / 2, static_cast<uint64_t>(P.E) * P.P, 128, 128);
    P.ts_gate = w->exp_gate_ts;
    P.ts_up = w->exp_up_ts;
    P.ts_down = w->exp_down_ts;
  } else if (st == MK_OK) {
    st = encode_tmap_2d(&P.tm_gate, w->w_gate, 2, P.H, P.F, 64, 128);
    if (st == MK_OK) st = encode_tmap_2d(&P.tm_up, w->w_up, 2, P.H, P.F, 64, 128);
    if (st == MK_OK) st = encode_tmap_2d(&P.tm_down, w->w_down, 2, P.F, P.H, 64, 128);
  }
  if (st != MK_OK) return st;

  // every library-owned buffer, carved out of the scratch array
  Carve cv{D.base};
  const size_t T = kMaxT;
  P.q_buf = cv.take<__nv_bfloat16>(T * qd);
  P.o_buf = cv.take<__nv_bfloat16>(T * qd);
  P.xmid = cv.take<__nv_bfloat16>(T * P.H);
  P.ssq_mid = cv.take<float>(T * (P.H / 128));
  P.ssq_out = cv.take<float>(T * (P.H / 128));
  if (P.fuse_next) {
    P.xn_img = cv.take<uint8_t>(T * P.H * 2);
    P.xt_flag = cv.take<uint32_t>(P.H / 128);
  }
  size_t part = static_cast<size_t>(P.ks_qkv) * T * P.tiles_qkv * 128;
  part = std::max(part, static_cast<size_t>(P.ks_o) * T * P.tiles_o * 128);
  size_t gu = 0, dn = 0;
  if (P.moe) {
    P.p_buf = cv.take<__nv_bfloat16>(T * P.P);
    P.a_buf = cv.take<__nv_bfloat16>(T * P.topk * P.I);
    P.z_buf = cv.take<__nv_bfloat16>(T * P.topk * P.P);
    P.y_buf = cv.take<__nv_bfloat16>(T * P.P);
    P.logits = cv.take<float>(T * kMaxE);
    P.idx = cv.take<int32_t>(T * kMaxK);
    P.wts = cv.take<float>(T * kMaxK);
    P.pamax = cv.take<float>(T * (P.P / 128));
    P.aamax = cv.take<float>(T * P.topk * (P.I / 128));
    P.comb_ctr = cv.take<uint32_t>(T * (P.P / 128));
    P.exp_sync = cv.take<uint32_t>(2 * kMaxE);
    P.srow_a = cv.take<float>(T * kMaxK);
    P.pq_img = cv.take<uint8_t>(image_bytes(P.P));
    P.aq_img = cv.take<uint8_t>(static_cast<size_t>(P.E) * image_bytes(P.I));
    part = std::max(part, static_cast<size_t>(P.ks_rp) * T * (P.tiles_router + P.tiles_pool) * 128);
    part = std::max(part, static_cast<size_t>(P.ks_unpool) * T * P.tiles_unpool * 128);
    gu = sf_repacked_bytes(P.E, P.I, P.P);
    dn = sf_repacked_bytes(P.E, P.P, P.I);
    uint8_t* sf = cv.take<uint8_t>(2 * gu + dn);
    P.sf_gate = sf;
    P.sf_up = sf ? sf + gu : nullptr;
    P.sf_down = sf ? sf + 2 * gu : nullptr;
  } else {
    P.a_buf = cv.take<__nv_bfloat16>(T * P.F);
    part = std::max(part, static_cast<size_t>(P.ks_dgu) * 2 * T * P.tiles_dgu * 128);
    part = std::max(part, static_cast<size_t>(P.ks_ddown) * T * P.tiles_ddown * 128);
  }
  P.part = cv.take<float>(part);
  P.part_o = cv.take<float>(static_cast<size_t>(P.ks_o) * T * P.tiles_o * 128);
  if (P.fuse_next) P.part_n = cv.take<float>(static_cast<size_t>(P.ks_qkv) * T * P.tiles_qkv * 128);
  L.attn_max_chunks = std::min(kNoAllocMaxChunks, std::max(1, D.sm_count / P.Hkv));
  P.attn_part = cv.take<float>(static_cast<size_t>(P.Hkv) * L.attn_max_chunks * 64 * (P.d + 2));
  // counters that must start at zero each call: one contiguous block
  uint32_t* zero = cv.take<uint32_t>(static_cast<size_t>(PH_COUNT) * 256 + 4 + kNumCounters + 2 + PH_COUNT +
                                     3 * kMaxGroups);
  if (cv.overflow) {
    if (log_enabled())
      std::fprintf(stderr, "mk: mk_decode_step_noalloc: this layer needs more than the %zu-byte scratch\n",
                   kNoAllocBytes);
    return MK_ERR_UNSUPPORTED;
  }
  P.fix_ctr = zero;
  P.misc_ctr = zero + PH_COUNT * 256;
  P.bar_ctr = P.misc_ctr + 4;
  P.epoch = P.bar_ctr + kNumCounters;
  P.status = P.epoch + 1;
  P.sched = P.status + 1;
  P.grp_sync = P.sched + PH_COUNT;
  P.ts = nullptr;

  // per-step fields and the attention split (same rules as mk_decode_step,
  // with the chunk count capped for the fixed scratch)
  LayerParams S;
  st = fill_step(&L, io, S);
  if (st != MK_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MK_CUDA_TRY(cudaMemsetAsync(zero, 0, (static_cast<size_t>(PH_COUNT) * 256 + 4 + kNumCounters + 2 + PH_COUNT +
                                        3 * kMaxGroups) * 4, s));
  if (P.comb_ctr) MK_CUDA_TRY(cudaMemsetAsync(P.comb_ctr, 0, T * (P.P / 128) * 4, s));
  if (P.xt_flag) MK_CUDA_TRY(cudaMemsetAsync(P.xt_flag, 0, (P.H / 128) * 4, s));
  if (P.exp_sync) MK_CUDA_TRY(cudaMemsetAsync(P.exp_sync, 0, 2 * kMaxE * 4, s));
  if (P.moe) {
    // the operand images' padding past K must read as zero (an earlier call
    // may have left other shapes' data in the array)
    MK_CUDA_TRY(cudaMemsetAsync(P.pq_img, 0, image_bytes(P.P), s));
    MK_CUDA_TRY(cudaMemsetAsync(P.aq_img, 0, static_cast<size_t>(P.E) * image_bytes(P.I), s));
    st = launch_sf_repack(w->exp_gate_s, const_cast<uint8_t*>(P.sf_gate), P.E, P.I, P.P, s);
    if (st == MK_OK) st = launch_sf_repack(w->exp_up_s, const_cast<uint8_t*>(P.sf_up), P.E, P.I, P.P, s);
    if (st == MK_OK) st = launch_sf_repack(w->exp_down_s, const_cast<uint8_t*>(P.sf_down), P.E, P.P, P.I, s);
    if (st != MK_OK) return st;
  }
  return launch(&L, S, s, false);
}
