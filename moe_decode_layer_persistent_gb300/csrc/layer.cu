// layer.cu -- the persistent decode-layer kernel: one launch runs one decoder
// layer's verify step (T <= 16 tokens) on every SM.
//
// Page "Muse Spark Open: 1,109 Tokens a Second Is a Kernel Change, Not a Model
// Change", section "Where the kernel boundary sits, and why it stops there":
// one launch per layer covering attention through the next layer's qkv
// projection and KV write, one block per SM, warps with specialised roles
// (loading, tensor cores, math).  Section "Three bills a kernel this big has to
// pay": weights are streamed ahead of use into a shared-memory ring.
//
// Roles (one CTA of 384 threads per SM):
//   warp 0      TMA producer: streams 128-row weight tiles (and NVFP4 scale
//               factors) of every phase into a kStages-deep ring; it never
//               waits on activations, only on the router for expert tiles.
//   warps 1-4   tcgen05 MMA issuers (one thread each, K-step w-1 of every
//               K-block): weights are operand A (M=128 rows), the T verify
//               tokens operand B (N=16), fp32 accumulators in tensor memory,
//               two accumulator buffers.
//   warps 5-6   stagers: wait for a phase's inputs, then write the token
//               operand (RMSNorm applied, or NVFP4-quantised) into shared
//               memory in the MMA's swizzled layout.
//   warp 7      spare; in CTA 0 it keeps the expert-prefetch statistics and
//               the next step's prediction.
//   warps 8-11  epilogue (TMEM lanes 0-127) and math: split-K fix-ups,
//               residuals, router top-k, SwiGLU, combine; attention with
//               warp-level MMA in the attention phase.
// Phases are separated by grid-wide dependency counters with bounded waits.
#include "layer.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mk {

// ------------------------------------------------------------ roles
constexpr int kStagerBase = 160;   // warps 5-6
constexpr int kEpiBase = 256;      // warps 8-11 (TMEM lane quadrants 0-3)
// registers per thread: at launch (65536 / 384, rounded down to a multiple of
// 8), for warp groups 0-1, for the epilogue warp group
constexpr uint32_t kLaunchRegs = 168, kRegsRoles = 120, kRegsEpi = 256;
static_assert(2 * 128 * kRegsRoles + 128 * kRegsEpi <= 384 * kLaunchRegs, "register split");

// ------------------------------------------------------------ smem layout
constexpr uint32_t kTileBytes = 16384;                       // 128 rows x 128 B
constexpr uint32_t kSfBytes = 2048;                          // 4 chunks x 512 B
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffSF = kOffA + kStages * kTileBytes;
constexpr uint32_t kOffB = kOffSF + kStages * kSfBytes;       // 2 operand buffers
constexpr uint32_t kBBufBytes = 40960;
constexpr uint32_t kBSfOff = 16384;                          // scales inside a B buffer
constexpr uint32_t kLandOff = 16384;   // bf16 units: raw input rows (<= 16 KB), then the gain slice
constexpr uint32_t kOffMisc = kOffB + 2 * kBBufBytes;
constexpr uint32_t kOffTs = kOffMisc + 8192;                 // self-timing block
constexpr uint32_t kOffRes = (kOffTs + kTsPerCta * 8 + 127) & ~127u;  // epilogue: residual rows of a tile
constexpr uint32_t kResBytes = kMaxT * 128 * 2;
constexpr uint32_t kOffTsc = kOffRes + kResBytes;            // epilogue: experts' NVFP4 tensor scales
constexpr uint32_t kTscBytes = 3 * kMaxE * 4;
constexpr uint32_t kSmemBytes = kOffTsc + kTscBytes + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Misc {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t bfull[2];
  uint64_t bempty[2];
  uint64_t accfull[2];
  uint64_t accempty[2];
  uint64_t route_ready;
  uint64_t mma_done;
  uint64_t land[2];                // stager copies into each operand buffer (bf16 input rows or an NVFP4 image)
  uint64_t attn_free;              // the epilogue's attention no longer uses the operand buffers
  uint64_t uq_full[8];             // unit queue: slot written by the producer
  uint64_t uq_empty[8];            // unit queue: slot read by the 4 MMA issuers, stager and epilogue leaders
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t epoch;
  int n_act;                       // active experts (MoE)
  int flag;                        // epilogue broadcast
  int act[kMaxE];                  // active experts, ascending
  int cnt[kMaxE];                  // tokens per expert
  int off[kMaxE + 1];              // first slot of expert e in `slots`
  int slots[kMaxT * kMaxK];        // slot (t*k + r) grouped by expert
  float rnorm[kMaxT];              // stager: RMSNorm factors of the phase input
  float srow_st[kMaxT];            // stager: row scales of p (its share of the p image)
  float srow_b[kMaxT];             // warp 7: row scales of the expert image it builds
  float srow_ep[kMaxT * kMaxK];    // epilogue: NVFP4 row scales of the phase input
  float rnorm_ep[kMaxT];           // epilogue: RMS factors of x_out (fused next-layer QKV)
  int rn_ready;                    // epilogue: rnorm_ep computed in this launch
  float red[4][kMaxT];             // epilogue cross-warp reductions
  uint32_t comb_local[kMaxT][16];  // epilogue: this CTA's z contributions per (token, tile)
  int done_pairs[kMaxT * 16];      // epilogue: (token, tile) pairs this CTA completes
  int n_done;
  int grp_ok[4];                   // shared outcome of a group's wait: [0] stagers, [1] epilogue, [2..3] stager warps
  int pref_ok[2];                  // stagers: a unit's first input rows were copied ahead (per buffer)
  int uq[8];                       // unit queue: the CTA's next units in order, -1 ends a phase
  uint32_t land_out[2];            // stager copies issued and not yet waited for (per buffer)
};
static_assert(sizeof(Misc) <= 8192, "misc region");

struct Smem {
  uint8_t* base;
  Misc* m;
  uint64_t* ts;  // self-timing block (used only when P.ts is set)
  MK_DEV uint8_t* a_tile(int s) const { return base + kOffA + s * kTileBytes; }
  MK_DEV uint8_t* sf(int s) const { return base + kOffSF + s * kSfBytes; }
  MK_DEV uint8_t* bbuf(int b) const { return base + kOffB + b * kBBufBytes; }
  MK_DEV uint8_t* res() const { return base + kOffRes; }
  // tensor scales of the launch's active experts: [0] gate, [1] up, [2] down, by expert
  MK_DEV float* tsc(int w) const { return reinterpret_cast<float*>(base + kOffTsc) + w * kMaxE; }
};

// ------------------------------------------------------------ errors / waits
enum : uint32_t {
  ERR_TIMEOUT_FULL = 0x100, ERR_TIMEOUT_EMPTY = 0x200, ERR_TIMEOUT_B = 0x300,
  ERR_TIMEOUT_ACC = 0x400, ERR_TIMEOUT_GRID = 0x500, ERR_TIMEOUT_ROUTE = 0x600,
  ERR_TIMEOUT_DATA = 0x700, ERR_TIMEOUT_QUEUE = 0x800
};

MK_DEV bool aborted(const LayerParams& P, const Smem& S) {
  return *reinterpret_cast<volatile uint32_t*>(&S.m->abort) != 0 ||
         *reinterpret_cast<volatile uint32_t*>(P.status) != 0;
}
MK_DEV void raise_error(const LayerParams& P, const Smem& S, uint32_t code) {
  atomicCAS(P.status, 0u, code | (blockIdx.x << 16) | 1u);
  atomicExch(&S.m->abort, 1u);
}

// Bounded mbarrier wait: gives up on timeout or when the CTA/grid aborted.
// The waiting thread sleeps in the barrier (woken when the phase completes)
// and checks for an abort or a timeout about every microsecond.
MK_DEV bool wait_bar(const LayerParams& P, const Smem& S, uint64_t* bar, uint32_t parity,
                     uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, 1000u)) {
    if (aborted(P, S)) return false;
    if (globaltimer() - t0 > P.timeout_ns) {
      raise_error(P, S, code);
      return false;
    }
  }
  return true;
}

// Self-timing: each slot has one writer; the block is copied to P.ts when
// the CTA exits, so that stamping costs a shared-memory access.
MK_DEV void stamp(const LayerParams& P, const Smem& S, int ph, int slot) {
  if (P.ts) S.ts[ph * kTsSlots + slot] = globaltimer();
}
MK_DEV void stamp_add(const LayerParams& P, const Smem& S, int ph, int slot, uint64_t ns) {
  if (P.ts) S.ts[ph * kTsSlots + slot] += ns;
}
// now() only when self-timing is on (0 otherwise)
MK_DEV uint64_t tnow(const LayerParams& P) { return P.ts ? globaltimer() : 0; }

MK_DEV uint32_t grid_target(const LayerParams& P, uint32_t epoch) {
  return (epoch + 1u) * static_cast<uint32_t>(P.grid);
}

// One thread polls grid counter `id` until every CTA of this launch arrived.
MK_DEV bool grid_wait(const LayerParams& P, const Smem& S, int id, uint32_t target) {
  const uint32_t* c = P.bar_ctr + id;
  if (static_cast<int32_t>(ld_acquire(c) - target) >= 0) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    // short sleeps between polls leave the issue slots to working warps
    for (int i = 0; i < 8; ++i) {
      __nanosleep(100);
      if (static_cast<int32_t>(ld_acquire(c) - target) >= 0) return true;
    }
    if (aborted(P, S)) return false;
    if (globaltimer() - t0 > P.timeout_ns) {
      raise_error(P, S, ERR_TIMEOUT_GRID | static_cast<uint32_t>(id << 4));
      return false;
    }
  }
}

// One thread polls a flag holding the epoch + 1 of the launch that set it.
MK_DEV bool flag_wait(const LayerParams& P, const Smem& S, const uint32_t* f, uint32_t value,
                      uint32_t code) {
  if (static_cast<int32_t>(ld_acquire(f) - value) >= 0) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 8; ++i) {
      __nanosleep(100);
      if (static_cast<int32_t>(ld_acquire(f) - value) >= 0) return true;
    }
    if (aborted(P, S)) return false;
    if (globaltimer() - t0 > P.timeout_ns) {
      raise_error(P, S, code);
      return false;
    }
  }
}

MK_DEV void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Waits of a named-barrier group: one leader waits, every member gets the
// same outcome (a member must never leave the group's barrier sequence while
// others go on -- that would hang them at the next barrier).
MK_DEV bool group_mbar_wait(const LayerParams& P, const Smem& S, uint64_t* bar, uint32_t parity,
                            uint32_t code, bool leader, int bar_id, int n, int slot) {
  if (leader) S.m->grp_ok[slot] = wait_bar(P, S, bar, parity, code) ? 1 : 0;
  named_bar(bar_id, n);
  const bool ok = *reinterpret_cast<volatile int*>(&S.m->grp_ok[slot]) != 0;
  named_bar(bar_id, n);
  return ok;
}
MK_DEV bool group_grid_wait(const LayerParams& P, const Smem& S, int id, uint32_t target,
                            bool leader, int bar_id, int n, int slot) {
  if (leader) {
    const bool ok = grid_wait(P, S, id, target);
    if (!ok) atomicExch(&S.m->abort, 1u);
    S.m->grp_ok[slot] = ok ? 1 : 0;
  }
  named_bar(bar_id, n);
  const bool ok = *reinterpret_cast<volatile int*>(&S.m->grp_ok[slot]) != 0;
  named_bar(bar_id, n);
  return ok;
}
MK_DEV bool group_flag_wait(const LayerParams& P, const Smem& S, const uint32_t* f, uint32_t value,
                            bool leader, int bar_id, int n, int slot) {
  if (leader) S.m->grp_ok[slot] = flag_wait(P, S, f, value, ERR_TIMEOUT_DATA) ? 1 : 0;
  named_bar(bar_id, n);
  const bool ok = *reinterpret_cast<volatile int*>(&S.m->grp_ok[slot]) != 0;
  named_bar(bar_id, n);
  return ok;
}

// ------------------------------------------------------------ per-group dataflow
// QKV -> attention -> merge -> o-proj proceed per KV-head group g: kind 0
// counts g's finished QKV tiles (it grows by the group's tile count per launch),
// 1 its attention chunks, 2 its merged (token, head) items (both reset by CTA 0
// at the end of a launch: their counts per launch change with ctx and T).  A
// thread counts in with a release once the data it counts is written (by it,
// or by its group before a barrier) and waits for no reply; a waiter acquires
// the counter against the launch's target.
MK_DEV uint32_t* grp_ctr(const LayerParams& P, int kind, int g) { return P.grp_sync + kind * kMaxGroups + g; }
// Does QKV tile t hold rows of group g (its 4 q heads, its k and v heads)?
MK_DEV bool tile_in_group(const LayerParams& P, int t, int g) {
  const int a = t * 128, b = a + 128;
  const int q0 = g * 4 * P.d, k0 = P.Hq * P.d + g * P.d, v0 = k0 + P.Hkv * P.d;
  return (q0 < b && q0 + 4 * P.d > a) || (k0 < b && k0 + P.d > a) || (v0 < b && v0 + P.d > a);
}

// ------------------------------------------------------------ unit queue
// The producer claims the CTA's units (statically in the launch's first weight
// phase, so that it can stream before the previous launch ends; from a grid
// counter in every later phase, so that faster CTAs take more units) and
// hands them, in order, to the MMA issuers, the stagers and the epilogue
// through a ring of kUQ slots; -1 ends a phase.
constexpr int kUQ = 8;
struct QCursor {
  uint32_t slot = 0, par = 0;
  MK_DEV void advance() {
    if (++slot == kUQ) { slot = 0; par ^= 1; }
  }
};
MK_DEV bool queue_push(const LayerParams& P, const Smem& S, QCursor& q, int v) {
  if (!wait_bar(P, S, &S.m->uq_empty[q.slot], q.par ^ 1, ERR_TIMEOUT_QUEUE)) return false;
  S.m->uq[q.slot] = v;
  mbar_arrive(&S.m->uq_full[q.slot]);
  q.advance();
  return true;
}
// One thread (an MMA issuer).
MK_DEV bool queue_pop1(const LayerParams& P, const Smem& S, QCursor& q, int& v) {
  if (!wait_bar(P, S, &S.m->uq_full[q.slot], q.par, ERR_TIMEOUT_QUEUE)) return false;
  v = *reinterpret_cast<volatile int*>(&S.m->uq[q.slot]);
  mbar_arrive(&S.m->uq_empty[q.slot]);
  q.advance();
  return true;
}
// A named-barrier group (stagers or epilogue): the leader waits, everyone reads
// the slot, then the leader frees it.
MK_DEV bool queue_pop_group(const LayerParams& P, const Smem& S, QCursor& q, int& v, bool leader,
                            int bar_id, int n, int slot) {
  if (leader) S.m->grp_ok[slot] = wait_bar(P, S, &S.m->uq_full[q.slot], q.par, ERR_TIMEOUT_QUEUE) ? 1 : 0;
  named_bar(bar_id, n);
  const bool ok = *reinterpret_cast<volatile int*>(&S.m->grp_ok[slot]) != 0;
  v = *reinterpret_cast<volatile int*>(&S.m->uq[q.slot]);
  named_bar(bar_id, n);
  if (ok && leader) mbar_arrive(&S.m->uq_empty[q.slot]);
  q.advance();
  return ok;
}
constexpr int kBarEpi = 1;     // epilogue warps 8-11
constexpr int kBarStage = 2;   // stager warps 5-6
MK_DEV void epi_sync() { named_bar(kBarEpi, 128); }
MK_DEV void stage_sync() { named_bar(kBarStage, 64); }

// ------------------------------------------------------------ bf16 helpers
MK_DEV float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }
// Loads of data other CTAs wrote during this launch go to L2 (never L1, which
// is not coherent across SMs).
MK_DEV float ld_bf(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldcg(reinterpret_cast<const unsigned short*>(p))) << 16);
}
MK_DEV __nv_bfloat16 to_bf(float v) { return __float2bfloat16_rn(v); }
MK_DEV float round_bf(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
MK_DEV float silu(float x) { return x / (1.0f + expf(-x)); }

// ------------------------------------------------------------ phase geometry
MK_DEV bool phase_is_gemm(int ph) {
  return ph == PH_QKV || ph == PH_O || ph == PH_RP || ph == PH_GU || ph == PH_DOWN ||
         ph == PH_UNPOOL || ph == PH_NQKV;
}

MK_DEV bool phase_active(const LayerParams& P, int ph) {
  switch (ph) {
    case PH_QKV: return P.first_layer != 0;
    case PH_GU: case PH_UNPOOL: return P.moe != 0;
    case PH_NQKV: return P.fuse_next != 0;
    default: return true;
  }
}

// MoE down units: two adjacent 128-row tiles of one expert each (the last
// unit of an odd tile count holds one), so that one copy of the expert's
// image and one accumulator hand-off serve 256 output rows.
MK_DEV int down_pairs(const LayerParams& P) { return (P.P / 128 + 1) / 2; }

MK_DEV int phase_units(const LayerParams& P, const Smem& S, int ph) {
  switch (ph) {
    case PH_QKV: case PH_NQKV: return P.tiles_qkv * P.ks_qkv;
    case PH_O: return P.tiles_o * P.ks_o;
    case PH_RP: return P.moe ? (P.tiles_router + P.tiles_pool) * P.ks_rp : P.tiles_dgu * P.ks_dgu;
    case PH_GU: return S.m->n_act * (P.I / 128);
    case PH_DOWN: return P.moe ? S.m->n_act * down_pairs(P) : P.tiles_ddown * P.ks_ddown;
    case PH_UNPOOL: return P.tiles_unpool * P.ks_unpool;
    case PH_ATTN: return P.Hkv * P.attn_chunks;
    case PH_MERGE: return P.T * P.Hq;
  }
  return 0;
}

// First unit of this CTA in a statically dealt phase (attention chunks, merge
// items, and the first unit of the launch's first weight phase): units are
// dealt round-robin, rotated by phase so that the CTAs holding a phase's
// extra units change.
MK_DEV int first_unit(const LayerParams& P, int ph) {
  const int rot = (ph * 37) % P.grid;
  return (static_cast<int>(blockIdx.x) + P.grid - rot) % P.grid;
}

// The grid counter a phase's token operand waits for (-1: none).
MK_DEV int phase_dep(const LayerParams& P, int ph) {
  switch (ph) {
    case PH_O: return -1;  // per group of merged heads (grp_sync)
    case PH_RP: return BAR_O;
    case PH_GU: return -1;                     // the p image (misc_ctr[2])
    case PH_DOWN: return P.moe ? -1 : BAR_RP;  // MoE: per expert (exp_sync)
    case PH_UNPOOL: return BAR_DOWN;
    case PH_NQKV: return -1;  // per 128-column tile of x_out (xt_flag)
  }
  return -1;
}
// The grid counter the epilogue arrives on when a phase is done.
MK_DEV int phase_arrive(const LayerParams& P, int ph) {
  switch (ph) {
    case PH_QKV: return BAR_QKV;
    case PH_ATTN: return BAR_ATTN;
    case PH_MERGE: return BAR_MERGE;
    case PH_O: return BAR_O;
    case PH_RP: return BAR_RP;
    case PH_GU: return BAR_GU;
    case PH_DOWN: return P.moe ? BAR_DOWN : BAR_X;
    case PH_UNPOOL: return BAR_X;
    case PH_NQKV: return BAR_END;
  }
  return -1;
}
MK_DEV int final_barrier(const LayerParams& P) { return P.fuse_next ? BAR_END : BAR_X; }

struct Unit {
  const CUtensorMap* map[2];
  const uint8_t* sf[2];  // repacked scales of K-block 0 (NVFP4)
  int pair;              // 1 or 2 weight tiles (gate + up; two adjacent down tiles)
  int fp4;
  int row0;              // TMA row of the tile
  int row1;              // TMA row of the second tile of a pair
  int x0;                // TMA x of K-block 0 (elements for bf16, bytes for NVFP4)
  int nkb;               // K-blocks of 128 bytes per row
  int tile;              // 128-row tile index within its matrix
  int ks;                // K-split index
  int ksplit;
  int expert;            // NVFP4 units
  int router;            // PH_RP (MoE): 1 = router tile, 0 = pooler tile
  int N;                 // rows of the weight matrix (outputs)
  int K;                 // inputs of the weight matrix
  int col_tile;          // tile index in the phase's split-K partial columns
  int col_tiles;         // tiles in the phase's split-K partial columns
};

MK_DEV Unit make_unit(const LayerParams& P, const Smem& S, int ph, int u) {
  Unit U{};
  U.pair = 1;
  U.map[1] = nullptr;
  U.sf[0] = U.sf[1] = nullptr;
  auto bf16_unit = [&](const CUtensorMap* m, int N, int K, int ks_count, int tile_base) {
    U.map[0] = m;
    U.fp4 = 0;
    U.col_tile = u / ks_count;
    U.ks = u % ks_count;
    if (ph == PH_QKV) {
      U.col_tile = u / ks_count < 64 ? P.qkv_order[u / ks_count] : u / ks_count;  // group by group
    } else if (ph == PH_O || ph == PH_NQKV) {
      // K-slice by K-slice: an o-proj slice is one group's merged heads; a
      // next-layer QKV slice waits for the tiles of x_out it covers
      const int nt = ph == PH_O ? P.tiles_o : P.tiles_qkv;
      U.col_tile = u % nt;
      U.ks = u / nt;
    }
    U.tile = U.col_tile - tile_base;
    U.ksplit = ks_count;
    U.row0 = U.row1 = U.tile * 128;
    const int kc = K / ks_count;
    U.x0 = U.ks * kc;
    U.nkb = kc / 64;
    U.N = N;
    U.K = K;
  };
  switch (ph) {
    case PH_QKV:
      bf16_unit(&P.tm_qkv, P.Nqkv, P.H, P.ks_qkv, 0);
      U.col_tiles = P.tiles_qkv;
      break;
    case PH_NQKV:
      bf16_unit(&P.tm_nqkv, P.Nqkv, P.H, P.ks_qkv, 0);
      U.col_tiles = P.tiles_qkv;
      break;
    case PH_O:
      bf16_unit(&P.tm_o, P.H, P.Hq * P.d, P.ks_o, 0);
      U.col_tiles = P.tiles_o;
      break;
    case PH_UNPOOL:
      bf16_unit(&P.tm_unpool, P.H, P.P, P.ks_unpool, 0);
      U.col_tiles = P.tiles_unpool;
      break;
    case PH_RP:
      U.col_tiles = P.moe ? P.tiles_router + P.tiles_pool : P.tiles_dgu;
      if (P.moe) {
        if (u < P.tiles_router * P.ks_rp) {
          bf16_unit(&P.tm_router, P.E, P.H, P.ks_rp, 0);
          U.router = 1;
        } else {
          bf16_unit(&P.tm_pool, P.P, P.H, P.ks_rp, P.tiles_router);
          U.router = 0;
        }
      } else {
        bf16_unit(&P.tm_gate, P.F, P.H, P.ks_dgu, 0);
        U.map[1] = &P.tm_up;
        U.pair = 2;
      }
      break;
    case PH_DOWN:
      if (!P.moe) {
        bf16_unit(&P.tm_down, P.H, P.F, P.ks_ddown, 0);
        U.col_tiles = P.tiles_ddown;
        break;
      }
      [[fallthrough]];
    case PH_GU: {
      const bool gu = ph == PH_GU;
      const int N = gu ? P.I : P.P, K = gu ? P.P : P.I;
      const int tiles = N / 128;
      const int per = gu ? tiles : down_pairs(P);  // units per expert
      const int e = S.m->act[u / per];
      U.fp4 = 1;
      U.expert = e;
      U.tile = gu ? u % per : 2 * (u % per);
      U.ks = 0;
      U.ksplit = 1;
      U.row0 = U.row1 = e * N + U.tile * 128;
      U.x0 = 0;
      U.nkb = (K + 255) / 256;
      U.N = N;
      U.K = K;
      const size_t sf_off = (static_cast<size_t>(e) * tiles + U.tile) * U.nkb * kSfBytes;
      if (gu) {
        U.map[0] = &P.tm_gate;
        U.map[1] = &P.tm_up;
        U.pair = 2;
        U.sf[0] = P.sf_gate + sf_off;
        U.sf[1] = P.sf_up + sf_off;
      } else {
        U.map[0] = &P.tm_down;
        U.sf[0] = P.sf_down + sf_off;
        if (U.tile + 1 < tiles) {
          U.pair = 2;
          U.map[1] = &P.tm_down;
          U.row1 = U.row0 + 128;
          U.sf[1] = U.sf[0] + U.nkb * kSfBytes;
        }
      }
      break;
    }
  }
  return U;
}

// o-proj unit: the groups whose heads its K-slice of o covers.
MK_DEV int o_group_lo(const LayerParams& P, const Unit& U) { return U.x0 / (4 * P.d); }
MK_DEV int o_group_hi(const LayerParams& P, const Unit& U) {
  return (U.x0 + U.nkb * 64 - 1) / (4 * P.d);
}

// ------------------------------------------------------------ routing table
// One warp: group the (token, rank) slots by expert, deterministically
// (experts ascending, slots ascending within an expert).
MK_DEV void build_routing(const LayerParams& P, const Smem& S) {
  Misc* m = S.m;
  const int lane = lane_id();
  for (int e = lane; e < P.E; e += 32) m->cnt[e] = 0;
  __syncwarp();
  const int nslot = P.T * P.topk;
  for (int s0 = 0; s0 < nslot; s0 += 32) {
    const int s = s0 + lane;
    const int e = s < nslot ? __ldcg(P.idx + s) : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (s < nslot && (peers & ((1u << lane) - 1)) == 0) m->cnt[e] += __popc(peers);
    __syncwarp();
  }
  // exclusive scan of cnt -> off, and the active list
  int base = 0, nact = 0;
  for (int e0 = 0; e0 < P.E; e0 += 32) {
    const int e = e0 + lane;
    const int c = e < P.E ? m->cnt[e] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t act = __ballot_sync(0xffffffffu, c > 0);
    if (e < P.E) {
      m->off[e] = base + incl - c;
      if (c > 0) m->act[nact + __popc(act & ((1u << lane) - 1))] = e;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
    nact += __popc(act);
  }
  if (lane == 0) {
    m->off[P.E] = base;
    m->n_act = nact;
  }
  __syncwarp();
  // place slots: rank within the expert = earlier slots with the same expert
  for (int e = lane; e < P.E; e += 32) m->cnt[e] = 0;
  __syncwarp();
  for (int s0 = 0; s0 < nslot; s0 += 32) {
    const int s = s0 + lane;
    const int e = s < nslot ? __ldcg(P.idx + s) : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (s < nslot) {
      const int rank = __popc(peers & ((1u << lane) - 1));
      m->slots[m->off[e] + m->cnt[e] + rank] = s;
    }
    __syncwarp();
    if (s < nslot && (peers & ((1u << lane) - 1)) == 0) m->cnt[e] += __popc(peers);
    __syncwarp();
  }
}

// ============================================================ producer (warp 0)
MK_DEV int first_gemm_phase(const LayerParams& P) { return P.first_layer ? PH_QKV : PH_O; }

// L2 prefetch of this CTA's share of the experts the previous step used most
// (the prediction for this step, by launch parity): per expert the gate, up
// and down code tiles and their 2 KB scale chunks, spread over the grid.
MK_DEV void prefetch_predicted_experts(const LayerParams& P) {
  const uint32_t ep = *reinterpret_cast<const volatile uint32_t*>(P.epoch);
  // the whole list in one round trip (64 bytes, 16-byte aligned)
  const int4* l4 = reinterpret_cast<const int4*>(P.pf_list + (ep & 1u) * kMaxPf);
  int list[kMaxPf];
#pragma unroll
  for (int q = 0; q < kMaxPf / 4; ++q) {
    const int4 v = __ldcg(l4 + q);
    list[4 * q] = v.x; list[4 * q + 1] = v.y; list[4 * q + 2] = v.z; list[4 * q + 3] = v.w;
  }
  const int gt = P.I / 128, gk = (P.P + 255) / 256, dt = P.P / 128, dk = (P.I + 255) / 256;
  const int ngu = gt * gk, ndn = dt * dk, nmat = 2 * ngu + ndn, per = 2 * nmat;
#pragma unroll 1
  for (int k = 0; k < P.pf_n; ++k) {
    int e = -1;
#pragma unroll
    for (int q = 0; q < kMaxPf; ++q)
      if (q == k) e = list[q];
    if (e < 0 || e >= P.E) break;
    const int start = ((static_cast<int>(blockIdx.x) - (k * per) % P.grid) % P.grid + P.grid) % P.grid;
    for (int i = start; i < per; i += P.grid) {
      const bool sf = i >= nmat;
      int j = sf ? i - nmat : i;
      const CUtensorMap* map;
      const uint8_t* sfp;
      int row, x;
      if (j < 2 * ngu) {  // gate or up
        const bool up = j >= ngu;
        j -= up ? ngu : 0;
        const int rt = j / gk, kb = j % gk;
        map = up ? &P.tm_up : &P.tm_gate;
        sfp = (up ? P.sf_up : P.sf_gate) + ((static_cast<size_t>(e) * gt + rt) * gk + kb) * kSfBytes;
        row = e * P.I + rt * 128;
        x = kb * 128;
      } else {            // down
        j -= 2 * ngu;
        const int rt = j / dk, kb = j % dk;
        map = &P.tm_down;
        sfp = P.sf_down + ((static_cast<size_t>(e) * dt + rt) * dk + kb) * kSfBytes;
        row = e * P.P + rt * 128;
        x = kb * 128;
      }
      if (sf) bulk_prefetch_l2(sfp, kSfBytes);
      else tma_prefetch_2d(map, x, row);
    }
  }
}

// Warp 7 of CTA 0, once the routing is known: how many of this step's
// prefetched experts were routed to, and the next step's prediction (the
// experts with the most tokens, an equal count going to the lower index).
MK_DEV void prefetch_bookkeeping(const LayerParams& P, const Smem& S, uint32_t epoch) {
  Misc* m = S.m;
  if (!wait_bar(P, S, &m->route_ready, 0, ERR_TIMEOUT_ROUTE)) return;
  const int lane = lane_id();
  const int32_t* cur = P.pf_list + (epoch & 1u) * kMaxPf;
  int32_t* nxt = P.pf_list + ((epoch + 1u) & 1u) * kMaxPf;
  uint32_t pred = 0, hit = 0;
  if (lane < P.pf_n) {
    const int e = cur[lane];
    if (e >= 0 && e < P.E) {
      pred = 1;
      hit = m->off[e + 1] > m->off[e] ? 1u : 0u;
    }
  }
  pred = __reduce_add_sync(0xffffffffu, pred);
  hit = __reduce_add_sync(0xffffffffu, hit);
  if (lane == 0) {
    atomicAdd(P.pf_stats + 0, 1ull);
    atomicAdd(P.pf_stats + 1, static_cast<unsigned long long>(pred));
    atomicAdd(P.pf_stats + 2, static_cast<unsigned long long>(m->n_act));
    atomicAdd(P.pf_stats + 3, static_cast<unsigned long long>(hit));
  }
  uint32_t key[kMaxE / 32];
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = lane + 32 * i;
    const int c = e < P.E ? m->off[e + 1] - m->off[e] : 0;
    key[i] = c > 0 ? (static_cast<uint32_t>(c) << 16) | (0xFFFFu - e) : 0u;
  }
#pragma unroll 1
  for (int r = 0; r < kMaxPf; ++r) {
    uint32_t b = 0u;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) b = max(b, key[i]);
    const uint32_t wk = r < P.pf_n ? __reduce_max_sync(0xffffffffu, b) : 0u;
    const int e = wk ? static_cast<int>(0xFFFFu - (wk & 0xFFFFu)) : -1;
    if (lane == 0) nxt[r] = e;
    if (e >= 0 && (e & 31) == lane) {
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i)
        if (i == (e >> 5)) key[i] = 0u;
    }
  }
}

// L2 prefetch of this CTA's 1/grid share of the next layer's old K and V rows
// (a stack's MK_PREFETCH_NEXT_KV), in 16 KB pieces.
MK_DEV void prefetch_next_kv(const LayerParams& P) {
  constexpr uint64_t kPiece = 16384;
  const uint64_t pieces = (P.nkv_bytes + kPiece - 1) / kPiece;
  for (int m = 0; m < 2; ++m)
    for (uint64_t i = blockIdx.x; i < pieces; i += P.grid) {
      const uint64_t off = i * kPiece;
      const uint64_t n = P.nkv_bytes - off < kPiece ? P.nkv_bytes - off : kPiece;
      bulk_prefetch_l2(P.nkv[m] + off, static_cast<uint32_t>(n & ~15ull));
    }
}


MK_DEV void run_producer(const LayerParams& P, const Smem& S) {
  Misc* m = S.m;
  const uint64_t pol = policy_evict_first();
  uint32_t stage = 0, phase = 0;
  QCursor q;
  bool route_known = false, prev_done = false;
  bool ok = true;
  const int ph0 = first_gemm_phase(P);
  for (int ph = 0; ph < PH_COUNT && ok; ++ph) {
    if (!phase_is_gemm(ph) || !phase_active(P, ph)) continue;
    if (P.moe && ph == PH_GU && !route_known) {
      // The unpooler and next-layer QKV weights are not fetched into L2 here:
      // that 66 MB burst delayed the first gate/up tiles and the epilogues'
      // stores more than it saved later (4.4 us per layer on the stack).
      if (P.pf_n > 0) {
        if (!prev_done) {
          pdl_wait();
          prev_done = true;
        }
        prefetch_predicted_experts(P);
      }
      if (!wait_bar(P, S, &m->route_ready, 0, ERR_TIMEOUT_ROUTE)) { ok = false; break; }
      route_known = true;
    }
    // the launch's last weight phases before the fused next QKV run from L2
    // (unpooler) or stream while HBM has room: fetch the next layer's old KV
    if (P.nkv_bytes && ph == (P.moe ? PH_UNPOOL : PH_DOWN)) prefetch_next_kv(P);
    // The launch's first weight phase starts with one unit per CTA dealt
    // statically (streamed before the previous launch ends); all other units
    // are claimed from the phase's counter, once the previous launch of this
    // layer (which resets the counters at its end) is complete.
    const int n = phase_units(P, S, ph);
    bool first = ph == ph0;
    int u = first_unit(P, ph);
    while (ok) {
      if (!first) {
        if (!prev_done) {
          pdl_wait();
          prev_done = true;
        }
        u = static_cast<int>(atomicAdd(P.sched + ph, 1u)) + (ph == ph0 ? P.grid : 0);
      }
      first = false;
      const bool end = u >= n;
      if (!queue_push(P, S, q, end ? -1 : u)) { ok = false; break; }
      if (end) break;
      const Unit U = make_unit(P, S, ph, u);
      const uint32_t bytes = kTileBytes + (U.fp4 ? kSfBytes : 0);
      for (int kb = 0; kb < U.nkb && ok; ++kb) {
        for (int j = 0; j < U.pair; ++j) {
          const uint64_t w0 = tnow(P);
          if (!wait_bar(P, S, &m->empty[stage], phase ^ 1, ERR_TIMEOUT_EMPTY)) { ok = false; break; }
          if (P.ts) stamp_add(P, S, ph, 4, globaltimer() - w0);
          mbar_arrive_expect_tx(&m->full[stage], bytes);
          const int x = U.x0 + kb * (U.fp4 ? 128 : 64);
          tma_load_2d(S.a_tile(stage), U.map[j], &m->full[stage], x, j ? U.row1 : U.row0, pol);
          if (U.fp4) bulk_load(S.sf(stage), U.sf[j] + kb * kSfBytes, kSfBytes, &m->full[stage], pol);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    }
    stamp(P, S, ph, 3);
  }
  // Drain: every issued copy must land before the CTA may exit.
  for (int s = 0; s < kStages; ++s) {
    // the most recent use of stage s had parity (phase ^ (s >= stage ? 1 : 0))
    const uint32_t par = s < static_cast<int>(stage) ? phase : phase ^ 1;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait_sleep(&m->full[s], par, 1000u)) {
      if (globaltimer() - t0 > P.timeout_ns) break;
    }
  }
}

// ============================================================ MMA (warps 1-4, one thread each)
// A 128-byte K-block of a weight tile holds four MMA K-steps (4 x 16 bf16 or
// 4 x 64 NVFP4 elements).  MMA warp l+1 issues K-step l of every K-block (and
// copies that step's scale factors) into its own accumulator: a thread waits
// ~100-200 cycles per tcgen05 instruction it issues, and four issuing warps
// keep four times as many in flight.  The epilogue adds the four partial
// accumulators.
// TMEM columns: accumulators at 128*b + 64*j + 16*l (buffer b, matrix j of a
// gate/up pair, lane l); scale factors at 256 + 48*r (r = K-block parity):
// token operand 16 columns, then 16 per weight matrix (4 per lane).
MK_DEV void run_mma(const LayerParams& P, const Smem& S) {
  Misc* m = S.m;
  const uint32_t l = (threadIdx.x >> 5) - 1;  // 0..3
  const uint32_t tbase = m->tmem_base;
  uint32_t stage = 0, phase = 0, acc_ph[2] = {0, 0}, b_ph[2] = {0, 0};
  uint32_t ucount = 0, sfreg = 0;
  QCursor q;
  bool ok = true;
  bool route_known = false;
  for (int ph = 0; ph < PH_COUNT && ok; ++ph) {
    if (!phase_is_gemm(ph) || !phase_active(P, ph)) continue;
    if (P.moe && ph == PH_GU && !route_known) {
      if (!wait_bar(P, S, &m->route_ready, 0, ERR_TIMEOUT_ROUTE)) { ok = false; break; }
      route_known = true;
    }
    if (l == 0) stamp(P, S, ph, 13);
    while (ok) {
      int u;
      if (!queue_pop1(P, S, q, u)) { ok = false; break; }
      if (u < 0) break;
      const Unit U = make_unit(P, S, ph, u);
      const uint32_t b = ucount & 1;
      uint64_t w0 = tnow(P);
      if (!wait_bar(P, S, &m->accempty[b], acc_ph[b] ^ 1, ERR_TIMEOUT_ACC)) { ok = false; break; }
      uint64_t w1 = tnow(P);
      if (!wait_bar(P, S, &m->bfull[b], b_ph[b], ERR_TIMEOUT_B)) { ok = false; break; }
      if (P.ts && l == 0) {
        const uint64_t w2 = globaltimer();
        stamp_add(P, S, ph, 7, w1 - w0);
        stamp_add(P, S, ph, 6, w2 - w1);
      }
      tc_fence_after();
      uint8_t* bb = S.bbuf(b);
      for (int kb = 0; kb < U.nkb && ok; ++kb) {
        for (int j = 0; j < U.pair; ++j) {
          const uint64_t wf = tnow(P);
          if (!wait_bar(P, S, &m->full[stage], phase, ERR_TIMEOUT_FULL)) { ok = false; break; }
          const uint64_t wi = tnow(P);
          if (P.ts && l == 0) stamp_add(P, S, ph, 5, wi - wf);
          tc_fence_after();
          const uint64_t da = sdesc_kmajor_sw128(smem_u32(S.a_tile(stage))) + 2 * l;
          const uint64_t db = sdesc_kmajor_sw128(smem_u32(bb + kb * 2048)) + 2 * l;
          const uint32_t d = tbase + 128 * b + 64 * j + 16 * l;
          if (U.fp4) {
            const uint32_t reg = tbase + 256 + 48 * (sfreg & 1);
            const uint32_t sfb = reg + 4 * l, sfa = reg + 16 + 16 * j + 4 * l;
            tmem_cp_sf(sfa, sdesc_sf_chunk(smem_u32(S.sf(stage) + l * 512)));
            if (j == 0)
              tmem_cp_sf(sfb, sdesc_sf_chunk(smem_u32(bb + kBSfOff + (kb * 4 + l) * 512)));
            mma_nvf4(d, da, db, idesc_nvf4(128, kMaxT), sfa, sfb, kb != 0);
            if (j == U.pair - 1) ++sfreg;
          } else {
            mma_bf16(d, da, db, idesc_bf16(128, kMaxT), kb != 0);
          }
          mma_commit(&m->empty[stage]);
          if (P.ts && l == 0) stamp_add(P, S, ph, 12, globaltimer() - wi);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) break;
      mma_commit(&m->accfull[b]);
      mma_commit(&m->bempty[b]);
      acc_ph[b] ^= 1;
      b_ph[b] ^= 1;
      ++ucount;
    }
    if (l == 0) stamp(P, S, ph, 2);
  }
  // all issued tensor-core work completes before TMEM is released
  mma_commit(&m->mma_done);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait_sleep(&m->mma_done, 0, 1000u)) {
    if (globaltimer() - t0 > P.timeout_ns) break;
  }
}

// ============================================================ stagers (warps 5-6)
// Token operand of a bf16 unit.  The stager leader bulk-copies rows t < T of
// src[t][k0 .. k0 + 64*nkb) (and the gain slice) into the landing area of the
// operand buffer (issue_bf16, possibly one unit ahead); then all stager
// threads write the swizzled operand, as bf16(x * rnorm[t] * gain[k]) when a
// gain is given (stage_bf16).  Rows >= T are zero.
struct BfSrc {
  const __nv_bfloat16* src;
  int ld;
  const __nv_bfloat16* gain;
};
MK_DEV BfSrc bf_source(const LayerParams& P, int ph) {
  switch (ph) {
    case PH_QKV: return {P.x_in, P.H, P.attn_norm_w};
    case PH_NQKV: return {P.x_out, P.H, P.next_attn_norm_w};
    case PH_RP: return {P.xmid, P.H, P.ffn_norm_w};
    default: return {P.a_buf, P.F, nullptr};  // dense down
  }
}

// bf16 operand images.  The o-proj input (the merged attention output) and
// the unpooler input (the combined expert output) are written by their
// producers straight into the layout of an operand buffer: K-blocks of 64
// inputs, each 16 rows x 128 B (2048 B), SW128-swizzled.  A unit's token
// operand is then one bulk copy of its K-slice (rows >= T hold whatever an
// earlier step left: each row only reaches its own accumulator column, which
// the epilogue does not read).
MK_DEV uint32_t bf_image_off(int t, int k) {
  return static_cast<uint32_t>(k >> 6) * 2048u + sw128_offset(t, (k & 63) * 2);
}
MK_DEV bool image_phase(int ph) { return ph == PH_O || ph == PH_UNPOOL || ph == PH_NQKV; }
MK_DEV const uint8_t* bf_image(const LayerParams& P, int ph) {
  if (ph == PH_NQKV) return P.xn_img;
  return reinterpret_cast<const uint8_t*>(ph == PH_O ? P.o_buf : P.y_buf);
}

MK_DEV void issue_bf16(const LayerParams& P, const Smem& S, int ph, const Unit& U, int buf) {
  const BfSrc src = bf_source(P, ph);
  uint8_t* raw = S.bbuf(buf) + kLandOff;
  uint8_t* graw = raw + kMaxT * U.nkb * 128;
  const uint32_t rowbytes = static_cast<uint32_t>(U.nkb) * 128u;
  // normal priority: each layer of a stack has its own activation buffers,
  // and evict-last lines of 62 layers would crowd L2
  const uint64_t pol = policy_evict_normal();
  uint64_t* lb = &S.m->land[buf];
  S.m->land_out[buf] = 1;
  // the rows were written by ordinary stores (of this and other CTAs),
  // released to this thread: order them before its async-proxy copies
  fence_proxy_async_global();
  mbar_arrive_expect_tx(lb, P.T * rowbytes + (src.gain ? rowbytes : 0u));
  for (int t = 0; t < P.T; ++t)
    bulk_load(raw + t * rowbytes, src.src + static_cast<size_t>(t) * src.ld + U.x0, rowbytes, lb, pol);
  if (src.gain) bulk_load(graw, src.gain + U.x0, rowbytes, lb, pol);
}

MK_DEV bool stage_bf16(const LayerParams& P, const Smem& S, int ph, const Unit& U, int buf,
                       bool issued, uint32_t& land_ph) {
  const int tid = threadIdx.x - kStagerBase;
  if (!issued && tid == 0) issue_bf16(P, S, ph, U, buf);
  uint8_t* bb = S.bbuf(buf);
  const int nkb = U.nkb;
  const bool gain = bf_source(P, ph).gain != nullptr;
  uint8_t* raw = bb + kLandOff;
  uint8_t* graw = raw + kMaxT * nkb * 128;
  const uint32_t rowbytes = static_cast<uint32_t>(nkb) * 128u;
  if (!group_mbar_wait(P, S, &S.m->land[buf], land_ph, ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0))
    return false;
  land_ph ^= 1;
  if (tid == 0) S.m->land_out[buf] = 0;
  const int chunks = nkb * 8;  // 16-byte chunks per row
  for (int i = tid; i < kMaxT * chunks; i += 64) {
    const int t = i / chunks, c = i % chunks;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (t < P.T) {
      v = *reinterpret_cast<const uint4*>(raw + t * rowbytes + c * 16);
      if (gain) {
        const uint4 g = *reinterpret_cast<const uint4*>(graw + c * 16);
        const float r = S.m->rnorm[t];
        uint32_t* pv = reinterpret_cast<uint32_t*>(&v);
        const uint32_t* pg = reinterpret_cast<const uint32_t*>(&g);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float x0 = __uint_as_float(pv[w] << 16), x1 = __uint_as_float(pv[w] & 0xFFFF0000u);
          const float g0 = __uint_as_float(pg[w] << 16), g1 = __uint_as_float(pg[w] & 0xFFFF0000u);
          const __nv_bfloat162 o = __floats2bfloat162_rn(x0 * r * g0, x1 * r * g1);
          pv[w] = *reinterpret_cast<const uint32_t*>(&o);
        }
      }
    }
    const int byte = c * 16;
    *reinterpret_cast<uint4*>(bb + (byte >> 7) * 2048 + sw128_offset(t, byte & 127)) = v;
  }
  return true;
}

// Router logits as 32-bit keys whose unsigned order is the float order.
MK_DEV uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);  // -0 ranks as +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
MK_DEV float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Router top-k of token t by one warp: the k largest float32 logits
// (descending, an exact tie going to the lower expert index), the softmax
// over all experts (maximum subtracted), the combine weights.  Lane l holds
// experts l + 32 i as order-preserving keys; a round takes the warp's maximum
// key, then the lowest expert index holding it, and clears that key.
MK_DEV void topk_token(const LayerParams& P, int t) {
  constexpr int kI = kMaxE / 32;  // experts per lane
  const int lane = lane_id();
  const float* lg = P.logits + static_cast<size_t>(t) * kMaxE;
  uint32_t k[kI];
#pragma unroll
  for (int i = 0; i < kI; ++i) {
    const int e = lane + 32 * i;
    k[i] = e < P.E ? order_key(__ldcg(lg + e)) : 0u;  // 0: no expert
  }
  uint32_t mk = 0u;
#pragma unroll
  for (int i = 0; i < kI; ++i) mk = max(mk, k[i]);
  const float mx = key_logit(__reduce_max_sync(0xffffffffu, mk));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kI; ++i)
    if (k[i] != 0u) s += __expf(key_logit(k[i]) - mx);
  s = warp_sum(s);
  int ek = 0;
  uint32_t wk = 0u;
#pragma unroll 1
  for (int r = 0; r < P.topk; ++r) {
    uint32_t b = 0u;
    int ib = 0;
#pragma unroll
    for (int i = kI - 1; i >= 0; --i)
      if (k[i] >= b && k[i] != 0u) { b = k[i]; ib = i; }
    const uint32_t x = __reduce_max_sync(0xffffffffu, b);
    const int c = static_cast<int>(__reduce_min_sync(
        0xffffffffu, (b == x && x != 0u) ? static_cast<uint32_t>(ib * 32 + lane) : 0xffffffffu));
#pragma unroll
    for (int i = 0; i < kI; ++i)
      if ((c & 31) == lane && i == (c >> 5)) k[i] = 0u;
    if (lane == r) { ek = c; wk = x; }
  }
  float wt = lane < P.topk ? __expf(key_logit(wk) - mx) / s : 0.f;
  if (P.renorm) wt = wt / warp_sum(wt);
  if (lane < P.topk) {
    P.idx[t * P.topk + lane] = ek;
    P.wts[t * P.topk + lane] = wt;
    if (P.topk_idx_out) P.topk_idx_out[t * P.topk + lane] = ek;
    if (P.topk_w_out) P.topk_w_out[t * P.topk + lane] = wt;
  }
}

// NVFP4 operand image (codes in K-blocks of 2048 B, then the scale chunks) of
// `rows` bf16 rows of K inputs, by `nthr` threads (this one: `tid`): image
// row i is the row at src + off(i), with row scale srow[i] (shared memory).
// The codes and scales go to `img` (global) and, when `sm` is given, to an
// operand buffer in shared memory (codes at its start, scales at kBSfOff).
// Each thread loads four 16-element blocks before quantising them, so that
// four L2 round trips overlap.  The readers of `img` copy it with the async
// proxy after acquiring the release that publishes it, behind a proxy fence
// of their own.
template <class Off>
MK_DEV void quantize_image(uint8_t* img, uint8_t* sm, int rows, int K, const float* srow,
                           const __nv_bfloat16* src, Off off, int tid, int nthr) {
  const int nblk = K / 16;
  const int total = rows * nblk;
  OperandSink sink{img, img + ((K + 255) / 256) * 2048, 0};
  OperandSink sink_s{sm, sm + kBSfOff, 0};
  for (int i0 = tid; i0 < total; i0 += 4 * nthr) {
    uint4 r[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * nthr;
      if (i < total) {
        const uint4* p = reinterpret_cast<const uint4*>(src + off(i / nblk) + (i % nblk) * 16);
        r[q][0] = __ldcg(p);
        r[q][1] = __ldcg(p + 1);
      }
    }
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * nthr;
      if (i >= total) break;
      // select the block's registers (no dynamically indexed array)
      const uint4 c0 = q == 0 ? r[0][0] : q == 1 ? r[1][0] : q == 2 ? r[2][0] : r[3][0];
      const uint4 c1 = q == 0 ? r[0][1] : q == 1 ? r[1][1] : q == 2 ? r[2][1] : r[3][1];
      const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      float x[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
      uint32_t w0, w1, sb;
      quantize_block16(x, srow[i / nblk], w0, w1, sb);
      sink.r = sink_s.r = static_cast<uint32_t>(i / nblk);
      if (img) sink.put(i % nblk, w0, w1, sb);
      if (sm) sink_s.put(i % nblk, w0, w1, sb);
    }
  }
}

// The sum (in index order, from 0) or the maximum (from 0) of the n
// per-tile partials p[j * stride], j < n.  The loads go out 32 at a time, so
// that the partials of a 4096-wide row cost one L2 round trip, not one per
// partial; the arithmetic is that of the plain loop.
template <bool kMax>
MK_DEV float reduce_partials(const float* p, int n, int stride) {
  float acc = 0.f;
  for (int j0 = 0; j0 < n; j0 += 32) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = j0 + k < n ? __ldcg(p + static_cast<size_t>(j0 + k) * stride) : 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k)
      if (j0 + k < n) acc = kMax ? fmaxf(acc, v[k]) : acc + v[k];
  }
  return acc;
}

// NVFP4 row scale of p's row t (amax over the pooler tiles' partials).
MK_DEV float p_row_scale(const LayerParams& P, int t) {
  const float a = reduce_partials<true>(P.pamax + t, P.P / 128, kMaxT);
  return a > 0.f ? __fdiv_rn(a, 2688.0f) : 1.0f;
}

// Share `sharer` (of `nsh`) of the p image's 16-element blocks (T rows of P),
// by the 64 stager threads: one block per thread at the full shapes.  The
// block's values are in flight while the row scales are gathered.
MK_DEV void p_image_share(const LayerParams& P, const Smem& S, int tid, int sharer, int nsh) {
  Misc* m = S.m;
  const int nblk = P.P / 16, total = P.T * nblk;
  const int per = (total + nsh - 1) / nsh;
  const int lo = sharer * per, hi = min(total, lo + per);
  float x[16];
  if (lo + tid < hi) load_bf16x16_cg(P.p_buf + static_cast<size_t>((lo + tid) / nblk) * P.P + ((lo + tid) % nblk) * 16, x);
  if (tid < P.T) m->srow_st[tid] = p_row_scale(P, tid);
  stage_sync();
  OperandSink sink{P.pq_img, P.pq_img + ((P.P + 255) / 256) * 2048, 0};
  for (int i = lo + tid; i < hi; i += 64) {
    const int t = i / nblk, b = i % nblk;
    if (i != lo + tid) load_bf16x16_cg(P.p_buf + static_cast<size_t>(t) * P.P + b * 16, x);
    uint32_t w0, w1, sb;
    quantize_block16(x, m->srow_st[t], w0, w1, sb);
    sink.r = static_cast<uint32_t>(t);
    sink.put(b, w0, w1, sb);
  }
}

// Warp 7 (MoE): once the routing is known, the SwiGLU images of the active
// experts i = blockIdx.x, blockIdx.x + grid, ... (at most one per CTA at the
// full shapes): wait until all of the expert's gate/up tiles are counted in,
// compute the NVFP4 row scales of its rows (amax over the tiles' partials),
// quantise the rows once into the expert's image and release it to the down
// units of every CTA.
MK_DEV void build_expert_images(const LayerParams& P, const Smem& S, uint32_t epoch) {
  Misc* m = S.m;
  const int lane = lane_id();
  if (!wait_bar(P, S, &m->route_ready, 0, ERR_TIMEOUT_ROUTE)) return;
  for (int i = blockIdx.x; i < m->n_act; i += P.grid) {
    const int e = m->act[i];
    int ok = 1;
    if (lane == 0) ok = flag_wait(P, S, P.exp_sync + e, static_cast<uint32_t>(P.I / 128), ERR_TIMEOUT_DATA) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    __syncwarp();  // the lanes' loads below follow lane 0's acquire
    const int n = m->off[e + 1] - m->off[e];
    const int* sl = m->slots + m->off[e];
    if (lane < n) {
      const float a = reduce_partials<true>(P.aamax + sl[lane] * (P.I / 128), P.I / 128, 1);
      const float sr = a > 0.f ? __fdiv_rn(a, 2688.0f) : 1.0f;
      P.srow_a[sl[lane]] = sr;
      m->srow_b[lane] = sr;
    }
    __syncwarp();
    const int ld = P.I;
    quantize_image(P.aq_img + static_cast<size_t>(e) * image_bytes(P.I), nullptr, n, P.I, m->srow_b, P.a_buf,
                   [sl, ld](int r) { return static_cast<size_t>(sl[r]) * ld; }, lane, 32);
    __syncwarp();  // every lane's image and scale writes precede lane 0's release
    if (lane == 0) st_release(P.exp_sync + kMaxE + e, epoch + 1u);
  }
}

// Token operand of an NVFP4 expert unit: an operand image quantised once per
// launch (the p image for every gate/up unit, the expert's SwiGLU image for a
// down unit), bulk-copied by the stager leader into operand buffer `buf`:
// codes to the buffer's start, scale chunks to kBSfOff.
MK_DEV void issue_image(const LayerParams& P, const Smem& S, const uint8_t* img, int K, int buf) {
  const uint32_t half = image_bytes(K) / 2;
  uint64_t* lb = &S.m->land[buf];
  S.m->land_out[buf] = 1;
  mbar_arrive_expect_tx(lb, 2 * half);
  const uint64_t pol = policy_evict_normal();  // see issue_bf16
  bulk_load(S.bbuf(buf), img, half, lb, pol);
  bulk_load(S.bbuf(buf) + kBSfOff, img + half, half, lb, pol);
}

// The stagers through a phase whose token operand is a bf16 image (o-proj,
// unpooler, fused next-layer QKV): per unit, once its buffer is free and its
// K-slice is written (o-proj: its head groups merged; next-layer QKV: the
// tiles of x_out it covers), the leader bulk-copies the unit's K-slice of the
// image into it.  With two buffers this runs one unit ahead of
// the MMA.
MK_DEV bool stage_image_phase(const LayerParams& P, const Smem& S, int ph, uint32_t epoch, QCursor& q,
                              uint32_t (&b_ph)[2], uint32_t& ucount, uint32_t (&land_ph)[2]) {
  Misc* m = S.m;
  const int tid = threadIdx.x - kStagerBase;
  const uint8_t* img = bf_image(P, ph);
  int u;
  if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) return false;
  while (u >= 0) {
    const Unit U = make_unit(P, S, ph, u);
    const uint32_t b = ucount & 1;
    const uint64_t w0 = tnow(P);
    if (!group_mbar_wait(P, S, &m->bempty[b], b_ph[b] ^ 1, ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0))
      return false;
    const uint64_t w1 = tnow(P);
    if (ph == PH_O)
      for (int g = o_group_lo(P, U); g <= o_group_hi(P, U); ++g)
        if (!group_flag_wait(P, S, grp_ctr(P, 2, g), static_cast<uint32_t>(P.T * 4), tid == 0, kBarStage, 64, 0))
          return false;
    if (ph == PH_NQKV)
      for (int j = U.x0 / 128; j <= (U.x0 + U.nkb * 64 - 1) / 128; ++j)
        if (!group_flag_wait(P, S, P.xt_flag + j, epoch + 1u, tid == 0, kBarStage, 64, 0)) return false;
    if (tid == 0) {
      // the image was written by ordinary stores (of this and other CTAs),
      // released to this thread: order them before its async-proxy copy
      fence_proxy_async_global();
      const uint32_t bytes = static_cast<uint32_t>(U.nkb) * 2048u;
      uint64_t* lb = &m->land[b];
      m->land_out[b] = 1;
      mbar_arrive_expect_tx(lb, bytes);
      bulk_load(S.bbuf(b), img + static_cast<size_t>(U.x0 / 64) * 2048, bytes, lb, policy_evict_normal());
    }
    if (!group_mbar_wait(P, S, &m->land[b], land_ph[b], ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0)) return false;
    land_ph[b] ^= 1;
    if (tid == 0) {
      m->land_out[b] = 0;
      mbar_arrive(&m->bfull[b]);
      if (P.ts) {
        stamp_add(P, S, ph, 8, w1 - w0);
        stamp_add(P, S, ph, 9, globaltimer() - w1);
      }
    }
    b_ph[b] ^= 1;
    ++ucount;
    if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) return false;
  }
  return true;
}

// The stagers through one NVFP4 expert phase.  Each unit's operand is a copy
// of an image, skipped when the buffer already holds that image (every gate/up
// unit uses the p image; consecutive down units may share an expert).  A down
// unit waits for its own expert's image only.
MK_DEV bool stage_expert_phase(const LayerParams& P, const Smem& S, int ph, uint32_t epoch, QCursor& q,
                               uint32_t (&b_ph)[2], uint32_t& ucount, uint32_t (&land_ph)[2]) {
  Misc* m = S.m;
  const int tid = threadIdx.x - kStagerBase;
  const bool gu = ph == PH_GU;
  const int K = gu ? P.P : P.I;
  int holds[2] = {-1, -1};  // image in each operand buffer: -2 the p image, e expert e's
  if (gu && !group_grid_wait(P, S, BAR_PQ, grid_target(P, epoch), tid == 0, kBarStage, 64, 0)) return false;
  if (tid == 0) stamp(P, S, ph, 14);
  int u;
  if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) return false;
  while (u >= 0) {
    const Unit U = make_unit(P, S, ph, u);
    const uint32_t b = ucount & 1;
    const uint64_t w0 = tnow(P);
    // down: the expert's SwiGLU image (built by warp 7 of one CTA)
    if (!gu && holds[b] != U.expert &&
        !group_flag_wait(P, S, P.exp_sync + kMaxE + U.expert, epoch + 1u, tid == 0, kBarStage, 64, 0))
      return false;
    if (!group_mbar_wait(P, S, &m->bempty[b], b_ph[b] ^ 1, ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0))
      return false;
    const uint64_t w1 = tnow(P);
    const int key = gu ? -2 : U.expert;
    if (holds[b] != key) {
      if (tid == 0) {
        // the image was written by ordinary stores of other CTAs, released to
        // this one: order them before this thread's async-proxy copy
        fence_proxy_async_global();
        issue_image(P, S, gu ? P.pq_img : P.aq_img + static_cast<size_t>(U.expert) * image_bytes(K), K, b);
      }
      if (!group_mbar_wait(P, S, &m->land[b], land_ph[b], ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0))
        return false;
      land_ph[b] ^= 1;
      if (tid == 0) m->land_out[b] = 0;
      holds[b] = key;
    }
    if (tid == 0) {
      mbar_arrive(&m->bfull[b]);
      if (P.ts) {
        stamp_add(P, S, ph, 8, w1 - w0);
        stamp_add(P, S, ph, 9, globaltimer() - w1);
      }
    }
    b_ph[b] ^= 1;
    ++ucount;
    if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) return false;
  }
  return true;
}

// RMSNorm factors of x_in (first layer), by the stager and epilogue warps: one row per warp at a
// time, each lane's 16-byte loads of the row issued together.
MK_DEV void rnorm_x_in(const LayerParams& P, const Smem& S) {
  const int wid = threadIdx.x >> 5;
  const int w = wid >= kEpiBase / 32 ? wid - kEpiBase / 32 + 2 : wid - kStagerBase / 32;  // 0..5
  const int per_lane = P.H / 256;         // 16-byte chunks per lane (H % 256 == 0)
  for (int t = w; t < P.T; t += 6) {
    const uint4* x = reinterpret_cast<const uint4*>(P.x_in + static_cast<size_t>(t) * P.H) + lane_id();
    float s = 0.f;
    for (int c0 = 0; c0 < per_lane; c0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = c0 + c < per_lane ? x[(c0 + c) * 32] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t* pv = reinterpret_cast<const uint32_t*>(&v[c]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(pv[k] << 16), b = __uint_as_float(pv[k] & 0xFFFF0000u);
          s += a * a + b * b;
        }
      }
    }
    s = warp_sum(s);
    if (lane_id() == 0) S.m->rnorm[t] = 1.0f / sqrtf(s / P.H + P.eps);
  }
  named_bar(4, 192);
}

MK_DEV void run_stager(const LayerParams& P, const Smem& S, uint32_t epoch) {
  Misc* m = S.m;
  const int tid = threadIdx.x - kStagerBase;  // 0..63
  const int warp = tid >> 5;
  const uint32_t target = grid_target(P, epoch);
  uint32_t b_ph[2] = {0, 0}, ucount = 0, land_ph[2] = {0, 0};
  QCursor q;
  bool ok = true;
  if (P.first_layer) rnorm_x_in(P, S);
  for (int ph = 0; ph < PH_COUNT && ok; ++ph) {
    if (!phase_is_gemm(ph) || !phase_active(P, ph)) continue;
    if (ph == PH_GU) {
      // the router top-k, one token per CTA: CTA t < T selects token t's
      // experts with its first stager warp once the logits are complete; the
      // arrivals add up to grid (CTA 0 adds the CTAs without a token).  The p
      // image is quantised in shares by the other CTAs (by all when grid == T):
      // a top-k CTA without a share arrives at once.
      const int nsh = P.grid > P.T ? P.grid - P.T : P.grid;
      const int sharer = static_cast<int>(blockIdx.x) - (P.grid - nsh);
      if (static_cast<int>(blockIdx.x) < P.T) {
        if (sharer < 0 && tid == 0) red_release_add(P.bar_ctr + BAR_PQ, 1u);
        if (!group_flag_wait(P, S, P.misc_ctr + 3, epoch + 1u, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
        if (warp == 0) {
          if (tid == 0) stamp(P, S, PH_COUNT, 3);
          topk_token(P, blockIdx.x);
          __syncwarp();  // the lanes' writes precede lane 0's release
          if (tid == 0) {
            red_release_add(P.bar_ctr + BAR_ROUTE,
                            blockIdx.x == 0 ? 1u + static_cast<uint32_t>(P.grid - P.T) : 1u);
            stamp(P, S, PH_COUNT, 4);
          }
        }
      }
      // once p is complete, this CTA's share of the p image
      if (sharer >= 0) {
        if (!group_flag_wait(P, S, P.misc_ctr + 2, epoch + 1u, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
        if (tid == 0) stamp(P, S, PH_COUNT, 6);
        p_image_share(P, S, tid, sharer, nsh);
        stage_sync();
        if (tid == 0) {
          red_release_add(P.bar_ctr + BAR_PQ, 1u);
          stamp(P, S, PH_COUNT, 7);
        }
      }
      // the expert weights depend only on the routing: publish it to the
      // producer before waiting for the rest of the p image
      if (!group_grid_wait(P, S, BAR_ROUTE, target, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
      if (warp == 0) {
        build_routing(P, S);
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&m->route_ready);
      }
    }
    if (ph == PH_GU || (ph == PH_DOWN && P.moe)) {
      ok = stage_expert_phase(P, S, ph, epoch, q, b_ph, ucount, land_ph);
      continue;
    }
    const int dep = phase_dep(P, ph);
    if (dep >= 0) {
      if (!group_grid_wait(P, S, dep, target, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
    }
    if (tid == 0) stamp(P, S, ph, 14);
    // per-phase inputs of the token operand
    if (ph == PH_RP) {
      if (tid < P.T) {
        const float s = reduce_partials<false>(P.ssq_mid + tid, P.H / 128, kMaxT);
        m->rnorm[tid] = 1.0f / sqrtf(s / P.H + P.eps);
      }
    }
    stage_sync();
    // The leader copies a unit's first inputs ahead into the buffer's landing
    // area and records that it did (read by all after the next barrier).
    auto try_prefetch = [&](const Unit& V, int buf) {
      if (tid != 0) return;
      issue_bf16(P, S, ph, V, buf);
      m->pref_ok[buf] = 1;
    };
    // attention keeps its tiles in the operand buffers: the o-proj (which
    // waits per head group, not for the whole merge) starts once this CTA's
    // attention is done
    if (ph == PH_O &&
        !group_mbar_wait(P, S, &m->attn_free, 0, ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0)) {
      ok = false;
      break;
    }
    if (image_phase(ph)) {
      ok = stage_image_phase(P, S, ph, epoch, q, b_ph, ucount, land_ph);
      continue;
    }
    // the phase's first unit, its inputs copied at once; later units' are
    // copied one unit ahead when the producer has already claimed them
    int u;
    if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
    if (u >= 0) try_prefetch(make_unit(P, S, ph, u), ucount & 1);
    while (u >= 0 && ok) {
      const Unit U = make_unit(P, S, ph, u);
      const uint32_t b = ucount & 1;
      // the next unit's inputs go into the other buffer's landing area, which
      // the MMA never reads (its previous contents were consumed last unit)
      if (tid == 0) {
        m->pref_ok[b ^ 1] = 0;
        if (mbar_test_wait(&m->uq_full[q.slot], q.par)) {
          const int nu = *reinterpret_cast<volatile int*>(&m->uq[q.slot]);
          if (nu >= 0) try_prefetch(make_unit(P, S, ph, nu), b ^ 1);
        }
      }
      const uint64_t w0 = tnow(P);
      if (!group_mbar_wait(P, S, &m->bempty[b], b_ph[b] ^ 1, ERR_TIMEOUT_B, tid == 0, kBarStage, 64, 0)) {
        ok = false;
        break;
      }
      const bool pre = *reinterpret_cast<volatile int*>(&m->pref_ok[b]) != 0;
      const uint64_t w1 = tnow(P);
      const bool sok = stage_bf16(P, S, ph, U, b, pre, land_ph[b]);
      // both stager warps agree on the outcome before the next barrier
      if (lane_id() == 0) m->grp_ok[2 + warp] = sok ? 1 : 0;
      fence_proxy_async_smem();
      stage_sync();
      if (!(*reinterpret_cast<volatile int*>(&m->grp_ok[2]) && *reinterpret_cast<volatile int*>(&m->grp_ok[3]))) {
        ok = false;
        break;
      }
      if (tid == 0) {
        mbar_arrive(&m->bfull[b]);
        if (P.ts) {
          stamp_add(P, S, ph, 8, w1 - w0);
          stamp_add(P, S, ph, 9, globaltimer() - w1);
        }
      }
      b_ph[b] ^= 1;
      ++ucount;
      if (!queue_pop_group(P, S, q, u, tid == 0, kBarStage, 64, 0)) { ok = false; break; }
    }
  }
  // copies still in flight (only after an abort) must land before exit
  stage_sync();
  if (tid == 0) {
    for (int buf = 0; buf < 2; ++buf) {
      if (!m->land_out[buf]) continue;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait_sleep(&m->land[buf], land_ph[buf], 1000u)) {
        if (globaltimer() - t0 > P.timeout_ns) break;
      }
    }
  }
}

// ============================================================ epilogue (warps 8-11)
// Cross-warp reduction over the 128 epilogue threads of 16 per-token values
// (the tokens in `mask`): returns, in thread t (< 16, in mask), the sum (or
// max) for token t.
template <bool kMax>
MK_DEV float epi_reduce16_mask(const Smem& S, float (&v)[kMaxT], int et, uint32_t mask) {
  const int q = et >> 5;
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) {
    if ((mask >> t) & 1u) {
      float x = v[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, o);
        x = kMax ? fmaxf(x, y) : x + y;
      }
      if (lane_id() == 0) S.m->red[q][t] = x;
    }
  }
  epi_sync();
  float r = 0.f;
  if (et < kMaxT && ((mask >> et) & 1u)) {
    r = S.m->red[0][et];
    for (int w = 1; w < 4; ++w) r = kMax ? fmaxf(r, S.m->red[w][et]) : r + S.m->red[w][et];
  }
  epi_sync();
  return r;
}
// The same over all 16 tokens (values of tokens >= T are 0): a butterfly
// reduce-scatter inside each warp -- at each step a lane sends the half of
// its values that its partner keeps, 8 + 4 + 2 + 1 + 1 shuffles instead of
// 16 x 5 -- leaves token (lane >> 1) in lane pair (2t, 2t+1); then the four
// warps through shared memory.  Thread t (< 16) gets token t's result.
template <bool kMax>
MK_DEV float epi_reduce16(const Smem& S, float (&v)[kMaxT], int et) {
  const int lane = lane_id();
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a8[8], a4[4], a2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a8[i] = op(b4 ? v[i + 8] : v[i], __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 8], 16));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    a4[i] = op(b3 ? a8[i + 4] : a8[i], __shfl_xor_sync(0xffffffffu, b3 ? a8[i] : a8[i + 4], 8));
#pragma unroll
  for (int i = 0; i < 2; ++i)
    a2[i] = op(b2 ? a4[i + 2] : a4[i], __shfl_xor_sync(0xffffffffu, b2 ? a4[i] : a4[i + 2], 4));
  float a1 = op(b1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, b1 ? a2[0] : a2[1], 2));
  a1 = op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
  if ((lane & 1) == 0) S.m->red[et >> 5][lane >> 1] = a1;
  epi_sync();
  float r = 0.f;
  if (et < kMaxT) {
    r = S.m->red[0][et];
    for (int w = 1; w < 4; ++w) r = op(r, S.m->red[w][et]);
  }
  epi_sync();
  return r;
}

// 16-byte global -> shared copies (zero fill when !valid), completed in groups.
MK_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
MK_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MK_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The residual phases (o-proj, unpooler, dense down) add the layer input
// x_in (o-proj) or x_mid to their output.
MK_DEV bool residual_phase(int ph) { return ph == PH_O || ph == PH_UNPOOL || ph == PH_DOWN; }
// The phase whose final step writes x_out.
MK_DEV int x_out_phase(const LayerParams& P) { return P.moe ? PH_UNPOOL : PH_DOWN; }
MK_DEV const __nv_bfloat16* residual_src(const LayerParams& P, int ph) { return ph == PH_O ? P.x_in : P.xmid; }
// Asynchronous copy of a tile's residual rows (T rows of 128 columns from
// U.row0) into the epilogue's staging area: two 16-byte chunks per thread,
// rows >= T zero.  Issued by the last unit of a split-K tile before it reads
// the partials, so that both round trips overlap; epi_bf16_final waits.
MK_DEV void stage_residual(const LayerParams& P, const Smem& S, int ph, const Unit& U, int et) {
  const __nv_bfloat16* res = residual_src(P, ph);
  for (int c = et; c < kMaxT * 16; c += 128) {
    const int t = c >> 4, col = U.row0 + (c & 15) * 8;
    const bool valid = t < P.T && col < U.N;
    cp_async16(smem_u32(S.res() + c * 16), res + (valid ? static_cast<size_t>(t) * P.H + col : 0), valid);
  }
  cp_async_commit();
}

// Final values of one 128-row tile of a bf16 phase: acc[j][t] for the row
// (feature) f of this thread.
// `staged`: the residual rows are in flight to the staging area
// (stage_residual), else they are loaded here.
MK_DEV void epi_bf16_final(const LayerParams& P, const Smem& S, int ph, const Unit& U, int et,
                           float (&g)[kMaxT], float (&u)[kMaxT], bool staged) {
  const int f = U.row0 + et;
  const bool valid = f < U.N;
  switch (ph) {
    case PH_QKV:
    case PH_NQKV: {
      if (!valid) break;
      __nv_bfloat16* qdst = ph == PH_QKV ? P.q_buf : P.q_out;
      __nv_bfloat16* kc = ph == PH_QKV ? P.k_cache : P.nk_cache;
      __nv_bfloat16* vc = ph == PH_QKV ? P.v_cache : P.nv_cache;
      const int nq = P.Hq * P.d, nk = P.Hkv * P.d;
      for (int t = 0; t < P.T; ++t) {
        const __nv_bfloat16 v = to_bf(ph == PH_NQKV ? g[t] * S.m->rnorm_ep[t] : g[t]);
        if (f < nq) qdst[static_cast<size_t>(t) * nq + f] = v;
        else if (f < nq + nk) kc[static_cast<size_t>(P.ctx + t) * nk + (f - nq)] = v;
        else vc[static_cast<size_t>(P.ctx + t) * nk + (f - nq - nk)] = v;
      }
      break;
    }
    case PH_O:
    case PH_UNPOOL:
    case PH_DOWN: {  // residual: x = bf16(res + acc); sum-of-squares partial
      __nv_bfloat16* dst = ph == PH_O ? P.xmid : P.x_out;
      // the phase that writes x_out also writes the fused next-layer QKV's
      // operand image, bf16(x_out * gain)
      const bool xn = P.fuse_next && ph == x_out_phase(P);
      const float gn = xn && valid ? __bfloat162float(P.next_attn_norm_w[f]) : 0.f;
      // every residual load is issued before the first store: a load may not
      // move past a store that could alias it, so interleaving them would cost
      // one memory round trip per token
      float rv[kMaxT];
      if (staged) {
        cp_async_wait<0>();
        epi_sync();  // every thread's chunks have landed
#pragma unroll
        for (int t = 0; t < kMaxT; ++t)
          rv[t] = valid ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(S.res() + t * 256)[et]) : 0.f;
      } else {
        const __nv_bfloat16* res = residual_src(P, ph);
#pragma unroll
        for (int t = 0; t < kMaxT; ++t)
          rv[t] = (valid && t < P.T) ? ld_bf(res + static_cast<size_t>(t) * P.H + f) : 0.f;
      }
      float sq[kMaxT];
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        sq[t] = 0.f;
        if (valid && t < P.T) {
          const float x = round_bf(rv[t] + g[t]);
          dst[static_cast<size_t>(t) * P.H + f] = to_bf(x);
          if (xn) *reinterpret_cast<__nv_bfloat16*>(P.xn_img + bf_image_off(t, f)) = to_bf(x * gn);
          sq[t] = x * x;
        }
      }
      const float r = epi_reduce16<false>(S, sq, et);
      if (et < P.T) (ph == PH_O ? P.ssq_mid : P.ssq_out)[U.tile * kMaxT + et] = r;
      break;
    }
    case PH_RP: {
      if (!P.moe) {  // dense SwiGLU
        if (valid)
          for (int t = 0; t < P.T; ++t)
            P.a_buf[static_cast<size_t>(t) * P.F + f] = to_bf(silu(g[t]) * u[t]);
        break;
      }
      if (U.router) {
        if (valid)
          for (int t = 0; t < P.T; ++t) P.logits[static_cast<size_t>(t) * kMaxE + f] = g[t];
      } else {
        float am[kMaxT];
#pragma unroll
        for (int t = 0; t < kMaxT; ++t) {
          am[t] = 0.f;
          if (valid && t < P.T) {
            const float x = round_bf(g[t]);
            P.p_buf[static_cast<size_t>(t) * P.P + f] = to_bf(x);
            am[t] = fabsf(x);
          }
        }
        const float r = epi_reduce16<true>(S, am, et);
        if (et < P.T) P.pamax[U.tile * kMaxT + et] = r;
      }
      break;
    }
  }
}

// Epilogue of one GEMM unit.
MK_DEV bool epi_gemm_unit(const LayerParams& P, const Smem& S, int ph, const Unit& U,
                          uint32_t b, uint32_t& acc_ph_b, int et) {
  Misc* m = S.m;
  const uint64_t w0 = tnow(P);
  if (!group_mbar_wait(P, S, &m->accfull[b], acc_ph_b, ERR_TIMEOUT_ACC, et == 0, kBarEpi, 128, 1))
    return false;
  if (P.ts && et == 0) stamp_add(P, S, ph, 10, globaltimer() - w0);
  acc_ph_b ^= 1;
  tc_fence_after();
  const int q = et >> 5;
  const uint32_t taddr = m->tmem_base + (static_cast<uint32_t>(32 * q) << 16) + 128 * b;
  float g[kMaxT], u[kMaxT];
  // the four MMA lanes' partial sums (K-steps 0..3 of every K-block)
  // the four MMA warps' partial sums (K-steps 0..3 of every K-block): all
  // loads issued, one wait
  auto load_sum = [&](uint32_t col, float (&acc)[kMaxT]) {
    uint32_t r[4][16];
#pragma unroll
    for (int l = 0; l < 4; ++l) tmem_ld16_nowait(col + 16 * l, r[l]);
    tmem_ld_wait();
#pragma unroll
    for (int t = 0; t < kMaxT; ++t)
      acc[t] = (__uint_as_float(r[0][t]) + __uint_as_float(r[1][t])) +
               (__uint_as_float(r[2][t]) + __uint_as_float(r[3][t]));
  };
  load_sum(taddr, g);
  if (U.pair == 2) load_sum(taddr + 64, u);
  tc_fence_before();
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(&m->accempty[b]);

  if (U.fp4) {
    const int e = U.expert;
    const int n = m->off[e + 1] - m->off[e];
    const int f = U.tile * 128 + et;
    if (ph == PH_GU) {
      // Accumulator column t is token t (the p image holds every token).  The
      // expert's slots, ascending, name its tokens in ascending order.
      const float tg = S.tsc(0)[e], tu = S.tsc(1)[e];
      const int* sl = m->slots + m->off[e];
      float am[kMaxT];
      uint32_t tmask = 0;
      int j = 0, sj = n > 0 ? sl[0] : 0;
      int tj = n > 0 ? sj / P.topk : -1;
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        am[t] = 0.f;
        if (tj == t) {
          const float sr = m->srow_ep[t];
          const float gv = g[t] * sr * tg, uv = u[t] * sr * tu;
          const float a = round_bf(silu(gv) * uv);
          P.a_buf[static_cast<size_t>(sj) * P.I + f] = to_bf(a);
          am[t] = fabsf(a);
          tmask |= 1u << t;
          if (++j < n) {
            sj = sl[j];
            tj = sj / P.topk;
          } else {
            tj = -1;
          }
        }
      }
      const float r = epi_reduce16_mask<true>(S, am, et, tmask);
      if (et < kMaxT && ((tmask >> et) & 1u))
        P.aamax[sl[__popc(tmask & ((1u << et) - 1u))] * (P.I / 128) + U.tile] = r;
      // this gate/up tile of the expert is written: count it in (no reply
      // waited for; warp 7 of one CTA builds the expert's image once all of
      // its tiles are in)
      epi_sync();
      if (et == 0) red_release_add(P.exp_sync + e, 1u);
    } else {
      // accumulator column i is the expert's i-th slot; the pair's second
      // tile holds the next 128 features
      const float td = S.tsc(2)[e];
      for (int i = 0; i < n; ++i) {
        const int s = m->slots[m->off[e] + i];
        const float sr = m->srow_ep[s];
        P.z_buf[static_cast<size_t>(s) * P.P + f] = to_bf(g[i] * sr * td);
        if (U.pair == 2) P.z_buf[static_cast<size_t>(s) * P.P + f + 128] = to_bf(u[i] * sr * td);
      }
      if (et < n) {
        const int t = m->slots[m->off[e] + et] / P.topk;
        atomicAdd(&m->comb_local[t][U.tile], 1u);
        if (U.pair == 2) atomicAdd(&m->comb_local[t][U.tile + 1], 1u);
      }
    }
    return true;
  }

  // bf16 phase: split-K partials + fix-up by the last arriving unit of a tile
  bool staged = false;
  if (U.ksplit > 1) {
    // the o-proj overlaps the QKV phase (per head group) and the fused
    // next-layer QKV the fix-ups of the phase before it, so each has its own
    float* part = ph == PH_O ? P.part_o : ph == PH_NQKV ? P.part_n : P.part;
    // partials: part[ks][j][col][16 tokens], col = col_tile * 128 + row in
    // tile: each thread moves its 16 token values as four 16-byte vectors
    const size_t ncol = static_cast<size_t>(U.col_tiles) * 128;
    const int col = U.col_tile * 128 + et;
    for (int j = 0; j < U.pair; ++j) {
      float4* dst = reinterpret_cast<float4*>(part + ((static_cast<size_t>(U.ks * U.pair + j)) * ncol + col) * kMaxT);
      const float* v = j ? u : g;
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    epi_sync();
    if (et == 0) {
      uint32_t* c = P.fix_ctr + ph * 256 + U.col_tile;
      const uint32_t old = atom_add_acq_rel(c, 1u);
      const bool last = old == static_cast<uint32_t>(U.ksplit - 1);
      if (last) *c = 0;  // this launch's arrivals are all in
      m->flag = last;
    }
    epi_sync();
    if (!m->flag) return true;
    // the last unit of the tile: its residual loads go out with the first
    // partials' loads
    if (residual_phase(ph)) {
      stage_residual(P, S, ph, U, et);
      staged = true;
    }
    for (int j = 0; j < U.pair; ++j) {
      float acc[kMaxT];
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) acc[t] = 0.f;
      // the partials are summed in split order, kFixBatch splits' loads at a
      // time (more would not fit in registers)
      constexpr int kFixBatch = 4;
      for (int ks = 0; ks < U.ksplit; ks += kFixBatch) {
        float4 v[kFixBatch][4];
#pragma unroll
        for (int kk = 0; kk < kFixBatch; ++kk) {
          if (ks + kk < U.ksplit) {
            const float4* src = reinterpret_cast<const float4*>(
                part + ((static_cast<size_t>((ks + kk) * U.pair + j)) * ncol + col) * kMaxT);
#pragma unroll
            for (int q = 0; q < 4; ++q) v[kk][q] = __ldcg(src + q);
          }
        }
#pragma unroll
        for (int kk = 0; kk < kFixBatch; ++kk) {
          if (ks + kk < U.ksplit) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[4 * q] += v[kk][q].x;
              acc[4 * q + 1] += v[kk][q].y;
              acc[4 * q + 2] += v[kk][q].z;
              acc[4 * q + 3] += v[kk][q].w;
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) (j ? u : g)[t] = acc[t];
    }
  }
  if (ph == PH_NQKV && !m->rn_ready) {
    // The next-layer QKV ran on bf16(x_out * gain): its RMS factors, once
    // per launch, when every tile of x_out (and its sum-of-squares partial)
    // is in.
    if (!group_grid_wait(P, S, BAR_X, grid_target(P, m->epoch), et == 0, kBarEpi, 128, 1)) return false;
    if (et < P.T)
      m->rnorm_ep[et] = 1.0f / sqrtf(reduce_partials<false>(P.ssq_out + et, P.H / 128, kMaxT) / P.H + P.eps);
    if (et == 0) m->rn_ready = 1;
    epi_sync();
  }
  epi_bf16_final(P, S, ph, U, et, g, u, staged);
  if (P.fuse_next && ph == x_out_phase(P)) {
    // this tile of x_out, its image columns and its sum-of-squares partial
    // are final: the next-layer QKV units of its K-slices may start
    epi_sync();
    if (et == 0) st_release(P.xt_flag + U.tile, m->epoch + 1u);
  }
  if (ph == PH_QKV) {
    // this tile's q, k and v rows are final: count it in for its groups (a
    // counter that grows by grp_tiles per launch; no reply is waited for)
    epi_sync();
    if (et == 0) {
      for (int gg = 0; gg < P.Hkv; ++gg)
        if (tile_in_group(P, U.tile, gg)) red_release_add(grp_ctr(P, 0, gg), 1u);
    }
  }
  if (ph == PH_RP && P.moe && !U.router) {
    // the last finished pooler tile announces that p and its amax partials
    // are complete (every CTA then quantises a share of the p image)
    epi_sync();
    if (et == 0) {
      const uint32_t old = atom_add_acq_rel(P.misc_ctr + 1, 1u);
      if (old == static_cast<uint32_t>(P.tiles_pool - 1)) {
        P.misc_ctr[1] = 0;  // this launch's arrivals are all in
        st_release(P.misc_ctr + 2, m->epoch + 1u);
      }
    }
  }
  if (ph == PH_RP && P.moe && U.router) {
    // the last finished router tile announces that the logits are complete
    // (the first T CTAs then select one token's experts each)
    epi_sync();
    if (et == 0) {
      const uint32_t old = atom_add_acq_rel(P.misc_ctr, 1u);
      if (old == static_cast<uint32_t>(P.tiles_router - 1)) {
        *P.misc_ctr = 0;  // this launch's arrivals are all in
        st_release(P.misc_ctr + 3, m->epoch + 1u);
        stamp(P, S, PH_COUNT, 5);
      }
    }
  }
  return true;
}

// ------------------------------------------------------------ attention (epilogue warps 8-11)
MK_DEV void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
MK_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MK_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
MK_DEV uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Row r, 16-byte chunk c of a [64][D] bf16 tile: chunks XOR-swizzled by r % 8.
template <int D>
MK_DEV uint32_t tile_off(int r, int c) {
  return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// One unit: KV head g, positions [lo, hi).  Each warp owns q head 4g + w and
// the T tokens (16 rows); flash-style online softmax in the log2 domain.
// kTree: the verify tokens form a token tree (visibility from tree_vis /
// tree_depth) instead of the causal chain (a separate instance, so that the
// chain's innermost loop keeps its registers).
template <int D, bool kTree>
MK_DEV void attention_unit(const LayerParams& P, const Smem& S, int g, int lo, int hi, int chunk_id,
                           int et) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  // Q and the double-buffered K/V tiles live in the two operand buffers (80 KB):
  // the stagers stay out of them until the epilogue arrives on attn_free
  uint8_t* sQ = S.bbuf(0);
  uint8_t* sK[2] = {sQ + 64 * D * 2, sQ + 64 * D * 2 + 2 * 64 * D * 2};
  uint8_t* sV[2] = {sK[0] + 64 * D * 2, sK[1] + 64 * D * 2};
  const int w = et >> 5, lane = lane_id();
  const int Hkv = P.Hkv;
  const size_t kv_row = static_cast<size_t>(Hkv) * D;  // elements per position
  const __nv_bfloat16* qsrc = P.first_layer ? P.q_buf : P.q_in;
  const int qld = P.Hq * D;

  // Q tile: row = w*16 + t (q head 4g+w, token t); rows t >= T read as zero
  for (int i = et; i < 64 * kChunks; i += 128) {
    const int r = i / kChunks, c = i % kChunks;
    const int hl = r >> 4, t = r & 15;
    const bool valid = t < P.T;
    const __nv_bfloat16* src = qsrc + static_cast<size_t>(valid ? t : 0) * qld + (4 * g + hl) * D + c * 8;
    cp_async16(smem_u32(sQ + tile_off<D>(r, c)), src, valid);
  }
  cp_async_commit();
  auto load_kv = [&](int buf, int p0) {
    for (int i = et; i < 64 * kChunks; i += 128) {
      const int r = i / kChunks, c = i % kChunks;
      const int pos = p0 + r;
      const bool valid = pos < hi;
      const size_t off = static_cast<size_t>(valid ? pos : lo) * kv_row + g * D + c * 8;
      cp_async16(smem_u32(sK[buf] + tile_off<D>(r, c)), P.k_cache + off, valid);
      cp_async16(smem_u32(sV[buf] + tile_off<D>(r, c)), P.v_cache + off, valid);
    }
    cp_async_commit();
  };
  load_kv(0, lo);
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  const int r0 = lane >> 2;            // rows r0 and r0 + 8 of this warp = tokens
  // each token's sequence position (prefix window) and, in a tree, its
  // visible verify tokens
  const int posq[2] = {P.ctx + (kTree ? P.tree_depth[r0] : r0), P.ctx + (kTree ? P.tree_depth[r0 + 8] : r0 + 8)};
  uint32_t vism[2] = {0u, 0u};
  if (kTree) {
    vism[0] = P.tree_vis[r0];
    vism[1] = P.tree_vis[r0 + 8];
  }

  const int ntiles = (hi - lo + 63) / 64;
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    const int p0 = lo + it * 64;
    if (it + 1 < ntiles) {
      load_kv(buf ^ 1, p0 + 64);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    epi_sync();
    // the 64-position tile in two halves of 32 (keeps the score fragment small)
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int q0 = p0 + 32 * half;
      if (q0 >= hi) break;
      // S = Q K^T (16 x 32)
      float s[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t qa[4];  // Q fragment of this warp (rows w*16 .. w*16+15), K-step ks
        {
          const int r = w * 16 + (lane & 15);
          const int c = ks * 2 + (lane >> 4);
          ldsm_x4(smem_u32(sQ + tile_off<D>(r, c)), qa[0], qa[1], qa[2], qa[3]);
        }
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // pairs of 8-position tiles
          const int r = 32 * half + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int c = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(sK[buf] + tile_off<D>(r, c)), b0, b1, b2, b3);
          mma16816(s[2 * np], qa, b0, b1);
          mma16816(s[2 * np + 1], qa, b2, b3);
        }
      }
      // mask + online softmax (log2 domain)
      float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = q0 + nt * 8 + 2 * (lane & 3) + (e & 1);
          const int rr = e >> 1;
          // chain: key j visible iff j <= the token's position, within the
          // window; tree: prefix keys by the window from the token's
          // position, verify tokens by the visibility mask
          const int pq = posq[rr];
          const bool vis =
              kTree ? j < hi && (j < P.ctx ? (P.window == 0 || pq - j < P.window)
                                           : ((vism[rr] >> (j - P.ctx)) & 1u) != 0)
                    : j < hi && j <= pq && (P.window == 0 || pq - j < P.window);
          const float v = vis ? s[nt][e] * sl2 : -INFINITY;
          s[nt][e] = v;
          mx[rr] = fmaxf(mx[rr], v);
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
        mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
      }
      float alpha[2], base[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        base[rr] = mx[rr] == -INFINITY ? 0.f : mx[rr];
        alpha[rr] = mrow[rr] == -INFINITY ? 0.f : exp2f(mrow[rr] - base[rr]);
        if (mx[rr] == -INFINITY) alpha[rr] = 1.f;
        mrow[rr] = mx[rr];
        lrow[rr] *= alpha[rr];
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      // P V over 2 K-steps of 16 positions.  P (as A fragments) is split into
      // a bf16 high part and the bf16 rounding of the remainder, so that P V
      // is accumulated from a ~16-bit-mantissa P rather than bf16's 8 bits.
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4], pl[4];
#pragma unroll
        for (int hi8 = 0; hi8 < 2; ++hi8) {
          const int nt = 2 * kk + hi8;
          const float p0v = exp2f(s[nt][0] - base[0]), p1v = exp2f(s[nt][1] - base[0]);
          const float p2v = exp2f(s[nt][2] - base[1]), p3v = exp2f(s[nt][3] - base[1]);
          lrow[0] += p0v + p1v;
          lrow[1] += p2v + p3v;
          const float h0 = round_bf(p0v), h1 = round_bf(p1v), h2 = round_bf(p2v), h3 = round_bf(p3v);
          pa[hi8 * 2 + 0] = pack_bf16(h0, h1);
          pa[hi8 * 2 + 1] = pack_bf16(h2, h3);
          pl[hi8 * 2 + 0] = pack_bf16(p0v - h0, p1v - h1);
          pl[hi8 * 2 + 1] = pack_bf16(p2v - h2, p3v - h3);
        }
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {  // pairs of 8-wide d tiles
          const int r = 32 * half + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int c = dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(sV[buf] + tile_off<D>(r, c)), b0, b1, b2, b3);
          mma16816(o[2 * dp], pa, b0, b1);
          mma16816(o[2 * dp + 1], pa, b2, b3);
          mma16816(o[2 * dp], pl, b0, b1);
          mma16816(o[2 * dp + 1], pl, b2, b3);
        }
      }
    }
    epi_sync();
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 1);
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 2);
  }
  // partial: [unit][row][D + 2] = o (unnormalised), m, l
  float* dst = P.attn_part + static_cast<size_t>(g * P.attn_chunks + chunk_id) * 64 * (D + 2);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = w * 16 + r0 + 8 * rr;
    float* pr = dst + static_cast<size_t>(row) * (D + 2);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int col = i * 8 + 2 * (lane & 3);
      *reinterpret_cast<float2*>(pr + col) = make_float2(o[i][2 * rr], o[i][2 * rr + 1]);
    }
    if ((lane & 3) == 0) {
      pr[D] = mrow[rr];
      pr[D + 1] = lrow[rr];
    }
  }
}

// Merge of the attention partials of one (token, q head) by one warp:
// o = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c over the chunks c, summed
// in chunk order.  The loads go out in batches (the chunk statistics one chunk
// per lane, the o partials 16 chunks at a time, the first batch together with
// the statistics), so that a merge costs a few L2 round trips, not one per
// four chunks.
template <int D>
MK_DEV void merge_item(const LayerParams& P, int item) {
  constexpr int V = D / 32;  // output elements per lane
  constexpr int kB = 16;     // chunks whose o partials are loaded together (divides 32)
  const int lane = lane_id();
  const int t = item / P.Hq, hq = item % P.Hq;
  const int g = hq / 4, hl = hq % 4;
  const int row = hl * 16 + t;
  const size_t stride = static_cast<size_t>(64) * (D + 2);
  const float* base = P.attn_part + static_cast<size_t>(g * P.attn_chunks) * stride +
                      static_cast<size_t>(row) * (D + 2);
  const int C = P.attn_chunks;
  // chunk statistics of the first 32 chunks (lane j: chunk j) and the first
  // batch of o partials go out together; then the maximum over all chunks
  float mc = -INFINITY, lc = 0.f;
  if (lane < C) {
    mc = __ldcg(base + lane * stride + D);
    lc = __ldcg(base + lane * stride + D + 1);
  }
  float ov[kB][V];
#pragma unroll
  for (int j = 0; j < kB; ++j)
#pragma unroll
    for (int v = 0; v < V; ++v) ov[j][v] = j < C ? __ldcg(base + j * stride + lane * V + v) : 0.f;
  float M = mc;
  for (int c = lane + 32; c < C; c += 32) M = fmaxf(M, __ldcg(base + c * stride + D));
  M = warp_max(M);
  float wl = mc == -INFINITY ? 0.f : exp2f(mc - M);
  float acc[V], L = 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int c0 = 0; c0 < C; c0 += kB) {
    if (c0 > 0) {
      if ((c0 & 31) == 0) {  // the next group of 32 chunks' statistics
        mc = -INFINITY;
        lc = 0.f;
        if (c0 + lane < C) {
          mc = __ldcg(base + (c0 + lane) * stride + D);
          lc = __ldcg(base + (c0 + lane) * stride + D + 1);
        }
        wl = mc == -INFINITY ? 0.f : exp2f(mc - M);
      }
#pragma unroll
      for (int j = 0; j < kB; ++j)
#pragma unroll
        for (int v = 0; v < V; ++v)
          ov[j][v] = c0 + j < C ? __ldcg(base + (c0 + j) * stride + lane * V + v) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      if (c0 + j < C) {  // the same for every lane
        const float wgt = __shfl_sync(0xffffffffu, wl, (c0 + j) & 31);
        L += wgt * __shfl_sync(0xffffffffu, lc, (c0 + j) & 31);
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] += wgt * ov[j][v];
      }
    }
  }
  // this lane's V outputs lie in one 16-byte chunk of the o-proj input image
  uint32_t w[V / 2];
#pragma unroll
  for (int v = 0; v < V / 2; ++v) w[v] = pack_bf16(acc[2 * v] / L, acc[2 * v + 1] / L);
  uint8_t* out = reinterpret_cast<uint8_t*>(P.o_buf) + bf_image_off(t, hq * D + lane * V);
  if constexpr (V == 4) *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
  else *reinterpret_cast<uint32_t*>(out) = w[0];
}

// End of the expert-down phase: publish this CTA's z contributions per
// (token, output tile) with one release, and combine every (token, tile) whose
// k contributions are now all written: y = bf16(sum_r w[t][r] z[t*k + r]),
// summed in rank order (page "Muse Spark Open ...", section "What the 5.9 ms
// is still spent on": the combine).
MK_DEV void combine_phase_end(const LayerParams& P, const Smem& S, int et) {
  Misc* m = S.m;
  const int tiles = P.P / 128;
  if (et == 0) m->n_done = 0;
  epi_sync();  // every thread's z writes precede the arrivals below
  for (int i = et; i < P.T * tiles; i += 128) {
    const int t = i / tiles, j = i % tiles;
    const uint32_t c = m->comb_local[t][j];
    if (c == 0) continue;
    uint32_t* ctr = P.comb_ctr + t * tiles + j;
    // releases this CTA's z rows, acquires the other contributors'
    const uint32_t old = atom_add_acq_rel(ctr, c);
    if (old + c == static_cast<uint32_t>(P.topk)) {
      *ctr = 0;
      m->done_pairs[atomicAdd(&m->n_done, 1)] = i;
    }
  }
  epi_sync();
  // 16 threads per completed (token, tile) pair, 8 features each with 16-byte
  // loads: 8 pairs at a time; each feature sums its k terms in rank order
  const int nd = m->n_done;
  for (int d0 = 0; d0 < nd; d0 += 8) {
    const int d = d0 + (et >> 4);
    if (d >= nd) continue;
    const int i = m->done_pairs[d];
    const int t = i / tiles, f0 = (i % tiles) * 128 + (et & 15) * 8;
    uint4 z[kMaxK];
    float wr[kMaxK];
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
      if (r < P.topk) {
        z[r] = __ldcg(reinterpret_cast<const uint4*>(P.z_buf + static_cast<size_t>(t * P.topk + r) * P.P + f0));
        wr[r] = __ldcg(P.wts + t * P.topk + r);
      }
    }
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
      if (r < P.topk) {
        const uint32_t* zw = reinterpret_cast<const uint32_t*>(&z[r]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] += wr[r] * __uint_as_float(zw[j] << 16);
          acc[2 * j + 1] += wr[r] * __uint_as_float(zw[j] & 0xFFFF0000u);
        }
      }
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      ow[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(P.y_buf) + bf_image_off(t, f0)) = o;
  }
}

MK_DEV bool epi_arrive(const LayerParams& P, const Smem& S, int id, int et) {
  epi_sync();
  if (et == 0) red_release_add(P.bar_ctr + id, 1u);  // releases the group's writes
  return true;
}

MK_DEV bool epi_wait(const LayerParams& P, const Smem& S, int id, uint32_t target, int et) {
  return group_grid_wait(P, S, id, target, et == 0, kBarEpi, 128, 1);
}

MK_DEV void run_epilogue(const LayerParams& P, const Smem& S, uint32_t epoch) {
  Misc* m = S.m;
  const int et = threadIdx.x - kEpiBase;  // 0..127
  const uint32_t target = grid_target(P, epoch);
  uint32_t acc_ph[2] = {0, 0}, ucount = 0;
  QCursor qe;
  bool ok = true;
  if (P.first_layer) rnorm_x_in(P, S);
  const int last_ph = P.fuse_next ? PH_NQKV : (P.moe ? PH_UNPOOL : PH_DOWN);
  for (int ph = 0; ph < PH_COUNT && ok; ++ph) {
    if (!phase_active(P, ph)) continue;
    if (ph == last_ph && et == 0) pdl_launch_dependents();
    if (et == 0) stamp(P, S, ph, 0);
    if (ph == PH_ATTN) {
      // a chunk of KV head g waits only for g's q, k and v rows
      const int n = phase_units(P, S, ph);
      for (int u = first_unit(P, ph); u < n && ok; u += P.grid) {
        const int g = u / P.attn_chunks, c = u % P.attn_chunks;
        if (P.first_layer &&
            !(ok = group_flag_wait(P, S, grp_ctr(P, 0, g), (epoch + 1u) * P.grp_tiles[g], et == 0, kBarEpi,
                                   128, 1)))
          break;
        const int lo = P.attn_lo + c * P.attn_chunk_len;
        const int hi = min(P.ctx + P.T, lo + P.attn_chunk_len);
        if (P.d == 128) {
          if (P.tree) attention_unit<128, true>(P, S, g, lo, hi, c, et);
          else attention_unit<128, false>(P, S, g, lo, hi, c, et);
        } else {
          if (P.tree) attention_unit<64, true>(P, S, g, lo, hi, c, et);
          else attention_unit<64, false>(P, S, g, lo, hi, c, et);
        }
        epi_sync();
        if (et == 0) red_release_add(grp_ctr(P, 1, g), 1u);  // no reply waited for
      }
      if (!ok) break;
      if (et == 0) {
        stamp(P, S, ph, 1);
        mbar_arrive(&m->attn_free);  // the o-proj stagers may now use the operand buffers
      }
      epi_arrive(P, S, BAR_ATTN, et);
      continue;
    }
    if (ph == PH_MERGE) {
      // an item (token, q head) waits only for its group's chunks
      const int n = phase_units(P, S, ph);
      const int w = et >> 5;
      int k = 0;
      bool wok = true;
      for (int u = first_unit(P, ph); u < n && wok; u += P.grid, ++k) {
        if ((k & 3) != w) continue;  // the CTA's k-th item goes to warp k % 4
        const int g = (u % P.Hq) / 4;
        int r = 1;
        if (lane_id() == 0)
          r = flag_wait(P, S, grp_ctr(P, 1, g), static_cast<uint32_t>(P.attn_chunks), ERR_TIMEOUT_DATA) ? 1 : 0;
        if (!(wok = __shfl_sync(0xffffffffu, r, 0) != 0)) break;
        __syncwarp();  // the lanes' loads below follow lane 0's acquire
        if (P.d == 128) merge_item<128>(P, u);
        else merge_item<64>(P, u);
        __syncwarp();
        if (lane_id() == 0) red_release_add(grp_ctr(P, 2, g), 1u);  // no reply waited for
      }
      // the epilogue warps agree on the outcome before their next barrier
      if (lane_id() == 0) m->red[0][w] = wok ? 1.f : 0.f;
      epi_sync();
      ok = m->red[0][0] != 0.f && m->red[0][1] != 0.f && m->red[0][2] != 0.f && m->red[0][3] != 0.f;
      epi_sync();
      if (!ok) break;
      if (et == 0) stamp(P, S, ph, 1);
      epi_arrive(P, S, BAR_MERGE, et);
      continue;
    }
    // GEMM phases: inputs the epilogue itself reads
    if (ph == PH_GU) {
      if (!(ok = group_mbar_wait(P, S, &m->route_ready, 0, ERR_TIMEOUT_ROUTE, et == 0, kBarEpi, 128, 1)))
        break;
      // p complete: its row scales from the amax partials
      if (!(ok = group_flag_wait(P, S, P.misc_ctr + 2, epoch + 1u, et == 0, kBarEpi, 128, 1))) break;
      if (et < P.T) m->srow_ep[et] = p_row_scale(P, et);
      // the active experts' tensor scales, read from shared memory by every
      // expert unit of the launch (one L2 round trip here, none per unit)
      for (int i = et; i < m->n_act; i += 128) {
        const int e = m->act[i];
        S.tsc(0)[e] = __ldg(P.ts_gate + e);
        S.tsc(1)[e] = __ldg(P.ts_up + e);
        S.tsc(2)[e] = __ldg(P.ts_down + e);
      }
      epi_sync();
    } else if (ph == PH_DOWN && P.moe) {
      for (int i = et; i < kMaxT * 16; i += 128) (&m->comb_local[0][0])[i] = 0;
      epi_sync();
    }
    if (et == 0) stamp(P, S, ph, 15);
    while (ok) {
      int u;
      if (!queue_pop_group(P, S, qe, u, et == 0, kBarEpi, 128, 1)) { ok = false; break; }
      if (u < 0) break;
      const Unit U = make_unit(P, S, ph, u);
      const uint32_t b = ucount & 1;
      const uint64_t w0 = tnow(P);
      if (ph == PH_DOWN && P.moe) {
        if (!(ok = group_flag_wait(P, S, P.exp_sync + kMaxE + U.expert, epoch + 1u, et == 0, kBarEpi, 128, 1)))
          break;
        const int e = U.expert;
        if (et < m->off[e + 1] - m->off[e]) {
          const int s = m->slots[m->off[e] + et];
          m->srow_ep[s] = __ldcg(P.srow_a + s);
        }
        epi_sync();
      }
      ok = epi_gemm_unit(P, S, ph, U, b, acc_ph[b], et);
      if (P.ts && et == 0) stamp_add(P, S, ph, 11, globaltimer() - w0);
      ++ucount;
    }
    if (!ok) break;
    if (ph == PH_DOWN && P.moe) combine_phase_end(P, S, et);
    if (et == 0) stamp(P, S, ph, 1);
    epi_arrive(P, S, phase_arrive(P, ph), et);
  }
  // CTA 0 advances the epoch once every CTA has finished this launch.
  if (ok && blockIdx.x == 0) {
    if (epi_wait(P, S, final_barrier(P), target, et)) {
      // every CTA has claimed its last unit and counted in its last gate/up
      // tile: the claim and per-expert counters start the next launch at zero
      if (P.moe)
        for (int i = et; i < P.E; i += 128) P.exp_sync[i] = 0;
      // and the per-group attention-chunk and merge-item counters
      for (int i = et; i < 2 * kMaxGroups; i += 128) grp_ctr(P, 1, 0)[i] = 0;
      epi_sync();
      if (et == 0) {
        for (int i = 0; i < PH_COUNT; ++i) P.sched[i] = 0;
        __threadfence();
        *P.epoch = epoch + 1u;
      }
    }
  }
}

// ============================================================ kernel
__global__ void __launch_bounds__(kThreads, 1) mk_layer_kernel(const __grid_constant__ LayerParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem S;
  S.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  S.m = reinterpret_cast<Misc*>(S.base + kOffMisc);
  S.ts = reinterpret_cast<uint64_t*>(S.base + kOffTs);
  const int warp = threadIdx.x >> 5;
  Misc* m = S.m;
  const uint64_t t_start = P.ts ? globaltimer() : 0;
  if (P.ts)
    for (int i = threadIdx.x; i < kTsPerCta; i += kThreads) S.ts[i] = 0;

  if (threadIdx.x == 0) {
    // barriers completed by tcgen05.commit count the four MMA lanes
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&m->full[s], 1);
      mbar_init(&m->empty[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&m->bfull[b], 1);
      mbar_init(&m->bempty[b], 4);
      mbar_init(&m->accfull[b], 4);
      mbar_init(&m->accempty[b], 4);
    }
    mbar_init(&m->route_ready, 1);
    mbar_init(&m->mma_done, 4);
    mbar_init(&m->attn_free, 1);
    for (int i = 0; i < kUQ; ++i) {
      mbar_init(&m->uq_full[i], 1);
      mbar_init(&m->uq_empty[i], 6);  // 4 MMA issuers, stager and epilogue leaders
    }
    for (int i = 0; i < 2; ++i) mbar_init(&m->land[i], 1);
    m->abort = 0;
    m->n_act = 0;
    m->rn_ready = 0;
    for (int i = 0; i < 2; ++i) m->land_out[i] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&m->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (P.ts && threadIdx.x == 0) S.ts[PH_COUNT * kTsSlots] = t_start;

  // Register split: the producer, MMA, stager and image-builder warps (warp
  // groups 0-1) need at most kRegsRoles registers; the epilogue warp group
  // (GEMM epilogues, attention, merge, combine) gets the rest, so that it
  // spills as little as possible (its local memory misses the 28 KB L1 that
  // the shared-memory carve-out leaves).  Sum: 2*128*kRegsRoles +
  // 128*kRegsEpi <= 384*168, the registers the block is launched with; both
  // budgets go back to 168 before the common tail.  Each budget change sits
  // inside its own branch, so that the compiler allocates each role's code
  // for its own budget.
  if (warp >= kEpiBase / 32) {
    reg_alloc<kRegsEpi>();
    pdl_wait();
    named_bar(3, kThreads - 32);  // the launch epoch is read (below)
    run_epilogue(P, S, m->epoch);
    __syncwarp();
    reg_dealloc<kLaunchRegs>();
  } else {
    reg_dealloc<kRegsRoles>();
    if (warp == 0) {
      // weights depend on nothing in flight: stream them before the previous
      // launch has finished
      if (lane_id() == 0) run_producer(P, S);
    } else {
      pdl_wait();
      // One read of the launch epoch per CTA, before any of its arrivals: CTA 0
      // advances the epoch only after every CTA has arrived on the last counter.
      if (threadIdx.x == 32) m->epoch = *reinterpret_cast<volatile uint32_t*>(P.epoch);
      named_bar(3, kThreads - 32);
      if (threadIdx.x == 32) stamp(P, S, PH_COUNT, 1);
      const uint32_t epoch = m->epoch;
      if (warp >= 1 && warp <= 4) {
        if (lane_id() == 0) run_mma(P, S);
      } else if (warp == 5 || warp == 6) {
        run_stager(P, S, epoch);
      } else if (warp == 7) {
        if (blockIdx.x == 0 && P.pf_n > 0) prefetch_bookkeeping(P, S, epoch);
        if (P.moe) build_expert_images(P, S, epoch);
      }
    }
    __syncwarp();
    reg_alloc<kLaunchRegs>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(m->tmem_base, kTmemCols);
  }
  if (P.ts) {
    if (threadIdx.x == 0) stamp(P, S, PH_COUNT, 2);
    __syncthreads();
    for (int i = threadIdx.x; i < kTsPerCta; i += kThreads)
      P.ts[static_cast<size_t>(blockIdx.x) * kTsPerCta + i] = S.ts[i];
  }
}

const void* layer_kernel_ptr() { return reinterpret_cast<const void*>(&mk_layer_kernel); }
uint32_t layer_smem_bytes() { return kSmemBytes; }

}  // namespace mk
