// moe_kernel.cu -- the MoE layer as one persistent megakernel coordinated by
// an Event Tensor ("Event Tensor: A Unified Abstraction for Compiling Dynamic
// Megakernel", Figure 2 and Figure 5(b); podcast cues 7, 9 and 11).
//
// Tasks (one per tile) and the events between them:
//
//   NORM(b,tb)      chain only: RMSNorm of token block tb -> xn   flag norm_flag[tb]
//   ROUTER(b,tb,c)  tcgen05 tile: logits of token block tb over H-chunk c.
//                   H unsplit (NC == 1): bias, top-k, softmax over the
//                   top-k and the block's expert histogram right here   -> ev_route (+1)
//                   H split: fixed-point partial sums                  -> ev_rblk[tb] (+1)
//   TOPK(b,tb)      H split only: sums the NC partials, top-k, softmax,
//                   expert histogram                                    -> ev_route (+1)
//   SCAN(b)         counts, exp_indptr, expert chunks; DATA-DEPENDENT
//                   EVENT UPDATE: ev_expert[e] := counts[e]; publishes
//                   the plan                                           flag plan_flag
//   PERM(b,tb)      writes x_perm rows [exp_indptr[e] + rank]           -> ev_expert[e] (-n)
//   GU(b,ch,n)      gate/up tile: 64 gate + 64 up weight rows x chunk
//                   tokens, SwiGLU -> act                               -> ev_act[ch] (-1)
//   DN(b,ch,n)      down tile: 128 output columns x chunk tokens -> y   -> ev_down[ch] (-1);
//                   the tile that brings ev_down[ch] to zero notifies the
//                   token blocks of the chunk's rows                    -> ev_tok[tb] (-rows)
//   COMB(b,tb)      out[t] = sum_j w[t,j] y[pos[t,j]] (+ residual)     flag comb_flag[tb]
//
// DATA-DEPENDENT TASK TRIGGERING: expert e owns the rows
// [exp_indptr[e], exp_indptr[e+1]) and fires exactly the GU tiles of the
// chunks covering them (ceil(counts[e]/128) chunks); an expert with no tokens
// fires none.
//
// Static scheduling: every CTA walks a fixed, stage-ordered list of task
// slots computed from (T, blockIdx) and from the published chunk count,
// spinning on each task's input event before handing it to its roles.
// Dynamic scheduling: the notify that brings an event to zero pushes the
// consumer tasks into a global queue at once (early push); CTAs pop.
//
// Inside a CTA (one per SM, 12 warps):
//   warp 0   scheduler (lane 0): walks or pops tasks, waits on their events,
//            writes them into a shared-memory ring
//   warp 1   TMA producer (lane 0): weight and token tiles -> smem stages
//   warp 2   tcgen05 issuer (lane 0); the warp owns 256 TMEM columns
//   warp 3   notifier: event updates and dynamic early pushes
//   warps 4-11  workers: TMEM epilogues of the router and GEMM tiles and
//            every SIMT task
//
// GEMM tiles are "swap-AB": the MMA's M = 128 weight rows, its N = the
// chunk's token rows rounded up to 16 (16..128).  Decode-sized chunks (a few
// tokens per expert) therefore waste at most 15 columns, and the weight
// stream is what the tile pays for.
#include <cstdio>

#include "../../include/etc_moe.h"
#include "etc_event.cuh"

namespace etc {

struct Task {
  int type, blk, a, b;
  int e, row0, rows, pad;  // expert chunks: act rows [row0, row0 + rows); token rows from
                           // x_perm row pad, or (pad < 0, heavy expert) x row -1 - pad
  unsigned long long t_disp;  // when the scheduler handed the task over (trace only)
};

constexpr int kNoti = 8;  // finished tasks waiting for the notifier warp
constexpr int kMbox = 4;  // pair tiles, dynamic queue: tasks the even CTA forwards to its peer
constexpr int kPermSlots = 6;                         // token rows in flight in a permute task
constexpr int kPermRowOff = 8 * 1024;                 // row slots' offset in the worker scratch
constexpr int kPermBytes = kSimtBytes - kPermRowOff;  // row slots' bytes

struct Ctrl {
  uint64_t full[kStagesMax];
  uint64_t empty[kStagesMax];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t rfull[kRing];
  uint64_t rempty[kRing];
  uint64_t nfull[kNoti];
  uint64_t nempty[kNoti];
  uint64_t pbar[kPermSlots];  // permute row loads
  Task ring[kRing];
  Task wtask[2];     // workers' broadcast of the current task (double-buffered)
  Task noti[kNoti];  // workers -> notifier
  Task mbox[kMbox];  // pair peer's scheduler -> this CTA's scheduler (dynamic queue)
  uint64_t mb_full[kMbox];
  uint64_t mb_empty[kMbox];
  uint32_t tmem_base;
  int wflag[2];      // workers' broadcast flags
  int started;       // tasks the workers have taken from the ring
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

constexpr int kRingConsumers = 3;  // TMA lane, MMA lane, worker thread 0
constexpr int kWarpNotifier = 3;

__device__ __forceinline__ QueueView queue_of(const MegaParams& p) {
  QueueView q;
  const int par = p.epoch & 1;
  q.slots = p.ws.qslots[par];
  q.head = p.ws.qhead[par];
  q.tail = p.ws.qtail[par];
  q.cap = p.ws.qcap;
  // DYNAMIC seeds the queue with the first tasks (virtual slots 0..n_seed-1).
  // (dense MLP: every gate/up tile).
  q.n_seed = p.mode != ETC_SCHED_DYNAMIC ? 0
             : p.dense                   ? p.n_chunks * p.NT_gu
             : p.use_norm                ? p.nb
                                         : p.n_router;
  q.epoch = p.epoch;
  return q;
}

__device__ __forceinline__ bool dynamic_mode(const MegaParams& p) { return p.mode == ETC_SCHED_DYNAMIC; }

// CTA pairs.  With pair tiles every task belongs to a pair of CTAs (a cluster
// of two): an expert or router tile is one cta_group::2 MMA over both CTAs'
// operands, and a SIMT task on pair token block a is split into the 32-token
// blocks 2a (even CTA) and 2a + 1 (odd CTA).
__device__ __forceinline__ int pair_rank(const MegaParams& p) {
  return p.pair ? static_cast<int>(cluster_ctarank()) : 0;
}
// This CTA's token block of a routing task on (pair) block a.
__device__ __forceinline__ int my_tb(const MegaParams& p, int a) { return p.pair ? 2 * a + pair_rank(p) : a; }
// Scheduling unit of this CTA (its own index, or its pair's) and the number of units.
__device__ __forceinline__ int sched_unit(const MegaParams& p) {
  return p.pair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
}
__device__ __forceinline__ int sched_units(const MegaParams& p) {
  return p.pair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
}
// Token rows a pair expert tile's MMA covers: the chunk rounded to 32, i.e.
// a multiple of 16 rows from each CTA.
__device__ __forceinline__ int pair_npad(int rows) { return (rows + 31) & ~31; }
// Whether the expert tiles and the finaliser go through the queue (DYNAMIC and
// MIXED); the routing tasks do only in DYNAMIC.
__device__ __forceinline__ bool tiles_queued(const MegaParams& p) { return p.mode != ETC_SCHED_STATIC; }

// Whether block blk's combine finaliser has work: releasing the next block's
// RMSNorm in the chain, or rounding the last block's rows to a bf16 output.
// Otherwise the down tiles' fp32 additions are the result and no COMB runs.
// The dense MLP's down tiles store their outputs themselves.
__device__ __forceinline__ bool needs_comb(const MegaParams& p, int blk) {
  return !p.dense && (blk < p.n_blocks - 1 || p.out_bf16 != 0 || p.ordered != 0);
}

// Dense MLP: the finished gate/up tiles chunk c's down tiles wait for (one more for the
// chunk a fault-injection call names, so that its wait runs out).
__device__ __forceinline__ int dense_gu_target(const MegaParams& p, int c) {
  return p.ev_mul * p.NT_gu + (((p.debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT) && c == p.debug_arg) ? 1 : 0);
}

// Operand stages of a call: narrow tiles 6 x 32 KB (16 KB of weights, then up
// to 16 KB of token rows), wide tiles 4 x 48 KB (32 KB of weights, then the
// token rows).  Calls whose chunks hold at most 32 rows (T <= 32) take 9 x
// 20 KB: 16 KB of weights and at most 4 KB of token rows (or a router block),
// so that half as many bytes again are in flight while weights stream.
struct StageGeom {
  int n;          // stages
  uint32_t bytes; // stride
  uint32_t boff;  // token operand offset in a stage
};
__device__ __forceinline__ StageGeom stage_geom(const MegaParams& p) {
  // Pair tiles: 6 x 32 KB per CTA, 16 KB of weights (its 128 of the pair's
  // 256 weight rows) and up to 16 KB of token rows (its half of the chunk).
  return p.pair   ? StageGeom{kStagesNarrow, kOpABytes + kStageBBytes, kOpABytes}
         : p.wide ? StageGeom{4, kStageABytes + kStageBBytes, kStageABytes}
         : p.thin ? StageGeom{kStagesMax, kStageThinBytes, kOpABytes}
                  : StageGeom{kStagesNarrow, kOpABytes + kStageBBytes, kOpABytes};
}

// Token-major MMA for this expert tile: wide gate/up tiles of full chunks
// (one M=128 x N=256 MMA per K step).  Partial chunks and down tiles measured
// faster swap-AB (M = weight rows, N = the chunk's rows rounded to 16; down
// tiles: the epilogue's coalesced reductions).
__device__ __forceinline__ bool tile_tokmaj(const MegaParams& p, const Task& t) {
  return p.tokmaj && t.type == TK_GU && t.rows == p.cw;
}

// K blocks of a router tile per operand stage: two when the stage holds two
// (weights 16 KB + 32 token rows 4 KB per K block: the wide geometry).
__device__ __forceinline__ int router_kpack(const StageGeom& g) {
  return (g.boff >= 2 * kOpABytes && g.bytes - g.boff >= 2 * kTB * kBK * 2) ? 2 : 1;
}

// Eight consecutive values of block blk's input row `tok` (columns 8c..8c+7):
// the caller's bf16 x for block 0, the fp32 residual stream after that.
__device__ __forceinline__ void load_block_input8(const MegaParams& p, int blk, int tok, int c,
                                                  float (&f)[8]);
__device__ void init_acc_rows(const MegaParams& p, int blk, int tb, int wt, uint8_t* zbuf = nullptr);
__device__ void scan_block(const MegaParams& p, int blk, uint8_t* simt, int wt,
                           const int* s_counts = nullptr);

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

__device__ __forceinline__ void load_block_input8(const MegaParams& p, int blk, int tok, int c,
                                                  float (&f)[8]) {
  if (blk == 0) {
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(tok) * p.H) + c), f);
  } else {
    // written earlier in this kernel by another CTA: L2-only load
    const float4* r = reinterpret_cast<const float4*>(
        p.ws.resid + (static_cast<size_t>(blk - 1) * p.T_max + tok) * p.H + 8 * c);
    const float4 a = __ldcg(r), b = __ldcg(r + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

// Exclusive prefix sum over the 256 worker threads (64-bit, so that two 32-bit
// sums can travel packed in one scan), also giving every thread the sum over
// all 256 values; `tmp` holds >= 8 values.
__device__ __forceinline__ unsigned long long workers_excl_scan_total(unsigned long long v,
                                                                      unsigned long long* tmp, int wt,
                                                                      unsigned long long& total) {
  const int lane = wt & 31, w = wt >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[w] = x;
  named_bar(1, kNumWorkers);
  unsigned long long base = 0, all = 0;
#pragma unroll
  for (int i = 0; i < kNumWorkers / 32; ++i) {
    if (i < w) base += tmp[i];
    all += tmp[i];
  }
  named_bar(1, kNumWorkers);
  total = all;
  return base + x - v;
}

// ---------------------------------------------------------------------------
// SIMT tasks (executed by the 256 worker threads)
// ---------------------------------------------------------------------------

// RMSNorm of token block tb: xn[t] = x[t] / sqrt(mean(x[t]^2) + eps) * g.
__device__ void task_norm(const MegaParams& p, const Task& t, int wt) {
  const int blk = t.blk, tb = t.a;
  const BlockWs& B = p.ws.blk[blk];
  const __nv_bfloat16* g = p.norm_w[blk];
  const int ww = wt >> 5, lane = wt & 31, n8 = p.H / 8;
  for (int r = ww; r < kTB; r += 8) {
    const int tok = tb * kTB + r;
    if (tok >= p.T) break;
    float ss = 0.f;
    for (int c = lane; c < n8; c += 32) {
      float f[8];
      load_block_input8(p, blk, tok, c, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += f[i] * f[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(p.H) + p.eps);
    uint4* dst = reinterpret_cast<uint4*>(p.ws.xn + static_cast<size_t>(tok) * p.H);
    uint4* dst_lo = reinterpret_cast<uint4*>(p.ws.xn_lo + static_cast<size_t>(tok) * p.H);
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    for (int c = lane; c < n8; c += 32) {
      float f[8], w[8], hi[8];
      load_block_input8(p, blk, tok, c, f);
      bf16x8_to_f32(gv[c], w);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = f[i] * inv * w[i];
      const uint4 h = f32_to_bf16x8(f);
      dst[c] = h;
      // The router also reads what the bf16 rounding dropped, so that its
      // logits see the normalised input to about 16 mantissa bits.
      bf16x8_to_f32(h, hi);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] -= hi[i];
      dst_lo[c] = f32_to_bf16x8(f);
    }
  }
  fence_proxy_async_global();  // xn / xn_lo are read next by TMA (router tiles)
  named_bar(1, kNumWorkers);   // notify: norm_flag (by the notifier warp)
  (void)B;
}

// ---------------------------------------------------------------------------
// Routing.  A router task is a tcgen05 tile: A = the router weight [H, E]
// read MN-major (TMEM lane = expert), B = the token block's 32 input rows
// (column = token), K = the task's H range.  With H unsplit (NC == 1) the
// epilogue adds the bias and runs the top-k at once; with H split over NC
// tasks each adds its partial into exact fixed-point sums and a top-k task
// of the block follows.
// ---------------------------------------------------------------------------

// Top-k by warps (blocks of 3 to 8 tokens): one warp per
// token, k rounds of a warp arg-max, ties to the lower expert id; weights the
// softmax over the k selected logits.  Counts the experts in s_cnt.
__device__ void topk_rows_warp(const MegaParams& p, const BlockWs& B, const float* s_log, int tok0,
                               int* s_cnt, int ww, int lane, int* s_sel_ids, float* s_sel_w) {
  const int E = p.E, k = p.k;
  for (int r = ww; r < kTB; r += 8) {
    const int tok = tok0 + r;
    if (tok >= p.T) break;
    float v[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i)
      v[i] = 32 * i + lane < E ? s_log[r * E + 32 * i + lane] : -INFINITY;
    unsigned taken = 0;
    float my_v = -INFINITY;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = 32 * i + lane;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_v = bv;
        my_id = bi;
      }
    }
    const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - v0) : 0.f;
    float z = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < k) {
      B.ids[tok * k + lane] = my_id;
      B.wts[tok * k + lane] = ex / z;
      s_sel_ids[r * k + lane] = my_id;
      s_sel_w[r * k + lane] = ex / z;
      atomicAdd(&s_cnt[my_id], 1);
    }
  }
}


// One level of a pairwise arg-max tree over 2W slots: slot i keeps the better
// of slots i and i + W (logit descending, expert id ascending).
template <int W>
__device__ __forceinline__ void tree_level(float (&cv)[kMaxE / 8], int (&ci)[kMaxE / 8]) {
#pragma unroll
  for (int i = 0; i < W; ++i) {
    if (cv[i + W] > cv[i] || (cv[i + W] == cv[i] && ci[i + W] < ci[i])) {
      cv[i] = cv[i + W];
      ci[i] = ci[i + W];
    }
  }
}

// Top-k by groups of eight threads (blocks of more than 8 tokens):
// the 256 workers hold 32 tokens, thread `sub` of a token's group the logits
// of experts sub, sub + 8, sub + 16, ... (E is a multiple of 8).  k rounds of
// an arg-max over the group (ties to the lower expert id) give the selection
// in rank order; weights: the softmax over the k selected logits.  Counts
// the experts in s_cnt; `logits_out`: also stores the block's logits.
__device__ void topk_rows_group(const MegaParams& p, const BlockWs& B, const float* s_log, int tok0,
                                int nt, int* s_cnt, int wt, int* s_sel_ids, float* s_sel_w,
                                bool logits_out) {
  const int E = p.E, k = p.k, per = E >> 3;
  const int r = wt >> 3, sub = wt & 7;
  const bool live = r < nt;
  float v[kMaxE / 8];
#pragma unroll
  for (int i = 0; i < kMaxE / 8; ++i) v[i] = live && i < per ? s_log[r * E + 8 * i + sub] : -INFINITY;
  if (live && logits_out) {
    float* lrow = B.logits + static_cast<size_t>(tok0 + r) * E;
#pragma unroll
    for (int i = 0; i < kMaxE / 8; ++i)
      if (i < per) lrow[8 * i + sub] = v[i];
  }
  unsigned taken = per >= 32 ? 0u : ~0u << per;  // slots past E count as taken
  float v0 = 0.f, sv0 = 0.f, sv1 = 0.f;
  int si0 = 0, si1 = 0;
  for (int j = 0; j < k; ++j) {
    // this thread's best untaken expert: a pairwise tree (depth 4), taken slots
    // entering as (-inf, no id), which any real entry beats
    float cv[kMaxE / 8];
    int ci[kMaxE / 8];
#pragma unroll
    for (int i = 0; i < kMaxE / 8; ++i) {
      const bool tk = (taken >> i) & 1u;
      cv[i] = tk ? -INFINITY : v[i];
      ci[i] = tk ? 0x7fffffff : 8 * i + sub;
    }
    tree_level<8>(cv, ci);
    tree_level<4>(cv, ci);
    tree_level<2>(cv, ci);
    tree_level<1>(cv, ci);
    float bv = cv[0];
    int bi = ci[0];
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 7) == sub && bi < E) taken |= 1u << (bi >> 3);
    if (j == 0) v0 = bv;
    if (j == sub) { sv0 = bv; si0 = bi; }
    if (j == sub + 8) { sv1 = bv; si1 = bi; }
  }
  const float ex0 = sub < k ? expf(sv0 - v0) : 0.f;
  const float ex1 = sub + 8 < k ? expf(sv1 - v0) : 0.f;
  float z = ex0 + ex1;
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (live) {
    const int tok = tok0 + r;
    if (sub < k) {
      const float wv = ex0 / z;
      B.ids[tok * k + sub] = si0;
      B.wts[tok * k + sub] = wv;
      s_sel_ids[r * k + sub] = si0;
      s_sel_w[r * k + sub] = wv;
      atomicAdd(&s_cnt[si0], 1);
    }
    if (sub + 8 < k) {
      const float wv = ex1 / z;
      B.ids[tok * k + sub + 8] = si1;
      B.wts[tok * k + sub + 8] = wv;
      s_sel_ids[r * k + sub + 8] = si1;
      s_sel_w[r * k + sub + 8] = wv;
      atomicAdd(&s_cnt[si1], 1);
    }
  }
}


// Top-k of the tokens tok0.. of a block whose fp32 logits (bias included) are
// in s_log [kTB][E].  Blocks of at most kTopkRankMax tokens (where this task
// is on the critical path of a one-token call) use all 256 workers at once:
// each (token, expert) pair counts the experts ahead of it in the order
// (logit descending, expert id ascending), two threads per pair for a single
// token; those of rank < k are the selection, in rank order, so ties go to the
// lower expert id.  Blocks of up to kTopkWarpMax tokens take the warp arg-max,
// larger ones the group arg-max above (the same selection; their cost grows
// with k, not with E * T).  Weights: the softmax
// over the k selected logits.  Counts the selected experts in s_cnt, and
// leaves the selection in s_sel_ids / s_sel_w ([kTB][k]).  `scr`: 4 KB of
// scratch.  `logits_out`: also stores the block's logits (router tiles with
// H whole).
constexpr int kTopkRankMax = 2;
constexpr int kTopkWarpMax = 8;
constexpr int kTopkScratchOff = 18 * 1024;  // offset of the top-k scratch in the SIMT region
constexpr int kDirectOff = 24 * 1024;       // direct mode: the scan's expert row offsets
constexpr int kSelBytes = 4 * kTB * kMaxK;  // a block's selected experts (or weights)
constexpr int kSelOff = kDirectOff + 4 * kMaxE;  // the top-k's selection, kept for the scan
constexpr int kGatherOff = 16 * 1024;       // direct mode: gate/up activations of all T tokens
constexpr int kZeroOff = 30 * 1024;         // router tiles: zeros for the block's output rows
constexpr int kDirectTokOff = 20 * 1024;    // direct-mode gate/up tiles: the chunk rows' tokens
constexpr int kZeroBytes = 2 * 1024;
static_assert(kSelOff + 2 * kSelBytes <= kZeroOff && kZeroOff + kZeroBytes <= kSimtBytes,
              "SIMT scratch layout");
__device__ void topk_rows(const MegaParams& p, const BlockWs& B, const float* s_log, int tok0,
                          int* s_cnt, int wt, uint8_t* scr, int* s_sel_ids, float* s_sel_w,
                          bool logits_out = false) {
  const int E = p.E, k = p.k;
  const int nt = max(0, min(kTB, p.T - tok0));
  if (nt > kTopkWarpMax) {
    topk_rows_group(p, B, s_log, tok0, nt, s_cnt, wt, s_sel_ids, s_sel_w, logits_out);
    return;
  }
  if (logits_out)
    for (int idx = wt; idx < nt * E; idx += kNumWorkers) B.logits[static_cast<size_t>(tok0) * E + idx] = s_log[idx];
  if (nt > kTopkRankMax) {
    topk_rows_warp(p, B, s_log, tok0, s_cnt, wt >> 5, wt & 31, s_sel_ids, s_sel_w);
    return;
  }
  float* s_v = reinterpret_cast<float*>(scr);                 // [kTB][kMaxK] selected logits by rank
  int* s_i = reinterpret_cast<int*>(scr + 4 * kTB * kMaxK);  // [kTB][kMaxK] selected experts by rank
  const int tpi = nt * E * 2 <= kNumWorkers ? 2 : 1;          // threads per (token, expert) pair
  const int n_items = nt * E * tpi;
  // every worker runs every round (whole warps meet at the pair shuffle)
  for (int base = 0; base < n_items; base += kNumWorkers) {
    const int it = base + wt;
    const bool act = it < n_items;
    const int idx = act ? it / tpi : 0, part = it - (it / tpi) * tpi;
    const int r = idx / E, e = idx - r * E;
    const float* row = s_log + r * E;
    const float v = row[e];
    int rank = 0;
    const int f_end = act ? (part + 1) * E / tpi : 0;
    for (int f = part * E / tpi; f < f_end; f += 4) {
      const float4 u = *reinterpret_cast<const float4*>(row + f);
      rank += static_cast<int>(u.x > v) | (static_cast<int>(u.x == v) & static_cast<int>(f < e));
      rank += static_cast<int>(u.y > v) | (static_cast<int>(u.y == v) & static_cast<int>(f + 1 < e));
      rank += static_cast<int>(u.z > v) | (static_cast<int>(u.z == v) & static_cast<int>(f + 2 < e));
      rank += static_cast<int>(u.w > v) | (static_cast<int>(u.w == v) & static_cast<int>(f + 3 < e));
    }
    if (tpi == 2) rank += __shfl_xor_sync(0xffffffffu, rank, 1);  // the pair's two halves
    if (act && part == 0 && rank < k) {
      s_v[r * kMaxK + rank] = v;
      s_i[r * kMaxK + rank] = e;
    }
  }
  named_bar(1, kNumWorkers);
  for (int idx = wt; idx < nt * k; idx += kNumWorkers) {
    const int r = idx / k, j = idx - r * k;
    const float* vr = s_v + r * kMaxK;
    const float v0 = vr[0];
    float z = 0.f;
    for (int q = 0; q < k; ++q) z += expf(vr[q] - v0);
    const int e = s_i[r * kMaxK + j], tok = tok0 + r;
    const float wv = expf(vr[j] - v0) / z;
    B.ids[tok * k + j] = e;
    B.wts[tok * k + j] = wv;
    s_sel_ids[r * k + j] = e;
    s_sel_w[r * k + j] = wv;
    atomicAdd(&s_cnt[e], 1);
  }
}

// The block's expert histogram: kept per block (the permute derives its row
// offsets from it) and added into the call's counts (what the scan reads),
// unless it is the call's only block and its task runs the scan itself.
__device__ __forceinline__ void publish_block_counts(const MegaParams& p, const BlockWs& B, int tb,
                                                     const int* s_cnt, int wt, bool sum = true) {
  for (int e = wt; e < p.E; e += kNumWorkers) {
    const int n = s_cnt[e];
    B.blk_cnt[tb * p.E + e] = n;
    if (n && sum) atomicAdd(B.cnt_acc + e, n);
  }
}

// The workers are done with accumulator buffer `acc`: the MMA issuer may
// reuse it.  Pair tiles: the issuer sits in the even CTA and waits for both
// CTAs' workers.
// (PAIR, here and below, is the kernel instantiation's compile-time copy of
// p.pair: the single-CTA kernel holds no pair-only instruction at all.)
template <bool PAIR>
__device__ __forceinline__ void release_acc(Ctrl* c, int acc) {
  if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(&c->tempty[acc], 0));
  else mbar_arrive(&c->tempty[acc]);
}

// Epilogue of a router tile of token block tb (TMEM lane = expert, column =
// token; each worker warp reads its 32 lanes x 16 columns).  Pair tiles: the
// MMA covered 64 tokens, columns 32r..32r+31 being CTA r's block 2a + r.
template <bool PAIR>
__device__ void task_router_epilogue(const MegaParams& p, Ctrl* c, uint8_t* simt, const Task& t,
                                     uint32_t& gemm_i, const Clock& clk, int wt, uint32_t iter) {
  const int acc = gemm_i & 1;
  const uint32_t aph = (gemm_i >> 1) & 1;
  ++gemm_i;
  const int tb = my_tb(p, t.a);
  // While the tile is still on the tensor cores: the block's combine rows.
  const bool zero_rows = t.b == 0;
  if (zero_rows) init_acc_rows(p, t.blk, tb, wt, simt + kZeroOff);
  int* flag = &c->wflag[iter & 1];
  if (wt == 0) *flag = mbar_wait(&c->tfull[acc], aph, clk, 231, PAIR) ? 1 : 0;
  named_bar(1, kNumWorkers);
  const bool ok = *flag != 0;
  tc_fence_after();
  const BlockWs& B = p.ws.blk[t.blk];
  const int w = warp_id(), q = w & 3, h = (w - kWorkerWarp0) >> 2, lane = lane_id();
  const int E = p.E, e = 32 * q + lane;
  const uint32_t col0 = p.pair ? 32u * pair_rank(p) : 0u;
  int* s_cnt = reinterpret_cast<int*>(simt);             // [E]
  float* s_log = reinterpret_cast<float*>(simt + 1024);  // [kTB][E]
  for (int i = wt; i < E; i += kNumWorkers) s_cnt[i] = 0;
  if (ok) {
    float v[16];
    tmem_ld16(c->tmem_base + acc * kAccCols + (static_cast<uint32_t>(32 * q) << 16) + col0 + h * 16, v);
    if (e < E) {
      if (p.NC == 1) {
        const float b = p.bias[t.blk] ? __ldg(p.bias[t.blk] + e) : 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) s_log[(h * 16 + i) * E + e] = v[i] + b;
      } else {
        // Partials over H-chunks are summed exactly, in any order, as 64-bit
        // fixed point (units of 2^-40): the logits do not depend on which
        // chunk lands first.
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int tok = tb * kTB + h * 16 + i;
          if (tok < p.T)
            red_add_u64(B.logit_fx + static_cast<size_t>(tok) * E + e,
                        static_cast<unsigned long long>(
                            __double2ll_rn(static_cast<double>(v[i]) * 1099511627776.0)));
        }
      }
    }
  }
  tc_fence_before();
  named_bar(1, kNumWorkers);
  if (wt == 0) release_acc<PAIR>(c, acc);  // accumulator free for the next tile
  if (ok && p.NC == 1 && tb < p.nb) {
    const int tok0 = tb * kTB;
    topk_rows(p, B, s_log, tok0, s_cnt, wt, simt + kTopkScratchOff,
              reinterpret_cast<int*>(simt + kSelOff), reinterpret_cast<float*>(simt + kSelOff + kSelBytes),
              /*logits_out=*/true);
    named_bar(1, kNumWorkers);
    publish_block_counts(p, B, tb, s_cnt, wt);
  }
  if (zero_rows && wt < 32) {
    bulk_wait_all();             // the zeroed rows are written
    fence_proxy_async_global();  // before any down tile adds into them
  }
  named_bar(1, kNumWorkers);  // notify: ev_route, or ev_rblk[tb] with H split (notifier warp)
}

// Top-k of token block tb as a SIMT task: from the NC summed partials (H
// split), or from logits the caller gave (routing-only calls).
__device__ void task_topk(const MegaParams& p, const Task& t, uint8_t* simt, int wt) {
  const int blk = t.blk, tb = my_tb(p, t.a);
  const BlockWs& B = p.ws.blk[blk];
  const int E = p.E;
  int* s_cnt = reinterpret_cast<int*>(simt);             // [E]
  float* s_log = reinterpret_cast<float*>(simt + 1024);  // [kTB][E]
  for (int i = wt; i < E; i += kNumWorkers) s_cnt[i] = 0;
  const float* bias = p.bias[blk];
  const int tok0 = tb * kTB;
  if (p.logits_in) init_acc_rows(p, blk, tb, wt);  // no router tile ran for this block
  const int ntok = max(0, min(kTB, p.T - tok0));
  const size_t o0 = static_cast<size_t>(tok0) * E;
  const int n = ntok * E;
  if (p.logits_in) {
    for (int idx = wt; idx < n; idx += kNumWorkers) {
      const float s = __ldg(p.logits_in + o0 + idx);
      s_log[idx] = s;
      B.logits[o0 + idx] = s;
    }
  } else {
    // Partial sums written by other CTAs' router tiles (L2-only loads), four
    // per thread in flight before any store.
    for (int base = wt; base < n; base += 4 * kNumWorkers) {
      long long v[4];
      float bi[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kNumWorkers;
        v[u] = 0;
        bi[u] = 0.f;
        if (idx < n) {
          v[u] = static_cast<long long>(__ldcg(B.logit_fx + o0 + idx));
          if (bias) bi[u] = __ldg(bias + (idx - (idx / E) * E));
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * kNumWorkers;
        if (idx < n) {
          float s = static_cast<float>(static_cast<double>(v[u]) * 9.094947017729282379e-13);  // 2^-40
          if (bias) s += bi[u];
          B.logit_fx[o0 + idx] = 0ull;  // consumed: re-armed for the next call
          s_log[idx] = s;
          B.logits[o0 + idx] = s;
        }
      }
    }
  }
  named_bar(1, kNumWorkers);
  topk_rows(p, B, s_log, tok0, s_cnt, wt, simt + kTopkScratchOff,
            reinterpret_cast<int*>(simt + kSelOff), reinterpret_cast<float*>(simt + kSelOff + kSelBytes));
  named_bar(1, kNumWorkers);
  if (tb < p.nb) publish_block_counts(p, B, tb, s_cnt, wt, !p.fuse_scan);
  if (p.fuse_scan) {
    // One token block: its histogram (in shared memory) is the call's counts,
    // so the scan runs here, one hop sooner (no separate scan task, no
    // round trip through the count accumulators; the notifier leaves
    // ev_route alone).
    named_bar(1, kNumWorkers);
    scan_block(p, blk, simt, wt, s_cnt);
  }
  named_bar(1, kNumWorkers);  // notify: ev_route (by the notifier warp)
}

// counts / exp_indptr / expert chunks / event inits, from the counts the
// routing tasks summed (thread e < E owns expert e).
__device__ void scan_block(const MegaParams& p, int blk, uint8_t* simt, int wt,
                           const int* s_counts) {
  const BlockWs& B = p.ws.blk[blk];
  const int E = p.E;
  int cnt = 0;
  if (wt < E) {
    if (s_counts) {
      cnt = s_counts[wt];
    } else {
      cnt = __ldcg(B.cnt_acc + wt);
      B.cnt_acc[wt] = 0;  // consumed: re-armed for the next call
    }
  }
  named_bar(1, kNumWorkers);  // the counts are read before the scan scratch is reused
  int* tmp = reinterpret_cast<int*>(simt);  // scan scratch [32]
  unsigned long long* scr = reinterpret_cast<unsigned long long*>(simt + 256);
  const int cw = p.cw;
  // A heavy expert runs over all T rows of x: T act rows, ceil(T / cw)
  // chunks, numbered before every other expert's (the static walk and the
  // queue take them first: they need no permuted rows).
  const bool heavy = p.heavy_min > 0 && wt < E && cnt >= p.heavy_min;
  const int arows = heavy ? p.T : cnt;
  const int nch = (arows + cw - 1) / cw;
  int row0, arow0, ch0, n_rows, n_chunks, n_heavy_ch = 0;
  unsigned long long tot = 0;
  if (p.heavy_min == 0) {
    // rows (low half) and chunks (high half) of the experts before this one, in one scan
    const unsigned long long pre = workers_excl_scan_total(
        (static_cast<unsigned long long>(nch) << 32) | static_cast<unsigned>(cnt), scr, wt, tot);
    row0 = arow0 = static_cast<int>(pre & 0xffffffffu);
    ch0 = static_cast<int>(pre >> 32);
    n_rows = static_cast<int>(tot & 0xffffffffu);
    n_chunks = static_cast<int>(tot >> 32);
  } else {
    // x_perm rows (low) and act rows (high); then heavy experts' chunks (low)
    // and the other experts' chunks (high)
    const unsigned long long pre = workers_excl_scan_total(
        (static_cast<unsigned long long>(arows) << 32) | static_cast<unsigned>(cnt), scr, wt, tot);
    row0 = static_cast<int>(pre & 0xffffffffu);
    arow0 = static_cast<int>(pre >> 32);
    n_rows = static_cast<int>(tot & 0xffffffffu);
    const unsigned long long pc = workers_excl_scan_total(
        (static_cast<unsigned long long>(heavy ? 0 : nch) << 32) | static_cast<unsigned>(heavy ? nch : 0),
        scr, wt, tot);
    n_heavy_ch = static_cast<int>(tot & 0xffffffffu);
    n_chunks = n_heavy_ch + static_cast<int>(tot >> 32);
    ch0 = heavy ? static_cast<int>(pc & 0xffffffffu) : n_heavy_ch + static_cast<int>(pc >> 32);
  }
  if (wt < E) {
    B.counts[wt] = cnt;
    B.exp_indptr[wt] = row0;
    B.chunk_indptr[wt] = ch0;  // (first chunk of the expert; its chunks are consecutive)
    B.heavy[wt] = heavy ? 1 : 0;
    if (wt == 0) {
      B.exp_indptr[E] = n_rows;
      B.chunk_indptr[E] = n_chunks;
      B.meta[0] = n_chunks;
      B.meta[1] = n_chunks * p.NT_gu;
      B.meta[2] = n_chunks * p.NT_dn;
      B.meta[3] = n_heavy_ch;
    }
    for (int c = 0; c < nch; ++c) {
      const int chn = ch0 + c;
      B.chunk_expert[chn] = wt;
      B.chunk_row0[chn] = arow0 + c * cw;
      B.chunk_rows[chn] = min(cw, arows - c * cw);
      B.chunk_src[chn] = heavy ? -1 - c * cw : row0 + c * cw;
      // one notify per tile, or per CTA of a pair tile
      B.ev_act[chn] = p.ev_mul * p.NT_gu;
      B.ev_down[chn] = p.ev_mul * p.NT_dn;
    }
    // Data-dependent event update: expert e waits for its counts[e] rows
    // (none in direct mode or for a heavy expert: their tiles read x itself).
    const int extra = ((p.debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT) && wt == p.debug_arg) ? 1 : 0;
    B.ev_expert[wt] = (p.direct || heavy ? 0 : cnt) + extra;
  }
  int* s_row0 = reinterpret_cast<int*>(simt + kDirectOff);  // [kMaxE]
  if (p.direct) {
    // Direct mode (one token block, no permute task): the expert-sorted row of
    // every slot (t, j) is exp_indptr[e] + the number of earlier slots routed
    // to the same expert (ascending token within an expert).
    // The selection of the call's single token block: still in shared memory
    // when the top-k task runs the scan itself, else read back.
    int* s_ids = reinterpret_cast<int*>(simt + kSelOff);                  // [kTB * k]
    float* s_w = reinterpret_cast<float*>(simt + kSelOff + kSelBytes);   // [kTB * k]
    const int ns = p.T * p.k;
    if (wt < E) s_row0[wt] = row0;
    if (!s_counts)
      for (int i = wt; i < ns; i += kNumWorkers) {
        s_ids[i] = __ldcg(B.ids + i);
        s_w[i] = __ldcg(B.wts + i);
      }
    named_bar(1, kNumWorkers);
    for (int sl = wt; sl < ns; sl += kNumWorkers) {
      const int e = s_ids[sl];
      int rank = 0;
      for (int s2 = 0; s2 < sl; ++s2) rank += s_ids[s2] == e;
      const int row = s_row0[e] + rank;
      B.pos[sl] = row;
      B.row_token[row] = sl / p.k;
      B.row_w[row] = s_w[sl];
    }
  }
  if (needs_comb(p, blk)) {
    // token rows the finaliser of (pair) token block tb waits for
    const int tbw = p.pair ? 2 * kTB : kTB;
    for (int tb = wt; tb < p.nbp; tb += kNumWorkers)
      B.ev_tok[tb] = p.k * (min(p.T, tb * tbw + tbw) - tb * tbw);
  }
  // No per-thread fence: the barrier orders every worker's plan writes before
  // worker 0's gpu-scope fence and plan-flag release below (and before each
  // queue-slot writer's fence), which publish them cumulatively.  A fence by
  // all 256 threads cost ~1.5 us of a decode call's critical path.
  named_bar(1, kNumWorkers);
  if (wt == 0) {
    st_relaxed(B.ev_route, 0);
    const bool dyn = dynamic_mode(p);
    if (tiles_queued(p)) {
      // Tasks of the block that pass through the queue: all of them in
      // DYNAMIC, the expert tiles and the finaliser in MIXED.
      const int nbp = p.nbp;
      const int routing = dyn ? (p.use_norm ? nbp : 0) + p.n_router + (p.NC > 1 ? nbp : 0) +
                                    (p.fuse_scan ? 0 : 1) + (p.direct ? 0 : nbp * p.PP)
                              : 0;
      const int blk_tasks = routing + n_chunks * (p.NT_gu + p.NT_dn) + (needs_comb(p, blk) ? nbp : 0);
      const int acc = (blk == 0 ? 0 : *p.ws.qacc) + blk_tasks;
      *p.ws.qacc = acc;
      if (blk == p.n_blocks - 1) *p.ws.qtotal = acc;
    }
    __threadfence();
    st_release(B.plan_flag, p.epoch);
    if (tiles_queued(p) && blk == p.n_blocks - 1) st_release(p.ws.qtotal_flag, p.epoch);
    // The tasks this plan makes ready at once: the block's permute tasks
    // (DYNAMIC), then the gate/up tiles that need no permuted rows (DYNAMIC
    // and MIXED): every one in direct mode, the heavy experts' otherwise.
    const int n_perm = (!p.direct && dyn) ? p.nbp * p.PP : 0;
    const int n_gu = tiles_queued(p) ? (p.direct ? n_chunks : n_heavy_ch) * p.NT_gu : 0;
    const int n_push = n_perm + n_gu;
    if (n_push) {
      const QueueView q = queue_of(p);
      tmp[0] = q.n_seed + atom_add_relaxed(q.tail, n_push);
    }
    tmp[1] = n_push;
    tmp[2] = n_perm;
  }
  if (tiles_queued(p)) {
    // Every worker writes some of the reserved slots.
    named_bar(1, kNumWorkers);
    const int base = tmp[0], n_push = tmp[1], n_perm = tmp[2];
    const QueueView q = queue_of(p);
    __threadfence();  // the plan above is published with the slots
    for (int i = wt; i < n_push; i += kNumWorkers) {
      if (base + i >= q.cap) {
        const Clock c0{~0ull, p.ws.status, p.ws.status_host};
        raise_error(c0, DERR_QUEUE_OVERFLOW, 3, base + i);
        break;
      }
      const int g = i - n_perm;  // gate/up tile g of the chunks pushed here
      // (fault injection: the tiles of the expert that waits for one row more
      // are never made ready, so a queue pop runs out of time)
      if (g >= 0 && (p.debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT) &&
          __ldcg(B.chunk_expert + g / p.NT_gu) == p.debug_arg)
        continue;
      const uint32_t d = g >= 0 ? task_enc(TK_GU, blk, g / p.NT_gu, g % p.NT_gu)
                                : task_enc(TK_PERM, blk, i / p.PP, i % p.PP);
      st_relaxed_u64(&q.slots[base + i], (static_cast<unsigned long long>(q.epoch) << 32) | d);
    }
  }
}

__device__ void task_scan(const MegaParams& p, const Task& t, uint8_t* simt, int wt) {
  scan_block(p, t.blk, simt, wt);
}

// fp32 rows that block blk's combine accumulates into: the residual stream of
// the next block, the caller's fp32 output, or the accumulator behind a bf16
// output.
__device__ __forceinline__ float* acc_rows(const MegaParams& p, int blk) {
  if (blk < p.n_blocks - 1) return p.ws.resid + static_cast<size_t>(blk) * p.T_max * p.H;
  return p.out_bf16 ? p.ws.acc : static_cast<float*>(p.out);
}

// Combine rows of token block tb start at 0 (or at the block's input in the
// chain) before any down tile adds into them.  Run by the block's routing
// task, which every down tile of the block follows.  (A routing-only call
// has no output rows.)
__device__ void init_acc_rows(const MegaParams& p, int blk, int tb, int wt, uint8_t* zbuf) {
  float* accr = acc_rows(p, blk);
  if (accr == nullptr || p.ordered) return;  // (ordered combine: the finaliser writes whole rows)
  const int ww = wt >> 5, lane = wt & 31, n8 = p.H / 8, t0 = tb * kTB, ntok = min(kTB, p.T - t0);
  if (zbuf != nullptr && !p.use_norm) {
    // Zeros, written by the bulk-copy engine from kZeroBytes of zeroed shared
    // memory (the lanes of worker warp 0 issue the copies and wait for them
    // before the task's notify): the workers go on to the tile's epilogue.
    for (int i = wt; i < kZeroBytes / 16; i += kNumWorkers)
      reinterpret_cast<uint4*>(zbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // visible to the bulk-copy engine
    named_bar(1, kNumWorkers);
    if (wt < 32 && ntok > 0) {
      uint8_t* dst = reinterpret_cast<uint8_t*>(accr + static_cast<size_t>(t0) * p.H);
      const uint32_t total = static_cast<uint32_t>(ntok) * static_cast<uint32_t>(p.H) * 4u;
      for (uint32_t off = wt * kZeroBytes; off < total; off += 32 * kZeroBytes)
        bulk_store(dst + off, zbuf, min(static_cast<uint32_t>(kZeroBytes), total - off));
      bulk_commit();
    }
    return;
  }
  for (int r = ww; r < ntok; r += 8) {
    const int tok = t0 + r;
    float4* d = reinterpret_cast<float4*>(accr + static_cast<size_t>(tok) * p.H);
    for (int c = lane; c < n8; c += 32) {
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (p.use_norm) load_block_input8(p, blk, tok, c, x);
      d[2 * c] = make_float4(x[0], x[1], x[2], x[3]);
      d[2 * c + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
}

// Writes the rows of part t.b of token block tb (kTB / PP tokens; PP > 1
// spreads the copies of few blocks over more CTAs) into x_perm at
// exp_indptr[e] + rank, records each row's token and routing weight, and the
// part's expert histogram (what its notify takes off ev_expert).  The rows
// move through shared memory with the bulk-copy engine: each token row is
// read once (kPermSlots rows in flight) and stored to its k expert-sorted
// rows by k lanes of worker warp 0.
__device__ void task_perm(const MegaParams& p, Ctrl* c, const Task& t, uint8_t* simt, int wt,
                          uint32_t& li, const Clock& clk) {
  const int blk = t.blk, tb = my_tb(p, t.a), part = t.b;
  const BlockWs& B = p.ws.blk[blk];
  const int E = p.E, k = p.k;
  int* s_run = reinterpret_cast<int*>(simt);
  int* s_slot = s_run + kMaxE;
  int* s_ids = s_slot + kTB * kMaxK;
  int* s_part = s_ids + kTB * kMaxK;  // [kNumWorkers]
  int* s_pcnt = s_part + kNumWorkers; // [E]
  unsigned* s_mask = reinterpret_cast<unsigned*>(s_pcnt + kMaxE);  // [E] tokens of the block per expert
  int* s_heavy = reinterpret_cast<int*>(s_mask + kMaxE);             // [E] experts that read x itself
  static_assert(4 * (5 * kMaxE + 2 * kTB * kMaxK + kNumWorkers) <= kPermRowOff, "permute tables");
  static_assert(kTB <= 32, "a token block's tokens form one 32-bit mask");
  uint8_t* rows = simt + kPermRowOff;
  const int t0 = tb * kTB, ntok = max(0, min(kTB, p.T - t0));  // (odd CTA of the last pair block: none)
  const int TP = kTB / p.PP, r_lo = min(ntok, part * TP), r_hi = min(ntok, r_lo + TP);
  const int nmine = r_hi - r_lo;
  const __nv_bfloat16* src = p.use_norm ? p.ws.xn : p.x;
  const uint32_t RB = static_cast<uint32_t>(p.H) * 2;
  const int nslot = min(kPermSlots, kPermBytes / static_cast<int>(RB));
  if (wt == 0) {
    for (int r = 0; r < min(nmine, nslot); ++r) {
      const int sl = (li + r) % nslot;
      mbar_arrive_expect_tx(&c->pbar[sl], RB);
      bulk_load(rows + sl * RB, src + static_cast<size_t>(t0 + r_lo + r) * p.H, RB, &c->pbar[sl]);
    }
  }
  // First row of each expert in this block: exp_indptr[e] plus the rows of e
  // in the blocks before tb, summed from the block histograms by `per`
  // threads per expert.
  // (16 loads in flight per thread).
  const int per = kNumWorkers / E;
  {
    const int e = wt % E, q = wt / E;
    int sum = 0;
    if (q < per) {
      for (int b0 = q; b0 < tb; b0 += 16 * per) {
        int x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int b = b0 + u * per;
          x[u] = b < tb ? __ldcg(B.blk_cnt + b * E + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) sum += x[u];
      }
    }
    s_part[wt] = sum;
  }
  for (int i = wt; i < r_hi * k; i += kNumWorkers) s_ids[i] = __ldcg(B.ids + t0 * k + i);
  for (int i = wt; i < E; i += kNumWorkers) {
    s_mask[i] = 0u;
    s_heavy[i] = p.heavy_min > 0 ? __ldcg(B.heavy + i) : 0;
  }
  named_bar(1, kNumWorkers);
  for (int e = wt; e < E; e += kNumWorkers) {
    int run = __ldcg(B.exp_indptr + e);
    for (int j = 0; j < per; ++j) run += s_part[j * E + e];
    s_run[e] = run;
  }
  // The block's tokens (up to this part's end) of each expert, as a bit mask
  // (a token block has 32 tokens; one token's k experts are distinct).
  for (int i = wt; i < r_hi * k; i += kNumWorkers) atomicOr(&s_mask[s_ids[i]], 1u << (i / k));
  named_bar(1, kNumWorkers);
  // Rank of slot (r, j) among the block's rows of its expert: the block's
  // tokens before r that chose the same expert (ascending token order).
  for (int i = r_lo * k + wt; i < r_hi * k; i += kNumWorkers) {
    const int e = s_ids[i], r = i / k;
    s_slot[i] = s_run[e] + __popc(s_mask[e] & ((1u << r) - 1u));
  }
  {
    const unsigned part_bits = (r_hi >= 32 ? ~0u : (1u << r_hi) - 1u) & ~((1u << r_lo) - 1u);
    for (int e = wt; e < E; e += kNumWorkers) s_pcnt[e] = __popc(s_mask[e] & part_bits);
  }
  named_bar(1, kNumWorkers);
  for (int i = r_lo * k + wt; i < r_hi * k; i += kNumWorkers) {
    const int row = s_slot[i];
    B.pos[t0 * k + i] = row;
    B.row_token[row] = t0 + i / k;
    B.row_w[row] = __ldcg(B.wts + t0 * k + i);
  }
  if (tb < p.nb)
    for (int e = wt; e < E; e += kNumWorkers)  // (a heavy expert waits for no rows)
      B.part_cnt[(tb * p.PP + part) * E + e] = s_heavy[e] ? 0 : s_pcnt[e];
  if (wt < 32) {
    // Warp 0 issues the copies: G groups of k lanes take every G-th row, lane
    // j of a group storing the row's slot j (one thread issuing all of them
    // measured 20 % slower); the group's first lane refills the row's shared
    // memory slot once the group's stores have read it.  G divides nslot, so
    // the rows that share a slot (nslot apart) fall to one group, which waits
    // for each of the slot's loads in turn (a parity wait could not tell a
    // load two phases ahead from the one before it).
    int G = 32 / k;
    while (nslot % G) --G;
    const int lane = wt, g = lane / k, j = lane - g * k;
    if (g < G) {
      const unsigned gm = (k >= 32 ? 0xffffffffu : ((1u << k) - 1u)) << (g * k);
      for (int r = g; r < nmine; r += G) {
        const uint32_t L = li + r;
        const int sl = L % nslot;
        const bool got = mbar_wait(&c->pbar[sl], (L / nslot) & 1, clk, 270);
        if (!__all_sync(gm, got)) break;
        const uint8_t* srow = rows + sl * RB;
        const int i = (r_lo + r) * k + j;
        if (!s_heavy[s_ids[i]])  // (a heavy expert's tiles read x itself)
          bulk_store(p.ws.x_perm + static_cast<size_t>(s_slot[i]) * p.H, srow, RB);
        bulk_commit();
        const int nx = r + nslot;
        if (nx < nmine) {
          bulk_wait_read_all();  // the slot's row has been read out before it is refilled
          __syncwarp(gm);
          if (j == 0) {
            mbar_arrive_expect_tx(&c->pbar[sl], RB);
            bulk_load(rows + sl * RB, src + static_cast<size_t>(t0 + r_lo + nx) * p.H, RB, &c->pbar[sl]);
          }
        }
      }
    }
    bulk_wait_all();  // x_perm rows written before the notify
    li += nmine;
  }
  fence_proxy_async_global();  // x_perm / row tables are read next by other CTAs' TMA
  named_bar(1, kNumWorkers);   // notify: ev_expert[e] per expert (by the notifier warp)
}

// Finaliser of token block tb once every down tile touching it has added its
// weighted expert rows: rounds the rows to bf16 when the output is bf16, and
// in the chain releases the next block's RMSNorm of tb.  Ordered combine: the
// down tiles stored their rows y; here out[t] = (residual +) sum over j in
// order 0..k-1 of w[t,j] * y[pos[t,j]], one fused multiply-add per term.
__device__ void task_comb(const MegaParams& p, const Task& t, uint8_t* simt, int wt) {
  const int blk = t.blk, tb = my_tb(p, t.a);
  const BlockWs& B = p.ws.blk[blk];
  const int ww = wt >> 5, lane = wt & 31, n8 = p.H / 8;
  const bool last = blk == p.n_blocks - 1;
  if (p.ordered) {
    float* resid = last ? nullptr : acc_rows(p, blk);
    // the block's rows and weights (written by other CTAs) into shared memory
    int* s_pos = reinterpret_cast<int*>(simt);                  // [kTB * kMaxK]
    float* s_w = reinterpret_cast<float*>(simt + 4 * kTB * kMaxK);
    const int t0 = tb * kTB, ntok = max(0, min(kTB, p.T - t0));
    for (int i = wt; i < ntok * p.k; i += kNumWorkers) {
      s_pos[i] = __ldcg(B.pos + t0 * p.k + i);
      s_w[i] = __ldcg(B.wts + t0 * p.k + i);
    }
    named_bar(1, kNumWorkers);
    for (int r = ww; r < ntok; r += 8) {
      const int tok = t0 + r;
      const int* rows = s_pos + r * p.k;
      const float* wj = s_w + r * p.k;
      for (int c = lane; c < n8; c += 32) {
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (p.use_norm) load_block_input8(p, blk, tok, c, f);
        for (int j = 0; j < p.k; ++j) {
          const float4* y = reinterpret_cast<const float4*>(p.ws.yperm + static_cast<size_t>(rows[j]) * p.H) + 2 * c;
          const float4 a = __ldcg(y), b = __ldcg(y + 1);
          f[0] = fmaf(wj[j], a.x, f[0]); f[1] = fmaf(wj[j], a.y, f[1]);
          f[2] = fmaf(wj[j], a.z, f[2]); f[3] = fmaf(wj[j], a.w, f[3]);
          f[4] = fmaf(wj[j], b.x, f[4]); f[5] = fmaf(wj[j], b.y, f[5]);
          f[6] = fmaf(wj[j], b.z, f[6]); f[7] = fmaf(wj[j], b.w, f[7]);
        }
        if (!last) {
          float4* d = reinterpret_cast<float4*>(resid + static_cast<size_t>(tok) * p.H) + 2 * c;
          d[0] = make_float4(f[0], f[1], f[2], f[3]);
          d[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else if (p.out_bf16) {
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(tok) * p.H)[c] =
              f32_to_bf16x8(f);
        } else {
          float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.out) + static_cast<size_t>(tok) * p.H) + 2 * c;
          d[0] = make_float4(f[0], f[1], f[2], f[3]);
          d[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
      }
    }
  } else if (last && p.out_bf16) {
    for (int r = ww; r < kTB; r += 8) {
      const int tok = tb * kTB + r;
      if (tok >= p.T) break;
      const float4* s = reinterpret_cast<const float4*>(p.ws.acc + static_cast<size_t>(tok) * p.H);
      uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(tok) * p.H);
      for (int c = lane; c < n8; c += 32) {
        const float4 a = __ldcg(s + 2 * c), b = __ldcg(s + 2 * c + 1);
        const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        d[c] = f32_to_bf16x8(f);
      }
    }
  }
  named_bar(1, kNumWorkers);  // notify: comb_flag (by the notifier warp)
}

// TMEM epilogue of a GU or DN tile, then its notify.
// act rows of the dense MLP (larger than L2, re-read only by the down
// phase) are stored evict-first, so that they do not push x and the weight
// slices in use out of L2; the MoE layer's act (re-read soon, from L2) is
// stored normally.
// SiLU, x * sigmoid(x), with the fast division (2 ulp): its result is rounded
// to bf16 right after, far coarser, and the IEEE division's refinement cost
// about 2 us of a one-token gate/up epilogue.  For x < -87 the denominator is
// past 2^126 and the result is 0, the function's limit.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ void store_act(const MegaParams& p, uint4* dst, const uint4& v) {
  if (p.dense) __stcs(dst, v);
  else *dst = v;
}

template <bool PAIR>
__device__ void task_gemm_epilogue(const MegaParams& p, Ctrl* c, uint8_t* epi, uint8_t* simt,
                                   const Task& t, uint32_t& gemm_i, const Clock& clk, int wt,
                                   uint32_t iter) {
  const int acc = gemm_i & 1;
  const uint32_t aph = (gemm_i >> 1) & 1;
  ++gemm_i;
  int* flag = &c->wflag[iter & 1];
  const BlockWs& B = p.ws.blk[t.blk];
  // Down tiles: each chunk row's token and routing weight, for the combine,
  // read while the tile is still on the tensor cores.
  int* s_rtok = reinterpret_cast<int*>(simt + 2 * kEpiHalfBytes);                 // [256]
  float* s_rw = reinterpret_cast<float*>(simt + 2 * kEpiHalfBytes + 4 * kBT2);    // [256]
  const bool fused_comb = t.type == TK_DN && !p.dense && !p.ordered;
  // Direct-mode gate/up tiles: each chunk row's token, read while the tile
  // is still on the tensor cores (the scan wrote them before the tile ran).
  int* s_dtok = reinterpret_cast<int*>(simt + kDirectTokOff);  // [kTB]
  if (t.type == TK_GU && p.direct)
    for (int i = wt; i < t.rows; i += kNumWorkers) s_dtok[i] = __ldcg(B.row_token + t.pad + i);
  if (fused_comb) {
    if (t.pad >= 0) {
      for (int r = wt; r < t.rows; r += kNumWorkers) {
        s_rtok[r] = __ldcg(B.row_token + t.pad + r);
        s_rw[r] = __ldcg(B.row_w + t.pad + r);
      }
    } else {
      // Heavy expert: chunk row r is token -1 - pad + r; its weight for this
      // expert from the token's selection (no row: a token that did not
      // choose the expert, which adds nothing).
      const int tok0 = -1 - t.pad;
      for (int r = wt; r < t.rows; r += kNumWorkers) {
        const int tok = tok0 + r;
        int hit = -1;
        float w = 0.f;
        for (int j = 0; j < p.k; ++j)
          if (__ldcg(B.ids + static_cast<size_t>(tok) * p.k + j) == t.e) {
            hit = tok;
            w = __ldcg(B.wts + static_cast<size_t>(tok) * p.k + j);
          }
        s_rtok[r] = hit;
        s_rw[r] = w;
      }
    }
  }
  if (wt == 0) *flag = mbar_wait(&c->tfull[acc], aph, clk, 230, PAIR) ? 1 : 0;
  named_bar(1, kNumWorkers);
  const bool ok = *flag != 0;
  tc_fence_after();
  const int w = warp_id(), q = w & 3, h = (w - kWorkerWarp0) >> 2, lane = lane_id();
  const int i128 = q * 32 + lane;
  float* U = reinterpret_cast<float*>(epi + h * kEpiHalfBytes);                     // [2][16][32]
  __nv_bfloat16* S = reinterpret_cast<__nv_bfloat16*>(epi + h * kEpiHalfBytes + 4096);  // [16][128]
  const uint32_t tbase = c->tmem_base + acc * kAccCols + (static_cast<uint32_t>(32 * q) << 16);
  const int ncb = (t.rows + 15) >> 4;
  // Pair tiles: this CTA's 64 intermediate columns (gate/up) or 128 output
  // columns (down) of the pair's tile; the accumulator holds all chunk rows.
  const int rank = pair_rank(p);
  if (ok) {
    if (t.type == TK_GU && tile_tokmaj(p, t)) {
      // Token-major: TMEM lane = chunk row, columns 0-127 gate and 128-255 up
      // of the tile's 128 intermediate columns; each worker half takes 64 of
      // them, so a thread writes one 128-byte piece of its row's act.
      const int r = 32 * q + lane;
      __nv_bfloat16* arow = p.ws.act + static_cast<size_t>(t.row0 + r) * p.I + t.b * kGuRowsW + 64 * h;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float g[16], u[16];
        tmem_ld16(tbase + 64 * h + 16 * cb, g);
        tmem_ld16(tbase + kGuRowsW + 64 * h + 16 * cb, u);
        if (r < t.rows) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float a0 = silu(g[2 * i]) * u[2 * i];
            const float a1 = silu(g[2 * i + 1]) * u[2 * i + 1];
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
            pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(arow + 16 * cb);
          store_act(p, dst, make_uint4(pk[0], pk[1], pk[2], pk[3]));
          store_act(p, dst + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]));
        }
      }
    } else if (t.type == TK_GU && p.wide) {
      // Wide: gate rows in the buffer's first half, up rows in its second;
      // lane = intermediate column, so SwiGLU pairs them in registers.
      for (int cb = h; cb < ncb; cb += 2) {
        float g[16], u[16];
        tmem_ld16(tbase + cb * 16, g);
        tmem_ld16(tbase + kAccCols / 2 + cb * 16, u);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          S[i * 128 + i128] = __float2bfloat16_rn(silu(g[i]) * u[i]);
        named_bar(2 + h, 128);
        // 16 token rows x 128 columns = 256 chunks of 16 bytes
#pragma unroll
        for (int rep = 0; rep < 2; ++rep) {
          const int idx = i128 + 128 * rep, r = idx >> 4, chunk = idx & 15, tok = cb * 16 + r;
          if (tok < t.rows) {
            const uint4 val = *reinterpret_cast<const uint4*>(S + r * 128 + chunk * 8);
            store_act(p, reinterpret_cast<uint4*>(p.ws.act + static_cast<size_t>(t.row0 + tok) * p.I +
                                                  t.b * kGuRowsW + chunk * 8), val);
          }
        }
        named_bar(2 + h, 128);
      }
    } else if (t.type == TK_GU && p.direct) {
      // Direct mode: the accumulator's columns are the call's T tokens.  The
      // activations of all of them go to shared memory, then each chunk row
      // takes its own token's.
      __nv_bfloat16* SA = reinterpret_cast<__nv_bfloat16*>(simt + kGatherOff);  // [kTB][64]
      const int ncbt = (p.T + 15) >> 4;
      for (int cb = h; cb < ncbt; cb += 2) {
        float v[16];
        tmem_ld16(tbase + cb * 16, v);
        if (q >= 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) U[((q - 2) * 16 + i) * 32 + lane] = v[i];
        }
        named_bar(2 + h, 128);
        if (q < 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gte = v[i];
            const float up = U[(q * 16 + i) * 32 + lane];
            SA[(cb * 16 + i) * 64 + 32 * q + lane] = __float2bfloat16_rn(silu(gte) * up);
          }
        }
        named_bar(2 + h, 128);
      }
      named_bar(1, kNumWorkers);
      for (int idx = wt; idx < t.rows * 8; idx += kNumWorkers) {
        const int i = idx >> 3, chunk = idx & 7;
        const int tok = s_dtok[i];
        const uint4 val = *reinterpret_cast<const uint4*>(SA + tok * 64 + chunk * 8);
        store_act(p, reinterpret_cast<uint4*>(p.ws.act + static_cast<size_t>(t.row0 + i) * p.I +
                                              t.b * kGuRows + chunk * 8), val);
      }
    } else if (t.type == TK_GU) {
      for (int cb = h; cb < ncb; cb += 2) {
        float v[16];
        tmem_ld16(tbase + cb * 16, v);
        if (q >= 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) U[((q - 2) * 16 + i) * 32 + lane] = v[i];
        }
        named_bar(2 + h, 128);
        if (q < 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gte = v[i];
            const float up = U[(q * 16 + i) * 32 + lane];
            const float a = silu(gte) * up;
            S[i * 64 + 32 * q + lane] = __float2bfloat16_rn(a);
          }
        }
        named_bar(2 + h, 128);
        const int tok = cb * 16 + (i128 >> 3), chunk = i128 & 7;
        if (tok < t.rows) {
          const uint4 val = *reinterpret_cast<const uint4*>(S + (i128 >> 3) * 64 + chunk * 8);
          const int gcol = p.pair ? t.b * 2 * kGuRows + kGuRows * rank : t.b * kGuRows;
          store_act(p, reinterpret_cast<uint4*>(p.ws.act + static_cast<size_t>(t.row0 + tok) * p.I +
                                                gcol + chunk * 8), val);
        }
        named_bar(2 + h, 128);
      }
    } else {
      // Down tile: TMEM lane = output column, TMEM column = chunk row.  Each
      // quad of lanes transposes its 4 x 4 blocks in registers, so that a
      // lane holds 4 consecutive output columns of one row and one warp
      // instruction writes 4 rows x 128 bytes; no shared-memory staging.
      // The two worker halves take alternate 16-row blocks (wide tiles: of
      // both 128-column halves of the accumulator); the next block's TMEM
      // load is in flight while one is written.  Weighted combine fused
      // here: out[token] += w * y (fp32 reductions).  The ordered combine
      // stores y; the dense MLP's tile owns its output rows and stores them.
      const int nhalf = p.wide ? 2 : 1;
      const int nmy = (ncb - h + 1) >> 1, nblk = nhalf * nmy;
      const int cq = 32 * q + 4 * (lane >> 2), rq = lane & 3;
      float* accr = fused_comb ? acc_rows(p, t.blk) : nullptr;
      auto taddr = [&](int b) {
        const int hf = b / nmy;
        return tbase + hf * (kAccCols / 2) + (h + 2 * (b - hf * nmy)) * 16;
      };
      auto put = [&](uint32_t(&r)[16], int b) {
        const int hf = b / nmy, cb = h + 2 * (b - hf * nmy);
        const int col = (p.pair ? t.b * kDnRowsW + kDnRows * rank
                                : t.b * (p.wide ? kDnRowsW : kDnRows) + hf * 128) + cq;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
        quad_transpose16(v, lane);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int rr = cb * 16 + 4 * g + rq;
          if (rr < t.rows) {
            const float4 val = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
            if (fused_comb) {
              const float wr = s_rw[rr];
              const int tok = s_rtok[rr];
              if (tok >= 0)
                red_add_v4(accr + static_cast<size_t>(tok) * p.H + col,
                           make_float4(wr * val.x, wr * val.y, wr * val.z, wr * val.w));
            } else if (p.ordered) {
              // ordered combine: the expert row y itself, in expert-sorted order
              *reinterpret_cast<float4*>(p.ws.yperm + static_cast<size_t>(t.pad + rr) * p.H + col) = val;
            } else {
              const size_t o = static_cast<size_t>(t.row0 + rr) * p.H + col;
              if (p.out_bf16) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(val.x, val.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(val.z, val.w);
                uint2 pk;
                pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + o), pk);
              } else {
                __stcs(reinterpret_cast<float4*>(static_cast<float*>(p.out) + o), val);
              }
            }
          }
        }
      };
      uint32_t ra[16], rb[16];
      if (nblk > 0) tmem_ld16_issue(taddr(0), ra);
      for (int b = 0; b < nblk; b += 2) {
        tmem_ld_wait(ra);
        if (b + 1 < nblk) tmem_ld16_issue(taddr(b + 1), rb);
        put(ra, b);
        if (b + 1 < nblk) {
          tmem_ld_wait(rb);
          if (b + 2 < nblk) tmem_ld16_issue(taddr(b + 2), ra);
          put(rb, b + 1);
        }
      }
    }
  }
  fence_proxy_async_global();  // act is read next by TMA
  tc_fence_before();
  named_bar(1, kNumWorkers);  // notify: ev_act / ev_down (by the notifier warp)
  if (wt == 0) release_acc<PAIR>(c, acc);
}

// ---------------------------------------------------------------------------
// Notifier warp: takes each finished task from the workers and performs its
// notify (and, in dynamic mode, the early push of the tasks it makes ready),
// so that the fence and atomic latency stays off the workers' path.
// ---------------------------------------------------------------------------
__device__ void hand_over(Ctrl* c, uint32_t& nit, const Task& t, const Clock& clk) {
  const int s = nit % kNoti;
  if (mbar_wait(&c->nempty[s], ((nit / kNoti) & 1) ^ 1, clk, 260)) {
    c->noti[s] = t;
    mbar_arrive(&c->nfull[s]);
  }
  ++nit;
}

// Warp-wide push: lane 0 reserves n slots, every lane writes some of them.
template <class DescOf>
__device__ void queue_push_warp(const QueueView& q, int n, DescOf desc_of, const Clock& c,
                                int lane) {
  int base = 0;
  if (lane == 0) base = q.n_seed + atom_add_relaxed(q.tail, n);
  base = __shfl_sync(0xffffffffu, base, 0);
  __threadfence();
  for (int i = lane; i < n; i += 32) {
    const int idx = base + i;
    if (idx >= q.cap) {
      raise_error(c, DERR_QUEUE_OVERFLOW, 1, idx);
      break;
    }
    st_relaxed_u64(&q.slots[idx], (static_cast<unsigned long long>(q.epoch) << 32) | desc_of(i));
  }
}

// Phase A of a notify: the one counter or flag a finished task updates,
// issued by one lane per record so that a batch costs one round trip.
// Returns whether the update completed the event (when that matters).
__device__ __forceinline__ int notify_primary(const MegaParams& p, const Task& t) {
  const BlockWs& B = p.ws.blk[t.blk];
  const bool dyn = dynamic_mode(p);
  switch (t.type) {
    case TK_NORM:
      st_relaxed(reinterpret_cast<int*>(&B.norm_flag[t.a]), static_cast<int>(p.epoch));
      return 0;
    case TK_ROUTER:
      if (p.NC == 1) {  // block tb routed (top-k ran in the router task)
        if (!dyn) {
          red_add_relaxed(B.ev_route, 1);
          return 0;
        }
        return atom_add_acq_rel(B.ev_route, 1) + 1 == p.ev_mul * p.nbp;
      }
      // partial logits of block tb landed ("ij->i" on ev_rblk)
      if (!dyn) {
        red_add_relaxed(&B.ev_rblk[t.a], 1);
        return 0;
      }
      return atom_add_acq_rel(&B.ev_rblk[t.a], 1) + 1 == p.ev_mul * p.NC;
    case TK_TOPK:
      st_relaxed(&B.ev_rblk[t.a], 0);  // consumed: re-armed for the next call
      if (p.fuse_scan) return 0;       // the task ran the scan itself
      if (!dyn) {
        red_add_relaxed(B.ev_route, 1);
        return 0;
      }
      return atom_add_acq_rel(B.ev_route, 1) + 1 == p.ev_mul * p.nbp;
    case TK_GU:
      if (p.dense) {  // count-up chunk counters (no scan to arm them)
        if (!tiles_queued(p)) {
          red_add_relaxed(&B.ev_act[t.a], 1);
          return 0;
        }
        return atom_add_acq_rel(&B.ev_act[t.a], 1) + 1 == dense_gu_target(p, t.a);
      }
      if (!tiles_queued(p)) {
        red_add_relaxed(&B.ev_act[t.a], -1);
        return 0;
      }
      return notify(&B.ev_act[t.a], 1) == 0;
    case TK_DN:  // both modes need to know which tile finished the chunk
      if (p.dense) return atom_add_acq_rel(&B.ev_down[t.a], 1) + 1 == p.ev_mul * p.NT_dn;
      return notify(&B.ev_down[t.a], 1) == 0;
    case TK_COMB:
      if (p.use_norm) st_relaxed(reinterpret_cast<int*>(&B.comb_flag[t.a]), static_cast<int>(p.epoch));
      return 0;
    default:
      return 0;
  }
}

// Phase B: what follows from the primary update, warp-wide.
__device__ void notify_follow(const MegaParams& p, Ctrl* c, const Task& t, int fire, int lane,
                              const Clock& clk) {
  const BlockWs& B = p.ws.blk[t.blk];
  const bool dyn = dynamic_mode(p);
  const QueueView q = queue_of(p);
  const unsigned full = 0xffffffffu;
  switch (t.type) {
    case TK_NORM:
      if (dyn) queue_push_warp(q, p.NC, [&](int i) { return task_enc(TK_ROUTER, t.blk, t.a, i); }, clk, lane);
      break;
    case TK_ROUTER:
      if (fire)
        queue_push_warp(q, 1, [&](int) {
          return p.NC == 1 ? task_enc(TK_SCAN, t.blk, 0, 0) : task_enc(TK_TOPK, t.blk, t.a, 0);
        }, clk, lane);
      break;
    case TK_TOPK:
      if (fire && !p.fuse_scan)
        queue_push_warp(q, 1, [&](int) { return task_enc(TK_SCAN, t.blk, 0, 0); }, clk, lane);
      break;
    case TK_PERM: {  // rows of expert e landed: ev_expert[e] -= rows of this block part
      // Lane l owns experts kEL*l .. kEL*l + kEL-1: their notifies go out
      // together, then the tiles of [exp_indptr[e], exp_indptr[e+1]) of every
      // expert this part completed are pushed under one queue reservation, in
      // expert order (the order the static walk takes them, so that tiles of
      // one expert run side by side and share its weights in L2).
      constexpr int kEL = kMaxE / 32;
      const int tb = my_tb(p, t.a);
      if (tb >= p.nb) break;  // the odd CTA's half of the last pair block holds no tokens
      int n[kEL], tiles[kEL], c0[kEL];
#pragma unroll
      for (int i = 0; i < kEL; ++i) {
        const int e = kEL * lane + i;
        n[i] = e < p.E ? __ldcg(B.part_cnt + (tb * p.PP + t.b) * p.E + e) : 0;
      }
      int mine = 0;
#pragma unroll
      for (int i = 0; i < kEL; ++i) {
        tiles[i] = 0;
        if (n[i] > 0) {
          const int e = kEL * lane + i;
          if (!tiles_queued(p)) {
            red_add_relaxed(&B.ev_expert[e], -n[i]);
          } else if (notify(&B.ev_expert[e], n[i]) == 0) {
            c0[i] = __ldcg(B.chunk_indptr + e);
            tiles[i] = ((__ldcg(B.counts + e) + p.cw - 1) / p.cw) * p.NT_gu;
            mine += tiles[i];
          }
        }
      }
      if (!tiles_queued(p)) break;
      int off = mine;  // inclusive prefix over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(full, off, o);
        if (lane >= o) off += y;
      }
      const int total = __shfl_sync(full, off, 31);
      if (total == 0) break;
      int base = 0;
      if (lane == 0) base = q.n_seed + atom_add_relaxed(q.tail, total);
      base = __shfl_sync(full, base, 0) + off - mine;
      __threadfence();  // what the notifies acquired is published with the slots
      const int NT = p.NT_gu;
#pragma unroll
      for (int i = 0; i < kEL; ++i) {
        for (int j = 0; j < tiles[i]; ++j, ++base) {
          if (base >= q.cap) {
            raise_error(clk, DERR_QUEUE_OVERFLOW, 2, base);
            break;
          }
          st_relaxed_u64(&q.slots[base], (static_cast<unsigned long long>(q.epoch) << 32) |
                                              task_enc(TK_GU, t.blk, c0[i] + j / NT, j % NT));
        }
      }
      break;
    }
    case TK_GU:
      if (fire) queue_push_warp(q, p.NT_dn, [&](int i) { return task_enc(TK_DN, t.blk, t.a, i); }, clk, lane);
      break;
    case TK_DN:
      if (p.dense) {
        // Last down tile of the chunk: every tile of the chunk has passed its
        // wait, so both counters go back to 0 for the next call.
        if (fire && lane == 0) {
          st_relaxed(&B.ev_act[t.a], 0);
          st_relaxed(&B.ev_down[t.a], 0);
        }
        break;
      }
      if (fire && needs_comb(p, t.blk)) {
        // Finisher of the chunk: notify each token block by its number of rows.
        // The chunk's rows are in ascending token order, so blocks form runs;
        // each lane takes a contiguous range of rows and notifies its runs (a
        // run split between lanes is notified in two parts).
        const int per = (t.rows + 31) / 32, r0 = min(t.rows, lane * per), r1 = min(t.rows, r0 + per);
        int run_tb = -1, run_n = 0;
        auto flush_run = [&]() {
          if (run_n == 0) return;
          if (!tiles_queued(p)) {
            red_add_relaxed(&B.ev_tok[run_tb], -run_n);
          } else if (notify(&B.ev_tok[run_tb], run_n) == 0) {
            queue_push(q, 1, [&](int) { return task_enc(TK_COMB, t.blk, run_tb, 0); }, clk);
          }
        };
        const int tbw = p.pair ? 2 * kTB : kTB;  // rows of a (pair) token block
        for (int r = r0; r < r1; ++r) {
          const int tb = __ldcg(B.row_token + t.pad + r) / tbw;
          if (tb != run_tb) {
            flush_run();
            run_tb = tb;
            run_n = 0;
          }
          ++run_n;
        }
        flush_run();
        __syncwarp();
      }
      break;
    case TK_COMB:
      if (dyn && t.blk + 1 < p.n_blocks)
        queue_push_warp(q, 1, [&](int) { return task_enc(TK_NORM, t.blk + 1, t.a, 0); }, clk, lane);
      break;
    default:
      break;
  }
}

// Takes the finished tasks in batches of up to 8: one fence for the batch,
// the primary updates in parallel (one lane per task), then the follow-ups.
__device__ void run_notifier(const MegaParams& p, Ctrl* c, const Clock& clk) {
  const int lane = lane_id();
  const unsigned full = 0xffffffffu;
  uint32_t nit = 0;
  bool done = false;
  while (!done) {
    int n = 0;
    if (lane == 0) {
      if (mbar_wait(&c->nfull[nit % kNoti], (nit / kNoti) & 1, clk, 250)) {
        n = 1;
        while (n < kNoti && mbar_try_wait(&c->nfull[(nit + n) % kNoti], ((nit + n) / kNoti) & 1)) ++n;
      } else {
        n = -1;
      }
    }
    n = __shfl_sync(full, n, 0);
    if (n < 0) break;
    __syncwarp();
    // Records up to (not including) a TERM are handled; TERM ends the loop.
    int m = n;
    for (int i = 0; i < n; ++i)
      if (c->noti[(nit + i) % kNoti].type == TK_TERM) {
        m = i;
        done = true;
        break;
      }
    __threadfence();  // the workers' writes (ordered by the mbarrier) precede the notifies
    int fire = 0;
    if (lane < m) fire = notify_primary(p, c->noti[(nit + lane) % kNoti]);
    for (int i = 0; i < m; ++i) {
      const Task t = c->noti[(nit + i) % kNoti];
      notify_follow(p, c, t, __shfl_sync(full, fire, i), lane, clk);
    }
    __syncwarp();
    if (lane == 0)
      for (int i = 0; i < n; ++i) mbar_arrive(&c->nempty[(nit + i) % kNoti]);
    nit += n;
  }
}

template <bool PAIR>
__device__ void run_workers(const MegaParams& p, Ctrl* c, uint8_t* simt, uint8_t* epi,
                            const Clock& clk) {
  const int wt = threadIdx.x - kWorkerWarp0 * 32;
  uint32_t gemm_i = 0, nit = 0, perm_li = 0;
  for (uint32_t ri = 0;; ++ri) {
    Task* slot = &c->wtask[ri & 1];
    if (wt == 0) {
      const int r = ri % kRing;
      if (mbar_wait(&c->rfull[r], (ri / kRing) & 1, clk, 210)) {
        *slot = c->ring[r];
        *reinterpret_cast<volatile int*>(&c->started) = static_cast<int>(ri + 1);
      } else {
        slot->type = TK_TERM;
      }
      mbar_arrive(&c->rempty[r]);
    }
    named_bar(1, kNumWorkers);
    const Task t = *slot;
    const unsigned long long t_start = p.ws.trace ? globaltimer_ns() : 0;
    switch (t.type) {
      case TK_NORM: task_norm(p, t, wt); break;
      case TK_ROUTER:
        if (p.logits_in) task_topk(p, t, simt, wt);
        else task_router_epilogue<PAIR>(p, c, simt, t, gemm_i, clk, wt, ri);
        break;
      case TK_TOPK: task_topk(p, t, simt, wt); break;
      case TK_SCAN:  // pair tiles: the even CTA of the pair runs it
        if (pair_rank(p) == 0) task_scan(p, t, simt, wt);
        break;
      case TK_PERM: task_perm(p, c, t, simt, wt, perm_li, clk); break;
      case TK_GU:
      case TK_DN: task_gemm_epilogue<PAIR>(p, c, epi, simt, t, gemm_i, clk, wt, ri); break;
      case TK_COMB: task_comb(p, t, simt, wt); break;
      default: break;
    }
    // Every task ends with a barrier of the 256 workers: its writes are done.
    if (wt == 0 && t.type != TK_SCAN) hand_over(c, nit, t, clk);
    if (t.type == TK_TERM) break;
    if (p.ws.trace && wt == 0) {
      const int idx = static_cast<int>(atomicAdd(p.ws.trace, 1ull));
      if (idx < p.ws.trace_cap) {
        unsigned long long* r = p.ws.trace + 1 + 4 * static_cast<size_t>(idx);
        r[0] = (static_cast<unsigned long long>(t.type) << 56) |
               (static_cast<unsigned long long>(t.blk) << 48) |
               (static_cast<unsigned long long>(blockIdx.x) << 32) |
               (static_cast<unsigned long long>(t.a) << 8) | static_cast<unsigned long long>(t.b & 0xFF);
        r[1] = t.t_disp;
        r[2] = t_start;
        r[3] = globaltimer_ns();
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA producer and tcgen05 issuer
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ring_take(Ctrl* c, uint32_t& ri, Task& t, const Clock& clk,
                                          int where) {
  const int r = ri % kRing;
  const bool ok = mbar_wait(&c->rfull[r], (ri / kRing) & 1, clk, where);
  if (ok) t = c->ring[r];
  mbar_arrive(&c->rempty[r]);
  ++ri;
  return ok;
}

template <bool PAIR>
__device__ void run_producer(const MegaParams& p, Ctrl* c, uint8_t* base, const Clock& clk) {
  uint32_t ri = 0, ph = 0;  // stage slot and its phase, advanced without division
  int st = 0;
  const StageGeom g = stage_geom(p);
  // Pair tiles: each CTA loads its half of the operands into its own stages;
  // every copy completes on the even CTA's `full` barrier, where the pair MMA
  // waits, and the even CTA's producer announces both CTAs' bytes.
  constexpr bool pair = PAIR;
  const int rank = pair_rank(p);
  const bool announce = !pair || rank == 0;
  const uint32_t tx_mul = pair ? 2u : 1u;
  auto load = [&](void* dst, const CUtensorMap* m, int s, int x, int y) {
    if constexpr (PAIR) tma_load_2d_pair(dst, m, mapa_shared(&c->full[s], 0), x, y);
    else tma_load_2d(dst, m, &c->full[s], x, y);
  };
  auto load3 = [&](void* dst, const CUtensorMap* m, int s, int x, int y, int z) {
    if constexpr (PAIR) tma_load_3d_pair(dst, m, mapa_shared(&c->full[s], 0), x, y, z);
    else tma_load_3d(dst, m, &c->full[s], x, y, z);
  };
  for (;;) {
    Task t;
    if (!ring_take(c, ri, t, clk, 220) || t.type == TK_TERM) break;
    if (t.type == TK_ROUTER && !p.logits_in) {
      // Router tile: per 64-row K block of H, the router weight's rows for
      // experts 0-63 and 64-127 (two MN-major boxes; experts >= E read as
      // zero) and the block's 32 input rows (the lo part second in the chain).
      // Pair tiles: both CTAs load the router weight, each its own 32 rows.
      // Stages large enough for two K blocks (wide geometry) take two: twice
      // the bytes in flight for a tile whose weight operand is the same
      // 512 KB for every token block.
      const int KB = p.KBr * (p.use_norm ? 2 : 1);
      const uint32_t bytes = kOpABytes + kTB * kBK * 2;  // two 64-expert boxes + 32 token rows
      const int per = router_kpack(g);
      const int tok0 = my_tb(p, t.a) * kTB;
      fence_proxy_async_global();
      for (int kb0 = 0; kb0 < KB; kb0 += per, st = st + 1 == g.n ? (ph ^= 1, 0) : st + 1) {
        const int s = st;
        if (!mbar_wait(&c->empty[s], ph ^ 1, clk, 222, pair)) return;
        uint8_t* sa = base + s * g.bytes;
        const int nk = min(per, KB - kb0);
        if (announce) mbar_arrive_expect_tx(&c->full[s], nk * bytes * tx_mul);
        for (int u = 0; u < nk; ++u) {
          const int kb = kb0 + u;
          const int part = kb >= p.KBr ? 1 : 0;
          const int h = t.b * p.HC + (kb - part * p.KBr) * kBK;
          load(sa + u * kOpABytes, &p.tm_wg[t.blk], s, 0, h);
          load(sa + u * kOpABytes + kOpABytes / 2, &p.tm_wg[t.blk], s, 64, h);
          load(sa + g.boff + u * (kTB * kBK * 2), part ? &p.tm_xrlo : &p.tm_xr, s, h, tok0);
        }
      }
      continue;
    }
    if (t.type != TK_GU && t.type != TK_DN) continue;
    const bool gu = t.type == TK_GU;
    const CUtensorMap* ta = gu ? &p.tm_wgu[t.blk] : &p.tm_wd[t.blk];
    // token operand: x_perm rows (a heavy expert's: x rows) for gate/up, act rows for down
    const bool heavy_x = gu && t.pad < 0;
    const CUtensorMap* tb = !gu ? &p.tm_act : heavy_x ? &p.tm_xh : &p.tm_xperm;
    const CUtensorMap* tb128 = !gu ? &p.tm_act128 : heavy_x ? &p.tm_xh128 : &p.tm_xperm128;
    const int src0 = !gu ? t.row0 : heavy_x ? -1 - t.pad : t.pad;
    const int KB = (gu ? p.H : p.I) / kBK;
    // Token rows of this CTA: the whole chunk, or its half of a pair tile
    // (the MMA takes rows [0, npad/2) from the even CTA, the rest from the odd).
    const int half = pair ? pair_npad(t.rows) / 2 : 0;
    const int brow0 = pair ? src0 + rank * half : src0;
    const int nb16 = pair ? half >> 4 : (t.rows + 15) >> 4;
    const int n128 = nb16 >> 3, r16 = nb16 & 7;  // token rows as 128-row boxes, then 16-row boxes
    // Weight rows, one box per K step.  Gate/up: R gate rows and the R up
    // rows beside them (3-D box, gate block then up block): R = 64 narrow (one
    // M=128 operand) and pair (this CTA's half of the 128 intermediate
    // columns), 128 wide (two operands).  Down tiles: 128 (wide: 256)
    // consecutive output rows of w_down.
    const bool wide = p.wide != 0;
    const int nA = wide ? 4 : 2;  // 64-row weight blocks per K step
    const int i0 = gu ? (pair ? t.b * 2 * kGuRows + kGuRows * rank : t.b * (wide ? kGuRowsW : kGuRows)) : 0;
    const int r0 = gu ? 0 : t.e * p.H + (pair ? t.b * kDnRowsW + kDnRows * rank : t.b * (wide ? kDnRowsW : kDnRows));
    // Direct mode: a gate/up tile's token operand is all T (<= 32) rows of x,
    // one 32-row box (rows past T read as zero).
    const bool direct_x = gu && p.direct;
    const uint32_t bytes = nA * (kOpABytes / 2) + (direct_x ? kTB : nb16 * 16) * kBK * 2;
    fence_proxy_async_global();
    for (int kb = 0; kb < KB; ++kb, st = st + 1 == g.n ? (ph ^= 1, 0) : st + 1) {
      const int s = st;
      if (!mbar_wait(&c->empty[s], ph ^ 1, clk, 221, pair)) return;
      uint8_t* sa = base + s * g.bytes;
      uint8_t* sb = sa + g.boff;
      if (announce) mbar_arrive_expect_tx(&c->full[s], bytes * tx_mul);
      if (gu) load3(sa, ta, s, kb * kBK, i0, 2 * t.e);
      else load(sa, ta, s, kb * kBK, r0);
      if (direct_x) {
        load(sb, &p.tm_xr, s, kb * kBK, 0);
        continue;
      }
      for (int i = 0; i < n128; ++i) load(sb + i * 128 * kBK * 2, tb128, s, kb * kBK, brow0 + 128 * i);
      for (int i = 0; i < r16; ++i)
        load(sb + (n128 * 128 + i * 16) * kBK * 2, tb, s, kb * kBK, brow0 + n128 * 128 + 16 * i);
    }
  }
}

// PAIR (a compile-time copy of p.pair): a kernel uses tcgen05 with one CTA
// group only, so the pair and single-CTA issuers are separate instantiations.
template <bool PAIR>
__device__ void run_mma(const MegaParams& p, Ctrl* c, uint8_t* base, const Clock& clk) {
  uint32_t ri = 0, tc = 0, ph = 0;  // stage slot and its phase, advanced without division
  int st = 0;
  const StageGeom g = stage_geom(p);
  const uint32_t tmem = c->tmem_base;
  // Pair tiles: the even CTA's issuer runs every MMA of the pair; the odd
  // CTA's only keeps its place in the task ring.
  constexpr bool pair = PAIR;
  const bool issuer = !pair || pair_rank(p) == 0;
  for (;;) {
    Task t;
    if (!ring_take(c, ri, t, clk, 240) || t.type == TK_TERM) break;
    const bool rt = t.type == TK_ROUTER && !p.logits_in;
    if (!issuer || (!rt && t.type != TK_GU && t.type != TK_DN)) continue;
    const int acc = tc & 1;
    if (!mbar_wait(&c->tempty[acc], ((tc >> 1) & 1) ^ 1, clk, 241, pair)) return;
    tc_fence_after();
    const uint32_t d = tmem + acc * kAccCols;
    // N = token columns: the 32-token router block (64 over a pair), the
    // chunk rounded to 16 (a pair's chunk rounded to 32).
    // (direct mode: a gate/up tile's columns are all T tokens)
    const int ncol = (t.type == TK_GU && p.direct) ? p.T : t.rows;
    const int npad = rt ? (pair ? 2 * kTB : kTB) : pair ? pair_npad(ncol) : (ncol + 15) & ~15;
    const int M = pair ? 256 : 128;
    // Token-major wide tiles: M = 128 token rows (rows past the chunk are
    // don't-care lanes), N = the 256 weight rows.
    const bool tmaj = !rt && tile_tokmaj(p, t);
    // Router tiles read A (the router weight) MN-major; expert tiles K-major.
    const uint32_t idesc = rt     ? idesc_bf16_f32_amn(M, npad)
                           : tmaj ? idesc_bf16_f32(128, 2 * kGuRowsW)
                                  : idesc_bf16_f32(M, npad);
    const int KB = rt ? p.KBr * (p.use_norm ? 2 : 1) : (t.type == TK_GU ? p.H : p.I) / kBK;
    const int per = rt ? router_kpack(g) : 1;  // K blocks per stage
    for (int kb = 0; kb < KB; kb += per, st = st + 1 == g.n ? (ph ^= 1, 0) : st + 1) {
      const int s = st;
      if (!mbar_wait(&c->full[s], ph, clk, 242, pair)) return;
      tc_fence_after();
      const uint32_t sa = smem_u32(base + s * g.bytes);
      const uint64_t bd = desc_kmajor_sw128(sa + g.boff);
      if constexpr (PAIR) {
        // 128 weight rows from each CTA, npad/2 token rows from each.
        const uint64_t ad = rt ? desc_mnmajor_sw128(sa, kOpABytes / 2) : desc_kmajor_sw128(sa);
        const uint64_t astep = rt ? (2048 >> 4) : 2;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16_pair(d, ad + astep * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
        umma_commit_pair(&c->empty[s]);  // both CTAs' stages free once these MMAs have read them
        continue;
      } else if (rt) {
        // 16 K rows per MMA: 2 KB further into each 64-expert box; the
        // stage's second K block (if any) 16 KB (weight) and 4 KB (tokens) on.
        const int nk = min(per, KB - kb);
        for (int u = 0; u < nk; ++u) {
          const uint64_t ad = desc_mnmajor_sw128(sa + u * kOpABytes, kOpABytes / 2);
          const uint64_t bdu = desc_kmajor_sw128(sa + g.boff + u * (kTB * kBK * 2));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d, ad + kk * (2048 >> 4), bdu + 2 * kk, idesc, (kb | u | kk) != 0 ? 1u : 0u);
        }
      } else if (tmaj) {
        // A = the token rows (the stage's token part), B = all 256 weight rows
        const uint64_t ta = desc_kmajor_sw128(sa + g.boff), wb = desc_kmajor_sw128(sa);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16(d, ta + 2 * kk, wb + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
      } else {
        const uint64_t ad = desc_kmajor_sw128(sa);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
        if (p.wide) {  // second 128 weight rows into the buffer's second half
          const uint64_t ad1 = desc_kmajor_sw128(sa + kOpABytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d + kAccCols / 2, ad1 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
      }
      if constexpr (!PAIR) umma_commit(&c->empty[s]);  // stage free once these MMAs have read it
    }
    if constexpr (PAIR) umma_commit_pair(&c->tfull[acc]);  // accumulator ready in both CTAs
    else umma_commit(&c->tfull[acc]);                      // accumulator ready
    ++tc;
  }
}

// ---------------------------------------------------------------------------
// Scheduler
// ---------------------------------------------------------------------------
struct RingWriter {
  Ctrl* c;
  uint32_t i;
  __device__ bool emit(const Task& t, const Clock& clk) {
    const int r = i % kRing;
    if (!mbar_wait(&c->rempty[r], ((i / kRing) & 1) ^ 1, clk, 200)) return false;
    c->ring[r] = t;
    c->ring[r].t_disp = globaltimer_ns();
    mbar_arrive(&c->rfull[r]);
    ++i;
    return true;
  }
};

__device__ __forceinline__ Task make_task(int type, int blk, int a, int b) {
  Task t;
  t.type = type;
  t.blk = blk;
  t.a = a;
  t.b = b;
  t.e = t.row0 = t.rows = t.pad = 0;
  return t;
}

__device__ __forceinline__ void resolve_chunk(const MegaParams& p, Task& t) {
  if (p.dense) {  // chunk a = rows [cw*a, min(cw*a + cw, T)) of x
    t.e = 0;
    t.row0 = t.a * p.cw;
    t.rows = min(p.cw, p.T - t.row0);
    t.pad = t.row0;
    return;
  }
  const BlockWs& B = p.ws.blk[t.blk];
  t.e = __ldcg(B.chunk_expert + t.a);
  t.row0 = __ldcg(B.chunk_row0 + t.a);
  t.rows = __ldcg(B.chunk_rows + t.a);
  t.pad = __ldcg(B.chunk_src + t.a);
}

// Dense MLP gate/up tile g of a call: groups of kGc chunks, each group taken
// weight-slice major.  The tiles that run side by side share a slice or two
// of w_gate_up (read from HBM once per group) and read only the group's rows
// of x (32 MB at H = 4096), which stay in L2; walking all of x at once
// (67 MB at H = 4096) had x re-read from HBM for every slice.
__device__ __forceinline__ Task dense_gu_task(const MegaParams& p, int g) {
  const int kGc = p.pair ? 16 : 32;  // chunks per group (4096 rows of x)
  const int per_group = kGc * p.NT_gu, grp = g / per_group, w = g - grp * per_group;
  const int c0 = grp * kGc, gs = min(kGc, p.n_chunks - c0);
  Task t = make_task(TK_GU, 0, c0 + w % gs, w / gs);
  resolve_chunk(p, t);
  return t;
}

// Static walk of the dense MLP: gate/up tiles (no input event), then the down
// tiles chunk by chunk, each after its chunk's gate/up tiles (count-up event).
__device__ bool sched_static_dense(const MegaParams& p, Ctrl* c, const Clock& clk, RingWriter& rw) {
  const int G = sched_units(p), cta = sched_unit(p);
  const BlockWs& B = p.ws.blk[0];
  bool ok = true;
  if (p.stage_lo <= TK_GU && p.stage_hi >= TK_GU)
    for (int g = cta; g < p.n_chunks * p.NT_gu && ok; g += G) ok = rw.emit(dense_gu_task(p, g), clk);
  if (p.stage_lo <= TK_DN && p.stage_hi >= TK_DN)
    for (int d = cta; d < p.n_chunks * p.NT_dn && ok; d += G) {
      Task t = make_task(TK_DN, 0, d / p.NT_dn, d % p.NT_dn);
      ok = wait_geq(&B.ev_act[t.a], dense_gu_target(p, t.a), clk, TK_DN, t.a);
      resolve_chunk(p, t);
      ok = ok && rw.emit(t, clk);
    }
  return ok;
}

// Static walk.  routing_only (MIXED): the walk stops after each block's
// permute tasks; the expert tiles then come from the queue.  Returns false
// after a failed wait.
__device__ bool sched_static(const MegaParams& p, Ctrl* c, const Clock& clk, RingWriter& rw,
                             bool routing_only) {
  // Pair tiles: both CTAs of a pair walk the same list of pair tasks.
  const int G = sched_units(p), cta = sched_unit(p);
  auto in = [&](int stage) { return stage >= p.stage_lo && stage <= p.stage_hi; };
  bool ok = true;
  for (int blk = 0; blk < p.n_blocks && ok; ++blk) {
    const BlockWs& B = p.ws.blk[blk];
    if (p.use_norm && in(TK_NORM)) {
      for (int tb = cta; tb < p.nb && ok; tb += G) {
        if (blk > 0) ok = wait_flag(&p.ws.blk[blk - 1].comb_flag[tb], p.epoch, clk, TK_NORM, tb);
        ok = ok && rw.emit(make_task(TK_NORM, blk, tb, 0), clk);
      }
    }
    if (in(TK_ROUTER)) {
      for (int i = cta; i < p.n_router && ok; i += G) {
        const int tb = i / p.NC;
        if (p.use_norm) ok = wait_flag(&B.norm_flag[tb], p.epoch, clk, TK_ROUTER, tb);
        ok = ok && rw.emit(make_task(TK_ROUTER, blk, tb, i % p.NC), clk);
      }
    }
    if (in(TK_TOPK) && p.NC > 1) {
      for (int tb = cta; tb < p.nbp && ok; tb += G) {
        ok = wait_geq(&B.ev_rblk[tb], p.ev_mul * p.NC, clk, TK_TOPK, tb);
        ok = ok && rw.emit(make_task(TK_TOPK, blk, tb, 0), clk);
      }
    }
    if (in(TK_SCAN) && !p.fuse_scan && cta == blk % G && ok) {
      ok = wait_geq(B.ev_route, p.ev_mul * p.nbp, clk, TK_SCAN, 0);
      ok = ok && rw.emit(make_task(TK_SCAN, blk, 0, 0), clk);
    }
    if (p.stage_hi < TK_PERM || !ok) continue;
    ok = wait_flag(B.plan_flag, p.epoch, clk, TK_PERM, 0);
    if (!ok) break;
    const int n_chunks = ld_acquire(&B.meta[0]);
    if (in(TK_PERM) && !p.direct)
      for (int i = cta; i < p.nbp * p.PP && ok; i += G)
        ok = rw.emit(make_task(TK_PERM, blk, i / p.PP, i % p.PP), clk);
    if (routing_only) continue;
    if (in(TK_GU)) {
      const int n = n_chunks * p.NT_gu;
      for (int g = cta; g < n && ok; g += G) {
        Task t = make_task(TK_GU, blk, g / p.NT_gu, g % p.NT_gu);
        resolve_chunk(p, t);
        ok = wait_zero(&B.ev_expert[t.e], clk, TK_GU, t.e);
        ok = ok && rw.emit(t, clk);
      }
    }
    if (in(TK_DN)) {
      const int n = n_chunks * p.NT_dn;
      for (int d = cta; d < n && ok; d += G) {
        Task t = make_task(TK_DN, blk, d / p.NT_dn, d % p.NT_dn);
        ok = wait_zero(&B.ev_act[t.a], clk, TK_DN, t.a);
        if (ok) resolve_chunk(p, t);
        ok = ok && rw.emit(t, clk);
      }
    }
    if (in(TK_COMB) && needs_comb(p, blk)) {
      for (int tb = cta; tb < p.nbp && ok; tb += G) {
        ok = wait_zero(&B.ev_tok[tb], clk, TK_COMB, tb);
        ok = ok && rw.emit(make_task(TK_COMB, blk, tb, 0), clk);
      }
    }
  }
  return ok;
}

// Pair tiles, dynamic queue: the even CTA pops each task and forwards it to
// the odd CTA's mailbox (shared memory written across the pair, completed on
// the peer's mbarrier); the odd CTA's scheduler hands the forwarded tasks to
// its own roles in the same order.
__device__ bool forward_task(Ctrl* c, uint32_t& fi, const Task& t, const Clock& clk) {
  const int s = fi % kMbox;
  if (!mbar_wait(&c->mb_empty[s], ((fi / kMbox) & 1) ^ 1, clk, 205, true)) return false;
  const uint32_t dst = mapa_shared(&c->mbox[s], 1);
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&t);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(Task) / 4); ++i) st_cluster_u32(dst + 4 * i, src[i]);
  mbar_arrive_cluster(mapa_shared(&c->mb_full[s], 1));  // release: the task is visible first
  ++fi;
  return true;
}

__device__ void relay_pair_tasks(Ctrl* c, const Clock& clk, RingWriter& rw) {
  for (uint32_t i = 0;; ++i) {
    const int s = i % kMbox;
    if (!mbar_wait(&c->mb_full[s], (i / kMbox) & 1, clk, 206, true)) break;
    const Task t = c->mbox[s];
    mbar_arrive_cluster(mapa_shared(&c->mb_empty[s], 0));
    if (t.type == TK_TERM || !rw.emit(t, clk)) break;
  }
}

// Queue pops until every task of the call that passes through the queue has
// been popped (the last scan publishes their number).
template <bool PAIR>
__device__ void sched_dynamic(const MegaParams& p, Ctrl* c, const Clock& clk, RingWriter& rw) {
  if constexpr (PAIR) {
    if (pair_rank(p) != 0) {
      relay_pair_tasks(c, clk, rw);
      return;
    }
  }
  const QueueView q = queue_of(p);
  constexpr int kLookahead = 2;  // tasks popped but not yet started by the workers
  uint32_t fi = 0;
  // Hands a task to this CTA's roles (and, with pair tiles, to the peer's).
  auto emit = [&](const Task& t) {
    if constexpr (PAIR) {
      if (!forward_task(c, fi, t, clk)) return false;
    }
    return rw.emit(t, clk);
  };
  for (;;) {
    // Pop only when this CTA is about to need work: a CTA that grabbed many
    // ready tasks would leave other SMs idle.
    const volatile int* started = &c->started;
    if (!spin_until([&] { return static_cast<int>(rw.i) - *started < kLookahead; }, clk,
                    DERR_TIMEOUT_QUEUE, 1, 0))
      break;
    const int idx = atom_add_relaxed(q.head, 1);
    uint32_t desc = 0;
    bool have = false;
    if (idx < q.n_seed && p.dense) {
      if (!emit(dense_gu_task(p, idx))) break;
      continue;
    }
    if (p.dense && idx >= p.q_total) break;  // every task of the call has been popped
    if (idx < q.n_seed) {
      desc = p.use_norm ? task_enc(TK_NORM, 0, idx, 0)
                        : task_enc(TK_ROUTER, 0, idx / p.NC, idx % p.NC);
      have = true;
    } else {
      unsigned long long v = 0;
      const bool got = spin_until(
          [&] {
            if (idx < q.cap) {
              v = ld_acquire(&q.slots[idx]);
              if (static_cast<unsigned>(v >> 32) == p.epoch) return true;
            }
            if (ld_acquire(p.ws.qtotal_flag) == p.epoch && idx >= ld_acquire(p.ws.qtotal)) {
              v = 0;
              return true;
            }
            return false;
          },
          clk, DERR_TIMEOUT_QUEUE, 0, idx);
      if (!got) break;
      if (static_cast<unsigned>(v >> 32) == p.epoch) {
        desc = static_cast<uint32_t>(v);
        have = true;
      }
    }
    if (!have) break;  // every task of the call has been popped
    Task t = make_task(task_type(desc), task_blk(desc), task_a(desc), task_b(desc));
    if (t.type == TK_GU || t.type == TK_DN) resolve_chunk(p, t);
    if (!emit(t)) break;
  }
  if constexpr (PAIR) forward_task(c, fi, make_task(TK_TERM, 0, 0, 0), clk);
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
// PAIR = 1: launched as clusters of two CTAs with pair tiles (p.pair == 1).
template <int PAIR>
__global__ void __launch_bounds__(kThreads, 1) etc_moe_megakernel(const __grid_constant__ MegaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* simt = base + kStageRegion;
  uint8_t* epi = simt;  // shared with the SIMT scratch (one worker task at a time)
  Ctrl* c = reinterpret_cast<Ctrl*>(simt + kWorkerBytes);
  const Clock clk{globaltimer_ns() + p.timeout_ns, p.ws.status, p.ws.status_host};
  const int w = warp_id();
  if (threadIdx.x == 0) {
    c->started = 0;
    for (int s = 0; s < kStagesMax; ++s) {
      mbar_init(&c->full[s], 1);
      mbar_init(&c->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&c->tfull[a], 1);
      mbar_init(&c->tempty[a], PAIR ? 2 : 1);  // pair: the workers of both CTAs release it
    }
    for (int s = 0; s < kMbox; ++s) {
      mbar_init(&c->mb_full[s], 1);
      mbar_init(&c->mb_empty[s], 1);
    }
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&c->rfull[r], 1);
      mbar_init(&c->rempty[r], kRingConsumers);
    }
    for (int s = 0; s < kNoti; ++s) {
      mbar_init(&c->nfull[s], 1);
      mbar_init(&c->nempty[s], 1);
    }
    for (int s = 0; s < kPermSlots; ++s) mbar_init(&c->pbar[s], 1);
    mbar_fence_init();
  }
  if (w == kWarpTma && lane_id() == 0 && p.stage_lo <= TK_ROUTER && !p.logits_in) {
    for (int b = 0; b < p.n_blocks; ++b) tma_prefetch_desc(&p.tm_wg[b]);
    tma_prefetch_desc(&p.tm_xr);
    if (p.use_norm) tma_prefetch_desc(&p.tm_xrlo);
  }
  if (w == kWarpTma && lane_id() == 0 && p.stage_hi >= TK_GU) {
    for (int b = 0; b < p.n_blocks; ++b) {
      tma_prefetch_desc(&p.tm_wgu[b]);
      tma_prefetch_desc(&p.tm_wd[b]);
    }
    tma_prefetch_desc(&p.tm_xperm);
    tma_prefetch_desc(&p.tm_act);
    tma_prefetch_desc(&p.tm_xperm128);
    tma_prefetch_desc(&p.tm_act128);
  }
  if (w == kWarpMma) {
    if constexpr (PAIR) {  // the same columns in both CTAs of the pair
      tmem_alloc_pair(&c->tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c->tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // the peer's barriers are initialised before any use
  tc_fence_after();

  if (w == kWarpSched) {
    if (lane_id() == 0) {
      RingWriter rw{c, 0};
      if (blockIdx.x == 0) {
        // Re-arm the other parity's queue for the next call: the call before
        // this one, which used it, has completed.
        const int other = (p.epoch + 1) & 1;
        *p.ws.qhead[other] = 0;
        *p.ws.qtail[other] = 0;
      }
      if (p.dense && p.mode != ETC_SCHED_DYNAMIC) {
        sched_static_dense(p, c, clk, rw);
      } else if (p.mode == ETC_SCHED_DYNAMIC) {
        sched_dynamic<PAIR != 0>(p, c, clk, rw);
      } else if (p.mode == ETC_SCHED_MIXED) {
        if (sched_static(p, c, clk, rw, true)) sched_dynamic<PAIR != 0>(p, c, clk, rw);
      } else {
        sched_static(p, c, clk, rw, false);
      }
      rw.emit(make_task(TK_TERM, 0, 0, 0), clk);
    }
  } else if (w == kWarpTma) {
    if (lane_id() == 0) run_producer<PAIR != 0>(p, c, base, clk);
  } else if (w == kWarpMma) {
    if (lane_id() == 0) run_mma<PAIR != 0>(p, c, base, clk);
  } else if (w == kWarpNotifier) {
    run_notifier(p, c, clk);
  } else if (w >= kWorkerWarp0) {
    run_workers<PAIR != 0>(p, c, simt, epi, clk);
  }

  tc_fence_before();
  __syncthreads();
  // Pair: neither CTA leaves while the peer may still signal its barriers,
  // read its operands or write its accumulators.
  if constexpr (PAIR) cluster_sync_all();
  if (w == kWarpMma) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(c->tmem_base, kTmemCols);
    else tmem_dealloc(c->tmem_base, kTmemCols);
  }
}

cudaError_t megakernel_configure() {
  cudaError_t e = cudaFuncSetAttribute(etc_moe_megakernel<0>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(etc_moe_megakernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

static cudaLaunchConfig_t launch_config(int grid, bool pair, cudaStream_t stream,
                                        cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: spin-waits are safe
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  return cfg;
}

cudaError_t launch_megakernel(const MegaParams& p, int grid, cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(grid, p.pair != 0, stream, attr);
  if (p.pair) return cudaLaunchKernelEx(&cfg, etc_moe_megakernel<1>, p);
  return cudaLaunchKernelEx(&cfg, etc_moe_megakernel<0>, p);
}

int megakernel_occupancy() {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, etc_moe_megakernel<0>, kThreads,
                                                    kSmemBytes) != cudaSuccess)
    return 0;
  return occ;
}

// CTA pairs that can be resident at once (0 if cluster launches are unavailable).
int megakernel_pair_clusters(int sms) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(2 * (sms / 2), true, nullptr, attr);
  cfg.attrs = &attr[1];  // the cluster shape alone
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, etc_moe_megakernel<1>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace etc
