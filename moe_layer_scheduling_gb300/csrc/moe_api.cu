// moe_api.cu -- plans, workspace and the C ABI of the MoE megakernel.
//
// A plan is created once per weight shape; every per-call quantity (T, the
// token-block count, the router's H split, the call's epoch) is a kernel
// argument, so one compiled kernel serves every token count without
// recompilation or graph capture ("Event Tensor: A Unified Abstraction for
// Compiling Dynamic Megakernel", Figure 4: the symbolic-shape template is
// instantiated per call).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "../../include/etc_moe.h"
#include "etc_host.h"
#include "etc_internal.h"

namespace etc {
int megakernel_occupancy();
int megakernel_pair_clusters(int sms);
}

using namespace etc;

struct etc_plan_s {
  int device = 0;
  etc_moe_opts opts{};
  int H = 0, E = 0, k = 0, I = 0, T_max = 0, n_blocks = 1;
  int grid = 0;
  int pair_grid = 0;          // CTAs of a launch in CTA pairs (0: cluster launches unavailable)
  int nb_max = 0, C_max = 0, R_max = 0;
  int R_act = 0;              // act rows: R_max plus what heavy experts add (up to 20 %)
  long long partial_max = 0;  // max NC * T_pad over T
  std::vector<void*> allocs;
  void* ctrl = nullptr;       // counters, flags, queue heads: cleared by reset
  size_t ctrl_bytes = 0;
  Workspace ws{};
  CUtensorMap tm_xperm{}, tm_act{}, tm_xperm128{}, tm_act128{};
  const void* cached_wgu[kMaxBlocks] = {};
  const void* cached_wd[kMaxBlocks] = {};
  // w_gate_up as [E * 2][I][H] (gate half, then up half of each expert): one
  // box = R gate rows and the R up rows beside them, R = 64 (narrow and pair
  // tiles) or 128 (wide); w_down [E * H][I] with 128-row (wide: 256-row) boxes
  const void* cached_wgu128[kMaxBlocks] = {};
  const void* cached_wd256[kMaxBlocks] = {};
  CUtensorMap tm_wgu[kMaxBlocks]{}, tm_wgu128[kMaxBlocks]{}, tm_wd[kMaxBlocks]{},
      tm_wd256[kMaxBlocks]{};
  const void* cached_wg[kMaxBlocks] = {};
  CUtensorMap tm_wg[kMaxBlocks]{};
  const void* cached_x = nullptr;  // router input map of the caller's x, per (pointer, T)
  int cached_xT = 0;
  CUtensorMap tm_x{};
  const void* cached_xh = nullptr;  // heavy experts' token-operand maps of x, per (pointer, T)
  int cached_xhT = 0;
  CUtensorMap tm_xh16{}, tm_xh128{};
  CUtensorMap tm_xn{}, tm_xnlo{};  // router input maps of the chain's normalised rows
  unsigned epoch = 0;
  long long launches = 0;
  int last_T = 0;
  int dense = 0;                    // dense MLP plan (etc_mlp_plan)
  const void* cached_xd = nullptr;  // dense MLP: token-operand maps of the caller's x, per (pointer, T)
  int cached_xdT = 0;
  CUtensorMap tm_xd16{}, tm_xd128{};
};

namespace {

// Router H-split for a call: with few token blocks, split H into NC chunks
// (multiples of 64 rows) so that the router tiles still spread over the grid;
// with enough blocks (nb > grid / 2) H stays whole and the top-k runs inside
// the router tile.
int choose_nc(int T, int H, int grid) {
  const int nb = (T + kTB - 1) / kTB;
  int nc = 1;
  while (nb * nc * 2 <= grid && (H / (nc * 2)) % kBK == 0) nc *= 2;
  return nc;
}

int alloc_dev(etc_plan_t p, void** out, size_t bytes) {
  void* d = nullptr;
  cudaError_t e = cudaMalloc(&d, std::max<size_t>(bytes, 256));
  if (e != cudaSuccess)
    return set_error(ETC_ERR_CUDA, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  p->allocs.push_back(d);
  *out = d;
  return ETC_OK;
}

// Bump allocator over one device buffer (256-byte aligned pieces).
struct Bump {
  char* base;
  size_t off;
  template <class T>
  T* take(size_t n) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* r = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += n * sizeof(T);
    return r;
  }
};

void carve_block(Bump& data, Bump& ctrl, BlockWs& b, const etc_plan_s& p) {
  const size_t E = p.E, k = p.k, T = p.T_max, nb = p.nb_max, C = p.C_max, R = p.R_max;
  b.logit_fx = ctrl.take<unsigned long long>(static_cast<size_t>(p.partial_max) * E);
  b.logits = data.take<float>(T * E);
  b.ids = data.take<int>(T * k);
  b.wts = data.take<float>(T * k);
  b.pos = data.take<int>(T * k);
  b.row_token = data.take<int>(R);
  b.row_w = data.take<float>(R);
  b.blk_cnt = data.take<int>(nb * E);
  b.part_cnt = data.take<int>(nb * kMaxPermParts * E);
  b.cnt_acc = ctrl.take<int>(E);
  b.counts = data.take<int>(E);
  b.exp_indptr = data.take<int>(E + 1);
  b.chunk_indptr = data.take<int>(E + 1);
  b.chunk_expert = data.take<int>(C);
  b.chunk_row0 = data.take<int>(C);
  b.chunk_rows = data.take<int>(C);
  b.chunk_src = data.take<int>(C);
  b.heavy = data.take<int>(E);
  b.meta = data.take<int>(8);
  b.ev_rblk = ctrl.take<int>(nb);
  b.ev_route = ctrl.take<int>(1);
  b.plan_flag = ctrl.take<unsigned>(1);
  b.ev_expert = ctrl.take<int>(E);
  b.ev_act = ctrl.take<int>(C);
  b.ev_down = ctrl.take<int>(C);
  b.ev_tok = ctrl.take<int>(nb);
  b.norm_flag = ctrl.take<unsigned>(nb);
  b.comb_flag = ctrl.take<unsigned>(nb);
}

void carve_globals(Bump& ctrl, Workspace& w) {
  for (int i = 0; i < 2; ++i) {
    w.qhead[i] = ctrl.take<int>(1);
    w.qtail[i] = ctrl.take<int>(1);
  }
  w.qtotal = ctrl.take<int>(1);
  w.qtotal_flag = ctrl.take<unsigned>(1);
  w.qacc = ctrl.take<int>(1);
  w.status = ctrl.take<DevStatus>(1);
}

int validate_opts(const etc_moe_opts* o) {
  if (!o) return set_error(ETC_ERR_INVALID, "opts is NULL");
  if (o->hidden <= 0 || o->hidden % 128 != 0 || o->hidden > 12288)
    return set_error(ETC_ERR_INVALID, "hidden=%d must be a multiple of 128 in [128, 12288]",
                     o->hidden);
  if (o->n_experts < 8 || o->n_experts > kMaxE || o->n_experts % 8 != 0)
    return set_error(ETC_ERR_INVALID, "n_experts=%d must be a multiple of 8 in [8, %d]",
                     o->n_experts, kMaxE);
  if (o->top_k < 1 || o->top_k > std::min(o->n_experts, kMaxK))
    return set_error(ETC_ERR_INVALID, "top_k=%d must be in [1, min(E, %d)]", o->top_k, kMaxK);
  if (o->inter <= 0 || o->inter % 64 != 0)
    return set_error(ETC_ERR_INVALID, "inter=%d must be a positive multiple of 64", o->inter);
  if (o->t_max < 1 || static_cast<long long>(o->t_max) * o->top_k > (1 << 24))
    return set_error(ETC_ERR_INVALID, "t_max=%d out of range", o->t_max);
  if (o->sched != ETC_SCHED_STATIC && o->sched != ETC_SCHED_DYNAMIC && o->sched != ETC_SCHED_MIXED)
    return set_error(ETC_ERR_INVALID, "sched=%d unknown", o->sched);
  if (o->sched == ETC_SCHED_MIXED && o->n_blocks != 1)
    return set_error(ETC_ERR_INVALID, "sched=MIXED needs n_blocks == 1 (got %d)", o->n_blocks);
  if (o->n_blocks < 1 || o->n_blocks > kMaxBlocks)
    return set_error(ETC_ERR_INVALID, "n_blocks=%d must be in [1, %d]", o->n_blocks, kMaxBlocks);
  if (o->router_bias && !aligned16(o->router_bias))
    return set_error(ETC_ERR_INVALID, "router_bias must be 16-byte aligned");
  if (o->out_dtype != ETC_OUT_F32 && o->out_dtype != ETC_OUT_BF16)
    return set_error(ETC_ERR_INVALID, "out_dtype=%d unknown", o->out_dtype);
  if (o->combine != ETC_COMBINE_FUSED && o->combine != ETC_COMBINE_ORDERED)
    return set_error(ETC_ERR_INVALID, "combine=%d unknown", o->combine);
  return ETC_OK;
}

int status_of(etc_plan_t p) {
  volatile DevStatus* h = p->ws.status_host;
  if (h->code == 0) return ETC_OK;
  return set_error(ETC_ERR_TIMEOUT,
                   "device wait timed out (code %d, task type/site %d, index %d, cta %d); "
                   "call etc_plan_reset",
                   h->code, h->where, h->aux, h->cta);
}

// Weight maps of block b for a call with wide (or narrow / pair) tiles.
int weight_maps(etc_plan_t p, int b, const void* wgu, const void* wd, bool wide,
                CUtensorMap* wgu_map, CUtensorMap* wd_map) {
  const unsigned long long halves = static_cast<unsigned long long>(p->E) * 2;
  const unsigned long long rows_dn = static_cast<unsigned long long>(p->E) * p->H;
  const void** cgu = wide ? p->cached_wgu128 : p->cached_wgu;
  CUtensorMap* mgu = wide ? p->tm_wgu128 : p->tm_wgu;
  if (cgu[b] != wgu) {
    CUresult r = encode_tensor_map_3d_bf16(&mgu[b], wgu, p->H, p->I, halves, kBK, wide ? 128 : 64, 2);
    if (r != CUDA_SUCCESS) return set_error(ETC_ERR_CUDA, "tensor map (w_gate_up) failed: %d", r);
    cgu[b] = wgu;
  }
  const void** cdn = wide ? p->cached_wd256 : p->cached_wd;
  CUtensorMap* mdn = wide ? p->tm_wd256 : p->tm_wd;
  if (cdn[b] != wd) {
    CUresult r = encode_tensor_map_2d_bf16(&mdn[b], wd, p->I, rows_dn, kBK, wide ? 256 : 128);
    if (r != CUDA_SUCCESS) return set_error(ETC_ERR_CUDA, "tensor map (w_down) failed: %d", r);
    cdn[b] = wd;
  }
  *wgu_map = mgu[b];
  *wd_map = mdn[b];
  return ETC_OK;
}

int router_weight_map(etc_plan_t p, int b, const void* gate_w) {
  if (p->cached_wg[b] != gate_w) {
    // [H, E] row-major, read as the MN-major A operand: boxes of 64 experts x 64 rows.
    CUresult r = encode_tensor_map_2d_bf16(&p->tm_wg[b], gate_w, p->E, p->H, 64, kBK);
    if (r != CUDA_SUCCESS) return set_error(ETC_ERR_CUDA, "tensor map (gate_w) failed: %d", r);
    p->cached_wg[b] = gate_w;
  }
  return ETC_OK;
}

struct CallArgs {
  const void* x = nullptr;
  void* out = nullptr;
  int T = 0;
  int n_blocks = 1;
  int use_norm = 0;
  const void* gate_w[kMaxBlocks] = {};
  const float* bias[kMaxBlocks] = {};
  const void* norm_w[kMaxBlocks] = {};
  const void* wgu[kMaxBlocks] = {};
  const void* wd[kMaxBlocks] = {};
  const float* logits_in = nullptr;
};

// One call: validation, params, then either one launch (stages lo..hi) or,
// for the unfused ablation, one launch per stage.
int run_call(etc_plan_t p, void* stream, const CallArgs& a, bool unfused, int stage_lo,
             int stage_hi, int mode) {
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  if (p->dense) return set_error(ETC_ERR_INVALID, "a dense MLP plan serves etc_mlp_forward only");
  if (a.T < 0 || a.T > p->T_max)
    return set_error(ETC_ERR_INVALID, "T=%d outside [0, t_max=%d]", a.T, p->T_max);
  if (a.T == 0) return ETC_OK;
  if (a.n_blocks > p->n_blocks)
    return set_error(ETC_ERR_INVALID, "plan holds %d blocks, call wants %d", p->n_blocks, a.n_blocks);
  if (!a.x || !aligned16(a.x) || (stage_hi >= TK_COMB && (!a.out || !aligned16(a.out))))
    return set_error(ETC_ERR_INVALID, "x/out must be 16-byte aligned device pointers");
  for (int b = 0; b < a.n_blocks; ++b) {
    if (!a.logits_in && (!a.gate_w[b] || !aligned16(a.gate_w[b])))
      return set_error(ETC_ERR_INVALID, "gate_w[%d] must be a 16-byte aligned device pointer", b);
    if (stage_hi >= TK_GU && (!a.wgu[b] || !a.wd[b] || !aligned16(a.wgu[b]) || !aligned16(a.wd[b])))
      return set_error(ETC_ERR_INVALID, "expert weights of block %d must be 16-byte aligned", b);
    if (a.use_norm && (!a.norm_w[b] || !aligned16(a.norm_w[b])))
      return set_error(ETC_ERR_INVALID, "norm_w[%d] must be a 16-byte aligned device pointer", b);
    if (a.bias[b] && !aligned16(a.bias[b]))
      return set_error(ETC_ERR_INVALID, "router_bias[%d] must be 16-byte aligned", b);
  }
  int st = status_of(p);
  if (st != ETC_OK) return set_error(ETC_ERR_STATE, "%s", last_error());
  int dev = 0;
  ETC_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != p->device)
    return set_error(ETC_ERR_INVALID, "plan belongs to device %d, current device is %d", p->device, dev);

  MegaParams prm;
  std::memset(&prm, 0, sizeof prm);
  const bool router_tiles = a.logits_in == nullptr;
  for (int b = 0; b < a.n_blocks; ++b) {
    if (router_tiles) {
      int r = router_weight_map(p, b, a.gate_w[b]);
      if (r != ETC_OK) return r;
      prm.tm_wg[b] = p->tm_wg[b];
    }
    prm.gate_w[b] = static_cast<const __nv_bfloat16*>(a.gate_w[b]);
    prm.bias[b] = a.bias[b];
    prm.norm_w[b] = static_cast<const __nv_bfloat16*>(a.norm_w[b]);
  }
  prm.tm_xperm = p->tm_xperm;
  prm.tm_act = p->tm_act;
  prm.tm_xperm128 = p->tm_xperm128;
  prm.tm_act128 = p->tm_act128;
  if (router_tiles) {
    if (a.use_norm) {
      prm.tm_xr = p->tm_xn;
      prm.tm_xrlo = p->tm_xnlo;
    } else {
      if (p->cached_x != a.x || p->cached_xT != a.T) {
        // Rows past T read as zero: the map's extent is the call's T.
        CUresult r = encode_tensor_map_2d_bf16(&p->tm_x, a.x, p->H, a.T, kBK, kTB);
        if (r != CUDA_SUCCESS) return set_error(ETC_ERR_CUDA, "tensor map (x) failed: %d", r);
        p->cached_x = a.x;
        p->cached_xT = a.T;
      }
      prm.tm_xr = p->tm_x;
    }
  }
  prm.ws = p->ws;
  prm.x = static_cast<const __nv_bfloat16*>(a.x);
  prm.out = a.out;
  prm.out_bf16 = p->opts.out_dtype == ETC_OUT_BF16 ? 1 : 0;
  prm.ordered = p->opts.combine == ETC_COMBINE_ORDERED ? 1 : 0;
  prm.logits_in = a.logits_in;
  prm.H = p->H;
  prm.E = p->E;
  prm.k = p->k;
  prm.I = p->I;
  prm.T_max = p->T_max;
  prm.n_blocks = a.n_blocks;
  prm.use_norm = a.use_norm;
  prm.eps = p->opts.rms_eps > 0.f ? p->opts.rms_eps : 1e-6f;
  prm.T = a.T;
  prm.nb = (a.T + kTB - 1) / kTB;
  prm.NC = router_tiles ? choose_nc(a.T, p->H, p->grid) : 1;
  prm.HC = p->H / prm.NC;
  prm.KBr = prm.HC / kBK;
  // Few token blocks: split each block's permute over kMaxPermParts tasks.
  prm.PP = prm.nb <= 32 ? kMaxPermParts : 1;
  // One token block with H split: the top-k task runs the scan (not in the
  // per-stage ablation, which launches every stage on its own).
  prm.fuse_scan = (prm.nb == 1 && prm.NC > 1 && !unfused) ? 1 : 0;
  prm.T_pad = prm.nb * kTB;
  // Wide expert tiles once experts average 64 rows or more (and the shapes divide).
  prm.wide = (static_cast<long long>(a.T) * p->k >= 64LL * p->E && p->I % kGuRowsW == 0 &&
              p->H % kDnRowsW == 0) ? 1 : 0;
  // On request the same calls run on CTA pairs (one cta_group::2 MMA over two
  // SMs: 256 weight rows x up to 256 chunk rows per tile) when clusters are
  // available.
  prm.pair = (prm.wide && a.n_blocks == 1 && !a.use_norm && router_tiles && p->pair_grid > 0 &&
              (p->opts.debug_flags & ETC_DEBUG_PAIR_MOE) && !(p->opts.debug_flags & ETC_DEBUG_NO_PAIR))
                 ? 1 : 0;
  if (prm.pair) prm.wide = 0;
  prm.tokmaj = (prm.wide && !(p->opts.debug_flags & ETC_DEBUG_WIDE_SWAP_AB)) ? 1 : 0;
  prm.cw = prm.pair ? kBT2 : kBT;
  prm.nbp = prm.pair ? (prm.nb + 1) / 2 : prm.nb;
  prm.ev_mul = prm.pair ? 2 : 1;
  prm.n_router = prm.nbp * prm.NC;
  prm.NT_gu = p->I / (prm.wide || prm.pair ? kGuRowsW : kGuRows);
  prm.NT_dn = p->H / (prm.wide || prm.pair ? kDnRowsW : kDnRows);
  // An expert holds at most one row per token: with T <= kTB no chunk is
  // above kTB rows, and the thin stages hold a whole token operand.
  prm.thin = (!prm.wide && !prm.pair && a.T <= kTB) ? 1 : 0;
  // One token block: gate/up tiles read the T token rows straight from x (or
  // the chain's normalised rows); no permute task, no x_perm rows.
  prm.direct = (prm.thin && prm.nb == 1 && router_tiles) ? 1 : 0;
  if (stage_hi >= TK_GU)
    for (int b = 0; b < a.n_blocks; ++b) {
      int r = weight_maps(p, b, a.wgu[b], a.wd[b], prm.wide != 0, &prm.tm_wgu[b], &prm.tm_wd[b]);
      if (r != ETC_OK) return r;
    }
  // Heavy experts: an expert that at least 85 % of the call's tokens chose
  // runs over all T rows of x, its gate/up tiles reading x itself (weight 0
  // for the tokens that did not choose it), so that its tiles need no
  // permuted rows and start as soon as the scan has run, while the permute of
  // the other experts is still in flight.  Calls whose output is the plain
  // fp32 sum of the fused combine, with the expert tiles taken from the
  // queue (dynamic and mixed scheduling: 21 us faster on the skewed T = 4096
  // prefill; the static walk measured no gain).
  prm.heavy_min = (prm.wide && !prm.pair && !prm.direct && a.n_blocks == 1 && !a.use_norm &&
                   router_tiles && !prm.out_bf16 && !prm.ordered && a.T >= kHeavyMinT &&
                   mode != ETC_SCHED_STATIC && !(p->opts.debug_flags & ETC_DEBUG_NO_HEAVY))
                      ? (17 * a.T + 19) / 20
                      : 0;
  if (prm.heavy_min > 0) {
    if (p->cached_xh != a.x || p->cached_xhT != a.T) {
      if (encode_tensor_map_2d_bf16(&p->tm_xh16, a.x, p->H, a.T, kBK, 16) != CUDA_SUCCESS ||
          encode_tensor_map_2d_bf16(&p->tm_xh128, a.x, p->H, a.T, kBK, 128) != CUDA_SUCCESS)
        return set_error(ETC_ERR_CUDA, "tensor map (x, heavy experts) failed");
      p->cached_xh = a.x;
      p->cached_xhT = a.T;
    }
    prm.tm_xh = p->tm_xh16;
    prm.tm_xh128 = p->tm_xh128;
  }
  if (++p->epoch == 0) p->epoch = 1;
  prm.epoch = p->epoch;
  prm.mode = mode;
  prm.timeout_ns = p->opts.wait_timeout_ns ? p->opts.wait_timeout_ns : 2000000000ull;
  prm.debug_flags = static_cast<int>(p->opts.debug_flags);
  prm.debug_arg = p->opts.debug_arg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (p->ws.trace) ETC_CUDA_TRY(cudaMemsetAsync(p->ws.trace, 0, 8, s));
  if (p->opts.debug_flags & ETC_DEBUG_POISON) {
    const size_t rows = static_cast<size_t>(p->R_max);
    ETC_CUDA_TRY(cudaMemsetAsync(p->ws.x_perm, 0xFF, rows * p->H * 2, s));
    ETC_CUDA_TRY(cudaMemsetAsync(p->ws.act, 0xFF, static_cast<size_t>(p->R_act) * p->I * 2, s));
    if (p->ws.acc)
      ETC_CUDA_TRY(cudaMemsetAsync(p->ws.acc, 0xFF, static_cast<size_t>(p->T_max) * p->H * 4, s));
  }
  const int grid = prm.pair ? p->pair_grid : p->grid;
  if (!unfused) {
    prm.stage_lo = stage_lo;
    prm.stage_hi = stage_hi;
    ETC_CUDA_TRY(launch_megakernel(prm, grid, s));
    ++p->launches;
    g_launches.fetch_add(1);
  } else {
    for (int stg = TK_ROUTER; stg <= TK_COMB; ++stg) {
      if (stg == TK_TOPK && prm.NC == 1) continue;  // top-k ran inside the router stage
      if (stg == TK_PERM && prm.direct) continue;   // no permute: tiles read x directly
      if (stg == TK_COMB && !prm.out_bf16 && !prm.ordered && a.n_blocks == 1) continue;  // nothing to finalise
      prm.stage_lo = prm.stage_hi = stg;
      ETC_CUDA_TRY(launch_megakernel(prm, grid, s));
      ++p->launches;
      g_launches.fetch_add(1);
    }
  }
  p->last_T = a.T;
  return ETC_OK;
}

int validate_mlp_opts(const etc_mlp_opts* o) {
  if (!o) return set_error(ETC_ERR_INVALID, "opts is NULL");
  if (o->hidden <= 0 || o->hidden % 128 != 0 || o->hidden > 16384)
    return set_error(ETC_ERR_INVALID, "hidden=%d must be a multiple of 128 in [128, 16384]",
                     o->hidden);
  if (o->inter <= 0 || o->inter % 64 != 0 || o->inter > 65536)
    return set_error(ETC_ERR_INVALID, "inter=%d must be a multiple of 64 in [64, 65536]", o->inter);
  if (o->t_max < 1 || o->t_max > 65536)
    return set_error(ETC_ERR_INVALID, "t_max=%d must be in [1, 65536]", o->t_max);
  if (o->sched != ETC_SCHED_STATIC && o->sched != ETC_SCHED_DYNAMIC)
    return set_error(ETC_ERR_INVALID, "sched=%d: the dense MLP takes STATIC or DYNAMIC", o->sched);
  if (o->out_dtype != ETC_OUT_F32 && o->out_dtype != ETC_OUT_BF16)
    return set_error(ETC_ERR_INVALID, "out_dtype=%d unknown", o->out_dtype);
  return ETC_OK;
}

// One dense MLP call: gate/up and down tiles of the same megakernel over
// 128-row chunks of x (one launch, or one per stage for the ablation).
int run_dense_call(etc_plan_t p, void* stream, const void* x, const void* wgu, const void* wd,
                   int T, void* out, bool unfused) {
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  if (!p->dense) return set_error(ETC_ERR_INVALID, "plan is not a dense MLP plan (etc_mlp_plan)");
  if (T < 0 || T > p->T_max)
    return set_error(ETC_ERR_INVALID, "T=%d outside [0, t_max=%d]", T, p->T_max);
  if (T == 0) return ETC_OK;
  if (!x || !out || !wgu || !wd || !aligned16(x) || !aligned16(out) || !aligned16(wgu) ||
      !aligned16(wd))
    return set_error(ETC_ERR_INVALID, "x, weights and out must be 16-byte aligned device pointers");
  int st = status_of(p);
  if (st != ETC_OK) return set_error(ETC_ERR_STATE, "%s", last_error());
  int dev = 0;
  ETC_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != p->device)
    return set_error(ETC_ERR_INVALID, "plan belongs to device %d, current device is %d", p->device, dev);
  if (p->cached_xd != x || p->cached_xdT != T) {
    // Rows past T read as zero: the maps' extent is the call's T.
    if (encode_tensor_map_2d_bf16(&p->tm_xd16, x, p->H, T, kBK, 16) != CUDA_SUCCESS ||
        encode_tensor_map_2d_bf16(&p->tm_xd128, x, p->H, T, kBK, 128) != CUDA_SUCCESS)
      return set_error(ETC_ERR_CUDA, "tensor map (x) failed");
    p->cached_xd = x;
    p->cached_xdT = T;
  }
  MegaParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.tm_xperm = p->tm_xd16;
  prm.tm_xperm128 = p->tm_xd128;
  prm.tm_act = p->tm_act;
  prm.tm_act128 = p->tm_act128;
  prm.ws = p->ws;
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.out = out;
  prm.out_bf16 = p->opts.out_dtype == ETC_OUT_BF16 ? 1 : 0;
  prm.H = p->H;
  prm.E = 1;
  prm.k = 1;
  prm.I = p->I;
  prm.T_max = p->T_max;
  prm.n_blocks = 1;
  prm.T = T;
  prm.nb = (T + kTB - 1) / kTB;
  prm.NC = 1;
  prm.HC = p->H;
  prm.PP = 1;
  prm.T_pad = prm.nb * kTB;
  prm.wide = (T >= 64 && p->I % kGuRowsW == 0 && p->H % kDnRowsW == 0) ? 1 : 0;
  prm.pair = (prm.wide && p->pair_grid > 0 && !(p->opts.debug_flags & ETC_DEBUG_NO_PAIR)) ? 1 : 0;
  if (prm.pair) prm.wide = 0;
  prm.tokmaj = (prm.wide && !(p->opts.debug_flags & ETC_DEBUG_WIDE_SWAP_AB)) ? 1 : 0;
  prm.cw = prm.pair ? kBT2 : kBT;
  prm.nbp = prm.nb;
  prm.ev_mul = prm.pair ? 2 : 1;
  prm.NT_gu = p->I / (prm.wide || prm.pair ? kGuRowsW : kGuRows);
  prm.NT_dn = p->H / (prm.wide || prm.pair ? kDnRowsW : kDnRows);
  prm.thin = (!prm.wide && !prm.pair && T <= kTB) ? 1 : 0;  // chunks of at most kTB rows
  int r = weight_maps(p, 0, wgu, wd, prm.wide != 0, &prm.tm_wgu[0], &prm.tm_wd[0]);
  if (r != ETC_OK) return r;
  prm.dense = 1;
  prm.n_chunks = (T + prm.cw - 1) / prm.cw;
  prm.q_total = prm.n_chunks * (prm.NT_gu + prm.NT_dn);
  if (++p->epoch == 0) p->epoch = 1;
  prm.epoch = p->epoch;
  prm.mode = unfused ? ETC_SCHED_STATIC : p->opts.sched;
  prm.timeout_ns = p->opts.wait_timeout_ns ? p->opts.wait_timeout_ns : 2000000000ull;
  prm.debug_flags = static_cast<int>(p->opts.debug_flags);
  prm.debug_arg = p->opts.debug_arg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->ws.trace) ETC_CUDA_TRY(cudaMemsetAsync(p->ws.trace, 0, 8, s));
  if (p->opts.debug_flags & ETC_DEBUG_POISON)
    ETC_CUDA_TRY(cudaMemsetAsync(p->ws.act, 0xFF, static_cast<size_t>(T) * p->I * 2, s));
  // Fused: one launch of both stages; unfused: the gate/up stage, then the down stage.
  const int stage[2] = {TK_GU, TK_DN};
  for (int i = 0; i < (unfused ? 2 : 1); ++i) {
    prm.stage_lo = unfused ? stage[i] : TK_GU;
    prm.stage_hi = unfused ? stage[i] : TK_DN;
    ETC_CUDA_TRY(launch_megakernel(prm, prm.pair ? p->pair_grid : p->grid, s));
    ++p->launches;
    g_launches.fetch_add(1);
  }
  p->last_T = T;
  return ETC_OK;
}

int plan_moe_buffers(etc_plan_t p);

// Plan body shared by the MoE layer and the dense MLP (options validated).
int make_plan(etc_plan_t* out, const etc_moe_opts* opts, bool dense) {
  int r = ETC_OK;
  etc_plan_t p = new etc_plan_s();
  p->dense = dense ? 1 : 0;
  p->opts = *opts;
  p->H = opts->hidden;
  p->E = opts->n_experts;
  p->k = opts->top_k;
  p->I = opts->inter;
  p->T_max = opts->t_max;
  p->n_blocks = opts->n_blocks;
  auto fail = [&](int code) {
    etc_plan_destroy(p);
    return code;
  };
  if (cudaGetDevice(&p->device) != cudaSuccess) return fail(set_error(ETC_ERR_CUDA, "no CUDA device"));
  if (megakernel_configure() != cudaSuccess)
    return fail(set_error(ETC_ERR_CUDA, "cannot configure %d bytes of shared memory", kSmemBytes));
  const int occ = megakernel_occupancy();
  if (occ < 1) return fail(set_error(ETC_ERR_CUDA, "megakernel does not fit on an SM"));
  p->grid = sm_count(p->device);  // one CTA per SM: TMEM and smem sized for that
  if (p->grid <= 0) return fail(set_error(ETC_ERR_CUDA, "cannot query SM count"));
  p->pair_grid = 2 * std::min(megakernel_pair_clusters(p->grid), p->grid / 2);

  p->nb_max = (p->T_max + kTB - 1) / kTB;
  p->R_max = p->T_max * p->k;
  // Heavy experts (at least ceil(0.85 T) rows each, so at most k / 0.85 of
  // them) take T act rows instead of their row count: at most
  // 0.15 / 0.85 < 0.2 of R_max more.
  p->R_act = dense ? p->R_max : p->R_max + p->R_max / 5 + kBT;
  p->C_max = (p->R_act + kBT - 1) / kBT + p->E;
  // Rows of fixed-point router sums: the token rows of the largest call whose
  // H is split (the split depends on T only through nb).
  p->partial_max = kTB;
  long long n_router_max = p->nb_max;
  for (int nb = 1; nb <= p->nb_max; ++nb) {
    const int nc = choose_nc(std::min(nb * kTB, p->T_max), p->H, p->grid);
    if (nc > 1) p->partial_max = std::max<long long>(p->partial_max, static_cast<long long>(nb) * kTB);
    n_router_max = std::max<long long>(n_router_max, static_cast<long long>(nb) * nc);
  }
  {
    const int nb = p->nb_max;
    const long long per_block = nb /*norm*/ + n_router_max + nb + 1 + nb * kMaxPermParts +
                                static_cast<long long>(p->C_max) * (p->I / kGuRows + p->H / kDnRows) + nb;
    p->ws.qcap = static_cast<int>(per_block * p->n_blocks + 64);
  }

  // Data region (no clearing needed) and control region (cleared on reset).
  Bump dsz{nullptr, 0}, csz{nullptr, 0};
  {
    BlockWs tmp{};
    Workspace wtmp{};
    for (int b = 0; b < p->n_blocks; ++b) carve_block(dsz, csz, tmp, *p);
    carve_globals(csz, wtmp);
  }
  void* data = nullptr;
  if ((r = alloc_dev(p, &data, dsz.off + 256)) != ETC_OK) return fail(r);
  if ((r = alloc_dev(p, &p->ctrl, csz.off + 256)) != ETC_OK) return fail(r);
  p->ctrl_bytes = csz.off + 256;
  Bump d{static_cast<char*>(data), 0}, c{static_cast<char*>(p->ctrl), 0};
  for (int b = 0; b < p->n_blocks; ++b) carve_block(d, c, p->ws.blk[b], *p);
  carve_globals(c, p->ws);
  if (cudaMemset(p->ctrl, 0, p->ctrl_bytes) != cudaSuccess)
    return fail(set_error(ETC_ERR_CUDA, "cudaMemset failed"));

  void* m = nullptr;
  const size_t R = static_cast<size_t>(p->R_act);
  if ((r = alloc_dev(p, &m, R * p->I * 2)) != ETC_OK) return fail(r);
  p->ws.act = static_cast<__nv_bfloat16*>(m);
  if (encode_tensor_map_2d_bf16(&p->tm_act, p->ws.act, p->I, R, kBK, 16) != CUDA_SUCCESS ||
      encode_tensor_map_2d_bf16(&p->tm_act128, p->ws.act, p->I, R, kBK, 128) != CUDA_SUCCESS)
    return fail(set_error(ETC_ERR_CUDA, "tensor map encoding of the workspace failed"));
  if (!dense && (r = plan_moe_buffers(p)) != ETC_OK) return fail(r);
  for (int i = 0; i < 2; ++i) {
    if ((r = alloc_dev(p, &m, static_cast<size_t>(p->ws.qcap) * 8)) != ETC_OK) return fail(r);
    p->ws.qslots[i] = static_cast<unsigned long long*>(m);
    if (cudaMemset(m, 0, static_cast<size_t>(p->ws.qcap) * 8) != cudaSuccess)
      return fail(set_error(ETC_ERR_CUDA, "cudaMemset failed"));
  }
  if (opts->debug_flags & ETC_DEBUG_TRACE) {
    p->ws.trace_cap = p->ws.qcap;
    if ((r = alloc_dev(p, &m, (1 + 4 * static_cast<size_t>(p->ws.trace_cap)) * 8)) != ETC_OK)
      return fail(r);
    p->ws.trace = static_cast<unsigned long long*>(m);
  }
  DevStatus* hs = nullptr;
  if (cudaHostAlloc(&hs, sizeof(DevStatus), cudaHostAllocMapped) != cudaSuccess)
    return fail(set_error(ETC_ERR_CUDA, "cudaHostAlloc failed"));
  std::memset(hs, 0, sizeof *hs);
  p->ws.status_host = hs;
  *out = p;
  return ETC_OK;
}

// Buffers only the MoE layer and the chain use: permuted rows, the fp32
// combine accumulator, the chain's normalised rows and residual stream.
int plan_moe_buffers(etc_plan_t p) {
  int r = ETC_OK;
  void* m = nullptr;
  const size_t R = static_cast<size_t>(p->R_max);
  if ((r = alloc_dev(p, &m, R * p->H * 2)) != ETC_OK) return r;
  p->ws.x_perm = static_cast<__nv_bfloat16*>(m);
  if (encode_tensor_map_2d_bf16(&p->tm_xperm, p->ws.x_perm, p->H, R, kBK, 16) != CUDA_SUCCESS ||
      encode_tensor_map_2d_bf16(&p->tm_xperm128, p->ws.x_perm, p->H, R, kBK, 128) != CUDA_SUCCESS)
    return set_error(ETC_ERR_CUDA, "tensor map encoding of the workspace failed");
  if (p->opts.combine == ETC_COMBINE_ORDERED) {  // the expert rows the ordered combine sums
    if ((r = alloc_dev(p, &m, R * p->H * 4)) != ETC_OK) return r;
    p->ws.yperm = static_cast<float*>(m);
  } else if (p->opts.out_dtype == ETC_OUT_BF16) {  // fp32 accumulator behind a bf16 output
    if ((r = alloc_dev(p, &m, static_cast<size_t>(p->T_max) * p->H * 4)) != ETC_OK) return r;
    p->ws.acc = static_cast<float*>(m);
  }
  // Normalised rows of the chain (any plan may be given to etc_chain_forward,
  // a one-block chain included).
  if ((r = alloc_dev(p, &m, static_cast<size_t>(p->T_max) * p->H * 2)) != ETC_OK) return r;
  p->ws.xn = static_cast<__nv_bfloat16*>(m);
  if ((r = alloc_dev(p, &m, static_cast<size_t>(p->T_max) * p->H * 2)) != ETC_OK) return r;
  p->ws.xn_lo = static_cast<__nv_bfloat16*>(m);
  if (encode_tensor_map_2d_bf16(&p->tm_xn, p->ws.xn, p->H, p->T_max, kBK, kTB) != CUDA_SUCCESS ||
      encode_tensor_map_2d_bf16(&p->tm_xnlo, p->ws.xn_lo, p->H, p->T_max, kBK, kTB) != CUDA_SUCCESS)
    return set_error(ETC_ERR_CUDA, "tensor map encoding of the normalised rows failed");
  if (p->n_blocks > 1) {
    if ((r = alloc_dev(p, &m, static_cast<size_t>(p->n_blocks - 1) * p->T_max * p->H * 4)) != ETC_OK)
      return r;
    p->ws.resid = static_cast<float*>(m);
  }
  return ETC_OK;
}

}  // namespace

extern "C" {

int etc_moe_plan(etc_plan_t* out, const etc_moe_opts* opts) {
  clear_error();
  if (!out) return set_error(ETC_ERR_INVALID, "plan pointer is NULL");
  *out = nullptr;
  const int r = validate_opts(opts);
  if (r != ETC_OK) return r;
  return make_plan(out, opts, false);
}

int etc_mlp_plan(etc_plan_t* out, const etc_mlp_opts* opts) {
  clear_error();
  if (!out) return set_error(ETC_ERR_INVALID, "plan pointer is NULL");
  *out = nullptr;
  const int r = validate_mlp_opts(opts);
  if (r != ETC_OK) return r;
  // One always-taken weight set: the plan of a one-expert, top-1 layer.
  etc_moe_opts o{};
  o.hidden = opts->hidden;
  o.n_experts = 1;
  o.top_k = 1;
  o.inter = opts->inter;
  o.t_max = opts->t_max;
  o.sched = opts->sched;
  o.n_blocks = 1;
  o.wait_timeout_ns = opts->wait_timeout_ns;
  o.debug_flags = opts->debug_flags & (ETC_DEBUG_POISON | ETC_DEBUG_TRACE | ETC_DEBUG_FAULT_EXTRA_WAIT |
                                      ETC_DEBUG_NO_PAIR);
  o.debug_arg = opts->debug_arg;
  o.out_dtype = opts->out_dtype;
  return make_plan(out, &o, true);
}

int etc_mlp_forward(etc_plan_t p, void* stream, const void* x, const void* w_gate_up,
                    const void* w_down, int T, void* out) {
  clear_error();
  return run_dense_call(p, stream, x, w_gate_up, w_down, T, out, false);
}

int etc_mlp_forward_unfused(etc_plan_t p, void* stream, const void* x, const void* w_gate_up,
                            const void* w_down, int T, void* out) {
  clear_error();
  return run_dense_call(p, stream, x, w_gate_up, w_down, T, out, true);
}

void etc_plan_destroy(etc_plan_t p) {
  if (!p) return;
  cudaDeviceSynchronize();
  for (void* d : p->allocs) cudaFree(d);
  if (p->ws.status_host) cudaFreeHost(p->ws.status_host);
  delete p;
}

int etc_moe_forward(etc_plan_t p, void* stream, const void* x, const void* gate_w,
                    const void* w_gate_up, const void* w_down, int T, void* out) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  CallArgs a;
  a.x = x;
  a.out = out;
  a.T = T;
  a.gate_w[0] = gate_w;
  a.bias[0] = p->opts.router_bias;
  a.wgu[0] = w_gate_up;
  a.wd[0] = w_down;
  return run_call(p, stream, a, false, TK_NORM, TK_COMB, p->opts.sched);
}

int etc_moe_forward_unfused(etc_plan_t p, void* stream, const void* x, const void* gate_w,
                            const void* w_gate_up, const void* w_down, int T, void* out) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  CallArgs a;
  a.x = x;
  a.out = out;
  a.T = T;
  a.gate_w[0] = gate_w;
  a.bias[0] = p->opts.router_bias;
  a.wgu[0] = w_gate_up;
  a.wd[0] = w_down;
  return run_call(p, stream, a, true, TK_ROUTER, TK_COMB, ETC_SCHED_STATIC);
}

int etc_moe_route_from_logits(etc_plan_t p, void* stream, const float* logits, const void* x,
                              int T) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  if (!logits) return set_error(ETC_ERR_INVALID, "logits is NULL");
  CallArgs a;
  a.x = x;
  a.T = T;
  a.logits_in = logits;
  return run_call(p, stream, a, false, TK_ROUTER, TK_PERM, ETC_SCHED_STATIC);
}

int etc_chain_forward(etc_plan_t p, void* stream, const void* x, const void* const* norm_w,
                      const void* const* gate_w, const float* const* router_bias,
                      const void* const* w_gate_up, const void* const* w_down, int T, void* out) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  if (!norm_w || !gate_w || !w_gate_up || !w_down)
    return set_error(ETC_ERR_INVALID, "weight pointer arrays must not be NULL");
  CallArgs a;
  a.x = x;
  a.out = out;
  a.T = T;
  a.n_blocks = p->n_blocks;
  a.use_norm = 1;
  for (int b = 0; b < p->n_blocks; ++b) {
    a.norm_w[b] = norm_w[b];
    a.gate_w[b] = gate_w[b];
    a.bias[b] = router_bias ? router_bias[b] : nullptr;
    a.wgu[b] = w_gate_up[b];
    a.wd[b] = w_down[b];
  }
  return run_call(p, stream, a, false, TK_NORM, TK_COMB, p->opts.sched);
}

int etc_moe_debug_routing(etc_plan_t p, void* stream, int block, void* logits, void* topk_ids,
                          void* topk_w, void* counts, void* exp_indptr, void* pos) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  if (p->dense) return set_error(ETC_ERR_INVALID, "a dense MLP plan has no routing");
  if (block < 0 || block >= p->n_blocks) return set_error(ETC_ERR_INVALID, "bad block %d", block);
  const BlockWs& b = p->ws.blk[block];
  const size_t T = p->last_T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaMemcpyKind kind = cudaMemcpyDeviceToDevice;
  if (logits) ETC_CUDA_TRY(cudaMemcpyAsync(logits, b.logits, T * p->E * 4, kind, s));
  if (topk_ids) ETC_CUDA_TRY(cudaMemcpyAsync(topk_ids, b.ids, T * p->k * 4, kind, s));
  if (topk_w) ETC_CUDA_TRY(cudaMemcpyAsync(topk_w, b.wts, T * p->k * 4, kind, s));
  if (counts) ETC_CUDA_TRY(cudaMemcpyAsync(counts, b.counts, p->E * 4, kind, s));
  if (exp_indptr) ETC_CUDA_TRY(cudaMemcpyAsync(exp_indptr, b.exp_indptr, (p->E + 1) * 4, kind, s));
  if (pos) ETC_CUDA_TRY(cudaMemcpyAsync(pos, b.pos, T * p->k * 4, kind, s));
  return ETC_OK;
}

int etc_moe_debug_buffer(etc_plan_t p, void* stream, int which, void* dst,
                         unsigned long long bytes) {
  clear_error();
  if (!p || !dst) return set_error(ETC_ERR_INVALID, "NULL argument");
  const unsigned long long R = static_cast<unsigned long long>(p->R_max);
  const void* src = nullptr;
  unsigned long long cap = 0;
  if (which == 0) {
    src = p->ws.x_perm;
    cap = R * p->H * 2;
  } else if (which == 1) {
    src = p->ws.act;
    cap = static_cast<unsigned long long>(p->R_act) * p->I * 2;
  } else {
    return set_error(ETC_ERR_INVALID, "unknown buffer %d", which);
  }
  if (!src) return set_error(ETC_ERR_INVALID, "this plan holds no buffer %d", which);
  if (bytes > cap) return set_error(ETC_ERR_INVALID, "buffer %d holds %llu bytes", which, cap);
  ETC_CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice,
                               static_cast<cudaStream_t>(stream)));
  return ETC_OK;
}

int etc_moe_debug_trace(etc_plan_t p, void* stream, void* dst, int max_records) {
  clear_error();
  if (!p || !dst || max_records < 0) return set_error(ETC_ERR_INVALID, "bad argument");
  if (!p->ws.trace) return set_error(ETC_ERR_INVALID, "plan was created without ETC_DEBUG_TRACE");
  const size_t n = 1 + 4 * static_cast<size_t>(std::min(max_records, p->ws.trace_cap));
  ETC_CUDA_TRY(cudaMemcpyAsync(dst, p->ws.trace, n * 8, cudaMemcpyDeviceToDevice,
                               static_cast<cudaStream_t>(stream)));
  return ETC_OK;
}

int etc_plan_check(etc_plan_t p) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  return status_of(p);
}

int etc_plan_reset(etc_plan_t p, void* stream) {
  clear_error();
  if (!p) return set_error(ETC_ERR_INVALID, "plan is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ETC_CUDA_TRY(cudaMemsetAsync(p->ctrl, 0, p->ctrl_bytes, s));
  ETC_CUDA_TRY(cudaStreamSynchronize(s));
  std::memset(const_cast<DevStatus*>(p->ws.status_host), 0, sizeof(DevStatus));
  // The epoch keeps counting: queue slots written by earlier calls carry
  // older epochs and can never be mistaken for this call's.
  return ETC_OK;
}

int etc_plan_stats(etc_plan_t p, long long* out, int n) {
  clear_error();
  if (!p || !out) return set_error(ETC_ERR_INVALID, "NULL argument");
  const long long v[8] = {p->launches, p->grid, kSmemBytes, p->epoch, kTB, kBT, p->ws.qcap, p->C_max};
  for (int i = 0; i < n && i < 8; ++i) out[i] = v[i];
  return ETC_OK;
}

}  // extern "C"
