// etc_internal.h -- structures shared by the host side and the kernels of the
// Event Tensor MoE library.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace etc {

// ---------------------------------------------------------------------------
// Megakernel geometry
// ---------------------------------------------------------------------------
constexpr int kThreads = 384;       // 12 warps per CTA, one CTA per SM
constexpr int kWarpSched = 0;       // lane 0: task scheduler (static walk or queue pop)
constexpr int kWarpTma = 1;         // lane 0: TMA producer
constexpr int kWarpMma = 2;         // lane 0: tcgen05 issuer; warp owns TMEM
constexpr int kWorkerWarp0 = 4;     // warps 4..11: epilogue + SIMT tasks
constexpr int kNumWorkers = 256;
constexpr int kStagesMax = 9;       // smem operand stages (9 x 20 KB thin, 6 x 32 KB narrow, 4 x 48 KB wide)
constexpr int kStagesNarrow = 6;
constexpr int kRing = 8;            // smem task ring depth
constexpr int kTB = 32;             // tokens per router/top-k/permute/combine task
constexpr int kMaxPermParts = 4;    // permute tasks per token block when blocks are few
constexpr int kHeavyMinT = 256;     // smallest call whose experts may run over all of x
constexpr int kBT = 128;            // max rows (tokens) per expert chunk = max MMA N
constexpr int kBT2 = 256;           // pair tiles: max rows per chunk (128 token rows per CTA)
constexpr int kBK = 64;             // K elements per stage (one 128-byte swizzle row)
// Expert tiles come in two widths.  Narrow (decode-sized calls): one M=128
// MMA per K step.  Wide (calls with many rows per expert): two M=128 MMAs
// that share the token operand, i.e. 256 weight rows per tile and 25% fewer
// operand bytes per FLOP.
constexpr int kGuRows = 64;         // narrow: gate rows (and up rows) per gate/up tile
constexpr int kDnRows = 128;        // narrow: output columns of H per down tile
constexpr int kGuRowsW = 128;       // wide: gate rows (and up rows) per gate/up tile
constexpr int kDnRowsW = 256;       // wide: output columns of H per down tile
constexpr int kAccCols = 256;       // TMEM columns per accumulator buffer (two 128-column halves)
constexpr int kTmemCols = 512;      // two accumulator buffers
constexpr int kMaxBlocks = 4;       // chain depth per launch
constexpr int kMaxE = 128;        // experts: one M=128 router MMA covers them all
constexpr int kMaxK = 16;
constexpr int kOpABytes = 128 * kBK * 2;      // 16 KB: one M=128 operand
constexpr int kStageABytes = 2 * kOpABytes;   // 32 KB: up to 256 weight rows
constexpr int kStageBBytes = kBT * kBK * 2;   // 16 KB: up to 128 token rows
constexpr int kStageRegion = 192 * 1024;      // the operand stages' shared memory
static_assert(kStageRegion >= 4 * (kStageABytes + kStageBBytes), "wide stages do not fit");
static_assert(kStageRegion >= kStagesNarrow * (kOpABytes + kStageBBytes), "narrow stages do not fit");
// Thin calls (no chunk above 32 rows): 16 KB of weights + 32 token rows.
constexpr int kStageThinBytes = kOpABytes + kTB * kBK * 2;
static_assert(kStageRegion >= kStagesMax * kStageThinBytes, "thin stages do not fit");
static_assert(kStageThinBytes % 1024 == 0, "thin stages must keep the 1 KB swizzle alignment");
// The worker warps run one task at a time, so the SIMT tasks' scratch and the
// GEMM epilogues' staging share one region.
constexpr int kSimtBytes = 32 * 1024;
constexpr int kEpiHalfBytes = 8 * 1024;       // U (4 KB fp32) + S (4 KB bf16) per half
constexpr int kWorkerBytes = kSimtBytes > 2 * kEpiHalfBytes ? kSimtBytes : 2 * kEpiHalfBytes;
constexpr int kCtrlBytes = 2048;
constexpr int kSmemBytes = 1024 /*align slack*/ + kStageRegion + kWorkerBytes + kCtrlBytes;
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA may use");

enum TaskType : int {
  TK_NONE = 0,
  TK_NORM = 1,
  TK_ROUTER = 2,
  TK_TOPK = 3,
  TK_SCAN = 4,
  TK_PERM = 5,
  TK_GU = 6,
  TK_DN = 7,
  TK_COMB = 8,
  TK_TERM = 15,
};

// Device error codes (DevStatus::code).
enum DevErr : int {
  DERR_NONE = 0,
  DERR_TIMEOUT_EVENT = 1,
  DERR_TIMEOUT_QUEUE = 2,
  DERR_TIMEOUT_MBAR = 3,
  DERR_QUEUE_OVERFLOW = 4,
  DERR_BAD_TASK = 5,
};

struct DevStatus {
  int code;   // first error wins
  int where;  // site id (task type or internal wait id)
  int aux;    // event index
  int cta;
};

// 32-bit task descriptor: type[31:28] blk[27:25] a[24:8] b[7:0].
__host__ __device__ inline uint32_t task_enc(int type, int blk, int a, int b) {
  return (static_cast<uint32_t>(type) << 28) | (static_cast<uint32_t>(blk) << 25) |
         (static_cast<uint32_t>(a) << 8) | static_cast<uint32_t>(b);
}
__host__ __device__ inline int task_type(uint32_t d) { return static_cast<int>(d >> 28); }
__host__ __device__ inline int task_blk(uint32_t d) { return static_cast<int>((d >> 25) & 7); }
__host__ __device__ inline int task_a(uint32_t d) { return static_cast<int>((d >> 8) & 0x1FFFF); }
__host__ __device__ inline int task_b(uint32_t d) { return static_cast<int>(d & 0xFF); }

// Per-block workspace (the chain keeps one per block).
struct BlockWs {
  unsigned long long* logit_fx;  // [T_pad, E] sum of H-chunk partials, fixed point 2^-40 (NC > 1)
  float* logits;       // [T_max, E] final fp32 logits (with bias)
  int* ids;            // [T_max, k]
  float* wts;          // [T_max, k]
  int* pos;            // [T_max, k] row of slot (t, j) in expert-sorted order
  int* row_token;      // [R_max] token of each expert-sorted row
  float* row_w;        // [R_max] routing weight of each expert-sorted row
  int* blk_cnt;        // [nb_max, E] per-token-block expert histogram
  int* cnt_acc;        // [E] counts summed by the routing tasks; the scan reads and re-arms it
  int* part_cnt;       // [nb_max * kMaxPermParts, E] expert histogram of each permute part
  int* counts;         // [E]
  int* exp_indptr;     // [E+1]
  int* chunk_indptr;   // [E+1]
  int* chunk_expert;   // [C_max]
  int* chunk_row0;     // [C_max]
  int* chunk_rows;     // [C_max]
  int* chunk_src;      // [C_max] token rows of the chunk: x_perm rows from chunk_src[c], or
                       // (heavy expert) x rows from -1 - chunk_src[c]
  int* heavy;          // [E] 1: this call runs the expert over all T rows of x (no permute)
  int* meta;           // [8] 0: n_chunks 1: n_gu 2: n_dn 3: heavy experts' chunks (first)
  // Event tensor counters
  int* ev_rblk;        // [nb_max] router partials landed per token block (count up to NC)
  int* ev_route;       // [1] top-k tasks done (count up to nb)
  unsigned* plan_flag; // [1] epoch once counts / exp_indptr / event inits are published
  int* ev_expert;      // [E] count-down from counts[e] (permuted rows still missing)
  int* ev_act;         // [C_max] count-down from gate/up tiles per chunk
  int* ev_down;        // [C_max] count-down from down tiles per chunk
                       // (dense MLP: ev_act / ev_down count up and are re-armed
                       // to 0 by the chunk's last down tile)
  int* ev_tok;         // [nb_max] count-down from expert rows per token block
  unsigned* norm_flag; // [nb_max] epoch once the token block is normalised (chain)
  unsigned* comb_flag; // [nb_max] epoch once the token block is combined (chain)
};

struct Workspace {
  BlockWs blk[kMaxBlocks];
  __nv_bfloat16* x_perm;  // [R_max, H]
  __nv_bfloat16* act;     // [R_act, I] (R_act: R_max plus the heavy experts' extra rows)
  float* acc;             // [T_max, H] fp32 combine accumulator when `out` is bf16
  float* yperm;           // [R_max, H] fp32 expert rows, expert-sorted (ordered combine)
  __nv_bfloat16* xn;      // [T_max, H] normalised input rounded to bf16 (chain)
  __nv_bfloat16* xn_lo;   // [T_max, H] bf16 of what that rounding dropped (router only)
  float* resid;           // [n_blocks-1, T_max, H] fp32 residual stream between blocks
  unsigned long long* qslots[2];  // dynamic queue, one per epoch parity
  int* qhead[2];
  int* qtail[2];
  int* qtotal;            // tasks of the whole call, known after the last scan
  unsigned* qtotal_flag;
  int* qacc;
  DevStatus* status;      // device copy, polled by spinning CTAs
  DevStatus* status_host; // host-mapped mirror written on error
  unsigned long long* trace;  // [1 + 4 * trace_cap] task trace (debug), or null
  int trace_cap;
  int qcap;
};

struct MegaParams {
  CUtensorMap tm_wgu[kMaxBlocks];  // [E*2][I][H] box 2 x 64 rows x 64 (wide tiles: 2 x 128 rows),
                                   // 128B swizzle: R gate rows, then the R up rows beside them
  CUtensorMap tm_wd[kMaxBlocks];   // [E*H, I]  box 128 rows x 64 (wide tiles: 256 rows)
  CUtensorMap tm_xperm;            // [R_max, H] box 16x64 (dense MLP: the caller's x [T, H])
  CUtensorMap tm_act;              // [R_max, I] box 16x64
  CUtensorMap tm_xperm128;         // [R_max, H] box 128 rows x 64 (dense MLP: x)
  CUtensorMap tm_act128;           // [R_act, I] box 128 rows x 64
  CUtensorMap tm_wg[kMaxBlocks];   // router weight [H, E], box 64 experts x 64 rows (MN-major A)
  CUtensorMap tm_xr;               // router input rows [T, H] (x, or xn in the chain), box 32x64
  CUtensorMap tm_xrlo;             // xn_lo [T_max, H] (chain), box 32x64
  CUtensorMap tm_xh;               // x [T, H] box 16x64: heavy experts' token rows
  CUtensorMap tm_xh128;            // x [T, H] box 128 rows x 64
  Workspace ws;
  const __nv_bfloat16* x;
  void* out;     // fp32 [T, H], or bf16 when out_bf16
  int out_bf16;
  int ordered;   // combine: down tiles store y rows, a finaliser sums them in j order
  const __nv_bfloat16* gate_w[kMaxBlocks];
  const float* bias[kMaxBlocks];
  const __nv_bfloat16* norm_w[kMaxBlocks];
  const float* logits_in;  // non-null: routing from given logits (router stage skipped)
  int H, E, k, I, T_max;
  int n_blocks;
  int use_norm;  // chain: RMSNorm before and residual after each block
  float eps;
  int T, nb, NC, HC, n_router, T_pad;
  int KBr;       // 64-wide K blocks per router task (HC / 64)
  int PP;        // permute parts per token block (1, or kMaxPermParts for few blocks)
  int fuse_scan; // one token block with H split: its top-k task runs the scan
  int NT_gu, NT_dn;
  int wide;      // expert tiles of 256 weight rows (two MMAs per K step)
  int pair;      // CTA-pair tiles (cta_group::2): 128 weight rows x up to 128 token rows per
                 // CTA; every task belongs to a pair, whose two CTAs each take half of it
  int cw;        // rows per expert chunk (kBT, or kBT2 with pair tiles)
  int nbp;       // token blocks as tasks see them: nb, or ceil(nb / 2) pair blocks
  int ev_mul;    // notifies per tile or routing task (2 with pair tiles: one per CTA)
  int thin;      // narrow tiles whose chunks hold at most kTB rows: 20 KB stages
  int direct;    // one token block: gate/up tiles read all T token rows of x (no permute)
  int tokmaj;    // wide gate/up tiles of full chunks token-major: M = the chunk's 128 token
                 // rows, N = 256 weight rows (one N=256 MMA per K step); other expert tiles
                 // swap-AB (M = weight rows, N = chunk rows)
  int heavy_min; // > 0: experts with at least this many rows run over all T rows of x,
                 // their tiles reading x itself (ready as soon as the scan has run); 0: off
  unsigned epoch;
  int mode;  // 0 static, 1 dynamic, 2 mixed
  int dense;     // dense MLP: one weight set, chunks are 128-row slices of x, no routing
  int n_chunks;  // dense MLP: chunks of this call
  int q_total;   // dense MLP: tasks of the call (known on the host)
  int stage_lo, stage_hi;
  unsigned long long timeout_ns;
  int debug_flags, debug_arg;
};

// Host-side launch helpers implemented next to the kernels.
cudaError_t launch_megakernel(const MegaParams& p, int grid, cudaStream_t stream);
cudaError_t megakernel_configure();

}  // namespace etc
