/*
 * etc_moe.h -- C ABI of the GB300 Event Tensor MoE library (libetc_moe.so).
 *
 * The library runs one Mixture-of-Experts layer (router -> top-k -> per-expert
 * counts and exp_indptr -> token permute -> GroupGEMM gate/up with SwiGLU ->
 * GroupGEMM down -> weighted combine) as ONE persistent CUDA kernel whose tiled
 * tasks are coordinated by an Event Tensor: a device array of counters.  It
 * also exports the split-K row-sum task graph and a chain of
 * RMSNorm -> MoE -> residual blocks run in one launch.
 *
 * Sources for the operations ("Event Tensor: A Unified Abstraction for
 * Compiling Dynamic Megakernel", paper summary page and podcast transcript):
 *   - MoE subgraph, runtime tensors topk and exp_indptr: Figure 2, Figure 5(b).
 *   - Data-dependent event update (an expert's wait_count is the number of
 *     tokens routed to it) and data-dependent task triggering (expert i fires
 *     the GroupGEMM tiles of rows [exp_indptr[i], exp_indptr[i+1])): podcast
 *     transcript, cues 7 and 9.
 *   - Symbolic shapes: the token count T is a per-call value; the same kernel
 *     serves every T with no recompilation and no graph capture: Figure 4,
 *     podcast cue 5, Table 1 (0 JIT captures).
 *   - Static scheduling (per-SM task lists, notify/wait on counters) and
 *     dynamic scheduling (a notify that brings a counter to zero pushes the
 *     ready task into a shared queue; idle SMs pop): Figures 6-9, podcast
 *     cue 11.
 *   - Split-K: partial_sum(i,j) notifies event i (wait_count = number of column
 *     tiles, map "ij->i"); final_sum(i) waits on event i only ("i->i"):
 *     Figure 3, podcast cue 3.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers, 16-byte aligned, contiguous
 *     row-major with the shapes given below.  bf16 means IEEE bfloat16 stored
 *     as uint16.  The caller owns all tensors it passes; the library never
 *     frees them and never keeps them past the call.
 *   - `stream` is a cudaStream_t passed as void*.  Calls are asynchronous on
 *     it: nothing is synchronised and nothing is copied to the host.
 *   - Return 0 (ETC_OK) or a negative ETC_ERR_* code; etc_last_error() then
 *     holds a message (per calling thread).
 *   - Device-side waits are bounded in time.  A wait that gives up records a
 *     timeout in the plan's status, makes every CTA exit cleanly, and leaves
 *     the CUDA context usable; etc_plan_check() reports it once the stream has
 *     completed, and etc_plan_reset() makes the plan usable again.
 */
#ifndef ETC_MOE_H_
#define ETC_MOE_H_

#ifdef __cplusplus
extern "C" {
#endif

#define ETC_OK 0
#define ETC_ERR_INVALID (-1)       /* bad shape, pointer, alignment or T */
#define ETC_ERR_CUDA (-2)          /* a CUDA runtime call failed */
#define ETC_ERR_TIMEOUT (-3)       /* a device wait gave up (see etc_plan_check) */
#define ETC_ERR_UNIMPLEMENTED (-4) /* option not supported by this library */
#define ETC_ERR_STATE (-5)         /* plan needs etc_plan_reset after a timeout */

/*
 * Schedulers of the megakernel's tasks:
 *   STATIC   every CTA walks a fixed, stage-ordered list of task slots and
 *            spin-waits on each task's input event (notify/wait);
 *   DYNAMIC  the notify that completes an event pushes the tasks it makes
 *            ready into a global queue, from which CTAs pop (push/pop);
 *   MIXED    (n_blocks == 1) router, top-k, scan and permute as STATIC, the
 *            expert tiles and the combine finaliser through the queue as
 *            DYNAMIC.  Not accepted by the split-K entry points.
 */
typedef enum { ETC_SCHED_STATIC = 0, ETC_SCHED_DYNAMIC = 1, ETC_SCHED_MIXED = 2 } etc_sched_t;

/* Debug bits for etc_moe_opts.debug_flags. */
#define ETC_DEBUG_FAULT_EXTRA_WAIT 0x1u /* add 1 to expert debug_arg's wait_count (dense MLP:
                                           chunk debug_arg's gate/up target): its tiles never
                                           become ready, so a wait times out */
#define ETC_DEBUG_POISON 0x2u           /* fill intermediate buffers with NaN before each call */
#define ETC_DEBUG_TRACE 0x4u            /* record every task's dispatch/start/end time and SM */
#define ETC_DEBUG_NO_PAIR 0x8u          /* never run expert tiles on CTA pairs (dense MLP: run its
                                           wide tiles on single CTAs; ablation of the pair tiles) */
#define ETC_DEBUG_PAIR_MOE 0x10u        /* run the wide expert tiles of MoE calls on CTA pairs too
                                           (by default only the dense MLP uses them: on the MoE
                                           layer's skewed chunks they measured no faster) */
#define ETC_DEBUG_WIDE_SWAP_AB 0x40u    /* wide gate/up tiles of full chunks with the weight rows as
                                           the MMA's M (two M=128 x N=128 MMAs per K step) instead of
                                           the token rows (one M=128 x N=256 MMA); ablation */
#define ETC_DEBUG_NO_HEAVY 0x20u        /* never run an expert over all T rows of x (by default, in
                                           dynamic and mixed scheduling, an expert that >= 85 % of a
                                           large call's tokens chose does, its tiles needing no
                                           permuted rows; ablation) */

typedef struct etc_plan_s* etc_plan_t;

typedef struct {
  int hidden;        /* H: model width; multiple of 128, at most 12288 */
  int n_experts;     /* E: 8..128, multiple of 8 (one router tile holds all experts) */
  int top_k;         /* k: 1..min(E,16) */
  int inter;         /* I: expert intermediate width; multiple of 64 */
  int t_max;         /* largest token count a call may pass (>= 1) */
  int sched;         /* etc_sched_t (MIXED only with n_blocks == 1) */
  int n_blocks;      /* 1 for etc_moe_forward; 1..4 for etc_chain_forward */
  float rms_eps;     /* RMSNorm epsilon of the chain (0 -> 1e-6) */
  const float* router_bias;          /* device fp32 [E] added to the logits, or NULL */
  unsigned long long wait_timeout_ns; /* device wait limit (0 -> 2 s) */
  unsigned debug_flags;              /* ETC_DEBUG_* */
  int debug_arg;                     /* expert id for ETC_DEBUG_FAULT_EXTRA_WAIT */
  int out_dtype;                     /* ETC_OUT_F32 (default) or ETC_OUT_BF16 */
  int combine;                       /* ETC_COMBINE_FUSED (default) or ETC_COMBINE_ORDERED */
} etc_moe_opts;

/* Element type of `out` (etc_moe_opts.out_dtype). */
#define ETC_OUT_F32 0  /* the fp32 combine sum, unrounded */
#define ETC_OUT_BF16 1 /* the same sum rounded to bf16 */

/*
 * How the k weighted expert rows of a token are added (etc_moe_opts.combine):
 *   FUSED    each down tile adds w * y into the token's fp32 output row with
 *            fp32 reductions in L2, in the order the tiles finish (no extra
 *            memory traffic; the last bits may differ from run to run);
 *   ORDERED  down tiles store their rows y to an fp32 buffer [T*k, H] of the
 *            plan, and a finaliser per 32-token block forms
 *            out[t] = sum_{j=0..k-1} w[t,j] * y[pos[t,j]] in j order (fp32 fused
 *            multiply-adds): the result is the same bit for bit from run to
 *            run and for every scheduler, at the cost of writing and reading
 *            the rows once more.
 */
#define ETC_COMBINE_FUSED 0
#define ETC_COMBINE_ORDERED 1

/*
 * Creates a plan for one weight shape: validates the options, allocates the
 * workspace (event counters, task queue, routing buffers, permuted
 * activations sized for t_max), builds the TMA descriptors of the workspace,
 * and sizes the persistent grid (one CTA per SM, all co-resident).  Nothing
 * in the plan depends on T.  The plan belongs to the current CUDA device.
 * Returns ETC_ERR_INVALID for unsupported shapes, ETC_ERR_CUDA if allocation
 * fails.  Free with etc_plan_destroy.
 */
int etc_moe_plan(etc_plan_t* plan, const etc_moe_opts* opts);

/*
 * One MoE layer, out = sum_j w[t,j] * FFN_{ids[t,j]}(x[t]), in ONE kernel
 * launch on `stream`.  (See etc_moe_opts.combine for how the sum is formed.)
 *   x          bf16 [T, H]
 *   gate_w     bf16 [H, E]       router weight (logits = x gate_w + bias)
 *   w_gate_up  bf16 [E, 2I, H]   rows 0..I-1 gate, rows I..2I-1 up (K-major)
 *   w_down     bf16 [E, H, I]    (K-major)
 *   out        fp32 [T, H] (bf16 [T, H] when opts.out_dtype = ETC_OUT_BF16)
 * Routing: the logits are bf16 x bf16 products summed in fp32 on the tensor
 * cores (when T is small, H is split into chunks whose partial sums are added
 * exactly as 64-bit fixed point); top-k of the fp32 logits, ties to the lower
 * expert id; weights = softmax over the k selected logits.  Accumulation is fp32; the SwiGLU
 * activation is rounded to bf16 (the operand of the second GEMM); each down
 * tile adds its weighted fp32 outputs into the token rows of `out` with
 * fp32 reductions in L2 (the order of the k additions per element is not
 * fixed, so results may differ in the last fp32 bits from run to run).
 * 0 <= T <= t_max; T == 0 returns ETC_OK without launching.
 * Concurrent calls on one plan are undefined: give each stream its own plan.
 */
int etc_moe_forward(etc_plan_t plan, void* stream, const void* x, const void* gate_w,
                    const void* w_gate_up, const void* w_down, int T, void* out);

/*
 * The same layer computed by the same task code, one kernel launch per stage
 * that has work (router, top-k, scan, permute, gate/up, down, combine: 5 to 7
 * launches: no top-k launch when the top-k runs inside the router stage, i.e.
 * when H is not split; no combine launch for an fp32 output, which is complete
 * after the down stage).  The ablation baseline for the one-launch
 * megakernel.  Same arguments and result.
 */
int etc_moe_forward_unfused(etc_plan_t plan, void* stream, const void* x, const void* gate_w,
                            const void* w_gate_up, const void* w_down, int T, void* out);

/*
 * Routing from caller-given fp32 logits [T, E] (device): runs the top-k,
 * count/scan and permute stages of the megakernel on `x` and leaves the
 * routing in the plan's workspace for etc_moe_debug_routing.  Used to check
 * the routing bit for bit against a reference fed the same logits.
 */
int etc_moe_route_from_logits(etc_plan_t plan, void* stream, const float* logits, const void* x,
                              int T);

/*
 * Copies the last call's routing of block `block` from the workspace into
 * caller buffers (device pointers, each may be NULL), asynchronously on
 * `stream`:  logits fp32 [T,E] (with bias), topk_ids int32 [T,k], topk_w fp32
 * [T,k], counts int32 [E], exp_indptr int32 [E+1], pos int32 [T,k] (row of
 * slot (t,j) in the expert-sorted order).  T is the last call's token count.
 */
int etc_moe_debug_routing(etc_plan_t plan, void* stream, int block, void* logits, void* topk_ids,
                          void* topk_w, void* counts, void* exp_indptr, void* pos);

/*
 * Copies `bytes` bytes from the start of an intermediate buffer of the last
 * call into `dst` (device), asynchronously on `stream`.  which: 0 = x_perm
 * bf16 [T*k, H] (expert-sorted input rows), 1 = act bf16 [T*k, I] (SwiGLU
 * output).  Returns ETC_ERR_INVALID if `bytes` exceeds the buffer.
 */
int etc_moe_debug_buffer(etc_plan_t plan, void* stream, int which, void* dst,
                         unsigned long long bytes);

/*
 * Task trace of the last call of a plan created with ETC_DEBUG_TRACE: copies
 * up to `max_records` records into `dst` (device, uint64 [1 + 4*max_records]),
 * asynchronously on `stream`.  dst[0] = number of records written by the call;
 * record i = dst[1+4i .. 4+4i]: (type<<56 | block<<48 | sm<<32 | a<<8 | b),
 * dispatch time, start time, end time (ns, %globaltimer).  The dispatch time
 * is when the scheduler handed the task to its CTA (after its input event);
 * start/end bracket the workers' part of the task.  Returns ETC_ERR_INVALID
 * if the plan has no trace buffer.
 */
int etc_moe_debug_trace(etc_plan_t plan, void* stream, void* dst, int max_records);

/*
 * A plan for a chain of n_blocks blocks (1..4) of the layer that opts
 * describes: the same as etc_moe_plan with opts->n_blocks replaced by
 * n_blocks (opts itself is not modified).  Same errors as etc_moe_plan.
 */
int etc_chain_plan(etc_plan_t* plan, const etc_moe_opts* opts, int n_blocks);

/*
 * Chain of opts.n_blocks blocks  x <- x + MoE_b(RMSNorm_b(x))  in ONE launch.
 * Arguments are HOST arrays of n_blocks DEVICE pointers:
 *   norm_w[b] bf16 [H], gate_w[b] bf16 [H,E], router_bias[b] fp32 [E] (the
 *   array or an entry may be NULL), w_gate_up[b] bf16 [E,2I,H],
 *   w_down[b] bf16 [E,H,I].  x bf16 [T,H]; out [T,H] of opts.out_dtype.  The
 *   residual stream between blocks stays fp32 in the workspace.  Each
 *   block's normalised input is rounded to bf16 (the GEMM operand).  Block
 *   b+1's work on a token block starts as soon as block
 *   b has combined that token block.  T may change on every call.
 */
int etc_chain_forward(etc_plan_t plan, void* stream, const void* x, const void* const* norm_w,
                      const void* const* gate_w, const float* const* router_bias,
                      const void* const* w_gate_up, const void* const* w_down, int T, void* out);

/*
 * Dense MLP, out = (silu(x Wg^T) * (x Wu^T)) Wd^T, run by the same persistent
 * megakernel, operand pipeline and event counters as the MoE layer, with one
 * always-taken weight set and no routing stages.  The shapes are the dense MLP
 * configurations of the paper summary page's appendix (Table 4: S, H, I); the
 * pages name no activation, and SwiGLU (the experts' FFN) is used.  Gate/up
 * tiles of 128-token chunks need no input event; the down tiles of chunk c
 * wait on chunk c's counter, which its gate/up tiles notify (count-up, re-armed
 * by the chunk's last down tile).  STATIC is the schedule the pages expect to
 * win on regular dense layers (Table 3; podcast transcript, cue 13); DYNAMIC
 * seeds the queue with every gate/up tile and pushes a chunk's down tiles
 * when its counter completes.
 */
typedef struct {
  int hidden;        /* H: multiple of 128, at most 16384 */
  int inter;         /* I: multiple of 64, at most 65536 */
  int t_max;         /* largest token count a call may pass: 1..65536 */
  int sched;         /* ETC_SCHED_STATIC or ETC_SCHED_DYNAMIC */
  unsigned long long wait_timeout_ns; /* device wait limit (0 -> 2 s) */
  unsigned debug_flags;              /* ETC_DEBUG_POISON, ETC_DEBUG_TRACE, ETC_DEBUG_FAULT_EXTRA_WAIT */
  int out_dtype;                     /* ETC_OUT_F32 (default) or ETC_OUT_BF16 */
  int debug_arg;                     /* chunk (128-row slice) for ETC_DEBUG_FAULT_EXTRA_WAIT */
} etc_mlp_opts;

/*
 * Creates a dense MLP plan: validates the options, allocates the event
 * counters, the task queue and the activation buffer act bf16 [t_max, I].
 * The plan serves etc_mlp_forward(_unfused) and the plan-level calls
 * (etc_plan_check, _reset, _stats, _destroy, etc_moe_debug_trace,
 * etc_moe_debug_buffer with which = 1); the MoE entry points refuse it with
 * ETC_ERR_INVALID, and etc_mlp_forward refuses MoE plans.
 */
int etc_mlp_plan(etc_plan_t* plan, const etc_mlp_opts* opts);

/*
 * One dense MLP in ONE kernel launch on `stream`:
 *   x          bf16 [T, H]
 *   w_gate_up  bf16 [2I, H]   rows 0..I-1 gate, rows I..2I-1 up (K-major)
 *   w_down     bf16 [H, I]    (K-major)
 *   out        fp32 [T, H] (bf16 [T, H] when opts.out_dtype = ETC_OUT_BF16)
 * Accumulation is fp32 on the tensor cores; the SwiGLU activation is rounded
 * to bf16 (the operand of the second GEMM); each output element is written
 * once, by the down tile that owns it (the result is deterministic).
 * 0 <= T <= t_max; T == 0 returns ETC_OK without launching.
 */
int etc_mlp_forward(etc_plan_t plan, void* stream, const void* x, const void* w_gate_up,
                    const void* w_down, int T, void* out);

/* The same MLP by the same task code in two launches (gate/up stage, then
 * down stage): the unfused baseline of the one-launch kernel. */
int etc_mlp_forward_unfused(etc_plan_t plan, void* stream, const void* x, const void* w_gate_up,
                            const void* w_down, int T, void* out);

/*
 * Reads the plan's device status (after the caller has synchronised the
 * stream of the last call): ETC_OK, or ETC_ERR_TIMEOUT with the site in
 * etc_last_error().  Does not synchronise anything itself.
 */
int etc_plan_check(etc_plan_t plan);

/* Clears the status and all event counters (async on `stream`). */
int etc_plan_reset(etc_plan_t plan, void* stream);

/*
 * Statistics of a plan: out[0] = kernel launches issued so far, out[1] =
 * persistent grid size, out[2] = dynamic shared memory per CTA, out[3] =
 * epoch (calls so far), out[4] = token-block size, out[5] = max tokens per
 * expert tile.  n = number of entries wanted (<= 8).
 */
int etc_plan_stats(etc_plan_t plan, long long* out, int n);

void etc_plan_destroy(etc_plan_t plan);

/*
 * Split-K row sum in one launch: B[i,j] = sum of A[i, j*tile : (j+1)*tile]
 * (tile = n_cols / n_split), C[i] = sum_{j} B[i,j] in j order, after event i
 * has received its n_split notifies.
 *   A fp32 [n_rows, n_cols] device, 16-byte aligned; C fp32 [n_rows] device.
 *   n_cols % n_split == 0, (n_cols / n_split) % 4 == 0, tile <= 16384,
 *   1 <= n_split <= 64.  n_rows == 0 returns ETC_OK without launching.
 *   sched: ETC_SCHED_STATIC or ETC_SCHED_DYNAMIC.
 * B and the per-row counters live in a scratch buffer the library allocates
 * on first use per device and grows as needed (freed at process exit).
 * Calls on one device must be ordered on one stream: overlapping calls share
 * that scratch.
 */
int etc_splitk_rowsum(void* stream, const float* A, long long n_rows, long long n_cols,
                      int n_split, float* C, int sched);

/*
 * etc_splitk_rowsum with a wait limit (0 -> 2 s) and fault injection:
 * debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT makes row debug_arg wait for one
 * notify more than it gets, so its final sum times out.
 */
int etc_splitk_rowsum_ex(void* stream, const float* A, long long n_rows, long long n_cols,
                         int n_split, float* C, int sched, unsigned long long wait_timeout_ns,
                         unsigned debug_flags, long long debug_arg);

/*
 * Status of the split-K calls on the current device since the last check,
 * both entry points (call it after synchronising their stream): ETC_OK, or
 * ETC_ERR_TIMEOUT with the row in etc_last_error(); the status is cleared.
 * For etc_splitk_rowsum_noalloc it reads the status word of the fixed array
 * with one synchronous 16-byte copy (nothing is allocated).
 */
int etc_splitk_check(void);

/*
 * etc_splitk_rowsum for callers that must not allocate device memory: code
 * inside an allocator or memory-pool callback that may not re-enter the
 * allocator, and runtimes that reserve all device memory up front and forbid
 * allocation afterwards.  Same arguments, result and tolerance
 * as etc_splitk_rowsum; the paper has no counterpart of this entry point.
 *
 * Its scratch (partial sums, per-row counters, queue counters, status) is a
 * fixed array of about 1.25 MiB compiled into the library: every GPU that
 * loads the library holds it until the process exits.  Limits:
 * n_rows <= 65536 and n_rows * n_split <= 262144; larger calls return
 * ETC_ERR_INVALID (use etc_splitk_rowsum instead).  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine; each call clears the
 * part of the array that must start at zero with an async memset on `stream`.
 * The first call on a device looks up the array's device address (a one-time
 * set-up, with that device current); make that first call before any stream
 * capture.  All calls on a device share the one array, so calls that overlap
 * on the GPU (other streams, other threads) race: order them on one stream.
 * A device wait that gives up (2 s) leaves the affected C rows unwritten and
 * records the site in the array's status word, which the calls do not clear:
 * until etc_splitk_check reports and clears it, the waits of later calls give
 * up at once and may leave C rows unwritten too.  Check after the calls whose
 * result matters.
 */
int etc_splitk_rowsum_noalloc(void* stream, const float* A, long long n_rows, long long n_cols,
                              int n_split, float* C, int sched);

/* Number of kernels launched by the library so far in this process. */
long long etc_launch_count(void);

/* Message of the last error on this thread ("" if none). */
const char* etc_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ETC_MOE_H_ */
