// splitk.cu -- the split-K row-sum task graph as one persistent kernel.
//
// "Event Tensor: A Unified Abstraction for Compiling Dynamic Megakernel",
// Figure 3 and podcast cue 3: partial_sum(i, j) sums row i over column tile j
// into B[i, j] and notifies event i (out_edges "ij->i", wait_count = number of
// column tiles); final_sum(i) waits on event i alone (in_edges "i->i") and
// sums B row i into C[i].  Row i is finished as soon as its own partials have
// landed, whatever the other rows are doing.
//
// GB300 layout: one CTA per SM.  Warp 0 (lane 0) streams each partial task's
// rows (R rows x one column tile, contiguous 16-byte-aligned segments) from
// HBM into a ring of shared-memory stages with bulk TMA copies; warps 1..8
// reduce a stage and notify.  Static scheduling: CTA c takes partial tasks
// c, c+G, ... and then the final sums of its row blocks, spinning on their
// events.  Dynamic scheduling: CTAs pop partial tasks from a shared counter;
// the notify that completes row i runs final_sum(i) on the spot (early push,
// popped by the same thread).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/etc_moe.h"
#include "etc_event.cuh"
#include "etc_host.h"

namespace etc {
namespace {

constexpr int kSkThreads = 320;  // warp 0 producer, 8 consumer warps, warp 9 notifier
constexpr int kSkNotifierWarp = 9;
constexpr int kSkConsumers = 256;
constexpr int kSkMaxStages = 6;
constexpr int kSkMaxRows = 8;
constexpr int kSkSmemBudget = 192 * 1024;
constexpr int kSkFinalRows = 256;

struct SkParams {
  const float* A;
  float* C;
  float* B;    // scratch [n_rows, n_split]
  int* ev;     // scratch [n_rows] count-up to n_split, reset by the final sum
  int* head;   // [2] dynamic pop counters, one per epoch parity
  long long n_rows, n_cols;
  int n_split, tile, R, stages, stage_bytes;
  long long n_tasks;
  unsigned epoch;
  int mode;
  unsigned long long timeout_ns;
  DevStatus* status;
  DevStatus* status_host;
  long long fault_row;  // row whose event waits for one notify more (-1: none)
};

constexpr int kSkNotiRing = 16;  // reduced stages waiting for their notify

struct SkCtrl {
  uint64_t full[kSkMaxStages];
  uint64_t empty[kSkMaxStages];
  uint64_t noti_full[kSkNotiRing];
  uint64_t noti_empty[kSkNotiRing];
  long long task[kSkMaxStages];
  long long noti_task[kSkNotiRing];  // partial task whose B entries are written (-1: stop)
  long long go;  // task handed to all consumers (-1: stop)
  float red[8][kSkMaxRows];
};

__device__ __forceinline__ int row_target(const SkParams& p, long long row) {
  return p.n_split + (row == p.fault_row ? 1 : 0);
}

// final_sum(i): C[i] = sum_j B[i, j], j ascending; then re-arm event i.
__device__ __forceinline__ void final_sum(const SkParams& p, long long row) {
  const float* b = p.B + row * p.n_split;
  float s = 0.f;
  for (int j = 0; j < p.n_split; ++j) s += b[j];
  p.C[row] = s;
  st_relaxed(&p.ev[row], 0);
}

__global__ void __launch_bounds__(kSkThreads, 1) splitk_kernel(const __grid_constant__ SkParams p) {
  extern __shared__ __align__(128) uint8_t sk_smem[];
  SkCtrl* ctrl = reinterpret_cast<SkCtrl*>(sk_smem);
  uint8_t* stage0 = sk_smem + ((sizeof(SkCtrl) + 127) / 128) * 128;
  const Clock clk{globaltimer_ns() + p.timeout_ns, p.status, p.status_host};
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    for (int s = 0; s < kSkNotiRing; ++s) {
      mbar_init(&ctrl->noti_full[s], 1);
      mbar_init(&ctrl->noti_empty[s], 1);
    }
    mbar_fence_init();
    if (blockIdx.x == 0)  // re-arm the other parity for the next call, whatever its mode
      st_relaxed(&p.head[(p.epoch + 1) & 1], 0);
  }
  __syncthreads();

  const long long n_row_blocks = (p.n_rows + p.R - 1) / p.R;
  const int tile_bytes = p.tile * 4;

  if (threadIdx.x == 0) {
    // ---- producer: one elected thread issues the bulk copies ----
    uint32_t it = 0;
    long long next_static = blockIdx.x;
    for (;;) {
      long long t;
      if (p.mode == ETC_SCHED_DYNAMIC) {
        t = atom_add_relaxed(&p.head[p.epoch & 1], 1);
      } else {
        t = next_static;
        next_static += G;
      }
      if (t >= p.n_tasks) t = -1;
      const int s = it % p.stages;
      if (!mbar_wait(&ctrl->empty[s], ((it / p.stages) & 1) ^ 1, clk, 100)) t = -1;
      ctrl->task[s] = t;
      if (t < 0) {
        mbar_arrive(&ctrl->full[s]);  // sentinel: no bytes
        break;
      }
      const long long rb = t / p.n_split;
      const int j = static_cast<int>(t % p.n_split);
      const int rows = static_cast<int>(min(static_cast<long long>(p.R), p.n_rows - rb * p.R));
      mbar_arrive_expect_tx(&ctrl->full[s], rows * tile_bytes);
      uint8_t* dst = stage0 + static_cast<size_t>(s) * p.stage_bytes;
      for (int r = 0; r < rows; ++r) {
        const float* src = p.A + (rb * p.R + r) * p.n_cols + static_cast<long long>(j) * p.tile;
        bulk_load(dst + r * tile_bytes, src, tile_bytes, &ctrl->full[s]);
      }
      ++it;
    }
  } else if (threadIdx.x >= 32 * kSkNotifierWarp) {
    // ---- notifier: partial_sum(i, j) notifies event i ("ij->i") ----
    // The fence and the atomics are paid here, off the consumers' path: one
    // fence covers every stage handed over so far, then one lane per row.
    const int lane = threadIdx.x & 31;
    uint32_t nit = 0;
    bool done = false;
    while (!done) {
      int n = 0;
      if (lane == 0) {
        if (mbar_wait(&ctrl->noti_full[nit % kSkNotiRing], (nit / kSkNotiRing) & 1, clk, 102)) {
          n = 1;
          while (n < 8 && mbar_try_wait(&ctrl->noti_full[(nit + n) % kSkNotiRing],
                                        ((nit + n) / kSkNotiRing) & 1))
            ++n;
        } else {
          n = -1;
        }
      }
      n = __shfl_sync(0xffffffffu, n, 0);
      if (n < 0) break;
      __syncwarp();
      __threadfence();  // the consumers' B writes (ordered by the mbarrier) before the notifies
      for (int i = 0; i < n; ++i) {
        const long long t = ctrl->noti_task[(nit + i) % kSkNotiRing];
        if (t < 0) {
          done = true;
          break;
        }
        const long long rb = t / p.n_split;
        const int rows = static_cast<int>(min(static_cast<long long>(p.R), p.n_rows - rb * p.R));
        if (lane < rows) {
          const long long row = rb * p.R + lane;
          if (p.mode == ETC_SCHED_DYNAMIC) {
            // The notify that completes row i runs final_sum(i) at once (early push).
            const int arrived = atom_add_acq_rel(&p.ev[row], 1) + 1;
            if (arrived == row_target(p, row)) final_sum(p, row);
          } else {
            red_add_relaxed(&p.ev[row], 1);
          }
        }
      }
      __syncwarp();
      if (lane == 0)
        for (int i = 0; i < n; ++i) mbar_arrive(&ctrl->noti_empty[(nit + i) % kSkNotiRing]);
      nit += n;
    }
  } else if (threadIdx.x >= 32) {
    // ---- consumers: reduce a stage, write B, hand the notify over ----
    const int ct = threadIdx.x - 32;
    const int cw = ct >> 5, lane = ct & 31;
    const int n4 = p.tile / 4;
    uint32_t nit = 0;
    auto hand_over = [&](long long t) {  // consumer thread 0 only
      const int ns = nit % kSkNotiRing;
      if (mbar_wait(&ctrl->noti_empty[ns], ((nit / kSkNotiRing) & 1) ^ 1, clk, 103)) {
        ctrl->noti_task[ns] = t;
        mbar_arrive(&ctrl->noti_full[ns]);
      }
      ++nit;
    };
    for (uint32_t it = 0;; ++it) {
      const int s = it % p.stages;
      const uint32_t par = (it / p.stages) & 1;
      // One thread does the bounded wait and broadcasts the task, so that a
      // timeout stops every consumer at the same point.
      if (ct == 0) ctrl->go = mbar_wait(&ctrl->full[s], par, clk, 101) ? ctrl->task[s] : -1;
      named_bar(1, kSkConsumers);
      const long long t = ctrl->go;
      if (t < 0) {
        if (ct == 0) hand_over(-1);
        break;
      }
      while (!mbar_try_wait(&ctrl->full[s], par)) {
      }  // phase already complete: makes the TMA bytes visible to this thread
      const long long rb = t / p.n_split;
      const int j = static_cast<int>(t % p.n_split);
      const int rows = static_cast<int>(min(static_cast<long long>(p.R), p.n_rows - rb * p.R));
      const float4* st = reinterpret_cast<const float4*>(stage0 + static_cast<size_t>(s) * p.stage_bytes);
      float part[kSkMaxRows];
#pragma unroll
      for (int r = 0; r < kSkMaxRows; ++r) {
        float acc = 0.f;
        if (r < rows) {
          const float4* row = st + r * n4;
          for (int i = ct; i < n4; i += kSkConsumers) {
            const float4 v = row[i];
            acc += (v.x + v.y) + (v.z + v.w);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        part[r] = acc;
      }
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kSkMaxRows; ++r)
          if (r < rows) ctrl->red[cw][r] = part[r];
      }
      named_bar(1, kSkConsumers);
      if (ct == 0) mbar_arrive(&ctrl->empty[s]);  // stage consumed
      if (ct < rows) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += ctrl->red[w][ct];
        const long long row = rb * p.R + ct;
        p.B[row * p.n_split + j] = v;
      }
      named_bar(1, kSkConsumers);  // B written; red[] reused next iteration
      if (ct == 0) hand_over(t);
    }
    if (p.mode == ETC_SCHED_STATIC) {
      // final_sum(i) for this CTA's row blocks, each waiting on event i ("i->i").
      const long long n_fb = (p.n_rows + kSkFinalRows - 1) / kSkFinalRows;
      for (long long fb = blockIdx.x; fb < n_fb; fb += G) {
        const long long row = fb * kSkFinalRows + ct;
        if (row < p.n_rows) {
          const int target = row_target(p, row);
          if (wait_geq(&p.ev[row], target, clk, TK_TERM, static_cast<int>(row)))
            final_sum(p, row);
        }
      }
    }
  }
  (void)n_row_blocks;
}

struct SkScratch {
  float* B = nullptr;
  int* ev = nullptr;
  int* head = nullptr;
  DevStatus* status = nullptr;
  DevStatus* status_host = nullptr;
  long long cap_B = 0, cap_rows = 0;
  unsigned epoch = 0;
  bool configured = false;
};

std::mutex g_sk_mu;
std::vector<SkScratch> g_sk;  // per device

SkScratch* scratch_for(int dev) {
  if (static_cast<int>(g_sk.size()) <= dev) g_sk.resize(dev + 1);
  return &g_sk[dev];
}

}  // namespace
}  // namespace etc

using namespace etc;

extern "C" {

int etc_splitk_rowsum_ex(void* stream, const float* A, long long n_rows, long long n_cols,
                         int n_split, float* C, int sched, unsigned long long wait_timeout_ns,
                         unsigned debug_flags, long long debug_arg) {
  clear_error();
  if (n_rows < 0 || n_cols <= 0 || n_split < 1 || n_split > 64)
    return set_error(ETC_ERR_INVALID, "splitk: bad sizes n_rows=%lld n_cols=%lld n_split=%d",
                     n_rows, n_cols, n_split);
  if (n_cols % n_split != 0 || (n_cols / n_split) % 4 != 0 || n_cols / n_split > 16384)
    return set_error(ETC_ERR_INVALID,
                     "splitk: tile = n_cols/n_split must be a multiple of 4 and <= 16384");
  if (sched != ETC_SCHED_STATIC && sched != ETC_SCHED_DYNAMIC)
    return set_error(ETC_ERR_INVALID, "splitk: bad sched %d", sched);
  if ((debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT) && sched != ETC_SCHED_STATIC)
    return set_error(ETC_ERR_UNIMPLEMENTED, "splitk: fault injection needs the static scheduler");
  if (n_rows == 0) return ETC_OK;
  if (!A || !C || !aligned16(A))
    return set_error(ETC_ERR_INVALID, "splitk: A and C must be device pointers, A 16-byte aligned");

  int dev = 0;
  ETC_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_sk_mu);
  SkScratch* sc = scratch_for(dev);
  const long long need_B = n_rows * n_split;
  if (!sc->status) {
    ETC_CUDA_TRY(cudaMalloc(&sc->status, sizeof(DevStatus)));
    ETC_CUDA_TRY(cudaMemset(sc->status, 0, sizeof(DevStatus)));
    ETC_CUDA_TRY(cudaHostAlloc(&sc->status_host, sizeof(DevStatus), cudaHostAllocMapped));
    std::memset(sc->status_host, 0, sizeof(DevStatus));
    ETC_CUDA_TRY(cudaMalloc(&sc->head, 2 * sizeof(int)));
    ETC_CUDA_TRY(cudaMemset(sc->head, 0, 2 * sizeof(int)));
  }
  if (sc->cap_B < need_B || sc->cap_rows < n_rows) {
    // cudaFree waits for work in flight that may still use the old scratch.
    if (sc->B) cudaFree(sc->B);
    if (sc->ev) cudaFree(sc->ev);
    sc->B = nullptr;
    sc->ev = nullptr;
    sc->cap_B = sc->cap_rows = 0;
    ETC_CUDA_TRY(cudaMalloc(&sc->B, need_B * sizeof(float)));
    ETC_CUDA_TRY(cudaMalloc(&sc->ev, n_rows * sizeof(int)));
    ETC_CUDA_TRY(cudaMemset(sc->ev, 0, n_rows * sizeof(int)));
    sc->cap_B = need_B;
    sc->cap_rows = n_rows;
  }
  if (!sc->configured) {
    ETC_CUDA_TRY(cudaFuncSetAttribute(splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSkSmemBudget + 1024));
    sc->configured = true;
  }
  DevStatus hs;
  std::memcpy(&hs, sc->status_host, sizeof hs);
  if (hs.code != 0)
    return set_error(ETC_ERR_STATE, "splitk: an earlier call timed out; call etc_splitk_check");

  SkParams p{};
  p.A = A;
  p.C = C;
  p.B = sc->B;
  p.ev = sc->ev;
  p.head = sc->head;
  p.n_rows = n_rows;
  p.n_cols = n_cols;
  p.n_split = n_split;
  p.tile = static_cast<int>(n_cols / n_split);
  const int tile_bytes = p.tile * 4;
  p.R = std::max(1, std::min(kSkMaxRows, 65536 / tile_bytes));
  p.stage_bytes = p.R * tile_bytes;
  p.stages = std::max(2, std::min(kSkMaxStages, kSkSmemBudget / p.stage_bytes));
  p.n_tasks = ((n_rows + p.R - 1) / p.R) * n_split;
  if (++sc->epoch == 0) sc->epoch = 1;
  p.epoch = sc->epoch;
  p.mode = sched;
  p.timeout_ns = wait_timeout_ns ? wait_timeout_ns : 2000000000ull;
  p.status = sc->status;
  p.status_host = sc->status_host;
  p.fault_row = (debug_flags & ETC_DEBUG_FAULT_EXTRA_WAIT) ? debug_arg : -1;
  const size_t smem = ((sizeof(SkCtrl) + 127) / 128) * 128 + static_cast<size_t>(p.stages) * p.stage_bytes;

  int occ = 0;
  ETC_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, splitk_kernel, kSkThreads, smem));
  if (occ < 1) return set_error(ETC_ERR_CUDA, "splitk: kernel does not fit on an SM");
  const int grid = sm_count(dev) * occ;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: spin-waits are safe
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ETC_CUDA_TRY(cudaLaunchKernelEx(&cfg, splitk_kernel, p));
  g_launches.fetch_add(1);
  return ETC_OK;
}

namespace etc {
int noalloc_check(int dev);
}

int etc_splitk_rowsum(void* stream, const float* A, long long n_rows, long long n_cols,
                      int n_split, float* C, int sched) {
  return etc_splitk_rowsum_ex(stream, A, n_rows, n_cols, n_split, C, sched, 0, 0, -1);
}

int etc_splitk_check(void) {
  clear_error();
  int dev = 0;
  ETC_CUDA_TRY(cudaGetDevice(&dev));
  const int na = etc::noalloc_check(dev);  // the no-allocation entry point's status word
  if (na != ETC_OK) return na;
  std::lock_guard<std::mutex> lk(g_sk_mu);
  SkScratch* sc = scratch_for(dev);
  if (!sc->status_host) return ETC_OK;
  DevStatus hs;
  std::memcpy(&hs, sc->status_host, sizeof hs);
  if (hs.code == 0) return ETC_OK;
  // Clear for the next call: counters of unfinished rows are re-armed too.
  std::memset(sc->status_host, 0, sizeof(DevStatus));
  ETC_CUDA_TRY(cudaMemset(sc->status, 0, sizeof(DevStatus)));
  if (sc->ev) ETC_CUDA_TRY(cudaMemset(sc->ev, 0, sc->cap_rows * sizeof(int)));
  ETC_CUDA_TRY(cudaMemset(sc->head, 0, 2 * sizeof(int)));
  return set_error(ETC_ERR_TIMEOUT, "splitk: device wait timed out (code %d, site %d, row %d, cta %d)",
                   hs.code, hs.where, hs.aux, hs.cta);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Split-K row sum that allocates nothing.
//
// Some callers cannot call cudaMalloc at the moment they need this operation:
// code inside an allocator or a memory-pool callback that must not re-enter
// the allocator, and runtimes that reserve all device memory up front and
// forbid allocation later.  For them the scratch this kernel needs (the per-row partial sums B,
// the per-row event counters and the queue counters) lives in one fixed-size
// array in the library's device image instead of a buffer from cudaMalloc.
// The array exists on every GPU that loads the library and stays there until
// the process exits.
// ---------------------------------------------------------------------------
namespace etc {
namespace {

constexpr long long kNoAllocMaxRows = 65536;           // n_rows limit
constexpr long long kNoAllocMaxPartials = 262144;      // n_rows * n_split limit
constexpr size_t kNoAllocHeader = 256;                 // status + queue counters
constexpr size_t kNoAllocCleared = 128;                // first byte a call clears (the queue counters)
constexpr size_t kNoAllocBytes =
    kNoAllocHeader + kNoAllocMaxRows * sizeof(int) + kNoAllocMaxPartials * sizeof(float);

// Layout: [DevStatus | pad to 128] [head[2] | pad to 256] [ev: int x 65536] [B: float x 262144].
// The status word sits outside what a call clears: it keeps the first wait
// that gave up until etc_splitk_check reads and clears it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch on this device
  unsigned epoch = 0;
};
std::mutex g_na_mu;
NoAllocDevice g_na[64];

}  // namespace

// Reads (and clears) the status word the no-allocation calls on device `dev`
// share: a synchronous 16-byte copy out of the fixed array, nothing allocated.
int noalloc_check(int dev) {
  if (dev < 0 || dev >= 64) return ETC_OK;
  std::lock_guard<std::mutex> lk(g_na_mu);
  NoAllocDevice& nd = g_na[dev];
  if (!nd.base) return ETC_OK;  // no call on this device yet
  DevStatus hs;
  ETC_CUDA_TRY(cudaMemcpy(&hs, nd.base, sizeof hs, cudaMemcpyDeviceToHost));
  if (hs.code == 0) return ETC_OK;
  ETC_CUDA_TRY(cudaMemset(nd.base, 0, sizeof(DevStatus)));
  return set_error(ETC_ERR_TIMEOUT,
                   "splitk_noalloc: device wait timed out (code %d, site %d, row %d, cta %d)",
                   hs.code, hs.where, hs.aux, hs.cta);
}

}  // namespace etc

extern "C" int etc_splitk_rowsum_noalloc(void* stream, const float* A, long long n_rows,
                                         long long n_cols, int n_split, float* C, int sched) {
  using namespace etc;
  clear_error();
  if (n_rows < 0 || n_cols <= 0 || n_split < 1 || n_split > 64)
    return set_error(ETC_ERR_INVALID, "splitk_noalloc: bad sizes n_rows=%lld n_cols=%lld n_split=%d",
                     n_rows, n_cols, n_split);
  if (n_cols % n_split != 0 || (n_cols / n_split) % 4 != 0 || n_cols / n_split > 16384)
    return set_error(ETC_ERR_INVALID,
                     "splitk_noalloc: tile = n_cols/n_split must be a multiple of 4 and <= 16384");
  if (n_rows > kNoAllocMaxRows || n_rows * n_split > kNoAllocMaxPartials)
    return set_error(ETC_ERR_INVALID,
                     "splitk_noalloc: n_rows=%lld, n_rows*n_split=%lld exceed the fixed scratch "
                     "(at most %lld rows and %lld partial sums); use etc_splitk_rowsum",
                     n_rows, n_rows * n_split, kNoAllocMaxRows, kNoAllocMaxPartials);
  if (sched != ETC_SCHED_STATIC && sched != ETC_SCHED_DYNAMIC)
    return set_error(ETC_ERR_INVALID, "splitk_noalloc: bad sched %d", sched);
  if (n_rows == 0) return ETC_OK;
  if (!A || !C || !aligned16(A))
    return set_error(ETC_ERR_INVALID,
                     "splitk_noalloc: A and C must be device pointers, A 16-byte aligned");
  int dev = 0;
  ETC_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return set_error(ETC_ERR_INVALID, "splitk_noalloc: device %d", dev);

  std::lock_guard<std::mutex> lk(g_na_mu);
  NoAllocDevice& nd = g_na[dev];
  if (!nd.base) {
    // One-time set-up on this device (the current one): the host-side name of
    // the array is not a device address, so ask the runtime for it.
    void* ptr = nullptr;
    ETC_CUDA_TRY(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
    ETC_CUDA_TRY(cudaFuncSetAttribute(splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSkSmemBudget + 1024));
    nd.base = static_cast<unsigned char*>(ptr);
  }
  int* ev = reinterpret_cast<int*>(nd.base + kNoAllocHeader);
  float* B = reinterpret_cast<float*>(nd.base + kNoAllocHeader + kNoAllocMaxRows * sizeof(int));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Queue counters and this call's row counters must start at zero; the array
  // keeps whatever the previous call left there.  (Not the status word.)
  ETC_CUDA_TRY(cudaMemsetAsync(nd.base + kNoAllocCleared, 0,
                               kNoAllocHeader - kNoAllocCleared + n_rows * sizeof(int), s));

  SkParams p{};
  p.A = A;
  p.C = C;
  p.B = B;
  p.ev = ev;
  p.head = reinterpret_cast<int*>(nd.base + kNoAllocCleared);
  p.n_rows = n_rows;
  p.n_cols = n_cols;
  p.n_split = n_split;
  p.tile = static_cast<int>(n_cols / n_split);
  const int tile_bytes = p.tile * 4;
  p.R = std::max(1, std::min(kSkMaxRows, 65536 / tile_bytes));
  p.stage_bytes = p.R * tile_bytes;
  p.stages = std::max(2, std::min(kSkMaxStages, kSkSmemBudget / p.stage_bytes));
  p.n_tasks = ((n_rows + p.R - 1) / p.R) * n_split;
  if (++nd.epoch == 0) nd.epoch = 1;
  p.epoch = nd.epoch;
  p.mode = sched;
  p.timeout_ns = 2000000000ull;
  p.status = reinterpret_cast<DevStatus*>(nd.base);
  p.status_host = nullptr;
  p.fault_row = -1;
  const size_t smem =
      ((sizeof(SkCtrl) + 127) / 128) * 128 + static_cast<size_t>(p.stages) * p.stage_bytes;
  int occ = 0;
  ETC_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, splitk_kernel, kSkThreads, smem));
  if (occ < 1) return set_error(ETC_ERR_CUDA, "splitk_noalloc: kernel does not fit on an SM");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count(dev) * occ);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ETC_CUDA_TRY(cudaLaunchKernelEx(&cfg, splitk_kernel, p));
  g_launches.fetch_add(1);
  return ETC_OK;
}
