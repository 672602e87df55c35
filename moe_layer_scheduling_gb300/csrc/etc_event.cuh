// etc_event.cuh -- Event Tensor primitives on the device: bounded waits on
// global-memory counters and flags, notify, error reporting, and the
// lock-free task queue of the dynamic scheduler.
//
// Semantics follow the Event Tensor pages ("Event Tensor: A Unified
// Abstraction for Compiling Dynamic Megakernel", Figures 7 and 9, podcast
// cue 11): an event counter starts at its wait_count and every notify takes
// one off; the waiter is released at zero.  In the dynamic form the notify
// that brings a counter to zero pushes the now-ready task into a shared queue
// at once ("early push"), and idle SMs pop from it.
#pragma once

#include "etc_internal.h"
#include "etc_ptx.cuh"

namespace etc {

struct Clock {
  uint64_t deadline;
  DevStatus* st;
  DevStatus* st_host;
};

__device__ __forceinline__ bool error_raised(const Clock& c) {
  return ld_relaxed(&c.st->code) != 0;
}

static __device__ __noinline__ void raise_error(const Clock& c, int code, int where, int aux) {
  if (atom_cas_relaxed(&c.st->code, 0, code) == 0) {
    c.st->where = where;
    c.st->aux = aux;
    c.st->cta = blockIdx.x;
    if (c.st_host) {
      volatile DevStatus* h = c.st_host;
      h->where = where;
      h->aux = aux;
      h->cta = blockIdx.x;
      __threadfence_system();
      h->code = code;
    }
    __threadfence();
  }
}

// Spins until pred() holds.  Returns false once the deadline passes (after
// recording a timeout) or once another CTA has recorded an error.
template <class Pred>
__device__ __forceinline__ bool spin_until(Pred pred, const Clock& c, int code, int where,
                                           int aux) {
  uint32_t it = 0;
  while (!pred()) {
    if ((++it & 31u) == 0) {
      if (error_raised(c)) return false;
      if (globaltimer_ns() > c.deadline) {
        raise_error(c, code, where, aux);
        return false;
      }
    }
    __nanosleep(20);
  }
  return true;
}

// Count-down event: ready when the counter reaches zero.
__device__ __forceinline__ bool wait_zero(const int* ev, const Clock& c, int where, int aux) {
  return spin_until([&] { return ld_acquire(ev) <= 0; }, c, DERR_TIMEOUT_EVENT, where, aux);
}
// Count-up event: ready when the counter reaches `target`.
__device__ __forceinline__ bool wait_geq(const int* ev, int target, const Clock& c, int where,
                                         int aux) {
  return spin_until([&] { return ld_acquire(ev) >= target; }, c, DERR_TIMEOUT_EVENT, where,
                    aux);
}
// One-shot flag carrying the call's epoch.
__device__ __forceinline__ bool wait_flag(const unsigned* f, unsigned epoch, const Clock& c,
                                          int where, int aux) {
  return spin_until([&] { return ld_acquire(f) == epoch; }, c, DERR_TIMEOUT_EVENT, where, aux);
}
// Notify: takes n off a count-down event; returns the value after the notify.
// acq_rel: publishes this thread's (and, through the barrier before it, its
// CTA's) writes and acquires those of earlier notifiers.
__device__ __forceinline__ int notify(int* ev, int n) { return atom_add_acq_rel(ev, -n) - n; }

// Bounded mbarrier wait used inside a CTA.  `cluster`: the barrier may be
// completed from the pair peer CTA or by a pair MMA (cluster-scope acquire).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Clock& c,
                                          int where, bool cluster = false) {
  auto tw = [&] { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (tw()) return true;
  uint32_t it = 0;
  while (!tw()) {
    if ((++it & 255u) == 0 && globaltimer_ns() > c.deadline + 1000000000ull) {
      raise_error(c, DERR_TIMEOUT_MBAR, where, 0);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// Dynamic task queue.  Slot i holds (epoch << 32 | descriptor) once written;
// slots [0, n_seed) are implicit (the initially ready tasks) and are never
// stored.  head/tail are reset for the next call of the same parity by the
// current call, so no call has to clear its own queue before using it.
// ---------------------------------------------------------------------------
struct QueueView {
  unsigned long long* slots;
  int* head;
  int* tail;
  int cap;
  int n_seed;
  unsigned epoch;
};

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Pushes n tasks desc_of(0..n-1); the caller's earlier writes become visible
// to whoever pops them.
template <class DescOf>
__device__ __forceinline__ void queue_push(const QueueView& q, int n, DescOf desc_of,
                                           const Clock& c) {
  if (n <= 0) return;
  __threadfence();
  const int base = q.n_seed + atom_add_relaxed(q.tail, n);
  for (int i = 0; i < n; ++i) {
    const int idx = base + i;
    if (idx >= q.cap) {
      raise_error(c, DERR_QUEUE_OVERFLOW, 0, idx);
      return;
    }
    st_relaxed_u64(&q.slots[idx],
                   (static_cast<unsigned long long>(q.epoch) << 32) | desc_of(i));
  }
}

}  // namespace etc
