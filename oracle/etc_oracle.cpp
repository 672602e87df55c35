// etc_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously correct CPU restatement, in fp64, of what the
// Event Tensor MoE layer, the split-K row sum and the RMSNorm -> MoE -> residual
// chain compute.  Only the test suite, the smoke check and the benchmark's CPU
// baseline leg may load this library; the CUDA path never calls it and the two
// share no code, headers or tables.
//
// Sources (all from the pages on "Event Tensor: A Unified Abstraction for
// Compiling Dynamic Megakernel"):
//   * MoE subgraph and its runtime tensors topk / exp_indptr: Figure 2 and
//     Figure 5(b) captions of the paper summary page.
//   * exp_indptr = prefix sum of tokens per expert, expert i owns the range
//     [exp_indptr[i], exp_indptr[i+1]): podcast transcript, cue 9.
//   * Per-expert wait_count = number of tokens the router gave the expert:
//     podcast transcript, cue 7.
//   * Split-K example (partial_sum(i,j) -> B, final_sum(i) sums B row i into C,
//     ETensor of shape n with wait_count 4, out_edges "ij->i", in_edges "i->i"):
//     Figure 3 caption and podcast transcript, cue 3.
//   * Count-down semantics of an event (starts at its wait_count, each notify
//     takes one off, ready at zero): podcast transcript, cue 11.
//
// Readings where the pages are silent (each listed in the design notes):
//   * top-k selects on the logits ordered by (value descending, expert id
//     ascending); weights are the softmax restricted to the k selected logits,
//     which equals a full softmax renormalised over the selected experts.
//   * Within an expert's row range, rows follow ascending token index.
//   * W_gate_up[e] holds the I gate rows first, then the I up rows; the
//     activation is silu(gate) * up with silu(z) = z / (1 + exp(-z)).
//   * The dense MLP of the appendix's Table 4 applies that same FFN to every
//     row with one weight set.
//   * The chain block is x <- x + MoE(RMSNorm(x)), RMSNorm(x) = x /
//     sqrt(mean(x^2) + eps) * g.
//
// Every floating-point step is done in double with no intermediate rounding;
// bf16 inputs are widened exactly.  Sums run in index order.
//
// Parity pins (closed forms, brute force, invariants) live in tests/.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <random>
#include <string>
#include <thread>
#include <vector>

namespace {

inline double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

int g_threads = 0;  // 0 = hardware concurrency

int thread_count() {
  if (g_threads > 0) return g_threads;
  unsigned hc = std::thread::hardware_concurrency();
  return hc == 0 ? 1 : static_cast<int>(hc);
}

// Runs fn(i) for i in [0, n) over a pool of threads, dynamic chunks of 1.
template <class Fn>
void parallel_for(long n, Fn fn) {
  int nt = std::min<long>(thread_count(), std::max<long>(n, 1));
  if (nt <= 1) {
    for (long i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<long> next{0};
  std::vector<std::thread> pool;
  pool.reserve(nt);
  for (int t = 0; t < nt; ++t) {
    pool.emplace_back([&]() {
      for (;;) {
        long i = next.fetch_add(1);
        if (i >= n) break;
        fn(i);
      }
    });
  }
  for (auto& th : pool) th.join();
}

// --- MoE steps -------------------------------------------------------------

// Router: logits[t,e] = sum_h x[t,h] * Wg[h,e] (+ bias[e]).  Wg is [H, E].
void router_logits(const uint16_t* x, const uint16_t* wg, const float* bias,
                   long T, int H, int E, double* logits) {
  parallel_for(T, [&](long t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += bf16_to_double(x[t * H + h]) * bf16_to_double(wg[static_cast<long>(h) * E + e]);
      if (bias) s += static_cast<double>(bias[e]);
      logits[t * E + e] = s;
    }
  });
}

// Weights of a token's k selected experts ids[0..k-1]:
// w_j = exp(L_j - L_0) / sum_j' exp(L_j' - L_0), the softmax over the selected
// logits (L_0 the logit of the first selected expert).
template <class Real>
void selected_weights(const Real* L, int k, const int32_t* ids, double* w) {
  const double l0 = static_cast<double>(L[ids[0]]);
  double z = 0.0;
  for (int j = 0; j < k; ++j) z += std::exp(static_cast<double>(L[ids[j]]) - l0);
  for (int j = 0; j < k; ++j) w[j] = std::exp(static_cast<double>(L[ids[j]]) - l0) / z;
}

// Routing for one token: the k largest logits, ties to the lower expert id,
// then the softmax over the selected k.
template <class Real>
void route_token(const Real* L, int E, int k, int32_t* ids, double* w) {
  std::vector<char> taken(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      // Strict '>' while scanning e upward keeps the lowest id among equals.
      if (best < 0 || static_cast<double>(L[e]) > static_cast<double>(L[best])) best = e;
    }
    taken[best] = 1;
    ids[j] = best;
  }
  selected_weights(L, k, ids, w);
}

// Dispatch: per-expert counts, exp_indptr (exclusive prefix sum of the counts),
// and the stable permutation: the row of slot (t, j) is exp_indptr[e] plus the
// number of earlier tokens routed to the same expert e.
void dispatch(const int32_t* ids, long T, int E, int k, int32_t* counts,
              int32_t* exp_indptr, int32_t* pos, int32_t* row_token) {
  std::vector<long> cnt(E, 0);
  for (long s = 0; s < T * k; ++s) cnt[ids[s]] += 1;
  exp_indptr[0] = 0;
  for (int e = 0; e < E; ++e) {
    counts[e] = static_cast<int32_t>(cnt[e]);
    exp_indptr[e + 1] = exp_indptr[e] + counts[e];
  }
  std::vector<long> seen(E, 0);
  for (long t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      const long r = exp_indptr[e] + seen[e]++;
      pos[t * k + j] = static_cast<int32_t>(r);
      if (row_token) row_token[r] = static_cast<int32_t>(t);
    }
  }
}

// Expert FFN on one input row: g = x Wg^T, u = x Wu^T, a = silu(g) * u, y = a Wd^T.
void expert_ffn(const double* xrow, const uint16_t* wgu_e, const uint16_t* wd_e, int H,
                int I, double* act, double* y) {
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    const uint16_t* wg_row = wgu_e + static_cast<long>(n) * H;
    const uint16_t* wu_row = wgu_e + static_cast<long>(I + n) * H;
    for (int h = 0; h < H; ++h) {
      g += xrow[h] * bf16_to_double(wg_row[h]);
      u += xrow[h] * bf16_to_double(wu_row[h]);
    }
    act[n] = g / (1.0 + std::exp(-g)) * u;
  }
  for (int m = 0; m < H; ++m) {
    double s = 0.0;
    const uint16_t* wd_row = wd_e + static_cast<long>(m) * I;
    for (int n = 0; n < I; ++n) s += act[n] * bf16_to_double(wd_row[n]);
    y[m] = s;
  }
}

// One MoE layer on fp64 input rows xin[T, H] (already widened).  ids_in
// (nullable, [T, k]): the experts each token is routed to, given instead of
// selected from the logits (the weights are still the softmax of this layer's
// own logits over the given experts).
void moe_layer_f64(const double* xin, const uint16_t* x_bf16_for_router, const uint16_t* wg,
                   const float* bias, const uint16_t* wgu, const uint16_t* wd, long T, int H,
                   int E, int k, int I, double* out, double* logits_out, int32_t* ids_out,
                   double* w_out, const int32_t* ids_in = nullptr) {
  std::vector<double> logits(static_cast<size_t>(T) * E);
  if (x_bf16_for_router) {
    router_logits(x_bf16_for_router, wg, bias, T, H, E, logits.data());
  } else {
    parallel_for(T, [&](long t) {
      for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int h = 0; h < H; ++h)
          s += xin[t * H + h] * bf16_to_double(wg[static_cast<long>(h) * E + e]);
        if (bias) s += static_cast<double>(bias[e]);
        logits[t * E + e] = s;
      }
    });
  }
  std::vector<int32_t> ids(static_cast<size_t>(T) * k);
  std::vector<double> w(static_cast<size_t>(T) * k);
  parallel_for(T, [&](long t) {
    if (ids_in) {
      std::copy(ids_in + t * k, ids_in + (t + 1) * k, &ids[t * k]);
      selected_weights(&logits[t * E], k, &ids[t * k], &w[t * k]);
    } else {
      route_token(&logits[t * E], E, k, &ids[t * k], &w[t * k]);
    }
  });

  std::vector<int32_t> counts(E), exp_indptr(E + 1), pos(static_cast<size_t>(T) * k),
      row_token(static_cast<size_t>(T) * k);
  dispatch(ids.data(), T, E, k, counts.data(), exp_indptr.data(), pos.data(), row_token.data());

  // Expert e computes the rows [exp_indptr[e], exp_indptr[e+1]) of the
  // permuted activations; each row is the FFN of its token's input.
  const long R = T * k;
  std::vector<double> y(static_cast<size_t>(R) * H);
  std::vector<int32_t> row_expert(R);
  for (int e = 0; e < E; ++e)
    for (long r = exp_indptr[e]; r < exp_indptr[e + 1]; ++r) row_expert[r] = e;
  parallel_for(R, [&](long r) {
    std::vector<double> act(I);
    const int e = row_expert[r];
    expert_ffn(xin + static_cast<long>(row_token[r]) * H,
               wgu + static_cast<long>(e) * 2 * I * H, wd + static_cast<long>(e) * H * I, H, I,
               act.data(), &y[r * H]);
  });
  // Weighted combine: out[t] = sum_j w[t,j] * y[pos[t,j]], j ascending.
  parallel_for(T, [&](long t) {
    for (int m = 0; m < H; ++m) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) s += w[t * k + j] * y[static_cast<long>(pos[t * k + j]) * H + m];
      out[t * H + m] = s;
    }
  });
  if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
  if (ids_out) std::copy(ids.begin(), ids.end(), ids_out);
  if (w_out) std::copy(w.begin(), w.end(), w_out);
}

// --- index maps for the event-graph simulator ------------------------------

// Parses an affine index map written like "ij->i": every letter on the left
// names a task coordinate; the right side picks coordinates by letter.
struct IndexMap {
  std::vector<int> pick;  // for each output coord, the index of the input coord
  bool parse(const char* spec) {
    std::string s(spec);
    size_t arrow = s.find("->");
    if (arrow == std::string::npos) return false;
    std::string lhs = s.substr(0, arrow), rhs = s.substr(arrow + 2);
    pick.clear();
    for (char c : rhs) {
      size_t p = lhs.find(c);
      if (p == std::string::npos) return false;
      pick.push_back(static_cast<int>(p));
    }
    return true;
  }
};

}  // namespace

extern "C" {

void oracle_set_threads(int n) { g_threads = n; }
int oracle_get_threads(void) { return thread_count(); }

// Router logits in fp64, [T, E].
int oracle_router_logits(const uint16_t* x, const uint16_t* wg, const float* bias, long T, int H,
                         int E, double* logits) {
  if (T < 0 || H <= 0 || E <= 0) return -1;
  router_logits(x, wg, bias, T, H, E, logits);
  return 0;
}

// Routing from fp64 logits: ids [T, k], weights [T, k].
int oracle_route_f64(const double* L, long T, int E, int k, int32_t* ids, double* w) {
  if (k <= 0 || k > E) return -1;
  for (long t = 0; t < T; ++t) route_token(L + t * E, E, k, ids + t * k, w + t * k);
  return 0;
}

// Routing from fp32 logits (the same rule, compared in double: exact for fp32).
int oracle_route_f32(const float* L, long T, int E, int k, int32_t* ids, double* w) {
  if (k <= 0 || k > E) return -1;
  for (long t = 0; t < T; ++t) route_token(L + t * E, E, k, ids + t * k, w + t * k);
  return 0;
}

// counts [E], exp_indptr [E+1], pos [T, k], row_token [T*k] (nullable).
int oracle_dispatch(const int32_t* ids, long T, int E, int k, int32_t* counts, int32_t* exp_indptr,
                    int32_t* pos, int32_t* row_token) {
  for (long s = 0; s < T * k; ++s)
    if (ids[s] < 0 || ids[s] >= E) return -1;
  dispatch(ids, T, E, k, counts, exp_indptr, pos, row_token);
  return 0;
}

// One expert FFN on one bf16 input row (for closed-form pins).
int oracle_expert_ffn(const uint16_t* x, const uint16_t* wgu_e, const uint16_t* wd_e, int H, int I,
                      double* y) {
  std::vector<double> xr(H), act(I);
  for (int h = 0; h < H; ++h) xr[h] = bf16_to_double(x[h]);
  expert_ffn(xr.data(), wgu_e, wd_e, H, I, act.data(), y);
  return 0;
}

// Dense MLP on chosen rows of x: out[i] = FFN(x[rows[i]]) with the single
// weight set w_gate_up bf16 [2I,H] (gate rows, then up rows) and w_down bf16
// [H,I].  The paper summary page's appendix Table 4 gives the MLP shapes (S,
// H, I) but no activation; the FFN is read as the experts' silu(gate) * up.
// rows == NULL takes rows 0 .. n-1 (n <= T); out is fp64 [n, H].
int oracle_mlp(const uint16_t* x, const uint16_t* wgu, const uint16_t* wd, long T, int H, int I,
               const int64_t* rows, long n, double* out) {
  if (T < 0 || H <= 0 || I <= 0 || n < 0 || (!rows && n > T)) return -1;
  for (long i = 0; rows && i < n; ++i)
    if (rows[i] < 0 || rows[i] >= T) return -1;
  parallel_for(n, [&](long i) {
    const long t = rows ? static_cast<long>(rows[i]) : i;
    std::vector<double> xr(H), act(I);
    for (int h = 0; h < H; ++h) xr[h] = bf16_to_double(x[t * H + h]);
    expert_ffn(xr.data(), wgu, wd, H, I, act.data(), out + i * H);
  });
  return 0;
}

// Full MoE layer: x bf16 [T,H], gate_w bf16 [H,E], bias fp32 [E] (nullable),
// w_gate_up bf16 [E,2I,H], w_down bf16 [E,H,I] -> out fp64 [T,H].
// logits_out [T,E], ids_out [T,k], w_out [T,k] are optional.
int oracle_moe_layer(const uint16_t* x, const uint16_t* wg, const float* bias, const uint16_t* wgu,
                     const uint16_t* wd, long T, int H, int E, int k, int I, double* out,
                     double* logits_out, int32_t* ids_out, double* w_out) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || I <= 0) return -1;
  std::vector<double> xin(static_cast<size_t>(T) * H);
  for (long i = 0; i < T * H; ++i) xin[i] = bf16_to_double(x[i]);
  moe_layer_f64(xin.data(), x, wg, bias, wgu, wd, T, H, E, k, I, out, logits_out, ids_out, w_out);
  return 0;
}

// Chain of n_blocks blocks x <- x + MoE_b(RMSNorm_b(x)); all pointers are
// arrays of n_blocks per-block tensors.  ids_out: [n_blocks, T, k] (nullable),
// logits_out: [n_blocks, T, E] (nullable), ids_in: [n_blocks, T, k] (nullable)
// routing given for every block instead of selected (see moe_layer_f64).
int oracle_chain_routed(const uint16_t* x, int n_blocks, const uint16_t* const* norm_w,
                        const uint16_t* const* wg, const float* const* bias,
                        const uint16_t* const* wgu, const uint16_t* const* wd, long T, int H,
                        int E, int k, int I, double eps, double* out, int32_t* ids_out,
                        double* logits_out, const int32_t* ids_in) {
  if (T < 0 || n_blocks <= 0) return -1;
  if (ids_in)
    for (long i = 0; i < static_cast<long>(n_blocks) * T * k; ++i)
      if (ids_in[i] < 0 || ids_in[i] >= E) return -1;
  std::vector<double> cur(static_cast<size_t>(T) * H), normed(static_cast<size_t>(T) * H),
      delta(static_cast<size_t>(T) * H);
  for (long i = 0; i < T * H; ++i) cur[i] = bf16_to_double(x[i]);
  for (int b = 0; b < n_blocks; ++b) {
    parallel_for(T, [&](long t) {
      double ss = 0.0;
      for (int h = 0; h < H; ++h) ss += cur[t * H + h] * cur[t * H + h];
      const double inv = 1.0 / std::sqrt(ss / H + eps);
      for (int h = 0; h < H; ++h)
        normed[t * H + h] = cur[t * H + h] * inv * bf16_to_double(norm_w[b][h]);
    });
    moe_layer_f64(normed.data(), nullptr, wg[b], bias ? bias[b] : nullptr, wgu[b], wd[b], T, H, E,
                  k, I, delta.data(), logits_out ? logits_out + static_cast<long>(b) * T * E : nullptr,
                  ids_out ? ids_out + static_cast<long>(b) * T * k : nullptr, nullptr,
                  ids_in ? ids_in + static_cast<long>(b) * T * k : nullptr);
    for (long i = 0; i < T * H; ++i) cur[i] += delta[i];
  }
  std::copy(cur.begin(), cur.end(), out);
  return 0;
}

int oracle_chain(const uint16_t* x, int n_blocks, const uint16_t* const* norm_w,
                 const uint16_t* const* wg, const float* const* bias, const uint16_t* const* wgu,
                 const uint16_t* const* wd, long T, int H, int E, int k, int I, double eps,
                 double* out, int32_t* ids_out, double* logits_out) {
  return oracle_chain_routed(x, n_blocks, norm_w, wg, bias, wgu, wd, T, H, E, k, I, eps, out,
                             ids_out, logits_out, nullptr);
}

// Split-K row sum: B[i,j] = sum of row i over column tile j, C[i] = sum_j B[i,j].
int oracle_splitk(const float* A, long n_rows, long n_cols, int n_split, double* B, double* C) {
  if (n_split <= 0 || n_cols % n_split != 0) return -1;
  const long tile = n_cols / n_split;
  parallel_for(n_rows, [&](long i) {
    double c = 0.0;
    for (int j = 0; j < n_split; ++j) {
      double s = 0.0;
      for (long col = j * tile; col < (j + 1) * tile; ++col) s += A[i * n_cols + col];
      if (B) B[i * n_split + j] = s;
      c += s;
    }
    C[i] = c;
  });
  return 0;
}

// Event-graph simulator for the split-K program: producer tasks partial(i,j)
// over the grid [n_rows, n_split] notify the events named by out_map; consumer
// tasks final(i) over [n_rows] wait on the events named by in_map.  Every event
// starts at wait_count and is ready at zero.  Ready tasks run in a random order
// drawn from `seed`.  Partial values are part_val[i*n_split+j]; final(i) sums
// its row's partials in j order into C[i].
//
// Outputs: notifies[i] = notifies event i received; early = number of
// consumers that started while one of their events was non-zero (always 0 for
// a correct graph); order[] = the executed task sequence (>=0: partial index
// i*n_split+j, <0: -(i+1) for final(i)).  Returns the number of tasks run.
long oracle_event_sim(long n_rows, int n_split, int wait_count, const char* out_map,
                      const char* in_map, unsigned long long seed, const double* part_val,
                      double* C, int32_t* notifies, int32_t* early, int64_t* order) {
  IndexMap om, im;
  if (!om.parse(out_map) || !im.parse(in_map)) return -1;
  if (om.pick.size() != 1 || im.pick.size() != 1) return -1;  // rank-1 event tensor
  std::vector<long> counter(n_rows, wait_count);
  std::vector<int32_t> notes(n_rows, 0);
  std::vector<double> B(static_cast<size_t>(n_rows) * n_split, 0.0);
  std::mt19937_64 rng(seed);
  // Ready set: all producers initially; a consumer joins when its event hits 0.
  std::vector<int64_t> ready;
  ready.reserve(n_rows * n_split + n_rows);
  for (long i = 0; i < n_rows; ++i)
    for (int j = 0; j < n_split; ++j) ready.push_back(i * n_split + j);
  std::vector<char> final_queued(n_rows, 0);
  if (wait_count <= 0) {  // an event with nothing to wait for is ready at launch
    for (long i = 0; i < n_rows; ++i) {
      final_queued[i] = 1;
      ready.push_back(-(i + 1));
    }
  }
  long ran = 0, early_count = 0;
  while (!ready.empty()) {
    std::uniform_int_distribution<size_t> pickd(0, ready.size() - 1);
    size_t p = pickd(rng);
    int64_t task = ready[p];
    ready[p] = ready.back();
    ready.pop_back();
    if (order) order[ran] = task;
    ++ran;
    if (task >= 0) {
      const long coords[2] = {task / n_split, task % n_split};
      const long ev = coords[om.pick[0]];
      B[task] = part_val[task];
      notes[ev] += 1;
      counter[ev] -= 1;
      if (counter[ev] == 0 && !final_queued[ev]) {
        // in_map "i->i": final(i) waits on event i; find consumers of ev.
        const long ci = ev;  // consumer grid is [n_rows]; identity in_map picks coord 0
        final_queued[ci] = 1;
        ready.push_back(-(ci + 1));
      }
    } else {
      const long i = -task - 1;
      const long coords[1] = {i};
      const long ev = coords[im.pick[0]];
      if (counter[ev] != 0) ++early_count;
      double s = 0.0;
      for (int j = 0; j < n_split; ++j) s += B[i * n_split + j];
      C[i] = s;
    }
  }
  for (long i = 0; i < n_rows; ++i) notifies[i] = notes[i];
  *early = static_cast<int32_t>(early_count);
  return ran;
}

}  // extern "C"
