// Plain fp64 CPU oracle for the chunk-level gated delta rule.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or
// call this file: only the test suite, the smoke check and the benchmark's
// CPU-baseline leg use it. It shares no code, header or constant with the
// CUDA library.
//
// What it computes (token by token, no blocking, no reordering):
//
//   Gated delta rule, Eq. (1) named in the StateFlow review (referee report,
//   major comment 1), written out as in Gated Delta Networks (reference [32]
//   of that review). With the state held as M = S^T (d_k x d_v):
//
//     alpha_t = exp(g_t)
//     e_t     = v_t - alpha_t * M_{t-1}^T k_t            (the "new value")
//     M_t     = alpha_t * M_{t-1} + beta_t * k_t e_t^T
//     o_t     = M_t^T q_t
//
//   which is S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//   o_t = S_t q_t, with S = M^T.
//
//   A call processes one chunk C_i of each sequence: M_0 = S_in, and the final
//   state is S_out, so the forward chain S_{i+1}^in = S_i^out (Eq. 5 in
//   "What carries the argument") is a plain hand-over of the state.
//
//   Backward: reverse-mode differentiation of the same loop (back-propagation
//   through time) for the loss <do, o> + <dS_out, S_out>. It returns dq, dk,
//   dv, dg, dbeta and dS_in; the backward chain (Eq. 7) hands dS_in of chunk
//   i+1 to chunk i as its dS_out. States are re-created from checkpoints
//   taken every L tokens (two-level checkpointing, memory O(sqrt(T))).
//
// Layouts (all contiguous, row-major):
//   q, k   : [ntok, H, dk]        v, o, do : [ntok, H, dv]
//   g, beta: [ntok, H]            states   : [nstate, H, dk, dv]
// For the fixed-length entry points ntok = B*T and sequence b occupies tokens
// [b*T, (b+1)*T); for the varlen entry points sequence s occupies
// [cu[s], cu[s+1]) and its state slot is s.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Problem {
  int H, dk, dv;
  const double *q, *k, *v, *g, *beta;
  const double* S_in;   // nullable: zero initial state
  double* o;            // fwd output (nullable in bwd)
  double* S_out;        // nullable
  // backward
  const double* dout;
  const double* dS_out;  // nullable: zero
  double *dq, *dk_, *dv_, *dg, *dbeta;
  double* dS_in;  // nullable
};

struct Item {
  long start;  // first token (flattened index)
  long len;
  int slot;    // state slot (batch index or sequence index)
  int h;
};

inline const double* tok(const double* base, long n, int H, int h, int d) {
  return base + ((size_t)n * H + h) * d;
}
inline double* tok(double* base, long n, int H, int h, int d) {
  return base + ((size_t)n * H + h) * d;
}

// One token of the recurrence: M <- alpha M + beta k e^T, e = v - alpha M^T k.
void step(const Problem& P, long n, int h, double* M, double* e /*dv scratch*/) {
  const int dk = P.dk, dv = P.dv, H = P.H;
  const double* kk = tok(P.k, n, H, h, dk);
  const double* vv = tok(P.v, n, H, h, dv);
  const double a = std::exp(P.g[(size_t)n * H + h]);
  const double b = P.beta[(size_t)n * H + h];
  for (int j = 0; j < dv; ++j) e[j] = 0.0;
  for (int i = 0; i < dk; ++i) {
    const double ki = kk[i];
    const double* row = M + (size_t)i * dv;
    for (int j = 0; j < dv; ++j) e[j] += ki * row[j];
  }
  for (int j = 0; j < dv; ++j) e[j] = vv[j] - a * e[j];
  for (int i = 0; i < dk; ++i) {
    const double bki = b * kk[i];
    double* row = M + (size_t)i * dv;
    for (int j = 0; j < dv; ++j) row[j] = a * row[j] + bki * e[j];
  }
}

void load_state(const double* S, const Item& it, int H, int dk, int dv, double* M) {
  const size_t sz = (size_t)dk * dv;
  if (S)
    std::memcpy(M, S + ((size_t)it.slot * H + it.h) * sz, sz * sizeof(double));
  else
    std::fill(M, M + sz, 0.0);
}

void fwd_item(const Problem& P, const Item& it) {
  const int dk = P.dk, dv = P.dv, H = P.H;
  const size_t sz = (size_t)dk * dv;
  std::vector<double> M(sz), e(dv);
  load_state(P.S_in, it, H, dk, dv, M.data());
  for (long t = 0; t < it.len; ++t) {
    const long n = it.start + t;
    step(P, n, it.h, M.data(), e.data());
    const double* qq = tok(P.q, n, H, it.h, dk);
    double* oo = tok(P.o, n, H, it.h, dv);
    for (int j = 0; j < dv; ++j) oo[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
      const double qi = qq[i];
      const double* row = M.data() + (size_t)i * dv;
      for (int j = 0; j < dv; ++j) oo[j] += qi * row[j];
    }
  }
  if (P.S_out) std::memcpy(P.S_out + ((size_t)it.slot * H + it.h) * sz, M.data(), sz * sizeof(double));
}

long checkpoint_interval(long len) {
  long L = 64;
  while (L * L < len) L *= 2;
  return L;
}

void bwd_item(const Problem& P, const Item& it) {
  const int dk = P.dk, dv = P.dv, H = P.H, h = it.h;
  const size_t sz = (size_t)dk * dv;
  const long L = checkpoint_interval(it.len);
  const long nseg = (it.len + L - 1) / L;
  std::vector<double> ck((size_t)std::max<long>(nseg, 1) * sz);
  std::vector<double> e(dv), de(dv), dqv(dk), dkv(dk);
  // forward sweep: keep the state at the start of every segment
  {
    std::vector<double> M(sz);
    load_state(P.S_in, it, H, dk, dv, M.data());
    for (long c = 0; c < nseg; ++c) {
      std::memcpy(ck.data() + (size_t)c * sz, M.data(), sz * sizeof(double));
      const long t1 = std::min(it.len, (c + 1) * L);
      for (long t = c * L; t < t1; ++t) step(P, it.start + t, h, M.data(), e.data());
    }
  }
  std::vector<double> D(sz);
  if (P.dS_out)
    std::memcpy(D.data(), P.dS_out + ((size_t)it.slot * H + h) * sz, sz * sizeof(double));
  else
    std::fill(D.begin(), D.end(), 0.0);
  std::vector<double> seg((size_t)(L + 1) * sz);
  for (long c = nseg - 1; c >= 0; --c) {
    const long t0 = c * L, t1 = std::min(it.len, (c + 1) * L);
    std::memcpy(seg.data(), ck.data() + (size_t)c * sz, sz * sizeof(double));
    for (long t = t0; t < t1; ++t) {
      double* nxt = seg.data() + (size_t)(t - t0 + 1) * sz;
      std::memcpy(nxt, nxt - sz, sz * sizeof(double));
      step(P, it.start + t, h, nxt, e.data());
    }
    for (long t = t1 - 1; t >= t0; --t) {
      const long n = it.start + t;
      const double* Mprev = seg.data() + (size_t)(t - t0) * sz;
      const double* Mcur = Mprev + sz;
      const double* qq = tok(P.q, n, H, h, dk);
      const double* kk = tok(P.k, n, H, h, dk);
      const double* vv = tok(P.v, n, H, h, dv);
      const double* dd = tok(P.dout, n, H, h, dv);
      const double a = std::exp(P.g[(size_t)n * H + h]);
      const double b = P.beta[(size_t)n * H + h];
      // o_t = M_t^T q_t
      for (int i = 0; i < dk; ++i) {
        double* Drow = D.data() + (size_t)i * dv;
        const double* Mrow = Mcur + (size_t)i * dv;
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) {
          Drow[j] += qq[i] * dd[j];
          acc += Mrow[j] * dd[j];
        }
        dqv[i] = acc;
      }
      // e = v - a Mprev^T k
      for (int j = 0; j < dv; ++j) e[j] = 0.0;
      for (int i = 0; i < dk; ++i) {
        const double* Mrow = Mprev + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) e[j] += kk[i] * Mrow[j];
      }
      for (int j = 0; j < dv; ++j) e[j] = vv[j] - a * e[j];
      // M_t = a Mprev + b k e^T
      for (int j = 0; j < dv; ++j) de[j] = 0.0;
      double dbeta = 0.0, dalpha = 0.0;
      for (int i = 0; i < dk; ++i) {
        const double* Drow = D.data() + (size_t)i * dv;
        const double* Mrow = Mprev + (size_t)i * dv;
        double De = 0.0;
        for (int j = 0; j < dv; ++j) {
          de[j] += Drow[j] * kk[i];
          De += Drow[j] * e[j];
          dalpha += Drow[j] * Mrow[j];
        }
        dkv[i] = b * De;
        dbeta += kk[i] * De;
      }
      for (int j = 0; j < dv; ++j) de[j] *= b;
      // through e: dv = de, dk -= a Mprev de, dalpha -= k^T Mprev de
      for (int i = 0; i < dk; ++i) {
        const double* Mrow = Mprev + (size_t)i * dv;
        double Mde = 0.0;
        for (int j = 0; j < dv; ++j) Mde += Mrow[j] * de[j];
        dkv[i] -= a * Mde;
        dalpha -= kk[i] * Mde;
      }
      // D <- a (D - k de^T)
      for (int i = 0; i < dk; ++i) {
        double* Drow = D.data() + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Drow[j] = a * (Drow[j] - kk[i] * de[j]);
      }
      std::memcpy(tok(P.dq, n, H, h, dk), dqv.data(), dk * sizeof(double));
      std::memcpy(tok(P.dk_, n, H, h, dk), dkv.data(), dk * sizeof(double));
      std::memcpy(tok(P.dv_, n, H, h, dv), de.data(), dv * sizeof(double));
      P.dg[(size_t)n * H + h] = a * dalpha;
      P.dbeta[(size_t)n * H + h] = dbeta;
    }
  }
  if (P.dS_in) std::memcpy(P.dS_in + ((size_t)it.slot * H + h) * sz, D.data(), sz * sizeof(double));
}

template <class F>
void run_items(const std::vector<Item>& items, int nthreads, F f) {
  if (nthreads < 1) nthreads = 1;
  nthreads = std::min<int>(nthreads, (int)items.size());
  if (nthreads <= 1) {
    for (const Item& it : items) f(it);
    return;
  }
  std::atomic<size_t> next{0};
  std::vector<std::thread> pool;
  for (int w = 0; w < nthreads; ++w)
    pool.emplace_back([&] {
      for (size_t i = next++; i < items.size(); i = next++) f(items[i]);
    });
  for (auto& th : pool) th.join();
}

std::vector<Item> fixed_items(int B, int T, int H) {
  std::vector<Item> items;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) items.push_back({(long)b * T, (long)T, b, h});
  return items;
}

int varlen_items(const int* cu, int nseq, int H, std::vector<Item>* items) {
  if (!cu || nseq < 1 || cu[0] != 0) return 1;
  for (int s = 0; s < nseq; ++s)
    if (cu[s + 1] < cu[s]) return 1;
  for (int s = 0; s < nseq; ++s)
    for (int h = 0; h < H; ++h) items->push_back({(long)cu[s], (long)(cu[s + 1] - cu[s]), s, h});
  return 0;
}

bool bad_dims(int H, int dk, int dv) { return H < 1 || dk < 1 || dv < 1; }

}  // namespace

extern "C" {

// Returns 0 on success, 1 on invalid arguments.
int gdn_oracle_fwd(int B, int T, int H, int dk, int dv, const double* q, const double* k,
                   const double* v, const double* g, const double* beta, const double* S_in,
                   double* o, double* S_out, int nthreads) {
  if (B < 1 || T < 0 || bad_dims(H, dk, dv)) return 1;
  Problem P{};
  P.H = H; P.dk = dk; P.dv = dv;
  P.q = q; P.k = k; P.v = v; P.g = g; P.beta = beta; P.S_in = S_in; P.o = o; P.S_out = S_out;
  run_items(fixed_items(B, T, H), nthreads, [&](const Item& it) { fwd_item(P, it); });
  return 0;
}

int gdn_oracle_bwd(int B, int T, int H, int dk, int dv, const double* q, const double* k,
                   const double* v, const double* g, const double* beta, const double* S_in,
                   const double* dout, const double* dS_out, double* dq, double* dk_,
                   double* dv_, double* dg, double* dbeta, double* dS_in, int nthreads) {
  if (B < 1 || T < 0 || bad_dims(H, dk, dv)) return 1;
  Problem P{};
  P.H = H; P.dk = dk; P.dv = dv;
  P.q = q; P.k = k; P.v = v; P.g = g; P.beta = beta; P.S_in = S_in;
  P.dout = dout; P.dS_out = dS_out;
  P.dq = dq; P.dk_ = dk_; P.dv_ = dv_; P.dg = dg; P.dbeta = dbeta; P.dS_in = dS_in;
  run_items(fixed_items(B, T, H), nthreads, [&](const Item& it) { bwd_item(P, it); });
  return 0;
}

int gdn_oracle_varlen_fwd(int H, int dk, int dv, const int* cu, int nseq, const double* q,
                          const double* k, const double* v, const double* g, const double* beta,
                          const double* S0, double* o, double* S_final, int nthreads) {
  std::vector<Item> items;
  if (bad_dims(H, dk, dv) || varlen_items(cu, nseq, H, &items)) return 1;
  Problem P{};
  P.H = H; P.dk = dk; P.dv = dv;
  P.q = q; P.k = k; P.v = v; P.g = g; P.beta = beta; P.S_in = S0; P.o = o; P.S_out = S_final;
  run_items(items, nthreads, [&](const Item& it) { fwd_item(P, it); });
  return 0;
}

int gdn_oracle_varlen_bwd(int H, int dk, int dv, const int* cu, int nseq, const double* q,
                          const double* k, const double* v, const double* g, const double* beta,
                          const double* S0, const double* dout, const double* dS_final,
                          double* dq, double* dk_, double* dv_, double* dg, double* dbeta,
                          double* dS0, int nthreads) {
  std::vector<Item> items;
  if (bad_dims(H, dk, dv) || varlen_items(cu, nseq, H, &items)) return 1;
  Problem P{};
  P.H = H; P.dk = dk; P.dv = dv;
  P.q = q; P.k = k; P.v = v; P.g = g; P.beta = beta; P.S_in = S0;
  P.dout = dout; P.dS_out = dS_final;
  P.dq = dq; P.dk_ = dk_; P.dv_ = dv_; P.dg = dg; P.dbeta = dbeta; P.dS_in = dS0;
  run_items(items, nthreads, [&](const Item& it) { bwd_item(P, it); });
  return 0;
}

}  // extern "C"
