// fp64 oracle for the gated delta rule over packed variable-length batches.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
// this file: only tests/, the smoke check and the benchmark's CPU-baseline leg
// use it, to produce reference values. It shares no code with the CUDA library.
//
// What it computes (the plain definition, token by token, in fp64):
//   For each document i = [cu[i], cu[i+1]) and value head h (key head
//   hk = h / (Hv / Hk)), the state S in R^{Dk x Dv} starts at S_init(i, h) and,
//   for every token t,
//       a  = exp(g_t)                          decay gate alpha_t = e^{g_t}
//       S' = a * S                             decay first
//       p  = S'^T k_t                          value the decayed memory predicts for k_t
//       d  = beta_t * (v_t - p)                delta-rule correction
//       S  = S' + k_t d^T                      write it back along k_t
//       o_t = S^T q_t                          the query reads the updated state
//   which is S_t = e^{g_t} (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T.
//   final_state[i, h] = S after the last token of the document.
// Sources: "How to Speed Up GDN Kernels for Qwen Models", section "What GDN
// actually computes" (S in R^{d_k x d_v} per head, alpha_t = e^{g_t}, the
// erase-then-write factor (I - beta_t k_t k_t^T)); "Musings on long-context
// fine-tuning", section "Isolating the recurrent layers" (decay the memory, then
// correct its prediction for the current key; the query reads the updated
// matrix; the state restarts at each document given by cu_seqlens and a
// continuation may start from another document's final state through
// initial_state).
//
// Initial states (init_idx[i]): -1 = zero; 0 <= x < n_init = initial_state[x];
// n_init + j with j < i = the final state of document j of the same call.
//
// Backward: hand-written reverse mode of the recurrence above, token by token,
// with dL/dS at the end of each document seeded by dfinal_state (or zero) plus,
// for a document whose final state was forked, the d(initial state) of every
// document that started from it. Gradients that reach a shared initial state
// are summed over all documents that share it ("Musings on long-context
// fine-tuning", section "Backward through P"). dq and dk are summed over the
// value heads that share a key head.
//
// Parallelism: the columns of S evolve independently given (k, g, beta), so the
// work is split over (value head, block of Dv columns); documents run in order
// inside a task (forks point backwards), and in reverse order in the backward.
// Sums over columns (dq, dk, dbeta, dg) are kept per column block and reduced
// afterwards in a fixed order, so results do not depend on the thread count.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Shape {
  int32_t N;
  int64_t T;
  int32_t Hk, Hv, Dk, Dv;
  int32_t n_init;
};

int validate(const Shape& s, const int32_t* cu, const int32_t* init_idx) {
  if (s.N < 0 || s.T < 0 || s.Hk <= 0 || s.Hv <= 0 || s.Dk <= 0 || s.Dv <= 0 || s.n_init < 0) return -1;
  if (s.Hv % s.Hk != 0) return -1;
  if (cu[0] != 0 || (int64_t)cu[s.N] != s.T) return -1;
  for (int i = 0; i < s.N; ++i)
    if (cu[i + 1] < cu[i]) return -1;
  if (init_idx) {
    for (int i = 0; i < s.N; ++i) {
      int x = init_idx[i];
      if (x < -1) return -1;
      if (x >= s.n_init && x - s.n_init >= i) return -1;
    }
  }
  return 0;
}

template <class F>
void run_tasks(int n_tasks, int n_threads, F&& f) {
  if (n_threads < 1) n_threads = 1;
  n_threads = std::min(n_threads, n_tasks);
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (;;) {
      int t = next.fetch_add(1);
      if (t >= n_tasks) break;
      f(t);
    }
  };
  if (n_threads <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int i = 0; i < n_threads; ++i) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

// Column blocks: enough tasks to occupy the threads, at least 4 columns each.
int pick_col_blocks(const Shape& s, int n_threads) {
  int want = std::max(1, (n_threads + s.Hv - 1) / s.Hv);
  int maxb = std::max(1, s.Dv / 4);
  return std::min(want, maxb);
}

// One token of the forward recurrence on a column block of width w.
// S is Dk x w (row-major, row stride w). Writes p (the prediction) and d (delta).
inline void token_step(double* S, int Dk, int w, double a, double b, const double* kt, const double* vt,
                       double* p, double* d) {
  for (int r = 0; r < Dk; ++r)
    for (int c = 0; c < w; ++c) S[r * w + c] *= a;
  for (int c = 0; c < w; ++c) p[c] = 0.0;
  for (int r = 0; r < Dk; ++r) {
    double kr = kt[r];
    for (int c = 0; c < w; ++c) p[c] += S[r * w + c] * kr;
  }
  for (int c = 0; c < w; ++c) d[c] = b * (vt[c] - p[c]);
  for (int r = 0; r < Dk; ++r) {
    double kr = kt[r];
    for (int c = 0; c < w; ++c) S[r * w + c] += kr * d[c];
  }
}

struct Inputs {
  const double *q, *k, *v, *g, *beta;
  const int32_t *cu, *init_idx;
  const double* initial_state;
};

// Load the start state of document i for head h, columns [c0, c0 + w).
void load_init(const Shape& s, const Inputs& in, int i, int h, int c0, int w,
               const std::vector<std::vector<double>>& fin, double* S) {
  int x = in.init_idx ? in.init_idx[i] : -1;
  if (x < 0) {
    std::fill(S, S + (size_t)s.Dk * w, 0.0);
  } else if (x < s.n_init) {
    const double* src = in.initial_state + (((size_t)x * s.Hv + h) * s.Dk) * s.Dv;
    for (int r = 0; r < s.Dk; ++r)
      for (int c = 0; c < w; ++c) S[r * w + c] = src[(size_t)r * s.Dv + c0 + c];
  } else {
    const std::vector<double>& f = fin[x - s.n_init];
    std::copy(f.begin(), f.end(), S);
  }
}

}  // namespace

extern "C" {

int gdn_oracle_fwd(const double* q, const double* k, const double* v, const double* g, const double* beta,
                   const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t Hk, int32_t Hv, int32_t Dk,
                   int32_t Dv, const int32_t* init_idx, const double* initial_state, int32_t n_init,
                   double* out, double* final_state, int32_t n_threads) {
  Shape s{N, T, Hk, Hv, Dk, Dv, n_init};
  if (!cu_seqlens || validate(s, cu_seqlens, init_idx) != 0) return -1;
  if (n_init > 0 && !initial_state) return -1;
  Inputs in{q, k, v, g, beta, cu_seqlens, init_idx, initial_state};
  const int nb = pick_col_blocks(s, n_threads);
  const int G = Hv / Hk;
  run_tasks(Hv * nb, n_threads, [&](int task) {
    const int h = task / nb, blk = task % nb;
    const int c0 = (int)((int64_t)Dv * blk / nb), c1 = (int)((int64_t)Dv * (blk + 1) / nb), w = c1 - c0;
    const int hk = h / G;
    std::vector<std::vector<double>> fin(N);
    std::vector<double> S((size_t)Dk * w), p(w), d(w);
    for (int i = 0; i < N; ++i) {
      load_init(s, in, i, h, c0, w, fin, S.data());
      for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
        const double a = std::exp(g[t * Hv + h]);
        const double b = beta[t * Hv + h];
        const double* kt = k + ((size_t)t * Hk + hk) * Dk;
        const double* qt = q + ((size_t)t * Hk + hk) * Dk;
        const double* vt = v + ((size_t)t * Hv + h) * Dv + c0;
        token_step(S.data(), Dk, w, a, b, kt, vt, p.data(), d.data());
        double* ot = out + ((size_t)t * Hv + h) * Dv + c0;
        for (int c = 0; c < w; ++c) ot[c] = 0.0;
        for (int r = 0; r < Dk; ++r) {
          double qr = qt[r];
          for (int c = 0; c < w; ++c) ot[c] += S[(size_t)r * w + c] * qr;
        }
      }
      fin[i] = S;
      if (final_state) {
        double* dst = final_state + (((size_t)i * Hv + h) * Dk) * Dv;
        for (int r = 0; r < Dk; ++r)
          for (int c = 0; c < w; ++c) dst[(size_t)r * Dv + c0 + c] = S[(size_t)r * w + c];
      }
    }
  });
  return 0;
}

// Backward. dout [T,Hv,Dv]; dfinal [N,Hv,Dk,Dv] or null. Outputs (all overwritten):
// dq, dk [T,Hk,Dk]; dv [T,Hv,Dv]; dg, dbeta [T,Hv]; dinit [n_init,Hv,Dk,Dv] (if n_init > 0).
int gdn_oracle_bwd(const double* q, const double* k, const double* v, const double* g, const double* beta,
                   const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t Hk, int32_t Hv, int32_t Dk,
                   int32_t Dv, const int32_t* init_idx, const double* initial_state, int32_t n_init,
                   const double* dout, const double* dfinal, double* dq, double* dk, double* dv, double* dg,
                   double* dbeta, double* dinit, int32_t n_threads) {
  Shape s{N, T, Hk, Hv, Dk, Dv, n_init};
  if (!cu_seqlens || validate(s, cu_seqlens, init_idx) != 0) return -1;
  if (n_init > 0 && (!initial_state || !dinit)) return -1;
  Inputs in{q, k, v, g, beta, cu_seqlens, init_idx, initial_state};
  const int nb = pick_col_blocks(s, n_threads);
  const int G = Hv / Hk;
  // Per column block partial sums: dq/dk per value head [nb][T][Hv][Dk], dbeta/dg [nb][T][Hv].
  std::vector<double> pq((size_t)nb * T * Hv * Dk, 0.0), pk((size_t)nb * T * Hv * Dk, 0.0);
  std::vector<double> pb((size_t)nb * T * Hv, 0.0), pg((size_t)nb * T * Hv, 0.0);
  if (n_init > 0) std::fill(dinit, dinit + (size_t)n_init * Hv * Dk * Dv, 0.0);
  constexpr int CK = 64;  // checkpoint interval (tokens)

  run_tasks(Hv * nb, n_threads, [&](int task) {
    const int h = task / nb, blk = task % nb;
    const int c0 = (int)((int64_t)Dv * blk / nb), c1 = (int)((int64_t)Dv * (blk + 1) / nb), w = c1 - c0;
    const int hk = h / G;
    const size_t SZ = (size_t)Dk * w;
    // Forward sweep: start state of every document and final states (for forks).
    std::vector<std::vector<double>> fin(N), start(N);
    std::vector<double> S(SZ), p(w), d(w);
    for (int i = 0; i < N; ++i) {
      load_init(s, in, i, h, c0, w, fin, S.data());
      start[i] = S;
      for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
        const double* kt = k + ((size_t)t * Hk + hk) * Dk;
        const double* vt = v + ((size_t)t * Hv + h) * Dv + c0;
        token_step(S.data(), Dk, w, std::exp(g[t * Hv + h]), beta[t * Hv + h], kt, vt, p.data(), d.data());
      }
      fin[i] = S;
    }
    // dL/dS at each document end: dfinal plus what forked documents send back.
    std::vector<std::vector<double>> dfin(N, std::vector<double>(SZ, 0.0));
    if (dfinal)
      for (int i = 0; i < N; ++i) {
        const double* src = dfinal + (((size_t)i * Hv + h) * Dk) * Dv;
        for (int r = 0; r < Dk; ++r)
          for (int c = 0; c < w; ++c) dfin[i][(size_t)r * w + c] = src[(size_t)r * Dv + c0 + c];
      }
    double* pqb = pq.data() + (size_t)blk * T * Hv * Dk;
    double* pkb = pk.data() + (size_t)blk * T * Hv * Dk;
    double* pbb = pb.data() + (size_t)blk * T * Hv;
    double* pgb = pg.data() + (size_t)blk * T * Hv;
    std::vector<double> dS(SZ), Sp(SZ), states((size_t)(CK + 1) * SZ), ddel(w), dp(w), vp(w);
    for (int i = N - 1; i >= 0; --i) {
      const int64_t t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
      dS = dfin[i];
      // Checkpoints: state before each block of CK tokens.
      const int64_t nblk = (t1 - t0 + CK - 1) / CK;
      std::vector<std::vector<double>> ckpt(nblk);
      S = start[i];
      for (int64_t bi = 0; bi < nblk; ++bi) {
        ckpt[bi] = S;
        for (int64_t t = t0 + bi * CK; t < std::min(t1, t0 + (bi + 1) * CK); ++t) {
          const double* kt = k + ((size_t)t * Hk + hk) * Dk;
          const double* vt = v + ((size_t)t * Hv + h) * Dv + c0;
          token_step(S.data(), Dk, w, std::exp(g[t * Hv + h]), beta[t * Hv + h], kt, vt, p.data(), d.data());
        }
      }
      for (int64_t bi = nblk - 1; bi >= 0; --bi) {
        const int64_t tb = t0 + bi * CK, te = std::min(t1, tb + CK);
        // states[j] = state before token tb + j; states[te - tb] = after the block.
        std::copy(ckpt[bi].begin(), ckpt[bi].end(), states.begin());
        for (int64_t t = tb; t < te; ++t) {
          double* cur = states.data() + (size_t)(t - tb + 1) * SZ;
          std::copy(states.begin() + (size_t)(t - tb) * SZ, states.begin() + (size_t)(t - tb + 1) * SZ, cur);
          const double* kt = k + ((size_t)t * Hk + hk) * Dk;
          const double* vt = v + ((size_t)t * Hv + h) * Dv + c0;
          token_step(cur, Dk, w, std::exp(g[t * Hv + h]), beta[t * Hv + h], kt, vt, p.data(), d.data());
        }
        for (int64_t t = te - 1; t >= tb; --t) {
          const double* Sprev = states.data() + (size_t)(t - tb) * SZ;
          const double* St = states.data() + (size_t)(t - tb + 1) * SZ;
          const double a = std::exp(g[t * Hv + h]);
          const double b = beta[t * Hv + h];
          const double* kt = k + ((size_t)t * Hk + hk) * Dk;
          const double* qt = q + ((size_t)t * Hk + hk) * Dk;
          const double* vt = v + ((size_t)t * Hv + h) * Dv + c0;
          const double* dot = dout + ((size_t)t * Hv + h) * Dv + c0;
          // Recompute S' = a S_{t-1}, p = S'^T k, delta = b (v - p).
          for (size_t e = 0; e < SZ; ++e) Sp[e] = a * Sprev[e];
          for (int c = 0; c < w; ++c) p[c] = 0.0;
          for (int r = 0; r < Dk; ++r)
            for (int c = 0; c < w; ++c) p[c] += Sp[(size_t)r * w + c] * kt[r];
          for (int c = 0; c < w; ++c) {
            vp[c] = vt[c] - p[c];
            d[c] = b * vp[c];
          }
          double* dqt = pqb + ((size_t)t * Hv + h) * Dk;
          double* dkt = pkb + ((size_t)t * Hv + h) * Dk;
          // o_t = S_t^T q_t
          for (int r = 0; r < Dk; ++r) {
            double acc = 0.0;
            for (int c = 0; c < w; ++c) {
              dS[(size_t)r * w + c] += qt[r] * dot[c];
              acc += St[(size_t)r * w + c] * dot[c];
            }
            dqt[r] += acc;
          }
          // S_t = S' + k d^T
          for (int c = 0; c < w; ++c) ddel[c] = 0.0;
          for (int r = 0; r < Dk; ++r) {
            double acc = 0.0;
            for (int c = 0; c < w; ++c) {
              ddel[c] += dS[(size_t)r * w + c] * kt[r];
              acc += dS[(size_t)r * w + c] * d[c];
            }
            dkt[r] += acc;
          }
          // d = b (v - p)
          double dbt = 0.0;
          double* dvt = dv + ((size_t)t * Hv + h) * Dv + c0;
          for (int c = 0; c < w; ++c) {
            dvt[c] = b * ddel[c];
            dbt += ddel[c] * vp[c];
            dp[c] = -b * ddel[c];
          }
          pbb[t * Hv + h] += dbt;
          // p = S'^T k: dS' = dS + k dp^T, dk += S' dp
          for (int r = 0; r < Dk; ++r) {
            double acc = 0.0;
            for (int c = 0; c < w; ++c) {
              dS[(size_t)r * w + c] += kt[r] * dp[c];
              acc += Sp[(size_t)r * w + c] * dp[c];
            }
            dkt[r] += acc;
          }
          // S' = a S_{t-1}: dg_t = <dS', S'>, dS_{t-1} = a dS'
          double dgt = 0.0;
          for (size_t e = 0; e < SZ; ++e) dgt += dS[e] * Sp[e];
          pgb[t * Hv + h] += dgt;
          for (size_t e = 0; e < SZ; ++e) dS[e] *= a;
        }
      }
      // Send dL/dS_init to wherever the start state came from.
      int x = init_idx ? init_idx[i] : -1;
      if (x >= 0 && x < n_init) {
        double* dst = dinit + (((size_t)x * Hv + h) * Dk) * Dv;
        for (int r = 0; r < Dk; ++r)
          for (int c = 0; c < w; ++c) dst[(size_t)r * Dv + c0 + c] += dS[(size_t)r * w + c];
      } else if (x >= n_init) {
        std::vector<double>& tgt = dfin[x - n_init];
        for (size_t e = 0; e < SZ; ++e) tgt[e] += dS[e];
      }
    }
  });

  // Fixed-order reductions: over column blocks, then over the value heads of each key head.
  for (int64_t t = 0; t < T; ++t) {
    for (int hk = 0; hk < Hk; ++hk) {
      double* oq = dq + ((size_t)t * Hk + hk) * Dk;
      double* ok = dk + ((size_t)t * Hk + hk) * Dk;
      for (int r = 0; r < Dk; ++r) oq[r] = ok[r] = 0.0;
      for (int hh = hk * G; hh < (hk + 1) * G; ++hh)
        for (int b = 0; b < nb; ++b) {
          const double* sq = pq.data() + (((size_t)b * T + t) * Hv + hh) * Dk;
          const double* sk = pk.data() + (((size_t)b * T + t) * Hv + hh) * Dk;
          for (int r = 0; r < Dk; ++r) {
            oq[r] += sq[r];
            ok[r] += sk[r];
          }
        }
    }
    for (int h = 0; h < Hv; ++h) {
      double sb = 0.0, sg = 0.0;
      for (int b = 0; b < nb; ++b) {
        sb += pb[((size_t)b * T + t) * Hv + h];
        sg += pg[((size_t)b * T + t) * Hv + h];
      }
      dbeta[t * Hv + h] = sb;
      dg[t * Hv + h] = sg;
    }
  }
  return 0;
}

int gdn_oracle_hw_threads(void) { return (int)std::thread::hardware_concurrency(); }

}  // extern "C"
