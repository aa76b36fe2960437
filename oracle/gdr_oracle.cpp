// gdr_oracle.cpp -- FP64 CPU oracle for the gated delta rule over packed
// variable-length documents (KDA and GDN).
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the benchmark's
// CPU-baseline leg load this library.  It shares no code, header, table or
// helper with the CUDA library; it is a plain token-by-token recurrence
// written for readability, not speed.
//
// What it computes (the method both pages train):
//   "feat(cake_kda): ... Cake KDA context-parallel (KCP) autograd backend"
//   (flashinfer PR #8218), opening description and "Workload" paragraph:
//   Kimi Delta Attention over packed documents at head dim 128, q and k
//   L2-normalized, a pre-activated FP32 log-decay gate g per (token, head,
//   channel), beta per (token, head).
//   "perf(cake_gdn): prefetch offset adjoint walk, default LPT segment plan"
//   (flashinfer PR #7723), opening description: Gated DeltaNet with a scalar
//   FP32 log-decay per (token, value head), grouped Q/K heads (H_qk, HV), and
//   dq/dk summed over the value heads that share a Q/K head.
// The pages name the method but never print its recurrence; the plain
// definition of the gated delta rule is used, per (document, value head),
// with the state reset to h0[doc] (or zero) at every document start:
//   a_t = exp(g_t)                      (a K-vector for KDA, a scalar for GDN)
//   P_t = diag(a_t) S_{t-1}             (S is K x V, S[k][v])
//   r_t = v_t - P_t^T k_t
//   S_t = P_t + beta_t k_t r_t^T        (= (I - beta k k^T) diag(a) S + beta k v^T)
//   o_t = scale * S_t^T q_t
//   ht[doc] = S after the document's last token.
// The reverse pass is the hand-derived adjoint of those five lines, run
// backwards over the tokens of each document (see oracle_chain_bwd).
//
// Everything is double precision.  Inputs arrive as doubles (the caller
// widens BF16/FP32 values exactly).  D is a parameter (the method uses 128;
// tests use 4 or 8 for finite differences).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

extern "C" {

// One problem: a packed batch of N documents, T tokens in total.
// Layouts (row-major, contiguous):
//   q, k, dq, dk : [T][Hqk][D]
//   v, out, dout, dv : [T][HV][D]
//   g, dg : [T][HV][D] when gate_per_channel (KDA) else [T][HV] (GDN)
//   beta, dbeta : [T][HV]
//   h0, ht, dht, dh0 : [N][HV][D][D], S[k][v]
// Value head j reads Q/K head j / (HV / Hqk) (contiguous groups).
struct gdr_oracle_problem {
  int64_t T;
  int32_t N;
  const int32_t* cu_seqlens;  // [N+1], 0 = cu[0] <= cu[1] <= ... <= cu[N] = T
  int32_t Hqk, HV, D;
  int32_t gate_per_channel;   // 1: KDA gate [T][HV][D]; 0: GDN gate [T][HV]
  double scale;
  const double *q, *k, *v, *g, *beta;
  const double* h0;           // nullable: zero initial state
  const double* dout;         // nullable: forward only
  const double* dht;          // nullable: zero adjoint of the final state
  double *out, *ht;           // ht nullable
  double *dq, *dk, *dv, *dg, *dbeta, *dh0;  // used when dout != null; dh0 nullable
  int32_t threads;            // 0: one per hardware thread
};

int gdr_oracle_hardware_threads(void) {
  unsigned n = std::thread::hardware_concurrency();
  return n == 0 ? 1 : (int)n;
}

}  // extern "C"

namespace {

struct Chain {
  const gdr_oracle_problem* p;
  int32_t doc;
  int32_t hv;       // value head
  int32_t hq;       // its Q/K head
  int64_t t0, len;  // token range of the document
};

inline const double* row_qk(const double* base, const gdr_oracle_problem* p, int64_t t, int32_t hq) {
  return base + ((size_t)t * p->Hqk + hq) * p->D;
}
inline const double* row_v(const double* base, const gdr_oracle_problem* p, int64_t t, int32_t hv) {
  return base + ((size_t)t * p->HV + hv) * p->D;
}
inline double* row_v_mut(double* base, const gdr_oracle_problem* p, int64_t t, int32_t hv) {
  return base + ((size_t)t * p->HV + hv) * p->D;
}

// Decay of token t for channel c.
inline double gate_at(const gdr_oracle_problem* p, int64_t t, int32_t hv, int c) {
  if (p->gate_per_channel) return p->g[((size_t)t * p->HV + hv) * p->D + c];
  return p->g[(size_t)t * p->HV + hv];
}

// One forward token step on state S (D x D, S[k][v]); writes r (D) when given.
// Returns nothing; S becomes S_t.
void token_step(const gdr_oracle_problem* p, const Chain& ch, int64_t t, std::vector<double>& S,
                std::vector<double>& r) {
  const int D = p->D;
  const double* kt = row_qk(p->k, p, t, ch.hq);
  const double* vt = row_v(p->v, p, t, ch.hv);
  const double bt = p->beta[(size_t)t * p->HV + ch.hv];
  // P = diag(exp(g)) S
  for (int c = 0; c < D; ++c) {
    const double a = std::exp(gate_at(p, t, ch.hv, c));
    double* Sc = &S[(size_t)c * D];
    for (int j = 0; j < D; ++j) Sc[j] *= a;
  }
  // r = v - P^T k
  for (int j = 0; j < D; ++j) r[j] = vt[j];
  for (int c = 0; c < D; ++c) {
    const double kc = kt[c];
    const double* Sc = &S[(size_t)c * D];
    for (int j = 0; j < D; ++j) r[j] -= Sc[j] * kc;
  }
  // S = P + beta k r^T
  for (int c = 0; c < D; ++c) {
    const double f = bt * kt[c];
    double* Sc = &S[(size_t)c * D];
    for (int j = 0; j < D; ++j) Sc[j] += f * r[j];
  }
}

// o = scale * S^T q
void token_out(const gdr_oracle_problem* p, const Chain& ch, int64_t t, const std::vector<double>& S,
               double* o) {
  const int D = p->D;
  const double* qt = row_qk(p->q, p, t, ch.hq);
  for (int j = 0; j < D; ++j) o[j] = 0.0;
  for (int c = 0; c < D; ++c) {
    const double qc = qt[c];
    const double* Sc = &S[(size_t)c * D];
    for (int j = 0; j < D; ++j) o[j] += Sc[j] * qc;
  }
  for (int j = 0; j < D; ++j) o[j] *= p->scale;
}

void load_h0(const gdr_oracle_problem* p, const Chain& ch, std::vector<double>& S) {
  const size_t DD = (size_t)p->D * p->D;
  if (p->h0) {
    const double* src = p->h0 + ((size_t)ch.doc * p->HV + ch.hv) * DD;
    std::copy(src, src + DD, S.begin());
  } else {
    std::fill(S.begin(), S.end(), 0.0);
  }
}

// Forward over one chain.  When `ckpt` is non-null, stores S_{t-1} (the
// state before token t0 + s*every) for every segment s.
void chain_fwd(const gdr_oracle_problem* p, const Chain& ch, int64_t every,
               std::vector<std::vector<double>>* ckpt) {
  const int D = p->D;
  const size_t DD = (size_t)D * D;
  std::vector<double> S(DD), r(D);
  load_h0(p, ch, S);
  for (int64_t i = 0; i < ch.len; ++i) {
    const int64_t t = ch.t0 + i;
    if (ckpt && i % every == 0) ckpt->push_back(S);
    token_step(p, ch, t, S, r);
    token_out(p, ch, t, S, row_v_mut(p->out, p, t, ch.hv));
  }
  if (p->ht) {
    double* dst = p->ht + ((size_t)ch.doc * p->HV + ch.hv) * DD;
    std::copy(S.begin(), S.end(), dst);
  }
}

// Reverse pass over one chain: the adjoint of token_step / token_out, with
// dS the adjoint of S_t on entry to token t's step (iterating t downwards):
//   dS   += scale * q_t do_t^T          (from o_t = scale S_t^T q_t)
//   dq_t  = scale * S_t do_t
//   dbeta = k_t^T dS r_t
//   dr    = beta dS^T k_t   (= dv_t)
//   dk_t  = beta dS r_t - P_t dr
//   dP    = dS - k_t dr^T
//   dg_t  = rowsum(dP * P_t)   (KDA per channel; GDN summed over channels)
//   dS   <- diag(a_t) dP        (adjoint of S_{t-1})
// dq/dk of the chain's Q/K head are accumulated (+=) into the outputs.
void chain_bwd(const gdr_oracle_problem* p, const Chain& ch) {
  const int D = p->D;
  const size_t DD = (size_t)D * D;
  if (ch.len == 0) {
    // Empty document: ht = h0, so dh0 = dht.
    if (p->dh0) {
      double* dst = p->dh0 + ((size_t)ch.doc * p->HV + ch.hv) * DD;
      if (p->dht) {
        const double* src = p->dht + ((size_t)ch.doc * p->HV + ch.hv) * DD;
        std::copy(src, src + DD, dst);
      } else {
        std::fill(dst, dst + DD, 0.0);
      }
    }
    if (p->ht) chain_fwd(p, ch, 1, nullptr);
    return;
  }
  // Square-root checkpointing keeps memory at O(sqrt(L) * D^2).
  int64_t every = (int64_t)std::ceil(std::sqrt((double)ch.len));
  if (every < 16) every = 16;
  std::vector<std::vector<double>> ckpt;
  chain_fwd(p, ch, every, &ckpt);

  std::vector<double> dS(DD, 0.0);
  if (p->dht) {
    const double* src = p->dht + ((size_t)ch.doc * p->HV + ch.hv) * DD;
    std::copy(src, src + DD, dS.begin());
  }
  std::vector<double> S(DD), P(DD), St(DD), r(D), u(D), dr(D), a(D);
  std::vector<std::vector<double>> seg;  // S_{t-1} for each t of the segment
  const int64_t nseg = (int64_t)ckpt.size();
  for (int64_t s = nseg - 1; s >= 0; --s) {
    const int64_t i0 = s * every;
    const int64_t i1 = std::min<int64_t>(ch.len, i0 + every);
    seg.clear();
    S = ckpt[(size_t)s];
    for (int64_t i = i0; i < i1; ++i) {
      seg.push_back(S);
      token_step(p, ch, ch.t0 + i, S, r);
    }
    for (int64_t i = i1 - 1; i >= i0; --i) {
      const int64_t t = ch.t0 + i;
      const double* qt = row_qk(p->q, p, t, ch.hq);
      const double* kt = row_qk(p->k, p, t, ch.hq);
      const double* vt = row_v(p->v, p, t, ch.hv);
      const double* dot = row_v(p->dout, p, t, ch.hv);
      const double bt = p->beta[(size_t)t * p->HV + ch.hv];
      const std::vector<double>& Sprev = seg[(size_t)(i - i0)];
      // Recompute P_t, r_t, S_t.
      for (int c = 0; c < D; ++c) a[c] = std::exp(gate_at(p, t, ch.hv, c));
      for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j) P[(size_t)c * D + j] = a[c] * Sprev[(size_t)c * D + j];
      for (int j = 0; j < D; ++j) {
        double acc = vt[j];
        for (int c = 0; c < D; ++c) acc -= P[(size_t)c * D + j] * kt[c];
        r[j] = acc;
      }
      for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j) St[(size_t)c * D + j] = P[(size_t)c * D + j] + bt * kt[c] * r[j];
      // dS += scale q do^T
      for (int c = 0; c < D; ++c)
        for (int j = 0; j < D; ++j) dS[(size_t)c * D + j] += p->scale * qt[c] * dot[j];
      // dq_t = scale S_t do_t
      double* dqt = p->dq + ((size_t)t * p->Hqk + ch.hq) * D;
      for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j) acc += St[(size_t)c * D + j] * dot[j];
        dqt[c] += p->scale * acc;
      }
      // u = dS r ; dbeta = k^T u ; dr = beta dS^T k
      double dbeta = 0.0;
      for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j) acc += dS[(size_t)c * D + j] * r[j];
        u[c] = acc;
        dbeta += kt[c] * acc;
      }
      p->dbeta[(size_t)t * p->HV + ch.hv] = dbeta;
      for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int c = 0; c < D; ++c) acc += dS[(size_t)c * D + j] * kt[c];
        dr[j] = bt * acc;
      }
      double* dvt = row_v_mut(p->dv, p, t, ch.hv);
      for (int j = 0; j < D; ++j) dvt[j] = dr[j];
      // dk_t = beta u - P dr
      double* dkt = p->dk + ((size_t)t * p->Hqk + ch.hq) * D;
      for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j) acc += P[(size_t)c * D + j] * dr[j];
        dkt[c] += bt * u[c] - acc;
      }
      // dP = dS - k dr^T ; dg = rowsum(dP * P) ; dS = diag(a) dP
      double dg_sum = 0.0;
      for (int c = 0; c < D; ++c) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j) {
          const double dP = dS[(size_t)c * D + j] - kt[c] * dr[j];
          acc += dP * P[(size_t)c * D + j];
          dS[(size_t)c * D + j] = a[c] * dP;
        }
        if (p->gate_per_channel)
          p->dg[((size_t)t * p->HV + ch.hv) * D + c] = acc;
        else
          dg_sum += acc;
      }
      if (!p->gate_per_channel) p->dg[(size_t)t * p->HV + ch.hv] = dg_sum;
    }
  }
  if (p->dh0) {
    double* dst = p->dh0 + ((size_t)ch.doc * p->HV + ch.hv) * DD;
    std::copy(dS.begin(), dS.end(), dst);
  }
}

}  // namespace

extern "C" {

// Runs the forward (and, when dout != null, the reverse pass) of every
// (document, value head) chain.  Work units are (document, Q/K head) groups,
// issued longest document first over a pool of threads; the value heads of a
// group run in order inside one unit, so dq/dk accumulate without races.
// Returns 0 on success, 1 on an invalid problem.
int gdr_oracle_run(const gdr_oracle_problem* p) {
  if (!p || p->N < 0 || p->T < 0 || p->D <= 0 || p->Hqk <= 0 || p->HV <= 0) return 1;
  if (p->HV % p->Hqk != 0) return 1;
  if (!p->cu_seqlens || p->cu_seqlens[0] != 0 || p->cu_seqlens[p->N] != p->T) return 1;
  for (int32_t n = 0; n < p->N; ++n)
    if (p->cu_seqlens[n + 1] < p->cu_seqlens[n]) return 1;
  const bool bwd = p->dout != nullptr;
  const int32_t G = p->HV / p->Hqk;
  if (bwd) {
    std::fill(p->dq, p->dq + (size_t)p->T * p->Hqk * p->D, 0.0);
    std::fill(p->dk, p->dk + (size_t)p->T * p->Hqk * p->D, 0.0);
  }
  struct Unit { int32_t doc, hq; int64_t len; };
  std::vector<Unit> units;
  for (int32_t n = 0; n < p->N; ++n)
    for (int32_t hq = 0; hq < p->Hqk; ++hq)
      units.push_back({n, hq, (int64_t)p->cu_seqlens[n + 1] - p->cu_seqlens[n]});
  std::stable_sort(units.begin(), units.end(), [](const Unit& a, const Unit& b) { return a.len > b.len; });

  int nthreads = p->threads > 0 ? p->threads : gdr_oracle_hardware_threads();
  if (nthreads > (int)units.size()) nthreads = (int)units.size();
  if (nthreads < 1) nthreads = 1;
  std::atomic<size_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const size_t i = next.fetch_add(1);
      if (i >= units.size()) return;
      const Unit& un = units[i];
      for (int32_t gi = 0; gi < G; ++gi) {
        Chain ch{p, un.doc, un.hq * G + gi, un.hq, (int64_t)p->cu_seqlens[un.doc], un.len};
        if (bwd)
          chain_bwd(p, ch);
        else
          chain_fwd(p, ch, 1, nullptr);
      }
    }
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nthreads; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return 0;
}

}  // extern "C"
