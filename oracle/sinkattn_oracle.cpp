// fp64 CPU oracle for causal / windowed / varlen attention with learnable
// per-head sink logits.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg may load this library. The CUDA library shares
// no code with it; the product path never calls it.
//
// What it computes (page "GPT-OSS Agentic RL Training: A Practical
// Retrospective", section "The Role of Attention Sinks": each head owns one
// learnable scalar that behaves like a virtual token inside the softmax; section
// "Implementation in FlashAttention v3": a forward with sinks and a backward
// that also yields dL/dS_h). The pages give no formula; the plain reading used
// here is: the sink adds exp(S_h) to the softmax denominator and carries no
// value. Per sequence b, query head h, local query row i, allowed key j:
//
//   s_ij    = scale * <q_i, k_j>             (k, v from kv head h / G)
//   LSE_i   = log( exp(S_h) + sum_j exp(s_ij) )
//   P_ij    = exp(s_ij - LSE_i),  p_sink_i = exp(S_h - LSE_i)
//   O_i     = sum_j P_ij v_j
//   D_i     = <dO_i, O_i>
//   dP_ij   = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i)
//   dq_i    = scale * sum_j dS_ij k_j
//   dk_j    = scale * sum_{h in group} sum_i dS_ij q_i
//   dv_j    = sum_{h in group} sum_i P_ij dO_i
//   dS_h    = - sum_{b,i} p_sink_i D_i
//
// allowed(i, j) = (causal ? j <= i : true) and (window > 0 ? i - j < window : true).
//
// Every quantity is fp64. Rows are processed one at a time, with two passes
// over the row's scores (max, then exponentials). No tiling, no online
// rescaling, no fusion: each output element is its defining sum.
//
// Threads only split independent output elements; the per-head sink gradient
// is formed from per-(b, h, chunk) partials that are added in a fixed order,
// so results do not depend on the thread count.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

struct Problem {
  const double* q;
  const double* k;
  const double* v;
  const double* sinks;  // may be null: no sink (S_h = -inf)
  const double* dout;   // may be null: forward only
  const int32_t* cu;
  int32_t nseq, Hq, Hkv, d, causal, window;
  int32_t first_row;  // rows and keys below this local index are skipped
  double scale;
};

constexpr int kChunk = 32;  // rows (or keys) per work unit

inline bool allowed(const Problem& p, int64_t i, int64_t j) {
  if (p.causal && j > i) return false;
  if (p.window > 0 && i - j >= p.window) return false;
  return true;
}

// The keys of row i that allowed() admits form one interval [lo, hi): the
// loops below walk that interval and still test allowed() on each pair.
inline void keys_of_row(const Problem& p, int64_t i, int64_t L, int64_t* lo, int64_t* hi) {
  *hi = p.causal ? i + 1 : L;
  *lo = p.window > 0 ? std::max<int64_t>(0, i - p.window + 1) : 0;
}

// Likewise the rows that may use key j.
inline void rows_of_key(const Problem& p, int64_t j, int64_t L, int64_t* lo, int64_t* hi) {
  *lo = p.causal ? j : 0;
  *hi = p.window > 0 ? std::min<int64_t>(L, j + p.window) : L;
}

inline double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
  for (int t = 0; t < d; ++t) acc += a[t] * b[t];
  return acc;
}

inline double sink_of(const Problem& p, int h) {
  return p.sinks ? p.sinks[h] : -std::numeric_limits<double>::infinity();
}

// Run fn(unit) for unit in [0, n) over nthreads std::threads.
template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (nthreads < 1) nthreads = 1;
  if (n <= 0) return;
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      int64_t u = next.fetch_add(1);
      if (u >= n) break;
      fn(u);
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

struct Unit {
  int32_t b, head;  // head: q head (row units) or kv head (key units)
  int64_t first;    // first local row / key of the chunk
};

std::vector<Unit> make_units(const Problem& p, int heads) {
  std::vector<Unit> units;
  for (int32_t b = 0; b < p.nseq; ++b) {
    const int64_t L = p.cu[b + 1] - p.cu[b];
    for (int h = 0; h < heads; ++h)
      for (int64_t r = p.first_row; r < L; r += kChunk) units.push_back({b, h, r});
  }
  return units;
}

}  // namespace

extern "C" {

// Returns 0 on success, nonzero on bad arguments.
//
// Layouts (contiguous, row-major):
//   q, dout, o, dq : [total, Hq, d]      k, v, dk, dv : [total, Hkv, d]
//   lse            : [Hq, total]         sinks, dsinks : [Hq]
// total = cu_seqlens[nseq]. Any output pointer may be null to skip it.
// dq/dk/dv/dsinks need dout. When sinks is null the sink is absent and
// dsinks, if requested, is all zero.
//
// first_row > 0 restricts the work to local rows >= first_row and keys >=
// first_row of every sequence (outputs elsewhere are left untouched, and
// dsinks sums only those rows). Under a causal mask the rows that see such a
// key all lie in that range, so dk and dv there are still complete; the rows
// themselves always see all their keys.
int oracle_sinkattn(const double* q, const double* k, const double* v,
                    const double* sinks, const double* dout,
                    const int32_t* cu_seqlens, int32_t nseq, int32_t Hq,
                    int32_t Hkv, int32_t d, int32_t causal, int32_t window,
                    double scale, int32_t first_row, double* o, double* lse,
                    double* dq, double* dk, double* dv, double* dsinks,
                    int32_t nthreads) {
  if (!q || !k || !v || !cu_seqlens || nseq < 0 || Hq <= 0 || Hkv <= 0 ||
      d <= 0 || Hq % Hkv != 0)
    return 1;
  if (window > 0 && !causal) return 1;
  if (first_row < 0 || (first_row > 0 && !causal)) return 1;
  if ((dq || dk || dv || dsinks) && !dout) return 1;
  for (int32_t b = 0; b < nseq; ++b)
    if (cu_seqlens[b + 1] < cu_seqlens[b]) return 1;
  if (cu_seqlens[0] != 0) return 1;

  Problem p{q, k, v, sinks, dout, cu_seqlens, nseq, Hq, Hkv, d, causal, window, first_row, scale};
  const int G = Hq / Hkv;
  const int64_t total = cu_seqlens[nseq];
  const bool want_bwd = dq || dk || dv || dsinks;

  // Row quantities kept for the key pass: LSE and D per (h, token).
  std::vector<double> lse_all((size_t)Hq * total, 0.0);
  std::vector<double> D_all(want_bwd ? (size_t)Hq * total : 0, 0.0);

  // ---- pass over query rows: LSE, O, D, dq, sink-gradient partials ----
  std::vector<Unit> rows = make_units(p, Hq);
  std::vector<double> sink_part(rows.size(), 0.0);
  parallel_for((int64_t)rows.size(), nthreads, [&](int64_t u) {
    const Unit un = rows[u];
    const int h = un.head, kvh = h / G;
    const int64_t base = cu_seqlens[un.b];
    const int64_t L = cu_seqlens[un.b + 1] - base;
    const double S = sink_of(p, h);
    std::vector<double> s(L), P(L), o_row(d), dq_row(d);
    double part = 0.0;
    for (int64_t i = un.first; i < std::min<int64_t>(un.first + kChunk, L); ++i) {
      const double* qi = q + ((base + i) * Hq + h) * d;
      int64_t jlo, jhi;
      keys_of_row(p, i, L, &jlo, &jhi);
      // first pass: scores and their maximum (the sink logit included)
      double M = S;
      for (int64_t j = jlo; j < jhi; ++j) {
        if (!allowed(p, i, j)) continue;
        s[j] = scale * dot(qi, k + ((base + j) * Hkv + kvh) * d, d);
        M = std::max(M, s[j]);
      }
      // second pass: normaliser, LSE, probabilities, output row
      double Z = std::isinf(S) ? 0.0 : std::exp(S - M);
      for (int64_t j = jlo; j < jhi; ++j)
        if (allowed(p, i, j)) Z += std::exp(s[j] - M);
      const double LSE = M + std::log(Z);
      lse_all[(size_t)h * total + base + i] = LSE;
      std::fill(o_row.begin(), o_row.end(), 0.0);
      for (int64_t j = jlo; j < jhi; ++j) {
        if (!allowed(p, i, j)) continue;
        P[j] = std::exp(s[j] - LSE);
        const double* vj = v + ((base + j) * Hkv + kvh) * d;
        for (int t = 0; t < d; ++t) o_row[t] += P[j] * vj[t];
      }
      if (o) std::copy(o_row.begin(), o_row.end(), o + ((base + i) * Hq + h) * d);
      if (!want_bwd) continue;
      const double* doi = dout + ((base + i) * Hq + h) * d;
      const double Di = dot(doi, o_row.data(), d);
      D_all[(size_t)h * total + base + i] = Di;
      const double p_sink = std::isinf(S) ? 0.0 : std::exp(S - LSE);
      part += -p_sink * Di;
      if (dq) {
        std::fill(dq_row.begin(), dq_row.end(), 0.0);
        for (int64_t j = jlo; j < jhi; ++j) {
          if (!allowed(p, i, j)) continue;
          const double* vj = v + ((base + j) * Hkv + kvh) * d;
          const double* kj = k + ((base + j) * Hkv + kvh) * d;
          const double dS = P[j] * (dot(doi, vj, d) - Di);
          for (int t = 0; t < d; ++t) dq_row[t] += scale * dS * kj[t];
        }
        std::copy(dq_row.begin(), dq_row.end(), dq + ((base + i) * Hq + h) * d);
      }
    }
    sink_part[u] = part;
  });

  if (lse)
    for (int32_t b = 0; b < nseq; ++b)
      for (int h = 0; h < Hq; ++h)
        for (int64_t t = cu_seqlens[b] + first_row; t < cu_seqlens[b + 1]; ++t)
          lse[(size_t)h * total + t] = lse_all[(size_t)h * total + t];

  if (dsinks) {
    for (int h = 0; h < Hq; ++h) dsinks[h] = 0.0;
    for (size_t u = 0; u < rows.size(); ++u) dsinks[rows[u].head] += sink_part[u];
  }

  // ---- pass over keys: dk, dv, summed over the kv head's query heads ----
  if (dk || dv) {
    std::vector<Unit> keys = make_units(p, Hkv);
    parallel_for((int64_t)keys.size(), nthreads, [&](int64_t u) {
      const Unit un = keys[u];
      const int kvh = un.head;
      const int64_t base = cu_seqlens[un.b];
      const int64_t L = cu_seqlens[un.b + 1] - base;
      std::vector<double> dk_row(d), dv_row(d);
      for (int64_t j = un.first; j < std::min<int64_t>(un.first + kChunk, L); ++j) {
        const double* kj = k + ((base + j) * Hkv + kvh) * d;
        const double* vj = v + ((base + j) * Hkv + kvh) * d;
        std::fill(dk_row.begin(), dk_row.end(), 0.0);
        std::fill(dv_row.begin(), dv_row.end(), 0.0);
        int64_t ilo, ihi;
        rows_of_key(p, j, L, &ilo, &ihi);
        for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
          for (int64_t i = ilo; i < ihi; ++i) {
            if (!allowed(p, i, j)) continue;
            const double* qi = q + ((base + i) * Hq + h) * d;
            const double* doi = dout + ((base + i) * Hq + h) * d;
            const double sij = scale * dot(qi, kj, d);
            const double Pij = std::exp(sij - lse_all[(size_t)h * total + base + i]);
            const double dS = Pij * (dot(doi, vj, d) - D_all[(size_t)h * total + base + i]);
            for (int t = 0; t < d; ++t) {
              dv_row[t] += Pij * doi[t];
              dk_row[t] += scale * dS * qi[t];
            }
          }
        }
        if (dk) std::copy(dk_row.begin(), dk_row.end(), dk + ((base + j) * Hkv + kvh) * d);
        if (dv) std::copy(dv_row.begin(), dv_row.end(), dv + ((base + j) * Hkv + kvh) * d);
      }
    });
  }
  return 0;
}

}  // extern "C"
