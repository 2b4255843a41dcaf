// FP64 CPU oracle for chunked-prefill causal GQA attention.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
// this file: only the test suite, the package smoke check and the benchmark's
// CPU-baseline leg use it. It shares no code, header or constant with the CUDA
// library.
//
// What it computes is the plain definition of the operation, written out with
// an explicit full-row softmax (no online rescaling, no tiling, no fusion):
//
//   For every query token t in [0, q_len) and query head h in [0, n_q_heads):
//     g    = h / (n_q_heads / n_kv_heads)
//            -- query heads 6g..6g+5 share KV head g: "KV head = query_head/6",
//               gfx936 DCU上实现INT8 QK MMAC：分页访存、Fragment映射与GQA适配, §5.2.
//     p    = kv_len - q_len + t
//            -- the chunk sits at the end of the K/V prefix, so token t has
//               absolute position p and its causal mask keeps keys 0..p
//               (DCU使用技术报告（中篇）, §3: later chunks of one request see a
//               longer kv_len; the chunk's own keys are the last q_len keys).
//     s_j  = scale * sum_c q[t,h,c] * k[j,g,c]        for j = 0..p  (QK^T)
//     m    = max_j s_j
//     e_j  = exp(s_j - m),  Z = sum_j e_j              (softmax)
//     out[t,h,c] = sum_j e_j * v[j,g,c] / Z            (PV)
//     lse[t,h]   = m + ln Z                            (natural log of the
//                                                        softmax normaliser of
//                                                        the scaled scores)
//   -- QK, causal mask, softmax, PV with wide accumulation:
//      DCU使用技术报告（中篇）, §2 "专用 Prefill Attention".
//
// Inputs are FP64 arrays (BF16 inputs are widened exactly by the caller).
// Rows are independent, so they are spread over std::threads; each row is
// computed by one thread start to finish, which makes the result independent
// of the thread count.
//
// Parity status: every output of this function is pinned by the CPU test
// suite (closed forms, textbook library special cases, invariants and a
// separate numpy restatement); nothing here is "parity unpinned".

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
  int64_t q_len, kv_len, hq, hkv, d;
  double scale;
  double* out;       // [n_rows, d] when rows given, else [q_len, hq, d]
  double* lse;       // [n_rows] or [q_len, hq]; may be null
  double* prob_sum;  // optional: sum_j e_j / Z per row
};

void one_row(const Problem& P, int64_t t, int64_t h, int64_t slot, std::vector<double>& s) {
  const int64_t group = P.hq / P.hkv;
  const int64_t g = h / group;
  const int64_t p = P.kv_len - P.q_len + t;  // last visible key
  const double* qrow = P.q + (t * P.hq + h) * P.d;
  s.assign(static_cast<size_t>(p + 1), 0.0);
  for (int64_t j = 0; j <= p; ++j) {
    const double* krow = P.k + (j * P.hkv + g) * P.d;
    double acc = 0.0;
    for (int64_t c = 0; c < P.d; ++c) acc += qrow[c] * krow[c];
    s[static_cast<size_t>(j)] = P.scale * acc;
  }
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j <= p; ++j) m = std::max(m, s[static_cast<size_t>(j)]);
  double Z = 0.0;
  for (int64_t j = 0; j <= p; ++j) {
    s[static_cast<size_t>(j)] = std::exp(s[static_cast<size_t>(j)] - m);
    Z += s[static_cast<size_t>(j)];
  }
  double* orow = P.out + slot * P.d;
  for (int64_t c = 0; c < P.d; ++c) orow[c] = 0.0;
  for (int64_t j = 0; j <= p; ++j) {
    const double w = s[static_cast<size_t>(j)];
    const double* vrow = P.v + (j * P.hkv + g) * P.d;
    for (int64_t c = 0; c < P.d; ++c) orow[c] += w * vrow[c];
  }
  for (int64_t c = 0; c < P.d; ++c) orow[c] /= Z;
  if (P.lse) P.lse[slot] = m + std::log(Z);
  if (P.prob_sum) {
    double sum = 0.0;
    for (int64_t j = 0; j <= p; ++j) sum += s[static_cast<size_t>(j)] / Z;
    P.prob_sum[slot] = sum;
  }
}

}  // namespace

extern "C" {

// Returns 0 on success, 1 on a bad argument.
//   q: [q_len, n_q_heads, head_dim]   k, v: [kv_len, n_kv_heads, head_dim]
//   rows: optional list of row ids t*n_q_heads + h (n_rows of them); when null,
//         every row is computed and out/lse/prob_sum are laid out
//         [q_len, n_q_heads, ...]; otherwise they are [n_rows, ...] in list order.
//   n_threads <= 0 means std::thread::hardware_concurrency().
int gqa_oracle_attn(const double* q, const double* k, const double* v,
                    int64_t q_len, int64_t kv_len, int64_t n_q_heads, int64_t n_kv_heads,
                    int64_t head_dim, double scale, const int64_t* rows, int64_t n_rows,
                    double* out, double* lse, double* prob_sum, int n_threads) {
  if (!q || !k || !v || !out) return 1;
  if (q_len < 0 || kv_len < q_len || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return 1;
  if (n_q_heads % n_kv_heads != 0) return 1;
  const int64_t total = rows ? n_rows : q_len * n_q_heads;
  if (rows) {
    for (int64_t i = 0; i < n_rows; ++i)
      if (rows[i] < 0 || rows[i] >= q_len * n_q_heads) return 1;
  }
  Problem P{q, k, v, q_len, kv_len, n_q_heads, n_kv_heads, head_dim, scale, out, lse, prob_sum};
  int nt = n_threads > 0 ? n_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (static_cast<int64_t>(nt) > total) nt = static_cast<int>(std::max<int64_t>(total, 1));
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    std::vector<double> s;
    for (;;) {
      const int64_t i = next.fetch_add(1);
      if (i >= total) break;
      const int64_t r = rows ? rows[i] : i;
      one_row(P, r / n_q_heads, r % n_q_heads, i, s);
    }
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return 0;
}

}  // extern "C"
