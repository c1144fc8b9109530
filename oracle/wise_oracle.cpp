/*
 * CPU oracle (C++) for WISE working-set paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, direct statement of
 * what one WISE decode call computes; the CUDA library is checked against it
 * and never links it, and it includes nothing of the library.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg load it (through
 * oracle/cpp_oracle.py).
 *
 * Every routine is a template over the arithmetic type T.  T = float is the
 * fp32 oracle (fp32 math throughout: scores, softmax, block masses, the
 * cumulative sum of the selection).  T = double is the same code in double
 * precision; the distance between the two bounds the fp32 oracle's own
 * rounding error.  No blocking, fusion or reordering: every sum runs in
 * ascending index order, one (row, query head) at a time.  Threads only split
 * the (row, query head) pairs among themselves, so the thread count never
 * changes a result.
 *
 * Source: the vllm-rlt pull request "WISE working-set decode" (PR #143), cited
 * as [WISE PR, <section>]:
 *   - dense rows attend the whole paged K/V; discover rows are dense and also
 *     record each 32-token tile's max and sum; sparse rows attend only their
 *     selected tiles ("What changes");
 *   - the finish merges and, for discover rows, applies the eta selection with
 *     B = 32 blocks and eta = 0.95 ("Summary") into a [slot, layer, head,
 *     block] support bitmask ("What changes"); union-discover ORs the new
 *     choice into the previous support (review "[P2] Distinguish discovery
 *     density from reused union density");
 *   - sparse output matches masked attention; LSE-derived block mass matches
 *     softmax block sums; compaction with every block selected is bitwise
 *     dense ("Tests").
 *
 * Readings where the pages are silent (the same ones the numpy oracle takes):
 *   - block = tile = 32 consecutive tokens from token 0; a row's last block
 *     holds only its valid tokens;
 *   - softmax scale 1/sqrt(D); LSE = natural log of sum exp(scale q.k);
 *   - selection: blocks in order of mass descending, equal masses by lower
 *     block index; the shortest prefix whose cumulative mass reaches eta;
 *     eta >= 1, or a cumulative sum that never reaches eta, keeps every
 *     block; at least one block is always kept;
 *   - grouped query heads: each query head selects on its own and the KV
 *     head's mask is the OR over its group;
 *   - padding rows (length 0): output 0, LSE -inf, mask untouched; a sparse
 *     row with no selected block attends the empty set (0, -inf);
 *   - a written mask has no bit at or past the row's block count.
 */
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <thread>
#include <vector>

namespace {

enum Mode { DENSE = 0, DISCOVER = 1, DISCOVER_UNION = 2, SPARSE = 3 };

}  // namespace

extern "C" {

/* One decode call's shapes.  Field order matches the ctypes mirror in
 * oracle/cpp_oracle.py. */
struct OracleProblem {
  int32_t rows, q_heads, kv_heads, head_dim;
  int32_t page_size, tile_tokens;
  int32_t max_pages_per_row, num_pages;
  int32_t mask_words;     /* W: u32 words per (row, KV head) mask */
  int32_t bf16_storage;   /* 1: q/K/V hold bfloat16 bit patterns (uint16); 0: float32 */
  double scale;           /* 0 means 1/sqrt(head_dim) */
  double eta;
};

/* Where the results go.  Arrays indexed [row][q head][block] have 32*W
 * blocks per (row, q head); the per-block and per-pair diagnostics are
 * written for discover and union-discover rows only. */
struct OracleResults {
  double* out;          /* [R, Hq, D]  attention output */
  double* lse;          /* [R, Hq] */
  uint32_t* support;    /* [R, Hkv, W]  the mask after the call */
  double* tile_max;     /* [R, Hq, 32W] m_b */
  double* tile_sum;     /* [R, Hq, 32W] l_b */
  double* mass;         /* [R, Hq, 32W] p_b */
  uint8_t* selected;    /* [R, Hq, 32W] 1 where block b is in this head's selection */
  int32_t* order;       /* [R, Hq, 32W] blocks in selection order */
  int32_t* k_star;      /* [R, Hq] */
  double* margin;       /* [R, Hq] */
  double* gap;          /* [R, Hq] */
};

}  // extern "C"

namespace {

/* The stored value of element idx: bfloat16 bits are the upper half of an
 * IEEE float32, so widening is exact. */
inline float stored(const void* base, bool bf16, size_t idx) {
  if (bf16) {
    uint32_t bits = uint32_t(static_cast<const uint16_t*>(base)[idx]) << 16;
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return f;
  }
  return static_cast<const float*>(base)[idx];
}

inline bool mask_bit(const uint32_t* words, int b) { return (words[b >> 5] >> (b & 31)) & 1u; }

/* The eta rule over n block masses [WISE PR, "Summary": B = 32 blocks and
 * the eta = 0.95 selection].  Writes the selection order, the chosen blocks
 * and k*; margin = min(C_k* - eta, eta - C_(k*-1)) with C_0 = 0 (+inf when
 * eta >= 1); gap = p_(k*) - p_(k*+1) in the order (+inf when k* = n). */
template <typename T>
int select_eta(const T* p, int n, double eta, int32_t* order, uint8_t* sel, double* margin,
               double* gap) {
  std::vector<int32_t> idx(n);
  std::iota(idx.begin(), idx.end(), 0);
  std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
    return p[a] > p[b] || (p[a] == p[b] && a < b);
  });
  const T eta_t = static_cast<T>(eta);
  std::vector<T> C(n);
  T run = 0;
  for (int i = 0; i < n; ++i) {
    run += p[idx[i]];
    C[i] = run;
  }
  int k = n;
  if (eta < 1.0) {
    for (int i = 0; i < n; ++i) {
      if (C[i] >= eta_t) {
        k = i + 1;
        break;
      }
    }
  }
  for (int i = 0; i < n; ++i) {
    order[i] = idx[i];
    sel[i] = 0;
  }
  for (int i = 0; i < k; ++i) sel[idx[i]] = 1;
  const double inf = std::numeric_limits<double>::infinity();
  if (eta >= 1.0) {
    *margin = inf;
  } else {
    double prev = k >= 2 ? double(C[k - 2]) : 0.0;
    *margin = std::min(double(C[k - 1]) - eta, eta - prev);
  }
  *gap = k < n ? double(p[idx[k - 1]]) - double(p[idx[k]]) : inf;
  return k;
}

/* One (row r, query head h) of one decode call. */
template <typename T>
void decode_pair(const OracleProblem& P, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* page_table, const int32_t* seq_lens, const int8_t* modes,
                 const uint32_t* support_in, OracleResults& res, int r, int h,
                 std::vector<T>& s, std::vector<T>& e, std::vector<T>& acc, std::vector<T>& pm) {
  const int D = P.head_dim, Hq = P.q_heads, Hkv = P.kv_heads, W = P.mask_words;
  const int NB = 32 * W;
  const int G = Hq / Hkv;
  const int g = h / G;
  const int B = P.tile_tokens, PS = P.page_size;
  const bool bf16 = P.bf16_storage != 0;
  const size_t pair = size_t(r) * Hq + h;
  double* out = res.out + pair * D;
  const int L = seq_lens[r];
  const int mode = modes[r];
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  res.lse[pair] = -std::numeric_limits<double>::infinity();
  res.k_star[pair] = 0;
  if (L <= 0) return;  // padding row
  const int nb = (L + B - 1) / B;
  const T scale = P.scale != 0.0 ? static_cast<T>(P.scale)
                                 : static_cast<T>(1) / std::sqrt(static_cast<T>(D));
  const uint32_t* words = support_in + (size_t(r) * Hkv + g) * W;

  // 1. Scores of every token: paged gather (token j sits in page
  //    page_table[r][j / page_size] at slot j % page_size) and a dot product
  //    accumulated in ascending d.
  s.assign(L, 0);
  for (int j = 0; j < L; ++j) {
    const int32_t page = page_table[size_t(r) * P.max_pages_per_row + j / PS];
    const size_t krow = ((size_t(page) * PS + j % PS) * Hkv + g) * D;
    T dot = 0;
    for (int d = 0; d < D; ++d)
      dot += static_cast<T>(stored(q, bf16, pair * D + d)) * static_cast<T>(stored(k_cache, bf16, krow + d));
    s[j] = scale * dot;
  }

  // 2. The active tokens: all of them, or for sparse rows those whose block
  //    is selected [WISE PR, "Tests": sparse output matches masked attention].
  auto active = [&](int j) { return mode != SPARSE || mask_bit(words, j / B); };

  // 3. Softmax over the active tokens: max, exponentials, their sum in
  //    ascending j, the weighted sum of V rows, then one division.
  bool any = false;
  T m = 0;
  for (int j = 0; j < L; ++j) {
    if (!active(j)) continue;
    if (!any || s[j] > m) m = s[j];
    any = true;
  }
  if (!any) return;  // empty support: output 0, LSE -inf
  e.assign(L, 0);
  T Z = 0;
  for (int j = 0; j < L; ++j) {
    if (!active(j)) continue;
    e[j] = std::exp(s[j] - m);
    Z += e[j];
  }
  acc.assign(D, 0);
  for (int j = 0; j < L; ++j) {
    if (!active(j)) continue;
    const int32_t page = page_table[size_t(r) * P.max_pages_per_row + j / PS];
    const size_t vrow = ((size_t(page) * PS + j % PS) * Hkv + g) * D;
    for (int d = 0; d < D; ++d) acc[d] += e[j] * static_cast<T>(stored(v_cache, bf16, vrow + d));
  }
  for (int d = 0; d < D; ++d) out[d] = double(acc[d] / Z);
  const T lse = m + std::log(Z);
  res.lse[pair] = double(lse);

  if (mode != DISCOVER && mode != DISCOVER_UNION) return;

  // 4. Discover rows: per tile the max and the sum of exp(s - m_b) [WISE PR,
  //    "What changes"], and the block masses p_b = (sum of the block's e_j) / Z,
  //    summed explicitly token by token; then the eta rule.
  pm.assign(nb, 0);
  double* tmax = res.tile_max + pair * NB;
  double* tsum = res.tile_sum + pair * NB;
  double* mass = res.mass + pair * NB;
  for (int b = 0; b < nb; ++b) {
    const int lo = b * B, hi = std::min(L, lo + B);
    T mb = s[lo];
    for (int j = lo + 1; j < hi; ++j) mb = std::max(mb, s[j]);
    T lb = 0, eb = 0;
    for (int j = lo; j < hi; ++j) {
      lb += std::exp(s[j] - mb);
      eb += e[j];
    }
    pm[b] = eb / Z;
    tmax[b] = double(mb);
    tsum[b] = double(lb);
    mass[b] = double(pm[b]);
  }
  res.k_star[pair] = select_eta<T>(pm.data(), nb, P.eta, res.order + pair * NB,
                                   res.selected + pair * NB, res.margin + pair, res.gap + pair);
}

/* One decode call over the batch. */
template <typename T>
int decode(const OracleProblem* Pp, const void* q, const void* k_cache, const void* v_cache,
           const int32_t* page_table, const int32_t* seq_lens, const int8_t* modes,
           const uint32_t* support_in, OracleResults* res, int threads) {
  const OracleProblem& P = *Pp;
  if (P.rows < 0 || P.q_heads <= 0 || P.kv_heads <= 0 || P.q_heads % P.kv_heads != 0 ||
      P.head_dim <= 0 || P.page_size <= 0 || P.tile_tokens <= 0 || P.mask_words <= 0)
    return -1;
  const int pairs = P.rows * P.q_heads;
  if (threads <= 0) threads = int(std::max(1u, std::thread::hardware_concurrency()));
  threads = std::max(1, std::min(threads, pairs));
  std::atomic<int> next{0};
  auto worker = [&]() {
    std::vector<T> s, e, acc, pm;
    for (int i = next.fetch_add(1); i < pairs; i = next.fetch_add(1))
      decode_pair<T>(P, q, k_cache, v_cache, page_table, seq_lens, modes, support_in, *res,
                     i / P.q_heads, i % P.q_heads, s, e, acc, pm);
  };
  if (threads == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < threads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
  }

  // 5. Masks: discover writes the OR of the group's selections, union-discover
  //    ORs it into the previous mask; bits at or past the row's block count
  //    are cleared; dense, sparse and padding rows keep the mask they had.
  const int W = P.mask_words, G = P.q_heads / P.kv_heads, NB = 32 * W;
  for (int r = 0; r < P.rows; ++r) {
    const int L = seq_lens[r];
    const int nb = L > 0 ? (L + P.tile_tokens - 1) / P.tile_tokens : 0;
    for (int g = 0; g < P.kv_heads; ++g) {
      const uint32_t* before = support_in + (size_t(r) * P.kv_heads + g) * W;
      uint32_t* after = res->support + (size_t(r) * P.kv_heads + g) * W;
      for (int w = 0; w < W; ++w) after[w] = before[w];
      if (L <= 0 || (modes[r] != DISCOVER && modes[r] != DISCOVER_UNION)) continue;
      for (int w = 0; w < W; ++w) after[w] = 0;
      for (int b = 0; b < nb; ++b) {
        bool bit = modes[r] == DISCOVER_UNION && mask_bit(before, b);
        for (int h = g * G; h < (g + 1) * G; ++h)
          bit = bit || res->selected[(size_t(r) * P.q_heads + h) * NB + b] != 0;
        if (bit) after[b >> 5] |= 1u << (b & 31);
      }
    }
  }
  return threads;
}

}  // namespace

extern "C" {

/* One WISE decode call (one layer at one depth) for the whole batch.
 * q [R, Hq, D]; k_cache, v_cache [num_pages, page_size, Hkv, D];
 * page_table int32 [R, max_pages_per_row]; seq_lens int32 [R]; modes int8 [R]
 * (0 dense, 1 discover, 2 union-discover, 3 sparse); support_in uint32
 * [R, Hkv, W], the mask before the call.  threads <= 0 uses every hardware
 * thread.  Returns the number of threads used, or -1 for an invalid shape. */
int wise_oracle_decode_f32(const OracleProblem* P, const void* q, const void* k, const void* v,
                           const int32_t* page_table, const int32_t* seq_lens, const int8_t* modes,
                           const uint32_t* support_in, OracleResults* res, int threads) {
  return decode<float>(P, q, k, v, page_table, seq_lens, modes, support_in, res, threads);
}

int wise_oracle_decode_f64(const OracleProblem* P, const void* q, const void* k, const void* v,
                           const int32_t* page_table, const int32_t* seq_lens, const int8_t* modes,
                           const uint32_t* support_in, OracleResults* res, int threads) {
  return decode<double>(P, q, k, v, page_table, seq_lens, modes, support_in, res, threads);
}

/* The eta rule alone on n given masses, taken in float (f32) or as they are
 * (f64).  Returns k*. */
int wise_oracle_select_f32(const double* p, int n, double eta, int32_t* order, uint8_t* sel,
                           double* margin, double* gap) {
  std::vector<float> pf(p, p + n);
  return select_eta<float>(pf.data(), n, eta, order, sel, margin, gap);
}

int wise_oracle_select_f64(const double* p, int n, double eta, int32_t* order, uint8_t* sel,
                           double* margin, double* gap) {
  return select_eta<double>(p, n, eta, order, sel, margin, gap);
}

/* dst | src, word by word [review "[P2] Distinguish discovery density from
 * reused union density": the chosen blocks are ORed into the support]. */
void wise_oracle_support_union(const uint32_t* dst, const uint32_t* src, uint32_t* out,
                               int64_t n_words) {
  for (int64_t i = 0; i < n_words; ++i) out[i] = dst[i] | src[i];
}

/* Head union [WISE PR, "What changes", FlashAttention decode bullet]: every
 * KV head of a row gets each block that any KV head of the row selected,
 * decided bit by bit. */
void wise_oracle_head_union(const uint32_t* support, int rows, int kv_heads, int words,
                            uint32_t* out) {
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < 32 * words; ++b) {
      bool any = false;
      for (int g = 0; g < kv_heads; ++g)
        any = any || mask_bit(support + (size_t(r) * kv_heads + g) * words, b);
      for (int g = 0; g < kv_heads; ++g) {
        uint32_t& w = out[(size_t(r) * kv_heads + g) * words + (b >> 5)];
        if (b % 32 == 0) w = 0;
        if (any) w |= 1u << (b & 31);
      }
    }
  }
}

/* Selected blocks of the final union over causal blocks, over every
 * (row, KV head) of a non-empty row [author's reply to the review: a union
 * depth adds only newly set blocks, so two disjoint one-block choices over
 * two blocks give 1.0]. */
double wise_oracle_union_density(const uint32_t* support, const int32_t* seq_lens, int rows,
                                 int kv_heads, int words, int tile_tokens) {
  int64_t sel = 0, causal = 0;
  for (int r = 0; r < rows; ++r) {
    const int nb = seq_lens[r] > 0 ? (seq_lens[r] + tile_tokens - 1) / tile_tokens : 0;
    for (int g = 0; g < kv_heads; ++g) {
      for (int b = 0; b < nb; ++b) sel += mask_bit(support + (size_t(r) * kv_heads + g) * words, b);
      causal += nb;
    }
  }
  return causal ? double(sel) / double(causal) : 0.0;
}

/* The compacted tile lists [WISE PR, "What changes": sparse rows attend only
 * their selected tiles, compacted first so the loop has no branch].  Per
 * (row, KV head) the list is the ascending selected blocks below the row's
 * block count (sparse rows) or every block (other modes), written to
 * lists [R, Hkv, 32W] with its length in counts [R, Hkv].  How the lists are
 * cut into work items is the kernel's scheduling choice, not part of the
 * definition. */
void wise_oracle_compact(const uint32_t* support, const int8_t* modes, const int32_t* seq_lens,
                         int rows, int kv_heads, int words, int tile_tokens, int32_t* lists,
                         int32_t* counts) {
  const int NB = 32 * words;
  for (int r = 0; r < rows; ++r) {
    const int nb = seq_lens[r] > 0 ? (seq_lens[r] + tile_tokens - 1) / tile_tokens : 0;
    for (int g = 0; g < kv_heads; ++g) {
      const uint32_t* w = support + (size_t(r) * kv_heads + g) * words;
      int32_t* lst = lists + (size_t(r) * kv_heads + g) * NB;
      int c = 0;
      for (int b = 0; b < nb; ++b)
        if (modes[r] != SPARSE || mask_bit(w, b)) lst[c++] = b;
      counts[size_t(r) * kv_heads + g] = c;
    }
  }
}

}  // extern "C"
