// BeaconKV eviction step -- plain CPU reference ("the oracle").
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
// calls this file: only the tests, the package smoke check and the
// benchmark's CPU-baseline leg do.  It shares no code, header, table or
// helper with the CUDA library.
//
// Every routine is single-threaded and works in fp64 from the same bf16
// inputs the GPU path reads.  It follows the method as the BeaconKV pages
// state it, step by step, with no blocking, fusion or reordering:
//
//  * FPS seed and greedy step, pre-rotation similarity:
//      wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫FPS的采样算法"
//      (start from the query with the lowest mean similarity to the others,
//      then repeatedly add the query farthest from / least similar to the
//      chosen set; similarity is taken before RoPE).
//  * Continual FPS buffer: same section (each head keeps a bounded buffer;
//    when it is full an FPS pass compresses it back to a smaller size; repeat).
//  * Beacon re-rotation to the current position, recent queries at their own
//    positions, max aggregation:
//      wzjinhao.cn explainer, section "信标查询怎么用：位置对齐与打分策略".
//  * I = TopK(score(K,V), B_KV): inkeast.github.io reading, section 三
//    (problem formalisation).
//  * A recent sliding window is always kept; highest-scoring entries
//    survive: aimodeling.com article, section "用信标 query 预判" /
//    "The mechanism has three parts".
//
// Readings taken where the pages are silent:
//  - an FPS item is the concatenated G*d pre-rotation vector of one decode
//    step of one KV head; distance = 1 - cosine; a zero vector has cosine 0
//    with everything;
//  - ties (seed, greedy, top-k) go to the lowest index;
//  - after a compress the survivors stay in arrival (ascending) order;
//  - beacons at an eviction = FPS of the current buffer contents;
//  - rotary embedding is rotate-half with freq_i = theta^(-2i/d);
//  - a recent query at position p sees keys with position <= p; beacons
//    (at the current position) see the whole cache;
//  - the B_KV kept entries include the always-kept window of R slots.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Cosine-similarity matrix of n items of dimension D (fp64).
std::vector<double> cosine_matrix(const uint16_t* X, int n, int D) {
  std::vector<double> unit(static_cast<size_t>(n) * D);
  for (int i = 0; i < n; ++i) {
    double ss = 0.0;
    for (int k = 0; k < D; ++k) {
      double v = bf16_value(X[static_cast<size_t>(i) * D + k]);
      ss += v * v;
    }
    double norm = std::sqrt(ss);
    for (int k = 0; k < D; ++k) {
      double v = bf16_value(X[static_cast<size_t>(i) * D + k]);
      unit[static_cast<size_t>(i) * D + k] = norm > 0.0 ? v / norm : 0.0;
    }
  }
  std::vector<double> S(static_cast<size_t>(n) * n);
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double s = 0.0;
      for (int k = 0; k < D; ++k)
        s += unit[static_cast<size_t>(i) * D + k] * unit[static_cast<size_t>(j) * D + k];
      S[static_cast<size_t>(i) * n + j] = s;
    }
  return S;
}

}  // namespace

extern "C" {

// Farthest point sampling of m items out of n (rows of X, each D bf16).
// Writes the selection order to sel[0..ret) and returns ret = min(n, m)
// (0 when m <= 0).  When radius is not null, radius[k] (k < ret) receives
// the covering radius max_i min_{s in first k+1 picks} (1 - cos(x_i, x_s)).
int ora_fps(const uint16_t* X, int n, int D, int m, int32_t* sel, double* radius) {
  if (m <= 0 || n <= 0) return 0;
  if (n <= m) {
    // fewer items than wanted: all of them, in index order
    for (int i = 0; i < n; ++i) {
      sel[i] = i;
      if (radius) radius[i] = 0.0;
    }
    return n;
  }
  std::vector<double> S = cosine_matrix(X, n, D);
  // seed: lowest mean similarity to the other items (ties -> lowest index).
  // The sum over the others is the whole row, summed in slot order, minus
  // the item's own term: two identical items then get the same value bit
  // for bit, so an exact tie is decided by the index, not by rounding.
  int seed = 0;
  double seed_val = std::numeric_limits<double>::infinity();
  for (int i = 0; i < n; ++i) {
    double sum = 0.0;
    for (int j = 0; j < n; ++j) sum += S[static_cast<size_t>(i) * n + j];
    sum -= S[static_cast<size_t>(i) * n + i];
    double mean = sum / static_cast<double>(n - 1);
    if (mean < seed_val) {
      seed_val = mean;
      seed = i;
    }
  }
  std::vector<char> chosen(n, 0);
  std::vector<double> dist(n);
  sel[0] = seed;
  chosen[seed] = 1;
  for (int i = 0; i < n; ++i) dist[i] = 1.0 - S[static_cast<size_t>(seed) * n + i];
  auto covering = [&]() {
    double r = 0.0;
    for (int i = 0; i < n; ++i)
      if (!chosen[i]) r = std::max(r, dist[i]);
    return r;
  };
  if (radius) radius[0] = covering();
  for (int k = 1; k < m; ++k) {
    // farthest unselected item (ties -> lowest index)
    int best = -1;
    double best_val = -std::numeric_limits<double>::infinity();
    for (int i = 0; i < n; ++i)
      if (!chosen[i] && dist[i] > best_val) {
        best_val = dist[i];
        best = i;
      }
    sel[k] = best;
    chosen[best] = 1;
    for (int i = 0; i < n; ++i)
      dist[i] = std::min(dist[i], 1.0 - S[static_cast<size_t>(best) * n + i]);
    if (radius) radius[k] = covering();
  }
  return m;
}

// One decode step of the continual buffer: append item x (D bf16) at slot
// *cnt; if the buffer then holds C items, keep the M FPS survivors in
// arrival order and set *cnt = M.  Returns 1 when a compress happened,
// -1 on a bad state, else 0.
int ora_buffer_push(uint16_t* buf, int32_t* cnt, const uint16_t* x, int D, int C, int M) {
  if (*cnt < 0 || *cnt >= C) return -1;
  std::memcpy(buf + static_cast<size_t>(*cnt) * D, x, sizeof(uint16_t) * D);
  *cnt += 1;
  if (*cnt < C) return 0;
  std::vector<int32_t> sel(C);
  int got = ora_fps(buf, C, D, M, sel.data(), nullptr);
  std::sort(sel.begin(), sel.begin() + got);
  std::vector<uint16_t> keep(static_cast<size_t>(got) * D);
  for (int i = 0; i < got; ++i)
    std::memcpy(keep.data() + static_cast<size_t>(i) * D, buf + static_cast<size_t>(sel[i]) * D,
                sizeof(uint16_t) * D);
  std::memcpy(buf, keep.data(), sizeof(uint16_t) * keep.size());
  *cnt = got;
  return 1;
}

// Rotate-half rotary embedding of one d-vector at integer position pos.
void ora_rope(const double* x, int d, int64_t pos, double theta, double* out) {
  int h = d / 2;
  for (int i = 0; i < h; ++i) {
    double freq = std::pow(theta, -2.0 * i / static_cast<double>(d));
    double a = static_cast<double>(pos) * freq;
    double c = std::cos(a), s = std::sin(a);
    double x0 = x[i], x1 = x[i + h];
    out[i] = x0 * c - x1 * s;
    out[i + h] = x1 * c + x0 * s;
  }
}

// Eviction scores of one unit.
//   K [L][d] bf16 (cached, already rotated), kpos [L]
//   ring [W][G][d] bf16 pre-rotation recent queries; slot s holds decode
//     step t with t % W == s; `step` is the newest step written
//   beacons [nb][G][d] bf16 pre-rotation
// Rows: every written ring slot (age a = (step - s) mod W <= step) at
// position cur_pos - a, and every beacon at cur_pos; each row carries its G
// head-queries.  A row sees key j when kpos[j] <= its position (causal != 0)
// or always (causal == 0).  P = softmax(q . k / sqrt(d)) over visible keys.
// agg == 0: score_j = max over rows of P[row][j]; agg == 1: mean over rows.
// Optional outputs: P [(W + nb) * G][L] (rows of unwritten ring slots and
// invisible entries are 0) and row_pos [(W + nb) * G] (-1 for unwritten).
void ora_score(int d, int G, int W, int nb, int L, double theta, int agg, int causal,
               const uint16_t* K, const int32_t* kpos, const uint16_t* ring, int64_t step,
               const uint16_t* beacons, int64_t cur_pos, double* scores, double* P,
               int64_t* row_pos) {
  const int rows = (W + nb) * G;
  std::vector<double> q(d), qr(d), logit(L);
  std::vector<char> vis(L);
  for (int j = 0; j < L; ++j) scores[j] = 0.0;
  if (P) std::fill(P, P + static_cast<size_t>(rows) * L, 0.0);
  int used_rows = 0;
  for (int r = 0; r < rows; ++r) {
    int item = r / G, g = r % G;
    const uint16_t* src;
    int64_t pos;
    if (item < W) {
      int64_t age = ((step - item) % W + W) % W;
      if (age > step) {  // slot never written
        if (row_pos) row_pos[r] = -1;
        continue;
      }
      pos = cur_pos - age;
      src = ring + (static_cast<size_t>(item) * G + g) * d;
    } else {
      pos = cur_pos;
      src = beacons + (static_cast<size_t>(item - W) * G + g) * d;
    }
    if (row_pos) row_pos[r] = pos;
    for (int k = 0; k < d; ++k) q[k] = bf16_value(src[k]);
    ora_rope(q.data(), d, pos, theta, qr.data());
    double mx = -std::numeric_limits<double>::infinity();
    int nvis = 0;
    for (int j = 0; j < L; ++j) {
      vis[j] = (!causal || kpos[j] <= pos) ? 1 : 0;
      if (!vis[j]) continue;
      double s = 0.0;
      for (int k = 0; k < d; ++k) s += qr[k] * bf16_value(K[static_cast<size_t>(j) * d + k]);
      logit[j] = s / std::sqrt(static_cast<double>(d));
      mx = std::max(mx, logit[j]);
      ++nvis;
    }
    ++used_rows;
    if (nvis == 0) continue;
    double z = 0.0;
    for (int j = 0; j < L; ++j)
      if (vis[j]) z += std::exp(logit[j] - mx);
    for (int j = 0; j < L; ++j) {
      if (!vis[j]) continue;
      double p = std::exp(logit[j] - mx) / z;
      if (P) P[static_cast<size_t>(r) * L + j] = p;
      if (agg == 0)
        scores[j] = std::max(scores[j], p);
      else
        scores[j] += p;
    }
  }
  if (agg == 1 && used_rows > 0)
    for (int j = 0; j < L; ++j) scores[j] /= static_cast<double>(used_rows);
}

// Kept slots of one unit (ascending) -> kept[0..ret).  If L <= B every slot
// stays.  Else the last R slots stay, plus the B - R highest-scoring of the
// other slots (ties -> lower slot).
int ora_select(int L, int B, int R, const double* scores, int32_t* kept) {
  if (L <= B) {
    for (int i = 0; i < L; ++i) kept[i] = i;
    return L;
  }
  int ncand = L - R;
  std::vector<int32_t> idx(ncand);
  for (int i = 0; i < ncand; ++i) idx[i] = i;
  std::stable_sort(idx.begin(), idx.end(),
                   [&](int32_t a, int32_t b) { return scores[a] > scores[b]; });
  std::vector<int32_t> keep(idx.begin(), idx.begin() + (B - R));
  for (int j = L - R; j < L; ++j) keep.push_back(j);
  std::sort(keep.begin(), keep.end());
  for (int i = 0; i < B; ++i) kept[i] = keep[i];
  return B;
}

// In-place compaction of one unit's rows (row_bytes each): row i <- row
// kept[i] for i < n.  A plain gather through a temporary copy.
void ora_compact(uint8_t* rows, int64_t row_bytes, const int32_t* kept, int n) {
  std::vector<uint8_t> tmp(static_cast<size_t>(n) * row_bytes);
  for (int i = 0; i < n; ++i)
    std::memcpy(tmp.data() + static_cast<size_t>(i) * row_bytes,
                rows + static_cast<size_t>(kept[i]) * row_bytes, row_bytes);
  std::memcpy(rows, tmp.data(), tmp.size());
}

}  // extern "C"
