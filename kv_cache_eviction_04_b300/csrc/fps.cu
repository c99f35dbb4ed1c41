// Continual farthest-point-sampling beacon buffer: per-step append, FPS
// compress when the buffer is full, and FPS beacon selection at eviction.
//
// BeaconKV pages: wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫FPS
// 的采样算法" -- seed = the query with the lowest mean similarity to the others;
// then repeatedly the query farthest from (least similar to) the chosen set;
// similarity on pre-RoPE queries; each head keeps a bounded buffer that is
// FPS-compressed to a smaller size whenever it fills up.
//
// One CTA (256 threads) per unit.  For a buffer of n items (each the G*d
// pre-RoPE vector of one decode step):
//   1. Gram matrix G = X X^T on the tensor core: TMA streams 64-column
//      slices of X (128-byte swizzle) into shared memory and one thread
//      issues tcgen05 MMAs; rows 0..127 and 128..255 land in TMEM columns
//      [0, 256) and [256, 512) with fp32 accumulation.  The Gram stays in
//      TMEM for the whole selection.
//      While a chunk is staged, thread i also accumulates the exact squared
//      norm of item i from it (exact bf16 products, TwoSum sums).
//   2. Thread i owns item i (its TMEM lane): its mean cosine to the others
//      from its TMEM row (error-free sum) -> seed = argmin.
//   3. Greedy: each step reads the new pick's Gram column (one TMEM column:
//      every thread gets its own item's entry), updates its min distance
//      1 - cos in a register and a block argmax (warp shuffles, then shared
//      memory) picks the next item.
//   4. Exactness guard: an fp32 decision is final only when the winner leads
//      the runner-up by more than twice a bound on the fp32 error; otherwise
//      every contender within that band is re-evaluated from the bf16 inputs
//      with exact products and error-free (TwoSum) sums, ~2^-44 accurate,
//      and those values decide (ties: lowest index).  The indices then equal
//      those of an fp64 evaluation except where two candidates' exact values
//      differ by less than ~1e-12; identical items tie exactly.
#include "common.cuh"
#include "fps_common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

using namespace fps;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 6;  // Gram chunk stages (8 chunks at D = 512: two refills)
constexpr int kMaxSel = 64;
constexpr int kMaxPairs = 256;   // near-minimum (contender, chosen) pairs per greedy recheck

struct __align__(16) FpsShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t n_sel;
  int32_t winner;
  int32_t npairs;
  float inv[256];         // fp32 1/||x_i|| (from the exact norm)
  int32_t sel[kMaxSel];
  int32_t surv[kMaxSel];
  int32_t wcount[kWarps];
  int32_t cont[256];      // contenders of a recheck, ascending item index
  double cont_val[256];
  double rn64[256];       // fp64 1/||x_i|| from the exact squared norm
  double n2_64[256];      // exact squared norm ||x_i||^2
  float rh[256], rl[256];  // 1/||x_i|| as an unevaluated float pair
  double pair64[kMaxPairs];
  int16_t pair_a[kMaxPairs];  // item of a pair's contender
  int16_t pair_s[kMaxPairs];  // its chosen item
  float red_v1[2][kWarps];
  float red_v2[2][kWarps];
  int32_t red_i1[2][kWarps];
};

// Block-wide Top2 (all threads call; result valid in every thread).  One
// barrier: consecutive calls alternate between two reduction buffers
// (`par` = call count & 1), so a call never overwrites what a thread of the
// previous call may still read.
__device__ Top2 block_top2(Top2 t, FpsShared* sh, int par) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 o2;
    o2.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
    o2.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    o2.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
    t = top2_merge(t, o2);
  }
  if (lane == 0) {
    sh->red_v1[par][warp] = t.v1;
    sh->red_i1[par][warp] = t.i1;
    sh->red_v2[par][warp] = t.v2;
  }
  __syncthreads();
  Top2 r{sh->red_v1[par][0], sh->red_i1[par][0], sh->red_v2[par][0]};
  for (int w = 1; w < kWarps; ++w)
    r = top2_merge(r, Top2{sh->red_v1[par][w], sh->red_i1[par][w], sh->red_v2[par][w]});
  return r;
}

// Ordered list of the items whose flag is set (thread i = item i): writes
// them to sh->cont in ascending index order and returns how many there are.
// Every thread calls; no cap, so a recheck always sees every contender.
__device__ int collect_contenders(bool flag, FpsShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t b = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) sh->wcount[warp] = __popc(b);
  __syncthreads();
  int off = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    const int c = sh->wcount[w];
    off += w < warp ? c : 0;
    total += c;
  }
  if (flag) sh->cont[off + __popc(b & ((1u << lane) - 1u))] = threadIdx.x;
  __syncthreads();
  return total;
}

// FPS of m items out of the first n rows of unit u's buffer.  Writes the
// selection order to sh->sel and returns its length.  A CTA runs at most one
// non-trivial selection per launch (after a compress the buffer holds M
// items and the beacon pass takes all of them), so the mbarriers start from
// phase 0 here.
__device__ int fps_select(const FpsParams& p, const CUtensorMap* bmap, FpsShared* sh,
                          uint8_t* stages, int stage_rows, int u, int n, int m) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (m <= 0) return 0;
  if (n <= m) {
    for (int i = tid; i < n; i += kThreads) sh->sel[i] = i;
    __syncthreads();
    return n;
  }
  const int D = p.D;
  const uint16_t* X = p.buf + static_cast<size_t>(u) * p.C * D;
  const int N = (n + 15) & ~15;
  const int nbands = (n + 127) / 128;
  const int nchunks = D / 64;
  const uint32_t stage_bytes = static_cast<uint32_t>(stage_rows) * 128;
  const uint32_t box_bytes = static_cast<uint32_t>(min(stage_rows, (p.C + 15) & ~15)) * 128;

  if (warp == 0) tmem_alloc(&sh->tmem_base, 512);  // no relinquish: a CTA may select twice
  if (tid == 0) sh->npairs = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sh->tmem_base;
  const int i = tid;  // this thread's item

  // ---- Gram on the tensor core (thread 0 issues TMA and MMA).  Meanwhile
  // every thread accumulates the exact squared norm of its own item from
  // the staged 64-column chunks (rows of 128 bytes, whose 16-byte pieces are
  // swizzled by row & 7).  A stage is refilled once the MMAs and all eight
  // warps are done with it.
  FF n2{0.f, 0.f};
  const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(N));
  if (tid == 0)
    for (int c = 0; c < min(kStages, nchunks); ++c) {
      mbar_arrive_expect_tx(&sh->full[c], box_bytes);
      tma_load_3d(stages + c * stage_bytes, bmap, &sh->full[c], 64 * c, 0, u);
    }
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kStages;
    ok = __all_sync(0xffffffffu, ok && wait_bar(&sh->full[st], (c / kStages) & 1));
    if (!ok) break;
    const uint8_t* sb = stages + st * stage_bytes;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t sbase = smem_u32(sb);
      for (int h = 0; h < nbands; ++h)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16(tbase + h * 256, sdesc_sw128(sbase + h * 16384 + kk * 32),
                   sdesc_sw128(sbase + kk * 32), idesc, (c | kk) != 0);
      mma_commit(&sh->empty[st]);
    }
    if (i < n) {
      const uint8_t* row = sb + i * 128;
#pragma unroll
      for (int lc = 0; lc < 8; ++lc) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((lc ^ (i & 7)) << 4));
        ff_add_products(n2, v, v);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->empty[st]);
    if (tid == 0 && c + kStages < nchunks) {
      if (!wait_bar(&sh->empty[st], (c / kStages) & 1)) {
        ok = false;
      } else {
        mbar_arrive_expect_tx(&sh->full[st], box_bytes);
        tma_load_3d(stages + st * stage_bytes, bmap, &sh->full[st], 64 * (c + kStages), 0, u);
      }
    }
  }
  if (tid == 0) mma_commit(&sh->done);
  if (!ok) {
    sh->abort_flag = 1;
    if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteFpsWait);
  }
  __syncthreads();
  warp_wait(&sh->done, 0, &sh->abort_flag);
  tc_fence_after();
  __syncthreads();
  const bool gram_ok = sh->abort_flag == 0;  // block-uniform

  // item of this thread: band h = warp / 4, TMEM lane quarter = warp % 4
  const int h = warp >> 2, q = warp & 3;
  const bool band_live = h < nbands;
  const uint32_t trow = tbase + (static_cast<uint32_t>(q * 32) << 16) + h * 256;
  {
    const double nn = i < n ? ff_value(n2) : 0.0;
    const double r = nn > 0.0 ? 1.0 / sqrt(nn) : 0.0;
    sh->rn64[i] = r;
    sh->n2_64[i] = nn;
    const float rhi = static_cast<float>(r);
    sh->rh[i] = rhi;
    sh->rl[i] = static_cast<float>(r - static_cast<double>(rhi));
    sh->inv[i] = static_cast<float>(r);
  }
  __syncthreads();
  const float inv_i = sh->inv[i];
  int tb = 0;  // block_top2 calls so far

  // ---- seed: lowest mean cosine to the other items (error-free sum of the
  // fp32 cosines, so the mean's error is that of one cosine)
  float mean = INFINITY;
  if (band_live) {
    FF acc{0.f, 0.f};
    for (int c = 0; c < (N + 31) / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(trow + c * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = c * 32 + k;  // columns past n were never written: skip them
        if (j < n && j != i) ff_add(acc, __uint_as_float(v[k]) * sh->inv[j]);
      }
    }
    if (i < n) mean = (acc.hi + acc.lo) * inv_i / static_cast<float>(n - 1);
  }
  Top2 t = block_top2(Top2{mean, i, INFINITY}, sh, tb++ & 1);
  int seed = t.i1;
  if (!(t.v2 - t.v1 > 2.f * kTauMean) && gram_ok) {
    // Near-tie: re-decide among the contenders with exact-product sums.
    // sum_j cos(a, j) = r_a * (x_a . T) with T = sum_j r_j x_j, so T is built
    // once (slot order, float-float, exact bf16 x fp32 products by TwoProd)
    // and each contender needs one dot product with it; the item's own term
    // (n2_a r_a) r_a is then removed.  Two identical items get bit-identical
    // values, so the lowest slot wins an exact tie.
    const int nc = collect_contenders(i < n && mean <= t.v1 + 2.f * kTauMean, sh);
    // T in two steps, in a fixed order: thread (group g, octet o) sums items
    // [g * per, (g + 1) * per) over columns 8o .. 8o + 7 (16-byte loads, many
    // in flight), then the groups' partial sums are merged in group order.
    const int noct = D / 8;
    const int ngrp = max(1, kThreads / noct);
    const int per = (n + ngrp - 1) / ngrp;
    FF* Tp = reinterpret_cast<FF*>(stages);  // [ngrp][D] partials (the Gram's stages are free)
    FF* T = Tp + static_cast<size_t>(ngrp) * D;
    for (int w = tid; w < ngrp * noct; w += kThreads) {
      const int g = w / noct, o = w % noct;
      FF acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = FF{0.f, 0.f};
      const int j0 = g * per, j1 = min(n, j0 + per);
      const uint4* col = reinterpret_cast<const uint4*>(X) + o;
#pragma unroll 8
      for (int j = j0; j < j1; ++j) {
        const uint4 v = col[static_cast<size_t>(j) * noct];
        const float rh = sh->rh[j], rl = sh->rl[j];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          ff_add_scaled(acc[2 * hh], __uint_as_float(wv[hh] << 16), rh, rl);
          ff_add_scaled(acc[2 * hh + 1], __uint_as_float(wv[hh] & 0xFFFF0000u), rh, rl);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) Tp[static_cast<size_t>(g) * D + 8 * o + e] = acc[e];
    }
    __syncthreads();
    for (int k = tid; k < D; k += kThreads) {
      FF tk = Tp[k];
      for (int g = 1; g < ngrp; ++g) tk = ff_merge(tk, Tp[static_cast<size_t>(g) * D + k]);
      T[k] = tk;
    }
    __syncthreads();
    for (int c = warp; c < nc; c += kWarps) {
      const int a = sh->cont[c];
      const uint32_t* xa = reinterpret_cast<const uint32_t*>(X + static_cast<size_t>(a) * D);
      FF acc{0.f, 0.f};
      for (int k2 = 2 * lane; k2 < D; k2 += 64) {
        const uint32_t w = xa[k2 / 2];
        ff_add_scaled(acc, __uint_as_float(w << 16), T[k2].hi, T[k2].lo);
        ff_add_scaled(acc, __uint_as_float(w & 0xFFFF0000u), T[k2 + 1].hi, T[k2 + 1].lo);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        FF other{__shfl_xor_sync(0xffffffffu, acc.hi, o), __shfl_xor_sync(0xffffffffu, acc.lo, o)};
        acc = ff_merge(acc, other);
      }
      if (lane == 0) {
        const double ra = sh->rn64[a];
        const double self = (sh->n2_64[a] * ra) * ra;
        sh->cont_val[c] = (ff_value(acc) * ra - self) / static_cast<double>(n - 1);
      }
    }
    __syncthreads();
    if (tid == 0) {
      int best = -1;
      double bv = 0.0;
      for (int c = 0; c < nc; ++c) {  // ascending index: strict < keeps the lowest
        const double v = sh->cont_val[c];
        if (best < 0 || v < bv) {
          best = sh->cont[c];
          bv = v;
        }
      }
      sh->winner = best;
    }
    __syncthreads();
    seed = sh->winner;
  }

  // ---- greedy farthest-point steps
  if (tid == 0) sh->sel[0] = seed;
  bool chosen = (i == seed);
  // 1 - cos lies in [0, 2]: start above it so the seed's column sets it
  float dist = INFINITY;
  auto gram = [&](int k) {  // this thread's fp32 cosine to item k (warp-collective)
    float gk = 0.f;
    if (band_live) {
      uint32_t v;
      tmem_ld1(trow + k, v);
      tmem_wait_ld();
      gk = __uint_as_float(v);
    }
    return gk * inv_i * sh->inv[k];
  };
  dist = fminf(dist, 1.f - gram(seed));
  for (int k = 1; k < m; ++k) {
    const bool live = i < n && !chosen;
    Top2 r = block_top2(Top2{live ? -dist : INFINITY, i, INFINITY}, sh, tb++ & 1);
    int win = r.i1;
    if (!(r.v2 - r.v1 > 2.f * kTauCos) && gram_ok) {
      const bool cont = live && -dist <= r.v1 + 2.f * kTauCos;
      const int nc = collect_contenders(cont, sh);
      // A contender's exact distance is the min over the chosen items; only
      // those whose fp32 distance is within 2 tau of its fp32 min can attain
      // it, so only those pairs are re-evaluated.
      for (int s2 = 0; s2 < k; ++s2) {
        const float dv = 1.f - gram(sh->sel[s2]);
        if (cont && dv <= dist + 2.f * kTauCos) {
          const int slot = atomicAdd(&sh->npairs, 1);
          if (slot < kMaxPairs) {
            sh->pair_a[slot] = static_cast<int16_t>(i);
            sh->pair_s[slot] = static_cast<int16_t>(sh->sel[s2]);
          }
        }
      }
      __syncthreads();
      const int np = sh->npairs;
      if (np <= kMaxPairs) {
        for (int pr = warp; pr < np; pr += kWarps) {
          const int a = sh->pair_a[pr], b = sh->pair_s[pr];
          const double cv = (warp_dot_rows(X, D, a, b) * sh->rn64[a]) * sh->rn64[b];
          if (lane == 0) sh->pair64[pr] = 1.0 - cv;
        }
        __syncthreads();
        for (int c = tid; c < nc; c += kThreads) {
          const int a = sh->cont[c];
          double dmin = INFINITY;
          for (int pr = 0; pr < np; ++pr)
            if (sh->pair_a[pr] == a) dmin = fmin(dmin, sh->pair64[pr]);
          sh->cont_val[c] = dmin;
        }
      } else {
        // too many near-minimum pairs: every (contender, chosen) pair
        for (int c = warp; c < nc; c += kWarps) {
          const int a = sh->cont[c];
          double dmin = INFINITY;
          for (int s2 = 0; s2 < k; ++s2) {
            const int b = sh->sel[s2];
            dmin = fmin(dmin, 1.0 - (warp_dot_rows(X, D, a, b) * sh->rn64[a]) * sh->rn64[b]);
          }
          if (lane == 0) sh->cont_val[c] = dmin;
        }
      }
      __syncthreads();
      if (tid == 0) {
        sh->npairs = 0;
        int best = -1;
        double bv = 0.0;
        for (int c = 0; c < nc; ++c) {  // ascending index: strict > keeps the lowest
          const double v = sh->cont_val[c];
          if (best < 0 || v > bv) {
            best = sh->cont[c];
            bv = v;
          }
        }
        sh->winner = best;
      }
      __syncthreads();
      win = sh->winner;
    }
    if (tid == 0) sh->sel[k] = win;
    chosen = chosen || (i == win);
    dist = fminf(dist, 1.f - gram(win));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
  return m;
}

__global__ void __launch_bounds__(kThreads, 1)
    fps_update_kernel(const __grid_constant__ FpsParams p,
                      const __grid_constant__ CUtensorMap bmap, int stage_rows) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // TMA destinations with the 128-byte swizzle need 1024-byte alignment
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  FpsShared* sh = reinterpret_cast<FpsShared*>(stages + kStages * stage_rows * 128);
  const int u = blockIdx.x, tid = threadIdx.x;
  const int D = p.D;
  uint16_t* buf = p.buf + static_cast<size_t>(u) * p.C * D;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], kWarps + 1);  // every warp read it + the MMAs ran
    }
    mbar_init(&sh->done, 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  int c = p.cnt[u];
  const bool ok_state = c >= 0 && c < p.C;
  if (!ok_state) {
    if (tid == 0) record_error(p.ws, BKV_EDEVICE, kSiteFpsState);
    c = 0;
  }
  // ---- 1. append the step's query to the ring and the buffer
  if (p.q_new != nullptr && ok_state) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q_new + static_cast<size_t>(u) * D);
    uint4* ring = p.W > 0 ? reinterpret_cast<uint4*>(
                                p.recent_q + (static_cast<size_t>(u) * p.W +
                                              static_cast<size_t>(p.step % p.W)) * D)
                          : nullptr;
    uint4* dst = reinterpret_cast<uint4*>(buf + static_cast<size_t>(c) * D);
    for (int k = tid; k < D / 8; k += kThreads) {
      const uint4 v = src[k];
      if (ring != nullptr) ring[k] = v;
      dst[k] = v;
    }
    c += 1;
  }
  fence_proxy_async();  // generic writes to the buffer -> later TMA reads
  __syncthreads();

  // ---- 2. compress a full buffer to its FPS survivors, in slot order
  if (ok_state && c == p.C) {
    const int got = fps_select(p, &bmap, sh, stages, stage_rows, u, c, p.M);
    if (tid == 0) {
      for (int k = 0; k < got; ++k) sh->surv[k] = sh->sel[k];
      for (int a = 1; a < got; ++a) {  // insertion sort, got <= 64
        const int v = sh->surv[a];
        int b = a - 1;
        while (b >= 0 && sh->surv[b] > v) {
          sh->surv[b + 1] = sh->surv[b];
          --b;
        }
        sh->surv[b + 1] = v;
      }
    }
    __syncthreads();
    // row k <- row surv[k] (surv ascending, surv[k] >= k): batches read into
    // shared memory first, then written
    const int row_vec = D / 8;  // uint4 per row
    const int batch = max(1, static_cast<int>((kStages * stage_rows * 128) / (D * 2)));
    uint4* tmp = reinterpret_cast<uint4*>(stages);
    for (int k0 = 0; k0 < got; k0 += batch) {
      const int k1 = min(got, k0 + batch);
      for (int e = tid; e < (k1 - k0) * row_vec; e += kThreads) {
        const int k = k0 + e / row_vec, v = e % row_vec;
        tmp[e] = reinterpret_cast<const uint4*>(buf + static_cast<size_t>(sh->surv[k]) * D)[v];
      }
      __syncthreads();
      for (int e = tid; e < (k1 - k0) * row_vec; e += kThreads) {
        const int k = k0 + e / row_vec, v = e % row_vec;
        reinterpret_cast<uint4*>(buf + static_cast<size_t>(k) * D)[v] = tmp[e];
      }
      __syncthreads();
    }
    c = got;
    fence_proxy_async();
    __syncthreads();
  }

  // ---- 3. beacons: FPS over the current buffer (read-only)
  if (p.want_beacons) {
    const int got = ok_state ? fps_select(p, &bmap, sh, stages, stage_rows, u, c, p.M) : 0;
    __syncthreads();
    if (p.beacon_idx != nullptr)
      for (int k = tid; k < p.M; k += kThreads)
        p.beacon_idx[static_cast<size_t>(u) * p.M + k] = k < got ? sh->sel[k] : -1;
    if (p.beacons != nullptr) {
      const int row_vec = D / 8;
      for (int e = tid; e < got * row_vec; e += kThreads) {
        const int k = e / row_vec, v = e % row_vec;
        reinterpret_cast<uint4*>(p.beacons + (static_cast<size_t>(u) * p.M + k) * D)[v] =
            reinterpret_cast<const uint4*>(buf + static_cast<size_t>(sh->sel[k]) * D)[v];
      }
    }
    if (p.n_beacons != nullptr && tid == 0) p.n_beacons[u] = got;
  }
  if (tid == 0 && ok_state) p.cnt[u] = c;
}

}  // namespace

// Stage rows cover every row a 128-row MMA band reads (one band up to C =
// 128, two bands beyond).
int fps_stage_rows(int C) { return C <= 128 ? 128 : 256; }

// At least 120 KB so that one CTA holds an SM (each takes all 512 TMEM columns).
size_t fps_smem_bytes(int C) {
  const size_t need =
      1024 + static_cast<size_t>(kStages) * fps_stage_rows(C) * 128 + sizeof(FpsShared);
  return need < 120 * 1024 ? 120 * 1024 : need;
}

cudaError_t launch_fps(const FpsParams& p, const CUtensorMap& bufmap, cudaStream_t st) {
  const int rows = fps_stage_rows(p.C);
  const size_t smem = fps_smem_bytes(p.C);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fps_update_kernel), smem);
  if (e != cudaSuccess) return e;
  fps_update_kernel<<<p.U, kThreads, smem, st>>>(p, bufmap, rows);
  return cudaGetLastError();
}

}  // namespace bkv
