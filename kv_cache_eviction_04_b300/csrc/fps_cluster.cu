// Continual FPS buffer for capacities of 257..512 items: the same steps as
// fps.cu (append, compress when full, beacon selection), with the n x n
// Gram matrix spread over a thread-block cluster.
//
// BeaconKV pages: wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫FPS
// 的采样算法" -- seed = the query with the lowest mean similarity to the others;
// then repeatedly the query farthest from the chosen set; similarity on
// pre-RoPE queries; a bounded per-head buffer compressed when full.
//
// A 512 x 512 fp32 Gram (1 MB) does not fit one SM's tensor memory (256 KB),
// so a unit runs on a cluster of R = ceil(C / 128) CTAs: CTA r owns items
// [128 r, 128 r + 128) and keeps their Gram rows (128 TMEM lanes x up to 512
// columns).  Every CTA streams all of the buffer (64-column chunks, two
// 256-row TMA boxes each) and issues its own MMAs; every CTA also forms the
// exact squared norms of all items from the staged chunks.  The seed and each
// greedy step reduce per CTA (top-2 of its items) and then across the
// cluster: each CTA posts its result in its own shared memory, the cluster
// meets at a hardware barrier, and every CTA merges all posts in rank order,
// so all CTAs take the same decision.  Near-ties are re-decided as in
// fps.cu (exact products, error-free sums), each CTA for its own contenders,
// and merged the same way.  Rank 0 does the append, the survivor compaction
// and the outputs.
#include "common.cuh"
#include "fps_common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

using namespace fps;

constexpr int kCT = 256;  // threads per CTA; threads 0..127 own the CTA's items
constexpr int kCW = kCT / 32;
constexpr int kCStages = 3;
constexpr int kMaxItems = 512;
constexpr int kMaxSelC = 64;
constexpr int kMaxPairsC = 256;
constexpr uint32_t kChunkBytes = kMaxItems * 128;  // 64 columns of 512 rows

struct __align__(16) ClShared {
  uint64_t full[kCStages];
  uint64_t empty[kCStages];
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t winner;
  int32_t npairs;
  double rn64[kMaxItems];  // fp64 1/||x_j|| from the exact squared norm
  double n2_64[kMaxItems];
  float rh[kMaxItems], rl[kMaxItems];  // 1/||x_j|| as a float pair
  float inv[kMaxItems];                // fp32 1/||x_j||
  int32_t sel[kMaxSelC];
  int32_t surv[kMaxSelC];
  int32_t wcount[kCW];
  int32_t cont[128];  // this CTA's contenders, ascending
  double cont_val[128];
  double pair64[kMaxPairsC];
  int16_t pair_a[kMaxPairsC], pair_s[kMaxPairsC];
  uint4 red4[2][kCW];  // per-warp {key, item, runner-up key, -} of a CTA top-2
  // posts read by the other CTAs of the cluster, double-buffered by the
  // parity of the exchange count
  uint4 mbk[2];  // this CTA's {key, item, runner-up key, -}
  double mb_cv[2];
  int32_t mb_ci[2];
};

// Top-2 of the CTA as keys (one barrier; alternating buffers, as in
// fps.cu).  v is this thread's value; its item is i = base + threadIdx.x.
__device__ uint4 cta_top2(float v, int i, ClShared* sh, int par) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const KeyTop2 w = warp_key_top2(fkey(v), i - lane);
  if (lane == 0) sh->red4[par][warp] = make_uint4(w.k1, static_cast<uint32_t>(w.i1), w.k2, 0u);
  __syncthreads();
  return merge_key_top2(lane < kCW ? sh->red4[par][lane]
                                   : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0u));
}

// Cluster-wide top-2: post the CTA's, meet, and lane q of every warp reads
// CTA q's post; the merge does not depend on the order.
__device__ Top2 cluster_top2(uint4 local, ClShared* sh, int par, int R) {
  if (threadIdx.x == 0) sh->mbk[par] = local;
  cluster_sync();
  const int lane = threadIdx.x & 31;
  const uint4 r = merge_key_top2(lane < R ? ld_cluster_u32x4(cluster_map(&sh->mbk[par], lane))
                                          : make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0u));
  return Top2{fkey_value(r.x), static_cast<int>(r.y), fkey_value(r.z)};
}

// Cluster-wide best contender: the largest value (or smallest, `maximize`
// false), ties to the lowest item; idx < 0 marks "no contender".
__device__ int cluster_best(double v, int idx, bool maximize, ClShared* sh, int par, int R) {
  if (threadIdx.x == 0) {
    sh->mb_cv[par] = v;
    sh->mb_ci[par] = idx;
  }
  cluster_sync();
  int best = -1;
  double bv = 0.0;
  for (int q = 0; q < R; ++q) {
    const int qi = ld_cluster_s32(cluster_map(&sh->mb_ci[par], q));
    if (qi < 0) continue;
    const double qv = ld_cluster_f64(cluster_map(&sh->mb_cv[par], q));
    const bool better = best < 0 || (maximize ? qv > bv : qv < bv) || (qv == bv && qi < best);
    if (better) {
      best = qi;
      bv = qv;
    }
  }
  return best;
}

// Ordered list of this CTA's flagged items (thread t < 128 = item base + t).
__device__ int collect_own(bool flag, int base, ClShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t b = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) sh->wcount[warp] = __popc(b);
  __syncthreads();
  int off = 0, total = 0;
  for (int w = 0; w < kCW; ++w) {
    const int c = sh->wcount[w];
    off += w < warp ? c : 0;
    total += c;
  }
  if (flag) sh->cont[off + __popc(b & ((1u << lane) - 1u))] = base + threadIdx.x;
  __syncthreads();
  return total;
}

// FPS of m out of the first n rows of unit u's buffer, cluster-wide; every
// CTA returns the same selection in sh->sel.  `xc` counts exchanges (their
// parity picks the post buffer) and must advance identically in all CTAs.
__device__ int fps_select_cl(const FpsParams& p, const CUtensorMap* bmap, ClShared* sh,
                             uint8_t* stages, int u, int n, int m, int rank, int R, int& xc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (m <= 0) return 0;
  if (n <= m || p.first_m) {  // every item, or the first m (in slot order)
    const int got = min(n, m);
    for (int i = tid; i < got; i += kCT) sh->sel[i] = i;
    __syncthreads();
    return got;
  }
  const int D = p.D;
  const float tauc = tau_cos(D), taum = tau_mean(D);
  const uint16_t* X = p.buf + static_cast<size_t>(u) * p.C * D;
  const int N = (n + 15) & ~15;
  const int N1 = min(N, 256), N2 = N - N1;  // column blocks: items 0..255, 256..N-1
  const int nchunks = D / 64;
  const int base = 128 * rank;              // this CTA's first item
  const int i = base + tid;                 // this thread's item (tid < 128)
  const bool owner = tid < 128;

  if (warp == 0) tmem_alloc(&sh->tmem_base, 512);
  if (tid == 0) sh->npairs = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sh->tmem_base;

  // ---- Gram rows of this CTA's items against all items; exact norms of all
  // items (thread t: items t and t + 256) from the staged chunks
  // squared norms of items t and t + 256: four partial sums each
  // (independent chains; sum e takes pieces e and e + 4 of every chunk),
  // merged in order at the end; sums 2h and 2h + 1 ride in halves 0 and 1
  // of n2p2[half][h] (packed f32x2 arithmetic, the same bits)
  FF2 n2p2[2][2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int e = 0; e < 2; ++e) n2p2[hh][e] = FF2{0ull, 0ull};
  const uint32_t id1 = idesc_bf16_f32(128, static_cast<uint32_t>(N1));
  const uint32_t id2 = idesc_bf16_f32(128, static_cast<uint32_t>(N2 > 0 ? N2 : 16));
  auto load_chunk = [&](int c, int st) {
    mbar_arrive_expect_tx(&sh->full[st], kChunkBytes);
    tma_load_3d(stages + st * kChunkBytes, bmap, &sh->full[st], 64 * c, 0, u);
    tma_load_3d(stages + st * kChunkBytes + 256 * 128, bmap, &sh->full[st], 64 * c, 256, u);
  };
  if (tid == 0) {
    fence_proxy_async();  // rank 0's append (before the cluster barrier) -> these TMA reads
    for (int c = 0; c < min(kCStages, nchunks); ++c) load_chunk(c, c);
  }
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kCStages;
    ok = __all_sync(0xffffffffu, ok && wait_bar(&sh->full[st], (c / kCStages) & 1));
    if (!ok) break;
    const uint8_t* sb = stages + st * kChunkBytes;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t sbase = smem_u32(sb);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sdesc_sw128(sbase + base * 128 + kk * 32);
        mma_bf16(tbase, ad, sdesc_sw128(sbase + kk * 32), id1, (c | kk) != 0);
        if (N2 > 0)
          mma_bf16(tbase + 256, ad, sdesc_sw128(sbase + 256 * 128 + kk * 32), id2, (c | kk) != 0);
      }
      mma_commit(&sh->empty[st]);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int j = tid + 256 * half;
      if (j < n) {
        const uint8_t* row = sb + j * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // pieces 2q and 2q + 1 -> sums (2q, 2q + 1) mod 4
          const uint4 v0 = *reinterpret_cast<const uint4*>(row + (((2 * q) ^ (j & 7)) << 4));
          const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((2 * q + 1) ^ (j & 7)) << 4));
          ff2_add_squares(n2p2[half][q & 1], v0, v1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh->empty[st]);
    if (tid == 0 && c + kCStages < nchunks) {
      if (!wait_bar(&sh->empty[st], (c / kCStages) & 1))
        ok = false;
      else
        load_chunk(c + kCStages, st);
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
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int j = tid + 256 * half;
    FF n2p[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      f2_unpack(n2p2[half][h].hi, n2p[2 * h].hi, n2p[2 * h + 1].hi);
      f2_unpack(n2p2[half][h].lo, n2p[2 * h].lo, n2p[2 * h + 1].lo);
    }
    const FF n2 = ff_merge(ff_merge(n2p[0], n2p[1]), ff_merge(n2p[2], n2p[3]));
    const FF r = j < n ? ff_rsqrt(n2) : FF{0.f, 0.f};
    sh->rn64[j] = ff_value(r);
    sh->n2_64[j] = j < n ? ff_value(n2) : 0.0;
    sh->rh[j] = r.hi;
    sh->rl[j] = r.lo;
    sh->inv[j] = r.hi;
  }
  __syncthreads();
  const uint32_t trow = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const bool live_item = owner && i < n;
  const float inv_i = live_item ? sh->inv[i] : 0.f;
  int tb = 0;

  // ---- seed: lowest mean cosine to the other items (error-free fp32 sum)
  float mean = INFINITY;
  if (owner) {
    FF acc{0.f, 0.f};
    for (int c = 0; c < N / 32 + ((N & 31) != 0); ++c) {
      const int col = c * 32;
      uint32_t v[32];
      tmem_ld32(trow + col, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = col + k;
        if (j < n && j != i) ff_add(acc, __uint_as_float(v[k]) * sh->inv[j]);
      }
    }
    if (live_item) mean = (acc.hi + acc.lo) * inv_i / static_cast<float>(n - 1);
  }
  Top2 t = cluster_top2(cta_top2(mean, i, sh, tb++ & 1), sh, xc++ & 1, R);
  int seed = t.i1;
  if (!(t.v2 - t.v1 > 2.f * taum)) {
    // near-tie: as in fps.cu, sum_j cos(a, j) = r_a (x_a . T), T = sum_j r_j x_j
    const int nc = collect_own(live_item && mean <= t.v1 + 2.f * taum, base, sh);
    const int noct = D / 8;
    const int ngrp = max(1, kCT / noct);
    const int per = (n + ngrp - 1) / ngrp;
    FF* Tp = reinterpret_cast<FF*>(stages);
    FF* T = Tp + static_cast<size_t>(ngrp) * D;
    for (int w = tid; w < ngrp * noct; w += kCT) {
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
    for (int k = tid; k < D; k += kCT) {
      FF tk = Tp[k];
      for (int g = 1; g < ngrp; ++g) tk = ff_merge(tk, Tp[static_cast<size_t>(g) * D + k]);
      T[k] = tk;
    }
    __syncthreads();
    for (int c = warp; c < nc; c += kCW) {
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
    int lb = -1;
    double lv = 0.0;
    for (int c = 0; c < nc; ++c)  // ascending index: strict < keeps the lowest
      if (lb < 0 || sh->cont_val[c] < lv) {
        lb = sh->cont[c];
        lv = sh->cont_val[c];
      }
    seed = cluster_best(lv, lb, false, sh, xc++ & 1, R);
  }

  // ---- greedy farthest-point steps (decisions merged across the cluster)
  if (tid == 0) sh->sel[0] = seed;
  bool chosen = (i == seed);
  float dist = INFINITY;
  auto gram = [&](int k) {  // fp32 cosine of this thread's item to item k
    float gk = 0.f;
    if (owner) {
      uint32_t v;
      tmem_ld1(trow + k, v);
      tmem_wait_ld();
      gk = __uint_as_float(v);
    }
    return gk * inv_i * sh->inv[k];
  };
  dist = fminf(dist, 1.f - gram(seed));
  for (int k = 1; k < m; ++k) {
    const bool live = live_item && !chosen;
    const Top2 r =
        cluster_top2(cta_top2(live ? -dist : INFINITY, i, sh, tb++ & 1), sh, xc++ & 1, R);
    int win = r.i1;
    if (!(r.v2 - r.v1 > 2.f * tauc)) {
      const bool cont = live && -dist <= r.v1 + 2.f * tauc;
      const int nc = collect_own(cont, base, sh);
      for (int s2 = 0; s2 < k; ++s2) {  // near-minimum pairs only (see fps.cu)
        const float dv = 1.f - gram(sh->sel[s2]);
        if (cont && dv <= dist + 2.f * tauc) {
          const int slot = atomicAdd(&sh->npairs, 1);
          if (slot < kMaxPairsC) {
            sh->pair_a[slot] = static_cast<int16_t>(i);
            sh->pair_s[slot] = static_cast<int16_t>(sh->sel[s2]);
          }
        }
      }
      __syncthreads();
      const int np = sh->npairs;
      if (np <= kMaxPairsC) {
        for (int pr = warp; pr < np; pr += kCW) {
          const int a = sh->pair_a[pr], b = sh->pair_s[pr];
          const double cv = (warp_dot_rows(X, D, a, b) * sh->rn64[a]) * sh->rn64[b];
          if (lane == 0) sh->pair64[pr] = 1.0 - cv;
        }
        __syncthreads();
        for (int c = tid; c < nc; c += kCT) {
          const int a = sh->cont[c];
          double dmin = INFINITY;
          for (int pr = 0; pr < np; ++pr)
            if (sh->pair_a[pr] == a) dmin = fmin(dmin, sh->pair64[pr]);
          sh->cont_val[c] = dmin;
        }
      } else {
        for (int c = warp; c < nc; c += kCW) {
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
      if (tid == 0) sh->npairs = 0;
      int lb = -1;
      double lv = 0.0;
      for (int c = 0; c < nc; ++c)  // ascending index: strict > keeps the lowest
        if (lb < 0 || sh->cont_val[c] > lv) {
          lb = sh->cont[c];
          lv = sh->cont_val[c];
        }
      win = cluster_best(lv, lb, true, sh, xc++ & 1, R);
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

__global__ void __launch_bounds__(kCT, 1)
    fps_cluster_kernel(const __grid_constant__ FpsParams p,
                       const __grid_constant__ CUtensorMap bmap) {
  pdl_trigger();  // scoring may set up on free SMs; it waits for this grid before reading it
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  ClShared* sh = reinterpret_cast<ClShared*>(stages + kCStages * kChunkBytes);
  const int R = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int u = blockIdx.x / R, tid = threadIdx.x;
  const int D = p.D;
  uint16_t* buf = p.buf + static_cast<size_t>(u) * p.C * D;
  int xc = 0;

  if (tid == 0) {
    for (int s = 0; s < kCStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], kCW + 1);  // every warp read it + the MMAs ran
    }
    mbar_init(&sh->done, 1);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  int c = p.cnt[u];  // every CTA reads cnt before rank 0 rewrites it (at the end)
  const bool ok_state = c >= 0 && c < p.C;
  if (!ok_state) {
    if (tid == 0 && rank == 0) record_error(p.ws, BKV_EDEVICE, kSiteFpsState);
    c = 0;
  }
  // ---- 1. append (rank 0)
  if (p.q_new != nullptr && ok_state) {
    if (rank == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q_new + static_cast<size_t>(u) * D);
      uint4* ring = p.W > 0 ? reinterpret_cast<uint4*>(
                                  p.recent_q + (static_cast<size_t>(u) * p.W +
                                                static_cast<size_t>(p.step % p.W)) * D)
                            : nullptr;
      uint4* dst = reinterpret_cast<uint4*>(buf + static_cast<size_t>(c) * D);
      for (int k = tid; k < D / 8; k += kCT) {
        const uint4 v = src[k];
        if (ring != nullptr) ring[k] = v;
        dst[k] = v;
      }
      fence_proxy_async();
    }
    c += 1;
  }
  cluster_sync();  // the appended row is visible to every CTA's reads

  // ---- 2. compress a full buffer to its FPS survivors, in slot order
  if (ok_state && c == p.C) {
    const int got = fps_select_cl(p, &bmap, sh, stages, u, c, p.M, rank, R, xc);
    cluster_sync();  // every CTA is done reading the buffer
    if (rank == 0) {
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
      const int row_vec = D / 8;
      const int batch = max(1, static_cast<int>((kCStages * kChunkBytes) / (D * 2)));
      uint4* tmp = reinterpret_cast<uint4*>(stages);
      for (int k0 = 0; k0 < got; k0 += batch) {
        const int k1 = min(got, k0 + batch);
        for (int e = tid; e < (k1 - k0) * row_vec; e += kCT) {
          const int k = k0 + e / row_vec, v = e % row_vec;
          tmp[e] = reinterpret_cast<const uint4*>(buf + static_cast<size_t>(sh->surv[k]) * D)[v];
        }
        __syncthreads();
        for (int e = tid; e < (k1 - k0) * row_vec; e += kCT) {
          const int k = k0 + e / row_vec, v = e % row_vec;
          reinterpret_cast<uint4*>(buf + static_cast<size_t>(k) * D)[v] = tmp[e];
        }
        __syncthreads();
      }
      fence_proxy_async();
    }
    c = got;
    cluster_sync();  // the compacted buffer is visible to every CTA
  }

  // ---- 3. beacons: FPS over the current buffer (read-only)
  if (p.want_beacons) {
    const int got = ok_state ? fps_select_cl(p, &bmap, sh, stages, u, c, p.M, rank, R, xc) : 0;
    __syncthreads();
    if (rank == 0) {
      if (p.beacon_idx != nullptr)
        for (int k = tid; k < p.M; k += kCT)
          p.beacon_idx[static_cast<size_t>(u) * p.M + k] = k < got ? sh->sel[k] : -1;
      if (p.beacons != nullptr) {
        const int row_vec = D / 8;
        for (int e = tid; e < got * row_vec; e += kCT) {
          const int k = e / row_vec, v = e % row_vec;
          reinterpret_cast<uint4*>(p.beacons + (static_cast<size_t>(u) * p.M + k) * D)[v] =
              reinterpret_cast<const uint4*>(buf + static_cast<size_t>(sh->sel[k]) * D)[v];
        }
      }
      if (p.n_beacons != nullptr && tid == 0) p.n_beacons[u] = got;
    }
  }
  if (tid == 0 && rank == 0 && ok_state) p.cnt[u] = c;
  cluster_sync();  // no CTA leaves while another may still read its posts
}

}  // namespace

size_t fps_cluster_smem_bytes() {
  return 1024 + static_cast<size_t>(kCStages) * kChunkBytes + sizeof(ClShared);
}

cudaError_t launch_fps_cluster(const FpsParams& p, const CUtensorMap& bufmap, cudaStream_t st) {
  const size_t smem = fps_cluster_smem_bytes();
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fps_cluster_kernel), smem);
  if (e != cudaSuccess) return e;
  const int R = (p.C + 127) / 128;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.U * R));
  cfg.blockDim = dim3(kCT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(R);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fps_cluster_kernel, p, bufmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace bkv
