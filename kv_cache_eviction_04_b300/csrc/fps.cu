// Continual farthest-point-sampling beacon buffer: per-step append, FPS
// compress when the buffer is full, and FPS beacon selection at eviction.
//
// BeaconKV pages: wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫FPS
// 的采样算法" -- seed = the query with the lowest mean similarity to the others;
// then repeatedly the query farthest from (least similar to) the chosen set;
// similarity on pre-RoPE queries; each head keeps a bounded buffer that is
// FPS-compressed to a smaller size whenever it fills up.
//
// One CTA per unit: eight item warps (thread i owns item i) and a producer
// warp.  For a buffer of n items (each the G*d pre-RoPE vector of one
// decode step):
//   1. Gram matrix G = X X^T on the tensor core: TMA streams 64-column
//      slices of X (128-byte swizzle) into shared memory and one thread of
//      the producer warp issues tcgen05 MMAs; rows 0..127 and 128..255 land
//      in TMEM columns [0, 256) and [256, 512) with fp32 accumulation.  The
//      Gram stays in TMEM for the whole selection.
//      While a chunk is staged, thread i also accumulates the exact squared
//      norm of item i from it (exact bf16 products, TwoSum sums, two float
//      pairs per packed f32x2 instruction).
//   2. Thread i owns item i (its TMEM lane): its mean cosine to the others
//      from its TMEM row (pairwise fp32 sum) -> seed = argmin.
//   3. Greedy: each step reads the new pick's Gram column (one TMEM column:
//      every thread gets its own item's entry), updates its min distance
//      1 - cos in a register, and a block argmax (redux.sync on
//      order-preserving keys per warp, then one barrier) picks the next item.
//   4. Exactness guard: an fp32 decision is final only when the winner leads
//      the runner-up by more than twice a bound on the fp32 error; otherwise
//      every contender within that band is re-evaluated from the bf16 inputs
//      with exact products and error-free (TwoSum) sums, ~2^-44 accurate,
//      and those values decide (ties: lowest index).  For the seed an fp32
//      pass with a proven error bound comes first and settles the choice
//      when one contender is certainly the lowest.  The indices then equal
//      those of an fp64 evaluation except where two candidates' exact values
//      differ by less than ~1e-12; identical items tie exactly.
#include "common.cuh"
#include "fps_common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

using namespace fps;

constexpr int kItems = 256;                // item threads: warps 0..7, thread t = item t
constexpr int kItemWarps = kItems / 32;
constexpr int kThreads = kItems + 32;      // + warp 8: TMA and MMA issue for the Gram
constexpr int kStages = 6;  // Gram chunk stages (8 chunks at D = 512: two refills)
constexpr int kMaxSel = 64;
constexpr int kMaxPairs = 256;   // near-minimum (contender, chosen) pairs per greedy recheck

struct __align__(16) FpsShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t done;
  uint64_t seeded;           // the eight item warps are past the seed (its scratch is free)
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t n_sel;
  int32_t winner;
  int32_t npairs;
  int32_t pad_;
  uint4 red[2][kItemWarps];  // per-warp {key, item, runner-up key, -} of a block top-2
  float inv[kItems];         // fp32 1/||x_i|| from the exact squared norm
  float n2h[kItems], n2l[kItems];  // exact squared norm ||x_i||^2 as an unevaluated float pair
  int32_t sel[kMaxSel];
  int32_t surv[kMaxSel];
  int32_t wcount[kItemWarps];
  int32_t cont[kItems];      // contenders of a recheck, ascending item index
  double cont_val[kItems];
  double cont_err[kItems];   // seed filter: error bound of a contender's fp32-pass value
  float2 rr[kItems];         // seed recheck: 1/||x_i|| as an unevaluated float pair
  double pair64[kMaxPairs];
  int16_t pair_a[kMaxPairs];  // item of a pair's contender
  int16_t pair_s[kMaxPairs];  // its chosen item
  int32_t ulist[kItems];      // compress pass: full units of the current batch
  int32_t ucount;
  int32_t preloaded;          // Gram chunks of the next selection already loaded
};

// Barrier of the eight item warps only (the producer warp idles after the
// Gram).
__device__ __forceinline__ void item_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kItems) : "memory"); }

// Top2 over the items (thread t < 256 = item t, every item thread calls)
// under the order "smaller value first, then smaller item"; the result is
// valid in every item thread.  Warps reduce order-preserving keys with
// redux.sync; one barrier; then lane q of every warp takes warp q's entry
// and three more reductions merge the eight: the smallest key, the lowest
// item holding it, and the runner-up (the winner's own second, or another
// warp's best).  Consecutive calls alternate between two buffers (`par` =
// call count & 1), so a call never overwrites what a thread of the previous
// call may still read.
__device__ Top2 block_top2(float v, FpsShared* sh, int par) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const KeyTop2 w = warp_key_top2(fkey(v), warp * 32);
  if (lane == 0) sh->red[par][warp] = make_uint4(w.k1, static_cast<uint32_t>(w.i1), w.k2, 0u);
  item_sync();
  const uint4 r = merge_key_top2(lane < kItemWarps ? sh->red[par][lane]
                                                  : make_uint4(0xffffffffu, 0xffffffffu,
                                                               0xffffffffu, 0u));
  return Top2{fkey_value(r.x), static_cast<int>(r.y), fkey_value(r.z)};
}

// Ordered list of the items whose flag is set (item threads): writes them
// to sh->cont in ascending index order and returns how many there are.
// No cap, so a recheck always sees every contender.
__device__ int collect_contenders(bool flag, FpsShared* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t b = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) sh->wcount[warp] = __popc(b);
  item_sync();
  int off = 0, total = 0;
  for (int w = 0; w < kItemWarps; ++w) {
    const int c = sh->wcount[w];
    off += w < warp ? c : 0;
    total += c;
  }
  if (flag) sh->cont[off + __popc(b & ((1u << lane) - 1u))] = threadIdx.x;
  item_sync();
  return total;
}

// fp64 1/||x_a|| from the exact squared norm (0 for a zero row).
__device__ __forceinline__ double exact_rnorm(const FpsShared* sh, int a) {
  return ff_value(ff_rsqrt(FF{sh->n2h[a], sh->n2l[a]}));
}

// The same, warp-collective, for a selection whose exact squared norms are
// formed on demand (a negative n2h marks one not formed yet): the warp forms
// it from the row in global memory and keeps it.  Two warps that form the
// same norm at once write the same value.
__device__ __forceinline__ double exact_rnorm_w(FpsShared* sh, const uint16_t* X, int D, int a) {
  if (sh->n2h[a] < 0.f) {
    const FF n2 = warp_dot_rows_ff(X, D, a, a);
    if ((threadIdx.x & 31) == 0) {
      sh->n2l[a] = n2.lo;
      sh->n2h[a] = n2.hi;
    }
    return ff_value(ff_rsqrt(n2));
  }
  return exact_rnorm(sh, a);
}

// Exact squared norm of item i's row (one thread), as the Gram phase forms
// it from the staged chunks: eight float pairs, one per 16-byte piece of a
// 64-column chunk, merged in a fixed order.
__device__ __forceinline__ FF row_norm_ff(const uint16_t* X, int D, int i) {
  FF n2p[8];
#pragma unroll
  for (int lc = 0; lc < 8; ++lc) n2p[lc] = FF{0.f, 0.f};
  const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(i) * D);
#pragma unroll 1
  for (int c = 0; c < D / 64; ++c) {
    uint4 v[8];
#pragma unroll
    for (int lc = 0; lc < 8; ++lc) v[lc] = row[c * 8 + lc];
#pragma unroll
    for (int lc = 0; lc < 8; ++lc) ff_add_products(n2p[lc], v[lc], v[lc]);
  }
  return ff_merge(ff_merge(ff_merge(n2p[0], n2p[1]), ff_merge(n2p[2], n2p[3])),
                  ff_merge(ff_merge(n2p[4], n2p[5]), ff_merge(n2p[6], n2p[7])));
}

// Seed and greedy steps over the Gram in TMEM (the eight item warps only;
// thread i owns item i and its TMEM lane).  Writes sh->sel[0, m).
// `stages` is free scratch here (the seed recheck's partial sums).
// With `lazy` the Gram phase formed 1/||x|| from an fp32 pairwise sum of
// the exact squares (relative error <= ~6 u instead of ~1 u from the exact
// norm): both bands widen by 1e-6, and the exact norms are formed only when
// a recheck needs them.
template <bool lazy>
__device__ void fps_pick(const FpsParams& p, FpsShared* sh, uint8_t* stages, uint32_t tbase,
                         bool gram_ok, int u, int n, int m) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = tid;
  const int D = p.D;
  const float widen = lazy ? 1e-6f : 0.f;
  const float tauc = tau_cos(D) + widen, taum = tau_mean(D) + widen;
  const uint16_t* X = p.buf + static_cast<size_t>(u) * p.C * D;
  const int N = (n + 15) & ~15;
  const int nbands = (n + 127) / 128;
  // item of this thread: band h = warp / 4, TMEM lane quarter = warp % 4
  const int h = warp >> 2, q = warp & 3;
  const bool band_live = h < nbands;
  const uint32_t trow = tbase + (static_cast<uint32_t>(q * 32) << 16) + h * 256;
  const float inv_i = sh->inv[i];
  int tb = 0;  // block_top2 calls so far

  // ---- seed: lowest mean cosine to the other items.  The fp32 cosines of a
  // 32-column block are summed pairwise, two blocks are added and the pair
  // sums accumulated in order (at most 9 roundings per term); the loop stays
  // rolled so that its code is fetched once.
  float mean = INFINITY;
  if (band_live) {
    float total = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < N; c0 += 64) {
      uint32_t v[2][32];
      tmem_ld32(trow + c0, v[0]);  // columns up to c0 + 63 < 512: inside the allocation
      tmem_ld32(trow + c0 + 32, v[1]);
      tmem_wait_ld();
      float ps[2];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        float s[32];
#pragma unroll
        for (int k4 = 0; k4 < 32; k4 += 4) {
          const float4 r4 = *reinterpret_cast<const float4*>(&sh->inv[c0 + 32 * b + k4]);
          const float rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = c0 + 32 * b + k4 + e;  // columns past n hold no item: skip them
            s[k4 + e] = (j < n && j != i) ? __uint_as_float(v[b][k4 + e]) * rv[e] : 0.f;
          }
        }
#pragma unroll
        for (int w = 16; w > 0; w >>= 1)
#pragma unroll
          for (int k = 0; k < w; ++k) s[k] += s[k + w];
        ps[b] = s[0];
      }
      total += ps[0] + ps[1];
    }
    if (i < n) mean = total * inv_i / static_cast<float>(n - 1);
  }
  Top2 t = block_top2(mean, sh, tb++ & 1);
  int seed = t.i1;
  if (!(t.v2 - t.v1 > 2.f * taum) && gram_ok) {
    // Near-tie: re-decide among the contenders with exact-product sums.
    // sum_j cos(a, j) = r_a * (x_a . T) with T = sum_j r_j x_j, so T is
    // built once and each contender needs one dot product with it; the
    // item's own term (n2_a r_a) r_a is then removed.  T is formed from the
    // buffer in global memory (it was just streamed, so it sits in L2) in
    // one compact loop: thread t takes the 16-byte column octet t % (D/8)
    // and every (256 / (D/8))-th item from t / (D/8) on, with eight
    // independent float pairs (exact bf16 x fp32 products by TwoProd,
    // TwoSum sums); the groups' partial sums are merged in a fixed order.
    // One warp per contender then forms x_a . T.  Two identical items get
    // bit-identical values, so the lowest slot wins an exact tie.  An fp32
    // pass with a proven error bound comes first and settles the seed on
    // its own when one contender is certainly the lowest; the float-float
    // pass runs only when it is not (as for exact ties).
    const int nc = collect_contenders(i < n && mean <= t.v1 + 2.f * taum, sh);
    if (lazy && i < n) {  // (a template parameter)
      // the exact norms were not formed in the Gram phase: every item's now
      const FF n2 = row_norm_ff(X, D, i);
      sh->n2h[i] = n2.hi;
      sh->n2l[i] = n2.lo;
    }
    {
      const FF r = i < n ? ff_rsqrt(FF{sh->n2h[i], sh->n2l[i]}) : FF{0.f, 0.f};
      sh->rr[i] = make_float2(r.hi, r.lo);
    }
    item_sync();
    const int noct = D / 8;               // 16-byte column octets: 8..256
    const int ngrp = kItems / noct;       // item groups: 1..32
    const uint4* Xv = reinterpret_cast<const uint4*>(X);
    // ---- fp32 filter.  T and A = sum_j |x_j| r_j are first formed in
    // plain fp32 (fma, r_j rounded to its high part), in the same item
    // groups, in blocks of eight items summed into a running total, and the
    // groups merged in order; the sum a term passes through is at most
    // m = 8 + (blocks per group) + (ngrp - 1) roundings deep, so
    // |T32_k - T_k| <= (gamma_m + 2^-23.9) A_k (Higham, Accuracy and
    // Stability of Numerical Algorithms, 2nd ed., 4.2; 2^-23.9 for r_j's
    // low part).  A contender's value S_a = r_a (x_a . T32) - 1 (float-float
    // dot) is then within E_a = 1.01 (gamma_m + 2^-22) r_a (|x_a| . A32)
    // of its exact value (the factor covers 1 / (1 - gamma_m), A32's own
    // rounding and the dot's).  When the lowest value's interval lies below
    // every other contender's, it is the exact minimum, unique; otherwise
    // the exact float-float pass below decides.
    {
      float* T32p = reinterpret_cast<float*>(stages);  // [ngrp][D]
      float* A32p = T32p + static_cast<size_t>(ngrp) * D;
      float* T32 = A32p + static_cast<size_t>(ngrp) * D;  // [D]
      float* A32 = T32 + D;                                // [D]
      if (tid < ngrp * noct) {
        const int g = tid / noct, o = tid - g * noct;
        uint64_t ta[4] = {0ull, 0ull, 0ull, 0ull}, aa[4] = {0ull, 0ull, 0ull, 0ull};
        // the next block's loads are issued before this block is summed
        auto load8 = [&](int j0, uint4 (&v)[8]) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j = j0 + q * ngrp;
            v[q] = j < n ? Xv[static_cast<size_t>(j) * noct + o] : make_uint4(0u, 0u, 0u, 0u);
          }
        };
        uint4 v[8];
        load8(g, v);
#pragma unroll 1
        for (int j0 = g; j0 < n; j0 += 8 * ngrp) {
          uint4 vn[8];
          load8(j0 + 8 * ngrp, vn);
          float rh[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j = j0 + q * ngrp;
            rh[q] = j < n ? sh->rr[j].x : 0.f;
          }
          uint64_t tb[4] = {0ull, 0ull, 0ull, 0ull}, ab[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t wv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
            const uint64_t r2 = f2_pack(rh[q], rh[q]);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              const uint32_t lo = wv[hh] << 16, hi = wv[hh] & 0xFFFF0000u;
              tb[hh] = f2_fma(f2_pack(__uint_as_float(lo), __uint_as_float(hi)), r2, tb[hh]);
              ab[hh] = f2_fma(f2_pack(__uint_as_float(lo & 0x7FFFFFFFu),
                                      __uint_as_float(hi & 0x7FFFFFFFu)),
                              r2, ab[hh]);
            }
          }
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            ta[hh] = f2_add(ta[hh], tb[hh]);
            aa[hh] = f2_add(aa[hh], ab[hh]);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = vn[q];
        }
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const size_t at = static_cast<size_t>(g) * D + 8 * o + 2 * hh;
          f2_unpack(ta[hh], T32p[at], T32p[at + 1]);
          f2_unpack(aa[hh], A32p[at], A32p[at + 1]);
        }
      }
      item_sync();
      for (int k = tid; k < D; k += kItems) {
        float tk = T32p[k], ak = A32p[k];
        for (int gg = 1; gg < ngrp; ++gg) {
          tk += T32p[static_cast<size_t>(gg) * D + k];
          ak += A32p[static_cast<size_t>(gg) * D + k];
        }
        T32[k] = tk;
        A32[k] = ak;
      }
      item_sync();
      const int per = (n + ngrp - 1) / ngrp;
      const double m = 8.0 + (per + 7) / 8 + (ngrp - 1);
      const double gm = m * 0x1p-24 / (1.0 - m * 0x1p-24);
      for (int cc = warp; cc < nc; cc += kItemWarps) {
        const int a = sh->cont[cc];
        const uint32_t* xa = reinterpret_cast<const uint32_t*>(X + static_cast<size_t>(a) * D);
        FF d{0.f, 0.f};
        float bs = 0.f;
        for (int k2 = 2 * lane; k2 < D; k2 += 64) {
          const uint32_t w = xa[k2 / 2];
          const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
          ff_add_scaled(d, x0, T32[k2], 0.f);
          ff_add_scaled(d, x1, T32[k2 + 1], 0.f);
          bs = fmaf(fabsf(x0), A32[k2], bs);
          bs = fmaf(fabsf(x1), A32[k2 + 1], bs);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const FF other{__shfl_xor_sync(0xffffffffu, d.hi, o),
                         __shfl_xor_sync(0xffffffffu, d.lo, o)};
          d = ff_merge(d, other);
          bs += __shfl_xor_sync(0xffffffffu, bs, o);
        }
        if (lane == 0) {
          const float2 ra = sh->rr[a];
          FF v = ff_mul(d, FF{ra.x, ra.y});
          if (ra.x != 0.f) ff_add(v, -1.f);
          sh->cont_val[cc] = ff_value(v);
          sh->cont_err[cc] = 1.01 * (gm + 0x1p-22) * static_cast<double>(ra.x) * bs;
        }
      }
      item_sync();
      if (tid == 0) {
        int best = 0;
        for (int c = 1; c < nc; ++c)
          if (sh->cont_val[c] < sh->cont_val[best]) best = c;
        bool sure = true;
        const double hi_best = sh->cont_val[best] + sh->cont_err[best];
        for (int c = 0; c < nc; ++c)
          if (c != best && !(sh->cont_val[c] - sh->cont_err[c] > hi_best)) sure = false;
        sh->winner = sure ? sh->cont[best] : -1;
      }
      item_sync();
    }
    if (sh->winner < 0) {  // block-uniform (read after the barrier above)
      // ---- exact float-float pass
      FF* Tp = reinterpret_cast<FF*>(stages);           // [ngrp][D] partial sums
      FF* T = Tp + static_cast<size_t>(ngrp) * D;       // [D]
      item_sync();  // every thread has read the winner before it is written again
      if (tid < ngrp * noct) {
        const int g = tid / noct, o = tid - g * noct;
        FF2 acc2[4];  // octet values 2h, 2h + 1 in halves 0, 1 of acc2[h]
#pragma unroll
        for (int e = 0; e < 4; ++e) acc2[e] = FF2{0ull, 0ull};
        const uint4* col = reinterpret_cast<const uint4*>(X) + o;
        // eight items' loads in flight before any is used, and the next
        // eight's issued before this eight's products are summed (the pass
        // waits on L2 otherwise); items past n are zero and add exactly nothing
        auto load8 = [&](int j0, uint4 (&v)[8]) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j = j0 + q * ngrp;
            v[q] = j < n ? col[static_cast<size_t>(j) * noct] : make_uint4(0u, 0u, 0u, 0u);
          }
        };
        uint4 v[8];
        load8(g, v);
#pragma unroll 1
        for (int j0 = g; j0 < n; j0 += 8 * ngrp) {
          uint4 vn[8];
          load8(j0 + 8 * ngrp, vn);
          float2 r[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int j = j0 + q * ngrp;
            r[q] = j < n ? sh->rr[j] : make_float2(0.f, 0.f);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t wv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
            const uint64_t rh2 = f2_pack(r[q].x, r[q].x), rl2 = f2_pack(r[q].y, r[q].y);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh)
              ff2_add_scaled(acc2[hh],
                             f2_pack(__uint_as_float(wv[hh] << 16),
                                     __uint_as_float(wv[hh] & 0xFFFF0000u)),
                             rh2, rl2);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) v[q] = vn[q];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          FF a, b;
          f2_unpack(acc2[e].hi, a.hi, b.hi);
          f2_unpack(acc2[e].lo, a.lo, b.lo);
          Tp[static_cast<size_t>(g) * D + 8 * o + 2 * e] = a;
          Tp[static_cast<size_t>(g) * D + 8 * o + 2 * e + 1] = b;
        }
      }
      item_sync();
      for (int k = tid; k < D; k += kItems) {
        FF tk = Tp[k];
        for (int g = 1; g < ngrp; ++g) tk = ff_merge(tk, Tp[static_cast<size_t>(g) * D + k]);
        T[k] = tk;
      }
      item_sync();
      for (int cc = warp; cc < nc; cc += kItemWarps) {
        const int a = sh->cont[cc];
        const uint32_t* xa = reinterpret_cast<const uint32_t*>(X + static_cast<size_t>(a) * D);
        FF d{0.f, 0.f};
        for (int k2 = 2 * lane; k2 < D; k2 += 64) {
          const uint32_t w = xa[k2 / 2];
          ff_add_scaled(d, __uint_as_float(w << 16), T[k2].hi, T[k2].lo);
          ff_add_scaled(d, __uint_as_float(w & 0xFFFF0000u), T[k2 + 1].hi, T[k2 + 1].lo);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const FF other{__shfl_xor_sync(0xffffffffu, d.hi, o), __shfl_xor_sync(0xffffffffu, d.lo, o)};
          d = ff_merge(d, other);
        }
        if (lane == 0) {
          // sum over j != a of cos(a, j) = r_a (x_a . T) - 1 for a nonzero
          // item (its own term r_a^2 ||x_a||^2 is 1), 0 for a zero one; the
          // common factor 1 / (n - 1) of the mean does not change the order
          const float2 ra = sh->rr[a];
          FF v = ff_mul(d, FF{ra.x, ra.y});
          if (ra.x != 0.f) ff_add(v, -1.f);
          sh->cont_val[cc] = ff_value(v);
        }
      }
      item_sync();
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
      item_sync();
    }
    seed = sh->winner;
    // the staged chunks were overwritten by the partial sums: none is
    // resident any more (the greedy steps read the buffer from global memory)
  }

  // The stages are free from here on (the recheck's scratch is done with):
  // the producer warp may load the next unit's chunks into them.
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh->seeded);

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
    Top2 r = block_top2(live ? -dist : INFINITY, sh, tb++ & 1);
    int win = r.i1;
    if (!(r.v2 - r.v1 > 2.f * tauc) && gram_ok) {
      const bool cont = live && -dist <= r.v1 + 2.f * tauc;
      const int nc = collect_contenders(cont, sh);
      // A contender's exact distance is the min over the chosen items; only
      // those whose fp32 distance is within 2 tau of its fp32 min can attain
      // it, so only those pairs are re-evaluated.
      for (int s2 = 0; s2 < k; ++s2) {
        const float dv = 1.f - gram(sh->sel[s2]);
        if (cont && dv <= dist + 2.f * tauc) {
          const int slot = atomicAdd(&sh->npairs, 1);
          if (slot < kMaxPairs) {
            sh->pair_a[slot] = static_cast<int16_t>(i);
            sh->pair_s[slot] = static_cast<int16_t>(sh->sel[s2]);
          }
        }
      }
      item_sync();
      const int np = sh->npairs;
      if (np <= kMaxPairs) {
        for (int pr = warp; pr < np; pr += kItemWarps) {
          const int a = sh->pair_a[pr], b = sh->pair_s[pr];
          const double cv =
              (warp_dot_rows(X, D, a, b) * exact_rnorm_w(sh, X, D, a)) * exact_rnorm_w(sh, X, D, b);
          if (lane == 0) sh->pair64[pr] = 1.0 - cv;
        }
        item_sync();
        for (int c = tid; c < nc; c += kItems) {
          const int a = sh->cont[c];
          double dmin = INFINITY;
          for (int pr = 0; pr < np; ++pr)
            if (sh->pair_a[pr] == a) dmin = fmin(dmin, sh->pair64[pr]);
          sh->cont_val[c] = dmin;
        }
      } else {
        // too many near-minimum pairs: every (contender, chosen) pair
        for (int c = warp; c < nc; c += kItemWarps) {
          const int a = sh->cont[c];
          const double ra = exact_rnorm_w(sh, X, D, a);
          double dmin = INFINITY;
          for (int s2 = 0; s2 < k; ++s2) {
            const int b = sh->sel[s2];
            dmin = fmin(dmin, 1.0 - (warp_dot_rows(X, D, a, b) * ra) * exact_rnorm_w(sh, X, D, b));
          }
          if (lane == 0) sh->cont_val[c] = dmin;
        }
      }
      item_sync();
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
      item_sync();
      win = sh->winner;
    }
    if (tid == 0) sh->sel[k] = win;
    chosen = chosen || (i == win);
    dist = fminf(dist, 1.f - gram(win));
  }
}

// FPS of m items out of the first n rows of unit u's buffer.  Writes the
// selection order to sh->sel and returns its length (all threads call).  A
// CTA runs at most one non-trivial selection per launch (after a compress
// the buffer holds M items and the beacon pass takes all of them), so the
// mbarriers start from phase 0 here, or the persistent beacon kernel
// initialises them again between units.  sh->preloaded of the unit's first
// Gram chunks are already loaded (or in flight) into their stages.  With
// next_u >= 0 the producer warp loads that unit's first chunks during the
// greedy steps (once the seed's scratch is free), initialising the
// barriers again first, and leaves their count in sh->preloaded.
// `lazy` (a template parameter, so that each kernel carries one copy of the
// selection): see fps_pick.
template <bool lazy>
__device__ __noinline__ int fps_select(const FpsParams& p, const CUtensorMap* bmap, FpsShared* sh,
                          uint8_t* stages, int stage_rows, int u, int n, int m,
                          int next_u) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pre = sh->preloaded;
  if (m <= 0) return 0;
  if (n <= m || p.first_m) {  // every item, or the first m (in slot order)
    const int got = min(n, m);
    for (int i = tid; i < got; i += kThreads) sh->sel[i] = i;
    __syncthreads();
    return got;
  }
  const int D = p.D;
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

  // Chunk c of the buffer goes to stage c % kStages.
  auto load_chunk = [&](int c, int st) {
    mbar_arrive_expect_tx(&sh->full[st], box_bytes);
    tma_load_3d(stages + st * stage_bytes, bmap, &sh->full[st], 64 * c, 0, u);
  };
  if (tid == kItems) sh->preloaded = 0;  // read by every thread above

  // ---- Gram on the tensor core.  One thread of the producer warp streams
  // 64-column chunks of the buffer into the stage ring by TMA and issues the
  // tcgen05 MMAs of every chunk as soon as it lands.  Meanwhile every item
  // thread accumulates the exact squared norm of its own item from the
  // staged chunks.  A stage is refilled once its MMAs have completed and
  // all eight item warps are done with it; the producer refills without
  // waiting while it still has landed chunks to multiply.
  // eight independent partial sums, one per 16-byte piece of a row: pieces
  // 2h and 2h + 1 in halves 0 and 1 of n2p2[h]
  FF2 n2p2[4];
  float f2[8];  // lazy: fp32 partial sums of the exact squares, the same pieces
#pragma unroll
  for (int lc = 0; lc < 8; ++lc) f2[lc] = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) n2p2[h] = FF2{0ull, 0ull};
  if (warp == kItemWarps) {
    if (lane == 0) {
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(N));
      for (int c = pre; c < min(kStages, nchunks); ++c) load_chunk(c, c);
      int next = min(kStages, nchunks);  // next chunk to load
      for (int c = 0; c < nchunks && ok; ++c) {
        // chunk c must have been loaded: block on its stage's release if not
        while (ok && next <= c) {
          ok = wait_bar(&sh->empty[next % kStages], ((next - kStages) / kStages) & 1);
          if (ok) load_chunk(next, next % kStages), ++next;
        }
        const int st = c % kStages;
        if (!ok || !wait_bar(&sh->full[st], (c / kStages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sbase = smem_u32(stages + st * stage_bytes);
        for (int h = 0; h < nbands; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + h * 256, sdesc_sw128(sbase + h * 16384 + kk * 32),
                     sdesc_sw128(sbase + kk * 32), idesc, (c | kk) != 0);
        mma_commit(&sh->empty[st]);
        // refill released stages without blocking
        while (next < nchunks &&
               mbar_test_wait(&sh->empty[next % kStages], ((next - kStages) / kStages) & 1)) {
          load_chunk(next, next % kStages);
          ++next;
        }
      }
      mma_commit(&sh->done);
      if (!ok) {
        sh->abort_flag = 1;
        record_error(p.ws, BKV_ETIMEOUT, kSiteFpsWait);
      }
    }
    __syncwarp();
  } else {
    const int i = tid;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % kStages;
      ok = __all_sync(0xffffffffu, ok && wait_bar(&sh->full[st], (c / kStages) & 1));
      if (!ok) break;
      if (i < n) {
        const uint8_t* row = stages + st * stage_bytes + i * 128;
        if constexpr (lazy) {
          // the eight squares of a piece (exact in fp32) summed pairwise,
          // then added to the piece's running sum
#pragma unroll
          for (int lc = 0; lc < 8; ++lc) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((lc ^ (i & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float sq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a = __uint_as_float(w[e] << 16), b = __uint_as_float(w[e] & 0xFFFF0000u);
              sq[e] = a * a + b * b;
            }
            f2[lc] += (sq[0] + sq[1]) + (sq[2] + sq[3]);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const uint4 v0 = *reinterpret_cast<const uint4*>(row + (((2 * h) ^ (i & 7)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((2 * h + 1) ^ (i & 7)) << 4));
            ff2_add_squares(n2p2[h], v0, v1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->empty[st]);
    }
    if (!ok) {
      sh->abort_flag = 1;
      if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteFpsWait);
    }
  }
  warp_wait(&sh->done, 0, &sh->abort_flag);
  tc_fence_after();
  if (tid < kItems) {
    const int i = tid;
    float nn;
    if constexpr (lazy) {
      // squared norm from the fp32 sums (at most 14 roundings of positive
      // terms for D = 512); the exact one is formed when a recheck needs it
      nn = ((f2[0] + f2[1]) + (f2[2] + f2[3])) + ((f2[4] + f2[5]) + (f2[6] + f2[7]));
      sh->n2h[i] = i < n ? -1.f : 0.f;
      sh->n2l[i] = 0.f;
    } else {
      FF n2p[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        f2_unpack(n2p2[h].hi, n2p[2 * h].hi, n2p[2 * h + 1].hi);
        f2_unpack(n2p2[h].lo, n2p[2 * h].lo, n2p[2 * h + 1].lo);
      }
      const FF n2 = ff_merge(ff_merge(ff_merge(n2p[0], n2p[1]), ff_merge(n2p[2], n2p[3])),
                             ff_merge(ff_merge(n2p[4], n2p[5]), ff_merge(n2p[6], n2p[7])));
      nn = n2.hi + n2.lo;
      sh->n2h[i] = i < n ? n2.hi : 0.f;
      sh->n2l[i] = i < n ? n2.lo : 0.f;
    }
    sh->inv[i] = (i < n && nn > 0.f) ? 1.f / sqrtf(nn) : 0.f;
  }
  __syncthreads();
  const bool gram_ok = sh->abort_flag == 0;  // block-uniform
  if (warp < kItemWarps) {
    fps_pick<lazy>(p, sh, stages, tbase, gram_ok, u, n, m);
  } else if (next_u >= 0 && lane == 0 && gram_ok) {
    // the next unit's first chunks, while the item warps run the greedy
    // steps: every wait on the barriers of this unit has completed (the
    // Gram is done and the seed is past), so they start again from phase 0
    // every arrival on the stage barriers has landed (the last phase of
    // each stage is complete) before they are initialised again
    bool quiet = wait_bar(&sh->seeded, 0);
    for (int c = max(0, nchunks - kStages); c < nchunks && quiet; ++c)
      quiet = wait_bar(&sh->empty[c % kStages], (c / kStages) & 1);
    if (quiet) {
      for (int st = 0; st < kStages; ++st) {
        mbar_inval(&sh->full[st]);
        mbar_inval(&sh->empty[st]);
        mbar_init(&sh->full[st], 1);
        mbar_init(&sh->empty[st], kItemWarps + 1);
      }
      mbar_inval(&sh->done);
      mbar_inval(&sh->seeded);
      mbar_init(&sh->done, 1);
      mbar_init(&sh->seeded, kItemWarps);
      fence_mbar_init();
      const int k = min(kStages, nchunks);
      for (int c = 0; c < k; ++c) {
        mbar_arrive_expect_tx(&sh->full[c], box_bytes);
        tma_load_3d(stages + c * stage_bytes, bmap, &sh->full[c], 64 * c, 0, next_u);
      }
      sh->preloaded = k;
    } else {
      sh->abort_flag = 1;
      record_error(p.ws, BKV_ETIMEOUT, kSiteFpsWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
  return m;
}

// The CTA's mbarriers and abort flag (thread 0).  With `again` the words
// were initialised before: every wait on them has completed and no copy
// still signals them (the whole CTA has passed a barrier since).
__device__ void init_fps_barriers(FpsShared* sh, bool again) {
  if (again) {
    for (int s = 0; s < kStages; ++s) {
      mbar_inval(&sh->full[s]);
      mbar_inval(&sh->empty[s]);
    }
    mbar_inval(&sh->done);
    mbar_inval(&sh->seeded);
  }
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&sh->full[s], 1);
    mbar_init(&sh->empty[s], kItemWarps + 1);  // every item warp read it + the MMAs ran
  }
  mbar_init(&sh->done, 1);
  mbar_init(&sh->seeded, kItemWarps);
  sh->abort_flag = 0;
  sh->preloaded = 0;
  fence_mbar_init();
}

// Compress unit u's full buffer (C items) to its FPS survivors, kept in slot
// order in buf[0, got); returns got (all threads call, block-uniform).
__device__ int compress_unit(const FpsParams& p, const CUtensorMap* bmap, FpsShared* sh,
                             uint8_t* stages, int stage_rows, int u, uint16_t* buf) {
  const int tid = threadIdx.x, D = p.D;
  const int got = fps_select<false>(p, bmap, sh, stages, stage_rows, u, p.C, p.M, -1);
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
  // generic writes (buffer rows, and the staging in shared memory) before
  // later TMA reads and writes of the same memory
  fence_proxy_async();
  __syncthreads();
  return got;
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
  pdl_trigger();  // scoring may set up on free SMs; it waits for this grid before reading it
  const int D = p.D;
  uint16_t* buf = p.buf + static_cast<size_t>(u) * p.C * D;

  if (tid == 0) init_fps_barriers(sh, false);
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
  if (ok_state && c == p.C) c = compress_unit(p, &bmap, sh, stages, stage_rows, u, buf);

  // ---- 3. beacons: FPS over the current buffer (read-only)
  if (p.want_beacons) {
    const int got =
        ok_state ? fps_select<false>(p, &bmap, sh, stages, stage_rows, u, c, p.M, -1) : 0;
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

// ---- Beacon selection alone (no append, so no count or buffer changes
// here), persistent: CTA b selects for units b, b + G, ... (G at most the
// SM count).  While the item warps run one unit's greedy steps the
// producer warp loads the next unit's first Gram chunks, so the next Gram
// starts with most of its buffer in shared memory.
__device__ __forceinline__ bool runs_gram(const FpsParams& p, int u) {
  const int c = p.cnt[u];
  return c >= 0 && c < p.C && c > p.M && p.M > 0 && !p.first_m;
}

// kLazy (several units per CTA): the exact norms only where a recheck
// needs them (fps_pick).
template <bool kLazy>
__global__ void __launch_bounds__(kThreads, 1)
    fps_beacons_kernel(const __grid_constant__ FpsParams p,
                       const __grid_constant__ CUtensorMap bmap, int stage_rows) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  FpsShared* sh = reinterpret_cast<FpsShared*>(stages + kStages * stage_rows * 128);
  const int tid = threadIdx.x, G = gridDim.x;
  pdl_trigger();  // scoring may set up on free SMs; it waits for this grid before reading it
  const int D = p.D;
  if (tid == 0) init_fps_barriers(sh, false);
  __syncthreads();
  for (int u = blockIdx.x; u < p.U; u += G) {
    const uint16_t* buf = p.buf + static_cast<size_t>(u) * p.C * D;
    int c = p.cnt[u];
    const bool ok_state = c >= 0 && c < p.C;
    if (!ok_state) {
      if (tid == 0) record_error(p.ws, BKV_EDEVICE, kSiteFpsState);
      c = 0;
    }
    const int un = u + G;
    const int next = (un < p.U && runs_gram(p, un)) ? un : -1;
    const int got =
        ok_state ? fps_select<kLazy>(p, &bmap, sh, stages, stage_rows, u, c, p.M, next) : 0;
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
    __syncthreads();  // sel is read before the next unit writes it
    const bool stop = sh->abort_flag != 0;  // block-uniform
    if (!stop && sh->preloaded == 0 && u + G < p.U) {
      // nothing was loaded ahead: the barriers start again here
      if (tid == 0) init_fps_barriers(sh, true);
      __syncthreads();
    }
    if (stop) break;
  }
  // no load may still target this CTA's shared memory when it leaves
  if (tid == kItems)
    for (int k = 0; k < sh->preloaded; ++k) wait_bar(&sh->full[k], 0);
  __syncthreads();
}

// ---- The per-step append on its own (a1), for steps that select no
// beacons: one warp per unit copies the step's query (G*d bf16, at most 256
// 16-byte pieces, at most 8 per lane) into ring slot step % W and buffer
// slot cnt, then counts it.  Only this warp touches the unit, so reading
// cnt and writing cnt + 1 need no atomics.  The query's loads are issued
// before cnt arrives.  A unit whose buffer this fills (cnt == C) is left
// for fps_compress_kernel, launched right after on the same stream.
constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32)
    fps_append_kernel(const __grid_constant__ FpsParams p) {
  pdl_trigger();  // the compress pass may set up; it waits for this grid before reading it
  const int lane = threadIdx.x & 31;
  const int64_t u = static_cast<int64_t>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  if (u >= p.U) return;
  const int nv = p.D / 8;  // 16-byte pieces of an item: 8..256
  const uint4* src = reinterpret_cast<const uint4*>(p.q_new + u * p.D);
  uint4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (lane + 32 * k < nv) v[k] = src[lane + 32 * k];
  const int c = p.cnt[u];
  if (c < 0 || c >= p.C) {  // not a valid buffer state: nothing is written
    if (lane == 0) record_error(p.ws, BKV_EDEVICE, kSiteFpsState);
    return;
  }
  uint4* ring = p.W > 0 ? reinterpret_cast<uint4*>(
                              p.recent_q + (u * p.W + static_cast<int64_t>(p.step % p.W)) * p.D)
                        : nullptr;
  uint4* dst = reinterpret_cast<uint4*>(p.buf + (u * p.C + c) * p.D);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (lane + 32 * k < nv) {
      if (ring != nullptr) ring[lane + 32 * k] = v[k];
      dst[lane + 32 * k] = v[k];
    }
  __syncwarp();
  if (lane == 0) p.cnt[u] = c + 1;
}

// ---- Compress on demand (a2) after fps_append_kernel: a persistent grid
// (at most one CTA per SM) finds the units whose buffer is full and
// compresses each to its FPS survivors, as step 2 of fps_update_kernel
// does.  CTA b takes units b, b + grid, b + 2 grid, ...: it reads their
// counts 256 at a time, lists the full ones in shared memory and compresses
// them one after another, re-initialising its mbarriers between units.  A
// step that fills no buffer costs one short scan per CTA.
__global__ void __launch_bounds__(kThreads, 1)
    fps_compress_kernel(const __grid_constant__ FpsParams p,
                        const __grid_constant__ CUtensorMap bmap, int stage_rows) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  FpsShared* sh = reinterpret_cast<FpsShared*>(stages + kStages * stage_rows * 128);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) init_fps_barriers(sh, false);
  __syncthreads();
  pdl_wait();  // the counts and buffers come from the append
  const int64_t grid = gridDim.x;
  bool again = false;
  for (int64_t k0 = 0; blockIdx.x + k0 * grid < p.U; k0 += kItems) {
    bool full = false;
    int u = -1;
    if (tid < kItems) {
      const int64_t uu = blockIdx.x + (k0 + tid) * grid;
      if (uu < p.U) {
        u = static_cast<int>(uu);
        full = p.cnt[u] == p.C;
      }
    }
    if (tid == 0) sh->ucount = 0;
    __syncthreads();
    if (warp < kItemWarps) {
      const uint32_t b = __ballot_sync(0xffffffffu, full);
      int base = 0;
      if (lane == 0 && b != 0u) base = atomicAdd(&sh->ucount, __popc(b));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (full) sh->ulist[base + __popc(b & ((1u << lane) - 1u))] = u;
    }
    __syncthreads();
    const int n = sh->ucount;
    for (int i = 0; i < n; ++i) {
      const int uu = sh->ulist[i];
      if (again) {
        if (tid == 0) init_fps_barriers(sh, true);
        __syncthreads();
      }
      again = true;
      uint16_t* buf = p.buf + static_cast<size_t>(uu) * p.C * p.D;
      const int got = compress_unit(p, &bmap, sh, stages, stage_rows, uu, buf);
      if (tid == 0) p.cnt[uu] = got;
      if (sh->abort_flag != 0) return;  // a wait timed out (recorded): copies may be in flight
    }
    __syncthreads();  // the list is read before the next batch rewrites it
  }
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

cudaError_t launch_fps(const FpsParams& p, const CUtensorMap& bufmap, int sms, cudaStream_t st) {
  const int rows = fps_stage_rows(p.C);
  const size_t smem = fps_smem_bytes(p.C);
  if (p.q_new == nullptr && p.want_beacons) {
    // beacon selection alone: the persistent kernel, in its throughput
    // form (exact norms on demand) when a CTA takes more than one unit
    const bool lazy = p.U > sms;
    auto* kernel = lazy ? fps_beacons_kernel<true> : fps_beacons_kernel<false>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    kernel<<<lazy ? sms : p.U, kThreads, smem, st>>>(p, bufmap, rows);
    return cudaGetLastError();
  }
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(fps_update_kernel), smem);
  if (e != cudaSuccess) return e;
  fps_update_kernel<<<p.U, kThreads, smem, st>>>(p, bufmap, rows);
  return cudaGetLastError();
}

cudaError_t launch_fps_append_compress(const FpsParams& p, const CUtensorMap& bufmap, int sms,
                                       cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>((p.U + kAppendWarps - 1) / kAppendWarps);
  fps_append_kernel<<<blocks, kAppendWarps * 32, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = fps_stage_rows(p.C);
  const size_t smem = fps_smem_bytes(p.C);
  e = set_smem_once(reinterpret_cast<const void*>(fps_compress_kernel), smem);
  if (e != cudaSuccess) return e;
  // a programmatic dependent of the append: it launches while the append
  // runs and waits for it before reading any count or buffer
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.U < sms ? p.U : sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fps_compress_kernel, p, bufmap, rows);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace bkv
