// Device helpers shared by the FPS kernels (single-CTA and cluster):
// error-free float-float arithmetic for the exactness rechecks, the top-2
// reduction, and the fp32 error bounds that decide when a recheck runs.
#pragma once
#include "common.cuh"

namespace bkv {
namespace fps {

// Bound on |fp32 cosine - exact cosine| for a tensor-core Gram over rows of
// D bf16 values, normalised by 1/||x|| from exact norms (rounded to fp32).
// bf16 products are exact; the fp32 accumulation in steps of 16 products is
// taken to lose at most 2 ulp (2^-22) of the running sum per step, so an
// entry is within e = (D / 16) 2^-22 ||x_i|| ||x_j||; the bound is 1.3 e
// plus 1e-6 for the fp32 normalisation (a few roundings of at most 2^-24).
// The seed's mean sums at most 512 such cosines in fp32 with at most 9
// roundings per term (below 1e-6 in all), so its bound is 1e-6 more.
__device__ __forceinline__ float tau_cos(int D) {
  return 1.3f * static_cast<float>(D / 16) * 0x1p-22f + 1e-6f;
}
__device__ __forceinline__ float tau_mean(int D) { return tau_cos(D) + 1e-6f; }
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* abort) {
  bool ok = *reinterpret_cast<volatile int32_t*>(abort) == 0 && wait_bar(bar, parity);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) *reinterpret_cast<volatile int32_t*>(abort) = 1;
  return ok;
}

// (best value, its index, runner-up value) under the order "smaller value
// first, then smaller index" (argmin; the argmax passes negated values).
struct Top2 {
  float v1;
  int i1;
  float v2;
};
// Order-preserving integer key of a float (smaller value -> smaller key,
// -0 counts as +0) and its inverse: the top-2 reductions compare keys with
// redux.sync.
__device__ __forceinline__ uint32_t fkey(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Warp-wide Top2 of (key, item) with item = lane + base: the minimum by
// redux.sync, its lowest lane by ballot, the runner-up by a second redux
// with that lane masked.  Every lane gets the result.
struct KeyTop2 {
  uint32_t k1;
  int i1;
  uint32_t k2;
};
__device__ __forceinline__ KeyTop2 warp_key_top2(uint32_t key, int base) {
  const int lane = threadIdx.x & 31;
  const uint32_t k1 = __reduce_min_sync(0xffffffffu, key);
  const int l1 = __ffs(__ballot_sync(0xffffffffu, key == k1)) - 1;
  const uint32_t k2 = __reduce_min_sync(0xffffffffu, lane == l1 ? 0xffffffffu : key);
  return KeyTop2{k1, base + l1, k2};
}
// Merge of up to 32 {key, item, runner-up key, -} entries, one per lane
// (lanes without one hold all-ones keys), under the order "smaller key
// first, then smaller item": the smallest key, the lowest item holding it,
// and the runner-up (the winner's own second, or another entry's best).
// Every lane gets the result.
__device__ __forceinline__ uint4 merge_key_top2(uint4 e) {
  const uint32_t k1 = __reduce_min_sync(0xffffffffu, e.x);
  const uint32_t i1 = __reduce_min_sync(0xffffffffu, e.x == k1 ? e.y : 0xffffffffu);
  const uint32_t k2 = __reduce_min_sync(0xffffffffu, (e.x == k1 && e.y == i1) ? e.z : e.x);
  return make_uint4(k1, i1, k2, 0u);
}

// ---- exact-product dot products for the near-tie rechecks.
// B300 runs fp64 at a small fraction of its fp32 rate, so the rechecks
// work on the fp32 pipes: a product of two bf16 values is exact in fp32
// (8-bit significands), and the sum is carried as an unevaluated pair
// hi + lo with Knuth's TwoSum (Knuth, TAOCP vol. 2, 4.2.2), which keeps the
// rounding error of every addition.  The pair is ~2^-44 accurate relative
// to the sum of |terms|; only then is it widened to fp64.  The result is a
// deterministic function of the two rows, symmetric in them, so identical
// items get identical values and exact ties stay exact.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ void ff_add(FF& acc, float p) {
  const float s = acc.hi + p;
  const float bb = s - acc.hi;
  const float e = (acc.hi - (s - bb)) + (p - bb);
  acc.hi = s;
  acc.lo += e;
}
__device__ __forceinline__ void ff_add_products(FF& acc, uint4 a, uint4 b) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    ff_add(acc, __uint_as_float(wa[h] << 16) * __uint_as_float(wb[h] << 16));
    ff_add(acc, __uint_as_float(wa[h] & 0xFFFF0000u) * __uint_as_float(wb[h] & 0xFFFF0000u));
  }
}
// acc += x * (rh + rl) for a bf16 value x: x * rh is split exactly into
// p + e (TwoProd by fma), x * rl is small enough to add rounded.
__device__ __forceinline__ void ff_add_scaled(FF& acc, float x, float rh, float rl) {
  const float p = x * rh;
  const float e = fmaf(x, rh, -p);
  ff_add(acc, p);
  acc.lo += fmaf(x, rl, e);
}
__device__ __forceinline__ FF ff_merge(FF a, FF b) {
  FF r{a.hi, a.lo + b.lo};
  ff_add(r, b.hi);
  return r;
}
// a * b for two unevaluated pairs, ~2^-46 relative: TwoProd of the high
// parts by fma, the cross terms added to its error, one Fast2Sum.
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
  const float s = p + e;
  return FF{s, e - (s - p)};
}
// Two independent float pairs at once.  sm_100 and later have packed fp32
// instructions (add / sub / mul / fma .f32x2) that round each half exactly
// as the scalar instruction does, so two sums carried this way are bit for
// bit the two scalar sums, in half the instructions (1.34x faster on B300
// for this accumulation, which is issue-bound at eight warps per SM).
struct FF2 {
  uint64_t hi, lo;  // {half 0, half 1} of each part
};
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// ff_add on both halves
__device__ __forceinline__ void ff2_add(FF2& acc, uint64_t p) {
  const uint64_t s = f2_add(acc.hi, p);
  const uint64_t bb = f2_sub(s, acc.hi);
  const uint64_t e = f2_add(f2_sub(acc.hi, f2_sub(s, bb)), f2_sub(p, bb));
  acc.hi = s;
  acc.lo = f2_add(acc.lo, e);
}
// ff_add_scaled on both halves: half h adds x_h * (rh + rl).  0 - p is -p
// (both are +0 only where the fma's sum is +0 either way).
__device__ __forceinline__ void ff2_add_scaled(FF2& acc, uint64_t x, uint64_t rh, uint64_t rl) {
  const uint64_t p = f2_mul(x, rh);
  const uint64_t e = f2_fma(x, rh, f2_sub(0ull, p));
  ff2_add(acc, p);
  acc.lo = f2_add(acc.lo, f2_fma(x, rl, e));
}
// ff_add_products(acc_h, v_h, v_h) on both halves: the squares of the eight
// bf16 values of piece v0 go to half 0, those of v1 to half 1, in the scalar
// order (per word: the low value, then the high one).
__device__ __forceinline__ void ff2_add_squares(FF2& acc, uint4 v0, uint4 v1) {
  const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint64_t lo = f2_pack(__uint_as_float(w0[h] << 16), __uint_as_float(w1[h] << 16));
    ff2_add(acc, f2_mul(lo, lo));
    const uint64_t hi =
        f2_pack(__uint_as_float(w0[h] & 0xFFFF0000u), __uint_as_float(w1[h] & 0xFFFF0000u));
    ff2_add(acc, f2_mul(hi, hi));
  }
}
__device__ __forceinline__ double ff_value(FF a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

// 1/sqrt(a) for a = a.hi + a.lo as an unevaluated pair, about 2^-46
// relative, on the fp32 pipes (B300's fp64 square root and division are
// slow): y0 = rsqrtf(a.hi), then one step of the series
// (1 - t)^(-1/2) = 1 + t/2 + 3 t^2 / 8 + O(t^3) with t = 1 - a y0^2 formed
// from exact products (TwoProd by fma); 1 - q below is exact (Sterbenz,
// q within 2^-20 of 1).  Far-from-unit a is scaled by a power of two first.
// a <= 0 gives 0.
__device__ __forceinline__ FF ff_rsqrt(FF a) {
  if (!(a.hi > 0.f)) return FF{0.f, 0.f};
  float sc = 1.f;
  if (a.hi < 0x1p-100f) {
    a.hi *= 0x1p100f;
    a.lo *= 0x1p100f;
    sc = 0x1p50f;
  } else if (a.hi > 0x1p100f) {
    a.hi *= 0x1p-100f;
    a.lo *= 0x1p-100f;
    sc = 0x1p-50f;
  }
  const float y0 = rsqrtf(a.hi);
  const float p = y0 * y0, pe = fmaf(y0, y0, -p);    // y0^2 = p + pe exactly
  const float q = a.hi * p, qe = fmaf(a.hi, p, -q);  // a.hi p = q + qe exactly
  const float t = (1.f - q) - (qe + fmaf(a.hi, pe, a.lo * p));
  const float d = y0 * fmaf(0.375f * t, t, 0.5f * t);
  const float rh = y0 + d;
  return FF{rh * sc, (d - (rh - y0)) * sc};
}

// Exact-product dot product of rows a and b of X by one warp: lane l takes
// the 16-byte pieces l, l + 32, ...; the partial pairs are merged by an
// xor butterfly (TwoSum is exact in either operand order, so every lane ends
// with the same value, and the result is symmetric in a and b).
__device__ __forceinline__ FF warp_dot_rows_ff(const uint16_t* X, int D, int a, int b) {
  const int lane = threadIdx.x & 31;
  const uint4* ra = reinterpret_cast<const uint4*>(X + static_cast<size_t>(a) * D);
  const uint4* rb = reinterpret_cast<const uint4*>(X + static_cast<size_t>(b) * D);
  FF acc{0.f, 0.f};
  for (int v = lane; v < D / 8; v += 32) ff_add_products(acc, ra[v], rb[v]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF other{__shfl_xor_sync(0xffffffffu, acc.hi, o), __shfl_xor_sync(0xffffffffu, acc.lo, o)};
    acc = ff_merge(acc, other);
  }
  return acc;
}
__device__ __forceinline__ double warp_dot_rows(const uint16_t* X, int D, int a, int b) {
  return ff_value(warp_dot_rows_ff(X, D, a, b));
}
// fp64 1/||x_a|| from the exact squared norm of row a (one warp).
__device__ __forceinline__ double warp_rnorm(const uint16_t* X, int D, int a) {
  return ff_value(ff_rsqrt(warp_dot_rows_ff(X, D, a, a)));
}

}  // namespace fps
}  // namespace bkv
