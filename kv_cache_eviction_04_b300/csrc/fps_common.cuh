// Device helpers shared by the FPS kernels (single-CTA and cluster):
// error-free float-float arithmetic for the exactness rechecks, the top-2
// reduction, and the fp32 error bounds that decide when a recheck runs.
#pragma once
#include "common.cuh"

namespace bkv {
namespace fps {

// Bound on |fp32 cosine - exact cosine| for the tensor-core Gram (bf16
// products are exact; fp32 accumulation over up to 2048 terms in blocks of
// 16, plus the normalisation by exact norms) with a safety factor.  The
// seed's mean sums its terms error-free, so its bound is the same plus the
// final rounding.
constexpr float kTauCos = 4e-5f;
constexpr float kTauMean = 4.1e-5f;
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
__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b) {
  const bool a_first = a.v1 < b.v1 || (a.v1 == b.v1 && a.i1 < b.i1);
  Top2 r;
  if (a_first) {
    r.v1 = a.v1;
    r.i1 = a.i1;
    r.v2 = fminf(a.v2, b.v1);
  } else {
    r.v1 = b.v1;
    r.i1 = b.i1;
    r.v2 = fminf(b.v2, a.v1);
  }
  return r;
}
// Warp-wide Top2 by xor shuffles (every lane gets the result).
__device__ __forceinline__ Top2 warp_top2(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 o2;
    o2.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
    o2.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    o2.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
    t = top2_merge(t, o2);
  }
  return t;
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
__device__ __forceinline__ double ff_value(FF a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

// Exact-product dot product of rows a and b of X by one warp: lane l takes
// the 16-byte pieces l, l + 32, ...; the partial pairs are merged by an
// xor butterfly (TwoSum is exact in either operand order, so every lane ends
// with the same value, and the result is symmetric in a and b).
__device__ __forceinline__ double warp_dot_rows(const uint16_t* X, int D, int a, int b) {
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
  return ff_value(acc);
}

}  // namespace fps
}  // namespace bkv
