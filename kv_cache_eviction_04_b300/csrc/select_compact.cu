// Top-B_KV selection and in-place, order-preserving K/V compaction.
//
// BeaconKV pages: inkeast.github.io reading, section 三 (the kept set is
// I = TopK(score(K,V), B_KV)); aimodeling.com article, section
// "用信标 query 预判" (only the highest-scoring entries survive while a recent
// sliding window is always kept).
//
// One thread-block cluster of `ncl` CTAs per unit.  Every CTA selects on its
// own (the scores of a unit are a few KB, far less than its K and V rows).
// The unit's scores are read once, as order-preserving integer keys, into
// shared memory (it reuses the copy ring, which is idle until then); longer
// caches than the ring holds read the keys from global memory instead.
//   * radix select on the keys in three passes of 11, 11 and 10 bits from
//     the top: a 2048-bin shared-memory histogram filled with shared-memory
//     atomics (cheaper here than aggregating lanes with match.any first),
//     then a block scan finds the bin holding the k-th largest;
//   * the ascending kept list: each warp scans its own span of slots, lanes
//     taking interleaved slots (conflict-free), with a ballot per step for
//     the order and a scan over the warps for the offsets (equal scores:
//     the lower slots first).
// The unit's old key positions are staged in the ring's last two buffers
// and gathered for the moved rows while the first waves' loads fly.
// Compaction (row i <- row kept[i], kept[i] >= i) runs in waves over the
// rows that move, [first, n_kept): wave w covers ncl consecutive slices of
// RS rows, one per CTA.  Each CTA gathers its slice's source rows of K and V
// into a shared-memory ring (TMA bulk copies per run of consecutive source
// rows when the unit's sources are dense, else 16-byte cp.async copies
// spread over all its threads), the cluster meets at a hardware barrier
// once every CTA's copies of the wave have landed, and only then is each
// slice stored back (two TMA bulk stores of contiguous rows).  Sources of a
// wave lie at or above its first row, so stores of earlier waves never
// touch them, and a wave's stores wait for all of its loads: in-place
// compaction needs no second buffer and no spin-wait between CTAs.  Loads
// run nbufs - 2 waves ahead.
// The hole-filling mode (an order-free layout: the holes below the new
// length take the kept rows past it) replaces the waves with direct copies
// of (hole, source) pairs; see fill_compact.
#include "common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

// Threads per CTA: 256, or 512 for long caches in the order-preserving
// layout, whose selection passes over tens of thousands of keys are
// latency-bound loops that more warps hide better (measured on 32768 keys:
// 2.76 against 3.42 ms for the 32K-cache round; on caches of 1 to 2 K keys
// 256 threads were faster).  The hole-filling copy loop holds 144
// registers per thread, so that layout stays at 256.
constexpr int kLongCache = 8192;  // L_cap from which the ordered layout takes 512 threads
constexpr int kMaxWarps = 16;
constexpr int kMaxBufs = 8;             // ring of wave buffers (count set by the host)
constexpr uint32_t kBufBig = 32768;     // bytes of one wave of one CTA (RS rows of K and V)
constexpr uint32_t kBufSmall = 16384;   // the same when a very large B_KV leaves less room
constexpr int kFillAhead = 16;          // 16-byte loads per thread in flight (hole-filling copy)

__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0;                         // -0.0 counts as +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // larger float -> larger key
}

// Inclusive block-wide prefix sum of one int per thread.
template <int NT>
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  int add = 0;
  for (int w = 0; w < warp; ++w) add += warp_tot[w];
  __syncthreads();
  return v + add;
}

// Block-wide sum of one int per thread (every thread gets it).
template <int NT>
__device__ __forceinline__ int block_sum(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  __syncthreads();  // earlier readers of warp_tot are done
  if (lane == 0) warp_tot[warp] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += warp_tot[w];
  return t;
}

struct __align__(16) Smem {
  uint64_t wbar[kMaxBufs];  // per ring buffer: a wave's gathered bytes have landed
  int32_t hist[2048];
  int32_t warp_tot[kMaxWarps];
  int32_t warp_eq[kMaxWarps];
  uint32_t prefix;
  int32_t krem;
  int32_t first;
  int32_t pad;
};

// Layout: Smem | kept list [B] | new kpos of this CTA's rows [B + 128] | ring.
// (A CTA's kpos entries are indexed wave * RS + row; the last wave may run
// up to RS - 1 <= 127 entries past its rows.)
__host__ __device__ constexpr size_t kept_offset() { return (sizeof(Smem) + 15) & ~size_t(15); }
__host__ __device__ inline size_t kpn_offset(int B) {
  return kept_offset() + static_cast<size_t>(B) * 4;
}
__host__ __device__ inline size_t bufs_offset(int B) {
  return (kpn_offset(B) + (static_cast<size_t>(B) + 128) * 4 + 1023) & ~static_cast<size_t>(1023);
}

// Select the kept slots of unit u into kept_s[0, n_kept); returns n_kept.
// keys_s: the unit's order keys in shared memory, or null (read scores).
// kStaged: the keys are read from keys_s (shared memory), else from the
// scores in global memory; a template parameter so that no key read
// carries a load of the other source (a runtime choice per read let both
// loads be issued, a global load for every key of every pass).
template <int NT, bool kStaged>
__device__ int select_kept(const SelectParams& p, const float* sc, const uint32_t* keys_s,
                           int L, int32_t* kept_s, Smem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int kWarps = NT / 32;
  constexpr int kBins = 2048 / NT;  // histogram bins each thread scans
  const int n_kept = L <= p.B ? L : p.B;
  if (L <= p.B) {
    for (int i = tid; i < n_kept; i += NT) kept_s[i] = i;
    __syncthreads();
    return n_kept;
  }
  auto key_at = [&](int j) {
    if constexpr (kStaged)
      return keys_s[j];
    else
      return order_key(sc[j]);
  };
  // ---------------- radix select of the (B - R)-th largest candidate:
  // digits of 11, 11 and 10 bits from the top; thread t owns the kBins bins
  // from 2047 - kBins t down (descending) in the scan of each pass
  const int ncand = L - p.R;
  const int k = p.B - p.R;
  uint32_t prefix = 0;
  int krem = k;
  if (k > 0) {
    constexpr int kShift[3] = {21, 10, 0};
    constexpr uint32_t kDigit[3] = {2047u, 2047u, 1023u};
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = kShift[pass];
      const uint32_t dmask = kDigit[pass];
      const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (kShift[pass - 1]));
#pragma unroll
      for (int b8 = 0; b8 < kBins; ++b8) sm->hist[tid * kBins + b8] = 0;
      __syncthreads();
      // four slots per thread per step, loaded before any is used (indices
      // clamped into range; slots past ncand are discarded)
      for (int j0 = 0; j0 < ncand; j0 += 4 * NT) {
        uint32_t kv[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) kv[q4] = key_at(min(j0 + q4 * NT + tid, ncand - 1));
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const bool in = j0 + q4 * NT + tid < ncand;
          const uint32_t key = kv[q4];
          const bool hit = in && (key & hmask) == prefix;
          const uint32_t bin = (key >> shift) & dmask;
          if (hit) atomicAdd(&sm->hist[bin], 1);
        }
      }
      __syncthreads();
      int c[kBins], loc = 0;
#pragma unroll
      for (int b8 = 0; b8 < kBins; ++b8) {
        c[b8] = sm->hist[2047 - tid * kBins - b8];
        loc += c[b8];
      }
      const int incl = block_incl_scan<NT>(loc, sm->warp_tot);
      int above = incl - loc;  // candidates in higher bins than this thread's
      if (above < krem && incl >= krem) {
#pragma unroll
        for (int b8 = 0; b8 < kBins; ++b8) {
          if (above < krem && above + c[b8] >= krem) {
            sm->prefix = prefix | (static_cast<uint32_t>(2047 - tid * kBins - b8) << shift);
            sm->krem = krem - above;
          }
          above += c[b8];
        }
      }
      __syncthreads();
      prefix = sm->prefix;
      krem = sm->krem;
    }
  } else {
    prefix = 0xFFFFFFFFu;  // keep no candidate: only the window
    krem = 0;
  }
  const uint32_t T = prefix;
  const int need_eq = krem;  // candidates equal to T kept, lowest slots first
  // ---------------- ascending kept list.  Warp w takes slots
  // [w s, w s + s) (s a multiple of 32), lane l the slot w s + 32 i + l in
  // step i: shared-memory reads are conflict-free and a ballot per step
  // keeps the slot order.  Pass 1 counts, per warp, the slots kept for sure
  // (key > T, or in the recent window) and the candidates equal to T; a scan
  // over the warps gives each warp the equal candidates before it and its
  // first output index; pass 2 keeps the first need_eq equal candidates in
  // slot order and writes the list.
  const int warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int span = ((L + 32 * kWarps - 1) / (32 * kWarps)) * 32;
  const int jb = min(warp * span, L), je = min(jb + span, L);
  // keys of four steps are loaded before any is used (indices clamped into
  // range; slots past the span are discarded)
  auto load4 = [&](int i0, uint32_t (&kv)[4]) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) kv[q4] = key_at(min(i0 + 32 * q4 + lane, L - 1));
  };
  auto classify = [&](int j, uint32_t key, bool& gt, bool& eq) {
    const bool in = j < je;
    const bool win = in && j >= ncand;  // the recent window: always kept
    gt = win || (in && key > T);
    eq = in && !win && key == T;
  };
  int n_gt = 0, n_eq = 0;  // per lane, summed over the warp below
  for (int i0 = jb; i0 < je; i0 += 128) {
    uint32_t kv[4];
    load4(i0, kv);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      bool gt, eq;
      classify(i0 + 32 * q4 + lane, kv[q4], gt, eq);
      n_gt += gt;
      n_eq += eq;
    }
  }
  n_gt = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n_gt)));
  n_eq = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n_eq)));
  if (lane == 0) {
    sm->warp_tot[warp] = n_gt;
    sm->warp_eq[warp] = n_eq;
  }
  __syncthreads();
  int out = 0, e = 0;  // this warp's first output index and equal candidates before it
  for (int w = 0; w < warp; ++w) {
    const int eq_w = sm->warp_eq[w];
    out += sm->warp_tot[w] + min(max(need_eq - e, 0), eq_w);
    e += eq_w;
  }
  // every equal candidate of this warp is kept, or none is, unless the cut
  // falls inside the warp (warp-uniform); only then are they ranked per step
  const bool eq_all = e + sm->warp_eq[warp] <= need_eq, eq_none = e >= need_eq;
  for (int i0 = jb; i0 < je; i0 += 128) {
    uint32_t kv[4];
    load4(i0, kv);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int j = i0 + 32 * q4 + lane;
      bool gt, eq;
      classify(j, kv[q4], gt, eq);
      bool keep;
      if (eq_all || eq_none) {
        keep = gt || (eq && eq_all);
      } else {
        const uint32_t beq = __ballot_sync(0xffffffffu, eq);
        keep = gt || (eq && e + __popc(beq & lt_mask) < need_eq);
        e += __popc(beq);
      }
      const uint32_t bk = __ballot_sync(0xffffffffu, keep);
      if (keep) kept_s[out + __popc(bk & lt_mask)] = j;
      out += __popc(bk);
    }
  }
  __syncthreads();
  return n_kept;
}

// Hole-filling (order-free) compaction of unit u, whose n = n_kept kept
// slots are kept_s[0, n) in ascending order: a kept slot below n keeps its
// row, and the slots below n that are not kept (the holes), ascending, take
// the kept slots at or past n, ascending.  Sources lie at or past n and
// destinations below it, so the copies need no order among themselves and
// no staging: every CTA of the cluster copies its share of the (hole,
// source) pairs with 16-byte loads and stores, kFillAhead per thread in
// flight (the copy is bound by the bytes each SM keeps in flight).
// `hole` holds up to n entries, `bits` up to n bits.
template <int NT>
__device__ void fill_compact(const SelectParams& p, int u, int rank, int ncl, int n,
                             const int32_t* kept_s, int32_t* hole, uint32_t* bits, Smem* sm,
                             int32_t* kp, uint8_t* Kb, uint8_t* Vb, uint32_t rb) {
  const int tid = threadIdx.x;
  const int nwords = (n + 31) >> 5;
  for (int w = tid; w < nwords; w += NT) bits[w] = 0u;
  int below = 0;  // kept slots below n: a prefix of the ascending list
  for (int j = tid; j < n; j += NT) below += kept_s[j] < n ? 1 : 0;
  const int c = block_sum<NT>(below, sm->warp_tot);  // its barriers also publish the zeroed bits
  for (int j = tid; j < c; j += NT) atomicOr(&bits[kept_s[j] >> 5], 1u << (kept_s[j] & 31));
  __syncthreads();
  // ascending hole list: thread t takes words [t wpt, (t + 1) wpt) of the map
  auto hole_bits = [&](int w) {
    uint32_t m = ~bits[w];
    const int valid = n - 32 * w;  // slots of this word below n
    return valid < 32 ? m & ((1u << valid) - 1u) : m;
  };
  const int wpt = (nwords + NT - 1) / NT;
  const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(hole_bits(w));
  int pos = block_incl_scan<NT>(cnt, sm->warp_tot) - cnt;
  for (int w = w0; w < w1; ++w) {
    uint32_t m = hole_bits(w);
    while (m != 0u) {
      hole[pos++] = 32 * w + __ffs(m) - 1;
      m &= m - 1u;
    }
  }
  __syncthreads();
  const int h = n - c;  // holes = kept slots at or past n
  if (rank == 0 && p.kept != nullptr) {  // the source slot of every row
    int32_t* ko = p.kept + static_cast<size_t>(u) * p.B;
    for (int i = tid; i < p.B; i += NT) ko[i] = i < n ? i : -1;
    __syncthreads();
    for (int k = tid; k < h; k += NT) ko[hole[k]] = kept_s[c + k];
  }
  const int k0 = static_cast<int>(static_cast<int64_t>(h) * rank / ncl);
  const int k1 = static_cast<int>(static_cast<int64_t>(h) * (rank + 1) / ncl);
  for (int k = k0 + tid; k < k1; k += NT) kp[hole[k]] = kp[kept_s[c + k]];
  // element e of this CTA's pairs: pair k0 + e / per_pair, 16-byte piece
  // e % per_pair (K pieces first, then V)
  const int ppr = static_cast<int>(rb / 16);
  const int per_pair = 2 * ppr;
  const int total = (k1 - k0) * per_pair;
  for (int e0 = tid; e0 < total; e0 += kFillAhead * NT) {
    uint4 v[kFillAhead];
    uint8_t* dst[kFillAhead];
#pragma unroll
    for (int q = 0; q < kFillAhead; ++q) {
      const int e = e0 + q * NT;
      const int ec = e < total ? e : total - 1;  // clamped: a valid address, store skipped
      const int k = k0 + ec / per_pair, pc = ec % per_pair;
      const bool is_v = pc >= ppr;
      const size_t off = static_cast<size_t>(is_v ? pc - ppr : pc) * 16;
      uint8_t* base = is_v ? Vb : Kb;
      v[q] = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(kept_s[c + k]) * rb + off);
      dst[q] = e < total ? base + static_cast<size_t>(hole[k]) * rb + off : nullptr;
    }
#pragma unroll
    for (int q = 0; q < kFillAhead; ++q)
      if (dst[q] != nullptr) *reinterpret_cast<uint4*>(dst[q]) = v[q];
  }
}

// kFill: the hole-filling compaction (p.fill), a separate instantiation so
// that its copy loop's registers do not lower the occupancy of the
// order-preserving one.
template <bool kFill, int NT>
__global__ void __launch_bounds__(NT)
    select_compact_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem* sm = reinterpret_cast<Smem*>(smem_raw);
  int32_t* kept_s = reinterpret_cast<int32_t*>(smem_raw + kept_offset());
  int32_t* kpn = reinterpret_cast<int32_t*>(smem_raw + kpn_offset(p.B));
  uint8_t* bufs = smem_raw + bufs_offset(p.B);
  const int nbufs = p.nbufs;
  const int ncl = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int u = blockIdx.x / ncl;
  const int tid = threadIdx.x;
  const float* sc = p.scores + static_cast<size_t>(u) * p.L_cap;
  // the scores, and the K rows that scoring reads, belong to the previous
  // kernel of the stream until it completes
  pdl_wait();

  int L = p.L[u];
  const bool valid = L >= 0 && L <= p.L_cap;
  if (!valid) {
    if (tid == 0 && rank == 0) record_error(p.ws, BKV_EDEVICE, kSiteSelectState);
    L = 0;
  }
  if (tid == 0) {
    sm->first = 0x7fffffff;
    for (int b = 0; b < nbufs; ++b) mbar_init(&sm->wbar[b], 1);
    fence_mbar_init();
  }
  const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
  const size_t ubase = static_cast<size_t>(u) * p.L_cap;
  int32_t* kp = p.kpos + ubase;
  // The unit's keys (from the start of the ring) and key positions (in its
  // last two buffers, which the first gathers below do not touch) are staged
  // in the still idle copy ring when they fit.
  const size_t lbytes = static_cast<size_t>(L) * 4;
  const uint32_t bufb = static_cast<uint32_t>(p.buf_bytes);
  const size_t tail_off = static_cast<size_t>(nbufs - 2) * bufb;
  int32_t* kpos_s = (L > p.B && lbytes <= 2 * static_cast<size_t>(bufb))
                        ? reinterpret_cast<int32_t*>(bufs + tail_off)
                        : nullptr;
  uint32_t* keys_s =
      (L > p.B && lbytes <= (kpos_s ? tail_off : static_cast<size_t>(nbufs) * bufb))
          ? reinterpret_cast<uint32_t*>(bufs)
          : nullptr;
  // When the unit's rows are 16-byte aligned (then so are keys_s + 4i and
  // kpos_s + 4i: the ring is 1024-byte aligned) the staging copies are
  // 16-byte cp.async copies, all of them in flight at once (a long cache's
  // 128 KB of scores would otherwise arrive a few loads per thread at a
  // time); the scores are then turned into order keys in place.
  const bool sc16 = (reinterpret_cast<uintptr_t>(sc) & 15u) == 0;
  const bool kp16 = (reinterpret_cast<uintptr_t>(kp) & 15u) == 0;
  const int n4 = L >> 2;
  if (keys_s != nullptr && sc16)
    for (int i = tid; i < n4; i += NT) cp_async16(keys_s + 4 * i, sc + 4 * i);
  if (kpos_s != nullptr && kp16)
    for (int i = tid; i < n4; i += NT) cp_async16(kpos_s + 4 * i, kp + 4 * i);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (keys_s != nullptr) {
    if (sc16) {
      uint4* k4 = reinterpret_cast<uint4*>(keys_s);
      for (int i = tid; i < n4; i += NT) {
        const uint4 v = k4[i];
        k4[i] = make_uint4(order_key(__uint_as_float(v.x)), order_key(__uint_as_float(v.y)),
                           order_key(__uint_as_float(v.z)), order_key(__uint_as_float(v.w)));
      }
      for (int j = 4 * n4 + tid; j < L; j += NT) keys_s[j] = order_key(sc[j]);
    } else {
#pragma unroll 8
      for (int j = tid; j < L; j += NT) keys_s[j] = order_key(sc[j]);
    }
  }
  if (kpos_s != nullptr) {
    if (kp16) {
      for (int j = 4 * n4 + tid; j < L; j += NT) kpos_s[j] = kp[j];
    } else {
#pragma unroll 8
      for (int j = tid; j < L; j += NT) kpos_s[j] = kp[j];
    }
  }
  __syncthreads();
  const int n_kept = keys_s != nullptr ? select_kept<NT, true>(p, sc, keys_s, L, kept_s, sm)
                                       : select_kept<NT, false>(p, sc, keys_s, L, kept_s, sm);
  // first destination row whose source differs (kept[i] == i before it)
  for (int i = tid; i < n_kept; i += NT)
    if (kept_s[i] != i) atomicMin(&sm->first, i);
  __syncthreads();  // the keys in the ring are dead from here on
  const int first = min(sm->first, n_kept);

  if constexpr (kFill) {
    fill_compact<NT>(p, u, rank, ncl, n_kept, kept_s, kpn, reinterpret_cast<uint32_t*>(bufs), sm, kp,
                 p.K + ubase * rb, p.V + ubase * rb, rb);
    cluster_sync();  // every CTA of the unit has read L and finished its copies
    if (rank == 0 && tid == 0 && valid) p.L[u] = n_kept;
    return;
  }

  if (rank == 0 && p.kept != nullptr)
    for (int i = tid; i < p.B; i += NT)
      p.kept[static_cast<size_t>(u) * p.B + i] = i < n_kept ? kept_s[i] : -1;

  // ---------------- compaction in cluster-wide waves
  const int RS = static_cast<int>(bufb / (2 * rb));  // rows per CTA per wave
  uint8_t* Kb = p.K + ubase * rb;
  uint8_t* Vb = p.V + ubase * rb;
  const int nmove = n_kept - first;
  const int per_wave = ncl * RS;
  const int nw = nmove > 0 ? (nmove + per_wave - 1) / per_wave : 0;

  auto slice = [&](int w, int& r0, int& cnt) {
    r0 = first + (w * ncl + rank) * RS;
    cnt = max(0, min(RS, n_kept - r0));
  };
  // A wave's source rows of K and V are gathered into one ring buffer (K
  // rows first, then V rows), and thread 0 then writes the wave's
  // contiguous destination rows back with two bulk stores.  The gather:
  //  * sources in runs of at least four consecutive rows on average (a
  //    block-uniform choice per unit): warp 0 issues one TMA bulk copy per
  //    run (runs cut at every 32 rows) and matrix, completion counted in
  //    bytes on the buffer's mbarrier;
  //  * scattered sources: every thread issues 16-byte cp.async copies, one
  //    commit group per wave.
  const int warp = tid >> 5, lane = tid & 31;
  int nruns = 0;
  for (int i = first + tid; i < n_kept; i += NT)
    nruns += (i == first || kept_s[i - 1] + 1 != kept_s[i]) ? 1 : 0;
  const bool use_tma = 4 * block_sum<NT>(nruns, sm->warp_tot) <= n_kept - first;
  const int ppr = static_cast<int>(rb / 16);  // 16-byte pieces per row
  auto issue_cp = [&](int w) {  // every thread
    int r0, cnt;
    slice(w, r0, cnt);
    uint8_t* buf = bufs + (w % nbufs) * bufb;
    for (int e = tid; e < 2 * cnt * ppr; e += NT) {
      const int t = e / ppr, pc = e % ppr;
      const bool is_v = t >= cnt;
      const int row = is_v ? t - cnt : t;
      const size_t src = static_cast<size_t>(kept_s[r0 + row]) * rb + pc * 16;
      cp_async16(buf + (is_v ? RS + row : row) * rb + pc * 16, (is_v ? Vb : Kb) + src);
    }
  };
  auto issue = [&](int w) {  // warp 0
    int r0, cnt;
    slice(w, r0, cnt);
    const int b = w % nbufs;
    uint8_t* buf = bufs + b * bufb;
    if (lane == 0) mbar_arrive_expect_tx(&sm->wbar[b], 2u * static_cast<uint32_t>(cnt) * rb);
    __syncwarp();
    for (int t0 = 0; t0 < cnt; t0 += 32) {
      const int t = t0 + lane;
      const bool live = t < cnt;
      const int src = live ? kept_s[r0 + t] : 0;
      const bool start = live && (lane == 0 || kept_s[r0 + t - 1] + 1 != src);
      const uint32_t starts = __ballot_sync(0xffffffffu, start);
      if (start) {
        const uint32_t above = starts & ~((2u << lane) - 1u);  // later run starts
        const int end = above != 0u ? __ffs(above) - 1 : min(32, cnt - t0);
        const uint32_t bytes = static_cast<uint32_t>(end - lane) * rb;
        const size_t off = static_cast<size_t>(src) * rb;
        bulk_load(buf + static_cast<size_t>(t) * rb, Kb + off, bytes, &sm->wbar[b]);
        bulk_load(buf + static_cast<size_t>(RS + t) * rb, Vb + off, bytes, &sm->wbar[b]);
      }
    }
  };
  // Waves w + 1 .. w + kAhead are in flight while wave w is stored.  Wave
  // w + kAhead reuses the buffer of wave w + kAhead - nbufs = w - 2, whose
  // store is the older of the two outstanding ones (waves w - 2 and w - 1).
  // Wave w is the (w / nbufs)-th use of its buffer: its mbarrier phase has
  // that parity.  The first kAhead waves use buffers 0 .. nbufs - 3 only.
  const int kAhead = nbufs - 2;
  if (use_tma) {
    if (warp == 0)
      for (int w = 0; w < min(kAhead, nw); ++w) issue(w);
  } else {
    for (int w = 0; w < kAhead; ++w) {  // one group per wave slot, empty past the last wave
      if (w < nw) issue_cp(w);
      cp_async_commit();
    }
  }
  bool failed = false;  // block-uniform
  int failed_at = nw;    // first wave whose gather never landed
  // New kpos of every row this CTA writes, gathered while those gathers fly
  // and before the first wave's barrier (no CTA writes kpos before it);
  // entry w * RS + t = wave w, row t.
  // (the staged and the global source in separate loops, so that no read
  // also issues a load of the other)
  if (kpos_s != nullptr) {
    for (int e = tid; e < nw * RS; e += NT) {
      int r0, cnt;
      slice(e / RS, r0, cnt);
      if (e % RS < cnt) kpn[e] = kpos_s[kept_s[r0 + e % RS]];
    }
  } else {
    for (int e = tid; e < nw * RS; e += NT) {
      int r0, cnt;
      slice(e / RS, r0, cnt);
      if (e % RS < cnt) kpn[e] = kp[kept_s[r0 + e % RS]];
    }
  }
  __syncthreads();  // the staged key positions are dead from here on

  for (int w = 0; w < nw; ++w) {
    if (tid == 0) bulk_wait_read<1>();  // all stores but wave w - 1's have read smem
    __syncthreads();
    bool here = true;
    if (use_tma) {
      if (warp == 0 && w + kAhead < nw && !failed) issue(w + kAhead);
      here = !failed && wait_bar(&sm->wbar[w % nbufs], (w / nbufs) & 1);
    } else {
      // "wave w landed" is "at most kAhead groups pending"
      if (w + kAhead < nw) issue_cp(w + kAhead);
      cp_async_commit();
      cp_async_wait_dyn(kAhead);
      fence_proxy_async_shared();  // this thread's smem writes -> the bulk stores
    }
    // A wave that never lands stops the copies but not the loop: every CTA
    // of the cluster still meets at each of its barriers.
    const bool landed = __syncthreads_and(here);
    if (!landed && !failed) {
      if (tid == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteSelectWait);
      failed_at = w;
    }
    failed = failed || !landed;
    int r0, cnt;
    slice(w, r0, cnt);
    // Every CTA's sources of wave w are in its shared memory, so only
    // execution order matters here; a one-CTA cluster needs nothing more.
    if (ncl > 1) cluster_sync_relaxed();
    if (cnt > 0 && !failed) {
      if (tid == 0) {
        const uint8_t* buf = bufs + (w % nbufs) * bufb;
        fence_proxy_async_shared();
        bulk_store(Kb + static_cast<size_t>(r0) * rb, buf, cnt * rb);
        bulk_store(Vb + static_cast<size_t>(r0) * rb, buf + RS * rb, cnt * rb);
        bulk_commit();
      }
      if (tid < cnt) kp[r0 + tid] = kpn[w * RS + tid];
    }
  }
  cp_async_wait<0>();
  if (tid == 0) bulk_wait<0>();
  // After a gather that never landed no further wave was issued, but waves
  // failed_at .. failed_at + kAhead may still have bulk loads in flight into
  // this CTA's shared memory: wait for them (bounded) before the CTA exits.
  // A wave that still has not landed then is left in flight; its error is
  // already recorded.
  if (use_tma && failed && tid == 0)
    for (int w = failed_at; w < min(nw, failed_at + kAhead + 1); ++w)
      wait_bar(&sm->wbar[w % nbufs], (w / nbufs) & 1);
  cluster_sync();  // every CTA of the unit has read L and finished its copies
  if (rank == 0 && tid == 0 && valid) p.L[u] = n_kept;
}

}  // namespace

// Ring of the copy waves: buffers of 32 KB (16 KB when a very large B_KV
// leaves no room for three of 32 KB).  As many as fit (at most 8) when there
// are few units, each CTA then streaming with a deep pipeline.  With many
// units, just enough to stage a unit's keys (at least 3) when that lets two
// CTAs share an SM, so that one copies while the other selects; when even
// that ring is too large for two CTAs per SM (long caches, large B_KV), the
// deep ring again, since a lone CTA per SM then needs every wave in flight
// it can hold.  nbufs = 0: not even three buffers fit.
void select_ring(int B, int L_cap, bool many_units, int* nbufs, int* buf_bytes) {
  const size_t off = bufs_offset(B);
  size_t bb = kBufBig;
  if (off + 3 * bb > 232448) bb = kBufSmall;
  *buf_bytes = static_cast<int>(bb);
  if (off + 3 * bb > 232448) {
    *nbufs = 0;
    return;
  }
  int n = static_cast<int>((232448 - off) / bb);
  if (n > kMaxBufs) n = kMaxBufs;
  if (many_units) {
    const size_t stage = (static_cast<size_t>(L_cap) * 4 + bb - 1) / bb;
    const int want = stage < 3 ? 3 : static_cast<int>(stage);
    // two CTAs share an SM's 228 KB (each also reserves 1 KB)
    const bool two_per_sm = off + static_cast<size_t>(want) * bb <= 113 * 1024;
    if (two_per_sm && want < n) n = want;
  }
  *nbufs = n;
}

size_t select_smem_bytes(int B, int nbufs, int buf_bytes) {
  return bufs_offset(B) + static_cast<size_t>(nbufs) * buf_bytes;
}

cudaError_t launch_select_compact(const SelectParams& p, cudaStream_t st) {
  const size_t smem = select_smem_bytes(p.B, p.nbufs, p.buf_bytes);
  const bool wide = !p.fill && p.L_cap >= kLongCache;
  auto* kernel = p.fill ? select_compact_kernel<true, 256>
                        : (wide ? select_compact_kernel<false, 512> : select_compact_kernel<false, 256>);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.U * p.ncl));
  cfg.blockDim = dim3(wide ? 512 : 256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.ncl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of the scoring kernel: it launches while that
  // kernel finishes and waits for it before touching any of its data
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace bkv
