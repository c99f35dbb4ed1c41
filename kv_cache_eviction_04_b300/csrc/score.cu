// Eviction scoring: per-key max (or mean) over (query, head) rows of the
// softmax attention of the W recent queries and the M beacons.
//
// BeaconKV pages: wzjinhao.cn explainer, section "信标查询怎么用：位置对齐与打分
// 策略" -- beacons are rotated to the current decode position, recent queries
// keep the positions they were generated at, and a key's importance is the
// maximum over queries (max beats mean); inkeast.github.io reading, section
// 三, scoring with the union of recent and beacon queries.
//
// Three paths, all tcgen05 kernels fed by TMA:
//   score_fused_kernel    both passes in one persistent kernel (one CTA per
//                         SM takes units in turn; more than 256 rows in
//                         groups of 256);
//   score_stats + final   the keys of a unit split over CTAs: pass 1 writes
//                         per-split (m, z), pass 2 merges them (few units
//                         with long caches);
//   score_cluster_kernel  one pass on a cluster, the logits kept in TMEM
//                         (small rounds, at most 128 rows).
// The two-pass kernels put, in
//   pass 1  rows on the 128 TMEM lanes, keys on the columns: D = Q * K^T;
//           each thread owns one row and keeps a running max and sum of
//           exp2 over its keys;
//   pass 2  keys on the TMEM lanes, rows on the columns: D = K * Q^T; each
//           thread owns one key and takes the max (or mean) of the
//           normalised probability over rows in registers.
// Queries are rotated in fp32 (angles reduced in extended precision) and
// carried as q = q_hi + q_lo, two bf16 terms; both terms run through the
// tensor core into one fp32 accumulator, so the logits carry ~2^-17
// relative query error instead of bf16's 2^-9.  Logits are kept in log2
// units (log2(e)/sqrt(d) is folded into the queries).
#include "common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

constexpr int kThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpiThreads = 128;
constexpr int kTileKeys = 128;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also ORs a predicate over its n threads: every thread
// gets the same verdict (for decisions that must be uniform across warps).
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " barrier.cta.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Every lane of the warp waits on `bar`; the verdict is warp-uniform.  Once
// any wait of the CTA has timed out (`abort` set) later waits fail at once,
// so every role drains its loop without blocking and all threads still meet
// at the CTA's barriers.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* abort,
                                          uint64_t budget_ns) {
  bool ok = *reinterpret_cast<volatile int32_t*>(abort) == 0 && wait_bar(bar, parity, budget_ns);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) *reinterpret_cast<volatile int32_t*>(abort) = 1;
  return ok;
}

// Reduce a position-times-frequency product to [-pi, pi] in fp32 with
// extra precision: the product is split into a rounded part and its exact
// error (fma), and 2*pi is subtracted in three pieces (Cody and Waite,
// "Software Manual for the Elementary Functions", 1980).  Valid for
// positions below 2^24 and frequencies <= 1.
__device__ __forceinline__ float reduce_angle(float pos, float f_hi, float f_lo) {
  const float ph = pos * f_hi;
  const float pe = fmaf(pos, f_hi, -ph);
  const float pl = pos * f_lo;
  const float k = rintf(ph * 0.15915494309189535f);
  // 2*pi = A + B + C, A with 8 significant bits so that k * A is exact
  constexpr float A = 6.28125f;
  constexpr float B = 1.9353071693331003e-03f;   // fp32(2*pi - A)
  constexpr float Cc = 1.0253376273028358e-11f;  // fp32(2*pi - A - B)
  float r = fmaf(-k, A, ph);
  r = fmaf(-k, B, r);
  r = fmaf(-k, Cc, r);
  return r + (pe + pl);
}

// Row metadata: row r = item * G + g; items 0..W-1 are ring slots, the
// rest beacons.  Returns the row's position, or INT32_MIN when the row is
// empty (ring slot never written, beacon past n_beacons, padding).
__device__ __forceinline__ int row_position(const ScoreParams& p, int u, int r, int nb,
                                            int32_t cur) {
  if (r >= p.NQ) return INT32_MIN;
  const int item = r / p.G;
  if (item < p.W) {
    // age of ring slot `item`: steps since it was written (slot_now = step % W)
    const int age = (p.slot_now - item + p.W) % p.W;
    if (age > p.step_cap) return INT32_MIN;  // never written (older than step 0)
    return cur - age;
  }
  return (item - p.W < nb) ? cur : INT32_MIN;
}

// The cos/sin table of the query build: entry (age, i) at
// age * (D/2 + 4) + (i % 8) * (D/16) + i / 8.  A warp of the build reads, for
// one k = i % 8, the D/16 consecutive entries of its rows' ages, and the
// padded row stride puts different ages on different banks.
__host__ __device__ constexpr int cs_stride(int D) { return D / 2 + 4; }
__host__ __device__ constexpr size_t cs_bytes(int W, int D) {
  return static_cast<size_t>(W > 0 ? W : 1) * cs_stride(D) * 8;
}

// Build the rotated, scaled, hi/lo-split query operand for rows
// [row0, row0 + nrows) in two K-major 128B-swizzled smem images.  Run by
// `nthr` threads with ids tid in [0, nthr); ends with named barrier `bar`.
// Loads the query rows of items idx0, idx0 + nthr, ... (kBatch of them) of
// build_queries: item = (row, group of 8 rotary pairs).  Rows past the
// recent and beacon slots load nothing (zeros).
template <int D, int kBatch>
__device__ __forceinline__ void load_query_batch(const ScoreParams& p, int u, int row0, int total,
                                                 int idx0, int nthr, uint4 (&va)[kBatch],
                                                 uint4 (&vb)[kBatch]) {
  constexpr int H = D / 2;
  constexpr int kGroups = H / 8;
#pragma unroll
  for (int t = 0; t < kBatch; ++t) {
    const int idx = idx0 + t * nthr;
    va[t] = vb[t] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < total) {
      const int rr = row0 + idx / kGroups, grp = idx % kGroups;
      const int item = rr / p.G, g = rr % p.G;
      if (item < p.W + p.M) {
        const uint16_t* src =
            item < p.W ? p.recent_q + ((static_cast<size_t>(u) * p.W + item) * p.G + g) * D
                       : p.beacons + ((static_cast<size_t>(u) * p.M + (item - p.W)) * p.G + g) * D;
        va[t] = *reinterpret_cast<const uint4*>(src + grp * 8);
        vb[t] = *reinterpret_cast<const uint4*>(src + H + grp * 8);
      }
    }
  }
}

// L1 prefetches of the addresses load_query_batch reads (no registers held).
template <int D, int kBatch>
__device__ __forceinline__ void prefetch_query_batch(const ScoreParams& p, int u, int row0,
                                                     int total, int idx0, int nthr) {
  constexpr int H = D / 2;
  constexpr int kGroups = H / 8;
#pragma unroll
  for (int t = 0; t < kBatch; ++t) {
    const int idx = idx0 + t * nthr;
    if (idx < total) {
      const int rr = row0 + idx / kGroups, grp = idx % kGroups;
      const int item = rr / p.G, g = rr % p.G;
      if (item < p.W + p.M) {
        const uint16_t* src =
            item < p.W ? p.recent_q + ((static_cast<size_t>(u) * p.W + item) * p.G + g) * D
                       : p.beacons + ((static_cast<size_t>(u) * p.M + (item - p.W)) * p.G + g) * D;
        asm volatile("prefetch.global.L1 [%0];" ::"l"(src + grp * 8));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(src + H + grp * 8));
      }
    }
  }
}

// cos/sin of every (age, frequency) of the query build; age 0 is the
// current position `cur`.  The positions are not written by the beacon
// selection.  A thread takes one frequency and a block of eight ages:
// sincosf at the block's first age, then seven rotations by -theta_i
// (cos/sin of theta_i from the host), each adding at most a couple of ulp.
// Consecutive threads take consecutive blocks of one frequency, so the lanes
// of a warp read the same few frequencies from the parameter space
// (different addresses in one warp would be served one after another).
template <int D>
__device__ __forceinline__ void build_cs_table(const ScoreParams& p, int32_t cur, float2* cs,
                                               int tid, int nthr) {
  constexpr int H = D / 2;
  const int nage = max(p.W, 1);
  const int nblk = (nage + 7) / 8;
  for (int idx = tid; idx < nblk * H; idx += nthr) {
    const int i = idx / nblk, a0 = (idx - i * nblk) * 8;
    const float ang = reduce_angle(static_cast<float>(cur - a0), p.freq_hi[i], p.freq_lo[i]);
    float s, c;
    sincosf(ang, &s, &c);
    const float c1 = p.step_cos[i], s1 = p.step_sin[i];
    float2* dst = cs + (i & 7) * (H / 8) + (i >> 3);
    const int a1 = min(a0 + 8, nage);
    for (int a = a0; a < a1; ++a) {
      dst[a * cs_stride(D)] = make_float2(c, s);
      const float cn = fmaf(c, c1, s * s1);  // angle of age a + 1: one step of theta_i less
      s = fmaf(s, c1, -(c * s1));
      c = cn;
    }
  }
}

// Rotate, scale and hi/lo-split the query items idx0, idx0 + nthr, ...
// (kBatch of them, as load_query_batch loaded them) and store them in the
// two K-major 128B-swizzled images of `nrows` rows.
template <int D, int kBatch>
__device__ __forceinline__ void store_query_batch(const ScoreParams& p, int nrows, int total,
                                                  int idx0, int nthr, const uint4 (&va)[kBatch],
                                                  const uint4 (&vb)[kBatch],
                                                  const int32_t* row_pos, const float2* cs,
                                                  int32_t cur, uint8_t* q_hi, uint8_t* q_lo) {
  constexpr int H = D / 2;
  constexpr int kGroups = H / 8;
#pragma unroll
  for (int t = 0; t < kBatch; ++t) {
    const int idx = idx0 + t * nthr;
    if (idx >= total) break;
    const int r = idx / kGroups, grp = idx % kGroups;
    const int32_t pos = row_pos[r];
    // rotated, scaled pairs, rounded to bf16 two at a time (hi), then the
    // exact remainders rounded likewise (lo); packed 32-bit words
    uint32_t hi0[4] = {0u, 0u, 0u, 0u}, hi1[4] = {0u, 0u, 0u, 0u};
    uint32_t lo0[4] = {0u, 0u, 0u, 0u}, lo1[4] = {0u, 0u, 0u, 0u};
    if (pos != INT32_MIN) {
      const float2* csa = cs + (cur - pos) * cs_stride(D) + grp;
      const uint32_t wa[4] = {va[t].x, va[t].y, va[t].z, va[t].w};
      const uint32_t wb[4] = {vb[t].x, vb[t].y, vb[t].z, vb[t].w};
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        float y0[2], y1[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 2 * k2 + e;  // pair grp * 8 + k
          const float2 csv = csa[k * (H / 8)];
          const float x0 = __uint_as_float(e ? (wa[k2] & 0xFFFF0000u) : (wa[k2] << 16));
          const float x1 = __uint_as_float(e ? (wb[k2] & 0xFFFF0000u) : (wb[k2] << 16));
          y0[e] = (x0 * csv.x - x1 * csv.y) * p.qscale;
          y1[e] = (x1 * csv.x + x0 * csv.y) * p.qscale;
        }
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(y0[0], y0[1]);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(y1[0], y1[1]);
        const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
        const __nv_bfloat162 l0 = __floats2bfloat162_rn(y0[0] - f0.x, y0[1] - f0.y);
        const __nv_bfloat162 l1 = __floats2bfloat162_rn(y1[0] - f1.x, y1[1] - f1.y);
        hi0[k2] = *reinterpret_cast<const uint32_t*>(&h0);
        hi1[k2] = *reinterpret_cast<const uint32_t*>(&h1);
        lo0[k2] = *reinterpret_cast<const uint32_t*>(&l0);
        lo1[k2] = *reinterpret_cast<const uint32_t*>(&l1);
      }
    }
    // 8 consecutive elements = one 16-byte chunk of the swizzled image
    const uint32_t o0 = sw128_offset(r, grp * 8, nrows);
    const uint32_t o1 = sw128_offset(r, H + grp * 8, nrows);
    *reinterpret_cast<uint4*>(q_hi + o0) = make_uint4(hi0[0], hi0[1], hi0[2], hi0[3]);
    *reinterpret_cast<uint4*>(q_hi + o1) = make_uint4(hi1[0], hi1[1], hi1[2], hi1[3]);
    *reinterpret_cast<uint4*>(q_lo + o0) = make_uint4(lo0[0], lo0[1], lo0[2], lo0[3]);
    *reinterpret_cast<uint4*>(q_lo + o1) = make_uint4(lo1[0], lo1[1], lo1[2], lo1[3]);
  }
}

template <int D>
__device__ void build_queries(const ScoreParams& p, int u, int row0, int nrows, uint8_t* q_hi,
                              uint8_t* q_lo, int32_t* row_pos, float2* cs, int tid, int nthr,
                              int bar) {
  constexpr int H = D / 2;
  // one thread per (row, pair of 8 consecutive rotary pairs), four items at
  // a time: all of a batch's global loads are issued before any is used.
  // Rows without an item (no beacon there) are loaded where the memory
  // exists and zeroed below.
  constexpr int kGroups = H / 8;
  constexpr int kBatch = 4;
  const int total = nrows * kGroups;
  uint4 va[kBatch], vb[kBatch];
  // The recent queries, beacons and beacon counts come from the previous
  // call (the beacon selection).  When the kernel has already waited for it
  // the first batch is prefetched into L1 at once, landing while the table
  // below is computed; inside a round the table is computed before the wait.
  const int32_t cur = p.cur_pos[u];
  if (!p.early_reads) prefetch_query_batch<D, kBatch>(p, u, row0, total, tid, nthr);
  build_cs_table<D>(p, cur, cs, tid, nthr);
  if (p.early_reads) pdl_wait();
  load_query_batch<D, kBatch>(p, u, row0, total, tid, nthr, va, vb);
  const int nb = p.M > 0 ? min(max(p.n_beacons[u], 0), p.M) : 0;
  for (int r = tid; r < nrows; r += nthr) row_pos[r] = row_position(p, u, row0 + r, nb, cur);
  named_sync(bar, nthr);
  for (int idx0 = tid; idx0 < total; idx0 += kBatch * nthr) {
    if (idx0 != tid) load_query_batch<D, kBatch>(p, u, row0, total, idx0, nthr, va, vb);
    store_query_batch<D, kBatch>(p, nrows, total, idx0, nthr, va, vb, row_pos, cs, cur, q_hi,
                                 q_lo);
  }
  fence_proxy_async_shared();  // generic smem writes -> visible to the tensor core
  named_sync(bar, nthr);
}

// Shared-memory arrays read with 16-byte vector loads follow this struct,
// so its size is a multiple of 16.
struct __align__(16) Barriers {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[4];   // accumulator buffers: 2 (split kernels, fused with 256 rows) or 4
  uint64_t tempty[4];
  uint64_t tmax_ready;  // fused kernel: the per-tile key-position maxima are in place
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t minpos;
  int32_t minrow;       // fused kernel: smallest key-position limit over the rows
};

static_assert(sizeof(Barriers) % 16 == 0, "arrays after the barriers need 16-byte alignment");

// The fused kernel keeps the largest key position of each of the first
// kTmaxTiles tiles in shared memory: a tile whose largest position is within
// every row's limit needs no causal mask and no per-key positions.
constexpr int kTmaxTiles = 512;

// Key tile range of split `s` for unit u.
__device__ __forceinline__ void split_tiles(const ScoreParams& p, int u, int s, int& t0, int& t1,
                                            int& L) {
  L = p.L[u];
  if (L < 0 || L > p.L_cap) {
    if (threadIdx.x == 0) record_error(p.ws, BKV_EDEVICE, kSiteScoreState);
    L = 0;
  }
  const int nt = (L + kTileKeys - 1) / kTileKeys;
  t0 = min(s * p.tiles_per_split, nt);
  t1 = min(t0 + p.tiles_per_split, nt);
}

__device__ __forceinline__ void init_barriers(Barriers* bars, int ns) {
  for (int i = 0; i < ns; ++i) {
    mbar_init(&bars->full[i], 1);
    mbar_init(&bars->empty[i], 1);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&bars->tfull[i], 1);
    mbar_init(&bars->tempty[i], 4);  // one arrival per epilogue warp
  }
  bars->abort_flag = 0;
  bars->minpos = INT32_MAX;
  fence_mbar_init();
}

// Before a TMA producer leaves: every tile load it issued has landed
// (bounded waits), so no copy into shared memory is still in flight when the
// CTA exits, even after another role gave up.  Only the last NS loads can
// still be pending: each earlier one was consumed before its stage was
// refilled.  On the normal path every phase has completed and this returns
// at once.
__device__ __forceinline__ void drain_loads(uint64_t* full, int NS, int issued, uint64_t budget) {
  for (int k = max(0, issued - NS); k < issued; ++k) wait_bar(&full[k % NS], (k / NS) & 1, budget);
}

// TMA producer (one elected lane of warp 0): stream the split's key tiles.
template <int D, int NS>
__device__ void produce_tiles(const ScoreParams& p, const CUtensorMap* kmap, Barriers* bars,
                              uint8_t* stages, int u, int t0, int ntl) {
  constexpr uint32_t kStageBytes = kTileKeys * D * 2;
  prefetch_tmap(kmap);
  int issued = 0;
  for (int i = 0; i < ntl; ++i) {
    const int st = i % NS;
    if (*reinterpret_cast<volatile int32_t*>(&bars->abort_flag) != 0 ||
        !wait_bar(&bars->empty[st], ((i / NS) & 1) ^ 1, p.wait_ns)) {
      bars->abort_flag = 1;
      record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
      break;
    }
    mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
    const int j0 = (t0 + i) * kTileKeys;
#pragma unroll
    for (int a = 0; a < D / 64; ++a)
      tma_load_3d(stages + st * kStageBytes + a * 16384, kmap, &bars->full[st], 64 * a, j0, u);
    issued = i + 1;
  }
  drain_loads(bars->full, NS, issued, p.wait_ns);
}

// --------------------------------------------------------------- pass 1
template <int D, int NS>
__global__ void __launch_bounds__(kThreads, 1)
    score_stats_kernel(const __grid_constant__ ScoreParams p,
                       const __grid_constant__ CUtensorMap kmap) {
  constexpr uint32_t kQBytes = 128 * D * 2;  // one 128-row operand image
  constexpr uint32_t kStageBytes = kTileKeys * D * 2;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, kTileKeys);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_hi = smem;
  uint8_t* q_lo = q_hi + kQBytes;
  uint8_t* stages = q_lo + kQBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(stages + NS * kStageBytes);
  int32_t* row_pos = reinterpret_cast<int32_t*>(bars + 1);  // [128]
  int32_t* kp = row_pos + 128;                              // [2][128] key positions
  float2* cs = reinterpret_cast<float2*>(kp + 256);         // [max(W,1)][D/2]

  const int s = blockIdx.x, rb = blockIdx.y, u = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t0, t1, L;
  split_tiles(p, u, s, t0, t1, L);
  const int ntl = t1 - t0;

  if (threadIdx.x == 0) init_barriers(bars, NS);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 2 * kTileKeys);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    if (elect_one()) produce_tiles<D, NS>(p, &kmap, bars, stages, u, t0, ntl);
  } else {
    build_queries<D>(p, u, rb * 128, 128, q_hi, q_lo, row_pos, cs, threadIdx.x - 32,
                     kThreads - 32, 1);
    if (warp == 1) {
      // ---------------- MMA issuer: D[row][key] = sum_k Q[row][k] K[key][k]
      int last = -1;
      for (int i = 0; i < (p.stall ? 0 : ntl); ++i) {
        const int st = i % NS, b = i & 1;
        if (!warp_wait(&bars->full[st], (i / NS) & 1, &bars->abort_flag, p.wait_ns) ||
            !warp_wait(&bars->tempty[b], ((i >> 1) & 1) ^ 1, &bars->abort_flag, p.wait_ns)) {
          if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t dt = tbase + b * kTileKeys;
          const uint32_t kbase = smem_u32(stages + st * kStageBytes);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t qbase = smem_u32(part ? q_lo : q_hi);
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(dt, sdesc_sw128(qbase + a * 16384 + kk * 32),
                         sdesc_sw128(kbase + a * 16384 + kk * 32), kIdesc,
                         (part | a | kk) != 0);
          }
          mma_commit(&bars->empty[st]);
          mma_commit(&bars->tfull[b]);
        }
        __syncwarp();
        last = i;
      }
      // the MMAs have completed before TMEM is released, even if the
      // epilogue gave up on them
      if (last >= 0) wait_bar(&bars->tfull[last & 1], (last >> 1) & 1, p.wait_ns);
    } else {
      // ---------------- epilogue: thread = one row; running max / sum of exp2
      const int q = warp & 3;
      const int et = threadIdx.x - 64;  // 0..127
      const int lrow = q * 32 + lane;   // TMEM lane = row within the block
      const int32_t rpos = row_pos[lrow];
      const int32_t lim = (p.causal || rpos == INT32_MIN) ? rpos : INT32_MAX - 1;
      float m = -INFINITY, z = 0.f;
      // key positions of the tiles, one tile ahead, in two buffers (the
      // barrier of tile i + 1 keeps tile i + 2 from rewriting tile i's)
      const int32_t* kpu = p.kpos + static_cast<size_t>(u) * p.L_cap;
      int32_t kp_next = (t0 * kTileKeys + et) < L && ntl > 0 ? kpu[t0 * kTileKeys + et] : INT32_MAX;
      for (int i = 0; i < ntl; ++i) {
        const int b = i & 1;
        int32_t* kpb = kp + (i & 1) * 128;
        kpb[et] = kp_next;
        const int jn = (t0 + i + 1) * kTileKeys + et;
        kp_next = (i + 1 < ntl && jn < L) ? kpu[jn] : INT32_MAX;
        named_sync(2, kEpiThreads);
        if (warp_wait(&bars->tfull[b], (i >> 1) & 1, &bars->abort_flag, p.wait_ns)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kTileKeys / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + (static_cast<uint32_t>(q * 32) << 16) + b * kTileKeys + c * 32, v);
            tmem_wait_ld();
            if (c == kTileKeys / 32 - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->tempty[b]);
            }
            const int4* kp4 = reinterpret_cast<const int4*>(kpb + c * 32);
            float t[32];
            float mx = -INFINITY;
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
              const int4 kk = kp4[k4];
              const int kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = k4 * 4 + e;
                t[k] = (kv[e] <= lim) ? __uint_as_float(v[k]) : -INFINITY;
                mx = fmaxf(mx, t[k]);
              }
            }
            const float mn = fmaxf(m, mx);
            if (mn != -INFINITY) {
              float acc = (m == -INFINITY) ? 0.f : z * ex2(m - mn);
#pragma unroll
              for (int k = 0; k < 32; ++k) acc += ex2(t[k] - mn);
              z = acc;
              m = mn;
            }
          }
        } else if (lane == 0) {
          record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
        }
      }
      const int row = rb * 128 + lrow;
      p.part[(static_cast<size_t>(u) * p.nsplit + s) * p.nrows_part + row] = make_float2(m, z);
      // several row groups combine through atomics in pass 2: start from 0
      if (p.ngrp > 1 && rb == 0)
        for (int jj = t0 * kTileKeys + et; jj < min(t1 * kTileKeys, L); jj += kEpiThreads)
          p.scores[static_cast<size_t>(u) * p.L_cap + jj] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 2 * kTileKeys);
}

// --------------------------------------------------------------- pass 2
template <int D, int NS, int NMAX, bool kMax>
__global__ void __launch_bounds__(kThreads, 1)
    score_final_kernel(const __grid_constant__ ScoreParams p,
                       const __grid_constant__ CUtensorMap kmap) {
  constexpr uint32_t kStageBytes = kTileKeys * D * 2;
  constexpr uint32_t kCols = NMAX <= 128 ? 256 : 512;  // two accumulator buffers
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int s = blockIdx.x, grp = blockIdx.y, u = blockIdx.z;
  const int row0 = grp * 256;
  const int N = min(256, p.NQ16 - row0);  // rows of this group, a multiple of 16
  uint8_t* q_hi = smem;
  uint8_t* q_lo = q_hi + NMAX * D * 2;
  uint8_t* stages = q_lo + NMAX * D * 2;
  Barriers* bars = reinterpret_cast<Barriers*>(stages + NS * kStageBytes);
  int32_t* row_pos = reinterpret_cast<int32_t*>(bars + 1);  // [256]
  float* lse = reinterpret_cast<float*>(row_pos + 256);      // [256]
  float2* cs = reinterpret_cast<float2*>(lse + 256);         // [max(W,1)][D/2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t0, t1, L;
  split_tiles(p, u, s, t0, t1, L);
  const int ntl = t1 - t0;

  if (threadIdx.x == 0) init_barriers(bars, NS);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    if (elect_one()) produce_tiles<D, NS>(p, &kmap, bars, stages, u, t0, ntl);
  } else {
    const int tid = threadIdx.x - 32, nthr = kThreads - 32;
    build_queries<D>(p, u, row0, N, q_hi, q_lo, row_pos, cs, tid, nthr, 1);
    // merge the per-split (max, sum) of each row into its log2-sum-exp
    for (int r = tid; r < N; r += nthr) {
      const int row = row0 + r;
      float l = INFINITY;  // empty rows: every probability is 0
      if (row_pos[r] != INT32_MIN) {
        const float2* pr = p.part + static_cast<size_t>(u) * p.nsplit * p.nrows_part + row;
        float mm = -INFINITY;
        for (int k = 0; k < p.nsplit; ++k)
          mm = fmaxf(mm, pr[static_cast<size_t>(k) * p.nrows_part].x);
        float zz = 0.f;
        if (mm != -INFINITY)
          for (int k = 0; k < p.nsplit; ++k) {
            const float2 mz = pr[static_cast<size_t>(k) * p.nrows_part];
            if (mz.x != -INFINITY) zz += mz.y * ex2(mz.x - mm);
          }
        if (zz > 0.f) l = mm + lg2(zz);
        atomicMin(&bars->minpos, row_pos[r]);
        if (!p.causal) row_pos[r] = INT32_MAX;
      }
      lse[r] = l;
    }
    named_sync(1, nthr);
    if (warp == 1) {
      // ---------------- MMA issuer: D[key][row] = sum_k K[key][k] Q[row][k]
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(N));
      int last = -1;
      for (int i = 0; i < (p.stall ? 0 : ntl); ++i) {
        const int st = i % NS, b = i & 1;
        if (!warp_wait(&bars->full[st], (i / NS) & 1, &bars->abort_flag, p.wait_ns) ||
            !warp_wait(&bars->tempty[b], ((i >> 1) & 1) ^ 1, &bars->abort_flag, p.wait_ns)) {
          if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t dt = tbase + b * (kCols / 2);
          const uint32_t kbase = smem_u32(stages + st * kStageBytes);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t qbase = smem_u32(part ? q_lo : q_hi);
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(dt, sdesc_sw128(kbase + a * 16384 + kk * 32),
                         sdesc_sw128(qbase + a * (N * 128) + kk * 32), idesc,
                         (part | a | kk) != 0);
          }
          mma_commit(&bars->empty[st]);
          mma_commit(&bars->tfull[b]);
        }
        __syncwarp();
        last = i;
      }
      if (last >= 0) wait_bar(&bars->tfull[last & 1], (last >> 1) & 1, p.wait_ns);
    } else {
      // ---------------- epilogue: thread = one key
      const int q = warp & 3;
      const int32_t minpos = bars->minpos;
      const int nb = p.M > 0 ? min(max(p.n_beacons[u], 0), p.M) : 0;
      const int nrec = p.step + 1 < p.W ? static_cast<int>(p.step + 1) : p.W;
      const float inv_rows = 1.f / static_cast<float>(max((nrec + nb) * p.G, 1));
      const int nchunks = (N + 31) / 32;
      const int32_t* kpu = p.kpos + static_cast<size_t>(u) * p.L_cap;
      // this key's position, fetched one tile ahead
      int32_t kp_ahead = INT32_MAX;
      {
        const int j0 = t0 * kTileKeys + q * 32 + lane;
        if (ntl > 0 && j0 < L) kp_ahead = kpu[j0];
      }
      for (int i = 0; i < ntl; ++i) {
        const int b = i & 1;
        const int j = (t0 + i) * kTileKeys + q * 32 + lane;
        const int32_t kpj = kp_ahead;
        kp_ahead = (i + 1 < ntl && j + kTileKeys < L) ? kpu[j + kTileKeys] : INT32_MAX;
        if (!warp_wait(&bars->tfull[b], (i >> 1) & 1, &bars->abort_flag, p.wait_ns)) {
          if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
          continue;
        }
        tc_fence_after();
        const bool nomask = __all_sync(0xffffffffu, kpj <= minpos);
        float best = -INFINITY, acc = 0.f;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + (static_cast<uint32_t>(q * 32) << 16) + b * (kCols / 2) + c * 32, v);
          tmem_wait_ld();
          if (c == nchunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[b]);
          }
          const int nv = min(32, N - c * 32);
          const float4* l4 = reinterpret_cast<const float4*>(lse + c * 32);
          const int4* p4 = reinterpret_cast<const int4*>(row_pos + c * 32);
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            if (k4 * 4 < nv) {
              const float4 lv = l4[k4];
              const int4 pv = p4[k4];
              const float ll[4] = {lv.x, lv.y, lv.z, lv.w};
              const int pp[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float x = __uint_as_float(v[k4 * 4 + e]) - ll[e];
                if (!nomask && kpj > pp[e]) x = -INFINITY;
                if constexpr (kMax)
                  best = fmaxf(best, x);
                else
                  acc += ex2(x);
              }
            }
          }
        }
        if (j < L) {
          float* dst = p.scores + static_cast<size_t>(u) * p.L_cap + j;
          if constexpr (kMax) {
            const float sc = best == -INFINITY ? 0.f : ex2(best);
            if (p.ngrp > 1)
              atomicMax(reinterpret_cast<int*>(dst), __float_as_int(sc));
            else
              *dst = sc;
          } else {
            const float sc = acc * inv_rows;
            if (p.ngrp > 1)
              atomicAdd(dst, sc);
            else
              *dst = sc;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kCols);
}

// --------------------------------------------------------------- fused
// Both passes in one CTA for a unit's rows (or a group of 256 of them): the
// queries are rotated once, pass 1 runs over every key tile of the unit,
// each row's log2-sum-exp is formed locally (no partials, no second
// launch), and pass 2 streams the same tiles again through TMA (a unit's
// keys are then usually still in L2).  NR = 128-row blocks of the query
// image (1 or 2).  score_fused_kernel (below) runs it persistently; its
// epilogue is fused_epilogue.  The cluster kernel uses the thread count
// and epilogue width here.
constexpr int kFusedThreads = 320;
constexpr int kFusedEpi = 256;

// Arrival of one of the four warps of a half on a TMEM-empty barrier that
// counts eight: each warp stands for two.
__device__ __forceinline__ void arrive_tempty(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], 2;" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier of one half of the epilogue (named barriers 3 and 4, 128 threads).
__device__ __forceinline__ void half_sync(int h) {
  if (h == 0)
    named_sync(3, 128);
  else
    named_sync(4, 128);
}

// Running max and sum of exp2 of one row over 64 keys (TMEM words).
__device__ __forceinline__ void row_update(float& m, float& z, const uint32_t (&v)[64]) {
  float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
  for (int k = 0; k < 64; k += 4) {
    mx0 = fmaxf(mx0, __uint_as_float(v[k]));
    mx1 = fmaxf(mx1, __uint_as_float(v[k + 1]));
    mx2 = fmaxf(mx2, __uint_as_float(v[k + 2]));
    mx3 = fmaxf(mx3, __uint_as_float(v[k + 3]));
  }
  const float mn = fmaxf(m, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)));
  if (mn != -INFINITY) {
    float a0 = (m == -INFINITY) ? 0.f : z * ex2(m - mn);
    float a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int k = 0; k < 64; k += 4) {
      a0 += ex2(__uint_as_float(v[k]) - mn);
      a1 += ex2(__uint_as_float(v[k + 1]) - mn);
      a2 += ex2(__uint_as_float(v[k + 2]) - mn);
      a3 += ex2(__uint_as_float(v[k + 3]) - mn);
    }
    z = (a0 + a1) + (a2 + a3);
    m = mn;
  }
}

// Barriers and per-unit hand-offs of the persistent two-pass kernel; what
// crosses from one unit to the next is double-buffered by unit parity.
struct __align__(16) FusedBars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[4];   // accumulator buffers: 4 (128 rows) or 2 (256 rows)
  uint64_t tempty[4];
  uint64_t qfull[2];   // a unit's query image is in place (its two builders)
  uint64_t qempty;     // the MMAs of a unit are done with the query image
  uint64_t tready[2];  // a unit's per-tile key-position maxima are in place
  uint64_t edone[2];   // the epilogue is done with a unit (8 warps)
  uint64_t bready[2];  // a unit's cos/sin table and row positions are in place
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t minrow[2];   // smallest key-position limit over a unit's live rows
  int32_t minpos[2];   // smallest position over a unit's live rows
  int32_t cur[2];      // a unit's current position
  int32_t pad[2];
};
static_assert(sizeof(FusedBars) % 16 == 0, "arrays after the barriers need 16-byte alignment");

// Warp 0 TMA, warp 1 MMA, warps 2-3 query build of the next unit, warps
// 4-11 epilogue.
constexpr int kPersistThreads = 384;

// One warp: the smallest key-position limit and the smallest position over
// the live rows of a unit's query build, then `count` arrivals on `bar`.
__device__ __forceinline__ void publish_rows(const ScoreParams& p, const int32_t* rp, int nrows,
                                             FusedBars* bars, int b, uint64_t* bar,
                                             uint32_t count) {
  const int lane = threadIdx.x & 31;
  int32_t lw = INT32_MAX, pw = INT32_MAX;
  for (int r = lane; r < nrows; r += 32) {
    const int32_t v = rp[r];
    if (v != INT32_MIN) {
      lw = min(lw, p.causal ? v : INT32_MAX - 1);
      pw = min(pw, v);
    }
  }
  lw = __reduce_min_sync(0xffffffffu, lw);
  pw = __reduce_min_sync(0xffffffffu, pw);
  if (lane == 0) {
    bars->minrow[b] = lw;
    bars->minpos[b] = pw;
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
  }
  __syncwarp();
}

// The query build of a unit after the first is shared: the builder warps
// take items [0, kBuildSplit * total) as soon as the MMAs of the previous
// unit are done with the image, the epilogue the rest once it has finished
// the previous unit.
constexpr int kBuildSplitNum = 3, kBuildSplitDen = 8;

// Work item n of CTA b in the persistent two-pass kernel: row group n % ngrp
// (kRows rows from row0) of unit b + (n / ngrp) * G.  More scoring rows than
// one CTA's operand holds are scored in groups one after another, all groups
// of a unit in the same CTA.
struct SubUnit {
  int u, grp, row0;
  int nq16;  // rows of the group, rounded up to 16 (the pass-2 MMA's N)
  int nblk;  // 128-row blocks of the group that hold rows (pass 1)
};
__device__ __forceinline__ SubUnit sub_unit(const ScoreParams& p, int n, int G, int kRows,
                                            int ngrp) {
  SubUnit w;
  w.u = blockIdx.x + (n / ngrp) * G;
  w.grp = n % ngrp;
  w.row0 = w.grp * kRows;
  const int nr = min(kRows, p.NQ16 - w.row0);
  w.nq16 = nr;
  w.nblk = (nr + 127) / 128;
  return w;
}

// Epilogue of one unit (warps 4..11).  Iteration i of the unit (tile i in
// pass 1, tile i - nt in pass 2) is the kernel's iteration g0 + i: it uses
// accumulator (g0 + i) % kNBuf and is taken by half (g0 + i) % 2, so each
// half owns every other accumulator.  kMax: max aggregation (else the
// mean), a template parameter so that the per-element loops carry no branch
// on it.
template <int D, int NR, uint32_t kBufCols, int kNBuf, bool kMax>
__device__ __forceinline__ void fused_epilogue(const ScoreParams& p, int u, int nt, int L, int g0,
                                               uint32_t tbase, FusedBars* bars, int32_t* row_pos,
                                               float* lse, float2* mz, int32_t* kp,
                                               const int32_t* tmax, int32_t minrow,
                                               int32_t minpos, int nq16, int nblk, int grp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                      // TMEM lane quarter
  const int h = (warp - 4) >> 2;               // half: 0 = warps 4..7, 1 = warps 8..11
  const int ht = (threadIdx.x - 128) & 127;    // thread within the half
  const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
  auto acc_of = [&](int g) { return tbase + lane_addr + (g % kNBuf) * kBufCols; };
  const int32_t* kpu = p.kpos + static_cast<size_t>(u) * p.L_cap;
  int32_t* kph = kp + h * 128;                 // this half's staged key positions

  // ---- pass 1: thread = row (of each row block) over all keys of its
  // half's tiles; running max and sum of exp2
  float m[NR], z[NR];
  int32_t lim[NR];
#pragma unroll
  for (int blk = 0; blk < NR; ++blk) {
    const int32_t rp = row_pos[blk * 128 + q * 32 + lane];
    lim[blk] = (p.causal || rp == INT32_MIN) ? rp : INT32_MAX - 1;
    m[blk] = -INFINITY;
    z[blk] = 0.f;
  }
  // A tile whose largest key position is within every live row's limit (and
  // that has no key past L) needs no mask; for another tile the half stages
  // its key positions in shared memory between two barriers of the half.
  for (int i = (h - g0) & 1; i < nt; i += 2) {
    const int g = g0 + i;
    const bool masked = !(i < kTmaxTiles && tmax[i] <= minrow);  // uniform
    if (masked) {
      half_sync(h);  // the half is done with its previous staged tile
      const int j = i * kTileKeys + ht;
      kph[ht] = j < L ? kpu[j] : INT32_MAX;
      half_sync(h);
    }
    if (warp_wait(&bars->tfull[g % kNBuf], (g / kNBuf) & 1, &bars->abort_flag, p.wait_ns)) {
      tc_fence_after();
      const uint32_t buf = acc_of(g);
#pragma unroll
      for (int blk = 0; blk < NR; ++blk)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (blk >= nblk) continue;  // a row block of the group without rows
          uint32_t v[64];  // keys 64 c .. 64 c + 63 of the tile
          const uint32_t col = buf + blk * 128 + c * 64;
          tmem_ld32(col, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          tmem_ld32(col + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tmem_wait_ld();
          if (blk == nblk - 1 && c == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_tempty(&bars->tempty[g % kNBuf]);
          }
          if (masked) {
            const int lm = lim[blk];
            const int* kh = kph + 64 * c;
#pragma unroll
            for (int k = 0; k < 64; ++k)
              v[k] = kh[k] > lm ? __float_as_uint(-INFINITY) : v[k];
          }
          row_update(m[blk], z[blk], v);
        }
    } else if (lane == 0) {
      record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
    }
  }
  // merge the two halves of every row into its log2-sum-exp (empty rows:
  // every probability is 0)
#pragma unroll
  for (int blk = 0; blk < NR; ++blk)
    if (h == 1) mz[blk * 128 + q * 32 + lane] = make_float2(m[blk], z[blk]);
  named_sync(2, kFusedEpi);
  if (h == 0) {
#pragma unroll
    for (int blk = 0; blk < NR; ++blk) {
      const int r = blk * 128 + q * 32 + lane;
      const int32_t rp = row_pos[r];
      const float2 o = mz[r];
      const float mm = fmaxf(m[blk], o.x);
      float l = INFINITY;
      if (rp != INT32_MIN) {
        float zz = 0.f;
        if (mm != -INFINITY) {
          if (m[blk] != -INFINITY) zz += z[blk] * ex2(m[blk] - mm);
          if (o.x != -INFINITY) zz += o.y * ex2(o.x - mm);
        }
        if (zz > 0.f) l = mm + lg2(zz);
        if (!p.causal) row_pos[r] = INT32_MAX;
      }
      lse[r] = l;
    }
  }
  named_sync(2, kFusedEpi);

  // ---- pass 2: thread = key q * 32 + lane of its half's tiles, over every
  // row; max (or mean) of exp2(s - lse), written directly
  const int nb = p.M > 0 ? min(max(p.n_beacons[u], 0), p.M) : 0;
  const int nrec = p.step + 1 < p.W ? static_cast<int>(p.step + 1) : p.W;
  const float inv_rows = 1.f / static_cast<float>(max((nrec + nb) * p.G, 1));
  const int N = nq16;
  const int nchunks = (N + 31) / 32;
  constexpr bool is_max = kMax;
  const int key = q * 32 + lane;
  for (int i = nt + ((h - g0 - nt) & 1); i < 2 * nt; i += 2) {
    const int g = g0 + i;
    const int ti = i - nt;
    const int j = ti * kTileKeys + key;
    // a tile whose largest key position is at most every row's position
    // (and that has no key past L) needs no mask and no per-key position
    const bool tile_open = ti < kTmaxTiles && tmax[ti] <= minpos;
    const int32_t kpj = tile_open ? INT32_MIN : (j < L ? kpu[j] : INT32_MAX);
    float r0 = -INFINITY, r1 = -INFINITY, r2 = -INFINITY, r3 = -INFINITY;  // max
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;                          // mean
    if (warp_wait(&bars->tfull[g % kNBuf], (g / kNBuf) & 1, &bars->abort_flag, p.wait_ns)) {
      tc_fence_after();
      const uint32_t buf = acc_of(g);
      const bool nomask = tile_open || __all_sync(0xffffffffu, kpj <= minpos);
      const int32_t kpm = nomask ? INT32_MIN : kpj;
      // chunks of 32 rows in pairs: both TMEM loads issued before one wait
#pragma unroll 1
      for (int c = 0; c < nchunks; c += 2) {
        const bool two = c + 1 < nchunks;
        uint32_t v[64];
        const uint32_t col = buf + c * 32;
        tmem_ld32(col, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        if (two) tmem_ld32(col + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_wait_ld();
        if (c + 2 >= nchunks) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_tempty(&bars->tempty[g % kNBuf]);
        }
        const int nv = min(two ? 64 : 32, N - c * 32);  // valid rows here (multiple of 16)
        const float4* l4 = reinterpret_cast<const float4*>(lse + c * 32);
        const int4* p4 = reinterpret_cast<const int4*>(row_pos + c * 32);
        if (is_max && nomask && nv == 64) {
          // every row of these 64 sees this key: no positions, no selects
#pragma unroll
          for (int k4 = 0; k4 < 16; ++k4) {
            const float4 lv = l4[k4];
            r0 = fmaxf(r0, __uint_as_float(v[k4 * 4 + 0]) - lv.x);
            r1 = fmaxf(r1, __uint_as_float(v[k4 * 4 + 1]) - lv.y);
            r2 = fmaxf(r2, __uint_as_float(v[k4 * 4 + 2]) - lv.z);
            r3 = fmaxf(r3, __uint_as_float(v[k4 * 4 + 3]) - lv.w);
          }
          continue;
        }
        // No branch per group of four rows: rows past nv read whatever lies
        // past them in shared memory (lse and row_pos are followed by other
        // arrays of the kernel) and are discarded by the selects.
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4) {
          const bool ok = k4 * 4 < nv;
          const float4 lv = l4[k4];
          const int4 pv = p4[k4];
          float x0 = __uint_as_float(v[k4 * 4 + 0]) - lv.x;
          float x1 = __uint_as_float(v[k4 * 4 + 1]) - lv.y;
          float x2 = __uint_as_float(v[k4 * 4 + 2]) - lv.z;
          float x3 = __uint_as_float(v[k4 * 4 + 3]) - lv.w;
          x0 = (ok && kpm <= pv.x) ? x0 : -INFINITY;
          x1 = (ok && kpm <= pv.y) ? x1 : -INFINITY;
          x2 = (ok && kpm <= pv.z) ? x2 : -INFINITY;
          x3 = (ok && kpm <= pv.w) ? x3 : -INFINITY;
          if constexpr (is_max) {
            r0 = fmaxf(r0, x0);
            r1 = fmaxf(r1, x1);
            r2 = fmaxf(r2, x2);
            r3 = fmaxf(r3, x3);
          } else {
            s0 += ex2(x0);
            s1 += ex2(x1);
            s2 += ex2(x2);
            s3 += ex2(x3);
          }
        }
      }
    } else if (lane == 0) {
      record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
    }
    if (j < L) {
      // the groups of a unit run one after another in this CTA (with the
      // epilogue's barriers between them): later groups fold into the score
      const float all = is_max ? fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)) : (s0 + s1) + (s2 + s3);
      const float sc = is_max ? (all == -INFINITY ? 0.f : ex2(all)) : all * inv_rows;
      float* dst = p.scores + static_cast<size_t>(u) * p.L_cap + j;
      *dst = grp == 0 ? sc : (is_max ? fmaxf(*dst, sc) : *dst + sc);
    }
  }
}

// Both passes in one persistent kernel: CTA b scores units b, b + G, b + 2G,
// ... (G = gridDim.x, at most one CTA per SM), and its roles overlap
// consecutive units: the key tiles of the next unit load while the current
// one finishes, and the next query operand is built as soon as the MMAs of
// the current one are done with the single query image.
//   warp 0      TMA: per unit, the largest key position of each tile, then
//               every tile twice (pass 1, then pass 2) through the ring;
//   warp 1      MMA: pass 1 D[row][key] = Q . K (rows on the TMEM lanes),
//               pass 2 D[key][row] = K . Q (keys on the lanes);
//   warps 2-3   query build of the next unit (all warps but the TMA warp
//               build the first unit's together);
//   warps 4-11  epilogue (fused_epilogue).
template <int D, int NS, int NR, bool kMax>
__global__ void __launch_bounds__(kPersistThreads, 1)
    score_fused_kernel(const __grid_constant__ ScoreParams p,
                       const __grid_constant__ CUtensorMap kmap) {
  pdl_trigger();  // select + compact may set up; it waits for this grid before reading it
  // Launched as a programmatic dependent: wait for the previous kernel before
  // reading anything, unless that kernel is known to be the beacon selection
  // (then only its outputs -- beacons, their counts, the recent ring -- wait,
  // in the query build).
  if (!p.early_reads) pdl_wait();
  constexpr int kRows = NR * 128;
  constexpr uint32_t kQBytes = kRows * D * 2;  // one query image (hi or lo)
  constexpr uint32_t kStageBytes = kTileKeys * D * 2;
  constexpr uint32_t kBufCols = NR == 1 ? 128 : 256;  // TMEM columns per accumulator
  // accumulators in TMEM: four of 128 columns (128 rows) or two of 256, so
  // that the MMAs of a tile can run while the epilogue still reads earlier
  // ones (each half of the epilogue owns every other accumulator)
  constexpr int kNBuf = NR == 1 ? 4 : 2;
  constexpr uint32_t kCols = kNBuf * kBufCols;
  constexpr uint32_t kIdesc1 = idesc_bf16_f32(128, kTileKeys);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_hi = smem;
  uint8_t* q_lo = q_hi + kQBytes;
  uint8_t* stages = q_lo + kQBytes;
  FusedBars* bars = reinterpret_cast<FusedBars*>(stages + NS * kStageBytes);
  int32_t* row_pos = reinterpret_cast<int32_t*>(bars + 1);  // [2][kRows], by unit parity
  float* lse = reinterpret_cast<float*>(row_pos + 2 * kRows);  // [kRows]
  float2* mz = reinterpret_cast<float2*>(lse + kRows);         // [kRows] second half's (m, z)
  int32_t* kp = reinterpret_cast<int32_t*>(mz + kRows);        // [2][128] pass-1 key positions
  float2* cs = reinterpret_cast<float2*>(kp + 256);            // [max(W,1)][D/2 + 4]
  int32_t* tmax = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(cs) + cs_bytes(p.W, D));  // [2][kTmaxTiles]

  const int G = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < kNBuf; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 8);  // two per warp of the owning half
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->qfull[b], 2);  // the builders' part and the epilogue's part
      mbar_init(&bars->tready[b], 1);
      mbar_init(&bars->edone[b], 8);  // one per epilogue warp
      mbar_init(&bars->bready[b], 1);
    }
    mbar_init(&bars->qempty, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  // row groups per unit (more rows than one operand holds)
  const int ngrp = (p.NQ16 + kRows - 1) / kRows;
  // the first work item's query operand: every warp but the TMA warp
  if (warp >= 1) {
    build_queries<D>(p, blockIdx.x, 0, kRows, q_hi, q_lo, row_pos, cs, threadIdx.x - 32,
                     kPersistThreads - 32, 1);
    if (warp == 2) {
      publish_rows(p, row_pos, kRows, bars, 0, &bars->qfull[0], 2);
      // unit 0 takes phase 0 of bready[0] too, so that unit n waits for
      // phase n / 2 of bready[n % 2]
      if (lane == 0) mbar_arrive(&bars->bready[0]);
    }
  }

  if (warp == 0) {
    // ---------------- TMA producer.  (An L2 run-ahead of bulk prefetches
    // measured slower and, on long caches, re-read tiles from HBM.)
    if (lane == 0) prefetch_tmap(&kmap);
    int g = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const SubUnit w = sub_unit(p, n, G, kRows, ngrp);
      const int u = w.u;
      if (u >= p.U) break;
      int t0, t1, L;
      split_tiles(p, u, 0, t0, t1, L);  // tiles_per_split covers the whole cache here
      const int nt = t1 - t0;
      // the epilogue is done with the tile maxima of two units back
      if (n >= 2 &&
          !warp_wait(&bars->edone[n & 1], ((n - 2) >> 1) & 1, &bars->abort_flag, p.wait_ns)) {
        if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
        break;
      }
      // Largest key position of every tile (keys past L count as
      // unbounded).  Lane l reads keys 4l .. 4l + 3 of a tile with one
      // 16-byte load (the address clamped into the row; clamped loads only
      // cover keys past L), so sixteen tiles' loads are in flight before any
      // is reduced.  Rows that are not 16-byte aligned take element loads.
      {
        int32_t* tm = tmax + (n & 1) * kTmaxTiles;
        const int32_t* kpu = p.kpos + static_cast<size_t>(u) * p.L_cap;
        const bool vec = (reinterpret_cast<uintptr_t>(p.kpos) & 15u) == 0 &&
                         (p.L_cap & 3) == 0 && p.L_cap >= 4;
        const int ntm = min(nt, kTmaxTiles);
        for (int ta = 0; ta < ntm; ta += 16) {
          int32_t mx[16];
          if (vec) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int j = (ta + k) * kTileKeys + 4 * lane;
              const int4 v = *reinterpret_cast<const int4*>(kpu + min(j, p.L_cap - 4));
              mx[k] = max(max(j < L ? v.x : INT32_MAX, j + 1 < L ? v.y : INT32_MAX),
                          max(j + 2 < L ? v.z : INT32_MAX, j + 3 < L ? v.w : INT32_MAX));
            }
          } else {
#pragma unroll 1
            for (int k = 0; k < 16; ++k) {
              const int j = (ta + k) * kTileKeys + 4 * lane;
              int32_t m = INT32_MIN;
              for (int e = 0; e < 4; ++e) m = max(m, j + e < L ? kpu[j + e] : INT32_MAX);
              mx[k] = m;
            }
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int32_t r = __reduce_max_sync(0xffffffffu, mx[k]);
            if (lane == 0 && ta + k < ntm) tm[ta + k] = r;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tready[n & 1]);
      }
      // every tile twice: iteration i loads tile i % nt
      if (lane == 0) {
        for (int i = 0; i < 2 * nt; ++i, ++g) {
          const int st = g % NS;
          if (*reinterpret_cast<volatile int32_t*>(&bars->abort_flag) != 0 ||
              !wait_bar(&bars->empty[st], ((g / NS) & 1) ^ 1, p.wait_ns)) {
            bars->abort_flag = 1;
            record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->full[st], kStageBytes);
          const int j0 = (i % nt) * kTileKeys;
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(stages + st * kStageBytes + a * 16384, &kmap, &bars->full[st], 64 * a,
                        j0, u);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      g = __shfl_sync(0xffffffffu, g, 0);
    }
    // every load has landed before the CTA can leave (bounded)
    if (lane == 0) drain_loads(bars->full, NS, g, p.wait_ns);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    int g = 0, commits = 0;
    bool ok = true;
    for (int n = 0; !p.stall && ok; ++n) {
      const SubUnit w = sub_unit(p, n, G, kRows, ngrp);
      const int u = w.u;
      if (u >= p.U) break;
      const uint32_t idesc2 = idesc_bf16_f32(128, static_cast<uint32_t>(w.nq16));
      int t0, t1, L;
      split_tiles(p, u, 0, t0, t1, L);
      const int nt = t1 - t0;
      ok = warp_wait(&bars->qfull[n & 1], (n >> 1) & 1, &bars->abort_flag, p.wait_ns);
      tc_fence_after();
      for (int i = 0; i < 2 * nt && ok; ++i, ++g) {
        const int st = g % NS, b = g % kNBuf;
        ok = warp_wait(&bars->full[st], (g / NS) & 1, &bars->abort_flag, p.wait_ns) &&
             warp_wait(&bars->tempty[b], ((g / kNBuf) & 1) ^ 1, &bars->abort_flag, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t dt = tbase + b * kBufCols;
          const uint32_t kbase = smem_u32(stages + st * kStageBytes);
          if (i < nt) {
            // pass 1: D[row][key] = Q[row] . K[key], one M = 128 block per row
            // block that holds rows
#pragma unroll
            for (int blk = 0; blk < NR; ++blk)
#pragma unroll
              for (int part2 = 0; part2 < 2; ++part2) {
                if (blk >= w.nblk) continue;
                const uint32_t qbase = smem_u32(part2 ? q_lo : q_hi) + blk * 128 * 128;
#pragma unroll
                for (int a = 0; a < D / 64; ++a)
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(dt + blk * 128, sdesc_sw128(qbase + a * (kRows * 128) + kk * 32),
                             sdesc_sw128(kbase + a * 16384 + kk * 32), kIdesc1,
                             (part2 | a | kk) != 0);
              }
          } else {
            // pass 2: D[key][row] = K[key] . Q[row], N = NQ16 rows
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2) {
              const uint32_t qbase = smem_u32(part2 ? q_lo : q_hi);
#pragma unroll
              for (int a = 0; a < D / 64; ++a)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16(dt, sdesc_sw128(kbase + a * 16384 + kk * 32),
                           sdesc_sw128(qbase + a * (kRows * 128) + kk * 32), idesc2,
                           (part2 | a | kk) != 0);
            }
          }
          mma_commit(&bars->empty[st]);
          mma_commit(&bars->tfull[b]);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
      // the query image is free once this unit's MMAs have finished (a
      // commit even after a failed wait: it covers every MMA issued)
      if (elect_one()) mma_commit(&bars->qempty);
      __syncwarp();
      ++commits;
    }
    // no MMA may still write TMEM when the CTA leaves (bounded)
    if (commits > 0) wait_bar(&bars->qempty, (commits - 1) & 1, p.wait_ns);
  } else if (warp < 4) {
    // ---------------- query build of the units after the first (64
    // threads).  (1) Once the epilogue is done with the row positions of two
    // units back: the cos/sin table, the row positions and the first batch
    // of this role's raw query rows, then the epilogue may join.  (2) Once
    // the MMAs of the previous unit are done with the image: rotate, split
    // and store this role's items (the epilogue stores the rest).  The raw
    // rows of the unit after are then pulled into L2 and its position read.
    constexpr int kGroups = D / 16;
    constexpr int kTotal = kRows * kGroups;
    constexpr int kX = kTotal * kBuildSplitNum / kBuildSplitDen;  // the builders' items
    constexpr int kPer = kX / 64;                 // items per builder thread
    constexpr int kB = kPer <= 6 ? kPer : kPer / 2;  // items per batch
    static_assert(kX % 64 == 0 && kPer % kB == 0, "whole batches");
    const int bt = threadIdx.x - 64;
    auto pull_rows = [&](int un) {
      const size_t rb = static_cast<size_t>(p.W) * p.G * D * 2;
      const size_t bb = static_cast<size_t>(p.M) * p.G * D * 2;
      const uint8_t* r0 = reinterpret_cast<const uint8_t*>(p.recent_q) + un * rb;
      for (size_t o = static_cast<size_t>(bt) * 128; o < rb; o += 64 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(r0 + o));
      if (bb > 0) {
        const uint8_t* b0 = reinterpret_cast<const uint8_t*>(p.beacons) + un * bb;
        for (size_t o = static_cast<size_t>(bt) * 128; o < bb; o += 64 * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(b0 + o));
      }
    };
    int32_t cur = 0;
    {
      const SubUnit w1 = sub_unit(p, 1, G, kRows, ngrp);
      if (w1.u < p.U) {
        if (w1.grp == 0) pull_rows(w1.u);
        cur = p.cur_pos[w1.u];
      }
    }
    for (int n = 1;; ++n) {
      const SubUnit w = sub_unit(p, n, G, kRows, ngrp);
      const int u = w.u;
      if (u >= p.U) break;
      bool ok = n < 2 || warp_wait(&bars->edone[n & 1], ((n - 2) >> 1) & 1, &bars->abort_flag,
                                   p.wait_ns);
      // both builder warps leave together (they meet at named barriers)
      if (named_sync_or(5, 64, !ok)) break;
      int32_t* rp = row_pos + (n & 1) * kRows;
      build_cs_table<D>(p, cur, cs, bt, 64);
      uint4 va[kB], vb[kB];
      load_query_batch<D, kB>(p, u, w.row0, kTotal, bt, 64, va, vb);
      const int nb = p.M > 0 ? min(max(p.n_beacons[u], 0), p.M) : 0;
      for (int r = bt; r < kRows; r += 64) rp[r] = row_position(p, u, w.row0 + r, nb, cur);
      named_sync(5, 64);
      if (warp == 2) {
        if (lane == 0) bars->cur[n & 1] = cur;
        publish_rows(p, rp, kRows, bars, n & 1, &bars->bready[n & 1], 1);
      }
      ok = warp_wait(&bars->qempty, (n - 1) & 1, &bars->abort_flag, p.wait_ns);
      if (named_sync_or(5, 64, !ok)) break;
#pragma unroll 1
      for (int k = 0; k < kPer; k += kB) {
        if (k > 0) load_query_batch<D, kB>(p, u, w.row0, kTotal, bt + k * 64, 64, va, vb);
        store_query_batch<D, kB>(p, kRows, kTotal, bt + k * 64, 64, va, vb, rp, cs, cur, q_hi,
                                 q_lo);
      }
      fence_proxy_async_shared();  // generic smem writes -> visible to the tensor core
      named_sync(5, 64);
      if (bt == 0) mbar_arrive(&bars->qfull[n & 1]);
      const SubUnit wn = sub_unit(p, n + 1, G, kRows, ngrp);
      if (wn.u < p.U) {
        if (wn.grp == 0) pull_rows(wn.u);
        cur = p.cur_pos[wn.u];
      }
    }
  } else {
    // ---------------- epilogue (warps 4..11)
    int g0 = 0;
    for (int n = 0;; ++n) {
      const SubUnit w = sub_unit(p, n, G, kRows, ngrp);
      const int u = w.u;
      if (u >= p.U) break;
      int t0, t1, L;
      split_tiles(p, u, 0, t0, t1, L);
      const int nt = t1 - t0;
      if (!(warp_wait(&bars->qfull[n & 1], (n >> 1) & 1, &bars->abort_flag, p.wait_ns) &&
            warp_wait(&bars->tready[n & 1], (n >> 1) & 1, &bars->abort_flag, p.wait_ns)) &&
          lane == 0)
        record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
      int32_t* rp = row_pos + (n & 1) * kRows;
      const int32_t* tm = tmax + (n & 1) * kTmaxTiles;
      const int32_t minrow = bars->minrow[n & 1], minpos = bars->minpos[n & 1];
      fused_epilogue<D, NR, kBufCols, kNBuf, kMax>(p, u, nt, L, g0, tbase, bars, rp, lse, mz, kp,
                                                   tm, minrow, minpos, w.nq16, w.nblk, w.grp);
      g0 += 2 * nt;
      // the epilogue's share of the next work item's query build (items
      // [kX, total)); the builders have placed the table and row positions
      const SubUnit wn = sub_unit(p, n + 1, G, kRows, ngrp);
      if (wn.u < p.U) {
        constexpr int kTotal = kRows * (D / 16);
        constexpr int kX = kTotal * kBuildSplitNum / kBuildSplitDen;
        constexpr int kEB = (kTotal - kX + kFusedEpi - 1) / kFusedEpi;
        const int nn = n + 1, et = threadIdx.x - 128;
        // The MMAs of this work item must be done with the image: each half
        // waited only for its own tiles, and the other half's last tile may
        // still be in the tensor core.  qempty completes once per work item.
        if (warp_wait(&bars->qempty, n & 1, &bars->abort_flag, p.wait_ns) &&
            warp_wait(&bars->bready[nn & 1], (nn >> 1) & 1, &bars->abort_flag, p.wait_ns)) {
          const int32_t cur = bars->cur[nn & 1];
          uint4 va[kEB], vb[kEB];
          load_query_batch<D, kEB>(p, wn.u, wn.row0, kTotal, kX + et, kFusedEpi, va, vb);
          store_query_batch<D, kEB>(p, kRows, kTotal, kX + et, kFusedEpi, va, vb,
                                    row_pos + (nn & 1) * kRows, cs, cur, q_hi, q_lo);
          fence_proxy_async_shared();  // generic smem writes -> visible to the tensor core
        } else if (lane == 0) {
          record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
        }
        named_sync(2, kFusedEpi);
        if (et == 0) mbar_arrive(&bars->qfull[nn & 1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->edone[n & 1]);
      // all epilogue warps leave together once any wait has failed
      if (named_sync_or(2, kFusedEpi,
                        *reinterpret_cast<volatile int32_t*>(&bars->abort_flag) != 0))
        break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kCols);
}

// --------------------------------------------------------------- cluster
// One pass over the keys, for max aggregation and up to 128 scoring rows:
// the keys of a unit are spread over a thread-block cluster of ncl CTAs,
// and each CTA keeps the logits of its own (at most four) 128-key tiles in
// its TMEM for the whole call (rows on the 128 lanes, one 128-column block
// per tile; 4 x 128 fp32 columns = all 512).  Nothing is computed twice and
// every key tile is read from memory once:
//   pass 1  thread = row: running max and sum of exp2 over the CTA's keys
//           (the two halves of the epilogue take alternate tiles and merge);
//   merge   every CTA posts its per-row (max, sum) in its shared memory, the
//           cluster meets at a hardware barrier, and every CTA merges all
//           posts of a row in rank order (distributed shared memory), so all
//           CTAs hold bit-identical log2-sum-exp values;
//   pass 2  the logits are read from TMEM once more: for each key the lanes
//           (rows) of a warp reduce max_r (s - lse_r) with redux.sync on
//           order-preserving keys, the four lane quarters combine through a
//           shared-memory atomicMax, and the score is exp2 of the maximum.
// Warp 0 issues the CTA's tile loads (one stage per tile, no refills), warp
// 1 the MMAs (hi and lo query terms into one accumulator per tile), warps
// 2..9 are the epilogue.
constexpr int kClTiles = 4;  // tiles per CTA: 4 x 128 TMEM columns

struct __align__(16) ClBars {
  uint64_t full[kClTiles];
  uint64_t tfull[kClTiles];
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t minrow;   // smallest key-position limit over the live rows
  int32_t minpos;   // smallest position over the live rows
  int32_t tmax[kClTiles];  // largest key position per tile (keys past L: unbounded)
};
static_assert(sizeof(ClBars) % 16 == 0, "arrays after the barriers need 16-byte alignment");

template <int D>
__global__ void __launch_bounds__(kFusedThreads, 1)
    score_cluster_kernel(const __grid_constant__ ScoreParams p,
                         const __grid_constant__ CUtensorMap kmap) {
  pdl_trigger();  // select + compact may set up; it waits for this grid before reading it
  if (!p.early_reads) pdl_wait();
  constexpr uint32_t kQBytes = 128 * D * 2;
  constexpr uint32_t kStageBytes = kTileKeys * D * 2;
  constexpr uint32_t kIdesc = idesc_bf16_f32(128, kTileKeys);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_hi = smem;
  uint8_t* q_lo = q_hi + kQBytes;
  uint8_t* stages = q_lo + kQBytes;
  ClBars* bars = reinterpret_cast<ClBars*>(stages + kClTiles * kStageBytes);
  int32_t* row_pos = reinterpret_cast<int32_t*>(bars + 1);        // [128]
  float2* mz = reinterpret_cast<float2*>(row_pos + 128);          // [128] second half's (m, z)
  float2* post = mz + 128;                                        // [128] this CTA's (m, z)
  int32_t* kp = reinterpret_cast<int32_t*>(post + 128);           // [4][128] key positions
  uint32_t* keymax = reinterpret_cast<uint32_t*>(kp + kClTiles * 128);  // [4][128]
  float2* cs = reinterpret_cast<float2*>(keymax + kClTiles * 128);      // [max(W,1)][D/2]

  const int ncl = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int u = blockIdx.x / ncl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L = p.L[u];
  if (L < 0 || L > p.L_cap) {
    if (threadIdx.x == 0 && rank == 0) record_error(p.ws, BKV_EDEVICE, kSiteScoreState);
    L = 0;
  }
  // tiles [t0, t1) of the unit: rank r takes its share of the layout's
  // tiles (at most kClTiles), cut at the unit's length
  const int ntc = (p.L_cap + kTileKeys - 1) / kTileKeys;
  const int nt = (L + kTileKeys - 1) / kTileKeys;
  const int t0 = min(rank * ntc / ncl, nt);
  const int t1 = min((rank + 1) * ntc / ncl, nt);
  const int ntl = t1 - t0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kClTiles; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->tfull[i], 1);
      bars->tmax[i] = INT32_MIN;
    }
    bars->abort_flag = 0;
    bars->minrow = INT32_MAX;
    bars->minpos = INT32_MAX;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer: every tile of the CTA at once
    if (lane == 0) {
      prefetch_tmap(&kmap);
      for (int i = 0; i < ntl; ++i) {
        mbar_arrive_expect_tx(&bars->full[i], kStageBytes);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(stages + i * kStageBytes + a * 16384, &kmap, &bars->full[i], 64 * a,
                      (t0 + i) * kTileKeys, u);
      }
      // every load has landed before the CTA can leave (bounded)
      for (int i = 0; i < ntl; ++i) wait_bar(&bars->full[i], 0, p.wait_ns);
    }
    __syncwarp();
  } else {
    // the epilogue stages the CTA's key positions while the queries build
    // (the positions are not written by the beacon selection)
    const int et = threadIdx.x - 64;  // 0..255 in the epilogue
    if (warp >= 2) {
      const int32_t* kpu = p.kpos + static_cast<size_t>(u) * p.L_cap;
      for (int e = et; e < kClTiles * 128; e += kFusedEpi) {
        const int j = t0 * kTileKeys + e;
        const int32_t v = (e < ntl * kTileKeys && j < L) ? kpu[j] : INT32_MAX;
        kp[e] = v;
        keymax[e] = 0u;
        const int32_t wm = __reduce_max_sync(0xffffffffu, v);
        if (lane == 0 && e < ntl * kTileKeys) atomicMax(&bars->tmax[e / kTileKeys], wm);
      }
    }
    build_queries<D>(p, u, 0, 128, q_hi, q_lo, row_pos, cs, threadIdx.x - 32,
                     kFusedThreads - 32, 1);
    if (warp == 1) {
      // ---------------- MMA issuer: tile i -> TMEM columns [128 i, 128 i + 128)
      int last = -1;
      for (int i = 0; i < (p.stall ? 0 : ntl); ++i) {
        if (!warp_wait(&bars->full[i], 0, &bars->abort_flag, p.wait_ns)) {
          if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t kbase = smem_u32(stages + i * kStageBytes);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint32_t qbase = smem_u32(part ? q_lo : q_hi);
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tbase + i * kTileKeys, sdesc_sw128(qbase + a * 16384 + kk * 32),
                         sdesc_sw128(kbase + a * 16384 + kk * 32), kIdesc, (part | a | kk) != 0);
          }
          mma_commit(&bars->tfull[i]);
        }
        __syncwarp();
        last = i;
      }
      if (last >= 0) wait_bar(&bars->tfull[last], 0, p.wait_ns);
    } else {
      // ---------------- pass 1: thread = row, running max / sum of exp2
      const int q = warp & 3, h = (warp - 2) >> 2;
      const int r = q * 32 + lane;  // TMEM lane = row
      const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
      const int32_t rp = row_pos[r];
      const int32_t lim = (p.causal || rp == INT32_MIN) ? rp : INT32_MAX - 1;
      const int32_t lw = __reduce_min_sync(0xffffffffu, rp != INT32_MIN ? lim : INT32_MAX);
      const int32_t pw = __reduce_min_sync(0xffffffffu, rp != INT32_MIN ? rp : INT32_MAX);
      if (lane == 0) {
        atomicMin(&bars->minrow, lw);
        atomicMin(&bars->minpos, pw);
      }
      named_sync(2, kFusedEpi);  // key positions, tile maxima and row limits in place
      const int32_t minrow = bars->minrow;
      float m = -INFINITY, z = 0.f;
      for (int i = h; i < ntl; i += 2) {
        const bool masked = !(bars->tmax[i] <= minrow);  // block-uniform
        if (warp_wait(&bars->tfull[i], 0, &bars->abort_flag, p.wait_ns)) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t v[64];  // keys 64 c .. 64 c + 63 of tile i
            const uint32_t col = tbase + lane_addr + i * kTileKeys + c * 64;
            tmem_ld32(col, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(col + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (masked) {
              const int* kh = kp + i * kTileKeys + 64 * c;
#pragma unroll
              for (int k = 0; k < 64; ++k)
                v[k] = kh[k] > lim ? __float_as_uint(-INFINITY) : v[k];
            }
            row_update(m, z, v);
          }
        } else if (lane == 0) {
          record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
        }
      }
      // the two halves of a row merge into this CTA's (max, sum) post
      if (h == 1) mz[r] = make_float2(m, z);
      named_sync(2, kFusedEpi);
      if (h == 0) {
        const float2 o = mz[r];
        const float mm = fmaxf(m, o.x);
        float zz = 0.f;
        if (mm != -INFINITY) {
          if (m != -INFINITY) zz += z * ex2(m - mm);
          if (o.x != -INFINITY) zz += o.y * ex2(o.x - mm);
        }
        post[r] = make_float2(mm, zz);
      }
    }
  }
  // every CTA's posts are in place and visible to the cluster
  __syncwarp();
  cluster_sync();
  if (warp >= 2) {
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int32_t rp = row_pos[r];
    const int32_t lim = (p.causal || rp == INT32_MIN) ? rp : INT32_MAX - 1;
    // log2-sum-exp of row r over the whole unit: every rank's post, merged
    // in rank order (the same order, so the same bits, in every CTA)
    float mm = -INFINITY;
    for (int k = 0; k < ncl; ++k) mm = fmaxf(mm, ld_cluster_f32(cluster_map(&post[r].x, k)));
    float zz = 0.f;
    if (mm != -INFINITY)
      for (int k = 0; k < ncl; ++k) {
        const float mk = ld_cluster_f32(cluster_map(&post[r].x, k));
        const float zk = ld_cluster_f32(cluster_map(&post[r].y, k));
        if (mk != -INFINITY) zz += zk * ex2(mk - mm);
      }
    // empty rows (no position, or no visible key): every probability is 0
    const float lse = (rp != INT32_MIN && zz > 0.f) ? mm + lg2(zz) : INFINITY;
    const int32_t minpos = bars->minpos;
    // ---------------- pass 2: per key, max over the rows of s - lse
    for (int i = h; i < ntl; i += 2) {
      const bool open = bars->tmax[i] <= minpos;  // every row sees every key of the tile
      if (warp_wait(&bars->tfull[i], 0, &bars->abort_flag, p.wait_ns)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kTileKeys / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_addr + i * kTileKeys + c * 32, v);
          tmem_wait_ld();
          const int* kh = kp + i * kTileKeys + 32 * c;
          uint32_t mine = 0u;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float x = __uint_as_float(v[k]) - lse;
            if (!open && kh[k] > lim) x = -INFINITY;
            // x <= 0 (lse is at least the row's largest logit); for x in
            // [-inf, 0] the complement of the bits orders like x
            const uint32_t key = ~__float_as_uint(fminf(x, 0.f));
            const uint32_t best = __reduce_max_sync(0xffffffffu, key);
            mine = lane == k ? best : mine;
          }
          atomicMax(&keymax[i * kTileKeys + 32 * c + lane], mine);
        }
      } else if (lane == 0) {
        record_error(p.ws, BKV_ETIMEOUT, kSiteScoreWait);
      }
    }
    named_sync(2, kFusedEpi);
    const int et = threadIdx.x - 64;
    float* dst = p.scores + static_cast<size_t>(u) * p.L_cap + t0 * kTileKeys;
    for (int e = et; e < ntl * kTileKeys; e += kFusedEpi)
      if (t0 * kTileKeys + e < L) dst[e] = ex2(__uint_as_float(~keymax[e]));
  }
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while another may still read its posts
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D>
size_t cluster_smem(int W) {
  return 1024 + 2 * static_cast<size_t>(128) * D * 2 + kClTiles * kTileKeys * D * 2 +
         sizeof(ClBars) + 128 * 4 + 2 * 128 * 8 + 2 * kClTiles * 128 * 4 +
         cs_bytes(W, D);
}

template <int D, int NS, int NR>
size_t fused_smem(int W) {
  return 1024 + 2 * static_cast<size_t>(NR) * 128 * D * 2 + NS * kTileKeys * D * 2 +
         sizeof(FusedBars) + NR * 128 * (2 * 4 + 4 + 8) + 256 * 4 + cs_bytes(W, D) +
         2 * kTmaxTiles * 4;
}

template <int D, int NS>
size_t stats_smem(int W) {
  return 1024 + 2 * 128 * D * 2 + NS * kTileKeys * D * 2 + sizeof(Barriers) + 128 * 4 + 256 * 4 +
         cs_bytes(W, D);
}
template <int D, int NS, int NMAX>
size_t final_smem(int W) {
  return 1024 + 2 * NMAX * D * 2 + NS * kTileKeys * D * 2 + sizeof(Barriers) + 256 * 4 +
         256 * 4 + cs_bytes(W, D);
}

int num_sms() {
  static const int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return 148;
    return v;
  }();
  return n;
}

// pdl: launched as a programmatic dependent of the previous kernel of the
// stream (its setup overlaps that kernel's tail; the kernel waits for it
// before reading what it wrote).
template <typename Kern>
cudaError_t launch(Kern kernel, dim3 grid, size_t smem, cudaStream_t st, const ScoreParams& p,
                   const CUtensorMap& map, int threads = kThreads, bool pdl = false) {
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, p, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

size_t score_smem_bytes(int d, int NQ16, int W, bool fused, int cluster) {
  if (cluster > 0) return d == 128 ? cluster_smem<128>(W) : cluster_smem<64>(W);
  if (fused) {
    const bool one = NQ16 <= 128;
    if (d == 128) return one ? fused_smem<128, 4, 1>(W) : fused_smem<128, 2, 2>(W);
    return one ? fused_smem<64, 4, 1>(W) : fused_smem<64, 4, 2>(W);
  }
  const bool small = NQ16 <= 128;
  if (d == 128) {
    const size_t a = stats_smem<128, 3>(W);
    const size_t b = small ? final_smem<128, 3, 128>(W) : final_smem<128, 2, 256>(W);
    return a > b ? a : b;
  }
  const size_t a = stats_smem<64, 4>(W);
  const size_t b = small ? final_smem<64, 4, 128>(W) : final_smem<64, 4, 256>(W);
  return a > b ? a : b;
}

cudaError_t launch_score(const ScoreParams& p, const CUtensorMap& kmap, cudaStream_t st) {
  if (p.cluster > 0) {
    auto* kernel = p.d == 128 ? score_cluster_kernel<128> : score_cluster_kernel<64>;
    const size_t smem = p.d == 128 ? cluster_smem<128>(p.W) : cluster_smem<64>(p.W);
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kernel), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.U * p.cluster));
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, p, kmap);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (p.fused) {
    // persistent: at most one CTA per SM, each taking units b, b + G, ...
    const dim3 g(static_cast<unsigned>(p.U < num_sms() ? p.U : num_sms()));
    const bool one = p.NQ16 <= 128;
    const int T = kPersistThreads;
    // max or mean aggregation as separate kernels (one epilogue each keeps
    // the register allocation free of spills)
    const bool mx = p.agg == BKV_AGG_MAX;
    if (p.d == 128) {
      if (one) {
        const size_t sm = fused_smem<128, 4, 1>(p.W);
        return mx ? launch(score_fused_kernel<128, 4, 1, true>, g, sm, st, p, kmap, T, true)
                  : launch(score_fused_kernel<128, 4, 1, false>, g, sm, st, p, kmap, T, true);
      }
      const size_t sm = fused_smem<128, 2, 2>(p.W);
      return mx ? launch(score_fused_kernel<128, 2, 2, true>, g, sm, st, p, kmap, T, true)
                : launch(score_fused_kernel<128, 2, 2, false>, g, sm, st, p, kmap, T, true);
    }
    if (one) {
      const size_t sm = fused_smem<64, 4, 1>(p.W);
      return mx ? launch(score_fused_kernel<64, 4, 1, true>, g, sm, st, p, kmap, T, true)
                : launch(score_fused_kernel<64, 4, 1, false>, g, sm, st, p, kmap, T, true);
    }
    const size_t sm = fused_smem<64, 4, 2>(p.W);
    return mx ? launch(score_fused_kernel<64, 4, 2, true>, g, sm, st, p, kmap, T, true)
              : launch(score_fused_kernel<64, 4, 2, false>, g, sm, st, p, kmap, T, true);
  }
  const dim3 g1(p.nsplit, p.nrows_part / 128, p.U);
  const dim3 g2(p.nsplit, p.ngrp, p.U);
  const bool small = p.NQ16 <= 128;
  const bool mx = p.agg == BKV_AGG_MAX;
  cudaError_t e;
  if (p.d == 128) {
    e = launch(score_stats_kernel<128, 3>, g1, stats_smem<128, 3>(p.W), st, p, kmap);
    if (e != cudaSuccess) return e;
    if (small) {
      const size_t sm = final_smem<128, 3, 128>(p.W);
      return mx ? launch(score_final_kernel<128, 3, 128, true>, g2, sm, st, p, kmap)
                : launch(score_final_kernel<128, 3, 128, false>, g2, sm, st, p, kmap);
    }
    const size_t sm = final_smem<128, 2, 256>(p.W);
    return mx ? launch(score_final_kernel<128, 2, 256, true>, g2, sm, st, p, kmap)
              : launch(score_final_kernel<128, 2, 256, false>, g2, sm, st, p, kmap);
  }
  e = launch(score_stats_kernel<64, 4>, g1, stats_smem<64, 4>(p.W), st, p, kmap);
  if (e != cudaSuccess) return e;
  if (small) {
    const size_t sm = final_smem<64, 4, 128>(p.W);
    return mx ? launch(score_final_kernel<64, 4, 128, true>, g2, sm, st, p, kmap)
              : launch(score_final_kernel<64, 4, 128, false>, g2, sm, st, p, kmap);
  }
  const size_t sm = final_smem<64, 4, 256>(p.W);
  return mx ? launch(score_final_kernel<64, 4, 256, true>, g2, sm, st, p, kmap)
            : launch(score_final_kernel<64, 4, 256, false>, g2, sm, st, p, kmap);
}

}  // namespace bkv
