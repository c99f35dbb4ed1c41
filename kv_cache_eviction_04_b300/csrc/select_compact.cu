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
//     the top: a 2048-bin shared-memory histogram with warp-aggregated
//     increments (match.any), then a block scan finds the bin holding the
//     k-th largest;
//   * the ascending kept list by block prefix sums (equal scores: the lower
//     slots first; when every key equal to the threshold is kept, one
//     comparison per slot decides).
// The unit's old key positions are staged in the ring's last two buffers
// and gathered for the moved rows while the first waves' loads fly.
// Compaction (row i <- row kept[i], kept[i] >= i) runs in waves over the
// rows that move, [first, n_kept): wave w covers ncl consecutive slices of
// RS rows, one per CTA.  Each CTA gathers its slice's source rows of K and V
// into a shared-memory ring with 16-byte cp.async copies spread over all its
// threads, the cluster meets at a hardware barrier once every CTA's copies
// of the wave have landed, and only then is each slice stored back (two TMA
// bulk stores of contiguous rows).  Sources of a wave lie at or above its
// first row, so stores of earlier waves never touch them, and a wave's
// stores wait for all of its loads: in-place compaction needs no second
// buffer and no spin-wait between CTAs.  Loads run nbufs - 2 waves ahead.
#include "common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBufs = 8;             // ring of wave buffers (count set by the host)
constexpr uint32_t kBufBig = 32768;     // bytes of one wave of one CTA (RS rows of K and V)
constexpr uint32_t kBufSmall = 16384;   // the same when a very large B_KV leaves less room

__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0;                         // -0.0 counts as +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // larger float -> larger key
}

// Inclusive block-wide prefix sum of one int per thread.
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

struct __align__(16) Smem {
  int32_t hist[2048];
  int32_t eq_total;  // candidates equal to the threshold key
  int32_t warp_tot[kWarps];
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
__device__ int select_kept(const SelectParams& p, const float* sc, const uint32_t* keys_s,
                           int L, int32_t* kept_s, Smem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n_kept = L <= p.B ? L : p.B;
  if (L <= p.B) {
    for (int i = tid; i < n_kept; i += kThreads) kept_s[i] = i;
    __syncthreads();
    return n_kept;
  }
  auto key_at = [&](int j) { return keys_s != nullptr ? keys_s[j] : order_key(sc[j]); };
  // ---------------- radix select of the (B - R)-th largest candidate:
  // digits of 11, 11 and 10 bits from the top; thread t owns the 8 bins
  // 2047 - 8t .. 2040 - 8t (descending) in the scan of each pass
  const int ncand = L - p.R;
  const int k = p.B - p.R;
  uint32_t prefix = 0;
  int krem = k;
  if (tid == 0) sm->eq_total = 0;
  if (k > 0) {
    constexpr int kShift[3] = {21, 10, 0};
    constexpr uint32_t kDigit[3] = {2047u, 2047u, 1023u};
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = kShift[pass];
      const uint32_t dmask = kDigit[pass];
      const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (kShift[pass - 1]));
#pragma unroll
      for (int b8 = 0; b8 < 8; ++b8) sm->hist[tid * 8 + b8] = 0;
      __syncthreads();
      for (int j0 = 0; j0 < ncand; j0 += kThreads) {
        const int j = j0 + tid;
        const bool in = j < ncand;
        const uint32_t key = in ? key_at(j) : 0u;
        const bool hit = in && (key & hmask) == prefix;
        const uint32_t bin = (key >> shift) & dmask;
        const uint32_t active = __ballot_sync(0xffffffffu, hit);
        if (hit) {
          const uint32_t same = __match_any_sync(active, bin);
          if ((__ffs(same) - 1) == lane) atomicAdd(&sm->hist[bin], __popc(same));
        }
      }
      __syncthreads();
      int c[8], loc = 0;
#pragma unroll
      for (int b8 = 0; b8 < 8; ++b8) {
        c[b8] = sm->hist[2047 - tid * 8 - b8];
        loc += c[b8];
      }
      const int incl = block_incl_scan(loc, sm->warp_tot);
      int above = incl - loc;  // candidates in higher bins than this thread's
      if (above < krem && incl >= krem) {
#pragma unroll
        for (int b8 = 0; b8 < 8; ++b8) {
          if (above < krem && above + c[b8] >= krem) {
            sm->prefix = prefix | (static_cast<uint32_t>(2047 - tid * 8 - b8) << shift);
            sm->krem = krem - above;
            if (pass == 2) sm->eq_total = c[b8];
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
  // ---------------- ascending kept list: contiguous segment per thread
  const int seg = (L + kThreads - 1) / kThreads;
  const int j0 = min(tid * seg, L), j1 = min(j0 + seg, L);
  if (k > 0 && sm->eq_total == need_eq) {
    // every candidate equal to T is kept: keep = key >= T
    int cnt = 0;
    for (int j = j0; j < j1; ++j) cnt += (j >= ncand || key_at(j) >= T);
    int pos = block_incl_scan(cnt, sm->warp_tot) - cnt;
    for (int j = j0; j < j1; ++j)
      if (j >= ncand || key_at(j) >= T) kept_s[pos++] = j;
    __syncthreads();
    return n_kept;
  }
  int eq_local = 0;
  for (int j = j0; j < j1 && j < ncand; ++j) eq_local += key_at(j) == T;
  const int eq_before = block_incl_scan(eq_local, sm->warp_tot) - eq_local;
  int kept_local = 0;
  {
    int e = eq_before;
    for (int j = j0; j < j1; ++j) {
      bool keep = j >= ncand;
      if (!keep) {
        const uint32_t key = key_at(j);
        keep = key > T || (key == T && e++ < need_eq);
      }
      kept_local += keep;
    }
  }
  int pos = block_incl_scan(kept_local, sm->warp_tot) - kept_local;
  {
    int e = eq_before;
    for (int j = j0; j < j1; ++j) {
      bool keep = j >= ncand;
      if (!keep) {
        const uint32_t key = key_at(j);
        keep = key > T || (key == T && e++ < need_eq);
      }
      if (keep) kept_s[pos++] = j;
    }
  }
  __syncthreads();
  return n_kept;
}

__global__ void __launch_bounds__(kThreads)
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
  if (tid == 0) sm->first = 0x7fffffff;
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
  if (keys_s != nullptr) {
#pragma unroll 8
    for (int j = tid; j < L; j += kThreads) keys_s[j] = order_key(sc[j]);
  }
  if (kpos_s != nullptr) {
#pragma unroll 8
    for (int j = tid; j < L; j += kThreads) kpos_s[j] = kp[j];
  }
  __syncthreads();
  const int n_kept = select_kept(p, sc, keys_s, L, kept_s, sm);
  // first destination row whose source differs (kept[i] == i before it)
  for (int i = tid; i < n_kept; i += kThreads)
    if (kept_s[i] != i) atomicMin(&sm->first, i);
  __syncthreads();  // the keys in the ring are dead from here on
  const int first = min(sm->first, n_kept);

  if (rank == 0 && p.kept != nullptr)
    for (int i = tid; i < p.B; i += kThreads)
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
  // All threads gather a wave's source rows of K and V into one ring buffer
  // with 16-byte cp.async copies (K rows first, then V rows); thread 0 then
  // writes the wave's contiguous destination rows back with two bulk stores.
  const int ppr = static_cast<int>(rb / 16);  // 16-byte pieces per row
  auto issue = [&](int w) {
    int r0, cnt;
    slice(w, r0, cnt);
    uint8_t* buf = bufs + (w % nbufs) * bufb;
    for (int e = tid; e < 2 * cnt * ppr; e += kThreads) {
      const int t = e / ppr, pc = e % ppr;
      const bool is_v = t >= cnt;
      const int row = is_v ? t - cnt : t;
      const size_t src = static_cast<size_t>(kept_s[r0 + row]) * rb + pc * 16;
      cp_async16(buf + (is_v ? RS + row : row) * rb + pc * 16, (is_v ? Vb : Kb) + src);
    }
  };
  // Waves w + 1 .. w + kAhead are in flight while wave w is stored.  Wave
  // w + kAhead reuses the buffer of wave w + kAhead - nbufs = w - 2, whose
  // store is the older of the two outstanding ones (waves w - 2 and w - 1).
  // Every thread commits one cp.async group per wave slot (empty past the
  // last wave), so "wave w landed" is "at most kAhead groups pending".
  // The first kAhead waves use buffers 0 .. nbufs - 3 only.
  const int kAhead = nbufs - 2;
  for (int w = 0; w < kAhead; ++w) {
    if (w < nw) issue(w);
    cp_async_commit();
  }
  // New kpos of every row this CTA writes, gathered while those gathers fly
  // and before the first wave's barrier (no CTA writes kpos before it);
  // entry w * RS + t = wave w, row t.
  for (int e = tid; e < nw * RS; e += kThreads) {
    int r0, cnt;
    slice(e / RS, r0, cnt);
    if (e % RS < cnt) {
      const int src = kept_s[r0 + e % RS];
      kpn[e] = kpos_s != nullptr ? kpos_s[src] : kp[src];
    }
  }
  __syncthreads();  // the staged key positions are dead from here on

  for (int w = 0; w < nw; ++w) {
    if (tid == 0) bulk_wait_read<1>();  // all stores but wave w - 1's have read smem
    __syncthreads();
    if (w + kAhead < nw) issue(w + kAhead);
    cp_async_commit();
    cp_async_wait_dyn(kAhead);
    fence_proxy_async_shared();  // this thread's smem writes -> the bulk stores
    __syncthreads();
    int r0, cnt;
    slice(w, r0, cnt);
    // Every CTA's sources of wave w are in its shared memory, so only
    // execution order matters here; a one-CTA cluster needs nothing more.
    if (ncl > 1) cluster_sync_relaxed();
    if (cnt > 0) {
      if (tid == 0) {
        const uint8_t* buf = bufs + (w % nbufs) * bufb;
        bulk_store(Kb + static_cast<size_t>(r0) * rb, buf, cnt * rb);
        bulk_store(Vb + static_cast<size_t>(r0) * rb, buf + RS * rb, cnt * rb);
        bulk_commit();
      }
      if (tid < cnt) kp[r0 + tid] = kpn[w * RS + tid];
    }
  }
  cp_async_wait<0>();
  if (tid == 0) bulk_wait<0>();
  cluster_sync();  // every CTA of the unit has read L and finished its copies
  if (rank == 0 && tid == 0 && valid) p.L[u] = n_kept;
}

}  // namespace

// Ring of the copy waves: buffers of 32 KB (16 KB when a very large B_KV
// leaves no room for three of 32 KB).  As many as fit (at most 8) when there
// are few units, each CTA then streaming with a deep pipeline; with many
// units, just enough to stage a unit's keys (at least 3), so that two CTAs
// share an SM and one copies while the other selects.  nbufs = 0: not even
// three buffers fit.
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
    n = want < n ? want : n;
  }
  *nbufs = n;
}

size_t select_smem_bytes(int B, int nbufs, int buf_bytes) {
  return bufs_offset(B) + static_cast<size_t>(nbufs) * buf_bytes;
}

cudaError_t launch_select_compact(const SelectParams& p, cudaStream_t st) {
  const size_t smem = select_smem_bytes(p.B, p.nbufs, p.buf_bytes);
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(select_compact_kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.U * p.ncl));
  cfg.blockDim = dim3(kThreads);
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
  e = cudaLaunchKernelEx(&cfg, select_compact_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace bkv
