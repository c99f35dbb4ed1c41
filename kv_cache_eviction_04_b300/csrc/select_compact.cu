// Top-B_KV selection and in-place, order-preserving K/V compaction.
//
// BeaconKV pages: inkeast.github.io reading, section 三 (the kept set is
// I = TopK(score(K,V), B_KV)); aimodeling.com article, section
// "用信标 query 预判" (only the highest-scoring entries survive while a recent
// sliding window is always kept).
//
// One CTA per (unit, tensor): part 0 compacts K (plus kpos, the kept list
// and the new length), part 1 compacts V.  Each CTA selects on its own (the
// scores of a unit are a few KB, far less than its K or V rows):
//   * radix select, 8 bits per pass from the top, on an order-preserving
//     integer image of the fp32 scores: a 256-bin shared-memory histogram
//     with warp-aggregated increments (match.any ballots), then a block
//     scan finds the bin holding the k-th largest;
//   * the ascending kept list by block prefix sums (equal scores: the lower
//     slots first);
//   * compaction: row i <- row kept[i] with kept[i] >= i.  Destination rows
//     are processed in ascending chunks by one warp: TMA bulk copies bring a
//     chunk's source rows into a shared-memory ring (one 16-byte-aligned
//     row per lane) and one bulk store writes the chunk's contiguous
//     destination rows back.  Sources of a later chunk lie at or above its
//     own first row, so they are never overwritten by earlier chunks' stores,
//     and a chunk is stored only after every earlier chunk's loads have
//     landed: in-place compaction needs no second buffer.
#include "common.cuh"
#include "kernels.h"

namespace bkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkRows = 32;  // rows per chunk: one per lane of the copy warp
constexpr int kStages = 8;

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
  uint64_t full[kStages];
  int32_t hist[256];
  int32_t warp_tot[kWarps];
  uint32_t prefix;
  int32_t krem;
  int32_t first;
  int32_t pad;
};

__global__ void __launch_bounds__(kThreads)
    select_compact_kernel(const __grid_constant__ SelectParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem* sm = reinterpret_cast<Smem*>(smem_raw);
  int32_t* kept_s = reinterpret_cast<int32_t*>(smem_raw + sizeof(Smem));
  uint8_t* stages =
      smem_raw + ((sizeof(Smem) + static_cast<size_t>(p.B) * 4 + 1023) & ~static_cast<size_t>(1023));
  const int u = blockIdx.x >> 1, part = blockIdx.x & 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* sc = p.scores + static_cast<size_t>(u) * p.L_cap;

  int L = p.L[u];
  const bool valid = L >= 0 && L <= p.L_cap;
  if (!valid) {
    if (tid == 0) record_error(p.ws, BKV_EDEVICE, kSiteSelectState);
    L = 0;
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&sm->full[i], 1);
    fence_mbar_init();
  }
  const int n_kept = L <= p.B ? L : p.B;

  if (L <= p.B) {
    for (int i = tid; i < n_kept; i += kThreads) kept_s[i] = i;
  } else {
    // ---------------- radix select of the (B - R)-th largest candidate
    const int ncand = L - p.R;
    const int k = p.B - p.R;
    uint32_t prefix = 0;
    int krem = k;
    if (k > 0) {
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        sm->hist[tid] = 0;
        __syncthreads();
        for (int j0 = 0; j0 < ncand; j0 += kThreads) {
          const int j = j0 + tid;
          const bool in = j < ncand;
          const uint32_t key = in ? order_key(sc[j]) : 0u;
          const bool hit = in && (key & hmask) == prefix;
          const uint32_t bin = (key >> shift) & 255u;
          const uint32_t active = __ballot_sync(0xffffffffu, hit);
          if (hit) {
            const uint32_t same = __match_any_sync(active, bin);
            if ((__ffs(same) - 1) == lane) atomicAdd(&sm->hist[bin], __popc(same));
          }
        }
        __syncthreads();
        // bins from the top: thread t holds bin 255 - t
        const int h = sm->hist[255 - tid];
        const int incl = block_incl_scan(h, sm->warp_tot);
        if (incl >= krem && incl - h < krem) {
          sm->prefix = prefix | (static_cast<uint32_t>(255 - tid) << shift);
          sm->krem = krem - (incl - h);
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
    int eq_local = 0;
    for (int j = j0; j < j1 && j < ncand; ++j) eq_local += order_key(sc[j]) == T;
    int eq_before = block_incl_scan(eq_local, sm->warp_tot) - eq_local;
    int kept_local = 0;
    {
      int e = eq_before;
      for (int j = j0; j < j1; ++j) {
        bool keep = j >= ncand;
        if (!keep) {
          const uint32_t key = order_key(sc[j]);
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
          const uint32_t key = order_key(sc[j]);
          keep = key > T || (key == T && e++ < need_eq);
        }
        if (keep) kept_s[pos++] = j;
      }
    }
  }
  if (tid == 0) sm->first = n_kept;
  __syncthreads();
  // first destination row whose source differs (kept[i] == i before it)
  for (int i = tid; i < n_kept; i += kThreads)
    if (kept_s[i] != i) atomicMin(&sm->first, i);
  __syncthreads();
  const int first = sm->first;

  if (part == 0) {
    if (p.kept != nullptr)
      for (int i = tid; i < p.B; i += kThreads)
        p.kept[static_cast<size_t>(u) * p.B + i] = i < n_kept ? kept_s[i] : -1;
    // kpos: gather everything first, then write (all reads precede writes)
    int32_t* kp = p.kpos + static_cast<size_t>(u) * p.L_cap;
    int32_t* tmp = reinterpret_cast<int32_t*>(stages);
    for (int i = first + tid; i < n_kept; i += kThreads) tmp[i - first] = kp[kept_s[i]];
    __syncthreads();
    for (int i = first + tid; i < n_kept; i += kThreads) kp[i] = tmp[i - first];
    __syncthreads();
  }

  // ---------------- compaction of this part's rows (one warp)
  if (warp == 0 && first < n_kept) {
    const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
    uint8_t* base = (part == 0 ? p.K : p.V) + static_cast<size_t>(u) * p.L_cap * rb;
    const int nrows = n_kept - first;
    const int nchunks = (nrows + kChunkRows - 1) / kChunkRows;
    const uint32_t stage_bytes = kChunkRows * rb;
    auto issue = [&](int c) {
      const int st = c % kStages;
      const int r0 = first + c * kChunkRows;
      const int cnt = min(kChunkRows, n_kept - r0);
      if (lane == 0) mbar_arrive_expect_tx(&sm->full[st], cnt * rb);
      __syncwarp();
      if (lane < cnt)
        bulk_load(stages + st * stage_bytes + lane * rb,
                  base + static_cast<size_t>(kept_s[r0 + lane]) * rb, rb, &sm->full[st]);
    };
    const int pro = min(kStages, nchunks);
    for (int c = 0; c < pro; ++c) issue(c);
    bool ok = true;
    int waited = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c % kStages;
      ok = __all_sync(0xffffffffu, wait_bar(&sm->full[st], (c / kStages) & 1));
      if (!ok) break;
      waited = c + 1;
      const int r0 = first + c * kChunkRows;
      const int cnt = min(kChunkRows, n_kept - r0);
      if (lane == 0) {
        bulk_store(base + static_cast<size_t>(r0) * rb, stages + st * stage_bytes, cnt * rb);
        bulk_commit();
      }
      // refill the stage of chunk c - 1 once its store has read the stage
      const int cn = c - 1 + kStages;
      if (c >= 1 && cn < nchunks) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        issue(cn);
      }
    }
    if (!ok) {
      if (lane == 0) record_error(p.ws, BKV_ETIMEOUT, kSiteSelectWait);
      // let copies already in flight land before the CTA exits (bounded)
      const int issued = min(nchunks, max(pro, waited - 1 + kStages));
      for (int c = waited; c < issued; ++c) wait_bar(&sm->full[c % kStages], (c / kStages) & 1);
    }
    if (lane == 0) bulk_wait<0>();
  }
  __syncthreads();
  // the second CTA of the unit to finish publishes the new length: both
  // CTAs have read L by then
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(&p.unit_done[u], 1);
    if (old == 1) {
      if (valid) p.L[u] = n_kept;
      p.unit_done[u] = 0;
    }
  }
}

}  // namespace

size_t select_smem_bytes(int B, int row_bytes) {
  const size_t ring = static_cast<size_t>(kStages) * kChunkRows * row_bytes;
  const size_t kpos_tmp = static_cast<size_t>(B) * 4;  // reuses the ring before the copy
  return ((sizeof(Smem) + static_cast<size_t>(B) * 4 + 1023) & ~static_cast<size_t>(1023)) +
         (ring > kpos_tmp ? ring : kpos_tmp);
}

cudaError_t launch_select_compact(const SelectParams& p, cudaStream_t st) {
  const size_t smem = select_smem_bytes(p.B, p.row_bytes);
  cudaError_t e = cudaFuncSetAttribute(select_compact_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  select_compact_kernel<<<2 * p.U, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
