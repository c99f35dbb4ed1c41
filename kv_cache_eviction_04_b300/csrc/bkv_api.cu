// C ABI of the BeaconKV eviction step (declared in include/bkv.h): argument
// validation, workspace layout, TMA descriptors and kernel launches.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bkv {
size_t select_smem_bytes(int B, int nbufs, int buf_bytes);
void select_ring(int B, int L_cap, bool many_units, int* nbufs, int* buf_bytes);
size_t fps_smem_bytes(int C);
}  // namespace bkv

namespace {

using bkv::WsHeader;

// The binding mirrors this layout (13 int32 fields, then the double).
static_assert(offsetof(bkv_dims, rope_theta) == 56 && sizeof(bkv_dims) == 64,
              "bkv_dims layout");

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const bkv_dims* d) {
  if (d == nullptr) return BKV_EINVAL;
  if (d->U < 1 || d->G < 1 || d->G > 16 || (d->d != 64 && d->d != 128)) return BKV_EINVAL;
  if (d->W < 0 || d->W > 64 || d->M < 0 || d->M > 64) return BKV_EINVAL;
  if (d->C < 2 || d->M >= d->C) return BKV_EINVAL;
  if (d->B_KV < 1 || d->B_KV > 16384 || d->R < 0 || d->R > d->B_KV) return BKV_EINVAL;
  if (d->L_cap < d->B_KV || d->L_cap > (1 << 24)) return BKV_EINVAL;
  if (d->agg != BKV_AGG_MAX && d->agg != BKV_AGG_MEAN) return BKV_EINVAL;
  if (d->causal_recent != 0 && d->causal_recent != 1) return BKV_EINVAL;
  if (d->beacon_select != BKV_BEACONS_FPS && d->beacon_select != BKV_BEACONS_FIRST) return BKV_EINVAL;
  if (d->compact != BKV_COMPACT_ORDERED && d->compact != BKV_COMPACT_FILL) return BKV_EINVAL;
  if (!(d->rope_theta > 1.0) || !std::isfinite(d->rope_theta)) return BKV_EINVAL;
  if (d->W + d->M < 1 || (d->W + d->M) * d->G > 1024) return BKV_EINVAL;
  if (static_cast<int64_t>(d->U) * d->L_cap * d->d >= (int64_t(1) << 40)) return BKV_EINVAL;
  if (d->C > 512) return BKV_EUNSUPPORTED;
  return BKV_OK;
}

int sm_count() {
  static int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      return 148;
    return v;
  }();
  return n;
}

struct ScoreShape {
  int NQ, NQ16, nrows_part, ngrp, ntiles, tiles_per_split, nsplit;
  bool fused;
  int cluster;  // > 0: single-pass scoring on a cluster of this many CTAs per unit
};

constexpr int kMaxSmem = 232448;  // bytes of shared memory a CTA may opt into on sm_103

ScoreShape score_shape(const bkv_dims* d) {
  ScoreShape s{};
  s.NQ = (d->W + d->M) * d->G;
  s.NQ16 = (s.NQ + 15) & ~15;
  s.nrows_part = (s.NQ + 127) / 128 * 128;
  s.ngrp = (s.NQ16 + 255) / 256;
  s.ntiles = (d->L_cap + 127) / 128;
  // Max aggregation over at most 128 rows, with a unit's logits fitting the
  // TMEM of at most 8 CTAs (4 key tiles each, L_cap <= 4096), and few
  // enough units that all their clusters run at once (one CTA per SM): one
  // pass, the keys of a unit spread over a thread-block cluster.  With more
  // units the one-CTA-per-unit kernel below keeps every SM busy with less
  // fixed work per key (each CTA builds its own query operand).
  const int ncl = (s.ntiles + 3) / 4;
  if (d->agg == BKV_AGG_MAX && s.NQ16 <= 128 && ncl <= 8 &&
      static_cast<int64_t>(d->U) * ncl <= sm_count() &&
      bkv::score_smem_bytes(d->d, s.NQ16, d->W, false, ncl) <= static_cast<size_t>(kMaxSmem)) {
    s.cluster = ncl;
    s.fused = false;
    s.tiles_per_split = s.ntiles;
    s.nsplit = 1;
    return s;
  }
  // The persistent two-pass kernel (one CTA per SM, units in turn) when
  // there are enough units to fill the GPU, or the rows fit one CTA's
  // operand and the caches are short; more than 256 rows are then scored
  // in groups of 256, one after another.  Otherwise the keys of a unit are
  // split over CTAs and the passes are two launches.
  s.fused = 2 * d->U >= sm_count() || (s.NQ16 <= 256 && s.ntiles <= 24);
  if (s.fused) {
    s.tiles_per_split = s.ntiles > 0 ? s.ntiles : 1;
    s.nsplit = 1;
    return s;
  }
  // about four CTAs per SM in the first pass, at least two tiles each
  const int64_t work = static_cast<int64_t>(d->U) * (s.nrows_part / 128) * s.ntiles;
  const int64_t target = 4ll * sm_count();
  int64_t tps = (work + target - 1) / target;
  if (tps < 2) tps = 2;
  if (tps > s.ntiles) tps = s.ntiles;
  if (tps < 1) tps = 1;
  s.tiles_per_split = static_cast<int>(tps);
  s.nsplit = (s.ntiles + s.tiles_per_split - 1) / s.tiles_per_split;
  if (s.nsplit < 1) s.nsplit = 1;
  return s;
}

struct WsLayout {
  size_t part, total;
};

WsLayout ws_layout(const bkv_dims* d) {
  WsLayout w{};
  const ScoreShape s = score_shape(d);
  w.part = bkv::kWsHeaderBytes;
  w.total = w.part + static_cast<size_t>(d->U) * s.nsplit * s.nrows_part * sizeof(float2);
  return w;
}

// CTAs per unit of the select + compact kernel: one CTA per SM in all, as
// one cluster of at most 8 (the portable cluster size) per unit.
int select_cluster_size(int U) {
  const int c = sm_count() / (U > 0 ? U : 1);
  return c < 1 ? 1 : (c > 8 ? 8 : c);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor map over [n2][n1][n0] (n0 contiguous), box {64, box1, 1},
// 128-byte swizzle, zero fill out of bounds.
int make_map(CUtensorMap* map, const void* base, uint64_t n0, uint64_t n1, uint64_t n2,
             uint32_t box1) {
  auto fn = encode_fn();
  if (fn == nullptr) return BKV_ECUDA;
  const cuuint64_t dims[3] = {n0, n1, n2};
  const cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
  const cuuint32_t box[3] = {64, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BKV_OK : BKV_ECUDA;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? BKV_OK : BKV_ECUDA; }

// Wait-timeout test setting of the scoring calls (bkv_test_wait_timeout),
// process-wide: the MMA issuer stalls and every wait gives up after wait_ns.
std::atomic<int32_t> g_test_stall{0};
std::atomic<int64_t> g_test_wait_ns{0};

}  // namespace

// Scratch of bkv_score_noalloc: a status header (as in a workspace) and the
// per-split (max, sum) partials of the scoring passes.  Lives in the
// library's device memory on every GPU that loads it, until process exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoAllocMaxDevices = 256;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return BKV_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BKV_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return BKV_OK;
}

}  // namespace

namespace {

// Validation and parameters of the beacon-selection call (nothing launched).
int fps_prepare(const bkv_dims* dims, const void* q_new, int64_t step, void* recent_q, void* buf,
                int32_t* cnt, int32_t want_beacons, int32_t* beacon_idx, void* beacons,
                int32_t* n_beacons, void* workspace, bkv::FpsParams* out, CUtensorMap* map,
                bool* cluster_out) {
  int v = validate(dims);
  if (v != BKV_OK) return v;
  if (buf == nullptr || cnt == nullptr || workspace == nullptr || step < 0) return BKV_EINVAL;
  if (q_new != nullptr && dims->W > 0 && recent_q == nullptr) return BKV_EINVAL;
  if (!aligned16(buf) || (q_new && !aligned16(q_new)) || (recent_q && !aligned16(recent_q)) ||
      (beacons && !aligned16(beacons)))
    return BKV_EINVAL;
  const bool cluster = dims->C > 256;
  *cluster_out = cluster;
  if ((cluster ? bkv::fps_cluster_smem_bytes() : bkv::fps_smem_bytes(dims->C)) >
      static_cast<size_t>(kMaxSmem))
    return BKV_EUNSUPPORTED;
  const int D = dims->G * dims->d;
  bkv::FpsParams& p = *out;
  p = bkv::FpsParams{};
  p.q_new = static_cast<const uint16_t*>(q_new);
  p.recent_q = static_cast<uint16_t*>(recent_q);
  p.buf = static_cast<uint16_t*>(buf);
  p.cnt = cnt;
  p.beacon_idx = beacon_idx;
  p.beacons = static_cast<uint16_t*>(beacons);
  p.n_beacons = n_beacons;
  p.ws = static_cast<WsHeader*>(workspace);
  p.step = step;
  p.U = dims->U;
  p.D = D;
  p.W = dims->W;
  p.M = dims->M;
  p.C = dims->C;
  p.want_beacons = want_beacons != 0;
  p.first_m = dims->beacon_select == BKV_BEACONS_FIRST ? 1 : 0;
  const uint32_t box_rows = static_cast<uint32_t>(std::min(256, (dims->C + 15) & ~15));
  return make_map(map, buf, static_cast<uint64_t>(D), static_cast<uint64_t>(dims->C),
                  static_cast<uint64_t>(dims->U), box_rows);
}

// Validation and parameters of the scoring call (nothing launched).  The
// partials and status word live in `workspace` (a caller workspace, or the
// library's static scratch).
int score_prepare(const bkv_dims* dims, const void* K, const int32_t* L, const int32_t* kpos,
                  const void* recent_q, int64_t step, const void* beacons,
                  const int32_t* n_beacons, const int32_t* cur_pos, float* scores,
                  void* workspace, bkv::ScoreParams* out, CUtensorMap* map) {
  int v = validate(dims);
  if (v != BKV_OK) return v;
  if (K == nullptr || L == nullptr || kpos == nullptr || cur_pos == nullptr ||
      scores == nullptr || step < 0)
    return BKV_EINVAL;
  if (dims->W > 0 && recent_q == nullptr) return BKV_EINVAL;
  if (dims->M > 0 && (beacons == nullptr || n_beacons == nullptr)) return BKV_EINVAL;
  if (!aligned16(K) || (recent_q && !aligned16(recent_q)) || (beacons && !aligned16(beacons)))
    return BKV_EINVAL;
  const ScoreShape s = score_shape(dims);
  if (bkv::score_smem_bytes(dims->d, s.NQ16, dims->W, s.fused, s.cluster) >
      static_cast<size_t>(kMaxSmem))
    return BKV_EUNSUPPORTED;
  bkv::ScoreParams& p = *out;
  p = bkv::ScoreParams{};
  p.L = L;
  p.kpos = kpos;
  p.recent_q = static_cast<const uint16_t*>(recent_q);
  p.beacons = static_cast<const uint16_t*>(beacons);
  p.n_beacons = n_beacons;
  p.cur_pos = cur_pos;
  p.scores = scores;
  p.part = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + bkv::kWsHeaderBytes);
  p.ws = static_cast<WsHeader*>(workspace);
  p.step = step;
  p.slot_now = dims->W > 0 ? static_cast<int32_t>(step % dims->W) : 0;
  p.step_cap = static_cast<int32_t>(step < (int64_t(1) << 30) ? step : (int64_t(1) << 30));
  p.U = dims->U;
  p.G = dims->G;
  p.d = dims->d;
  p.W = dims->W;
  p.M = dims->M;
  p.L_cap = dims->L_cap;
  p.NQ = s.NQ;
  p.NQ16 = s.NQ16;
  p.nrows_part = s.nrows_part;
  p.ngrp = s.ngrp;
  p.nsplit = s.nsplit;
  p.tiles_per_split = s.tiles_per_split;
  p.fused = s.fused ? 1 : 0;
  p.cluster = s.cluster;
  p.agg = dims->agg;
  p.causal = dims->causal_recent;
  p.early_reads = 0;
  const int64_t wns = g_test_wait_ns.load();
  p.wait_ns = wns > 0 ? static_cast<uint64_t>(wns) : bkv::kWaitBudgetNs;
  p.stall = g_test_stall.load();
  p.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(dims->d)));
  for (int i = 0; i < dims->d / 2; ++i) {
    const double f = std::pow(dims->rope_theta, -2.0 * i / static_cast<double>(dims->d));
    p.freq_hi[i] = static_cast<float>(f);
    p.freq_lo[i] = static_cast<float>(f - static_cast<double>(p.freq_hi[i]));
    p.step_cos[i] = static_cast<float>(std::cos(f));
    p.step_sin[i] = static_cast<float>(std::sin(f));
  }
  return make_map(map, K, static_cast<uint64_t>(dims->d), static_cast<uint64_t>(dims->L_cap),
                  static_cast<uint64_t>(dims->U), 128);
}

// Validation and parameters of the select + compact call (nothing launched).
int select_prepare(const bkv_dims* dims, const float* scores, void* K, void* V, int32_t* kpos,
                   int32_t* L, int32_t* kept, void* workspace, bkv::SelectParams* out) {
  const int v = validate(dims);
  if (v != BKV_OK) return v;
  if (scores == nullptr || K == nullptr || V == nullptr || kpos == nullptr || L == nullptr ||
      workspace == nullptr)
    return BKV_EINVAL;
  if (!aligned16(K) || !aligned16(V)) return BKV_EINVAL;
  int nbufs = 0, buf_bytes = 0;
  bkv::select_ring(dims->B_KV, dims->L_cap, dims->U >= 2 * sm_count(), &nbufs, &buf_bytes);
  if (nbufs < 3 ||
      bkv::select_smem_bytes(dims->B_KV, nbufs, buf_bytes) > static_cast<size_t>(kMaxSmem))
    return BKV_EUNSUPPORTED;
  bkv::SelectParams& p = *out;
  p = bkv::SelectParams{};
  p.scores = scores;
  p.K = static_cast<uint8_t*>(K);
  p.V = static_cast<uint8_t*>(V);
  p.kpos = kpos;
  p.L = L;
  p.kept = kept;
  p.ws = static_cast<WsHeader*>(workspace);
  p.U = dims->U;
  p.L_cap = dims->L_cap;
  p.B = dims->B_KV;
  p.R = dims->R;
  p.row_bytes = dims->d * 2;
  p.ncl = select_cluster_size(dims->U);
  p.nbufs = nbufs;
  p.buf_bytes = buf_bytes;
  p.fill = dims->compact == BKV_COMPACT_FILL ? 1 : 0;
  return BKV_OK;
}

}  // namespace

extern "C" {

int bkv_version(void) { return 1; }

const char* bkv_strerror(int code) {
  switch (code) {
    case BKV_OK: return "ok";
    case BKV_EINVAL: return "invalid argument";
    case BKV_ECUDA: return "CUDA runtime or launch failure";
    case BKV_ETIMEOUT: return "a device-side wait timed out";
    case BKV_EDEVICE: return "invalid per-unit device data";
    case BKV_EUNSUPPORTED: return "shape not supported by this build";
    default: return "unknown error code";
  }
}

int bkv_workspace_size(const bkv_dims* dims, size_t* bytes) {
  const int v = validate(dims);
  if (v != BKV_OK) return v;
  if (bytes == nullptr) return BKV_EINVAL;
  *bytes = ws_layout(dims).total;
  return BKV_OK;
}

int bkv_workspace_init(void* workspace, size_t bytes, bkv_stream_t stream) {
  if (workspace == nullptr || bytes < bkv::kWsHeaderBytes) return BKV_EINVAL;
  return cuda_rc(cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int bkv_fps_update(const bkv_dims* dims, const void* q_new, int64_t step, void* recent_q,
                   void* buf, int32_t* cnt, int32_t want_beacons, int32_t* beacon_idx,
                   void* beacons, int32_t* n_beacons, void* workspace, bkv_stream_t stream) {
  bkv::FpsParams p{};
  CUtensorMap map;
  bool cluster = false;
  const int v = fps_prepare(dims, q_new, step, recent_q, buf, cnt, want_beacons, beacon_idx,
                            beacons, n_beacons, workspace, &p, &map, &cluster);
  if (v != BKV_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // A decode step that selects no beacons appends with a light copy kernel
  // and compresses only the buffers that step filled.
  if (q_new != nullptr && want_beacons == 0 && !cluster)
    return cuda_rc(bkv::launch_fps_append_compress(p, map, sm_count(), st));
  return cuda_rc(cluster ? bkv::launch_fps_cluster(p, map, st) : bkv::launch_fps(p, map, sm_count(), st));
}

int bkv_score(const bkv_dims* dims, const void* K, const int32_t* L, const int32_t* kpos,
              const void* recent_q, int64_t step, const void* beacons,
              const int32_t* n_beacons, const int32_t* cur_pos, float* scores,
              void* workspace, bkv_stream_t stream) {
  if (workspace == nullptr) return BKV_EINVAL;
  bkv::ScoreParams p{};
  CUtensorMap map;
  const int v = score_prepare(dims, K, L, kpos, recent_q, step, beacons, n_beacons, cur_pos,
                              scores, workspace, &p, &map);
  if (v != BKV_OK) return v;
  return cuda_rc(bkv::launch_score(p, map, reinterpret_cast<cudaStream_t>(stream)));
}

int bkv_select_compact(const bkv_dims* dims, const float* scores, void* K, void* V,
                       int32_t* kpos, int32_t* L, int32_t* kept, void* workspace,
                       bkv_stream_t stream) {
  bkv::SelectParams p{};
  const int v = select_prepare(dims, scores, K, V, kpos, L, kept, workspace, &p);
  if (v != BKV_OK) return v;
  return cuda_rc(bkv::launch_select_compact(p, reinterpret_cast<cudaStream_t>(stream)));
}

int bkv_round(const bkv_dims* dims, const void* q_new, int64_t step, void* recent_q, void* buf,
              int32_t* cnt, int32_t* beacon_idx, void* beacons, int32_t* n_beacons,
              void* K, void* V, int32_t* L, int32_t* kpos, const int32_t* cur_pos,
              float* scores, int32_t* kept, void* workspace, bkv_stream_t stream) {
  if (workspace == nullptr) return BKV_EINVAL;
  if (dims != nullptr && dims->M > 0 && (beacons == nullptr || n_beacons == nullptr))
    return BKV_EINVAL;
  bkv::FpsParams fp{};
  CUtensorMap fmap;
  bool cluster = false;
  int v = fps_prepare(dims, q_new, step, recent_q, buf, cnt, 1, beacon_idx, beacons, n_beacons,
                      workspace, &fp, &fmap, &cluster);
  if (v != BKV_OK) return v;
  bkv::ScoreParams sp{};
  CUtensorMap smap;
  v = score_prepare(dims, K, L, kpos, recent_q, step, beacons, n_beacons, cur_pos, scores,
                    workspace, &sp, &smap);
  if (v != BKV_OK) return v;
  bkv::SelectParams cp{};
  v = select_prepare(dims, scores, K, V, kpos, L, kept, workspace, &cp);
  if (v != BKV_OK) return v;
  // scoring follows the beacon selection directly on the stream, and the
  // selection writes none of K, kpos, L or cur_pos: scoring may read them
  // before it waits for the selection
  sp.early_reads = 1;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  v = cuda_rc(cluster ? bkv::launch_fps_cluster(fp, fmap, st) : bkv::launch_fps(fp, fmap, sm_count(), st));
  if (v != BKV_OK) return v;
  v = cuda_rc(bkv::launch_score(sp, smap, st));
  if (v != BKV_OK) return v;
  return cuda_rc(bkv::launch_select_compact(cp, st));
}

int bkv_score_noalloc(const bkv_dims* dims, const void* K, const int32_t* L,
                      const int32_t* kpos, const void* recent_q, int64_t step,
                      const void* beacons, const int32_t* n_beacons, const int32_t* cur_pos,
                      float* scores, int32_t* device_status, bkv_stream_t stream) {
  int v = validate(dims);
  if (v != BKV_OK) return v;
  const ScoreShape s = score_shape(dims);
  const size_t need = bkv::kWsHeaderBytes +
                      static_cast<size_t>(dims->U) * s.nsplit * s.nrows_part * sizeof(float2);
  if (need > static_cast<size_t>(BKV_NOALLOC_SCRATCH_BYTES)) return BKV_EUNSUPPORTED;
  void* base = nullptr;
  v = noalloc_scratch(&base);
  if (v != BKV_OK) return v;
  bkv::ScoreParams p{};
  CUtensorMap map;
  v = score_prepare(dims, K, L, kpos, recent_q, step, beacons, n_beacons, cur_pos, scores, base,
                    &p, &map);
  if (v != BKV_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the previous call's status must not leak into this one
  if (cudaMemsetAsync(base, 0, bkv::kWsHeaderBytes, st) != cudaSuccess) return BKV_ECUDA;
  v = cuda_rc(bkv::launch_score(p, map, st));
  if (v != BKV_OK) return v;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, base, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return BKV_ECUDA;
  return BKV_OK;
}

int bkv_test_wait_timeout(int32_t stall, int64_t wait_ns) {
  if ((stall != 0 && stall != 1) || wait_ns < 0 ||
      wait_ns > static_cast<int64_t>(bkv::kWaitBudgetNs))
    return BKV_EINVAL;
  g_test_wait_ns.store(wait_ns);
  g_test_stall.store(stall);
  return BKV_OK;
}

int bkv_get_status(void* workspace, bkv_stream_t stream, int32_t* device_status) {
  if (workspace == nullptr || device_status == nullptr) return BKV_EINVAL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return BKV_ECUDA;
  WsHeader h{};
  if (cudaMemcpy(&h, workspace, 8, cudaMemcpyDeviceToHost) != cudaSuccess) return BKV_ECUDA;
  if (cudaMemset(workspace, 0, 8) != cudaSuccess) return BKV_ECUDA;
  *device_status = h.status;
  return BKV_OK;
}

}  // extern "C"
