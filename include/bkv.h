/*
 * bkv.h -- C ABI of the BeaconKV eviction step on NVIDIA B300 (sm_103a).
 *
 * BeaconKV ("Key-Value Cache Compression Guided by Beacon Queries for
 * Efficient Large Reasoning Model Inference", arXiv 2609.04971) evicts KV
 * cache entries by scoring every cached key with the attention of the most
 * recent queries together with a few "beacon" queries: representatives of
 * the far-looking ("global") queries of the decode so far, kept by a
 * continual farthest-point-sampling (FPS) buffer.  This library runs one
 * eviction step for many independent units at once.  A unit is one
 * (layer, sequence, KV head); all arrays are laid out unit-major.
 *
 * Passages each call follows (page titles of the BeaconKV pages):
 *   - wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫FPS的采样算法":
 *     FPS seed = the query with the lowest mean similarity to the others;
 *     each further pick is the query farthest from the chosen set; the
 *     similarity is taken on pre-RoPE queries; each head keeps a bounded
 *     buffer that an FPS pass compresses when it fills up.
 *   - same page, section "信标查询怎么用：位置对齐与打分策略": beacons are
 *     re-rotated to the current decode position, recent queries keep their
 *     own positions, and per-key importance is the max over queries.
 *   - inkeast.github.io reading, section 三 (formalisation): at eviction time
 *     the kept set is I = TopK(score(K,V), B_KV).
 *   - aimodeling.com article, section "用信标 query 预判" ("The mechanism has
 *     three parts"): only the highest-scoring entries survive while a recent
 *     sliding window is always kept; defaults 16 beacons and 16 recent queries.
 *
 * Conventions
 *   - All pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory and keeps no state between calls; scratch
 *     lives in a caller-allocated workspace (see bkv_workspace_size).  The
 *     one exception is bkv_score_noalloc, whose scratch is a fixed array in
 *     the library's own device memory: calls sharing that array must be
 *     ordered (see its declaration below).
 *   - bf16 arrays are raw 16-bit patterns.  Every array is dense, unit-major.
 *   - Every call only enqueues work on `stream` and returns; nothing
 *     synchronises except bkv_get_status.
 *   - Return codes: BKV_OK (0) or a negative BKV_E* value.  BKV_EINVAL and
 *     BKV_EUNSUPPORTED are detected on the host before anything is enqueued.
 *     Errors found on the device (a bad per-unit value, a wait that timed
 *     out) are recorded in the workspace's status word; read them with
 *     bkv_get_status.
 *   - Calls on one workspace must be ordered (one stream, or the caller's
 *     own events): kernels of overlapping calls would share its scratch.
 */
#ifndef BKV_H
#define BKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* bkv_stream_t;

enum {
  BKV_OK = 0,
  BKV_EINVAL = -1,       /* bad argument; nothing was enqueued            */
  BKV_ECUDA = -2,        /* a CUDA runtime call or launch failed          */
  BKV_ETIMEOUT = -3,     /* a device-side wait gave up (status word)      */
  BKV_EDEVICE = -4,      /* bad per-unit device data, e.g. L > L_cap      */
  BKV_EUNSUPPORTED = -5  /* valid but outside what this build implements  */
};

enum { BKV_AGG_MAX = 0, BKV_AGG_MEAN = 1 };

/*
 * Problem shape shared by all calls.
 *   U      units (layers x sequences x KV heads), U >= 1
 *   G      GQA group: query heads sharing one KV head, 1 <= G <= 16
 *   d      head dimension: 64 or 128
 *   W      recent queries scored (ring of the last W decode steps), 0 <= W <= 64
 *   M      beacons (FPS target size), 0 <= M <= 64, M < C
 *   C      continual-buffer capacity, 2 <= C <= 512
 *   B_KV   entries an eviction keeps, 1 <= B_KV <= 16384
 *   R      always-kept recent window: the last R cache slots, 0 <= R <= B_KV
 *   L_cap  row stride (slots) of K, V, kpos and scores; L_cap >= B_KV
 *   agg    BKV_AGG_MAX (the method) or BKV_AGG_MEAN
 *   causal_recent  1: a recent query at position p sees keys with kpos <= p;
 *                  0: every row sees every key
 *   beacon_select  BKV_BEACONS_FPS (0): beacons by farthest-point
 *                  sampling over the continual buffer, which is FPS-
 *                  compressed when full (the method);
 *                  BKV_BEACONS_FIRST (1): the first M buffered queries,
 *                  the buffer keeping its first M items when it fills (the
 *                  InitialRecent comparison of the BeaconKV pages: initial
 *                  queries plus the recent window)
 *   compact        BKV_COMPACT_ORDERED (0): the kept rows in slot order;
 *                  BKV_COMPACT_FILL (1): order-free, kept rows below the
 *                  new length stay and the holes there take the kept rows
 *                  past it (moves at most L - B_KV rows; see
 *                  bkv_select_compact)
 *   rope_theta     rotary base (rotate-half pairs (i, i + d/2),
 *                  frequency theta^(-2i/d))
 * Limits: (W + M) * G <= 1024 scoring rows; positions < 2^24.
 */
#define BKV_BEACONS_FPS 0
#define BKV_BEACONS_FIRST 1
#define BKV_COMPACT_ORDERED 0
#define BKV_COMPACT_FILL 1

typedef struct bkv_dims {
  int32_t U, G, d, W, M, C, B_KV, R;
  int32_t L_cap;
  int32_t agg;
  int32_t causal_recent;
  int32_t beacon_select; /* BKV_BEACONS_FPS (the method) or BKV_BEACONS_FIRST */
  int32_t compact;       /* BKV_COMPACT_ORDERED (default) or BKV_COMPACT_FILL */
  double rope_theta;
} bkv_dims;

/* Bytes of workspace the calls need for `dims` (same for all three calls). */
int bkv_workspace_size(const bkv_dims* dims, size_t* bytes);

/* Zero-fill a workspace (required once before first use; enqueued on
 * stream).  Calls leave the workspace ready for the next call. */
int bkv_workspace_init(void* workspace, size_t bytes, bkv_stream_t stream);

/*
 * One decode step of the continual FPS beacon buffer, for every unit.
 *
 *   q_new      [U][G][d] bf16, pre-RoPE queries of decode step `step`;
 *              may be NULL (no append: only the beacon selection runs)
 *   step       decode-step index (>= 0); its ring slot is step % W
 *   recent_q   [U][W][G][d] bf16 ring of recent pre-RoPE queries (in/out)
 *   buf        [U][C][G][d] bf16 FPS buffer (in/out); an item is the G*d
 *              vector of one decode step
 *   cnt        [U] int32 items in buf (in/out), 0 <= cnt < C on entry
 *   want_beacons  nonzero: also select beacons (below)
 *   beacon_idx [U][M] int32 or NULL: buffer slots of the beacons in FPS
 *              selection order; -1 past n_beacons
 *   beacons    [U][M][G][d] bf16 or NULL: the beacon vectors, same order
 *   n_beacons  [U] int32 or NULL: min(M, cnt) after the step
 *
 * Per unit, in order: (1) if q_new: ring[step % W] = q_new, buf[cnt] =
 * q_new, cnt += 1; (2) if cnt == C: FPS picks M of the C items (seed =
 * lowest mean cosine to the others, then greedily the item with the largest
 * 1 - cosine to its nearest chosen item; ties to the lowest slot), the
 * survivors stay in slot order in buf[0..M), cnt = M; (3) if want_beacons:
 * FPS picks min(M, cnt) of the cnt items (read-only; all of them, in slot
 * order, when cnt <= M).  Beacon and survivor indices match an fp64
 * evaluation: near-ties of the fp32 tensor-core pass are re-decided from the
 * bf16 inputs with exact products and error-free sums (~2^-44 relative), and
 * identical items tie exactly (lowest slot).  Requires a workspace of
 * bkv_workspace_size(dims) bytes.
 *
 * BeaconKV pages: the wzjinhao.cn explainer, section "怎么挑出这几个信标：一种叫
 * FPS的采样算法" (seed = the query least similar on average to the others,
 * then the query farthest from the chosen set; a bounded per-head buffer
 * of pre-RoPE queries, FPS-compressed when it fills), and the aimodeling.com
 * article, section "用信标 query 预判" (16 beacons by default).
 */
int bkv_fps_update(const bkv_dims* dims, const void* q_new, int64_t step, void* recent_q,
                   void* buf, int32_t* cnt, int32_t want_beacons, int32_t* beacon_idx,
                   void* beacons, int32_t* n_beacons, void* workspace, bkv_stream_t stream);

/*
 * Eviction scores of every cached key, for every unit.
 *
 *   K          [U][L_cap][d] bf16 cached keys (already rotated, as stored)
 *   L          [U] int32 current cache lengths, 0 <= L <= L_cap
 *   kpos       [U][L_cap] int32 position of each cached key
 *   recent_q   [U][W][G][d] bf16 ring (as maintained by bkv_fps_update)
 *   step       newest decode step written to the ring; ring slot s holds
 *              the step t <= step with t % W == s, at position
 *              cur_pos - ((step - s) mod W); slots older than step 0 are
 *              skipped
 *   beacons    [U][M][G][d] bf16 pre-RoPE beacons; n_beacons [U] valid ones
 *              (beacons / n_beacons may be NULL when M == 0)
 *   cur_pos    [U] int32 position of the current decode step
 *   scores     [U][L_cap] fp32 out: entries j < L written
 *
 * Rows are (query, head) pairs: each recent query with each of its G heads
 * at its own position, each beacon with each head rotated to cur_pos.  For
 * row r and key j: P_r(j) = softmax_j(q_r . K_j / sqrt(d)) over the keys row
 * r sees.  score_j = max_r P_r(j) (BKV_AGG_MAX) or the mean over rows.
 * Accuracy: |score - exact| <= 1e-6 + 2e-3 |exact| (fp32 accumulation of
 * bf16 products, queries carried as a two-term bf16 split).
 *
 * BeaconKV pages: the wzjinhao.cn explainer, section "信标查询怎么用：位置对齐与
 * 打分策略" (beacons re-rotated to the current position, recent queries at
 * their own positions, max over queries beats the mean), and the
 * inkeast.github.io reading, section 三 (score(K, V) from the union of the
 * recent and beacon queries).  M = 0 is recent-only scoring, the RPC
 * comparison on the same pages.
 */
int bkv_score(const bkv_dims* dims, const void* K, const int32_t* L, const int32_t* kpos,
              const void* recent_q, int64_t step, const void* beacons,
              const int32_t* n_beacons, const int32_t* cur_pos, float* scores,
              void* workspace, bkv_stream_t stream);

/*
 * Keep B_KV entries per unit and compact the cache in place.
 *
 *   scores     [U][L_cap] fp32 (from bkv_score; entries j < L read)
 *   K, V       [U][L_cap][d] bf16, compacted in place
 *   kpos       [U][L_cap] int32, compacted in place
 *   L          [U] int32 in: lengths; out: min(L, B_KV)
 *   kept       [U][B_KV] int32 or NULL: the source slot of each row after
 *              compaction (BKV_COMPACT_ORDERED: the kept slots in ascending
 *              order), -1 past the new length
 *
 * If L <= B_KV nothing moves.  Else the last R slots are kept, plus the
 * B_KV - R highest-scoring of the other L - R slots (equal scores: the lower
 * slot wins; -0.0 counts as +0.0; scores must not be NaN).  Rows of K, V and
 * kpos move alike; with n = B_KV kept:
 *   BKV_COMPACT_ORDERED  slot order is preserved: row i takes the row of the
 *                        i-th kept slot;
 *   BKV_COMPACT_FILL     a kept slot below n keeps its row, and the slots
 *                        below n that are not kept, in ascending order, take
 *                        the kept slots at or past n, in ascending order.  At
 *                        most L - n rows move.  Attention over the cache is
 *                        order-free (kpos carries each row's position), so
 *                        the row order is a layout choice; the BeaconKV pages
 *                        fix only the kept set (inkeast.github.io reading,
 *                        section 三).
 */
int bkv_select_compact(const bkv_dims* dims, const float* scores, void* K, void* V,
                       int32_t* kpos, int32_t* L, int32_t* kept, void* workspace,
                       bkv_stream_t stream);

/*
 * One eviction round: bkv_fps_update (want_beacons = 1), bkv_score and
 * bkv_select_compact on `stream`, with the arguments of those calls (K is
 * both the scored and the compacted cache).  BeaconKV pages: the
 * inkeast.github.io reading, section 三 (scoring with recent and beacon
 * queries, then I = TopK over the scores), and the wzjinhao.cn explainer on
 * FPS beacons.
 *
 * The results equal those of the three calls made one after the other.
 * Inside a round the library knows that scoring follows the beacon
 * selection, which writes none of K, kpos, L and cur_pos, so the scoring
 * kernel launches while the selection finishes and sets itself up (tile
 * maxima of the key positions, first key tiles, RoPE table) before waiting
 * for the beacons; select + compact likewise launches while scoring
 * finishes and waits for it before touching memory.  Every argument is
 * validated before anything is enqueued; on an error nothing runs.
 */
int bkv_round(const bkv_dims* dims, const void* q_new, int64_t step, void* recent_q, void* buf,
              int32_t* cnt, int32_t* beacon_idx, void* beacons, int32_t* n_beacons, void* K,
              void* V, int32_t* L, int32_t* kpos, const int32_t* cur_pos, float* scores,
              int32_t* kept, void* workspace, bkv_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the workspace status word:
 * *device_status = BKV_OK or the first BKV_ETIMEOUT / BKV_EDEVICE recorded
 * by a kernel since the last read.  Returns BKV_OK or BKV_ECUDA.
 */
int bkv_get_status(void* workspace, bkv_stream_t stream, int32_t* device_status);

/*
 * bkv_score without a caller-provided workspace.  (The BeaconKV paper has
 * no counterpart: this is a deployment variant of bkv_score.)
 *
 * For callers that cannot allocate device memory themselves: plugins
 * hosted by a framework that owns every device allocation and offers no
 * allocation hook, or loops where cudaMalloc's implicit device-wide
 * synchronisation is not acceptable.  The call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine); its scratch is a
 * fixed array of BKV_NOALLOC_SCRATCH_BYTES bytes in the library's own
 * device memory, which every GPU that loads the library holds until the
 * process exits.
 *
 * Arguments and results are those of bkv_score, except:
 *   device_status  optional device pointer to one int32; when the call's
 *                  kernels finish it holds BKV_OK or the BKV_ETIMEOUT /
 *                  BKV_EDEVICE they recorded (NULL: not reported)
 * Returns BKV_EUNSUPPORTED, before enqueuing anything, when the shape needs
 * more scratch than the array holds: 256 + U * nsplit * ceil(NQ/128)*128 * 8
 * bytes (NQ = (W + M) * G scoring rows).  nsplit, the key-range splits of
 * the launch, is 1 when one CTA scores a whole unit (NQ <= 256 and either
 * 2 U >= the SM count or L_cap <= 3072); otherwise the splits take about
 * U * ceil(NQ/128) * ceil(L_cap/128) / (4 * SMs) key tiles each, at least 2.
 * For example 112 units of 128 rows need 0.11 MB.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress) and caches it; make that first call before
 * any stream capture.  Every call on a device shares the one array, so
 * calls whose kernels overlap on the GPU (different streams without an
 * ordering between them) race: order them.  Each call clears the status
 * word it uses before its kernels run.
 */
#define BKV_NOALLOC_SCRATCH_BYTES (8u << 20)
int bkv_score_noalloc(const bkv_dims* dims, const void* K, const int32_t* L,
                      const int32_t* kpos, const void* recent_q, int64_t step,
                      const void* beacons, const int32_t* n_beacons, const int32_t* cur_pos,
                      float* scores, int32_t* device_status, bkv_stream_t stream);

/*
 * Test hook for the device-side timeout path of the scoring calls
 * (bkv_score, bkv_score_noalloc and the scoring step of bkv_round).  Every
 * mbarrier wait of those kernels is bounded; with wait_ns > 0 the bound is
 * wait_ns nanoseconds instead of 2 s.  With stall = 1 the MMA issuer of
 * each scoring CTA issues nothing, so the waits on its accumulator
 * barriers run out: the kernels then record BKV_ETIMEOUT in the status
 * word, let every role drain (loads already issued land, no MMA is left
 * running) and return normally, leaving the device usable.  Scores are
 * then undefined.  stall = 0 and wait_ns = 0 restore normal operation.
 * The setting is process-wide and is read when a call is made; it is meant
 * for tests of the error path only.  (The BeaconKV paper has no
 * counterpart.)  Returns BKV_EINVAL for stall outside {0, 1} or wait_ns
 * outside [0, 2e9].
 */
int bkv_test_wait_timeout(int32_t stall, int64_t wait_ns);

/* Static description of a return code. */
const char* bkv_strerror(int code);

/* ABI version: 1. */
int bkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BKV_H */
