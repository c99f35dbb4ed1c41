// Launch interfaces of the eviction-step kernels (internal to libbkv).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace bkv {

struct WsHeader;

// ------------------------------------------------------------------ score
struct ScoreParams {
  const int32_t* L;
  const int32_t* kpos;
  const uint16_t* recent_q;
  const uint16_t* beacons;
  const int32_t* n_beacons;
  const int32_t* cur_pos;
  float* scores;
  float2* part;  // [U][nsplit][nrows_part] (running max, sum of exp2), log2 units
  WsHeader* ws;
  int64_t step;
  int32_t slot_now;         // step % W: the ring slot of the newest query (0 when W = 0)
  int32_t step_cap;         // min(step, 2^30): ring slots older than this were never written
  int32_t U, G, d, W, M, L_cap;
  int32_t NQ;               // (W + M) * G scoring rows
  int32_t NQ16;             // NQ rounded up to 16
  int32_t nrows_part;       // NQ rounded up to 128 (pass-1 row blocks)
  int32_t ngrp;             // pass-2 row groups of <= 256
  int32_t nsplit;           // key-range splits per unit
  int32_t tiles_per_split;  // 128-key tiles per split
  int32_t agg, causal;
  int32_t fused;            // 1: the persistent two-pass kernel (row groups of 256)
  int32_t cluster;          // > 0: one pass on a cluster of this many CTAs per unit
                            // (max aggregation, NQ16 <= 128, at most 4 key tiles per CTA)
  int32_t early_reads;      // 1: the previous kernel of the stream is the beacon selection,
                            // which writes none of K, kpos, L, cur_pos (read before waiting)
  uint64_t wait_ns;         // budget of every mbarrier wait (ns)
  int32_t stall;            // wait-timeout test: the MMA issuer issues nothing, so the waits
                            // on its accumulator barriers run out after wait_ns
  float qscale;             // log2(e) / sqrt(d)
  float freq_hi[64];        // theta^(-2i/d) = freq_hi + freq_lo
  float freq_lo[64];
  float step_cos[64];       // cos and sin of theta^(-2i/d) (one position step)
  float step_sin[64];
};

cudaError_t launch_score(const ScoreParams& p, const CUtensorMap& kmap, cudaStream_t st);
size_t score_smem_bytes(int d, int NQ16, int W, bool fused, int cluster);

// --------------------------------------------------------- select+compact
struct SelectParams {
  const float* scores;
  uint8_t* K;
  uint8_t* V;
  int32_t* kpos;
  int32_t* L;
  int32_t* kept;  // optional [U][B]
  WsHeader* ws;
  int32_t U, L_cap, B, R, row_bytes;
  int32_t ncl;    // CTAs (one cluster) per unit, 1..8
  int32_t nbufs;      // wave buffers in the ring, 3..8
  int32_t buf_bytes;  // bytes of one wave buffer (32768 or 16384)
  int32_t fill;       // 1: hole-filling (order-free) compaction
};

cudaError_t launch_select_compact(const SelectParams& p, cudaStream_t st);

// ---------------------------------------------------------------- FPS
struct FpsParams {
  const uint16_t* q_new;  // [U][D] or null
  uint16_t* recent_q;     // [U][W][D]
  uint16_t* buf;          // [U][C][D]
  int32_t* cnt;
  int32_t* beacon_idx;    // [U][M] or null
  uint16_t* beacons;      // [U][M][D] or null
  int32_t* n_beacons;     // [U] or null
  WsHeader* ws;
  int64_t step;
  int32_t U, D, W, M, C;
  int32_t want_beacons;
  int32_t first_m;        // 1: the first M items instead of FPS (compress keeps them)
};

cudaError_t launch_fps(const FpsParams& p, const CUtensorMap& bufmap, int sms, cudaStream_t st);
// The append alone (one warp per unit), then the compress of the buffers it
// filled (a persistent grid of at most `sms` CTAs); C <= 256, no beacons.
cudaError_t launch_fps_append_compress(const FpsParams& p, const CUtensorMap& bufmap, int sms,
                                       cudaStream_t st);
// Capacities of 257..512: one cluster of ceil(C / 128) CTAs per unit.
cudaError_t launch_fps_cluster(const FpsParams& p, const CUtensorMap& bufmap, cudaStream_t st);
size_t fps_cluster_smem_bytes();

}  // namespace bkv
