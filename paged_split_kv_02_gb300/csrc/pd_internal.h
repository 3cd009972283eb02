// Internal host/device contract between the C ABI (pd_api.cu) and the
// decode kernels (pd_kernel.cuh, instantiated per head size).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "paged_decode.h"

namespace pd {

constexpr int kBlockKeys = 16;        // keys per TMA box and per mma m-tile
constexpr int kStageBytes = 32768;    // K + V bytes of one shared-memory ring stage
constexpr int kMaxRowGroups = 8;      // row groups of one kv head at most
// int32 counters reserved per (sequence, kv head): arrivals and finished
// mergers of every row group
constexpr int kCountersPerPair = 2 * kMaxRowGroups;
static_assert(kCountersPerPair == PD_COUNTERS_PER_PAIR, "counter reservation of the C ABI");
constexpr int kMaxConsumerWarps = 8;  // warps that compute; one more loads
constexpr int kMaxThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kSmemAlign = 1024;      // the 128-byte TMA swizzle repeats every 1 KiB
constexpr int kBlockIds = 512;        // page ids of 16-key blocks staged in shared memory
constexpr int kMaxBatchSegBlocks = 384;  // longest planned segment of a batch (6144 keys)
constexpr int64_t kNoSplitBytes = 256 << 10;  // K+V per (sequence, kv head) left unsplit
// Tensor-memory path: 4 softmax warps (one per tensor-memory sub-partition)
// and one warp that issues the tcgen05 MMAs, plus the producer warp; the
// packed rows (<= 64) are the M = 64 side of every MMA.
constexpr int kTcConsumerWarps = 5;
constexpr int kTcThreads = 32 * (kTcConsumerWarps + 1);
constexpr int kTcRows = 64;
constexpr int kTcBarriers = 9;  // S full/free, P full, PV done (x2 each), all MMAs done

// Everything a launch needs besides the two tensor maps.
struct Params {
  const void *q;
  int64_t q_s0, q_s1;  // element strides of q[t][hq][:]
  void *out;
  int64_t o_s0, o_s1;
  const int32_t *block_table;
  int64_t bt_stride;
  int bt_width;
  const int32_t *seq_lens;
  const int32_t *query_start;  // [S + 1] first q / out row of each sequence, or null
                               // (then sequence s owns rows s * M .. s * M + M - 1)
  int num_tokens;              // rows of q and out
  int num_pool_blocks;  // pages in the pool, for the page-id bounds check
  int Hq, Hkv, G, M, P, window, layout;
  float scale_log2;  // scale * log2(e): softmax runs on exp2
  int R;             // packed rows per kv head, G * M
  int rg;            // row groups (CTAs per kv head and segment)
  int rows_cta;      // packed rows per CTA, ceil(R / rg)
  int NT;            // 8-row mma n-tiles per CTA
  int KG;            // consumer warp groups; group g takes tiles g, g + KG, ...
  int NS;            // ring stages
  int seg_blocks;    // 16-key blocks per segment (lower bound)
  int max_seg;       // segments per (sequence, kv head, row group) in the grid
  int CS;            // cluster size of the merge
  int max_parts;     // partial slots per group, max_seg / CS
  float *part_acc;   // [S][Hkv][rg][max_parts][NT*8][D]
  float *part_ml;    // [S][Hkv][rg][max_parts][NT*8][2]
  int *counters;     // [S][Hkv][rg][2]: arrivals, finished mergers
  unsigned int *status;
  int64_t epi_floats;  // floats of the epilogue region (dead ring + Q tile)
  int coop;            // 1: co-resident grid, the last `mergers` arrivals merge
  int mergers;         // K_max of the cooperative merge (a power of two)
  unsigned long long wait_limit_ns;  // bound of a cooperative merger's wait for arrivals
  int num_seqs;                      // sequences of the call (rows of seq_lens)
  // 1: the block table, seq_lens, query_start and every key / value older
  // than a sequence's newest M tokens are complete before the previous grid
  // on the stream started, so they are read (and those pages streamed)
  // before the dependency wait; q, the newest keys and every write wait
  int early;
  // prefill: the work list (int32 [items][8]: sequence, tile, segment,
  // segments, split tile, first partial slot, blocks, 0), or null; the
  // split tiles and partial slots (per kv head) the scratch holds
  const int32_t *work;
  int pf_groups, pf_slots;
};

struct Launch {
  dim3 grid;
  dim3 block;
  int smem;
  int cluster;
  int cooperative;
};

// Dynamic shared memory of a launch: ring + Q tile + barriers + flags +
// the staged page ids.
inline int smem_bytes(int D, int NT, int NS) {
  return kSmemAlign + NS * kStageBytes + NT * D * 16 + 2 * NS * 8 + 16 + 4 * kBlockIds;
}
// The warp dot-product path (one n-tile) adds, 16-byte aligned, the Q rows
// in fp32 [8][D] and a P buffer [stage keys][8] fp32 per warp group.
inline int smem_bytes_dot(int D, int KG, int NS) {
  const int stage_keys = kStageBytes / 2 / (kBlockKeys * D * 2) * kBlockKeys;
  return smem_bytes(D, 1, NS) + 16 + 8 * D * 4 + KG * stage_keys * 8 * 4;
}

// Bytes of the epilogue region (the ring and the Q tile once they are dead).
inline int64_t epilogue_bytes(int D, int NT, int NS) {
  return (int64_t)NS * kStageBytes + (int64_t)NT * D * 16;
}

// Tensor-memory path: keys per stage, bytes of one P tile (64 rows of
// 128-byte swizzled rows per 64 keys), tensor-memory columns (two S buffers
// and O, rounded up to a power of two).
constexpr int tc_stage_keys(int D) { return kStageBytes / 2 / (kBlockKeys * D * 2) * kBlockKeys; }
constexpr int tc_p_tile_bytes(int D) {
  return kTcRows * (tc_stage_keys(D) > 64 ? tc_stage_keys(D) : 64) * 2;
}
constexpr int tc_tmem_cols(int D) {
  return 2 * tc_stage_keys(D) + D <= 32    ? 32
         : 2 * tc_stage_keys(D) + D <= 64  ? 64
         : 2 * tc_stage_keys(D) + D <= 128 ? 128
         : 2 * tc_stage_keys(D) + D <= 256 ? 256
                                            : 512;
}
// Dynamic shared memory of a tensor-memory launch: ring + 64-row Q tile +
// two P tiles + barriers + flags + staged page ids + tensor-memory address.
inline int smem_bytes_tc(int D, int NS) {
  return kSmemAlign + NS * kStageBytes + kTcRows * D * 2 + 2 * tc_p_tile_bytes(D) + 2 * NS * 8 +
         kTcBarriers * 8 + 16 + 4 * kBlockIds + 16;
}
inline int64_t epilogue_bytes_tc(int D, int NS) {
  return (int64_t)NS * kStageBytes + (int64_t)kTcRows * D * 2 + 2LL * tc_p_tile_bytes(D);
}

// Tensor-memory prefill path (TP, head size 128): two tiles of 128 packed
// rows share each K/V stage, one row of a tile per tensor-memory lane, each
// tile with its own four softmax warps; one warp issues the S MMAs of both
// tiles, one warp per tile the PV MMAs.  Both tiles' Q are in shared
// memory.  Columns: one S buffer per tile (fp32), two P buffers per tile
// (16-bit pairs), one O per tile (fp32): 512 at D = 128.
constexpr int kTpRows = 128;
constexpr int kTpSoftmaxWarps = 8;
constexpr int kTpConsumerWarps = kTpSoftmaxWarps + 1;  // + the warp that issues S
// warps: softmax 0..7, S issue 8, producer 9, PV issue 10 (tile 0) and 11
constexpr int kTpThreads = 32 * (kTpConsumerWarps + 3);
// barriers (per tile x and S / P buffer b): [0..3] S full (2 x + b), [4..7]
// P written (4 + 2 x + b), [8..11] PV done (8 + 2 x + b), [12] every MMA done
constexpr int kTpBarriers = 13;
constexpr int kTpBlockIds = 256;  // page ids staged at a time (room for a fifth stage)
// tensor-memory columns of a prefill CTA: two S buffers per tile (P of a
// stage overwrites its S), then O of both tiles
constexpr int tp_s_col(int D) { return 0 * D; }
constexpr int tp_o_col(int D) { return 4 * tc_stage_keys(D); }
constexpr int tp_tmem_cols(int D) {
  return tp_o_col(D) + 2 * D <= 128 ? 128 : tp_o_col(D) + 2 * D <= 256 ? 256 : 512;
}
static_assert(tp_o_col(128) + 2 * 128 <= 512, "tensor memory of a prefill tile");
// Dynamic shared memory of a tensor-memory prefill launch: ring + both
// tiles' Q + barriers + flags + staged page ids + tensor-memory address;
// its epilogue region is the dead ring and Q tiles.
inline int smem_bytes_tp(int D, int NS) {
  return kSmemAlign + NS * kStageBytes + 2 * kTpRows * D * 2 + 2 * NS * 8 + kTpBarriers * 8 + 16 +
         4 * kTpBlockIds + 16;
}
inline int64_t epilogue_bytes_tp(int D, int NS) {
  return (int64_t)NS * kStageBytes + 2LL * kTpRows * D * 2;
}

// Floats the epilogue needs: combine phase and final-merge phase.
inline int64_t epilogue_floats(int D, int NT, int KG, int CS, int ncl_max) {
  const int64_t nt8 = 8LL * NT;
  // the cluster combine (CS > 1) adds a D/CS slice, its (m, l) and weights
  const int64_t combine = KG * nt8 * D + 2LL * KG * nt8 + 2 * nt8 +
                          (CS > 1 ? nt8 * (D / CS) + 2 * nt8 + (int64_t)CS * nt8 : 0) + 16;
  // weights and sums of every part, then a chunk buffer of >= one row chunk
  // of one part (rows * D/CS <= 16 floats per thread)
  const int64_t final_merge = 2LL * ncl_max * nt8 + nt8 + 16 +
                              16LL * (kMaxThreads > kTpThreads ? kMaxThreads : kTpThreads) + D;
  return combine > final_merge ? combine : final_merge;
}

// path: 1 = mma.sync consumers, 2 = warp dot products (D <= 256, one 8-row
// n-tile), 3 = tcgen05 / tensor memory (D <= 256), 4 = mma.sync with the
// rows on the M side, 16 rows per warp (prefill tiles, D <= 128), 5 =
// tcgen05 prefill tiles of 128 rows with Q, S, P and O in tensor memory
// (D = 128)
cudaError_t launch_mma(int D, bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                       const Params &p, const Launch &l, cudaStream_t stream);

// The current device, checked (an sm_103 part): its SM count and the
// device status word.  Returns a pd_status.
int device_check(int *num_sms, unsigned int **status);

// Argument check of a paged cache pool descriptor and of a [rows, Hq, D]
// token-row descriptor, and the TMA tensor map of a pool (pd_api.cu).
int check_cache_tensor(const pd_tensor *t, int layout, int Hkv, int P, int D);
int check_rows(const pd_tensor *t, int64_t rows, int Hq, int D);
// one_box: a copy lands one 64-dim box of a 16-key block instead of all of
// them (the tensor-memory prefill's K, landed box-major).
int cache_tensor_map(const pd_tensor *t, int layout, CUtensorMap *out, bool one_box = false);

// The rotary embedding + paged KV-cache write (pd_rope.cu).
struct RopeParams {
  const void *q, *k, *v;
  int64_t q_s0, q_s1, k_s0, k_s1, v_s0, v_s1;  // element strides of [t][head][:]
  void *q_out;
  int64_t qo_s0, qo_s1;
  void *k_cache, *v_cache;
  int64_t kc_page, kc_tok, kc_head;  // element strides of (page, token, kv head)
  int64_t vc_page, vc_tok, vc_head;
  const int32_t *positions, *slots;
  const float *cos_sin;
  int64_t cs_s0;  // floats between table rows
  int max_pos;
  int T, Hq, Hkv, D, rot, P;
  int64_t num_slots;  // pages x page_size
  unsigned int *status;
};

}  // namespace pd
