// Paged prefill: the host work-list planner and the launch of the decode
// kernel over a work list (plan_prefill, prefill_target_workgroups and
// _BuiltinPrefill.prefill_attn on the vllm.v1.attention.ops.rocm_rdna_hip
// page).
//
// A request's query tokens are packed token-major into rows (token i, q
// head h*G + j -> row i*G + j) and cut into tiles of PD_PREFILL_TILE_ROWS
// rows (PD_PREFILL_TILE_ROWS_D128 at head size 128, the tensor-memory
// tiles); a tile's keys run from its window start (rounded down to a 16-key
// block) to the last key its last token sees.  A tile heavier than the mean
// load per resident CTA is cut into segments, merged in the kernel by the
// last-arriving segment.  Items are ordered heaviest first, so the longest
// tiles start in the first wave and the short ones fill the tail.
#include <algorithm>
#include <cmath>
#include <vector>

#include "paged_decode.h"
#include "pd_internal.h"

namespace pd {
namespace {

// packed rows of a tile: 256 (two tiles of one row per tensor-memory lane)
// where the tensor-memory consumer serves the head size, else 64
int tile_rows_for(int D) { return D == 128 ? PD_PREFILL_TILE_ROWS_D128 : PD_PREFILL_TILE_ROWS; }
static_assert(PD_PREFILL_TILE_ROWS_D128 == 2 * kTpRows, "two tensor-memory tiles per CTA");
bool head_size_ok(int D) { return D == 64 || D == 128 || D == 256 || D == 512; }
constexpr int kMaxSegments = PD_PREFILL_MAX_SEGMENTS;
// a segment reads at least this many 16-key blocks (two ring stages at
// D = 128), so that its partial stays small next to the keys it read
constexpr int kMinSegmentBlocks = 8;
constexpr int kSmemLimit = 232448;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Tile {
  int32_t seq, tile;
  int64_t blocks;
  int32_t nseg;
};

// The plan shared by paged_prefill_plan and paged_prefill_attn's checks.
int plan_tiles(const int32_t *query_start, const int32_t *seq_lens, int S, int Hq, int Hkv,
               int rows, int window, int target, std::vector<Tile> *tiles,
               pd_prefill_plan_info *info) {
  if (S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || window < 0 || target <= 0 || rows <= 0)
    return PD_EINVAL;
  if (S > 0 && (!query_start || !seq_lens)) return PD_EINVAL;
  const int G = Hq / Hkv;
  tiles->clear();
  int64_t total = 0;
  for (int s = 0; s < S; ++s) {
    const int64_t q_len = (int64_t)query_start[s + 1] - query_start[s];
    if (query_start[s] < 0 || q_len < 0) return PD_EINVAL;
    if (q_len == 0) continue;
    // the request's keys include its new tokens (a shorter seq_len counts
    // as the query length: no context)
    const int64_t L = std::max<int64_t>(seq_lens[s], q_len);
    const int64_t context = L - q_len;
    const int64_t ntiles = cdiv(q_len * G, rows);
    if (ntiles > INT32_MAX) return PD_EINVAL;
    // the request's last tile first (it sees the most keys)
    for (int64_t t = ntiles - 1; t >= 0; --t) {
      const int64_t first = t * rows / G;
      const int64_t last = std::min(q_len - 1, ((t + 1) * rows - 1) / G);
      const int64_t key_end = context + last + 1;
      const int64_t key_begin =
          window ? std::max<int64_t>(0, context + first - window + 1) / kBlockKeys * kBlockKeys : 0;
      const int64_t blocks = cdiv(key_end - key_begin, kBlockKeys);
      tiles->push_back({s, (int32_t)t, blocks, 1});
      total += blocks;
    }
  }
  // the load each resident CTA would carry with every tile on every kv head
  // spread evenly; a heavier tile is cut into about load-sized segments
  const double load = std::max((double)Hkv * (double)total / target, (double)kMinSegmentBlocks);
  int32_t n_split = 0, n_slots = 0;
  for (Tile &t : *tiles) {
    if ((double)t.blocks > load) {
      const int64_t by_load = (int64_t)std::ceil((double)t.blocks / load);
      const int64_t by_floor = t.blocks / kMinSegmentBlocks;
      t.nseg = (int32_t)std::max<int64_t>(1, std::min<int64_t>({by_load, by_floor, kMaxSegments}));
    }
    if (t.nseg > 1) {
      ++n_split;
      n_slots += t.nseg;
    }
  }
  // heaviest per-segment load first; equal loads keep the order above
  std::stable_sort(tiles->begin(), tiles->end(), [](const Tile &a, const Tile &b) {
    return (double)a.blocks / a.nseg > (double)b.blocks / b.nseg;
  });
  int64_t items = 0;
  for (const Tile &t : *tiles) items += t.nseg;
  info->num_items = items;
  info->num_split_tiles = n_split;
  info->num_slots = n_slots;
  info->tile_rows = rows;
  info->max_segments = kMaxSegments;
  info->total_blocks = total;
  info->load_blocks = load;
  info->target_ctas = target;
  return PD_OK;
}

// Launch shape of a prefill tile.  At D = 128: 256 rows on the tensor
// cores (path 5: two tiles of 128 rows sharing each K/V stage, S, P and O
// in tensor memory, four softmax warps per tile and one MMA warp), as many
// 32 KiB ring stages as fit next to the second tile's Q.  Otherwise 8 n-tiles of 8
// rows, as many stages as fit next to the Q tile; at D = 64 the rows sit on
// the MMA's M side, one warp per 16 rows (path 4: each stage is read from
// shared memory once per 16 rows); larger heads keep the keys on the M side,
// one warp per 8 rows (path 1).
struct PrefillShape {
  int NT, KG, NS, smem, threads, path;
  int64_t epi;  // bytes of the epilogue region
};

int prefill_shape(int D, PrefillShape *sh) {
  if (D == 128) {
    sh->path = 5;
    sh->NT = 2 * kTpRows / 8;
    sh->KG = 1;
    sh->NS = std::min(8, (kSmemLimit - smem_bytes_tp(D, 0)) / (kStageBytes + 16));
    if (sh->NS < 2) return PD_EINVAL;
    sh->smem = smem_bytes_tp(D, sh->NS);
    sh->epi = epilogue_bytes_tp(D, sh->NS);
    if (epilogue_floats(D, sh->NT, sh->KG, 1, kMaxSegments) * 4 > sh->epi) return PD_EINVAL;
    sh->threads = kTpThreads;
    return PD_OK;
  }
  sh->NT = PD_PREFILL_TILE_ROWS / 8;
  sh->path = D <= 128 ? 4 : 1;
  // path 4: two warp groups of four warps take alternate stages
  sh->KG = sh->path == 4 ? 2 : 1;
  const int fixed = smem_bytes(D, sh->NT, 0);
  sh->NS = std::min(8, (kSmemLimit - fixed - 16 * 8) / kStageBytes) / sh->KG * sh->KG;
  if (sh->NS < 2) return PD_EINVAL;
  if (epilogue_floats(D, sh->NT, sh->KG, 1, kMaxSegments) * 4 > epilogue_bytes(D, sh->NT, sh->NS))
    return PD_EINVAL;
  sh->smem = smem_bytes(D, sh->NT, sh->NS);
  sh->epi = epilogue_bytes(D, sh->NT, sh->NS);
  sh->threads = 32 * ((sh->path == 4 ? sh->NT / 2 : sh->NT) * sh->KG + 1);
  return PD_OK;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace
}  // namespace pd

using namespace pd;

extern "C" {

PD_API int paged_prefill_plan(const int32_t *query_start, const int32_t *seq_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_size, int window,
                              int num_sms, pd_prefill_item *items, int64_t capacity,
                              pd_prefill_plan_info *info) {
  if (!info) return PD_EINVAL;
  if (!head_size_ok(head_size)) return PD_EHEAD;
  if (num_sms <= 0) {
    int rc = device_check(&num_sms, nullptr);
    if (rc != PD_OK) return rc;
  }
  std::vector<Tile> tiles;
  int rc = plan_tiles(query_start, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                      tile_rows_for(head_size), window, num_sms, &tiles, info);
  if (rc != PD_OK) return rc;
  if (!items) return PD_OK;  // a size query
  if (capacity < info->num_items) return PD_EINVAL;
  int64_t k = 0;
  int32_t split = 0, slot = 0;
  for (const Tile &t : tiles) {
    for (int32_t g = 0; g < t.nseg; ++g) {
      pd_prefill_item &it = items[k++];
      it.seq = t.seq;
      it.tile = t.tile;
      it.seg = g;
      it.nseg = t.nseg;
      it.split = t.nseg > 1 ? split : -1;
      it.slot = t.nseg > 1 ? slot : -1;
      it.blocks = (int32_t)std::min<int64_t>(t.blocks, INT32_MAX);
      it.reserved = 0;
    }
    if (t.nseg > 1) {
      ++split;
      slot += t.nseg;
    }
  }
  return PD_OK;
}

PD_API size_t paged_prefill_scratch_bytes(int num_kv_heads, int head_size, int num_sms) {
  if (num_kv_heads <= 0 || num_sms <= 0) return 0;
  if (!head_size_ok(head_size)) return 0;
  const int rows = tile_rows_for(head_size);
  // counters of paged_decode_scratch_init(.., max_num_seqs = num_sms,
  // num_kv_heads = 1, ..) and partials of 2 x num_sms slots: a plan splits
  // fewer than num_sms tiles x kv heads into fewer than 2 x num_sms
  // segments x kv heads
  const int64_t counters = round256((int64_t)num_sms * PD_COUNTERS_PER_PAIR * 4);
  const int64_t slots = 2LL * num_sms;
  const int64_t acc = round256(slots * rows * head_size * 4);
  const int64_t ml = round256(slots * rows * 2 * 4);
  return (size_t)(counters + acc + ml);
}

PD_API int paged_prefill_attn(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
                              const pd_tensor *block_table, const pd_tensor *seq_lens,
                              const pd_tensor *query_start, const pd_tensor *work,
                              const pd_prefill_plan_info *info, pd_tensor *out, int num_q_heads,
                              int num_kv_heads, int head_size, int page_size, int window,
                              float scale, int layout, pd_scratch *scratch, void *stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !query_start || !work ||
      !info || !out)
    return PD_EINVAL;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PD_EINVAL;
  if (!head_size_ok(head_size)) return PD_EHEAD;
  const int rows = tile_rows_for(head_size);
  if (page_size <= 0 || page_size % kBlockKeys != 0 || window < 0 || !std::isfinite(scale))
    return PD_EINVAL;
  if (layout != PD_NHD && layout != PD_HND) return PD_EINVAL;
  if (seq_lens->ndim != 1 || !seq_lens->data || seq_lens->stride[0] != 1) return PD_EINVAL;
  if (seq_lens->dtype != PD_I32 || block_table->dtype != PD_I32 || query_start->dtype != PD_I32 ||
      work->dtype != PD_I32)
    return PD_EDTYPE;
  const int64_t S = seq_lens->shape[0];
  if (S < 0 || S > INT32_MAX) return PD_EINVAL;
  if (block_table->ndim != 2 || !block_table->data || block_table->shape[0] != S ||
      block_table->shape[1] < 1 || block_table->stride[1] != 1 || block_table->stride[0] < 0)
    return PD_EINVAL;
  if (block_table->shape[1] * (int64_t)page_size > INT32_MAX) return PD_EINVAL;
  if (query_start->ndim != 1 || !query_start->data || query_start->shape[0] != S + 1 ||
      query_start->stride[0] != 1)
    return PD_EINVAL;
  if (q->ndim != 3) return PD_EINVAL;
  const int64_t T = q->shape[0];
  if (T < 0 || T > INT32_MAX) return PD_EINVAL;
  int rc;
  if (T > 0) {
    if ((rc = check_rows(q, T, num_q_heads, head_size)) != PD_OK) return rc;
    if ((rc = check_rows(out, T, num_q_heads, head_size)) != PD_OK) return rc;
  }
  if ((rc = check_cache_tensor(k_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK)
    return rc;
  if ((rc = check_cache_tensor(v_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK)
    return rc;
  if (q->dtype != out->dtype || q->dtype != k_cache->dtype || q->dtype != v_cache->dtype)
    return PD_EDTYPE;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return PD_EINVAL;
  // the plan: its work list on the device, its sizes from paged_prefill_plan
  if (info->num_items < 0 || info->num_items > INT32_MAX || info->tile_rows != rows ||
      info->num_split_tiles < 0 || info->num_slots < 0 || info->max_segments != kMaxSegments)
    return PD_EINVAL;
  if (work->ndim != 2 || work->shape[0] != info->num_items || work->shape[1] != 8 ||
      work->stride[1] != 1 || work->stride[0] != 8 || (info->num_items > 0 && !work->data) ||
      (reinterpret_cast<uintptr_t>(work->data) & 15u) != 0)
    return PD_EINVAL;
  if (S == 0 || T == 0 || info->num_items == 0) return PD_OK;

  int num_sms = 0;
  unsigned int *status = nullptr;
  if ((rc = device_check(&num_sms, &status)) != PD_OK) return rc;
  PrefillShape sh;
  if ((rc = prefill_shape(head_size, &sh)) != PD_OK) return rc;

  Params p{};
  // split tiles need scratch: counters for every (split tile, kv head) and
  // partials for every (slot, kv head)
  if (info->num_split_tiles > 0) {
    if (!scratch || !scratch->data) return PD_ESCRATCH;
    const int64_t cbytes = round256(scratch->counter_slots * 4);
    const int64_t parts = (int64_t)info->num_slots * num_kv_heads;
    const int64_t acc = round256(parts * rows * head_size * 4);
    const int64_t ml = round256(parts * rows * 2 * 4);
    if (scratch->counter_slots < 2LL * info->num_split_tiles * num_kv_heads ||
        (int64_t)scratch->bytes < cbytes + acc + ml)
      return PD_ESCRATCH;
    char *base = static_cast<char *>(scratch->data);
    p.counters = reinterpret_cast<int *>(base);
    p.part_acc = reinterpret_cast<float *>(base + cbytes);
    p.part_ml = reinterpret_cast<float *>(base + cbytes + acc);
  }

  CUtensorMap tk, tv;
  if ((rc = cache_tensor_map(k_cache, layout, &tk, sh.path == 5)) != PD_OK) return rc;
  if ((rc = cache_tensor_map(v_cache, layout, &tv)) != PD_OK) return rc;

  p.q = q->data;
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.out = out->data;
  p.o_s0 = out->stride[0];
  p.o_s1 = out->stride[1];
  p.block_table = static_cast<const int32_t *>(block_table->data);
  p.bt_stride = block_table->stride[0];
  p.bt_width = (int)block_table->shape[1];
  p.seq_lens = static_cast<const int32_t *>(seq_lens->data);
  p.query_start = static_cast<const int32_t *>(query_start->data);
  p.num_tokens = (int)T;
  p.num_pool_blocks = (int)k_cache->shape[0];
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = num_q_heads / num_kv_heads;
  p.M = 1 << 30;  // a request's query length is not bounded here
  p.P = page_size;
  p.window = window;
  p.layout = layout;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.R = 1 << 30;
  p.rg = 1;
  p.rows_cta = rows;
  p.NT = sh.NT;
  p.KG = sh.KG;
  p.NS = sh.NS;
  p.seg_blocks = 1;
  p.max_seg = 1;
  p.CS = 1;
  p.max_parts = kMaxSegments;
  p.status = status;
  p.epi_floats = sh.epi / 4;
  p.coop = 0;
  p.mergers = 1;
  p.wait_limit_ns = 1000000000ull;
  p.num_seqs = (int)S;
  p.work = static_cast<const int32_t *>(work->data);
  p.pf_groups = info->num_split_tiles;
  p.pf_slots = info->num_slots;

  Launch l;
  l.grid = dim3((unsigned)info->num_items, (unsigned)num_kv_heads, 1);
  l.block = dim3(sh.threads, 1, 1);
  l.smem = sh.smem;
  l.cluster = 1;
  l.cooperative = 0;
  if (num_kv_heads > 65535) return PD_EINVAL;
  cudaError_t e = launch_mma(head_size, q->dtype == PD_BF16, sh.path, tk, tv, p, l,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  return PD_OK;
}

}  // extern "C"
