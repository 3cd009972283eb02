// C ABI of the paged decode-attention library: argument checks, the launch
// plan (segments, clusters, warp groups, ring stages), TMA tensor maps of
// the paged caches, scratch handling and the device status word.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "paged_decode.h"
#include "pd_internal.h"
#include "pd_ptx.cuh"

namespace pd {

__device__ unsigned int g_status;  // PD_DEV_* bits; read by paged_decode_device_status

namespace {

constexpr int kVersion = 10300;  // 1.3.0
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block on sm_100-class parts
constexpr int kMaxDevices = 64;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Device facts (cached per device).
struct DeviceInfo {
  int ok = 0;        // 1 = sm_103 device
  int num_sms = 0;
  unsigned int *status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PD_ENODEV;
  }
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PD_ENODEV;
    }
    if (major != 10 || minor != 3) return PD_ENODEV;  // built for sm_103a only
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) {
      cudaGetLastError();
      return PD_ECUDA;
    }
    d.num_sms = sms;
    d.status = static_cast<unsigned int *>(ptr);
    d.ok = 1;
  }
  *out = d;
  return PD_OK;
}

// ---------------------------------------------------------------------------
// TMA tensor maps of the caches, cached by (address, shape, strides).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

struct MapKey {
  const void *ptr;
  int layout;
  int one_box;
  int64_t dims[4];
  int64_t strides[3];
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && layout == o.layout && one_box == o.one_box &&
           std::memcmp(dims, o.dims, sizeof dims) == 0 &&
           std::memcmp(strides, o.strides, sizeof strides) == 0;
  }
};
struct MapEntry {
  int dev = -1;
  MapKey key{};
  CUtensorMap map;
};
constexpr int kMapCache = 64;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
std::mutex g_map_mu;

// One copy moves one 16-token block of one kv head of one page, all D dims:
// dims (innermost first) = d within a 128-byte row (64), token, 128-byte row
// of the head dim (D/64, stride 128 B), kv head, page.  The copy lands as
// [D/64][16 tokens][128 B] with the 128-byte swizzle, the layout the
// consumers' ldmatrix reads.  A TMA copy has a fixed per-copy cost (2 KiB
// boxes stream at ~33 GB/s per SM on GB300); one copy per block is 32*D
// bytes (4 KiB at D = 128, 16 KiB at D = 512).
int encode_cache_map(const pd_tensor *t, int layout, CUtensorMap *out, bool one_box = false) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  if (!g_encode) return PD_ECUDA;
  int dev = 0;
  cudaGetDevice(&dev);
  // NHD [NB, P, Hkv, D]; HND [NB, Hkv, P, D]
  const int ti = layout == PD_NHD ? 1 : 2, hi = layout == PD_NHD ? 2 : 1;
  MapKey key{};
  key.ptr = t->data;
  key.layout = layout;
  key.one_box = one_box ? 1 : 0;
  for (int i = 0; i < 4; ++i) key.dims[i] = t->shape[i];
  for (int i = 0; i < 3; ++i) key.strides[i] = t->stride[i];
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (auto &e : g_maps)
    if (e.dev == dev && e.key == key) {
      *out = e.map;
      return PD_OK;
    }
  const int64_t D = t->shape[3];
  cuuint64_t dims[5] = {64, (cuuint64_t)t->shape[ti], (cuuint64_t)(D / 64),
                        (cuuint64_t)t->shape[hi], (cuuint64_t)t->shape[0]};
  cuuint64_t strides[4] = {(cuuint64_t)t->stride[ti] * 2, 128, (cuuint64_t)t->stride[hi] * 2,
                           (cuuint64_t)t->stride[0] * 2};  // bytes
  // a copy lands a 16-key block with all of its D/64 128-byte rows, or
  // (one_box) one 64-dim box of it
  cuuint32_t box[5] = {64, (cuuint32_t)kBlockKeys, one_box ? 1u : (cuuint32_t)(D / 64), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUtensorMap m;
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, t->data, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return PD_EALIGN;
  MapEntry &e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  e.dev = dev;
  e.key = key;
  e.map = m;
  *out = m;
  return PD_OK;
}

// ---------------------------------------------------------------------------
// Argument checks.
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_rows_tensor(const pd_tensor *t, int64_t rows, int Hq, int D) {
  if (!t || !t->data || t->ndim != 3) return PD_EINVAL;
  if (t->shape[0] != rows || t->shape[1] != Hq || t->shape[2] != D) return PD_EINVAL;
  if (t->dtype != PD_F16 && t->dtype != PD_BF16) return PD_EDTYPE;
  if (t->stride[2] != 1) return PD_EALIGN;
  if (t->stride[0] % 8 != 0 || t->stride[1] % 8 != 0 || !aligned16(t->data)) return PD_EALIGN;
  if (t->stride[0] < 0 || t->stride[1] < 0) return PD_EINVAL;
  return PD_OK;
}

int check_cache(const pd_tensor *t, int layout, int Hkv, int P, int D) {
  if (!t || !t->data || t->ndim != 4) return PD_EINVAL;
  const int64_t hdim = layout == PD_NHD ? t->shape[2] : t->shape[1];
  const int64_t pdim = layout == PD_NHD ? t->shape[1] : t->shape[2];
  if (t->shape[0] < 1 || hdim != Hkv || pdim != P || t->shape[3] != D) return PD_EINVAL;
  if (t->dtype != PD_F16 && t->dtype != PD_BF16) return PD_EDTYPE;
  if (t->stride[3] != 1) return PD_EALIGN;
  for (int i = 0; i < 3; ++i) {
    if (t->stride[i] <= 0) return PD_EINVAL;
    if (t->stride[i] % 8 != 0) return PD_EALIGN;  // TMA: strides are multiples of 16 bytes
  }
  if (!aligned16(t->data)) return PD_EALIGN;
  if (t->shape[0] > INT32_MAX) return PD_EINVAL;
  return PD_OK;
}

// ---------------------------------------------------------------------------
// The launch plan.
struct PlanOut {
  pd_plan pub;
  int nt, kg, ns;
};

int make_plan(int S, int Hq, int Hkv, int D, int P, int M, int window, int bt_width, int num_sms,
              const pd_scratch *scratch, const pd_options *opts, pd_plan *plan) {
  pd_options o{};
  if (opts) o = *opts;
  if (S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || P <= 0 || P % kBlockKeys != 0 ||
      window < 0 || bt_width < 1 || num_sms <= 0)
    return PD_EINVAL;
  if (D != 64 && D != 128 && D != 256 && D != 512) return PD_EHEAD;
  if (M < 1 || M > 8) return PD_EQLEN;
  // path: 0 = auto (mma.sync), 1 = mma.sync, 2 = warp dot products (D <=
  // 256, one 8-row n-tile per CTA), 3 = tcgen05 with tensor memory (D <= 256)
  if (o.path < 0 || o.path > 3) return PD_EINVAL;
  if (o.wait_limit_us < 0) return PD_EINVAL;
  if (o.early_reads != 0 && o.early_reads != 1) return PD_EINVAL;
  if (o.mergers < 0 || (o.mergers & (o.mergers - 1)) != 0) return PD_EINVAL;
  const bool tc = o.path == 3, dot = o.path == 2;
  if ((tc || dot) && D > 256) return PD_EINVAL;
  if ((tc || dot) && o.cluster > 1) return PD_EINVAL;
  const int G = Hq / Hkv, R = G * M;
  // One sequence: at most 16 packed rows per CTA.  Every n-tile warp of a
  // warp group reads the whole stage from shared memory, so more rows per
  // CTA cost shared-memory bandwidth and per-warp latency, while the row
  // groups of one segment, resident together, read the same pages at about
  // the same time (mostly L2 hits).  Measured at D=512, 64 rows, 32k keys:
  // 81 -> 52 us.  A batch runs several waves and is bound by HBM, where a
  // second read of the pages costs more than it saves: up to 64 rows.
  // (the tensor-memory path takes 16 rows per CTA, four copies of them)
  const int64_t rows_max = dot ? 8 : (S <= 1 || tc) ? 16 : 64;
  int rg = o.row_groups > 0
               ? o.row_groups
               : (int)std::min<int64_t>(kMaxRowGroups, std::max<int64_t>(1, cdiv(R, rows_max)));
  if (rg > kMaxRowGroups || rg > R) return PD_EINVAL;
  const int rows_cta = (int)cdiv(R, rg);
  const int NT = (int)cdiv(rows_cta, 8);
  if (NT > kMaxConsumerWarps) return PD_EINVAL;
  const int TB = kStageBytes / 2 / (kBlockKeys * D * 2);
  // (the dot path's P buffers grow with the warp groups: sized for the
  // most it may use)
  const int kg_dot = o.key_groups > 0 ? o.key_groups : 3;
  const int fixed = tc ? smem_bytes_tc(D, 0) : dot ? smem_bytes_dot(D, kg_dot, 0) : smem_bytes(D, NT, 0);
  const int ns_max = std::min(8, (kSmemLimit - fixed - 16 * 8) / kStageBytes);
  // dead ring (+ Q and P tiles) available to the epilogue with NS stages
  auto epi_bytes = [&](int ns) { return tc ? epilogue_bytes_tc(D, ns) : epilogue_bytes(D, NT, ns); };
  if (ns_max < 1) return PD_EINVAL;
  // warp groups take alternate stages; with >= 2 stages each, a group's next
  // stage loads while it computes on the current one (3 groups measured
  // fastest for up to 16 packed rows)
  int KG = o.key_groups > 0 ? o.key_groups : (NT <= 2 ? 3 : std::max(1, kMaxConsumerWarps / NT));
  if (tc) KG = 4;  // four copies of the rows, each over a quarter of the keys
  int NS = 0;
  while (true) {
    // (the tensor-memory path's copies share every stage: any count)
    NS = o.stages > 0 ? o.stages : (tc ? ns_max : (ns_max / KG) * KG);
    // the warp groups' partials (KG copies of NT*8 x D fp32) must fit in the
    // dead ring at the end; fewer groups when they do not
    if (o.key_groups > 0 || KG == 1 || NS < 1 ||
        epilogue_floats(D, NT, KG, 1, 1) * 4 <= epi_bytes(NS))
      break;
    KG /= 2;
  }
  if (!tc && NT * KG > kMaxConsumerWarps) return PD_EINVAL;
  if (NS < 1 || NS > ns_max || (!tc && NS % KG != 0) || (NS < 2 && o.stages == 0))
    return PD_EINVAL;

  // KV blocks (16 keys) a (sequence, kv head, row group) can span at most.
  int64_t nb_max = cdiv((int64_t)bt_width * P, kBlockKeys);
  if (window > 0) nb_max = std::min<int64_t>(nb_max, cdiv(window + M - 1, kBlockKeys) + 1);
  const int64_t units = (int64_t)S * Hkv * rg;
  const int64_t target = o.max_ctas_hint > 0 ? o.max_ctas_hint : num_sms;
  // a segment reads at least one and a half stages (~10 segments of 1k keys
  // measured best at D=128: 9.9 -> 9.4 us), and at least four keys per
  // packed row so its partial stays small next to the keys it read
  const int64_t min_seg_blocks = std::max<int64_t>({4, (3LL * TB) / 2, 2LL * NT});
  int64_t nseg;
  if (o.segments > 0) {
    nseg = o.segments;
  } else if (S <= 1) {
    // (a windowed call split into row groups is latency-bound: finer
    // segments, two blocks each, measured faster: 512-key window, D=256,
    // M=4, 2 row groups: 8 segments 9.4 us, 17 segments 8.9 us; with one
    // row group, M=1, they measured slower: 7.8 against 7.3 us)
    const int64_t seg_floor = (window > 0 && rg > 1) ? 2 : min_seg_blocks;
    nseg = std::max<int64_t>(1, target / std::max<int64_t>(units, 1));
    nseg = std::min(nseg, std::max<int64_t>(1, nb_max / seg_floor));
    // With 1-8 MiB of K and V per (sequence, kv head), fewer and longer
    // segments: the merge's parts then cost more than the shorter stream
    // saves.  Measured at D=128, 8 kv heads, M=1 and 4 (us per call,
    // segments per head): 2k keys 9.3 (12) against 10.1 (19); 4k 11.4 (14)
    // against 12.1 (19); 8k 14.3 (16) against 14.7 (19); 16k and 32k as
    // good or better with 19.  The CTAs are capped at (12 + 7/3 log2(MiB))
    // / 19 of the resident ones, which passes through those optima.
    const int64_t unit_bytes = nb_max * kBlockKeys * 4LL * D;  // K + V of a unit
    if (!(window > 0 && rg > 1) && unit_bytes >= (1LL << 20) && unit_bytes < (8LL << 20)) {
      const double frac = (12.0 + 7.0 / 3.0 * std::log2((double)unit_bytes / (1 << 20))) / 19.0;
      const int64_t cap = (int64_t)(frac * (double)target) / std::max<int64_t>(units, 1);
      nseg = std::min(nseg, std::max<int64_t>(1, cap));
    }
    // Below 1 MiB (no window) the optimum keeps about 85 KiB per segment,
    // the size the rule above gives at 1 MiB (1k keys, 512 KiB per head: 6
    // segments 6.8 us at M=1 and 7.3 at M=4, against 7.1 and 7.7 with 10)
    if (window == 0 && unit_bytes < (1LL << 20))
      nseg = std::min(nseg, std::max<int64_t>(2, unit_bytes / ((1LL << 20) / 12)));
    // a CTA that would move at most kNoSplitBytes of K and V alone is not
    // split: the merge's round trips cost more than the stream time a split
    // saves (300 keys at D=128: 5.8 us unsplit, 6.6 us in 3 segments)
    if (nb_max * kBlockKeys * 4LL * D <= kNoSplitBytes) nseg = 1;
  } else {
    // a batch: lengths are only known on the device; aim at ~1.5 waves of
    // equal segments assuming an average length of half the table width
    // (fewer, longer segments measured faster than ~4 waves: 300 -> 288 us
    // for 64 sequences of U[1, 16384] keys at D=256; the last-arriver merge
    // of a (sequence, kv head) then reads fewer parts)
    // Segments are also capped at 384 blocks (6144 keys): with many groups
    // the estimate alone gives segments of ~9k keys, and the last wave of
    // such long CTAs runs unbalanced (32 requests x 8 kv heads of 1k-16k
    // keys: 2 segments 220 us, 3-6 segments 205 us; 64 sequences x 2 kv
    // heads at D=256 keep their 4).
    const int64_t est = std::max<int64_t>(1, units * nb_max / 2);
    int64_t sb = std::max(min_seg_blocks, cdiv(2 * est, 3 * target));
    sb = std::min(sb, std::max<int64_t>(min_seg_blocks, kMaxBatchSegBlocks));
    nseg = cdiv(nb_max, sb);
  }
  nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, nb_max));
  const int64_t part_floats = 8LL * NT * D;  // one partial's acc
  int CS = o.cluster > 0 ? o.cluster : 1;
  // A cooperative merger needs room for one part's (m, l) and share at least
  // (it pulls the parts a window at a time; K >= 2 mergers).
  const int64_t coop_floats = 16LL * NT + 8LL * NT * D / 2 + 64;
  const bool coop_possible = o.merge != 1 && (int64_t)S * Hkv * rg * nseg <= num_sms &&
                             coop_floats * 4 <= epi_bytes(NS);
  // Clusters only in the one-wave regime (a batch runs several waves, where
  // the last-arriving CTA's merge overlaps other CTAs' work) and only when
  // the cooperative merge is not possible (it measured faster).
  if (o.cluster == 0 && !tc && !dot && S <= 1 && nseg >= 8 && nseg * part_floats * 4 > (256 << 10) &&
      !coop_possible)
    CS = 8;
  if (CS != 1 && CS != 2 && CS != 4 && CS != 8) return PD_EINVAL;
  if (CS > 1) {
    if (o.segments > 0) {
      if (nseg % CS) return PD_EINVAL;
    } else {
      nseg = std::max<int64_t>(CS, (nseg / CS) * CS);
    }
  }
  int64_t max_parts = nseg > CS ? nseg / CS : 0;  // partial slots per group (0: none)

  // Scratch: counters for every group, partials for every cluster.
  const int64_t counter_need = 2 * units;  // arrivals and finished mergers per group
  auto partial_bytes = [&](int64_t parts) -> int64_t {
    const int64_t acc = ((units * parts * part_floats * 4) + 255) / 256 * 256;
    const int64_t ml = ((units * parts * 8LL * NT * 2 * 4) + 255) / 256 * 256;
    return acc + ml;
  };
  int64_t avail = -1;
  if (scratch && scratch->data) {
    const int64_t cbytes = (scratch->counter_slots * 4 + 255) / 256 * 256;
    avail = (int64_t)scratch->bytes - cbytes;
    if (scratch->counter_slots < counter_need) avail = -1;
  }
  if (max_parts > 0) {
    if (avail < 0 || partial_bytes(max_parts) > avail) {
      if (o.segments > 0) return PD_ESCRATCH;
      // shrink the split to what the scratch holds (one cluster needs none)
      int64_t fit = 0;
      if (avail > 0) {
        int64_t lo = 0, hi = max_parts;
        while (lo < hi) {
          const int64_t mid = (lo + hi + 1) / 2;
          if (partial_bytes(mid) <= avail) lo = mid; else hi = mid - 1;
        }
        fit = lo;
      }
      if (fit >= 2) {
        max_parts = fit;
        nseg = max_parts * CS;
      } else {
        if (CS == 1) {
          nseg = 1;
        } else {
          nseg = CS;
        }
        max_parts = 0;
      }
    }
  }
  // The epilogue must fit in the ring + Q region.
  while (max_parts > 0 &&
         epilogue_floats(D, NT, KG, CS, (int)max_parts) * 4 > epi_bytes(NS)) {
    if (o.segments > 0) return PD_EINVAL;
    max_parts = max_parts - 1;
    nseg = max_parts > 1 ? max_parts * CS : CS;
    if (max_parts <= 1) max_parts = 0;
  }
  if (epilogue_floats(D, NT, KG, CS, 1) * 4 > epi_bytes(NS)) return PD_EINVAL;
  const int64_t seg_blocks = cdiv(nb_max, nseg);
  // Merge.  A grid that fits on the GPU at once (one CTA per SM) can be
  // launched cooperatively; then the last K arrivals of a group each merge
  // one D/K slice instead of the last arrival merging all of it alone.
  if (o.merge < 0 || o.merge > 2) return PD_EINVAL;
  const bool coop_ok = max_parts > 1 && CS == 1 && (int64_t)S * Hkv * rg * nseg <= num_sms &&
                       coop_floats * 4 <= epi_bytes(NS);
  int merge = max_parts > 1 ? 1 : 0, mergers = 0;
  if (coop_ok && o.merge != 1) {
    merge = 2;
    // K mergers, each taking a slice of D / K >= 8 columns of every part: K a
    // power of two <= min(D / 8, 64, parts), and no larger than it takes to
    // keep a merger's share of the parts near 8192 fp32 elements (at least
    // 4).  A merger's time is mostly round trips until its share grows past
    // that, while every extra merger holds an SM the next call could start
    // on (measured at D = 128, 4k-32k keys: 4 mergers for 4-12 rows, 8 for
    // 16 rows at 16k, 2-5 % faster per call than 16; at D = 512 with 152
    // parts the bound stays at 64)
    const int64_t share = max_parts * rows_cta * (int64_t)D;
    int64_t by_work = 4;
    while (by_work * 8192 < share) by_work *= 2;
    mergers = 1;
    while (2 * mergers <= std::min<int64_t>({(int64_t)D / 8, 64, max_parts, by_work})) mergers *= 2;
    if (o.mergers > 0) mergers = std::min(mergers, o.mergers);
  } else if (o.merge == 2 && max_parts > 1) {
    return PD_EINVAL;  // the grid does not fit at once, or a cluster was asked for
  }
  // launched as (segments, kv heads x row groups, sequences)
  if ((int64_t)Hkv * rg * nseg > INT32_MAX || (int64_t)Hkv * rg > 65535 || S > 65535)
    return PD_EINVAL;

  plan->path = tc ? 3 : dot ? 2 : 1;
  plan->merge = merge;
  plan->mergers = mergers;
  plan->rows = R;
  plan->row_groups = rg;
  plan->rows_per_cta = rows_cta;
  plan->n_tiles = NT;
  plan->key_groups = KG;
  plan->stages = NS;
  plan->seg_blocks = (int)seg_blocks;
  plan->max_segments = (int)nseg;
  plan->cluster = CS;
  plan->max_parts = (int)max_parts;
  plan->grid_x = (int)(Hkv * rg * nseg);
  plan->grid_y = S;
  plan->block_threads = tc ? kTcThreads : 32 * (NT * KG + 1);
  plan->smem_bytes = tc ? smem_bytes_tc(D, NS) : dot ? smem_bytes_dot(D, KG, NS) : smem_bytes(D, NT, NS);
  plan->scratch_needed = max_parts > 0 ? partial_bytes(max_parts) : 0;
  return PD_OK;
}

int element_dtype_ok(const pd_tensor *t, int want) { return t->dtype == want; }

int attn_impl(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
              const pd_tensor *block_table, const pd_tensor *seq_lens,
              const pd_tensor *query_start, pd_tensor *out, int num_q_heads, int num_kv_heads,
              int head_size, int page_size, int max_query_len, int window, float scale,
              int layout, pd_scratch *scratch, void *stream, const pd_options *opts) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return PD_EINVAL;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return PD_EINVAL;
  if (head_size != 64 && head_size != 128 && head_size != 256 && head_size != 512) return PD_EHEAD;
  if (max_query_len < 1 || max_query_len > 8) return PD_EQLEN;
  if (page_size <= 0 || page_size % kBlockKeys != 0) return PD_EINVAL;
  if (window < 0 || !std::isfinite(scale)) return PD_EINVAL;
  if (layout != PD_NHD && layout != PD_HND) return PD_EINVAL;
  if (seq_lens->ndim != 1 || !seq_lens->data || seq_lens->stride[0] != 1) return PD_EINVAL;
  if (!element_dtype_ok(seq_lens, PD_I32) || !element_dtype_ok(block_table, PD_I32)) return PD_EDTYPE;
  const int64_t S = seq_lens->shape[0];
  if (S < 0) return PD_EINVAL;
  if (block_table->ndim != 2 || !block_table->data || block_table->shape[0] != S ||
      block_table->shape[1] < 1 || block_table->stride[1] != 1 || block_table->stride[0] < 0)
    return PD_EINVAL;
  // rows of q and out: S * M (uniform), or any count T with query_start
  // [S + 1] giving each sequence's first row (variable query lengths)
  int64_t T = S * max_query_len;
  if (query_start) {
    if (query_start->ndim != 1 || !query_start->data || query_start->shape[0] != S + 1 ||
        query_start->stride[0] != 1)
      return PD_EINVAL;
    if (!element_dtype_ok(query_start, PD_I32)) return PD_EDTYPE;
    if (!q->data || q->ndim != 3) return PD_EINVAL;
    T = q->shape[0];
    if (T < 0 || T > INT32_MAX) return PD_EINVAL;
  }
  int rc;
  if ((rc = check_rows_tensor(q, T, num_q_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_rows_tensor(out, T, num_q_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_cache(k_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK) return rc;
  if ((rc = check_cache(v_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK) return rc;
  if (q->dtype != out->dtype || q->dtype != k_cache->dtype || q->dtype != v_cache->dtype)
    return PD_EDTYPE;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return PD_EINVAL;
  if (block_table->shape[1] > INT32_MAX || block_table->shape[1] * (int64_t)page_size > INT32_MAX)
    return PD_EINVAL;
  if (S == 0 || T == 0) return PD_OK;

  DeviceInfo dev;
  if ((rc = device_info(&dev)) != PD_OK) return rc;
  pd_plan plan;
  rc = make_plan((int)S, num_q_heads, num_kv_heads, head_size, page_size, max_query_len, window,
                 (int)block_table->shape[1], dev.num_sms, scratch, opts, &plan);
  if (rc != PD_OK) return rc;
  if (query_start && plan.path == 3) return PD_EINVAL;  // not built for variable lengths

  CUtensorMap tk, tv;
  // (the tensor-memory path lands K box-major: one box per 64 dims)
  if ((rc = encode_cache_map(k_cache, layout, &tk, plan.path == 3)) != PD_OK) return rc;
  if ((rc = encode_cache_map(v_cache, layout, &tv)) != PD_OK) return rc;

  Params p{};
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
  p.query_start = query_start ? static_cast<const int32_t *>(query_start->data) : nullptr;
  p.num_tokens = (int)T;
  p.num_pool_blocks = (int)k_cache->shape[0];
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = num_q_heads / num_kv_heads;
  p.M = max_query_len;
  p.P = page_size;
  p.window = window;
  p.layout = layout;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.R = plan.rows;
  p.rg = plan.row_groups;
  p.rows_cta = plan.rows_per_cta;
  p.NT = plan.n_tiles;
  p.KG = plan.key_groups;
  p.NS = plan.stages;
  p.seg_blocks = plan.seg_blocks;
  p.max_seg = plan.max_segments;
  p.CS = plan.cluster;
  p.max_parts = std::max(plan.max_parts, 1);
  p.status = dev.status;
  p.coop = plan.merge == 2 ? 1 : 0;
  p.mergers = plan.mergers > 0 ? plan.mergers : 1;
  p.num_seqs = (int)S;
  p.work = nullptr;
  p.early = (opts && opts->early_reads) ? 1 : 0;
  p.wait_limit_ns = (opts && opts->wait_limit_us > 0)
                        ? (unsigned long long)opts->wait_limit_us * 1000ull
                        : kWaitLimitNs;
  p.epi_floats = (plan.path == 3 ? epilogue_bytes_tc(head_size, plan.stages)
                                  : epilogue_bytes(head_size, plan.n_tiles, plan.stages)) / 4;
  if (plan.max_parts > 0) {
    char *base = static_cast<char *>(scratch->data);
    const int64_t cbytes = (scratch->counter_slots * 4 + 255) / 256 * 256;
    const int64_t units = S * num_kv_heads * plan.row_groups;
    const int64_t acc_bytes =
        (units * p.max_parts * 8LL * plan.n_tiles * head_size * 4 + 255) / 256 * 256;
    p.counters = reinterpret_cast<int *>(base);
    p.part_acc = reinterpret_cast<float *>(base + cbytes);
    p.part_ml = reinterpret_cast<float *>(base + cbytes + acc_bytes);
  }

  Launch l;
  // (segment, kv head x row group, sequence): plan.grid_x CTAs per sequence
  l.grid = dim3(plan.max_segments, num_kv_heads * plan.row_groups, plan.grid_y);
  l.block = dim3(plan.block_threads, 1, 1);
  l.smem = plan.smem_bytes;
  l.cluster = plan.cluster;
  // The cooperative merge needs every CTA of the grid resident at once; the
  // planner sizes such a grid to fit.  Launched with the cooperative
  // attribute, a grid does not start before all of its CTAs fit, so under
  // early reads a grid that fills more than ~58 % of the SMs is launched
  // plainly: its CTAs then start, and stream the older pages, on the SMs the
  // previous call frees while that call's mergers finish (measured at 32 / 8
  // heads, D = 128, 2k-32k keys: 0.4-1.5 us less per call; with 80 CTAs the
  // cooperative launch was 1.1 us faster).  This grid never waits on a later
  // one (the next call launches only once every CTA of this one has
  // started), so all of its CTAs still become resident; a kernel on another
  // stream that held SMs for longer than the mergers' wait limit would end
  // in PD_DEV_WAIT_TIMEOUT.
  const int64_t ctas = (int64_t)plan.max_segments * num_kv_heads * plan.row_groups * plan.grid_y;
  l.cooperative = plan.merge == 2 && !(p.early && ctas * 100 > 58LL * dev.num_sms) ? 1 : 0;
  cudaError_t e = launch_mma(head_size, q->dtype == PD_BF16, plan.path, tk, tv, p, l,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  return PD_OK;
}

}  // namespace

int device_check(int *num_sms, unsigned int **status) {
  DeviceInfo d;
  const int rc = device_info(&d);
  if (rc != PD_OK) return rc;
  if (num_sms) *num_sms = d.num_sms;
  if (status) *status = d.status;
  return PD_OK;
}

int check_cache_tensor(const pd_tensor *t, int layout, int Hkv, int P, int D) {
  return check_cache(t, layout, Hkv, P, D);
}

int check_rows(const pd_tensor *t, int64_t rows, int Hq, int D) {
  return check_rows_tensor(t, rows, Hq, D);
}

int cache_tensor_map(const pd_tensor *t, int layout, CUtensorMap *out, bool one_box) {
  return encode_cache_map(t, layout, out, one_box);
}

}  // namespace pd

using namespace pd;

extern "C" {

size_t paged_decode_scratch_bytes(int max_num_seqs, int num_q_heads, int num_kv_heads,
                                  int head_size, int max_query_len, int max_splits) {
  if (max_num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || max_query_len < 1 || max_query_len > 8 ||
      max_splits < 0)
    return 0;
  if (head_size != 64 && head_size != 128 && head_size != 256 && head_size != 512) return 0;
  const int64_t R = (int64_t)(num_q_heads / num_kv_heads) * max_query_len;
  // padded rows over all row groups, for the larger of the two row-group
  // rules of the planner (at most 64 rows per CTA for a batch, 16 for one
  // sequence)
  int64_t nt8 = 0;
  for (int64_t rows_max : {64, 16}) {
    const int64_t rg = std::min<int64_t>(kMaxRowGroups, std::max<int64_t>(1, cdiv(R, rows_max)));
    nt8 = std::max(nt8, rg * 8 * cdiv(cdiv(R, rg), 8));
  }
  const int64_t counters =
      ((int64_t)max_num_seqs * num_kv_heads * kCountersPerPair * 4 + 255) / 256 * 256;
  const int64_t parts = (int64_t)max_num_seqs * num_kv_heads * max_splits;
  const int64_t acc = (parts * nt8 * head_size * 4 + 255) / 256 * 256;
  const int64_t ml = (parts * nt8 * 2 * 4 + 255) / 256 * 256;
  return (size_t)(counters + acc + ml + 256);
}

int paged_decode_scratch_init(pd_scratch *scratch, void *data, size_t bytes, int max_num_seqs,
                              int num_kv_heads, void *stream) {
  if (!scratch || !data || max_num_seqs < 0 || num_kv_heads <= 0) return PD_EINVAL;
  if ((reinterpret_cast<uintptr_t>(data) & 255u) != 0) return PD_EALIGN;
  const int64_t slots = (int64_t)max_num_seqs * num_kv_heads * kCountersPerPair;
  const int64_t cbytes = (slots * 4 + 255) / 256 * 256;
  if ((int64_t)bytes < cbytes) return PD_ESCRATCH;
  scratch->data = data;
  scratch->bytes = bytes;
  scratch->counter_slots = slots;
  if (cbytes > 0 &&
      cudaMemsetAsync(data, 0, (size_t)cbytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  return PD_OK;
}

int paged_decode_attn(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
                      const pd_tensor *block_table, const pd_tensor *seq_lens, pd_tensor *out,
                      int num_q_heads, int num_kv_heads, int head_size, int page_size,
                      int max_query_len, int window, float scale, int layout,
                      pd_scratch *scratch, void *stream) {
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, nullptr, out, num_q_heads,
                   num_kv_heads, head_size, page_size, max_query_len, window, scale, layout,
                   scratch, stream, nullptr);
}

int paged_decode_attn_opts(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
                           const pd_tensor *block_table, const pd_tensor *seq_lens, pd_tensor *out,
                           int num_q_heads, int num_kv_heads, int head_size, int page_size,
                           int max_query_len, int window, float scale, int layout,
                           pd_scratch *scratch, void *stream, const pd_options *opts) {
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, nullptr, out, num_q_heads,
                   num_kv_heads, head_size, page_size, max_query_len, window, scale, layout,
                   scratch, stream, opts);
}

int paged_decode_attn_varlen(const pd_tensor *q, const pd_tensor *k_cache,
                             const pd_tensor *v_cache, const pd_tensor *block_table,
                             const pd_tensor *seq_lens, const pd_tensor *query_start,
                             pd_tensor *out, int num_q_heads, int num_kv_heads, int head_size,
                             int page_size, int max_query_len, int window, float scale,
                             int layout, pd_scratch *scratch, void *stream,
                             const pd_options *opts) {
  if (!query_start) return PD_EINVAL;
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, query_start, out, num_q_heads,
                   num_kv_heads, head_size, page_size, max_query_len, window, scale, layout,
                   scratch, stream, opts);
}

int paged_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                      int page_size, int max_query_len, int window, int block_table_width,
                      int num_sms, const pd_scratch *scratch, const pd_options *opts,
                      pd_plan *plan) {
  if (!plan) return PD_EINVAL;
  return make_plan(num_seqs, num_q_heads, num_kv_heads, head_size, page_size, max_query_len,
                   window, block_table_width, num_sms, scratch, opts, plan);
}

int paged_decode_device_status(unsigned int *status, int reset, void *stream) {
  if (!status) return PD_EINVAL;
  DeviceInfo dev;
  int rc = device_info(&dev);
  if (rc != PD_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, dev.status, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  if (reset && cudaMemsetAsync(dev.status, 0, sizeof v, st) != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  *status = v;
  return PD_OK;
}

const char *paged_decode_strerror(int code) {
  switch (code) {
    case PD_OK: return "ok";
    case PD_EINVAL: return "invalid argument (null pointer, size, shape, layout or option)";
    case PD_EDTYPE: return "unsupported or mismatched dtype (q, caches and out must share fp16 or bf16; block_table and seq_lens int32)";
    case PD_EHEAD: return "head_size must be 64, 128, 256 or 512";
    case PD_EQLEN: return "max_query_len must be in 1..8";
    case PD_EALIGN: return "misaligned tensor (16-byte rows and bases, innermost stride 1)";
    case PD_ESCRATCH: return "scratch missing, not initialised or too small";
    case PD_ECUDA: return "CUDA runtime error";
    case PD_ENODEV: return "no sm_103 CUDA device";
    default: return "unknown status";
  }
}

int paged_decode_version(void) { return kVersion; }

}  // extern "C"
