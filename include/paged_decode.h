/*
 * paged_decode.h — C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The operation (vllm.v1.attention.ops.rocm_rdna_hip, the decode entry point
 * `_Builtin.decode_attn(q, kv_cache, block_table, out, *scratch_and_args)`,
 * and vllm.v1.attention.backends.rocm_octave_attn, `RocmOctaveAttentionImpl
 * .forward` / `_decode`):
 *
 *   For every sequence s (L_s = seq_lens[s] keys, which include its M new
 *   query tokens), query token i in [0, M) and query head hq:
 *     h   = hq / G, G = Hq / Hkv             (contiguous GQA groups)
 *     n_i = L_s - M + i + 1                  (keys query i sees; the K
 *                                             length of rocm_octave_attn
 *                                             `_fill_query_maps`)
 *     keys k in [lo_i, n_i), lo_i = window ? max(0, n_i - window) : 0
 *                                            (window in keys, 0 = full
 *                                             causal: KernelVariant.window)
 *     K_k = k_cache[block_table[s][k / P]] at token k % P, kv head h
 *     out[s*M + i][hq] = softmax_k(scale * q . K_k) . V_k, fp32 arithmetic,
 *                        rounded to the input dtype; 0 if no key is visible.
 *
 * Split-KV (KernelVariant.max_segments, scratch_shapes, make_scratch): the
 * keys of one (sequence, kv head, row group) are cut into segments, one CTA
 * each; each writes unnormalised partials (acc, m, l) to the caller's
 * scratch, and the CTA that arrives last at a per-group counter merges them
 * and resets the counter to 0: the counters start every launch at zero.
 *
 * Threading and streams: every call is asynchronous on `stream`, performs
 * no host synchronisation and allocates nothing (no cudaMalloc, no host
 * allocation that outlives the call), so a call may be captured in a CUDA
 * graph.  A scratch buffer may serve one stream at a time: two calls in
 * flight on different streams with one scratch race on its counters.
 *
 * Errors: every function returns PD_OK (0) or a negative pd_status, checked
 * on the host before any launch.  Nothing falls back to another
 * implementation.  Faults the host cannot see (a page id outside the pool,
 * a seq_len beyond the block table, an internal wait that timed out) are
 * recorded in a device status word (paged_decode_device_status) and the
 * kernel clamps the access instead of faulting.
 */
#ifndef PAGED_DECODE_H
#define PAGED_DECODE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PD_API __attribute__((visibility("default")))
#else
#define PD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  q, the caches and out share one of PD_F16 / PD_BF16
 * (KernelVariant.__post_init__: fp16 or bf16 only); block_table and
 * seq_lens are PD_I32. */
typedef enum { PD_F16 = 0, PD_BF16 = 1, PD_I32 = 2, PD_F32 = 3 } pd_dtype;

/* Cache layouts (KernelVariant.layout: 0 = NHD, 1 = HND).
 *   PD_NHD: [num_blocks, page_size, num_kv_heads, head_size]
 *   PD_HND: [num_blocks, num_kv_heads, page_size, head_size]            */
typedef enum { PD_NHD = 0, PD_HND = 1 } pd_layout;

/* A strided view of device memory.  Strides are in elements; the innermost
 * (head_size) stride must be 1.  `data` is a device pointer; the library
 * never frees it or keeps it past the call. */
typedef struct pd_tensor {
  void *data;
  int32_t dtype; /* pd_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} pd_tensor;

/* Caller-owned split-KV scratch (make_scratch / scratch_bytes).  Filled by
 * paged_decode_scratch_init; the library reads the fields, never resizes or
 * frees `data`. */
typedef struct pd_scratch {
  void *data;             /* device memory, 256-byte aligned                  */
  size_t bytes;           /* its size                                          */
  int64_t counter_slots;  /* int32 counters at the start of data (set by init) */
} pd_scratch;

typedef enum {
  PD_OK = 0,
  PD_EINVAL = -1,    /* null pointer, size <= 0, Hq % Hkv != 0, shape or
                        descriptor mismatch, window < 0, page_size % 16 != 0 */
  PD_EDTYPE = -2,    /* not fp16/bf16, or q/k/v/out dtypes differ            */
  PD_EHEAD = -3,     /* head_size not in {64, 128, 256, 512}                 */
  PD_EQLEN = -4,     /* max_query_len < 1 or > 8                             */
  PD_EALIGN = -5,    /* a row or base not 16-byte aligned, inner stride != 1 */
  PD_ESCRATCH = -6,  /* scratch missing, not initialised or too small        */
  PD_ECUDA = -7,     /* a CUDA runtime call failed (launch, attribute, ...)  */
  PD_ENODEV = -8     /* no CUDA device, or not an sm_103 device              */
} pd_status;

/* Bits of the device status word. */
#define PD_DEV_WAIT_TIMEOUT 0x1u  /* an internal barrier wait gave up       */
#define PD_DEV_BAD_PAGE     0x2u  /* a block-table entry outside the pool   */
#define PD_DEV_BAD_SEQLEN   0x4u  /* seq_len > block-table width * page_size */
#define PD_DEV_BAD_QSTART   0x8u  /* query_start out of order or out of range */
#define PD_DEV_BAD_SCRATCH  0x10u /* a split-KV counter did not start the call at
                                     zero: the scratch served two overlapping
                                     calls, or a merger gave up waiting
                                     (PD_DEV_WAIT_TIMEOUT) in an earlier call;
                                     the groups concerned are not merged and
                                     the scratch must be initialised again */

#define PD_DEV_BAD_POSITION 0x20u /* paged_rope_cache_write: a position outside
                                     the cos/sin table (clamped into it)     */
#define PD_DEV_BAD_SLOT     0x40u /* paged_rope_cache_write: a slot past the
                                     pool's pages x page_size (not written)  */
#define PD_DEV_BAD_WORK     0x80u /* paged_prefill_attn: a work item outside
                                     the launch (skipped)                    */

/* int32 counters a scratch reserves per (sequence, kv head): an arrival
 * count and a finished-merger count for each of up to 8 row groups. */
#define PD_COUNTERS_PER_PAIR 16

/* Bytes of scratch for calls of up to `max_num_seqs` sequences
 * (scratch_bytes: 4 * (rows * D + 2 * rows + counters) per sequence).
 * `max_splits` is the most KV segments (split-KV partials) one
 * (sequence, kv head) may use; a larger buffer allows more segments.
 * Returns 0 on invalid arguments. */
PD_API size_t paged_decode_scratch_bytes(int max_num_seqs, int num_q_heads, int num_kv_heads,
                                  int head_size, int max_query_len, int max_splits);

/* Prepare a scratch buffer: record its counter area (PD_COUNTERS_PER_PAIR
 * int32 per (sequence, kv head)) and zero the counters once, asynchronously
 * on `stream` (as the RDNA backend's make_scratch does: the calls leave them
 * at zero afterwards).  `data` must stay allocated while calls use it.
 * Call it outside graph capture.  Call it again on a buffer after a call
 * that reported PD_DEV_WAIT_TIMEOUT or PD_DEV_BAD_SCRATCH: a merger that
 * gave up leaves its group's counter deliberately out of range, and every
 * later call on that buffer skips the merge of that group (reporting
 * PD_DEV_BAD_SCRATCH) until the counters are zeroed again. */
PD_API int paged_decode_scratch_init(pd_scratch *scratch, void *data, size_t bytes, int max_num_seqs,
                              int num_kv_heads, void *stream);

/* The decode call.
 *   q           [S*M, Hq, D]  fp16/bf16, rows of sequence s at s*M .. s*M+M-1
 *   k_cache     NHD or HND pool (any strides, innermost 1)
 *   v_cache     same shape and dtype as k_cache; may alias k_cache + D with
 *               the packed K|V strides of expected_kv_cache_strides
 *   block_table [S, W] int32, logical page -> physical page
 *   seq_lens    [S] int32 device array: keys per sequence, including the M
 *               new tokens (0 = empty slot: its rows are written as zeros)
 *   out         [S*M, Hq, D], same dtype as q; may not overlap the inputs
 *   scale       multiplies q . k before the softmax (usually 1/sqrt(D))
 *   scratch     from paged_decode_scratch_init; NULL allowed when a call
 *               needs no split (then every (sequence, kv head) is one CTA)
 *   stream      cudaStream_t (NULL = the legacy default stream)
 * The library reads block_table only for pages that hold visible keys, so
 * entries before a sliding window's first page may be anything. */
PD_API int paged_decode_attn(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
                      const pd_tensor *block_table, const pd_tensor *seq_lens, pd_tensor *out,
                      int num_q_heads, int num_kv_heads, int head_size, int page_size,
                      int max_query_len, int window, float scale, int layout,
                      pd_scratch *scratch, void *stream);

/* Launch knobs (KernelVariant's max_segments / row_groups / waves /
 * dot_product knobs, chosen per call here).  Zero means "choose". */
typedef struct pd_options {
  int segments;      /* KV segments per (sequence, kv head, row group)        */
  int row_groups;    /* CTAs sharing one kv head's packed query rows          */
  int key_groups;    /* warp groups of a CTA that take alternate KV tiles     */
  int stages;        /* shared-memory ring stages (32 KiB each)               */
  int cluster;       /* thread-block cluster size of the merge (1, 2, 4, 8)   */
  int path;          /* 0 = auto (= 1), 1 = mma.sync, 2 = warp dot products in
                        fp32 (D <= 256, 8 packed rows per CTA, more in row
                        groups), 3 = tcgen05 MMAs with tensor memory
                        (D <= 256, 16 packed rows per CTA)                     */
  int max_ctas_hint; /* CTAs the split aims for (0 = the SM count)            */
  int merge;         /* split-KV merge: 0 = auto, 1 = the last-arriving CTA,
                        2 = the last K arrivals of a co-resident (cooperative)
                        grid, one D/K slice each                                */
  int wait_limit_us; /* how long a cooperative merger waits for the remaining
                        arrivals before it gives up and reports
                        PD_DEV_WAIT_TIMEOUT (0 = one second); for tests of
                        that path                                              */
  int early_reads;   /* 1 = the caller vouches that block_table, seq_lens,
                        query_start and every cached key and value older than
                        each sequence's newest max_query_len tokens are not
                        written by the kernel that precedes this call on the
                        stream (anything else that writes them completes
                        before the call is launched: earlier kernels, copies
                        the stream waits for).  The call then reads them,
                        and streams those pages into shared memory, while
                        that kernel finishes
                        (programmatic dependent launch); q, the newest keys
                        and values, and every write still wait for it to
                        complete.  This is the case of a decode step whose
                        previous kernel writes only the new tokens' keys and
                        values (paged_rope_cache_write) or is an attention
                        call of another layer.  A split call whose grid
                        fills more than ~58 % of the SMs is then launched
                        without the cooperative attribute (so that it starts
                        on the SMs the previous call frees); its mergers
                        still wait for every CTA of the call, which a kernel
                        on another stream holding SMs for longer than the
                        wait limit would turn into PD_DEV_WAIT_TIMEOUT.
                        0 = read nothing before the previous kernel has
                        completed.  Anything else: PD_EINVAL.                  */
  int mergers;       /* at most this many mergers K of the cooperative merge
                        (a power of two; 0 = auto: the largest power of two
                        <= min(D / 8, 64, segments, W), W the smallest power
                        of two >= 4 with W x 8192 >= segments x rows per CTA
                        x D, i.e. about 8192 partial elements per merger)     */
} pd_options;

/* paged_decode_attn with explicit knobs (opts may be NULL). */
PD_API int paged_decode_attn_opts(const pd_tensor *q, const pd_tensor *k_cache, const pd_tensor *v_cache,
                           const pd_tensor *block_table, const pd_tensor *seq_lens, pd_tensor *out,
                           int num_q_heads, int num_kv_heads, int head_size, int page_size,
                           int max_query_len, int window, float scale, int layout,
                           pd_scratch *scratch, void *stream, const pd_options *opts);

/* A decode batch whose requests have different query lengths (the
 * query_start_loc / q_to_klen maps of the vLLM ROCm Octave backend,
 * `_fill_query_maps`): request s owns the rows query_start[s] ..
 * query_start[s+1] - 1 of q and out, q_len_s = query_start[s+1] -
 * query_start[s] <= max_query_len <= 8, and its token i sees the keys
 * [lo, seq_lens[s] - q_len_s + i + 1) (lo as in paged_decode_attn).  Rows at
 * and past query_start[S] (padding of a captured batch) see no key and are
 * written as zeros.
 *   q, out       [T, Hq, D] for any T >= 0 (T = 0: nothing to do)
 *   query_start  [S + 1] int32 device array, non-decreasing, 0 <= entries <= T
 * The other arguments are those of paged_decode_attn_opts (opts may be
 * NULL; path 3 is not built for this call: PD_EINVAL).  Entries outside
 * [0, T], decreasing ones or a q_len above max_query_len are clamped on the
 * device and reported as PD_DEV_BAD_QSTART. */
PD_API int paged_decode_attn_varlen(const pd_tensor *q, const pd_tensor *k_cache,
                                    const pd_tensor *v_cache, const pd_tensor *block_table,
                                    const pd_tensor *seq_lens, const pd_tensor *query_start,
                                    pd_tensor *out, int num_q_heads, int num_kv_heads,
                                    int head_size, int page_size, int max_query_len, int window,
                                    float scale, int layout, pd_scratch *scratch, void *stream,
                                    const pd_options *opts);

/* The launch plan chosen for a call shape, computed on the host only (no
 * device access), for inspection and tests. */
typedef struct pd_plan {
  int path;          /* 1 = mma.sync, 3 = tcgen05 / tensor memory             */
  int merge;         /* 0 = none, 1 = last arriver, 2 = cooperative mergers    */
  int mergers;       /* K of the cooperative merge                             */
  int rows;          /* packed rows per kv head, G * M                         */
  int row_groups, rows_per_cta, n_tiles, key_groups, stages;
  int seg_blocks;    /* 16-key blocks per segment                              */
  int max_segments;  /* segments per (sequence, kv head, row group) in the grid */
  int cluster;
  int max_parts;     /* partial slots per group in the scratch                 */
  int grid_x;        /* CTAs per sequence: kv heads x row_groups x max_segments */
  int grid_y;        /* sequences (the launch grid is (max_segments,            */
                     /* kv heads x row_groups, sequences))                      */
  int block_threads;
  int smem_bytes;
  int64_t scratch_needed; /* bytes of scratch this call needs (0 = none)       */
} pd_plan;

PD_API int paged_decode_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
                      int page_size, int max_query_len, int window, int block_table_width,
                      int num_sms, const pd_scratch *scratch, const pd_options *opts,
                      pd_plan *plan);

/* Size of the scratch array compiled into the library for
 * paged_decode_attn_static, and the part of it kept for counters. */
#define PD_STATIC_SCRATCH_BYTES (16u << 20)
#define PD_STATIC_COUNTER_BYTES (512u << 10)

/* The decode call without caller scratch.  The paper has no counterpart to
 * it.  For callers that cannot allocate device memory (a host
 * framework that owns all device allocation, a runtime that forbids
 * allocation after start-up, an integration that only hands over inputs and
 * outputs), the split-KV scratch is a fixed array of
 * PD_STATIC_SCRATCH_BYTES inside the library, present on every GPU that
 * loads the library until the process exits.  Arguments, layouts and
 * results are those of paged_decode_attn; the split is fitted to the array,
 * so long or large calls may use fewer segments than with a larger caller
 * buffer.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - Each call clears its counters with cudaMemsetAsync on `stream` and
 *     allocates nothing (no cudaMalloc, no cudaFree, no allocating library).
 *   - Every call shares the one array: calls that overlap on the GPU (on two
 *     streams, or two host threads) race on it.  Serialise them.
 *   - A call whose sequences x kv heads need more than
 *     PD_STATIC_COUNTER_BYTES of counters (PD_COUNTERS_PER_PAIR int32 per
 *     pair, i.e. more than 8192 pairs) returns PD_ESCRATCH before it
 *     touches the device.
 *   - On a device that is not sm_103 it returns PD_ENODEV, as the other
 *     entry points do. */
PD_API int paged_decode_attn_static(const pd_tensor *q, const pd_tensor *k_cache,
                                    const pd_tensor *v_cache, const pd_tensor *block_table,
                                    const pd_tensor *seq_lens, pd_tensor *out, int num_q_heads,
                                    int num_kv_heads, int head_size, int page_size,
                                    int max_query_len, int window, float scale, int layout,
                                    void *stream);

/* The rotary position embedding of the new tokens' q and k and the store of
 * their k and v into the paged cache, in one kernel, ahead of the decode call
 * that reads the cache.  The pages only name this step (the fused RoPE /
 * KV-cache write that ROCm/vllm PR #1330, "Summary", moved to a stacked draft
 * PR); the slot convention is the cache store of the vLLM ROCm Octave
 * backend (`do_kv_cache_update(layer, key, value, kv_cache, slot_mapping)`)
 * and the rotary part of the head its `rope_dim`.  For token t, head h and
 * rotated pair i < rot_dim / 2 with (c, s) = cos_sin_cache[positions[t]]
 * [i], [rot_dim / 2 + i]:
 *     x1' = x1 c - x2 s,   x2' = x2 c + x1 s       (fp32, rounded once)
 * where (x1, x2) = dims (i, i + rot_dim/2) when is_neox, else (2i, 2i + 1);
 * dims at and past rot_dim pass through.  q' goes to q_out; k' and v go to
 * the cache slot slot_mapping[t] (page slot / page_size, token slot %
 * page_size) of every kv head; a slot of -1 (a padding token) writes
 * nothing.
 *   q, q_out      [T, Hq, D], fp16/bf16; q_out may be q itself (in place)
 *   k, v          [T, Hkv, D], the same dtype
 *   positions     [T] int32 device array, rows of the table
 *   slot_mapping  [T] int32 device array, distinct slots or -1
 *   cos_sin_cache [max_pos, >= rot_dim] fp32 (PD_F32), rows 16-byte aligned
 *   k_cache, v_cache  the decode call's pools (NHD or HND, packed allowed)
 *   rot_dim       rotated dims, <= D; a multiple of 16 (NeoX) or 8 (GPT-J)
 * Asynchronous on `stream`, allocates nothing.  A position outside the table
 * is clamped into it and a slot past the pool is skipped, both reported in
 * the device status word (PD_DEV_BAD_POSITION, PD_DEV_BAD_SLOT). */
PD_API int paged_rope_cache_write(const pd_tensor *q, const pd_tensor *k, const pd_tensor *v,
                                  const pd_tensor *positions, const pd_tensor *slot_mapping,
                                  const pd_tensor *cos_sin_cache, pd_tensor *q_out,
                                  pd_tensor *k_cache, pd_tensor *v_cache, int num_q_heads,
                                  int num_kv_heads, int head_size, int rot_dim, int page_size,
                                  int layout, int is_neox, void *stream);

/* ---- Paged prefill (plan_prefill, prefill_target_workgroups and
 * _BuiltinPrefill.prefill_attn on the vllm.v1.attention.ops.rocm_rdna_hip
 * page) ----
 *
 * The same attention as paged_decode_attn_varlen, for requests of any query
 * length: request s owns the rows query_start[s] .. query_start[s+1] - 1 of
 * q and out, and its token i sees the keys [lo, seq_lens[s] - q_len_s + i +
 * 1) (lo as in paged_decode_attn).  A launch runs a host-made work list: a
 * request's query tokens are packed token-major into rows (token i, q head
 * h*G + j -> row i*G + j), cut into tiles of PD_PREFILL_TILE_ROWS rows
 * (PD_PREFILL_TILE_ROWS_D128 at head size 128, whose tiles run on the
 * 5th-generation tensor cores as two halves of one row per tensor-memory
 * lane), and
 * a tile whose keys (from its window start rounded down to 16 keys, to the
 * last key its last token sees) exceed the mean load per resident CTA is cut
 * into segments, merged in the kernel by the last-arriving segment.  Items
 * are ordered heaviest first.  Each item runs once per kv head. */
#define PD_PREFILL_TILE_ROWS 64
#define PD_PREFILL_TILE_ROWS_D128 256
#define PD_PREFILL_MAX_SEGMENTS 32

/* One work item: a segment of the keys of one tile of one request. */
typedef struct pd_prefill_item {
  int32_t seq;      /* request of the batch                                   */
  int32_t tile;     /* tile of info.tile_rows packed rows of it               */
  int32_t seg;      /* segment of the tile's keys, 0 .. nseg - 1               */
  int32_t nseg;     /* segments of the tile (1: not split)                    */
  int32_t split;    /* index of the split tile, -1 when nseg == 1             */
  int32_t slot;     /* first partial slot of the split tile's segments, or -1 */
  int32_t blocks;   /* 16-key blocks of the tile's keys (its load)            */
  int32_t reserved; /* 0                                                      */
} pd_prefill_item;

typedef struct pd_prefill_plan_info {
  int64_t num_items;       /* work items (each runs once per kv head)         */
  int32_t num_split_tiles; /* tiles cut into segments                         */
  int32_t num_slots;       /* partial slots of their segments (per kv head)  */
  int32_t tile_rows;       /* packed rows per tile: PD_PREFILL_TILE_ROWS, or  *
                            * PD_PREFILL_TILE_ROWS_D128 at head size 128     */
  int32_t max_segments;    /* PD_PREFILL_MAX_SEGMENTS                         */
  int32_t target_ctas;     /* CTAs resident at once the split aims at         */
  int32_t reserved;
  int64_t total_blocks;    /* 16-key blocks over all tiles (one kv head)      */
  double load_blocks;      /* blocks per CTA a tile is split above            */
} pd_prefill_plan_info;

/* The work list of a prefill launch, computed on the host from host copies
 * of query_start [num_seqs + 1] and seq_lens [num_seqs] (each length, or an
 * upper bound).  head_size (64, 128, 256 or 512; else PD_EHEAD) sets the
 * tile rows.  num_sms: CTAs resident at once (0 = the current device's SM
 * count; this kernel runs one CTA per SM).  items NULL: fill `info` only (a
 * size query); else items[0 .. info->num_items) are written and `capacity`
 * must hold them.  Returns PD_EINVAL on a malformed query_start (negative
 * or decreasing). */
PD_API int paged_prefill_plan(const int32_t *query_start, const int32_t *seq_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_size, int window,
                              int num_sms, pd_prefill_item *items, int64_t capacity,
                              pd_prefill_plan_info *info);

/* Scratch bytes that serve every prefill plan made with this num_sms.
 * Prepare the buffer with paged_decode_scratch_init(scratch, data, bytes,
 * num_sms, 1, stream). */
PD_API size_t paged_prefill_scratch_bytes(int num_kv_heads, int head_size, int num_sms);

/* The prefill call.
 *   q, out       [T, Hq, D] fp16/bf16, T = query_start's last entry or more
 *                (rows past it are written as zeros)
 *   k_cache, v_cache, block_table, seq_lens: as paged_decode_attn
 *   query_start  [S + 1] int32 device array (the plan's, on the device)
 *   work         [num_items, 8] int32 device copy of the plan's items
 *   info         the plan's info (host), made for this head_size
 *   scratch      needed when info->num_split_tiles > 0 (else may be NULL)
 * Items that do not fit the launch (a request, tile, segment or slot out of
 * range) are skipped and reported as PD_DEV_BAD_WORK. */
PD_API int paged_prefill_attn(const pd_tensor *q, const pd_tensor *k_cache,
                              const pd_tensor *v_cache, const pd_tensor *block_table,
                              const pd_tensor *seq_lens, const pd_tensor *query_start,
                              const pd_tensor *work, const pd_prefill_plan_info *info,
                              pd_tensor *out, int num_q_heads, int num_kv_heads, int head_size,
                              int page_size, int window, float scale, int layout,
                              pd_scratch *scratch, void *stream);

/* Read the device status word (PD_DEV_* bits) of the current device after
 * synchronising `stream`; reset it to 0 when `reset` is non-zero. */
PD_API int paged_decode_device_status(unsigned int *status, int reset, void *stream);

/* A static description of a status code. */
PD_API const char *paged_decode_strerror(int code);

/* Library version, major * 10000 + minor * 100 + patch. */
PD_API int paged_decode_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_DECODE_H */
