// Paged split-KV decode attention on sm_103a.
//
// One CTA per (KV segment, kv head x row group, sequence) = blockIdx (x, y,
// z): the work unit of the gfx1151 decode kernel (ROCm/vllm PR #1330,
// "Kernel"), where all the query rows of a kv head share a CTA so that its K
// and V are read from memory once, and a batch puts one sequence on each
// grid slice.  A sequence's query rows are s * M .. s * M + M - 1, or, with
// variable query lengths, query_start[s] .. query_start[s+1] - 1 (the query
// maps of the vLLM ROCm Octave backend, _fill_query_maps); packed rows are
// token-major, so a shorter request only shortens the CTA's valid rows.
//
// Warp roles
//   * one producer warp: per 32 KiB ring stage, TMA-loads the K and V
//     16-key x 64-dim boxes of the stage's keys, one box per lane, straight
//     from the physical page the block table names (the page gather);
//   * NT * KG consumer warps: warp (t, g) owns the 8 packed query rows of
//     n-tile t and consumes the stages g, g + KG, g + 2 KG, ...
//
// Per stage, a consumer warp computes for each 16-key block
//   S^T[16 keys x 8 rows] = K[16 x D] . Q^T[D x 8]        (mma m16n8k16)
// so keys sit on the MMA's M side and the packed rows on its 8-wide N side:
// few rows (G * M = 4 .. 64) waste at most 7 rows of the tile.  The online
// softmax (running max m, sum l, in exp2 form, all fp32) needs no cross-warp
// exchange because every row lives in one warp.  P^T is cast to the input
// dtype and moved into the B-operand layout with movmatrix.trans, then
//   O^T[D x 8] += V^T[D x 16 keys] . P^T[16 x 8]           (mma m16n8k16)
// with V^T read by ldmatrix.trans from the same swizzled stage.
//
// A second consumer (TC = true) runs the products on the 5th-generation
// tensor cores instead: tcgen05 MMAs issued by one thread, accumulators in
// tensor memory, four softmax warps (see the TC branch below).  A third
// (TP = true) serves prefill tiles of 256 packed rows: two halves of 128
// rows share each K/V stage, one row per tensor-memory lane, with S, P and
// O in tensor memory (see the TP branch).
//
// Epilogue: the warp groups' (acc, m, l) are combined in shared memory into
// the CTA's partial.  A sequence cut into several segments publishes the
// partials to scratch and counts arrivals per (sequence, kv head, row group);
// in a grid that fits on the GPU at once the last K arrivals merge one slice
// of the head dim each (cooperative launch), otherwise the last arrival
// merges alone (or, with a thread-block cluster, after a combine through
// distributed shared memory).  The mergers reset the counters, so every
// launch starts them at zero (split-KV with an in-kernel merge, as in the
// vLLM RDNA backend's make_scratch).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pd_internal.h"
#include "pd_ptx.cuh"

namespace pd {

__device__ __forceinline__ uint32_t pack2(float lo, float hi, std::true_type /*bf16*/) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, std::false_type /*fp16*/) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// The largest element of 32 packed pairs, widened to fp32 (NaN skipped).
template <int N>
__device__ __forceinline__ float max2_of(const uint32_t (&w)[N], std::true_type /*bf16*/) {
  __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162 *>(&w[0]);
#pragma unroll
  for (int i = 1; i < N; ++i) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
  return fmaxf(__low2float(m), __high2float(m));
}
template <int N>
__device__ __forceinline__ float max2_of(const uint32_t (&w)[N], std::false_type /*fp16*/) {
  __half2 m = *reinterpret_cast<const __half2 *>(&w[0]);
#pragma unroll
  for (int i = 1; i < N; ++i) m = __hmax2(m, *reinterpret_cast<const __half2 *>(&w[i]));
  return fmaxf(__low2float(m), __high2float(m));
}

// acc + lo + hi of a packed pair, each half widened exactly to fp32 inside a
// mixed-precision add (one instruction per element)
__device__ __forceinline__ float add2_f32(float acc, uint32_t w, std::true_type /*bf16*/) {
  asm("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nadd.rn.f32.bf16 %0, lo, %0;\n"
      "add.rn.f32.bf16 %0, hi, %0;\n}\n"
      : "+f"(acc)
      : "r"(w));
  return acc;
}
__device__ __forceinline__ float add2_f32(float acc, uint32_t w, std::false_type /*fp16*/) {
  asm("{\n.reg .b16 lo, hi;\nmov.b32 {lo, hi}, %1;\nadd.rn.f32.f16 %0, lo, %0;\n"
      "add.rn.f32.f16 %0, hi, %0;\n}\n"
      : "+f"(acc)
      : "r"(w));
  return acc;
}

// Column swizzle of the fp32 partial tiles in shared memory: rows 2x and 2x+1
// of an n-tile are spread over four 8-word bank groups.
__device__ __forceinline__ int psw(int d, int r) { return d ^ (((r >> 1) & 3) << 3); }

template <bool BF16>
__device__ __forceinline__ void store8(void *dst, const float (&v)[8]) {
  using tag = std::integral_constant<bool, BF16>;
  uint4 w;
  w.x = pack2(v[0], v[1], tag{});
  w.y = pack2(v[2], v[3], tag{});
  w.z = pack2(v[4], v[5], tag{});
  w.w = pack2(v[6], v[7], tag{});
  *reinterpret_cast<uint4 *>(dst) = w;
}

template <bool BF16>
__device__ __forceinline__ void store4(void *dst, const float (&v)[4]) {
  using tag = std::integral_constant<bool, BF16>;
  uint2 w;
  w.x = pack2(v[0], v[1], tag{});
  w.y = pack2(v[2], v[3], tag{});
  *reinterpret_cast<uint2 *>(dst) = w;
}

// 2^x by the SFU (ex2.approx.ftz: relative error ~2^-22, -inf -> +0); the
// main-loop probabilities are rounded to 16 bits right after.
__device__ __forceinline__ float sfu_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1/x by the SFU (rcp.approx.ftz: ~1 ulp) for the output normalisation
__device__ __forceinline__ float sfu_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float exp2_or_zero(float x, float m) {
  // e^(x - m) in exp2 form; 0 for an empty row (x = -inf; m is always
  // finite here: 0 stands in for the max of an empty row)
  return sfu_exp2(x - m);
}

template <int D, bool BF16, bool TC, bool DOT, bool RM, bool TP>
__global__ void __launch_bounds__(TC ? kTcThreads : TP ? kTpThreads : kMaxThreads, 1)
    pd_decode_mma(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ Params p) {
  static_assert((int)TC + (int)DOT + (int)RM + (int)TP <= 1, "one consumer kind per instance");
  static_assert(!TP || D == 128, "the tensor-memory prefill consumer serves head size 128");
  static_assert(!RM || D <= 128, "the rows-on-M consumer keeps Q and O of 16 rows in registers");
  static_assert(!DOT || D <= 256, "the warp dot-product consumer serves head sizes up to 256");
  using tag = std::integral_constant<bool, BF16>;
  using T = std::conditional_t<BF16, __nv_bfloat16, __half>;
  constexpr int NBOX = D / 64;                  // 128-byte boxes across the head dim
  constexpr int BLOCK_BYTES = kBlockKeys * D * 2;
  constexpr int STAGE = kStageBytes;
  constexpr int TB = STAGE / 2 / BLOCK_BYTES;  // 16-key blocks per stage
  constexpr int KS = D / 16;                    // mma k-steps over d, and m-tiles of O^T
  constexpr bool Q_IN_REGS = D <= 256;

  extern __shared__ unsigned char smem_raw[];
  // aligned by pointer arithmetic on the shared array (not through an
  // integer), so every pointer derived from it stays in the shared space
  unsigned char *smem =
      smem_raw + ((kSmemAlign - (smem_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  // Tensor-memory path (TC): keys per stage, P tile bytes, TMEM columns.
  constexpr int SC = TB * kBlockKeys;
  constexpr int PTILE = tc_p_tile_bytes(D);
  constexpr int TMEM_COLS = TP ? tp_tmem_cols(D) : tc_tmem_cols(D);
  // (RM: one warp per 16 packed rows, the n-tiles taken in pairs)
  const int NS = p.NS, NT = p.NT, KG = p.KG,
            NC = TC ? kTcConsumerWarps : TP ? kTpConsumerWarps : RM ? (NT >> 1) * KG : NT * KG;
  const int NT8 = NT * 8;
  // 8-row groups of the Q tile in shared memory (TP: both tiles')
  const int NTQ = TC ? kTcRows / 8 : TP ? 2 * kTpRows / 8 : NT;
  // page ids of 16-key blocks staged in shared memory at a time
  constexpr int BIDS = TP ? kTpBlockIds : kBlockIds;
  unsigned char *ring = smem;
  unsigned char *qs = ring + NS * STAGE;
  unsigned char *pts = qs + NTQ * D * 16;  // TC: two P tiles
  uint64_t *full = reinterpret_cast<uint64_t *>(pts + (TC ? 2 * PTILE : 0));
  uint64_t *empty = full + NS;
  // TC barriers: [0,1] S full, [2,3] S read, [4,5] P written, [6,7] PV done,
  // [8] every MMA done
  uint64_t *tcb = empty + NS;
  uint64_t *fl64 = tcb + (TC ? kTcBarriers : TP ? kTpBarriers : 0);
  volatile int *flags = reinterpret_cast<volatile int *>(fl64);  // [0] abort, [1] last
  uint64_t *mbar_merge = fl64 + 1;                               // flags[2..3]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fl64) + 4 + BIDS;  // after the page ids
  uint32_t tmem_base = 0;
  // Warp dot-product path (DOT): Q rows in fp32 [8][D], then one P buffer
  // [stage keys][8] fp32 per warp group, 16-byte aligned after the page ids
  float *dot_q = reinterpret_cast<float *>(
      smem + ((reinterpret_cast<unsigned char *>(tmem_slot) - smem + 15) & ~15));
  float *dot_p = dot_q + 8 * D;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid (segment, kv head x row group, sequence); a prefill launch's grid
  // is (work item, kv head) and its item names the sequence, the tile of
  // packed rows (the row group) and the segment
  const bool prefill = p.work != nullptr;
  int seg = blockIdx.x, hg = blockIdx.y, s = blockIdx.z;
  int h = p.rg == 1 ? hg : hg / p.rg, grow = hg - h * p.rg;

  // ---- set-up that reads no global memory (it overlaps the previous grid's
  // tail): barriers, the tensor-map prefetch (the Q tile is loaded by the
  // consumers later) ----
  // (one barrier per lane of warp 0)
  if (warp == 0) {
    if (lane < NS) {
      mbar_init(smem_u32(full + lane), 1);
      // (TC: freed by the PV MMAs' commit; TP: by both tiles' PV commits;
      // RM: by its NT / 2 warps)
      mbar_init(smem_u32(empty + lane), TC ? 1 : TP ? 2 : RM ? NT >> 1 : NT);
    }
    if constexpr (TC) {
      if (lane < kTcBarriers) mbar_init(smem_u32(tcb + lane), (lane >= 2 && lane <= 5) ? 4 : 1);
    }
    if constexpr (TP) {
      // P written: a tile's four softmax warps; every MMA done: the S warp's
      // and both PV warps' last commits
      if (lane < kTpBarriers)
        mbar_init(smem_u32(tcb + lane), (lane >= 4 && lane <= 7) ? 4 : lane == 12 ? 3 : 1);
    }
    if (lane == 31) {
      mbar_init(smem_u32(mbar_merge), 1);
      flags[0] = 0;
      flags[1] = 0;
    }
    fence_mbar_init();
  }
  if (warp == NC && lane == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  __syncthreads();

  // ---- index arithmetic that reads no global memory, done before the wait
  // so that only loads and a few compares lie between the wait and the
  // first page copy ----
  int rr0 = grow * p.rows_cta;
  int rr1 = min(p.R, rr0 + p.rows_cta);
  const int lg_g = (p.G & (p.G - 1)) == 0 ? __ffs(p.G) - 1 : -1;  // G a power of two
  auto token_of = [&](int rr) { return lg_g >= 0 ? rr >> lg_g : rr / p.G; };  // packed row -> token
  int tok0 = token_of(rr0), tok1 = token_of(rr1 - 1);  // tokens of the first and last row
  const int lg_nt = (NT & (NT - 1)) == 0 ? __ffs(NT) - 1 : -1;
  // consumer n-tile and warp group (RM: warp w of a group takes rows 16w ..)
  const int t_n = RM ? warp % (NT >> 1) : lg_nt >= 0 ? warp & (NT - 1) : warp % NT;
  const int g_k = RM ? warp / (NT >> 1) : lg_nt >= 0 ? warp >> lg_nt : warp / NT;
  int cl_id = seg / p.CS;
  const int bpp = p.P / kBlockKeys;  // 16-key blocks per page
  const int lg_bpp = (bpp & (bpp - 1)) == 0 ? __ffs(bpp) - 1 : -1;
  const int seg_cover = p.max_seg * p.seg_blocks;  // blocks the plan's segments cover
  // Speculative page ids: without a window, segment `seg` starts at block
  // seg * seg_blocks whenever the sequence fits the plan; the producer reads
  // those block-table entries while seq_lens is still in flight.
  constexpr int kSpec = 256;
  int spec[kSpec / 32];  // block-table column of each block, then its page id
  const int spec_b0 = seg * p.seg_blocks;
  const int32_t *bt_row = p.block_table + (int64_t)s * p.bt_stride;
  const int bt_blocks = p.bt_width * bpp;
  const bool spec_on = warp == NC && p.window == 0 && !prefill;
  if (spec_on) {
#pragma unroll
    for (int k = 0; k < kSpec / 32; ++k) {
      const int i = lane + 32 * k, b = spec_b0 + i;
      spec[k] = (i < p.seg_blocks && b < bt_blocks) ? (lg_bpp >= 0 ? b >> lg_bpp : b / bpp) : -1;
    }
  }

  // Launched with programmatic stream serialisation: wait here until the
  // previous grid on the stream (which may have written q, the caches, the
  // block table or the scratch) has completed, before reading any of them.
  // With p.early the caller vouches for the block table, seq_lens,
  // query_start and the older keys: the producer streams those pages while
  // the previous grid finishes, and every other warp waits at the top of
  // its branch below.
  if (!p.early) grid_dependency_wait();

  // prefill: the work item (sequence, tile, segment, segments, split tile,
  // first partial slot), checked against the launch before anything is
  // addressed with it
  int pf_nseg = 1, pf_split = 0, pf_slot = 0;
  if (prefill) {
    const int4 w0 = __ldg(reinterpret_cast<const int4 *>(p.work) + 2 * (int64_t)blockIdx.x);
    const int4 w1 = __ldg(reinterpret_cast<const int4 *>(p.work) + 2 * (int64_t)blockIdx.x + 1);
    s = w0.x;
    grow = w0.y;
    seg = w0.z;
    pf_nseg = w0.w;
    pf_split = w1.x;
    pf_slot = w1.y;
    h = hg = blockIdx.y;
    const bool ok = s >= 0 && s < p.num_seqs && grow >= 0 && grow <= (INT32_MAX - 64) / p.rows_cta &&
                    pf_nseg >= 1 && pf_nseg <= p.max_parts && seg >= 0 && seg < pf_nseg &&
                    (pf_nseg == 1 || (pf_split >= 0 && pf_split < p.pf_groups && pf_slot >= 0 &&
                                      pf_slot <= p.pf_slots - pf_nseg));
    if (!ok) {
      if (tid == 0) atomicOr(p.status, 0x80u);
      return;
    }
    rr0 = grow * p.rows_cta;
    rr1 = rr0 + p.rows_cta;
    tok0 = token_of(rr0);
    tok1 = token_of(rr1 - 1);
    cl_id = seg;
    bt_row = p.block_table + (int64_t)s * p.bt_stride;
  }

  // (the block-table entries of the segment's first blocks are loaded in
  // the same round trip as seq_lens)
  if (spec_on) {
#pragma unroll
    for (int k = 0; k < kSpec / 32; ++k) spec[k] = spec[k] >= 0 ? ld_nc_now(bt_row + spec[k]) : 0;
  }
  int L = __ldg(p.seq_lens + s);
  // q / out rows of the sequence: [s * M, s * M + M), or from query_start
  int qa, qb;
  if (p.query_start) {
    qa = __ldg(p.query_start + s);
    qb = __ldg(p.query_start + s + 1);
  } else {
    qa = s * p.M;
    qb = qa + p.M;
  }

  // ---- key ranges --------------------------------------------------------
  if (L < 0) L = 0;
  if (L > p.bt_width * p.P) {
    if (tid == 0 && seg == 0) atomicOr(p.status, 0x4u);
    L = p.bt_width * p.P;
  }
  // first row and query tokens of the sequence (clamped into [0, num_tokens]
  // and to M, and reported, when query_start is out of order or range)
  int q0 = qa, ml = p.M;
  if (p.query_start) {
    const int a = min(max(qa, 0), p.num_tokens), b = min(max(qb, a), p.num_tokens);
    if ((a != qa || b != qb || b - a > p.M) && tid == 0 && seg == 0 && hg == 0)
      atomicOr(p.status, 0x8u);
    q0 = a;
    ml = min(b - a, p.M);
  }
  // rows of real query tokens: a prefix of the CTA's rows (token-major packing)
  const int rr1v = min(rr1, ml * p.G);
  const int tok1v = rr1v < rr1 ? ml - 1 : tok1;
  int u_lo = 0, u_hi = 0, v_lo = 0, v_hi = 0;  // union / intersection of the rows' key ranges
  if (rr1v > rr0) {
    const int n0 = max(L - ml + tok0 + 1, 0);
    const int n1 = max(L - ml + tok1v + 1, 0);
    u_hi = n1;
    v_hi = n0;
    u_lo = p.window ? max(0, n0 - p.window) : 0;
    v_lo = p.window ? max(0, n1 - p.window) : 0;
  }
  const int b_first = u_lo / kBlockKeys;
  const int nb = u_hi > u_lo ? (u_hi + kBlockKeys - 1) / kBlockKeys - b_first : 0;
  // blocks per segment: the plan's, unless the sequence is longer than
  // planned; a prefill tile's segments are its work items' (every one of
  // them arrives at the merge, an empty one with an empty partial)
  const int sb = prefill ? max(1, (nb + pf_nseg - 1) / pf_nseg)
                         : (nb <= seg_cover ? p.seg_blocks : (nb + p.max_seg - 1) / p.max_seg);
  // Segment x works iff x == 0 or x * sb < nb.
  if (!prefill) {
    if (cl_id > 0 && cl_id * p.CS * sb >= nb) return;  // uniform over the cluster
    if (seg > 0 && nb <= sb) return;                     // no merge: only segment 0 works
  }
  const int my_b0 = b_first + seg * sb;
  const int my_nb = max(0, min(b_first + nb, my_b0 + sb) - my_b0);
  const int ntile = (my_nb + TB - 1) / TB;
  // segments of this (sequence, head, row group) and merge clusters
  const int nseg = prefill ? pf_nseg : max(1, (nb + sb - 1) / sb);
  const int ncl = (nseg + p.CS - 1) / p.CS;
  if constexpr (TC || TP) {
    // tensor memory for the two S buffers and O (TP: and Q and two P
    // buffers); freed once the epilogue has read O (every path of the CTA
    // reaches that point)
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // (broadcast from lane 0 so the compiler knows it is warp-uniform: the
    // tensor-memory operands then stay in uniform registers)
    tmem_base = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile uint32_t *>(tmem_slot), 0);
  }


  // Consumer state (kept in registers across the main loop).
  // (DOT: lane i holds dims [i * DPL, (i + 1) * DPL) of all 8 rows)
  constexpr int DPL = DOT ? D / 32 : 1;
  float dacc[DOT ? 8 : 1][DPL], dm[DOT ? 8 : 1], dl[DOT ? 8 : 1];
#pragma unroll
  for (int r = 0; r < (DOT ? 8 : 1); ++r) {
    dm[r] = -INFINITY;
    dl[r] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) dacc[r][j] = 0.f;
  }
  // (RM: O of this warp's 16 rows, D/8 n-tiles of 8 dims)
  float racc[RM ? D / 8 : 1][4];
#pragma unroll
  for (int i = 0; i < (RM ? D / 8 : 1); ++i) racc[i][0] = racc[i][1] = racc[i][2] = racc[i][3] = 0.f;
  float acc[KS][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int i = 0; i < KS; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int r0 = t_n * 8 + 2 * (lane & 3), r1 = r0 + 1;

  if (warp == NC) {
    // ================= producer: the page gather ===========================
    const uint64_t pol = policy_evict_first();
    // Physical page of every 16-key block of the segment, read from the
    // block table kBlockIds at a time ahead of the copies that need them, so
    // no TMA issue waits on a dependent global load.
    int *pids = const_cast<int *>(flags + 4);
    int pid_base = 0;
    const bool spec_ok = spec_on && my_b0 == spec_b0;
    auto load_pids = [&](int base) {
      __syncwarp();
      const int n = min(BIDS, my_nb - base);
      int i0 = 0;
      if (base == 0 && spec_ok) {
#pragma unroll
        for (int k = 0; k < kSpec / 32; ++k)
          if (lane + 32 * k < n) pids[lane + 32 * k] = spec[k];
        i0 = kSpec;
      }
      for (int i = i0 + lane; i < n; i += 32)
        pids[i] = __ldg(bt_row + (lg_bpp >= 0 ? (my_b0 + base + i) >> lg_bpp : (my_b0 + base + i) / bpp));
      __syncwarp();
    };
    if (my_nb > 0) load_pids(0);
    int issued = 0;
    int slot = 0, phase = 0;  // ring slot of stage j and the parity of its round
    // (p.early: keys at and past `fresh` may come from the previous grid)
    bool waited = !p.early;
    const int fresh = max(L - p.M, 0);
    for (int j = 0; j < ntile; ++j) {
      if (j * TB >= pid_base + BIDS) {
        pid_base = j * TB;
        load_pids(pid_base);
      }
      if (!waited && (my_b0 + j * TB + min(TB, my_nb - j * TB)) * kBlockKeys > fresh) {
        grid_dependency_wait();
        waited = true;
      }
      if (j >= NS) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait_bounded(smem_u32(empty + slot), phase ^ 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.status, 0x1u);
          }
          break;
        }
      }
      if (flags[0]) break;
      const int nbt = min(TB, my_nb - j * TB);
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(full + slot), nbt * 2 * BLOCK_BYTES);
      __syncwarp();
      if ((TP || TC) && lane < nbt * NBOX) {
        // K of the tensor-memory consumers: one copy per (16-key block,
        // 64-dim box), box-major in the stage ([box][block][16 keys][128 B])
        // so that one box's keys are consecutive 128-byte rows (one MMA
        // descriptor spans the stage)
        const int b = lane / NBOX, x = lane - b * NBOX;
        const int blk = my_b0 + j * TB + b;
        const int key_in_page = (lg_bpp >= 0 ? blk & (bpp - 1) : blk % bpp) * kBlockKeys;
        int phys = pids[j * TB + b - pid_base];
        if ((unsigned)phys >= (unsigned)p.num_pool_blocks) {
          atomicOr(p.status, 0x2u);  // a page id outside the pool: report, read page 0
          phys = 0;
        }
        const uint32_t dst = smem_u32(ring + slot * STAGE + x * (TB * BLOCK_BYTES / NBOX) +
                                      b * (BLOCK_BYTES / NBOX));
        tma_load_5d(dst, &tmK, smem_u32(full + slot), 0, key_in_page, x, h, phys, pol);
      } else if ((TP || TC) ? lane >= nbt * NBOX && lane < nbt * (NBOX + 1) : lane < 2 * nbt) {
        // one copy per 16-key block of K or V (all D/64 swizzle rows at once;
        // the tensor-memory consumers: V only)
        const int kv = (TP || TC) ? 1 : lane >= nbt, b = (TP || TC) ? lane - nbt * NBOX : lane - kv * nbt;
        const int blk = my_b0 + j * TB + b;
        const int key_in_page = (lg_bpp >= 0 ? blk & (bpp - 1) : blk % bpp) * kBlockKeys;
        int phys = pids[j * TB + b - pid_base];
        if ((unsigned)phys >= (unsigned)p.num_pool_blocks) {
          atomicOr(p.status, 0x2u);  // a page id outside the pool: report, read page 0
          phys = 0;
        }
        const uint32_t dst =
            smem_u32(ring + slot * STAGE + kv * (TB * BLOCK_BYTES) + b * BLOCK_BYTES);
        tma_load_5d(dst, kv ? &tmV : &tmK, smem_u32(full + slot), 0, key_in_page, 0, h, phys, pol);
      }
      issued = j + 1;
      if (++slot == NS) {
        slot = 0;
        phase ^= 1;
      }
    }
    // Leave no copy in flight: wait (bounded) for the last stages issued.
    if (lane == 0) {
      for (int j = max(0, issued - NS); j < issued; ++j)
        if (!mbar_wait_bounded(smem_u32(full + j % NS), (j / NS) & 1)) atomicOr(p.status, 0x1u);
    }
    if (!waited) grid_dependency_wait();  // before the epilogue's writes
  } else {
    if (p.early) grid_dependency_wait();  // before q and any write
    if constexpr (TP) {
    // ================= tensor-memory prefill consumers ====================
    // Two tiles of 128 packed rows share every K/V stage: tile X (X = 0, 1)
    // is rows 128 X .. 128 X + 127, one row per tensor-memory lane, and its
    // own four softmax warps 4 X .. 4 X + 3 (warp w owns lanes 32 (w % 4) ..
    // 32 (w % 4) + 31, one row per thread).  Warp 8 issues the S MMAs, warp
    // 10 + X the PV MMAs of tile X, each as soon as its inputs are ready:
    //   S_X[128 x stage keys] = Q_X . K^T  (A = Q_X from shared memory; B =
    //                                     the stage's K, landed box-major,
    //                                     K-major; N = 64, one MMA per 16 dims)
    //   O_X[128 x D]         += P_X . V    (A = P_X from tensor memory; B = one
    //                                     V block, MN-major as the copies land)
    // S of stage j goes to buffer j & 1 of its tile and P of stage j over it,
    // so S of stage j + 1 is computed while the softmax of stage j runs, and
    // buffer j & 1 takes S of stage j + 2 once the PV MMAs of stage j have
    // read its P; only a rescale of O waits for a PV MMA.  O_X is rescaled in
    // tensor memory only when a row's max grows more than 8 past the
    // reference its P values use (so P <= 2^8), the online-softmax update in
    // exp2 form.  Two tiles per stage halve the K/V copies per row: the
    // per-SM copy rate bounds a 128-row tile.
    static_assert(!TP || SC == 64, "a stage holds 64 keys at head size 128");
    const int X = (warp >> 2) & 1;             // this softmax warp's tile
    const int r_tp = 32 * (warp & 3) + lane;   // its row in the tile
    const int rr_tp = rr0 + kTpRows * X + r_tp;
    const bool live = warp < kTpSoftmaxWarps && rr_tp < rr1v;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // S of tile x, stage j in buffer tS + (2 x + (j & 1)) * SC; P of that
    // stage overwrites the buffer's first SC / 2 columns once the softmax has
    // read S (so S of stage j + 1 is computed while the softmax of stage j
    // runs, and S of stage j + 2 once the PV MMAs of stage j have read P)
    const uint32_t tS = tmem_base + tp_s_col(D), tO = tmem_base + tp_o_col(D);
    if (warp < kTpSoftmaxWarps) {
      // Q rows of tile X into its 128-byte-swizzled K-major tile in shared
      // memory ([tile][64-dim box][128 rows][128 B]); zeros for rows past
      // the requests
      const uint4 *src = nullptr;
      if (live) {
        const int i = token_of(rr_tp), jq = rr_tp - i * p.G;
        src = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.q) +
                                              (int64_t)(q0 + i) * p.q_s0 +
                                              (int64_t)(h * p.G + jq) * p.q_s1);
      }
      unsigned char *qx = qs + X * (kTpRows * D * 2);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(qx + (c >> 3) * (kTpRows * 128) + r_tp * 128 +
                                   (((c & 7) ^ (r_tp & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();  // the tensor core reads the tiles
    }
    // both Q tiles are in place (softmax warps and the S warp)
    if (warp < kTpConsumerWarps) asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
    if (warp == kTpConsumerWarps - 1) {
      // ---- S issue: the whole warp runs the loop (every operand is
      // warp-uniform), one elected lane issues each MMA and commit ----
      tc_fence_after();
      const uint32_t idS = umma_idesc_f16(kTpRows, SC, BF16, 0, 0);
      const uint32_t ring_u = smem_u32(ring), qb_u = smem_u32(qs);
      // S of both tiles for stage j, once its stage has landed and (j >= 2)
      // the PV MMAs of stage j - 2 have read the P in its buffer
      auto issue_s = [&](int j) -> bool {
        const int slot = j % NS, sb = j & 1;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(full + slot), (j / NS) & 1)))
          return false;
        const uint32_t kst = ring_u + slot * STAGE;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 8 + 2 * x + sb),
                                                                  ((j - 2) >> 1) & 1)))
            return false;
          tc_fence_after();
          // all SC keys of the stage at once (keys of blocks a short stage
          // did not load give scores the softmax masks)
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const uint64_t bk =
                umma_desc_sw128(kst + (ks >> 2) * (TB * BLOCK_BYTES / NBOX) + (ks & 3) * 32, 16, 1024);
            umma_f16_warp(tS + (2 * x + sb) * SC,
                          umma_desc_sw128(qb_u + x * (kTpRows * D * 2) + (ks >> 2) * (kTpRows * 128) +
                                              (ks & 3) * 32,
                                          16, 1024),
                          bk, idS, ks > 0 ? 1u : 0u);
          }
          umma_commit_warp(smem_u32(tcb + 2 * x + sb));  // S_x of stage j is ready
        }
        return true;
      };
      // S of stage 0, then of each next stage as soon as its buffer is free
      // (the PV MMAs are the PV warps')
      bool ok = ntile == 0 || issue_s(0);
      for (int k = 1; k < ntile && ok; ++k) ok = issue_s(k);
      if (!ok && lane == 0) {
        flags[0] = 1;
        atomicOr(p.status, 0x1u);
      }
      umma_commit_warp(smem_u32(tcb + 12));  // this warp's MMAs have completed
    } else if (warp >= kTpConsumerWarps + 1) {
      // ---- PV issue of tile x = warp - 10: the whole warp runs the loop,
      // one elected lane issues ----
      const int x = warp - (kTpConsumerWarps + 1);
      tc_fence_after();
      const uint32_t idO = umma_idesc_f16(kTpRows, D, BF16, 0, 1);
      const uint32_t ring_u = smem_u32(ring);
      bool ok = true;
      for (int k = 0; k < ntile; ++k) {
        // P of stage k is in buffer k & 1 (its barriers complete once per
        // two stages, so a parity never stands for two phases)
        const int pb = k & 1;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 4 + 2 * x + pb), (k >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const int slot = k % NS;
        const int nbt = min(TB, my_nb - k * TB);
        const uint64_t dv = umma_desc_sw128(ring_u + slot * STAGE + TB * BLOCK_BYTES, 2048, 1024);
#pragma unroll
        for (int b = 0; b < TB; ++b)
          if (b < nbt)
            umma_f16_ts_warp(tO + x * D, tS + (2 * x + pb) * SC + 8 * b,
                             dv + (uint64_t)(b * BLOCK_BYTES / 16), idO, (k > 0 || b > 0) ? 1u : 0u);
        umma_commit_warp(smem_u32(tcb + 8 + 2 * x + pb));  // P buffer pb free, O_x current
        umma_commit_warp(smem_u32(empty + slot));  // (with the other tile's) the stage is free
      }
      if (!ok && lane == 0) {
        flags[0] = 1;
        atomicOr(p.status, 0x1u);
      }
      umma_commit_warp(smem_u32(tcb + 12));  // this warp's MMAs have completed
    } else {
      // ---- softmax: one row per thread, every stage, this tile ----
      int lo = 0, hi = 0;
      if (live) {
        hi = max(L - ml + token_of(rr_tp) + 1, 0);
        lo = p.window ? max(0, hi - p.window) : 0;
      }
      const uint32_t tOx = tO + X * D;
      float m_used = -INFINITY, lsum = 0.f;
      for (int j = 0; j < ntile; ++j) {
        const uint32_t tSx = tS + (2 * X + (j & 1)) * SC;  // S, then P, of stage j
        if (!__all_sync(0xffffffffu,
                        mbar_wait_bounded(smem_u32(tcb + 2 * X + (j & 1)), (j >> 1) & 1))) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.status, 0x1u);
          }
          break;
        }
        tc_fence_after();
        uint32_t sr[SC];  // the row's scores of the stage (fp32 bits)
        {
          uint32_t x0[32], x1[32];
          tmem_ld32(tSx + lane_base, x0);
          tmem_ld32(tSx + lane_base + 32, x1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            sr[i] = x0[i];
            sr[32 + i] = x1[i];
          }
        }
        const int nbt = min(TB, my_nb - j * TB);
        const int key_t0 = (my_b0 + j * TB) * kBlockKeys;
        const int slot = j % NS;
        // every row of the CTA sees every key of the stage: no mask, and the
        // scale is applied inside the exponent (rows past the requests'
        // tokens have Q = 0, finite scores, and are never stored)
        const bool fast = nbt == TB && key_t0 >= v_lo && key_t0 + SC <= v_hi;
        const float sl2 = p.scale_log2;
        // the largest scaled score of an unmasked stage: the largest (scale
        // >= 0) or smallest raw score, eight independent chains
        auto fast_max = [&]() -> float {
          float a[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) a[u] = __uint_as_float(sr[u]);
          if (sl2 >= 0.f) {
#pragma unroll
            for (int c = 8; c < SC; ++c) a[c & 7] = fmaxf(a[c & 7], __uint_as_float(sr[c]));
#pragma unroll
            for (int u = 4; u >= 1; u >>= 1)
#pragma unroll
              for (int v = 0; v < u; ++v) a[v] = fmaxf(a[v], a[v + u]);
          } else {
#pragma unroll
            for (int c = 8; c < SC; ++c) a[c & 7] = fminf(a[c & 7], __uint_as_float(sr[c]));
#pragma unroll
            for (int u = 4; u >= 1; u >>= 1)
#pragma unroll
              for (int v = 0; v < u; ++v) a[v] = fminf(a[v], a[v + u]);
          }
          return a[0] * sl2;
        };
        // O_X *= alpha row by row in tensor memory (the whole warp), once the
        // PV MMAs of stage j - 1 have completed
        auto rescale_o = [&](float alpha) -> bool {
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 8 + 2 * X + ((j - 1) & 1)),
                                                         ((j - 1) >> 1) & 1)))
            return false;
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tOx + lane_base + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tOx + lane_base + c0, o);
          }
          tmem_wait_st();
          tc_fence_before();
          return true;
        };
        // An unmasked stage with a reference on every row takes its
        // exponentials straight against that reference, tracking the largest
        // P; only a row whose P exceeds 2^8 (its max grew more than 8 past
        // the reference) needs the max, a rescale and the stage again.
        const bool direct = fast && __all_sync(0xffffffffu, m_used != -INFINITY);
        bool ok = true;
        if (!direct) {
          float mx;
          if (fast) {
            mx = fast_max();
          } else {
            // scaled scores with the mask applied (-inf), kept as fp32 bits
            float a[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) a[u] = -INFINITY;
#pragma unroll
            for (int c = 0; c < SC; ++c) {
              const int k = key_t0 + c;
              float x = __uint_as_float(sr[c]) * sl2;
              if (!live || !(c < nbt * kBlockKeys && k >= lo && k < hi)) x = -INFINITY;
              sr[c] = __float_as_uint(x);
              a[c & 7] = fmaxf(a[c & 7], x);
            }
#pragma unroll
            for (int u = 4; u >= 1; u >>= 1)
#pragma unroll
              for (int v = 0; v < u; ++v) a[v] = fmaxf(a[v], a[v + u]);
            mx = a[0];
          }
          const float m_new = fmaxf(m_used, mx);
          const bool need = m_used != -INFINITY && m_new > m_used + 8.f;
          // (need implies j >= 1)
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? sfu_exp2(m_used - m_new) : 1.f;
            ok = rescale_o(alpha);
            if (need) {
              lsum *= alpha;
              m_used = m_new;
            }
          }
          if (m_used == -INFINITY) m_used = m_new;
        }
        // (P goes over S in the buffer this warp has just read: its other
        // readers, the PV MMAs of stage j - 2, completed before S of stage j
        // was written there)
        if (!ok) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.status, 0x1u);
          }
          break;
        }
        {
          // P = 2^(x - m) rounded to the input type; the row sum takes P as
          // rounded for the MMA (four chains), so O is normalised by the
          // weights it was formed with
          uint32_t w[SC / 2];
          auto exps = [&](float mu) -> float {  // returns the largest P (direct stages)
            float pmax = 0.f;
            if (fast) {
#pragma unroll
              for (int c = 0; c < SC; c += 2)
                w[c >> 1] = pack2(sfu_exp2(fmaf(__uint_as_float(sr[c]), sl2, -mu)),
                                  sfu_exp2(fmaf(__uint_as_float(sr[c + 1]), sl2, -mu)), tag{});
              // the largest P as rounded: packed maxima, two per instruction
              pmax = max2_of(w, tag{});
            } else {
#pragma unroll
              for (int c = 0; c < SC; c += 2)
                w[c >> 1] = pack2(sfu_exp2(__uint_as_float(sr[c]) - mu),
                                  sfu_exp2(__uint_as_float(sr[c + 1]) - mu), tag{});
            }
            return pmax;
          };
          const float pmax = exps(m_used == -INFINITY ? 0.f : m_used);
          // (fmaxf skips a NaN P, as the max skipped a NaN score)
          if (direct && __any_sync(0xffffffffu, pmax > 256.f)) {
            const float m_new = fmaxf(m_used, fast_max());
            const bool need = m_new > m_used + 8.f;
            const float alpha = need ? sfu_exp2(m_used - m_new) : 1.f;
            if (!rescale_o(alpha)) {
              if (lane == 0) {
                flags[0] = 1;
                atomicOr(p.status, 0x1u);
              }
              break;
            }
            if (need) {
              lsum *= alpha;
              m_used = m_new;
            }
            exps(m_used);
          }
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < SC / 2; ++c) ls[c & 3] = add2_f32(ls[c & 3], w[c], tag{});
          lsum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          tmem_st32(tSx + lane_base, w);
        }
        // zero V of keys no row sees (outside the union, stale or NaN slots);
        // each tile does it before its own PV MMAs (the other tile's writes
        // are the same zeros)
        if (!(nbt == TB && key_t0 >= u_lo && key_t0 + SC <= u_hi)) {
          unsigned char *vb = ring + slot * STAGE + TB * BLOCK_BYTES;
          for (int c = 32 * (warp & 3) + lane; c < nbt * kBlockKeys; c += 128) {
            const int k = key_t0 + c;
            if (k < u_lo || k >= u_hi) {
#pragma unroll 1
              for (int x = 0; x < NBOX * 8; ++x)
                *reinterpret_cast<uint4 *>(vb + (c >> 4) * BLOCK_BYTES + (x >> 3) * 2048 +
                                           (c & 15) * 128 + (x & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();  // the zeroed V reaches the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tcb + 4 + 2 * X + (j & 1)));  // P of stage j written
      }
      m0 = m_used;
      l0 = lsum;
    }
    } else if constexpr (TC) {
    // ================= tensor-memory consumers ============================
    // The CTA's packed rows (<= 16) are copied four times into the 64 rows
    // of the Q tile (row 16 q + r = packed row r), so the M = 64 MMAs give
    // four copies of every score row, one per tensor-memory sub-partition
    // (lanes 0-15).  Softmax warp q takes its copy and a quarter of every
    // stage's keys, one row per thread (lanes < 16), and keeps its own
    // running (m, l) and O rows: four independent online softmaxes over
    // disjoint keys, merged in the epilogue like warp groups.  Warp 4
    // issues the MMAs (one elected lane of the whole warp):
    //   S[64 x stage keys] = Q[64 x D] . K^T   (one MMA per 16-key block and
    //                                          16-dim step, K-major operands)
    //   O[64 x D]         += P[64 x keys] . V  (one MMA per 16-key block, V
    //                                          MN-major as the copies land)
    // S has two tensor-memory buffers so the MMAs of stage j + 1 overlap
    // the softmax of stage j; P has two shared-memory tiles (row 16 q + r
    // holds copy q's keys only, the rest stays zero).  O is rescaled in
    // tensor memory only when a stage's max exceeds a row's reference max by
    // more than 8 (so P <= 2^8).
    constexpr int KPC = SC / 4;  // keys of a stage per copy
    {
      // the Q tile: 64 rows = 4 copies of the 16 packed rows (others zero);
      // both P tiles zeroed (each thread later writes its own keys only)
      const T *qbase = static_cast<const T *>(p.q);
      for (int idx = tid; idx < kTcRows * (D / 8); idx += NC * 32) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const int rp = r & 15, rr = rr0 + rp;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rp < p.rows_cta && rr < rr1v) {
          const int i = rr / p.G, jq = rr % p.G;
          v = __ldg(reinterpret_cast<const uint4 *>(qbase + (int64_t)(q0 + i) * p.q_s0 +
                                                    (int64_t)(h * p.G + jq) * p.q_s1 + c * 8));
        }
        const int tn = r >> 3, rw = r & 7, box = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(qs + (tn * NBOX + box) * 1024 + rw * 128 + ((cc ^ rw) << 4)) = v;
      }
      for (int idx = tid; idx < 2 * PTILE / 16; idx += NC * 32)
        reinterpret_cast<uint4 *>(pts)[idx] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();  // the tensor core reads both tiles
      asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
    }
    const uint32_t tS = tmem_base, tO = tmem_base + 2 * SC;
    if (warp == kTcConsumerWarps - 1) {
      // ---- MMA issue: the whole warp runs the loop (every operand is
      // warp-uniform), one elected lane issues each MMA and commit ----
      const uint32_t idS = umma_idesc_f16(kTcRows, SC, BF16, 0, 0);
      const uint32_t idO = umma_idesc_f16(kTcRows, D, BF16, 0, 1);
      const uint32_t q_u = smem_u32(qs), p_u = smem_u32(pts), ring_u = smem_u32(ring);
      const uint64_t dq = umma_desc_sw128(q_u, 16, NBOX * 1024);
      bool ok = true;
      for (int j = 0; j <= ntile; ++j) {
        if (j < ntile) {
          const int slot = j % NS;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(full + slot), (j / NS) & 1));
          if (ok && j >= 2)
            ok = __all_sync(0xffffffffu,
                            mbar_wait_bounded(smem_u32(tcb + 2 + (j & 1)), ((j - 2) >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          // K landed box-major ([64-dim box][block][16 keys][128 B]), so one
          // 128-byte-swizzled K-major descriptor spans the stage's keys: one
          // MMA per 16-dim step with N = every key of the stage (keys of
          // blocks a short stage did not load give scores the softmax masks)
          const uint32_t kst = ring_u + slot * STAGE;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
            umma_f16_warp(tS + (j & 1) * SC,
                          dq + (uint64_t)(((ks >> 2) * 1024 + (ks & 3) * 32) / 16),
                          umma_desc_sw128(kst + (ks >> 2) * (TB * BLOCK_BYTES / NBOX) + (ks & 3) * 32,
                                          16, 1024),
                          idS, ks > 0 ? 1u : 0u);
          umma_commit_warp(smem_u32(tcb + (j & 1)));  // S of stage j is ready
        }
        if (j >= 1) {
          const int jj = j - 1, slot = jj % NS;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 4 + (jj & 1)), (jj >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const int nbt = min(TB, my_nb - jj * TB);
          const uint64_t dv = umma_desc_sw128(ring_u + slot * STAGE + TB * BLOCK_BYTES, 2048, 1024);
          const uint64_t dp = umma_desc_sw128(p_u + (jj & 1) * PTILE, 16, 1024);
#pragma unroll
          for (int b = 0; b < TB; ++b)
            if (b < nbt)
              umma_f16_warp(tO, dp + (uint64_t)(((b >> 2) * 8192 + (b & 3) * 32) / 16),
                            dv + (uint64_t)(b * BLOCK_BYTES / 16), idO, (jj > 0 || b > 0) ? 1u : 0u);
          umma_commit_warp(smem_u32(empty + slot));       // the stage may be refilled
          umma_commit_warp(smem_u32(tcb + 6 + (jj & 1)));  // P tile jj & 1 is free, O is current
        }
      }
      if (!ok && lane == 0) {
        flags[0] = 1;
        atomicOr(p.status, 0x1u);
      }
      umma_commit_warp(smem_u32(tcb + 8));  // every MMA issued above has completed
    } else {
      // ---- softmax (warp q = copy q, keys [q KPC, (q + 1) KPC) of a stage) ----
      const int r = lane & 15, prow = 16 * warp + r;  // packed row, P / MMA row
      const bool live = lane < 16 && r < p.rows_cta && rr0 + r < rr1v;
      int lo = 0, hi = 0;
      if (live) {
        hi = max(L - ml + (rr0 + r) / p.G + 1, 0);
        lo = p.window ? max(0, hi - p.window) : 0;
      }
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      const int c_first = KPC * warp;  // this copy's first key of a stage
      float m_used = -INFINITY, lsum_all = 0.f;
      for (int j = 0; j < ntile; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + (j & 1)), (j >> 1) & 1))) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.status, 0x1u);
          }
          break;
        }
        tc_fence_after();
        float sv[KPC];
#pragma unroll
        for (int c0 = 0; c0 < KPC; c0 += 8) {
          uint32_t rr[8];
          tmem_ld8(tS + lane_base + (j & 1) * SC + c_first + c0, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) sv[c0 + i] = __uint_as_float(rr[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tcb + 2 + (j & 1)));  // S buffer read
        const int nbt = min(TB, my_nb - j * TB);
        const int key_t0 = (my_b0 + j * TB) * kBlockKeys;
        const int slot = j % NS;
        const bool fast = nbt == TB && key_t0 >= v_lo && key_t0 + SC <= v_hi;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < KPC; ++c) {
          float x = sv[c] * p.scale_log2;
          const int cs = c_first + c, k = key_t0 + cs;
          if (!live || (!fast && !(cs < nbt * kBlockKeys && k >= lo && k < hi))) x = -INFINITY;
          sv[c] = x;
          mx = fmaxf(mx, x);
        }
        const float m_new = fmaxf(m_used, mx);
        const bool need = m_used != -INFINITY && m_new > m_used + 8.f;
        bool ok = true;
        if (__any_sync(0xffffffffu, need)) {
          // O must be current: the PV MMAs of stage j - 1 have completed
          ok = __all_sync(0xffffffffu,
                          mbar_wait_bounded(smem_u32(tcb + 6 + ((j - 1) & 1)), ((j - 1) >> 1) & 1));
          if (ok) {
            tc_fence_after();
            const float alpha = need ? sfu_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tO + lane_base + c0, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + lane_base + c0, o);
            }
            tmem_wait_st();
            tc_fence_before();
            if (need) {
              lsum_all *= alpha;
              m_used = m_new;
            }
          }
        }
        if (m_used == -INFINITY) m_used = m_new;
        // P tile j & 1 is free once the PV MMAs of stage j - 2 have completed
        if (ok && j >= 2)
          ok = __all_sync(0xffffffffu,
                          mbar_wait_bounded(smem_u32(tcb + 6 + (j & 1)), ((j - 2) >> 1) & 1));
        if (!ok) {
          if (lane == 0) {
            flags[0] = 1;
            atomicOr(p.status, 0x1u);
          }
          break;
        }
        {
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          unsigned char *pt = pts + (j & 1) * PTILE;
          float ls = 0.f;
#pragma unroll
          for (int u = 0; u < KPC / 8; ++u) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              pv[e] = sfu_exp2(sv[8 * u + e] - mu);
              ls += pv[e];
            }
            uint4 w;
            w.x = pack2(pv[0], pv[1], tag{});
            w.y = pack2(pv[2], pv[3], tag{});
            w.z = pack2(pv[4], pv[5], tag{});
            w.w = pack2(pv[6], pv[7], tag{});
            const int key = c_first + 8 * u;           // first key of the 16-byte unit
            const int kc = key >> 6, uu = (key >> 3) & 7;  // 64-key chunk, unit of the row
            if (lane < 16)
              *reinterpret_cast<uint4 *>(pt + kc * 8192 + prow * 128 + ((uu ^ (prow & 7)) << 4)) = w;
          }
          lsum_all += ls;
        }
        // zero V of keys no row sees (outside the union, stale or NaN slots)
        if (!(nbt == TB && key_t0 >= u_lo && key_t0 + SC <= u_hi)) {
          unsigned char *vb = ring + slot * STAGE + TB * BLOCK_BYTES;
          for (int c = 32 * warp + lane; c < nbt * kBlockKeys; c += 128) {
            const int k = key_t0 + c;
            if (k < u_lo || k >= u_hi) {
#pragma unroll 1
              for (int x = 0; x < NBOX * 8; ++x)
                *reinterpret_cast<uint4 *>(vb + (c >> 4) * BLOCK_BYTES + (x >> 3) * 2048 +
                                           (c & 15) * 128 + (x & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();  // P and the zeroed V reach the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tcb + 4 + (j & 1)));  // P of stage j written
      }
      m0 = m_used;
      l0 = lsum_all;
    }
    } else if constexpr (DOT) {
    // ================= warp dot-product consumers (path 2) ================
    // A CTA of at most 8 packed rows (one n-tile), each warp group one warp.
    // Per stage, lane i takes keys i, i + 32, .. of the stage (KPL of them)
    // for S = Q K^T, dot products in fp32 over 8-dim chunks of its keys'
    // rows; the row maxima are shared by shuffles (sums stay per lane until
    // the end); P goes to the warp's buffer in shared memory; then lane i
    // takes dims [i * DPL, (i + 1) * DPL) of every row for O += P V, key by
    // key.  P stays fp32 (it is not rounded to the input dtype as the
    // tensor paths do).
    constexpr int SKEYS = TB * kBlockKeys;  // keys per stage
    constexpr int KPL = SKEYS / 32;         // keys per lane
    static_assert(!DOT || KPL >= 1, "a stage has at least 32 keys");
    const int nr = max(0, min(8, rr1v - rr0));  // real rows of this CTA
    int rlo[8], rhi[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      rlo[r] = 0;
      rhi[r] = 0;
      if (r < nr) {
        rhi[r] = max(L - ml + token_of(rr0 + r) + 1, 0);
        rlo[r] = p.window ? max(0, rhi[r] - p.window) : 0;
      }
    }
    {
      // the CTA's Q rows, widened to fp32 once (zeros past the real rows)
      const T *qbase = static_cast<const T *>(p.q);
      for (int idx = tid; idx < 8 * D; idx += NC * 32) {
        const int r = idx / D, d = idx - r * D;
        float v = 0.f;
        if (r < nr) {
          const int rr = rr0 + r, i = token_of(rr), jq = rr - i * p.G;
          const T qv = qbase[(int64_t)(q0 + i) * p.q_s0 + (int64_t)(h * p.G + jq) * p.q_s1 + d];
          if constexpr (BF16) v = __bfloat162float(qv);
          else v = __half2float(qv);
        }
        dot_q[idx] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
    }
    float *pbuf = dot_p + g_k * SKEYS * 8;
    int slot = g_k % NS, phase = (g_k / NS) & 1;
    for (int j = g_k; j < ntile; j += KG) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(full + slot), phase))) {
        if (lane == 0) {
          flags[0] = 1;
          atomicOr(p.status, 0x1u);
        }
        break;
      }
      const int nbt = min(TB, my_nb - j * TB);
      const unsigned char *kb = ring + slot * STAGE;
      const unsigned char *vb = kb + TB * BLOCK_BYTES;
      const int key_t0 = (my_b0 + j * TB) * kBlockKeys;
      // S = Q K^T for this lane's keys
      float sv[KPL][8];
#pragma unroll
      for (int i = 0; i < KPL; ++i)
#pragma unroll
        for (int r = 0; r < 8; ++r) sv[i][r] = 0.f;
#pragma unroll 2
      for (int c = 0; c < D / 8; ++c) {
        float kf[KPL][8];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
          const int key = lane + 32 * i, b = key >> 4, kk = key & 15;
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (b < nbt)
            w = *reinterpret_cast<const uint4 *>(kb + b * BLOCK_BYTES + (c >> 3) * 2048 + kk * 128 +
                                                 (((c & 7) ^ (kk & 7)) << 4));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f;
            if constexpr (BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ws[e]));
            else f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
            kf[i][2 * e] = f.x;
            kf[i][2 * e + 1] = f.y;
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < nr) {
            const float4 qa = *reinterpret_cast<const float4 *>(dot_q + r * D + 8 * c);
            const float4 qb = *reinterpret_cast<const float4 *>(dot_q + r * D + 8 * c + 4);
#pragma unroll
            for (int i = 0; i < KPL; ++i)
              sv[i][r] += qa.x * kf[i][0] + qa.y * kf[i][1] + qa.z * kf[i][2] + qa.w * kf[i][3] +
                          qb.x * kf[i][4] + qb.y * kf[i][5] + qb.z * kf[i][6] + qb.w * kf[i][7];
          }
        }
      }
      // scale, mask (keys past the stage, outside a row's range), row maxima
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < nr) {
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < KPL; ++i) {
            const int key = lane + 32 * i, k = key_t0 + key;
            const bool ok = key < nbt * kBlockKeys && k >= rlo[r] && k < rhi[r];
            sv[i][r] = ok ? sv[i][r] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, sv[i][r]);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float mn = fmaxf(dm[r], mx);
          const float mu = mn == -INFINITY ? 0.f : mn;
          const float al = sfu_exp2(dm[r] - mu);  // dm = -inf -> 0
          dm[r] = mn;
          float ls = 0.f;
#pragma unroll
          for (int i = 0; i < KPL; ++i) {
            sv[i][r] = sfu_exp2(sv[i][r] - mu);
            ls += sv[i][r];
          }
          dl[r] = dl[r] * al + ls;
#pragma unroll
          for (int jd = 0; jd < DPL; ++jd) dacc[r][jd] *= al;
        } else {
#pragma unroll
          for (int i = 0; i < KPL; ++i) sv[i][r] = 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < KPL; ++i) {
        float *dst = pbuf + (lane + 32 * i) * 8;
        *reinterpret_cast<float4 *>(dst) = make_float4(sv[i][0], sv[i][1], sv[i][2], sv[i][3]);
        *reinterpret_cast<float4 *>(dst + 4) = make_float4(sv[i][4], sv[i][5], sv[i][6], sv[i][7]);
      }
      __syncwarp();
      // O += P V: this lane's dims of every key the rows can see (keys
      // outside every row's range hold stale or NaN values: skipped)
      const int d0 = lane * DPL, box = d0 >> 6, chunk = (d0 & 63) >> 3, within = d0 & 7;
      const int kbeg = max(0, u_lo - key_t0), kend = min(nbt * kBlockKeys, u_hi - key_t0);
#pragma unroll 4
      for (int k = kbeg; k < kend; ++k) {
        const int b = k >> 4, kk = k & 15;
        const unsigned char *vp =
            vb + b * BLOCK_BYTES + box * 2048 + kk * 128 + ((chunk ^ (kk & 7)) << 4) + within * 2;
        float vf[DPL];
        if constexpr (DPL == 8) {
          const uint4 w = *reinterpret_cast<const uint4 *>(vp);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f;
            if constexpr (BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ws[e]));
            else f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
            vf[2 * e] = f.x;
            vf[2 * e + 1] = f.y;
          }
        } else if constexpr (DPL == 4) {
          const uint2 w = *reinterpret_cast<const uint2 *>(vp);
          const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float2 f;
            if constexpr (BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ws[e]));
            else f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
            vf[2 * e] = f.x;
            vf[2 * e + 1] = f.y;
          }
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(vp);
          float2 f;
          if constexpr (BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
          else f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
          vf[0] = f.x;
          if constexpr (DPL > 1) vf[1] = f.y;
        }
        const float4 pa = *reinterpret_cast<const float4 *>(pbuf + k * 8);
        const float4 pb = *reinterpret_cast<const float4 *>(pbuf + k * 8 + 4);
        const float pr[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (r < nr)
#pragma unroll
            for (int jd = 0; jd < DPL; ++jd) dacc[r][jd] += pr[r] * vf[jd];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + slot));
      slot += KG;
      while (slot >= NS) {
        slot -= NS;
        phase ^= 1;
      }
    }
    // full row sums (each lane summed its own keys)
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dl[r] += __shfl_xor_sync(0xffffffffu, dl[r], o);
    } else if constexpr (RM) {
    // ================= rows-on-M consumers (prefill tiles) =================
    // Warp w owns the packed rows 16w .. 16w + 15 (two n-tiles of the Q
    // tile) and every key of every stage, with the rows on the MMA's M side:
    //   S[16 rows x 8 keys]  = Q[16 x D] . K^T       (Q fragments in registers)
    //   O[16 rows x 8 dims] += P[16 x 16 keys] . V   (P straight from S's
    //                                                 accumulators)
    // so each stage is read from shared memory once per 16 rows, not once
    // per 8.  A row lives in the four lanes of one lane >> 2 class: two
    // xor-shuffles give its maximum.
    const int gq = lane >> 2, tq = lane & 3;  // fragment row and column pair
    const int ra = 16 * t_n + gq, rb = ra + 8;  // this lane's two rows
    int lo_a = 0, hi_a = 0, lo_b = 0, hi_b = 0;
    if (rr0 + ra < rr1v) {
      hi_a = max(L - ml + token_of(rr0 + ra) + 1, 0);
      lo_a = p.window ? max(0, hi_a - p.window) : 0;
    }
    if (rr0 + rb < rr1v) {
      hi_b = max(L - ml + token_of(rr0 + rb) + 1, 0);
      lo_b = p.window ? max(0, hi_b - p.window) : 0;
    }
    {
      // the Q tile, as for the other consumers
      const T *qbase = static_cast<const T *>(p.q);
      for (int idx = tid; idx < NT8 * (D / 8); idx += NC * 32) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const int rr = rr0 + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr < rr1v) {
          const int i = token_of(rr), jq = rr - i * p.G;
          v = __ldg(reinterpret_cast<const uint4 *>(qbase + (int64_t)(q0 + i) * p.q_s0 +
                                                    (int64_t)(h * p.G + jq) * p.q_s1 + c * 8));
        }
        const int tn = r >> 3, rw = r & 7, box = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(qs + (tn * NBOX + box) * 1024 + rw * 128 + ((cc ^ rw) << 4)) = v;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
    }
    // Q as the A operand (16 rows x 16 dims per k-step): matrices (rows 0-7 |
    // 8-15) x (dims 0-7 | 8-15) of the k-step
    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int j = lane >> 3, row = lane & 7;
      const int tn = 2 * t_n + (j & 1), chunk = 2 * ks + (j >> 1);
      ldsm_x4(smem_u32(qs) + (tn * NBOX + (chunk >> 3)) * 1024 + row * 128 +
                  (((chunk & 7) ^ row) << 4),
              qa[ks]);
    }
    // warp group g_k takes the stages g_k, g_k + KG, ..
    int slot = g_k % NS, phase = (g_k / NS) & 1;
    for (int j = g_k; j < ntile; j += KG) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(full + slot), phase))) {
        if (lane == 0) {
          flags[0] = 1;
          atomicOr(p.status, 0x1u);
        }
        break;
      }
      const int nbt = min(TB, my_nb - j * TB);
      const uint32_t kbase = smem_u32(ring + slot * STAGE);
      const uint32_t vbase = kbase + TB * BLOCK_BYTES;
      const int key_t0 = (my_b0 + j * TB) * kBlockKeys;
      constexpr int KN = TB * 2;  // 8-key n-tiles of the stage
      float sc[KN][4];
#pragma unroll
      for (int kn = 0; kn < KN; ++kn) sc[kn][0] = sc[kn][1] = sc[kn][2] = sc[kn][3] = 0.f;
      // S = Q K^T: K rows are [key][dims], the col-major B of the MMA;
      // one ldmatrix.x4 serves two n-tiles of one k-step
#pragma unroll
      for (int kn = 0; kn < KN; kn += 2) {
        if ((kn >> 1) < nbt) {  // both n-tiles of block kn / 2
          const int jm = lane >> 3, kk = (jm >> 1) * 8 + (lane & 7);  // key in the block
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int chunk = 2 * ks + (jm & 1);
            uint32_t b[4];
            ldsm_x4(kbase + (kn >> 1) * BLOCK_BYTES + (chunk >> 3) * 2048 + kk * 128 +
                        (((chunk & 7) ^ (kk & 7)) << 4),
                    b);
            mma_16816<BF16>(sc[kn], qa[ks], b[0], b[1]);
            mma_16816<BF16>(sc[kn + 1], qa[ks], b[2], b[3]);
          }
        }
      }
      // scale, mask, running max of rows ra and rb
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int kn = 0; kn < KN; ++kn) {
        const int k0 = key_t0 + kn * 8 + 2 * tq;
        const bool blk = (kn >> 1) < nbt;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = k0 + (e & 1);
          const bool ok = blk && ((e < 2) ? (k >= lo_a && k < hi_a) : (k >= lo_b && k < hi_b));
          sc[kn][e] = ok ? sc[kn][e] * p.scale_log2 : -INFINITY;
        }
        mxa = fmaxf(mxa, fmaxf(sc[kn][0], sc[kn][1]));
        mxb = fmaxf(mxb, fmaxf(sc[kn][2], sc[kn][3]));
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, o));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, o));
      }
      const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
      const float mua = mna == -INFINITY ? 0.f : mna, mub = mnb == -INFINITY ? 0.f : mnb;
      const float ala = sfu_exp2(m0 - mua), alb = sfu_exp2(m1 - mub);  // m = -inf -> 0
      m0 = mna;
      m1 = mnb;
      if (__any_sync(0xffffffffu, ala != 1.f || alb != 1.f)) {
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          racc[dn][0] *= ala;
          racc[dn][1] *= ala;
          racc[dn][2] *= alb;
          racc[dn][3] *= alb;
        }
      }
      l0 *= ala;
      l1 *= alb;
      // P = exp2(S - m) as the A operand of PV, 16 keys (two n-tiles) at a
      // time; V^T fragments by ldmatrix.trans, V of keys outside every row's
      // range zeroed (stale or NaN slots)
#pragma unroll
      for (int kb = 0; kb < TB; ++kb) {
        if (kb < nbt) {
          float pv[2][4];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            pv[u][0] = sfu_exp2(sc[2 * kb + u][0] - mua);
            pv[u][1] = sfu_exp2(sc[2 * kb + u][1] - mua);
            pv[u][2] = sfu_exp2(sc[2 * kb + u][2] - mub);
            pv[u][3] = sfu_exp2(sc[2 * kb + u][3] - mub);
            l0 += pv[u][0] + pv[u][1];
            l1 += pv[u][2] + pv[u][3];
          }
          uint32_t pa[4];
          pa[0] = pack2(pv[0][0], pv[0][1], tag{});
          pa[1] = pack2(pv[0][2], pv[0][3], tag{});
          pa[2] = pack2(pv[1][0], pv[1][1], tag{});
          pa[3] = pack2(pv[1][2], pv[1][3], tag{});
          const int key0 = key_t0 + kb * kBlockKeys;
          const bool vmask = !(key0 >= u_lo && key0 + kBlockKeys <= u_hi);
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (vmask) {
            const int ke = key0 + 2 * tq;
            mlo = ((ke >= u_lo && ke < u_hi) ? 0x0000ffffu : 0u) |
                  ((ke + 1 >= u_lo && ke + 1 < u_hi) ? 0xffff0000u : 0u);
            mhi = ((ke + 8 >= u_lo && ke + 8 < u_hi) ? 0x0000ffffu : 0u) |
                  ((ke + 9 >= u_lo && ke + 9 < u_hi) ? 0xffff0000u : 0u);
          }
          const int jm = lane >> 3, kk = (jm & 1) * 8 + (lane & 7);  // key of the block
          const uint32_t vb = vbase + kb * BLOCK_BYTES + kk * 128;
#pragma unroll
          for (int dn = 0; dn < D / 8; dn += 2) {
            const int chunk = dn + (jm >> 1);
            uint32_t b[4];
            ldsm_x4_trans(vb + (chunk >> 3) * 2048 + (((chunk & 7) ^ (kk & 7)) << 4), b);
            if (vmask) {
              b[0] &= mlo;
              b[1] &= mhi;
              b[2] &= mlo;
              b[3] &= mhi;
            }
            mma_16816<BF16>(racc[dn], pa, b[0], b[1]);
            mma_16816<BF16>(racc[dn + 1], pa, b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + slot));
      slot += KG;
      while (slot >= NS) {
        slot -= NS;
        phase ^= 1;
      }
    }
    // full row sums over the four lanes of a row
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    } else {
    // ================= consumers ==========================================
    // Visible key range of this thread's two rows (empty for padding rows).
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    {
      const int rra = rr0 + r0, rrb = rr0 + r1;
      if (rra < rr1v) {
        hi0 = max(L - ml + token_of(rra) + 1, 0);
        lo0 = p.window ? max(0, hi0 - p.window) : 0;
      }
      if (rrb < rr1v) {
        hi1 = max(L - ml + token_of(rrb) + 1, 0);
        lo1 = p.window ? max(0, hi1 - p.window) : 0;
      }
    }
    {
      // the Q tile: packed rows of this CTA, 16-byte chunks, 128B-swizzled
      const T *qbase = static_cast<const T *>(p.q);
      for (int idx = tid; idx < NT8 * (D / 8); idx += NC * 32) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const int rr = rr0 + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rr < rr1v) {
          const int i = token_of(rr), j = rr - i * p.G;
          v = __ldg(reinterpret_cast<const uint4 *>(qbase + (int64_t)(q0 + i) * p.q_s0 +
                                                    (int64_t)(h * p.G + j) * p.q_s1 + c * 8));
        }
        const int tn = r >> 3, rw = r & 7, box = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(qs + (tn * NBOX + box) * 1024 + rw * 128 + ((cc ^ rw) << 4)) = v;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
    }
    const uint32_t qs_u32 = smem_u32(qs) + t_n * NBOX * 1024;
    uint32_t qf[Q_IN_REGS ? KS : 1][2];
    if constexpr (Q_IN_REGS) {
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        const int row = lane & 7, chunk = 2 * ks + (lane >> 3);
        uint32_t r[4];
        ldsm_x4(qs_u32 + (chunk >> 3) * 1024 + row * 128 + (((chunk & 7) ^ row) << 4), r);
        qf[ks][0] = r[0];
        qf[ks][1] = r[1];
        qf[ks + 1][0] = r[2];
        qf[ks + 1][1] = r[3];
      }
    }
    const int k_row = lane & 15, k_hi = lane >> 4;                     // K ldmatrix roles
    const int v_row = (lane & 7) + ((lane >> 4) << 3), v_hi = (lane >> 3) & 1;  // V^T roles

    int slot = g_k % NS, phase = (g_k / NS) & 1;  // ring slot of tile j and its round parity
    for (int j = g_k; j < ntile; j += KG) {
      // one verdict for the warp, so no lane leaves the shuffles alone
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(full + slot), phase))) {
        if (lane == 0) {
          flags[0] = 1;
          atomicOr(p.status, 0x1u);
        }
        break;
      }
      const int nbt = min(TB, my_nb - j * TB);
      const uint32_t kbase = smem_u32(ring + slot * STAGE);
      const uint32_t vbase = kbase + TB * BLOCK_BYTES;
      const int key_t0 = (my_b0 + j * TB) * kBlockKeys;

      // S^T = K Q^T for every block of the stage
      float sc[TB][4];
#pragma unroll
      for (int b = 0; b < TB; ++b) sc[b][0] = sc[b][1] = sc[b][2] = sc[b][3] = 0.f;
      if constexpr (Q_IN_REGS) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int chunk = 2 * ks + k_hi;
          const uint32_t off = (chunk >> 3) * 2048 + k_row * 128 + (((chunk & 7) ^ (k_row & 7)) << 4);
#pragma unroll
          for (int b = 0; b < TB; ++b) {
            if (b < nbt) {
              uint32_t a[4];
              ldsm_x4(kbase + b * BLOCK_BYTES + off, a);
              mma_16816<BF16>(sc[b], a, qf[ks][0], qf[ks][1]);
            }
          }
        }
      } else {
        // D = 512: one block per stage; two accumulators break the k-step chain
        float sc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          uint32_t qr[4];
          {
            const int row = lane & 7, chunk = 2 * ks + (lane >> 3);
            ldsm_x4(qs_u32 + (chunk >> 3) * 1024 + row * 128 + (((chunk & 7) ^ row) << 4), qr);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int chunk = 2 * (ks + u) + k_hi;
            uint32_t a[4];
            ldsm_x4(kbase + (chunk >> 3) * 2048 + k_row * 128 +
                        (((chunk & 7) ^ (k_row & 7)) << 4),
                    a);
            if (u == 0)
              mma_16816<BF16>(sc[0], a, qr[0], qr[1]);
            else
              mma_16816<BF16>(sc2, a, qr[2], qr[3]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[0][e] += sc2[e];
      }

      // scale, mask, running max
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int b = 0; b < TB; ++b) {
        const int key0 = key_t0 + b * kBlockKeys;
        if (b >= nbt) {
          sc[b][0] = sc[b][1] = sc[b][2] = sc[b][3] = -INFINITY;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[b][e] *= p.scale_log2;
          if (!(key0 >= v_lo && key0 + kBlockKeys <= v_hi)) {
            const int ka = key0 + (lane >> 2), kb = ka + 8;
            if (!(ka >= lo0 && ka < hi0)) sc[b][0] = -INFINITY;
            if (!(ka >= lo1 && ka < hi1)) sc[b][1] = -INFINITY;
            if (!(kb >= lo0 && kb < hi0)) sc[b][2] = -INFINITY;
            if (!(kb >= lo1 && kb < hi1)) sc[b][3] = -INFINITY;
          }
        }
        mx0 = fmaxf(mx0, fmaxf(sc[b][0], sc[b][2]));
        mx1 = fmaxf(mx1, fmaxf(sc[b][1], sc[b][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = sfu_exp2(m0 - mu0), al1 = sfu_exp2(m1 - mu1);  // m = -inf -> 0
      m0 = mn0;
      m1 = mn1;
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          acc[i][0] *= al0;
          acc[i][1] *= al1;
          acc[i][2] *= al0;
          acc[i][3] *= al1;
        }
      }
      l0 *= al0;
      l1 *= al1;

      // P = exp2(S - m); PV
#pragma unroll
      for (int b = 0; b < TB; ++b) {
        if (b < nbt) {
          const float p0 = sfu_exp2(sc[b][0] - mu0), p1 = sfu_exp2(sc[b][1] - mu1);
          const float p2 = sfu_exp2(sc[b][2] - mu0), p3 = sfu_exp2(sc[b][3] - mu1);
          l0 += p0 + p2;
          l1 += p1 + p3;
          const uint32_t pb0 = movmatrix_trans(pack2(p0, p1, tag{}));
          const uint32_t pb1 = movmatrix_trans(pack2(p2, p3, tag{}));
          const int key0 = key_t0 + b * kBlockKeys;
          const bool vmask = !(key0 >= u_lo && key0 + kBlockKeys <= u_hi);
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (vmask) {
            // zero V of keys outside every row's range (stale or NaN slots)
            const int ke = key0 + 2 * (lane & 3);
            mlo = ((ke >= u_lo && ke < u_hi) ? 0x0000ffffu : 0u) |
                  ((ke + 1 >= u_lo && ke + 1 < u_hi) ? 0xffff0000u : 0u);
            mhi = ((ke + 8 >= u_lo && ke + 8 < u_hi) ? 0x0000ffffu : 0u) |
                  ((ke + 9 >= u_lo && ke + 9 < u_hi) ? 0xffff0000u : 0u);
          }
          const uint32_t vb = vbase + b * BLOCK_BYTES;
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            const int chunk = 2 * mt + v_hi;
            uint32_t a[4];
            ldsm_x4_trans(vb + (chunk >> 3) * 2048 + v_row * 128 + (((chunk & 7) ^ (v_row & 7)) << 4),
                          a);
            if (vmask) {
              a[0] &= mlo;
              a[1] &= mlo;
              a[2] &= mhi;
              a[3] &= mhi;
            }
            mma_16816<BF16>(acc[mt], a, pb0, pb1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + slot));
      slot += KG;
      while (slot >= NS) {
        slot -= NS;
        phase ^= 1;
      }
    }
    // full row sums: the 8 lanes of one (lane & 3) class hold one row pair
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    }
  }

  // ================= epilogue ==============================================
  // The next grid on the stream may start launching now (its CTAs wait at
  // their own grid_dependency_wait until this grid has completed).
  grid_dependents_launch();
  __syncthreads();  // ring and Q tile are dead from here on
  float *ep = reinterpret_cast<float *>(smem);
  float *cp = ep;                          // [KG][NT8][D] (swizzled columns)
  float *mrow = cp + (size_t)KG * NT8 * D;  // [KG][NT8]
  float *lrow = mrow + KG * NT8;
  float *mfin = lrow + KG * NT8;  // [NT8]
  float *lfin = mfin + NT8;

  T *obase = static_cast<T *>(p.out);
  auto out_row = [&](int r) -> T * {
    const int rr = rr0 + r;
    const int i = token_of(rr);
    const int j = rr - i * p.G;
    return obase + (int64_t)(q0 + i) * p.o_s0 + (int64_t)(h * p.G + j) * p.o_s1;
  };
  const int nrows = max(0, rr1v - rr0);  // valid rows of this CTA
  if (p.query_start && (prefill ? blockIdx.x == 0 && blockIdx.y == 0 : seg == 0 && hg == 0 && s == 0)) {
    // rows at and past the last request's end (padding of a captured batch)
    // see no key: zeros
    const int t0 = min(max(__ldg(p.query_start + p.num_seqs), 0), p.num_tokens);
    const int per_row = p.Hq * (D / 8);
#pragma unroll 1
    for (int64_t i = tid; i < (int64_t)(p.num_tokens - t0) * per_row; i += blockDim.x) {
      const int t = t0 + (int)(i / per_row), rem = (int)(i - (int64_t)(t - t0) * per_row);
      const int hq = rem / (D / 8), c = rem - hq * (D / 8);
      *reinterpret_cast<uint4 *>(obase + (int64_t)t * p.o_s0 + (int64_t)hq * p.o_s1 + c * 8) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }

  const int CS = p.CS;
  const int DS = D / CS;
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0u;
  // split-KV counters and partial slots of this (sequence, kv head, row
  // group), or of this prefill tile and kv head (its segments' slots are
  // consecutive from the item's first slot)
  const int group = prefill ? pf_split * p.Hkv + h : (s * p.Hkv + h) * p.rg + grow;
  const int64_t gbase =
      prefill ? (int64_t)pf_slot * p.Hkv + (int64_t)h * pf_nseg : (int64_t)group * p.max_parts;
  const int64_t slice_floats = (int64_t)NT8 * DS;

  if constexpr (TP) {
    // O of each tile (tensor memory) -> the CTA's partial in shared memory
    // (KG = 1): row 128 X + 32 (w % 4) + lane of softmax warp w of tile X,
    // once every MMA has completed
    if (warp < kTpSoftmaxWarps) {
      const bool done = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 12), 0));
      tc_fence_after();
      const int g = warp >> 2, r = kTpRows * g + 32 * (warp & 3) + lane;
      const bool keep = r < NT8;
      const bool have = ntile > 0 && done;
      const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
      float *dst = cp + (size_t)r * D;
      if (nseg == 1) {
        // an unsplit tile: each row normalised and stored from here
        const float inv = (have && l0 > 0.f) ? sfu_rcp(l0) : 0.f;
        T *orow = r < nrows ? out_row(r) : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem_base + tp_o_col(D) + g * D + lane_base + c0, o);
          tmem_wait_ld();
          if (orow) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              const float v[8] = {__uint_as_float(o[i]) * inv,     __uint_as_float(o[i + 1]) * inv,
                                  __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv,
                                  __uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv,
                                  __uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv};
              store8<BF16>(orow + c0 + i, v);
            }
          }
        }
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D && nseg > 1; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem_base + tp_o_col(D) + g * D + lane_base + c0, o);
        tmem_wait_ld();
        if (keep) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 v = have ? make_float4(__uint_as_float(o[i]), __uint_as_float(o[i + 1]),
                                                __uint_as_float(o[i + 2]), __uint_as_float(o[i + 3]))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(dst + psw(c0 + i, r)) = v;
          }
        }
      }
      if (keep) {
        mrow[r] = have ? m0 : -INFINITY;
        lrow[r] = have ? l0 : 0.f;
      }
      if (!done && lane == 0) atomicOr(p.status, 0x1u);
    }
    tc_fence_before();
  } else if constexpr (TC) {
    // O (tensor memory) -> the CTA's partial in shared memory (one warp group,
    // KG = 1), one row per thread, once every MMA has completed
    if (warp < kTcConsumerWarps - 1) {
      const bool done = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(tcb + 8), 0));
      tc_fence_after();
      // copy q = warp q is warp group q of the partial pass (KG = 4)
      const int r = lane & 15;
      const bool keep = lane < 16 && r < NT8;
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      float *dst = cp + ((size_t)warp * NT8 + r) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem_base + 2 * SC + lane_base + c0, o);
        tmem_wait_ld();
        if (keep) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 v = (ntile > 0 && done)
                                 ? make_float4(__uint_as_float(o[i]), __uint_as_float(o[i + 1]),
                                               __uint_as_float(o[i + 2]), __uint_as_float(o[i + 3]))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(dst + psw(c0 + i, r)) = v;
          }
        }
      }
      if (keep) {
        mrow[warp * NT8 + r] = (ntile > 0 && done) ? m0 : -INFINITY;
        lrow[warp * NT8 + r] = (ntile > 0 && done) ? l0 : 0.f;
      }
      if (!done && lane == 0) atomicOr(p.status, 0x1u);
    }
    tc_fence_before();
  } else if (DOT && warp < NC && lane == 0) {
    // (the row maxima and sums are the same in every lane)
#pragma unroll
    for (int r = 0; r < (DOT ? 8 : 1); ++r) {
      mrow[g_k * NT8 + r] = dm[r];
      lrow[g_k * NT8 + r] = dl[r];
    }
  } else if (RM && warp < NC && (lane & 3) == 0) {
    const int ra = g_k * NT8 + 16 * t_n + (lane >> 2);
    mrow[ra] = m0;
    mrow[ra + 8] = m1;
    lrow[ra] = l0;
    lrow[ra + 8] = l1;
  } else if (!DOT && !RM && warp < NC && lane < 4) {
    mrow[g_k * NT8 + r0] = m0;
    mrow[g_k * NT8 + r1] = m1;
    lrow[g_k * NT8 + r0] = l0;
    lrow[g_k * NT8 + r1] = l1;
  }
  if constexpr (TP) {
    if (nseg == 1) {
      // every row was stored from tensor memory above: free it and leave
      __syncthreads();
      if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
      }
      return;
    }
  }
  if (CS == 1) {
    // ---- no cluster: one pass over the warp groups' raw accumulators -------
    // Each warp stores its fragment unscaled (rows of D fp32, columns
    // swizzled) next to its rows' (m, l), so one barrier separates the
    // stores from the pass that forms every (row, 4 columns) item of the
    // CTA's partial: sum over the groups of acc_g * exp2(m_g - m*), then
    // normalised (one segment) or published (several).
    if (DOT && warp < NC) {
      float *dst = cp + (size_t)g_k * NT8 * D;
#pragma unroll
      for (int r = 0; r < (DOT ? 8 : 1); ++r)
#pragma unroll
        for (int jd = 0; jd < DPL; ++jd) {
          const int d = lane * DPL + jd;
          dst[r * D + psw(d, r)] = dacc[r][jd];
        }
    } else if (RM && warp < NC) {
      float *dst = cp + (size_t)g_k * NT8 * D;
      const int ra = 16 * t_n + (lane >> 2), rb = ra + 8;
#pragma unroll
      for (int dn = 0; dn < (RM ? D / 8 : 1); ++dn) {
        const int d = dn * 8 + 2 * (lane & 3);
        dst[ra * D + psw(d, ra)] = racc[dn][0];
        dst[ra * D + psw(d + 1, ra)] = racc[dn][1];
        dst[rb * D + psw(d, rb)] = racc[dn][2];
        dst[rb * D + psw(d + 1, rb)] = racc[dn][3];
      }
    } else if (!TC && !TP && warp < NC) {
      float *dst = cp + (size_t)g_k * NT8 * D;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d = mt * 16 + (lane >> 2);
        dst[r0 * D + psw(d, r0)] = acc[mt][0];
        dst[r1 * D + psw(d, r1)] = acc[mt][1];
        dst[r0 * D + psw(d + 8, r0)] = acc[mt][2];
        dst[r1 * D + psw(d + 8, r1)] = acc[mt][3];
      }
    }
    __syncthreads();
    if constexpr (TC || TP) {
      // every read of tensor memory is done
      if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
      }
    }
    const int DKm = p.coop ? D >> (__ffs(p.mergers) - 1) : D;  // K_max a power of two
    const int lg_dkm = __ffs(DKm) - 1;
    float *pa = p.part_acc + (gbase + cl_id) * (int64_t)NT8 * D;
    float2 *pm = reinterpret_cast<float2 *>(p.part_ml + (gbase + cl_id) * NT8 * 2);
    // one item = (row, kCols columns), every load of an item issued at once;
    // 4 columns when that gives every thread at most one item, else 16
    auto items_pass = [&](auto cols) {
    constexpr int kCols = decltype(cols)::value, kItemsPerRow = D / kCols;
#pragma unroll 1
    for (int idx = tid; idx < nrows * kItemsPerRow; idx += blockDim.x) {
      // the item's 4-column groups are kItemsPerRow groups apart, so the
      // threads of a row read consecutive 16-byte words (no bank conflicts)
      const int r = idx / kItemsPerRow, t4 = (idx % kItemsPerRow) * 4;
      constexpr int kStride = 4 * kItemsPerRow;
      float ms = -INFINITY;
#pragma unroll
      for (int gg = 0; gg < kMaxConsumerWarps; ++gg)
        if (gg < KG) ms = fmaxf(ms, mrow[gg * NT8 + r]);
      const float mu = ms == -INFINITY ? 0.f : ms;
      float4 a[kCols / 4];
#pragma unroll
      for (int v = 0; v < kCols / 4; ++v) a[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      float lsum = 0.f;
      constexpr int kGroupChunk = 4;  // warp groups whose loads are in flight at once
#pragma unroll 1
      for (int g0 = 0; g0 < KG; g0 += kGroupChunk) {
        float mg[kGroupChunk], lg[kGroupChunk];
        float4 b[kGroupChunk][kCols / 4];
#pragma unroll
        for (int u = 0; u < kGroupChunk; ++u) {
          const int gg = g0 + u;
          if (gg < KG) {
            mg[u] = mrow[gg * NT8 + r];
            lg[u] = lrow[gg * NT8 + r];
#pragma unroll
            for (int v = 0; v < kCols / 4; ++v)
              b[u][v] = *reinterpret_cast<const float4 *>(cp + ((size_t)gg * NT8 + r) * D +
                                                          psw(t4 + kStride * v, r));
          } else {
            mg[u] = -INFINITY;
            lg[u] = 0.f;
#pragma unroll
            for (int v = 0; v < kCols / 4; ++v) b[u][v] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < kGroupChunk; ++u) {
          if (g0 + u >= KG) break;
          const float w = exp2_or_zero(mg[u], mu);
          lsum += w * lg[u];
#pragma unroll
          for (int v = 0; v < kCols / 4; ++v) {
            a[v].x += w * b[u][v].x;
            a[v].y += w * b[u][v].y;
            a[v].z += w * b[u][v].z;
            a[v].w += w * b[u][v].w;
          }
        }
      }
      if (nseg == 1) {
        const float inv = lsum > 0.f ? sfu_rcp(lsum) : 0.f;
#pragma unroll
        for (int v = 0; v < kCols / 4; ++v) {
          const float o[4] = {a[v].x * inv, a[v].y * inv, a[v].z * inv, a[v].w * inv};
          store4<BF16>(out_row(r) + t4 + kStride * v, o);
        }
      } else {
        // DKm is a power of two (>= 4)
#pragma unroll
        for (int v = 0; v < kCols / 4; ++v) {
          const int d4 = t4 + kStride * v, k = d4 >> lg_dkm, dk = d4 & (DKm - 1);
          __stcg(reinterpret_cast<float4 *>(pa + ((int64_t)k * NT8 + r) * DKm + dk), a[v]);
        }
        if (t4 == 0) __stcg(pm + r, make_float2(ms, lsum));
      }
    }
    };
    if (nrows * (D / 4) <= (int)blockDim.x)
      items_pass(std::integral_constant<int, 4>{});
    else
      items_pass(std::integral_constant<int, 16>{});
    if (nseg == 1) return;
  } else {
  __syncthreads();
  if constexpr (TC || TP) {
    // (clusters are not planned on the tensor-memory paths; free it anyway)
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem_base, TMEM_COLS);
    }
  }
  if (!TC && !TP && warp < NC) {
    float ms0 = -INFINITY, ms1 = -INFINITY;
#pragma unroll 1
    for (int gg = 0; gg < KG; ++gg) {
      ms0 = fmaxf(ms0, mrow[gg * NT8 + r0]);
      ms1 = fmaxf(ms1, mrow[gg * NT8 + r1]);
    }
    const float f0 = exp2_or_zero(m0, ms0 == -INFINITY ? 0.f : ms0);
    const float f1 = exp2_or_zero(m1, ms1 == -INFINITY ? 0.f : ms1);
    float *dst = cp + (size_t)g_k * NT8 * D;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      const int d = mt * 16 + (lane >> 2);
      dst[r0 * D + psw(d, r0)] = acc[mt][0] * f0;
      dst[r1 * D + psw(d, r1)] = acc[mt][1] * f1;
      dst[r0 * D + psw(d + 8, r0)] = acc[mt][2] * f0;
      dst[r1 * D + psw(d + 8, r1)] = acc[mt][3] * f1;
    }
  }
  __syncthreads();
  if (KG > 1) {
#pragma unroll 1
    for (int idx = tid; idx < NT8 * D / 4; idx += blockDim.x) {
      float4 a = reinterpret_cast<float4 *>(cp)[idx];
#pragma unroll 1
      for (int gg = 1; gg < KG; ++gg) {
        const float4 b = reinterpret_cast<float4 *>(cp + (size_t)gg * NT8 * D)[idx];
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      reinterpret_cast<float4 *>(cp)[idx] = a;
    }
  }
#pragma unroll 1
  for (int r = tid; r < NT8; r += blockDim.x) {
    float ms = -INFINITY;
#pragma unroll 1
    for (int gg = 0; gg < KG; ++gg) ms = fmaxf(ms, mrow[gg * NT8 + r]);
    const float mu = ms == -INFINITY ? 0.f : ms;
    float lsum = 0.f;
#pragma unroll 1
    for (int gg = 0; gg < KG; ++gg) lsum += lrow[gg * NT8 + r] * exp2_or_zero(mrow[gg * NT8 + r], mu);
    mfin[r] = ms;
    lfin[r] = lsum;
  }
  __syncthreads();

  if (nseg == 1) {
    // one segment: normalise and store
#pragma unroll 1
    for (int idx = tid; idx < nrows * (D / 8); idx += blockDim.x) {
      const int r = idx / (D / 8), c8 = (idx % (D / 8)) * 8;
      const float lr = lfin[r];
      const float inv = lr > 0.f ? sfu_rcp(lr) : 0.f;
      const float4 a = *reinterpret_cast<const float4 *>(cp + r * D + psw(c8, r));
      const float4 b = *reinterpret_cast<const float4 *>(cp + r * D + psw(c8 + 4, r));
      const float v[8] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv,
                          b.x * inv, b.y * inv, b.z * inv, b.w * inv};
      store8<BF16>(out_row(r) + c8, v);
    }
    return;
  }

  // ---- combine the segments of this cluster ------------------------------
  // cluster size 1: the CTA partial (cp, swizzled, full D) is the cluster's
  float *clp = lfin + NT8;               // [NT8][DS] cluster partial slice (CS > 1)
  float *mcl = CS > 1 ? clp + NT8 * DS : mfin;
  float *lcl = CS > 1 ? mcl + NT8 : lfin;
  if (CS > 1) {
    float *wts = lcl + NT8;  // [CS][NT8]
    cluster_sync();          // every CTA's partial is in its shared memory
#pragma unroll 1
    for (int r = tid; r < NT8; r += blockDim.x) {
      float mr[8];
      float ms = -INFINITY;
#pragma unroll 1
      for (int x = 0; x < CS; ++x) {
        mr[x] = ld_dsmem_f32(mapa(smem_u32(mfin + r), x));
        ms = fmaxf(ms, mr[x]);
      }
      const float mu = ms == -INFINITY ? 0.f : ms;
      float lsum = 0.f;
#pragma unroll 1
      for (int x = 0; x < CS; ++x) {
        const float w = exp2_or_zero(mr[x], mu);
        lsum += ld_dsmem_f32(mapa(smem_u32(lfin + r), x)) * w;
        wts[x * NT8 + r] = w;
      }
      mcl[r] = ms;
      lcl[r] = lsum;
    }
    __syncthreads();
#pragma unroll 1
    for (int idx = tid; idx < NT8 * (DS / 4); idx += blockDim.x) {
      const int r = idx / (DS / 4), d = (int)rank * DS + (idx % (DS / 4)) * 4;
      const uint32_t local = smem_u32(cp + r * D + psw(d, r));
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int x = 0; x < CS; ++x) {
        const float w = wts[x * NT8 + r];
        const float4 b = ld_dsmem_f32x4(mapa(local, x));
        a.x += w * b.x;
        a.y += w * b.y;
        a.z += w * b.z;
        a.w += w * b.w;
      }
      *reinterpret_cast<float4 *>(clp + r * DS + (d - (int)rank * DS)) = a;
    }
    cluster_sync();  // no CTA reads another's shared memory after this
  }
  // element (r, d) of this CTA's slice of the cluster partial
  auto part4 = [&](int r, int d4) -> float4 {
    return CS > 1 ? *reinterpret_cast<const float4 *>(clp + r * DS + d4)
                  : *reinterpret_cast<const float4 *>(cp + r * D + psw(d4, r));
  };

  if (ncl == 1) {
#pragma unroll 1
    for (int idx = tid; idx < nrows * (DS / 8); idx += blockDim.x) {
      const int r = idx / (DS / 8), c8 = (idx % (DS / 8)) * 8;
      const float lr = lcl[r];
      const float inv = lr > 0.f ? sfu_rcp(lr) : 0.f;
      const float4 a = part4(r, c8), b = part4(r, c8 + 4);
      const float v[8] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv,
                          b.x * inv, b.y * inv, b.z * inv, b.w * inv};
      store8<BF16>(out_row(r) + (int)rank * DS + c8, v);
    }
    return;
  }

  // ---- several clusters: publish this cluster's partial, count arrivals ----
  // Global partials of a group: acc [max_parts][CS][NT8][DS] (each CTA's
  // slice contiguous, valid rows only), (m, l) [max_parts][NT8].
  if (p.coop) {
    // layout [part][K_max][NT8][D/K_max]: a merger's slice is one block
    const int DKm = D / p.mergers;
    float *pa = p.part_acc + (gbase + cl_id) * (int64_t)NT8 * D;
#pragma unroll 1
    for (int idx = tid; idx < nrows * (D / 4); idx += blockDim.x) {
      const int r = idx / (D / 4), d4 = (idx % (D / 4)) * 4;
      const int k = d4 / DKm, dk = d4 % DKm;
      __stcg(reinterpret_cast<float4 *>(pa + ((int64_t)k * NT8 + r) * DKm + dk), part4(r, d4));
    }
  } else {
    float *pa = p.part_acc + ((gbase + cl_id) * CS + rank) * slice_floats;
#pragma unroll 1
    for (int idx = tid; idx < nrows * (DS / 4); idx += blockDim.x) {
      const int r = idx / (DS / 4), d4 = (idx % (DS / 4)) * 4;
      __stcg(reinterpret_cast<float4 *>(pa + (int64_t)r * DS + d4), part4(r, d4));
    }
  }
  {
    if (rank == 0) {
      float2 *pm = reinterpret_cast<float2 *>(p.part_ml + (gbase + cl_id) * NT8 * 2);
#pragma unroll 1
      for (int r = tid; r < nrows; r += blockDim.x) __stcg(pm + r, make_float2(mcl[r], lcl[r]));
    }
  }
  }
  // The barrier orders every thread's stores before thread 0's release
  // (acq_rel) increment of the counter; the last arriver's acquire then
  // orders every cluster's partial before its reads (the split-K semaphore
  // pattern: stores, barrier, one release by one thread).
  if (CS > 1)
    cluster_sync();
  else
    __syncthreads();

  if (p.coop) {
    // ---- co-resident grid: the last K arrivals merge one D/K slice each ----
    // Every CTA of a cooperative launch is resident, so a merger waiting for
    // the remaining arrivals waits on CTAs that are running (bounded).
    // K = the largest power of two <= min(K_max, arrivals of this group).
    int K = 1, lg_k = 0;
    while (2 * K <= min(p.mergers, ncl)) {
      K *= 2;
      ++lg_k;
    }
    // Thread 0 counts the CTA in; a merger that is not the last arrival
    // waits there for the rest (the last one knows from the count that
    // every part is published, and its acquire already covers them).
    if (tid == 0) {
      const int old = atomic_add_acq_rel_gpu(p.counters + 2 * group, 1);
      int m = old - (ncl - K);
      int ok = 1;
      if (old < 0 || old >= ncl) {
        // the counter did not start this launch at zero (a scratch shared by
        // overlapping calls, or left behind by a merger that gave up): no
        // merge from it; every later index stays in bounds
        atomicOr(p.status, 0x10u);
        m = -1;
      } else if (m >= 0 && old != ncl - 1 && ld_acquire_gpu(p.counters + 2 * group) < ncl) {
        const unsigned long long t0 = global_timer_ns();
        while (ld_acquire_gpu(p.counters + 2 * group) < ncl) {
          __nanosleep(64);
          if (global_timer_ns() - t0 > p.wait_limit_ns) {
            ok = 0;
            atomicOr(p.status, 0x1u);
            // poison the group's arrival count so that the next launch on
            // this scratch sees it out of range (and reports it) instead of
            // electing mergers from a stale count; the scratch must be
            // initialised again before it serves another call.  The sign bit
            // keeps the count below ncl, so a merger of this launch still
            // polling keeps waiting (and gives up in turn) rather than take
            // the poison for the last arrival.
            atomicOr(p.counters + 2 * group, (int)0x80000000u);
            break;
          }
        }
      }
      flags[1] = m;
      flags[2] = ok;
    }
    __syncthreads();
    const int mi = flags[1];
    if (mi < 0 || mi >= K) return;  // not one of the last K arrivals
    if (!flags[2]) return;
    // count this merger past its wait now; the answer is needed only at the
    // end, so the round trip overlaps the merge
    const int fin_old = tid == 0 ? atomicAdd(p.counters + 2 * group + 1, 1) : 0;
    // this merger's layout slices: [mi * q, (mi + 1) * q) of the K_max slices
    const int lg_km = __ffs(p.mergers) - 1;
    const int DKm = D >> lg_km, q = p.mergers >> lg_k, DK = q * DKm;
    const int64_t part_floats = (int64_t)NT8 * D;
    const int slab = q * NT8 * DKm;  // floats of one part's share
    if (ncl * (2 * NT8 + slab) + 64 <= p.epi_floats &&
        nrows * (DK / 4) <= (int)blockDim.x) {
    // every part fits in shared memory at once and each thread has at most
    // one item: one round of copies, one pass
    float *ml_s = ep;                    // [ncl][NT8][2] (m, l) of every part
    float *buf = ml_s + 2 * ncl * NT8;   // [ncl][q][NT8][DKm]
    // Every part's (m, l) and this merger's share of every part, brought into
    // shared memory by 16-byte asynchronous copies from every thread, all in
    // flight at once (one L2 round trip).
    {
      const int slab4 = slab / 4, n_ml4 = ncl * NT8 / 2;
      const int64_t part4 = part_floats / 4;
      const float4 *ml_g = reinterpret_cast<const float4 *>(p.part_ml + gbase * NT8 * 2);
      const float4 *acc_g = reinterpret_cast<const float4 *>(p.part_acc + gbase * part_floats) +
                            (int64_t)mi * slab4;
      const int nwarps = blockDim.x >> 5;
#pragma unroll 1
      for (int i = tid; i < n_ml4; i += blockDim.x) cp_async16(ml_s + 4 * i, ml_g + i);
#pragma unroll 1
      for (int c = warp; c < ncl; c += nwarps) {
#pragma unroll 1
        for (int j = lane; j < slab4; j += 32)
          cp_async16(buf + ((int64_t)c * slab4 + j) * 4, acc_g + c * part4 + j);
      }
      cp_async_wait_all();
    }
    __syncthreads();
    // TPI threads (a power of two, adjacent lanes) per (row, 4 columns) item
    // of the slice.  Parts are taken 8 * TPI at a time: each thread loads its
    // eight (m, l) and accumulator rows at once, the chunk's largest m is
    // shared by shuffles, and the running sums are rescaled when it grows
    // (online softmax over the parts); the TPI threads' sums are then added
    // by shuffles.  DKm and DK / 4 are powers of two.
    const int lg_dkm = __ffs(DKm) - 1, lg_i = __ffs(DK / 4) - 1;
    const int n_items = nrows << lg_i;
    int lgT = 0;
    while (lgT < 5 && (2 << lgT) * n_items <= (int)blockDim.x) ++lgT;
    const int TPI = 1 << lgT;  // threads per item
    constexpr int kChunk = 8;
#pragma unroll 1
    for (int base = 0; base < n_items * TPI; base += blockDim.x) {
      const int item = (base + tid) >> lgT, sub = (base + tid) & (TPI - 1);
      const bool active = item < n_items;
      const int r = active ? item >> lg_i : 0, dd = active ? (item & ((DK >> 2) - 1)) * 4 : 0;
      const float2 *mlr = reinterpret_cast<const float2 *>(ml_s) + r;
      const float *src = buf + ((int64_t)(dd >> lg_dkm) * NT8 + r) * DKm + (dd & (DKm - 1));
      float M = -INFINITY, lr = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int c0 = 0; c0 < ncl; c0 += kChunk * TPI) {
        float2 mv[kChunk];
        float4 bv[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
          const int c = c0 + sub + u * TPI;
          if (active && c < ncl) {
            mv[u] = mlr[c * NT8];
            bv[u] = *reinterpret_cast<const float4 *>(src + (int64_t)c * slab);
          } else {
            mv[u] = make_float2(-INFINITY, 0.f);
            bv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        float cm = M;
#pragma unroll
        for (int u = 0; u < kChunk; ++u) cm = fmaxf(cm, mv[u].x);
#pragma unroll 1
        for (int o = 1; o < TPI; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        const float mu = cm == -INFINITY ? 0.f : cm;
        const float sc = exp2_or_zero(M, mu);
        lr *= sc;
        a.x *= sc;
        a.y *= sc;
        a.z *= sc;
        a.w *= sc;
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
          const float w = exp2_or_zero(mv[u].x, mu);
          lr += w * mv[u].y;
          a.x += w * bv[u].x;
          a.y += w * bv[u].y;
          a.z += w * bv[u].z;
          a.w += w * bv[u].w;
        }
        M = cm;
      }
#pragma unroll 1
      for (int o = 1; o < TPI; o <<= 1) {
        lr += __shfl_xor_sync(0xffffffffu, lr, o);
        a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
        a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
        a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
        a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
      }
      if (active && sub == 0) {
        const float inv = lr > 0.f ? sfu_rcp(lr) : 0.f;
        const float v[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
        store4<BF16>(out_row(r) + mi * DK + dd, v);
      }
    }
    } else {
    // Parts are pulled into shared memory a window at a time ([win][NT8][2]
    // (m, l), then [win][q][NT8][DKm] shares), as many as the dead ring holds.
    const int win = max(1, min(ncl, (int)((p.epi_floats - 64) / (2 * NT8 + slab))));
    float *ml_s = ep;
    float *buf = ml_s + 2 * win * NT8;
    // TPI threads (a power of two, adjacent lanes) per (row, 4 columns) item
    // of the slice, up to kMaxRounds items per thread.  Parts are taken
    // 8 * TPI at a time: each thread loads its eight (m, l) and accumulator
    // rows at once, the chunk's largest m is shared by shuffles, and the
    // running sums are rescaled when it grows (online softmax over the
    // parts); the TPI threads' sums are added by shuffles at the end.  DKm
    // and DK / 4 are powers of two.
    const int lg_dkm = __ffs(DKm) - 1, lg_i = __ffs(DK / 4) - 1;
    const int n_items = nrows << lg_i;
    int lgT = 0;
    while (lgT < 5 && (2 << lgT) * n_items <= (int)blockDim.x) ++lgT;
    const int TPI = 1 << lgT;  // threads per item
    constexpr int kChunk = 8, kMaxRounds = 4;
    const int slab4 = slab / 4;
    const int64_t part4 = part_floats / 4;
    const float4 *ml_g = reinterpret_cast<const float4 *>(p.part_ml + gbase * NT8 * 2);
    const float4 *acc_g =
        reinterpret_cast<const float4 *>(p.part_acc + gbase * part_floats) + (int64_t)mi * slab4;
    const int nwarps = blockDim.x >> 5;
    // items beyond kMaxRounds per thread (a large slice) go in further
    // batches, each over all the windows again
#pragma unroll 1
    for (int ib = 0; ib < n_items * TPI; ib += kMaxRounds * blockDim.x) {
    const int rounds = min(kMaxRounds, (n_items * TPI - ib + blockDim.x - 1) / blockDim.x);
    float Ms[kMaxRounds], Ls[kMaxRounds];
    float4 As[kMaxRounds];
#pragma unroll
    for (int ri = 0; ri < kMaxRounds; ++ri) {
      Ms[ri] = -INFINITY;
      Ls[ri] = 0.f;
      As[ri] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 1
    for (int w0 = 0; w0 < ncl; w0 += win) {
      const int nw = min(win, ncl - w0);
      if (w0 > 0 || ib > 0) __syncthreads();  // the previous window is consumed
      // the window's (m, l) and shares: 16-byte asynchronous copies from
      // every thread, all in flight at once (one L2 round trip)
#pragma unroll 1
      for (int i = tid; i < nw * NT8 / 2; i += blockDim.x)
        cp_async16(ml_s + 4 * i, ml_g + (int64_t)w0 * NT8 / 2 + i);
#pragma unroll 1
      for (int c = warp; c < nw; c += nwarps) {
#pragma unroll 1
        for (int j = lane; j < slab4; j += 32)
          cp_async16(buf + ((int64_t)c * slab4 + j) * 4, acc_g + (int64_t)(w0 + c) * part4 + j);
      }
      cp_async_wait_all();
      __syncthreads();
#pragma unroll
      for (int ri = 0; ri < kMaxRounds; ++ri) {
        if (ri >= rounds) break;
        const int gi = ib + ri * blockDim.x + tid;
        const int item = gi >> lgT, sub = gi & (TPI - 1);
        const bool active = item < n_items;
        const int r = active ? item >> lg_i : 0, dd = active ? (item & ((DK >> 2) - 1)) * 4 : 0;
        const float2 *mlr = reinterpret_cast<const float2 *>(ml_s) + r;
        const float *src = buf + ((int64_t)(dd >> lg_dkm) * NT8 + r) * DKm + (dd & (DKm - 1));
#pragma unroll 1
        for (int c0 = 0; c0 < nw; c0 += kChunk * TPI) {
          float2 mv[kChunk];
          float4 bv[kChunk];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            const int c = c0 + sub + u * TPI;
            if (active && c < nw) {
              mv[u] = mlr[c * NT8];
              bv[u] = *reinterpret_cast<const float4 *>(src + (int64_t)c * slab);
            } else {
              mv[u] = make_float2(-INFINITY, 0.f);
              bv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          float cm = Ms[ri];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) cm = fmaxf(cm, mv[u].x);
#pragma unroll 1
          for (int o = 1; o < TPI; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
          const float mu = cm == -INFINITY ? 0.f : cm;
          const float sc = exp2_or_zero(Ms[ri], mu);
          float lr = Ls[ri] * sc;
          float4 a = As[ri];
          a.x *= sc;
          a.y *= sc;
          a.z *= sc;
          a.w *= sc;
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            const float w = exp2_or_zero(mv[u].x, mu);
            lr += w * mv[u].y;
            a.x += w * bv[u].x;
            a.y += w * bv[u].y;
            a.z += w * bv[u].z;
            a.w += w * bv[u].w;
          }
          Ms[ri] = cm;
          Ls[ri] = lr;
          As[ri] = a;
        }
      }
    }
#pragma unroll
    for (int ri = 0; ri < kMaxRounds; ++ri) {
      if (ri >= rounds) break;
      const int gi = ib + ri * blockDim.x + tid;
      const int item = gi >> lgT, sub = gi & (TPI - 1);
      const bool active = item < n_items;
      float lr = Ls[ri];
      float4 a = As[ri];
#pragma unroll 1
      for (int o = 1; o < TPI; o <<= 1) {
        lr += __shfl_xor_sync(0xffffffffu, lr, o);
        a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
        a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
        a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
        a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
      }
      if (active && sub == 0) {
        const int r = item >> lg_i, dd = (item & ((DK >> 2) - 1)) * 4;
        const float inv = lr > 0.f ? sfu_rcp(lr) : 0.f;
        const float v[4] = {a.x * inv, a.y * inv, a.z * inv, a.w * inv};
        store4<BF16>(out_row(r) + mi * DK + dd, v);
      }
    }
    }
    }
    if (tid == 0 && fin_old == K - 1) {
      // the last merger past its wait resets both counters: every merger
      // has passed its wait by then and every arrival has been counted
      atomicExch(p.counters + 2 * group, 0);
      atomicExch(p.counters + 2 * group + 1, 0);
    }
    return;
  }

  if (rank == 0 && tid == 0) {
    const int old = atomic_add_acq_rel_gpu(p.counters + 2 * group, 1);
    const int last = old == ncl - 1;
    if (last) atomicExch(p.counters + 2 * group, 0);
    if (old < 0 || old >= ncl) atomicOr(p.status, 0x10u);  // did not start at zero
    flags[1] = last;
#pragma unroll 1
    for (int x = 1; x < CS; ++x)
      st_dsmem_u32(mapa(smem_u32((const void *)(flags + 1)), x), (uint32_t)last);
  }
  if (CS > 1)
    cluster_sync();
  else
    __syncthreads();
  if (!flags[1]) return;

  // ---- the last cluster merges every cluster partial (its own slice) ----
  // By row chunks that keep at most four float4 sums per thread, the parts'
  // rows are pulled into shared memory with bulk copies (a chunk of parts in
  // flight at once); the first chunk is requested before the parts' (m, l)
  // are read, so both round trips overlap.
  float *pm_s = ep;                // [ncl][NT8] max, then weights
  float *pl_s = pm_s + ncl * NT8;  // [ncl][NT8] sums
  float *lall = pl_s + ncl * NT8;  // [NT8]
  float *buf = lall + NT8;         // [chunk][RC][DS]
  const int nthr = blockDim.x;
  const int RC = max(1, min(nrows, (16 * nthr) / DS));  // rows per chunk: <= 4 float4 per thread
  const int PC = max(1, min(ncl, (int)((p.epi_floats - (2 * ncl + 1) * NT8 - 16) / (RC * DS))));
  const uint32_t mb = smem_u32(mbar_merge);
  auto request = [&](int rc0, int p0) {
    if (tid == 0) {
      const int nr = min(RC, nrows - rc0), np = min(PC, ncl - p0);
      fence_proxy_async();
      const uint32_t bytes = (uint32_t)(nr * DS * 4);
      mbar_arrive_expect_tx(mb, bytes * np);
#pragma unroll 1
      for (int c = 0; c < np; ++c)
        bulk_load(smem_u32(buf + (int64_t)c * RC * DS),
                  p.part_acc + ((gbase + p0 + c) * CS + rank) * slice_floats + (int64_t)rc0 * DS,
                  bytes, mb);
    }
  };
  if (nrows > 0) request(0, 0);
#pragma unroll 1
  for (int idx = tid; idx < ncl * NT8; idx += blockDim.x) {
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + gbase * NT8 * 2) + idx);
    pm_s[idx] = ml.x;
    pl_s[idx] = ml.y;
  }
  __syncthreads();
#pragma unroll 1
  for (int r = tid; r < nrows; r += blockDim.x) {
    float ms = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < ncl; ++c) ms = fmaxf(ms, pm_s[c * NT8 + r]);
    const float mu = ms == -INFINITY ? 0.f : ms;
    float lsum = 0.f;
#pragma unroll 1
    for (int c = 0; c < ncl; ++c) {
      const float w = exp2_or_zero(pm_s[c * NT8 + r], mu);
      pm_s[c * NT8 + r] = w;
      lsum += pl_s[c * NT8 + r] * w;
    }
    lall[r] = lsum;
  }
  uint32_t phase = 0;
  bool ok = true, first = true;
#pragma unroll 1
  for (int rc0 = 0; rc0 < nrows && ok; rc0 += RC) {
    const int nr = min(RC, nrows - rc0);
    const int nitems = nr * (DS / 4);
    float4 a[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int p0 = 0; p0 < ncl; p0 += PC) {
      const int np = min(PC, ncl - p0);
      __syncthreads();  // the weights are in place; the previous chunk is consumed
      if (!first) request(rc0, p0);
      first = false;
      // one verdict for the whole CTA, so no thread leaves a barrier alone
      if (!__syncthreads_and(mbar_wait_bounded(mb, phase))) {
        if (tid == 0) atomicOr(p.status, 0x1u);
        ok = false;
        break;
      }
      phase ^= 1;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int it = tid + k * nthr;
        if (it < nitems) {
          const int rl = it / (DS / 4), d4 = (it % (DS / 4)) * 4;
#pragma unroll 1
          for (int c = 0; c < np; ++c) {
            const float w = pm_s[(p0 + c) * NT8 + rc0 + rl];
            const float4 b = *reinterpret_cast<const float4 *>(buf + ((int64_t)c * RC + rl) * DS + d4);
            a[k].x += w * b.x;
            a[k].y += w * b.y;
            a[k].z += w * b.z;
            a[k].w += w * b.w;
          }
        }
      }
    }
    if (!ok) break;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int it = tid + k * nthr;
      if (it < nitems) {
        const int rl = it / (DS / 4), d4 = (it % (DS / 4)) * 4;
        const float lr = lall[rc0 + rl];
        const float inv = lr > 0.f ? sfu_rcp(lr) : 0.f;
        const float v[4] = {a[k].x * inv, a[k].y * inv, a[k].z * inv, a[k].w * inv};
        store4<BF16>(out_row(rc0 + rl) + (int)rank * DS + d4, v);
      }
    }
  }
}

template <int D, bool BF16, bool TC, bool DOT = false, bool RM = false, bool TP = false>
cudaError_t launch_mma_t(const CUtensorMap &tk, const CUtensorMap &tv, const Params &p,
                         const Launch &l, cudaStream_t stream) {
  auto kern = pd_decode_mma<D, BF16, TC, DOT, RM, TP>;
  // largest dynamic shared memory opted into so far, per device
  static int configured_smem[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (l.smem > configured_smem[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem);
    if (e != cudaSuccess) return e;
    configured_smem[dev] = l.smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = l.grid;
  cfg.blockDim = l.block;
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (l.cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = l.cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (l.cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace pd
