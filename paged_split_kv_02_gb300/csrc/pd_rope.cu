// Rotary position embedding of the new tokens' q and k, and the store of k
// and v into the paged cache, in one kernel that runs ahead of decode
// attention (the fused RoPE / KV-cache write ROCm/vllm PR #1330, "Summary",
// names; cache slots as in the vLLM ROCm Octave backend's
// do_kv_cache_update(layer, key, value, kv_cache, slot_mapping)).
//
// One CTA per token.  Its work items are 16-byte chunks: for every q and
// k head the rotated chunks (NeoX: chunk c of each half, dims 8c.. and
// rot/2 + 8c..; GPT-J: 4 interleaved pairs, dims 8c..8c+7), then the
// pass-through chunks past rot_dim, then every v chunk.  Rotated values
// are computed in fp32 from the fp16/bf16 inputs and the fp32 table and
// rounded once.  Memory-bound: every byte is read or written once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "paged_decode.h"
#include "pd_internal.h"
#include "pd_ptx.cuh"

namespace pd {
namespace {

template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float2 to2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const T2 *>(&w));
  }
  static __device__ __forceinline__ uint32_t from2(float a, float b) {
    T2 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <>
struct Elem<false> {
  using T2 = __half2;
  static __device__ __forceinline__ float2 to2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const T2 *>(&w));
  }
  static __device__ __forceinline__ uint32_t from2(float a, float b) {
    T2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &w, float (&x)[8]) {
  using E = Elem<BF16>;
  const float2 a = E::to2(w.x), b = E::to2(w.y), c = E::to2(w.z), d = E::to2(w.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
  uint4 w;
  w.x = Elem<BF16>::from2(y[0], y[1]);
  w.y = Elem<BF16>::from2(y[2], y[3]);
  w.z = Elem<BF16>::from2(y[4], y[5]);
  w.w = Elem<BF16>::from2(y[6], y[7]);
  return w;
}

template <bool BF16, bool NEOX, int kU>
__global__ void __launch_bounds__(128) pd_rope_cache(const __grid_constant__ RopeParams p) {
  const int t = blockIdx.x;
  // the inputs may be the previous kernel's outputs
  grid_dependency_wait();
  grid_dependents_launch();
  int pos = __ldg(p.positions + t);
  if (pos < 0 || pos >= p.max_pos) {
    if (threadIdx.x == 0) atomicOr(p.status, PD_DEV_BAD_POSITION);
    pos = min(max(pos, 0), p.max_pos - 1);
  }
  const int slot = __ldg(p.slots + t);
  const bool write_kv = slot >= 0 && (int64_t)slot < p.num_slots;
  if (slot >= 0 && !write_kv && threadIdx.x == 0) atomicOr(p.status, PD_DEV_BAD_SLOT);
  const int page = write_kv ? slot / p.P : 0, off = write_kv ? slot - page * p.P : 0;

  const float *cs = p.cos_sin + (int64_t)pos * p.cs_s0;
  const int half = p.rot >> 1;
  const int heads = p.Hq + p.Hkv;
  const int rot_items = NEOX ? p.rot / 16 : p.rot / 8;  // per head
  const int pass_items = (p.D - p.rot) / 8;             // per head
  const int n_rot = heads * rot_items, n_pass = heads * pass_items;
  const int n_v = p.Hkv * (p.D / 8);
  const int n = n_rot + n_pass + (write_kv ? n_v : 0);

  // address of dims [d, d + 8) of head hh (q heads first, then k heads):
  // source and destination (q_out, or the k cache when the slot is valid).
  // Sources are read with coherent loads: q_out may be q itself, and each
  // chunk is read and then written by the same thread.
  auto src_ptr = [&](int hh, int d) -> const uint4 * {
    const unsigned short *b = hh < p.Hq
        ? static_cast<const unsigned short *>(p.q) + (int64_t)t * p.q_s0 + (int64_t)hh * p.q_s1
        : static_cast<const unsigned short *>(p.k) + (int64_t)t * p.k_s0 +
              (int64_t)(hh - p.Hq) * p.k_s1;
    return reinterpret_cast<const uint4 *>(b + d);
  };
  auto dst_ptr = [&](int hh, int d) -> uint4 * {
    unsigned short *b = hh < p.Hq
        ? static_cast<unsigned short *>(p.q_out) + (int64_t)t * p.qo_s0 + (int64_t)hh * p.qo_s1
        : static_cast<unsigned short *>(p.k_cache) + (int64_t)page * p.kc_page +
              (int64_t)off * p.kc_tok + (int64_t)(hh - p.Hq) * p.kc_head;
    return reinterpret_cast<uint4 *>(b + d);
  };

  auto v_src = [&](int h, int c) -> const uint4 * {
    return reinterpret_cast<const uint4 *>(static_cast<const unsigned short *>(p.v) +
                                           (int64_t)t * p.v_s0 + (int64_t)h * p.v_s1 + 8 * c);
  };
  auto v_dst = [&](int h, int c) -> uint4 * {
    return reinterpret_cast<uint4 *>(static_cast<unsigned short *>(p.v_cache) +
                                     (int64_t)page * p.vc_page + (int64_t)off * p.vc_tok +
                                     (int64_t)h * p.vc_head + 8 * c);
  };
  // Up to kU items per thread per pass: every item's loads are issued before
  // any item is computed and stored, so a thread has several 16-byte loads
  // in flight.  A few tokens (a decode batch) leave most warp slots empty and
  // take kU = 4; many tokens fill the SMs with warps instead and take kU = 1
  // (more registers per thread would cost resident CTAs).  Items touch
  // disjoint chunks and each chunk is loaded and stored by the same thread,
  // so the early loads are safe when q_out is q.
#pragma unroll 1
  for (int i0 = threadIdx.x; i0 < n; i0 += kU * blockDim.x) {
    uint4 w1[kU], w2[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * blockDim.x;
      w1[u] = w2[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i >= n) continue;
      if (i < n_rot) {
        const int hh = i / rot_items, c = i - hh * rot_items;
        w1[u] = *src_ptr(hh, 8 * c);
        if (NEOX) w2[u] = *src_ptr(hh, half + 8 * c);
      } else if (i < n_rot + n_pass) {
        const int j = i - n_rot, hh = j / pass_items, c = j - hh * pass_items;
        w1[u] = *src_ptr(hh, p.rot + 8 * c);
      } else {
        const int j = i - n_rot - n_pass, h = j / (p.D / 8), c = j - h * (p.D / 8);
        w1[u] = *v_src(h, c);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i >= n) continue;
      if (i < n_rot) {
        const int hh = i / rot_items, c = i - hh * rot_items;
        const bool store = hh < p.Hq || write_kv;
        if (NEOX) {
          // dims [8c, 8c + 8) pair with [half + 8c, half + 8c + 8), angles 8c..
          float x1[8], x2[8], co[8], si[8], y1[8], y2[8];
          unpack8<BF16>(w1[u], x1);
          unpack8<BF16>(w2[u], x2);
          const float4 c0 = __ldg(reinterpret_cast<const float4 *>(cs + 8 * c));
          const float4 c1 = __ldg(reinterpret_cast<const float4 *>(cs + 8 * c + 4));
          const float4 s0 = __ldg(reinterpret_cast<const float4 *>(cs + half + 8 * c));
          const float4 s1 = __ldg(reinterpret_cast<const float4 *>(cs + half + 8 * c + 4));
          co[0] = c0.x; co[1] = c0.y; co[2] = c0.z; co[3] = c0.w;
          co[4] = c1.x; co[5] = c1.y; co[6] = c1.z; co[7] = c1.w;
          si[0] = s0.x; si[1] = s0.y; si[2] = s0.z; si[3] = s0.w;
          si[4] = s1.x; si[5] = s1.y; si[6] = s1.z; si[7] = s1.w;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            y1[e] = x1[e] * co[e] - x2[e] * si[e];
            y2[e] = x2[e] * co[e] + x1[e] * si[e];
          }
          if (store) {
            *dst_ptr(hh, 8 * c) = pack8<BF16>(y1);
            *dst_ptr(hh, half + 8 * c) = pack8<BF16>(y2);
          }
        } else {
          // dims [8c, 8c + 8): pairs (2j, 2j + 1) of angles 4c .. 4c + 3
          float x[8], y[8];
          unpack8<BF16>(w1[u], x);
          const float4 cc = __ldg(reinterpret_cast<const float4 *>(cs + 4 * c));
          const float4 ss = __ldg(reinterpret_cast<const float4 *>(cs + half + 4 * c));
          const float co[4] = {cc.x, cc.y, cc.z, cc.w}, si[4] = {ss.x, ss.y, ss.z, ss.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[2 * j] = x[2 * j] * co[j] - x[2 * j + 1] * si[j];
            y[2 * j + 1] = x[2 * j + 1] * co[j] + x[2 * j] * si[j];
          }
          if (store) *dst_ptr(hh, 8 * c) = pack8<BF16>(y);
        }
      } else if (i < n_rot + n_pass) {
        const int j = i - n_rot, hh = j / pass_items, c = j - hh * pass_items;
        if (hh < p.Hq || write_kv) *dst_ptr(hh, p.rot + 8 * c) = w1[u];
      } else {
        const int j = i - n_rot - n_pass, h = j / (p.D / 8), c = j - h * (p.D / 8);
        *v_dst(h, c) = w1[u];
      }
    }
  }
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// [T, H, D] fp16/bf16 token rows: 16-byte aligned rows, innermost stride 1
int check_token_rows(const pd_tensor *t, int64_t T, int H, int D) {
  if (!t || t->ndim != 3 || (!t->data && T != 0)) return PD_EINVAL;  // (empty: any pointer)
  if (t->shape[0] != T || t->shape[1] != H || t->shape[2] != D) return PD_EINVAL;
  if (t->dtype != PD_F16 && t->dtype != PD_BF16) return PD_EDTYPE;
  if (t->stride[2] != 1) return PD_EALIGN;
  if (t->stride[0] < 0 || t->stride[1] < 0) return PD_EINVAL;
  if (t->stride[0] % 8 != 0 || t->stride[1] % 8 != 0 || !aligned16(t->data)) return PD_EALIGN;
  return PD_OK;
}

int check_i32_vector(const pd_tensor *t, int64_t n) {
  if (!t || (!t->data && n != 0) || t->ndim != 1 || t->shape[0] != n || t->stride[0] != 1)
    return PD_EINVAL;
  if (t->dtype != PD_I32) return PD_EDTYPE;
  return PD_OK;
}

// (page, token, kv head) element strides of a pool in its layout
void pool_strides(const pd_tensor *t, int layout, int64_t *page, int64_t *tok, int64_t *head) {
  *page = t->stride[0];
  *tok = layout == PD_NHD ? t->stride[1] : t->stride[2];
  *head = layout == PD_NHD ? t->stride[2] : t->stride[1];
}

}  // namespace
}  // namespace pd

using namespace pd;

extern "C" PD_API int paged_rope_cache_write(
    const pd_tensor *q, const pd_tensor *k, const pd_tensor *v, const pd_tensor *positions,
    const pd_tensor *slot_mapping, const pd_tensor *cos_sin_cache, pd_tensor *q_out,
    pd_tensor *k_cache, pd_tensor *v_cache, int num_q_heads, int num_kv_heads, int head_size,
    int rot_dim, int page_size, int layout, int is_neox, void *stream) {
  if (!q || !k || !v || !positions || !slot_mapping || !cos_sin_cache || !q_out || !k_cache ||
      !v_cache)
    return PD_EINVAL;
  if (num_q_heads <= 0 || num_kv_heads <= 0) return PD_EINVAL;
  if (head_size != 64 && head_size != 128 && head_size != 256 && head_size != 512) return PD_EHEAD;
  if (page_size <= 0 || (layout != PD_NHD && layout != PD_HND)) return PD_EINVAL;
  if (rot_dim <= 0 || rot_dim > head_size || rot_dim % (is_neox ? 16 : 8) != 0) return PD_EINVAL;
  if (q->ndim != 3 || q->shape[0] < 0 || q->shape[0] > INT32_MAX) return PD_EINVAL;
  const int64_t T = q->shape[0];
  int rc;
  if ((rc = check_token_rows(q, T, num_q_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_token_rows(q_out, T, num_q_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_token_rows(k, T, num_kv_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_token_rows(v, T, num_kv_heads, head_size)) != PD_OK) return rc;
  if ((rc = check_i32_vector(positions, T)) != PD_OK) return rc;
  if ((rc = check_i32_vector(slot_mapping, T)) != PD_OK) return rc;
  if ((rc = check_cache_tensor(k_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK)
    return rc;
  if ((rc = check_cache_tensor(v_cache, layout, num_kv_heads, page_size, head_size)) != PD_OK)
    return rc;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return PD_EINVAL;
  const int dt = q->dtype;
  if (q_out->dtype != dt || k->dtype != dt || v->dtype != dt || k_cache->dtype != dt ||
      v_cache->dtype != dt)
    return PD_EDTYPE;
  const pd_tensor *cs = cos_sin_cache;
  if (!cs->data || cs->ndim != 2 || cs->shape[0] < 1 || cs->shape[0] > INT32_MAX ||
      cs->shape[1] < rot_dim || cs->stride[1] != 1 || cs->stride[0] < rot_dim)
    return PD_EINVAL;
  if (cs->dtype != PD_F32) return PD_EDTYPE;
  if (cs->stride[0] % 4 != 0 || !aligned16(cs->data)) return PD_EALIGN;
  if (T == 0) return PD_OK;

  unsigned int *status = nullptr;
  if ((rc = device_check(nullptr, &status)) != PD_OK) return rc;

  RopeParams p{};
  p.q = q->data;
  p.q_s0 = q->stride[0];
  p.q_s1 = q->stride[1];
  p.k = k->data;
  p.k_s0 = k->stride[0];
  p.k_s1 = k->stride[1];
  p.v = v->data;
  p.v_s0 = v->stride[0];
  p.v_s1 = v->stride[1];
  p.q_out = q_out->data;
  p.qo_s0 = q_out->stride[0];
  p.qo_s1 = q_out->stride[1];
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  pool_strides(k_cache, layout, &p.kc_page, &p.kc_tok, &p.kc_head);
  pool_strides(v_cache, layout, &p.vc_page, &p.vc_tok, &p.vc_head);
  p.positions = static_cast<const int32_t *>(positions->data);
  p.slots = static_cast<const int32_t *>(slot_mapping->data);
  p.cos_sin = static_cast<const float *>(cs->data);
  p.cs_s0 = cs->stride[0];
  p.max_pos = (int)cs->shape[0];
  p.T = (int)T;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.D = head_size;
  p.rot = rot_dim;
  p.P = page_size;
  p.num_slots = k_cache->shape[0] * (int64_t)page_size;
  p.status = status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)T);
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool bf16 = dt == PD_BF16;
  int num_sms = 0;
  if ((rc = device_check(&num_sms, nullptr)) != PD_OK) return rc;
  // (4 warps per token; a GB300 SM holds 64)
  const bool few = T * 4 < (int64_t)num_sms * 32;
  cudaError_t e;
  if (few) {
    if (bf16)
      e = is_neox ? cudaLaunchKernelEx(&cfg, pd_rope_cache<true, true, 4>, p)
                  : cudaLaunchKernelEx(&cfg, pd_rope_cache<true, false, 4>, p);
    else
      e = is_neox ? cudaLaunchKernelEx(&cfg, pd_rope_cache<false, true, 4>, p)
                  : cudaLaunchKernelEx(&cfg, pd_rope_cache<false, false, 4>, p);
  } else {
    if (bf16)
      e = is_neox ? cudaLaunchKernelEx(&cfg, pd_rope_cache<true, true, 1>, p)
                  : cudaLaunchKernelEx(&cfg, pd_rope_cache<true, false, 1>, p);
    else
      e = is_neox ? cudaLaunchKernelEx(&cfg, pd_rope_cache<false, true, 1>, p)
                  : cudaLaunchKernelEx(&cfg, pd_rope_cache<false, false, 1>, p);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PD_ECUDA;
  }
  return PD_OK;
}
