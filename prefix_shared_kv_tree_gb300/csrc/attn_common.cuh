// Device helpers shared by the attention kernels: element conversion, warp
// reductions, and the online-softmax merge of a row's partial results
// (ChunkAttention, Knowl 3: attn_reduce, then O = o / n).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "pst_internal.h"
#include "ptx.cuh"

namespace pst {

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& raw, float* f) {
  if constexpr (sizeof(T) == 4) {
    f[0] = __uint_as_float(raw.x);
    f[1] = __uint_as_float(raw.y);
    f[2] = __uint_as_float(raw.z);
    f[3] = __uint_as_float(raw.w);
  } else if constexpr (std::is_same<T, __half>::value) {
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Two fp32 values rounded to nearest into one 32-bit word of 16-bit T
// (a first, in the low half).  T is __half or __nv_bfloat16.
template <typename T>
__device__ __forceinline__ uint32_t pack2_16(float a, float b) {
  if constexpr (std::is_same<T, __half>::value) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Merge the partial rows of one output row -- query head kv*g + hg of batch
// row u, task = (u * Hkv + kv) * g + hg -- whose pair owns entries [e0, e1)
// (entry e: partial row e*g + hg), and write the normalised output row.
// Whole warp; lane owns D/32 contiguous features.  Partials are read through
// L2 (other SMs wrote them): the (m, n) of every entry at once (lane = entry)
// for the row max, then the weighted sums taken in entry order, then one
// multiply by 1/n (ChunkAttention, Knowl 3: attn_reduce, then O = o / n).
template <typename T, int D>
__device__ __forceinline__ void merge_row(const AttnParams& p, int task, int e0, int e1, int lane) {
  constexpr int DPL = D / 32;
  constexpr int kFast = 16;  // entries merged from registers after one round of loads
  const int g = p.g, hg = task % g;
  const int cnt = e1 - e0;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  if (cnt <= kFast) {
    // Every load first -- each entry's (m, n) (lane = entry) and this lane's
    // features of every entry's o row -- then the same arithmetic, in the same
    // entry order, as the general path below.
    using VecT = typename std::conditional<DPL == 4, float4, float2>::type;
    VecT ov[kFast];
#pragma unroll
    for (int j = 0; j < kFast; ++j)
      if (j < cnt)
        ov[j] = __ldcg(reinterpret_cast<const VecT*>(p.part_o + (static_cast<size_t>(e0 + j) * g + hg) * D + lane * DPL));
    const float2 mn = lane < cnt ? __ldcg(ml + static_cast<size_t>(e0 + lane) * g + hg) : make_float2(-INFINITY, 0.f);
    const float m = warp_max(mn.x);
    float o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.f;
    float n = 0.f;
#pragma unroll
    for (int j = 0; j < kFast; ++j) {
      if (j < cnt) {
        const float mj = __shfl_sync(0xffffffffu, mn.x, j);
        const float nj = __shfl_sync(0xffffffffu, mn.y, j);
        const float wj = mj == -INFINITY ? 0.f : ptx::ex2(mj - m);
        n = fmaf(wj, nj, n);
        if constexpr (DPL == 4) {
          o[0] = fmaf(wj, ov[j].x, o[0]);
          o[1] = fmaf(wj, ov[j].y, o[1]);
          o[2] = fmaf(wj, ov[j].z, o[2]);
          o[3] = fmaf(wj, ov[j].w, o[3]);
        } else {
          o[0] = fmaf(wj, ov[j].x, o[0]);
          o[1] = fmaf(wj, ov[j].y, o[1]);
        }
      }
    }
    const float inv = 1.f / n;
    T* out = static_cast<T*>(p.out) + static_cast<size_t>(task) * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) out[i] = from_float<T>(o[i] * inv);
    return;
  }
  float2 first = make_float2(-INFINITY, 0.f);  // entry `lane` of the first 32
  float m = -INFINITY;
  for (int e = lane; e < cnt; e += 32) {
    const float2 t = __ldcg(ml + static_cast<size_t>(e0 + e) * g + hg);
    if (e < 32) first = t;
    m = fmaxf(m, t.x);
  }
  m = warp_max(m);
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  float n = 0.f;
  for (int base = 0; base < cnt; base += 32) {
    float2 mn = first;
    if (base > 0) mn = lane < cnt - base ? __ldcg(ml + static_cast<size_t>(e0 + base + lane) * g + hg)
                                         : make_float2(-INFINITY, 0.f);
    const int c = min(32, cnt - base);
#pragma unroll 8
    for (int j = 0; j < c; ++j) {
      const float mj = __shfl_sync(0xffffffffu, mn.x, j);
      const float nj = __shfl_sync(0xffffffffu, mn.y, j);
      const float wj = mj == -INFINITY ? 0.f : ptx::ex2(mj - m);  // an entry with no valid key adds nothing
      n = fmaf(wj, nj, n);
      const float* src = p.part_o + (static_cast<size_t>(e0 + base + j) * g + hg) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
        o[0] = fmaf(wj, t.x, o[0]);
        o[1] = fmaf(wj, t.y, o[1]);
        o[2] = fmaf(wj, t.z, o[2]);
        o[3] = fmaf(wj, t.w, o[3]);
      } else {
        const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
        o[0] = fmaf(wj, t.x, o[0]);
        o[1] = fmaf(wj, t.y, o[1]);
      }
    }
  }
  const float inv = 1.f / n;
  T* out = static_cast<T*>(p.out) + static_cast<size_t>(task) * D + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) out[i] = from_float<T>(o[i] * inv);
}

}  // namespace pst
