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

// Merge all partial rows of query head kv*g + hg of batch row u and write the
// normalised output row.  Whole warp; lane owns D/32 contiguous features.
// Partials are read through L2 (they were written by other SMs): first the
// row max over all entries, then the weighted sums taken in entry order, then
// one multiply by 1/n.
template <typename T, int D>
__device__ __forceinline__ void merge_row(const AttnParams& p, int u, int kv, int hg, int lane) {
  constexpr int DPL = D / 32;
  const int key = u * p.Hkv + kv;
  const int e0 = __ldcg(p.m_off + key), e1 = __ldcg(p.m_off + key + 1);
  float m = -INFINITY;
  for (int e = e0 + lane; e < e1; e += 32) {
    const int pr = __ldcg(p.m_ent + e) + hg;
    m = fmaxf(m, __ldcg(p.part_ml + 2 * static_cast<size_t>(pr)));
  }
  m = warp_max(m);
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  float n = 0.f;
  for (int base = e0; base < e1; base += 32) {
    const int cnt = min(32, e1 - base);
    int pr = 0;
    float2 mn = make_float2(-INFINITY, 0.f);
    if (lane < cnt) {
      pr = __ldcg(p.m_ent + base + lane) + hg;
      mn = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + pr);
    }
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const int prj = __shfl_sync(0xffffffffu, pr, j);
      const float mj = __shfl_sync(0xffffffffu, mn.x, j);
      const float nj = __shfl_sync(0xffffffffu, mn.y, j);
      if (mj == -INFINITY) continue;
      const float wj = ptx::ex2(mj - m);
      n = fmaf(wj, nj, n);
      const float* src = p.part_o + static_cast<size_t>(prj) * D + lane * DPL;
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
  T* out = static_cast<T*>(p.out) + (static_cast<size_t>(u) * p.Hq + kv * p.g + hg) * D + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) out[i] = from_float<T>(o[i] * inv);
}

}  // namespace pst
