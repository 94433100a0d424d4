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

// The low / high 16-bit value packed in w (as pack2_16 wrote them),
// converted exactly to fp32.
template <typename T>
__device__ __forceinline__ float lo16(uint32_t w) {
  if constexpr (std::is_same<T, __half>::value) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  } else {
    return __uint_as_float(w << 16);
  }
}
template <typename T>
__device__ __forceinline__ float hi16(uint32_t w) {
  if constexpr (std::is_same<T, __half>::value) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  } else {
    return __uint_as_float(w & 0xffff0000u);
  }
}
// Sum of both: the row sum of two rounded probabilities.
template <typename T>
__device__ __forceinline__ float sum2_16(uint32_t w) {
  return lo16<T>(w) + hi16<T>(w);
}

// Element `elem` of an output tensor whose elements are T, or fp32 when
// out_f32 is set (the value before the final rounding to T).
template <typename T>
__device__ __forceinline__ void store_out1(void* out, size_t elem, float x, int out_f32) {
  if (out_f32) static_cast<float*>(out)[elem] = x;
  else static_cast<T*>(out)[elem] = from_float<T>(x);
}

// Four consecutive output elements from elem (a multiple of 4).
template <typename T>
__device__ __forceinline__ void store_out4(void* out, size_t elem, float a, float b, float c, float d, int out_f32) {
  if (out_f32 || sizeof(T) == 4) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + elem) = make_float4(a, b, c, d);
  } else {
    *reinterpret_cast<uint2*>(static_cast<T*>(out) + elem) = make_uint2(pack2_16<T>(a, b), pack2_16<T>(c, d));
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

// Merge the partial rows of one (batch row u, KV head kv) pair, key =
// u * Hkv + kv, whose entries are [e0, e1): entry e holds the G partial rows
// e*G .. e*G + G-1 (query heads kv*G + hg), so an entry is one contiguous
// block of G*D floats and the (m, n) of all the pair's rows are the
// contiguous float2s [e0*G, e1*G).  Writes output rows key*G + hg.
// Whole warp.  Lane l takes float4 l + 32 i of every entry block (row
// (l + 32 i) / (D/4)); (m, n) pair x = j*G + hg sits in lane x mod 32.  Per
// query row: the max of the entries' m, each entry's weight 2^(m_j - max),
// n = sum of weight * n_j, o = sum of weight * o_j taken in entry order, then
// one multiply by 1/n (ChunkAttention, Knowl 3: attn_reduce, then O = o / n).
// Partials are read through L2: other SMs wrote them.
template <typename T, int D, int G>
__device__ __forceinline__ void merge_task(const AttnParams& p, int key, int e0, int e1, int lane) {
  constexpr int RF = D / 4;                   // float4 per row
  constexpr int F4 = G * RF;                  // float4 per entry block
  constexpr int NI = (F4 + 31) / 32;          // float4 per lane per entry
  constexpr int kFast = NI >= 16 ? 1 : 16 / NI;  // entries merged from registers after one round of loads
  constexpr int EPR = 32 / G;                 // entries per 32 (m, n) pairs
  const int cnt = e1 - e0;
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + static_cast<size_t>(e0) * F4 + lane;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + static_cast<size_t>(e0) * G;
  int hg_i[NI];  // query row of this lane's float4 i
#pragma unroll
  for (int i = 0; i < NI; ++i) hg_i[i] = min((lane + 32 * i) / RF, G - 1);
  float4 acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  float mx, nn;  // lanes with lane % G == hg end up holding row hg's max and n
  if (cnt <= kFast && cnt <= EPR) {
    // Every load first -- the pairs' (m, n) (lane = pair) and this lane's
    // float4s of every entry block -- then the arithmetic.
    float4 ov[kFast][NI];
#pragma unroll
    for (int j = 0; j < kFast; ++j)
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (j < cnt && lane + 32 * i < F4) ov[j][i] = __ldcg(po + j * F4 + 32 * i);
    const float2 mn = lane < cnt * G ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
    mx = mn.x;
#pragma unroll
    for (int s = G; s < 32; s <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    const float w = mn.x == -INFINITY ? 0.f : ptx::ex2(mn.x - mx);  // an entry with no valid key adds nothing
    nn = w * mn.y;
#pragma unroll
    for (int s = G; s < 32; s <<= 1) nn += __shfl_xor_sync(0xffffffffu, nn, s);
#pragma unroll
    for (int j = 0; j < kFast; ++j) {
      if (j < cnt) {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const float wj = __shfl_sync(0xffffffffu, w, j * G + hg_i[i]);
          acc[i].x = fmaf(wj, ov[j][i].x, acc[i].x);
          acc[i].y = fmaf(wj, ov[j][i].y, acc[i].y);
          acc[i].z = fmaf(wj, ov[j][i].z, acc[i].z);
          acc[i].w = fmaf(wj, ov[j][i].w, acc[i].w);
        }
      }
    }
  } else {
    // Rounds of 32 pairs (EPR entries): the max over every round first, then
    // per round the weights, n, and the weighted entry blocks.
    const int rounds = (cnt + EPR - 1) / EPR;
    mx = -INFINITY;
    for (int r = 0; r < rounds; ++r) {
      const int x = r * 32 + lane;
      if (x < cnt * G) mx = fmaxf(mx, __ldcg(ml + x).x);
    }
#pragma unroll
    for (int s = G; s < 32; s <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    nn = 0.f;
    for (int r = 0; r < rounds; ++r) {
      const int x = r * 32 + lane;
      const float2 mn = x < cnt * G ? __ldcg(ml + x) : make_float2(-INFINITY, 0.f);
      const float w = mn.x == -INFINITY ? 0.f : ptx::ex2(mn.x - mx);
      nn = fmaf(w, mn.y, nn);
      const int c = min(EPR, cnt - r * EPR);
#pragma unroll 4
      for (int j = 0; j < c; ++j) {
        const float4* src = po + static_cast<size_t>(r * EPR + j) * F4;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const float wj = __shfl_sync(0xffffffffu, w, j * G + hg_i[i]);
          if (lane + 32 * i < F4) {
            const float4 t = __ldcg(src + 32 * i);
            acc[i].x = fmaf(wj, t.x, acc[i].x);
            acc[i].y = fmaf(wj, t.y, acc[i].y);
            acc[i].z = fmaf(wj, t.z, acc[i].z);
            acc[i].w = fmaf(wj, t.w, acc[i].w);
          }
        }
      }
    }
#pragma unroll
    for (int s = G; s < 32; s <<= 1) nn += __shfl_xor_sync(0xffffffffu, nn, s);
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const float inv = 1.f / __shfl_sync(0xffffffffu, nn, hg_i[i]);
    const int f = lane + 32 * i;
    if (f < F4)
      store_out4<T>(p.out, (static_cast<size_t>(key) * G + f / RF) * D + (f % RF) * 4, acc[i].x * inv, acc[i].y * inv,
                    acc[i].z * inv, acc[i].w * inv, p.out_f32);
  }
}

// merge_task with every entry block of the pair staged in shared memory by
// 16-byte asynchronous copies through L2 (all of them in flight at once, no
// registers held), then the same arithmetic in the same order.  buf holds
// cnt * G * D floats; cnt * G <= 32 (one round of (m, n) pairs).
template <typename T, int D, int G>
__device__ __forceinline__ void merge_task_staged(const AttnParams& p, int key, int e0, int e1, int lane,
                                                  float4* buf) {
  constexpr int RF = D / 4;
  constexpr int F4 = G * RF;
  constexpr int NI = (F4 + 31) / 32;
  const int cnt = e1 - e0;
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + static_cast<size_t>(e0) * F4;
  const uint32_t sb = ptx::smem_u32(buf);
  for (int x = lane; x < cnt * F4; x += 32)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sb + x * 16), "l"(po + x) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + static_cast<size_t>(e0) * G;
  const float2 mn = lane < cnt * G ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
  int hg_i[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) hg_i[i] = min((lane + 32 * i) / RF, G - 1);
  float mx = mn.x;
#pragma unroll
  for (int s = G; s < 32; s <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
  const float w = mn.x == -INFINITY ? 0.f : ptx::ex2(mn.x - mx);  // an entry with no valid key adds nothing
  float nn = w * mn.y;
#pragma unroll
  for (int s = G; s < 32; s <<= 1) nn += __shfl_xor_sync(0xffffffffu, nn, s);
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();
  float4 acc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < cnt; ++j) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const float wj = __shfl_sync(0xffffffffu, w, j * G + hg_i[i]);
      if (lane + 32 * i < F4) {
        const float4 t = buf[j * F4 + lane + 32 * i];
        acc[i].x = fmaf(wj, t.x, acc[i].x);
        acc[i].y = fmaf(wj, t.y, acc[i].y);
        acc[i].z = fmaf(wj, t.z, acc[i].z);
        acc[i].w = fmaf(wj, t.w, acc[i].w);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const float inv = 1.f / __shfl_sync(0xffffffffu, nn, hg_i[i]);
    const int f = lane + 32 * i;
    if (f < F4)
      store_out4<T>(p.out, (static_cast<size_t>(key) * G + f / RF) * D + (f % RF) * 4, acc[i].x * inv, acc[i].y * inv,
                    acc[i].z * inv, acc[i].w * inv, p.out_f32);
  }
}

}  // namespace pst
