// CUDA-core kernels: K/V scatter into the chunk pool (and gather back), the
// sequence-first partial attention (ChunkAttention, Knowl 2 phase 2, with the
// partial_attn / attn_reduce of Knowl 3), and the online-softmax merge with the
// final divide.
//
// The attention kernel is a warp-per-stream design: every warp walks its own
// contiguous share of the grid's (chunk, KV head) tiles, staging each K or V^T
// half-tile into shared memory with a bulk async copy (TMA engine) several
// half-tiles ahead of the math, so each SM keeps tens of kilobytes of HBM
// reads in flight.  Scores use 128-bit shared-memory reads and fp32 FMAs; row
// max uses warp shuffles; row sums stay lane-local until the end of an item.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "ptx.cuh"
#include "pst_internal.h"

namespace pst {

namespace {

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

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared memory of one warp: [stages x half-tile][q rows fp32][p fp32][barriers].
__host__ __device__ inline size_t simt_warp_bytes(int C, int D, int G, int S, int es) {
  const size_t half = static_cast<size_t>(C) * D * es;
  size_t b = S * half;
  b += static_cast<size_t>(G) * D * 4;
  b += static_cast<size_t>(G) * C * 4;
  b = align_up(b, 8) + S * 8;
  return align_up(b, 128);
}

// ---------------------------------------------------------------------------
// Sequence-first partial attention.
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) attn_simt_kernel(const AttnParams p) {
  constexpr int ES = sizeof(T);
  constexpr int VEC = 16 / ES;
  constexpr int DCH = D / VEC;  // 16-byte chunks per K row
  constexpr int DPL = D / 32;   // V^T rows (output features) per lane
  const int C = p.chunk_size;
  const int CCH = C / VEC;      // 16-byte chunks per V^T row
  const int KPL = C / 32;       // keys per lane (1 or 2)
  const uint32_t half_bytes = static_cast<uint32_t>(C) * D * ES;
  const size_t tile_bytes = 2 * static_cast<size_t>(half_bytes);
  const int S = p.stages;

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * p.warps_per_cta + warp;
  if (gw >= p.n_warps) return;
  const int it0 = p.warp_items[gw];
  const int it1 = p.warp_items[gw + 1];
  if (it0 >= it1) return;

  uint8_t* wb = smem + static_cast<size_t>(warp) * simt_warp_bytes(C, D, G, S, ES);
  uint8_t* stages = wb;
  float* qbuf = reinterpret_cast<float*>(wb + static_cast<size_t>(S) * half_bytes);
  float* pbuf = qbuf + G * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(align_up(reinterpret_cast<size_t>(pbuf + G * C), 8));

  if (lane == 0) {
    for (int s = 0; s < S; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  // Producer cursor (lane 0 only): next half-tile to stage.
  int pi = it0, pc = 0, ppart = 0;
  uint32_t issued = 0;
  WorkItem pw = p.items[it0];
  auto issue_next = [&]() {
    if (pi >= it1) return;
    const int chunk = p.chunks[pw.chunk_off + pc];
    const uint8_t* src = p.pool + (static_cast<size_t>(chunk) * p.Hkv + pw.kv) * tile_bytes +
                         static_cast<size_t>(ppart) * half_bytes;
    const int s = issued % S;
    ptx::mbar_arrive_expect_tx(&full[s], half_bytes);
    ptx::bulk_g2s(stages + static_cast<size_t>(s) * half_bytes, src, half_bytes, &full[s]);
    ++issued;
    ppart ^= 1;
    if (ppart == 0 && ++pc == pw.n_chunks) {
      pc = 0;
      if (++pi < it1) pw = p.items[pi];
    }
  };
  if (lane == 0) {
    for (int s = 0; s < S; ++s) issue_next();
  }
  __syncwarp();

  uint32_t consumed = 0;
  bool aborted = false;
  const T* qptr = static_cast<const T*>(p.q);

  for (int it = it0; it < it1 && !aborted; ++it) {
    const WorkItem w = p.items[it];
    const int grp = w.group0;
    // Query rows of this group, pre-scaled into log2 units.
    for (int idx = lane; idx < G * DCH; idx += 32) {
      const int h = idx / DCH, j = idx % DCH;
      const T* src = qptr + (static_cast<size_t>(grp) * p.Hq + w.kv * p.g + h) * D + j * VEC;
      const uint4 raw = *reinterpret_cast<const uint4*>(src);
      float f[VEC];
      unpack16<T>(raw, f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) qbuf[h * D + j * VEC + e] = f[e] * p.scale_log2;
    }
    __syncwarp();

    float m[G], nl[G], o[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      nl[h] = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[h][i] = 0.f;
    }

    for (int c = 0; c < w.n_chunks; ++c) {
      const int chunk = p.chunks[w.chunk_off + c];
      int lim = p.chunk_len[chunk];
      if (p.causal_p0 >= 0) lim = min(lim, p.causal_p0 + grp + 1 - c * C);

      // ---- K half-tile: scores
      int s = consumed % S;
      if (!ptx::mbar_wait(&full[s], (consumed / S) & 1, nullptr, p.err)) {
        aborted = true;
        break;
      }
      const uint8_t* kt = stages + static_cast<size_t>(s) * half_bytes;
      float sc[G][2];
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h][0] = sc[h][1] = 0.f;
#pragma unroll 4
      for (int j = 0; j < DCH; ++j) {
        float kf0[VEC], kf1[VEC];
        unpack16<T>(*reinterpret_cast<const uint4*>(kt + cm_off(lane, j, DCH)), kf0);
        if (KPL == 2) unpack16<T>(*reinterpret_cast<const uint4*>(kt + cm_off(lane + 32, j, DCH)), kf1);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4* qv = reinterpret_cast<const float4*>(qbuf + h * D + j * VEC);
#pragma unroll
          for (int e4 = 0; e4 < VEC / 4; ++e4) {
            const float4 qq = qv[e4];
            sc[h][0] = fmaf(qq.x, kf0[4 * e4 + 0], sc[h][0]);
            sc[h][0] = fmaf(qq.y, kf0[4 * e4 + 1], sc[h][0]);
            sc[h][0] = fmaf(qq.z, kf0[4 * e4 + 2], sc[h][0]);
            sc[h][0] = fmaf(qq.w, kf0[4 * e4 + 3], sc[h][0]);
            if (KPL == 2) {
              sc[h][1] = fmaf(qq.x, kf1[4 * e4 + 0], sc[h][1]);
              sc[h][1] = fmaf(qq.y, kf1[4 * e4 + 1], sc[h][1]);
              sc[h][1] = fmaf(qq.z, kf1[4 * e4 + 2], sc[h][1]);
              sc[h][1] = fmaf(qq.w, kf1[4 * e4 + 3], sc[h][1]);
            }
          }
        }
      }
      __syncwarp();
      ++consumed;
      if (lane == 0) issue_next();

      // ---- online softmax over this chunk (Knowl 3, in log2 units)
      const bool v0 = lane < lim;
      const bool v1 = (KPL == 2) && (lane + 32 < lim);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float s0 = v0 ? sc[h][0] : -INFINITY;
        const float s1 = v1 ? sc[h][1] : -INFINITY;
        const float mt = warp_max(fmaxf(s0, s1));
        const float m_new = fmaxf(m[h], mt);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m[h] - m_use);
        const float p0 = exp2f(s0 - m_use);
        const float p1 = exp2f(s1 - m_use);
        nl[h] = nl[h] * alpha + p0 + p1;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[h][i] *= alpha;
        m[h] = m_new;
        pbuf[h * C + lane] = p0;
        if (KPL == 2) pbuf[h * C + lane + 32] = p1;
      }
      __syncwarp();

      // ---- V^T half-tile: o += p V
      s = consumed % S;
      if (!ptx::mbar_wait(&full[s], (consumed / S) & 1, nullptr, p.err)) {
        aborted = true;
        break;
      }
      const uint8_t* vt = stages + static_cast<size_t>(s) * half_bytes;
      for (int j = 0; j < CCH; ++j) {
        float pv[G][VEC];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4* pp = reinterpret_cast<const float4*>(pbuf + h * C + j * VEC);
#pragma unroll
          for (int e4 = 0; e4 < VEC / 4; ++e4) {
            const float4 t = pp[e4];
            pv[h][4 * e4 + 0] = t.x;
            pv[h][4 * e4 + 1] = t.y;
            pv[h][4 * e4 + 2] = t.z;
            pv[h][4 * e4 + 3] = t.w;
          }
        }
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          float vf[VEC];
          unpack16<T>(*reinterpret_cast<const uint4*>(vt + cm_off(lane + 32 * i, j, CCH)), vf);
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[h][i] = fmaf(pv[h][e], vf[e], o[h][i]);
          }
        }
      }
      __syncwarp();
      ++consumed;
      if (lane == 0) issue_next();
    }
    if (aborted) break;

    // ---- item result
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float n = warp_sum(nl[h]);
      if (p.final_mode) {
        T* out = static_cast<T*>(p.out) + (static_cast<size_t>(grp) * p.Hq + w.kv * p.g + h) * D;
        const float inv = 1.f / n;
#pragma unroll
        for (int i = 0; i < DPL; ++i) out[lane + 32 * i] = from_float<T>(o[h][i] * inv);
      } else {
        const size_t row = static_cast<size_t>(w.part_base) + h;
        float* po = p.part_o + row * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) po[lane + 32 * i] = o[h][i];
        if (lane == 0) {
          p.part_ml[2 * row] = m[h];
          p.part_ml[2 * row + 1] = n;
        }
      }
    }
    __syncwarp();
  }

  if (aborted && lane == 0) {
    // Let every copy still in flight land before the warp leaves.
    for (uint32_t k = consumed; k < issued; ++k) ptx::mbar_wait(&full[k % S], (k / S) & 1, nullptr, p.err);
  }
}

// ---------------------------------------------------------------------------
// Merge (Knowl 3 attn_reduce over all partials of a row, then O = o / n).
// One warp per (batch row, query head); each lane owns D/32 contiguous features.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  constexpr int DPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= p.B * p.Hq) return;
  const int u = row / p.Hq, h = row % p.Hq;
  const int kv = h / p.g, hg = h % p.g;
  const int e0 = p.off[u * p.Hkv + kv], e1 = p.off[u * p.Hkv + kv + 1];
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  float m = -INFINITY, n = 0.f;
  for (int e = e0; e < e1; ++e) {
    const size_t pr = static_cast<size_t>(p.ent[e]) + hg;
    const float mc = p.part_ml[2 * pr];
    const float nc = p.part_ml[2 * pr + 1];
    if (mc == -INFINITY) continue;
    const float mx = fmaxf(m, mc);
    const float x = exp2f(mc - mx);
    const float y = (m == -INFINITY) ? 0.f : exp2f(m - mx);
    const float* src = p.part_o + pr * D + lane * DPL;
    float oc[DPL];
    if constexpr (DPL == 4) {
      const float4 t = *reinterpret_cast<const float4*>(src);
      oc[0] = t.x; oc[1] = t.y; oc[2] = t.z; oc[3] = t.w;
    } else {
#pragma unroll
      for (int i = 0; i < DPL; ++i) oc[i] = src[i];
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = x * oc[i] + y * o[i];
    n = x * nc + y * n;
    m = mx;
  }
  T* out = static_cast<T*>(p.out) + static_cast<size_t>(row) * D + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) out[i] = from_float<T>(o[i] / n);
}

// ---------------------------------------------------------------------------
// Scatter user rows [rows][Hkv][D] into pool tiles (K rows and V^T columns).
// grid = (ops, Hkv).
// ---------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(256) scatter_kernel(const ScatterParams p, int D, int C) {
  constexpr int VEC = 16 / ES;
  const ScatterOp op = p.ops[blockIdx.x];
  const int kv = blockIdx.y;
  const int DCH = D / VEC, CCH = C / VEC;
  const size_t half = static_cast<size_t>(C) * D * ES;
  uint8_t* tile = p.pool + (static_cast<size_t>(op.chunk) * p.Hkv + kv) * 2 * half;
  const int rend = op.zero_tail ? C : op.r1;
  const size_t src_row_bytes = static_cast<size_t>(p.Hkv) * D * ES;
  // K: whole 16-byte chunks of rows [r0, rend)
  for (int idx = threadIdx.x; idx < (rend - op.r0) * DCH; idx += blockDim.x) {
    const int r = op.r0 + idx / DCH, j = idx % DCH;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < op.r1) {
      val = *reinterpret_cast<const uint4*>(p.k + static_cast<size_t>(op.src_row + r - op.r0) * src_row_bytes +
                                            static_cast<size_t>(kv) * D * ES + j * 16);
    }
    *reinterpret_cast<uint4*>(tile + cm_off(r, j, DCH)) = val;
  }
  // V^T: the 16-byte chunks holding keys [r0, rend), patched element by element
  const int jb = op.r0 / VEC, je = (rend + VEC - 1) / VEC, nj = je - jb;
  for (int idx = threadIdx.x; idx < D * nj; idx += blockDim.x) {
    const int dr = idx / nj, j = jb + idx % nj;
    uint4* dst = reinterpret_cast<uint4*>(tile + half + cm_off(dr, j, CCH));
    union {
      uint4 v;
      uint8_t b[16];
    } cur;
    cur.v = *dst;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const int key = j * VEC + e;
      if (key >= op.r0 && key < op.r1) {
        const uint8_t* s = p.v + static_cast<size_t>(op.src_row + key - op.r0) * src_row_bytes +
                           (static_cast<size_t>(kv) * D + dr) * ES;
#pragma unroll
        for (int b = 0; b < ES; ++b) cur.b[e * ES + b] = s[b];
      } else if (key >= op.r1 && op.zero_tail) {
#pragma unroll
        for (int b = 0; b < ES; ++b) cur.b[e * ES + b] = 0;
      }
    }
    *dst = cur.v;
  }
  if (kv == 0 && threadIdx.x == 0) p.chunk_len[op.chunk] = op.r1;
}

// Gather pool rows [r0, r1) of each op back to user layout (p.k / p.v are
// the destinations).
template <int ES>
__global__ void __launch_bounds__(256) gather_kernel(const ScatterParams p, int D, int C) {
  constexpr int VEC = 16 / ES;
  const ScatterOp op = p.ops[blockIdx.x];
  const int kv = blockIdx.y;
  const int DCH = D / VEC, CCH = C / VEC;
  const size_t half = static_cast<size_t>(C) * D * ES;
  const uint8_t* tile = p.pool + (static_cast<size_t>(op.chunk) * p.Hkv + kv) * 2 * half;
  const size_t row_bytes = static_cast<size_t>(p.Hkv) * D * ES;
  uint8_t* kd = const_cast<uint8_t*>(p.k);
  uint8_t* vd = const_cast<uint8_t*>(p.v);
  for (int idx = threadIdx.x; idx < (op.r1 - op.r0) * DCH; idx += blockDim.x) {
    const int r = op.r0 + idx / DCH, j = idx % DCH;
    *reinterpret_cast<uint4*>(kd + static_cast<size_t>(op.src_row + r - op.r0) * row_bytes +
                              static_cast<size_t>(kv) * D * ES + j * 16) =
        *reinterpret_cast<const uint4*>(tile + cm_off(r, j, DCH));
  }
  for (int idx = threadIdx.x; idx < (op.r1 - op.r0) * D; idx += blockDim.x) {
    const int r = op.r0 + idx / D, dr = idx % D;
    const uint8_t* s = tile + half + cm_off(dr, r / VEC, CCH) + (r % VEC) * ES;
    uint8_t* d = vd + static_cast<size_t>(op.src_row + r - op.r0) * row_bytes + (static_cast<size_t>(kv) * D + dr) * ES;
#pragma unroll
    for (int b = 0; b < ES; ++b) d[b] = s[b];
  }
}

template <typename T, int D, int G>
cudaError_t launch_simt_t(const AttnParams& p, int grid, cudaStream_t s) {
  const size_t smem = simt_warp_bytes(p.chunk_size, D, G, p.stages, sizeof(T)) * p.warps_per_cta;
  auto fn = attn_simt_kernel<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  fn<<<grid, p.warps_per_cta * 32, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_simt_g(int g, const AttnParams& p, int grid, cudaStream_t s) {
  switch (g) {
    case 1: return launch_simt_t<T, D, 1>(p, grid, s);
    case 2: return launch_simt_t<T, D, 2>(p, grid, s);
    case 4: return launch_simt_t<T, D, 4>(p, grid, s);
    case 8: return launch_simt_t<T, D, 8>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_simt_d(int D, int g, const AttnParams& p, int grid, cudaStream_t s) {
  if (D == 64) return launch_simt_g<T, 64>(g, p, grid, s);
  if (D == 128) return launch_simt_g<T, 128>(g, p, grid, s);
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_merge_d(int D, const MergeParams& p, cudaStream_t s) {
  const int rows = p.B * p.Hq;
  const int grid = (rows + 3) / 4;
  if (grid == 0) return cudaSuccess;
  if (D == 64) merge_kernel<T, 64><<<grid, 128, 0, s>>>(p);
  else if (D == 128) merge_kernel<T, 128><<<grid, 128, 0, s>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

bool simt_supported(int dtype, int D, int g) {
  return (dtype == kF16 || dtype == kBF16 || dtype == kF32) && (D == 64 || D == 128) &&
         (g == 1 || g == 2 || g == 4 || g == 8);
}

size_t attn_simt_smem(int dtype, int D, int C, int g, int stages, int warps_per_cta) {
  return simt_warp_bytes(C, D, g, stages, dtype_size(dtype)) * warps_per_cta;
}

cudaError_t launch_attn_simt(int dtype, int D, int g, const AttnParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  switch (dtype) {
    case kF16: return launch_simt_d<__half>(D, g, p, grid, s);
    case kBF16: return launch_simt_d<__nv_bfloat16>(D, g, p, grid, s);
    case kF32: return launch_simt_d<float>(D, g, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge(int dtype, int D, const MergeParams& p, cudaStream_t s) {
  switch (dtype) {
    case kF16: return launch_merge_d<__half>(D, p, s);
    case kBF16: return launch_merge_d<__nv_bfloat16>(D, p, s);
    case kF32: return launch_merge_d<float>(D, p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_scatter(int dtype, int D, int C, const ScatterParams& p, cudaStream_t s) {
  if (p.n_ops <= 0) return cudaSuccess;
  dim3 grid(p.n_ops, p.Hkv);
  if (dtype_size(dtype) == 2) scatter_kernel<2><<<grid, 256, 0, s>>>(p, D, C);
  else scatter_kernel<4><<<grid, 256, 0, s>>>(p, D, C);
  return cudaGetLastError();
}

cudaError_t launch_gather(int dtype, int D, int C, const ScatterParams& p, cudaStream_t s) {
  if (p.n_ops <= 0) return cudaSuccess;
  dim3 grid(p.n_ops, p.Hkv);
  if (dtype_size(dtype) == 2) gather_kernel<2><<<grid, 256, 0, s>>>(p, D, C);
  else gather_kernel<4><<<grid, 256, 0, s>>>(p, D, C);
  return cudaGetLastError();
}

}  // namespace pst
