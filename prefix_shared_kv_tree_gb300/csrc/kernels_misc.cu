// K/V scatter into the chunk pool (and gather back out), the merge kernel,
// and the dtype dispatch of the CUDA-core attention kernel.  The pool stores each (chunk, KV
// head) as a K block and a transposed V block in the core-matrix layout of
// pst_internal.h; the scatter builds that layout from user rows [n][Hkv][D]
// (ChunkAttention, Knowl 1: K and V slices of h x c x d per chunk), see tile_off.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "attn_simt.cuh"

namespace pst {

namespace {

// ---------------------------------------------------------------------------
// Scatter user rows [rows][Hkv][D] into pool tiles (K rows and V^T columns).
// grid = (ops, Hkv).
// ---------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(256) scatter_kernel(const ScatterParams p, int D, int C) {
  constexpr int VEC = 16 / ES;
  const ScatterOp op = p.ops[blockIdx.x];
  const int kv = blockIdx.y;
  const int DCH = D / VEC;
  const size_t half = static_cast<size_t>(C) * D * ES;
  uint8_t* tile = p.pool + (static_cast<size_t>(op.chunk) * p.Hkv + kv) * 2 * half;
  const int rend = op.zero_tail ? C : op.r1;
  const size_t src_row_bytes = static_cast<size_t>(p.Hkv) * D * ES;
  if (op.r1 == op.r0 + 1 && !op.zero_tail) {
    // One row into a chunk that already holds rows [0, r0): a decode append.
    // K: the row's 16-byte chunks; V^T: one element in each of the D feature
    // rows, stored on its own (the rest of each 16-byte chunk is left alone).
    const uint8_t* ks = p.k + static_cast<size_t>(op.src_row) * src_row_bytes + static_cast<size_t>(kv) * D * ES;
    const uint8_t* vs = p.v + static_cast<size_t>(op.src_row) * src_row_bytes + static_cast<size_t>(kv) * D * ES;
    for (int j = threadIdx.x; j < DCH; j += blockDim.x)
      *reinterpret_cast<uint4*>(tile + tile_off(op.r0, j, D * ES, C)) = *reinterpret_cast<const uint4*>(ks + j * 16);
    const int j = op.r0 / VEC, e = op.r0 % VEC;
    for (int dr = threadIdx.x; dr < D; dr += blockDim.x) {
      uint8_t* dst = tile + half + tile_off(dr, j, C * ES, D) + e * ES;
      if constexpr (ES == 2) {
        *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(vs + dr * ES);
      } else {
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(vs + dr * ES);
      }
    }
    if (kv == 0 && threadIdx.x == 0) p.chunk_len[op.chunk] = op.r1;
    return;
  }
  // K: whole 16-byte chunks of rows [r0, rend)
  for (int idx = threadIdx.x; idx < (rend - op.r0) * DCH; idx += blockDim.x) {
    const int r = op.r0 + idx / DCH, j = idx % DCH;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < op.r1) {
      val = *reinterpret_cast<const uint4*>(p.k + static_cast<size_t>(op.src_row + r - op.r0) * src_row_bytes +
                                            static_cast<size_t>(kv) * D * ES + j * 16);
    }
    *reinterpret_cast<uint4*>(tile + tile_off(r, j, D * ES, C)) = val;
  }
  // V^T: the 16-byte chunks holding keys [r0, rend), patched element by element
  const int jb = op.r0 / VEC, je = (rend + VEC - 1) / VEC, nj = je - jb;
  for (int idx = threadIdx.x; idx < D * nj; idx += blockDim.x) {
    const int dr = idx / nj, j = jb + idx % nj;
    uint4* dst = reinterpret_cast<uint4*>(tile + half + tile_off(dr, j, C * ES, D));
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
  const int DCH = D / VEC;
  const size_t half = static_cast<size_t>(C) * D * ES;
  const uint8_t* tile = p.pool + (static_cast<size_t>(op.chunk) * p.Hkv + kv) * 2 * half;
  const size_t row_bytes = static_cast<size_t>(p.Hkv) * D * ES;
  uint8_t* kd = const_cast<uint8_t*>(p.k);
  uint8_t* vd = const_cast<uint8_t*>(p.v);
  for (int idx = threadIdx.x; idx < (op.r1 - op.r0) * DCH; idx += blockDim.x) {
    const int r = op.r0 + idx / DCH, j = idx % DCH;
    *reinterpret_cast<uint4*>(kd + static_cast<size_t>(op.src_row + r - op.r0) * row_bytes +
                              static_cast<size_t>(kv) * D * ES + j * 16) =
        *reinterpret_cast<const uint4*>(tile + tile_off(r, j, D * ES, C));
  }
  for (int idx = threadIdx.x; idx < (op.r1 - op.r0) * D; idx += blockDim.x) {
    const int r = op.r0 + idx / D, dr = idx % D;
    const uint8_t* s = tile + half + tile_off(dr, r / VEC, C * ES, D) + (r % VEC) * ES;
    uint8_t* d = vd + static_cast<size_t>(op.src_row + r - op.r0) * row_bytes + (static_cast<size_t>(kv) * D + dr) * ES;
#pragma unroll
    for (int b = 0; b < ES; ++b) d[b] = s[b];
  }
}

// ---------------------------------------------------------------------------
// Merge (ChunkAttention, Knowl 3: attn_reduce over all partial rows of a
// query row, then O = o / n).  One warp per (batch row, KV head) pair; the
// partials come from the chunk-first and sequence-first kernels that precede
// it on the stream.  A pair with at most merge_cap entries stages them in the
// warp's part of shared memory, all copies in flight at once.  Launched as a
// programmatic dependent: it becomes resident while they run and waits for
// their completion before reading.
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) merge_kernel(const AttnParams p, int B) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int key = blockIdx.x * 4 + warp;  // (batch row, KV head) pair: u * Hkv + kv
  const bool live = key < B * p.Hkv;
  int e0 = 0, e1 = 0;
  if (live) {  // the merge table was uploaded before the attention kernels ran
    e0 = __ldg(p.m_off + key);
    e1 = __ldg(p.m_off + key + 1);
  }
  if (p.pdl) ptx::pdl_wait();
  // every attention kernel of the step has completed: clear the work-claim
  // counter for the next step
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.sched != nullptr) *p.sched = 0;
  if (live) {
    extern __shared__ float4 merge_smem[];
    if (e1 - e0 <= p.merge_cap)
      merge_task_staged<T, D, G>(p, key, e0, e1, lane, merge_smem + static_cast<size_t>(warp) * p.merge_cap * (G * D / 4));
    else
      merge_task<T, D, G>(p, key, e0, e1, lane);
  }
}

template <typename T, int D, int G>
cudaError_t launch_merge_g(cudaLaunchConfig_t cfg, const AttnParams& p, int B) {
  auto fn = merge_kernel<T, D, G>;
  cfg.dynamicSmemBytes = static_cast<size_t>(4) * p.merge_cap * G * D * sizeof(float);
  if (cfg.dynamicSmemBytes > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(cfg.dynamicSmemBytes));
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, fn, p, B);
}

template <typename T, int D>
cudaError_t launch_merge_d(const cudaLaunchConfig_t& cfg, int g, const AttnParams& p, int B) {
  switch (g) {
    case 1: return launch_merge_g<T, D, 1>(cfg, p, B);
    case 2: return launch_merge_g<T, D, 2>(cfg, p, B);
    case 4: return launch_merge_g<T, D, 4>(cfg, p, B);
    case 8: return launch_merge_g<T, D, 8>(cfg, p, B);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_merge_t(int D, const AttnParams& p, int B, cudaStream_t s) {
  const int keys = B * p.Hkv;
  if (keys == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((keys + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  if (D == 64) return launch_merge_d<T, 64>(cfg, p.g, p, B);
  if (D == 128) return launch_merge_d<T, 128>(cfg, p.g, p, B);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_merge(int dtype, int D, const AttnParams& p, int B, cudaStream_t s) {
  switch (dtype) {
    case kF16: return launch_merge_t<__half>(D, p, B, s);
    case kBF16: return launch_merge_t<__nv_bfloat16>(D, p, B, s);
    case kF32: return launch_merge_t<float>(D, p, B, s);
  }
  return cudaErrorInvalidValue;
}

bool simt_supported(int dtype, int D, int g) {
  return (dtype == kF16 || dtype == kBF16 || dtype == kF32) && (D == 64 || D == 128) &&
         (g == 1 || g == 2 || g == 4 || g == 8);
}

int attn_simt_max_warps(int dtype, int g) { return simt_max_warps(g, dtype_size(dtype)); }

size_t attn_simt_piece_bytes(int dtype, int D, int C) { return simt_stage_bytes(C, D, dtype_size(dtype)); }

size_t attn_simt_smem(int dtype, int D, int C, int g, int stages, int warps_per_cta) {
  return simt_warp_bytes(C, D, g, stages, dtype_size(dtype), dtype == kBF16) * warps_per_cta;
}

cudaError_t launch_attn_simt(int dtype, int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s) {
  const bool large = C >= 64;
  switch (dtype) {
    case kF16: return large ? launch_attn_simt_f16_large(D, C, g, p, grid, s) : launch_attn_simt_f16_small(D, C, g, p, grid, s);
    case kBF16:
      return large ? launch_attn_simt_bf16_large(D, C, g, p, grid, s) : launch_attn_simt_bf16_small(D, C, g, p, grid, s);
    case kF32: return large ? launch_attn_simt_f32_large(D, C, g, p, grid, s) : launch_attn_simt_f32_small(D, C, g, p, grid, s);
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
