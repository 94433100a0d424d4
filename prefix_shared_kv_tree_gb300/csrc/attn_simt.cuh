// Sequence-first partial attention on the CUDA cores (ChunkAttention, Knowl 2
// phase 2, with partial_attn / attn_reduce of Knowl 3).  Also runs the
// chunk-first phase when the tensor-core kernel does not apply (fp32, c = 32),
// and causal prefill blocks in that case.
//
// Warp-per-stream design.  Each warp owns a contiguous share of the grid's
// (chunk, KV head) tiles, split on the host into work items of one
// (group, KV head) each.  A tile is consumed as pieces -- each 128-byte column
// block of K (all C keys), then each 64-row group of V^T -- each a contiguous
// block of the pool's tile image; lane 0 of the warp keeps `stages` pieces in
// flight with bulk async copies (TMA engine) into the warp's shared-memory
// ring.  Scores: lane = key, 128-bit shared loads, fp32 FMAs split over 4
// accumulators; tile max by warp shuffles; row sums stay lane-local until the
// item ends.  Values: lane = output feature row of V^T, 2 accumulators per row.
// The item's (o, m, n) rows then go to the partial buffer; the merge kernel
// that follows combines the rows of every (batch row, KV head).
#pragma once

#include "attn_common.cuh"
#include "ptx.cuh"

namespace pst {

__host__ __device__ inline size_t simt_align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Pieces of a tile (see tile_off): each 128-byte column block of K (C rows),
// then each 64-row group of every column block of V^T.
__host__ __device__ inline size_t simt_stage_bytes(int C, int D, int es) {
  const size_t kpb = static_cast<size_t>(C) * 128;
  const size_t vpb = ((C * es) % 128 == 0) ? static_cast<size_t>(64) * 128 : static_cast<size_t>(64) * C * es;
  return kpb > vpb ? kpb : vpb;
}

// Shared memory of one warp: [stages x piece][q rows fp32][p fp32][barriers].
__host__ __device__ inline size_t simt_warp_bytes(int C, int D, int G, int S, int es) {
  size_t b = S * simt_stage_bytes(C, D, es);
  b += static_cast<size_t>(G) * D * 4;
  b += static_cast<size_t>(G) * C * 4;
  b = simt_align_up(b, 8) + S * 8;
  return simt_align_up(b, 128);
}

template <typename T, int D, int G, int C>
__global__ void __launch_bounds__(256, 1) attn_simt_kernel(const AttnParams p) {
  constexpr int ES = sizeof(T);
  constexpr int VEC = 16 / ES;
  constexpr int DCH = D / VEC;    // 16-byte chunks per K row
  constexpr int CCH = C / VEC;    // 16-byte chunks per V^T row
  constexpr int KPL = C / 32;     // keys per lane
  constexpr int KB = D * ES / 128;                 // K pieces: 128-byte column blocks, C rows each
  constexpr bool VSW = (C * ES) % 128 == 0;         // V^T rows in 128-byte swizzled blocks
  constexpr int VB = VSW ? C * ES / 128 : 1;        // V^T column blocks
  constexpr int VR = D / 64;                        // 64-row groups per V^T block
  constexpr int VP = VB * VR;                       // V^T pieces
  constexpr int NP = KB + VP;
  constexpr int DPL = D / 32;     // output features per lane
  constexpr int KCH = 128 / 16;   // 16-byte chunks per K piece row
  constexpr int VCH = VSW ? 8 : C * ES / 16;        // 16-byte chunks per V^T piece row
  constexpr uint32_t KPB = static_cast<uint32_t>(C) * 128u;
  constexpr uint32_t VPB = VSW ? 64u * 128u : 64u * C * ES;
  constexpr uint32_t HALF = static_cast<uint32_t>(C) * D * ES;
  constexpr size_t TILE = 2 * static_cast<size_t>(HALF);
  const int S = p.stages;
  const uint32_t SB = static_cast<uint32_t>(simt_stage_bytes(C, D, ES));

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  ptx::pdl_launch_dependents();  // the merge kernel may become resident; it waits for us
  const int gw = blockIdx.x * p.warps_per_cta + warp;
  const int it0 = gw < p.n_warps ? p.warp_items[gw] : 0;
  const int it1 = gw < p.n_warps ? p.warp_items[gw + 1] : 0;
  if (it0 >= it1) {
    if (p.pdl) ptx::pdl_wait();  // never complete before the kernel we overlap
    return;
  }

  uint8_t* wb = smem + static_cast<size_t>(warp) * simt_warp_bytes(C, D, G, S, ES);
  uint8_t* stages = wb;
  float* qbuf = reinterpret_cast<float*>(wb + static_cast<size_t>(S) * SB);
  float* pbuf = qbuf + G * D;
  uint64_t* full = reinterpret_cast<uint64_t*>(simt_align_up(reinterpret_cast<size_t>(pbuf + G * C), 8));

  if (lane == 0) {
    for (int s = 0; s < S; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  // Producer cursor (lane 0 only): next piece to stage.
  int pi = it0, pc = 0, pp = 0;
  uint32_t issued = 0;
  WorkItem pw = p.items[it0];
  auto issue_next = [&]() {
    if (pi >= it1) return;
    const int chunk = p.chunks[pw.chunk_off + pc];
    const uint8_t* tile = p.pool + (static_cast<size_t>(chunk) * p.Hkv + pw.kv) * TILE;
    const uint8_t* src;
    if (pp < KB) {
      src = tile + pp * KPB;
    } else {
      const int vb = (pp - KB) / VR, vr = (pp - KB) % VR;
      src = tile + HALF + (VSW ? (static_cast<size_t>(vb) * D * 128 + vr * 64 * 128) : static_cast<size_t>(vr) * VPB);
    }
    const uint32_t bytes = pp < KB ? KPB : VPB;
    const int s = issued % S;
    ptx::mbar_arrive_expect_tx(&full[s], bytes);
    ptx::bulk_g2s(stages + static_cast<size_t>(s) * SB, src, bytes, &full[s]);
    ++issued;
    if (++pp == NP) {
      pp = 0;
      if (++pc == pw.n_chunks) {
        pc = 0;
        if (++pi < it1) pw = p.items[pi];
      }
    }
  };
  if (lane == 0) {
    for (int s = 0; s < S; ++s) issue_next();
  }
  __syncwarp();

  uint32_t consumed = 0;
  bool aborted = false;
  const T* qptr = static_cast<const T*>(p.q);

  // The next item's query rows and chunk lengths (lane c: chunk c, first 32
  // chunks) are fetched into registers one item ahead.
  constexpr int NQ = (G * DCH + 31) / 32;
  uint4 qnext[NQ];
  int len_next = 0;
  auto fetch_q = [&](int it_idx) {
    const WorkItem wn = p.items[it_idx];
    len_next = lane < wn.n_chunks ? p.chunk_len[p.chunks[wn.chunk_off + lane]] : 0;
#pragma unroll
    for (int k = 0; k < NQ; ++k) {
      const int idx = lane + 32 * k;
      if (idx < G * DCH) {
        const int h = idx / DCH, j = idx % DCH;
        qnext[k] = *reinterpret_cast<const uint4*>(qptr + (static_cast<size_t>(wn.group0) * p.Hq + wn.kv * p.g + h) * D +
                                                  j * VEC);
      }
    }
  };
  fetch_q(it0);

  for (int it = it0; it < it1 && !aborted; ++it) {
    const WorkItem w = p.items[it];
    const int grp = w.group0;
    // Query rows of this group, pre-scaled into log2 units.
#pragma unroll
    for (int k = 0; k < NQ; ++k) {
      const int idx = lane + 32 * k;
      if (idx < G * DCH) {
        const int h = idx / DCH, j = idx % DCH;
        float f[VEC];
        unpack16<T>(qnext[k], f);
#pragma unroll
        for (int e = 0; e < VEC; ++e) qbuf[h * D + j * VEC + e] = f[e] * p.scale_log2;
      }
    }
    __syncwarp();
    int my_len = len_next;
    if (it + 1 < it1) fetch_q(it + 1);

    float m[G], nl[G], o[G][DPL][2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      nl[h] = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[h][i][0] = o[h][i][1] = 0.f;
    }

    for (int c = 0; c < w.n_chunks && !aborted; ++c) {
      if ((c & 31) == 0 && c > 0) {  // valid tokens of chunks c .. c+31 of this item, one per lane
        my_len = 0;
        if (c + lane < w.n_chunks) my_len = p.chunk_len[p.chunks[w.chunk_off + c + lane]];
      }
      int lim = __shfl_sync(0xffffffffu, my_len, c & 31);
      if (p.causal_p0 >= 0) lim = min(lim, p.causal_p0 + grp + 1 - c * C);

      // ---- scores over the K pieces (one 128-byte column block of all keys each)
      float acc[G][KPL][4];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int kk = 0; kk < KPL; ++kk) acc[h][kk][0] = acc[h][kk][1] = acc[h][kk][2] = acc[h][kk][3] = 0.f;
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        const int s = consumed % S;
        if (!ptx::mbar_wait(&full[s], (consumed / S) & 1, nullptr, p.err)) {
          aborted = true;
          break;
        }
        const uint8_t* kt = stages + static_cast<size_t>(s) * SB;
#pragma unroll 4
        for (int jj = 0; jj < KCH; ++jj) {
#pragma unroll
          for (int kk = 0; kk < KPL; ++kk) {
            const int r = lane + 32 * kk;
            float kf[VEC];
            unpack16<T>(*reinterpret_cast<const uint4*>(kt + r * 128 + ((jj ^ (r & 7)) << 4)), kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float4* qv = reinterpret_cast<const float4*>(qbuf + h * D + kb * (128 / ES) + jj * VEC);
#pragma unroll
              for (int e4 = 0; e4 < VEC / 4; ++e4) {
                const float4 qq = qv[e4];
                acc[h][kk][0] = fmaf(qq.x, kf[4 * e4 + 0], acc[h][kk][0]);
                acc[h][kk][1] = fmaf(qq.y, kf[4 * e4 + 1], acc[h][kk][1]);
                acc[h][kk][2] = fmaf(qq.z, kf[4 * e4 + 2], acc[h][kk][2]);
                acc[h][kk][3] = fmaf(qq.w, kf[4 * e4 + 3], acc[h][kk][3]);
              }
            }
          }
        }
        __syncwarp();
        ++consumed;
        if (lane == 0) issue_next();
      }
      if (aborted) break;
      float sc[G][KPL];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int kk = 0; kk < KPL; ++kk)
          sc[h][kk] = (acc[h][kk][0] + acc[h][kk][1]) + (acc[h][kk][2] + acc[h][kk][3]);

      // ---- online softmax over the chunk's C keys (Knowl 3, log2 units)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int kp = 0; kp < KPL; ++kp) {
          if (kp * 32 + lane >= lim) sc[h][kp] = -INFINITY;
          mx = fmaxf(mx, sc[h][kp]);
        }
        const float m_new = fmaxf(m[h], warp_max(mx));
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ptx::ex2(m[h] - m_use);
        float ps = 0.f;
#pragma unroll
        for (int kp = 0; kp < KPL; ++kp) {
          const float pr = ptx::ex2(sc[h][kp] - m_use);
          ps += pr;
          pbuf[h * C + kp * 32 + lane] = pr;
        }
        nl[h] = nl[h] * alpha + ps;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          o[h][i][0] *= alpha;
          o[h][i][1] *= alpha;
        }
        m[h] = m_new;
      }
      __syncwarp();

      // ---- o += p V over the V^T pieces (64 feature rows of one key block each)
#pragma unroll
      for (int vp = 0; vp < VP; ++vp) {
        const int vb = vp / VR, vr = vp % VR;
        const int s = consumed % S;
        if (!ptx::mbar_wait(&full[s], (consumed / S) & 1, nullptr, p.err)) {
          aborted = true;
          break;
        }
        const uint8_t* vt = stages + static_cast<size_t>(s) * SB;
#pragma unroll 2
        for (int j = 0; j < VCH; ++j) {
          const int key0 = (VSW ? vb * (128 / ES) : 0) + j * VEC;
          float pv[G][VEC];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float4* pp4 = reinterpret_cast<const float4*>(pbuf + h * C + key0);
#pragma unroll
            for (int e4 = 0; e4 < VEC / 4; ++e4) {
              const float4 t = pp4[e4];
              pv[h][4 * e4 + 0] = t.x;
              pv[h][4 * e4 + 1] = t.y;
              pv[h][4 * e4 + 2] = t.z;
              pv[h][4 * e4 + 3] = t.w;
            }
          }
#pragma unroll
          for (int r2 = 0; r2 < 2; ++r2) {
            const int r = lane + 32 * r2;
            float vf[VEC];
            const uint32_t off = VSW ? r * 128 + ((j ^ (r & 7)) << 4) : cm_off(r, j, VCH);
            unpack16<T>(*reinterpret_cast<const uint4*>(vt + off), vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
              for (int e = 0; e < VEC; ++e)
                o[h][2 * vr + r2][e & 1] = fmaf(pv[h][e], vf[e], o[h][2 * vr + r2][e & 1]);
            }
          }
        }
        __syncwarp();
        ++consumed;
        if (lane == 0) issue_next();
      }
    }
    if (aborted) break;

    // ---- item result
    if (p.final_mode) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float inv = 1.f / warp_sum(nl[h]);
        T* out = static_cast<T*>(p.out) + (static_cast<size_t>(grp) * p.Hq + w.kv * p.g + h) * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) out[lane + 32 * i] = from_float<T>((o[h][i][0] + o[h][i][1]) * inv);
      }
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float n = warp_sum(nl[h]);
        const size_t row = static_cast<size_t>(w.part_base) + h;
        float* po = p.part_o + row * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) po[lane + 32 * i] = o[h][i][0] + o[h][i][1];
        if (lane == 0) reinterpret_cast<float2*>(p.part_ml)[row] = make_float2(m[h], n);
      }
    }
    __syncwarp();
  }

  if (aborted && lane == 0) {
    // Let every copy still in flight land before the warp leaves.
    for (uint32_t k = consumed; k < issued; ++k) ptx::mbar_wait(&full[k % S], (k / S) & 1, nullptr, p.err);
  }
  if (p.pdl) ptx::pdl_wait();  // never complete before the kernel we overlap
}

template <typename T, int D, int G, int C>
cudaError_t launch_simt_t(const AttnParams& p, int grid, cudaStream_t s) {
  const size_t smem = simt_warp_bytes(C, D, G, p.stages, sizeof(T)) * p.warps_per_cta;
  auto fn = attn_simt_kernel<T, D, G, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(p.warps_per_cta * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename T, int D, int C>
cudaError_t launch_simt_g(int g, const AttnParams& p, int grid, cudaStream_t s) {
  switch (g) {
    case 1: return launch_simt_t<T, D, 1, C>(p, grid, s);
    case 2: return launch_simt_t<T, D, 2, C>(p, grid, s);
    case 4: return launch_simt_t<T, D, 4, C>(p, grid, s);
    case 8: return launch_simt_t<T, D, 8, C>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_simt_dc(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (D == 64 && C == 32) return launch_simt_g<T, 64, 32>(g, p, grid, s);
  if (D == 64 && C == 64) return launch_simt_g<T, 64, 64>(g, p, grid, s);
  if (D == 128 && C == 32) return launch_simt_g<T, 128, 32>(g, p, grid, s);
  if (D == 128 && C == 64) return launch_simt_g<T, 128, 64>(g, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pst
