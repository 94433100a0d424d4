// Chunk-first partial attention on the 5th-generation tensor cores (tcgen05).
//
// ChunkAttention, Knowl 2 phase 1: the queries of every sequence that shares
// a chunk are stacked into one matrix and multiplied by the chunk's K/V, which
// turns per-sequence matrix-vector work into a small dense contraction
// (Knowl 9).  Knowl 3 gives partial_attn: W = Q K^T, m = rowmax W,
// E = exp(W - m), n = rowsum E, O = E V.  The same kernel, with a per-row
// causal key limit and a normalised output, runs a W-row chunked-prefill block
// (Chunked Prefill, sections 1-2).
//
// Persistent: each CTA walks its own list of work items (up to 128 stacked
// query rows of one KV head against a list of chunks of 16, 32, 64 or 128
// tokens, taken as tiles of 64 keys: four or two chunks, one chunk, or half
// of one); TMEM and the mbarriers are set up once and the pipelines run
// across item boundaries.
// Warp roles (512 threads):
//   warp 0      : producer.  Lane 0 moves each tile's 32 KB K + V^T image
//                 from the pool into a 5-stage shared-memory ring by bulk
//                 async copy (TMA engine): one copy for a 64-token chunk; for
//                 keys [64h, 64h + 64) of a 128-token chunk, rows 64h .. of
//                 each 128-byte column block of K and column block h of V^T;
//                 for 16- or 32-token chunks, per chunk of the tile its K
//                 rows into each K column block and its V^T core matrices.
//                 The pool already stores K blocks in the tensor cores'
//                 128-byte-swizzled K-major layout (the swizzle follows the
//                 row index mod 8, so a part of a block whose rows start at a
//                 multiple of 8 is itself a block of that layout), V^T blocks
//                 with 128-byte rows likewise and shorter ones as plain 8-row
//                 core matrices; Q is written in the swizzled layout.
//   warp 1      : allocates TMEM and issues S = Q K^T (M=128, N=64, K=D) into
//                 three TMEM buffers (two for bf16), as far ahead of the
//                 softmax as they allow, across item boundaries.
//   warp 2      : issues O += P V (M=128, N=D, K=64, A = P read from TMEM) into
//                 the item's O buffer (double-buffered by item).
//                 Both issuer warps run their loops whole; one elected lane
//                 issues each tcgen05 instruction and commit.  Two issuers,
//                 because one thread's stream of MMAs and commits for a chunk
//                 takes longer than the tensor cores need for it.
//   warp 3      : gathers the next item's query rows into the other half of a
//                 double-buffered Q tile while the current item computes.
//   warps 4..11 : two threads per query row, each with half of the row's
//                 keys and O columns (half-split TMEM access puts both in one
//                 warp, so they combine by shuffles): read S from TMEM, online
//                 softmax in log2 units against a reference max that moves
//                 only when a chunk's max passes it by more than 2^8 (then O
//                 and the row sum are rescaled in TMEM), write the rounded
//                 probabilities P into TMEM as the A operand of the PV product
//                 (for bf16 also the rounded remainders, a second PV
//                 product); at an item's end they leave the row max and sum in
//                 shared memory and go on with the next item.
//   warps 12..15: epilogue, one thread per query row: stream each item's O
//                 out of TMEM (double-buffered by item) once its last PV
//                 product has completed: the item's partial rows (the merge
//                 kernel combines them) or, for a prefill block, the
//                 normalised output rows.
// Every wait is bounded; on a timeout the CTA records an error, drains its
// copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <type_traits>

#include "attn_common.cuh"
#include "ptx.cuh"

namespace pst {

namespace {

constexpr int kC = 64;     // keys per tile
constexpr int kBM = 128;   // stacked query rows per item
constexpr int kNS = 5;     // K/V tile stages
constexpr int kSB = 3;     // S buffers in TMEM at most: S runs up to kSB - 1 chunks ahead of the PV product
constexpr int kSoftmaxWarps = 8;   // warps 4..11, two threads per query row; each arrives once per barrier phase
constexpr int kEpilogueWarps = 4;  // warps 12..15, one thread per query row

__host__ __device__ constexpr uint32_t tc_tile_bytes(int D) { return 2u * kC * D * 2u; }
__host__ __device__ constexpr uint32_t tc_q_bytes(int D) { return kBM * D * 2u; }
__host__ __device__ constexpr size_t tc_smem_bytes(int D) {
  return 2 * tc_q_bytes(D) + kNS * tc_tile_bytes(D) + 320 + 2 * kBM * 8;
}

template <typename T>
__device__ __forceinline__ uint32_t pack2_plain(float a, float b) {
  if constexpr (std::is_same<T, __half>::value) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <typename T, int D, int CP>
__global__ void __launch_bounds__(512, 1) attn_tc_kernel(const AttnParams p) {
  constexpr uint32_t HALF = kC * D * 2;
  constexpr uint32_t TILE = tc_tile_bytes(D);
  // A 64-key tile is one pool chunk (CP = 64), half of one (CP = 128: SUB = 2
  // tiles per chunk), or CPT consecutive chunks (CP = 16, 32).
  constexpr int SUB = CP >= kC ? CP / kC : 1;     // 64-key tiles per pool chunk
  constexpr int CPT = CP < kC ? kC / CP : 1;      // pool chunks per 64-key tile
  constexpr uint32_t PHALF = CP * D * 2;          // a pool chunk's K block (per KV head)
  constexpr uint32_t PTILE = 2 * PHALF;           // a pool chunk's K + V^T blocks
  static_assert(CP == 16 || CP == 32 || CP == 64 || CP == 128, "chunk size");
  constexpr uint32_t QB = tc_q_bytes(D);
  constexpr int DCH = D / 8;    // 16-byte chunks per row when the reduction runs over D
  constexpr int CCH = kC / 8;   // 16-byte chunks per row when the reduction runs over keys
  constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
  // bf16 probabilities go to the PV product as two bf16 terms, the rounded
  // value and the rounded remainder (16 significant bits instead of 8, so a
  // row dominated by a few keys keeps its accuracy); their room in TMEM comes
  // from one S buffer less
  constexpr bool PSPLIT = BF;
  constexpr int SB = PSPLIT ? 2 : kSB;               // S buffers in use
  constexpr uint32_t PW = PSPLIT ? 64 : 32;          // TMEM columns of one P buffer
  constexpr uint32_t S_COL = 0;  // S buffers: columns [kC b, kC b + kC), b < SB
  // O of an item, double-buffered by item: [O_COL, O_COL + D), [O_COL + D, O_COL + 2D)
  constexpr uint32_t O_COL = SB * kC;
  // P double buffer, the A operand of the PV product: a row's kC 16-bit
  // probabilities packed two per column, [P_COL + PW b, .. + 32) (and, split,
  // the remainders in the next 32 columns)
  constexpr uint32_t P_COL = O_COL + 2 * D;
  constexpr uint32_t TMEM_COLS = (P_COL + 2 * PW) <= 256 ? 256u : 512u;
  static_assert(P_COL + 2 * PW <= 512, "tensor memory columns");
  constexpr uint32_t ID_S = ptx::idesc_f16(kBM, kC, BF);
  constexpr uint32_t ID_O = ptx::idesc_f16(kBM, D, BF);

  // The swizzled tiles need 1024-byte alignment; the dynamic shared memory
  // of this kernel (which has no static shared memory) starts there.  A base
  // that is not aligned is reported and nothing is touched.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (ptx::smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadIndex);
    if (p.pdl) ptx::pdl_wait();
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* qs = smem;                 // [2] Q tiles
  uint8_t* kvs = qs + 2 * QB;         // [kNS] K + V^T tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(kvs + kNS * TILE);
  uint64_t* full = bars;             // [kNS] tile landed
  uint64_t* empty = bars + kNS;      // [kNS] tile no longer read by the tensor cores
  uint64_t* qfull = bars + 2 * kNS;  // [2] Q tile written (32 Q-loader lanes)
  uint64_t* qfree = qfull + 2;       // [2] Q tile no longer read by the tensor cores
  uint64_t* sfull = qfree + 2;       // [kSB] S ready in TMEM
  uint64_t* sfree = sfull + kSB;     // [kSB] S read by the softmax warps (8)
  uint64_t* pfull = sfree + kSB;     // [2] P written, O rescaled if needed (8)
  uint64_t* pfree = pfull + 2;       // [2] the PV product that read P buffer b has completed
  uint64_t* ofull = pfree + 2;       // [2] every PV product of an item has completed (O buffer by item)
  uint64_t* oempty = ofull + 2;      // [2] the item's O was read out (4 epilogue warps)
  uint64_t* mlfull = oempty + 2;     // [2] the item's row max and sum are in ml_buf (8 softmax warps)
  uint64_t* done = mlfull + 2;       // [2] all MMAs of the S / PV issuer completed
  float2* ml_buf = reinterpret_cast<float2*>(done + 2);  // [2][kBM] (m, n) of each row, by O buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ml_buf + 2 * kBM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* issued_slot = abort_flag + 1;
  volatile int* consumed_slot = abort_flag + 2;

  ptx::pdl_launch_dependents();  // the kernels that follow wait for our results themselves
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int i0 = p.warp_items[blockIdx.x];
  const int i1 = p.warp_items[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < SB; ++b) {
      ptx::mbar_init(&sfull[b], 1);
      ptx::mbar_init(&sfree[b], kSoftmaxWarps);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&qfull[b], 32);
      ptx::mbar_init(&qfree[b], 1);
      ptx::mbar_init(&pfull[b], kSoftmaxWarps);
      ptx::mbar_init(&pfree[b], 1);
      ptx::mbar_init(&ofull[b], 1);
      ptx::mbar_init(&oempty[b], kEpilogueWarps);
      ptx::mbar_init(&mlfull[b], kSoftmaxWarps);
    }
    ptx::mbar_init(&done[0], 1);
    ptx::mbar_init(&done[1], 1);
    *abort_flag = 0;
    *issued_slot = 0;
    *consumed_slot = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, TMEM_COLS);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const T* qbase = static_cast<const T*>(p.q);

  if (warp == 0) {
    // ------------------------------------------------------- tile producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();
      int t = 0;
      bool ok = true;
      for (int ii = i0; ii < i1 && ok; ++ii) {
        const WorkItem w = p.items[ii];
        const int nt = (w.n_chunks * SUB + CPT - 1) / CPT;
        for (int c = 0; c < nt; ++c, ++t) {
          const int s = t % kNS;
          if (t >= kNS && !ptx::mbar_wait(&empty[s], ((t / kNS) - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* dst = kvs + s * TILE;
          ptx::mbar_arrive_expect_tx(&full[s], TILE);
          if constexpr (CPT > 1) {
            // chunks c CPT .. c CPT + CPT - 1: chunk i's K rows become rows
            // [i CP, i CP + CP) of each 128-byte K column block (CP is a
            // multiple of 8, so the swizzle phase of every row is kept) and
            // its V^T core matrices block i of the V^T part.  Past the item's
            // last chunk the slot gets its first chunk again: finite values,
            // masked by the softmax.
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
              const int ch = c * CPT + i < w.n_chunks ? c * CPT + i : c * CPT;
              const int chunk = p.chunks[w.chunk_off + ch];
              const uint8_t* src = p.pool + (static_cast<size_t>(chunk) * p.Hkv + w.kv) * PTILE;
#pragma unroll
              for (int kb = 0; kb < D / 64; ++kb)
                ptx::bulk_g2s_hint(dst + kb * (kC * 128) + i * (CP * 128), src + kb * (CP * 128), CP * 128, &full[s], pol);
              ptx::bulk_g2s_hint(dst + HALF + i * PHALF, src + PHALF, PHALF, &full[s], pol);
            }
          } else if constexpr (SUB == 1) {
            const int chunk = p.chunks[w.chunk_off + c];
            const uint8_t* src = p.pool + (static_cast<size_t>(chunk) * p.Hkv + w.kv) * PTILE;
            ptx::bulk_g2s_hint(dst, src, TILE, &full[s], pol);
          } else {
            const int chunk = p.chunks[w.chunk_off + c / SUB];
            const uint8_t* src = p.pool + (static_cast<size_t>(chunk) * p.Hkv + w.kv) * PTILE;
            const int h = c % SUB;
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb)  // K column block kb: rows 64h .. 64h + 63
              ptx::bulk_g2s_hint(dst + kb * (kC * 128), src + kb * (CP * 128) + h * (kC * 128), kC * 128, &full[s], pol);
            ptx::bulk_g2s_hint(dst + HALF, src + PHALF + h * (D * 128), D * 128, &full[s], pol);  // V^T column block h
          }
          *issued_slot = t + 1;
        }
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------- Q loader
    // Gathers each item's 128 query rows (zero past n_rows) into one half of
    // the double-buffered Q tile, one item ahead of the tensor cores: 16-byte
    // asynchronous copies, all of an item's in flight at once.
    for (int ii = i0; ii < i1; ++ii) {
      const int it = ii - i0, qb = it & 1;
      bool ok = true;
      if (it >= 2) ok = ptx::mbar_wait(&qfree[qb], ((it - 2) >> 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) break;
      const WorkItem w = p.items[ii];
      const uint32_t dst = ptx::smem_u32(qs + qb * QB);
#pragma unroll
      for (int i = 0; i < kBM / 32; ++i) {
        const int r = lane + 32 * i;
        const bool valid = r < w.n_rows;
        const int rr = w.row0 + r;
        const T* src = valid ? qbase + (static_cast<size_t>(w.group0 + rr / p.g) * p.Hq + w.kv * p.g + rr % p.g) * D
                             : qbase;
#pragma unroll
        for (int j = 0; j < DCH; ++j) ptx::cp_async_16(dst + tile_off(r, j, D * 2, kBM), src + 8 * j, valid ? 16u : 0u);
      }
      ptx::cp_async_wait_all();
      ptx::fence_proxy_async_smem();  // the tensor cores read the tile through the async proxy
      ptx::mbar_arrive(&qfull[qb]);
    }
  } else if (warp == 1 || warp == 2) {
    // ---------------------------------------------------- MMA issuers (S, PV)
    // The whole warp runs its loop (operands stay warp-uniform); one elected
    // lane issues each tcgen05 instruction.
    {
      const uint32_t q_addr = ptx::smem_u32(qs);
      const uint32_t kv_addr = ptx::smem_u32(kvs);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, p.err));
      };
      auto issue_s = [&](int t, int qb) -> bool {
        const int s = t % kNS, b = t % SB;
        if (!wait_all(&full[s], (t / kNS) & 1)) return false;
        if (lane == 0) *consumed_slot = t + 1;
        if (t >= SB && !wait_all(&sfree[b], ((t - SB) / SB) & 1)) return false;
        ptx::tc_fence_after();
        // Descriptors of each K step = the tile's base descriptor + the step's
        // byte offset / 16 (the 14-bit start-address field never carries).
        const uint64_t a0 = ptx::smem_desc_sw128(q_addr + qb * QB, 1024);
        const uint64_t b0 = ptx::smem_desc_sw128(kv_addr + s * TILE, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K step kk covers features [16kk, 16kk+16): column block kk/4, 32-byte offset (kk%4)
          constexpr uint32_t kA = kBM * 128 / 16, kB = kC * 128 / 16;
          const uint64_t da = (kk >> 2) * kA + (kk & 3) * 2, db = (kk >> 2) * kB + (kk & 3) * 2;
          ptx::mma_f16_warp(tbase + S_COL + b * kC, a0 + da, b0 + db, ID_S, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_warp(&sfull[b]);
        return true;
      };
      // O += P V for chunk c of item it: accumulates in the item's TMEM buffer
      // across its chunks (the softmax threads rescale it when their
      // reference max moves); the first chunk overwrites.
      auto issue_pv = [&](int t, int it, int c, bool last) -> bool {
        const int s = t % kNS, b = t & 1, ob = it & 1;
        if (!wait_all(&pfull[b], (t >> 1) & 1)) return false;
        if (c == 0 && it >= 2 && !wait_all(&oempty[ob], ((it - 2) >> 1) & 1)) return false;
        ptx::tc_fence_after();
        // V^T operand of K step kk (keys [16kk, 16kk+16)): at CP >= 64 the
        // tile's 128-byte-swizzled block, 32 bytes further per step; at
        // CP < 64 the core matrices of chunk (16 kk) / CP, unswizzled
        // (16-byte rows, CP / 8 core matrices per 8-row group, two per step)
        auto vdesc = [&](int kk) -> uint64_t {
          if constexpr (CPT > 1) {
            const uint32_t at = kv_addr + s * TILE + HALF + (16 * kk / CP) * PHALF + ((16 * kk) % CP) / 16 * 256;
            return ptx::smem_desc(at, 128, 16 * CP);
          } else {
            return ptx::smem_desc_sw128(kv_addr + s * TILE + HALF, 1024) + kk * 2;
          }
        };
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)  // K step kk: keys [16kk, 16kk+16) = P columns [8kk, 8kk+8)
          ptx::mma_f16_tmem_a_warp(tbase + O_COL + ob * D, tbase + P_COL + b * PW + kk * 8, vdesc(kk), ID_O,
                                   (c > 0 || kk > 0) ? 1u : 0u);
        if constexpr (PSPLIT) {
#pragma unroll
          for (int kk = 0; kk < kC / 16; ++kk)  // the remainders: P columns 32 + [8kk, 8kk+8)
            ptx::mma_f16_tmem_a_warp(tbase + O_COL + ob * D, tbase + P_COL + b * PW + 32 + kk * 8, vdesc(kk), ID_O,
                                     1u);
        }
        ptx::mma_commit_warp(&pfree[b]);
        ptx::mma_commit_warp(&empty[s]);
        if (last) ptx::mma_commit_warp(&ofull[ob]);
        return true;
      };
      // S runs over this CTA's chunk sequence (across item boundaries) as far
      // ahead as the kSB S buffers allow, so the softmax threads find each S
      // ready when they finish the previous chunk.
      int s_ii = i0, s_c = 0, s_t = 0;
      auto tiles_of = [](const WorkItem& w) { return (w.n_chunks * SUB + CPT - 1) / CPT; };
      int s_nk = i0 < i1 ? tiles_of(p.items[i0]) : 0;
      auto issue_next_s = [&]() -> bool {
        const int it = s_ii - i0, qb = it & 1;
        if (s_c == 0) {  // the item's Q tile
          if (!wait_all(&qfull[qb], (it >> 1) & 1)) return false;
          ptx::tc_fence_after();
        }
        if (!issue_s(s_t, qb)) return false;
        if (s_c + 1 == s_nk) ptx::mma_commit_warp(&qfree[qb]);  // every S of this item is issued
        ++s_t;
        if (++s_c == s_nk) {
          s_c = 0;
          ++s_ii;
          s_nk = s_ii < i1 ? tiles_of(p.items[s_ii]) : 0;
        }
        return true;
      };
      bool ok = true;
      if (warp == 1) {
        while (ok && s_ii < i1) ok = issue_next_s();
      } else {
        int t = 0;
        for (int ii = i0; ii < i1 && ok; ++ii) {
          const int it = ii - i0;
          const int nk = tiles_of(p.items[ii]);
          for (int c = 0; c < nk && ok; ++c, ++t) ok = issue_pv(t, it, c, c + 1 == nk);
        }
      }
      // Every MMA of this issuer must have finished before TMEM is released.
      uint64_t* my_done = &done[warp == 1 ? 0 : 1];  // S issuer, PV issuer
      ptx::mma_commit_warp(my_done);
      ptx::mbar_wait(my_done, 0, nullptr, p.err);
    }
    __syncwarp();
  } else if (warp < 12) {
    // ---------------------------------------------------------------- softmax
    // Two threads per query row.  Warps 4..11 each take 16 rows: the TMEM
    // lane quadrant is fixed by warp % 4, warps 8..11 take its upper 16
    // lanes; with half-split TMEM access thread t holds row (t mod 16) of the
    // warp's 16 and half hf = t div 16 of the row's columns -- keys
    // [32 hf, 32 hf + 32) of each S tile, O columns [hf D/2, (hf + 1) D/2).
    // The two halves of a row meet by warp shuffles (xor 16).  The item's O
    // accumulates in TMEM; scores are exponentiated against a per-row
    // reference max that only moves when a chunk's max exceeds it by more
    // than kRescale (log2 units), so P stays below 2^kRescale and O (with the
    // row sum) is rescaled rarely.
    constexpr float kRescale = 8.f;
    constexpr int HK = kC / 2;  // keys of a tile per thread
    constexpr int HD = D / 2;   // O columns per thread
    const int quad = warp & 3, sub = (warp >> 3) & 1, hf = lane >> 4;
    const int r = quad * 32 + sub * 16 + (lane & 15);
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32 + sub * 16) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, p.err));
    };
    // Valid keys of tile c of item w: the tile's chunks are full but for the
    // item's last chunk (only a sequence's last chunk is partial), whose
    // valid tokens the scatter kernel keeps in chunk_len.
    auto tile_len = [&](const WorkItem& w, int c) -> int {
      if constexpr (CPT > 1) {
        const int first = c * CPT, cnt = min(CPT, w.n_chunks - first);
        return (cnt - 1) * CP + p.chunk_len[p.chunks[w.chunk_off + first + cnt - 1]];
      } else {
        return min(kC, max(0, p.chunk_len[p.chunks[w.chunk_off + c / SUB]] - (c % SUB) * kC));
      }
    };
    auto tiles_of = [](const WorkItem& w) { return (w.n_chunks * SUB + CPT - 1) / CPT; };
    // An item's descriptor and the valid keys of its first 32 tiles are
    // loaded while the previous item ends, so their latency is hidden.
    WorkItem wn{};
    int len_n = 0;
    auto prefetch = [&](int ii) {
      if (ii >= i1) return;
      wn = p.items[ii];
      len_n = lane < tiles_of(wn) ? tile_len(wn, lane) : 0;
    };
    prefetch(i0);
    const float sc = p.scale_log2;
    int t = 0;
    bool ok = true;
    for (int ii = i0; ii < i1 && ok; ++ii) {
      const int it = ii - i0, ob = it & 1;
      const WorkItem w = wn;
      const int nk = tiles_of(w);  // 64-key tiles
      const bool row_valid = r < w.n_rows;
      const int grp = row_valid ? w.group0 + (w.row0 + r) / p.g : 0;
      // causal: keys of this item up to position p0 + token (item key 0 is at w.key0)
      const int key_limit = (p.causal_p0 >= 0 && row_valid) ? p.causal_p0 + grp + 1 - w.key0 : INT_MAX;
      float m = -INFINITY, l = 0.f;  // reference max; this half's row sum relative to it
      int my_len = len_n;

      for (int c = 0; c < nk; ++c, ++t) {
        if ((c & 31) == 0 && c > 0)  // valid keys of tiles c .. c+31, one per lane
          my_len = c + lane < nk ? tile_len(w, c + lane) : 0;
        // valid keys of this thread's half of the tile
        const int lim = min(__shfl_sync(0xffffffffu, my_len, c & 31), key_limit - c * kC) - hf * HK;
        const int b = t & 1, sb = t % SB;
        // polled now, waited for below: the answer arrives during the exponentials
        const bool p_ready = t < 2 || ptx::mbar_test_wait(&pfree[b], ((t - 2) >> 1) & 1);
        if (!wait_all(&sfull[sb], (t / SB) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        uint32_t sv[32];
        ptx::tmem_ld32_half<HK>(tl + S_COL + sb * kC, sv);
        ptx::tmem_ld_wait(sv);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sfree[sb]);  // one arrival per warp

        // Raw scores; the max is taken before scaling (the scale is positive),
        // and the scale is folded into the exponent's FMA.
        float x[HK];
#pragma unroll
        for (int k2 = 0; k2 < HK; ++k2) x[k2] = __uint_as_float(sv[k2]);
        if (lim < HK) {  // a partial tile (the sequence's last chunk, or the causal limit)
#pragma unroll
          for (int k2 = 0; k2 < HK; ++k2)
            if (k2 >= lim) x[k2] = -INFINITY;
        }
        // P = 2^(x * scale - m), rounded to the operand type (bf16: plus the
        // rounded remainder); the row sum adds the values the PV product reads
        // (so o / n stays a weighted mean of V rows): the rounded ones for
        // fp16, for bf16 the unrounded ones, which hi + lo matches to 2^-17.
        uint32_t pw[HK / 2], pr[HK / 2];  // pr: the remainders (bf16 only)
        float2 ps[2];
        auto exps = [&](float m_ref) {
          const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_ref, -m_ref);
          ps[0] = ps[1] = make_float2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < HK / 2; ++q) {
            const float2 a = __ffma2_rn(make_float2(x[2 * q], x[2 * q + 1]), sc2, nm2);
            const float2 e = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
            pw[q] = pack2_plain<T>(e.x, e.y);
            if constexpr (PSPLIT) {
              const float2 h = make_float2(lo16<T>(pw[q]), hi16<T>(pw[q]));
              const float2 d = __ffma2_rn(h, make_float2(-1.f, -1.f), e);  // e - h, exact
              pr[q] = pack2_plain<T>(d.x, d.y);
              ps[q & 1] = __fadd2_rn(ps[q & 1], e);
            } else {
              ps[q & 1] = __fadd2_rn(ps[q & 1], make_float2(lo16<T>(pw[q]), hi16<T>(pw[q])));
            }
          }
        };
        // this half's max
        float mq[HK / 4];
#pragma unroll
        for (int k2 = 0; k2 < HK / 4; ++k2)
          mq[k2] = ptx::fmax3(fmaxf(x[4 * k2], x[4 * k2 + 1]), x[4 * k2 + 2], x[4 * k2 + 3]);
#pragma unroll
        for (int w2 = HK / 8; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int k2 = 0; k2 < w2; ++k2) mq[k2] = fmaxf(mq[k2], mq[k2 + w2]);
        const float hmax = mq[0];
        // Past an item's first tile the exponentials are taken against the
        // current reference at once; they stand unless some row of the warp
        // has a score past the reference by more than kRescale (then the
        // reference moves and they are taken again below).
        bool redo = (c == 0);
        if (!redo) {
          exps(m == -INFINITY ? 0.f : m);
          redo = __any_sync(0xffffffffu, hmax * sc > m + kRescale);
        }
        if (redo) {
          const float mxr = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 16));  // the row's other half
          const float mx = mxr * sc;
          // Move the reference max: always on the item's first tile (nothing
          // accumulated yet); later only when this tile's max runs past it.
          // Both halves of a row take the same decision.
          const bool move = (c == 0) || (mx > m + kRescale);
          const float m_old_use = (m == -INFINITY) ? 0.f : m;
          if (move) m = fmaxf(m, mx);
          const float m_use = (m == -INFINITY) ? 0.f : m;
          if (c > 0 && __any_sync(0xffffffffu, move)) {
            // O so far (through tile c-1) and l get the factor 2^(old - new):
            // wait for that tile's PV product, then rescale this half in place.
            const float alpha = move ? ptx::ex2(m_old_use - m_use) : 1.f;
            if (!wait_all(&pfree[(t - 1) & 1], ((t - 1) >> 1) & 1)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cg = 0; cg < HD / 32; ++cg) {
              uint32_t ov[32];
              ptx::tmem_ld32_half<HD>(tl + O_COL + ob * D + 32 * cg, ov);
              ptx::tmem_ld_wait(ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              ptx::tmem_st32_half<HD>(tl + O_COL + ob * D + 32 * cg, ov);
            }
            ptx::tmem_st_wait();
            l *= alpha;
          }
          exps(m_use);
        }
        // P buffer b is free once the PV product of tile t-2 has completed.
        if (__any_sync(0xffffffffu, !p_ready) && !wait_all(&pfree[b], ((t - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        // this half's 32 keys are P columns [16 hf, 16 hf + 16) (two keys per column)
        ptx::tmem_st16_half<HK / 2>(tl + P_COL + b * PW, pw);
        if constexpr (PSPLIT) ptx::tmem_st16_half<HK / 2>(tl + P_COL + b * PW + 32, pr);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();  // orders the TMEM stores above before the PV product
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&pfull[b]);  // one arrival per warp
        const float2 ps2 = __fadd2_rn(ps[0], ps[1]);
        l += ps2.x + ps2.y;
      }
      if (!ok) break;
      prefetch(ii + 1);
      // ---- hand the row's max and sum to the epilogue warps, which stream
      // O out once its last PV product has completed (ml_buf[ob] is free once
      // the epilogue of item it - 2 has read it)
      if (it >= 2 && !wait_all(&oempty[ob], ((it - 2) >> 1) & 1)) {
        ok = false;
        break;
      }
      const float lrow = l + __shfl_xor_sync(0xffffffffu, l, 16);  // the row sum of both halves
      if (hf == 0) ml_buf[ob * kBM + r] = make_float2(m, lrow);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&mlfull[ob]);  // one arrival per warp (release: ml_buf above)
    }
  } else {
    // --------------------------------------------------------------- epilogue
    // One thread per query row (TMEM lane quadrant warp % 4): once an item's
    // last PV product has completed and the softmax warps have left the row
    // max and sum in ml_buf, read O out of TMEM and write the item's partial
    // rows (the merge kernel combines them) or, for a prefill block, the
    // normalised output rows; meanwhile the softmax warps run the next item
    // into the other O buffer.
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(quad * 32) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, abort_flag, p.err));
    };
    for (int ii = i0; ii < i1; ++ii) {
      const int it = ii - i0, ob = it & 1;
      const WorkItem w = p.items[ii];
      const bool row_valid = r < w.n_rows;
      int grp = 0, hg = 0;
      if (row_valid) {
        const int rr = w.row0 + r;
        grp = w.group0 + rr / p.g;
        hg = rr % p.g;
      }
      // partial row: from the decode tables' row map, or, for a prefill block
      // cut along the keys (piece part_base of its rows), entry part_base of
      // the (token, KV head) pair's entries
      int part_row = 0;
      if (row_valid && !p.final_mode)
        part_row = p.causal_p0 >= 0 ? (__ldg(p.m_off + grp * p.Hkv + w.kv) + w.part_base) * p.g + hg
                                    : __ldg(p.row_idx + w.part_base + r);
      if (!wait_all(&ofull[ob], (it >> 1) & 1)) break;
      if (!wait_all(&mlfull[ob], (it >> 1) & 1)) break;
      ptx::tc_fence_after();
      const float2 ml = ml_buf[ob * kBM + r];
      const float inv = 1.f / ml.y;
      const size_t out_row = (static_cast<size_t>(grp) * p.Hq + w.kv * p.g + hg) * D;
      float* po = p.part_o + static_cast<size_t>(part_row) * D;
#pragma unroll
      for (int cg = 0; cg < D / 32; ++cg) {
        uint32_t ov[32];
        ptx::tmem_ld32(tl + O_COL + ob * D + 32 * cg, ov);
        ptx::tmem_ld_wait(ov);
        if (row_valid) {
          if (p.final_mode && p.out_f32) {
            float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row + 32 * cg);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                                  __uint_as_float(ov[4 * j + 2]) * inv, __uint_as_float(ov[4 * j + 3]) * inv);
          } else if (p.final_mode) {
            T* out = static_cast<T*>(p.out) + out_row + 32 * cg;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float* o8 = reinterpret_cast<const float*>(ov) + 8 * j;
              uint4 pk;
              pk.x = pack2_plain<T>(o8[0] * inv, o8[1] * inv);
              pk.y = pack2_plain<T>(o8[2] * inv, o8[3] * inv);
              pk.z = pack2_plain<T>(o8[4] * inv, o8[5] * inv);
              pk.w = pack2_plain<T>(o8[6] * inv, o8[7] * inv);
              *reinterpret_cast<uint4*>(out + 8 * j) = pk;
            }
          } else {
            float4* o4 = reinterpret_cast<float4*>(po + 32 * cg);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              o4[j] = make_float4(__uint_as_float(ov[4 * j]), __uint_as_float(ov[4 * j + 1]),
                                  __uint_as_float(ov[4 * j + 2]), __uint_as_float(ov[4 * j + 3]));
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&oempty[ob]);  // one arrival per warp
      if (row_valid && !p.final_mode) reinterpret_cast<float2*>(p.part_ml)[part_row] = ml;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // Let every bulk copy still in flight land before the CTA exits.
    for (int k = *consumed_slot; k < *issued_slot; ++k) ptx::mbar_wait(&full[k % kNS], (k / kNS) & 1, nullptr, p.err);
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, TMEM_COLS);
  }
  if (p.pdl) ptx::pdl_wait();  // never complete before the kernel we overlap
}

template <typename T, int D, int CP>
cudaError_t launch_tc_t(const AttnParams& p, int grid, cudaStream_t s) {
  const size_t smem = tc_smem_bytes(D);
  auto fn = attn_tc_kernel<T, D, CP>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <typename T, int D>
cudaError_t launch_tc_c(int C, const AttnParams& p, int grid, cudaStream_t s) {
  switch (C) {
    case 16: return launch_tc_t<T, D, 16>(p, grid, s);
    case 32: return launch_tc_t<T, D, 32>(p, grid, s);
    case 64: return launch_tc_t<T, D, 64>(p, grid, s);
    case 128: return launch_tc_t<T, D, 128>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool tc_supported(int dtype, int D, int C) {
  return (dtype == kF16 || dtype == kBF16) && (D == 64 || D == 128) && (C == 16 || C == 32 || C == 64 || C == 128);
}

size_t attn_tc_smem(int D) { return tc_smem_bytes(D); }

cudaError_t launch_attn_tc(int dtype, int D, int C, const AttnParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (dtype == kF16) {
    if (D == 128) return launch_tc_c<__half, 128>(C, p, grid, s);
    if (D == 64) return launch_tc_c<__half, 64>(C, p, grid, s);
  } else if (dtype == kBF16) {
    if (D == 128) return launch_tc_c<__nv_bfloat16, 128>(C, p, grid, s);
    if (D == 64) return launch_tc_c<__nv_bfloat16, 64>(C, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pst
