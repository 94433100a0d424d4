// Internal types shared by the host tree manager (pool.cpp) and the CUDA
// kernels (*.cu).  Not part of the public ABI.
#pragma once

#include <stdint.h>
#include <cuda_runtime.h>

namespace pst {

enum Dtype : int32_t { kF16 = 0, kBF16 = 1, kF32 = 2 };

inline int dtype_size(int dt) { return dt == kF32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// Pool layout.  The slab holds, per (chunk, KV head), one contiguous tile of
// 2 * C * D elements: first the K block (C key rows of D elements), then the
// transposed V block (D feature rows of C keys).  A block whose rows are a
// multiple of 128 bytes is stored as 128-byte column blocks one after another,
// each [rows][128 B], with the eight 16-byte chunks of row r permuted by XOR
// with (r mod 8).  That is the 128-byte-swizzled K-major operand image the
// tcgen05 tensor cores read from shared memory (so one bulk copy stages a
// tile ready for MMA), and it gives conflict-free 16-byte shared-memory reads
// to the CUDA-core kernel.  64-byte rows (16-bit V^T with c = 32) use plain
// 8-row x 16-byte core matrices.
// ---------------------------------------------------------------------------
__host__ __device__ inline uint32_t cm_off(uint32_t r, uint32_t j, uint32_t chunks_per_row) {
  return ((r >> 3) * chunks_per_row + j) * 128u + (r & 7u) * 16u;
}

// Byte offset of 16-byte chunk j of row r in a block of `rows` rows of
// `row_bytes` bytes.
__host__ __device__ inline uint32_t tile_off(uint32_t r, uint32_t j, uint32_t row_bytes, uint32_t rows) {
  if ((row_bytes & 127u) == 0) {
    return (j >> 3) * rows * 128u + r * 128u + (((j & 7u) ^ (r & 7u)) << 4);
  }
  return cm_off(r, j, row_bytes >> 4);
}

// One unit of partial-attention work: a list of chunks of one KV head against
// n_rows query rows.  Query rows are numbered in a "group-row" space: row
// rr = row0 + r belongs to group group0 + rr / g and query head kv * g + rr % g,
// where a group is a batch row (decode) or a token of the prefill block.
struct WorkItem {
  int32_t chunk_off;  // first entry in the chunk-id list
  int32_t n_chunks;
  int32_t kv;
  int32_t group0;
  int32_t row0;
  int32_t n_rows;
  int32_t part_base;  // partial mode: row r's partial row is row_idx[part_base + r] (decode), or,
                      // for a prefill block cut along the keys, entry m_off[pair] + part_base
  int32_t key0;       // causal mode: position of the item's first key in its sequence
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// Work item of the CUDA-core kernel: a run of chunks of one (batch row, KV
// head).  Runs of up to kSimtInline chunks carry their pool chunk ids in the
// item itself, so one 32-byte load tells a warp everything it needs to stage
// the run; longer runs (prefill) keep their ids in the chunk-id list.
constexpr int kSimtInline = 4;
struct alignas(16) SimtItem {
  int32_t chunk[kSimtInline];  // n_chunks <= kSimtInline: chunk ids; else chunk[0] = first entry in the id list
  int32_t n_chunks;            // 0 only in the kernel's "no more work" sentinel
  int32_t kv;
  int32_t group0;              // batch row (decode) or query position (prefill)
  int32_t part_base;           // partial-result row of head 0 (partial mode)
};
static_assert(sizeof(SimtItem) == 32, "SimtItem layout");

struct AttnParams {
  const uint8_t* pool;        // chunk slab
  const int32_t* chunk_len;   // valid tokens of each physical chunk
  const int32_t* chunks;      // chunk-id lists
  const WorkItem* items;      // tensor-core kernel items, or the CUDA-core kernel's SimtItem array
  const int32_t* warp_items;  // tensor-core kernel: item range [warp_items[c], warp_items[c+1]) of CTA c
  int32_t* sched;             // CUDA-core kernel: claim counter (zero at the step's start)
  int32_t first_items;        // CUDA-core kernel: items [0, first_items) go to consumer blockIdx * NW + warp
  int32_t claim_base;         // CUDA-core kernel: claimed index = counter value + claim_base
  int32_t n_items;
  int32_t claim_batch;        // CUDA-core kernel: items per claim once at most claim_tail are left
  int32_t claim_tail;         //   (before that, warps_per_cta per claim)
  const void* q;              // [groups][Hq][D]
  void* out;                  // final mode: [groups][Hq][D]
  float* part_o;              // partial mode: [rows][D]
  float* part_ml;             // partial mode: [rows][2] = (m, n), m in log2 units
  int32_t Hq, Hkv, g;
  int32_t chunk_size;
  int32_t final_mode;         // 0: write (o, m, n) partials; 1: write o / n to out
  int32_t causal_p0;          // >= 0: group t sees keys [0, causal_p0 + t]; < 0: no causal limit
  float scale_log2;           // log2(e) / sqrt(D), computed on the host
  int32_t stages;             // CUDA-core kernel: piece stages per warp
  int32_t warps_per_cta;      // CUDA-core kernel
  int32_t* err;               // device error word
  // Partial rows are grouped per (batch row, KV head) pair: entry e of the
  // pair (m_off[key] <= e < m_off[key + 1], key = u * Hkv + kv) holds head
  // kv*g + hg at row e*g + hg.
  const int32_t* m_off;       // [B * Hkv + 1]
  const int32_t* row_idx;     // tensor-core kernel: partial row of item row r at row_idx[item.part_base + r]
  // CUDA-core kernel: 1 when every K/V tile it stages is read by one item
  // only (decode with the shared chunks on the tensor cores): its copies then
  // take the L2 evict-first priority, so the streamed tiles do not push the
  // partial rows that the merge reads next out of L2.
  int32_t kv_evict_first;
  // merge kernel: pairs with at most this many entries stage them in shared
  // memory (0: none do)
  int32_t merge_cap;
  // 1: launched as a programmatic dependent of the previous kernel on the
  // stream (it may start while that kernel drains; it must not finish first)
  int32_t pdl;
  // 1: `out` holds fp32 rows whatever the K/V type (the value before the
  // final rounding to the K/V type; PST_FLAG_F32_OUT)
  int32_t out_f32;
};



// Copies user K/V rows into pool tiles (or back out, for gather).
struct ScatterOp {
  int32_t chunk;     // physical chunk
  int32_t src_row;   // first user row (token) of this op
  int32_t r0, r1;    // rows [r0, r1) of the chunk are written from src_row...
  int32_t zero_tail; // 1: rows [r1, C) are zero-filled (freshly allocated chunk)
};
// Ops per scatter launch: they travel in the kernel parameters (20 bytes
// each), so a decode step's batched append of up to 512 sequences is one launch.
constexpr int kScatterMax = 512;
struct ScatterParams {
  const uint8_t* k;   // scatter: source [rows][Hkv][D]; gather: destination
  const uint8_t* v;
  uint8_t* pool;
  int32_t* chunk_len;
  int32_t n_ops;
  int32_t Hkv;
  ScatterOp ops[kScatterMax];
};

// Error codes OR-ed into the device error word.
enum : int32_t {
  kErrWaitTimeout = 1,   // a bounded mbarrier wait ran out
  kErrBadIndex = 2,      // an index check failed
};

// Fixed device scratch used by pst_decode_attention_noalloc (static_scratch.cu).
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
// Device address of that area on `device` (looked up once per device, with
// the device made current for the lookup).
cudaError_t static_scratch_address(int device, void** ptr);

// Launchers (defined in the .cu files).  All return the launch status.
cudaError_t launch_scatter(int dtype, int D, int C, const ScatterParams& p, cudaStream_t s);
cudaError_t launch_gather(int dtype, int D, int C, const ScatterParams& p, cudaStream_t s);
cudaError_t launch_attn_simt(int dtype, int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s);
size_t attn_simt_smem(int dtype, int D, int C, int g, int stages, int warps_per_cta);
size_t attn_simt_piece_bytes(int dtype, int D, int C);  // bytes of one ring stage of the CUDA-core kernel
int attn_simt_max_warps(int dtype, int g);  // consumer warps per CTA of the CUDA-core kernel, at most
// per-dtype launchers for chunk sizes 64 / 128 (large) and 16 / 32 (small),
// one translation unit each
#define PST_SIMT_LAUNCHER(dt)                                                                                   \
  cudaError_t launch_attn_simt_##dt##_large(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s); \
  cudaError_t launch_attn_simt_##dt##_small(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s);
PST_SIMT_LAUNCHER(f16)
PST_SIMT_LAUNCHER(bf16)
PST_SIMT_LAUNCHER(f32)
#undef PST_SIMT_LAUNCHER
cudaError_t launch_attn_tc(int dtype, int D, int C, const AttnParams& p, int grid, cudaStream_t s);
size_t attn_tc_smem(int D);
// Merge of the partial rows of every (batch row, KV head) pair into `out`
// (one warp per pair); a programmatic dependent of the previous kernel when
// p.pdl is set.
cudaError_t launch_merge(int dtype, int D, const AttnParams& p, int B, cudaStream_t s);
bool simt_supported(int dtype, int D, int g);
bool tc_supported(int dtype, int D, int C);

}  // namespace pst
