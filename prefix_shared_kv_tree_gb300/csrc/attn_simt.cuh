// Sequence-first partial attention (ChunkAttention, Knowl 2 phase 2, with
// partial_attn / attn_reduce of Knowl 3).  Also runs the chunk-first phase
// when the tensor-core kernel does not apply (fp32 K/V, or the
// PST_FLAG_NO_TENSOR_CORES flag), and causal prefill blocks in that case.
//
// Warp-specialised, warp-per-stream design.  A CTA holds NW consumer warps and
// one producer warp; lane c of the producer serves consumer c:
//   * it claims work items (a run of up to four chunks of one (group, KV
//     head), chunk ids inline; longer prefill runs keep theirs in the chunk
//     list) for the whole CTA, NW consecutive indices per atomic on a global
//     counter, largest first: two batches are in hand and the claim of a third
//     is in flight, and a batch's descriptors land in shared memory by one
//     bulk copy, so consumers whose SM came free late (an earlier kernel held
//     it) simply get fewer;
//   * it fills the consumer's two item slots: the item header by shared
//     stores, the chunks' valid-token counts by 4-byte async copies, the
//     query rows by one bulk async copy;
//   * the consumer's lane 0 keeps its ring of `stages` pieces full with bulk
//     async copies (TMA engine): a tile is consumed as pieces of up to 64
//     rows -- each key run of every 128-byte column block of K, then each
//     row group of V^T -- each a contiguous block of the pool's tile image.
// The consumer warps issue no global load and no atomic: every latency of the
// item pipeline (claim, descriptor, chunk lengths, query rows) sits in the
// producer, which waits for none of them in the step that issued it.  For
// 16-bit K/V the products run on the tensor cores as warp-level mma.sync
// m16n8k16: S^T = K Q^T and O^T = V^T P^T with keys / output features on the
// 16-row side and the item's <= 8 query rows on the 8-column side (bf16
// probabilities as two bf16 terms, the rounded value and the rounded
// remainder); the online softmax per query column uses shuffles over the 8
// lanes that hold it.  fp32 K/V: lane = key, packed fp32 FMAs, warp-shuffle
// tile max, row sums lane-local until the item ends; values with lane =
// output feature row of V^T.  The item's (o, m, n) rows then go to the
// partial buffer; the merge kernel that follows combines the rows of every
// (batch row, KV head).
#pragma once

#include "attn_common.cuh"
#include "ptx.cuh"

namespace pst {

__host__ __device__ inline size_t simt_align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rows per piece of a tile (see tile_off): each run of kSimtPieceRows keys of
// every 128-byte column block of K, then each run of kSimtPieceRows rows of
// every column block of V^T -- each a contiguous block of the tile image.
#ifndef PST_SIMT_PIECE_ROWS
#define PST_SIMT_PIECE_ROWS 64
#endif
constexpr int kSimtPieceRows = PST_SIMT_PIECE_ROWS;

static_assert(kSimtPieceRows == 32 || kSimtPieceRows == 64, "piece rows");

// Pieces per ring stage.  With 16-bit K/V, chunks shorter than a piece
// (16 or 32 keys) make pieces of 2 or 4 KB that are consecutive, equal blocks
// of the tile image (each 128-byte K column block of C rows, then each run of
// 64 V^T rows of C * 2 bytes): a stage then holds up to 8 KB of consecutive
// pieces, staged by one bulk copy and waited for once.
__host__ __device__ inline int simt_pieces_per_stage(int C, int D, int es) {
  if (es != 2 || C >= kSimtPieceRows) return 1;
  const int np = D / 32;         // pieces per tile: 2 C D bytes in pieces of 128 C bytes
  const int fit = 8192 / (128 * C);
  return np < fit ? np : fit;
}

__host__ __device__ inline size_t simt_stage_bytes(int C, int D, int es) {
  const int kr = C < kSimtPieceRows ? C : kSimtPieceRows;
  const int vr = D < kSimtPieceRows ? D : kSimtPieceRows;
  const size_t kpb = static_cast<size_t>(kr) * 128;
  const size_t vpb = ((C * es) % 128 == 0) ? static_cast<size_t>(vr) * 128 : static_cast<size_t>(vr) * C * es;
  return (kpb > vpb ? kpb : vpb) * simt_pieces_per_stage(C, D, es);
}

// Consumer warps per CTA at most (one more warp produces).  16-bit K/V take
// the tensor-core consumer (about 100 registers at any query group).  The fp32
// consumer keeps its G query rows' partial sums in registers: with nine warps
// one SM sub-partition holds three, which caps registers at 168 per thread,
// so query groups of four and more take seven consumers (255 registers).
#ifndef PST_SIMT_MMA_WARPS
#define PST_SIMT_MMA_WARPS 8
#endif
#ifndef PST_SIMT_G4_WARPS
#define PST_SIMT_G4_WARPS 7
#endif
#ifndef PST_SIMT_G1_WARPS
#define PST_SIMT_G1_WARPS 8
#endif
constexpr int kSimtMaxWarps = 12;  // capacity of the producer's per-CTA structures
__host__ __device__ constexpr int simt_max_warps(int G, int es) {
  return es == 2 ? PST_SIMT_MMA_WARPS : G >= 8 ? 7 : G >= 4 ? PST_SIMT_G4_WARPS : G >= 2 ? 8 : PST_SIMT_G1_WARPS;
}
static_assert(PST_SIMT_G1_WARPS <= kSimtMaxWarps && PST_SIMT_G4_WARPS <= kSimtMaxWarps &&
                  PST_SIMT_MMA_WARPS <= kSimtMaxWarps,
              "consumer warps");

// Item slot: a 64-byte header -- [0] n_chunks (0: no more work), [1] kv,
// [2] group0, [3] part_base, [4..7] valid tokens of the first four chunks,
// [8] chunk-list offset of a longer run, [12..15] the chunk ids of a run of
// at most four -- then the item's G query rows as stored (G * D elements).
constexpr int kSlotHeader = 64;

// Shared memory of one consumer warp, all offsets from the warp's base:
// [stages x piece][q rows fp32][p][2 item slots][barriers: full[S], empty[S],
// slot_full[2], slot_empty[2]].  The fp32 consumer keeps the scaled query rows
// and the probabilities (G x C fp32); the tensor-core consumer (16-bit K/V)
// keeps its query rows in registers and the probabilities as the transposed
// C x 8 block of 16-bit values (one 16-byte row per key, columns past G
// unused) that the P V product reads back -- for bf16 two such blocks, P's
// rounded value and the rounded remainder (see the consumer).
struct SimtLayout {
  uint32_t stage, q, p, slot, slot_bytes, bars, total;
};

__host__ __device__ inline SimtLayout simt_layout(int C, int D, int G, int S, int es, bool p_split) {
  SimtLayout L;
  L.stage = static_cast<uint32_t>(simt_stage_bytes(C, D, es));
  size_t off = static_cast<size_t>(S) * L.stage;
  const bool mma = es == 2;
  L.q = static_cast<uint32_t>(off);
  off += mma ? 0 : static_cast<size_t>(G) * D * 4;
  L.p = static_cast<uint32_t>(off);
  off += mma ? static_cast<size_t>(C) * 16 * (p_split ? 2 : 1) : static_cast<size_t>(G) * C * 4;
  off = simt_align_up(off, 128);
  L.slot = static_cast<uint32_t>(off);
  L.slot_bytes = static_cast<uint32_t>(kSlotHeader + static_cast<size_t>(G) * D * es);
  off += 2 * static_cast<size_t>(L.slot_bytes);
  off = simt_align_up(off, 8);
  L.bars = static_cast<uint32_t>(off);
  off += static_cast<size_t>(2 * S + 4) * 8;
  L.total = static_cast<uint32_t>(simt_align_up(off, 128));
  return L;
}

__host__ __device__ inline size_t simt_warp_bytes(int C, int D, int G, int S, int es, bool p_split) {
  return simt_layout(C, D, G, S, es, p_split).total;
}

// A work item as loaded: the two raw 16-byte halves of the SimtItem and
// whether the claimed index was a real item.  The producer lets a loaded item
// sit for a whole item before touching it, so the load's latency never stalls.
struct SimtMeta {
  int4 a;  // chunk[0..3]
  int4 b;  // n_chunks, kv, group0, part_base
  int valid;
  __device__ __forceinline__ int n_chunks() const { return valid ? b.x : 0; }
  __device__ __forceinline__ int kv() const { return b.y; }
  __device__ __forceinline__ int group0() const { return b.z; }
  __device__ __forceinline__ int part_base() const { return b.w; }
};

// Loads item idx (a claimed index; past the end it reads the last item and
// marks the result invalid).  n_items >= 1.
__device__ __forceinline__ SimtMeta simt_load_item(const SimtItem* items, int idx, int n_items) {
  SimtMeta m;
  const int4* src = reinterpret_cast<const int4*>(items + min(idx, n_items - 1));
  m.a = __ldg(src);
  m.b = __ldg(src + 1);
  m.valid = idx < n_items;
  return m;
}

// Chunk id c of an item (inline ids, or the id list for long runs); c < n.
__device__ __forceinline__ int simt_chunk_id(const SimtMeta& m, int c, const int32_t* chunks) {
  if (m.b.x > kSimtInline) return chunks[m.a.x + c];
  return c == 0 ? m.a.x : c == 1 ? m.a.y : c == 2 ? m.a.z : m.a.w;
}

template <typename T, int D, int G, int C>
__global__ void __launch_bounds__(32 * (simt_max_warps(G, sizeof(T)) + 1), 1) attn_simt_kernel(const AttnParams p) {
  constexpr int ES = sizeof(T);
  constexpr int VEC = 16 / ES;
  constexpr int DCH = D / VEC;     // 16-byte chunks per query row
  constexpr int KB = D * ES / 128;                       // K: 128-byte column blocks of C rows
  constexpr int KPR = C < kSimtPieceRows ? C : kSimtPieceRows;  // keys per K piece
  constexpr int KPC = C / KPR;                           // K pieces per column block
  // fp32 consumer, lane = key: keys per lane per K piece and per chunk (a
  // chunk shorter than a warp leaves lanes C .. 31 on masked duplicates)
  constexpr int KT = KPR >= 32 ? KPR / 32 : 1;
  constexpr int KPL = C >= 32 ? C / 32 : 1;
  constexpr bool VSW = (C * ES) % 128 == 0;              // V^T rows in 128-byte swizzled blocks
  constexpr int VB = VSW ? C * ES / 128 : 1;             // V^T column blocks
  constexpr int VPR = D < kSimtPieceRows ? D : kSimtPieceRows;  // feature rows per V^T piece
  constexpr int VG = D / VPR;                            // V^T pieces per column block
  constexpr int VT = VPR / 32;                           // feature rows per lane per V^T piece
  constexpr int NP = KB * KPC + VB * VG;                 // pieces per tile
  constexpr int PPS = C < kSimtPieceRows && ES == 2 ? (D / 32 < 8192 / (128 * C) ? D / 32 : 8192 / (128 * C)) : 1;
  constexpr int DPL = D / 32;      // output features per lane
  constexpr int KCH = 128 / 16;    // 16-byte chunks per K piece row
  constexpr int VCH = VSW ? 8 : C * ES / 16;             // 16-byte chunks per V^T piece row
  constexpr uint32_t KPB = static_cast<uint32_t>(KPR) * 128u;
  constexpr uint32_t VPB = VSW ? static_cast<uint32_t>(VPR) * 128u : static_cast<uint32_t>(VPR) * C * ES;
  // several pieces per stage (see simt_pieces_per_stage): equal, consecutive
  // blocks of the tile image
  static_assert(PPS == 1 || (KPC == 1 && !VSW && VPR == 64 && KPB == VPB && NP % PPS == 0 && PPS * KPB <= 8192),
                "pieces per stage");
  constexpr uint32_t HALF = static_cast<uint32_t>(C) * D * ES;
  constexpr size_t TILE = 2 * static_cast<size_t>(HALF);
  constexpr uint32_t QBYTES = static_cast<uint32_t>(G) * D * ES;
  constexpr int NQ = (G * DCH + 31) / 32;  // 16-byte query pieces per lane
  // 16-bit K/V: warp-level tensor-core products with the keys (scores) and
  // the output features (values) as the 16-row M side and the item's query
  // rows as the 8-column N side.
  constexpr bool kMma = ES == 2;
  static_assert(!kMma || (G <= 8 && C % 16 == 0 && KPR % 16 == 0 && VPR % 16 == 0), "mma shape");
  const int S = p.stages;
  const int NW = p.warps_per_cta;  // consumer warps; warp NW produces
  // bf16 probabilities go to the tensor cores as two bf16 terms, the rounded
  // value and the rounded remainder: 16 significant bits instead of 8, so a
  // row dominated by a few keys keeps its accuracy
  constexpr bool kPSplit = std::is_same<T, __nv_bfloat16>::value;
  const SimtLayout L = simt_layout(C, D, G, S, ES, kPSplit);

  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ __align__(16) SimtItem s_batch[2][kSimtMaxWarps];  // claimed item descriptors, two batches of NW
  __shared__ uint64_t s_bbar[2];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  ptx::pdl_launch_dependents();  // the merge kernel may become resident; it waits for us
  const int n_items = p.n_items;
  const SimtItem* items = reinterpret_cast<const SimtItem*>(p.items);

  if (threadIdx.x == 0) {
    s_abort = 0;
    ptx::mbar_init(&s_bbar[0], 1);
    ptx::mbar_init(&s_bbar[1], 1);
  }
  if (warp < NW && lane == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(warp) * L.total + L.bars);
    for (int s = 0; s < 2 * S + 4; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  if (warp == NW) {
    // ================================================================ producer
    // Fills lane c's consumer's two item slots (c < NW).  Items are claimed
    // for the whole CTA, NW consecutive indices per atomic while more than
    // p.claim_tail items are left, then p.claim_batch (fewer items reserved by
    // one CTA when the list runs out, so the warps end closer together); a
    // batch's descriptors land in s_batch by one bulk copy.  Two batches are
    // in hand and the claim of a third is in flight, so this warp never reads
    // a register that a global load or atomic of the current step still
    // fills (its lanes share one scoreboard: such a read would stall every
    // lane).
    const int small = min(NW, max(1, p.claim_batch));
    auto claim_size = [&](int next) { return n_items - next > p.claim_tail ? NW : small; };
    const bool mine = lane < NW;
    uint8_t* rb = smem + static_cast<size_t>(mine ? lane : 0) * L.total;
    uint8_t* slots = rb + L.slot;
    uint64_t* bars = reinterpret_cast<uint64_t*>(rb + L.bars);
    uint64_t* sfull = bars + 2 * S;
    uint64_t* sempty = bars + 2 * S + 2;
    const T* qptr = static_cast<const T*>(p.q);
    auto fill_batch = [&](int buf, int base, int sz) {  // lane 0
      const int valid = max(0, min(n_items - base, sz));
      if (valid > 0) {
        ptx::mbar_arrive_expect_tx(&s_bbar[buf], valid * static_cast<uint32_t>(sizeof(SimtItem)));
        ptx::bulk_g2s(&s_batch[buf][0], items + base, valid * static_cast<uint32_t>(sizeof(SimtItem)), &s_bbar[buf]);
      } else {
        ptx::mbar_arrive(&s_bbar[buf]);
      }
    };
    // batch b: items [base_b, base_b + sz_b); pend: the claim in flight
    int base0 = 0, base1 = 0, pend = 0;
    int sz0 = claim_size(p.claim_base), sz1 = sz0, pend_sz = sz0;
    if (lane == 0) {
      base0 = atomicAdd(p.sched, sz0) + p.claim_base;
      base1 = atomicAdd(p.sched, sz1) + p.claim_base;
    }
    base0 = __shfl_sync(0xffffffffu, base0, 0);
    base1 = __shfl_sync(0xffffffffu, base1, 0);
    if (lane == 0) {
      fill_batch(0, base0, sz0);
      fill_batch(1, base1, sz1);
      pend_sz = claim_size(base1 + sz1);
      pend = base1 + sz1 < n_items ? atomicAdd(p.sched, pend_sz) + p.claim_base : n_items;
    }
    uint32_t fills0 = 1, fills1 = 1;
    int bcur = 0, bpos = 0;
    bool finished = !mine;
    int qs = 0;
    uint32_t written = 0, idle = 0;
    uint64_t idle_since = 0;
    while (true) {
      // ---- next item into the consumer's next slot, once it has released it
      bool want = !finished && (written < 2 || ptx::mbar_test_wait(&sempty[qs], ((written >> 1) - 1) & 1));
      unsigned wm = __ballot_sync(0xffffffffu, want);
      // at most the rest of the two batches in hand on this pass
      const int szc = bcur ? sz1 : sz0;
      const int room = szc + (bcur ? sz0 : sz1) - bpos;
      if (__popc(wm) > room) {
        want = want && __popc(wm & ((1u << lane) - 1u)) < room;
        wm = __ballot_sync(0xffffffffu, want);
      }
      if (wm != 0u) {
        const int cnt = __popc(wm);
        // the current batch (and, past its end, the next) must have landed
        bool ok = ptx::mbar_wait(&s_bbar[bcur], ((bcur ? fills1 : fills0) - 1) & 1, abort_flag, p.err);
        if (bpos + cnt > szc)
          ok = ok && ptx::mbar_wait(&s_bbar[bcur ^ 1], ((bcur ? fills0 : fills1) - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (want) {
          const int pos = bpos + __popc(wm & ((1u << lane) - 1u));
          const int buf = pos < szc ? bcur : (bcur ^ 1);
          const int i = pos < szc ? pos : pos - szc;
          const int idx = (buf ? base1 : base0) + i;
          const int4* d = reinterpret_cast<const int4*>(&s_batch[buf][i]);
          SimtMeta cur;
          cur.a = d[0];
          cur.b = d[1];
          cur.valid = idx < n_items;
          uint8_t* sl = slots + static_cast<size_t>(qs) * L.slot_bytes;
          int* hdr = reinterpret_cast<int*>(sl);
          const int n = cur.n_chunks();
          hdr[0] = n;
          if (n > 0) {
            hdr[1] = cur.kv();
            hdr[2] = cur.group0();
            hdr[3] = cur.part_base();
            hdr[8] = cur.a.x;
            *reinterpret_cast<int4*>(hdr + 12) = cur.a;  // chunk ids of a short run (words 12..15)
            if (n <= kSimtInline) {
              for (int c = 0; c < n; ++c) ptx::cp_async_4(hdr + 4 + c, p.chunk_len + simt_chunk_id(cur, c, p.chunks));
              ptx::cp_async_mbar_arrive(&sfull[qs]);  // the slot completes only once they landed
            }
            ptx::mbar_arrive_expect_tx(&sfull[qs], QBYTES);  // release: the header stores above
            ptx::bulk_g2s(sl + kSlotHeader, qptr + (static_cast<size_t>(cur.group0()) * p.Hq + cur.kv() * p.g) * D,
                          QBYTES, &sfull[qs]);
          } else {
            ptx::mbar_arrive(&sfull[qs]);  // end marker
            finished = true;
          }
          ++written;
          if (++qs == 2) qs = 0;
        }
        bpos += cnt;
        if (bpos >= szc) {
          // The current batch is used up (every read of it above fed a store
          // that has issued): refill its buffer with the batch claimed last time.
          const int nb = __shfl_sync(0xffffffffu, pend, 0);
          const int nsz = __shfl_sync(0xffffffffu, pend_sz, 0);
          if (bcur == 0) {
            base0 = nb;
            sz0 = nsz;
            ++fills0;
          } else {
            base1 = nb;
            sz1 = nsz;
            ++fills1;
          }
          if (lane == 0) {
            fill_batch(bcur, nb, nsz);
            pend_sz = claim_size(nb + nsz);
            pend = nb + nsz < n_items ? atomicAdd(p.sched, pend_sz) + p.claim_base : n_items;
          }
          bcur ^= 1;
          bpos -= szc;
        }
      }
      if (__all_sync(0xffffffffu, finished)) break;
      if (*abort_flag) break;
      if (wm != 0u) {
        idle = 0;
      } else if ((++idle & 255u) == 0) {  // the timer is read now and then only
        const uint64_t t = ptx::globaltimer();
        if (idle == 256) {
          idle_since = t;
        } else if (t - idle_since > ptx::kWaitLimitNs) {
          if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
          *abort_flag = 1;
        }
      }
    }
    // Every bulk copy this warp started must land before the CTA exits: the
    // last fill of each batch buffer and of each of this lane's slots.
    ptx::mbar_wait(&s_bbar[0], (fills0 - 1) & 1, nullptr, p.err);
    ptx::mbar_wait(&s_bbar[1], (fills1 - 1) & 1, nullptr, p.err);
    if (mine)
      for (int q = 0; q < 2; ++q)
        if (written > static_cast<uint32_t>(q)) {
          const uint32_t last = q + ((written - 1 - q) / 2) * 2;
          ptx::mbar_wait(&sfull[q], (last >> 1) & 1, nullptr, p.err);
        }
  } else {
    // ================================================================ consumer
    uint8_t* rb = smem + static_cast<size_t>(warp) * L.total;
    uint8_t* stages = rb;
    float* qbuf = reinterpret_cast<float*>(rb + L.q);
    float* pbuf = reinterpret_cast<float*>(rb + L.p);
    uint8_t* pbuf_b = rb + L.p;  // tensor-core consumer: P^T, C rows of 16 bytes
    const uint8_t* slots = rb + L.slot;
    uint64_t* bars = reinterpret_cast<uint64_t*>(rb + L.bars);
    uint64_t* full = bars;
    uint64_t* sfull = bars + 2 * S;
    uint64_t* sempty = bars + 2 * S + 2;

    // The first item may be handed out statically (item blockIdx * NW + warp
    // of the launch's first wave) and read straight from the item table, so
    // the warp starts streaming without waiting for its producer; items after
    // it come through the slots.
    const int sidx = static_cast<int>(blockIdx.x) * NW + warp;
    const bool has_static = sidx < min(p.first_items, n_items);
    const uint32_t kofs = has_static ? 1u : 0u;
    const SimtMeta st = simt_load_item(items, has_static ? sidx : n_items, n_items);
    const T* qptr_g = static_cast<const T*>(p.q);

    // Staging (whole warp, all lanes in step): the tiles of item si (this
    // item or the next) go into the warp's ring of S pieces; an item's chunk
    // ids come from its slot header, which the producer wrote before that
    // slot completed.
    uint32_t k = 0;  // items started
    uint32_t si = 0;          // item being staged
    bool s_ready = false;     // its header is in s_* below
    bool s_done = false;      // no more items to stage
    int s_n = 0, s_kv = 0, s_list = 0, pc = 0, pp = 0, ps = 0;
    int4 s_ids = make_int4(0, 0, 0, 0);
    uint32_t issued = 0;
    const uint64_t kv_policy = ptx::policy_evict_first();
    auto issue_next = [&]() -> bool {  // false: nothing can be issued now
      if (s_done || si > k + 1) return false;
      if (!s_ready) {
        if (si < kofs) {
          s_n = st.b.x;
          s_kv = st.b.y;
          s_list = st.a.x;
          s_ids = st.a;
        } else {
          const uint32_t js = si - kofs;
          // every lane observes the phase (each read below is ordered by its
          // own acquire); the decision is the warp's
          if (!__all_sync(0xffffffffu, ptx::mbar_test_wait(&sfull[js & 1], (js >> 1) & 1))) return false;
          const int* h = reinterpret_cast<const int*>(slots + static_cast<size_t>(js & 1) * L.slot_bytes);
          s_n = h[0];
          if (s_n == 0) {
            s_done = true;
            return false;
          }
          s_kv = h[1];
          s_list = h[8];
          s_ids = *reinterpret_cast<const int4*>(h + 12);
        }
        s_ready = true;
        pc = 0;
        pp = 0;
      }
      const int chunk = s_n > kSimtInline ? p.chunks[s_list + pc]
                                          : (pc == 0 ? s_ids.x : pc == 1 ? s_ids.y : pc == 2 ? s_ids.z : s_ids.w);
      const uint8_t* tile = p.pool + (static_cast<size_t>(chunk) * p.Hkv + s_kv) * TILE;
      const uint8_t* src;
      uint32_t bytes;
      if (pp < KB * KPC) {
        src = tile + (pp / KPC) * (C * 128) + (pp % KPC) * KPB;
        bytes = KPB;
      } else {
        const int vb = (pp - KB * KPC) / VG, vg = (pp - KB * KPC) % VG;
        src = tile + HALF + (VSW ? (static_cast<size_t>(vb) * D * 128 + vg * VPB) : static_cast<size_t>(vg) * VPB);
        bytes = VPB;
      }
      bytes *= PPS;  // the stage's PPS consecutive pieces
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx_relaxed(&full[ps], bytes);
        if (p.kv_evict_first)
          ptx::bulk_g2s_hint(stages + static_cast<size_t>(ps) * L.stage, src, bytes, &full[ps], kv_policy);
        else
          ptx::bulk_g2s(stages + static_cast<size_t>(ps) * L.stage, src, bytes, &full[ps]);
      }
      ++issued;
      if (++ps == S) ps = 0;
      pp += PPS;
      if (pp == NP) {
        pp = 0;
        if (++pc == s_n) {
          ++si;
          s_ready = false;
        }
      }
      return true;
    };
    uint32_t consumed = 0;
    int cs = 0;          // stage of the next piece
    uint32_t cph = 0;    // its mbarrier phase parity
    bool aborted = false;

    for (; !aborted; ++k) {
      const bool stat = k < kofs;
      const uint32_t js = k - kofs;  // slot sequence number of a non-static item
      const int qs = js & 1;
      const uint8_t* sl = slots + static_cast<size_t>(qs) * L.slot_bytes;
      int n_chunks, kv, grp, part_base, list_off, my_len;
      const uint8_t* qsrc;  // the item's G query rows as stored
      if (stat) {
        n_chunks = st.b.x;
        kv = st.b.y;
        grp = st.b.z;
        part_base = st.b.w;
        list_off = st.a.x;
        my_len = (lane < n_chunks && n_chunks <= kSimtInline)
                     ? p.chunk_len[simt_chunk_id(st, min(lane, kSimtInline - 1), p.chunks)]
                     : 0;
        qsrc = reinterpret_cast<const uint8_t*>(qptr_g + (static_cast<size_t>(grp) * p.Hq + kv * p.g) * D);
      } else {
        if (!ptx::mbar_wait(&sfull[qs], (js >> 1) & 1, abort_flag, p.err)) break;
        const int* hdr = reinterpret_cast<const int*>(sl);
        n_chunks = hdr[0];
        if (n_chunks == 0) break;  // end marker
        kv = hdr[1];
        grp = hdr[2];
        part_base = hdr[3];
        list_off = hdr[8];
        // valid tokens of chunks 0 .. 31 of this item, one per lane
        my_len = lane < n_chunks ? hdr[4 + min(lane, kSimtInline - 1)] : 0;
        qsrc = sl + kSlotHeader;
      }
      // long runs (prefill only) read their chunk lengths from the chunk-length array
      if (n_chunks > kSimtInline) my_len = lane < n_chunks ? p.chunk_len[p.chunks[list_off + lane]] : 0;
      // query rows of this item: the tensor-core consumer holds them as the
      // B operand of S^T = K Q^T (column n = query row lane / 4, zero past G);
      // the fp32 consumer keeps them in qbuf, pre-scaled into log2 units
      uint32_t qf[kMma ? D / 16 : 1][2];
      if constexpr (kMma) {
        if (!stat) {
          // from the slot, two k-steps per ldmatrix: matrix i holds features
          // 8 i .. 8 i + 7 of the pair's 16-feature span, rows = query rows
          // (rows past G repeat row G-1: their columns are never stored)
          const uint32_t qb = ptx::smem_u32(qsrc) + static_cast<uint32_t>(min(lane & 7, G - 1) * D * ES) + (lane >> 3) * 16;
#pragma unroll
          for (int k2 = 0; k2 < D / 32; ++k2) {
            uint32_t r[4];
            ptx::ldsm_x4(qb + k2 * 64, r);
            qf[2 * k2][0] = r[0];
            qf[2 * k2][1] = r[1];
            qf[2 * k2 + 1][0] = r[2];
            qf[2 * k2 + 1][1] = r[3];
          }
        } else {
          const int n = lane >> 2;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            if (n < G) {
              const uint8_t* qr = qsrc + (static_cast<size_t>(n) * D + ks * 16 + 2 * (lane & 3)) * ES;
              qf[ks][0] = *reinterpret_cast<const uint32_t*>(qr);
              qf[ks][1] = *reinterpret_cast<const uint32_t*>(qr + 16);
            } else {
              qf[ks][0] = qf[ks][1] = 0u;
            }
          }
        }
      } else {
#pragma unroll
        for (int kq = 0; kq < NQ; ++kq) {
          const int idx = lane + 32 * kq;
          if (idx < G * DCH) {
            const int h = idx / DCH, j = idx % DCH;
            float f[VEC];
            unpack16<T>(*reinterpret_cast<const uint4*>(qsrc + (static_cast<size_t>(h) * D + j * VEC) * ES), f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qbuf[h * D + j * VEC + e] = f[e] * p.scale_log2;
          }
        }
      }
      // stage ahead: the rest of this item and the start of the next
      while (issued < consumed + S && issue_next()) {
      }
      __syncwarp();
      // The slot is free once the header and rows are in registers / qbuf;
      // staging (above) read item k+1's slot, never item k's after this.
      if (!stat && lane == 0) ptx::mbar_arrive_relaxed(&sempty[qs]);

      if constexpr (kMma) {
        // ---- tensor-core consumer.  Lane roles of the m16n8k16 fragments:
        // rows (keys of S^T, features of O^T) lg = lane / 4 and lg + 8 of
        // each 16-row tile, query columns 2 lq and 2 lq + 1, lq = lane % 4.
        constexpr int MT = C / 16;        // key tiles of a chunk
        constexpr int KMT = KPR / 16;     // key tiles of a K piece
        constexpr int VMT = VPR / 16;     // feature tiles of a V^T piece
        constexpr int OMT = D / 16;       // feature tiles of the output
        constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
        const int lg = lane >> 2, lq = lane & 3;
        // ldmatrix row of this lane within a 16-row tile, and its 16-byte
        // column half: matrices 0..3 = (rows 0-7, k 0-7), (rows 8-15, k 0-7),
        // (rows 0-7, k 8-15), (rows 8-15, k 8-15) -- the A fragment order
        const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int a_hi = lane >> 4;
        const uint32_t pb = ptx::smem_u32(pbuf);
        float m2[2] = {-INFINITY, -INFINITY}, nl2[2] = {0.f, 0.f};
        float o[OMT][4];
#pragma unroll
        for (int t = 0; t < OMT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;

        for (int c = 0; c < n_chunks && !aborted; ++c) {
          if ((c & 31) == 0 && c > 0) {  // valid tokens of chunks c .. c+31 (long runs only)
            my_len = c + lane < n_chunks ? p.chunk_len[p.chunks[list_off + c + lane]] : 0;
          }
          int lim = __shfl_sync(0xffffffffu, my_len, c & 31);
          if (p.causal_p0 >= 0) lim = min(lim, p.causal_p0 + grp + 1 - c * C);

          // ---- S^T = K Q^T over the K pieces (raw scores, fp32)
          float sacc[MT][4];
#pragma unroll
          for (int t = 0; t < MT; ++t) sacc[t][0] = sacc[t][1] = sacc[t][2] = sacc[t][3] = 0.f;
#pragma unroll
          for (int kp = 0; kp < KB * KPC; ++kp) {
            const int kb = kp / KPC, kh = kp % KPC;  // feature block of 64, key run kh * KPR
            if (kp % PPS == 0 && !ptx::mbar_wait(&full[cs], cph, abort_flag, p.err)) {
              aborted = true;
              break;
            }
            const uint32_t kt = ptx::smem_u32(stages + static_cast<size_t>(cs) * L.stage) + (kp % PPS) * KPB;
            // A fragments one k-step ahead of the products that use them, so
            // every product finds its operands loaded
            uint32_t af[2][KMT][4];
            auto load_k = [&](int ks, uint32_t (&dst)[KMT][4]) {
#pragma unroll
              for (int t = 0; t < KMT; ++t) {
                const int r = t * 16 + a_row;
                ptx::ldsm_x4(kt + r * 128 + (((ks * 2 + a_hi) ^ (r & 7)) << 4), dst[t]);
              }
            };
            load_k(0, af[0]);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (ks + 1 < 4) load_k(ks + 1, af[(ks + 1) & 1]);
#pragma unroll
              for (int t = 0; t < KMT; ++t)
                ptx::mma_16816<BF>(sacc[kh * KMT + t], af[ks & 1][t], qf[kb * 4 + ks][0], qf[kb * 4 + ks][1]);
            }
            if (kp % PPS == PPS - 1) {
              __syncwarp();  // every lane is done with the stage
              ++consumed;
              if (++cs == S) {
                cs = 0;
                cph ^= 1u;
              }
              issue_next();
            }
          }
          if (aborted) break;

          // ---- online softmax (Knowl 3, log2 units): the running max of a
          // query column is taken on raw scores and scaled once; the scale
          // is folded into the exponent's FMA
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if (t * 16 + lg >= lim) sacc[t][0] = sacc[t][1] = -INFINITY;
            if (t * 16 + lg + 8 >= lim) sacc[t][2] = sacc[t][3] = -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(sacc[t][0], sacc[t][2]));
            mx1 = fmaxf(mx1, fmaxf(sacc[t][1], sacc[t][3]));
          }
#pragma unroll
          for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
          }
          const float sl2 = p.scale_log2;
          const float mn0 = fmaxf(m2[0], mx0 * sl2), mn1 = fmaxf(m2[1], mx1 * sl2);
          const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = ptx::ex2(m2[0] - mu0), al1 = ptx::ex2(m2[1] - mu1);
          m2[0] = mn0;
          m2[1] = mn1;
          float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            const float e0 = ptx::ex2(fmaf(sacc[t][0], sl2, -mu0));
            const float e1 = ptx::ex2(fmaf(sacc[t][1], sl2, -mu1));
            const float e2 = ptx::ex2(fmaf(sacc[t][2], sl2, -mu0));
            const float e3 = ptx::ex2(fmaf(sacc[t][3], sl2, -mu1));
            // P^T row of key t*16 + lg (+8): query columns 2 lq, 2 lq + 1.
            // The row sums add the rounded probabilities the product reads,
            // so o / n stays a weighted mean of V rows.
            const uint32_t w01 = pack2_16<T>(e0, e1), w23 = pack2_16<T>(e2, e3);
            *reinterpret_cast<uint32_t*>(pbuf_b + (t * 16 + lg) * 16 + lq * 4) = w01;
            *reinterpret_cast<uint32_t*>(pbuf_b + (t * 16 + lg + 8) * 16 + lq * 4) = w23;
            if constexpr (kPSplit) {
              const float h0 = lo16<T>(w01), h1 = hi16<T>(w01), h2 = lo16<T>(w23), h3 = hi16<T>(w23);
              const uint32_t r01 = pack2_16<T>(e0 - h0, e1 - h1), r23 = pack2_16<T>(e2 - h2, e3 - h3);
              *reinterpret_cast<uint32_t*>(pbuf_b + C * 16 + (t * 16 + lg) * 16 + lq * 4) = r01;
              *reinterpret_cast<uint32_t*>(pbuf_b + C * 16 + (t * 16 + lg + 8) * 16 + lq * 4) = r23;
              ps0 += (h0 + lo16<T>(r01)) + (h2 + lo16<T>(r23));
              ps1 += (h1 + hi16<T>(r01)) + (h3 + hi16<T>(r23));
            } else {
              ps0 += lo16<T>(w01) + lo16<T>(w23);
              ps1 += hi16<T>(w01) + hi16<T>(w23);
            }
          }
          nl2[0] = nl2[0] * al0 + ps0;
          nl2[1] = nl2[1] * al1 + ps1;
#pragma unroll
          for (int t = 0; t < OMT; ++t) {
            o[t][0] *= al0;
            o[t][1] *= al1;
            o[t][2] *= al0;
            o[t][3] *= al1;
          }
          __syncwarp();  // P^T is written
          // B fragments of P^T (keys x query columns), k-steps of 16 keys:
          // matrices of 8 key rows, transposed on load
          uint32_t pf[MT][2], pfr[kPSplit ? MT : 1][2];  // P (rounded) and, for bf16, its rounded remainder
          auto load_p = [&](uint32_t base, uint32_t (*dst)[2]) {
            if constexpr (MT == 1) {
              ptx::ldsm_x2_trans(base + (lane & 15) * 16, dst[0]);
            } else {
#pragma unroll
              for (int t2 = 0; t2 < MT / 2; ++t2) {
                uint32_t r[4];
                ptx::ldsm_x4_trans(base + (t2 * 32 + lane) * 16, r);
                dst[2 * t2][0] = r[0];
                dst[2 * t2][1] = r[1];
                dst[2 * t2 + 1][0] = r[2];
                dst[2 * t2 + 1][1] = r[3];
              }
            }
          };
          load_p(pb, pf);
          if constexpr (kPSplit) load_p(pb + C * 16, pfr);

          // ---- O^T += V^T P^T over the V^T pieces (VPR feature rows of one
          // key block each: VKS k-steps of 16 keys from key vb * 16 VKS)
          constexpr int VKS = VSW ? 128 / ES / 16 : MT;
          static_assert(VB * VKS == MT, "V^T key blocks");
#pragma unroll
          for (int vp = 0; vp < VB * VG; ++vp) {
            const int vb = vp / VG, vg = vp % VG;
            const int jp = KB * KPC + vp;  // the piece's index in the tile
            if (jp % PPS == 0 && !ptx::mbar_wait(&full[cs], cph, abort_flag, p.err)) {
              aborted = true;
              break;
            }
            const uint32_t vt = ptx::smem_u32(stages + static_cast<size_t>(cs) * L.stage) + (jp % PPS) * VPB;
            uint32_t af[2][VMT][4];
            auto load_v = [&](int ks, uint32_t (&dst)[VMT][4]) {
              const int j = ks * 2 + a_hi;
#pragma unroll
              for (int t = 0; t < VMT; ++t) {
                const int r = t * 16 + a_row;
                ptx::ldsm_x4(vt + (VSW ? r * 128 + ((j ^ (r & 7)) << 4) : cm_off(r, j, VCH)), dst[t]);
              }
            };
            load_v(0, af[0]);
#pragma unroll
            for (int ks = 0; ks < VKS; ++ks) {
              if (ks + 1 < VKS) load_v(ks + 1, af[(ks + 1) & 1]);
#pragma unroll
              for (int t = 0; t < VMT; ++t) {
                ptx::mma_16816<BF>(o[vg * VMT + t], af[ks & 1][t], pf[vb * VKS + ks][0], pf[vb * VKS + ks][1]);
                if constexpr (kPSplit)
                  ptx::mma_16816<BF>(o[vg * VMT + t], af[ks & 1][t], pfr[vb * VKS + ks][0], pfr[vb * VKS + ks][1]);
              }
            }
            if (jp % PPS == PPS - 1) {
              __syncwarp();  // every lane is done with the stage (and with P^T before the next chunk)
              ++consumed;
              if (++cs == S) {
                cs = 0;
                cph ^= 1u;
              }
              issue_next();
            }
          }
        }
        if (aborted) break;

        // ---- item result: lane holds features t*16 + lg (+8) of query
        // columns 2 lq, 2 lq + 1; the row sums are lane-partial until here
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          nl2[0] += __shfl_xor_sync(0xffffffffu, nl2[0], sh);
          nl2[1] += __shfl_xor_sync(0xffffffffu, nl2[1], sh);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = 2 * lq + j;
          if (h < G) {
            if (p.final_mode) {
              const float inv = 1.f / nl2[j];
              const size_t row = (static_cast<size_t>(grp) * p.Hq + kv * p.g + h) * D;
#pragma unroll
              for (int t = 0; t < OMT; ++t) {
                store_out1<T>(p.out, row + t * 16 + lg, o[t][j] * inv, p.out_f32);
                store_out1<T>(p.out, row + t * 16 + lg + 8, o[t][2 + j] * inv, p.out_f32);
              }
            } else {
              const size_t row = static_cast<size_t>(part_base) + h;
              float* po = p.part_o + row * D;
#pragma unroll
              for (int t = 0; t < OMT; ++t) {
                po[t * 16 + lg] = o[t][j];
                po[t * 16 + lg + 8] = o[t][2 + j];
              }
              if (lg == 0) reinterpret_cast<float2*>(p.part_ml)[row] = make_float2(m2[j], nl2[j]);
            }
          }
        }
      } else {
      // o[h][i]: two partial sums (even / odd keys of each 16-byte run) of
      // output feature lane + 32 i, added at the end; packed fp32x2 FMAs
      float m[G], nl[G];
      float2 o[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        nl[h] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[h][i] = make_float2(0.f, 0.f);
      }

      for (int c = 0; c < n_chunks && !aborted; ++c) {
        if ((c & 31) == 0 && c > 0) {  // valid tokens of chunks c .. c+31 (long runs only)
          my_len = c + lane < n_chunks ? p.chunk_len[p.chunks[list_off + c + lane]] : 0;
        }
        int lim = __shfl_sync(0xffffffffu, my_len, c & 31);
        if (p.causal_p0 >= 0) lim = min(lim, p.causal_p0 + grp + 1 - c * C);

        // ---- scores over the K pieces.  Per key four partial sums (feature
        // i mod 4) as two pairs; at four keys per lane and G >= 4 the G * KPL
        // keys give independent FMA chains enough, and one pair (feature i
        // mod 2) keeps the accumulators in registers
        constexpr int NA = (KPL >= 4 && G >= 4) ? 1 : 2;
        float2 acc[G][KPL][NA];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int kk = 0; kk < KPL; ++kk)
#pragma unroll
            for (int a = 0; a < NA; ++a) acc[h][kk][a] = make_float2(0.f, 0.f);
#pragma unroll
        for (int kp = 0; kp < KB * KPC; ++kp) {
          const int kb = kp / KPC, kh = kp % KPC;  // column block, key run: keys kh*KPR + lane + 32 t
          if (!ptx::mbar_wait(&full[cs], cph, abort_flag, p.err)) {
            aborted = true;
            break;
          }
          const uint8_t* kt = stages + static_cast<size_t>(cs) * L.stage;
#pragma unroll 4
          for (int jj = 0; jj < KCH; ++jj) {
#pragma unroll
            for (int t = 0; t < KT; ++t) {
              const int r = KPR >= 32 ? lane + 32 * t : (lane & (KPR - 1));
              float kf[VEC];
              unpack16<T>(*reinterpret_cast<const uint4*>(kt + r * 128 + ((jj ^ (r & 7)) << 4)), kf);
#pragma unroll
              for (int h = 0; h < G; ++h) {
                const float4* qv = reinterpret_cast<const float4*>(qbuf + h * D + kb * (128 / ES) + jj * VEC);
#pragma unroll
                for (int e4 = 0; e4 < VEC / 4; ++e4) {
                  const float4 qq = qv[e4];
                  float2* a = acc[h][kh * KT + t];
                  a[0] = __ffma2_rn(make_float2(qq.x, qq.y), make_float2(kf[4 * e4 + 0], kf[4 * e4 + 1]), a[0]);
                  a[NA - 1] = __ffma2_rn(make_float2(qq.z, qq.w), make_float2(kf[4 * e4 + 2], kf[4 * e4 + 3]), a[NA - 1]);
                }
              }
            }
          }
          __syncwarp();  // every lane is done with the stage
          ++consumed;
          if (++cs == S) {
            cs = 0;
            cph ^= 1u;
          }
          issue_next();
        }
        if (aborted) break;
        float sc[G][KPL];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int kk = 0; kk < KPL; ++kk)
            sc[h][kk] = NA == 2 ? (acc[h][kk][0].x + acc[h][kk][0].y) + (acc[h][kk][NA - 1].x + acc[h][kk][NA - 1].y)
                                : acc[h][kk][0].x + acc[h][kk][0].y;

        // ---- online softmax over the chunk's C keys (Knowl 3, log2 units)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mx = -INFINITY;
#pragma unroll
          for (int kk = 0; kk < KPL; ++kk) {
            if (kk * 32 + lane >= lim) sc[h][kk] = -INFINITY;
            mx = fmaxf(mx, sc[h][kk]);
          }
          const float m_new = fmaxf(m[h], warp_max(mx));
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float alpha = ptx::ex2(m[h] - m_use);
          float ps_ = 0.f;
#pragma unroll
          for (int kk = 0; kk < KPL; ++kk) {
            const float pr = ptx::ex2(sc[h][kk] - m_use);
            ps_ += pr;
            if (C >= 32 || lane < C) pbuf[h * C + kk * 32 + lane] = pr;
          }
          nl[h] = nl[h] * alpha + ps_;
#pragma unroll
          for (int i = 0; i < DPL; ++i) o[h][i] = __fmul2_rn(o[h][i], make_float2(alpha, alpha));
          m[h] = m_new;
        }
        __syncwarp();

        // ---- o += p V over the V^T pieces (VPR feature rows of one key block each)
#pragma unroll
        for (int vp = 0; vp < VB * VG; ++vp) {
          const int vb = vp / VG, vg = vp % VG;  // key block, feature rows vg*VPR + lane + 32 t
          if (!ptx::mbar_wait(&full[cs], cph, abort_flag, p.err)) {
            aborted = true;
            break;
          }
          const uint8_t* vt = stages + static_cast<size_t>(cs) * L.stage;
#pragma unroll 2
          for (int j = 0; j < VCH; ++j) {
            const int key0 = (VSW ? vb * (128 / ES) : 0) + j * VEC;
            float pv[G][VEC];
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float4* pp4 = reinterpret_cast<const float4*>(pbuf + h * C + key0);
#pragma unroll
              for (int e4 = 0; e4 < VEC / 4; ++e4) {
                const float4 t4 = pp4[e4];
                pv[h][4 * e4 + 0] = t4.x;
                pv[h][4 * e4 + 1] = t4.y;
                pv[h][4 * e4 + 2] = t4.z;
                pv[h][4 * e4 + 3] = t4.w;
              }
            }
#pragma unroll
            for (int t = 0; t < VT; ++t) {
              const int r = lane + 32 * t;
              float vf[VEC];
              const uint32_t off = VSW ? r * 128 + ((j ^ (r & 7)) << 4) : cm_off(r, j, VCH);
              unpack16<T>(*reinterpret_cast<const uint4*>(vt + off), vf);
#pragma unroll
              for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int e = 0; e < VEC; e += 2)
                  o[h][vg * VT + t] = __ffma2_rn(make_float2(pv[h][e], pv[h][e + 1]), make_float2(vf[e], vf[e + 1]),
                                                 o[h][vg * VT + t]);
              }
            }
          }
          __syncwarp();  // every lane is done with the stage, and with pbuf before the next chunk rewrites it
          ++consumed;
          if (++cs == S) {
            cs = 0;
            cph ^= 1u;
          }
          issue_next();
        }
      }
      if (aborted) break;

      // ---- item result
      if (p.final_mode) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float inv = 1.f / warp_sum(nl[h]);
          const size_t row = (static_cast<size_t>(grp) * p.Hq + kv * p.g + h) * D;
#pragma unroll
          for (int i = 0; i < DPL; ++i) store_out1<T>(p.out, row + lane + 32 * i, (o[h][i].x + o[h][i].y) * inv, p.out_f32);
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float n = warp_sum(nl[h]);
          const size_t row = static_cast<size_t>(part_base) + h;
          float* po = p.part_o + row * D;
#pragma unroll
          for (int i = 0; i < DPL; ++i) po[lane + 32 * i] = o[h][i].x + o[h][i].y;
          if (lane == 0) reinterpret_cast<float2*>(p.part_ml)[row] = make_float2(m[h], n);
        }
      }
      }  // fp32 consumer
    }
    if (lane == 0) {
      // Let every copy still in flight land before the warp leaves (only
      // after an abort are there any).
      for (uint32_t x = consumed; x < issued; ++x) {
        const int s = static_cast<int>(x % S);
        ptx::mbar_wait(&full[s], (x / S) & 1, nullptr, p.err);
      }
    }
  }
  if (p.pdl) ptx::pdl_wait();  // never complete before the kernel we overlap
}

template <typename T, int D, int G, int C>
cudaError_t launch_simt_t(const AttnParams& p, int grid, cudaStream_t s) {
  if (p.warps_per_cta < 1 || p.warps_per_cta > simt_max_warps(G, sizeof(T))) return cudaErrorInvalidValue;
  const size_t smem = simt_warp_bytes(C, D, G, p.stages, sizeof(T), std::is_same<T, __nv_bfloat16>::value) *
                     p.warps_per_cta;
  auto fn = attn_simt_kernel<T, D, G, C>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((p.warps_per_cta + 1) * 32);
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

// Chunk sizes C0 and C1 at both head dims (each translation unit instantiates
// one pair, so the build compiles the kernel's variants in parallel).
template <typename T, int C0, int C1>
cudaError_t launch_simt_dc(int D, int C, int g, const AttnParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (D == 64 && C == C0) return launch_simt_g<T, 64, C0>(g, p, grid, s);
  if (D == 64 && C == C1) return launch_simt_g<T, 64, C1>(g, p, grid, s);
  if (D == 128 && C == C0) return launch_simt_g<T, 128, C0>(g, p, grid, s);
  if (D == 128 && C == C1) return launch_simt_g<T, 128, C1>(g, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace pst
