// Host side of libpst: the prefix-aware KV cache tree, the chunk pool's free
// list, the table builder, and the C ABI declared in include/pst.h.
//
// ChunkAttention, Knowl 1 (PAKV): a forest of c-token chunks; arrival does a
// prefix lookup and shares matched full chunks, decode appends to the leaf,
// departure prunes and frees chunks nobody uses (device memory is kept).
// Knowl 5: the kernels are driven by flattened chunk -> batch-range tables that
// are rebuilt on the host and copied to the GPU only when the tree changes
// structurally (a chunk is added or freed, a sequence joins or leaves); the
// per-chunk valid length lives on the device and is updated by the scatter
// kernel, so ordinary decode appends need no table copy.
//
// Readings taken where the pages leave a step open:
//   * only full chunks are matched/shared, by equality of all c token ids under
//     an already matched parent; the first such child in creation order wins;
//   * batch order: depth-first preorder from a virtual root, children in
//     creation order, sequences ending at a node (by id) before its children;
//   * a chunk covered by >= min_share live sequences is computed chunk-first;
//   * sequence ids count up from 0 and are never reused.
#include <algorithm>
#include <chrono>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pst.h"
#include "pst_internal.h"

using namespace pst;

namespace pst {
// selftest.cu: one warp waits on an mbarrier nothing arrives on, through the
// kernels' bounded-wait helper; returns the error word and how many lanes gave up.
cudaError_t run_bounded_wait_selftest(int device, int32_t* err_word, int32_t* lanes_gave_up);
}  // namespace pst

namespace {

thread_local std::string g_last_error;

pst_status fail(pst_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                  \
  do {                                                                                  \
    cudaError_t _e = (expr);                                                            \
    if (_e != cudaSuccess) return fail(PST_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)

uint64_t hash_tokens(const int32_t* t, int n) {
  uint64_t h = 1469598103934665603ull;
  for (int i = 0; i < n; ++i) {
    h ^= static_cast<uint32_t>(t[i]);
    h *= 1099511628211ull;
  }
  return h;
}

struct Node {
  int32_t parent = -1;
  int32_t depth = -1;
  int32_t chunk = -1;
  int32_t n_tokens = 0;
  int32_t refs = 0;
  uint64_t hash = 0;  // of the tokens once the chunk is full
  bool live = false;
  std::vector<int32_t> tokens;
  std::vector<int32_t> children;  // creation order
  std::vector<int64_t> ending;     // ids of sequences whose path ends here, ascending
};

struct Seq {
  std::vector<int32_t> path;  // node ids, root to leaf
  int64_t length = 0;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Stream {  // a run of tiles for the CUDA-core kernel: chunks of one list, one KV head, one group
  int32_t chunk_off, n, kv, group;
};

// Partial results, one entry per (batch row, KV head) pair and item that
// covers it.  The rows of one pair end up contiguous in entry order (slot e of
// the pair holds heads kv*g .. kv*g+g-1 at rows e*g ..), so the merge reads
// one contiguous block per pair.  An entry points back at its producer: a
// tensor-core row-index slot (rows of head 0 at tc_rows[pos]) or a CUDA-core
// item (x).
struct Entry {
  int32_t key;  // u * Hkv + kv
  int32_t pos;  // >= 0: index into tc_rows of head 0; < 0: -1 - CUDA-core item index
};

// The table builder's large work arrays, kept by the pool between builds so a
// rebuild reuses their memory instead of allocating (and first touching) it.
struct BuildScratch {
  std::vector<int32_t> chunks, tc_items, simt_items, tc_rows, sorted, moff, fill;
  std::vector<Entry> ents;
  std::vector<Stream> streams, units, ordered;
};

}  // namespace

struct pst_pool {
  pst_config cfg{};
  int device = -1;
  bool host_only = true;
  int es = 2;
  int C = 64, D = 128, g = 1;
  size_t half_bytes = 0, tile_bytes = 0;
  int32_t n_layers = 1;
  size_t layer_bytes = 0;  // one layer's K/V: max_chunks x Hkv tiles
  int n_sm = 1;
  bool use_tc = false;
  float scale_log2 = 0.f;

  // ---- tree
  std::vector<Node> nodes;  // nodes[0] is the virtual root
  std::vector<int32_t> free_nodes;
  std::vector<int32_t> free_chunks;  // LIFO
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_seq = 0;

  // ---- tables
  bool dirty = true;
  int64_t version = 0, rebuild_count = 0;
  double last_rebuild_us = 0;
  std::vector<int64_t> batch;  // live ids in batch order
  std::vector<int32_t> h_tab;
  size_t off_chunks = 0, off_tc = 0, off_tc_cta = 0, off_simt = 0, off_warp = 0, off_moff = 0, off_rows = 0;
  int32_t n_tc_items = 0, n_tc_ctas = 0, n_simt_items = 0, n_simt_warps = 0;
  // Cost model for splitting the SMs between the phases (GB300, 64-token
  // chunks, head size 128): one chunk of one tensor-core item, the fixed cost
  // of an item, one CUDA-core tile when the phases run on split SMs, the
  // DRAM rate one SM of the CUDA-core kernel sustains (query groups of one),
  // and the whole GPU's.
  // SM-split model: chunk-first cost per chunk (plus tc_hbm_us when the item
  // is the first row tile of its run, i.e. its tiles come from DRAM, not L2)
  // and per item; sequence-first bytes per microsecond per SM; DRAM rate
  double tc_chunk_us = 1.1, tc_hbm_us = 0.3, tc_item_us = 1.0, simt_tile_us = 0.75, simt_sm_gbs = 60.0,
         hbm_gbs = 6500.0;
  int32_t simt_unit = 0;      // CUDA-core work-item size in chunks; 0 = automatic
  int32_t simt_max_ctas = 0;  // cap on the CUDA-core grid; 0 = one CTA per SM
  bool simt_first = false;     // launch order of the decode step (see launch_overlapped)
  bool tc_first_forced = false;
  bool simt_first_forced = false;
  int32_t tc_ctas_forced = 0;  // > 0: chunk-first CTAs when both phases run (tuning knob)
  // sequence-first items: about g * T / (simt_unit_div * W) chunks each when
  // every tile they stage is read once (at most kSimtInline; an item's set-up
  // and partial rows grow with g), the last simt_tail * W chunks as
  // single-chunk items.  Measured, us per step, this rule against
  // sqrt(g) * T / (8 W): share4k 96.0 / 98.4, noshare 303.2 / 306.8, the
  // others equal (the same items at g = 4 and for share1k)
  double simt_unit_div = 16.0, simt_tail = 2.0;
  int32_t tc_max_run = 32;  // chunk-first items: at most this many 64-key tiles
  int32_t tc_tiles_forced = 0;  // > 0: chunk-first item length in tiles (tuning knob)
  // chunk-first kernel first: the sequence-first CTAs that start at once take
  // their first items statically (measured 1.5 to 3.4 us per step faster)
  bool tcf_static = true;
  int32_t merge_cap = 0, merge_cap_forced = -1;
  int32_t simt_grid = 0, simt_stages = 3, simt_wpc = 8;
  // sequence-first claims: simt_wpc items each until at most
  // simt_claim_tail * (consumer warps) items are left, then simt_batch_end
  // (simt_batch when set, else chosen at each table build)
  int32_t simt_batch = 0, simt_batch_end = 2;
  double simt_claim_tail = 4.0;
  int64_t n_part_rows = 0, shared_chunks = 0;
  std::vector<int32_t> canon_shared;   // 4 per row
  std::vector<int32_t> canon_entries;  // 2 per entry
  std::vector<int64_t> canon_offsets;  // B + 1
  BuildScratch scratch;                // the table builder's work arrays, reused between builds
  bool canon_valid = false;            // built on demand by pst_export_tables from the last rebuild's
  std::vector<int32_t> tab_ni, tab_nj, tab_preorder;  // batch ranges and node preorder

  // ---- device
  uint8_t* d_pool = nullptr;
  int32_t* d_chunk_len = nullptr;
  int32_t* d_tab = nullptr;
  size_t tab_cap = 0;  // int32 elements
  bool tab_uploaded = false;
  float* d_part_o = nullptr;
  float* d_part_ml = nullptr;
  size_t part_cap = 0;  // rows
  int32_t* d_err = nullptr;
  int32_t* d_sched = nullptr;  // work-claim counter of the CUDA-core kernel
  // d_sched is zero when the next decode starts: every decode's merge kernel
  // clears it at its end; a prefill (no merge) or a failed launch leaves it set
  bool sched_zero = true;
  int32_t* d_pre = nullptr;
  size_t pre_cap = 0;
  // partial rows of a tensor-core prefill block cut along the keys
  float* d_ppart_o = nullptr;
  float* d_ppart_ml = nullptr;
  size_t ppart_cap = 0;  // rows
  bool split_prefill = true;
  // pinned upload staging, two buffers used in turn: an upload waits only for
  // the copy out of the buffer two uploads back, not for the one just issued
  int32_t* h_stage[2] = {nullptr, nullptr};
  size_t stage_cap[2] = {0, 0};
  cudaEvent_t ev_stage[2] = {nullptr, nullptr};
  bool stage_pending[2] = {false, false};
  int stage_next = 0;
  void* d_q = nullptr;
  void* d_out = nullptr;
  size_t qo_cap = 0;  // bytes each
  cudaStream_t aux = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  bool profiling = false;
  cudaEvent_t pev[6] = {};
  bool pran[3] = {false, false, false};
  int32_t last_launches = 0;
  // pst_decode_attention_graph(_layer): the capture stream, and one captured
  // decode step per layer, replayed while the table version and the q / out
  // pointers it was captured with still hold
  cudaStream_t cap_stream = nullptr;
  struct GraphCache {
    cudaGraphExec_t exec = nullptr;
    int64_t version = -1;
    const void* q = nullptr;
    void* out = nullptr;
    int32_t launches = 0;
  };
  std::vector<GraphCache> graphs;
  int64_t graph_captures = 0;
};

namespace {

// =========================================================== tree operations
int32_t new_node(pst_pool* p, int32_t parent) {
  int32_t id;
  if (!p->free_nodes.empty()) {
    id = p->free_nodes.back();
    p->free_nodes.pop_back();
  } else {
    id = static_cast<int32_t>(p->nodes.size());
    p->nodes.emplace_back();
  }
  Node& n = p->nodes[id];
  n = Node();
  n.parent = parent;
  n.depth = p->nodes[parent].depth + 1;
  n.live = true;
  n.chunk = p->free_chunks.back();
  p->free_chunks.pop_back();
  n.tokens.reserve(p->C);
  p->nodes[parent].children.push_back(id);
  return id;
}

void release_node(pst_pool* p, int32_t id) {
  Node& n = p->nodes[id];
  auto& sib = p->nodes[n.parent].children;
  sib.erase(std::find(sib.begin(), sib.end(), id));
  p->free_chunks.push_back(n.chunk);
  n.live = false;
  n.tokens.clear();
  n.tokens.shrink_to_fit();
  n.children.clear();
  n.ending.clear();
  p->free_nodes.push_back(id);
}

int32_t find_full_child(const pst_pool* p, int32_t parent, const int32_t* tok) {
  const uint64_t h = hash_tokens(tok, p->C);
  for (int32_t ch : p->nodes[parent].children) {
    const Node& n = p->nodes[ch];
    if (n.n_tokens == p->C && n.hash == h && std::memcmp(n.tokens.data(), tok, sizeof(int32_t) * p->C) == 0) return ch;
  }
  return -1;
}

// Longest run of existing full chunks matching the leading tokens.
int64_t match_path(const pst_pool* p, const int32_t* tokens, int64_t n, std::vector<int32_t>* path) {
  int32_t cur = 0;
  int64_t pos = 0;
  while (pos + p->C <= n) {
    const int32_t ch = find_full_child(p, cur, tokens + pos);
    if (ch < 0) break;
    if (path) path->push_back(ch);
    cur = ch;
    pos += p->C;
  }
  return pos;
}

void push_token(pst_pool* p, int32_t id, int32_t tok) {
  Node& n = p->nodes[id];
  n.tokens.push_back(tok);
  n.n_tokens++;
  if (n.n_tokens == p->C) n.hash = hash_tokens(n.tokens.data(), p->C);
}

void mark_structural(pst_pool* p) {
  p->dirty = true;
  p->version++;
}

// Launch scatter ops into (or, gathering, out of) one layer's K/V, in batches
// of kScatterMax.
pst_status run_scatter(pst_pool* p, const std::vector<ScatterOp>& ops, const void* k, const void* v,
                       cudaStream_t s, bool gather, int32_t layer = 0) {
  if (p->host_only || ops.empty()) return PST_OK;
  ScatterParams sp;
  sp.k = static_cast<const uint8_t*>(k);
  sp.v = static_cast<const uint8_t*>(v);
  sp.pool = p->d_pool + static_cast<size_t>(layer) * p->layer_bytes;
  sp.chunk_len = p->d_chunk_len;
  sp.Hkv = p->cfg.n_kv_heads;
  for (size_t i = 0; i < ops.size(); i += kScatterMax) {
    const size_t n = std::min<size_t>(kScatterMax, ops.size() - i);
    sp.n_ops = static_cast<int32_t>(n);
    std::memcpy(sp.ops, ops.data() + i, n * sizeof(ScatterOp));
    cudaError_t e = gather ? launch_gather(p->cfg.dtype, p->D, p->C, sp, s) : launch_scatter(p->cfg.dtype, p->D, p->C, sp, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "scatter launch: %s", cudaGetErrorString(e));
  }
  return PST_OK;
}

// The same ops for every layer: k and v hold n_rows source rows per layer,
// layer-major ([n_layers][n_rows][Hkv][D]).  Null k / v: nothing to write
// (the caller writes each layer's rows later with pst_write_kv).
pst_status scatter_layers(pst_pool* p, const std::vector<ScatterOp>& ops, const void* k, const void* v, int64_t n_rows,
                          cudaStream_t s, bool gather = false) {
  if (!k || !v) return PST_OK;
  const size_t lb = static_cast<size_t>(n_rows) * p->cfg.n_kv_heads * p->D * p->es;
  for (int32_t l = 0; l < p->n_layers; ++l) {
    const pst_status st = run_scatter(p, ops, static_cast<const uint8_t*>(k) + l * lb,
                                      static_cast<const uint8_t*>(v) + l * lb, s, gather, l);
    if (st != PST_OK) return st;
  }
  return PST_OK;
}

// ================================================================ tables

pst_status upload(pst_pool* p, int32_t** dbuf, size_t* dcap, const std::vector<int32_t>& src, cudaStream_t s) {
  const size_t n = src.size();
  if (n == 0) return PST_OK;
  if (n > *dcap) {
    if (*dbuf) {
      CUDA_TRY(cudaStreamSynchronize(s));
      CUDA_TRY(cudaFree(*dbuf));
    }
    size_t cap = std::max<size_t>(n * 3 / 2, 4096);
    CUDA_TRY(cudaMalloc(dbuf, cap * sizeof(int32_t)));
    *dcap = cap;
  }
  const int b = p->stage_next;
  p->stage_next ^= 1;
  if (p->stage_pending[b]) {
    CUDA_TRY(cudaEventSynchronize(p->ev_stage[b]));
    p->stage_pending[b] = false;
  }
  if (n > p->stage_cap[b]) {
    if (p->h_stage[b]) CUDA_TRY(cudaFreeHost(p->h_stage[b]));
    size_t cap = std::max<size_t>(n * 3 / 2, 4096);
    CUDA_TRY(cudaMallocHost(&p->h_stage[b], cap * sizeof(int32_t)));
    p->stage_cap[b] = cap;
  }
  std::memcpy(p->h_stage[b], src.data(), n * sizeof(int32_t));
  CUDA_TRY(cudaMemcpyAsync(*dbuf, p->h_stage[b], n * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaEventRecord(p->ev_stage[b], s));
  p->stage_pending[b] = true;
  return PST_OK;
}

// Query rows are fetched with bulk async copies and outputs written with
// 16-byte stores: both buffers must start on a 16-byte boundary.
bool misaligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

// CUDA-core work item (SimtItem): chunk ids inline for runs of up to
// kSimtInline chunks, else the run's offset in the chunk-id list.
void push_simt_item(std::vector<int32_t>& v, const std::vector<int32_t>& ids, int32_t off, int32_t n, int32_t kv,
                    int32_t group0, int32_t part_base) {
  static_assert(kSimtInline == 4, "inline chunk slots");
  int32_t c[kSimtInline] = {0, 0, 0, 0};
  if (n <= kSimtInline) {
    for (int32_t x = 0; x < n; ++x) c[x] = ids[off + x];
  } else {
    c[0] = off;
  }
  v.insert(v.end(), {c[0], c[1], c[2], c[3], n, kv, group0, part_base});
}

void push_item(std::vector<int32_t>& v, const WorkItem& w) {
  const int32_t* x = reinterpret_cast<const int32_t*>(&w);
  v.insert(v.end(), x, x + 8);
}

// Rebuild batch order, canonical tables and the device work tables.
pst_status rebuild(pst_pool* p) {
  const auto t0 = std::chrono::steady_clock::now();
  const int g = p->g, Hkv = p->cfg.n_kv_heads;
  const int min_share = p->cfg.min_share;
  const size_t NN = p->nodes.size();
  std::vector<int32_t> ni(NN, 0), nj(NN, 0);
  std::vector<int32_t> preorder;
  p->batch.clear();
  // iterative DFS from the virtual root
  {
    std::vector<std::pair<int32_t, size_t>> st;
    st.emplace_back(0, 0);
    ni[0] = 0;
    while (!st.empty()) {
      auto& top = st.back();
      const int32_t id = top.first;
      if (top.second == 0) {
        ni[id] = static_cast<int32_t>(p->batch.size());
        if (id != 0) preorder.push_back(id);
        for (int64_t sid : p->nodes[id].ending) p->batch.push_back(sid);
      }
      const auto& ch = p->nodes[id].children;
      if (top.second < ch.size()) {
        const int32_t c = ch[top.second++];
        st.emplace_back(c, 0);
      } else {
        nj[id] = static_cast<int32_t>(p->batch.size());
        st.pop_back();
      }
    }
  }
  const int32_t B = static_cast<int32_t>(p->batch.size());
  auto shared = [&](int32_t id) { return nj[id] - ni[id] >= min_share; };

  // canonical tables: only counted here (pst_export_tables builds them)
  int64_t n_shared = 0;
  for (int32_t id : preorder) n_shared += shared(id) ? 1 : 0;
  p->shared_chunks = n_shared;

  // runs of shared chunks with an identical batch range
  std::vector<int32_t> run_of(NN, -1);
  std::vector<std::vector<int32_t>> runs;  // node ids root->leaf
  for (int32_t id : preorder) {
    if (!shared(id)) continue;
    const int32_t par = p->nodes[id].parent;
    if (par != 0 && run_of[par] >= 0 && ni[par] == ni[id] && nj[par] == nj[id]) {
      run_of[id] = run_of[par];
    } else {
      run_of[id] = static_cast<int32_t>(runs.size());
      runs.emplace_back();
    }
    runs[run_of[id]].push_back(id);
  }

  BuildScratch& sc = p->scratch;
  auto& chunks = sc.chunks;
  auto& tc_items = sc.tc_items;
  auto& simt_items = sc.simt_items;
  auto& ents = sc.ents;      // partial-result entries (see Entry)
  auto& tc_rows = sc.tc_rows;  // tensor-core item row -> partial row
  auto& streams = sc.streams;
  chunks.clear();
  tc_items.clear();
  simt_items.clear();
  ents.clear();
  tc_rows.clear();
  streams.clear();
  std::vector<int32_t> warp_items;

  // ---- phase 1: chunk-first over the runs.  The tensor-core kernel takes
  // chunks as tiles of 64 keys (two per 128-token chunk, a 64-token chunk,
  // two 32- or four 16-token chunks): its costs and item lengths are counted
  // in tiles, tpc per chunk.
  const double tpc = p->use_tc ? p->C / 64.0 : 1.0;
  double p1_iters = 0;
  for (const auto& r : runs) {
    const int32_t id0 = r.front();
    const int64_t rows = static_cast<int64_t>(nj[id0] - ni[id0]) * g;
    p1_iters += static_cast<double>(r.size()) * tpc * Hkv * (p->use_tc ? ceil_div(rows, 128) : (nj[id0] - ni[id0]));
  }
  // chunk-first items: enough of them to cover every SM when the phases run
  // back to back; fewer, longer ones when they share the GPU (in tiles, then
  // chunks)
  const int64_t tiles1 =
      (p->cfg.flags & PST_FLAG_CONCURRENT_PHASES)
          ? 8
          : std::min<int64_t>(p->tc_max_run,
                              std::max<int64_t>(2, static_cast<int64_t>(std::ceil(p1_iters / std::max(1, p->n_sm)))));
  const int64_t split1 =
      std::max<int64_t>(1, static_cast<int64_t>(std::floor((p->tc_tiles_forced > 0 ? p->tc_tiles_forced : tiles1) / tpc)));
  for (const auto& r : runs) {
    const int32_t i = ni[r.front()], j = nj[r.front()];
    const int32_t rows = (j - i) * g;
    const int32_t L = static_cast<int32_t>(r.size());
    const int32_t nsplit = static_cast<int32_t>(ceil_div(L, split1));
    for (int32_t sp = 0; sp < nsplit; ++sp) {
      const int32_t a = static_cast<int32_t>(static_cast<int64_t>(sp) * L / nsplit);
      const int32_t b = static_cast<int32_t>(static_cast<int64_t>(sp + 1) * L / nsplit);
      const int32_t off = static_cast<int32_t>(chunks.size());
      for (int32_t x = a; x < b; ++x) chunks.push_back(p->nodes[r[x]].chunk);
      if (p->use_tc) {
        for (int kv = 0; kv < Hkv; ++kv) {
          for (int32_t r0 = 0; r0 < rows; r0 += 128) {
            WorkItem w{};
            w.chunk_off = off;
            w.n_chunks = b - a;
            w.kv = kv;
            w.group0 = i;
            w.row0 = r0;
            w.n_rows = std::min(128, rows - r0);
            w.part_base = static_cast<int32_t>(tc_rows.size());
            push_item(tc_items, w);
            for (int32_t u = i + r0 / g; u < i + (r0 + w.n_rows) / g; ++u)
              ents.push_back({u * Hkv + kv, static_cast<int32_t>(tc_rows.size()) + (u - i) * g - r0});
            tc_rows.resize(tc_rows.size() + w.n_rows, 0);
          }
        }
      } else {
        for (int32_t u = i; u < j; ++u)
          for (int kv = 0; kv < Hkv; ++kv) streams.push_back({off, b - a, kv, u});
      }
    }
  }
  p->n_tc_items = static_cast<int32_t>(tc_items.size() / 8);

  // ---- phase 2: sequence-first over each sequence's own chunks
  for (int32_t u = 0; u < B; ++u) {
    const Seq& sq = p->seqs[p->batch[u]];
    const int32_t off = static_cast<int32_t>(chunks.size());
    int32_t n = 0;
    for (int32_t id : sq.path) {
      if (shared(id)) continue;
      chunks.push_back(p->nodes[id].chunk);
      ++n;
    }
    if (n == 0) continue;
    for (int kv = 0; kv < Hkv; ++kv) streams.push_back({off, n, kv, u});
  }

  int64_t T = 0;
  for (const auto& st : streams) T += st.n;

  // ---- tensor-core items -> persistent CTAs.  When both phases run at once,
  // each kernel's CTA fills an SM, so the GPU is split: k SMs for the
  // chunk-first kernel, the rest for the sequence-first kernel, k chosen by a
  // simple cost model so both finish together; items go to CTAs longest first.
  std::vector<int32_t> tc_cta_off(1, 0);
  p->n_tc_ctas = 0;
  p->simt_first = false;
  if (p->n_tc_items > 0) {
    const int32_t n = p->n_tc_items;
    const bool concurrent = T > 0 && (p->cfg.flags & PST_FLAG_CONCURRENT_PHASES);
    std::vector<double> cost(n);
    double w_tc = 0;
    for (int32_t x = 0; x < n; ++x) {
      const bool first_tile = tc_items[8 * x + 4] == 0;  // row0: the run's first row tile reads its tiles from DRAM
      cost[x] = std::ceil(tc_items[8 * x + 1] * tpc) * (p->tc_chunk_us + (first_tile ? p->tc_hbm_us : 0.0)) +
                p->tc_item_us;
      w_tc += cost[x];
    }
    const double max_cost = *std::max_element(cost.begin(), cost.end());
    int32_t k = std::min(p->n_sm, n);
    if (!concurrent && T > 0 && p->n_sm > 1) {
      // The sequence-first kernel is launched right behind this one
      // (programmatic dependent launch) and starts on the SMs this kernel
      // leaves free; its CTAs claim work dynamically, so those that start
      // late, on SMs this kernel releases, just take less.  The chunk-first
      // phase is compute-bound, the sequence-first phase DRAM-bound: pick the
      // k that minimises the modelled end time of both (with 20% margin on the
      // chunk-first estimate, fewer SMs on ties).
      const double simt_bytes = static_cast<double>(T) * p->tile_bytes;
      // bytes per microsecond; with fp32 K/V the sequence-first kernel's
      // per-SM rate falls with the query-group size g (its FMAs per byte grow
      // with g); its tensor-core products for 16-bit K/V cover g <= 8 alike
      const double g_exp = p->cfg.dtype == kF32 ? 0.7 : 0.0;
      const double hbm = p->hbm_gbs * 1e3,
                   per_sm = p->simt_sm_gbs * 1e3 / std::pow(static_cast<double>(g), g_exp);
      double best = 1e300;
      for (int32_t kk = 1; kk <= std::min(p->n_sm, n); ++kk) {
        const double t_tc = 1.2 * std::max(w_tc / kk, max_cost);
        const double r = std::min(hbm, (p->n_sm - kk) * per_sm);
        const double done = r * t_tc;
        const double t = done >= simt_bytes ? std::max(t_tc, simt_bytes / r) : t_tc + (simt_bytes - done) / hbm;
        if (t < best * (1.0 - 1e-9)) {
          best = t;
          k = kk;
        }
      }
      if (p->tc_ctas_forced > 0) k = std::min({p->tc_ctas_forced, p->n_sm, n});
      // Sequence-first kernel first when the chunk-first phase is the shorter
      // one (it then waits for the first kernel without holding its SMs long).
      const double t_tc = 1.2 * std::max(w_tc / k, max_cost);
      const double t_simt = simt_bytes / std::min(hbm, std::max(1, p->n_sm - k) * per_sm);
      p->simt_first = k < p->n_sm && ((t_tc <= 1.1 * t_simt && !p->tc_first_forced) || p->simt_first_forced);
    }
    if (concurrent && p->n_sm > 1) {
      const double w_simt = static_cast<double>(T) * p->simt_tile_us;
      k = static_cast<int32_t>(std::lround(p->n_sm * w_tc / (w_tc + w_simt)));
      k = std::max(1, std::min({k, n, p->n_sm - 1}));
    }
    std::vector<int32_t> order(n);
    for (int32_t x = 0; x < n; ++x) order[x] = x;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });
    // each item to the least-loaded CTA, the lowest index among equals: a
    // min-heap on (load, CTA)
    std::vector<std::pair<double, int32_t>> heap(k);
    for (int32_t c = 0; c < k; ++c) heap[c] = {0.0, c};
    std::vector<int32_t> cta_of(n), count(k + 1, 0);
    for (int32_t x : order) {
      std::pop_heap(heap.begin(), heap.end(), std::greater<>());
      auto& top = heap.back();
      cta_of[x] = top.second;
      ++count[top.second + 1];
      top.first += cost[x];
      std::push_heap(heap.begin(), heap.end(), std::greater<>());
    }
    // items grouped by CTA, each CTA's in assignment order
    for (int32_t c = 0; c < k; ++c) count[c + 1] += count[c];
    auto& sorted = sc.sorted;
    sorted.resize(tc_items.size());
    std::vector<int32_t> fill_at(count.begin(), count.end() - 1);
    for (int32_t x : order) {
      const int32_t at = fill_at[cta_of[x]]++;
      std::copy(tc_items.begin() + 8 * x, tc_items.begin() + 8 * x + 8, sorted.begin() + 8 * at);
    }
    for (int32_t c = 0; c < k; ++c) tc_cta_off.push_back(count[c + 1]);
    tc_items.swap(sorted);
    p->n_tc_ctas = k;
  }

  // ---- cut the CUDA-core tile streams into work items that warps claim at
  // run time: items of about g T / (16 W) chunks (W = warps in the grid; see
  // below) and at least 16 KiB, the largest claimed first, and the last ~2W
  // chunks as single-chunk items so the kernel ends evenly.
  const int32_t simt_sms = (p->n_tc_ctas > 0 && (p->cfg.flags & PST_FLAG_CONCURRENT_PHASES))
                               ? std::max(1, p->n_sm - p->n_tc_ctas)
                               : p->n_sm;
  p->simt_grid = static_cast<int32_t>(std::min<int64_t>(simt_sms, std::max<int64_t>(1, ceil_div(T, p->simt_wpc))));
  if (p->simt_max_ctas > 0) p->simt_grid = std::min(p->simt_grid, p->simt_max_ctas);
  p->n_simt_warps = p->simt_grid * p->simt_wpc;
  {
    // W: the warps that stream from the start -- with the chunk-first
    // kernel alongside, those on the SMs it leaves free
    const bool beside_tc = p->n_tc_ctas > 0 && p->n_tc_ctas < p->n_sm;
    const int64_t W =
        static_cast<int64_t>(beside_tc ? std::min(p->simt_grid, p->n_sm - p->n_tc_ctas) : p->simt_grid) * p->simt_wpc;
    // items of at least 16 KiB of K/V, for small chunks (an item's fixed cost
    // against its bytes; measured at d = 64, c = 16: 54 us per step with 16 KiB
    // items, 60 with 8 KiB)
    const int64_t min_unit = ceil_div(int64_t{16384}, static_cast<int64_t>(2) * p->C * p->D * p->es);
    // g T / (16 W) chunks when every tile staged here is read by one item
    // only (the shared chunks on the tensor cores); when shared chunks are
    // streamed here by every sequence that holds them (read again from L2),
    // larger items pay: sqrt(g) T / (8 W) (measured, share1k with no sharing:
    // 67.7 us per step against 76.5 with the first rule)
    const bool read_once = p->use_tc && p->cfg.min_share <= 2;
    const double per_warp = read_once ? static_cast<double>(g) / p->simt_unit_div
                                      : std::sqrt(static_cast<double>(g)) / 8.0;
    const int32_t unit = std::min<int32_t>(
        kSimtInline,
        p->simt_unit > 0 ? p->simt_unit
                         : static_cast<int32_t>(std::max<int64_t>(
                               min_unit, static_cast<int64_t>(static_cast<double>(T) * per_warp / W))));
    // the units, largest first and in stream order among equals: a stable
    // bucket pass (a unit has 1 .. unit <= kSimtInline chunks)
    std::vector<int32_t> of_len(kSimtInline + 2, 0);
    for (const auto& st : streams) {
      of_len[std::min(unit, st.n) + 1] += st.n / unit;
      if (st.n % unit) ++of_len[st.n % unit + 1];
    }
    std::vector<int32_t> at(kSimtInline + 1, 0);  // first slot of each length, longest first
    for (int32_t len = kSimtInline, pos = 0; len >= 1; --len) {
      at[len] = pos;
      pos += of_len[len + 1];
    }
    auto& units = sc.units;
    units.resize(static_cast<size_t>(at[1] + of_len[2]));
    for (const auto& st : streams)
      for (int32_t a = 0; a < st.n; a += unit) {
        const int32_t len = std::min(unit, st.n - a);
        units[at[len]++] = {st.chunk_off + a, len, st.kv, st.group};
      }
    int64_t tail = 0;
    size_t cut = units.size();
    while (cut > 0 && static_cast<double>(tail) < p->simt_tail * W) tail += units[--cut].n;
    auto& ordered = sc.ordered;
    ordered.assign(units.begin(), units.begin() + cut);
    for (size_t x = cut; x < units.size(); ++x)
      for (int32_t a = 0; a < units[x].n; ++a) ordered.push_back({units[x].chunk_off + a, 1, units[x].kv, units[x].group});
    // one entry and one 8-word item per unit, written in place
    const size_t e0 = ents.size(), i0 = simt_items.size() / 8;
    ents.resize(e0 + ordered.size());
    simt_items.resize(8 * (i0 + ordered.size()));
    for (size_t x = 0; x < ordered.size(); ++x) {
      const Stream& un = ordered[x];
      ents[e0 + x] = {un.group * Hkv + un.kv, -1 - static_cast<int32_t>(i0 + x)};
      int32_t* it = simt_items.data() + 8 * (i0 + x);
      for (int32_t c = 0; c < kSimtInline; ++c) it[c] = c < un.n ? chunks[un.chunk_off + c] : 0;
      it[4] = un.n;
      it[5] = un.kv;
      it[6] = un.group;
      it[7] = 0;
    }
    warp_items.assign(1, 0);
    // Claims near the end of the list: two items (fewer items reserved by one
    // CTA, so the warps end together) where that was measured to pay: this
    // kernel's end is the step's end (it runs alone, or first as the longer
    // phase), the last items take a warp at least ~2.7 us each (about two
    // claim round trips, so a claim of two comes back before the warps run
    // out), and the chunk-first kernel holds at most a quarter of the SMs or
    // the query group is 2 or more.  Otherwise one item per consumer warp.
    // (Measured, two against eight, us per step: share1k 52.2 / 53.6,
    // gqa_tree 60.9 / 63.6, d = 128 with c = 16 58.9 / 59.7, noshare
    // 302 / 308; against: d = 64, c = 64 44.0 / 32.6, b = 96 with 64
    // private tokens 39.9 / 34.3, 4096 shared + 512 private tokens 66.6 /
    // 60.6, 1024 + 256 35.9 / 32.9.)  A warp streams at the GPU's DRAM rate
    // shared by the W streaming warps, at most ~110 GB/s per SM.
    const size_t n_tail = std::min(ordered.size(), static_cast<size_t>(p->simt_claim_tail * p->n_simt_warps));
    int64_t tail_chunks = 0;
    for (size_t x = ordered.size() - n_tail; x < ordered.size(); ++x) tail_chunks += ordered[x].n;
    const double tile_bytes = 2.0 * p->C * p->D * p->es;
    const double mean_bytes = n_tail > 0 ? tile_bytes * static_cast<double>(tail_chunks) / n_tail : 0.0;
    const double warp_gbs = std::min(p->hbm_gbs / std::max<int64_t>(1, W), 110.0 / p->simt_wpc);
    const double item_us = mean_bytes / (warp_gbs * 1e3);
    const bool ends_step = p->n_tc_items == 0 || p->simt_first;
    const bool pays = 4 * p->n_tc_ctas <= p->n_sm || g >= 2;
    p->simt_batch_end = (ends_step && pays && item_us >= 2.7) ? 2 : p->simt_wpc;
  }
  p->n_simt_items = static_cast<int32_t>(simt_items.size() / 8);
  p->n_part_rows = static_cast<int64_t>(ents.size()) * g;

  // ---- merge CSR per (batch row, KV head): entry slots in emission order,
  // and each producer told its rows
  auto& moff = sc.moff;
  moff.assign(static_cast<size_t>(B) * Hkv + 1, 0);
  for (const auto& e : ents) moff[e.key + 1]++;
  for (size_t x = 1; x < moff.size(); ++x) moff[x] += moff[x - 1];
  {
    // merge: pairs with up to merge_cap entries stage them in shared memory
    // (G rows of d floats per entry, 4 warps per CTA, at most 64 KiB, and
    // one round of 32 (m, n) pairs)
    int32_t max_ent = 0;
    for (size_t x = 0; x + 1 < moff.size(); ++x) max_ent = std::max(max_ent, moff[x + 1] - moff[x]);
    const int32_t by_smem = static_cast<int32_t>((64 * 1024) / (4 * static_cast<size_t>(g) * p->D * sizeof(float)));
    p->merge_cap = std::min({max_ent, by_smem, 32 / g});
    if (p->merge_cap_forced >= 0) p->merge_cap = std::min(p->merge_cap, p->merge_cap_forced);
  }
  {
    auto& fill = sc.fill;
    fill.assign(moff.begin(), moff.end() - 1);
    for (const auto& e : ents) {
      const int32_t slot = fill[e.key]++;
      if (e.pos >= 0) {
        for (int hg = 0; hg < g; ++hg) tc_rows[e.pos + hg] = slot * g + hg;
      } else {
        simt_items[8 * static_cast<size_t>(-1 - e.pos) + 7] = slot * g;
      }
    }
  }

  // ---- pack the table image
  auto& t = p->h_tab;
  t.clear();
  p->off_chunks = t.size();
  t.insert(t.end(), chunks.begin(), chunks.end());
  while (t.size() % 8) t.push_back(0);  // 32-byte alignment of the item arrays
  p->off_tc = t.size();
  t.insert(t.end(), tc_items.begin(), tc_items.end());
  p->off_tc_cta = t.size();
  t.insert(t.end(), tc_cta_off.begin(), tc_cta_off.end());
  while (t.size() % 4) t.push_back(0);  // SimtItem: 16-byte alignment
  p->off_simt = t.size();
  t.insert(t.end(), simt_items.begin(), simt_items.end());
  p->off_warp = t.size();
  t.insert(t.end(), warp_items.begin(), warp_items.end());
  p->off_moff = t.size();
  t.insert(t.end(), moff.begin(), moff.end());
  p->off_rows = t.size();
  t.insert(t.end(), tc_rows.begin(), tc_rows.end());
  if (t.empty()) t.push_back(0);

  p->tab_ni.swap(ni);
  p->tab_nj.swap(nj);
  p->tab_preorder.swap(preorder);
  p->canon_valid = false;
  p->rebuild_count++;
  p->dirty = false;
  p->tab_uploaded = false;
  p->last_rebuild_us =
      std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
  return PST_OK;
}

// Copy the table image and size the partial buffers, on the decode stream.
pst_status sync_device_tables(pst_pool* p, cudaStream_t s) {
  if (p->tab_uploaded) return PST_OK;
  if (static_cast<size_t>(p->n_part_rows) > p->part_cap) {
    if (p->d_part_o) {
      CUDA_TRY(cudaStreamSynchronize(s));
      CUDA_TRY(cudaFree(p->d_part_o));
      CUDA_TRY(cudaFree(p->d_part_ml));
    }
    const size_t cap = std::max<size_t>(static_cast<size_t>(p->n_part_rows) * 3 / 2, 1024);
    CUDA_TRY(cudaMalloc(&p->d_part_o, cap * p->D * sizeof(float)));
    CUDA_TRY(cudaMalloc(&p->d_part_ml, cap * 2 * sizeof(float)));
    p->part_cap = cap;
  }
  pst_status st = upload(p, &p->d_tab, &p->tab_cap, p->h_tab, s);
  if (st != PST_OK) return st;
  p->tab_uploaded = true;
  return PST_OK;
}

pst_status ensure_tables(const pst_pool* cp) {
  pst_pool* p = const_cast<pst_pool*>(cp);
  if (!p->dirty) return PST_OK;
  return rebuild(p);
}

pst_status need_device(const pst_pool* p) {
  if (!p) return fail(PST_ERR_INVALID, "null pool");
  if (p->host_only) return fail(PST_ERR_STATE, "host-only pool has no device");
  cudaError_t e = cudaSetDevice(p->device);
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
  return PST_OK;
}

// Decode: with the shared chunks on the tensor cores and min_share <= 2,
// every sequence-first tile belongs to one sequence, so each is read once.
int32_t decode_evict_first(const pst_pool* p) { return (p->use_tc && p->cfg.min_share <= 2) ? 1 : 0; }

AttnParams base_params(const pst_pool* p, int32_t layer) {
  AttnParams a{};
  a.pool = p->d_pool + static_cast<size_t>(layer) * p->layer_bytes;
  a.chunk_len = p->d_chunk_len;
  a.Hq = p->cfg.n_q_heads;
  a.Hkv = p->cfg.n_kv_heads;
  a.g = p->g;
  a.chunk_size = p->C;
  a.causal_p0 = -1;
  a.scale_log2 = p->scale_log2;
  a.stages = p->simt_stages;
  a.warps_per_cta = p->simt_wpc;
  a.claim_batch = p->simt_batch > 0 ? p->simt_batch : p->simt_batch_end;
  a.claim_tail = static_cast<int32_t>(std::min<double>(INT32_MAX, p->simt_claim_tail * p->n_simt_warps));
  a.err = p->d_err;
  a.sched = p->d_sched;
  a.merge_cap = p->merge_cap;
  a.out_f32 = (p->cfg.flags & PST_FLAG_F32_OUT) ? 1 : 0;
  return a;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* pst_last_error(void) { return g_last_error.c_str(); }

const char* pst_version(void) { return "pst 0.1 (sm_103a)"; }

pst_status pst_pool_create(const pst_config* cfg, int device, pst_pool** out) {
  g_last_error.clear();
  if (!cfg || !out) return fail(PST_ERR_INVALID, "null argument");
  const pst_config& c = *cfg;
  if (c.n_q_heads < 1 || c.n_kv_heads < 1 || c.n_q_heads % c.n_kv_heads)
    return fail(PST_ERR_INVALID, "n_q_heads must be a positive multiple of n_kv_heads");
  const int g = c.n_q_heads / c.n_kv_heads;
  if (c.dtype < 0 || c.dtype > 2) return fail(PST_ERR_INVALID, "bad dtype %d", c.dtype);
  if (!simt_supported(c.dtype, c.head_dim, g))
    return fail(PST_ERR_INVALID, "unsupported head_dim %d / group %d", c.head_dim, g);
  if (c.chunk_size != 16 && c.chunk_size != 32 && c.chunk_size != 64 && c.chunk_size != 128)
    return fail(PST_ERR_INVALID, "chunk_size must be 16, 32, 64 or 128");
  if (c.max_chunks < 1 || c.max_chunks > (int64_t(1) << 30)) return fail(PST_ERR_INVALID, "bad max_chunks");
  if (c.min_share < 0 || c.max_seqs < 0) return fail(PST_ERR_INVALID, "negative min_share / max_seqs");
  if (c.n_layers < 0 || c.n_layers > 1024) return fail(PST_ERR_INVALID, "n_layers %d outside [0, 1024]", c.n_layers);
  if (device < -1) return fail(PST_ERR_INVALID, "bad device");

  pst_pool* p = new pst_pool();
  p->cfg = c;
  if (p->cfg.min_share == 0) p->cfg.min_share = 2;
  if (p->cfg.max_seqs == 0) p->cfg.max_seqs = 4096;
  p->device = device;
  p->host_only = device < 0;
  p->es = dtype_size(c.dtype);
  p->C = c.chunk_size;
  p->D = c.head_dim;
  p->g = g;
  p->half_bytes = static_cast<size_t>(p->C) * p->D * p->es;
  p->tile_bytes = 2 * p->half_bytes;
  p->n_layers = c.n_layers > 0 ? c.n_layers : 1;
  p->layer_bytes = static_cast<size_t>(c.max_chunks) * c.n_kv_heads * p->tile_bytes;
  p->scale_log2 = static_cast<float>(1.0 / std::log(2.0) / std::sqrt(static_cast<double>(p->D)));
  p->nodes.emplace_back();  // virtual root
  p->nodes[0].live = true;
  p->free_chunks.reserve(c.max_chunks);
  for (int64_t x = c.max_chunks - 1; x >= 0; --x) p->free_chunks.push_back(static_cast<int32_t>(x));

  if (const char* e = std::getenv("PST_TC_CHUNK_US")) p->tc_chunk_us = std::atof(e);
  if (const char* e = std::getenv("PST_TC_HBM_US")) p->tc_hbm_us = std::atof(e);
  if (const char* e = std::getenv("PST_SIMT_TILE_US")) p->simt_tile_us = std::atof(e);
  if (const char* e = std::getenv("PST_TC_ITEM_US")) p->tc_item_us = std::atof(e);
  if (const char* e = std::getenv("PST_SIMT_SM_GBS")) p->simt_sm_gbs = std::atof(e);
  if (const char* e = std::getenv("PST_HBM_GBS")) p->hbm_gbs = std::atof(e);
  if (const char* e = std::getenv("PST_SIMT_UNIT")) p->simt_unit = std::atoi(e);
  if (const char* e = std::getenv("PST_TC_FIRST")) p->tc_first_forced = std::atoi(e) != 0;
  if (const char* e = std::getenv("PST_SIMT_FIRST")) p->simt_first_forced = std::atoi(e) != 0;
  if (const char* e = std::getenv("PST_TC_CTAS")) p->tc_ctas_forced = std::max(0, std::atoi(e));
  if (const char* e = std::getenv("PST_SIMT_UNIT_DIV")) p->simt_unit_div = std::max(0.25, std::atof(e));
  if (const char* e = std::getenv("PST_TC_MAX_RUN")) p->tc_max_run = std::max(2, std::atoi(e));
  if (const char* e = std::getenv("PST_TC_TILES")) p->tc_tiles_forced = std::max(0, std::atoi(e));
  if (const char* e = std::getenv("PST_TCF_STATIC")) p->tcf_static = std::atoi(e) != 0;
  if (const char* e = std::getenv("PST_MERGE_CAP")) p->merge_cap_forced = std::max(0, std::atoi(e));
  if (const char* e = std::getenv("PST_SIMT_TAIL")) p->simt_tail = std::max(0.0, std::atof(e));
  if (const char* e = std::getenv("PST_SPLIT_PREFILL")) p->split_prefill = std::atoi(e) != 0;
  if (const char* e = std::getenv("PST_SIMT_BATCH")) p->simt_batch = std::max(0, std::atoi(e));
  if (const char* e = std::getenv("PST_SIMT_CLAIM_TAIL")) p->simt_claim_tail = std::max(0.0, std::atof(e));
  // Sequence-first kernel shape: up to 8 consumer warps (plus the producer
  // warp) x up to 6 stages of 8 KB pieces, as far as shared memory allows
  p->simt_wpc = attn_simt_max_warps(c.dtype, g);
  // 16-bit K/V with one query row per KV head: two stages keep the DRAM-bound
  // stream fed (fewer bytes in flight, shorter queues); larger groups compute
  // longer per piece and want a deeper ring
  p->simt_stages = (c.dtype != kF32 && g == 1) ? 2 : 6;
  // pieces smaller than 8 KB (chunks of 16 keys, 16-bit V^T rows of 32 keys)
  // keep about the same bytes in flight with proportionally more stages
  p->simt_stages = std::min<int>(16, p->simt_stages * std::max<int>(1, static_cast<int>(8192 / attn_simt_piece_bytes(c.dtype, p->D, p->C))));
  if (const char* e = std::getenv("PST_SIMT_WPC"))
    p->simt_wpc = std::max(1, std::min(attn_simt_max_warps(c.dtype, g), std::atoi(e)));
  if (const char* e = std::getenv("PST_SIMT_STAGES")) p->simt_stages = std::max(2, std::min(16, std::atoi(e)));
  if (const char* e = std::getenv("PST_SIMT_SMS")) p->simt_max_ctas = std::max(1, std::atoi(e));
  // dynamic shared memory per CTA: 227 KiB less the kernel's static part (under 1 KiB)
  while (attn_simt_smem(c.dtype, p->D, p->C, g, p->simt_stages, p->simt_wpc) > 226 * 1024) {
    if (p->simt_stages > 2) p->simt_stages--;
    else p->simt_wpc--;
  }

  if (!p->host_only) {
    auto bail = [&](cudaError_t e, const char* what) {
      pst_status st = fail(PST_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
      pst_pool_free(p);
      return st;
    };
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return bail(e, "cudaSetDevice");
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&p->n_sm, cudaDevAttrMultiProcessorCount, device);
    p->use_tc = major == 10 && tc_supported(c.dtype, p->D, p->C) && !(c.flags & PST_FLAG_NO_TENSOR_CORES);
    const size_t slab = p->layer_bytes * p->n_layers;
    if ((e = cudaMalloc(&p->d_pool, slab)) != cudaSuccess) return bail(e, "cudaMalloc(pool)");
    if ((e = cudaMemset(p->d_pool, 0, slab)) != cudaSuccess) return bail(e, "cudaMemset(pool)");
    if ((e = cudaMalloc(&p->d_chunk_len, sizeof(int32_t) * c.max_chunks)) != cudaSuccess) return bail(e, "cudaMalloc");
    if ((e = cudaMemset(p->d_chunk_len, 0, sizeof(int32_t) * c.max_chunks)) != cudaSuccess) return bail(e, "cudaMemset");
    if ((e = cudaMalloc(&p->d_err, sizeof(int32_t))) != cudaSuccess) return bail(e, "cudaMalloc");
    if ((e = cudaMemset(p->d_err, 0, sizeof(int32_t))) != cudaSuccess) return bail(e, "cudaMemset");
    if ((e = cudaMalloc(&p->d_sched, 256)) != cudaSuccess) return bail(e, "cudaMalloc");
    if ((e = cudaMemset(p->d_sched, 0, 256)) != cudaSuccess) return bail(e, "cudaMemset");
    if ((e = cudaStreamCreateWithFlags(&p->aux, cudaStreamNonBlocking)) != cudaSuccess) return bail(e, "stream");
    if ((e = cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming)) != cudaSuccess) return bail(e, "event");
    if ((e = cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming)) != cudaSuccess) return bail(e, "event");
    for (int b = 0; b < 2; ++b)
      if ((e = cudaEventCreateWithFlags(&p->ev_stage[b], cudaEventDisableTiming)) != cudaSuccess) return bail(e, "event");
    for (auto& ev : p->pev)
      if ((e = cudaEventCreate(&ev)) != cudaSuccess) return bail(e, "event");
    // The fixed area of pst_decode_attention_noalloc belongs to a module of
    // its own, which the CUDA runtime may load lazily, at the first use of one
    // of its symbols.  Looking its address up here commits the area while
    // this call allocates anyway, so the allocation-free call never triggers
    // that load (and its allocation) itself.
    void* scratch = nullptr;
    if ((e = static_scratch_address(device, &scratch)) != cudaSuccess) return bail(e, "cudaGetSymbolAddress(scratch)");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return bail(e, "cudaDeviceSynchronize");
  }
  *out = p;
  return PST_OK;
}

pst_status pst_pool_free(pst_pool* p) {
  if (!p) return fail(PST_ERR_INVALID, "null pool");
  if (!p->host_only) {
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    cudaFree(p->d_pool);
    cudaFree(p->d_chunk_len);
    cudaFree(p->d_tab);
    cudaFree(p->d_part_o);
    cudaFree(p->d_part_ml);
    cudaFree(p->d_err);
    cudaFree(p->d_sched);
    cudaFree(p->d_pre);
    cudaFree(p->d_ppart_o);
    cudaFree(p->d_ppart_ml);
    cudaFree(p->d_q);
    cudaFree(p->d_out);
    for (int b = 0; b < 2; ++b)
      if (p->h_stage[b]) cudaFreeHost(p->h_stage[b]);
    if (p->aux) cudaStreamDestroy(p->aux);
    for (auto& gc : p->graphs)
      if (gc.exec) cudaGraphExecDestroy(gc.exec);
    if (p->cap_stream) cudaStreamDestroy(p->cap_stream);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    for (int b = 0; b < 2; ++b)
      if (p->ev_stage[b]) cudaEventDestroy(p->ev_stage[b]);
    for (auto& ev : p->pev)
      if (ev) cudaEventDestroy(ev);
  }
  delete p;
  return PST_OK;
}

pst_status pst_match(const pst_pool* p, const int32_t* tokens, int64_t n, int64_t* n_matched) {
  if (!p || !n_matched || (n > 0 && !tokens) || n < 0) return fail(PST_ERR_INVALID, "bad argument");
  *n_matched = match_path(p, tokens, n, nullptr);
  return PST_OK;
}

pst_status pst_insert(pst_pool* p, const int32_t* tokens, int64_t n, const void* k, const void* v, void* stream,
                      int64_t* seq_id, int64_t* n_matched) {
  if (!p || !tokens || n < 1 || !seq_id) return fail(PST_ERR_INVALID, "bad argument");
  if (static_cast<int64_t>(p->seqs.size()) >= p->cfg.max_seqs)
    return fail(PST_ERR_OOM, "max_seqs (%d) live sequences", p->cfg.max_seqs);
  std::vector<int32_t> path;
  const int64_t m = match_path(p, tokens, n, &path);
  const int64_t need = ceil_div(n - m, p->C);
  if (need > static_cast<int64_t>(p->free_chunks.size()))
    return fail(PST_ERR_OOM, "pool exhausted: need %lld chunks, %zu free", (long long)need, p->free_chunks.size());
  if (p->host_only ? (k || v) : (!k != !v))
    return fail(p->host_only ? PST_ERR_STATE : PST_ERR_INVALID,
                p->host_only ? "host-only pool takes no K/V" : "k and v must both be given or both be null");
  if (!p->host_only) {
    pst_status st = need_device(p);
    if (st != PST_OK) return st;
  }
  std::vector<ScatterOp> ops;
  int32_t cur = path.empty() ? 0 : path.back();
  for (int64_t pos = m; pos < n; pos += p->C) {
    const int32_t id = new_node(p, cur);
    const int64_t end = std::min<int64_t>(pos + p->C, n);
    for (int64_t x = pos; x < end; ++x) push_token(p, id, tokens[x]);
    ops.push_back({p->nodes[id].chunk, static_cast<int32_t>(pos), 0, static_cast<int32_t>(end - pos), 1});
    path.push_back(id);
    cur = id;
  }
  for (int32_t id : path) p->nodes[id].refs++;
  const int64_t sid = p->next_seq++;
  p->nodes[path.back()].ending.push_back(sid);
  Seq sq;
  sq.path = std::move(path);
  sq.length = n;
  p->seqs.emplace(sid, std::move(sq));
  mark_structural(p);
  *seq_id = sid;
  if (n_matched) *n_matched = m;
  return scatter_layers(p, ops, k, v, n, static_cast<cudaStream_t>(stream));
}

// Apply one appended token to the tree; fills *op with its scatter op.
static void append_one(pst_pool* p, Seq& sq, int64_t sid, int32_t token, ScatterOp* op, int32_t src_row) {
  const int32_t leaf = sq.path.back();
  if (p->nodes[leaf].n_tokens < p->C) {
    const int32_t r = p->nodes[leaf].n_tokens;
    push_token(p, leaf, token);
    *op = {p->nodes[leaf].chunk, src_row, r, r + 1, 0};
  } else {
    const int32_t id = new_node(p, leaf);
    push_token(p, id, token);
    p->nodes[id].refs = 1;
    auto& end = p->nodes[leaf].ending;
    end.erase(std::find(end.begin(), end.end(), sid));
    p->nodes[id].ending.push_back(sid);
    sq.path.push_back(id);
    *op = {p->nodes[id].chunk, src_row, 0, 1, 1};
    mark_structural(p);
  }
  sq.length++;
}

pst_status pst_append(pst_pool* p, int64_t seq_id, int32_t token, const void* k, const void* v, void* stream) {
  return pst_append_batch(p, 1, &seq_id, &token, k, v, stream);
}

pst_status pst_append_batch(pst_pool* p, int64_t n, const int64_t* seq_ids, const int32_t* tokens, const void* k,
                            const void* v, void* stream) {
  if (!p || n < 0 || (n > 0 && (!seq_ids || !tokens))) return fail(PST_ERR_INVALID, "bad argument");
  if (n == 0) return PST_OK;
  if (p->host_only ? (k || v) : (!k != !v)) return fail(PST_ERR_INVALID, "k/v pointers do not match pool kind");
  int64_t need = 0;
  std::vector<int64_t> sorted(seq_ids, seq_ids + n);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
    return fail(PST_ERR_INVALID, "duplicate sequence id in batch append");
  for (int64_t x = 0; x < n; ++x) {
    auto it = p->seqs.find(seq_ids[x]);
    if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_ids[x]);
    if (p->nodes[it->second.path.back()].n_tokens == p->C) ++need;
  }
  if (need > static_cast<int64_t>(p->free_chunks.size())) return fail(PST_ERR_OOM, "pool exhausted on append");
  if (!p->host_only) {
    pst_status st = need_device(p);
    if (st != PST_OK) return st;
  }
  std::vector<ScatterOp> ops(n);
  for (int64_t x = 0; x < n; ++x) append_one(p, p->seqs[seq_ids[x]], seq_ids[x], tokens[x], &ops[x], static_cast<int32_t>(x));
  return scatter_layers(p, ops, k, v, n, static_cast<cudaStream_t>(stream));
}

pst_status pst_remove(pst_pool* p, int64_t seq_id) {
  if (!p) return fail(PST_ERR_INVALID, "null pool");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  Seq& sq = it->second;
  auto& end = p->nodes[sq.path.back()].ending;
  end.erase(std::find(end.begin(), end.end(), seq_id));
  for (int32_t id : sq.path) p->nodes[id].refs--;
  for (auto r = sq.path.rbegin(); r != sq.path.rend(); ++r)
    if (p->nodes[*r].refs == 0) release_node(p, *r);
  p->seqs.erase(it);
  mark_structural(p);
  return PST_OK;
}

pst_status pst_batch_order(const pst_pool* p, int64_t* seq_ids, int64_t cap, int64_t* B) {
  if (!p || !B || cap < 0 || (cap > 0 && !seq_ids)) return fail(PST_ERR_INVALID, "bad argument");
  pst_status st = ensure_tables(p);
  if (st != PST_OK) return st;
  *B = static_cast<int64_t>(p->batch.size());
  for (int64_t x = 0; x < std::min<int64_t>(cap, *B); ++x) seq_ids[x] = p->batch[x];
  return PST_OK;
}

pst_status pst_seq_length(const pst_pool* p, int64_t seq_id, int64_t* n_tokens) {
  if (!p || !n_tokens) return fail(PST_ERR_INVALID, "bad argument");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  *n_tokens = it->second.length;
  return PST_OK;
}

// Launch the decode kernels on one stream, overlapped, each later kernel a
// programmatic dependent that waits at its end for the one before (so the
// merge sees every partial row).  When the chunk-first phase is the shorter
// one: the sequence-first kernel first, on the SMs the chunk-first kernel will
// not use; the chunk-first kernel (its CTAs take the free SMs at once); the
// merge.  Otherwise the chunk-first kernel first and the
// sequence-first kernel behind it on the whole grid (its CTAs start on the
// free SMs at once, each of their warps on one item of the first wave, and on
// the others as chunk-first CTAs leave, claiming every item); the merge.
static pst_status launch_overlapped(pst_pool* p, const AttnParams& a, int32_t B, cudaStream_t s) {
  const bool tc = p->n_tc_items > 0, simt = p->n_simt_items > 0;
  const int32_t grid_a =
      simt ? (tc ? (p->simt_first ? std::min(p->simt_grid, std::max(0, p->n_sm - p->n_tc_ctas)) : 0) : p->simt_grid) : 0;
  // (With the sequence-first kernel first, the chunk-first CTAs hold their SMs
  // until that kernel ends, so a second sequence-first launch could start only
  // when no work is left: there is none.)
  const int32_t grid_b = (simt && grid_a == 0) ? p->simt_grid : 0;
  AttnParams a2 = a;
  a2.items = reinterpret_cast<const WorkItem*>(p->d_tab + p->off_simt);
  a2.n_items = p->n_simt_items;
  bool before = false;  // a kernel of this step is already on the stream
  if (grid_a > 0) {
    a2.pdl = 0;
    // every consumer of this launch starts on one item of the first wave
    a2.first_items = grid_a * p->simt_wpc;
    a2.claim_base = a2.first_items;
    cudaError_t e = launch_attn_simt(p->cfg.dtype, p->D, p->C, p->g, a2, grid_a, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "sequence-first launch: %s", cudaGetErrorString(e));
    p->last_launches++;
    before = true;
  }
  if (tc) {
    AttnParams a1 = a;
    a1.items = reinterpret_cast<const WorkItem*>(p->d_tab + p->off_tc);
    a1.n_items = p->n_tc_items;
    a1.warp_items = p->d_tab + p->off_tc_cta;
    a1.pdl = before ? 1 : 0;
    cudaError_t e = launch_attn_tc(p->cfg.dtype, p->D, p->C, a1, p->n_tc_ctas, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "chunk-first launch: %s", cudaGetErrorString(e));
    p->last_launches++;
    before = true;
  }
  if (grid_b > 0) {
    a2.pdl = before ? 1 : 0;
    // CTAs that find a free SM at once (those the chunk-first kernel leaves)
    // start on one item each of the first wave; the others, which start as
    // chunk-first CTAs leave, claim every item
    a2.first_items = p->tcf_static ? std::min(grid_b, std::max(0, p->n_sm - (tc ? p->n_tc_ctas : 0))) * p->simt_wpc : 0;
    a2.claim_base = a2.first_items;
    cudaError_t e = launch_attn_simt(p->cfg.dtype, p->D, p->C, p->g, a2, grid_b, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "sequence-first launch: %s", cudaGetErrorString(e));
    p->last_launches++;
    before = true;
  }
  AttnParams am = a;
  am.pdl = before ? 1 : 0;
  cudaError_t e = launch_merge(p->cfg.dtype, p->D, am, B, s);
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  p->last_launches++;
  return PST_OK;
}

static pst_status launch_step(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s);
static cudaError_t clear_sched(pst_pool* p, cudaStream_t s);

static pst_status decode_impl(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s) {
  pst_status st = ensure_tables(p);
  if (st != PST_OK) return st;
  p->last_launches = 0;
  p->pran[0] = p->pran[1] = p->pran[2] = false;
  const int32_t B = static_cast<int32_t>(p->batch.size());
  if (B == 0) return PST_OK;
  if (!q || !out) return fail(PST_ERR_INVALID, "null q/out with %d live sequences", B);
  if (misaligned16(q) || misaligned16(out)) return fail(PST_ERR_INVALID, "q and out must be 16-byte aligned");
  st = sync_device_tables(p, s);
  if (st != PST_OK) return st;
  CUDA_TRY(clear_sched(p, s));
  return launch_step(p, layer, q, out, s);
}

// Zero the claim counter on stream s unless it is known to be zero already;
// the decode step about to run leaves it zero (its merge kernel clears it).
static cudaError_t clear_sched(pst_pool* p, cudaStream_t s) {
  if (!p->sched_zero) {
    const cudaError_t e = cudaMemsetAsync(p->d_sched, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
  }
  p->sched_zero = true;
  return cudaSuccess;
}

// The step's device work once the tables are on the device: zero the claim
// counter, launch the attention kernels and the merge on stream s.
static pst_status launch_step_impl(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s);

// A step whose launches all went out leaves the claim counter zero (its
// merge kernel clears it); after a failed launch its state is unknown.
static pst_status launch_step(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s) {
  const pst_status st = launch_step_impl(p, layer, q, out, s);
  p->sched_zero = st == PST_OK;
  return st;
}

static pst_status launch_step_impl(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s) {
  p->last_launches = 0;
  const int32_t B = static_cast<int32_t>(p->batch.size());
  AttnParams a = base_params(p, layer);
  a.q = q;
  a.out = out;
  a.part_o = p->d_part_o;
  a.part_ml = p->d_part_ml;
  a.chunks = p->d_tab + p->off_chunks;
  a.kv_evict_first = decode_evict_first(p);
  a.m_off = p->d_tab + p->off_moff;
  a.row_idx = p->d_tab + p->off_rows;
  const bool fork = p->n_tc_items > 0 && p->n_simt_items > 0 && (p->cfg.flags & PST_FLAG_CONCURRENT_PHASES);
  cudaStream_t s1 = fork ? p->aux : s;
  if (!fork && !p->profiling) return launch_overlapped(p, a, B, s);
  // Profiling (per-phase events between the kernels, so no overlap) or forked
  // phases: chunk-first, then sequence-first on the whole grid, then merge.
  if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[4], s));
  if (fork) {
    CUDA_TRY(cudaEventRecord(p->ev_fork, s));
    CUDA_TRY(cudaStreamWaitEvent(p->aux, p->ev_fork, 0));
  }
  if (p->n_tc_items > 0) {
    AttnParams a1 = a;
    a1.items = reinterpret_cast<const WorkItem*>(p->d_tab + p->off_tc);
    a1.n_items = p->n_tc_items;
    a1.warp_items = p->d_tab + p->off_tc_cta;
    if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[0], s1));
    cudaError_t e = launch_attn_tc(p->cfg.dtype, p->D, p->C, a1, p->n_tc_ctas, s1);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "chunk-first launch: %s", cudaGetErrorString(e));
    if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[1], s1));
    p->pran[0] = true;
    p->last_launches++;
  }
  if (p->n_simt_items > 0) {
    AttnParams a2 = a;
    a2.items = reinterpret_cast<const WorkItem*>(p->d_tab + p->off_simt);
    a2.n_items = p->n_simt_items;
    if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[2], s));
    a2.pdl = (p->n_tc_items > 0 && !fork) ? 1 : 0;
    cudaError_t e = launch_attn_simt(p->cfg.dtype, p->D, p->C, p->g, a2, p->simt_grid, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "sequence-first launch: %s", cudaGetErrorString(e));
    if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[3], s));
    p->pran[1] = true;
    p->last_launches++;
  }
  if (fork) {
    CUDA_TRY(cudaEventRecord(p->ev_join, p->aux));
    CUDA_TRY(cudaStreamWaitEvent(s, p->ev_join, 0));
  }
  {
    AttnParams am = a;
    am.pdl = fork ? 0 : 1;  // right behind the attention kernel(s) on this stream
    cudaError_t e = launch_merge(p->cfg.dtype, p->D, am, B, s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
    p->last_launches++;
  }
  if (p->profiling) {
    CUDA_TRY(cudaEventRecord(p->pev[5], s));
    p->pran[2] = true;
  }
  return PST_OK;
}

pst_status pst_decode_attention(pst_pool* p, const void* q, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  return decode_impl(p, 0, q, out, static_cast<cudaStream_t>(stream));
}

pst_status pst_decode_attention_layer(pst_pool* p, int32_t layer, const void* q, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (layer < 0 || layer >= p->n_layers) return fail(PST_ERR_INVALID, "layer %d outside [0, %d)", layer, p->n_layers);
  return decode_impl(p, layer, q, out, static_cast<cudaStream_t>(stream));
}

static pst_status decode_graph_impl(pst_pool* p, int32_t layer, const void* q, void* out, cudaStream_t s) {
  if (p->profiling) return decode_impl(p, layer, q, out, s);  // per-phase events are not captured
  pst_status st = ensure_tables(p);
  if (st != PST_OK) return st;
  p->pran[0] = p->pran[1] = p->pran[2] = false;
  const int32_t B = static_cast<int32_t>(p->batch.size());
  if (B == 0) {
    p->last_launches = 0;
    return PST_OK;
  }
  if (!q || !out) return fail(PST_ERR_INVALID, "null q/out with %d live sequences", B);
  if (misaligned16(q) || misaligned16(out)) return fail(PST_ERR_INVALID, "q and out must be 16-byte aligned");
  st = sync_device_tables(p, s);  // on the caller's stream, before the graph
  if (st != PST_OK) return st;
  CUDA_TRY(clear_sched(p, s));  // the graph holds no counter reset: the previous step's merge cleared it
  if (p->graphs.size() < static_cast<size_t>(p->n_layers)) p->graphs.resize(p->n_layers);
  auto& gc = p->graphs[layer];
  if (!gc.exec || gc.version != p->version || gc.q != q || gc.out != out) {
    if (!p->cap_stream) CUDA_TRY(cudaStreamCreateWithFlags(&p->cap_stream, cudaStreamNonBlocking));
    if (gc.exec) {
      cudaGraphExecDestroy(gc.exec);
      gc.exec = nullptr;
    }
    CUDA_TRY(cudaStreamBeginCapture(p->cap_stream, cudaStreamCaptureModeRelaxed));
    const pst_status ls = launch_step(p, layer, q, out, p->cap_stream);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(p->cap_stream, &graph);
    if (ls != PST_OK) {
      if (graph) cudaGraphDestroy(graph);
      return ls;
    }
    if (ce != cudaSuccess) return fail(PST_ERR_CUDA, "decode graph capture: %s", cudaGetErrorString(ce));
    const cudaError_t ie = cudaGraphInstantiate(&gc.exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) {
      gc.exec = nullptr;
      return fail(PST_ERR_CUDA, "decode graph instantiate: %s", cudaGetErrorString(ie));
    }
    gc.version = p->version;
    gc.q = q;
    gc.out = out;
    gc.launches = p->last_launches;
    ++p->graph_captures;
  }
  CUDA_TRY(cudaGraphLaunch(gc.exec, s));
  p->last_launches = gc.launches;
  return PST_OK;
}

pst_status pst_decode_attention_graph(pst_pool* p, const void* q, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  return decode_graph_impl(p, 0, q, out, static_cast<cudaStream_t>(stream));
}

pst_status pst_decode_attention_graph_layer(pst_pool* p, int32_t layer, const void* q, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (layer < 0 || layer >= p->n_layers) return fail(PST_ERR_INVALID, "layer %d outside [0, %d)", layer, p->n_layers);
  return decode_graph_impl(p, layer, q, out, static_cast<cudaStream_t>(stream));
}

// Decode attention without any allocation: the partial rows and the work
// counter go to the library's fixed device scratch instead of the pool's own
// buffers.  Only a 4-byte memset and kernel launches on `stream`.
pst_status pst_decode_attention_noalloc(pst_pool* p, const void* q, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (p->dirty || !p->tab_uploaded)
    return fail(PST_ERR_STATE,
                "the chunk tables changed since the last pst_decode_attention; call it once first "
                "(that call may allocate) before using the allocation-free variant");
  const int32_t B = static_cast<int32_t>(p->batch.size());
  if (B == 0) return PST_OK;
  if (!q || !out) return fail(PST_ERR_INVALID, "null q/out with %d live sequences", B);
  if (misaligned16(q) || misaligned16(out)) return fail(PST_ERR_INVALID, "q and out must be 16-byte aligned");
  auto align256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t sched_bytes = 256;  // the CUDA-core kernel's work-claim counter
  const size_t ml_bytes = align256(static_cast<size_t>(p->n_part_rows) * 2 * sizeof(float));
  const size_t o_bytes = static_cast<size_t>(p->n_part_rows) * p->D * sizeof(float);
  const size_t need = sched_bytes + ml_bytes + o_bytes;
  if (need > kStaticScratchBytes)
    return fail(PST_ERR_INVALID, "this batch needs %zu bytes of scratch; the fixed area holds %zu", need,
                kStaticScratchBytes);
  void* base = nullptr;  // resolved by pst_pool_create: no module load happens here
  cudaError_t e = static_scratch_address(p->device, &base);
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  p->pran[0] = p->pran[1] = p->pran[2] = false;  // no per-phase timings for this call
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* b8 = static_cast<uint8_t*>(base);
  AttnParams a = base_params(p, 0);
  a.q = q;
  a.out = out;
  a.sched = reinterpret_cast<int32_t*>(b8);  // must start at zero: cleared below
  a.part_ml = reinterpret_cast<float*>(b8 + sched_bytes);
  a.part_o = reinterpret_cast<float*>(b8 + sched_bytes + ml_bytes);
  CUDA_TRY(cudaMemsetAsync(a.sched, 0, sizeof(int32_t), s));
  a.chunks = p->d_tab + p->off_chunks;
  a.kv_evict_first = decode_evict_first(p);
  a.m_off = p->d_tab + p->off_moff;
  a.row_idx = p->d_tab + p->off_rows;
  p->last_launches = 0;
  return launch_overlapped(p, a, B, s);
}

pst_status pst_decode_attention_host(pst_pool* p, const void* q_host, void* out_host, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (!q_host || !out_host) return fail(PST_ERR_INVALID, "null q/out");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = ensure_tables(p);
  if (st != PST_OK) return st;
  const size_t bytes = p->batch.size() * p->cfg.n_q_heads * p->D * p->es;
  const size_t out_bytes = bytes / p->es * ((p->cfg.flags & PST_FLAG_F32_OUT) ? 4 : p->es);
  if (bytes == 0) return PST_OK;
  if (bytes > p->qo_cap) {
    CUDA_TRY(cudaStreamSynchronize(s));
    cudaFree(p->d_q);
    cudaFree(p->d_out);
    p->d_q = p->d_out = nullptr;
    CUDA_TRY(cudaMalloc(&p->d_q, bytes));
    CUDA_TRY(cudaMalloc(&p->d_out, bytes / p->es * 4));  // room for fp32 rows
    p->qo_cap = bytes;
  }
  CUDA_TRY(cudaMemcpyAsync(p->d_q, q_host, bytes, cudaMemcpyHostToDevice, s));
  // the staging buffers stay put between calls, so the step is replayed from
  // its CUDA graph until the tables change structurally
  st = pst_decode_attention_graph(p, p->d_q, p->d_out, stream);
  if (st != PST_OK) return st;
  CUDA_TRY(cudaMemcpyAsync(out_host, p->d_out, out_bytes, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return PST_OK;
}

// Append a block of W tokens to sequence seq_id (sq): first the free rows of
// its leaf (a partial leaf belongs to one sequence), then new private chunks.
// *out_ops gets one scatter op per chunk touched, source rows 0 .. W-1.  Checks
// the capacity before changing anything.
static pst_status append_block(pst_pool* p, int64_t seq_id, Seq& sq, const int32_t* tokens, int64_t W,
                               std::vector<ScatterOp>* out_ops) {
  const int32_t leaf = sq.path.back();
  const int64_t room = p->C - p->nodes[leaf].n_tokens;
  const int64_t need = ceil_div(std::max<int64_t>(0, W - room), p->C);
  if (need > static_cast<int64_t>(p->free_chunks.size())) return fail(PST_ERR_OOM, "pool exhausted on prefill");
  if (sq.length + W > INT32_MAX / 2) return fail(PST_ERR_INVALID, "sequence too long");
  std::vector<ScatterOp> ops;
  int64_t pos = 0;
  if (room > 0) {
    const int32_t r0 = p->nodes[leaf].n_tokens;
    const int64_t take = std::min<int64_t>(room, W);
    for (int64_t x = 0; x < take; ++x) push_token(p, leaf, tokens[x]);
    ops.push_back({p->nodes[leaf].chunk, 0, r0, static_cast<int32_t>(r0 + take), 0});
    pos = take;
  }
  while (pos < W) {
    const int32_t cur = sq.path.back();
    const int32_t id = new_node(p, cur);
    const int64_t end = std::min<int64_t>(pos + p->C, W);
    for (int64_t x = pos; x < end; ++x) push_token(p, id, tokens[x]);
    p->nodes[id].refs = 1;
    auto& e = p->nodes[cur].ending;
    e.erase(std::find(e.begin(), e.end(), seq_id));
    p->nodes[id].ending.push_back(seq_id);
    sq.path.push_back(id);
    ops.push_back({p->nodes[id].chunk, static_cast<int32_t>(pos), 0, static_cast<int32_t>(end - pos), 1});
    pos = end;
  }
  sq.length += W;
  if (need > 0) mark_structural(p);
  *out_ops = std::move(ops);
  return PST_OK;
}

// Causal attention of the W query rows at positions [p0, p0 + W) of sequence
// sq over its keys [0, p0 + r] in layer `layer` (Chunked Prefill, sections
// 1-2), normalised rows into out.
// Causal attention of a W-row block on the tensor-core kernel.  Items are
// (KV head, 128-row tile) over keys [0, p0 + last token of the tile].  When
// those items are too few to keep the SMs busy, each is cut
// along the keys into pieces of about T / (2 #SMs) 64-key tiles (T: all
// tiles of the block); the pieces write (o, m, n) partial rows, grouped per
// (token, KV head) in key order, and the merge kernel combines them
// (attn_reduce, then O = o / n; ChunkAttention, Knowl 3) into out.  Pieces
// go to CTAs longest first, each to the least-loaded CTA.
static pst_status prefill_attention_tc(pst_pool* p, const AttnParams& base, const std::vector<int32_t>& path_chunks,
                                       int64_t p0, int64_t W, cudaStream_t s) {
  const int g = p->g, Hkv = p->cfg.n_kv_heads, C = p->C;
  const double tpc = C / 64.0;  // 64-key tiles per chunk
  const int64_t rows = W * g;
  struct Tile {
    int32_t kv, r0, n_rows, n_ch, nsplit;
  };
  std::vector<Tile> tiles;
  int64_t T = 0;
  for (int kv = 0; kv < Hkv; ++kv)
    for (int64_t r0 = 0; r0 < rows; r0 += 128) {
      const int32_t n_rows = static_cast<int32_t>(std::min<int64_t>(128, rows - r0));
      const int64_t t_last = (r0 + n_rows - 1) / g;
      const int32_t n_ch = static_cast<int32_t>(ceil_div(p0 + t_last + 1, C));
      tiles.push_back({kv, static_cast<int32_t>(r0), n_rows, n_ch, 1});
      T += static_cast<int64_t>(std::ceil(n_ch * tpc));
    }
  // pieces of about T / (2 #SMs) tiles, at least kMinPiece, when the items
  // would leave at least half of the SMs idle (measured on the GQA tree's
  // prompt: with 128 items on 152 SMs the pieces' partial rows and the merge
  // cost more than the idle SMs; with 32 items cutting them pays)
  constexpr int64_t kMinPiece = 6;
  const int64_t piece = std::max<int64_t>(kMinPiece, ceil_div(T, 2 * std::max(1, p->n_sm)));
  int64_t n_pieces = 0;
  const bool split = p->split_prefill && 2 * static_cast<int64_t>(tiles.size()) <= p->n_sm;
  for (auto& t : tiles) {
    if (split)
      t.nsplit = static_cast<int32_t>(
          std::max<int64_t>(1, std::min<int64_t>(t.n_ch, std::llround(t.n_ch * tpc / static_cast<double>(piece)))));
    n_pieces += t.nsplit;
  }

  // table image: chunk ids, items, per-CTA item ranges, merge CSR
  std::vector<int32_t> tab(path_chunks);
  while (tab.size() % 8) tab.push_back(0);
  const size_t off_items = tab.size();
  std::vector<WorkItem> items;
  items.reserve(n_pieces);
  std::vector<int32_t> moff;
  if (split) {
    moff.assign(static_cast<size_t>(W) * Hkv + 1, 0);
    for (const auto& t : tiles)
      for (int32_t r = 0; r < t.n_rows; r += g) moff[static_cast<size_t>((t.r0 + r) / g) * Hkv + t.kv + 1] = t.nsplit;
    for (size_t x = 1; x < moff.size(); ++x) moff[x] += moff[x - 1];
  }
  for (const auto& t : tiles) {
    for (int32_t sp = 0; sp < t.nsplit; ++sp) {
      const int32_t c0 = static_cast<int32_t>(static_cast<int64_t>(sp) * t.n_ch / t.nsplit);
      const int32_t c1 = static_cast<int32_t>(static_cast<int64_t>(sp + 1) * t.n_ch / t.nsplit);
      WorkItem w{};
      w.chunk_off = c0;
      w.n_chunks = c1 - c0;
      w.kv = t.kv;
      w.group0 = 0;
      w.row0 = t.r0;
      w.n_rows = t.n_rows;
      w.key0 = c0 * C;
      w.part_base = sp;  // partial rows: entry moff[token * Hkv + kv] + sp of each row's pair (the kernel)
      items.push_back(w);
    }
  }
  // pieces to CTAs: longest first, each to the least-loaded CTA
  const int32_t n = static_cast<int32_t>(items.size());
  const int32_t k = std::max<int32_t>(1, std::min<int32_t>(p->n_sm, n));
  std::vector<int32_t> order(n);
  for (int32_t x = 0; x < n; ++x) order[x] = x;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return items[x].n_chunks > items[y].n_chunks; });
  std::vector<std::pair<int64_t, int32_t>> heap(k);
  for (int32_t c = 0; c < k; ++c) heap[c] = {0, c};
  std::vector<int32_t> cta_of(n), count(k + 1, 0);
  for (int32_t x : order) {
    std::pop_heap(heap.begin(), heap.end(), std::greater<>());
    cta_of[x] = heap.back().second;
    heap.back().first += items[x].n_chunks + 2;  // + the item's set-up and write-out, in chunk units
    ++count[heap.back().second + 1];
    std::push_heap(heap.begin(), heap.end(), std::greater<>());
  }
  for (int32_t c = 0; c < k; ++c) count[c + 1] += count[c];
  std::vector<int32_t> at(count.begin(), count.end() - 1);
  std::vector<WorkItem> sorted(n);
  for (int32_t x : order) sorted[at[cta_of[x]]++] = items[x];
  for (const auto& w : sorted) push_item(tab, w);
  const size_t off_warp = tab.size();
  tab.insert(tab.end(), count.begin(), count.end());
  const size_t off_moff = tab.size();
  tab.insert(tab.end(), moff.begin(), moff.end());
  pst_status st = upload(p, &p->d_pre, &p->pre_cap, tab, s);
  if (st != PST_OK) return st;

  AttnParams a = base;
  a.chunks = p->d_pre;
  a.items = reinterpret_cast<const WorkItem*>(p->d_pre + off_items);
  a.n_items = n;
  a.warp_items = p->d_pre + off_warp;
  int32_t merge_cap = 0;
  if (split) {
    const size_t part_rows = static_cast<size_t>(moff.back()) * g;
    if (part_rows > p->ppart_cap) {
      if (p->d_ppart_o) {
        CUDA_TRY(cudaStreamSynchronize(s));
        CUDA_TRY(cudaFree(p->d_ppart_o));
        CUDA_TRY(cudaFree(p->d_ppart_ml));
        p->d_ppart_o = p->d_ppart_ml = nullptr;
        p->ppart_cap = 0;
      }
      const size_t cap = std::max<size_t>(part_rows * 3 / 2, 4096);
      CUDA_TRY(cudaMalloc(&p->d_ppart_o, cap * p->D * sizeof(float)));
      CUDA_TRY(cudaMalloc(&p->d_ppart_ml, cap * 2 * sizeof(float)));
      p->ppart_cap = cap;
    }
    a.final_mode = 0;
    a.part_o = p->d_ppart_o;
    a.part_ml = p->d_ppart_ml;
    a.m_off = p->d_pre + off_moff;
    a.row_idx = nullptr;  // the kernel places each row from m_off and its piece index
    int32_t max_ent = 0;
    for (const auto& t : tiles) max_ent = std::max(max_ent, t.nsplit);
    const int32_t by_smem = static_cast<int32_t>((64 * 1024) / (4 * static_cast<size_t>(g) * p->D * sizeof(float)));
    merge_cap = std::min({max_ent, by_smem, 32 / g});
  }
  if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[0], s));
  cudaError_t e = launch_attn_tc(p->cfg.dtype, p->D, p->C, a, k, s);
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  if (split) {
    AttnParams am = a;
    am.final_mode = 1;
    am.pdl = 1;  // a programmatic dependent of the attention kernel: waits for its partial rows
    am.merge_cap = merge_cap;
    am.sched = nullptr;
    e = launch_merge(p->cfg.dtype, p->D, am, static_cast<int32_t>(W), s);
    if (e != cudaSuccess) return fail(PST_ERR_CUDA, "prefill merge launch: %s", cudaGetErrorString(e));
  }
  if (p->profiling) {
    CUDA_TRY(cudaEventRecord(p->pev[1], s));
    p->pran[0] = true;
  }
  return PST_OK;
}

// Causal attention of the W query rows at positions [p0, p0 + W) of sequence
// sq over its keys [0, p0 + r] in layer `layer` (Chunked Prefill, sections
// 1-2), normalised rows into out.
static pst_status prefill_attention(pst_pool* p, int32_t layer, Seq& sq, int64_t p0, int64_t W, const void* q,
                                    void* out, cudaStream_t s) {
  AttnParams a = base_params(p, layer);
  a.q = q;
  a.out = out;
  a.final_mode = 1;
  a.causal_p0 = static_cast<int32_t>(p0);
  p->pran[0] = p->pran[1] = p->pran[2] = false;
  std::vector<int32_t> path_chunks;
  for (int32_t id : sq.path) path_chunks.push_back(p->nodes[id].chunk);
  if (p->use_tc) return prefill_attention_tc(p, a, path_chunks, p0, W, s);

  // CUDA cores: one item per (token, KV head) over keys [0, p0 + t], one warp each
  std::vector<int32_t> tab(path_chunks);
  while (tab.size() % 8) tab.push_back(0);
  const size_t off_items = tab.size();
  const int g = p->g, Hkv = p->cfg.n_kv_heads;
  int32_t n_items = 0;
  for (int64_t t = 0; t < W; ++t)
    for (int kv = 0; kv < Hkv; ++kv) {
      push_simt_item(tab, path_chunks, 0, static_cast<int32_t>(ceil_div(p0 + t + 1, p->C)), kv, static_cast<int32_t>(t),
                     0);
      ++n_items;
    }
  const size_t off_warp = tab.size();
  const int32_t grid = static_cast<int32_t>(ceil_div(n_items, p->simt_wpc));
  for (int32_t x = 0; x <= n_items; ++x) tab.push_back(x);
  pst_status st = upload(p, &p->d_pre, &p->pre_cap, tab, s);
  if (st != PST_OK) return st;
  a.chunks = p->d_pre;
  a.items = reinterpret_cast<const WorkItem*>(p->d_pre + off_items);
  a.n_items = n_items;
  a.warp_items = p->d_pre + off_warp;
  // with profiling on, the attention kernel alone is timed: phase 1 (pst_phase_times)
  CUDA_TRY(cudaMemsetAsync(p->d_sched, 0, sizeof(int32_t), s));
  if (p->profiling) CUDA_TRY(cudaEventRecord(p->pev[2], s));
  const cudaError_t e = launch_attn_simt(p->cfg.dtype, p->D, p->C, g, a, std::min<int32_t>(grid, p->n_sm), s);
  p->sched_zero = false;  // no merge follows to clear it
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  if (p->profiling) {
    CUDA_TRY(cudaEventRecord(p->pev[3], s));
    p->pran[1] = true;
  }
  return PST_OK;
}


pst_status pst_prefill_attend(pst_pool* p, int64_t seq_id, const int32_t* tokens, int64_t W, const void* q,
                              const void* k_new, const void* v_new, void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (!tokens || W < 1 || !q || !k_new || !v_new || !out) return fail(PST_ERR_INVALID, "bad argument");
  if (misaligned16(q) || misaligned16(out)) return fail(PST_ERR_INVALID, "q and out must be 16-byte aligned");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Seq& sq = it->second;
  const int64_t p0 = sq.length;
  std::vector<ScatterOp> ops;
  st = append_block(p, seq_id, sq, tokens, W, &ops);
  if (st != PST_OK) return st;
  st = scatter_layers(p, ops, k_new, v_new, W, s);
  if (st != PST_OK) return st;
  return prefill_attention(p, 0, sq, p0, W, q, out, s);
}

pst_status pst_extend(pst_pool* p, int64_t seq_id, const int32_t* tokens, int64_t W) {
  if (!p || !tokens || W < 1) return fail(PST_ERR_INVALID, "bad argument");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  std::vector<ScatterOp> ops;
  return append_block(p, seq_id, it->second, tokens, W, &ops);
}

pst_status pst_prefill_attend_layer(pst_pool* p, int32_t layer, int64_t seq_id, int64_t p0, int64_t W, const void* q,
                                    void* out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (layer < 0 || layer >= p->n_layers) return fail(PST_ERR_INVALID, "layer %d outside [0, %d)", layer, p->n_layers);
  if (W < 1 || p0 < 0 || !q || !out) return fail(PST_ERR_INVALID, "bad argument");
  if (misaligned16(q) || misaligned16(out)) return fail(PST_ERR_INVALID, "q and out must be 16-byte aligned");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  if (p0 + W > it->second.length)
    return fail(PST_ERR_INVALID, "rows [%lld, %lld) past the sequence's %lld tokens", (long long)p0,
                (long long)(p0 + W), (long long)it->second.length);
  return prefill_attention(p, layer, it->second, p0, W, q, out, static_cast<cudaStream_t>(stream));
}

pst_status pst_gather_kv(const pst_pool* p, int64_t seq_id, void* k_out, void* v_out, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (!k_out || !v_out) return fail(PST_ERR_INVALID, "null output");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  std::vector<ScatterOp> ops;
  int32_t pos = 0;
  for (int32_t id : it->second.path) {
    const Node& n = p->nodes[id];
    ops.push_back({n.chunk, pos, 0, n.n_tokens, 0});
    pos += n.n_tokens;
  }
  return scatter_layers(const_cast<pst_pool*>(p), ops, k_out, v_out, it->second.length, static_cast<cudaStream_t>(stream),
                        true);
}

pst_status pst_write_kv(pst_pool* p, int32_t layer, int64_t seq_id, int64_t n, const void* k, const void* v,
                        void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (layer < 0 || layer >= p->n_layers) return fail(PST_ERR_INVALID, "layer %d outside [0, %d)", layer, p->n_layers);
  if (!k || !v || n < 1) return fail(PST_ERR_INVALID, "bad argument");
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_id);
  const Seq& sq = it->second;
  if (n > sq.length)
    return fail(PST_ERR_INVALID, "%lld rows for a sequence of %lld tokens", (long long)n, (long long)sq.length);
  // the last n rows: every node but the leaf is full, so node i holds
  // positions [i C, i C + n_tokens); each op runs to its chunk's last row
  // (the chunk's device length is set from it)
  const int64_t pos0 = sq.length - n;
  std::vector<ScatterOp> ops;
  for (int64_t i = pos0 / p->C; i < static_cast<int64_t>(sq.path.size()); ++i) {
    const Node& nd = p->nodes[sq.path[i]];
    if (nd.refs > 1)
      return fail(PST_ERR_STATE,
                  "chunk %lld of the sequence is shared by %d sequences; shared rows are written once, by the "
                  "insert that created them",
                  (long long)i, nd.refs);
    const int32_t r0 = static_cast<int32_t>(std::max<int64_t>(pos0, i * p->C) - i * p->C);
    // a chunk written from its first row also clears the rest of it, as on insert
    ops.push_back({nd.chunk, static_cast<int32_t>(i * p->C + r0 - pos0), r0, nd.n_tokens, r0 == 0 ? 1 : 0});
  }
  return run_scatter(p, ops, k, v, static_cast<cudaStream_t>(stream), false, layer);
}

pst_status pst_write_kv_last(pst_pool* p, int32_t layer, int64_t n, const int64_t* seq_ids, const void* k,
                             const void* v, void* stream) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (layer < 0 || layer >= p->n_layers) return fail(PST_ERR_INVALID, "layer %d outside [0, %d)", layer, p->n_layers);
  if (n < 0 || (n > 0 && (!seq_ids || !k || !v))) return fail(PST_ERR_INVALID, "bad argument");
  std::vector<int64_t> sorted(seq_ids, seq_ids + n);
  std::sort(sorted.begin(), sorted.end());
  if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
    return fail(PST_ERR_INVALID, "duplicate sequence id in batch write");  // one launch: rows must not collide
  std::vector<ScatterOp> ops(n);
  for (int64_t x = 0; x < n; ++x) {
    auto it = p->seqs.find(seq_ids[x]);
    if (it == p->seqs.end()) return fail(PST_ERR_NOT_FOUND, "unknown sequence %lld", (long long)seq_ids[x]);
    const Node& nd = p->nodes[it->second.path.back()];
    if (nd.refs > 1)
      return fail(PST_ERR_STATE, "the last token of sequence %lld lies in a chunk shared with %d sequences",
                  (long long)seq_ids[x], nd.refs);
    const int32_t r = nd.n_tokens - 1;
    // as a decode append: a chunk's first row also clears the rest of it
    ops[x] = {nd.chunk, static_cast<int32_t>(x), r, r + 1, r == 0 ? 1 : 0};
  }
  return run_scatter(p, ops, k, v, static_cast<cudaStream_t>(stream), false, layer);
}

// Canonical (chunk-id free) tables of the last rebuild: per shared chunk in
// preorder (depth, i, j, tokens), per sequence in batch order its path's
// (depth, shared) entries.
static void build_canonical(pst_pool* p) {
  if (p->canon_valid) return;
  const auto& ni = p->tab_ni;
  const auto& nj = p->tab_nj;
  auto shared = [&](int32_t id) { return nj[id] - ni[id] >= p->cfg.min_share; };
  p->canon_shared.clear();
  p->canon_entries.clear();
  p->canon_offsets.assign(1, 0);
  for (int32_t id : p->tab_preorder) {
    if (!shared(id)) continue;
    const Node& n = p->nodes[id];
    p->canon_shared.insert(p->canon_shared.end(), {n.depth, ni[id], nj[id], n.n_tokens});
  }
  for (int64_t sid : p->batch) {
    for (int32_t id : p->seqs[sid].path) {
      p->canon_entries.push_back(p->nodes[id].depth);
      p->canon_entries.push_back(shared(id) ? 1 : 0);
    }
    p->canon_offsets.push_back(static_cast<int64_t>(p->canon_entries.size() / 2));
  }
  p->canon_valid = true;
}

pst_status pst_export_tables(const pst_pool* p, int32_t* shared_rows, int64_t shared_cap, int64_t* n_shared,
                             int32_t* seq_entries, int64_t entries_cap, int64_t* n_entries, int64_t* seq_offsets,
                             int64_t offsets_cap, int64_t* B) {
  if (!p || !n_shared || !n_entries || !B) return fail(PST_ERR_INVALID, "null count pointer");
  pst_status st = ensure_tables(p);
  if (st != PST_OK) return st;
  build_canonical(const_cast<pst_pool*>(p));
  *n_shared = static_cast<int64_t>(p->canon_shared.size() / 4);
  *n_entries = static_cast<int64_t>(p->canon_entries.size() / 2);
  *B = static_cast<int64_t>(p->batch.size());
  if (shared_cap < *n_shared || entries_cap < *n_entries || offsets_cap < *B + 1) {
    if (shared_cap == 0 && entries_cap == 0 && offsets_cap == 0) return PST_OK;
    return fail(PST_ERR_INVALID, "export buffers too small");
  }
  if (*n_shared) std::memcpy(shared_rows, p->canon_shared.data(), p->canon_shared.size() * sizeof(int32_t));
  if (*n_entries) std::memcpy(seq_entries, p->canon_entries.data(), p->canon_entries.size() * sizeof(int32_t));
  std::memcpy(seq_offsets, p->canon_offsets.data(), p->canon_offsets.size() * sizeof(int64_t));
  return PST_OK;
}

pst_status pst_stats(const pst_pool* p, pst_stats_t* o) {
  if (!p || !o) return fail(PST_ERR_INVALID, "bad argument");
  std::memset(o, 0, sizeof(*o));
  o->live_seqs = static_cast<int64_t>(p->seqs.size());
  o->max_chunks = p->cfg.max_chunks;
  o->free_chunks = static_cast<int64_t>(p->free_chunks.size());
  o->used_chunks = o->max_chunks - o->free_chunks;
  int64_t uniq = 0;
  for (size_t i = 1; i < p->nodes.size(); ++i)
    if (p->nodes[i].live) uniq += p->nodes[i].n_tokens;
  o->unique_tokens = uniq;
  for (const auto& kv : p->seqs) o->logical_tokens += kv.second.length;
  o->shared_chunks = p->shared_chunks;
  o->table_version = p->version;
  o->rebuild_count = p->rebuild_count;
  o->last_rebuild_us = p->last_rebuild_us;
  o->phase1_items = p->n_tc_items;
  o->phase2_items = p->n_simt_items;
  o->partial_rows = p->n_part_rows;
  o->graph_captures = p->graph_captures;
  o->phase1_ctas = p->n_tc_ctas;
  o->phase2_ctas = p->n_simt_items > 0 ? p->simt_grid : 0;
  o->simt_first = p->simt_first ? 1 : 0;
  return PST_OK;
}

pst_status pst_set_profiling(pst_pool* p, int enable) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  p->profiling = enable != 0;
  return PST_OK;
}

pst_status pst_phase_times(pst_pool* p, float* ms3) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (!ms3) return fail(PST_ERR_INVALID, "null output");
  if (!p->profiling) return fail(PST_ERR_STATE, "profiling is off");
  for (int i = 0; i < 3; ++i) {
    ms3[i] = 0.f;
    if (!p->pran[i]) continue;
    CUDA_TRY(cudaEventSynchronize(p->pev[2 * i + 1]));
    CUDA_TRY(cudaEventElapsedTime(&ms3[i], p->pev[2 * i], p->pev[2 * i + 1]));
  }
  return PST_OK;
}

pst_status pst_selftest_bounded_wait(int device, int32_t* err_code, int32_t* lanes_gave_up) {
  if (device < 0 || !err_code || !lanes_gave_up) return fail(PST_ERR_INVALID, "bad argument");
  const cudaError_t e = run_bounded_wait_selftest(device, err_code, lanes_gave_up);
  if (e != cudaSuccess) return fail(PST_ERR_CUDA, "bounded-wait self-test: %s", cudaGetErrorString(e));
  return PST_OK;
}

pst_status pst_last_launch_count(const pst_pool* p, int32_t* n) {
  if (!p || !n) return fail(PST_ERR_INVALID, "bad argument");
  *n = p->last_launches;
  return PST_OK;
}

pst_status pst_check_device(pst_pool* p, int32_t* code) {
  pst_status st = need_device(p);
  if (st != PST_OK) return st;
  if (!code) return fail(PST_ERR_INVALID, "null output");
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemcpy(code, p->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(p->d_err, 0, sizeof(int32_t)));
  if (*code) return fail(PST_ERR_DEVICE, "device error word 0x%x", *code);
  return PST_OK;
}

}  // extern "C"
