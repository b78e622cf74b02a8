// Host core of the paged-KV attention library: page allocator, reference
// counts, prefix dedup table, working-set state machine, per-pass slot
// reservation and attention planner, and the C ABI declared in pie_attn.h.
//
// Working-set semantics follow "How Pie thinks", section 4 "Working sets"
// (frozen prefix, writable buffer, fork without copying, dedup of frozen
// pages across requests); the per-pass planning step is the runtime's
// packing of many passes into shared launches ("How Pie thinks", "Batching
// is still the engine's job") and the role of ops.attn.plan_prefill ("Poem
// ops", Operations table).
#include <cudaTypedefs.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/pie_attn.h"
#include "plan.h"

using pie::CopyItem;
using pie::kPageSize;
using pie::WorkItem;

namespace {

// Rows x query-heads per item above which the tensor-core kernel takes the
// item (it tiles 256 of them per CTA); the decode kernel takes up to 64.
constexpr int kDecodeMaxM = 64;
constexpr int kPrefillTileM = 256;
// A shared run (fork / dedup group) of at most this many rows x query heads
// goes to the decode kernel in row tiles of at most kDecodeMaxM, each tile
// reading the run's pages (from L2 after the first): the whole pass then
// stays in one decode launch.  Larger runs take the tensor-core kernel.
constexpr int kDecodeSharedMaxM = 64;
constexpr int kMinSplitPages = 16;

struct DedupKey {
  std::array<int32_t, kPageSize + 1> v;  // predecessor page (-1 at page 0), token ids
  bool operator==(const DedupKey& o) const { return v == o.v; }
};
struct DedupHash {
  size_t operator()(const DedupKey& k) const {
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (int32_t x : k.v) {
      h ^= static_cast<uint32_t>(x);
      h *= 0xBF58476D1CE4E5B9ull;
      h ^= h >> 31;
    }
    return static_cast<size_t>(h);
  }
};

struct WorkingSet {
  std::vector<int32_t> tokens;  // token ids, -1 = unknown
  int32_t n_frozen = 0;
  std::vector<int32_t> pages;
  int32_t n_tokens() const { return static_cast<int32_t>(tokens.size()); }
};

inline int32_t cdiv(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

}  // namespace

struct pie_batch {
  pie_ctx* ctx = nullptr;
  int32_t n_rows = 0;
  std::vector<int32_t> row_pos, row_slot;
  std::vector<WorkItem> dec, pre;  // host copies of the work items
  pie::PlanView view{};
  bool appended_any = false;
};

struct pie_ctx {
  pie_config cfg{};
  pie::Geometry geo{};
  int32_t num_sms = 152;
  bool plan_only = true;
  cudaStream_t stream = nullptr;
  std::string err;

  std::vector<int32_t> free_stack;  // back() = next page to allocate
  std::vector<int32_t> refcount;
  std::unordered_map<DedupKey, int32_t, DedupHash> dedup;
  std::unordered_map<int32_t, DedupKey> page_key;
  std::unordered_map<int32_t, WorkingSet> ws;
  int32_t next_ws = 1;
  std::vector<float> k_scale, v_scale;

  // device buffers owned by the context
  float* d_scales = nullptr;  // [4][L*Hkv]: k_scale, v_scale, 1/k_scale, 1/v_scale
  float* d_rope = nullptr;    // [rope_max_positions][d/2][2] (cos, sin), when rope_theta > 0
  int* d_err = nullptr;       // error bits set by kernels (bounded waits that ran out)
  uint8_t* d_plan = nullptr;
  size_t plan_cap = 0;
  uint8_t* h_plan = nullptr;  // pinned staging
  size_t h_plan_cap = 0;
  cudaEvent_t upload_done = nullptr;
  // a second stream, so a pass's decode items run beside its tensor-core
  // items (fork: side waits on main; join: main waits on side)
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  // the last Q tensor map built, for the Q pointer and row count it covers
  CUtensorMap q_map{};
  const void* q_map_ptr = nullptr;
  int32_t q_map_rows = -1;
  bool upload_pending = false;
  float* d_part = nullptr;  // partial (acc | m,l) results
  size_t part_cap = 0;      // floats
  // per (merged row, query head): parts stored so far, for the decode
  // kernels' own merge; zero between launches (each row's last part resets
  // its counters), cleared again after a failed launch
  int32_t* d_cnt = nullptr;
  size_t cnt_cap = 0;       // counters
  bool cnt_dirty = false;
  int32_t merge_mode = 0;   // pie_ctx_set_merge_mode
  pie_batch* open = nullptr;
  bool fail_next_begin = false;  // self-test: fake a CUDA failure at the plan upload
};

namespace {

// Device pointers the kernels read or write with 16-byte (or 4-byte) vector
// accesses and bulk copies must be aligned to that; null passes (its own
// checks come later).
bool aligned(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0; }

pie_status fail(pie_ctx* c, pie_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return st;
}

pie_status cuda_fail(pie_ctx* c, cudaError_t e, const char* what) {
  return fail(c, PIE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

WorkingSet* find_ws(pie_ctx* c, pie_ws h) {
  auto it = c->ws.find(h);
  return it == c->ws.end() ? nullptr : &it->second;
}

int32_t alloc_page(pie_ctx* c) {
  int32_t p = c->free_stack.back();
  c->free_stack.pop_back();
  c->refcount[p] = 1;
  return p;
}

void release_page(pie_ctx* c, int32_t p) {
  if (--c->refcount[p] == 0) {
    auto it = c->page_key.find(p);
    if (it != c->page_key.end()) {
      c->dedup.erase(it->second);
      c->page_key.erase(it);
    }
    c->free_stack.push_back(p);
  }
}

void release_from(pie_ctx* c, WorkingSet& w, size_t keep) {
  while (w.pages.size() > keep) {
    int32_t p = w.pages.back();
    w.pages.pop_back();
    release_page(c, p);
  }
}

// Grow a device buffer; the stream is synchronised first because work still
// queued may read the old buffer.
template <class T>
pie_status ensure_device(pie_ctx* c, T** buf, size_t* cap, size_t need) {
  if (need <= *cap) return PIE_OK;
  size_t n = std::max(need, *cap + *cap / 2);
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamSynchronize");
  if (*buf) cudaFree(*buf);
  *buf = nullptr;
  *cap = 0;
  e = cudaMalloc(reinterpret_cast<void**>(buf), n * sizeof(T));
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaMalloc");
  *cap = n;
  return PIE_OK;
}

// -------------------------------------------------------------- planner
struct PlanBuilder {
  std::vector<int32_t> page_ids, row_pos, row_slot, row_part_base, row_list, row_merge;
  std::vector<int4> merge_info;
  std::vector<CopyItem> copies;
  std::vector<WorkItem> dec, pre;
};

struct SegInfo {
  int32_t seg, n0, n_new, row0, table_off, n_pages, shared_pages;
};

void split_pages(int32_t n_pages, int32_t chunk, std::vector<std::pair<int32_t, int32_t>>& out) {
  out.clear();
  if (n_pages <= 0) return;
  int32_t n = std::max(1, cdiv(n_pages, chunk));
  for (int32_t i = 0; i < n; ++i) {
    int32_t a = static_cast<int32_t>(static_cast<int64_t>(n_pages) * i / n);
    int32_t b = static_cast<int32_t>(static_cast<int64_t>(n_pages) * (i + 1) / n);
    if (b > a) out.push_back({a, b - a});
  }
}

// A run of pages [p0, p1) that every member segment's table holds: the
// shared item of a fork / dedup group, attended once for all members' rows.
struct SharedRun {
  std::vector<int32_t> members;  // segment indices
  int32_t p0, p1;
};

// Prefix tree over the page tables of the segments that may share: at each
// depth, segments holding the same physical page there form a group; the
// group's run extends while all its members hold the same pages, and the
// group then splits by the page where they part.  A fork of a fork thus
// shares its parent's pages with all its relatives and its own frozen pages
// with its siblings only.  Only pages before every member's new tokens (full
// frozen pages) are shared.  shared_end[i] = pages of segment i covered by
// runs (its private keys start there).
void shared_runs(const std::vector<SegInfo>& segs, const std::vector<int32_t>& page_ids,
                 const std::vector<int32_t>& cand, std::vector<SharedRun>& runs, std::vector<int32_t>& shared_end) {
  auto page_at = [&](int32_t i, int32_t j) { return page_ids[segs[i].table_off + j]; };
  auto full = [&](int32_t i) { return segs[i].n0 / kPageSize; };
  struct Work {
    std::vector<int32_t> members;
    int32_t depth;
  };
  std::vector<Work> stack{{cand, 0}};
  std::vector<int32_t> order;
  std::unordered_map<int32_t, std::vector<int32_t>> by_page;
  while (!stack.empty()) {
    Work w = std::move(stack.back());
    stack.pop_back();
    // partition by the page at `depth`, in order of first appearance
    by_page.clear();
    order.clear();
    for (int32_t i : w.members) {
      if (full(i) <= w.depth) {
        shared_end[i] = w.depth;
        continue;
      }
      auto& v = by_page[page_at(i, w.depth)];
      if (v.empty()) order.push_back(page_at(i, w.depth));
      v.push_back(i);
    }
    std::vector<Work> next;
    for (int32_t pg : order) {
      std::vector<int32_t>& m = by_page[pg];
      if (m.size() < 2) {
        shared_end[m[0]] = w.depth;
        continue;
      }
      int32_t lim = INT32_MAX;
      for (int32_t i : m) lim = std::min(lim, full(i));
      int32_t L = w.depth + 1;
      for (; L < lim; ++L) {
        const int32_t p0 = page_at(m[0], L);
        bool same = true;
        for (int32_t i : m) same = same && page_at(i, L) == p0;
        if (!same) break;
      }
      runs.push_back({m, w.depth, L});
      next.push_back({std::move(m), L});
    }
    // depth-first, in order: a segment's runs come out shallowest first
    for (auto it = next.rbegin(); it != next.rend(); ++it) stack.push_back(std::move(*it));
  }
}

void build_plan(pie_ctx* c, const std::vector<SegInfo>& segs_in, int32_t n_rows, PlanBuilder& pb) {
  const int32_t G = c->geo.hq / c->geo.hkv;
  std::vector<SegInfo> segs = segs_in;
  // Segments of up to one tensor-core row tile (decode rows, speculative
  // drafts) share: a long prefill chunk reads its whole context itself,
  // tile by tile, and sharing would only add partial results for each of
  // its many rows.
  std::vector<int32_t> cand;
  for (size_t i = 0; i < segs.size(); ++i)
    if (static_cast<int64_t>(segs[i].n_new) * G <= kPrefillTileM) cand.push_back(static_cast<int32_t>(i));
  std::vector<SharedRun> runs;
  std::vector<int32_t> shared_end(segs.size(), 0);
  shared_runs(segs, pb.page_ids, cand, runs, shared_end);
  for (size_t i = 0; i < segs.size(); ++i) segs[i].shared_pages = shared_end[i];

  auto run_rows = [&](const SharedRun& r) {
    int64_t rows = 0;
    for (int32_t i : r.members) rows += segs[i].n_new;
    return rows;
  };
  // pages of decode-kernel work, to size the KV splits
  int64_t dec_pages = 0;
  for (auto& r : runs)
    if (run_rows(r) * G <= kDecodeSharedMaxM) dec_pages += (r.p1 - r.p0) * cdiv(run_rows(r) * G, kDecodeMaxM);
  for (auto& s : segs)
    if (static_cast<int64_t>(s.n_new) * G <= kDecodeMaxM) dec_pages += s.n_pages - s.shared_pages;
  // KV splits aim at about 8 decode CTAs per SM for bf16 pages and 16 for
  // e4m3 (measured on the 8B and 70B-FP8 decode batches: 1x and 2x were the
  // best of 0.75x..3x; the e4m3 kernel spends more time per byte converting,
  // and shorter splits keep its long tails off the end of the launch)
  const int64_t per_sm = c->geo.kv_dtype == PIE_KV_E4M3 ? 16 : 8;
  int64_t target_items = std::max<int64_t>(1, static_cast<int64_t>(c->num_sms) * per_sm / c->geo.hkv);
  int32_t chunk = static_cast<int32_t>(std::max<int64_t>(kMinSplitPages, (dec_pages + target_items - 1) / target_items));

  std::vector<int32_t> n_parts(n_rows, 0);
  struct Pending {
    WorkItem it;
    bool decode;
  };
  std::vector<Pending> items;
  std::vector<std::pair<int32_t, int32_t>> sp;

  // shared items first: a member row's parts are numbered along its runs,
  // shallowest first, then its private parts
  std::vector<int32_t> seg_parts(segs.size(), 0);
  for (const SharedRun& g : runs) {
    int32_t rows_off = static_cast<int32_t>(pb.row_list.size());
    for (int32_t i : g.members)
      for (int32_t r = 0; r < segs[i].n_new; ++r) pb.row_list.push_back(segs[i].row0 + r);
    int32_t rows = static_cast<int32_t>(pb.row_list.size()) - rows_off;
    // members whose rows are consecutive batch rows (a fork group's drafts,
    // usually) are addressed through the identity prefix of row_list, so
    // the kernels skip the lookup
    bool consecutive = true;
    for (int32_t r = 1; r < rows && consecutive; ++r)
      consecutive = pb.row_list[rows_off + r] == pb.row_list[rows_off] + r;
    if (consecutive) {
      const int32_t first = pb.row_list[rows_off];
      pb.row_list.resize(rows_off);
      rows_off = first;
    }
    const SegInfo& s0 = segs[g.members[0]];
    const int32_t run = g.p1 - g.p0;
    bool decode = static_cast<int64_t>(rows) * G <= kDecodeSharedMaxM;
    int32_t kv_chunk = chunk;
    int32_t rt_rows = rows;
    if (decode) {
      rt_rows = cdiv(rows, cdiv(static_cast<int64_t>(rows) * G, kDecodeMaxM));
    } else {
      // tensor-core items: rows in balanced tiles of at most one 128-row Q
      // tile (a CTA with one Q tile runs S, softmax and PV of a key tile in
      // about 2500 cycles, two Q tiles take about 4000: for the short runs
      // of a shared prefix the shorter chain wins); keys split so the
      // group's items fill about the SMs, each page still read once per row
      // tile.  At least 4 key tiles (32 pages) per item: shorter splits add
      // start-up and partials, and more CTAs than SMs keep the pass's
      // decode CTAs waiting (fork pass, 4096-token prompt, 32 layers: one
      // Q tile 0.81 ms, two 0.86 ms; 16-page splits with one Q tile 0.96 ms).
      int32_t tiles = cdiv(static_cast<int64_t>(rows) * G, kPrefillTileM / 2);
      rt_rows = cdiv(rows, tiles);
      int64_t want = std::max<int64_t>(1, static_cast<int64_t>(c->num_sms) / (c->geo.hkv * tiles));
      kv_chunk = std::max<int32_t>(32, cdiv(run, want));
    }
    split_pages(run, kv_chunk, sp);
    // every member row takes the run's parts at its own next part indices;
    // the kernels index parts per row (row_part_base[row] + part), so the
    // members of one run must agree on the index: they do, because a run's
    // members share every run before it on their paths
    const int32_t base_part = seg_parts[g.members[0]];
    for (int32_t r0 = 0; r0 < rows; r0 += rt_rows) {
      int32_t nr = std::min(rt_rows, rows - r0);
      for (size_t j = 0; j < sp.size(); ++j) {
        WorkItem it{};
        it.pages_off = s0.table_off + g.p0 + sp[j].first;
        it.n_pages = sp[j].second;
        it.key_base = (g.p0 + sp[j].first) * kPageSize;
        it.n_keys = sp[j].second * kPageSize;
        it.rows_off = rows_off + r0;
        it.n_rows = nr;
        it.direct_rows = consecutive ? 1 : 0;
        it.part = base_part + static_cast<int32_t>(j);
        items.push_back({it, decode});
      }
    }
    for (int32_t i : g.members) {
      seg_parts[i] += static_cast<int32_t>(sp.size());
      for (int32_t r = 0; r < segs[i].n_new; ++r) n_parts[segs[i].row0 + r] += static_cast<int32_t>(sp.size());
    }
  }

  // private items of each segment
  for (size_t si = 0; si < segs.size(); ++si) {
    const SegInfo& s = segs[si];
    int32_t base_part = seg_parts[si];
    int32_t priv = s.n_pages - s.shared_pages;
    if (static_cast<int64_t>(s.n_new) * G <= kDecodeMaxM) {
      split_pages(priv, chunk, sp);
      for (size_t j = 0; j < sp.size(); ++j) {
        WorkItem it{};
        int32_t first = s.shared_pages + sp[j].first;
        it.pages_off = s.table_off + first;
        it.n_pages = sp[j].second;
        it.key_base = first * kPageSize;
        it.n_keys = std::min(sp[j].second * kPageSize, s.n0 + s.n_new - it.key_base);
        it.rows_off = s.row0;  // row_list[0..n_rows) is the identity
        it.n_rows = s.n_new;
        it.direct_rows = 1;
        it.part = base_part + static_cast<int32_t>(j);
        items.push_back({it, true});
      }
      for (int32_t r = 0; r < s.n_new; ++r) n_parts[s.row0 + r] += static_cast<int32_t>(sp.size());
    } else {
      int32_t rt_rows = std::max(1, kPrefillTileM / G);
      for (int32_t r0 = 0; r0 < s.n_new; r0 += rt_rows) {
        int32_t nr = std::min(rt_rows, s.n_new - r0);
        int32_t last_pos = s.n0 + r0 + nr - 1;
        WorkItem it{};
        it.pages_off = s.table_off + s.shared_pages;
        it.key_base = s.shared_pages * kPageSize;
        it.n_pages = cdiv(last_pos + 1, kPageSize) - s.shared_pages;
        it.n_keys = last_pos + 1 - it.key_base;
        it.rows_off = s.row0 + r0;
        it.n_rows = nr;
        it.direct_rows = 1;
        it.part = base_part;
        items.push_back({it, false});
        for (int32_t r = 0; r < nr; ++r) n_parts[s.row0 + r0 + r] += 1;
      }
    }
  }

  // part bases: rows with a single part are written directly
  int32_t total = 0;
  pb.row_part_base.assign(n_rows, -1);
  pb.row_merge.assign(n_rows, -1);
  for (int32_t r = 0; r < n_rows; ++r) {
    if (n_parts[r] >= 2) {
      pb.row_part_base[r] = total;
      pb.row_merge[r] = static_cast<int32_t>(pb.merge_info.size());
      total += n_parts[r];
      pb.merge_info.push_back(make_int4(r, n_parts[r], pb.row_part_base[r], 0));
    }
  }
  for (auto& p : items) {
    int32_t r0 = pb.row_list[p.it.rows_off];
    if (n_parts[r0] < 2) p.it.part = -1;
    (p.decode ? pb.dec : pb.pre).push_back(p.it);
  }
  // longest first, so the tail of each launch is made of short items
  auto longer = [](const WorkItem& a, const WorkItem& b) {
    int64_t ca = static_cast<int64_t>(a.n_pages) * a.n_rows, cb = static_cast<int64_t>(b.n_pages) * b.n_rows;
    if (ca != cb) return ca > cb;
    return a.pages_off < b.pages_off;
  };
  // wide items (more than kDecodeNarrowM rows x heads) first, each kind
  // longest first: the two kinds go to two launches of the decode kernel
  std::stable_sort(pb.dec.begin(), pb.dec.end(), [G](const WorkItem& a, const WorkItem& b) {
    const bool wa = a.n_rows * G > pie::kDecodeNarrowM, wb = b.n_rows * G > pie::kDecodeNarrowM;
    if (wa != wb) return wa;
    return a.n_pages > b.n_pages;
  });
  std::stable_sort(pb.pre.begin(), pb.pre.end(), longer);
}

// What pie_batch_begin changed in the host state, in order: per segment the
// working set's length and page count before the pass (and the shared tail
// page a copy-on-write replaced), and every page taken from the free stack.
struct Undo {
  struct Seg {
    pie_ws ws;
    int32_t n_tokens, n_pages, cow_tail;
  };
  std::vector<Seg> segs;
  std::vector<int32_t> allocated;
};

// Puts the host state back as it was before the reservation: tokens and
// pages dropped, shared tails restored, and the pages returned to the free
// stack in reverse order of allocation, so the stack's order is unchanged.
void undo_reservation(pie_ctx* c, const Undo& u) {
  for (auto it = u.segs.rbegin(); it != u.segs.rend(); ++it) {
    WorkingSet& w = c->ws[it->ws];
    w.tokens.resize(it->n_tokens);
    w.pages.resize(it->n_pages);
    if (it->cow_tail >= 0) {
      w.pages[it->n_tokens / kPageSize] = it->cow_tail;
      c->refcount[it->cow_tail] += 1;
    }
  }
  for (auto it = u.allocated.rbegin(); it != u.allocated.rend(); ++it) {
    c->refcount[*it] = 0;
    c->free_stack.push_back(*it);
  }
}

template <class T>
size_t put(std::vector<uint8_t>& blob, const std::vector<T>& v, size_t align = 16) {
  size_t off = (blob.size() + align - 1) / align * align;
  blob.resize(off + v.size() * sizeof(T));
  if (!v.empty()) std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
  return off;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* pie_last_error(const pie_ctx* c) { return c ? c->err.c_str() : "null context"; }

pie_status pie_ctx_create(const pie_config* cfg, pie_ctx** out) {
  if (!cfg || !out) return PIE_ERR_INVALID;
  *out = nullptr;
  const pie_config& k = *cfg;
  int esize = k.kv_dtype == PIE_KV_BF16 ? 2 : (k.kv_dtype == PIE_KV_E4M3 ? 1 : 0);
  if (k.num_layers <= 0 || k.num_q_heads <= 0 || k.num_kv_heads <= 0 || k.num_pages <= 0 || esize == 0 ||
      k.page_size != kPageSize || k.num_q_heads % k.num_kv_heads)
    return PIE_ERR_INVALID;
  int G = k.num_q_heads / k.num_kv_heads;
  bool dim_ok = (k.kv_dtype == PIE_KV_BF16 && (k.head_dim == 64 || k.head_dim == 128)) ||
                (k.kv_dtype == PIE_KV_E4M3 && k.head_dim == 128);
  if (!dim_ok || G > 64 || (G & (G - 1))) return PIE_ERR_INVALID;
  if ((k.k_pool == nullptr) != (k.v_pool == nullptr)) return PIE_ERR_INVALID;
  if (!aligned(k.k_pool, 16) || !aligned(k.v_pool, 16)) return PIE_ERR_INVALID;
  if (k.kv_dtype == PIE_KV_E4M3 && (!k.k_scale || !k.v_scale)) return PIE_ERR_INVALID;
  if (!(k.logit_softcap >= 0.0f) || !std::isfinite(k.logit_softcap)) return PIE_ERR_INVALID;
  if (!(k.rope_theta >= 0.0f) || !std::isfinite(k.rope_theta)) return PIE_ERR_INVALID;
  if (k.rope_theta > 0.0f && (k.rope_theta <= 1.0f || k.rope_max_positions <= 0)) return PIE_ERR_INVALID;

  auto* c = new pie_ctx();
  c->cfg = k;
  c->geo = {k.num_layers, k.num_q_heads, k.num_kv_heads, k.head_dim, k.num_pages, k.kv_dtype,
            static_cast<int64_t>(kPageSize) * k.head_dim * esize, k.logit_softcap};
  c->plan_only = k.k_pool == nullptr;
  c->stream = static_cast<cudaStream_t>(k.stream);
  c->refcount.assign(k.num_pages, 0);
  c->free_stack.resize(k.num_pages);
  if (k.free_list) {
    std::vector<char> seen(k.num_pages, 0);
    for (int32_t i = 0; i < k.num_pages; ++i) {
      int32_t p = k.free_list[i];
      if (p < 0 || p >= k.num_pages || seen[p]) {
        delete c;
        return PIE_ERR_INVALID;
      }
      seen[p] = 1;
      c->free_stack[k.num_pages - 1 - i] = p;
    }
  } else {
    for (int32_t i = 0; i < k.num_pages; ++i) c->free_stack[k.num_pages - 1 - i] = i;
  }
  const int32_t nsc = k.num_layers * k.num_kv_heads;
  c->k_scale.assign(nsc, 1.0f);
  c->v_scale.assign(nsc, 1.0f);
  if (k.kv_dtype == PIE_KV_E4M3) {
    for (int32_t i = 0; i < nsc; ++i) {
      if (!(k.k_scale[i] > 0.0f) || !(k.v_scale[i] > 0.0f)) {
        delete c;
        return PIE_ERR_INVALID;
      }
      c->k_scale[i] = k.k_scale[i];
      c->v_scale[i] = k.v_scale[i];
    }
  }
  c->cfg.free_list = nullptr;
  c->cfg.k_scale = c->cfg.v_scale = nullptr;
  c->num_sms = k.num_sms > 0 ? k.num_sms : 152;
  if (!c->plan_only) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && k.num_sms <= 0) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
    std::vector<float> sc(4 * nsc);
    for (int32_t i = 0; i < nsc; ++i) {
      sc[i] = c->k_scale[i];
      sc[nsc + i] = c->v_scale[i];
      sc[2 * nsc + i] = 1.0f / c->k_scale[i];
      sc[3 * nsc + i] = 1.0f / c->v_scale[i];
    }
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&c->d_scales), sc.size() * sizeof(float));
    if (e == cudaSuccess) e = cudaMemcpy(c->d_scales, sc.data(), sc.size() * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&c->d_err), sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->upload_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->fork_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->join_ev, cudaEventDisableTiming);
    if (e == cudaSuccess && k.rope_theta > 0.0f) {
      std::vector<float> tab(static_cast<size_t>(k.rope_max_positions) * k.head_dim);
      pie_rope_table(k.rope_theta, k.head_dim, k.rope_max_positions, tab.data());
      e = cudaMalloc(reinterpret_cast<void**>(&c->d_rope), tab.size() * sizeof(float));
      if (e == cudaSuccess) e = cudaMemcpy(c->d_rope, tab.data(), tab.size() * sizeof(float), cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      pie_ctx_destroy(c);
      return PIE_ERR_CUDA;
    }
  }
  *out = c;
  return PIE_OK;
}

pie_status pie_ctx_destroy(pie_ctx* c) {
  if (!c) return PIE_ERR_INVALID;
  if (!c->plan_only) {
    cudaStreamSynchronize(c->stream);
    if (c->d_scales) cudaFree(c->d_scales);
    if (c->d_rope) cudaFree(c->d_rope);
    if (c->d_err) cudaFree(c->d_err);
    if (c->d_plan) cudaFree(c->d_plan);
    if (c->d_part) cudaFree(c->d_part);
    if (c->d_cnt) cudaFree(c->d_cnt);
    if (c->h_plan) cudaFreeHost(c->h_plan);
    if (c->upload_done) cudaEventDestroy(c->upload_done);
    if (c->side) {
      cudaStreamSynchronize(c->side);
      cudaStreamDestroy(c->side);
    }
    if (c->fork_ev) cudaEventDestroy(c->fork_ev);
    if (c->join_ev) cudaEventDestroy(c->join_ev);
  }
  delete c->open;
  delete c;
  return PIE_OK;
}

pie_status pie_ws_create(pie_ctx* c, pie_ws* out) {
  if (!c || !out) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  *out = c->next_ws++;
  c->ws.emplace(*out, WorkingSet{});
  return PIE_OK;
}

pie_status pie_ws_destroy(pie_ctx* c, pie_ws h) {
  if (!c) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  WorkingSet* w = find_ws(c, h);
  if (!w) return fail(c, PIE_ERR_BAD_HANDLE, "no working set %d", h);
  release_from(c, *w, 0);
  c->ws.erase(h);
  return PIE_OK;
}

pie_status pie_ws_fork(pie_ctx* c, pie_ws parent, pie_ws* child) {
  if (!c || !child) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  WorkingSet* p = find_ws(c, parent);
  if (!p) return fail(c, PIE_ERR_BAD_HANDLE, "no working set %d", parent);
  WorkingSet w;
  w.n_frozen = p->n_frozen;
  w.tokens.assign(p->tokens.begin(), p->tokens.begin() + p->n_frozen);
  w.pages.assign(p->pages.begin(), p->pages.begin() + cdiv(p->n_frozen, kPageSize));
  for (int32_t pg : w.pages) c->refcount[pg] += 1;
  *child = c->next_ws++;
  c->ws.emplace(*child, std::move(w));
  return PIE_OK;
}

pie_status pie_ws_freeze(pie_ctx* c, pie_ws h, int32_t n) {
  if (!c) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  WorkingSet* w = find_ws(c, h);
  if (!w) return fail(c, PIE_ERR_BAD_HANDLE, "no working set %d", h);
  int32_t writable = w->n_tokens() - w->n_frozen;
  if (n < 0) n = writable;
  if (n > writable) return fail(c, PIE_ERR_RANGE, "freeze %d > %d writable tokens", n, writable);
  int32_t old_full = w->n_frozen / kPageSize;
  w->n_frozen += n;
  for (int32_t i = old_full; i < w->n_frozen / kPageSize; ++i) {
    int32_t page = w->pages[i];
    if (c->page_key.count(page)) continue;
    DedupKey key;
    bool known = true;
    for (int32_t j = 0; j < kPageSize; ++j) {
      key.v[1 + j] = w->tokens[i * kPageSize + j];
      known = known && key.v[1 + j] >= 0;
    }
    if (!known) continue;
    key.v[0] = i == 0 ? -1 : w->pages[i - 1];
    if (i > 0 && !c->page_key.count(key.v[0])) continue;
    if (c->dedup.count(key)) continue;
    c->dedup.emplace(key, page);
    c->page_key.emplace(page, key);
  }
  return PIE_OK;
}

pie_status pie_ws_rollback(pie_ctx* c, pie_ws h, int32_t n) {
  if (!c) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  WorkingSet* w = find_ws(c, h);
  if (!w) return fail(c, PIE_ERR_BAD_HANDLE, "no working set %d", h);
  if (n < 0 || n > w->n_tokens() - w->n_frozen)
    return fail(c, PIE_ERR_RANGE, "rollback %d > %d writable tokens", n, w->n_tokens() - w->n_frozen);
  w->tokens.resize(w->tokens.size() - n);
  release_from(c, *w, cdiv(w->n_tokens(), kPageSize));
  return PIE_OK;
}

pie_status pie_ws_match_prefix(pie_ctx* c, pie_ws h, const int32_t* toks, int32_t n, int32_t* n_reused) {
  if (!c || n < 0 || (n > 0 && !toks)) return PIE_ERR_INVALID;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is open");
  WorkingSet* w = find_ws(c, h);
  if (!w) return fail(c, PIE_ERR_BAD_HANDLE, "no working set %d", h);
  if (w->n_tokens()) return fail(c, PIE_ERR_STATE, "match_prefix needs an empty working set");
  int32_t parent = -1, matched = 0;
  while ((matched + 1) * kPageSize <= n) {
    DedupKey key;
    key.v[0] = parent;
    for (int32_t j = 0; j < kPageSize; ++j) key.v[1 + j] = toks[matched * kPageSize + j];
    auto it = c->dedup.find(key);
    if (it == c->dedup.end()) break;
    w->pages.push_back(it->second);
    c->refcount[it->second] += 1;
    parent = it->second;
    ++matched;
  }
  w->tokens.assign(toks, toks + matched * kPageSize);
  w->n_frozen = matched * kPageSize;
  if (n_reused) *n_reused = matched * kPageSize;
  return PIE_OK;
}

pie_status pie_ws_info(const pie_ctx* c, pie_ws h, int32_t* nt, int32_t* nf, int32_t* np) {
  if (!c) return PIE_ERR_INVALID;
  auto it = c->ws.find(h);
  if (it == c->ws.end()) return PIE_ERR_BAD_HANDLE;
  if (nt) *nt = it->second.n_tokens();
  if (nf) *nf = it->second.n_frozen;
  if (np) *np = static_cast<int32_t>(it->second.pages.size());
  return PIE_OK;
}

pie_status pie_ws_page_table(const pie_ctx* c, pie_ws h, int32_t* out, int32_t cap, int32_t* n) {
  if (!c) return PIE_ERR_INVALID;
  auto it = c->ws.find(h);
  if (it == c->ws.end()) return PIE_ERR_BAD_HANDLE;
  const auto& p = it->second.pages;
  int32_t m = std::min<int32_t>(cap, static_cast<int32_t>(p.size()));
  if (out && m > 0) std::memcpy(out, p.data(), m * sizeof(int32_t));
  if (n) *n = static_cast<int32_t>(p.size());
  return PIE_OK;
}

pie_status pie_page_refcount(const pie_ctx* c, int32_t page, int32_t* rc) {
  if (!c || !rc || page < 0 || page >= c->geo.num_pages) return PIE_ERR_INVALID;
  *rc = c->refcount[page];
  return PIE_OK;
}

pie_status pie_free_pages(const pie_ctx* c, int32_t* n) {
  if (!c || !n) return PIE_ERR_INVALID;
  *n = static_cast<int32_t>(c->free_stack.size());
  return PIE_OK;
}

pie_status pie_batch_begin(pie_ctx* c, const pie_seg* segs, int32_t n_segs, pie_batch** out) {
  if (!c || !out || n_segs < 0 || (n_segs > 0 && !segs)) return PIE_ERR_INVALID;
  *out = nullptr;
  if (c->open) return fail(c, PIE_ERR_STATE, "a batch is already open");
  // validate and count pages, touching nothing
  std::unordered_set<int32_t> seen;
  int64_t need = 0, n_rows = 0;
  for (int32_t i = 0; i < n_segs; ++i) {
    const pie_seg& s = segs[i];
    WorkingSet* w = find_ws(c, s.ws);
    if (!w) return fail(c, PIE_ERR_BAD_HANDLE, "segment %d: no working set %d", i, s.ws);
    if (!seen.insert(s.ws).second) return fail(c, PIE_ERR_INVALID, "working set %d twice in one pass", s.ws);
    if (s.n_new < 0) return fail(c, PIE_ERR_INVALID, "segment %d: n_new < 0", i);
    if (s.n_new == 0) continue;
    int32_t n0 = w->n_tokens();
    need += cdiv(static_cast<int64_t>(n0) + s.n_new, kPageSize) - cdiv(n0, kPageSize);
    if (n0 % kPageSize && c->refcount[w->pages[n0 / kPageSize]] > 1) need += 1;
    n_rows += s.n_new;
  }
  if (need > static_cast<int64_t>(c->free_stack.size()))
    return fail(c, PIE_ERR_NO_PAGES, "pass needs %lld pages, %zu free", static_cast<long long>(need),
                c->free_stack.size());
  if (n_rows > INT32_MAX / 2) return fail(c, PIE_ERR_INVALID, "too many rows");

  // reserve slots; `undo` records what changes, so that a failure further
  // down (a CUDA call) can put the host state back as it was
  auto* b = new pie_batch();
  b->ctx = c;
  b->n_rows = static_cast<int32_t>(n_rows);
  PlanBuilder pb;
  std::vector<SegInfo> infos;
  Undo undo;
  b->row_pos.reserve(n_rows);
  b->row_slot.reserve(n_rows);
  for (int32_t i = 0; i < n_segs; ++i) {
    const pie_seg& s = segs[i];
    if (s.n_new == 0) continue;
    WorkingSet& w = c->ws[s.ws];
    int32_t n0 = w.n_tokens();
    undo.segs.push_back({s.ws, n0, static_cast<int32_t>(w.pages.size()), -1});
    if (n0 % kPageSize) {
      int32_t tail = w.pages[n0 / kPageSize];
      if (c->refcount[tail] > 1) {
        int32_t fresh = alloc_page(c);
        undo.allocated.push_back(fresh);
        c->refcount[tail] -= 1;
        w.pages[n0 / kPageSize] = fresh;
        pb.copies.push_back({tail, fresh});
        undo.segs.back().cow_tail = tail;
      }
    }
    SegInfo si{};
    si.seg = i;
    si.n0 = n0;
    si.n_new = s.n_new;
    si.row0 = static_cast<int32_t>(b->row_pos.size());
    for (int32_t t = 0; t < s.n_new; ++t) {
      int32_t pos = n0 + t;
      if (pos % kPageSize == 0) {
        w.pages.push_back(alloc_page(c));
        undo.allocated.push_back(w.pages.back());
      }
      b->row_pos.push_back(pos);
      b->row_slot.push_back(w.pages[pos / kPageSize] * kPageSize + pos % kPageSize);
    }
    for (int32_t t = 0; t < s.n_new; ++t) w.tokens.push_back(s.token_ids ? s.token_ids[t] : -1);
    si.table_off = static_cast<int32_t>(pb.page_ids.size());
    si.n_pages = static_cast<int32_t>(w.pages.size());
    pb.page_ids.insert(pb.page_ids.end(), w.pages.begin(), w.pages.end());
    infos.push_back(si);
  }
  pb.row_list.resize(n_rows);
  for (int32_t r = 0; r < n_rows; ++r) pb.row_list[r] = r;
  build_plan(c, infos, b->n_rows, pb);
  pb.row_pos = b->row_pos;
  pb.row_slot = b->row_slot;
  b->dec = pb.dec;
  b->pre = pb.pre;

  // lay out and upload
  std::vector<uint8_t> blob;
  size_t o_pages = put(blob, pb.page_ids), o_pos = put(blob, pb.row_pos), o_slot = put(blob, pb.row_slot);
  size_t o_base = put(blob, pb.row_part_base), o_list = put(blob, pb.row_list);
  size_t o_mi = put(blob, pb.merge_info), o_rm = put(blob, pb.row_merge);
  size_t o_cp = put(blob, pb.copies), o_dec = put(blob, pb.dec, 32), o_pre = put(blob, pb.pre, 32);
  int64_t total_parts = 0;
  for (const int4& mi : pb.merge_info) total_parts += mi.y;

  pie::PlanView& v = b->view;
  v.n_rows = b->n_rows;
  v.n_dec = static_cast<int32_t>(pb.dec.size());
  v.n_pre = static_cast<int32_t>(pb.pre.size());
  v.n_merge = static_cast<int32_t>(pb.merge_info.size());
  v.n_copies = static_cast<int32_t>(pb.copies.size());
  v.max_dec_m = 0;
  v.n_dec_wide = 0;
  for (const WorkItem& it : pb.dec) {
    const int32_t m = it.n_rows * (c->geo.hq / c->geo.hkv);
    v.max_dec_m = std::max(v.max_dec_m, m);
    v.n_dec_wide += m > pie::kDecodeNarrowM;
  }
  // Merge mode 1: the decode kernels merge split rows themselves when every
  // part comes from a decode item (the tensor-core kernel does not count its
  // parts); otherwise, and by default, a merge launch follows.
  bool fused_merge = v.n_merge > 0 && !c->plan_only && c->merge_mode == 1;
  for (const WorkItem& it : pb.pre) fused_merge = fused_merge && it.part < 0;
  if (c->fail_next_begin) {
    c->fail_next_begin = false;
    undo_reservation(c, undo);
    delete b;
    return fail(c, PIE_ERR_CUDA, "plan upload: failure injected by pie_selftest_fail_next_begin");
  }
  if (!c->plan_only && !blob.empty()) {
    pie_status st = ensure_device(c, &c->d_plan, &c->plan_cap, blob.size());
    size_t part_need = static_cast<size_t>(total_parts) * c->geo.hq * (c->geo.d + 2);
    if (st == PIE_OK) st = ensure_device(c, &c->d_part, &c->part_cap, std::max<size_t>(part_need, 1));
    const size_t cnt_need = static_cast<size_t>(v.n_merge) * c->geo.hq;
    if (st == PIE_OK && fused_merge && cnt_need > c->cnt_cap) {
      st = ensure_device(c, &c->d_cnt, &c->cnt_cap, cnt_need);
      c->cnt_dirty = true;  // a new buffer is not zeroed yet
    }
    if (st == PIE_OK && fused_merge && c->cnt_dirty) {
      cudaError_t e = cudaMemsetAsync(c->d_cnt, 0, c->cnt_cap * sizeof(int32_t), c->stream);
      if (e != cudaSuccess) st = cuda_fail(c, e, "cudaMemsetAsync");
      else c->cnt_dirty = false;
    }
    if (st == PIE_OK && c->upload_pending) {
      cudaError_t e = cudaEventSynchronize(c->upload_done);
      if (e != cudaSuccess) st = cuda_fail(c, e, "cudaEventSynchronize");
      c->upload_pending = false;
    }
    if (st == PIE_OK && blob.size() > c->h_plan_cap) {
      if (c->h_plan) cudaFreeHost(c->h_plan);
      c->h_plan = nullptr;
      c->h_plan_cap = 0;
      size_t n = std::max(blob.size(), c->h_plan_cap + c->h_plan_cap / 2);
      cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&c->h_plan), n);
      if (e != cudaSuccess) st = cuda_fail(c, e, "cudaMallocHost");
      else c->h_plan_cap = n;
    }
    if (st == PIE_OK) {
      std::memcpy(c->h_plan, blob.data(), blob.size());
      cudaError_t e = cudaMemcpyAsync(c->d_plan, c->h_plan, blob.size(), cudaMemcpyHostToDevice, c->stream);
      if (e == cudaSuccess) e = cudaEventRecord(c->upload_done, c->stream);
      if (e != cudaSuccess) st = cuda_fail(c, e, "plan upload");
      c->upload_pending = e == cudaSuccess;
    }
    if (st != PIE_OK) {
      undo_reservation(c, undo);
      delete b;
      return st;
    }
    uint8_t* d = c->d_plan;
    v.page_ids = reinterpret_cast<const int32_t*>(d + o_pages);
    v.row_pos = reinterpret_cast<const int32_t*>(d + o_pos);
    v.row_slot = reinterpret_cast<const int32_t*>(d + o_slot);
    v.row_part_base = reinterpret_cast<const int32_t*>(d + o_base);
    v.row_list = reinterpret_cast<const int32_t*>(d + o_list);
    v.merge_info = reinterpret_cast<const int4*>(d + o_mi);
    v.row_merge = reinterpret_cast<const int32_t*>(d + o_rm);
    v.merge_cnt = fused_merge ? c->d_cnt : nullptr;
    v.copies = reinterpret_cast<const CopyItem*>(d + o_cp);
    v.dec_items = reinterpret_cast<const WorkItem*>(d + o_dec);
    v.pre_items = reinterpret_cast<const WorkItem*>(d + o_pre);
    if (v.n_copies) {
      cudaError_t e = pie::launch_page_copy(c->geo, v, c->cfg.k_pool, c->cfg.v_pool, c->stream);
      if (e != cudaSuccess) {
        // The plan upload is enqueued, but nothing reads it before the next
        // pie_batch_begin, which waits for it (upload_pending).
        undo_reservation(c, undo);
        delete b;
        return cuda_fail(c, e, "page copy launch");
      }
    }
  }
  c->open = b;
  *out = b;
  return PIE_OK;
}

pie_status pie_batch_rows(const pie_batch* b, int32_t* n) {
  if (!b || !n) return PIE_ERR_INVALID;
  *n = b->n_rows;
  return PIE_OK;
}

pie_status pie_batch_slots(const pie_batch* b, int32_t* pos, int32_t* slot) {
  if (!b) return PIE_ERR_INVALID;
  if (pos && b->n_rows) std::memcpy(pos, b->row_pos.data(), b->n_rows * sizeof(int32_t));
  if (slot && b->n_rows) std::memcpy(slot, b->row_slot.data(), b->n_rows * sizeof(int32_t));
  return PIE_OK;
}

pie_status pie_kv_append(pie_ctx* c, pie_batch* b, int32_t layer, const void* k, const void* v) {
  if (!c || !b || b != c->open) return c ? fail(c, PIE_ERR_BAD_HANDLE, "not the open batch") : PIE_ERR_INVALID;
  if (!aligned(k, 16) || !aligned(v, 16)) return fail(c, PIE_ERR_INVALID, "K or V not 16-byte aligned");
  if (c->plan_only) return fail(c, PIE_ERR_STATE, "plan-only context");
  if (layer < 0 || layer >= c->geo.num_layers) return fail(c, PIE_ERR_INVALID, "layer %d", layer);
  if (b->n_rows == 0) return PIE_OK;
  if (!k || !v) return fail(c, PIE_ERR_INVALID, "null K or V");
  const int32_t nsc = c->geo.num_layers * c->geo.hkv;
  cudaError_t e = pie::launch_kv_append(c->geo, b->view, layer, k, v, c->cfg.k_pool, c->cfg.v_pool,
                                        c->d_scales + 2 * nsc, c->d_scales + 3 * nsc, c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "kv_append launch");
  b->appended_any = true;
  return PIE_OK;
}

pie_status pie_rope_table(float theta, int32_t head_dim, int32_t positions, float* out) {
  if (!out || head_dim <= 0 || head_dim % 2 || positions <= 0 || !(theta > 1.0f) || !std::isfinite(theta))
    return PIE_ERR_INVALID;
  const int32_t half = head_dim / 2;
  std::vector<double> w(half);
  for (int32_t i = 0; i < half; ++i) w[i] = std::pow(static_cast<double>(theta), -2.0 * i / head_dim);
  for (int32_t p = 0; p < positions; ++p)
    for (int32_t i = 0; i < half; ++i) {
      const double a = static_cast<double>(p) * w[i];
      out[(static_cast<size_t>(p) * half + i) * 2] = static_cast<float>(std::cos(a));
      out[(static_cast<size_t>(p) * half + i) * 2 + 1] = static_cast<float>(std::sin(a));
    }
  return PIE_OK;
}

pie_status pie_kv_append_rope(pie_ctx* c, pie_batch* b, int32_t layer, const void* k, const void* v, const void* q,
                              void* q_out) {
  if (!c || !b || b != c->open) return c ? fail(c, PIE_ERR_BAD_HANDLE, "not the open batch") : PIE_ERR_INVALID;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(q, 16) || !aligned(q_out, 16))
    return fail(c, PIE_ERR_INVALID, "K, V, Q or the rotated Q not 16-byte aligned");
  if (c->plan_only) return fail(c, PIE_ERR_STATE, "plan-only context");
  if (!c->d_rope) return fail(c, PIE_ERR_STATE, "context has no rotary table (rope_theta = 0)");
  if (layer < 0 || layer >= c->geo.num_layers) return fail(c, PIE_ERR_INVALID, "layer %d", layer);
  if (b->n_rows == 0) return PIE_OK;
  if (!k || !v) return fail(c, PIE_ERR_INVALID, "null K or V");
  if ((q == nullptr) != (q_out == nullptr)) return fail(c, PIE_ERR_INVALID, "q and q_out go together");
  for (int32_t pos : b->row_pos)
    if (pos >= c->cfg.rope_max_positions)
      return fail(c, PIE_ERR_RANGE, "position %d beyond the rotary table (%d)", pos, c->cfg.rope_max_positions);
  const int32_t nsc = c->geo.num_layers * c->geo.hkv;
  cudaError_t e = pie::launch_kv_append_rope(c->geo, b->view, layer, k, v, q, q_out, c->d_rope, c->cfg.k_pool,
                                             c->cfg.v_pool, c->d_scales + 2 * nsc, c->d_scales + 3 * nsc, c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "kv_append_rope launch");
  b->appended_any = true;
  return PIE_OK;
}

// cuTensorMapEncodeTiled through the CUDA runtime's driver entry point (no link
// against the CUDA driver library); null when the driver does not offer it.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult found{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &found) !=
            cudaSuccess ||
        found != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Tensor map over a bf16 Q ([n_rows][Hq][d]) for the tensor-core kernel's Q
// tiles: box d 64 x G heads x 128/G rows with the 128-byte swizzle, which is
// the tiles' K-major operand layout.  False when it cannot be built; the
// kernel then loads Q by cp.async.
static bool q_tensor_map(pie_ctx* c, const void* q, int32_t n_rows, CUtensorMap* map) {
  if (q == c->q_map_ptr && n_rows == c->q_map_rows) {
    *map = c->q_map;
    return true;
  }
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || c->geo.kv_dtype != PIE_KV_BF16 || (reinterpret_cast<uintptr_t>(q) & 15) != 0) return false;
  const cuuint64_t d = static_cast<cuuint64_t>(c->geo.d), hq = static_cast<cuuint64_t>(c->geo.hq);
  const cuuint32_t G = static_cast<cuuint32_t>(c->geo.hq / c->geo.hkv);
  const cuuint64_t dim[3] = {d, hq, static_cast<cuuint64_t>(n_rows)};
  const cuuint64_t stride[2] = {d * 2, hq * d * 2};  // bytes, dimensions 1 and 2
  const cuuint32_t box[3] = {64, G, 128 / G};
  const cuuint32_t elem[3] = {1, 1, 1};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dim, stride, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  c->q_map = *map;
  c->q_map_ptr = q;
  c->q_map_rows = n_rows;
  return true;
}

pie_status pie_attend(pie_ctx* c, pie_batch* b, int32_t layer, const void* q, void* out, float* lse) {
  if (!c || !b || b != c->open) return c ? fail(c, PIE_ERR_BAD_HANDLE, "not the open batch") : PIE_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return fail(c, PIE_ERR_INVALID, "Q or output not 16-byte aligned, or LSE not 4-byte aligned");
  if (c->plan_only) return fail(c, PIE_ERR_STATE, "plan-only context");
  if (layer < 0 || layer >= c->geo.num_layers) return fail(c, PIE_ERR_INVALID, "layer %d", layer);
  if (b->n_rows == 0) return PIE_OK;
  if (!q || !out) return fail(c, PIE_ERR_INVALID, "null Q or output");
  const pie::PlanView& v = b->view;
  const int32_t nsc = c->geo.num_layers * c->geo.hkv;
  float* acc = c->d_part;
  size_t total_parts = c->part_cap / (static_cast<size_t>(c->geo.hq) * (c->geo.d + 2));
  float* ml = c->d_part + total_parts * c->geo.hq * c->geo.d;
  cudaError_t e = cudaSuccess;
  // Up to three launches write disjoint outputs and partials: tensor-core
  // items, wide decode items (fork / dedup groups of more than 32 rows x
  // heads, two N tiles per warp) and narrow decode items.  The largest kind
  // goes on the caller's stream -- tensor-core items if any, else the narrow
  // decode items -- and the others on the context's second stream, forked
  // from and joined back into the caller's stream, so they take the SMs the
  // first leaves free; the merge waits for all.  The tensor-core grid is
  // submitted first: its CTAs need a whole SM each (224 KB of shared
  // memory), and decode CTAs spread over the SMs first would keep them out.
  pie::PlanView wide = v, narrow = v;
  wide.n_dec = v.n_dec_wide;
  narrow.dec_items = v.dec_items + v.n_dec_wide;
  narrow.n_dec = v.n_dec - v.n_dec_wide;
  narrow.max_dec_m = std::min(v.max_dec_m, pie::kDecodeNarrowM);
  const bool narrow_main = v.n_pre == 0;
  const bool side = (v.n_pre > 0) + (wide.n_dec > 0) + (narrow.n_dec > 0) > 1;
  if (side) {
    e = cudaEventRecord(c->fork_ev, c->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->side, c->fork_ev, 0);
  }
  cudaStream_t other = side ? c->side : c->stream;
  if (e == cudaSuccess && v.n_pre) {
    // Encoding a map costs about 0.15 us of host time per new Q address (the
    // last one is kept), and the map shortens every tensor-core CTA's start
    CUtensorMap q_map;
    const bool mapped = q_tensor_map(c, q, b->n_rows, &q_map);
    e = pie::launch_prefill(c->geo, v, layer, q, mapped ? &q_map : nullptr, c->cfg.k_pool, c->cfg.v_pool,
                            c->d_scales, c->d_scales + nsc, out, lse, acc, ml, c->d_err, c->stream);
  }
  if (e == cudaSuccess && narrow.n_dec && narrow_main)
    e = pie::launch_decode(c->geo, narrow, layer, q, c->cfg.k_pool, c->cfg.v_pool, c->d_scales, c->d_scales + nsc,
                           out, lse, acc, ml, c->d_err, c->stream);
  if (e == cudaSuccess && wide.n_dec)
    e = pie::launch_decode(c->geo, wide, layer, q, c->cfg.k_pool, c->cfg.v_pool, c->d_scales, c->d_scales + nsc, out,
                           lse, acc, ml, c->d_err, other);
  if (e == cudaSuccess && narrow.n_dec && !narrow_main)
    e = pie::launch_decode(c->geo, narrow, layer, q, c->cfg.k_pool, c->cfg.v_pool, c->d_scales, c->d_scales + nsc,
                           out, lse, acc, ml, c->d_err, other);
  if (e == cudaSuccess && side) e = cudaEventRecord(c->join_ev, c->side);
  if (e == cudaSuccess && side) e = cudaStreamWaitEvent(c->stream, c->join_ev, 0);
  if (e == cudaSuccess && v.n_merge && !v.merge_cnt) e = pie::launch_merge(c->geo, v, out, lse, acc, ml, c->stream);
  if (e != cudaSuccess) {
    c->cnt_dirty = true;  // some parts may be counted without their row's merge
    return cuda_fail(c, e, "attend launch");
  }
  return PIE_OK;
}

pie_status pie_ctx_set_merge_mode(pie_ctx* c, int32_t mode) {
  if (!c || mode < 0 || mode > 1) return PIE_ERR_INVALID;
  c->merge_mode = mode;
  return PIE_OK;
}

pie_status pie_ctx_check(pie_ctx* c, int32_t* flags) {
  if (!c || !flags) return PIE_ERR_INVALID;
  *flags = 0;
  if (c->plan_only) return PIE_OK;
  cudaError_t e = cudaStreamSynchronize(c->stream);
  if (e == cudaSuccess) e = cudaMemcpy(flags, c->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(int));
  if (e == cudaSuccess && *flags) c->cnt_dirty = true;  // the next pass clears the merge counters
  if (e != cudaSuccess) return cuda_fail(c, e, "pie_ctx_check");
  return PIE_OK;
}

pie_status pie_selftest_wait_timeout(pie_ctx* c, int32_t polls) {
  if (!c || polls <= 0) return PIE_ERR_INVALID;
  if (c->plan_only) return fail(c, PIE_ERR_STATE, "plan-only context");
  cudaError_t e = pie::launch_wait_selftest(c->d_err, static_cast<uint32_t>(polls), c->stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "self-test launch");
  return PIE_OK;
}

pie_status pie_selftest_fail_next_begin(pie_ctx* c) {
  if (!c) return PIE_ERR_INVALID;
  c->fail_next_begin = true;
  return PIE_OK;
}

pie_status pie_batch_plan_info(const pie_batch* b, int32_t* info) {
  if (!b || !info) return PIE_ERR_INVALID;
  info[0] = b->view.n_dec;
  info[1] = b->view.n_pre;
  info[2] = b->view.n_merge;
  info[3] = b->view.n_copies;
  info[4] = b->view.n_merge > 0 && !b->view.merge_cnt;
  return PIE_OK;
}

pie_status pie_batch_items(const pie_batch* b, int32_t kind, int32_t* out, int32_t cap, int32_t* n) {
  if (!b || !n || (kind != 0 && kind != 1)) return PIE_ERR_INVALID;
  const auto& v = kind == 0 ? b->dec : b->pre;
  *n = static_cast<int32_t>(v.size());
  int32_t m = std::min<int32_t>(cap, *n);
  if (out && m > 0) std::memcpy(out, v.data(), static_cast<size_t>(m) * sizeof(WorkItem));
  return PIE_OK;
}

pie_status pie_batch_end(pie_ctx* c, pie_batch* b) {
  if (!c || !b || b != c->open) return c ? fail(c, PIE_ERR_BAD_HANDLE, "not the open batch") : PIE_ERR_INVALID;
  delete b;
  c->open = nullptr;
  return PIE_OK;
}

}  // extern "C"
