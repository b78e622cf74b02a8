// Internal plan structures shared by the host planner and the CUDA kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pie {

constexpr int kPageSize = 16;

// One unit of attention work for one KV head (the head is blockIdx.y): a set
// of query rows that all read the same run of pages of one working set.
// Private items cover one segment's rows over part of its own pages; shared
// items cover the rows of every segment of a fork/dedup group over the
// pages they all hold.
struct WorkItem {
  int32_t pages_off;  // index into page_ids of the first page of the run
  int32_t n_pages;    // pages in the run
  int32_t key_base;   // position of the run's first key (16 * logical page)
  int32_t rows_off;   // index into row_list of the item's first row
  int32_t n_rows;     // rows (each row contributes Hq/Hkv query heads)
  int32_t part;       // -1: rows are written straight to the output;
                      // else partial index = row_part_base[row] + part
  int32_t n_keys;     // keys in the run that lie before its end (<= 16*n_pages)
  int32_t direct_rows;  // 1: the item's rows are batch rows rows_off,
                        // rows_off + 1, ... in order (row_list is the
                        // identity there), so a kernel skips the lookup
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

struct CopyItem {  // copy-on-write: page src -> page dst, every layer, K and V
  int32_t src, dst;
};

// Device views of one batch's plan (all arrays live in one uploaded buffer).
struct PlanView {
  const int32_t* page_ids;
  const int32_t* row_pos;        // [n_rows]
  const int32_t* row_slot;       // [n_rows] page * 16 + slot
  const int32_t* row_part_base;  // [n_rows], -1 for direct rows
  const int32_t* row_list;       // item row lists
  const WorkItem* dec_items;     // decode-kernel items
  const WorkItem* pre_items;     // tensor-core (prefill) items
  const int4* merge_info;        // rows with >= 2 parts: (row, parts, first
                                 // part index = row_part_base[row], 0)
  const int32_t* row_merge;      // [n_rows]: index into merge_info, -1 for direct rows
  int32_t* merge_cnt;            // [n_merge][Hq] parts stored so far, zero
                                 // between launches; non-null: the decode
                                 // kernels merge split rows themselves (no
                                 // tensor-core item writes partials), else a
                                 // merge launch follows
  const CopyItem* copies;
  int32_t n_rows, n_dec, n_pre, n_merge, n_copies;
  int32_t max_dec_m;             // largest rows x query heads of a decode item
  int32_t n_dec_wide;            // decode items [0, n_dec_wide) have more than
                                 // kDecodeNarrowM rows x heads, the rest at most
};

#ifdef __CUDACC__
// Batch row of an item's i-th row.
__device__ __forceinline__ int item_row(const PlanView& p, const WorkItem& it, int i) {
  return it.direct_rows ? it.rows_off + i : p.row_list[it.rows_off + i];
}
#endif

// Decode items of at most this many rows x query heads run in the decode
// kernel variant with one 8-wide N tile per warp (fewer registers, 4 CTAs
// per SM); wider items (fork / dedup groups up to 64) take two per warp.
constexpr int kDecodeNarrowM = 32;

struct Geometry {
  int32_t num_layers, hq, hkv, d, num_pages, kv_dtype;
  int64_t block_bytes;  // 16 * d * esize
  float softcap;        // > 0: scores s become softcap * tanh(s / softcap)
};

// Kernel launchers (defined in the .cu files); all return cudaGetLastError().
cudaError_t launch_kv_append(const Geometry& g, const PlanView& p, int layer,
                             const void* k, const void* v, void* kpool, void* vpool,
                             const float* inv_scale_k, const float* inv_scale_v,
                             cudaStream_t st);
cudaError_t launch_kv_append_rope(const Geometry& g, const PlanView& p, int layer, const void* k,
                                  const void* v, const void* q, void* q_out, const float* rope,
                                  void* kpool, void* vpool, const float* inv_scale_k,
                                  const float* inv_scale_v, cudaStream_t st);
cudaError_t launch_page_copy(const Geometry& g, const PlanView& p, void* kpool, void* vpool,
                             cudaStream_t st);
cudaError_t launch_decode(const Geometry& g, const PlanView& p, int layer, const void* q,
                          const void* kpool, const void* vpool, const float* scale_k,
                          const float* scale_v, void* out, float* lse, float* part_acc,
                          float* part_ml, int* err, cudaStream_t st);
// q_map: a tiled tensor map over Q ([rows][Hq][d] bf16, box d 64 x G heads x
// 128/G rows, 128-byte swizzle), or null; with it, items whose rows are in
// batch order load their Q tiles by tensor copies.
cudaError_t launch_prefill(const Geometry& g, const PlanView& p, int layer, const void* q,
                           const CUtensorMap* q_map, const void* kpool, const void* vpool,
                           const float* scale_k, const float* scale_v, void* out, float* lse,
                           float* part_acc, float* part_ml, int* err, cudaStream_t st);
cudaError_t launch_wait_selftest(int* err, uint32_t polls, cudaStream_t st);
cudaError_t launch_merge(const Geometry& g, const PlanView& p, void* out, float* lse,
                         const float* part_acc, const float* part_ml, cudaStream_t st);

}  // namespace pie
