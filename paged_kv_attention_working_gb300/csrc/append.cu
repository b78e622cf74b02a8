// ops.attn.kv_append ("Poem ops", Operations table): scatter one layer's new
// K and V rows into their reserved page slots, as bf16 or as OCP FP8 E4M3;
// and the copy-on-write page copy that a write into a shared page needs
// ("How Pie thinks", section 4: forks share the frozen prefix without
// copying it, so a shared partial page is copied only when written).
//
// Both kernels are HBM streaming kernels: 16-byte vector loads and stores,
// one thread per 16-byte output chunk, consecutive threads on consecutive
// chunks of a key row (whole 128-byte lines per 8 threads).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "plan.h"

namespace pie {
namespace {

__device__ __forceinline__ int64_t slot_chunk_offset(const Geometry& g, int layer, int page, int head,
                                                     int s, int chunk16) {
  // pool layout: [layer][page][head][block]; a block is panels of 128 bytes
  // per key; 16-byte chunk c of key slot s sits at s*128 + 16*(c ^ (s % 8)).
  int64_t blk = ((static_cast<int64_t>(layer) * g.num_pages + page) * g.hkv + head) * g.block_bytes;
  int panel = chunk16 >> 3, c = chunk16 & 7;
  return blk + panel * (kPageSize * 128) + s * 128 + 16 * (c ^ (s & 7));
}

// bf16: one thread per (row, head, 16-byte chunk), K and V.
__global__ void kv_append_bf16(Geometry g, PlanView p, int layer, const uint4* __restrict__ k,
                               const uint4* __restrict__ v, uint8_t* __restrict__ kpool,
                               uint8_t* __restrict__ vpool) {
  const int chunks = g.d * 2 / 16;
  int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t total = static_cast<int64_t>(p.n_rows) * g.hkv * chunks;
  if (idx >= total) return;
  int c = static_cast<int>(idx % chunks);
  int64_t rh = idx / chunks;
  int head = static_cast<int>(rh % g.hkv);
  int row = static_cast<int>(rh / g.hkv);
  int slot = p.row_slot[row];
  int64_t off = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c);
  uint4 kk = __ldg(k + idx), vv = __ldg(v + idx);
  *reinterpret_cast<uint4*>(kpool + off) = kk;
  *reinterpret_cast<uint4*>(vpool + off) = vv;
}

__device__ __forceinline__ uint32_t quant4(uint2 bits, float inv) {
  // four bf16 -> four e4m3 bytes (element 0 in the low byte)
  float f0 = __uint_as_float(bits.x << 16) * inv, f1 = __uint_as_float(bits.x & 0xFFFF0000u) * inv;
  float f2 = __uint_as_float(bits.y << 16) * inv, f3 = __uint_as_float(bits.y & 0xFFFF0000u) * inv;
  uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f0, f1), __NV_SATFINITE, __NV_E4M3);
  uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f2, f3), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// e4m3: one thread per (row, head, 16-element chunk); 32 bytes in, 16 out.
__global__ void kv_append_e4m3(Geometry g, PlanView p, int layer, const uint4* __restrict__ k,
                               const uint4* __restrict__ v, uint8_t* __restrict__ kpool,
                               uint8_t* __restrict__ vpool, const float* __restrict__ inv_k,
                               const float* __restrict__ inv_v) {
  const int chunks = g.d / 16;
  int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t total = static_cast<int64_t>(p.n_rows) * g.hkv * chunks;
  if (idx >= total) return;
  int c = static_cast<int>(idx % chunks);
  int64_t rh = idx / chunks;
  int head = static_cast<int>(rh % g.hkv);
  int row = static_cast<int>(rh / g.hkv);
  int slot = p.row_slot[row];
  int64_t off = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c);
  float ik = inv_k[layer * g.hkv + head], iv = inv_v[layer * g.hkv + head];
  uint4 k0 = __ldg(k + 2 * idx), k1 = __ldg(k + 2 * idx + 1);
  uint4 v0 = __ldg(v + 2 * idx), v1 = __ldg(v + 2 * idx + 1);
  uint4 ko, vo;
  ko.x = quant4(make_uint2(k0.x, k0.y), ik);
  ko.y = quant4(make_uint2(k0.z, k0.w), ik);
  ko.z = quant4(make_uint2(k1.x, k1.y), ik);
  ko.w = quant4(make_uint2(k1.z, k1.w), ik);
  vo.x = quant4(make_uint2(v0.x, v0.y), iv);
  vo.y = quant4(make_uint2(v0.z, v0.w), iv);
  vo.z = quant4(make_uint2(v1.x, v1.y), iv);
  vo.w = quant4(make_uint2(v1.z, v1.w), iv);
  *reinterpret_cast<uint4*>(kpool + off) = ko;
  *reinterpret_cast<uint4*>(vpool + off) = vo;
}

// copy-on-write: blockIdx.x = copy * layers + layer, blockIdx.y = K / V.
// A page's blocks for all heads are contiguous, so one page of one layer is
// hkv * block_bytes consecutive bytes.
__global__ void page_copy(Geometry g, PlanView p, uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool) {
  int ci = blockIdx.x / g.num_layers, layer = blockIdx.x % g.num_layers;
  uint8_t* pool = blockIdx.y ? vpool : kpool;
  CopyItem cp = p.copies[ci];
  int64_t bytes = g.hkv * g.block_bytes;
  const uint4* src = reinterpret_cast<const uint4*>(pool + (static_cast<int64_t>(layer) * g.num_pages + cp.src) * bytes);
  uint4* dst = reinterpret_cast<uint4*>(pool + (static_cast<int64_t>(layer) * g.num_pages + cp.dst) * bytes);
  for (int64_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_kv_append(const Geometry& g, const PlanView& p, int layer, const void* k, const void* v,
                             void* kpool, void* vpool, const float* inv_scale_k, const float* inv_scale_v,
                             cudaStream_t st) {
  const int chunks = g.kv_dtype == 0 ? g.d * 2 / 16 : g.d / 16;
  int64_t total = static_cast<int64_t>(p.n_rows) * g.hkv * chunks;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  unsigned blocks = static_cast<unsigned>((total + threads - 1) / threads);
  if (g.kv_dtype == 0)
    kv_append_bf16<<<blocks, threads, 0, st>>>(g, p, layer, static_cast<const uint4*>(k),
                                                static_cast<const uint4*>(v), static_cast<uint8_t*>(kpool),
                                                static_cast<uint8_t*>(vpool));
  else
    kv_append_e4m3<<<blocks, threads, 0, st>>>(g, p, layer, static_cast<const uint4*>(k),
                                                static_cast<const uint4*>(v), static_cast<uint8_t*>(kpool),
                                                static_cast<uint8_t*>(vpool), inv_scale_k, inv_scale_v);
  return cudaGetLastError();
}

cudaError_t launch_page_copy(const Geometry& g, const PlanView& p, void* kpool, void* vpool, cudaStream_t st) {
  if (p.n_copies == 0) return cudaSuccess;
  dim3 grid(p.n_copies * g.num_layers, 2);
  page_copy<<<grid, 256, 0, st>>>(g, p, static_cast<uint8_t*>(kpool), static_cast<uint8_t*>(vpool));
  return cudaGetLastError();
}

}  // namespace pie
