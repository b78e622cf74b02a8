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

#include "launch.h"
#include "plan.h"
#include "ptx.cuh"

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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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

// ---------------------------------------------------------------- rope
// Rotary embedding fused into the append ("Poem ops": ops.elemwise.rope
// feeding ops.attn.kv_append): dimension i of a head pairs with i + d/2 and
// turns by the row position's angle from the (cos, sin) table,
//   y_i = x_i c - x_{i+d/2} s,   y_{i+d/2} = x_{i+d/2} c + x_i s,
// each product and the sum rounded to float32 (no fused multiply-add), the
// result rounded to bf16 -- the same bytes as rotating to bf16 first and
// appending after.  One thread takes 16 dimensions of each half of one head
// of one row: K heads (rotated, then stored or quantised like
// kv_append_bf16 / kv_append_e4m3, with their V unrotated), then, when q is
// given, Q heads (rotated into q_out).

// Rotates 8 bf16 pairs: a holds dims j..j+7 of the first half, b the same of
// the second half, cs the 8 (cos, sin) pairs.
__device__ __forceinline__ void rotate8(uint4& a, uint4& b, const float4* cs) {
  uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
  uint32_t* pb = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 t = __ldg(cs + w);  // (c0, s0, c1, s1) of the two dims in word w
    float x0[2] = {__uint_as_float(pa[w] << 16), __uint_as_float(pa[w] & 0xFFFF0000u)};
    float x1[2] = {__uint_as_float(pb[w] << 16), __uint_as_float(pb[w] & 0xFFFF0000u)};
    const float c[2] = {t.x, t.z}, sn[2] = {t.y, t.w};
    float y0[2], y1[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      y0[e] = __fsub_rn(__fmul_rn(x0[e], c[e]), __fmul_rn(x1[e], sn[e]));
      y1[e] = __fadd_rn(__fmul_rn(x1[e], c[e]), __fmul_rn(x0[e], sn[e]));
    }
    const __nv_bfloat162 r0 = __floats2bfloat162_rn(y0[0], y0[1]);  // .x (low half) = first dim
    const __nv_bfloat162 r1 = __floats2bfloat162_rn(y1[0], y1[1]);
    pa[w] = *reinterpret_cast<const uint32_t*>(&r0);
    pb[w] = *reinterpret_cast<const uint32_t*>(&r1);
  }
}

template <bool E4M3>
__global__ void kv_append_rope(Geometry g, PlanView p, int layer, const uint4* __restrict__ k,
                               const uint4* __restrict__ v, const uint4* __restrict__ q, uint4* __restrict__ q_out,
                               const float* __restrict__ rope, uint8_t* __restrict__ kpool,
                               uint8_t* __restrict__ vpool, const float* __restrict__ inv_k,
                               const float* __restrict__ inv_v) {
  pdl_wait();
  pdl_trigger();
  const int nc = g.d / 32;        // 16-dimension groups per half
  const int hd = g.d / 8;         // 16-byte chunks per head row
  const int heads = g.hkv + (q ? g.hq : 0);
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(p.n_rows) * heads * nc) return;
  const int c = static_cast<int>(idx % nc);
  const int64_t rh = idx / nc;
  const int hh = static_cast<int>(rh % heads);
  const int row = static_cast<int>(rh / heads);
  const int pos = p.row_pos[row];
  const float4* cs = reinterpret_cast<const float4*>(rope + (static_cast<int64_t>(pos) * (g.d / 2) + 16 * c) * 2);
  // chunk indices (16-byte bf16 units) of the thread's dims in a head row
  const int c0 = 2 * c, c1 = hd / 2 + 2 * c;
  if (hh >= g.hkv) {
    const int64_t base = (static_cast<int64_t>(row) * g.hq + (hh - g.hkv)) * hd;
    uint4 a0 = __ldg(q + base + c0), a1 = __ldg(q + base + c0 + 1);
    uint4 b0 = __ldg(q + base + c1), b1 = __ldg(q + base + c1 + 1);
    rotate8(a0, b0, cs);
    rotate8(a1, b1, cs + 4);
    q_out[base + c0] = a0;
    q_out[base + c0 + 1] = a1;
    q_out[base + c1] = b0;
    q_out[base + c1 + 1] = b1;
    return;
  }
  const int head = hh;
  const int64_t base = (static_cast<int64_t>(row) * g.hkv + head) * hd;
  uint4 a0 = __ldg(k + base + c0), a1 = __ldg(k + base + c0 + 1);
  uint4 b0 = __ldg(k + base + c1), b1 = __ldg(k + base + c1 + 1);
  rotate8(a0, b0, cs);
  rotate8(a1, b1, cs + 4);
  const uint4 va0 = __ldg(v + base + c0), va1 = __ldg(v + base + c0 + 1);
  const uint4 vb0 = __ldg(v + base + c1), vb1 = __ldg(v + base + c1 + 1);
  const int slot = p.row_slot[row];
  if constexpr (!E4M3) {
    const int64_t o0 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c0);
    const int64_t o1 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c0 + 1);
    const int64_t o2 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c1);
    const int64_t o3 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c1 + 1);
    *reinterpret_cast<uint4*>(kpool + o0) = a0;
    *reinterpret_cast<uint4*>(kpool + o1) = a1;
    *reinterpret_cast<uint4*>(kpool + o2) = b0;
    *reinterpret_cast<uint4*>(kpool + o3) = b1;
    *reinterpret_cast<uint4*>(vpool + o0) = va0;
    *reinterpret_cast<uint4*>(vpool + o1) = va1;
    *reinterpret_cast<uint4*>(vpool + o2) = vb0;
    *reinterpret_cast<uint4*>(vpool + o3) = vb1;
  } else {
    // e4m3 chunk e holds dims 16e..16e+15: this thread's are chunks c and d/32 + c
    const float ik = inv_k[layer * g.hkv + head], iv = inv_v[layer * g.hkv + head];
    const int64_t o0 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, c);
    const int64_t o1 = slot_chunk_offset(g, layer, slot >> 4, head, slot & 15, nc + c);
    auto q16 = [](uint4 lo, uint4 hi, float inv) {
      return make_uint4(quant4(make_uint2(lo.x, lo.y), inv), quant4(make_uint2(lo.z, lo.w), inv),
                        quant4(make_uint2(hi.x, hi.y), inv), quant4(make_uint2(hi.z, hi.w), inv));
    };
    *reinterpret_cast<uint4*>(kpool + o0) = q16(a0, a1, ik);
    *reinterpret_cast<uint4*>(kpool + o1) = q16(b0, b1, ik);
    *reinterpret_cast<uint4*>(vpool + o0) = q16(va0, va1, iv);
    *reinterpret_cast<uint4*>(vpool + o1) = q16(vb0, vb1, iv);
  }
}

// copy-on-write: blockIdx.x = copy * layers + layer, blockIdx.y = K / V.
// A page's blocks for all heads are contiguous, so one page of one layer is
// hkv * block_bytes consecutive bytes.
__global__ void page_copy(Geometry g, PlanView p, uint8_t* __restrict__ kpool, uint8_t* __restrict__ vpool) {
  pdl_wait();
  pdl_trigger();
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
  cudaError_t e;
  if (g.kv_dtype == 0)
    e = launch_pdl(kv_append_bf16, blocks, threads, 0, st, g, p, layer, static_cast<const uint4*>(k),
                   static_cast<const uint4*>(v), static_cast<uint8_t*>(kpool), static_cast<uint8_t*>(vpool));
  else
    e = launch_pdl(kv_append_e4m3, blocks, threads, 0, st, g, p, layer, static_cast<const uint4*>(k),
                   static_cast<const uint4*>(v), static_cast<uint8_t*>(kpool), static_cast<uint8_t*>(vpool),
                   inv_scale_k, inv_scale_v);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_kv_append_rope(const Geometry& g, const PlanView& p, int layer, const void* k, const void* v,
                                  const void* q, void* q_out, const float* rope, void* kpool, void* vpool,
                                  const float* inv_scale_k, const float* inv_scale_v, cudaStream_t st) {
  const int heads = g.hkv + (q ? g.hq : 0);
  int64_t total = static_cast<int64_t>(p.n_rows) * heads * (g.d / 32);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  unsigned blocks = static_cast<unsigned>((total + threads - 1) / threads);
  auto args = [&](auto kern) {
    return launch_pdl(kern, blocks, threads, 0, st, g, p, layer, static_cast<const uint4*>(k),
                      static_cast<const uint4*>(v), static_cast<const uint4*>(q), static_cast<uint4*>(q_out), rope,
                      static_cast<uint8_t*>(kpool), static_cast<uint8_t*>(vpool), inv_scale_k, inv_scale_v);
  };
  const cudaError_t e = g.kv_dtype == 0 ? args(kv_append_rope<false>) : args(kv_append_rope<true>);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_page_copy(const Geometry& g, const PlanView& p, void* kpool, void* vpool, cudaStream_t st) {
  if (p.n_copies == 0) return cudaSuccess;
  dim3 grid(p.n_copies * g.num_layers, 2);
  const cudaError_t e =
      launch_pdl(page_copy, grid, 256, 0, st, g, p, static_cast<uint8_t*>(kpool), static_cast<uint8_t*>(vpool));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pie
