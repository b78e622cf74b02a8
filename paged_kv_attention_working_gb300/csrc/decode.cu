// Decode attention over paged KV ("Poem ops", ops.attn.attend) and the merge
// of split / shared partial results.
//
// One CTA takes one work item for one KV head: up to 64 query rows x query
// heads of that KV group (one decode token, a few speculative drafts, or the
// rows of a small fork / dedup group) over a run of pages of one working set.
// The item's pages stream through a ring of shared-memory stages, one 1-D
// bulk async copy per K and per V page block (the pool's block layout is
// already bank-conflict free for ldmatrix, see pie_attn.h), filled by a
// producer warp.  Four consumer warps run QK^T and PV on the tensor cores
// with warp-level m16n8k16 MMA (M = 16 query heads x rows, N = 8 keys or 8
// head-dim columns) and keep an online softmax in registers.  When the item
// has a single 16-row M tile the four warps take alternate pages and merge
// their softmax states at the end; with 2 or 4 M tiles each warp owns a
// tile and every page is read from HBM once for all of them, which is what
// makes a fork group's shared pages cost one read per group ("How Pie
// thinks", section 4: the prompt is computed once and shared).
//
// E4M3 pages are converted in registers to f16 (exact) and the per-head
// scales are folded into the softmax and output scaling.  With a logit soft
// cap (CAP) each visible score s becomes c * tanh(s / c) before the running
// max and the exponentials.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "../../include/pie_attn.h"
#include "func_attr.h"
#include "plan.h"
#include "ptx.cuh"

namespace pie {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <bool E4M3, int D>
struct DecodeCfg {
  static constexpr int kEsize = E4M3 ? 1 : 2;
  static constexpr int kBlock = kPageSize * D * kEsize;  // bytes per page-head block
  static constexpr int kStages = E4M3 ? 12 : 8;
  static constexpr int kStageBytes = 2 * kBlock;
  static constexpr int kNT = D / 8;  // n-tiles of the output (head dim)
  static constexpr int kKS = D / 16; // k-steps of QK^T
  static constexpr int kCombineFloats = kConsumerWarps * 32 * (kNT * 4 + 4);
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kSmem = (kRing > kCombineFloats * 4 ? kRing : kCombineFloats * 4) + 2 * kStages * 8 + 16;
};

template <bool E4M3, int D, bool CAP>
__global__ void __launch_bounds__(kThreads, 3) decode_kernel(Geometry g, PlanView p, int layer,
                                                          const __nv_bfloat16* __restrict__ q,
                                                          const uint8_t* __restrict__ kpool,
                                                          const uint8_t* __restrict__ vpool,
                                                          const float* __restrict__ kscale,
                                                          const float* __restrict__ vscale,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                          float* __restrict__ part_acc, float* __restrict__ part_ml,
                                                          int* err) {
  using C = DecodeCfg<E4M3, D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (C::kSmem - 2 * C::kStages * 8 - 16));
  uint64_t* empty = full + C::kStages;

  const WorkItem it = p.dec_items[blockIdx.x];
  const int head = blockIdx.y;
  const int G = g.hq / g.hkv;
  const int M = it.n_rows * G;
  const int n_mt = M <= 16 ? 1 : (M <= 32 ? 2 : 4);
  const int n_grp = kConsumerWarps / n_mt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t layer_blk = (static_cast<int64_t>(layer) * g.num_pages) * g.hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_mt);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < it.n_pages; ++j) {
        int s = j % C::kStages;
        if (j >= C::kStages && !mbar_wait(&empty[s], ((j / C::kStages) - 1) & 1, err)) break;
        int page = p.page_ids[it.pages_off + j];
        int64_t boff = (layer_blk + static_cast<int64_t>(page) * g.hkv + head) * C::kBlock;
        uint8_t* st = smem + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], 2 * C::kBlock);
        bulk_g2s(st, kpool + boff, C::kBlock, &full[s]);
        bulk_g2s(st + C::kBlock, vpool + boff, C::kBlock, &full[s]);
        issued = j + 1;
      }
      // Before this thread leaves, the copies it issued into the last stages
      // have landed (bounded): the consumers already waited for them unless
      // a wait of theirs ran out, and then no copy may outlive the CTA.
      for (int j = issued > C::kStages ? issued - C::kStages : 0; j < issued; ++j)
        if (!mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1, err)) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int mt = warp % n_mt, grp = warp / n_mt;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group / thread in quad
  const float kdq = E4M3 ? kscale[layer * g.hkv + head] : 1.0f;
  const float vdq = E4M3 ? vscale[layer * g.hkv + head] : 1.0f;
  // scores in log2 units: s * qk_scale, or with the soft cap c,
  // tanh(s * cap_pre) * cap_post = c * tanh(s / c) * log2(e)
  const float qk_scale = kdq * rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;
  const float cap_pre = CAP ? kdq * rsqrtf(static_cast<float>(D)) / g.softcap : 0.f;
  const float cap_post = CAP ? g.softcap * 1.4426950408889634f : 0.f;

  // the two M rows this thread holds: m = 16*mt + gq (+8)
  int mrow[2], mpos[2];
  const __nv_bfloat16* qptr[2];
  for (int h = 0; h < 2; ++h) {
    int m = 16 * mt + gq + 8 * h;
    mrow[h] = -1;
    mpos[h] = -1;
    qptr[h] = nullptr;
    if (m < M) {
      int rl = m / G, hl = m % G;
      int row = p.row_list[it.rows_off + rl];
      mrow[h] = row;
      mpos[h] = p.row_pos[row];
      qptr[h] = q + (static_cast<int64_t>(row) * g.hq + head * G + hl) * D;
    }
  }
  // Q as A fragments: qa[ks][0..3] = (row g, k 2t..) (row g+8, k 2t..) (row g, k 2t+8..) (row g+8, k 2t+8..)
  uint32_t qa[C::kKS][4];
#pragma unroll
  for (int ks = 0; ks < C::kKS; ++ks) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo = 0, hi = 0;
      if (qptr[h]) {
        if constexpr (!E4M3) {
          lo = *reinterpret_cast<const uint32_t*>(qptr[h] + 16 * ks + 2 * tq);
          hi = *reinterpret_cast<const uint32_t*>(qptr[h] + 16 * ks + 8 + 2 * tq);
        } else {
          // k-slots 2t,2t+1 <-> d 16ks+4t, +1 ; 2t+8,2t+9 <-> d 16ks+4t+2, +3
          uint2 w = *reinterpret_cast<const uint2*>(qptr[h] + 16 * ks + 4 * tq);
          float f0 = __uint_as_float(w.x << 16), f1 = __uint_as_float(w.x & 0xFFFF0000u);
          float f2 = __uint_as_float(w.y << 16), f3 = __uint_as_float(w.y & 0xFFFF0000u);
          lo = pack_f16(f0, f1);
          hi = pack_f16(f2, f3);
        }
      }
      qa[ks][h] = lo;
      qa[ks][2 + h] = hi;
    }
  }

  float o[C::kNT][4];
#pragma unroll
  for (int i = 0; i < C::kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mx[2] = {-INFINITY, -INFINITY}, sum[2] = {0.f, 0.f};

  for (int j = grp; j < it.n_pages; j += n_grp) {
    const int s = j % C::kStages;
    // warp-uniform: the shuffles and MMAs below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / C::kStages) & 1, err))) break;
    const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
    const uint32_t vb = kb + C::kBlock;

    // ---- S = Q K^T for 16 keys: two n-tiles of 8 keys
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (!E4M3) {
      const int key = (lane & 7) + ((lane >> 4) << 3);
      const int csel = (lane >> 3) & 1;
#pragma unroll
      for (int ks = 0; ks < C::kKS; ++ks) {
        int panel = ks >> 2, c = 2 * (ks & 3) + csel;
        uint32_t addr = kb + panel * 2048 + key * 128 + 16 * (c ^ (key & 7));
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma16816<true>(sc[0], qa[ks], b0, b1);
        mma16816<true>(sc[1], qa[ks], b2, b3);
      }
    } else {
      const int key = (lane & 7) + ((lane >> 4) << 3);
      const int csel = (lane >> 3) & 1;
#pragma unroll
      for (int kp = 0; kp < C::kKS / 2; ++kp) {
        int c = 2 * kp + csel;
        uint32_t addr = kb + key * 128 + 16 * (c ^ (key & 7));
        uint32_t r0, r1, r2, r3;  // (keys 0-7, chunk 2kp) (0-7, 2kp+1) (8-15, 2kp) (8-15, 2kp+1)
        ldsm_x4(addr, r0, r1, r2, r3);
        // bytes 4t, 4t+1 -> k-slots 2t, 2t+1; bytes 4t+2, 4t+3 -> k-slots 2t+8, 2t+9
        mma16816<false>(sc[0], qa[2 * kp], e4m3x2_lo_to_f16x2(r0), e4m3x2_hi_to_f16x2(r0));
        mma16816<false>(sc[1], qa[2 * kp], e4m3x2_lo_to_f16x2(r2), e4m3x2_hi_to_f16x2(r2));
        mma16816<false>(sc[0], qa[2 * kp + 1], e4m3x2_lo_to_f16x2(r1), e4m3x2_hi_to_f16x2(r1));
        mma16816<false>(sc[1], qa[2 * kp + 1], e4m3x2_lo_to_f16x2(r3), e4m3x2_hi_to_f16x2(r3));
      }
    }

    // ---- mask, online softmax (log2 domain)
    const int kbase = it.key_base + 16 * j;
    float pm[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float best = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          int kpos = kbase + nt * 8 + 2 * tq + e;
          float v;
          if constexpr (CAP)
            v = kpos <= mpos[h] ? tanh_approx(sc[nt][2 * h + e] * cap_pre) * cap_post : -INFINITY;
          else
            v = kpos <= mpos[h] ? sc[nt][2 * h + e] * qk_scale : -INFINITY;
          sc[nt][2 * h + e] = v;
          best = fmaxf(best, v);
        }
      best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 1));
      best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 2));
      // The reference max only moves when the row max exceeds it by more
      // than 8 (log2 units): weights stay <= 2^8, and O is rescaled rarely.
      const bool up = best > mx[h] + 8.f;
      const float mnew = up ? best : mx[h];
      const float base = mnew == -INFINITY ? 0.f : mnew;
      pm[h] = base;
      if (__any_sync(0xffffffffu, up)) {
        const float alpha = up ? ex2(mx[h] - base) : 1.f;
        sum[h] *= alpha;
#pragma unroll
        for (int i = 0; i < C::kNT; ++i) {
          o[i][2 * h] *= alpha;
          o[i][2 * h + 1] *= alpha;
        }
      }
      mx[h] = mnew;
    }
    uint32_t pa[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float e0 = ex2(sc[nt][2 * h] - pm[h]), e1 = ex2(sc[nt][2 * h + 1] - pm[h]);
        sum[h] += e0 + e1;
        pa[2 * nt + h] = E4M3 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
      }

    // ---- O += P V
    if constexpr (!E4M3) {
      const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int csel = lane >> 4;
#pragma unroll
      for (int np = 0; np < C::kNT / 2; ++np) {
        int cc = 2 * np + csel;  // 16-byte d chunk (8 columns)
        int panel = cc >> 3, c = cc & 7;
        uint32_t addr = vb + panel * 2048 + key * 128 + 16 * (c ^ (key & 7));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma16816<true>(o[2 * np], pa, b0, b1);
        mma16816<true>(o[2 * np + 1], pa, b2, b3);
      }
    } else {
      // Transposing loads of 16-bit units (two e4m3 dims): matrices (keys
      // 0-7, chunk 2cp), (keys 8-15, 2cp), (0-7, 2cp+1), (8-15, 2cp+1); each
      // register holds (key 2t: dims 2g, 2g+1) (key 2t+1: dims 2g, 2g+1),
      // and one byte permute pairs the keys per dim.  n-tile 2c takes dims
      // 16c + 2n, n-tile 2c+1 dims 16c + 2n + 1 (undone when writing out).
      const int vkey = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int vsel = lane >> 4;
#pragma unroll
      for (int cp = 0; cp < D / 32; ++cp) {
        const int c = 2 * cp + vsel;
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(vb + vkey * 128 + 16 * (c ^ (vkey & 7)), r0, r1, r2, r3);
        const uint32_t x0 = prmt(r0, r0, 0x3120), x1 = prmt(r1, r1, 0x3120);
        const uint32_t x2 = prmt(r2, r2, 0x3120), x3 = prmt(r3, r3, 0x3120);
        mma16816<false>(o[4 * cp], pa, e4m3x2_lo_to_f16x2(x0), e4m3x2_lo_to_f16x2(x1));
        mma16816<false>(o[4 * cp + 1], pa, e4m3x2_hi_to_f16x2(x0), e4m3x2_hi_to_f16x2(x1));
        mma16816<false>(o[4 * cp + 2], pa, e4m3x2_lo_to_f16x2(x2), e4m3x2_lo_to_f16x2(x3));
        mma16816<false>(o[4 * cp + 3], pa, e4m3x2_hi_to_f16x2(x2), e4m3x2_hi_to_f16x2(x3));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- finish: quad sums, then merge warps that shared an M tile
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
    sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
  }
  if (n_grp > 1) {
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32));
    float* cm = reinterpret_cast<float*>(smem);
    const int stride = C::kNT * 4 + 4;
    float* mine = cm + (warp * 32 + lane) * stride;
    if (grp > 0) {
#pragma unroll
      for (int i = 0; i < C::kNT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) mine[i * 4 + e] = o[i][e];
      mine[C::kNT * 4 + 0] = mx[0];
      mine[C::kNT * 4 + 1] = mx[1];
      mine[C::kNT * 4 + 2] = sum[0];
      mine[C::kNT * 4 + 3] = sum[1];
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32));
    if (grp > 0) return;
    for (int og = 1; og < n_grp; ++og) {
      const float* th = cm + ((og * n_mt + mt) * 32 + lane) * stride;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m2 = th[C::kNT * 4 + h], l2 = th[C::kNT * 4 + 2 + h];
        float mnew = fmaxf(mx[h], m2);
        float base = mnew == -INFINITY ? 0.f : mnew;
        float a1 = ex2(mx[h] - base), a2 = ex2(m2 - base);
        sum[h] = sum[h] * a1 + l2 * a2;
        mx[h] = mnew;
#pragma unroll
        for (int i = 0; i < C::kNT; ++i) {
          o[i][2 * h] = o[i][2 * h] * a1 + th[i * 4 + 2 * h] * a2;
          o[i][2 * h + 1] = o[i][2 * h + 1] * a1 + th[i * 4 + 2 * h + 1] * a2;
        }
      }
    }
  }

  // ---- write: direct bf16 output, or fp32 partial (acc, m, l) for merging
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (mrow[h] < 0) continue;
    int m = 16 * mt + gq + 8 * h;
    int qh = head * G + m % G;
    int row = mrow[h];
    if (it.part < 0) {
      float inv = sum[h] > 0.f ? vdq / sum[h] : 0.f;
      __nv_bfloat16* dst = out + (static_cast<int64_t>(row) * g.hq + qh) * D;
#pragma unroll
      for (int i = 0; i < C::kNT; ++i) {
        if constexpr (!E4M3) {
          *reinterpret_cast<uint32_t*>(dst + 8 * i + 2 * tq) =
              pack_bf16(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
        } else if ((i & 1) == 0) {
          // n-tiles i (even dims) and i+1 (odd dims) of chunk i/2: dims
          // 8i + 4t .. 8i + 4t + 3
          uint2 wv;
          wv.x = pack_bf16(o[i][2 * h] * inv, o[i + 1][2 * h] * inv);
          wv.y = pack_bf16(o[i][2 * h + 1] * inv, o[i + 1][2 * h + 1] * inv);
          *reinterpret_cast<uint2*>(dst + 8 * i + 4 * tq) = wv;
        }
      }
      if (lse && tq == 0) lse[static_cast<int64_t>(row) * g.hq + qh] = (mx[h] + __log2f(sum[h])) * 0.6931471805599453f;
    } else {
      int64_t slot = static_cast<int64_t>(p.row_part_base[row] + it.part) * g.hq + qh;
      float* dst = part_acc + slot * D;
#pragma unroll
      for (int i = 0; i < C::kNT; ++i) {
        if constexpr (!E4M3) {
          *reinterpret_cast<float2*>(dst + 8 * i + 2 * tq) = make_float2(o[i][2 * h] * vdq, o[i][2 * h + 1] * vdq);
        } else if ((i & 1) == 0) {
          *reinterpret_cast<float4*>(dst + 8 * i + 4 * tq) =
              make_float4(o[i][2 * h] * vdq, o[i + 1][2 * h] * vdq, o[i][2 * h + 1] * vdq, o[i + 1][2 * h + 1] * vdq);
        }
      }
      if (tq == 0) *reinterpret_cast<float2*>(part_ml + slot * 2) = make_float2(mx[h], sum[h]);
    }
  }
}

// One warp per (merged row, query head): combine the row's parts
// (m_i, l_i, acc_i) in the log2 domain:
//   m = max m_i,  l = sum l_i 2^(m_i - m),  o = sum acc_i 2^(m_i - m) / l.
template <int D>
__global__ void merge_kernel(Geometry g, PlanView p, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                             const float* __restrict__ part_acc, const float* __restrict__ part_ml) {
  // One warp per (merged row, query head).  Lane k holds part k's (m, l)
  // (32 parts at a time), so the parts' loads are issued together; the
  // weights reach every lane by shuffle, and each lane accumulates E dims of
  // the parts' partial outputs with vector loads, four parts in flight.
  int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= p.n_merge * g.hq) return;
  int i = wid / g.hq, qh = wid % g.hq;
  int row = p.merge_rows[i], np = p.merge_nparts[i], base = p.row_part_base[row];
  auto ml_at = [&](int k) {
    return k < np ? *reinterpret_cast<const float2*>(part_ml + (static_cast<int64_t>(base + k) * g.hq + qh) * 2)
                  : make_float2(-INFINITY, 0.f);
  };
  const float2 ml0 = ml_at(lane);
  float m = ml0.x;
  for (int k0 = 32; k0 < np; k0 += 32) m = fmaxf(m, ml_at(k0 + lane).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float base_m = m == -INFINITY ? 0.f : m;
  constexpr int E = D / 32;
  using Vec = typename std::conditional<E == 4, float4, float2>::type;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float l = 0.f;
  for (int k0 = 0; k0 < np; k0 += 32) {
    const float2 ml = k0 == 0 ? ml0 : ml_at(k0 + lane);
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - base_m);
    l += ml.y * w;
    const int n = min(32, np - k0);
    const float* a = part_acc + (static_cast<int64_t>(base + k0) * g.hq + qh) * D + lane * E;
#pragma unroll 4
    for (int kk = 0; kk < n; ++kk) {
      const float wk = __shfl_sync(0xffffffffu, w, kk);
      const Vec v = *reinterpret_cast<const Vec*>(a + static_cast<int64_t>(kk) * g.hq * D);
      acc[0] += v.x * wk;
      acc[1] += v.y * wk;
      if constexpr (E == 4) {
        acc[2] += reinterpret_cast<const float4&>(v).z * wk;
        acc[3] += reinterpret_cast<const float4&>(v).w * wk;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16* dst = out + (static_cast<int64_t>(row) * g.hq + qh) * D + lane * E;
  if constexpr (E == 4) {
    uint2 wv;
    wv.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    wv.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = wv;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
  }
  if (lse && lane == 0) lse[static_cast<int64_t>(row) * g.hq + qh] = (m + __log2f(l)) * 0.6931471805599453f;
}

template <bool E4M3, int D, bool CAP = false>
cudaError_t launch_decode_t(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                            const void* vpool, const float* ks, const float* vs, void* out, float* lse,
                            float* acc, float* ml, int* err, cudaStream_t st) {
  using C = DecodeCfg<E4M3, D>;
  cudaError_t e = ensure_smem_attr<decode_kernel<E4M3, D, CAP>>(C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_dec, g.hkv);
  decode_kernel<E4M3, D, CAP><<<grid, kThreads, C::kSmem, st>>>(
      g, p, layer, static_cast<const __nv_bfloat16*>(q), static_cast<const uint8_t*>(kpool),
      static_cast<const uint8_t*>(vpool), ks, vs, static_cast<__nv_bfloat16*>(out), lse, acc, ml, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                          const void* vpool, const float* scale_k, const float* scale_v, void* out, float* lse,
                          float* part_acc, float* part_ml, int* err, cudaStream_t st) {
  if (p.n_dec == 0) return cudaSuccess;
#define PIE_DECODE(E, DD, CP) \
  launch_decode_t<E, DD, CP>(g, p, layer, q, kpool, vpool, scale_k, scale_v, out, lse, part_acc, part_ml, err, st)
  const bool cap = g.softcap > 0.f;
  if (g.kv_dtype == 0 && g.d == 128) return cap ? PIE_DECODE(false, 128, true) : PIE_DECODE(false, 128, false);
  if (g.kv_dtype == 0 && g.d == 64) return cap ? PIE_DECODE(false, 64, true) : PIE_DECODE(false, 64, false);
  if (g.kv_dtype == 1 && g.d == 128) return cap ? PIE_DECODE(true, 128, true) : PIE_DECODE(true, 128, false);
#undef PIE_DECODE
  return cudaErrorInvalidValue;
}

namespace {
// One thread waits on an mbarrier that nothing ever completes; the bounded
// wait gives up after `polls` polls and records the timeout bit.
__global__ void wait_selftest_kernel(int* err, uint32_t polls) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, err, polls);
}
}  // namespace

cudaError_t launch_wait_selftest(int* err, uint32_t polls, cudaStream_t st) {
  wait_selftest_kernel<<<1, 1, 0, st>>>(err, polls);
  return cudaGetLastError();
}

cudaError_t launch_merge(const Geometry& g, const PlanView& p, void* out, float* lse, const float* part_acc,
                         const float* part_ml, cudaStream_t st) {
  if (p.n_merge == 0) return cudaSuccess;
  int64_t warps = static_cast<int64_t>(p.n_merge) * g.hq;
  unsigned blocks = static_cast<unsigned>((warps * 32 + 255) / 256);
  if (g.d == 128)
    merge_kernel<128><<<blocks, 256, 0, st>>>(g, p, static_cast<__nv_bfloat16*>(out), lse, part_acc, part_ml);
  else
    merge_kernel<64><<<blocks, 256, 0, st>>>(g, p, static_cast<__nv_bfloat16*>(out), lse, part_acc, part_ml);
  return cudaGetLastError();
}

}  // namespace pie

// ===========================================================================
// Decode attention that allocates nothing (pie_attend_decode_noalloc): the
// same decode and merge kernels, with the KV-split work list and the split
// partials in a file-scope device array instead of context buffers.
namespace pie {
namespace {

constexpr size_t kNoAllocBytes = PIE_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch per device ordinal, looked up once.
std::mutex g_noalloc_mu;
constexpr int kMaxDevices = 256;
void* g_noalloc_addr[kMaxDevices] = {};

// One thread per (row, split): the split's work item; split 0 also writes
// the row's entries.
__global__ void noalloc_plan(int n_rows, int n_splits, int chunk, int max_pages, const int32_t* __restrict__ seq_lens,
                             WorkItem* items, int32_t* row_pos, int32_t* row_list, int32_t* part_base,
                             int32_t* merge_rows, int32_t* merge_np) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_rows * n_splits) return;
  int r = i / n_splits, s = i % n_splits;
  int len = seq_lens[r];
  int pages = (len + kPageSize - 1) / kPageSize;
  int first = s * chunk;
  int np = min(chunk, max(0, pages - first));
  WorkItem it;
  it.pages_off = r * max_pages + first;
  it.n_pages = np;
  it.key_base = first * kPageSize;
  it.rows_off = r;
  it.n_rows = 1;
  it.part = n_splits > 1 ? s : -1;
  it.n_keys = max(0, min(np * kPageSize, len - first * kPageSize));
  it.pad = 0;
  items[i] = it;
  if (s == 0) {
    row_pos[r] = len - 1;
    row_list[r] = r;
    part_base[r] = n_splits > 1 ? r * n_splits : -1;
    merge_rows[r] = r;
    merge_np[r] = n_splits;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct NoAllocLayout {
  size_t items, row_pos, row_list, part_base, merge_rows, merge_np, acc, ml, total;
};

NoAllocLayout noalloc_layout(int64_t R, int64_t S, int64_t hq, int64_t d) {
  NoAllocLayout l{};
  size_t o = 0;
  l.items = o;
  o = align256(o + R * S * sizeof(WorkItem));
  l.row_pos = o;
  o = align256(o + R * 4);
  l.row_list = o;
  o = align256(o + R * 4);
  l.part_base = o;
  o = align256(o + R * 4);
  l.merge_rows = o;
  o = align256(o + R * 4);
  l.merge_np = o;
  o = align256(o + R * 4);
  l.acc = o;
  if (S > 1) o = align256(o + R * S * hq * d * 4);
  l.ml = o;
  if (S > 1) o = align256(o + R * S * hq * 2 * 4);
  l.total = o;
  return l;
}

}  // namespace
}  // namespace pie

extern "C" pie_status pie_attend_decode_noalloc(const pie_decode_args* a) {
  using namespace pie;
  if (!a) return PIE_ERR_INVALID;
  const int R = a->num_rows, hq = a->num_q_heads, hkv = a->num_kv_heads, d = a->head_dim;
  if (R < 0 || hq <= 0 || hkv <= 0 || hq % hkv || (d != 64 && d != 128) || a->num_layers <= 0 ||
      a->num_pages <= 0 || a->layer < 0 || a->layer >= a->num_layers || a->max_pages_per_row <= 0)
    return PIE_ERR_INVALID;
  const int G = hq / hkv;
  if (G > 64 || (G & (G - 1))) return PIE_ERR_INVALID;
  if (static_cast<int64_t>(R) * a->max_pages_per_row >= (int64_t{1} << 31)) return PIE_ERR_RANGE;
  if (R == 0) return PIE_OK;
  if (!a->q || !a->k_pool || !a->v_pool || !a->block_table || !a->seq_lens || !a->out) return PIE_ERR_INVALID;
  if (noalloc_layout(R, 1, hq, d).total > kNoAllocBytes) return PIE_ERR_RANGE;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PIE_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PIE_ERR_CUDA;
      g_noalloc_addr[dev] = ptr;
    }
    base = g_noalloc_addr[dev];
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PIE_ERR_CUDA;

  // KV splits: about 8 CTAs per SM over rows x splits x KV heads, lowered
  // until the split partials fit in the array.
  const int maxp = a->max_pages_per_row;
  int S = static_cast<int>(std::min<int64_t>(maxp, std::max<int64_t>(1, (int64_t{sms} * 8 + int64_t{hkv} * R - 1) /
                                                                              (int64_t{hkv} * R))));
  while (S > 1 && noalloc_layout(R, S, hq, d).total > kNoAllocBytes) --S;
  int chunk = (maxp + S - 1) / S;
  S = (maxp + chunk - 1) / chunk;
  const NoAllocLayout lay = noalloc_layout(R, S, hq, d);
  if (lay.total > kNoAllocBytes) return PIE_ERR_RANGE;

  uint8_t* sc = static_cast<uint8_t*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(a->stream);
  WorkItem* items = reinterpret_cast<WorkItem*>(sc + lay.items);
  int32_t* row_pos = reinterpret_cast<int32_t*>(sc + lay.row_pos);
  int32_t* row_list = reinterpret_cast<int32_t*>(sc + lay.row_list);
  int32_t* part_base = reinterpret_cast<int32_t*>(sc + lay.part_base);
  int32_t* merge_rows = reinterpret_cast<int32_t*>(sc + lay.merge_rows);
  int32_t* merge_np = reinterpret_cast<int32_t*>(sc + lay.merge_np);
  float* acc = reinterpret_cast<float*>(sc + lay.acc);
  float* ml = reinterpret_cast<float*>(sc + lay.ml);

  const int n_items = R * S;
  noalloc_plan<<<(n_items + 255) / 256, 256, 0, st>>>(R, S, chunk, maxp, a->seq_lens, items, row_pos, row_list,
                                                       part_base, merge_rows, merge_np);
  if (cudaGetLastError() != cudaSuccess) return PIE_ERR_CUDA;

  Geometry g{a->num_layers, hq, hkv, d, a->num_pages, 0, static_cast<int64_t>(kPageSize) * d * 2};
  PlanView v{};
  v.page_ids = a->block_table;
  v.row_pos = row_pos;
  v.row_slot = nullptr;
  v.row_part_base = part_base;
  v.row_list = row_list;
  v.dec_items = items;
  v.pre_items = nullptr;
  v.merge_rows = merge_rows;
  v.merge_nparts = merge_np;
  v.copies = nullptr;
  v.n_rows = R;
  v.n_dec = n_items;
  v.n_pre = 0;
  v.n_merge = S > 1 ? R : 0;
  v.n_copies = 0;
  cudaError_t e = d == 128 ? launch_decode_t<false, 128>(g, v, a->layer, a->q, a->k_pool, a->v_pool, nullptr, nullptr,
                                                         a->out, a->lse, acc, ml, nullptr, st)
                           : launch_decode_t<false, 64>(g, v, a->layer, a->q, a->k_pool, a->v_pool, nullptr, nullptr,
                                                        a->out, a->lse, acc, ml, nullptr, st);
  if (e == cudaSuccess && S > 1) e = launch_merge(g, v, a->out, a->lse, acc, ml, st);
  return e == cudaSuccess ? PIE_OK : PIE_ERR_CUDA;
}
