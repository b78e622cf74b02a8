// Decode attention over paged KV ("Poem ops", ops.attn.attend) and the merge
// of split / shared partial results.
//
// One CTA takes one work item for one KV head: up to 64 query rows x query
// heads of that KV group (one decode token, a few speculative drafts, or the
// rows of a small fork / dedup group) over a run of pages of one working set.
// The item's pages stream through a ring of shared-memory stages, one 1-D
// bulk async copy per K and per V page block (the pool's block layout is
// already bank-conflict free for ldmatrix, see pie_attn.h), filled by a
// producer warp.  Four consumer warps run the products on the tensor cores
// with warp-level m16n8k16 MMA, keys and head dims on the MMA's 16-wide M
// side and the item's rows x heads on its 8-wide N side (S^T = K Q^T, O^T
// += V^T P^T), and keep an online softmax per column in registers.  With a
// single N tile the four warps take alternate pages and merge their softmax
// states at the end; with more, each warp owns one or two N tiles and every
// page is read from HBM once for all of them, which is what makes a fork
// group's shared pages cost one read per group ("How Pie thinks", section
// 4: the prompt is computed once and shared).
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
#include "launch.h"
#include "plan.h"
#include "ptx.cuh"

namespace pie {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <bool E4M3, int D, int NTW>
struct DecodeCfg {
  static constexpr int kEsize = E4M3 ? 1 : 2;
  static constexpr int kBlock = kPageSize * D * kEsize;  // bytes per page-head block
  static constexpr int kStages = E4M3 ? 12 : 8;
  // Warps that take alternate pages (up to kConsumerWarps groups) must each
  // own their stages: with the stage count a multiple of the group count a
  // stage is only ever consumed by one warp, in order, so no warp can wait
  // on a stage's phase before the previous phase of that stage completed
  // (a parity wait cannot tell the two apart).
  static_assert(kStages % kConsumerWarps == 0, "ring stages per page group");
  static constexpr int kStageBytes = 2 * kBlock;
  static constexpr int kNTW = NTW;   // N tiles (8 rows x heads each) per warp at most
  static constexpr int kMT = D / 16; // M tiles of the head dim in O^T
  static constexpr int kKS = D / 16; // k-steps of S^T
  // per thread: O^T fragments and (max, max, sum, sum) per N tile; the
  // float4 stride is odd, so 8 lanes' float4 stores hit 8 bank groups
  static constexpr int kCombineBase = kNTW * kMT * 4 + kNTW * 4;
  static constexpr int kCombineStride = (kCombineBase / 4) % 2 ? kCombineBase : kCombineBase + 4;
  static constexpr int kCombineFloats = kConsumerWarps * 32 * kCombineStride;
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kSmem = (kRing > kCombineFloats * 4 ? kRing : kCombineFloats * 4) + 2 * kStages * 8 + 16;
};

// One warp combines the np parts (m_i, l_i, acc_i) of (row, query head qh),
// stored from part index base on, in the log2 domain:
//   m = max m_i,  l = sum l_i 2^(m_i - m),  o = sum acc_i 2^(m_i - m) / l,
// and writes o (bf16) and the LSE.  Lane k holds part k's (m, l) (32 parts
// at a time), so the parts' loads are issued together; the weights reach
// every lane by shuffle, and each lane accumulates E dims of the parts'
// partial outputs with vector loads (the first eight issued with the (m, l)
// loads, the rest four at a time).  The loads bypass L1: inside a decode
// launch the parts were written by other CTAs moments earlier.
template <int D>
__device__ __forceinline__ void merge_parts(const Geometry& g, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                            const float* __restrict__ part_acc, const float* __restrict__ part_ml,
                                            int row, int np, int base, int qh, int lane) {
  auto ml_at = [&](int k) {
    return k < np ? __ldcg(reinterpret_cast<const float2*>(part_ml + (static_cast<int64_t>(base + k) * g.hq + qh) * 2))
                  : make_float2(-INFINITY, 0.f);
  };
  constexpr int E = D / 32;
  using Vec = typename std::conditional<E == 4, float4, float2>::type;
  const float* a = part_acc + (static_cast<int64_t>(base) * g.hq + qh) * D + lane * E;
  const int64_t part_stride = static_cast<int64_t>(g.hq) * D;
  // The first kPre parts' partial outputs are loaded together with the (m, l)
  // values (they do not depend on the weights): one round trip to L2 fewer
  // before the sums, which is most of this kernel's time in a small pass.
  constexpr int kPre = 8;
  Vec pre[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    if (k < np) {
      pre[k] = __ldcg(reinterpret_cast<const Vec*>(a + k * part_stride));
    } else {
      reinterpret_cast<float*>(&pre[k])[0] = 0.f;
      reinterpret_cast<float*>(&pre[k])[1] = 0.f;
      if constexpr (E == 4) {
        reinterpret_cast<float*>(&pre[k])[2] = 0.f;
        reinterpret_cast<float*>(&pre[k])[3] = 0.f;
      }
    }
  }
  const float2 ml0 = ml_at(lane);
  float m = ml0.x;
  for (int k0 = 32; k0 < np; k0 += 32) m = fmaxf(m, ml_at(k0 + lane).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float base_m = m == -INFINITY ? 0.f : m;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  auto add = [&](const Vec& v, float wk) {
    acc[0] += v.x * wk;
    acc[1] += v.y * wk;
    if constexpr (E == 4) {
      acc[2] += reinterpret_cast<const float4&>(v).z * wk;
      acc[3] += reinterpret_cast<const float4&>(v).w * wk;
    }
  };
  float l = 0.f;
  for (int k0 = 0; k0 < np; k0 += 32) {
    const float2 ml = k0 == 0 ? ml0 : ml_at(k0 + lane);
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - base_m);
    l += ml.y * w;
    const int n = min(32, np - k0);
    if (k0 == 0) {
#pragma unroll
      for (int kk = 0; kk < kPre; ++kk) add(pre[kk], __shfl_sync(0xffffffffu, w, kk));
    }
    const int first = k0 == 0 ? kPre : 0;
#pragma unroll 4
    for (int kk = first; kk < n; ++kk)
      add(__ldcg(reinterpret_cast<const Vec*>(a + (k0 + kk) * part_stride)), __shfl_sync(0xffffffffu, w, kk));
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

// Merge inside the attention launch: a warp has just stored its partial
// results for the columns (colrow[e], colqh[e]) of one N tile (the 8 lanes
// of one tq hold the same two columns).  Each (row, query head) has a
// counter of the parts stored so far; one lane per column counts its part,
// and the warp that stores a column's last part resets the counter and
// combines the column's parts at once, so no separate merge launch follows.
// Each column lies in one warp's N tile per CTA, and each of the row's parts
// is one CTA, so the count reaches the row's number of parts exactly once.
template <int D>
__device__ __forceinline__ void count_and_merge(const Geometry& g, const PlanView& p, __nv_bfloat16* out, float* lse,
                                                const float* part_acc, const float* part_ml, const int (&colrow)[2],
                                                const int (&colqh)[2], int gq, int lane) {
  __threadfence();  // this lane's partial stores, before the count
  __syncwarp();
  uint32_t last = 0;
  if (gq == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (colrow[e] < 0) continue;
      const int i = p.row_merge[colrow[e]];
      int* cnt = p.merge_cnt + static_cast<int64_t>(i) * g.hq + colqh[e];
      if (atomicAdd(cnt, 1) == p.merge_info[i].y - 1) {
        *cnt = 0;  // every part is counted: the next launch starts from zero
        last |= 1u << e;
      }
    }
  }
  __threadfence();  // the other parts' stores, before the loads of the merge
  __syncwarp();
  uint32_t todo = __ballot_sync(0xffffffffu, last != 0);
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const uint32_t cols = __shfl_sync(0xffffffffu, last, src);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = __shfl_sync(0xffffffffu, colrow[e], src), qh = __shfl_sync(0xffffffffu, colqh[e], src);
      if (cols >> e & 1u) {
        const int4 mi = p.merge_info[p.row_merge[row]];
        merge_parts<D>(g, out, lse, part_acc, part_ml, row, mi.y, mi.z, qh, lane);
      }
    }
  }
}

template <bool E4M3, int D, bool CAP, int NTW>
__global__ void __launch_bounds__(kThreads, NTW == 1 ? 4 : 3) decode_kernel(Geometry g, PlanView p, int layer,
                                                          const __nv_bfloat16* __restrict__ q,
                                                          const uint8_t* __restrict__ kpool,
                                                          const uint8_t* __restrict__ vpool,
                                                          const float* __restrict__ kscale,
                                                          const float* __restrict__ vscale,
                                                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                          float* __restrict__ part_acc, float* __restrict__ part_ml,
                                                          int* err) {
  using C = DecodeCfg<E4M3, D, NTW>;
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (C::kSmem - 2 * C::kStages * 8 - 16));
  uint64_t* empty = full + C::kStages;

  const WorkItem it = p.dec_items[blockIdx.x];
  const int head = blockIdx.y;
  const int G = g.hq / g.hkv;
  const int M = it.n_rows * G;
  // N tiles of 8 rows x heads; owner warps hold two each and read every page
  // of the item, the others take alternate pages (n_grp groups)
  const int n_nt = (M + 7) >> 3;
  const int n_own = n_nt <= C::kNTW ? 1 : (n_nt <= 2 * C::kNTW ? 2 : 4);  // n_nt <= 4 * kNTW
  const int n_grp = kConsumerWarps / n_own;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t layer_blk = (static_cast<int64_t>(layer) * g.num_pages) * g.hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_own);
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
  // Keys and head dims are the MMA's M side, the item's rows x query heads
  // its N side: S^T = K Q^T (M = 16 keys, N = 8 columns, K = head dim) and
  // O^T += V^T P^T (M = 16 dims, N = 8 columns, K = 16 keys).  A decode row
  // of 4 or 8 query heads then fills half or all of an 8-wide N tile instead
  // of a quarter or half of a 16-row M tile, which halves the MMAs and the
  // softmax work per page.  Thread (g = lane / 4, t = lane % 4) holds, per
  // N tile, the scores of keys g and g + 8 for columns 2t and 2t + 1, and
  // the B fragment of Q^T for column g.
  const int ow = warp % n_own, grp = warp / n_own;
  const int ntw = max(0, min(C::kNTW, n_nt - C::kNTW * ow));  // N tiles of this warp
  const int gq = lane >> 2, tq = lane & 3;
  const float kdq = E4M3 ? kscale[layer * g.hkv + head] : 1.0f;
  const float vdq = E4M3 ? vscale[layer * g.hkv + head] : 1.0f;
  // scores in log2 units: s * qk_scale, or with the soft cap c,
  // tanh(s * cap_pre) * cap_post = c * tanh(s / c) * log2(e)
  const float qk_scale = kdq * rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;
  const float cap_pre = CAP ? kdq * rsqrtf(static_cast<float>(D)) / g.softcap : 0.f;
  const float cap_post = CAP ? g.softcap * 1.4426950408889634f : 0.f;

  // Q^T as B fragments: qb[i][ks] = (k 2t, 2t+1 ; column g) (k 2t+8, 2t+9 ;
  // column g).  e4m3: k slots 2t, 2t+1, 2t+8, 2t+9 of a 16-dim step are dims
  // 4t .. 4t+3 (the order the e4m3 K bytes arrive in; the sum over k is the
  // same).  colpos[i][e]: position of the row of column 2t + e (-1 = none).
  uint32_t qb[C::kNTW][C::kKS][2];
  int colpos[C::kNTW][2];
#pragma unroll
  for (int i = 0; i < C::kNTW; ++i) {
    const int mq = 8 * (C::kNTW * ow + i) + gq;
    const __nv_bfloat16* qp = nullptr;
    if (i < ntw && mq < M)
      qp = q + (static_cast<int64_t>(item_row(p, it, mq / G)) * g.hq + head * G + mq % G) * D;
#pragma unroll
    for (int ks = 0; ks < C::kKS; ++ks) {
      uint32_t b0 = 0, b1 = 0;
      if (qp) {
        if constexpr (!E4M3) {
          b0 = __ldcg(reinterpret_cast<const unsigned int*>(qp + 16 * ks + 2 * tq));
          b1 = __ldcg(reinterpret_cast<const unsigned int*>(qp + 16 * ks + 8 + 2 * tq));
        } else {
          const uint2 w = __ldcg(reinterpret_cast<const uint2*>(qp + 16 * ks + 4 * tq));
          b0 = pack_f16(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
          b1 = pack_f16(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        }
      }
      qb[i][ks][0] = b0;
      qb[i][ks][1] = b1;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int m = 8 * (C::kNTW * ow + i) + 2 * tq + e;
      colpos[i][e] = i < ntw && m < M ? p.row_pos[item_row(p, it, m / G)] : -1;
    }
  }

  // O^T accumulators: o[i][mt] = (dim row g, columns 2t, 2t+1), (dim row
  // g + 8, columns 2t, 2t+1) of M tile mt; bf16 rows are dims 16mt + g and
  // 16mt + g + 8, e4m3 rows dims 16mt + 2g and 16mt + 2g + 1.
  float o[C::kNTW][C::kMT][4];
#pragma unroll
  for (int i = 0; i < C::kNTW; ++i)
#pragma unroll
    for (int mt = 0; mt < C::kMT; ++mt) o[i][mt][0] = o[i][mt][1] = o[i][mt][2] = o[i][mt][3] = 0.f;
  // per column: the running reference max (log2 units) and this thread's
  // share of the row sum (keys g and g + 8 of every page it saw)
  float mx[C::kNTW][2], sum[C::kNTW][2];
#pragma unroll
  for (int i = 0; i < C::kNTW; ++i) mx[i][0] = mx[i][1] = -INFINITY, sum[i][0] = sum[i][1] = 0.f;

  for (int j = grp; j < it.n_pages; j += n_grp) {
    const int s = j % C::kStages;
    // warp-uniform: the shuffles and MMAs below need every lane
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / C::kStages) & 1, err))) break;
    if (ntw > 0) {
      const uint32_t kb = smem_u32(smem + s * C::kStageBytes);
      const uint32_t vb = kb + C::kBlock;

      // ---- S^T = K Q^T: A = K (16 keys x 16 dims per step) by ldmatrix:
      // matrices (keys 0-7, low chunk) (keys 8-15, low) (keys 0-7, high) (keys 8-15, high)
      float sc[C::kNTW][4];
#pragma unroll
      for (int i = 0; i < C::kNTW; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      const int key = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int csel = lane >> 4;
      if constexpr (!E4M3) {
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          const int c = 2 * (ks & 3) + csel;
          uint32_t a[4];
          ldsm_x4(kb + (ks >> 2) * 2048 + key * 128 + 16 * (c ^ (key & 7)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int i = 0; i < C::kNTW; ++i)
            if (i < ntw) mma16816<true>(sc[i], a, qb[i][ks][0], qb[i][ks][1]);
        }
      } else {
        // e4m3 bytes: (keys 0-7, chunk 2kp) (keys 8-15, 2kp) (keys 0-7, 2kp+1)
        // (keys 8-15, 2kp+1); a lane's 4 bytes are dims 4t .. 4t+3 of its key
#pragma unroll
        for (int kp = 0; kp < C::kKS / 2; ++kp) {
          const int c = 2 * kp + csel;
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + key * 128 + 16 * (c ^ (key & 7)), r0, r1, r2, r3);
          const uint32_t a0[4] = {e4m3x2_lo_to_f16x2(r0), e4m3x2_lo_to_f16x2(r1), e4m3x2_hi_to_f16x2(r0),
                                  e4m3x2_hi_to_f16x2(r1)};
          const uint32_t a1[4] = {e4m3x2_lo_to_f16x2(r2), e4m3x2_lo_to_f16x2(r3), e4m3x2_hi_to_f16x2(r2),
                                  e4m3x2_hi_to_f16x2(r3)};
#pragma unroll
          for (int i = 0; i < C::kNTW; ++i)
            if (i < ntw) {
              mma16816<false>(sc[i], a0, qb[i][2 * kp][0], qb[i][2 * kp][1]);
              mma16816<false>(sc[i], a1, qb[i][2 * kp + 1][0], qb[i][2 * kp + 1][1]);
            }
        }
      }

      // ---- mask, online softmax per column (log2 domain); P^T to B fragments
      const int kpos0 = it.key_base + 16 * j + gq, kpos1 = kpos0 + 8;
      uint32_t pb[C::kNTW][2];
#pragma unroll
      for (int i = 0; i < C::kNTW; ++i) {
        if (i >= ntw) break;
        float v[2][2];  // [column e][key g, g + 8]
        bool grow = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if constexpr (CAP) {
            v[e][0] = kpos0 <= colpos[i][e] ? tanh_approx(sc[i][e] * cap_pre) * cap_post : -INFINITY;
            v[e][1] = kpos1 <= colpos[i][e] ? tanh_approx(sc[i][2 + e] * cap_pre) * cap_post : -INFINITY;
          } else {
            v[e][0] = kpos0 <= colpos[i][e] ? sc[i][e] * qk_scale : -INFINITY;
            v[e][1] = kpos1 <= colpos[i][e] ? sc[i][2 + e] * qk_scale : -INFINITY;
          }
          grow |= fmaxf(v[e][0], v[e][1]) > mx[i][e] + 8.f;
        }
        // The reference max of a column only moves when one of its scores
        // exceeds it by more than 8 (log2 units): weights stay <= 2^8 and the
        // column's 8 lanes must agree on it, so the cross-lane max is taken
        // only then (after the first page, rarely).
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float best = fmaxf(v[e][0], v[e][1]);
            best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 4));
            best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 8));
            best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 16));
            if (best > mx[i][e] + 8.f) {
              const float alpha = mx[i][e] == -INFINITY ? 0.f : ex2(mx[i][e] - best);
              sum[i][e] *= alpha;
#pragma unroll
              for (int mt = 0; mt < C::kMT; ++mt) {
                o[i][mt][e] *= alpha;
                o[i][mt][2 + e] *= alpha;
              }
              mx[i][e] = best;
            }
          }
        }
        float w[2][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float base = mx[i][e] == -INFINITY ? 0.f : mx[i][e];
          w[e][0] = ex2(v[e][0] - base);
          w[e][1] = ex2(v[e][1] - base);
          sum[i][e] += w[e][0] + w[e][1];
        }
        // (key g: columns 2t, 2t+1) and (key g + 8: ...) are 8x8 blocks in
        // the layout ldmatrix gives; transposed they are the B fragment
        // (keys 2t, 2t+1 ; column g) and (keys 2t+8, 2t+9 ; column g)
        pb[i][0] = movmatrix_t(E4M3 ? pack_f16(w[0][0], w[1][0]) : pack_bf16(w[0][0], w[1][0]));
        pb[i][1] = movmatrix_t(E4M3 ? pack_f16(w[0][1], w[1][1]) : pack_bf16(w[0][1], w[1][1]));
      }

      // ---- O^T += V^T P^T: A = V^T (16 dims x 16 keys) by transposing ldmatrix
      if constexpr (!E4M3) {
        // matrices (keys 0-7, dims 16mt..+7) (keys 0-7, +8..+15) (keys 8-15, ..) (keys 8-15, ..)
        const int vkey = (lane & 7) + ((lane >> 4) << 3);
        const int vch = (lane >> 3) & 1;
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          const int c = 2 * (mt & 3) + vch;
          uint32_t a[4];
          ldsm_x4_t(vb + (mt >> 2) * 2048 + vkey * 128 + 16 * (c ^ (vkey & 7)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int i = 0; i < C::kNTW; ++i)
            if (i < ntw) mma16816<true>(o[i][mt], a, pb[i][0], pb[i][1]);
        }
      } else {
        // 16-bit units of two e4m3 dims: matrices (keys 0-7, chunk 2cp) (keys
        // 8-15, 2cp) (keys 0-7, 2cp+1) (keys 8-15, 2cp+1); a lane gets (key 2t:
        // dims 2g, 2g+1) (key 2t+1: dims 2g, 2g+1) and one byte permute pairs
        // the keys per dim: M rows g and g + 8 are dims 2g and 2g + 1
        const int vkey = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int vsel = lane >> 4;
#pragma unroll
        for (int cp = 0; cp < D / 32; ++cp) {
          const int c = 2 * cp + vsel;
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vb + vkey * 128 + 16 * (c ^ (vkey & 7)), r0, r1, r2, r3);
          const uint32_t x0 = prmt(r0, r0, 0x3120), x1 = prmt(r1, r1, 0x3120);
          const uint32_t x2 = prmt(r2, r2, 0x3120), x3 = prmt(r3, r3, 0x3120);
          const uint32_t a0[4] = {e4m3x2_lo_to_f16x2(x0), e4m3x2_hi_to_f16x2(x0), e4m3x2_lo_to_f16x2(x1),
                                  e4m3x2_hi_to_f16x2(x1)};
          const uint32_t a1[4] = {e4m3x2_lo_to_f16x2(x2), e4m3x2_hi_to_f16x2(x2), e4m3x2_lo_to_f16x2(x3),
                                  e4m3x2_hi_to_f16x2(x3)};
#pragma unroll
          for (int i = 0; i < C::kNTW; ++i)
            if (i < ntw) {
              mma16816<false>(o[i][2 * cp], a0, pb[i][0], pb[i][1]);
              mma16816<false>(o[i][2 * cp + 1], a1, pb[i][0], pb[i][1]);
            }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- finish: each column's sum over its 8 lanes, then merge the warps
  // that took alternate pages of the same columns
#pragma unroll
  for (int i = 0; i < C::kNTW; ++i)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      sum[i][e] += __shfl_xor_sync(0xffffffffu, sum[i][e], 4);
      sum[i][e] += __shfl_xor_sync(0xffffffffu, sum[i][e], 8);
      sum[i][e] += __shfl_xor_sync(0xffffffffu, sum[i][e], 16);
    }
  if (n_grp > 1) {
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32));
    float* cm = reinterpret_cast<float*>(smem);
    float* mine = cm + (warp * 32 + lane) * C::kCombineStride;
    if (grp > 0) {
#pragma unroll
      for (int i = 0; i < C::kNTW; ++i) {
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
          *reinterpret_cast<float4*>(mine + (i * C::kMT + mt) * 4) =
              make_float4(o[i][mt][0], o[i][mt][1], o[i][mt][2], o[i][mt][3]);
        *reinterpret_cast<float4*>(mine + (C::kNTW * C::kMT + i) * 4) =
            make_float4(mx[i][0], mx[i][1], sum[i][0], sum[i][1]);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32));
    if (grp > 0) return;
    for (int og = 1; og < n_grp; ++og) {
      const float* th = cm + ((og * n_own + ow) * 32 + lane) * C::kCombineStride;
#pragma unroll
      for (int i = 0; i < C::kNTW; ++i) {
        const float4 st = *reinterpret_cast<const float4*>(th + (C::kNTW * C::kMT + i) * 4);
        const float m2[2] = {st.x, st.y}, l2[2] = {st.z, st.w};
        float a1[2], a2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mnew = fmaxf(mx[i][e], m2[e]);
          const float base = mnew == -INFINITY ? 0.f : mnew;
          a1[e] = ex2(mx[i][e] - base);
          a2[e] = ex2(m2[e] - base);
          sum[i][e] = sum[i][e] * a1[e] + l2[e] * a2[e];
          mx[i][e] = mnew;
        }
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          const float4 v = *reinterpret_cast<const float4*>(th + (i * C::kMT + mt) * 4);
          o[i][mt][0] = o[i][mt][0] * a1[0] + v.x * a2[0];
          o[i][mt][1] = o[i][mt][1] * a1[1] + v.y * a2[1];
          o[i][mt][2] = o[i][mt][2] * a1[0] + v.z * a2[0];
          o[i][mt][3] = o[i][mt][3] * a1[1] + v.w * a2[1];
        }
      }
    }
  }

  // ---- write: direct bf16 output, or fp32 partial (acc, m, l) for merging
#pragma unroll
  for (int i = 0; i < C::kNTW; ++i) {
    if (i >= ntw) break;
    const int nt = C::kNTW * ow + i;
    int colrow[2], colqh[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int m = 8 * nt + 2 * tq + e;
      colrow[e] = m < M ? item_row(p, it, m / G) : -1;
      colqh[e] = head * G + m % G;
    }
    if (it.part < 0) {
      float inv[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) inv[e] = sum[i][e] > 0.f ? vdq / sum[i][e] : 0.f;
      if constexpr (!E4M3) {
        // transpose (dim g: columns 2t, 2t+1) blocks to (column g: dims 2t,
        // 2t+1): each lane then stores whole bf16 pairs of one head
        const int m = 8 * nt + gq;
        __nv_bfloat16* dst =
            m < M ? out + (static_cast<int64_t>(item_row(p, it, m / G)) * g.hq + head * G + m % G) * D
                  : nullptr;
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          const uint32_t lo = movmatrix_t(pack_bf16(o[i][mt][0] * inv[0], o[i][mt][1] * inv[1]));
          const uint32_t hi = movmatrix_t(pack_bf16(o[i][mt][2] * inv[0], o[i][mt][3] * inv[1]));
          if (dst) {
            *reinterpret_cast<uint32_t*>(dst + 16 * mt + 2 * tq) = lo;
            *reinterpret_cast<uint32_t*>(dst + 16 * mt + 8 + 2 * tq) = hi;
          }
        }
      } else {
        // rows g and g + 8 of M tile mt are dims 16mt + 2g and 16mt + 2g + 1
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (colrow[e] < 0) continue;
          __nv_bfloat16* dst = out + (static_cast<int64_t>(colrow[e]) * g.hq + colqh[e]) * D;
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt)
            *reinterpret_cast<uint32_t*>(dst + 16 * mt + 2 * gq) =
                pack_bf16(o[i][mt][e] * inv[e], o[i][mt][2 + e] * inv[e]);
        }
      }
      if (lse && gq == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (colrow[e] >= 0)
            lse[static_cast<int64_t>(colrow[e]) * g.hq + colqh[e]] = (mx[i][e] + __log2f(sum[i][e])) * 0.6931471805599453f;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (colrow[e] < 0) continue;
        const int64_t slot = static_cast<int64_t>(p.row_part_base[colrow[e]] + it.part) * g.hq + colqh[e];
        float* dst = part_acc + slot * D;
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          if constexpr (!E4M3) {
            dst[16 * mt + gq] = o[i][mt][e] * vdq;
            dst[16 * mt + 8 + gq] = o[i][mt][2 + e] * vdq;
          } else {
            *reinterpret_cast<float2*>(dst + 16 * mt + 2 * gq) = make_float2(o[i][mt][e] * vdq, o[i][mt][2 + e] * vdq);
          }
        }
        if (gq == 0) *reinterpret_cast<float2*>(part_ml + slot * 2) = make_float2(mx[i][e], sum[i][e]);
      }
      if (p.merge_cnt) count_and_merge<D>(g, p, out, lse, part_acc, part_ml, colrow, colqh, gq, lane);
    }
  }
}

// One warp per (merged row, query head): the separate merge launch, for
// passes whose split rows are not merged inside the attention kernels.
template <int D>
__global__ void merge_kernel(Geometry g, PlanView p, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                             const float* __restrict__ part_acc, const float* __restrict__ part_ml) {
  pdl_wait();
  pdl_trigger();
  int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= p.n_merge * g.hq) return;
  const int4 mi = p.merge_info[wid / g.hq];  // one load: (row, parts, first part)
  merge_parts<D>(g, out, lse, part_acc, part_ml, mi.x, mi.y, mi.z, wid % g.hq, lane);
}

template <bool E4M3, int D, bool CAP, int NTW>
cudaError_t launch_decode_t(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                            const void* vpool, const float* ks, const float* vs, void* out, float* lse,
                            float* acc, float* ml, int* err, cudaStream_t st) {
  using C = DecodeCfg<E4M3, D, NTW>;
  cudaError_t e = ensure_smem_attr<decode_kernel<E4M3, D, CAP, NTW>>(C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_dec, g.hkv);
  e = launch_pdl(decode_kernel<E4M3, D, CAP, NTW>, grid, kThreads, C::kSmem, st, g, p, layer,
                 static_cast<const __nv_bfloat16*>(q), static_cast<const uint8_t*>(kpool),
                 static_cast<const uint8_t*>(vpool), ks, vs, static_cast<__nv_bfloat16*>(out), lse, acc, ml, err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Items of up to kDecodeNarrowM rows x heads take one N tile per warp (96
// registers: 4 CTAs per SM where the shared memory allows, e4m3 pages); a
// launch with wider items (fork / dedup groups of up to 64) takes two.
template <bool E4M3, int D, bool CAP>
cudaError_t launch_decode_n(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                            const void* vpool, const float* ks, const float* vs, void* out, float* lse,
                            float* acc, float* ml, int* err, cudaStream_t st) {
  return p.max_dec_m > kDecodeNarrowM
             ? launch_decode_t<E4M3, D, CAP, 2>(g, p, layer, q, kpool, vpool, ks, vs, out, lse, acc, ml, err, st)
             : launch_decode_t<E4M3, D, CAP, 1>(g, p, layer, q, kpool, vpool, ks, vs, out, lse, acc, ml, err, st);
}

}  // namespace

cudaError_t launch_decode(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                          const void* vpool, const float* scale_k, const float* scale_v, void* out, float* lse,
                          float* part_acc, float* part_ml, int* err, cudaStream_t st) {
  if (p.n_dec == 0) return cudaSuccess;
#define PIE_DECODE(E, DD, CP) \
  launch_decode_n<E, DD, CP>(g, p, layer, q, kpool, vpool, scale_k, scale_v, out, lse, part_acc, part_ml, err, st)
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
  const cudaError_t e =
      g.d == 128 ? launch_pdl(merge_kernel<128>, blocks, 256, 0, st, g, p, static_cast<__nv_bfloat16*>(out), lse,
                              part_acc, part_ml)
                 : launch_pdl(merge_kernel<64>, blocks, 256, 0, st, g, p, static_cast<__nv_bfloat16*>(out), lse,
                              part_acc, part_ml);
  return e != cudaSuccess ? e : cudaGetLastError();
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
                             int4* merge_info) {
  pdl_wait();
  pdl_trigger();
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
  it.direct_rows = 1;  // row_list[r] = r
  items[i] = it;
  if (s == 0) {
    row_pos[r] = len - 1;
    row_list[r] = r;
    part_base[r] = n_splits > 1 ? r * n_splits : -1;
    merge_info[r] = make_int4(r, n_splits, r * n_splits, 0);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct NoAllocLayout {
  size_t items, row_pos, row_list, part_base, merge_info, acc, ml, total;
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
  l.merge_info = o;
  o = align256(o + R * 16);
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
  {
    auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; };
    if (!al(a->q, 16) || !al(a->k_pool, 16) || !al(a->v_pool, 16) || !al(a->out, 16) || !al(a->block_table, 4) ||
        !al(a->seq_lens, 4) || !al(a->lse, 4))
      return PIE_ERR_INVALID;
  }
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
  int4* merge_info = reinterpret_cast<int4*>(sc + lay.merge_info);
  float* acc = reinterpret_cast<float*>(sc + lay.acc);
  float* ml = reinterpret_cast<float*>(sc + lay.ml);

  const int n_items = R * S;
  if (launch_pdl(noalloc_plan, (n_items + 255) / 256, 256, 0, st, R, S, chunk, maxp, a->seq_lens, items, row_pos,
                 row_list, part_base, merge_info) != cudaSuccess ||
      cudaGetLastError() != cudaSuccess)
    return PIE_ERR_CUDA;

  Geometry g{a->num_layers, hq, hkv, d, a->num_pages, 0, static_cast<int64_t>(kPageSize) * d * 2};
  PlanView v{};
  v.page_ids = a->block_table;
  v.row_pos = row_pos;
  v.row_slot = nullptr;
  v.row_part_base = part_base;
  v.row_list = row_list;
  v.dec_items = items;
  v.pre_items = nullptr;
  v.merge_info = merge_info;
  v.copies = nullptr;
  v.n_rows = R;
  v.n_dec = n_items;
  v.n_pre = 0;
  v.n_merge = S > 1 ? R : 0;
  v.n_copies = 0;
  v.max_dec_m = G;
  cudaError_t e = d == 128 ? launch_decode_n<false, 128, false>(g, v, a->layer, a->q, a->k_pool, a->v_pool, nullptr,
                                                                nullptr, a->out, a->lse, acc, ml, nullptr, st)
                           : launch_decode_n<false, 64, false>(g, v, a->layer, a->q, a->k_pool, a->v_pool, nullptr,
                                                               nullptr, a->out, a->lse, acc, ml, nullptr, st);
  if (e == cudaSuccess && S > 1) e = launch_merge(g, v, a->out, a->lse, acc, ml, st);
  return e == cudaSuccess ? PIE_OK : PIE_ERR_CUDA;
}
