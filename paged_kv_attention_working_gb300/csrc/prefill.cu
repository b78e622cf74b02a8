// Ragged prefill / speculative-buffer attention over paged KV on the 5th
// generation tensor cores ("Poem ops", ops.attn.prefill; "How Pie thinks",
// section 4: the writable buffer of speculative drafts, and the shared
// frozen prefix of a fork group).
//
// One CTA takes one work item for one KV head: up to 256 query rows x query
// heads of that KV group (M, in two 128-row tiles), which all read the same
// run of pages, causally (key position <= row position).  Per 64-key tile
// (4 pages):
//   producer warp   16 one-dimensional bulk copies (K and V, 4 pages x 2
//                   panels of 2 KB) into a 3-stage ring; the pool's block
//                   layout is exactly the 128-byte-swizzled K-major (K) and
//                   MN-major (V) operand layout, so pages land ready for MMA;
//   MMA warp        S_t = Q_t K^T   (tcgen05.mma M=128 N=64 K=16, fp32 in
//                   tensor memory) for both Q tiles, then
//                   O_t += P_t V    (M=128 N=d K=16, A operand P read from
//                   tensor memory, O in tensor memory);
//   softmax warps   one warpgroup per Q tile, one thread per row: loads its
//                   S row from tensor memory (freeing S for the next tile at
//                   once), masks, keeps the running max and sum, rescales O
//                   in tensor memory only when the max grew by more than 2^8
//                   (otherwise the stale max is kept), and writes P as bf16
//                   pairs into one of two tensor-memory P buffers.
// Tensor memory: S 2 x 64 columns, P 2 x 2 x 32, O 2 x d (512 in all); with
// P there, shared memory holds Q and a 5-stage K/V ring.
// Rows with one part are normalised and written as bf16; otherwise the
// fp32 (acc, m, l) partial goes to the merge kernel.
#include <cuda_bf16.h>

#include <cmath>

#include "plan.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pie {
namespace {

constexpr int kThreadsPre = 320;  // 8 softmax warps, MMA warp, producer warp

template <int D>
struct PreCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kKeys = 64;
  static constexpr int kPagesPerTile = kKeys / kPageSize;
  static constexpr int kStages = D == 128 ? 5 : 6;
  static constexpr int kQTile = 128 * D * 2;
  static constexpr int kKVTile = kKeys * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kQTile;
  static constexpr int kOffBar = kOffKV + kStages * 2 * kKVTile;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 4 + 4;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S of tile t at t * 64
  static constexpr uint32_t kColP = 128;  // P of tile t, buffer b at 128 + t * 64 + b * 32
  static constexpr uint32_t kColO = 256;  // O of tile t at 256 + t * d
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  bool ok = mbar_wait(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreadsPre, 1)
    prefill_kernel(Geometry g, PlanView p, int layer, const __nv_bfloat16* __restrict__ q,
                   const uint8_t* __restrict__ kpool, const uint8_t* __restrict__ vpool,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_acc,
                   float* __restrict__ part_ml, int* err) {
  using C = PreCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::kStages;
  uint64_t* s_full = bars + 2 * C::kStages;  // [tile]: S(j) in tensor memory
  uint64_t* s_free = s_full + 2;             // [tile]: S(j) loaded into registers
  uint64_t* p_full = s_free + 2;             // [tile][buffer]: P(j) written
  uint64_t* o_done = p_full + 4;             // [tile][buffer]: PV(j) that read P buffer b done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);

  const WorkItem it = p.pre_items[blockIdx.x];
  const int head = blockIdx.y;
  const int G = g.hq / g.hkv;
  const int M = it.n_rows * G;
  const int n_qt = M > 128 ? 2 : 1;
  const int nkv = (it.n_keys + C::kKeys - 1) / C::kKeys;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    fence_mbar_init();
  }
  // Q tiles -> shared memory, 128-byte swizzled K-major; rows past M are zero
  {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int total = n_qt * 128 * kChunks;
    for (int idx = threadIdx.x; idx < total; idx += kThreadsPre) {
      int m = idx / kChunks, c16 = idx % kChunks;
      int t = m >> 7, r = m & 127;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m < M) {
        int row = p.row_list[it.rows_off + m / G];
        int qh = head * G + m % G;
        v = *reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(row) * g.hq + qh) * D + c16 * 8);
      }
      int panel = c16 >> 3, c = c16 & 7;
      *reinterpret_cast<uint4*>(smem + C::kOffQ + t * C::kQTile + panel * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
  }
  tc::fence_proxy_async_smem();
  if (warp == 8) {
    tc::alloc(tmem_slot, C::kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    const int64_t layer_blk = static_cast<int64_t>(layer) * g.num_pages * g.hkv;
    constexpr int kCopies = C::kPagesPerTile * C::kPanels * 2;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      const int s = j % C::kStages;
      if (j >= C::kStages) ok = warp_wait(&kv_empty[s], ((j / C::kStages) - 1) & 1, err);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[s], 2 * C::kKVTile);
      __syncwarp();
      if (lane < kCopies) {
        const int kv = lane / (C::kPagesPerTile * C::kPanels);
        const int rem = lane % (C::kPagesPerTile * C::kPanels);
        const int pg = rem / C::kPanels, panel = rem % C::kPanels;
        int pj = C::kPagesPerTile * j + pg;
        if (pj >= it.n_pages) pj = it.n_pages - 1;  // keys there are masked; any finite page will do
        const int page = p.page_ids[it.pages_off + pj];
        const int64_t off = (layer_blk + static_cast<int64_t>(page) * g.hkv + head) * g.block_bytes + panel * 2048;
        uint8_t* dst = smem + C::kOffKV + s * 2 * C::kKVTile + kv * C::kKVTile + panel * (C::kKeys * 128) + pg * 2048;
        bulk_g2s(dst, (kv ? vpool : kpool) + off, 2048, &kv_full[s]);
      }
      __syncwarp();
    }
  } else if (warp == 8) {
    // ----------------------------------------------------------------- MMA
    // One thread issues everything, event-driven: S(j) for both Q tiles as
    // soon as K tile j has landed and both tiles' S(j-1) are in registers,
    // PV(j) of a Q tile as soon as its P(j) is written; K/V stage j is
    // released right after the last PV(j).  Nothing waits on a later tile
    // to release an earlier one.
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_bf16(128, C::kKeys, false, false);
      const uint32_t id_o = tc::idesc_bf16(128, D, false, true);
      int s_next = 0;
      int pv_next[2] = {0, n_qt > 1 ? 0 : nkv};
      uint32_t idle = 0;
      while ((pv_next[0] < nkv || pv_next[1] < nkv) && idle < kWaitLimit) {
        bool progressed = false;
        if (s_next < nkv) {
          const int j = s_next, st = j % C::kStages, b = j & 1;
          bool ready = mbar_test_wait(&kv_full[st], (j / C::kStages) & 1);
          for (int t = 0; t < n_qt && ready && j > 0; ++t) ready = mbar_test_wait(&s_free[t], (j - 1) & 1);
          if (ready) {
            tc::fence_after();
            const uint32_t kaddr = sbase + C::kOffKV + st * 2 * C::kKVTile;
            for (int t = 0; t < n_qt; ++t) {
              const uint32_t d_s = tmem + C::kColS + t * C::kKeys;
              const uint32_t qaddr = sbase + C::kOffQ + t * C::kQTile;
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off_q = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint32_t off_k = (ks >> 2) * (C::kKeys * 128) + (ks & 3) * 32;
                tc::mma_bf16(d_s, tc::sw128_desc(qaddr + off_q, 16, 1024),
                             tc::sw128_desc(kaddr + off_k, 16, 1024), id_s, ks > 0);
              }
              tc::commit(&s_full[t]);
            }
            ++s_next;
            progressed = true;
          }
        }
        for (int t = 0; t < n_qt; ++t) {
          const int j = pv_next[t];
          if (j >= s_next) continue;  // S(j) not issued yet (nor P(j) written)
          const int b = j & 1;
          if (!mbar_test_wait(&p_full[2 * t + b], (j >> 1) & 1)) continue;
          tc::fence_after();
          const int st = j % C::kStages;
          const uint32_t vaddr = sbase + C::kOffKV + st * 2 * C::kKVTile + C::kKVTile;
          const uint32_t p_tmem = tmem + C::kColP + t * 64 + b * 32;  // 16 keys = 8 columns per k-step
          const uint32_t d_o = tmem + C::kColO + t * D;
#pragma unroll
          for (int ks = 0; ks < C::kKeys / 16; ++ks)
            tc::mma_bf16_ts(d_o, p_tmem + ks * 8, tc::sw128_desc(vaddr + ks * 2048, C::kKeys * 128, 1024), id_o,
                            j > 0 || ks > 0);
          tc::commit(&o_done[2 * t + b]);
          pv_next[t] = j + 1;
          progressed = true;
          // the stage is free once both tiles' PV(j) are issued (commit
          // arrives after every MMA issued so far has completed)
          const int other = n_qt > 1 ? pv_next[1 - t] : nkv;
          if (other > j) tc::commit(&kv_empty[st]);
        }
        idle = progressed ? 0 : idle + 1;
      }
      if (idle >= kWaitLimit && err) atomicOr(err, kErrWaitTimeout);
    }
    __syncwarp();
  } else if (warp / 4 < n_qt) {
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const int m = t * 128 + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) << 5) << 16;
    int row = -1, pos = -1, qh = 0;
    if (m < M) {
      row = p.row_list[it.rows_off + m / G];
      pos = p.row_pos[row];
      qh = head * G + m % G;
    }
    const float qk_scale = 1.4426950408889634f * rsqrtf(static_cast<float>(D));
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      const int b = j & 1;
      ok = warp_wait(&s_full[t], j & 1, err);
      if (!ok) break;
      tc::fence_after();
      uint32_t sr[64];
      tc::ld32(tmem + lane_base + C::kColS + t * C::kKeys, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tc::ld32(tmem + lane_base + C::kColS + t * C::kKeys + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[t]);

      // columns <= lim are visible: causal, and inside the item's key run
      // (the tile past the run's end holds stand-in pages)
      const int lim = min(pos - (it.key_base + C::kKeys * j), it.n_keys - 1 - C::kKeys * j);
      float f[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) f[c] = __uint_as_float(sr[c]);
      if (!__all_sync(0xffffffffu, lim >= 63)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) f[c] = c <= lim ? f[c] : -INFINITY;
      }
      // row max with 8 independent chains (scale > 0, so the max commutes with it)
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = f[i];
#pragma unroll
      for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], f[c]);
#pragma unroll
      for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) m8[i] = fmaxf(m8[i], m8[i + w2]);
      const float mx = m8[0] * qk_scale;
      float alpha = 1.f;
      bool resc = false;
      const float m_new = fmaxf(m_run, mx);
      if (m_new > m_run + 8.f) {
        alpha = ex2(m_run - m_new);
        m_run = m_new;
        resc = true;
      }
      const float nb = m_run == -INFINITY ? 0.f : -m_run;
      float s8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) s8[i] = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float e0 = ex2(fmaf(f[2 * c], qk_scale, nb)), e1 = ex2(fmaf(f[2 * c + 1], qk_scale, nb));
        s8[(2 * c) & 7] += e0;
        s8[(2 * c + 1) & 7] += e1;
        pk[c] = pack_bf16(e0, e1);
      }
#pragma unroll
      for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) s8[i] += s8[i + w2];
      const float sum = s8[0];
      l_run = l_run * alpha + sum;
      // P buffer b is free once PV(j-2) is done; a rescale of O needs every
      // PV so far (up to j-1) done -- commits complete in issue order.
      const bool any_resc = j > 0 && __any_sync(0xffffffffu, resc);
      if (any_resc) {
        ok = warp_wait(&o_done[2 * t + ((j - 1) & 1)], ((j - 1) >> 1) & 1, err);
      } else if (j >= 2) {
        ok = warp_wait(&o_done[2 * t + b], ((j - 2) >> 1) & 1, err);
      }
      if (!ok) break;
      tc::fence_after();
      if (any_resc) {
        {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + C::kColO + t * D + cc * 32;
            tc::ld32(ta, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st32(ta, o);
          }
          tc::wait_st();
        }
      }
      // P as bf16 pairs (key 2c in the low half of column c): the A operand of PV(j)
      tc::st32(tmem + lane_base + C::kColP + t * 64 + b * 32, pk);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[2 * t + b]);
    }
    if (ok) ok = warp_wait(&o_done[2 * t + ((nkv - 1) & 1)], ((nkv - 1) >> 1) & 1, err);
    tc::fence_after();
    if (ok) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tc::ld32(tmem + lane_base + C::kColO + t * D + cc * 32, o);
        tc::wait_ld();
        if (row < 0) continue;
        if (it.part < 0) {
          uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(row) * g.hq + qh) * D + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        } else {
          const int64_t slot = static_cast<int64_t>(p.row_part_base[row] + it.part) * g.hq + qh;
          float4* dst = reinterpret_cast<float4*>(part_acc + slot * D + cc * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                 __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
        }
      }
      if (row >= 0) {
        if (it.part < 0) {
          if (lse) lse[static_cast<int64_t>(row) * g.hq + qh] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
        } else {
          const int64_t slot = static_cast<int64_t>(p.row_part_base[row] + it.part) * g.hq + qh;
          *reinterpret_cast<float2*>(part_ml + slot * 2) = make_float2(m_run, l_run);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after();
    tc::dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_t(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                     const void* vpool, void* out, float* lse, float* acc, float* ml, int* err, cudaStream_t st) {
  using C = PreCfg<D>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(p.n_pre, g.hkv);
  prefill_kernel<D><<<grid, kThreadsPre, C::kSmem, st>>>(
      g, p, layer, static_cast<const __nv_bfloat16*>(q), static_cast<const uint8_t*>(kpool),
      static_cast<const uint8_t*>(vpool), static_cast<__nv_bfloat16*>(out), lse, acc, ml, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const Geometry& g, const PlanView& p, int layer, const void* q, const void* kpool,
                           const void* vpool, void* out, float* lse, float* part_acc, float* part_ml, int* err,
                           cudaStream_t st) {
  if (p.n_pre == 0) return cudaSuccess;
  if (g.kv_dtype != 0) return cudaErrorNotSupported;  // e4m3 prefill is not built yet
  if (g.d == 128) return launch_t<128>(g, p, layer, q, kpool, vpool, out, lse, part_acc, part_ml, err, st);
  if (g.d == 64) return launch_t<64>(g, p, layer, q, kpool, vpool, out, lse, part_acc, part_ml, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace pie
