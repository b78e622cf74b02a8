// Ragged prefill / speculative-buffer attention over paged KV on the 5th
// generation tensor cores ("Poem ops", ops.attn.prefill; "How Pie thinks",
// section 4: the writable buffer of speculative drafts, and the shared
// frozen prefix of a fork group).
//
// One CTA takes one work item for one KV head: up to 256 query rows x query
// heads of that KV group (M, in two 128-row tiles t = 0, 1), which all read
// the same run of pages, causally (key position <= row position).  Keys go
// in tiles of 128 (8 pages):
//   producer warps  one for K, one for V (each issue of a bulk copy costs
//                   about a hundred cycles, so one warp for both lagged):
//                   2-KB page panels into a K ring, whole page blocks into a
//                   V ring (separate rings, so a K tile is refilled as soon
//                   as both S products have read it); the pool's block
//                   layout is the 128-byte-swizzled operand layout, so pages
//                   land ready for the tensor cores (K-major for K, MN-major
//                   for V, one page per K = 16 step);
//   MMA thread      event-driven issue of S_t = Q_t K^T (tcgen05.mma M=128
//                   N=128 K=16, fp32 in tensor memory) and O_t += P_t V
//                   (M=128 N=d K=16, A = P read from tensor memory, O in
//                   tensor memory); S_t(j+1) overwrites S_t(j) / P_t(j), so it
//                   is issued once PV_t(j) has completed -- the two Q tiles
//                   keep the tensor pipe busy in turn;
//   softmax warps   one warpgroup per Q tile, one thread per row: loads its
//                   128-score S row from tensor memory, takes the row max,
//                   keeps the running max stale unless the row max grew by
//                   more than 2^8 (then O is rescaled in tensor memory),
//                   computes the weights with packed f32x2 arithmetic and
//                   writes P back as bf16 pairs over the row's first 64 S
//                   columns.
// Tensor memory: S/P of tile t at columns t*128, O of tile t at 256 + t*d.
// Q tiles: items whose rows are in batch order take them by tensor copies
// (one box of a 3-D map over [rows][Hq][d] per 64-column panel), the others
// by the softmax warps' cp.async copies.  Rows with one part are normalised
// and written as bf16; otherwise the fp32 (acc, m, l) partial goes to the
// merge kernel; either way through the tile's Q buffer, whole rows per store.
//
// With a logit soft cap c (CAP), the softmax warps map each raw score to
// tanh(s * scale / c) before masking, and c * log2(e) takes the place of the
// score scale.
//
// e4m3 pools (d = 128): the tensor cores take the dequantised codes.  The
// producer copies raw e4m3 page blocks into a small staging ring; two
// converter warps turn each 16-key page into f16 (every e4m3 value is exact
// in f16) at its place in the 128-byte-swizzled K / V tile, and hand the
// tile to the MMA thread.  Q is rounded to f16 on load and P is written as
// f16 pairs, so both products are f16 x f16 with fp32 accumulation; the
// per-(layer, KV head) scales fold into the softmax scale (K) and the
// output (V), as in the decode kernel.
#include <cuda_bf16.h>

#include <cmath>

#include "launch.h"
#include "plan.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pie {
namespace {

// Warps 0-7 softmax, warp 8 MMA; bf16: warp 9 produces K and warp 10 V;
// e4m3: warp 9 produces raw K and V, warps 10 and 11 convert them.
template <int D, bool E4M3>
struct PreCfg {
  static constexpr int kThreads = E4M3 ? 384 : 352;
  static constexpr int kPanels = D / 64;
  static constexpr int kKeys = 128;                       // keys per tile
  static constexpr int kPagesPerTile = kKeys / kPageSize;  // 8
  static constexpr int kQTile = 128 * D * 2;
  static constexpr int kKVTile = kKeys * D * 2;            // one K (or V) tile, 16-bit elements
  static constexpr int kPanelBytes = kKeys * 128;          // one 64-column panel of a tile
  static constexpr int kKStages = E4M3 ? 2 : (D == 128 ? 3 : 4);
  static constexpr int kVStages = E4M3 ? 2 : (D == 128 ? 2 : 3);
  static constexpr int kRawRing = 2;                       // e4m3 staging: K(j), V(j) alternate
  static constexpr int kRawStages = E4M3 ? kRawRing : 0;
  static constexpr int kRawTile = kKeys * D;               // one e4m3 tile (8 page blocks)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQTile;
  static constexpr int kOffV = kOffK + kKStages * kKVTile;
  static constexpr int kOffRaw = kOffV + kVStages * kKVTile;
  static constexpr int kOffBar = kOffRaw + kRawStages * kRawTile;
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 * kRawStages + 2;
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;
};

// Position given to rows past an item's last row: after every key.
constexpr int kNoRowPos = 0x3fffffff;

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two softmax weights: e = 2^(s * scale + nb) for a pair of scores (one
// packed f32x2 FMA, two ex2), added to a packed pair of running sums;
// returns the pair as bf16x2, or f16x2 when F16 (element 0 low).
template <bool F16>
__device__ __forceinline__ uint32_t softmax_pair(float s0, float s1, float scale, float nb, uint64_t& acc) {
  uint32_t pk;
  if constexpr (F16) {
    asm("{\n"
        " .reg .b64 s, k, n, x, e;\n"
        " .reg .f32 x0, x1, e0, e1;\n"
        " mov.b64 s, {%2, %3};\n"
        " mov.b64 k, {%4, %4};\n"
        " mov.b64 n, {%5, %5};\n"
        " fma.rn.f32x2 x, s, k, n;\n"
        " mov.b64 {x0, x1}, x;\n"
        " ex2.approx.ftz.f32 e0, x0;\n"
        " ex2.approx.ftz.f32 e1, x1;\n"
        " mov.b64 e, {e0, e1};\n"
        " add.rn.f32x2 %1, %1, e;\n"
        " cvt.rn.f16x2.f32 %0, e1, e0;\n"
        "}"
        : "=r"(pk), "+l"(acc)
        : "f"(s0), "f"(s1), "f"(scale), "f"(nb));
  } else {
    asm("{\n"
        " .reg .b64 s, k, n, x, e;\n"
        " .reg .f32 x0, x1, e0, e1;\n"
        " mov.b64 s, {%2, %3};\n"
        " mov.b64 k, {%4, %4};\n"
        " mov.b64 n, {%5, %5};\n"
        " fma.rn.f32x2 x, s, k, n;\n"
        " mov.b64 {x0, x1}, x;\n"
        " ex2.approx.ftz.f32 e0, x0;\n"
        " ex2.approx.ftz.f32 e1, x1;\n"
        " mov.b64 e, {e0, e1};\n"
        " add.rn.f32x2 %1, %1, e;\n"
        " cvt.rn.bf16x2.f32 %0, e1, e0;\n"
        "}"
        : "=r"(pk), "+l"(acc)
        : "f"(s0), "f"(s1), "f"(scale), "f"(nb));
  }
  return pk;
}

// Eight bf16 (one 16-byte chunk) -> eight f16, round to nearest even.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  auto cv = [](uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    return pack_f16(lo, hi);
  };
  return make_uint4(cv(v.x), cv(v.y), cv(v.z), cv(v.w));
}

__device__ __forceinline__ float sum_pair(uint64_t acc) {
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(acc));
  return a + b;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err) {
  bool ok = mbar_wait(bar, parity, err);
  return __all_sync(0xffffffffu, ok);
}

template <int D, bool E4M3, bool CAP>
__global__ void __launch_bounds__(PreCfg<D, E4M3>::kThreads, 1)
    prefill_kernel(Geometry g, PlanView p, int layer, const __nv_bfloat16* __restrict__ q,
                   const __grid_constant__ CUtensorMap q_map, int q_tma,
                   const uint8_t* __restrict__ kpool, const uint8_t* __restrict__ vpool,
                   const float* __restrict__ kscale, const float* __restrict__ vscale,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_acc,
                   float* __restrict__ part_ml, int* err) {
  using C = PreCfg<D, E4M3>;
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* k_full = bars;                        // [K stage]
  uint64_t* k_empty = k_full + C::kKStages;
  uint64_t* v_full = k_empty + C::kKStages;       // [V stage]
  uint64_t* v_empty = v_full + C::kVStages;
  uint64_t* s_full = v_empty + C::kVStages;       // [tile]: S_t(j) in tensor memory
  uint64_t* p_full = s_full + 2;                  // [tile]: P_t(j) written (and O rescaled)
  uint64_t* o_done = p_full + 2;                  // [tile]: PV_t(j) complete
  uint64_t* raw_full = o_done + 2;                // [raw stage] (e4m3 only)
  uint64_t* raw_empty = raw_full + C::kRawStages;
  uint64_t* mma_drain = raw_empty + C::kRawStages;  // every issued MMA complete
  uint64_t* q_full = mma_drain + 1;                 // Q tiles landed (tensor-copy path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);

  const WorkItem it = p.pre_items[blockIdx.x];
  const int head = blockIdx.y;
  const int G = g.hq / g.hkv;
  const int M = it.n_rows * G;
  const int n_qt = M > 128 ? 2 : 1;
  const int nkv = (it.n_keys + C::kKeys - 1) / C::kKeys;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // bf16 items whose rows are in batch order take their Q tiles by tensor
  // copies (the MMA thread issues them); the others by the softmax warps'
  // cp.async copies, which the SM keeps only so many of in flight at once:
  // a CTA's 4,096 of them took about 7,000 cycles
  const bool q_by_map = !E4M3 && q_tma && it.direct_rows;

  if (threadIdx.x == 0) {
    // e4m3: a K / V stage is filled by the two converter warps' arrivals
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&k_full[s], E4M3 ? 2 : 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&v_full[s], E4M3 ? 2 : 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < C::kRawStages; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(mma_drain, 1);
    mbar_init(q_full, 1);
    fence_mbar_init();
  }

  // Q tiles that do not come by tensor copies -> shared memory, 128-byte
  // swizzled K-major, rows past M zero; loaded by the softmax warps while the
  // producers already fetch K and V.
  // Every load of a thread is in flight at once (16-byte cp.async copies,
  // or, for e4m3 contexts, register loads for the f16 conversion, issued
  // before the barriers and tensor memory are set up); a load loop that
  // waited for each copy in turn cost a few microseconds per CTA, the whole
  // run time of a short item.  The MMA thread issues no product before the
  // named barrier below.
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  constexpr int kPer = 2 * 128 * kChunks / 256;
  const int q_total = n_qt * 128 * kChunks;
  // e4m3: every row first, then every load (-1: past M, stays zero)
  int e_row[E4M3 ? kPer : 1];
  uint4 e_val[E4M3 ? kPer : 1];
  if constexpr (E4M3) {
    if (warp < 8) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks;
        e_row[k] = idx < q_total && m < M ? item_row(p, it, m / G) : -1;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks, c16 = idx % kChunks;
        if (e_row[k] >= 0)
          e_val[k] = *reinterpret_cast<const uint4*>(
              q + (static_cast<int64_t>(e_row[k]) * g.hq + head * G + m % G) * D + c16 * 8);
      }
    }
  }

  if (warp == 8) {
    tc::alloc(tmem_slot, C::kTmemCols);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    if constexpr (E4M3) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks, c16 = idx % kChunks;
        if (idx >= q_total) continue;
        const int t = m >> 7, r = m & 127, panel = c16 >> 3, c = c16 & 7;
        const uint4 w = e_row[k] >= 0 ? bf16x8_to_f16x8(e_val[k]) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + C::kOffQ + t * C::kQTile + panel * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = w;
      }
    } else if (!q_by_map) {
      int src_row[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks;
        src_row[k] = idx < q_total && m < M ? item_row(p, it, m / G) : -1;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks, c16 = idx % kChunks;
        if (src_row[k] < 0) continue;
        const int t = m >> 7, r = m & 127, panel = c16 >> 3, c = c16 & 7;
        cp_async16(smem + C::kOffQ + t * C::kQTile + panel * 16384 + r * 128 + ((c ^ (r & 7)) << 4),
                   q + (static_cast<int64_t>(src_row[k]) * g.hq + head * G + m % G) * D + c16 * 8);
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = threadIdx.x + 256 * k, m = idx / kChunks, c16 = idx % kChunks;
        if (idx >= q_total || src_row[k] >= 0) continue;
        const int t = m >> 7, r = m & 127, panel = c16 >> 3, c = c16 & 7;
        *reinterpret_cast<uint4*>(smem + C::kOffQ + t * C::kQTile + panel * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) =
            make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_wait_all();
    tc::fence_proxy_async_smem();
  }
  if (warp <= 8) asm volatile("bar.sync 1, 288;" ::: "memory");  // Q in shared memory

  if (E4M3 && warp == 9) {
    // ------------------------------------------------- producer (e4m3)
    // Raw tiles in order K(0), V(0), K(1), V(1), ...: one 2-KB page block
    // per lane 0..7 into the staging ring.
    const int64_t layer_blk = static_cast<int64_t>(layer) * g.num_pages * g.hkv;
    int issued = 0;
    for (int i = 0; i < 2 * nkv; ++i) {
      const int r = i % C::kRawRing, j = i >> 1;
      if (i >= C::kRawRing && !warp_wait(&raw_empty[r], ((i / C::kRawRing) - 1) & 1, err)) break;
      if (lane == 0) mbar_arrive_expect_tx(&raw_full[r], C::kRawTile);
      __syncwarp();
      if (lane < C::kPagesPerTile) {
        int pj = C::kPagesPerTile * j + lane;
        if (pj >= it.n_pages) pj = it.n_pages - 1;  // keys there are masked; any finite page will do
        const int page = p.page_ids[it.pages_off + pj];
        const int64_t off = (layer_blk + static_cast<int64_t>(page) * g.hkv + head) * g.block_bytes;
        bulk_g2s(smem + C::kOffRaw + r * C::kRawTile + lane * 2048, ((i & 1) ? vpool : kpool) + off, 2048,
                 &raw_full[r]);
      }
      __syncwarp();
      issued = i + 1;
    }
    // no copy outlives the CTA, even when a consumer's wait ran out
    for (int i = issued > C::kRawRing ? issued - C::kRawRing : 0; i < issued; ++i)
      if (!warp_wait(&raw_full[i % C::kRawRing], (i / C::kRawRing) & 1, err)) break;
  } else if (E4M3 && warp >= 10) {
    // ------------------------------------------------ converters (e4m3)
    // Raw page block pg holds key s's 16-byte chunk c (dims 16c..16c+15) at
    // s*128 + 16*(c ^ (s%8)); the 8 blocks of a tile are contiguous, so raw
    // chunk qc belongs to tile key qc/8.  Its f16 values go to dims
    // 16c..16c+15 of that key's tile row: panel c/4, 16-byte f16 chunks
    // 2(c%4) and 2(c%4)+1, each at key*128 + 16*(chunk ^ (key%8)).
    // Thread ct takes raw chunks ct + 64n (n = 0..15): keys ct/8 + 8n, all
    // with key%8 = ct/8 and the same physical chunk ct%8, so every address
    // offset but the 1-KB row step is fixed per thread.  Threads with c >= 4
    // store their second chunk first, so the 8 lanes of a store phase hit 8
    // distinct bank groups.
    const int ct = threadIdx.x - 320;
    const int kr = ct >> 3, c = (ct & 7) ^ kr, ca = 2 * (c & 3);
    const int off_lo = (c >> 2) * C::kPanelBytes + kr * 128 + ((ca ^ kr) << 4);
    const int off_hi = (c >> 2) * C::kPanelBytes + kr * 128 + (((ca + 1) ^ kr) << 4);
    const int off_1 = (c & 4) ? off_hi : off_lo, off_2 = (c & 4) ? off_lo : off_hi;
    bool ok = true;
    for (int i = 0; i < 2 * nkv && ok; ++i) {
      const int r = i % C::kRawRing, j = i >> 1;
      const bool is_v = i & 1;
      const int nst = is_v ? C::kVStages : C::kKStages;
      const int st = j % nst;
      ok = warp_wait(&raw_full[r], (i / C::kRawRing) & 1, err);
      if (ok && j >= nst) ok = warp_wait(is_v ? &v_empty[st] : &k_empty[st], ((j / nst) - 1) & 1, err);
      if (!ok) break;
      const uint8_t* src = smem + C::kOffRaw + r * C::kRawTile + ct * 16;
      uint8_t* dst = smem + (is_v ? C::kOffV : C::kOffK) + st * C::kKVTile;
#pragma unroll 1
      for (int n0 = 0; n0 < C::kKeys / 8; n0 += 4) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = *reinterpret_cast<const uint4*>(src + (n0 + u) * 1024);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 a = make_uint4(e4m3x2_lo_to_f16x2(w[u].x), e4m3x2_hi_to_f16x2(w[u].x),
                                     e4m3x2_lo_to_f16x2(w[u].y), e4m3x2_hi_to_f16x2(w[u].y));
          const uint4 b = make_uint4(e4m3x2_lo_to_f16x2(w[u].z), e4m3x2_hi_to_f16x2(w[u].z),
                                     e4m3x2_lo_to_f16x2(w[u].w), e4m3x2_hi_to_f16x2(w[u].w));
          uint8_t* rowp = dst + (n0 + u) * 1024;
          *reinterpret_cast<uint4*>(rowp + off_1) = (c & 4) ? b : a;
          *reinterpret_cast<uint4*>(rowp + off_2) = (c & 4) ? a : b;
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[r]);
        mbar_arrive(is_v ? &v_full[st] : &k_full[st]);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ----------------------------------------------------------- producers
    // warp 9: K(j), one 2-KB copy per page panel (8 pages x kPanels) into
    // the panel-major tile (the S product's K-major operand spans pages);
    // warp 10: V(j), one copy of each whole page block (8 pages), blocks
    // side by side (the PV product takes one page per K = 16 step, its two
    // panels block_bytes / 2 apart).  In tile order, a stage once the MMAs
    // that read it are done; the page ids are loaded a tile ahead.
    const bool is_v = warp == 10;
    const int nst = is_v ? C::kVStages : C::kKStages;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    const int ncopy = is_v ? C::kPagesPerTile : C::kPagesPerTile * C::kPanels;
    const int64_t layer_blk = static_cast<int64_t>(layer) * g.num_pages * g.hkv;
    auto page_of = [&](int j) {
      int pj = C::kPagesPerTile * j + (is_v ? lane : lane / C::kPanels);
      if (pj >= it.n_pages) pj = it.n_pages - 1;  // keys there are masked; any finite page will do
      return lane < ncopy ? p.page_ids[it.pages_off + pj] : 0;
    };
    int page = nkv > 0 ? page_of(0) : 0;
    int issued = 0;
    for (int j = 0; j < nkv; ++j) {
      const int st = j % nst;
      if (j >= nst && !warp_wait(&empty[st], ((j / nst) - 1) & 1, err)) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], C::kKVTile);
      __syncwarp();
      if (lane < ncopy) {
        const int64_t blk = (layer_blk + static_cast<int64_t>(page) * g.hkv + head) * g.block_bytes;
        if (is_v) {
          bulk_g2s(smem + C::kOffV + st * C::kKVTile + lane * g.block_bytes, vpool + blk,
                   static_cast<uint32_t>(g.block_bytes), &full[st]);
        } else {
          const int pg = lane / C::kPanels, panel = lane % C::kPanels;
          bulk_g2s(smem + C::kOffK + st * C::kKVTile + panel * C::kPanelBytes + pg * 2048, kpool + blk + panel * 2048,
                   2048, &full[st]);
        }
      }
      if (j + 1 < nkv) page = page_of(j + 1);
      __syncwarp();
      issued = j + 1;
    }
    // no copy outlives the CTA, even when a consumer's wait ran out
    for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
      if (!warp_wait(&full[j % nst], (j / nst) & 1, err)) break;
  } else if (warp == 8) {
    // ----------------------------------------------------------------- MMA
    // One thread issues everything, event-driven, PVs first (they gate the
    // next S of their tile): PV_t(j) once P_t(j) is written and V(j)
    // landed; S_t(j) once K(j) landed and PV_t(j-1) is complete (S_t(j)
    // overwrites P_t(j-1)).  A K (V) stage is released by a commit after the
    // last S (PV) that reads it.  (Issuing S first measured the same.)
    if (lane == 0) {
      uint32_t idle = 0;
      if (q_by_map) {
        // box: d 64 x G heads x 128/G rows = one 128-row panel of one Q tile;
        // rows past M bring later rows' Q (or zeros past the batch's last
        // row), whose results are dropped
        mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(n_qt * C::kQTile));
        for (int t = 0; t < n_qt; ++t)
          for (int panel = 0; panel < C::kPanels; ++panel)
            tma_load_3d(smem + C::kOffQ + t * C::kQTile + panel * 16384, &q_map, 64 * panel, head * G,
                        it.rows_off + t * (128 / G), q_full);
        if (!mbar_wait(q_full, 0, err)) idle = kWaitLimit;
      }
      const uint32_t id_s = tc::idesc_f16kind(128, C::kKeys, false, false, !E4M3);
      const uint32_t id_o = tc::idesc_f16kind(128, D, false, true, !E4M3);
      // Per tile: the next S and PV, and the K / V ring stage and phase they
      // read; the tile loops are unrolled so that all of it stays in
      // registers (the thread's instruction count paces every hand-off).
      int s_next[2] = {0, n_qt > 1 ? 0 : nkv};
      int pv_next[2] = {0, n_qt > 1 ? 0 : nkv};
      int k_st[2] = {0, 0}, v_st[2] = {0, 0};
      uint32_t k_ph[2] = {0, 0}, v_ph[2] = {0, 0};
      while ((pv_next[0] < nkv || pv_next[1] < nkv) && idle < kWaitLimit) {
        bool progressed = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int j = pv_next[t];
          if (j < s_next[t] && mbar_test_wait(&p_full[t], j & 1) && mbar_test_wait(&v_full[v_st[t]], v_ph[t])) {
            tc::fence_after();
            const uint32_t vaddr = sbase + C::kOffV + v_st[t] * C::kKVTile;
            const uint32_t p_tmem = tmem + t * C::kKeys;  // 16 keys = 8 columns per k-step
            const uint32_t d_o = tmem + C::kColO + t * D;
            const uint32_t v_lo = tc::sw128_lo(vaddr, E4M3 ? C::kPanelBytes : 2048);
            constexpr uint32_t v_hi = tc::sw128_hi(1024);
#pragma unroll
            for (int ks = 0; ks < C::kKeys / 16; ++ks)
              tc::mma_bf16_ts_w(d_o, p_tmem + ks * 8, v_lo + ((E4M3 ? ks * 2048 : ks * (16 * D * 2)) >> 4), v_hi,
                                id_o, j > 0 || ks > 0);
            tc::commit(&o_done[t]);
            pv_next[t] = j + 1;
            if (pv_next[1 - t] > j) tc::commit(&v_empty[v_st[t]]);
            if (++v_st[t] == C::kVStages) {
              v_st[t] = 0;
              v_ph[t] ^= 1u;
            }
            progressed = true;
          }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int j = s_next[t];
          if (j < nkv && pv_next[t] == j && mbar_test_wait(&k_full[k_st[t]], k_ph[t]) &&
              (j == 0 || mbar_test_wait(&o_done[t], (j - 1) & 1))) {
            tc::fence_after();
            const uint32_t kaddr = sbase + C::kOffK + k_st[t] * C::kKVTile;
            const uint32_t qaddr = sbase + C::kOffQ + t * C::kQTile;
            const uint32_t d_s = tmem + t * C::kKeys;
            const uint32_t q_lo = tc::sw128_lo(qaddr, 16), k_lo = tc::sw128_lo(kaddr, 16);
            constexpr uint32_t qk_hi = tc::sw128_hi(1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint32_t off_q = (ks >> 2) * 16384 + (ks & 3) * 32;
              const uint32_t off_k = (ks >> 2) * C::kPanelBytes + (ks & 3) * 32;
              tc::mma_bf16_w(d_s, q_lo + (off_q >> 4), qk_hi, k_lo + (off_k >> 4), qk_hi, id_s, ks > 0);
            }
            tc::commit(&s_full[t]);
            s_next[t] = j + 1;
            if (s_next[1 - t] > j) tc::commit(&k_empty[k_st[t]]);
            if (++k_st[t] == C::kKStages) {
              k_st[t] = 0;
              k_ph[t] ^= 1u;
            }
            progressed = true;
          }
        }
        idle = progressed ? 0 : idle + 1;
      }
      if (idle >= kWaitLimit && err) atomicOr(err, kErrWaitTimeout);
      // Tensor memory is freed only after every MMA issued here has
      // completed (normally they have: the softmax warps waited for them).
      tc::commit(mma_drain);
      mbar_wait(mma_drain, 0, err);
    }
    __syncwarp();
  } else if (warp / 4 < n_qt) {
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int r = ((warp & 3) << 5) + lane;
    const int m = t * 128 + r;
    const uint32_t row_s = tmem + (static_cast<uint32_t>((warp & 3) << 5) << 16) + t * C::kKeys;
    const uint32_t row_o = tmem + (static_cast<uint32_t>((warp & 3) << 5) << 16) + C::kColO + t * D;
    // rows past M (zero Q) take a position past every key, so that they do
    // not force the masked path on their warp; their results are dropped
    int row = -1, pos = kNoRowPos, qh = 0;
    if (m < M) {
      row = item_row(p, it, m / G);
      pos = p.row_pos[row];
      qh = head * G + m % G;
    }
    // a warp with no row below M computes nothing: it only keeps the
    // barrier protocol (the P lanes it leaves hold S values, which reach
    // only the O rows of those lanes, never stored)
    const bool idle = __all_sync(0xffffffffu, row < 0);
    // scores in log2 units: s * qk_scale; with the soft cap c the scores
    // are first mapped to tanh(s * cap_pre) and then scaled by
    // qk_scale = c * log2(e) (c * tanh(s / c) in log2 units)
    const float s_scale = (E4M3 ? kscale[layer * g.hkv + head] : 1.0f) * rsqrtf(static_cast<float>(D));
    const float qk_scale = CAP ? g.softcap * 1.4426950408889634f : s_scale * 1.4426950408889634f;
    const float cap_pre = CAP ? s_scale / g.softcap : 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      ok = warp_wait(&s_full[t], j & 1, err);
      if (!ok) break;
      if (idle) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
        continue;
      }
      tc::fence_after();
      // columns <= lim are visible: causal, and inside the item's key run
      // (the tile past the run's end holds stand-in pages)
      const int lim = min(pos - (it.key_base + C::kKeys * j), it.n_keys - 1 - C::kKeys * j);
      const bool masked = !__all_sync(0xffffffffu, lim >= C::kKeys - 1);
      // The whole S row in registers (4 loads of 32 columns in flight at
      // once), its max (scale > 0 commutes with max), then the weights per
      // chunk of 32 columns; P (bf16 pairs) of chunk c goes to columns
      // 16c..16c+15, which hold scores already in registers.
      uint32_t sr[C::kKeys];
#pragma unroll
      for (int c = 0; c < C::kKeys / 32; ++c) tc::ld32(row_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tc::wait_ld();
      if constexpr (CAP) {
#pragma unroll
        for (int e = 0; e < C::kKeys; ++e) sr[e] = __float_as_uint(tanh_approx(__uint_as_float(sr[e]) * cap_pre));
      }
      if (masked) {
#pragma unroll
        for (int e = 0; e < C::kKeys; ++e)
          if (e > lim) sr[e] = __float_as_uint(-INFINITY);
      }
      float m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) m4[i] = -INFINITY;
#pragma unroll
      for (int e = 0; e < C::kKeys / 2; ++e)
        m4[e & 3] = max3(m4[e & 3], __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
      m4[0] = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      const float mx = m4[0] * qk_scale;
      float alpha = 1.f;
      bool resc = false;
      const float m_new = fmaxf(m_run, mx);
      if (m_new > m_run + 8.f) {
        alpha = ex2(m_run - m_new);
        m_run = m_new;
        resc = true;
      }
      const float nb = m_run == -INFINITY ? 0.f : -m_run;
      uint64_t acc[4] = {0, 0, 0, 0};  // packed pairs of partial row sums
#pragma unroll
      for (int c = 0; c < C::kKeys / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = softmax_pair<E4M3>(__uint_as_float(sr[32 * c + 2 * e]), __uint_as_float(sr[32 * c + 2 * e + 1]), qk_scale,
                               nb, acc[e & 3]);
        tc::st16(row_s + 16 * c, pk);
      }
      const float row_sum = (sum_pair(acc[0]) + sum_pair(acc[1])) + (sum_pair(acc[2]) + sum_pair(acc[3]));
      l_run = l_run * alpha + row_sum;
      // O rescale: PV_t(j-1) is complete (S_t(j) was issued after it)
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tc::ld32(row_o + cc * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::st32(row_o + cc * 32, o);
        }
      }
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    if (ok) ok = warp_wait(&o_done[t], (nkv - 1) & 1, err);
    tc::fence_after();
    if (ok && !idle) {
      // O of the warp's 32 rows goes out through shared memory: each lane
      // writes its row (tensor-memory lane) into the warp's quarter of Q
      // tile t's buffer (free: every S_t has completed), in 16-byte chunks
      // XOR-swizzled by row so that neither the row-wise writes nor the
      // chunk-wise reads meet a bank conflict; then 32 / kCh lanes store one
      // row per instruction, each 32-byte sector of the output written
      // whole.  (Storing each lane's own row straight from registers wrote
      // 32 half sectors per instruction and took about 4,000 cycles per CTA.)
      // Direct rows stage the bf16 row (2d bytes) once, split rows their
      // fp32 partial in two halves of 2d bytes.
      constexpr int kRowB = 2 * D;     // staged bytes per row and round
      constexpr int kCh = kRowB / 16;  // 16-byte chunks per staged row
      constexpr int kRpi = 32 / kCh;   // rows per store instruction
      static_assert(4 * 32 * kRowB == C::kQTile, "staging fills the Q tile buffer");
      uint8_t* stage = smem + C::kOffQ + t * C::kQTile + (warp & 3) * 32 * kRowB;
      auto put = [&](int c, uint4 w) {
        *reinterpret_cast<uint4*>(stage + lane * kRowB + ((c ^ (lane % kCh)) << 4)) = w;
      };
      auto get = [&](int rr, int c) {
        return *reinterpret_cast<const uint4*>(stage + rr * kRowB + ((c ^ (rr % kCh)) << 4));
      };
      const float vdq = E4M3 ? vscale[layer * g.hkv + head] : 1.0f;
      if (it.part < 0) {
        const float inv = l_run > 0.f ? vdq / l_run : 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tc::ld32(row_o + cc * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            put(4 * cc + v, w);
          }
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kCh; ++i) {
          const int rr = i * kRpi + lane / kCh, c = lane % kCh;
          const int rrow = __shfl_sync(0xffffffffu, row, rr), rqh = __shfl_sync(0xffffffffu, qh, rr);
          const uint4 w = get(rr, c);
          if (rrow >= 0) *reinterpret_cast<uint4*>(out + (static_cast<int64_t>(rrow) * g.hq + rqh) * D + c * 8) = w;
        }
        if (row >= 0 && lse) lse[static_cast<int64_t>(row) * g.hq + qh] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
      } else {
        const int slot = row >= 0 ? (p.row_part_base[row] + it.part) * g.hq + qh : -1;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t o[32];
            tc::ld32(row_o + half * (D / 2) + cc * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int v = 0; v < 8; ++v)
              put(8 * cc + v, make_uint4(__float_as_uint(__uint_as_float(o[4 * v]) * vdq),
                                         __float_as_uint(__uint_as_float(o[4 * v + 1]) * vdq),
                                         __float_as_uint(__uint_as_float(o[4 * v + 2]) * vdq),
                                         __float_as_uint(__uint_as_float(o[4 * v + 3]) * vdq)));
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kCh; ++i) {
            const int rr = i * kRpi + lane / kCh, c = lane % kCh;
            const int rslot = __shfl_sync(0xffffffffu, slot, rr);
            const uint4 w = get(rr, c);
            if (rslot >= 0)
              *reinterpret_cast<uint4*>(part_acc + static_cast<int64_t>(rslot) * D + half * (D / 2) + c * 4) = w;
          }
          __syncwarp();  // the next half overwrites the staging rows
        }
        if (row >= 0) *reinterpret_cast<float2*>(part_ml + static_cast<int64_t>(slot) * 2) = make_float2(m_run, l_run);
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

template <int D, bool E4M3, bool CAP>
cudaError_t launch_t(const Geometry& g, const PlanView& p, int layer, const void* q, const CUtensorMap* q_map,
                     const void* kpool, const void* vpool, const float* kscale, const float* vscale, void* out,
                     float* lse, float* acc, float* ml, int* err, cudaStream_t st) {
  using C = PreCfg<D, E4M3>;
  static_assert(C::kSmem <= 227 * 1024, "shared memory budget");
  cudaError_t e = ensure_smem_attr<prefill_kernel<D, E4M3, CAP>>(C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_pre, g.hkv);
  const CUtensorMap no_map{};
  e = launch_pdl(prefill_kernel<D, E4M3, CAP>, grid, C::kThreads, C::kSmem, st, g, p, layer,
                 static_cast<const __nv_bfloat16*>(q), q_map ? *q_map : no_map, q_map ? 1 : 0,
                 static_cast<const uint8_t*>(kpool),
                 static_cast<const uint8_t*>(vpool), kscale, vscale, static_cast<__nv_bfloat16*>(out), lse, acc, ml,
                 err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const Geometry& g, const PlanView& p, int layer, const void* q, const CUtensorMap* q_map,
                           const void* kpool, const void* vpool, const float* scale_k, const float* scale_v,
                           void* out, float* lse, float* part_acc, float* part_ml, int* err, cudaStream_t st) {
  if (p.n_pre == 0) return cudaSuccess;
#define PIE_PREFILL(DD, E, CP) \
  launch_t<DD, E, CP>(g, p, layer, q, q_map, kpool, vpool, scale_k, scale_v, out, lse, part_acc, part_ml, err, st)
  const bool cap = g.softcap > 0.f;
  if (g.kv_dtype != 0) {
    if (g.d != 128) return cudaErrorInvalidValue;
    return cap ? PIE_PREFILL(128, true, true) : PIE_PREFILL(128, true, false);
  }
  if (g.d == 128) return cap ? PIE_PREFILL(128, false, true) : PIE_PREFILL(128, false, false);
  if (g.d == 64) return cap ? PIE_PREFILL(64, false, true) : PIE_PREFILL(64, false, false);
#undef PIE_PREFILL
  return cudaErrorInvalidValue;
}

}  // namespace pie
