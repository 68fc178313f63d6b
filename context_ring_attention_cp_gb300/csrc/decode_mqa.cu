// Pass-Q decode for query heads that share one K/V head (MQA / MLA-style), on
// sm_103a tensor cores.
//
// "G5 上下文并行建模设计规格": Terms table row "Pass-Q" (query to every rank,
// local partial attention per KV shard, then the reduce), c_kv row (for MLA the
// compressed per-token K/V), use-case decode paragraph.  With g = h_q / h_kv
// query heads on one K/V head (g = 16 x 512 on the pypto-lib issue page's per-card
// shapes), every K/V byte feeds 16 dot products: at HBM speed that is ~16 FLOP/B,
// beyond the FP32 pipes, so both contractions run on tcgen05.
//
// Transposed formulation; one persistent CTA per SM walks work items (KV range,
// sequence, kv head) strided by the grid, keeping its barriers, ring and TMEM:
//   S^T = K Q^T   M = 128 keys, N = g heads, K = d      (A = K tile, B = Q, both K-major)
//   O^T += V^T P^T  M = 128-wide d block, N = g, K = 128 keys
//                   (A = V tile read MN-major, B = P^T written by the softmax warps)
// so g = 16 heads fill an N = 16 instruction with no padding.  K and V stream
// through a ring of 16 KB slots (128 keys x 64 d, 128-byte swizzle), loaded in
// exactly the order the MMAs consume them: K_0, then (K_{j+1}, V_j) per tile; V_j
// is requested only once P(j) is written, so its slots hold loads in flight, not
// landed data waiting for softmax(j).
// A tile's V slabs come in groups of d/64 >= 2 starting on an even slot of an
// even-sized ring, so the two 64-wide halves of a d block sit in adjacent slots
// and the MN-major descriptor's leading offset is one slot.
//
// Warps: 0 TMA producer, 1 TMEM owner + MMA issuer (one lane), 4-7 softmax and
// epilogue (thread = key lane of S^T, and = d lane of O^T).  Per-head maxima over
// the 128 keys of a tile come from a warp max reduction (redux.sync) plus a
// shared-memory reduction across the four warps; the exponent reference is raised
// only when a head's max
// grows by more than 8 (log2 units), O^T columns are then rescaled in TMEM.  Row
// sums stay per thread until the epilogue.  The CTA writes its partial triple per
// query head to the decode workspace, which the LSE merge kernel reduces.
//
// Across items: Q is double-buffered (released after an item's last S^T), and the
// next item's first O^T waits until the epilogue has read the previous O^T out of
// TMEM, so the next item's first S^T overlaps the previous epilogue.
//
// Every mbarrier wait is bounded (tc_ptx.h); on expiry CP_ERR_TIMEOUT goes to this
// file's status word and the CTA returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "internal.h"
#include "tc_ptx.h"

namespace cpattn {
namespace {

using namespace tc;

constexpr int BK = 128;        // keys per tile (M of S^T)
constexpr int kSlabBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

__device__ int32_t g_mqa_status = 0;

template <int D, int G>
struct MqaCfg {
  static constexpr int kSlabsPerTile = D / 64;      // K or V slabs per 128-key tile
  static constexpr int kQSlab = G * 128;            // bytes of one Q slab (G rows x 64 d)
  static constexpr int kQBytes = kSlabsPerTile * kQSlab;
  static constexpr int kPSlab = G * 128;            // bytes of one P^T slab (G rows x 64 keys)
  static constexpr int kPBytes = 2 * kPSlab;        // one P^T buffer (128 keys)
  static constexpr int kSlots = (G == 16) ? 10 : 8;  // even ring size
  static constexpr int kQOff = 0;                   // two Q buffers (consecutive work items)
  static constexpr int kPOff = 2 * kQBytes;         // two P^T buffers
  static constexpr int kRingOff = kPOff + 2 * kPBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kSlabBytes;
  static constexpr int kRedOff = kBarOff + 512;     // [2][4][G] per-warp maxima, then [4][G] row sums
  static constexpr int kSmemBytes = kRedOff + 3 * 4 * G * 4 + 1024;
  static constexpr uint32_t kOCol = 2 * G;          // S^T buffers at [0, G) and [G, 2G)
  static constexpr uint32_t kTmemCols = (2 * G + (D / 128) * G) <= 64 ? 64 : ((2 * G + (D / 128) * G) <= 128 ? 128 : 256);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kSlots % 2 == 0, "V slab pairs must not wrap the ring");
  static_assert(kQSlab % 1024 == 0 && kPSlab % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
};

struct MqaParams {
  CUtensorMap tmap_q;  // dims (d, h_q, b), box (64, G, 1)
  CUtensorMap tmap_k;  // dims (d, h_kv, L, b), box (64, 1, 128, 1)
  CUtensorMap tmap_v;
  float* o_parts;  // [n_parts, b, h_q, d]
  float* m_parts;  // [n_parts, b, h_q]
  float* l_parts;
  int64_t b, L, h_q, h_kv;
  int64_t shard_len;              // keys per KV shard (L / cp)
  int32_t cp;                     // shards per sequence
  int32_t splits;                 // key ranges per shard
  int32_t tiles_base, tiles_rem;  // a shard's T tiles: ranges j < T % splits get one more
  int32_t n_units;                // b * h_kv * cp shards in all
  int32_t n_parts;                // cp * splits partial triples per (sequence, head)
  int32_t n_items;  // n_parts * b * h_kv work items, strided over the persistent grid
  float sl;         // scale * log2(e)
};

// Maximum over the warp's 32 lanes in one instruction.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) mqa_decode_kernel(const __grid_constant__ MqaParams p) {
  using K = MqaCfg<D, G>;
  constexpr int NS = K::kSlabsPerTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K::kBarOff);
  auto bar_qf = [&](int b) { return smem_u32(&bars[0 + b]); };   // Q buffer b loaded
  auto bar_qe = [&](int b) { return smem_u32(&bars[2 + b]); };   // Q buffer b no longer read
  auto bar_full = [&](int s) { return smem_u32(&bars[4 + s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[4 + K::kSlots + s]); };
  auto bar_s = [&](int b) { return smem_u32(&bars[4 + 2 * K::kSlots + b]); };
  auto bar_p = [&](int b) { return smem_u32(&bars[6 + 2 * K::kSlots + b]); };
  // O^T of tile t complete: barrier t % 2 (phase t / 2), so a wait for tile t - 2 is never
  // ambiguous (tile t cannot complete before this softmax writes P(t)).
  auto bar_o = [&](int32_t t) { return smem_u32(&bars[8 + 2 * K::kSlots + (t & 1)]); };
  const uint32_t bar_of = smem_u32(&bars[10 + 2 * K::kSlots]);    // O^T read by the epilogue
  const uint32_t bar_red = smem_u32(&bars[11 + 2 * K::kSlots]);   // the four softmax warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[12 + 2 * K::kSlots]);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + K::kRedOff);  // [2][4][G] maxima
  float* red_l = red + 2 * 4 * G;                             // [4][G] row sums

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Work item -> (key range, sequence, kv head).  Items go range-major: range j of
  // every shard of every (sequence, kv head), then range j + 1.  A shard's ranges are
  // whole tiles, the longer ones first, so the grid-strided walk hands every CTA
  // nearly the same number of tiles.
  struct ItemRange {
    int32_t part, kvh, bi, n_tiles;
    int64_t k_begin, k_end;
  };
  auto decode_item = [&](int32_t item) {
    ItemRange r;
    const int32_t j = item / p.n_units;
    const int32_t rest = item - j * p.n_units;
    const int32_t bk = rest / p.cp;  // sequence * h_kv + kv head
    const int32_t shard = rest - bk * p.cp;
    r.bi = bk / int32_t(p.h_kv);
    r.kvh = bk - r.bi * int32_t(p.h_kv);
    r.part = shard * p.splits + j;
    r.n_tiles = p.tiles_base + (j < p.tiles_rem ? 1 : 0);
    const int32_t t0 = j * p.tiles_base + (j < p.tiles_rem ? j : p.tiles_rem);
    const int64_t s0 = int64_t(shard) * p.shard_len;
    r.k_begin = s0 + int64_t(t0) * BK;
    const int64_t end = r.k_begin + int64_t(r.n_tiles) * BK;
    r.k_end = end < s0 + p.shard_len ? end : s0 + p.shard_len;
    return r;
  };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_qf(b), 1);
      mbar_init(bar_qe(b), 1);
      mbar_init(bar_s(b), 1);
      mbar_init(bar_p(b), 4);
    }
    for (int s = 0; s < K::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_o(0), 1);
    mbar_init(bar_o(1), 1);
    mbar_init(bar_of, 4);
    mbar_init(bar_red, 4);
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(&g_mqa_status) != 0) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(K::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;
  auto wait = [&](uint32_t bar, uint32_t parity) { return mbar_wait_bounded(bar, parity, abort_flag, &g_mqa_status); };

  if (skip) {
    // an earlier wait gave up: nothing to do
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int32_t li = 0;  // running slab index, in MMA consumption order
      int32_t jt = 0;  // running tile index (P barrier phases)
      bool ok = true;
      int32_t ic = 0;  // items of this CTA so far
      for (int32_t item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++ic) {
        const ItemRange ir = decode_item(item);
        const int32_t kvh = ir.kvh, bi = ir.bi, n_tiles = ir.n_tiles;
        const int32_t k_begin = int32_t(ir.k_begin);
        const int qb = ic & 1;
        if (ic >= 2 && !wait(bar_qe(qb), uint32_t(((ic >> 1) - 1) & 1))) { ok = false; break; }
        mbar_expect_tx(bar_qf(qb), uint32_t(K::kQBytes));
        for (int sl = 0; sl < NS; ++sl)
          tma_load_3d(sbase + K::kQOff + qb * K::kQBytes + sl * K::kQSlab, &p.tmap_q, bar_qf(qb), sl * 64, kvh * G,
                      bi);
        auto load_tile = [&](const CUtensorMap* map, int32_t tile) {
          const int32_t key0 = k_begin + tile * BK;
          for (int sl = 0; sl < NS && ok; ++sl, ++li) {
            const int s = li % K::kSlots, round = li / K::kSlots;
            if (round > 0 && !wait(bar_empty(s), uint32_t((round - 1) & 1))) { ok = false; break; }
            mbar_expect_tx(bar_full(s), uint32_t(kSlabBytes));
            tma_load_4d(sbase + K::kRingOff + s * kSlabBytes, map, bar_full(s), sl * 64, kvh, key0, bi);
          }
        };
        load_tile(&p.tmap_k, 0);
        for (int32_t j = 0; ok && j < n_tiles; ++j) {
          if (j + 1 < n_tiles) load_tile(&p.tmap_k, j + 1);
          // V_j is consumed only once P(j) is written: loading it then keeps its slots
          // free for loads in flight while softmax(j) runs.
          const int32_t t = jt + j;
          if (ok && !wait(bar_p(t & 1), uint32_t((t >> 1) & 1))) { ok = false; break; }
          if (ok) load_tile(&p.tmap_v, j);
        }
        jt += n_tiles;
      }
      if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc_bf16(128, G, false, false);
      constexpr uint32_t idesc_o = instr_desc_bf16(128, G, true, false);
      int32_t li = 0;   // running slab index
      int32_t jt = 0;   // running tile index (S / P buffer and barrier phases)
      bool ok = true;
      int32_t ic = 0;
      for (int32_t item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++ic) {
        const int32_t n_tiles = decode_item(item).n_tiles;
        const int qb = ic & 1;
        if (!wait(bar_qf(qb), uint32_t((ic >> 1) & 1))) { ok = false; break; }
        // S^T of global tile t into S buffer t % 2 from the next NS K slabs
        auto issue_s = [&](int32_t t) {
          const uint32_t d_tm = tmem + uint32_t(t & 1) * G;
          for (int sl = 0; sl < NS && ok; ++sl, ++li) {
            const int s = li % K::kSlots;
            if (!wait(bar_full(s), uint32_t((li / K::kSlots) & 1))) { ok = false; break; }
            tc_fence_after();
            const uint32_t ka = sbase + K::kRingOff + s * kSlabBytes;
            const uint32_t qa = sbase + K::kQOff + qb * K::kQBytes + sl * K::kQSlab;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 d per k-step = 32 bytes into the 128-byte row
              mma_ss(d_tm, smem_desc(ka + kk * 32, 16, 1024), smem_desc(qa + kk * 32, 16, 1024), idesc_s,
                     (sl > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar_empty(s));
          }
        };
        // O^T += V^T(t) P^T(t): d blocks of 128 = slab pairs, 8 k-steps of 16 keys each
        auto issue_o = [&](int32_t t, bool first) {
          const uint32_t pa = sbase + K::kPOff + uint32_t(t & 1) * K::kPBytes;
          for (int blk = 0; blk < NS / 2 && ok; ++blk, li += 2) {
            const int s0 = li % K::kSlots, s1 = (li + 1) % K::kSlots;
            if (!wait(bar_full(s0), uint32_t((li / K::kSlots) & 1)) ||
                !wait(bar_full(s1), uint32_t(((li + 1) / K::kSlots) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t va = sbase + K::kRingOff + s0 * kSlabBytes;  // s1 == s0 + 1 (even slot, even ring)
            const uint32_t d_tm = tmem + K::kOCol + uint32_t(blk) * G;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_ss(d_tm, smem_desc(va + kk * 2048, kSlabBytes, 1024),
                     smem_desc(pa + (kk / 4) * K::kPSlab + (kk % 4) * 32, 16, 1024), idesc_o,
                     (!first || kk > 0) ? 1u : 0u);
            mma_commit(bar_empty(s0));
            mma_commit(bar_empty(s1));
          }
        };
        issue_s(jt);
        if (!ok) break;
        mma_commit(bar_s(jt & 1));
        if (n_tiles == 1) mma_commit(bar_qe(qb));
        for (int32_t j = 0; ok && j < n_tiles; ++j) {
          const int32_t t = jt + j;
          if (j + 1 < n_tiles) {
            issue_s(t + 1);
            if (!ok) break;
            mma_commit(bar_s((t + 1) & 1));
            if (j + 2 == n_tiles) mma_commit(bar_qe(qb));  // the item's last S^T: Q buffer free
          }
          if (!wait(bar_p(t & 1), uint32_t((t >> 1) & 1))) { ok = false; break; }
          // the previous item's O^T must have been read out before this item overwrites it
          if (j == 0 && ic > 0 && !wait(bar_of, uint32_t((ic - 1) & 1))) { ok = false; break; }
          tc_fence_after();
          issue_o(t, j == 0);
          if (!ok) break;
          mma_commit(bar_o(t));
        }
        jt += n_tiles;
      }
      if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int t_ = threadIdx.x - 128;  // key lane of S^T, d lane of O^T
    const int wq = warp - 4;
    const uint32_t lane_base = uint32_t(wq * 32) << 16;
    bool ok = true;
    int32_t jt = 0;  // running tile index
    int32_t rc = 0;  // running phase of the cross-warp barrier
    for (int32_t item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      const ItemRange ir = decode_item(item);
      const int32_t part = ir.part, kvh = ir.kvh, bi = ir.bi, n_tiles = ir.n_tiles;
      const int64_t k_begin = ir.k_begin;
      const int64_t k_end = ir.k_end;
      float m_ref[G], m_true[G], l_t[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_ref[h] = -INFINITY;
        m_true[h] = -INFINITY;
        l_t[h] = 0.f;
      }
      for (int32_t j = 0; j < n_tiles; ++j) {
        const int32_t t = jt + j;
        if (!__all_sync(0xffffffffu, wait(bar_s(t & 1), uint32_t((t >> 1) & 1)))) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[G];
        if constexpr (G == 16) {
          tmem_ld16(tmem + lane_base + uint32_t(t & 1) * G, sr);
          tmem_ld_wait16(sr);
        } else {
          tmem_ld32(tmem + lane_base + uint32_t(t & 1) * G, sr);
          tmem_ld_wait(sr);
        }
        const int64_t key = k_begin + int64_t(j) * BK + t_;
        const bool valid = key < k_end;
        float x[G], mx[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          x[h] = valid ? __uint_as_float(sr[h]) : -INFINITY;
          mx[h] = x[h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) mx[h] = warp_max(mx[h]);
        // Cross-warp maxima through shared memory, double-buffered by phase; the
        // barrier is an mbarrier (bounded wait), not bar.sync, so a warp that gave
        // up cannot leave the others waiting forever.
        float* rb = red + (rc & 1) * 4 * G;
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) rb[wq * G + h] = mx[h];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_red);
        if (!__all_sync(0xffffffffu, wait(bar_red, uint32_t(rc & 1)))) { ok = false; break; }
        ++rc;
        bool any_raise = false;
        float f[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float tmax = fmaxf(fmaxf(rb[h], rb[G + h]), fmaxf(rb[2 * G + h], rb[3 * G + h])) * p.sl;
          m_true[h] = fmaxf(m_true[h], tmax);
          const bool raise = tmax > m_ref[h] + kRescaleThreshold;
          f[h] = 1.f;
          if (raise) {
            f[h] = (m_ref[h] == -INFINITY) ? 0.f : ex2(m_ref[h] - tmax);
            any_raise = any_raise || (j > 0 && m_ref[h] != -INFINITY);
            l_t[h] *= f[h];
            m_ref[h] = tmax;
          }
        }
        // P buffer t % 2 was last read by O^T(t - 2): that must be complete before it is
        // rewritten (within an item's first two tiles the previous item's epilogue has
        // already waited for it).  A rescale of O^T also needs O^T(t - 1) complete.
        if (j >= 2 && !__all_sync(0xffffffffu, wait(bar_o(t - 2), uint32_t(((t - 2) >> 1) & 1)))) {
          ok = false;
          break;
        }
        if (any_raise && !__all_sync(0xffffffffu, wait(bar_o(t - 1), uint32_t(((t - 1) >> 1) & 1)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (any_raise) {  // identical in every thread: decided from the shared maxima
#pragma unroll
          for (int blk = 0; blk < D / 128; ++blk) {
            const uint32_t oaddr = tmem + lane_base + K::kOCol + uint32_t(blk) * G;
            uint32_t r[G];
            if constexpr (G == 16) {
              tmem_ld16(oaddr, r);
              tmem_ld_wait16(r);
#pragma unroll
              for (int h = 0; h < G; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * f[h]);
              tmem_st16(oaddr, r);
            } else {
              tmem_ld32(oaddr, r);
              tmem_ld_wait(r);
#pragma unroll
              for (int h = 0; h < G; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * f[h]);
              tmem_st32(oaddr, r);
            }
          }
          tmem_st_wait();
        }
        // P^T(t): row h, key column t_ of a [G x 128] K-major, 128-byte-swizzled operand
        uint8_t* pbuf = smem + K::kPOff + (t & 1) * K::kPBytes + (t_ / 64) * K::kPSlab;
        const int c16 = (t_ % 64) / 8, within = (t_ % 8) * 2;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pv = ex2(fmaf(x[h], p.sl, -((m_ref[h] == -INFINITY) ? 0.f : m_ref[h])));
          l_t[h] += pv;
          *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + ((c16 ^ (h % 8)) << 4) + within) =
              __float2bfloat16_rn(pv);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p(t & 1));
      }
      if (!ok) break;

      // ---------------- epilogue: this item's partial triple per query head
      const int32_t t_last = jt + n_tiles - 1;
      if (!__all_sync(0xffffffffu, wait(bar_o(t_last), uint32_t((t_last >> 1) & 1)))) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) l_t[h] += __shfl_xor_sync(0xffffffffu, l_t[h], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) red_l[wq * G + h] = l_t[h];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_red);
      if (!__all_sync(0xffffffffu, wait(bar_red, uint32_t(rc & 1)))) { ok = false; break; }
      ++rc;
      const int64_t row0 = (int64_t(part) * p.b + bi) * p.h_q + int64_t(kvh) * G;
#pragma unroll
      for (int blk = 0; blk < D / 128; ++blk) {
        uint32_t r[G];
        const uint32_t oaddr = tmem + lane_base + K::kOCol + uint32_t(blk) * G;
        if constexpr (G == 16) {
          tmem_ld16(oaddr, r);
          tmem_ld_wait16(r);
        } else {
          tmem_ld32(oaddr, r);
          tmem_ld_wait(r);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          // re-express against the true max: factor 2^(m_ref - m_true) <= 1
          const float fre = (m_true[h] == -INFINITY) ? 0.f : ex2(m_ref[h] - m_true[h]);
          p.o_parts[(row0 + h) * D + blk * 128 + t_] = __uint_as_float(r[h]) * fre;
        }
      }
      // O^T has been read into registers: the next item may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_of);
      if (t_ < G) {
        float mt = 0.f, mr = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h == t_) {
            mt = m_true[h];
            mr = m_ref[h];
          }
        }
        const float lsum = red_l[t_] + red_l[G + t_] + red_l[2 * G + t_] + red_l[3 * G + t_];
        const float fre = (mt == -INFINITY) ? 0.f : ex2(mr - mt);
        p.m_parts[row0 + t_] = mt * kLn2;  // natural-log units
        p.l_parts[row0 + t_] = lsum * fre;
      }
      jt += n_tiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(K::kTmemCols));
  }
}

bool encode(CUtensorMap* map, const void* base, cuuint32_t rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_dg(const MqaParams& p, dim3 grid, cudaStream_t stream) {
  using K = MqaCfg<D, G>;
  static SmemLimit lim;
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(mqa_decode_kernel<D, G>), K::kSmemBytes, &lim);
  if (e != cudaSuccess) return e;
  mqa_decode_kernel<D, G><<<grid, kThreads, K::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool decode_mqa_supported(const cp_attn_desc& d) {
  const int64_t g = d.h_q / d.h_kv;
  return (g == 16 || g == 32) && (d.d == 128 || d.d == 256 || d.d == 512) && d.S < (int64_t(1) << 31) &&
         d.b <= 65535 && d.h_kv <= 65535;
}

// Key ranges per shard.  Each candidate count (ranges of at least four tiles, at most
// CP_MAX_MERGE_PARTS parts) is scored as the kernel's grid walks the items: the
// busiest CTA's tiles, plus one tile per item for the switch between items
// (measured: 19 ranges, 0.2 % from even, ran slower than 16 ranges, 4 % from even).
// The lowest score wins, the fewer ranges on a tie.
int32_t decode_mqa_splits(const cp_attn_desc& d, int sm_count) {
  const int64_t tiles = (d.S / d.cp + BK - 1) / BK;  // per shard
  const int64_t units = d.b * d.h_kv * d.cp;
  const int64_t sms = sm_count > 0 ? sm_count : 148;
  int64_t best = 1;
  double best_score = 0.0;
  for (int64_t s = 1; s <= tiles && d.cp * s <= CP_MAX_MERGE_PARTS; ++s) {
    if (s > 1 && tiles / s < 4) break;
    const int64_t items = s * units;
    const int64_t grid = items < sms ? items : sms;
    const int64_t base = tiles / s, rem = tiles % s;
    // CTA c walks items c, c + grid, ...; the first rem * units items are one tile
    // longer.  Both counts fall with c, so CTA 0 is the busiest.
    const int64_t per_cta = (items + grid - 1) / grid;
    const int64_t worst = per_cta * base + (rem * units + grid - 1) / grid;
    const double score = double(worst) + double(per_cta);
    if (s == 1 || score < best_score) {
      best = s;
      best_score = score;
    }
  }
  return int32_t(best);
}

cudaError_t launch_decode_mqa(const cp_attn_desc& d, int32_t splits, const void* q, const void* k, const void* v,
                              float* o_parts, float* m_parts, float* l_parts, cudaStream_t stream) {
  MqaParams p;
  memset(&p, 0, sizeof(p));
  const int G = int(d.h_q / d.h_kv);
  {
    const cuuint64_t dims[3] = {cuuint64_t(d.d), cuuint64_t(d.h_q), cuuint64_t(d.b)};
    const cuuint64_t strides[2] = {cuuint64_t(d.d * 2), cuuint64_t(d.h_q * d.d * 2)};
    const cuuint32_t box[3] = {64, cuuint32_t(G), 1};
    if (!encode(&p.tmap_q, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[4] = {cuuint64_t(d.d), cuuint64_t(d.h_kv), cuuint64_t(d.S), cuuint64_t(d.b)};
    const cuuint64_t strides[3] = {cuuint64_t(d.d * 2), cuuint64_t(d.h_kv * d.d * 2),
                                   cuuint64_t(d.S * d.h_kv * d.d * 2)};
    const cuuint32_t box[4] = {64, 1, BK, 1};
    if (!encode(&p.tmap_k, k, 4, dims, strides, box) || !encode(&p.tmap_v, v, 4, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  p.b = d.b;
  p.L = d.S;
  p.h_q = d.h_q;
  p.h_kv = d.h_kv;
  p.n_parts = int32_t(d.cp * splits);
  p.cp = int32_t(d.cp);
  p.splits = splits;
  p.shard_len = d.S / d.cp;
  {
    const int32_t tiles = int32_t((p.shard_len + BK - 1) / BK);
    if (splits < 1 || splits > tiles) return cudaErrorInvalidValue;
    p.tiles_base = tiles / splits;
    p.tiles_rem = tiles % splits;
  }
  p.n_units = int32_t(d.b * d.h_kv * d.cp);
  p.sl = d.scale * kLog2e;
  const int64_t n_items = int64_t(p.n_parts) * d.b * d.h_kv;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.n_items = int32_t(n_items);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const dim3 grid(unsigned(n_items < sms ? n_items : sms));  // persistent: one CTA per SM
#define CP_MQA(DD, GG) \
  if (d.d == DD && G == GG) return launch_dg<DD, GG>(p, grid, stream);
  CP_MQA(128, 16) CP_MQA(256, 16) CP_MQA(512, 16)
  CP_MQA(128, 32) CP_MQA(256, 32) CP_MQA(512, 32)
#undef CP_MQA
  return cudaErrorInvalidValue;
}

cudaError_t mqa_take_status(int32_t* status) {
  int32_t s = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&s, g_mqa_status, sizeof(s));
  if (e != cudaSuccess) return e;
  const int32_t zero = 0;
  e = cudaMemcpyToSymbol(g_mqa_status, &zero, sizeof(zero));
  *status = s;
  return e;
}

}  // namespace cpattn
