// Ring-step partial attention for all cp virtual ranks, on sm_103a tensor cores.
//
// Method ("G5 上下文并行建模设计规格", G5 CP modelling spec):
//  * Terms table, "Balanced chunk split": the sequence is cut into 2*cp chunks of
//    C tokens; rank r owns chunk r (head) and chunk 2cp-1-r (tail).
//  * Terms table, "Pass-KV" / "Ring step": in step t rank r computes partial
//    attention of its rows against the K/V block it holds, the block of source
//    rank s = (r - t) mod cp.  On one GPU the rotation is an index change: the
//    kernel reads the source rank's chunks straight from HBM.
//  * Terms table, "Partial attention": each step yields the online-softmax
//    triple (max m, denominator l, numerator O); triples merge associatively.
//  * eq. g5cp-step-flops: every (rank, step) holds the same 2*C^2 visible pairs
//    (plus C on step 0), F_attn / cp^2.
//
// Layouts.  Balanced (the method): rank r owns chunks r and 2cp-1-r.  Sequential
// (the plain split the spec contrasts it with, kept for measuring imbalance):
// rank r owns chunks 2r and 2r+1.  A launch covers the ranks [rank_begin,
// rank_end) and the steps [step_begin, step_end).
//
// Work decomposition.  One CTA owns one 128-row query tile of one chunk for up
// to two query heads that share a kv head (grouped-query attention), and walks
// the ring steps [step_begin, step_end) in order.  For each step it visits the
// 128-key tiles of the source rank's two chunks that its rows can see: chunks
// before the query chunk are fully visible, the query chunk itself (step 0 only)
// is the causal diagonal, later chunks are skipped.  The running triple stays on
// chip across all steps, so the between-step merge is the online-softmax update
// itself; the epilogue emits the triple, or merges it into the triple already in
// HBM, and optionally normalises.  CTAs are ordered in groups of (sequence, kv head)
// units whose K/V fits in L2 together (so each K/V tile comes from DRAM about once),
// latest chunk first (longest first) within a group; the hardware block scheduler
// hands them out as SMs free up.
//
// Per CTA (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q tiles once, then K_j, V_j into a ring of smem slots
//   warp 1      TMEM owner and MMA issuer (converged warp, one elected lane issues)
//   warps 4-7   softmax of query tile A (thread = row = TMEM lane)
//   warps 8-11  softmax of query tile B
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D), O_B.  At d = 128
// P (bf16) is written over the first 64 columns of its S tile and fed to the PV MMA
// from TMEM.  The MMA warp issues PV_T(j) before S_T(j+1), and tcgen05.mma executes
// in issue order, so P_T(j) is consumed before S_T(j+1) overwrites it.  The commit
// that signals S_T(j+1) also covers PV_T(j), so softmax may rescale O_T then.  At
// d = 64 P_A, P_B have columns of their own, [384,448) and [448,512): S_T(j+1) is
// issued as soon as the softmax has read S_T(j), and the softmax waits for PV_T(j-1)
// before it stores P or rescales O.  A launch of few single query tiles splits each
// tile's key walk over a cluster of CTAs instead (three S buffers, see below).
//
// A launch with CP_MODE_OVERLAP_PREVIOUS is a programmatic dependent of the kernel
// before it: its CTAs may start in that kernel's tail and touch (o, m, l) only after
// griddepcontrol.wait.
//
// Softmax runs in base 2 on logits scaled by scale*log2(e).  The reference max
// used for the exponent is only raised when the row max grows by more than 8
// (a factor 256): the triple (m_ref, l, O) stays exact, P <= 256 fits bf16, and
// O is rescaled in TMEM only on those rare raises.  The true max is tracked on
// the side and the epilogue re-expresses (l, O) against it, so the stored m is
// the definition's max.
//
// Every mbarrier wait is bounded (about 1 s); on expiry the CTA records
// CP_ERR_TIMEOUT in a device status word, every role bails out, in-flight async
// copies are given time to land, TMEM is freed and the CTA returns.  While that
// word holds an error, CTAs of later launches return at once without writing
// (the outputs are undefined until cp_take_device_status clears it).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"
#include "tc_ptx.h"

namespace cpattn {
namespace {

constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // keys per KV tile
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int64_t kL2UnitBudget = int64_t(40) << 20;  // K/V bytes of one group of work items

__device__ int32_t g_ring_status = 0;

template <int D>
struct Cfg {
  static constexpr int kSlab = BM * 128;             // bytes of one 64-column swizzled slab
  static constexpr int kSlabs = D / 64;
  static constexpr int kTileBytes = BM * D * 2;      // Q tile, K tile and V tile alike
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr int kQOff = 0;
  static constexpr int kKvOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKvOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 1024 + 1024;  // barriers/flags + alignment slack
  // A launch whose key walks are split over a cluster also exchanges each row's (m, l)
  // and the merge weights through shared memory after the barriers.
  static constexpr int kSplitOff = kBarOff + 1024;
  static constexpr int kSplitSmemBytes = kSmemBytes + 2048;
  static constexpr uint32_t kOCol = 256;
  // d = 64 (unsplit): O takes columns 256-383, so P gets columns of its own, 384 + 64 tt,
  // and S is free as soon as the softmax has read it.
  static constexpr bool kEarlyS = D == 64;
  static constexpr uint32_t kPCol = 384;
};

struct RingParams {
  CUtensorMap tmap_q;  // dims (d, h_q, S, b)
  CUtensorMap tmap_k;  // dims (d, h_kv, S, b)
  CUtensorMap tmap_v;
  CUtensorMap tmap_o;  // fp32, dims (d, h_q, S, b), box 32 x 1 x 128 x 1: O tile stores
  float* o;
  float* m;
  float* l;
  int64_t b, S, h_q, h_kv;
  int32_t C;          // chunk length S / (2 cp)
  int32_t cp;
  int32_t tpc;        // query tiles per chunk
  int32_t row_pairs;  // 1: a CTA takes two consecutive query tiles of one head (odd group)
  int32_t ipc;        // work items per chunk along its rows: tpc, or ceil(tpc / 2) with row_pairs
  int32_t n_pairs;    // items per batch entry and row item: h_kv * ppg
  int32_t ppg;        // items per kv group and row item: head pairs, or heads with row_pairs
  int32_t group;      // h_q / h_kv
  int32_t step_begin, step_end;
  int32_t mode;
  int32_t rank_begin, rank_end;  // virtual ranks whose rows this launch computes
  int32_t chunks;                // RingChunks: both chunks of each rank, or only the first / second
  int32_t unit_groups;           // (sequence, kv head) units are taken in this many groups
  float sl;           // scale * log2(e)
  int32_t kv_split;   // CTAs (one cluster) that share each item's key walk; 1 = not split
};

// ---------------------------------------------------------------------------
// PTX wrappers (tc_ptx.h) and this kernel's status word
// ---------------------------------------------------------------------------

using namespace tc;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag) {
  return mbar_wait_bounded(bar, parity, abort_flag, &g_ring_status);
}

__host__ __device__ constexpr uint32_t instr_desc(int n, bool b_mn_major) {
  return instr_desc_bf16(BM, n, false, b_mn_major);
}

// ---------------------------------------------------------------------------
// Ring schedule: the KV tiles one query tile visits over steps [t0, t1)
// ---------------------------------------------------------------------------

template <int LAYOUT>
struct KvCursor {
  int32_t cp, r, c_q, t, t_end, half;
  int32_t C, q_last;
  int32_t seg_key0, seg_n, seg_end, seg_i;
  bool seg_diag;

  __device__ void init(int32_t cp_, int32_t r_, int32_t c_q_, int32_t t0, int32_t t1, int32_t C_,
                       int32_t q_last_) {
    cp = cp_; r = r_; c_q = c_q_; t = t0; t_end = t1; half = 0;
    C = C_; q_last = q_last_;
    seg_key0 = seg_n = seg_end = seg_i = 0;
    seg_diag = false;
  }

  // Next non-empty chunk segment: per step the first chunk of the source rank,
  // then its second chunk (balanced: s and 2cp-1-s; sequential: 2s and 2s+1).
  __device__ void find() {
    seg_n = 0;
    while (t < t_end) {
      const int32_t s = ((r - t) % cp + cp) % cp;
      const int32_t c = (LAYOUT == CP_LAYOUT_SEQUENTIAL) ? (2 * s + half)
                                                       : ((half == 0) ? s : 2 * cp - 1 - s);
      half ^= 1;
      if (half == 0) ++t;
      seg_i = 0;
      seg_key0 = c * C;
      seg_end = (c + 1) * C;
      if (c < c_q) {
        seg_diag = false;
        seg_n = (C + BN - 1) / BN;
        return;
      }
      if (c == c_q) {
        seg_diag = true;
        seg_n = (q_last - c * C) / BN + 1;
        return;
      }
    }
  }

  // Number of tiles next() yields over [t0, t1): the same segments, counted per
  // segment instead of per tile.
  __device__ static int32_t count(int32_t cp, int32_t r, int32_t c_q, int32_t t0, int32_t t1, int32_t C,
                                  int32_t q_last) {
    const int32_t full = (C + BN - 1) / BN;
    int32_t n = 0;
    int32_t s = ((r - t0) % cp + cp) % cp;
    for (int32_t t = t0; t < t1; ++t) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int32_t c = (LAYOUT == CP_LAYOUT_SEQUENTIAL) ? (2 * s + half) : ((half == 0) ? s : 2 * cp - 1 - s);
        if (c < c_q) {
          n += full;
        } else if (c == c_q) {
          n += (q_last - c * C) / BN + 1;
        }
      }
      s = (s == 0) ? cp - 1 : s - 1;
    }
    return n;
  }

  __device__ bool next(int32_t& key0, int32_t& key_end, bool& diag) {
    if (seg_i >= seg_n) {
      find();
      if (seg_n == 0) return false;
    }
    key0 = seg_key0 + BN * seg_i;
    key_end = seg_end;
    diag = seg_diag;
    ++seg_i;
    return true;
  }
};

// One CTA's work: query tile A and, when has_b, tile B, which share every K/V tile.
// Tile B is the next query head of the kv group (dh = 1, same rows; even groups) or
// the next 128 rows of the same head (drow = BM; odd groups, so that no head is left
// without a partner).
struct Item {
  int32_t bi, h0, has_b, kvh;
  int32_t c_q, r, q_row0, q_rows;
  int32_t dh, drow, q_rows_b, q_last;  // tile B's offsets and rows; the last row of either tile
};

template <int LAYOUT>
__device__ __forceinline__ Item decode_item(const RingParams& p, int32_t item) {
  Item it;
  const int32_t nr = p.rank_end - p.rank_begin;
  const int32_t n_qt = (p.chunks == kRingBothChunks ? 2 : 1) * nr * p.ipc;  // row items of the selected chunks
  // Units (sequence, kv head) in groups whose K/V fits in L2; within a group, the
  // latest chunk (most keys) first, then the group's head pairs (or heads).
  // The launch has fewer than 2^31 items, so every index here fits 32 bits.
  const int32_t upg = int32_t(p.b * p.h_kv) / p.unit_groups;  // units per group
  const int32_t per_tile = upg * p.ppg;
  const int32_t per_group = n_qt * per_tile;
  const int32_t g = item / per_group;
  const int32_t idx = item - g * per_group;
  const int32_t gq = n_qt - 1 - idx / per_tile;
  const int32_t bp = idx - (n_qt - 1 - gq) * per_tile;
  const int32_t u = bp / p.ppg;
  const int32_t i = bp - u * p.ppg;
  const int32_t unit = g * upg + u;
  it.bi = unit / int32_t(p.h_kv);
  it.kvh = unit - it.bi * int32_t(p.h_kv);
  it.h0 = it.kvh * p.group + (p.row_pairs ? i : 2 * i);
  // a-th selected chunk in ascending order.  Balanced: the ranks' head chunks
  // [rank_begin, rank_end) then their tail chunks [2cp-rank_end, 2cp-rank_begin);
  // sequential: chunks [2 rank_begin, 2 rank_end).  With one chunk per rank selected,
  // only the head (first) or only the tail (second) chunks, in ascending order.
  int32_t a = gq / p.ipc;
  const int32_t kq = gq % p.ipc;
  if (p.chunks == kRingSecondChunk) a += nr;
  if (LAYOUT == CP_LAYOUT_SEQUENTIAL) {
    it.c_q = (p.chunks == kRingBothChunks) ? 2 * p.rank_begin + a
                                           : 2 * (p.rank_begin + (a % nr)) + (a >= nr ? 1 : 0);
    it.r = it.c_q / 2;
  } else {
    it.c_q = (a < nr) ? p.rank_begin + a : 2 * p.cp - p.rank_end + (a - nr);
    it.r = (it.c_q < p.cp) ? it.c_q : 2 * p.cp - 1 - it.c_q;
  }
  const int32_t tile0 = p.row_pairs ? 2 * kq : kq;  // first query tile of the item in its chunk
  it.q_row0 = it.c_q * p.C + BM * tile0;
  it.q_rows = min(BM, p.C - BM * tile0);
  if (p.row_pairs) {
    it.dh = 0;
    it.drow = BM;
    it.q_rows_b = max(0, min(BM, p.C - BM * (tile0 + 1)));
    it.has_b = it.q_rows_b > 0 ? 1 : 0;
    it.q_last = it.has_b ? it.q_row0 + BM + it.q_rows_b - 1 : it.q_row0 + it.q_rows - 1;
  } else {
    it.dh = 1;
    it.drow = 0;
    it.q_rows_b = it.q_rows;
    it.has_b = (2 * i + 1 < p.group) ? 1 : 0;
    it.q_last = it.q_row0 + it.q_rows - 1;
  }
  return it;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Cluster-wide barrier of all threads: arrive with release semantics (this CTA's
// shared-memory writes become visible to the cluster), wait with acquire semantics.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr) : "memory");
  return v;
}

// The merge of a split item, run by the 256 threads of warps 4-11 of cluster CTA `part`
// after the first cluster barrier: rows [part * R, (part + 1) * R) of the tile, R = 128 / P.  Per row: m =
// max over the parts, part weights w = e^{m_part - m} (0 for a part that saw no key),
// l = sum of w * l_part in part order; then O = sum of w * O_part in part order, and the
// launch's mode (EMIT / ACCUMULATE, FINALIZE) as in the unsplit epilogue.  Every peer's
// values are loaded before any is used, so the distributed shared-memory loads of a row
// or a column block are in flight together.
template <int D, int P>
__device__ __noinline__ void split_merge(const RingParams& p, const Item& it, int32_t part, uint8_t* smem,
                                         uint32_t sbase) {
  using K = Cfg<D>;
  constexpr int R = BM / P;
  constexpr int kMergeThreads = 256;
  const int t = threadIdx.x - 128;
  float* xm = reinterpret_cast<float*>(smem + K::kSplitOff);
  float* wt = xm + 2 * BM;       // [R][P] part weights
  float* wo = wt + BM;           // [R] weight of the merged O (new part)
  float* wold = wo + R;          // [R] weight of the O already in memory (ACCUMULATE)
  const uint32_t xm_a = smem_u32(xm);
  const uint32_t stage = sbase + uint32_t(K::kQOff);
  const bool accumulate = (p.mode & CP_MODE_ACCUMULATE) != 0;
  const bool fin = (p.mode & CP_MODE_FINALIZE) != 0;
  if (t < R) {
    const int r = part * R + t;  // row within the tile
    const int32_t row = it.q_row0 + r;
    float mq[P], lq[P];
#pragma unroll
    for (int q = 0; q < P; ++q) {
      mq[q] = ld_cluster_f32(cluster_addr(xm_a + uint32_t(r * 4), uint32_t(q)));
      lq[q] = ld_cluster_f32(cluster_addr(xm_a + uint32_t((BM + r) * 4), uint32_t(q)));
    }
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < P; ++q) mx = fmaxf(mx, mq[q]);
    const float sh = (mx == -INFINITY) ? 0.f : mx;
    float l = 0.f;
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const float w = __expf(mq[q] - sh);
      wt[t * P + q] = w;
      l = fmaf(w, lq[q], l);
    }
    // The merged triple (mx, l, O) against the mode, as the unsplit epilogue does.
    float alpha = 0.f, beta = 1.f, l_out = l, m_out = mx;
    const bool row_ok = r < it.q_rows && row < p.S;
    const int64_t ml_off = (int64_t(it.bi) * p.h_q + it.h0) * p.S + row;
    if (accumulate && row_ok) {
      const float m_old = p.m[ml_off];
      const float l_old = p.l[ml_off];
      m_out = fmaxf(m_old, mx);
      const float s2 = (m_out == -INFINITY) ? 0.f : m_out;
      alpha = __expf(m_old - s2);
      beta = __expf(mx - s2);
      l_out = alpha * l_old + beta * l;
    }
    const float inv = (fin && l_out > 0.f) ? 1.f / l_out : (fin ? 0.f : 1.f);
    wo[t] = beta * inv;
    wold[t] = alpha * inv;
    if (row_ok) {
      p.m[ml_off] = m_out;
      p.l[ml_off] = l_out;
    }
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");  // warps 4-11
  constexpr int kVec = D / 4;  // float4 columns of a row
  for (int e = t; e < R * kVec; e += kMergeThreads) {
    const int rl = e / kVec, c4 = e - rl * kVec;
    const int r = part * R + rl;
    const int32_t row = it.q_row0 + r;
    // box c4 / 8, row r, 16-byte chunk (c4 % 8) at position (c4 % 8) ^ (r % 8)
    const uint32_t off = stage + uint32_t((c4 / 8) * BM * 128 + r * 128 + (((c4 % 8) ^ (r & 7)) << 4));
    float4 x[P];
#pragma unroll
    for (int q = 0; q < P; ++q) x[q] = ld_cluster_v4(cluster_addr(off, uint32_t(q)));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const float w = wt[rl * P + q];
      acc.x = fmaf(w, x[q].x, acc.x);
      acc.y = fmaf(w, x[q].y, acc.y);
      acc.z = fmaf(w, x[q].z, acc.z);
      acc.w = fmaf(w, x[q].w, acc.w);
    }
    if (r < it.q_rows && row < p.S) {
      float4* dst = reinterpret_cast<float4*>(p.o + ((int64_t(it.bi) * p.S + row) * p.h_q + it.h0) * D) + c4;
      const float wn = wo[rl];
      float4 v;
      if (accumulate) {
        const float4 old = *dst;
        const float wd = wold[rl];
        v = make_float4(fmaf(old.x, wd, acc.x * wn), fmaf(old.y, wd, acc.y * wn), fmaf(old.z, wd, acc.z * wn),
                        fmaf(old.w, wd, acc.w * wn));
      } else {
        v = make_float4(acc.x * wn, acc.y * wn, acc.z * wn, acc.w * wn);
      }
      *dst = v;
    }
  }
}

// SPLIT: the CTAs of a cluster of p.kv_split share one item (one query tile): each walks a
// contiguous part of its K/V tiles, stages its partial triple in shared memory, and after
// a cluster barrier each merges a slice of the tile's rows from every part through
// distributed shared memory (the associative merge of the Terms table's "Partial
// attention" row) and writes them.  Used for launches of single query tiles that fill
// less than half the GPU, which otherwise run as one CTA's chain of K/V tiles.
template <int D, int LAYOUT, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) ring_attn_kernel(const __grid_constant__ RingParams p) {
  using K = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + K::kBarOff);
  // barrier slots
  const uint32_t bar_q = smem_u32(&bars[0]);  // Q of tile A
  const uint32_t bar_qb = smem_u32(&bars[16 + 2 * K::kStages]);  // Q of tile B (d = 64)
  constexpr bool kQSplit = D == 64;
  auto bar_full = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto bar_empty = [&](int s) { return smem_u32(&bars[1 + K::kStages + s]); };
  auto bar_s = [&](int tt) { return smem_u32(&bars[1 + 2 * K::kStages + tt]); };
  auto bar_p = [&](int tt) { return smem_u32(&bars[3 + 2 * K::kStages + tt]); };
  auto bar_o = [&](int tt) { return smem_u32(&bars[5 + 2 * K::kStages + tt]); };
  auto bar_e = [&](int tt) { return smem_u32(&bars[7 + 2 * K::kStages + tt]); };  // O tile staged
  auto bar_l = [&](int tt) { return smem_u32(&bars[9 + 2 * K::kStages + tt]); };  // old O tile loaded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[11 + 2 * K::kStages]);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  // A split launch has one query tile per CTA and three S buffers (TMEM columns 0, 128 and
  // 384; O at 256): buffer b's S-ready and P-ready barriers are bar_s3(b) and bar_p3(b)
  // (tile B's slots for buffer 1 and two more for buffer 2), and bar_o(0) completes one
  // phase per PV.
  auto bar_s3 = [&](int b) { return b < 2 ? bar_s(b) : smem_u32(&bars[12 + 2 * K::kStages]); };
  auto bar_p3 = [&](int b) { return b < 2 ? bar_p(b) : smem_u32(&bars[13 + 2 * K::kStages]); };
  // Unsplit at d = 64, P lives apart from S: bar_sf(tt) completes when the tile's four
  // softmax warps have read S (the next S may then be issued into it), and bar_o(tt)
  // completes once per PV, which the softmax waits for before it reuses the P columns
  // or rescales O.
  constexpr bool kEarlyS = K::kEarlyS && !SPLIT;
  auto bar_sf = [&](int tt) { return smem_u32(&bars[14 + 2 * K::kStages + tt]); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int32_t part = SPLIT ? int32_t(blockIdx.x) % p.kv_split : 0;  // this CTA's rank in its cluster
  const Item it = decode_item<LAYOUT>(p, SPLIT ? int32_t(blockIdx.x) / p.kv_split : int32_t(blockIdx.x));
  // A ring launch that follows this one on the stream with CP_MODE_OVERLAP_PREVIOUS may
  // start its CTAs as soon as all of this grid's CTAs are running: it touches (o, m, l)
  // only after grid_dependency_wait, that is, after this grid has finished.
  grid_launch_dependents();

  if constexpr (!SPLIT) {
    // An item that sees no key over the step range (a head chunk whose source chunks all
    // lie after it): merging the identity into a running triple changes nothing, so
    // ACCUMULATE without FINALIZE leaves it as it is; EMIT writes the identity (O = 0,
    // m = -inf, l = 0; FINALIZE gives O = 0 as well) with plain stores.  No barrier,
    // TMEM or copy is set up.  (ACCUMULATE | FINALIZE normalises the old triple below.)
    if (KvCursor<LAYOUT>::count(p.cp, it.r, it.c_q, p.step_begin, p.step_end, p.C, it.q_last) == 0) {
      const bool acc = (p.mode & CP_MODE_ACCUMULATE) != 0;
      if (acc && (p.mode & CP_MODE_FINALIZE) == 0) return;
      if (!acc) {
        grid_dependency_wait();  // the kernel before this one may still own (o, m, l)
        if (*reinterpret_cast<volatile int32_t*>(&g_ring_status) != 0) return;  // an earlier wait gave up
        for (int tt = 0; tt <= it.has_b; ++tt) {
          const int h = it.h0 + tt * it.dh;
          const int32_t row0 = it.q_row0 + tt * it.drow;
          const int32_t rows = tt ? it.q_rows_b : it.q_rows;
          for (int e = threadIdx.x; e < rows * (D / 4); e += kThreads) {
            const int32_t row = row0 + e / (D / 4);
            reinterpret_cast<float4*>(p.o + ((int64_t(it.bi) * p.S + row) * p.h_q + h) * D)[e % (D / 4)] =
                make_float4(0.f, 0.f, 0.f, 0.f);
          }
          for (int r = threadIdx.x; r < rows; r += kThreads) {
            const int64_t ml = (int64_t(it.bi) * p.h_q + h) * p.S + row0 + r;
            p.m[ml] = -INFINITY;
            p.l[ml] = 0.f;
          }
        }
        return;
      }
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_qb, 1);
    for (int s = 0; s < K::kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int tt = 0; tt < 2; ++tt) {
      mbar_init(bar_s(tt), 1);
      mbar_init(bar_p(tt), BM / 32);
      mbar_init(bar_o(tt), 1);
      mbar_init(bar_e(tt), BM / 32);
      mbar_init(bar_l(tt), 1);
    }
    if constexpr (SPLIT) {
      mbar_init(bar_s3(2), 1);
      mbar_init(bar_p3(2), BM / 32);
    }
    if constexpr (kEarlyS) {
      mbar_init(bar_sf(0), BM / 32);
      mbar_init(bar_sf(1), BM / 32);
    }
    // An earlier wait gave up: the whole CTA skips its work (decided once, CTA-uniform).
    *abort_flag = (*reinterpret_cast<volatile int32_t*>(&g_ring_status) != 0) ? 1 : 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;
  // Number of KV tiles this query tile visits over the step range; split, this CTA's
  // contiguous part of them, from tile kv_lo on.
  const int32_t n_all = KvCursor<LAYOUT>::count(p.cp, it.r, it.c_q, p.step_begin, p.step_end, p.C,
                                                it.q_last);
  const int32_t kv_lo = SPLIT ? part * n_all / p.kv_split : 0;
  const int32_t n_kv = SPLIT ? (part + 1) * n_all / p.kv_split - kv_lo : n_all;
  const int n_q = 1 + it.has_b;

  // Register split (launched with 168 per thread, 64,512 in all): the producer /
  // MMA warpgroup gives registers to the two softmax warpgroups.
  // 128 x 72 + 256 x 216 = 64,512 <= 64,512, so the increase never waits.  Each
  // role's code is reachable only after its own setmaxnreg; the common tail is tiny.
  // A split launch's cluster barriers: every thread of every CTA of the cluster passes
  // exactly two, in whichever branch below it takes (no role returns early and every wait
  // before them is bounded), so they always complete.  The first makes the parts' staged
  // triples visible across the cluster; the second keeps each CTA's shared memory alive
  // until every peer has read it.  The merge between them runs in the softmax warps.
  if (skip) {
    // nothing to do: fall through to the teardown
    if constexpr (SPLIT) {
      cluster_sync_all();
      cluster_sync_all();
    }
  } else if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_kv > 0) {
      // L2 policy: a Q tile is read by this CTA alone, while every query tile of the
      // kv head re-reads its K/V tiles, so K/V should outlive Q (and O) in L2.
      const uint64_t pol_once = l2_policy_evict_first();
      // d = 64: Q of tile A, then K_0, then Q of tile B (right after K_0 in the loop below),
      // so tile A's first QK^T can start before tile B's Q is in.  d = 128: both Q tiles
      // first, on one barrier.
      auto load_q = [&](int tt) {
        const uint32_t bar = (kQSplit && tt == 1) ? bar_qb : bar_q;
        for (int sl = 0; sl < K::kSlabs; ++sl)
          tma_load_4d_hint(sbase + K::kQOff + tt * K::kTileBytes + sl * K::kSlab, &p.tmap_q, bar, sl * 64,
                           it.h0 + tt * it.dh, it.q_row0 + tt * it.drow, it.bi, pol_once);
      };
      if constexpr (kQSplit) {
        mbar_expect_tx(bar_q, uint32_t(K::kTileBytes));
        load_q(0);
      } else {
        mbar_expect_tx(bar_q, uint32_t(n_q * K::kTileBytes));
        for (int tt = 0; tt < n_q; ++tt) load_q(tt);
      }
      KvCursor<LAYOUT> cur;
      cur.init(p.cp, it.r, it.c_q, p.step_begin, p.step_end, p.C, it.q_last);
      int32_t key0, key_end;
      bool diag;
      if constexpr (SPLIT)
        for (int32_t i = 0; i < kv_lo; ++i) cur.next(key0, key_end, diag);
      int32_t li = 0;  // load index: K_j = 2j, V_j = 2j + 1
      bool ok = true;
      // ACCUMULATE reads the running triple at the end: bring its O tiles and m, l rows
      // into L2 once the K/V pipeline is full, so that they do not delay the first loads.
      bool prefetched = (p.mode & CP_MODE_ACCUMULATE) == 0;
      auto prefetch_old = [&]() {
        for (int tt = 0; tt < n_q; ++tt) {
          const int32_t row0 = it.q_row0 + tt * it.drow;
          const int32_t rows = tt ? it.q_rows_b : it.q_rows;
          const bool staged = rows == BM && row0 + BM <= p.S;
          const int64_t ml = (int64_t(it.bi) * p.h_q + it.h0 + tt * it.dh) * p.S + row0;
          for (int i = 0; i < rows; i += 32) {
            prefetch_l2(p.m + ml + i);
            prefetch_l2(p.l + ml + i);
          }
          prefetch_l2(p.m + ml + rows - 1);
          prefetch_l2(p.l + ml + rows - 1);
          if (staged)
            for (int c = 0; c < D / 32; ++c) tma_prefetch_4d(&p.tmap_o, c * 32, it.h0 + tt * it.dh, row0, it.bi);
        }
        prefetched = true;
      };
      while (ok && (!SPLIT || li < 2 * n_kv) && cur.next(key0, key_end, diag)) {
        for (int which = 0; which < 2 && ok; ++which, ++li) {
          if (!prefetched && li == K::kStages) prefetch_old();
          const int s = li % K::kStages;
          const int round = li / K::kStages;
          if (round > 0 && !mbar_wait(bar_empty(s), uint32_t((round - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar_full(s), uint32_t(K::kTileBytes));
          const CUtensorMap* map = which == 0 ? &p.tmap_k : &p.tmap_v;
          for (int sl = 0; sl < K::kSlabs; ++sl)
            tma_load_4d_hint(sbase + K::kKvOff + s * K::kTileBytes + sl * K::kSlab, map, bar_full(s), sl * 64,
                             it.kvh, key0, it.bi, l2_policy_evict_last());
          if (kQSplit && li == 0 && n_q == 2) {
            mbar_expect_tx(bar_qb, uint32_t(K::kTileBytes));
            load_q(1);
          }
        }
      }
      if (ok && !prefetched) prefetch_old();
      if (!ok) {  // let copies in flight land before the CTA can exit
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop in step (waits, descriptors, counters); one
    // elected lane issues each MMA and commit.
    if (n_kv > 0) {
      const uint32_t is = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
      };
      constexpr uint32_t idesc_s = instr_desc(BN, false);
      constexpr uint32_t idesc_pv = instr_desc(D, true);
      const uint32_t s_col[2] = {0u, 128u};
      const uint32_t o_col[2] = {K::kOCol, K::kOCol + uint32_t(D)};
      bool ok = wait(bar_q, 0);
      auto issue_s = [&](int tt, int slot) {
        const uint32_t qa = sbase + K::kQOff + tt * K::kTileBytes;
        const uint32_t ka = sbase + K::kKvOff + slot * K::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * K::kSlab + (kk % 4) * 32;
          mma_ss_if(is, tmem + s_col[tt], smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), idesc_s,
                    kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int tt, int slot, bool accumulate) {
        const uint32_t va = sbase + K::kKvOff + slot * K::kTileBytes;
        const uint32_t pa = kEarlyS ? K::kPCol + uint32_t(tt * 64) : s_col[tt];  // P's columns
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_ts_if(is, tmem + o_col[tt], tmem + pa + uint32_t(kk * 8),
                    smem_desc(va + kk * 2048, K::kSlab, 1024), idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      if constexpr (SPLIT) {
        // One query tile, three S buffers: S of K/V tile j goes to buffer j % 3 and is
        // issued right after the PV of tile j - 3 (the last reader of that buffer's P),
        // so the softmax of tile j + 1 need not wait for PV(j).  tcgen05.mma executes in
        // issue order, so a buffer's P is consumed before the next S overwrites it.
        auto s3_col = [](int b) { return b == 2 ? 384u : uint32_t(b) * 128u; };
        auto s_step = [&](int32_t jj) -> bool {
          const int lk = 2 * jj, sk = lk % K::kStages;
          if (!wait(bar_full(sk), uint32_t((lk / K::kStages) & 1))) return false;
          tc_fence_after();
          const int b = jj % 3;
          const uint32_t qa = sbase + K::kQOff;
          const uint32_t ka = sbase + K::kKvOff + sk * K::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * K::kSlab + (kk % 4) * 32;
            mma_ss_if(is, tmem + s3_col(b), smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), idesc_s,
                      kk > 0 ? 1u : 0u);
          }
          mma_commit_if(is, bar_s3(b));
          mma_commit_if(is, bar_empty(sk));  // K_jj consumed
          return true;
        };
        for (int32_t jj = 0; ok && jj < 3 && jj < n_kv; ++jj) ok = s_step(jj);
        for (int32_t j = 0; ok && j < n_kv; ++j) {
          const int lv = 2 * j + 1, sv = lv % K::kStages;
          if (!wait(bar_full(sv), uint32_t((lv / K::kStages) & 1))) { ok = false; break; }
          const int b = j % 3;
          if (!wait(bar_p3(b), uint32_t((j / 3) & 1))) { ok = false; break; }
          tc_fence_after();
          const uint32_t va = sbase + K::kKvOff + sv * K::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            mma_ts_if(is, tmem + K::kOCol, tmem + s3_col(b) + uint32_t(kk * 8),
                      smem_desc(va + kk * 2048, K::kSlab, 1024), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_if(is, bar_empty(sv));  // V_j consumed
          mma_commit_if(is, bar_o(0));       // PV(j) done: one phase per K/V tile
          if (j + 3 < n_kv && !s_step(j + 3)) { ok = false; break; }
        }
      } else if constexpr (kEarlyS) {
        // S(j + 1) of a tile is issued as soon as its softmax has read S(j) and K_{j+1} is in,
        // so it runs during that softmax; PV(j) follows once P(j) is stored.  bar_o(tt)
        // completes after every PV.  Per K/V tile the order is S_A(j + 1), PV_A(j),
        // S_B(j + 1), PV_B(j), so tile B's last PV is the last MMA and tile A's comes after
        // every S: the epilogue's staging (tile A in the Q tiles, tile B in K/V slots)
        // relies on that.  (Both S before both PV measured 1 % slower on row-paired tiles
        // and 2-4 % faster on head-paired ones; a warp that polls both tiles and issues
        // whichever MMA is ready was slower than either and breaks that staging order.)
        if (ok) ok = wait(bar_full(0), 0);
        if (ok) {
          tc_fence_after();
          for (int tt = 0; ok && tt < n_q; ++tt) {
            if (kQSplit && tt == 1 && !(ok = wait(bar_qb, 0))) break;
            issue_s(tt, 0);
            mma_commit_if(is, bar_s(tt));
          }
          if (ok) mma_commit_if(is, bar_empty(0));
        }
        for (int32_t j = 0; ok && j < n_kv; ++j) {
          const int lv = 2 * j + 1, lk = 2 * j + 2;
          const int sv = lv % K::kStages, sk = lk % K::kStages;
          const bool more = (j + 1 < n_kv);
          if (more && !wait(bar_full(sk), uint32_t((lk / K::kStages) & 1))) { ok = false; break; }
          if (!wait(bar_full(sv), uint32_t((lv / K::kStages) & 1))) { ok = false; break; }
          for (int tt = 0; tt < n_q; ++tt) {
            if (more) {
              if (!wait(bar_sf(tt), uint32_t(j & 1))) { ok = false; break; }
              tc_fence_after();
              issue_s(tt, sk);
              mma_commit_if(is, bar_s(tt));
              if (tt == n_q - 1) mma_commit_if(is, bar_empty(sk));  // K_{j+1} consumed by every tile
            }
            if (!wait(bar_p(tt), uint32_t(j & 1))) { ok = false; break; }
            tc_fence_after();
            issue_pv(tt, sv, j > 0);
            mma_commit_if(is, bar_o(tt));
            if (tt == n_q - 1) mma_commit_if(is, bar_empty(sv));  // V_j consumed by every tile
          }
        }
      } else {
      // prologue: S(0) for both tiles
      if (ok) ok = wait(bar_full(0), 0);
      if (ok) {
        tc_fence_after();
        for (int tt = 0; ok && tt < n_q; ++tt) {
          if (kQSplit && tt == 1 && !(ok = wait(bar_qb, 0))) break;
          issue_s(tt, 0);
          mma_commit_if(is, bar_s(tt));
        }
        if (ok) mma_commit_if(is, bar_empty(0));
      }
      for (int32_t j = 0; ok && j < n_kv; ++j) {
        const int lv = 2 * j + 1, lk = 2 * j + 2;
        const int sv = lv % K::kStages, sk = lk % K::kStages;
        if (!wait(bar_full(sv), uint32_t((lv / K::kStages) & 1))) { ok = false; break; }
        const bool more = (j + 1 < n_kv);
        bool k_ready = false;
        for (int tt = 0; tt < n_q; ++tt) {
          if (!wait(bar_p(tt), uint32_t(j & 1))) { ok = false; break; }
          tc_fence_after();
          issue_pv(tt, sv, j > 0);
          if (tt == n_q - 1) mma_commit_if(is, bar_empty(sv));  // V_j consumed by every tile
          if (more) {
            if (!k_ready) {
              if (!wait(bar_full(sk), uint32_t((lk / K::kStages) & 1))) { ok = false; break; }
              tc_fence_after();
              k_ready = true;
            }
            issue_s(tt, sk);
            mma_commit_if(is, bar_s(tt));
            if (tt == n_q - 1) mma_commit_if(is, bar_empty(sk));  // K_{j+1} consumed
          } else {
            mma_commit_if(is, bar_o(tt));
          }
        }
      }
      }  // !SPLIT
      if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
  }
  if constexpr (SPLIT) {
    cluster_sync_all();
    cluster_sync_all();
  }
  } else {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
  if (warp < 8 || it.has_b) {
    // ------------------------------------------------------------ softmax + epilogue
    const int tt = (warp - 4) / 4;
    const int t = threadIdx.x - 128 * (1 + tt);  // row within the tile == TMEM lane
    const int h = it.h0 + tt * it.dh;
    const int32_t row0 = it.q_row0 + tt * it.drow;  // this tile's first row
    const int32_t rows = tt ? it.q_rows_b : it.q_rows;
    const int32_t row = row0 + t;
    const uint32_t lane_base = uint32_t((warp % 4) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + uint32_t(tt * 128);
    const uint32_t o_addr = tmem + lane_base + K::kOCol + uint32_t(tt * D);
    const uint32_t p_addr = tmem + lane_base + K::kPCol + uint32_t(tt * 64);  // d = 64 unsplit
    float m_ref = -INFINITY;   // exponent reference (log2 units)
    float m_true = -INFINITY;  // true running max (log2 units)
    float l_run = 0.f;
    bool ok = true;

    KvCursor<LAYOUT> cur;
    cur.init(p.cp, it.r, it.c_q, p.step_begin, p.step_end, p.C, it.q_last);
    if constexpr (SPLIT) {
      int32_t key0, key_end;
      bool diag;
      for (int32_t i = 0; i < kv_lo; ++i) cur.next(key0, key_end, diag);
    }
    for (int32_t j = 0; j < n_kv; ++j) {
      int32_t key0 = 0, key_end = 0;
      bool diag = false;
      cur.next(key0, key_end, diag);
      // Warp-uniform outcome: the TMEM accesses below are warp-collective.
      // Split: this tile's S buffer for K/V tile j is j % 3 (its j / 3-th use).
      const int b3 = SPLIT ? int(j % 3) : tt;
      const uint32_t s_cur = SPLIT ? tmem + lane_base + (b3 == 2 ? 384u : uint32_t(b3) * 128u) : s_addr;
      if (!__all_sync(0xffffffffu, mbar_wait(SPLIT ? bar_s3(b3) : bar_s(tt), SPLIT ? uint32_t((j / 3) & 1)
                                                                                  : uint32_t(j & 1),
                                             abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Raw logits of this row (the scale is applied inside the exponent's FFMA).
      uint32_t sr[BN];
      tmem_ld128(s_cur, sr);
      tmem_ld_wait128(sr);
      if constexpr (kEarlyS) {  // S is in registers: the next S may overwrite its columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sf(tt));
      }
      float x[BN];
#pragma unroll
      for (int i = 0; i < BN; ++i) x[i] = __uint_as_float(sr[i]);
      const bool full = (key0 + BN <= key_end) && (!diag || key0 + BN - 1 <= row0);
      if (!full) {
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int32_t key = key0 + i;
          const bool vis = key < key_end && (!diag || key <= row);
          x[i] = vis ? x[i] : -INFINITY;
        }
      }
      // Row max: eight independent chains of three-input max (short dependency depth).
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        mx8[a] = fmaxf(x[a], x[a + 8]);
#pragma unroll
        for (int kk = 2; kk < BN / 8; kk += 2) mx8[a] = max3(mx8[a], x[a + 8 * kk], x[a + 8 * kk + 8]);
      }
      const float tmax = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], max3(mx8[5], mx8[6], mx8[7]))) *
                         p.sl;
      m_true = fmaxf(m_true, tmax);
      // Raise the exponent reference only when the max grew by more than the threshold.
      const bool raise = tmax > m_ref + kRescaleThreshold;
      const float m_new = raise ? tmax : m_ref;
      const float corr = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
      const bool rescale_o = raise && j > 0 && m_ref != -INFINITY;
      if (raise) {
        l_run *= corr;
        m_ref = m_new;
      }
      const float nmu = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // p = 2^(x*sl - m_ref): paired FFMA, MUFU ex2, paired adds into four pair accumulators.
      float ps8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) ps8[a] = 0.f;
      // All 64 packed columns of P go back in one TMEM store (fewer store instructions
      // measured faster than four or eight smaller ones).
      {
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float ya, yb;
          fma2(ya, yb, x[2 * i], x[2 * i + 1], p.sl, p.sl, nmu, nmu);
          const float a = ex2(ya);
          const float b = ex2(yb);
          const int acc = (2 * i) % 8;
          add2(ps8[acc], ps8[acc + 1], ps8[acc], ps8[acc + 1], a, b);
          pk[i] = pack_bf16(a, b);
        }
        if constexpr (kEarlyS) {
          // P's columns and O are free once PV(j - 1) has completed (S(j) no longer implies it).
          if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(bar_o(tt), uint32_t((j - 1) & 1), abort_flag)))
            ok = false;
          if (ok) {
            tc_fence_after();
            tmem_st64(p_addr, pk);
          }
        } else {
          tmem_st64(s_cur, pk);
        }
      }
      if (!ok) break;
      const float psum = ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
      // O is rescaled after P is out (the logits are dead by then); PV_T(j)
      // cannot start before this thread's arrive below.  Split, this S was issued before
      // PV(j - 1), so first wait for PV(j - 1) (every K/V tile, one phase each).
      if (SPLIT && j > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(bar_o(0), uint32_t((j - 1) & 1), abort_flag))) {
        ok = false;
        break;
      }
      if (__any_sync(0xffffffffu, rescale_o)) {
        const float f = rescale_o ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + uint32_t(c * 32), r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
          tmem_st32(o_addr + uint32_t(c * 32), r);
        }
      }
      l_run += psum;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(SPLIT ? bar_p3(b3) : bar_p(tt));  // one arrival per warp (count 4)
    }

    // ---------------- epilogue: this row's triple, merged / normalised as asked
    // (o, m, l) are read and written only from here on: under CP_MODE_OVERLAP_PREVIOUS
    // the kernel before this one on the stream may have been running until now.
    grid_dependency_wait();
    const bool have = ok && n_kv > 0;
    if (have && !__all_sync(0xffffffffu, mbar_wait(bar_o(tt), (SPLIT || kEarlyS) ? uint32_t((n_kv - 1) & 1) : 0u,
                                                   abort_flag)))
      ok = false;
    if (ok) {
      tc_fence_after();
      // Re-express (l, O) against the true max: factor 2^(m_ref - m_true) <= 1.
      const float fre = (m_true == -INFINITY) ? 0.f : ex2(m_ref - m_true);
      const float m_new_nat = m_true * kLn2;
      const float l_new = l_run * fre;
      if constexpr (SPLIT) {
        // This part's triple of every row of the tile, against the part's own max: m and
        // l into the exchange arrays, O * 2^(m_ref - m_true) into the Q tiles' space
        // (every MMA that read it has completed) in the 128-byte-swizzled layout of the
        // staged stores.  The merge after the cluster barrier reads them.
        float* xm = reinterpret_cast<float*>(smem + K::kSplitOff);
        xm[t] = m_new_nat;
        xm[BM + t] = l_new;
        const uint32_t stage = sbase + uint32_t(K::kQOff);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (have) {
            tmem_ld32(o_addr + uint32_t(c * 32), r);
            tmem_ld_wait(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          const uint32_t rowa = stage + uint32_t(c * BM * 128 + t * 128);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_shared_v4(rowa + uint32_t(((k ^ (t & 7)) << 4)), __uint_as_float(r[4 * k]) * fre,
                         __uint_as_float(r[4 * k + 1]) * fre, __uint_as_float(r[4 * k + 2]) * fre,
                         __uint_as_float(r[4 * k + 3]) * fre);
        }
      } else {
      const bool row_ok = t < rows && row < p.S;
      const bool accumulate = (p.mode & CP_MODE_ACCUMULATE) != 0;
      // A whole 128-row tile moves its O rows through shared memory with TMA.
      const bool staged = rows == BM && row0 + BM <= p.S;
      const int64_t ml_off = (int64_t(it.bi) * p.h_q + h) * p.S + row;
      float alpha = 0.f, beta = 1.f, l_out = l_new, m_out = m_new_nat;
      if (accumulate && row_ok) {
        const float m_old = p.m[ml_off];
        const float l_old = p.l[ml_off];
        m_out = fmaxf(m_old, m_new_nat);
        const float sh = (m_out == -INFINITY) ? 0.f : m_out;
        alpha = __expf(m_old - sh);
        beta = __expf(m_new_nat - sh);
        l_out = alpha * l_old + beta * l_new;
      }
      const bool fin = (p.mode & CP_MODE_FINALIZE) != 0;
      const float inv = (fin && l_out > 0.f) ? 1.f / l_out : (fin ? 0.f : 1.f);
      const float wnew = beta * fre * inv;
      const float wold = alpha * inv;
      // Without ACCUMULATE the two factors are applied in turn, (O * 2^(m_ref - m_true)) / l,
      // exactly as an EMIT launch followed by a one-part finalising merge does, so the
      // fused result is bit for bit the same as that pair.
      const float wre = beta * fre;
      auto plain = [&](uint32_t bits) { return (__uint_as_float(bits) * wre) * inv; };
      // A whole 128-row tile goes through shared memory: ACCUMULATE first loads the
      // old O tile there, each thread combines its row in place, and TMA tile stores
      // (128 rows x 32 floats a box) write it out.  Partial tiles read and store each
      // row directly.  Staging: tile A uses the Q tiles' space, tile B two K/V slots;
      // every MMA that read them has completed once bar_o(tt) has fired.
      const uint32_t stage = sbase + (tt == 0 ? uint32_t(K::kQOff) : uint32_t(K::kKvOff));
      if (staged && accumulate) {
        const bool leader = warp == 4 + 4 * tt && lane == 0;
        if (leader) {
          mbar_expect_tx(bar_l(tt), uint32_t(BM * D * 4));
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            tma_load_4d(stage + uint32_t(c * BM * 128), &p.tmap_o, bar_l(tt), c * 32, h, row0, it.bi);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar_l(tt), 0, abort_flag))) {
          ok = false;
          if (leader) {  // let the copies in flight land before the CTA can exit
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 50000ull) {
            }
          }
        }
      }
      if (staged && ok) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (have) {
            tmem_ld32(o_addr + uint32_t(c * 32), r);
            tmem_ld_wait(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          // box c, row t, 16-byte chunk k at position k ^ (t % 8) (128-byte swizzle)
          const uint32_t rowa = stage + uint32_t(c * BM * 128 + t * 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t a = rowa + uint32_t(((k ^ (t & 7)) << 4));
            if (accumulate) {
              const float4 old = ld_shared_v4(a);
              st_shared_v4(a, fmaf(old.x, wold, __uint_as_float(r[4 * k]) * wnew),
                           fmaf(old.y, wold, __uint_as_float(r[4 * k + 1]) * wnew),
                           fmaf(old.z, wold, __uint_as_float(r[4 * k + 2]) * wnew),
                           fmaf(old.w, wold, __uint_as_float(r[4 * k + 3]) * wnew));
            } else {
              st_shared_v4(a, plain(r[4 * k]), plain(r[4 * k + 1]), plain(r[4 * k + 2]), plain(r[4 * k + 3]));
            }
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_e(tt));
        if (warp == 4 + 4 * tt && lane == 0) {
          if (mbar_wait(bar_e(tt), 0, abort_flag)) {
            const uint64_t pol_once = l2_policy_evict_first();
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
              tma_store_4d_hint(&p.tmap_o, stage + uint32_t(c * BM * 128), c * 32, h, row0, it.bi, pol_once);
            bulk_commit();
            bulk_wait_all();
          }
        }
      } else if (ok) {
        float* orow = p.o + ((int64_t(it.bi) * p.S + row) * p.h_q + h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (have) {
            tmem_ld32(o_addr + uint32_t(c * 32), r);
            tmem_ld_wait(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 v;
              if (accumulate) {
                const float4 old = *reinterpret_cast<const float4*>(orow + c * 32 + i);
                v.x = fmaf(old.x, wold, __uint_as_float(r[i]) * wnew);
                v.y = fmaf(old.y, wold, __uint_as_float(r[i + 1]) * wnew);
                v.z = fmaf(old.z, wold, __uint_as_float(r[i + 2]) * wnew);
                v.w = fmaf(old.w, wold, __uint_as_float(r[i + 3]) * wnew);
              } else {
                v = make_float4(plain(r[i]), plain(r[i + 1]), plain(r[i + 2]), plain(r[i + 3]));
              }
              *reinterpret_cast<float4*>(orow + c * 32 + i) = v;
            }
          }
        }
      }
      if (row_ok && ok) {
        p.m[ml_off] = m_out;
        p.l[ml_off] = l_out;
      }
      }  // !SPLIT
    }
  }
  if constexpr (SPLIT) {
    // warps 4-11 (all 256 of them, whether or not they had a tile) merge the rows
    grid_dependency_wait();
    cluster_sync_all();
    if (p.kv_split == 2)
      split_merge<D, 2>(p, it, part, smem, sbase);
    else if (p.kv_split == 4)
      split_merge<D, 4>(p, it, part, smem, sbase);
    else
      split_merge<D, 8>(p, it, part, smem, sbase);
    cluster_sync_all();
  }

  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// One CTA waits, with the ring kernel's bounded wait, on an mbarrier that nothing
// will ever complete: after about a second the wait gives up and records
// CP_ERR_TIMEOUT in the ring kernel's status word, exactly as a stalled ring
// launch would.  Used to test the failure path without faulting the GPU.
__global__ void ring_wait_timeout_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, &abort_flag);
  __syncthreads();
}

// 4-D bf16 map over a [b, S, h, d] tensor: dims (d, h, S, b), box (64, 1, 128, 1), 128-byte swizzle.
// 4-D fp32 map over the [b, S, h, d] output: box (32, 1, 128, 1), 128-byte swizzle.
bool encode_map_o(CUtensorMap* map, const void* base, int64_t b, int64_t S, int64_t h, int64_t d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(h), cuuint64_t(S), cuuint64_t(b)};
  const cuuint64_t strides[3] = {cuuint64_t(d * 4), cuuint64_t(h * d * 4), cuuint64_t(S * h * d * 4)};
  const cuuint32_t box[4] = {32, 1, BM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_map(CUtensorMap* map, const void* base, int64_t b, int64_t S, int64_t h, int64_t d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(h), cuuint64_t(S), cuuint64_t(b)};
  const cuuint64_t strides[3] = {cuuint64_t(d * 2), cuuint64_t(h * d * 2), cuuint64_t(S * h * d * 2)};
  const cuuint32_t box[4] = {64, 1, BM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int LAYOUT>
cp_status launch_d(const RingParams& p, int64_t n_items, cudaStream_t stream) {
  using K = Cfg<D>;
  if (LAYOUT == CP_LAYOUT_BALANCED && p.kv_split > 1) {
    // One cluster of kv_split CTAs per item (at most 8, the portable cluster size).
    auto kern = ring_attn_kernel<D, CP_LAYOUT_BALANCED, true>;
    static SmemLimit lim_split;
    if (raise_smem_limit(reinterpret_cast<const void*>(kern), K::kSplitSmemBytes, &lim_split) != cudaSuccess)
      return CP_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(unsigned(n_items * p.kv_split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = K::kSplitSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.kv_split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  }
  static SmemLimit lim;
  if (raise_smem_limit(reinterpret_cast<const void*>(ring_attn_kernel<D, LAYOUT, false>), K::kSmemBytes, &lim) !=
      cudaSuccess)
    return CP_ERR_CUDA;
  if ((p.mode & CP_MODE_OVERLAP_PREVIOUS) != 0) {
    // Programmatic dependent launch: the CTAs may start while the kernel before this one
    // on the stream still runs; each waits for it before touching (o, m, l).
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(unsigned(n_items), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = K::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ring_attn_kernel<D, LAYOUT, false>, p) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  }
  ring_attn_kernel<D, LAYOUT, false><<<unsigned(n_items), kThreads, K::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace

bool ring_supported(const cp_attn_desc& d) {
  // Keys and rows are indexed with int32 inside the kernel.
  return (d.d == 64 || d.d == 128) && d.S < (int64_t(1) << 30) && d.b <= 65535 && d.h_q <= 65535;
}

cp_status launch_ring_attn(const cp_attn_desc& d, int32_t layout, int32_t rank_begin, int32_t rank_end,
                           int32_t step_begin, int32_t step_end, const void* q, const void* k, const void* v,
                           float* o, float* m, float* l, int32_t mode, cudaStream_t stream, int32_t chunks,
                           bool allow_split) {
  RingParams p;
  memset(&p, 0, sizeof(p));
  if (!encode_map(&p.tmap_q, q, d.b, d.S, d.h_q, d.d) || !encode_map(&p.tmap_k, k, d.b, d.S, d.h_kv, d.d) ||
      !encode_map(&p.tmap_v, v, d.b, d.S, d.h_kv, d.d) || !encode_map_o(&p.tmap_o, o, d.b, d.S, d.h_q, d.d))
    return CP_ERR_CUDA;
  p.o = o;
  p.m = m;
  p.l = l;
  p.b = d.b;
  p.S = d.S;
  p.h_q = d.h_q;
  p.h_kv = d.h_kv;
  p.cp = int32_t(d.cp);
  p.C = int32_t(d.S / (2 * d.cp));
  p.tpc = (p.C + BM - 1) / BM;
  p.group = int32_t(d.h_q / d.h_kv);
  // Two query tiles share each K/V tile in a CTA: two heads of a kv group (even groups),
  // or two consecutive row tiles of one head (odd groups, unless a chunk is one tile).
  bool row_pairs = p.group % 2 == 1 && (p.group == 1 || p.tpc > 1);
  // With one query head per kv head, a launch whose single tiles fit in one wave runs one
  // tile per CTA (the head-pair form, which finds no second head): pairing would halve its
  // CTAs and lengthen each CTA's chain (a tiny prefill: 15.5 against 19.4 us).
  // The CP_KNOB_RING_PAIRING setting overrides the choice; the results are the same bits.
  if (p.group == 1) {
    const int64_t n_single =
        int64_t(chunks == kRingBothChunks ? 2 : 1) * (rank_end - rank_begin) * p.tpc * d.b * d.h_q;
    const int32_t forced = kernel_choice(CP_KNOB_RING_PAIRING);
    int sms = 0;
    if (forced < 0 && current_sm_count(&sms) != cudaSuccess) return CP_ERR_CUDA;
    if (forced == 0 || (forced < 0 && n_single <= int64_t(sms))) row_pairs = false;
  }
  p.row_pairs = row_pairs ? 1 : 0;
  p.ipc = p.row_pairs ? (p.tpc + 1) / 2 : p.tpc;
  p.ppg = p.row_pairs ? p.group : (p.group + 1) / 2;
  p.n_pairs = int32_t(d.h_kv) * p.ppg;
  p.step_begin = step_begin;
  p.step_end = step_end;
  p.mode = mode;
  p.rank_begin = rank_begin;
  p.rank_end = rank_end;
  p.chunks = chunks;
  p.sl = d.scale * kLog2e;
  {
    // The fewest groups of equal size whose K/V stays under the budget (at least one
    // unit each): a group's K/V then stays in L2 while its CTAs run, next to the Q and O
    // streams.  40 MB measured best (0.40 GB of DRAM reads per GQA launch, 0.56 GB at
    // 70 MB, 1.68 GB ungrouped).
    // One ring step needs no grouping: the CTAs that share a K/V block lie within about
    // two waves of each other in the plain order (grouping measured 1 % slower there).
    const int64_t units = d.b * d.h_kv;
    const int64_t unit_bytes = d.S * d.d * 2 * 2;
    const int64_t budget = kL2UnitBudget;
    int64_t groups = 1;
    while (step_end - step_begin > 1 && groups < units && (units / groups) * unit_bytes > budget) {
      int64_t next = groups + 1;
      while (units % next != 0) ++next;
      groups = next;
    }
    p.unit_groups = int32_t(groups);
  }
  const int64_t n_items =
      int64_t(chunks == kRingBothChunks ? 2 : 1) * (rank_end - rank_begin) * p.ipc * d.b * p.n_pairs;
  if (n_items > 0x7fffffffLL) return CP_ERR_UNSUPPORTED;
  // Single query tiles that fill at most half the GPU: each item's key walk is split over
  // a cluster of 2, 4 or 8 CTAs (the most that still fit in one wave), which shortens the
  // chain of K/V tiles each CTA runs.  CP_KNOB_RING_KV_SPLIT = 0 turns this off.
  p.kv_split = 1;
  if (allow_split && layout == CP_LAYOUT_BALANCED && !p.row_pairs && p.group == 1 &&
      kernel_choice(CP_KNOB_RING_KV_SPLIT) != 0) {
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess) return CP_ERR_CUDA;
    while (p.kv_split < 8 && n_items * p.kv_split * 2 <= int64_t(sms)) p.kv_split *= 2;
  }
  if (layout == CP_LAYOUT_SEQUENTIAL)
    return d.d == 128 ? launch_d<128, CP_LAYOUT_SEQUENTIAL>(p, n_items, stream)
                      : launch_d<64, CP_LAYOUT_SEQUENTIAL>(p, n_items, stream);
  return d.d == 128 ? launch_d<128, CP_LAYOUT_BALANCED>(p, n_items, stream)
                    : launch_d<64, CP_LAYOUT_BALANCED>(p, n_items, stream);
}

cudaError_t ring_wait_timeout_selftest(cudaStream_t stream) {
  ring_wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t ring_take_status(int32_t* status) {
  int32_t s = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&s, g_ring_status, sizeof(s));
  if (e != cudaSuccess) return e;
  const int32_t zero = 0;
  e = cudaMemcpyToSymbol(g_ring_status, &zero, sizeof(zero));
  *status = s;
  return e;
}

}  // namespace cpattn
