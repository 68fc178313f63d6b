// LSE merge of partial attention triples (the "three-quantity reduce").
//
// "G5 上下文并行建模设计规格", Terms table, row "Partial attention": the triple
// (max / numerator / denominator) of disjoint key sets merges associatively and
// in any order.  For parts p taken in the caller's order:
//   m = max_p m_p,  l = sum_p e^{m_p - m} l_p,  O = sum_p e^{m_p - m} O_p.
// Taking m first (exact, order-free) and then summing the weighted parts is the
// same quantity as a left fold of pairwise merges; only rounding differs.
//
// HBM-bound: each (batch, head, row) reads n_parts x (d + 2) floats and writes
// d + 2.  One CTA covers kRowsPerCta consecutive rows of one (batch, head): it first
// stages the 2 x n_parts x kRowsPerCta scalars (m, l) with coalesced loads into shared
// memory, then each warp streams the O rows of its rows part by part, lanes
// owning float4 slices of d, with eight (d <= 128) down to two (d = 512) parts of loads
// in flight per lane.  For d = 128 and up to 64 parts, one thread per CTA instead
// streams every part's block of O rows into a ring of shared-memory slots with TMA, and
// the warps fold the same parts in the same order (the same bits).

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"
#include "tc_ptx.h"

namespace cpattn {
namespace {

constexpr int kRowsPerCta = 16;  // 0.680 ms on the merge-stress workload against 0.684 at 32
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

template <int NCH>  // float4 slices of d owned by one lane (d <= 128 * NCH)
__global__ void __launch_bounds__(kThreads, NCH == 1 ? 5 : 1) lse_merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int kUnroll = (8 / NCH) < 2 ? 2 : (8 / NCH);  // parts in flight per lane
  extern __shared__ float smem[];
  const int n_parts = p.n_parts;
  float* sm_m = smem;                          // [n_parts][kRowsPerCta] in fold order
  float* sm_l = smem + n_parts * kRowsPerCta;  // [n_parts][kRowsPerCta]

  const int64_t row_blocks = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t tile = blockIdx.x;
  const int64_t rb = tile % row_blocks;
  const int64_t bh = tile / row_blocks;  // batch * heads + head
  const int64_t h = bh % p.heads;
  const int64_t bi = bh / p.heads;
  const int64_t row0 = rb * kRowsPerCta;

  // Stage m and l of every part for the CTA's rows (consecutive threads -> consecutive rows).
  for (int idx = threadIdx.x; idx < n_parts * kRowsPerCta; idx += kThreads) {
    const int kpos = idx / kRowsPerCta;
    const int r = idx % kRowsPerCta;
    const int part = p.order[kpos];
    const int64_t row = row0 + r;
    float mv = -INFINITY, lv = 0.f;
    if (row < p.rows) {
      const int64_t off = ((int64_t(part) * p.batch + bi) * p.heads + h) * p.rows + row;
      mv = p.m_parts[off];
      lv = p.l_parts[off];
    }
    sm_m[idx] = mv;
    sm_l[idx] = lv;
  }
  __syncthreads();

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int64_t n_vec = p.d / 4;
  const int64_t part_stride = p.batch * p.rows * p.heads * p.d;  // floats between parts of O

  for (int r = warp; r < kRowsPerCta; r += kWarps) {
    const int64_t row = row0 + r;
    if (row >= p.rows) break;
    // m = max over parts (exact in any order).
    float mx = -INFINITY;
    for (int kpos = lane; kpos < n_parts; kpos += 32) mx = fmaxf(mx, sm_m[kpos * kRowsPerCta + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // All parts the identity: the row stays the identity (never NaN).
    const float shift = (mx == -INFINITY) ? 0.f : mx;

    float lsum = 0.f;
    float4 acc[NCH];
#pragma unroll
    for (int c = 0; c < NCH; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t obase = ((bi * p.rows + row) * p.heads + h) * p.d;

    for (int k0 = 0; k0 < n_parts; k0 += kUnroll) {
      float4 x[kUnroll][NCH];
      float w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int kpos = k0 + u;
        const bool ok = kpos < n_parts;
        const int part = ok ? p.order[kpos] : 0;
        w[u] = ok ? expf(sm_m[kpos * kRowsPerCta + r] - shift) : 0.f;
        const float4* src = reinterpret_cast<const float4*>(p.o_parts + int64_t(part) * part_stride + obase);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int64_t vi = lane + 32 * c;
          x[u][c] = (ok && vi < n_vec) ? ld_stream(src + vi) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int kpos = k0 + u;
        if (kpos < n_parts) lsum = fmaf(w[u], sm_l[kpos * kRowsPerCta + r], lsum);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          acc[c].x = fmaf(w[u], x[u][c].x, acc[c].x);
          acc[c].y = fmaf(w[u], x[u][c].y, acc[c].y);
          acc[c].z = fmaf(w[u], x[u][c].z, acc[c].z);
          acc[c].w = fmaf(w[u], x[u][c].w, acc[c].w);
        }
      }
    }
    const float inv = (p.finalize && lsum > 0.f) ? 1.f / lsum : 1.f;
    const bool zero = p.finalize && !(lsum > 0.f);
    float4* dst = reinterpret_cast<float4*>(p.o_out + obase);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int64_t vi = lane + 32 * c;
      if (vi < n_vec) {
        float4 y = acc[c];
        if (zero) {
          y = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (p.finalize) {
          y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
        }
        dst[vi] = y;
      }
    }
    if (lane == 0) {
      const int64_t off = (bi * p.heads + h) * p.rows + row;
      if (p.m_out) p.m_out[off] = mx;
      if (p.l_out) p.l_out[off] = lsum;
    }
  }
}

// d = 128, up to 64 parts: the same fold fed by TMA.  The kernel above keeps at
// most eight parts of loads in flight per warp and drains between batches (82 % of
// DRAM peak on the merge stress).  Here one thread streams each part's block of
// kRowsPerCta x 128 O values into a ring of shared-memory slots, kTmaSlots parts
// ahead of the slowest warp; each warp folds two rows from shared memory with the
// same arithmetic in the same order, so the result is the same bits.
constexpr int kTmaD = 128;
constexpr int kTmaSlots = 6;  // 4 CTAs per SM; 4 slots (5 CTAs) measured the same, 12 (2 CTAs) 10 % slower
constexpr uint32_t kTmaSlotBytes = kRowsPerCta * kTmaD * 4;  // 8 KB
constexpr int kTmaMaxParts = 64;  // m and l staging stays at most 8 KB (58 KB of shared memory a CTA)
constexpr int kTmaRowsPerWarp = kRowsPerCta / kWarps;

__device__ int32_t g_merge_status = 0;

struct MergeTmaParams {
  CUtensorMap map_o;  // o_parts as fp32 (d, heads, rows, n_parts * batch), box (128, 1, kRowsPerCta, 1)
  MergeParams p;
};

size_t merge_tma_smem_bytes(int32_t n_parts) {
  return 1024 + size_t(kTmaSlots) * kTmaSlotBytes + size_t(2) * n_parts * kRowsPerCta * 4 +
         size_t(2) * kTmaSlots * 8 + 16;
}

__global__ void __launch_bounds__(kThreads, 4) lse_merge_tma_kernel(const __grid_constant__ MergeTmaParams tp) {
  using namespace tc;
  const MergeParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_parts = p.n_parts;
  const uint32_t ring = smem_u32(base);
  float* sm_m = reinterpret_cast<float*>(base + kTmaSlots * kTmaSlotBytes);  // [n_parts][kRowsPerCta]
  float* sm_l = sm_m + n_parts * kRowsPerCta;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm_l + n_parts * kRowsPerCta);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(bars + 2 * kTmaSlots);
  auto full = [&](int sl) { return smem_u32(&bars[sl]); };
  auto empty = [&](int sl) { return smem_u32(&bars[kTmaSlots + sl]); };

  const int64_t row_blocks = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t tile = blockIdx.x;
  const int64_t rb = tile % row_blocks;
  const int64_t bh = tile / row_blocks;
  const int64_t h = bh % p.heads;
  const int64_t bi = bh / p.heads;
  const int64_t row0 = rb * kRowsPerCta;

  // Part kpos (fold order) into slot kpos % kTmaSlots.
  auto issue = [&](int kpos) {
    const int sl = kpos % kTmaSlots;
    mbar_expect_tx(full(sl), kTmaSlotBytes);
    tma_load_4d(ring + sl * kTmaSlotBytes, &tp.map_o, full(sl), 0, int32_t(h), int32_t(row0),
                int32_t(int64_t(p.order[kpos]) * p.batch + bi));
  };
  // The first parts stream in while the m and l scalars are staged.
  int issued = 0;  // copies issued (thread 0 only)
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < kTmaSlots; ++sl) {
      mbar_init(full(sl), 1);
      mbar_init(empty(sl), kWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int kpos = 0; kpos < n_parts && kpos < kTmaSlots; ++kpos) issue(kpos);
    issued = n_parts < kTmaSlots ? n_parts : kTmaSlots;
  }
  for (int idx = threadIdx.x; idx < n_parts * kRowsPerCta; idx += kThreads) {
    const int kpos = idx / kRowsPerCta;
    const int r = idx % kRowsPerCta;
    const int part = p.order[kpos];
    const int64_t row = row0 + r;
    float mv = -INFINITY, lv = 0.f;
    if (row < p.rows) {
      const int64_t off = ((int64_t(part) * p.batch + bi) * p.heads + h) * p.rows + row;
      mv = p.m_parts[off];
      lv = p.l_parts[off];
    }
    sm_m[idx] = mv;
    sm_l[idx] = lv;
  }
  __syncthreads();

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  float shift[kTmaRowsPerWarp], mxr[kTmaRowsPerWarp], lsum[kTmaRowsPerWarp];
  float4 acc[kTmaRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kTmaRowsPerWarp; ++rr) {
    const int r = warp * kTmaRowsPerWarp + rr;
    float mx = -INFINITY;
    for (int kpos = lane; kpos < n_parts; kpos += 32) mx = fmaxf(mx, sm_m[kpos * kRowsPerCta + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    mxr[rr] = mx;
    shift[rr] = (mx == -INFINITY) ? 0.f : mx;
    lsum[rr] = 0.f;
    acc[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  bool ok = true;
  for (int kpos = 0; kpos < n_parts; ++kpos) {
    const int sl = kpos % kTmaSlots;
    const uint32_t ph = uint32_t((kpos / kTmaSlots) & 1);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(full(sl), ph, abort_flag, &g_merge_status))) {
      ok = false;
      break;
    }
#pragma unroll
    for (int rr = 0; rr < kTmaRowsPerWarp; ++rr) {
      const int r = warp * kTmaRowsPerWarp + rr;
      const float w = expf(sm_m[kpos * kRowsPerCta + r] - shift[rr]);
      lsum[rr] = fmaf(w, sm_l[kpos * kRowsPerCta + r], lsum[rr]);
      const float4 x = ld_shared_v4(ring + sl * kTmaSlotBytes + uint32_t((r * kTmaD + lane * 4) * 4));
      acc[rr].x = fmaf(w, x.x, acc[rr].x);
      acc[rr].y = fmaf(w, x.y, acc[rr].y);
      acc[rr].z = fmaf(w, x.z, acc[rr].z);
      acc[rr].w = fmaf(w, x.w, acc[rr].w);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(sl));
    // The slot is refilled once every warp has read it.
    if (threadIdx.x == 0 && kpos + kTmaSlots < n_parts) {
      if (!mbar_wait_bounded(empty(sl), ph, abort_flag, &g_merge_status)) {
        ok = false;
      } else {
        issue(kpos + kTmaSlots);
        ++issued;
      }
    }
    if (!__all_sync(0xffffffffu, ok)) break;
  }
  if (!ok || *abort_flag) {
    // Thread 0 issued every copy: before it leaves, it waits for the last copy issued
    // into each slot to land (its full barrier's phase to complete), which keeps the
    // CTA's shared memory allocated meanwhile; the other threads leave at once.  The
    // wait is bounded (10 ms for all slots): a copy later than that is not waited for.
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer();
      for (int kpos = issued > kTmaSlots ? issued - kTmaSlots : 0; kpos < issued; ++kpos) {
        const uint32_t bar = full(kpos % kTmaSlots);
        const uint32_t ph = uint32_t((kpos / kTmaSlots) & 1);
        while (!mbar_try_wait(bar, ph) && globaltimer() - t0 < 10000000ull) {
        }
      }
    }
    return;
  }
#pragma unroll
  for (int rr = 0; rr < kTmaRowsPerWarp; ++rr) {
    const int r = warp * kTmaRowsPerWarp + rr;
    const int64_t row = row0 + r;
    if (row >= p.rows) break;
    const float ls = lsum[rr];
    const float inv = (p.finalize && ls > 0.f) ? 1.f / ls : 1.f;
    const bool zero = p.finalize && !(ls > 0.f);
    float4 y = acc[rr];
    if (zero) {
      y = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (p.finalize) {
      y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
    }
    reinterpret_cast<float4*>(p.o_out + ((bi * p.rows + row) * p.heads + h) * kTmaD)[lane] = y;
    if (lane == 0) {
      const int64_t off = (bi * p.heads + h) * p.rows + row;
      if (p.m_out) p.m_out[off] = mxr[rr];
      if (p.l_out) p.l_out[off] = ls;
    }
  }
}

bool merge_tma_enabled() { return kernel_choice(CP_KNOB_MERGE_KERNEL) != 0; }

// rows == 1 (the decode reduce: one triple per sequence and head).  One CTA per
// (batch, head, slice of 128 columns), so the grid has batch * heads * ceil(d/128)
// CTAs.  The part weights e^{m_p - m} are computed once into shared memory.  Each
// of the four warps then folds a contiguous quarter of the parts, in the caller's
// order, into one float4 column per lane with eight loads in flight; the quarters
// are added in order.
constexpr int kR1Threads = 128;
constexpr int kR1Warps = kR1Threads / 32;
constexpr int kR1SliceVec = 32;  // float4 columns per CTA: 128 floats

__global__ void __launch_bounds__(kR1Threads) lse_merge_rows1_kernel(const __grid_constant__ MergeParams p) {
  __shared__ float w[CP_MAX_MERGE_PARTS];  // weights in fold order
  __shared__ float red[kR1Warps];          // partial maxima / sums
  __shared__ float4 part_sum[kR1Warps][kR1SliceVec];
  const int n = p.n_parts;
  const int64_t bh = blockIdx.x;
  const int64_t h = bh % p.heads, bi = bh / p.heads;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  auto ml_off = [&](int part) { return (int64_t(part) * p.batch + bi) * p.heads + h; };  // rows == 1

  float mx = -INFINITY;
  for (int k = threadIdx.x; k < n; k += kR1Threads) {
    const float m = p.m_parts[ml_off(p.order[k])];
    w[k] = m;
    mx = fmaxf(mx, m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int i = 1; i < kR1Warps; ++i) mx = fmaxf(mx, red[i]);
  const float shift = (mx == -INFINITY) ? 0.f : mx;  // all parts the identity: stays the identity
  __syncthreads();
  float ls = 0.f;
  for (int k = threadIdx.x; k < n; k += kR1Threads) {
    const float wk = expf(w[k] - shift);
    w[k] = wk;
    ls = fmaf(wk, p.l_parts[ml_off(p.order[k])], ls);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
  if (lane == 0) red[warp] = ls;
  __syncthreads();
  float lsum = 0.f;
#pragma unroll
  for (int i = 0; i < kR1Warps; ++i) lsum += red[i];

  const int64_t n_vec = p.d / 4;
  const int64_t c = int64_t(blockIdx.y) * kR1SliceVec + lane;  // this lane's float4 column
  const bool col_ok = c < n_vec;
  const int64_t part_stride = p.batch * p.heads * p.d;  // rows == 1
  const int64_t obase = (bi * p.heads + h) * p.d;
  const int k_begin = int(int64_t(n) * warp / kR1Warps);
  const int k_end = int(int64_t(n) * (warp + 1) / kR1Warps);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col_ok) {
    int k = k_begin;
    for (; k + 8 <= k_end; k += 8) {
      float4 x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        x[u] = ld_stream(reinterpret_cast<const float4*>(p.o_parts + int64_t(p.order[k + u]) * part_stride + obase) + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float wk = w[k + u];
        acc.x = fmaf(wk, x[u].x, acc.x);
        acc.y = fmaf(wk, x[u].y, acc.y);
        acc.z = fmaf(wk, x[u].z, acc.z);
        acc.w = fmaf(wk, x[u].w, acc.w);
      }
    }
    for (; k < k_end; ++k) {
      const float4 x = ld_stream(reinterpret_cast<const float4*>(p.o_parts + int64_t(p.order[k]) * part_stride + obase) + c);
      const float wk = w[k];
      acc.x = fmaf(wk, x.x, acc.x);
      acc.y = fmaf(wk, x.y, acc.y);
      acc.z = fmaf(wk, x.z, acc.z);
      acc.w = fmaf(wk, x.w, acc.w);
    }
  }
  part_sum[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && col_ok) {
    float4 o = part_sum[0][lane];
#pragma unroll
    for (int i = 1; i < kR1Warps; ++i) {
      const float4 q = part_sum[i][lane];
      o.x += q.x;
      o.y += q.y;
      o.z += q.z;
      o.w += q.w;
    }
    if (p.finalize) {
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;  // no visible key at all: output 0
      o.x *= inv;
      o.y *= inv;
      o.z *= inv;
      o.w *= inv;
    }
    reinterpret_cast<float4*>(p.o_out + obase)[c] = o;
  }
  if (threadIdx.x == 0 && blockIdx.y == 0) {
    if (p.m_out) p.m_out[bi * p.heads + h] = mx;
    if (p.l_out) p.l_out[bi * p.heads + h] = lsum;
  }
}

// Tree merge (the halving tree: at each level part i merges with part i + n/2), in
// one pass.  That tree equals a pairwise tree over the parts taken in bit-reversed
// index order, so each lane streams its float4 column through a stack of partial
// results (one per level), merging whenever two of a level meet.  Every node does
// what the two-part merge does: m = max of the children; weights e^{m_child - m}
// (shift 0 when both are -inf); l = fmaf(w_r, l_r, w_l * l_l); O = fmaf(w_r, O_r,
// w_l * O_l); the root is finalised like the flat merge.  The node weights of a
// CTA's rows are computed first into shared memory, one warp per row.
constexpr int kTreeThreads = 256;
constexpr int kTreeWarps = kTreeThreads / 32;
// Leaves whose O rows a CTA prefetches to L2 before its node-weight phase.  32-part stress
// merge: 0.686 ms with none, 0.679 / 0.670 / 0.661 / 0.796 ms with 4 / 8 / 16 / 32 (all of them).
constexpr int kTreePrefetchLeaves = 16;
constexpr int kTreeGroupLg = 5;  // trees above 32 leaves run as a loop over 32-leaf subtrees
constexpr int kRing = 8;         // parts of loads in flight per lane in that loop

__device__ __forceinline__ int bit_reverse(int k, int lg) { return int(__brev(uint32_t(k)) >> (32 - lg)); }

template <int LG>  // n_parts = 2^LG; the part loop below unrolls completely
__global__ void __launch_bounds__(kTreeThreads, 3) lse_merge_tree_kernel(const __grid_constant__ MergeParams p,
                                                                        int rows_per_cta) {
  extern __shared__ float smem[];
  constexpr int lg = LG;
  constexpr int n = 1 << LG;
  const int nodes = n - 1;
  float* wl = smem;                            // [rows_per_cta][nodes] left-child weights
  float* wr = wl + rows_per_cta * nodes;       // [rows_per_cta][nodes] right-child weights
  float* mroot = wr + rows_per_cta * nodes;    // [rows_per_cta]
  float* lroot = mroot + rows_per_cta;         // [rows_per_cta]
  float* scratch = lroot + rows_per_cta;       // [warps][2][n] one level's (m, l) per warp

  const int64_t row_blocks = (p.rows + rows_per_cta - 1) / rows_per_cta;
  const int64_t tile = blockIdx.x;
  const int64_t rb = tile % row_blocks;
  const int64_t bh = tile / row_blocks;
  const int64_t h = bh % p.heads;
  const int64_t bi = bh / p.heads;
  const int64_t row0 = rb * rows_per_cta;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float* sm = scratch + warp * 2 * n;
  float* sl = sm + n;

  // The first leaves' O rows of this CTA go to L2 while the node weights below are
  // computed: one bulk prefetch per (leaf, row) of d floats, no registers held.
  {
    const int64_t pstride = p.batch * p.rows * p.heads * p.d;
    const int nr = int(min(int64_t(rows_per_cta), p.rows - row0));
    const int total = (kTreePrefetchLeaves < n ? kTreePrefetchLeaves : n) * nr;
    for (int t = threadIdx.x; t < total; t += kTreeThreads) {
      const int k = t / nr, r = t - (t / nr) * nr;
      const float* src = p.o_parts + int64_t(bit_reverse(k, lg)) * pstride + ((bi * p.rows + row0 + r) * p.heads + h) * p.d;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(uint32_t(p.d * 4)) : "memory");
    }
  }

  // Node weights, level by level; node (level L >= 1, index i) is stored at
  // (n - (n >> (L - 1))) + i, so level 1 comes first and the root last.
  for (int r = warp; r < rows_per_cta; r += kTreeWarps) {
    const int64_t row = row0 + r;
    if (row >= p.rows) break;
    for (int k = lane; k < n; k += 32) {  // leaves in bit-reversed order
      const int part = bit_reverse(k, lg);
      const int64_t off = ((int64_t(part) * p.batch + bi) * p.heads + h) * p.rows + row;
      sm[k] = p.m_parts[off];
      sl[k] = p.l_parts[off];
    }
    __syncwarp();
    int base = 0;
    for (int L = 1; L <= lg; ++L) {
      const int cnt = n >> L;
      float m_new[8], l_new[8];  // up to 256 leaves: at most 128 nodes, 4 per lane
      int c = 0;
      for (int i = lane; i < cnt; i += 32, ++c) {
        const float ma = sm[2 * i], mb = sm[2 * i + 1];
        const float mx = fmaxf(ma, mb);
        const float shift = (mx == -INFINITY) ? 0.f : mx;
        const float wa = expf(ma - shift), wb = expf(mb - shift);
        const float lsum = fmaf(wb, sl[2 * i + 1], fmaf(wa, sl[2 * i], 0.f));
        wl[r * nodes + base + i] = wa;
        wr[r * nodes + base + i] = wb;
        m_new[c] = mx;
        l_new[c] = lsum;
      }
      __syncwarp();
      c = 0;
      for (int i = lane; i < cnt; i += 32, ++c) {
        sm[i] = m_new[c];
        sl[i] = l_new[c];
      }
      __syncwarp();
      base += cnt;
    }
    if (lane == 0) {
      mroot[r] = sm[0];
      lroot[r] = sl[0];
    }
    __syncwarp();
  }
  __syncthreads();

  const int64_t n_vec = p.d / 4;
  const int64_t part_stride = p.batch * p.rows * p.heads * p.d;
  constexpr int kAhead = 14;  // parts of loads in flight per lane
  for (int r = warp; r < rows_per_cta; r += kTreeWarps) {
    const int64_t row = row0 + r;
    if (row >= p.rows) break;
    const int64_t obase = ((bi * p.rows + row) * p.heads + h) * p.d;
    const float* wlr = wl + r * nodes;
    const float* wrr = wr + r * nodes;
    for (int64_t vi = lane; vi < n_vec; vi += 32) {
      float4 y;
      // One tree node: cur = w_r * cur + w_l * left, weights from shared memory.
      auto node_merge = [&](float4& cur, const float4& left, int node) {
        const float a = wlr[node], b = wrr[node];
        cur.x = fmaf(b, cur.x, a * left.x);
        cur.y = fmaf(b, cur.y, a * left.y);
        cur.z = fmaf(b, cur.z, a * left.z);
        cur.w = fmaf(b, cur.w, a * left.w);
      };
      if constexpr (LG <= kTreeGroupLg) {
        // All n leaves unrolled: a stack of one partial per level.
        float4 stk[lg + 1];
        float4 x[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead && u < n; ++u)
          x[u] = ld_stream(reinterpret_cast<const float4*>(p.o_parts + int64_t(bit_reverse(u, lg)) * part_stride +
                                                           obase) + vi);
#pragma unroll
        for (int k = 0; k < n; ++k) {
          float4 cur = x[k % kAhead];
          if (k + kAhead < n)  // refill this slot with a later part
            x[k % kAhead] = ld_stream(reinterpret_cast<const float4*>(
                                          p.o_parts + int64_t(bit_reverse(k + kAhead, lg)) * part_stride + obase) + vi);
          // binary counter on k: merge with the level's left partial while bit `level` of k is set
          int base = 0;
#pragma unroll
          for (int level = 0; level < lg; ++level) {
            if (((k >> level) & 1) == 0) {
              stk[level] = cur;
              break;
            }
            node_merge(cur, stk[level], base + (k >> (level + 1)));
            base += n >> (level + 1);
            if (level == lg - 1) stk[lg] = cur;  // k = n - 1: the root
          }
        }
        y = stk[lg];
      } else {
        // Leaves in groups of 2^kTreeGroupLg: each group's subtree is unrolled as above,
        // the groups run in a loop, and the levels above a group keep their own stack.
        // The same nodes in the same order as the single unrolled tree.
        constexpr int G = kTreeGroupLg;
        constexpr int ng = 1 << G;
        constexpr int UP = LG - G;
        const float* col = p.o_parts + obase + 4 * vi;
        auto leaf = [&](int k) {
          return ld_stream(reinterpret_cast<const float4*>(col + int64_t(bit_reverse(k, lg)) * part_stride));
        };
        float4 up[UP];
        float4 x[kRing];  // kRing divides ng, so a leaf's slot is the same in every group
#pragma unroll
        for (int u = 0; u < kRing; ++u) x[u] = leaf(u);
#pragma unroll 1
        for (int g = 0; g < (1 << UP); ++g) {
          float4 stk[G];
          float4 cur;
#pragma unroll
          for (int k = 0; k < ng; ++k) {
            cur = x[k % kRing];
            const int next = g * ng + k + kRing;
            if (next < n) x[k % kRing] = leaf(next);
            int base = 0;
#pragma unroll
            for (int level = 0; level < G; ++level) {
              if (((k >> level) & 1) == 0) {
                stk[level] = cur;
                break;
              }
              node_merge(cur, stk[level], base + g * (ng >> (level + 1)) + (k >> (level + 1)));
              base += n >> (level + 1);
            }
          }
          // cur is group g's subtree root: carry it up the binary counter on g
          int base = n - (n >> G);
#pragma unroll
          for (int lv = 0; lv < UP; ++lv) {
            if (((g >> lv) & 1) == 0) {
              up[lv] = cur;
              break;
            }
            node_merge(cur, up[lv], base + (g >> (lv + 1)));
            base += n >> (G + lv + 1);
          }
          y = cur;  // the root after the last group
        }
      }
      const float lsum = lroot[r];
      if (p.finalize) {
        if (lsum > 0.f) {
          const float inv = 1.f / lsum;
          y.x *= inv; y.y *= inv; y.z *= inv; y.w *= inv;
        } else {
          y = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      reinterpret_cast<float4*>(p.o_out + obase)[vi] = y;
    }
    if (lane == 0) {
      const int64_t off = (bi * p.heads + h) * p.rows + row;
      if (p.m_out) p.m_out[off] = mroot[r];
      if (p.l_out) p.l_out[off] = lroot[r];
    }
  }
}

}  // namespace

cudaError_t launch_merge_tree(const MergeParams& p, cudaStream_t stream) {
  int lg = 0;
  while ((1 << lg) < p.n_parts) ++lg;
  if ((1 << lg) != p.n_parts || lg < 1 || lg > 8) return cudaErrorInvalidValue;
  // Rows per CTA, measured per size: 8 except 16 at 64 parts (32 parts: 0.701 ms at 8,
  // 0.704 at 16, 0.721 at 32; 64 parts: 0.723 at 16, 0.737 at 8).
  const int rows_per_cta = p.n_parts == 64 ? 16 : 8;
  const int64_t row_blocks = (p.rows + rows_per_cta - 1) / rows_per_cta;
  const int64_t ctas = p.batch * p.heads * row_blocks;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  const size_t smem = (size_t(rows_per_cta) * (2 * (p.n_parts - 1) + 2) + size_t(kTreeWarps) * 2 * p.n_parts) *
                      sizeof(float);
  switch (lg) {
#define CPATTN_TREE_CASE(L)                                                                                      \
  case L:                                                                                                        \
    if (smem > 48 * 1024) {                                                                                      \
      static SmemLimit lim;                                                                                      \
      if (raise_smem_limit(reinterpret_cast<const void*>(lse_merge_tree_kernel<L>), int(smem), &lim) !=          \
          cudaSuccess)                                                                                           \
        return cudaErrorInvalidValue;                                                                            \
    }                                                                                                            \
    lse_merge_tree_kernel<L><<<unsigned(ctas), kTreeThreads, smem, stream>>>(p, rows_per_cta);                   \
    break;
    CPATTN_TREE_CASE(1) CPATTN_TREE_CASE(2) CPATTN_TREE_CASE(3) CPATTN_TREE_CASE(4)
    CPATTN_TREE_CASE(5) CPATTN_TREE_CASE(6) CPATTN_TREE_CASE(7) CPATTN_TREE_CASE(8)
#undef CPATTN_TREE_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.rows == 1) {
    const int64_t ctas = p.batch * p.heads;
    const int64_t slices = (p.d / 4 + kR1SliceVec - 1) / kR1SliceVec;
    if (ctas > 0x7fffffffLL || slices > 65535) return cudaErrorInvalidValue;
    lse_merge_rows1_kernel<<<dim3(unsigned(ctas), unsigned(slices)), kR1Threads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  const int64_t row_blocks = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t tiles = row_blocks * p.batch * p.heads;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  // TMA coordinates are 32-bit and its strides below 2^40 bytes (rows * heads * 512 B).
  if (p.d == kTmaD && p.n_parts <= kTmaMaxParts && p.rows * p.heads < (int64_t(1) << 31) &&
      int64_t(p.n_parts) * p.batch < (int64_t(1) << 31) && enc != nullptr && merge_tma_enabled()) {
    MergeTmaParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.p = p;
    const cuuint64_t dims[4] = {cuuint64_t(kTmaD), cuuint64_t(p.heads), cuuint64_t(p.rows),
                                cuuint64_t(int64_t(p.n_parts) * p.batch)};
    const cuuint64_t strides[3] = {cuuint64_t(kTmaD * 4), cuuint64_t(p.heads * kTmaD * 4),
                                   cuuint64_t(p.rows * p.heads * kTmaD * 4)};
    const cuuint32_t box[4] = {kTmaD, 1, kRowsPerCta, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&tp.map_o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(p.o_parts), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const size_t tsmem = merge_tma_smem_bytes(p.n_parts);
    static SmemLimit lim_tma;
    const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(lse_merge_tma_kernel), int(tsmem), &lim_tma);
    if (e != cudaSuccess) return e;
    lse_merge_tma_kernel<<<unsigned(tiles), kThreads, tsmem, stream>>>(tp);
    return cudaGetLastError();
  }
  const size_t smem = size_t(2) * p.n_parts * kRowsPerCta * sizeof(float);
  const int nch = int((p.d / 4 + 31) / 32);
  cudaError_t e = cudaSuccess;
  switch (nch) {
#define CP_MERGE_CASE(N)                                                                       \
  case N: {                                                                                    \
    static SmemLimit lim;                                                                      \
    e = raise_smem_limit(reinterpret_cast<const void*>(lse_merge_kernel<N>), int(smem), &lim); \
    if (e != cudaSuccess) return e;                                                            \
  }                                                                                            \
    lse_merge_kernel<N><<<unsigned(tiles), kThreads, smem, stream>>>(p);                       \
    break;
    CP_MERGE_CASE(1)
    CP_MERGE_CASE(2)
    CP_MERGE_CASE(3)
    CP_MERGE_CASE(4)
#undef CP_MERGE_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t merge_take_status(int32_t* status) {
  int32_t s = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&s, g_merge_status, sizeof(s));
  if (e != cudaSuccess) return e;
  const int32_t zero = 0;
  e = cudaMemcpyToSymbol(g_merge_status, &zero, sizeof(zero));
  *status = s;
  return e;
}

}  // namespace cpattn
