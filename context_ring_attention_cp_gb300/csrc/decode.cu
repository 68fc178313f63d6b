// Pass-Q decode: one query per sequence against cp KV shards.
//
// "G5 上下文并行建模设计规格": Terms table row "Pass-Q" (the query goes to every
// rank, each rank computes partial attention on its local KV shard, then the
// partials are reduced), use-case decode paragraph (each rank scores its local
// shard), and the pass-Q paragraph of the Algorithm / formulas section (the
// reduce message is the partial output plus a max and a denominator per head).
//
// Shard s holds keys [s*L/cp, (s+1)*L/cp).  To stream K/V with the whole GPU,
// each shard is cut further into `splits` equal key ranges; every (range,
// sequence, kv head) is one CTA that writes one partial triple per query head of
// the group.  The reduce is the LSE merge kernel (merge.cu) over the cp*splits
// parts in shard order.
//
// The work is a streaming GEMV (about 1 FLOP per byte): HBM-bound.  A warp scores
// 32/LPK keys per iteration, LPK = d/16 lanes per key row (each lane holds 16
// elements: two 16-byte loads of K and two of V), with four iterations' loads in
// flight; dot products reduce across the LPK lanes with xor shuffles.  Softmax
// runs in base 2 on logits pre-scaled by scale*log2(e); m is stored in natural
// units.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace cpattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
  const uint16_t* q;  // [b, h_q, d] bf16
  const uint16_t* k;  // [b, L, h_kv, d] bf16
  const uint16_t* v;
  float* o_parts;  // [n_parts, b, h_q, d]
  float* m_parts;  // [n_parts, b, h_q]
  float* l_parts;
  int64_t b, L, h_q, h_kv;
  int64_t part_len;  // keys per part
  int32_t n_parts;
  float qscale;  // scale * log2(e)
};

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Merge (m2, l, o[16]) of the other lane group into this one; m2 in base-2 units.
__device__ __forceinline__ void merge_into(float& m, float& l, float* o, float m_o, float l_o,
                                           const float* o_o) {
  const float mn = fmaxf(m, m_o);
  const float sh = (mn == -INFINITY) ? 0.f : mn;
  const float a = exp2f(m - sh), c = exp2f(m_o - sh);
  l = a * l + c * l_o;
#pragma unroll
  for (int e = 0; e < 16; ++e) o[e] = a * o[e] + c * o_o[e];
  m = mn;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) passq_partial_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int LPK = D / 16;       // lanes per key row
  constexpr int KPW = 32 / LPK;     // keys per warp per iteration
  constexpr int NS = kWarps * KPW;  // key streams per CTA
  constexpr int U = (G == 1) ? 4 : (G == 2 ? 2 : 1);  // iterations of loads in flight

  __shared__ float sm_o[kWarps][G][D];
  __shared__ float sm_ml[kWarps][G][2];

  const int part = blockIdx.x;
  const int64_t bk = blockIdx.y;  // b * h_kv + kv head
  const int64_t kh = bk % p.h_kv;
  const int64_t bi = bk / p.h_kv;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int sub = lane / LPK;          // key slot of this lane group within the warp
  const int e0 = (lane % LPK) * 16;    // first element of the row held by this lane

  // Queries of the group, pre-scaled into base-2 logit units.
  float qr[G][16];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint16_t* qp = p.q + ((bi * p.h_q + kh * G + g) * D + e0);
    const uint4 a = *reinterpret_cast<const uint4*>(qp);
    const uint4 c = *reinterpret_cast<const uint4*>(qp + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qr[g][2 * i] = bf_lo(w[i]) * p.qscale;
      qr[g][2 * i + 1] = bf_hi(w[i]) * p.qscale;
    }
  }

  float m[G], l[G], o[G][16];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) o[g][e] = 0.f;
  }

  const int64_t k_begin = int64_t(part) * p.part_len;
  const int64_t k_end = k_begin + p.part_len;
  const int64_t row_stride = p.h_kv * D;  // elements between consecutive keys
  const uint16_t* kbase = p.k + (bi * p.L * p.h_kv + kh) * D + e0;
  const uint16_t* vbase = p.v + (bi * p.L * p.h_kv + kh) * D + e0;

  // The loop bound is warp-uniform (every lane takes part in the shuffles); lane
  // groups whose key falls past the range see -inf logits.
  for (int64_t wbase = k_begin + warp * KPW; wbase < k_end; wbase += int64_t(U) * NS) {
    uint4 kr[U][2], vr[U][2];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t key = wbase + sub + int64_t(u) * NS;
      ok[u] = key < k_end;
      if (ok[u]) {
        const uint16_t* kp = kbase + key * row_stride;
        const uint16_t* vp = vbase + key * row_stride;
        kr[u][0] = ld_stream_u4(kp);
        kr[u][1] = ld_stream_u4(kp + 8);
        vr[u][0] = ld_stream_u4(vp);
        vr[u][1] = ld_stream_u4(vp + 8);
      } else {
        kr[u][0] = kr[u][1] = vr[u][0] = vr[u][1] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float s[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t w[8] = {kr[u][0].x, kr[u][0].y, kr[u][0].z, kr[u][0].w,
                               kr[u][1].x, kr[u][1].y, kr[u][1].z, kr[u][1].w};
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = fmaf(qr[g][2 * i], bf_lo(w[i]), acc);
          acc = fmaf(qr[g][2 * i + 1], bf_hi(w[i]), acc);
        }
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        s[u] = ok[u] ? acc : -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u]);
      const float mn = fmaxf(m[g], mx);
      const float sh = (mn == -INFINITY) ? 0.f : mn;  // nothing seen yet: weights stay 0
      const float corr = exp2f(m[g] - sh);
      float pr[U];
      float ps = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        pr[u] = exp2f(s[u] - sh);
        ps += pr[u];
      }
      l[g] = fmaf(l[g], corr, ps);
      m[g] = mn;
#pragma unroll
      for (int e = 0; e < 16; ++e) o[g][e] *= corr;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t w[8] = {vr[u][0].x, vr[u][0].y, vr[u][0].z, vr[u][0].w,
                               vr[u][1].x, vr[u][1].y, vr[u][1].z, vr[u][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[g][2 * i] = fmaf(pr[u], bf_lo(w[i]), o[g][2 * i]);
          o[g][2 * i + 1] = fmaf(pr[u], bf_hi(w[i]), o[g][2 * i + 1]);
        }
      }
    }
  }

  // Merge the KPW lane groups of the warp (lanes with the same e0).
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
      float oo[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) oo[e] = __shfl_xor_sync(0xffffffffu, o[g][e], off);
      merge_into(m[g], l[g], o[g], mo, lo, oo);
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < 16; ++e) sm_o[warp][g][e0 + e] = o[g][e];
      if (lane == 0) {
        sm_ml[warp][g][0] = m[g];
        sm_ml[warp][g][1] = l[g];
      }
    }
  }
  __syncthreads();

  // Merge the warps: thread t handles element t of every query of the group.
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int g = idx / D, e = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, sm_ml[w][g][0]);
    const float sh = (mx == -INFINITY) ? 0.f : mx;
    float acc = 0.f, ls = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float a = exp2f(sm_ml[w][g][0] - sh);
      acc = fmaf(a, sm_o[w][g][e], acc);
      ls = fmaf(a, sm_ml[w][g][1], ls);
    }
    const int64_t row = (int64_t(part) * p.b + bi) * p.h_q + kh * G + g;
    p.o_parts[row * D + e] = acc;
    if (e == 0) {
      p.m_parts[row] = mx * kLn2;  // natural-log units
      p.l_parts[row] = ls;
    }
  }
}

}  // namespace

namespace {
// The streaming SIMT kernel of this file: small query groups.
bool simt_supported(const cp_attn_desc& d) {
  const int64_t g = d.h_q / d.h_kv;
  const bool dim_ok = d.d == 64 || d.d == 128 || d.d == 256 || d.d == 512;
  // Shared memory holds kWarps x g x d floats of per-warp partials: g * d <= 1024.
  return dim_ok && (g == 1 || g == 2 || g == 4) && g * d.d <= 1024;
}
}  // namespace

// g in {1, 2, 4}: the SIMT streaming kernel below; g in {16, 32} (heads sharing
// one K/V head): the tensor-core kernel of decode_mqa.cu.
bool decode_supported(const cp_attn_desc& d) { return simt_supported(d) || decode_mqa_supported(d); }

// Cut every shard into `splits` ranges so that about eight CTAs per SM are
// launched in total (a whole number of waves matters less than a short tail).
// `splits` divides the shard length; parts stay within CP_MAX_MERGE_PARTS.
int32_t decode_splits_per_shard(const cp_attn_desc& d, int sm_count) {
  if (!simt_supported(d)) return decode_mqa_splits(d, sm_count);
  const int64_t shard = d.S / d.cp;
  const int64_t groups = d.b * d.h_kv * d.cp;
  const int64_t target = int64_t(sm_count > 0 ? sm_count : 148) * 8;
  int64_t splits = 1;
  while (groups * splits < target && shard % (splits * 2) == 0 && shard / (splits * 2) >= 256 &&
         d.cp * splits * 2 <= CP_MAX_MERGE_PARTS)
    splits *= 2;
  return int32_t(splits);
}

namespace {
size_t pad4(size_t x) { return (x + 3) & ~size_t(3); }
}  // namespace

size_t decode_workspace_bytes(const cp_attn_desc& d, int32_t splits) {
  const size_t rows = size_t(d.cp) * size_t(splits) * size_t(d.b) * size_t(d.h_q);
  return (pad4(rows * size_t(d.d)) + 2 * pad4(rows)) * sizeof(float);
}

void decode_workspace_sections(const cp_attn_desc& d, int32_t splits, float* ws, float** o_parts,
                               float** m_parts, float** l_parts) {
  const size_t rows = size_t(d.cp) * size_t(splits) * size_t(d.b) * size_t(d.h_q);
  *o_parts = ws;
  *m_parts = ws + pad4(rows * size_t(d.d));
  *l_parts = *m_parts + pad4(rows);
}

cudaError_t launch_decode_partials(const cp_attn_desc& d, int32_t splits, const void* q,
                                   const void* k, const void* v, float* o_parts,
                                   float* m_parts, float* l_parts, cudaStream_t stream) {
  if (!simt_supported(d)) return launch_decode_mqa(d, splits, q, k, v, o_parts, m_parts, l_parts, stream);
  DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.b = d.b;
  p.L = d.S;
  p.h_q = d.h_q;
  p.h_kv = d.h_kv;
  p.n_parts = int32_t(d.cp * splits);
  p.part_len = d.S / p.n_parts;
  p.qscale = d.scale * kLog2e;
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  const int64_t gy = d.b * d.h_kv;
  if (gy > 65535) return cudaErrorInvalidValue;
  dim3 grid(unsigned(p.n_parts), unsigned(gy));
  const int g = int(d.h_q / d.h_kv);
#define CP_DEC(DD, GG)                                                     \
  if (d.d == DD && g == GG) {                                              \
    passq_partial_kernel<DD, GG><<<grid, kThreads, 0, stream>>>(p);        \
    return cudaGetLastError();                                             \
  }
  CP_DEC(64, 1) CP_DEC(64, 2) CP_DEC(64, 4)
  CP_DEC(128, 1) CP_DEC(128, 2) CP_DEC(128, 4)
  CP_DEC(256, 1) CP_DEC(256, 2) CP_DEC(256, 4)
  CP_DEC(512, 1) CP_DEC(512, 2)
#undef CP_DEC
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Fixed scratch for cp_passq_decode_noalloc
// ---------------------------------------------------------------------------
//
// Some callers cannot allocate device memory at the point where they decode:
// a plug-in whose host runtime owns all of HBM and hands it only the input and
// output buffers, or a latency-bound token loop that must not call cudaMalloc
// (which may synchronise the device).  For them the decode partials live in this
// array instead of a caller workspace.  It is part of the module image, so every
// GPU that loads the library holds its 8 MiB until the process exits.
// All calls share it and it keeps the last call's contents; nothing in it needs
// to start at zero (every partial is written before the reduce reads it), and
// calls that overlap on the GPU race on it.

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(2) << 20;  // 8 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // the context the address belongs to
  float* ptr;
};
ScratchAddr g_noalloc_addr[kMaxDevices] = {};

}  // namespace

size_t decode_noalloc_scratch_bytes() { return kNoAllocScratchFloats * sizeof(float); }

// The array's name in host code is only a host-side stand-in; its device address is
// looked up with the device current, once per device and context: the first call on
// a device does it, and so does the first call after a device reset.
cudaError_t decode_noalloc_scratch(float** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // Makes the device's primary context current (and creates it if a reset destroyed
  // it), so that the id read below is the context the kernels will run in.
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_context_id();
  ScratchAddr& a = g_noalloc_addr[dev];
  if (a.ptr == nullptr || ctx == 0 || ctx != a.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    a.ptr = static_cast<float*>(p);
    a.ctx_id = ctx;
  }
  *ptr = a.ptr;
  return cudaSuccess;
}

}  // namespace cpattn
