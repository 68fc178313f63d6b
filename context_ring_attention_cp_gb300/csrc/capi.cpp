// C-ABI entry points: argument validation, the host-side chunk planner and the
// closed-form byte counts.  Kernels are launched through internal.h only after
// every check here has passed; an invalid request launches nothing.
//
// Source of the operations: "G5 上下文并行建模设计规格" (G5 CP modelling spec) —
// Terms table (名词定义), Algorithm / formulas (算法 / 公式), Constraints
// (约束与规则: no silent fallback), Appendix C (cp is an explicit positive integer).

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"

using namespace cpattn;

cudaError_t cpattn::current_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

// Id of the calling thread's current context, 0 when it cannot be read.  A device
// reset destroys the current context; the next one has a new id.
unsigned long long cpattn::current_context_id() {
  struct Fns {
    PFN_cuCtxGetCurrent_v4000 get_current;
    PFN_cuCtxGetId_v12000 get_id;
  };
  static const Fns fns = []() {
    Fns f{nullptr, nullptr};
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return f;
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fns.get_current == nullptr || fns.get_id == nullptr || fns.get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || fns.get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

cudaError_t cpattn::raise_smem_limit(const void* func, int bytes, SmemLimit* lim) {
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(lim->mu);
  if (ctx != 0 && lim->ctx == ctx && lim->bytes >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  lim->ctx = ctx;  // the context's limit is now exactly `bytes`
  lim->bytes = bytes;
  return cudaSuccess;
}

namespace {
constexpr int kKnobs = 3;
std::atomic<int32_t> g_kernel_choice[kKnobs] = {{-1}, {-1}, {-1}};
}  // namespace

int32_t cpattn::kernel_choice(int32_t knob) {
  return (knob >= 0 && knob < kKnobs) ? g_kernel_choice[knob].load(std::memory_order_relaxed) : -1;
}

PFN_cuTensorMapEncodeTiled_v12000 cpattn::tensor_map_encoder() {
  // A function-local static is initialised once, even under concurrent first calls.
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) !=
            cudaSuccess ||
        qres != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

namespace {

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every element count a kernel indexes must fit int64 with room to spare.
bool product_fits(int64_t a, int64_t b, int64_t c, int64_t d) {
  int64_t x;
  return !__builtin_mul_overflow(a, b, &x) && !__builtin_mul_overflow(x, c, &x) &&
         !__builtin_mul_overflow(x, d, &x) && x < (int64_t(1) << 60);
}

cp_status check_desc_common(const cp_attn_desc* d) {
  if (d == nullptr) return CP_ERR_INVALID_ARGUMENT;
  if (d->b < 1 || d->S < 1 || d->h_q < 1 || d->h_kv < 1 || d->d < 1 || d->cp < 1)
    return CP_ERR_INVALID_ARGUMENT;
  if (d->cp > (1 << 20)) return CP_ERR_INVALID_ARGUMENT;
  if (d->h_q % d->h_kv != 0) return CP_ERR_INVALID_ARGUMENT;
  if (!(d->scale > 0.0f) || !isfinite(d->scale)) return CP_ERR_INVALID_ARGUMENT;
  if (!product_fits(d->b, d->S, d->h_q, d->d)) return CP_ERR_INVALID_ARGUMENT;
  return CP_OK;
}

cp_status check_decode_desc(const cp_attn_desc* d) {
  cp_status st = check_desc_common(d);
  if (st != CP_OK) return st;
  if (d->S % d->cp != 0) return CP_ERR_INVALID_ARGUMENT;
  if (d->causal != 0) return CP_ERR_UNSUPPORTED;
  if (!decode_supported(*d)) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

// ---------------------------------------------------------------------------
// Host-buffer ring: device workspace layout and the pipeline's streams
// ---------------------------------------------------------------------------

constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

struct HostRingLayout {
  size_t q, k, v, o, m, l;  // byte offsets into the workspace
  size_t total;
};

HostRingLayout host_ring_layout(const cp_attn_desc& d) {
  HostRingLayout w;
  const size_t qb = size_t(d.b) * d.S * d.h_q * d.d * 2;
  const size_t kb = size_t(d.b) * d.S * d.h_kv * d.d * 2;
  const size_t ob = size_t(d.b) * d.S * d.h_q * d.d * 4;
  const size_t mb = size_t(d.b) * d.h_q * d.S * 4;
  w.q = 0;
  w.k = w.q + round_up(qb);
  w.v = w.k + round_up(kb);
  w.o = w.v + round_up(kb);
  w.m = w.o + round_up(ob);
  w.l = w.m + round_up(mb);
  w.total = w.l + round_up(mb);
  return w;
}

cp_status check_host_ring(const cp_attn_desc* desc) {
  cp_status st = check_desc_common(desc);
  if (st != CP_OK) return st;
  if (desc->S % (2 * desc->cp) != 0) return CP_ERR_INVALID_ARGUMENT;
  if (desc->causal != 1) return CP_ERR_UNSUPPORTED;
  if (!ring_supported(*desc)) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

struct PipeStreams {
  cudaStream_t in, comp[2], out;
};

// Created on first use per device and kept for the life of the process.
bool pipe_streams(PipeStreams* out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static PipeStreams per_dev[kMaxDev];
  static bool made[kMaxDev] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!made[dev]) {
    PipeStreams s;
    cudaStream_t* all[4] = {&s.in, &s.comp[0], &s.comp[1], &s.out};
    for (int i = 0; i < 4; ++i) {
      if (cudaStreamCreateWithFlags(all[i], cudaStreamNonBlocking) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(*all[j]);
        return false;
      }
    }
    per_dev[dev] = s;
    made[dev] = true;
  }
  *out = per_dev[dev];
  return true;
}

// Merge of n_parts triples in index order (the caller may set another order).
MergeParams merge_params(int64_t batch, int64_t rows, int64_t heads, int64_t d, int32_t n_parts,
                         const float* o_parts, const float* m_parts, const float* l_parts, float* o_out,
                         float* m_out, float* l_out, bool finalize) {
  MergeParams p;
  memset(&p, 0, sizeof(p));
  p.batch = batch;
  p.rows = rows;
  p.heads = heads;
  p.d = d;
  p.n_parts = n_parts;
  p.finalize = finalize;
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  p.o_out = o_out;
  p.m_out = m_out;
  p.l_out = l_out;
  for (int32_t i = 0; i < n_parts; ++i) p.order[i] = static_cast<uint16_t>(i);
  return p;
}

// Pass-Q decode after the checks: the shard partials into the given sections, then the
// three-quantity reduce (the LSE merge over the parts in shard order, finalised).
cp_status run_passq_decode(const cp_attn_desc& desc, int32_t splits, const void* q, const void* k, const void* v,
                           float* sections, float* out, float* m_out, float* l_out, cudaStream_t s) {
  const int64_t n_parts = desc.cp * splits;
  if (n_parts > CP_MAX_MERGE_PARTS) return CP_ERR_UNSUPPORTED;
  float *o_parts = nullptr, *m_parts = nullptr, *l_parts = nullptr;
  decode_workspace_sections(desc, splits, sections, &o_parts, &m_parts, &l_parts);
  if (launch_decode_partials(desc, splits, q, k, v, o_parts, m_parts, l_parts, s) != cudaSuccess) return CP_ERR_CUDA;
  const MergeParams p =
      merge_params(desc.b, 1, desc.h_q, desc.d, int32_t(n_parts), o_parts, m_parts, l_parts, out, m_out, l_out, true);
  return launch_merge(p, s) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* cp_status_string(int32_t status) {
  switch (status) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARGUMENT: return "CP_ERR_INVALID_ARGUMENT";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_OVERFLOW: return "CP_ERR_OVERFLOW";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT";
    default: return "CP_ERR_UNKNOWN";
  }
}

cp_status cp_plan_chunks(int64_t S, int32_t cp, int32_t layout, int64_t* chunk_begin, int32_t* rank_chunks,
                         int32_t* step_src, int64_t* step_pairs) {
  if (cp < 1 || S < 1 || cp > (1 << 20)) return CP_ERR_INVALID_ARGUMENT;
  if (S % (2 * int64_t(cp)) != 0) return CP_ERR_INVALID_ARGUMENT;
  if (layout != CP_LAYOUT_BALANCED && layout != CP_LAYOUT_SEQUENTIAL) return CP_ERR_INVALID_ARGUMENT;
  if (!chunk_begin || !rank_chunks || !step_src || !step_pairs) return CP_ERR_INVALID_ARGUMENT;
  const int64_t C = S / (2 * int64_t(cp));
  const int64_t n = 2 * C;  // rows per rank
  int64_t pairs_off = 0, pairs_diag = 0, seq_full = 0, seq_tri = 0;
  if (__builtin_mul_overflow(2 * C, C, &pairs_off) || __builtin_add_overflow(pairs_off, C, &pairs_diag) ||
      __builtin_mul_overflow(n, n, &seq_full) || __builtin_mul_overflow(n, n + 1, &seq_tri))
    return CP_ERR_OVERFLOW;
  seq_tri /= 2;
  for (int64_t kk = 0; kk <= 2 * int64_t(cp); ++kk) chunk_begin[kk] = kk * C;
  for (int32_t r = 0; r < cp; ++r) {
    if (layout == CP_LAYOUT_BALANCED) {
      rank_chunks[2 * r] = r;                   // head chunk
      rank_chunks[2 * r + 1] = 2 * cp - 1 - r;  // tail chunk
    } else {
      rank_chunks[2 * r] = 2 * r;
      rank_chunks[2 * r + 1] = 2 * r + 1;
    }
    for (int32_t t = 0; t < cp; ++t) {
      const int32_t s = ((r - t) % cp + cp) % cp;
      step_src[int64_t(r) * cp + t] = s;
      if (layout == CP_LAYOUT_BALANCED)
        step_pairs[int64_t(r) * cp + t] = (t == 0) ? pairs_diag : pairs_off;
      else  // sequential: earlier source fully visible, own block causal, later source nothing
        step_pairs[int64_t(r) * cp + t] = (s < r) ? seq_full : (s == r ? seq_tri : 0);
    }
  }
  return CP_OK;
}

cp_status cp_plan_balanced_chunks(int64_t S, int32_t cp, int64_t* chunk_begin,
                                  int32_t* rank_chunks, int32_t* step_src,
                                  int64_t* step_pairs) {
  return cp_plan_chunks(S, cp, CP_LAYOUT_BALANCED, chunk_begin, rank_chunks, step_src, step_pairs);
}

cp_status cp_comm_bytes(const cp_comm_query* q, cp_comm_result* res) {
  if (q == nullptr || res == nullptr) return CP_ERR_INVALID_ARGUMENT;
  if (q->S < 0 || q->cp < 1 || q->c_kv < 0 || q->b < 0 || q->d < 0 || q->n_h < 0 || q->s_dtype < 0 ||
      q->layers_local < 0)
    return CP_ERR_INVALID_ARGUMENT;
  if (q->S % q->cp != 0) return CP_ERR_INVALID_ARGUMENT;
  uint64_t per_step, total, dispatch, width, reduce;
  const uint64_t tokens = uint64_t(q->S / q->cp);
  if (__builtin_mul_overflow(tokens, uint64_t(q->c_kv), &per_step)) return CP_ERR_OVERFLOW;
  if (__builtin_mul_overflow(uint64_t(q->cp - 1), per_step, &total)) return CP_ERR_OVERFLOW;
  if (__builtin_mul_overflow(uint64_t(q->b), uint64_t(q->d), &dispatch) ||
      __builtin_mul_overflow(dispatch, uint64_t(q->s_dtype), &dispatch))
    return CP_ERR_OVERFLOW;
  if (__builtin_mul_overflow(uint64_t(2), uint64_t(q->n_h), &width) ||
      __builtin_add_overflow(width, uint64_t(q->d), &width) ||
      __builtin_mul_overflow(uint64_t(q->b), width, &reduce) ||
      __builtin_mul_overflow(reduce, uint64_t(q->s_dtype), &reduce))
    return CP_ERR_OVERFLOW;
  uint64_t kv_rank;
  if (__builtin_mul_overflow(uint64_t(q->b), tokens, &kv_rank) ||
      __builtin_mul_overflow(kv_rank, uint64_t(q->c_kv), &kv_rank) ||
      __builtin_mul_overflow(kv_rank, uint64_t(q->layers_local), &kv_rank))
    return CP_ERR_OVERFLOW;
  res->passkv_total = total;
  res->passkv_per_step = per_step;
  res->passq_dispatch = dispatch;
  res->passq_reduce = reduce;
  res->kv_bytes_per_rank = kv_rank;
  return CP_OK;
}

cp_status cp_ring_rank_partial_attn(const cp_attn_desc* desc, int32_t layout, int32_t rank_begin,
                                    int32_t rank_end, int32_t step_begin, int32_t step_end, const void* q,
                                    const void* k, const void* v, float* o, float* m, float* l, int32_t mode,
                                    void* cuda_stream) {
  cp_status st = check_desc_common(desc);
  if (st != CP_OK) return st;
  if (desc->S % (2 * desc->cp) != 0) return CP_ERR_INVALID_ARGUMENT;
  if (layout != CP_LAYOUT_BALANCED && layout != CP_LAYOUT_SEQUENTIAL) return CP_ERR_INVALID_ARGUMENT;
  if (rank_begin < 0 || rank_end <= rank_begin || rank_end > desc->cp) return CP_ERR_INVALID_ARGUMENT;
  if (step_begin < 0 || step_end <= step_begin || step_end > desc->cp) return CP_ERR_INVALID_ARGUMENT;
  if ((mode & ~(CP_MODE_ACCUMULATE | CP_MODE_FINALIZE | CP_MODE_OVERLAP_PREVIOUS)) != 0)
    return CP_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(m) || !aligned16(l))
    return CP_ERR_INVALID_ARGUMENT;
  if (desc->causal != 1) return CP_ERR_UNSUPPORTED;
  if (!ring_supported(*desc)) return CP_ERR_UNSUPPORTED;
  return launch_ring_attn(*desc, layout, rank_begin, rank_end, step_begin, step_end, q, k, v, o, m, l, mode,
                          static_cast<cudaStream_t>(cuda_stream));
}

cp_status cp_ring_step_partial_attn(const cp_attn_desc* desc, int32_t step_begin,
                                    int32_t step_end, const void* q, const void* k,
                                    const void* v, float* o, float* m, float* l,
                                    int32_t mode, void* cuda_stream) {
  if (desc == nullptr) return CP_ERR_INVALID_ARGUMENT;
  if (desc->cp < 1 || desc->cp > (1 << 20)) return CP_ERR_INVALID_ARGUMENT;
  return cp_ring_rank_partial_attn(desc, CP_LAYOUT_BALANCED, 0, int32_t(desc->cp), step_begin, step_end, q, k, v,
                                   o, m, l, mode, cuda_stream);
}

cp_status cp_ring_attn_host_workspace_bytes(const cp_attn_desc* desc, size_t* bytes) {
  cp_status st = check_host_ring(desc);
  if (st != CP_OK) return st;
  if (bytes == nullptr) return CP_ERR_INVALID_ARGUMENT;
  *bytes = host_ring_layout(*desc).total;
  return CP_OK;
}

cp_status cp_ring_attn_host(const cp_attn_desc* desc, const void* q_host, const void* k_host, const void* v_host,
                            float* o_host, float* m_host, float* l_host, void* workspace, size_t workspace_bytes,
                            void* cuda_stream) {
  cp_status st = check_host_ring(desc);
  if (st != CP_OK) return st;
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr || m_host == nullptr ||
      l_host == nullptr)
    return CP_ERR_INVALID_ARGUMENT;
  const HostRingLayout w = host_ring_layout(*desc);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) != 0 || workspace_bytes < w.total)
    return CP_ERR_INVALID_ARGUMENT;
  PipeStreams ps;
  if (!pipe_streams(&ps)) return CP_ERR_CUDA;

  const cp_attn_desc& d = *desc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dq = ws + w.q;
  void* dk = ws + w.k;
  void* dv = ws + w.v;
  float* dout = reinterpret_cast<float*>(ws + w.o);
  float* dm = reinterpret_cast<float*>(ws + w.m);
  float* dl = reinterpret_cast<float*>(ws + w.l);
  const int32_t cp = int32_t(d.cp);
  const int64_t C = d.S / (2 * d.cp);
  const size_t q_row = size_t(d.h_q) * d.d * 2;   // bytes of one token's Q
  const size_t kv_row = size_t(d.h_kv) * d.d * 2;
  const size_t o_row = size_t(d.h_q) * d.d * 4;
  cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);

  // Work units in launch order: head chunks in ascending order (head chunk c sees
  // keys [0, (c+1) C) only, so the first can start once the first K/V chunks are in),
  // then tail chunks in descending order (they need all of K/V, which has arrived by
  // then).  Each unit is a contiguous range of ranks with one chunk selector.
  const int32_t n_half = cp < 8 ? cp : 8;
  const int32_t n_units = 2 * n_half;
  auto unit_ranks = [&](int u, int32_t* r0, int32_t* r1) {
    const int g = u % n_half;
    *r0 = int32_t(int64_t(g) * cp / n_half);
    *r1 = int32_t(int64_t(g + 1) * cp / n_half);
  };
  // chunk range [c0, c1) of unit u
  auto unit_chunks = [&](int u, int64_t* c0, int64_t* c1) {
    int32_t r0, r1;
    unit_ranks(u, &r0, &r1);
    if (u < n_half) {
      *c0 = r0;
      *c1 = r1;
    } else {
      *c0 = 2 * cp - r1;
      *c1 = 2 * cp - r0;
    }
  };

  constexpr int kMaxEv = 6 + 2 * 16 + 8 + 1;  // fixed, per unit (q, compute), K/V prefixes
  cudaEvent_t ev[kMaxEv];
  const int n_need = 6 + 2 * n_units + n_half + 1;
  int n_ev = 0;
  bool ok = true;
  for (int i = 0; i < n_need && ok; ++i, ++n_ev)
    ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    for (int i = 0; i + 1 < n_ev; ++i) cudaEventDestroy(ev[i]);
    return CP_ERR_CUDA;
  }
  cudaEvent_t e_start = ev[0], e_done = ev[1];
  cudaEvent_t e_tail[3] = {ev[2], ev[3], ev[4]};  // end of the in / compute streams' work
  auto e_q = [&](int u) { return ev[6 + u]; };
  auto e_c = [&](int u) { return ev[6 + n_units + u]; };
  auto e_kv = [&](int g) { return ev[6 + 2 * n_units + g]; };  // g < n_half: head units' K/V; n_half: all
  auto chk = [&](cudaError_t e) {
    if (e != cudaSuccess) ok = false;
  };
  // Chunks [c0, c1) of a [b, S, ...] tensor (row bytes given): one strided copy per call.
  auto copy_tok = [&](void* dst, const void* src, int64_t c0, int64_t c1, size_t row, cudaMemcpyKind kind,
                      cudaStream_t s) {
    const size_t off = size_t(c0 * C) * row;
    chk(cudaMemcpy2DAsync(static_cast<uint8_t*>(dst) + off, size_t(d.S) * row,
                          static_cast<const uint8_t*>(src) + off, size_t(d.S) * row, size_t((c1 - c0) * C) * row,
                          size_t(d.b), kind, s));
  };
  // Chunks [c0, c1) of a [b, h, S] fp32 tensor back to the host.
  auto copy_ml = [&](float* dst, const float* src, int64_t c0, int64_t c1, cudaStream_t s) {
    chk(cudaMemcpy2DAsync(dst + c0 * C, size_t(d.S) * 4, src + c0 * C, size_t(d.S) * 4, size_t((c1 - c0) * C) * 4,
                          size_t(d.b * d.h_q), cudaMemcpyDeviceToHost, s));
  };

  chk(cudaEventRecord(e_start, caller));
  chk(cudaStreamWaitEvent(ps.in, e_start, 0));
  chk(cudaStreamWaitEvent(ps.comp[0], e_start, 0));
  chk(cudaStreamWaitEvent(ps.comp[1], e_start, 0));
  chk(cudaStreamWaitEvent(ps.out, e_start, 0));
  // Copies in: each head unit's new K/V chunks and its Q, then the remaining K/V
  // (the tail half), then the tail units' Q.
  int64_t kv_done = 0;
  for (int u = 0; u < n_half && ok; ++u) {
    int64_t c0, c1;
    unit_chunks(u, &c0, &c1);
    if (c1 > kv_done) {
      copy_tok(dk, k_host, kv_done, c1, kv_row, cudaMemcpyHostToDevice, ps.in);
      copy_tok(dv, v_host, kv_done, c1, kv_row, cudaMemcpyHostToDevice, ps.in);
      kv_done = c1;
    }
    chk(cudaEventRecord(e_kv(u), ps.in));
    copy_tok(dq, q_host, c0, c1, q_row, cudaMemcpyHostToDevice, ps.in);
    chk(cudaEventRecord(e_q(u), ps.in));
  }
  if (ok) {
    copy_tok(dk, k_host, kv_done, 2 * cp, kv_row, cudaMemcpyHostToDevice, ps.in);
    copy_tok(dv, v_host, kv_done, 2 * cp, kv_row, cudaMemcpyHostToDevice, ps.in);
    chk(cudaEventRecord(e_kv(n_half), ps.in));
  }
  for (int u = n_half; u < n_units && ok; ++u) {
    int64_t c0, c1;
    unit_chunks(u, &c0, &c1);
    copy_tok(dq, q_host, c0, c1, q_row, cudaMemcpyHostToDevice, ps.in);
    chk(cudaEventRecord(e_q(u), ps.in));
  }
  // Launches (alternating compute streams) and copies out, unit by unit.
  for (int u = 0; u < n_units && ok; ++u) {
    int32_t r0, r1;
    int64_t c0, c1;
    unit_ranks(u, &r0, &r1);
    unit_chunks(u, &c0, &c1);
    cudaStream_t cs = ps.comp[u & 1];
    chk(cudaStreamWaitEvent(cs, e_kv(u < n_half ? u : n_half), 0));
    chk(cudaStreamWaitEvent(cs, e_q(u), 0));
    if (!ok) break;
    st = launch_ring_attn(d, CP_LAYOUT_BALANCED, r0, r1, 0, cp, dq, dk, dv, dout, dm, dl,
                          CP_MODE_EMIT | CP_MODE_FINALIZE, cs, u < n_half ? kRingFirstChunk : kRingSecondChunk,
                          false);
    if (st != CP_OK) {
      ok = false;
      break;
    }
    chk(cudaEventRecord(e_c(u), cs));
    chk(cudaStreamWaitEvent(ps.out, e_c(u), 0));
    copy_tok(o_host, dout, c0, c1, o_row, cudaMemcpyDeviceToHost, ps.out);
    copy_ml(m_host, dm, c0, c1, ps.out);
    copy_ml(l_host, dl, c0, c1, ps.out);
  }
  // Whatever was queued (also after a failure part-way), the caller's stream waits
  // for all of it, so no copy still reads or writes the caller's buffers afterwards.
  cudaStream_t others[3] = {ps.in, ps.comp[0], ps.comp[1]};
  for (int i = 0; i < 3; ++i) {
    cudaEventRecord(e_tail[i], others[i]);
    cudaStreamWaitEvent(ps.out, e_tail[i], 0);
  }
  cudaEventRecord(e_done, ps.out);
  cudaStreamWaitEvent(caller, e_done, 0);
  for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);
  if (!ok) return st != CP_OK ? st : CP_ERR_CUDA;
  return CP_OK;
}

cp_status cp_merge_partials(int64_t batch, int64_t rows, int64_t heads, int64_t d,
                            int32_t n_parts, const float* o_parts, const float* m_parts,
                            const float* l_parts, const int32_t* order, float* o_out,
                            float* m_out, float* l_out, int32_t finalize,
                            void* cuda_stream) {
  if (batch < 1 || rows < 1 || heads < 1 || d < 1 || n_parts < 1) return CP_ERR_INVALID_ARGUMENT;
  if (n_parts > CP_MAX_MERGE_PARTS) return CP_ERR_INVALID_ARGUMENT;
  if (d % 4 != 0) return CP_ERR_INVALID_ARGUMENT;
  if (d > 512) return CP_ERR_UNSUPPORTED;
  if (!product_fits(n_parts, batch, rows, heads * d)) return CP_ERR_INVALID_ARGUMENT;
  if (!aligned16(o_parts) || !aligned16(m_parts) || !aligned16(l_parts) || !aligned16(o_out) ||
      !aligned16(m_out) || !aligned16(l_out))
    return CP_ERR_INVALID_ARGUMENT;
  MergeParams p = merge_params(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out, l_out,
                               finalize != 0);
  if (order != nullptr) {
    bool seen[CP_MAX_MERGE_PARTS] = {false};
    for (int32_t i = 0; i < n_parts; ++i) {
      const int32_t x = order[i];
      if (x < 0 || x >= n_parts || seen[x]) return CP_ERR_INVALID_ARGUMENT;
      seen[x] = true;
      p.order[i] = static_cast<uint16_t>(x);
    }
  }
  return launch_merge(p, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_merge_tree_workspace_bytes(int64_t batch, int64_t rows, int64_t heads, int64_t d, int32_t n_parts,
                                        size_t* bytes) {
  if (bytes == nullptr || batch < 1 || rows < 1 || heads < 1 || d < 1 || n_parts < 2) return CP_ERR_INVALID_ARGUMENT;
  if ((n_parts & (n_parts - 1)) != 0 || n_parts > CP_MAX_MERGE_PARTS) return CP_ERR_INVALID_ARGUMENT;
  if (!product_fits(n_parts, batch, rows, heads * d)) return CP_ERR_INVALID_ARGUMENT;
  *bytes = 0;  // the tree is computed in one pass, with no intermediate levels in memory
  return CP_OK;
}

cp_status cp_merge_partials_tree(int64_t batch, int64_t rows, int64_t heads, int64_t d, int32_t n_parts,
                                 const float* o_parts, const float* m_parts, const float* l_parts,
                                 float* workspace, size_t workspace_bytes, float* o_out, float* m_out,
                                 float* l_out, int32_t finalize, void* cuda_stream) {
  (void)workspace;
  (void)workspace_bytes;
  size_t need = 0;
  cp_status st = cp_merge_tree_workspace_bytes(batch, rows, heads, d, n_parts, &need);
  if (st != CP_OK) return st;
  if (d % 4 != 0) return CP_ERR_INVALID_ARGUMENT;
  if (d > 512) return CP_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(m_parts) || !aligned16(l_parts) || !aligned16(o_out) ||
      !aligned16(m_out) || !aligned16(l_out))
    return CP_ERR_INVALID_ARGUMENT;
  const MergeParams p = merge_params(batch, rows, heads, d, n_parts, o_parts, m_parts, l_parts, o_out, m_out, l_out,
                                     finalize != 0);
  return launch_merge_tree(p, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_passq_workspace_bytes(const cp_attn_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return CP_ERR_INVALID_ARGUMENT;
  cp_status st = check_decode_desc(desc);
  if (st != CP_OK) return st;
  int sms = 0;
  if (current_sm_count(&sms) != cudaSuccess) return CP_ERR_CUDA;
  *bytes = decode_workspace_bytes(*desc, decode_splits_per_shard(*desc, sms));
  return CP_OK;
}

cp_status cp_passq_decode(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                          float* workspace, size_t workspace_bytes, float* out, float* m_out,
                          float* l_out, void* cuda_stream) {
  cp_status st = check_decode_desc(desc);
  if (st != CP_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(workspace) || !aligned16(out))
    return CP_ERR_INVALID_ARGUMENT;
  if ((m_out != nullptr && !aligned16(m_out)) || (l_out != nullptr && !aligned16(l_out)))
    return CP_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if (current_sm_count(&sms) != cudaSuccess) return CP_ERR_CUDA;
  const int32_t splits = decode_splits_per_shard(*desc, sms);
  const size_t need = decode_workspace_bytes(*desc, splits);
  if (workspace_bytes < need) return CP_ERR_INVALID_ARGUMENT;
  return run_passq_decode(*desc, splits, q, k, v, workspace, out, m_out, l_out,
                          static_cast<cudaStream_t>(cuda_stream));
}

cp_status cp_passq_decode_noalloc(const cp_attn_desc* desc, const void* q, const void* k, const void* v,
                                  float* out, float* m_out, float* l_out, void* cuda_stream) {
  cp_status st = check_decode_desc(desc);
  if (st != CP_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return CP_ERR_INVALID_ARGUMENT;
  if ((m_out != nullptr && !aligned16(m_out)) || (l_out != nullptr && !aligned16(l_out)))
    return CP_ERR_INVALID_ARGUMENT;
  int sms = 0;
  if (current_sm_count(&sms) != cudaSuccess) return CP_ERR_CUDA;
  // Same split of the shards as cp_passq_decode while the partials fit the fixed
  // scratch; fewer splits (halving keeps them dividing the shard) otherwise.
  const size_t cap = decode_noalloc_scratch_bytes();
  int32_t splits = decode_splits_per_shard(*desc, sms);
  while (splits > 1 && decode_workspace_bytes(*desc, splits) > cap) splits /= 2;
  if (decode_workspace_bytes(*desc, splits) > cap) return CP_ERR_UNSUPPORTED;
  if (desc->cp * splits > CP_MAX_MERGE_PARTS) return CP_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  if (decode_noalloc_scratch(&scratch) != cudaSuccess) return CP_ERR_CUDA;
  return run_passq_decode(*desc, splits, q, k, v, scratch, out, m_out, l_out, static_cast<cudaStream_t>(cuda_stream));
}

cp_status cp_set_kernel_choice(int32_t knob, int32_t value) {
  if (knob < 0 || knob >= kKnobs || value < -1 || value > 1) return CP_ERR_INVALID_ARGUMENT;
  g_kernel_choice[knob].store(value, std::memory_order_relaxed);
  return CP_OK;
}

cp_status cp_selftest_wait_timeout(void* cuda_stream) {
  return ring_wait_timeout_selftest(static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_take_device_status(void* cuda_stream, int32_t* status) {
  if (status == nullptr) return CP_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return CP_ERR_CUDA;
  int32_t s = CP_OK, s2 = CP_OK, s3 = CP_OK;
  if (ring_take_status(&s) != cudaSuccess || mqa_take_status(&s2) != cudaSuccess ||
      merge_take_status(&s3) != cudaSuccess)
    return CP_ERR_CUDA;
  *status = (s != CP_OK) ? s : (s2 != CP_OK ? s2 : s3);
  return CP_OK;
}

}  // extern "C"
