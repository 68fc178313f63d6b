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

#include "internal.h"

using namespace cpattn;

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

cudaError_t current_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
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
  if ((mode & ~(CP_MODE_ACCUMULATE | CP_MODE_FINALIZE)) != 0) return CP_ERR_INVALID_ARGUMENT;
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
  MergeParams p;
  memset(&p, 0, sizeof(p));
  if (order != nullptr) {
    bool seen[CP_MAX_MERGE_PARTS] = {false};
    for (int32_t i = 0; i < n_parts; ++i) {
      const int32_t x = order[i];
      if (x < 0 || x >= n_parts || seen[x]) return CP_ERR_INVALID_ARGUMENT;
      seen[x] = true;
      p.order[i] = static_cast<uint16_t>(x);
    }
  } else {
    for (int32_t i = 0; i < n_parts; ++i) p.order[i] = static_cast<uint16_t>(i);
  }
  p.batch = batch;
  p.rows = rows;
  p.heads = heads;
  p.d = d;
  p.n_parts = n_parts;
  p.finalize = finalize != 0;
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  p.o_out = o_out;
  p.m_out = m_out;
  p.l_out = l_out;
  return launch_merge(p, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_merge_tree_workspace_bytes(int64_t batch, int64_t rows, int64_t heads, int64_t d, int32_t n_parts,
                                        size_t* bytes) {
  if (bytes == nullptr || batch < 1 || rows < 1 || heads < 1 || d < 1 || n_parts < 2) return CP_ERR_INVALID_ARGUMENT;
  if ((n_parts & (n_parts - 1)) != 0 || n_parts > (1 << 20)) return CP_ERR_INVALID_ARGUMENT;
  if (!product_fits(n_parts, batch, rows, heads * d)) return CP_ERR_INVALID_ARGUMENT;
  // Two ping-pong levels of at most n_parts / 2 partial triples, O then m then l, 16-byte aligned sections.
  auto pad = [](size_t x) { return (x + 3) & ~size_t(3); };
  const size_t half = size_t(n_parts / 2) * size_t(batch) * size_t(rows) * size_t(heads);
  *bytes = 2 * (pad(half * size_t(d)) + 2 * pad(half)) * sizeof(float);
  return CP_OK;
}

cp_status cp_merge_partials_tree(int64_t batch, int64_t rows, int64_t heads, int64_t d, int32_t n_parts,
                                 const float* o_parts, const float* m_parts, const float* l_parts,
                                 float* workspace, size_t workspace_bytes, float* o_out, float* m_out,
                                 float* l_out, int32_t finalize, void* cuda_stream) {
  size_t need = 0;
  cp_status st = cp_merge_tree_workspace_bytes(batch, rows, heads, d, n_parts, &need);
  if (st != CP_OK) return st;
  if (d % 4 != 0) return CP_ERR_INVALID_ARGUMENT;
  if (d > 512) return CP_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(m_parts) || !aligned16(l_parts) || !aligned16(workspace) ||
      !aligned16(o_out) || !aligned16(m_out) || !aligned16(l_out))
    return CP_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < need) return CP_ERR_INVALID_ARGUMENT;
  auto pad = [](size_t x) { return (x + 3) & ~size_t(3); };
  const size_t half_rows = size_t(n_parts / 2) * size_t(batch) * size_t(rows) * size_t(heads);
  const size_t level_floats = pad(half_rows * size_t(d)) + 2 * pad(half_rows);
  float* lvl_o[2];
  float* lvl_m[2];
  float* lvl_l[2];
  for (int i = 0; i < 2; ++i) {
    lvl_o[i] = workspace + size_t(i) * level_floats;
    lvl_m[i] = lvl_o[i] + pad(half_rows * size_t(d));
    lvl_l[i] = lvl_m[i] + pad(half_rows);
  }
  // Level k merges part i with part i + n/2 for every i < n/2: a two-part merge whose
  // "batch" runs over (i, batch), because the part stride then is exactly n/2 parts.
  const float* src_o = o_parts;
  const float* src_m = m_parts;
  const float* src_l = l_parts;
  int cur = 0;
  for (int64_t n = n_parts; n >= 2; n /= 2) {
    const bool last = (n == 2);
    MergeParams p;
    memset(&p, 0, sizeof(p));
    p.batch = (n / 2) * batch;
    p.rows = rows;
    p.heads = heads;
    p.d = d;
    p.n_parts = 2;
    p.order[0] = 0;
    p.order[1] = 1;
    p.finalize = last && finalize != 0;
    p.o_parts = src_o;
    p.m_parts = src_m;
    p.l_parts = src_l;
    p.o_out = last ? o_out : lvl_o[cur];
    p.m_out = last ? m_out : lvl_m[cur];
    p.l_out = last ? l_out : lvl_l[cur];
    if (launch_merge(p, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return CP_ERR_CUDA;
    src_o = lvl_o[cur];
    src_m = lvl_m[cur];
    src_l = lvl_l[cur];
    cur ^= 1;
  }
  return CP_OK;
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
  const int64_t n_parts = desc->cp * splits;
  if (n_parts > CP_MAX_MERGE_PARTS) return CP_ERR_UNSUPPORTED;
  float *o_parts = nullptr, *m_parts = nullptr, *l_parts = nullptr;
  decode_workspace_sections(*desc, splits, workspace, &o_parts, &m_parts, &l_parts);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (launch_decode_partials(*desc, splits, q, k, v, o_parts, m_parts, l_parts, s) != cudaSuccess)
    return CP_ERR_CUDA;
  // Three-quantity reduce: the LSE merge over the parts in shard order, finalised.
  MergeParams p;
  memset(&p, 0, sizeof(p));
  p.batch = desc->b;
  p.rows = 1;
  p.heads = desc->h_q;
  p.d = desc->d;
  p.n_parts = static_cast<int32_t>(n_parts);
  p.finalize = 1;
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  p.o_out = out;
  p.m_out = m_out;
  p.l_out = l_out;
  for (int32_t i = 0; i < p.n_parts; ++i) p.order[i] = static_cast<uint16_t>(i);
  return launch_merge(p, s) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
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
  const int64_t n_parts = desc->cp * splits;
  if (n_parts > CP_MAX_MERGE_PARTS) return CP_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  if (decode_noalloc_scratch(&scratch) != cudaSuccess) return CP_ERR_CUDA;
  float *o_parts = nullptr, *m_parts = nullptr, *l_parts = nullptr;
  decode_workspace_sections(*desc, splits, scratch, &o_parts, &m_parts, &l_parts);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (launch_decode_partials(*desc, splits, q, k, v, o_parts, m_parts, l_parts, s) != cudaSuccess)
    return CP_ERR_CUDA;
  MergeParams p;
  memset(&p, 0, sizeof(p));
  p.batch = desc->b;
  p.rows = 1;
  p.heads = desc->h_q;
  p.d = desc->d;
  p.n_parts = static_cast<int32_t>(n_parts);
  p.finalize = 1;
  p.o_parts = o_parts;
  p.m_parts = m_parts;
  p.l_parts = l_parts;
  p.o_out = out;
  p.m_out = m_out;
  p.l_out = l_out;
  for (int32_t i = 0; i < p.n_parts; ++i) p.order[i] = static_cast<uint16_t>(i);
  return launch_merge(p, s) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_selftest_wait_timeout(void* cuda_stream) {
  return ring_wait_timeout_selftest(static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_take_device_status(void* cuda_stream, int32_t* status) {
  if (status == nullptr) return CP_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return CP_ERR_CUDA;
  int32_t s = CP_OK, s2 = CP_OK;
  if (ring_take_status(&s) != cudaSuccess || mqa_take_status(&s2) != cudaSuccess) return CP_ERR_CUDA;
  *status = (s != CP_OK) ? s : s2;
  return CP_OK;
}

}  // extern "C"
