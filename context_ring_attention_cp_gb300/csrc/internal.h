// Internal interface between the C-ABI layer (capi.cpp) and the kernel files.
// Every function here is called only after capi.cpp has validated its arguments.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/cpattn.h"

namespace cpattn {

// ---- host helpers shared by the kernel files (capi.cpp) ----------------------
// The driver's cuTensorMapEncodeTiled, looked up once per process; null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// SM count of the calling thread's current device.
cudaError_t current_sm_count(int* sms);
// Current value of a cp_set_kernel_choice knob (-1 = automatic).
int32_t kernel_choice(int32_t knob);
// Id of the calling thread's current CUDA context (0 when none can be read).
unsigned long long current_context_id();
// A kernel's dynamic shared-memory limit, raised with cudaFuncSetAttribute only when the
// current context has not yet been given at least `bytes` (the attribute belongs to the
// context's copy of the kernel: another device, or a device reset, needs it again).
// One SmemLimit per kernel (function-local static); calls may come from any thread.
struct SmemLimit {
  std::mutex mu;
  unsigned long long ctx = 0;
  int bytes = 0;
};
cudaError_t raise_smem_limit(const void* func, int bytes, SmemLimit* lim);

// ---- LSE merge (merge.cu) --------------------------------------------------
struct MergeParams {
  int64_t batch, rows, heads, d;
  int32_t n_parts;
  int32_t finalize;
  const float* o_parts;
  const float* m_parts;
  const float* l_parts;
  float* o_out;
  float* m_out;  // may be null
  float* l_out;  // may be null
  uint16_t order[CP_MAX_MERGE_PARTS];  // fold order (a permutation of 0..n_parts-1)
};
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
// The halving tree over n_parts = 2^k parts (k in 1..8) in one pass; order[] is not used.
cudaError_t launch_merge_tree(const MergeParams& p, cudaStream_t stream);
// Reads and clears the merge kernels' device status word (after the caller synchronised).
cudaError_t merge_take_status(int32_t* status);

// ---- pass-Q decode partials (decode.cu) ------------------------------------
// Key ranges per shard chosen for the device's SM count; n_parts = cp * splits.
int32_t decode_splits_per_shard(const cp_attn_desc& d, int sm_count);
size_t decode_workspace_bytes(const cp_attn_desc& d, int32_t splits);
// Splits the workspace into O partials [n_parts, b, h_q, d], then m and l [n_parts, b, h_q],
// each section starting on a 16-byte boundary.
void decode_workspace_sections(const cp_attn_desc& d, int32_t splits, float* ws, float** o_parts,
                               float** m_parts, float** l_parts);
bool decode_supported(const cp_attn_desc& d);
cudaError_t launch_decode_partials(const cp_attn_desc& d, int32_t splits, const void* q,
                                   const void* k, const void* v, float* o_parts,
                                   float* m_parts, float* l_parts, cudaStream_t stream);

// Fixed 8 MiB device scratch used by cp_passq_decode_noalloc (decode.cu): its size,
// and its device address on the current device (looked up once per device and context).
size_t decode_noalloc_scratch_bytes();
cudaError_t decode_noalloc_scratch(float** ptr);

// ---- pass-Q decode for heads sharing one K/V head, tensor cores (decode_mqa.cu)
bool decode_mqa_supported(const cp_attn_desc& d);
int32_t decode_mqa_splits(const cp_attn_desc& d, int sm_count);
cudaError_t launch_decode_mqa(const cp_attn_desc& d, int32_t splits, const void* q, const void* k, const void* v,
                              float* o_parts, float* m_parts, float* l_parts, cudaStream_t stream);
cudaError_t mqa_take_status(int32_t* status);

// ---- ring-step attention (ring_attn.cu) ------------------------------------
bool ring_supported(const cp_attn_desc& d);
// Returns CP_OK, or CP_ERR_CUDA when a tensor map cannot be encoded or the launch fails.
// Which of each selected rank's two chunks a ring launch computes.
enum RingChunks : int32_t { kRingBothChunks = 0, kRingFirstChunk = 1, kRingSecondChunk = 2 };
// allow_split: a launch of few single query tiles may split their key walks over CTA
// clusters (results equal within rounding); the host-buffer ring's partial launches do
// not, so that they compute exactly what the one device launch would without the split.
cp_status launch_ring_attn(const cp_attn_desc& d, int32_t layout, int32_t rank_begin, int32_t rank_end,
                           int32_t step_begin, int32_t step_end, const void* q, const void* k,
                           const void* v, float* o, float* m, float* l, int32_t mode,
                           cudaStream_t stream, int32_t chunks = kRingBothChunks, bool allow_split = true);
// Reads and clears the ring kernel's device status word (after the caller synchronised).
cudaError_t ring_take_status(int32_t* status);
// Launches one CTA whose bounded wait can never complete (records CP_ERR_TIMEOUT).
cudaError_t ring_wait_timeout_selftest(cudaStream_t stream);

}  // namespace cpattn
