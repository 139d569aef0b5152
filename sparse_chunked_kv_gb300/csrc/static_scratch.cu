// pfd_decode_attention_static_scratch: the static-KV decode attention call
// with its split-KV partials kept in one fixed, statically allocated device
// buffer instead of caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point of
// the call.  A plain C or C++ host program that links only libpfd holds no
// device allocator to size and own a workspace with, and a hook run inside
// another runtime's step (a scheduler callback, a plug-in of an inference
// engine) may be barred from allocating there because that runtime owns and
// accounts every device byte.  Such a caller passes no workspace at all.
//
// The buffer is a file-scope __device__ array, one copy per device, created
// when the CUDA runtime loads this module on that device.  Every call looks
// up the current device's copy with cudaGetSymbolAddress, with that device
// current, and passes the address to the kernels.  No address is cached, so
// a device reset (after which the module may load at another address) needs
// nothing from the caller.  Nothing here calls cudaMalloc, cudaFree or any
// other allocating routine.
//
// Nothing in the buffer has to start at zero: for every (split, row, head)
// the merge reads, the attention kernel of the same call writes it first:
// the split's running max m (log2 units), its denominator l and its output
// row normalised by l, in bf16.  A split that saw no key writes m = -inf,
// l = 0 and a zero row, and the merge gives it weight 0.  Because every call
// on a device shares the one buffer, two calls whose kernels overlap on that
// GPU (different streams with no ordering between them) race on it; calls
// on one stream are safe.
#include <cuda_runtime.h>

#include "pfd.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[PFD_DECODE_STATIC_SCRATCH_BYTES];

// Address of the current device's copy of the buffer (nullptr on failure).
void* scratch_on_current_device() {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_decode_scratch) != cudaSuccess) return nullptr;
  return addr;
}

}  // namespace

extern "C" pfd_status pfd_decode_attention_static_scratch(
    const pfd_bf16* q, const pfd_bf16* k_self, const pfd_bf16* v_self, const int32_t* cu_lq,
    const int32_t* cu_lq_host, const pfd_bf16* pool_k, const pfd_bf16* pool_v, int64_t pool_rows,
    const pfd_chunk_entry* table, int32_t table_len, const int32_t* sel, const int32_t* cu_k,
    const int32_t* cu_k_host, int batch, int Hq, int Hkv, int D, int max_chunk_len,
    float sm_scale, int n_splits, pfd_bf16* out, float* lse, int32_t* dev_err,
    pfd_stream_t stream) {
  if (batch < 1 || cu_lq_host == nullptr || cu_k_host == nullptr) return PFD_ERR_INVALID_ARG;
  if (n_splits < 0) return PFD_ERR_INVALID_ARG;
  int splits = n_splits;
  if (splits == 0) {
    // The planned split count, lowered until its partials fit the buffer
    // (one split needs none).
    splits = pfd_decode_plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len);
    while (splits > 1 && pfd_decode_workspace(batch, cu_lq_host, cu_k_host, Hq, Hkv, D,
                                              max_chunk_len, splits) >
                             PFD_DECODE_STATIC_SCRATCH_BYTES)
      --splits;
    if (splits < 1) splits = 1;
  }
  const size_t need = pfd_decode_workspace(batch, cu_lq_host, cu_k_host, Hq, Hkv, D,
                                           max_chunk_len, splits);
  if (need > PFD_DECODE_STATIC_SCRATCH_BYTES) return PFD_ERR_UNSUPPORTED;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return PFD_ERR_CUDA;
  return pfd_decode_attention(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v, pool_rows,
                              table, table_len, sel, cu_k, cu_k_host, batch, Hq, Hkv, D,
                              max_chunk_len, sm_scale, splits, out, lse, dev_err, scratch,
                              PFD_DECODE_STATIC_SCRATCH_BYTES, stream);
}
