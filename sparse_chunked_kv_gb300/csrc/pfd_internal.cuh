// Definitions shared by the kernels of libpfd and its C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "pfd.h"

namespace pfd {

using bf16 = __nv_bfloat16;

// ----------------------------------------------------------- attention --
// One CTA computes one 128-row tile of packed query rows against one
// contiguous range ("split") of a key sequence.  Query rows of a tile are
// (token t, head j of the KV group) pairs packed as m = t * G + j, so the G
// query heads that share KV head g share every K/V tile (GQA packing).
// The key sequence is a list of segments (row ranges of a K/V tensor); it is
// consumed in groups of 16 rows, 8 groups per 128-key tile, so segments of
// any length share tiles and only a segment's last group is ragged.
constexpr int kBlockM = 128;
constexpr int kGroupRows = 16;
constexpr int kGroupsPerTile = 8;
constexpr int kBlockN = kGroupRows * kGroupsPerTile;
constexpr int kBoxLevels = 4;      // K/V box heights 16, 32, 64, 128 rows
constexpr int kMaxSegments = 512;   // selected chunks per sequence + the live block

enum AttnMode : int { kModePrefill = 0, kModeDecode = 1, kModeMass = 2 };
constexpr int kMaxMassBatch = 64;   // sequences of one chunk-mass call
constexpr int kMassChunks = 8;      // most consecutive chunks of one chunk-mass item

struct AttnParams {
  // Query tensors addressed by TMA: index 0 = prefill chunk rows or decode
  // live rows, index 1 = prefill window rows.  3-D maps over [tokens, Hq, D],
  // box = Tq tokens x G heads x 64 columns, 128-byte swizzle.
  CUtensorMap tm_q[2];
  // Key/value tensors: [box level][tensor], tensor 0 = prefill K/V or the
  // decode pool, tensor 1 = the decode live block.  3-D maps over
  // [rows, Hkv, D], 128-byte swizzle, box = (16 << level) rows x 1 head x 64
  // columns: a run of consecutive 16-row groups is loaded with one box per
  // set bit of its length.
  CUtensorMap tm_k[kBoxLevels][2];
  CUtensorMap tm_v[kBoxLevels][2];

  const bf16* q;        // prefill: chunk rows; decode: live rows
  const bf16* q_win;    // prefill: window rows
  bf16* out;            // [rows, Hq, D]
  float* lse;           // decode, one split: [total_lq, Hq] (may be null)
  float* part_m;        // decode, several splits: [S, total_lq, Hq] (log2 units)
  float* part_l;        // [S, total_lq, Hq]
  bf16* part_acc;       // [S, total_lq, Hq, D] normalised (acc / l) bf16
  float* win_b;         // prefill: [N, Hkv, win_stride] per window row n = w*G + j of
                        // each KV group: m + log2(l) of its softmax over the chunk
  int win_stride;       // (W*G rounded up to 32)
  const float* win_self_b;  // prefill, window keys in the denominator: [W, Hq]
                            // log2-sum-exp of each window row over the W window
                            // keys, folded into win_b (null: chunk keys only)

  const pfd_chunk_entry* table;
  const int32_t* sel;
  const int32_t* cu_k;
  const int32_t* cu_lq;
  int32_t* dev_err;

  long long pool_rows;
  int table_len;
  int mode;
  int Hq, Hkv, G, D;
  int Tq;               // tokens per query tile: floor(128 / G)
  int n_items;          // work items (pairs of query tiles x key range)

  // prefill
  int n_chunks, chunk_rows, n_win;
  int layer_chunks;     // chunks per layer (window rows of chunk c: layer c / layer_chunks)
  int mt_chunk;         // query tiles per (chunk, KV head) of chunk rows
  int mt_win;           // query tiles per (chunk, KV head) of window rows
  int n_chunk_items;    // n_chunks * Hkv * mt_chunk

  // decode
  int batch, mt_max, n_splits, total_lq, total_sel;
  int self_keys;        // 1: the live block is the last key segment; 0: selected chunks only

  float scale_log2;     // sm_scale * log2(e)
  int out_v8;           // out is 32-byte aligned: whole-sector (32-byte) stores

  // chunk mass (kModeMass): items of sequence b are mass_item0[b] ..
  // mass_item0[b+1]-1, item = (chunk group cg * Hkv + g) * mass_pairs[b] +
  // pair; chunk group cg holds table entries mass_n0[b] + cg * mass_chunks ..
  // (at most mass_chunks <= kMassChunks of them, ending before mass_n0[b + 1])
  const float* mass_lse;   // [total_lq, Hq] the step's decode log-sum-exp (natural log)
  float* mass_part;        // [n_items, mass_chunks, 8] partial sums per chunk of the item
                           // (two query tiles x four warps)
  int mass_chunks;
  int mass_batch;
  int mass_item0[kMaxMassBatch + 1];
  int mass_n0[kMaxMassBatch + 1];
  int mass_pairs[kMaxMassBatch];
};

cudaError_t launch_attention(const AttnParams& p, int grid, cudaStream_t stream);
size_t attention_smem_bytes(int D, bool prefill);

// ------------------------------------------------------- window scores --
struct WinScoreParams {
  CUtensorMap tm_k;         // prefill K, 128-row box (as AttnParams::tm_k[3][0])
  CUtensorMap tm_qwin;      // q_win [W, Hq, D], box = W tokens x G heads x 64 columns
  const bf16* q_win;        // [W, Hq, D]
  const float* win_b;       // [N, Hkv, win_stride], as AttnParams::win_b
  int win_stride;
  float* part_scores;       // [N, Hkv, C+1]
  int n_chunks, chunk_rows, n_win, Hq, Hkv, G, D;
  int k_tiles;              // ceil((C+1) / 128)
  int concat;               // 1: 128-row tiles over the chunks laid end to end (C+1 >= 128)
  int n_items;              // tiles per KV group and layer
  int n_layers;             // stacked layers: layer l's chunks are l*N .. l*N+N-1, its
                            // window rows l*W .. l*W+W-1 of the q_win map
  float scale_log2;
  int32_t* dev_err;
};

cudaError_t launch_window_scores(const WinScoreParams& p, cudaStream_t stream);
cudaError_t launch_window_self_stats(const bf16* q_win, const bf16* k_win, int W, int Hq, int Hkv,
                                     int D, float scale_log2, float* b_self, cudaStream_t stream);

// ------------------------------------------------- top-B + compaction --
struct TopBParams {
  const float* part_scores;  // [N, Hkv, C+1] or null when W == 0
  float* scores;             // [N, C+1] ([N, Hkv, C+1] per head)
  int32_t* kept_idx;         // [N, B] ([N, Hkv, B] per head)
  const bf16* k;             // [N*(C+1), Hkv, D]
  const bf16* v;
  bf16* pool_k;              // [pool_rows, Hkv, D]
  bf16* pool_v;
  const int32_t* slot_row;   // [N]
  pfd_chunk_entry* table;    // [N]
  int32_t* dev_err;
  long long pool_rows;
  int n_chunks, chunk_size, n_keep, Hkv, D;
  int copy_splits;
  int layer_chunks;          // chunks per layer: chunk c writes layer c / layer_chunks's
                             // pool (layer_pool_rows rows further per layer) at slot
                             // slot_row[c % layer_chunks], table entries relative to it
  long long layer_pool_rows;
  int slot_per_chunk;        // 1: chunk c's slot is slot_row[c], a row of the one pool of
                             // pool_rows rows (a batch of requests), table rows absolute
  int per_head;              // 1: one ranking per (chunk, KV head): scores [N, Hkv, C+1],
                             // kept_idx [N, Hkv, B], head g's slot column from head g's set
};

cudaError_t launch_topb_compact(const TopBParams& p, cudaStream_t stream);

// ----------------------------------------------------------- selection --
// s = fl32(s_i + fl32(lambda * s_p)) per chunk (lambda = 1: fl32(s_i + s_p)).
cudaError_t launch_select(const float* s_i, const float* s_p, const int32_t* cu_n,
                          const int32_t* cu_k, int n_scalar, int k_scalar, int batch, int max_n,
                          float lambda, int32_t* sel, float* s_out, cudaStream_t stream);

// ------------------------------------------------------------ LSE merge --
struct MergeParams {
  // Split states: part_m = max (log2 units) and part_l = denominator, or,
  // when part_l is null, part_m = natural-log log-sum-exp of the split (its
  // denominator relative to a max of 0: m = lse * log2(e), l = 1).
  const float* part_m;
  const float* part_l;
  const bf16* part_acc;     // normalised (acc / l) bf16
  bf16* out;
  float* lse;
  int n_splits, total_lq, Hq, D;
  int early_trigger;        // set by launch_lse_merge
};

// sm_count: SMs of the current device (the grid is one wave of resident CTAs).
cudaError_t launch_lse_merge(const MergeParams& p, int sm_count, cudaStream_t stream);

// Per-chunk sums of the chunk-mass partials: mass[n0[b] + c] = (sum of the
// partials of chunk c of sequence b) / (Lq_b * Hq).
cudaError_t launch_mass_sum(const AttnParams& p, const int32_t* cu_lq_host, int n_chunks_total,
                            float* mass, cudaStream_t stream);

// -------------------------------------------------------- chunk scores --
cudaError_t launch_chunk_loglik(const bf16* logits, const int32_t* labels, int n_chunks,
                                int n_rows, long long vocab, float* row_ll, float* score,
                                int32_t* dev_err, cudaStream_t stream);

// ------------------------------------------------------------- helpers --
// Raises a kernel's dynamic shared-memory limit once per (kernel, device), so
// that later calls -- including calls made while a stream is being captured
// into a CUDA graph -- only launch.
inline cudaError_t ensure_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<const void*, int>, int>> done;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : done)
    if (e.first.first == func && e.first.second == dev && e.second >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess) done.push_back({{func, dev}, bytes});
  return err;
}

// Launch that lets the kernel start while the previous kernel on the stream
// is still finishing (programmatic dependent launch): its CTAs may be
// scheduled early and run their prologue, and each one calls
// grid_dependency_wait() before it touches global memory, which returns once
// the previous grid has completed and its writes are visible.  Every kernel of
// this library is launched this way and waits before its first global access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Waits until the grid launched before this one on the stream has completed
// and its memory writes are visible (a no-op without a programmatic launch).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next grid on the stream be scheduled now; it still waits in
// grid_dependency_wait() for this grid to complete.
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Maps an fp32 value to an unsigned key whose unsigned order is the rank
// order: larger value = larger key, -0.0 and +0.0 share a key, NaN gets the
// smallest key.
__device__ __forceinline__ uint32_t rank_key(float x) {
  if (x != x) return 0u;
  if (x == 0.0f) x = 0.0f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void raise_dev_err(int32_t* dev_err, int bits) {
  if (dev_err != nullptr) atomicOr(dev_err, bits);
}

}  // namespace pfd
