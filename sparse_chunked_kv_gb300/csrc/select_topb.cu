// Integer-exact selection kernels of the Prefilling-dLLM path.
//
// topb_compact: per chunk, adds the Hkv partial window scores in a fixed
//   order, keeps the B content tokens with the largest fp32 score (ties to the
//   lower index; "Two-Level Sparsity", intra-chunk), and copies BOS + the kept
//   K/V rows, ascending, into the chunk's pool slot ("Chunked Prefill and KV
//   Caching": the selected chunks' KV is cached), writing the chunk table.
//   The B-th largest score is found by an MSB-first radix select over
//   order-preserving 32-bit keys; positions come from block-wide prefix sums,
//   so the result is deterministic and exact.  Several CTAs per chunk redo the
//   (cheap) selection and each copies a slice of the rows, so the copy uses
//   the whole GPU.
//
// select: s = fl32(s_I + s_P) per chunk and the K best chunks in rank order
//   ("Selection" of Methodology 1): each chunk's rank is the number of chunks
//   that beat it, counted exactly.
#include "pfd_internal.cuh"

namespace pfd {
namespace {

// Threads of a top-B CTA: 256 for chunks of up to 2048 tokens (more CTAs
// resident per SM, more copy splits per chunk), 1024 up to 8192.
constexpr int kTopBThreadsSmall = 256;
constexpr int kTopBThreadsLarge = 1024;
constexpr int kMaxPerThread = 8;   // C <= 8 * threads

// Block-wide exclusive prefix sum of one value per thread (kThreads threads,
// at most 32 warps).
template <int kThreads>
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) warp_sums[lane] = wi - w;   // exclusive warp offsets
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int res = warp_sums[warp] + incl - v;
  total = warp_sums[32];
  __syncthreads();
  return res;
}

// 4. Chunk table and the copy of BOS + kept rows (kept_src, slot order) into
// chunk j's pool slot; CTA `part` of copy_splits copies its share of the rows.
// Per-head ranking (head >= 0): only KV head `head`'s columns of the rows.
template <int kThreads>
__device__ __forceinline__ void copy_kept_rows(const TopBParams& p, int j, int head, int part,
                                               int rows, const int* kept_src, int tid) {
  const int B = p.n_keep;
  // Layer of chunk j: its pool starts layer_pool_rows rows further per layer.
  // A batch of requests shares one pool: every chunk has its own slot there.
  const int layer = j / p.layer_chunks;
  const long long slot = p.slot_row[p.slot_per_chunk ? j : j % p.layer_chunks];
  const long long slot_limit = p.slot_per_chunk ? p.pool_rows : p.layer_pool_rows;
  const bool slot_ok = slot >= 0 && slot + B + 1 <= slot_limit;
  const long long pool0 = p.slot_per_chunk ? 0 : static_cast<long long>(layer) * p.layer_pool_rows;
  if (part == 0 && tid == 0 && head <= 0) {
    pfd_chunk_entry e;
    e.row = slot_ok ? static_cast<int32_t>(slot) : 0;
    e.len = slot_ok ? B + 1 : 0;
    p.table[j] = e;
    if (!slot_ok) raise_dev_err(p.dev_err, PFD_DEVERR_SLOT);
  }
  if (!slot_ok) return;
  const int n_rows_out = B + 1;
  const int r0 = static_cast<int>(static_cast<long long>(n_rows_out) * part / p.copy_splits);
  const int r1 = static_cast<int>(static_cast<long long>(n_rows_out) * (part + 1) / p.copy_splits);
  const int row_units = p.Hkv * p.D / 8;              // 16-byte units per token row
  const int units = head < 0 ? row_units : p.D / 8;   // units copied per row
  const int u0 = head < 0 ? 0 : head * (p.D / 8);     // first unit copied
  const long long chunk_row0 = static_cast<long long>(j) * rows;
  for (int idx = tid; idx < (r1 - r0) * units; idx += kThreads) {
    const int r = r0 + idx / units, u = u0 + idx % units;
    const long long src = (chunk_row0 + kept_src[r]) * row_units + u;
    const long long dst = (pool0 + slot + r) * row_units + u;
    reinterpret_cast<uint4*>(p.pool_k)[dst] = __ldg(reinterpret_cast<const uint4*>(p.k) + src);
    reinterpret_cast<uint4*>(p.pool_v)[dst] = __ldg(reinterpret_cast<const uint4*>(p.v) + src);
  }
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads)
topb_compact_kernel(const TopBParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t hist[256];
  __shared__ int warp_sums[33];
  __shared__ uint32_t sel_prefix;
  __shared__ int sel_remaining;
  __shared__ int sel_eq_total;   // keys equal to the threshold (last round)

  grid_dependency_wait();
  grid_dependents_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Ranking unit: chunk j, or (chunk j, KV head g) with per-head ranking.
  const int vj = blockIdx.x;
  const int j = p.per_head ? vj / p.Hkv : vj;
  const int head = p.per_head ? vj % p.Hkv : -1;
  const int part = blockIdx.y;
  const int C = p.chunk_size, rows = C + 1, B = p.n_keep;
  float* sc = reinterpret_cast<float*>(smem_raw);                   // [rows]
  int* kept_src = reinterpret_cast<int*>(smem_raw + ((rows * 4 + 15) & ~15));  // [B+1]

  // 1. Scores: fixed-order sum of the Hkv partial column sums (per-head
  // ranking: that head's partial alone).
  for (int t = tid; t < rows; t += kThreads) {
    float s = 0.0f;
    if (p.part_scores != nullptr) {
      if (head >= 0) {
        s = p.part_scores[static_cast<long long>(vj) * rows + t];
      } else {
        for (int g = 0; g < p.Hkv; ++g)
          s += p.part_scores[(static_cast<long long>(j) * p.Hkv + g) * rows + t];
      }
    }
    sc[t] = s;
    if (part == 0) p.scores[static_cast<long long>(vj) * rows + t] = s;
  }
  if (tid == 0) kept_src[0] = 0;  // BOS is slot row 0
  __syncthreads();

  // 2. Threshold key T (the B-th largest) and how many keys equal to T to keep.
  const int per = (C + kThreads - 1) / kThreads;
  const int i0 = tid * per;
  uint32_t key[kMaxPerThread];
#pragma unroll
  for (int u = 0; u < kMaxPerThread; ++u)
    key[u] = (u < per && i0 + u < C) ? rank_key(sc[1 + i0 + u]) : 0u;

  uint32_t thr = 0u;
  int need_eq = 0;
  if (B > 0 && B < C) {
    uint32_t prefix = 0u, pmask = 0u;
    int remaining = B;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kMaxPerThread; ++u)
        if (u < per && i0 + u < C && (key[u] & pmask) == prefix)
          atomicAdd(&hist[(key[u] >> shift) & 255u], 1u);
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255-8l .. 248-8l (descending digit order)
        uint32_t cnt[8];
        int lsum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          cnt[b] = hist[255 - 8 * lane - b];
          lsum += static_cast<int>(cnt[b]);
        }
        int incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - lsum;
        if (excl < remaining && incl >= remaining) {
          int above = excl;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (above + static_cast<int>(cnt[b]) >= remaining) {
              sel_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - b) << shift);
              sel_remaining = remaining - above;
              sel_eq_total = static_cast<int>(cnt[b]);
              break;
            }
            above += static_cast<int>(cnt[b]);
          }
        }
      }
      __syncthreads();
      prefix = sel_prefix;
      remaining = sel_remaining;
      pmask |= 255u << shift;
    }
    thr = prefix;
    need_eq = remaining;
  }

  // 3. Kept flags in index order, then their positions.  Keys equal to the
  // threshold are kept lowest index first; when all of them are kept (the
  // B-th largest score is unique, say) their ranks are not needed.
  const bool all_eq = !(B > 0 && B < C) || sel_eq_total == need_eq;
  int total;
  int eq_base = 0;
  if (!all_eq) {
    int n_eq = 0;
#pragma unroll
    for (int u = 0; u < kMaxPerThread; ++u)
      if (u < per && i0 + u < C && key[u] == thr) ++n_eq;
    eq_base = block_exclusive_scan<kThreads>(n_eq, warp_sums, total);
  }
  uint32_t kept_mask = 0u;
  int n_kept = 0, eq_seen = 0;
#pragma unroll
  for (int u = 0; u < kMaxPerThread; ++u) {
    if (!(u < per && i0 + u < C)) continue;
    bool kept;
    if (B == 0) kept = false;
    else if (B >= C) kept = true;
    else if (key[u] > thr) kept = true;
    else if (key[u] == thr) kept = all_eq || (eq_base + eq_seen++) < need_eq;
    else kept = false;
    if (kept) {
      kept_mask |= 1u << u;
      ++n_kept;
    }
  }
  int pos = block_exclusive_scan<kThreads>(n_kept, warp_sums, total);
#pragma unroll
  for (int u = 0; u < kMaxPerThread; ++u) {
    if (kept_mask & (1u << u)) {
      kept_src[1 + pos] = 1 + i0 + u;
      if (part == 0) p.kept_idx[static_cast<long long>(vj) * B + pos] = i0 + u;
      ++pos;
    }
  }
  __syncthreads();

  copy_kept_rows<kThreads>(p, j, head, part, rows, kept_src, tid);
}

constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads)
select_kernel(const float* __restrict__ s_i, const float* __restrict__ s_p,
              const int32_t* __restrict__ cu_n, const int32_t* __restrict__ cu_k, int n_scalar,
              int k_scalar, int max_n, float lambda, int32_t* __restrict__ sel,
              float* __restrict__ s_out) {
  extern __shared__ uint32_t keys[];
  grid_dependency_wait();
  grid_dependents_launch();
  const int b = blockIdx.x;
  const int off = cu_n ? cu_n[b] : 0;
  const int n = cu_n ? cu_n[b + 1] - off : n_scalar;
  const int koff = cu_k ? cu_k[b] : 0;
  const int k = cu_k ? cu_k[b + 1] - koff : k_scalar;
  if (n <= 0 || n > max_n || k < 0 || k > n) {
    // A malformed segment: its selection slots get -1, so that a decode
    // call reading them reports PFD_DEVERR_SEL instead of using stale
    // indices.  Only a range a valid cu_k could describe is written.
    if (koff >= 0 && k > 0 && k <= max_n)
      for (int t = threadIdx.x; t < k; t += kSelectThreads) sel[koff + t] = -1;
    return;
  }
  for (int t = threadIdx.x; t < n; t += kSelectThreads) {
    // fl32(s_i + fl32(lambda * s_p)), each step rounded to nearest even (no
    // contraction); lambda = 1 gives fl32(s_i + s_p) exactly.
    const float s = __fadd_rn(s_i[off + t], __fmul_rn(lambda, s_p[off + t]));
    if (s_out) s_out[off + t] = s;
    keys[t] = rank_key(s);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < n; t += kSelectThreads) {
    const uint32_t kt = keys[t];
    int rank = 0;
    for (int u = 0; u < n; ++u) {
      const uint32_t ku = keys[u];
      rank += (ku > kt) || (ku == kt && u < t);
    }
    if (rank < k) sel[koff + rank] = off + t;
  }
}

}  // namespace

// Launches (n_chunks x copy_splits) CTAs, with copy_splits chosen here from
// the kernel's occupancy so that the grid is about one resident wave.
template <int kThreads>
cudaError_t launch_topb_compact_t(TopBParams p, int sm_count, cudaStream_t stream) {
  const int rows = p.chunk_size + 1;
  const size_t smem = static_cast<size_t>((rows * 4 + 15) & ~15) + static_cast<size_t>(p.n_keep + 1) * 4;
  const void* fn = reinterpret_cast<const void*>(topb_compact_kernel<kThreads>);
  cudaError_t err = ensure_smem_limit(fn, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // Every CTA of a chunk redoes the selection and copies a share of its rows
  // (at least 16 rows each): as many CTAs per chunk as one resident wave holds.
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topb_compact_kernel<kThreads>,
                                                    kThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int wave = std::max(sm_count, 1) * per_sm;
  const int units = p.n_chunks * (p.per_head ? p.Hkv : 1);   // rankings
  p.copy_splits = std::max(1, std::min(wave / std::max(units, 1), std::max(1, (p.n_keep + 1) / 16)));
  dim3 grid(units, p.copy_splits);
  return launch_pdl(topb_compact_kernel<kThreads>, grid, dim3(kThreads), smem, stream, p);
}

cudaError_t launch_topb_compact(const TopBParams& params, cudaStream_t stream) {
  int dev = 0, sm_count = 1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sm_count = 1;
  if (params.chunk_size <= kMaxPerThread * kTopBThreadsSmall)
    return launch_topb_compact_t<kTopBThreadsSmall>(params, sm_count, stream);
  return launch_topb_compact_t<kTopBThreadsLarge>(params, sm_count, stream);
}

cudaError_t launch_select(const float* s_i, const float* s_p, const int32_t* cu_n,
                          const int32_t* cu_k, int n_scalar, int k_scalar, int batch, int max_n,
                          float lambda, int32_t* sel, float* s_out, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(max_n) * 4;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(select_kernel), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(select_kernel, dim3(batch), dim3(kSelectThreads), smem, stream, s_i, s_p, cu_n,
                    cu_k, n_scalar, k_scalar, max_n, lambda, sel, s_out);
}

}  // namespace pfd
