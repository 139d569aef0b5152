// Log-sum-exp merge of split-KV partial softmax states ("Attention Kernel
// Optimization" of the Prefilling-dLLM summary: chunks are processed
// independently and the results are merged by a log-sum-exp reduction).
//
// For one (row, head) with partials (m_s, l_s, O_s = acc_s / l_s), m in log2
// units:  M = max_s m_s,  w_s = 2^(m_s - M) l_s,  L = sum_s w_s,
//         out = sum_s w_s O_s / L,  lse = (M + log2 L) * ln 2.
// Up to four splits, a warp merges two (row, head) pairs; more, one pair.  Each
// lane owns 4 consecutive columns of D.
#include <algorithm>
#include <atomic>

#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kAccBatch = 8;   // split partials of O loaded per round trip (one-pair kernel)
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 v) {
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
}

// One split's (m, l) for a (row, head): stored as (max in log2 units,
// denominator), or, without part_l, as a natural-log log-sum-exp, which is
// the state (lse * log2(e), 1).  A split that saw no key has m = -inf.
__device__ __forceinline__ void load_state(const MergeParams& p, long long idx, float& m, float& l) {
  if (p.part_l != nullptr) {
    m = __ldg(p.part_m + idx);
    l = __ldg(p.part_l + idx);
  } else {
    const float lse = __ldg(p.part_m + idx);
    m = lse * kLog2e;
    l = lse == -INFINITY ? 0.0f : 1.0f;
  }
}

// More than 4 splits: one warp per (row, head).  Lane s loads split s's (m, l) (lanes loop when
// S > 32), so the statistics of every split arrive in one round trip; the O
// rows of up to kAccBatch splits are loaded in the same round trip.
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel_one(const MergeParams p) {
  grid_dependency_wait();
  // With p.early_trigger (a grid of at most two waves of resident CTAs) the
  // next kernel on the stream may be scheduled once every CTA has started:
  // its CTAs take the SMs as this grid's last wave leaves them.  A longer
  // grid signals only at its end, as an early next grid slowed its later
  // waves down.
  if (p.early_trigger) grid_dependents_launch();
  const long long pair = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const long long n_pairs = static_cast<long long>(p.total_lq) * p.Hq;
  if (pair >= n_pairs) return;
  const int lane = threadIdx.x & 31;
  const int S = p.n_splits;
  const bool active = lane * 4 < p.D;
  const bf16* o_base = p.part_acc + pair * p.D + lane * 4;
  const long long o_stride = n_pairs * p.D;

  uint2 a[kAccBatch];
#pragma unroll
  for (int s = 0; s < kAccBatch; ++s)
    if (active && s < S) a[s] = __ldg(reinterpret_cast<const uint2*>(o_base + s * o_stride));

  float m_lane = -INFINITY, l_lane = 0.0f;   // lane's own splits s = lane, lane + 32
  float m_hi = -INFINITY, l_hi = 0.0f;
  if (lane < S) load_state(p, lane * n_pairs + pair, m_lane, l_lane);
  if (lane + 32 < S) load_state(p, (lane + 32) * n_pairs + pair, m_hi, l_hi);
  float big_m = fmaxf(m_lane, m_hi);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) big_m = fmaxf(big_m, __shfl_xor_sync(0xFFFFFFFFu, big_m, o));
  // Weight of each split: 2^(m_s - M) * l_s (0 for a split that saw no key).
  const float w_lane = (m_lane == -INFINITY) ? 0.0f : ex2_approx(m_lane - big_m) * l_lane;
  const float w_hi = (m_hi == -INFINITY) ? 0.0f : ex2_approx(m_hi - big_m) * l_hi;
  float big_l = w_lane + w_hi;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) big_l += __shfl_xor_sync(0xFFFFFFFFu, big_l, o);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += kAccBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int s = 0; s < kAccBatch; ++s)
        if (active && s0 + s < S) a[s] = __ldg(reinterpret_cast<const uint2*>(o_base + (s0 + s) * o_stride));
    }
#pragma unroll
    for (int s = 0; s < kAccBatch; ++s) {
      const int src = (s0 + s) & 31;
      const float wl = __shfl_sync(0xFFFFFFFFu, w_lane, src);
      const float wh = __shfl_sync(0xFFFFFFFFu, w_hi, src);
      const float w = (s0 + s) < 32 ? wl : wh;
      if (active && s0 + s < S && w != 0.0f) {
        const float4 v = bf16x4_to_float4(a[s]);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
  }
  const float inv = big_l > 0.0f ? 1.0f / big_l : 0.0f;
  if (active) {
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + pair * p.D + lane * 4) = packed;
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[pair] = big_l > 0.0f ? (big_m + log2f(big_l)) * kLn2 : -INFINITY;
  grid_dependents_launch();
}

// Up to kB splits: kP (row, head) pairs per warp, their loads in flight
// together (fewer CTAs, fewer rounds of L2 latency): lane s
// loads split s's (m, l) (lanes loop when S > 32), so the statistics of every
// split arrive in one round trip, and the O rows of up to kB splits are
// loaded in the same round trip.
template <int kP, int kB>
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(const MergeParams p) {
  grid_dependency_wait();
  // With p.early_trigger (a grid of at most two waves of resident CTAs) the
  // next kernel on the stream may be scheduled once every CTA has started:
  // its CTAs take the SMs as this grid's last wave leaves them.  A longer
  // grid signals only at its end, as an early next grid slowed its later
  // waves down.
  if (p.early_trigger) grid_dependents_launch();
  const long long pair0 =
      (static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5)) * kP;
  const long long n_pairs = static_cast<long long>(p.total_lq) * p.Hq;
  if (pair0 >= n_pairs) return;
  const int lane = threadIdx.x & 31;
  const int S = p.n_splits;
  const bool active = lane * 4 < p.D;
  const long long o_stride = n_pairs * p.D;

  uint2 a[kP][kB];
  float m_lane[kP], l_lane[kP], m_hi[kP], l_hi[kP];   // lane's own splits s = lane, lane + 32
#pragma unroll
  for (int i = 0; i < kP; ++i) {
    const long long pair = pair0 + i;
    const bool valid = pair < n_pairs;
    const bf16* o_base = p.part_acc + pair * p.D + lane * 4;
#pragma unroll
    for (int s = 0; s < kB; ++s)
      if (valid && active && s < S) a[i][s] = __ldg(reinterpret_cast<const uint2*>(o_base + s * o_stride));
    m_lane[i] = m_hi[i] = -INFINITY;
    l_lane[i] = l_hi[i] = 0.0f;
    if (valid && lane < S) load_state(p, lane * n_pairs + pair, m_lane[i], l_lane[i]);
    if (valid && lane + 32 < S) load_state(p, (lane + 32) * n_pairs + pair, m_hi[i], l_hi[i]);
  }
#pragma unroll
  for (int i = 0; i < kP; ++i) {
    const long long pair = pair0 + i;
    if (pair >= n_pairs) break;   // warp-uniform
    const bf16* o_base = p.part_acc + pair * p.D + lane * 4;
    float big_m = fmaxf(m_lane[i], m_hi[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) big_m = fmaxf(big_m, __shfl_xor_sync(0xFFFFFFFFu, big_m, o));
    // Weight of each split: 2^(m_s - M) * l_s (0 for a split that saw no key).
    const float w_lane = (m_lane[i] == -INFINITY) ? 0.0f : ex2_approx(m_lane[i] - big_m) * l_lane[i];
    const float w_hi = (m_hi[i] == -INFINITY) ? 0.0f : ex2_approx(m_hi[i] - big_m) * l_hi[i];
    float big_l = w_lane + w_hi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) big_l += __shfl_xor_sync(0xFFFFFFFFu, big_l, o);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += kB) {
      if (s0 > 0) {
#pragma unroll
        for (int s = 0; s < kB; ++s)
          if (active && s0 + s < S)
            a[i][s] = __ldg(reinterpret_cast<const uint2*>(o_base + (s0 + s) * o_stride));
      }
#pragma unroll
      for (int s = 0; s < kB; ++s) {
        const int src = (s0 + s) & 31;
        const float wl = __shfl_sync(0xFFFFFFFFu, w_lane, src);
        const float wh = __shfl_sync(0xFFFFFFFFu, w_hi, src);
        const float w = (s0 + s) < 32 ? wl : wh;
        if (active && s0 + s < S && w != 0.0f) {
          const float4 v = bf16x4_to_float4(a[i][s]);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
    const float inv = big_l > 0.0f ? 1.0f / big_l : 0.0f;
    if (active) {
      uint2 packed;
      packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(p.out + pair * p.D + lane * 4) = packed;
    }
    if (lane == 0 && p.lse != nullptr)
      p.lse[pair] = big_l > 0.0f ? (big_m + log2f(big_l)) * kLn2 : -INFINITY;
  }
  grid_dependents_launch();
}

// CTAs of a merge kernel resident on an SM at once (cached per device and
// kernel; 1 if the query fails).
template <typename Kernel>
int merge_ctas_per_sm(Kernel kernel, int which) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
  int n = cache[dev][which].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kMergeThreads, 0) != cudaSuccess ||
      n < 1)
    n = 1;
  cache[dev][which].store(n, std::memory_order_relaxed);
  return n;
}

template <typename Kernel>
cudaError_t launch_merge_with(Kernel kernel, int which, int pairs_per_warp, MergeParams p,
                              int sm_count, cudaStream_t stream) {
  const long long n_pairs = static_cast<long long>(p.total_lq) * p.Hq;
  const long long per_cta = (kMergeThreads / 32) * pairs_per_warp;
  const long long blocks = (n_pairs + per_cta - 1) / per_cta;
  if (blocks <= 0) return cudaSuccess;
  const long long wave = static_cast<long long>(std::max(sm_count, 1)) * merge_ctas_per_sm(kernel, which);
  p.early_trigger = blocks <= 2 * wave ? 1 : 0;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kMergeThreads), 0, stream, p);
}

}  // namespace

// Up to 4 splits: two (row, head) pairs per warp with all their partials in
// flight at once (half the CTAs, about one wave); more: one pair per warp,
// 8 splits per round trip.
cudaError_t launch_lse_merge(const MergeParams& params, int sm_count, cudaStream_t stream) {
  if (params.n_splits <= 4)
    return launch_merge_with(lse_merge_kernel<2, 4>, 0, 2, params, sm_count, stream);
  return launch_merge_with(lse_merge_kernel_one, 1, 1, params, sm_count, stream);
}

namespace {

// Per-chunk sums of the chunk-mass partials (see AttnParams::mass_*): one
// warp per chunk of every sequence; lane l adds values l, l + 32, ... of
// the chunk's contiguous partials in order, then a fixed shuffle tree.
struct MassSumParams {
  const float* part;
  float* mass;
  int batch, Hkv;
  int chunks_per_item;                 // consecutive chunks of one item
  int chunk_base[kMaxMassBatch + 1];   // prefix of the sequences' chunk counts
  int n0[kMaxMassBatch];
  int item0[kMaxMassBatch];
  int pairs[kMaxMassBatch];
  float inv_rows[kMaxMassBatch];       // 1 / (Lq_b * Hq), 0 when Lq_b = 0
};

__global__ void __launch_bounds__(128) mass_sum_kernel(const __grid_constant__ MassSumParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (i >= p.chunk_base[p.batch]) return;
  int b = 0;
  while (b + 1 < p.batch && p.chunk_base[b + 1] <= i) ++b;
  const int c = i - p.chunk_base[b];
  // Chunk c of sequence b is chunk s of chunk group cg; the items of that
  // group (KV head x pair of query tiles) each hold 8 partials for it.
  const int M = p.chunks_per_item;
  const int cg = c / M, s = c % M;
  const int n_items = p.Hkv * p.pairs[b];
  const float* src = p.part +
                     (static_cast<long long>(p.item0[b]) + static_cast<long long>(cg) * n_items) *
                         M * 8 +
                     s * 8;
  float acc = 0.0f;
  for (int k = lane; k < n_items * 8; k += 32)
    acc += src[static_cast<long long>(k >> 3) * M * 8 + (k & 7)];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) p.mass[p.n0[b] + c] = acc * p.inv_rows[b];
}

}  // namespace

cudaError_t launch_mass_sum(const AttnParams& ap, const int32_t* cu_lq_host, int n_chunks_total,
                            float* mass, cudaStream_t stream) {
  if (n_chunks_total <= 0) return cudaSuccess;
  MassSumParams p;
  p.part = ap.mass_part;
  p.mass = mass;
  p.batch = ap.mass_batch;
  p.Hkv = ap.Hkv;
  p.chunks_per_item = ap.mass_chunks;
  p.chunk_base[0] = 0;
  for (int b = 0; b < ap.mass_batch; ++b) {
    // a sequence without query rows has no items, and its chunks no mass
    const int n_b = ap.mass_pairs[b] > 0 ? ap.mass_n0[b + 1] - ap.mass_n0[b] : 0;
    p.chunk_base[b + 1] = p.chunk_base[b] + n_b;
    p.n0[b] = ap.mass_n0[b];
    p.item0[b] = ap.mass_item0[b];
    p.pairs[b] = ap.mass_pairs[b];
    const long long rows = static_cast<long long>(cu_lq_host[b + 1] - cu_lq_host[b]) * ap.Hq;
    p.inv_rows[b] = rows > 0 ? static_cast<float>(1.0 / static_cast<double>(rows)) : 0.0f;
  }
  const int n = p.chunk_base[ap.mass_batch];
  if (n <= 0) return cudaSuccess;
  return launch_pdl(mass_sum_kernel, dim3((n + 3) / 4), dim3(128), 0, stream, p);
}

}  // namespace pfd
