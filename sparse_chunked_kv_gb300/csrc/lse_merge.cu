// Log-sum-exp merge of split-KV partial softmax states ("Attention Kernel
// Optimization" of the Prefilling-dLLM summary: chunks are processed
// independently and the results are merged by a log-sum-exp reduction).
//
// For one (row, head) with partials (m_s, l_s, acc_s), m in log2 units:
//   M = max_s m_s,  w_s = 2^(m_s - M),  L = sum_s w_s l_s,
//   out = sum_s w_s acc_s / L,  lse = (M + log2 L) * ln 2.
// One warp per (row, head); each lane owns 4 consecutive columns of D.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kMergeThreads = 256;
constexpr float kLn2 = 0.69314718055994530942f;

__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const MergeParams p) {
  const long long pair = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const long long n_pairs = static_cast<long long>(p.total_lq) * p.Hq;
  if (pair >= n_pairs) return;
  const int lane = threadIdx.x & 31;
  float big_m = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) big_m = fmaxf(big_m, p.part_m[s * n_pairs + pair]);
  float big_l = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool active = lane * 4 < p.D;
  for (int s = 0; s < p.n_splits; ++s) {
    const float m = p.part_m[s * n_pairs + pair];
    const float w = (m == -INFINITY) ? 0.0f : ex2_approx(m - big_m);
    big_l = fmaf(w, p.part_l[s * n_pairs + pair], big_l);
    if (active && w != 0.0f) {
      const float4 a = *reinterpret_cast<const float4*>(p.part_acc + (s * n_pairs + pair) * p.D + lane * 4);
      acc.x = fmaf(w, a.x, acc.x);
      acc.y = fmaf(w, a.y, acc.y);
      acc.z = fmaf(w, a.z, acc.z);
      acc.w = fmaf(w, a.w, acc.w);
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

}  // namespace

cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream) {
  const long long n_pairs = static_cast<long long>(p.total_lq) * p.Hq;
  const long long blocks = (n_pairs + kMergeThreads / 32 - 1) / (kMergeThreads / 32);
  if (blocks <= 0) return cudaSuccess;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pfd
