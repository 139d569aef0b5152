// Chunk scores from vocabulary logits: the summed label log-likelihood of
// each chunk ("Chunked Prefill and KV Caching", predictive scoring: s_I is
// the (negated) negative log-likelihood of the query window given the chunk,
// s_P the likelihood of the pseudo-labels given the chunk and the query).
//
//   row_ll[j][r] = logits[j][r][y_r] - log(sum_v exp(logits[j][r][v]))
//   score[j]     = sum_r row_ll[j][r]
//
// The work is one streaming pass over N * R * V bf16 logits, so the kernel is
// HBM-bound: one 256-thread CTA per (chunk, row) reads its row with 16-byte
// non-allocating loads, four in flight per thread, and keeps an online
// log-sum-exp in base 2 (m = running max of z * log2(e), s = sum of
// 2^(z * log2(e) - m)).  The CTA reduces the 256 states in a fixed order,
// so the result does not depend on scheduling.  A second small kernel sums
// each chunk's rows in a fixed order.
#include <cmath>

#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kRowThreads = 256;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

struct LseState {
  float m;   // max of z * log2(e) (-inf when empty)
  float s;   // sum of 2^(z * log2(e) - m)
};

__device__ __forceinline__ LseState lse_combine(LseState a, LseState b) {
  const float mm = fmaxf(a.m, b.m);
  if (mm == -INFINITY) return {mm, 0.0f};
  return {mm, a.s * ex2_approx(a.m - mm) + b.s * ex2_approx(b.m - mm)};
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Folds 8 logits (one 16-byte vector) into the state.
__device__ __forceinline__ void fold8(LseState& st, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_lo(w[i]) * kLog2e;
    x[2 * i + 1] = bf16_hi(w[i]) * kLog2e;
  }
  const float m8 = fmaxf(fmaxf(max3(x[0], x[1], x[2]), max3(x[3], x[4], x[5])), fmaxf(x[6], x[7]));
  if (m8 == -INFINITY) return;   // all eight are -inf: nothing to add
  if (m8 > st.m) {
    st.s = st.m == -INFINITY ? 0.0f : st.s * ex2_approx(st.m - m8);
    st.m = m8;
  }
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += ex2_approx(x[i] - st.m);
  st.s += acc;
}

__device__ __forceinline__ void fold1(LseState& st, float z) {
  const float x = z * kLog2e;
  if (x == -INFINITY) return;
  if (x > st.m) {
    st.s = st.m == -INFINITY ? 0.0f : st.s * ex2_approx(st.m - x);
    st.m = x;
  }
  st.s += ex2_approx(x - st.m);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kRowThreads)
row_loglik_kernel(const bf16* __restrict__ logits, const int32_t* __restrict__ labels, int n_rows,
                  long long vocab, float* __restrict__ row_ll, int32_t* dev_err) {
  grid_dependency_wait();
  const long long row = blockIdx.x;   // chunk j = row / R, r = row % R
  const int tid = threadIdx.x;
  const bf16* z = logits + row * vocab;
  // Elements before the first 16-byte boundary of the row, then whole
  // vectors, then the tail.
  const uintptr_t addr = reinterpret_cast<uintptr_t>(z);
  const long long head = static_cast<long long>(((16u - (addr & 15u)) & 15u) >> 1);
  const long long n_head = head < vocab ? head : vocab;
  const long long n_vec = (vocab - n_head) >> 3;
  const uint4* body = reinterpret_cast<const uint4*>(z + n_head);
  const long long tail0 = n_head + n_vec * 8;

  LseState st{-INFINITY, 0.0f};
  const uint16_t* zs = reinterpret_cast<const uint16_t*>(z);
  for (long long i = tid; i < n_head; i += kRowThreads)
    fold1(st, __uint_as_float(static_cast<uint32_t>(zs[i]) << 16));
  long long i = tid;
  for (; i + (kUnroll - 1) * kRowThreads < n_vec; i += kUnroll * kRowThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(body + i + u * kRowThreads);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) fold8(st, v[u]);
  }
  for (; i < n_vec; i += kRowThreads) fold8(st, ld_stream(body + i));
  for (long long t = tail0 + tid; t < vocab; t += kRowThreads)
    fold1(st, __uint_as_float(static_cast<uint32_t>(zs[t]) << 16));

  // Fixed-order reduction: warp tree, then warp 0 over the 8 warp states.
  __shared__ LseState warp_st[kRowThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LseState other{__shfl_xor_sync(0xFFFFFFFFu, st.m, o), __shfl_xor_sync(0xFFFFFFFFu, st.s, o)};
    st = lse_combine(st, other);
  }
  if ((tid & 31) == 0) warp_st[tid >> 5] = st;
  __syncthreads();
  grid_dependents_launch();
  if (tid == 0) {
    LseState all = warp_st[0];
    for (int w = 1; w < kRowThreads / 32; ++w) all = lse_combine(all, warp_st[w]);
    const int r = static_cast<int>(row % n_rows);
    const int y = labels[r];
    float out;
    if (y < 0 || static_cast<long long>(y) >= vocab) {
      raise_dev_err(dev_err, PFD_DEVERR_LABEL);
      out = __int_as_float(0x7FC00000);   // NaN: ranks below every chunk
    } else {
      const float zy = __uint_as_float(static_cast<uint32_t>(zs[y]) << 16);
      out = zy - (all.m + log2f(all.s)) * kLn2;
    }
    row_ll[row] = out;
  }
}

// score[j] = sum of row_ll[j][0..R-1]: lane l adds rows l, l + 32, ... in
// order, then a fixed shuffle tree.
__global__ void __launch_bounds__(32)
chunk_sum_kernel(const float* __restrict__ row_ll, int n_rows, float* __restrict__ score) {
  grid_dependency_wait();
  grid_dependents_launch();
  const int j = blockIdx.x, lane = threadIdx.x;
  float acc = 0.0f;
  for (int r = lane; r < n_rows; r += 32) acc += row_ll[static_cast<long long>(j) * n_rows + r];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) score[j] = acc;
}

}  // namespace

cudaError_t launch_chunk_loglik(const bf16* logits, const int32_t* labels, int n_chunks,
                                int n_rows, long long vocab, float* row_ll, float* score,
                                int32_t* dev_err, cudaStream_t stream) {
  const long long rows = static_cast<long long>(n_chunks) * n_rows;
  cudaError_t err = launch_pdl(row_loglik_kernel, dim3(static_cast<unsigned>(rows)),
                               dim3(kRowThreads), 0, stream, logits, labels, n_rows, vocab,
                               row_ll, dev_err);
  if (err != cudaSuccess) return err;
  return launch_pdl(chunk_sum_kernel, dim3(n_chunks), dim3(32), 0, stream,
                    static_cast<const float*>(row_ll), n_rows, score);
}

}  // namespace pfd
