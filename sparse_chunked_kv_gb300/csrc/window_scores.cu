// Cumulative attention weight each chunk row receives from the query window
// ("Two-Level Sparsity", intra-chunk ranking of the Prefilling-dLLM summary).
//
// score[j][t] = sum over window rows w and query heads h of
//               softmax over the C+1 rows of chunk j of (scale * q_win[w,h] . k[t,g]).
//
// The attention kernel has already produced, for every (chunk, head, window
// row), the row maximum m (log2 units) and the denominator l, folded here into
// one constant b = m + log2(l) per window row (p = 2^(s*scale - b)).  This kernel
// recomputes the logits transposed -- S^T = K Q_win^T with the 128 key rows of
// one tile on the TMEM lanes and the W*G window rows of one KV group on the
// TMEM columns -- so each thread owns one key and sums exp2(scale*s - b_n)
// over its TMEM row with no cross-thread reduction.  One CTA = (chunk, KV
// head, 128-key tile); it writes that head group's partial score, and the
// top-B kernel adds the Hkv partials in a fixed order.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kThreads = 160;       // warp 0: TMA + MMA; warps 1..4: one key row each thread
constexpr uint32_t kPanelBytes = 128u * 128u;
constexpr int kMaxWindowRows = 512;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
window_score_kernel(const __grid_constant__ WinScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_k;
  __shared__ uint64_t bar_mma[2];
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  __shared__ __align__(16) float b_sh[kMaxWindowRows];   // per column: m_n + log2(l_n)

  grid_dependency_wait();
  grid_dependents_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bid = blockIdx.x;
  const int kt = bid % p.k_tiles;
  bid /= p.k_tiles;
  const int g = bid % p.Hkv;
  const int chunk = bid / p.Hkv;
  const int nw = p.n_win * p.G;                         // window rows of this group
  const int nwp = (nw + 15) & ~15;                      // padded to the MMA N granule
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(nwp)) tmem_cols <<= 1;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* k_tile = smem;                               // [128 keys x D], D/64 panels
  uint8_t* q_tile = smem + 128 * D * 2;                 // [nwp rows x D], panels of nwp*128 B
  const uint32_t q_panel = static_cast<uint32_t>(nwp) * 128u;

  if (warp >= 1) {
    // Padding rows of the window tile are never loaded: keep them zero.
    const int ts = tid - 32;
    for (int idx = ts; idx < (nwp - nw) * (D / 8); idx += 128) {
      const int n = nw + idx / (D / 8), c = idx % (D / 8);
      *reinterpret_cast<uint4*>(q_tile + sw128_offset(n, c * 8, nwp)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    for (int n = ts; n < nwp; n += 128) {
      float b = INFINITY;  // padding columns contribute exp2(-inf) = 0
      if (n < nw) {
        const int w = n / p.G, jj = n - w * p.G;
        const long long idx = (static_cast<long long>(chunk) * p.Hq + g * p.G + jj) * p.n_win + w;
        const float l = p.win_l[idx];
        b = l > 0.0f ? p.win_m[idx] + log2f(l) : INFINITY;
      }
      b_sh[n] = b;
    }
  } else if (lane == 0) {
    mbar_init(&bar_k, 1);
    mbar_init(&bar_mma[0], 1);
    mbar_init(&bar_mma[1], 1);
    fence_barrier_init();
    failed = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int n_chunks_n = (nwp + 255) / 256;

  if (warp == 0) {
    if (lane == 0) {
      // K rows of this tile (rows past the chunk are loaded but never written
      // out) and the group's window rows, one box per 64-column panel each.
      const uint32_t bytes = 128u * D * 2u + static_cast<uint32_t>(nw) * D * 2u;
      mbar_arrive_expect_tx(&bar_k, bytes);
      const int row0 = chunk * p.chunk_rows + kt * 128;
      for (int pn = 0; pn < D / 64; ++pn) {
        tma_load_3d(k_tile + pn * kPanelBytes, &p.tm_k, &bar_k, pn * 64, g, row0);
        tma_load_3d(q_tile + pn * q_panel, &p.tm_qwin, &bar_k, pn * 64, g * p.G, 0);
      }
      bool ok = mbar_wait(&bar_k, 0);
      tc_fence_after_sync();
      const uint32_t ka = smem_u32(k_tile), qa = smem_u32(q_tile);
      for (int nc = 0; ok && nc < n_chunks_n; ++nc) {
        const int n0 = nc * 256;
        const int nn = min(256, nwp - n0);
        const uint32_t idesc = idesc_bf16(128, nn, false, false);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sw128_desc(ka + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t b =
              sw128_desc(qa + (kk >> 2) * q_panel + n0 * 128 + (kk & 3) * 32, 16, 1024);
          mma_bf16_ss(tmem + n0, a, b, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_mma[nc]);
      }
      if (!ok) {
        atomicOr(&failed, 1);
        // Nothing was issued; release the consumers.
        mbar_arrive(&bar_mma[0]);
        mbar_arrive(&bar_mma[1]);
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    for (int nc = 0; nc < n_chunks_n; ++nc) {
      if (!mbar_wait_warp(&bar_mma[nc], 0)) { ok = false; break; }
      tc_fence_after_sync();
      const int n0 = nc * 256;
      const int nn = min(256, nwp - n0);
      for (int cc = 0; cc < nn; cc += 32) {
        uint32_t s[32];
        tmem_ld32(lane_base + n0 + cc, s);
        tmem_ld_wait(s);
        const float4* b4 = reinterpret_cast<const float4*>(b_sh + n0 + cc);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (n0 + cc + 4 * i < nwp) {
            const float4 b = b4[i];
            acc[0] += ex2_approx(fmaf(__uint_as_float(s[4 * i + 0]), p.scale_log2, -b.x));
            acc[1] += ex2_approx(fmaf(__uint_as_float(s[4 * i + 1]), p.scale_log2, -b.y));
            acc[2] += ex2_approx(fmaf(__uint_as_float(s[4 * i + 2]), p.scale_log2, -b.z));
            acc[3] += ex2_approx(fmaf(__uint_as_float(s[4 * i + 3]), p.scale_log2, -b.w));
          }
        }
      }
    }
    if (!ok) atomicOr(&failed, 2);
    const int t = kt * 128 + row;
    if (t < p.chunk_rows)
      p.part_scores[(static_cast<long long>(chunk) * p.Hkv + g) * p.chunk_rows + t] =
          (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && failed) raise_dev_err(p.dev_err, PFD_DEVERR_TIMEOUT);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

cudaError_t launch_window_scores(const WinScoreParams& p, cudaStream_t stream) {
  const int grid = p.n_chunks * p.Hkv * p.k_tiles;
  if (grid <= 0 || p.n_win <= 0) return cudaSuccess;
  const int nwp = (p.n_win * p.G + 15) & ~15;
  const size_t smem = 1024 + static_cast<size_t>(128 + nwp) * p.D * 2;
  cudaError_t err;
  if (p.D == 64) {
    err = ensure_smem_limit(reinterpret_cast<const void*>(window_score_kernel<64>), static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(window_score_kernel<64>, dim3(grid), dim3(kThreads), smem, stream, p);
  } else {
    err = ensure_smem_limit(reinterpret_cast<const void*>(window_score_kernel<128>), static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(window_score_kernel<128>, dim3(grid), dim3(kThreads), smem, stream, p);
  }
  return cudaGetLastError();
}

}  // namespace pfd
