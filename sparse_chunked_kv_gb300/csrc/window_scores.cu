// Cumulative attention weight each chunk row receives from the query window
// ("Two-Level Sparsity", intra-chunk ranking of the Prefilling-dLLM summary).
//
// score[j][t] = sum over window rows w and query heads h of
//               softmax over the C+1 rows of chunk j of (scale * q_win[w,h] . k[t,g]).
//
// The attention kernel has already produced, for every (chunk, head, window
// row), the constant b = m + log2(l) of that row's softmax over the chunk (m
// the row maximum in log2 units, l the denominator), so p = 2^(s*scale - b).  This kernel
// recomputes the logits transposed -- S^T = K Q_win^T with the 128 key rows of
// one tile on the TMEM lanes and the W*G window rows of one KV group on the
// TMEM columns -- so each thread owns one key and sums exp2(scale*s - b_n)
// along its TMEM row with no cross-thread reduction.  The result is one
// partial score per KV group; the top-B kernel adds the Hkv partials in a
// fixed order.
//
// The kernel is persistent: CTA c serves KV group c % Hkv of one layer (of
// several stacked layers, each with its own window rows), loads that group's
// window rows once and streams that layer's 128-row K tiles through a
// two-slot ring.  When
// a chunk has at least 128 rows the tiles run over the chunks' rows laid end to
// end (a tile then spans at most two chunks, so no tile is mostly padding);
// otherwise each tile is a piece of one chunk.  S^T is split into two column
// halves in TMEM so the tensor core computes one half while the warps
// exponentiate the other.
//   warp 0      TMA loads and the single-thread MMA issuer;
//   warps 1..16 four warps per TMEM lane quarter (one thread per key row), each
//               taking every fourth 32-column piece of every half; their four
//               partial sums are added in a fixed order.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kSubs = kConsumerWarps / 4;        // consumer warps per lane quarter
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr uint32_t kPanelBytes = 128u * 128u;   // a 128-row, 64-column K panel
constexpr int kMaxWindowRows = 512;
constexpr uint32_t kConsumerBarrier = 1;         // named barrier of warps 1..16

// Rows [row0, row0 + nrows) of the concatenated chunks, starting in chunk c0.
struct Tile {
  long long row0;
  int nrows;
  int c0;
};

__device__ __forceinline__ Tile tile_of(const WinScoreParams& p, int i) {
  Tile t;
  const long long total = static_cast<long long>(p.n_chunks) * p.chunk_rows;
  if (p.concat) {
    t.row0 = static_cast<long long>(i) * 128;
    t.nrows = static_cast<int>(min(128ll, total - t.row0));
    t.c0 = static_cast<int>(t.row0 / p.chunk_rows);
  } else {
    const int chunk = i / p.k_tiles, kt = i % p.k_tiles;
    t.row0 = static_cast<long long>(chunk) * p.chunk_rows + kt * 128;
    t.nrows = min(128, p.chunk_rows - kt * 128);
    t.c0 = chunk;
  }
  return t;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
window_score_kernel(const __grid_constant__ WinScoreParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, k_full[2], k_empty[2], s_full[2], s_free[2];
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  __shared__ __align__(16) float b_sh[2][2][kMaxWindowRows];   // [item parity][chunk of tile][column]
  __shared__ float red[2][kSubs - 1][128];   // partials of warps sub = 1.. per key row

  grid_dependency_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA -> (KV group g, layer, index among the CTAs of that pair).
  const int g = blockIdx.x % p.Hkv;
  const int layer = (blockIdx.x / p.Hkv) % p.n_layers;
  const int cta_g = blockIdx.x / (p.Hkv * p.n_layers);
  const int n_cta_g = gridDim.x / (p.Hkv * p.n_layers);
  const long long layer_row0 = static_cast<long long>(layer) * p.n_chunks * p.chunk_rows;
  const long long layer_chunk0 = static_cast<long long>(layer) * p.n_chunks;
  const int nw = p.n_win * p.G;          // window rows of this group (TMEM columns)
  const int nwp = (nw + 31) & ~31;       // padded: two halves of a multiple of 16
  const int half = nwp / 2;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(nwp)) tmem_cols <<= 1;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_tile = smem;                                   // [nwp rows x D], panels of nwp*128 B
  const uint32_t q_panel = static_cast<uint32_t>(nwp) * 128u;
  uint8_t* k_ring = smem + ((static_cast<uint32_t>(nwp) * D * 2 + 1023) & ~1023u);   // 2 x [128 x D]
  constexpr uint32_t kKBytes = 128u * D * 2u;

  // b of chunk c, column n (n = w*G + j); padding and missing chunks get +inf
  // (2^(s - inf) = 0).
  auto b_src = [&](int c, int n) -> const float* {
    if (c >= p.n_chunks || n >= nw) return nullptr;
    return p.win_b + ((layer_chunk0 + c) * p.Hkv + g) * p.win_stride + n;
  };
  const int n_items = p.n_items;

  if (warp == 0) {
    if (lane == 0) {
      mbar_init(&q_full, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&k_full[i], 1);
        mbar_init(&k_empty[i], 1);
        mbar_init(&s_full[i], 1);
        mbar_init(&s_free[i], kConsumerWarps);
      }
      fence_barrier_init();
      failed = 0;
    }
    tmem_alloc(&tmem_base, tmem_cols);
    tmem_relinquish();
  } else {
    // Padding rows of the window tile are never loaded: keep them zero.
    const int ts = tid - 32;
    for (int idx = ts; idx < (nwp - nw) * (D / 8); idx += kConsumers) {
      const int n = nw + idx / (D / 8), c = idx % (D / 8);
      *reinterpret_cast<uint4*>(q_tile + sw128_offset(n, c * 8, nwp)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    // Statistics of the first tile.
    if (cta_g < n_items) {
      const Tile t0 = tile_of(p, cta_g);
      for (int idx = ts; idx < 2 * nwp; idx += kConsumers) {
        const float* src = b_src(t0.c0 + idx / nwp, idx % nwp);
        b_sh[0][idx / nwp][idx % nwp] = src != nullptr ? *src : INFINITY;
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(&q_full, static_cast<uint32_t>(nw) * D * 2u);
      for (int pn = 0; pn < D / 64; ++pn)
        tma_load_3d(q_tile + pn * q_panel, &p.tm_qwin, &q_full, pn * 64, g * p.G,
                    layer * p.n_win);
      auto load_k = [&](int k, int i) {
        const int slot = k & 1;
        mbar_arrive_expect_tx(&k_full[slot], kKBytes);
        const Tile t = tile_of(p, i);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d(k_ring + slot * kKBytes + pn * kPanelBytes, &p.tm_k, &k_full[slot], pn * 64, g,
                      static_cast<int>(layer_row0 + t.row0));
      };
      int k = 0;
      if (cta_g < n_items) load_k(0, cta_g);
      if (cta_g + n_cta_g < n_items) load_k(1, cta_g + n_cta_g);
      ok = mbar_wait(&q_full, 0);
      tc_fence_after_sync();
      const uint32_t qa = smem_u32(q_tile);
      for (int i = cta_g; ok && i < n_items; i += n_cta_g, ++k) {
        const int slot = k & 1;
        if (!mbar_wait(&k_full[slot], (k >> 1) & 1)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t ka = smem_u32(k_ring + slot * kKBytes);
        for (int hf = 0; hf < 2; ++hf) {
          // The warps have finished this half of the previous tile.
          if (k > 0 && !mbar_wait(&s_free[hf], (k - 1) & 1)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t idesc = idesc_bf16(128, half, false, false);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = sw128_desc(ka + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t b =
                sw128_desc(qa + (kk >> 2) * q_panel + hf * half * 128 + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(tmem + hf * half, a, b, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[hf]);
        }
        if (!ok) break;
        mma_commit(&k_empty[slot]);
        // The slot is refilled with the tile two ahead once these MMAs are done.
        const int i2 = i + 2 * n_cta_g;
        if (i2 < n_items) {
          if (!mbar_wait(&k_empty[slot], (k >> 1) & 1)) { ok = false; break; }
          load_k(k + 2, i2);
        }
      }
      if (!ok) atomicOr(&failed, 1);
      // Loads still in flight land before the CTA exits.
      const int n_mine = cta_g < n_items ? (n_items - 1 - cta_g) / n_cta_g + 1 : 0;
      for (int kk = max(0, n_mine - 2); kk < n_mine; ++kk) mbar_wait(&k_full[kk & 1], (kk >> 1) & 1);
    }
  } else {
    const int quarter = warp & 3;
    const int sub = (warp - 1) >> 2;   // 0 for warps 1..4, 1 for warps 5..8, ...
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
    const int pieces = (half + 31) / 32;
    bool ok = true;
    int k = 0;
    for (int i = cta_g; i < n_items; i += n_cta_g, ++k) {
      const Tile t = tile_of(p, i);
      const long long r = t.row0 + row;
      const int c_row = static_cast<int>(r / p.chunk_rows);
      const float* bv = b_sh[k & 1][min(c_row - t.c0, 1)];
      // Statistics of the next tile, copied asynchronously into the other
      // buffer while this tile is processed (the buffer's last reader was the
      // tile before this one, which every consumer has finished).
      const int i_next = i + n_cta_g;
      if (i_next < n_items) {
        const Tile tn = tile_of(p, i_next);
        for (int idx = tid - 32; idx < 2 * nwp; idx += kConsumers) {
          float* dst = &b_sh[(k + 1) & 1][idx / nwp][idx % nwp];
          const float* src = b_src(tn.c0 + idx / nwp, idx % nwp);
          if (src != nullptr) cp_async_4(dst, src);
          else *dst = INFINITY;
        }
        cp_async_commit();
      }
      uint64_t acc2 = f2_pack(0.f, 0.f);
      for (int hf = 0; hf < 2; ++hf) {
        if (ok && !mbar_wait_warp(&s_full[hf], k & 1)) ok = false;
        tc_fence_after_sync();
        if (ok) {
          for (int pc = sub; pc < pieces; pc += kSubs) {
            const int c0 = hf * half + pc * 32;
            uint32_t s[32];
            tmem_ld32(lane_base + c0, s);
            tmem_ld_wait(s);
            const int ncols = min(32, (hf + 1) * half - c0);
#pragma unroll
            for (int q = 0; q < 32; q += 2) {
              if (q < ncols) {
                const float2 b = *reinterpret_cast<const float2*>(bv + c0 + q);
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(s[q]), __uint_as_float(s[q + 1])), scale2,
                                 f2_pack(-b.x, -b.y)),
                          x0, x1);
                acc2 = f2_add(acc2, f2_pack(ex2_approx(x0), ex2_approx(x1)));
              }
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[hf]);
      }
      float a0, a1;
      f2_unpack(acc2, a0, a1);
      const float acc = a0 + a1;
      if (i_next < n_items) cp_async_wait_all();
      if (sub > 0) red[k & 1][sub - 1][row] = acc;
      named_barrier_sync(kConsumerBarrier, kConsumers);
      if (sub == 0 && row < t.nrows && c_row < p.n_chunks) {
        const int tt = static_cast<int>(r - static_cast<long long>(c_row) * p.chunk_rows);
        float total = acc;
#pragma unroll
        for (int u = 0; u < kSubs - 1; ++u) total += red[k & 1][u][row];
        p.part_scores[((layer_chunk0 + c_row) * p.Hkv + g) * p.chunk_rows + tt] = total;
      }
    }
    if (!ok) atomicOr(&failed, 2);
  }
  tc_fence_before_sync();
  __syncthreads();
  grid_dependents_launch();
  if (tid == 0 && failed) raise_dev_err(p.dev_err, PFD_DEVERR_TIMEOUT);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

cudaError_t launch_window_scores(const WinScoreParams& p, cudaStream_t stream) {
  if (p.n_items <= 0 || p.n_win <= 0) return cudaSuccess;
  const int nwp = (p.n_win * p.G + 31) & ~31;
  if (nwp > kMaxWindowRows) return cudaErrorInvalidValue;
  int sms = 0, dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int pairs = p.Hkv * std::max(1, p.n_layers);   // (KV group, layer) pairs
  const int per_g = std::max(1, std::min(sms / pairs, p.n_items));
  const int grid = per_g * pairs;
  const size_t smem =
      1024 + ((static_cast<size_t>(nwp) * p.D * 2 + 1023) & ~static_cast<size_t>(1023)) +
      2 * 128 * static_cast<size_t>(p.D) * 2;
  if (p.D == 64) {
    err = ensure_smem_limit(reinterpret_cast<const void*>(window_score_kernel<64>), static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(window_score_kernel<64>, dim3(grid), dim3(kThreads), smem, stream, p);
  }
  err = ensure_smem_limit(reinterpret_cast<const void*>(window_score_kernel<128>), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(window_score_kernel<128>, dim3(grid), dim3(kThreads), smem, stream, p);
}

// Each window row's log-sum-exp over the window's own W keys, for the reading
// of "Two-Level Sparsity" in which a window row's softmax runs over the
// chunk's keys and the window keys together:
//   b_self[w][h] = log2 sum_{w'} 2^(x_{w'}),  x = sm_scale log2(e) q_{w,h} . k_win_{w',g}.
// One warp per (w, h): the query row is staged in shared memory, lane l
// takes keys l, l + 32, ... (W <= 256: at most 8) and computes their whole
// dot products with 16-byte loads, all in flight together; then one
// (max, sum) reduction over the warp.  Once per prefill call.
__global__ void __launch_bounds__(128)
window_self_stats_kernel(const bf16* __restrict__ q_win, const bf16* __restrict__ k_win, int W,
                         int Hq, int Hkv, int D, float scale_log2, float* __restrict__ b_self) {
  __shared__ float q_sh[4][128];
  grid_dependency_wait();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const long long pair = static_cast<long long>(blockIdx.x) * 4 + wib;
  const bool live = pair < static_cast<long long>(W) * Hq;
  const int w = live ? static_cast<int>(pair / Hq) : 0, h = live ? static_cast<int>(pair % Hq) : 0;
  const int g = h / (Hq / Hkv);
  const uint16_t* q = reinterpret_cast<const uint16_t*>(q_win) + (static_cast<long long>(w) * Hq + h) * D;
  for (int e = lane; e < D; e += 32)
    q_sh[wib][e] = live ? __uint_as_float(static_cast<uint32_t>(q[e]) << 16) : 0.0f;
  __syncwarp();
  float m = -INFINITY, l = 0.0f;
  if (live) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k2 = lane + 32 * i;
      x[i] = -INFINITY;
      if (k2 < W) {
        const uint4* k = reinterpret_cast<const uint4*>(k_win) +
                         ((static_cast<long long>(k2) * Hkv + g) * D) / 8;
        float dot = 0.0f;
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint4 kv = __ldg(k + c8);
          const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dot = fmaf(q_sh[wib][c8 * 8 + 2 * j], __uint_as_float(kw[j] << 16), dot);
            dot = fmaf(q_sh[wib][c8 * 8 + 2 * j + 1], __uint_as_float(kw[j] & 0xFFFF0000u), dot);
          }
        }
        x[i] = dot * scale_log2;
      }
      m = fmaxf(m, x[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (x[i] != -INFINITY) l += ex2_approx(x[i] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
    if (lane == 0) b_self[pair] = m + log2f(l);
  }
  grid_dependents_launch();
}

cudaError_t launch_window_self_stats(const bf16* q_win, const bf16* k_win, int W, int Hq, int Hkv,
                                     int D, float scale_log2, float* b_self, cudaStream_t stream) {
  const long long pairs = static_cast<long long>(W) * Hq;
  if (pairs <= 0) return cudaSuccess;
  return launch_pdl(window_self_stats_kernel, dim3(static_cast<unsigned>((pairs + 3) / 4)),
                    dim3(128), 0, stream, q_win, k_win, W, Hq, Hkv, D, scale_log2, b_self);
}

}  // namespace pfd
