// Bidirectional softmax attention of 128-row query tiles over a list of key
// segments, on tcgen05 tensor cores with TMA-fed K/V tiles.
//
// One kernel serves three kinds of work item:
//   chunk   (prefill)  rows of chunk j attend to chunk j's own C+1 rows
//                      ("Chunked Prefill and KV Caching": each BOS-prefixed
//                      chunk is processed on its own, bidirectionally);
//   window  (prefill)  query-window rows against chunk j, statistics only
//                      (row max and softmax denominator), consumed by the
//                      window-score kernel ("Two-Level Sparsity", ranking by
//                      cumulative attention weight from the query tokens);
//   decode             live rows of one sequence against one contiguous range
//                      of [selected chunks' pool slots ; live rows], read in
//                      place through the chunk table ("Decoding with Static KV
//                      Reuse"; split-KV with log-sum-exp merge from "Attention
//                      Kernel Optimization").
//
// Warp roles (192 threads):
//   warp 0      TMA producer: walks the key segments in 16-row groups and
//               loads K (and V) tiles of 8 groups into a 2-stage ring.
//   warp 1      allocates TMEM and issues all tcgen05.mma from one thread:
//               S = Q K^T into one of two TMEM S buffers, O += P V into TMEM.
//   warps 2..5  one thread per query row (= TMEM lane): masked row max, exp2,
//               bf16 P into shared memory, rescale of O in TMEM only when the
//               running max grows by more than 2^8, and the epilogue.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint32_t kPanelBytes = 128u * 128u;  // 128 rows x 128 B
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t tmem_s(int st) { return st ? 128u : 0u; }
constexpr uint32_t kTmemO = 256u;
constexpr float kLn2 = 0.69314718055994530942f;

enum ItemKind : int { kChunk = 0, kWindow = 1, kDecode = 2 };

struct TileMeta {
  uint32_t nvalid_lo;  // valid rows of groups 0..3, one byte each
  uint32_t nvalid_hi;  // groups 4..7
  int32_t ngroups;
  int32_t pad;
};

struct Shared {
  uint64_t qfull;
  uint64_t kfull[2], vfull[2], kvempty[2];
  uint64_t sfull[2], sempty[2];
  uint64_t pfull[2], pvdone[2];
  uint64_t drain;
  TileMeta meta[2];
  uint32_t tmem_base;
  int32_t g_lo, g_hi, n_tiles;
  int32_t failed;
};

struct Item {
  int kind;
  int g, mt;
  const bf16* qsrc;
  long long q_row0;   // token row of t = 0 in qsrc (and in the output)
  int n_t;            // tokens in this item's query block
  int chunk;          // prefill
  int seq, split;     // decode
  int k0, k1;         // decode: selected-chunk range in sel
};

struct Segment {
  int tensor;
  long long row;
  int len;
};

// Segment i of an item's key sequence.
__device__ __forceinline__ Segment get_segment(const AttnParams& p, const Item& it, int i) {
  Segment s;
  if (it.kind != kDecode) {
    s.tensor = 0;
    s.row = static_cast<long long>(it.chunk) * p.chunk_rows;
    s.len = p.chunk_rows;
    return s;
  }
  const int n_sel = it.k1 - it.k0;
  if (i < n_sel) {
    const int c = p.sel[it.k0 + i];
    s.tensor = 0;
    s.row = 0;
    s.len = 0;
    if (c < 0 || c >= p.table_len) {
      raise_dev_err(p.dev_err, PFD_DEVERR_SEL);
      return s;
    }
    const pfd_chunk_entry e = p.table[c];
    if (e.row < 0 || e.len < 0 || static_cast<long long>(e.row) + e.len > p.pool_rows) {
      raise_dev_err(p.dev_err, PFD_DEVERR_TABLE);
      return s;
    }
    s.row = e.row;
    s.len = e.len;
    return s;
  }
  s.tensor = 1;
  s.row = it.q_row0;
  s.len = it.n_t;
  return s;
}

__device__ __forceinline__ int num_segments(const Item& it) {
  return it.kind == kDecode ? (it.k1 - it.k0 + 1) : 1;
}

__device__ __forceinline__ int groups_of(int len) { return (len + kGroupRows - 1) / kGroupRows; }

// Resolves blockIdx.x into a work item; returns false when the CTA has no work.
__device__ __forceinline__ bool resolve_item(const AttnParams& p, Item& it) {
  int bid = blockIdx.x;
  if (p.mode == kModePrefill) {
    if (bid < p.n_chunk_items) {
      it.kind = kChunk;
      it.mt = bid % p.mt_chunk;
      bid /= p.mt_chunk;
      it.qsrc = p.q;
      it.n_t = p.chunk_rows;
    } else {
      bid -= p.n_chunk_items;
      it.kind = kWindow;
      it.mt = bid % p.mt_win;
      bid /= p.mt_win;
      it.qsrc = p.q_win;
      it.n_t = p.n_win;
    }
    it.g = bid % p.Hkv;
    it.chunk = bid / p.Hkv;
    it.q_row0 = it.kind == kChunk ? static_cast<long long>(it.chunk) * p.chunk_rows : 0;
    it.seq = 0;
    it.split = 0;
    it.k0 = it.k1 = 0;
    return it.mt * kBlockM < it.n_t * p.G;
  }
  it.kind = kDecode;
  it.mt = bid % p.mt_max;
  bid /= p.mt_max;
  it.split = bid % p.n_splits;
  bid /= p.n_splits;
  it.g = bid % p.Hkv;
  it.seq = bid / p.Hkv;
  it.qsrc = p.q;
  it.chunk = 0;
  const int lq0 = p.cu_lq[it.seq], lq1 = p.cu_lq[it.seq + 1];
  const int k0 = p.cu_k[it.seq], k1 = p.cu_k[it.seq + 1];
  if (lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq || k0 < 0 || k1 < k0 || k1 > p.total_sel) {
    if (threadIdx.x == 0) raise_dev_err(p.dev_err, PFD_DEVERR_SHAPE);
    return false;
  }
  it.q_row0 = lq0;
  it.n_t = lq1 - lq0;
  it.k0 = k0;
  it.k1 = k1;
  return it.mt * kBlockM < it.n_t * p.G;
}

template <int D>
struct Layout {
  static constexpr uint32_t kQBytes = kBlockM * D * 2;
  static constexpr uint32_t kKVBytes = kBlockN * D * 2;
  static constexpr uint32_t kPBytes = kBlockM * kBlockN * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK0 = kQ + kQBytes;
  static constexpr uint32_t kV0 = kK0 + kKVBytes;
  static constexpr uint32_t kK1 = kV0 + kKVBytes;
  static constexpr uint32_t kV1 = kK1 + kKVBytes;
  static constexpr uint32_t kP0 = kV1 + kKVBytes;
  static constexpr uint32_t kP1 = kP0 + kPBytes;
  static constexpr uint32_t kTotal = kP1 + kPBytes;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attention_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;

  Item it;
  if (!resolve_item(p, it)) return;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool with_pv = it.kind != kWindow;

  if (tid == 0) {
    mbar_init(&sh.qfull, kSoftmaxThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.kfull[i], 1);
      mbar_init(&sh.vfull[i], 1);
      mbar_init(&sh.kvempty[i], 1);
      mbar_init(&sh.sfull[i], 1);
      mbar_init(&sh.sempty[i], kSoftmaxThreads);
      mbar_init(&sh.pfull[i], kSoftmaxThreads);
      mbar_init(&sh.pvdone[i], 1);
    }
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
    // Group range of this item's split.
    const int nseg = num_segments(it);
    long long total = 0;
    for (int i = 0; i < nseg; ++i) total += groups_of(get_segment(p, it, i).len);
    const int n_splits = it.kind == kDecode ? p.n_splits : 1;
    const long long lo = total * it.split / n_splits;
    const long long hi = total * (it.split + 1) / n_splits;
    sh.g_lo = static_cast<int>(lo);
    sh.g_hi = static_cast<int>(hi);
    sh.n_tiles = static_cast<int>((hi - lo + kGroupsPerTile - 1) / kGroupsPerTile);
    sh.failed = 0;
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem = sh.tmem_base;
  const int n_tiles = sh.n_tiles;
  const int g_lo = sh.g_lo, g_hi = sh.g_hi;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&p.tm_k[0]);
      const int nseg = num_segments(it);
      int seg = 0, gofs = 0;
      {
        long long acc = 0;
        for (; seg < nseg; ++seg) {
          const int n = groups_of(get_segment(p, it, seg).len);
          if (acc + n > g_lo) {
            gofs = static_cast<int>(g_lo - acc);
            break;
          }
          acc += n;
        }
      }
      Segment cur = get_segment(p, it, seg < nseg ? seg : 0);
      int g_cur = g_lo;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&sh.kvempty[st], ((j >> 1) - 1) & 1)) {
          atomicOr(&sh.failed, 1);
          break;
        }
        int tens[kGroupsPerTile];
        int rows[kGroupsPerTile];
        uint32_t nv_lo = 0, nv_hi = 0;
        int ng = 0;
        for (; ng < kGroupsPerTile && g_cur < g_hi; ++ng, ++g_cur) {
          const int nv = min(kGroupRows, cur.len - gofs * kGroupRows);
          tens[ng] = cur.tensor;
          rows[ng] = static_cast<int>(cur.row) + gofs * kGroupRows;
          if (ng < 4) nv_lo |= static_cast<uint32_t>(nv) << (8 * ng);
          else nv_hi |= static_cast<uint32_t>(nv) << (8 * (ng - 4));
          ++gofs;
          if (gofs * kGroupRows >= cur.len) {
            gofs = 0;
            ++seg;
            while (seg < nseg) {
              cur = get_segment(p, it, seg);
              if (cur.len > 0) break;
              ++seg;
            }
          }
        }
        sh.meta[st].nvalid_lo = nv_lo;
        sh.meta[st].nvalid_hi = nv_hi;
        sh.meta[st].ngroups = ng;
        const uint32_t bytes = static_cast<uint32_t>(ng) * kGroupRows * D * 2;
        const uint32_t k_dst = s_base + (st ? L::kK1 : L::kK0);
        const uint32_t v_dst = s_base + (st ? L::kV1 : L::kV0);
        mbar_arrive_expect_tx(&sh.kfull[st], bytes);
        for (int k = 0; k < ng; ++k)
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + (k_dst - s_base) + pn * kPanelBytes + k * 2048, &p.tm_k[tens[k]],
                        &sh.kfull[st], pn * 64, it.g, rows[k]);
        if (with_pv) {
          mbar_arrive_expect_tx(&sh.vfull[st], bytes);
          for (int k = 0; k < ng; ++k)
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d(smem + (v_dst - s_base) + pn * kPanelBytes + k * 2048,
                          &p.tm_v[tens[k]], &sh.vfull[st], pn * 64, it.g, rows[k]);
        }
      }
      // Drain: the last tiles' loads must have landed before the CTA exits.
      for (int j = max(0, n_tiles - 2); j < n_tiles; ++j) {
        mbar_wait(&sh.kfull[j & 1], (j >> 1) & 1);
        if (with_pv) mbar_wait(&sh.vfull[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(&sh.qfull, 0);
      tc_fence_after_sync();
      const uint32_t q_addr = s_base + L::kQ;
      auto issue_pv = [&](int i) -> bool {
        const int b = i & 1;
        if (!mbar_wait(&sh.pfull[b], (i >> 1) & 1)) return false;
        if (with_pv) {
          if (!mbar_wait(&sh.vfull[b], (i >> 1) & 1)) return false;
          tc_fence_after_sync();
          const int ng = min(sh.meta[b].ngroups, kGroupsPerTile);
          const uint32_t p_addr = s_base + (b ? L::kP1 : L::kP0);
          const uint32_t v_addr = s_base + (b ? L::kV1 : L::kV0);
          constexpr uint32_t idesc = idesc_bf16(kBlockM, D, false, true);
          for (int kk = 0; kk < ng; ++kk) {
            const uint64_t a = sw128_desc(p_addr + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t v = sw128_desc(v_addr + kk * 2048, kPanelBytes, 1024);
            mma_bf16_ss(tmem + kTmemO, a, v, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&sh.pvdone[b]);
        mma_commit(&sh.kvempty[b]);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&sh.kfull[st], (j >> 1) & 1)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&sh.sempty[st], ((j >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after_sync();
        const int ng = min(sh.meta[st].ngroups, kGroupsPerTile);
        const uint32_t idesc = idesc_bf16(kBlockM, max(ng, 1) * kGroupRows, false, false);
        const uint32_t k_addr = s_base + (st ? L::kK1 : L::kK0);
#pragma unroll
        for (int kk = 0; kk < (ng > 0 ? D / 16 : 0); ++kk) {
          const uint64_t a = sw128_desc(q_addr + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sw128_desc(k_addr + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
          mma_bf16_ss(tmem + tmem_s(st), a, b, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sh.sfull[st]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) atomicOr(&sh.failed, 2);
      // Every MMA issued above has completed once `drain` flips.
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0);
    }
  } else {
    // ---------------------------------------------- softmax + epilogue --
    const int ts = tid - 64;              // 0..127
    const int quarter = warp & 3;         // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;  // tile row of this thread
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int n_rows = it.n_t * p.G;

    if (n_tiles > 0) {
      // Q tile -> shared memory, 128-byte swizzled K-major panels.
      constexpr int kChunks = D / 8;
      for (int idx = ts; idx < kBlockM * kChunks; idx += kSoftmaxThreads) {
        const int r = idx / kChunks, c = idx % kChunks;
        const int m = it.mt * kBlockM + r;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (m < n_rows) {
          const int t = m / p.G, jj = m - t * p.G;
          const bf16* src = it.qsrc + ((it.q_row0 + t) * p.Hq + it.g * p.G + jj) * D + c * 8;
          val = __ldg(reinterpret_cast<const uint4*>(src));
        }
        *reinterpret_cast<uint4*>(smem + L::kQ + sw128_offset(r, c * 8, kBlockM)) = val;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh.qfull);
    }

    float m_used = -INFINITY;
    float l_sum = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!mbar_wait_warp(&sh.sfull[st], ph) || !mbar_wait_warp(&sh.kfull[st], ph)) { ok = false; break; }
      tc_fence_after_sync();
      const TileMeta meta = sh.meta[st];
      const int ncol = meta.ngroups * kGroupRows;
      const bool full = meta.ngroups == kGroupsPerTile && meta.nvalid_lo == 0x10101010u &&
                        meta.nvalid_hi == 0x10101010u;

      uint32_t s0[32], s1[32], s2[32], s3[32];
      const uint32_t s_addr = lane_base + tmem_s(st);
      tmem_ld32(s_addr + 0, s0);
      if (ncol > 32) tmem_ld32(s_addr + 32, s1);
      if (ncol > 64) tmem_ld32(s_addr + 64, s2);
      if (ncol > 96) tmem_ld32(s_addr + 96, s3);
      tmem_ld_wait(s0);
      reg_fence(s1);
      reg_fence(s2);
      reg_fence(s3);
      tc_fence_before_sync();
      mbar_arrive(&sh.sempty[st]);

      // Masked logits: a column is valid when its row exists in its group.
      auto nv_of = [&](int grp) -> int {
        const uint32_t w = grp < 4 ? meta.nvalid_lo : meta.nvalid_hi;
        return static_cast<int>((w >> (8 * (grp & 3))) & 0xFFu);
      };
      float x[128];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = __uint_as_float(s0[i]);
        x[32 + i] = __uint_as_float(s1[i]);
        x[64 + i] = __uint_as_float(s2[i]);
        x[96 + i] = __uint_as_float(s3[i]);
      }
      if (!full) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if ((c & 15) >= nv_of(c >> 4)) x[c] = -INFINITY;
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) tmax = fmaxf(tmax, x[c]);
      const float m_tile = tmax * p.scale_log2;

      // P buffer st was read by PV(j-2).
      if (j >= 2 && !mbar_wait_warp(&sh.pvdone[st], ((j >> 1) - 1) & 1)) { ok = false; break; }
      // Rescale decision per row; the TMEM rescale itself is warp-collective,
      // so a warp rescales when any of its rows needs it (alpha = 1 elsewhere).
      const bool mine = m_tile > m_used + kRescaleThreshold;
      if (__any_sync(0xFFFFFFFFu, mine)) {
        const float m_new = mine ? m_tile : m_used;
        const float alpha = mine ? ex2_approx(m_used - m_new) : 1.0f;
        if (j >= 1 && with_pv) {
          // O holds tiles 0..j-1 relative to the old max: rescale it in TMEM
          // once PV(j-1) has landed.
          if (!mbar_wait_warp(&sh.pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(lane_base + kTmemO + ch * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + kTmemO + ch * 32, o);
          }
          tmem_st_wait();
        }
        l_sum *= alpha;
        m_used = m_new;
      }

      // Probabilities (relative to m_used) -> bf16 P tile, row sum in fp32.
      const float neg_m = -m_used;
      float part = 0.0f;
      uint8_t* p_tile = smem + (st ? L::kP1 : L::kP0);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = ex2_approx(fmaf(x[ch * 32 + 2 * i], p.scale_log2, neg_m));
          const float b = ex2_approx(fmaf(x[ch * 32 + 2 * i + 1], p.scale_log2, neg_m));
          part += a + b;
          packed[i] = pack_bf16x2(a, b);
        }
        if (with_pv && ch * 32 < ncol) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint32_t off = sw128_offset(row, ch * 32 + q4 * 8, kBlockM);
            *reinterpret_cast<uint4*>(p_tile + off) =
                make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
          }
        }
      }
      l_sum += part;

      if (with_pv && !full) {
        // Rows of a ragged group that lie past its segment may hold anything
        // (another slot, padding): zero them in V so that 0 * v stays 0.
        if (!mbar_wait_warp(&sh.vfull[st], ph)) { ok = false; break; }
        uint8_t* v_tile = smem + (st ? L::kV1 : L::kV0);
        for (int grp = 0; grp < meta.ngroups; ++grp) {
          const int nv = nv_of(grp);
          const int n_bad = (kGroupRows - nv) * (D / 64) * 8;  // 16-byte chunks to clear
          for (int u = ts; u < n_bad; u += kSoftmaxThreads) {
            const int c16 = u & 7;
            const int rest = u >> 3;
            const int pn = rest % (D / 64);
            const int r = nv + rest / (D / 64);
            *reinterpret_cast<uint4*>(v_tile + pn * kPanelBytes + (grp * kGroupRows + r) * 128 +
                                      c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&sh.pfull[st]);
    }

    // ------------------------------------------------------------ epilogue --
    if (ok && n_tiles > 0 &&
        !mbar_wait_warp(&sh.pvdone[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1))
      ok = false;
    tc_fence_after_sync();
    if (!ok) atomicOr(&sh.failed, 4);

    const int m = it.mt * kBlockM + row;
    const bool row_ok = m < n_rows;
    const int t = row_ok ? m / p.G : 0;
    const int jj = m - t * p.G;
    const int head = it.g * p.G + jj;
    if (it.kind == kWindow) {
      if (row_ok) {
        const long long idx = (static_cast<long long>(it.chunk) * p.Hq + head) * p.n_win + t;
        p.win_m[idx] = m_used;
        p.win_l[idx] = l_sum;
      }
    } else {
      const long long tok = it.q_row0 + t;
      const bool final_out = it.kind == kChunk || p.n_splits == 1;
      const float inv_l = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(lane_base + kTmemO + ch * 32, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (!row_ok) continue;
        if (final_out) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                    __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(p.out + (tok * p.Hq + head) * D + ch * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_uint4(packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2],
                                 packed[4 * q4 + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.part_acc + ((static_cast<long long>(it.split) * p.total_lq + tok) * p.Hq + head) * D +
              ch * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                                  __uint_as_float(o[4 * q4 + 2]), __uint_as_float(o[4 * q4 + 3]));
        }
      }
      if (row_ok && it.kind == kDecode) {
        if (p.n_splits == 1) {
          if (p.lse != nullptr)
            p.lse[tok * p.Hq + head] = l_sum > 0.0f ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
        } else {
          const long long idx = (static_cast<long long>(it.split) * p.total_lq + tok) * p.Hq + head;
          p.part_m[idx] = m_used;
          p.part_l[idx] = l_sum;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (tid == 0 && sh.failed != 0) raise_dev_err(p.dev_err, PFD_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attention_smem_bytes(int D) {
  return 1024 + (D == 64 ? Layout<64>::kTotal : Layout<128>::kTotal);
}

cudaError_t launch_attention(const AttnParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  const size_t smem = attention_smem_bytes(p.D);
  cudaError_t err;
  if (p.D == 64) {
    err = ensure_smem_limit(reinterpret_cast<const void*>(attention_kernel<64>), static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    attention_kernel<64><<<grid, kThreads, smem, stream>>>(p);
  } else {
    err = ensure_smem_limit(reinterpret_cast<const void*>(attention_kernel<128>), static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    attention_kernel<128><<<grid, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace pfd
