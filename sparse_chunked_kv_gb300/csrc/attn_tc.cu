// Bidirectional softmax attention of packed query tiles over a list of key
// segments, on tcgen05 tensor cores with TMA-fed Q/K/V tiles.
//
// One kernel serves three kinds of work item:
//   chunk   (prefill)  rows of chunk j attend to chunk j's own C+1 rows
//                      ("Chunked Prefill and KV Caching": each BOS-prefixed
//                      chunk is processed on its own, bidirectionally);
//   window  (prefill)  query-window rows against chunk j, statistics only
//                      (row max and softmax denominator), consumed by the
//                      window-score kernel ("Two-Level Sparsity": ranking by
//                      the cumulative attention weight from the query tokens);
//   decode             live rows of one sequence against one contiguous range
//                      of [selected chunks' pool slots ; live rows], read in
//                      place through the chunk table ("Decoding with Static KV
//                      Reuse"; split-KV with a log-sum-exp merge from
//                      "Attention Kernel Optimization").
//
// A query tile packs Tq = floor(128 / G) tokens x the G query heads of one KV
// head (row m = t * G + j), so one 3-D TMA box loads it and every K/V tile is
// shared by the whole GQA group.  The key sequence is consumed in 16-row
// groups, 8 per 128-key tile; a tile lying inside one segment is loaded with
// one 128-row box per 64-column panel, other tiles group by group.
//
// Per SM two CTAs are resident (96 KB shared memory, 256 TMEM columns each),
// so one CTA's softmax overlaps the other's MMAs and TMA latency.  Inside a
// CTA (192 threads):
//   warp 0      TMA producer (Q once; K and V per tile, single-buffered, the
//               next K loads while the current tile's softmax runs);
//   warp 1      TMEM owner and single-thread MMA issuer:
//               S = Q K^T into TMEM columns [0, 128),
//               O += P V with P read from TMEM columns [0, 64) (bf16 pairs
//               written over S) and V from shared memory;
//   warps 2..5  one thread per tile row (TMEM lane): masked row max, exp2,
//               P into TMEM, O rescale in TMEM only when the running max grows
//               by more than 2^8, epilogue.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr uint32_t kPanelBytes = 128u * 128u;    // 128 rows x 128 B
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;                   // S fp32 [0,128), P bf16x2 [0,64)
constexpr uint32_t kTmemO = 128;
constexpr float kLn2 = 0.69314718055994530942f;

enum ItemKind : int { kChunk = 0, kWindow = 1, kDecode = 2 };

struct TileMeta {
  uint32_t nvalid_lo;  // valid rows of groups 0..3, one byte each
  uint32_t nvalid_hi;  // groups 4..7
  int32_t ngroups;
  int32_t pad;
};

struct Shared {
  uint64_t qfull, kfull, vfull, kempty, vempty, sfull, pfull, ofinal, drain;
  uint64_t mfull[2];
  TileMeta meta[2];
  uint32_t tmem_base;
  int32_t g_lo, g_hi, n_tiles, n_seg;
  int32_t failed;
};

struct Item {
  int kind;
  int g, mt;
  int q_map;          // 0 = main q tensor, 1 = q_win
  long long q_row0;   // token row of t = 0 in the q tensor (and in the output)
  int n_t;            // tokens in this item's query block
  int chunk;          // prefill
  int split;          // decode
  int k0, k1;         // decode: selected-chunk range in sel
};

// Resolves blockIdx.x into a work item; returns false when the CTA has no work.
__device__ __forceinline__ bool resolve_item(const AttnParams& p, Item& it) {
  int bid = blockIdx.x;
  if (p.mode == kModePrefill) {
    if (bid < p.n_chunk_items) {
      it.kind = kChunk;
      it.mt = bid % p.mt_chunk;
      bid /= p.mt_chunk;
      it.q_map = 0;
      it.n_t = p.chunk_rows;
    } else {
      bid -= p.n_chunk_items;
      it.kind = kWindow;
      it.mt = bid % p.mt_win;
      bid /= p.mt_win;
      it.q_map = 1;
      it.n_t = p.n_win;
    }
    it.g = bid % p.Hkv;
    it.chunk = bid / p.Hkv;
    it.q_row0 = it.kind == kChunk ? static_cast<long long>(it.chunk) * p.chunk_rows : 0;
    it.split = 0;
    it.k0 = it.k1 = 0;
    return it.mt * p.Tq < it.n_t;
  }
  it.kind = kDecode;
  it.mt = bid % p.mt_max;
  bid /= p.mt_max;
  it.split = bid % p.n_splits;
  bid /= p.n_splits;
  it.g = bid % p.Hkv;
  const int seq = bid / p.Hkv;
  it.q_map = 0;
  it.chunk = 0;
  const int lq0 = p.cu_lq[seq], lq1 = p.cu_lq[seq + 1];
  const int k0 = p.cu_k[seq], k1 = p.cu_k[seq + 1];
  if (lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq || k0 < 0 || k1 < k0 || k1 > p.total_sel ||
      k1 - k0 >= kMaxSegments) {
    if (threadIdx.x == 0) raise_dev_err(p.dev_err, PFD_DEVERR_SHAPE);
    return false;
  }
  it.q_row0 = lq0;
  it.n_t = lq1 - lq0;
  it.k0 = k0;
  it.k1 = k1;
  return it.mt * p.Tq < it.n_t;
}

template <int D>
struct Layout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;   // Q, K or V tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTileBytes;
  static constexpr uint32_t kV = kK + kTileBytes;
  static constexpr uint32_t kSegRow = kV + kTileBytes;              // int32 [kMaxSegments]
  static constexpr uint32_t kSegLen = kSegRow + 4u * kMaxSegments;  // int32
  static constexpr uint32_t kSegG0 = kSegLen + 4u * kMaxSegments;   // int32 [+1], first group
  static constexpr uint32_t kTotal = kSegG0 + 4u * (kMaxSegments + 1);
};

__device__ __forceinline__ int groups_of(int len) { return (len + kGroupRows - 1) / kGroupRows; }

// Fills the segment list of the item (row, length, first global group) in
// shared memory; run by one full warp.  Decode: the selected chunks' slots
// through the table, then the live block (the last segment, tensor 1).
__device__ __forceinline__ int load_segments(const AttnParams& p, const Item& it, int32_t* seg_row,
                                             int32_t* seg_len, int32_t* seg_g0, int lane) {
  int nseg;
  if (it.kind != kDecode) {
    nseg = 1;
    if (lane == 0) {
      seg_row[0] = it.chunk * p.chunk_rows;
      seg_len[0] = p.chunk_rows;
    }
  } else {
    const int nsel = it.k1 - it.k0;
    nseg = nsel + 1;
    for (int i = lane; i < nsel; i += 32) {
      const int c = p.sel[it.k0 + i];
      int row = 0, len = 0;
      if (c < 0 || c >= p.table_len) {
        raise_dev_err(p.dev_err, PFD_DEVERR_SEL);
      } else {
        const pfd_chunk_entry e = p.table[c];
        if (e.row < 0 || e.len < 0 || static_cast<long long>(e.row) + e.len > p.pool_rows) {
          raise_dev_err(p.dev_err, PFD_DEVERR_TABLE);
        } else {
          row = e.row;
          len = e.len;
        }
      }
      seg_row[i] = row;
      seg_len[i] = len;
    }
    if (lane == 0) {
      seg_row[nsel] = static_cast<int32_t>(it.q_row0);
      seg_len[nsel] = it.n_t;
    }
  }
  __syncwarp();
  int carry = 0;
  for (int base = 0; base < nseg; base += 32) {
    const int i = base + lane;
    const int n = i < nseg ? groups_of(seg_len[i]) : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (i < nseg) seg_g0[i] = carry + incl - n;
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) seg_g0[nseg] = carry;
  __syncwarp();
  return nseg;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
attention_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;

  Item it;
  if (!resolve_item(p, it)) return;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int32_t* seg_row = reinterpret_cast<int32_t*>(smem + L::kSegRow);
  int32_t* seg_len = reinterpret_cast<int32_t*>(smem + L::kSegLen);
  int32_t* seg_g0 = reinterpret_cast<int32_t*>(smem + L::kSegG0);
  const uint32_t s_base = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool with_pv = it.kind != kWindow;
  const int G = p.G;
  const int q_rows = G * p.Tq;                 // rows of the tile filled by the Q box

  // ----------------------------------------------------------- prologue --
  if (warp == 0) {
    const int nseg = load_segments(p, it, seg_row, seg_len, seg_g0, lane);
    if (lane == 0) {
      mbar_init(&sh.qfull, 1);
      mbar_init(&sh.kfull, 1);
      mbar_init(&sh.vfull, 1);
      mbar_init(&sh.kempty, 1);
      mbar_init(&sh.vempty, 1);
      mbar_init(&sh.sfull, 1);
      mbar_init(&sh.pfull, kSoftmaxThreads);
      mbar_init(&sh.ofinal, 1);
      mbar_init(&sh.drain, 1);
      mbar_init(&sh.mfull[0], 1);
      mbar_init(&sh.mfull[1], 1);
      fence_barrier_init();
      const long long total = seg_g0[nseg];
      const int n_splits = it.kind == kDecode ? p.n_splits : 1;
      const long long lo = total * it.split / n_splits;
      const long long hi = total * (it.split + 1) / n_splits;
      sh.g_lo = static_cast<int>(lo);
      sh.g_hi = static_cast<int>(hi);
      sh.n_tiles = static_cast<int>((hi - lo + kGroupsPerTile - 1) / kGroupsPerTile);
      sh.n_seg = nseg;
      sh.failed = 0;
    }
  } else if (warp == 1) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  } else if (q_rows < kBlockM) {
    // Tile rows past the Q box are never loaded: keep them zero.
    const int ts = tid - 64;
    for (int idx = ts; idx < (kBlockM - q_rows) * (D / 8); idx += kSoftmaxThreads) {
      const int r = q_rows + idx / (D / 8), c = idx % (D / 8);
      *reinterpret_cast<uint4*>(smem + L::kQ + sw128_offset(r, c * 8, kBlockM)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
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
      const int nseg = sh.n_seg;
      const int qm = it.q_map;
      mbar_arrive_expect_tx(&sh.qfull, static_cast<uint32_t>(q_rows) * D * 2);
      for (int pn = 0; pn < D / 64; ++pn)
        tma_load_3d(smem + L::kQ + pn * kPanelBytes, &p.tm_q[qm], &sh.qfull, pn * 64, it.g * G,
                    static_cast<int>(it.q_row0) + it.mt * p.Tq);
      int seg = 0;
      while (seg + 1 < nseg && seg_g0[seg + 1] <= g_lo) ++seg;
      int gofs = g_lo - seg_g0[seg];
      int g_cur = g_lo;
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        // Group list of tile j.
        int tens[kGroupsPerTile];
        int rows[kGroupsPerTile];
        uint32_t nv_lo = 0, nv_hi = 0;
        int ng = 0;
        const bool one_box = (g_hi - g_cur >= kGroupsPerTile) &&
                             ((gofs + kGroupsPerTile) * kGroupRows <= seg_len[seg]);
        for (; ng < kGroupsPerTile && g_cur < g_hi; ++ng, ++g_cur) {
          const int len = seg_len[seg];
          const int nv = min(kGroupRows, len - gofs * kGroupRows);
          tens[ng] = (it.kind == kDecode && seg == nseg - 1) ? 1 : 0;
          rows[ng] = seg_row[seg] + gofs * kGroupRows;
          if (ng < 4) nv_lo |= static_cast<uint32_t>(nv) << (8 * ng);
          else nv_hi |= static_cast<uint32_t>(nv) << (8 * (ng - 4));
          ++gofs;
          if (gofs * kGroupRows >= len) {
            gofs = 0;
            ++seg;
            while (seg < nseg && seg_len[seg] == 0) ++seg;
          }
        }
        // K(j) replaces K(j-1): wait for QK(j-1).  The metadata slot j & 1 was
        // last read by the softmax of tile j-2, which ended before QK(j-1).
        if (j >= 1 && !mbar_wait(&sh.kempty, (j - 1) & 1)) { ok = false; break; }
        TileMeta& m = sh.meta[j & 1];
        m.nvalid_lo = nv_lo;
        m.nvalid_hi = nv_hi;
        m.ngroups = ng;
        mbar_arrive(&sh.mfull[j & 1]);
        const uint32_t bytes = one_box ? static_cast<uint32_t>(kBlockN) * D * 2
                                       : static_cast<uint32_t>(ng) * kGroupRows * D * 2;
        mbar_arrive_expect_tx(&sh.kfull, bytes);
        if (one_box) {
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + L::kK + pn * kPanelBytes, &p.tm_k128[tens[0]], &sh.kfull, pn * 64,
                        it.g, rows[0]);
        } else {
          for (int k = 0; k < ng; ++k)
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d(smem + L::kK + pn * kPanelBytes + k * 2048, &p.tm_k16[tens[k]],
                          &sh.kfull, pn * 64, it.g, rows[k]);
        }
        if (with_pv) {
          // V(j) replaces V(j-1): wait for PV(j-1).
          if (j >= 1 && !mbar_wait(&sh.vempty, (j - 1) & 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh.vfull, bytes);
          if (one_box) {
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d(smem + L::kV + pn * kPanelBytes, &p.tm_v128[tens[0]], &sh.vfull,
                          pn * 64, it.g, rows[0]);
          } else {
            for (int k = 0; k < ng; ++k)
              for (int pn = 0; pn < D / 64; ++pn)
                tma_load_3d(smem + L::kV + pn * kPanelBytes + k * 2048, &p.tm_v16[tens[k]],
                            &sh.vfull, pn * 64, it.g, rows[k]);
          }
        }
      }
      if (!ok) atomicOr(&sh.failed, 1);
      // The last tile's loads must have landed before the CTA exits.
      const int jl = n_tiles - 1;
      mbar_wait(&sh.kfull, jl & 1);
      if (with_pv) mbar_wait(&sh.vfull, jl & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait(&sh.qfull, 0);
      const uint32_t q_addr = s_base + L::kQ;
      const uint32_t k_addr = s_base + L::kK;
      const uint32_t v_addr = s_base + L::kV;
      for (int j = 0; ok && j < n_tiles; ++j) {
        const uint32_t ph = j & 1;
        if (!mbar_wait(&sh.kfull, ph)) { ok = false; break; }
        tc_fence_after_sync();
        const int ng = min(sh.meta[j & 1].ngroups, kGroupsPerTile);
        const uint32_t idesc_s = idesc_bf16(kBlockM, max(ng, 1) * kGroupRows, false, false);
        if (ng > 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = sw128_desc(q_addr + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t b = sw128_desc(k_addr + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(tmem + kTmemS, a, b, idesc_s, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sh.sfull);
        mma_commit(&sh.kempty);
        if (!mbar_wait(&sh.pfull, ph)) { ok = false; break; }
        if (with_pv) {
          if (!mbar_wait(&sh.vfull, ph)) { ok = false; break; }
          tc_fence_after_sync();
          constexpr uint32_t idesc_o = idesc_bf16(kBlockM, D, false, true);
          for (int kk = 0; kk < ng; ++kk) {
            const uint64_t v = sw128_desc(v_addr + kk * 2048, kPanelBytes, 1024);
            mma_bf16_ts(tmem + kTmemO, tmem + kTmemS + kk * 8, v, idesc_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&sh.vempty);
      }
      if (!ok) atomicOr(&sh.failed, 2);
      mma_commit(&sh.ofinal);
      // Every MMA issued above has completed once `drain` flips.
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0);
    }
  } else {
    // ---------------------------------------------- softmax + epilogue --
    const int quarter = warp & 3;         // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;  // tile row of this thread
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float scale = p.scale_log2;

    float m_used = -INFINITY;
    float l_sum = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const uint32_t ph = j & 1;
      if (!mbar_wait_warp(&sh.mfull[j & 1], (j >> 1) & 1) || !mbar_wait_warp(&sh.sfull, ph)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const TileMeta meta = sh.meta[j & 1];
      const int ncol = meta.ngroups * kGroupRows;
      const bool full = meta.ngroups == kGroupsPerTile && meta.nvalid_lo == 0x10101010u &&
                        meta.nvalid_hi == 0x10101010u;
      auto nv_of = [&](int grp) -> int {
        const uint32_t w = grp < 4 ? meta.nvalid_lo : meta.nvalid_hi;
        return static_cast<int>((w >> (8 * (grp & 3))) & 0xFFu);
      };

      // Pass 1: row max of the valid logits.
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if (ch * 32 < ncol) {
          uint32_t s[32];
          tmem_ld32(lane_base + kTmemS + ch * 32, s);
          tmem_ld_wait(s);
          if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              mx0 = fmaxf(mx0, __uint_as_float(s[i]));
              mx1 = fmaxf(mx1, __uint_as_float(s[i + 1]));
              mx2 = fmaxf(mx2, __uint_as_float(s[i + 2]));
              mx3 = fmaxf(mx3, __uint_as_float(s[i + 3]));
            }
          } else {
            const int nva = nv_of(2 * ch), nvb = nv_of(2 * ch + 1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const bool valid = (i & 15) < (i < 16 ? nva : nvb);
              const float x = valid ? __uint_as_float(s[i]) : -INFINITY;
              if ((i & 3) == 0) mx0 = fmaxf(mx0, x);
              else if ((i & 3) == 1) mx1 = fmaxf(mx1, x);
              else if ((i & 3) == 2) mx2 = fmaxf(mx2, x);
              else mx3 = fmaxf(mx3, x);
            }
          }
        }
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale;

      // Rescale decision per row; the TMEM rescale of O is warp-collective,
      // so a warp rescales when any of its rows needs it (alpha = 1 for the
      // others).  sfull(j) also covers PV(j-1): O is complete here.
      const bool mine = m_tile > m_used + kRescaleThreshold;
      if (__any_sync(0xFFFFFFFFu, mine)) {
        const float m_new = mine ? m_tile : m_used;
        const float alpha = mine ? ex2_approx(m_used - m_new) : 1.0f;
        if (j >= 1 && with_pv) {
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(lane_base + kTmemO + ch * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + kTmemO + ch * 32, o);
          }
        }
        l_sum *= alpha;
        m_used = m_new;
      }

      // Pass 2: probabilities relative to m_used -> bf16 pairs in TMEM
      // columns [0, 64) (over S columns already read), fp32 row sum.
      const float neg_m = -m_used;
      float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (half * 64 < ncol) {
          uint32_t packed[32];
#pragma unroll
          for (int sub = 0; sub < 2; ++sub) {
            const int ch = half * 2 + sub;
            uint32_t s[32];
            tmem_ld32(lane_base + kTmemS + ch * 32, s);
            tmem_ld_wait(s);
            if (full) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float a = ex2_approx(fmaf(__uint_as_float(s[2 * i]), scale, neg_m));
                const float b = ex2_approx(fmaf(__uint_as_float(s[2 * i + 1]), scale, neg_m));
                if (i & 1) { sum2 += a; sum3 += b; } else { sum0 += a; sum1 += b; }
                packed[sub * 16 + i] = pack_bf16x2(a, b);
              }
            } else {
              const int nva = nv_of(2 * ch), nvb = nv_of(2 * ch + 1);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c0 = 2 * i, c1 = 2 * i + 1;
                const bool v0 = (c0 & 15) < (c0 < 16 ? nva : nvb);
                const bool v1 = (c1 & 15) < (c1 < 16 ? nva : nvb);
                const float a = v0 ? ex2_approx(fmaf(__uint_as_float(s[c0]), scale, neg_m)) : 0.0f;
                const float b = v1 ? ex2_approx(fmaf(__uint_as_float(s[c1]), scale, neg_m)) : 0.0f;
                if (i & 1) { sum2 += a; sum3 += b; } else { sum0 += a; sum1 += b; }
                packed[sub * 16 + i] = pack_bf16x2(a, b);
              }
            }
          }
          if (with_pv) tmem_st32(lane_base + kTmemS + half * 32, packed);
        }
      }
      l_sum += (sum0 + sum1) + (sum2 + sum3);
      if (with_pv) tmem_st_wait();

      if (with_pv && !full) {
        // Rows of a ragged group that lie past its segment may hold anything
        // (another slot, padding): zero them in V so that 0 * v stays 0.
        if (!mbar_wait_warp(&sh.vfull, ph)) { ok = false; break; }
        const int ts = tid - 64;
        uint8_t* v_tile = smem + L::kV;
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
        fence_proxy_async_smem();
      }
      tc_fence_before_sync();
      mbar_arrive(&sh.pfull);
    }

    // ------------------------------------------------------------ epilogue --
    if (ok && n_tiles > 0 && !mbar_wait_warp(&sh.ofinal, 0)) ok = false;
    tc_fence_after_sync();
    if (!ok) atomicOr(&sh.failed, 4);

    const int t_local = row / G;
    const int jj = row - t_local * G;
    const int t = it.mt * p.Tq + t_local;
    const bool row_ok = row < q_rows && t < it.n_t;
    const int head = it.g * G + jj;
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
