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
// shared by the whole GQA group.  A work item holds two such tiles (a, b) and
// one key range; the key sequence is consumed in 16-row groups, 8 per 128-key
// tile, and a tile inside one segment is loaded with one 128-row box per
// 64-column panel.
//
// The kernel is persistent (one CTA per SM, items strided over the grid) and
// warp-specialised (352 threads):
//   warp 0      TMA producer of K and V tiles into a 4-slot ring (K(j), V(j),
//               K(j+1), ...), so loads run two tiles ahead, also across item
//               boundaries; it also publishes each tile's group metadata;
//   warp 10     TMA loader of the item's two Q tiles (once every MMA of the
//               previous item, the last QK included, has completed);
//   warp 1      TMEM owner and single-thread MMA issuer, ping-ponging the two
//               query tiles:  QK_a(0) QK_b(0) | PV_a(j) QK_a(j+1) PV_b(j)
//               QK_b(j+1) | ...  so the tensor core works on one tile while
//               the other tile's softmax runs;
//   warps 2..5  softmax warpgroup of tile a, warps 6..9 of tile b: one thread
//               per row (TMEM lane): masked row max, exp2, P as bf16 pairs in
//               TMEM over the S columns already read (the A operand of PV),
//               O rescale in TMEM only when the running max grows by more than
//               2^8, and the epilogue of the item.
// TMEM (512 columns): S_a [0,128), S_b [128,256), O_a [256,..), O_b [384,..).
//
// A prefill chunk has C + 1 keys: its BOS row and C content rows.  The tensor
// cores take only the content rows (C = 256, 512, 1024 fill whole 128-key
// tiles, where the BOS row would add a tile of one key); the BOS key enters
// analytically.  The Q loader brings its K and V rows to shared memory with
// the item's Q, each softmax thread computes its BOS logit from the Q tile
// during the first key tile, and the epilogue folds it into the row's max,
// denominator and output: M = max(m, s0), l' = l 2^(m - M) + 2^(s0 - M),
// O' = O 2^(m - M) + 2^(s0 - M) v0.
#include "pfd_internal.cuh"
#include "sm103_ptx.cuh"

namespace pfd {
namespace {

constexpr int kThreads = 352;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kSoftmaxWarp0 = 2;                  // warps 2..5: tile a, 6..9: tile b
constexpr int kQLoaderWarp = 10;

constexpr int kWgThreads = 128;
constexpr int kRing = 4;
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr uint32_t kPanelBytes = 128u * 128u;    // 128 rows x 128 B
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ uint32_t tmem_s_col(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t tmem_o_col(int x) { return x ? 384u : 256u; }

enum ItemKind : int { kChunk = 0, kWindow = 1, kDecode = 2, kMass = 3 };

// Valid rows of a 16-row key group, one byte per group: 16 for a full
// group, 0 for a group past the tile's end, n (1..15) for the last group of a
// segment loaded from its first row (rows n..15 lie past the segment), and
// kShifted | n for that group loaded as the 16 rows ending at the segment's
// end (rows 0..15-n repeat keys of the previous group).  A segment of 16 or
// more rows is always loaded shifted, so every V row the tensor core reads
// belongs to the segment.
constexpr uint32_t kShifted = 0x80u;

struct TileMeta {
  uint32_t nvalid_lo;  // valid-row codes of groups 0..3, one byte each
  uint32_t nvalid_hi;  // groups 4..7
  int32_t ngroups;     // 0 only for the single tile of an empty item
  int32_t last;        // 1 on the last tile of an item
  int32_t fix_v;       // 1 when a group is ragged and unshifted: its V rows
                       // past the segment must be zeroed before PV.  Chunk-mass
                       // items (no PV): the segment (chunk of the item) of
                       // group g in bits [4g, 4g + 4)
};

struct Shared {
  uint64_t q_full, q_empty;
  uint64_t ring_full[kRing], ring_empty[kRing];
  uint64_t meta_full[kRing], meta_empty[kRing];
  uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
  uint64_t drain;
  TileMeta meta[kRing];
  uint32_t tmem_base;
  int32_t failed;
};

struct Item {
  int kind;
  int g;
  int ta;             // query tile index of tile a (tile b = ta + 1)
  bool has_b;
  int q_map;          // 0 = main q tensor, 1 = q_win
  long long q_row0;   // token row of t = 0 in the q tensor (and in the output)
  int n_t;            // tokens in this item's query block
  int chunk;          // prefill
  int split;          // decode
  int k0, k1;         // decode: selected-chunk range in sel
};

// Work item `idx`; returns false when it holds no query rows.  The decode
// and chunk-mass instantiations compile only their own mode's branch (their
// mode is fixed); the prefill instantiation dispatches on p.mode, which
// measured faster for it.
template <bool kPrefill, bool kMassMode>
__device__ __forceinline__ bool resolve_item(const AttnParams& p, int idx, Item& it) {
  constexpr bool kDecodeOnly = !kPrefill && !kMassMode;
  if (kPrefill && p.mode == kModePrefill) {
    int pairs;
    if (idx < p.n_chunk_items) {
      it.kind = kChunk;
      pairs = (p.mt_chunk + 1) / 2;
      it.q_map = 0;
      it.n_t = p.chunk_rows;
    } else {
      idx -= p.n_chunk_items;
      it.kind = kWindow;
      pairs = (p.mt_win + 1) / 2;
      it.q_map = 1;
      it.n_t = p.n_win;
    }
    it.ta = 2 * (idx % pairs);
    idx /= pairs;
    it.g = idx % p.Hkv;
    it.chunk = idx / p.Hkv;
    it.q_row0 = it.kind == kChunk ? static_cast<long long>(it.chunk) * p.chunk_rows
                                  : static_cast<long long>(it.chunk / p.layer_chunks) * p.n_win;
    it.split = 0;
    it.k0 = it.k1 = 0;
  } else if (!kDecodeOnly && (kMassMode || p.mode == kModeMass)) {
    // sequence b of the item (mass_item0 is non-decreasing, b < 64)
    int b = 0;
    while (b + 1 < p.mass_batch && p.mass_item0[b + 1] <= idx) ++b;
    const int local = idx - p.mass_item0[b];
    const int pairs = p.mass_pairs[b];
    it.kind = kMass;
    it.ta = 2 * (local % pairs);
    const int rest = local / pairs;
    it.g = rest % p.Hkv;
    // the item's chunks: table entries [k0, k1), at most mass_chunks
    it.k0 = p.mass_n0[b] + (rest / p.Hkv) * p.mass_chunks;
    it.k1 = min(it.k0 + p.mass_chunks, p.mass_n0[b + 1]);
    it.chunk = it.k0;
    it.q_map = 0;
    it.split = 0;
    const int lq0 = p.cu_lq[b], lq1 = p.cu_lq[b + 1];
    if (lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq) return false;   // reported by the producer
    it.q_row0 = lq0;
    it.n_t = lq1 - lq0;
  } else {
    const int pairs = (p.mt_max + 1) / 2;
    it.kind = kDecode;
    it.ta = 2 * (idx % pairs);
    idx /= pairs;
    it.split = idx % p.n_splits;
    idx /= p.n_splits;
    it.g = idx % p.Hkv;
    const int seq = idx / p.Hkv;
    it.q_map = 0;
    it.chunk = 0;
    const int lq0 = p.cu_lq[seq], lq1 = p.cu_lq[seq + 1];
    const int k0 = p.cu_k[seq], k1 = p.cu_k[seq + 1];
    if (lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq || k0 < 0 || k1 < k0 || k1 > p.total_sel ||
        k1 - k0 >= kMaxSegments)
      return false;  // reported by the producer
    it.q_row0 = lq0;
    it.n_t = lq1 - lq0;
    it.k0 = k0;
    it.k1 = k1;
  }
  it.has_b = (it.ta + 1) * p.Tq < it.n_t;
  return it.ta * p.Tq < it.n_t;
}

template <bool kPrefill, bool kMassMode>
__device__ __forceinline__ bool item_shape_error(const AttnParams& p, int idx) {
  if (kPrefill && p.mode == kModePrefill) return false;
  if (!(!kPrefill && !kMassMode) && (kMassMode || p.mode == kModeMass)) {
    int b = 0;
    while (b + 1 < p.mass_batch && p.mass_item0[b + 1] <= idx) ++b;
    const int lq0 = p.cu_lq[b], lq1 = p.cu_lq[b + 1];
    return lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq;
  }
  const int pairs = (p.mt_max + 1) / 2;
  const int seq = idx / pairs / p.n_splits / p.Hkv;
  const int lq0 = p.cu_lq[seq], lq1 = p.cu_lq[seq + 1];
  const int k0 = p.cu_k[seq], k1 = p.cu_k[seq + 1];
  return lq0 < 0 || lq1 < lq0 || lq1 > p.total_lq || k0 < 0 || k1 < k0 || k1 > p.total_sel ||
         k1 - k0 >= kMaxSegments;
}

// Prefill item of cost rank r: first the pairs of two query tiles, then the
// pairs of one (the last pair of an odd tile count), first of chunk rows,
// then of window rows; returns the item index resolve_item decodes.
__device__ __forceinline__ int prefill_item_of_rank(const AttnParams& p, int r) {
  const int pairs_c = (p.mt_chunk + 1) / 2, pairs_w = (p.mt_win + 1) / 2;
  const int half_c = p.mt_chunk & 1, half_w = p.mt_win & 1;
  const int full_c = pairs_c - half_c, full_w = pairs_w - half_w;
  const int groups = p.n_chunks * p.Hkv;   // (chunk, KV head); all counts below n_items < 2^31
  int n = groups * full_c;
  if (r < n) return (r / full_c) * pairs_c + r % full_c;
  r -= n;
  if (half_c) {
    if (r < groups) return r * pairs_c + pairs_c - 1;
    r -= groups;
  }
  n = groups * full_w;
  if (r < n) return p.n_chunk_items + (r / full_w) * pairs_w + r % full_w;
  r -= n;
  return p.n_chunk_items + r * pairs_w + pairs_w - 1;
}

// The k-th work item of this CTA, or -1 past its last.  Decode: the items
// strided over the grid.  Prefill: the items in cost order dealt back and
// forth over the CTAs (rank k G + b on even rounds, k G + G - 1 - b on odd
// ones), which evens out the CTAs' totals.
template <bool kPrefill>
__device__ __forceinline__ int nth_item(const AttnParams& p, int k) {
  const int grid = static_cast<int>(gridDim.x);
  if constexpr (!kPrefill) {
    const int idx = static_cast<int>(blockIdx.x) + k * grid;   // n_items < 2^31
    return idx < p.n_items ? idx : -1;
  } else {
    const int b = static_cast<int>(blockIdx.x);
    const int r = k * grid + ((k & 1) ? grid - 1 - b : b);
    return r < p.n_items ? prefill_item_of_rank(p, r) : -1;
  }
}

template <int D>
struct Layout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;   // Q, K or V tile
  static constexpr uint32_t kQ0 = 0;
  static constexpr uint32_t kQ1 = kQ0 + kTileBytes;
  static constexpr uint32_t kRing0 = kQ1 + kTileBytes;     // kRing slots of one tile
  static constexpr uint32_t kSegRow = kRing0 + kRing * kTileBytes;   // int32 [kMaxSegments]
  static constexpr uint32_t kSegLen = kSegRow + 4u * kMaxSegments;
  static constexpr uint32_t kSegG0 = kSegLen + 4u * kMaxSegments;    // [kMaxSegments + 1]
  static constexpr uint32_t kTotalDecode = kSegG0 + 4u * (kMaxSegments + 1);
  // Prefill only: the BOS rows of the item's chunk, double-buffered by item
  // parity: one 16-row TMA box of K, then one of V (row 0 is the BOS row).
  static constexpr uint32_t kBosBox = (D / 64) * 16u * 128u;
  static constexpr uint32_t kBos0 = (kTotalDecode + 1023u) & ~1023u;
  static constexpr uint32_t kTotalPrefill = kBos0 + 2u * 2u * kBosBox;
};

__device__ __forceinline__ int groups_of(int len) { return (len + kGroupRows - 1) / kGroupRows; }

// Fills the item's segment list (row, length, first global group) in shared
// memory; run by the whole producer warp.  Decode: the selected chunks' slots
// through the table, then (unless the call leaves it out) the live block,
// the last segment, read from tensor 1.
template <bool kPrefill, bool kMassMode>
__device__ __forceinline__ int load_segments(const AttnParams& p, const Item& it, int32_t* seg_row,
                                             int32_t* seg_len, int32_t* seg_g0, int lane) {
  int nseg;
  __syncwarp();
  constexpr bool kDecodeOnly = !kPrefill && !kMassMode;
  if (!kDecodeOnly && (kMassMode || it.kind == kMass)) {
    // one segment per chunk of the item, in table order
    nseg = it.k1 - it.k0;
    for (int i = lane; i < nseg; i += 32) {
      const pfd_chunk_entry e = p.table[it.k0 + i];
      const bool bad = e.row < 0 || e.len < 0 || static_cast<long long>(e.row) + e.len > p.pool_rows;
      if (bad) raise_dev_err(p.dev_err, PFD_DEVERR_TABLE);
      seg_row[i] = bad ? 0 : e.row;
      seg_len[i] = bad ? 0 : e.len;
    }
  } else if (!kDecodeOnly && !kMassMode && it.kind != kDecode) {
    nseg = 1;
    if (lane == 0) {
      seg_row[0] = it.chunk * p.chunk_rows + 1;   // the content rows; BOS enters analytically
      seg_len[0] = p.chunk_rows - 1;
    }
  } else {
    const int nsel = it.k1 - it.k0;
    nseg = nsel + (p.self_keys ? 1 : 0);
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
    if (lane == 0 && p.self_keys) {
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

// Softmax warpgroup state that persists over the tiles of one item.
struct RowState {
  float m_used;
  float l_sum;
};

// kPrefill: a prefill launch (chunk and window items, with the analytic BOS
// key); else a decode launch, compiled without that code.  kMassMode: a
// chunk-mass launch (decode-shaped, mass items only); kMassMulti: its items
// hold several chunks each, with per-chunk sums (one chunk per item needs
// only the row sum).
template <int D, bool kPrefill, bool kMassMode, bool kMassMulti>
__global__ void __launch_bounds__(kThreads, 1)
attention_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  int32_t* seg_row = reinterpret_cast<int32_t*>(smem + L::kSegRow);
  int32_t* seg_len = reinterpret_cast<int32_t*>(smem + L::kSegLen);
  int32_t* seg_g0 = reinterpret_cast<int32_t*>(smem + L::kSegG0);
  const uint32_t s_base = smem_u32(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.G;
  const int q_rows = G * p.Tq;   // rows of a query tile filled by the Q box

  // ----------------------------------------------------------- prologue --
  if (tid == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&sh.ring_full[i], 1);
      mbar_init(&sh.ring_empty[i], 1);
      mbar_init(&sh.meta_full[i], 1);
      mbar_init(&sh.meta_empty[i], 1 + 8);   // the MMA thread + one lane per softmax warp
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sh.s_full[x], 1);
      // one arrival per softmax warp (after a warp sync), not per thread
      mbar_init(&sh.p_full[x], kWgThreads / 32);
      mbar_init(&sh.o_full[x], 1);
      mbar_init(&sh.o_free[x], kWgThreads / 32);
    }
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
    sh.failed = 0;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sh.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 8 && q_rows < kBlockM) {
    // Rows of the Q tiles past the Q box are never loaded: keep them zero.
    const int ts = tid - kSoftmaxWarp0 * 32;
    for (int idx = ts; idx < 2 * (kBlockM - q_rows) * (D / 8); idx += 2 * kWgThreads) {
      const int x = idx / ((kBlockM - q_rows) * (D / 8));
      const int rem = idx % ((kBlockM - q_rows) * (D / 8));
      const int r = q_rows + rem / (D / 8), c = rem % (D / 8);
      *reinterpret_cast<uint4*>(smem + (x ? L::kQ1 : L::kQ0) + sw128_offset(r, c * 8, kBlockM)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Everything above touched only this CTA's shared memory and TMEM; global
  // inputs may come from the previous kernel on the stream.
  grid_dependency_wait();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer --
    uint32_t ring_ctr = 0;   // ring loads issued
    uint32_t tile_ctr = 0;   // tiles published
    int items_done = 0;
    bool ok = true;
    for (int kk = 0, idx; ok && (idx = nth_item<kPrefill>(p, kk)) >= 0; ++kk) {
      Item it;
      if (!resolve_item<kPrefill, kMassMode>(p, idx, it)) {
        if (lane == 0 && item_shape_error<kPrefill, kMassMode>(p, idx))
          raise_dev_err(p.dev_err, PFD_DEVERR_SHAPE);
        continue;
      }
      const bool with_pv = it.kind != kWindow && it.kind != kMass;
      const int nseg = load_segments<kPrefill, kMassMode>(p, it, seg_row, seg_len, seg_g0, lane);
      const long long total = seg_g0[nseg];
      const int n_splits = it.kind == kDecode ? p.n_splits : 1;
      const int g_lo = static_cast<int>(total * it.split / n_splits);
      const int g_hi = static_cast<int>(total * (it.split + 1) / n_splits);
      const int n_tiles = (g_hi - g_lo + kGroupsPerTile - 1) / kGroupsPerTile;
      const int tiles_to_publish = n_tiles > 0 ? n_tiles : 1;
      // Segment of each lane's group: found by binary search for the item's
      // first tile, then carried from tile to tile (a lane's group moves 8
      // groups on per tile, so its segment can only move forward).
      int lseg = 0;
      for (int j = 0; ok && j < tiles_to_publish; ++j) {
        // Lanes 0..ng-1 each place one 16-row key group of the tile: its
        // segment (seg_g0[s] <= g < seg_g0[s + 1]), source row, tensor and
        // valid-row code.
        const int g0 = g_lo + j * kGroupsPerTile;
        const int ng = n_tiles > 0 ? min(kGroupsPerTile, g_hi - g0) : 0;
        int row = 0, t = 0;
        uint32_t code = 0;
        if (lane < ng) {
          const int g = g0 + lane;
          int lo = lseg;
          if (j == 0) {
            int hi = nseg;
            while (hi - lo > 1) {
              const int mid = (lo + hi) >> 1;
              if (seg_g0[mid] <= g) lo = mid;
              else hi = mid;
            }
          } else {
            while (lo + 1 < nseg && seg_g0[lo + 1] <= g) ++lo;
          }
          lseg = lo;
          const int len = seg_len[lo];
          const int gofs = g - seg_g0[lo];
          const int nv = min(kGroupRows, len - gofs * kGroupRows);
          const bool shifted = nv < kGroupRows && len >= kGroupRows;
          t = (it.kind == kDecode && p.self_keys && lo == nseg - 1) ? 1 : 0;
          row = seg_row[lo] + (shifted ? len - kGroupRows : gofs * kGroupRows);
          code = static_cast<uint32_t>(nv) | (shifted ? kShifted : 0u);
        }
        uint32_t packed = lane < kGroupsPerTile ? code << (8 * (lane & 3)) : 0u;
        packed |= __shfl_xor_sync(0xFFFFFFFFu, packed, 1);
        packed |= __shfl_xor_sync(0xFFFFFFFFu, packed, 2);
        const uint32_t nv_lo = __shfl_sync(0xFFFFFFFFu, packed, 0);
        const uint32_t nv_hi = __shfl_sync(0xFFFFFFFFu, packed, 4);
        const bool fix_v = __any_sync(0xFFFFFFFFu, lane < ng && code < kGroupRows);
        uint32_t seg4 = 0;
        if constexpr (kMassMulti) {
          seg4 = lane < ng ? static_cast<uint32_t>(lseg & 0xF) << (4 * lane) : 0u;
          seg4 |= __shfl_xor_sync(0xFFFFFFFFu, seg4, 1);
          seg4 |= __shfl_xor_sync(0xFFFFFFFFu, seg4, 2);
          seg4 |= __shfl_xor_sync(0xFFFFFFFFu, seg4, 4);
          seg4 = __shfl_sync(0xFFFFFFFFu, seg4, 0);
        }
        // Runs: group k continues group k-1's run when it is the next 16 rows
        // of the same tensor.  A lane that starts a run loads the whole run,
        // one box per set bit of its length (16..128 rows).
        const int prev_row = __shfl_up_sync(0xFFFFFFFFu, row, 1);
        const int prev_t = __shfl_up_sync(0xFFFFFFFFu, t, 1);
        const bool cont = lane > 0 && lane < ng && t == prev_t && row == prev_row + kGroupRows;
        const uint32_t cont_mask = __ballot_sync(0xFFFFFFFFu, cont);
        const bool starts = lane < ng && !cont;
        const int run_len = starts ? __ffs(~(cont_mask >> (lane + 1))) : 0;   // 1 + continuing groups

        // Metadata slot tile_ctr % kRing: every consumer must have read the
        // tile published there kRing tiles ago.
        const int ms = tile_ctr % kRing;
        if (tile_ctr >= kRing && !mbar_wait_warp(&sh.meta_empty[ms], ((tile_ctr / kRing) - 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          TileMeta& m = sh.meta[ms];
          m.nvalid_lo = nv_lo;
          m.nvalid_hi = nv_hi;
          m.ngroups = ng;
          m.last = (j == tiles_to_publish - 1) ? 1 : 0;
          m.fix_v = kMassMode ? static_cast<int32_t>(seg4) : (fix_v ? 1 : 0);
          mbar_arrive(&sh.meta_full[ms]);
        }
        ++tile_ctr;
        if (ng == 0) break;
        const uint32_t bytes = static_cast<uint32_t>(ng) * kGroupRows * D * 2;
        for (int kv = 0; kv < (with_pv ? 2 : 1); ++kv) {
          const int rs = ring_ctr % kRing;
          if (ring_ctr >= kRing && !mbar_wait_warp(&sh.ring_empty[rs], ((ring_ctr / kRing) - 1) & 1)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&sh.ring_full[rs], bytes);
          __syncwarp();
          if (starts) {
            uint8_t* dst = smem + L::kRing0 + rs * L::kTileBytes;
            const CUtensorMap(*maps)[2] = kv ? p.tm_v : p.tm_k;
            int off = 0;
#pragma unroll
            for (int lv = kBoxLevels - 1; lv >= 0; --lv) {
              if (run_len - off < (1 << lv)) continue;
#pragma unroll
              for (int pn = 0; pn < D / 64; ++pn)
                tma_load_3d(dst + pn * kPanelBytes + (lane + off) * 2048, &maps[lv][t],
                            &sh.ring_full[rs], pn * 64, it.g, row + off * kGroupRows);
              off += 1 << lv;
            }
          }
          ++ring_ctr;
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      ++items_done;
    }
    if (lane == 0) {
      if (!ok) atomicOr(&sh.failed, 1);
      // Loads still in flight must land before the CTA exits.
      for (uint32_t c = ring_ctr > kRing ? ring_ctr - kRing : 0; c < ring_ctr; ++c)
        mbar_wait(&sh.ring_full[c % kRing], (c / kRing) & 1);
    }
  } else if (warp == kQLoaderWarp) {
    // -------------------------------------------------------- Q loader --
    if (lane == 0) {
      int items_done = 0;
      bool ok = true;
      const uint32_t q_bytes = static_cast<uint32_t>(q_rows) * D * 2;
      for (int kk = 0, idx; ok && (idx = nth_item<kPrefill>(p, kk)) >= 0; ++kk) {
        Item it;
        if (!resolve_item<kPrefill, kMassMode>(p, idx, it)) continue;
        // The Q buffers are free once every MMA of the previous item has
        // completed (q_empty), its last QK included.  Its first PV was issued
        // only after the epilogue two items back had released O (o_free), so
        // the BOS buffer of this parity, last read by that epilogue, is free
        // as well.
        if (items_done > 0 && !mbar_wait(&sh.q_empty, (items_done - 1) & 1)) { ok = false; break; }
        const int n_bos = !kPrefill ? 0 : it.kind == kChunk ? 2 : 1;   // K (and V) rows
        mbar_arrive_expect_tx(&sh.q_full, (it.has_b ? 2 * q_bytes : q_bytes) + n_bos * L::kBosBox);
        for (int x = 0; x < (it.has_b ? 2 : 1); ++x)
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(smem + (x ? L::kQ1 : L::kQ0) + pn * kPanelBytes, &p.tm_q[it.q_map],
                        &sh.q_full, pn * 64, it.g * G,
                        static_cast<int>(it.q_row0) + (it.ta + x) * p.Tq);
        uint8_t* bos = smem + L::kBos0 + (items_done & 1) * 2 * L::kBosBox;
        for (int kv = 0; kv < n_bos; ++kv)
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d(bos + kv * L::kBosBox + pn * 2048, kv ? &p.tm_v[0][0] : &p.tm_k[0][0],
                        &sh.q_full, pn * 64, it.g, it.chunk * p.chunk_rows);
        ++items_done;
      }
      if (!ok) atomicOr(&sh.failed, 8);
      if (items_done > 0) mbar_wait(&sh.q_full, (items_done - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t ring_ctr = 0, tile_ctr = 0;
      uint32_t p_ph[2] = {0, 0};
      int items_done = 0;
      bool ok = true;
      constexpr uint32_t idesc_o = idesc_bf16(kBlockM, D, false, true);
      // Base descriptors: Q tile 0 and K in ring slot 0 (K-major), V in ring
      // slot 0 (MN-major, 64-column panels kPanelBytes apart).
      const uint64_t desc_q0 = sw128_desc(s_base + L::kQ0, 16, 1024);
      const uint64_t desc_ring_k = sw128_desc(s_base + L::kRing0, 16, 1024);
      const uint64_t desc_ring_v = sw128_desc(s_base + L::kRing0, kPanelBytes, 1024);
      for (int kk = 0, idx; ok && (idx = nth_item<kPrefill>(p, kk)) >= 0; ++kk) {
        Item it;
        if (!resolve_item<kPrefill, kMassMode>(p, idx, it)) continue;
        const bool with_pv = it.kind != kWindow && it.kind != kMass;
        const int nx = it.has_b ? 2 : 1;
        bool ofree_done[2] = {items_done == 0, items_done == 0};
        bool ofull_sent[2] = {false, false};
        auto wait_ofree = [&](int x) -> bool {
          if (ofree_done[x]) return true;
          ofree_done[x] = true;
          const bool r = mbar_wait(&sh.o_free[x], (items_done - 1) & 1);
          tc_fence_after_sync();
          return r;
        };
        if (!mbar_wait(&sh.q_full, items_done & 1)) { ok = false; break; }
        // QK of one tile into S_x from the K slot `ks`.  A descriptor's
        // address field holds (address >> 4) in 14 bits and every operand
        // here lies in this CTA's shared memory, so the descriptor of base +
        // offset is the base descriptor plus offset >> 4: the loop adds
        // constants to descriptors made once per kernel.
        auto issue_qk = [&](int x, int ng, uint32_t ks) {
          const uint64_t a0 = desc_q0 + (x ? (L::kTileBytes >> 4) : 0u);
          const uint64_t b0 = desc_ring_k + ks * (L::kTileBytes >> 4);
          const uint32_t idesc_s = ng == kGroupsPerTile
                                       ? idesc_bf16(kBlockM, kBlockN, false, false)
                                       : idesc_bf16(kBlockM, ng * kGroupRows, false, false);
          const uint32_t d_s = tmem + tmem_s_col(x);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4;
            mma_bf16_ss(d_s, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&sh.s_full[x]);
        };
        // Rows of an unshifted ragged group past its (shorter than 16 rows)
        // segment may hold anything (another slot, padding): zero them in V so
        // that 0 * v stays 0 in PV.
        auto fix_v = [&](const TileMeta& m, uint32_t vs) {
          uint8_t* v_tile = smem + L::kRing0 + vs * L::kTileBytes;
          bool wrote = false;
          for (int grp = 0; grp < m.ngroups; ++grp) {
            const uint32_t w = grp < 4 ? m.nvalid_lo : m.nvalid_hi;
            const int nv = static_cast<int>((w >> (8 * (grp & 3))) & 0xFFu);
            if (nv & kShifted) continue;   // all 16 rows belong to the segment
            wrote = wrote || nv < kGroupRows;
            for (int r = nv; r < kGroupRows; ++r)
              for (int pn = 0; pn < D / 64; ++pn) {
                uint4* dst = reinterpret_cast<uint4*>(v_tile + pn * kPanelBytes + (grp * kGroupRows + r) * 128);
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) dst[c16] = make_uint4(0u, 0u, 0u, 0u);
              }
          }
          if (wrote) fence_proxy_async_smem();
        };
        auto issue_pv = [&](int x, int ng, uint32_t vs, bool first) {
          const uint64_t v0 = desc_ring_v + vs * (L::kTileBytes >> 4);
          const uint32_t d_o = tmem + tmem_o_col(x), a_p = tmem + tmem_s_col(x);
          if (ng == kGroupsPerTile) {
#pragma unroll
            for (int kk = 0; kk < kGroupsPerTile; ++kk)
              mma_bf16_ts(d_o, a_p + kk * 8, v0 + kk * (2048 >> 4), idesc_o,
                          (!first || kk > 0) ? 1u : 0u);
          } else {
            for (int kk = 0; kk < ng; ++kk)
              mma_bf16_ts(d_o, a_p + kk * 8, v0 + kk * (2048 >> 4), idesc_o,
                          (!first || kk > 0) ? 1u : 0u);
          }
        };
        // Tile 0.
        int ms = tile_ctr % kRing;
        if (!mbar_wait(&sh.meta_full[ms], (tile_ctr / kRing) & 1)) { ok = false; break; }
        TileMeta mt = sh.meta[ms];
        mbar_arrive(&sh.meta_empty[ms]);
        ++tile_ctr;
        if (mt.ngroups > 0) {
          uint32_t ks = ring_ctr % kRing;
          if (!mbar_wait(&sh.ring_full[ks], (ring_ctr / kRing) & 1)) { ok = false; break; }
          tc_fence_after_sync();
          for (int x = 0; x < nx; ++x) issue_qk(x, mt.ngroups, ks);
          mma_commit(&sh.ring_empty[ks]);
          ++ring_ctr;
          for (int j = 0;; ++j) {
            const bool last = mt.last != 0;
            const int ng = mt.ngroups;
            uint32_t vs = 0;
            if (with_pv) {
              vs = ring_ctr % kRing;
              if (!mbar_wait(&sh.ring_full[vs], (ring_ctr / kRing) & 1)) { ok = false; break; }
              ++ring_ctr;
              if (mt.fix_v) fix_v(mt, vs);
            }
            TileMeta mn = mt;
            uint32_t ks_next = 0;
            if (!last) {
              ms = tile_ctr % kRing;
              if (!mbar_wait(&sh.meta_full[ms], (tile_ctr / kRing) & 1)) { ok = false; break; }
              mn = sh.meta[ms];
              mbar_arrive(&sh.meta_empty[ms]);
              ++tile_ctr;
              ks_next = ring_ctr % kRing;
            }
            for (int x = 0; x < nx; ++x) {
              // softmax x finished tile j (S_x read, P_x written)
              if (!mbar_wait(&sh.p_full[x], p_ph[x])) { ok = false; break; }
              p_ph[x] ^= 1u;
              tc_fence_after_sync();
              if (with_pv) {
                if (j == 0 && !wait_ofree(x)) { ok = false; break; }
                issue_pv(x, ng, vs, j == 0);
                if (last) {
                  // O_x is final once this PV completes: its epilogue need
                  // not wait for the other tile's last PV.
                  mma_commit(&sh.o_full[x]);
                  ofull_sent[x] = true;
                }
              }
              if (!last) {
                if (x == 0 && !mbar_wait(&sh.ring_full[ks_next], (ring_ctr / kRing) & 1)) {
                  ok = false;
                  break;
                }
                tc_fence_after_sync();
                issue_qk(x, mn.ngroups, ks_next);
              }
            }
            if (!ok) break;
            if (with_pv) mma_commit(&sh.ring_empty[vs]);
            if (last) break;
            mma_commit(&sh.ring_empty[ks_next]);
            ++ring_ctr;
            mt = mn;
          }
          if (!ok) break;
        }
        // Every item waits for the previous item's epilogue of both tiles
        // exactly once (before its first PV into O_x, else here), so the
        // o_free phases are consumed in order.
        for (int x = 0; ok && x < 2; ++x)
          if (!wait_ofree(x)) ok = false;
        if (!ok) break;
        // O_x of this item is final once every MMA issued so far completes
        // (one o_full phase per tile and item, committed early above after
        // the tile's last PV).
        for (int x = 0; x < 2; ++x)
          if (!ofull_sent[x]) mma_commit(&sh.o_full[x]);
        mma_commit(&sh.q_empty);
        ++items_done;
      }
      if (!ok) atomicOr(&sh.failed, 2);
      mma_commit(&sh.drain);
      mbar_wait(&sh.drain, 0);
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 8) {
    // ------------------------------------------------- softmax warpgroups --
    const int x = warp >= kSoftmaxWarp0 + 4 ? 1 : 0;   // query tile of this warpgroup
    const int quarter = warp & 3;         // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;  // tile row of this thread
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = tmem_s_col(x), o_col = tmem_o_col(x);
    const float scale = p.scale_log2;
    uint32_t tile_ctr = 0, ring_ctr = 0, s_ph = 0;
    int items_done = 0;
    bool ok = true;
    for (int kk = 0, idx; ok && (idx = nth_item<kPrefill>(p, kk)) >= 0; ++kk) {
      Item it;
      if (!resolve_item<kPrefill, kMassMode>(p, idx, it)) continue;
      const bool with_pv = it.kind != kWindow && it.kind != kMass;
      const bool active = x == 0 || it.has_b;
      float m_used = -INFINITY, l_sum = 0.0f;
      // Chunk-mass items: this row's probability mass in each of the item's
      // chunks (segments), accumulated group by group.
      float seg_mass[kMassChunks];
#pragma unroll
      for (int c = 0; c < kMassChunks; ++c) seg_mass[c] = 0.0f;
      if constexpr (kMassMode) {
        // Mass items: every probability is taken at the step's normaliser,
        // p = 2^(s * scale - lse * log2(e)), so the row's reference is its
        // lse and never moves (rows past the block, or with no finite lse,
        // get +inf: their probabilities are 0).
        const int t_local = row / G;
        const int t = (it.ta + x) * p.Tq + t_local;
        float b = INFINITY;
        if (active && row < q_rows && t < it.n_t) {
          const float lse_row =
              p.mass_lse[(it.q_row0 + t) * p.Hq + it.g * G + (row - t_local * G)];
          if (isfinite(lse_row)) b = lse_row * kLog2e;
        }
        m_used = b;
      }
      float s_bos = 0.0f;   // prefill: this row's BOS logit q . k0 (unscaled)
      int n_seen = 0;
      const uint8_t* bos = smem + L::kBos0 + (items_done & 1) * 2 * L::kBosBox;
      // q . k0 from the Q tile in shared memory and the BOS K row, in fp32.
      // Both arrived by TMA on q_full (phase items_done, complete since the
      // first QK ran; the next phase needs this item's last P first).
      auto bos_logit = [&]() -> float {
        if (!mbar_wait_warp(&sh.q_full, items_done & 1)) ok = false;
        const uint8_t* qt = smem + (x ? L::kQ1 : L::kQ0);
        float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll 4
        for (int c8 = 0; c8 < D / 8; ++c8) {
          const uint4 qv = *reinterpret_cast<const uint4*>(qt + sw128_offset(row, c8 * 8, kBlockM));
          const uint4 kv = *reinterpret_cast<const uint4*>(bos + sw128_offset(0, c8 * 8, 16));
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc0 = fmaf(__uint_as_float(qw[i] << 16), __uint_as_float(kw[i] << 16), acc0);
            acc1 = fmaf(__uint_as_float(qw[i] & 0xFFFF0000u), __uint_as_float(kw[i] & 0xFFFF0000u), acc1);
          }
        }
        return acc0 + acc1;
      };
      for (;;) {
        const int ms = tile_ctr % kRing;
        if (!mbar_wait_warp(&sh.meta_full[ms], (tile_ctr / kRing) & 1)) { ok = false; break; }
        const TileMeta meta = sh.meta[ms];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.meta_empty[ms]);
        ++tile_ctr;
        if (meta.ngroups == 0) break;
        ring_ctr += with_pv ? 2 : 1;
        ++n_seen;
        if (!active) {
          if (meta.last) break;
          continue;
        }
        if (!mbar_wait_warp(&sh.s_full[x], s_ph)) { ok = false; break; }
        s_ph ^= 1u;
        tc_fence_after_sync();
        const int ncol = meta.ngroups * kGroupRows;
        const bool full = meta.ngroups == kGroupsPerTile && meta.nvalid_lo == 0x10101010u &&
                          meta.nvalid_hi == 0x10101010u;
        auto nv_of = [&](int grp) -> int {
          const uint32_t w = grp < 4 ? meta.nvalid_lo : meta.nvalid_hi;
          return static_cast<int>((w >> (8 * (grp & 3))) & 0xFFu);
        };

        // Ragged tiles: logits of key rows outside a group's valid rows become
        // -inf (their exp2 is then 0): the rows past the count, or for a
        // shifted group the leading rows that repeat the previous group's keys.
        // valid16(code): bit i set when row i of the group is one of its keys.
        auto valid16 = [](int code) -> uint32_t {
          if (code & kShifted) return (0xFFFFu << (kGroupRows - (code & 0x1f))) & 0xFFFFu;
          return (1u << code) - 1u;   // code 16: all rows; 0: none
        };
        // Masks the groups of this half whose bit is set in `which` (a
        // warp-uniform 4-bit set); each group is one uniform branch, so tiles
        // with one ragged group pay for that group only.
        auto mask_half = [&](uint32_t (&sr)[2][32], int half, uint32_t which) {
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            if (which & (1u << gq)) {
              const uint32_t vm = valid16(nv_of(half * 4 + gq));
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (!((vm >> i) & 1u)) sr[gq >> 1][(gq & 1) * 16 + i] = __float_as_uint(-INFINITY);
            }
          }
        };
        // Groups that need masking (not 16 keys), per half.
        uint32_t rag2 = 0;
        if (!full) {
#pragma unroll
          for (int g = 0; g < kGroupsPerTile; ++g)
            if (nv_of(g) != kGroupRows) rag2 |= 1u << g;
        }

        // One pass over the tile, 64 columns (two TMEM loads) at a time: the
        // masked logits, their max, the rescale decision, then probabilities
        // relative to m_used -> bf16 pairs in TMEM columns [32 half, 32 half
        // + 32) of S_x (over logits already read) and the fp32 row sum.
        // A half whose max exceeds m_used by more than the threshold moves
        // m_used (per row; alpha = 1 for the warp's other rows, as the TMEM
        // accesses are warp-collective) and rescales what was summed against
        // the old reference: l, O (complete here: s_full covers PV(j-1)) and,
        // in the second half, the first half's P.  Masked logits are -inf:
        // they add nothing to the max or the sum.
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          if (half * 64 < ncol) {
            uint32_t sr[2][32];
            tmem_ld32(lane_base + s_col + half * 64, sr[0]);
            tmem_ld32(lane_base + s_col + half * 64 + 32, sr[1]);
            tmem_ld_wait(sr[0]);
            reg_fence(sr[1]);
            const uint32_t m2 = (rag2 >> (4 * half)) & 0xFu;
            if (m2) mask_half(sr, half, m2);
            if constexpr (!kMassMode) {
              float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const int a = (i >> 1) & 1;
                mx[a] = max3(mx[a], __uint_as_float(sr[0][i]), __uint_as_float(sr[0][i + 1]));
                mx[2 + a] = max3(mx[2 + a], __uint_as_float(sr[1][i]), __uint_as_float(sr[1][i + 1]));
              }
              const float m_half = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale;
              const bool mine = m_half > m_used + kRescaleThreshold;
              if (__any_sync(0xFFFFFFFFu, mine)) {
                const float m_new = mine ? m_half : m_used;
                const float alpha = mine ? ex2_approx(m_used - m_new) : 1.0f;
                if (n_seen > 1 && with_pv) {
#pragma unroll 1
                  for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o0[32];
                    tmem_ld32(lane_base + o_col + ch * 32, o0);
                    tmem_ld_wait(o0);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
                    tmem_st32(lane_base + o_col + ch * 32, o0);
                  }
                }
                if (half == 1 && with_pv) {
                  uint32_t p0[32];
                  tmem_st_wait();   // the first half's P is in TMEM
                  tmem_ld32(lane_base + s_col, p0);
                  tmem_ld_wait(p0);
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    p0[i] = pack_bf16x2(__uint_as_float(p0[i] << 16) * alpha,
                                        __uint_as_float(p0[i] & 0xFFFF0000u) * alpha);
                  tmem_st32(lane_base + s_col, p0);
                }
                l_sum *= alpha;
                m_used = m_new;
              }
            }
            const float neg_m = -m_used;
            const uint64_t scale2 = f2_pack(scale, scale), neg_m2 = f2_pack(neg_m, neg_m);
            uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
            uint64_t gsum2[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f),
                                 f2_pack(0.f, 0.f)};   // mass items: per 16-key group
            uint32_t packed[32];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float xa0, xa1, xb0, xb1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[0][i]), __uint_as_float(sr[0][i + 1])),
                               scale2, neg_m2), xa0, xa1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[1][i]), __uint_as_float(sr[1][i + 1])),
                               scale2, neg_m2), xb0, xb1);
              const float a0 = ex2_approx(xa0), a1 = ex2_approx(xa1);
              const float b0 = ex2_approx(xb0), b1 = ex2_approx(xb1);
              if constexpr (kMassMulti) {
                gsum2[i >> 4] = f2_add(gsum2[i >> 4], f2_pack(a0, a1));
                gsum2[2 + (i >> 4)] = f2_add(gsum2[2 + (i >> 4)], f2_pack(b0, b1));
              } else {
                sum2[0] = f2_add(sum2[0], f2_pack(a0, a1));
                sum2[1] = f2_add(sum2[1], f2_pack(b0, b1));
                packed[i >> 1] = pack_bf16x2(a0, a1);
                packed[16 + (i >> 1)] = pack_bf16x2(b0, b1);
              }
            }
            if constexpr (kMassMulti) {
              // Each group's sum goes to its chunk (segment) of the item.
#pragma unroll
              for (int gq = 0; gq < 4; ++gq) {
                float g0, g1;
                f2_unpack(gsum2[gq], g0, g1);
                const float gs = g0 + g1;
                const uint32_t seg =
                    (static_cast<uint32_t>(meta.fix_v) >> (4 * (half * 4 + gq))) & 0xFu;
#pragma unroll
                for (int c = 0; c < kMassChunks; ++c)
                  seg_mass[c] += seg == static_cast<uint32_t>(c) ? gs : 0.0f;
              }
            }
            if (with_pv) tmem_st32(lane_base + s_col + half * 32, packed);
            float sum[4];
            f2_unpack(sum2[0], sum[0], sum[1]);
            f2_unpack(sum2[1], sum[2], sum[3]);
            l_sum += (sum[0] + sum[1]) + (sum[2] + sum[3]);
          }
        }
        if (with_pv) tmem_st_wait();
        // The BOS logit, while the Q tile is certainly resident: before the
        // item's last P is handed over (after it the last PV may complete and
        // the next item's Q arrive), else right after the first tile's P.
        const bool bos_now = kPrefill && n_seen == 1;
        if (bos_now && meta.last) s_bos = bos_logit();
        // Every lane's TMEM reads of S and stores of P are complete (waited
        // above); the warp sync orders them before lane 0's arrival.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full[x]);
        if (bos_now && !meta.last) s_bos = bos_logit();
        if (meta.last) break;
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue --
      if (!mbar_wait_warp(&sh.o_full[x], items_done & 1)) { ok = false; break; }
      tc_fence_after_sync();
      // Prefill: fold the BOS key into (m, l) and, through o_alpha / o_bos,
      // into the output row (every prefill item has content keys, so s_bos
      // was computed).
      float o_alpha = 1.0f, o_bos = 0.0f;
      if constexpr (kPrefill) {
        const float sb = s_bos * scale;
        const float m_new = fmaxf(m_used, sb);
        o_alpha = ex2_approx(m_used - m_new);
        o_bos = ex2_approx(sb - m_new);
        l_sum = l_sum * o_alpha + o_bos;
        m_used = m_new;
      }
      if constexpr (kMassMode) {
        // This warp's rows' mass over each chunk of the item (its row sum
        // when the item holds one chunk): one partial per (item, chunk,
        // query tile, warp), summed per chunk in a fixed order by the
        // mass-sum kernel.
        const int t_local = row / G;
        const int t = (it.ta + x) * p.Tq + t_local;
        const bool row_in = active && row < q_rows && t < it.n_t;
        if constexpr (kMassMulti) {
          const int nchunks = it.k1 - it.k0;
#pragma unroll
          for (int c = 0; c < kMassChunks; ++c) {
            if (c < nchunks) {
              float v = row_in ? seg_mass[c] : 0.0f;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
              if (lane == 0)
                p.mass_part[(static_cast<long long>(idx) * p.mass_chunks + c) * 8 + x * 4 +
                            quarter] = v;
            }
          }
        } else {
          float v = row_in ? l_sum : 0.0f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
          if (lane == 0) p.mass_part[static_cast<long long>(idx) * 8 + x * 4 + quarter] = v;
        }
      }
      if (!kMassMode && active) {
        const int t_local = row / G;
        const int jj = row - t_local * G;
        const int t = (it.ta + x) * p.Tq + t_local;
        const bool row_ok = row < q_rows && t < it.n_t;
        const int head = it.g * G + jj;
        if (it.kind == kWindow) {
          // The window-score kernel's per-column constant b = m + log2(l)
          // (+inf when the row saw no key, so its probabilities are 0).  With
          // the window keys in the denominator, their log2-sum-exp is added:
          // b = log2(2^b + 2^b_self).
          if (row_ok) {
            float b = l_sum > 0.0f ? m_used + log2f(l_sum) : -INFINITY;
            if (p.win_self_b != nullptr) {
              const float bw = p.win_self_b[static_cast<long long>(t) * p.Hq + head];
              const float hi = fmaxf(b, bw), lo = fminf(b, bw);
              b = hi + log2f(1.0f + ex2_approx(lo - hi));
            }
            p.win_b[(static_cast<long long>(it.chunk) * p.Hkv + it.g) * p.win_stride + t * G + jj] =
                b == -INFINITY ? INFINITY : b;
          }
        } else {
          const long long tok = it.q_row0 + t;
          const bool final_out = it.kind == kChunk || p.n_splits == 1;
          const float inv_l = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
          bf16* const row_dst =
              final_out ? p.out + (tok * p.Hq + head) * D
                        : p.part_acc +
                              ((static_cast<long long>(it.split) * p.total_lq + tok) * p.Hq + head) * D;
          // Normalised bf16 row: the output, or one split's partial O / l
          // (the merge weighs it by the split's l and max).  Each lane
          // writes its own row; whole 32-byte sectors where the destination
          // allows it (the workspace always does).
          const uint8_t* v_bos = bos + L::kBosBox;
          auto emit32 = [&](int ch, const uint32_t (&o)[32]) {
            uint32_t packed[16];
            if (kPrefill && it.kind == kChunk) {
              // (O 2^(m - M) + 2^(s0 - M) v0) / l' over these 32 columns.
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const uint4 vv = *reinterpret_cast<const uint4*>(v_bos + sw128_offset(0, ch * 32 + q4 * 8, 16));
                const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int e = 8 * q4 + 2 * i;
                  const float lo = fmaf(__uint_as_float(o[e]), o_alpha, o_bos * __uint_as_float(vw[i] << 16));
                  const float hi = fmaf(__uint_as_float(o[e + 1]), o_alpha,
                                        o_bos * __uint_as_float(vw[i] & 0xFFFF0000u));
                  packed[4 * q4 + i] = pack_bf16x2(lo * inv_l, hi * inv_l);
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                packed[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                        __uint_as_float(o[2 * i + 1]) * inv_l);
            }
            bf16* dst = row_dst + ch * 32;
            if (!final_out || p.out_v8) {
#pragma unroll
              for (int q8 = 0; q8 < 2; ++q8)
                st_global_v8(dst + q8 * 16, packed[8 * q8], packed[8 * q8 + 1], packed[8 * q8 + 2],
                             packed[8 * q8 + 3], packed[8 * q8 + 4], packed[8 * q8 + 5],
                             packed[8 * q8 + 6], packed[8 * q8 + 7]);
            } else {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                reinterpret_cast<uint4*>(dst)[q4] = make_uint4(
                    packed[4 * q4], packed[4 * q4 + 1], packed[4 * q4 + 2], packed[4 * q4 + 3]);
            }
          };
          // 64 columns of O per TMEM round trip.
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ch += 2) {
            uint32_t o0[32], o1[32];
            if (n_seen > 0) {
              tmem_ld32(lane_base + o_col + ch * 32, o0);
              tmem_ld32(lane_base + o_col + ch * 32 + 32, o1);
              tmem_ld_wait(o0);
              reg_fence(o1);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o0[i] = o1[i] = 0u;
            }
            if (!row_ok) continue;
            emit32(ch, o0);
            emit32(ch + 1, o1);
          }
          if (row_ok && it.kind == kDecode) {
            if (p.n_splits == 1) {
              if (p.lse != nullptr)
                p.lse[tok * p.Hq + head] =
                    l_sum > 0.0f ? (m_used + log2f(l_sum)) * kLn2 : -INFINITY;
            } else {
              const long long idx2 =
                  (static_cast<long long>(it.split) * p.total_lq + tok) * p.Hq + head;
              p.part_m[idx2] = m_used;
              p.part_l[idx2] = l_sum;
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.o_free[x]);
      ++items_done;
    }
    if (!ok) atomicOr(&sh.failed, 4);
  }

  tc_fence_before_sync();
  __syncthreads();
  // Only now may the next kernel's CTAs be scheduled: launched earlier they
  // would sit on the SMs (registers, warp slots) while this grid still works.
  grid_dependents_launch();
  if (tid == 0 && sh.failed != 0) raise_dev_err(p.dev_err, PFD_DEVERR_TIMEOUT);
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t attention_smem_bytes(int D, bool prefill) {
  if (D == 64) return 1024 + (prefill ? Layout<64>::kTotalPrefill : Layout<64>::kTotalDecode);
  return 1024 + (prefill ? Layout<128>::kTotalPrefill : Layout<128>::kTotalDecode);
}

template <int D, bool kPrefill, bool kMassMode, bool kMassMulti = false>
cudaError_t launch_attention_t(const AttnParams& p, int grid, size_t smem, cudaStream_t stream) {
  const cudaError_t err = ensure_smem_limit(
      reinterpret_cast<const void*>(attention_kernel<D, kPrefill, kMassMode, kMassMulti>),
      static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  return launch_pdl(attention_kernel<D, kPrefill, kMassMode, kMassMulti>, dim3(grid),
                    dim3(kThreads), smem, stream, p);
}

cudaError_t launch_attention(const AttnParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0 || p.n_items <= 0) return cudaSuccess;
  const bool prefill = p.mode == kModePrefill;
  const size_t smem = attention_smem_bytes(p.D, prefill);
  if (p.mode == kModeMass) {
    if (p.mass_chunks > 1)
      return p.D == 64 ? launch_attention_t<64, false, true, true>(p, grid, smem, stream)
                       : launch_attention_t<128, false, true, true>(p, grid, smem, stream);
    return p.D == 64 ? launch_attention_t<64, false, true>(p, grid, smem, stream)
                     : launch_attention_t<128, false, true>(p, grid, smem, stream);
  }
  if (p.D == 64)
    return prefill ? launch_attention_t<64, true, false>(p, grid, smem, stream)
                   : launch_attention_t<64, false, false>(p, grid, smem, stream);
  return prefill ? launch_attention_t<128, true, false>(p, grid, smem, stream)
                 : launch_attention_t<128, false, false>(p, grid, smem, stream);
}

}  // namespace pfd
