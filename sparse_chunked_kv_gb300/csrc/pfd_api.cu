// C ABI of libpfd: argument checks, TMA tensor maps, workspace layout, split
// planning and kernel launches.  Declarations and contracts: include/pfd.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pfd_internal.cuh"

namespace pfd {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// 3-D map over a [rows, heads, D] bf16 tensor with a box of box_rows rows x
// box_heads heads x 64 columns (128 B), 128-byte swizzle; out-of-range rows
// read as zero.
bool encode_map(CUtensorMap* map, const void* base, long long rows, int heads, int D, int box_heads,
                int box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || base == nullptr || rows <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(heads) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A tensor map depends only on (base, rows, heads, D, box), so encoded maps
// are kept in a small process-wide table: a decode loop that calls with the
// same buffers step after step encodes each map once.  Round-robin
// replacement; the table is guarded by a mutex.
struct MapKey {
  const void* base;
  long long rows;
  int heads, D, box_heads, box_rows;
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && heads == o.heads && D == o.D &&
           box_heads == o.box_heads && box_rows == o.box_rows;
  }
};

bool make_map(CUtensorMap* map, const void* base, long long rows, int heads, int D, int box_heads,
              int box_rows) {
  constexpr int kEntries = 128;
  static std::mutex mu;
  static MapKey keys[kEntries];
  static CUtensorMap maps[kEntries];
  static int used = 0, next = 0;
  const MapKey key{base, rows, heads, D, box_heads, box_rows};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == key) {
        *map = maps[i];
        return true;
      }
  }
  if (!encode_map(map, base, rows, heads, D, box_heads, box_rows)) return false;
  std::lock_guard<std::mutex> lock(mu);
  const int slot = used < kEntries ? used++ : (next++ % kEntries);
  keys[slot] = key;
  maps[slot] = *map;
  return true;
}

// K or V maps of one tensor (slot t of maps[level][t]): boxes of 16, 32, 64
// and 128 rows.
bool make_kv_maps(CUtensorMap (*maps)[2], int t, const void* base, long long rows, int heads,
                  int D) {
  for (int lv = 0; lv < kBoxLevels; ++lv)
    if (!make_map(&maps[lv][t], base, rows, heads, D, 1, kGroupRows << lv)) return false;
  return true;
}

void copy_kv_maps(CUtensorMap (*maps)[2], int to, int from) {
  for (int lv = 0; lv < kBoxLevels; ++lv) maps[lv][to] = maps[lv][from];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct PrefillWs {
  size_t win_b, part_scores, win_self, total;
  int win_stride;
};

// Window statistics [N, Hkv, W*G rounded up to 32], per-KV-group partial
// scores [N, Hkv, C+1] and the window rows' statistics over the window's own
// keys [W, Hq] (used when those keys are in the denominator).
PrefillWs prefill_ws_layout(int N, int C, int W, int Hq, int Hkv) {
  PrefillWs w;
  w.win_stride = (W * (Hq / Hkv) + 31) & ~31;
  const size_t stats = static_cast<size_t>(N) * Hkv * w.win_stride * sizeof(float);
  w.win_b = 0;
  w.part_scores = align256(stats);
  const size_t ps = W > 0 ? static_cast<size_t>(N) * Hkv * (C + 1) * sizeof(float) : 0;
  w.win_self = w.part_scores + align256(ps);
  w.total = w.win_self + align256(static_cast<size_t>(W) * Hq * sizeof(float));
  return w;
}

bool shapes_ok(int Hq, int Hkv, int D) {
  return Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && (D == 64 || D == 128);
}

pfd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PFD_OK : PFD_ERR_CUDA; }

struct DecodeWs {
  size_t part_m, part_l, part_acc, total;
};

DecodeWs decode_ws_layout(int n_splits, long long total_lq, int Hq, int D) {
  DecodeWs w{0, 0, 0, 0};
  if (n_splits <= 1) return w;
  const size_t ml = static_cast<size_t>(n_splits) * total_lq * Hq * sizeof(float);
  w.part_m = 0;
  w.part_l = align256(ml);
  w.part_acc = w.part_l + align256(ml);
  w.total = w.part_acc + align256(ml / sizeof(float) * D * 2);   // bf16 partials
  return w;
}

bool decode_host_ok(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host) {
  if (batch < 1 || cu_lq_host == nullptr || cu_k_host == nullptr) return false;
  if (cu_lq_host[0] != 0 || cu_k_host[0] != 0) return false;
  for (int b = 0; b < batch; ++b)
    if (cu_lq_host[b + 1] < cu_lq_host[b] || cu_k_host[b + 1] < cu_k_host[b]) return false;
  return cu_lq_host[batch] >= 1;
}

constexpr int kMaxSplits = 64;

// Chunked prefill (pfd_chunk_prefill, pfd_chunk_prefill_ex,
// pfd_chunk_prefill_layers, pfd_chunk_prefill_batch): L stacked layers (or
// requests) of N chunks (layer l's chunk j is chunk l*N + j of the stacked
// tensors, its window rows l*W..; its slot slot_row[j] in its own pool
// l*pool_rows rows further, or with shared_pool slot_row[l*N + j] in the
// one pool); per_kv_head ranks per (chunk, KV head); k_win (may be null;
// L == 1) puts the window keys into the window rows' softmax denominator.
pfd_status prefill_impl(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                        const pfd_bf16* q_win, int L, int N, int C, int W, int Hq, int Hkv, int D,
                        int B,
                        float sm_scale, pfd_bf16* out, float* scores, int32_t* kept_idx,
                        pfd_bf16* pool_k, pfd_bf16* pool_v, int64_t pool_rows,
                        const int32_t* slot_row, pfd_chunk_entry* table, int32_t* dev_err,
                        void* workspace, size_t workspace_bytes, bool per_kv_head,
                        const pfd_bf16* k_win, pfd_stream_t stream, bool shared_pool = false) {
  if (L < 1 || N < 1 || C < 1 || W < 0 || B < 0 || B > C) return PFD_ERR_INVALID_ARG;
  if (k_win != nullptr && L != 1) return PFD_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return PFD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return PFD_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (C > 8192 || G > kBlockM || W > 256 || static_cast<long long>(W) * G > 512)
    return PFD_ERR_UNSUPPORTED;
  if (static_cast<long long>(L) * N * (C + 1) * Hq * D >= (1ll << 40) ||
      static_cast<long long>(L) * N * (C + 1) >= (1ll << 31) ||
      static_cast<long long>(L) * N >= (1ll << 24))
    return PFD_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out || !scores || !pool_k || !pool_v || !slot_row || !table)
    return PFD_ERR_INVALID_ARG;
  if (B > 0 && !kept_idx) return PFD_ERR_INVALID_ARG;
  if (W > 0 && !q_win) return PFD_ERR_INVALID_ARG;
  if (k_win != nullptr && (W == 0 || !aligned16(k_win))) return PFD_ERR_INVALID_ARG;
  if (pool_rows < B + 1 || pool_rows >= (1ll << 31)) return PFD_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(pool_k) ||
      !aligned16(pool_v) || (W > 0 && !aligned16(q_win)))
    return PFD_ERR_INVALID_ARG;
  const int NL = L * N;   // chunks of all layers
  const PrefillWs ws = prefill_ws_layout(NL, C, W, Hq, Hkv);
  if (workspace_bytes < ws.total || (ws.total > 0 && workspace == nullptr) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PFD_ERR_INVALID_ARG;
  const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  const long long rows = static_cast<long long>(NL) * (C + 1);

  const int Tq = kBlockM / G;
  AttnParams ap;
  std::memset(&ap, 0, sizeof(ap));
  if (!make_kv_maps(ap.tm_k, 0, k, rows, Hkv, D) || !make_kv_maps(ap.tm_v, 0, v, rows, Hkv, D) ||
      !make_map(&ap.tm_q[0], q, rows, Hq, D, G, Tq))
    return PFD_ERR_CUDA;
  copy_kv_maps(ap.tm_k, 1, 0);
  copy_kv_maps(ap.tm_v, 1, 0);
  if (W > 0) {
    if (!make_map(&ap.tm_q[1], q_win, static_cast<long long>(L) * W, Hq, D, G, Tq))
      return PFD_ERR_CUDA;
  } else {
    ap.tm_q[1] = ap.tm_q[0];
  }
  ap.Tq = Tq;
  ap.q = reinterpret_cast<const bf16*>(q);
  ap.q_win = reinterpret_cast<const bf16*>(q_win);
  ap.out = reinterpret_cast<bf16*>(out);
  ap.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  ap.win_b = reinterpret_cast<float*>(wsb + ws.win_b);
  ap.win_stride = ws.win_stride;
  ap.dev_err = dev_err;
  ap.mode = kModePrefill;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.G = G;
  ap.D = D;
  ap.n_chunks = NL;
  ap.layer_chunks = N;
  ap.chunk_rows = C + 1;
  ap.n_win = W;
  ap.mt_chunk = ceil_div(C + 1, Tq);
  ap.mt_win = W > 0 ? ceil_div(W, Tq) : 0;
  ap.n_chunk_items = NL * Hkv * ceil_div(ap.mt_chunk, 2);
  ap.n_splits = 1;
  ap.scale_log2 = scale * kLog2e;
  const long long items =
      static_cast<long long>(ap.n_chunk_items) + static_cast<long long>(NL) * Hkv * ceil_div(ap.mt_win, 2);
  if (items >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  ap.n_items = static_cast<int>(items);
  // Every tensor map is encoded before the first launch, so that a failure
  // to encode one launches nothing.
  WinScoreParams wp;
  std::memset(&wp, 0, sizeof(wp));
  wp.k_tiles = ceil_div(C + 1, 128);
  wp.concat = (C + 1 >= 128) ? 1 : 0;
  const long long layer_rows = static_cast<long long>(N) * (C + 1);   // tiles per layer
  const long long ws_items =
      wp.concat ? (layer_rows + 127) / 128 : static_cast<long long>(N) * wp.k_tiles;
  if (ws_items >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  if (W > 0 && !make_map(&wp.tm_qwin, q_win, static_cast<long long>(L) * W, Hq, D, G, W))
    return PFD_ERR_CUDA;
  const int grid = static_cast<int>(std::min<long long>(items, device_sm_count()));
  pfd_status s = PFD_OK;
  if (k_win != nullptr) {
    ap.win_self_b = reinterpret_cast<float*>(wsb + ws.win_self);
    s = from_cuda(launch_window_self_stats(reinterpret_cast<const bf16*>(q_win),
                                           reinterpret_cast<const bf16*>(k_win), W, Hq, Hkv, D,
                                           ap.scale_log2, reinterpret_cast<float*>(wsb + ws.win_self),
                                           st));
    if (s != PFD_OK) return s;
  }
  s = from_cuda(launch_attention(ap, grid, st));
  if (s != PFD_OK) return s;

  if (W > 0) {
    wp.tm_k = ap.tm_k[kBoxLevels - 1][0];
    wp.q_win = ap.q_win;
    wp.win_b = ap.win_b;
    wp.win_stride = ap.win_stride;
    wp.part_scores = reinterpret_cast<float*>(wsb + ws.part_scores);
    wp.n_chunks = N;
    wp.n_layers = L;
    wp.chunk_rows = C + 1;
    wp.n_win = W;
    wp.Hq = Hq;
    wp.Hkv = Hkv;
    wp.G = G;
    wp.D = D;
    wp.n_items = static_cast<int>(ws_items);
    wp.scale_log2 = ap.scale_log2;
    wp.dev_err = dev_err;
    s = from_cuda(launch_window_scores(wp, st));
    if (s != PFD_OK) return s;
  }

  TopBParams tp;
  std::memset(&tp, 0, sizeof(tp));
  tp.part_scores = W > 0 ? reinterpret_cast<const float*>(wsb + ws.part_scores) : nullptr;
  tp.scores = scores;
  tp.kept_idx = kept_idx;
  tp.k = reinterpret_cast<const bf16*>(k);
  tp.v = reinterpret_cast<const bf16*>(v);
  tp.pool_k = reinterpret_cast<bf16*>(pool_k);
  tp.pool_v = reinterpret_cast<bf16*>(pool_v);
  tp.slot_row = slot_row;
  tp.table = table;
  tp.dev_err = dev_err;
  tp.pool_rows = pool_rows;
  tp.layer_pool_rows = pool_rows;
  tp.slot_per_chunk = shared_pool ? 1 : 0;
  tp.layer_chunks = N;
  tp.n_chunks = NL;
  tp.chunk_size = C;
  tp.n_keep = B;
  tp.Hkv = Hkv;
  tp.D = D;
  tp.per_head = per_kv_head ? 1 : 0;
  return from_cuda(launch_topb_compact(tp, st));   // sets the copy splits
}

int plan_splits(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host, int Hq,
                int Hkv, int D, int max_chunk_len, bool self_keys) {
  (void)D;
  if (!decode_host_ok(batch, cu_lq_host, cu_k_host) || !shapes_ok(Hq, Hkv, 128)) return 1;
  const int G = Hq / Hkv;
  if (G > kBlockM) return 1;
  const int Tq = kBlockM / G;
  long long items = 0, keys_max = 0;
  for (int b = 0; b < batch; ++b) {
    const long long lq = cu_lq_host[b + 1] - cu_lq_host[b];
    const long long kb = cu_k_host[b + 1] - cu_k_host[b];
    items += Hkv * (((lq + Tq - 1) / Tq + 1) / 2);   // two query tiles per item
    keys_max = std::max(keys_max, kb * std::max(0, max_chunk_len) + (self_keys ? lq : 0));
  }
  if (items <= 0) return 1;
  const long long sms = device_sm_count();   // one persistent CTA per SM
  int best = 1;
  double best_cost = 1e300;
  const long long max_s = std::max<long long>(1, std::min<long long>(kMaxSplits, (keys_max + kBlockN - 1) / kBlockN));
  for (int S = 1; S <= max_s; ++S) {
    const long long waves = (items * S + sms - 1) / sms;
    const long long tiles = (keys_max + static_cast<long long>(S) * kBlockN - 1) / (static_cast<long long>(S) * kBlockN);
    // an item costs ~2 units per key tile (two query tiles) plus ~3 units of
    // fixed cost (Q load, pipeline fill, epilogue); the merge ~ 2 units
    const double cost = static_cast<double>(waves) * (2.0 * tiles + 3.0) + (S > 1 ? 2.0 : 0.0);
    if (cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

// Decode attention of one step over [selected chunks ; live block when
// self_keys]: pfd_decode_attention (self_keys) and pfd_decode_partial.
pfd_status decode_impl(const pfd_bf16* q, const pfd_bf16* k_self, const pfd_bf16* v_self,
                       const int32_t* cu_lq, const int32_t* cu_lq_host, const pfd_bf16* pool_k,
                       const pfd_bf16* pool_v, int64_t pool_rows, const pfd_chunk_entry* table,
                       int32_t table_len, const int32_t* sel, const int32_t* cu_k,
                       const int32_t* cu_k_host, int batch, int Hq, int Hkv, int D,
                       int max_chunk_len, float sm_scale, bool self_keys, int n_splits,
                       pfd_bf16* out, float* lse, int32_t* dev_err, void* workspace,
                       size_t workspace_bytes, pfd_stream_t stream) {
  if (!decode_host_ok(batch, cu_lq_host, cu_k_host)) return PFD_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return PFD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return PFD_ERR_UNSUPPORTED;
  if (!q || !k_self || !v_self || !cu_lq || !cu_k || !out) return PFD_ERR_INVALID_ARG;
  if (n_splits < 0 || n_splits > kMaxSplits) return PFD_ERR_INVALID_ARG;
  if (Hq / Hkv > kBlockM) return PFD_ERR_UNSUPPORTED;
  for (int b = 0; b < batch; ++b)
    if (cu_k_host[b + 1] - cu_k_host[b] >= kMaxSegments) return PFD_ERR_UNSUPPORTED;
  const int total_lq = cu_lq_host[batch];
  const int total_sel = cu_k_host[batch];
  if (total_sel > 0 && (!pool_k || !pool_v || !table || !sel || pool_rows < 1 || table_len < 1))
    return PFD_ERR_INVALID_ARG;
  if (pool_rows >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_self) || !aligned16(v_self) || !aligned16(out) ||
      (total_sel > 0 && (!aligned16(pool_k) || !aligned16(pool_v))))
    return PFD_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const int S = n_splits > 0 ? n_splits
                             : plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D,
                                           max_chunk_len, self_keys);
  const DecodeWs ws = decode_ws_layout(S, total_lq, Hq, D);
  if (workspace_bytes < ws.total || (ws.total > 0 && workspace == nullptr) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PFD_ERR_INVALID_ARG;
  const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);

  const int Tq = kBlockM / G;
  AttnParams ap;
  std::memset(&ap, 0, sizeof(ap));
  if (!make_kv_maps(ap.tm_k, 1, k_self, total_lq, Hkv, D) ||
      !make_kv_maps(ap.tm_v, 1, v_self, total_lq, Hkv, D) ||
      !make_map(&ap.tm_q[0], q, total_lq, Hq, D, G, Tq))
    return PFD_ERR_CUDA;
  ap.tm_q[1] = ap.tm_q[0];
  if (total_sel > 0) {
    if (!make_kv_maps(ap.tm_k, 0, pool_k, pool_rows, Hkv, D) ||
        !make_kv_maps(ap.tm_v, 0, pool_v, pool_rows, Hkv, D))
      return PFD_ERR_CUDA;
  } else {
    copy_kv_maps(ap.tm_k, 0, 1);
    copy_kv_maps(ap.tm_v, 0, 1);
  }
  ap.Tq = Tq;
  int mt_max = 0;
  for (int b = 0; b < batch; ++b)
    mt_max = std::max(mt_max, ceil_div(cu_lq_host[b + 1] - cu_lq_host[b], Tq));
  ap.q = reinterpret_cast<const bf16*>(q);
  ap.out = reinterpret_cast<bf16*>(out);
  ap.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  ap.lse = lse;
  ap.part_m = S > 1 ? reinterpret_cast<float*>(wsb + ws.part_m) : nullptr;
  ap.part_l = S > 1 ? reinterpret_cast<float*>(wsb + ws.part_l) : nullptr;
  ap.part_acc = S > 1 ? reinterpret_cast<bf16*>(wsb + ws.part_acc) : nullptr;
  ap.table = table;
  ap.sel = sel;
  ap.cu_k = cu_k;
  ap.cu_lq = cu_lq;
  ap.dev_err = dev_err;
  ap.pool_rows = pool_rows;
  ap.table_len = table_len;
  ap.mode = kModeDecode;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.G = G;
  ap.D = D;
  ap.batch = batch;
  ap.mt_max = mt_max;
  ap.n_splits = S;
  ap.total_lq = total_lq;
  ap.total_sel = total_sel;
  ap.self_keys = self_keys ? 1 : 0;
  ap.scale_log2 = scale * kLog2e;
  const long long items = static_cast<long long>(batch) * Hkv * S * ceil_div(mt_max, 2);
  if (items >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  ap.n_items = static_cast<int>(items);
  const int grid = static_cast<int>(std::min<long long>(items, device_sm_count()));
  pfd_status s = from_cuda(launch_attention(ap, grid, st));
  if (s != PFD_OK || S == 1) return s;
  MergeParams mp;
  mp.part_m = ap.part_m;
  mp.part_l = ap.part_l;
  mp.part_acc = ap.part_acc;
  mp.out = ap.out;
  mp.lse = lse;
  mp.n_splits = S;
  mp.total_lq = total_lq;
  mp.Hq = Hq;
  mp.D = D;
  return from_cuda(launch_lse_merge(mp, device_sm_count(), st));
}

}  // namespace
}  // namespace pfd

using namespace pfd;

extern "C" {

int pfd_abi_version(void) { return PFD_ABI_VERSION; }

const char* pfd_status_string(pfd_status s) {
  switch (s) {
    case PFD_OK: return "PFD_OK";
    case PFD_ERR_INVALID_ARG: return "PFD_ERR_INVALID_ARG";
    case PFD_ERR_UNSUPPORTED: return "PFD_ERR_UNSUPPORTED";
    case PFD_ERR_CUDA: return "PFD_ERR_CUDA";
  }
  return "PFD_UNKNOWN_STATUS";
}

size_t pfd_chunk_prefill_workspace(int N, int C, int W, int Hq, int Hkv, int D, int B) {
  (void)D;
  (void)B;
  if (N < 1 || C < 1 || W < 0 || Hq < 1 || Hkv < 1) return 0;
  return prefill_ws_layout(N, C, W, Hq, Hkv).total;
}

pfd_status pfd_chunk_prefill(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                             const pfd_bf16* q_win, int N, int C, int W, int Hq, int Hkv, int D,
                             int B, float sm_scale, pfd_bf16* out, float* scores,
                             int32_t* kept_idx, pfd_bf16* pool_k, pfd_bf16* pool_v,
                             int64_t pool_rows, const int32_t* slot_row, pfd_chunk_entry* table,
                             int32_t* dev_err, void* workspace, size_t workspace_bytes,
                             pfd_stream_t stream) {
  return prefill_impl(q, k, v, q_win, 1, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores, kept_idx,
                      pool_k, pool_v, pool_rows, slot_row, table, dev_err, workspace,
                      workspace_bytes, false, nullptr, stream);
}

pfd_status pfd_chunk_prefill_ex(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                const pfd_bf16* q_win, const pfd_bf16* k_win, int N, int C, int W,
                                int Hq, int Hkv, int D, int B, float sm_scale, int per_kv_head,
                                pfd_bf16* out, float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                size_t workspace_bytes, pfd_stream_t stream) {
  if (per_kv_head != 0 && per_kv_head != 1) return PFD_ERR_INVALID_ARG;
  return prefill_impl(q, k, v, q_win, 1, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores, kept_idx,
                      pool_k, pool_v, pool_rows, slot_row, table, dev_err, workspace,
                      workspace_bytes, per_kv_head != 0, k_win, stream);
}

size_t pfd_chunk_prefill_layers_workspace(int L, int N, int C, int W, int Hq, int Hkv, int D,
                                          int B) {
  (void)D;
  (void)B;
  if (L < 1 || N < 1 || C < 1 || W < 0 || Hq < 1 || Hkv < 1) return 0;
  return prefill_ws_layout(L * N, C, W, Hq, Hkv).total;
}

pfd_status pfd_chunk_prefill_layers(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                    const pfd_bf16* q_win, int L, int N, int C, int W, int Hq,
                                    int Hkv, int D, int B, float sm_scale, pfd_bf16* out,
                                    float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                    pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                    pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                    size_t workspace_bytes, pfd_stream_t stream) {
  return prefill_impl(q, k, v, q_win, L, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores, kept_idx,
                      pool_k, pool_v, pool_rows, slot_row, table, dev_err, workspace,
                      workspace_bytes, false, nullptr, stream);
}

pfd_status pfd_chunk_prefill_batch(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                   const pfd_bf16* q_win, int L, int N, int C, int W, int Hq,
                                   int Hkv, int D, int B, float sm_scale, pfd_bf16* out,
                                   float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                   pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                   pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                   size_t workspace_bytes, pfd_stream_t stream) {
  return prefill_impl(q, k, v, q_win, L, N, C, W, Hq, Hkv, D, B, sm_scale, out, scores, kept_idx,
                      pool_k, pool_v, pool_rows, slot_row, table, dev_err, workspace,
                      workspace_bytes, false, nullptr, stream, true);
}

pfd_status pfd_chunk_loglik(const pfd_bf16* logits, const int32_t* labels, int N, int R,
                            int64_t V, float* row_ll, float* score, int32_t* dev_err,
                            pfd_stream_t stream) {
  if (!logits || !labels || !row_ll || !score || N < 1 || R < 1 || V < 1)
    return PFD_ERR_INVALID_ARG;
  if (static_cast<long long>(N) * R >= (1ll << 31) || V >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  return from_cuda(launch_chunk_loglik(reinterpret_cast<const bf16*>(logits), labels, N, R, V,
                                       row_ll, score, dev_err,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

pfd_status pfd_select_chunks(const float* s_I, const float* s_P, int N, int K, int32_t* sel,
                             float* s_out, pfd_stream_t stream) {
  if (!s_I || !s_P || !sel || N < 1 || K < 1 || K > N) return PFD_ERR_INVALID_ARG;
  if (N > 16384) return PFD_ERR_UNSUPPORTED;
  return from_cuda(launch_select(s_I, s_P, nullptr, nullptr, N, K, 1, N, 1.0f, sel, s_out,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

pfd_status pfd_select_chunks_batched(const float* s_I, const float* s_P, const int32_t* cu_n,
                                     const int32_t* cu_k, int batch, int max_n, int32_t* sel,
                                     float* s_out, pfd_stream_t stream) {
  if (!s_I || !s_P || !sel || !cu_n || !cu_k || batch < 1 || max_n < 1)
    return PFD_ERR_INVALID_ARG;
  if (max_n > 16384) return PFD_ERR_UNSUPPORTED;
  return from_cuda(launch_select(s_I, s_P, cu_n, cu_k, 0, 0, batch, max_n, 1.0f, sel, s_out,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

int pfd_decode_plan_splits(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host,
                           int Hq, int Hkv, int D, int max_chunk_len) {
  return plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D, max_chunk_len, true);
}

size_t pfd_decode_workspace(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host,
                            int Hq, int Hkv, int D, int max_chunk_len, int n_splits) {
  if (!decode_host_ok(batch, cu_lq_host, cu_k_host)) return 0;
  const int S = n_splits > 0 ? n_splits
                             : plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D,
                                           max_chunk_len, true);
  return decode_ws_layout(S, cu_lq_host[batch], Hq, D).total;
}

size_t pfd_decode_partial_workspace(int batch, const int32_t* cu_lq_host,
                                    const int32_t* cu_k_host, int Hq, int Hkv, int D,
                                    int max_chunk_len, int self_keys, int n_splits) {
  if (!decode_host_ok(batch, cu_lq_host, cu_k_host)) return 0;
  const int S = n_splits > 0 ? n_splits
                             : plan_splits(batch, cu_lq_host, cu_k_host, Hq, Hkv, D,
                                           max_chunk_len, self_keys != 0);
  return decode_ws_layout(S, cu_lq_host[batch], Hq, D).total;
}

pfd_status pfd_decode_attention(const pfd_bf16* q, const pfd_bf16* k_self,
                                const pfd_bf16* v_self, const int32_t* cu_lq,
                                const int32_t* cu_lq_host, const pfd_bf16* pool_k,
                                const pfd_bf16* pool_v, int64_t pool_rows,
                                const pfd_chunk_entry* table, int32_t table_len,
                                const int32_t* sel, const int32_t* cu_k, const int32_t* cu_k_host,
                                int batch, int Hq, int Hkv, int D, int max_chunk_len,
                                float sm_scale, int n_splits, pfd_bf16* out, float* lse,
                                int32_t* dev_err, void* workspace, size_t workspace_bytes,
                                pfd_stream_t stream) {
  return decode_impl(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v, pool_rows, table,
                     table_len, sel, cu_k, cu_k_host, batch, Hq, Hkv, D, max_chunk_len, sm_scale,
                     true, n_splits, out, lse, dev_err, workspace, workspace_bytes, stream);
}

pfd_status pfd_decode_partial(const pfd_bf16* q, const pfd_bf16* k_self, const pfd_bf16* v_self,
                              const int32_t* cu_lq, const int32_t* cu_lq_host,
                              const pfd_bf16* pool_k, const pfd_bf16* pool_v, int64_t pool_rows,
                              const pfd_chunk_entry* table, int32_t table_len, const int32_t* sel,
                              const int32_t* cu_k, const int32_t* cu_k_host, int batch, int Hq,
                              int Hkv, int D, int max_chunk_len, float sm_scale, int self_keys,
                              int n_splits, pfd_bf16* part_o, float* part_lse, int32_t* dev_err,
                              void* workspace, size_t workspace_bytes, pfd_stream_t stream) {
  if (part_lse == nullptr || (self_keys != 0 && self_keys != 1)) return PFD_ERR_INVALID_ARG;
  return decode_impl(q, k_self, v_self, cu_lq, cu_lq_host, pool_k, pool_v, pool_rows, table,
                     table_len, sel, cu_k, cu_k_host, batch, Hq, Hkv, D, max_chunk_len, sm_scale,
                     self_keys != 0, n_splits, part_o, part_lse, dev_err, workspace,
                     workspace_bytes, stream);
}

pfd_status pfd_lse_merge(const pfd_bf16* part_o, const float* part_lse, int n_parts, int rows,
                         int Hq, int D, pfd_bf16* out, float* lse, pfd_stream_t stream) {
  if (!part_o || !part_lse || !out || n_parts < 1 || rows < 1 || Hq < 1)
    return PFD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return PFD_ERR_UNSUPPORTED;
  if (n_parts > kMaxSplits) return PFD_ERR_UNSUPPORTED;
  if (static_cast<long long>(n_parts) * rows * Hq * D >= (1ll << 40)) return PFD_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(part_o) & 7u) != 0 || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return PFD_ERR_INVALID_ARG;
  MergeParams mp;
  std::memset(&mp, 0, sizeof(mp));
  mp.part_m = part_lse;
  mp.part_l = nullptr;   // states given as log-sum-exp
  mp.part_acc = reinterpret_cast<const bf16*>(part_o);
  mp.out = reinterpret_cast<bf16*>(out);
  mp.lse = lse;
  mp.n_splits = n_parts;
  mp.total_lq = rows;
  mp.Hq = Hq;
  mp.D = D;
  return from_cuda(launch_lse_merge(mp, device_sm_count(), reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------- reselection --

namespace {

struct MassPlan {
  int batch = 0;
  int item0[kMaxMassBatch + 1];
  int n0[kMaxMassBatch];
  int n1[kMaxMassBatch];
  int pairs[kMaxMassBatch];
  int chunks_per_item = 1;
  long long items = 0;
  int chunks = 0;
};

bool mass_plan(int batch, const int32_t* cu_lq_host, const int32_t* cu_n_host, int Hq, int Hkv,
               MassPlan* mp) {
  if (batch < 1 || batch > kMaxMassBatch || !cu_lq_host || !cu_n_host) return false;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Hq / Hkv > kBlockM) return false;
  if (cu_lq_host[0] != 0 || cu_n_host[0] != 0) return false;
  const int Tq = kBlockM / (Hq / Hkv);
  mp->batch = batch;
  for (int b = 0; b < batch; ++b) {
    const int lq = cu_lq_host[b + 1] - cu_lq_host[b], n = cu_n_host[b + 1] - cu_n_host[b];
    if (lq < 0 || n < 0) return false;
    mp->n0[b] = cu_n_host[b];
    mp->n1[b] = cu_n_host[b + 1];
    mp->pairs[b] = (ceil_div(lq, Tq) + 1) / 2;
  }
  // One item per (group of M consecutive chunks, KV head, pair of query
  // tiles): the largest M <= kMassChunks that still leaves kMassMinItems
  // items (short items are mostly start and end; too few leave SMs idle).
  // The choice depends only on the shapes, so the workspace size does too.
  constexpr long long kMassMinItems = 512;
  auto items_for = [&](int M) {
    long long items = 0;
    for (int b = 0; b < batch; ++b)
      items += static_cast<long long>(ceil_div(mp->n1[b] - mp->n0[b], M)) * Hkv * mp->pairs[b];
    return items;
  };
  int M = kMassChunks;
  while (M > 1 && items_for(M) < kMassMinItems) M >>= 1;
  mp->chunks_per_item = M;
  long long items = 0;
  for (int b = 0; b < batch; ++b) {
    mp->item0[b] = static_cast<int>(items);
    items += static_cast<long long>(ceil_div(mp->n1[b] - mp->n0[b], M)) * Hkv * mp->pairs[b];
    if (items >= (1ll << 31)) return false;
  }
  mp->item0[batch] = static_cast<int>(items);
  mp->items = items;
  mp->chunks = cu_n_host[batch];
  return true;
}

}  // namespace

extern "C" {

size_t pfd_chunk_mass_workspace(int batch, const int32_t* cu_lq_host, const int32_t* cu_n_host,
                                int Hq, int Hkv) {
  MassPlan mp;
  if (!mass_plan(batch, cu_lq_host, cu_n_host, Hq, Hkv, &mp)) return 0;
  return align256(static_cast<size_t>(mp.items) * mp.chunks_per_item * 8 * sizeof(float));
}

pfd_status pfd_chunk_mass(const pfd_bf16* q, const int32_t* cu_lq, const int32_t* cu_lq_host,
                          const pfd_bf16* pool_k, int64_t pool_rows, const pfd_chunk_entry* table,
                          int32_t table_len, const int32_t* cu_n_host, const float* lse, int batch,
                          int Hq, int Hkv, int D, float sm_scale, float* mass, int32_t* dev_err,
                          void* workspace, size_t workspace_bytes, pfd_stream_t stream) {
  if (!q || !cu_lq || !pool_k || !table || !lse || !mass) return PFD_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return PFD_ERR_UNSUPPORTED;
  if (batch > kMaxMassBatch) return PFD_ERR_UNSUPPORTED;
  MassPlan mp;
  if (!mass_plan(batch, cu_lq_host, cu_n_host, Hq, Hkv, &mp)) return PFD_ERR_INVALID_ARG;
  const int total_lq = cu_lq_host[batch];
  if (total_lq < 1 || cu_n_host[batch] > table_len || table_len < 1 || pool_rows < 1)
    return PFD_ERR_INVALID_ARG;
  if (pool_rows >= (1ll << 31)) return PFD_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(pool_k)) return PFD_ERR_INVALID_ARG;
  const size_t need =
      align256(static_cast<size_t>(mp.items) * mp.chunks_per_item * 8 * sizeof(float));
  if (workspace_bytes < need || (need > 0 && workspace == nullptr) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PFD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (mp.items == 0) return PFD_OK;
  const int G = Hq / Hkv;
  const int Tq = kBlockM / G;
  AttnParams ap;
  std::memset(&ap, 0, sizeof(ap));
  if (!make_map(&ap.tm_q[0], q, total_lq, Hq, D, G, Tq) ||
      !make_kv_maps(ap.tm_k, 0, pool_k, pool_rows, Hkv, D))
    return PFD_ERR_CUDA;
  ap.tm_q[1] = ap.tm_q[0];
  copy_kv_maps(ap.tm_k, 1, 0);
  for (int lv = 0; lv < kBoxLevels; ++lv)
    for (int t = 0; t < 2; ++t) ap.tm_v[lv][t] = ap.tm_k[lv][t];   // no PV in mass items
  const float scale = sm_scale > 0.0f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  ap.Tq = Tq;
  ap.q = reinterpret_cast<const bf16*>(q);
  ap.table = table;
  ap.table_len = table_len;
  ap.pool_rows = pool_rows;
  ap.cu_lq = cu_lq;
  ap.total_lq = total_lq;
  ap.dev_err = dev_err;
  ap.mode = kModeMass;
  ap.Hq = Hq;
  ap.Hkv = Hkv;
  ap.G = G;
  ap.D = D;
  ap.batch = batch;
  ap.n_splits = 1;
  ap.scale_log2 = scale * kLog2e;
  ap.mass_lse = lse;
  ap.mass_part = static_cast<float*>(workspace);
  ap.mass_chunks = mp.chunks_per_item;
  ap.mass_batch = batch;
  for (int b = 0; b <= batch; ++b) ap.mass_item0[b] = mp.item0[b];
  for (int b = 0; b < batch; ++b) {
    ap.mass_n0[b] = mp.n0[b];
    ap.mass_pairs[b] = mp.pairs[b];
  }
  ap.mass_n0[batch] = mp.n1[batch - 1];
  ap.n_items = static_cast<int>(mp.items);
  const int grid = static_cast<int>(std::min<long long>(mp.items, device_sm_count()));
  pfd_status s = from_cuda(launch_attention(ap, grid, st));
  if (s != PFD_OK) return s;
  return from_cuda(launch_mass_sum(ap, cu_lq_host, mp.chunks, mass, st));
}

pfd_status pfd_reselect_chunks(const float* s, const float* mass, float lambda,
                               const int32_t* cu_n, const int32_t* cu_k, int batch, int max_n,
                               int32_t* sel, float* s_out, pfd_stream_t stream) {
  if (!s || !mass || !sel || !cu_n || !cu_k || batch < 1 || max_n < 1 || !(lambda >= 0.0f))
    return PFD_ERR_INVALID_ARG;
  if (max_n > 16384) return PFD_ERR_UNSUPPORTED;
  return from_cuda(launch_select(s, mass, cu_n, cu_k, 0, 0, batch, max_n, lambda, sel, s_out,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
