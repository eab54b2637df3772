// Host side of the C ABI declared in include/lmhead.h: argument checks, the
// tile/split/block plan, the workspace carve-up, TMA descriptor encoding and
// the stream-ordered launches.  No device memory is allocated here and no
// call synchronises the stream except the explicit status readers.
#include "lmhead.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"

using namespace lmh;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 32;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t x, int64_t m) { return (x + m - 1) / m; }

// ------------------------------------------------------------------ launches
std::atomic<uint64_t> g_launches{0};

struct ProfRecord {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

template <class F>
cudaError_t launch(const char* name, cudaStream_t s, F&& f) {
  cudaEvent_t a = nullptr, b = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) {
      a = pooled_event();
      b = pooled_event();
    }
  }
  if (a && b) cudaEventRecord(a, s);
  const cudaError_t e = f();
  if (a && b) {
    cudaEventRecord(b, s);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({name, a, b});
  }
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// ------------------------------------------------------------------ device facts
int sm_count() {
  static std::atomic<int> cache[64];   // per device; 0 = not yet known
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    if (const int c = cache[dev].load(std::memory_order_relaxed); c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Tiles run on CTA pairs (tcgen05 cta_group::2) unless the environment sets
// LMHEAD_CTA_PAIR=0 (single-CTA tiles; a diagnostic fallback).
bool use_pair() {
  static const bool on = [] {
    const char* e = std::getenv("LMHEAD_CTA_PAIR");
    return !(e && e[0] == '0');
  }();
  return on;
}

// Backward launch structure, from LMHEAD_BWD_PERSISTENT (read on every call
// so that the forms can be compared in one process; all give the same bits):
//   unset       chosen by block size (below);
//   1           one persistent launch for all blocks, tiles ordered by
//               completion flags;
//   0           two launches per block (dz, then dh + dW);
//   2           windows: blocks + 1 launches, each a block's dh + dW tiles
//               followed by the next block's dz tiles.
// The persistent forms need CTA pairs and at most BWD_ALL_MAX_TOKEN_BLOCKS
// token blocks; otherwise the backward runs as two launches per block.
int bwd_mode() {
  const char* e = std::getenv("LMHEAD_BWD_PERSISTENT");
  if (!e || !e[0]) return -1;
  return e[0] == '0' ? 0 : (e[0] == '2' ? 2 : 1);
}

// Unset mode: the persistent launch removes two launch boundaries and their
// tails per block, which pays while blocks are small (Qwen3-4B-sized head,
// 4096 x 16896 x 2560 MACs per block: 5.55 vs 5.86 ms).  With blocks of
// 1e12 MACs and more (chunk 4096 on a 61k-token row or a 200,000-token
// trace) the boundaries cost under 1% and the persistent launch measured
// 1.0-1.3% slower than two launches per block, so those take the latter.
constexpr double kPersistentMaxBlockMacs = 5e11;

bool persistent_pays(int64_t Tb, int64_t Vb, int64_t H) {
  return static_cast<double>(Tb) * static_cast<double>(Vb) * static_cast<double>(H) <=
         kPersistentMaxBlockMacs;
}

int unit_rows() { return use_pair() ? 2 * BM : BM; }
uint32_t b_box_rows() { return use_pair() ? BN / 2 : BN; }

bool make_map_k3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_rows);
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer);

// Map of a K-major operand with K = H of the forward and dz GEMMs: on CTA
// pairs those kernels stage two K steps per operand (3-D boxes), single-CTA
// tiles one (2-D boxes).
bool make_map_hk(CUtensorMap* m, const void* base, uint64_t H, uint64_t rows, uint32_t box_rows) {
  return use_pair() ? make_map_k3(m, base, H, rows, 2 * H, box_rows)
                    : make_map(m, base, H, rows, 2 * H, BK, box_rows);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map: `inner` contiguous elements per row, `outer` rows, rows
// `row_bytes` apart; boxes of box_inner x box_outer with 128-byte swizzle.
// Elements outside the map read as zero.
bool make_map_typed(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto enc = encode_fn();
  if (!enc || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, type, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major bf16 operand map: the matrix [rows][inner] (rows `row_bytes`
// apart, K along the rows) viewed as 64-element chunks, (64, rows,
// ceil(inner / 64)), the chunks 128 bytes apart.  A box of 64 x 64 x `chunks`
// lands in shared memory as `chunks` swizzled 64 x 64 images 8 KB apart: one
// instruction per K step instead of one per chunk.  Rows past `rows` read as
// zero; a partial last chunk reads the row's padding (callers discard those
// M rows, or the row is padded with zeros).
bool make_map_mn(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t row_bytes, uint32_t chunks) {
  auto enc = encode_fn();
  if (!enc || inner == 0 || rows == 0) return false;
  cuuint64_t dims[3] = {64, rows, (inner + 63) / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, 64, chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer) {
  return make_map_typed(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_bytes,
                        box_inner, box_outer);
}

// K-major bf16 operand [rows][inner] (inner a multiple of 64: K = H) viewed
// as (64, rows, inner / 64), the 64-element K chunks 128 bytes apart.  A box
// of 64 x box_rows x 2 loads two 64-wide K steps with one instruction; each
// lands as the swizzled image a 2-D 64 x box_rows box would give, 16 KB
// apart for 128 rows.  Rows past `rows`, and a chunk past the last, read as
// zero.
bool make_map_k3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc || inner == 0 || rows == 0 || inner % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, inner / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_f16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_map_typed(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, inner, outer, row_bytes,
                        box_inner, box_outer);
}

// fp32 output map with 128-row x 32-column (128-byte) boxes for staged
// epilogue stores and reduce-adds.
bool make_out_map_f32(CUtensorMap* m, const float* base, uint64_t cols, uint64_t rows,
                      uint64_t ld) {
  return make_map_typed(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, cols, rows, 4 * ld, 32, BM);
}

// ------------------------------------------------------------------ plans
// Vocabulary splits for the forward: each CTA takes (token block, split)
// units round robin; pick the split count whose largest per-CTA tile count
// is smallest (ties: fewer splits, i.e. fewer partial statistics).
int choose_splits(int64_t m_tiles, int64_t n_tiles, int sms) {
  struct Key {
    int64_t m, n;
    int sms, splits;
  };
  static std::mutex mu;
  static std::vector<Key> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Key& k : cache)
      if (k.m == m_tiles && k.n == n_tiles && k.sms == sms) return k.splits;
  }
  int best = 1;
  int64_t best_span = INT64_MAX;
  const int smax = static_cast<int>(std::min<int64_t>(n_tiles, kMaxSplits));
  std::vector<int64_t> load;
  for (int S = 1; S <= smax; ++S) {
    const int64_t units = m_tiles * S;
    const int64_t G = std::min<int64_t>(units, sms);
    load.assign(static_cast<size_t>(G), 0);
    for (int64_t u = 0; u < units; ++u) {
      const int64_t j = u / m_tiles;
      load[static_cast<size_t>(u % G)] += (j + 1) * n_tiles / S - j * n_tiles / S;
    }
    const int64_t span = *std::max_element(load.begin(), load.end());
    if (span < best_span) {
      best_span = span;
      best = S;
    }
  }
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() > 64) cache.clear();
  cache.push_back({m_tiles, n_tiles, sms, best});
  return best;
}

struct BwdPlan {
  int64_t Tb, Vb, n_tb, n_vb;
};

// Backward blocks T_b x V_b with T_b * V_b <= chunk_size * V (the scratch
// bound).  T_b ~ V_b ~ sqrt(chunk_size * V) would minimise the fp32
// read-modify-write traffic of dh and dW, 8 T V H (1/T_b + 1/V_b) bytes, but
// a token block's hidden rows are read again for every dz column tile and
// every dW tile, so T_b is also capped to keep them (T_b x H bf16) within
// kHiddenBlockBytes of L2; V_b then takes the rest of the bound.  On a
// 200,000-token trace (H 2048) and a 61k-token row (H 4096) at chunk 4096
// the cap makes the backward 6-8% faster than square blocks; where the
// square block is already small enough (H 2560 at chunk 512) nothing changes.
// T_b is a multiple of 256 rows (one CTA pair's tile), V_b of 256 columns.
constexpr int64_t kHiddenBlockBytes = 40ll << 20;

BwdPlan plan_bwd(int64_t T, int64_t H, int64_t V, int64_t chunk) {
  BwdPlan p;
  constexpr int64_t TU = 2 * BM;
  const int64_t T_alloc = round_up(T, BM);
  const int64_t V_pad = round_up(V, BN);
  const double S = static_cast<double>(chunk) * static_cast<double>(V);
  int64_t tb_max = static_cast<int64_t>(std::floor(std::sqrt(S) / TU)) * TU;
  tb_max = std::min<int64_t>(tb_max, kHiddenBlockBytes / (2 * H) / TU * TU);
  tb_max = std::max<int64_t>(TU, std::min<int64_t>(tb_max, round_up(T_alloc, TU)));
  p.n_tb = ceil_div(T_alloc, tb_max);
  p.Tb = round_up(ceil_div(T_alloc, p.n_tb), TU);
  p.n_tb = ceil_div(T_alloc, p.Tb);
  int64_t vb_max = static_cast<int64_t>(std::floor(S / static_cast<double>(p.Tb) / BN)) * BN;
  vb_max = std::max<int64_t>(BN, std::min<int64_t>(vb_max, V_pad));
  p.n_vb = ceil_div(V_pad, vb_max);
  p.Vb = round_up(ceil_div(V_pad, p.n_vb), BN);
  p.n_vb = ceil_div(V, p.Vb);
  return p;
}

// Forward unit order.  The forward's units (token block, vocabulary split)
// are handed out token-block fastest, so the CTAs running at one time sweep
// the same split's W tiles together (one DRAM read, the rest L2 hits) while
// each re-reads its own token block's hidden rows (256 x H bf16) once per
// 256-column vocabulary tile.  With every SM on a different token block
// those rows alone can outgrow L2 (76 pairs x 256 rows x 4096 x 2 B =
// 152 MB at H = 4096), and then the re-reads go to DRAM.  So token blocks
// are taken in groups whose hidden rows fit in kFwdGroupBytes (a quarter of
// L2); a group runs through all splits before the next one starts, which
// costs one more read of W per group (a few hundred GB/s at most).
// Measured on GB300, forward alone, interleaved against the plain order:
// 61k-token row at H = 4096 -10 to -15%, 45k scored tokens at H = 2560
// -3 to -4%, 160k at H = 2048 -1 to -2%, for any budget from 20 to 48 MB;
// 16 token blocks at H = 2560 (4096 tokens) fit in one group (unchanged).
// LMHEAD_FWD_GROUP_MB, read on every call, overrides the budget (0: one
// group, the plain order); the order changes no result bit, since every
// unit is computed whole by one CTA pair.
constexpr int64_t kFwdGroupBytes = 32ll << 20;

int fwd_m_group(int64_t H) {
  int64_t budget = kFwdGroupBytes;
  if (const char* e = std::getenv("LMHEAD_FWD_GROUP_MB"); e && e[0]) {
    const long long mb = std::atoll(e);
    if (mb <= 0) return 0;
    budget = static_cast<int64_t>(std::min<long long>(mb, 1ll << 20)) << 20;
  }
  const int64_t panel = static_cast<int64_t>(unit_rows()) * 2 * H;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(budget / panel, 1 << 20)));
}

// Work units of the per-block dz GEMM: k adjacent 256-column tiles of one
// token block, k the largest of 4, 2, 1 that still leaves at least
// kDzUnitsPerPair units per CTA pair (so the launch's tail stays short).
// Each unit pays one fetch from the unit counter and one hand-off through
// the scheduler ring, which shows where a tile is short (K = H).  Measured on
// GB300, interleaved, results bitwise equal: dz launches of the 200,000-token
// trace (H 2048, 40 x 198 tiles per block) 64.7 ms per step with one tile per
// unit, 62.2 with two, 61.0 with four; a Qwen3-4B-sized block (H 2560,
// 16 x 66 tiles) 2.04 / 1.96 / 2.10 ms, four tiles leaving too few units.
constexpr int64_t kDzUnitsPerPair = 6;

int dz_splits(int64_t m_tiles, int64_t n_tiles, int sms) {
  const int64_t pairs = std::max(1, use_pair() ? sms / 2 : sms);
  for (int64_t k = 4; k > 1; k /= 2) {
    const int64_t splits = ceil_div(n_tiles, k);
    if (m_tiles * splits >= kDzUnitsPerPair * pairs) return static_cast<int>(splits);
  }
  return 0;   // one tile per unit
}

// Single-call forward + backward that keeps each token block's logits over
// the whole vocabulary (T_b x V_pad 16-bit values <= chunk_size x V) instead
// of recomputing them.  It pays when the recompute GEMM (2 T H V flops)
// costs more than what keeping the logits adds: writing and re-reading them
// (about 4 T V bytes) and the extra fp32 read-modify-write passes over dW
// that the smaller token blocks cause (8 V H bytes each).
struct FusedPlan {
  int64_t Tb, n_tb, V_pad, n_tiles;
  bool preferred;
};

FusedPlan plan_fused(int64_t T, int64_t H, int64_t V, int64_t chunk) {
  FusedPlan p;
  const int64_t T_alloc = round_up(T, BM);
  p.V_pad = round_up(V, BN);
  p.n_tiles = p.V_pad / BN;
  const int64_t unit = 2 * BM;
  int64_t tb = static_cast<int64_t>(static_cast<double>(chunk) * static_cast<double>(V) /
                                    static_cast<double>(p.V_pad)) / unit * unit;
  tb = std::max<int64_t>(unit, std::min<int64_t>(tb, round_up(T_alloc, unit)));
  p.Tb = tb;
  p.n_tb = ceil_div(T_alloc, tb);
  const BwdPlan bp = plan_bwd(T, H, V, chunk);
  const double flops_rate = 1.6e15, bytes_rate = 5.0e12;   // GB300 sustained, rounded down
  const double TVd = static_cast<double>(T) * static_cast<double>(V);
  const double dw_pass = 8.0 * static_cast<double>(V) * static_cast<double>(H) / bytes_rate;
  const double split_cost = 2.0 * TVd * static_cast<double>(H) / flops_rate +
                            static_cast<double>(bp.n_tb) * dw_pass;
  const double fused_cost = 4.0 * TVd / bytes_rate + static_cast<double>(p.n_tb) * dw_pass;
  p.preferred = fused_cost < split_cost;
  return p;
}

struct Layout {
  size_t state, counters, chunk_counts, idx, y_c, h_c, part, coef, dz, m_tile, total;
  int64_t n_counters;   // dynamic work-unit counters, one per GEMM launch
};

Layout layout(int op, int64_t T, int64_t H, int64_t V, int64_t chunk) {
  Layout L{};
  const int64_t T_alloc = round_up(T, BM);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.state = take(sizeof(DeviceState));
  if (op == LMHEAD_OP_FWD) {
    L.n_counters = 1;
  } else if (op == LMHEAD_OP_BWD) {
    // two unit counters per block (per-block launches), or one counter and
    // the tile completion flags of the persistent launch
    const BwdPlan bp = plan_bwd(T, H, V, chunk);
    const int64_t blocks = bp.n_tb * bp.n_vb;
    L.n_counters =
        std::max<int64_t>(2 * blocks, (blocks + 1) + blocks * (1 + bp.Tb / (2 * BM) + 2 * bp.Vb / BN));
  } else {
    L.n_counters = 2 * plan_fused(T, H, V, chunk).n_tb;
  }
  L.counters = take(4 * static_cast<size_t>(L.n_counters));
  L.chunk_counts = take(4 * static_cast<size_t>(compact_chunks(static_cast<int>(T_alloc))));
  L.idx = take(4 * static_cast<size_t>(T_alloc));
  L.y_c = take(4 * static_cast<size_t>(T_alloc));
  L.h_c = take(2 * static_cast<size_t>(T_alloc) * static_cast<size_t>(H));
  if (op == LMHEAD_OP_FWD) {
    L.part = take(16 * static_cast<size_t>(kMaxSplits) * static_cast<size_t>(T_alloc));
  } else if (op == LMHEAD_OP_BWD) {
    const BwdPlan bp = plan_bwd(T, H, V, chunk);
    L.coef = take(16 * static_cast<size_t>(T_alloc));
    L.dz = take(2 * static_cast<size_t>(bp.Tb) * static_cast<size_t>(bp.Vb));
  } else {
    const FusedPlan fp = plan_fused(T, H, V, chunk);
    L.part = take(16 * static_cast<size_t>(kMaxSplits) * static_cast<size_t>(T_alloc));
    L.coef = take(16 * static_cast<size_t>(T_alloc));
    L.dz = take(2 * static_cast<size_t>(fp.Tb) * static_cast<size_t>(fp.V_pad));
    L.m_tile = take(4 * static_cast<size_t>(fp.Tb) * static_cast<size_t>(fp.n_tiles));
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

lmhead_status check_sizes(int64_t T, int32_t H, int32_t V, float tau, int32_t chunk) {
  if (T < 0 || H <= 0 || V <= 0 || chunk <= 0 || !std::isfinite(tau) || !(tau > 0.f))
    return LMHEAD_ERR_INVALID_ARG;
  if (H % 64 != 0 || T >= (int64_t{1} << 31) - 256) return LMHEAD_ERR_UNSUPPORTED;
  return LMHEAD_OK;
}

#define LMH_TRY(expr)                               \
  do {                                              \
    if ((expr) != cudaSuccess) return LMHEAD_ERR_CUDA; \
  } while (0)

// Shared front half of both calls: status reset, mask compaction / target
// wrap, and the gather of scored rows.  Sets the row source for the GEMMs.
struct Front {
  DeviceState* st;
  int* counters;        // zeroed work-unit counters, one per GEMM launch
  int* idx;             // NULL when every token is scored
  int* y_c;
  const uint16_t* h_src;
  int64_t rows_avail;   // rows addressable in h_src
  int64_t T_alloc;
};

// The call holds vocabulary rows [v0, v0 + V) of a vocabulary of Vt ids
// (v0 = 0, Vt = V outside the vocabulary-sharded calls).
lmhead_status front(const uint16_t* hidden, const int32_t* targets, const uint8_t* mask, int64_t T,
                    int32_t H, int32_t V, int32_t v0, int32_t Vt, char* ws, const Layout& L,
                    cudaStream_t s, Front* f) {
  f->T_alloc = round_up(T, BM);
  f->st = reinterpret_cast<DeviceState*>(ws + L.state);
  f->y_c = reinterpret_cast<int*>(ws + L.y_c);
  const int Ti = static_cast<int>(T), Ta = static_cast<int>(f->T_alloc);
  f->counters = reinterpret_cast<int*>(ws + L.counters);
  LMH_TRY(launch("clear_state", s, [&] {
    return launch_clear_state(f->st, mask ? 0 : Ti, f->counters, L.n_counters, s);
  }));
  if (mask) {
    f->idx = reinterpret_cast<int*>(ws + L.idx);
    uint16_t* h_c = reinterpret_cast<uint16_t*>(ws + L.h_c);
    LMH_TRY(launch("compact", s, [&] {
      return launch_compact(mask, targets, Ti, v0, V, Vt, Ta,
                            reinterpret_cast<int*>(ws + L.chunk_counts), f->idx, f->y_c, f->st, s);
    }));
    LMH_TRY(launch("gather_rows", s, [&] {
      return launch_gather_rows(hidden, H, f->idx, Ta, f->st, h_c, s);
    }));
    f->h_src = h_c;
    f->rows_avail = f->T_alloc;
  } else {
    f->idx = nullptr;
    LMH_TRY(launch("targets_dense", s, [&] {
      return launch_targets_dense(targets, Ti, v0, V, Vt, Ta, f->y_c, f->st, s);
    }));
    f->h_src = hidden;
    f->rows_avail = T;
  }
  return LMHEAD_OK;
}

}  // namespace

extern "C" {

size_t lmhead_workspace_size(int op, int64_t T, int32_t H, int32_t V, int32_t chunk_size) {
  if ((op != LMHEAD_OP_FWD && op != LMHEAD_OP_BWD && op != LMHEAD_OP_FWD_BWD) ||
      check_sizes(T, H, V, 1.0f, chunk_size) != LMHEAD_OK)
    return 0;
  if (op == LMHEAD_OP_FWD_BWD)
    return std::max({layout(LMHEAD_OP_FWD, T, H, V, chunk_size).total,
                     layout(LMHEAD_OP_BWD, T, H, V, chunk_size).total,
                     layout(LMHEAD_OP_FWD_BWD, T, H, V, chunk_size).total});
  return layout(op, T, H, V, chunk_size).total;
}

const char* lmhead_status_string(lmhead_status status) {
  switch (status) {
    case LMHEAD_OK: return "LMHEAD_OK";
    case LMHEAD_ERR_INVALID_ARG: return "LMHEAD_ERR_INVALID_ARG: invalid argument";
    case LMHEAD_ERR_UNSUPPORTED: return "LMHEAD_ERR_UNSUPPORTED: unsupported size or alignment";
    case LMHEAD_ERR_WORKSPACE_TOO_SMALL: return "LMHEAD_ERR_WORKSPACE_TOO_SMALL: workspace too small";
    case LMHEAD_ERR_CUDA: return "LMHEAD_ERR_CUDA: CUDA launch or runtime error";
    case LMHEAD_ERR_DEVICE_TIMEOUT: return "LMHEAD_ERR_DEVICE_TIMEOUT: a device wait exceeded its limit";
    case LMHEAD_ERR_BAD_TARGET: return "LMHEAD_ERR_BAD_TARGET: a scored target lies outside [-V, V)";
    case LMHEAD_ERR_INTERNAL:
      return "LMHEAD_ERR_INTERNAL: a kernel refused a tile store at an invalid coordinate";
  }
  return "unknown lmhead_status";
}

lmhead_status lmhead_plan_info(int64_t T, int32_t H, int32_t V, int32_t chunk_size,
                               int32_t* fwd_splits, int32_t* bwd_tokens, int32_t* bwd_vocab) {
  if (check_sizes(T, H, V, 1.0f, chunk_size) != LMHEAD_OK || T == 0) return LMHEAD_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (fwd_splits)
    *fwd_splits = sms > 0 ? choose_splits(ceil_div(T, unit_rows()), ceil_div(V, BN),
                                          use_pair() ? sms / 2 : sms)
                          : 0;
  const BwdPlan bp = plan_bwd(T, H, V, chunk_size);
  if (bwd_tokens) *bwd_tokens = static_cast<int32_t>(bp.Tb);
  if (bwd_vocab) *bwd_vocab = static_cast<int32_t>(bp.Vb);
  return LMHEAD_OK;
}

}  // extern "C"

namespace {

// Forward over vocabulary rows [v0, v0 + V) of a vocabulary of Vt ids.  With
// shard_part == NULL (the whole vocabulary: v0 = 0, Vt = V) it writes logp /
// entropy / lse; otherwise the token's statistics over these rows go to
// shard_part, for lmhead_combine_shards.
lmhead_status fwd_impl(const uint16_t* hidden, const uint16_t* weight, const int32_t* targets,
                       const uint8_t* loss_mask, int64_t T, int32_t H, int32_t V, int32_t v0,
                       int32_t Vt, float temperature, int32_t chunk_size, float* logp,
                       float* entropy, float* lse, float4* shard_part, void* workspace,
                       size_t workspace_bytes, lmhead_stream_t stream) {
  lmhead_status rc = check_sizes(T, H, V, temperature, chunk_size);
  if (rc != LMHEAD_OK) return rc;
  if (T == 0) return LMHEAD_OK;
  if (!hidden || !weight || !targets || !workspace || (!shard_part && (!logp || !lse)))
    return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return LMHEAD_ERR_UNSUPPORTED;
  const Layout L = layout(LMHEAD_OP_FWD, T, H, V, chunk_size);
  if (workspace_bytes < L.total) return LMHEAD_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return LMHEAD_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  Front f;
  rc = front(hidden, targets, loss_mask, T, H, V, v0, Vt, ws, L, s, &f);
  if (rc != LMHEAD_OK) return rc;

  const bool pair = use_pair();
  const int64_t m_tiles = ceil_div(T, unit_rows()), n_tiles = ceil_div(V, BN);
  const int splits = choose_splits(m_tiles, n_tiles, pair ? sms / 2 : sms);
  float4* part = reinterpret_cast<float4*>(ws + L.part);

  LaunchArgs la;
  std::memset(&la, 0, sizeof(la));
  if (!make_map_hk(&la.map_a[0], f.h_src, H, f.rows_avail, BM)) return LMHEAD_ERR_CUDA;
  if (!make_map_hk(&la.map_b[0], weight, H, V, b_box_rows())) return LMHEAD_ERR_CUDA;
  GemmArgs& p = la.prob[0].p;
  p.m_cap = static_cast<int>(T);
  p.n_extent = V;
  p.k_cap = H;
  p.m_dynamic = 1;
  p.dyn_base = 0;
  p.dev_rows = &f.st->rows;
  p.n_splits = splits;
  p.m_group = fwd_m_group(H);
  p.status = &f.st->status;
  p.scale = kLog2e / temperature;
  p.y_c = f.y_c;
  p.partials = part;
  p.part_ld = static_cast<int>(f.T_alloc);
  la.n_problems = 1;
  la.counter = f.counters;
  const int grid = static_cast<int>(std::min<int64_t>(m_tiles * splits * (pair ? 2 : 1), sms));
  LMH_TRY(launch("fwd_stats_gemm", s, [&] { return launch_gemm_fwd_stats(la, grid, pair, s); }));
  LMH_TRY(launch("fwd_merge", s, [&] {
    return launch_fwd_merge(part, splits, static_cast<int>(f.T_alloc), f.idx, f.y_c, f.st, 0,
                            static_cast<int>(f.T_alloc), logp, entropy, lse, shard_part, s);
  }));
  if (loss_mask) {
    LMH_TRY(launch("zero_masked_outputs", s, [&] {
      return launch_zero_masked_outputs(loss_mask, static_cast<int>(T), logp, entropy, lse,
                                        shard_part, s);
    }));
  }
  return LMHEAD_OK;
}

// Backward over vocabulary rows [v0, v0 + V) of a vocabulary of Vt ids, given
// the whole vocabulary's lse (and entropy): d_hidden gets these rows' share of
// the gradient, d_weight the gradient of these rows.
lmhead_status bwd_impl(const uint16_t* hidden, const uint16_t* weight, const int32_t* targets,
                       const uint8_t* loss_mask, int64_t T, int32_t H, int32_t V, int32_t v0,
                       int32_t Vt, float temperature, int32_t chunk_size,
                       const float* grad_logp, const float* grad_entropy, const float* lse,
                       const float* entropy, float* d_hidden, float* d_weight,
                       int accumulate_dweight, void* workspace, size_t workspace_bytes,
                       lmhead_stream_t stream) {
  lmhead_status rc = check_sizes(T, H, V, temperature, chunk_size);
  if (rc != LMHEAD_OK) return rc;
  if (!weight || !d_weight) return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(weight) || !aligned16(d_weight)) return LMHEAD_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (!accumulate_dweight &&
        cudaMemsetAsync(d_weight, 0, sizeof(float) * static_cast<size_t>(V) * H, s) != cudaSuccess)
      return LMHEAD_ERR_CUDA;
    return LMHEAD_OK;
  }
  if (!hidden || !targets || !lse || !d_hidden || !workspace || (grad_entropy && !entropy))
    return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(d_hidden) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return LMHEAD_ERR_UNSUPPORTED;
  const Layout L = layout(LMHEAD_OP_BWD, T, H, V, chunk_size);
  if (workspace_bytes < L.total) return LMHEAD_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return LMHEAD_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);

  Front f;
  rc = front(hidden, targets, loss_mask, T, H, V, v0, Vt, ws, L, s, &f);
  if (rc != LMHEAD_OK) return rc;

  float4* coef = reinterpret_cast<float4*>(ws + L.coef);
  uint16_t* dz = reinterpret_cast<uint16_t*>(ws + L.dz);
  LMH_TRY(launch("bwd_prep", s, [&] {
    return launch_bwd_prep(f.idx, f.st, 0, static_cast<int>(f.T_alloc), lse, entropy, grad_logp,
                           grad_entropy, temperature, coef, s);
  }));
  if (loss_mask) {
    LMH_TRY(launch("zero_masked_rows", s, [&] {
      return launch_zero_masked_rows(loss_mask, static_cast<int>(T), H, d_hidden, s);
    }));
  }

  const BwdPlan bp = plan_bwd(T, H, V, chunk_size);
  const float scale = kLog2e / temperature;
  const bool pair = use_pair();
  const int64_t um = unit_rows();
  const int64_t ctas = pair ? 2 : 1;

  int mode = bwd_mode();
  if (mode < 0) mode = persistent_pays(bp.Tb, bp.Vb, H) ? 1 : 0;
  if (pair && mode != 0 && bp.n_tb <= BWD_ALL_MAX_TOKEN_BLOCKS) {
    // every block's dz, dh and dW tiles in one launch, ordered by tile flags
    BwdAllArgs a;
    std::memset(&a, 0, sizeof(a));
    const uint64_t Tb = static_cast<uint64_t>(bp.Tb), Vb = static_cast<uint64_t>(bp.Vb);
    if (!make_map(&a.h_k, f.h_src, H, f.rows_avail, 2ull * H, BK, BM) ||
        !make_map(&a.w_k, weight, H, V, 2ull * H, BK, BN / 2) ||
        !make_map(&a.dz_k, dz, Vb, Tb, 2ull * Vb, 64, BM) ||
        !make_map_mn(&a.w_mn, weight, H, V, 2ull * H, 2) ||
        !make_map_mn(&a.dz_mn, dz, Vb, Tb, 2ull * Vb, 2) ||
        !make_map_mn(&a.h_mn, f.h_src, H, f.rows_avail, 2ull * H, 2) ||
        (!f.idx && !make_out_map_f32(&a.dh_out, d_hidden, H, T, H)) ||
        !make_out_map_f32(&a.dw_out, d_weight, H, V, H))
      return LMHEAD_ERR_CUDA;
    a.T_b = static_cast<int>(bp.Tb);
    a.V_b = static_cast<int>(bp.Vb);
    a.n_tb = static_cast<int>(bp.n_tb);
    a.n_vb = static_cast<int>(bp.n_vb);
    a.V = V;
    a.H = H;
    a.T_alloc = static_cast<int>(f.T_alloc);
    a.MT = static_cast<int>(bp.Tb / (2 * BM));
    a.NT = static_cast<int>(bp.Vb / BN);
    a.st = f.st;
    a.scale = scale;
    a.y_c = f.y_c;
    a.coef = coef;
    a.row_map = f.idx;
    a.d_hidden = d_hidden;
    a.d_weight = d_weight;
    a.accumulate_dweight = accumulate_dweight ? 1 : 0;
    const int blocks = static_cast<int>(bp.n_tb * bp.n_vb);
    a.flags = f.counters + (blocks + 1);
    if (mode == 1) {
      a.window = -1;
      a.unit_counter = f.counters;
      LMH_TRY(launch("bwd_all_gemm", s, [&] { return launch_gemm_bwd_all(a, sms, s); }));
    } else {
      for (int w = 0; w <= blocks; ++w) {
        a.window = w;
        a.unit_counter = f.counters + w;
        LMH_TRY(launch("bwd_window_gemm", s, [&] { return launch_gemm_bwd_all(a, sms, s); }));
      }
    }
    return LMHEAD_OK;
  }

  for (int64_t tb = 0; tb < bp.n_tb; ++tb) {
    const int64_t t0 = tb * bp.Tb;
    if (t0 >= f.T_alloc) break;
    const int64_t m_cap = std::min<int64_t>(bp.Tb, f.T_alloc - t0);
    const int64_t h_rows = std::min<int64_t>(bp.Tb, f.rows_avail - t0);
    const uint16_t* h_blk = f.h_src + t0 * H;
    for (int64_t vb = 0; vb < bp.n_vb; ++vb) {
      const int64_t v0 = vb * bp.Vb;
      if (v0 >= V) break;
      const int64_t vact = std::min<int64_t>(bp.Vb, V - v0);
      const uint16_t* w_blk = weight + v0 * H;
      int* counter = f.counters + 2 * (tb * bp.n_vb + vb);

      // dz = cotangent of the recomputed logits of this block, bf16 scratch
      LaunchArgs lz;
      std::memset(&lz, 0, sizeof(lz));
      if (!make_map_hk(&lz.map_a[0], h_blk, H, h_rows, BM)) return LMHEAD_ERR_CUDA;
      if (!make_map_hk(&lz.map_b[0], w_blk, H, vact, b_box_rows())) return LMHEAD_ERR_CUDA;
      GemmArgs& pz = lz.prob[0].p;
      pz.m_cap = static_cast<int>(m_cap);
      pz.n_extent = static_cast<int>(vact);
      pz.k_cap = H;
      pz.m_dynamic = 1;
      pz.dyn_base = static_cast<int>(t0);
      pz.dev_rows = &f.st->rows;
      pz.status = &f.st->status;
      pz.scale = scale;
      pz.row_base = static_cast<int>(t0);
      pz.col_base = static_cast<int>(v0);
      pz.y_c = f.y_c;
      pz.coef = coef;
      pz.dz_out = dz;
      pz.dz_ld = static_cast<int>(bp.Vb);
      pz.out_mode = 1;
      pz.n_splits = dz_splits(ceil_div(m_cap, um), ceil_div(vact, BN), sms);
      if (!make_map(&lz.map_out[0], dz, vact, m_cap, 2ull * bp.Vb, 64, BM)) return LMHEAD_ERR_CUDA;
      lz.n_problems = 1;
      lz.counter = counter;
      const int gz = static_cast<int>(
          std::min<int64_t>(ceil_div(m_cap, um) * ceil_div(vact, BN) * ctas, sms));
      LMH_TRY(launch("bwd_dz_gemm", s, [&] { return launch_gemm_bwd_dz(lz, gz, pair, s); }));

      // one launch for both gradient contractions of the block
      LaunchArgs lg;
      std::memset(&lg, 0, sizeof(lg));
      // problem 0: dh[block rows] (+)= dz . W_block   (K = vocabulary of the block)
      if (!make_map(&lg.map_a[0], dz, vact, m_cap, 2ull * bp.Vb, BK, BM)) return LMHEAD_ERR_CUDA;
      if (!make_map_mn(&lg.map_b[0], w_blk, H, vact, 2ull * H, b_box_rows() / 64))
        return LMHEAD_ERR_CUDA;
      GemmArgs& ph = lg.prob[0].p;
      lg.prob[0].a_mn = 0;
      ph.m_cap = static_cast<int>(m_cap);
      ph.n_extent = H;
      ph.k_cap = static_cast<int>(vact);
      ph.m_dynamic = 1;
      ph.dyn_base = static_cast<int>(t0);
      ph.dev_rows = &f.st->rows;
      ph.status = &f.st->status;
      ph.row_base = static_cast<int>(t0);
      ph.out = d_hidden;
      ph.out_ld = H;
      ph.row_map = f.idx;
      ph.accumulate = vb > 0 ? 1 : 0;
      ph.n_fastest = 1;
      if (!f.idx) {
        // every token scored: compacted rows are the rows of d_hidden
        ph.out_mode = ph.accumulate ? 2 : 1;
        if (!make_out_map_f32(&lg.map_out[0], d_hidden + t0 * H, H,
                              std::min<int64_t>(m_cap, T - t0), H))
          return LMHEAD_ERR_CUDA;
      }
      // problem 1: dW[block vocab rows] (+)= dz^T . h_block (K = tokens, ascending blocks)
      if (!make_map_mn(&lg.map_a[1], dz, vact, m_cap, 2ull * bp.Vb, BM / 64) ||
          !make_map_mn(&lg.map_b[1], h_blk, H, h_rows, 2ull * H, b_box_rows() / 64))
        return LMHEAD_ERR_CUDA;
      GemmArgs& pw = lg.prob[1].p;
      lg.prob[1].a_mn = 1;
      pw.m_cap = static_cast<int>(vact);
      pw.n_extent = H;
      pw.k_cap = static_cast<int>(m_cap);
      pw.k_dynamic = 1;
      pw.dyn_base = static_cast<int>(t0);
      pw.dev_rows = &f.st->rows;
      pw.status = &f.st->status;
      pw.row_base = 0;
      pw.out = d_weight + v0 * H;
      pw.out_ld = H;
      pw.accumulate = (tb > 0 || accumulate_dweight) ? 1 : 0;
      pw.zero_if_empty = 1;
      pw.n_fastest = 1;
      pw.out_mode = pw.accumulate ? 2 : 1;
      if (!make_out_map_f32(&lg.map_out[1], d_weight + v0 * H, H, vact, H)) return LMHEAD_ERR_CUDA;
      lg.n_problems = 2;
      lg.counter = counter + 1;
      const int gg = static_cast<int>(std::min<int64_t>(
          (ceil_div(m_cap, um) + ceil_div(vact, um)) * ceil_div(H, BN) * ctas, sms));
      LMH_TRY(launch("bwd_grad_gemm", s, [&] { return launch_gemm_bwd_grad(lg, gg, pair, s); }));
    }
  }
  return LMHEAD_OK;
}

// Arguments of the vocabulary-sharded calls: rows [vocab_offset, vocab_offset +
// V_shard) of a vocabulary of vocab_total ids.
lmhead_status check_shard(int32_t V_shard, int32_t vocab_offset, int32_t vocab_total) {
  if (V_shard <= 0 || vocab_offset < 0 || vocab_total <= 0 ||
      static_cast<int64_t>(vocab_offset) + V_shard > vocab_total)
    return LMHEAD_ERR_INVALID_ARG;
  return LMHEAD_OK;
}

}  // namespace

extern "C" {

lmhead_status lmhead_logps_fwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                               int32_t H, int32_t V, float temperature, int32_t chunk_size,
                               float* logp, float* entropy, float* lse, void* workspace,
                               size_t workspace_bytes, lmhead_stream_t stream) {
  return fwd_impl(hidden, weight, targets, loss_mask, T, H, V, 0, V, temperature, chunk_size,
                  logp, entropy, lse, nullptr, workspace, workspace_bytes, stream);
}

lmhead_status lmhead_logps_bwd(const uint16_t* hidden, const uint16_t* weight,
                               const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                               int32_t H, int32_t V, float temperature, int32_t chunk_size,
                               const float* grad_logp, const float* grad_entropy,
                               const float* lse, const float* entropy, float* d_hidden,
                               float* d_weight, int accumulate_dweight, void* workspace,
                               size_t workspace_bytes, lmhead_stream_t stream) {
  return bwd_impl(hidden, weight, targets, loss_mask, T, H, V, 0, V, temperature, chunk_size,
                  grad_logp, grad_entropy, lse, entropy, d_hidden, d_weight, accumulate_dweight,
                  workspace, workspace_bytes, stream);
}

lmhead_status lmhead_logps_fwd_shard(const uint16_t* hidden, const uint16_t* weight_shard,
                                     const int32_t* targets, const uint8_t* loss_mask,
                                     int64_t T, int32_t H, int32_t V_shard, int32_t vocab_offset,
                                     int32_t vocab_total, float temperature, int32_t chunk_size,
                                     float* partials, void* workspace, size_t workspace_bytes,
                                     lmhead_stream_t stream) {
  lmhead_status rc = check_shard(V_shard, vocab_offset, vocab_total);
  if (rc != LMHEAD_OK) return rc;
  if (T > 0 && !partials) return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(partials)) return LMHEAD_ERR_UNSUPPORTED;
  return fwd_impl(hidden, weight_shard, targets, loss_mask, T, H, V_shard, vocab_offset,
                  vocab_total, temperature, chunk_size, nullptr, nullptr, nullptr,
                  reinterpret_cast<float4*>(partials), workspace, workspace_bytes, stream);
}

lmhead_status lmhead_logps_bwd_shard(const uint16_t* hidden, const uint16_t* weight_shard,
                                     const int32_t* targets, const uint8_t* loss_mask,
                                     int64_t T, int32_t H, int32_t V_shard, int32_t vocab_offset,
                                     int32_t vocab_total, float temperature, int32_t chunk_size,
                                     const float* grad_logp, const float* grad_entropy,
                                     const float* lse, const float* entropy, float* d_hidden,
                                     float* d_weight_shard, int accumulate_dweight,
                                     void* workspace, size_t workspace_bytes,
                                     lmhead_stream_t stream) {
  const lmhead_status rc = check_shard(V_shard, vocab_offset, vocab_total);
  if (rc != LMHEAD_OK) return rc;
  return bwd_impl(hidden, weight_shard, targets, loss_mask, T, H, V_shard, vocab_offset,
                  vocab_total, temperature, chunk_size, grad_logp, grad_entropy, lse, entropy,
                  d_hidden, d_weight_shard, accumulate_dweight, workspace, workspace_bytes,
                  stream);
}

lmhead_status lmhead_combine_shards(const float* partials, int32_t n_shards,
                                    const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                                    int32_t vocab_total, float* logp, float* entropy, float* lse,
                                    lmhead_stream_t stream) {
  if (n_shards <= 0 || T < 0 || vocab_total <= 0) return LMHEAD_ERR_INVALID_ARG;
  if (T >= (int64_t{1} << 31) - 256) return LMHEAD_ERR_UNSUPPORTED;
  if (T == 0) return LMHEAD_OK;
  if (!partials || !targets || !logp || !lse) return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(partials)) return LMHEAD_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LMH_TRY(launch("combine_shards", s, [&] {
    return launch_combine_shards(reinterpret_cast<const float4*>(partials), n_shards, T, targets,
                                 loss_mask, vocab_total, logp, entropy, lse, s);
  }));
  return LMHEAD_OK;
}

lmhead_status lmhead_logps_fwd_bwd(const uint16_t* hidden, const uint16_t* weight,
                                   const int32_t* targets, const uint8_t* loss_mask, int64_t T,
                                   int32_t H, int32_t V, float temperature, int32_t chunk_size,
                                   const float* grad_logp, const float* grad_entropy,
                                   float* logp, float* entropy, float* lse, float* d_hidden,
                                   float* d_weight, int accumulate_dweight, int strategy,
                                   void* workspace, size_t workspace_bytes,
                                   lmhead_stream_t stream) {
  lmhead_status rc = check_sizes(T, H, V, temperature, chunk_size);
  if (rc != LMHEAD_OK) return rc;
  if (strategy < LMHEAD_STRATEGY_AUTO || strategy > LMHEAD_STRATEGY_KEEP_LOGITS)
    return LMHEAD_ERR_INVALID_ARG;
  if (!weight || !d_weight) return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(weight) || !aligned16(d_weight)) return LMHEAD_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (!accumulate_dweight &&
        cudaMemsetAsync(d_weight, 0, sizeof(float) * static_cast<size_t>(V) * H, s) != cudaSuccess)
      return LMHEAD_ERR_CUDA;
    return LMHEAD_OK;
  }
  if (!hidden || !targets || !logp || !lse || !d_hidden || !workspace ||
      (grad_entropy && !entropy))
    return LMHEAD_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(d_hidden) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return LMHEAD_ERR_UNSUPPORTED;
  if (workspace_bytes < lmhead_workspace_size(LMHEAD_OP_FWD_BWD, T, H, V, chunk_size))
    return LMHEAD_ERR_WORKSPACE_TOO_SMALL;

  const FusedPlan fp = plan_fused(T, H, V, chunk_size);
  const bool keep = strategy == LMHEAD_STRATEGY_KEEP_LOGITS ||
                    (strategy == LMHEAD_STRATEGY_AUTO && fp.preferred);
  if (!keep) {
    rc = lmhead_logps_fwd(hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size,
                          logp, entropy, lse, workspace, workspace_bytes, stream);
    if (rc != LMHEAD_OK) return rc;
    return lmhead_logps_bwd(hidden, weight, targets, loss_mask, T, H, V, temperature, chunk_size,
                            grad_logp, grad_entropy, lse, entropy, d_hidden, d_weight,
                            accumulate_dweight, workspace, workspace_bytes, stream);
  }

  const int sms = sm_count();
  if (sms <= 0) return LMHEAD_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  const Layout L = layout(LMHEAD_OP_FWD_BWD, T, H, V, chunk_size);
  Front f;
  rc = front(hidden, targets, loss_mask, T, H, V, 0, V, ws, L, s, &f);
  if (rc != LMHEAD_OK) return rc;
  if (loss_mask) {
    LMH_TRY(launch("zero_masked_outputs", s, [&] {
      return launch_zero_masked_outputs(loss_mask, static_cast<int>(T), logp, entropy, lse,
                                        nullptr, s);
    }));
    LMH_TRY(launch("zero_masked_rows", s, [&] {
      return launch_zero_masked_rows(loss_mask, static_cast<int>(T), H, d_hidden, s);
    }));
  }
  float4* part = reinterpret_cast<float4*>(ws + L.part);
  float4* coef = reinterpret_cast<float4*>(ws + L.coef);
  uint16_t* zbuf = reinterpret_cast<uint16_t*>(ws + L.dz);
  float* m_tile = reinterpret_cast<float*>(ws + L.m_tile);
  const bool pair = use_pair();
  const int64_t um = unit_rows();
  const int64_t ctas = pair ? 2 : 1;
  const int splits = choose_splits(ceil_div(fp.Tb, um), fp.n_tiles, pair ? sms / 2 : sms);
  const float scale = kLog2e / temperature;

  for (int64_t tb = 0; tb < fp.n_tb; ++tb) {
    const int64_t t0 = tb * fp.Tb;
    if (t0 >= f.T_alloc) break;
    const int64_t m_cap = std::min<int64_t>(fp.Tb, f.T_alloc - t0);
    const int64_t h_rows = std::min<int64_t>(fp.Tb, f.rows_avail - t0);
    const uint16_t* h_blk = f.h_src + t0 * H;
    int* counter = f.counters + 2 * tb;

    // forward over the whole vocabulary for this block, keeping the logits
    LaunchArgs lf;
    std::memset(&lf, 0, sizeof(lf));
    if (!make_map_hk(&lf.map_a[0], h_blk, H, h_rows, BM)) return LMHEAD_ERR_CUDA;
    if (!make_map_hk(&lf.map_b[0], weight, H, V, b_box_rows())) return LMHEAD_ERR_CUDA;
    if (!make_map_f16(&lf.map_out[0], zbuf, V, m_cap, 2ull * fp.V_pad, 64, BM))
      return LMHEAD_ERR_CUDA;
    GemmArgs& pf = lf.prob[0].p;
    pf.m_cap = static_cast<int>(m_cap);
    pf.n_extent = V;
    pf.k_cap = H;
    pf.m_dynamic = 1;
    pf.dyn_base = static_cast<int>(t0);
    pf.dev_rows = &f.st->rows;
    pf.n_splits = splits;
    pf.m_group = fwd_m_group(H);
    pf.status = &f.st->status;
    pf.scale = scale;
    pf.row_base = static_cast<int>(t0);
    pf.y_c = f.y_c;
    pf.partials = part;
    pf.part_ld = static_cast<int>(f.T_alloc);
    pf.m_tile = m_tile;
    pf.m_tile_ld = static_cast<int>(fp.n_tiles);
    pf.out_mode = 1;
    lf.n_problems = 1;
    lf.counter = counter;
    const int gf = static_cast<int>(
        std::min<int64_t>(ceil_div(m_cap, um) * splits * ctas, sms));
    LMH_TRY(launch("fwd_keep_gemm", s, [&] { return launch_gemm_fwd_z(lf, gf, pair, s); }));

    const int r0 = static_cast<int>(t0), r1 = static_cast<int>(t0 + m_cap);
    LMH_TRY(launch("fwd_merge", s, [&] {
      return launch_fwd_merge(part, splits, static_cast<int>(f.T_alloc), f.idx, f.y_c, f.st, r0,
                              r1, logp, entropy, lse, nullptr, s);
    }));
    LMH_TRY(launch("bwd_prep", s, [&] {
      return launch_bwd_prep(f.idx, f.st, r0, r1, lse, entropy, grad_logp, grad_entropy,
                             temperature, coef, s);
    }));
    LMH_TRY(launch("keep_dz", s, [&] {
      return launch_fused_dz(zbuf, static_cast<int>(fp.V_pad), m_tile,
                             static_cast<int>(fp.n_tiles), coef, f.y_c, f.st, r0,
                             static_cast<int>(m_cap), V, s);
    }));

    // both gradient contractions over the whole vocabulary
    LaunchArgs lg;
    std::memset(&lg, 0, sizeof(lg));
    if (!make_map(&lg.map_a[0], zbuf, V, m_cap, 2ull * fp.V_pad, BK, BM)) return LMHEAD_ERR_CUDA;
    if (!make_map_mn(&lg.map_b[0], weight, H, V, 2ull * H, b_box_rows() / 64))
      return LMHEAD_ERR_CUDA;
    GemmArgs& ph = lg.prob[0].p;
    lg.prob[0].a_mn = 0;
    ph.m_cap = static_cast<int>(m_cap);
    ph.n_extent = H;
    ph.k_cap = V;
    ph.m_dynamic = 1;
    ph.dyn_base = static_cast<int>(t0);
    ph.dev_rows = &f.st->rows;
    ph.status = &f.st->status;
    ph.row_base = static_cast<int>(t0);
    ph.out = d_hidden;
    ph.out_ld = H;
    ph.row_map = f.idx;
    ph.accumulate = 0;
    ph.n_fastest = 1;
    if (!f.idx) {
      ph.out_mode = 1;
      if (!make_out_map_f32(&lg.map_out[0], d_hidden + t0 * H, H,
                            std::min<int64_t>(m_cap, T - t0), H))
        return LMHEAD_ERR_CUDA;
    }
    if (!make_map_mn(&lg.map_a[1], zbuf, V, m_cap, 2ull * fp.V_pad, BM / 64) ||
        !make_map_mn(&lg.map_b[1], h_blk, H, h_rows, 2ull * H, b_box_rows() / 64))
      return LMHEAD_ERR_CUDA;
    GemmArgs& pw = lg.prob[1].p;
    lg.prob[1].a_mn = 1;
    pw.m_cap = V;
    pw.n_extent = H;
    pw.k_cap = static_cast<int>(m_cap);
    pw.k_dynamic = 1;
    pw.dyn_base = static_cast<int>(t0);
    pw.dev_rows = &f.st->rows;
    pw.status = &f.st->status;
    pw.out = d_weight;
    pw.out_ld = H;
    pw.accumulate = (tb > 0 || accumulate_dweight) ? 1 : 0;
    pw.zero_if_empty = 1;
    pw.n_fastest = 1;
    pw.out_mode = pw.accumulate ? 2 : 1;
    if (!make_out_map_f32(&lg.map_out[1], d_weight, H, V, H)) return LMHEAD_ERR_CUDA;
    lg.n_problems = 2;
    lg.counter = counter + 1;
    const int gg = static_cast<int>(std::min<int64_t>(
        (ceil_div(m_cap, um) + ceil_div(V, um)) * ceil_div(H, BN) * ctas, sms));
    LMH_TRY(launch("bwd_grad_gemm", s, [&] { return launch_gemm_bwd_grad(lg, gg, pair, s); }));
  }
  return LMHEAD_OK;
}

lmhead_status lmhead_score_logits_fwd(const float* logits, const int32_t* targets,
                                      const uint8_t* loss_mask, int64_t T, int32_t V,
                                      float temperature, float* logp, float* entropy, float* lse,
                                      lmhead_stream_t stream) {
  if (T < 0 || V <= 0 || !std::isfinite(temperature) || !(temperature > 0.f))
    return LMHEAD_ERR_INVALID_ARG;
  if (T >= (int64_t{1} << 31)) return LMHEAD_ERR_UNSUPPORTED;
  if (T == 0) return LMHEAD_OK;
  if (!logits || !targets || !logp || !lse) return LMHEAD_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LMH_TRY(launch("score_logits_fwd", s, [&] {
    return launch_score_logits_fwd(logits, targets, loss_mask, T, V, temperature, logp, entropy,
                                   lse, s);
  }));
  return LMHEAD_OK;
}

lmhead_status lmhead_score_logits_bwd(const float* logits, const int32_t* targets,
                                      const uint8_t* loss_mask, int64_t T, int32_t V,
                                      float temperature, const float* grad_logp,
                                      const float* grad_entropy, const float* lse,
                                      const float* entropy, float* d_logits,
                                      lmhead_stream_t stream) {
  if (T < 0 || V <= 0 || !std::isfinite(temperature) || !(temperature > 0.f))
    return LMHEAD_ERR_INVALID_ARG;
  if (T >= (int64_t{1} << 31)) return LMHEAD_ERR_UNSUPPORTED;
  if (T == 0) return LMHEAD_OK;
  if (!logits || !targets || !lse || !d_logits || (grad_entropy && !entropy))
    return LMHEAD_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LMH_TRY(launch("score_logits_bwd", s, [&] {
    return launch_score_logits_bwd(logits, targets, loss_mask, T, V, temperature, grad_logp,
                                   grad_entropy, lse, entropy, d_logits, s);
  }));
  return LMHEAD_OK;
}

lmhead_status lmhead_selftest_bounded_wait(void* workspace, size_t workspace_bytes,
                                           uint32_t limit_ms, lmhead_stream_t stream) {
  if (!workspace || workspace_bytes < sizeof(DeviceState) || limit_ms == 0 || limit_ms > 10000)
    return LMHEAD_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return LMHEAD_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceState* st = static_cast<DeviceState*>(workspace);
  LMH_TRY(launch("clear_state", s, [&] { return launch_clear_state(st, 0, nullptr, 0, s); }));
  LMH_TRY(launch("bounded_wait_selftest", s, [&] {
    return launch_bounded_wait_selftest(&st->status, uint64_t{limit_ms} * 1000000ull, s);
  }));
  return LMHEAD_OK;
}

lmhead_status lmhead_read_device_status(const void* workspace, lmhead_stream_t stream) {
  if (!workspace) return LMHEAD_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LMHEAD_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LMHEAD_ERR_CUDA;
  return static_cast<lmhead_status>(v);
}

int64_t lmhead_read_scored_count(const void* workspace, lmhead_stream_t stream) {
  if (!workspace) return -1;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return -1;
  DeviceState st;
  if (cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  return st.rows;
}

void lmhead_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) {
    for (ProfRecord& r : g_prof) {
      cudaEventSynchronize(r.stop);
      g_event_pool.push_back(r.start);
      g_event_pool.push_back(r.stop);
    }
    g_prof.clear();
  }
  g_prof_on = on != 0;
}

int lmhead_profile_count(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  return static_cast<int>(g_prof.size());
}

lmhead_status lmhead_profile_record(int i, const char** name, float* ms) {
  ProfRecord r;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (i < 0 || i >= static_cast<int>(g_prof.size())) return LMHEAD_ERR_INVALID_ARG;
    r = g_prof[static_cast<size_t>(i)];
  }
  if (cudaEventSynchronize(r.stop) != cudaSuccess) return LMHEAD_ERR_CUDA;
  float t = 0.f;
  if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) return LMHEAD_ERR_CUDA;
  if (name) *name = r.name;
  if (ms) *ms = t;
  return LMHEAD_OK;
}

uint64_t lmhead_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int lmhead_fwd_bwd_keeps_logits(int64_t T, int32_t H, int32_t V, int32_t chunk_size,
                                int32_t* block_tokens) {
  if (check_sizes(T, H, V, 1.0f, chunk_size) != LMHEAD_OK || T == 0) return -1;
  const FusedPlan fp = plan_fused(T, H, V, chunk_size);
  if (block_tokens) *block_tokens = static_cast<int32_t>(fp.Tb);
  return fp.preferred ? 1 : 0;
}

}  // extern "C"
