// Internal interface between the host planner (lmhead_api.cu) and the
// sm_103a kernels.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace lmh {

// Tile shape of every tensor-core GEMM in the head: 128 rows (one TMEM lane
// per row) x 256 columns (fp32 accumulator columns), K staged 64 bf16 = one
// 128-byte swizzle row at a time.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr uint32_t A_TILE_BYTES = BM * BK * 2;
constexpr uint32_t B_TILE_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int EPI_WARPS = 4;
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 2 * BN;   // two accumulators, double buffered
// Epilogue staging: two 16 KB buffers (128 rows x 128 bytes, 128-byte
// swizzled) that TMA bulk-stores write out.
constexpr uint32_t STAGING_BYTES = 2 * 16384;
constexpr size_t GEMM_SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + 256 + 1024;
constexpr size_t BWD_ALL_SMEM_BYTES = GEMM_SMEM_BYTES + 1024;   // + the token-block unit table

// Device status word values (same numbers as the public lmhead_status).
constexpr int STATUS_DEVICE_TIMEOUT = 5;
constexpr int STATUS_BAD_TARGET = 6;
constexpr int STATUS_INTERNAL = 7;

// Small block of device state at the head of the workspace.
struct DeviceState {
  int status;       // first error seen on the device (0 = none)
  int rows;         // number of scored tokens T_v (written by the compaction step)
  int abort_all;    // set by a persistent kernel's CTA that gave up, so the others stop too
  int pad[61];
};

enum EpiKind : int {
  EPI_FWD_STATS = 0,   // online max / exp-sum / sum p*z / target logit per vocab split
  EPI_BWD_DZ = 1,      // dz = g_l (onehot - p) - g_e p (log p + H), divided by tau, to bf16
  EPI_STORE_F32 = 2,   // plain fp32 tile store or read-modify-write (dh, dW)
  EPI_FWD_Z = 3,       // EPI_FWD_STATS, and also keep the logits: fp16 (u - m_tile) tiles
                       // through map_out plus the per-(row, tile) reference m_tile
};

struct GemmArgs {
  // Problem extents.  M and K can be bounded by the device count of scored
  // tokens: extent = clamp(*dev_rows - dyn_base, 0, cap).
  int m_cap;
  int n_extent;
  int k_cap;
  int m_dynamic;
  int k_dynamic;
  int dyn_base;
  const int* dev_rows;
  int n_splits;          // EPI_FWD_STATS: vocab splits per token block; else 0
  int* status;
  // epilogue inputs
  float scale;           // log2(e) / tau
  int row_base;          // offset of row 0 in the per-row arrays
  int col_base;          // vocabulary id of column 0 (targets are global ids)
  const int* y_c;        // per-row wrapped target id, or -1
  float4* partials;      // EPI_FWD_STATS: [n_splits][part_ld] {m, s, S1, zy} in log2 units
  int part_ld;
  const float4* coef;    // EPI_BWD_DZ: per row {lse*log2e, g_e ln2/tau, (g_l + g_e H)/tau, g_l/tau}
  uint16_t* dz_out;      // EPI_BWD_DZ: bf16 scratch, row-major, ld = dz_ld
  int dz_ld;
  float* out;            // EPI_STORE_F32: output rows
  int64_t out_ld;
  const int* row_map;    // EPI_STORE_F32: optional output row of row (row_base + r)
  int accumulate;        // EPI_STORE_F32: 1 = add to the existing values
  int zero_if_empty;     // EPI_STORE_F32: K == 0 and !accumulate writes zeros
  float* m_tile;         // EPI_FWD_Z: [rows][m_tile_ld] reference max of each 256-column tile
  int m_tile_ld;
  int n_fastest;         // unit order: 1 = N tiles of one M block consecutively (one tile per unit)
  int m_group;           // unit order otherwise: M blocks fastest, taken in groups of m_group
                         // blocks that run through every N split before the next group
                         // starts (0 = all M blocks in one group)
  int out_mode;          // 0: per-thread global stores; 1: TMA store of map_out tiles;
                         // 2: TMA reduce-add into map_out (EPI_STORE_F32 accumulation)
};

// One launch of the tensor-core GEMM runs one or two problems (GEMMs with
// the same epilogue kind).  Work units of problem 0 come first, then those of
// problem 1; CTAs fetch units from a device counter (zeroed before the
// launch), so units with long K (put first) start first and short ones fill
// the tail.
constexpr int MAX_PROBLEMS = 2;

struct Problem {
  GemmArgs p;
  int a_mn;   // 1: the A operand is MN-major in memory (B majorness is a template flag).
              // MN-major operands take 3-D maps (64 elements, K rows, 64-element
              // chunks) with boxes of 64 x 64 x (rows per CTA / 64).
};

struct LaunchArgs {
  CUtensorMap map_a[MAX_PROBLEMS];
  CUtensorMap map_b[MAX_PROBLEMS];
  CUtensorMap map_out[MAX_PROBLEMS];   // output tiles for out_mode 1 / 2 (box 128 rows x 128 bytes)
  Problem prob[MAX_PROBLEMS];
  int n_problems;
  int* counter;
};

// The whole backward in one persistent launch on CTA pairs: the dz, dh and
// dW tiles of every backward block in one dynamically fetched sequence,
// ordered by per-tile completion flags instead of launch boundaries.  Blocks
// (token block tb, vocabulary block vb) are numbered b = tb * n_vb + vb; T_b
// and V_b are multiples of 256.  Per block the units are its dz tiles (column
// major), its dh tiles (row major) and its dW tiles (vocabulary-tile major).
// The first unit of each token block is kept in shared memory (1 KB).
constexpr int BWD_ALL_MAX_TOKEN_BLOCKS = 255;

struct BwdAllArgs {
  CUtensorMap h_k;     // hidden rows [rows, H], K-major, boxes 64 x 128: A of dz
  CUtensorMap w_k;     // W [V, H], K-major, boxes 64 x 128: B of dz (half of N per CTA)
  CUtensorMap dz_k;    // dz scratch [T_b, V_b], boxes 64 x 128: dz tile stores and A of dh
  CUtensorMap w_mn;    // W as (64, V rows, H / 64 chunks), boxes 64 x 64 x 2: MN-major B of dh
  CUtensorMap dz_mn;   // dz scratch as (64, T_b rows, V_b / 64 chunks), boxes 64 x 64 x 2: A of dW
  CUtensorMap h_mn;    // hidden rows as (64, rows, H / 64 chunks), boxes 64 x 64 x 2: B of dW
  CUtensorMap dh_out;  // d_hidden fp32 [T, H], boxes 32 x 128 (when rows are not scattered)
  CUtensorMap dw_out;  // d_weight fp32 [V, H], boxes 32 x 128
  int T_b, V_b, n_tb, n_vb, V, H, T_alloc;
  int MT, NT;          // T_b / 256 and V_b / 256: flags per block and kind
  DeviceState* st;     // scored count, status word, abort word
  float scale;         // log2(e) / tau
  const int* y_c;
  const float4* coef;
  const int* row_map;  // compaction index (d_hidden rows scattered), or NULL
  float* d_hidden;
  float* d_weight;
  int accumulate_dweight;
  int* unit_counter;   // zeroed; one per launch
  int* flags;          // per block: all dz [1], dz columns [NT], dh rows [MT], dW columns [NT]
  // -1: every unit in one launch.  w in [0, blocks]: launch w of a sequence of
  // blocks + 1 launches runs the units from block w-1's first dh tile up to
  // block w's first dh tile (launch 0: block 0's dz tiles; the last: the
  // last block's dh and dW tiles), so each launch starts with one block's
  // gradient tiles on every SM together and ends with the next block's dz
  // tiles filling its tail.
  int window;
};

// Launchers.  Each returns the launch error (cudaSuccess when enqueued).
cudaError_t launch_gemm_bwd_all(const BwdAllArgs& a, int grid, cudaStream_t s);
// pair = true runs each tile on a cluster of two CTAs (tcgen05 cta_group::2,
// 256-row units, B staged half per CTA); the B maps must then use 128-row
// K-major boxes.  `grid` is the number of CTAs wanted.
cudaError_t launch_gemm_fwd_stats(const LaunchArgs& a, int grid, bool pair, cudaStream_t s);
cudaError_t launch_gemm_bwd_dz(const LaunchArgs& a, int grid, bool pair, cudaStream_t s);
cudaError_t launch_gemm_bwd_grad(const LaunchArgs& a, int grid, bool pair, cudaStream_t s);
cudaError_t launch_gemm_fwd_z(const LaunchArgs& a, int grid, bool pair, cudaStream_t s);

// Auxiliary kernels (aux.cu).
// Mask compaction works on chunks of this many tokens; `counts` holds one
// int per chunk (compact_chunks(T) of them).
constexpr int kCompactChunk = 4096;
int compact_chunks(int T);
// Targets are ids of a vocabulary of Vt entries; the call holds rows
// [v0, v0 + Vs) of it (the whole vocabulary: v0 = 0, Vs = Vt).  y_c gets the
// local row of each scored target, -2 for a valid id held by another
// vocabulary shard, -1 for an invalid id (which also sets the status word).
cudaError_t launch_compact(const uint8_t* mask, const int32_t* targets, int T, int v0, int Vs,
                           int Vt, int T_alloc, int* counts, int* idx, int* y_c, DeviceState* st,
                           cudaStream_t s);
cudaError_t launch_targets_dense(const int32_t* targets, int T, int v0, int Vs, int Vt,
                                 int T_alloc, int* y_c, DeviceState* st, cudaStream_t s);
cudaError_t launch_gather_rows(const uint16_t* hidden, int H, const int* idx, int T_alloc,
                               const DeviceState* st, uint16_t* h_c, cudaStream_t s);
// Unscored tokens' outputs +0.0: logp / entropy / lse, or, when shard_part
// is not NULL, only the shard's partial statistics.
cudaError_t launch_zero_masked_outputs(const uint8_t* mask, int T, float* logp, float* entropy,
                                       float* lse, float4* shard_part, cudaStream_t s);
// Rows [r0, r1) of the compacted order (clipped to the scored count).  With
// shard_part != NULL the merged statistics {m, s, S1, zy} (log2 units) go
// there, in token order, instead of logp / entropy / lse.
cudaError_t launch_fwd_merge(const float4* partials, int n_splits, int part_ld, const int* idx,
                             const int* y_c, const DeviceState* st, int r0, int r1, float* logp,
                             float* entropy, float* lse, float4* shard_part, cudaStream_t s);
// logp / entropy / lse of T tokens from n_shards sets of shard statistics
// partials[j][t] (token order); Vt is the whole vocabulary's size.
cudaError_t launch_combine_shards(const float4* partials, int n_shards, int64_t T,
                                  const int32_t* targets, const uint8_t* mask, int Vt, float* logp,
                                  float* entropy, float* lse, cudaStream_t s);
// Rows [r0, r1): coefficients of scored rows, zeros past the scored count.
cudaError_t launch_bwd_prep(const int* idx, const DeviceState* st, int r0, int r1, const float* lse,
                            const float* entropy, const float* grad_logp,
                            const float* grad_entropy, float tau, float4* coef, cudaStream_t s);
// In-place logits -> dz pass over a token block of the single-call path:
// z16 holds fp16 (u - m_tile) for rows [0, rows_cap) of the block and
// columns [0, V); it becomes bf16 dz / tau.
cudaError_t launch_fused_dz(uint16_t* z16, int ld, const float* m_tile, int m_tile_ld,
                            const float4* coef, const int* y_c, const DeviceState* st, int t0,
                            int rows_cap, int V, cudaStream_t s);
cudaError_t launch_zero_masked_rows(const uint8_t* mask, int T, int H, float* d_hidden,
                                    cudaStream_t s);
// Resets the device state (status, scored count, abort word) and zeroes
// `n_counters` work-unit counters.
cudaError_t launch_clear_state(DeviceState* st, int rows_if_dense, int* counters,
                               int64_t n_counters, cudaStream_t s);

// Self-test of the bounded mbarrier wait (selftest.cu).
cudaError_t launch_bounded_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s);

// Logits-level scoring (score_logits.cu).
cudaError_t launch_score_logits_fwd(const float* logits, const int32_t* targets,
                                    const uint8_t* mask, int64_t T, int V, float tau, float* logp,
                                    float* entropy, float* lse, cudaStream_t s);
cudaError_t launch_score_logits_bwd(const float* logits, const int32_t* targets,
                                    const uint8_t* mask, int64_t T, int V, float tau,
                                    const float* grad_logp, const float* grad_entropy,
                                    const float* lse, const float* entropy, float* d_logits,
                                    cudaStream_t s);

}  // namespace lmh
