// Memory-bound helper kernels around the tensor-core GEMMs: mask
// compaction and target wrap, the gather of scored hidden rows, the
// log-sum-exp combine of per-split statistics, the per-row backward
// coefficients and the zeroing of unscored rows.
#include "kernels.h"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <utility>

namespace lmh {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kCompactThreads = 256;

// Target id of a call that holds vocabulary rows [v0, v0 + Vs) of a
// vocabulary of Vt ids (the whole vocabulary: v0 = 0, Vs = Vt = V).  Negative
// ids wrap (y in [-Vt, 0) -> y + Vt); a wrapped id in this call's rows becomes
// its local row, one held by another vocabulary shard becomes kTargetElsewhere
// (never matched by a column, no error), and an id outside [-Vt, Vt) becomes
// kTargetInvalid.
constexpr int kTargetInvalid = -1;
constexpr int kTargetElsewhere = -2;

__device__ __forceinline__ int shard_target(int y, int v0, int Vs, int Vt) {
  if (y < 0) y += Vt;
  if (y < 0 || y >= Vt) return kTargetInvalid;
  y -= v0;
  return (y >= 0 && y < Vs) ? y : kTargetElsewhere;
}

// Start of every call: status, scored count (known on the host only when no
// mask is given) and abort word, and the zeroed work-unit counters.
__global__ void clear_state_kernel(DeviceState* st, int rows, int* counters, int64_t n) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    st->status = 0;
    st->rows = rows;
    st->abort_all = 0;
  }
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    counters[i] = 0;
}

// Stable compaction of the scored positions, in two launches over chunks of
// kCompactChunk tokens (one CTA each, kCompactThreads threads).  In a chunk,
// thread t owns positions t, t + 256, ..., t + 15 * 256, so every load is
// coalesced; within one round of 256 positions a warp ballot orders them.
// (1) compact_count_kernel: scored tokens per chunk.
// (2) compact_scatter_kernel: the chunk's offset (sum of the counts before
//     it), the compact index and wrapped targets in ascending token order,
//     the scored count, and -1 targets for the padding rows.
constexpr int kCompactRounds = kCompactChunk / kCompactThreads;   // 16

__device__ __forceinline__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int k = 0; k < kCompactThreads / 32; ++k) t += red[k];
  return t;
}

__global__ void __launch_bounds__(kCompactThreads)
    compact_count_kernel(const uint8_t* __restrict__ mask, int T, int* __restrict__ counts) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  __shared__ int red[kCompactThreads / 32];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kCompactChunk;
  int cnt = 0;
#pragma unroll
  for (int c = 0; c < kCompactRounds; ++c) {
    const int64_t t = base + c * kCompactThreads + threadIdx.x;
    if (t < T) cnt += mask[t] != 0;
  }
  const int tot = block_sum(cnt, red);
  if (threadIdx.x == 0) counts[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kCompactThreads)
    compact_scatter_kernel(const uint8_t* __restrict__ mask, const int32_t* __restrict__ targets,
                           int T, int v0, int Vs, int Vt, int T_alloc,
                           const int* __restrict__ counts, int n_chunks, int* __restrict__ idx,
                           int* __restrict__ y_c, DeviceState* st) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  __shared__ int red[kCompactThreads / 32];
  __shared__ int round_warp[kCompactRounds][kCompactThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // offset of this chunk and the total, from the per-chunk counts
  int before = 0, all = 0;
  for (int k = threadIdx.x; k < n_chunks; k += kCompactThreads) {
    const int c = counts[k];
    all += c;
    if (k < static_cast<int>(blockIdx.x)) before += c;
  }
  before = block_sum(before, red);
  all = block_sum(all, red);
  // per round: a ballot orders this warp's 32 positions; warp totals in shared memory
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kCompactChunk;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t live = 0;          // bit c: position of round c is scored
  int rank[kCompactRounds];   // rank among the scored positions of this warp's round
#pragma unroll
  for (int c = 0; c < kCompactRounds; ++c) {
    const int64_t t = base + c * kCompactThreads + threadIdx.x;
    const bool f = t < T && mask[t] != 0;
    const uint32_t b = __ballot_sync(0xffffffffu, f);
    rank[c] = __popc(b & lt);
    if (f) live |= 1u << c;
    if (lane == 0) round_warp[c][w] = __popc(b);
  }
  __syncthreads();
  // exclusive prefix over (round, warp) in position order: one warp scans 128 totals
  if (w == 0) {
    int carry = 0;
    for (int c = 0; c < kCompactRounds; ++c) {
      const int v = lane < kCompactThreads / 32 ? round_warp[c][lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      if (lane < kCompactThreads / 32) round_warp[c][lane] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  int bad = 0;
#pragma unroll
  for (int c = 0; c < kCompactRounds; ++c) {
    if (live & (1u << c)) {
      const int t = static_cast<int>(base) + c * kCompactThreads + threadIdx.x;
      const int pos = before + round_warp[c][w] + rank[c];
      const int y = shard_target(targets[t], v0, Vs, Vt);
      bad |= y == kTargetInvalid;
      idx[pos] = t;
      y_c[pos] = y;
    }
  }
  for (int r = all + static_cast<int>(blockIdx.x) * kCompactThreads + threadIdx.x; r < T_alloc;
       r += n_chunks * kCompactThreads)
    y_c[r] = -1;
  if (bad) atomicCAS(&st->status, 0, STATUS_BAD_TARGET);
  if (blockIdx.x == 0 && threadIdx.x == 0) st->rows = all;
}

__global__ void targets_dense_kernel(const int32_t* __restrict__ targets, int T, int v0, int Vs,
                                     int Vt, int T_alloc, int* __restrict__ y_c, DeviceState* st) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= T_alloc) return;
  int y = kTargetInvalid;
  if (r < T) {
    y = shard_target(targets[r], v0, Vs, Vt);
    if (y == kTargetInvalid) atomicCAS(&st->status, 0, STATUS_BAD_TARGET);
  }
  y_c[r] = y;
}

// h_c[r] = hidden[idx[r]] for scored rows; zero rows up to T_alloc so that
// every tile edge past the scored count reads exact zeros.  One row per CTA
// iteration, 16-byte accesses.
__global__ void gather_rows_kernel(const uint4* __restrict__ hidden, int H8, const int* __restrict__ idx,
                                   int T_alloc, const DeviceState* st, uint4* __restrict__ h_c) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int rows = st->rows;
  for (int r = blockIdx.x; r < T_alloc; r += gridDim.x) {
    uint4* dst = h_c + static_cast<int64_t>(r) * H8;
    if (r < rows) {
      const uint4* src = hidden + static_cast<int64_t>(idx[r]) * H8;
      for (int c = threadIdx.x; c < H8; c += blockDim.x) dst[c] = src[c];
    } else {
      for (int c = threadIdx.x; c < H8; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Outputs of unscored tokens: +0.0 (the forward's logp / entropy / lse, or a
// vocabulary shard's partial statistics).
__global__ void zero_masked_outputs_kernel(const uint8_t* __restrict__ mask, int T, float* logp,
                                           float* entropy, float* lse, float4* shard_part) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T || mask[t]) return;
  if (shard_part) {
    shard_part[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  logp[t] = 0.f;
  lse[t] = 0.f;
  if (entropy) entropy[t] = 0.f;
}

// Log-sum-exp combine of n sets of statistics {m_j, s_j, S1_j, zy_j} of one
// token over disjoint parts of the vocabulary, all in log2 units: m_j the
// part's largest scaled logit u = z log2(e), s_j = sum 2^(u - m_j),
// S1_j = sum 2^(u - m_j) (u - m_j), zy_j the target's u if the target lies in
// the part, else -inf.  With M = max_j m_j and w_j = 2^(m_j - M):
//   s = sum_j w_j s_j,  S1 = sum_j w_j (S1_j + (m_j - M) s_j),  zy = max_j zy_j.
// The parts are taken in index order, so the result is deterministic.
struct Stats {
  float M, s, s1, zy;
};

__device__ __forceinline__ Stats merge_stats(const float4* __restrict__ part, int n,
                                             int64_t stride) {
  Stats r{-INFINITY, 0.f, 0.f, -INFINITY};
  for (int j = 0; j < n; ++j) r.M = fmaxf(r.M, part[j * stride].x);
  for (int j = 0; j < n; ++j) {
    const float4 q = part[j * stride];
    const float dm = q.x - r.M;
    const float wgt = exp2f(dm);
    r.s = fmaf(q.y, wgt, r.s);
    r.s1 = fmaf(wgt, fmaf(dm, q.y, q.z), r.s1);
    r.zy = fmaxf(r.zy, q.w);
  }
  return r;
}

// The forward's merge of its per-split statistics.  Writes the token's logp /
// entropy / lse in original order (lse = (M + log2 s) ln 2, logp = (zy - M -
// log2 s) ln 2, entropy = (log2 s - S1 / s) ln 2; NaN logp for an invalid
// target), or, for a vocabulary shard (shard_part != NULL), the statistics
// merged over this call's splits, which lmhead_combine_shards merges across
// shards by the same rule.
__global__ void fwd_merge_kernel(const float4* __restrict__ part, int n_splits, int part_ld,
                                 const int* __restrict__ idx, const int* __restrict__ y_c,
                                 const DeviceState* st, int r0, int r1, float* logp,
                                 float* entropy, float* lse, float4* shard_part) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int r = r0 + blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= r1 || r >= st->rows) return;
  const Stats m = merge_stats(part + r, n_splits, part_ld);
  const int t = idx ? idx[r] : r;
  if (shard_part) {
    shard_part[t] = make_float4(m.M, m.s, m.s1, m.zy);
    return;
  }
  const float l2s = log2f(m.s);
  lse[t] = (m.M + l2s) * kLn2;
  logp[t] = y_c[r] >= 0 ? (m.zy - m.M - l2s) * kLn2 : __int_as_float(0x7fc00000);
  if (entropy) entropy[t] = kLn2 * (l2s - m.s1 / m.s);
}

// Combine of vocabulary shards' statistics part[j][t] (j < n_shards, each from
// lmhead_logps_fwd_shard over one shard) into logp / entropy / lse, as the
// forward's merge does over its splits.  Unscored tokens give +0.0; an id
// outside [-Vt, Vt) gives NaN logp.
__global__ void combine_shards_kernel(const float4* __restrict__ part, int n_shards, int64_t T,
                                      const int32_t* __restrict__ targets,
                                      const uint8_t* __restrict__ mask, int Vt, float* logp,
                                      float* entropy, float* lse) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (t >= T) return;
  if (mask && !mask[t]) {
    logp[t] = 0.f;
    lse[t] = 0.f;
    if (entropy) entropy[t] = 0.f;
    return;
  }
  const Stats m = merge_stats(part + t, n_shards, T);
  const bool valid = shard_target(targets[t], 0, Vt, Vt) >= 0;
  const float l2s = log2f(m.s);
  lse[t] = (m.M + l2s) * kLn2;
  logp[t] = valid ? (m.zy - m.M - l2s) * kLn2 : __int_as_float(0x7fc00000);
  if (entropy) entropy[t] = kLn2 * (l2s - m.s1 / m.s);
}

// Per scored row: {lse * log2 e, g_e ln2 / tau, (g_l + g_e H) / tau, g_l / tau}
// so that dz / tau = -p (a d + b) + c [v == y], with d = log2 p.  Rows past
// the scored count get zeros (their dz is then exactly zero).
__global__ void bwd_prep_kernel(const int* __restrict__ idx, const DeviceState* st, int r0, int r1,
                                const float* __restrict__ lse, const float* __restrict__ entropy,
                                const float* __restrict__ grad_logp,
                                const float* __restrict__ grad_entropy, float inv_tau,
                                float4* __restrict__ coef) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  const int r = r0 + blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= r1) return;
  float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r < st->rows) {
    const int t = idx ? idx[r] : r;
    const float gl = grad_logp ? grad_logp[t] : 0.f;
    const float ge = grad_entropy ? grad_entropy[t] : 0.f;
    const float Hh = (grad_entropy && entropy) ? entropy[t] : 0.f;
    c.x = lse[t] * kLog2e;
    c.y = ge * kLn2 * inv_tau;
    c.z = fmaf(ge, Hh, gl) * inv_tau;
    c.w = gl * inv_tau;
  }
  coef[r] = c;
}

__global__ void zero_masked_rows_kernel(const uint8_t* __restrict__ mask, int T, int H4,
                                        float4* __restrict__ d_hidden) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    if (mask[t]) continue;
    float4* row = d_hidden + static_cast<int64_t>(t) * H4;
    for (int c = threadIdx.x; c < H4; c += blockDim.x) row[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// In-place logits -> dz for a token block of the single-call path.  Element
// (r, c): u - m' is stored as fp16 with m' = m_tile[r][c / 256]; with
// d = u - lse_u = log2 p:  dz / tau = -p (a d + b) + c1 [c == y]  (the
// per-row coefficients of bwd_prep_kernel), written back as bf16.  Rows
// past the scored count have zero coefficients and become exact zeros.
// Work items are (row, column range) pairs, `parts` ranges of 8-element
// groups per row, so that the CTAs share the pass evenly (with whole rows per
// CTA, 3,840 rows on 1,216 CTAs left the fourth round on a sixth of them).
// Every element is read and written by one thread.  By count, the one ex2
// per logit occupies the special-function units for about 40% of the pass,
// and four loads in flight per thread (fewer resident warps) measured slower.
__device__ __forceinline__ uint4 dz_group(uint4 raw, int c0, float base, float4 cf, int y) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 u = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    float g[2];
    const float uu[2] = {u.x, u.y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float d = uu[e] + base;
      const float pr = ex2_approx(d);
      g[e] = -pr * fmaf(cf.y, d, cf.z);
      if (c0 + 2 * k + e == y) g[e] += cf.w;
    }
    const __nv_bfloat162 bv = __floats2bfloat162_rn(g[0], g[1]);
    out[k] = *reinterpret_cast<const uint32_t*>(&bv);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void fused_dz_kernel(uint16_t* __restrict__ z, int ld, const float* __restrict__ m_tile,
                                int mt_ld, const float4* __restrict__ coef,
                                const int* __restrict__ y_c, const DeviceState* st, int t0,
                                int rows_cap, int V, int parts) {
  pdl_wait_prerequisites();
  pdl_launch_dependents();
  int dyn = st->rows - t0;
  dyn = dyn < 0 ? 0 : (dyn > rows_cap ? rows_cap : dyn);
  // rows the gradient GEMMs read: whole 128-row tiles (zero padding rows included)
  const int rows = min(rows_cap, (dyn + BM - 1) / BM * BM);
  const int groups = (V + 7) / 8;
  for (int64_t w = blockIdx.x; w < static_cast<int64_t>(rows) * parts; w += gridDim.x) {
    const int r = static_cast<int>(w / parts);
    const int part = static_cast<int>(w - static_cast<int64_t>(r) * parts);
    const int g0 = static_cast<int>(static_cast<int64_t>(groups) * part / parts);
    const int g1 = static_cast<int>(static_cast<int64_t>(groups) * (part + 1) / parts);
    const float4 cf = coef[t0 + r];
    const int y = y_c[t0 + r];
    const float* mt = m_tile + static_cast<int64_t>(r) * mt_ld;
    uint16_t* zr = z + static_cast<int64_t>(r) * ld;
    for (int gi = g0 + threadIdx.x; gi < g1; gi += blockDim.x) {
      const int c0 = gi * 8;
      uint16_t* row = zr + c0;
      const uint4 o = dz_group(*reinterpret_cast<const uint4*>(row), c0, mt[c0 / BN] - cf.x, cf, y);
      if (c0 + 8 <= V) {
        *reinterpret_cast<uint4*>(row) = o;
      } else {
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < V)
            row[j] = static_cast<uint16_t>((j & 1) ? (ow[j >> 1] >> 16) : (ow[j >> 1] & 0xFFFFu));
      }
    }
  }
}

// Launch with programmatic dependent launch: the kernel may start while its
// predecessor in the stream finishes; every helper kernel waits for the
// predecessor's completion (griddepcontrol.wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid < 1 ? 1 : grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Threads per CTA for a kernel that sweeps one row of `vecs` 16-byte
// vectors per CTA iteration: the largest of 256, 128, 64, 32 that divides the
// row, so that no pass over a row leaves warps idle.
int row_threads(int vecs) {
  for (int t = 256; t >= 32; t >>= 1)
    if (vecs % t == 0) return t;
  return 256;
}

int grid_for(int64_t n, int threads, int cap = 4 * 152 * 8) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  return static_cast<int>(g < cap ? g : cap);
}

}  // namespace

cudaError_t launch_clear_state(DeviceState* st, int rows_if_dense, int* counters,
                               int64_t n_counters, cudaStream_t s) {
  return launch_pdl(clear_state_kernel, grid_for(n_counters, 256, 152), 256, s, st,
                    rows_if_dense, counters, n_counters);
}

int compact_chunks(int T) { return (T + kCompactChunk - 1) / kCompactChunk; }

cudaError_t launch_compact(const uint8_t* mask, const int32_t* targets, int T, int v0, int Vs,
                           int Vt, int T_alloc, int* counts, int* idx, int* y_c, DeviceState* st,
                           cudaStream_t s) {
  const int n = compact_chunks(T);
  if (n < 1) return cudaSuccess;
  const cudaError_t e = launch_pdl(compact_count_kernel, n, kCompactThreads, s, mask, T, counts);
  if (e != cudaSuccess) return e;
  return launch_pdl(compact_scatter_kernel, n, kCompactThreads, s, mask, targets, T, v0, Vs, Vt,
                    T_alloc, static_cast<const int*>(counts), n, idx, y_c, st);
}

cudaError_t launch_targets_dense(const int32_t* targets, int T, int v0, int Vs, int Vt,
                                 int T_alloc, int* y_c, DeviceState* st, cudaStream_t s) {
  return launch_pdl(targets_dense_kernel, (T_alloc + 255) / 256, 256, s, targets, T, v0, Vs, Vt,
                    T_alloc, y_c, st);
}

cudaError_t launch_gather_rows(const uint16_t* hidden, int H, const int* idx, int T_alloc,
                               const DeviceState* st, uint16_t* h_c, cudaStream_t s) {
  const int H8 = H / 8;
  return launch_pdl(gather_rows_kernel, grid_for(T_alloc, 1, 152 * 32), row_threads(H8), s,
                    reinterpret_cast<const uint4*>(hidden), H8, idx, T_alloc, st,
                    reinterpret_cast<uint4*>(h_c));
}

cudaError_t launch_zero_masked_outputs(const uint8_t* mask, int T, float* logp, float* entropy,
                                       float* lse, float4* shard_part, cudaStream_t s) {
  return launch_pdl(zero_masked_outputs_kernel, (T + 255) / 256, 256, s, mask, T, logp, entropy,
                    lse, shard_part);
}

cudaError_t launch_fwd_merge(const float4* partials, int n_splits, int part_ld, const int* idx,
                             const int* y_c, const DeviceState* st, int r0, int r1, float* logp,
                             float* entropy, float* lse, float4* shard_part, cudaStream_t s) {
  if (r1 <= r0) return cudaSuccess;
  return launch_pdl(fwd_merge_kernel, (r1 - r0 + 255) / 256, 256, s, partials, n_splits, part_ld,
                    idx, y_c, st, r0, r1, logp, entropy, lse, shard_part);
}

cudaError_t launch_combine_shards(const float4* partials, int n_shards, int64_t T,
                                  const int32_t* targets, const uint8_t* mask, int Vt, float* logp,
                                  float* entropy, float* lse, cudaStream_t s) {
  const int64_t blocks = (T + 255) / 256;
  return launch_pdl(combine_shards_kernel, static_cast<int>(blocks), 256, s, partials, n_shards,
                    T, targets, mask, Vt, logp, entropy, lse);
}

cudaError_t launch_bwd_prep(const int* idx, const DeviceState* st, int r0, int r1, const float* lse,
                            const float* entropy, const float* grad_logp,
                            const float* grad_entropy, float tau, float4* coef, cudaStream_t s) {
  if (r1 <= r0) return cudaSuccess;
  return launch_pdl(bwd_prep_kernel, (r1 - r0 + 255) / 256, 256, s, idx, st, r0, r1, lse, entropy,
                    grad_logp, grad_entropy, 1.0f / tau, coef);
}

cudaError_t launch_fused_dz(uint16_t* z16, int ld, const float* m_tile, int m_tile_ld,
                            const float4* coef, const int* y_c, const DeviceState* st, int t0,
                            int rows_cap, int V, cudaStream_t s) {
  // ranges of about 4096 groups (32,768 logits, 64 KB read and written) per row
  const int groups = (V + 7) / 8;
  const int parts = (groups + 4095) / 4096;
  return launch_pdl(fused_dz_kernel, grid_for(static_cast<int64_t>(rows_cap) * parts, 1, 152 * 8),
                    256, s, z16, ld, m_tile, m_tile_ld, coef, y_c, st, t0, rows_cap, V, parts);
}

cudaError_t launch_zero_masked_rows(const uint8_t* mask, int T, int H, float* d_hidden,
                                    cudaStream_t s) {
  const int H4 = H / 4;
  return launch_pdl(zero_masked_rows_kernel, grid_for(T, 1, 152 * 32), row_threads(H4), s, mask, T,
                    H4, reinterpret_cast<float4*>(d_hidden));
}

}  // namespace lmh
