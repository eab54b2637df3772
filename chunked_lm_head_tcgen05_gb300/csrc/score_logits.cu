// Logits-level scoring for callers that already hold a chunk's logits:
// per-row log-sum-exp, target log-prob and entropy (forward), and the
// cotangent of the logits (backward), with the non-finite semantics stated
// in include/lmhead.h.  Both passes are HBM-bound: one read of the logits
// forward; one read and one write backward.  The forward reduces a row in one
// CTA; the backward, whose elements need only per-row values, spreads each
// row over several CTAs (independent column ranges) so that the last wave of
// rows does not leave most SMs idle.  16-byte loads when the row layout allows
// them.
#include "kernels.h"
#include "ptx.cuh"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

namespace {

constexpr int kFwdThreads = 256;    // forward: one CTA per row
constexpr int kFwdUnroll = 8;       // forward: 16-byte loads in flight per thread
constexpr int kThreads = 256;       // backward: one CTA per (row, column range)
constexpr int kUnroll = 4;          // 16-byte loads in flight per thread
constexpr int kMaxRowParts = 16;    // column ranges per row in the backward
constexpr int kColsPerPart = 16384; // about 64 KB of fp32 logits per range
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int wrap_target(int y, int V) {
  if (y < 0) y += V;
  return (y >= 0 && y < V) ? y : -1;
}

// Running base-2 statistics over the finite entries seen by one thread.
struct Stats {
  float m, s, s1;   // max, sum 2^(u-m), sum 2^(u-m)(u-m)
  int bad;          // saw NaN or +inf
};

// Fold n values into the running statistics: one max over the chunk, then
// the exponentials against it.  NaN or +inf set `bad` (NaN by its failed
// self-comparison, +inf through the maximum); -inf adds exactly nothing: its
// exponent d is clamped to -1e30, whose ex2 is +0, so e and e * d are zeros.
// A NaN's exponent is clamped the same way; its row is reported as NaN anyway.
template <int N>
__device__ __forceinline__ void stats_add_chunk(Stats& st, const float (&x)[N], float scale) {
  float cmax = -INFINITY;
  bool nan = false;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    cmax = fmaxf(cmax, x[j]);   // ignores NaN
    nan |= x[j] != x[j];
  }
  if (nan || cmax == INFINITY) {
    st.bad = 1;
    return;   // the row's results are NaN: its sums are never used
  }
  const float cm = cmax * scale;
  if (cm > st.m) {
    const float dm = st.m - cm;   // -inf on the first finite entry
    const float r = lmh::ex2_approx(dm);
    st.s1 = st.s > 0.f ? r * fmaf(dm, st.s, st.s1) : 0.f;
    st.s *= r;
    st.m = cm;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const float d = fmaxf(fmaf(x[j], scale, -st.m), -1e30f);
    const float e = lmh::ex2_approx(d);
    st.s += e;
    st.s1 = fmaf(e, d, st.s1);
  }
}

__device__ __forceinline__ Stats stats_merge(Stats a, Stats b) {
  const int bad = a.bad | b.bad;
  if (b.s == 0.f) {
    a.bad = bad;
    return a;
  }
  if (a.s == 0.f) {
    b.bad = bad;
    return b;
  }
  const float M = fmaxf(a.m, b.m);
  const float da = a.m - M, db = b.m - M;
  const float wa = exp2f(da), wb = exp2f(db);
  Stats r;
  r.m = M;
  r.s = fmaf(a.s, wa, b.s * wb);
  r.s1 = fmaf(wa, fmaf(da, a.s, a.s1), wb * fmaf(db, b.s, b.s1));
  r.bad = bad;
  return r;
}

// One CTA per row (rows taken in turn when there are more rows than CTAs).
__global__ void __launch_bounds__(kFwdThreads)
    score_logits_fwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ targets,
                            const uint8_t* __restrict__ mask, int64_t T, int V, float scale,
                            int vec4, float* logp, float* entropy, float* lse) {
  __shared__ Stats red[kFwdThreads / 32];
  __shared__ float zy_s;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    if (mask && !mask[t]) {
      if (threadIdx.x == 0) {
        logp[t] = 0.f;
        lse[t] = 0.f;
        if (entropy) entropy[t] = 0.f;
      }
      continue;
    }
    const float* row = logits + t * static_cast<int64_t>(V);
    const int y = wrap_target(targets[t], V);
    Stats st{-INFINITY, 0.f, 0.f, 0};
    if (vec4) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int n4 = V / 4;
      int i = threadIdx.x;
      for (; i + (kFwdUnroll - 1) * kFwdThreads < n4; i += kFwdUnroll * kFwdThreads) {
        float x[4 * kFwdUnroll];
#pragma unroll
        for (int k = 0; k < kFwdUnroll; ++k) {
          const float4 q = r4[i + k * kFwdThreads];
          x[4 * k] = q.x;
          x[4 * k + 1] = q.y;
          x[4 * k + 2] = q.z;
          x[4 * k + 3] = q.w;
        }
        stats_add_chunk(st, x, scale);
      }
      for (; i < n4; i += kFwdThreads) {
        const float4 q = r4[i];
        const float x[4] = {q.x, q.y, q.z, q.w};
        stats_add_chunk(st, x, scale);
      }
    } else {
      for (int i = threadIdx.x; i < V; i += kFwdThreads) {
        const float x[1] = {row[i]};
        stats_add_chunk(st, x, scale);
      }
    }
    if (threadIdx.x == 0) zy_s = y >= 0 ? row[y] * scale : __int_as_float(0x7fc00000);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Stats b;
      b.m = __shfl_xor_sync(0xffffffffu, st.m, o);
      b.s = __shfl_xor_sync(0xffffffffu, st.s, o);
      b.s1 = __shfl_xor_sync(0xffffffffu, st.s1, o);
      b.bad = __shfl_xor_sync(0xffffffffu, st.bad, o);
      st = stats_merge(st, b);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
      Stats a = red[0];
      for (int w = 1; w < kFwdThreads / 32; ++w) a = stats_merge(a, red[w]);
      float L, H, lp;
      if (a.bad) {
        L = H = lp = __int_as_float(0x7fc00000);
      } else if (a.s == 0.f) {   // no finite logit in the row
        L = -INFINITY;
        H = lp = __int_as_float(0x7fc00000);
      } else {
        const float l2s = log2f(a.s);
        L = (a.m + l2s) * kLn2;
        H = kLn2 * (l2s - a.s1 / a.s);
        lp = (zy_s - a.m - l2s) * kLn2;   // NaN for an invalid id, -inf for a -inf logit
      }
      lse[t] = L;
      logp[t] = lp;
      if (entropy) entropy[t] = H;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float cotangent(float x, float scale, float lse_u, float a, float b,
                                           float c1, bool is_target) {
  if (!isfinite(x)) return 0.f;   // isfinite mask
  const float d = fmaf(x, scale, -lse_u);
  const float p = lmh::ex2_approx(d);
  float g = -p * fmaf(a, d, b);
  if (is_target) g += c1;
  return g;
}

// Independent CTAs over (row, column range): kp ranges per row, work item w is
// row w / kp, range w % kp.  Every element is read and written by one thread,
// so d_logits may be the logits buffer itself.
__global__ void __launch_bounds__(kThreads)
    score_logits_bwd_kernel(const float* logits, const int32_t* __restrict__ targets,
                            const uint8_t* __restrict__ mask, int64_t T, int V, int kp,
                            float scale, float inv_tau, int vec4,
                            const float* __restrict__ grad_logp,
                            const float* __restrict__ grad_entropy,
                            const float* __restrict__ lse, const float* __restrict__ entropy,
                            float* d_logits) {
  const int n = vec4 ? V / 4 : V;
  for (int64_t w = blockIdx.x; w < T * kp; w += gridDim.x) {
    const int64_t t = w / kp;
    const int part = static_cast<int>(w - t * kp);
    const int b = static_cast<int>(static_cast<int64_t>(n) * part / kp);
    const int e = static_cast<int>(static_cast<int64_t>(n) * (part + 1) / kp);
    const float* row = logits + t * static_cast<int64_t>(V);
    float* out = d_logits + t * static_cast<int64_t>(V);
    const bool scored = !mask || mask[t];
    if (!scored) {
      if (vec4) {
        float4* o4 = reinterpret_cast<float4*>(out);
        for (int i = b + threadIdx.x; i < e; i += kThreads) o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int i = b + threadIdx.x; i < e; i += kThreads) out[i] = 0.f;
      }
      continue;
    }
    const float gl = grad_logp ? grad_logp[t] : 0.f;
    const float ge = grad_entropy ? grad_entropy[t] : 0.f;
    const float Hh = grad_entropy ? entropy[t] : 0.f;
    const float lse_u = lse[t] * kLog2e;
    const float a = ge * kLn2 * inv_tau;
    const float bb = fmaf(ge, Hh, gl) * inv_tau;
    const float c1 = gl * inv_tau;
    const int y = wrap_target(targets[t], V);
    if (vec4) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      float4* o4 = reinterpret_cast<float4*>(out);
      int i = b + threadIdx.x;
      for (; i + (kUnroll - 1) * kThreads < e; i += kUnroll * kThreads) {
        float4 q[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) q[k] = r4[i + k * kThreads];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
          const int c = 4 * (i + k * kThreads);
          float4 g;
          g.x = cotangent(q[k].x, scale, lse_u, a, bb, c1, c == y);
          g.y = cotangent(q[k].y, scale, lse_u, a, bb, c1, c + 1 == y);
          g.z = cotangent(q[k].z, scale, lse_u, a, bb, c1, c + 2 == y);
          g.w = cotangent(q[k].w, scale, lse_u, a, bb, c1, c + 3 == y);
          o4[i + k * kThreads] = g;
        }
      }
      for (; i < e; i += kThreads) {
        const float4 q = r4[i];
        const int c = 4 * i;
        float4 g;
        g.x = cotangent(q.x, scale, lse_u, a, bb, c1, c == y);
        g.y = cotangent(q.y, scale, lse_u, a, bb, c1, c + 1 == y);
        g.z = cotangent(q.z, scale, lse_u, a, bb, c1, c + 2 == y);
        g.w = cotangent(q.w, scale, lse_u, a, bb, c1, c + 3 == y);
        o4[i] = g;
      }
    } else {
      for (int i = b + threadIdx.x; i < e; i += kThreads)
        out[i] = cotangent(row[i], scale, lse_u, a, bb, c1, i == y);
    }
  }
}

int sm_count_now() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  return sms;
}

// Column ranges per row in the backward: about kColsPerPart columns each, at
// most `cap`.
int parts_per_row(int V, int cap) {
  const int k = V / kColsPerPart;
  return k < 1 ? 1 : (k > cap ? cap : k);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace lmh {

cudaError_t launch_score_logits_fwd(const float* logits, const int32_t* targets,
                                    const uint8_t* mask, int64_t T, int V, float tau, float* logp,
                                    float* entropy, float* lse, cudaStream_t s) {
  const int vec4 = (V % 4 == 0 && aligned16(logits)) ? 1 : 0;
  const int64_t cap = static_cast<int64_t>(sm_count_now()) * 4;
  const int grid = static_cast<int>(T < cap ? T : cap);
  score_logits_fwd_kernel<<<grid, kFwdThreads, 0, s>>>(logits, targets, mask, T, V,
                                                        kLog2e / tau, vec4, logp, entropy, lse);
  return cudaGetLastError();
}

cudaError_t launch_score_logits_bwd(const float* logits, const int32_t* targets,
                                    const uint8_t* mask, int64_t T, int V, float tau,
                                    const float* grad_logp, const float* grad_entropy,
                                    const float* lse, const float* entropy, float* d_logits,
                                    cudaStream_t s) {
  const int vec4 = (V % 4 == 0 && aligned16(logits) && aligned16(d_logits)) ? 1 : 0;
  const int kp = parts_per_row(V, kMaxRowParts);
  const int64_t cap = static_cast<int64_t>(sm_count_now()) * 16;
  const int64_t items = T * kp;
  const int grid = static_cast<int>(items < cap ? items : cap);
  score_logits_bwd_kernel<<<grid, kThreads, 0, s>>>(logits, targets, mask, T, V, kp,
                                                     kLog2e / tau, 1.0f / tau, vec4, grad_logp,
                                                     grad_entropy, lse, entropy, d_logits);
  return cudaGetLastError();
}

}  // namespace lmh
