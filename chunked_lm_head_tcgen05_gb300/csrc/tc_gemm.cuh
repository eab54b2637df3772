// Persistent, warp-specialised tcgen05 GEMM with fused epilogues for the
// chunked LM head (sm_103a).
//
// Per CTA, 192 threads:
//   warp 0      scheduler + TMA producer (one elected lane): fetches work
//               units from a device counter, passes each unit index to the
//               other roles through a small shared-memory ring, and streams
//               the unit's A and B tiles into a shared-memory ring,
//               128-byte swizzled.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and issues tcgen05.mma (one elected lane).
//   warps 2..5  epilogue: each thread owns one accumulator row (TMEM lane)
//               and reads it 32 columns at a time with tcgen05.ld.
// Accumulators are double buffered, so the epilogue of one tile overlaps the
// MMAs of the next.
//
// PAIR = true runs the same roles on a cluster of two CTAs (two SMs) that
// share one 256 x 256 output tile: each CTA stages its own 128 rows of A and
// half (128 columns) of B, the even CTA issues tcgen05.mma.cta_group::2
// (M = 256) over both CTAs' shared memory, and each CTA's TMEM receives its
// 128 rows of D.  Per SM this halves the B traffic and the B staging space,
// so six 64-wide K steps fit instead of four.  Where both operands are
// K-major with K = H (forward and dz tiles), a pair stages them two K steps
// at a time (three 64 KB stages, one 3-D TMA box per operand each).  The even CTA fetches the work units and
// forwards them to its peer; the peer's loads complete on the even CTA's
// barriers, and MMA completion is multicast back to both CTAs.
//
// A launch holds one or two problems (see LaunchArgs).  A work unit is one
// block of M rows (128, or 256 for a pair) and a contiguous range of
// 256-column N tiles: for the forward statistics the range is a vocabulary
// split (the running softmax statistics stay in registers across it); for
// the per-block dz GEMM a few adjacent tiles (the host sets n_splits);
// otherwise one tile.  Units of problem 0 are numbered first.
// Fetching units dynamically keeps every SM busy until the end when units
// differ in length or speed.  Every unit is computed entirely by one CTA (or
// pair) in a fixed order, so results do not depend on who took it.
//
// Every wait on an mbarrier is bounded (about 2 s of wall time); when one
// gives up the CTA records STATUS_DEVICE_TIMEOUT in the device status word,
// lets its in-flight copies and MMAs finish, frees TMEM and exits.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

#include <atomic>
#include <climits>
#include <type_traits>

namespace lmh {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int SCHED_DEPTH = 4;
constexpr int MAX_STAGES = 6;
// The next unit's index is fetched this many K steps before the current
// unit's last load, so that the fetch's latency is hidden behind the loads.
constexpr int FETCH_AHEAD_KB = 8;

template <bool PAIR>
struct TileCfg {
  static constexpr int CTAS = PAIR ? 2 : 1;
  static constexpr int UNIT_M = BM * CTAS;            // output rows per work unit
  static constexpr int B_ROWS = BN / CTAS;            // N columns of B staged per CTA
  static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;
  static constexpr uint32_t STAGE = A_TILE_BYTES + B_BYTES;
  static constexpr int NSTAGE = PAIR ? 6 : 4;
  static_assert(NSTAGE * STAGE <= STAGES * STAGE_BYTES, "stage ring exceeds the shared memory plan");
  static_assert(NSTAGE <= MAX_STAGES, "too many stages");
};

struct SharedCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t sfull[SCHED_DEPTH];
  uint64_t sempty[SCHED_DEPTH];
  uint64_t drain;
  int sched[SCHED_DEPTH];
  uint32_t tmem_base;
  int abort;
  int epi_u;    // unit index broadcast to the epilogue warps
  int epi_ok;   // accumulator-ready flag broadcast to the epilogue warps
};
static_assert(sizeof(SharedCtl) <= 256, "control block exceeds its shared memory slot");

// Wait for `parity` on `bar`; false if it gave up (time limit, or another
// role of this CTA gave up first).  CLUSTER selects acquire at cluster scope
// (the barrier is also arrived on by the peer CTA).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                             int* status, uint64_t limit_ns = WAIT_LIMIT_NS) {
  auto poll = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (poll()) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort = 1;
      atomicCAS(status, 0, STATUS_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Time-limited wait used only while draining after an abort.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ void pause_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

struct Sched {
  int M, K, m_tiles, n_tiles, n_splits, k_blocks, units, n_fastest, m_group;

  __device__ __forceinline__ void init(const GemmArgs& p, int unit_m) {
    int dev = 0;
    if (p.m_dynamic || p.k_dynamic) dev = *p.dev_rows - p.dyn_base;
    dev = dev < 0 ? 0 : dev;
    M = p.m_dynamic ? min(dev, p.m_cap) : p.m_cap;
    K = p.k_dynamic ? min(dev, p.k_cap) : p.k_cap;
    m_tiles = (M + unit_m - 1) / unit_m;
    n_tiles = (p.n_extent + BN - 1) / BN;
    n_splits = p.n_splits > 0 ? min(p.n_splits, n_tiles) : n_tiles;
    k_blocks = (K + BK - 1) / BK;
    units = m_tiles * n_splits;
    n_fastest = p.n_fastest && n_splits == n_tiles;
    m_group = (p.m_group > 0 && p.m_group < m_tiles) ? p.m_group : m_tiles;
  }

  // Unit u -> M block m and N tiles [nb, ne).  M-fastest order lets units
  // that run together share the B panel; N-fastest lets them share A.  In
  // M-fastest order the M blocks are taken m_group at a time: a group's
  // units (its blocks x every split) are numbered before the next group's,
  // so the A panels in use at once stay within m_group blocks (the last
  // group may be smaller).  With one group this is plain M-fastest order.
  __device__ __forceinline__ void unit(int u, int& m, int& split, int& nb, int& ne) const {
    if (n_fastest) {
      m = u / n_splits;
      split = u - m * n_splits;
    } else {
      const int per_group = m_group * n_splits;
      const int m0 = (u / per_group) * m_group;
      const int gm = min(m_group, m_tiles - m0);
      const int r = u - (m0 / m_group) * per_group;
      split = r / gm;
      m = m0 + (r - split * gm);
    }
    nb = static_cast<int>(static_cast<long long>(split) * n_tiles / n_splits);
    ne = static_cast<int>(static_cast<long long>(split + 1) * n_tiles / n_splits);
  }
};

// Global unit index -> (problem, unit within it).
__device__ __forceinline__ int split_unit(const Sched& s0, int u, int& q) {
  if (u < s0.units) {
    q = 0;
    return u;
  }
  q = 1;
  return u - s0.units;
}

// Write one thread's 128-byte row piece (8 x 16 bytes) into staging buffer
// (nstore & 1) in the 128-byte swizzled layout and hand the 128-row tile to
// TMA (store, or reduce-add for mode 2).  All 128 epilogue threads call it
// together; `issuer` is the one thread that drives TMA.  Every tile store
// starts at a non-negative row and at a column that is a multiple of 32
// elements; a coordinate outside that is never issued (a TMA store there
// would fault the context): it is recorded as STATUS_INTERNAL instead.
__device__ __forceinline__ void stage_out(const uint32_t* w, uint32_t stg0, uint32_t nstore,
                                          int lrow, bool issuer, const CUtensorMap* map, int mode,
                                          int x, int y, int* status) {
  const uint32_t buf = stg0 + (nstore & 1u) * 16384u;
  if (issuer && nstore >= 2) bulk_wait_read<1>();
  named_bar_sync(1, 128);
  const uint32_t rowb = buf + static_cast<uint32_t>(lrow) * 128u;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(rowb + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(lrow) & 7u)) << 4),
                 w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  fence_async_smem();
  named_bar_sync(1, 128);
  if (issuer) {
    if (x < 0 || y < 0 || (x & 31) != 0)
      atomicCAS(status, 0, STATUS_INTERNAL);
    else if (mode == 2)
      tma_reduce_add_2d(map, buf, x, y);
    else
      tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
}

template <int EPI, bool B_MN, bool PAIR>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ LaunchArgs L) {
  using C = TileCfg<PAIR>;
  // K steps per operand stage.  Where both operands are K-major with K = H
  // (the forward kernels and the per-block dz GEMM) and the tile is a CTA
  // pair's, a stage holds two 64-wide K steps of each operand, loaded by one
  // 3-D TMA box per operand (64 elements x rows x 2 K chunks): half the TMA
  // instructions and barrier round trips per K step.  The host passes
  // K-major 3-D maps (make_map_k3) and never an MN-major A for these.
  constexpr int KS = (PAIR && !B_MN && EPI != EPI_STORE_F32) ? 2 : 1;
  constexpr int NST = C::NSTAGE / KS;
  constexpr uint32_t STG = C::STAGE * KS;
  constexpr uint32_t ABYTES = A_TILE_BYTES * KS;
  static_assert(NST * KS == C::NSTAGE, "stage ring does not divide into K-step pairs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + STAGES * STAGE_BYTES + STAGING_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int* const status = L.prob[0].p.status;
  const uint32_t rank = PAIR ? cluster_cta_rank() : 0u;
  const bool leader = rank == 0;

  // The next kernel in the stream may begin its own prologue once every CTA
  // of this one is resident; it waits for this grid's results before use.
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&ctl->tfull[b]), 1);
      mbar_init(smem_addr(&ctl->tempty[b]), EPI_WARPS * C::CTAS);
    }
    for (int s = 0; s < SCHED_DEPTH; ++s) {
      mbar_init(smem_addr(&ctl->sfull[s]), 1);
      mbar_init(smem_addr(&ctl->sempty[s]), 2 * C::CTAS);
    }
    mbar_init(smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_addr(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort = &ctl->abort;
  const uint32_t smem_base = smem_addr(smem);

  // Everything above only touched this CTA's own resources; inputs written
  // by earlier kernels (scored count, counters, operands) are read below.
  pdl_wait_prerequisites();
  Sched sc0, sc1;
  sc0.init(L.prob[0].p, C::UNIT_M);
  if (L.n_problems > 1) {
    sc1.init(L.prob[1].p, C::UNIT_M);
  } else {
    sc1 = sc0;
    sc1.units = 0;
  }
  const int total_units = sc0.units + sc1.units;

  // scheduler ring: the even CTA fetches, the odd CTA reads its copy
  auto sched_take = [&](int slot, uint32_t spar, int& u) -> bool {
    if (!wait_bounded<PAIR>(smem_addr(&ctl->sfull[slot]), spar, abort, status)) return false;
    u = ctl->sched[slot];
    return true;
  };
  auto sched_release = [&](int slot) {
    if (PAIR && !leader)
      mbar_arrive_remote(map_to_cta(smem_addr(&ctl->sempty[slot]), 0));
    else
      mbar_arrive(smem_addr(&ctl->sempty[slot]));
  };

  if (warp == 0) {
    // ------------------------------------------------------ scheduler + producer
    if (lane == 0) {
      for (int q = 0; q < L.n_problems; ++q) {
        tma_prefetch_map(&L.map_a[q]);
        tma_prefetch_map(&L.map_b[q]);
      }
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_par = 0;
      bool ok = true;
      int ahead = -1;   // unit index fetched ahead, -1 = none
      for (int i = 0; ok; ++i) {
        const int slot = i & (SCHED_DEPTH - 1);
        const uint32_t spar = (i / SCHED_DEPTH) & 1;
        int u;
        if (leader) {
          if (!wait_bounded<PAIR>(smem_addr(&ctl->sempty[slot]), spar ^ 1, abort, status)) {
            ok = false;
            break;
          }
          u = ahead >= 0 ? ahead : atomicAdd(L.counter, 1);
          ahead = -1;
          if (u >= total_units) u = -1;
          ctl->sched[slot] = u;
          if constexpr (PAIR) {
            st_shared_remote(map_to_cta(smem_addr(&ctl->sched[slot]), 1), u);
            mbar_arrive_remote(map_to_cta(smem_addr(&ctl->sfull[slot]), 1));
          }
          mbar_arrive(smem_addr(&ctl->sfull[slot]));
        } else {
          if (!sched_take(slot, spar, u)) {
            ok = false;
            break;
          }
          sched_release(slot);
        }
        if (u < 0) break;
        int q;
        const int lu = split_unit(sc0, u, q);
        const Sched s = q ? sc1 : sc0;
        if (s.k_blocks == 0) continue;
        const CUtensorMap* ma = &L.map_a[q];
        const CUtensorMap* mb = &L.map_b[q];
        // the A layout is fixed per problem: the K loop is compiled for each
        // so that no per-step test of it is left in the issue path
        auto produce = [&](auto amn_tag) {
          constexpr bool A_MN = decltype(amn_tag)::value;
          int m, split, nb, ne;
          s.unit(lu, m, split, nb, ne);
          const int arow = m * C::UNIT_M + static_cast<int>(rank) * BM;
          for (int n = nb; ok && n < ne; ++n) {
            const int bcol = n * BN + static_cast<int>(rank) * C::B_ROWS;
            const int kb_fetch = (max(0, s.k_blocks - FETCH_AHEAD_KB) / KS) * KS;
            for (int kb = 0; kb < s.k_blocks; kb += KS) {
              if (leader && ahead < 0 && n == ne - 1 && kb == kb_fetch)
                ahead = atomicAdd(L.counter, 1);
              if (!wait_bounded<PAIR>(smem_addr(&ctl->empty[stage]), phase ^ 1, abort, status)) {
                ok = false;
                break;
              }
              const uint32_t fb_local = smem_addr(&ctl->full[stage]);
              if (leader) mbar_arrive_expect_tx(fb_local, STG * C::CTAS);
              const uint32_t sa = smem_base + stage * STG;
              const uint32_t sb = sa + ABYTES;
              // MN-major operands use 3-D maps (64 elements, K rows, 64-element
              // chunks): one instruction loads all of this CTA's chunks
              if constexpr (KS == 2) {
                // K chunks kb and kb + 1 of the K-major 3-D maps land 16 KB
                // apart, each the swizzled image of one 64-wide K step; past
                // the last chunk the box reads zeros (never multiplied)
                const uint32_t fb = map_to_cta(fb_local, 0);
                tma_load_3d_pair(sa, ma, fb, 0, arow, kb);
                tma_load_3d_pair(sb, mb, fb, 0, bcol, kb);
              } else if constexpr (PAIR) {
                const uint32_t fb = map_to_cta(fb_local, 0);
                if constexpr (!A_MN)
                  tma_load_2d_pair(sa, ma, fb, kb * BK, arow);
                else
                  tma_load_3d_pair(sa, ma, fb, 0, kb * BK, arow / 64);
                if constexpr (!B_MN)
                  tma_load_2d_pair(sb, mb, fb, kb * BK, bcol);
                else
                  tma_load_3d_pair(sb, mb, fb, 0, kb * BK, bcol / 64);
              } else {
                if constexpr (!A_MN)
                  tma_load_2d(sa, ma, fb_local, kb * BK, arow);
                else
                  tma_load_3d(sa, ma, fb_local, 0, kb * BK, arow / 64);
                if constexpr (!B_MN)
                  tma_load_2d(sb, mb, fb_local, kb * BK, bcol);
                else
                  tma_load_3d(sb, mb, fb_local, 0, kb * BK, bcol / 64);
              }
              issued_mask |= 1u << stage;
              issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
              if (++stage == NST) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        };
        if (KS == 1 && L.prob[q].a_mn != 0)
          produce(std::true_type{});
        else
          produce(std::false_type{});
      }
      if (!ok) {
        if constexpr (PAIR) {
          pause_ns(100000);   // let copies already issued land before exit
        } else {
          for (int s = 0; s < NST; ++s)
            if (issued_mask & (1u << s))
              wait_drain(smem_addr(&ctl->full[s]), (issued_par >> s) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t B_LBO = 8192;   // MN-major: the 64-wide N chunks are 8 KB apart
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int slot = i & (SCHED_DEPTH - 1);
        const uint32_t spar = (i / SCHED_DEPTH) & 1;
        int u;
        if (!sched_take(slot, spar, u)) {
          ok = false;
          break;
        }
        sched_release(slot);
        if (u < 0) break;
        int q;
        const int lu = split_unit(sc0, u, q);
        const Sched s = q ? sc1 : sc0;
        if (s.k_blocks == 0) continue;
        auto issue = [&](auto amn_tag) {
          constexpr bool A_MN = decltype(amn_tag)::value;
          constexpr uint32_t IDESC = idesc_bf16_f32(C::UNIT_M, BN, A_MN, B_MN);
          int m, split, nb, ne;
          s.unit(lu, m, split, nb, ne);
          for (int n = nb; ok && n < ne; ++n) {
            if (!wait_bounded<PAIR>(smem_addr(&ctl->tempty[acc]), acc_phase ^ 1, abort, status)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < s.k_blocks; kb += KS) {
              if (!wait_bounded<PAIR>(smem_addr(&ctl->full[stage]), phase, abort, status)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              const uint32_t sa0 = smem_base + stage * STG;
              const uint32_t sb0 = sa0 + ABYTES;
#pragma unroll
              for (int j = 0; j < KS; ++j) {
                if (kb + j >= s.k_blocks) break;   // zero-filled K step past the end
                const uint32_t sa = sa0 + j * A_TILE_BYTES;
                const uint32_t sb = sb0 + j * C::B_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                  // K-major: the next 16 K elements are 32 bytes further along the
                  // swizzled 128-byte row.  MN-major: 16 more K rows, 2 KB further,
                  // with the 64-wide MN chunks 8 KB apart.
                  const uint64_t ad = A_MN ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                           : smem_desc_sw128(sa + k * 32, 16, 1024);
                  const uint64_t bd = B_MN ? smem_desc_sw128(sb + k * 2048, B_LBO, 1024)
                                           : smem_desc_sw128(sb + k * 32, 16, 1024);
                  const uint32_t accum = (kb | j | k) != 0 ? 1u : 0u;
                  if constexpr (PAIR)
                    umma_bf16_pair(d_tmem, ad, bd, IDESC, accum);
                  else
                    umma_bf16(d_tmem, ad, bd, IDESC, accum);
                }
              }
              if constexpr (PAIR)
                umma_commit_pair(smem_addr(&ctl->empty[stage]), 0x3);
              else
                umma_commit(smem_addr(&ctl->empty[stage]));
              if (++stage == NST) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (!ok) break;
            if constexpr (PAIR)
              umma_commit_pair(smem_addr(&ctl->tfull[acc]), 0x3);
            else
              umma_commit(smem_addr(&ctl->tfull[acc]));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
          }
        };
        if (KS == 1 && L.prob[q].a_mn != 0)
          issue(std::true_type{});
        else
          issue(std::false_type{});
      }
      if (!ok) {
        if constexpr (PAIR) {
          umma_commit_pair(smem_addr(&ctl->drain), 0x1);
        } else {
          umma_commit(smem_addr(&ctl->drain));
        }
        wait_drain(smem_addr(&ctl->drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Decisions that all four epilogue warps must take together (the next
    // unit, whether an accumulator is ready) are made by one issuer thread
    // and broadcast through shared memory between named barriers, so the
    // warps can never part ways at a barrier.
    const int qw = warp & 3;            // TMEM lane quarter this warp may read
    const int lrow = qw * 32 + lane;    // accumulator row of this thread
    const bool issuer = lrow == 0;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t stg0 = smem_base + STAGES * STAGE_BYTES;
    uint32_t acc = 0, acc_phase = 0;
    uint32_t nstore = 0;   // staged TMA stores issued so far (buffer parity)
    const uint32_t tempty_leader =
        PAIR ? map_to_cta(smem_addr(&ctl->tempty[0]), 0) : smem_addr(&ctl->tempty[0]);
    volatile int* epi_u = &ctl->epi_u;
    volatile int* epi_ok = &ctl->epi_ok;

    for (int i = 0;; ++i) {
      const int slot = i & (SCHED_DEPTH - 1);
      const uint32_t spar = (i / SCHED_DEPTH) & 1;
      if (issuer) {
        int uu = 0;
        const bool got = sched_take(slot, spar, uu);
        if (got) sched_release(slot);
        *epi_u = got ? uu : INT_MIN;
      }
      named_bar_sync(1, 128);
      const int u = *epi_u;
      named_bar_sync(1, 128);
      if (u < 0) break;   // no more work, or the scheduler gave up
      int q;
      const int lu = split_unit(sc0, u, q);
      const Sched s = q ? sc1 : sc0;
      const GemmArgs& p = L.prob[q].p;
      const CUtensorMap* map_out = &L.map_out[q];
      int m, split, nb, ne;
      s.unit(lu, m, split, nb, ne);
      const int row_t = m * C::UNIT_M + static_cast<int>(rank) * BM;   // first row of this CTA's tile
      const int row = row_t + lrow;

      if (s.k_blocks == 0) {
        if constexpr (EPI == EPI_STORE_F32) {
          if (p.zero_if_empty && !p.accumulate && row < s.M) {
            const int64_t orow = p.row_map ? p.row_map[p.row_base + row] : p.row_base + row;
            for (int n = nb; n < ne; ++n) {
              float* dst = p.out + orow * p.out_ld + n * BN;
              const int lim = min(BN, p.n_extent - n * BN);
              for (int j = 0; j < lim; ++j) dst[j] = 0.f;
            }
          }
        }
        continue;
      }

      // per-unit state
      float mrun = -INFINITY, ssum = 0.f, s1 = 0.f, zy = -INFINITY;   // EPI_FWD_STATS
      float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);                   // EPI_BWD_DZ
      int y = -1;
      bool row_ok = false;
      int64_t orow = 0;
      if constexpr (EPI == EPI_FWD_STATS || EPI == EPI_FWD_Z) {
        row_ok = row < s.M;
        if (row_ok) y = p.y_c[p.row_base + row];
      } else if constexpr (EPI == EPI_BWD_DZ) {
        row_ok = row < p.m_cap;
        if (row_ok) {
          cf = p.coef[p.row_base + row];
          y = p.y_c[p.row_base + row];
        }
      } else {
        row_ok = row < s.M;
        if (row_ok && p.out_mode == 0)
          orow = p.row_map ? p.row_map[p.row_base + row] : p.row_base + row;
      }

      bool ok = true;
      for (int n = nb; n < ne; ++n) {
        if (issuer)
          *epi_ok = wait_bounded<PAIR>(smem_addr(&ctl->tfull[acc]), acc_phase, abort, status) ? 1 : 0;
        named_bar_sync(1, 128);
        const int t_ok = *epi_ok;
        named_bar_sync(1, 128);
        if (!t_ok) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int col0 = n * BN;
        const uint32_t tcol = tmem_base + lane_off + acc * BN;
        const int yt = y - p.col_base - col0;
        // hand the accumulator back to the MMA warp once this warp has read it all
        auto release_acc = [&]() {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR)
              mbar_arrive_remote(tempty_leader + acc * sizeof(uint64_t));
            else
              mbar_arrive(smem_addr(&ctl->tempty[acc]));
          }
        };

        if constexpr (EPI == EPI_FWD_STATS) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load_32(tcol + c * 32, v);
            if (c == BN / 32 - 1) release_acc();
            const int cb = c * 32;
            const int lim = p.n_extent - col0 - cb;   // valid columns in this chunk
            float cmax = -INFINITY;
            if (lim >= 32) {
#pragma unroll
              for (int j = 0; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < lim) cmax = fmaxf(cmax, v[j]);
            }
            const float cm = cmax * p.scale;
            if (cm > mrun) {
              const float dm = mrun - cm;
              const float r = ex2_approx(dm);
              s1 = ssum > 0.f ? r * fmaf(dm, ssum, s1) : 0.f;
              ssum *= r;
              mrun = cm;
            }
            if (lim >= 32) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float d = fmaf(v[j], p.scale, -mrun);
                const float e = ex2_approx(d);
                ssum += e;
                s1 = fmaf(e, d, s1);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (j < lim) {
                  const float d = fmaf(v[j], p.scale, -mrun);
                  const float e = ex2_approx(d);
                  ssum += e;
                  s1 = fmaf(e, d, s1);
                }
              }
            }
            if (static_cast<unsigned>(yt - cb) < 32u) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == yt - cb) zy = v[j] * p.scale;
            }
          }
        } else if constexpr (EPI == EPI_FWD_Z) {
          // pass 1: the tile's maximum sets this tile's reference m' (>= every
          // logit in it), so the kept values u - m' are <= 0 and fp16 keeps
          // most precision where p is largest
          float tmax = -INFINITY;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load_32(tcol + c * 32, v);
            const int lim = p.n_extent - col0 - c * 32;
            if (lim >= 32) {
#pragma unroll
              for (int j = 0; j < 32; ++j) tmax = fmaxf(tmax, v[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < lim) tmax = fmaxf(tmax, v[j]);
            }
          }
          const float cm = tmax * p.scale;
          if (cm > mrun) {
            const float dm = mrun - cm;
            const float r = ex2_approx(dm);
            s1 = ssum > 0.f ? r * fmaf(dm, ssum, s1) : 0.f;
            ssum *= r;
            mrun = cm;
          }
          const float mref = mrun;
          // pass 2: statistics from the same exponentials, and the kept logits
#pragma unroll 1
          for (int cc = 0; cc < BN / 64; ++cc) {
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float v[32];
              tmem_load_32(tcol + cc * 64 + h * 32, v);
              if (cc == BN / 64 - 1 && h == 1) release_acc();
              const int cb = cc * 64 + h * 32;
              const int lim = p.n_extent - col0 - cb;
              float d[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) d[j] = fmaf(v[j], p.scale, -mref);
              if (lim >= 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float e = ex2_approx(d[j]);
                  ssum += e;
                  s1 = fmaf(e, d[j], s1);
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  if (j < lim) {
                    const float e = ex2_approx(d[j]);
                    ssum += e;
                    s1 = fmaf(e, d[j], s1);
                  }
                }
              }
              if (static_cast<unsigned>(yt - cb) < 32u) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j == yt - cb) zy = v[j] * p.scale;
              }
#pragma unroll
              for (int k = 0; k < 16; ++k) pk[h * 16 + k] = pack_f16x2(d[2 * k], d[2 * k + 1]);
            }
            stage_out(pk, stg0, nstore++, lrow, issuer, map_out, 1, col0 + cc * 64, row_t, status);
          }
          if (row < p.m_cap) p.m_tile[static_cast<int64_t>(row) * p.m_tile_ld + n] = mref;
        } else if constexpr (EPI == EPI_BWD_DZ) {
          // 64 columns per staged chunk: 128 bytes of bf16 per row
#pragma unroll 1
          for (int cc = 0; cc < BN / 64; ++cc) {
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float v[32];
              tmem_load_32(tcol + cc * 64 + h * 32, v);
              if (cc == BN / 64 - 1 && h == 1) release_acc();
              const int cb = cc * 64 + h * 32;
              float g[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float d = fmaf(v[j], p.scale, -cf.x);
                const float pr = ex2_approx(d);
                g[j] = -pr * fmaf(cf.y, d, cf.z);
              }
              if (static_cast<unsigned>(yt - cb) < 32u) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j == yt - cb) g[j] += cf.w;
              }
#pragma unroll
              for (int k = 0; k < 16; ++k) pk[h * 16 + k] = pack_bf16x2(g[2 * k], g[2 * k + 1]);
            }
            if (p.out_mode == 1) {
              stage_out(pk, stg0, nstore++, lrow, issuer, map_out, 1, col0 + cc * 64, row_t, status);
            } else if (row_ok) {
              const int lim = p.n_extent - col0 - cc * 64;
              uint16_t* dst = p.dz_out + static_cast<int64_t>(row) * p.dz_ld + col0 + cc * 64;
              if (lim >= 64) {
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                  if (j < lim)
                    dst[j] = static_cast<uint16_t>((j & 1) ? (pk[j >> 1] >> 16)
                                                           : (pk[j >> 1] & 0xFFFFu));
              }
            }
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load_32(tcol + c * 32, v);
            if (c == BN / 32 - 1) release_acc();
            const int cb = c * 32;
            if (p.out_mode != 0) {
              uint32_t w[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(v[j]);
              stage_out(w, stg0, nstore++, lrow, issuer, map_out, p.out_mode, col0 + cb, row_t,
                        status);
            } else if (row_ok) {
              const int lim = p.n_extent - col0 - cb;
              float* dst = p.out + orow * p.out_ld + col0 + cb;
              if (lim >= 32) {
                float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                  if (p.accumulate) {
                    const float4 old = d4[k];
                    o.x += old.x;
                    o.y += old.y;
                    o.z += old.z;
                    o.w += old.w;
                  }
                  d4[k] = o;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j < lim) dst[j] = p.accumulate ? dst[j] + v[j] : v[j];
              }
            }
          }
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) break;
      if constexpr (EPI == EPI_FWD_STATS || EPI == EPI_FWD_Z) {
        if (row_ok)
          p.partials[static_cast<int64_t>(split) * p.part_ld + p.row_base + row] =
              make_float4(mrun, ssum, s1, zy);
      }
    }
    if (issuer) bulk_wait_all();   // staged stores done before the staging memory goes away
  }

  tc_fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // no remote arrive may target an exited CTA
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Co-resident clusters of two CTAs of `kern` with `smem` bytes of dynamic
// shared memory each (0 if the query fails).
inline int cluster_pairs(const void* kern, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

// Once per kernel and device: allow its dynamic shared memory and count its
// co-resident pairs.  `ready` holds 0 (not yet done) or 1 + that count, so
// later launches make no configuration calls (which also keeps them legal
// inside a stream capture).
inline cudaError_t prepare_kernel(std::atomic<int>* ready, const void* kern, size_t smem,
                                  bool pair, int* pairs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int r = ready[dev].load(std::memory_order_relaxed);
  if (r == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int n = pair ? cluster_pairs(kern, smem) : 0;
    if (pair && n <= 0) return cudaErrorInvalidConfiguration;
    r = 1 + n;
    ready[dev].store(r, std::memory_order_relaxed);
  }
  *pairs = r - 1;
  return cudaSuccess;
}

// grid = CTAs wanted (ignored beyond the co-resident limit).  For pairs the
// grid is rounded to whole clusters.
template <int EPI, bool B_MN, bool PAIR>
cudaError_t launch_tc_gemm(const LaunchArgs& a, int grid, cudaStream_t s) {
  auto kern = tc_gemm_kernel<EPI, B_MN, PAIR>;
  static std::atomic<int> ready[64];   // per device, for this kernel
  int pairs_max = 0;
  const cudaError_t e = prepare_kernel(ready, reinterpret_cast<const void*>(kern),
                                       GEMM_SMEM_BYTES, PAIR, &pairs_max);
  if (e != cudaSuccess) return e;
  int ctas = grid < 1 ? 1 : grid;
  if constexpr (PAIR) {
    int pairs = (ctas + 1) / 2;
    if (pairs > pairs_max) pairs = pairs_max;
    ctas = 2 * pairs;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if constexpr (PAIR) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace lmh
