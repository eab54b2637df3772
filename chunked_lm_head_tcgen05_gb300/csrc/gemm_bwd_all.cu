// The whole backward of the chunked LM head in one persistent launch
// (sm_103a, CTA pairs, tcgen05.mma.cta_group::2).
//
// The backward (the entropy / log-prob head pages, "backward" and "chunked
// loss" sections) works block by block: for T_b scored tokens and V_b
// vocabulary rows it recomputes the logits and turns them into the cotangent
// dz (bf16 scratch), then dh (+)= dz . W_blk and dW_blk (+)= dz^T . h_blk.
// The per-block path runs that as two launches per block.  Here the tiles of
// every block form one sequence of work units, fetched from a device counter
// by persistent CTA pairs, and the order that the launch boundaries gave is
// kept by per-tile completion counters in the workspace:
//   * a dh tile of rows m of block b loads each 256-column K step of dz
//     once every dz tile of that column is stored (dz tiles run column by
//     column, so a dh tile follows the dz wavefront instead of waiting for
//     whole rows);
//   * a dW tile of vocabulary rows j loads dz column tile j once every dz
//     tile of that column is stored;
//   * a dz tile (m, n) overwrites the scratch only after the previous block's
//     readers of rows m (its dh tiles) and of column tile n (its dW tiles)
//     are done;
//   * a dh tile that adds into d_hidden waits for the previous vocabulary
//     block's tile of the same rows, and a dW tile that adds into d_weight
//     for the previous token block's tile of the same rows of W.
// Each tile is computed as in the per-block path (same operands, tile shape,
// K order and epilogue arithmetic) and the additions into d_hidden and
// d_weight happen in the same order, so both paths give the same bits.
//
// Units are numbered token block by token block; within a block: its dz
// tiles (column major: the tiles running together share one W tile in L2),
// its dh tiles (row major), its dW tiles (vocabulary-tile major).  Every unit
// depends only on units with smaller numbers and units are handed out in
// increasing order, so the smallest unfinished unit can always run: the
// schedule cannot deadlock.  Every wait is still bounded: a CTA that gives up
// records STATUS_DEVICE_TIMEOUT and raises the state's abort word, which all
// other CTAs poll, so the whole grid winds down.
#include "tc_gemm.cuh"

#include <type_traits>

namespace lmh {
namespace {

enum : int { U_DZ = 0, U_DH = 1, U_DW = 2 };
constexpr int PAIR_M = 2 * BM;   // rows of a pair's tile

struct Blk {
  int tb, vb, t0, v0, vact, mcap, rows, mt, nt;
};

__device__ __forceinline__ Blk block_of(const BwdAllArgs& a, int tb, int vb, int scored) {
  Blk k;
  k.tb = tb;
  k.vb = vb;
  k.t0 = tb * a.T_b;
  k.v0 = vb * a.V_b;
  k.vact = min(a.V_b, a.V - k.v0);
  k.mcap = min(a.T_b, a.T_alloc - k.t0);
  k.rows = max(0, min(scored - k.t0, k.mcap));
  k.mt = (k.rows + PAIR_M - 1) / PAIR_M;
  k.nt = (k.vact + BN - 1) / BN;
  return k;
}

// A dz unit covers DZW adjacent 256-column tiles of one row tile (the last
// of a block's columns may be alone): each unit pays a fetch from the unit
// counter, a scheduler hand-off and a decode, and dz tiles are short (K = H).
constexpr int DZW = 2;

__device__ __forceinline__ int dz_units(int mt, int nt) { return mt * ((nt + DZW - 1) / DZW); }

// Work units of one full-width block whose token block has `mt` row tiles.
__device__ __forceinline__ int units_full(const BwdAllArgs& a, int mt, int ht) {
  return dz_units(mt, a.NT) + mt * ht + a.NT * ht;
}

struct Unit {
  int kind, b, m, n, ntiles, kblocks;   // dz units: tiles n .. n + ntiles - 1; others: 1 tile
  Blk k;
};

// Unit number -> block, kind and tile.  `tb_prefix` holds the first unit of
// each token block; within a token block all vocabulary blocks but the last
// are full width, so their units follow one stride.
__device__ __forceinline__ Unit decode(const BwdAllArgs& a, const int* tb_prefix, int scored,
                                       int ht, int u) {
  int lo = 0, hi = a.n_tb - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb_prefix[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  int r = u - tb_prefix[lo];
  const Blk k0 = block_of(a, lo, 0, scored);
  const int stride = units_full(a, k0.mt, ht);
  const int vb = min(r / stride, a.n_vb - 1);
  r -= vb * stride;
  Unit x;
  x.k = block_of(a, lo, vb, scored);
  x.b = lo * a.n_vb + vb;
  const int n_dz = dz_units(x.k.mt, x.k.nt), n_dh = x.k.mt * ht;
  x.ntiles = 1;
  if (r < n_dz) {
    // column pairs, row tiles fastest: a block's dz columns complete in order
    x.kind = U_DZ;
    const int np = r / x.k.mt;
    x.m = r - np * x.k.mt;
    x.n = np * DZW;
    x.ntiles = min(DZW, x.k.nt - x.n);
    x.kblocks = a.H / BK;
  } else if (r - n_dz < n_dh) {
    r -= n_dz;
    x.kind = U_DH;
    x.m = r / ht;
    x.n = r - x.m * ht;
    x.kblocks = (x.k.vact + BK - 1) / BK;
  } else {
    r -= n_dz + n_dh;
    x.kind = U_DW;
    x.m = r / ht;
    x.n = r - x.m * ht;
    x.kblocks = (x.k.rows + BK - 1) / BK;
  }
  return x;
}

// Completion counters of block b (each CTA of a pair adds 1 per tile): all
// dz tiles, dz tiles per column, dh tiles per row tile, dW tiles per
// vocabulary tile.
struct Flags {
  int* base;
  int MT, NT;
  __device__ __forceinline__ int* blk(int b) const {
    return base + static_cast<int64_t>(b) * (1 + MT + 2 * NT);
  }
  __device__ __forceinline__ int* dz_all(int b) const { return blk(b); }
  __device__ __forceinline__ int* dz_col(int b, int n) const { return blk(b) + 1 + n; }
  __device__ __forceinline__ int* dh_row(int b, int m) const { return blk(b) + 1 + NT + m; }
  __device__ __forceinline__ int* dw_col(int b, int n) const { return blk(b) + 1 + NT + MT + n; }
};


// True when this CTA must stop: it gave up earlier, another CTA did, or this
// wait has run past its limit (then it records the timeout for everyone).
__device__ __forceinline__ bool give_up(volatile int* abort, DeviceState* st, uint64_t t0) {
  if (*abort) return true;
  if (*reinterpret_cast<volatile int*>(&st->abort_all)) {
    *abort = 1;
    return true;
  }
  if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
    *abort = 1;
    atomicExch(&st->abort_all, 1);
    atomicCAS(&st->status, 0, STATUS_DEVICE_TIMEOUT);
    return true;
  }
  return false;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         DeviceState* st) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (give_up(abort, st, t0)) return false;
  }
}

// Wait until *f >= target (acquire at GPU scope).
__device__ __forceinline__ bool wait_flag(const int* f, int target, volatile int* abort,
                                          DeviceState* st) {
  if (ld_acquire_gpu(f) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
      __nanosleep(128);
      if (ld_acquire_gpu(f) >= target) return true;
    }
    if (give_up(abort, st, t0)) return false;
  }
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
    bwd_all_kernel(const __grid_constant__ BwdAllArgs A) {
  using C = TileCfg<true>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + STAGES * STAGE_BYTES + STAGING_BYTES);
  int* tb_prefix = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + STAGING_BYTES + 256);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  DeviceState* const st = A.st;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;
  const int r128 = static_cast<int>(rank) * BM;
  const Flags F{A.flags, A.MT, A.NT};
  const int ht = (A.H + BN - 1) / BN;

  if (threadIdx.x == 0) pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(smem_addr(&ctl->full[s]), 1);
      mbar_init(smem_addr(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&ctl->tfull[b]), 1);
      mbar_init(smem_addr(&ctl->tempty[b]), EPI_WARPS * 2);
    }
    for (int s = 0; s < SCHED_DEPTH; ++s) {
      mbar_init(smem_addr(&ctl->sfull[s]), 1);
      mbar_init(smem_addr(&ctl->sempty[s]), 4);
    }
    mbar_init(smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();   // the peer's barriers exist before any remote arrive
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort = &ctl->abort;
  const uint32_t smem_base = smem_addr(smem);

  // Inputs written by earlier kernels (scored count, counters, coefficients)
  // are read from here on.
  pdl_wait_prerequisites();
  const int scored = st->rows;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int tb = 0; tb < A.n_tb; ++tb) {
      tb_prefix[tb] = acc;
      const Blk k = block_of(A, tb, 0, scored);
      acc += (A.n_vb - 1) * units_full(A, k.mt, ht);
      const Blk kl = block_of(A, tb, A.n_vb - 1, scored);
      acc += dz_units(kl.mt, kl.nt) + kl.mt * ht + kl.nt * ht;
    }
    tb_prefix[A.n_tb] = acc;
  }
  __syncthreads();
  // This launch's units: all of them, or one window (see BwdAllArgs::window).
  int unit_begin = 0, unit_end = tb_prefix[A.n_tb];
  if (A.window >= 0) {
    const int n_blocks = A.n_tb * A.n_vb;
    auto first_dh = [&](int b) {   // number of the first dh unit of block b
      const int tb = b / A.n_vb, vb = b - tb * A.n_vb;
      const Blk k0 = block_of(A, tb, 0, scored);
      const Blk k = block_of(A, tb, vb, scored);
      return tb_prefix[tb] + vb * units_full(A, k0.mt, ht) + dz_units(k.mt, k.nt);
    };
    if (A.window > 0) unit_begin = first_dh(A.window - 1);
    if (A.window < n_blocks) unit_end = first_dh(A.window);
  }

  auto sched_take = [&](int slot, uint32_t spar, int& u) -> bool {
    if (!wait_bar(smem_addr(&ctl->sfull[slot]), spar, abort, st)) return false;
    u = ctl->sched[slot];
    return true;
  };
  auto sched_release = [&](int slot) {
    if (!leader)
      mbar_arrive_remote(map_to_cta(smem_addr(&ctl->sempty[slot]), 0));
    else
      mbar_arrive(smem_addr(&ctl->sempty[slot]));
  };

  if (warp == 0) {
    // ------------------------------------------------------ scheduler + producer
    if (lane == 0) {
      tma_prefetch_map(&A.h_k);
      tma_prefetch_map(&A.w_k);
      tma_prefetch_map(&A.dz_k);
      tma_prefetch_map(&A.w_mn);
      tma_prefetch_map(&A.dz_mn);
      tma_prefetch_map(&A.h_mn);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int ahead = -1;   // unit index fetched ahead, -1 = none
      for (int i = 0; ok; ++i) {
        const int slot = i & (SCHED_DEPTH - 1);
        const uint32_t spar = (i / SCHED_DEPTH) & 1;
        int u;
        if (leader) {
          if (!wait_bar(smem_addr(&ctl->sempty[slot]), spar ^ 1, abort, st)) {
            ok = false;
            break;
          }
          u = unit_begin + (ahead >= 0 ? ahead : atomicAdd(A.unit_counter, 1));
          ahead = -1;
          if (u >= unit_end) u = -1;
          ctl->sched[slot] = u;
          st_shared_remote(map_to_cta(smem_addr(&ctl->sched[slot]), 1), u);
          mbar_arrive_remote(map_to_cta(smem_addr(&ctl->sfull[slot]), 1));
          mbar_arrive(smem_addr(&ctl->sfull[slot]));
        } else {
          if (!sched_take(slot, spar, u)) {
            ok = false;
            break;
          }
          sched_release(slot);
        }
        if (u < 0) break;
        const Unit x = decode(A, tb_prefix, scored, ht, u);
        if (x.kblocks == 0) continue;
        // The dz tiles this unit reads must be stored; each acquire is then
        // ordered before this thread's async-proxy loads.  A dW tile needs
        // one dz column.  A dh tile needs them all, and usually finds every
        // dz tile of its block stored; otherwise it checks each column as
        // its K loop reaches it.
        const int dz_target = 2 * x.k.mt * x.k.nt;
        bool dz_ready = x.kind != U_DH;
        if (!dz_ready && ld_acquire_gpu(F.dz_all(x.b)) >= dz_target) {
          fence_async_global();
          dz_ready = true;
        }
        if (x.kind == U_DW) {
          if (!wait_flag(F.dz_col(x.b, x.m), 2 * x.k.mt, abort, st)) {
            ok = false;
            break;
          }
          fence_async_global();
        }
        const int mrow = x.m * PAIR_M + r128;   // this CTA's first M row (or M column)
        const int ncol = x.n * BN + r128;       // this CTA's half of the N tile
        // The K loop is compiled once per tile kind: a kind test inside it costs
        // this TMA-issue-bound thread about a tenth of the kernel's speed.
        auto produce = [&](auto kind_tag) {
          constexpr int KIND = decltype(kind_tag)::value;
          const int ntl = KIND == U_DZ ? x.ntiles : 1;
          for (int t = 0; ok && t < ntl; ++t) {
            const int ncol_t = ncol + t * BN;
            const bool last_tile = t == ntl - 1;
            for (int kb = 0; kb < x.kblocks; ++kb) {
              if constexpr (KIND == U_DH) {
                if (!dz_ready && kb % (BN / BK) == 0) {
                  if (ld_acquire_gpu(F.dz_all(x.b)) >= dz_target) {
                    dz_ready = true;
                  } else if (!wait_flag(F.dz_col(x.b, kb / (BN / BK)), 2 * x.k.mt, abort, st)) {
                    ok = false;
                    break;
                  }
                  fence_async_global();
                }
              }
              if (leader && ahead < 0 && last_tile && kb == max(0, x.kblocks - FETCH_AHEAD_KB))
                ahead = atomicAdd(A.unit_counter, 1);
              if (!wait_bar(smem_addr(&ctl->empty[stage]), phase ^ 1, abort, st)) {
                ok = false;
                break;
              }
              const uint32_t fb_local = smem_addr(&ctl->full[stage]);
              if (leader) mbar_arrive_expect_tx(fb_local, C::STAGE * 2);
              const uint32_t fb = map_to_cta(fb_local, 0);
              const uint32_t sa = smem_base + stage * C::STAGE;
              const uint32_t sb = sa + A_TILE_BYTES;
              const int k0 = kb * BK;
              if constexpr (KIND == U_DZ) {
                tma_load_2d_pair(sa, &A.h_k, fb, k0, x.k.t0 + mrow);
                tma_load_2d_pair(sb, &A.w_k, fb, k0, x.k.v0 + ncol_t);
              } else if constexpr (KIND == U_DH) {
                tma_load_2d_pair(sa, &A.dz_k, fb, k0, mrow);
                tma_load_3d_pair(sb, &A.w_mn, fb, 0, x.k.v0 + k0, ncol_t / 64);
              } else {
                tma_load_3d_pair(sa, &A.dz_mn, fb, 0, k0, mrow / 64);
                tma_load_3d_pair(sb, &A.h_mn, fb, 0, x.k.t0 + k0, ncol_t / 64);
              }
              if (++stage == C::NSTAGE) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        };
        if (x.kind == U_DZ)
          produce(std::integral_constant<int, U_DZ>{});
        else if (x.kind == U_DH)
          produce(std::integral_constant<int, U_DH>{});
        else
          produce(std::integral_constant<int, U_DW>{});
      }
      if (!ok) pause_ns(100000);   // let copies already issued land before exit
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
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
        const Unit x = decode(A, tb_prefix, scored, ht, u);
        if (x.kblocks == 0) continue;
        uint32_t d_tmem = 0;
        // one K loop per tile kind, operand layouts and descriptor fixed at compile time
        auto issue = [&](auto kind_tag) {
          constexpr int KIND = decltype(kind_tag)::value;
          constexpr bool AMN = KIND == U_DW, BMN = KIND != U_DZ;
          constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, BN, AMN, BMN);
          for (int kb = 0; kb < x.kblocks; ++kb) {
            if (!wait_bar(smem_addr(&ctl->full[stage]), phase, abort, st)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t sa = smem_base + stage * C::STAGE;
            const uint32_t sb = sa + A_TILE_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // K-major: 16 more K elements are 32 bytes along the swizzled row;
              // MN-major: 16 more K rows are 2 KB further, 64-wide MN chunks 8 KB apart.
              const uint64_t ad = AMN ? smem_desc_sw128(sa + k * 2048, 8192, 1024)
                                      : smem_desc_sw128(sa + k * 32, 16, 1024);
              const uint64_t bd = BMN ? smem_desc_sw128(sb + k * 2048, 8192, 1024)
                                      : smem_desc_sw128(sb + k * 32, 16, 1024);
              umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
            }
            umma_commit_pair(smem_addr(&ctl->empty[stage]), 0x3);
            if (++stage == C::NSTAGE) {
              stage = 0;
              phase ^= 1;
            }
          }
        };
        // each tile of the unit into the next free accumulator
        for (int t = 0; t < x.ntiles; ++t) {
          if (!wait_bar(smem_addr(&ctl->tempty[acc]), acc_phase ^ 1, abort, st)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          d_tmem = tmem_base + acc * BN;
          if (x.kind == U_DZ)
            issue(std::integral_constant<int, U_DZ>{});
          else if (x.kind == U_DH)
            issue(std::integral_constant<int, U_DH>{});
          else
            issue(std::integral_constant<int, U_DW>{});
          if (!ok) break;
          umma_commit_pair(smem_addr(&ctl->tfull[acc]), 0x3);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!ok) break;
      }
      // every MMA issued by this thread has completed before TMEM is freed
      umma_commit_pair(smem_addr(&ctl->drain), 0x1);
      wait_drain(smem_addr(&ctl->drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Decisions the four epilogue warps take together (next unit, accumulator
    // ready, dependencies met) are made by one issuer thread and broadcast
    // through shared memory between named barriers.
    const int qw = warp & 3;
    const int lrow = qw * 32 + lane;
    const bool issuer = lrow == 0;
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t stg0 = smem_base + STAGES * STAGE_BYTES;
    uint32_t acc = 0, acc_phase = 0;
    uint32_t nstore = 0;
    const uint32_t tempty_leader = map_to_cta(smem_addr(&ctl->tempty[0]), 0);
    volatile int* epi_u = &ctl->epi_u;
    volatile int* epi_ok = &ctl->epi_ok;

    auto broadcast = [&](int v) -> int {
      if (issuer) *epi_ok = v;
      named_bar_sync(1, 128);
      const int r = *epi_ok;
      named_bar_sync(1, 128);
      return r;
    };
    // Dependencies of this tile's stores (the issuer waits, then orders its
    // later async-proxy stores after the acquire).
    auto wait_deps = [&](const int* f0, int t0v, const int* f1, int t1v) -> bool {
      int okv = 1;
      if (issuer) {
        bool ok = true;
        if (f0) ok = wait_flag(f0, t0v, abort, st);
        if (ok && f1) ok = wait_flag(f1, t1v, abort, st);
        if (ok) fence_async_global();
        okv = ok ? 1 : 0;
      }
      return broadcast(okv) != 0;
    };
    // Publish this tile: its stores are complete and visible before the counter moves.
    auto signal = [&](int* f0, int* f1, bool staged) {
      if (staged) {
        if (issuer) bulk_wait_all();
      } else {
        __threadfence();
      }
      named_bar_sync(1, 128);
      if (issuer) {
        fence_async_global();
        red_release_gpu_add(f0, 1);
        if (f1) red_release_gpu_add(f1, 1);
      }
    };

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
      if (u < 0) break;
      const Unit x = decode(A, tb_prefix, scored, ht, u);
      const int rloc = x.m * PAIR_M + r128 + lrow;   // this thread's row within the block's tile grid

      if (x.kblocks == 0) {
        // a dW tile of a token block without scored tokens: zeros unless it adds
        const int col0 = x.n * BN;
        if (x.k.tb == 0 && !A.accumulate_dweight && rloc < x.k.vact) {
          float* dst = A.d_weight + static_cast<int64_t>(x.k.v0 + rloc) * A.H + col0;
          const int lim = min(BN, A.H - col0);
          for (int j = 0; j < lim; ++j) dst[j] = 0.f;
        }
        signal(F.dw_col(x.b, x.m), nullptr, false);
        continue;
      }

      // the unit's tiles in order (dz units may hold two), each from the next
      // accumulator the MMA warp filled
      bool fail = false;
      for (int t = 0; t < x.ntiles; ++t) {
        const int xn = x.n + t;
        const int col0 = xn * BN;
        // dependencies of this tile's stores
        bool dep_ok = true;
        if (x.kind == U_DZ) {
          if (x.b > 0) {
            const Blk kp = block_of(A, (x.b - 1) / A.n_vb, (x.b - 1) % A.n_vb, scored);
            const int bp = xn < kp.nt ? x.b - 1 : x.b - 2;
            dep_ok = wait_deps(F.dh_row(x.b - 1, x.m), 2 * ht, bp >= 0 ? F.dw_col(bp, xn) : nullptr,
                               2 * ht);
          }
        } else if (x.kind == U_DH) {
          if (x.k.vb > 0) dep_ok = wait_deps(F.dh_row(x.b - 1, x.m), 2 * ht, nullptr, 0);
        } else {
          if (x.k.tb > 0) dep_ok = wait_deps(F.dw_col(x.b - A.n_vb, x.m), 2 * ht, nullptr, 0);
        }
        if (!dep_ok) {
          fail = true;
          break;
        }

        int t_ok = 0;
        if (issuer) t_ok = wait_bar(smem_addr(&ctl->tfull[acc]), acc_phase, abort, st) ? 1 : 0;
        if (!broadcast(t_ok)) {
          fail = true;
          break;
        }
        tc_fence_after_sync();
        const uint32_t tcol = tmem_base + lane_off + acc * BN;
        auto release_acc = [&]() {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(tempty_leader + acc * sizeof(uint64_t));
        };

        if (x.kind == U_DZ) {
          const bool row_ok = rloc < x.k.mcap;
          float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
          int y = -1;
          if (row_ok) {
            cf = A.coef[x.k.t0 + rloc];
            y = A.y_c[x.k.t0 + rloc];
          }
          const int yt = y - x.k.v0 - col0;
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
                const float d = fmaf(v[j], A.scale, -cf.x);
                const float pr = ex2_approx(d);
                g[j] = -pr * fmaf(cf.y, d, cf.z);
              }
              if (static_cast<unsigned>(yt - cb) < 32u) {
  #pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j == yt - cb) g[j] += cf.w;
              }
              // columns past the vocabulary block hold zeros: the dh and dW
              // tiles read whole 64-wide K steps of the scratch
              const int lim = x.k.vact - col0 - cb;
              if (lim < 32) {
  #pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (j >= lim) g[j] = 0.f;
              }
  #pragma unroll
              for (int k = 0; k < 16; ++k) pk[h * 16 + k] = pack_bf16x2(g[2 * k], g[2 * k + 1]);
            }
            stage_out(pk, stg0, nstore++, lrow, issuer, &A.dz_k, 1, col0 + cc * 64,
                      x.m * PAIR_M + r128, &st->status);
          }
          signal(F.dz_col(x.b, xn), F.dz_all(x.b), true);
        } else if (x.kind == U_DH) {
          const bool scatter = A.row_map != nullptr;
          const bool add = x.k.vb > 0;
          const bool row_ok = rloc < x.k.rows;
          const int64_t orow = (scatter && row_ok) ? A.row_map[x.k.t0 + rloc] : 0;
  #pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load_32(tcol + c * 32, v);
            if (c == BN / 32 - 1) release_acc();
            const int cb = c * 32;
            if (!scatter) {
              uint32_t w[32];
  #pragma unroll
              for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(v[j]);
              stage_out(w, stg0, nstore++, lrow, issuer, &A.dh_out, add ? 2 : 1, col0 + cb,
                        x.k.t0 + x.m * PAIR_M + r128, &st->status);
            } else if (row_ok) {
              const int lim = A.H - col0 - cb;
              float* dst = A.d_hidden + orow * A.H + col0 + cb;
              if (lim >= 32) {
                float4* d4 = reinterpret_cast<float4*>(dst);
  #pragma unroll
                for (int k = 0; k < 8; ++k) {
                  float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                  if (add) {
                    // from L2: the previous value was written by another SM
                    const float4 old = __ldcg(d4 + k);
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
                  if (j < lim) dst[j] = add ? __ldcg(dst + j) + v[j] : v[j];
              }
            }
          }
          signal(F.dh_row(x.b, x.m), nullptr, !scatter);
        } else {
          const int mode = (x.k.tb > 0 || A.accumulate_dweight) ? 2 : 1;
  #pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tmem_load_32(tcol + c * 32, v);
            if (c == BN / 32 - 1) release_acc();
            uint32_t w[32];
  #pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(v[j]);
            stage_out(w, stg0, nstore++, lrow, issuer, &A.dw_out, mode, col0 + c * 32,
                      x.k.v0 + x.m * PAIR_M + r128, &st->status);
          }
          signal(F.dw_col(x.b, x.m), nullptr, true);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (fail) break;
    }
    if (issuer) bulk_wait_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();   // no remote arrive may target an exited CTA
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_gemm_bwd_all(const BwdAllArgs& a, int grid, cudaStream_t s) {
  if (a.n_tb < 1 || a.n_tb > BWD_ALL_MAX_TOKEN_BLOCKS || a.n_vb < 1 || a.T_b % (2 * BM) != 0 ||
      a.V_b % BN != 0 || a.H % BK != 0)
    return cudaErrorInvalidValue;
  static std::atomic<int> ready[64];   // per device
  int pairs_max = 0;
  const cudaError_t e = prepare_kernel(ready, reinterpret_cast<const void*>(bwd_all_kernel),
                                       BWD_ALL_SMEM_BYTES, true, &pairs_max);
  if (e != cudaSuccess) return e;
  int pairs = (grid + 1) / 2;
  if (pairs < 1) pairs = 1;
  if (pairs > pairs_max) pairs = pairs_max;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = BWD_ALL_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, bwd_all_kernel, a);
}

}  // namespace lmh
