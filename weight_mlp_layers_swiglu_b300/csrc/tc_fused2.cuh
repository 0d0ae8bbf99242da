// The fused chunk-state + apply kernel of tc_fused.cuh on CTA pairs (clusters of two CTAs).
//
// zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.2 Steps 1-3, in one
// cooperative persistent launch: every pair first runs its state units (as tc_state2.cuh:
// 256 x 256 units, tcgen05.mma.cta_group::2, each CTA loading its own halves of V and Z), then
// claims apply tiles from a global queue in chunk order.
//
// The apply tiles are 256 rows x 512 columns of O when there are enough of them (p.a_halves = 2):
// each CTA's whole tensor memory (512 columns) holds one accumulator, and every k-block issues
// two N = 256 MMAs that share the A tile (the chunk's Z rows).  Against 256 x 256 tiles this
// loads a quarter fewer operand bytes per FLOP, which is what the apply's MMAs wait for (its
// W_eff rows come from DRAM); the epilogue of a tile is no longer hidden behind the next tile's
// MMAs, but a tile runs 2 x d_ff/64 k-blocks and its epilogue a few microseconds.  Calls with
// few tiles (a short sequence) take 256 x 256 tiles (p.a_halves = 1) with two accumulators in
// turn, so that twice as many pairs share the work, and continue on the state phase's stage
// ring.  Wide tiles reuse the ring's memory as 4 stages of 48 KB (A 16 KB, B 2 x 16 KB) with
// barriers of their own; a CTA's producer starts them once the MMAs have consumed every state
// stage it issued.
//
// Hand-offs, as in tc_fused.cuh: each epilogue warp of both CTAs publishes a W_eff slice on the
// slice's counter once its TMA stores of the slice have completed (ready_target = pair units
// per sequence x 8 warps); both CTAs' producers wait for the counter before loading their
// halves of the slice.  The even CTA claims each apply tile and hands it to the odd CTA
// through the odd CTA's shared memory (a remote store, then a remote arrive with release
// semantics on the odd CTA's tile_full); the slot is reused once all ten readers of both CTAs
// have arrived on the even CTA's tile_empty.  All clusters are co-resident (cooperative
// launch), so the waits on other clusters' counters always end; every wait is bounded.
#pragma once

#include "tc_fused.cuh"
#include "tc_gemm2.cuh"
#include "tc_state2.cuh"

namespace ipttt {
namespace fused2 {

constexpr int STAGES = 6;
constexpr int STAGE_BYTES = 32 * 1024;
static_assert(state2::STAGE_BYTES == STAGE_BYTES && gemm2::STAGE_BYTES == STAGE_BYTES, "one ring for both phases");
static_assert(state2::A_BYTES == gemm2::A_BYTES, "A tiles share the stage layout");
constexpr int A_BYTES = gemm2::A_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int TILE_SLOTS = 4;
constexpr int APPLY_STAGES = 4;
constexpr int APPLY_B_HALF = gemm2::B_BYTES;                       // 128 rows x 64 k of one N-half
constexpr int APPLY_STAGE_BYTES = gemm2::A_BYTES + 2 * APPLY_B_HALF;  // 48 KB
static_assert(APPLY_STAGES * APPLY_STAGE_BYTES <= STAGES * STAGE_BYTES, "the apply ring fits the state ring");
static_assert(APPLY_STAGE_BYTES % 1024 == 0, "apply stages keep the 1024-byte alignment");
constexpr int TILE_READERS = 10;  // MMA + 4 epilogue warps (even CTA), producer + 4 epilogue warps (odd)
constexpr int BAR_BYTES = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert((2 * STAGES + 2 * APPLY_STAGES + 8 + 2 * TILE_SLOTS + 1) * 8 + TILE_SLOTS * 4 + 8 <= BAR_BYTES,
              "barrier block");

using fused::Params;  // s: pair units (m_units counts 256-row blocks); a: 256 x 512 apply tiles

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// HALVES (= Params::a_halves): 256-column halves per apply tile, a template parameter so that
// each tile width compiles to its own fixed loops.
template <int HALVES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    tc_state_apply2_kernel(const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_z,
                           const __grid_constant__ CUtensorMap map_weff_st,
                           const __grid_constant__ CUtensorMap map_wfin, const __grid_constant__ CUtensorMap map_za,
                           const __grid_constant__ CUtensorMap map_weff_ld, const __grid_constant__ CUtensorMap map_w0,
                           const __grid_constant__ CUtensorMap map_o, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                          // [STAGES]  even CTA
  uint64_t* empty = full + STAGES;                // [STAGES]  each CTA
  uint64_t* chunk_done = empty + STAGES;          // [2] state: MMA -> epilogues (both)
  uint64_t* snap_done = chunk_done + 2;           // [2] state: epilogues -> MMA (even)
  uint64_t* acc_full = snap_done + 2;             // [2] apply: MMA -> epilogues (both)
  uint64_t* acc_empty = acc_full + 2;             // [2] apply: epilogues -> MMA (even)
  uint64_t* a_full = acc_empty + 2;               // [APPLY_STAGES] apply ring, even CTA
  uint64_t* a_empty = a_full + APPLY_STAGES;      // [APPLY_STAGES] apply ring, each CTA
  uint64_t* tile_full = a_empty + APPLY_STAGES;   // [TILE_SLOTS] even producer -> readers (both)
  uint64_t* tile_empty = tile_full + TILE_SLOTS;  // [TILE_SLOTS] readers -> even producer
  uint64_t* drain = tile_empty + TILE_SLOTS;
  int* tile_q = reinterpret_cast<int*>(drain + 1);  // [TILE_SLOTS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_q + TILE_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const state::Params& S = p.s;
  const gemm::Params& A = p.a;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1;
  const int n_cl = gridDim.x >> 1;
  const int upairs = (S.units + 1) / 2;
  const int total_tiles = A.problems * A.m_tiles * A.n_tiles;
  constexpr int halves = HALVES;                 // 1 or 2
  const int tile_n = halves * gemm2::BN;         // O columns per apply tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&chunk_done[s], 1);
      mbar_init(&snap_done[s], 8);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);
    }
    for (int s = 0; s < APPLY_STAGES; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < TILE_SLOTS; ++s) {
      mbar_init(&tile_full[s], 1);
      mbar_init(&tile_empty[s], TILE_READERS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int p_stage = 0;
  uint32_t p_phase = 0;
  long p_issued = 0;
  long a_issued = 0;  // apply-ring stages the producer issued (for the drain after an abort)

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ producer (both CTAs)
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_z);
    tma_prefetch_desc(&map_za);
    tma_prefetch_desc(&map_weff_ld);
    tma_prefetch_desc(&map_w0);
    bool ok = true;
    for (int pr = cl; pr < upairs && ok; pr += n_cl) {
      for (int i = 0; i < S.n_chunks && ok; ++i) {
        const int nkb = state::chunk_kblocks(S, i);
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= S.units) break;
          int b, mb, nb;
          state::decode_unit(S, u, b, mb, nb);
          const int d0 = mb * state2::PAIR_D + (int)rank * state2::BMD;
          const int f0 = nb * state2::BNF + (int)rank * state2::BNF_HALF;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, S.st, abort_flag, 0x701)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + p_stage * STAGE_BYTES;
            uint8_t* sb = sa + A_BYTES;
            const uint32_t bar = cluster_addr(smem_u32(&full[p_stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[p_stage], 2 * STAGE_BYTES);
            const int tok = i * S.C + kb * state2::BKT;
            if (S.blocked) {  // the CTA's two 64-column blocks of V, then of Z, one request each
              tma_load_4d_pair(sa, &map_v, bar, 0, tok, d0 >> 6, b);
              tma_load_4d_pair(sb, &map_z, bar, 0, tok, f0 >> 6, b);
            } else {
              tma_load_3d_pair(sa, &map_v, bar, d0, tok, b);
              tma_load_3d_pair(sa + state2::BKT * 128, &map_v, bar, d0 + 64, tok, b);
              tma_load_3d_pair(sb, &map_z, bar, f0, tok, b);
              tma_load_3d_pair(sb + state2::BKT * 128, &map_z, bar, f0 + 64, tok, b);
            }
            ++p_issued;
            if (++p_stage == STAGES) {
              p_stage = 0;
              p_phase ^= 1u;
            }
          }
        }
      }
    }
    // wide tiles' ring overlays the state ring: first let the MMAs consume every state stage
    // issued (one more lap of waits on the state ring's empty barriers)
    for (int j = 0; j < STAGES && ok && halves == 2; ++j) {
      if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, S.st, abort_flag, 0x706)) ok = false;
      if (++p_stage == STAGES) {
        p_stage = 0;
        p_phase ^= 1u;
      }
    }
    // apply tiles: the even CTA claims them from the global queue and hands each to the odd CTA
    const uint32_t peer_tile_q = cluster_addr(smem_u32(tile_q), 1);
    const uint32_t peer_tile_full = cluster_addr(smem_u32(tile_full), 1);
    const uint32_t lead_tile_empty = cluster_addr(smem_u32(tile_empty), 0);
    // narrow tiles continue on the state ring (its stages, barriers and phases), wide tiles use
    // the apply ring from its start
    const bool wide = halves == 2;
    uint64_t* r_full = wide ? a_full : full;
    uint64_t* r_empty = wide ? a_empty : empty;
    const int r_stages = wide ? APPLY_STAGES : STAGES;
    const int r_bytes = wide ? APPLY_STAGE_BYTES : STAGE_BYTES;
    int a_stage = wide ? 0 : p_stage;
    uint32_t a_phase = wide ? 0u : p_phase;
    for (uint32_t k = 0; ok; ++k) {
      const int qs = (int)(k % TILE_SLOTS);
      const uint32_t par = (k / TILE_SLOTS) & 1u;
      int tile;
      if (rank == 0) {
        do {
          tile = (int)atomicAdd(p.next_tile, 1u);
          if (tile >= total_tiles) break;
          int prob, mt, nt;
          gemm::decode_tile(A, tile, prob, mt, nt);
          if (gemm2::pair_tile_active<gemm::kApply>(A, prob, mt)) break;
        } while (true);
        if (tile >= total_tiles) tile = -1;
        if (!wait_bounded_cluster(&tile_empty[qs], par ^ 1u, A.st, abort_flag, 0x702)) break;
        tile_q[qs] = tile;
        st_shared_cluster_u32(peer_tile_q + 4u * qs, (uint32_t)tile);
        mbar_arrive(&tile_full[qs]);
        mbar_arrive_cluster(peer_tile_full + 8u * qs);
      } else {
        if (!wait_bounded_cluster(&tile_full[qs], par, A.st, abort_flag, 0x703)) break;
        tile = tile_q[qs];
        mbar_arrive_cluster(lead_tile_empty + 8u * qs);
      }
      if (tile < 0) break;
      int prob, mt, nt;
      gemm::decode_tile(A, tile, prob, mt, nt);
      const int b = prob / A.n_chunks;
      const int i = prob - b * A.n_chunks;
      const bool from_w0 = i == 0 && A.first_from_w0;
      if (!from_w0) {
        if (!fused::wait_counter(&p.ready[prob], p.ready_target, A.st, abort_flag, 0x704)) break;
        fused::fence_proxy_async_global();
      }
      const int m0 = i * A.C + mt * gemm2::PAIR_M + (int)rank * gemm2::BM;
      for (int kb = 0; kb < A.k_blocks; ++kb) {
        if (!wait_bounded(&r_empty[a_stage], a_phase ^ 1u, A.st, abort_flag, 0x705)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + a_stage * r_bytes;
        uint8_t* sb = sa + gemm2::A_BYTES;
        const uint32_t bar = cluster_addr(smem_u32(&r_full[a_stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&r_full[a_stage], 2 * (gemm2::A_BYTES + halves * APPLY_B_HALF));
        const int k0 = kb * gemm2::BK;
        tma_load_3d_pair(sa, &map_za, bar, k0, m0, b);
        for (int j = 0; j < halves; ++j) {  // this CTA's 128 rows of each 256-column half of the tile
          const int n0 = nt * tile_n + j * gemm2::BN + (int)rank * gemm2::BN_HALF;
          if (from_w0)
            tma_load_2d_pair(sb + j * APPLY_B_HALF, &map_w0, bar, k0, n0);
          else
            tma_load_3d_pair(sb + j * APPLY_B_HALF, &map_weff_ld, bar, k0, n0, prob);
        }
        if (wide)
          ++a_issued;
        else
          ++p_issued;
        if (++a_stage == r_stages) {
          a_stage = 0;
          a_phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    {
      constexpr uint32_t idesc = idesc_bf16(state2::PAIR_D, state2::BNF, true, true);
      uint32_t snap_waits[2] = {0, 0};
      for (int pr = cl; pr < upairs && ok; pr += n_cl) {
        for (int i = 0; i < S.n_chunks && ok; ++i) {
          const int nkb = state::chunk_kblocks(S, i);
          for (int slot = 0; slot < 2 && ok; ++slot) {
            const int u = 2 * pr + slot;
            if (u >= S.units) break;
            if (!wait_bounded_cluster(&snap_done[slot], snap_waits[slot] & 1u, S.st, abort_flag, 0x711)) {
              ok = false;
              break;
            }
            ++snap_waits[slot];
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(slot * state2::BNF);
            for (int kb = 0; kb < nkb; ++kb) {
              if (!wait_bounded(&full[stage], phase, S.st, abort_flag, 0x712)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
              const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
              for (int kk = 0; kk < state2::BKT / 16; ++kk)
                tc_mma_bf16_pair(d_tmem, sdesc_sw128(a_addr + kk * 2048, state2::BKT * 128, 1024),
                                 sdesc_sw128(b_addr + kk * 2048, state2::BKT * 128, 1024), idesc, 1u);
              tc_commit_pair(&empty[stage], 0x3);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            tc_commit_pair(&chunk_done[slot], 0x3);
          }
        }
      }
    }
    {
      constexpr uint32_t idesc = idesc_bf16(gemm2::PAIR_M, gemm2::BN, false, false);
      const bool wide = halves == 2;
      uint64_t* r_full = wide ? a_full : full;
      uint64_t* r_empty = wide ? a_empty : empty;
      const int r_stages = wide ? APPLY_STAGES : STAGES;
      const int r_bytes = wide ? APPLY_STAGE_BYTES : STAGE_BYTES;
      int a_stage = wide ? 0 : stage;
      uint32_t a_phase = wide ? 0u : phase;
      int it = 0;
      for (uint32_t k = 0; ok; ++k) {
        const int qs = (int)(k % TILE_SLOTS);
        if (!wait_bounded(&tile_full[qs], (k / TILE_SLOTS) & 1u, A.st, abort_flag, 0x713)) break;
        const int tile = tile_q[qs];
        mbar_arrive(&tile_empty[qs]);
        if (tile < 0) break;
        // one accumulator (two halves) or two in turn; the first wait of each is released by the
        // epilogues' end of the state phase
        const int buf = halves == 2 ? 0 : (it & 1);
        const uint32_t use = (uint32_t)(halves == 2 ? it : it >> 1);
        if (!wait_bounded_cluster(&acc_empty[buf], use & 1u, A.st, abort_flag, 0x714)) break;
        tc_fence_after();
        for (int kb = 0; kb < A.k_blocks; ++kb) {
          if (!wait_bounded(&r_full[a_stage], a_phase, A.st, abort_flag, 0x715)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + a_stage * r_bytes);
          const uint32_t b_addr = a_addr + gemm2::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < gemm2::BK / 16; ++kk)
            for (int j = 0; j < halves; ++j)
              tc_mma_bf16_pair(tmem_base + (uint32_t)((buf + j) * gemm2::BN), sdesc_sw128(a_addr + kk * 32, 16, 1024),
                               sdesc_sw128(b_addr + j * APPLY_B_HALF + kk * 32, 16, 1024), idesc,
                               (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair(&r_empty[a_stage], 0x3);
          if (++a_stage == r_stages) {
            a_stage = 0;
            a_phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[buf], 0x3);
        ++it;
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_weff_st);
    tma_prefetch_desc(&map_wfin);
    tma_prefetch_desc(&map_o);
    const uint32_t lead_snap_done = cluster_addr(smem_u32(snap_done), 0);
    const uint32_t lead_acc_empty = cluster_addr(smem_u32(acc_empty), 0);
    const uint32_t lead_tile_empty = cluster_addr(smem_u32(tile_empty), 0);
    // this warp is done with an accumulator: after initialising it (tcgen05.st, release
    // semantics) or after reading it (relaxed: the reads have completed)
    auto release = [&](uint32_t lead_bar, bool after_reads = true) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (after_reads)
          mbar_arrive_cluster_relaxed(lead_bar);
        else
          mbar_arrive_cluster(lead_bar);
      }
    };
    bool ok = true;
    int pending = -1;  // slice whose stores this warp issued last and has not published yet
    auto publish = [&](int slice) {
      if (lane == 0) {
        fused::fence_proxy_async_global();
        fused::red_release_gpu_add(&p.ready[slice], 1u);
      }
    };
    uint32_t chunk_waits[2] = {0, 0};
    for (int pr = cl; pr < upairs && ok; pr += n_cl) {
      for (int slot = 0; slot < 2; ++slot) {
        const int u = 2 * pr + slot;
        if (u >= S.units) break;
        int b, mb, nb;
        state::decode_unit(S, u, b, mb, nb);
        const int row0 = mb * state2::PAIR_D + (int)rank * state2::BMD;
        const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * state2::BNF);
#pragma unroll 1
        for (int c = 0; c < state2::BNF / 32; ++c) {
          uint32_t r[32];
          state::load_init32(S, b, row0 + r_in_tile, nb * state2::BNF + c * 32, r);
          tmem_st32(t_row + c * 32, r);
        }
        tmem_st_wait();
        if (!S.skip_first) {  // per-sequence starting state: W_eff[b, 0] is this state in bf16
          const int slice = b * S.n_chunks;
          state::snapshot_bf16(out, t_row, &map_weff_st, nb * state2::BNF, row0 + q * 32, slice);
          if (lane == 0) fused::bulk_wait_pending<4>();
          if (pending >= 0) publish(pending);
          pending = slice;
        }
        release(lead_snap_done + 8u * slot, false);
      }
      for (int i = 1; i <= S.n_chunks && ok; ++i) {
        for (int slot = 0; slot < 2; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= S.units) break;
          if (!wait_bounded(&chunk_done[slot], chunk_waits[slot] & 1u, S.st, abort_flag, 0x721)) {
            ok = false;
            break;
          }
          ++chunk_waits[slot];
          tc_fence_after();
          int b, mb, nb;
          state::decode_unit(S, u, b, mb, nb);
          const int row0 = mb * state2::PAIR_D + (int)rank * state2::BMD;
          const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * state2::BNF);
          if (i < S.n_chunks) {
            const int slice = b * S.n_chunks + i;
            state::snapshot_bf16(out, t_row, &map_weff_st, nb * state2::BNF, row0 + q * 32, slice);
            release(lead_snap_done + 8u * slot);
            // every snapshot is 4 bulk groups: all groups before this one's have completed
            if (lane == 0) fused::bulk_wait_pending<4>();
            if (pending >= 0) publish(pending);
            pending = slice;
          } else {
            if (lane == 0) bulk_wait_all();
            if (pending >= 0) publish(pending);
            pending = -1;
            state::snapshot_f32(out, t_row, &map_wfin, nb * state2::BNF, row0 + q * 32, b);
            tc_fence_before();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    if (pending >= 0) publish(pending);
    // the tensor memory is free: release the accumulator(s) to the apply phase
    release(lead_acc_empty);
    if (halves == 1) release(lead_acc_empty + 8u);
    int it = 0;
    for (uint32_t k = 0; ok; ++k) {
      const int qs = (int)(k % TILE_SLOTS);
      if (!wait_bounded_cluster(&tile_full[qs], (k / TILE_SLOTS) & 1u, A.st, abort_flag, 0x722)) break;
      const int tile = tile_q[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_tile_empty + 8u * qs);
      if (tile < 0) break;
      int prob, mt, nt;
      gemm::decode_tile(A, tile, prob, mt, nt);
      const int b = prob / A.n_chunks;
      const int i = prob - b * A.n_chunks;
      const int buf = halves == 2 ? 0 : (it & 1);
      const uint32_t use = (uint32_t)(halves == 2 ? it : it >> 1);
      if (!wait_bounded(&acc_full[buf], use & 1u, A.st, abort_flag, 0x723)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * gemm2::BN);
      const int row = i * A.C + mt * gemm2::PAIR_M + (int)rank * gemm2::BM + q * 32;
#pragma unroll 1
      for (int h = 0; h < tile_n / 64; ++h) {
        uint32_t rw[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t a[32];
          tmem_ld32(t_row + h * 64 + half * 32, a);
          tmem_ld_wait(a);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            rw[half * 16 + e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
        }
        out.put(rw, &map_o, nt * tile_n + h * 64, row, b);
      }
      release(lead_acc_empty + 8u * buf);
      ++it;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 1 && lane == 0 && rank == 0) {
      tc_commit_pair(drain, 0x1);
      drain_wait(drain, 0, 50000000ull);
    }
    if (warp == 0 && lane == 0 && rank == 0) {
      for (long j = p_issued - 1; j >= 0 && j >= p_issued - STAGES; --j)
        drain_wait(&full[j % STAGES], (uint32_t)((j / STAGES) & 1), 50000000ull);
      for (long j = a_issued - 1; j >= 0 && j >= a_issued - APPLY_STAGES; --j)
        drain_wait(&a_full[j % APPLY_STAGES], (uint32_t)((j / APPLY_STAGES) & 1), 50000000ull);
    }
    __syncthreads();
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace fused2
}  // namespace ipttt
