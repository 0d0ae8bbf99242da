// The chunk-state kernel of tc_state.cuh on CTA pairs (clusters of two CTAs on two SMs).
//
// zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.2 Steps 1-2 and the
// §3.3 update rule, exactly as in tc_state.cuh: each unit's fp32 state stays in tensor memory,
// is snapshotted to the bf16 W_eff stack before every chunk and accumulates V_i^T Z_i.
//
// Why pairs: with 128 (d) x 256 (d_ff) units a CTA loads 48 KB of V and Z from L2 for every
// 4.2 MFLOP, and the single-CTA kernel is bound by that L2-to-SM traffic (it runs as fast
// with its MMAs removed).  A pair unit is 256 (d) x 256 (d_ff): each CTA loads its own 128
// columns of V and 128 columns of Z (32 KB per 4.2 MFLOP, one third less), the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256 state rows, N = 256), and each CTA's tensor memory holds
// its own 128 state rows.  Two units per pair run side by side, as in tc_state.cuh, so the
// snapshot of one overlaps the MMAs of the other.
//
//   warp 0      TMA producer of its CTA (6 stages of 32 KB); both CTAs' copies complete on the
//               even CTA's `full` barrier.
//   warp 1      the even CTA's lane 0 issues the pair's MMAs; commits go to both CTAs.
//   warps 2-5   each CTA initialises, snapshots and finally stores its own 128 state rows, and
//               releases the unit to the MMA issuer (one arrival per warp on the even CTA's
//               `snap_done`).
#pragma once

#include "tc_state.cuh"

namespace ipttt {
namespace state2 {

using state::Params;

constexpr int BMD = 128;     // state rows per CTA
constexpr int PAIR_D = 256;  // state rows per pair unit
constexpr int BNF = 256;     // state columns per unit
constexpr int BNF_HALF = 128;
constexpr int BKT = 64;  // tokens per stage
constexpr int STAGES = 6;
constexpr int A_BYTES = BMD * BKT * 2;       // 2 boxes of 64 d x 64 tokens
constexpr int B_BYTES = BNF_HALF * BKT * 2;  // 2 boxes of 64 d_ff x 64 tokens
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier block");

// Pair units are decoded by state::decode_unit (sequence b, state block mb, column block nb,
// mb fastest); p.m_units counts 256-row blocks here.

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    tc_state2_kernel(const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_z,
                     const __grid_constant__ CUtensorMap map_weff, const __grid_constant__ CUtensorMap map_wfin,
                     const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                     // [STAGES], used in the even CTA
  uint64_t* empty = bars + STAGES;           // [STAGES], each CTA
  uint64_t* chunk_done = bars + 2 * STAGES;  // [2] MMA -> epilogues (both CTAs)
  uint64_t* snap_done = chunk_done + 2;      // [2] epilogues -> MMA (even CTA)
  uint64_t* drain = snap_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1;
  const int n_cl = gridDim.x >> 1;
  const int upairs = (p.units + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&chunk_done[s], 1);
      mbar_init(&snap_done[s], 8);  // one arrival per epilogue warp of both CTAs
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

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_z);
    bool ok = true;
    for (int pr = cl; pr < upairs && ok; pr += n_cl) {
      for (int j = 0; j < p.n_chunks && ok; ++j) {
        const int i = state::chunk_at(p, j);
        const int nkb = state::chunk_kblocks(p, i);
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          int b, mb, nb;
          state::decode_unit(p, u, b, mb, nb);
          const int d0 = mb * PAIR_D + (int)rank * BMD;
          const int f0 = nb * BNF + (int)rank * BNF_HALF;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, p.st, abort_flag, 0x601)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + p_stage * STAGE_BYTES;
            uint8_t* sb = sa + A_BYTES;
            const uint32_t bar = cluster_addr(smem_u32(&full[p_stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[p_stage], 2 * STAGE_BYTES);
            const int tok = i * p.C + kb * BKT;
            if (p.blocked) {  // the CTA's two 64-column blocks of V, then of Z, one request each
              tma_load_4d_pair(sa, &map_v, bar, 0, tok, d0 >> 6, b);
              tma_load_4d_pair(sb, &map_z, bar, 0, tok, f0 >> 6, b);
            } else {
              tma_load_3d_pair(sa, &map_v, bar, d0, tok, b);
              tma_load_3d_pair(sa + BKT * 128, &map_v, bar, d0 + 64, tok, b);
              tma_load_3d_pair(sb, &map_z, bar, f0, tok, b);
              tma_load_3d_pair(sb + BKT * 128, &map_z, bar, f0 + 64, tok, b);
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
  } else if (warp == 1 && lane == 0 && rank == 0) {
    constexpr uint32_t idesc = idesc_bf16(PAIR_D, BNF, true, true);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t snap_waits[2] = {0, 0};
    bool ok = true;
    for (int pr = cl; pr < upairs && ok; pr += n_cl) {
      for (int j = 0; j < p.n_chunks && ok; ++j) {
        const int nkb = state::chunk_kblocks(p, state::chunk_at(p, j));
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          if (!wait_bounded_cluster(&snap_done[slot], snap_waits[slot] & 1u, p.st, abort_flag, 0x602)) {
            ok = false;
            break;
          }
          ++snap_waits[slot];
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(slot * BNF);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&full[stage], phase, p.st, abort_flag, 0x603)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BKT / 16; ++kk) {
              // 16 tokens = 16 rows of 128 B; the two 64-wide blocks along d / d_ff are BKT*128 B apart
              const uint64_t adesc = sdesc_sw128(a_addr + kk * 2048, BKT * 128, 1024);
              const uint64_t bdesc = sdesc_sw128(b_addr + kk * 2048, BKT * 128, 1024);
              tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, 1u);
            }
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
  } else if (warp >= 2) {
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_weff);
    tma_prefetch_desc(&map_wfin);
    // this warp is done with the unit's accumulator: after initialising it (tcgen05.st, release
    // semantics) or after reading it (relaxed: the reads have completed)
    auto release = [&](int slot, bool after_reads) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = cluster_addr(smem_u32(&snap_done[slot]), 0);
        if (after_reads)
          mbar_arrive_cluster_relaxed(bar);
        else
          mbar_arrive_cluster(bar);
      }
    };
    uint32_t chunk_waits[2] = {0, 0};
    bool ok = true;
    for (int pr = cl; pr < upairs && ok; pr += n_cl) {
      for (int slot = 0; slot < 2; ++slot) {
        const int u = 2 * pr + slot;
        if (u >= p.units) break;
        int b, mb, nb;
        state::decode_unit(p, u, b, mb, nb);
        const int row0 = mb * PAIR_D + (int)rank * BMD;
        const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * BNF);
#pragma unroll 1
        for (int c = 0; c < BNF / 32; ++c) {
          uint32_t r[32];
          state::load_init32(p, b, row0 + r_in_tile, nb * BNF + c * 32, r);
          tmem_st32(t_row + c * 32, r);
        }
        tmem_st_wait();
        if (!p.skip_first && !p.no_snap)
          state::snapshot_bf16(out, t_row, &map_weff, nb * BNF, row0 + q * 32, b * p.n_chunks + state::chunk_at(p, 0));
        release(slot, false);
      }
      for (int i = 1; i <= p.n_chunks && ok; ++i) {
        for (int slot = 0; slot < 2; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          if (!wait_bounded(&chunk_done[slot], chunk_waits[slot] & 1u, p.st, abort_flag, 0x604)) {
            ok = false;
            break;
          }
          ++chunk_waits[slot];
          tc_fence_after();
          int b, mb, nb;
          state::decode_unit(p, u, b, mb, nb);
          const int row0 = mb * PAIR_D + (int)rank * BMD;
          const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * BNF);
          if (i < p.n_chunks) {
            if (!p.no_snap)
              state::snapshot_bf16(out, t_row, &map_weff, nb * BNF, row0 + q * 32,
                                   b * p.n_chunks + state::chunk_at(p, i));
            release(slot, true);
          } else {
            state::snapshot_f32(out, t_row, &map_wfin, nb * BNF, row0 + q * 32, b);
            tc_fence_before();
          }
        }
      }
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

}  // namespace state2
}  // namespace ipttt
