// Fused chunk-state + per-chunk apply: one cooperative persistent launch for steps (3)-(5).
//
// zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.2 Steps 1-3: the
// state units (tc_state.cuh) produce the per-chunk weights W_eff[i]; the apply tiles
// (tc_gemm.cuh, kind Apply) consume them.  Run as two kernels, the state kernel ends with a
// partial round (the d x d_ff state is larger than all TMEM at once), leaving SMs idle.  Here
// every CTA first runs its state unit pairs, then pulls apply tiles from a global queue in
// chunk order, so the apply work fills the SMs that the state work leaves idle.
//
// Hand-off: after the TMA stores of a W_eff slice have completed, each epilogue warp makes
// them visible (fence.proxy.async + a release add) on the slice's counter; an apply tile of
// chunk i >= 1 waits (bounded) until all units of its sequence have published chunk i, then
// fences (fence.proxy.async) before its TMA loads.  Chunk 0 is applied with W_down0 itself,
// or, when each sequence starts from its own state (a resumed call), with W_eff[b, 0], which
// the state phase then writes and publishes like the other slices.
// All CTAs are co-resident (cooperative launch, one CTA per SM), so these waits always end.
#pragma once

#include "ptx.cuh"
#include "tc_gemm.cuh"
#include "tc_state.cuh"

namespace ipttt {
namespace fused {

constexpr int STAGES = 4;
constexpr int STAGE_BYTES = 48 * 1024;
static_assert(state::STAGE_BYTES == STAGE_BYTES && gemm::STAGE_BYTES == STAGE_BYTES, "one ring serves both phases");
static_assert(state::A_BYTES == gemm::A_BYTES, "A tiles share the stage layout");
constexpr int A_BYTES = gemm::A_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int TILE_SLOTS = 4;  // apply tiles in flight between the producer and the epilogue
constexpr int BAR_BYTES = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;

struct Params {
  state::Params s;        // skip_first = 1 (W_eff[b, 0] not written) unless s.W_init is given
  gemm::Params a;         // Apply tiling; first_from_w0 = s.skip_first
  uint32_t* ready;        // [B * n_chunks]: published (unit, epilogue warp) snapshots of each slice
  uint32_t* next_tile;    // apply-tile queue head
  uint32_t ready_target;  // m_units * n_units * 4
  int a_halves;           // CTA-pair kernel: 256-column halves per apply tile (2: 512 columns, one
                          // accumulator; 1: 256 columns, two accumulators in turn); the host
                          // launches the kernel instantiation of that width
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_pending() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Bounded wait until *p >= target (another CTA's release add).
__device__ __forceinline__ bool wait_counter(const uint32_t* p, uint32_t target, const DevStatus& st,
                                             volatile int* abort, uint32_t site) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
    if (*abort) return false;
    if (global_ns() - t0 > st.limit_ns) {
      *abort = 1;
      record_error(st, kDevStatusTimeout, site);
      return false;
    }
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_state_apply_kernel(const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_z,
                          const __grid_constant__ CUtensorMap map_weff_st, const __grid_constant__ CUtensorMap map_wfin,
                          const __grid_constant__ CUtensorMap map_za, const __grid_constant__ CUtensorMap map_weff_ld,
                          const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_o,
                          const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                        // [STAGES]
  uint64_t* empty = full + STAGES;              // [STAGES]
  uint64_t* chunk_done = empty + STAGES;        // [2]  state: MMA -> epilogue
  uint64_t* snap_done = chunk_done + 2;         // [2]  state: epilogue -> MMA
  uint64_t* acc_full = snap_done + 2;           // [2]  apply: MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;           // [2]  apply: epilogue -> MMA
  uint64_t* tile_full = acc_empty + 2;          // [TILE_SLOTS] producer -> MMA + epilogue
  uint64_t* tile_empty = tile_full + TILE_SLOTS;  // [TILE_SLOTS] MMA + epilogue -> producer
  uint64_t* drain = tile_empty + TILE_SLOTS;
  int* tile_q = reinterpret_cast<int*>(drain + 1);  // [TILE_SLOTS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_q + TILE_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const state::Params& S = p.s;
  const gemm::Params& A = p.a;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pairs = (S.units + 1) / 2;
  const int total_tiles = A.problems * A.m_tiles * A.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&chunk_done[s], 1);
      mbar_init(&snap_done[s], 128);
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 128);
    }
    for (int s = 0; s < TILE_SLOTS; ++s) {
      mbar_init(&tile_full[s], 1);
      mbar_init(&tile_empty[s], 129);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int p_stage = 0;
  uint32_t p_phase = 0;
  long p_issued = 0;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ producer
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_z);
    tma_prefetch_desc(&map_za);
    tma_prefetch_desc(&map_weff_ld);
    tma_prefetch_desc(&map_w0);
    bool ok = true;
    for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
      for (int i = 0; i < S.n_chunks && ok; ++i) {
        const int nkb = state::chunk_kblocks(S, i);
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= S.units) break;
          int b, mb, nb;
          state::decode_unit(S, u, b, mb, nb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, S.st, abort_flag, 0x401)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + p_stage * STAGE_BYTES;
            uint8_t* sb = sa + A_BYTES;
            mbar_arrive_expect_tx(&full[p_stage], STAGE_BYTES);
            const int tok = i * S.C + kb * state::BKT;
            tma_load_3d(sa, &map_v, &full[p_stage], mb * state::BMD, tok, b);
            tma_load_3d(sa + state::BKT * 128, &map_v, &full[p_stage], mb * state::BMD + 64, tok, b);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_3d(sb + j * (state::BKT * 128), &map_z, &full[p_stage], nb * state::BNF + j * 64, tok, b);
            ++p_issued;
            if (++p_stage == STAGES) {
              p_stage = 0;
              p_phase ^= 1u;
            }
          }
        }
      }
    }
    // apply tiles, claimed from the global queue in chunk order
    for (uint32_t k = 0; ok; ++k) {
      int tile;
      do {
        tile = (int)atomicAdd(p.next_tile, 1u);
        if (tile >= total_tiles) break;
        int prob, mt, nt;
        gemm::decode_tile(A, tile, prob, mt, nt);
        if (gemm::tile_active<gemm::kApply>(A, prob, mt)) break;
      } while (true);
      if (tile >= total_tiles) tile = -1;
      const int qs = (int)(k % TILE_SLOTS);
      if (!wait_bounded(&tile_empty[qs], ((k / TILE_SLOTS) & 1u) ^ 1u, A.st, abort_flag, 0x402)) break;
      tile_q[qs] = tile;
      mbar_arrive(&tile_full[qs]);
      if (tile < 0) break;
      int prob, mt, nt;
      gemm::decode_tile(A, tile, prob, mt, nt);
      const int b = prob / A.n_chunks;
      const int i = prob - b * A.n_chunks;
      const bool from_w0 = i == 0 && A.first_from_w0;
      if (!from_w0) {
        if (!wait_counter(&p.ready[prob], p.ready_target, A.st, abort_flag, 0x403)) break;
        fence_proxy_async_global();
      }
      for (int kb = 0; kb < A.k_blocks; ++kb) {
        if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, A.st, abort_flag, 0x404)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + p_stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        mbar_arrive_expect_tx(&full[p_stage], STAGE_BYTES);
        const int k0 = kb * gemm::BK;
        tma_load_3d(sa, &map_za, &full[p_stage], k0, i * A.C + mt * gemm::BM, b);
        if (from_w0)
          tma_load_2d(sb, &map_w0, &full[p_stage], k0, nt * gemm::BN);
        else
          tma_load_3d(sb, &map_weff_ld, &full[p_stage], k0, nt * gemm::BN, prob);
        ++p_issued;
        if (++p_stage == STAGES) {
          p_stage = 0;
          p_phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    {
      constexpr uint32_t idesc = idesc_bf16(state::BMD, state::BNF, true, true);
      uint32_t snap_waits[2] = {0, 0};
      for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
        for (int i = 0; i < S.n_chunks && ok; ++i) {
          const int nkb = state::chunk_kblocks(S, i);
          for (int slot = 0; slot < 2 && ok; ++slot) {
            const int u = 2 * pr + slot;
            if (u >= S.units) break;
            if (!wait_bounded(&snap_done[slot], snap_waits[slot] & 1u, S.st, abort_flag, 0x411)) {
              ok = false;
              break;
            }
            ++snap_waits[slot];
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(slot * state::BNF);
            for (int kb = 0; kb < nkb; ++kb) {
              if (!wait_bounded(&full[stage], phase, S.st, abort_flag, 0x412)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
              const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
              for (int kk = 0; kk < state::BKT / 16; ++kk)
                tc_mma_bf16(d_tmem, sdesc_sw128(a_addr + kk * 2048, state::BKT * 128, 1024),
                            sdesc_sw128(b_addr + kk * 2048, state::BKT * 128, 1024), idesc, 1u);
              tc_commit(&empty[stage]);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            tc_commit(&chunk_done[slot]);
          }
        }
      }
    }
    {
      constexpr uint32_t idesc = idesc_bf16(gemm::BM, gemm::BN, false, false);
      int it = 0;
      for (uint32_t k = 0; ok; ++k) {
        const int qs = (int)(k % TILE_SLOTS);
        if (!wait_bounded(&tile_full[qs], (k / TILE_SLOTS) & 1u, A.st, abort_flag, 0x413)) break;
        const int tile = tile_q[qs];
        mbar_arrive(&tile_empty[qs]);
        if (tile < 0) break;
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        // the first wait of each buffer is released by the epilogue's end of the state phase
        if (!wait_bounded(&acc_empty[buf], use & 1u, A.st, abort_flag, 0x414)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * gemm::BN);
        for (int kb = 0; kb < A.k_blocks; ++kb) {
          if (!wait_bounded(&full[stage], phase, A.st, abort_flag, 0x415)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < gemm::BK / 16; ++kk)
            tc_mma_bf16(d_tmem, sdesc_sw128(a_addr + kk * 32, 16, 1024), sdesc_sw128(b_addr + kk * 32, 16, 1024),
                        idesc, (kb | kk) != 0 ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        ++it;
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_weff_st);
    tma_prefetch_desc(&map_wfin);
    tma_prefetch_desc(&map_o);
    bool ok = true;
    int pending = -1;  // slice whose stores this warp issued last and has not published yet
    auto publish = [&](int slice) {
      if (lane == 0) {
        fence_proxy_async_global();
        red_release_gpu_add(&p.ready[slice], 1u);
      }
    };
    uint32_t chunk_waits[2] = {0, 0};
    for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
      for (int slot = 0; slot < 2; ++slot) {
        const int u = 2 * pr + slot;
        if (u >= S.units) break;
        int b, mb, nb;
        state::decode_unit(S, u, b, mb, nb);
        const int row = mb * state::BMD + r_in_tile;
        const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * state::BNF);
#pragma unroll 1
        for (int c = 0; c < state::BNF / 32; ++c) {
          uint32_t r[32];
          state::load_init32(S, b, row, nb * state::BNF + c * 32, r);
          tmem_st32(t_row + c * 32, r);
        }
        tmem_st_wait();
        if (!S.skip_first) {  // per-sequence starting state: W_eff[b, 0] is this state in bf16
          const int slice = b * S.n_chunks;
          state::snapshot_bf16(out, t_row, &map_weff_st, nb * state::BNF, mb * state::BMD + q * 32, slice);
          if (lane == 0) bulk_wait_pending<4>();
          if (pending >= 0) publish(pending);
          pending = slice;
        }
        tc_fence_before();
        mbar_arrive(&snap_done[slot]);
      }
      for (int i = 1; i <= S.n_chunks && ok; ++i) {
        for (int slot = 0; slot < 2; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= S.units) break;
          if (!wait_bounded(&chunk_done[slot], chunk_waits[slot] & 1u, S.st, abort_flag, 0x421)) {
            ok = false;
            break;
          }
          ++chunk_waits[slot];
          tc_fence_after();
          int b, mb, nb;
          state::decode_unit(S, u, b, mb, nb);
          const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * state::BNF);
          if (i < S.n_chunks) {
            const int slice = b * S.n_chunks + i;
            state::snapshot_bf16(out, t_row, &map_weff_st, nb * state::BNF, mb * state::BMD + q * 32, slice);
            tc_fence_before();
            mbar_arrive(&snap_done[slot]);
            // every snapshot is 4 bulk groups: all groups before this one's have completed
            if (lane == 0) bulk_wait_pending<4>();
            if (pending >= 0) publish(pending);
            pending = slice;
          } else {
            if (lane == 0) bulk_wait_all();
            if (pending >= 0) publish(pending);
            pending = -1;
            state::snapshot_f32(out, t_row, &map_wfin, nb * state::BNF, mb * state::BMD + q * 32, b);
            tc_fence_before();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    if (pending >= 0) publish(pending);
    // the accumulators are free: release them to the apply phase
    tc_fence_before();
    mbar_arrive(&acc_empty[0]);
    mbar_arrive(&acc_empty[1]);
    int it = 0;
    for (uint32_t k = 0; ok; ++k) {
      const int qs = (int)(k % TILE_SLOTS);
      if (!wait_bounded(&tile_full[qs], (k / TILE_SLOTS) & 1u, A.st, abort_flag, 0x422)) break;
      const int tile = tile_q[qs];
      mbar_arrive(&tile_empty[qs]);
      if (tile < 0) break;
      int prob, mt, nt;
      gemm::decode_tile(A, tile, prob, mt, nt);
      const int b = prob / A.n_chunks;
      const int i = prob - b * A.n_chunks;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded(&acc_full[buf], use & 1u, A.st, abort_flag, 0x423)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * gemm::BN);
#pragma unroll 1
      for (int h = 0; h < gemm::BN / 64; ++h) {
        uint32_t a[32], c2[32], row[32];
        tmem_ld32(t_row + h * 64, a);
        tmem_ld32(t_row + h * 64 + 32, c2);
        tmem_ld_wait(a);
        tmem_ld_wait(c2);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          row[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
          row[16 + e] = pack_bf16x2(__uint_as_float(c2[2 * e]), __uint_as_float(c2[2 * e + 1]));
        }
        out.put(row, &map_o, nt * gemm::BN + h * 64, i * A.C + mt * gemm::BM + q * 32, b);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      ++it;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 1 && lane == 0) {
      tc_commit(drain);
      drain_wait(drain, 0, 50000000ull);
    }
    if (warp == 0 && lane == 0) {
      for (long j = p_issued - 1; j >= 0 && j >= p_issued - STAGES; --j)
        drain_wait(&full[j % STAGES], (uint32_t)((j / STAGES) & 1), 50000000ull);
    }
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace fused
}  // namespace ipttt
