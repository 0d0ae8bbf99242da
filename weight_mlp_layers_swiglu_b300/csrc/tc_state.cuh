// Chunk-state kernel: the running fast weight, held in tensor memory.
//
// The same kernel runs the backward pass's reverse scan (chunks last to first, started from
// dW_final: its snapshots are the exclusive suffix sums R_i = dW_final + sum_{l>i} dO_l^T Z_l)
// and, with one chunk and a zero start, plain reductions over tokens (A^T B of two
// token-major matrices, the weight gradients).
//
// zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.2 Steps 1-2 and the
// §3.3 update rule: for each chunk i of a sequence, Delta_i = V_i^T Z_i, and chunk i is
// applied with W_eff[i] = W_down0 + sum_{j<i} Delta_j (V arrives pre-scaled by eta), so
// W_eff is the exclusive prefix sum of the chunk updates.
//
// One work unit is a 128 (d) x 256 (d_ff) tile of the state of one sequence.  Its fp32
// accumulator lives in TMEM for the whole sequence: it is initialised with the W_down0 tile
// (tcgen05.st), and for every chunk the epilogue first snapshots it to the bf16 W_eff stack,
// then the MMA warp adds the chunk's V_i^T Z_i with tcgen05.mma contracting over the chunk's
// tokens (both operands token-major, i.e. MN-major in shared memory).  After the last chunk
// the accumulator is the final fp32 W_down.
//
// Each CTA runs two units side by side (2 x 256 TMEM columns) in lock step, so the snapshot
// of one unit overlaps the MMAs of the other and the tensor pipe never waits for a snapshot.
// Warp roles as in the GEMM: warp 0 TMA, warp 1 MMA, warps 2-5 snapshot/epilogue.
#pragma once

#include "ptx.cuh"

namespace ipttt {
namespace state {

constexpr int BMD = 128;  // state rows (d) per unit
constexpr int BNF = 256;  // state columns (d_ff) per unit
constexpr int BKT = 64;   // tokens per pipeline stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BMD * BKT * 2;  // V tile: 2 boxes of 64 d x 64 tokens
constexpr int B_BYTES = BNF * BKT * 2;  // Z tile: 4 boxes of 64 d_ff x 64 tokens
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
// Output staging: each epilogue warp owns two 4 KB boxes (32 rows x 128 B, 128-byte swizzle)
// that alternate between TMA tensor stores.
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;

struct Params {
  int B, T, d, f, C, n_chunks;
  int m_units, n_units, units;  // units = B * n_units * m_units
  const __nv_bfloat16* W0;      // [d, f]; W_eff [B, n_chunks, d, f] and W_final [B, d, f] via tensor maps
  int skip_first;               // 1: W_eff[b, 0] (= W_down0) is not written (the apply reads W_down0)
  const float* W_init;          // optional [B, d, f] fp32: each sequence's own starting state
  int reverse;                  // 1: chunks run last to first (the backward pass's suffix scan)
  int no_snap;                  // 1: no W_eff snapshot at all, only the final state (update totals)
  int blocked;                  // 1 (CTA-pair kernels): V and Z maps are 4-D, [B][n/64][T][64] blocks
  DevStatus st;
};

// The chunk processed at step j: j, or n-1-j when the scan runs backwards.
__device__ __forceinline__ int chunk_at(const Params& p, int j) { return p.reverse ? p.n_chunks - 1 - j : j; }

// The accumulator's starting value for state rows `row`, columns col .. col+31 of sequence b:
// W_init[b] (fp32) when given, else W_down0 (bf16), else zero (a plain reduction over tokens).
__device__ __forceinline__ void load_init32(const Params& p, int b, int row, int col, uint32_t (&r)[32]) {
  const bool row_ok = row < p.d;
  if (p.W_init == nullptr && p.W0 == nullptr) {
#pragma unroll
    for (int e = 0; e < 32; ++e) r[e] = 0u;
    return;
  }
  if (p.W_init != nullptr) {
    const float* src = p.W_init + ((int64_t)b * p.d + row) * p.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row_ok && col + g * 4 < p.f) v = *reinterpret_cast<const float4*>(src + col + g * 4);
      r[g * 4 + 0] = __float_as_uint(v.x);
      r[g * 4 + 1] = __float_as_uint(v.y);
      r[g * 4 + 2] = __float_as_uint(v.z);
      r[g * 4 + 3] = __float_as_uint(v.w);
    }
    return;
  }
  const __nv_bfloat16* src = p.W0 + (int64_t)row * p.f;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (row_ok && col + g * 8 < p.f) w = *reinterpret_cast<const uint4*>(src + col + g * 8);
    r[g * 8 + 0] = __float_as_uint(bf16_lo(w.x));
    r[g * 8 + 1] = __float_as_uint(bf16_hi(w.x));
    r[g * 8 + 2] = __float_as_uint(bf16_lo(w.y));
    r[g * 8 + 3] = __float_as_uint(bf16_hi(w.y));
    r[g * 8 + 4] = __float_as_uint(bf16_lo(w.z));
    r[g * 8 + 5] = __float_as_uint(bf16_hi(w.z));
    r[g * 8 + 6] = __float_as_uint(bf16_lo(w.w));
    r[g * 8 + 7] = __float_as_uint(bf16_hi(w.w));
  }
}

// Reads the 256 accumulator columns of this thread's TMEM lane and stores them as bf16
// W_eff rows (4 boxes of 64 columns) for state rows y.. y+31 of slice z.
__device__ __forceinline__ void snapshot_bf16(OutStager& out, uint32_t t_row, const CUtensorMap* map, int x0, int y,
                                              int z) {
#pragma unroll 1
  for (int g = 0; g < BNF / 64; ++g) {
    uint32_t a[32], b[32], row[32];
    tmem_ld32(t_row + g * 64, a);
    tmem_ld32(t_row + g * 64 + 32, b);
    tmem_ld_wait(a);
    tmem_ld_wait(b);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      row[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
      row[16 + e] = pack_bf16x2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
    }
    out.put(row, map, x0 + g * 64, y, z);
  }
}

// The same for the fp32 final state (8 boxes of 32 columns).
__device__ __forceinline__ void snapshot_f32(OutStager& out, uint32_t t_row, const CUtensorMap* map, int x0, int y,
                                             int z) {
#pragma unroll 1
  for (int g = 0; g < BNF / 32; ++g) {
    uint32_t a[32];
    tmem_ld32(t_row + g * 32, a);
    tmem_ld_wait(a);
    out.put(a, map, x0 + g * 32, y, z);
  }
}

// Unit order: d-tile fastest, so that concurrently running CTAs share the same Z columns.
__device__ __forceinline__ void decode_unit(const Params& p, int u, int& b, int& mb, int& nb) {
  mb = u % p.m_units;
  const int r = u / p.m_units;
  nb = r % p.n_units;
  b = r / p.n_units;
}

__device__ __forceinline__ int chunk_kblocks(const Params& p, int i) {
  const int len = min(p.C, p.T - i * p.C);
  return (len + BKT - 1) / BKT;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_state_kernel(const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_z,
                    const __grid_constant__ CUtensorMap map_weff, const __grid_constant__ CUtensorMap map_wfin,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* chunk_done = bars + 2 * STAGES;  // [2]  MMA -> epilogue: chunk's MMAs finished
  uint64_t* snap_done = chunk_done + 2;      // [2]  epilogue -> MMA: accumulator read / initialised
  uint64_t* drain = snap_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pairs = (p.units + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&chunk_done[s], 1);
      mbar_init(&snap_done[s], 128);
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
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_z);
    bool ok = true;
    for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
      for (int j = 0; j < p.n_chunks && ok; ++j) {
        const int i = chunk_at(p, j);
        const int nkb = chunk_kblocks(p, i);
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          int b, mb, nb;
          decode_unit(p, u, b, mb, nb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, p.st, abort_flag, 0x201)) {
              ok = false;
              break;
            }
            uint8_t* sa = smem + p_stage * STAGE_BYTES;
            uint8_t* sb = sa + A_BYTES;
            mbar_arrive_expect_tx(&full[p_stage], STAGE_BYTES);
            const int tok = i * p.C + kb * BKT;
            tma_load_3d(sa, &map_v, &full[p_stage], mb * BMD, tok, b);
            tma_load_3d(sa + BKT * 128, &map_v, &full[p_stage], mb * BMD + 64, tok, b);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_3d(sb + j * (BKT * 128), &map_z, &full[p_stage], nb * BNF + j * 64, tok, b);
            ++p_issued;
            if (++p_stage == STAGES) {
              p_stage = 0;
              p_phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16(BMD, BNF, true, true);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t snap_waits[2] = {0, 0};
    bool ok = true;
    for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
      for (int j = 0; j < p.n_chunks && ok; ++j) {
        const int nkb = chunk_kblocks(p, chunk_at(p, j));
        for (int slot = 0; slot < 2 && ok; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          if (!wait_bounded(&snap_done[slot], snap_waits[slot] & 1u, p.st, abort_flag, 0x202)) {
            ok = false;
            break;
          }
          ++snap_waits[slot];
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(slot * BNF);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_bounded(&full[stage], phase, p.st, abort_flag, 0x203)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BKT / 16; ++kk) {
              // 16 tokens = 16 rows of 128 B; 64-wide blocks along d / d_ff are BKT*128 B apart
              const uint64_t adesc = sdesc_sw128(a_addr + kk * 2048, BKT * 128, 1024);
              const uint64_t bdesc = sdesc_sw128(b_addr + kk * 2048, BKT * 128, 1024);
              tc_mma_bf16(d_tmem, adesc, bdesc, idesc, 1u);
            }
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
  } else if (warp >= 2) {
    const int q = warp & 3;
    const int r_in_tile = q * 32 + lane;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_weff);
    tma_prefetch_desc(&map_wfin);
    uint32_t chunk_waits[2] = {0, 0};
    bool ok = true;
    for (int pr = blockIdx.x; pr < pairs && ok; pr += gridDim.x) {
      // initialise both accumulators with W_down0; the snapshot right after emits W_eff[0] = W_down0
      for (int slot = 0; slot < 2; ++slot) {
        const int u = 2 * pr + slot;
        if (u >= p.units) break;
        int b, mb, nb;
        decode_unit(p, u, b, mb, nb);
        const int row = mb * BMD + r_in_tile;
        const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * BNF);
#pragma unroll 1
        for (int c = 0; c < BNF / 32; ++c) {
          uint32_t r[32];
          load_init32(p, b, row, nb * BNF + c * 32, r);
          tmem_st32(t_row + c * 32, r);
        }
        tmem_st_wait();
        if (!p.skip_first && !p.no_snap)
          snapshot_bf16(out, t_row, &map_weff, nb * BNF, mb * BMD + q * 32, b * p.n_chunks + chunk_at(p, 0));
        tc_fence_before();
        mbar_arrive(&snap_done[slot]);
      }
      // after chunk i-1 completes the accumulator holds W_eff[i]; after the last, the final state
      for (int i = 1; i <= p.n_chunks && ok; ++i) {
        for (int slot = 0; slot < 2; ++slot) {
          const int u = 2 * pr + slot;
          if (u >= p.units) break;
          if (!wait_bounded(&chunk_done[slot], chunk_waits[slot] & 1u, p.st, abort_flag, 0x204)) {
            ok = false;
            break;
          }
          ++chunk_waits[slot];
          tc_fence_after();
          int b, mb, nb;
          decode_unit(p, u, b, mb, nb);
          const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * BNF);
          if (i < p.n_chunks) {
            if (!p.no_snap)
              snapshot_bf16(out, t_row, &map_weff, nb * BNF, mb * BMD + q * 32, b * p.n_chunks + chunk_at(p, i));
            tc_fence_before();
            mbar_arrive(&snap_done[slot]);
          } else {
            snapshot_f32(out, t_row, &map_wfin, nb * BNF, mb * BMD + q * 32, b);
            tc_fence_before();
          }
        }
      }
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

}  // namespace state
}  // namespace ipttt
