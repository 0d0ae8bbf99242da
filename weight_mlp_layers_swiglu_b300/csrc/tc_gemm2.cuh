// The persistent bf16 GEMM of tc_gemm.cuh on CTA pairs (clusters of two CTAs on two SMs).
//
// One tcgen05.mma.cta_group::2 computes a 256 x 256 x 16 product: each CTA of the pair holds
// its own 128 rows of A and one half (128 columns) of B in shared memory, and receives its own
// 128 rows of the accumulator in tensor memory.  Against the single-CTA 128 x 256 tile this
// halves the B operand each SM loads from L2 and reads from shared memory per FLOP (one third
// less operand traffic in all), which is what the tensor cores pay for at the board power limit.
//
//   warp 0      TMA producer of its CTA: 128 x 64 A and 128 x 64 B per stage (32 KB), 6 stages;
//               both CTAs' copies complete on the even CTA's `full` barrier.
//   warp 1      the even CTA's lane 0 issues the pair's MMAs and commits them to both CTAs'
//               barriers (multicast); warp 1 of each CTA allocates the pair's tensor memory.
//   warps 2-5   epilogue of each CTA for its own 128 rows, as in tc_gemm.cuh; the accumulator
//               buffer is released to the MMA issuer once both CTAs' epilogues have read it.
//
// Steps served (zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学"):
//   kSwiglu      §3.1 gated MLP; B half 0 = 128 rows of W_gate, half 1 = the same rows of W_up.
//   kTarget      §3.3 target projection (B = W_target, MN-major).
//   kApply       §3.2 Step 3 per chunk (requires C % 256 == 0 so a pair tile never spans chunks).
//   kSwigluSave  kSwiglu that also stores [A | U] through map_x ([rows][2][d_ff]), for the
//                backward pass.
//   kTwoSeg      the backward pass's A1 B1 + A2 B2 (B operands MN-major), per chunk like kApply,
//                with the optional SwiGLU-adjoint epilogue of tc_gemm.cuh (p.au).
#pragma once

#include "tc_gemm.cuh"

namespace ipttt {
namespace gemm2 {

using gemm::Kind;
using gemm::kApply;
using gemm::kSwiglu;
using gemm::kSwigluSave;
using gemm::kTarget;
using gemm::kTwoSeg;
using gemm::Params;

constexpr int BM = 128;        // rows per CTA (the pair tile has 256)
constexpr int PAIR_M = 256;
constexpr int BN = 256;        // accumulator columns (each CTA loads 128 of B's N)
constexpr int BN_HALF = 128;
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_HALF * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier block");

template <int KIND>
__device__ __forceinline__ bool pair_tile_active(const Params& p, int prob, int mt) {
  if (KIND == kApply || KIND == kTwoSeg) {
    const int i = prob % p.n_chunks;
    return i * p.C + mt * PAIR_M < p.T;
  }
  return true;
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    tc_gemm2_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                    const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_out,
                    const __grid_constant__ CUtensorMap map_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                    // [STAGES], used in the even CTA
  uint64_t* empty = bars + STAGES;          // [STAGES], each CTA's own ring
  uint64_t* acc_full = bars + 2 * STAGES;   // [2], each CTA
  uint64_t* acc_empty = acc_full + 2;       // [2], used in the even CTA
  uint64_t* drain = acc_empty + 2;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int total_tiles = p.problems * p.m_tiles * p.n_tiles;
  const int k_total = p.k_blocks + (KIND == kTwoSeg ? p.k_blocks2 : 0);

  if (p.zero_ptr != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.zero_count; i += blockDim.x) p.zero_ptr[i] = 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // one arrival per epilogue warp of both CTAs
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
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int p_stage = 0;
  uint32_t p_phase = 0;
  long p_issued = 0;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b0);
    if (KIND != kTarget) tma_prefetch_desc(&map_b1);
    if (KIND == kTwoSeg) tma_prefetch_desc(&map_x);
    for (int tile = pair; tile < total_tiles; tile += n_pairs) {
      int prob, mt, nt;
      gemm::decode_tile(p, tile, prob, mt, nt);
      if (!pair_tile_active<KIND>(p, prob, mt)) continue;
      const int m0 = mt * PAIR_M + (int)rank * BM;
      bool ok = true;
      for (int kb = 0; kb < k_total; ++kb) {
        if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, p.st, abort_flag, 0x501)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + p_stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        const uint32_t bar = cluster_addr(smem_u32(&full[p_stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[p_stage], 2 * STAGE_BYTES);
        const int k0 = kb * BK;
        if (KIND == kSwiglu || KIND == kSwigluSave) {
          tma_load_2d_pair(sa, &map_a, bar, k0, m0);
          tma_load_2d_pair(sb, rank == 0 ? &map_b0 : &map_b1, bar, k0, nt * BN_HALF);
        } else if (KIND == kTwoSeg) {
          const int b = prob / p.n_chunks;
          const int i = prob - b * p.n_chunks;
          const bool second = kb >= p.k_blocks;
          const int kk0 = second ? (kb - p.k_blocks) * BK : k0;
          const int bslice = p.b_per_problem ? prob : 0;
          tma_load_3d_pair(sa, second ? &map_b1 : &map_a, bar, kk0 + (second ? p.a2_koff : 0), i * p.C + m0, b);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma_load_3d_pair(sb + j * (BK * 128), second ? &map_x : &map_b0, bar,
                             nt * BN + (int)rank * BN_HALF + j * 64, kk0, bslice);
        } else if (KIND == kTarget) {
          tma_load_2d_pair(sa, &map_a, bar, k0, m0);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma_load_2d_pair(sb + j * (BK * 128), &map_b0, bar, nt * BN + (int)rank * BN_HALF + j * 64, k0);
        } else {
          const int b = prob / p.n_chunks;
          const int i = prob - b * p.n_chunks;
          tma_load_3d_pair(sa, &map_a, bar, k0, i * p.C + m0, b);
          if (i == 0 && p.first_from_w0)
            tma_load_2d_pair(sb, &map_b1, bar, k0, nt * BN + (int)rank * BN_HALF);
          else
            tma_load_3d_pair(sb, &map_b0, bar, k0, nt * BN + (int)rank * BN_HALF, prob);
        }
        ++p_issued;
        if (++p_stage == STAGES) {
          p_stage = 0;
          p_phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    constexpr bool b_mn = KIND == kTarget || KIND == kTwoSeg;
    constexpr uint32_t idesc = idesc_bf16(PAIR_M, BN, false, b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int tile = pair; tile < total_tiles; tile += n_pairs) {
      int prob, mt, nt;
      gemm::decode_tile(p, tile, prob, mt, nt);
      if (!pair_tile_active<KIND>(p, prob, mt)) continue;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded_cluster(&acc_empty[buf], (use & 1u) ^ 1u, p.st, abort_flag, 0x502)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
      bool ok = true;
      for (int kb = 0; kb < k_total; ++kb) {
        if (!wait_bounded(&full[stage], phase, p.st, abort_flag, 0x503)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t adesc = sdesc_sw128(a_addr + kk * 32, 16, 1024);
          const uint64_t bdesc = b_mn ? sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024)
                                      : sdesc_sw128(b_addr + kk * 32, 16, 1024);
          tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        tc_commit_pair(&empty[stage], 0x3);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_pair(&acc_full[buf], 0x3);
      ++it;
    }
  } else if (warp >= 2) {
    const int q = warp & 3;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_out);
    int it = 0;
    for (int tile = pair; tile < total_tiles; tile += n_pairs) {
      int prob, mt, nt;
      gemm::decode_tile(p, tile, prob, mt, nt);
      if (!pair_tile_active<KIND>(p, prob, mt)) continue;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded(&acc_full[buf], use & 1u, p.st, abort_flag, 0x504)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      const int row0 = mt * PAIR_M + (int)rank * BM + q * 32;
      if (KIND == kSwiglu || KIND == kSwigluSave) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t row[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t g[32], u[32];
            tmem_ld32(t_row + h * 64 + c * 32, g);
            tmem_ld32(t_row + BN_HALF + h * 64 + c * 32, u);
            tmem_ld_wait(g);
            tmem_ld_wait(u);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float a0 = __uint_as_float(g[2 * e]), a1 = __uint_as_float(g[2 * e + 1]);
              const float z0 = silu_bf16ep(a0) * __uint_as_float(u[2 * e]);
              const float z1 = silu_bf16ep(a1) * __uint_as_float(u[2 * e + 1]);
              row[c * 16 + e] = pack_bf16x2(z0, z1);
            }
          }
          out.put(row, &map_out, nt * BN_HALF + h * 64, row0);
          if (KIND == kSwigluSave) {  // the gate and up pre-activations: map_x is [rows][2][d_ff]
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
              uint32_t pre[32];
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                uint32_t g[32];
                tmem_ld32(t_row + part * BN_HALF + h * 64 + c * 32, g);
                tmem_ld_wait(g);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  pre[c * 16 + e] = pack_bf16x2(__uint_as_float(g[2 * e]), __uint_as_float(g[2 * e + 1]));
              }
              out.put(pre, &map_x, nt * BN_HALF + h * 64, part, row0);
            }
          }
        }
      } else if (KIND == kTwoSeg && p.au != nullptr) {
        // dZ stays in registers: the SwiGLU adjoints overwrite [A | U] in place (tc_gemm.cuh)
        const int bq = prob / p.n_chunks;
        const int i = prob - bq * p.n_chunks;
        const int tok = i * p.C + row0 + lane;
        __nv_bfloat16* au_row = p.au + ((int64_t)bq * p.T + tok) * (2 * (int64_t)p.au_f);
#pragma unroll 1
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t lo[32], hi[32];
          tmem_ld32(t_row + h * 64, lo);
          tmem_ld32(t_row + h * 64 + 32, hi);
          tmem_ld_wait(lo);
          tmem_ld_wait(hi);
          const int n0 = nt * BN + h * 64;
          if (tok < p.T) gemm::swiglu_adjoint_row64(lo, hi, au_row, n0, p.au_f);
        }
      } else {
#pragma unroll 1
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t a[32], b[32], row[32];
          tmem_ld32(t_row + h * 64, a);
          tmem_ld32(t_row + h * 64 + 32, b);
          tmem_ld_wait(a);
          tmem_ld_wait(b);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            row[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
            row[16 + e] = pack_bf16x2(__uint_as_float(b[2 * e]) * p.scale, __uint_as_float(b[2 * e + 1]) * p.scale);
          }
          if (KIND == kApply || KIND == kTwoSeg) {
            const int bq = prob / p.n_chunks;
            const int i = prob - bq * p.n_chunks;
            out.put(row, &map_out, nt * BN + h * 64, i * p.C + row0, bq);
          } else {
            out.put(row, &map_out, nt * BN + h * 64, row0);
          }
        }
      }
      // release the accumulator buffer to the even CTA's MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&acc_empty[buf]), 0));
      ++it;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (*abort_flag) {
    // Drain (bounded): the pair's MMAs (even CTA) and the copies that complete on its barriers.
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
  cluster_sync();  // neither CTA leaves while the other may still signal it or use its operands
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace gemm2
}  // namespace ipttt
