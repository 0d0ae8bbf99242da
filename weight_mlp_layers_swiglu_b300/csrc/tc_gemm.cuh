// Persistent, warp-specialised bf16 GEMM on the 5th-generation tensor cores.
//
// One CTA per SM (192 threads):
//   warp 0      TMA producer: streams 128x64 A tiles and 256x64 B tiles into a
//               4-stage shared-memory ring (128-byte swizzle).
//   warp 1      MMA issuer (one thread): tcgen05.mma 128x256x16 into one of two
//               TMEM accumulators (2 x 256 fp32 columns), so the epilogue of one
//               tile overlaps the main loop of the next.
//   warps 2-5   epilogue: tcgen05.ld the accumulator (one TMEM lane = one output
//               row per thread), apply the step's epilogue, stage 32 x 64 bf16 boxes
//               in swizzled shared memory and write them with TMA tensor stores.
//
// The same kernel serves three steps of the layer (zhichai.net "In-Place TTT：给LLM装上
// "临时记忆插槽"，让它边读边学"):
//   Swiglu  §3.1 gated MLP:   Z = SiLU(H W_gate^T) * (H W_up^T).  The B tile holds 128
//           rows of W_gate and the same 128 rows of W_up, so one N=256 MMA produces
//           both halves and the epilogue fuses SiLU and the product.
//   Target  §3.3 target:      V = scale * (Y W_target), Y = causal conv of X0 (computed
//           by the conv kernel).  W_target is [d_in, d_out], so B is MN-major.
//   Apply   §3.2 Step 3:      O_i = Z_i W_eff[i]^T for every chunk i of every sequence;
//           the problem index selects the chunk's rows of Z and its slice of the
//           W_eff stack (3-D tensor maps); chunk 0 may read W_down0 directly, since
//           W_eff[0] = W_down0.
#pragma once

#include "ptx.cuh"

namespace ipttt {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int BAR_BYTES = 256;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;  // two staging boxes per epilogue warp
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + BAR_BYTES;

// kSwigluSave: kSwiglu that also writes the gate and up pre-activations (for the backward pass).
// kTwoSeg: C = A1 B1 + A2 B2 over two K segments, B operands MN-major ([K, N] row-major), per
// chunk like kApply (the backward pass's dZ_i = dO_i W_i + V_i R_i and dH = dA W_gate + dU W_up).
enum Kind : int { kSwiglu = 0, kTarget = 1, kApply = 2, kSwigluSave = 3, kTwoSeg = 4 };

struct Params {
  int m_tiles, n_tiles, k_blocks;  // per problem
  int problems;                    // Apply: B * n_chunks, else 1
  int group_m;                     // rasterisation: m-tiles per group
  float scale;
  int T, C, n_chunks;  // Apply only
  int first_from_w0;   // Apply: chunk 0 of each sequence reads W_down0 (map_b1) instead of the stack
  uint32_t* zero_ptr;  // optional: CTA 0 clears zero_count words here (counters of a later kernel)
  int zero_count;
  int k_blocks2;       // kTwoSeg: k-blocks of the second segment (the first has k_blocks)
  int a2_koff;         // kTwoSeg: column offset of the second segment within its A map
  int b_per_problem;   // kTwoSeg: 1 = each problem (chunk) has its own B slice, 0 = one shared B
  // kTwoSeg, optional: the result is dZ and is not stored; instead the SwiGLU adjoints overwrite
  // the saved pre-activations au = [A | U] ([B*T, 2*au_f] bf16, the output's rows):
  // dA = dZ U s (1 + A (1 - s)), dU = dZ A s with s = sigmoid(A)
  __nv_bfloat16* au;
  int au_f;
  DevStatus st;
};

__device__ __forceinline__ void decode_tile(const Params& p, int tile, int& prob, int& mt, int& nt) {
  const int per_prob = p.m_tiles * p.n_tiles;
  prob = tile / per_prob;
  const int r = tile - prob * per_prob;
  const int group = p.group_m * p.n_tiles;
  const int g = r / group;
  const int rr = r - g * group;
  const int gm = min(p.group_m, p.m_tiles - g * p.group_m);
  mt = g * p.group_m + rr % gm;
  nt = rr / gm;
}

template <int KIND>
__device__ __forceinline__ bool tile_active(const Params& p, int prob, int mt) {
  if (KIND == kApply || KIND == kTwoSeg) {
    const int i = prob % p.n_chunks;
    return i * p.C + mt * BM < p.T;
  }
  return true;
}

// The SwiGLU adjoint for 64 columns n0.. of one token's row: dZ (fp32) in lo/hi, A and U read
// from au_row = [A | U] (bf16, au_f columns each) and overwritten with dA and dU:
// dA = dZ U s (1 + A (1 - s)), dU = dZ A s, s = sigmoid(A).  d_ff % 8 == 0, so each group of 8
// columns lies wholly inside or outside the row.
__device__ __forceinline__ void swiglu_adjoint_row64(const uint32_t (&lo)[32], const uint32_t (&hi)[32],
                                                     __nv_bfloat16* au_row, int n0, int au_f) {
  uint4 av[8], uv[8];
#pragma unroll
  for (int v = 0; v < 8; ++v)
    if (n0 + v * 8 < au_f) {
      av[v] = *reinterpret_cast<const uint4*>(au_row + n0 + v * 8);
      uv[v] = *reinterpret_cast<const uint4*>(au_row + au_f + n0 + v * 8);
    }
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    if (n0 + v * 8 >= au_f) continue;
    const uint32_t* aw = reinterpret_cast<const uint32_t*>(&av[v]);
    const uint32_t* uw = reinterpret_cast<const uint32_t*>(&uv[v]);
    uint4 da, du;
    uint32_t* daw = reinterpret_cast<uint32_t*>(&da);
    uint32_t* duw = reinterpret_cast<uint32_t*>(&du);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = (v & 3) * 8 + 2 * e;
      const float z0 = __uint_as_float(v < 4 ? lo[j] : hi[j]);
      const float z1 = __uint_as_float(v < 4 ? lo[j + 1] : hi[j + 1]);
      const float A0 = bf16_lo(aw[e]), A1 = bf16_hi(aw[e]);
      const float U0 = bf16_lo(uw[e]), U1 = bf16_hi(uw[e]);
      const float s0 = sigmoid_bf16ep(A0), s1 = sigmoid_bf16ep(A1);
      daw[e] = pack_bf16x2(z0 * U0 * s0 * (1.0f + A0 * (1.0f - s0)), z1 * U1 * s1 * (1.0f + A1 * (1.0f - s1)));
      duw[e] = pack_bf16x2(z0 * A0 * s0, z1 * A1 * s1);
    }
    *reinterpret_cast<uint4*>(au_row + n0 + v * 8) = da;
    *reinterpret_cast<uint4*>(au_row + au_f + n0 + v * 8) = du;
  }
}

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_out,
                   const __grid_constant__ CUtensorMap map_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                // [STAGES]
  uint64_t* empty = bars + STAGES;      // [STAGES]
  uint64_t* acc_full = bars + 2 * STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* drain = acc_empty + 2;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
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
      mbar_init(&acc_empty[b], 128);
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

  // producer state, kept at function scope for the drain after an abort
  int p_stage = 0;
  uint32_t p_phase = 0;
  long p_issued = 0;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b0);
    if (KIND != kTarget) tma_prefetch_desc(&map_b1);
    if (KIND == kTwoSeg) tma_prefetch_desc(&map_x);
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int prob, mt, nt;
      decode_tile(p, tile, prob, mt, nt);
      if (!tile_active<KIND>(p, prob, mt)) continue;
      bool ok = true;
      for (int kb = 0; kb < k_total; ++kb) {
        if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, p.st, abort_flag, 0x101)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + p_stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        mbar_arrive_expect_tx(&full[p_stage], STAGE_BYTES);
        const int k0 = kb * BK;
        if (KIND == kSwiglu || KIND == kSwigluSave) {
          tma_load_2d(sa, &map_a, &full[p_stage], k0, mt * BM);
          tma_load_2d(sb, &map_b0, &full[p_stage], k0, nt * 128);
          tma_load_2d(sb + B_BYTES / 2, &map_b1, &full[p_stage], k0, nt * 128);
        } else if (KIND == kTwoSeg) {
          const int b = prob / p.n_chunks;
          const int i = prob - b * p.n_chunks;
          const bool second = kb >= p.k_blocks;
          const int kk0 = second ? (kb - p.k_blocks) * BK : k0;
          const int bslice = p.b_per_problem ? prob : 0;
          tma_load_3d(sa, second ? &map_b1 : &map_a, &full[p_stage], kk0 + (second ? p.a2_koff : 0),
                      i * p.C + mt * BM, b);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tma_load_3d(sb + j * (BK * 128), second ? &map_x : &map_b0, &full[p_stage], nt * BN + j * 64, kk0,
                        bslice);
        } else if (KIND == kTarget) {
          tma_load_2d(sa, &map_a, &full[p_stage], k0, mt * BM);
#pragma unroll
          for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * (BK * 128), &map_b0, &full[p_stage], nt * BN + j * 64, k0);
        } else {
          const int b = prob / p.n_chunks;
          const int i = prob - b * p.n_chunks;
          tma_load_3d(sa, &map_a, &full[p_stage], k0, i * p.C + mt * BM, b);
          if (i == 0 && p.first_from_w0)
            tma_load_2d(sb, &map_b1, &full[p_stage], k0, nt * BN);
          else
            tma_load_3d(sb, &map_b0, &full[p_stage], k0, nt * BN, prob);
        }
        ++p_issued;
        if (++p_stage == STAGES) {
          p_stage = 0;
          p_phase ^= 1u;
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1 && lane == 0) {
    constexpr bool b_mn = KIND == kTarget || KIND == kTwoSeg;
    constexpr uint32_t idesc = idesc_bf16(BM, BN, false, b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int prob, mt, nt;
      decode_tile(p, tile, prob, mt, nt);
      if (!tile_active<KIND>(p, prob, mt)) continue;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded(&acc_empty[buf], (use & 1u) ^ 1u, p.st, abort_flag, 0x102)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
      bool ok = true;
      for (int kb = 0; kb < k_total; ++kb) {
        if (!wait_bounded(&full[stage], phase, p.st, abort_flag, 0x103)) {
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
          tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
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
  } else if (warp >= 2) {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_out);
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int prob, mt, nt;
      decode_tile(p, tile, prob, mt, nt);
      if (!tile_active<KIND>(p, prob, mt)) continue;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded(&acc_full[buf], use & 1u, p.st, abort_flag, 0x104)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      if (KIND == kSwiglu || KIND == kSwigluSave) {
        // 128 output columns: two boxes of 64, each from 64 gate and 64 up accumulator columns
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t row[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t g[32], u[32];
            tmem_ld32(t_row + h * 64 + c * 32, g);
            tmem_ld32(t_row + 128 + h * 64 + c * 32, u);
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
          out.put(row, &map_out, nt * 128 + h * 64, mt * BM + q * 32);
          if (KIND == kSwigluSave) {  // the gate and up pre-activations: map_x is [rows][2][d_ff]
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
              uint32_t pre[32];
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                uint32_t g[32];
                tmem_ld32(t_row + part * 128 + h * 64 + c * 32, g);
                tmem_ld_wait(g);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  pre[c * 16 + e] = pack_bf16x2(__uint_as_float(g[2 * e]), __uint_as_float(g[2 * e + 1]));
              }
              out.put(pre, &map_x, nt * 128 + h * 64, part, mt * BM + q * 32);
            }
          }
        }
      } else if (KIND == kTwoSeg && p.au != nullptr) {
        const int bq = prob / p.n_chunks;
        const int i = prob - bq * p.n_chunks;
        const int tok = i * p.C + mt * BM + q * 32 + lane;
        __nv_bfloat16* au_row = p.au + ((int64_t)bq * p.T + tok) * (2 * (int64_t)p.au_f);
#pragma unroll 1
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t lo[32], hi[32];
          tmem_ld32(t_row + h * 64, lo);
          tmem_ld32(t_row + h * 64 + 32, hi);
          tmem_ld_wait(lo);
          tmem_ld_wait(hi);
          const int n0 = nt * BN + h * 64;
          if (tok < p.T) swiglu_adjoint_row64(lo, hi, au_row, n0, p.au_f);
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
            out.put(row, &map_out, nt * BN + h * 64, i * p.C + mt * BM + q * 32, bq);
          } else {
            out.put(row, &map_out, nt * BN + h * 64, mt * BM + q * 32);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      ++it;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncthreads();
  if (*abort_flag) {
    // Drain: wait (bounded) for this CTA's own MMAs and TMA copies still in flight.
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

}  // namespace gemm
}  // namespace ipttt
