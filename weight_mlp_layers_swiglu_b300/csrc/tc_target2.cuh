// Step (2) of the layer as one kernel on CTA pairs: V = scale * (CausalConv1D(X0) W_target)
// (zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学", §3.3, the target equation).
//
// The GEMM is the pair GEMM of tc_gemm2.cuh (kind kTarget: 256 x 256 pair tiles, W_target
// MN-major), but its A operand, the conv output Y, is never stored: four extra warps per CTA
// form each 128 x 64 A tile from a window of X0 rows and write it straight into the stage, in
// the 128-byte-swizzled layout the MMA reads.  The TMA producer loads, per k-block, the
// 64-channel X0 window of the CTA's 128 tokens (7 rows before them and 1 after, zero outside
// the sequence), and the 64 channels' conv taps, into a small ring of its own.
//
//   warp 0      TMA producer of W_target half-tiles into the stage ring (both CTAs' copies
//               complete on the even CTA's `full`).
//   warp 14     TMA producer of the X0 windows and the taps (a bulk copy) into the CTA's own
//               X0 ring (a thread of its own, so that neither stream waits for the other's slots).
//   warp 1      the even CTA's lane 0 issues the pair's MMAs once `full` (B landed) and
//               `a_ready` (both CTAs' A written) complete; warp 1 of each CTA allocates TMEM.
//   warps 2-5   epilogue, as in tc_gemm2.cuh: V = scale * acc in bf16 through TMA stores.
//   warps 6-13  conv, two groups of four taking alternate k-blocks (so that one group's load,
//               wait and fence latencies overlap the other's work): in its group, thread
//               (cg, rg) forms channels 8cg..8cg+7 of tile rows 8rg..8rg+7:
//               Y[t, c] = sum_{s<K} conv_w[c, s] X0[t + shift - (K-1) + s, c], an fp32 fma chain
//               over s from zero (the order of simt.cuh's causal_conv_kernel, two channels per
//               fma.rn.f32x2, each lane an IEEE fma, so Y, and hence V, is the same bf16 value
//               bit for bit), rounded to bf16 into the A stage, then fence.proxy.async and one
//               arrival per warp on the even CTA's a_ready.
//
// Rows of a sequence before its first token are zero, or the caller's halo rows (a resumed
// call); rows after its last token are zero (the shifted window's last target).  Tiles never
// span two sequences: the tile grid is (sequence, 256-token block, 256-column block).
#pragma once

#include "tc_gemm.cuh"

namespace ipttt {
namespace tconv2 {

constexpr int BM = 128;  // tokens per CTA (the pair tile has 256)
constexpr int PAIR_M = 256;
constexpr int BN = 256;
constexpr int BN_HALF = 128;
constexpr int BK = 64;  // channels per k-block
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_HALF * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int XHALO = 7;                  // X0 rows loaded before a tile's first token (K - 1 <= 7)
constexpr int XROWS = BM + XHALO + 1;     // ... and one after its last (the shifted window)
constexpr int XWIN_BYTES = XROWS * BK * 2;         // 64 channels x 136 rows, unswizzled
constexpr int TAP_BYTES = BK * 8 * 2;               // the k-block's conv taps: 64 channels x K <= 8
constexpr int X_BYTES = XWIN_BYTES + TAP_BYTES;     // one X0 slot: window, then taps
constexpr int XSLOTS = 3;
constexpr int CONV_WARP0 = 6;
constexpr int CONV_WARPS = 8;   // two groups of four, taking alternate k-blocks
constexpr int CONV_GROUP = 4;   // warps per group: 128 threads, one per (8 channels, 8 rows) block
constexpr int CONV_ROWS = BM / (CONV_GROUP * 4);  // tile rows per conv thread (8 channels each)
constexpr int XLOAD_WARP = CONV_WARP0 + CONV_WARPS;  // issues the X0 windows, apart from the W_target stream
constexpr int NUM_THREADS = 32 * (XLOAD_WARP + 1);
constexpr uint32_t TMEM_COLS = 512;
constexpr int OUT_BYTES = 4 * 2 * OUT_BOX_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + XSLOTS * X_BYTES + OUT_BYTES + 1024 + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(X_BYTES % 1024 == 0, "X0 slots keep the stage alignment");
static_assert((3 * STAGES + 2 * XSLOTS + 5) * 8 + 8 <= BAR_BYTES, "barrier block");

struct Params {
  int B, T, d;
  int m_tiles, n_tiles, k_blocks, group_m;  // m_tiles: 256-token blocks per sequence
  int shift;                                // 1: the window ends at the next token
  float scale;
  const __nv_bfloat16* conv_w;  // [d, K]
  const __nv_bfloat16* halo;    // optional [B, K-1, d]: the rows before each sequence's first token
  uint32_t* zero_ptr;           // optional: CTA 0 clears zero_count words (counters of a later kernel)
  int zero_count;
  DevStatus st;
};

// tile -> (sequence b, token block mt, column block nt), in groups of group_m token blocks
__device__ __forceinline__ void decode_tile(const Params& p, int tile, int& b, int& mt, int& nt) {
  const int per_seq = p.m_tiles * p.n_tiles;
  b = tile / per_seq;
  const int r = tile - b * per_seq;
  const int group = p.group_m * p.n_tiles;
  const int g = r / group;
  const int rr = r - g * group;
  const int gm = min(p.group_m, p.m_tiles - g * p.group_m);
  mt = g * p.group_m + rr % gm;
  nt = rr / gm;
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint4& v) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
}

// Two fp32 values in one 64-bit register (element 0 in the low half) and the packed fused
// multiply-add of sm_100+: each half is an IEEE fma rounded to nearest, as fmaf.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// The bf16 pair in one 32-bit word as two fp32 values (widening is exact).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) { return f2_pack(bf16_lo(w), bf16_hi(w)); }

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  v[0] = bf16_lo(w.x), v[1] = bf16_hi(w.x), v[2] = bf16_lo(w.y), v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z), v[5] = bf16_hi(w.z), v[6] = bf16_lo(w.w), v[7] = bf16_hi(w.w);
}

template <int K>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    tc_target_conv2_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_b,
                           const __grid_constant__ CUtensorMap map_out, const Params p) {
  static_assert(K >= 1 && K - 1 <= XHALO, "conv kernel size");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xring = smem + STAGES * STAGE_BYTES;
  uint8_t* out_stage = xring + XSLOTS * X_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + OUT_BYTES);
  uint64_t* full = bars;                   // [STAGES] even CTA: W_target halves landed (tx)
  uint64_t* a_ready = full + STAGES;       // [STAGES] even CTA: both CTAs' conv warps wrote their A tiles
  uint64_t* empty = a_ready + STAGES;      // [STAGES] each CTA: the MMAs have read the stage
  uint64_t* x_full = empty + STAGES;       // [XSLOTS] each CTA: X0 window landed (tx)
  uint64_t* x_empty = x_full + XSLOTS;     // [XSLOTS] each CTA: its conv warps have read it
  uint64_t* acc_full = x_empty + XSLOTS;   // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2] even CTA
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int total_tiles = p.B * p.m_tiles * p.n_tiles;

  if (p.zero_ptr != nullptr && blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.zero_count; i += blockDim.x) p.zero_ptr[i] = 0u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&a_ready[s], 2 * CONV_GROUP);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < XSLOTS; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], CONV_GROUP);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], 8);
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
  int x_slot = 0;
  uint32_t x_phase = 0;
  long x_issued = 0;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&map_b);
    bool ok = true;
    for (int tile = pair; tile < total_tiles && ok; tile += n_pairs) {
      int b, mt, nt;
      decode_tile(p, tile, b, mt, nt);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!wait_bounded(&empty[p_stage], p_phase ^ 1u, p.st, abort_flag, 0x802)) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + p_stage * STAGE_BYTES + A_BYTES;
        const uint32_t bar = cluster_addr(smem_u32(&full[p_stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[p_stage], 2 * B_BYTES);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_2d_pair(sb + j * (BK * 128), &map_b, bar, nt * BN + (int)rank * BN_HALF + j * 64, kb * BK);
        ++p_issued;
        if (++p_stage == STAGES) {
          p_stage = 0;
          p_phase ^= 1u;
        }
      }
    }
  } else if (warp == XLOAD_WARP && lane == 0) {
    // ------------------------------------------------------------------ X0 window producer
    tma_prefetch_desc(&map_x);
    bool ok = true;
    for (int tile = pair; tile < total_tiles && ok; tile += n_pairs) {
      int b, mt, nt;
      decode_tile(p, tile, b, mt, nt);
      const int t0 = mt * PAIR_M + (int)rank * BM;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!wait_bounded(&x_empty[x_slot], x_phase ^ 1u, p.st, abort_flag, 0x801)) {
          ok = false;
          break;
        }
        // taps of channels kb*64 .. : min(64, d - kb*64) rows of K bf16 (a multiple of 16 bytes)
        const uint32_t tap_bytes = (uint32_t)(min(BK, p.d - kb * BK) * K * 2);
        uint8_t* slot = xring + x_slot * X_BYTES;
        mbar_arrive_expect_tx(&x_full[x_slot], XWIN_BYTES + tap_bytes);
        tma_load_3d(slot, &map_x, &x_full[x_slot], kb * BK, t0 - XHALO, b);
        bulk_load(slot + XWIN_BYTES, p.conv_w + (int64_t)kb * BK * K, tap_bytes, &x_full[x_slot]);
        ++x_issued;
        if (++x_slot == XSLOTS) {
          x_slot = 0;
          x_phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    constexpr uint32_t idesc = idesc_bf16(PAIR_M, BN, false, true);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int tile = pair; tile < total_tiles && ok; tile += n_pairs) {
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded_cluster(&acc_empty[buf], (use & 1u) ^ 1u, p.st, abort_flag, 0x811)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        if (!wait_bounded(&full[stage], phase, p.st, abort_flag, 0x812) ||
            !wait_bounded_cluster(&a_ready[stage], phase, p.st, abort_flag, 0x813)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_bf16_pair(d_tmem, sdesc_sw128(a_addr + kk * 32, 16, 1024),
                           sdesc_sw128(b_addr + kk * 2048, BK * 128, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
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
  } else if (warp >= 2 && warp < CONV_WARP0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;
    OutStager out{out_stage + (warp - 2) * 2 * OUT_BOX_BYTES, 0u, lane};
    tma_prefetch_desc(&map_out);
    int it = 0;
    for (int tile = pair; tile < total_tiles; tile += n_pairs) {
      int b, mt, nt;
      decode_tile(p, tile, b, mt, nt);
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!wait_bounded(&acc_full[buf], use & 1u, p.st, abort_flag, 0x821)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      const int row0 = mt * PAIR_M + (int)rank * BM + q * 32;
#pragma unroll 1
      for (int h = 0; h < BN / 64; ++h) {
        uint32_t row[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 32 columns at a time keeps the registers low
          uint32_t a[32];
          tmem_ld32(t_row + h * 64 + half * 32, a);
          tmem_ld_wait(a);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            row[half * 16 + e] =
                pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
        }
        out.put(row, &map_out, nt * BN + h * 64, row0, b);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(&acc_empty[buf]), 0));
      ++it;
    }
    if (lane == 0) bulk_wait_all();
  } else if (warp >= CONV_WARP0 && warp < XLOAD_WARP) {
    // ------------------------------------------------------------------ conv warps
    // group g takes the k-blocks n = g, g+2, g+4, ... of this CTA's k-block sequence (n counts
    // the k-blocks of all its tiles in order), which fixes their stage and X0 slot
    const int grp = (warp - CONV_WARP0) / CONV_GROUP;
    const int cw = (warp - CONV_WARP0) % CONV_GROUP;
    const int cg = lane & 7;                              // channels 8cg .. 8cg+7 of the k-block
    const int r0 = (cw * 4 + (lane >> 3)) * CONV_ROWS;    // tile rows r0 .. r0+CONV_ROWS-1
    const uint32_t lead_ready = cluster_addr(smem_u32(a_ready), 0);
    const int my_tiles = pair < total_tiles ? (total_tiles - 1 - pair) / n_pairs + 1 : 0;
    const long n_end = (long)my_tiles * p.k_blocks;
    for (long n = grp; n < n_end; n += 2) {
      const int tile = pair + (int)(n / p.k_blocks) * n_pairs;
      const int kb = (int)(n % p.k_blocks);
      int b, mt, nt;
      decode_tile(p, tile, b, mt, nt);
      const int t0 = mt * PAIR_M + (int)rank * BM;
      const int c0 = kb * BK + cg * 8;
      const int xs = (int)(n % XSLOTS);
      const int stage = (int)(n % STAGES);
      if (!wait_bounded(&x_full[xs], (uint32_t)((n / XSLOTS) & 1), p.st, abort_flag, 0x831) ||
          !wait_bounded(&empty[stage], (uint32_t)(((n / STAGES) & 1) ^ 1), p.st, abort_flag, 0x832))
        break;
      // the taps of this thread's 8 channels as channel pairs, w2[e2][s] = (w[2e2][s], w[2e2+1][s]):
      // 8K contiguous bf16 at 16K bytes per channel group in the slot's tap block (zero past d)
      uint64_t w2[4][K];
      {
        const uint4* tp = reinterpret_cast<const uint4*>(xring + xs * X_BYTES + XWIN_BYTES) + cg * K;
        float w[8][K];
#pragma unroll
        for (int v = 0; v < K; ++v) {
          float u[8];
          unpack8(c0 < p.d ? tp[v] : make_uint4(0u, 0u, 0u, 0u), u);
#pragma unroll
          for (int m = 0; m < 8; ++m) w[(v * 8 + m) / K][(v * 8 + m) % K] = u[m];
        }
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
#pragma unroll
          for (int s2 = 0; s2 < K; ++s2) w2[e2][s2] = f2_pack(w[2 * e2][s2], w[2 * e2 + 1][s2]);
      }
      const uint4* xrow = reinterpret_cast<const uint4*>(xring + xs * X_BYTES) + cg;  // 8 uint4 per row
      // rows of the sequence before its first token come from the caller's halo (first tile only)
      const bool use_halo = p.halo != nullptr && t0 == 0;
      auto load_row = [&](int j, uint64_t (&v)[4]) {
        const int tr = r0 + j - (K - 1) + p.shift;  // tile-relative input row, >= -(K-1)
        uint4 q;
        if (use_halo && tr < 0)
          q = c0 < p.d ? *reinterpret_cast<const uint4*>(p.halo + ((int64_t)b * (K - 1) + (K - 1) + tr) * p.d + c0)
                       : make_uint4(0u, 0u, 0u, 0u);
        else
          q = xrow[(tr + XHALO) * 8];
        v[0] = bf16x2_to_f2(q.x);
        v[1] = bf16x2_to_f2(q.y);
        v[2] = bf16x2_to_f2(q.z);
        v[3] = bf16x2_to_f2(q.w);
      };
      const uint32_t abase = smem_u32(smem + stage * STAGE_BYTES);
      uint64_t win[K][4];  // the last K input rows
#pragma unroll
      for (int j = 0; j < K - 1; ++j) load_row(j, win[j]);
#pragma unroll
      for (int j = 0; j < CONV_ROWS; ++j) {
        load_row(j + K - 1, win[K - 1]);
        uint32_t packed[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          uint64_t acc = 0ull;  // (+0, +0)
#pragma unroll
          for (int s2 = 0; s2 < K; ++s2) acc = ffma2(w2[e2][s2], win[s2][e2], acc);
          float lo, hi;
          f2_unpack(acc, lo, hi);
          packed[e2] = pack_bf16x2(lo, hi);
        }
        const int r = r0 + j;
        st_shared_v4(abase + (uint32_t)(r * 128 + ((cg ^ (r & 7)) << 4)), packed[0], packed[1], packed[2], packed[3]);
#pragma unroll
        for (int s2 = 0; s2 < K - 1; ++s2)
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) win[s2][e2] = win[s2 + 1][e2];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&x_empty[xs]);
        mbar_arrive_cluster(lead_ready + 8u * stage);
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 1 && lane == 0 && rank == 0) {
      tc_commit_pair(drain, 0x1);
      drain_wait(drain, 0, 50000000ull);
    }
    if (warp == 0 && lane == 0 && rank == 0)
      for (long j = p_issued - 1; j >= 0 && j >= p_issued - STAGES; --j)
        drain_wait(&full[j % STAGES], (uint32_t)((j / STAGES) & 1), 50000000ull);
    if (warp == XLOAD_WARP && lane == 0)
      for (long j = x_issued - 1; j >= 0 && j >= x_issued - XSLOTS; --j)
        drain_wait(&x_full[j % XSLOTS], (uint32_t)((j / XSLOTS) & 1), 50000000ull);
    __syncthreads();
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace tconv2
}  // namespace ipttt
