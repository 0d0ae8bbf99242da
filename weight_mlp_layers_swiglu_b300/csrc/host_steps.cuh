// Step launchers: one kernel launch per step of the layer, no argument validation.
// Part of the host side of libipttt (one translation unit: ipttt.cu includes the host_*.cuh
// files in order).  Everything here is internal; the C ABI is at the end of ipttt.cu.
#pragma once

#include "host_context.cuh"

namespace {

// ------------------------------------------------------------------ step launchers (no validation)

// allow_pairs = false keeps the single-CTA tiles (bit-identical results); a few rows then take
// d_ff/128 tiles in one wave over the SMs instead of two waves of pair tiles.
ipttt_status run_swiglu(ipttt_ctx* ctx, const void* H, const void* Wg, const void* Wu, int64_t rows, int64_t d,
                        int64_t f, ipttt_dtype dt, void* Z, bool allow_pairs = true) {
  if (rows == 0) return IPTTT_OK;
  if (dt == IPTTT_BF16) {
    CUtensorMap ma, mb0, mb1, mo;
    if (!map_2d(ctx, &ma, H, rows, d, 64, 128) || !map_2d(ctx, &mb0, Wg, f, d, 64, 128) ||
        !map_2d(ctx, &mb1, Wu, f, d, 64, 128) || !map_2d(ctx, &mo, Z, rows, f, 64, 32))
      return IPTTT_ERR_CUDA;
    gemm::Params p{};
    const bool pairs = allow_pairs && use_pairs(ctx);
    p.m_tiles = ceil_div(rows, pairs ? gemm2::PAIR_M : gemm::BM);
    p.n_tiles = ceil_div(f, 128);
    p.k_blocks = ceil_div(d, gemm::BK);
    p.problems = 1;
    // 32 pair tiles (8192 rows) share each weight tile: the weights are read from DRAM once per
    // 8192 rows (measured at the 4B shape under the power limit: 1309 TFLOP/s with groups of 8,
    // 1341 with 16, 1352 with 32, 1210 with 64, whose H rows no longer stay in L2)
    p.group_m = pairs ? 32 : 16;
    p.scale = 1.f;
    p.st = dev_status(ctx);
    const int tiles = p.m_tiles * p.n_tiles;
    if (pairs) {
      gemm2::tc_gemm2_kernel<gemm::kSwiglu><<<pair_grid(ctx, tiles), gemm2::NUM_THREADS, gemm2::SMEM_BYTES,
                                             ctx->stream>>>(ma, mb0, mb1, mo, mo, p);
    } else {
      const int grid = tiles < ctx->sm_count ? tiles : ctx->sm_count;
      gemm::tc_gemm_kernel<gemm::kSwiglu><<<grid, gemm::NUM_THREADS, gemm::SMEM_BYTES, ctx->stream>>>(ma, mb0, mb1,
                                                                                                      mo, mo, p);
    }
  } else {
    simt::SgemmParams p{};
    p.A = static_cast<const float*>(H);
    p.B = static_cast<const float*>(Wg);
    p.B2 = static_cast<const float*>(Wu);
    p.Cm = static_cast<float*>(Z);
    p.M = (int)rows;
    p.N = (int)f;
    p.K = (int)d;
    p.a_sm = d, p.a_sk = 1, p.b_sk = 1, p.b_sn = d, p.c_sm = f;
    p.scale = 1.f;
    dim3 grid(ceil_div(f, simt::SG_BN), ceil_div(rows, simt::SG_BM), 1);
    simt::sgemm_kernel<true><<<grid, 256, 0, ctx->stream>>>(p);
  }
  return check_launch(ctx, "swiglu launch");
}

template <typename E>
void launch_conv(ipttt_ctx* ctx, dim3 grid, dim3 block, const void* X0, const void* cw, void* Y, int T_len, int d,
                 int k, const void* halo, int shift, float scale) {
  const E* x = static_cast<const E*>(X0);
  const E* w = static_cast<const E*>(cw);
  E* y = static_cast<E*>(Y);
  const E* h = static_cast<const E*>(halo);
  switch (k) {
#define IPTTT_CONV_CASE(KK) \
  case KK: simt::causal_conv_kernel<E, KK><<<grid, block, 0, ctx->stream>>>(x, w, y, T_len, d, h, shift, scale); break;
    IPTTT_CONV_CASE(1) IPTTT_CONV_CASE(2) IPTTT_CONV_CASE(3) IPTTT_CONV_CASE(4)
    IPTTT_CONV_CASE(5) IPTTT_CONV_CASE(6) IPTTT_CONV_CASE(7) IPTTT_CONV_CASE(8)
#undef IPTTT_CONV_CASE
    default: break;
  }
}

// Y = scale * CausalConv1D(X0), window shifted by ctx->target_shift (0 or 1).
ipttt_status run_conv(ipttt_ctx* ctx, const void* X0, const void* cw, int64_t B, int64_t T, int64_t d, int k,
                      ipttt_dtype dt, void* Y, const void* halo = nullptr, float scale = 1.f) {
  if (B == 0 || T == 0) return IPTTT_OK;
  const int rows = dt == IPTTT_BF16 ? simt::conv_rows<__nv_bfloat16>() : simt::conv_rows<float>();
  dim3 block(32, simt::CONV_STRIPS);
  dim3 grid(ceil_div(d / 8, 32), ceil_div(T, (int64_t)rows * simt::CONV_STRIPS), (unsigned)B);
  if (dt == IPTTT_BF16)
    launch_conv<__nv_bfloat16>(ctx, grid, block, X0, cw, Y, (int)T, (int)d, k, halo, ctx->target_shift, scale);
  else
    launch_conv<float>(ctx, grid, block, X0, cw, Y, (int)T, (int)d, k, halo, ctx->target_shift, scale);
  return check_launch(ctx, "conv launch");
}

// zero_ptr / zero_count (bf16 only): words the kernel clears before the fused state + apply
// kernel that follows it on the stream uses them as counters.
ipttt_status run_target_gemm(ipttt_ctx* ctx, const void* Y, const void* Wt, int64_t rows, int64_t d, float scale,
                             ipttt_dtype dt, void* V, uint32_t* zero_ptr = nullptr, int zero_count = 0) {
  if (rows == 0) return IPTTT_OK;
  if (dt == IPTTT_BF16) {
    CUtensorMap ma, mb, mo;
    if (!map_2d(ctx, &ma, Y, rows, d, 64, 128) || !map_2d(ctx, &mb, Wt, d, d, 64, 64) ||
        !map_2d(ctx, &mo, V, rows, d, 64, 32))
      return IPTTT_ERR_CUDA;
    gemm::Params p{};
    p.m_tiles = ceil_div(rows, gemm::BM);
    p.n_tiles = ceil_div(d, gemm::BN);
    p.k_blocks = ceil_div(d, gemm::BK);
    p.problems = 1;
    p.group_m = 16;
    p.scale = scale;
    p.zero_ptr = zero_ptr;
    p.zero_count = zero_count;
    p.st = dev_status(ctx);
    const bool pairs = use_pairs(ctx);
    if (pairs) {
      p.m_tiles = ceil_div(rows, gemm2::PAIR_M);
      p.group_m = 8;
      const int tiles = p.m_tiles * p.n_tiles;
      gemm2::tc_gemm2_kernel<gemm::kTarget><<<pair_grid(ctx, tiles), gemm2::NUM_THREADS, gemm2::SMEM_BYTES,
                                             ctx->stream>>>(ma, mb, mb, mo, mo, p);
    } else {
      const int tiles = p.m_tiles * p.n_tiles;
      const int grid = tiles < ctx->sm_count ? tiles : ctx->sm_count;
      gemm::tc_gemm_kernel<gemm::kTarget><<<grid, gemm::NUM_THREADS, gemm::SMEM_BYTES, ctx->stream>>>(ma, mb, mb, mo,
                                                                                                      mo, p);
    }
  } else {
    simt::SgemmParams p{};
    p.A = static_cast<const float*>(Y);
    p.B = static_cast<const float*>(Wt);
    p.Cm = static_cast<float*>(V);
    p.M = (int)rows;
    p.N = (int)d;
    p.K = (int)d;
    p.a_sm = d, p.a_sk = 1, p.b_sk = d, p.b_sn = 1, p.c_sm = d;
    p.scale = scale;
    dim3 grid(ceil_div(d, simt::SG_BN), ceil_div(rows, simt::SG_BM), 1);
    simt::sgemm_kernel<false><<<grid, 256, 0, ctx->stream>>>(p);
  }
  return check_launch(ctx, "target launch");
}

// Step (2) as one kernel on CTA pairs (tc_target2.cuh), bf16, W_target given:
// V = scale * (CausalConv1D(X0) W_target), the conv window shifted by ctx->target_shift and
// continuing from `halo` ([B, k-1, d], NULL = zeros); Y is never stored.  zero_ptr / zero_count:
// words CTA 0 clears for the fused state + apply kernel that follows.
ipttt_status run_target_conv(ipttt_ctx* ctx, const void* X0, const void* cw, const void* Wt, int64_t B, int64_t T,
                             int64_t d, int k, float scale, void* V, const void* halo = nullptr,
                             uint32_t* zero_ptr = nullptr, int zero_count = 0) {
  if (B == 0 || T == 0) return IPTTT_OK;
  CUtensorMap mx, mb, mo;
  if (!map_3d_plain(ctx, &mx, X0, B, T, d, tconv2::XROWS) || !map_2d(ctx, &mb, Wt, d, d, 64, 64) ||
      !map_3d(ctx, &mo, V, B, T, d, 32))
    return IPTTT_ERR_CUDA;
  tconv2::Params p{};
  p.B = (int)B;
  p.T = (int)T;
  p.d = (int)d;
  p.m_tiles = ceil_div(T, tconv2::PAIR_M);
  p.n_tiles = ceil_div(d, tconv2::BN);
  p.k_blocks = ceil_div(d, tconv2::BK);
  p.group_m = 8;
  p.shift = ctx->target_shift;
  p.scale = scale;
  p.conv_w = static_cast<const __nv_bfloat16*>(cw);
  p.halo = k > 1 ? static_cast<const __nv_bfloat16*>(halo) : nullptr;
  p.zero_ptr = zero_ptr;
  p.zero_count = zero_count;
  p.st = dev_status(ctx);
  const int64_t tiles = (int64_t)p.B * p.m_tiles * p.n_tiles;
  const dim3 grid((unsigned)pair_grid(ctx, tiles)), block(tconv2::NUM_THREADS);
  const size_t sm = tconv2::SMEM_BYTES;
  switch (k) {
#define IPTTT_TCONV_CASE(KK) \
  case KK: tconv2::tc_target_conv2_kernel<KK><<<grid, block, sm, ctx->stream>>>(mx, mb, mo, p); break;
    IPTTT_TCONV_CASE(1) IPTTT_TCONV_CASE(2) IPTTT_TCONV_CASE(3) IPTTT_TCONV_CASE(4)
    IPTTT_TCONV_CASE(5) IPTTT_TCONV_CASE(6) IPTTT_TCONV_CASE(7) IPTTT_TCONV_CASE(8)
#undef IPTTT_TCONV_CASE
    default:
      set_err(ctx, "conv kernel size k=%d > %d", k, simt::CONV_MAXK);
      return IPTTT_ERR_UNSUPPORTED;
  }
  return check_launch(ctx, "target launch");
}

// The bf16 state kernel on CTA pairs (256-row units) or single CTAs (128-row units); p's
// m_units / units are given for 128-row units and recomputed here for pairs.
ipttt_status launch_state_kernel(ipttt_ctx* ctx, const CUtensorMap& mv, const CUtensorMap& mz, const CUtensorMap& mw,
                                 const CUtensorMap& mf, state::Params p) {
  if (use_pairs(ctx)) {
    p.m_units = ceil_div(p.d, state2::PAIR_D);
    p.units = p.B * p.m_units * p.n_units;
    state2::tc_state2_kernel<<<pair_grid(ctx, (p.units + 1) / 2), state2::NUM_THREADS, state2::SMEM_BYTES,
                               ctx->stream>>>(mv, mz, mw, mf, p);
  } else {
    if (p.blocked) {  // the single-CTA kernel loads 3-D maps only
      set_err(ctx, "state kernel: blocked operand maps without CTA pairs");
      return IPTTT_ERR_UNSUPPORTED;
    }
    const int pairs = (p.units + 1) / 2;
    const int grid = pairs < ctx->sm_count ? pairs : ctx->sm_count;
    state::tc_state_kernel<<<grid, state::NUM_THREADS, state::SMEM_BYTES, ctx->stream>>>(mv, mz, mw, mf, p);
  }
  return check_launch(ctx, "state launch");
}

// Steps (3)+(4).  fp32: Step 1 (all Delta_i) then Step 2 (scan); bf16: one fused kernel.
// skip_first (bf16): leave W_eff[b, 0] (= W_down0) unwritten; the layer's apply then reads
// W_down0 for chunk 0 directly.
// W_init (optional, [B, d, f] fp32): each sequence's own starting state instead of W0.
ipttt_status run_state(ipttt_ctx* ctx, const void* V, const void* Z, const void* W0, int64_t B, int64_t T,
                       int64_t d, int64_t f, int64_t C, ipttt_dtype dt, void* W_eff, float* W_final,
                       bool skip_first = false, const float* W_init = nullptr) {
  const int64_t n = n_chunks_of(T, C);
  if (B == 0 || n == 0) return IPTTT_OK;
  if (dt == IPTTT_BF16) {
    CUtensorMap mv, mz, mw, mf;
    int blocked = 0;
    if (!map_state_operands(ctx, &mv, &mz, V, d, Z, f, B, T, d, f, use_pairs(ctx), &blocked) ||
        !map_3d(ctx, &mw, W_eff, B * n, d, f, 32) || !map_3d_f32(ctx, &mf, W_final, B, d, f, 32))
      return IPTTT_ERR_CUDA;
    state::Params p{};
    p.blocked = blocked;
    p.B = (int)B;
    p.T = (int)T;
    p.d = (int)d;
    p.f = (int)f;
    p.C = (int)C;
    p.n_chunks = (int)n;
    p.m_units = ceil_div(d, state::BMD);
    p.n_units = ceil_div(f, state::BNF);
    p.units = (int)(B * p.m_units * p.n_units);
    p.W0 = static_cast<const __nv_bfloat16*>(W0);
    p.skip_first = (skip_first && W_init == nullptr) ? 1 : 0;
    p.W_init = W_init;
    p.st = dev_status(ctx);
    return launch_state_kernel(ctx, mv, mz, mw, mf, p);
  }
  simt::SgemmParams p{};
  p.A = static_cast<const float*>(V);
  p.B = static_cast<const float*>(Z);
  p.Cm = static_cast<float*>(W_eff);
  p.M = (int)d;
  p.N = (int)f;
  p.K = (int)C;
  p.a_sm = 1, p.a_sk = d, p.b_sk = f, p.b_sn = 1, p.c_sm = f;
  p.a_tok = d, p.b_tok = f, p.c_tok = 0;
  p.a_z = 0, p.b_z = 0, p.c_z = d * f;
  p.chunked = 2;
  p.T = (int)T, p.C = (int)C, p.n_chunks = (int)n;
  p.scale = 1.f;
  dim3 grid(ceil_div(f, simt::SG_BN), ceil_div(d, simt::SG_BM), (unsigned)(B * n));
  simt::sgemm_kernel<false><<<grid, 256, 0, ctx->stream>>>(p);
  ipttt_status s = check_launch(ctx, "delta launch");
  if (s != IPTTT_OK) return s;
  const int64_t df = d * f;
  dim3 g2(ceil_div(df, 256), (unsigned)B);
  simt::chunk_scan_f32_kernel<<<g2, 256, 0, ctx->stream>>>(static_cast<float*>(W_eff), static_cast<const float*>(W0),
                                                             W_final, (int)B, (int)n, df, W_init, 0);
  return check_launch(ctx, "scan launch");
}

// W0 (bf16, optional): chunk 0 of every sequence is applied with W0 instead of W_eff[b, 0].
ipttt_status run_apply(ipttt_ctx* ctx, const void* Z, const void* W_eff, int64_t B, int64_t T, int64_t d, int64_t f,
                       int64_t C, ipttt_dtype dt, void* O, const void* W0 = nullptr, float scale = 1.f) {
  const int64_t n = n_chunks_of(T, C);
  if (B == 0 || n == 0) return IPTTT_OK;
  if (dt == IPTTT_BF16) {
    // pairs: 256-row tiles (each CTA loads 128 rows of the chunk's weight), whole tiles per chunk
    const bool pairs = use_pairs(ctx) && C % gemm2::PAIR_M == 0;
    const uint32_t w_rows = pairs ? gemm2::BN_HALF : gemm::BN;
    CUtensorMap ma, mb, mw0, mo;
    if (!map_3d(ctx, &ma, Z, B, T, f, 128) || !map_3d(ctx, &mb, W_eff, B * n, d, f, w_rows) ||
        !map_3d(ctx, &mo, O, B, T, d, 32))
      return IPTTT_ERR_CUDA;
    if (W0 != nullptr) {
      if (!map_2d(ctx, &mw0, W0, d, f, 64, w_rows)) return IPTTT_ERR_CUDA;
    } else {
      mw0 = mb;
    }
    gemm::Params p{};
    p.m_tiles = (int)(C / (pairs ? gemm2::PAIR_M : gemm::BM));
    p.n_tiles = ceil_div(d, gemm::BN);
    p.k_blocks = ceil_div(f, gemm::BK);
    p.problems = (int)(B * n);
    p.group_m = 16;
    p.scale = scale;
    p.T = (int)T, p.C = (int)C, p.n_chunks = (int)n;
    p.first_from_w0 = W0 != nullptr ? 1 : 0;
    p.st = dev_status(ctx);
    const int tiles = p.problems * p.m_tiles * p.n_tiles;
    if (pairs) {
      p.group_m = 8;
      gemm2::tc_gemm2_kernel<gemm::kApply><<<pair_grid(ctx, tiles), gemm2::NUM_THREADS, gemm2::SMEM_BYTES,
                                            ctx->stream>>>(ma, mb, mw0, mo, mo, p);
    } else {
      const int grid = tiles < ctx->sm_count ? tiles : ctx->sm_count;
      gemm::tc_gemm_kernel<gemm::kApply><<<grid, gemm::NUM_THREADS, gemm::SMEM_BYTES, ctx->stream>>>(ma, mb, mw0, mo,
                                                                                                     mo, p);
    }
  } else {
    simt::SgemmParams p{};
    p.A = static_cast<const float*>(Z);
    p.B = static_cast<const float*>(W_eff);
    p.Cm = static_cast<float*>(O);
    p.M = (int)C;
    p.N = (int)d;
    p.K = (int)f;
    p.a_sm = f, p.a_sk = 1, p.b_sk = 1, p.b_sn = f, p.c_sm = d;
    p.a_tok = f, p.b_tok = 0, p.c_tok = d;
    p.a_z = 0, p.b_z = d * f, p.c_z = 0;
    p.chunked = 1;
    p.T = (int)T, p.C = (int)C, p.n_chunks = (int)n;
    p.scale = scale;
    dim3 grid(ceil_div(d, simt::SG_BN), ceil_div(C, simt::SG_BM), (unsigned)(B * n));
    simt::sgemm_kernel<false><<<grid, 256, 0, ctx->stream>>>(p);
  }
  return check_launch(ctx, "apply launch");
}

// Steps (3)-(5) as one cooperative kernel: state unit pairs, then apply tiles from a queue
// (tc_fused.cuh).  `ctr` holds B*n slice counters and the queue head, zeroed beforehand.
// The pair version (tc_fused2.cuh): 256-row state units and apply tiles (C % 256 == 0).
// Returns false, having launched nothing, when the cooperative cluster launch is refused.
bool launch_state_apply_pairs(ipttt_ctx* ctx, const void* V, const void* Z, const void* W0, int64_t B, int64_t T,
                              int64_t d, int64_t f, int64_t C, void* W_eff, float* W_final, void* O, uint32_t* ctr,
                              const float* W_init, bool write_first, ipttt_status* st) {
  const int64_t n = n_chunks_of(T, C);
  CUtensorMap mv, mz, mw_st, mf, mza, mw_ld, mw0, mo;
  int blocked = 0;
  *st = IPTTT_ERR_CUDA;
  if (!map_state_operands(ctx, &mv, &mz, V, d, Z, f, B, T, d, f, true, &blocked) ||
      !map_3d(ctx, &mw_st, W_eff, B * n, d, f, 32) || !map_3d_f32(ctx, &mf, W_final, B, d, f, 32) ||
      !map_3d(ctx, &mza, Z, B, T, f, 128) || !map_3d(ctx, &mw_ld, W_eff, B * n, d, f, 128) ||
      !map_3d(ctx, &mo, O, B, T, d, 32))
    return true;
  if (W_init == nullptr && !write_first) {
    if (!map_2d(ctx, &mw0, W0, d, f, 64, 128)) return true;
  } else {
    mw0 = mw_ld;  // unused: chunk 0 reads W_eff[b, 0]
  }
  fused::Params p{};
  p.s.B = (int)B;
  p.s.T = (int)T;
  p.s.d = (int)d;
  p.s.f = (int)f;
  p.s.C = (int)C;
  p.s.n_chunks = (int)n;
  p.s.m_units = ceil_div(d, state2::PAIR_D);
  p.s.n_units = ceil_div(f, state2::BNF);
  p.s.units = (int)(B * p.s.m_units * p.s.n_units);
  p.s.W0 = static_cast<const __nv_bfloat16*>(W0);
  p.s.skip_first = (W_init == nullptr && !write_first) ? 1 : 0;
  p.s.W_init = W_init;
  p.s.blocked = blocked;
  p.s.st = dev_status(ctx);
  // 256 x 512 apply tiles (a quarter fewer operand bytes per FLOP, one accumulator whose epilogue
  // is not hidden) when a tile is long, d_ff / 64 >= 128 k-blocks, and the wide tiles still
  // make two waves over the co-resident pairs; else 256 x 256 tiles, two accumulators in turn.
  // Measured on one box with both instantiations: wide 0.5-1.2 % faster at d_ff = 9728 (152
  // k-blocks), narrow 2-4.5 % faster at d_ff = 4096 (64 k-blocks).
  const int64_t wide_tiles = B * n * (C / gemm2::PAIR_M) * ceil_div(d, 2 * gemm2::BN);
  p.a_halves = ctx->apply_halves != 0 ? ctx->apply_halves
               : (wide_tiles >= (int64_t)ctx->pair_ctas && ceil_div(f, gemm2::BK) >= 128) ? 2 : 1;
  p.a.m_tiles = (int)(C / gemm2::PAIR_M);
  p.a.n_tiles = ceil_div(d, p.a_halves * gemm2::BN);
  p.a.k_blocks = ceil_div(f, gemm2::BK);
  p.a.problems = (int)(B * n);
  p.a.group_m = 8;
  p.a.scale = 1.f;
  p.a.T = (int)T, p.a.C = (int)C, p.a.n_chunks = (int)n;
  p.a.first_from_w0 = p.s.skip_first;
  p.a.st = dev_status(ctx);
  p.ready = ctr;
  p.next_tile = ctr + B * n;
  p.ready_target = (uint32_t)(p.s.m_units * p.s.n_units * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctx->pair_ctas);
  cfg.blockDim = dim3(fused2::NUM_THREADS);
  cfg.dynamicSmemBytes = fused2::SMEM_BYTES;
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      p.a_halves == 2
          ? cudaLaunchKernelEx(&cfg, fused2::tc_state_apply2_kernel<2>, mv, mz, mw_st, mf, mza, mw_ld, mw0, mo, p)
          : cudaLaunchKernelEx(&cfg, fused2::tc_state_apply2_kernel<1>, mv, mz, mw_st, mf, mza, mw_ld, mw0, mo, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // a refused launch configuration is not sticky
    // "too large": this context now has fewer SMs than the grid was sized for (the next call
    // may fit again); anything else: the driver does not take cooperative launches of
    // clusters, so stop trying
    if (e != cudaErrorCooperativeLaunchTooLarge) ctx->fused_pairs = false;
    return false;
  }
  *st = check_launch(ctx, "state+apply launch");
  return true;
}

// write_first: W_eff[b, 0] is written (and chunk 0 applied from it) even without W_init.
ipttt_status run_state_apply_fused(ipttt_ctx* ctx, const void* V, const void* Z, const void* W0, int64_t B, int64_t T,
                                   int64_t d, int64_t f, int64_t C, void* W_eff, float* W_final, void* O,
                                   uint32_t* ctr, const float* W_init = nullptr, bool write_first = false) {
  if (use_pairs(ctx) && ctx->fused_pairs && C % gemm2::PAIR_M == 0) {
    ipttt_status st;
    if (launch_state_apply_pairs(ctx, V, Z, W0, B, T, d, f, C, W_eff, W_final, O, ctr, W_init, write_first, &st))
      return st;
  }
  const int64_t n = n_chunks_of(T, C);
  CUtensorMap mv, mz, mw_st, mf, mza, mw_ld, mw0, mo;
  if (!map_3d(ctx, &mv, V, B, T, d, 64) || !map_3d(ctx, &mz, Z, B, T, f, 64) ||
      !map_3d(ctx, &mw_st, W_eff, B * n, d, f, 32) || !map_3d_f32(ctx, &mf, W_final, B, d, f, 32) ||
      !map_3d(ctx, &mza, Z, B, T, f, 128) || !map_3d(ctx, &mw_ld, W_eff, B * n, d, f, 256) ||
      !map_3d(ctx, &mo, O, B, T, d, 32))
    return IPTTT_ERR_CUDA;
  if (W_init == nullptr && !write_first) {
    if (!map_2d(ctx, &mw0, W0, d, f, 64, 256)) return IPTTT_ERR_CUDA;
  } else {
    mw0 = mw_ld;  // unused: chunk 0 reads W_eff[b, 0]
  }
  fused::Params p{};
  p.s.B = (int)B;
  p.s.T = (int)T;
  p.s.d = (int)d;
  p.s.f = (int)f;
  p.s.C = (int)C;
  p.s.n_chunks = (int)n;
  p.s.m_units = ceil_div(d, state::BMD);
  p.s.n_units = ceil_div(f, state::BNF);
  p.s.units = (int)(B * p.s.m_units * p.s.n_units);
  p.s.W0 = static_cast<const __nv_bfloat16*>(W0);
  p.s.skip_first = (W_init == nullptr && !write_first) ? 1 : 0;
  p.s.W_init = W_init;
  p.s.st = dev_status(ctx);
  p.a.m_tiles = (int)(C / gemm::BM);
  p.a.n_tiles = ceil_div(d, gemm::BN);
  p.a.k_blocks = ceil_div(f, gemm::BK);
  p.a.problems = (int)(B * n);
  p.a.group_m = 16;
  p.a.scale = 1.f;
  p.a.T = (int)T, p.a.C = (int)C, p.a.n_chunks = (int)n;
  p.a.first_from_w0 = p.s.skip_first;
  p.a.st = dev_status(ctx);
  p.ready = ctr;
  p.next_tile = ctr + B * n;
  p.ready_target = (uint32_t)(p.s.m_units * p.s.n_units * 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctx->sm_count);
  cfg.blockDim = dim3(fused::NUM_THREADS);
  cfg.dynamicSmemBytes = fused::SMEM_BYTES;
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, fused::tc_state_apply_kernel, mv, mz, mw_st, mf, mza, mw_ld, mw0, mo, p);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    // more CTAs than this context can hold at once (fewer SMs than at sizing time): the
    // caller runs steps (3)-(5) as separate kernels instead
    cudaGetLastError();
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "state+apply launch");
  return check_launch(ctx, "state+apply launch");
}

// A decode step's rows (simt.cuh, decode rows).  The SwiGLU of one token row streams the
// weights on the CUDA cores (2 columns per block, 2 slices per warp in flight); several bf16
// rows go through the tensor-core SwiGLU GEMM, which streams them as fast whatever the row
// count up to a tile (the fp32 path has no tensor-core GEMM: its rows stay on the CUDA cores,
// in launches of up to DEC_ROWS rows).  The first SwiGLU launch fills the chunk buffers, or two
// strided copies do.  Then each sequence's m rows are applied with its weight W_cur[b] on the
// CUDA cores (one row: 2 weight rows per block; more: 8 weight rows per block).
template <typename E>
ipttt_status run_decode_rows(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                             const void* Wc, int64_t B, int64_t m, int64_t d, int64_t f, int64_t C, int64_t pos,
                             void* Z, void* O, void* H_buf, void* X0_buf) {
  constexpr int R = simt::DEC_ROWS;
  constexpr bool kF32 = std::is_same<E, float>::value;
  const E* h = static_cast<const E*>(H);
  E* z = static_cast<E*>(Z);
  const int64_t rows = B * m;
  const int64_t cap = (int64_t)ctx->sm_count * 8;
  auto grid = [&](int64_t groups) { return (unsigned)(groups < cap ? groups : cap); };
  ipttt_status s = IPTTT_OK;
  if (kF32 || rows == 1) {
    for (int64_t r0 = 0; r0 < rows; r0 += R) {
      const int nr = (int)(rows - r0 < R ? rows - r0 : R);
      const bool copy = r0 == 0 && H_buf != nullptr;
      const E* hc = copy ? h : nullptr;
      const E* xc = copy ? static_cast<const E*>(X0) : nullptr;
      E* hb = copy ? static_cast<E*>(H_buf) : nullptr;
      E* xb = copy ? static_cast<E*>(X0_buf) : nullptr;
      if (nr == 1)
        simt::decode_swiglu_kernel<E, 1, 2, 2><<<grid(ceil_div(f, 2)), simt::DEC_THREADS, 0, ctx->stream>>>(
            h + r0 * d, static_cast<const E*>(Wg), static_cast<const E*>(Wu), z + r0 * f, nr, (int)d, (int)f, hc, xc,
            hb, xb, (int)B, (int)m, C, pos);
      else
        simt::decode_swiglu_kernel<E, R, 2, 1><<<grid(ceil_div(f, 2)), simt::DEC_THREADS, 0, ctx->stream>>>(
            h + r0 * d, static_cast<const E*>(Wg), static_cast<const E*>(Wu), z + r0 * f, nr, (int)d, (int)f, hc, xc,
            hb, xb, (int)B, (int)m, C, pos);
      if ((s = check_launch(ctx, "decode SwiGLU launch")) != IPTTT_OK) return s;
    }
  } else {
    if (H_buf != nullptr) {  // [B, m, d] -> rows pos.. of [B, C, d]
      const size_t w = (size_t)(m * d) * sizeof(E), dp = (size_t)(C * d) * sizeof(E), off = (size_t)(pos * d);
      cudaError_t e;
      if ((e = cudaMemcpy2DAsync(static_cast<E*>(H_buf) + off, dp, H, w, w, (size_t)B, cudaMemcpyDeviceToDevice,
                                 ctx->stream)) != cudaSuccess ||
          (e = cudaMemcpy2DAsync(static_cast<E*>(X0_buf) + off, dp, X0, w, w, (size_t)B, cudaMemcpyDeviceToDevice,
                                 ctx->stream)) != cudaSuccess)
        return cuda_fail(ctx, e, "decode chunk buffers");
    }
    if ((s = ensure_attrs(ctx)) != IPTTT_OK) return s;
    if ((s = run_swiglu(ctx, H, Wg, Wu, rows, d, f, IPTTT_BF16, Z, rows > gemm::BM)) != IPTTT_OK) return s;
  }
  // the apply starts as a dependent launch: it prefetches W_cur into L2 while the SwiGLU rows
  // stream theirs (when W_cur takes at most half the L2), then waits for Z
  const int64_t wc_bytes = B * d * f * (int64_t)sizeof(E);
  const int prefetch = wc_bytes <= (int64_t)64 << 20;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(simt::DEC_THREADS);
  cfg.stream = ctx->stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const E* wc = static_cast<const E*>(Wc);
  E* o = static_cast<E*>(O);
  cudaError_t e;
  if (m == 1) {
    cfg.gridDim = dim3(grid(B * d / 2));
    e = cudaLaunchKernelEx(&cfg, simt::decode_apply_kernel<E, 1, 2, 2>, (const E*)z, wc, o, (int)B, (int)m, (int)d,
                           (int)f, prefetch);
  } else {
    cfg.gridDim = dim3(grid(B * d / 8));
    e = cudaLaunchKernelEx(&cfg, simt::decode_apply_kernel<E, R, 8, 1>, (const E*)z, wc, o, (int)B, (int)m, (int)d,
                           (int)f, prefetch);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "decode apply launch");
  return check_launch(ctx, "decode apply launch");
}

}  // namespace
