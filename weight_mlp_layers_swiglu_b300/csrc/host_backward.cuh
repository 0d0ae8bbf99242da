// The backward pass, the training pair and the workspace layouts of the host-buffer entry.
// Part of the host side of libipttt (one translation unit: ipttt.cu includes the host_*.cuh
// files in order).  Everything here is internal; the C ABI is at the end of ipttt.cu.
#pragma once

#include "host_steps.cuh"

namespace {

// ------------------------------------------------------------------ backward pass

// One state-kernel launch in its general form (bf16): accumulator rows are the M columns of the
// token-major A operand (rows of V apart by v_stride elements), accumulator columns the N
// columns of Z (apart by z_stride); start from W_init (fp32), W0 (bf16) or zero; chunks in
// order or reversed; snapshots (bf16) into W_eff unless skip_first with one chunk.
ipttt_status launch_state_general(ipttt_ctx* ctx, const void* V, int64_t v_stride, const void* Z, int64_t z_stride,
                                  int64_t B, int64_t T, int64_t M, int64_t N, int64_t C, const void* W0,
                                  const float* W_init, bool skip_first, bool reverse, void* W_eff, float* W_final) {
  const int64_t n = n_chunks_of(T, C);
  CUtensorMap mv, mz, mw, mf;
  int blocked = 0;
  if (!map_state_operands(ctx, &mv, &mz, V, v_stride, Z, z_stride, B, T, M, N, use_pairs(ctx), &blocked) ||
      !map_3d_f32(ctx, &mf, W_final, B, M, N, 32))
    return IPTTT_ERR_CUDA;
  if (W_eff != nullptr) {
    if (!map_3d(ctx, &mw, W_eff, B * n, M, N, 32)) return IPTTT_ERR_CUDA;
  } else {
    mw = mv;  // never stored through: one chunk and no first snapshot
  }
  state::Params p{};
  p.B = (int)B;
  p.T = (int)T;
  p.d = (int)M;
  p.f = (int)N;
  p.C = (int)C;
  p.n_chunks = (int)n;
  p.m_units = ceil_div(M, state::BMD);
  p.n_units = ceil_div(N, state::BNF);
  p.units = (int)(B * p.m_units * p.n_units);
  p.W0 = static_cast<const __nv_bfloat16*>(W0);
  p.skip_first = skip_first ? 1 : 0;
  p.W_init = W_init;
  p.reverse = reverse ? 1 : 0;
  p.blocked = blocked;
  p.st = dev_status(ctx);
  return launch_state_kernel(ctx, mv, mz, mw, mf, p);
}

// C = A1 B1 + A2 B2 (bf16, kTwoSeg): A segments token-major [B, T, K] (a2 = A1's map shifted by
// a2_koff columns when a2 is NULL), B segments [slices, K, N]; per chunk when b_per_problem.
// With au != NULL, C is dZ and is not stored: the epilogue turns au = [A | U] ([B*T, 2N]) into
// [dA | dU] in place (out is then unused and may be NULL).
ipttt_status launch_two_seg(ipttt_ctx* ctx, const void* A1, int64_t a1_stride, const void* A2, int64_t a2_stride,
                            int64_t a2_koff, const void* B1, const void* B2, int64_t b_slices, bool b_per_problem,
                            int64_t B, int64_t T, int64_t C, int64_t K1, int64_t K2, int64_t N, void* out,
                            void* au = nullptr) {
  const int64_t n = n_chunks_of(T, C);
  CUtensorMap ma1, ma2, mb1, mb2, mo;
  // segment 1 is cut at K1 columns (its ragged K block reads zeros, not segment 2); without its
  // own pointer segment 2 is read through a map over [A1 | A2] at column offset a2_koff
  const bool shared = A2 == nullptr;
  if (!map_3d_strided(ctx, &ma1, A1, B, T, K1, a1_stride, 128) ||
      !map_3d_strided(ctx, &ma2, shared ? A1 : A2, B, T, shared ? a2_koff + K2 : K2, shared ? a1_stride : a2_stride,
                      128) ||
      !map_3d(ctx, &mb1, B1, b_slices, K1, N, 64) || !map_3d(ctx, &mb2, B2, b_slices, K2, N, 64))
    return IPTTT_ERR_CUDA;
  if (out != nullptr) {
    if (!map_3d(ctx, &mo, out, B, T, N, 32)) return IPTTT_ERR_CUDA;
  } else {
    mo = ma1;  // never stored through
  }
  const bool pairs = use_pairs(ctx) && C % gemm2::PAIR_M == 0;
  gemm::Params p{};
  p.m_tiles = (int)(C / (pairs ? gemm2::PAIR_M : gemm::BM));
  p.n_tiles = ceil_div(N, gemm::BN);
  p.k_blocks = ceil_div(K1, gemm::BK);
  p.k_blocks2 = ceil_div(K2, gemm::BK);
  p.a2_koff = shared ? (int)a2_koff : 0;
  p.b_per_problem = b_per_problem ? 1 : 0;
  p.au = static_cast<__nv_bfloat16*>(au);
  p.au_f = (int)N;
  p.problems = (int)(B * n);
  p.group_m = 16;
  p.scale = 1.f;
  p.T = (int)T, p.C = (int)C, p.n_chunks = (int)n;
  p.st = dev_status(ctx);
  const int tiles = p.problems * p.m_tiles * p.n_tiles;
  if (pairs) {
    p.group_m = b_per_problem ? 8 : 32;  // one shared B (dH): as the SwiGLU GEMM
    gemm2::tc_gemm2_kernel<gemm::kTwoSeg><<<pair_grid(ctx, tiles), gemm2::NUM_THREADS, gemm2::SMEM_BYTES,
                                           ctx->stream>>>(ma1, mb1, ma2, mo, mb2, p);
  } else {
    const int grid = tiles < ctx->sm_count ? tiles : ctx->sm_count;
    gemm::tc_gemm_kernel<gemm::kTwoSeg><<<grid, gemm::NUM_THREADS, gemm::SMEM_BYTES, ctx->stream>>>(ma1, mb1, ma2,
                                                                                                      mo, mb2, p);
  }
  return check_launch(ctx, "two-segment launch");
}

// fp32 CUDA-core GEMM helper: C[z] = scale * A B (+ beta C) with element strides.
ipttt_status sgemm(ipttt_ctx* ctx, const float* A, int64_t a_sm, int64_t a_sk, const float* Bm, int64_t b_sk,
                   int64_t b_sn, float* Cm, int64_t c_sm, int64_t M, int64_t N, int64_t K, float scale, float beta,
                   int chunked = 0, int64_t T = 0, int64_t C = 0, int64_t n = 0, int64_t Bseq = 1, int64_t a_tok = 0,
                   int64_t b_tok = 0, int64_t c_tok = 0, int64_t a_z = 0, int64_t b_z = 0, int64_t c_z = 0) {
  simt::SgemmParams p{};
  p.A = A, p.B = Bm, p.Cm = Cm;
  p.M = (int)M, p.N = (int)N, p.K = (int)K;
  p.a_sm = a_sm, p.a_sk = a_sk, p.b_sk = b_sk, p.b_sn = b_sn, p.c_sm = c_sm;
  p.a_tok = a_tok, p.b_tok = b_tok, p.c_tok = c_tok, p.a_z = a_z, p.b_z = b_z, p.c_z = c_z;
  p.chunked = chunked;
  p.T = (int)T, p.C = (int)C, p.n_chunks = (int)n;
  p.scale = scale;
  p.beta = beta;
  dim3 grid(ceil_div(N, simt::SG_BN), ceil_div(M, simt::SG_BM), (unsigned)(chunked ? Bseq * n : 1));
  simt::sgemm_kernel<false><<<grid, 256, 0, ctx->stream>>>(p);
  return check_launch(ctx, "sgemm launch");
}

// Step (1) that also keeps the gate and up pre-activations AU = [A | U] ([rows, 2 d_ff]) for
// the backward pass: bf16 through the SwiGLU GEMM's saving epilogue, fp32 as two GEMMs and an
// elementwise combine.
ipttt_status run_swiglu_save(ipttt_ctx* ctx, const void* H, const void* Wg, const void* Wu, int64_t BT, int64_t d,
                             int64_t f, ipttt_dtype dt, void* Z, void* AU) {
  ipttt_status s = IPTTT_OK;
  if (BT == 0) return s;
  if (dt == IPTTT_BF16) {
    // [A | U] as [rows][2][d_ff]: a box never crosses from the gate half into the up half
    CUtensorMap ma, mb0, mb1, mo, mx;
    const uint64_t au_dims[3] = {(uint64_t)f, 2, (uint64_t)BT};
    const uint64_t au_strides[2] = {(uint64_t)f * 2, (uint64_t)f * 4};
    const uint32_t au_box[3] = {64, 1, 32};
    if (!map_2d(ctx, &ma, H, BT, d, 64, 128) || !map_2d(ctx, &mb0, Wg, f, d, 64, 128) ||
        !map_2d(ctx, &mb1, Wu, f, d, 64, 128) || !map_2d(ctx, &mo, Z, BT, f, 64, 32) ||
        !encode_map(ctx, &mx, AU, 3, au_dims, au_strides, au_box))
      return IPTTT_ERR_CUDA;
    const bool pairs = use_pairs(ctx);
    gemm::Params p{};
    p.m_tiles = ceil_div(BT, pairs ? gemm2::PAIR_M : gemm::BM);
    p.n_tiles = ceil_div(f, 128);
    p.k_blocks = ceil_div(d, gemm::BK);
    p.problems = 1;
    p.group_m = pairs ? 32 : 16;  // as the SwiGLU GEMM of the forward
    p.scale = 1.f;
    p.st = dev_status(ctx);
    const int tiles = p.m_tiles * p.n_tiles;
    if (pairs) {
      gemm2::tc_gemm2_kernel<gemm::kSwigluSave><<<pair_grid(ctx, tiles), gemm2::NUM_THREADS, gemm2::SMEM_BYTES,
                                                 ctx->stream>>>(ma, mb0, mb1, mo, mx, p);
    } else {
      const int grid = tiles < ctx->sm_count ? tiles : ctx->sm_count;
      gemm::tc_gemm_kernel<gemm::kSwigluSave><<<grid, gemm::NUM_THREADS, gemm::SMEM_BYTES, ctx->stream>>>(
          ma, mb0, mb1, mo, mx, p);
    }
    return check_launch(ctx, "swiglu save launch");
  }
  // A -> AU[:, :f], U -> AU[:, f:], then Z = SiLU(A) U
  float* au = static_cast<float*>(AU);
  if ((s = sgemm(ctx, static_cast<const float*>(H), d, 1, static_cast<const float*>(Wg), 1, d, au, 2 * f, BT, f, d,
                 1.f, 0.f)) != IPTTT_OK ||
      (s = sgemm(ctx, static_cast<const float*>(H), d, 1, static_cast<const float*>(Wu), 1, d, au + f, 2 * f, BT, f, d,
                 1.f, 0.f)) != IPTTT_OK)
    return s;
  simt::swiglu_combine_kernel<float><<<ceil_div(BT * f, 256), 256, 0, ctx->stream>>>(au, static_cast<float*>(Z), BT,
                                                                                     (int)f);
  return check_launch(ctx, "combine launch");
}

// Forward activations the backward pass reads (all dtype): Z [B,T,d_ff], [A | U] [B,T,2 d_ff],
// Y = conv(X0) [B,T,d], V = eta * Y W_target [B,T,d] and the W_i stack [B,n,d,d_ff] with every
// slice (W_0 = W_down0 included); then the fused kernel's counters.  Each region 256-byte aligned.
struct SavedLayout {
  size_t z, au, y, v, wst, ctr, total;
};

SavedLayout saved_layout(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, ipttt_dtype dt) {
  const size_t es = esize(dt);
  const int64_t n = n_chunks_of(T, C);
  SavedLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.z = take((size_t)B * T * f * es);
  L.au = take((size_t)B * T * 2 * f * es);
  L.y = take((size_t)B * T * d * es);
  L.v = take((size_t)B * T * d * es);
  L.wst = take((size_t)B * n * d * f * es);
  L.ctr = take((size_t)(B * n + 1) * 4);
  L.total = off;
  return L;
}

struct SavedPtrs {
  void *z, *au, *y, *v, *wst;
  uint32_t* ctr;
};

SavedPtrs saved_ptrs(void* base, const SavedLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(base);
  return SavedPtrs{b + L.z, b + L.au, b + L.y, b + L.v, b + L.wst, reinterpret_cast<uint32_t*>(b + L.ctr)};
}

// The backward pass's own scratch: dZ (fp32 path only), dV, dY, the R_i stack, per-sequence
// dW_down0 (fp32) and the conv-tap partial sums (fp32).
struct BwdScratch {
  size_t dz, dv, dy, rst, dw0b, part, total;
  int64_t strips;
};

BwdScratch scratch_layout(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, int k, ipttt_dtype dt) {
  const size_t es = esize(dt);
  const int64_t n = n_chunks_of(T, C);
  BwdScratch L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.dz = take(dt == IPTTT_BF16 ? 0 : (size_t)B * T * f * es);  // bf16: dZ never leaves the GEMM epilogue
  L.dv = take((size_t)B * T * d * es);
  L.dy = take((size_t)B * T * d * es);
  L.rst = take((size_t)B * n * d * f * es);
  L.dw0b = take((size_t)B * d * f * 4);
  L.strips = B * ((T + simt::CONVW_STRIP - 1) / simt::CONVW_STRIP);
  L.part = take((size_t)L.strips * d * k * 4);
  L.total = off;
  return L;
}

// Workspace of the backward pass with recompute: the saved activations, then the scratch.
size_t bwd_total(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, int k, ipttt_dtype dt) {
  return saved_layout(B, T, d, f, C, dt).total + scratch_layout(B, T, d, f, C, k, dt).total;
}

// Pieces of a host-buffer call: a multiple of C near kPieceTokens, at most kMaxPieces of them.
int64_t piece_len(int64_t T, int64_t C) {
  int64_t P = (kPieceTokens + C - 1) / C * C;
  const int64_t min_p = ((T + kMaxPieces - 1) / kMaxPieces + C - 1) / C * C;
  if (P < min_p) P = min_p;
  return P < T ? P : T;
}

// Device workspace of the host-buffer entry: the layer's workspace for one piece, then H, X0
// and O staged whole (piece j at offset B * lo * d), the fp32 state and two conv halos.
struct HostLayout {
  size_t h, x, o, w, halo0, halo1, total;
  int64_t piece;
};

HostLayout host_layout(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, int k, ipttt_dtype dt) {
  const size_t es = esize(dt);
  HostLayout L;
  L.piece = piece_len(T, C);
  size_t off = ws_layout(B, L.piece, d, f, C, dt).total;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.h = take((size_t)B * T * d * es);
  L.x = take((size_t)B * T * d * es);
  L.o = take((size_t)B * T * d * es);
  L.w = take((size_t)B * d * f * 4);
  L.halo0 = take((size_t)B * (k - 1) * d * es);
  L.halo1 = take((size_t)B * (k - 1) * d * es);
  L.total = off;
  return L;
}

// Recompute of the forward activations the backward pass reads (Z, [A | U], Y, V and every W_i;
// the forward's final state goes to W_fin_scratch).
ipttt_status run_forward_saved(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                               const void* W0, const void* Wt, const void* cw, int64_t B, int64_t T, int64_t d,
                               int64_t f, int64_t C, int k, float eta, ipttt_dtype dt, const SavedPtrs& sv,
                               float* W_fin_scratch) {
  ipttt_status s = IPTTT_OK;
  const int64_t BT = B * T;
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  if ((s = run_swiglu_save(ctx, H, Wg, Wu, BT, d, f, dt, sv.z, sv.au)) != IPTTT_OK) return s;
  if (Wt != nullptr) {
    if ((s = run_conv(ctx, X0, cw, B, T, d, k, dt, sv.y)) != IPTTT_OK) return s;
    if ((s = run_target_gemm(ctx, sv.y, Wt, BT, d, eta, dt, sv.v)) != IPTTT_OK) return s;
  } else if ((s = run_conv(ctx, X0, cw, B, T, d, k, dt, sv.v, nullptr, eta)) != IPTTT_OK) {  // V = eta * conv(X0)
    return s;
  }
  return run_state(ctx, sv.v, sv.z, W0, B, T, d, f, C, dt, sv.wst, W_fin_scratch, false);
}

// dX0 and the per-strip tap partials of the conv adjoint (kernels templated on the tap count).
template <typename E>
void launch_conv_adjoints(ipttt_ctx* ctx, dim3 gx, dim3 gw, const void* dY, const void* cw, const void* X0,
                          void* dX0, float* part, int T_len, int d, int k) {
  const E* dy = static_cast<const E*>(dY);
  const E* w = static_cast<const E*>(cw);
  const E* x = static_cast<const E*>(X0);
  E* dx = static_cast<E*>(dX0);
  const int sh = ctx->target_shift;
  switch (k) {
#define IPTTT_ADJ_CASE(KK)                                                                              \
  case KK:                                                                                              \
    simt::conv_backward_x_kernel<E, KK><<<gx, 64, 0, ctx->stream>>>(dy, w, dx, T_len, d, sh);           \
    simt::conv_backward_w_partial_kernel<E, KK><<<gw, 64, 0, ctx->stream>>>(dy, x, part, T_len, d, sh); \
    break;
    IPTTT_ADJ_CASE(1) IPTTT_ADJ_CASE(2) IPTTT_ADJ_CASE(3) IPTTT_ADJ_CASE(4)
    IPTTT_ADJ_CASE(5) IPTTT_ADJ_CASE(6) IPTTT_ADJ_CASE(7) IPTTT_ADJ_CASE(8)
#undef IPTTT_ADJ_CASE
    default: break;
  }
}

// The backward pass from the saved forward activations (validated by the caller; T >= 1).  It
// overwrites sv.au with [dA | dU].
ipttt_status run_backward_core(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                               const void* Wt, const void* cw, int64_t B, int64_t T, int64_t d, int64_t f, int64_t C,
                               int k, float eta, ipttt_dtype dt, const void* dO, const float* dW_final, void* dH,
                               void* dX0, float* dWg, float* dWu, float* dW0, float* dWt, float* dcw,
                               const SavedPtrs& sv, void* scratch) {
  ipttt_status s = IPTTT_OK;
  const BwdScratch L = scratch_layout(B, T, d, f, C, k, dt);
  uint8_t* base = static_cast<uint8_t*>(scratch);
  const void* Y = sv.y;
  const void* V = sv.v;
  const void* Z = sv.z;
  void* AU = sv.au;
  const void* Wst = sv.wst;
  void* dZ = base + L.dz;
  void* dV = base + L.dv;
  void* dY = base + L.dy;
  void* Rst = base + L.rst;
  float* dW0b = reinterpret_cast<float*>(base + L.dw0b);
  float* part = reinterpret_cast<float*>(base + L.part);
  const int64_t n = n_chunks_of(T, C);
  const int64_t BT = B * T;
  const int64_t CT = (BT + 255) / 256 * 256;  // all tokens as one chunk (flat GEMMs and reductions)
  const bool bf16 = dt == IPTTT_BF16;
  const int64_t df = d * f;
  if (bf16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  // The target branch needs only R (the reverse scan): dV = eta Z R^T (per chunk),
  // dY = dV W_target^T, dW_target = Y^T dV (without a projection dY is dV itself), and the
  // causal conv's adjoints.
  auto target_branch = [&]() -> ipttt_status {
    ipttt_status r;
    if ((r = run_apply(ctx, Z, Rst, B, T, d, f, C, dt, dV, nullptr, eta)) != IPTTT_OK) return r;
    if (Wt == nullptr) {
      dY = dV;
    } else if (bf16) {
      if ((r = run_apply(ctx, dV, Wt, 1, BT, d, d, CT, dt, dY)) != IPTTT_OK) return r;
      if ((r = launch_state_general(ctx, Y, d, dV, d, 1, BT, d, d, CT, nullptr, nullptr, true, false, nullptr, dWt)) !=
          IPTTT_OK)
        return r;
    } else {
      if ((r = sgemm(ctx, static_cast<const float*>(dV), d, 1, static_cast<const float*>(Wt), 1, d,
                     static_cast<float*>(dY), d, BT, d, d, 1.f, 0.f)) != IPTTT_OK ||
          (r = sgemm(ctx, static_cast<const float*>(Y), 1, d, static_cast<const float*>(dV), d, 1, dWt, d, d, d, BT, 1.f,
                     0.f)) != IPTTT_OK)
        return r;
    }
    const int64_t groups = d / (bf16 ? 8 : 4);  // 16-byte channel groups
    dim3 gx(ceil_div(groups, 64), ceil_div(T, simt::CONVX_ROWS), (unsigned)B);
    dim3 gw((unsigned)L.strips, ceil_div(groups, 64));
    if (bf16)
      launch_conv_adjoints<__nv_bfloat16>(ctx, gx, gw, dY, cw, X0, dX0, part, (int)T, (int)d, k);
    else
      launch_conv_adjoints<float>(ctx, gx, gw, dY, cw, X0, dX0, part, (int)T, (int)d, k);
    simt::sum_strips_kernel<<<ceil_div(d * k, 256), 256, 0, ctx->stream>>>(part, dcw, (int)L.strips, d * k);
    return check_launch(ctx, "conv backward launch");
  };
  if (bf16) {
    // reverse scan: R_i = dW_final + sum_{l>i} dO_l^T Z_l, final = dW_final + sum_i dO_i^T Z_i
    if ((s = launch_state_general(ctx, dO, d, Z, f, B, T, d, f, C, nullptr, dW_final, false, true, Rst,
                                  B == 1 ? dW0 : dW0b)) != IPTTT_OK)
      return s;
    // After the scan the target branch can run on the context's side stream, beside dZ, dH,
    // dW_gate and dW_up on the caller's stream, so that the persistent kernels of one branch
    // fill the SMs the other leaves idle.  That pays when the weight-gradient reductions have
    // fewer 256 x 256 units than the grid has CTAs (at d = 1024, d_ff = 4096: 64 units, 12 %
    // faster); with a full round of units or more (the 4B widths: 380) the two branches only
    // contend, and it ran 1-4 % slower, so the branches then run in turn.  The branches read
    // only what was written before the fork (the dZ step rewrites [A | U], which the target
    // branch does not read) and write disjoint buffers; the caller's stream waits for the side
    // stream at the end.
    const bool fork = ceil_div(f, state2::BNF) * ceil_div(d, state2::PAIR_D) < (int64_t)ctx->pair_ctas;
    cudaStream_t main = ctx->stream;
    cudaError_t e;
    if (fork && ((e = cudaEventRecord(ctx->b_fork, main)) != cudaSuccess ||
                 (e = cudaStreamWaitEvent(ctx->side, ctx->b_fork, 0)) != cudaSuccess))
      return cuda_fail(ctx, e, "backward fork");
    if (fork) ctx->stream = ctx->side;
    const ipttt_status sb = target_branch();
    ctx->stream = main;
    const size_t es = 2;
    // dZ_i = dO_i W_i + V_i R_i (V carries eta), and in the same epilogue the gated-MLP
    // adjoints: AU = [A | U] becomes [dA | dU]
    if (sb == IPTTT_OK &&
        (s = launch_two_seg(ctx, dO, d, V, d, 0, Wst, Rst, B * n, true, B, T, C, d, d, f, nullptr, AU)) == IPTTT_OK &&
        // dH = dA W_gate + dU W_up
        (s = launch_two_seg(ctx, AU, 2 * f, nullptr, 2 * f, f, Wg, Wu, 1, false, 1, BT, CT, f, f, d, dH)) ==
            IPTTT_OK &&
        // dW_gate = dA^T H, dW_up = dU^T H (reductions over all tokens)
        (s = launch_state_general(ctx, AU, 2 * f, H, d, 1, BT, f, d, CT, nullptr, nullptr, true, false, nullptr,
                                  dWg)) == IPTTT_OK)
      s = launch_state_general(ctx, static_cast<uint8_t*>(AU) + f * es, 2 * f, H, d, 1, BT, f, d, CT, nullptr,
                               nullptr, true, false, nullptr, dWu);
    // join even after an error, so that no work of this call is left unordered on the side stream
    if (fork && ((e = cudaEventRecord(ctx->b_join, ctx->side)) != cudaSuccess ||
                 (e = cudaStreamWaitEvent(main, ctx->b_join, 0)) != cudaSuccess))
      return cuda_fail(ctx, e, "backward join");
    if (sb != IPTTT_OK) return sb;
    if (s != IPTTT_OK) return s;
  } else {
    float* rst = static_cast<float*>(Rst);
    // G_i = dO_i^T Z_i per chunk, then the reverse exclusive scan
    if ((s = sgemm(ctx, static_cast<const float*>(dO), 1, d, static_cast<const float*>(Z), f, 1, rst, f, d, f, C, 1.f,
                   0.f, 2, T, C, n, B, d, f, 0, 0, 0, df)) != IPTTT_OK)
      return s;
    dim3 g2(ceil_div(df, 256), (unsigned)B);
    simt::chunk_scan_f32_kernel<<<g2, 256, 0, ctx->stream>>>(rst, nullptr, B == 1 ? dW0 : dW0b, (int)B, (int)n, df,
                                                             dW_final, 1);
    if ((s = check_launch(ctx, "reverse scan launch")) != IPTTT_OK) return s;
    // dZ_i = dO_i W_i + V_i R_i
    if ((s = sgemm(ctx, static_cast<const float*>(dO), d, 1, static_cast<const float*>(Wst), f, 1,
                   static_cast<float*>(dZ), f, C, f, d, 1.f, 0.f, 1, T, C, n, B, d, 0, f, 0, df, 0)) != IPTTT_OK ||
        (s = sgemm(ctx, static_cast<const float*>(V), d, 1, rst, f, 1, static_cast<float*>(dZ), f, C, f, d, 1.f, 1.f,
                   1, T, C, n, B, d, 0, f, 0, df, 0)) != IPTTT_OK)
      return s;
    // the gated-MLP backward in place, AU -> [dA | dU] (bf16 does it in the dZ epilogue)
    simt::swiglu_backward_kernel<float><<<ceil_div(BT * f, 256), 256, 0, ctx->stream>>>(
        static_cast<const float*>(dZ), static_cast<float*>(AU), BT, (int)f);
    if ((s = check_launch(ctx, "swiglu backward launch")) != IPTTT_OK) return s;
    const float* au = static_cast<const float*>(AU);
    if ((s = sgemm(ctx, au, 2 * f, 1, static_cast<const float*>(Wg), d, 1, static_cast<float*>(dH), d, BT, d, f, 1.f,
                   0.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au + f, 2 * f, 1, static_cast<const float*>(Wu), d, 1, static_cast<float*>(dH), d, BT, d, f,
                   1.f, 1.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au, 1, 2 * f, static_cast<const float*>(H), d, 1, dWg, d, f, d, BT, 1.f, 0.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au + f, 1, 2 * f, static_cast<const float*>(H), d, 1, dWu, d, f, d, BT, 1.f, 0.f)) != IPTTT_OK)
      return s;
    if ((s = target_branch()) != IPTTT_OK) return s;
  }
  // the shared initial fast weight: sum over sequences (one sequence wrote it directly)
  if (B > 1) simt::sum_strips_kernel<<<ceil_div(df, 256), 256, 0, ctx->stream>>>(dW0b, dW0, (int)B, df);
  return check_launch(ctx, "batch sum launch");
}

// The backward pass with the forward recomputed into the first part of the workspace.
ipttt_status run_backward(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                          const void* W0, const void* Wt, const void* cw, int64_t B, int64_t T, int64_t d, int64_t f,
                          int64_t C, int k, float eta, ipttt_dtype dt, const void* dO, const float* dW_final,
                          void* dH, void* dX0, float* dWg, float* dWu, float* dW0, float* dWt, float* dcw, void* ws) {
  const SavedLayout SL = saved_layout(B, T, d, f, C, dt);
  const SavedPtrs sv = saved_ptrs(ws, SL);
  void* scratch = static_cast<uint8_t*>(ws) + SL.total;
  float* w_fin = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + scratch_layout(B, T, d, f, C, k, dt).dw0b);
  ipttt_status s = run_forward_saved(ctx, H, X0, Wg, Wu, W0, Wt, cw, B, T, d, f, C, k, eta, dt, sv, w_fin);
  if (s != IPTTT_OK) return s;
  return run_backward_core(ctx, H, X0, Wg, Wu, Wt, cw, B, T, d, f, C, k, eta, dt, dO, dW_final, dH, dX0, dWg, dWu,
                           dW0, dWt, dcw, sv, scratch);
}

}  // namespace
