// The layer: steps (1)-(5) in order on the context stream, and its argument validation.
// Part of the host side of libipttt (one translation unit: ipttt.cu includes the host_*.cuh
// files in order).  Everything here is internal; the C ABI is at the end of ipttt.cu.
#pragma once

#include "host_backward.cuh"

namespace {

void mark(ipttt_ctx* ctx, int call, int which, cudaStream_t stream) {
  if (call >= 0) cudaEventRecord(ctx->events[(size_t)call * kEventsPerCall + which], stream);
}

// Steps (3)-(5) from V (eta-scaled) and Z: the fused cooperative kernel when *fuse (its
// counters `ctr` already cleared), else, or when its launch is refused, the state kernel and the
// apply; *fuse tells which ran.  W_init (optional) is each sequence's starting state, else W0;
// write_first keeps W_0 in the stack Wst too (else chunk 0 reads W0 itself when W_init is NULL).
ipttt_status run_tail(ipttt_ctx* ctx, const void* V, const void* Z, const void* W0, const float* W_init, int64_t B,
                      int64_t T, int64_t d, int64_t f, int64_t C, ipttt_dtype dt, void* Wst, uint32_t* ctr, void* O,
                      float* W_final, bool write_first, int call, bool* fuse) {
  ipttt_status s = IPTTT_OK;
  const bool bf16 = dt == IPTTT_BF16;
  if (*fuse) {
    s = run_state_apply_fused(ctx, V, Z, W0, B, T, d, f, C, Wst, W_final, O, ctr, W_init, write_first);
    if (s == IPTTT_ERR_UNSUPPORTED) {
      *fuse = false;  // the cooperative launch was refused: separate kernels below
    } else if (s != IPTTT_OK) {
      return s;
    } else {
      mark(ctx, call, kEvStateEnd, ctx->stream);
      mark(ctx, call, kEvApplyEnd, ctx->stream);
      if (call >= 0) ctx->timed_fused[call] = 1;
      return IPTTT_OK;
    }
  }
  const bool skip_first = bf16 && !write_first;
  if ((s = run_state(ctx, V, Z, W0, B, T, d, f, C, dt, Wst, W_final, skip_first, W_init)) != IPTTT_OK) return s;
  mark(ctx, call, kEvStateEnd, ctx->stream);
  const void* w0_first = (skip_first && W_init == nullptr) ? W0 : nullptr;
  if ((s = run_apply(ctx, Z, Wst, B, T, d, f, C, dt, O, w0_first)) != IPTTT_OK) return s;
  mark(ctx, call, kEvApplyEnd, ctx->stream);
  return IPTTT_OK;
}

// Step 1 of the pages' three-step scheme for one range of tokens (a rank of context
// parallelism): Z and V of the range (the conv continuing from halo_in) into sv, and each
// sequence's update total S[b] = sum_i V_i^T Z_i (V eta-scaled), accumulated from zero with no
// per-chunk weight written.
ipttt_status run_totals(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu, const void* Wt,
                        const void* cw, const void* halo_in, int64_t B, int64_t T, int64_t d, int64_t f, int64_t C,
                        int k, float eta, ipttt_dtype dt, float* S, const SavedPtrs& sv) {
  ipttt_status s = IPTTT_OK;
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  if ((s = run_swiglu(ctx, H, Wg, Wu, B * T, d, f, dt, sv.z)) != IPTTT_OK) return s;
  if (Wt != nullptr && dt == IPTTT_BF16 && use_fused_target(ctx)) {
    if ((s = run_target_conv(ctx, X0, cw, Wt, B, T, d, k, eta, sv.v, halo_in)) != IPTTT_OK) return s;
  } else if (Wt != nullptr) {
    if ((s = run_conv(ctx, X0, cw, B, T, d, k, dt, sv.y, halo_in)) != IPTTT_OK) return s;
    if ((s = run_target_gemm(ctx, sv.y, Wt, B * T, d, eta, dt, sv.v)) != IPTTT_OK) return s;
  } else if ((s = run_conv(ctx, X0, cw, B, T, d, k, dt, sv.v, halo_in, eta)) != IPTTT_OK) {
    return s;
  }
  if (dt != IPTTT_BF16)  // fp32: the delta stack and the scan from zero (the stack is scratch)
    return run_state(ctx, sv.v, sv.z, nullptr, B, T, d, f, C, dt, sv.wst, S, false, nullptr);
  const int64_t n = n_chunks_of(T, C);
  CUtensorMap mv, mz, mf;
  int blocked = 0;
  if (!map_state_operands(ctx, &mv, &mz, sv.v, d, sv.z, f, B, T, d, f, use_pairs(ctx), &blocked) ||
      !map_3d_f32(ctx, &mf, S, B, d, f, 32))
    return IPTTT_ERR_CUDA;
  state::Params p{};
  p.B = (int)B;
  p.T = (int)T;
  p.d = (int)d;
  p.f = (int)f;
  p.C = (int)C;
  p.n_chunks = (int)n;
  p.m_units = ceil_div(d, state::BMD);
  p.n_units = ceil_div(f, state::BNF);
  p.units = (int)(B * p.m_units * p.n_units);
  p.skip_first = 1;
  p.no_snap = 1;  // zero start (W0 and W_init NULL), only the final state is stored
  p.blocked = blocked;
  p.st = dev_status(ctx);
  return launch_state_kernel(ctx, mv, mz, mv, mf, p);
}

// The layer on device buffers, validated by the caller.
// W_init (optional, fp32 [B, d, f]): per-sequence starting state instead of W0; halo_in /
// halo_out (optional, [B, k-1, d]): the X0 rows before this call / after it (resumed calls).
// sv (optional, with ws unused then): the training forward, which keeps the activations the
// backward pass reads (Z, [A | U], Y, V and every W_i, W_0 included) in the saved buffer.
ipttt_status run_layer(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                       const void* W0, const void* Wt, const void* cw, int64_t B, int64_t T, int64_t d, int64_t f,
                       int64_t C, int k, float eta, ipttt_dtype dt, void* O, float* W_final, void* ws,
                       const float* W_init = nullptr, const void* halo_in = nullptr, void* halo_out = nullptr,
                       const SavedPtrs* sv = nullptr) {
  if (B == 0) return IPTTT_OK;
  if (halo_out != nullptr && k > 1) {
    const int64_t nh = B * (k - 1) * d;
    dim3 g(ceil_div(nh, 256));
    if (dt == IPTTT_BF16)
      simt::halo_out_kernel<__nv_bfloat16><<<g, 256, 0, ctx->stream>>>(
          static_cast<const __nv_bfloat16*>(X0), static_cast<const __nv_bfloat16*>(halo_in),
          static_cast<__nv_bfloat16*>(halo_out), (int)B, (int)T, (int)d, k - 1);
    else
      simt::halo_out_kernel<float><<<g, 256, 0, ctx->stream>>>(static_cast<const float*>(X0),
                                                               static_cast<const float*>(halo_in),
                                                               static_cast<float*>(halo_out), (int)B, (int)T,
                                                               (int)d, k - 1);
    ipttt_status hs = check_launch(ctx, "halo launch");
    if (hs != IPTTT_OK) return hs;
  }
  if (T == 0 && W_init != nullptr) {
    const cudaError_t e = cudaMemcpyAsync(W_final, W_init, (size_t)B * d * f * sizeof(float),
                                          cudaMemcpyDeviceToDevice, ctx->stream);
    return e == cudaSuccess ? IPTTT_OK : cuda_fail(ctx, e, "state copy");
  }
  if (T == 0) {
    const int64_t df = d * f;
    dim3 g(ceil_div(df, 256), (unsigned)B);
    if (dt == IPTTT_BF16)
      simt::broadcast_state_kernel<__nv_bfloat16><<<g, 256, 0, ctx->stream>>>(static_cast<const __nv_bfloat16*>(W0),
                                                                              W_final, df);
    else
      simt::broadcast_state_kernel<float><<<g, 256, 0, ctx->stream>>>(static_cast<const float*>(W0), W_final, df);
    return check_launch(ctx, "broadcast launch");
  }
  ipttt_status s = IPTTT_OK;
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  const WsLayout L = ws_layout(B, T, d, f, C, dt);
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* Y = sv ? sv->y : base + L.y;
  void* V = sv ? sv->v : base + L.v;
  void* Z = sv ? sv->z : base + L.z;
  void* Wst = sv ? sv->wst : base + L.w;
  int call = -1;
  if (ctx->timing && ctx->timed_calls < kMaxTimedCalls) {
    call = ctx->timed_calls++;
    ctx->timed_fused[call] = 0;
  }
  mark(ctx, call, kEvStart, ctx->stream);
  // Step (2) as one kernel (the conv inside the target GEMM, Y never stored) when selected,
  // unless the training forward needs Y kept or the projection is left out; else the conv
  // kernel first (memory bound, about 0.15 ms at the 4B shape and 32k tokens)
  const bool fuse_target = Wt != nullptr && dt == IPTTT_BF16 && sv == nullptr && use_fused_target(ctx);
  mark(ctx, call, kEvConvStart, ctx->stream);
  if (!fuse_target) {
    // without W_target (the "w/o Proj" ablation) the conv writes V = eta * conv(X0) directly
    s = Wt != nullptr ? run_conv(ctx, X0, cw, B, T, d, k, dt, Y, halo_in)
                      : run_conv(ctx, X0, cw, B, T, d, k, dt, V, halo_in, eta);
    if (s != IPTTT_OK) return s;
  }
  mark(ctx, call, kEvConvEnd, ctx->stream);
  if ((s = sv ? run_swiglu_save(ctx, H, Wg, Wu, B * T, d, f, dt, Z, sv->au)
              : run_swiglu(ctx, H, Wg, Wu, B * T, d, f, dt, Z)) != IPTTT_OK)
    return s;
  mark(ctx, call, kEvSwigluEnd, ctx->stream);
  mark(ctx, call, kEvJoined, ctx->stream);
  const bool bf16 = dt == IPTTT_BF16;  // W_eff[b, 0] = W_down0: the apply reads W_down0 itself
  bool fuse = bf16 && ctx->fused_tail && ctx->coop;
  uint32_t* ctr = sv ? sv->ctr : reinterpret_cast<uint32_t*>(base + L.ctr);
  const int n_ctr = (int)(B * n_chunks_of(T, C) + 1);
  if (fuse_target) {
    if ((s = run_target_conv(ctx, X0, cw, Wt, B, T, d, k, eta, V, halo_in, fuse ? ctr : nullptr, fuse ? n_ctr : 0)) !=
        IPTTT_OK)
      return s;
  } else if (Wt != nullptr) {
    if ((s = run_target_gemm(ctx, Y, Wt, B * T, d, eta, dt, V, fuse ? ctr : nullptr, fuse ? n_ctr : 0)) != IPTTT_OK)
      return s;
  } else if (fuse) {
    const cudaError_t ez = cudaMemsetAsync(ctr, 0, (size_t)n_ctr * sizeof(uint32_t), ctx->stream);
    if (ez != cudaSuccess) return cuda_fail(ctx, ez, "counter reset");
  }
  mark(ctx, call, kEvTargetEnd, ctx->stream);
  if ((s = run_tail(ctx, V, Z, W0, W_init, B, T, d, f, C, dt, Wst, ctr, O, W_final, sv != nullptr, call, &fuse)) !=
      IPTTT_OK)
    return s;
  if (call >= 0)
    ctx->timed_launches += (bf16 ? (fuse ? 4 : 5) : 6) + ((halo_out != nullptr && k > 1) ? 1 : 0) - (Wt ? 0 : 1) -
                           (fuse_target ? 1 : 0);
  return IPTTT_OK;
}

// Validation of the device-buffer layer call (everything except the buffers' residency).
// ws_need: bytes the workspace must hold (0: the layer's own, ipttt_workspace_size()).
ipttt_status validate_layer(ipttt_ctx* ctx, const void* H, const void* X0, const void* Wg, const void* Wu,
                            const void* W0, const void* Wt, const void* cw, int64_t B, int64_t T, int64_t d,
                            int64_t f, int64_t C, int k, float eta, ipttt_dtype dt, const void* O,
                            const float* W_final, const void* ws, size_t ws_bytes, bool check_overlap,
                            size_t ws_need = 0) {
  ipttt_status s = check_shape(ctx, B, T, d, f, C, k, dt);
  if (s != IPTTT_OK) return s;
  if (!std::isfinite(eta)) {
    set_err(ctx, "eta is not finite");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B == 0) return IPTTT_OK;
  const size_t es = esize(dt);
  const size_t act = (size_t)B * T * d * es;
  struct P {
    const void* p;
    const char* n;
    bool needed;
  } ptrs[] = {{H, "H", T > 0},        {X0, "X0", T > 0},  {Wg, "W_gate", T > 0}, {Wu, "W_up", T > 0},
              {W0, "W_down0", true},  {Wt, "W_target", false}, {cw, "conv_w", T > 0}, {O, "O", T > 0},
              {W_final, "W_final", true}, {ws, "workspace", T > 0}};
  for (const P& q : ptrs) {
    if (!q.needed) continue;
    if (!q.p) {
      set_err(ctx, "%s is NULL", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
    if (!aligned16(q.p)) {
      set_err(ctx, "%s is not 16-byte aligned", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  if (Wt != nullptr && !aligned16(Wt)) {
    set_err(ctx, "W_target is not 16-byte aligned");
    return IPTTT_ERR_INVALID_ARG;
  }
  const size_t need = ws_need != 0 ? ws_need : ws_layout(B, T, d, f, C, dt).total;
  if (T > 0 && ws_bytes < need) {
    set_err(ctx, "workspace too small: %zu < %zu bytes", ws_bytes, need);
    return IPTTT_ERR_WORKSPACE;
  }
  if (check_overlap) {
    const size_t wdf = (size_t)d * f * es;
    std::vector<Region> all = {{H, act, "H"},
                               {X0, act, "X0"},
                               {Wg, wdf, "W_gate"},
                               {Wu, wdf, "W_up"},
                               {W0, wdf, "W_down0"},
                               {Wt, (size_t)d * d * es, "W_target"},
                               {cw, (size_t)d * k * es, "conv_w"},
                               {O, act, "O"},
                               {W_final, (size_t)B * d * f * 4, "W_final"},
                               {ws, T > 0 ? need : 0, "workspace"}};
    std::vector<Region> outs = {all[7], all[8], all[9]};
    std::string what;
    if (find_overlap(outs, all, what)) {
      set_err(ctx, "overlapping buffers: %s", what.c_str());
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  return IPTTT_OK;
}

}  // namespace
