// Host orchestration and C ABI of the In-Place TTT fast-weight SwiGLU layer (see
// include/ipttt.h for the contract).  bf16 runs on the tcgen05 kernels (tc_gemm.cuh,
// tc_state.cuh); fp32 runs on the CUDA-core kernels (simt.cuh).  Nothing here computes on
// the host: every step of the layer is a kernel launch on the context's stream.
//
// The host code is split over host_context.cuh (context, checks, tensor maps), host_steps.cuh
// (one launcher per step), host_backward.cuh (the backward pass and buffer layouts) and
// host_layer.cuh (the layer call); this file holds the C ABI.
#include "host_layer.cuh"

// ====================================================================== C ABI

extern "C" {

const char* ipttt_version(void) { return "0.1.0"; }

const char* ipttt_status_string(ipttt_status s) {
  switch (s) {
    case IPTTT_OK: return "IPTTT_OK";
    case IPTTT_ERR_INVALID_ARG: return "IPTTT_ERR_INVALID_ARG";
    case IPTTT_ERR_UNSUPPORTED: return "IPTTT_ERR_UNSUPPORTED";
    case IPTTT_ERR_WORKSPACE: return "IPTTT_ERR_WORKSPACE";
    case IPTTT_ERR_CUDA: return "IPTTT_ERR_CUDA";
    case IPTTT_ERR_TIMEOUT: return "IPTTT_ERR_TIMEOUT";
  }
  return "IPTTT_ERR_UNKNOWN";
}

ipttt_status ipttt_create(ipttt_ctx** out, int device, void* stream) {
  if (!out) return IPTTT_ERR_INVALID_ARG;
  *out = nullptr;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return IPTTT_ERR_INVALID_ARG;
  }
  ipttt_ctx* ctx = new ipttt_ctx();
  ctx->device = device;
  ctx->stream = static_cast<cudaStream_t>(stream);
  DeviceGuard g(device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    delete ctx;
    return IPTTT_ERR_CUDA;
  }
  ctx->sm_count = prop.multiProcessorCount;
  ctx->coop = prop.cooperativeLaunch != 0;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete ctx;
    return IPTTT_ERR_CUDA;
  }
  ctx->encode = reinterpret_cast<EncodeTiledFn>(fn);
  if (cudaMalloc(&ctx->status, 2 * sizeof(uint32_t)) != cudaSuccess) {
    delete ctx;
    return IPTTT_ERR_CUDA;
  }
  if (cudaMemset(ctx->status, 0, 2 * sizeof(uint32_t)) != cudaSuccess) {
    cudaFree(ctx->status);
    delete ctx;
    return IPTTT_ERR_CUDA;
  }
  if (cudaStreamCreateWithFlags(&ctx->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->copy_out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->h_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->h_join, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->b_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->b_join, cudaEventDisableTiming) != cudaSuccess) {
    ipttt_destroy(ctx);
    return IPTTT_ERR_CUDA;
  }
  ctx->piece_ev.assign(2 * kMaxPieces, nullptr);
  for (auto& e : ctx->piece_ev) {
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      e = nullptr;
      ipttt_destroy(ctx);
      return IPTTT_ERR_CUDA;
    }
  }
  ctx->events.resize((size_t)kMaxTimedCalls * kEventsPerCall, nullptr);
  ctx->timed_fused.assign(kMaxTimedCalls, 0);
  for (auto& e : ctx->events) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      ipttt_destroy(ctx);
      return IPTTT_ERR_CUDA;
    }
  }
  *out = ctx;
  return IPTTT_OK;
}

ipttt_status ipttt_set_stream(ipttt_ctx* ctx, void* stream) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->stream = static_cast<cudaStream_t>(stream);
  return IPTTT_OK;
}

ipttt_status ipttt_set_cta_pairs(ipttt_ctx* ctx, int enable) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->cta_pairs = enable != 0;
  return IPTTT_OK;
}

ipttt_status ipttt_set_target_shift(ipttt_ctx* ctx, int shift) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  if (shift != 0 && shift != 1) {
    set_err(ctx, "target shift must be 0 or 1 (got %d)", shift);
    return IPTTT_ERR_INVALID_ARG;
  }
  ctx->target_shift = shift;
  return IPTTT_OK;
}

ipttt_status ipttt_set_fused_target(ipttt_ctx* ctx, int enable) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->fused_target = enable != 0;
  return IPTTT_OK;
}

ipttt_status ipttt_set_fused_tail(ipttt_ctx* ctx, int enable) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->fused_tail = enable != 0;
  return IPTTT_OK;
}

ipttt_status ipttt_set_apply_tiles(ipttt_ctx* ctx, int halves) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  if (halves < 0 || halves > 2) {
    set_err(ctx, "apply tiles: halves = %d (0 = per call, 1 = 256 x 256, 2 = 256 x 512)", halves);
    return IPTTT_ERR_INVALID_ARG;
  }
  ctx->apply_halves = halves;
  return IPTTT_OK;
}

ipttt_status ipttt_set_wait_limit_ns(ipttt_ctx* ctx, uint64_t ns) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  if (ns == 0) {
    set_err(ctx, "wait limit must be > 0");
    return IPTTT_ERR_INVALID_ARG;
  }
  ctx->wait_limit_ns = ns;
  return IPTTT_OK;
}

ipttt_status ipttt_sync(ipttt_ctx* ctx) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream synchronize");
  uint32_t h[2] = {0, 0};
  e = cudaMemcpyAsync(h, ctx->status, sizeof(h), cudaMemcpyDeviceToHost, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
  if (h[0] != 0) {
    const uint32_t zero[2] = {0, 0};
    e = cudaMemcpyAsync(ctx->status, zero, sizeof(zero), cudaMemcpyHostToDevice, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "status reset");
    set_err(ctx, "device wait gave up after %llu ns (site 0x%x)", (unsigned long long)ctx->wait_limit_ns, h[1]);
    return h[0] == kDevStatusTimeout ? IPTTT_ERR_TIMEOUT : IPTTT_ERR_CUDA;
  }
  return IPTTT_OK;
}

const char* ipttt_last_error(const ipttt_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

void ipttt_destroy(ipttt_ctx* ctx) {
  if (!ctx) return;
  DeviceGuard g(ctx->device);
  for (auto& e : ctx->events)
    if (e) cudaEventDestroy(e);
  for (auto& e : ctx->piece_ev)
    if (e) cudaEventDestroy(e);
  if (ctx->h_fork) cudaEventDestroy(ctx->h_fork);
  if (ctx->h_join) cudaEventDestroy(ctx->h_join);
  if (ctx->b_fork) cudaEventDestroy(ctx->b_fork);
  if (ctx->b_join) cudaEventDestroy(ctx->b_join);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  if (ctx->copy_in) cudaStreamDestroy(ctx->copy_in);
  if (ctx->copy_out) cudaStreamDestroy(ctx->copy_out);
  if (ctx->status) cudaFree(ctx->status);
  delete ctx;
}

ipttt_status ipttt_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, ipttt_dtype dt,
                                  size_t* bytes) {
  if (!bytes) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_shape(nullptr, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  *bytes = ws_layout(B, T, d, d_ff, C, dt).total;
  return IPTTT_OK;
}

ipttt_status ipttt_host_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                       ipttt_dtype dt, size_t* bytes) {
  if (!bytes) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_shape(nullptr, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  *bytes = host_layout(B, T, d, d_ff, C, k, dt).total;
  return IPTTT_OK;
}

int64_t ipttt_layer_launches(int64_t B, int64_t T, ipttt_dtype dt) {
  if (B <= 0) return 0;
  if (T <= 0) return 1;
  return dt == IPTTT_BF16 ? 4 : 6;
}

ipttt_status ipttt_layer_forward(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate, const void* W_up,
                                 const void* W_down0, const void* W_target, const void* conv_w, int64_t B, int64_t T,
                                 int64_t d, int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dt, void* O,
                                 float* W_final, void* ws, size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = validate_layer(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt,
                                  O, W_final, ws, ws_bytes, true);
  if (s != IPTTT_OK) return s;
  DeviceGuard g(ctx->device);
  return run_layer(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, O, W_final, ws);
}

ipttt_status ipttt_backward_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                           ipttt_dtype dt, size_t* bytes) {
  if (!bytes) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_shape(nullptr, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  *bytes = bwd_total(B, T, d, d_ff, C, k, dt);
  return IPTTT_OK;
}

namespace {

// Argument checks shared by the two backward entries.  W_down0 is read only by the recomputing
// entry (need_w0); `saved` (the second entry's saved activations, NULL for the first) is an
// input that the call overwrites.
ipttt_status check_backward(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate, const void* W_up,
                            const void* W_down0, bool need_w0, const void* W_target, const void* conv_w, int64_t B,
                            int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dt,
                            const void* dO, const float* dW_final, void* dH, void* dX0, float* dW_gate, float* dW_up,
                            float* dW_down0, float* dW_target, float* dconv_w, const void* saved, size_t saved_need,
                            size_t saved_bytes, void* ws, size_t ws_need, size_t ws_bytes) {
  ipttt_status s = check_shape(ctx, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  if (!std::isfinite(eta)) {
    set_err(ctx, "eta is not finite");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B * T >= (int64_t)1 << 31) {
    set_err(ctx, "B*T must be < 2^31");
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (B > 65535 || (T + simt::CONVX_ROWS - 1) / simt::CONVX_ROWS > 65535) {
    set_err(ctx, "B (%lld) and ceil(T/%d) must be <= 65535", (long long)B, simt::CONVX_ROWS);
    return IPTTT_ERR_UNSUPPORTED;
  }
  const bool work = B > 0 && T > 0;
  const bool with_saved = saved_need > 0;
  struct P {
    const void* p;
    const char* n;
    bool needed;
  } ptrs[] = {{H, "H", work},         {X0, "X0", work},         {W_gate, "W_gate", work}, {W_up, "W_up", work},
              {W_down0, "W_down0", work && need_w0}, {conv_w, "conv_w", work}, {dO, "dO", work}, {dH, "dH", work},
              {dX0, "dX0", work},     {dW_gate, "dW_gate", true}, {dW_up, "dW_up", true}, {dW_down0, "dW_down0", true},
              {dconv_w, "dconv_w", true}, {ws, "workspace", work}, {W_target, "W_target", false},
              {dW_target, "dW_target", W_target != nullptr}, {dW_final, "dW_final", false},
              {saved, "saved", work && with_saved}};
  for (const P& q : ptrs) {
    if (q.needed && !q.p) {
      set_err(ctx, "%s is NULL", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
    if (q.p && !aligned16(q.p)) {
      set_err(ctx, "%s is not 16-byte aligned", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  if (work && ws_bytes < ws_need) {
    set_err(ctx, "workspace too small: %zu < %zu bytes", ws_bytes, ws_need);
    return IPTTT_ERR_WORKSPACE;
  }
  if (work && with_saved && saved_bytes < saved_need) {
    set_err(ctx, "saved-activation buffer too small: %zu < %zu bytes", saved_bytes, saved_need);
    return IPTTT_ERR_WORKSPACE;
  }
  const size_t es = esize(dt);
  const size_t act = (size_t)B * T * d * es, wdf = (size_t)d * d_ff * es, gdf = (size_t)d * d_ff * 4;
  std::vector<Region> all = {{H, act, "H"},
                             {X0, act, "X0"},
                             {W_gate, wdf, "W_gate"},
                             {W_up, wdf, "W_up"},
                             {W_down0, need_w0 ? wdf : 0, "W_down0"},
                             {W_target, (size_t)d * d * es, "W_target"},
                             {conv_w, (size_t)d * k * es, "conv_w"},
                             {dO, act, "dO"},
                             {dW_final, (size_t)B * gdf, "dW_final"},
                             {dH, act, "dH"},
                             {dX0, act, "dX0"},
                             {dW_gate, gdf, "dW_gate"},
                             {dW_up, gdf, "dW_up"},
                             {dW_down0, gdf, "dW_down0"},
                             {dW_target, W_target ? (size_t)d * d * 4 : 0, "dW_target"},
                             {dconv_w, (size_t)d * k * 4, "dconv_w"},
                             {ws, work ? ws_need : 0, "workspace"},
                             {saved, work && with_saved ? saved_need : 0, "saved"}};
  std::vector<Region> outs(all.begin() + 9, all.end());
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  return IPTTT_OK;
}

// No tokens: every gradient is zero except dW_down0 = sum_b dW_final[b].
ipttt_status backward_no_tokens(ipttt_ctx* ctx, int64_t B, int64_t d, int64_t d_ff, int k, const float* dW_final,
                                float* dW_gate, float* dW_up, float* dW_down0, float* dW_target, float* dconv_w) {
  const size_t gdf = (size_t)d * d_ff * 4;
  cudaError_t e;
  if ((e = cudaMemsetAsync(dW_gate, 0, gdf, ctx->stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(dW_up, 0, gdf, ctx->stream)) != cudaSuccess ||
      (dW_target && (e = cudaMemsetAsync(dW_target, 0, (size_t)d * d * 4, ctx->stream)) != cudaSuccess) ||
      (e = cudaMemsetAsync(dconv_w, 0, (size_t)d * k * 4, ctx->stream)) != cudaSuccess)
    return cuda_fail(ctx, e, "gradient clear");
  if (dW_final != nullptr && B > 0) {
    simt::sum_strips_kernel<<<ceil_div(d * d_ff, 256), 256, 0, ctx->stream>>>(dW_final, dW_down0, (int)B, d * d_ff);
    return check_launch(ctx, "empty backward");
  }
  if ((e = cudaMemsetAsync(dW_down0, 0, gdf, ctx->stream)) != cudaSuccess) return cuda_fail(ctx, e, "gradient clear");
  return IPTTT_OK;
}

}  // namespace

ipttt_status ipttt_layer_backward(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                  const void* W_up, const void* W_down0, const void* W_target, const void* conv_w,
                                  int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                  ipttt_dtype dt, const void* dO, const float* dW_final, void* dH, void* dX0,
                                  float* dW_gate, float* dW_up, float* dW_down0, float* dW_target, float* dconv_w,
                                  void* ws, size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_backward(ctx, H, X0, W_gate, W_up, W_down0, true, W_target, conv_w, B, T, d, d_ff, C,
                                        k, eta, dt, dO, dW_final, dH, dX0, dW_gate, dW_up, dW_down0, dW_target,
                                        dconv_w, nullptr, 0, 0, ws, bwd_total(B, T, d, d_ff, C, k, dt), ws_bytes);
  if (s != IPTTT_OK) return s;
  DeviceGuard g(ctx->device);
  if (B == 0 || T == 0)
    return backward_no_tokens(ctx, B, d, d_ff, k, dW_final, dW_gate, dW_up, dW_down0, dW_target, dconv_w);
  return run_backward(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, dO, dW_final,
                      dH, dX0, dW_gate, dW_up, dW_down0, dW_target, dconv_w, ws);
}

ipttt_status ipttt_saved_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, ipttt_dtype dt,
                              size_t* bytes) {
  if (!bytes) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_shape(nullptr, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  *bytes = saved_layout(B, T, d, d_ff, C, dt).total;
  return IPTTT_OK;
}

ipttt_status ipttt_backward_saved_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                                 ipttt_dtype dt, size_t* bytes) {
  if (!bytes) return IPTTT_ERR_INVALID_ARG;
  const ipttt_status s = check_shape(nullptr, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  *bytes = scratch_layout(B, T, d, d_ff, C, k, dt).total;
  return IPTTT_OK;
}

ipttt_status ipttt_layer_forward_train(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                       const void* W_up, const void* W_down0, const void* W_target,
                                       const void* conv_w, int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C,
                                       int k, float eta, ipttt_dtype dt, void* O, float* W_final, void* saved,
                                       size_t saved_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  const size_t need = saved_layout(B, T, d, d_ff, C, dt).total;
  ipttt_status s = validate_layer(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt,
                                  O, W_final, saved, saved_bytes, true, need);
  if (s != IPTTT_OK) return s;
  DeviceGuard g(ctx->device);
  if (B == 0 || T == 0)
    return run_layer(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, O, W_final,
                     saved);
  const SavedPtrs sv = saved_ptrs(saved, saved_layout(B, T, d, d_ff, C, dt));
  return run_layer(ctx, H, X0, W_gate, W_up, W_down0, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, O, W_final,
                   nullptr, nullptr, nullptr, nullptr, &sv);
}

ipttt_status ipttt_layer_backward_saved(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                        const void* W_up, const void* W_target, const void* conv_w, int64_t B,
                                        int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                        ipttt_dtype dt, void* saved, size_t saved_bytes, const void* dO,
                                        const float* dW_final, void* dH, void* dX0, float* dW_gate, float* dW_up,
                                        float* dW_down0, float* dW_target, float* dconv_w, void* ws,
                                        size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  const SavedLayout SL = saved_layout(B, T, d, d_ff, C, dt);
  const ipttt_status s =
      check_backward(ctx, H, X0, W_gate, W_up, nullptr, false, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, dO,
                     dW_final, dH, dX0, dW_gate, dW_up, dW_down0, dW_target, dconv_w, saved, SL.total, saved_bytes, ws,
                     scratch_layout(B, T, d, d_ff, C, k, dt).total, ws_bytes);
  if (s != IPTTT_OK) return s;
  DeviceGuard g(ctx->device);
  if (B == 0 || T == 0)
    return backward_no_tokens(ctx, B, d, d_ff, k, dW_final, dW_gate, dW_up, dW_down0, dW_target, dconv_w);
  return run_backward_core(ctx, H, X0, W_gate, W_up, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, dO, dW_final, dH,
                           dX0, dW_gate, dW_up, dW_down0, dW_target, dconv_w, saved_ptrs(saved, SL), ws);
}

ipttt_status ipttt_layer_totals(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate, const void* W_up,
                                const void* W_target, const void* conv_w, const void* X0_halo, int64_t B, int64_t T,
                                int64_t d, int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dt, float* S,
                                void* saved, size_t saved_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  if (ctx->target_shift != 0) {
    set_err(ctx, "the shifted target window needs the next rank's first X0 row: not supported by layer_totals");
    return IPTTT_ERR_UNSUPPORTED;
  }
  const SavedLayout SL = saved_layout(B, T, d, d_ff, C, dt);
  ipttt_status s = check_shape(ctx, B, T, d, d_ff, C, k, dt);
  if (s != IPTTT_OK) return s;
  if (!std::isfinite(eta)) {
    set_err(ctx, "eta is not finite");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B == 0) return IPTTT_OK;
  const bool work = T > 0;
  struct P {
    const void* p;
    const char* n;
    bool needed;
  } ptrs[] = {{H, "H", work},           {X0, "X0", work},       {W_gate, "W_gate", work}, {W_up, "W_up", work},
              {conv_w, "conv_w", work}, {saved, "saved", work}, {S, "S", true},           {W_target, "W_target", false},
              {X0_halo, "X0_halo", false}};
  for (const P& q : ptrs) {
    if (q.needed && !q.p) {
      set_err(ctx, "%s is NULL", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
    if (q.p && !aligned16(q.p)) {
      set_err(ctx, "%s is not 16-byte aligned", q.n);
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  if (work && saved_bytes < SL.total) {
    set_err(ctx, "saved-activation buffer too small: %zu < %zu bytes", saved_bytes, SL.total);
    return IPTTT_ERR_WORKSPACE;
  }
  const size_t es = esize(dt);
  const size_t act = (size_t)B * T * d * es, wdf = (size_t)d * d_ff * es;
  std::vector<Region> all = {{H, act, "H"},
                             {X0, act, "X0"},
                             {W_gate, wdf, "W_gate"},
                             {W_up, wdf, "W_up"},
                             {W_target, (size_t)d * d * es, "W_target"},
                             {conv_w, (size_t)d * k * es, "conv_w"},
                             {X0_halo, (size_t)B * (k - 1) * d * es, "X0_halo"},
                             {S, (size_t)B * d * d_ff * 4, "S"},
                             {saved, T > 0 ? SL.total : 0, "saved"}};
  std::vector<Region> outs = {all[7], all[8]};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (T == 0) {
    const cudaError_t e = cudaMemsetAsync(S, 0, (size_t)B * d * d_ff * 4, ctx->stream);
    return e == cudaSuccess ? IPTTT_OK : cuda_fail(ctx, e, "total clear");
  }
  return run_totals(ctx, H, X0, W_gate, W_up, W_target, conv_w, X0_halo, B, T, d, d_ff, C, k, eta, dt, S,
                    saved_ptrs(saved, SL));
}

ipttt_status ipttt_layer_apply_saved(ipttt_ctx* ctx, const float* W_init, int64_t B, int64_t T, int64_t d,
                                     int64_t d_ff, int64_t C, ipttt_dtype dt, void* saved, size_t saved_bytes,
                                     void* O, float* W_final) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, T, d, d_ff, C, 1, dt);
  if (s != IPTTT_OK) return s;
  if (B == 0) return IPTTT_OK;
  const SavedLayout SL = saved_layout(B, T, d, d_ff, C, dt);
  const bool work = T > 0;
  if (!W_init || !W_final || !aligned16(W_init) || !aligned16(W_final) ||
      (work && (!saved || !O || !aligned16(saved) || !aligned16(O)))) {
    set_err(ctx, "apply_saved: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (work && saved_bytes < SL.total) {
    set_err(ctx, "saved-activation buffer too small: %zu < %zu bytes", saved_bytes, SL.total);
    return IPTTT_ERR_WORKSPACE;
  }
  const size_t state = (size_t)B * d * d_ff * 4;
  std::vector<Region> all = {{saved, work ? SL.total : 0, "saved"}, {O, work ? (size_t)B * T * d * esize(dt) : 0, "O"},
                             {W_init, state, "W_init"}};
  std::vector<Region> outs = {all[1]};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  // W_final may be W_init itself (each state element is read before it is rewritten)
  all.pop_back();
  std::vector<Region> st_out = {{W_final, state, "W_final"}};
  if (W_final != W_init) all.push_back({W_init, state, "W_init"});
  if (find_overlap(st_out, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  cudaError_t e;
  if (!work) {
    if (W_final == W_init) return IPTTT_OK;
    e = cudaMemcpyAsync(W_final, W_init, state, cudaMemcpyDeviceToDevice, ctx->stream);
    return e == cudaSuccess ? IPTTT_OK : cuda_fail(ctx, e, "state copy");
  }
  const bool bf16 = dt == IPTTT_BF16;
  if (bf16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  const SavedPtrs sv = saved_ptrs(saved, SL);
  bool fuse = bf16 && ctx->fused_tail && ctx->coop;
  if (fuse && (e = cudaMemsetAsync(sv.ctr, 0, (size_t)(B * n_chunks_of(T, C) + 1) * 4, ctx->stream)) != cudaSuccess)
    return cuda_fail(ctx, e, "counter reset");
  return run_tail(ctx, sv.v, sv.z, nullptr, W_init, B, T, d, d_ff, C, dt, sv.wst, sv.ctr, O, W_final, false, -1,
                  &fuse);
}

ipttt_status ipttt_prefix_step(ipttt_ctx* ctx, const float* P_in, const void* W_down0, const float* S, int64_t B,
                               int64_t d, int64_t d_ff, ipttt_dtype dt, int64_t first, int64_t count, float* P_out) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, 1, d, d_ff, 1, 1, dt, false);
  if (s != IPTTT_OK) return s;
  const int64_t n = B * d * d_ff;
  if (first < 0 || count < 0 || first > n || count > n - first) {
    set_err(ctx, "prefix_step: elements [%lld, %lld) outside the state of %lld", (long long)first,
            (long long)(first + count), (long long)n);
    return IPTTT_ERR_INVALID_ARG;
  }
  if (count == 0) return IPTTT_OK;
  if (!P_out || (!P_in && !W_down0)) {
    set_err(ctx, "prefix_step: P_out and one of P_in / W_down0 are needed");
    return IPTTT_ERR_INVALID_ARG;
  }
  auto al4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!al4(P_out) || (P_in && !al4(P_in)) || (S && !al4(S)) || (W_down0 && !al4(W_down0) && dt == IPTTT_F32) ||
      (W_down0 && (reinterpret_cast<uintptr_t>(W_down0) & 1u))) {
    set_err(ctx, "prefix_step: misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  // P_out may be P_in or S itself (element for element), but must not partly overlap them or W_down0
  const size_t state = (size_t)n * 4;
  std::vector<Region> all;
  if (P_in && P_in != P_out) all.push_back({P_in, state, "P_in"});
  if (S && S != P_out) all.push_back({S, state, "S"});
  if (W_down0) all.push_back({W_down0, (size_t)d * d_ff * esize(dt), "W_down0"});
  std::vector<Region> outs = {{P_out, state, "P_out"}};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  const int vec = (first % 4 == 0 && count % 4 == 0 && aligned16(P_out) && (!P_in || aligned16(P_in)) &&
                   (!S || aligned16(S)))
                      ? 1
                      : 0;
  const int64_t items = vec ? count / 4 : count;
  const int64_t cap = (int64_t)ctx->sm_count * 8;
  const int64_t blocks = ceil_div(items, 256) < cap ? ceil_div(items, 256) : cap;
  if (dt == IPTTT_BF16)
    simt::prefix_step_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, ctx->stream>>>(
        P_in, static_cast<const __nv_bfloat16*>(W_down0), S, P_out, first, count, d * d_ff, vec);
  else
    simt::prefix_step_kernel<float><<<(unsigned)blocks, 256, 0, ctx->stream>>>(
        P_in, static_cast<const float*>(W_down0), S, P_out, first, count, d * d_ff, vec);
  return check_launch(ctx, "prefix step launch");
}

ipttt_status ipttt_layer_forward_resume(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                        const void* W_up, const void* W_target, const void* conv_w,
                                        const float* W_state, const void* X0_halo, int64_t B, int64_t T, int64_t d,
                                        int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dt, void* O,
                                        float* W_state_out, void* X0_halo_out, void* ws, size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  if (ctx->target_shift != 0) {
    set_err(ctx, "the shifted target window needs the next call's first X0 row: not supported by resumed calls");
    return IPTTT_ERR_UNSUPPORTED;
  }
  // the shared-weight checks of the plain layer, with W_state standing in for W_down0
  ipttt_status s = validate_layer(ctx, H, X0, W_gate, W_up, W_state, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt,
                                  O, W_state_out, ws, ws_bytes, false);
  if (s != IPTTT_OK) return s;
  if (B == 0) return IPTTT_OK;
  if ((X0_halo && !aligned16(X0_halo)) || (X0_halo_out && !aligned16(X0_halo_out))) {
    set_err(ctx, "halo buffer is not 16-byte aligned");
    return IPTTT_ERR_INVALID_ARG;
  }
  const size_t es = esize(dt);
  const size_t act = (size_t)B * T * d * es, wdf = (size_t)d * d_ff * es, state = (size_t)B * d * d_ff * 4;
  const size_t halo = (size_t)B * (k - 1) * d * es;
  const WsLayout L = ws_layout(B, T, d, d_ff, C, dt);
  std::vector<Region> all = {{H, act, "H"},
                             {X0, act, "X0"},
                             {W_gate, wdf, "W_gate"},
                             {W_up, wdf, "W_up"},
                             {W_target, (size_t)d * d * es, "W_target"},
                             {conv_w, (size_t)d * k * es, "conv_w"},
                             {X0_halo, halo, "X0_halo"},
                             {O, act, "O"},
                             {X0_halo_out, halo, "X0_halo_out"},
                             {ws, T > 0 ? L.total : 0, "workspace"}};
  std::vector<Region> outs = {all[7], all[8], all[9]};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  // W_state_out may be W_state itself (each state element is read before it is rewritten), but
  // must not partly overlap it or touch any other buffer
  all.push_back({W_state, state, "W_state"});
  std::vector<Region> st_out = {{W_state_out, state, "W_state_out"}};
  if (W_state_out == W_state) all.pop_back();
  if (find_overlap(st_out, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  return run_layer(ctx, H, X0, W_gate, W_up, nullptr, W_target, conv_w, B, T, d, d_ff, C, k, eta, dt, O,
                   W_state_out, ws, W_state, X0_halo, X0_halo_out);
}

ipttt_status ipttt_layer_forward_host(ipttt_ctx* ctx, const void* H_host, const void* X0_host, const void* W_gate,
                                      const void* W_up, const void* W_down0, const void* W_target, const void* conv_w,
                                      int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                      ipttt_dtype dt, void* O_host, float* W_final_host, void* ws, size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  size_t need = 0;
  ipttt_status s = ipttt_host_workspace_size(B, T, d, d_ff, C, k, dt, &need);
  if (s != IPTTT_OK) {
    check_shape(ctx, B, T, d, d_ff, C, k, dt);
    return s;
  }
  if (B == 0) return IPTTT_OK;
  if (!ws || ws_bytes < need || !aligned16(ws)) {
    set_err(ctx, "workspace missing, misaligned or too small: %zu < %zu bytes", ws_bytes, need);
    return IPTTT_ERR_WORKSPACE;
  }
  if ((T > 0 && (!H_host || !X0_host || !O_host)) || !W_final_host) {
    set_err(ctx, "host buffer is NULL");
    return IPTTT_ERR_INVALID_ARG;
  }
  const size_t es = esize(dt);
  const HostLayout HL = host_layout(B, T, d, d_ff, C, k, dt);
  const int64_t P = HL.piece;
  if (ctx->target_shift != 0 && T > P) {
    set_err(ctx, "the shifted target window needs the next piece's first X0 row: T=%lld spans pieces of %lld tokens",
            (long long)T, (long long)P);
    return IPTTT_ERR_UNSUPPORTED;
  }
  const size_t layer_ws = ws_layout(B, P, d, d_ff, C, dt).total;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint8_t* Hd = base + HL.h;
  uint8_t* Xd = base + HL.x;
  uint8_t* Od = base + HL.o;
  float* Wst = reinterpret_cast<float*>(base + HL.w);
  void* halo[2] = {base + HL.halo0, base + HL.halo1};
  s = validate_layer(ctx, P > 0 ? Hd : nullptr, P > 0 ? Xd : nullptr, W_gate, W_up, W_down0, W_target, conv_w, B, P, d,
                     d_ff, C, k, eta, dt, P > 0 ? Od : nullptr, Wst, ws, layer_ws, false);
  if (s != IPTTT_OK) return s;
  DeviceGuard g(ctx->device);
  cudaError_t e;
  const size_t state_bytes = (size_t)B * d * d_ff * 4;
  if (T == 0) {  // W_final[b] = W_down0
    if ((s = run_layer(ctx, nullptr, nullptr, W_gate, W_up, W_down0, W_target, conv_w, B, 0, d, d_ff, C, k, eta, dt,
                       nullptr, Wst, ws)) != IPTTT_OK)
      return s;
    if ((e = cudaMemcpyAsync(W_final_host, Wst, state_bytes, cudaMemcpyDeviceToHost, ctx->stream)) != cudaSuccess)
      return cuda_fail(ctx, e, "W_final download");
    return IPTTT_OK;
  }
  // fork the copy streams from the caller's stream, and start every sequence from W_down0
  if ((e = cudaEventRecord(ctx->h_fork, ctx->stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ctx->copy_in, ctx->h_fork, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ctx->copy_out, ctx->h_fork, 0)) != cudaSuccess)
    return cuda_fail(ctx, e, "copy fork");
  if ((s = run_layer(ctx, nullptr, nullptr, W_gate, W_up, W_down0, W_target, conv_w, B, 0, d, d_ff, C, k, eta, dt,
                     nullptr, Wst, ws)) != IPTTT_OK)
    return s;
  const size_t row_bytes = (size_t)T * d * es;  // one sequence in the host arrays
  // Pieces of P tokens, except that when there are several, the last P tokens (or what remains)
  // go in halves of halves down to C: after the last upload only a short piece computes and
  // downloads before the final state does.  Every piece but the last is a multiple of C.
  int64_t lens[kMaxPieces];
  int n_pieces = 0;
  {
    int64_t rem = T;
    while (rem > P) {
      lens[n_pieces++] = P;
      rem -= P;
    }
    if (n_pieces > 0) {
      while (rem > C && n_pieces + 1 < kMaxPieces) {
        const int64_t h = (rem / 2 + C - 1) / C * C;  // a multiple of C, at least half
        if (h >= rem) break;
        lens[n_pieces++] = h;
        rem -= h;
      }
    }
    lens[n_pieces++] = rem;
  }
  int64_t lo = 0;
  for (int j = 0; j < n_pieces; lo += lens[j], ++j) {
    const int64_t len = lens[j];
    const size_t off = (size_t)B * lo * d * es;   // piece j's [B, len, d] block of the staging
    const size_t width = (size_t)len * d * es;
    cudaEvent_t in_done = ctx->piece_ev[2 * j], comp_done = ctx->piece_ev[2 * j + 1];
    const uint8_t* hsrc = static_cast<const uint8_t*>(H_host) + (size_t)lo * d * es;
    const uint8_t* xsrc = static_cast<const uint8_t*>(X0_host) + (size_t)lo * d * es;
    if ((e = cudaMemcpy2DAsync(Hd + off, width, hsrc, row_bytes, width, (size_t)B, cudaMemcpyHostToDevice,
                               ctx->copy_in)) != cudaSuccess ||
        (e = cudaMemcpy2DAsync(Xd + off, width, xsrc, row_bytes, width, (size_t)B, cudaMemcpyHostToDevice,
                               ctx->copy_in)) != cudaSuccess ||
        (e = cudaEventRecord(in_done, ctx->copy_in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->stream, in_done, 0)) != cudaSuccess)
      return cuda_fail(ctx, e, "piece upload");
    // continue every sequence from the state and conv halo the previous piece left
    if ((s = run_layer(ctx, Hd + off, Xd + off, W_gate, W_up, nullptr, W_target, conv_w, B, len, d, d_ff, C, k, eta,
                       dt, Od + off, Wst, ws, Wst, j > 0 ? halo[j & 1] : nullptr, halo[(j + 1) & 1])) != IPTTT_OK)
      return s;
    uint8_t* odst = static_cast<uint8_t*>(O_host) + (size_t)lo * d * es;
    if ((e = cudaEventRecord(comp_done, ctx->stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(ctx->copy_out, comp_done, 0)) != cudaSuccess ||
        (e = cudaMemcpy2DAsync(odst, row_bytes, Od + off, width, width, (size_t)B, cudaMemcpyDeviceToHost,
                               ctx->copy_out)) != cudaSuccess)
      return cuda_fail(ctx, e, "piece download");
  }
  // the final state follows the last piece on copy_out; the caller's stream joins both copy streams
  if ((e = cudaMemcpyAsync(W_final_host, Wst, state_bytes, cudaMemcpyDeviceToHost, ctx->copy_out)) != cudaSuccess ||
      (e = cudaEventRecord(ctx->h_join, ctx->copy_out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ctx->stream, ctx->h_join, 0)) != cudaSuccess ||
      (e = cudaEventRecord(ctx->h_join, ctx->copy_in)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ctx->stream, ctx->h_join, 0)) != cudaSuccess)
    return cuda_fail(ctx, e, "copy join");
  return IPTTT_OK;
}

ipttt_status ipttt_swiglu(ipttt_ctx* ctx, const void* H, const void* W_gate, const void* W_up, int64_t rows, int64_t d,
                          int64_t d_ff, ipttt_dtype dt, void* Z) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, rows, 1, d, d_ff, 1, 1, dt, false);
  if (s != IPTTT_OK) return s;
  if (rows == 0) return IPTTT_OK;
  if (!H || !W_gate || !W_up || !Z || !aligned16(H) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(Z)) {
    set_err(ctx, "swiglu: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  return run_swiglu(ctx, H, W_gate, W_up, rows, d, d_ff, dt, Z);
}

ipttt_status ipttt_target(ipttt_ctx* ctx, const void* X0, const void* conv_w, const void* W_target, int64_t B,
                          int64_t T, int64_t d, int k, float scale, ipttt_dtype dt, void* Y, void* V) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, T, d, 8, 1, k, dt, false);
  if (s != IPTTT_OK) return s;
  if (B == 0 || T == 0) return IPTTT_OK;
  if (!X0 || !conv_w || !V || !aligned16(X0) || (W_target && (!aligned16(W_target) || !Y || !aligned16(Y))) ||
      !aligned16(V)) {
    set_err(ctx, "target: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (!std::isfinite(scale)) {
    set_err(ctx, "scale is not finite");
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  if (W_target == nullptr) return run_conv(ctx, X0, conv_w, B, T, d, k, dt, V, nullptr, scale);
  if ((s = run_conv(ctx, X0, conv_w, B, T, d, k, dt, Y)) != IPTTT_OK) return s;
  return run_target_gemm(ctx, Y, W_target, B * T, d, scale, dt, V);
}

ipttt_status ipttt_chunk_state(ipttt_ctx* ctx, const void* V, const void* Z, const void* W_down0, int64_t B, int64_t T,
                               int64_t d, int64_t d_ff, int64_t C, ipttt_dtype dt, void* W_eff, float* W_final) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, T, d, d_ff, C, 1, dt);
  if (s != IPTTT_OK) return s;
  if (T < 1) {
    set_err(ctx, "chunk_state needs T >= 1");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B == 0) return IPTTT_OK;
  if (!V || !Z || !W_down0 || !W_eff || !W_final || !aligned16(V) || !aligned16(Z) || !aligned16(W_down0) ||
      !aligned16(W_eff) || !aligned16(W_final)) {
    set_err(ctx, "chunk_state: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  return run_state(ctx, V, Z, W_down0, B, T, d, d_ff, C, dt, W_eff, W_final);
}

ipttt_status ipttt_chunk_apply(ipttt_ctx* ctx, const void* Z, const void* W_eff, int64_t B, int64_t T, int64_t d,
                               int64_t d_ff, int64_t C, ipttt_dtype dt, void* O) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, T, d, d_ff, C, 1, dt);
  if (s != IPTTT_OK) return s;
  if (T < 1) {
    set_err(ctx, "chunk_apply needs T >= 1");
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B == 0) return IPTTT_OK;
  if (!Z || !W_eff || !O || !aligned16(Z) || !aligned16(W_eff) || !aligned16(O)) {
    set_err(ctx, "chunk_apply: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16 && (s = ensure_attrs(ctx)) != IPTTT_OK) return s;
  return run_apply(ctx, Z, W_eff, B, T, d, d_ff, C, dt, O);
}

ipttt_status ipttt_state_weight(ipttt_ctx* ctx, const float* W_state, int64_t B, int64_t d, int64_t d_ff,
                                ipttt_dtype dt, void* W) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, 1, d, d_ff, 1, 1, dt, false);
  if (s != IPTTT_OK) return s;
  if (B == 0) return IPTTT_OK;
  if (!W_state || !W || !aligned16(W_state) || !aligned16(W)) {
    set_err(ctx, "state_weight: NULL or misaligned pointer");
    return IPTTT_ERR_INVALID_ARG;
  }
  const int64_t n = B * d * d_ff;
  std::vector<Region> all = {{W_state, (size_t)n * 4, "W_state"}, {W, (size_t)n * esize(dt), "W"}};
  std::vector<Region> outs = {all[1]};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16)
    simt::state_weight_kernel<__nv_bfloat16><<<ceil_div(n, 256), 256, 0, ctx->stream>>>(
        W_state, static_cast<__nv_bfloat16*>(W), n);
  else
    simt::state_weight_kernel<float><<<ceil_div(n, 256), 256, 0, ctx->stream>>>(W_state, static_cast<float*>(W), n);
  return check_launch(ctx, "state weight launch");
}

ipttt_status ipttt_decode_step(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate, const void* W_up,
                               const void* W_cur, int64_t B, int64_t m, int64_t d, int64_t d_ff, ipttt_dtype dt,
                               void* Z, void* O, void* H_buf, void* X0_buf, int64_t C, int64_t pos) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ipttt_status s = check_shape(ctx, B, m, d, d_ff, 1, 1, dt, false);
  if (s != IPTTT_OK) return s;
  if (m < 1 || m > simt::DEC_ROWS) {
    set_err(ctx, "decode step takes 1..%d tokens per sequence (m=%lld)", simt::DEC_ROWS, (long long)m);
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (B == 0) return IPTTT_OK;
  const void* need[] = {H, W_gate, W_up, W_cur, Z, O};
  for (const void* q : need) {
    if (!q || !aligned16(q)) {
      set_err(ctx, "decode step: NULL or misaligned pointer");
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  const bool buf = H_buf != nullptr || X0_buf != nullptr;
  if (buf) {
    if (!H_buf || !X0_buf || !X0 || !aligned16(H_buf) || !aligned16(X0_buf) || !aligned16(X0)) {
      set_err(ctx, "decode step: the chunk buffers need H_buf, X0_buf and X0, 16-byte aligned");
      return IPTTT_ERR_INVALID_ARG;
    }
    if (C < 1 || pos < 0 || pos + m > C || B * C > (int64_t(1) << 31)) {
      set_err(ctx, "decode step: tokens %lld..%lld do not fit a chunk buffer of %lld", (long long)pos,
              (long long)(pos + m), (long long)C);
      return IPTTT_ERR_INVALID_ARG;
    }
  }
  const size_t es = esize(dt);
  const size_t act = (size_t)(B * m * d) * es, wdf = (size_t)(d * d_ff) * es, bufb = buf ? (size_t)(B * C * d) * es : 0;
  std::vector<Region> all = {{H, act, "H"},
                             {buf ? X0 : nullptr, buf ? act : 0, "X0"},
                             {W_gate, wdf, "W_gate"},
                             {W_up, wdf, "W_up"},
                             {W_cur, (size_t)B * wdf, "W_cur"},
                             {Z, (size_t)(B * m * d_ff) * es, "Z"},
                             {O, act, "O"},
                             {H_buf, bufb, "H_buf"},
                             {X0_buf, bufb, "X0_buf"}};
  std::vector<Region> outs = {all[5], all[6], all[7], all[8]};
  std::string what;
  if (find_overlap(outs, all, what)) {
    set_err(ctx, "overlapping buffers: %s", what.c_str());
    return IPTTT_ERR_INVALID_ARG;
  }
  DeviceGuard g(ctx->device);
  if (dt == IPTTT_BF16)
    return run_decode_rows<__nv_bfloat16>(ctx, H, X0, W_gate, W_up, W_cur, B, m, d, d_ff, C, pos, Z, O, H_buf, X0_buf);
  return run_decode_rows<float>(ctx, H, X0, W_gate, W_up, W_cur, B, m, d, d_ff, C, pos, Z, O, H_buf, X0_buf);
}

ipttt_status ipttt_timing_begin(ipttt_ctx* ctx) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->timing = true;
  ctx->timed_calls = 0;
  ctx->timed_launches = 0;
  return IPTTT_OK;
}

ipttt_status ipttt_timing_read(ipttt_ctx* ctx, double* ms, int64_t* calls, int64_t* launches) {
  if (!ctx || !ms || !calls || !launches) return IPTTT_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  ctx->timing = false;
  for (int s = 0; s < IPTTT_NUM_STAGES; ++s) ms[s] = 0.0;
  // stage intervals, in stream order: conv [conv start, conv end], swiglu [conv end, swiglu
  // end], target [swiglu end, target end], state, apply
  const int iv[IPTTT_NUM_STAGES][2] = {{kEvConvEnd, kEvSwigluEnd},
                                       {kEvConvStart, kEvConvEnd},
                                       {kEvSwigluEnd, kEvTargetEnd},
                                       {kEvTargetEnd, kEvStateEnd},
                                       {kEvStateEnd, kEvApplyEnd}};
  for (int c = 0; c < ctx->timed_calls; ++c) {
    cudaEvent_t* ev = &ctx->events[(size_t)c * kEventsPerCall];
    cudaError_t e = cudaEventSynchronize(ev[kEvApplyEnd]);
    if (e == cudaSuccess) e = cudaEventSynchronize(ev[kEvConvEnd]);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "timing event");
    for (int s = 0; s < IPTTT_NUM_STAGES; ++s) {
      float t = 0.f;
      if (s == IPTTT_STAGE_APPLY && ctx->timed_fused[c]) continue;  // included in the state stage
      e = cudaEventElapsedTime(&t, ev[iv[s][0]], ev[iv[s][1]]);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "timing elapsed");
      ms[s] += t;
    }
  }
  *calls = ctx->timed_calls;
  *launches = ctx->timed_launches;
  return IPTTT_OK;
}

ipttt_status ipttt_selftest_wait_timeout(ipttt_ctx* ctx) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  simt::wait_probe_kernel<<<1, 32, 0, ctx->stream>>>(dev_status(ctx));
  return check_launch(ctx, "wait probe launch");
}

int ipttt_sm_count(const ipttt_ctx* ctx) { return ctx ? ctx->sm_count : 0; }

}  // extern "C"

// ====================================================================== allocation-free variant
//
// ipttt_target_noalloc: the target step for callers that cannot allocate device memory.  Its
// scratch is this file-scope array, which the CUDA runtime places in every GPU that loads the
// library.  In host code the name g_noalloc_scratch is only a host-side stand-in, so the
// device address is looked up once per device with cudaGetSymbolAddress and passed to the
// kernels.  Layout: [0, 256) fallback status word, [256, end) the conv output Y.

static __device__ __align__(256) uint8_t g_noalloc_scratch[IPTTT_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoAllocStatusBytes = 256;
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on that device
  EncodeTiledFn encode = nullptr;
  int sm_count = 0;
  int pair_ctas = 0;  // CTAs of a CTA-pair grid on that device (0: the single-CTA kernels run)
};

NoAllocDevice g_noalloc_devices[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// One-time set-up of the current device `dev` (which must be current).
ipttt_status noalloc_device(int dev, NoAllocDevice* out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice& nd = g_noalloc_devices[dev];
  if (!nd.ready) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return IPTTT_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return IPTTT_ERR_CUDA;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return IPTTT_ERR_CUDA;
    }
    // holds nothing on the device: it sets the kernel attributes and sizes the CTA-pair grids
    // (which need the SM count) exactly as ipttt_create's context does
    ipttt_ctx probe;
    probe.device = dev;
    probe.sm_count = sms;
    if (ensure_attrs(&probe) != IPTTT_OK) return IPTTT_ERR_CUDA;
    nd.scratch = static_cast<uint8_t*>(addr);
    nd.encode = reinterpret_cast<EncodeTiledFn>(fn);
    nd.sm_count = sms;
    nd.pair_ctas = probe.pair_ctas;
    nd.ready = true;
  }
  *out = nd;
  return IPTTT_OK;
}

}  // namespace

extern "C" ipttt_status ipttt_target_noalloc(const void* X0, const void* conv_w, const void* W_target, int64_t B,
                                             int64_t T, int64_t d, int k, float scale, ipttt_dtype dtype, void* V,
                                             uint32_t* status, void* cuda_stream) {
  ipttt_status s = check_shape(nullptr, B, T, d, 8, 1, k, dtype, false);
  if (s != IPTTT_OK) return s;
  if (!std::isfinite(scale)) return IPTTT_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return IPTTT_OK;
  if (!X0 || !conv_w || !W_target || !V || !aligned16(X0) || !aligned16(W_target) || !aligned16(V) ||
      (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return IPTTT_ERR_INVALID_ARG;
  const size_t y_bytes = (size_t)B * (size_t)T * (size_t)d * esize(dtype);
  if (y_bytes > IPTTT_NOALLOC_SCRATCH_BYTES - kNoAllocStatusBytes) return IPTTT_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    cudaGetLastError();
    return IPTTT_ERR_CUDA;
  }
  NoAllocDevice nd;
  if ((s = noalloc_device(dev, &nd)) != IPTTT_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  uint32_t* word = status;
  if (word == nullptr) {
    word = reinterpret_cast<uint32_t*>(nd.scratch);
    if (cudaMemsetAsync(word, 0, 2 * sizeof(uint32_t), stream) != cudaSuccess) {
      cudaGetLastError();
      return IPTTT_ERR_CUDA;
    }
  }
  ipttt_ctx c;  // a view for the launchers: it owns no device memory and no events
  c.device = dev;
  c.stream = stream;
  c.sm_count = nd.sm_count;
  c.status = word;
  c.encode = nd.encode;
  c.pair_ctas = nd.pair_ctas;
  c.attrs_set = true;
  void* Y = nd.scratch + kNoAllocStatusBytes;
  if ((s = run_conv(&c, X0, conv_w, B, T, d, k, dtype, Y)) != IPTTT_OK) return s;
  return run_target_gemm(&c, Y, W_target, B * T, d, scale, dtype, V);
}
