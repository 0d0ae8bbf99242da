// Host orchestration and C ABI of the In-Place TTT fast-weight SwiGLU layer (see
// include/ipttt.h for the contract).  bf16 runs on the tcgen05 kernels (tc_gemm.cuh,
// tc_state.cuh); fp32 runs on the CUDA-core kernels (simt.cuh).  Nothing here computes on
// the host: every step of the layer is a kernel launch on the context's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/ipttt.h"
#include "ptx.cuh"
#include "simt.cuh"
#include "tc_fused.cuh"
#include "tc_fused2.cuh"
#include "tc_gemm.cuh"
#include "tc_gemm2.cuh"
#include "tc_state.cuh"
#include "tc_state2.cuh"

using namespace ipttt;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {

constexpr int kMaxTimedCalls = 256;
constexpr int kMaxPieces = 64;           // pieces of one host-buffer call
constexpr int64_t kPieceTokens = 4096;   // target piece length (rounded up to a multiple of C)
// Timing events recorded per timed layer call.
enum : int {
  kEvStart = 0,       // context stream, before the fork
  kEvConvStart = 1,   // side stream
  kEvConvEnd = 2,     // side stream
  kEvSwigluEnd = 3,   // context stream
  kEvJoined = 4,      // context stream, after waiting for the conv
  kEvTargetEnd = 5,
  kEvStateEnd = 6,
  kEvApplyEnd = 7,
  kEventsPerCall = 8
};

}  // namespace

struct ipttt_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  int sm_count = 0;
  uint32_t* status = nullptr;  // device, 2 words
  uint64_t wait_limit_ns = 2000000000ull;
  EncodeTiledFn encode = nullptr;
  bool attrs_set = false;
  bool coop = false;       // device supports cooperative launches
  bool fused_tail = true;  // run steps (3)-(5) as one cooperative kernel when possible
  bool cta_pairs = true;   // bf16 GEMMs on CTA pairs (cta_group::2) when the device allows
  int pair_ctas = 0;       // CTAs of the pair GEMM grid (2 x co-resident clusters; 0 = unavailable)
  bool fused_pairs = true; // the cooperative launch of the fused pair kernel has not been refused
  int target_shift = 0;    // 1: the conv window of the target ends at the next token
  // The causal conv runs on an internal side stream, forked from and joined back into
  // `stream` with these events, so that it overlaps the SwiGLU GEMM.
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  // The host-buffer entry pipelines pieces of a call: uploads on copy_in and downloads on
  // copy_out overlap the compute on `stream` (per-piece events in piece_ev).
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t h_fork = nullptr, h_join = nullptr;
  std::vector<cudaEvent_t> piece_ev;  // [2 * kMaxPieces]: upload done, compute done
  // timing
  bool timing = false;
  int timed_calls = 0;
  int64_t timed_launches = 0;
  std::vector<cudaEvent_t> events;
  std::vector<char> timed_fused;  // per timed call: steps (3)-(5) ran as one kernel
  std::string err;
};

namespace {

void set_err(ipttt_ctx* ctx, const char* fmt, ...) {
  if (!ctx) return;
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  ctx->err = buf;
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

size_t esize(ipttt_dtype dt) { return dt == IPTTT_BF16 ? 2 : 4; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Region {
  const void* p;
  size_t bytes;
  const char* name;
};

// Finds the first pair (output region, any other region) whose byte ranges intersect.
bool find_overlap(const std::vector<Region>& outs, const std::vector<Region>& all, std::string& what) {
  for (const Region& o : outs) {
    if (!o.p || o.bytes == 0) continue;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(o.p), a1 = a0 + o.bytes;
    for (const Region& r : all) {
      if (!r.p || r.bytes == 0 || std::strcmp(r.name, o.name) == 0) continue;
      const uintptr_t b0 = reinterpret_cast<uintptr_t>(r.p), b1 = b0 + r.bytes;
      if (a0 < b1 && b0 < a1) {
        what = std::string(o.name) + " / " + r.name;
        return true;
      }
    }
  }
  return false;
}

// Shape rules shared by every entry point.  ctx may be null (host-only callers).
ipttt_status check_shape(ipttt_ctx* ctx, int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, int k,
                         ipttt_dtype dt, bool need_C = true) {
  if (dt != IPTTT_F32 && dt != IPTTT_BF16) {
    set_err(ctx, "unknown dtype %d", (int)dt);
    return IPTTT_ERR_INVALID_ARG;
  }
  if (B < 0 || T < 0 || d < 1 || f < 1 || k < 1 || (need_C && C < 1)) {
    set_err(ctx, "invalid sizes B=%lld T=%lld d=%lld d_ff=%lld C=%lld k=%d", (long long)B, (long long)T,
            (long long)d, (long long)f, (long long)C, k);
    return IPTTT_ERR_INVALID_ARG;
  }
  if (d % 8 || f % 8) {
    set_err(ctx, "d (%lld) and d_ff (%lld) must be multiples of 8", (long long)d, (long long)f);
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (k > simt::CONV_MAXK) {
    set_err(ctx, "conv kernel size k=%d > %d", k, simt::CONV_MAXK);
    return IPTTT_ERR_UNSUPPORTED;
  }
  if (dt == IPTTT_BF16 && need_C && C % 128) {
    set_err(ctx, "bf16 path needs C %% 128 == 0 (C=%lld)", (long long)C);
    return IPTTT_ERR_UNSUPPORTED;
  }
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (B * T > lim || d > (1 << 20) || f > (1 << 22) || (need_C && C > lim)) {
    set_err(ctx, "sizes exceed the supported range");
    return IPTTT_ERR_UNSUPPORTED;
  }
  return IPTTT_OK;
}

int64_t n_chunks_of(int64_t T, int64_t C) { return T == 0 ? 0 : (T + C - 1) / C; }

struct WsLayout {
  size_t y, v, z, w, ctr, total;
};

WsLayout ws_layout(int64_t B, int64_t T, int64_t d, int64_t f, int64_t C, ipttt_dtype dt) {
  const size_t es = esize(dt);
  WsLayout L;
  size_t off = 0;
  L.y = off;
  off += align256((size_t)B * T * d * es);
  L.v = off;
  off += align256((size_t)B * T * d * es);
  L.z = off;
  off += align256((size_t)B * T * f * es);
  L.w = off;
  off += align256((size_t)B * n_chunks_of(T, C) * d * f * es);
  L.ctr = off;  // hand-off counters of the fused state + apply kernel: B*n slices + queue head
  off += align256(((size_t)B * n_chunks_of(T, C) + 1) * sizeof(uint32_t));
  L.total = off;
  return L;
}

ipttt_status cuda_fail(ipttt_ctx* ctx, cudaError_t e, const char* what) {
  set_err(ctx, "%s: %s", what, cudaGetErrorString(e));
  return IPTTT_ERR_CUDA;
}

ipttt_status check_launch(ipttt_ctx* ctx, const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  return IPTTT_OK;
}

// ------------------------------------------------------------------ tensor maps

bool encode_map(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUresult r =
      ctx->encode(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_err(ctx, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return false;
  }
  return true;
}

// [rows, cols] bf16 row-major, box = 64 columns x box_rows rows.
bool map_2d(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_cols,
            uint32_t box_rows) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {box_cols, box_rows};
  return encode_map(ctx, m, base, 2, dims, strides, box);
}

// [outer, mid, inner] bf16 row-major, box = 64 inner x box_mid x 1.
bool map_3d(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t outer, int64_t mid, int64_t inner,
            uint32_t box_mid) {
  const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)mid, (uint64_t)outer};
  const uint64_t strides[2] = {(uint64_t)inner * 2, (uint64_t)inner * mid * 2};
  const uint32_t box[3] = {64, box_mid, 1};
  return encode_map(ctx, m, base, 3, dims, strides, box);
}

// [outer, mid, inner] bf16 whose rows are row_stride elements apart (inner <= row_stride).
bool map_3d_strided(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t outer, int64_t mid, int64_t inner,
                    int64_t row_stride, uint32_t box_mid) {
  const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)mid, (uint64_t)outer};
  const uint64_t strides[2] = {(uint64_t)row_stride * 2, (uint64_t)row_stride * mid * 2};
  const uint32_t box[3] = {64, box_mid, 1};
  return encode_map(ctx, m, base, 3, dims, strides, box);
}

// [outer, mid, inner] fp32 row-major, box = 32 inner (128 bytes) x box_mid x 1.
bool map_3d_f32(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t outer, int64_t mid, int64_t inner,
                uint32_t box_mid) {
  const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)mid, (uint64_t)outer};
  const uint64_t strides[2] = {(uint64_t)inner * 4, (uint64_t)inner * mid * 4};
  const uint32_t box[3] = {32, box_mid, 1};
  return encode_map(ctx, m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

ipttt_status ensure_attrs(ipttt_ctx* ctx) {
  if (ctx->attrs_set) return IPTTT_OK;
  cudaError_t e;
  e = cudaFuncSetAttribute(gemm::tc_gemm_kernel<gemm::kSwiglu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemm::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (swiglu)");
  e = cudaFuncSetAttribute(gemm::tc_gemm_kernel<gemm::kTarget>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemm::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (target)");
  e = cudaFuncSetAttribute(gemm::tc_gemm_kernel<gemm::kApply>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemm::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (apply)");
  e = cudaFuncSetAttribute(gemm::tc_gemm_kernel<gemm::kSwigluSave>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemm::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (swiglu save)");
  e = cudaFuncSetAttribute(gemm::tc_gemm_kernel<gemm::kTwoSeg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           gemm::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (two-segment)");
  {
    const void* pk[7] = {(const void*)gemm2::tc_gemm2_kernel<gemm::kSwiglu>,
                         (const void*)gemm2::tc_gemm2_kernel<gemm::kTarget>,
                         (const void*)gemm2::tc_gemm2_kernel<gemm::kApply>,
                         (const void*)gemm2::tc_gemm2_kernel<gemm::kSwigluSave>,
                         (const void*)gemm2::tc_gemm2_kernel<gemm::kTwoSeg>, (const void*)state2::tc_state2_kernel,
                         (const void*)fused2::tc_state_apply2_kernel};
    const int pk_smem[7] = {gemm2::SMEM_BYTES, gemm2::SMEM_BYTES, gemm2::SMEM_BYTES, gemm2::SMEM_BYTES,
                            gemm2::SMEM_BYTES, state2::SMEM_BYTES, fused2::SMEM_BYTES};
    int clusters = 1 << 30;
    for (int ki = 0; ki < 7; ++ki) {
      const void* k = pk[ki];
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pk_smem[ki]);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (pair kernels)");
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(ctx->sm_count & ~1), 1, 1);
      cfg.blockDim = dim3(gemm2::NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = pk_smem[ki];
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      clusters = n < clusters ? n : clusters;
    }
    ctx->pair_ctas = 2 * clusters;
  }
  e = cudaFuncSetAttribute(state::tc_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           state::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (state)");
  e = cudaFuncSetAttribute(fused::tc_state_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           fused::SMEM_BYTES);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (state+apply)");
  ctx->attrs_set = true;
  return IPTTT_OK;
}

DevStatus dev_status(ipttt_ctx* ctx) { return DevStatus{ctx->status, ctx->wait_limit_ns}; }

bool use_pairs(const ipttt_ctx* ctx) { return ctx->cta_pairs && ctx->pair_ctas >= 2; }

// Grid of a pair-GEMM launch: one CTA pair per tile, at most the co-resident pairs.
int pair_grid(const ipttt_ctx* ctx, int64_t tiles) {
  return 2 * (int)(tiles < ctx->pair_ctas / 2 ? tiles : ctx->pair_ctas / 2);
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// ------------------------------------------------------------------ step launchers (no validation)

ipttt_status run_swiglu(ipttt_ctx* ctx, const void* H, const void* Wg, const void* Wu, int64_t rows, int64_t d,
                        int64_t f, ipttt_dtype dt, void* Z) {
  if (rows == 0) return IPTTT_OK;
  if (dt == IPTTT_BF16) {
    CUtensorMap ma, mb0, mb1, mo;
    if (!map_2d(ctx, &ma, H, rows, d, 64, 128) || !map_2d(ctx, &mb0, Wg, f, d, 64, 128) ||
        !map_2d(ctx, &mb1, Wu, f, d, 64, 128) || !map_2d(ctx, &mo, Z, rows, f, 64, 32))
      return IPTTT_ERR_CUDA;
    gemm::Params p{};
    const bool pairs = use_pairs(ctx);
    p.m_tiles = ceil_div(rows, pairs ? gemm2::PAIR_M : gemm::BM);
    p.n_tiles = ceil_div(f, 128);
    p.k_blocks = ceil_div(d, gemm::BK);
    p.problems = 1;
    p.group_m = pairs ? 8 : 16;
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
  dim3 block(32, 4);
  dim3 grid(ceil_div(d / 8, 32), ceil_div(T, (int64_t)simt::CONV_TS * 4), (unsigned)B);
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
    if (!map_3d(ctx, &mv, V, B, T, d, 64) || !map_3d(ctx, &mz, Z, B, T, f, 64) ||
        !map_3d(ctx, &mw, W_eff, B * n, d, f, 32) || !map_3d_f32(ctx, &mf, W_final, B, d, f, 32))
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
  *st = IPTTT_ERR_CUDA;
  if (!map_3d(ctx, &mv, V, B, T, d, 64) || !map_3d(ctx, &mz, Z, B, T, f, 64) ||
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
  p.s.st = dev_status(ctx);
  p.a.m_tiles = (int)(C / gemm2::PAIR_M);
  p.a.n_tiles = ceil_div(d, gemm2::BN);
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
      cudaLaunchKernelEx(&cfg, fused2::tc_state_apply2_kernel, mv, mz, mw_st, mf, mza, mw_ld, mw0, mo, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // a refused launch configuration is not sticky
    ctx->fused_pairs = false;
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
  if (e != cudaSuccess) return cuda_fail(ctx, e, "state+apply launch");
  return check_launch(ctx, "state+apply launch");
}

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
  if (!map_3d_strided(ctx, &mv, V, B, T, M, v_stride, 64) || !map_3d_strided(ctx, &mz, Z, B, T, N, z_stride, 64) ||
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
    p.group_m = 8;
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
    p.group_m = pairs ? 8 : 16;
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
  if (bf16) {
    // reverse scan: R_i = dW_final + sum_{l>i} dO_l^T Z_l, final = dW_final + sum_i dO_i^T Z_i
    if ((s = launch_state_general(ctx, dO, d, Z, f, B, T, d, f, C, nullptr, dW_final, false, true, Rst,
                                  B == 1 ? dW0 : dW0b)) != IPTTT_OK)
      return s;
    // dZ_i = dO_i W_i + V_i R_i (V carries eta), and in the same epilogue the gated-MLP
    // adjoints: AU = [A | U] becomes [dA | dU]
    if ((s = launch_two_seg(ctx, dO, d, V, d, 0, Wst, Rst, B * n, true, B, T, C, d, d, f, nullptr, AU)) != IPTTT_OK)
      return s;
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
  }
  // fp32: the gated-MLP backward in place, AU -> [dA | dU] (bf16 did it in the dZ epilogue)
  if (!bf16) {
    simt::swiglu_backward_kernel<float><<<ceil_div(BT * f, 256), 256, 0, ctx->stream>>>(
        static_cast<const float*>(dZ), static_cast<float*>(AU), BT, (int)f);
    if ((s = check_launch(ctx, "swiglu backward launch")) != IPTTT_OK) return s;
  }
  if (bf16) {
    const size_t es = 2;
    // dH = dA W_gate + dU W_up
    if ((s = launch_two_seg(ctx, AU, 2 * f, nullptr, 2 * f, f, Wg, Wu, 1, false, 1, BT, CT, f, f, d, dH)) != IPTTT_OK)
      return s;
    // dW_gate = dA^T H, dW_up = dU^T H (reductions over all tokens)
    if ((s = launch_state_general(ctx, AU, 2 * f, H, d, 1, BT, f, d, CT, nullptr, nullptr, true, false, nullptr,
                                  dWg)) != IPTTT_OK ||
        (s = launch_state_general(ctx, static_cast<uint8_t*>(AU) + f * es, 2 * f, H, d, 1, BT, f, d, CT, nullptr,
                                  nullptr, true, false, nullptr, dWu)) != IPTTT_OK)
      return s;
  } else {
    const float* au = static_cast<const float*>(AU);
    if ((s = sgemm(ctx, au, 2 * f, 1, static_cast<const float*>(Wg), d, 1, static_cast<float*>(dH), d, BT, d, f, 1.f,
                   0.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au + f, 2 * f, 1, static_cast<const float*>(Wu), d, 1, static_cast<float*>(dH), d, BT, d, f,
                   1.f, 1.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au, 1, 2 * f, static_cast<const float*>(H), d, 1, dWg, d, f, d, BT, 1.f, 0.f)) != IPTTT_OK ||
        (s = sgemm(ctx, au + f, 1, 2 * f, static_cast<const float*>(H), d, 1, dWu, d, f, d, BT, 1.f, 0.f)) != IPTTT_OK)
      return s;
  }
  // dV = eta Z R^T (per chunk), dY = dV W_target^T, dW_target = Y^T dV (without a projection
  // dY is dV itself)
  if ((s = run_apply(ctx, Z, Rst, B, T, d, f, C, dt, dV, nullptr, eta)) != IPTTT_OK) return s;
  if (Wt == nullptr) {
    dY = dV;
  } else if (bf16) {
    if ((s = run_apply(ctx, dV, Wt, 1, BT, d, d, CT, dt, dY)) != IPTTT_OK) return s;
    if ((s = launch_state_general(ctx, Y, d, dV, d, 1, BT, d, d, CT, nullptr, nullptr, true, false, nullptr, dWt)) !=
        IPTTT_OK)
      return s;
  } else {
    if ((s = sgemm(ctx, static_cast<const float*>(dV), d, 1, static_cast<const float*>(Wt), 1, d,
                   static_cast<float*>(dY), d, BT, d, d, 1.f, 0.f)) != IPTTT_OK ||
        (s = sgemm(ctx, static_cast<const float*>(Y), 1, d, static_cast<const float*>(dV), d, 1, dWt, d, d, d, BT, 1.f,
                   0.f)) != IPTTT_OK)
      return s;
  }
  // the causal conv's adjoints
  {
    const int64_t groups = d / (bf16 ? 8 : 4);  // 16-byte channel groups
    dim3 gx(ceil_div(groups, 64), ceil_div(T, simt::CONVX_ROWS), (unsigned)B);
    dim3 gw((unsigned)L.strips, ceil_div(groups, 64));
    if (bf16)
      launch_conv_adjoints<__nv_bfloat16>(ctx, gx, gw, dY, cw, X0, dX0, part, (int)T, (int)d, k);
    else
      launch_conv_adjoints<float>(ctx, gx, gw, dY, cw, X0, dX0, part, (int)T, (int)d, k);
    simt::sum_strips_kernel<<<ceil_div(d * k, 256), 256, 0, ctx->stream>>>(part, dcw, (int)L.strips, d * k);
    if ((s = check_launch(ctx, "conv backward launch")) != IPTTT_OK) return s;
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

void mark(ipttt_ctx* ctx, int call, int which, cudaStream_t stream) {
  if (call >= 0) cudaEventRecord(ctx->events[(size_t)call * kEventsPerCall + which], stream);
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
  cudaError_t e;
  mark(ctx, call, kEvStart, ctx->stream);
  // fork: the causal conv (memory bound) overlaps the SwiGLU GEMM (tensor bound)
  if ((e = cudaEventRecord(ctx->fork, ctx->stream)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(ctx->side, ctx->fork, 0)) != cudaSuccess)
    return cuda_fail(ctx, e, "fork");
  {
    cudaStream_t main_stream = ctx->stream;
    ctx->stream = ctx->side;
    mark(ctx, call, kEvConvStart, ctx->side);
    // without W_target (the "w/o Proj" ablation) the conv writes V = eta * conv(X0) directly
    s = Wt != nullptr ? run_conv(ctx, X0, cw, B, T, d, k, dt, Y, halo_in)
                      : run_conv(ctx, X0, cw, B, T, d, k, dt, V, halo_in, eta);
    mark(ctx, call, kEvConvEnd, ctx->side);
    ctx->stream = main_stream;
    if (s != IPTTT_OK) return s;
  }
  if ((e = cudaEventRecord(ctx->join, ctx->side)) != cudaSuccess) return cuda_fail(ctx, e, "join record");
  if ((s = sv ? run_swiglu_save(ctx, H, Wg, Wu, B * T, d, f, dt, Z, sv->au)
              : run_swiglu(ctx, H, Wg, Wu, B * T, d, f, dt, Z)) != IPTTT_OK)
    return s;
  mark(ctx, call, kEvSwigluEnd, ctx->stream);
  if ((e = cudaStreamWaitEvent(ctx->stream, ctx->join, 0)) != cudaSuccess) return cuda_fail(ctx, e, "join");
  mark(ctx, call, kEvJoined, ctx->stream);
  const bool bf16 = dt == IPTTT_BF16;  // W_eff[b, 0] = W_down0: the apply reads W_down0 itself
  const bool fuse = bf16 && ctx->fused_tail && ctx->coop;
  uint32_t* ctr = sv ? sv->ctr : reinterpret_cast<uint32_t*>(base + L.ctr);
  const int n_ctr = (int)(B * n_chunks_of(T, C) + 1);
  if (Wt != nullptr) {
    if ((s = run_target_gemm(ctx, Y, Wt, B * T, d, eta, dt, V, fuse ? ctr : nullptr, fuse ? n_ctr : 0)) != IPTTT_OK)
      return s;
  } else if (fuse) {
    const cudaError_t ez = cudaMemsetAsync(ctr, 0, (size_t)n_ctr * sizeof(uint32_t), ctx->stream);
    if (ez != cudaSuccess) return cuda_fail(ctx, ez, "counter reset");
  }
  mark(ctx, call, kEvTargetEnd, ctx->stream);
  if (fuse) {
    if ((s = run_state_apply_fused(ctx, V, Z, W0, B, T, d, f, C, Wst, W_final, O, ctr, W_init, sv != nullptr)) !=
        IPTTT_OK)
      return s;
    mark(ctx, call, kEvStateEnd, ctx->stream);
    mark(ctx, call, kEvApplyEnd, ctx->stream);
    if (call >= 0) ctx->timed_fused[call] = 1;
  } else {
    const bool skip_first = bf16 && sv == nullptr;  // the training forward keeps W_0 in the stack too
    if ((s = run_state(ctx, V, Z, W0, B, T, d, f, C, dt, Wst, W_final, skip_first, W_init)) != IPTTT_OK) return s;
    mark(ctx, call, kEvStateEnd, ctx->stream);
    const void* w0_first = (skip_first && W_init == nullptr) ? W0 : nullptr;
    if ((s = run_apply(ctx, Z, Wst, B, T, d, f, C, dt, O, w0_first)) != IPTTT_OK) return s;
    mark(ctx, call, kEvApplyEnd, ctx->stream);
  }
  if (call >= 0)
    ctx->timed_launches += (bf16 ? (fuse ? 4 : 5) : 6) + ((halo_out != nullptr && k > 1) ? 1 : 0) - (Wt ? 0 : 1);
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
  if (cudaStreamCreateWithFlags(&ctx->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->join, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&ctx->copy_out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->h_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ctx->h_join, cudaEventDisableTiming) != cudaSuccess) {
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

ipttt_status ipttt_set_fused_tail(ipttt_ctx* ctx, int enable) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
  ctx->fused_tail = enable != 0;
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
  if (ctx->fork) cudaEventDestroy(ctx->fork);
  if (ctx->join) cudaEventDestroy(ctx->join);
  if (ctx->side) cudaStreamDestroy(ctx->side);
  for (auto& e : ctx->piece_ev)
    if (e) cudaEventDestroy(e);
  if (ctx->h_fork) cudaEventDestroy(ctx->h_fork);
  if (ctx->h_join) cudaEventDestroy(ctx->h_join);
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
  cudaMemsetAsync(dW_gate, 0, gdf, ctx->stream);
  cudaMemsetAsync(dW_up, 0, gdf, ctx->stream);
  if (dW_target) cudaMemsetAsync(dW_target, 0, (size_t)d * d * 4, ctx->stream);
  cudaMemsetAsync(dconv_w, 0, (size_t)d * k * 4, ctx->stream);
  if (dW_final != nullptr && B > 0)
    simt::sum_strips_kernel<<<ceil_div(d * d_ff, 256), 256, 0, ctx->stream>>>(dW_final, dW_down0, (int)B, d * d_ff);
  else
    cudaMemsetAsync(dW_down0, 0, gdf, ctx->stream);
  return check_launch(ctx, "empty backward");
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

ipttt_status ipttt_layer_forward_resume(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                        const void* W_up, const void* W_target, const void* conv_w,
                                        const float* W_state, const void* X0_halo, int64_t B, int64_t T, int64_t d,
                                        int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dt, void* O,
                                        float* W_state_out, void* X0_halo_out, void* ws, size_t ws_bytes) {
  if (!ctx) return IPTTT_ERR_INVALID_ARG;
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
  const int n_pieces = (int)((T + P - 1) / P);
  for (int j = 0; j < n_pieces; ++j) {
    const int64_t lo = j * P;
    const int64_t len = (lo + P < T ? P : T - lo);
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
  // stage intervals: swiglu [start, swiglu end], conv [conv start, conv end] on the side stream
  // (overlapping the SwiGLU GEMM), target [joined, target end], state, apply
  const int iv[IPTTT_NUM_STAGES][2] = {{kEvStart, kEvSwigluEnd},
                                       {kEvConvStart, kEvConvEnd},
                                       {kEvJoined, kEvTargetEnd},
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
    ipttt_ctx probe;  // holds nothing on the device; only used to set the kernel attributes
    probe.device = dev;
    if (ensure_attrs(&probe) != IPTTT_OK) return IPTTT_ERR_CUDA;
    nd.scratch = static_cast<uint8_t*>(addr);
    nd.encode = reinterpret_cast<EncodeTiledFn>(fn);
    nd.sm_count = sms;
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
  c.attrs_set = true;
  void* Y = nd.scratch + kNoAllocStatusBytes;
  if ((s = run_conv(&c, X0, conv_w, B, T, d, k, dtype, Y)) != IPTTT_OK) return s;
  return run_target_gemm(&c, Y, W_target, B * T, d, scale, dtype, V);
}
