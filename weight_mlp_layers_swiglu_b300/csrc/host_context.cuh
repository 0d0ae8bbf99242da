// Host context, errors, argument checks, tensor maps and kernel attributes.
// Part of the host side of libipttt (one translation unit: ipttt.cu includes the host_*.cuh
// files in order).  Everything here is internal; the C ABI is at the end of ipttt.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>
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
#include "tc_target2.cuh"

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
  kEvStart = 0,       // context stream, before the call's first kernel
  kEvConvStart = 1,
  kEvConvEnd = 2,     // the conv kernel (or nothing, when step (2) runs as one kernel)
  kEvSwigluEnd = 3,
  kEvJoined = 4,      // unused (kept for the event layout)
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
  int apply_halves = 0;    // fused pair kernel's apply tiles: 0 per call, 1 = 256 x 256, 2 = 256 x 512
  bool fused_target = false;  // step (2) as one kernel (conv inside the target GEMM) when pairs run
  int target_shift = 0;    // 1: the conv window of the target ends at the next token
  // The host-buffer entry pipelines pieces of a call: uploads on copy_in and downloads on
  // copy_out overlap the compute on `stream` (per-piece events in piece_ev).
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t h_fork = nullptr, h_join = nullptr;
  // The bf16 backward pass runs its target branch (dV, dY, dW_target, the conv adjoints) on
  // `side`, forked from and joined back into `stream` with b_fork / b_join.
  cudaStream_t side = nullptr;
  cudaEvent_t b_fork = nullptr, b_join = nullptr;
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
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t gd[4], gs[3];
  cuuint32_t bx[4], es[4];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  const CUresult r =
      ctx->encode(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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

// [outer, mid, inner] bf16 row-major, box = 64 inner x box_mid x 1, unswizzled (rows of 128
// bytes one after another in shared memory, for CUDA-core readers).
bool map_3d_plain(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t outer, int64_t mid, int64_t inner,
                  uint32_t box_mid) {
  const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)mid, (uint64_t)outer};
  const uint64_t strides[2] = {(uint64_t)inner * 2, (uint64_t)inner * mid * 2};
  const uint32_t box[3] = {64, box_mid, 1};
  return encode_map(ctx, m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// [outer, mid, inner] bf16 (rows row_stride elements apart, inner a multiple of 64) seen as
// [outer][inner / 64][mid][64]: blocks of 64 columns.  The box is two blocks of 64 columns x
// 64 rows, so one request brings what two requests of the 3-D map with box_mid = 64 bring, in
// the same shared-memory layout (block 0's 64 rows of 128 bytes, then block 1's).
bool map_blocks(ipttt_ctx* ctx, CUtensorMap* m, const void* base, int64_t outer, int64_t mid, int64_t inner,
                int64_t row_stride) {
  const uint64_t dims[4] = {64, (uint64_t)mid, (uint64_t)(inner / 64), (uint64_t)outer};
  const uint64_t strides[3] = {(uint64_t)row_stride * 2, 128, (uint64_t)row_stride * mid * 2};
  const uint32_t box[4] = {64, 64, 2, 1};
  return encode_map(ctx, m, base, 4, dims, strides, box);
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
    constexpr int NPK = 16;
    const void* pk[NPK] = {(const void*)gemm2::tc_gemm2_kernel<gemm::kSwiglu>,
                           (const void*)gemm2::tc_gemm2_kernel<gemm::kTarget>,
                           (const void*)gemm2::tc_gemm2_kernel<gemm::kApply>,
                           (const void*)gemm2::tc_gemm2_kernel<gemm::kSwigluSave>,
                           (const void*)gemm2::tc_gemm2_kernel<gemm::kTwoSeg>,
                           (const void*)state2::tc_state2_kernel,
                           (const void*)fused2::tc_state_apply2_kernel<1>,
                           (const void*)fused2::tc_state_apply2_kernel<2>,
                           (const void*)tconv2::tc_target_conv2_kernel<1>,
                           (const void*)tconv2::tc_target_conv2_kernel<2>,
                           (const void*)tconv2::tc_target_conv2_kernel<3>,
                           (const void*)tconv2::tc_target_conv2_kernel<4>,
                           (const void*)tconv2::tc_target_conv2_kernel<5>,
                           (const void*)tconv2::tc_target_conv2_kernel<6>,
                           (const void*)tconv2::tc_target_conv2_kernel<7>,
                           (const void*)tconv2::tc_target_conv2_kernel<8>};
    int pk_smem[NPK], pk_threads[NPK];
    for (int ki = 0; ki < NPK; ++ki) {
      pk_smem[ki] = ki < 5    ? gemm2::SMEM_BYTES
                    : ki == 5 ? state2::SMEM_BYTES
                    : ki < 8  ? fused2::SMEM_BYTES
                              : tconv2::SMEM_BYTES;
      pk_threads[ki] = ki < 8 ? gemm2::NUM_THREADS : tconv2::NUM_THREADS;
    }
    int clusters = 1 << 30;
    for (int ki = 0; ki < NPK; ++ki) {
      const void* k = pk[ki];
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pk_smem[ki]);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "smem attribute (pair kernels)");
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(ctx->sm_count & ~1), 1, 1);
      cfg.blockDim = dim3(pk_threads[ki], 1, 1);
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

// The token-major operands of a state kernel (V: [B, T, M], Z: [B, T, N], rows v_stride and
// z_stride elements apart) as the kernel loads them: for the CTA-pair kernels, with M and N
// multiples of 64, as blocks of 64 columns (map_blocks, one request per operand and k-block;
// p.blocked = 1), else as 3-D maps with 64-token boxes (two requests each).
bool map_state_operands(ipttt_ctx* ctx, CUtensorMap* mv, CUtensorMap* mz, const void* V, int64_t v_stride,
                        const void* Z, int64_t z_stride, int64_t B, int64_t T, int64_t M, int64_t N, bool pairs,
                        int* blocked) {
  *blocked = (pairs && M % 64 == 0 && N % 64 == 0) ? 1 : 0;
  if (*blocked)
    return map_blocks(ctx, mv, V, B, T, M, v_stride) && map_blocks(ctx, mz, Z, B, T, N, z_stride);
  return map_3d_strided(ctx, mv, V, B, T, M, v_stride, 64) && map_3d_strided(ctx, mz, Z, B, T, N, z_stride, 64);
}

// Step (2) of a bf16 layer call runs as the one conv + projection kernel (tc_target2.cuh).
bool use_fused_target(const ipttt_ctx* ctx) { return ctx->fused_target && use_pairs(ctx); }

// Grid of a pair-GEMM launch: one CTA pair per tile, at most the co-resident pairs.
int pair_grid(const ipttt_ctx* ctx, int64_t tiles) {
  return 2 * (int)(tiles < ctx->pair_ctas / 2 ? tiles : ctx->pair_ctas / 2);
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace
