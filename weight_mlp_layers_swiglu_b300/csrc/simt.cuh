// CUDA-core kernels: the causal depthwise convolution (both precisions), the fp32 path of
// the layer (generic tiled SGEMM, exclusive chunk scan), and small helpers.
//
// The fp32 path keeps fp32 end to end (tensor-core TF32 would not meet a 1e-4 relative
// bound); it follows the three steps of zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，
// 让它边读边学" §3.2 literally: Step 1 every chunk's Delta_i = V_i^T Z_i in parallel (one
// batched GEMM), Step 2 one exclusive prefix sum over chunks (scan kernel), Step 3 every
// chunk applied with its own weight (one batched GEMM).
#pragma once

#include "ptx.cuh"

namespace ipttt {
namespace simt {

// --------------------------------------------------------------------------- causal conv
// Y[b, t, c] = sum_{s<k} conv_w[c, s] * X0[b, t-(k-1)+s, c], zero for t-(k-1)+s < 0
// (zhichai.net page, §3.3: Conv1D with causal padding).  The conv reads and writes each
// element once, so it is bound by memory bandwidth: each thread owns 8 channels (one 16- or
// 32-byte vector) of a strip of conv_rows<T>() tokens and issues the loads of all its input
// rows (the strip and the k-1 rows before it) before any arithmetic, so that every thread
// keeps that many vector loads in flight.  The sum for one output is an fp32 fma chain over
// the taps from zero, s = 0 .. k-1.
constexpr int CONV_MAXK = 8;
constexpr int CONV_STRIPS = 4;  // token strips per block (blockDim.y); blockDim.x = 32 channel groups

template <typename T>
__host__ __device__ constexpr int conv_rows() {
  return sizeof(T) == 2 ? 8 : 4;
}

// One row's 8 channels as loaded: a 16-byte vector (bf16) or two (fp32), widened when used.
template <typename T>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void zero() { v = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void widen(float (&f)[8]) const {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  }
};
template <>
struct Row8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void widen(float (&f)[8]) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
};

// The K taps of channels c0 .. c0+N-1, widened: w[e][s] = conv_w[c0 + e, s].  Those N*K values
// are contiguous; with conv_w 16-byte aligned (c0 a multiple of 8 keeps the offset aligned) they
// are read as N*K*sizeof(T)/16 vectors instead of N*K scalars, which had bounded the conv
// kernel's rate (one scalar load per tap and channel against 11 row vectors of data).
template <typename T, int K, int N>
__device__ __forceinline__ void load_taps(const T* __restrict__ conv_w, int c0, float (&w)[N][K]) {
  static_assert((N * K * (int)sizeof(T)) % 16 == 0, "taps in whole vectors");
  const T* src = conv_w + (int64_t)c0 * K;
  if ((reinterpret_cast<uintptr_t>(conv_w) & 15u) == 0) {
    constexpr int NV = N * K * (int)sizeof(T) / 16;
    uint4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = reinterpret_cast<const uint4*>(src)[i];
    const T* t = reinterpret_cast<const T*>(v);
#pragma unroll
    for (int e = 0; e < N; ++e)
#pragma unroll
      for (int s = 0; s < K; ++s) w[e][s] = static_cast<float>(t[e * K + s]);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e)
#pragma unroll
      for (int s = 0; s < K; ++s) w[e][s] = static_cast<float>(src[e * K + s]);
  }
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]) {
  Row8<T> r;
  r.load(p);
  r.widen(v);
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = w;
}

// halo (optional, [B, K-1, d]): the K-1 rows that precede X0's first token of each sequence
// (rows of an earlier call); without it those rows are zero.  shift = 1 moves the window one
// token later (it ends at t+1; the token after the last one reads as zero).  The output is
// multiplied by `scale`.
template <typename T, int K>
__global__ void __launch_bounds__(32 * CONV_STRIPS, 4)
    causal_conv_kernel(const T* __restrict__ X0, const T* __restrict__ conv_w, T* __restrict__ Y, int T_len, int d,
                       const T* __restrict__ halo, int shift, float scale) {
  constexpr int R = conv_rows<T>();
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  const int t0 = (blockIdx.y * blockDim.y + threadIdx.y) * R;
  const int b = blockIdx.z;
  if (c0 >= d || t0 >= T_len) return;
  const T* xb = X0 + (int64_t)b * T_len * d + c0;
  T* yb = Y + (int64_t)b * T_len * d + c0;
  // input row j is X0[t0 + shift - (K-1) + j]: issue every load first
  Row8<T> raw[R + K - 1];
#pragma unroll
  for (int j = 0; j < R + K - 1; ++j) {
    const int src = t0 + shift - (K - 1) + j;
    if (src >= 0 && src < T_len)
      raw[j].load(xb + (int64_t)src * d);
    else if (src < 0 && halo != nullptr)
      raw[j].load(halo + ((int64_t)b * (K - 1) + (K - 1) + src) * d + c0);
    else
      raw[j].zero();
  }
  float w[8][K];
  load_taps<T, K, 8>(conv_w, c0, w);
  float win[K][8];  // the last K input rows, widened
#pragma unroll
  for (int j = 0; j < K - 1; ++j) raw[j].widen(win[j]);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    raw[r + K - 1].widen(win[K - 1]);
    if (t0 + r < T_len) {
      float out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < K; ++s) acc = fmaf(w[e][s], win[s][e], acc);
        out[e] = acc * scale;
      }
      store8<T>(yb + (int64_t)(t0 + r) * d, out);
    }
#pragma unroll
    for (int s = 0; s < K - 1; ++s)
#pragma unroll
      for (int e = 0; e < 8; ++e) win[s][e] = win[s + 1][e];
  }
}

// halo_out[b, j] = row T-(k-1)+j of [halo_in[b], X0[b]] (the k-1 rows the next call of the
// sequence needs); rows before the sequence start are halo_in rows or zero.
template <typename T>
__global__ void halo_out_kernel(const T* __restrict__ X0, const T* __restrict__ halo_in, T* __restrict__ halo_out,
                                int B, int T_len, int d, int km1) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_b = (int64_t)km1 * d;
  if (e >= (int64_t)B * per_b) return;
  const int b = (int)(e / per_b);
  const int j = (int)((e % per_b) / d);
  const int c = (int)(e % d);
  const int src = T_len - km1 + j;
  T v = static_cast<T>(0.f);
  if (src >= 0)
    v = X0[((int64_t)b * T_len + src) * d + c];
  else if (halo_in != nullptr)
    v = halo_in[((int64_t)b * km1 + km1 + src) * d + c];
  halo_out[e] = v;
}

// --------------------------------------------------------------------------- fp32 GEMM
// C[z](m, n) = scale * sum_k A[z](m, k) * B[z](k, n), with arbitrary element strides.
// Swiglu mode: C = SiLU(A B) * (A B2).  Chunk mode: z = b * n_chunks + i addresses chunk i of
// sequence b; its token rows [iC, min(iC+C, T)) move the A/B/C bases by (b*T + iC) * *_tok and
// the chunk index moves them by z * *_z; the chunk length replaces M (apply) or K (delta).
struct SgemmParams {
  const float* A;
  const float* B;
  const float* B2;
  float* Cm;
  int M, N, K;
  int64_t a_sm, a_sk, b_sk, b_sn, c_sm;
  int64_t a_tok, b_tok, c_tok;  // chunk mode: base step per token row
  int64_t a_z, b_z, c_z;        // chunk mode: base step per chunk index
  int chunked;                  // 0: plain; 1: chunk length is M; 2: chunk length is K
  int T, C, n_chunks;
  float scale;
  float beta;  // C = scale * A B + beta * C (beta = 0: C is only written)
};

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <bool SWIGLU>
__global__ void __launch_bounds__(256) sgemm_kernel(const SgemmParams p) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  __shared__ float B2s[SWIGLU ? SG_BK : 1][SWIGLU ? SG_BN + 4 : 1];
  const int z = blockIdx.z;
  const float* A = p.A;
  const float* Bm = p.B;
  const float* B2 = p.B2;
  float* Cm = p.Cm;
  int M = p.M, K = p.K;
  if (p.chunked) {
    const int b = z / p.n_chunks;
    const int i = z - b * p.n_chunks;
    const int lo = i * p.C;
    const int len = min(p.C, p.T - lo);
    const int64_t tok = (int64_t)b * p.T + lo;
    A += tok * p.a_tok + (int64_t)z * p.a_z;
    Bm += tok * p.b_tok + (int64_t)z * p.b_z;
    Cm += tok * p.c_tok + (int64_t)z * p.c_z;
    if (p.chunked == 1) M = len; else K = len;
  }
  const int m0 = blockIdx.y * SG_BM;
  const int n0 = blockIdx.x * SG_BN;
  if (m0 >= M) return;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  float acc2[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
    for (int e = threadIdx.x; e < SG_BK * SG_BM; e += 256) {
      const int kk = e / SG_BM, mm = e % SG_BM;
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < M && gk < K) ? A[gm * p.a_sm + gk * p.a_sk] : 0.f;
    }
    for (int e = threadIdx.x; e < SG_BK * SG_BN; e += 256) {
      const int kk = e / SG_BN, nn = e % SG_BN;
      const int gn = n0 + nn, gk = k0 + kk;
      const bool in = gn < p.N && gk < K;
      Bs[kk][nn] = in ? Bm[gk * p.b_sk + gn * p.b_sn] : 0.f;
      if (SWIGLU) B2s[kk][nn] = in ? B2[gk * p.b_sk + gn * p.b_sn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], bv[4], b2v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = Bs[kk][tx * 4 + j];
        if (SWIGLU) b2v[j] = B2s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
          if (SWIGLU) acc2[i][j] = fmaf(a[i], b2v[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= p.N) continue;
      float v;
      if (SWIGLU) {
        const float g = acc[i][j];
        v = g / (1.0f + expf(-g)) * acc2[i][j];
      } else {
        v = acc[i][j] * p.scale;
      }
      if (p.beta != 0.f) v += p.beta * Cm[gm * p.c_sm + gn];
      Cm[gm * p.c_sm + gn] = v;
    }
  }
}

// --------------------------------------------------------------------------- exclusive scan
// In place over the stack: on entry W[b, i] holds Delta_i (already scaled by eta); on exit
// W[b, i] = W0 + sum_{j<i} Delta_j and W_final[b] = W0 + sum_j Delta_j.
// W_init (optional, [B, d, d_ff]): each sequence's own starting state instead of W0 (W0 NULL
// too: zero).  reverse = 1 scans the chunks last to first (exclusive suffix sums).
__global__ void chunk_scan_f32_kernel(float* __restrict__ W, const float* __restrict__ W0,
                                      float* __restrict__ W_final, int B, int n_chunks, int64_t df,
                                      const float* __restrict__ W_init, int reverse) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (e >= df) return;
  float acc = W_init != nullptr ? W_init[(int64_t)b * df + e] : (W0 != nullptr ? W0[e] : 0.f);
  float* w = W + (int64_t)b * n_chunks * df + e;
  for (int j = 0; j < n_chunks; ++j) {
    const int i = reverse ? n_chunks - 1 - j : j;
    const float delta = w[(int64_t)i * df];
    w[(int64_t)i * df] = acc;
    acc += delta;
  }
  W_final[(int64_t)b * df + e] = acc;
}

// ------------------------------------------------------------------ backward-pass helpers

template <typename T>
__device__ __forceinline__ float ld_f(const T* p) { return static_cast<float>(*p); }
template <typename T>
__device__ __forceinline__ void st_f(T* p, float v) { *p = static_cast<T>(v); }

// Z = SiLU(A) * U from the saved pre-activations AU = [A | U] ([rows, 2f]).
template <typename T>
__global__ void swiglu_combine_kernel(const T* __restrict__ AU, T* __restrict__ Z, int64_t rows, int f) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= rows * f) return;
  const int64_t r = e / f;
  const int j = (int)(e % f);
  const float a = ld_f(AU + r * 2 * f + j), u = ld_f(AU + r * 2 * f + f + j);
  st_f(Z + e, a / (1.0f + expf(-a)) * u);
}

// Gated-MLP backward, in place: AU = [A | U] becomes [dA | dU] with
// dA = dZ * U * s * (1 + A (1 - s)), s = sigmoid(A), and dU = dZ * A * s (the derivative of
// SiLU(a) = a * sigmoid(a) is s (1 + a (1 - s))).
template <typename T>
__global__ void swiglu_backward_kernel(const T* __restrict__ dZ, T* __restrict__ AU, int64_t rows, int f) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= rows * f) return;
  const int64_t r = e / f;
  const int j = (int)(e % f);
  T* pa = AU + r * 2 * f + j;
  T* pu = pa + f;
  const float a = ld_f(pa), u = ld_f(pu), dz = ld_f(dZ + e);
  const float sg = 1.0f / (1.0f + expf(-a));
  st_f(pa, dz * u * sg * (1.0f + a * (1.0f - sg)));
  st_f(pu, dz * a * sg);
}

// Adjoint of the causal depthwise conv for its input: with the window shifted by `shift` tokens,
// dX0[u, c] = sum_s w[c, s] dY[u - shift + (K-1) - s, c] over the rows that exist.  Grid:
// x = blocks of 16-byte channel groups, y = blocks of CONVX_ROWS tokens, z = sequence.  Each
// thread keeps its channels' taps and a sliding window of the last K dY rows in registers, so
// it loads every dY row it needs once.
constexpr int CONVX_ROWS = 32;

template <typename T>
__device__ __forceinline__ void load_row16(const T* p, bool ok, float (&v)[16 / sizeof(T)]) {
  constexpr int VEC = 16 / sizeof(T);
  uint4 raw = make_uint4(0, 0, 0, 0);
  if (ok) raw = *reinterpret_cast<const uint4*>(p);
  const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
  for (int j = 0; j < VEC; ++j) v[j] = static_cast<float>(e[j]);
}

template <typename T, int K>
__global__ void conv_backward_x_kernel(const T* __restrict__ dY, const T* __restrict__ conv_w, T* __restrict__ dX0,
                                       int T_len, int d, int shift) {
  constexpr int VEC = 16 / sizeof(T);
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= d / VEC) return;
  const int c0 = g * VEC;
  const int u0 = blockIdx.y * CONVX_ROWS;
  const int u1 = min(u0 + CONVX_ROWS, T_len);
  const T* dy = dY + (int64_t)blockIdx.z * T_len * d + c0;
  T* dx = dX0 + (int64_t)blockIdx.z * T_len * d + c0;
  float w[K][VEC];
#pragma unroll
  for (int s = 0; s < K; ++s)
#pragma unroll
    for (int j = 0; j < VEC; ++j) w[s][j] = static_cast<float>(conv_w[(int64_t)(c0 + j) * K + s]);
  // win[m] = dY row u - shift + m (m = 0 .. K-1) for the current output row u
  float win[K][VEC];
#pragma unroll
  for (int m = 1; m < K; ++m) {
    const int r = u0 - shift + m - 1;
    load_row16(dy + (int64_t)r * d, r >= 0 && r < T_len, win[m]);
  }
  for (int u = u0; u < u1; ++u) {
#pragma unroll
    for (int m = 0; m + 1 < K; ++m)
#pragma unroll
      for (int j = 0; j < VEC; ++j) win[m][j] = win[m + 1][j];
    const int r = u - shift + K - 1;
    load_row16(dy + (int64_t)r * d, r >= 0 && r < T_len, win[K - 1]);
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
#pragma unroll
    for (int s = 0; s < K; ++s)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[j] = fmaf(w[s][j], win[K - 1 - s][j], acc[j]);
    uint4 out;
    T* o = reinterpret_cast<T*>(&out);
#pragma unroll
    for (int j = 0; j < VEC; ++j) o[j] = static_cast<T>(acc[j]);
    *reinterpret_cast<uint4*>(dx + (int64_t)u * d) = out;
  }
}

// Adjoint for the taps, in two passes (deterministic): partial[strip, c, s] = sum over the strip's
// tokens of dY[t, c] X0[t + shift - (K-1) + s, c]; then dconv_w[c, s] = sum over strips in order.
// Grid: x = strip (B * ceil(T / CONVW_STRIP)), y = blocks of 16-byte channel groups.  A sliding
// window of the last K X0 rows in registers: every row is loaded once per strip.
constexpr int CONVW_STRIP = 64;

template <typename T, int K>
__global__ void conv_backward_w_partial_kernel(const T* __restrict__ dY, const T* __restrict__ X0,
                                               float* __restrict__ partial, int T_len, int d, int shift) {
  constexpr int VEC = 16 / sizeof(T);
  const int g = blockIdx.y * blockDim.x + threadIdx.x;
  if (g >= d / VEC) return;
  const int c0 = g * VEC;
  const int strip = blockIdx.x;
  const int per_b = (T_len + CONVW_STRIP - 1) / CONVW_STRIP;
  const int b = strip / per_b;
  const int t0 = (strip % per_b) * CONVW_STRIP;
  const int t1 = min(t0 + CONVW_STRIP, T_len);
  const T* dy = dY + (int64_t)b * T_len * d + c0;
  const T* x = X0 + (int64_t)b * T_len * d + c0;
  float acc[K][VEC];
#pragma unroll
  for (int s = 0; s < K; ++s)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[s][j] = 0.f;
  // win[s] = X0 row t + shift - (K-1) + s for the current token t
  float win[K][VEC];
#pragma unroll
  for (int s = 1; s < K; ++s) {
    const int r = t0 + shift - K + s;
    load_row16(x + (int64_t)r * d, r >= 0 && r < T_len, win[s]);
  }
  for (int t = t0; t < t1; ++t) {
#pragma unroll
    for (int s = 0; s + 1 < K; ++s)
#pragma unroll
      for (int j = 0; j < VEC; ++j) win[s][j] = win[s + 1][j];
    const int r = t + shift;
    load_row16(x + (int64_t)r * d, r >= 0 && r < T_len, win[K - 1]);
    float dv[VEC];
    load_row16(dy + (int64_t)t * d, true, dv);
#pragma unroll
    for (int s = 0; s < K; ++s)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[s][j] = fmaf(dv[j], win[s][j], acc[s][j]);
  }
  float* out = partial + ((int64_t)strip * d + c0) * K;
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int s = 0; s < K; ++s) out[j * K + s] = acc[s][j];
}

__global__ void sum_strips_kernel(const float* __restrict__ partial, float* __restrict__ out, int strips, int64_t n) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  float acc = 0.f;
  for (int i = 0; i < strips; ++i) acc += partial[(int64_t)i * n + e];
  out[e] = acc;
}

// W_final[b] = W0 (as fp32) for every sequence: the state of an empty sequence.  (A resumed
// empty call copies its fp32 state with cudaMemcpyAsync instead.)
template <typename T>
__global__ void broadcast_state_kernel(const T* __restrict__ W0, float* __restrict__ W_final, int64_t df) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e < df) W_final[(int64_t)blockIdx.y * df + e] = static_cast<float>(W0[e]);
}

// One hop of the exclusive prefix over ranks (zhichai.net page, §3.2 Step 2), on elements
// [first, first + count) of a flattened [B, d, d_ff] fp32 state:
//   out[j] = base[j] + (S ? S[j] : 0),  base[j] = P_in ? P_in[j] : W0[j mod (d * d_ff)].
// Vectors of four where the range allows (first and count multiples of 4, 16-byte aligned
// pointers), single elements otherwise.  out may alias P_in or S element for element.
template <typename T>
__global__ void prefix_step_kernel(const float* P_in, const T* __restrict__ W0, const float* S, float* out,
                                   int64_t first, int64_t count, int64_t df, int vec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec) {
    for (int64_t v = i0; v < count / 4; v += stride) {
      const int64_t j = first + 4 * v;
      float4 b;
      if (P_in != nullptr) {
        b = *reinterpret_cast<const float4*>(P_in + j);
      } else {
        const int64_t e = j % df;  // df % 4 == 0: the four elements stay in one row of W0
        b = make_float4(static_cast<float>(W0[e]), static_cast<float>(W0[e + 1]), static_cast<float>(W0[e + 2]),
                        static_cast<float>(W0[e + 3]));
      }
      if (S != nullptr) {
        const float4 s = *reinterpret_cast<const float4*>(S + j);
        b.x += s.x, b.y += s.y, b.z += s.z, b.w += s.w;
      }
      *reinterpret_cast<float4*>(out + j) = b;
    }
  } else {
    for (int64_t v = i0; v < count; v += stride) {
      const int64_t j = first + v;
      float b = P_in != nullptr ? P_in[j] : static_cast<float>(W0[j % df]);
      if (S != nullptr) b += S[j];
      out[j] = b;
    }
  }
}

// The weight a chunk is applied with, from the running fp32 state: W[e] = T(state[e]) (bf16
// round to nearest even, or an fp32 copy).
template <typename T>
__global__ void state_weight_kernel(const float* __restrict__ state, T* __restrict__ W, int64_t n) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e < n) W[e] = static_cast<T>(state[e]);
}

// --------------------------------------------------------------------------- decode rows
// The few token rows of a decode step (zhichai.net page, §3.2 Step 3: the tokens of a chunk
// that is not complete yet see the weight at the chunk's start).  For a handful of rows these
// products stream each weight once at about one FLOP per byte, so they run on the CUDA cores
// across every SM: one warp per output column, each lane summing its 8-element slices in k
// order in fp32, then a fixed butterfly across the warp (the same result on every run).  The
// weights are read with the streaming cache hint; the few rows they meet stay in L1.
constexpr int DEC_ROWS = 8;  // rows of one SwiGLU launch; tokens per sequence of the apply
constexpr int DEC_THREADS = 256;

// Eight weight elements as loaded (streaming cache hint), widened to fp32 when used.
template <typename T>
struct Raw8;
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldcs(reinterpret_cast<const float4*>(p));
    b = __ldcs(reinterpret_cast<const float4*>(p + 4));
  }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};
template <>
struct Raw8<__nv_bfloat16> {
  uint4 w;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { w = __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z); v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
  }
};

// SiLU as each path computes it: the IEEE quotient in fp32, the fast one before a bf16 rounding.
template <typename T>
__device__ __forceinline__ float silu_of(float a);
template <>
__device__ __forceinline__ float silu_of<float>(float a) { return a / (1.0f + expf(-a)); }
template <>
__device__ __forceinline__ float silu_of<__nv_bfloat16>(float a) { return silu_bf16ep(a); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Z[r, n] = SiLU(H[r] . W_gate[n]) * (H[r] . W_up[n]) for the R <= RMAX rows of H [R, d].
// A block takes NB columns n at a time; its 8 warps split each dot product over interleaved
// 256-element slices of d (warp w: slices w, w+8, ...), with NB*NBATCH slices' weight loads in
// flight per lane, and the warps' partial sums meet in shared memory in warp order.  The
// block's weight rows are prefetched into L2 up front.
// The first launch of a step may also copy the step's tokens into the chunk buffers:
// H_buf[b, pos + t] = Hc[b, t] and X0_buf[b, pos + t] = X0c[b, t] for b < Bc, t < mc
// ([Bc, mc, d] in, [Bc, C, d] buffers; H_buf NULL: no copy).
template <typename T, int RMAX, int NB, int NBATCH>
__global__ void __launch_bounds__(DEC_THREADS) decode_swiglu_kernel(const T* __restrict__ H, const T* __restrict__ Wg,
                                                                    const T* __restrict__ Wu, T* __restrict__ Z, int R,
                                                                    int d, int f, const T* __restrict__ Hc,
                                                                    const T* __restrict__ X0c, T* __restrict__ H_buf,
                                                                    T* __restrict__ X0_buf, int Bc, int mc, int64_t C,
                                                                    int64_t pos) {
  constexpr int NW = DEC_THREADS / 32;
  __shared__ float part[NW][NB][RMAX][2];
  pdl_launch_dependents();  // the apply may start prefetching its weights now
  if (H_buf != nullptr) {
    const int64_t per_row = d / 8;
    const int64_t nvec = (int64_t)Bc * mc * per_row;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
      const int64_t row = v / per_row, c = (v - row * per_row) * 8;
      const int64_t b = row / mc, t = row - b * mc;
      const int64_t dst = (b * C + pos + t) * d + c;
      float x[8];
      load8(Hc + row * d + c, x);
      store8(H_buf + dst, x);
      load8(X0c + row * d + c, x);
      store8(X0_buf + dst, x);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // every weight row this block will stream, queued at once as bulk L2 prefetches: the DRAM
  // then works through one deep queue, whatever the loads in flight per lane
  if ((int)threadIdx.x < 2 * NB)
    for (int n0 = blockIdx.x * NB; n0 < f; n0 += gridDim.x * NB) {
      const int c = threadIdx.x % NB;
      if (n0 + c < f)
        prefetch_l2_bulk(((int)threadIdx.x < NB ? Wg : Wu) + (int64_t)(n0 + c) * d, (uint32_t)((int64_t)d * sizeof(T)));
    }
  for (int n0 = blockIdx.x * NB; n0 < f; n0 += gridDim.x * NB) {
    float ag[NB][RMAX], au[NB][RMAX];
#pragma unroll
    for (int c = 0; c < NB; ++c)
#pragma unroll
      for (int r = 0; r < RMAX; ++r) ag[c][r] = au[c][r] = 0.f;
    for (int k0 = (warp * 32 + lane) * 8; k0 < d; k0 += NW * 256 * NBATCH) {
      Raw8<T> gw[NBATCH][NB], uw[NBATCH][NB];
#pragma unroll
      for (int j = 0; j < NBATCH; ++j)
#pragma unroll
        for (int c = 0; c < NB; ++c)
          if (k0 + j * NW * 256 < d && n0 + c < f) {
            gw[j][c].load(Wg + (int64_t)(n0 + c) * d + k0 + j * NW * 256);
            uw[j][c].load(Wu + (int64_t)(n0 + c) * d + k0 + j * NW * 256);
          }
#pragma unroll
      for (int j = 0; j < NBATCH; ++j) {
        const int k = k0 + j * NW * 256;
        if (k >= d) break;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            float h[8];
            load8(H + (int64_t)r * d + k, h);
#pragma unroll
            for (int c = 0; c < NB; ++c) {
              if (n0 + c < f) {
                float g[8], u[8];
                gw[j][c].get(g);
                uw[j][c].get(u);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  ag[c][r] = fmaf(g[e], h[e], ag[c][r]);
                  au[c][r] = fmaf(u[e], h[e], au[c][r]);
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < NB; ++c)
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        if (r < R) {
          const float a = warp_sum(ag[c][r]), u = warp_sum(au[c][r]);
          if (lane == 0) {
            part[warp][c][r][0] = a;
            part[warp][c][r][1] = u;
          }
        }
    __syncthreads();
    if ((int)threadIdx.x < NB * R) {
      const int c = threadIdx.x / R, r = threadIdx.x - c * R;
      if (n0 + c < f) {
        float a = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          a += part[w][c][r][0];
          u += part[w][c][r][1];
        }
        Z[(int64_t)r * f + n0 + c] = static_cast<T>(silu_of<T>(a) * u);
      }
    }
    __syncthreads();
  }
}

// O[b, t, e] = sum_n Z[b, t, n] * W[b, e, n] for the R <= RMAX rows t of each of the Bq
// sequences: Z [Bq, R, f], W [Bq, d, f] (each sequence's current chunk weight), O [Bq, R, d].
// A block takes NB rows e of one sequence at a time (d % NB == 0), split over its warps as in
// decode_swiglu_kernel.  Launched as a dependent of the SwiGLU rows, it first prefetches its
// weight rows into L2 (when `prefetch`: the weights fit in L2 beside what the SwiGLU streams),
// then waits for Z.
template <typename T, int RMAX, int NB, int NBATCH>
__global__ void __launch_bounds__(DEC_THREADS) decode_apply_kernel(const T* __restrict__ Z, const T* __restrict__ W,
                                                                   T* __restrict__ O, int Bq, int R, int d, int f,
                                                                   int prefetch) {
  constexpr int NW = DEC_THREADS / 32;
  __shared__ float part[NW][NB][RMAX];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t groups = (int64_t)Bq * d / NB;
  if (prefetch && (int)threadIdx.x < NB)
    for (int64_t q = blockIdx.x; q < groups; q += gridDim.x)
      prefetch_l2_bulk(W + (q * NB + threadIdx.x) * f, (uint32_t)((int64_t)f * sizeof(T)));
  pdl_wait();
  for (int64_t q = blockIdx.x; q < groups; q += gridDim.x) {
    const int64_t row0 = q * NB;  // rows row0 .. row0+NB-1 of the [Bq*d, f] weight stack
    const int64_t b = row0 / d;
    const T* z = Z + b * R * f;
    float acc[NB][RMAX];
#pragma unroll
    for (int c = 0; c < NB; ++c)
#pragma unroll
      for (int r = 0; r < RMAX; ++r) acc[c][r] = 0.f;
    for (int n0 = (warp * 32 + lane) * 8; n0 < f; n0 += NW * 256 * NBATCH) {
      Raw8<T> ww[NBATCH][NB];
#pragma unroll
      for (int j = 0; j < NBATCH; ++j)
#pragma unroll
        for (int c = 0; c < NB; ++c)
          if (n0 + j * NW * 256 < f) ww[j][c].load(W + (row0 + c) * f + n0 + j * NW * 256);
#pragma unroll
      for (int j = 0; j < NBATCH; ++j) {
        const int n = n0 + j * NW * 256;
        if (n >= f) break;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            float zv[8];
            load8(z + (int64_t)r * f + n, zv);
#pragma unroll
            for (int c = 0; c < NB; ++c) {
              float wv[8];
              ww[j][c].get(wv);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[c][r] = fmaf(wv[i], zv[i], acc[c][r]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < NB; ++c)
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        if (r < R) {
          const float o = warp_sum(acc[c][r]);
          if (lane == 0) part[warp][c][r] = o;
        }
    __syncthreads();
    if ((int)threadIdx.x < NB * R) {
      const int c = threadIdx.x / R, r = threadIdx.x - c * R;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) o += part[w][c][r];
      const int64_t e = row0 + c - b * d;
      O[(b * R + r) * d + e] = static_cast<T>(o);
    }
    __syncthreads();
  }
}

// Device-side wait that nothing ever signals: exercises the bounded-wait path.
__global__ void wait_probe_kernel(DevStatus st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(&bar, 0, st, reinterpret_cast<volatile int*>(&abort_flag), 0x301);
  __syncthreads();
}

}  // namespace simt
}  // namespace ipttt
