/*
 * ipttt.h -- C ABI of the In-Place TTT fast-weight SwiGLU layer for NVIDIA B300 (sm_103a).
 *
 * The layer (zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，让它边读边学"; ordering also in
 * the xiaoxiang.io summary "原位测试时训练", 核心方法 item 3) computes, for each sequence b:
 *
 *   (1) Z      = SiLU(H W_gate^T) * (H W_up^T)                    §3.1 gated-MLP equation
 *   (2) V      = CausalConv1D(X0) W_target                         §3.3 LM-aligned target
 *   (3) D_i    = V_i^T Z_i for every C-token chunk i               §3.2 Step 1, §3.3 update rule
 *   (4) W_i    = W_down0 + eta * sum_{j<i} D_j  (exclusive prefix) §3.2 Step 2, bullets 2-4
 *   (5) O_i    = Z_i W_i^T                                          §3.1, §3.2 Step 3
 *   and returns O and the final state W_down0 + eta * sum_j D_j.
 *
 * Readings fixed by this ABI (the pages are silent or garbled there):
 *   - the conv is depthwise, zero left-padded by k-1 per sequence, no bias; conv_w[c, k-1]
 *     multiplies the current token, conv_w[c, 0] the token k-1 steps back;
 *   - V = Y W_target with W_target stored [d_in, d_out] (right-multiplied, as printed);
 *   - the loss printed as -<V, Z W_down>_F is read as -<V, Z W_down^T>_F, whose negative
 *     gradient is the printed update direction V^T Z;
 *   - eta is applied as given; a last chunk shorter than C is a chunk of its own;
 *   - a batch holds independent sequences, each with its own padding and its own state.
 *
 * Conventions for every entry point
 *   - All tensors are dense row-major.  Device pointers are allocated and owned by the
 *     caller; the library never allocates device memory in a compute call.  Every pointer
 *     passed to a compute call must be 16-byte aligned.  Inputs are read only; outputs
 *     and the workspace must not overlap the inputs or each other.
 *   - dtype IPTTT_BF16: H, X0, weights, O, workspace tensors are bf16; products accumulate
 *     in fp32 on the tensor cores; the running state is fp32; Z, V and the per-chunk
 *     weights W_i are rounded to bf16 (round-to-nearest-even).  Requires C % 128 == 0.
 *     dtype IPTTT_F32: everything fp32 on CUDA cores (any C >= 1).
 *     Both require d % 8 == 0, d_ff % 8 == 0, 1 <= k <= 8, B*T < 2^31.
 *   - Compute calls are asynchronous on the context's stream.  Argument errors are
 *     reported before anything is launched.  A device-side wait that runs past the
 *     context's limit makes the kernel record IPTTT_ERR_TIMEOUT and return; the code is
 *     reported by the next ipttt_sync().  No call throws or aborts the process.
 *   - Every failing call stores a message retrievable with ipttt_last_error().
 *   - A context is used by one host thread at a time (calls on one context are not
 *     synchronised with each other); separate contexts may be used from separate threads
 *     (ipttt_target_noalloc, which takes no context, shares one scratch: see there).
 */
#ifndef IPTTT_H
#define IPTTT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ipttt_ctx ipttt_ctx; /* opaque */

typedef enum {
  IPTTT_OK = 0,
  IPTTT_ERR_INVALID_ARG = 1, /* null / misaligned / overlapping pointer, negative size ... */
  IPTTT_ERR_UNSUPPORTED = 2, /* valid but unsupported shape or dtype combination          */
  IPTTT_ERR_WORKSPACE = 3,   /* workspace missing or smaller than ipttt_workspace_size() */
  IPTTT_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed                      */
  IPTTT_ERR_TIMEOUT = 5      /* a device-side wait ran past the limit (see ipttt_sync)  */
} ipttt_status;

typedef enum { IPTTT_F32 = 0, IPTTT_BF16 = 1 } ipttt_dtype;

/* Kernel stages as reported by ipttt_timing_read(), in the order a layer call runs them on
 * the context's stream: the causal conv, the SwiGLU GEMM, the W_target projection, the
 * chunk updates and the apply.  With step (2) as one kernel (ipttt_set_fused_target) the
 * conv stage has zero length and the target stage holds both. */
typedef enum {
  IPTTT_STAGE_SWIGLU = 0, /* step (1)                                     */
  IPTTT_STAGE_CONV = 1,   /* causal conv of step (2), run before (1)       */
  IPTTT_STAGE_TARGET = 2, /* W_target projection of step (2), times eta   */
  IPTTT_STAGE_STATE = 3,  /* steps (3)+(4); with the fused kernel (3)-(5) */
  IPTTT_STAGE_APPLY = 4,  /* step (5); 0 with the fused kernel            */
  IPTTT_NUM_STAGES = 5
} ipttt_stage;

/* Library version as "major.minor.patch"; static string. */
const char* ipttt_version(void);

/* Human-readable name of a status code; static string. */
const char* ipttt_status_string(ipttt_status s);

/* Create a context on CUDA device `device`, bound to `cuda_stream` (a cudaStream_t; NULL =
 * the legacy default stream).  Allocates a 8-byte device status word, CUDA events and three
 * internal streams (the upload and download streams of ipttt_layer_forward_host, and the
 * stream of the bf16 backward pass's target branch), each ordered after and joined back into
 * the context's stream by events; this is the only call that allocates device memory.  *out
 * receives the context.
 * Errors: INVALID_ARG (out == NULL, bad device), CUDA. */
ipttt_status ipttt_create(ipttt_ctx** out, int device, void* cuda_stream);

/* Rebind the context to another stream of the same device. */
ipttt_status ipttt_set_stream(ipttt_ctx* ctx, void* cuda_stream);

/* bf16 layer calls run steps (3)-(5) as one cooperative kernel by default: the state units
 * run first and the per-chunk apply tiles fill the SMs the state work leaves idle (each tile
 * waits on device-side counters until the weights of its chunk are written).  enable = 0
 * selects two separate kernels instead (same results, bit for bit); devices without
 * cooperative launch, and calls whose cooperative grid no longer fits the SMs available to the
 * context, use two. */
ipttt_status ipttt_set_fused_tail(ipttt_ctx* ctx, int enable);

/* Width of the apply tiles of that cooperative kernel on CTA pairs: halves = 0 (default)
 * chooses per call (256 x 512 tiles when d_ff / 64 >= 128 and they make at least two waves
 * over the co-resident pairs, else 256 x 256), 1 always 256 x 256 (two accumulators in turn),
 * 2 always 256 x 512 (one accumulator, a quarter fewer operand bytes per FLOP).  Results are
 * bit-identical: every output element is the same fp32 sum in the same order.
 * Errors: INVALID_ARG (halves not 0, 1 or 2). */
ipttt_status ipttt_set_apply_tiles(ipttt_ctx* ctx, int halves);

/* Choose how step (2) of a bf16 layer call runs: enable = 0 (default) as the conv kernel
 * (memory bound, before step (1)) followed by the W_target GEMM; enable = 1 as one kernel on
 * CTA pairs whose extra warps form each tile of the conv output Y = CausalConv1D(X0) in
 * shared memory straight from X0 for the GEMM, so that Y is never stored.  Results are
 * bit-identical: Y is the same fp32 fma chain rounded to bf16 either way.  The one-kernel form
 * forms each Y tile once per 256-column block of V (d/256 times in all) on the CUDA cores, and
 * at the 4B shape it is the slower of the two.  The training forward, calls without W_target
 * and the single-CTA GEMMs always run the two kernels; ipttt_target always does (it returns
 * Y). */
ipttt_status ipttt_set_fused_target(ipttt_ctx* ctx, int enable);

/* Choose how the bf16 GEMMs of steps (1), (2) and (5) run: enable = 1 (default) on CTA pairs
 * (clusters of two SMs issuing tcgen05.mma.cta_group::2 on 256-row tiles; the chunk apply
 * only when C % 256 == 0), 0 on single CTAs (128-row tiles).  Results are bit-identical:
 * every output element is the same fp32 sum in the same order, only the tiling differs. */
ipttt_status ipttt_set_cta_pairs(ipttt_ctx* ctx, int enable);

/* Ablation variant of the target (zhichai.net page §6, conv/proj ablation; its Theorem 1 uses
 * the next token's embedding as target): shift = 1 moves the conv window one token later, so
 * that the target of token t ends at X0[t+1] (the token after a call's last one reads as
 * zero); shift = 0 (default) is the causal window.  A piece of a sequence would need the
 * next piece's first X0 row for its last target, so with shift = 1 the entry points that
 * run a sequence in pieces return UNSUPPORTED: ipttt_layer_forward_resume,
 * ipttt_layer_totals, and ipttt_layer_forward_host when T spans more than one of its
 * pieces.  ipttt_layer_forward, ipttt_target and the backward pass take it.
 * The other ablations need no switch: W_target = NULL is "w/o Proj" (identity projection;
 * the projection GEMM is skipped), k = 1 with conv_w = 1 is "w/o Conv". */
ipttt_status ipttt_set_target_shift(ipttt_ctx* ctx, int shift);

/* Limit, in nanoseconds, on every device-side wait of later launches (default 2e9). */
ipttt_status ipttt_set_wait_limit_ns(ipttt_ctx* ctx, uint64_t ns);

/* Wait for the context's stream, then read and clear the device status word.
 * Returns IPTTT_ERR_TIMEOUT if a kernel gave up a wait since the last sync, CUDA on a
 * CUDA error, else OK. */
ipttt_status ipttt_sync(ipttt_ctx* ctx);

/* Message of the last failing call on this context (empty string if none). */
const char* ipttt_last_error(const ipttt_ctx* ctx);

/* Destroy a context (NULL is ignored).  Waits for nothing: sync first. */
void ipttt_destroy(ipttt_ctx* ctx);

/* Bytes of device workspace ipttt_layer_forward needs for this shape (host-only call, no
 * GPU needed).  Layout: Y [B,T,d], V [B,T,d], Z [B,T,d_ff], W stack [B,ceil(T/C),d,d_ff],
 * each in `dtype`, then B*ceil(T/C)+1 uint32 counters; each region 256-byte aligned.
 * Errors: INVALID_ARG (bytes == NULL, negative sizes, C < 1, k < 1), UNSUPPORTED. */
ipttt_status ipttt_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                  ipttt_dtype dtype, size_t* bytes);

/* The whole layer, steps (1)-(5).
 *   H, X0     [B, T, d]        dtype, device      hidden state; embedding output
 *   W_gate    [d_ff, d]        dtype, device      frozen, shared by all sequences
 *   W_up      [d_ff, d]        dtype, device      frozen
 *   W_down0   [d, d_ff]        dtype, device      initial fast weight
 *   W_target  [d, d]           dtype, device      [d_in, d_out], V = Y W_target; NULL = identity
 *   conv_w    [d, k]           dtype, device      depthwise causal taps
 *   O         [B, T, d]        dtype, device      output
 *   W_final   [B, d, d_ff]     fp32,  device      state after the last chunk's update
 *   workspace                  device, >= ipttt_workspace_size() bytes, overwritten
 * B = 0 is a no-op; T = 0 sets W_final[b] = W_down0 for every b.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA (launch). */
ipttt_status ipttt_layer_forward(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                 const void* W_up, const void* W_down0, const void* W_target,
                                 const void* conv_w, int64_t B, int64_t T, int64_t d, int64_t d_ff,
                                 int64_t C, int k, float eta, ipttt_dtype dtype, void* O,
                                 float* W_final, void* workspace, size_t workspace_bytes);

/* Continue B sequences where an earlier call left them: streaming, read-while-learn use
 * (zhichai.net page §9, future directions; one fast-weight state per session as in the
 * travelaiplan.net engineering blog §4).  Same computation as ipttt_layer_forward, except that
 *   W_state     [B, d, d_ff]  fp32, device   each sequence's fast weight at this call's first
 *                                            token (W_down0 broadcast for a new sequence; the
 *                                            W_state_out of the previous call otherwise)
 *   X0_halo     [B, k-1, d]   dtype, device  the k-1 X0 rows before this call's first token
 *                                            (NULL = zeros: a new sequence)
 *   W_state_out [B, d, d_ff]  fp32, device   the state after this call's last chunk; may be
 *                                            W_state itself (updated in place)
 *   X0_halo_out [B, k-1, d]   dtype, device  (NULL = not written) the last k-1 rows of
 *                                            [X0_halo, X0], the next call's X0_halo; must not
 *                                            overlap X0_halo
 * Chunks are counted from this call's first token, so a sequence cut at multiples of C and
 * fed call by call gives exactly the results of one call over the whole sequence (bit for bit
 * on the GPU).  A call of T = C tokens is the decode step: buffer C tokens, then run them.
 * The workspace is that of ipttt_layer_forward.  Errors as ipttt_layer_forward. */
ipttt_status ipttt_layer_forward_resume(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                        const void* W_up, const void* W_target, const void* conv_w,
                                        const float* W_state, const void* X0_halo, int64_t B, int64_t T,
                                        int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                        ipttt_dtype dtype, void* O, float* W_state_out, void* X0_halo_out,
                                        void* workspace, size_t workspace_bytes);

/* ---- context parallelism: the pages' three steps (§3.2) on one rank ----
 * Step 1, ipttt_layer_totals: for a rank's range of tokens of every sequence (the conv
 * continuing from X0_halo, the k-1 X0 rows before the range, NULL = zeros), Z and V go to
 * `saved` (the ipttt_saved_size() layout) and S[b] = eta * sum_i V_i^T Z_i [B, d, d_ff] fp32
 * is the range's update total, accumulated from zero with no per-chunk weight written.
 * Step 2, ipttt_prefix_step: the rank's starting state is W_down0 plus the totals of the
 * ranks before it, carried from rank to rank as a chain: rank 0's state is W_down0, and each
 * rank adds its own total to the state it received and passes the sum on (the caller moves
 * the buffers between ranks).  Step 3, ipttt_layer_apply_saved: from that state W_init [B, d, d_ff]
 * fp32 and the same `saved`, O [B, T, d] and the state after the range W_final [B, d, d_ff]
 * fp32 (W_final may be W_init itself); Z and V are not computed again.  Errors as the layer
 * calls. */
ipttt_status ipttt_layer_totals(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                const void* W_up, const void* W_target, const void* conv_w,
                                const void* X0_halo, int64_t B, int64_t T, int64_t d, int64_t d_ff,
                                int64_t C, int k, float eta, ipttt_dtype dtype, float* S, void* saved,
                                size_t saved_bytes);

/* Step 2, one hop of the chain, on the elements [first, first + count) of the flattened
 * [B, d, d_ff] fp32 state (so that a caller can pass the state on in pieces while later pieces
 * are still arriving):
 *   P_out[j] = base[j] + S[j],   base[j] = P_in[j], or W_down0[j mod (d * d_ff)] widened to
 *                                fp32 when P_in is NULL (rank 0; the same W_down0 for every b)
 *   P_in, S, P_out  [B, d, d_ff] fp32, device; S NULL = zeros (the state itself, e.g. rank 0's
 *                   own starting state); P_out may be P_in or S itself (elementwise in place)
 *   W_down0         [d, d_ff] dtype, device (read only when P_in is NULL)
 * One fp32 addition per element, so every rank of a chain gets the sum of the totals before
 * it in rank order whatever the pieces.  Errors: INVALID_ARG (NULL or misaligned pointers,
 * a range outside the state, partial overlap), UNSUPPORTED (sizes as ipttt_layer_forward). */
ipttt_status ipttt_prefix_step(ipttt_ctx* ctx, const float* P_in, const void* W_down0, const float* S,
                               int64_t B, int64_t d, int64_t d_ff, ipttt_dtype dtype, int64_t first,
                               int64_t count, float* P_out);

ipttt_status ipttt_layer_apply_saved(ipttt_ctx* ctx, const float* W_init, int64_t B, int64_t T,
                                     int64_t d, int64_t d_ff, int64_t C, ipttt_dtype dtype, void* saved,
                                     size_t saved_bytes, void* O, float* W_final);

/* Bytes of device workspace ipttt_layer_forward_host needs: ipttt_workspace_size() for one
 * piece (see below), then device staging for the whole H, X0 and O, the fp32 state [B,d,d_ff]
 * and two conv halos [B,k-1,d]. */
ipttt_status ipttt_host_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                       ipttt_dtype dtype, size_t* bytes);

/* The whole layer with the activations and results in HOST memory (pinned memory gives
 * asynchronous copies): H_host, X0_host [B,T,d] dtype in, O_host [B,T,d] dtype and
 * W_final_host [B,d,d_ff] fp32 out; the frozen weights stay device pointers.  The call runs in
 * pieces of about 4096 tokens (a multiple of C, at most 64 pieces; with several pieces the
 * last one's tokens are cut into halves of halves down to C): piece j is uploaded on an
 * internal copy stream, computed on the context's stream as a resumed call (the state and conv
 * halo of piece j-1), and its O downloaded on a second copy stream, so the copies of one piece
 * overlap the compute of its neighbours.  Pieces start at multiples of C, so the results equal
 * ipttt_layer_forward's bit for bit.  Everything is ordered after the work already on the
 * context's stream, and the context's stream waits for all of it at the end: the host buffers
 * must stay valid until ipttt_sync() returns.  Errors as ipttt_layer_forward. */
ipttt_status ipttt_layer_forward_host(ipttt_ctx* ctx, const void* H_host, const void* X0_host,
                                      const void* W_gate, const void* W_up, const void* W_down0,
                                      const void* W_target, const void* conv_w, int64_t B, int64_t T,
                                      int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                      ipttt_dtype dtype, void* O_host, float* W_final_host,
                                      void* workspace, size_t workspace_bytes);

/* The weight a chunk is applied with, from a running fp32 state (the decode path of a stream:
 * tokens of a chunk that is not complete yet are applied with the weight at the chunk's start,
 * §3.2 Step 3): W[b] = W_state[b] rounded to dtype (bf16 round to nearest even; fp32 copies).
 * W_state [B, d, d_ff] fp32, W [B, d, d_ff] dtype, both device; they must not overlap.
 * Errors: INVALID_ARG, UNSUPPORTED (as ipttt_workspace_size for d, d_ff, dtype), CUDA. */
ipttt_status ipttt_state_weight(ipttt_ctx* ctx, const float* W_state, int64_t B, int64_t d, int64_t d_ff,
                                ipttt_dtype dtype, void* W);

/* One decode step of a stream (§3.2 Step 3 for the tokens of a chunk that is not complete yet):
 * for m (1..8) new tokens of each of B sequences, Z = SiLU(H W_gate^T) * (H W_up^T) and
 * O[b] = Z[b] W_cur[b]^T, W_cur [B, d, d_ff] dtype being each sequence's weight at the
 * chunk's start (ipttt_state_weight of its state).  H [B, m, d] in; Z [B, m, d_ff] and
 * O [B, m, d] out, all dtype, all device.  With the chunk buffers H_buf and X0_buf
 * ([B, C, d], both or neither), the step also stores H[b, t] and X0[b, t] (X0 [B, m, d]) at
 * token pos + t of the buffers (pos + m <= C), so that the chunk's update can be committed
 * with ipttt_layer_forward_resume once it completes.  The apply, and the SwiGLU of a single
 * token row (or of any rows in fp32), run on the CUDA cores as weight-streaming dot products
 * over every SM with fp32 sums in a fixed order (the same on every run); several bf16 rows take
 * the tensor-core SwiGLU.  The outputs agree with the chunked path's to rounding, not bit for
 * bit.
 * Outputs must not overlap inputs or each other.  Errors: INVALID_ARG, UNSUPPORTED (m outside
 * 1..8; as ipttt_workspace_size for d, d_ff, dtype), CUDA. */
ipttt_status ipttt_decode_step(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                               const void* W_up, const void* W_cur, int64_t B, int64_t m, int64_t d,
                               int64_t d_ff, ipttt_dtype dtype, void* Z, void* O, void* H_buf,
                               void* X0_buf, int64_t C, int64_t pos);

/* ---- backward pass ----
 * The pages train the layer (§5 results: continued training of a 4B model, experiment 1, and
 * pretraining from scratch, experiment 3) but print no gradient formulas; these are the exact
 * derivatives of steps (1)-(5) by the chain rule, for a loss L(O, W_final).  With
 * G_i = dO_i^T Z_i and R_i = dW_final + sum_{l>i} G_l (the gradient reaching the state after
 * chunk i, an exclusive suffix sum: the forward's prefix scan run backwards):
 *   dW_down0 = sum_b (dW_final[b] + sum_i G_i)
 *   dZ_i     = dO_i W_i + eta V_i R_i              dV_i = eta Z_i R_i^T
 *   dA, dU   = the SwiGLU adjoints of dZ            (A = H W_gate^T, U = H W_up^T)
 *   dH = dA W_gate + dU W_up    dW_gate = dA^T H    dW_up = dU^T H
 *   dY = dV W_target^T          dW_target = Y^T dV  (Y = CausalConv1D(X0))
 *   dX0, dconv_w                the conv's adjoints (the window shift of
 *                               ipttt_set_target_shift is honoured).
 * The forward quantities (Z, A, U, Y, V and every W_i) are recomputed, not passed in. */

/* Bytes of device workspace ipttt_layer_backward needs (host-only call).  Layout: Y, V [B,T,d],
 * Z [B,T,d_ff], [A|U] [B,T,2*d_ff], dZ [B,T,d_ff] (fp32 only), dV, dY [B,T,d], the W_i and
 * R_i stacks [B,ceil(T/C),d,d_ff] (all dtype), per-sequence dW_down0 [B,d,d_ff] fp32 and the
 * conv-tap partial sums [B*ceil(T/64),d,k] fp32; each region 256-byte aligned.  Errors as
 * ipttt_workspace_size. */
ipttt_status ipttt_backward_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                                           ipttt_dtype dtype, size_t* bytes);

/* Gradients of the whole layer.  Inputs as ipttt_layer_forward, plus
 *   dO        [B, T, d]        dtype, device      gradient of the loss w.r.t. O
 *   dW_final  [B, d, d_ff]     fp32,  device      gradient w.r.t. W_final; NULL = zero
 * Outputs (overwritten, never accumulated into):
 *   dH, dX0   [B, T, d]        dtype, device
 *   dW_gate, dW_up [d_ff, d]   fp32,  device      summed over the batch
 *   dW_down0  [d, d_ff]        fp32,  device      summed over the batch
 *   dW_target [d, d]           fp32,  device      NULL allowed (and ignored) iff W_target is NULL
 *   dconv_w   [d, k]           fp32,  device
 *   workspace                  device, >= ipttt_backward_workspace_size() bytes, overwritten
 * bf16: every product on the tensor cores with fp32 accumulation; the intermediates (Z, V,
 * W_i, R_i, dA, dU, dV, dY) are rounded to bf16 between steps (dZ stays fp32: the SwiGLU
 * adjoints are taken in the epilogue of the GEMM that forms it).  B*T = 0 writes zeros
 * (dW_down0 = sum_b dW_final[b]).  Also requires B <= 65535 and T <= 2097120.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. */
ipttt_status ipttt_layer_backward(ipttt_ctx* ctx, const void* H, const void* X0, const void* W_gate,
                                  const void* W_up, const void* W_down0, const void* W_target,
                                  const void* conv_w, int64_t B, int64_t T, int64_t d, int64_t d_ff,
                                  int64_t C, int k, float eta, ipttt_dtype dtype, const void* dO,
                                  const float* dW_final, void* dH, void* dX0, float* dW_gate, float* dW_up,
                                  float* dW_down0, float* dW_target, float* dconv_w, void* workspace,
                                  size_t workspace_bytes);

/* ---- training: the forward keeps what the backward pass reads ----
 * ipttt_layer_forward_train computes what ipttt_layer_forward computes, bit for bit, and also
 * keeps in `saved` the activations the backward pass would otherwise recompute: Z
 * [B,T,d_ff], the gate and up pre-activations [A | U] [B,T,2 d_ff], Y = CausalConv1D(X0)
 * [B,T,d], V = eta * Y W_target [B,T,d] and the weight of every chunk W_i [B,n,d,d_ff]
 * (W_0 = W_down0 included), all dtype, then n*B+1 uint32 counters; each region 256-byte
 * aligned.  ipttt_layer_backward_saved then runs only the backward half; it overwrites the
 * [A | U] region with [dA | dU], so a saved buffer serves one backward call. */

/* Bytes of the saved-activation buffer (host-only call).  Errors as ipttt_workspace_size. */
ipttt_status ipttt_saved_size(int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C, int k,
                              ipttt_dtype dtype, size_t* bytes);

/* Bytes of device workspace ipttt_layer_backward_saved needs: dZ (fp32 only), dV, dY, the
 * R_i stack, per-sequence dW_down0 and the conv-tap partial sums, as in
 * ipttt_backward_workspace_size.  Errors as ipttt_workspace_size. */
ipttt_status ipttt_backward_saved_workspace_size(int64_t B, int64_t T, int64_t d, int64_t d_ff,
                                                 int64_t C, int k, ipttt_dtype dtype, size_t* bytes);

/* The layer (arguments as ipttt_layer_forward) with `saved` (device, >= ipttt_saved_size()
 * bytes, overwritten) in place of the workspace.  Errors as ipttt_layer_forward. */
ipttt_status ipttt_layer_forward_train(ipttt_ctx* ctx, const void* H, const void* X0,
                                       const void* W_gate, const void* W_up, const void* W_down0,
                                       const void* W_target, const void* conv_w, int64_t B, int64_t T,
                                       int64_t d, int64_t d_ff, int64_t C, int k, float eta,
                                       ipttt_dtype dtype, void* O, float* W_final, void* saved,
                                       size_t saved_bytes);

/* The gradients of ipttt_layer_backward from a saved buffer that ipttt_layer_forward_train
 * filled with the same inputs (W_down0 is not needed: every W_i is saved).  Arguments and
 * outputs as ipttt_layer_backward; the workspace is >= ipttt_backward_saved_workspace_size()
 * bytes.  The [A | U] region of `saved` is overwritten.  Errors as ipttt_layer_backward. */
ipttt_status ipttt_layer_backward_saved(ipttt_ctx* ctx, const void* H, const void* X0,
                                        const void* W_gate, const void* W_up, const void* W_target,
                                        const void* conv_w, int64_t B, int64_t T, int64_t d,
                                        int64_t d_ff, int64_t C, int k, float eta, ipttt_dtype dtype,
                                        void* saved, size_t saved_bytes, const void* dO,
                                        const float* dW_final, void* dH, void* dX0, float* dW_gate,
                                        float* dW_up, float* dW_down0, float* dW_target,
                                        float* dconv_w, void* workspace, size_t workspace_bytes);

/* ---- the individual steps (the layer is exactly these calls in this order) ---- */

/* Step (1), §3.1: Z[r] = SiLU(H[r] W_gate^T) * (H[r] W_up^T) for rows r < rows (rows = B*T).
 * H [rows, d], W_gate/W_up [d_ff, d], Z [rows, d_ff], all dtype. */
ipttt_status ipttt_swiglu(ipttt_ctx* ctx, const void* H, const void* W_gate, const void* W_up,
                          int64_t rows, int64_t d, int64_t d_ff, ipttt_dtype dtype, void* Z);

/* Step (2), §3.3: Y = CausalConv1D(X0) (per sequence), V = scale * (Y W_target).
 * X0 [B,T,d], conv_w [d,k], W_target [d,d], Y (scratch, written) [B,T,d], V [B,T,d].
 * W_target = NULL: V = scale * Y written directly (Y may then be NULL). */
ipttt_status ipttt_target(ipttt_ctx* ctx, const void* X0, const void* conv_w, const void* W_target,
                          int64_t B, int64_t T, int64_t d, int k, float scale, ipttt_dtype dtype,
                          void* Y, void* V);

/* Steps (3)+(4), §3.2 Steps 1-2, §3.3 update: with V already scaled by eta,
 * W_eff[b, i] = W_down0 + sum_{j<i} V_j^T Z_j and W_final[b] = W_down0 + sum_j V_j^T Z_j.
 * V [B,T,d], Z [B,T,d_ff], W_down0 [d,d_ff] dtype; W_eff [B,ceil(T/C),d,d_ff] dtype;
 * W_final [B,d,d_ff] fp32.  Requires T >= 1. */
ipttt_status ipttt_chunk_state(ipttt_ctx* ctx, const void* V, const void* Z, const void* W_down0,
                               int64_t B, int64_t T, int64_t d, int64_t d_ff, int64_t C,
                               ipttt_dtype dtype, void* W_eff, float* W_final);

/* Step (5), §3.2 Step 3: O[b, chunk i] = Z[b, chunk i] W_eff[b, i]^T.
 * Z [B,T,d_ff], W_eff [B,ceil(T/C),d,d_ff], O [B,T,d], all dtype.  Requires T >= 1. */
ipttt_status ipttt_chunk_apply(ipttt_ctx* ctx, const void* Z, const void* W_eff, int64_t B, int64_t T,
                               int64_t d, int64_t d_ff, int64_t C, ipttt_dtype dtype, void* O);

/* ---- allocation-free variant ----
 *
 * The paper has no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory.  Examples: code that runs inside a host application whose device
 * memory belongs to that application's own allocator or pool (and that therefore holds no
 * right to call cudaMalloc), latency-critical loops where cudaMalloc / cudaFree could
 * synchronise the device, and deployments whose device footprint must be fixed when the
 * library is loaded.  Such callers cannot provide the Y scratch that ipttt_target needs.
 */

/* Size of the built-in scratch of ipttt_target_noalloc: 16 MiB of device memory that every
 * GPU which loads this library reserves until the process exits.  The first 256 bytes hold
 * a fallback status word; the rest holds the conv output Y. */
#define IPTTT_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Step (2) exactly as ipttt_target computes it (same kernels, same results), but with the
 * conv output Y kept in the library's built-in scratch instead of a caller buffer, and
 * without a context.  It allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library call.
 *   X0 [B,T,d], conv_w [d,k], W_target [d,d], V [B,T,d] (output), all `dtype`, device,
 *   16-byte aligned.  V = scale * (CausalConv1D(X0) W_target).
 *   status: optional device pointer to two uint32 words owned by the caller (zero them
 *   before the first call); a device-side wait that runs past 2 s writes IPTTT_ERR_TIMEOUT
 *   and a site code there.  With NULL a word inside the built-in scratch is used instead
 *   and such a timeout is not reported.
 *   cuda_stream: the stream to launch on (NULL = legacy default stream).
 * Runs on the calling thread's current CUDA device.  The first call on each device sets
 * up that device (looks up the scratch's device address with cudaGetSymbolAddress, finds
 * the tensor-map encoder, sets kernel attributes): make that first call before any CUDA
 * stream capture begins.  Later calls only launch two kernels.
 * All calls share the one scratch, which keeps the last call's contents; nothing in it has
 * to start at zero, because each call writes every element of Y it later reads.  Calls
 * whose kernels may overlap on the GPU (other streams, or other host threads without
 * ordering between them) race on the scratch and give wrong results: serialise them.
 * Errors: INVALID_ARG (NULL / misaligned pointer, bad sizes), UNSUPPORTED (as
 * ipttt_target), WORKSPACE when B*T*d*sizeof(dtype) > IPTTT_NOALLOC_SCRATCH_BYTES - 256
 * (nothing is launched), CUDA. */
ipttt_status ipttt_target_noalloc(const void* X0, const void* conv_w, const void* W_target, int64_t B,
                                  int64_t T, int64_t d, int k, float scale, ipttt_dtype dtype, void* V,
                                  uint32_t* status, void* cuda_stream);

/* ---- measurement and self-test ---- */

/* Start timing: later layer calls record a CUDA event at every stage boundary (up to 256
 * calls); earlier records are discarded. */
ipttt_status ipttt_timing_begin(ipttt_ctx* ctx);

/* Stop timing and read it: waits for the recorded events, then writes the summed device
 * time in ms of each stage to ms[IPTTT_NUM_STAGES], the number of timed layer calls to
 * *calls and the number of kernels those calls launched to *launches. */
ipttt_status ipttt_timing_read(ipttt_ctx* ctx, double* ms, int64_t* calls, int64_t* launches);

/* Number of kernels one ipttt_layer_forward call launches for this shape with the default
 * settings (host only): bf16 3 (step (2) and steps (3)-(5) each one kernel), fp32 6; T = 0:
 * 1; B = 0: 0. */
int64_t ipttt_layer_launches(int64_t B, int64_t T, ipttt_dtype dtype);

/* Launch one block that waits on a shared-memory barrier nothing ever signals, through
 * the same bounded wait as the layer's kernels; it returns after the context's wait limit.
 * The following ipttt_sync() must return IPTTT_ERR_TIMEOUT and the context stays usable. */
ipttt_status ipttt_selftest_wait_timeout(ipttt_ctx* ctx);

/* Number of streaming multiprocessors of the context's device. */
int ipttt_sm_count(const ipttt_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* IPTTT_H */
