/*
 * ne_attn.h -- C ABI of the GB300 (sm_103a) causal self-attention library with
 * rotary position embedding (RoPE), forward and backward.
 *
 * The operation (per sequence, per head, positions m, n = 0..L-1; the pages
 * print no equations, so the standard definitions are restated here):
 *   q'_m = R(m) q_m, k'_n = R(n) k_n        RoPE, rotate-half pairing (element
 *                                           i with i + D/2), theta_i =
 *                                           base^(-(2i)/D), angle m * theta_i
 *   S_mn = scale * q'_m . k'_n              for n <= m (causal)
 *   LSE_m = log sum_{n<=m} exp(S_mn)        natural log, scale included
 *   O_m = sum_{n<=m} exp(S_mn - LSE_m) v_n
 * and the backward returns dq, dk, dv with respect to the UN-rotated q and k
 * (the rotation is inside the operation).
 * Sources: causal self-attention with RoPE applied to the projections --
 * "Tiny Hackable CUDA: C ve CUDA ile Sifirdan Dil Modeli Gelistirmek",
 * section 3; a hand-written FlashAttention with RoPE in a CUDA engine whose
 * analytic gradients (including through RoPE) are checked against a centred
 * finite difference -- NanoEuler Show HN page, paragraph 2; 12 heads of width
 * 64 (GPT-2 small) -- techinfos.ro NanoEuler article, section "Arhitectura si
 * tehnologii folosite".  RoPE itself: RoFormer (Su et al. 2021).
 *
 * Conventions shared by every entry point:
 *  - Head dimension D must be 64 (NE_ERR_UNSUPPORTED otherwise).
 *  - q, k, v, out, dout, dq, dk, dv are bf16 (raw 16-bit words, type
 *    ne_bf16), row-major [B, T, H, 64] for the fixed-length calls and
 *    [N_tot, H, 64] for the varlen calls, 64 contiguous.  Every one of these
 *    pointers must be 16-byte aligned (NE_ERR_MISALIGNED).
 *  - lse is fp32 [B, H, T] (fixed length) or [H, N_tot] (varlen), 4-byte
 *    aligned.
 *  - Sizes: fewer than 2^31 rows (B * T or N_tot) and fewer than 2^31
 *    (row, head) pairs (rows * H: each tensor then stays under 256 GB), at
 *    most 65535 key tiles of 128 rows per sequence; a larger problem is
 *    refused with NE_ERR_INVALID_ARG.
 *  - Every pointer is DEVICE memory owned by the caller; the library keeps no
 *    reference to it after the call returns.  The library owns only its RoPE
 *    cos/sin tables, one temporary per stream for the forward's rotated keys
 *    (k' = R(n) k, 128 bytes per token and head, allocated stream-ordered on
 *    the first call on that stream outside graph capture and grown when
 *    needed; inside a capture each call allocates and frees its own), the
 *    backward's work-schedule tables (one per fixed-length shape, a few KB,
 *    made on first use outside graph capture) -- all released by
 *    ne_attn_release -- and, when a backward is given no workspace, a
 *    stream-ordered temporary it frees itself.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *    enqueued asynchronously on it; the call returns after the launch.
 *  - Calls may be captured into a CUDA graph once a call with the same
 *    rope_base and at least as many positions has run outside a capture:
 *    that first call builds the RoPE table with a synchronous copy, which a
 *    capture does not allow (inside one it returns NE_ERR_UNSUPPORTED and
 *    enqueues nothing).  Workspaces, temporaries and work lists that a
 *    captured call needs are allocated stream-ordered inside the graph.
 *  - Argument errors are detected on the host before anything is launched
 *    and return a nonzero ne_status.  Errors found on the device (a varlen
 *    sequence longer than max_seqlen, a pipeline wait that timed out) are
 *    recorded in a device status word read by ne_attn_get_device_status.
 *  - Nothing here calls exit, abort or traps the GPU.
 *  - Calls are thread-safe; the RoPE table cache is per device.
 */
#ifndef NE_ATTN_H
#define NE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int ne_status;
#define NE_OK 0
#define NE_ERR_INVALID_ARG 1 /* null pointer, non-positive size, bad cu_seqlens count */
#define NE_ERR_UNSUPPORTED 2 /* D != 64, or a device without sm_100-family tensor cores */
#define NE_ERR_MISALIGNED 3  /* a tensor pointer not 16-byte aligned */
#define NE_ERR_CUDA 4        /* a CUDA runtime / driver call failed */
#define NE_ERR_TIMEOUT 5     /* a device pipeline wait expired (reported by get_device_status) */
#define NE_ERR_OOM 6         /* allocation of a table or temporary failed */
#define NE_ERR_BAD_SEQLEN 7  /* a varlen sequence was longer than max_seqlen (device-detected) */
#define NE_ERR_TOO_LARGE 8   /* problem exceeds the fixed scratch of ne_attn_bwd_noalloc */

typedef uint16_t ne_bf16; /* raw bfloat16 bits */

/* Forward, fixed length.  q, k, v: [B, T, H, 64] bf16.  out: [B, T, H, 64]
 * bf16 (written).  lse: [B, H, T] fp32 (written), natural log.  scale is the
 * softmax scale, finite and > 0 (1/sqrt(64) = 0.125 for the usual choice);
 * rope_base is the RoPE theta base, finite and > 0 (10000 for the usual
 * choice).  B, H, T >= 1. */
ne_status ne_attn_fwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H, int T,
                      int D, float rope_base, float scale, ne_bf16* out, float* lse,
                      void* stream);

/* Same as ne_attn_fwd but writes O as fp32 (before any bf16 rounding). */
ne_status ne_attn_fwd_f32out(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H,
                             int T, int D, float rope_base, float scale, float* out, float* lse,
                             void* stream);

/* Bytes of workspace ne_attn_bwd / ne_attn_varlen_bwd need for n_tot tokens
 * (B*T for fixed length) and H heads: an fp32 dQ accumulator [n_tot, H, D],
 * the fp32 row terms D_m = dO_m . O_m [H, n_tot] and the rotated copies
 * q' = R(m) q and k' = R(n) k (bf16 [n_tot, H, D] each), every part 256-byte
 * aligned: 516 bytes per token and head at D = 64, plus alignment. */
size_t ne_attn_bwd_workspace_bytes(int n_tot, int H, int D);

/* Backward, fixed length.  q, k, v, out (the forward's O), dout: [B, T, H, 64]
 * bf16; lse: the forward's [B, H, T] fp32.  dq, dk, dv: [B, T, H, 64] bf16
 * (written), gradients w.r.t. the un-rotated q, k and v.  workspace: device
 * memory of at least ne_attn_bwd_workspace_bytes(B*T, H, D) bytes, 256-byte
 * aligned, or NULL to let the library allocate (and free) a temporary on
 * `stream` with cudaMallocAsync.  dq is accumulated with fp32 atomics, so its
 * last bits may differ from run to run; dk and dv are deterministic. */
ne_status ne_attn_bwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, const ne_bf16* out,
                      const ne_bf16* dout, const float* lse, int B, int H, int T, int D,
                      float rope_base, float scale, ne_bf16* dq, ne_bf16* dk, ne_bf16* dv,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Forward and backward on inputs already rotated: q' = R(m) q and k' = R(n) k
 * as ne_rmsnorm_qkv_rope writes them (the projection applied RoPE in its
 * epilogue), so nothing is rotated here.  Fixed length, arguments as in
 * ne_attn_fwd / ne_attn_bwd without rope_base; qr, kr replace q, k.  The
 * backward returns dqr, dkr -- the gradients with respect to q' and k' (the
 * rotated frame; dq = R(m)^T dqr, dk = R(n)^T dkr) -- and dv.  With q', k'
 * equal to the bf16 rotation ne_attn_fwd performs internally, O and LSE are
 * bitwise those of ne_attn_fwd on q, k. */
ne_status ne_attn_fwd_rotated(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v, int B,
                              int H, int T, int D, float scale, ne_bf16* out, float* lse,
                              void* stream);
ne_status ne_attn_bwd_rotated(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                              const ne_bf16* out, const ne_bf16* dout, const float* lse, int B,
                              int H, int T, int D, float scale, ne_bf16* dqr, ne_bf16* dkr,
                              ne_bf16* dv, void* workspace, size_t workspace_bytes, void* stream);

/* Training pair: the forward keeps the rotated operands for the backward, so
 * RoPE is applied to q and k once per training step instead of once in the
 * forward and again in the backward.  ne_attn_fwd_train takes the un-rotated
 * q, k, v (arguments as in ne_attn_fwd) and also writes qr = R(m) q and
 * kr = R(n) k (bf16 [B, T, H, 64], 16-byte aligned, caller-owned; the same
 * bf16 values ne_attn_fwd forms internally); O and LSE are bitwise those of
 * ne_attn_fwd.  ne_attn_bwd_train takes those qr, kr in place of q, k (q, k
 * themselves are not needed) with the other arguments as in ne_attn_bwd, and
 * returns dq, dk w.r.t. the UN-rotated q, k and dv -- bitwise what
 * ne_attn_bwd returns on q, k (dq up to its fp32 accumulation order).  The
 * workspace of ne_attn_bwd_workspace_bytes is enough (its q', k' part goes
 * unused).  qr, kr must be left as the forward wrote them; the gradients are
 * computed from them as they are. */
ne_status ne_attn_fwd_train(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H,
                            int T, int D, float rope_base, float scale, ne_bf16* out, float* lse,
                            ne_bf16* qr, ne_bf16* kr, void* stream);
ne_status ne_attn_bwd_train(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                            const ne_bf16* out, const ne_bf16* dout, const float* lse, int B,
                            int H, int T, int D, float rope_base, float scale, ne_bf16* dq,
                            ne_bf16* dk, ne_bf16* dv, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Forward, packed variable-length batch.  Sequence s occupies rows
 * cu_seqlens[s] .. cu_seqlens[s+1]-1 of q, k, v, out ([n_tot, H, 64] bf16);
 * cu_seqlens is DEVICE int32 [nseq + 1], nondecreasing, cu_seqlens[0] = 0,
 * cu_seqlens[nseq] = n_tot.  RoPE positions restart at 0 in every sequence and
 * attention never crosses a sequence boundary.  max_seqlen must be >= every
 * sequence length: a longer sequence (or one that cu_seqlens puts outside
 * [0, n_tot]) is reported as NE_ERR_BAD_SEQLEN by ne_attn_get_device_status
 * and skipped -- its rows of out and lse (and, in the backward, of dq, dk,
 * dv) are not written; the other sequences are computed as usual.  lse: [H, n_tot]
 * fp32.  With equal lengths T this computes exactly what ne_attn_fwd computes
 * on [B, T, H, 64] (LSE layout aside). */
ne_status ne_attn_varlen_fwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                             const int* cu_seqlens, int nseq, int n_tot, int max_seqlen, int H,
                             int D, float rope_base, float scale, ne_bf16* out, float* lse,
                             void* stream);

/* Same as ne_attn_varlen_fwd but writes O as fp32. */
ne_status ne_attn_varlen_fwd_f32out(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                                    const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                    int H, int D, float rope_base, float scale, float* out,
                                    float* lse, void* stream);

/* Backward of ne_attn_varlen_fwd; arguments as there and as in ne_attn_bwd.
 * workspace: ne_attn_bwd_workspace_bytes(n_tot, H, D) bytes or NULL. */
ne_status ne_attn_varlen_bwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                             const ne_bf16* out, const ne_bf16* dout, const float* lse,
                             const int* cu_seqlens, int nseq, int n_tot, int max_seqlen, int H,
                             int D, float rope_base, float scale, ne_bf16* dq, ne_bf16* dk,
                             ne_bf16* dv, void* workspace, size_t workspace_bytes, void* stream);

/* The training pair (see ne_attn_fwd_train) for packed variable-length
 * batches; qr, kr: [n_tot, H, 64] bf16, positions restarting at 0 in every
 * sequence; other arguments as in ne_attn_varlen_fwd / ne_attn_varlen_bwd. */
ne_status ne_attn_varlen_fwd_train(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                                   const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                   int H, int D, float rope_base, float scale, ne_bf16* out,
                                   float* lse, ne_bf16* qr, ne_bf16* kr, void* stream);
ne_status ne_attn_varlen_bwd_train(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                                   const ne_bf16* out, const ne_bf16* dout, const float* lse,
                                   const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                   int H, int D, float rope_base, float scale, ne_bf16* dq,
                                   ne_bf16* dk, ne_bf16* dv, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* Timing hook for profilers and benchmarks.  When set (non-NULL cudaEvent_t
 * handles created by the caller on the current device), every following
 * backward call (ne_attn_bwd, ne_attn_varlen_bwd and their _rotated / _train
 * forms) records ev_after_preprocess right after its preprocess kernel and
 * ev_after_main right after its main kernel, on the call's stream, so the
 * three backward kernels can be timed apart.  Pass NULL, NULL to turn it off.
 * Process-wide; not for concurrent callers. */
ne_status ne_attn_set_bwd_phase_events(void* ev_after_preprocess, void* ev_after_main);

/* The same for the forward: every following forward call that runs a
 * rotation pass before its attention kernel (the _train forms; ne_attn_fwd
 * from 2048 positions on) records ev_after_rotation between the two.  NULL
 * turns it off. */
ne_status ne_attn_set_fwd_phase_event(void* ev_after_rotation);

/* Backward that allocates no device memory at all, for callers that cannot
 * call cudaMalloc (or let a library do it for them): for example code running
 * under an allocator that must own every byte of device memory, a serving
 * process whose memory budget is fixed after start-up, or a plug-in that is
 * handed tensors but no allocator.  The paper pages have no counterpart; this
 * is a property of the library's interface, not of the method.
 *
 * Arguments are those of ne_attn_bwd without the workspace.  Instead of a
 * workspace and the library's RoPE-table cache, it uses one fixed scratch
 * array of NE_NOALLOC_SCRATCH_BYTES in the library's own device memory (a
 * static array that every GPU which loads the library holds until the process
 * exits).  Limits: B*T*H <= NE_NOALLOC_MAX_ROWS (token-head rows of the fp32
 * dQ accumulator) and T <= NE_NOALLOC_MAX_POSITIONS; beyond them the call
 * returns NE_ERR_TOO_LARGE before touching the device.
 *
 * The first call on a device looks up the array's device address (with that
 * device current).  The first call, and any call whose rope_base differs from
 * the previous call's, writes the RoPE table for that base into the array with
 * a copy from host memory enqueued on `stream`: it runs after the earlier work
 * of that stream (whose kernels may still read the old table) and before this
 * call's kernels.  Make the first call, and any call with a new rope_base,
 * outside a stream capture: inside one such a call returns NE_ERR_UNSUPPORTED
 * and enqueues nothing (a captured copy would read the host image when the
 * graph is replayed, after later calls may have rebuilt it).  Every call
 * shares the one array and leaves the last call's contents in it (the parts
 * that must start from zero are cleared on every call), so calls whose work
 * overlaps on the GPU -- on different streams, or on different host threads --
 * race and must be serialized by the caller.  Results equal those
 * of ne_attn_bwd (dq up to the order of its fp32 atomic adds). */
#define NE_NOALLOC_SCRATCH_BYTES (64u << 20)
#define NE_NOALLOC_MAX_POSITIONS 16384
#define NE_NOALLOC_MAX_ROWS 108000
ne_status ne_attn_bwd_noalloc(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                              const ne_bf16* out, const ne_bf16* dout, const float* lse, int B,
                              int H, int T, int D, float rope_base, float scale, ne_bf16* dq,
                              ne_bf16* dk, ne_bf16* dv, void* stream);

/* Decode attention over a KV cache: one new token per sequence attends to
 * every cached position up to and including its own (the generation path:
 * the interactive text generation of the NanoEuler Show HN page and of "Tiny
 * Hackable CUDA", section 7).
 *   q:        [B, H, 64] bf16, the new tokens' un-rotated queries;
 *   k_cache,
 *   v_cache:  [B, Tmax, H, 64] bf16, un-rotated keys and values; rows
 *             0..pos[b] of sequence b are attended (the new token's own key
 *             and value already written at row pos[b]);
 *   pos:      DEVICE int32 [B], the new token's position, 0 <= pos[b] < Tmax
 *             (an entry outside that range is reported as NE_ERR_BAD_SEQLEN
 *             by ne_attn_get_device_status and its outputs are zero / -inf);
 *   out:      [B, H, 64] bf16 (written);  lse: [B, H] fp32, natural log
 *             (written).
 * RoPE and the softmax are those of ne_attn_fwd: the query is rotated at
 * pos[b], each key at its own position (same fp32 rule and table), so a
 * decode at pos = T-1 reproduces row T-1 of the training forward.
 * workspace: ne_attn_decode_workspace_bytes(B, H, Tmax) bytes (split-K
 * partials), 16-byte aligned, or NULL for a stream-ordered temporary. */
size_t ne_attn_decode_workspace_bytes(int B, int H, int Tmax);
ne_status ne_attn_decode(const ne_bf16* q, const ne_bf16* k_cache, const ne_bf16* v_cache,
                         const int* pos, int B, int H, int Tmax, int D, float rope_base,
                         float scale, ne_bf16* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Decode over a cache of ROTATED keys: kr_cache holds k'_n = R(n) k_n (as
 * ne_attn_fwd_train's kr or ne_rmsnorm_qkv_rope's k write them) and qr is the
 * new token's q' = R(pos[b]) q, so nothing is rotated and no table is read;
 * the cache traffic is the K' and V rows alone.  Arguments, layouts, status
 * and workspace as in ne_attn_decode (no rope_base).  With the rotation of
 * ne_attn_decode (fp32 products, one bf16 rounding) applied to q and the
 * keys, the results equal ne_attn_decode's bit for bit. */
ne_status ne_attn_decode_rotated(const ne_bf16* qr, const ne_bf16* kr_cache,
                                 const ne_bf16* v_cache, const int* pos, int B, int H, int Tmax,
                                 int D, float scale, ne_bf16* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* The step before the attention in a transformer layer: RMSNorm, then the
 * QKV projection, with RoPE applied to q and k in the projection's epilogue
 * (NanoEuler Show HN page, paragraph 2: the CUDA engine has RMSNorm and RoPE
 * kernels and computes the layer's matrix products; "Tiny Hackable CUDA",
 * section 3: the projections are computed, then RoPE encodes relative
 * position).  For a fixed-length batch of B sequences of T tokens, C = H*64
 * with H a multiple of 4 (C a multiple of 256; NE_ERR_UNSUPPORTED otherwise),
 * D = 64:
 *   x_norm[n][c] = x[n][c] / sqrt(mean_c' x[n][c']^2 + eps) * g[c]   (rstd[n]
 *                  = 1 / sqrt(mean + eps) in fp32; the bf16 x_norm is what the
 *                  projection multiplies)
 *   [q | k | v]  = x_norm . w_qkv^T             (w_qkv [3C, C], no bias)
 *   q' = R(t) q, k' = R(t) k per head of 64, t = n mod T, in fp32 from the
 *   fp32 accumulators with the library's RoPE table for rope_base, then bf16.
 *   x:      [B*T, C] bf16 (input);  g: [C] bf16;  w_qkv: [3C, C] bf16
 *   x_norm: [B*T, C] bf16 (written);  rstd: [B*T] fp32 (written; may be NULL)
 *   q, k, v: [B, T, H, 64] bf16 (written) -- the attention's input layout.
 * All pointers are device memory owned by the caller, 16-byte aligned (rstd:
 * 4-byte).  eps finite and >= 0; rope_base finite and > 0.  Asynchronous on
 * `stream`; argument errors return before anything is launched. */
ne_status ne_rmsnorm_qkv_rope(const ne_bf16* x, const ne_bf16* g, const ne_bf16* w_qkv, int B,
                              int T, int H, int D, float eps, float rope_base, ne_bf16* x_norm,
                              float* rstd, ne_bf16* q, ne_bf16* k, ne_bf16* v, void* stream);

/* The step after the attention: the output projection with the residual
 * added in its epilogue ("Tiny Hackable CUDA", section 3: the attention is
 * wrapped in a residual connection):  y = residual + o . w_o^T  in fp32, then
 * bf16.  o (the attention output [N, H, 64] viewed as [N, C]), residual, y:
 * [N, C] bf16; w_o: [C, C] bf16 ([out, in], no bias); C a multiple of 256.
 * Conventions as above. */
ne_status ne_out_proj_residual(const ne_bf16* o, const ne_bf16* w_o, const ne_bf16* residual,
                               int N, int C, ne_bf16* y, void* stream);

/* Multi-token prediction (MTP) head with its softmax cross-entropy loss and
 * analytic gradients, the loss-side layer whose gradients the NanoEuler Show
 * HN page (paragraph 2) checks against double-precision finite differences
 * "including the RoPE and MTP layers".  K linear heads on the hidden states,
 * head j (0-based) predicting the token j + 1 positions ahead:
 *   logit_j(t) = h_t . W_j^T,   W_j = rows j*V .. j*V+V-1 of w
 *   loss = (1/n) sum over (t, j) with a target y_tj of (lse_j(t) - logit_j(t)[y_tj])
 *   dh = sum_j dlogit_j W_j,  dW_j = dlogit_j^T h,  dlogit_j(t) = (softmax - onehot(y_tj)) / n
 * (n: the number of (t, j) with a target; all zero when n = 0).
 * h: [M, C] bf16; w: [K*V, C] bf16 ([out, in], no bias); targets: [M, K]
 * int32 DEVICE array, each in [0, V) or -1 (no target there; a value outside
 * [-1, V) gives an unspecified loss for that row).  V must be 256 (a
 * byte-level vocabulary: one 256-wide GEMM tile per head), C a multiple of 8.
 * Writes loss [1] fp32 (the mean), row_loss [M, K] fp32 (each (t, j)'s term,
 * 0 where there is no target), dh [M, C] bf16 and dw [K*V, C] fp32.
 * workspace: ne_mtp_head_workspace_bytes(M, K, V) bytes of device memory,
 * 256-byte aligned (it holds dlogits [M, K*V] bf16), or NULL to let the
 * library allocate a stream-ordered temporary.  The loss sums are fp32
 * atomics, so the loss's last bits may differ from run to run.  Pointers
 * 16-byte aligned (targets, loss, row_loss 4-byte).  Asynchronous on
 * `stream`; argument errors return before anything is launched. */
size_t ne_mtp_head_workspace_bytes(int M, int K, int V);
ne_status ne_mtp_head(const ne_bf16* h, const ne_bf16* w, const int* targets, int M, int C, int K,
                      int V, float* loss, float* row_loss, ne_bf16* dh, float* dw,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Synchronize `stream`, then return and clear the device status word of the
 * current device: NE_OK, NE_ERR_TIMEOUT or NE_ERR_BAD_SEQLEN (or NE_ERR_CUDA
 * if the synchronization itself failed). */
ne_status ne_attn_get_device_status(void* stream);

/* Detail of the last device status read by ne_attn_get_device_status: the raw
 * device code (for a timeout, 0x100 + the id of the wait that expired). */
int ne_attn_last_device_code(void);

/* Human-readable name of a status code (static string). */
const char* ne_status_string(ne_status s);

/* Free the RoPE tables, the work-schedule tables and the per-stream
 * temporaries kept for every device.  Call only when no launch that may read them is still pending, and
 * before destroying a stream the library was given. */
void ne_attn_release(void);

#ifdef __cplusplus
}
#endif

#endif /* NE_ATTN_H */
