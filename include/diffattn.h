/*
 * diffattn.h -- C ABI of libdiffattn.so: causal differential-attention forward
 * on one GB300 (sm_103a).
 *
 * Operations (page titles as printed on the pages):
 *   diffattn_v1_fwd     "Differential Transformer V2", pseudo-code DiffAttnV1:
 *                       out = (1 - lam_init) * RMSNorm(softmax(Q1 K1^T / sqrt(d)) V
 *                                                     - lam * softmax(Q2 K2^T / sqrt(d)) V)
 *                       lam_init = 0.8 - 0.6 exp(-0.3 layer_index)
 *                       lam = exp(sum(lam_q1*lam_k1)) - exp(sum(lam_q2*lam_k2)) + lam_init
 *                       RMSNorm over the 2d channels of each (token, diff head),
 *                       eps = 1e-5, no weight ("How best to implement a
 *                       differential transformer?", first CausalSelfAttention, subln).
 *   diffattn_v2_fwd     same page, pseudo-code DiffAttnV2: one causal GQA attention
 *                       over Hq query heads, then out = attn[:, 0::2]
 *                       - sigmoid(lam) * attn[:, 1::2] (heads of one GQA group are
 *                       contiguous, so heads 2i and 2i+1 share kv head 2i/(Hq/Hkv)).
 *   diffattn_v2_decode  same page, the decoding remark after DiffAttnV2: the V2
 *                       operation for one new query token per sequence against an
 *                       L-row KV cache (the token attends all L rows).
 *   diffattn_v2_decode_varlen  the same with a cache length per sequence.
 *   diffattn_v1_fwd_train / diffattn_v2_fwd_train, diffattn_v1_bwd /
 *   diffattn_v2_bwd     the same forwards saving what their gradients need,
 *                       and the gradients of DiffAttnV1 (q1, q2, k1, k2, v and
 *                       the four lambda vectors) and DiffAttnV2 (q, k, v and
 *                       the lambda logits) for an upstream gradient dout; the
 *                       pages train these models, the backward is the chain
 *                       rule of the same definitions.
 *   diffattn_prologue   the neighbours before the attention: rotary embedding of
 *                       q and k, and V2's projected lambda logits.
 *   diffattn_v2_fwd_rope  diffattn_v2_fwd with the rotary embedding folded in:
 *                       q is rotated tile by tile inside the prefill kernel.
 *   diffattn_v1_fwd_host  the same DiffAttnV1 forward on host buffers, copies
 *                       overlapped with the forward (the end-to-end call).
 *   diffattn_paired_fwd modded-nanogpt pull request "New Record: Paired Head
 *                       Attention (-3.5s, -65 steps)": heads 2i and 2i+1
 *                       interleaved into one causal sequence of length 2T with
 *                       one softmax (a second workload on the prefill kernel).
 *   diffattn_v1_decode  DiffAttnV1 for one new query token per sequence against
 *                       cached k1, k2, v rows (all L, or a length per sequence);
 *                       the remark names V1 decoding as the case that needs
 *                       custom kernels, because its v head is 2d wide.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates and frees nothing and keeps no per-call state; it may be called
 *     concurrently on different streams.
 *   - The head dimension of every tensor is contiguous (stride 1).  Base pointers
 *     must be 16-byte aligned and every other stride, in bytes, a multiple of 16.
 *   - Softmax scale is fixed at 1/sqrt(d) (d = query/key head dim); causal mask
 *     j <= i with queries and keys aligned at position 0 (prefill).
 *   - dtype DA_BF16: bf16 q/k/v/out; softmax, lambda, norm and gate math in
 *     fp32; prefill runs on the tcgen05 tensor-core kernels, decode on the
 *     split-KV tensor-core kernel.  dtype DA_F32: fp32 everywhere on CUDA cores.
 *     Lambda vectors and lambda logits are fp32 for both dtypes.
 *   - `out` must not overlap any input.
 *   - Arguments are checked on the host before anything is enqueued; on any
 *     error the call returns a non-zero da_status and enqueues nothing.  A CUDA
 *     launch error is returned as DA_ERR_CUDA.  Work is asynchronous on
 *     `stream` (NULL = legacy default stream).
 *   - Device-side waits are bounded: a kernel that gives up waiting records a
 *     code in the error word of the stream it was launched on and returns;
 *     read it with diffattn_stream_error() (that stream only) or
 *     diffattn_device_error() (every stream of the device).  Each stream has
 *     a word of its own, so an error on one stream neither cuts short the
 *     kernels of another stream nor is reported to its caller.
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DA_OK = 0,
    DA_ERR_NULL_PTR = 1,          /* a required pointer is NULL                        */
    DA_ERR_BAD_SHAPE = 2,         /* a size is < 1 or too large                         */
    DA_ERR_UNSUPPORTED_DIM = 3,   /* head dim not supported for this dtype             */
    DA_ERR_BAD_GROUP = 4,         /* Hq % Hkv != 0, Hq/Hkv odd, or too large for dtype  */
    DA_ERR_MISALIGNED = 5,        /* pointer or stride breaks the 16-byte rule, or the  */
                                  /* head dimension is not contiguous                   */
    DA_ERR_WORKSPACE_TOO_SMALL = 6,
    DA_ERR_CUDA = 7,              /* CUDA runtime / driver error                        */
    DA_ERR_BAD_DTYPE = 8,
    DA_ERR_DEVICE_TIMEOUT = 9,    /* reported by diffattn_device_error()               */
    DA_ERR_SCRATCH_LIMIT = 10,    /* the call needs more scratch than the library's     */
                                  /* static buffer holds (diffattn_v2_decode_noalloc)  */
    DA_ERR_BAD_LENGTH = 11,       /* reported by diffattn_device_error(): a decode     */
                                  /* cache length was outside 1..L (it was clamped)    */
    DA_ERR_DEVICE_BOUNDS = 12     /* reported by the error-word calls of the debug     */
                                  /* build: an index failed its bounds check            */
} da_status;

typedef enum { DA_F32 = 0, DA_BF16 = 1 } da_dtype;

/* DIFF V1 causal forward.
 *   q1, q2, k1, k2 : (B, T, H, d) tensors given by base pointer + element strides
 *                    (q_sb, q_st, q_sh) shared by q1 and q2, (k_sb, k_st, k_sh)
 *                    shared by k1 and k2.  The nanoGPT-issue layout -- one
 *                    interleaved (B, T, 2H, d) tensor, q1 = heads 0::2,
 *                    q2 = heads 1::2 -- is q1 = q, q2 = q + d, q_sh = 2d,
 *                    q_st = 2Hd, q_sb = 2HdT.
 *   v              : (B, T, H, 2d), strides (v_sb, v_st, v_sh).
 *   lam_q1 .. lam_k2 : fp32 device vectors of length d.
 *   out            : (B, T, H, 2d), strides (o_sb, o_st, o_sh), dtype as inputs.
 *   layer_index    : >= 0, used as given (0-based) in lam_init.
 *   Supported: d in {32, 64, 128} for both dtypes (DA_BF16 at d = 32 runs the
 *   d = 64 tensor-core kernel on q / k boxes zero-filled past column 32).
 */
da_status diffattn_v1_fwd(const void *q1, const void *q2, const void *k1, const void *k2,
                          const void *v,
                          const float *lam_q1, const float *lam_k1,
                          const float *lam_q2, const float *lam_k2,
                          void *out,
                          int B, int T, int H, int d, int layer_index,
                          int64_t q_sb, int64_t q_st, int64_t q_sh,
                          int64_t k_sb, int64_t k_st, int64_t k_sh,
                          int64_t v_sb, int64_t v_st, int64_t v_sh,
                          int64_t o_sb, int64_t o_st, int64_t o_sh,
                          da_dtype dtype, cudaStream_t stream);

/* DIFF V1 forward from HOST buffers (the end-to-end call): the same operation
 * as diffattn_v1_fwd on host-resident inputs and output, with the copies of
 * the inputs in, the forward and the copy of the output back overlapped,
 * chunk by chunk of batch entries (up to 8 chunks), on two copy streams of
 * the library's own and `stream`.  The call is ordered on `stream`: work
 * queued on it afterwards sees the output in host memory.  Layouts (host,
 * contiguous; the nanoGPT issue's reshape(B, T, n_head, 2, d)):
 *   q, k   : (B, T, 2H, d)   branch 1 of head h in channel block 2h, branch 2 in 2h + 1
 *   v, out : (B, T, H, 2d)
 *   lam_q1, lam_k1, lam_q2, lam_k2 : d fp32 each, host
 *   workspace : device memory of diffattn_v1_fwd_host_workspace_size() bytes,
 *               256-byte aligned, owned by the caller; holds the device copies.
 * Host buffers should be pinned (page-locked) for the copies to run
 * asynchronously and overlap.  Concurrent calls on one device are correct;
 * they take the library's copy streams in turn.  Supported sizes as for
 * diffattn_v1_fwd; errors as there, DA_ERR_WORKSPACE_TOO_SMALL for a short
 * workspace.
 */
size_t diffattn_v1_fwd_host_workspace_size(int B, int T, int H, int d, da_dtype dtype);
da_status diffattn_v1_fwd_host(const void *q, const void *k, const void *v,
                               const float *lam_q1, const float *lam_k1,
                               const float *lam_q2, const float *lam_k2,
                               void *out, int B, int T, int H, int d, int layer_index,
                               void *workspace, size_t workspace_bytes,
                               da_dtype dtype, cudaStream_t stream);

/* DIFF V2 causal prefill (contiguous tensors).
 *   q   : (B, T, Hq, D)        Hq even; G = Hq / Hkv must be an even integer
 *   k, v: (B, T, Hkv, D)
 *   lam : (B, T, Hq/2) fp32 lambda logits, one per token and output head
 *   out : (B, T, Hq/2, D), dtype as inputs
 *   Supported: D in {64, 128} for both dtypes.
 */
da_status diffattn_v2_fwd(const void *q, const void *k, const void *v, const float *lam,
                          void *out, int B, int T, int Hq, int Hkv, int D,
                          da_dtype dtype, cudaStream_t stream);

/* DIFF V2 forward with the rotary embedding of q and k folded in: the result
 * of diffattn_prologue(q, k, ..., pos0, base) (rotate-half form, see there)
 * followed by diffattn_v2_fwd, bit for bit, with q left as it is.
 *   - k is rotated in place, as diffattn_prologue does (first launch);
 *   - q is read once per query tile by the prefill kernel and each tile is
 *     rotated in shared memory before its first product (cos and sin formed
 *     in registers with the same arithmetic as the prologue), so q is never
 *     written back; the tile is loaded once per query tile, so this repeats
 *     no work.
 * Arguments as for diffattn_v2_fwd, plus pos0, base: the position of token t
 * is pos0 + t, theta = pos * base^(-2i/D).  No workspace.
 * Supported: DA_BF16, D in {64, 128} (DA_F32 returns DA_ERR_UNSUPPORTED_DIM).
 * Errors as for the other entry points. */
da_status diffattn_v2_fwd_rope(const void *q, void *k, const void *v, const float *lam,
                               void *out, int B, int T, int Hq, int Hkv, int D,
                               int64_t pos0, float base, da_dtype dtype, cudaStream_t stream);

/* Paired Head Attention, causal (modded-nanogpt pull request "New Record:
 * Paired Head Attention (-3.5s, -65 steps)", section "Updates in PR"): the k,
 * q and v of heads 2i and 2i+1 are interleaved into one sequence of 2T
 * positions (position 2t + e is token t of head 2i + e), attended with one
 * causal softmax over it (scale 1/sqrt(D)), and the outputs are returned to
 * their (token, head) places.  So the query of token t of head 2i + e sees
 * both heads' keys of tokens < t, head 2i's key of token t, and for e = 1 its
 * own.  Contiguous tensors:
 *   q, k, v : (B, T, H, D)         H even, D in {64, 128}
 *   out     : (B, T, H, D)
 *   Supported: DA_BF16 only (tcgen05 one-pass kernel); DA_F32 returns
 *   DA_ERR_UNSUPPORTED_DIM.  Errors as for the other entry points.
 */
da_status diffattn_paired_fwd(const void *q, const void *k, const void *v, void *out,
                              int B, int T, int H, int D, da_dtype dtype, cudaStream_t stream);

/* Bytes of device scratch that diffattn_v2_decode needs for these sizes on the
 * current device (depends on its SM count).  Returns 0 for invalid sizes. */
size_t diffattn_v2_decode_workspace_size(int B, int L, int Hq, int Hkv, int D, da_dtype dtype);

/* DIFF V2 decode: one new query token per sequence against a KV cache.
 *   q           : (B, Hq, D)            G = Hq / Hkv even, G <= 8 for DA_BF16
 *   k_cache, v_cache : (B, L, Hkv, D)   rows 0..L-1 all valid (the new token's
 *                                        own K/V already written at row L-1)
 *   lam         : (B, Hq/2) fp32 lambda logits
 *   out         : (B, Hq/2, D)
 *   workspace   : device scratch of at least diffattn_v2_decode_workspace_size()
 *                 bytes, 256-byte aligned, owned by the caller; contents on entry
 *                 are ignored and on exit undefined.  Calls that share one
 *                 workspace must be ordered on the GPU (same stream).
 *   Supported: D in {64, 128}.
 */
da_status diffattn_v2_decode(const void *q, const void *k_cache, const void *v_cache,
                             const float *lam, void *out, void *workspace,
                             size_t workspace_bytes, int B, int L, int Hq, int Hkv, int D,
                             da_dtype dtype, cudaStream_t stream);

/* DIFF V2 decode that allocates nothing and takes no workspace.
 *   The paper has no counterpart: this exists for callers that are not
 *   allowed to allocate device memory themselves -- for example a host
 *   framework that owns every byte of device memory through its own pool and
 *   hands this library only inputs and outputs, or a decode loop that cannot
 *   afford the device-wide synchronisation a cudaMalloc may cause.
 *   Same operation, arguments, layouts and limits as diffattn_v2_decode, minus
 *   the workspace.  The split-KV partials live instead in one static device
 *   buffer of 8 MiB inside the library; every GPU that loads the library
 *   holds that buffer until the process exits.
 *   - Sizes whose partials need more than 8 MiB (see
 *     diffattn_v2_decode_workspace_size) return DA_ERR_SCRATCH_LIMIT with
 *     nothing enqueued; the workspace entry point has no such limit.
 *   - The first call on each device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the one buffer and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (each call writes every partial it
 *     reads back), but calls that overlap on the GPU -- on different streams,
 *     or from different host threads -- race on it: order them.
 *   - dtype DA_F32 needs no scratch and runs the same fp32 kernel as
 *     diffattn_v2_decode.
 */
da_status diffattn_v2_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                     const float *lam, void *out, int B, int L, int Hq, int Hkv,
                                     int D, da_dtype dtype, cudaStream_t stream);

/* DIFF V2 decode with a cache length per sequence: sequence b's new token
 * attends cache rows 0 .. cache_lens[b]-1 (its own K/V already written at row
 * cache_lens[b]-1); rows at and past that length are never used, whatever they
 * hold.  The split-KV work is rebalanced over the SMs by the actual lengths.
 *   cache_lens : DEVICE int32 array of B lengths, each in 1..L (L = rows
 *                allocated per sequence, the cache's row stride).  A length
 *                outside that range is clamped into it and recorded in the
 *                device error word (diffattn_device_error -> DA_ERR_BAD_LENGTH).
 *   workspace  : as diffattn_v2_decode (the same size function covers both).
 *   Every other argument, layout and limit as diffattn_v2_decode.  dtype
 *   DA_F32 runs the fp32 kernel, which takes no workspace.
 */
da_status diffattn_v2_decode_varlen(const void *q, const void *k_cache, const void *v_cache,
                                    const float *lam, const int32_t *cache_lens, void *out,
                                    void *workspace, size_t workspace_bytes, int B, int L, int Hq,
                                    int Hkv, int D, da_dtype dtype, cudaStream_t stream);

/* Bytes of device scratch that diffattn_v1_decode needs (either length mode)
 * on the current device.  Returns 0 for invalid sizes or dtype DA_F32. */
size_t diffattn_v1_decode_workspace_size(int B, int L, int H, int d, da_dtype dtype);

/* DIFF V1 decode: the DiffAttnV1 operation for one new query token per
 * sequence against a KV cache.
 *   q1, q2          : (B, H, d) contiguous
 *   k1_cache, k2_cache : (B, L, H, d) contiguous
 *   v_cache         : (B, L, H, 2d) contiguous
 *   lam_q1 .. lam_k2 : (d) fp32 lambda vectors; layer_index gives lam_init
 *   cache_lens      : NULL (every sequence attends all L rows) or a DEVICE
 *                     int32 array of B lengths in 1..L, as in
 *                     diffattn_v2_decode_varlen
 *   out             : (B, H, 2d) = (B, C), dtype as inputs
 *   workspace       : DA_BF16 only; at least diffattn_v1_decode_workspace_size()
 *                     bytes, 256-byte aligned, as in diffattn_v2_decode
 *   Supported: d in {32, 64, 128} for both dtypes (DA_BF16 at d = 32 runs the
 *   d = 64 kernels on k / v boxes zero-filled past d / 2d).
 */
da_status diffattn_v1_decode(const void *q1, const void *q2, const void *k1_cache,
                             const void *k2_cache, const void *v_cache, const float *lam_q1,
                             const float *lam_k1, const float *lam_q2, const float *lam_k2,
                             const int32_t *cache_lens, void *out, void *workspace,
                             size_t workspace_bytes, int B, int L, int H, int d, int layer_index,
                             da_dtype dtype, cudaStream_t stream);

/* ---- training: forward with saved tensors, and the backward -----------
 * Supported: DA_BF16 on the tensor cores: V1 d in {32, 64, 128} (d = 32 on
 * the d = 64 kernels with zero-filled q / k boxes; d = 128, dv = 256, with a
 * training forward of two launches and a backward of five: a row pass, the
 * lambda reduction, dK per branch, dV, dQ per branch), V2 D in {64, 128};
 * DA_F32 on CUDA cores: V1 d in {32, 64, 128}, V2 D in {64, 128}
 * (every tensor, dout and the gradients fp32).  Other combinations return
 * DA_ERR_UNSUPPORTED_DIM.  The size functions take the same dtype.
 *
 * `saved` (DEVICE, caller-owned, at least *_train_saved_size() bytes,
 * 16-byte aligned) receives what the backward needs -- V2: each branch's
 * normalised attention output a_b (bf16); V1: x = a1 - lam a2, the RMSNorm
 * input, and a2 (fp32) -- and each branch's row log-sum-exp (fp32); its
 * contents are private to this library: pass it unchanged to the matching
 * *_bwd call.  The forward output
 * is the same as the plain forward's.  `workspace` (DEVICE, at least
 * *_bwd_workspace_size() bytes) is scratch for the backward; contents on
 * entry are ignored.  Gradient outputs must not overlap any input; they are
 * fully overwritten (not accumulated into).  Sizes functions return 0 for
 * unsupported sizes. */
size_t diffattn_v1_train_saved_size(int B, int T, int H, int d, da_dtype dtype);
size_t diffattn_v1_bwd_workspace_size(int B, int T, int H, int d, da_dtype dtype);
size_t diffattn_v2_train_saved_size(int B, int T, int Hq, int Hkv, int D, da_dtype dtype);
size_t diffattn_v2_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D, da_dtype dtype);

/* Byte offset inside `saved` of each branch's row log-sum-exp: fp32
 * (2, B, H, T) for V1 (branch 1, then branch 2) and (2, B, Hq/2, T) for V2
 * (the even heads, then the odd heads), lse = log sum_j exp(q . k_j / sqrt(d))
 * over the causal keys j <= t, in log2 units (times log2(e)) for DA_BF16 and
 * natural units for DA_F32.  Arguments as the size functions; 0 for
 * unsupported sizes.  The rest of `saved` stays private. */
size_t diffattn_v1_train_saved_lse_offset(int B, int T, int H, int d, da_dtype dtype);
size_t diffattn_v2_train_saved_lse_offset(int B, int T, int Hq, int Hkv, int D, da_dtype dtype);

/* DIFF V1 training forward: arguments, layouts and strides as
 * diffattn_v1_fwd, plus `saved`. */
da_status diffattn_v1_fwd_train(const void *q1, const void *q2, const void *k1, const void *k2,
                                const void *v, const float *lam_q1, const float *lam_k1,
                                const float *lam_q2, const float *lam_k2, void *out, void *saved,
                                size_t saved_bytes, int B, int T, int H, int d, int layer_index,
                                int64_t q_sb, int64_t q_st, int64_t q_sh, int64_t k_sb,
                                int64_t k_st, int64_t k_sh, int64_t v_sb, int64_t v_st,
                                int64_t v_sh, int64_t o_sb, int64_t o_st, int64_t o_sh,
                                da_dtype dtype, cudaStream_t stream);

/* DIFF V1 backward.  Inputs as the training forward that filled `saved`;
 * dout has the output's strides (o_*).  dq1, dq2 take q's strides, dk1, dk2
 * k's, dv v's (bf16).  dlam_q1 .. dlam_k2: fp32 (d) gradients of the lambda
 * vectors. */
da_status diffattn_v1_bwd(const void *q1, const void *q2, const void *k1, const void *k2,
                          const void *v, const float *lam_q1, const float *lam_k1,
                          const float *lam_q2, const float *lam_k2, const void *dout,
                          const void *saved, size_t saved_bytes, void *dq1, void *dq2, void *dk1,
                          void *dk2, void *dv, float *dlam_q1, float *dlam_k1, float *dlam_q2,
                          float *dlam_k2, void *workspace, size_t workspace_bytes, int B, int T,
                          int H, int d, int layer_index, int64_t q_sb, int64_t q_st, int64_t q_sh,
                          int64_t k_sb, int64_t k_st, int64_t k_sh, int64_t v_sb, int64_t v_st,
                          int64_t v_sh, int64_t o_sb, int64_t o_st, int64_t o_sh, da_dtype dtype,
                          cudaStream_t stream);

/* DIFF V2 training forward: as diffattn_v2_fwd, plus `saved`. */
da_status diffattn_v2_fwd_train(const void *q, const void *k, const void *v, const float *lam,
                                void *out, void *saved, size_t saved_bytes, int B, int T, int Hq,
                                int Hkv, int D, da_dtype dtype, cudaStream_t stream);

/* DIFF V2 backward.  dout (B, T, Hq/2, D) contiguous; dq (B, T, Hq, D), dk, dv
 * (B, T, Hkv, D) bf16 contiguous; dlam (B, T, Hq/2) fp32 gradient of the
 * lambda logits. */
da_status diffattn_v2_bwd(const void *q, const void *k, const void *v, const float *lam,
                          const void *dout, const void *saved, size_t saved_bytes, void *dq,
                          void *dk, void *dv, float *dlam, void *workspace, size_t workspace_bytes,
                          int B, int T, int Hq, int Hkv, int D, da_dtype dtype, cudaStream_t stream);

/* Prologue of the attention call, in one pass over device memory:
 *   - rotary position embedding of q (B, T, Hq, D) and k (B, T, Hk, D) in
 *     place (contiguous, dtype as given), the rotate-half form: for the
 *     token at position pos0 + t and i < D/2, theta = pos * base^(-2i/D),
 *     (x_i, x_{i+D/2}) -> (x_i cos - x_{i+D/2} sin, x_{i+D/2} cos + x_i sin)
 *     ("How best to implement a differential transformer?", the issue's
 *     RotaryEmbedding / apply_rotary_pos_emb applied to q and k before the
 *     attention; base 10000 there).  Hq or Hk may be 0 (that tensor is
 *     skipped).  For DIFF V1 pass the interleaved (B, T, 2H, d) q and k.
 *   - if x != NULL, DIFF V2's projected lambda ("Differential Transformer
 *     V2": a projected lambda for each token and head): lam (B, T, P) fp32
 *     = x (B, T, C) @ w_lam (C, P), x and w_lam in dtype, fp32 sums.
 * Supported: D in {32, 64, 128}; C a multiple of 64; P a multiple of 8 in
 * 8..64.  Pointers 16-byte aligned. */
da_status diffattn_prologue(void *q, void *k, int B, int T, int Hq, int Hk, int D, int64_t pos0,
                            float base, const void *x, const void *w_lam, float *lam, int C, int P,
                            da_dtype dtype, cudaStream_t stream);

/* Static string for a status code (never NULL). */
const char *diffattn_status_string(da_status s);

/* Error words.  The library keeps one 32-bit error word per stream that has
 * called it (per device, handed out on a stream's first call; past 256
 * streams on one device, further streams share words).  A kernel that gives
 * up a bounded wait, or that meets a decode cache length outside 1..L, sets a
 * bit in the word of the stream it runs on; the other kernels of that stream
 * then give up their waits at once, those of other streams do not notice.
 *
 * diffattn_stream_error synchronises `stream` only, then reads and clears
 * its word.  diffattn_device_error synchronises the whole current device,
 * then reads and clears every stream's word and returns their OR.
 * *code (may be NULL) receives the raw word (0 = no error).  Both return
 * DA_OK if the word was 0, DA_ERR_DEVICE_TIMEOUT if a kernel recorded a
 * give-up, else DA_ERR_DEVICE_BOUNDS if a bounds check of the debug build
 * failed, else DA_ERR_BAD_LENGTH if the record is a decode cache length
 * outside 1..L; DA_ERR_CUDA if the synchronisation or the read failed. */
da_status diffattn_stream_error(uint32_t *code, cudaStream_t stream);
da_status diffattn_device_error(uint32_t *code);

/* Failure-path self-test: one warp waits on an mbarrier phase that nothing
 * completes.  Its bounded wait gives up after the library's limit (2 s of
 * global time), records the timeout bit in the error word of `stream` and
 * returns; the call then reads and clears that word (the raw value into
 * *code, which may be NULL), synchronising `stream` only.  Returns DA_OK when the wait gave up and
 * recorded the bit -- the context stays usable for the next call -- and
 * DA_ERR_CUDA if a launch or copy failed or the wait did not give up.  Any
 * error recorded on `stream` before the call is cleared first.  Takes about
 * 2 s.  Run one self-test at a time per device. */
da_status diffattn_selftest_wait_limit(uint32_t *code, cudaStream_t stream);

/* Debug build.  libdiffattn_debug.so is the same library compiled with
 * DA_DEBUG_CHECKS: every kernel tests the indices through which it writes
 * memory (output rows, channels, heads and batch entries against the call's
 * sizes; partial slots against the workspace; shared-memory staging offsets
 * against the tile; TMEM columns against the allocation) before the access.
 * A failed test skips the access and records a bit in the stream's error
 * word, which diffattn_stream_error / diffattn_device_error report as
 * DA_ERR_DEVICE_BOUNDS; nothing traps.  (No tool of the image checks device
 * memory accesses on this system, so this build stands in for one.)
 *
 * diffattn_debug_checks returns 1 in the debug build and 0 in the release
 * build.  diffattn_selftest_bounds launches one warp that tests an index one
 * past the end of a 32-entry buffer through the same check (the write is
 * skipped), then reads and clears the error word of `stream` (raw value into
 * *code, may be NULL).  Debug build: DA_OK when the bit was recorded.
 * Release build: DA_OK with a zero word (the check is compiled out).
 * DA_ERR_CUDA if a launch or copy failed or the result is not the one of
 * the build. */
int diffattn_debug_checks(void);
da_status diffattn_selftest_bounds(uint32_t *code, cudaStream_t stream);

/* Number of kernel launches the last successful call on this host thread
 * enqueued (launch accounting for benchmarks). */
int diffattn_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DIFFATTN_H */
