// da_internal.h -- parameter blocks and launchers shared between the C-ABI
// host code (da_api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace da {

// Bits of the device error word.
enum : uint32_t {
    kErrWaitTimeout = 1u,      // a bounded mbarrier wait gave up
    kErrAborted = 2u,          // a kernel saw an earlier error and returned early
    kErrBadLength = 4u,        // a decode cache length outside 1 .. L (clamped)
    kErrBounds = 8u,           // debug builds: an index failed its bounds check (access skipped)
    kErrFatal = kErrWaitTimeout | kErrAborted,   // bits after which kernels stop waiting
};

// Built with the debug bounds checks (-DDA_DEBUG_CHECKS, libdiffattn_debug.so).
#ifdef DA_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Runs set() once per device and remembers success in one bit of *done.
// Kernel attributes such as the dynamic shared-memory opt-in belong to the
// current device's context, so a launcher that sets them must do so on every
// device it launches on; the bitmask is read and updated atomically so that
// host threads may launch concurrently (set() may then run more than once on
// a device, which is harmless).  Devices past 63 run set() on every call.
template <typename F>
inline cudaError_t once_on_device(unsigned long long *done, int dev, F &&set) {
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (__atomic_load_n(done, __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    const cudaError_t e = set();
    if (e == cudaSuccess && bit) __atomic_fetch_or(done, bit, __ATOMIC_RELEASE);
    return e;
}
template <typename F>
inline cudaError_t once_per_device(unsigned long long *done, F &&set) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return once_on_device(done, dev, static_cast<F &&>(set));
}

// ---------------------------------------------------------------- SIMT fp32
// One warp per output row.  mode 1 = DIFF V1, mode 2 = DIFF V2 (prefill or
// decode).  Query t attends keys 0 .. t + (Lk - Tq): Lk == Tq is the causal
// prefill, Tq == 1 is decode against Lk cached rows.
struct SimtParams {
    const float *q1, *q2, *k1, *k2, *v;
    int64_t q_sb, q_st, q_sh;
    int64_t k_sb, k_st, k_sh;
    int64_t v_sb, v_st, v_sh;
    int64_t o_sb, o_st, o_sh;
    float *out;
    const float *lam;              // V2 logits at lam[b*lam_sb + t*lam_st + i]
    int64_t lam_sb, lam_st;
    const float *lq1, *lk1, *lq2, *lk2;
    int layer_index;
    int B, Tq, Lk, H, G, mode;
    const int *lens;               // decode (Tq == 1): keys per sequence, or NULL
    uint32_t *err;
    // training forward (prefill) only, else NULL: per row (B, T, H, DV)
    // contiguous fp32, V1 x = a1 - lam a2 and a2, V2 a_e and a_o; and each
    // branch's log-sum-exp of the scaled scores in natural units,
    // lse_b = m + log(l), P = exp(s * scale - lse_b) ((2, B, H, T) fp32)
    float *sa1, *sa2, *slse;
};
cudaError_t launch_simt(const SimtParams &p, int dqk, int dv, cudaStream_t s);

// ------------------------------------------------------- tcgen05 prefill
// V1: H diff heads; tensor maps over q1, q2, k1, k2, v.
// V2: H = Hq/2 pairs; tq1 == tq2 over q, tk1 == tk2 over k, G = Hq/Hkv.
struct PrefillParams {
    void *out;
    int64_t o_sb, o_st, o_sh;      // elements
    const float *lam;              // V2 logits (B, T, H) contiguous
    const float *lq1, *lk1, *lq2, *lk2;
    int dlam;                      // V1: length d of the lambda vectors
    int layer_index;
    int B, T, H, G;
    float scale_log2;              // log2(e) / sqrt(dqk)
    uint32_t *err;
    int num_sms;                   // SMs of the device (the persistent grid)
    // training forward only ((B, T, H, DV) contiguous; NULL for the plain
    // forward): V1 saves x = a1 - lam a2 (the RMSNorm input) and a2 in fp32,
    // V2 saves a_e and a_o in bf16 (a_b = O_b / l_b); both save each branch's
    // log-sum-exp in log2 units, lse_b = m + log2(l), so that
    // P = 2^(s * scale_log2 - lse_b) (fp32, (2, B, H, T))
    void *sa1, *sa2;
    float *slse;
    int64_t rope_pos0;             // V2 with rotary embedding (q rotated in shared memory as each
    double rope_base;              // Q tile lands): position of token t = rope_pos0 + t, base
};
struct PrefillMaps {
    CUtensorMap q1, q2, k1, k2, v;
    CUtensorMap out;   // one-pass kernel: output tile stores (box 64 x 1 x 128 x 1)
};
// dqk/dv in {32/64, 64/128 (V1), 128/256 (V1 two-pass), 64/64, 128/128 (V2)}
cudaError_t launch_prefill(const PrefillMaps &m, const PrefillParams &p, int dqk, int dv, bool v2,
                           cudaStream_t s);
// The same kernel with the training epilogue (p.sa1, p.sa2, p.slse written).
// Paired Head Attention forward on the one-pass kernel (bf16, D in {64, 128}):
// m.q1 = m.q2 = a 4-D map of q, m.k1 = m.k2 and m.v 5-D interleaved maps of
// k and v (encode_map_pairs); p.H = pairs, p.G = 2, p.out / p.o_* the output.
// V2 prefill whose Q tiles are rotated (rotary embedding, table p.rope_cs) in
// shared memory before their first product; D in {64, 128}, bf16.
cudaError_t launch_prefill_v2_rope(const PrefillMaps &m, const PrefillParams &p, int d, cudaStream_t s);
bool paired_supported(int d);
cudaError_t launch_paired(const PrefillMaps &m, const PrefillParams &p, int d, cudaStream_t s);
// 5-D map over a contiguous (B, T, H, D) bf16 tensor read as {D, 2, H/2, T, B}
// with boxes {64, 2, 1, 64, 1}: 64 tokens of both heads of one pair, in the
// interleaved order (token, head) -- 128 rows of 128 bytes, 128-byte swizzle.
bool encode_map_pairs(CUtensorMap *m, const void *base, uint64_t D, uint64_t H, uint64_t T, uint64_t B);
// The count diffattn_last_launch_count() reports for this thread's last call.
void set_last_launches(int n);
cudaError_t launch_prefill_train(const PrefillMaps &m, const PrefillParams &p, int dqk, int dv, bool v2,
                                 cudaStream_t s);
bool prefill_supported(int dqk, int dv, bool v2);
// DIFF V1 in two passes over the keys (row statistics, then one combined PV);
// dqk in {64, 128}, dv = 2 dqk.  The V tensor map's box has
// prefill_v1_twopass_v_rows(dqk) rows (the Q/K maps 128).
cudaError_t launch_prefill_v1_twopass(const PrefillMaps &m, const PrefillParams &p, int dqk, cudaStream_t s);
// Its training forward at dqk = 128 (two launches): the output, x = a1 - lam a2
// (p.sa1, fp32), a2 (p.sa2, fp32) and each branch's log-sum-exp (p.slse, log2
// units), the layout the V1 backward reads.
cudaError_t launch_prefill_v1_twopass_train(const PrefillMaps &m, const PrefillParams &p, cudaStream_t s);
int prefill_v1_twopass_v_rows(int dqk);

// -------------------------------------------------------------- backward
// Gradients of the V1 / V2 prefill (k_backward.cu).  H = diff heads (V1) or
// pairs (V2); row vectors are (2, B, H, T) fp32 (branch-major).
struct BwdParams {
    __nv_bfloat16 *dq1, *dq2, *dk1, *dk2, *dv;   // V2: dq1 == dq2 (head 2i / 2i+1), dk1 == dk2
    int64_t q_sb, q_st, q_sh;                    // element strides of q1/q2 and dq1/dq2
    int64_t k_sb, k_st, k_sh;                    // of k1/k2 and dk1/dk2
    int64_t v_sb, v_st, v_sh;                    // of v and dv
    const float *lse;                            // forward log-sum-exp, log2 units
    const float *dd;                             // D_b = g_b . a_b
    const float *cv;                             // c (B, H, T): V1 -lam, V2 -sigmoid(lam[t])
    int B, T, H, G, Hkv;
    int dqk_store;                               // channels of dq / dk stored (the real d; the
                                                 // kernels may run on zero-padded q / k boxes)
    float scale_log2, scale;                     // log2(e) / sqrt(dqk), 1 / sqrt(dqk)
    uint32_t *err;
};
struct BwdPreParams {
    const void *sa1, *sa2;                       // saved: V1 x, a2 (fp32); V2 a_e, a_o (bf16)
    const __nv_bfloat16 *dout;                   // upstream gradient, the output's layout
    int64_t o_sb, o_st, o_sh;
    const float *lam;                            // V2 logits (B, T, H)
    int layer_index;                             // V1
    const float *lq1, *lk1, *lq2, *lk2;          // V1 lambda vectors (d)
    float *dlq1, *dlk1, *dlq2, *dlk2;            // V1 outputs (d)
    float *dlam;                                 // V2 output (B, T, H)
    float *dlam_rows;                            // V1 scratch: shares of dL/dlam (n_shares of them)
    int64_t n_shares;                            // set by the launchers: one per row-pass block (tensor-core
                                                 // path) or one per row (fp32 path)
    __nv_bfloat16 *g;                            // V1 g_1 = dx, (B, T, H, DV) contiguous
    float *dd, *cv;                              // outputs D (2, B, H, T); c (B, H, T)
    int B, T, H, d;
    uint32_t *err;                               // error word (debug bounds checks)
};
struct BwdMaps {
    CUtensorMap q1r, q2r, gr, k1c, k2c, vc;      // dQ kernel: 128-row Q / G boxes, 64-row K / V boxes
    CUtensorMap k1r, k2r, vr, q1c, q2c, gc;      // dK dV kernel: 128-row K / V boxes, 64-row Q / G boxes
};
bool backward_supported(int dqk, int dv, bool v2);
// One warp waits on an mbarrier phase nothing completes (the bounded-wait
// failure path); *gave_up is true once the wait gave up as designed.
cudaError_t run_wait_selftest(uint32_t *err, bool *gave_up, cudaStream_t s);
// One warp tests index 32 of a 32-entry buffer through DA_CHECK; *wrote says
// whether any write reached the buffer (it must not, in either build).
cudaError_t run_bounds_selftest(uint32_t *err, bool *wrote, cudaStream_t s);
// dL/dlam summed from the per-row shares in pp.dlam_rows, then the four
// lambda-vector gradients (one CTA; used by the bf16 and the fp32 backward).
cudaError_t launch_bwd_lambda(const BwdPreParams &pp, cudaStream_t s);

// fp32 backward on CUDA cores (k_simt_bwd.cu).  mode 1 = V1 (H diff heads),
// mode 2 = V2 (H = pairs, query heads 2h / 2h+1, kv head 2h / G).
struct SimtBwdParams {
    const float *q1, *q2, *k1, *k2, *v;          // V2: q1 == q2, k1 == k2
    int64_t q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh;   // elements
    const float *dout;
    int64_t o_sb, o_st, o_sh;
    const float *sa1, *sa2, *slse;               // saved by the fp32 training forward
    const float *lam;                            // V2 logits (B, T, H)
    const float *lq1, *lk1, *lq2, *lk2;          // V1
    int layer_index;
    float *dq1, *dq2, *dk1, *dk2, *dv;           // outputs with the inputs' strides (V2: dq1 == dq2, dk1 == dk2)
    float *dlam;                                 // V2 (B, T, H)
    float *dlq1, *dlk1, *dlq2, *dlk2;            // V1 lambda-vector gradients (d)
    const float *g;                              // upstream gradient of branch 1: V1 workspace, V2 dout
    int64_t g_sb, g_st, g_sh;
    float *gw, *dd, *cv, *dlam_rows;             // workspace: V1 g (B,T,H,DV); D (2,B,H,T); c (B,H,T); V1 rows
    int B, T, H, G, Hkv, mode;
    uint32_t *err;
};
cudaError_t launch_simt_backward(const SimtBwdParams &p, int dqk, int dv, cudaStream_t s);
cudaError_t launch_backward(const BwdMaps &m, const BwdParams &p, const BwdPreParams &pp, int dqk, int dv, bool v2,
                            cudaStream_t s);

// -------------------------------------------------------------- prologue
// Rotary embedding of q, k in place and the V2 projected lambda (k_prologue.cu).
struct PrologueParams {
    void *q, *k;                   // (B, T, Hq, D), (B, T, Hk, D) contiguous; either may be NULL
    int Hq, Hk, D;
    const void *x, *w;             // (B, T, C), (C, P) contiguous; x NULL = no projection
    float *lam;                    // (B, T, P) fp32
    int C, P;
    int B, T;
    int64_t pos0;                  // position of token t is pos0 + t
    double base;
    uint32_t *err;                 // error word (debug bounds checks)
};
bool prologue_supported(int D, int C, int P);
cudaError_t launch_prologue(const PrologueParams &p, bool bf16, cudaStream_t s);

// --------------------------------------------------------------- decode
// One kernel family serves three decodes:
//   V2      : kv head g of sequence b feeds the G query heads g*G .. g*G+G-1;
//   V1      : "kv head" = diff head h; the two score columns are q1 . k1 and
//             q2 . k2 (K tile = k1 channels, then k2 channels), V is 2d wide;
// and either with every sequence attending all L cached rows (lens == NULL)
// or sequence b attending rows 0 .. lens[b]-1.
struct DecodeParams {
    const __nv_bfloat16 *q;        // V2: (B, Hq, D).  V1: q1 (B, H, d)
    const __nv_bfloat16 *q2;       // V1: q2 (B, H, d)
    const float *lam;              // V2 logits (B, Hq/2)
    const float *lq1, *lk1, *lq2, *lk2;   // V1 lambda vectors (d)
    int layer_index;               // V1
    __nv_bfloat16 *out;            // V2: (B, Hq/2, D).  V1: (B, H, 2d)
    float *ws;                     // partial slots: B * Hkv + grid - 1
    const int *lens;               // per-sequence rows (B), or NULL for all L
    int64_t *cum;                  // lens != NULL: units before sequence b (B + 1)
    int B, L, Hq, Hkv, G, D;       // V1: Hq = Hkv = H, G = 2, D = 2d (128 for d = 32)
    int dq, dv;                    // V1: the real head dims d and 2d (D = 2d, or 128 for d = 32,
                                   // which runs on k / v boxes zero-filled past d / 2d)
    int grid;                      // CTAs of the split kernel
    int64_t units;                 // lens == NULL: B * Hkv * spb
    int spb;                       // 64-key units per (b, kv head) at L rows
    float scale_log2;              // log2(e) / sqrt(q/k head dim)
    uint32_t *err;
};
struct DecodeMaps {
    CUtensorMap k, k2, v;          // k2: V1 only (k1 in k)
};
// Sizes the decode plan on the current device.  Returns false on bad sizes.
// ws_bytes covers the partial slots and, for per-sequence lengths, the unit
// prefix (which sits first, cum_bytes long).
bool decode_plan(int B, int L, int Hkv, int D, int num_sms, bool varlen, int *grid, int64_t *units,
                 int *spb, size_t *cum_bytes, size_t *ws_bytes);
cudaError_t launch_decode(const DecodeMaps &m, const DecodeParams &p, bool v1, cudaStream_t s);
constexpr int kDecodeKeysPerUnit = 64;

// Tensor-map helper (da_api.cu): 4-D bf16 map over (inner, d1, d2, d3) with
// element strides s1, s2, s3, box (64, 1, box_rows, 1), 128-byte swizzle.
// l2_promo_bytes (128 or 256) is the L2 fetch granularity: a map whose rows
// are 128 bytes apart from the next row it reads should not promote to 256,
// or every row pulls in 128 bytes it does not use.
bool encode_map_4d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t d1, uint64_t d2,
                   uint64_t d3, int64_t s1, int64_t s2, int64_t s3, uint32_t box_rows,
                   int l2_promo_bytes = 256);

}  // namespace da
