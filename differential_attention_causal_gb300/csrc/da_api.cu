// da_api.cu -- the C ABI of libdiffattn.so (declared in include/diffattn.h).
//
// Host side only: argument checks (nothing is enqueued when one fails), TMA
// tensor-map encoding, the device error word, and the launch of the kernels
// in k_prefill.cu (tcgen05 prefill), k_decode.cu (split-KV decode) and
// k_simt.cu (fp32).  The library allocates no memory.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <cudaTypedefs.h>

#include "da_internal.h"
#include "diffattn.h"

namespace da {

// Sticky device error words, set by bounded waits that give up.  Each stream
// that calls the library gets a word of its own (slots handed out in order of
// first use per device), so that an error on one stream neither stops the
// kernels of another stream (a wait gives up at once when its word already
// holds a fatal bit) nor shows up when another stream's word is read.  Past
// kErrSlots streams on one device, later streams share words by hash.
constexpr int kErrSlots = 256;
__device__ uint32_t g_err_words[kErrSlots];

namespace {

thread_local int t_last_launches = 0;

struct DeviceState {
    uint32_t *words = nullptr;   // device address of this device's g_err_words
    int num_sms = 0;
    int used = 0;                // slots handed out so far
    std::unordered_map<uintptr_t, int> slot;   // stream handle -> slot
};
std::mutex g_mu;
DeviceState g_dev[64];

// Looks up (once per device, with that device current) the address of the
// device's error words and its SM count; if err is not NULL, *err receives
// the error word of `stream` on this device.
bool device_state(cudaStream_t stream, uint32_t **err, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &ds = g_dev[dev];
    if (!ds.words) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_words) != cudaSuccess || !p) return false;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return false;
        ds.words = static_cast<uint32_t *>(p);
        ds.num_sms = n;
    }
    if (err) {
        const uintptr_t key = reinterpret_cast<uintptr_t>(stream);
        auto it = ds.slot.find(key);
        int s;
        if (it != ds.slot.end()) {
            s = it->second;
        } else if (ds.used < kErrSlots) {
            s = ds.used++;
            ds.slot.emplace(key, s);
        } else {
            s = static_cast<int>((key >> 4) % kErrSlots);
        }
        *err = ds.words + s;
    }
    if (num_sms) *num_sms = ds.num_sms;
    return true;
}

// Error words of every slot handed out on the current device (for the
// device-wide read).
bool device_words(uint32_t **words, int *used) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!device_state(nullptr, nullptr, nullptr)) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    *words = g_dev[dev].words;
    *used = g_dev[dev].used;
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s, int esize) { return s > 0 && ((s * esize) % 16) == 0 && s < (int64_t(1) << 36); }

da_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DA_OK : DA_ERR_CUDA; }

}  // namespace

bool encode_map_4d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t d1, uint64_t d2, uint64_t d3,
                   int64_t s1, int64_t s2, int64_t s3, uint32_t box_rows, int l2_promo_bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {inner, d1, d2, d3};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(s1) * 2, static_cast<cuuint64_t>(s2) * 2,
                             static_cast<cuuint64_t>(s3) * 2};
    cuuint32_t box[4] = {64, 1, box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          l2_promo_bytes == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_map_pairs(CUtensorMap *m, const void *base, uint64_t D, uint64_t H, uint64_t T, uint64_t B) {
    auto fn = encode_fn();
    if (!fn || (H & 1) || D % 64 != 0) return false;
    cuuint64_t dims[5] = {D, 2, H / 2, T, B};
    cuuint64_t strides[4] = {D * 2, 2 * D * 2, H * D * 2, T * H * D * 2};
    cuuint32_t box[5] = {64, 2, 1, 64, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void set_last_launches(int n) { t_last_launches = n; }

}  // namespace da

using namespace da;

extern "C" {

const char *diffattn_status_string(da_status s) {
    switch (s) {
        case DA_OK: return "ok";
        case DA_ERR_NULL_PTR: return "a required pointer is NULL";
        case DA_ERR_BAD_SHAPE: return "a size is out of range";
        case DA_ERR_UNSUPPORTED_DIM: return "head dimension not supported for this dtype";
        case DA_ERR_BAD_GROUP: return "Hq must be a multiple of Hkv with an even group size (<= 8 for bf16 decode)";
        case DA_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
        case DA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case DA_ERR_CUDA: return "CUDA error";
        case DA_ERR_BAD_DTYPE: return "unknown dtype";
        case DA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (device error word set)";
        case DA_ERR_SCRATCH_LIMIT:
            return "sizes need more decode scratch than the library's static 8 MiB buffer; "
                   "use diffattn_v2_decode with a workspace";
        case DA_ERR_BAD_LENGTH: return "a decode cache length was outside 1..L and was clamped";
        case DA_ERR_DEVICE_BOUNDS: return "a bounds check of the debug build failed (the access was skipped)";
    }
    return "unknown status";
}

int diffattn_last_launch_count(void) { return t_last_launches; }

static da_status status_of_word(uint32_t v) {
    if (v == 0) return DA_OK;
    if (v & kErrFatal) return DA_ERR_DEVICE_TIMEOUT;
    if (v & kErrBounds) return DA_ERR_DEVICE_BOUNDS;
    if (v & kErrBadLength) return DA_ERR_BAD_LENGTH;
    return DA_ERR_DEVICE_TIMEOUT;
}

da_status diffattn_device_error(uint32_t *code) {
    uint32_t *words = nullptr;
    int used = 0;
    if (!device_words(&words, &used)) return DA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DA_ERR_CUDA;
    uint32_t v = 0;
    if (used > 0) {
        uint32_t w[kErrSlots];
        if (cudaMemcpy(w, words, sizeof(uint32_t) * used, cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
        for (int i = 0; i < used; ++i) v |= w[i];
        if (v != 0 && cudaMemset(words, 0, sizeof(uint32_t) * used) != cudaSuccess) return DA_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return DA_ERR_CUDA;
    }
    if (code) *code = v;
    return status_of_word(v);
}

da_status diffattn_stream_error(uint32_t *code, cudaStream_t stream) {
    uint32_t *err = nullptr;
    if (!device_state(stream, &err, nullptr)) return DA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
    if (v != 0) {
        if (cudaMemsetAsync(err, 0, sizeof(v), stream) != cudaSuccess) return DA_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
    }
    if (code) *code = v;
    return status_of_word(v);
}

da_status diffattn_selftest_wait_limit(uint32_t *code, cudaStream_t stream) {
    uint32_t *err = nullptr;
    if (!device_state(stream, &err, nullptr)) return DA_ERR_CUDA;
    uint32_t before = 0;
    if (diffattn_stream_error(&before, stream) == DA_ERR_CUDA) return DA_ERR_CUDA;   // start from a clear word
    bool gave_up = false;
    if (run_wait_selftest(err, &gave_up, stream) != cudaSuccess) return DA_ERR_CUDA;
    uint32_t v = 0;
    if (diffattn_stream_error(&v, stream) == DA_ERR_CUDA) return DA_ERR_CUDA;   // reads and clears the word
    if (code) *code = v;
    t_last_launches = 1;
    return (gave_up && (v & kErrWaitTimeout) != 0) ? DA_OK : DA_ERR_CUDA;
}

int diffattn_debug_checks(void) { return kDebugChecks ? 1 : 0; }

da_status diffattn_selftest_bounds(uint32_t *code, cudaStream_t stream) {
    uint32_t *err = nullptr;
    if (!device_state(stream, &err, nullptr)) return DA_ERR_CUDA;
    uint32_t before = 0;
    if (diffattn_stream_error(&before, stream) == DA_ERR_CUDA) return DA_ERR_CUDA;   // start from a clear word
    bool wrote = true;
    if (run_bounds_selftest(err, &wrote, stream) != cudaSuccess) return DA_ERR_CUDA;
    uint32_t v = 0;
    if (diffattn_stream_error(&v, stream) == DA_ERR_CUDA) return DA_ERR_CUDA;   // reads and clears the word
    if (code) *code = v;
    t_last_launches = 1;
    if (wrote) return DA_ERR_CUDA;   // the write past the end must be skipped in both builds
    return (kDebugChecks ? v == kErrBounds : v == 0) ? DA_OK : DA_ERR_CUDA;
}

da_status diffattn_v1_fwd(const void *q1, const void *q2, const void *k1, const void *k2, const void *v,
                          const float *lam_q1, const float *lam_k1, const float *lam_q2, const float *lam_k2,
                          void *out, int B, int T, int H, int d, int layer_index,
                          int64_t q_sb, int64_t q_st, int64_t q_sh, int64_t k_sb, int64_t k_st, int64_t k_sh,
                          int64_t v_sb, int64_t v_st, int64_t v_sh, int64_t o_sb, int64_t o_st, int64_t o_sh,
                          da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q1 || !q2 || !k1 || !k2 || !v || !lam_q1 || !lam_k1 || !lam_q2 || !lam_k2 || !out)
        return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || H < 1 || layer_index < 0) return DA_ERR_BAD_SHAPE;
    const int es = dtype == DA_BF16 ? 2 : 4;
    // bf16: d = 64 runs the one-pass kernel, d = 32 the same kernel with q and
    // k read through 64-column boxes whose upper half the copy fills with
    // zeros (Q K^T unchanged), d = 128 (dv = 256: two fp32 accumulators would
    // not fit in TMEM next to S) the two-pass kernel
    const bool twopass = dtype == DA_BF16 && d == 128;
    if (dtype == DA_BF16 ? !(twopass || prefill_supported(d, 2 * d, false)) : (d != 32 && d != 64 && d != 128))
        return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q1, q2, k1, k2, v, static_cast<const void *>(out)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    for (int64_t s : {q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh, o_sb, o_st, o_sh})
        if (!stride_ok(s, es)) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = static_cast<const float *>(q1); p.q2 = static_cast<const float *>(q2);
        p.k1 = static_cast<const float *>(k1); p.k2 = static_cast<const float *>(k2);
        p.v = static_cast<const float *>(v);
        p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
        p.k_sb = k_sb; p.k_st = k_st; p.k_sh = k_sh;
        p.v_sb = v_sb; p.v_st = v_st; p.v_sh = v_sh;
        p.o_sb = o_sb; p.o_st = o_st; p.o_sh = o_sh;
        p.out = static_cast<float *>(out);
        p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
        p.layer_index = layer_index;
        p.B = B; p.Tq = T; p.Lk = T; p.H = H; p.G = 1; p.mode = 1;
        p.err = err;
        const da_status st = cuda_status(launch_simt(p, d, 2 * d, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uH = static_cast<uint64_t>(H), uB = static_cast<uint64_t>(B);
    if (!encode_map_4d(&m.q1, q1, d, uH, uT, uB, q_sh, q_st, q_sb, 128) ||
        !encode_map_4d(&m.q2, q2, d, uH, uT, uB, q_sh, q_st, q_sb, 128) ||
        !encode_map_4d(&m.k1, k1, d, uH, uT, uB, k_sh, k_st, k_sb, 128) ||
        !encode_map_4d(&m.k2, k2, d, uH, uT, uB, k_sh, k_st, k_sb, 128) ||
        !encode_map_4d(&m.v, v, 2 * d, uH, uT, uB, v_sh, v_st, v_sb,
                       twopass ? static_cast<uint32_t>(prefill_v1_twopass_v_rows(d)) : 128u) ||
        !encode_map_4d(&m.out, out, 2 * d, uH, uT, uB, o_sh, o_st, o_sb, 128))
        return DA_ERR_CUDA;
    PrefillParams p{};
    p.out = out; p.o_sb = o_sb; p.o_st = o_st; p.o_sh = o_sh;
    p.lam = nullptr;
    p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
    p.dlam = d;
    p.layer_index = layer_index;
    p.B = B; p.T = T; p.H = H; p.G = 1;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    p.num_sms = nsm;
    p.err = err;
    const da_status st = cuda_status(twopass ? launch_prefill_v1_twopass(m, p, d, stream)
                                             : launch_prefill(m, p, d, 2 * d, false, stream));
    if (st == DA_OK) t_last_launches = 1;
    return st;
}

da_status diffattn_v2_fwd(const void *q, const void *k, const void *v, const float *lam, void *out, int B, int T,
                          int Hq, int Hkv, int D, da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !lam || !out) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || Hq < 2 || Hkv < 1) return DA_ERR_BAD_SHAPE;
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1)) return DA_ERR_BAD_GROUP;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    const int P = Hq / 2, G = Hq / Hkv;
    t_last_launches = 0;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = p.q2 = static_cast<const float *>(q);
        p.k1 = p.k2 = static_cast<const float *>(k);
        p.v = static_cast<const float *>(v);
        p.q_sh = D; p.q_st = static_cast<int64_t>(Hq) * D; p.q_sb = p.q_st * T;
        p.k_sh = D; p.k_st = static_cast<int64_t>(Hkv) * D; p.k_sb = p.k_st * T;
        p.v_sh = p.k_sh; p.v_st = p.k_st; p.v_sb = p.k_sb;
        p.o_sh = D; p.o_st = static_cast<int64_t>(P) * D; p.o_sb = p.o_st * T;
        p.out = static_cast<float *>(out);
        p.lam = lam; p.lam_st = P; p.lam_sb = static_cast<int64_t>(P) * T;
        p.B = B; p.Tq = T; p.Lk = T; p.H = P; p.G = G; p.mode = 2;
        p.err = err;
        const da_status st = cuda_status(launch_simt(p, D, D, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uB = static_cast<uint64_t>(B);
    const int64_t qst = static_cast<int64_t>(Hq) * D, kst = static_cast<int64_t>(Hkv) * D;
    if (!encode_map_4d(&m.q1, q, D, Hq, uT, uB, D, qst, qst * T, 128) ||
        !encode_map_4d(&m.k1, k, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.v, v, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.out, out, D, P, uT, uB, D, static_cast<int64_t>(P) * D, static_cast<int64_t>(P) * D * T, 128))
        return DA_ERR_CUDA;
    m.q2 = m.q1;
    m.k2 = m.k1;
    PrefillParams p{};
    p.out = out;
    p.o_sh = D; p.o_st = static_cast<int64_t>(P) * D; p.o_sb = p.o_st * T;
    p.lam = lam;
    p.B = B; p.T = T; p.H = P; p.G = G;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.num_sms = nsm;
    p.err = err;
    const da_status st = cuda_status(launch_prefill(m, p, D, D, true, stream));
    if (st == DA_OK) t_last_launches = 1;
    return st;
}

da_status diffattn_v2_fwd_rope(const void *q, void *k, const void *v, const float *lam, void *out, int B, int T,
                               int Hq, int Hkv, int D, int64_t pos0, float base, da_dtype dtype,
                               cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !lam || !out) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || Hq < 2 || Hkv < 1 || !(base > 0.f)) return DA_ERR_BAD_SHAPE;
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1)) return DA_ERR_BAD_GROUP;
    if (dtype != DA_BF16 || (D != 64 && D != 128)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, static_cast<const void *>(k), v, static_cast<const void *>(out)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    const int P = Hq / 2, G = Hq / Hkv;
    t_last_launches = 0;
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uB = static_cast<uint64_t>(B);
    const int64_t qst = static_cast<int64_t>(Hq) * D, kst = static_cast<int64_t>(Hkv) * D;
    if (!encode_map_4d(&m.q1, q, D, Hq, uT, uB, D, qst, qst * T, 128) ||
        !encode_map_4d(&m.k1, k, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.v, v, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.out, out, D, P, uT, uB, D, static_cast<int64_t>(P) * D, static_cast<int64_t>(P) * D * T, 128))
        return DA_ERR_CUDA;
    m.q2 = m.q1;
    m.k2 = m.k1;
    // k rotated in place
    PrologueParams r{};
    r.k = k;
    r.Hq = 0; r.Hk = Hkv; r.D = D;
    r.B = B; r.T = T;
    r.pos0 = pos0;
    r.base = static_cast<double>(base);
    r.err = err;
    da_status st = cuda_status(launch_prologue(r, true, stream));
    if (st != DA_OK) return st;
    t_last_launches = 1;
    PrefillParams p{};
    p.out = out;
    p.o_sh = D; p.o_st = static_cast<int64_t>(P) * D; p.o_sb = p.o_st * T;
    p.lam = lam;
    p.B = B; p.T = T; p.H = P; p.G = G;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.num_sms = nsm;
    p.err = err;
    p.rope_pos0 = pos0;
    p.rope_base = static_cast<double>(base);
    st = cuda_status(launch_prefill_v2_rope(m, p, D, stream));
    if (st == DA_OK) t_last_launches = 2;
    return st;
}

da_status diffattn_paired_fwd(const void *q, const void *k, const void *v, void *out, int B, int T, int H, int D,
                              da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !out) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || H < 2 || (H & 1)) return DA_ERR_BAD_SHAPE;
    if (dtype != DA_BF16 || !paired_supported(D)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uB = static_cast<uint64_t>(B), uH = static_cast<uint64_t>(H);
    const int64_t st = static_cast<int64_t>(H) * D;
    if (!encode_map_4d(&m.q1, q, D, uH, uT, uB, D, st, st * T, 128) ||
        !encode_map_pairs(&m.k1, k, D, uH, uT, uB) || !encode_map_pairs(&m.v, v, D, uH, uT, uB))
        return DA_ERR_CUDA;
    m.q2 = m.q1;
    m.k2 = m.k1;
    m.out = m.q1;   // not read: the paired epilogue stores directly
    PrefillParams p{};
    p.out = out;
    p.o_sh = D; p.o_st = st; p.o_sb = st * T;
    p.B = B; p.T = T; p.H = H / 2; p.G = 2;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.num_sms = nsm;
    p.err = err;
    const da_status s = cuda_status(launch_paired(m, p, D, stream));
    if (s == DA_OK) t_last_launches = 1;
    return s;
}

size_t diffattn_v2_decode_workspace_size(int B, int L, int Hq, int Hkv, int D, da_dtype dtype) {
    if (dtype == DA_F32) return 0;
    if (dtype != DA_BF16 || Hkv < 1 || Hq % Hkv != 0) return 0;
    if (D != 64 && D != 128) return 0;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(nullptr, nullptr, &nsm)) return 0;
    int grid, spb;
    int64_t units;
    size_t cum = 0, ws = 0;
    // sized for per-sequence lengths, which also covers the all-L call
    if (!decode_plan(B, L, Hkv, D, nsm, true, &grid, &units, &spb, &cum, &ws)) return 0;
    return ws;
}

size_t diffattn_v1_decode_workspace_size(int B, int L, int H, int d, da_dtype dtype) {
    if (dtype != DA_BF16 || (d != 32 && d != 64 && d != 128)) return 0;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(nullptr, nullptr, &nsm)) return 0;
    int grid, spb;
    int64_t units;
    size_t cum = 0, ws = 0;
    if (!decode_plan(B, L, H, d == 32 ? 128 : 2 * d, nsm, true, &grid, &units, &spb, &cum, &ws)) return 0;
    return ws;
}

}  // extern "C"

namespace {

// bf16 split-KV decode shared by the V2 and V1 entry points (arguments
// already checked): plan, tensor maps, workspace split, launch.
da_status decode_bf16(bool v1, const DecodeMaps &m, DecodeParams p, const int32_t *lens, void *workspace,
                      size_t workspace_bytes, int nsm, cudaStream_t stream) {
    int grid, spb;
    int64_t units;
    size_t cum = 0, need = 0;
    if (!decode_plan(p.B, p.L, p.Hkv, p.D, nsm, lens != nullptr, &grid, &units, &spb, &cum, &need))
        return DA_ERR_BAD_SHAPE;
    if (!workspace) return DA_ERR_NULL_PTR;
    if (!aligned16(workspace)) return DA_ERR_MISALIGNED;
    if (workspace_bytes < need) return DA_ERR_WORKSPACE_TOO_SMALL;
    p.lens = lens;
    p.cum = lens ? static_cast<int64_t *>(workspace) : nullptr;
    p.ws = reinterpret_cast<float *>(static_cast<char *>(workspace) + cum);
    p.grid = grid;
    p.units = units;
    p.spb = spb;
    const da_status st = cuda_status(launch_decode(m, p, v1, stream));
    if (st == DA_OK) t_last_launches = lens ? 3 : 2;
    return st;
}

}  // namespace

// Argument checks of the V2 decode entry points (nothing enqueued on failure).
static da_status v2_decode_check(const void *q, const void *k_cache, const void *v_cache, const float *lam,
                                 const void *out, int B, int L, int Hq, int Hkv, int D, da_dtype dtype) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k_cache || !v_cache || !lam || !out) return DA_ERR_NULL_PTR;
    if (B < 1 || L < 1 || Hq < 2 || Hkv < 1) return DA_ERR_BAD_SHAPE;
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1)) return DA_ERR_BAD_GROUP;
    if (D != 64 && D != 128) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, k_cache, v_cache, out})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    if (dtype == DA_BF16 && Hq / Hkv > 8) return DA_ERR_BAD_GROUP;
    return DA_OK;
}

namespace {

da_status v2_decode_impl(const void *q, const void *k_cache, const void *v_cache, const float *lam,
                         const int32_t *lens, void *out, void *workspace, size_t workspace_bytes, int B, int L,
                         int Hq, int Hkv, int D, da_dtype dtype, cudaStream_t stream) {
    const da_status chk = v2_decode_check(q, k_cache, v_cache, lam, out, B, L, Hq, Hkv, D, dtype);
    if (chk != DA_OK) return chk;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    const int P = Hq / 2, G = Hq / Hkv;
    t_last_launches = 0;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = p.q2 = static_cast<const float *>(q);
        p.k1 = p.k2 = static_cast<const float *>(k_cache);
        p.v = static_cast<const float *>(v_cache);
        p.q_sh = D; p.q_st = 0; p.q_sb = static_cast<int64_t>(Hq) * D;
        p.k_sh = D; p.k_st = static_cast<int64_t>(Hkv) * D; p.k_sb = p.k_st * L;
        p.v_sh = p.k_sh; p.v_st = p.k_st; p.v_sb = p.k_sb;
        p.o_sh = D; p.o_st = 0; p.o_sb = static_cast<int64_t>(P) * D;
        p.out = static_cast<float *>(out);
        p.lam = lam; p.lam_st = 0; p.lam_sb = P;
        p.B = B; p.Tq = 1; p.Lk = L; p.H = P; p.G = G; p.mode = 2;
        p.lens = lens;
        p.err = err;
        const da_status st = cuda_status(launch_simt(p, D, D, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    if (G > 8) return DA_ERR_BAD_GROUP;
    DecodeMaps m;
    const int64_t st_row = static_cast<int64_t>(Hkv) * D;
    // a decode unit reads D * 2 bytes of each cache row and the neighbouring
    // bytes belong to another head: promote L2 fills no wider than a row
    const int promo = D * 2 <= 128 ? 128 : 256;
    if (!encode_map_4d(&m.k, k_cache, D, Hkv, static_cast<uint64_t>(L), B, D, st_row, st_row * L,
                       kDecodeKeysPerUnit, promo) ||
        !encode_map_4d(&m.v, v_cache, D, Hkv, static_cast<uint64_t>(L), B, D, st_row, st_row * L,
                       kDecodeKeysPerUnit, promo))
        return DA_ERR_CUDA;
    m.k2 = m.k;
    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.lam = lam;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.B = B; p.L = L; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.D = D;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.err = err;
    return decode_bf16(false, m, p, lens, workspace, workspace_bytes, nsm, stream);
}

}  // namespace

extern "C" {

da_status diffattn_v2_decode(const void *q, const void *k_cache, const void *v_cache, const float *lam, void *out,
                             void *workspace, size_t workspace_bytes, int B, int L, int Hq, int Hkv, int D,
                             da_dtype dtype, cudaStream_t stream) {
    return v2_decode_impl(q, k_cache, v_cache, lam, nullptr, out, workspace, workspace_bytes, B, L, Hq, Hkv, D,
                          dtype, stream);
}

da_status diffattn_v2_decode_varlen(const void *q, const void *k_cache, const void *v_cache, const float *lam,
                                    const int32_t *cache_lens, void *out, void *workspace, size_t workspace_bytes,
                                    int B, int L, int Hq, int Hkv, int D, da_dtype dtype, cudaStream_t stream) {
    if (!cache_lens) return DA_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return DA_ERR_MISALIGNED;
    return v2_decode_impl(q, k_cache, v_cache, lam, cache_lens, out, workspace, workspace_bytes, B, L, Hq, Hkv,
                          D, dtype, stream);
}

da_status diffattn_v1_decode(const void *q1, const void *q2, const void *k1_cache, const void *k2_cache,
                             const void *v_cache, const float *lam_q1, const float *lam_k1, const float *lam_q2,
                             const float *lam_k2, const int32_t *cache_lens, void *out, void *workspace,
                             size_t workspace_bytes, int B, int L, int H, int d, int layer_index, da_dtype dtype,
                             cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q1 || !q2 || !k1_cache || !k2_cache || !v_cache || !lam_q1 || !lam_k1 || !lam_q2 || !lam_k2 || !out)
        return DA_ERR_NULL_PTR;
    if (B < 1 || L < 1 || H < 1 || layer_index < 0) return DA_ERR_BAD_SHAPE;
    if (d != 32 && d != 64 && d != 128)
        return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q1, q2, k1_cache, k2_cache, v_cache, static_cast<const void *>(out)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    if (cache_lens && (reinterpret_cast<uintptr_t>(cache_lens) & 3u) != 0) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    const int dv = 2 * d;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = static_cast<const float *>(q1);
        p.q2 = static_cast<const float *>(q2);
        p.k1 = static_cast<const float *>(k1_cache);
        p.k2 = static_cast<const float *>(k2_cache);
        p.v = static_cast<const float *>(v_cache);
        p.q_sh = d; p.q_st = 0; p.q_sb = static_cast<int64_t>(H) * d;
        p.k_sh = d; p.k_st = static_cast<int64_t>(H) * d; p.k_sb = p.k_st * L;
        p.v_sh = dv; p.v_st = static_cast<int64_t>(H) * dv; p.v_sb = p.v_st * L;
        p.o_sh = dv; p.o_st = 0; p.o_sb = static_cast<int64_t>(H) * dv;
        p.out = static_cast<float *>(out);
        p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
        p.layer_index = layer_index;
        p.B = B; p.Tq = 1; p.Lk = L; p.H = H; p.G = 1; p.mode = 1;
        p.lens = cache_lens;
        p.err = err;
        const da_status st = cuda_status(launch_simt(p, d, dv, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    DecodeMaps m;
    const int64_t kr = static_cast<int64_t>(H) * d, vr = static_cast<int64_t>(H) * dv;
    const int kpromo = d * 2 <= 128 ? 128 : 256;   // as for the V2 cache maps
    if (!encode_map_4d(&m.k, k1_cache, d, H, static_cast<uint64_t>(L), B, d, kr, kr * L, kDecodeKeysPerUnit,
                       kpromo) ||
        !encode_map_4d(&m.k2, k2_cache, d, H, static_cast<uint64_t>(L), B, d, kr, kr * L, kDecodeKeysPerUnit,
                       kpromo) ||
        !encode_map_4d(&m.v, v_cache, dv, H, static_cast<uint64_t>(L), B, dv, vr, vr * L, kDecodeKeysPerUnit))
        return DA_ERR_CUDA;
    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(q1);
    p.q2 = static_cast<const __nv_bfloat16 *>(q2);
    p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
    p.layer_index = layer_index;
    p.out = static_cast<__nv_bfloat16 *>(out);
    // d = 32 runs the d = 64 configuration: the k maps are d wide and the v map
    // 2d wide, their 64-column boxes zero-filled past that (q is zero-padded in
    // the kernel), so the scores and the first 2d output channels are the same
    p.B = B; p.L = L; p.Hq = H; p.Hkv = H; p.G = 2; p.D = d == 32 ? 128 : dv;
    p.dq = d; p.dv = dv;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    p.err = err;
    return decode_bf16(true, m, p, cache_lens, workspace, workspace_bytes, nsm, stream);
}

}  // extern "C"

// ------------------------------------------------------------ training

namespace {
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Saved-tensor layout of a training forward: two (B, T, H, DV) tensors
// (V1: x and a2 in fp32; V2: a_e and a_o in bf16) | lse (fp32, (2, B, H, T)),
// each part 256-byte aligned.
struct SavedLayout {
    size_t a_bytes, off_a2, off_lse, total;
    SavedLayout(int B, int T, int H, int DV, int esize) {
        a_bytes = round256(static_cast<size_t>(B) * T * H * DV * esize);
        off_a2 = a_bytes;
        off_lse = 2 * a_bytes;
        total = off_lse + round256(static_cast<size_t>(2) * B * H * T * 4);
    }
};
// Backward workspace: D (2, B, H, T) | c (B, H, T) | V1: dlam rows (B, T, H) | g ((B, T, H, DV),
// gsize bytes per element: bf16 on the tensor-core path, fp32 on the CUDA-core one)
struct BwdWsLayout {
    size_t off_c, off_rows, off_g, total;
    BwdWsLayout(int B, int T, int H, int DV, bool v1, int gsize) {
        const size_t n = static_cast<size_t>(B) * H * T;
        off_c = round256(2 * n * 4);
        off_rows = off_c + round256(n * 4);
        off_g = off_rows + (v1 ? round256(n * 4) : 0);
        total = off_g + (v1 ? round256(n * DV * gsize) : 0);
    }
};
bool shape_ok_bytes(int B, int T, int H, int DV) {
    return B >= 1 && T >= 1 && H >= 1 && static_cast<double>(B) * T * H * DV < 4.0e12;
}
// Training support: bf16 on the tcgen05 kernels, fp32 on the CUDA-core ones.
bool train_supported(int dqk, bool v2, da_dtype dtype) {
    if (dtype == DA_BF16) return backward_supported(dqk, v2 ? dqk : 2 * dqk, v2);
    if (dtype == DA_F32) return v2 ? (dqk == 64 || dqk == 128) : (dqk == 32 || dqk == 64 || dqk == 128);
    return false;
}
int saved_esize(bool v2, da_dtype dtype) { return (v2 && dtype == DA_BF16) ? 2 : 4; }
}  // namespace

extern "C" {

size_t diffattn_v1_train_saved_size(int B, int T, int H, int d, da_dtype dtype) {
    if (!shape_ok_bytes(B, T, H, 2 * d) || !train_supported(d, false, dtype)) return 0;
    return SavedLayout(B, T, H, 2 * d, saved_esize(false, dtype)).total;
}
size_t diffattn_v2_train_saved_size(int B, int T, int Hq, int Hkv, int D, da_dtype dtype) {
    if (Hq < 2 || Hkv < 1 || !shape_ok_bytes(B, T, Hq / 2, D) || !train_supported(D, true, dtype)) return 0;
    return SavedLayout(B, T, Hq / 2, D, saved_esize(true, dtype)).total;
}
size_t diffattn_v1_train_saved_lse_offset(int B, int T, int H, int d, da_dtype dtype) {
    if (!shape_ok_bytes(B, T, H, 2 * d) || !train_supported(d, false, dtype)) return 0;
    return SavedLayout(B, T, H, 2 * d, saved_esize(false, dtype)).off_lse;
}
size_t diffattn_v2_train_saved_lse_offset(int B, int T, int Hq, int Hkv, int D, da_dtype dtype) {
    if (Hq < 2 || Hkv < 1 || !shape_ok_bytes(B, T, Hq / 2, D) || !train_supported(D, true, dtype)) return 0;
    return SavedLayout(B, T, Hq / 2, D, saved_esize(true, dtype)).off_lse;
}
size_t diffattn_v1_bwd_workspace_size(int B, int T, int H, int d, da_dtype dtype) {
    if (!shape_ok_bytes(B, T, H, 2 * d) || !train_supported(d, false, dtype)) return 0;
    return BwdWsLayout(B, T, H, 2 * d, true, dtype == DA_F32 ? 4 : 2).total;
}
size_t diffattn_v2_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D, da_dtype dtype) {
    if (Hq < 2 || Hkv < 1 || !shape_ok_bytes(B, T, Hq / 2, D) || !train_supported(D, true, dtype)) return 0;
    return BwdWsLayout(B, T, Hq / 2, D, false, 4).total;
}

da_status diffattn_v1_fwd_train(const void *q1, const void *q2, const void *k1, const void *k2, const void *v,
                                const float *lam_q1, const float *lam_k1, const float *lam_q2, const float *lam_k2,
                                void *out, void *saved, size_t saved_bytes, int B, int T, int H, int d,
                                int layer_index, int64_t q_sb, int64_t q_st, int64_t q_sh, int64_t k_sb,
                                int64_t k_st, int64_t k_sh, int64_t v_sb, int64_t v_st, int64_t v_sh, int64_t o_sb,
                                int64_t o_st, int64_t o_sh, da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q1 || !q2 || !k1 || !k2 || !v || !lam_q1 || !lam_k1 || !lam_q2 || !lam_k2 || !out || !saved)
        return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || H < 1 || layer_index < 0) return DA_ERR_BAD_SHAPE;
    if (!train_supported(d, false, dtype)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q1, q2, k1, k2, v, static_cast<const void *>(out), static_cast<const void *>(saved)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    for (int64_t st : {q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh, o_sb, o_st, o_sh})
        if (!stride_ok(st, dtype == DA_F32 ? 4 : 2)) return DA_ERR_MISALIGNED;
    const SavedLayout sl(B, T, H, 2 * d, saved_esize(false, dtype));
    if (saved_bytes < sl.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = static_cast<const float *>(q1); p.q2 = static_cast<const float *>(q2);
        p.k1 = static_cast<const float *>(k1); p.k2 = static_cast<const float *>(k2);
        p.v = static_cast<const float *>(v);
        p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
        p.k_sb = k_sb; p.k_st = k_st; p.k_sh = k_sh;
        p.v_sb = v_sb; p.v_st = v_st; p.v_sh = v_sh;
        p.o_sb = o_sb; p.o_st = o_st; p.o_sh = o_sh;
        p.out = static_cast<float *>(out);
        p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
        p.layer_index = layer_index;
        p.B = B; p.Tq = T; p.Lk = T; p.H = H; p.G = 1; p.mode = 1;
        p.err = err;
        char *sv = static_cast<char *>(saved);
        p.sa1 = reinterpret_cast<float *>(sv);
        p.sa2 = reinterpret_cast<float *>(sv + sl.off_a2);
        p.slse = reinterpret_cast<float *>(sv + sl.off_lse);
        const da_status st = cuda_status(launch_simt(p, d, 2 * d, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uH = static_cast<uint64_t>(H), uB = static_cast<uint64_t>(B);
    // d = 128: the two-pass kernel (its V map has the item-sized box)
    const bool twopass = d == 128;
    if (!encode_map_4d(&m.q1, q1, d, uH, uT, uB, q_sh, q_st, q_sb, 128) ||
        !encode_map_4d(&m.q2, q2, d, uH, uT, uB, q_sh, q_st, q_sb, 128) ||
        !encode_map_4d(&m.k1, k1, d, uH, uT, uB, k_sh, k_st, k_sb, 128) ||
        !encode_map_4d(&m.k2, k2, d, uH, uT, uB, k_sh, k_st, k_sb, 128) ||
        !encode_map_4d(&m.v, v, 2 * d, uH, uT, uB, v_sh, v_st, v_sb,
                       twopass ? static_cast<uint32_t>(prefill_v1_twopass_v_rows(d)) : 128u) ||
        !encode_map_4d(&m.out, out, 2 * d, uH, uT, uB, o_sh, o_st, o_sb, 128))
        return DA_ERR_CUDA;
    PrefillParams p{};
    p.out = out; p.o_sb = o_sb; p.o_st = o_st; p.o_sh = o_sh;
    p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
    p.dlam = d;
    p.layer_index = layer_index;
    p.B = B; p.T = T; p.H = H; p.G = 1;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    p.num_sms = nsm;
    p.err = err;
    char *sv = static_cast<char *>(saved);
    p.sa1 = sv;
    p.sa2 = sv + sl.off_a2;
    p.slse = reinterpret_cast<float *>(sv + sl.off_lse);
    const da_status st = cuda_status(twopass ? launch_prefill_v1_twopass_train(m, p, stream)
                                             : launch_prefill_train(m, p, d, 2 * d, false, stream));
    if (st == DA_OK) t_last_launches = twopass ? 2 : 1;
    return st;
}

da_status diffattn_v2_fwd_train(const void *q, const void *k, const void *v, const float *lam, void *out,
                                void *saved, size_t saved_bytes, int B, int T, int Hq, int Hkv, int D,
                                da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !lam || !out || !saved) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || Hq < 2 || Hkv < 1) return DA_ERR_BAD_SHAPE;
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1)) return DA_ERR_BAD_GROUP;
    if (!train_supported(D, true, dtype)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out), static_cast<const void *>(saved)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    const int P = Hq / 2, G = Hq / Hkv;
    const SavedLayout sl(B, T, P, D, saved_esize(true, dtype));
    if (saved_bytes < sl.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    if (dtype == DA_F32) {
        SimtParams p{};
        p.q1 = p.q2 = static_cast<const float *>(q);
        p.k1 = p.k2 = static_cast<const float *>(k);
        p.v = static_cast<const float *>(v);
        p.q_sh = D; p.q_st = static_cast<int64_t>(Hq) * D; p.q_sb = p.q_st * T;
        p.k_sh = D; p.k_st = static_cast<int64_t>(Hkv) * D; p.k_sb = p.k_st * T;
        p.v_sh = p.k_sh; p.v_st = p.k_st; p.v_sb = p.k_sb;
        p.o_sh = D; p.o_st = static_cast<int64_t>(P) * D; p.o_sb = p.o_st * T;
        p.out = static_cast<float *>(out);
        p.lam = lam; p.lam_st = P; p.lam_sb = static_cast<int64_t>(P) * T;
        p.B = B; p.Tq = T; p.Lk = T; p.H = P; p.G = G; p.mode = 2;
        p.err = err;
        char *sv = static_cast<char *>(saved);
        p.sa1 = reinterpret_cast<float *>(sv);
        p.sa2 = reinterpret_cast<float *>(sv + sl.off_a2);
        p.slse = reinterpret_cast<float *>(sv + sl.off_lse);
        const da_status st = cuda_status(launch_simt(p, D, D, stream));
        if (st == DA_OK) t_last_launches = 1;
        return st;
    }
    PrefillMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uB = static_cast<uint64_t>(B);
    const int64_t qst = static_cast<int64_t>(Hq) * D, kst = static_cast<int64_t>(Hkv) * D;
    if (!encode_map_4d(&m.q1, q, D, Hq, uT, uB, D, qst, qst * T, 128) ||
        !encode_map_4d(&m.k1, k, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.v, v, D, Hkv, uT, uB, D, kst, kst * T, 128) ||
        !encode_map_4d(&m.out, out, D, P, uT, uB, D, static_cast<int64_t>(P) * D, static_cast<int64_t>(P) * D * T, 128))
        return DA_ERR_CUDA;
    m.q2 = m.q1;
    m.k2 = m.k1;
    PrefillParams p{};
    p.out = out;
    p.o_sh = D; p.o_st = static_cast<int64_t>(P) * D; p.o_sb = p.o_st * T;
    p.lam = lam;
    p.B = B; p.T = T; p.H = P; p.G = G;
    p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    p.num_sms = nsm;
    p.err = err;
    char *sv = static_cast<char *>(saved);
    p.sa1 = sv;
    p.sa2 = sv + sl.off_a2;
    p.slse = reinterpret_cast<float *>(sv + sl.off_lse);
    const da_status st = cuda_status(launch_prefill_train(m, p, D, D, true, stream));
    if (st == DA_OK) t_last_launches = 1;
    return st;
}

da_status diffattn_v1_bwd(const void *q1, const void *q2, const void *k1, const void *k2, const void *v,
                          const float *lam_q1, const float *lam_k1, const float *lam_q2, const float *lam_k2,
                          const void *dout, const void *saved, size_t saved_bytes, void *dq1, void *dq2, void *dk1,
                          void *dk2, void *dv, float *dlam_q1, float *dlam_k1, float *dlam_q2, float *dlam_k2,
                          void *workspace, size_t workspace_bytes, int B, int T, int H, int d, int layer_index,
                          int64_t q_sb, int64_t q_st, int64_t q_sh, int64_t k_sb, int64_t k_st, int64_t k_sh,
                          int64_t v_sb, int64_t v_st, int64_t v_sh, int64_t o_sb, int64_t o_st, int64_t o_sh,
                          da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q1 || !q2 || !k1 || !k2 || !v || !lam_q1 || !lam_k1 || !lam_q2 || !lam_k2 || !dout || !saved || !dq1 ||
        !dq2 || !dk1 || !dk2 || !dv || !dlam_q1 || !dlam_k1 || !dlam_q2 || !dlam_k2 || !workspace)
        return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || H < 1 || layer_index < 0) return DA_ERR_BAD_SHAPE;
    if (!train_supported(d, false, dtype)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q1, q2, k1, k2, v, dout, saved, static_cast<const void *>(dq1),
                            static_cast<const void *>(dq2), static_cast<const void *>(dk1),
                            static_cast<const void *>(dk2), static_cast<const void *>(dv),
                            static_cast<const void *>(workspace)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    const bool f32 = dtype == DA_F32;
    for (int64_t st : {q_sb, q_st, q_sh, k_sb, k_st, k_sh, v_sb, v_st, v_sh, o_sb, o_st, o_sh})
        if (!stride_ok(st, f32 ? 4 : 2)) return DA_ERR_MISALIGNED;
    const int DV = 2 * d;
    const SavedLayout sl(B, T, H, DV, saved_esize(false, dtype));
    const BwdWsLayout wl(B, T, H, DV, true, f32 ? 4 : 2);
    if (saved_bytes < sl.total || workspace_bytes < wl.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    char *ws = static_cast<char *>(workspace);
    const char *sv = static_cast<const char *>(saved);
    if (f32) {
        SimtBwdParams p{};
        p.q1 = static_cast<const float *>(q1); p.q2 = static_cast<const float *>(q2);
        p.k1 = static_cast<const float *>(k1); p.k2 = static_cast<const float *>(k2);
        p.v = static_cast<const float *>(v);
        p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
        p.k_sb = k_sb; p.k_st = k_st; p.k_sh = k_sh;
        p.v_sb = v_sb; p.v_st = v_st; p.v_sh = v_sh;
        p.dout = static_cast<const float *>(dout);
        p.o_sb = o_sb; p.o_st = o_st; p.o_sh = o_sh;
        p.sa1 = reinterpret_cast<const float *>(sv);
        p.sa2 = reinterpret_cast<const float *>(sv + sl.off_a2);
        p.slse = reinterpret_cast<const float *>(sv + sl.off_lse);
        p.lq1 = lam_q1; p.lk1 = lam_k1; p.lq2 = lam_q2; p.lk2 = lam_k2;
        p.layer_index = layer_index;
        p.dq1 = static_cast<float *>(dq1); p.dq2 = static_cast<float *>(dq2);
        p.dk1 = static_cast<float *>(dk1); p.dk2 = static_cast<float *>(dk2);
        p.dv = static_cast<float *>(dv);
        p.dlq1 = dlam_q1; p.dlk1 = dlam_k1; p.dlq2 = dlam_q2; p.dlk2 = dlam_k2;
        p.gw = reinterpret_cast<float *>(ws + wl.off_g);
        p.g = p.gw;
        p.g_sh = DV; p.g_st = static_cast<int64_t>(H) * DV; p.g_sb = p.g_st * T;
        p.dd = reinterpret_cast<float *>(ws);
        p.cv = reinterpret_cast<float *>(ws + wl.off_c);
        p.dlam_rows = reinterpret_cast<float *>(ws + wl.off_rows);
        p.B = B; p.T = T; p.H = H; p.G = 1; p.Hkv = H; p.mode = 1;
        p.err = err;
        const da_status st = cuda_status(launch_simt_backward(p, d, DV, stream));
        if (st == DA_OK) t_last_launches = 4;
        return st;
    }
    __nv_bfloat16 *g = reinterpret_cast<__nv_bfloat16 *>(ws + wl.off_g);
    BwdMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uH = static_cast<uint64_t>(H), uB = static_cast<uint64_t>(B);
    const int64_t g_st = static_cast<int64_t>(H) * DV;
    bool okm = true;
    for (int rows : {128, 64}) {
        const bool r = rows == 128;
        okm = okm && encode_map_4d(r ? &m.q1r : &m.q1c, q1, d, uH, uT, uB, q_sh, q_st, q_sb, rows) &&
              encode_map_4d(r ? &m.q2r : &m.q2c, q2, d, uH, uT, uB, q_sh, q_st, q_sb, rows) &&
              encode_map_4d(r ? &m.k1r : &m.k1c, k1, d, uH, uT, uB, k_sh, k_st, k_sb, rows) &&
              encode_map_4d(r ? &m.k2r : &m.k2c, k2, d, uH, uT, uB, k_sh, k_st, k_sb, rows) &&
              encode_map_4d(r ? &m.vr : &m.vc, v, DV, uH, uT, uB, v_sh, v_st, v_sb, rows) &&
              encode_map_4d(r ? &m.gr : &m.gc, g, DV, uH, uT, uB, DV, g_st, g_st * T, rows);
    }
    if (!okm) return DA_ERR_CUDA;
    BwdPreParams pp{};
    pp.sa1 = sv;
    pp.sa2 = sv + sl.off_a2;
    pp.dout = static_cast<const __nv_bfloat16 *>(dout);
    pp.o_sb = o_sb; pp.o_st = o_st; pp.o_sh = o_sh;
    pp.layer_index = layer_index;
    pp.lq1 = lam_q1; pp.lk1 = lam_k1; pp.lq2 = lam_q2; pp.lk2 = lam_k2;
    pp.dlq1 = dlam_q1; pp.dlk1 = dlam_k1; pp.dlq2 = dlam_q2; pp.dlk2 = dlam_k2;
    pp.dlam_rows = reinterpret_cast<float *>(ws + wl.off_rows);
    pp.g = g;
    pp.dd = reinterpret_cast<float *>(ws);
    pp.cv = reinterpret_cast<float *>(ws + wl.off_c);
    pp.B = B; pp.T = T; pp.H = H; pp.d = d;
    pp.err = err;
    BwdParams p{};
    p.dq1 = static_cast<__nv_bfloat16 *>(dq1); p.dq2 = static_cast<__nv_bfloat16 *>(dq2);
    p.dk1 = static_cast<__nv_bfloat16 *>(dk1); p.dk2 = static_cast<__nv_bfloat16 *>(dk2);
    p.dv = static_cast<__nv_bfloat16 *>(dv);
    p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
    p.k_sb = k_sb; p.k_st = k_st; p.k_sh = k_sh;
    p.v_sb = v_sb; p.v_st = v_st; p.v_sh = v_sh;
    p.lse = reinterpret_cast<const float *>(sv + sl.off_lse);
    p.dd = pp.dd;
    p.cv = pp.cv;
    p.B = B; p.T = T; p.H = H; p.G = 1; p.Hkv = H;
    p.dqk_store = d;
    p.scale = 1.f / sqrtf(static_cast<float>(d));
    p.scale_log2 = 1.4426950408889634f * p.scale;
    p.err = err;
    const da_status st = cuda_status(launch_backward(m, p, pp, d, DV, false, stream));
    if (st == DA_OK) t_last_launches = d == 128 ? 5 : 4;
    return st;
}

da_status diffattn_v2_bwd(const void *q, const void *k, const void *v, const float *lam, const void *dout,
                          const void *saved, size_t saved_bytes, void *dq, void *dk, void *dv, float *dlam,
                          void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D,
                          da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !lam || !dout || !saved || !dq || !dk || !dv || !dlam || !workspace)
        return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || Hq < 2 || Hkv < 1) return DA_ERR_BAD_SHAPE;
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1)) return DA_ERR_BAD_GROUP;
    if (!train_supported(D, true, dtype)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {q, k, v, dout, saved, static_cast<const void *>(dq), static_cast<const void *>(dk),
                            static_cast<const void *>(dv), static_cast<const void *>(workspace)})
        if (!aligned16(ptr)) return DA_ERR_MISALIGNED;
    const int P = Hq / 2, G = Hq / Hkv;
    const SavedLayout sl(B, T, P, D, saved_esize(true, dtype));
    const BwdWsLayout wl(B, T, P, D, false, 4);
    if (saved_bytes < sl.total || workspace_bytes < wl.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    char *ws = static_cast<char *>(workspace);
    const char *sv = static_cast<const char *>(saved);
    if (dtype == DA_F32) {
        SimtBwdParams p{};
        p.q1 = p.q2 = static_cast<const float *>(q);
        p.k1 = p.k2 = static_cast<const float *>(k);
        p.v = static_cast<const float *>(v);
        const int64_t qst = static_cast<int64_t>(Hq) * D, kst = static_cast<int64_t>(Hkv) * D;
        const int64_t ost = static_cast<int64_t>(P) * D;
        p.q_sh = D; p.q_st = qst; p.q_sb = qst * T;
        p.k_sh = D; p.k_st = kst; p.k_sb = kst * T;
        p.v_sh = D; p.v_st = kst; p.v_sb = kst * T;
        p.dout = static_cast<const float *>(dout);
        p.o_sh = D; p.o_st = ost; p.o_sb = ost * T;
        p.g = p.dout;
        p.g_sh = D; p.g_st = ost; p.g_sb = ost * T;
        p.sa1 = reinterpret_cast<const float *>(sv);
        p.sa2 = reinterpret_cast<const float *>(sv + sl.off_a2);
        p.slse = reinterpret_cast<const float *>(sv + sl.off_lse);
        p.lam = lam;
        p.dq1 = p.dq2 = static_cast<float *>(dq);
        p.dk1 = p.dk2 = static_cast<float *>(dk);
        p.dv = static_cast<float *>(dv);
        p.dlam = dlam;
        p.dd = reinterpret_cast<float *>(ws);
        p.cv = reinterpret_cast<float *>(ws + wl.off_c);
        p.B = B; p.T = T; p.H = P; p.G = G; p.Hkv = Hkv; p.mode = 2;
        p.err = err;
        const da_status st = cuda_status(launch_simt_backward(p, D, D, stream));
        if (st == DA_OK) t_last_launches = 3;
        return st;
    }
    BwdMaps m;
    const uint64_t uT = static_cast<uint64_t>(T), uB = static_cast<uint64_t>(B);
    const int64_t qst = static_cast<int64_t>(Hq) * D, kst = static_cast<int64_t>(Hkv) * D;
    const int64_t ost = static_cast<int64_t>(P) * D;
    bool okm = true;
    for (int rows : {128, 64}) {
        const bool r = rows == 128;
        okm = okm && encode_map_4d(r ? &m.q1r : &m.q1c, q, D, Hq, uT, uB, D, qst, qst * T, rows) &&
              encode_map_4d(r ? &m.k1r : &m.k1c, k, D, Hkv, uT, uB, D, kst, kst * T, rows) &&
              encode_map_4d(r ? &m.vr : &m.vc, v, D, Hkv, uT, uB, D, kst, kst * T, rows) &&
              encode_map_4d(r ? &m.gr : &m.gc, dout, D, P, uT, uB, D, ost, ost * T, rows);
    }
    if (!okm) return DA_ERR_CUDA;
    m.q2r = m.q1r; m.q2c = m.q1c; m.k2r = m.k1r; m.k2c = m.k1c;
    BwdPreParams pp{};
    pp.sa1 = sv;
    pp.sa2 = sv + sl.off_a2;
    pp.dout = static_cast<const __nv_bfloat16 *>(dout);
    pp.o_sh = D; pp.o_st = ost; pp.o_sb = ost * T;
    pp.lam = lam;
    pp.dlam = dlam;
    pp.dd = reinterpret_cast<float *>(ws);
    pp.cv = reinterpret_cast<float *>(ws + wl.off_c);
    pp.B = B; pp.T = T; pp.H = P; pp.d = D;
    pp.err = err;
    BwdParams p{};
    p.dq1 = p.dq2 = static_cast<__nv_bfloat16 *>(dq);
    p.dk1 = p.dk2 = static_cast<__nv_bfloat16 *>(dk);
    p.dv = static_cast<__nv_bfloat16 *>(dv);
    p.q_sh = D; p.q_st = qst; p.q_sb = qst * T;
    p.k_sh = D; p.k_st = kst; p.k_sb = kst * T;
    p.v_sh = D; p.v_st = kst; p.v_sb = kst * T;
    p.lse = reinterpret_cast<const float *>(sv + sl.off_lse);
    p.dd = pp.dd;
    p.cv = pp.cv;
    p.B = B; p.T = T; p.H = P; p.G = G; p.Hkv = Hkv;
    p.dqk_store = D;
    p.scale = 1.f / sqrtf(static_cast<float>(D));
    p.scale_log2 = 1.4426950408889634f * p.scale;
    p.err = err;
    const da_status st = cuda_status(launch_backward(m, p, pp, D, D, true, stream));
    if (st == DA_OK) t_last_launches = 3;
    return st;
}

}  // extern "C"

// ------------------------------------------------------------ prologue

extern "C" da_status diffattn_prologue(void *q, void *k, int B, int T, int Hq, int Hk, int D, int64_t pos0,
                                       float base, const void *x, const void *w_lam, float *lam, int C, int P,
                                       da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if ((Hq > 0 && !q) || (Hk > 0 && !k) || (x && (!w_lam || !lam))) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || Hq < 0 || Hk < 0 || !(base > 0.f) || (x && (C < 1 || P < 1))) return DA_ERR_BAD_SHAPE;
    if (!prologue_supported(D, x ? C : 0, x ? P : 0)) return DA_ERR_UNSUPPORTED_DIM;
    for (const void *ptr : {static_cast<const void *>(q), static_cast<const void *>(k), x, w_lam})
        if (ptr && !aligned16(ptr)) return DA_ERR_MISALIGNED;
    if (lam && !aligned16(lam)) return DA_ERR_MISALIGNED;
    uint32_t *err = nullptr;
    int nsm = 0;
    if (!device_state(stream, &err, &nsm)) return DA_ERR_CUDA;
    t_last_launches = 0;
    if (Hq + Hk == 0 && !x) return DA_OK;   // nothing to do
    PrologueParams p{};
    p.q = Hq > 0 ? q : nullptr;
    p.k = Hk > 0 ? k : nullptr;
    p.Hq = Hq; p.Hk = Hk; p.D = D;
    p.x = x; p.w = w_lam; p.lam = lam;
    p.C = x ? C : 0; p.P = x ? P : 0;
    p.B = B; p.T = T;
    p.pos0 = pos0;
    p.base = static_cast<double>(base);
    p.err = err;
    const da_status st = cuda_status(launch_prologue(p, dtype == DA_BF16, stream));
    if (st == DA_OK) t_last_launches = (Hq + Hk > 0 ? 1 : 0) + (x ? 1 : 0);
    return st;
}

// ---------------------------------------------------------------------------
// Decode without allocation: the split-KV partials go to a buffer the library
// owns, so a caller that may not allocate device memory passes only inputs
// and outputs.  The buffer is a file-scope __device__ array; in host code its
// name is only a stand-in, so its device address is looked up per device with
// cudaGetSymbolAddress and that address is what the kernels receive.
namespace da {
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_ptr[64];

// Device address of this device's copy of g_noalloc_scratch; looked up on
// the first call per device, with that device current.
bool noalloc_scratch(void **p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return false;
        g_scratch_ptr[dev] = a;
    }
    *p = g_scratch_ptr[dev];
    return true;
}
}  // namespace
}  // namespace da

extern "C" da_status diffattn_v2_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                                const float *lam, void *out, int B, int L, int Hq, int Hkv,
                                                int D, da_dtype dtype, cudaStream_t stream) {
    // every argument check of the workspace entry point first, so that an
    // invalid call gets the same status there and here
    const da_status chk = v2_decode_check(q, k_cache, v_cache, lam, out, B, L, Hq, Hkv, D, dtype);
    if (chk != DA_OK) return chk;
    if (dtype == DA_F32)   // the fp32 kernel uses no scratch
        return diffattn_v2_decode(q, k_cache, v_cache, lam, out, nullptr, 0, B, L, Hq, Hkv, D, dtype, stream);
    int nsm = 0;
    int grid, spb;
    int64_t units;
    size_t cum = 0, need = 0;
    if (!device_state(nullptr, nullptr, &nsm)) return DA_ERR_CUDA;
    if (!decode_plan(B, L, Hkv, D, nsm, false, &grid, &units, &spb, &cum, &need)) return DA_ERR_BAD_SHAPE;
    if (need > kNoAllocScratchBytes) return DA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if (!noalloc_scratch(&scratch)) return DA_ERR_CUDA;
    return diffattn_v2_decode(q, k_cache, v_cache, lam, out, scratch, kNoAllocScratchBytes, B, L, Hq, Hkv, D,
                              dtype, stream);
}
