// da_host.cu -- the DIFF V1 forward called with HOST buffers: the copies of
// the inputs in, the forward and the copy of the output back overlap, chunk
// by chunk of batch entries, instead of running one after the other.
//
//   copy stream in     H2D q, k, v of chunk 0 | chunk 1 | chunk 2 | ...
//   caller's stream               forward(0)  | forward(1) | ...
//   copy stream out                           | D2H out(0) | D2H out(1) ...
//
// Each forward waits for its chunk's inputs (an event), each copy out for its
// chunk's forward; the caller's stream finally waits for the last copy out,
// so the call is ordered on `stream` like any other.  The two copy streams
// are the library's own (one pair per device, created on first use); the
// enqueue of one call holds a per-device lock, so calls from several host
// threads are correct and share the copy engines in turn.  No kernel lives
// here: every chunk runs diffattn_v1_fwd on the device copies.
#include <mutex>

#include "da_internal.h"
#include "diffattn.h"

namespace da {
namespace {

constexpr int kMaxChunks = 8;
constexpr size_t kAlign = 256;

struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in[kMaxChunks] = {}, ev_fwd[kMaxChunks] = {};
    bool ready = false;
};
HostPipe g_pipe[64];
std::mutex g_pipe_mu[64];

bool make_pipe(HostPipe &h) {
    if (h.ready) return true;
    if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&h.ev_start, cudaEventDisableTiming) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&h.ev_end, cudaEventDisableTiming) != cudaSuccess) return false;
    for (int c = 0; c < kMaxChunks; ++c) {
        if (cudaEventCreateWithFlags(&h.ev_in[c], cudaEventDisableTiming) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&h.ev_fwd[c], cudaEventDisableTiming) != cudaSuccess) return false;
    }
    h.ready = true;
    return true;
}

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// device workspace: q | k | v | out | the four lambda vectors
struct HostLayout {
    size_t q, k, v, out, lam, total;
    HostLayout(int B, int T, int H, int d, int es) {
        const size_t qk = static_cast<size_t>(B) * T * 2 * H * d * es;   // (B, T, 2H, d)
        const size_t vo = static_cast<size_t>(B) * T * H * 2 * d * es;   // (B, T, H, 2d)
        q = 0;
        k = q + round_up(qk);
        v = k + round_up(qk);
        out = v + round_up(vo);
        lam = out + round_up(vo);
        total = lam + round_up(4 * static_cast<size_t>(d) * sizeof(float));
    }
};

}  // namespace
}  // namespace da

using namespace da;

extern "C" {

size_t diffattn_v1_fwd_host_workspace_size(int B, int T, int H, int d, da_dtype dtype) {
    if (dtype != DA_F32 && dtype != DA_BF16) return 0;
    if (B < 1 || T < 1 || H < 1 || d < 1) return 0;
    return HostLayout(B, T, H, d, dtype == DA_BF16 ? 2 : 4).total;
}

da_status diffattn_v1_fwd_host(const void *q, const void *k, const void *v, const float *lam_q1,
                               const float *lam_k1, const float *lam_q2, const float *lam_k2, void *out, int B,
                               int T, int H, int d, int layer_index, void *workspace, size_t workspace_bytes,
                               da_dtype dtype, cudaStream_t stream) {
    if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_BAD_DTYPE;
    if (!q || !k || !v || !lam_q1 || !lam_k1 || !lam_q2 || !lam_k2 || !out || !workspace) return DA_ERR_NULL_PTR;
    if (B < 1 || T < 1 || H < 1 || layer_index < 0) return DA_ERR_BAD_SHAPE;
    if (d != 32 && d != 64 && d != 128) return DA_ERR_UNSUPPORTED_DIM;
    const int es = dtype == DA_BF16 ? 2 : 4;
    const HostLayout L(B, T, H, d, es);
    if (workspace_bytes < L.total) return DA_ERR_WORKSPACE_TOO_SMALL;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DA_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_pipe_mu[dev]);
    HostPipe &hp = g_pipe[dev];
    if (!make_pipe(hp)) return DA_ERR_CUDA;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *dq = ws + L.q, *dk = ws + L.k, *dv = ws + L.v, *dout = ws + L.out;
    float *dlam = reinterpret_cast<float *>(ws + L.lam);
    const int64_t qk_sb = static_cast<int64_t>(T) * 2 * H * d, vo_sb = static_cast<int64_t>(T) * H * 2 * d;
    const size_t qk_b = static_cast<size_t>(qk_sb) * es, vo_b = static_cast<size_t>(vo_sb) * es;
    const int nch = B < kMaxChunks ? B : kMaxChunks;

    auto cuda = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = cuda(cudaEventRecord(hp.ev_start, stream)) && cuda(cudaStreamWaitEvent(hp.in, hp.ev_start, 0)) &&
              cuda(cudaStreamWaitEvent(hp.out, hp.ev_start, 0));
    // the lambda vectors, then each chunk's q, k, v
    const float *lams[4] = {lam_q1, lam_k1, lam_q2, lam_k2};
    for (int i = 0; ok && i < 4; ++i)
        ok = cuda(cudaMemcpyAsync(dlam + static_cast<size_t>(i) * d, lams[i], d * sizeof(float),
                                  cudaMemcpyHostToDevice, hp.in));
    int b0s[kMaxChunks + 1];
    for (int c = 0; c <= nch; ++c) b0s[c] = static_cast<int>(static_cast<int64_t>(B) * c / nch);
    for (int c = 0; ok && c < nch; ++c) {
        const size_t o_qk = static_cast<size_t>(b0s[c]) * qk_b, n_qk = static_cast<size_t>(b0s[c + 1] - b0s[c]) * qk_b;
        const size_t o_v = static_cast<size_t>(b0s[c]) * vo_b, n_v = static_cast<size_t>(b0s[c + 1] - b0s[c]) * vo_b;
        ok = cuda(cudaMemcpyAsync(dq + o_qk, static_cast<const uint8_t *>(q) + o_qk, n_qk, cudaMemcpyHostToDevice, hp.in)) &&
             cuda(cudaMemcpyAsync(dk + o_qk, static_cast<const uint8_t *>(k) + o_qk, n_qk, cudaMemcpyHostToDevice, hp.in)) &&
             cuda(cudaMemcpyAsync(dv + o_v, static_cast<const uint8_t *>(v) + o_v, n_v, cudaMemcpyHostToDevice, hp.in)) &&
             cuda(cudaEventRecord(hp.ev_in[c], hp.in));
    }
    // forward of each chunk on the caller's stream, its output copied back on the other copy stream
    da_status st = ok ? DA_OK : DA_ERR_CUDA;
    int launches = 0;
    for (int c = 0; st == DA_OK && c < nch; ++c) {
        const int bc = b0s[c + 1] - b0s[c];
        const size_t o_qk = static_cast<size_t>(b0s[c]) * qk_b, o_v = static_cast<size_t>(b0s[c]) * vo_b;
        if (!cuda(cudaStreamWaitEvent(stream, hp.ev_in[c], 0))) { st = DA_ERR_CUDA; break; }
        // q1 = heads 0::2 and q2 = heads 1::2 of the interleaved (T, 2H, d) rows; likewise k
        st = diffattn_v1_fwd(dq + o_qk, dq + o_qk + static_cast<size_t>(d) * es, dk + o_qk,
                             dk + o_qk + static_cast<size_t>(d) * es, dv + o_v, dlam, dlam + d, dlam + 2 * d,
                             dlam + 3 * d, dout + o_v, bc, T, H, d, layer_index, qk_sb, 2 * H * d, 2 * d, qk_sb,
                             2 * H * d, 2 * d, vo_sb, H * 2 * d, 2 * d, vo_sb, H * 2 * d, 2 * d, dtype, stream);
        if (st != DA_OK) break;
        launches += diffattn_last_launch_count();
        if (!(cuda(cudaEventRecord(hp.ev_fwd[c], stream)) && cuda(cudaStreamWaitEvent(hp.out, hp.ev_fwd[c], 0)) &&
              cuda(cudaMemcpyAsync(static_cast<uint8_t *>(out) + o_v, dout + o_v, static_cast<size_t>(bc) * vo_b,
                                   cudaMemcpyDeviceToHost, hp.out))))
            st = DA_ERR_CUDA;
    }
    // the call ends on `stream` when the last output bytes are in host memory
    // (also after an error, so that nothing enqueued here outlives the call's order)
    const bool joined = cuda(cudaEventRecord(hp.ev_end, hp.out)) && cuda(cudaStreamWaitEvent(stream, hp.ev_end, 0));
    set_last_launches(st == DA_OK ? launches : 0);
    if (st != DA_OK) return st;
    return joined ? DA_OK : DA_ERR_CUDA;
}

}  // extern "C"
