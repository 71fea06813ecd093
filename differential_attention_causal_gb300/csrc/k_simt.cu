// k_simt.cu -- fp32 differential attention on CUDA cores (dtype DA_F32).
//
// "Differential Transformer V2", DiffAttnV1 / DiffAttnV2: both branches are
// plain causal softmax attentions; V1 combines them as
// RMSNorm(a1 - lam a2) (1 - lam_init), V2 as a1 - sigmoid(lam) a2.
//
// One warp owns one output row and walks the keys 32 at a time: lane j forms
// the scores of key j0 + j (its own dot products, q from shared memory), the
// chunk's max and sum are two warp reductions per branch, and the exact online
// softmax update (running max m, running sum l, rescaled accumulator) then
// adds the chunk's P V with lanes over the value channels (p_j broadcast by a
// shuffle).  This path exists for fp32 accuracy (the tf32 tensor-core rate
// would not hold a 1e-4 bound after the RMSNorm) and for the small fp32
// workloads; it is not the throughput path.
#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(128) simt_fwd(SimtParams p) {
    constexpr int NQ = DQK / 32;   // q/k elements per lane
    constexpr int NV = DV / 32;    // v/out elements per lane
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int64_t nrows = static_cast<int64_t>(p.B) * p.Tq * p.H;
    if (row >= nrows) return;
    // an earlier kernel gave up: do not compute (decided for the whole warp)
    if (__any_sync(0xffffffffu, (ld_volatile_u32(p.err) & kErrFatal) != 0)) {
        if (lane == 0) atomicOr(p.err, kErrAborted);
        return;
    }
    const int h = static_cast<int>(row % p.H);
    const int t = static_cast<int>((row / p.H) % p.Tq);
    const int b = static_cast<int>(row / (static_cast<int64_t>(p.H) * p.Tq));
    if (!DA_CHECK(b < p.B && t < p.Tq && h < p.H, p.err)) return;

    // Head selection: V1 diff head h reads q1/k1 and q2/k2 at head h and v at
    // head h; V2 pair h reads query heads 2h (kept) and 2h+1 (subtracted) and
    // kv head 2h / G (heads of one GQA group are contiguous).
    int hq1, hq2, hk;
    if (p.mode == 1) { hq1 = h; hq2 = h; hk = h; }
    else { hq1 = 2 * h; hq2 = 2 * h + 1; hk = (2 * h) / p.G; }

    const float *q1 = p.q1 + b * p.q_sb + t * p.q_st + hq1 * p.q_sh;
    const float *q2 = p.q2 + b * p.q_sb + t * p.q_st + hq2 * p.q_sh;
    const float *k1 = p.k1 + b * p.k_sb + hk * p.k_sh;
    const float *k2 = p.k2 + b * p.k_sb + hk * p.k_sh;
    const float *vv = p.v + b * p.v_sb + hk * p.v_sh;

    // this row's q1, q2 in shared memory: every lane reads all channels
    __shared__ __align__(16) float qsh[4][2][DQK];
    const int w = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        qsh[w][0][lane + 32 * i] = q1[lane + 32 * i];
        qsh[w][1][lane + 32 * i] = q2[lane + 32 * i];
    }
    __syncwarp();
    const float4 *qa4 = reinterpret_cast<const float4 *>(qsh[w][0]);
    const float4 *qb4 = reinterpret_cast<const float4 *>(qsh[w][1]);
    const float scale = rsqrtf(static_cast<float>(DQK));
    float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
    float o1[NV], o2[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) { o1[i] = 0.f; o2[i] = 0.f; }

    // keys 0 .. t + (Lk - Tq), or for decode with per-sequence lengths the
    // first lens[b] cached rows (clamped into 1 .. Lk)
    int nkeys = t + (p.Lk - p.Tq) + 1;
    if (p.lens) {
        const int n = p.lens[b];
        if (n < 1 || n > p.Lk) {
            if (lane == 0) atomicOr(p.err, kErrBadLength);
            nkeys = n < 1 ? 1 : p.Lk;
        } else {
            nkeys = n;
        }
    }
    for (int j0 = 0; j0 < nkeys; j0 += 32) {
        // scores of keys j0 .. j0 + 31, one per lane (past the last key: -inf)
        const int j = j0 + lane;
        float s1 = -INFINITY, s2 = -INFINITY;
        if (j < nkeys) {
            const float4 *kj1 = reinterpret_cast<const float4 *>(k1 + static_cast<int64_t>(j) * p.k_st);
            const float4 *kj2 = reinterpret_cast<const float4 *>(k2 + static_cast<int64_t>(j) * p.k_st);
            float d1 = 0.f, d2 = 0.f;
#pragma unroll 8
            for (int c4 = 0; c4 < DQK / 4; ++c4) {
                const float4 x = kj1[c4], y = kj2[c4], qa = qa4[c4], qb = qb4[c4];
                d1 = fmaf(qa.x, x.x, d1); d1 = fmaf(qa.y, x.y, d1); d1 = fmaf(qa.z, x.z, d1); d1 = fmaf(qa.w, x.w, d1);
                d2 = fmaf(qb.x, y.x, d2); d2 = fmaf(qb.y, y.y, d2); d2 = fmaf(qb.z, y.z, d2); d2 = fmaf(qb.w, y.w, d2);
            }
            s1 = d1 * scale;
            s2 = d2 * scale;
        }
        const float n1 = fmaxf(m1, warp_max(s1)), n2 = fmaxf(m2, warp_max(s2));
        const float a1 = expf(m1 - n1), a2 = expf(m2 - n2);   // 0 on the first chunk
        const float p1 = j < nkeys ? expf(s1 - n1) : 0.f, p2 = j < nkeys ? expf(s2 - n2) : 0.f;
        l1 = l1 * a1 + warp_sum(p1);
        l2 = l2 * a2 + warp_sum(p2);
        m1 = n1;
        m2 = n2;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            o1[i] *= a1;
            o2[i] *= a2;
        }
        // O_b += sum_j p_j v_j over the chunk's keys, lanes over the channels;
        // eight keys' value rows are loaded before they are used, so that
        // their loads are in flight together
        const int jn = nkeys - j0 < 32 ? nkeys - j0 : 32;
        for (int g = 0; g < jn; g += 8) {
            float vx[8][NV];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float *vj = vv + static_cast<int64_t>(j0 + g + u) * p.v_st;
#pragma unroll
                for (int i = 0; i < NV; ++i) vx[u][i] = g + u < jn ? vj[lane + 32 * i] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                // keys past the chunk's last have p = 0 and v = 0: adding them changes nothing
                const float pa = __shfl_sync(0xffffffffu, p1, g + u), pb = __shfl_sync(0xffffffffu, p2, g + u);
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    o1[i] = fmaf(pa, vx[u][i], o1[i]);
                    o2[i] = fmaf(pb, vx[u][i], o2[i]);
                }
            }
        }
    }

    float *out = p.out + b * p.o_sb + t * p.o_st + h * p.o_sh;
    // training forward: saved tensors of this row for the backward
    const bool train = p.sa1 != nullptr;
    const int64_t srow = ((static_cast<int64_t>(b) * p.Tq + t) * p.H + h) * DV;
    if (train && lane == 0) {
        const int64_t li = (static_cast<int64_t>(b) * p.H + h) * p.Tq + t;
        p.slse[li] = m1 + logf(l1);
        p.slse[static_cast<int64_t>(p.B) * p.H * p.Tq + li] = m2 + logf(l2);
    }
    if (p.mode == 1) {
        // lam = exp(lq1 . lk1) - exp(lq2 . lk2) + lam_init ; lam_init = 0.8 - 0.6 exp(-0.3 layer)
        float d1 = 0.f, d2 = 0.f;
        for (int c = lane; c < DQK; c += 32) {
            d1 = fmaf(p.lq1[c], p.lk1[c], d1);
            d2 = fmaf(p.lq2[c], p.lk2[c], d2);
        }
        d1 = warp_sum(d1);
        d2 = warp_sum(d2);
        const float lam_init = 0.8f - 0.6f * expf(-0.3f * static_cast<float>(p.layer_index));
        const float lam = expf(d1) - expf(d2) + lam_init;
        const float i1 = 1.f / l1, i2 = lam / l2;
        float x[NV], ss = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            x[i] = o1[i] * i1 - o2[i] * i2;
            ss = fmaf(x[i], x[i], ss);
        }
        ss = warp_sum(ss);
        if (train) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                p.sa1[srow + lane + 32 * i] = x[i];
                p.sa2[srow + lane + 32 * i] = o2[i] / l2;
            }
        }
        // RMSNorm over the DV channels, eps 1e-5, no weight; then (1 - lam_init)
        const float r = (1.f - lam_init) / sqrtf(ss / static_cast<float>(DV) + 1e-5f);
#pragma unroll
        for (int i = 0; i < NV; ++i) out[lane + 32 * i] = x[i] * r;
    } else {
        const float lg = p.lam[b * p.lam_sb + t * p.lam_st + h];
        const float sg = 1.f / (1.f + expf(-lg));
        const float i1 = 1.f / l1, i2 = sg / l2;
#pragma unroll
        for (int i = 0; i < NV; ++i) out[lane + 32 * i] = o1[i] * i1 - o2[i] * i2;
        if (train) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                p.sa1[srow + lane + 32 * i] = o1[i] * i1;
                p.sa2[srow + lane + 32 * i] = o2[i] / l2;
            }
        }
    }
}

}  // namespace

cudaError_t launch_simt(const SimtParams &p, int dqk, int dv, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.Tq * p.H;
    const int64_t blocks = (rows + 3) / 4;
    if (blocks <= 0 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks)), block(128);
    if (dqk == 32 && dv == 64) simt_fwd<32, 64><<<grid, block, 0, s>>>(p);
    else if (dqk == 64 && dv == 128) simt_fwd<64, 128><<<grid, block, 0, s>>>(p);
    else if (dqk == 128 && dv == 256) simt_fwd<128, 256><<<grid, block, 0, s>>>(p);
    else if (dqk == 64 && dv == 64) simt_fwd<64, 64><<<grid, block, 0, s>>>(p);
    else if (dqk == 128 && dv == 128) simt_fwd<128, 128><<<grid, block, 0, s>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace da
