// k_simt_bwd.cu -- fp32 backward of the causal differential attention on
// CUDA cores (dtype DA_F32), DIFF V1 and DIFF V2.
//
// The same chain rule as the bf16 backward ("Differential Transformer V2",
// DiffAttnV1 / DiffAttnV2 differentiated): per branch b, with g_b the
// upstream gradient of a_b = softmax(S_b) V (g_2 = c g_1 row by row),
//     dP = g_1 . v_j,  dS_b = P_b (c_b dP - D_b),  D_b = g_b . a_b,
//     dQ_b = scale sum_j dS_b k_b,j,  dK_b = scale sum_i dS_b q_b,i,
//     dV = sum_i (P_1 + c P_2) g_1,i.
// P_b is recomputed from the scaled scores and the training forward's
// log-sum-exp (natural units).  One warp per row: bwd_simt_pre forms g_1,
// D_1, D_2, c and the lambda gradient; bwd_simt_dq walks the keys of one
// query row, bwd_simt_dkdv the queries of one key row (for V2 those of every
// pair in the key's GQA group).  Every sum is exact fp32 in a fixed order.
// This path exists for fp32 accuracy and small workloads, like the fp32
// forward; it is not the throughput path.
#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// One warp per row (b, t, h).  Lanes take channels lane + 32 i.
template <int DQK, int DV>
__global__ void __launch_bounds__(128) bwd_simt_pre(const SimtBwdParams p) {
    constexpr int NV = DV / 32;
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int64_t nrows = static_cast<int64_t>(p.B) * p.T * p.H;
    if (r >= nrows) return;
    const int h = static_cast<int>(r % p.H);
    const int t = static_cast<int>((r / p.H) % p.T);
    const int b = static_cast<int>(r / (static_cast<int64_t>(p.H) * p.T));
    if (!DA_CHECK(b < p.B && t < p.T && h < p.H, p.err)) return;
    const float *go = p.dout + b * p.o_sb + static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(h) * p.o_sh;
    const int64_t vi = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
    float x1[NV], x2[NV], dy[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        x1[i] = p.sa1[r * DV + lane + 32 * i];
        x2[i] = p.sa2[r * DV + lane + 32 * i];
        dy[i] = go[lane + 32 * i];
    }
    if (p.mode == 2) {
        // x1 = a_e, x2 = a_o; g_1 = dout, c = -sigmoid(lam[t])
        float e = 0.f, o = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            e = fmaf(dy[i], x1[i], e);
            o = fmaf(dy[i], x2[i], o);
        }
        e = wsum(e);
        o = wsum(o);
        if (lane == 0) {
            const float sg = 1.f / (1.f + expf(-p.lam[(static_cast<int64_t>(b) * p.T + t) * p.H + h]));
            p.dd[vi] = e;
            p.dd[nrows + vi] = -sg * o;
            p.cv[vi] = -sg;
            p.dlam[(static_cast<int64_t>(b) * p.T + t) * p.H + h] = -sg * (1.f - sg) * o;
        }
        return;
    }
    // V1: x1 = x (the RMSNorm input), x2 = a2; a1 = x + lam a2
    float s1 = 0.f, s2 = 0.f;
    for (int c = lane; c < DQK; c += 32) {
        s1 = fmaf(p.lq1[c], p.lk1[c], s1);
        s2 = fmaf(p.lq2[c], p.lk2[c], s2);
    }
    s1 = wsum(s1);
    s2 = wsum(s2);
    const float lam_init = 0.8f - 0.6f * expf(-0.3f * static_cast<float>(p.layer_index));
    const float lam = expf(s1) - expf(s2) + lam_init;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        ss = fmaf(x1[i], x1[i], ss);
        dy[i] *= (1.f - lam_init);
    }
    ss = wsum(ss);
    const float rr = 1.f / sqrtf(ss / static_cast<float>(DV) + 1e-5f);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) m = fmaf(dy[i], x1[i] * rr, m);
    m = wsum(m) / static_cast<float>(DV);
    float d1 = 0.f, d2 = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const float dx = rr * (dy[i] - x1[i] * rr * m);
        p.gw[r * DV + lane + 32 * i] = dx;
        d1 = fmaf(dx, fmaf(lam, x2[i], x1[i]), d1);
        d2 = fmaf(dx, x2[i], d2);
    }
    d1 = wsum(d1);
    d2 = wsum(d2);
    if (lane == 0) {
        p.dd[vi] = d1;
        p.dd[nrows + vi] = -lam * d2;
        p.cv[vi] = -lam;
        p.dlam_rows[r] = -d2;
    }
}

// One warp per query row (b, t, h): dQ_1, dQ_2 over keys 0 .. t.
template <int DQK, int DV>
__global__ void __launch_bounds__(128) bwd_simt_dq(const SimtBwdParams p) {
    constexpr int NQ = DQK / 32, NV = DV / 32;
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int64_t nrows = static_cast<int64_t>(p.B) * p.T * p.H;
    if (r >= nrows) return;
    const int h = static_cast<int>(r % p.H);
    const int t = static_cast<int>((r / p.H) % p.T);
    const int b = static_cast<int>(r / (static_cast<int64_t>(p.H) * p.T));
    if (!DA_CHECK(b < p.B && t < p.T && h < p.H, p.err)) return;
    const bool v2 = p.mode == 2;
    const int hq1 = v2 ? 2 * h : h, hq2 = v2 ? 2 * h + 1 : h, hk = v2 ? (2 * h) / p.G : h;
    const float scale = rsqrtf(static_cast<float>(DQK));
    const float *q1 = p.q1 + b * p.q_sb + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(hq1) * p.q_sh;
    const float *q2 = p.q2 + b * p.q_sb + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(hq2) * p.q_sh;
    const float *g = p.g + b * p.g_sb + static_cast<int64_t>(t) * p.g_st + static_cast<int64_t>(h) * p.g_sh;
    const int64_t vi = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
    const float lse1 = p.slse[vi], lse2 = p.slse[nrows + vi];
    const float dd1 = p.dd[vi], dd2 = p.dd[nrows + vi], cc = p.cv[vi];
    float qa[NQ], qb[NQ], ga[NV], dqa[NQ], dqb[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        qa[i] = q1[lane + 32 * i];
        qb[i] = q2[lane + 32 * i];
        dqa[i] = dqb[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) ga[i] = g[lane + 32 * i];
    const float *k1 = p.k1 + b * p.k_sb + static_cast<int64_t>(hk) * p.k_sh;
    const float *k2 = p.k2 + b * p.k_sb + static_cast<int64_t>(hk) * p.k_sh;
    const float *vv = p.v + b * p.v_sb + static_cast<int64_t>(hk) * p.v_sh;
    for (int j = 0; j <= t; ++j) {
        const float *kj1 = k1 + static_cast<int64_t>(j) * p.k_st;
        const float *kj2 = k2 + static_cast<int64_t>(j) * p.k_st;
        const float *vj = vv + static_cast<int64_t>(j) * p.v_st;
        float s1 = 0.f, s2 = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            s1 = fmaf(qa[i], kj1[lane + 32 * i], s1);
            s2 = fmaf(qb[i], kj2[lane + 32 * i], s2);
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) dp = fmaf(ga[i], vj[lane + 32 * i], dp);
        s1 = wsum(s1);
        s2 = wsum(s2);
        dp = wsum(dp);
        const float p1 = expf(s1 * scale - lse1), p2 = expf(s2 * scale - lse2);
        const float ds1 = p1 * (dp - dd1), ds2 = p2 * (cc * dp - dd2);
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            dqa[i] = fmaf(ds1, kj1[lane + 32 * i], dqa[i]);
            dqb[i] = fmaf(ds2, kj2[lane + 32 * i], dqb[i]);
        }
    }
    float *o1 = p.dq1 + b * p.q_sb + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(hq1) * p.q_sh;
    float *o2 = p.dq2 + b * p.q_sb + static_cast<int64_t>(t) * p.q_st + static_cast<int64_t>(hq2) * p.q_sh;
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        o1[lane + 32 * i] = dqa[i] * scale;
        o2[lane + 32 * i] = dqb[i] * scale;
    }
}

// One warp per key row (b, j, kv head): dK_1, dK_2 (V2: one dK) and dV over
// the queries j .. T-1 of every head (V1) or pair (V2) that reads this row.
template <int DQK, int DV>
__global__ void __launch_bounds__(128) bwd_simt_dkdv(const SimtBwdParams p) {
    constexpr int NQ = DQK / 32, NV = DV / 32;
    const int lane = threadIdx.x & 31;
    const bool v2 = p.mode == 2;
    const int nh = v2 ? p.Hkv : p.H;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int64_t nrows = static_cast<int64_t>(p.B) * p.T * nh;
    if (r >= nrows) return;
    const int hk = static_cast<int>(r % nh);
    const int j = static_cast<int>((r / nh) % p.T);
    const int b = static_cast<int>(r / (static_cast<int64_t>(nh) * p.T));
    if (!DA_CHECK(b < p.B && j < p.T && hk < nh, p.err)) return;
    const float scale = rsqrtf(static_cast<float>(DQK));
    const int64_t vrows = static_cast<int64_t>(p.B) * p.H * p.T;
    const float *kj1 = p.k1 + b * p.k_sb + static_cast<int64_t>(j) * p.k_st + static_cast<int64_t>(hk) * p.k_sh;
    const float *kj2 = p.k2 + b * p.k_sb + static_cast<int64_t>(j) * p.k_st + static_cast<int64_t>(hk) * p.k_sh;
    const float *vj = p.v + b * p.v_sb + static_cast<int64_t>(j) * p.v_st + static_cast<int64_t>(hk) * p.v_sh;
    float ka[NQ], kb[NQ], va[NV], dka[NQ], dkb[NQ], dva[NV];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        ka[i] = kj1[lane + 32 * i];
        kb[i] = kj2[lane + 32 * i];
        dka[i] = dkb[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        va[i] = vj[lane + 32 * i];
        dva[i] = 0.f;
    }
    const int np = v2 ? p.G / 2 : 1;
    for (int pi = 0; pi < np; ++pi) {
        const int hp = v2 ? hk * (p.G / 2) + pi : hk;
        const int hq1 = v2 ? 2 * hp : hp, hq2 = v2 ? 2 * hp + 1 : hp;
        for (int i = j; i < p.T; ++i) {
            const float *q1 = p.q1 + b * p.q_sb + static_cast<int64_t>(i) * p.q_st + static_cast<int64_t>(hq1) * p.q_sh;
            const float *q2 = p.q2 + b * p.q_sb + static_cast<int64_t>(i) * p.q_st + static_cast<int64_t>(hq2) * p.q_sh;
            const float *g = p.g + b * p.g_sb + static_cast<int64_t>(i) * p.g_st + static_cast<int64_t>(hp) * p.g_sh;
            const int64_t vi = (static_cast<int64_t>(b) * p.H + hp) * p.T + i;
            float qa[NQ], qb[NQ], ga[NV];
            float s1 = 0.f, s2 = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < NQ; ++c) {
                qa[c] = q1[lane + 32 * c];
                qb[c] = q2[lane + 32 * c];
                s1 = fmaf(qa[c], ka[c], s1);
                s2 = fmaf(qb[c], kb[c], s2);
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) {
                ga[c] = g[lane + 32 * c];
                dp = fmaf(ga[c], va[c], dp);
            }
            s1 = wsum(s1);
            s2 = wsum(s2);
            dp = wsum(dp);
            const float cc = p.cv[vi];
            const float p1 = expf(s1 * scale - p.slse[vi]), p2 = expf(s2 * scale - p.slse[vrows + vi]);
            const float ds1 = p1 * (dp - p.dd[vi]), ds2 = p2 * (cc * dp - p.dd[vrows + vi]);
            const float pt = fmaf(cc, p2, p1);
#pragma unroll
            for (int c = 0; c < NQ; ++c) {
                dka[c] = fmaf(ds1, qa[c], dka[c]);
                dkb[c] = fmaf(ds2, qb[c], dkb[c]);
            }
#pragma unroll
            for (int c = 0; c < NV; ++c) dva[c] = fmaf(pt, ga[c], dva[c]);
        }
    }
    float *o1 = p.dk1 + b * p.k_sb + static_cast<int64_t>(j) * p.k_st + static_cast<int64_t>(hk) * p.k_sh;
    float *o2 = p.dk2 + b * p.k_sb + static_cast<int64_t>(j) * p.k_st + static_cast<int64_t>(hk) * p.k_sh;
    float *ov = p.dv + b * p.v_sb + static_cast<int64_t>(j) * p.v_st + static_cast<int64_t>(hk) * p.v_sh;
#pragma unroll
    for (int c = 0; c < NQ; ++c) {
        if (v2) {
            o1[lane + 32 * c] = (dka[c] + dkb[c]) * scale;   // both branches read the one K
        } else {
            o1[lane + 32 * c] = dka[c] * scale;
            o2[lane + 32 * c] = dkb[c] * scale;
        }
    }
#pragma unroll
    for (int c = 0; c < NV; ++c) ov[lane + 32 * c] = dva[c];
}

template <int DQK, int DV>
cudaError_t launch_t(const SimtBwdParams &p, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(p.B) * p.T * p.H;
    const int64_t krows = static_cast<int64_t>(p.B) * p.T * (p.mode == 2 ? p.Hkv : p.H);
    const int64_t blocks = (rows + 3) / 4, kblocks = (krows + 3) / 4;
    if (blocks < 1 || blocks > 0x7fffffff || kblocks > 0x7fffffff) return cudaErrorInvalidValue;
    bwd_simt_pre<DQK, DV><<<static_cast<unsigned>(blocks), 128, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.mode == 1) {
        // dL/dlam from the row shares, then the four lambda-vector gradients
        BwdPreParams pp{};
        pp.dlam_rows = p.dlam_rows;
        pp.lq1 = p.lq1; pp.lk1 = p.lk1; pp.lq2 = p.lq2; pp.lk2 = p.lk2;
        pp.dlq1 = p.dlq1; pp.dlk1 = p.dlk1; pp.dlq2 = p.dlq2; pp.dlk2 = p.dlk2;
        pp.B = p.B; pp.T = p.T; pp.H = p.H; pp.d = DQK;
        pp.n_shares = rows;
        pp.err = p.err;
        e = launch_bwd_lambda(pp, s);
        if (e != cudaSuccess) return e;
    }
    bwd_simt_dq<DQK, DV><<<static_cast<unsigned>(blocks), 128, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_simt_dkdv<DQK, DV><<<static_cast<unsigned>(kblocks), 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_backward(const SimtBwdParams &p, int dqk, int dv, cudaStream_t s) {
    if (p.mode == 1 && dqk == 32 && dv == 64) return launch_t<32, 64>(p, s);
    if (p.mode == 1 && dqk == 64 && dv == 128) return launch_t<64, 128>(p, s);
    if (p.mode == 1 && dqk == 128 && dv == 256) return launch_t<128, 256>(p, s);
    if (p.mode == 2 && dqk == 64 && dv == 64) return launch_t<64, 64>(p, s);
    if (p.mode == 2 && dqk == 128 && dv == 128) return launch_t<128, 128>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace da
