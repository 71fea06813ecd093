// k_decode.cu -- DIFF V2 decode (bf16): one new query token per sequence
// against an L-row KV cache.
//
// "Differential Transformer V2", DiffAttnV2 and the decoding remark after it:
// the query heads 2i and 2i+1 of one GQA group share kv head g = 2i/G, so a
// cache row is read once for all G query heads of its group; decoding is
// memory-bound.  out[b, i] = a_{2i} - sigmoid(lam[b, i]) a_{2i+1}.
//
// Design (HBM-bound: every K/V byte is read exactly once):
//   * Work is the flat list of 64-key units over (b, kv head, key block);
//     CTA c takes units [c N / grid, (c+1) N / grid) -- one CTA per SM,
//     balanced to within one unit.  A CTA's range covers a few (b, kv head)
//     segments; each segment yields one partial (m, l, o) per head.
//   * Warp 0 streams K and V units with TMA (128-byte swizzled 64x64 boxes)
//     into a STAGES-deep shared-memory ring.
//   * Warps 1..4 each take 16 keys of every unit.  Scores S^T (16 keys x 8
//     heads) = K Q^T with mma.sync m16n8k16 (the G <= 8 heads of the group are
//     the N = 8 columns); per-head online softmax in fp32 with warp shuffles;
//     P^T is turned into the B operand with movmatrix; O^T (D x 8) += V^T P^T
//     with ldmatrix.trans fragments.  The tensor-core work is ~8 flop/byte,
//     far below its rate; the loop is paced by HBM.
//   * At a segment end the four warps merge their (m, l, O^T) in shared memory
//     and write one partial.  A second kernel merges the partials of each
//     (b, kv head) and applies the sigmoid-gated pair subtraction.
#include <cfloat>

#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

template <int D>
struct DecCfg {
    static constexpr int KEYS = kDecodeKeysPerUnit;   // keys per unit / stage
    static constexpr int STAGES = 4;
    static constexpr int NBOX = D / 64;                // 64-element boxes per row
    static constexpr int BOX_BYTES = KEYS * 128;       // one 64 x 64 bf16 box
    static constexpr int TILE = KEYS * D * 2;          // K (or V) bytes per unit
    static constexpr int STAGE = 2 * TILE;
    static constexpr int NCW = 4;                      // consumer warps
    static constexpr int THREADS = 32 * (NCW + 1);
    static constexpr int XW = (D * 8 + 16) * 4;        // per-warp merge scratch
    static constexpr int OFF_XCH = STAGES * STAGE;
    static constexpr int OFF_BAR = OFF_XCH + NCW * XW;
    static constexpr int SMEM = OFF_BAR + 2 * STAGES * 8 + 1024;   // + alignment slack
    static constexpr int SLOT = 8 * D + 16;            // floats per partial slot
};

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    decode_split(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                 const DecodeParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t bar_full = sbase + C::OFF_BAR;           // STAGES x 8 bytes
    const uint32_t bar_empty = bar_full + C::STAGES * 8;    // STAGES x 8 bytes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t N = p.units;
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * N / p.grid;
    const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * N / p.grid;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            int64_t i = 0;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int st = static_cast<int>(i % C::STAGES);
                if (i >= C::STAGES &&
                    !mbar_wait(bar_empty + 8 * st, static_cast<uint32_t>((i / C::STAGES - 1) & 1), p.err))
                    break;
                const int64_t bg = u / p.spb;
                const int b = static_cast<int>(bg / p.Hkv), g = static_cast<int>(bg % p.Hkv);
                const int key0 = static_cast<int>(u % p.spb) * C::KEYS;
                const uint32_t sk = sbase + st * C::STAGE, sv = sk + C::TILE;
                mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE);
#pragma unroll
                for (int c = 0; c < C::NBOX; ++c) {
                    tma_load_4d(sk + c * C::BOX_BYTES, &tk, bar_full + 8 * st, c * 64, g, key0, b);
                    tma_load_4d(sv + c * C::BOX_BYTES, &tv, bar_full + 8 * st, c * 64, g, key0, b);
                }
            }
            // Leave no copy in flight: wait for the last fills issued.
            const int64_t first = i > C::STAGES ? i - C::STAGES : 0;
            for (int64_t k = first; k < i; ++k)
                mbar_wait(bar_full + 8 * static_cast<int>(k % C::STAGES),
                          static_cast<uint32_t>((k / C::STAGES) & 1), p.err);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int w = warp - 1;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[D / 16][4];
    uint32_t bq[D / 16][2];
    bool ok = true;
    int64_t cur_bg = -1;
    int seg = 0;
    float *xw = reinterpret_cast<float *>(smem + C::OFF_XCH);

    // Merge the four warps' (m, l, O^T) of the current segment into one partial.
    auto flush = [&](int segment) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
        float *mine = xw + w * (C::XW / 4);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = 16 * mt + g8;
            mine[d0 * 8 + 2 * t4] = o[mt][0];
            mine[d0 * 8 + 2 * t4 + 1] = o[mt][1];
            mine[(d0 + 8) * 8 + 2 * t4] = o[mt][2];
            mine[(d0 + 8) * 8 + 2 * t4 + 1] = o[mt][3];
        }
        if (g8 == 0) {
            mine[D * 8 + 2 * t4] = m0;
            mine[D * 8 + 2 * t4 + 1] = m1;
            mine[D * 8 + 8 + 2 * t4] = l0;
            mine[D * 8 + 8 + 2 * t4 + 1] = l1;
        }
        named_bar_sync(1, 32 * C::NCW);
        const int tid = w * 32 + lane;
        float *dst = p.ws + (static_cast<int64_t>(blockIdx.x) * p.max_seg + segment) * C::SLOT;
        for (int e = tid; e < D * 8; e += 32 * C::NCW) {
            const int n = e & 7, dd = e >> 3;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < C::NCW; ++ww) M = fmaxf(M, xw[ww * (C::XW / 4) + D * 8 + n]);
            const float Mb = (M == -INFINITY) ? 0.f : M;
            float acc = 0.f;
#pragma unroll
            for (int ww = 0; ww < C::NCW; ++ww) {
                const float *src = xw + ww * (C::XW / 4);
                acc = fmaf(src[dd * 8 + n], ex2(src[D * 8 + n] - Mb), acc);
            }
            dst[n * D + dd] = acc;
        }
        if (tid < 8) {
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < C::NCW; ++ww) M = fmaxf(M, xw[ww * (C::XW / 4) + D * 8 + tid]);
            const float Mb = (M == -INFINITY) ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int ww = 0; ww < C::NCW; ++ww) {
                const float *src = xw + ww * (C::XW / 4);
                L = fmaf(src[D * 8 + 8 + tid], ex2(src[D * 8 + tid] - Mb), L);
            }
            dst[8 * D + tid] = M;
            dst[8 * D + 8 + tid] = L;
        }
        named_bar_sync(1, 32 * C::NCW);
    };

    int64_t i = 0;
    for (int64_t u = u0; u < u1; ++u, ++i) {
        const int64_t bg = u / p.spb;
        if (bg != cur_bg) {
            if (cur_bg >= 0) flush(seg++);
            cur_bg = bg;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            // Q^T as the B operand: column n = head g*G + n of this group (zero past G).
            const int b = static_cast<int>(bg / p.Hkv), g = static_cast<int>(bg % p.Hkv);
            const bool valid = g8 < p.G;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                p.q + (static_cast<int64_t>(b) * p.Hq + g * p.G + (valid ? g8 : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                bq[ks][0] = valid ? qrow[(16 * ks + 2 * t4) >> 1] : 0u;
                bq[ks][1] = valid ? qrow[(16 * ks + 2 * t4 + 8) >> 1] : 0u;
            }
        }
        const int st = static_cast<int>(i % C::STAGES);
        ok = warp_wait(bar_full + 8 * st, static_cast<uint32_t>((i / C::STAGES) & 1), p.err, ok);
        if (!ok) continue;   // keep the flush sequence identical across warps
        const uint32_t sk = sbase + st * C::STAGE, sv = sk + C::TILE;

        // S^T[16 keys x 8 heads] = K[16 x D] * Q^T[D x 8]
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int krow = 16 * w + r8 + (mi & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int chunk = 2 * ks + (mi >> 1);
                const uint32_t addr = sk + (chunk >> 3) * C::BOX_BYTES + krow * 128 +
                                      (((chunk & 7) ^ (krow & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
                mma_16816(sc, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
            }
        }
        // mask keys past L, scale into log2 units
        const int key0 = static_cast<int>(u % p.spb) * C::KEYS + 16 * w + g8;
        const bool va = key0 < p.L, vb = key0 + 8 < p.L;
        const float x0 = va ? sc[0] * p.scale_log2 : -INFINITY;
        const float x1 = va ? sc[1] * p.scale_log2 : -INFINITY;
        const float x2 = vb ? sc[2] * p.scale_log2 : -INFINITY;
        const float x3 = vb ? sc[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int s = 4; s < 32; s <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, s));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, s));
        }
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float b0s = (n0 == -INFINITY) ? 0.f : n0, b1s = (n1 == -INFINITY) ? 0.f : n1;
        const float al0 = ex2(m0 - b0s), al1 = ex2(m1 - b1s);
        const float p0 = ex2(x0 - b0s), p1 = ex2(x1 - b1s), p2 = ex2(x2 - b0s), p3 = ex2(x3 - b1s);
        l0 = fmaf(l0, al0, p0 + p2);
        l1 = fmaf(l1, al1, p1 + p3);
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= al0;
            o[mt][2] *= al0;
            o[mt][1] *= al1;
            o[mt][3] *= al1;
        }
        // P^T as the B operand of O^T += V^T P^T
        const uint32_t pb0 = movmatrix_trans(pack_bf16(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16(p2, p3));
        {
            const int vrow = 16 * w + r8 + (mi >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int chunk = 2 * mt + (mi & 1);
                const uint32_t addr = sv + (chunk >> 3) * C::BOX_BYTES + vrow * 128 +
                                      (((chunk & 7) ^ (vrow & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(addr, a0, a1, a2, a3);
                mma_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    if (cur_bg >= 0) flush(seg);
}

// One CTA per (b, pair i), D threads: merge the partials of kv head g over the
// CTAs that covered it, normalise, apply out = a_even - sigmoid(lam) a_odd.
template <int D>
__global__ void __launch_bounds__(D) decode_combine(const DecodeParams p) {
    using C = DecCfg<D>;
    const int P = p.Hq / 2;
    const int b = blockIdx.x / P, i = blockIdx.x % P;
    const int he = 2 * i, ho = 2 * i + 1;
    const int g = he / p.G;
    const int ne = he % p.G, no = ho % p.G;
    const int64_t bg = static_cast<int64_t>(b) * p.Hkv + g;
    const int64_t N = p.units;
    auto cta_of = [&](int64_t u) -> int64_t { return ((u + 1) * p.grid - 1) / N; };
    auto first_unit = [&](int64_t c) -> int64_t { return c * N / p.grid; };
    const int64_t c_lo = cta_of(bg * p.spb), c_hi = cta_of(bg * p.spb + p.spb - 1);
    const int dd = threadIdx.x;
    float Me = -INFINITY, Mo = -INFINITY;
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        const int64_t seg = bg - first_unit(c) / p.spb;
        const float *src = p.ws + (c * p.max_seg + seg) * C::SLOT;
        Me = fmaxf(Me, src[8 * D + ne]);
        Mo = fmaxf(Mo, src[8 * D + no]);
    }
    float Le = 0.f, Lo = 0.f, Oe = 0.f, Oo = 0.f;
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        const int64_t seg = bg - first_unit(c) / p.spb;
        const float *src = p.ws + (c * p.max_seg + seg) * C::SLOT;
        const float we = ex2(src[8 * D + ne] - Me), wo = ex2(src[8 * D + no] - Mo);
        Le = fmaf(src[8 * D + 8 + ne], we, Le);
        Lo = fmaf(src[8 * D + 8 + no], wo, Lo);
        Oe = fmaf(src[ne * D + dd], we, Oe);
        Oo = fmaf(src[no * D + dd], wo, Oo);
    }
    const float sg = 1.f / (1.f + __expf(-p.lam[static_cast<int64_t>(b) * P + i]));
    const float y = Oe / Le - sg * (Oo / Lo);
    p.out[(static_cast<int64_t>(b) * P + i) * D + dd] = __float2bfloat16_rn(y);
}

template <int D>
cudaError_t launch_decode_t(const DecodeMaps &m, const DecodeParams &p, cudaStream_t s) {
    using C = DecCfg<D>;
    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_split<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    decode_split<D><<<p.grid, C::THREADS, C::SMEM, s>>>(m.k, m.v, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine<D><<<p.B * (p.Hq / 2), D, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool decode_plan(int B, int L, int Hq, int Hkv, int D, int num_sms, int *grid, int *max_seg,
                 int64_t *units, int *spb, size_t *ws_bytes) {
    if (B < 1 || L < 1 || Hq < 2 || Hkv < 1 || num_sms < 1) return false;
    if (D != 64 && D != 128) return false;
    const int s = (L + kDecodeKeysPerUnit - 1) / kDecodeKeysPerUnit;
    const int64_t n = static_cast<int64_t>(B) * Hkv * s;
    const int gr = static_cast<int>(n < num_sms ? n : num_sms);
    int ms = 1;
    for (int c = 0; c < gr; ++c) {
        const int64_t a = static_cast<int64_t>(c) * n / gr, e = static_cast<int64_t>(c + 1) * n / gr - 1;
        const int segs = static_cast<int>(e / s - a / s + 1);
        if (segs > ms) ms = segs;
    }
    *grid = gr;
    *max_seg = ms;
    *units = n;
    *spb = s;
    *ws_bytes = static_cast<size_t>(gr) * ms * (8 * D + 16) * sizeof(float);
    return true;
}

cudaError_t launch_decode(const DecodeMaps &m, const DecodeParams &p, cudaStream_t s) {
    if (p.D == 128) return launch_decode_t<128>(m, p, s);
    if (p.D == 64) return launch_decode_t<64>(m, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace da
