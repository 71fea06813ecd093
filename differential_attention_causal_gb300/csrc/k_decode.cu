// k_decode.cu -- single-token decode (bf16) against a KV cache: DIFF V2 and
// DIFF V1, every sequence attending all L cached rows or its own length.
//
// "Differential Transformer V2", DiffAttnV2 and the decoding remark after it:
// the query heads 2i and 2i+1 of one GQA group share kv head g = 2i/G, so a
// cache row is read once for all G query heads of its group; decoding is
// memory-bound.  out[b, i] = a_{2i} - sigmoid(lam[b, i]) a_{2i+1}.
// DiffAttnV1 for one new token: a1 = softmax(q1 K1^T / sqrt(d)) V and a2 the
// same with q2, K2; out = RMSNorm(a1 - lam a2) (1 - lam_init) over 2d channels.
//
// Design (HBM-bound: every K/V byte is read exactly once):
//   * Work is the flat list of 64-key units over (b, kv head, key block);
//     CTA c takes units [c N / grid, (c+1) N / grid) -- one CTA per SM,
//     balanced to within one unit.  With per-sequence lengths a small kernel
//     first writes the prefix of units per sequence, so the split stays
//     balanced however the lengths vary.  A CTA's range covers a few
//     (b, kv head) segments; each segment yields one partial (m, l, o) per
//     score column, in slot (b * Hkv + g) + cta (unique: along the unit order
//     both terms never decrease and at least one grows at every new segment).
//   * Warp 0 streams K and V units with TMA (128-byte swizzled 64x64 boxes)
//     into a shared-memory ring.
//   * Warps 1..4 each take 16 keys of every unit.  Scores S^T (16 keys x 8
//     columns) = K Q^T with mma.sync m16n8k16; per-column online softmax in
//     fp32 with warp shuffles; P^T is turned into the B operand with
//     movmatrix; O^T (D x 8) += V^T P^T with ldmatrix.trans fragments.  The
//     tensor-core work is ~8 flop/byte, far below its rate; HBM paces the loop.
//     V2: the columns are the G <= 8 query heads of the group.  V1: the K tile
//     is [k1 | k2] (2d channels) and the columns are [q1 | 0] and [0 | q2], so
//     column 0 scores q1 . k1 and column 1 scores q2 . k2 over the shared V.
//   * At a segment end the four warps merge their (m, l, O^T) in shared memory
//     and write one partial.  A second kernel merges the partials of each
//     (b, kv head) and applies the V2 gate or the V1 lambda / RMSNorm epilogue.
#include <cfloat>

#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

template <int D>
struct DecCfg {
    static constexpr int KEYS = kDecodeKeysPerUnit;   // keys per unit / stage
    static constexpr int STAGES = D >= 256 ? 3 : 4;    // D = 256: capped by shared memory
    static constexpr int NBOX = D / 64;                // 64-element boxes per row
    static constexpr int NBOX_LOG2 = NBOX == 1 ? 0 : (NBOX == 2 ? 1 : 2);
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
static_assert(DecCfg<256>::SMEM <= 232448, "decode ring exceeds the opt-in shared memory");

// Rows sequence b attends; lengths outside 1 .. L are clamped (and flagged by
// decode_prefix).
__device__ __forceinline__ int seq_len(const DecodeParams &p, int b) {
    if (!p.lens) return p.L;
    const int n = p.lens[b];
    return n < 1 ? 1 : (n > p.L ? p.L : n);
}
// First unit of sequence b, and the total.
__device__ __forceinline__ int64_t seq_first(const DecodeParams &p, int b) {
    return p.lens ? p.cum[b] : static_cast<int64_t>(b) * p.Hkv * p.spb;
}
__device__ __forceinline__ int64_t total_units(const DecodeParams &p) {
    return p.lens ? p.cum[p.B] : p.units;
}
// The sequence holding unit u: the last b with seq_first(b) <= u.
__device__ __forceinline__ int seq_of(const DecodeParams &p, int64_t u) {
    if (!p.lens) return static_cast<int>(u / (static_cast<int64_t>(p.Hkv) * p.spb));
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cum[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Walks the units of one CTA in order, tracking the sequence they belong to.
struct UnitCursor {
    int b, len, sb;          // sequence, its rows, its units per kv head
    int64_t first, end;      // its units [first, end)
    __device__ __forceinline__ void load(const DecodeParams &p, int bb) {
        b = bb;
        len = seq_len(p, bb);
        sb = (len + kDecodeKeysPerUnit - 1) / kDecodeKeysPerUnit;
        first = seq_first(p, bb);
        end = first + static_cast<int64_t>(p.Hkv) * sb;
    }
    __device__ __forceinline__ void seek(const DecodeParams &p, int64_t u) {
        while (u >= end && b + 1 < p.B) load(p, b + 1);
    }
};

// cum[b] = units of sequences 0 .. b-1 (B + 1 entries), one CTA of 1024.
__global__ void __launch_bounds__(1024) decode_prefix(const DecodeParams p) {
    __shared__ long long wsum[32];
    __shared__ long long carry_s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) {
        p.cum[0] = 0;
        carry_s = 0;
    }
    __syncthreads();
    for (int base = 0; base < p.B; base += 1024) {
        const int b = base + tid;
        long long x = 0;
        if (b < p.B) {
            const int n = p.lens[b];
            if (n < 1 || n > p.L) atomicOr(p.err, kErrBadLength);
            const int len = n < 1 ? 1 : (n > p.L ? p.L : n);
            x = static_cast<long long>(p.Hkv) * ((len + kDecodeKeysPerUnit - 1) / kDecodeKeysPerUnit);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            long long t = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            wsum[lane] = t;
        }
        __syncthreads();
        const long long incl = x + (w > 0 ? wsum[w - 1] : 0) + carry_s;
        if (b < p.B) p.cum[b + 1] = incl;
        __syncthreads();
        if (tid == 1023) carry_s = incl;
        __syncthreads();
    }
}

template <int D, bool V1>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    decode_split(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tk2,
                 const __grid_constant__ CUtensorMap tv, const DecodeParams p) {
    using C = DecCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t bar_full = sbase + C::OFF_BAR;           // STAGES x 8 bytes
    const uint32_t bar_empty = bar_full + C::STAGES * 8;    // STAGES x 8 bytes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t N = total_units(p);
    const int64_t u0 = static_cast<int64_t>(blockIdx.x) * N / p.grid;
    const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * N / p.grid;
    if (u0 >= u1) return;   // shorter sequences than L can leave a CTA without work

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    UnitCursor cu;
    cu.load(p, seq_of(p, u0));

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tk);
            if (V1) prefetch_tmap(&tk2);
            prefetch_tmap(&tv);
            int64_t i = 0;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int st = static_cast<int>(i % C::STAGES);
                if (i >= C::STAGES &&
                    !mbar_wait(bar_empty + 8 * st, static_cast<uint32_t>((i / C::STAGES - 1) & 1), p.err))
                    break;
                cu.seek(p, u);
                const int64_t local = u - cu.first;
                const int g = static_cast<int>(local / cu.sb);
                const int key0 = static_cast<int>(local % cu.sb) * C::KEYS;
                const uint32_t sk = sbase + st * C::STAGE, sv = sk + C::TILE;
                mbar_arrive_expect_tx(bar_full + 8 * st, C::STAGE);
#pragma unroll
                for (int c = 0; c < C::NBOX; ++c) {
                    if (V1 && c >= C::NBOX / 2)   // V1: channels d .. 2d-1 of the K tile are k2
                        tma_load_4d(sk + c * C::BOX_BYTES, &tk2, bar_full + 8 * st, (c - C::NBOX / 2) * 64, g,
                                    key0, cu.b);
                    else
                        tma_load_4d(sk + c * C::BOX_BYTES, &tk, bar_full + 8 * st, c * 64, g, key0, cu.b);
                    tma_load_4d(sv + c * C::BOX_BYTES, &tv, bar_full + 8 * st, c * 64, g, key0, cu.b);
                }
            }
            // Leave no copy in flight: wait for the last fills issued.
            const int64_t first = i > C::STAGES ? i - C::STAGES : 0;
            for (int64_t k = first; k < i; ++k)
                mbar_wait_drain(bar_full + 8 * static_cast<int>(k % C::STAGES),
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
    float *xw = reinterpret_cast<float *>(smem + C::OFF_XCH);

    // Merge the four warps' (m, l, O^T) of segment bg into its partial slot.
    auto flush = [&](int64_t bg) {
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
        float *dst = p.ws + (bg + blockIdx.x) * C::SLOT;
        // the partial slots: B * Hkv + grid - 1
        const bool in_ws = DA_CHECK(bg + blockIdx.x < static_cast<int64_t>(p.B) * p.Hkv + p.grid - 1, p.err);
        for (int e = tid; in_ws && e < D * 8; e += 32 * C::NCW) {
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
        if (tid < 8 && in_ws) {
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
        cu.seek(p, u);
        const int64_t local = u - cu.first;
        const int g = static_cast<int>(local / cu.sb);
        const int64_t bg = static_cast<int64_t>(cu.b) * p.Hkv + g;
        if (bg != cur_bg) {
            if (cur_bg >= 0) flush(cur_bg);
            cur_bg = bg;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            if (V1) {
                // column 0 = [q1 | 0], column 1 = [0 | q2]; q1, q2 rows at (b * H + h) * d
                constexpr int DQ = D / 2;
                // (d = p.dq may be less than DQ: the channels past it are zero, as in the
                // zero-filled k boxes)
                const uint32_t *q1r = reinterpret_cast<const uint32_t *>(p.q + bg * p.dq);
                const uint32_t *q2r = reinterpret_cast<const uint32_t *>(p.q2 + bg * p.dq);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c0 = 16 * ks + 2 * t4;
                    const bool lo_half = 16 * ks < DQ;
                    if (g8 == 0 && lo_half) {
                        bq[ks][0] = c0 < p.dq ? q1r[c0 >> 1] : 0u;
                        bq[ks][1] = c0 + 8 < p.dq ? q1r[(c0 + 8) >> 1] : 0u;
                    } else if (g8 == 1 && !lo_half) {
                        bq[ks][0] = c0 - DQ < p.dq ? q2r[(c0 - DQ) >> 1] : 0u;
                        bq[ks][1] = c0 - DQ + 8 < p.dq ? q2r[(c0 - DQ + 8) >> 1] : 0u;
                    } else {
                        bq[ks][0] = bq[ks][1] = 0u;
                    }
                }
            } else {
                // Q^T as the B operand: column n = head g*G + n of this group (zero past G).
                const bool valid = g8 < p.G;
                const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                    p.q + (static_cast<int64_t>(cu.b) * p.Hq + g * p.G + (valid ? g8 : 0)) * D);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    bq[ks][0] = valid ? qrow[(16 * ks + 2 * t4) >> 1] : 0u;
                    bq[ks][1] = valid ? qrow[(16 * ks + 2 * t4 + 8) >> 1] : 0u;
                }
            }
        }
        const int st = static_cast<int>(i % C::STAGES);
        ok = warp_wait(bar_full + 8 * st, static_cast<uint32_t>((i / C::STAGES) & 1), p.err, ok);
        if (!ok) continue;   // keep the flush sequence identical across warps
        const uint32_t sk = sbase + st * C::STAGE, sv = sk + C::TILE;
        const int ukey0 = static_cast<int>(local % cu.sb) * C::KEYS;

        // Rows of the last unit past this sequence's length may hold anything
        // (a longer sequence's cache area, uninitialised memory): zero their V
        // so that p = 0 cannot meet a NaN in the PV product.  K needs nothing:
        // those scores are replaced by -inf below.
        const bool tail = ukey0 + C::KEYS > cu.len;
        if (tail) {
            for (int e = lane; e < 16 * C::NBOX * 8; e += 32) {
                const int r = 16 * w + (e >> (3 + C::NBOX_LOG2));
                const int c = (e >> 3) & (C::NBOX - 1);
                if (ukey0 + r >= cu.len)
                    *reinterpret_cast<uint4 *>(smem + (sv - sbase) + c * C::BOX_BYTES + r * 128 + (e & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // S^T[16 keys x 8 columns] = K[16 x D] * Q^T[D x 8]
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
        // mask keys past the sequence length, scale into log2 units
        const int key0 = ukey0 + 16 * w + g8;
        const bool va = key0 < cu.len, vb = key0 + 8 < cu.len;
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
        // the zeroed rows were written through the generic proxy; order them
        // before the next TMA fill of this stage
        if (tail) fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
    if (cur_bg >= 0) flush(cur_bg);
}

__device__ __forceinline__ float block_sum(float x, float *red) {   // blockDim.x <= 256
    x = warp_sum(x);
    __syncthreads();   // red may still be read from the previous call
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float t = 0.f;
    for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) t += red[k];
    return t;
}

// One CTA per output row, D threads: merge the partials of (b, kv head g)
// over the CTAs that covered it, normalise both score columns, then
//   V2 (row (b, pair i), columns 2i % G and (2i+1) % G):
//       out = a_even - sigmoid(lam[b, i]) a_odd;
//   V1 (row (b, h), columns 0 and 1):
//       out = RMSNorm(a1 - lam a2) (1 - lam_init), lam from the lambda vectors.
template <int D, bool V1>
__global__ void __launch_bounds__(D) decode_combine(const DecodeParams p) {
    using C = DecCfg<D>;
    __shared__ float red[8];
    int b, g, ne, no;
    if (V1) {
        b = blockIdx.x / p.Hkv;
        g = blockIdx.x % p.Hkv;
        ne = 0;
        no = 1;
    } else {
        const int P = p.Hq / 2;
        b = blockIdx.x / P;
        const int i = blockIdx.x % P;
        g = (2 * i) / p.G;
        ne = (2 * i) % p.G;
        no = (2 * i + 1) % p.G;
    }
    const int64_t bg = static_cast<int64_t>(b) * p.Hkv + g;
    const int64_t N = total_units(p);
    const int sb = (seq_len(p, b) + kDecodeKeysPerUnit - 1) / kDecodeKeysPerUnit;
    const int64_t f = seq_first(p, b) + static_cast<int64_t>(g) * sb;
    // CTA c holds units [c N / grid, (c+1) N / grid); with fewer units than
    // CTAs (short sequences) some of those ranges are empty and wrote nothing.
    auto cta_of = [&](int64_t u) -> int64_t { return ((u + 1) * p.grid - 1) / N; };
    auto empty = [&](int64_t c) -> bool { return c * N / p.grid == (c + 1) * N / p.grid; };
    const int64_t c_lo = cta_of(f), c_hi = cta_of(f + sb - 1);
    const int dd = threadIdx.x;
    float Me = -INFINITY, Mo = -INFINITY;
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        if (empty(c)) continue;
        const float *src = p.ws + (bg + c) * C::SLOT;
        Me = fmaxf(Me, src[8 * D + ne]);
        Mo = fmaxf(Mo, src[8 * D + no]);
    }
    float Le = 0.f, Lo = 0.f, Oe = 0.f, Oo = 0.f;
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        if (empty(c)) continue;
        const float *src = p.ws + (bg + c) * C::SLOT;
        const float we = ex2(src[8 * D + ne] - Me), wo = ex2(src[8 * D + no] - Mo);
        Le = fmaf(src[8 * D + 8 + ne], we, Le);
        Lo = fmaf(src[8 * D + 8 + no], wo, Lo);
        Oe = fmaf(src[ne * D + dd], we, Oe);
        Oo = fmaf(src[no * D + dd], wo, Oo);
    }
    float y;
    if (V1) {
        // lam = exp(lq1 . lk1) - exp(lq2 . lk2) + lam_init, lam_init = 0.8 - 0.6 exp(-0.3 layer)
        const float d1 = block_sum(dd < p.dq ? p.lq1[dd] * p.lk1[dd] : 0.f, red);
        const float d2 = block_sum(dd < p.dq ? p.lq2[dd] * p.lk2[dd] : 0.f, red);
        const float lam_init = 0.8f - 0.6f * expf(-0.3f * static_cast<float>(p.layer_index));
        const float lam = expf(d1) - expf(d2) + lam_init;
        const float x = Oe / Le - lam * (Oo / Lo);
        const float ss = block_sum(x * x, red);
        // RMSNorm over the 2d channels (those past p.dv are zero), eps 1e-5, no
        // weight; then (1 - lam_init)
        y = x * ((1.f - lam_init) / sqrtf(ss / static_cast<float>(p.dv) + 1e-5f));
        if (dd < p.dv && DA_CHECK(blockIdx.x < static_cast<int64_t>(p.B) * p.Hq, p.err))
            p.out[static_cast<int64_t>(blockIdx.x) * p.dv + dd] = __float2bfloat16_rn(y);
    } else {
        const float sg = 1.f / (1.f + __expf(-p.lam[blockIdx.x]));
        y = Oe / Le - sg * (Oo / Lo);
        if (DA_CHECK(blockIdx.x < static_cast<int64_t>(p.B) * (p.Hq / 2), p.err))
            p.out[static_cast<int64_t>(blockIdx.x) * D + dd] = __float2bfloat16_rn(y);
    }
}

template <int D, bool V1>
cudaError_t launch_decode_t(const DecodeMaps &m, const DecodeParams &p, cudaStream_t s) {
    using C = DecCfg<D>;
    static unsigned long long attr_done = 0;   // one bit per device
    cudaError_t ea = once_per_device(&attr_done, [] {
        return cudaFuncSetAttribute(decode_split<D, V1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (ea != cudaSuccess) return ea;
    if (p.lens) {
        decode_prefix<<<1, 1024, 0, s>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    decode_split<D, V1><<<p.grid, C::THREADS, C::SMEM, s>>>(m.k, m.k2, m.v, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int rows = V1 ? p.B * p.Hkv : p.B * (p.Hq / 2);
    decode_combine<D, V1><<<rows, D, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool decode_plan(int B, int L, int Hkv, int D, int num_sms, bool varlen, int *grid, int64_t *units, int *spb,
                 size_t *cum_bytes, size_t *ws_bytes) {
    if (B < 1 || L < 1 || Hkv < 1 || num_sms < 1) return false;
    if (D != 64 && D != 128 && D != 256) return false;
    const int s = (L + kDecodeKeysPerUnit - 1) / kDecodeKeysPerUnit;
    const int64_t n = static_cast<int64_t>(B) * Hkv * s;   // all sequences at L rows: an upper bound
    const int gr = static_cast<int>(n < num_sms ? n : num_sms);
    const size_t cb = varlen ? ((static_cast<size_t>(B) + 1) * sizeof(int64_t) + 255) / 256 * 256 : 0;
    *grid = gr;
    *units = n;
    *spb = s;
    *cum_bytes = cb;
    *ws_bytes = cb + (static_cast<size_t>(B) * Hkv + gr - 1) * (8 * D + 16) * sizeof(float);
    return true;
}

cudaError_t launch_decode(const DecodeMaps &m, const DecodeParams &p, bool v1, cudaStream_t s) {
    if (v1) {
        if (p.D == 128) return launch_decode_t<128, true>(m, p, s);
        if (p.D == 256) return launch_decode_t<256, true>(m, p, s);
        return cudaErrorInvalidValue;
    }
    if (p.D == 128) return launch_decode_t<128, false>(m, p, s);
    if (p.D == 64) return launch_decode_t<64, false>(m, p, s);
    return cudaErrorInvalidValue;
}

}  // namespace da
