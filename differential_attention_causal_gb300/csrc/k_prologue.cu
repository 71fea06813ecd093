// k_prologue.cu -- the attention call's prologue in one pass over HBM:
// rotary position embedding of q and k in place, and DIFF V2's projected
// lambda logits.
//
// Rotary embedding as the nanoGPT issue applies it to q and k before the
// attention (RotaryEmbedding(dim = head_dim), apply_rotary_pos_emb), read as
// the rotate-half form with base 10000: for position p and i < D/2, with
// theta = p * base^(-2i/D), (x_i, x_{i+D/2}) -> (x_i cos - x_{i+D/2} sin,
// x_{i+D/2} cos + x_i sin).  "Differential Transformer V2": a projected lambda
// for each token and head, lam[n, i] = x[n, :] . w[:, i].
//
// Two kernels of 256 threads (q, k and x are disjoint, so one pass over each
// is all the fusion there is; the two need different shapes):
//   rotary, persistent (three CTAs per SM), blocks of TS = 16 tokens:
//   1. cos / sin of the block's positions (rope_cs, shared with the prefill's
//      in-place Q rotation): the angle is formed and reduced modulo 2 pi with
//      an extra float of precision (positions reach 10^5, where a plain float
//      product would already be off by ~1e-3 rad), the sine and cosine of
//      the reduced angle from the hardware approximations;
//   2. every (token, head, 8-pair chunk) of q and k: two 16-byte loads, the
//      rotation in fp32, two stores;
//   lambda, one CTA of 256 threads per 128 tokens:
//   3. the logits of the CTA's 128 tokens: bf16 on the tensor cores
//      (mma.sync, fp32 accumulators, x and w staged in shared memory 64
//      channels at a time), fp32 on CUDA cores (one warp per token).
// The work is HBM-bound (q and k read and written once, x read once); w
// stays in L2.
#include <cmath>

#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

constexpr int TB = 128;         // tokens per lambda CTA (16 per warp, 8 warps)
constexpr int LT = 256;         // threads of a lambda CTA
constexpr int TS = 16;          // tokens per rotary sub-block (one cos / sin table)
constexpr int MAXP = 64;        // lambda logits per token
// dynamic shared memory of the lambda kernel: LSTAGES x (TB x KC channels of
// x + KC rows of w, each P logits padded by 16 bytes)
constexpr int KC = 64;          // channels per stage of the lambda product
constexpr int LSTAGES = 4;      // 4 x 19.5 KB at P = 16: two CTAs per SM
__host__ __device__ constexpr int lstage(int P) { return TB * KC * 2 + KC * (P * 2 + 16); }
constexpr int SMEM_MAX = LSTAGES * lstage(MAXP);

template <typename E>
struct Vec8;                    // 8 elements <-> 8 floats
template <>
struct Vec8<__nv_bfloat16> {
    using Raw = uint4;   // the 8 elements as loaded, unpacked only when used
    static __device__ __forceinline__ Raw ld(const __nv_bfloat16 *p) { return *reinterpret_cast<const uint4 *>(p); }
    static __device__ __forceinline__ void unpack(const Raw &u, float *f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            f[2 * i] = a.x;
            f[2 * i + 1] = a.y;
        }
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *f) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            f[2 * i] = a.x;
            f[2 * i + 1] = a.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float *f) {
        *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                                   pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
    }
};
template <>
struct Vec8<float> {
    struct Raw {
        float4 a, b;
    };
    static __device__ __forceinline__ Raw ld(const float *p) {
        return Raw{*reinterpret_cast<const float4 *>(p), *reinterpret_cast<const float4 *>(p + 4)};
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float *f) {
        f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
        f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
    }
    static __device__ __forceinline__ void load(const float *p, float *f) {
        const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    static __device__ __forceinline__ void store(float *p, const float *f) {
        *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// base^(-2i/D) for the D/2 pairs, once per CTA, into shared memory
template <int D>
__device__ __forceinline__ void rope_freqs(double base, float *freq_hi, float *freq_lo) {
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) rope_freq(base, i, D, freq_hi[i], freq_lo[i]);
}

// Rotate every (token, head, 8-pair chunk) of q and k in tokens [t0, t0 + TS)
// for heads [h0, h1) of the Hq + Hk (q heads first, then k heads).  The cos /
// sin table of the block's TS tokens is stored [token][k][chunk] (entry
// i = 8 chunk + k at (token * 8 + k) * CH + chunk), so that the lanes of a
// warp, which take consecutive chunks, read consecutive entries.
template <typename E, int D>
__device__ __forceinline__ void rope_tokens(const PrologueParams &p, int64_t t0, int h0, int h1,
                                            float2 *cs, const float *freq_hi, const float *freq_lo) {
    constexpr int HALF = D / 2, CH = HALF / 8;
    const int64_t ntok = static_cast<int64_t>(p.B) * p.T;
    for (int e = threadIdx.x; e < TS * HALF; e += blockDim.x) {
        const int tt = e / HALF, i = e % HALF;
        const int64_t n = t0 + tt;
        float2 csv = make_float2(1.f, 0.f);
        if (n < ntok) csv = rope_cs(static_cast<float>(p.pos0 + n % p.T), freq_hi[i], freq_lo[i]);
        cs[(tt * 8 + i % 8) * CH + i / 8] = csv;
    }
    __syncthreads();
    const int heads = h1 - h0;
    const int units = TS * heads * CH;
    // U units per thread per round: all their loads are issued (and kept
    // packed) before the first rotation, so 2 U 16-byte reads are in flight
    // per thread
    constexpr int U = sizeof(E) == 2 ? 4 : 2;
    using Raw = typename Vec8<E>::Raw;
    for (int u0 = threadIdx.x; u0 < units; u0 += U * blockDim.x) {
        E *row[U];
        int tt[U], ch[U];
        Raw a[U], b[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int u = u0 + j * blockDim.x;
            row[j] = nullptr;
            ch[j] = u % CH;
            const int hh = h0 + (u / CH) % heads;
            tt[j] = u / (CH * heads);
            const int64_t n = t0 + tt[j];
            if (u < units && n < ntok && (hh < p.Hq ? p.q != nullptr : p.k != nullptr) &&
                DA_CHECK(hh < p.Hq + p.Hk && 8 * ch[j] + 8 <= HALF, p.err)) {
                row[j] = hh < p.Hq ? static_cast<E *>(p.q) + (n * p.Hq + hh) * D
                                   : static_cast<E *>(p.k) + (n * p.Hk + (hh - p.Hq)) * D;
                a[j] = Vec8<E>::ld(row[j] + 8 * ch[j]);
                b[j] = Vec8<E>::ld(row[j] + HALF + 8 * ch[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (!row[j]) continue;
            float fa[8], fb[8], ra[8], rb[8];
            Vec8<E>::unpack(a[j], fa);
            Vec8<E>::unpack(b[j], fb);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 t = cs[(tt[j] * 8 + k) * CH + ch[j]];
                rope_rotate(fa[k], fb[k], t.x, t.y, ra[k], rb[k]);
            }
            Vec8<E>::store(row[j] + 8 * ch[j], ra);
            Vec8<E>::store(row[j] + HALF + 8 * ch[j], rb);
        }
    }
    __syncthreads();   // cs is rewritten by the next sub-block
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    // the 256-byte L2 prefetch brings in the neighbouring 16-byte pieces of
    // the same row segment, which this CTA reads next
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// bf16 lambda logits of the block's TB tokens on the tensor cores:
// lam[tokens, :] = x[tokens, :] @ w, K in chunks of KC channels through an
// LSTAGES-deep ring of shared-memory buffers filled with cp.async (x rows
// 128-byte swizzled; w rows padded by 16 bytes so that ldmatrix reads them
// without bank conflicts), so several chunks are in flight per CTA.  Warp w
// owns tokens 16 w .. 16 w + 15 (8 warps); mma.sync m16n8k16 with fp32
// accumulators.
__device__ __forceinline__ void lambda_bf16(const PrologueParams &p, int64_t tok0, uint8_t *sm) {
    const int64_t ntok = static_cast<int64_t>(p.B) * p.T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wrow = p.P * 2 + 16;                         // padded w row, bytes
    const uint32_t sbase = smem_u32(sm);
    const int lst = lstage(p.P);
    auto xs = [&](int b) { return sbase + b * lst; };
    auto ws = [&](int b) { return sbase + b * lst + TB * KC * 2; };
    // x tile: rows of KC * 2 = 128 bytes, 16-byte chunk ch at
    // ((ch & 8) | ((ch & 7) ^ (row & 7))): ldmatrix's 8 rows hit 8 bank groups
    auto xoff = [](int row, int ch) { return row * (KC * 2) + (((ch & 8) | ((ch & 7) ^ (row & 7))) << 4); };
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(p.x);
    const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(p.w);
    const int wch = p.P / 8;                               // 16-byte chunks per w row
    const int nchunks = p.C / KC;
    auto issue = [&](int ci) {
        if (ci < nchunks) {
            const int c0 = ci * KC, b = ci % LSTAGES;
            for (int e = threadIdx.x; e < TB * (KC / 8); e += LT) {
                const int row = e / (KC / 8), ch = e % (KC / 8);
                const int64_t n = tok0 + row;
                cp_async16(xs(b) + xoff(row, ch), x + (n < ntok ? n : 0) * p.C + c0 + 8 * ch, n < ntok);
            }
            for (int e = threadIdx.x; e < KC * wch; e += LT) {
                const int row = e / wch, ch = e % wch;
                cp_async16(ws(b) + row * wrow + 16 * ch, w + static_cast<int64_t>(c0 + row) * p.P + 8 * ch, true);
            }
        }
        cp_async_commit();   // one group per chunk, empty past the end
    };
    float acc[MAXP / 8][4];
#pragma unroll
    for (int j = 0; j < MAXP / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int st = 0; st < LSTAGES - 1; ++st) issue(st);
    for (int ci = 0; ci < nchunks; ++ci) {
        cp_async_wait<LSTAGES - 2>();   // chunk ci has landed (this thread's copies)
        __syncthreads();                // ... and every thread's; buffer (ci - 1) is free
        issue(ci + LSTAGES - 1);
        const int b = ci % LSTAGES;
        const uint32_t xa = xs(b), wa = ws(b);
#pragma unroll
        for (int ks = 0; ks < KC / 16; ++ks) {
            const int row = 16 * warp + r8 + (mi & 1) * 8, chunk = 2 * ks + (mi >> 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(xa + xoff(row, chunk), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < MAXP / 16; ++np) {
                if (16 * np < p.P) {
                    // matrices (k 0-7 | 8-15) x (n 0-7 | 8-15) of this 16 x 16 block of w
                    const int kr = 16 * ks + (mi & 1) * 8 + r8, nc = 16 * np + (mi >> 1) * 8;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(wa + kr * wrow + nc * 2, b0, b1, b2, b3);
                    mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                    if (16 * np + 8 < p.P) mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
    }
    cp_async_wait<0>();
    // accumulator (16 tokens x 8 logits per tile): rows g, g + 8, columns 2 t, 2 t + 1
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int j = 0; j < MAXP / 8; ++j) {
        if (8 * j < p.P) {
            const int col = 8 * j + 2 * t4;
            const int64_t n0 = tok0 + 16 * warp + g, n1 = n0 + 8;
            if (!DA_CHECK(col + 2 <= p.P, p.err)) continue;
            if (n0 < ntok) *reinterpret_cast<float2 *>(p.lam + n0 * p.P + col) = make_float2(acc[j][0], acc[j][1]);
            if (n1 < ntok) *reinterpret_cast<float2 *>(p.lam + n1 * p.P + col) = make_float2(acc[j][2], acc[j][3]);
        }
    }
}

// fp32 lambda logits on CUDA cores: one warp per token, lanes over 8-channel chunks.
__device__ __forceinline__ void lambda_f32(const PrologueParams &p, int64_t tok0) {
    const int64_t ntok = static_cast<int64_t>(p.B) * p.T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *x = static_cast<const float *>(p.x);
    const float *w = static_cast<const float *>(p.w);
    for (int tt = warp; tt < TB; tt += LT / 32) {
        const int64_t n = tok0 + tt;
        if (n >= ntok) break;
        float acc[MAXP];
#pragma unroll
        for (int i = 0; i < MAXP; ++i) acc[i] = 0.f;
        for (int c0 = 8 * lane; c0 < p.C; c0 += 256) {
            float xv[8];
            Vec8<float>::load(x + n * p.C + c0, xv);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float *wr = w + static_cast<int64_t>(c0 + k) * p.P;
#pragma unroll
                for (int i0 = 0; i0 < MAXP; i0 += 8) {
                    if (i0 < p.P) {
                        float wv[8];
                        Vec8<float>::load(wr + i0, wv);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i0 + i] = fmaf(xv[k], wv[i], acc[i0 + i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < MAXP; ++i) {
            if (i < p.P) {
                const float v = warp_sum(acc[i]);
                if (lane == 0) p.lam[n * p.P + i] = v;
            }
        }
    }
}

// Rotary embedding: one CTA per TS tokens (one cos / sin table), all heads.
template <typename E, int D>
__global__ void __launch_bounds__(256, 3) prologue_rope(const PrologueParams p) {
    constexpr int HALF = D / 2;
    __shared__ float2 cs[TS * HALF];
    __shared__ float freq_hi[HALF], freq_lo[HALF];
    rope_freqs<D>(p.base, freq_hi, freq_lo);   // once per CTA
    __syncthreads();
    // persistent: the grid fills the GPU once and walks the token blocks
    const int64_t nblk = (static_cast<int64_t>(p.B) * p.T + TS - 1) / TS;
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x)
        rope_tokens<E, D>(p, blk * TS, 0, p.Hq + p.Hk, cs, freq_hi, freq_lo);
}

// Lambda logits: one CTA per TB tokens.
template <typename E>
__global__ void __launch_bounds__(LT) prologue_lambda(const PrologueParams p) {
    extern __shared__ __align__(16) uint8_t sm[];
    const int64_t tok0 = static_cast<int64_t>(blockIdx.x) * TB;
    if constexpr (sizeof(E) == 2) lambda_bf16(p, tok0, sm);
    else lambda_f32(p, tok0);
}

template <typename E>
cudaError_t launch_e(const PrologueParams &p, cudaStream_t s) {
    const int64_t ntok = static_cast<int64_t>(p.B) * p.T;
    if (p.q || p.k) {
        const int64_t blocks = (ntok + TS - 1) / TS;
        if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
        // three 256-thread CTAs per SM (the launch bound), one wave
        int dev = 0, nsm = 0;
        cudaError_t e0 = cudaGetDevice(&dev);
        if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e0 != cudaSuccess) return e0;
        const unsigned grid = static_cast<unsigned>(blocks < 3LL * nsm ? blocks : 3LL * nsm);
        if (p.D == 32) prologue_rope<E, 32><<<grid, 256, 0, s>>>(p);
        else if (p.D == 64) prologue_rope<E, 64><<<grid, 256, 0, s>>>(p);
        else if (p.D == 128) prologue_rope<E, 128><<<grid, 256, 0, s>>>(p);
        else return cudaErrorInvalidValue;
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.x) {
        static unsigned long long attr_done = 0;   // one bit per device
        const cudaError_t ea = once_per_device(&attr_done, [] {
            return cudaFuncSetAttribute(prologue_lambda<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        });
        if (ea != cudaSuccess) return ea;
        const int64_t blocks = (ntok + TB - 1) / TB;
        if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
        const int smem = sizeof(E) == 2 ? LSTAGES * lstage(p.P) : 0;   // the fp32 path stages nothing
        prologue_lambda<E><<<static_cast<unsigned>(blocks), LT, smem, s>>>(p);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

bool prologue_supported(int D, int C, int P) {
    const bool dim_ok = D == 32 || D == 64 || D == 128;
    // the bf16 product takes the channels KC = 64 at a time
    const bool proj_ok = C == 0 || (C % KC == 0 && P >= 8 && P <= MAXP && P % 8 == 0);
    return dim_ok && proj_ok;
}

cudaError_t launch_prologue(const PrologueParams &p, bool bf16, cudaStream_t s) {
    return bf16 ? launch_e<__nv_bfloat16>(p, s) : launch_e<float>(p, s);
}


}  // namespace da
