// k_prefill.cu -- fused causal differential-attention prefill on tcgen05
// tensor cores (bf16 in, fp32 accumulate), DIFF V1 and DIFF V2.
//
// "Differential Transformer V2": DiffAttnV1 computes two causal attentions
// attn_b = softmax(Q_b K_b^T / sqrt(d)) V over one shared V (2d wide) and
// returns RMSNorm(attn1 - lam attn2) (1 - lam_init); DiffAttnV2 runs one GQA
// attention whose even / odd query heads of a group share K and V and returns
// attn[:,0::2] - sigmoid(lam) attn[:,1::2].  Both are the same shape of work:
// two branches (Q1,K1) and (Q2,K2) against one V, combined per row at the end.
//
// Work tile = 128 query rows of one diff head (V1) or one head pair (V2).
// The kernel is persistent: one CTA per SM walks a snake-ordered list of work
// tiles, heaviest (most key tiles) first, so that every CTA gets the same
// amount of causal work and one tile's epilogue overlaps the next tile's
// loads and first products.
//   warp 0      TMA producer (converged, elected lane; lane 0 alone for
//               Paired Head Attention): Q1, Q2 per work tile (as soon as the previous
//               tile's last QK has been issued); K tiles (K1 and K2 for V1)
//               into a KS-deep ring and V tiles into a VS-deep ring, causal
//               tiles only, in the order the MMAs consume them.  K tile 0
//               completes on the Q tiles' barrier and K tile j + 1 on V tile
//               j's, so the MMA warp waits once per key tile for its operands
//               (measured on GB300: V1 d = 64 2 % faster than a K barrier of
//               its own).
//   warp 1      TMEM owner and MMA issuer (the whole warp runs the issue
//               loop converged; one lane chosen by elect.sync issues each
//               MMA and commit).
// The waits of these two roles and of the softmax warps are warp-uniform
// vote loops (warp_wait_vote), so those warps never run a divergent branch.
//   warp 2      V1: the lambda scalar (lam_init and the two exp terms) into
//               shared memory while the main loop runs.
//   warps 4-7   softmax for branch 1 (thread = query row = TMEM lane)
//   warps 8-11  softmax for branch 2
// TMEM (512 columns): S1 | S2 (128 fp32 columns each) | O1 | O2 (DV each).
// Per KV tile j the MMA warp issues   PV1(j) S1(j+1) ... PV2(j) S2(j+1):
//   S_b = Q_b K_b^T      (SS MMA, K-major operands, 128-byte swizzle)
//   P_b (bf16) is written by the softmax threads over the first 64 columns
//   of S_b in two key halves, and O_b += P_b V is a TS MMA (A = P from
//   TMEM, B = V MN-major), per half as it is published (V1) or once both
//   are (V2).
// While branch 1's threads exponentiate, the tensor core runs branch 2's
// products and vice versa.  The online softmax keeps a per-row reference
// max and rescales O only when the running max grows by more than 2^8; P
// stays below 2^8 and the final division by l uses the same reference, so
// the result is exact up to rounding.
// Epilogue (same kernel): x = O1/l1 - c O2/l2 with c = lam (V1) or
// sigmoid(lam[b,t,pair]) (V2); V1 then applies RMSNorm over the DV channels
// (eps 1e-5) and the (1 - lam_init) scale; the bf16 tile is staged in shared
// memory and written with TMA stores.
//
// Paired Head Attention (modded-nanogpt pull request "New Record: Paired Head
// Attention (-3.5s, -65 steps)", section "Updates in PR") runs on the same
// machinery (PAIRED, a V2-shaped instantiation): the keys and values of heads
// 2i and 2i+1 form one interleaved sequence of 2T positions (position 2t + e
// = token t of head 2i + e), which a 5-D tensor map reads directly as
// 64 tokens x 2 heads per 128-row key tile.  Branch e takes the queries of
// head 2i + e for 128 tokens, so both branches need the same key tiles
// (0 .. 2 qt + 1) and differ only in the causal limit of the last two: row r
// of branch e sees interleaved key columns c <= 2r + e - 128 (j - 2 qt).  The
// epilogue writes O_e / l_e of each branch to its own head with direct stores.
//
// Rotary embedding (ROPE, V2): when a work tile's Q tiles land, the two
// softmax threads of each row turn half of the row's channel pairs each, in
// shared memory, before the tile's first QK (see rope_q_row); the MMA warp
// then waits on a "Q rotated" barrier instead of "Q landed".
//
// L2: the Q tiles and the output are copied with an evict-first policy (read
// or written once), K and V with evict-last (every later query tile of the
// head reads them again), which keeps a head's K / V in L2 across its query
// tiles: the headline workload's DRAM traffic is within 3 % of its
// algorithmic bytes.
#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

template <int DQK, int DV, bool V2>
struct PreCfg {
    static constexpr int BM = 128, BN = 128;
    static constexpr int QB = DQK / 64;                // 64-column boxes per Q/K tile
    static constexpr int VB = DV / 64;
    static constexpr int BOX = 128 * 128;              // bytes of one 128-row x 64-col box
    static constexpr int Q_TILE = QB * BOX;
    static constexpr int K_TILE = QB * BOX;
    static constexpr int NK = V2 ? 1 : 2;              // K tiles per key block (K1, K2)
    static constexpr int K_SLOT = NK * K_TILE;
    static constexpr int V_SLOT = VB * BOX;
    static constexpr int OUT_TILE = VB * BOX;          // bf16 output tile staged for TMA stores
    // Ring depths when shared memory is short: V2 D = 128 2 / 2; V1 d = 64
    // K 3 / V 2 (measured on GB300 with the converged issuing warps: 0.4 %
    // faster than K 2 / V 3).
    static constexpr bool ROOMY = 2 * Q_TILE + 3 * (K_SLOT + V_SLOT) + OUT_TILE + 2048 <= 232448;
    static constexpr int KS = ROOMY ? 3 : (V2 ? 2 : 3);
    static constexpr int VS = ROOMY ? 3 : 2;
    static constexpr int OFF_Q1 = 0;
    static constexpr int OFF_Q2 = Q_TILE;
    static constexpr int OFF_K = 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * K_SLOT;
    static constexpr int OFF_OUT = OFF_V + VS * V_SLOT;
    // epilogue exchange of l (and for V1 the RMS partials): the first 2 KB of
    // the output staging tile, used before the tile is written
    static constexpr int OFF_X = OFF_OUT;
    static constexpr int OFF_BAR = OFF_OUT + OUT_TILE;
    // qfull, qfree, kfull[KS], kempty[KS], vfull[VS], vempty[VS], s[2], p[2][2], o[2], odrain, drain, lam,
    // staged, store-free, drain2, q rotated
    static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 2 + 4 + 2 + 7;
    static constexpr int OFF_LAM = OFF_BAR + NBAR * 8;        // 2 floats
    static constexpr int OFF_TSLOT = OFF_LAM + 8;
    static constexpr int OFF_FREQ = OFF_TSLOT + 8;            // rotary f_i as float pairs (DQK / 2 x 2)
    static constexpr int SMEM = OFF_FREQ + DQK * 4 + 1024;    // + alignment slack
    static constexpr int COL_S1 = 0, COL_S2 = BN, COL_O1 = 2 * BN, COL_O2 = 2 * BN + DV;
    static constexpr uint32_t TMEM_COLS = 512;
    // registers per thread after the split: warps 0-3 (producer, MMA,
    // lambda, idle) give up registers, the two softmax warpgroups take them
    static constexpr uint32_t REGS_LOW = 88, REGS_HIGH = 192;
    // measured on GB300 with the converged issuing warps: V1 and V2 both
    // faster with the split (V2 D = 128 4.7 %; before that change it cost V2)
    static constexpr bool REG_SPLIT = true;
    // the row max of keys 0-63 taken while keys 64-127 are still being read
    // out of TMEM (off the diagonal): measured on GB300 with the converged
    // issuing warps, V1 d = 64 1 % slower, V2 D = 128 2 % slower, so off
    static constexpr bool LD_SPLIT = false;
    // PV issued per key half as the softmax publishes each (P_HALVES) or once
    // both halves are published; measured on GB300: halves keep V1 d = 64 1-2 %
    // faster, the single wait makes V2 D = 128 and Paired Head Attention 2-4 %
    // faster (one barrier wait fewer per branch and key tile in the MMA warp)
    static constexpr bool P_HALVES = !V2;
    // one MMA-issuing warp per branch (warp 1: S1, O1; warp 2: S2, O2) instead
    // of one for both; measured on GB300 at the V1 d = 64 / V2 D = 128 prefill
    // shapes: 13 % / 25 % slower with lane-0 issuers, 19 % / 20 % slower with
    // converged ones, so off
    static constexpr bool TWO_ISSUERS = false;
    // the MMA issue loop run by all of warp 1, converged, each MMA and commit
    // issued by one lane chosen with elect.sync, instead of by lane 0 alone
    // (whose loop runs divergent from the rest of its warp), and the same for
    // the TMA producer (warp 0; not for Paired Head Attention, whose 5-D key
    // loads stay on lane 0).  Measured on GB300 with the vote-based waits:
    // V1 d = 64 2.7 % faster, V2 D = 128 0.7 % faster.
    static constexpr bool ELECT_ISSUE = true;
    static constexpr bool ELECT_LOAD = true;
    static constexpr uint32_t NISS = TWO_ISSUERS ? 2 : 1;     // arrivals on stage-release barriers
    static constexpr int REGS_NEEDED_AT_LAUNCH = (128 * REGS_LOW + 256 * REGS_HIGH + 383) / 384;
    static constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, true);
    static_assert(COL_O2 + DV <= 512, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

// p = 2^(s*scale - m) for 64 scores, in place as 32 packed bf16 pairs in
// s[0..31]; returns the fp32 sum of the 64 values.
__device__ __forceinline__ float exp_pack64(uint32_t *s, float scale, float m) {
    const float2 sc2 = make_float2(scale, scale);
    const float2 nm2 = make_float2(-m, -m);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const float2 x =
            __ffma2_rn(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nm2);
        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
        switch (c & 3) {
            case 0: acc0 = __fadd2_rn(acc0, pp); break;
            case 1: acc1 = __fadd2_rn(acc1, pp); break;
            case 2: acc2 = __fadd2_rn(acc2, pp); break;
            default: acc3 = __fadd2_rn(acc3, pp); break;
        }
        s[c] = pack_bf16(pp.x, pp.y);
    }
    const float2 t = __fadd2_rn(__fadd2_rn(acc0, acc1), __fadd2_rn(acc2, acc3));
    return t.x + t.y;
}

// Number of the k-th work tile of CTA c when G CTAs walk NT tiles in snake
// order (c, 2G-1-c, 2G+c, ...): consecutive rounds go in opposite directions,
// so with tiles sorted by decreasing weight every CTA's total is within one
// tile of the others.  Returns -1 past the end.
__device__ __forceinline__ int snake_tile(int k, int c, int G, int NT) {
    const int w = k * G + ((k & 1) ? (G - 1 - c) : c);
    return w < NT ? w : -1;
}

// Rotary embedding of one query row (position pos) of both Q tiles in shared
// memory (each DQK channels as DQK / 64 boxes of 128 rows x 128 bytes,
// 128-byte swizzle): the pairs (i, i + DQK/2) for i in this thread's half of
// the pairs (half 0: i < DQK/4, half 1: the rest), turned by the angle
// pos * f_i (f_i = fhi[i] + flo[i]), every value rounded back to bf16.
// 8-channel chunk c of the first half pairs with chunk c + DQK/16 at the same
// place in its group.  The two branches' threads of one row take the two
// halves, so each (cos, sin) is formed once per row and applied to both tiles.
template <int DQK>
__device__ __forceinline__ void rope_q_row(uint8_t *q1, uint8_t *q2, int row, int half, float pos,
                                           const float *fhi, const float *flo) {
    constexpr int NCH = DQK / 16;          // 8-channel chunks per half of the channels
    constexpr int MY = DQK / 32;           // chunks of this thread per tile
    constexpr int BOX = 128 * 128;
    auto at = [&](uint8_t *q, int c) { return q + (c >> 3) * BOX + row * 128 + (((c & 7) ^ (row & 7)) << 4); };
#pragma unroll 1
    for (int c = half * MY; c < half * MY + MY; ++c) {
        float2 cs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) cs[e] = rope_cs(pos, fhi[8 * c + e], flo[8 * c + e]);
#pragma unroll
        for (int tile = 0; tile < 2; ++tile) {
            uint4 *pa = reinterpret_cast<uint4 *>(at(tile ? q2 : q1, c));
            uint4 *pb = reinterpret_cast<uint4 *>(at(tile ? q2 : q1, c + NCH));
            const uint4 ua = *pa, ub = *pb;
            const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
            uint32_t ra[4], rb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wa[k]));
                const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wb[k]));
                float2 xa, xb;
                rope_rotate2(a, b, make_float2(cs[2 * k].x, cs[2 * k + 1].x), make_float2(cs[2 * k].y, cs[2 * k + 1].y),
                             xa, xb);
                ra[k] = pack_bf16(xa.x, xa.y);
                rb[k] = pack_bf16(xb.x, xb.y);
            }
            *pa = make_uint4(ra[0], ra[1], ra[2], ra[3]);
            *pb = make_uint4(rb[0], rb[1], rb[2], rb[3]);
        }
    }
}

template <int DQK, int DV, bool V2, bool TRAIN, bool PAIRED, bool ROPE>
__global__ void __launch_bounds__(384, 1)
    prefill_onepass(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tq2,
                    const __grid_constant__ CUtensorMap tk1, const __grid_constant__ CUtensorMap tk2,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tout,
                    const PrefillParams p) {
    using C = PreCfg<DQK, DV, V2>;
    static_assert(!PAIRED || (V2 && !TRAIN && DQK == DV), "paired heads: V2-shaped forward only");
    static_assert(!ROPE || (V2 && !TRAIN && !PAIRED), "rotated Q tiles: V2 forward only");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // work tiles: index w -> query tile n_qt-1-w/(H*B) (heaviest first), head, batch
    const int n_qt = (p.T + C::BM - 1) / C::BM;
    const int per_qt = p.H * p.B;
    const int NT = n_qt * per_qt;
    // key tiles of query tile qt: the causal ones; for paired heads the keys are
    // the interleaved sequence (two positions per token, 2T in all)
    const int n_kt = PAIRED ? (2 * p.T + C::BN - 1) / C::BN : n_qt;
    auto kv_tiles = [&](int qt) { return PAIRED ? min(2 * qt + 2, n_kt) : qt + 1; };
    const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);

    const uint32_t bar_qf = sbase + C::OFF_BAR;
    const uint32_t bar_qe = bar_qf + 8;                // Q tiles free (last QK of a tile issued)
    const uint32_t bar_kf = bar_qe + 8;                // [KS] (unused: K lands on the Q / V barriers)
    const uint32_t bar_ke = bar_kf + 8 * C::KS;        // [KS]
    const uint32_t bar_vf = bar_ke + 8 * C::KS;        // [VS]
    const uint32_t bar_ve = bar_vf + 8 * C::VS;        // [VS]
    const uint32_t bar_s = bar_ve + 8 * C::VS;         // [2]
    const uint32_t bar_p = bar_s + 16;                 // [2 branches][2 halves]
    const uint32_t bar_o = bar_p + 32;                 // [2]
    const uint32_t bar_od = bar_o + 16;                // O read by the epilogue (8 warps)
    const uint32_t bar_dr = bar_od + 8;
    const uint32_t bar_lam = bar_dr + 8;
    const uint32_t bar_stg = bar_lam + 8, bar_stf = bar_stg + 8;
    const uint32_t bar_dr2 = bar_stf + 8;              // drain of the second issuer
    const uint32_t bar_qr = bar_dr2 + 8;               // Q tiles rotated (8 softmax warps)
    const uint32_t tslot = sbase + C::OFF_TSLOT;
    const uint32_t sQ1 = sbase + C::OFF_Q1, sQ2 = sbase + C::OFF_Q2;
    float *lam_smem = reinterpret_cast<float *>(smem + C::OFF_LAM);

    if (threadIdx.x == 0) {
        mbar_init(bar_qf, 1);
        mbar_init(bar_qe, C::NISS);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, C::NISS);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(bar_vf + 8 * s, 1);
            mbar_init(bar_ve + 8 * s, C::NISS);
        }
        for (int br = 0; br < 2; ++br) {
            mbar_init(bar_s + 8 * br, 1);
            mbar_init(bar_p + 16 * br, 4);     // keys 0-63 of P: one arrival per softmax warp
            mbar_init(bar_p + 16 * br + 8, 4); // keys 64-127
            mbar_init(bar_o + 8 * br, 1);
        }
        mbar_init(bar_od, 8);
        mbar_init(bar_dr, 1);
        mbar_init(bar_lam, 1);
        mbar_init(bar_stg, 8);
        mbar_init(bar_stf, 1);
        mbar_init(bar_dr2, 1);
        mbar_init(bar_qr, 8);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::OFF_TSLOT);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (C::REG_SPLIT) regs_decrease<C::REGS_LOW>();
        constexpr bool kElectLoad = C::ELECT_LOAD && !PAIRED;
        if (kElectLoad || lane == 0) {
            // load primitives of this thread (lane 0) or of the converged warp
            auto wait_p = [&](uint32_t bar, uint32_t parity, uint32_t *err) -> bool {
                if constexpr (kElectLoad) return warp_wait_vote(bar, parity, err, true);
                else return mbar_wait(bar, parity, err);
            };
            auto expect_p = [&](uint32_t bar, uint32_t bytes) {
                if constexpr (kElectLoad) mbar_arrive_expect_tx_elect(bar, bytes);
                else mbar_arrive_expect_tx(bar, bytes);
            };
            auto load4_p = [&](uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1, int c2, int c3,
                               uint64_t pol) {
                if constexpr (kElectLoad) tma_load_4d_hint_elect(dst, m, bar, c0, c1, c2, c3, pol);
                else tma_load_4d_hint(dst, m, bar, c0, c1, c2, c3, pol);
            };
            prefetch_tmap(&tq1);
            prefetch_tmap(&tk1);
            prefetch_tmap(&tv);
            if (!V2) {
                prefetch_tmap(&tq2);
                prefetch_tmap(&tk2);
            }
            int kc = 0, vc = 0, tc = 0;   // ring and tile counters (the MMA warp keeps the same)
            bool ok = true;
            // Q tiles are read once; K and V tiles are read again by the other
            // query tiles of their head (from L2, if they are kept there)
            const uint64_t pol_once = l2_evict_first(), pol_reuse = l2_evict_last();
            // A K slot / V slot is free once the products that read its previous
            // contents have completed.
            auto k_free = [&]() {
                return kc < C::KS ||
                       wait_p(bar_ke + 8 * (kc % C::KS), static_cast<uint32_t>((kc / C::KS - 1) & 1), p.err);
            };
            auto v_free = [&]() {
                return vc < C::VS ||
                       wait_p(bar_ve + 8 * (vc % C::VS), static_cast<uint32_t>((vc / C::VS - 1) & 1), p.err);
            };
            // K tile j (K1 and K2 for V1) into the next K slot, completing on `bar`
            auto put_k = [&](int j, int hk, int b, uint32_t bar) {
                const uint32_t dst = sbase + C::OFF_K + (kc % C::KS) * C::K_SLOT;
#pragma unroll
                for (int c = 0; c < C::QB; ++c) {
                    if (PAIRED)   // 64 tokens x both heads of pair hk, interleaved
                        tma_load_5d(dst + c * C::BOX, &tk1, bar, 64 * c, 0, hk, j * (C::BN / 2), b);
                    else
                        load4_p(dst + c * C::BOX, &tk1, bar, 64 * c, hk, j * C::BN, b, pol_reuse);
                    if (!V2) load4_p(dst + C::K_TILE + c * C::BOX, &tk2, bar, 64 * c, hk, j * C::BN, b, pol_reuse);
                }
                ++kc;
            };
            auto put_v = [&](int j, int hk, int b, uint32_t bar) {
                const uint32_t dst = sbase + C::OFF_V + (vc % C::VS) * C::V_SLOT;
#pragma unroll
                for (int c = 0; c < C::VB; ++c) {
                    if (PAIRED)
                        tma_load_5d(dst + c * C::BOX, &tv, bar, 64 * c, 0, hk, j * (C::BN / 2), b);
                    else
                        load4_p(dst + c * C::BOX, &tv, bar, 64 * c, hk, j * C::BN, b, pol_reuse);
                }
                ++vc;
            };
            for (int k = 0; ok; ++k) {
                const int w = snake_tile(k, cta, G, NT);
                if (w < 0) break;
                const int qt = n_qt - 1 - w / per_qt, rest = w % per_qt;
                const int h = rest % p.H, b = rest / p.H, n_kv = kv_tiles(qt);
                const int hq1 = V2 ? 2 * h : h, hq2 = V2 ? 2 * h + 1 : h;
                const int hk = V2 ? (2 * h) / p.G : h;
                // Q of this tile, with K tile 0, once the previous tile's last QK
                // has been issued: one barrier for both
                if (tc > 0 && !wait_p(bar_qe, static_cast<uint32_t>((tc - 1) & 1), p.err)) break;
                if (!k_free()) break;
                expect_p(bar_qf, 2 * C::Q_TILE + C::K_SLOT);
#pragma unroll
                for (int c = 0; c < C::QB; ++c) {
                    load4_p(sQ1 + c * C::BOX, &tq1, bar_qf, 64 * c, hq1, qt * C::BM, b, pol_once);
                    load4_p(sQ2 + c * C::BOX, &tq2, bar_qf, 64 * c, hq2, qt * C::BM, b, pol_once);
                }
                put_k(0, hk, b, bar_qf);
                ++tc;
                // then V tile j with K tile j + 1 on V(j)'s barrier, in the order the
                // MMAs consume them (one wait per key tile in the MMA warp)
                for (int j = 0; ok && j < n_kv; ++j) {
                    const bool next_k = j + 1 < n_kv;
                    ok = v_free() && (!next_k || k_free());
                    if (!ok) break;
                    const uint32_t bv = bar_vf + 8 * (vc % C::VS);
                    expect_p(bv, C::V_SLOT + (next_k ? C::K_SLOT : 0));
                    put_v(j, hk, b, bv);
                    if (next_k) put_k(j + 1, hk, b, bv);
                }
            }
            // leave no copy in flight
            auto drain_p = [&](uint32_t bar, uint32_t parity) {
                if constexpr (kElectLoad) warp_wait_drain(bar, parity, p.err);
                else mbar_wait_drain(bar, parity, p.err);
            };
            if (tc > 0) drain_p(bar_qf, static_cast<uint32_t>((tc - 1) & 1));
            for (int k = (vc > C::VS ? vc - C::VS : 0); k < vc; ++k)
                drain_p(bar_vf + 8 * (k % C::VS), static_cast<uint32_t>((k / C::VS) & 1));
        }
    } else if (warp == 1 || warp == 2) {
        if (C::REG_SPLIT) regs_decrease<C::REGS_LOW>();
        if (warp == 2) {
            // --------------------------------------------- lambda (V1 only)
            if (!V2) {
                // lam_init = 0.8 - 0.6 exp(-0.3 layer); lam = exp(lq1.lk1) - exp(lq2.lk2) + lam_init
                float d1 = 0.f, d2 = 0.f;
                for (int c = lane; c < p.dlam; c += 32) {
                    d1 = fmaf(p.lq1[c], p.lk1[c], d1);
                    d2 = fmaf(p.lq2[c], p.lk2[c], d2);
                }
                d1 = warp_sum(d1);
                d2 = warp_sum(d2);
                if (lane == 0) {
                    const float lam_init = 0.8f - 0.6f * expf(-0.3f * static_cast<float>(p.layer_index));
                    lam_smem[0] = expf(d1) - expf(d2) + lam_init;
                    lam_smem[1] = lam_init;
                    mbar_arrive(bar_lam);
                }
            }
        }
        // ------------------------------------------------------------ MMA
        if ((C::ELECT_ISSUE || lane == 0) && (warp == 1 || C::TWO_ISSUERS)) {
            // issue primitives of this thread (lane 0) or of the converged warp
            auto wait_i = [&](uint32_t bar, uint32_t parity, uint32_t *err) -> bool {
                if constexpr (C::ELECT_ISSUE) return warp_wait_vote(bar, parity, err, true);
                else return mbar_wait(bar, parity, err);
            };
            auto ss_i = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
                if constexpr (C::ELECT_ISSUE) mma_ss_elect(d, a, b, idesc, acc);
                else mma_ss(d, a, b, idesc, acc);
            };
            auto ts_i = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
                if constexpr (C::ELECT_ISSUE) mma_ts_elect(d, a, b, idesc, acc);
                else mma_ts(d, a, b, idesc, acc);
            };
            auto commit_i = [&](uint32_t bar) {
                if constexpr (C::ELECT_ISSUE) mma_commit_elect(bar);
                else mma_commit(bar);
            };
            // branches issued by this thread: both, or branch warp - 1
            const int br0 = C::TWO_ISSUERS ? warp - 1 : 0, br1 = C::TWO_ISSUERS ? warp - 1 : 1;
            // Descriptors are built once per operand; a K step only moves the
            // start address field (bits 0-13, in 16-byte units), which never
            // carries for shared-memory addresses.
            auto issue_qk = [&](uint32_t dcol, uint32_t sq, uint32_t sk) {
                const uint64_t da = sdesc_sw128(sq, 16, 1024), db = sdesc_sw128(sk, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DQK / 16; ++ks) {
                    const uint32_t off = ((ks >> 2) * C::BOX + (ks & 3) * 32) >> 4;
                    ss_i(tmem + dcol, da + off, db + off, C::IDESC_QK, ks > 0 ? 1u : 0u);
                }
            };
            // O += P V over one half of the key tile (64 keys = 4 K-steps).
            auto issue_pv_half = [&](uint32_t dcol, uint32_t pcol, uint32_t sv, int half, bool acc) {
                const uint64_t dv = sdesc_sw128(sv, C::BOX, 1024);
#pragma unroll
                for (int k = 0; k < C::BN / 32; ++k) {
                    const int ks = half * (C::BN / 32) + k;
                    ts_i(tmem + dcol, tmem + pcol + ks * 8, dv + ((ks * 2048) >> 4), C::IDESC_PV,
                           (acc || ks > 0) ? 1u : 0u);
                }
            };
            int kc = 0, vc = 0, tc = 0, it = 0;
            bool ok = true;
            auto k_at = [&](int br) {
                return sbase + C::OFF_K + (kc % C::KS) * C::K_SLOT + ((br && !V2) ? C::K_TILE : 0);
            };
            // S_b = Q_b K_b^T for this thread's branches, then the K slot's release
            auto scores = [&]() {
                for (int br = br0; br <= br1; ++br) {
                    issue_qk(br ? C::COL_S2 : C::COL_S1, br ? sQ2 : sQ1, k_at(br));
                    commit_i(bar_s + 8 * br);
                }
                commit_i(bar_ke + 8 * (kc % C::KS));
                ++kc;
            };
            for (int k = 0; ok; ++k) {
                const int w = snake_tile(k, cta, G, NT);
                if (w < 0) break;
                const int n_kv = kv_tiles(n_qt - 1 - w / per_qt);
                // Q of this tile landed (and, with the rotary embedding, rotated in place)
                ok = wait_i(ROPE ? bar_qr : bar_qf, static_cast<uint32_t>(tc & 1), p.err);
                if (!ok) break;
                tc_fence_after();
                scores();
                if (n_kv == 1) commit_i(bar_qe);
                for (int j = 0; ok && j < n_kv; ++j, ++it) {
                    const uint32_t pj = static_cast<uint32_t>(it & 1);
                    const int vst = vc % C::VS;
                    const uint32_t sv = sbase + C::OFF_V + vst * C::V_SLOT;
                    const bool more = j + 1 < n_kv;
                    ok = wait_i(bar_vf + 8 * vst, static_cast<uint32_t>((vc / C::VS) & 1), p.err);
                    // the first PV of a tile overwrites O: the previous epilogue must have read it
                    if (ok && j == 0 && tc > 0) ok = wait_i(bar_od, static_cast<uint32_t>((tc - 1) & 1), p.err);
                    // per branch: O_b += P_b V in two key halves as the softmax publishes them,
                    // then S_b of the next key tile (in order after the PV that reads P_b)
                    for (int br = br0; ok && br <= br1; ++br) {
                        const uint32_t colS = br ? C::COL_S2 : C::COL_S1, colO = br ? C::COL_O2 : C::COL_O1;
                        if (C::P_HALVES) {
                            ok = wait_i(bar_p + 16 * br, pj, p.err);
                            if (!ok) break;
                            tc_fence_after();
                            issue_pv_half(colO, colS, sv, 0, j > 0);
                        }
                        ok = wait_i(bar_p + 16 * br + 8, pj, p.err);
                        if (!ok) break;
                        tc_fence_after();
                        if (!C::P_HALVES) issue_pv_half(colO, colS, sv, 0, j > 0);
                        issue_pv_half(colO, colS, sv, 1, j > 0);
                        if (br == br1) {
                            commit_i(bar_ve + 8 * vst);
                            ++vc;
                        }
                        if (more) {
                            // K tile j + 1 landed with V tile j
                            issue_qk(colS, br ? sQ2 : sQ1, k_at(br));
                            commit_i(bar_s + 8 * br);
                            if (br == br1) {
                                commit_i(bar_ke + 8 * (kc % C::KS));
                                ++kc;
                                if (j + 2 == n_kv) commit_i(bar_qe);   // last QK of the tile issued
                            }
                        } else {
                            commit_i(bar_o + 8 * br);
                        }
                    }
                }
                ++tc;
            }
            // no MMA may be in flight when TMEM is released
            const uint32_t drain = warp == 1 ? bar_dr : bar_dr2;
            commit_i(drain);
            if constexpr (C::ELECT_ISSUE) warp_wait_drain(drain, 0, p.err);
            else mbar_wait_drain(drain, 0, p.err);
        }
    } else if (warp == 3) {
        if (C::REG_SPLIT) regs_decrease<C::REGS_LOW>();
        if (lane == 0 && !PAIRED) {
            bool ok = true;
            const uint64_t pol_once = l2_evict_first();   // the output is written once
            for (int k = 0;; ++k) {
                const int w = snake_tile(k, cta, G, NT);
                if (w < 0) break;
                const int qt = n_qt - 1 - w / per_qt, rest = w % per_qt;
                const int h = rest % p.H, b = rest / p.H;
                ok = ok && mbar_wait(bar_stg, static_cast<uint32_t>(k & 1), p.err);
                if (ok && DA_CHECK(qt * C::BM < p.T && h < p.H && b < p.B, p.err)) {
#pragma unroll
                    for (int bx = 0; bx < C::VB; ++bx)
                        tma_store_4d_hint(&tout, sbase + C::OFF_OUT + bx * C::BOX, 64 * bx, h, qt * C::BM, b, pol_once);
                    bulk_commit();
                }
                bulk_wait_read_all();
                mbar_arrive(bar_stf);
            }
            bulk_wait_all();
        }
    } else {
        // -------------------------------------------------------- softmax
        if (C::REG_SPLIT) regs_increase<C::REGS_HIGH>();
        const int br = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + (br ? C::COL_S2 : C::COL_S1);
        const uint32_t tO = tmem + lane_off + (br ? C::COL_O2 : C::COL_O1);
        const uint32_t my_s = bar_s + 8 * br, my_p = bar_p + 16 * br, my_o = bar_o + 8 * br;
        const float sl2 = p.scale_log2;
        float *xch = reinterpret_cast<float *>(smem + C::OFF_X);
        float *freq = reinterpret_cast<float *>(smem + C::OFF_FREQ);
        bool ok = true;
        float lam = 0.f, lam_init = 0.f;
        if (!V2) {
            ok = warp_wait_vote(bar_lam, 0, p.err, ok);
            lam = lam_smem[0];
            lam_init = lam_smem[1];
        }
        int it = 0;
        // Rotary embedding: the two softmax threads of a row turn half of the
        // row's channel pairs each, in both Q tiles of work tile kk (query
        // tile of work w), once the tiles have landed (cos and sin formed in
        // registers, no table); the MMA thread issues the tile's first QK
        // after all 8 warps have arrived.  Tile 0 is rotated before the first key tile,
        // tile kk + 1 right after the last P of tile kk (its Q load was issued
        // when the last QK of tile kk was), while the last PV runs.
        auto rotate_q = [&](int kk, int w) {
            if constexpr (ROPE) {
                const int tq = (n_qt - 1 - w / per_qt) * C::BM + row;
                ok = warp_wait_vote(bar_qf, static_cast<uint32_t>(kk & 1), p.err, ok);
                if (ok && tq < p.T && DA_CHECK(row < C::BM, p.err))
                    rope_q_row<DQK>(smem + C::OFF_Q1, smem + C::OFF_Q2, row, br, static_cast<float>(p.rope_pos0 + tq),
                                    freq, freq + DQK / 2);
                fence_async_smem();
                __syncwarp();
                mbar_arrive_elect(bar_qr);
            }
        };
        if (ROPE) {
            // f_i of the rotary embedding, once per CTA
            for (int i = (warp - 4) * 32 + lane; i < DQK / 2; i += 256) rope_freq(p.rope_base, i, DQK, freq[i], freq[DQK / 2 + i]);
            named_bar_sync(1, 256);
            const int w0 = snake_tile(0, cta, G, NT);
            if (w0 >= 0) rotate_q(0, w0);
        }
        // Every softmax warp walks the same tile list and reaches the same
        // named barriers, also after an error (then it skips waits and work).
        for (int k = 0;; ++k) {
            const int w = snake_tile(k, cta, G, NT);
            if (w < 0) break;
            const int qt = n_qt - 1 - w / per_qt, rest = w % per_qt;
            const int h = rest % p.H, b = rest / p.H, n_kv = kv_tiles(qt);
            const int t = qt * C::BM + row;   // query token of this thread's row
            // V2 gate logit of this row, fetched now and used in the epilogue
            const float lg = (V2 && !PAIRED && t < p.T) ? p.lam[(static_cast<int64_t>(b) * p.T + t) * p.H + h] : 0.f;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < n_kv; ++j, ++it) {
                ok = warp_wait_vote(my_s, static_cast<uint32_t>(it & 1), p.err, ok);
                if (!ok) continue;
                tc_fence_after();
                uint32_t s[C::BN];
                tmem_ld32(tS + 0, s);
                tmem_ld32(tS + 32, s + 32);
                if (C::LD_SPLIT) tmem_wait_ld();
                tmem_ld32(tS + 64, s + 64);
                tmem_ld32(tS + 96, s + 96);
                const bool diag = PAIRED ? j >= 2 * qt : j == qt;
                float rmax;
                if (!C::LD_SPLIT || diag) {
                    tmem_wait_ld();
                    if (diag) {   // diagonal tile(s): keys past this row are masked
                        const int lim = PAIRED ? 2 * row + br - C::BN * (j - 2 * qt) : row;   // last visible column
#pragma unroll
                        for (int c = 0; c < C::BN; ++c)
                            if (c > lim) s[c] = 0xff800000u;   // -inf
                    }
                    rmax = row_max128(s);
                } else {
                    // max of keys 0-63 while keys 64-127 are still coming out of TMEM
                    float a[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) a[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
                    for (int k2 = 8; k2 < 64; k2 += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            a[i] = fmax3(a[i], __uint_as_float(s[k2 + 2 * i]), __uint_as_float(s[k2 + 2 * i + 1]));
                    tmem_wait_ld();
#pragma unroll
                    for (int k2 = 64; k2 < 128; k2 += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            a[i] = fmax3(a[i], __uint_as_float(s[k2 + 2 * i]), __uint_as_float(s[k2 + 2 * i + 1]));
                    rmax = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
                }
                const float m_new = fmaxf(m_ref, rmax * sl2);
                const bool resc = m_new > m_ref + 8.f;
                const float alpha = resc ? ex2(m_ref - m_new) : 1.f;
                l *= alpha;
                m_ref = resc ? m_new : m_ref;
                if (j > 0 && __any_sync(0xffffffffu, resc)) {
                    // O_b is quiescent: PV_b(j-1) completed before S_b(j) was signalled.
#pragma unroll 1
                    for (int c0 = 0; c0 < DV; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32(tO + c0, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int kk = 0; kk < 32; ++kk) ov[kk] = __float_as_uint(__uint_as_float(ov[kk]) * alpha);
                        tmem_st32(tO + c0, ov);
                    }
                    tmem_wait_st();
                }
                // P in two halves: with P_HALVES the tensor core starts O += P V
                // on keys 0-63 while keys 64-127 are still being exponentiated;
                // without, the MMA thread waits for the second half only (the
                // first half's store wait is kept: measured, dropping it costs V2
                // the 2 % that the single wait gains).
                l += exp_pack64(s, sl2, m_ref);
                tmem_st32(tS + 0, s);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_elect(my_p);
                l += exp_pack64(s + 64, sl2, m_ref);
                tmem_st32(tS + 32, s + 64);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_elect(my_p + 8);
            }
            if (ROPE) {
                const int wn = snake_tile(k + 1, cta, G, NT);
                if (wn >= 0) rotate_q(k + 1, wn);
            }

            // --------------------------------------------------- epilogue
            if constexpr (PAIRED) {
                // each branch is one head of the pair: O_e / l_e to its rows, directly
                ok = warp_wait_vote(my_o, static_cast<uint32_t>(k & 1), p.err, ok);
                tc_fence_after();
                const float il = 1.f / l;
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + static_cast<int64_t>(b) * p.o_sb +
                                     static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(2 * h + br) * p.o_sh;
#pragma unroll
                for (int cc = 0; cc < DV; cc += 32) {
                    uint32_t a[32];
                    tmem_ld32(tO + cc, a);
                    tmem_wait_ld();
                    if (ok && t < p.T && DA_CHECK(2 * h + br < 2 * p.H && b < p.B && cc + 32 <= DV, p.err)) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const uint32_t *aa = a + 8 * q8;
                            d4[q8] = make_uint4(pack_bf16(__uint_as_float(aa[0]) * il, __uint_as_float(aa[1]) * il),
                                                pack_bf16(__uint_as_float(aa[2]) * il, __uint_as_float(aa[3]) * il),
                                                pack_bf16(__uint_as_float(aa[4]) * il, __uint_as_float(aa[5]) * il),
                                                pack_bf16(__uint_as_float(aa[6]) * il, __uint_as_float(aa[7]) * il));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                mbar_arrive_elect(bar_od);   // O read: the next tile's first PV may overwrite it
                continue;
            }
            ok = warp_wait_vote(my_o, static_cast<uint32_t>(k & 1), p.err, ok);
            if (k > 0) ok = warp_wait_vote(bar_stf, static_cast<uint32_t>((k - 1) & 1), p.err, ok);
            tc_fence_after();
            if (TRAIN && t < p.T && DA_CHECK(b < p.B && h < p.H, p.err))   // this branch's log-sum-exp (log2 units) for the backward
                p.slse[((static_cast<int64_t>(br) * p.B + b) * p.H + h) * p.T + t] = m_ref + __log2f(l);
            xch[br * 128 + row] = l;
            named_bar_sync(1, 256);   // both branches' final O are complete past this point
            tc_fence_after();
            const float l1 = xch[row], l2 = xch[128 + row];
            const float c2 = V2 ? 1.f / (1.f + __expf(-lg)) / l2 : lam / l2;
            const float c1 = 1.f / l1;
            constexpr int HALF = DV / 2;
            const int col0 = br * HALF;
            float x[HALF];
            float ss = 0.f;
#pragma unroll
            for (int cc = 0; cc < HALF; cc += 32) {
                uint32_t a[32], bb[32];
                tmem_ld32(tmem + lane_off + C::COL_O1 + col0 + cc, a);
                tmem_ld32(tmem + lane_off + C::COL_O2 + col0 + cc, bb);
                tmem_wait_ld();
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    const float v = __uint_as_float(a[kk]) * c1 - __uint_as_float(bb[kk]) * c2;
                    x[cc + kk] = v;
                    ss = fmaf(v, v, ss);
                }
                if (TRAIN && !V2 && t < p.T && DA_CHECK(b < p.B && h < p.H && col0 + cc + 32 <= DV, p.err)) {
                    // V1: x (the RMSNorm input) and a2 = O2 / l2 in fp32, channels col0 + cc .. + 31
                    const float i2 = 1.f / l2;
                    const int64_t off = ((static_cast<int64_t>(b) * p.T + t) * p.H + h) * DV + col0 + cc;
                    float4 *d1 = reinterpret_cast<float4 *>(static_cast<float *>(p.sa1) + off);
                    float4 *d2 = reinterpret_cast<float4 *>(static_cast<float *>(p.sa2) + off);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        d1[q4] = make_float4(x[cc + 4 * q4], x[cc + 4 * q4 + 1], x[cc + 4 * q4 + 2], x[cc + 4 * q4 + 3]);
                        d2[q4] = make_float4(__uint_as_float(bb[4 * q4]) * i2, __uint_as_float(bb[4 * q4 + 1]) * i2,
                                             __uint_as_float(bb[4 * q4 + 2]) * i2,
                                             __uint_as_float(bb[4 * q4 + 3]) * i2);
                    }
                }
                if (TRAIN && V2 && t < p.T && DA_CHECK(b < p.B && h < p.H && col0 + cc + 32 <= DV, p.err)) {
                    // V2: a_b = O_b / l_b of this row's channels col0 + cc .. + 31, both heads, bf16
                    const float i2 = 1.f / l2;
                    const int64_t off = ((static_cast<int64_t>(b) * p.T + t) * p.H + h) * DV + col0 + cc;
                    uint4 *d1 = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.sa1) + off);
                    uint4 *d2 = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.sa2) + off);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const uint32_t *aa = a + 8 * q8, *bq = bb + 8 * q8;
                        d1[q8] = make_uint4(pack_bf16(__uint_as_float(aa[0]) * c1, __uint_as_float(aa[1]) * c1),
                                            pack_bf16(__uint_as_float(aa[2]) * c1, __uint_as_float(aa[3]) * c1),
                                            pack_bf16(__uint_as_float(aa[4]) * c1, __uint_as_float(aa[5]) * c1),
                                            pack_bf16(__uint_as_float(aa[6]) * c1, __uint_as_float(aa[7]) * c1));
                        d2[q8] = make_uint4(pack_bf16(__uint_as_float(bq[0]) * i2, __uint_as_float(bq[1]) * i2),
                                            pack_bf16(__uint_as_float(bq[2]) * i2, __uint_as_float(bq[3]) * i2),
                                            pack_bf16(__uint_as_float(bq[4]) * i2, __uint_as_float(bq[5]) * i2),
                                            pack_bf16(__uint_as_float(bq[6]) * i2, __uint_as_float(bq[7]) * i2));
                    }
                }
            }
            // O has been read: the next tile's first PV may overwrite it
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elect(bar_od);
            if (!V2) {
                xch[256 + br * 128 + row] = ss;
                named_bar_sync(1, 256);
                const float ms = (xch[256 + row] + xch[384 + row]) * (1.f / static_cast<float>(DV));
                const float r = (1.f - lam_init) * rsqrtf(ms + 1e-5f);
#pragma unroll
                for (int kk = 0; kk < HALF; ++kk) x[kk] *= r;
            }
            named_bar_sync(1, 256);   // exchange area read: the staging tile may be written
            // Stage the bf16 row in the 128-byte-swizzled layout of the output
            // map's 128 x 64 boxes, then one thread stores the tile with TMA
            // (rows past T are clipped by the map's bounds).
#pragma unroll
            for (int kk = 0; kk < HALF; kk += 8) {
                const int col = col0 + kk, ch = (col & 63) >> 3;
                if (!DA_CHECK((col >> 6) * C::BOX + row * 128 + 16 * ch + 16 <= C::OUT_TILE, p.err)) continue;
                uint4 v;
                v.x = pack_bf16(x[kk], x[kk + 1]);
                v.y = pack_bf16(x[kk + 2], x[kk + 3]);
                v.z = pack_bf16(x[kk + 4], x[kk + 5]);
                v.w = pack_bf16(x[kk + 6], x[kk + 7]);
                *reinterpret_cast<uint4 *>(smem + C::OFF_OUT + (col >> 6) * C::BOX + row * 128 +
                                           ((ch ^ (row & 7)) << 4)) = v;
            }
            fence_async_smem();
            __syncwarp();
            mbar_arrive_elect(bar_stg);
        }
    }

    // ------------------------------------------------------------ teardown
    if (warp == 3 && lane == 0) bulk_wait_all();   // output stores complete before exit
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int DQK, int DV, bool V2, bool TRAIN, bool PAIRED = false, bool ROPE = false>
cudaError_t launch_t(const PrefillMaps &m, const PrefillParams &p, cudaStream_t s) {
    using C = PreCfg<DQK, DV, V2>;
    static unsigned long long attr_done = 0;   // one bit per device
    const cudaError_t ea = once_per_device(&attr_done, [] {
        // The register split inside the kernel must fit in what the launch
        // grants (384 threads x registers per thread), or its increase would
        // never complete: refuse to launch otherwise.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, prefill_onepass<DQK, DV, V2, TRAIN, PAIRED, ROPE>);
        if (e != cudaSuccess) return e;
        if (C::REG_SPLIT && fa.numRegs < C::REGS_NEEDED_AT_LAUNCH) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(prefill_onepass<DQK, DV, V2, TRAIN, PAIRED, ROPE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    });
    if (ea != cudaSuccess) return ea;
    const int n_qt = (p.T + C::BM - 1) / C::BM;
    const long long tiles = static_cast<long long>(n_qt) * p.H * p.B;
    if (tiles < 1 || tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    // persistent: one CTA per SM (shared memory and TMEM allow no more)
    if (p.num_sms < 1) return cudaErrorInvalidValue;
    const unsigned grid = static_cast<unsigned>(tiles < p.num_sms ? tiles : p.num_sms);
    prefill_onepass<DQK, DV, V2, TRAIN, PAIRED, ROPE><<<grid, 384, C::SMEM, s>>>(m.q1, m.q2, m.k1, m.k2, m.v, m.out, p);
    return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int dqk, int dv, bool v2) {
    if (v2) return (dqk == 128 && dv == 128) || (dqk == 64 && dv == 64);
    return (dqk == 64 && dv == 128) || (dqk == 32 && dv == 64);
}

cudaError_t launch_prefill(const PrefillMaps &m, const PrefillParams &p, int dqk, int dv, bool v2,
                           cudaStream_t s) {
    if (v2 && dqk == 128 && dv == 128) return launch_t<128, 128, true, false>(m, p, s);
    if (v2 && dqk == 64 && dv == 64) return launch_t<64, 64, true, false>(m, p, s);
    if (!v2 && dqk == 64 && dv == 128) return launch_t<64, 128, false, false>(m, p, s);
    // d = 32: the q / k maps are 32 columns wide and their 64-column boxes are
    // zero-filled past column 32, so the d = 64 kernel computes the same S
    if (!v2 && dqk == 32 && dv == 64) return launch_t<64, 64, false, false>(m, p, s);
    return cudaErrorInvalidValue;
}

bool paired_supported(int d) { return d == 64 || d == 128; }

cudaError_t launch_paired(const PrefillMaps &m, const PrefillParams &p, int d, cudaStream_t s) {
    if (p.G != 2) return cudaErrorInvalidValue;   // kv coordinate = pair index
    if (d == 128) return launch_t<128, 128, true, false, true>(m, p, s);
    if (d == 64) return launch_t<64, 64, true, false, true>(m, p, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_v2_rope(const PrefillMaps &m, const PrefillParams &p, int d, cudaStream_t s) {
    if (!(p.rope_base > 0.0)) return cudaErrorInvalidValue;
    if (d == 128) return launch_t<128, 128, true, false, false, true>(m, p, s);
    if (d == 64) return launch_t<64, 64, true, false, false, true>(m, p, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_train(const PrefillMaps &m, const PrefillParams &p, int dqk, int dv, bool v2,
                                 cudaStream_t s) {
    if (!p.sa1 || !p.sa2 || !p.slse) return cudaErrorInvalidValue;
    if (v2 && dqk == 128 && dv == 128) return launch_t<128, 128, true, true>(m, p, s);
    if (v2 && dqk == 64 && dv == 64) return launch_t<64, 64, true, true>(m, p, s);
    if (!v2 && dqk == 64 && dv == 128) return launch_t<64, 128, false, true>(m, p, s);
    if (!v2 && dqk == 32 && dv == 64) return launch_t<64, 64, false, true>(m, p, s);   // zero-filled q / k boxes
    return cudaErrorInvalidValue;
}

}  // namespace da
