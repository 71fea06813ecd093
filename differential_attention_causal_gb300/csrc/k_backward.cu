// k_backward.cu -- backward of the causal differential attention on tcgen05
// tensor cores (bf16 in, fp32 accumulate): DIFF V1 (d = 64, dv = 128) and
// DIFF V2 (D = 64 / 128).
//
// "Differential Transformer V2", DiffAttnV1 / DiffAttnV2, differentiated.
// Both operations are two softmax attentions a_b = softmax(S_b) V, b = 1, 2,
// S_b = scale Q_b K_b^T (causal), combined per row.  With g_b = dL/da_b the
// upstream gradient of branch b, each branch backward is
//     dV += P_b^T g_b,   dP_b = g_b V^T,   dS_b = P_b o (dP_b - D_b),
//     D_b[i] = sum_j P_b[i,j] dP_b[i,j] = g_b[i] . a_b[i],
//     dQ_b = scale dS_b K_b,   dK_b = scale dS_b^T Q_b.
// Here g_2 = c g_1 row by row (V1: g_1 = dx, c = -lam, dx the RMSNorm
// backward of (1 - lam_init) dout; V2: g_1 = dout, c = -sigmoid(lam[t])), so
//     dP_2 = c dP_1            (one dP product for both branches)
//     dV  += (P_1 + c P_2)^T g_1   (one dV product for both branches).
// P_b is recomputed from the scores and the forward's log-sum-exp.
//
// Kernels (the row pre-pass and the lambda reduction at the end of the file):
//   bwd_pre     one warp per row: g_1 (V1: the RMSNorm backward), D_1, D_2,
//               c, and the lambda gradient (V1: per-row share of dL/dlam;
//               V2: dL/dlam[t] directly).
//   bwd_dq      query-stationary: 128 query rows, 64-key sub-tiles.  TMEM:
//               S1 | S2 | dP (64 columns each) | dQ1 | dQ2.
//   bwd_dkdv    key-stationary: 128 key rows, 64-query sub-tiles (for V2 of
//               every pair of the kv group).  TMEM: S1^T | S2^T | dP^T (64
//               each) | dK1 (| dK2) | dV.
// In both, warp 0 streams the sub-tiles with TMA, warp 1 issues the score
// MMAs (S, dP), warp 2 the accumulating ones, and two row warpgroups (warps
// 4-7, 8-11; thread = TMEM lane = row) each take 32 of a sub-tile's 64
// columns.  The rows load S and dP, release that TMEM at once (the next
// sub-tile's products start on the tensor cores), form P, dS in fp32 and
// write them in bf16 to 128-byte-swizzled shared tiles, the A operands of
// the accumulating MMAs (dV, dK_b or dQ_b).  Two issuing warps because a
// thread's barrier wait returns only after the MMAs it issued before it
// have drained: with one issuer every wait left the tensor pipe idle.
// The TMA warp and the two issuing warps run converged (one lane chosen by
// elect.sync issues each copy, MMA and commit; their waits are warp-vote
// loops), which measured 0.7 % faster on GB300 than lane 0 alone at d = 64
// (the d = 128 split kernels 1.5-3 % slower, kept the same for one code path).  The row
// warps arrive on barriers through elect.sync as well (V2 2 % faster), but
// keep the per-lane polling wait (warp_wait): the vote-based one costs the
// V1 backward 4-5 %.
#include <type_traits>

#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

// MODE 0: both branches in one kernel (dq: dQ1 and dQ2; dkdv: dK1, dK2 and dV).
// MODE 1: one branch per CTA, the branch = work index & 1 (dq: dQ_b; dkdv: dK_b).
// MODE 2: dkdv kernel computing dV only.
// DIFF V1 at d = 128 (dv = 256) runs MODE 1 dq, MODE 1 dkdv and MODE 2 dkdv:
// with both branches, dK1 | dK2 | dV (512 fp32 columns) next to S1 | S2 | dP
// would not fit in TMEM, nor the resident tiles in shared memory.
template <int DQK, int DV, bool V2, int MODE = 0>
struct BwdCfg {
    static constexpr int BM = 128, BN = 64;
    static constexpr int QB = DQK / 64, VB = DV / 64;   // 64-column boxes
    static constexpr int RBOX = 128 * 128;              // 128 rows x 64 bf16
    static constexpr int CBOX = 64 * 128;               // 64 rows x 64 bf16
    static constexpr int NK = V2 ? 1 : 2;               // distinct K tiles (V1: K1, K2)
    static constexpr int NQ = MODE == 1 ? 1 : 2;        // Q tiles a CTA reads (both branches, or its own)
    static constexpr int NKT = MODE == 1 ? 1 : NK;      // K tiles a CTA reads
    static constexpr bool HAS_DP = MODE != 2;           // dP = G V^T is formed (and V read)
    static constexpr int COL_S1 = 0, COL_S2 = 64, COL_DP = 128, COL_ACC = 192;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t IDESC_S = idesc_bf16(128, 64, false);
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, DQK, true);
    static constexpr uint32_t IDESC_V = idesc_bf16(128, DV, true);
    // warp 0 TMA, warps 1-2 MMA, warps 4.. NRG row warpgroups, each taking RC of a
    // sub-tile's 64 columns (measured on GB300: four groups of 16 columns are 3-8 %
    // slower than two of 32)
    static constexpr int NRG = 2, RC = BN / NRG;
    static constexpr int THREADS = 128 + 128 * NRG;
    // MMAs issued by two threads: warp 1 the score products (S, dP), warp 2 the
    // accumulating ones; each thread's barrier waits then stall only its own
    // stream while the other's MMAs keep the tensor pipe busy
    static constexpr bool TWO_ISSUERS = true;
    static constexpr int MIN_SMEM = 120 * 1024;   // one CTA per SM (each takes all of TMEM)

    // ---- dq kernel: resident Q1 (, Q2), G (128 rows); ring of K1 (, K2), V (64 rows);
    //      result tiles dS1 (, dS2) (128 x 64 bf16, the A operands of dQ += dS K)
    static constexpr int DQ_NRES = MODE == 1 ? 1 : 2;
    static constexpr int DQ_STAGES = MODE == 1 ? 2 : (DQK == 64 ? 4 : 3);   // shared memory
    static constexpr int DQ_OFF_Q1 = 0;
    static constexpr int DQ_OFF_Q2 = QB * RBOX;
    static constexpr int DQ_OFF_G = NQ * QB * RBOX;
    static constexpr int DQ_OFF_RES = DQ_OFF_G + VB * RBOX;
    static constexpr int DQ_OFF_RING = DQ_OFF_RES + DQ_NRES * RBOX;
    static constexpr int DQ_STAGE = NKT * QB * CBOX + VB * CBOX;
    static constexpr int DQ_OFF_BAR = DQ_OFF_RING + DQ_STAGES * DQ_STAGE;
    // res, full[S], empty[S], s, sfree, rready, rfree, done, drain, drain of the score issuer
    static constexpr int DQ_NBAR = 1 + 2 * DQ_STAGES + 7;
    static constexpr int DQ_OFF_TSLOT = DQ_OFF_BAR + DQ_NBAR * 8;
    static constexpr int DQ_SMEM_RAW = DQ_OFF_TSLOT + 8 + 1024;
    static constexpr int DQ_SMEM = DQ_SMEM_RAW > MIN_SMEM ? DQ_SMEM_RAW : MIN_SMEM;
    static constexpr int COL_DQ1 = COL_ACC, COL_DQ2 = COL_ACC + DQK;

    // ---- dkdv kernel: resident K1 (, K2) (, V) (128 rows); ring of Q1 (, Q2), G (64 rows)
    //      + row vectors; result tiles (P~^T,) dS1^T (, dS2^T) or P~^T alone (128 x 64
    //      bf16, the A operands of dV, dK)
    static constexpr int KV_NRES = MODE == 0 ? 3 : 1;
    static constexpr int KV_STAGES = MODE != 0 ? 2 : ((V2 && DQK == 128) ? 2 : 3);   // shared memory
    static constexpr int KV_OFF_K1 = 0;
    static constexpr int KV_OFF_K2 = QB * RBOX;                    // V1, MODE 0 / 2
    static constexpr int KV_OFF_V = NKT * QB * RBOX;
    static constexpr int KV_OFF_RES = KV_OFF_V + (HAS_DP ? VB * RBOX : 0);
    static constexpr int KV_OFF_RING = KV_OFF_RES + KV_NRES * RBOX;
    static constexpr int KV_VEC = 5 * 64 * 4;                      // lse1, lse2, d1, d2, c
    static constexpr int KV_STAGE_TMA = NQ * QB * CBOX + VB * CBOX;
    static constexpr int KV_STAGE = KV_STAGE_TMA + 2048;           // vectors, padded to keep 1 KB alignment
    static constexpr int KV_OFF_BAR = KV_OFF_RING + KV_STAGES * KV_STAGE;
    static constexpr int KV_NBAR = 1 + 2 * KV_STAGES + 7;
    static constexpr int KV_OFF_TSLOT = KV_OFF_BAR + KV_NBAR * 8;
    static constexpr int KV_SMEM_RAW = KV_OFF_TSLOT + 8 + 1024;
    static constexpr int KV_SMEM = KV_SMEM_RAW > MIN_SMEM ? KV_SMEM_RAW : MIN_SMEM;
    static constexpr int COL_DK1 = COL_ACC;
    static constexpr int COL_DK2 = V2 ? COL_ACC : COL_ACC + DQK;   // V2: both branches hit one K
    static constexpr int COL_DV = MODE == 2 ? COL_ACC : COL_ACC + NK * DQK;

    static_assert(MODE == 0 || (!V2 && DQK == 128 && DV == 256), "split modes: V1 at d = 128");
    static_assert((MODE == 1 ? COL_DQ1 + DQK : COL_DQ2 + DQK) <= 512, "TMEM budget (dq)");
    static_assert((MODE == 1 ? COL_DK1 + DQK : COL_DV + DV) <= 512, "TMEM budget (dkdv)");
    static_assert((MODE == 2 || DQ_SMEM <= 232448) && KV_SMEM <= 232448, "shared memory budget");
    static_assert(KV_VEC <= 2048, "vector area");
};

// RC consecutive fp32 columns of this thread's TMEM lane (RC = 16 or 32)
template <int RC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t *r) {
    static_assert(RC == 16 || RC == 32, "columns per row thread");
    if constexpr (RC == 32)
        tmem_ld32(taddr, r);
    else
        tmem_ld16(taddr, r);
}

// RC / 2 bf16 pairs from RC floats held as bit patterns
template <int RC>
__device__ __forceinline__ void pack_cols(const uint32_t *x, uint32_t *u) {
#pragma unroll
    for (int i = 0; i < RC / 2; ++i) u[i] = pack_bf16(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
}

// Write RC bf16 values (RC / 2 packed words) of one row into a 128-row x
// 64-col K-major tile with 128-byte swizzle (the layout a TMA box of that
// shape has), at the row's 16-byte chunks RC / 8 * part .. RC / 8 * part + RC / 8 - 1.
template <int RC>
__device__ __forceinline__ void store_row_part(uint8_t *tile, int row, int part, const uint32_t *u) {
#pragma unroll
    for (int k = 0; k < RC / 8; ++k) {
        const int ch = RC / 8 * part + k;
        *reinterpret_cast<uint4 *>(tile + row * 128 + ((ch ^ (row & 7)) << 4)) =
            make_uint4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
    }
}

// ===================================================================== dQ
// Pipeline per 64-key sub-tile j (one MMA issuer, two row warpgroups):
//   MMA:  S(j), dP(j) into TMEM once the rows have loaded S(j-1), dP(j-1)
//         ("sfree"); then dQ += dS(j-1) K(j-1) from the shared-memory result
//         tiles once the rows have written them ("rready").
//   rows: load S(j), dP(j) -> sfree; compute dS; wait until dQ(j-1) has read
//         the result tiles ("rfree"); write dS(j) -> rready.
// So S(j+1) and dP(j+1) run on the tensor cores while the rows work on j.
template <int DQK, int DV, bool V2, int MODE = 0>
__global__ void __launch_bounds__(BwdCfg<DQK, DV, V2, MODE>::THREADS, 1)
    bwd_dq(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tq2,
           const __grid_constant__ CUtensorMap tg, const __grid_constant__ CUtensorMap tk1,
           const __grid_constant__ CUtensorMap tk2, const __grid_constant__ CUtensorMap tv, const BwdParams p) {
    using C = BwdCfg<DQK, DV, V2, MODE>;
    static_assert(MODE != 2, "dq kernel: MODE 0 or 1");
    constexpr int ST = C::DQ_STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // tile w -> query tile (heaviest first), head / pair, batch; MODE 1: the two
    // branches of a tile are neighbouring CTAs, branch = index & 1
    const int n_qt = (p.T + C::BM - 1) / C::BM;
    const int per_qt = p.H * p.B;
    const int w = static_cast<int>(blockIdx.x) >> (MODE == 1 ? 1 : 0);
    const int brc = MODE == 1 ? static_cast<int>(blockIdx.x & 1u) : 0;   // this CTA's branch (MODE 1)
    const int qt = n_qt - 1 - w / per_qt, rest = w % per_qt;
    const int h = rest % p.H, b = rest / p.H;
    const int n_kt = (p.T + C::BN - 1) / C::BN;
    const int kend = (qt + 1) * (C::BM / C::BN);
    const int n_kv = kend < n_kt ? kend : n_kt;   // 64-key sub-tiles at or before the diagonal
    const int hq1 = V2 ? 2 * h : h, hq2 = V2 ? 2 * h + 1 : h;
    const int hk = V2 ? (2 * h) / p.G : h;

    const uint32_t bar_res = sbase + C::DQ_OFF_BAR;
    const uint32_t bar_full = bar_res + 8;
    const uint32_t bar_empty = bar_full + 8 * ST;
    const uint32_t bar_s = bar_empty + 8 * ST;
    const uint32_t bar_sfree = bar_s + 8;
    const uint32_t bar_rready = bar_sfree + 8;
    const uint32_t bar_rfree = bar_rready + 8;
    const uint32_t bar_done = bar_rfree + 8;
    const uint32_t bar_dr = bar_done + 8;
    const uint32_t bar_dra = bar_dr + 8;
    const uint32_t tslot = sbase + C::DQ_OFF_TSLOT;

    if (threadIdx.x == 0) {
        mbar_init(bar_res, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_sfree, 4 * C::NRG);   // one arrival per row warp
        mbar_init(bar_rready, 4 * C::NRG);
        mbar_init(bar_rfree, 1);
        mbar_init(bar_done, 1);
        mbar_init(bar_dr, 1);
        mbar_init(bar_dra, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::DQ_OFF_TSLOT);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        {
            // the whole warp, converged; one elected lane issues each copy
            auto wait_c = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
                return warp_wait_vote(bar, parity, err, true);
            };
            // MODE 1: only this branch's Q and K
            const CUtensorMap *mq = (MODE == 1 && brc) ? &tq2 : &tq1;
            const CUtensorMap *mk = (MODE == 1 && brc) ? &tk2 : &tk1;
            prefetch_tmap(mq);
            prefetch_tmap(&tg);
            prefetch_tmap(mk);
            prefetch_tmap(&tv);
            mbar_arrive_expect_tx_elect(bar_res, C::NQ * C::QB * C::RBOX + C::VB * C::RBOX);
#pragma unroll
            for (int c = 0; c < C::QB; ++c) {
                tma_load_4d_elect(sbase + C::DQ_OFF_Q1 + c * C::RBOX, mq, bar_res, 64 * c, (MODE == 1 && brc) ? hq2 : hq1,
                            qt * C::BM, b);
                if (MODE == 0)
                    tma_load_4d_elect(sbase + C::DQ_OFF_Q2 + c * C::RBOX, &tq2, bar_res, 64 * c, hq2, qt * C::BM, b);
            }
#pragma unroll
            for (int c = 0; c < C::VB; ++c)
                tma_load_4d_elect(sbase + C::DQ_OFF_G + c * C::RBOX, &tg, bar_res, 64 * c, h, qt * C::BM, b);
            int j = 0;
            for (; j < n_kv; ++j) {
                const int st = j % ST;
                if (j >= ST && !wait_c(bar_empty + 8 * st, static_cast<uint32_t>((j / ST - 1) & 1), p.err))
                    break;
                const uint32_t dst = sbase + C::DQ_OFF_RING + st * C::DQ_STAGE;
                mbar_arrive_expect_tx_elect(bar_full + 8 * st, C::DQ_STAGE);
#pragma unroll
                for (int c = 0; c < C::QB; ++c) {
                    tma_load_4d_elect(dst + c * C::CBOX, mk, bar_full + 8 * st, 64 * c, hk, j * C::BN, b);
                    if (!V2 && MODE == 0)
                        tma_load_4d_elect(dst + (C::QB + c) * C::CBOX, &tk2, bar_full + 8 * st, 64 * c, hk, j * C::BN, b);
                }
#pragma unroll
                for (int c = 0; c < C::VB; ++c)
                    tma_load_4d_elect(dst + (C::NKT * C::QB + c) * C::CBOX, &tv, bar_full + 8 * st, 64 * c, hk, j * C::BN,
                                b);
            }
            // leave no copy in flight
            warp_wait_drain(bar_res, 0, p.err);
            for (int k = (j > ST ? j - ST : 0); k < j; ++k)
                warp_wait_drain(bar_full + 8 * (k % ST), static_cast<uint32_t>((k / ST) & 1), p.err);
        }
    } else if (warp == 1 || (C::TWO_ISSUERS && warp == 2)) {
        // ------------------------------------------------------------ MMA
        {
            // the whole warp, converged; one elected lane issues each MMA and commit
            auto wait_c = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
                return warp_wait_vote(bar, parity, err, true);
            };
            const uint32_t sQ1 = sbase + C::DQ_OFF_Q1, sQ2 = sbase + C::DQ_OFF_Q2, sG = sbase + C::DQ_OFF_G;
            const uint32_t sR1 = sbase + C::DQ_OFF_RES, sR2 = sR1 + C::RBOX;
            auto k1_at = [&](int j) { return sbase + C::DQ_OFF_RING + (j % ST) * C::DQ_STAGE; };
            // dQ_b += dS_b K_b for sub-tile jj: A = dS_b (shared, K-major), B = K_b tile MN-major
            auto acc = [&](int jj) {
                const uint32_t sK1 = k1_at(jj), sK2 = (V2 || MODE == 1) ? sK1 : sK1 + C::QB * C::CBOX;
                const uint64_t a1 = sdesc_sw128(sR1, 16, 1024), a2 = sdesc_sw128(sR2, 16, 1024);
                const uint64_t k1 = sdesc_sw128(sK1, C::CBOX, 1024), k2 = sdesc_sw128(sK2, C::CBOX, 1024);
#pragma unroll
                for (int ks = 0; ks < C::BN / 16; ++ks) {
                    const uint32_t oa = (ks * 32) >> 4, ob = (ks * 2048) >> 4;
                    const uint32_t first = (jj > 0 || ks > 0) ? 1u : 0u;
                    mma_ss_elect(tmem + C::COL_DQ1, a1 + oa, k1 + ob, C::IDESC_QK, first);
                    if (MODE == 0) mma_ss_elect(tmem + C::COL_DQ2, a2 + oa, k2 + ob, C::IDESC_QK, first);
                }
                mma_commit_elect(bar_empty + 8 * (jj % ST));   // K, V of jj no longer needed
                mma_commit_elect(bar_rfree);                    // result tiles read
            };
            // S_b = Q_b K_b^T (N = 64 keys), dP = G V^T for sub-tile j
            auto scores = [&](int j) {
                const uint32_t sK1 = k1_at(j);
                const uint32_t sK2 = (V2 || MODE == 1) ? sK1 : sK1 + C::QB * C::CBOX;
                const uint32_t sV = sK1 + C::NKT * C::QB * C::CBOX;
                const uint64_t a1 = sdesc_sw128(sQ1, 16, 1024), a2 = sdesc_sw128(sQ2, 16, 1024);
                const uint64_t b1 = sdesc_sw128(sK1, 16, 1024), b2 = sdesc_sw128(sK2, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DQK / 16; ++ks) {
                    const uint32_t oa = ((ks >> 2) * C::RBOX + (ks & 3) * 32) >> 4;
                    const uint32_t ob = ((ks >> 2) * C::CBOX + (ks & 3) * 32) >> 4;
                    mma_ss_elect(tmem + C::COL_S1, a1 + oa, b1 + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                    if (MODE == 0) mma_ss_elect(tmem + C::COL_S2, a2 + oa, b2 + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                }
                const uint64_t ag = sdesc_sw128(sG, 16, 1024), bv = sdesc_sw128(sV, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DV / 16; ++ks) {
                    const uint32_t oa = ((ks >> 2) * C::RBOX + (ks & 3) * 32) >> 4;
                    const uint32_t ob = ((ks >> 2) * C::CBOX + (ks & 3) * 32) >> 4;
                    mma_ss_elect(tmem + C::COL_DP, ag + oa, bv + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                }
                mma_commit_elect(bar_s);
            };
            // S(j) needs sub-tile j in the ring and the rows done loading S(j-1)
            auto wait_scores = [&](int j) {
                return wait_c(bar_full + 8 * (j % ST), static_cast<uint32_t>((j / ST) & 1), p.err) &&
                       (j == 0 || wait_c(bar_sfree, static_cast<uint32_t>((j - 1) & 1), p.err));
            };
            if (C::TWO_ISSUERS && warp == 1) {
                bool ok = wait_c(bar_res, 0, p.err);
                for (int j = 0; ok && j < n_kv; ++j) {
                    ok = wait_scores(j);
                    if (!ok) break;
                    tc_fence_after();
                    scores(j);
                }
                // no MMA of this thread may be in flight when TMEM is released
                mma_commit_elect(bar_dra);
                warp_wait_drain(bar_dra, 0, p.err);
            } else if (C::TWO_ISSUERS) {
                // dQ(j) waits for the rows' dS(j), which they form after S(j) completed
                bool ok = true;
                for (int j = 0; ok && j < n_kv; ++j) {
                    ok = wait_c(bar_rready, static_cast<uint32_t>(j & 1), p.err);
                    if (!ok) break;
                    tc_fence_after();
                    acc(j);
                }
                mma_commit_elect(bar_done);
                mma_commit_elect(bar_dr);
                warp_wait_drain(bar_dr, 0, p.err);
            } else {
                bool ok = wait_c(bar_res, 0, p.err);
                int j = 0;
                for (; ok && j < n_kv; ++j) {
                    ok = wait_scores(j);
                    if (!ok) break;
                    tc_fence_after();
                    scores(j);
                    if (j > 0) {
                        ok = wait_c(bar_rready, static_cast<uint32_t>((j - 1) & 1), p.err);
                        if (!ok) break;
                        tc_fence_after();
                        acc(j - 1);
                    }
                }
                if (ok && j == n_kv && wait_c(bar_rready, static_cast<uint32_t>((n_kv - 1) & 1), p.err)) {
                    tc_fence_after();
                    acc(n_kv - 1);
                }
                mma_commit_elect(bar_done);
                // no MMA may be in flight when TMEM is released
                mma_commit_elect(bar_dr);
                warp_wait_drain(bar_dr, 0, p.err);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ rows (query i)
        constexpr int RC = C::RC;
        const int wq = warp & 3, wg = (warp - 4) >> 2;   // lane quadrant, key part
        const int row = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const int t = qt * C::BM + row;
        const bool live = t < p.T;
        const int64_t vi = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
        const int64_t vstride = static_cast<int64_t>(p.B) * p.H * p.T;
        // MODE 1: branch 2's values sit in the first pair (lse1, d1): one formula below
        const int64_t v1i = vi + (MODE == 1 && brc ? vstride : 0);
        const float lse1 = live ? p.lse[v1i] : 0.f, lse2 = live && MODE == 0 ? p.lse[vstride + vi] : 0.f;
        const float d1 = live ? p.dd[v1i] : 0.f, d2 = live && MODE == 0 ? p.dd[vstride + vi] : 0.f;
        const float cc = live ? p.cv[vi] : 0.f;
        // dS_b = P_b (cb dP - D_b): cb = 1 for branch 1, c for branch 2
        const float cb1 = (MODE == 1 && brc) ? cc : 1.f;
        const float sl2 = p.scale_log2;
        uint8_t *res1 = smem + C::DQ_OFF_RES, *res2 = res1 + C::RBOX;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            ok = warp_wait(bar_s, static_cast<uint32_t>(j & 1), p.err, ok);
            uint32_t s1[RC], s2[RC], dp[RC];
            if (ok) {
                tc_fence_after();
                tmem_ld_cols<RC>(tmem + lane_off + C::COL_S1 + RC * wg, s1);
                if (MODE == 0) tmem_ld_cols<RC>(tmem + lane_off + C::COL_S2 + RC * wg, s2);
                tmem_ld_cols<RC>(tmem + lane_off + C::COL_DP + RC * wg, dp);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elect(bar_sfree);   // the next S, dP may overwrite TMEM
            if (ok) {
                const int key0 = j * C::BN + RC * wg;
                // every key of this part is at or before every query of the tile: no mask
                const bool full = key0 + RC - 1 <= qt * C::BM;
                // two unrolled copies: without the per-element mask where it is all true
                // two columns at a time on the packed fp32 pipe (the same roundings per element)
                auto form = [&](auto masked) {
                    const float2 sc2 = make_float2(sl2, sl2), cc2 = make_float2(cc, cc);
                    const float2 nl1 = make_float2(-lse1, -lse1), nl2 = make_float2(-lse2, -lse2);
                    const float2 nd1 = make_float2(-d1, -d1), nd2 = make_float2(-d2, -d2);
                    const float2 cb2 = make_float2(cb1, cb1);
#pragma unroll
                    for (int c = 0; c < RC; c += 2) {
                        const float2 dpv = make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1]));
                        const float2 x1 =
                            __ffma2_rn(make_float2(__uint_as_float(s1[c]), __uint_as_float(s1[c + 1])), sc2, nl1);
                        float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                        if (decltype(masked)::value) {
                            const bool v0 = live && key0 + c <= t, v1 = live && key0 + c + 1 <= t;
                            p1 = make_float2(v0 ? p1.x : 0.f, v1 ? p1.y : 0.f);
                        }
                        if constexpr (MODE == 1) {
                            // one branch: dS = P (cb dP - D)
                            const float2 r1 = __fmul2_rn(p1, __ffma2_rn(cb2, dpv, nd1));
                            s1[c] = __float_as_uint(r1.x);
                            s1[c + 1] = __float_as_uint(r1.y);
                        } else {
                            const float2 x2 =
                                __ffma2_rn(make_float2(__uint_as_float(s2[c]), __uint_as_float(s2[c + 1])), sc2, nl2);
                            float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
                            if (decltype(masked)::value) {
                                const bool v0 = live && key0 + c <= t, v1 = live && key0 + c + 1 <= t;
                                p2 = make_float2(v0 ? p2.x : 0.f, v1 ? p2.y : 0.f);
                            }
                            const float2 r1 = __fmul2_rn(p1, __fadd2_rn(dpv, nd1));
                            const float2 r2 = __fmul2_rn(p2, __ffma2_rn(cc2, dpv, nd2));
                            s1[c] = __float_as_uint(r1.x);
                            s1[c + 1] = __float_as_uint(r1.y);
                            s2[c] = __float_as_uint(r2.x);
                            s2[c + 1] = __float_as_uint(r2.y);
                        }
                    }
                };
                if (live && full)
                    form(std::false_type{});
                else
                    form(std::true_type{});
            }
            // the previous dQ MMAs must have read the result tiles
            if (j > 0) ok = warp_wait(bar_rfree, static_cast<uint32_t>((j - 1) & 1), p.err, ok);
            if (ok) {
                uint32_t u[RC / 2];
                pack_cols<RC>(s1, u);
                store_row_part<RC>(res1, row, wg, u);
                if (MODE == 0) {
                    pack_cols<RC>(s2, u);
                    store_row_part<RC>(res2, row, wg, u);
                }
                fence_async_smem();   // generic-proxy writes -> tensor core reads
            }
            __syncwarp();
            mbar_arrive_elect(bar_rready);
        }
        // epilogue: dQ_b * scale -> bf16 rows (MODE 0: warpgroup wg takes branch
        // wg % 2, channels DQK / (NRG / 2) * (wg / 2) onwards; MODE 1: this CTA's
        // branch, channels DQK / NRG * wg onwards, from the first accumulator)
        ok = warp_wait(bar_done, 0, p.err, ok);
        tc_fence_after();
        if (ok) {
            constexpr int NCH = MODE == 1 ? DQK / C::NRG : DQK / (C::NRG / 2);
            const int br = MODE == 1 ? brc : (wg & 1), ch0 = MODE == 1 ? NCH * wg : NCH * (wg >> 1);
            const int acol = (MODE == 0 && br) ? C::COL_DQ2 : C::COL_DQ1;
            __nv_bfloat16 *dst = (br ? p.dq2 : p.dq1) + b * p.q_sb + static_cast<int64_t>(t) * p.q_st +
                                 static_cast<int64_t>(br ? hq2 : hq1) * p.q_sh + ch0;
#pragma unroll
            for (int c0 = 0; c0 < NCH; c0 += 32) {
                if (ch0 + c0 >= p.dqk_store) break;   // zero-padded channels
                uint32_t a[32];
                tmem_ld32(tmem + lane_off + acol + ch0 + c0, a);
                tmem_wait_ld();
                if (live && DA_CHECK(b < p.B && ch0 + c0 + 32 <= DQK, p.err)) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const uint32_t *aa = a + 8 * q8;
                        d4[q8] = make_uint4(
                            pack_bf16(__uint_as_float(aa[0]) * p.scale, __uint_as_float(aa[1]) * p.scale),
                            pack_bf16(__uint_as_float(aa[2]) * p.scale, __uint_as_float(aa[3]) * p.scale),
                            pack_bf16(__uint_as_float(aa[4]) * p.scale, __uint_as_float(aa[5]) * p.scale),
                            pack_bf16(__uint_as_float(aa[6]) * p.scale, __uint_as_float(aa[7]) * p.scale));
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// =================================================================== dK dV
// Same pipeline over 64-query sub-tiles (items; V2: of every pair of the kv
// group): S1^T, S2^T, dP^T of item i run while the rows turn item i-1 into
// P~^T = P1^T + c P2^T, dS1^T, dS2^T; dV += P~^T G, dK_b += dS_b^T Q_b read
// those from shared memory.
template <int DQK, int DV, bool V2, int MODE = 0>
__global__ void __launch_bounds__(BwdCfg<DQK, DV, V2, MODE>::THREADS, 1)
    bwd_dkdv(const __grid_constant__ CUtensorMap tk1, const __grid_constant__ CUtensorMap tk2,
             const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq1,
             const __grid_constant__ CUtensorMap tq2, const __grid_constant__ CUtensorMap tg, const BwdParams p) {
    using C = BwdCfg<DQK, DV, V2, MODE>;
    constexpr int ST = C::KV_STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // tile w -> key tile (heaviest = earliest first), head (V1) / kv head (V2), batch
    const int n_kt = (p.T + C::BM - 1) / C::BM;
    const int nh = V2 ? p.Hkv : p.H;
    const int per_kt = nh * p.B;
    // MODE 1: the two branches of a key tile are neighbouring CTAs, branch = index & 1
    const int w = static_cast<int>(blockIdx.x) >> (MODE == 1 ? 1 : 0);
    const int brc = MODE == 1 ? static_cast<int>(blockIdx.x & 1u) : 0;
    const int kt = w / per_kt, rest = w % per_kt;
    const int hk = rest % nh, b = rest / nh;
    const int n_qs = (p.T + C::BN - 1) / C::BN;
    const int i0 = kt * (C::BM / C::BN);
    const int nq = n_qs - i0;                       // query sub-tiles at or after the diagonal
    const int npairs = V2 ? p.G / 2 : 1;
    const int n_items = npairs * nq;
    // item -> (pair or head for the row vectors, query sub-tile)
    auto item_head = [&](int it) { return V2 ? hk * (p.G / 2) + it / nq : hk; };
    auto item_qs = [&](int it) { return i0 + it % nq; };

    const uint32_t bar_res = sbase + C::KV_OFF_BAR;
    const uint32_t bar_full = bar_res + 8;
    const uint32_t bar_empty = bar_full + 8 * ST;
    const uint32_t bar_s = bar_empty + 8 * ST;
    const uint32_t bar_sfree = bar_s + 8;
    const uint32_t bar_rready = bar_sfree + 8;
    const uint32_t bar_rfree = bar_rready + 8;
    const uint32_t bar_done = bar_rfree + 8;
    const uint32_t bar_dr = bar_done + 8;
    const uint32_t bar_dra = bar_dr + 8;
    const uint32_t tslot = sbase + C::KV_OFF_TSLOT;

    if (threadIdx.x == 0) {
        mbar_init(bar_res, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_full + 8 * s, 1 + 32);   // TMA bytes + 32 lanes' row vectors
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_s, 1);
        mbar_init(bar_sfree, 4 * C::NRG);   // one arrival per row warp
        mbar_init(bar_rready, 4 * C::NRG);
        mbar_init(bar_rfree, 1);
        mbar_init(bar_done, 1);
        mbar_init(bar_dr, 1);
        mbar_init(bar_dra, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::KV_OFF_TSLOT);
    const int64_t vstride = static_cast<int64_t>(p.B) * p.H * p.T;

    if (warp == 0) {
        // ------------------------------------------ TMA + row vectors (32 lanes)
        // MODE 1: only this branch's K and Q
        const CUtensorMap *mk = (MODE == 1 && brc) ? &tk2 : &tk1;
        const CUtensorMap *mq = (MODE == 1 && brc) ? &tq2 : &tq1;
        auto wait_c = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
            return warp_wait_vote(bar, parity, err, true);
        };
        {
            prefetch_tmap(mk);
            prefetch_tmap(&tv);
            prefetch_tmap(mq);
            prefetch_tmap(&tg);
            mbar_arrive_expect_tx_elect(bar_res, C::NKT * C::QB * C::RBOX + (C::HAS_DP ? C::VB * C::RBOX : 0));
#pragma unroll
            for (int c = 0; c < C::QB; ++c) {
                tma_load_4d_elect(sbase + C::KV_OFF_K1 + c * C::RBOX, mk, bar_res, 64 * c, hk, kt * C::BM, b);
                if (!V2 && MODE != 1)
                    tma_load_4d_elect(sbase + C::KV_OFF_K2 + c * C::RBOX, &tk2, bar_res, 64 * c, hk, kt * C::BM, b);
            }
            if (C::HAS_DP) {
#pragma unroll
                for (int c = 0; c < C::VB; ++c)
                    tma_load_4d_elect(sbase + C::KV_OFF_V + c * C::RBOX, &tv, bar_res, 64 * c, hk, kt * C::BM, b);
            }
        }
        bool ok = true;
        int it = 0;
        for (; ok && it < n_items; ++it) {
            const int st = it % ST;
            if (it >= ST) ok = warp_wait_vote(bar_empty + 8 * st, static_cast<uint32_t>((it / ST - 1) & 1), p.err, ok);
            if (!ok) break;
            const int hp = item_head(it), qs = item_qs(it);
            const uint32_t dst = sbase + C::KV_OFF_RING + st * C::KV_STAGE;
            {
                const int hq1 = V2 ? 2 * hp : hp, hq2 = V2 ? 2 * hp + 1 : hp;
                mbar_arrive_expect_tx_elect(bar_full + 8 * st, C::KV_STAGE_TMA);
#pragma unroll
                for (int c = 0; c < C::QB; ++c) {
                    tma_load_4d_elect(dst + c * C::CBOX, mq, bar_full + 8 * st, 64 * c, (MODE == 1 && brc) ? hq2 : hq1,
                                qs * C::BN, b);
                    if (MODE != 1)
                        tma_load_4d_elect(dst + (C::QB + c) * C::CBOX, &tq2, bar_full + 8 * st, 64 * c, hq2, qs * C::BN, b);
                }
#pragma unroll
                for (int c = 0; c < C::VB; ++c)
                    tma_load_4d_elect(dst + (C::NQ * C::QB + c) * C::CBOX, &tg, bar_full + 8 * st, 64 * c, hp, qs * C::BN,
                                b);
            }
            // row vectors of the 64 query rows: lse (+inf past T so that P = 0), D, c
            float *vec = reinterpret_cast<float *>(smem + (dst - sbase) + C::KV_STAGE_TMA);
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int r = lane + 32 * r2;
                const int tq = qs * C::BN + r;
                const bool live = tq < p.T;
                const int64_t vi = (static_cast<int64_t>(b) * p.H + hp) * p.T + tq;
                vec[r] = live ? p.lse[vi] : INFINITY;
                vec[64 + r] = live ? p.lse[vstride + vi] : INFINITY;
                vec[128 + r] = live ? p.dd[vi] : 0.f;
                vec[192 + r] = live ? p.dd[vstride + vi] : 0.f;
                vec[256 + r] = live ? p.cv[vi] : 0.f;
            }
            mbar_arrive(bar_full + 8 * st);   // release: the vectors are visible to the waiters
        }
        // leave no copy in flight
        {
            warp_wait_drain(bar_res, 0, p.err);
            for (int k = (it > ST ? it - ST : 0); k < it; ++k)
                warp_wait_drain(bar_full + 8 * (k % ST), static_cast<uint32_t>((k / ST) & 1), p.err);
        }
    } else if (warp == 1 || (C::TWO_ISSUERS && warp == 2)) {
        // ------------------------------------------------------------ MMA
        {
            // the whole warp, converged; one elected lane issues each MMA and commit
            auto wait_c = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
                return warp_wait_vote(bar, parity, err, true);
            };
            const uint32_t sK1 = sbase + C::KV_OFF_K1, sK2 = (V2 || MODE == 1) ? sK1 : sbase + C::KV_OFF_K2;
            const uint32_t sV = sbase + C::KV_OFF_V;
            const uint32_t sRP = sbase + C::KV_OFF_RES, sR1 = sRP + C::RBOX, sR2 = sR1 + C::RBOX;
            auto q1_at = [&](int it) { return sbase + C::KV_OFF_RING + (it % ST) * C::KV_STAGE; };
            // dV += P~^T G; dK_b += dS_b^T Q_b for item jj (A = result tiles, B = MN-major sub-tiles)
            auto acc = [&](int jj) {
                const uint32_t sQ1 = q1_at(jj), sQ2 = sQ1 + C::QB * C::CBOX, sG = sQ1 + C::NQ * C::QB * C::CBOX;
                const uint64_t ap = sdesc_sw128(sRP, 16, 1024), a1 = sdesc_sw128(sR1, 16, 1024),
                               a2 = sdesc_sw128(sR2, 16, 1024);
                const uint64_t gdesc = sdesc_sw128(sG, C::CBOX, 1024);
                const uint64_t q1d = sdesc_sw128(sQ1, C::CBOX, 1024), q2d = sdesc_sw128(sQ2, C::CBOX, 1024);
#pragma unroll
                for (int ks = 0; ks < C::BN / 16; ++ks) {
                    const uint32_t oa = (ks * 32) >> 4, ob = (ks * 2048) >> 4;
                    const uint32_t first = (jj > 0 || ks > 0) ? 1u : 0u;
                    if constexpr (MODE == 1) {
                        // dK_b += dS_b^T Q_b: the one result tile sits first
                        mma_ss_elect(tmem + C::COL_DK1, ap + oa, q1d + ob, C::IDESC_QK, first);
                    } else if constexpr (MODE == 2) {
                        mma_ss_elect(tmem + C::COL_DV, ap + oa, gdesc + ob, C::IDESC_V, first);
                    } else {
                        mma_ss_elect(tmem + C::COL_DV, ap + oa, gdesc + ob, C::IDESC_V, first);
                        mma_ss_elect(tmem + C::COL_DK1, a1 + oa, q1d + ob, C::IDESC_QK, first);
                        mma_ss_elect(tmem + C::COL_DK2, a2 + oa, q2d + ob, C::IDESC_QK, V2 ? 1u : first);
                    }
                }
                mma_commit_elect(bar_empty + 8 * (jj % ST));   // Q, G of jj no longer needed
                mma_commit_elect(bar_rfree);                    // result tiles read
            };
            // S_b^T = K_b Q_b^T (N = 64 queries), dP^T = V G^T for item it
            auto scores = [&](int it) {
                const uint32_t sQ1 = q1_at(it);
                const uint32_t sQ2 = sQ1 + C::QB * C::CBOX, sG = sQ1 + C::NQ * C::QB * C::CBOX;
                const uint64_t a1 = sdesc_sw128(sK1, 16, 1024), a2 = sdesc_sw128(sK2, 16, 1024);
                const uint64_t b1 = sdesc_sw128(sQ1, 16, 1024), b2 = sdesc_sw128(sQ2, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DQK / 16; ++ks) {
                    const uint32_t oa = ((ks >> 2) * C::RBOX + (ks & 3) * 32) >> 4;
                    const uint32_t ob = ((ks >> 2) * C::CBOX + (ks & 3) * 32) >> 4;
                    mma_ss_elect(tmem + C::COL_S1, a1 + oa, b1 + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                    if (MODE != 1) mma_ss_elect(tmem + C::COL_S2, a2 + oa, b2 + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                }
                if (C::HAS_DP) {
                    const uint64_t av = sdesc_sw128(sV, 16, 1024), bg = sdesc_sw128(sG, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < DV / 16; ++ks) {
                        const uint32_t oa = ((ks >> 2) * C::RBOX + (ks & 3) * 32) >> 4;
                        const uint32_t ob = ((ks >> 2) * C::CBOX + (ks & 3) * 32) >> 4;
                        mma_ss_elect(tmem + C::COL_DP, av + oa, bg + ob, C::IDESC_S, ks > 0 ? 1u : 0u);
                    }
                }
                mma_commit_elect(bar_s);
            };
            // S(it) needs item it in the ring and the rows done loading S(it-1)
            auto wait_scores = [&](int it) {
                return wait_c(bar_full + 8 * (it % ST), static_cast<uint32_t>((it / ST) & 1), p.err) &&
                       (it == 0 || wait_c(bar_sfree, static_cast<uint32_t>((it - 1) & 1), p.err));
            };
            if (C::TWO_ISSUERS && warp == 1) {
                bool ok = wait_c(bar_res, 0, p.err);
                for (int it = 0; ok && it < n_items; ++it) {
                    ok = wait_scores(it);
                    if (!ok) break;
                    tc_fence_after();
                    scores(it);
                }
                // no MMA of this thread may be in flight when TMEM is released
                mma_commit_elect(bar_dra);
                warp_wait_drain(bar_dra, 0, p.err);
            } else if (C::TWO_ISSUERS) {
                // dV, dK(it) wait for the rows' P~, dS(it), formed after S(it) completed
                bool ok = true;
                for (int it = 0; ok && it < n_items; ++it) {
                    ok = wait_c(bar_rready, static_cast<uint32_t>(it & 1), p.err);
                    if (!ok) break;
                    tc_fence_after();
                    acc(it);
                }
                mma_commit_elect(bar_done);
                mma_commit_elect(bar_dr);
                warp_wait_drain(bar_dr, 0, p.err);
            } else {
                bool ok = wait_c(bar_res, 0, p.err);
                int it = 0;
                for (; ok && it < n_items; ++it) {
                    ok = wait_scores(it);
                    if (!ok) break;
                    tc_fence_after();
                    scores(it);
                    if (it > 0) {
                        ok = wait_c(bar_rready, static_cast<uint32_t>((it - 1) & 1), p.err);
                        if (!ok) break;
                        tc_fence_after();
                        acc(it - 1);
                    }
                }
                if (ok && it == n_items &&
                    wait_c(bar_rready, static_cast<uint32_t>((n_items - 1) & 1), p.err)) {
                    tc_fence_after();
                    acc(n_items - 1);
                }
                mma_commit_elect(bar_done);
                mma_commit_elect(bar_dr);
                warp_wait_drain(bar_dr, 0, p.err);
            }
        }
    } else if (warp >= 4) {
        // -------------------------------------------------- rows (key j)
        constexpr int RC = C::RC;
        const int wq = warp & 3, wg = (warp - 4) >> 2;   // lane quadrant, query part
        const int row = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const int j = kt * C::BM + row;
        const float sl2 = p.scale_log2;
        uint8_t *resP = smem + C::KV_OFF_RES, *res1 = resP + C::RBOX, *res2 = res1 + C::RBOX;
        bool ok = true;
        for (int it = 0; it < n_items; ++it) {
            const int st = it % ST;
            ok = warp_wait(bar_s, static_cast<uint32_t>(it & 1), p.err, ok);
            // the stage's row vectors were written by warp 0 before it arrived on
            // the stage's full barrier: acquire them there (that phase is complete)
            ok = warp_wait(bar_full + 8 * st, static_cast<uint32_t>((it / ST) & 1), p.err, ok);
            uint32_t s1[RC], s2[RC], dp[RC];
            if (ok) {
                tc_fence_after();
                tmem_ld_cols<RC>(tmem + lane_off + C::COL_S1 + RC * wg, s1);
                if (MODE != 1) tmem_ld_cols<RC>(tmem + lane_off + C::COL_S2 + RC * wg, s2);
                if (C::HAS_DP) tmem_ld_cols<RC>(tmem + lane_off + C::COL_DP + RC * wg, dp);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            mbar_arrive_elect(bar_sfree);   // the next S^T, dP^T may overwrite TMEM
            if (ok) {
                // this warpgroup's RC query columns of the row vectors, 16 bytes at a time
                const float4 *vec = reinterpret_cast<const float4 *>(smem + C::KV_OFF_RING + st * C::KV_STAGE +
                                                                     C::KV_STAGE_TMA) + RC / 4 * wg;
                const int q0 = item_qs(it) * C::BN + RC * wg;
                // every query of this part is at or after every key of the tile: no mask
                const bool full = q0 >= kt * C::BM + C::BM - 1;
                // in place: s1 <- P~ = P1 + c P2, s2 <- dS1, dp <- dS2 (MODE 1: s1 <- dS_b;
                // MODE 2: s1 <- P~); two unrolled copies, without the per-element mask
                // where it is all true
                auto form = [&](auto masked) {
#pragma unroll
                    for (int c4 = 0; c4 < RC / 4; ++c4) {
                        // MODE 1, branch 2: its lse and D in the place of branch 1's
                        const float4 l1 = vec[(MODE == 1 && brc ? 16 : 0) + c4], l2 = vec[16 + c4],
                                     e1 = vec[(MODE == 1 && brc ? 48 : 32) + c4], e2 = vec[48 + c4], cv = vec[64 + c4];
                        const float l1a[4] = {l1.x, l1.y, l1.z, l1.w}, l2a[4] = {l2.x, l2.y, l2.z, l2.w};
                        const float e1a[4] = {e1.x, e1.y, e1.z, e1.w}, e2a[4] = {e2.x, e2.y, e2.z, e2.w};
                        const float cva[4] = {cv.x, cv.y, cv.z, cv.w};
                        // two columns at a time on the packed fp32 pipe (the same roundings per element)
#pragma unroll
                        for (int k = 0; k < 4; k += 2) {
                            const int c = 4 * c4 + k;
                            const float2 sc2 = make_float2(sl2, sl2), cv2 = make_float2(cva[k], cva[k + 1]);
                            const float2 dpv = make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1]));
                            const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(s1[c]), __uint_as_float(s1[c + 1])),
                                                         sc2, make_float2(-l1a[k], -l1a[k + 1]));
                            const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(s2[c]), __uint_as_float(s2[c + 1])),
                                                         sc2, make_float2(-l2a[k], -l2a[k + 1]));
                            float2 p1 = make_float2(ex2(x1.x), ex2(x1.y)), p2 = make_float2(ex2(x2.x), ex2(x2.y));
                            if (decltype(masked)::value) {
                                // key j <= query q0 + c; rows past T carry lse = +inf
                                const bool v0 = q0 + c >= j, v1 = q0 + c + 1 >= j;
                                p1 = make_float2(v0 ? p1.x : 0.f, v1 ? p1.y : 0.f);
                                p2 = make_float2(v0 ? p2.x : 0.f, v1 ? p2.y : 0.f);
                            }
                            if constexpr (MODE == 1) {
                                // dS_b = P_b (cb dP - D_b), cb = 1 (branch 1) or c (branch 2)
                                const float2 cb2 = brc ? cv2 : make_float2(1.f, 1.f);
                                const float2 r1 = __fmul2_rn(p1, __ffma2_rn(cb2, dpv, make_float2(-e1a[k], -e1a[k + 1])));
                                s1[c] = __float_as_uint(r1.x);
                                s1[c + 1] = __float_as_uint(r1.y);
                            } else if constexpr (MODE == 2) {
                                const float2 r0 = __ffma2_rn(cv2, p2, p1);
                                s1[c] = __float_as_uint(r0.x);
                                s1[c + 1] = __float_as_uint(r0.y);
                            } else {
                                const float2 r0 = __ffma2_rn(cv2, p2, p1);
                                const float2 r1 = __fmul2_rn(p1, __fadd2_rn(dpv, make_float2(-e1a[k], -e1a[k + 1])));
                                const float2 r2 =
                                    __fmul2_rn(p2, __ffma2_rn(cv2, dpv, make_float2(-e2a[k], -e2a[k + 1])));
                                s1[c] = __float_as_uint(r0.x);
                                s1[c + 1] = __float_as_uint(r0.y);
                                s2[c] = __float_as_uint(r1.x);
                                s2[c + 1] = __float_as_uint(r1.y);
                                dp[c] = __float_as_uint(r2.x);
                                dp[c + 1] = __float_as_uint(r2.y);
                            }
                        }
                    }
                };
                if (full)
                    form(std::false_type{});
                else
                    form(std::true_type{});
            }
            // the previous item's dV / dK MMAs must have read the result tiles
            if (it > 0) ok = warp_wait(bar_rfree, static_cast<uint32_t>((it - 1) & 1), p.err, ok);
            if (ok) {
                uint32_t u[RC / 2];
                pack_cols<RC>(s1, u);
                store_row_part<RC>(resP, row, wg, u);
                if (MODE == 0) {
                    pack_cols<RC>(s2, u);
                    store_row_part<RC>(res1, row, wg, u);
                    pack_cols<RC>(dp, u);
                    store_row_part<RC>(res2, row, wg, u);
                }
                fence_async_smem();   // generic-proxy writes -> tensor core reads
            }
            __syncwarp();
            mbar_arrive_elect(bar_rready);
        }
        // epilogue: dK_b * scale, dV -> bf16 rows of key j
        ok = warp_wait(bar_done, 0, p.err, ok);
        tc_fence_after();
        if (ok) {
            const bool live = j < p.T;
            auto store = [&](int col, int n, __nv_bfloat16 *dst, float f) {
                for (int c0 = 0; c0 < n; c0 += 32) {
                    uint32_t a[32];
                    tmem_ld32(tmem + lane_off + col + c0, a);
                    tmem_wait_ld();
                    if (live && DA_CHECK(b < p.B && col + c0 + 32 <= static_cast<int>(C::TMEM_COLS), p.err)) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const uint32_t *aa = a + 8 * q8;
                            d4[q8] = make_uint4(pack_bf16(__uint_as_float(aa[0]) * f, __uint_as_float(aa[1]) * f),
                                                pack_bf16(__uint_as_float(aa[2]) * f, __uint_as_float(aa[3]) * f),
                                                pack_bf16(__uint_as_float(aa[4]) * f, __uint_as_float(aa[5]) * f),
                                                pack_bf16(__uint_as_float(aa[6]) * f, __uint_as_float(aa[7]) * f));
                        }
                    }
                }
            };
            // MODE 0: the first half of the warpgroups stores dK (both branches for V1),
            // the second half dV, each warpgroup an equal share of the channels;
            // MODE 1 / 2: every warpgroup an equal share of dK_b / dV
            constexpr int HG = C::NRG / 2;
            const int part = wg % HG;
            const int64_t krow = b * p.k_sb + static_cast<int64_t>(j) * p.k_st + static_cast<int64_t>(hk) * p.k_sh;
            if constexpr (MODE == 1) {
                constexpr int NK = DQK / C::NRG;
                const int nk = min(NK, p.dqk_store - NK * wg);
                if (nk > 0) store(C::COL_DK1 + NK * wg, nk, (brc ? p.dk2 : p.dk1) + krow + NK * wg, p.scale);
            } else if constexpr (MODE == 2) {
                constexpr int NV = DV / C::NRG;
                store(C::COL_DV + NV * wg, NV,
                      p.dv + b * p.v_sb + static_cast<int64_t>(j) * p.v_st + static_cast<int64_t>(hk) * p.v_sh +
                          NV * wg,
                      1.f);
            } else if (wg < HG) {
                constexpr int NK = DQK / HG;
                // only the stored channels (the rest are zero padding)
                const int nk = min(NK, p.dqk_store - NK * part);
                store(C::COL_DK1 + NK * part, nk, p.dk1 + krow + NK * part, p.scale);
                if (!V2) store(C::COL_DK2 + NK * part, nk, p.dk2 + krow + NK * part, p.scale);
            } else {
                constexpr int NV = DV / HG;
                store(C::COL_DV + NV * part, NV,
                      p.dv + b * p.v_sb + static_cast<int64_t>(j) * p.v_st + static_cast<int64_t>(hk) * p.v_sh +
                          NV * part,
                      1.f);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ================================================================ row pass
// Per row (b, t, head (V1) / pair (V2)):
//   V1: x = a1 - lam a2 (saved by the forward), r = (mean(x^2) + 1e-5)^(-1/2), y = x r,
//       dy = (1 - lam_init) dout, dx = r (dy - y mean(dy y));
//       g = dx (bf16), D1 = dx . a1, D2 = -lam dx . a2, row share of
//       dL/dlam = -dx . a2.
//   V2: D1 = dout . a_e, D2 = -s dout . a_o, c = -s, dL/dlam = -s (1 - s)
//       dout . a_o with s = sigmoid(lam[t]).
// A row takes LPR = DV / 16 lanes of a warp, each holding 16 channels in four
// groups of four: lane j of the row owns channels 4 (j + LPR i) + k, i, k < 4,
// so that the row's lanes read consecutive 16-byte (fp32) or 8-byte (bf16)
// pieces with each instruction; a warp takes 32 / LPR rows at once and a
// row's sums need log2(LPR) shuffle steps.  (One warp per row, with four
// channels per lane, spent most of its issue slots on five-step shuffle
// reductions: 59 us against 41 us for this layout, measured on GB300 at the
// backward of the V1 B 4, T 2048, 16-head, d 64 workload.)
template <int DV>
struct PreCfgRows {
    static constexpr int LPR = DV / 16;                  // lanes per row
    static constexpr int RPW = 32 / LPR;                 // rows per warp
    static constexpr int ROWS = 8 * RPW;                 // rows per 256-thread block
    static_assert(DV == 64 || DV == 128 || DV == 256, "row pass: DV of 64, 128 or 256");
};

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void bf16x4_to_f32(uint2 u, float *dst) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    dst[0] = a.x; dst[1] = a.y; dst[2] = c.x; dst[3] = c.y;
}

template <int DV, bool V2>
__global__ void __launch_bounds__(256) bwd_pre(const BwdPreParams p) {
    using R = PreCfgRows<DV>;
    constexpr int LPR = R::LPR;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j = lane % LPR, rw = lane / LPR;                 // lane within its row; row within the warp
    const int row_in_block = warp * R::RPW + rw;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * R::ROWS + row_in_block;
    const int64_t nrows = static_cast<int64_t>(p.B) * p.T * p.H;
    const int h = static_cast<int>(r % p.H);
    const int t = static_cast<int>((r / p.H) % p.T);
    const int b = static_cast<int>(r / (static_cast<int64_t>(p.H) * p.T));
    // rows past the end compute on zeros and store nothing (the shuffles stay warp-wide)
    const bool live = r < nrows && DA_CHECK(b < p.B && t < p.T && h < p.H, p.err);
    float x1[16], x2[16], dy[16];
    const int64_t rbase = r * DV;
    const __nv_bfloat16 *go = p.dout + b * p.o_sb + static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(h) * p.o_sh;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = 4 * (j + LPR * i);
        if (live) {
            if constexpr (V2) {
                bf16x4_to_f32(*reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.sa1) + rbase + c),
                              x1 + 4 * i);
                bf16x4_to_f32(*reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.sa2) + rbase + c),
                              x2 + 4 * i);
            } else {
                const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.sa1) + rbase + c);
                const float4 e = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.sa2) + rbase + c);
                x1[4 * i] = a.x; x1[4 * i + 1] = a.y; x1[4 * i + 2] = a.z; x1[4 * i + 3] = a.w;
                x2[4 * i] = e.x; x2[4 * i + 1] = e.y; x2[4 * i + 2] = e.z; x2[4 * i + 3] = e.w;
            }
            bf16x4_to_f32(*reinterpret_cast<const uint2 *>(go + c), dy + 4 * i);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) x1[4 * i + k] = x2[4 * i + k] = dy[4 * i + k] = 0.f;
        }
    }
    const int64_t vi = (static_cast<int64_t>(b) * p.H + h) * p.T + t;
    const int64_t vstride = nrows;
    if constexpr (V2) {
        float e = 0.f, o = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            e = fmaf(dy[k], x1[k], e);
            o = fmaf(dy[k], x2[k], o);
        }
        e = group_sum<LPR>(e);
        o = group_sum<LPR>(o);
        if (live && j == 0) {
            const float s = 1.f / (1.f + expf(-p.lam[(static_cast<int64_t>(b) * p.T + t) * p.H + h]));
            p.dd[vi] = e;
            p.dd[vstride + vi] = -s * o;
            p.cv[vi] = -s;
            p.dlam[(static_cast<int64_t>(b) * p.T + t) * p.H + h] = -s * (1.f - s) * o;
        }
    } else {
        // lam_init = 0.8 - 0.6 exp(-0.3 layer); lam = exp(lq1 . lk1) - exp(lq2 . lk2) + lam_init,
        // once per block
        __shared__ float sh[2 + R::ROWS];
        if (warp == 0) {
            float s1 = 0.f, s2 = 0.f;
            for (int c = lane; c < p.d; c += 32) {
                s1 = fmaf(p.lq1[c], p.lk1[c], s1);
                s2 = fmaf(p.lq2[c], p.lk2[c], s2);
            }
            s1 = warp_sum(s1);
            s2 = warp_sum(s2);
            if (lane == 0) {
                const float li = 0.8f - 0.6f * expf(-0.3f * static_cast<float>(p.layer_index));
                sh[0] = expf(s1) - expf(s2) + li;
                sh[1] = li;
            }
        }
        __syncthreads();
        const float lam = sh[0], lam_init = sh[1];
        // x as the forward normalised it; a1 = x + lam a2
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            ss = fmaf(x1[k], x1[k], ss);
            dy[k] *= (1.f - lam_init);
        }
        ss = group_sum<LPR>(ss);
        const float rr = rsqrtf(ss / static_cast<float>(DV) + 1e-5f);
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) m = fmaf(dy[k], x1[k] * rr, m);
        m = group_sum<LPR>(m) / static_cast<float>(DV);
        float d1 = 0.f, d2 = 0.f, dl = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            alignas(8) __nv_bfloat16 gb[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float xv = x1[4 * i + k], a2v = x2[4 * i + k];
                const float dx = rr * (dy[4 * i + k] - xv * rr * m);
                // D is formed from the bf16 g that the dP product will use, so
                // that dP - D cancels where it should (one key: dP = D exactly)
                gb[k] = __float2bfloat16_rn(dx);
                const float gr = __bfloat162float(gb[k]);
                d1 = fmaf(gr, fmaf(lam, a2v, xv), d1);   // a1 = x + lam a2
                d2 = fmaf(gr, a2v, d2);
                dl = fmaf(dx, a2v, dl);
            }
            if (live) *reinterpret_cast<uint2 *>(p.g + rbase + 4 * (j + LPR * i)) = *reinterpret_cast<const uint2 *>(gb);
        }
        d1 = group_sum<LPR>(d1);
        d2 = group_sum<LPR>(d2);
        dl = group_sum<LPR>(dl);
        if (live && j == 0) {
            p.dd[vi] = d1;
            p.dd[vstride + vi] = -lam * d2;
            p.cv[vi] = -lam;
        }
        // the block's share of dL/dlam, its rows added in order (so the result
        // does not depend on scheduling); the lambda reduction then reads one
        // value per block
        if (j == 0) sh[2 + row_in_block] = live ? -dl : 0.f;
        __syncthreads();
        if (threadIdx.x == 0) {
            float acc = 0.f;
            for (int k = 0; k < R::ROWS; ++k) acc += sh[2 + k];
            p.dlam_rows[blockIdx.x] = acc;
        }
    }
}

// V1: dL/dlam = sum of the shares (one per row-pass block on the tensor-core
// path, one per row on the fp32 path; one CTA, fixed order), then the
// lambda-vector gradients dlq1 = dlam e1 lk1, dlk1 = dlam e1 lq1,
// dlq2 = -dlam e2 lk2, dlk2 = -dlam e2 lq2 with e_b = exp(lq_b . lk_b).
__global__ void __launch_bounds__(1024) bwd_lambda(const BwdPreParams p) {
    __shared__ float red[34];
    const int64_t n = p.n_shares;
    // eight independent 16-byte loads in flight per thread (the partials sit
    // at a 256-byte aligned workspace offset); fixed order, so deterministic
    const float4 *r4 = reinterpret_cast<const float4 *>(p.dlam_rows);
    const int64_t n4 = n / 4, nt = blockDim.x;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int64_t i = threadIdx.x;
    for (; i + 7 * nt < n4; i += 8 * nt) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = r4[i + k * nt];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] += (v[k].x + v[k].y) + (v[k].z + v[k].w);
    }
    for (; i < n4; i += nt) {
        const float4 v = r4[i];
        a[0] += (v.x + v.y) + (v.z + v.w);
    }
    for (int64_t j = n4 * 4 + threadIdx.x; j < n; j += nt) a[1] += p.dlam_rows[j];
    float acc = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    if (threadIdx.x < 32) {   // lq_b . lk_b, lanes over the d channels
        float s1 = 0.f, s2 = 0.f;
        for (int c = threadIdx.x; c < p.d; c += 32) {
            s1 = fmaf(p.lq1[c], p.lk1[c], s1);
            s2 = fmaf(p.lq2[c], p.lk2[c], s2);
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if (threadIdx.x == 0) {
            red[32] = s1;
            red[33] = s2;
        }
    }
    __syncthreads();
    float dlam = 0.f;
    for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) dlam += red[k];
    const float e1 = expf(red[32]), e2 = expf(red[33]);
    for (int c = threadIdx.x; c < p.d; c += blockDim.x) {
        p.dlq1[c] = dlam * e1 * p.lk1[c];
        p.dlk1[c] = dlam * e1 * p.lq1[c];
        p.dlq2[c] = -dlam * e2 * p.lk2[c];
        p.dlk2[c] = -dlam * e2 * p.lq2[c];
    }
}

template <int DQK, int DV, bool V2>
cudaError_t launch_bwd_t(const BwdMaps &m, const BwdParams &p, const BwdPreParams &pp, cudaStream_t s) {
    using C = BwdCfg<DQK, DV, V2>;
    static unsigned long long attr_done = 0;   // one bit per device
    cudaError_t ea = once_per_device(&attr_done, [] {
        cudaError_t e = cudaFuncSetAttribute(bwd_dq<DQK, DV, V2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::DQ_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_dkdv<DQK, DV, V2>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM);
        return e;
    });
    if (ea != cudaSuccess) return ea;
    const int64_t rows = static_cast<int64_t>(pp.B) * pp.T * pp.H;
    const int64_t pre_blocks = (rows + PreCfgRows<DV>::ROWS - 1) / PreCfgRows<DV>::ROWS;
    if (pre_blocks < 1 || pre_blocks > 0x7fffffff) return cudaErrorInvalidValue;
    BwdPreParams q = pp;
    q.n_shares = pre_blocks;   // V1: one share of dL/dlam per row-pass block
    bwd_pre<DV, V2><<<static_cast<unsigned>(pre_blocks), 256, 0, s>>>(q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!V2) {
        bwd_lambda<<<1, 1024, 0, s>>>(q);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t dq_tiles = static_cast<int64_t>((p.T + C::BM - 1) / C::BM) * p.H * p.B;
    const int64_t kv_tiles = static_cast<int64_t>((p.T + C::BM - 1) / C::BM) * (V2 ? p.Hkv : p.H) * p.B;
    if (dq_tiles > 0x7fffffff || kv_tiles > 0x7fffffff) return cudaErrorInvalidValue;
    bwd_dkdv<DQK, DV, V2><<<static_cast<unsigned>(kv_tiles), C::THREADS, C::KV_SMEM, s>>>(m.k1r, m.k2r, m.vr, m.q1c,
                                                                                          m.q2c, m.gc, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq<DQK, DV, V2><<<static_cast<unsigned>(dq_tiles), C::THREADS, C::DQ_SMEM, s>>>(m.q1r, m.q2r, m.gr, m.k1c,
                                                                                       m.k2c, m.vc, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_lambda(const BwdPreParams &pp, cudaStream_t s) {
    bwd_lambda<<<1, 1024, 0, s>>>(pp);
    return cudaGetLastError();
}

// DIFF V1 at d = 128 (dv = 256): per-branch dQ and dK kernels (two CTAs per
// tile) and a dV kernel, after the row pass and the lambda reduction.
cudaError_t launch_bwd_v1_d128(const BwdMaps &m, const BwdParams &p, const BwdPreParams &pp, cudaStream_t s) {
    using CQ = BwdCfg<128, 256, false, 1>;
    using CK = BwdCfg<128, 256, false, 1>;
    using CV = BwdCfg<128, 256, false, 2>;
    static unsigned long long attr_done = 0;   // one bit per device
    cudaError_t ea = once_per_device(&attr_done, [] {
        cudaError_t e = cudaFuncSetAttribute(bwd_dq<128, 256, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             CQ::DQ_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_dkdv<128, 256, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     CK::KV_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_dkdv<128, 256, false, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     CV::KV_SMEM);
        return e;
    });
    if (ea != cudaSuccess) return ea;
    const int64_t rows = static_cast<int64_t>(pp.B) * pp.T * pp.H;
    const int64_t pre_blocks = (rows + PreCfgRows<256>::ROWS - 1) / PreCfgRows<256>::ROWS;
    if (pre_blocks < 1 || pre_blocks > 0x7fffffff) return cudaErrorInvalidValue;
    BwdPreParams q = pp;
    q.n_shares = pre_blocks;   // one share of dL/dlam per row-pass block
    bwd_pre<256, false><<<static_cast<unsigned>(pre_blocks), 256, 0, s>>>(q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_lambda<<<1, 1024, 0, s>>>(q);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t tiles = static_cast<int64_t>((p.T + 127) / 128) * p.H * p.B;
    if (2 * tiles > 0x7fffffff) return cudaErrorInvalidValue;
    bwd_dkdv<128, 256, false, 1><<<static_cast<unsigned>(2 * tiles), CK::THREADS, CK::KV_SMEM, s>>>(
        m.k1r, m.k2r, m.vr, m.q1c, m.q2c, m.gc, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dkdv<128, 256, false, 2><<<static_cast<unsigned>(tiles), CV::THREADS, CV::KV_SMEM, s>>>(
        m.k1r, m.k2r, m.vr, m.q1c, m.q2c, m.gc, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq<128, 256, false, 1><<<static_cast<unsigned>(2 * tiles), CQ::THREADS, CQ::DQ_SMEM, s>>>(
        m.q1r, m.q2r, m.gr, m.k1c, m.k2c, m.vc, p);
    return cudaGetLastError();
}

bool backward_supported(int dqk, int dv, bool v2) {
    if (v2) return (dqk == 128 && dv == 128) || (dqk == 64 && dv == 64);
    return (dqk == 64 && dv == 128) || (dqk == 32 && dv == 64) || (dqk == 128 && dv == 256);
}

cudaError_t launch_backward(const BwdMaps &m, const BwdParams &p, const BwdPreParams &pp, int dqk, int dv, bool v2,
                            cudaStream_t s) {
    if (v2 && dqk == 128 && dv == 128) return launch_bwd_t<128, 128, true>(m, p, pp, s);
    if (v2 && dqk == 64 && dv == 64) return launch_bwd_t<64, 64, true>(m, p, pp, s);
    if (!v2 && dqk == 64 && dv == 128) return launch_bwd_t<64, 128, false>(m, p, pp, s);
    // d = 32: the q / k maps are 32 columns wide and their 64-column boxes are
    // zero-filled, so the d = 64 kernels compute the same S; the padded halves
    // of dq and dk come out zero and are not stored (p.dqk_store)
    if (!v2 && dqk == 32 && dv == 64) return launch_bwd_t<64, 64, false>(m, p, pp, s);
    if (!v2 && dqk == 128 && dv == 256) return launch_bwd_v1_d128(m, p, pp, s);
    return cudaErrorInvalidValue;
}

}  // namespace da
