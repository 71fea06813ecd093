// k_prefill_v1x2.cu -- DIFF V1 causal prefill in two passes over the keys,
// on tcgen05 tensor cores (bf16 in, fp32 accumulate).
//
// "Differential Transformer V2", DiffAttnV1: out = (1 - lam_init) *
// RMSNorm(softmax(Q1 K1^T/sqrt(d)) V - lam softmax(Q2 K2^T/sqrt(d)) V).
// Because softmax(.) V is linear in the probabilities, the difference can be
// taken before the value product:  a1 - lam a2 = (P1 - lam P2) V  with
// P_b = exp(S_b - m_b) / l_b -- the same identity as the materialised-weights
// form "(attn1 - lambda attn2) @ v" of the nanoGPT issue.  That needs the
// final row max m_b and sum l_b before any P is formed, hence two passes:
//
//   pass A  S1 = Q1 K1^T, S2 = Q2 K2^T per key tile; each branch's softmax
//           warpgroup keeps an exact online (m, l) per row.  S is double
//           buffered in TMEM so the next tile's products overlap the
//           exponentials of this one.
//   pass B  S1, S2 again; the two warpgroups split the 128 keys of a tile
//           (keys 0-63 and 64-127) and write P = e1/l1 - lam e2/l2 (bf16) to
//           TMEM; one accumulator O += P V (TS MMA, V MN-major).
//   epilogue  RMSNorm over the dv = 2d channels (eps 1e-5), (1 - lam_init)
//           scale, bf16 store.
//
// TMEM (512 columns): pass A uses all of it for S[buffer][branch]; pass B
// puts O in [0, dv) and S1, S2 after it.  With d = 64 (dv = 128) P has two
// buffers of its own, so the next tile's S1, S2 are computed as soon as this
// tile's have been read; with d = 128 (dv = 256) P is written over the part of
// S1 its own warpgroup has already read, so the next S2 is computed before
// the PV and only the next S1 follows it.
// With dv = 256 a key tile of V is 64 KB, so V streams in 32-key items.
//
// Roles: warp 0 TMA producer and warp 1 MMA issuer, each run by the whole
// warp converged with one lane chosen by elect.sync issuing (measured on
// GB300: 3 % faster at B1 T32768 H12 than lane 0 alone); warp 2 the lambda
// scalar; warps 4-11 two softmax warpgroups.  All waits of the converged
// warps are warp-uniform vote loops (warp_wait_vote).
//
// Executed work per causal (query, key) pair: 2d (S1) + 2d (S2) in each pass
// and 2 dv for the single PV = 12d, the same as two attentions with separate
// PV products; exponentials: 2 per pass.
#include "da_common.cuh"
#include "da_internal.h"

namespace da {
namespace {

template <int DQK>
struct V1x2Cfg {
    static constexpr int DV = 2 * DQK;
    static constexpr int BM = 128, BN = 128;
    static constexpr bool BIG = DQK == 128;          // dv = 256: P over S1, V in 32-key items
    static constexpr int QB = DQK / 64;
    static constexpr int BOX = 128 * 128;            // 128 rows x 64 bf16
    static constexpr int Q_TILE = QB * BOX;
    static constexpr int K_TILE = QB * BOX;
    // K ring item: K1 and K2 of a tile (d = 64) or one of them (d = 128)
    static constexpr int K_PER_ITEM = BIG ? 1 : 2;
    static constexpr int K_SLOT = K_PER_ITEM * K_TILE;   // 32 KB
    // ring depths (d = 128: measured on GB300, K 2 / V 5 deep 1167 TFLOP/s against
    // 1145 for 3 / 3 at B1 T32768 H12; the V items are 32 keys)
    static constexpr int KS = BIG ? 2 : 3;
    // V ring item: a whole key tile (d = 64) or 32 keys (d = 128, dv = 256)
    static constexpr int V_ROWS = BIG ? 32 : 128;
    static constexpr int V_ITEMS = BN / V_ROWS;
    static constexpr int VB = DV / 64;
    static constexpr int V_BOX = V_ROWS * 128;
    static constexpr int V_SLOT = VB * V_BOX;            // 32 KB or 16 KB
    static constexpr int VS = BIG ? 5 : 2;
    static constexpr int OFF_Q1 = 0, OFF_Q2 = Q_TILE;
    static constexpr int OFF_K = 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * K_SLOT;
    static constexpr int OFF_X = OFF_V + VS * V_SLOT;    // 4 x 128 floats
    static constexpr int OFF_BAR = OFF_X + 4 * 128 * 4;
    // q, kf[KS], ke[KS], vf[VS], ve[VS], saf[2][2], sae[2], sbf, sbe, pb[2], pfree[2], o, drain, lam
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 4 + 2 + 2 + 2 + 2 + 3;
    static constexpr int OFF_LAM = OFF_BAR + NBAR * 8;
    static constexpr int OFF_TSLOT = OFF_LAM + 8;
    static constexpr int SMEM = OFF_TSLOT + 8 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int COL_O = 0, COL_S1 = DV, COL_S2 = DV + 128;
    static constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(BM, DV, true);
    static constexpr uint32_t REGS_LOW = 56, REGS_HIGH = 208;
    static constexpr int REGS_NEEDED_AT_LAUNCH = (128 * REGS_LOW + 256 * REGS_HIGH + 383) / 384;
    static_assert(COL_S2 + 128 <= 512, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    // TMEM column of half h (keys 64h .. 64h+63) of P for tile j
    __device__ static constexpr int p_col(int j, int h) {
        return BIG ? COL_S1 + 64 * h : 384 + 64 * (j & 1) + 32 * h;
    }
};

// sum over 128 scores of 2^(s*scale - m)
__device__ __forceinline__ float sum_exp128(const uint32_t *s, float scale, float m) {
    const float2 sc2 = make_float2(scale, scale);
    const float2 nm2 = make_float2(-m, -m);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
    for (int c = 0; c < 64; ++c) {
        const float2 x =
            __ffma2_rn(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nm2);
        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
        switch (c & 3) {
            case 0: acc0 = __fadd2_rn(acc0, pp); break;
            case 1: acc1 = __fadd2_rn(acc1, pp); break;
            case 2: acc2 = __fadd2_rn(acc2, pp); break;
            default: acc3 = __fadd2_rn(acc3, pp); break;
        }
    }
    const float2 t = __fadd2_rn(__fadd2_rn(acc0, acc1), __fadd2_rn(acc2, acc3));
    return t.x + t.y;
}

// TRAIN (the training forward, DQK = 128): run 1 saves each branch's row
// log-sum-exp (log2 units, m + log2 l of pass A) and x = a1 - lam a2 (fp32,
// the RMSNorm input) besides the output; run 2 (A2) saves a2 (fp32) and
// writes no output: with branch 2's log-sum-exp known from run 1 it needs
// neither pass A nor branch 1, so it loads Q2, K2 and V only and computes
// S2 and P = 2^(s2 scale - lse2) = e2 / l2 once per key (half the products
// and a quarter of the exponentials of run 1).
template <int DQK, bool TRAIN = false, bool A2 = false>
__global__ void __launch_bounds__(384, 1)
    prefill_v1_twopass(const __grid_constant__ CUtensorMap tq1, const __grid_constant__ CUtensorMap tq2,
                       const __grid_constant__ CUtensorMap tk1, const __grid_constant__ CUtensorMap tk2,
                       const __grid_constant__ CUtensorMap tv, const PrefillParams p) {
    using C = V1x2Cfg<DQK>;
    static_assert(!A2 || (TRAIN && DQK == 128), "the a2 run: training forward, d = 128");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int n_qt = (p.T + C::BM - 1) / C::BM;
    const int per_qt = p.H * p.B;
    const int qt = n_qt - 1 - static_cast<int>(blockIdx.x) / per_qt;
    const int rest = static_cast<int>(blockIdx.x) % per_qt;
    const int h = rest % p.H, b = rest / p.H;
    const int q0 = qt * C::BM;
    const int n = qt + 1;

    const uint32_t bar_q = sbase + C::OFF_BAR;
    const uint32_t bar_kf = bar_q + 8;
    const uint32_t bar_ke = bar_kf + 8 * C::KS;
    const uint32_t bar_vf = bar_ke + 8 * C::KS;
    const uint32_t bar_ve = bar_vf + 8 * C::VS;
    const uint32_t bar_saf = bar_ve + 8 * C::VS;   // [buffer][branch]: pass-A S ready
    const uint32_t bar_sae = bar_saf + 32;         // [buffer]: pass-A S read by both branches
    const uint32_t bar_sbf = bar_sae + 16;         // pass-B S1, S2 ready
    const uint32_t bar_sbe = bar_sbf + 8;          // pass-B S1, S2 read
    const uint32_t bar_pb = bar_sbe + 8;           // [half]: P half written
    const uint32_t bar_pfree = bar_pb + 16;        // [P buffer]: PV done with it
    const uint32_t bar_o = bar_pfree + 16;
    const uint32_t bar_dr = bar_o + 8;
    const uint32_t bar_lam = bar_dr + 8;
    const uint32_t sQ1 = sbase + C::OFF_Q1, sQ2 = sbase + C::OFF_Q2;
    float *lam_smem = reinterpret_cast<float *>(smem + C::OFF_LAM);
    float *xch = reinterpret_cast<float *>(smem + C::OFF_X);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar_kf + 8 * s, 1);
            mbar_init(bar_ke + 8 * s, 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(bar_vf + 8 * s, 1);
            mbar_init(bar_ve + 8 * s, 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar_saf + 8 * i, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_sae + 8 * i, 8);
            mbar_init(bar_pb + 8 * i, 4);
            mbar_init(bar_pfree + 8 * i, 1);
        }
        mbar_init(bar_sbf, 1);
        mbar_init(bar_sbe, 8);
        mbar_init(bar_o, 1);
        mbar_init(bar_dr, 1);
        mbar_init(bar_lam, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + C::OFF_TSLOT, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::OFF_TSLOT);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        regs_decrease<C::REGS_LOW>();
        {
            // the whole warp, converged; one elected lane issues each copy
            auto wait_p = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
                return warp_wait_vote(bar, parity, err, true);
            };
            prefetch_tmap(&tq1);
            prefetch_tmap(&tq2);
            prefetch_tmap(&tk1);
            prefetch_tmap(&tk2);
            prefetch_tmap(&tv);
            mbar_arrive_expect_tx_elect(bar_q, (A2 ? 1 : 2) * C::Q_TILE);
#pragma unroll
            for (int c = 0; c < C::QB; ++c) {
                if (!A2) tma_load_4d_elect(sQ1 + c * C::BOX, &tq1, bar_q, 64 * c, h, q0, b);
                tma_load_4d_elect(sQ2 + c * C::BOX, &tq2, bar_q, 64 * c, h, q0, b);
            }
            int ki = 0, vi = 0;
            bool ok = true;
            // K ring item for tile j; `which` selects K1 / K2 when an item holds one of them
            auto load_k = [&](int j, int which) {
                const int st = ki % C::KS;
                if (ki >= C::KS && !wait_p(bar_ke + 8 * st, static_cast<uint32_t>((ki / C::KS - 1) & 1), p.err))
                    return false;
                const uint32_t dst = sbase + C::OFF_K + st * C::K_SLOT;
                mbar_arrive_expect_tx_elect(bar_kf + 8 * st, C::K_SLOT);
#pragma unroll
                for (int c = 0; c < C::QB; ++c) {
                    if (C::BIG) {
                        tma_load_4d_elect(dst + c * C::BOX, which ? &tk2 : &tk1, bar_kf + 8 * st, 64 * c, h, j * C::BN, b);
                    } else {
                        tma_load_4d_elect(dst + c * C::BOX, &tk1, bar_kf + 8 * st, 64 * c, h, j * C::BN, b);
                        tma_load_4d_elect(dst + C::K_TILE + c * C::BOX, &tk2, bar_kf + 8 * st, 64 * c, h, j * C::BN, b);
                    }
                }
                ++ki;
                return true;
            };
            auto load_tile_k = [&](int j) {
                if (!load_k(j, 0)) return false;
                return C::BIG ? load_k(j, 1) : true;
            };
            auto load_v = [&](int j, int item) {
                const int st = vi % C::VS;
                if (vi >= C::VS && !wait_p(bar_ve + 8 * st, static_cast<uint32_t>((vi / C::VS - 1) & 1), p.err))
                    return false;
                const uint32_t dst = sbase + C::OFF_V + st * C::V_SLOT;
                mbar_arrive_expect_tx_elect(bar_vf + 8 * st, C::V_SLOT);
#pragma unroll
                for (int c = 0; c < C::VB; ++c)
                    tma_load_4d_elect(dst + c * C::V_BOX, &tv, bar_vf + 8 * st, 64 * c, h, j * C::BN + item * C::V_ROWS, b);
                ++vi;
                return true;
            };
            // pass A: K tiles in order (none for the a2 run)
            for (int j = 0; !A2 && ok && j < n; ++j) ok = load_tile_k(j);
            // pass B, in the order the MMA warp consumes the items (the a2 run: K2 items only)
            if (ok) ok = A2 ? load_k(0, 1) : load_tile_k(0);
            for (int j = 0; ok && j < n; ++j) {
                if (C::BIG) {
                    // K2 of the next tile first: its S2 is computed before this tile's PV
                    if (j + 1 < n) ok = load_k(j + 1, 1);
                    for (int it = 0; ok && it < C::V_ITEMS; ++it) ok = load_v(j, it);
                    if (!A2 && ok && j + 1 < n) ok = load_k(j + 1, 0);
                } else {
                    if (j + 1 < n) ok = load_tile_k(j + 1);
                    if (ok) ok = load_v(j, 0);
                }
            }
            // leave no copy in flight
            warp_wait_drain(bar_q, 0, p.err);
            for (int k = (ki > C::KS ? ki - C::KS : 0); k < ki; ++k)
                warp_wait_drain(bar_kf + 8 * (k % C::KS), static_cast<uint32_t>((k / C::KS) & 1), p.err);
            for (int k = (vi > C::VS ? vi - C::VS : 0); k < vi; ++k)
                warp_wait_drain(bar_vf + 8 * (k % C::VS), static_cast<uint32_t>((k / C::VS) & 1), p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        regs_decrease<C::REGS_LOW>();
        {
            // the whole warp, converged; one elected lane issues each MMA and commit
            auto wait_i = [&](uint32_t bar, uint32_t parity, uint32_t *err) {
                return warp_wait_vote(bar, parity, err, true);
            };
            int ki = 0, vi = 0;
            auto wait_k = [&]() {
                return wait_i(bar_kf + 8 * (ki % C::KS), static_cast<uint32_t>((ki / C::KS) & 1), p.err);
            };
            auto k_at = [&]() { return sbase + C::OFF_K + (ki % C::KS) * C::K_SLOT; };
            auto issue_qk = [&](uint32_t dcol, uint32_t sq, uint32_t sk) {
                const uint64_t da = sdesc_sw128(sq, 16, 1024), db = sdesc_sw128(sk, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DQK / 16; ++ks) {
                    const uint32_t off = ((ks >> 2) * C::BOX + (ks & 3) * 32) >> 4;
                    mma_ss_elect(tmem + dcol, da + off, db + off, C::IDESC_QK, ks > 0 ? 1u : 0u);
                }
            };
            // S1 -> col1, S2 -> col2 for the next tile's K items; commits the K slots.
            auto qk_pair = [&](uint32_t col1, uint32_t col2, uint32_t bar1, uint32_t bar2) {
                if (!wait_k()) return false;
                tc_fence_after();
                const uint32_t sk = k_at();
                issue_qk(col1, sQ1, sk);
                if (bar1) mma_commit_elect(bar1);
                if (C::BIG) {
                    mma_commit_elect(bar_ke + 8 * (ki % C::KS));
                    ++ki;
                    if (!wait_k()) return false;
                    tc_fence_after();
                    issue_qk(col2, sQ2, k_at());
                } else {
                    issue_qk(col2, sQ2, sk + C::K_TILE);
                }
                mma_commit_elect(bar2);
                mma_commit_elect(bar_ke + 8 * (ki % C::KS));
                ++ki;
                return true;
            };
            // one QK from the next K ring item (d = 128: items hold K1 or K2)
            auto qk_one = [&](uint32_t col, uint32_t sq, uint32_t bar) {
                if (!wait_k()) return false;
                tc_fence_after();
                issue_qk(col, sq, k_at());
                if (bar) mma_commit_elect(bar);
                mma_commit_elect(bar_ke + 8 * (ki % C::KS));
                ++ki;
                return true;
            };
            // O += P V over V item `item` of tile j (keys item*V_ROWS ..); a P half
            // (64 keys) is waited for before its first K step.
            auto pv_item = [&](int j, int item) {
                const int st = vi % C::VS;
                if (!wait_i(bar_vf + 8 * st, static_cast<uint32_t>((vi / C::VS) & 1), p.err)) return false;
                const uint64_t dv = sdesc_sw128(sbase + C::OFF_V + st * C::V_SLOT, C::V_BOX, 1024);
#pragma unroll
                for (int ks = 0; ks < C::V_ROWS / 16; ++ks) {
                    const int g = item * (C::V_ROWS / 16) + ks;   // K step within the tile (16 keys)
                    if ((g & 3) == 0) {
                        if (!wait_i(bar_pb + 8 * (g >> 2), static_cast<uint32_t>(j & 1), p.err)) return false;
                        tc_fence_after();
                    }
                    mma_ts_elect(tmem + C::COL_O, tmem + C::p_col(j, g >> 2) + 8 * (g & 3), dv + ((ks * 2048) >> 4),
                           C::IDESC_PV, (j > 0 || g > 0) ? 1u : 0u);
                }
                mma_commit_elect(bar_ve + 8 * st);
                ++vi;
                return true;
            };
            bool ok = wait_i(bar_q, 0, p.err);
            if constexpr (A2) {
                // S2 only; S2(j+1) as soon as S2(j) has been read, P(j) (over the
                // S1 columns) read by PV(j); "S ready" is committed after PV(j),
                // so that the softmax writes P(j+1) only once P(j) has been read.
                if (ok) ok = qk_one(C::COL_S2, sQ2, 0);
                if (ok) mma_commit_elect(bar_sbf);
                for (int j = 0; ok && j < n; ++j) {
                    if (j + 1 < n)
                        ok = wait_i(bar_sbe, static_cast<uint32_t>(j & 1), p.err) && qk_one(C::COL_S2, sQ2, 0);
                    for (int it = 0; ok && it < C::V_ITEMS; ++it) ok = pv_item(j, it);
                    if (ok && j + 1 < n) mma_commit_elect(bar_sbf);
                }
            }
            // ------------------------------------------------------ pass A
            for (int j = 0; !A2 && ok && j < n; ++j) {
                const int buf = j & 1;
                if (j >= 2) ok = wait_i(bar_sae + 8 * buf, static_cast<uint32_t>(((j >> 1) - 1) & 1), p.err);
                if (ok) ok = qk_pair(256 * buf, 256 * buf + 128, bar_saf + 16 * buf, bar_saf + 16 * buf + 8);
            }
            // pass B overwrites TMEM that pass A used: wait until both tiles' S were read
            for (int j = (n > 2 ? n - 2 : 0); !A2 && ok && j < n; ++j)
                ok = wait_i(bar_sae + 8 * (j & 1), static_cast<uint32_t>((j >> 1) & 1), p.err);
            // ------------------------------------------------------ pass B
            if (!A2 && ok) ok = qk_pair(C::COL_S1, C::COL_S2, 0, bar_sbf);
            for (int j = 0; !A2 && ok && j < n; ++j) {
                if (C::BIG) {
                    // P(j) lies over S1 only: S2 of the next tile goes first, once
                    // this tile's S has been read, then the PV, then S1.
                    if (j + 1 < n)
                        ok = wait_i(bar_sbe, static_cast<uint32_t>(j & 1), p.err) && qk_one(C::COL_S2, sQ2, 0);
                    for (int it = 0; ok && it < C::V_ITEMS; ++it) ok = pv_item(j, it);
                    if (ok && j + 1 < n) ok = qk_one(C::COL_S1, sQ1, bar_sbf);
                } else {
                    if (j + 1 < n) {
                        ok = wait_i(bar_sbe, static_cast<uint32_t>(j & 1), p.err) &&
                             qk_pair(C::COL_S1, C::COL_S2, 0, bar_sbf);
                    }
                    if (ok) ok = pv_item(j, 0);
                    if (ok) mma_commit_elect(bar_pfree + 8 * (j & 1));
                }
            }
            if (ok) mma_commit_elect(bar_o);
            mma_commit_elect(bar_dr);
            warp_wait_drain(bar_dr, 0, p.err);
        }
    } else if (warp == 2) {
        regs_decrease<C::REGS_LOW>();
        // lam_init = 0.8 - 0.6 exp(-0.3 layer); lam = exp(lq1.lk1) - exp(lq2.lk2) + lam_init
        float d1 = 0.f, d2 = 0.f;
        for (int c = lane; c < DQK; c += 32) {
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
    } else if (warp == 3) {
        regs_decrease<C::REGS_LOW>();
    } else {
        // -------------------------------------------------------- softmax
        regs_increase<C::REGS_HIGH>();
        const int br = (warp - 4) >> 2;      // pass A: branch; pass B: key half
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int t = q0 + row;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        uint32_t s[128];

        // pass A: exact online row max / sum of branch br (not in the a2 run)
        float m = -INFINITY, l = 0.f;
        for (int j = 0; !A2 && j < n; ++j) {
            const int buf = j & 1;
            ok = warp_wait_vote(bar_saf + 16 * buf + 8 * br, static_cast<uint32_t>((j >> 1) & 1), p.err, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t ts = tmem + lane_off + 256 * buf + 128 * br;
            tmem_ld32(ts + 0, s);
            tmem_ld32(ts + 32, s + 32);
            tmem_ld32(ts + 64, s + 64);
            tmem_ld32(ts + 96, s + 96);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sae + 8 * buf);
            if (j == qt) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > row) s[c] = 0xff800000u;
            }
            const float m_new = fmaxf(m, row_max128(s) * sl2);
            l = l * ex2(m - m_new) + sum_exp128(s, sl2, m_new);
            m = m_new;
        }
        // both branches' statistics for this row
        xch[br * 256 + row] = m;
        xch[br * 256 + 128 + row] = l;
        named_bar_sync(1, 256);
        const float m1 = xch[row], l1 = xch[128 + row];
        const float m2 = xch[256 + row], l2 = xch[384 + row];
        ok = warp_wait_vote(bar_lam, 0, p.err, ok);
        const float lam = lam_smem[0], lam_init = lam_smem[1];
        constexpr bool a2_run = A2;
        if (TRAIN && !a2_run && t < p.T && DA_CHECK(b < p.B && h < p.H, p.err))   // this branch's log-sum-exp
            p.slse[((static_cast<int64_t>(br) * p.B + b) * p.H + h) * p.T + t] = m + __log2f(l);
        // P = c1 e1 - c2 e2: x = a1 - lam a2
        const float c1 = 1.f / l1, c2 = lam / l2;

        // the a2 run: P = 2^(s2 scale - lse2) from branch 2's saved log-sum-exp
        if constexpr (A2) {
            const float lse2 = (t < p.T && DA_CHECK(b < p.B && h < p.H, p.err))
                                   ? p.slse[((static_cast<int64_t>(p.B) + b) * p.H + h) * p.T + t]
                                   : 0.f;
            for (int j = 0; j < n; ++j) {
                ok = warp_wait_vote(bar_sbf, static_cast<uint32_t>(j & 1), p.err, ok);
                if (!ok) break;
                tc_fence_after();
                tmem_ld32(tmem + lane_off + C::COL_S2 + 64 * br, s);
                tmem_ld32(tmem + lane_off + C::COL_S2 + 64 * br + 32, s + 32);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sbe);   // this tile's S2 has been read
                if (j == qt) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (64 * br + c > row) s[c] = 0xff800000u;
                }
                const float2 sc2 = make_float2(sl2, sl2), nl2 = make_float2(-lse2, -lse2);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                                sc2, nl2);
                    s[c] = pack_bf16(ex2(x.x), ex2(x.y));
                }
                tmem_st32(tmem + lane_off + C::p_col(j, br), s);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pb + 8 * br);
            }
        }

        // pass B: keys 64*br .. 64*br+63 of each tile
        for (int j = 0; !A2 && j < n; ++j) {
            ok = warp_wait_vote(bar_sbf, static_cast<uint32_t>(j & 1), p.err, ok);
            if (!ok) break;
            tc_fence_after();
            tmem_ld32(tmem + lane_off + C::COL_S1 + 64 * br, s);
            tmem_ld32(tmem + lane_off + C::COL_S1 + 64 * br + 32, s + 32);
            tmem_ld32(tmem + lane_off + C::COL_S2 + 64 * br, s + 64);
            tmem_ld32(tmem + lane_off + C::COL_S2 + 64 * br + 32, s + 96);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sbe);   // this tile's S has been read
            if (j == qt) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (64 * br + c > row) {
                        s[c] = 0xff800000u;
                        s[64 + c] = 0xff800000u;
                    }
            }
            // P = 2^(s1 sc - m1) / l1 - lam 2^(s2 sc - m2) / l2, packed bf16 pairs into s[0..31]
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m1, -m2), cc = make_float2(c1, -c2);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float pv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 2 * c + e;
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[k]), __uint_as_float(s[64 + k])), sc2, nm2);
                    const float2 w = __fmul2_rn(make_float2(ex2(x.x), ex2(x.y)), cc);
                    pv[e] = w.x + w.y;
                }
                s[c] = pack_bf16(pv[0], pv[1]);
            }
            if (!C::BIG && j >= 2)
                ok = warp_wait_vote(bar_pfree + 8 * (j & 1), static_cast<uint32_t>(((j >> 1) - 1) & 1), p.err, ok);
            tmem_st32(tmem + lane_off + C::p_col(j, br), s);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pb + 8 * br);
        }

        // -------------------------------------------- epilogue: RMSNorm, scale
        ok = warp_wait_vote(bar_o, 0, p.err, ok);
        tc_fence_after();
        constexpr int HALF = C::DV / 2;
        const int col0 = br * HALF;
        float x[HALF];
        float ss = 0.f;
#pragma unroll
        for (int cc0 = 0; cc0 < HALF; cc0 += 32) {
            uint32_t a[32];
            tmem_ld32(tmem + lane_off + C::COL_O + col0 + cc0, a);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                x[cc0 + k] = __uint_as_float(a[k]);
                ss = fmaf(x[cc0 + k], x[cc0 + k], ss);
            }
        }
        if (TRAIN && ok && t < p.T && DA_CHECK(b < p.B && h < p.H && col0 + HALF <= C::DV, p.err)) {
            // x (run 1) or a2 (run 2), fp32, this warpgroup's half of the channels
            float4 *d4 = reinterpret_cast<float4 *>(static_cast<float *>(a2_run ? p.sa2 : p.sa1) +
                                                    ((static_cast<int64_t>(b) * p.T + t) * p.H + h) * C::DV + col0);
#pragma unroll
            for (int k = 0; k < HALF; k += 4) d4[k / 4] = make_float4(x[k], x[k + 1], x[k + 2], x[k + 3]);
        }
        // the statistics area is free again: both warpgroups read it before pass B
        xch[br * 128 + row] = ss;
        named_bar_sync(1, 256);
        const float ms = (xch[row] + xch[128 + row]) * (1.f / static_cast<float>(C::DV));
        const float r = (1.f - lam_init) * rsqrtf(ms + 1e-5f);
        if (ok && t < p.T && !a2_run && DA_CHECK(b < p.B && h < p.H && col0 + HALF <= C::DV, p.err)) {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + static_cast<int64_t>(b) * p.o_sb +
                                 static_cast<int64_t>(t) * p.o_st + static_cast<int64_t>(h) * p.o_sh + col0;
#pragma unroll
            for (int k = 0; k < HALF; k += 8) {
                uint4 v;
                v.x = pack_bf16(x[k] * r, x[k + 1] * r);
                v.y = pack_bf16(x[k + 2] * r, x[k + 3] * r);
                v.z = pack_bf16(x[k + 4] * r, x[k + 5] * r);
                v.w = pack_bf16(x[k + 6] * r, x[k + 7] * r);
                *reinterpret_cast<uint4 *>(dst + k) = v;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int DQK, bool TRAIN = false, bool A2 = false>
cudaError_t launch_t(const PrefillMaps &m, const PrefillParams &p, cudaStream_t s) {
    using C = V1x2Cfg<DQK>;
    static unsigned long long attr_done = 0;   // one bit per device
    const cudaError_t ea = once_per_device(&attr_done, [] {
        // the in-kernel register split must fit in the launch-time budget
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, prefill_v1_twopass<DQK, TRAIN, A2>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < C::REGS_NEEDED_AT_LAUNCH) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(prefill_v1_twopass<DQK, TRAIN, A2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM);
    });
    if (ea != cudaSuccess) return ea;
    const int n_qt = (p.T + C::BM - 1) / C::BM;
    const long long grid = static_cast<long long>(n_qt) * p.H * p.B;
    if (grid < 1 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    prefill_v1_twopass<DQK, TRAIN, A2><<<static_cast<unsigned>(grid), 384, C::SMEM, s>>>(m.q1, m.q2, m.k1, m.k2, m.v,
                                                                                     p);
    return cudaGetLastError();
}

}  // namespace

int prefill_v1_twopass_v_rows(int dqk) { return dqk == 128 ? V1x2Cfg<128>::V_ROWS : V1x2Cfg<64>::V_ROWS; }

cudaError_t launch_prefill_v1_twopass(const PrefillMaps &m, const PrefillParams &p, int dqk, cudaStream_t s) {
    if (dqk == 128) return launch_t<128>(m, p, s);
    if (dqk == 64) return launch_t<64>(m, p, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_v1_twopass_train(const PrefillMaps &m, const PrefillParams &p, cudaStream_t s) {
    if (!p.sa1 || !p.sa2 || !p.slse) return cudaErrorInvalidValue;
    // run 1: output, x and the log-sum-exp; run 2: a2, from branch 2's log-sum-exp
    cudaError_t e = launch_t<128, true, false>(m, p, s);
    if (e != cudaSuccess) return e;
    return launch_t<128, true, true>(m, p, s);
}

}  // namespace da
