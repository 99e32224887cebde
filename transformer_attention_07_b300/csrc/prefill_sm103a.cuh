// Fused differential-attention prefill for sm_103a.
//
// Computes, per head and per query row i (Differential Transformer pages:
// the DiffAttn formula of the iloveeagents.com Q&A, "Mathematical Formula";
// steps 2-4 of llmbytes.dev "How Differential Attention Cancels Common-Mode
// Noise"):
//     o_i = sum_j (A1_ij - lambda A2_ij) v_j
//     y_i = (1 - lambda_init) * gamma * (o_i - mean(o_i)) / sqrt(var(o_i) + eps)
// without ever forming an N x N map.  Because the product with V is linear,
// (A1 - lambda A2) V = A1 V - lambda A2 V, so each map keeps its own online
// softmax state (running max m_r, normaliser l_r) and its own unnormalised
// accumulator O_r, and the two are combined once per row at the end:
//     o = O1 / l1 - lambda * O2 / l2.
//
// One CTA owns a tile of 128 query rows of one (b, h) and walks the key tiles
// (128 keys each; under causal masking only the tiles at or left of the
// diagonal).  In the persistent form (PERSIST) a grid of one CTA per SM walks
// the query tiles in heaviest-first order, each CTA taking every G-th tile in
// alternating direction (G = grid size); the key/value rings and barrier
// phases run on across tiles, so the next tile's Q load and first scores
// overlap the current tile's epilogue.  Warp roles:
//   warp 0       TMA producer: Q1/Q2 once, then K1/K2 and V tiles into
//                shared-memory rings (128-byte swizzle).
//   warp 1       tensor-core issuer (one thread) and TMEM owner:
//                  S_r = Q_r K_r^T           (tcgen05.mma, A and B in smem)
//                  O_r += P_r V              (tcgen05.mma, A = P in TMEM)
//   warps 4-7    softmax of map 1; warps 8-11 softmax of map 2.  Thread t of
//                the group owns query row t: it reads its row of S_r from
//                TMEM, updates (m_r, l_r), writes P_r (bf16) back over S_r,
//                and rescales O_r in TMEM when its max has grown by more than
//                2^8 (values stay bounded by 2^8 in between).
//   epilogue     both softmax groups: o = O1/l1 - lambda O2/l2 per row, the
//                GroupNorm statistics over dv, gain, (1 - lambda_init), bf16
//                store (and the optional fp32 pre-norm copy; for training,
//                also each map's log-sum-exp and A2 V, which the backward
//                pass reads).  The persistent form at dv = 128 stages each
//                warp's 32-row x 64-column share of the bf16 output in
//                shared memory and writes it with one TMA store, so the
//                next tile's softmax does not queue behind per-row stores.
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   [0,128) S1 (P1 aliases its first 64 columns)   [128,256) S2 / P2
//   [256,256+dv) O1                                [256+dv,256+2dv) O2
#pragma once

#include "sm103_ptx.cuh"

namespace diffattn {

struct PrefillParams {
    int B, H, Nq, Nk;
    float lambda, lambda_init, eps;
    float scale_log2;       // log2(e) / sqrt(d)
    const float* gamma;     // [H*dv] or null
    uint16_t* out;          // bf16 [B,H,Nq,dv]
    float* o_prenorm;       // fp32 [B,H,Nq,dv] or null
    float* o2;              // fp32 [B,H,Nq,dv] or null: A2 V (the second map's normalised output)
    float* lse;             // fp32 [2,B,H,Nq] or null: log sum_j exp(s_r,ij), natural log, per map
    const float* qk_scale;  // [4,H] dequantisation scales of q1, k1, q2, k2 per head (fp8 inputs), or null
    int weight_major;       // persistent form: order the tiles by weight across all heads (see prefill_kernel)
    int head_group;         // one-tile form, > 0: a 1-D grid in weight order within groups of this many heads
    // Persistent form: tile numbers are divided by the major extent (heads
    // B H in weight-major order, else the query tiles of a head) and head
    // numbers by H through div_inv with these multipliers and shifts.
    unsigned div_major_m, div_h_m;
    int div_major_s, div_h_s;
};

// QK8: Q1, Q2, K1, K2 are fp8 (e4m3) with per-head scales, and Q K^T runs
// as an 8-bit tensor-core product (kind::f8f6f4, K = 32 per instruction);
// P V stays bf16.
// PERSIST: the layout of the persistent form (see prefill_kernel).
template <int D, int DV, bool QK8 = false, bool PERSIST = false>
struct PrefillLayout {
    static constexpr int BM = 128;   // query rows per tile (MMA M)
    static constexpr int BN = 128;   // keys per tile (MMA N of QK^T, K of PV)
    // Persistent form at dv = 128: the bf16 output leaves through shared
    // memory by TMA stores (one 32-row x 64-column box per softmax warp,
    // 128-byte swizzle), so the epilogue's stores do not occupy the
    // load/store unit.  Its 32 KB of staging take one K stage.
    static constexpr bool OST = PERSIST && DV == 128;
    static constexpr int KST = OST ? 2 : 3;    // K1/K2 ring depth
    // V ring depth.  A V tile can be loaded only once the P V product two
    // (three) tiles back has completed, and from L2 under full load it takes
    // about as long as one key tile's work to arrive, so a third stage keeps
    // the tensor core from waiting on it.  The persistent form needs its own
    // epilogue slots (the next tile's loads run during the epilogue) and has
    // no room for it.
    static constexpr int VST = PERSIST ? 2 : 3;
    static constexpr uint32_t QK_ELEM = QK8 ? 1 : 2;   // bytes per Q/K element
    static constexpr uint32_t QK_ROW = D * QK_ELEM;    // bytes per Q/K row: 128, 64 or 32
    static constexpr uint32_t Q_BYTES = BM * QK_ROW;
    static constexpr uint32_t K_BYTES = BN * QK_ROW;
    static constexpr uint32_t V_BOX = BN * 128;   // one 64-column V box: BN rows x 128 bytes
    static constexpr uint32_t V_BYTES = BN * DV * 2;
    static constexpr uint32_t OFF_Q1 = 0;
    static constexpr uint32_t OFF_Q2 = Q_BYTES;
    static constexpr uint32_t OFF_K = 2 * Q_BYTES;              // stage s: K1 then K2
    static constexpr uint32_t OFF_V = OFF_K + KST * 2 * K_BYTES;
    // 6 x 128 fp32 exchange slots of the epilogue.  With one query tile per
    // CTA they lie over Q1, which nothing reads once the epilogue may start.
    static constexpr uint32_t EPI_BYTES = 6 * BM * 4;
    static_assert(EPI_BYTES <= Q_BYTES, "epilogue slots");
    static constexpr uint32_t OST_WARP = 32 * 128;   // one warp's staging: 32 rows x 128 bytes
    static constexpr uint32_t OFF_OST = OFF_V + VST * V_BYTES;   // 1024-byte aligned (swizzle atoms)
    static constexpr uint32_t OST_BYTES = OST ? 8 * OST_WARP : 0;
    static_assert(OFF_OST % 1024 == 0, "staging alignment");
    static constexpr uint32_t OFF_EPI = PERSIST ? OFF_OST + OST_BYTES : OFF_Q1;
    static constexpr uint32_t OFF_BAR = PERSIST ? OFF_EPI + EPI_BYTES : OFF_V + VST * V_BYTES;
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + KST;
    static constexpr int B_VFULL = B_KEMPTY + KST;
    static constexpr int B_VEMPTY = B_VFULL + VST;
    static constexpr int B_SFULL = B_VEMPTY + VST;   // 2 (one per map)
    // P is handed to the issuer in PSPLIT parts of BN / PSPLIT keys each.
    static constexpr int PSPLIT = 2;
    static constexpr int PKEYS = BN / PSPLIT;
    static constexpr int B_PFULL = B_SFULL + 2;      // 2 PSPLIT: map r, part hh at PSPLIT r + hh
    static constexpr int B_OFULL = B_PFULL + 2 * PSPLIT;
    static constexpr int B_OFREE = B_OFULL + 1;      // persistent: O read by the epilogue (count 256)
    static constexpr int B_QEMPTY = B_OFREE + 1;     // persistent: Q tiles no longer read
    static constexpr int B_DRAIN = B_QEMPTY + 1;     // issuer: every issued MMA complete (error path)
    static constexpr int NBAR = B_DRAIN + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
    static constexpr uint32_t USED = OFF_TMEM_SLOT + 16;
    // +1024 for aligning the dynamic base; at least 120 KB so that a single
    // CTA (which takes all 512 TMEM columns) is resident per SM.
    static constexpr uint32_t SMEM_BYTES = (USED + 1024 > 120u * 1024u) ? USED + 1024 : 120u * 1024u;
    // The swizzle span equals the row width, so each row is one span.
    static constexpr uint32_t QK_SWZ = QK_ROW == 128 ? SWZ_128B : QK_ROW == 64 ? SWZ_64B : SWZ_32B;
    static constexpr uint32_t QK_SBO = 8 * QK_ROW;   // bytes between 8-row groups
    static constexpr int QK_KSTEPS = QK_ROW / 32;    // 32 bytes of the row per MMA (16 bf16 or 32 fp8)
    static constexpr uint32_t TM_S1 = 0, TM_S2 = 128, TM_O1 = 256, TM_O2 = 256 + DV;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 384;
    static_assert(D == 64 || D == 32, "d");
    static_assert(DV == 128 || DV == 64, "dv");
    static_assert(USED + 1024 <= 227u * 1024u, "shared memory");
};

template <int D, int DV, bool CAUSAL, bool QK8 = false, bool PERSIST = false>
__global__ void __launch_bounds__(384, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_q2,
               const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
               const PrefillParams p) {
    using L = PrefillLayout<D, DV, QK8, PERSIST>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Tiles: heaviest (right-most under causal masking) query tiles first.
    // Without PERSIST the CTA owns tile (blockIdx.x, y, z); with it, tile
    // number t = k G + (k even ? c : G - 1 - c) for k = 0, 1, ... (c =
    // blockIdx.x, G = gridDim.x) of one of two orders:
    //   * (b, h)-major, heaviest first within each (b, h): the CTAs at work at
    //     any time share a few heads' K and V, which stay in L2;
    //   * weight-major (p.weight_major), heaviest first across all heads: the
    //     alternating walk then hands every CTA nearly the same number of key
    //     tiles (at causal 2K, B4 H8: the busiest CTA 4% above the mean
    //     instead of 16%), but the CTAs at work span all heads, so the launcher
    //     takes it only when every head's K and V fit in L2 together.
    // The one-tile form under causal masking runs a 1-D grid (p.head_group >
    // 0): the hardware starts the CTAs in index order, and the index walks
    // groups of p.head_group heads (as many as fit 16 MB of K and V, when that
    // is at least four; otherwise the (b, h)-major 3-D grid), heaviest tiles
    // of the whole group first.  The last CTAs to start are then the
    // lightest tiles of the last group, not the lightest tiles of each head
    // behind the heaviest of the next (at causal 8K, B2 H16, the modelled
    // finish moves from 6.6% above a perfect split to 0.3%).
    const int num_qt = (p.Nq + L::BM - 1) / L::BM;
    const int diag = p.Nk - p.Nq;   // key j visible to query i iff j <= i + diag (causal)
    auto tile = [&](int k, int& qt, int& h, int& b) -> bool {
        if constexpr (!PERSIST) {
            if (p.head_group > 0) {
                const unsigned BH = (unsigned)p.H * (unsigned)p.B, HG = p.head_group, t = blockIdx.x;
                const unsigned NT = (unsigned)num_qt;
                const unsigned g = t / (HG * NT), r = t - g * HG * NT;
                const unsigned ng = BH - g * HG < HG ? BH - g * HG : HG;   // heads in this group
                const unsigned w = r / ng, bh = g * HG + (r - w * ng);
                qt = num_qt - 1 - (int)w;
                const unsigned bb = bh / (unsigned)p.H;
                h = (int)(bh - bb * (unsigned)p.H);
                b = (int)bb;
            } else {
                qt = num_qt - 1 - (int)blockIdx.x;
                h = blockIdx.y;
                b = blockIdx.z;
            }
            return k == 0;
        } else {
            // 32-bit index arithmetic (the launcher keeps the tile count
            // below 2^30) with divisions by invariant multipliers: the
            // softmax warps compute the next tile's indices between two
            // tiles, where a division's latency delays the next scores.
            const unsigned G = gridDim.x, c = blockIdx.x;
            const unsigned t = (unsigned)k * G + ((k & 1) ? G - 1 - c : c);
            const unsigned BH = (unsigned)p.H * (unsigned)p.B, NT = (unsigned)num_qt;
            if (t >= NT * BH) return false;
            unsigned bh, w;
            if (p.weight_major) {
                w = div_inv(t, p.div_major_m, p.div_major_s);
                bh = t - w * BH;
            } else {
                bh = div_inv(t, p.div_major_m, p.div_major_s);
                w = t - bh * NT;
            }
            qt = num_qt - 1 - (int)w;
            const unsigned bb = div_inv(bh, p.div_h_m, p.div_h_s);
            h = (int)(bh - bb * (unsigned)p.H);
            b = (int)bb;
            return true;
        }
    };
    auto kv_tiles = [&](int qt) -> int {
        int kv_end = p.Nk;
        if (CAUSAL) kv_end = min(p.Nk, qt * L::BM + L::BM + diag);
        return (kv_end + L::BN - 1) / L::BN;
    };

    auto bar = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_Q), 1);
        for (int s = 0; s < L::KST; ++s) {
            mbar_init(bar(L::B_KFULL + s), 1);
            mbar_init(bar(L::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < L::VST; ++s) {
            mbar_init(bar(L::B_VFULL + s), 1);
            mbar_init(bar(L::B_VEMPTY + s), 1);
        }
        for (int r = 0; r < 2; ++r) {
            mbar_init(bar(L::B_SFULL + r), 1);
            for (int hh = 0; hh < L::PSPLIT; ++hh) mbar_init(bar(L::B_PFULL + L::PSPLIT * r + hh), 128);
        }
        mbar_init(bar(L::B_OFULL), 1);
        mbar_init(bar(L::B_OFREE), 256);
        mbar_init(bar(L::B_QEMPTY), 1);
        mbar_init(bar(L::B_DRAIN), 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q1);
        prefetch_tensormap(&tm_q2);
        prefetch_tensormap(&tm_k1);
        prefetch_tensormap(&tm_k2);
        prefetch_tensormap(&tm_v);
        if constexpr (L::OST) prefetch_tensormap(&tm_out);
    }
    if (warp == 1) {
        tmem_alloc(sb + L::OFF_TMEM_SLOT, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM_SLOT);
    // Launched as a dependent grid (programmatic stream serialisation): no
    // global memory is read or written before the previous grid on the stream
    // has completed, since its output may be this call's input.  The next
    // grid may be scheduled from here on: its CTAs take SMs as this grid's
    // CTAs leave and set up while the last of them finish.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            // Stage counters run on across query tiles: the g-th key tile of
            // the CTA uses ring stage g % depth in phase (g / depth) & 1.
            int k_issued = 0, v_issued = 0, q_issued = 0;
            int qt, h, b;
            for (int k = 0; ok && tile(k, qt, h, b); ++k) {
                if (k > 0) {
                    ok = mbar_wait(bar(L::B_QEMPTY), (k - 1) & 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(bar(L::B_Q), 2 * L::Q_BYTES);
                tma_load_4d(sb + L::OFF_Q1, &tm_q1, bar(L::B_Q), 0, qt * L::BM, h, b);
                tma_load_4d(sb + L::OFF_Q2, &tm_q2, bar(L::B_Q), 0, qt * L::BM, h, b);
                ++q_issued;
                const int n_kv = kv_tiles(qt);
                for (int j = 0; j < n_kv; ++j) {
                    const int ks = k_issued % L::KST;
                    ok = mbar_wait(bar(L::B_KEMPTY + ks), ((k_issued / L::KST) & 1) ^ 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                    const uint32_t k1s = sb + L::OFF_K + (uint32_t)ks * 2 * L::K_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_KFULL + ks), 2 * L::K_BYTES);
                    tma_load_4d(k1s, &tm_k1, bar(L::B_KFULL + ks), 0, j * L::BN, h, b);
                    tma_load_4d(k1s + L::K_BYTES, &tm_k2, bar(L::B_KFULL + ks), 0, j * L::BN, h, b);
                    ++k_issued;
                    const int vs = v_issued % L::VST;
                    ok = mbar_wait(bar(L::B_VEMPTY + vs), ((v_issued / L::VST) & 1) ^ 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                    const uint32_t vsm = sb + L::OFF_V + (uint32_t)vs * L::V_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_VFULL + vs), L::V_BYTES);
#pragma unroll
                    for (int c = 0; c < DV / 64; ++c)
                        tma_load_4d(vsm + (uint32_t)c * L::V_BOX, &tm_v, bar(L::B_VFULL + vs), c * 64, j * L::BN, h,
                                    b);
                    ++v_issued;
                }
                if constexpr (!PERSIST) break;
            }
            // Never leave with copies in flight: wait (bounded) for the last
            // phase armed on every stage.
            if (q_issued > 0) mbar_wait(bar(L::B_Q), (q_issued - 1) & 1, ERR_SITE_PREFILL_DRAIN);
            for (int s = 0; s < L::KST && s < k_issued; ++s) {
                const int last = s + ((k_issued - 1 - s) / L::KST) * L::KST;
                mbar_wait(bar(L::B_KFULL + s), (last / L::KST) & 1, ERR_SITE_PREFILL_DRAIN);
            }
            for (int s = 0; s < L::VST && s < v_issued; ++s) {
                const int last = s + ((v_issued - 1 - s) / L::VST) * L::VST;
                mbar_wait(bar(L::B_VFULL + s), (last / L::VST) & 1, ERR_SITE_PREFILL_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop with warp-uniform values; each MMA and
        // commit is issued by one elected lane (the *_warp wrappers).
        {
            constexpr uint32_t idesc_qk = QK8 ? idesc_e4m3_f32(L::BM, L::BN) : idesc_bf16_f32(L::BM, L::BN, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(L::BM, DV, true);
            // Every lane waits; a wait that ran out on any lane ends the loop on all.
            auto wait = [&](int i, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ERR_SITE_PREFILL_MMA));
            };
            bool ok = wait(L::B_Q, 0);
            tc_fence_after();
            // Operand descriptors are built once; stages and k-steps are
            // compile-time offsets in the descriptor's address field (units of
            // 16 bytes), so each MMA costs one add: the issuing warp's own
            // instruction latency otherwise bounds the tensor pipe.
            const uint64_t dq1 = smem_desc(sb + L::OFF_Q1, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t dq2 = smem_desc(sb + L::OFF_Q2, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t dk0 = smem_desc(sb + L::OFF_K, 16, L::QK_SBO, L::QK_SWZ);   // K1 of stage 0
            const uint64_t dv0 = smem_desc(sb + L::OFF_V, L::V_BOX, 1024, SWZ_128B);   // V of stage 0
            constexpr uint64_t K2_OFF = L::K_BYTES >> 4, KSTAGE = (2 * L::K_BYTES) >> 4, VSTAGE = L::V_BYTES >> 4;
            const uint32_t t_s1 = tmem + L::TM_S1, t_s2 = tmem + L::TM_S2;
            const uint32_t t_o1 = tmem + L::TM_O1, t_o2 = tmem + L::TM_O2;
            // O += P V over part hh of one key tile (keys PKEYS hh .. PKEYS
            // (hh + 1) - 1): 16-key steps, P from TMEM columns 8k.
            auto pv = [&](uint32_t t_o, uint32_t t_p, uint64_t dvs, uint32_t acc0, int hh) {
#pragma unroll
                for (int kk = 0; kk < L::PKEYS / 16; ++kk) {
                    const int k = hh * (L::PKEYS / 16) + kk;
                    mma_ts_warp(t_o, t_p + 8u * k, dvs + (uint64_t)(k * (16 * 128 >> 4)), idesc_pv,
                                k == 0 ? acc0 : 1u);
                }
            };
            // S = Q K^T over one key tile: 16-column steps of d (32 bytes).
            auto qk = [&](uint32_t t_s, uint64_t dq, uint64_t dks) {
#pragma unroll
                for (int k = 0; k < L::QK_KSTEPS; ++k) {
                    if constexpr (QK8)
                        mma_ss_f8_warp(t_s, dq + (uint64_t)(2 * k), dks + (uint64_t)(2 * k), idesc_qk,
                                       k > 0 ? 1u : 0u);
                    else
                        mma_ss_warp(t_s, dq + (uint64_t)(2 * k), dks + (uint64_t)(2 * k), idesc_qk, k > 0 ? 1u : 0u);
                }
            };
            int g = 0;   // key tiles of earlier query tiles (ring stage and phase counter)
            int qt, h, b;
            for (int k = 0; ok && tile(k, qt, h, b); ++k) {
                const int n_kv = kv_tiles(qt);
                if (k > 0) {
                    ok = wait(L::B_Q, k & 1);
                    if (!ok) break;
                    tc_fence_after();
                }
                // Step j: P V of key tile j - 1, then the scores of tile j, per
                // map.  P_r V waits only for V and P_r, the scores only for K,
                // so a late K tile does not hold up the P V products.
                for (int j = 0; j <= n_kv; ++j) {
                    const int gj = g + j;
                    const int ks = gj % L::KST;
                    const int jv = j - 1, gv = gj - 1;
                    const int vs = (gv + L::VST) % L::VST;
                    const uint64_t dvs = dv0 + (uint64_t)vs * VSTAGE;
                    const uint64_t dks = dk0 + (uint64_t)ks * KSTAGE;
                    const uint32_t acc0 = jv > 0 ? 1u : 0u;
                    // map 1: O1 += P1 V (previous tile), then S1 = Q1 K1^T (this tile)
                    if (jv >= 0) {
                        ok = wait(L::B_VFULL + vs, (gv / L::VST) & 1) && wait(L::B_PFULL + 0, gv & 1);
                        if (!ok) break;
                        if (PERSIST && jv == 0 && k > 0) {
                            // The first product of a query tile overwrites O:
                            // the previous tile's epilogue must have read it.
                            ok = wait(L::B_OFREE, (k - 1) & 1);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        pv(t_o1, t_s1, dvs, acc0, 0);
#pragma unroll
                        for (int hh = 1; hh < L::PSPLIT && ok; ++hh) {
                            ok = wait(L::B_PFULL + hh, gv & 1);
                            tc_fence_after();
                            if (ok) pv(t_o1, t_s1, dvs, acc0, hh);
                        }
                        if (!ok) break;
                    }
                    if (j < n_kv) {
                        ok = wait(L::B_KFULL + ks, (gj / L::KST) & 1);
                        if (!ok) break;
                        tc_fence_after();
                        qk(t_s1, dq1, dks);
                        mma_commit_warp(bar(L::B_SFULL + 0));
                    }
                    // map 2
                    if (jv >= 0) {
#pragma unroll
                        for (int hh = 0; hh < L::PSPLIT && ok; ++hh) {
                            ok = wait(L::B_PFULL + L::PSPLIT + hh, gv & 1);
                            tc_fence_after();
                            if (ok) pv(t_o2, t_s2, dvs, acc0, hh);
                        }
                        if (!ok) break;
                        mma_commit_warp(bar(L::B_VEMPTY + vs));
                    }
                    if (j < n_kv) {
                        qk(t_s2, dq2, dks + K2_OFF);
                        mma_commit_warp(bar(L::B_SFULL + 1));
                        mma_commit_warp(bar(L::B_KEMPTY + ks));
                        if (PERSIST && j == n_kv - 1) mma_commit_warp(bar(L::B_QEMPTY));
                    }
                }
                g += n_kv;
                // The epilogue of this query tile may start once every MMA
                // issued so far has completed.
                if (ok) mma_commit_warp(bar(L::B_OFULL));
                if constexpr (!PERSIST) break;
            }
            if (!ok) {
                // Error: signal the epilogue anyway, and let no MMA outlive
                // the kernel's tensor memory.
                mma_commit_warp(bar(L::B_OFULL));
                mma_commit_warp(bar(L::B_DRAIN));
                mbar_wait(bar(L::B_DRAIN), 0, ERR_SITE_PREFILL_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        const int r = (warp - 4) >> 2;           // map
        const int wq = warp & 3;                 // TMEM lane quarter of this warp
        const int row = wq * 32 + lane;          // row within the tile
        const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
        const uint32_t s_col = r ? L::TM_S2 : L::TM_S1;
        const uint32_t o_col = r ? L::TM_O2 : L::TM_O1;
        bool ok = true;
        int g = 0;   // key tiles of earlier query tiles (barrier phase counter)
        int qt, h, b;
        bool more = tile(0, qt, h, b);
        for (int k = 0; ok && more; ++k) {
        const int n_kv = kv_tiles(qt);
        const int qi = qt * L::BM + row;
        const int kmax = CAUSAL ? min(qi + diag, p.Nk - 1) : p.Nk - 1;   // last visible key
        // log2(e)/sqrt(d), times the map's q and k dequantisation scales.
        float sl2 = p.scale_log2;
        if constexpr (QK8) sl2 *= p.qk_scale[(2 * r) * p.H + h] * p.qk_scale[(2 * r + 1) * p.H + h];
        float m = -INFINITY;   // running max of scaled logits (log2 domain)
        float l = 0.f;         // running sum of the bf16-rounded probabilities
        for (int j = 0; j < n_kv; ++j) {
            ok = mbar_wait(bar(L::B_SFULL + r), (g + j) & 1, ERR_SITE_PREFILL_SOFTMAX);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // S_r row: 128 columns in one TMEM load.
            uint32_t sv[128];
            tmem_ld128(tmem + t_lane + s_col, sv);
            const int kb = j * L::BN;
            if (kb + L::BN - 1 > kmax) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (kb + i > kmax) sv[i] = __float_as_uint(-INFINITY);
            }
            // Row max: four independent chains of three-input maxima.
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 128; i += 8) {
                mx0 = fmax3(mx0, __uint_as_float(sv[i + 0]), __uint_as_float(sv[i + 1]));
                mx1 = fmax3(mx1, __uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3]));
                mx2 = fmax3(mx2, __uint_as_float(sv[i + 4]), __uint_as_float(sv[i + 5]));
                mx3 = fmax3(mx3, __uint_as_float(sv[i + 6]), __uint_as_float(sv[i + 7]));
            }
            const float m_new = fmaxf(m, fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2);
            const bool grow = m_new > m + 8.0f;
            const bool rescale = __any_sync(0xffffffffu, grow) && j > 0;   // warp-uniform
            float alpha = 1.0f;
            if (grow) {
                alpha = fast_exp2(m - m_new);
                l *= alpha;
                m = m_new;
            }
            // p = 2^(s * log2(e)/sqrt(d) - m): scale and shift two columns per
            // packed FMA, exponential on the SFU, round to bf16 in pairs.  The
            // row sum accumulates the rounded values (the P the MMA multiplies),
            // so a row dominated by one key keeps that key's rounding out of
            // O/l; four packed chains.
            const float nm = (m == -INFINITY) ? 0.f : -m;
            // P goes to the issuer in PSPLIT parts: the P V of a part runs
            // while the next part's exponentials are computed.  The rare O
            // rescale happens before the first part is handed over (that
            // part's P V accumulates into O); the previous P_r V has
            // completed (it was issued before this tile's S_r, whose commit
            // we waited on).
            constexpr int PK = L::PKEYS;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, a4 = 0.f, a5 = 0.f, a6 = 0.f, a7 = 0.f;
#pragma unroll
            for (int hh = 0; hh < L::PSPLIT; ++hh) {
                uint32_t pk[PK / 2];
#pragma unroll
                for (int i = PK * hh; i < PK * hh + PK; i += 8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        fma2_bcast(x[e], x[e + 1], __uint_as_float(sv[i + e]), __uint_as_float(sv[i + e + 1]), sl2,
                                   nm);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = fast_exp2(x[e]);
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) pk[((i - PK * hh) >> 1) + e] = w[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                    acc_bf16x2(a0, a1, w[0]);
                    acc_bf16x2(a2, a3, w[1]);
                    acc_bf16x2(a4, a5, w[2]);
                    acc_bf16x2(a6, a7, w[3]);
                }
                if constexpr (PK == 64)
                    tmem_st32(tmem + t_lane + s_col + 32u * hh, pk);
                else
                    tmem_st16(tmem + t_lane + s_col + 16u * hh, pk);
                if (hh == 0 && rescale) {
#pragma unroll
                    for (int c = 0; c < DV / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tmem + t_lane + o_col + 32u * c, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(tmem + t_lane + o_col + 32u * c, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(L::B_PFULL + L::PSPLIT * r + hh));
            }
            l += ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
        }

        // ------------------------------------------------------------ epilogue
        g += n_kv;
        constexpr int HALF = DV / 2;
        const int c0 = r * HALF;
        // Bring this thread's GroupNorm gains into L1 while the last products
        // complete: read from L2 inside the store loop, their latency was paid
        // once per group of columns.
        if (p.gamma != nullptr && lane < HALF * 4 / 128)
            prefetch_l1(p.gamma + (size_t)h * DV + c0 + lane * 32);
        if (!mbar_wait(bar(L::B_OFULL), k & 1, ERR_SITE_PREFILL_EPILOGUE)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        __syncwarp();
        tc_fence_after();
        float* epi = reinterpret_cast<float*>(smem + L::OFF_EPI);
        epi[r * L::BM + row] = l;
        named_barrier_sync(1, 256);
        const float inv1 = 1.0f / epi[row];
        const float inv2 = p.lambda / epi[L::BM + row];
        const size_t rowoff = (((size_t)b * p.H + h) * p.Nq + qi) * DV + c0;
        // Training outputs for the backward pass: each map's log-sum-exp of
        // the scaled logits (natural log; m is in log2 units) and A2 V.
        if (p.lse != nullptr && qi < p.Nq)
            p.lse[((size_t)r * p.B * p.H + (size_t)b * p.H + h) * p.Nq + qi] = (m + log2f(l)) * 0.6931471805599453f;
        if (p.o2 != nullptr) {   // uniform: every lane takes part in the warp-wide TMEM loads
            const float inv2n = 1.0f / epi[L::BM + row];
#pragma unroll
            for (int c = 0; c < HALF / 32; ++c) {
                uint32_t bb[32];
                tmem_ld32(tmem + t_lane + L::TM_O2 + c0 + 32u * c, bb);
                if (qi < p.Nq) {
                    float4* dst = reinterpret_cast<float4*>(p.o2 + rowoff + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(bb[4 * i]) * inv2n, __uint_as_float(bb[4 * i + 1]) * inv2n,
                                             __uint_as_float(bb[4 * i + 2]) * inv2n,
                                             __uint_as_float(bb[4 * i + 3]) * inv2n);
                }
            }
        }
        float o[HALF];
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) {
            uint32_t a[32], bb[32];
            tmem_ld32(tmem + t_lane + L::TM_O1 + c0 + 32u * c, a);
            tmem_ld32(tmem + t_lane + L::TM_O2 + c0 + 32u * c, bb);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                // Both products rounded before the subtraction (no FMA
                // contraction), so identical maps with lambda = 1 cancel to 0.
                o[32 * c + i] = __fmul_rn(__uint_as_float(a[i]), inv1) - __fmul_rn(__uint_as_float(bb[i]), inv2);
        }
        if constexpr (PERSIST) {
            // O1, O2 are in registers: the next tile's products may overwrite them.
            tc_fence_before();
            mbar_arrive(bar(L::B_OFREE));
        }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < HALF; ++i) s4[i & 3] += o[i];
        const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        epi[(2 + r) * L::BM + row] = sum;
        named_barrier_sync(1, 256);
        const float mu = (epi[2 * L::BM + row] + epi[3 * L::BM + row]) * (1.0f / DV);
        float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < HALF; ++i) q4[i & 3] += (o[i] - mu) * (o[i] - mu);
        const float sq = (q4[0] + q4[1]) + (q4[2] + q4[3]);
        epi[(4 + r) * L::BM + row] = sq;
        named_barrier_sync(1, 256);
        const float var = (epi[4 * L::BM + row] + epi[5 * L::BM + row]) * (1.0f / DV);
        const float sc = (1.0f - p.lambda_init) * rsqrtf(var + p.eps);
        if constexpr (L::OST) {
            // Row `row` of this warp's 32 x 64 box: 16-byte chunk i at chunk
            // position i ^ (row & 7) (the 128-byte swizzle).  Rows at or past
            // Nq are staged too; the TMA store does not write them.
            if (p.o_prenorm && qi < p.Nq) {
                float4* dst = reinterpret_cast<float4*>(p.o_prenorm + rowoff);
#pragma unroll
                for (int i = 0; i < HALF / 4; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
            const float* __restrict__ g = p.gamma ? p.gamma + (size_t)h * DV + c0 : nullptr;
            const uint32_t box = L::OFF_OST + (uint32_t)(r * 4 + wq) * L::OST_WARP;
            // The previous tile's store from this buffer must have read it.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            uint8_t* srow = smem + box + (uint32_t)lane * 128u;
#pragma unroll
            for (int i = 0; i < HALF / 8; ++i) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = (o[8 * i + e] - mu) * sc * (g ? __ldg(g + 8 * i + e) : 1.0f);
                *reinterpret_cast<uint4*>(srow + (((uint32_t)i ^ (uint32_t)(lane & 7)) << 4)) =
                    make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                               pack_bf16x2(y[6], y[7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_4d(&tm_out, sb + box, c0, qt * L::BM + wq * 32, h, b);
                bulk_commit_group();
            }
        } else if (qi < p.Nq) {
            if (p.o_prenorm) {
                float4* dst = reinterpret_cast<float4*>(p.o_prenorm + rowoff);
#pragma unroll
                for (int i = 0; i < HALF / 4; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
            const float* __restrict__ g = p.gamma ? p.gamma + (size_t)h * DV + c0 : nullptr;
            uint4* dst = reinterpret_cast<uint4*>(p.out + rowoff);
#pragma unroll
            for (int i = 0; i < HALF / 8; ++i) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = (o[8 * i + e] - mu) * sc * (g ? __ldg(g + 8 * i + e) : 1.0f);
                dst[i] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                    pack_bf16x2(y[6], y[7]));
            }
        }
        if constexpr (!PERSIST) break;
        more = tile(k + 1, qt, h, b);
        }   // query tiles
        // Leave with no TMA store reading shared memory or still writing.
        if constexpr (L::OST)
            if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

}  // namespace diffattn
