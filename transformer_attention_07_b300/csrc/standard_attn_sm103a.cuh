// Standard softmax attention for sm_103a: the single-map baseline that the
// Differential Transformer pages measure differential attention against
// (llmbytes.dev "Throughput and Hardware Realities": DiffAttn compared with
// FlashAttention; the operator itself is softmax(Q K^T / sqrt d) V, the
// standard attention of the iloveeagents.com Q&A "Detail" section).
//
//     out_i = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j
//
// It is built from the same parts as the differential kernel so that the
// two can be compared on the same hardware path: at equal parameters a
// differential head (q = [q1; q2], k = [k1; k2] of width 2 x 64, v of width
// 128) is compared with a standard head of width d = dv = 128.
//
// One CTA owns two 128-row query tiles of one (b, h) (rows q0 .. q0+255),
// which share every K and V tile; they take the places of the two maps of
// the differential kernel.  As in the differential kernel, a persistent form
// (PERSIST) walks such tile pairs with one CTA per SM for short sequences.
// Warp roles:
//   warp 0       TMA producer: both Q tiles once, then K and V tiles.
//   warp 1       tensor-core issuer (the whole warp; one elected lane
//                issues): per key tile and query tile r,
//                O_r += P_r V (previous key tile, A = P in TMEM) then
//                S_r = Q_r K^T (A and B in smem, K-dim 128 = two 64-column
//                swizzle atoms).
//   warps 4-7    softmax of query tile 0; warps 8-11 of query tile 1; one
//                thread per row; the same online softmax as the
//                differential kernel; epilogue out = O_r / l_r, bf16
//                (in the persistent form through shared memory and TMA
//                stores, as in the differential kernel).
// Tensor memory: [0,128) S0 / P0, [128,256) S1 / P1, [256,384) O0, [384,512) O1.
#pragma once

#include "sm103_ptx.cuh"

namespace diffattn {

struct StandardParams {
    int B, H, Nq, Nk;
    float scale_log2;       // log2(e) / sqrt(d)
    uint16_t* out;          // bf16 [B,H,Nq,dv]
    float* out_f32;         // fp32 [B,H,Nq,dv] or null
    int weight_major;       // persistent form: order the tile pairs by weight across all heads
    int head_group;         // one-pair form, > 0: a 1-D grid in weight order within groups of this many heads
    // Persistent form: tile numbers are divided by the major extent (heads
    // B H in weight-major order, else the query tiles of a head) and head
    // numbers by H through div_inv with these multipliers and shifts.
    unsigned div_major_m, div_h_m;
    int div_major_s, div_h_s;
};

struct StandardLayout {
    static constexpr int D = 128, DV = 128;
    static constexpr int BM = 128;   // rows per query tile; two tiles per CTA
    static constexpr int BN = 128;   // keys per tile
    static constexpr int KST = 2;
    static constexpr int VST = 2;
    static constexpr uint32_t ATOM = 128 * 128;       // 128 rows x 128 bytes (64 bf16 columns)
    static constexpr uint32_t Q_BYTES = BM * D * 2;   // one query tile: two atoms
    static constexpr uint32_t K_BYTES = BN * D * 2;
    static constexpr uint32_t V_BYTES = BN * DV * 2;
    static constexpr uint32_t OFF_Q = 0;              // tile r at r * Q_BYTES
    static constexpr uint32_t OFF_K = 2 * Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KST * K_BYTES;
    // Persistent form: the bf16 output leaves through shared memory by TMA
    // stores, one 32-row x 64-column box (128-byte swizzle) per softmax warp
    // at a time, two per row block.
    static constexpr uint32_t OST_WARP = 32 * 128;
    static constexpr uint32_t OFF_OST = OFF_V + VST * V_BYTES;   // 1024-byte aligned
    static_assert(OFF_OST % 1024 == 0, "staging alignment");
    static constexpr uint32_t OFF_BAR = OFF_OST + 8 * OST_WARP;
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + KST;
    static constexpr int B_VFULL = B_KEMPTY + KST;
    static constexpr int B_VEMPTY = B_VFULL + VST;
    static constexpr int B_SFULL = B_VEMPTY + VST;   // [tile]
    static constexpr int B_PFULL = B_SFULL + 2;      // [tile]
    static constexpr int B_OFULL = B_PFULL + 2;
    static constexpr int B_OFREE = B_OFULL + 1;      // persistent: O read by the epilogue (count 256)
    static constexpr int B_QEMPTY = B_OFREE + 1;     // persistent: Q tiles no longer read
    static constexpr int B_DRAIN = B_QEMPTY + 1;     // issuer: every issued MMA complete (error path)
    static constexpr int NBAR = B_DRAIN + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
    static constexpr uint32_t USED = OFF_TMEM_SLOT + 16;
    static constexpr uint32_t SMEM_BYTES = USED + 1024;
    static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 384;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 384;
    static_assert(USED + 1024 <= 227u * 1024u, "shared memory");
};

template <bool CAUSAL, bool PERSIST = false>
__global__ void __launch_bounds__(384, 1)
standard_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                     const StandardParams p) {
    using L = StandardLayout;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Two query tiles per CTA; heaviest pairs first under causal masking.
    // Without PERSIST the CTA owns pair (blockIdx.x, y, z); with it, pair
    // number t = k G + (k even ? c : G - 1 - c) of the (b, h)-major,
    // heaviest-first order for k = 0, 1, ... (c = blockIdx.x, G = gridDim.x).
    const int num_pairs = (p.Nq + 2 * L::BM - 1) / (2 * L::BM);
    const int diag = p.Nk - p.Nq;
    auto tile = [&](int k, int& pr, int& h, int& b) -> bool {
        if constexpr (!PERSIST) {
            if (p.head_group > 0) {   // as in the differential prefill
                const unsigned BH = (unsigned)p.H * (unsigned)p.B, HG = p.head_group, t = blockIdx.x;
                const unsigned NT = (unsigned)num_pairs;
                const unsigned g = t / (HG * NT), r = t - g * HG * NT;
                const unsigned ng = BH - g * HG < HG ? BH - g * HG : HG;
                const unsigned w = r / ng, bh = g * HG + (r - w * ng);
                pr = num_pairs - 1 - (int)w;
                const unsigned bb = bh / (unsigned)p.H;
                h = (int)(bh - bb * (unsigned)p.H);
                b = (int)bb;
            } else {
                pr = num_pairs - 1 - (int)blockIdx.x;
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
            const unsigned BH = (unsigned)p.H * (unsigned)p.B, NT = (unsigned)num_pairs;
            if (t >= NT * BH) return false;
            unsigned bh, w;
            if (p.weight_major) {   // as in the differential prefill
                w = div_inv(t, p.div_major_m, p.div_major_s);
                bh = t - w * BH;
            } else {
                bh = div_inv(t, p.div_major_m, p.div_major_s);
                w = t - bh * NT;
            }
            pr = num_pairs - 1 - (int)w;
            const unsigned bb = div_inv(bh, p.div_h_m, p.div_h_s);
            h = (int)(bh - bb * (unsigned)p.H);
            b = (int)bb;
            return true;
        }
    };
    auto kv_tiles = [&](int pr) -> int {
        int kv_end = p.Nk;
        if (CAUSAL) kv_end = min(p.Nk, pr * 2 * L::BM + 2 * L::BM + diag);
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
            mbar_init(bar(L::B_PFULL + r), 4);   // one elected lane per softmax warp
        }
        mbar_init(bar(L::B_OFULL), 1);
        mbar_init(bar(L::B_OFREE), 256);
        mbar_init(bar(L::B_QEMPTY), 1);
        mbar_init(bar(L::B_DRAIN), 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        if constexpr (PERSIST) prefetch_tensormap(&tm_out);
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
            // Stage counters run on across tile pairs.
            int k_issued = 0, v_issued = 0, q_issued = 0;
            int pr, h, b;
            for (int k = 0; ok && tile(k, pr, h, b); ++k) {
                if (k > 0) {
                    ok = mbar_wait(bar(L::B_QEMPTY), (k - 1) & 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                }
                const int q0 = pr * 2 * L::BM;
                mbar_arrive_expect_tx(bar(L::B_Q), 2 * L::Q_BYTES);
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int a = 0; a < 2; ++a)
                        tma_load_4d(sb + L::OFF_Q + (uint32_t)r * L::Q_BYTES + (uint32_t)a * L::ATOM, &tm_q,
                                    bar(L::B_Q), a * 64, q0 + r * L::BM, h, b);
                ++q_issued;
                const int n_kv = kv_tiles(pr);
                for (int j = 0; j < n_kv; ++j) {
                    const int ks = k_issued % L::KST;
                    ok = mbar_wait(bar(L::B_KEMPTY + ks), ((k_issued / L::KST) & 1) ^ 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                    const uint32_t kst = sb + L::OFF_K + (uint32_t)ks * L::K_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_KFULL + ks), L::K_BYTES);
#pragma unroll
                    for (int a = 0; a < 2; ++a)
                        tma_load_4d(kst + (uint32_t)a * L::ATOM, &tm_k, bar(L::B_KFULL + ks), a * 64, j * L::BN, h, b);
                    ++k_issued;
                    const int vs = v_issued % L::VST;
                    ok = mbar_wait(bar(L::B_VEMPTY + vs), ((v_issued / L::VST) & 1) ^ 1, ERR_SITE_PREFILL_PRODUCER);
                    if (!ok) break;
                    const uint32_t vsm = sb + L::OFF_V + (uint32_t)vs * L::V_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_VFULL + vs), L::V_BYTES);
#pragma unroll
                    for (int a = 0; a < 2; ++a)
                        tma_load_4d(vsm + (uint32_t)a * L::ATOM, &tm_v, bar(L::B_VFULL + vs), a * 64, j * L::BN, h, b);
                    ++v_issued;
                }
                if constexpr (!PERSIST) break;
            }
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
            constexpr uint32_t idesc_qk = idesc_bf16_f32(L::BM, L::BN, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(L::BM, L::DV, true);
            // Every lane waits; a wait that ran out on any lane ends the loop on all.
            auto wait = [&](int i, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ERR_SITE_PREFILL_MMA));
            };
            bool ok = wait(L::B_Q, 0);
            tc_fence_after();
            const uint32_t s_col[2] = {L::TM_S0, L::TM_S1};
            const uint32_t o_col[2] = {L::TM_O0, L::TM_O1};
            int g = 0;   // key tiles of earlier tile pairs (ring stage and phase counter)
            int pr, h, b;
            for (int k = 0; ok && tile(k, pr, h, b); ++k) {
            const int n_kv = kv_tiles(pr);
            if (k > 0) {
                ok = wait(L::B_Q, k & 1);
                if (!ok) break;
                tc_fence_after();
            }
            // Step j: P V of key tile j - 1, then the scores of tile j, per
            // query tile.  P V waits only for V and P, the scores only for K.
            for (int j = 0; j <= n_kv && ok; ++j) {
                const int gj = g + j;
                const int ks = gj % L::KST;
                const int jv = j - 1, gv = gj - 1;
                const int vs = (gv + L::VST) % L::VST;
                const uint32_t vsm = sb + L::OFF_V + (uint32_t)vs * L::V_BYTES;
                const uint32_t kst = sb + L::OFF_K + (uint32_t)ks * L::K_BYTES;
                for (int r = 0; r < 2; ++r) {
                    if (jv >= 0) {
                        ok = (r > 0 || wait(L::B_VFULL + vs, (gv / L::VST) & 1)) && wait(L::B_PFULL + r, gv & 1);
                        if (!ok) break;
                        if (PERSIST && jv == 0 && r == 0 && k > 0) {
                            // The first product of a tile pair overwrites O:
                            // the previous pair's epilogue must have read it.
                            ok = wait(L::B_OFREE, (k - 1) & 1);
                            if (!ok) break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < L::BN / 16; ++kk) {
                            const uint64_t bdesc = smem_desc(vsm + (uint32_t)kk * 16 * 128, L::ATOM, 1024, SWZ_128B);
                            mma_ts_warp(tmem + o_col[r], tmem + s_col[r] + (uint32_t)kk * 8, bdesc, idesc_pv,
                                        (jv > 0 || kk > 0) ? 1u : 0u);
                        }
                        if (r == 1) mma_commit_warp(bar(L::B_VEMPTY + vs));
                    }
                    if (j < n_kv) {
                        if (r == 0) {
                            ok = wait(L::B_KFULL + ks, (gj / L::KST) & 1);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        const uint32_t qt = sb + L::OFF_Q + (uint32_t)r * L::Q_BYTES;
#pragma unroll
                        for (int kk = 0; kk < L::D / 16; ++kk) {
                            // K-step kk: 64-column atom kk / 4, 32-byte slice kk % 4 within it.
                            const uint32_t off = (uint32_t)(kk >> 2) * L::ATOM + (uint32_t)(kk & 3) * 32;
                            mma_ss_warp(tmem + s_col[r], smem_desc(qt + off, 16, 1024, SWZ_128B),
                                        smem_desc(kst + off, 16, 1024, SWZ_128B), idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        mma_commit_warp(bar(L::B_SFULL + r));
                        if (r == 1) mma_commit_warp(bar(L::B_KEMPTY + ks));
                        if (PERSIST && r == 1 && j == n_kv - 1) mma_commit_warp(bar(L::B_QEMPTY));
                    }
                }
            }
            g += n_kv;
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
        const int r = (warp - 4) >> 2;           // query tile
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
        const uint32_t s_col = r ? L::TM_S1 : L::TM_S0;
        const uint32_t o_col = r ? L::TM_O1 : L::TM_O0;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int g = 0;   // key tiles of earlier tile pairs (barrier phase counter)
        int pr, h, b;
        for (int k = 0; ok && tile(k, pr, h, b); ++k) {
        const int n_kv = kv_tiles(pr);
        const int qi = pr * 2 * L::BM + r * L::BM + row;
        const int kmax = CAUSAL ? min(qi + diag, p.Nk - 1) : p.Nk - 1;
        float m = -INFINITY;
        float l = 0.f;
        for (int j = 0; j < n_kv; ++j) {
            ok = mbar_wait(bar(L::B_SFULL + r), (g + j) & 1, ERR_SITE_PREFILL_SOFTMAX);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t sv[128];
            tmem_ld128(tmem + t_lane + s_col, sv);
            const int kb = j * L::BN;
            if (kb + L::BN - 1 > kmax) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (kb + i > kmax) sv[i] = __float_as_uint(-INFINITY);
            }
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
            const float nm = (m == -INFINITY) ? 0.f : -m;
            uint32_t pk[64];
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, a4 = 0.f, a5 = 0.f, a6 = 0.f, a7 = 0.f;
#pragma unroll
            for (int i = 0; i < 128; i += 8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2)
                    fma2_bcast(x[e], x[e + 1], __uint_as_float(sv[i + e]), __uint_as_float(sv[i + e + 1]), sl2, nm);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = fast_exp2(x[e]);
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pk[(i >> 1) + e] = w[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                acc_bf16x2(a0, a1, w[0]);
                acc_bf16x2(a2, a3, w[1]);
                acc_bf16x2(a4, a5, w[2]);
                acc_bf16x2(a6, a7, w[3]);
            }
            l += ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
            tmem_st64(tmem + t_lane + s_col, pk);
            if (rescale) {
                // O *= alpha once the scores' registers are free; the
                // previous P V has completed and this tile's waits for the
                // hand-off below.
#pragma unroll
                for (int c = 0; c < L::DV / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + t_lane + o_col + 32u * c, ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(tmem + t_lane + o_col + 32u * c, ov);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::B_PFULL + r));
        }

        // ------------------------------------------------------------ epilogue: out = O_r / l_r
        g += n_kv;
        if (!mbar_wait(bar(L::B_OFULL), k & 1, ERR_SITE_PREFILL_EPILOGUE)) ok = false;
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        const float inv = 1.0f / l;
        if constexpr (PERSIST) {
            // Two 64-column halves through this warp's staging box: row `row`
            // puts 16-byte chunk i at chunk position i ^ (row & 7).  Rows at
            // or past Nq are staged too; the TMA store does not write them.
            const uint32_t box = L::OFF_OST + (uint32_t)(r * 4 + wq) * L::OST_WARP;
            uint8_t* srow = smem + box + (uint32_t)lane * 128u;
            const size_t rowoff = (((size_t)b * p.H + h) * p.Nq + qi) * L::DV;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + t_lane + o_col + 64u * c2 + 32u * c, ov);
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(ov[i]) * inv;
                    if (p.out_f32 && qi < p.Nq) {
                        float4* dst = reinterpret_cast<float4*>(p.out_f32 + rowoff + 64 * c2 + 32 * c);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[16 * c + i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
                }
                if (c2 == 1) {
                    // O has been read: the next pair's products may overwrite it.
                    tc_fence_before();
                    mbar_arrive(bar(L::B_OFREE));
                }
                // The previous store from this buffer must have read it.
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    *reinterpret_cast<uint4*>(srow + (((uint32_t)i ^ (uint32_t)(lane & 7)) << 4)) =
                        make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_4d(&tm_out, sb + box, 64 * c2, pr * 2 * L::BM + r * L::BM + wq * 32, h, b);
                    bulk_commit_group();
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < L::DV / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tmem + t_lane + o_col + 32u * c, ov);
                if (qi < p.Nq) {
                    const size_t off = (((size_t)b * p.H + h) * p.Nq + qi) * L::DV + 32 * c;
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(ov[i]) * inv;
                    if (p.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(p.out_f32 + off);
#pragma unroll
                        for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(p.out + off);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_bf16x2(o[8 * i], o[8 * i + 1]), pack_bf16x2(o[8 * i + 2], o[8 * i + 3]),
                                            pack_bf16x2(o[8 * i + 4], o[8 * i + 5]), pack_bf16x2(o[8 * i + 6], o[8 * i + 7]));
                }
            }
        }
        if constexpr (!PERSIST) break;
        }   // tile pairs
        // Leave with no TMA store reading shared memory or still writing.
        if constexpr (PERSIST)
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
