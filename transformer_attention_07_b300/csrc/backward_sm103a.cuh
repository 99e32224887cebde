// Differential-attention backward pass for sm_103a.
//
// The forward pass (Differential Transformer pages: the DiffAttn formula of
// the iloveeagents.com Q&A, "Mathematical Formula", where lambda is a
// learnable scalar; steps 2-4 of llmbytes.dev "How Differential Attention
// Cancels Common-Mode Noise") is, per head and query row i,
//     o_i = sum_j (A1_ij - lambda A2_ij) v_j,   A_r = softmax(s Q_r K_r^T), s = 1/sqrt(d)
//     y_i = (1 - lambda_init) gamma * (o_i - mu_i) * rstd_i.
// Given dy = dL/dy, the chain rule in reverse order gives
//     do_i    = rstd (g - mean(g) - xhat mean(g xhat)),  g = (1 - lambda_init) gamma dy
//     dgamma  = (1 - lambda_init) sum_i dy_i xhat_i
//     dP_ij   = do_i . v_j                     (shared by both maps)
//     D1_i    = do_i . (A1 V)_i,  D2_i = do_i . (A2 V)_i
//     dS1_ij  = A1_ij (dP_ij - D1_i),   dS2_ij = -lambda A2_ij (dP_ij - D2_i)
//     dV_j    = sum_i (A1_ij - lambda A2_ij) do_i
//     dQ_r,i  = s sum_j dS_r,ij k_r,j,    dK_r,j = s sum_i dS_r,ij q_r,i
//     dlambda = -sum_i D2_i.
// The forward stores each map's log-sum-exp and A2 V, so both maps' rows
// A_r,ij = exp(s q_r,i . k_r,j - lse_r,i) are recomputed tile by tile and no
// N x N matrix is ever formed.
//
// Four kernels:
//   bwd_prep_kernel     one warp per row: GroupNorm backward, do (bf16),
//                       D1, D2, per-row constants for the tile kernels, and
//                       fixed-order partial sums of dgamma and dlambda.
//   bwd_dq_kernel       one CTA per 128 query rows; walks 128-key tiles:
//                       S_r = Q_r K_r^T, dP = dO V^T on the tensor core,
//                       dS_r in registers, dQ_r += dS_r K_r (dS_r from TMEM);
//                       the next tile's scores follow each map's dQ product.
//   bwd_dkv_kernel      one CTA per 128 keys; walks the query tiles in
//                       64-query units through two tensor-memory slots:
//                       S_r^T = K_r Q_r^T, dP^T = V dO^T, then
//                       dV += (A1 - lambda A2)^T dO, dK_r += dS_r^T Q_r;
//                       one unit's products run while the dS warps work on
//                       the other, the dS arithmetic in 16-query chunks that
//                       overlap the previous chunk's products.
//   bwd_finalize_kernel the dgamma and dlambda sums, in a fixed order.
// dQ and dK/dV come from separate sweeps (the dQ sweep recomputes S and dP),
// so every gradient is written once, by one CTA, without atomics: results
// are deterministic.
#pragma once

#include "sm103_ptx.cuh"

namespace diffattn {

struct BwdParams {
    int B, H, Nq, Nk;
    int Nq_pad;             // Nq rounded up to 128: rows of the per-row constants
    int nchunk;             // Nq_pad / 64: row blocks of the prep kernel
    float lambda, lambda_init, eps;
    float scale_log2;       // log2(e) / sqrt(d)
    float scale;            // 1 / sqrt(d)
    const float* gamma;     // [H*dv] or null (ones)
    const uint16_t* dy;     // bf16 [B,H,Nq,dv]
    const float* o;         // fp32 [B,H,Nq,dv]: pre-norm forward output
    const float* o2;        // fp32 [B,H,Nq,dv]: A2 V
    const float* lse;       // fp32 [2,B,H,Nq]: per-map log-sum-exp (natural log)
    uint16_t* dout;         // bf16 [B,H,Nq,dv]: gradient of the pre-norm output
    float4* rowc;           // [B*H*Nq_pad]: (lse1 log2 e, lse2 log2 e, D1, D2); padding rows (inf, inf, 0, 0)
    float* rowt;            // [B*H*Nq_pad/128][4][128]: the same constants negated, one row of 128
                            // per constant and 128-row block (padding rows: -inf, -inf, 0, 0)
    float* gpart;           // [B*H*nchunk, dv]: dgamma partial sums
    float* lpart;           // [B*H*nchunk]: dlambda partial sums
    uint16_t *dq1, *dq2;    // bf16 [B,H,Nq,d]
    uint16_t *dk1, *dk2;    // bf16 [B,H,Nk,d]
    uint16_t* dv;           // bf16 [B,H,Nk,dv]
    float* dlambda;         // one float, or null
    float* dgamma;          // [H*dv], or null
};

constexpr int kBwdPrepRows = 64;   // rows per prep block (8 warps x 8 rows)
constexpr int kBwdRowPad = 128;    // Nq_pad granularity

// ----------------------------------------------------------------- prep

template <int DV>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdParams p) {
    constexpr int CPL = DV / 32;   // channels per lane, contiguous
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * p.H + h;
    const size_t BH = (size_t)p.B * p.H;
    const float kappa = 1.0f - p.lambda_init;
    const float log2e = 1.4426950408889634f;
    const int c0 = lane * CPL;
    float gam[CPL], gacc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        gam[e] = p.gamma ? p.gamma[(size_t)h * DV + c0 + e] : 1.0f;
        gacc[e] = 0.0f;
    }
    float lacc = 0.0f;
    constexpr int RPW = kBwdPrepRows / 8;
    for (int rr = 0; rr < RPW; ++rr) {
        const int i = chunk * kBwdPrepRows + warp * RPW + rr;
        float4 rc = make_float4(INFINITY, INFINITY, 0.0f, 0.0f);
        if (i < p.Nq) {
            const size_t row = bh * p.Nq + i;
            float o[CPL], o2[CPL], dy[CPL];
#pragma unroll
            for (int e = 0; e < CPL; ++e) {
                o[e] = p.o[row * DV + c0 + e];
                o2[e] = p.o2[row * DV + c0 + e];
                dy[e] = __uint_as_float((uint32_t)p.dy[row * DV + c0 + e] << 16);
            }
            // GroupNorm statistics of the row (one group = this head).
            float s = 0.0f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) s += o[e];
            const float mu = warp_sum(s) * (1.0f / DV);
            float q = 0.0f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) q += (o[e] - mu) * (o[e] - mu);
            const float rstd = rsqrtf(warp_sum(q) * (1.0f / DV) + p.eps);
            // Through the gain and scale, then the normalisation.
            float xh[CPL], g[CPL];
            float sg = 0.0f, sgx = 0.0f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) {
                xh[e] = (o[e] - mu) * rstd;
                g[e] = kappa * gam[e] * dy[e];
                gacc[e] += kappa * dy[e] * xh[e];
                sg += g[e];
                sgx += g[e] * xh[e];
            }
            const float mg = warp_sum(sg) * (1.0f / DV);
            const float mgx = warp_sum(sgx) * (1.0f / DV);
            // do, rounded to bf16 as the tile kernels' MMAs consume it; D1 and
            // D2 use the rounded values so that sum_j dS_r,ij = 0 holds for the
            // operand the tensor core sees.
            // dlambda takes the unrounded do: its terms cancel to rounding
            // level when the norm makes y insensitive to lambda.
            float d1 = 0.0f, d2 = 0.0f, dl = 0.0f;
            uint32_t packed[CPL / 2];
#pragma unroll
            for (int e = 0; e < CPL; e += 2) {
                const float a0 = rstd * (g[e] - mg - xh[e] * mgx);
                const float a1 = rstd * (g[e + 1] - mg - xh[e + 1] * mgx);
                dl += a0 * o2[e] + a1 * o2[e + 1];
                packed[e / 2] = pack_bf16x2(a0, a1);
                const float r0 = bf16lo_to_f32(packed[e / 2]), r1 = bf16hi_to_f32(packed[e / 2]);
                d2 += r0 * o2[e] + r1 * o2[e + 1];
                d1 += r0 * (o[e] + p.lambda * o2[e]) + r1 * (o[e + 1] + p.lambda * o2[e + 1]);
            }
            if constexpr (CPL == 4) {
                *reinterpret_cast<uint2*>(p.dout + row * DV + c0) = make_uint2(packed[0], packed[1]);
            } else {
                *reinterpret_cast<uint32_t*>(p.dout + row * DV + c0) = packed[0];
            }
            d1 = warp_sum(d1);
            d2 = warp_sum(d2);
            lacc -= warp_sum(dl);
            rc = make_float4(p.lse[bh * p.Nq + i] * log2e, p.lse[(BH + bh) * p.Nq + i] * log2e, d1, d2);
        }
        if (lane == 0 && i < p.Nq_pad) p.rowc[bh * p.Nq_pad + i] = rc;
        if (lane < 4 && i < p.Nq_pad) {
            const float c = lane == 0 ? rc.x : lane == 1 ? rc.y : lane == 2 ? rc.z : rc.w;
            p.rowt[(bh * p.Nq_pad + (i & ~127)) * 4 + lane * 128 + (i & 127)] = -c;
        }
    }
    // Block sums of the dgamma and dlambda contributions, warps in order.
    __shared__ float sg_part[8][DV];
    __shared__ float sl_part[8];
#pragma unroll
    for (int e = 0; e < CPL; ++e) sg_part[warp][c0 + e] = gacc[e];
    if (lane == 0) sl_part[warp] = lacc;
    __syncthreads();
    const size_t part = bh * p.nchunk + chunk;
    for (int c = threadIdx.x; c < DV; c += blockDim.x) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += sg_part[w][c];
        p.gpart[part * DV + c] = t;
    }
    if (threadIdx.x == 0) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += sl_part[w];
        p.lpart[part] = t;
    }
}

// ----------------------------------------------------------------- finalize

// Blocks 0..H-1: dgamma of head h (sum over batches and row blocks); block H:
// dlambda.  Fixed summation order, so repeated runs agree bit for bit.
template <int DV>
__global__ void __launch_bounds__(256) bwd_finalize_kernel(const BwdParams p) {
    __shared__ float red[256];
    const int t = threadIdx.x;
    if ((int)blockIdx.x < p.H) {
        if (!p.dgamma) return;
        const int h = blockIdx.x;
        constexpr int G = 256 / DV;
        const int c = t % DV, g = t / DV;
        float acc = 0.0f;
        for (int b = 0; b < p.B; ++b) {
            const float* base = p.gpart + ((size_t)b * p.H + h) * p.nchunk * DV;
#pragma unroll 8
            for (int x = g; x < p.nchunk; x += G) acc += base[(size_t)x * DV + c];
        }
        red[t] = acc;
        __syncthreads();
        if (g == 0) {
            float s = 0.0f;
            for (int k = 0; k < G; ++k) s += red[k * DV + c];
            p.dgamma[(size_t)h * DV + c] = s;
        }
    } else {
        if (!p.dlambda) return;
        const size_t n = (size_t)p.B * p.H * p.nchunk;
        float acc = 0.0f;
        for (size_t x = t; x < n; x += 256) acc += p.lpart[x];
        red[t] = acc;
        __syncthreads();
        for (int s = 128; s > 0; s >>= 1) {
            if (t < s) red[t] += red[t + s];
            __syncthreads();
        }
        if (t == 0) *p.dlambda = red[0];
    }
}

// ----------------------------------------------------------------- dQ sweep

template <int D, int DV>
struct BwdDqLayout {
    static constexpr int BM = 128;   // query rows per CTA (MMA M)
    static constexpr int BN = 128;   // keys per tile (MMA N of S and dP)
    // K1/K2 and V come in separate rings: V is read by the first product of
    // a tile (dP, issued a tile ahead), K by the last (dQ), so V runs deeper.
    static constexpr int KST = 2;    // K1/K2 ring depth
    static constexpr int VST = 3;    // V ring depth
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t DO_BOX = BM * 128;       // one 64-column box of dO
    static constexpr uint32_t DO_BYTES = BM * DV * 2;
    static constexpr uint32_t K_BYTES = BN * D * 2;
    static constexpr uint32_t V_BOX = BN * 128;
    static constexpr uint32_t V_BYTES = BN * DV * 2;
    static constexpr uint32_t KSTAGE = 2 * K_BYTES;   // K1, K2
    static constexpr uint32_t OFF_Q1 = 0;
    static constexpr uint32_t OFF_Q2 = Q_BYTES;
    static constexpr uint32_t OFF_DO = 2 * Q_BYTES;
    static constexpr uint32_t OFF_K = OFF_DO + DO_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KST * KSTAGE;
    static constexpr uint32_t OFF_BAR = OFF_V + VST * V_BYTES;
    static constexpr int B_Q = 0;
    static constexpr int B_KFULL = 1;
    static constexpr int B_KEMPTY = B_KFULL + KST;
    static constexpr int B_VFULL = B_KEMPTY + KST;
    static constexpr int B_VEMPTY = B_VFULL + VST;
    static constexpr int B_SFULL = B_VEMPTY + VST;   // [map]: S_r (and dP) of the tile in TMEM
    static constexpr int B_DPFREE = B_SFULL + 2;     // both maps have dP in registers
    static constexpr int B_PFULL = B_DPFREE + 1;     // [map]: dS_r written over S_r
    static constexpr int B_DQFULL = B_PFULL + 2;
    static constexpr int NBAR = B_DQFULL + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
    static constexpr uint32_t USED = OFF_TMEM_SLOT + 16;
    // +1024 for aligning the dynamic base; at least 120 KB so that a single
    // CTA (which takes all 512 TMEM columns) is resident per SM.
    static constexpr uint32_t SMEM_BYTES = (USED + 1024 > 120u * 1024u) ? USED + 1024 : 120u * 1024u;
    // Tensor memory: S1, S2, dP (128 columns each; dS_r in bf16 is written
    // over the first 64 columns of S_r), then the two dQ accumulators.
    static constexpr uint32_t TM_S1 = 0, TM_S2 = 128, TM_DP = 256, TM_DQ1 = 384, TM_DQ2 = 384 + D;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 320;
    // Q/K rows are one swizzle span wide (128 or 64 bytes); dO and V come in
    // 64-column boxes of 128-byte rows.
    static constexpr uint32_t QK_ROW = D * 2;
    static constexpr uint32_t QK_SWZ = QK_ROW == 128 ? SWZ_128B : SWZ_64B;
    static constexpr uint32_t QK_SBO = 8 * QK_ROW;
    static_assert((D == 64 && DV == 128) || (D == 32 && DV == 64), "backward widths");
    static_assert(SMEM_BYTES <= 227u * 1024u && SMEM_BYTES > 114u * 1024u, "one CTA per SM");
};

template <int D, int DV, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_q2,
              const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k1,
              const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v,
              const BwdParams p) {
    using L = BwdDqLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_qt = (p.Nq + L::BM - 1) / L::BM;
    const int qt = num_qt - 1 - (int)blockIdx.x;   // heaviest tiles first under causal masking
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * p.H + h;
    const int q0 = qt * L::BM;
    const int diag = p.Nk - p.Nq;
    int kv_end = p.Nk;
    if (CAUSAL) kv_end = min(p.Nk, q0 + L::BM + diag);
    const int n_kv = (kv_end + L::BN - 1) / L::BN;

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
            mbar_init(bar(L::B_PFULL + r), 4);
        }
        mbar_init(bar(L::B_DPFREE), 8);
        mbar_init(bar(L::B_DQFULL), 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q1);
        prefetch_tensormap(&tm_q2);
        prefetch_tensormap(&tm_do);
        prefetch_tensormap(&tm_k1);
        prefetch_tensormap(&tm_k2);
        prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(sb + L::OFF_TMEM_SLOT, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM_SLOT);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(bar(L::B_Q), 2 * L::Q_BYTES + L::DO_BYTES);
            tma_load_4d(sb + L::OFF_Q1, &tm_q1, bar(L::B_Q), 0, q0, h, b);
            tma_load_4d(sb + L::OFF_Q2, &tm_q2, bar(L::B_Q), 0, q0, h, b);
#pragma unroll
            for (int c = 0; c < DV / 64; ++c)
                tma_load_4d(sb + L::OFF_DO + (uint32_t)c * L::DO_BOX, &tm_do, bar(L::B_Q), c * 64, q0, h, b);
            // V tile j goes VST - 1 tiles ahead of K tile j.
            auto load_v = [&](int j) -> bool {
                const int vs = j % L::VST;
                if (!mbar_wait(bar(L::B_VEMPTY + vs), ((j / L::VST) & 1) ^ 1, ERR_SITE_BWD_PRODUCER)) return false;
                const uint32_t st = sb + L::OFF_V + (uint32_t)vs * L::V_BYTES;
                mbar_arrive_expect_tx(bar(L::B_VFULL + vs), L::V_BYTES);
#pragma unroll
                for (int c = 0; c < DV / 64; ++c)
                    tma_load_4d(st + (uint32_t)c * L::V_BOX, &tm_v, bar(L::B_VFULL + vs), c * 64, j * L::BN, h, b);
                return true;
            };
            int issued_k = 0, issued_v = 0;
            for (int j = 0; j < L::VST - 1 && j < n_kv && ok; ++j) ok = load_v(j), issued_v += ok;
            for (int j = 0; j < n_kv && ok; ++j) {
                const int ks = j % L::KST;
                ok = mbar_wait(bar(L::B_KEMPTY + ks), ((j / L::KST) & 1) ^ 1, ERR_SITE_BWD_PRODUCER);
                if (!ok) break;
                const uint32_t st = sb + L::OFF_K + (uint32_t)ks * L::KSTAGE;
                mbar_arrive_expect_tx(bar(L::B_KFULL + ks), L::KSTAGE);
                tma_load_4d(st, &tm_k1, bar(L::B_KFULL + ks), 0, j * L::BN, h, b);
                tma_load_4d(st + L::K_BYTES, &tm_k2, bar(L::B_KFULL + ks), 0, j * L::BN, h, b);
                ++issued_k;
                if (j + L::VST - 1 < n_kv) {
                    ok = load_v(j + L::VST - 1);
                    issued_v += ok;
                }
            }
            // Every copy lands before the CTA exits.
            mbar_wait(bar(L::B_Q), 0, ERR_SITE_BWD_DRAIN);
            for (int s = 0; s < L::KST && s < issued_k; ++s) {
                const int last = s + ((issued_k - 1 - s) / L::KST) * L::KST;
                mbar_wait(bar(L::B_KFULL + s), (last / L::KST) & 1, ERR_SITE_BWD_DRAIN);
            }
            for (int s = 0; s < L::VST && s < issued_v; ++s) {
                const int last = s + ((issued_v - 1 - s) / L::VST) * L::VST;
                mbar_wait(bar(L::B_VFULL + s), (last / L::VST) & 1, ERR_SITE_BWD_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop with warp-uniform values; each MMA and
        // commit is issued by one elected lane (the *_warp wrappers).
        {
            // Every lane waits; a wait that ran out on any lane ends the loop on all.
            auto wait = [&](uint32_t b, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, ERR_SITE_BWD_MMA));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(L::BM, L::BN, false);   // S, dP: K-major operands
            constexpr uint32_t idesc_dq = idesc_bf16_f32(L::BM, D, true);       // dQ: K tile MN-major
            bool ok = wait(bar(L::B_Q), 0);
            tc_fence_after();
            const uint64_t dq1 = smem_desc(sb + L::OFF_Q1, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t dq2 = smem_desc(sb + L::OFF_Q2, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t ddo = smem_desc(sb + L::OFF_DO, 16, 1024, SWZ_128B);
            const uint64_t dk0 = smem_desc(sb + L::OFF_K, 16, L::QK_SBO, L::QK_SWZ);                 // K1, stage 0
            const uint64_t dkm0 = smem_desc(sb + L::OFF_K, L::K_BYTES, L::QK_SBO, L::QK_SWZ);        // K1 as MN-major B
            const uint64_t dv0 = smem_desc(sb + L::OFF_V, 16, 1024, SWZ_128B);                       // V, stage 0
            constexpr uint64_t KSTAGE16 = L::KSTAGE >> 4, VSTAGE16 = L::V_BYTES >> 4, K2OFF = L::K_BYTES >> 4;
            // dP = dO V^T: k over dv, two 64-column boxes of each operand.
            auto dp_mma = [&](uint64_t so) {
#pragma unroll
                for (int k = 0; k < DV / 16; ++k)
                    mma_ss_warp(tmem + L::TM_DP, ddo + (uint64_t)(((k >> 2) * L::DO_BOX + (k & 3) * 32) >> 4),
                           dv0 + so + (uint64_t)(((k >> 2) * L::V_BOX + (k & 3) * 32) >> 4), idesc_s,
                           k > 0 ? 1u : 0u);
            };
            // S_r = Q_r K_r^T.
            auto s_mma = [&](int r, uint64_t so) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_warp(tmem + (r ? L::TM_S2 : L::TM_S1), (r ? dq2 : dq1) + (uint64_t)(2 * k),
                           dk0 + so + (r ? K2OFF : 0) + (uint64_t)(2 * k), idesc_s, k > 0 ? 1u : 0u);
            };
            // dQ_r += dS_r K_r: dS_r (bf16) in the first 64 columns of S_r,
            // 8 columns per 16 keys; the K tile read MN-major.
            auto dq_mma = [&](int r, uint64_t so, bool first) {
#pragma unroll
                for (int k = 0; k < L::BN / 16; ++k)
                    mma_ts_warp(tmem + (r ? L::TM_DQ2 : L::TM_DQ1), tmem + (r ? L::TM_S2 : L::TM_S1) + 8u * k,
                           dkm0 + so + (r ? K2OFF : 0) + (uint64_t)(k * (16 * L::QK_ROW >> 4)), idesc_dq,
                           (!first || k > 0) ? 1u : 0u);
            };
            if (ok) ok = wait(bar(L::B_VFULL + 0), 0);
            if (ok) ok = wait(bar(L::B_KFULL + 0), 0);
            if (ok) {
                tc_fence_after();
                dp_mma(0);
                mma_commit_warp(bar(L::B_VEMPTY + 0));
                s_mma(0, 0);
                mma_commit_warp(bar(L::B_SFULL + 0));
                s_mma(1, 0);
                mma_commit_warp(bar(L::B_SFULL + 1));
            }
            // Per tile j: map 1's dQ product, its next scores, then the next
            // dP (once both maps hold this tile's dP), which completes the
            // next tile's inputs for map 1; then map 2's dQ product and next
            // scores.  Map 2's dS warps load dP last, so the next dP waits for
            // them only after map 1's products are queued.
            for (int j = 0; j < n_kv && ok; ++j) {
                const uint64_t so = (uint64_t)(j % L::KST) * KSTAGE16;
                const bool more = j + 1 < n_kv;
                const uint64_t sn = (uint64_t)((j + 1) % L::KST) * KSTAGE16;
                ok = wait(bar(L::B_PFULL + 0), j & 1);
                if (!ok) break;
                tc_fence_after();
                dq_mma(0, so, j == 0);
                if (more) {
                    ok = wait(bar(L::B_KFULL + (j + 1) % L::KST), ((j + 1) / L::KST) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    s_mma(0, sn);
                    const int vs = (j + 1) % L::VST;
                    ok = wait(bar(L::B_VFULL + vs), ((j + 1) / L::VST) & 1);
                    ok = ok && wait(bar(L::B_DPFREE), j & 1);
                    if (!ok) break;
                    tc_fence_after();
                    dp_mma((uint64_t)vs * VSTAGE16);
                    mma_commit_warp(bar(L::B_VEMPTY + vs));
                    mma_commit_warp(bar(L::B_SFULL + 0));
                }
                ok = wait(bar(L::B_PFULL + 1), j & 1);
                if (!ok) break;
                tc_fence_after();
                dq_mma(1, so, j == 0);
                mma_commit_warp(bar(L::B_KEMPTY + j % L::KST));
                if (more) {
                    s_mma(1, sn);
                    mma_commit_warp(bar(L::B_SFULL + 1));
                }
            }
            mma_commit_warp(bar(L::B_DQFULL));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ dS (warps 2-9)
        const int r = (warp - 2) >> 2;          // map
        const int wq = warp & 3;                // TMEM lane quarter
        const int row = wq * 32 + lane;
        const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
        const int qi = q0 + row;
        const int kmax = CAUSAL ? min(qi + diag, p.Nk - 1) : p.Nk - 1;
        const float4 rc = p.rowc[bh * p.Nq_pad + qi];
        const float nlse = -(r ? rc.y : rc.x);
        const float Dr = r ? rc.w : rc.z;
        const float coef = r ? -p.lambda : 1.0f;
        const float ncd = -coef * Dr;   // dS_r = A_r (coef dP + ncd)
        const float sl2 = p.scale_log2;
        const uint32_t s_col = tmem + t_lane + (r ? L::TM_S2 : L::TM_S1);
        const uint32_t dp_col = tmem + t_lane + L::TM_DP;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            ok = mbar_wait(bar(L::B_SFULL + r), j & 1, ERR_SITE_BWD_SOFTMAX);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int kb = j * L::BN;
            const bool edge = kb + L::BN - 1 > kmax;
            // Four 32-key chunks; chunk c's bf16 dS lands in columns [16c, 16c+16),
            // which this thread has already read.
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t sv[32], dp[32];
                tmem_ld32x2(s_col + 32u * c, sv, dp_col + 32u * c, dp);
                if (c == 3) {
                    // dP is in registers for this map: the next tile's dP may
                    // overwrite it once the other map is there too.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(L::B_DPFREE));
                }
                if (edge) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (kb + 32 * c + i > kmax) sv[i] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float x0, x1;
                    fma2_bcast(x0, x1, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]), sl2, nlse);
                    float t0, t1, d0, d1;
                    fma2_bcast(t0, t1, __uint_as_float(dp[i]), __uint_as_float(dp[i + 1]), coef, ncd);
                    mul2(d0, d1, fast_exp2(x0), fast_exp2(x1), t0, t1);
                    pk[i >> 1] = pack_bf16x2(d0, d1);
                }
                tmem_st16(s_col + 16u * c, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::B_PFULL + r));
        }
        // ------------------------------------------------------------ epilogue
        mbar_wait(bar(L::B_DQFULL), 0, ERR_SITE_BWD_EPILOGUE);
        __syncwarp();
        tc_fence_after();
        uint32_t a[D];
        if constexpr (D == 64)
            tmem_ld64(tmem + t_lane + (r ? L::TM_DQ2 : L::TM_DQ1), a);
        else
            tmem_ld32(tmem + t_lane + (r ? L::TM_DQ2 : L::TM_DQ1), a);
        if (qi < p.Nq) {
            uint4* dst = reinterpret_cast<uint4*>((r ? p.dq2 : p.dq1) + (bh * p.Nq + qi) * D);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(a[8 * i + 2 * e]) * p.scale,
                                       __uint_as_float(a[8 * i + 2 * e + 1]) * p.scale);
                dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ----------------------------------------------------------------- dK/dV sweep

// N fp32 columns of this thread's TMEM lane, times s, rounded to bf16 and
// stored to dst (16-byte aligned) when `store`; the load runs on every lane.
template <int N>
__device__ __forceinline__ void tmem_cols_to_bf16(uint32_t taddr, uint16_t* dst, float s, bool store) {
    static_assert(N == 16 || N == 32, "column count");
    uint32_t a[N];
    if constexpr (N == 16)
        tmem_ld16(taddr, a);
    else
        tmem_ld32(taddr, a);
    if (store) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < N / 8; ++i)
            d4[i] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * i]) * s, __uint_as_float(a[8 * i + 1]) * s),
                               pack_bf16x2(__uint_as_float(a[8 * i + 2]) * s, __uint_as_float(a[8 * i + 3]) * s),
                               pack_bf16x2(__uint_as_float(a[8 * i + 4]) * s, __uint_as_float(a[8 * i + 5]) * s),
                               pack_bf16x2(__uint_as_float(a[8 * i + 6]) * s, __uint_as_float(a[8 * i + 7]) * s));
    }
}

template <int D, int DV>
struct BwdDkvLayout {
    static constexpr int BK = 128;   // keys per CTA (MMA M)
    static constexpr int BQ = 128;   // query rows per staged tile
    static constexpr int BU = 64;    // query rows per unit: half a staged tile (MMA N of S^T and dP^T)
    static constexpr int QST = 2;    // ring depth of (Q1, Q2, dO, row constants)
    static constexpr uint32_t K_BYTES = BK * D * 2;
    static constexpr uint32_t V_BOX = BK * 128;
    static constexpr uint32_t V_BYTES = BK * DV * 2;
    static constexpr uint32_t Q_BYTES = BQ * D * 2;
    static constexpr uint32_t DO_BOX = BQ * 128;
    static constexpr uint32_t DO_BYTES = BQ * DV * 2;
    static constexpr uint32_t RC_BYTES = BQ * 16;
    static constexpr uint32_t STAGE = 2 * Q_BYTES + DO_BYTES + RC_BYTES;   // Q1, Q2, dO, row constants
    static constexpr uint32_t ST_Q2 = Q_BYTES, ST_DO = 2 * Q_BYTES, ST_RC = 2 * Q_BYTES + DO_BYTES;
    static constexpr uint32_t OFF_K1 = 0;
    static constexpr uint32_t OFF_K2 = K_BYTES;
    static constexpr uint32_t OFF_V = 2 * K_BYTES;
    static constexpr uint32_t OFF_Q = OFF_V + V_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_Q + QST * STAGE;
    // dS warps: one per TMEM lane quarter in each of NG column groups of a unit.
    static constexpr int NG = 2;
    static constexpr int GC = BU / NG;               // columns per group (32)
    static constexpr int NDS = 4 * NG;               // dS warps
    static constexpr int CW = 16;                    // queries per chunk: one k-step of the gradient products
    static constexpr int NCH = GC / CW;              // chunks per group
    static constexpr int B_KV = 0;
    static constexpr int B_QFULL = 1;
    static constexpr int B_QEMPTY = B_QFULL + QST;
    static constexpr int B_SFULL = B_QEMPTY + QST;   // [slot]: S1^T and S2^T of the slot's unit complete
    static constexpr int B_SFREE = B_SFULL + 2;      // [slot]: the dS warps hold both in registers
    static constexpr int B_DPFULL = B_SFREE + 2;     // [slot]: dP^T complete
    static constexpr int B_PFULL = B_DPFULL + 2;     // [slot][chunk]: bf16 operands of one chunk of every group
    static constexpr int B_GDONE = B_PFULL + 2 * NCH;   // [slot]: the slot's gradient products complete
    static constexpr int B_DONE = B_GDONE + 2;
    static constexpr int NBAR = B_DONE + 1;
    static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
    static constexpr uint32_t USED = OFF_TMEM_SLOT + 16;
    // +1024 for aligning the dynamic base; at least 120 KB so that a single
    // CTA (which takes all 512 TMEM columns) is resident per SM.
    static constexpr uint32_t SMEM_BYTES = (USED + 1024 > 120u * 1024u) ? USED + 1024 : 120u * 1024u;
    // Tensor memory: the dV, dK1, dK2 accumulators (dv + 2d columns), then two
    // unit slots of 128 columns.  Slot h takes the units of query rows
    // [64 h, 64 h + 64) of each staged tile.  Its region A (64 columns) holds
    // S1^T, then dP^T, then the bf16 dS1^T and dS2^T; its region B (64
    // columns) holds S2^T, then the bf16 (A1 - lambda A2)^T.  In bf16 each
    // 16-query chunk packs inside the columns its own fp32 values came from:
    // dS1^T then dS2^T (8 columns each) in region A, (A1 - lambda A2)^T in the
    // first 8 of the chunk's columns of region B.
    static constexpr uint32_t TM_DV = 0, TM_DK1 = DV, TM_DK2 = DV + D, TM_SLOTS = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int W_GRAD = 2 + NDS;           // the warp that issues the gradient products
    static constexpr int THREADS = 96 + 32 * NDS;   // producer, score/dP issuer, dS warps, gradient issuer
    // Q/K rows are one swizzle span wide (128 or 64 bytes); dO and V come in
    // 64-column boxes of 128-byte rows.
    static constexpr uint32_t QK_ROW = D * 2;
    static constexpr uint32_t QK_SWZ = QK_ROW == 128 ? SWZ_128B : SWZ_64B;
    static constexpr uint32_t QK_SBO = 8 * QK_ROW;
    static_assert((D == 64 && DV == 128) || (D == 32 && DV == 64), "backward widths");
    static_assert(STAGE % 1024 == 0, "stage layout");
    static_assert(DV + 2 * D <= TM_SLOTS, "accumulators below the unit slots");
    static_assert((BU * QK_ROW) % 1024 == 0 && (BU * 128) % 1024 == 0, "unit offsets keep the swizzle atoms");
    static_assert(SMEM_BYTES <= 227u * 1024u && SMEM_BYTES > 114u * 1024u, "one CTA per SM");
};

// One CTA owns 128 keys and walks the 128-query tiles that see them, half a
// tile (a 64-query unit) at a time, with two unit slots in tensor memory so
// that one unit's products run while the dS warps work on the other.
//   * Per unit the tensor core computes S1^T = K1 Q1^T and S2^T = K2 Q2^T
//     (M = 128 keys, N = 64 queries).
//   * The dS warps (two per TMEM lane quarter, 32 queries each) take both
//     into registers and release the slot; dP^T = V dO^T then goes over
//     S1^T while the dS warps form A1^T and A2^T.
//   * From dP^T, in 16-query chunks, they form dS1^T, dS2^T and
//     (A1 - lambda A2)^T in bf16; the gradient products
//     dV += (A1 - lambda A2)^T dO and dK_r += dS_r^T Q_r of chunk c run while
//     chunk c + 1 is computed.
//   * Two warps issue: one the score and dP^T products, one the gradient
//     products, so that dP^T of unit u + 1 goes in as soon as the dS warps
//     hold its scores, whatever gradient products are still queued.  The
//     scores of unit u + 2 go into unit u's slot once a barrier committed
//     behind unit u's gradient products reports them complete.

template <int D, int DV, bool CAUSAL>
__global__ void __launch_bounds__(BwdDkvLayout<D, DV>::THREADS, 1)
bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_q2,
               const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k1,
               const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v,
               const BwdParams p) {
    using L = BwdDkvLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kt = blockIdx.x;   // key tile 0 sees the most queries under causal masking: first
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * p.H + h;
    const int k0 = kt * L::BK;
    const int diag = p.Nk - p.Nq;
    // Query tiles that see at least one of this CTA's keys: key j is seen by
    // query i iff j <= i + diag.  Unit u is half u % 2 of tile u / 2.
    const int t0 = CAUSAL ? max(0, k0 - diag) / L::BQ : 0;
    const int n_t = (p.Nq + L::BQ - 1) / L::BQ - t0;
    const int n_u = 2 * n_t;

    auto bar = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_KV), 1);
        for (int s = 0; s < L::QST; ++s) {
            mbar_init(bar(L::B_QFULL + s), 1);
            mbar_init(bar(L::B_QEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::B_SFULL + s), 1);
            mbar_init(bar(L::B_SFREE + s), L::NDS);
            mbar_init(bar(L::B_DPFULL + s), 1);
        }
        for (int c = 0; c < 2 * L::NCH; ++c) mbar_init(bar(L::B_PFULL + c), L::NDS);
        for (int s = 0; s < 2; ++s) mbar_init(bar(L::B_GDONE + s), 1);
        mbar_init(bar(L::B_DONE), 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q1);
        prefetch_tensormap(&tm_q2);
        prefetch_tensormap(&tm_do);
        prefetch_tensormap(&tm_k1);
        prefetch_tensormap(&tm_k2);
        prefetch_tensormap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(sb + L::OFF_TMEM_SLOT, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM_SLOT);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(bar(L::B_KV), 2 * L::K_BYTES + L::V_BYTES);
            tma_load_4d(sb + L::OFF_K1, &tm_k1, bar(L::B_KV), 0, k0, h, b);
            tma_load_4d(sb + L::OFF_K2, &tm_k2, bar(L::B_KV), 0, k0, h, b);
#pragma unroll
            for (int c = 0; c < DV / 64; ++c)
                tma_load_4d(sb + L::OFF_V + (uint32_t)c * L::V_BOX, &tm_v, bar(L::B_KV), c * 64, k0, h, b);
            int issued = 0;
            for (int t = 0; t < n_t && ok; ++t) {
                const int qs = t % L::QST;
                ok = mbar_wait(bar(L::B_QEMPTY + qs), ((t / L::QST) & 1) ^ 1, ERR_SITE_BWD_PRODUCER);
                if (!ok) break;
                const int i0 = (t0 + t) * L::BQ;
                const uint32_t st = sb + L::OFF_Q + (uint32_t)qs * L::STAGE;
                mbar_arrive_expect_tx(bar(L::B_QFULL + qs), 2 * L::Q_BYTES + L::DO_BYTES + L::RC_BYTES);
                tma_load_4d(st, &tm_q1, bar(L::B_QFULL + qs), 0, i0, h, b);
                tma_load_4d(st + L::ST_Q2, &tm_q2, bar(L::B_QFULL + qs), 0, i0, h, b);
#pragma unroll
                for (int c = 0; c < DV / 64; ++c)
                    tma_load_4d(st + L::ST_DO + (uint32_t)c * L::DO_BOX, &tm_do, bar(L::B_QFULL + qs), c * 64, i0, h,
                                b);
                bulk_load(st + L::ST_RC, p.rowt + (bh * p.Nq_pad + i0) * 4, L::RC_BYTES, bar(L::B_QFULL + qs));
                ++issued;
            }
            mbar_wait(bar(L::B_KV), 0, ERR_SITE_BWD_DRAIN);
            for (int s = 0; s < L::QST && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / L::QST) * L::QST;
                mbar_wait(bar(L::B_QFULL + s), (last / L::QST) & 1, ERR_SITE_BWD_DRAIN);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == L::W_GRAD) {
        // ------------------------------------------------------------ MMA issuers
        // Each issuing warp runs its loop with warp-uniform values; each MMA
        // and commit is issued by one elected lane (the *_warp wrappers).
        // Every lane waits; a wait that ran out on any lane ends the loop on all.
        auto wait = [&](uint32_t b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, ERR_SITE_BWD_MMA));
        };
        constexpr uint64_t STAGE16 = L::STAGE >> 4, Q2OFF = L::ST_Q2 >> 4;
        auto slot_a = [&](int hu) -> uint32_t { return tmem + L::TM_SLOTS + 128u * (uint32_t)hu; };
        if (warp == 1) {
            // Scores and dP^T.
            constexpr uint32_t idesc_s = idesc_bf16_f32(L::BK, L::BU, false);   // S^T, dP^T of one unit
            bool ok = wait(bar(L::B_KV), 0);
            tc_fence_after();
            const uint64_t dk1 = smem_desc(sb + L::OFF_K1, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t dk2 = smem_desc(sb + L::OFF_K2, 16, L::QK_SBO, L::QK_SWZ);
            const uint64_t dvv = smem_desc(sb + L::OFF_V, 16, 1024, SWZ_128B);
            const uint64_t dq0 = smem_desc(sb + L::OFF_Q, 16, L::QK_SBO, L::QK_SWZ);           // Q1 (K-major), stage 0
            const uint64_t ddo0 = smem_desc(sb + L::OFF_Q + L::ST_DO, 16, 1024, SWZ_128B);   // dO (K-major)
            constexpr uint64_t QU16 = (L::BU * L::QK_ROW) >> 4, DOU16 = (L::BU * 128) >> 4;   // unit row offsets
            // S1^T into region A and S2^T into region B of the unit's slot,
            // once the gradient products of the unit that used it before are
            // complete.
            auto issue_scores = [&](int u) -> bool {
                const int t = u >> 1, hu = u & 1;
                if (u >= 2 && !wait(bar(L::B_GDONE + hu), (t - 1) & 1)) return false;
                if (!wait(bar(L::B_QFULL + t % L::QST), (t / L::QST) & 1)) return false;
                tc_fence_after();
                const uint64_t q = dq0 + (uint64_t)(t % L::QST) * STAGE16 + (uint64_t)hu * QU16;
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_warp(slot_a(hu), dk1 + (uint64_t)(2 * k), q + (uint64_t)(2 * k), idesc_s, k > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    mma_ss_warp(slot_a(hu) + 64u, dk2 + (uint64_t)(2 * k), q + Q2OFF + (uint64_t)(2 * k), idesc_s,
                                k > 0 ? 1u : 0u);
                mma_commit_warp(bar(L::B_SFULL + hu));
                return true;
            };
            // dP^T = V dO^T over S1^T once the dS warps hold the slot's
            // scores: k over dv, two 64-column boxes of each operand.
            auto issue_dp = [&](int u) -> bool {
                const int t = u >> 1, hu = u & 1;
                if (!wait(bar(L::B_SFREE + hu), t & 1)) return false;
                tc_fence_after();
                const uint64_t o = ddo0 + (uint64_t)(t % L::QST) * STAGE16 + (uint64_t)hu * DOU16;
#pragma unroll
                for (int k = 0; k < DV / 16; ++k)
                    mma_ss_warp(slot_a(hu), dvv + (uint64_t)(((k >> 2) * L::V_BOX + (k & 3) * 32) >> 4),
                                o + (uint64_t)(((k >> 2) * L::DO_BOX + (k & 3) * 32) >> 4), idesc_s, k > 0 ? 1u : 0u);
                mma_commit_warp(bar(L::B_DPFULL + hu));
                return true;
            };
            if (ok && n_u > 0) ok = issue_scores(0) && issue_scores(1) && issue_dp(0);
            for (int u = 0; u < n_u && ok; ++u) {
                if (u + 1 < n_u) ok = issue_dp(u + 1);
                if (ok && u + 2 < n_u) ok = issue_scores(u + 2);
            }
        } else {
            // Gradient products, chunk by chunk: chunk c of group g is the
            // unit's queries [GC g + CW c, GC g + CW c + CW), CW / 16 k-steps
            // (k-step kq: queries [16 kq, 16 kq + 16) of the staged tile).
            constexpr uint32_t idesc_dv = idesc_bf16_f32(L::BK, DV, true);   // dV: dO MN-major
            constexpr uint32_t idesc_dk = idesc_bf16_f32(L::BK, D, true);    // dK: Q MN-major
            const uint64_t dqm0 = smem_desc(sb + L::OFF_Q, L::Q_BYTES, L::QK_SBO, L::QK_SWZ);     // Q1 as MN-major B
            const uint64_t ddom0 = smem_desc(sb + L::OFF_Q + L::ST_DO, L::DO_BOX, 1024, SWZ_128B);   // dO MN-major
            bool ok = true;
            for (int u = 0; u < n_u && ok; ++u) {
                const int t = u >> 1, hu = u & 1, qs = t % L::QST;
                const uint64_t st = (uint64_t)qs * STAGE16;
                // This warp reads the staged Q and dO: observe their copies.
                ok = wait(bar(L::B_QFULL + qs), (t / L::QST) & 1);
#pragma unroll
                for (int c = 0; c < L::NCH && ok; ++c) {
                    ok = wait(bar(L::B_PFULL + hu * L::NCH + c), t & 1);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int g = 0; g < L::NG; ++g) {
#pragma unroll
                        for (int sub = 0; sub < L::CW / 16; ++sub) {
                            const int kq = (L::BU * hu + L::GC * g + L::CW * c) / 16 + sub;
                            const uint64_t kd = (uint64_t)(kq * (16 * 128 >> 4)),
                                           kqq = (uint64_t)(kq * (16 * L::QK_ROW >> 4));
                            const uint32_t acc = (t > 0 || kq > 0) ? 1u : 0u;
                            // bf16 operands of k-step sub: 8 columns at 8 sub
                            // of the chunk's [dS1 | dS2] (CW / 2 columns each)
                            // and of its (A1 - lambda A2) columns.
                            const uint32_t col = (uint32_t)(L::GC * g + L::CW * c) + 8u * sub;
                            mma_ts_warp(tmem + L::TM_DV, slot_a(hu) + 64u + col, ddom0 + st + kd, idesc_dv, acc);
                            mma_ts_warp(tmem + L::TM_DK1, slot_a(hu) + col, dqm0 + st + kqq, idesc_dk, acc);
                            mma_ts_warp(tmem + L::TM_DK2, slot_a(hu) + col + L::CW / 2, dqm0 + st + Q2OFF + kqq,
                                        idesc_dk, acc);
                        }
                    }
                }
                if (!ok) break;
                mma_commit_warp(bar(L::B_GDONE + hu));
                // Both units of the staged tile are done with it once these
                // products complete (the score and dP^T products that read it
                // completed before the dS warps released these chunks).
                if (hu == 1) mma_commit_warp(bar(L::B_QEMPTY + qs));
            }
            mma_commit_warp(bar(L::B_DONE));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ dS (warps 2 .. 2 + NDS - 1)
        constexpr int GC = L::GC, CW = L::CW;
        const int grp = (warp - 2) >> 2;        // column group: the unit's query columns [GC grp, GC grp + GC)
        const int wq = warp & 3;                // TMEM lane quarter
        const int row = wq * 32 + lane;         // key row within the tile
        const uint32_t t_lane = (uint32_t)(wq * 32) << 16;
        const int kj = k0 + row;
        const float sl2 = p.scale_log2;
        const float nlam = -p.lambda;
        bool ok = true;
        for (int u = 0; u < n_u; ++u) {
            const int t = u >> 1, hu = u & 1, qs = t % L::QST;
            const uint32_t ta = tmem + t_lane + L::TM_SLOTS + 128u * (uint32_t)hu + (uint32_t)(GC * grp);
            const uint32_t tb = ta + 64u;
            ok = mbar_wait(bar(L::B_SFULL + hu), t & 1, ERR_SITE_BWD_SOFTMAX);
            // The row constants came in with this stage's copies: observe that
            // barrier too (its phase cannot move on before this tile's PFULL
            // arrivals).
            ok = ok && mbar_wait(bar(L::B_QFULL + qs), (t / L::QST) & 1, ERR_SITE_BWD_SOFTMAX);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // Row constants of this group's GC queries, negated: -lse1 log2 e,
            // -lse2 log2 e, -D1, -D2 at rows 0, 128, 256, 384.
            const float* rct = reinterpret_cast<const float*>(smem + L::OFF_Q + (uint32_t)qs * L::STAGE + L::ST_RC) +
                               L::BU * hu + GC * grp;
            const int qbase = (t0 + t) * L::BQ + L::BU * hu + GC * grp;   // query of column 0
            // Causal: key kj is hidden from query qbase + i iff i < lim.  The
            // test runs only in warps that hold a hidden pair (warp-uniform).
            const int lim = kj - qbase - diag;
            const bool wmask = CAUSAL && (k0 + 32 * wq + 31 - qbase - diag > 0);
            float p1[GC], p2[GC];
            {
                uint32_t s1[GC], s2[GC];
                tmem_ld32x2(ta, s1, tb, s2);
                // Both score blocks are in registers: the slot may take dP^T.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::B_SFREE + hu));
#pragma unroll
                for (int j = 0; j < GC; j += 4) {
                    const float4 l1 = *reinterpret_cast<const float4*>(rct + j);
                    const float4 l2 = *reinterpret_cast<const float4*>(rct + 128 + j);
                    float x0, x1, x2, x3;
                    fma2(x0, x1, __uint_as_float(s1[j]), __uint_as_float(s1[j + 1]), sl2, sl2, l1.x, l1.y);
                    fma2(x2, x3, __uint_as_float(s1[j + 2]), __uint_as_float(s1[j + 3]), sl2, sl2, l1.z, l1.w);
                    p1[j] = fast_exp2(x0);
                    p1[j + 1] = fast_exp2(x1);
                    p1[j + 2] = fast_exp2(x2);
                    p1[j + 3] = fast_exp2(x3);
                    fma2(x0, x1, __uint_as_float(s2[j]), __uint_as_float(s2[j + 1]), sl2, sl2, l2.x, l2.y);
                    fma2(x2, x3, __uint_as_float(s2[j + 2]), __uint_as_float(s2[j + 3]), sl2, sl2, l2.z, l2.w);
                    p2[j] = fast_exp2(x0);
                    p2[j + 1] = fast_exp2(x1);
                    p2[j + 2] = fast_exp2(x2);
                    p2[j + 3] = fast_exp2(x3);
                }
                if (wmask) {
#pragma unroll
                    for (int j = 0; j < GC; ++j) {
                        p1[j] = j < lim ? 0.0f : p1[j];
                        p2[j] = j < lim ? 0.0f : p2[j];
                    }
                }
            }
            ok = mbar_wait(bar(L::B_DPFULL + hu), t & 1, ERR_SITE_BWD_SOFTMAX);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            // NCH chunks of CW queries; the gradient products of chunk c start
            // while chunk c + 1 is computed.
#pragma unroll
            for (int c = 0; c < L::NCH; ++c) {
                uint32_t dp[CW];
                tmem_ld16(ta + CW * c, dp);
                uint32_t w1[CW / 2], w2[CW / 2], wd[CW / 2];
#pragma unroll
                for (int j = 0; j < CW; j += 4) {
                    const float4 n1 = *reinterpret_cast<const float4*>(rct + 256 + CW * c + j);
                    const float4 n2 = *reinterpret_cast<const float4*>(rct + 384 + CW * c + j);
#pragma unroll
                    for (int h2 = 0; h2 < 4; h2 += 2) {
                        const int q = CW * c + j + h2;   // column within the group
                        const float d0 = __uint_as_float(dp[j + h2]), d1 = __uint_as_float(dp[j + h2 + 1]);
                        float u0, u1, v0, v1, g0, g1, a0, a1, b0, b1, c0, c1;
                        add2(u0, u1, d0, d1, h2 ? n1.z : n1.x, h2 ? n1.w : n1.y);   // dP - D1
                        add2(v0, v1, d0, d1, h2 ? n2.z : n2.x, h2 ? n2.w : n2.y);   // dP - D2
                        mul2(g0, g1, p2[q], p2[q + 1], nlam, nlam);                // -lambda A2
                        mul2(a0, a1, p1[q], p1[q + 1], u0, u1);                    // dS1
                        mul2(b0, b1, g0, g1, v0, v1);                              // dS2
                        add2(c0, c1, p1[q], p1[q + 1], g0, g1);                    // A1 - lambda A2
                        w1[(j + h2) >> 1] = pack_bf16x2(a0, a1);
                        w2[(j + h2) >> 1] = pack_bf16x2(b0, b1);
                        wd[(j + h2) >> 1] = pack_bf16x2(c0, c1);
                    }
                }
                tmem_st8(ta + CW * c, w1);
                tmem_st8(ta + CW * c + CW / 2, w2);
                tmem_st8(tb + CW * c, wd);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::B_PFULL + hu * L::NCH + c));
            }
        }
        // ------------------------------------------------------------ epilogue
        mbar_wait(bar(L::B_DONE), 0, ERR_SITE_BWD_EPILOGUE);
        __syncwarp();
        tc_fence_after();
        const bool store = kj < p.Nk;
        // dV: columns [dv/2 grp, dv/2 (grp + 1)); dK1, dK2: columns
        // [d/2 grp, d/2 (grp + 1)), times 1/sqrt(d).
        constexpr int VC = DV / L::NG, KC = D / L::NG;
#pragma unroll
        for (int c = 0; c < VC; c += 32)
            tmem_cols_to_bf16<32>(tmem + t_lane + L::TM_DV + (uint32_t)(VC * grp + c),
                                  p.dv + (bh * p.Nk + kj) * DV + VC * grp + c, 1.0f, store);
#pragma unroll
        for (int r = 0; r < 2; ++r)
            tmem_cols_to_bf16<KC>(tmem + t_lane + (r ? L::TM_DK2 : L::TM_DK1) + (uint32_t)(KC * grp),
                                  (r ? p.dk2 : p.dk1) + (bh * p.Nk + kj) * D + KC * grp, p.scale, store);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

}  // namespace diffattn
