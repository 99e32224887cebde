// Split-KV differential-attention decode for sm_103a: one query per (b, h)
// against a cache of Nk keys, no mask.  HBM-bound: every K1, K2 and V byte is
// read exactly once.
//
// Pass 1 (decode_split_kernel), grid (splits, H, B): a CTA owns one key range
// of one (b, h).  A producer warp streams 32-key chunks of K1 and K2 (tiled
// TMA, 128/64-byte swizzle so that lane-per-key reads are conflict-free) and
// of V (bulk copy) into a 12-16 stage shared-memory ring.  Six (d = 64) or
// eight (d = 32) consumer warps take chunks round-robin, each always from the
// same stages of the ring; in a warp, lane t scores key t against q1
// and q2, the warp keeps one online-softmax state per map (max m_r, per-lane
// partial normaliser l_r, unnormalised output O_r spread over the lanes by dv
// column) and accumulates O_r += p_r[j] v_j with the probabilities broadcast
// by shuffle.  The warps' states are merged in shared memory and one partial
// (m_r, l_r, O_r) per map is written to the workspace.
//
// Pass 2 (decode_merge_kernel), one warp per (b, h): merges the split
// partials with warp shuffles — M = max m_s, L = sum l_s 2^(m_s - M),
// O = sum O_s 2^(m_s - M) — the same associative rescaling the online
// softmax uses, then o = O1/L1 - lambda O2/L2, GroupNorm over dv, gain and
// (1 - lambda_init), bf16 store.  (Differential Transformer pages: the
// DiffAttn formula of the iloveeagents.com Q&A, "Mathematical Formula";
// steps 2-4 of llmbytes.dev "How Differential Attention Cancels Common-Mode
// Noise".)
#pragma once

#include "launch.h"
#include "sm103_ptx.cuh"

namespace diffattn {

struct DecodeParams {
    const uint16_t* q1;
    const uint16_t* q2;
    const uint16_t* v;
    int B, H, Nk, S;
    int keys_per_split;   // multiple of 32
    float scale_log2;     // log2(e) / sqrt(d)
    float* ws;            // [B*H*S][2][DV + 4] partials: m, l, pad, pad, O[DV]
    // Paged caches only: page p holds page_size consecutive keys of every
    // head (K rows (p*H + h)*page_size + i of the [num_pages*H*page_size, d]
    // view; V likewise); sequence b's pages are block_table[b*max_pages + .]
    // and its length is seq_lens[b].
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, page_size, num_pages;
};

struct MergeParams {
    int B, H, S;
    int parts;            // partial sets gathered from separate key ranges (1 on one GPU)
    float lambda, lambda_init, eps;
    const float* ws;
    const float* gamma;   // [H*DV] or null
    uint16_t* out;        // bf16 [B*H, DV]
    float* o_prenorm;     // fp32 [B*H, DV] or null
};

template <int D, int DV>
struct DecodeLayout {
    static constexpr int KC = 32;                       // keys per chunk (one per lane)
    // Chunk c goes to stage c % NST and to consumer warp c % NCW.  NST is a
    // multiple of NCW, so every stage is always consumed by the same warp,
    // which takes that stage's phases in order.  (If another warp could own
    // the next phase of a stage, it might wait on that stage's full barrier
    // while the earlier phase is still incomplete; a parity wait cannot tell
    // the two apart and would return at once.)
    static constexpr int NCW = (D == 64) ? 6 : 8;       // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;      // + producer warp
    static constexpr uint32_t K_BYTES = KC * D * 2;
    static constexpr uint32_t V_BYTES = KC * DV * 2;
    static constexpr uint32_t STAGE = 2 * K_BYTES + V_BYTES;
    static constexpr int NST = (D == 64) ? 12 : 16;
    static_assert(NST % NCW == 0, "each stage must belong to one consumer warp");
    static constexpr uint32_t OFF_RING = 0;
    static constexpr int PART = DV + 4;                 // floats per (map) partial
    static constexpr uint32_t OFF_RED = NST * STAGE;    // NCW x 2 x PART floats
    static constexpr uint32_t OFF_BAR = OFF_RED + NCW * 2 * PART * 4;
    static constexpr uint32_t OFF_PAGES = OFF_BAR + 2 * NST * 8;   // paged caches: the split's page indices
    static constexpr int MAX_SPLIT_PAGES = kDecodeMaxSplitPages;
    static constexpr uint32_t USED = OFF_PAGES + MAX_SPLIT_PAGES * 4;
    static constexpr uint32_t SMEM_BYTES = USED + 1024;
    static constexpr uint32_t SWZ_BYTES = (D == 64) ? 128 : 64;   // K row = swizzle span
    static_assert(USED + 1024 <= 227u * 1024u, "shared memory");
    static_assert(STAGE % 1024 == 0, "stage alignment");
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Dot product of a bf16 key row held in swizzled shared memory with q (fp32
// registers).  Row r of the tile starts at r*2D bytes; the 16-byte chunk c of
// the row sits at chunk position c ^ ((row byte offset >> 7) & (span/16 - 1)).
template <int D>
__device__ __forceinline__ float dot_row_swizzled(const uint8_t* tile, int r, const float (&q)[D]) {
    constexpr int RB = D * 2;
    constexpr int MASK = (D == 64) ? 7 : 3;
    const int sw = ((r * RB) >> 7) & MASK;
    const uint8_t* row = tile + r * RB;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const uint4 kk = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
        acc0 = fmaf(q[8 * c + 0], bf16lo_to_f32(kk.x), acc0);
        acc1 = fmaf(q[8 * c + 1], bf16hi_to_f32(kk.x), acc1);
        acc0 = fmaf(q[8 * c + 2], bf16lo_to_f32(kk.y), acc0);
        acc1 = fmaf(q[8 * c + 3], bf16hi_to_f32(kk.y), acc1);
        acc0 = fmaf(q[8 * c + 4], bf16lo_to_f32(kk.z), acc0);
        acc1 = fmaf(q[8 * c + 5], bf16hi_to_f32(kk.z), acc1);
        acc0 = fmaf(q[8 * c + 6], bf16lo_to_f32(kk.w), acc0);
        acc1 = fmaf(q[8 * c + 7], bf16hi_to_f32(kk.w), acc1);
    }
    return acc0 + acc1;
}

// PAGED = false: contiguous caches [B, H, Nk, width].  PAGED = true: paged
// caches with per-sequence lengths (see DecodeParams); a 32-key chunk never
// straddles a page because page_size is a multiple of 32.
template <int D, int DV, bool PAGED>
__global__ void __launch_bounds__(DecodeLayout<D, DV>::THREADS, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
                    const DecodeParams p) {
    using L = DecodeLayout<D, DV>;
    constexpr int CPL = DV / 32;   // dv columns per lane
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * p.H + h;
    // Launched as a dependent grid: the inputs, and the partials buffer that
    // the previous call's merge may still be reading, are touched only after
    // the previous grid on the stream has completed.
    grid_dependency_wait();
    grid_launch_dependents();
    int seq_len = p.Nk;
    if (PAGED) {
        // Lengths and pages come from device memory the host cannot check:
        // out-of-range values are clamped (and reported), never dereferenced.
        seq_len = p.seq_lens[b];
        const int cap = p.max_pages * p.page_size;
        if (seq_len < 1 || seq_len > cap) {
            if (threadIdx.x == 0) atomicCAS(&g_device_error, 0, ERR_DECODE_BAD_LENGTH);
            seq_len = min(max(seq_len, 1), cap);
        }
    }
    const int key_begin = s * p.keys_per_split;
    const int key_end = min(seq_len, key_begin + p.keys_per_split);
    const int nkeys = max(0, key_end - key_begin);
    const int nchunks = (nkeys + L::KC - 1) / L::KC;
    const int first_page = PAGED ? key_begin / p.page_size : 0;

    auto full = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8u * (uint32_t)i; };
    auto empty = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8u * (uint32_t)(L::NST + i); };

    if (PAGED && nkeys > 0) {
        int* pages = reinterpret_cast<int*>(smem + L::OFF_PAGES);
        const int npages = (key_end - 1) / p.page_size - first_page + 1;   // <= MAX_SPLIT_PAGES (host check)
        for (int i = threadIdx.x; i < npages; i += blockDim.x) {
            int pg = p.block_table[(size_t)b * p.max_pages + first_page + i];
            if (pg < 0 || pg >= p.num_pages) {
                atomicCAS(&g_device_error, 0, ERR_DECODE_BAD_PAGE);
                pg = 0;
            }
            pages[i] = pg;
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NST; ++i) {
            mbar_init(full(i), 1);
            mbar_init(empty(i), 1);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_k1);
        prefetch_tensormap(&tm_k2);
    }
    __syncthreads();

    float* red = reinterpret_cast<float*>(smem + L::OFF_RED);

    if (warp == L::NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const int* pages = reinterpret_cast<const int*>(smem + L::OFF_PAGES);
            // Paged caches: the chunk's page (index into the staged list) and
            // its key offset in that page, advanced chunk by chunk (key_begin
            // and page_size are multiples of the 32-key chunk).
            int pi = 0, off = PAGED ? key_begin - first_page * p.page_size : 0;
            size_t page_row = 0;   // first K row of the current page for this head
            if (PAGED && nchunks > 0) page_row = ((size_t)pages[0] * p.H + h) * p.page_size;
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int st = c % L::NST;
                if (!mbar_wait(empty(st), ((c / L::NST) & 1) ^ 1, ERR_SITE_DECODE_PRODUCER)) break;
                const int k0 = key_begin + c * L::KC;
                const int rows = min(L::KC, key_end - k0);
                // Row of this chunk's first key in the [rows, D] view of the K
                // caches (the V cache has the same row order).
                size_t krow;
                if (PAGED) {
                    krow = page_row + off;
                    off += L::KC;
                    if (off == p.page_size && c + 1 < nchunks) {
                        off = 0;
                        page_row = ((size_t)pages[++pi] * p.H + h) * p.page_size;
                    }
                } else {
                    krow = bh * (size_t)p.Nk + k0;
                }
                const uint32_t base = sb + L::OFF_RING + (uint32_t)st * L::STAGE;
                mbar_arrive_expect_tx(full(st), 2 * L::K_BYTES + (uint32_t)rows * DV * 2);
                tma_load_4d(base, &tm_k1, full(st), 0, (int)krow, 0, 0);
                tma_load_4d(base + L::K_BYTES, &tm_k2, full(st), 0, (int)krow, 0, 0);
                bulk_load(base + 2 * L::K_BYTES, p.v + krow * DV, (uint32_t)rows * DV * 2, full(st));
                ++issued;
            }
            for (int st = 0; st < L::NST && st < issued; ++st) {
                const int last = st + ((issued - 1 - st) / L::NST) * L::NST;
                mbar_wait(full(st), (last / L::NST) & 1, ERR_SITE_DECODE_DRAIN);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        float q1[D], q2[D];
#pragma unroll
        for (int i = 0; i < D; ++i) {
            q1[i] = __uint_as_float((uint32_t)p.q1[bh * D + i] << 16);
            q2[i] = __uint_as_float((uint32_t)p.q2[bh * D + i] << 16);
        }
        float m1 = -INFINITY, m2 = -INFINITY, l1 = 0.f, l2 = 0.f;
        float o1[CPL], o2[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) o1[i] = o2[i] = 0.f;
        const float sl2 = p.scale_log2;
        for (int c = warp; c < nchunks; c += L::NCW) {
            const int st = c % L::NST;
            bool ok = mbar_wait(full(st), (c / L::NST) & 1, ERR_SITE_DECODE_CONSUMER);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint8_t* base = smem + L::OFF_RING + (size_t)st * L::STAGE;
            const int rows = min(L::KC, key_end - (key_begin + c * L::KC));
            const bool valid = lane < rows;
            float s1 = dot_row_swizzled<D>(base, lane, q1) * sl2;
            float s2 = dot_row_swizzled<D>(base + L::K_BYTES, lane, q2) * sl2;
            if (!valid) s1 = s2 = -INFINITY;
            const float n1 = fmaxf(m1, warp_max(s1));
            const float n2 = fmaxf(m2, warp_max(s2));
            const float a1 = fast_exp2(m1 - n1), a2 = fast_exp2(m2 - n2);   // m = -inf -> 0
            const float p1 = fast_exp2(s1 - n1), p2 = fast_exp2(s2 - n2);
            m1 = n1;
            m2 = n2;
            l1 = l1 * a1 + p1;
            l2 = l2 * a2 + p2;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                o1[i] *= a1;
                o2[i] *= a2;
            }
            const uint8_t* vt = base + 2 * L::K_BYTES;
            for (int j = 0; j < rows; ++j) {
                const float pj1 = __shfl_sync(0xffffffffu, p1, j);
                const float pj2 = __shfl_sync(0xffffffffu, p2, j);
                const uint8_t* vr = vt + (size_t)j * DV * 2 + lane * CPL * 2;
                float vv[CPL];
                if constexpr (CPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vr);
                    vv[0] = bf16lo_to_f32(w.x); vv[1] = bf16hi_to_f32(w.x);
                    vv[2] = bf16lo_to_f32(w.y); vv[3] = bf16hi_to_f32(w.y);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(vr);
                    vv[0] = bf16lo_to_f32(w); vv[1] = bf16hi_to_f32(w);
                }
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    o1[i] = fmaf(pj1, vv[i], o1[i]);
                    o2[i] = fmaf(pj2, vv[i], o2[i]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(st));
        }
        // Per-warp state -> shared memory.
        l1 = warp_sum(l1);
        l2 = warp_sum(l2);
        float* w1 = red + (warp * 2 + 0) * L::PART;
        float* w2 = red + (warp * 2 + 1) * L::PART;
        if (lane == 0) {
            w1[0] = m1; w1[1] = l1;
            w2[0] = m2; w2[1] = l2;
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            w1[4 + lane * CPL + i] = o1[i];
            w2[4 + lane * CPL + i] = o2[i];
        }
        named_barrier_sync(1, L::NCW * 32);
        // Merge the warps: thread t -> (map t / DV, column t % DV).
        for (int t = threadIdx.x; t < 2 * DV; t += L::NCW * 32) {
            const int r = t / DV, col = t % DV;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < L::NCW; ++w) M = fmaxf(M, red[(w * 2 + r) * L::PART]);
            float Ls = 0.f, Os = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < L::NCW; ++w) {
                    const float* src = red + (w * 2 + r) * L::PART;
                    const float e = fast_exp2(src[0] - M);
                    Ls = fmaf(src[1], e, Ls);
                    Os = fmaf(src[4 + col], e, Os);
                }
            }
            float* dst = p.ws + ((bh * p.S + s) * 2 + r) * L::PART;
            dst[4 + col] = Os;
            if (col == 0) {
                dst[0] = M;
                dst[1] = Ls;
            }
        }
    }
}

template <int DV>
__global__ void __launch_bounds__(128)
decode_merge_kernel(const MergeParams p) {
    constexpr int PART = DV + 4;
    constexpr int CPL = DV / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = (size_t)blockIdx.x * 4 + warp;
    // Launched as a dependent grid of the split kernel: its partials are read
    // only once that grid has completed.
    grid_dependency_wait();
    grid_launch_dependents();
    if (bh >= (size_t)p.B * p.H) return;
    const int h = (int)(bh % p.H);
    // Partial t = (part, split) of this head: parts are [parts][B*H][S] blocks.
    const size_t BH = (size_t)p.B * p.H;
    const int T = p.parts * p.S;
    auto part = [&](int t, int r) -> const float* {
        const int pt = t / p.S, s = t - pt * p.S;
        return p.ws + ((((size_t)pt * BH + bh) * p.S + s) * 2 + r) * PART;
    };
    float O[2][CPL], Lr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float M = -INFINITY;
        for (int t = lane; t < T; t += 32) M = fmaxf(M, part(t, r)[0]);
        M = warp_max(M);
        float Ls = 0.f;
        for (int t = lane; t < T; t += 32) {
            const float m = part(t, r)[0];
            if (m != -INFINITY) Ls = fmaf(part(t, r)[1], fast_exp2(m - M), Ls);
        }
        Lr[r] = warp_sum(Ls);
#pragma unroll
        for (int i = 0; i < CPL; ++i) O[r][i] = 0.f;
        for (int t = 0; t < T; ++t) {
            const float* src = part(t, r);
            const float m = src[0];
            if (m == -INFINITY) continue;
            const float e = fast_exp2(m - M);
#pragma unroll
            for (int i = 0; i < CPL; ++i) O[r][i] = fmaf(src[4 + lane * CPL + i], e, O[r][i]);
        }
    }
    const float inv1 = 1.0f / Lr[0], inv2 = p.lambda / Lr[1];
    float o[CPL], sum = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        o[i] = __fmul_rn(O[0][i], inv1) - __fmul_rn(O[1][i], inv2);   // no contraction: exact cancel
        sum += o[i];
    }
    const float mu = warp_sum(sum) * (1.0f / DV);
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i) sq += (o[i] - mu) * (o[i] - mu);
    const float var = warp_sum(sq) * (1.0f / DV);
    const float sc = (1.0f - p.lambda_init) * rsqrtf(var + p.eps);
    const int col0 = lane * CPL;
    if (p.o_prenorm) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) p.o_prenorm[bh * DV + col0 + i] = o[i];
    }
    uint32_t packed[CPL / 2];
#pragma unroll
    for (int i = 0; i < CPL / 2; ++i) {
        const float g0 = p.gamma ? p.gamma[(size_t)h * DV + col0 + 2 * i] : 1.0f;
        const float g1 = p.gamma ? p.gamma[(size_t)h * DV + col0 + 2 * i + 1] : 1.0f;
        packed[i] = pack_bf16x2((o[2 * i] - mu) * sc * g0, (o[2 * i + 1] - mu) * sc * g1);
    }
    if constexpr (CPL == 4) {
        *reinterpret_cast<uint2*>(p.out + bh * DV + col0) = make_uint2(packed[0], packed[1]);
    } else {
        *reinterpret_cast<uint32_t*>(p.out + bh * DV + col0) = packed[0];
    }
}

// Merge with one CTA per (b, h) and one thread per output column, for heads
// with at most TMAX partial states: every load of the merge is issued at once
// (one round of memory latency instead of one per partial), the normaliser
// and the GroupNorm statistics are block reductions.  Same algebra as
// merge_head; the per-column output sum runs over the partials in the same
// order.
constexpr int kMergeWideMax = 16;

template <int DV>
__global__ void __launch_bounds__(DV)
decode_merge_wide_kernel(const MergeParams p) {
    constexpr int PART = DV + 4, TMAX = kMergeWideMax, NW = DV / 32;
    __shared__ float red[2][NW];
    const int c = threadIdx.x, lane = c & 31, warp = c >> 5;
    const size_t bh = blockIdx.x;
    grid_dependency_wait();
    grid_launch_dependents();
    const int h = (int)(bh % p.H);
    const size_t BH = (size_t)p.B * p.H;
    const int T = p.parts * p.S;   // <= TMAX (the launcher's choice)
    float m[2][TMAX], l[2][TMAX], o[2][TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
            const int pt = t / p.S, sp = t - pt * p.S;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float* src = p.ws + ((((size_t)pt * BH + bh) * p.S + sp) * 2 + r) * PART;
                m[r][t] = __ldcg(src);
                l[r][t] = __ldcg(src + 1);
                o[r][t] = __ldcg(src + 4 + c);
            }
        }
    }
    float O[2], L[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float M = -INFINITY;
#pragma unroll
        for (int t = 0; t < TMAX; ++t)
            if (t < T) M = fmaxf(M, m[r][t]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            if (t < T && m[r][t] != -INFINITY) {
                const float e = fast_exp2(m[r][t] - M);
                Ls = fmaf(l[r][t], e, Ls);
                Os = fmaf(o[r][t], e, Os);
            }
        }
        O[r] = Os;
        L[r] = Ls;
    }
    const float inv1 = 1.0f / L[0], inv2 = p.lambda / L[1];
    const float ov = __fmul_rn(O[0], inv1) - __fmul_rn(O[1], inv2);   // no contraction: exact cancel
    float x = warp_sum(ov);
    if (lane == 0) red[0][warp] = x;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += red[0][w];
    const float mu = tot * (1.0f / DV);
    x = warp_sum((ov - mu) * (ov - mu));
    if (lane == 0) red[1][warp] = x;
    __syncthreads();
    tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += red[1][w];
    const float var = tot * (1.0f / DV);
    const float sc = (1.0f - p.lambda_init) * rsqrtf(var + p.eps);
    if (p.o_prenorm) p.o_prenorm[bh * DV + c] = ov;
    const float g = p.gamma ? p.gamma[(size_t)h * DV + c] : 1.0f;
    const float y = (ov - mu) * sc * g;
    p.out[bh * DV + c] = (uint16_t)(pack_bf16x2(y, 0.0f) & 0xffffu);
}

}  // namespace diffattn
