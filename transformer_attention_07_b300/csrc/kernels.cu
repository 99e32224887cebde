// Device code of the library and the host launchers that configure it.
// Everything that runs on the GPU is in this translation unit, so the device
// error word is a single object per device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <utility>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace diffattn {

__device__ int g_device_error = 0;

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int site) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*reinterpret_cast<volatile int*>(&g_device_error) != 0) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicCAS(&g_device_error, 0, site);
                return false;
            }
        }
    }
}

}  // namespace diffattn

#include "backward_sm103a.cuh"
#include "decode_sm103a.cuh"
#include "prefill_sm103a.cuh"
#include "standard_attn_sm103a.cuh"

namespace diffattn {

// ----------------------------------------------------------------- diagnostics

bool cuda_ok(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    static const bool debug = std::getenv("DIFFATTN_DEBUG") != nullptr;
    if (debug) std::fprintf(stderr, "[diffattn] %s failed: %s (%d)\n", what, cudaGetErrorString(e), (int)e);
    return false;
}

// ----------------------------------------------------------------- tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 4-D map over a BHND tensor [B][H][N][W] of bf16 (or of bytes, esize 1):
// dims (W, N, H, B).
static bool make_map_bhnd(CUtensorMap* m, const void* base, int B, int H, int N, int W, int box_w, int box_n,
                          CUtensorMapSwizzle swz, int esize = 2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = (cuuint64_t)esize;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)W * e, (cuuint64_t)N * W * e, (cuuint64_t)H * N * W * e};
    const cuuint32_t box[4] = {(cuuint32_t)box_w, (cuuint32_t)box_n, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUresult r = fn(m, dt, 4, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && std::getenv("DIFFATTN_DEBUG"))
        std::fprintf(stderr, "[diffattn] cuTensorMapEncodeTiled failed: %d\n", (int)r);
    return r == CUDA_SUCCESS;
}

// Launches a decode kernel as a dependent grid (programmatic stream
// serialisation): it may be scheduled while the previous grid on the stream
// drains, and waits for that grid's completion inside the kernel before it
// touches memory.  The split and merge kernels of one call then follow each
// other without a full launch gap.
template <typename... Params, typename... Args>
static cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- prefill

// Streaming multiprocessors of the current device (0 if unknown), cached per
// device; safe to call from several host threads.
int sm_count() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMaxDevices) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Key lengths up to which the prefill runs as a persistent grid (one CTA per
// SM walking the query tiles).  With few key tiles per query tile, the
// per-tile setup and epilogue that the persistent form overlaps weigh more.
#ifndef DIFFATTN_PERSIST_MAX_NK
#define DIFFATTN_PERSIST_MAX_NK 4096
#endif
static constexpr int kPersistMaxNk = DIFFATTN_PERSIST_MAX_NK;

// The differential prefill also stays persistent up to this many keys when
// its tile list is weight-major (all heads' K and V in half the L2): at
// causal 8K, B1 H16 that gains 4-5%.  With a (b, h)-major list the one-tile
// grid's grouped order balances better (causal 8K, B2 H16: 1.7% slower
// persistent).
static constexpr int kPersistMaxNkWeightMajor = 8192;

// The persistent grids walk their tiles weight-major across all heads (the
// better balance) under causal masking when every head's K and V together
// take at most this many bytes, half the B300's 126 MB L2; larger problems
// walk (b, h)-major so that the tiles in flight share their heads' K and V.
static constexpr long long kWeightMajorMaxBytes = 64ll << 20;

static int weight_major_order(bool causal, int B, int H, int Nk, long long bytes_per_key) {
    return causal && (long long)B * H * Nk * bytes_per_key <= kWeightMajorMaxBytes ? 1 : 0;
}

// The one-tile grids under causal masking: heads per weight-ordered group,
// as many as fit kHeadGroupBytes of K and V, at most all; 0 (the (b, h)-major
// 3-D grid) when fewer than four heads fit.  The CTAs in flight then span a
// few heads more than in (b, h)-major order: groups of 64 MB cost 3% at 16K
// (B4 H16), groups of two 16K heads were 2% slower or even; four 8K heads
// (16 MB) gain 2.3% at causal 8K, B2 H16.
static constexpr long long kHeadGroupBytes = 16ll << 20;

// The 1-D tile orders (persistent list, grouped one-tile grid) compute tile
// indices in 32-bit arithmetic; larger problems take the 3-D grid.
static constexpr long long kMaxTiles1D = 1ll << 30;

// Multiplier and shift of div_inv for divisor d >= 1 (quotients exact for
// dividends below 2^31).
static void inv_div(unsigned d, unsigned& m, int& s) {
    if (d == 0) d = 1;   // empty problems: never used
    int l = 0;
    while ((1ull << l) < d) ++l;
    s = 31 + l;
    m = (unsigned)(((1ull << s) + d - 1) / d);
}

static int head_group_size(int B, int H, int Nk, long long bytes_per_key) {
    const long long per_head = (long long)Nk * bytes_per_key;
    long long g = per_head > 0 ? kHeadGroupBytes / per_head : 0;
    if (g > (long long)B * H) g = (long long)B * H;
    return g >= 4 ? (int)g : 0;
}

PrefillPlan prefill_plan(int B, int H, int Nq, int Nk, int d, int dv, bool causal, bool qk8, int sms) {
    constexpr int BM = 128;   // query rows per tile (PrefillLayout::BM)
    const long long bytes_per_key = 2ll * d * (qk8 ? 1 : 2) + 2ll * dv;
    const long long num_qt = (Nq + BM - 1) / BM;
    const long long tiles = num_qt * H * B;
    PrefillPlan pl;
    pl.weight_major = weight_major_order(causal, B, H, Nk, bytes_per_key);
    // Both 1-D orders index their tiles with 32-bit arithmetic.
    const bool small = tiles < kMaxTiles1D;
    const bool persist = sms > 0 && tiles > sms && small &&
                         (Nk <= kPersistMaxNk || (pl.weight_major && Nk <= kPersistMaxNkWeightMajor));
    pl.head_group = causal && !persist && small ? head_group_size(B, H, Nk, bytes_per_key) : 0;
    pl.form = persist ? (pl.weight_major ? 3 : 2) : pl.head_group > 0 ? 1 : 0;
    pl.ctas = persist ? sms : tiles;
    return pl;
}

template <int D, int DV, bool CAUSAL, bool QK8>
static int launch_prefill_t(const PrefillArgs& a, cudaStream_t st) {
    using L = PrefillLayout<D, DV, QK8>;
    CUtensorMap mq1, mq2, mk1, mk2, mv, mo;
    // Q/K rows are one swizzle span wide (128, 64 or 32 bytes).
    const CUtensorMapSwizzle qk_swz = L::QK_ROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                      : L::QK_ROW == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B;
    const int qe = (int)L::QK_ELEM;
    if (!make_map_bhnd(&mq1, a.q1, a.B, a.H, a.Nq, D, D, L::BM, qk_swz, qe) ||
        !make_map_bhnd(&mq2, a.q2, a.B, a.H, a.Nq, D, D, L::BM, qk_swz, qe) ||
        !make_map_bhnd(&mk1, a.k1, a.B, a.H, a.Nk, D, D, L::BN, qk_swz, qe) ||
        !make_map_bhnd(&mk2, a.k2, a.B, a.H, a.Nk, D, D, L::BN, qk_swz, qe) ||
        !make_map_bhnd(&mv, a.v, a.B, a.H, a.Nk, DV, 64, L::BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        // output boxes of the persistent form's TMA stores: 32 rows x 64 columns
        !make_map_bhnd(&mo, a.out, a.B, a.H, a.Nq, DV, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return LAUNCH_ERR_CUDA;
    PrefillParams p;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.lambda = a.lambda;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    p.gamma = a.gamma;
    p.out = static_cast<uint16_t*>(a.out);
    p.o_prenorm = a.o_prenorm;
    p.o2 = a.o2;
    p.lse = a.lse;
    p.qk_scale = a.qk_scale;
    const long long tiles = (long long)((a.Nq + L::BM - 1) / L::BM) * a.H * a.B;
    const int sms = sm_count();
    const PrefillPlan plan = prefill_plan(a.B, a.H, a.Nq, a.Nk, D, DV, CAUSAL, QK8, sms);
    p.weight_major = plan.weight_major;
    const bool persist = plan.form >= 2;
    inv_div(p.weight_major ? (unsigned)((long long)a.H * a.B) : (unsigned)((a.Nq + L::BM - 1) / L::BM), p.div_major_m,
            p.div_major_s);
    inv_div((unsigned)a.H, p.div_h_m, p.div_h_s);
    p.head_group = plan.head_group;
    auto kern = persist ? prefill_kernel<D, DV, CAUSAL, QK8, true> : prefill_kernel<D, DV, CAUSAL, QK8, false>;
    const int smem = (int)(persist ? PrefillLayout<D, DV, QK8, true>::SMEM_BYTES : L::SMEM_BYTES);
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                 "prefill: set shared memory"))
        return LAUNCH_ERR_CUDA;
    const dim3 grid = persist          ? dim3(sms, 1, 1)
                      : p.head_group ? dim3((unsigned)tiles, 1, 1)
                                     : dim3((a.Nq + L::BM - 1) / L::BM, a.H, a.B);
    return cuda_ok(launch_dependent(kern, grid, dim3(L::THREADS), (size_t)smem, st, mq1, mq2, mk1, mk2, mv, mo, p),
                   "prefill: launch")
               ? LAUNCH_OK
               : LAUNCH_ERR_CUDA;
}

template <bool QK8>
static int launch_prefill_q(const PrefillArgs& a, cudaStream_t st) {
    if (a.d == 64 && a.dv == 128)
        return a.causal ? launch_prefill_t<64, 128, true, QK8>(a, st) : launch_prefill_t<64, 128, false, QK8>(a, st);
    if (a.d == 32 && a.dv == 64)
        return a.causal ? launch_prefill_t<32, 64, true, QK8>(a, st) : launch_prefill_t<32, 64, false, QK8>(a, st);
    return LAUNCH_ERR_UNSUPPORTED;
}

int launch_prefill(const PrefillArgs& a, cudaStream_t st) {
    return a.qk_scale ? launch_prefill_q<true>(a, st) : launch_prefill_q<false>(a, st);
}

// ----------------------------------------------------------------- backward

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

BwdWorkspace bwd_workspace_layout(int B, int H, int Nq, int dv) {
    BwdWorkspace w;
    const size_t BH = (size_t)B * H;
    w.Nq_pad = (Nq + kBwdRowPad - 1) / kBwdRowPad * kBwdRowPad;
    w.nchunk = w.Nq_pad / kBwdPrepRows;
    w.off_do = 0;
    w.off_rowc = align256(BH * Nq * dv * 2);
    w.off_rowt = w.off_rowc + align256(BH * w.Nq_pad * 16);
    w.off_gpart = w.off_rowt + align256(BH * w.Nq_pad * 16);
    w.off_lpart = w.off_gpart + align256(BH * w.nchunk * dv * 4);
    w.total = w.off_lpart + align256(BH * w.nchunk * 4);
    return w;
}

template <int D, int DV, bool CAUSAL>
static int launch_backward_t(const BwdArgs& a, cudaStream_t st) {
    using LQ = BwdDqLayout<D, DV>;
    using LK = BwdDkvLayout<D, DV>;
    const BwdWorkspace w = bwd_workspace_layout(a.B, a.H, a.Nq, DV);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    BwdParams p;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.Nq_pad = w.Nq_pad;
    p.nchunk = w.nchunk;
    p.lambda = a.lambda;
    p.lambda_init = a.lambda_init;
    p.eps = a.eps;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    p.scale = (float)(1.0 / std::sqrt((double)D));
    p.gamma = a.gamma;
    p.dy = static_cast<const uint16_t*>(a.dy);
    p.o = a.o;
    p.o2 = a.o2;
    p.lse = a.lse;
    p.dout = reinterpret_cast<uint16_t*>(ws + w.off_do);
    p.rowc = reinterpret_cast<float4*>(ws + w.off_rowc);
    p.rowt = reinterpret_cast<float*>(ws + w.off_rowt);
    p.gpart = reinterpret_cast<float*>(ws + w.off_gpart);
    p.lpart = reinterpret_cast<float*>(ws + w.off_lpart);
    p.dq1 = static_cast<uint16_t*>(a.dq1);
    p.dq2 = static_cast<uint16_t*>(a.dq2);
    p.dk1 = static_cast<uint16_t*>(a.dk1);
    p.dk2 = static_cast<uint16_t*>(a.dk2);
    p.dv = static_cast<uint16_t*>(a.dv_grad);
    p.dlambda = a.dlambda;
    p.dgamma = a.dgamma;

    bwd_prep_kernel<DV><<<dim3(w.nchunk, a.H, a.B), 256, 0, st>>>(p);
    if (!cuda_ok(cudaGetLastError(), "backward: prep launch")) return LAUNCH_ERR_CUDA;

    CUtensorMap q1a, q2a, doa, k1a, k2a, va;   // dQ sweep: 128-row Q/dO boxes, BN-row K/V boxes
    CUtensorMap q1b, q2b, dob, k1b, k2b, vb;   // dK/dV sweep: 128-row Q/dO boxes (two 64-query units), 128-row K/V boxes
    const auto S = CU_TENSOR_MAP_SWIZZLE_128B;
    // Q/K rows are one swizzle span wide: 128 bytes (d = 64) or 64 bytes (d = 32).
    const auto SQ = D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make_map_bhnd(&q1a, a.q1, a.B, a.H, a.Nq, D, D, LQ::BM, SQ) ||
        !make_map_bhnd(&q2a, a.q2, a.B, a.H, a.Nq, D, D, LQ::BM, SQ) ||
        !make_map_bhnd(&doa, p.dout, a.B, a.H, a.Nq, DV, 64, LQ::BM, S) ||
        !make_map_bhnd(&k1a, a.k1, a.B, a.H, a.Nk, D, D, LQ::BN, SQ) ||
        !make_map_bhnd(&k2a, a.k2, a.B, a.H, a.Nk, D, D, LQ::BN, SQ) ||
        !make_map_bhnd(&va, a.v, a.B, a.H, a.Nk, DV, 64, LQ::BN, S) ||
        !make_map_bhnd(&q1b, a.q1, a.B, a.H, a.Nq, D, D, LK::BQ, SQ) ||
        !make_map_bhnd(&q2b, a.q2, a.B, a.H, a.Nq, D, D, LK::BQ, SQ) ||
        !make_map_bhnd(&dob, p.dout, a.B, a.H, a.Nq, DV, 64, LK::BQ, S) ||
        !make_map_bhnd(&k1b, a.k1, a.B, a.H, a.Nk, D, D, LK::BK, SQ) ||
        !make_map_bhnd(&k2b, a.k2, a.B, a.H, a.Nk, D, D, LK::BK, SQ) ||
        !make_map_bhnd(&vb, a.v, a.B, a.H, a.Nk, DV, 64, LK::BK, S))
        return LAUNCH_ERR_CUDA;

    auto kq = bwd_dq_kernel<D, DV, CAUSAL>;
    if (!cuda_ok(cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LQ::SMEM_BYTES),
                 "backward: dq shared memory"))
        return LAUNCH_ERR_CUDA;
    kq<<<dim3((a.Nq + LQ::BM - 1) / LQ::BM, a.H, a.B), LQ::THREADS, LQ::SMEM_BYTES, st>>>(q1a, q2a, doa, k1a, k2a,
                                                                                          va, p);
    if (!cuda_ok(cudaGetLastError(), "backward: dq launch")) return LAUNCH_ERR_CUDA;

    auto kk = bwd_dkv_kernel<D, DV, CAUSAL>;
    if (!cuda_ok(cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LK::SMEM_BYTES),
                 "backward: dkv shared memory"))
        return LAUNCH_ERR_CUDA;
    kk<<<dim3((a.Nk + LK::BK - 1) / LK::BK, a.H, a.B), LK::THREADS, LK::SMEM_BYTES, st>>>(q1b, q2b, dob, k1b, k2b,
                                                                                          vb, p);
    if (!cuda_ok(cudaGetLastError(), "backward: dkv launch")) return LAUNCH_ERR_CUDA;

    if (a.dgamma || a.dlambda) {
        bwd_finalize_kernel<DV><<<a.H + 1, 256, 0, st>>>(p);
        if (!cuda_ok(cudaGetLastError(), "backward: finalize launch")) return LAUNCH_ERR_CUDA;
    }
    return LAUNCH_OK;
}

int launch_backward(const BwdArgs& a, cudaStream_t st) {
    if (a.d == 64 && a.dv == 128)
        return a.causal ? launch_backward_t<64, 128, true>(a, st) : launch_backward_t<64, 128, false>(a, st);
    if (a.d == 32 && a.dv == 64)
        return a.causal ? launch_backward_t<32, 64, true>(a, st) : launch_backward_t<32, 64, false>(a, st);
    return LAUNCH_ERR_UNSUPPORTED;
}

// ----------------------------------------------------------------- standard attention

template <bool CAUSAL>
static int launch_standard_t(const StandardArgs& a, cudaStream_t st) {
    using L = StandardLayout;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map_bhnd(&mq, a.q, a.B, a.H, a.Nq, L::D, 64, L::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bhnd(&mk, a.k, a.B, a.H, a.Nk, L::D, 64, L::BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_bhnd(&mv, a.v, a.B, a.H, a.Nk, L::DV, 64, L::BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        // output boxes of the persistent form's TMA stores: 32 rows x 64 columns
        !make_map_bhnd(&mo, a.out, a.B, a.H, a.Nq, L::DV, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return LAUNCH_ERR_CUDA;
    StandardParams p;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)L::D));
    p.out = static_cast<uint16_t*>(a.out);
    p.out_f32 = a.out_f32;
    p.weight_major = weight_major_order(CAUSAL, a.B, a.H, a.Nk, 2ll * (L::D + L::DV));
    // Persistent for short sequences, as the differential prefill.
    const long long pairs = (long long)((a.Nq + 2 * L::BM - 1) / (2 * L::BM)) * a.H * a.B;
    const int sms = sm_count();
    const bool small = pairs < kMaxTiles1D;
    const bool persist = sms > 0 && pairs > sms && a.Nk <= kPersistMaxNk && small;
    inv_div(p.weight_major ? (unsigned)((long long)a.H * a.B) : (unsigned)((a.Nq + 2 * L::BM - 1) / (2 * L::BM)),
            p.div_major_m, p.div_major_s);
    inv_div((unsigned)a.H, p.div_h_m, p.div_h_s);
    p.head_group = CAUSAL && !persist && small ? head_group_size(a.B, a.H, a.Nk, 2ll * (L::D + L::DV)) : 0;
    auto kern = persist ? standard_attn_kernel<CAUSAL, true> : standard_attn_kernel<CAUSAL, false>;
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM_BYTES),
                 "standard attention: set shared memory"))
        return LAUNCH_ERR_CUDA;
    const dim3 grid = persist          ? dim3(sms, 1, 1)
                      : p.head_group ? dim3((unsigned)pairs, 1, 1)
                                     : dim3((a.Nq + 2 * L::BM - 1) / (2 * L::BM), a.H, a.B);
    return cuda_ok(launch_dependent(kern, grid, dim3(L::THREADS), (size_t)L::SMEM_BYTES, st, mq, mk, mv, mo, p),
                   "standard attention: launch")
               ? LAUNCH_OK
               : LAUNCH_ERR_CUDA;
}

int launch_standard(const StandardArgs& a, cudaStream_t st) {
    if (a.d != StandardLayout::D || a.dv != StandardLayout::DV) return LAUNCH_ERR_UNSUPPORTED;
    return a.causal ? launch_standard_t<true>(a, st) : launch_standard_t<false>(a, st);
}

// ----------------------------------------------------------------- decode


template <int D, int DV, bool PAGED>
static int launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
    using L = DecodeLayout<D, DV>;
    // K1/K2 viewed as [B*H*Nk rows, D]: 32-row boxes with the swizzle that
    // matches the row width.
    CUtensorMap mk1, mk2;
    const CUtensorMapSwizzle swz = D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const int rows = PAGED ? a.num_pages * a.H * a.page_size : a.B * a.H * a.Nk;
    if (!make_map_bhnd(&mk1, a.k1, 1, 1, rows, D, D, L::KC, swz) ||
        !make_map_bhnd(&mk2, a.k2, 1, 1, rows, D, D, L::KC, swz))
        return LAUNCH_ERR_CUDA;
    DecodeParams p;
    p.q1 = static_cast<const uint16_t*>(a.q1);
    p.q2 = static_cast<const uint16_t*>(a.q2);
    p.v = static_cast<const uint16_t*>(a.v);
    p.B = a.B;
    p.H = a.H;
    p.Nk = a.Nk;
    p.S = a.splits;
    p.keys_per_split = a.keys_per_split;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    p.ws = a.ws;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.max_pages = a.max_pages;
    p.page_size = a.page_size;
    p.num_pages = a.num_pages;
    auto kern = decode_split_kernel<D, DV, PAGED>;
    if (!cuda_ok(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::SMEM_BYTES),
                 "decode: set shared memory"))
        return LAUNCH_ERR_CUDA;
    if (!cuda_ok(launch_dependent(kern, dim3(a.splits, a.H, a.B), dim3(L::THREADS), L::SMEM_BYTES, st, mk1, mk2, p),
                 "decode: split launch"))
        return LAUNCH_ERR_CUDA;
    if (a.partials_only) return LAUNCH_OK;
    MergeParams mp;
    mp.B = a.B;
    mp.H = a.H;
    mp.S = a.splits;
    mp.parts = 1;
    mp.lambda = a.lambda;
    mp.lambda_init = a.lambda_init;
    mp.eps = a.eps;
    mp.ws = a.ws;
    mp.gamma = a.gamma;
    mp.out = static_cast<uint16_t*>(a.out);
    mp.o_prenorm = a.o_prenorm;
    const int heads = a.B * a.H;
    const cudaError_t e = mp.parts * mp.S <= kMergeWideMax
                              ? launch_dependent(decode_merge_wide_kernel<DV>, dim3(heads), dim3(DV), 0, st, mp)
                              : launch_dependent(decode_merge_kernel<DV>, dim3((heads + 3) / 4), dim3(128), 0, st, mp);
    return cuda_ok(e, "decode: merge launch")
               ? LAUNCH_OK
               : LAUNCH_ERR_CUDA;
}

int launch_decode_merge(const MergeArgs& a, cudaStream_t st) {
    MergeParams mp;
    mp.B = a.B;
    mp.H = a.H;
    mp.S = a.splits;
    mp.parts = a.parts;
    mp.lambda = a.lambda;
    mp.lambda_init = a.lambda_init;
    mp.eps = a.eps;
    mp.ws = a.ws;
    mp.gamma = a.gamma;
    mp.out = static_cast<uint16_t*>(a.out);
    mp.o_prenorm = a.o_prenorm;
    const int heads = a.B * a.H;
    cudaError_t e;
    const bool wide = a.parts * a.splits <= kMergeWideMax;
    if (a.dv == 128)
        e = wide ? launch_dependent(decode_merge_wide_kernel<128>, dim3(heads), dim3(128), 0, st, mp)
                 : launch_dependent(decode_merge_kernel<128>, dim3((heads + 3) / 4), dim3(128), 0, st, mp);
    else if (a.dv == 64)
        e = wide ? launch_dependent(decode_merge_wide_kernel<64>, dim3(heads), dim3(64), 0, st, mp)
                 : launch_dependent(decode_merge_kernel<64>, dim3((heads + 3) / 4), dim3(128), 0, st, mp);
    else
        return LAUNCH_ERR_UNSUPPORTED;
    return cuda_ok(e, "decode: merge of gathered partials") ? LAUNCH_OK : LAUNCH_ERR_CUDA;
}

int launch_decode(const DecodeArgs& a, cudaStream_t st) {
    const bool paged = a.block_table != nullptr;
    if (a.d == 64 && a.dv == 128)
        return paged ? launch_decode_t<64, 128, true>(a, st) : launch_decode_t<64, 128, false>(a, st);
    if (a.d == 32 && a.dv == 64)
        return paged ? launch_decode_t<32, 64, true>(a, st) : launch_decode_t<32, 64, false>(a, st);
    return LAUNCH_ERR_UNSUPPORTED;
}

// ----------------------------------------------------------------- decode without allocation
//
// Scratch for diffattn_decode_noalloc: the split partials live in this
// file-scope device array instead of a caller-provided workspace.  Every
// device that loads the library holds these 8 MiB until the process exits.
// In host code the array's name is only a stand-in, so its device address is
// looked up with cudaGetSymbolAddress, once per device, with that device
// current, and cached.
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

int decode_noalloc_scratch(void** ptr, size_t* bytes) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = -1;
    if (!cuda_ok(cudaGetDevice(&dev), "no-alloc decode: get device") || dev < 0 || dev >= kMaxDevices)
        return LAUNCH_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (!cuda_ok(cudaGetSymbolAddress(&p, g_decode_scratch), "no-alloc decode: scratch address") || !p)
            return LAUNCH_ERR_CUDA;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    *bytes = kNoAllocScratchBytes;
    return LAUNCH_OK;
}

// One thread waits, through the library's bounded wait, for a phase of a
// freshly initialised mbarrier that nothing arrives on: the wait runs out,
// records its site in the device error word and returns, and the kernel
// exits normally.
__global__ void __launch_bounds__(32, 1) selftest_wait_kernel() {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
        mbar_wait(smem_addr(&bar), 0, ERR_SITE_SELFTEST);
    }
}

int launch_selftest_wait(cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>();
    return cuda_ok(cudaGetLastError(), "self-test: launch") ? LAUNCH_OK : LAUNCH_ERR_CUDA;
}

int read_and_clear_device_error(cudaStream_t st, int* value) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return LAUNCH_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return LAUNCH_ERR_CUDA;
    const int zero = 0;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return LAUNCH_ERR_CUDA;
    *value = v;
    return LAUNCH_OK;
}

}  // namespace diffattn
