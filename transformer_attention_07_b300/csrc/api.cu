// C ABI of the differential-attention library (declared in include/diffattn.h).
// Each entry point checks every argument on the host first and launches
// nothing when one is wrong; the launchers in kernels.cu do the rest.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/diffattn.h"
#include "launch.h"

namespace {

constexpr int kMaxAutoSplits = 32;
constexpr int kMaxSplits = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool supported_widths(int d, int dv) { return (d == 64 && dv == 128) || (d == 32 && dv == 64); }

int from_launch(int s) {
    if (s == diffattn::LAUNCH_OK) return DIFFATTN_OK;
    if (s == diffattn::LAUNCH_ERR_UNSUPPORTED) return DIFFATTN_ERR_UNSUPPORTED;
    return DIFFATTN_ERR_CUDA;
}

// Per-call scalars shared by both entry points.
int check_scalars(float lambda, float lambda_init, float eps) {
    if (!std::isfinite(lambda) || !std::isfinite(lambda_init)) return DIFFATTN_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return DIFFATTN_ERR_INVALID_ARG;
    return DIFFATTN_OK;
}

// A BHND tensor of this shape must be describable by a 4-D tensor map:
// every byte stride below 2^40.
bool fits_tensor_map(int64_t H, int64_t N, int64_t W) { return H * N * W * 2 < (int64_t(1) << 40); }

// Checks shared by every prefill entry point, then the launch.  Optional
// outputs (o_prenorm, o2, lse) and inputs (gamma, qk_scale) may be null.
int prefill(const diffattn::PrefillArgs& a, void* stream) {
    if (!a.q1 || !a.k1 || !a.q2 || !a.k2 || !a.v || !a.out) return DIFFATTN_ERR_INVALID_ARG;
    if (a.B < 0 || a.H < 0 || a.Nq < 0 || a.Nk < 1 || a.d < 1 || a.dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (a.causal != 0 && a.causal != 1) return DIFFATTN_ERR_INVALID_ARG;
    if (a.causal && a.Nq > a.Nk) return DIFFATTN_ERR_INVALID_ARG;
    if (int s = check_scalars(a.lambda, a.lambda_init, a.eps)) return s;
    if (!supported_widths(a.d, a.dv)) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(a.q1) || !aligned16(a.k1) || !aligned16(a.q2) || !aligned16(a.k2) || !aligned16(a.v) ||
        !aligned16(a.out) || !aligned16(a.o_prenorm) || !aligned16(a.o2) || !aligned4(a.lse) ||
        !aligned4(a.gamma) || !aligned4(a.qk_scale))
        return DIFFATTN_ERR_INVALID_ARG;
    if (a.B > 65535 || a.H > 65535) return DIFFATTN_ERR_INVALID_ARG;   // grid y/z limits
    if (!fits_tensor_map(a.H, a.Nq, a.d) || !fits_tensor_map(a.H, a.Nk, a.dv)) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)a.B * a.H * a.Nq == 0) return DIFFATTN_OK;
    return from_launch(diffattn::launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

size_t workspace_for(int B, int H, int dv, int splits) {
    return (size_t)B * (size_t)H * (size_t)splits * 2u * (size_t)(dv + 4) * sizeof(float);
}

// Key ranges per (b, h): the count that minimises a cost model of the split
// kernel, fitted to B300 timings of B1-B8, H8-H32 and 1K-32K keys.
//   * One CTA streams one key range.  In a wave that occupies every SM, a CTA
//     gets the fair per-SM share of HBM bandwidth; in a wave with idle SMs it
//     gets up to 1.3 times that share (measured: 55-60 GB/s per CTA against
//     44 GB/s).
//   * Every wave adds a fixed cost (CTA start, the first loads' latency, the
//     partials' write) worth about 128 KB of streaming (3 us).
//   * Ranges are whole 32-key chunks, none empty, at least 256 keys, and at
//     most max_splits.  A count must beat the previous best by 1% to be taken,
//     so ties go to fewer ranges (less merge work).
// Filling whole waves with many short ranges, the previous rule, cost up to
// 40% at B4 H32 with 4K keys.
int choose_splits(int64_t heads, int Nk, int bytes_per_key, int sms, int max_splits = kMaxAutoSplits) {
    if (heads < 1 || Nk < 1 || sms < 1) return 1;
    constexpr double kWaveCost = 128.0 * 1024.0;   // bytes
    constexpr double kIdleBoost = 1.3;
    const int by_keys = (Nk + 255) / 256;
    const int cap = std::max(1, std::min(by_keys, max_splits));
    int best = 1;
    double best_cost = -1.0;
    for (int s = 1; s <= cap; ++s) {
        const int per = ((Nk + s - 1) / s + 31) / 32 * 32;
        if ((int64_t)(s - 1) * per >= Nk) continue;   // the last range would be empty
        const double bytes = (double)per * bytes_per_key;
        const int64_t ctas = heads * s;
        const int64_t full = ctas / sms, rem = ctas % sms;
        double cost = (double)full * (kWaveCost + bytes);
        if (rem) cost += kWaveCost + bytes * std::max(1.0 / kIdleBoost, (double)rem / sms);
        if (best_cost < 0.0 || cost < 0.99 * best_cost) {
            best = s;
            best_cost = cost;
        }
    }
    return best;
}

int key_bytes(int d, int dv) { return (2 * d + dv) * 2; }

// Streaming multiprocessors of the current device (cached per device), or 0.
int device_sms() { return diffattn::sm_count(); }

// Argument checks of the contiguous-cache decode entry points (everything
// but the workspace); DIFFATTN_OK when the call may proceed.
int check_decode(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, float lambda,
                 float lambda_init, int B, int H, int Nk, int d, int dv, const float* gn_gamma, float eps,
                 int num_splits, const void* out, const float* o_prenorm) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !out) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nk < 1 || d < 1 || dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (num_splits < 0 || num_splits > kMaxSplits) return DIFFATTN_ERR_INVALID_ARG;
    if (int s = check_scalars(lambda, lambda_init, eps)) return s;
    if (!supported_widths(d, dv)) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
        !aligned16(out) || !aligned16(o_prenorm) || !aligned4(gn_gamma))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B > 65535 || H > 65535) return DIFFATTN_ERR_INVALID_ARG;
    // The key caches are addressed as one [B*H*Nk, d] matrix with 32-bit rows.
    if ((int64_t)B * H * Nk >= (int64_t(1) << 31) - 64) return DIFFATTN_ERR_INVALID_ARG;
    return DIFFATTN_OK;
}

// The launch part of diffattn_decode, once the split count is fixed.
int decode_with_splits(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, float lambda,
                       float lambda_init, int B, int H, int Nk, int d, int dv, const float* gn_gamma, float eps,
                       int splits, void* workspace, size_t workspace_bytes, void* out, float* o_prenorm,
                       void* stream) {
    if (!workspace || workspace_bytes < workspace_for(B, H, dv, splits)) return DIFFATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DIFFATTN_ERR_INVALID_ARG;
    const int per = (Nk + splits - 1) / splits;
    const int keys_per_split = (per + 31) / 32 * 32;
    diffattn::DecodeArgs a{q1, k1, q2, k2, v, lambda, lambda_init, eps, B, H, Nk, d, dv,
                           splits, keys_per_split, gn_gamma, static_cast<float*>(workspace), out, o_prenorm,
                           nullptr, nullptr, 0, 0, 0, false};
    return from_launch(diffattn::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int diffattn_fwd_ex(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                    float lambda, float lambda_init, int causal, int B, int H, int Nq, int Nk, int d, int dv,
                    const float* gn_gamma, float eps, void* out, float* o_prenorm, void* stream) {
    diffattn::PrefillArgs a{q1, k1, q2, k2, v, lambda, lambda_init, eps, causal, B, H, Nq, Nk, d, dv,
                            gn_gamma, out, o_prenorm, nullptr, nullptr, nullptr};
    return prefill(a, stream);
}

int diffattn_fwd_fp8(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                     const float* qk_scale, float lambda, float lambda_init, int causal, int B, int H, int Nq, int Nk,
                     int d, int dv, const float* gn_gamma, float eps, void* out, float* o_prenorm, void* stream) {
    if (!qk_scale) return DIFFATTN_ERR_INVALID_ARG;
    diffattn::PrefillArgs a{q1, k1, q2, k2, v, lambda, lambda_init, eps, causal, B, H, Nq, Nk, d, dv,
                            gn_gamma, out, o_prenorm, nullptr, nullptr, qk_scale};
    return prefill(a, stream);
}

int diffattn_fwd_train(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                       float lambda, float lambda_init, int causal, int B, int H, int Nq, int Nk, int d, int dv,
                       const float* gn_gamma, float eps, void* out, float* o_prenorm, float* o2, float* lse,
                       void* stream) {
    if (!o_prenorm || !o2 || !lse) return DIFFATTN_ERR_INVALID_ARG;
    diffattn::PrefillArgs a{q1, k1, q2, k2, v, lambda, lambda_init, eps, causal, B, H, Nq, Nk, d, dv,
                            gn_gamma, out, o_prenorm, o2, lse, nullptr};
    return prefill(a, stream);
}

size_t diffattn_bwd_workspace_bytes(int B, int H, int Nq, int dv) {
    if (B < 0 || H < 0 || Nq < 0 || dv < 1) return 0;
    return diffattn::bwd_workspace_layout(B, H, Nq, dv).total;
}

int diffattn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, const void* dy,
                 const float* o_prenorm, const float* o2, const float* lse, float lambda, float lambda_init,
                 int causal, int B, int H, int Nq, int Nk, int d, int dv, const float* gn_gamma, float eps,
                 void* dq1, void* dk1, void* dq2, void* dk2, void* dv_grad, float* dlambda, float* dgamma,
                 void* workspace, size_t workspace_bytes, void* stream) {
    // With no query rows the query-side tensors are empty and may be NULL.
    const bool rows = Nq != 0;
    if (!k1 || !k2 || !v || !dk1 || !dk2 || !dv_grad) return DIFFATTN_ERR_INVALID_ARG;
    if (rows && (!q1 || !q2 || !dy || !o_prenorm || !o2 || !lse || !dq1 || !dq2)) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return DIFFATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return DIFFATTN_ERR_INVALID_ARG;
    if (int s = check_scalars(lambda, lambda_init, eps)) return s;
    if (!supported_widths(d, dv)) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v) ||
        !aligned16(dy) || !aligned16(o_prenorm) || !aligned16(o2) || !aligned4(lse) || !aligned4(gn_gamma) ||
        !aligned16(dq1) || !aligned16(dk1) || !aligned16(dq2) || !aligned16(dk2) || !aligned16(dv_grad) ||
        !aligned4(dlambda) || !aligned4(dgamma))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B > 65535 || H > 65535) return DIFFATTN_ERR_INVALID_ARG;
    if (!fits_tensor_map(H, Nq, dv) || !fits_tensor_map(H, Nk, dv)) return DIFFATTN_ERR_INVALID_ARG;
    const diffattn::BwdWorkspace w = diffattn::bwd_workspace_layout(B, H, Nq, dv);
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    if (!workspace || workspace_bytes < w.total) return DIFFATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DIFFATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (Nq == 0) {
        // No query rows: every key gradient is zero and so are dlambda and dgamma.
        const size_t kd = (size_t)B * H * Nk * d * 2, kv = (size_t)B * H * Nk * dv * 2;
        if (cudaMemsetAsync(dk1, 0, kd, st) != cudaSuccess || cudaMemsetAsync(dk2, 0, kd, st) != cudaSuccess ||
            cudaMemsetAsync(dv_grad, 0, kv, st) != cudaSuccess ||
            (dlambda && cudaMemsetAsync(dlambda, 0, sizeof(float), st) != cudaSuccess) ||
            (dgamma && cudaMemsetAsync(dgamma, 0, (size_t)H * dv * sizeof(float), st) != cudaSuccess))
            return DIFFATTN_ERR_CUDA;
        return DIFFATTN_OK;
    }
    diffattn::BwdArgs a{q1, k1, q2, k2, v, dy, o_prenorm, o2, lse, lambda, lambda_init, eps, causal, B, H, Nq, Nk,
                        d, dv, gn_gamma, dq1, dk1, dq2, dk2, dv_grad, dlambda, dgamma, workspace};
    return from_launch(diffattn::launch_backward(a, st));
}

int diffattn_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, float lambda,
                 float lambda_init, int causal, int B, int H, int Nq, int Nk, int d, int dv, const float* gn_gamma,
                 float eps, void* out, void* stream) {
    return diffattn_fwd_ex(q1, k1, q2, k2, v, lambda, lambda_init, causal, B, H, Nq, Nk, d, dv, gn_gamma, eps, out,
                           nullptr, stream);
}

int diffattn_standard_fwd(const void* q, const void* k, const void* v, int causal, int B, int H, int Nq, int Nk,
                          int d, int dv, void* out, float* out_f32, void* stream) {
    if (!q || !k || !v || !out) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return DIFFATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return DIFFATTN_ERR_INVALID_ARG;
    if (d != 128 || dv != 128) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(out_f32))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B > 65535 || H > 65535) return DIFFATTN_ERR_INVALID_ARG;
    if (!fits_tensor_map(H, Nq, d) || !fits_tensor_map(H, Nk, dv)) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H * Nq == 0) return DIFFATTN_OK;
    diffattn::StandardArgs a{q, k, v, causal, B, H, Nq, Nk, d, dv, out, out_f32};
    return from_launch(diffattn::launch_standard(a, static_cast<cudaStream_t>(stream)));
}

int diffattn_prefill_plan(int B, int H, int Nq, int Nk, int d, int dv, int causal, int fp8, int sms, int* form,
                          long long* ctas) {
    if (form == nullptr || ctas == nullptr) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 1 || sms < 1 || (causal != 0 && causal != 1) || (fp8 != 0 && fp8 != 1))
        return DIFFATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return DIFFATTN_ERR_INVALID_ARG;
    if (!supported_widths(d, dv)) return DIFFATTN_ERR_UNSUPPORTED;
    const diffattn::PrefillPlan pl = diffattn::prefill_plan(B, H, Nq, Nk, d, dv, causal != 0, fp8 != 0, sms);
    *form = pl.form;
    *ctas = pl.ctas;
    return DIFFATTN_OK;
}

int diffattn_decode_auto_splits(int B, int H, int Nk, int d, int dv, int sms, int max_splits) {
    if (B < 1 || H < 1 || Nk < 1 || sms < 1 || max_splits < 0 || max_splits > kMaxSplits) return 0;
    if (!supported_widths(d, dv)) return 0;
    return choose_splits((int64_t)B * H, Nk, key_bytes(d, dv), sms, max_splits == 0 ? kMaxAutoSplits : max_splits);
}

size_t diffattn_decode_workspace_bytes(int B, int H, int Nk, int dv, int num_splits) {
    if (B < 0 || H < 0 || Nk < 1 || dv < 1 || num_splits < 0 || num_splits > kMaxSplits) return 0;
    return workspace_for(B, H, dv, num_splits == 0 ? kMaxAutoSplits : num_splits);
}

int diffattn_decode(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, float lambda,
                    float lambda_init, int B, int H, int Nk, int d, int dv, const float* gn_gamma, float eps,
                    int num_splits, void* workspace, size_t workspace_bytes, void* out, float* o_prenorm,
                    void* stream) {
    if (int s = check_decode(q1, k1, q2, k2, v, lambda, lambda_init, B, H, Nk, d, dv, gn_gamma, eps, num_splits,
                             out, o_prenorm))
        return s;
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    int splits = num_splits;
    if (splits == 0) {
        const int sms = device_sms();
        if (sms < 1) return DIFFATTN_ERR_CUDA;
        splits = choose_splits((int64_t)B * H, Nk, key_bytes(d, dv), sms);
    }
    return decode_with_splits(q1, k1, q2, k2, v, lambda, lambda_init, B, H, Nk, d, dv, gn_gamma, eps, splits,
                              workspace, workspace_bytes, out, o_prenorm, stream);
}

size_t diffattn_decode_partials_bytes(int B, int H, int dv, int num_splits) {
    if (B < 0 || H < 0 || dv < 1 || num_splits < 1 || num_splits > kMaxSplits) return 0;
    return workspace_for(B, H, dv, num_splits);
}

int diffattn_decode_partials(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, int B,
                             int H, int Nk, int d, int dv, int num_splits, float* partials, size_t partials_bytes,
                             void* stream) {
    if (!q1 || !k1 || !q2 || !k2 || !v) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nk < 1 || d < 1 || dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (num_splits < 1 || num_splits > kMaxSplits) return DIFFATTN_ERR_INVALID_ARG;
    if (!supported_widths(d, dv)) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q1) || !aligned16(k1) || !aligned16(q2) || !aligned16(k2) || !aligned16(v))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B > 65535 || H > 65535) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H * Nk >= (int64_t(1) << 31) - 64) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    if (!partials || partials_bytes < workspace_for(B, H, dv, num_splits)) return DIFFATTN_ERR_WORKSPACE;
    if (!aligned16(partials)) return DIFFATTN_ERR_INVALID_ARG;
    const int per = (Nk + num_splits - 1) / num_splits;
    const int keys_per_split = (per + 31) / 32 * 32;
    // lambda, lambda_init, eps, gamma and out belong to the merge; the split
    // kernel does not read them.
    diffattn::DecodeArgs a{q1, k1, q2, k2, v, 0.0f, 0.0f, 0.0f, B, H, Nk, d, dv, num_splits, keys_per_split,
                           nullptr, partials, nullptr, nullptr, nullptr, nullptr, 0, 0, 0, true};
    return from_launch(diffattn::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

int diffattn_decode_merge(const float* partials, int num_parts, int B, int H, int dv, int num_splits, float lambda,
                          float lambda_init, const float* gn_gamma, float eps, void* out, float* o_prenorm,
                          void* stream) {
    if (!partials || !out) return DIFFATTN_ERR_INVALID_ARG;
    if (num_parts < 1 || B < 0 || H < 0 || num_splits < 1 || num_splits > kMaxSplits) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)num_parts * num_splits > 4096) return DIFFATTN_ERR_INVALID_ARG;
    if (dv != 128 && dv != 64) return DIFFATTN_ERR_UNSUPPORTED;
    if (int s = check_scalars(lambda, lambda_init, eps)) return s;
    if (!aligned16(partials) || !aligned16(out) || !aligned16(o_prenorm) || !aligned4(gn_gamma))
        return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    diffattn::MergeArgs a{partials, num_parts, B, H, num_splits, dv, lambda, lambda_init, eps, gn_gamma, out,
                          o_prenorm};
    return from_launch(diffattn::launch_decode_merge(a, static_cast<cudaStream_t>(stream)));
}

// Decode for callers that cannot allocate device memory: the split partials
// go to the library's own static scratch instead of a caller workspace.  The
// arguments are checked exactly as in diffattn_decode, before the runtime is
// asked for anything.  With num_splits = 0 the split count is chosen as there
// but never above what the scratch holds; DIFFATTN_ERR_WORKSPACE only when
// even one range per head, or the count the caller fixed, does not fit.
int diffattn_decode_noalloc(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                            float lambda, float lambda_init, int B, int H, int Nk, int d, int dv,
                            const float* gn_gamma, float eps, int num_splits, void* out, float* o_prenorm,
                            void* stream) {
    if (int s = check_decode(q1, k1, q2, k2, v, lambda, lambda_init, B, H, Nk, d, dv, gn_gamma, eps, num_splits,
                             out, o_prenorm))
        return s;
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    const size_t per_split = workspace_for(B, H, dv, 1);
    const size_t fit = diffattn::kNoAllocScratchBytes / per_split;
    if (fit < 1 || (size_t)num_splits > fit) return DIFFATTN_ERR_WORKSPACE;
    int splits = num_splits;
    if (splits == 0) {
        const int sms = device_sms();
        if (sms < 1) return DIFFATTN_ERR_CUDA;
        splits = choose_splits((int64_t)B * H, Nk, key_bytes(d, dv), sms,
                               fit < (size_t)kMaxAutoSplits ? (int)fit : kMaxAutoSplits);
    }
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    if (diffattn::decode_noalloc_scratch(&scratch, &scratch_bytes) != diffattn::LAUNCH_OK) return DIFFATTN_ERR_CUDA;
    return decode_with_splits(q1, k1, q2, k2, v, lambda, lambda_init, B, H, Nk, d, dv, gn_gamma, eps, splits,
                              scratch, scratch_bytes, out, o_prenorm, stream);
}

int diffattn_decode_paged(const void* q1, const void* q2, const void* k1_pages, const void* k2_pages,
                          const void* v_pages, const int32_t* block_table, const int32_t* seq_lens, int max_pages,
                          int page_size, int num_pages, float lambda, float lambda_init, int B, int H, int d, int dv,
                          const float* gn_gamma, float eps, int num_splits, void* workspace, size_t workspace_bytes,
                          void* out, float* o_prenorm, void* stream) {
    if (!q1 || !q2 || !k1_pages || !k2_pages || !v_pages || !block_table || !seq_lens || !out)
        return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || d < 1 || dv < 1 || max_pages < 1 || num_pages < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (page_size < 32 || page_size % 32 != 0) return DIFFATTN_ERR_INVALID_ARG;
    if (num_splits < 0 || num_splits > kMaxSplits) return DIFFATTN_ERR_INVALID_ARG;
    if (int s = check_scalars(lambda, lambda_init, eps)) return s;
    if (!supported_widths(d, dv)) return DIFFATTN_ERR_UNSUPPORTED;
    if (!aligned16(q1) || !aligned16(q2) || !aligned16(k1_pages) || !aligned16(k2_pages) || !aligned16(v_pages) ||
        !aligned16(out) || !aligned16(o_prenorm) || !aligned4(gn_gamma) || !aligned4(block_table) ||
        !aligned4(seq_lens))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B > 65535 || H > 65535) return DIFFATTN_ERR_INVALID_ARG;
    // Page caches are addressed as one [num_pages*H*page_size, d] matrix with
    // 32-bit rows; the longest sequence is max_pages * page_size keys.
    if ((int64_t)num_pages * H * page_size >= (int64_t(1) << 31) - 64) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)max_pages * page_size >= (int64_t(1) << 31) - 64) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H == 0) return DIFFATTN_OK;
    const int max_len = max_pages * page_size;
    // Each key range may span at most kDecodeMaxSplitPages pages.
    auto pages_ok = [&](int splits) {
        const int per = ((max_len + splits - 1) / splits + 31) / 32 * 32;
        return per / page_size + 1 <= diffattn::kDecodeMaxSplitPages;
    };
    int splits = num_splits;
    if (splits == 0) {
        const int sms = device_sms();
        if (sms < 1) return DIFFATTN_ERR_CUDA;
        splits = choose_splits((int64_t)B * H, max_len, key_bytes(d, dv), sms);
        while (!pages_ok(splits) && splits < kMaxSplits) ++splits;
    }
    if (!pages_ok(splits)) return DIFFATTN_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < workspace_for(B, H, dv, splits)) return DIFFATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DIFFATTN_ERR_INVALID_ARG;
    const int per = (max_len + splits - 1) / splits;
    const int keys_per_split = (per + 31) / 32 * 32;
    diffattn::DecodeArgs a{q1, k1_pages, q2, k2_pages, v_pages, lambda, lambda_init, eps, B, H, max_len, d, dv,
                           splits, keys_per_split, gn_gamma, static_cast<float*>(workspace), out, o_prenorm,
                           block_table, seq_lens, max_pages, page_size, num_pages, false};
    return from_launch(diffattn::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

const char* diffattn_status_string(int status) {
    switch (status) {
        case DIFFATTN_OK: return "ok";
        case DIFFATTN_ERR_INVALID_ARG: return "invalid argument";
        case DIFFATTN_ERR_UNSUPPORTED: return "unsupported head widths (d, dv)";
        case DIFFATTN_ERR_CUDA: return "CUDA runtime error";
        case DIFFATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case DIFFATTN_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int diffattn_selftest_wait_timeout(void* stream) {
    return diffattn::launch_selftest_wait(static_cast<cudaStream_t>(stream)) == diffattn::LAUNCH_OK
               ? DIFFATTN_OK
               : DIFFATTN_ERR_CUDA;
}

int diffattn_last_device_error(void* stream) {
    int v = 0;
    if (diffattn::read_and_clear_device_error(static_cast<cudaStream_t>(stream), &v) != diffattn::LAUNCH_OK)
        return -1;
    return v;
}

}  // extern "C"
