// Differential-attention oracle: a plain, slow, fp64 CPU statement of what the
// forward pass computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
// and the benchmark's CPU-baseline leg call it; the product path never does.
// It shares no code, header, table or helper with the CUDA library.
//
// What it follows (Differential Transformer pages):
//  * "How does Differential Attention work…" (iloveeagents.com), section
//    "Mathematical Formula": DiffAttn(Q,K,V) = (softmax(Q1 K1^T/sqrt d)
//    - lambda * softmax(Q2 K2^T/sqrt d)) V.  One softmax per map; the Example
//    snippet on that page applies a second softmax to the second map, which
//    this oracle deliberately does not do.
//  * "Differential Transformer: How Noise-Canceling Attention Reinvents LLMs"
//    (llmbytes.dev), section "How Differential Attention Cancels Common-Mode
//    Noise", steps 2-4: two independent softmax maps, the lambda-weighted
//    subtraction, then GroupNorm of the multi-head output and the
//    (1 - lambda_init) scale.
//
// Readings taken where the pages are silent:
//  * scale 1/sqrt(d) with d the query/key head width;
//  * causal mask, when asked for, is the same on both maps and bottom-right
//    aligned: key j is visible to query i iff j <= i + Nk - Nq;
//  * GroupNorm has one group per head; statistics are taken per token over
//    that head's dv channels (biased variance, eps inside the square root),
//    with a per-channel gain gamma[h*dv + c] and no bias; the (1 - lambda_init)
//    factor multiplies the normalised value.
//
// Every row is computed from its definition: the logits of both maps, the two
// max-subtracted softmax rows materialised in full, then the weighted sum over
// the keys.  No tiling, no online softmax, no fusion.
//
// The backward pass (oracle_diffattn_bwd) is the chain rule through the same
// steps, taken in reverse for one query row at a time: the GroupNorm and gain,
// the product with V, the lambda-weighted subtraction, each softmax, and the
// two logit products.  lambda is a learnable scalar on the pages (the
// iloveeagents.com Q&A, "Mathematical Formula"), so its gradient is returned
// too, as is that of the GroupNorm gain.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <atomic>

namespace {

// Input element types the oracle accepts.  bf16 values are passed as their raw
// 16-bit patterns and widened exactly (a bf16 is the top half of an fp32).
enum InType { IN_F64 = 0, IN_F32 = 1, IN_BF16 = 2 };

inline double load_elem(const void* base, int type, int64_t idx) {
    if (type == IN_F64) return static_cast<const double*>(base)[idx];
    if (type == IN_F32) return static_cast<const float*>(base)[idx];
    uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return f;
}

struct Problem {
    const void *q1, *k1, *q2, *k2, *v;
    int type;
    double lambda, lambda_init;
    int causal;
    int B, H, Nq, Nk, d, dv;
    const double* gamma;  // [H*dv] or null (all ones)
    double eps;
};

// Number of keys query i may attend to.
inline int64_t visible_keys(const Problem& p, int64_t i) {
    if (!p.causal) return p.Nk;
    int64_t last = i + (int64_t)p.Nk - (int64_t)p.Nq;  // last visible key index
    if (last < 0) return 0;
    return std::min<int64_t>(last + 1, p.Nk);
}

// softmax of one map's logits row, in place: a_j = exp(s_j - max s) / sum.
void softmax_row(std::vector<double>& s, int64_t n) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) m = std::max(m, s[j]);
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = std::exp(s[j] - m);
        z += s[j];
    }
    for (int64_t j = 0; j < n; ++j) s[j] /= z;
}

// The two attention rows of query i over its visible keys: the logits
// s_r[j] = (q_r . k_r[j]) / sqrt(d) of each map, then one softmax per map.
void attention_rows(const Problem& p, int b, int h, int64_t i,
                    std::vector<double>& a1, std::vector<double>& a2) {
    const int64_t n = visible_keys(p, i);
    const int64_t bh = (int64_t)b * p.H + h;
    const int64_t qoff = (bh * p.Nq + i) * p.d;
    const int64_t koff = bh * p.Nk * p.d;
    const double inv_sqrt_d = 1.0 / std::sqrt((double)p.d);
    a1.assign(n, 0.0);
    a2.assign(n, 0.0);
    for (int64_t j = 0; j < n; ++j) {
        double s1 = 0.0, s2 = 0.0;
        for (int c = 0; c < p.d; ++c) {
            s1 += load_elem(p.q1, p.type, qoff + c) * load_elem(p.k1, p.type, koff + j * p.d + c);
            s2 += load_elem(p.q2, p.type, qoff + c) * load_elem(p.k2, p.type, koff + j * p.d + c);
        }
        a1[j] = s1 * inv_sqrt_d;
        a2[j] = s2 * inv_sqrt_d;
    }
    softmax_row(a1, n);
    softmax_row(a2, n);
}

// One query row of one head: fills a1/a2 (the two attention rows over the
// visible keys), o_pre (dv values) and y (dv normalised values).
void one_row(const Problem& p, int b, int h, int64_t i,
             std::vector<double>& a1, std::vector<double>& a2,
             double* o_pre, double* y) {
    attention_rows(p, b, h, i, a1, a2);
    const int64_t n = (int64_t)a1.size();
    const int64_t voff = ((int64_t)b * p.H + h) * p.Nk * p.dv;
    // Differential subtraction, then the product with V.
    for (int c = 0; c < p.dv; ++c) o_pre[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double w = a1[j] - p.lambda * a2[j];
        for (int c = 0; c < p.dv; ++c) o_pre[c] += w * load_elem(p.v, p.type, voff + j * p.dv + c);
    }
    // GroupNorm (group = this head, statistics over its dv channels), gain,
    // then the (1 - lambda_init) scale.
    double mu = 0.0;
    for (int c = 0; c < p.dv; ++c) mu += o_pre[c];
    mu /= p.dv;
    double var = 0.0;
    for (int c = 0; c < p.dv; ++c) var += (o_pre[c] - mu) * (o_pre[c] - mu);
    var /= p.dv;
    const double rstd = 1.0 / std::sqrt(var + p.eps);
    for (int c = 0; c < p.dv; ++c) {
        const double g = p.gamma ? p.gamma[(int64_t)h * p.dv + c] : 1.0;
        y[c] = (1.0 - p.lambda_init) * g * (o_pre[c] - mu) * rstd;
    }
}

// Gradient of one query row, given dy (the gradient of the loss with respect
// to this row's normalised output y).  Recomputes the row's forward pass, then
// applies the chain rule step by step, in reverse order:
//   y_c  = k g_c xhat_c, k = 1 - lambda_init, xhat_c = (o_c - mu) * rstd
//        -> dgamma_c += k dy_c xhat_c; gx_c = k g_c dy_c
//   xhat -> do_c = rstd (gx_c - mean(gx) - xhat_c mean(gx * xhat))
//   o    = sum_j (a1_j - lambda a2_j) v_j
//        -> dv_j += (a1_j - lambda a2_j) do; da1_j = do . v_j; da2_j = -lambda do . v_j;
//           dlambda += -sum_j a2_j (do . v_j)
//   a_r  = softmax(s_r) -> ds_r,j = a_r,j (da_r,j - sum_k a_r,k da_r,k)
//   s_r,j = (q_r . k_r,j) / sqrt(d) -> dq_r += ds_r,j k_r,j / sqrt(d); dk_r,j += ds_r,j q_r / sqrt(d)
// ds1/ds2 receive the logit gradients of the visible keys, do the pre-norm
// gradient (dv values); returns this row's contribution to dlambda and adds
// its contribution to dgamma_h (dv values).
struct RowGrad {
    std::vector<double> a1, a2, dp, ds1, ds2, o, dout;
};

double row_backward(const Problem& p, const void* dy, int dy_type, int b, int h, int64_t i, RowGrad& w,
                    double* dgamma_h) {
    const int dv = p.dv;
    w.o.assign(dv, 0.0);
    std::vector<double> ytmp(dv);
    one_row(p, b, h, i, w.a1, w.a2, w.o.data(), ytmp.data());
    const int64_t n = (int64_t)w.a1.size();
    const int64_t bh = (int64_t)b * p.H + h;
    const int64_t voff = bh * p.Nk * dv;
    const int64_t yoff = (bh * p.Nq + i) * dv;
    // GroupNorm statistics of this row (as in the forward).
    double mu = 0.0;
    for (int c = 0; c < dv; ++c) mu += w.o[c];
    mu /= dv;
    double var = 0.0;
    for (int c = 0; c < dv; ++c) var += (w.o[c] - mu) * (w.o[c] - mu);
    var /= dv;
    const double rstd = 1.0 / std::sqrt(var + p.eps);
    const double kappa = 1.0 - p.lambda_init;
    // Through the gain and scale, then through the normalisation.
    std::vector<double> gx(dv), xhat(dv);
    double mean_gx = 0.0, mean_gx_xhat = 0.0;
    for (int c = 0; c < dv; ++c) {
        const double gam = p.gamma ? p.gamma[(int64_t)h * dv + c] : 1.0;
        const double dyc = load_elem(dy, dy_type, yoff + c);
        xhat[c] = (w.o[c] - mu) * rstd;
        if (dgamma_h) dgamma_h[c] += kappa * dyc * xhat[c];
        gx[c] = kappa * gam * dyc;
        mean_gx += gx[c];
        mean_gx_xhat += gx[c] * xhat[c];
    }
    mean_gx /= dv;
    mean_gx_xhat /= dv;
    w.dout.assign(dv, 0.0);
    for (int c = 0; c < dv; ++c) w.dout[c] = rstd * (gx[c] - mean_gx - xhat[c] * mean_gx_xhat);
    // Through the product with V: dp_j = do . v_j is the gradient reaching
    // both maps (with weight 1 and -lambda).
    w.dp.assign(n, 0.0);
    for (int64_t j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dv; ++c) acc += w.dout[c] * load_elem(p.v, p.type, voff + j * dv + c);
        w.dp[j] = acc;
    }
    // Through each softmax.
    double dot1 = 0.0, dot2 = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        dot1 += w.a1[j] * w.dp[j];
        dot2 += w.a2[j] * (-p.lambda * w.dp[j]);
    }
    w.ds1.assign(n, 0.0);
    w.ds2.assign(n, 0.0);
    double dlam = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        w.ds1[j] = w.a1[j] * (w.dp[j] - dot1);
        w.ds2[j] = w.a2[j] * (-p.lambda * w.dp[j] - dot2);
        dlam -= w.a2[j] * w.dp[j];
    }
    return dlam;
}

int check(const Problem& p) {
    if (!p.q1 || !p.k1 || !p.q2 || !p.k2 || !p.v) return 1;
    if (p.B < 0 || p.H < 0 || p.Nq < 0 || p.Nk < 1 || p.d < 1 || p.dv < 1) return 1;
    if (p.type < IN_F64 || p.type > IN_BF16) return 1;
    if (p.causal && p.Nq > p.Nk) return 1;
    return 0;
}

template <class F>
void parallel_for(int64_t n, int threads, F f) {
    if (threads <= 0) threads = (int)std::max(1u, std::thread::hardware_concurrency());
    threads = (int)std::min<int64_t>(threads, std::max<int64_t>(n, 1));
    std::atomic<int64_t> next{0};
    auto worker = [&]() {
        for (;;) {
            int64_t k = next.fetch_add(1);
            if (k >= n) break;
            f(k);
        }
    };
    std::vector<std::thread> pool;
    for (int t = 1; t < threads; ++t) pool.emplace_back(worker);
    worker();
    for (auto& t : pool) t.join();
}

}  // namespace

extern "C" {

// Rows of the forward pass.  Inputs are BHND contiguous: q1,q2 [B,H,Nq,d];
// k1,k2 [B,H,Nk,d]; v [B,H,Nk,dv].  When `rows` is null every query row is
// computed and the outputs are [B,H,Nq,dv]; otherwise the same n_rows query
// indices are computed for every (b,h) and the outputs are [B,H,n_rows,dv].
// o_pre receives (A1 - lambda A2) V, y the normalised and scaled output;
// either may be null.  Returns 0, or 1 on an invalid argument.
int oracle_diffattn_fwd(const void* q1, const void* k1, const void* q2, const void* k2,
                        const void* v, int in_type, double lambda, double lambda_init,
                        int causal, int B, int H, int Nq, int Nk, int d, int dv,
                        const double* gamma, double eps, const int64_t* rows, int64_t n_rows,
                        double* o_pre, double* y, int threads) {
    Problem p{q1, k1, q2, k2, v, in_type, lambda, lambda_init, causal, B, H, Nq, Nk, d, dv, gamma, eps};
    if (check(p)) return 1;
    const int64_t R = rows ? n_rows : (int64_t)Nq;
    if (rows) {
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= Nq) return 1;
    }
    const int64_t items = (int64_t)B * H * R;
    parallel_for(items, threads, [&](int64_t k) {
        thread_local std::vector<double> a1, a2, op, yy;
        op.resize(dv);
        yy.resize(dv);
        const int64_t r = k % R;
        const int64_t bh = k / R;
        const int b = (int)(bh / H), h = (int)(bh % H);
        const int64_t i = rows ? rows[r] : r;
        one_row(p, b, h, i, a1, a2, op.data(), yy.data());
        if (o_pre) std::memcpy(o_pre + k * dv, op.data(), sizeof(double) * dv);
        if (y) std::memcpy(y + k * dv, yy.data(), sizeof(double) * dv);
    });
    return 0;
}

// The two attention maps materialised in full, for small problems:
// a1, a2 are [B,H,Nq,Nk]; masked entries are 0.
int oracle_diffattn_maps(const void* q1, const void* k1, const void* q2, const void* k2,
                         int in_type, int causal, int B, int H, int Nq, int Nk, int d,
                         double* a1_out, double* a2_out) {
    // V is not used for the maps; a valid pointer keeps the shared check simple.
    Problem p{q1, k1, q2, k2, q1, in_type, 0.0, 0.0, causal, B, H, Nq, Nk, d, 1, nullptr, 0.0};
    if (check(p) || !a1_out || !a2_out) return 1;
    std::vector<double> a1, a2;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (int64_t i = 0; i < Nq; ++i) {
                attention_rows(p, b, h, i, a1, a2);
                const int64_t n = (int64_t)a1.size();
                const int64_t row = (((int64_t)b * H + h) * Nq + i) * Nk;
                for (int64_t j = 0; j < Nk; ++j) {
                    a1_out[row + j] = j < n ? a1[j] : 0.0;
                    a2_out[row + j] = j < n ? a2[j] : 0.0;
                }
            }
    return 0;
}

// Gradients of the loss sum(dy * y) with respect to every input of the
// forward pass.  dy is [B,H,Nq,dv] of type dy_type.  Outputs (fp64):
//  * dq1, dq2 [B,H,R,d] for the query rows `rows` (R = n_rows; all rows, in
//    order, when rows is null);
//  * dk1, dk2 [B,H,K,d] and dv [B,H,K,dv] for the keys `keys` (K = n_keys;
//    all keys when keys is null);
//  * dlambda (one value) and dgamma [H*dv], which sum over every row: they
//    may be non-null only when rows and keys are both null;
//  * dlambda_rss (one value, same condition): the root-sum-square of the
//    per-row terms of dlambda, the scale of its rounding error (the terms
//    cancel, so the sum itself can be much smaller than its terms).
// Any output may be null.  Only the query rows that are requested, or that
// see a requested key, are visited.  Returns 0, or 1 on an invalid argument.
int oracle_diffattn_bwd(const void* q1, const void* k1, const void* q2, const void* k2,
                        const void* v, int in_type, const void* dy, int dy_type,
                        double lambda, double lambda_init, int causal,
                        int B, int H, int Nq, int Nk, int d, int dv,
                        const double* gamma, double eps,
                        const int64_t* rows, int64_t n_rows, const int64_t* keys, int64_t n_keys,
                        double* dq1, double* dq2, double* dk1, double* dk2, double* dv_out,
                        double* dlambda, double* dgamma, double* dlambda_rss, int threads) {
    Problem p{q1, k1, q2, k2, v, in_type, lambda, lambda_init, causal, B, H, Nq, Nk, d, dv, gamma, eps};
    if (check(p) || !dy || dy_type < IN_F64 || dy_type > IN_BF16) return 1;
    if ((rows || keys) && (dlambda || dgamma || dlambda_rss)) return 1;
    const int64_t R = rows ? n_rows : (int64_t)Nq;
    const int64_t K = keys ? n_keys : (int64_t)Nk;
    // Position of each query row / key in the outputs (-1: not requested).
    std::vector<int64_t> row_slot(Nq, -1), key_slot(Nk, -1);
    for (int64_t r = 0; r < R; ++r) {
        const int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= Nq) return 1;
        row_slot[i] = r;
    }
    int64_t min_key = Nk;
    for (int64_t t = 0; t < K; ++t) {
        const int64_t j = keys ? keys[t] : t;
        if (j < 0 || j >= Nk) return 1;
        key_slot[j] = t;
        min_key = std::min(min_key, j);
    }
    const double inv_sqrt_d = 1.0 / std::sqrt((double)d);
    const int64_t BH = (int64_t)B * H;
    std::vector<double> dlam_bh(BH, 0.0), dlam_sq_bh(BH, 0.0), dgam_bh(dgamma ? BH * dv : 0, 0.0);
    if (dq1) std::fill(dq1, dq1 + BH * R * d, 0.0);
    if (dq2) std::fill(dq2, dq2 + BH * R * d, 0.0);
    if (dk1) std::fill(dk1, dk1 + BH * K * d, 0.0);
    if (dk2) std::fill(dk2, dk2 + BH * K * d, 0.0);
    if (dv_out) std::fill(dv_out, dv_out + BH * K * dv, 0.0);
    // One task per (b, h): it owns that head's slices of every output.
    parallel_for(BH, threads, [&](int64_t bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        RowGrad w;
        const int64_t qbase = bh * Nq * d, kbase = bh * Nk * d;
        for (int64_t i = 0; i < Nq; ++i) {
            const bool want_row = row_slot[i] >= 0;
            const bool sees_key = visible_keys(p, i) > min_key;
            if (!want_row && !sees_key && !dlambda && !dgamma && !dlambda_rss) continue;
            const double term = row_backward(p, dy, dy_type, b, h, i, w, dgamma ? &dgam_bh[bh * dv] : nullptr);
            dlam_bh[bh] += term;
            dlam_sq_bh[bh] += term * term;
            const int64_t n = (int64_t)w.ds1.size();
            if (want_row) {
                const int64_t o = (bh * R + row_slot[i]) * d;
                for (int64_t j = 0; j < n; ++j)
                    for (int c = 0; c < d; ++c) {
                        if (dq1) dq1[o + c] += w.ds1[j] * load_elem(k1, in_type, kbase + j * d + c) * inv_sqrt_d;
                        if (dq2) dq2[o + c] += w.ds2[j] * load_elem(k2, in_type, kbase + j * d + c) * inv_sqrt_d;
                    }
            }
            for (int64_t j = 0; j < n; ++j) {
                const int64_t t = key_slot[j];
                if (t < 0) continue;
                const int64_t ok = (bh * K + t) * d, ov = (bh * K + t) * dv;
                for (int c = 0; c < d; ++c) {
                    if (dk1) dk1[ok + c] += w.ds1[j] * load_elem(q1, in_type, qbase + i * d + c) * inv_sqrt_d;
                    if (dk2) dk2[ok + c] += w.ds2[j] * load_elem(q2, in_type, qbase + i * d + c) * inv_sqrt_d;
                }
                if (dv_out) {
                    const double a = w.a1[j] - lambda * w.a2[j];
                    for (int c = 0; c < dv; ++c) dv_out[ov + c] += a * w.dout[c];
                }
            }
        }
    });
    // Sums over heads in a fixed order.
    if (dlambda) {
        double s = 0.0;
        for (int64_t bh = 0; bh < BH; ++bh) s += dlam_bh[bh];
        *dlambda = s;
    }
    if (dlambda_rss) {
        double s = 0.0;
        for (int64_t bh = 0; bh < BH; ++bh) s += dlam_sq_bh[bh];
        *dlambda_rss = std::sqrt(s);
    }
    if (dgamma) {
        std::fill(dgamma, dgamma + (int64_t)H * dv, 0.0);
        for (int64_t bh = 0; bh < BH; ++bh)
            for (int c = 0; c < dv; ++c) dgamma[(bh % H) * dv + c] += dgam_bh[bh * dv + c];
    }
    return 0;
}

}  // extern "C"
