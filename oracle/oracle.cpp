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

}  // extern "C"
