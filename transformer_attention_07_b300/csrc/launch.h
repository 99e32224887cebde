// Internal interface between the C ABI (argument checking) and the launchers
// (tensor maps, grids, kernels).  Not installed; the public header is
// include/diffattn.h.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

namespace diffattn {

enum LaunchStatus { LAUNCH_OK = 0, LAUNCH_ERR_CUDA = 1, LAUNCH_ERR_UNSUPPORTED = 2 };

// Paged decode: most pages one key range (split) may span; their indices are
// staged in shared memory.
constexpr int kDecodeMaxSplitPages = 1024;

struct PrefillArgs {
    const void *q1, *k1, *q2, *k2, *v;
    float lambda, lambda_init, eps;
    int causal, B, H, Nq, Nk, d, dv;
    const float* gamma;
    void* out;
    float* o_prenorm;
    float* o2;    // training outputs (null for inference)
    float* lse;
    const float* qk_scale;   // non-null: q1, k1, q2, k2 are e4m3 with these [4,H] per-head scales
};

struct DecodeArgs {
    const void *q1, *k1, *q2, *k2, *v;
    float lambda, lambda_init, eps;
    int B, H, Nk, d, dv;
    int splits, keys_per_split;
    const float* gamma;
    float* ws;
    void* out;
    float* o_prenorm;
    // Paged caches (block_table != nullptr): Nk is then max_pages * page_size.
    const int32_t* block_table;
    const int32_t* seq_lens;
    int max_pages, page_size, num_pages;
    bool partials_only;   // stop after the split kernel (the partials stay in ws)
};

// Merge of gathered decode partials: ws holds [parts][B*H][splits][2][dv + 4].
struct MergeArgs {
    const float* ws;
    int parts, B, H, splits, dv;
    float lambda, lambda_init, eps;
    const float* gamma;
    void* out;
    float* o_prenorm;
};
int launch_decode_merge(const MergeArgs& a, cudaStream_t st);

// With DIFFATTN_DEBUG set in the environment, a failing CUDA call is
// reported on stderr (call site and the runtime's error string).
bool cuda_ok(cudaError_t e, const char* what);

struct StandardArgs {
    const void *q, *k, *v;
    int causal, B, H, Nq, Nk, d, dv;
    void* out;
    float* out_f32;
};

struct BwdArgs {
    const void *q1, *k1, *q2, *k2, *v, *dy;
    const float *o, *o2, *lse;
    float lambda, lambda_init, eps;
    int causal, B, H, Nq, Nk, d, dv;
    const float* gamma;
    void *dq1, *dk1, *dq2, *dk2, *dv_grad;
    float *dlambda, *dgamma;
    void* ws;   // >= bwd_workspace_bytes(B, H, Nq, dv), 256-byte aligned
};

// Workspace of the backward pass: do (bf16), the per-row constants, and the
// dgamma / dlambda partial sums, each 256-byte aligned.
struct BwdWorkspace {
    size_t off_do, off_rowc, off_rowt, off_gpart, off_lpart, total;
    int Nq_pad, nchunk;
};
BwdWorkspace bwd_workspace_layout(int B, int H, int Nq, int dv);

// How the prefill is launched for a shape on a device with `sms` SMs (host
// arithmetic; the launcher uses exactly this).  form: 0 = one CTA per query
// tile on the (tile, h, b) grid, 1 = one CTA per query tile on a 1-D grid in
// weight order within head groups, 2 = persistent grid over a (b, h)-major
// tile list, 3 = persistent grid over a weight-major list.
struct PrefillPlan {
    int form;
    long long ctas;     // CTAs launched
    int weight_major;   // the persistent list's order (kernel parameter)
    int head_group;     // heads per group of form 1, else 0 (kernel parameter)
};
PrefillPlan prefill_plan(int B, int H, int Nq, int Nk, int d, int dv, bool causal, bool qk8, int sms);

int launch_prefill(const PrefillArgs& a, cudaStream_t st);
int launch_backward(const BwdArgs& a, cudaStream_t st);
int launch_standard(const StandardArgs& a, cudaStream_t st);
int launch_decode(const DecodeArgs& a, cudaStream_t st);
int read_and_clear_device_error(cudaStream_t st, int* value);
int launch_selftest_wait(cudaStream_t st);

// Capacity of the library-owned decode scratch (diffattn_decode_noalloc).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// Streaming multiprocessors of the current device, looked up once per device
// and cached; 0 if the runtime cannot say.
int sm_count();

// Device address and size of that scratch on the current device (looked up
// on the first call per device).
int decode_noalloc_scratch(void** ptr, size_t* bytes);

}  // namespace diffattn
