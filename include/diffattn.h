/*
 * diffattn.h — C ABI of the B300 (sm_103a) differential-attention forward and backward.
 *
 * The operation (Differential Transformer pages):
 *   "How does Differential Attention work to suppress noise and improve
 *   long-context focus?" (iloveeagents.com), section "Mathematical Formula":
 *       DiffAttn(Q,K,V) = ( softmax(Q1 K1^T / sqrt d) - lambda * softmax(Q2 K2^T / sqrt d) ) V
 *   "Differential Transformer: How Noise-Canceling Attention Reinvents LLMs"
 *   (llmbytes.dev), section "How Differential Attention Cancels Common-Mode
 *   Noise", steps 2-4: two independent softmax maps, the lambda-weighted
 *   subtraction, then GroupNorm of the multi-head output and a
 *   (1 - lambda_init) scale.
 *
 * Readings fixed by this interface where the pages are silent:
 *   - the logit scale is 1/sqrt(d), d = the Q/K head width;
 *   - causal masking (optional) applies the same mask to both maps and is
 *     bottom-right aligned: key j is visible to query i iff j <= i + Nk - Nq;
 *   - GroupNorm: one group per head, statistics per token over that head's
 *     dv channels, biased variance, eps inside the square root, per-channel
 *     gain gamma[h*dv + c], no bias; the result is multiplied by
 *     (1 - lambda_init).  lambda only weights the subtraction.
 *
 * Conventions shared by every entry point:
 *   - Tensors are device pointers, bf16 stored as 16-bit words, BHND row-major
 *     and contiguous ([B][H][N][width], last dimension fastest), each 16-byte
 *     aligned.  The caller owns all memory; the library never allocates device
 *     memory and keeps no per-call state.
 *   - Supported head widths: (d, dv) = (64, 128) or (32, 64).
 *   - Arguments are validated on the host before anything is launched; on any
 *     error nothing is launched and nothing is written.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream).  No entry point synchronises.
 *   - A launch failure reported by the CUDA runtime returns DIFFATTN_ERR_CUDA.
 *     Device-side waits are bounded: a wait that runs out records a code that
 *     diffattn_last_device_error() returns, and the kernel exits.
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, bad eps/lambda */
    DIFFATTN_ERR_UNSUPPORTED = 2, /* (d, dv) pair without a compiled kernel */
    DIFFATTN_ERR_CUDA = 3,        /* the CUDA runtime reported an error at launch */
    DIFFATTN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
    DIFFATTN_ERR_TIMEOUT = 5      /* a device-side wait ran out (see diffattn_last_device_error) */
} diffattn_status;

/*
 * Prefill forward: y = (1 - lambda_init) * GroupNorm_h( (A1 - lambda A2) V ).
 *   q1, q2      [B,H,Nq,d]  bf16
 *   k1, k2      [B,H,Nk,d]  bf16
 *   v           [B,H,Nk,dv] bf16
 *   lambda      weight of the second map in the subtraction (any finite value)
 *   lambda_init output scale is (1 - lambda_init) (any finite value)
 *   causal      0 or 1; with 1, Nq <= Nk is required
 *   gn_gamma    [H*dv] fp32 per-channel gain, or NULL for all ones
 *   eps         GroupNorm epsilon, >= 0
 *   out         [B,H,Nq,dv] bf16 result (round to nearest even)
 * B, H or Nq equal to 0 is a valid empty problem (returns DIFFATTN_OK, no launch);
 * Nk must be >= 1.
 */
int diffattn_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                 float lambda, float lambda_init, int causal,
                 int B, int H, int Nq, int Nk, int d, int dv,
                 const float* gn_gamma, float eps, void* out, void* stream);

/*
 * As diffattn_fwd, and additionally writes the pre-norm output
 * (A1 - lambda A2) V in fp32 to o_prenorm ([B,H,Nq,dv]) when it is not NULL.
 */
int diffattn_fwd_ex(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                    float lambda, float lambda_init, int causal,
                    int B, int H, int Nq, int Nk, int d, int dv,
                    const float* gn_gamma, float eps, void* out, float* o_prenorm, void* stream);

/*
 * How diffattn_fwd, diffattn_fwd_ex, diffattn_fwd_train and diffattn_fwd_fp8
 * (fp8 = 1) launch the prefill for a shape on a device with `sms` streaming
 * multiprocessors (148 on a B300).  The operation is the one diffattn_fwd
 * computes (iloveeagents.com Q&A, "Mathematical Formula"); how its query
 * tiles of 128 rows are spread over the GPU is this library's own.  Pure
 * host arithmetic, no CUDA call; every form gives the same bits.
 *   *form  DIFFATTN_PLAN_TILE_GRID (0): one CTA per query tile, grid (tile, h, b)
 *          DIFFATTN_PLAN_TILE_GROUPED (1): one CTA per query tile, a 1-D grid
 *            in weight order within groups of heads (causal, K and V of at
 *            least four heads fit in 16 MB)
 *          DIFFATTN_PLAN_PERSISTENT (2): one CTA per SM walking a (b, h)-major
 *            tile list (more tiles than SMs, Nk <= 4096)
 *          DIFFATTN_PLAN_PERSISTENT_WEIGHT (3): the same over a weight-major
 *            list (causal, all heads' K and V within 64 MB; Nk <= 8192)
 *   *ctas  CTAs launched (0 for an empty problem)
 * Returns DIFFATTN_ERR_INVALID_ARG for bad sizes, sms < 1 or null outputs,
 * DIFFATTN_ERR_UNSUPPORTED for a (d, dv) pair without a kernel.
 */
enum {
    DIFFATTN_PLAN_TILE_GRID = 0,
    DIFFATTN_PLAN_TILE_GROUPED = 1,
    DIFFATTN_PLAN_PERSISTENT = 2,
    DIFFATTN_PLAN_PERSISTENT_WEIGHT = 3
};
int diffattn_prefill_plan(int B, int H, int Nq, int Nk, int d, int dv, int causal, int fp8, int sms, int* form,
                          long long* ctas);

/*
 * Prefill forward with 8-bit queries and keys.  The pages link differential
 * attention to low-bit quantisation through its smaller activation outliers
 * (llmbytes.dev, "Quantization Friendliness").  Here q1, k1, q2, k2 are
 * stored as fp8 e4m3 bytes [B,H,N,d] (16-byte aligned), and each
 * (tensor, head) has a dequantisation scale:
 *   qk_scale    [4*H] fp32, device: rows sq1, sk1, sq2, sk2, each H long,
 *               so q_r = sq_r[h] * q8_r and k_r = sk_r[h] * k8_r
 * The logits are s_r = sq_r[h] sk_r[h] (q8_r . k8_r) / sqrt(d), computed by
 * the 8-bit tensor-core product with fp32 accumulation.  V, P, the output
 * and everything after the scores are as in diffattn_fwd_ex.  The scales are
 * read on the device, so the host cannot check them; they must be finite.
 */
int diffattn_fwd_fp8(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                     const float* qk_scale, float lambda, float lambda_init, int causal,
                     int B, int H, int Nq, int Nk, int d, int dv,
                     const float* gn_gamma, float eps, void* out, float* o_prenorm, void* stream);

/*
 * Prefill with host-resident tensors: the same operation as diffattn_fwd, with
 * q1, k1, q2, k2, v and out in HOST memory (BHND bf16; page-locked memory
 * lets the copies overlap the computation, pageable memory works but
 * serialises them).  gn_gamma, if given, is a device pointer as elsewhere.
 * The B*H heads are processed in chunks of heads_per_chunk heads of one
 * batch entry (0 = about sixteen chunks per call): each chunk's inputs are
 * copied to a device slot on an internal stream, the prefill kernel runs on
 * `stream`, and the chunk's output is copied back on a second internal
 * stream, with three slots in flight.
 *   workspace   device memory of >= diffattn_fwd_host_workspace_bytes(...)
 *               bytes, 256-byte aligned (the slots)
 * The call only enqueues work.  `out` is complete when `stream` has
 * completed.  The result equals diffattn_fwd's bit for bit.
 */
size_t diffattn_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d, int dv, int heads_per_chunk);
int diffattn_fwd_host(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                      float lambda, float lambda_init, int causal,
                      int B, int H, int Nq, int Nk, int d, int dv,
                      const float* gn_gamma, float eps, void* out, int heads_per_chunk,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Training forward: diffattn_fwd_ex plus what the backward pass reads.
 *   o_prenorm   [B,H,Nq,dv] fp32, required: (A1 - lambda A2) V
 *   o2          [B,H,Nq,dv] fp32, required, 16-byte aligned: A2 V
 *   lse         [2,B,H,Nq] fp32, required, 4-byte aligned: for map r and row
 *               i, log sum_j exp(q_r,i . k_r,j / sqrt d) over the visible keys
 *               (natural log); map 1 first
 * Other arguments, checks and statuses as diffattn_fwd.
 */
int diffattn_fwd_train(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                       float lambda, float lambda_init, int causal,
                       int B, int H, int Nq, int Nk, int d, int dv,
                       const float* gn_gamma, float eps, void* out,
                       float* o_prenorm, float* o2, float* lse, void* stream);

/*
 * Bytes of device workspace diffattn_bwd needs (0 for invalid sizes).
 */
size_t diffattn_bwd_workspace_bytes(int B, int H, int Nq, int dv);

/*
 * Backward pass: the gradients of a loss L with respect to every input of
 * the forward pass, given dy = dL/dy.  lambda is learnable on the pages (the
 * iloveeagents.com Q&A, "Mathematical Formula"), so dL/dlambda is returned
 * with the GroupNorm gain's gradient and the five input gradients:
 *   do      = GroupNorm backward of dy (per row, through gamma and (1 - lambda_init))
 *   dS1     = A1 o (do V^T - rowsum(A1 o do V^T)),  dS2 = -lambda A2 o (do V^T - rowsum(...))
 *   dq_r    = dS_r k_r / sqrt d,   dk_r = dS_r^T q_r / sqrt d,   dv = (A1 - lambda A2)^T do
 *   dlambda = -sum do . (A2 V),    dgamma = (1 - lambda_init) sum_rows dy o xhat
 * Inputs: q1, k1, q2, k2, v, lambda, lambda_init, causal, gn_gamma, eps as in
 *   the forward call; dy [B,H,Nq,dv] bf16; o_prenorm, o2, lse as written by
 *   diffattn_fwd_train for those inputs.
 * Outputs (bf16, the inputs' shapes): dq1, dq2 [B,H,Nq,d]; dk1, dk2 [B,H,Nk,d];
 *   dv_grad [B,H,Nk,dv].  dlambda (one float) and dgamma ([H*dv] fp32) may be
 *   NULL when not wanted; dlambda sums over every (b, h, i).
 * workspace: >= diffattn_bwd_workspace_bytes(B, H, Nq, dv) bytes, 256-byte
 *   aligned, no initialisation needed; concurrent calls need separate ones.
 * Supported widths: (d, dv) = (64, 128) or (32, 64), as for the forward.  Nq = 0 writes zero key gradients (the
 * query-side pointers may then be NULL).  Results are
 * deterministic: no atomics, fixed summation orders.
 */
int diffattn_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                 const void* dy, const float* o_prenorm, const float* o2, const float* lse,
                 float lambda, float lambda_init, int causal,
                 int B, int H, int Nq, int Nk, int d, int dv,
                 const float* gn_gamma, float eps,
                 void* dq1, void* dk1, void* dq2, void* dk2, void* dv_grad,
                 float* dlambda, float* dgamma,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Standard softmax attention, the single-map baseline the pages compare
 * differential attention against ("Throughput and Hardware Realities",
 * llmbytes.dev, against FlashAttention; the operator is the standard
 * attention of the iloveeagents.com Q&A, "Detail"):
 *     out = softmax(Q K^T / sqrt(d)) V        (no lambda, no GroupNorm)
 *   q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,dv] bf16, (d, dv) = (128, 128):
 *   the width of one differential head's [q1; q2] and v, so that the two
 *   operators are compared at equal parameters.
 *   causal      0 or 1 (bottom-right aligned as above; Nq <= Nk)
 *   out         [B,H,Nq,dv] bf16;  out_f32: NULL or [B,H,Nq,dv] fp32
 * Same conventions and statuses as diffattn_fwd.
 */
int diffattn_standard_fwd(const void* q, const void* k, const void* v, int causal,
                          int B, int H, int Nq, int Nk, int d, int dv,
                          void* out, float* out_f32, void* stream);

/*
 * Bytes of device workspace diffattn_decode needs for this shape and split
 * count (num_splits = 0: enough for any split count the library chooses).
 * Returns 0 for invalid sizes.
 */
size_t diffattn_decode_workspace_bytes(int B, int H, int Nk, int dv, int num_splits);

/*
 * The key-range count diffattn_decode, diffattn_decode_paged (with Nk =
 * max_pages * page_size) and diffattn_decode_noalloc use when num_splits = 0,
 * for a device with `sms` streaming multiprocessors (148 on a B300).  Pure
 * host arithmetic, no CUDA call:
 *   * it minimises a cost model of the split kernel: each wave of CTAs costs a
 *     fixed start-up worth about 128 KB of streaming, plus its largest key
 *     range streamed at the per-SM share of HBM bandwidth (up to 1.3 times
 *     that share when the wave leaves SMs idle);
 *   * ranges are whole 32-key chunks, none empty, at least 256 keys;
 *   * max_splits caps the count (0 = the default cap of 32; at most 64);
 *     the no-alloc entry point passes what its scratch holds.
 * Returns 0 for invalid arguments or unsupported widths.
 */
int diffattn_decode_auto_splits(int B, int H, int Nk, int d, int dv, int sms, int max_splits);

/*
 * Split-KV decode: one query per (b, h) against a key/value cache of Nk rows,
 * no mask (the same operation as diffattn_fwd with Nq = 1, causal = 0).
 *   q1, q2      [B,H,1,d] bf16;  k1, k2 [B,H,Nk,d] bf16;  v [B,H,Nk,dv] bf16
 *   num_splits  0 = chosen by the library, else 1..64 key ranges per (b, h)
 *   workspace   device scratch of >= diffattn_decode_workspace_bytes(...) bytes,
 *               16-byte aligned; holds per-split partial softmax states.  It
 *               needs no initialisation; concurrent calls need separate
 *               workspaces.
 *   out         [B,H,1,dv] bf16;  o_prenorm: NULL or [B,H,1,dv] fp32
 * The key range of each (b, h) is cut into num_splits pieces; each piece
 * yields the running maximum, normaliser and unnormalised output of both maps,
 * and a second kernel merges the pieces (the associativity of the online
 * softmax), forms O1/L1 - lambda O2/L2 and applies the GroupNorm and scale.
 */
int diffattn_decode(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                    float lambda, float lambda_init, int B, int H, int Nk, int d, int dv,
                    const float* gn_gamma, float eps, int num_splits,
                    void* workspace, size_t workspace_bytes,
                    void* out, float* o_prenorm, void* stream);

/*
 * Paged split-KV decode with per-sequence lengths: the computation of
 * diffattn_decode (one query per (b, h), no mask) over key/value caches kept
 * in pages, as a serving system stores them.
 *   k1_pages, k2_pages [num_pages, H, page_size, d] bf16;
 *   v_pages            [num_pages, H, page_size, dv] bf16:
 *                      page p holds page_size consecutive keys of every head.
 *   block_table        [B, max_pages] int32 (device): the pages of sequence b,
 *                      in key order; entries past the sequence are ignored.
 *   seq_lens           [B] int32 (device): keys of sequence b, in
 *                      [1, max_pages * page_size].
 *   page_size          a multiple of 32.
 *   q1, q2 [B,H,1,d]; out [B,H,1,dv] bf16; o_prenorm NULL or fp32 [B,H,1,dv];
 *   num_splits, workspace, workspace_bytes: as diffattn_decode, sized with
 *   diffattn_decode_workspace_bytes(B, H, max_pages * page_size, dv, num_splits).
 * Table entries and lengths live on the device, so the host cannot check
 * them: a page index outside [0, num_pages) or a length outside the range is
 * clamped, never dereferenced, and reported by diffattn_last_device_error()
 * (0x301 page, 0x302 length).  The pages one key range spans are staged in
 * shared memory: a split count for which one range would span more than 1024
 * pages is refused (DIFFATTN_ERR_INVALID_ARG; num_splits = 0 avoids it).
 */
int diffattn_decode_paged(const void* q1, const void* q2, const void* k1_pages, const void* k2_pages,
                          const void* v_pages, const int32_t* block_table, const int32_t* seq_lens,
                          int max_pages, int page_size, int num_pages,
                          float lambda, float lambda_init, int B, int H, int d, int dv,
                          const float* gn_gamma, float eps, int num_splits,
                          void* workspace, size_t workspace_bytes,
                          void* out, float* o_prenorm, void* stream);

/*
 * Split-KV decode over key ranges held by different GPUs (sequence sharding
 * for caches longer than one GPU holds).  Each GPU computes the partial
 * softmax states of its own range; the states of all ranges are gathered
 * (e.g. an all-gather over the GPUs) and merged.  The merge is the
 * associativity of the online softmax, the same algebra that combines the
 * key ranges of one GPU in diffattn_decode.
 *
 * diffattn_decode_partials: q1, q2 [B,H,1,d]; k1, k2 [B,H,Nk,d]; v [B,H,Nk,dv]
 *   (this GPU's Nk keys) bf16.  Writes to `partials` (fp32, 16-byte aligned,
 *   >= diffattn_decode_partials_bytes(B, H, dv, num_splits) bytes) the states
 *   [B*H][num_splits][2 maps][dv + 4]: m (running max of the scaled logits, in
 *   log2 units: logit * log2(e)), l (sum of 2^(logit*log2(e) - m)), two unused
 *   words, then the dv-wide unnormalised output.  A range with no keys has
 *   m = -inf, l = 0.  num_splits (1..64) must be the same on every GPU.
 * diffattn_decode_merge: `partials` holds num_parts such blocks back to back
 *   ([num_parts][B*H][num_splits][2][dv + 4], the layout of an all-gather);
 *   writes out [B,H,1,dv] bf16 (and o_prenorm, if given) exactly as
 *   diffattn_decode.  num_parts * num_splits <= 4096.
 */
size_t diffattn_decode_partials_bytes(int B, int H, int dv, int num_splits);
int diffattn_decode_partials(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                             int B, int H, int Nk, int d, int dv, int num_splits,
                             float* partials, size_t partials_bytes, void* stream);
int diffattn_decode_merge(const float* partials, int num_parts, int B, int H, int dv, int num_splits,
                          float lambda, float lambda_init, const float* gn_gamma, float eps,
                          void* out, float* o_prenorm, void* stream);

/*
 * Split-KV decode that allocates nothing: the same computation and arguments
 * as diffattn_decode, minus the workspace.  (The Differential Transformer
 * pages have no counterpart to this entry point; it exists for callers.)
 *
 * Who needs it: callers that cannot call cudaMalloc at the point of use —
 * for example a plugin or operator inside a serving framework that owns all
 * device memory through a pool planned ahead of time and forbids allocation
 * on the request path, or an interface that hands the operator only its
 * input and output pointers and no allocator.
 *
 * Scratch: the per-split partial softmax states go to one library-owned
 * device array of 8 MiB (8388608 bytes), a file-scope static that every GPU
 * which loads the library holds until the process exits.  A problem needs
 * B*H*splits*2*(dv + 4)*4 bytes of it.  With num_splits = 0 the split count
 * is chosen as diffattn_decode chooses it, but never above the largest count
 * that fits; DIFFATTN_ERR_WORKSPACE (nothing launched) is returned only when
 * a single key range per head, or the num_splits the caller fixed, needs more
 * than 8 MiB.  The arguments are checked before any CUDA runtime call.  No
 * call allocates or frees device memory (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address once (cudaGetSymbolAddress) and caches it; make
 * that first call before any stream capture.
 *
 * Sharing: every call uses the same array and it keeps the last call's
 * contents.  Nothing in it needs to start at zero: each call writes every
 * partial before reading it.  Calls whose kernels overlap on the GPU (two
 * streams, or two host threads) race on the array and corrupt each other's
 * results; serialise them.
 *
 * Returns the same statuses as diffattn_decode; DIFFATTN_ERR_CUDA also when
 * the scratch address cannot be obtained.
 */
int diffattn_decode_noalloc(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                            float lambda, float lambda_init, int B, int H, int Nk, int d, int dv,
                            const float* gn_gamma, float eps, int num_splits,
                            void* out, float* o_prenorm, void* stream);

/* Static description of a status code. */
const char* diffattn_status_string(int status);

/*
 * Reads and clears the device error word of the current device (synchronous:
 * it waits for `stream`).  0 = no device-side error; otherwise a code naming
 * the wait that ran out.  Returns -1 if the read itself failed.
 */
int diffattn_last_device_error(void* stream);

/*
 * Diagnostic for the failure path above: launches on `stream` a one-warp
 * kernel whose only thread waits, through the same bounded wait every kernel
 * uses, for an mbarrier phase that nothing completes.  After the wait limit
 * (2 s) the kernel records code 0x601 in the device error word and exits;
 * the CUDA context stays usable.  Returns DIFFATTN_OK when the launch was
 * accepted (the code is then read with diffattn_last_device_error), or
 * DIFFATTN_ERR_CUDA.  While the word is set, every bounded wait of the
 * library's kernels gives up at its first slow-path check (a failed wait
 * makes the rest of the grid stop early), so read the word, which clears it,
 * before launching other work.
 */
int diffattn_selftest_wait_timeout(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
