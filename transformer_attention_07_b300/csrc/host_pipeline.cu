// Prefill with host-resident tensors (diffattn_fwd_host): the library's own
// staging of a host-to-host call.  The B*H heads are cut into chunks of whole
// heads; each chunk moves through three stages on three streams:
//   copy-in stream    q1, k1, q2, k2, v of the chunk, host -> device slot
//   compute streams   the prefill kernel on that slot, alternating between
//                     the caller's stream and a second one, so that a
//                     chunk's kernel starts filling SMs while the previous
//                     chunk's last CTAs are still running
//   copy-out stream   the chunk's output, device slot -> host
// A ring of device slots (in the caller's workspace) lets chunk i's copy-in
// overlap chunk i-1's kernel and chunk i-2's copy-out, so the transfers hide
// behind the computation except for the first copy-in and the last copy-out.
// Every head is computed by the same kernel as in diffattn_fwd, so the result
// equals the device-resident call bit for bit.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "../../include/diffattn.h"
#include "launch.h"

namespace {

constexpr int kSlots = 3;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct SlotLayout {
    size_t q, k, v, o;     // bytes of one tensor of the chunk
    size_t slot;           // bytes of one slot: q1, q2, k1, k2, v, out
};

SlotLayout slot_layout(int heads, int Nq, int Nk, int d, int dv) {
    SlotLayout s;
    s.q = align256((size_t)heads * Nq * d * 2);
    s.k = align256((size_t)heads * Nk * d * 2);
    s.v = align256((size_t)heads * Nk * dv * 2);
    s.o = align256((size_t)heads * Nq * dv * 2);
    s.slot = 2 * s.q + 2 * s.k + s.v + s.o;
    return s;
}

// Heads per chunk when the caller passes 0: about sixteen chunks per call
// (the first copy-in and the last copy-out are not hidden, so smaller chunks
// expose less; measured at causal 64K, 16 heads: one head per chunk 24.6 ms,
// two 25.1 ms, eight 31.3 ms per call), never across a batch boundary (a
// chunk is heads h0..h0+c-1 of one batch entry).
int auto_chunk(int B, int H) {
    const int c = (int)(((int64_t)B * H + 15) / 16);
    return std::max(1, std::min(c, H));
}

int chunk_heads(int B, int H, int heads_per_chunk) {
    return heads_per_chunk > 0 ? std::min(heads_per_chunk, H) : auto_chunk(B, H);
}

// Streams and events of one call, released when the call returns (the
// runtime defers the release of objects whose work is still pending).
struct Pipeline {
    cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t loaded[kSlots] = {}, computed[kSlots] = {}, drained[kSlots] = {};
    bool ok = true;

    Pipeline() {
        ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&comp, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&end, cudaEventDisableTiming) == cudaSuccess;
        for (int s = 0; s < kSlots && ok; ++s)
            ok = cudaEventCreateWithFlags(&loaded[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&computed[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&drained[s], cudaEventDisableTiming) == cudaSuccess;
    }
    ~Pipeline() {
        for (int s = 0; s < kSlots; ++s) {
            if (loaded[s]) cudaEventDestroy(loaded[s]);
            if (computed[s]) cudaEventDestroy(computed[s]);
            if (drained[s]) cudaEventDestroy(drained[s]);
        }
        if (start) cudaEventDestroy(start);
        if (end) cudaEventDestroy(end);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
        if (comp) cudaStreamDestroy(comp);
    }
};

}  // namespace

extern "C" {

size_t diffattn_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d, int dv, int heads_per_chunk) {
    if (B < 0 || H < 1 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || heads_per_chunk < 0) return 0;
    return kSlots * slot_layout(chunk_heads(B, H, heads_per_chunk), Nq, Nk, d, dv).slot;
}

int diffattn_fwd_host(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                      float lambda, float lambda_init, int causal, int B, int H, int Nq, int Nk, int d, int dv,
                      const float* gn_gamma, float eps, void* out, int heads_per_chunk, void* workspace,
                      size_t workspace_bytes, void* stream) {
    if (!q1 || !k1 || !q2 || !k2 || !v || !out) return DIFFATTN_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 1 || d < 1 || dv < 1 || heads_per_chunk < 0) return DIFFATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return DIFFATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk) return DIFFATTN_ERR_INVALID_ARG;
    if (!std::isfinite(lambda) || !std::isfinite(lambda_init) || !(eps >= 0.0f) || !std::isfinite(eps))
        return DIFFATTN_ERR_INVALID_ARG;
    if (!((d == 64 && dv == 128) || (d == 32 && dv == 64))) return DIFFATTN_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(gn_gamma) & 3u) != 0) return DIFFATTN_ERR_INVALID_ARG;
    if (H > 65535 || (int64_t)H * Nk * dv * 2 >= (int64_t(1) << 40)) return DIFFATTN_ERR_INVALID_ARG;
    if ((int64_t)B * H * Nq == 0) return DIFFATTN_OK;
    const int c = chunk_heads(B, H, heads_per_chunk);
    const SlotLayout L = slot_layout(c, Nq, Nk, d, dv);
    if (!workspace || workspace_bytes < kSlots * L.slot) return DIFFATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DIFFATTN_ERR_INVALID_ARG;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    Pipeline pl;
    if (!pl.ok) return DIFFATTN_ERR_CUDA;
    // The copies start after the caller's earlier work on its stream.
    if (cudaEventRecord(pl.start, cs) != cudaSuccess || cudaStreamWaitEvent(pl.in, pl.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pl.out, pl.start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(pl.comp, pl.start, 0) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;

    const size_t qh = (size_t)Nq * d * 2, kh = (size_t)Nk * d * 2, vh = (size_t)Nk * dv * 2, oh = (size_t)Nq * dv * 2;
    auto host = [](const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; };
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int idx = 0;
    for (int b = 0; b < B; ++b) {
        for (int h0 = 0; h0 < H; h0 += c, ++idx) {
            const int hc = std::min(c, H - h0);
            const int s = idx % kSlots;
            const size_t head = (size_t)b * H + h0;
            uint8_t* base = ws + (size_t)s * L.slot;
            uint8_t *dq1 = base, *dq2 = base + L.q, *dk1 = base + 2 * L.q, *dk2 = dk1 + L.k, *dvs = dk2 + L.k,
                    *dout = dvs + L.v;
            // Copy-in: the slot's inputs were last read by the kernel of chunk idx - kSlots.
            bool ok = idx < kSlots || cudaStreamWaitEvent(pl.in, pl.computed[s], 0) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(dq1, host(q1, head * qh), hc * qh, cudaMemcpyHostToDevice, pl.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(dk1, host(k1, head * kh), hc * kh, cudaMemcpyHostToDevice, pl.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(dq2, host(q2, head * qh), hc * qh, cudaMemcpyHostToDevice, pl.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(dk2, host(k2, head * kh), hc * kh, cudaMemcpyHostToDevice, pl.in) == cudaSuccess;
            ok = ok && cudaMemcpyAsync(dvs, host(v, head * vh), hc * vh, cudaMemcpyHostToDevice, pl.in) == cudaSuccess;
            ok = ok && cudaEventRecord(pl.loaded[s], pl.in) == cudaSuccess;
            // Kernel: after the inputs landed and the slot's previous output
            // left; even chunks on the caller's stream, odd ones on the second.
            cudaStream_t ks = (idx & 1) ? pl.comp : cs;
            ok = ok && cudaStreamWaitEvent(ks, pl.loaded[s], 0) == cudaSuccess;
            ok = ok && (idx < kSlots || cudaStreamWaitEvent(ks, pl.drained[s], 0) == cudaSuccess);
            if (!ok) return DIFFATTN_ERR_CUDA;
            diffattn::PrefillArgs a{dq1, dk1, dq2, dk2, dvs, lambda, lambda_init, eps, causal, 1, hc, Nq, Nk, d, dv,
                                    gn_gamma ? gn_gamma + (size_t)h0 * dv : nullptr, dout, nullptr, nullptr,
                                    nullptr, nullptr};
            const int rc = diffattn::launch_prefill(a, ks);
            if (rc != diffattn::LAUNCH_OK) return rc == diffattn::LAUNCH_ERR_UNSUPPORTED ? DIFFATTN_ERR_UNSUPPORTED
                                                                                         : DIFFATTN_ERR_CUDA;
            // Copy-out.
            ok = cudaEventRecord(pl.computed[s], ks) == cudaSuccess &&
                 cudaStreamWaitEvent(pl.out, pl.computed[s], 0) == cudaSuccess &&
                 cudaMemcpyAsync(static_cast<uint8_t*>(out) + head * oh, dout, hc * oh, cudaMemcpyDeviceToHost,
                                 pl.out) == cudaSuccess &&
                 cudaEventRecord(pl.drained[s], pl.out) == cudaSuccess;
            if (!ok) return DIFFATTN_ERR_CUDA;
        }
    }
    // The caller's stream completes only after the last output has reached
    // the host (the copy-out stream waited for every kernel, on both compute
    // streams).
    if (cudaEventRecord(pl.end, pl.out) != cudaSuccess || cudaStreamWaitEvent(cs, pl.end, 0) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    return DIFFATTN_OK;
}

}  // extern "C"
