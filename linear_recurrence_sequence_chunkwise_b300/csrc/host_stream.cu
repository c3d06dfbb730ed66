// host_stream.cu -- chunkwise retention over host-resident Q/K/V/O: the sequence moves
// through the device in segments, with the copies of one segment overlapping the
// compute of its neighbours.  Host code only (copies, events, library calls); every
// arithmetic step runs in the kernels behind retention_chunkwise.
//
// The split is exact: eq.(7) of "Transformer取代者登場！…RetNet…（2）", section
// "Retention" 3), carries the state R from one chunk to the next, so a segment of whole
// chunks continues from the fp32 state the previous segment left on the device.
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
size_t esize(int dtype) { return dtype == RET_BF16 ? 2 : 4; }

struct Layout {
    size_t state, q, k, v, o;     // bytes of each part (rounded up)
    size_t total() const { return state + 2 * (q + k + v + o); }
};

Layout layout(int in_dtype, int out_dtype, int b, int H, int dk, int dv, int seg) {
    const size_t rows = (size_t)b * H * (size_t)seg;
    Layout L;
    L.state = round_up((size_t)b * H * dk * dv * sizeof(float));
    L.q = round_up(rows * dk * esize(in_dtype));
    L.k = L.q;
    L.v = round_up(rows * dv * esize(in_dtype));
    L.o = round_up(rows * dv * esize(out_dtype));
    return L;
}

bool valid_dtype(int d) { return d == RET_F32 || d == RET_BF16; }

int status_of(cudaError_t e) { return ret::record_cuda_status(e); }

// Every argument check of retention_chunkwise_host (host-side, no GPU access).  Returns
// RET_OK to proceed, kNoWork when b, H or N is zero, or the status to return.
constexpr int kNoWork = -1;
int check_args(const void* q, const void* k, const void* v, const void* o, int in_dtype,
               int out_dtype, int b, int H, int N, int dk, int dv, int chunk, const double* gamma,
               const float* state_in, const float* state_out, int seg_len, const void* workspace,
               size_t workspace_bytes) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (dk <= 0 || dv <= 0 || dk % 16 || dv % 16 || dk > 256 || dv > 512) return RET_ERR_UNSUPPORTED;
    if (chunk < 16 || chunk > 256 || chunk % 16 != 0 || N % chunk != 0) return RET_ERR_SHAPE;
    if (seg_len <= 0 || seg_len % chunk != 0 || N % seg_len != 0) return RET_ERR_SHAPE;
    if (H > ret::kMaxHeads) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0) return kNoWork;
    if (!gamma) return RET_ERR_NULL;
    for (int h = 0; h < H; ++h)
        if (!(gamma[h] >= 0.0 && gamma[h] <= 1.0)) return RET_ERR_UNSUPPORTED;
    if (N == 0) return kNoWork;
    if (!q || !k || !v || !o || !workspace) return RET_ERR_NULL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if ((mis & 15u) || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return RET_ERR_ALIGN;
    if ((state_in && (reinterpret_cast<uintptr_t>(state_in) & 15u)) ||
        (state_out && (reinterpret_cast<uintptr_t>(state_out) & 15u)))
        return RET_ERR_ALIGN;
    if (workspace_bytes < layout(in_dtype, out_dtype, b, H, dk, dv, seg_len).total())
        return RET_ERR_SHAPE;
    return RET_OK;
}

// Scratch of the no-allocation entry point: a file-scope device array, reserved when the
// library's module loads on a device, so calls need no workspace from the caller.
constexpr size_t kStaticScratchBytes = size_t(48) << 20;
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device, looked up once per device
// and context: after cudaDeviceReset the module loads again in a new context, possibly at
// another address, so a changed context triggers a new lookup.
cudaError_t static_scratch(void** out) {
    static std::mutex mu;
    static void* addr[ret::kMaxDevices] = {};
    static void* ctx[ret::kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= ret::kMaxDevices) return cudaErrorInvalidDevice;
    // cudaFree(0) makes the device's primary context current if no context is yet
    e = cudaFree(nullptr);
    if (e != cudaSuccess) return e;
    void* const cur = ret::current_context();
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || !cur || cur != ctx[dev]) {
        e = cudaGetSymbolAddress(&addr[dev], g_static_scratch);
        if (e != cudaSuccess) {
            addr[dev] = nullptr;
            ctx[dev] = nullptr;
            return e;
        }
        ctx[dev] = cur;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

namespace ret {

void* current_context() {
    using Fn = CUresult (*)(CUcontext*);
    static Fn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<Fn>(p);
        return static_cast<Fn>(nullptr);
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

}  // namespace ret

extern "C" {

size_t retention_chunkwise_host_workspace_bytes(ret_dtype in_dtype, ret_dtype out_dtype, int b,
                                                int H, int dk, int dv, int seg_len) {
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || b < 0 || H < 0 || dk < 0 || dv < 0 ||
        seg_len < 0)
        return 0;
    return layout(in_dtype, out_dtype, b, H, dk, dv, seg_len).total();
}

int retention_chunkwise_host(const void* q, const void* k, const void* v, void* o,
                             ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N, int dk,
                             int dv, int chunk, const double* gamma, const float* state_in,
                             float* state_out, int seg_len, void* workspace,
                             size_t workspace_bytes, void* stream, void* h2d_stream,
                             void* d2h_stream) {
    const int rc = check_args(q, k, v, o, in_dtype, out_dtype, b, H, N, dk, dv, chunk, gamma,
                              state_in, state_out, seg_len, workspace, workspace_bytes);
    if (rc == kNoWork)   // zero sizes; with no tokens retention_chunkwise hands the state over
        return (N == 0 && b > 0 && H > 0)
                   ? retention_chunkwise(nullptr, nullptr, nullptr, nullptr, in_dtype, out_dtype, b,
                                         H, 0, dk, dv, chunk, gamma, state_in, state_out, stream)
                   : RET_OK;
    if (rc != RET_OK) return rc;
    const Layout L = layout(in_dtype, out_dtype, b, H, dk, dv, seg_len);

    // ---- workspace: carried state, then two buffer sets (q, k, v, o) of one segment each
    uint8_t* base = static_cast<uint8_t*>(workspace);
    float* st = reinterpret_cast<float*>(base);
    uint8_t* qd[2];
    uint8_t* kd[2];
    uint8_t* vd[2];
    uint8_t* od[2];
    {
        uint8_t* p = base + L.state;
        for (int j = 0; j < 2; ++j) {
            qd[j] = p; p += L.q;
            kd[j] = p; p += L.k;
            vd[j] = p; p += L.v;
            od[j] = p; p += L.o;
        }
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t hs = static_cast<cudaStream_t>(h2d_stream);
    cudaStream_t ds = static_cast<cudaStream_t>(d2h_stream);
    const size_t ein = esize(in_dtype), eout = esize(out_dtype);
    const size_t rows = (size_t)b * H;
    const int nseg = N / seg_len;

    // events live for this call only; destroying a recorded event frees it once it completes
    cudaEvent_t ev_start, h2d_done[2], comp_done[2], d2h_done[2], join_h, join_d;
    cudaEvent_t* all[] = {&ev_start, &h2d_done[0], &h2d_done[1], &comp_done[0], &comp_done[1],
                          &d2h_done[0], &d2h_done[1], &join_h, &join_d};
    constexpr int kEvents = sizeof(all) / sizeof(all[0]);
    int made = 0;
    cudaError_t e = cudaSuccess;
    for (; made < kEvents && e == cudaSuccess; ++made)
        e = cudaEventCreateWithFlags(all[made], cudaEventDisableTiming);
    auto finish = [&](int rc) {
        for (int i = 0; i < made; ++i) cudaEventDestroy(*all[i]);
        return rc;
    };
    if (e != cudaSuccess) {
        --made;   // the failed one was not created
        return finish(status_of(e));
    }
    // An error after copies were queued: stream still waits for whatever the copy streams
    // hold, so that work already queued never outlives the ordering the header promises
    // (best effort: the calls below may fail too if the error came from the device).
    auto fail = [&](int rc) {
        if (cudaEventRecord(join_h, hs) == cudaSuccess) cudaStreamWaitEvent(cs, join_h, 0);
        if (cudaEventRecord(join_d, ds) == cudaSuccess) cudaStreamWaitEvent(cs, join_d, 0);
        return finish(rc);
    };
    // the copy streams start after the work already queued on the compute stream
    e = cudaEventRecord(ev_start, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ds, ev_start, 0);
    if (e != cudaSuccess) return fail(status_of(e));

    for (int s = 0; s < nseg; ++s) {
        const int j = s & 1;
        const size_t t0 = (size_t)s * seg_len;
        // host -> device: one 2-D copy per tensor (b*H rows of seg_len*d elements)
        if (s >= 2) e = cudaStreamWaitEvent(hs, comp_done[j], 0);   // buffer j read by s-2
        const void* srcs[3] = {q, k, v};
        uint8_t* dsts[3] = {qd[j], kd[j], vd[j]};
        const int widths[3] = {dk, dk, dv};
        for (int t = 0; t < 3 && e == cudaSuccess; ++t) {
            const size_t w = (size_t)seg_len * widths[t] * ein;
            const size_t pitch = (size_t)N * widths[t] * ein;
            e = cudaMemcpy2DAsync(dsts[t], w,
                                  static_cast<const uint8_t*>(srcs[t]) + t0 * widths[t] * ein, pitch,
                                  w, rows, cudaMemcpyHostToDevice, hs);
        }
        if (e == cudaSuccess) e = cudaEventRecord(h2d_done[j], hs);
        // compute, continuing from the state the previous segment left
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, h2d_done[j], 0);
        if (e == cudaSuccess && s >= 2) e = cudaStreamWaitEvent(cs, d2h_done[j], 0);
        if (e != cudaSuccess) return fail(status_of(e));
        const int rc = retention_chunkwise(qd[j], kd[j], vd[j], od[j], in_dtype, out_dtype, b, H,
                                           seg_len, dk, dv, chunk, gamma,
                                           s == 0 ? state_in : st, st, stream);
        if (rc != RET_OK) return fail(rc);
        e = cudaEventRecord(comp_done[j], cs);
        // device -> host
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ds, comp_done[j], 0);
        if (e == cudaSuccess) {
            const size_t w = (size_t)seg_len * dv * eout;
            e = cudaMemcpy2DAsync(static_cast<uint8_t*>(o) + t0 * dv * eout, (size_t)N * dv * eout,
                                  od[j], w, w, rows, cudaMemcpyDeviceToHost, ds);
        }
        if (e == cudaSuccess) e = cudaEventRecord(d2h_done[j], ds);
        if (e != cudaSuccess) return fail(status_of(e));
    }
    // the compute stream orders everything: the last copies out, then the final state
    e = cudaStreamWaitEvent(cs, d2h_done[(nseg - 1) & 1], 0);
    if (e == cudaSuccess && nseg >= 2) e = cudaStreamWaitEvent(cs, d2h_done[nseg & 1], 0);
    if (e != cudaSuccess) return fail(status_of(e));
    if (state_out)
        e = cudaMemcpyAsync(state_out, st, (size_t)b * H * dk * dv * sizeof(float),
                            cudaMemcpyDeviceToDevice, cs);
    return finish(status_of(e));
}

size_t retention_chunkwise_host_static_scratch_bytes(void) { return kStaticScratchBytes; }

int retention_chunkwise_host_noalloc(const void* q, const void* k, const void* v, void* o,
                                     ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                                     int dk, int dv, int chunk, const double* gamma,
                                     const float* state_in, float* state_out, int seg_len,
                                     void* stream, void* h2d_stream, void* d2h_stream) {
    // every check, the size of the static scratch included, before any device access (the
    // placeholder stands for the scratch address, which is 256-byte aligned)
    const int rc = check_args(q, k, v, o, in_dtype, out_dtype, b, H, N, dk, dv, chunk, gamma,
                              state_in, state_out, seg_len, reinterpret_cast<const void*>(kAlign),
                              kStaticScratchBytes);
    if (rc != RET_OK && rc != kNoWork) return rc;
    void* scratch = nullptr;
    if (rc == RET_OK) {
        const cudaError_t e = static_scratch(&scratch);
        if (e != cudaSuccess) return status_of(e);
    }
    return retention_chunkwise_host(q, k, v, o, in_dtype, out_dtype, b, H, N, dk, dv, chunk, gamma,
                                    state_in, state_out, seg_len, scratch, kStaticScratchBytes,
                                    stream, h2d_stream, d2h_stream);
}

}  // extern "C"
