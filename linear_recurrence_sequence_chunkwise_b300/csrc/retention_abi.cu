// retention_abi.cu -- the C ABI of include/retention.h: argument checks, per-head
// constants, kernel selection.  Host code only; kernels live in the other files.
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "gemm.cuh"

using ret::HeadConsts;

namespace ret {
namespace {
std::atomic<unsigned long long> g_launches{0};
thread_local int t_last_kernel = RET_KERNEL_NONE;
thread_local int t_last_cuda_error = 0;
}
void count_launch(int kernel_code) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    t_last_kernel = kernel_code;
}
int record_cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return RET_OK;
    t_last_cuda_error = (int)e;
    return RET_ERR_CUDA;
}
}  // namespace ret

namespace {

bool is_dtype(int d) { return d == RET_F32 || d == RET_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dims_ok(int dk, int dv) {
    return dk > 0 && dv > 0 && dk % 16 == 0 && dv % 16 == 0 && dk <= 256 && dv <= 512;
}

// Decay constants of each head in fp64, rounded to fp32 once.  gamma must lie
// in [0, 1] ([RN2] "門控多尺度 Retention": a fixed decay per head).
int head_consts(const double* gamma, int H, int B, HeadConsts* hc) {
    if (H > ret::kMaxHeads) return RET_ERR_UNSUPPORTED;
    memset(hc, 0, sizeof(*hc));
    for (int h = 0; h < H; ++h) {
        double g = gamma[h];
        if (!(g >= 0.0 && g <= 1.0)) return RET_ERR_UNSUPPORTED;  // also rejects NaN
        hc->l2g[h] = (g == 0.0) ? -INFINITY : (float)log2(g);
        hc->lng[h] = (g == 0.0) ? -INFINITY : (float)log(g);
        hc->omg[h] = (float)(1.0 - g);
        hc->g1[h] = (float)g;
        hc->g128[h] = (float)pow(g, 128.0);
        hc->gB[h] = (float)pow(g, (double)B);
        hc->ginvB[h] = (g == 0.0) ? INFINITY : (float)pow(g, -(double)B);
    }
    return RET_OK;
}

int cuda_status(cudaError_t e) { return ret::record_cuda_status(e); }

}  // namespace

extern "C" {

const char* retention_status_string(int status) {
    switch (status) {
        case RET_OK: return "ok";
        case RET_ERR_NULL: return "a required pointer is NULL";
        case RET_ERR_SHAPE: return "invalid shape (negative size, or N not a multiple of a valid chunk)";
        case RET_ERR_DTYPE: return "dtype code is neither RET_F32 nor RET_BF16";
        case RET_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case RET_ERR_UNSUPPORTED: return "unsupported dims, heads, flags, gamma or eps";
        case RET_ERR_CUDA: return "CUDA launch or runtime error";
        case RET_ERR_TIMEOUT: return "a bounded on-chip wait expired inside a kernel";
        default: return "unknown status";
    }
}

int retention_parallel(const void* q, const void* k, const void* v, void* o,
                       ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N, int dk,
                       int dv, const double* gamma, unsigned flags, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (flags & ~(RET_NORM_SCALE | RET_NORM_DECAY | RET_NORM_ROWSUM)) return RET_ERR_UNSUPPORTED;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0 || N == 0) return RET_OK;
    if (!q || !k || !v || !o || !gamma) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RET_ERR_ALIGN;
    HeadConsts hc;
    int rc = head_consts(gamma, H, 1, &hc);
    if (rc != RET_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int ob = out_dtype == RET_BF16;
    if (in_dtype == RET_BF16) {
        cudaError_t e = ret::launch_parallel_tc(q, k, v, o, ob, b, H, N, dk, dv, hc, flags, s);
        if (e != cudaErrorNotSupported) return cuda_status(e);
    }
    return cuda_status(ret::launch_parallel_simt(q, k, v, o, in_dtype == RET_BF16, ob, b, H, N,
                                                 dk, dv, hc, flags, s));
}

int retention_parallel_gated(const void* q, const void* k, const void* v, const void* g,
                             void* out, ret_dtype in_dtype, ret_dtype g_dtype,
                             ret_dtype out_dtype, int b, int H, int N, int dk, int dv,
                             const double* gamma, unsigned flags, float eps,
                             const float* weight, const float* bias, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(g_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (flags & ~(RET_NORM_SCALE | RET_NORM_DECAY | RET_NORM_ROWSUM)) return RET_ERR_UNSUPPORTED;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || isinf(eps)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0 || N == 0) return RET_OK;
    if (!q || !k || !v || !g || !out || !gamma) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out))
        return RET_ERR_ALIGN;
    if ((weight && !aligned16(weight)) || (bias && !aligned16(bias))) return RET_ERR_ALIGN;
    // tensor-core shapes only (see the header)
    if (in_dtype != RET_BF16 || !(dk == 128 || dk == 256) || dv % 128 != 0 || N < 128)
        return RET_ERR_UNSUPPORTED;
    HeadConsts hc;
    int rc = head_consts(gamma, H, 1, &hc);
    if (rc != RET_OK) return rc;
    cudaError_t e = ret::launch_parallel_gated_tc(q, k, v, g, out, g_dtype == RET_BF16,
                                                  out_dtype == RET_BF16, b, H, N, dk, dv, hc,
                                                  flags, eps, weight, bias,
                                                  static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return RET_ERR_UNSUPPORTED;
    return cuda_status(e);
}

int retention_chunkwise(const void* q, const void* k, const void* v, void* o,
                        ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N, int dk,
                        int dv, int chunk, const double* gamma, const float* state_in,
                        float* state_out, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (chunk < 16 || chunk > 256 || chunk % 16 != 0) return RET_ERR_SHAPE;
    if (N % chunk != 0) return RET_ERR_SHAPE;
    if (b == 0 || H == 0) return RET_OK;
    if (!gamma) return RET_ERR_NULL;
    if (N == 0) {
        // No tokens: the final state is the incoming one.
        if (!state_out) return RET_OK;
        if (!aligned16(state_out) || (state_in && !aligned16(state_in))) return RET_ERR_ALIGN;
        size_t bytes = (size_t)b * H * dk * dv * sizeof(float);
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (state_in) {
            if (state_in == state_out) return RET_OK;
            return cuda_status(cudaMemcpyAsync(state_out, state_in, bytes,
                                               cudaMemcpyDeviceToDevice, s));
        }
        return cuda_status(cudaMemsetAsync(state_out, 0, bytes, s));
    }
    if (!q || !k || !v || !o) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RET_ERR_ALIGN;
    if ((state_in && !aligned16(state_in)) || (state_out && !aligned16(state_out)))
        return RET_ERR_ALIGN;
    HeadConsts hc;
    int rc = head_consts(gamma, H, chunk, &hc);
    if (rc != RET_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int ob = out_dtype == RET_BF16;
    if (in_dtype == RET_BF16) {
        // eq.(7) gives the same function for every chunk length (the chunk only orders the
        // work: R_i carries everything before the chunk exactly), so the call runs on the
        // fastest schedule that applies: the pair kernel with 256-token chunks when N splits
        // into them, else the caller's chunk length (pair kernel, then one-SM kernel), else
        // 256- or 128-token chunks -- a chunk below 128 has no tensor-core schedule of its
        // own, and decays too small for the folded factors at 256 tokens (g^-256 > 2^64)
        // still fit them at 128 -- and the CUDA-core kernel when none applies.
        const int schedule[4] = {256, chunk, 256, 128};
        for (int i = 0; i < 4; ++i) {
            const int cb = schedule[i];
            if (N % cb != 0 || (i == 0 && cb == chunk) || (i >= 2 && cb == chunk)) continue;
            HeadConsts hcb;
            if (head_consts(gamma, H, cb, &hcb) != RET_OK) continue;
            cudaError_t e = ret::launch_chunkwise_tc_pair(q, k, v, o, ob, b, H, N, dk, dv, cb,
                                                          hcb, state_in, state_out, s);
            if (e != cudaErrorNotSupported) return cuda_status(e);
            if (i == 0) continue;          // the first entry is for the pair kernel only
            e = ret::launch_chunkwise_tc(q, k, v, o, ob, b, H, N, dk, dv, cb, hcb, state_in,
                                         state_out, s);
            if (e != cudaErrorNotSupported) return cuda_status(e);
        }
    }
    return cuda_status(ret::launch_chunkwise_simt(q, k, v, o, in_dtype == RET_BF16, ob, b, H, N,
                                                  dk, dv, chunk, hc, state_in, state_out, s));
}

int retention_chunkwise_backward(const void* q, const void* k, const void* v,
                                 const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                 ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                                 int dk, int dv, int chunk, const double* gamma,
                                 const float* state_in, const float* dstate_out,
                                 float* dstate_in, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (chunk < 16 || chunk > 256 || chunk % 16 != 0) return RET_ERR_SHAPE;
    if (N % chunk != 0) return RET_ERR_SHAPE;
    if (b == 0 || H == 0) return RET_OK;
    if (!gamma) return RET_ERR_NULL;
    if ((state_in && !aligned16(state_in)) || (dstate_out && !aligned16(dstate_out)) ||
        (dstate_in && !aligned16(dstate_in)))
        return RET_ERR_ALIGN;
    // The gradient is the same function for every chunk length: scan in chunks of 64
    // (the register-blocked kernel) whenever N allows it.
    const int kchunk = (N % 64 == 0) ? 64 : chunk;
    HeadConsts hc;
    int rc = head_consts(gamma, H, kchunk, &hc);
    if (rc != RET_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        // No tokens: L = <dstate_out, S0>, so the incoming state's gradient is dstate_out.
        if (!dstate_in) return RET_OK;
        size_t bytes = (size_t)b * H * dk * dv * sizeof(float);
        if (dstate_out) {
            if (dstate_out == dstate_in) return RET_OK;
            return cuda_status(cudaMemcpyAsync(dstate_in, dstate_out, bytes,
                                               cudaMemcpyDeviceToDevice, s));
        }
        return cuda_status(cudaMemsetAsync(dstate_in, 0, bytes, s));
    }
    if (!q || !k || !v || !dout || !grad_q || !grad_k || !grad_v) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) ||
        !aligned16(grad_q) || !aligned16(grad_k) || !aligned16(grad_v))
        return RET_ERR_ALIGN;
    return cuda_status(ret::launch_chunkwise_backward_simt(
        q, k, v, dout, grad_q, grad_k, grad_v, in_dtype == RET_BF16, out_dtype == RET_BF16, b,
        H, N, dk, dv, kchunk, hc, state_in, dstate_out, dstate_in, s));
}

size_t retention_chunkwise_backward_workspace_bytes(ret_dtype out_dtype, int b, int H, int N,
                                                    int dk, int dv) {
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0 || dk != 256 || dv % 256 != 0) return 0;
    return ret::chunkwise_backward_tc_workspace(out_dtype == RET_BF16, b, H, N, dk, dv);
}

int retention_chunkwise_backward_ws(const void* q, const void* k, const void* v,
                                    const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                    ret_dtype in_dtype, ret_dtype out_dtype, int b, int H,
                                    int N, int dk, int dv, int chunk, const double* gamma,
                                    const float* state_in, const float* dstate_out,
                                    float* dstate_in, void* workspace, size_t workspace_bytes,
                                    void* stream) {
    // the checks of retention_chunkwise_backward first (it also handles every case the
    // tensor-core passes do not take)
    if (b < 0 || H < 0 || N < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (chunk < 16 || chunk > 256 || chunk % 16 != 0) return RET_ERR_SHAPE;
    if (N % chunk != 0) return RET_ERR_SHAPE;
    if (b == 0 || H == 0 || N == 0 || !gamma || H > ret::kMaxHeads)
        return retention_chunkwise_backward(q, k, v, dout, grad_q, grad_k, grad_v, in_dtype,
                                            out_dtype, b, H, N, dk, dv, chunk, gamma, state_in,
                                            dstate_out, dstate_in, stream);
    HeadConsts hc256;
    int rc = head_consts(gamma, H, 256, &hc256);
    if (rc != RET_OK) return rc;
    if (!ret::chunkwise_backward_tc_supported(in_dtype == RET_BF16, H, N, dk, dv, hc256))
        return retention_chunkwise_backward(q, k, v, dout, grad_q, grad_k, grad_v, in_dtype,
                                            out_dtype, b, H, N, dk, dv, chunk, gamma, state_in,
                                            dstate_out, dstate_in, stream);
    if (!q || !k || !v || !dout || !grad_q || !grad_k || !grad_v || !workspace) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) ||
        !aligned16(grad_q) || !aligned16(grad_k) || !aligned16(grad_v) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RET_ERR_ALIGN;
    if ((state_in && !aligned16(state_in)) || (dstate_out && !aligned16(dstate_out)) ||
        (dstate_in && !aligned16(dstate_in)))
        return RET_ERR_ALIGN;
    if (workspace_bytes < ret::chunkwise_backward_tc_workspace(out_dtype == RET_BF16, b, H, N, dk, dv))
        return RET_ERR_SHAPE;
    if ((long long)b * H * N >= (1LL << 31)) return RET_ERR_UNSUPPORTED;
    return cuda_status(ret::launch_chunkwise_backward_tc(
        q, k, v, dout, grad_q, grad_k, grad_v, out_dtype == RET_BF16, b, H, N, dk, dv, hc256,
        state_in, dstate_out, dstate_in, workspace, static_cast<cudaStream_t>(stream)));
}

int retention_recurrent_step(const void* q, const void* k, const void* v, float* state, void* o,
                             ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int dk,
                             int dv, const double* gamma, void* stream) {
    if (b < 0 || H < 0 || dk < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (!dims_ok(dk, dv)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0) return RET_OK;
    if (!q || !k || !v || !state || !o || !gamma) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(o))
        return RET_ERR_ALIGN;
    HeadConsts hc;
    int rc = head_consts(gamma, H, 1, &hc);
    if (rc != RET_OK) return rc;
    return cuda_status(ret::launch_recurrent_step(q, k, v, state, o, in_dtype == RET_BF16,
                                                  out_dtype == RET_BF16, b, H, dk, dv, hc,
                                                  static_cast<cudaStream_t>(stream)));
}

int msr_epilogue(const void* y, const void* g, void* out, ret_dtype y_dtype, ret_dtype g_dtype,
                 ret_dtype out_dtype, int b, int H, int N, int dv, float eps,
                 const float* weight, const float* bias, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dv < 0) return RET_ERR_SHAPE;
    if (!is_dtype(y_dtype) || !is_dtype(g_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (dv <= 0 || dv % 16 != 0 || dv > 512) return RET_ERR_UNSUPPORTED;
    if (H > ret::kMaxHeads) return RET_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || isinf(eps)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0 || N == 0) return RET_OK;
    if (!y || !g || !out) return RET_ERR_NULL;
    if (!aligned16(y) || !aligned16(g) || !aligned16(out)) return RET_ERR_ALIGN;
    if ((weight && !aligned16(weight)) || (bias && !aligned16(bias))) return RET_ERR_ALIGN;
    return cuda_status(ret::launch_msr_epilogue(y, g, out, y_dtype == RET_BF16,
                                                g_dtype == RET_BF16, out_dtype == RET_BF16, b, H,
                                                N, dv, eps, weight, bias,
                                                static_cast<cudaStream_t>(stream)));
}

int retention_xpos_rotate(const void* q, const void* k, void* q_out, void* k_out,
                          ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                          int dk, const double* theta, long long pos0, void* stream) {
    if (b < 0 || H < 0 || N < 0 || dk < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (!dims_ok(dk, 16)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || H == 0 || N == 0) return RET_OK;
    if (!q || !q_out || !theta || (k && !k_out)) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(q_out) || (k && (!aligned16(k) || !aligned16(k_out))))
        return RET_ERR_ALIGN;
    if (in_dtype != out_dtype && (q_out == q || (k && k_out == k))) return RET_ERR_DTYPE;
    for (int j = 0; j < dk / 2; ++j)
        if (!isfinite(theta[j])) return RET_ERR_UNSUPPORTED;
    return cuda_status(ret::launch_xpos_rotate(q, k, q_out, k ? k_out : nullptr,
                                               in_dtype == RET_BF16, out_dtype == RET_BF16, b,
                                               H, N, dk, theta, pos0,
                                               static_cast<cudaStream_t>(stream)));
}

int rglru_scan(const void* x, const void* gate_a, const void* gate_x, const float* lambda_,
               const float* h0, void* y, float* h_last, ret_dtype in_dtype,
               ret_dtype out_dtype, int b, int T, int D, float c, void* stream) {
    if (b < 0 || T < 0 || D < 0) return RET_ERR_SHAPE;
    if (!is_dtype(in_dtype) || !is_dtype(out_dtype)) return RET_ERR_DTYPE;
    if (D % 64 != 0) return RET_ERR_UNSUPPORTED;
    if (!(c >= 0.0f) || isinf(c)) return RET_ERR_UNSUPPORTED;
    if (b == 0 || D == 0) return RET_OK;
    if ((h0 && !aligned16(h0)) || (h_last && !aligned16(h_last))) return RET_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // No steps: the final state is the incoming one.
        if (!h_last) return RET_OK;
        size_t bytes = (size_t)b * D * sizeof(float);
        if (h0) {
            if (h0 == h_last) return RET_OK;
            return cuda_status(cudaMemcpyAsync(h_last, h0, bytes, cudaMemcpyDeviceToDevice, s));
        }
        return cuda_status(cudaMemsetAsync(h_last, 0, bytes, s));
    }
    if (!x || !gate_a || !gate_x || !lambda_ || !y) return RET_ERR_NULL;
    if (!aligned16(x) || !aligned16(gate_a) || !aligned16(gate_x) || !aligned16(lambda_) ||
        !aligned16(y))
        return RET_ERR_ALIGN;
    return cuda_status(ret::launch_rglru_scan(x, gate_a, gate_x, lambda_, h0, y, h_last,
                                              in_dtype == RET_BF16, out_dtype == RET_BF16, b,
                                              T, D, c, s));
}

unsigned long long retention_kernel_launches(void) { return ret::g_launches.load(); }

int retention_last_kernel(void) { return ret::t_last_kernel; }

int retention_last_cuda_error(void) { return ret::t_last_cuda_error; }

const char* retention_cuda_error_string(int cuda_error) {
    static thread_local char buf[256];
    const cudaError_t e = static_cast<cudaError_t>(cuda_error);
    snprintf(buf, sizeof(buf), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return buf;
}

int retention_chunkwise_wait_selftest(const void* q, const void* k, const void* v, void* o,
                                      void* stream) {
    if (!q || !k || !v || !o) return RET_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RET_ERR_ALIGN;
    const int H = 1, N = 256, dk = 256, dv = 128, chunk = 256;
    const double gamma[1] = {0.96875};
    HeadConsts hc;
    int rc = head_consts(gamma, H, chunk, &hc);
    if (rc != RET_OK) return rc;
    // every wait gives up after 1 ms; the TMA producer issues no load, so nothing is in
    // flight when the CTAs unwind
    return cuda_status(ret::launch_chunkwise_tc_pair(q, k, v, o, 0, 1, H, N, dk, dv, chunk, hc,
                                                     nullptr, nullptr,
                                                     static_cast<cudaStream_t>(stream),
                                                     1000000ull, 1));
}

int retention_chunkwise_format_reruns(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return (int)ret::read_clear_reruns_tc_chunkwise_pair(s);
}

int retention_parallel_format_reruns(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    return (int)ret::read_clear_reruns_parallel_pair(s);
}

int retention_check_device_error(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) return cuda_status(ce);
    unsigned e = ret::read_clear_error_tc_chunkwise(s) | ret::read_clear_error_tc_chunkwise_pair(s) |
                 ret::read_clear_error_tc_parallel(s) | ret::read_clear_error_gemm(s) |
                 ret::read_clear_error_rglru(s) | ret::read_clear_error_parallel_pair(s);
    ce = cudaGetLastError();
    if (ce != cudaSuccess) return cuda_status(ce);
    return e ? RET_ERR_TIMEOUT : RET_OK;
}

}  // extern "C"
