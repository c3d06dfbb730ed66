// msr_layer.cu -- the gated multi-scale retention layer as a chain of library calls.
//
// [RN2] "Transformer取代者登場！…RetNet…（2）", section "門控多尺度 Retention": per head h
// the layer computes Q = X W_Q, K = X W_K, V = X W_V (head h owns the columns h*dk.. of
// W_Q and W_K and h*dv.. of W_V), with xPos applied to Q and K ([RN2] "Retention" eqs.(2)-
// (3)), runs retention with the head's decay, normalises each head's output with
// GroupNorm, gates it with swish(X W_G) and projects the result with W_O.  Host code only:
//   1-4  four projection GEMMs (tc_gemm.cu): Q and K head-major with the rotation in the
//        epilogue, V head-major, G token-major, all bf16
//   5    the parallel form with the gated GroupNorm epilogue fused (retention_parallel_gated)
//        or, with chunk > 0, the chunkwise form (fp32 rows) followed by msr_epilogue
//   6    the W_O GEMM of the gated rows into the caller's output (fp32 or bf16)
// Every intermediate lives in the caller's workspace; the library allocates nothing.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "gemm.cuh"

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct LayerWs {
    size_t q, k, v, g, yg, y;
    size_t total() const { return q + k + v + g + yg + y; }
};

LayerWs layer_ws(int b, int N, int H, int dk, int dv, int chunk) {
    const size_t rows = (size_t)b * N;
    LayerWs w;
    w.q = round_up(rows * H * dk * 2);
    w.k = w.q;
    w.v = round_up(rows * H * dv * 2);
    w.g = w.v;
    w.yg = w.v;
    w.y = chunk > 0 ? round_up(rows * H * dv * 4) : 0;   // chunkwise rows before the epilogue
    return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// T_j = 2^64 frac(theta_j / 2 pi) in extended precision (the GEMM epilogue's phase table)
bool xpos_turns(const double* theta, int pairs, ret::GemmEpilogue* ep) {
    const long double two_pi = 6.283185307179586476925286766559L;
    for (int j = 0; j < pairs; ++j) {
        if (!isfinite(theta[j])) return false;
        long double t = fmodl((long double)theta[j] / two_pi, 1.0L);
        if (t < 0) t += 1.0L;
        long double s = t * 18446744073709551616.0L;           // 2^64
        unsigned long long T = (s >= 18446744073709551615.0L) ? 0ull : (unsigned long long)s;
        ep->turns_lo[j] = (uint32_t)T;
        ep->turns_hi[j] = (uint32_t)(T >> 32);
    }
    return true;
}

}  // namespace

extern "C" {

size_t retention_msr_layer_workspace_bytes(int b, int N, int H, int dk, int dv, int chunk) {
    if (b < 0 || N < 0 || H < 0 || dk < 0 || dv < 0 || chunk < 0) return 0;
    return layer_ws(b, N, H, dk, dv, chunk).total();
}

int retention_msr_layer(const void* x, const void* wq, const void* wk, const void* wv,
                        const void* wg, const void* wo, void* out, ret_dtype out_dtype, int b,
                        int N, int d_model, int H, int dk, int dv, int d_out,
                        const double* gamma, const double* theta, long long pos0,
                        unsigned flags, float eps, int chunk, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (b < 0 || N < 0 || d_model < 0 || H < 0 || dk < 0 || dv < 0 || d_out < 0 || chunk < 0)
        return RET_ERR_SHAPE;
    if (out_dtype != RET_F32 && out_dtype != RET_BF16) return RET_ERR_DTYPE;
    if (flags & ~(RET_NORM_SCALE | RET_NORM_DECAY | RET_NORM_ROWSUM)) return RET_ERR_UNSUPPORTED;
    if (chunk > 0 && flags) return RET_ERR_UNSUPPORTED;   // the chunkwise form is unnormalised
    if (!(eps >= 0.0f) || isinf(eps)) return RET_ERR_UNSUPPORTED;
    // tensor-core shapes: the projection GEMMs take 256-column tiles and 64-deep K steps,
    // the retention step the tensor-core kernels (see the header)
    if (H > ret::kMaxHeads || !(dk == 128 || dk == 256) || dv % 128 != 0 || dv > 512 ||
        d_model % 64 != 0 || (H * dk) % 256 != 0 || (H * dv) % 256 != 0 || d_out % 256 != 0)
        return RET_ERR_UNSUPPORTED;
    if (chunk > 0 && (chunk % 16 != 0 || chunk > 256 || N % chunk != 0)) return RET_ERR_SHAPE;
    if (chunk == 0 && N > 0 && N < 128) return RET_ERR_UNSUPPORTED;
    if (b == 0 || N == 0 || H == 0) return RET_OK;
    if (!x || !wq || !wk || !wv || !wg || !wo || !out || !gamma || !workspace) return RET_ERR_NULL;
    if (!aligned16(x) || !aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(wg) ||
        !aligned16(wo) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return RET_ERR_ALIGN;
    for (int h = 0; h < H; ++h)
        if (!(gamma[h] >= 0.0 && gamma[h] <= 1.0)) return RET_ERR_UNSUPPORTED;
    const LayerWs L = layer_ws(b, N, H, dk, dv, chunk);
    if (workspace_bytes < L.total()) return RET_ERR_SHAPE;
    if ((long long)b * N >= (1LL << 31)) return RET_ERR_UNSUPPORTED;

    ret::GemmEpilogue qk;
    memset(&qk, 0, sizeof(qk));
    if (theta && !xpos_turns(theta, dk / 2, &qk)) return RET_ERR_UNSUPPORTED;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* q = base;
    void* k = base + L.q;
    void* v = base + L.q + L.k;
    void* g = base + L.q + L.k + L.v;
    void* yg = base + L.q + L.k + L.v + L.g;
    void* y = base + L.q + L.k + L.v + L.g + L.yg;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int M = b * N;

    // 1-4: projections
    qk.mode = 1; qk.out_bf16 = 1; qk.nseq = N; qk.H = H; qk.d = dk;
    qk.xpos = theta != nullptr; qk.pos0 = pos0;
    qk.out = q;
    cudaError_t e = ret::launch_gemm_bf16(x, wq, M, H * dk, d_model, qk, s);
    if (e == cudaSuccess) { qk.out = k; e = ret::launch_gemm_bf16(x, wk, M, H * dk, d_model, qk, s); }
    if (e == cudaSuccess) {
        ret::GemmEpilogue ev;
        memset(&ev, 0, sizeof(ev));
        ev.mode = 1; ev.out_bf16 = 1; ev.out = v; ev.nseq = N; ev.H = H; ev.d = dv;
        e = ret::launch_gemm_bf16(x, wv, M, H * dv, d_model, ev, s);
    }
    if (e == cudaSuccess) {
        ret::GemmEpilogue eg;
        memset(&eg, 0, sizeof(eg));
        eg.mode = 0; eg.out_bf16 = 1; eg.out = g; eg.ldo = (long long)H * dv;
        e = ret::launch_gemm_bf16(x, wg, M, H * dv, d_model, eg, s);
    }
    if (e != cudaSuccess) return ret::record_cuda_status(e == cudaErrorNotSupported ? cudaErrorInvalidValue : e);
    // 5: retention + GroupNorm + swish gate -> yg [b][N][H*dv] bf16
    int rc;
    if (chunk == 0) {
        rc = retention_parallel_gated(q, k, v, g, yg, RET_BF16, RET_BF16, RET_BF16, b, H, N, dk, dv,
                                      gamma, flags, eps, nullptr, nullptr, stream);
    } else {
        rc = retention_chunkwise(q, k, v, y, RET_BF16, RET_F32, b, H, N, dk, dv, chunk, gamma,
                                 nullptr, nullptr, stream);
        if (rc == RET_OK)
            rc = msr_epilogue(y, g, yg, RET_F32, RET_BF16, RET_BF16, b, H, N, dv, eps, nullptr,
                              nullptr, stream);
    }
    if (rc != RET_OK) return rc;
    // 6: output projection
    ret::GemmEpilogue eo;
    memset(&eo, 0, sizeof(eo));
    eo.mode = 0; eo.out_bf16 = out_dtype == RET_BF16; eo.out = out; eo.ldo = d_out;
    e = ret::launch_gemm_bf16(yg, wo, M, d_out, H * dv, eo, s);
    if (e != cudaSuccess) return ret::record_cuda_status(e == cudaErrorNotSupported ? cudaErrorInvalidValue : e);
    return RET_OK;
}

}  // extern "C"

extern "C" {

int retention_gemm(const void* a, const void* w, void* c, ret_dtype c_dtype, int M, int Nc, int K,
                   void* stream) {
    if (M < 0 || Nc < 0 || K < 0) return RET_ERR_SHAPE;
    if (c_dtype != RET_F32 && c_dtype != RET_BF16) return RET_ERR_DTYPE;
    if (Nc % 256 != 0 || K % 64 != 0) return RET_ERR_UNSUPPORTED;
    if (M == 0 || Nc == 0 || K == 0) return RET_OK;
    if (!a || !w || !c) return RET_ERR_NULL;
    if (!aligned16(a) || !aligned16(w) || !aligned16(c)) return RET_ERR_ALIGN;
    ret::GemmEpilogue ep;
    memset(&ep, 0, sizeof(ep));
    ep.mode = 0; ep.out_bf16 = c_dtype == RET_BF16; ep.out = c; ep.ldo = Nc;
    const cudaError_t e = ret::launch_gemm_bf16(a, w, M, Nc, K, ep, static_cast<cudaStream_t>(stream));
    return e == cudaErrorNotSupported ? RET_ERR_UNSUPPORTED : ret::record_cuda_status(e);
}

int retention_project_heads(const void* x, const void* w, void* out, int b, int N, int d_in, int H,
                            int d, const double* theta, long long pos0, void* stream) {
    if (b < 0 || N < 0 || d_in < 0 || H < 0 || d < 0) return RET_ERR_SHAPE;
    if (d % 64 != 0 || d > 2 * ret::kGemmMaxPairs || (H * d) % 256 != 0 || d_in % 64 != 0)
        return RET_ERR_UNSUPPORTED;
    if (b == 0 || N == 0 || H == 0 || d_in == 0) return RET_OK;
    if (!x || !w || !out) return RET_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(out)) return RET_ERR_ALIGN;
    if ((long long)b * N >= (1LL << 31)) return RET_ERR_UNSUPPORTED;
    ret::GemmEpilogue ep;
    memset(&ep, 0, sizeof(ep));
    if (theta && !xpos_turns(theta, d / 2, &ep)) return RET_ERR_UNSUPPORTED;
    ep.mode = 1; ep.out_bf16 = 1; ep.out = out; ep.nseq = N; ep.H = H; ep.d = d;
    ep.xpos = theta != nullptr; ep.pos0 = pos0;
    const cudaError_t e = ret::launch_gemm_bf16(x, w, b * N, H * d, d_in, ep,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaErrorNotSupported ? RET_ERR_UNSUPPORTED : ret::record_cuda_status(e);
}

}  // extern "C"
