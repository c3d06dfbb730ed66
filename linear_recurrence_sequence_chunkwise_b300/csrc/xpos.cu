// xpos.cu -- xPos rotation of Q and K, "Transformer取代者登場！…RetNet…（2）",
// "Retention", eqs.(2)-(3): Q_n e^{i n theta}, K_m e^{i m theta}, so that the score
// of eq.(4) (conjugate transpose) depends on n - m only.  For real inputs the pair of
// coordinates (2j, 2j+1) is one complex number, multiplied by e^{i p theta_j} at
// position p = pos0 + n.
//
// Memory-bound prologue (each element read and written once).  The phase depends on
// (p, j) only, so a thread owns one (position, pair) and applies the same rotation to
// that pair in every (batch, head) row; a warp covers 32 consecutive pairs of one
// position (128 or 256 contiguous bytes per row).  The phase is exact to fp32: the
// fraction of turns p theta_j / (2 pi) is reduced in fp64 (one multiply, rint and a
// subtraction, exact for |p theta_j / 2pi| < 2^52), then sincospi in fp32.
#include "common.cuh"

namespace ret {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxPairs = 128;   // dk <= 256

struct Turns {
    double c[kMaxPairs];         // theta_j / (2 pi), computed on the host in fp64
};

template <typename T> struct Pair;
template <> struct Pair<float> {
    static __device__ __forceinline__ float2 load(const float* p) {
        return *reinterpret_cast<const float2*>(p);
    }
    static __device__ __forceinline__ void store(float* p, float2 v) {
        *reinterpret_cast<float2*>(p) = v;
    }
};
template <> struct Pair<__nv_bfloat16> {
    static __device__ __forceinline__ float2 load(const __nv_bfloat16* p) {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float2 v) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
    }
};

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
xpos_kernel(const TI* q, const TI* k, TO* q_out, TO* k_out, int bH, int N, int d,
            long long pos0, const Turns turns) {
    const int pairs = d >> 1;
    const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (idx >= (long long)N * pairs) return;
    const int n = (int)(idx / pairs), j = (int)(idx % pairs);
    const double t = (double)(pos0 + n) * turns.c[j];
    const float f = (float)(t - rint(t));        // in [-1/2, 1/2] turns
    float sn, cs;
    sincospif(2.0f * f, &sn, &cs);
    const size_t row = (size_t)N * d;
    const size_t off0 = (size_t)n * d + 2 * j;
#pragma unroll 4
    for (int r = 0; r < bH; ++r) {
        const size_t off = (size_t)r * row + off0;
        const float2 a = Pair<TI>::load(q + off);
        Pair<TO>::store(q_out + off, make_float2(a.x * cs - a.y * sn, a.x * sn + a.y * cs));
        if (k) {
            const float2 b = Pair<TI>::load(k + off);
            Pair<TO>::store(k_out + off, make_float2(b.x * cs - b.y * sn, b.x * sn + b.y * cs));
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch_x(const void* q, const void* k, void* q_out, void* k_out, int bH, int N,
                     int d, long long pos0, const Turns& turns, cudaStream_t s) {
    const long long threads = (long long)N * (d / 2);
    const long long blocks = (threads + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    xpos_kernel<TI, TO><<<(unsigned)blocks, kThreads, 0, s>>>(
        static_cast<const TI*>(q), static_cast<const TI*>(k), static_cast<TO*>(q_out),
        static_cast<TO*>(k_out), bH, N, d, pos0, turns);
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launch(RET_KERNEL_XPOS);
    return err;
}

}  // namespace

cudaError_t launch_xpos_rotate(const void* q, const void* k, void* q_out, void* k_out,
                               int in_bf16, int out_bf16, int b, int H, int N, int d,
                               const double* theta, long long pos0, cudaStream_t s) {
    if (d / 2 > kMaxPairs) return cudaErrorInvalidValue;
    Turns turns;
    for (int j = 0; j < d / 2; ++j) turns.c[j] = theta[j] / (2.0 * M_PI);
    for (int j = d / 2; j < kMaxPairs; ++j) turns.c[j] = 0.0;
    using bf = __nv_bfloat16;
    const int bH = b * H;
    if (in_bf16)
        return out_bf16 ? launch_x<bf, bf>(q, k, q_out, k_out, bH, N, d, pos0, turns, s)
                        : launch_x<bf, float>(q, k, q_out, k_out, bH, N, d, pos0, turns, s);
    return out_bf16 ? launch_x<float, bf>(q, k, q_out, k_out, bH, N, d, pos0, turns, s)
                    : launch_x<float, float>(q, k, q_out, k_out, bH, N, d, pos0, turns, s);
}

}  // namespace ret
