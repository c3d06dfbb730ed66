// common.cuh -- shared types and small device helpers of the retention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/retention.h"

namespace ret {

constexpr int kMaxHeads = 128;
constexpr int kMaxDevices = 64;   // per-device caches of the host code

// Per-head decay constants, computed on the host in fp64 and rounded once.
//   l2g  = log2(gamma)            (-inf for gamma = 0)
//   lng  = ln(gamma)              (-inf for gamma = 0)
//   omg  = 1 - gamma
//   gB   = gamma^B                (chunkwise only; gamma^1 elsewhere)
//   g1   = gamma
//   g128 = gamma^128
//   ginvB = gamma^(-B)          (chunkwise only; +inf for gamma = 0)
struct HeadConsts {
    float g1[kMaxHeads];
    float g128[kMaxHeads];
    float l2g[kMaxHeads];
    float lng[kMaxHeads];
    float omg[kMaxHeads];
    float gB[kMaxHeads];
    float ginvB[kMaxHeads];
};

// gamma^e for an integer exponent e >= 0 from log2(gamma): exp2(e * log2 gamma),
// with gamma = 0 handled exactly (0^0 = 1, 0^e = 0).
__device__ __forceinline__ float decay_pow(float l2g, float e) {
    if (e == 0.0f) return 1.0f;
    return exp2f(e * l2g);  // l2g = -inf -> 0
}

// Row sum of D, s_n = sum_{i<=n} gamma^(n-i) = (1 - gamma^(n+1)) / (1 - gamma),
// written with expm1 so that gamma close to 1 keeps full precision.
__device__ __forceinline__ float decay_rowsum(float lng, float omg, int n) {
    if (omg == 0.0f) return (float)(n + 1);          // gamma = 1
    if (isinf(lng)) return 1.0f;                      // gamma = 0
    return -expm1f((float)(n + 1) * lng) / omg;
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return *p; }
    static __device__ __forceinline__ void store(float* p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float x) {
        *p = __float2bfloat16_rn(x);
    }
};

template <typename T> __device__ __forceinline__ float ld(const T* p) { return Elem<T>::load(p); }
template <typename T> __device__ __forceinline__ void st(T* p, float x) { Elem<T>::store(p, x); }

}  // namespace ret

// Host-side launchers implemented by the kernel files (all return cudaError_t
// of the launch; argument checks have already passed).
namespace ret {
cudaError_t launch_recurrent_step(const void* q, const void* k, const void* v, float* state,
                                  void* o, int in_bf16, int out_bf16, int b, int H, int dk,
                                  int dv, const HeadConsts& hc, cudaStream_t s);
cudaError_t launch_msr_epilogue(const void* y, const void* g, void* out, int y_bf16,
                                int g_bf16, int out_bf16, int b, int H, int N, int dv,
                                float eps, const float* weight, const float* bias,
                                cudaStream_t s);
cudaError_t launch_parallel_simt(const void* q, const void* k, const void* v, void* o,
                                 int in_bf16, int out_bf16, int b, int H, int N, int dk, int dv,
                                 const HeadConsts& hc, unsigned flags, cudaStream_t s);
cudaError_t launch_chunkwise_simt(const void* q, const void* k, const void* v, void* o,
                                  int in_bf16, int out_bf16, int b, int H, int N, int dk,
                                  int dv, int chunk, const HeadConsts& hc,
                                  const float* state_in, float* state_out, cudaStream_t s);
cudaError_t launch_chunkwise_backward_simt(const void* q, const void* k, const void* v,
                                           const void* dout, void* dq, void* dk, void* dv,
                                           int in_bf16, int out_bf16, int b, int H, int N,
                                           int dkk, int dvv, int chunk, const HeadConsts& hc,
                                           const float* state_in, const float* dstate_out,
                                           float* dstate_in, cudaStream_t s);
unsigned read_clear_error_rglru(cudaStream_t s);
cudaError_t launch_rglru_scan(const void* x, const void* ga, const void* gx, const float* lam,
                              const float* h0, void* y, float* h_last, int in_bf16, int out_bf16,
                              int b, int T, int D, float c, cudaStream_t s);
cudaError_t launch_xpos_rotate(const void* q, const void* k, void* q_out, void* k_out,
                               int in_bf16, int out_bf16, int b, int H, int N, int d,
                               const double* theta, long long pos0, cudaStream_t s);
// Tensor-core paths: return cudaErrorNotSupported when the shape is outside
// what the kernel handles, so the caller can pick the CUDA-core kernel.
cudaError_t launch_chunkwise_tc(const void* q, const void* k, const void* v, void* o,
                                int out_bf16, int b, int H, int N, int dk, int dv, int chunk,
                                const HeadConsts& hc, const float* state_in, float* state_out,
                                cudaStream_t s);
// Pair-of-SMs chunkwise kernel (cta_group::2): chunk 256, dk 256, dv a multiple of 128.
// wait_ns bounds every on-chip wait (0: the default of 2 s); no_loads makes the TMA
// producer issue nothing (self-test of the bounded waits: every wait then expires).
// ldq, ldk, ldv, ldo: elements between rows of q, k, v and o (0: dk, dk, dv, dv), so that
// column slices of wider matrices are read and written in place.  rev != 0 runs eq.(7) in
// reversed time on the rows as stored (row n collects the keys m >= n with g^(m-n); the
// chunks are scanned from the last; state_in enters at the end, state_out leaves at the
// start).  acc (fp32) is added to the output: with fp32 output it must be o itself (the
// kernel adds its rows to o by reductions in L2); with bf16 output it is a separate array of
// pitch ldo.
cudaError_t launch_chunkwise_tc_pair(const void* q, const void* k, const void* v, void* o,
                                     int out_bf16, int b, int H, int N, int dk, int dv, int chunk,
                                     const HeadConsts& hc, const float* state_in, float* state_out,
                                     cudaStream_t s, uint64_t wait_ns = 0, int no_loads = 0,
                                     int ldq = 0, int ldk = 0, int ldv = 0, int ldo = 0,
                                     int rev = 0, const float* acc = nullptr);
cudaError_t launch_parallel_tc(const void* q, const void* k, const void* v, void* o,
                               int out_bf16, int b, int H, int N, int dk, int dv,
                               const HeadConsts& hc, unsigned flags, cudaStream_t s);
cudaError_t launch_parallel_gated_tc(const void* q, const void* k, const void* v, const void* g,
                                     void* out, int g_bf16, int out_bf16, int b, int H, int N,
                                     int dk, int dv, const HeadConsts& hc, unsigned flags,
                                     float eps, const float* weight, const float* bias,
                                     cudaStream_t s);
// Parallel form on pairs of SMs (tc_parallel_pair.cu): bf16 inputs, dk 256, dv a multiple
// of 256, N a multiple of 256; epi 0 plain output ([b][H][N][dv]), 1 / 2 the gated
// GroupNorm epilogue with an fp32 / bf16 gate ([b][N][H*dv]).  cudaErrorNotSupported
// for other shapes.
cudaError_t launch_parallel_pair(const void* q, const void* k, const void* v, const void* g,
                                 void* out, int out_bf16, int epi, int b, int H, int N, int dk,
                                 int dv, const HeadConsts& hc, unsigned flags, float eps,
                                 const float* weight, const float* bias, cudaStream_t s);
unsigned read_clear_error_parallel_pair(cudaStream_t s);
unsigned read_clear_reruns_parallel_pair(cudaStream_t s);
// Gradient of the chunkwise form as pair-kernel passes (backward_tc.cu): bf16 inputs,
// dk 256, dv a multiple of 256, N a multiple of 256, decays the pair kernel takes at chunk
// 256 (hc256: head constants for chunk 256).  workspace: chunkwise_backward_tc_workspace
// bytes, 256-byte aligned.
bool chunkwise_pair_supported(int dk, int dv, int chunk, const HeadConsts& hc, int H);
bool chunkwise_backward_tc_supported(int in_bf16, int H, int N, int dk, int dv,
                                     const HeadConsts& hc256);
size_t chunkwise_backward_tc_workspace(int out_bf16, int b, int H, int N, int dk, int dv);
cudaError_t launch_chunkwise_backward_tc(const void* q, const void* k, const void* v,
                                         const void* dout, void* grad_q, void* grad_k,
                                         void* grad_v, int out_bf16, int b, int H, int N, int dk,
                                         int dv, const HeadConsts& hc256, const float* state_in,
                                         const float* dstate_out, float* dstate_in,
                                         void* workspace, cudaStream_t s);
// The current CUDA context (driver entry point fetched through the runtime, so the
// library needs no link to libcuda); nullptr if it cannot be queried.  Per-device caches
// compare it to notice a context made after a device reset.
void* current_context();
// Count one successful kernel launch (host-side, process-wide) and record its
// RET_KERNEL_* code for the launching host thread.
void count_launch(int kernel_code);
// RET_OK for cudaSuccess; otherwise records the error for retention_last_cuda_error and
// returns RET_ERR_CUDA.
int record_cuda_status(cudaError_t e);
// Device error words of the kernels with bounded waits: read and clear.
unsigned read_clear_error_tc_chunkwise(cudaStream_t s);
unsigned read_clear_error_tc_chunkwise_pair(cudaStream_t s);
// Units of the pair chunkwise kernel that re-ran in the hi/lo bf16 format: read and clear.
unsigned read_clear_reruns_tc_chunkwise_pair(cudaStream_t s);
unsigned read_clear_error_tc_parallel(cudaStream_t s);
}  // namespace ret
