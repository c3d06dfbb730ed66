// gemm.cuh -- the projection GEMM of the gated multi-scale retention layer (tc_gemm.cu):
// C = A W with A [M][K] and W [K][Nc] bf16 row-major, fp32 accumulation, and the epilogue
// that places C where the next step of the layer reads it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ret {

constexpr int kGemmMaxPairs = 128;   // xPos: coordinate pairs per head (d <= 256)

struct GemmEpilogue {
    int mode;          // 0: row-major out[M][ldo]; 1: head-major out[b][H][nseq][d]
    int out_bf16;      // output element type: bf16 (1) or fp32 (0)
    void* out;
    long long ldo;     // mode 0: elements between rows
    int nseq, H, d;    // mode 1: rows are (b, n) with n < nseq; columns (h, i) with i < d
    int xpos;          // mode 1: rotate the pairs (2j, 2j+1) of each head by e^{i p theta_j}
    long long pos0;    // position of the first row of every sequence
    // T_j = 2^64 frac(theta_j / 2 pi), split into 32-bit halves
    uint32_t turns_lo[kGemmMaxPairs], turns_hi[kGemmMaxPairs];
};

// Address of element (row r, column c) of the output.
__device__ __forceinline__ char* gemm_out_addr(const GemmEpilogue& ep, int r, int c, int esize) {
    size_t off;
    if (ep.mode == 0) {
        off = (size_t)r * (size_t)ep.ldo + (size_t)c;
    } else {
        const int bi = r / ep.nseq, n = r - bi * ep.nseq;
        const int h = c / ep.d, i = c - h * ep.d;
        off = (((size_t)bi * ep.H + h) * ep.nseq + n) * ep.d + i;
    }
    return static_cast<char*>(ep.out) + off * (size_t)esize;
}

// Launch the GEMM on `s`: Nc % 256 == 0, K % 64 == 0, any M > 0; pointers 16-byte aligned.
// Returns cudaErrorNotSupported for shapes outside that.
cudaError_t launch_gemm_bf16(const void* a, const void* w, int M, int Nc, int K,
                             const GemmEpilogue& ep, cudaStream_t s);
unsigned read_clear_error_gemm(cudaStream_t s);

}  // namespace ret
