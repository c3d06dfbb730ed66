// tcgen05_mma_cost.cu -- cost of one tcgen05.mma (bf16, K=16) on this GPU versus N, the
// source of operand A (shared or tensor memory) and the number of issuing threads, for
// one SM (M=128) and for a pair of SMs (cta_group::2, M=256).
// Standalone program (not part of the library); build and run:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -I linear_recurrence_sequence_chunkwise_b300/csrc \
//        -o /tmp/tcgen05_mma_cost linear_recurrence_sequence_chunkwise_b300/microbench/tcgen05_mma_cost.cu
//   /tmp/tcgen05_mma_cost
// One CTA, 512 MMAs per issuing thread into its own accumulator, operands zero-filled;
// every wait is bounded.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include "tc_ptx.cuh"
using namespace ret::tc;

template <int N, int TS>
__device__ __forceinline__ void run8(uint32_t d, uint64_t dA, uint64_t dB, uint32_t ta, uint32_t id) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint64_t off = (uint64_t)(((k & 3) * 32 + (k >> 2) * 16384) >> 4);
        if (TS) mma_ts(d, ta + 8 * k, dB + off, id, 1);
        else mma_bf16(d, dA + off, dB + off, id, 1);
    }
}

template <int N, int TS>
__global__ void __launch_bounds__(128, 1) mb(int issuers, int reps, unsigned long long* out) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar[4];
    __shared__ uint32_t slot;
    for (int i = threadIdx.x; i < 96 * 1024 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) { for (int j = 0; j < 4; ++j) mbar_init(&bar[j], 1); fence_barrier_init(); }
    if (warp == 1) { tmem_alloc(&slot, 512); tmem_relinquish(); }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (lane == 0 && warp < issuers) {
        const uint32_t a = smem_u32(sm), b = a + 32768;
        const uint64_t dA = sdesc_sw128(a, 16, 1024), dB = sdesc_sw128(b, 16, 1024);
        const uint32_t id = TS ? idesc_bf16(128, N, 0, 0) : idesc_bf16(128, N, 0, 0);
        const uint32_t d = tmem + (uint32_t)((warp * N) % 256);
        const uint32_t ta = tmem + 256 + 64 * warp;
        unsigned long long t0 = clock64();
        for (int r = 0; r < reps; ++r) run8<N, TS>(d, dA, dB, ta, id);
        mma_commit(&bar[warp]);
        mbar_wait(&bar[warp], 0, nullptr, 1000000000ull);
        unsigned long long t2 = clock64();
        out[warp] = t2 - t0;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

template <int N, int TS>
void go(const char* name) {
    unsigned long long* d; cudaMalloc(&d, 64);
    unsigned long long h[4];
    cudaFuncSetAttribute(mb<N, TS>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
    for (int iss = 1; iss <= 4; iss *= 2) {
        for (int rep = 0; rep < 2; ++rep) {
            mb<N, TS><<<1, 128, 120 * 1024>>>(iss, 64, d);
            if (cudaDeviceSynchronize() != cudaSuccess) { printf("error\n"); exit(1); }
        }
        cudaMemcpy(h, d, 32, cudaMemcpyDeviceToHost);
        unsigned long long mx = 0;
        for (int j = 0; j < iss; ++j) mx = h[j] > mx ? h[j] : mx;
        printf("%-16s issuers %d: %6.1f cyc per MMA per issuer, %6.1f cyc per MMA aggregate\n", name, iss,
               (double)mx / 512.0, (double)mx / (512.0 * iss));
    }
}

// Pair MMAs (cta_group::2, M = 256: 128 rows per SM, operand B split by N between the two
// SMs), issued by one thread of the even CTA of a 2-CTA cluster.  Variant: 0 = A and B
// K-major from shared memory, 1 = A K-major / B MN-major, 2 = A MN-major / B MN-major,
// 3 = A from tensor memory / B MN-major.
template <int N, int VAR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) mb_pair(int reps, unsigned long long* out) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar;
    __shared__ uint32_t slot;
    for (int i = threadIdx.x; i < 64 * 1024 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    if (threadIdx.x == 0) { mbar_init(&bar, 1); fence_barrier_init(); }
    if (warp == 0) { tmem_alloc_pair(&slot, 512); tmem_relinquish_pair(); }
    fence_proxy_async();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = slot;
    if (rank == 0 && warp == 0 && lane == 0) {
        const uint32_t a = smem_u32(sm), b = a + 32768;
        const uint64_t dAk = sdesc_sw128(a, 16, 1024), dBk = sdesc_sw128(b, 16, 1024);
        const uint64_t dAm = sdesc_sw128(a, 16384, 1024), dBm = sdesc_sw128(b, 16384, 1024);
        const uint32_t id = idesc_bf16(256, N, VAR == 2 ? 1 : 0, VAR == 0 ? 0 : 1);
        unsigned long long t0 = clock64();
        for (int r = 0; r < reps; ++r) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t koff = (uint64_t)(((k & 3) * 32 + (k >> 2) * 16384) >> 4);   // K-major
                const uint64_t moff = (uint64_t)((k * 2048) >> 4);                          // MN-major
                if (VAR == 0) mma_pair(tmem, dAk + koff, dBk + koff, id, 1);
                else if (VAR == 1) mma_pair(tmem, dAk + koff, dBm + moff, id, 1);
                else if (VAR == 2) mma_pair(tmem, dAm + moff, dBm + moff, id, 1);
                else mma_pair_ts(tmem, tmem + 256 + 8 * k, dBm + moff, id, 1);
            }
        }
        mma_commit_pair(&bar, 1);
        mbar_wait(&bar, 0, nullptr, 1000000000ull);
        out[0] = clock64() - t0;
    }
    tc_fence_before();
    cluster_sync_all();
    if (warp == 0) { tc_fence_after(); tmem_dealloc_pair(tmem, 512); }
}

template <int N, int VAR>
void go_pair(const char* name) {
    unsigned long long* d; cudaMalloc(&d, 64);
    unsigned long long h = 0;
    cudaFuncSetAttribute(mb_pair<N, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
    for (int rep = 0; rep < 2; ++rep) {
        mb_pair<N, VAR><<<2, 128, 120 * 1024>>>(64, d);
        if (cudaDeviceSynchronize() != cudaSuccess) { printf("error\n"); exit(1); }
    }
    cudaMemcpy(&h, d, 8, cudaMemcpyDeviceToHost);
    printf("%-26s pair, 1 issuer: %6.1f cyc per MMA\n", name, (double)h / 512.0);
}

int main() {
    go<64, 0>("N64 smem");
    go<128, 0>("N128 smem");
    go<256, 0>("N256 smem");
    go<64, 1>("N64 tmem");
    go<128, 1>("N128 tmem");
    go<16, 0>("N16 smem");
    go_pair<256, 0>("M256 N256 A,B K-major");
    go_pair<128, 1>("M256 N128 A K, B MN");
    go_pair<128, 2>("M256 N128 A MN, B MN");
    go_pair<128, 3>("M256 N128 A tmem, B MN");
    return 0;
}
