// backward_tc.cu -- the gradient of the chunkwise form on tensor cores, as forward passes.
//
// The pages train with eqs.(5)/(7) ([RN2] "訓練/推理") and print no backward pass; the
// gradient is the exact derivative of eq.(7) for L = sum dout . o + <dS_final, S_final>.
// With o_n = sum_{m<=n} g^(n-m) (q_n . k_m) v_m + g^(n+1) q_n S0 and
// S_final = sum_m g^(N-1-m) k_m^T v_m + g^N S0, every gradient is itself a retention of
// the forward kind ("F(Q', K', V'; S0')" below, eq.(7) with chunk 256 on the pair kernel:
// the gradient does not depend on the chunk length):
//   dq_n = sum_{m<=n} g^(n-m) (dout_n . v_m) k_m + g^(n+1) dout_n S0^T
//        = F(dout, v, k; S0^T)
//   dv_m = sum_{n>=m} g^(n-m) (q_n . k_m) dout_n + g^(N-1-m) k_m dS_final
//        = rev F(rev k, rev q, rev dout; dS_final / g)          (rev: the token order reversed)
//   dk_m = sum_{n>=m} g^(n-m) (dout_n . v_m) q_n + g^(N-1-m) v_m dS_final^T
//        = rev F(rev v, rev dout, rev q; dS_final^T / g)
//   dS0  = sum_n g^(n+1) q_n^T dout_n + g^N dS_final = g * (final state of the dv pass)
// In reversed time the row m' = N-1-m collects the keys n' <= m' with g^(m'-n'), which is
// the forward form; its incoming-state term g^(m'+1) Q' S0' equals g^(N-1-m) Q' dS when
// S0' = dS / g.  The dq and dk passes have a 512-wide score dimension (dv); the scores
// are sums over that dimension and the state term is linear in it, so each pass runs as two
// passes over 256-column halves (read in place through pitched tensor maps) whose outputs
// add.  Host code plus small memory-bound kernels: the reversed copies of q, k, v and dout,
// the state transposes (scaled by 1/g), the sums of the halves with the reversal back,
// and dS0.  Five pair-kernel passes do all the contractions.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
constexpr int kPart = 256;             // width of one half of the 512-wide score dimension

struct BwdWs {
    size_t rq, rk, rv, rdo, op, odv, stq, stk, stv, sout, sc;
    size_t total() const { return rq + rk + rv + rdo + op + odv + stq + stk + stv + sout + sc; }
};

BwdWs bwd_ws(int b, int H, int N, int dk, int dv) {
    const size_t bh = (size_t)b * H, tok = bh * (size_t)N;
    const size_t parts = (size_t)(dv / kPart);
    BwdWs w;
    w.rq = round_up(tok * dk * 2);
    w.rk = w.rq;
    w.rv = round_up(tok * dv * 2);
    w.rdo = w.rv;
    w.op = round_up(parts * tok * dk * 4);          // partial outputs of the halves (fp32)
    w.odv = round_up(tok * dv * 4);
    w.stq = round_up(parts * bh * kPart * dk * 4);  // S0^T halves
    w.stk = w.stq;                                   // dS^T halves / g
    w.stv = round_up(bh * dk * dv * 4);              // dS / g
    w.sout = w.stv;                                  // final state of the dv pass
    w.sc = round_up(3 * ret::kMaxHeads * sizeof(float));   // per-head scales 1, 1/g, g
    return w;
}

// out[bh][n][:] = in[bh][N-1-n][:], rows of w bf16 (w % 8 == 0), 16-byte vectors
__global__ void reverse_rows_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                    long long rows_total, int N, int vec_per_row) {
    const long long total = rows_total * vec_per_row;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / vec_per_row;
        const int c = (int)(i - row * vec_per_row);
        const long long bh = row / N;
        const int n = (int)(row - bh * N);
        out[i] = __ldcs(in + ((bh * N + (N - 1 - n)) * vec_per_row + c));
    }
}

// out[p][bh][i][j] = scale_h * S[bh][j][p*256 + i] (transpose == 1: the dk x dv state's
// column halves, transposed) or out[bh][i][j] = scale_h * S[bh][i][j] (transpose == 0)
__global__ void state_prep_kernel(const float* __restrict__ S, float* __restrict__ out, int BH,
                                  int H, int dk, int dv, int transpose, const float* __restrict__ scale) {
    const long long total = (long long)BH * dk * dv;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int bh = (int)(i / ((long long)dk * dv));
        const long long r = i - (long long)bh * dk * dv;
        const float sc = scale[bh % H];
        if (!transpose) {
            out[i] = sc * S[i];
        } else {
            // i enumerates the output: part p, row ii (< 256), column j (< dk)
            const int per_part = kPart * dk;
            const int p = (int)(r / per_part);
            const int rr = (int)(r - (long long)p * per_part);
            const int ii = rr / dk, j = rr - ii * dk;
            const float x = S[((long long)bh * dk + j) * dv + p * kPart + ii];
            out[((long long)p * BH + bh) * per_part + rr] = sc * x;
        }
    }
}

// grad[bh][n][c] = sum_p src_p[bh][rev ? N-1-n : n][c], src_p = src + p * part_stride (fp32)
template <bool OUT_BF16>
__global__ void combine_kernel(const float* __restrict__ src, long long part_stride, int parts,
                               void* __restrict__ grad, long long rows_total, int N, int width,
                               int rev) {
    const int v4 = width / 4;
    const long long total = rows_total * v4;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / v4;
        const int c = (int)(i - row * v4);
        const long long bh = row / N;
        const int n = (int)(row - bh * N);
        const long long srow = bh * N + (rev ? (N - 1 - n) : n);
        float4 acc = __ldcs(reinterpret_cast<const float4*>(src) + srow * v4 + c);
        for (int p = 1; p < parts; ++p) {
            const float4 t = __ldcs(reinterpret_cast<const float4*>(src + p * part_stride) + srow * v4 + c);
            acc.x += t.x; acc.y += t.y; acc.z += t.z; acc.w += t.w;
        }
        if (OUT_BF16) {
            __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b2 = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t*>(&a);
            u.y = *reinterpret_cast<uint32_t*>(&b2);
            reinterpret_cast<uint2*>(grad)[i] = u;
        } else {
            reinterpret_cast<float4*>(grad)[i] = acc;
        }
    }
}

int grid_for(long long n) {
    long long g = (n + 255) / 256;
    return (int)(g < 148 * 16 ? (g > 0 ? g : 1) : 148 * 16);
}

}  // namespace

namespace ret {

bool chunkwise_backward_tc_supported(int in_bf16, int H, int N, int dk, int dv, const HeadConsts& hc256) {
    if (!in_bf16 || dk != 256 || dv % kPart != 0 || N % 256 != 0) return false;
    for (int h = 0; h < H; ++h)
        if (!(hc256.g1[h] > 0.0f)) return false;
    return chunkwise_pair_supported(256, 256, 256, hc256, H) &&
           chunkwise_pair_supported(256, dv, 256, hc256, H);
}

size_t chunkwise_backward_tc_workspace(int b, int H, int N, int dk, int dv) {
    return bwd_ws(b, H, N, dk, dv).total();
}

cudaError_t launch_chunkwise_backward_tc(const void* q, const void* k, const void* v,
                                         const void* dout, void* grad_q, void* grad_k,
                                         void* grad_v, int out_bf16, int b, int H, int N, int dk,
                                         int dv, const HeadConsts& hc256, const float* state_in,
                                         const float* dstate_out, float* dstate_in,
                                         void* workspace, cudaStream_t s) {
    const BwdWs L = bwd_ws(b, H, N, dk, dv);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    auto take = [&](size_t n) { uint8_t* r = p; p += n; return r; };
    void* rq = take(L.rq);
    void* rk = take(L.rk);
    void* rv = take(L.rv);
    void* rdo = take(L.rdo);
    float* op = reinterpret_cast<float*>(take(L.op));
    float* odv = reinterpret_cast<float*>(take(L.odv));
    float* stq = reinterpret_cast<float*>(take(L.stq));
    float* stk = reinterpret_cast<float*>(take(L.stk));
    float* stv = reinterpret_cast<float*>(take(L.stv));
    float* sout = reinterpret_cast<float*>(take(L.sout));
    float* scales = reinterpret_cast<float*>(take(L.sc));   // [0,H): 1, [H,2H): 1/g, [2H,3H): g
    const int BH = b * H, parts = dv / kPart;
    const long long rows = (long long)BH * N;
    const long long part_stride = rows * dk;           // elements between partial outputs

    {
        // pageable source: the copy has consumed it when cudaMemcpyAsync returns
        float host[3 * kMaxHeads];
        for (int h = 0; h < H; ++h) {
            host[h] = 1.0f;
            host[H + h] = 1.0f / hc256.g1[h];
            host[2 * H + h] = hc256.g1[h];
        }
        cudaError_t e = cudaMemcpyAsync(scales, host, 3 * H * sizeof(float), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
    }
    // reversed copies of q, k, v, dout
    const void* srcs[4] = {q, k, v, dout};
    void* dsts[4] = {rq, rk, rv, rdo};
    const int widths[4] = {dk, dk, dv, dv};
    for (int t = 0; t < 4; ++t) {
        const int vpr = widths[t] / 8;
        reverse_rows_kernel<<<grid_for(rows * vpr), 256, 0, s>>>(
            static_cast<const uint4*>(srcs[t]), static_cast<uint4*>(dsts[t]), rows, N, vpr);
    }
    // incoming states of the passes
    if (state_in)
        state_prep_kernel<<<grid_for((long long)BH * dk * dv), 256, 0, s>>>(state_in, stq, BH, H,
                                                                            dk, dv, 1, scales);
    if (dstate_out) {
        state_prep_kernel<<<grid_for((long long)BH * dk * dv), 256, 0, s>>>(dstate_out, stk, BH, H,
                                                                            dk, dv, 1, scales + H);
        state_prep_kernel<<<grid_for((long long)BH * dk * dv), 256, 0, s>>>(dstate_out, stv, BH, H,
                                                                            dk, dv, 0, scales + H);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dv = rev F(rev k, rev q, rev dout; dS / g); its final state gives dS0
    e = launch_chunkwise_tc_pair(rk, rq, rdo, odv, 0, b, H, N, dk, dv, 256, hc256,
                                 dstate_out ? stv : nullptr, dstate_in ? sout : nullptr, s);
    if (e != cudaSuccess) return e;
    if (dstate_in) {
        // dS0 = g * (final state of the dv pass)
        state_prep_kernel<<<grid_for((long long)BH * dk * dv), 256, 0, s>>>(sout, dstate_in, BH, H,
                                                                            dk, dv, 0, scales + 2 * H);
    }
    if (out_bf16)
        combine_kernel<true><<<grid_for(rows * dv / 4), 256, 0, s>>>(odv, 0, 1, grad_v, rows, N, dv, 1);
    else
        combine_kernel<false><<<grid_for(rows * dv / 4), 256, 0, s>>>(odv, 0, 1, grad_v, rows, N, dv, 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dq = sum over halves of F(dout_p, v_p, k; (S0^T)_p), halves read in place (pitch dv)
    const char* dob = static_cast<const char*>(dout);
    const char* vb = static_cast<const char*>(v);
    for (int pp = 0; pp < parts; ++pp) {
        e = launch_chunkwise_tc_pair(dob + (size_t)pp * kPart * 2, vb + (size_t)pp * kPart * 2, k,
                                     op + pp * part_stride, 0, b, H, N, kPart, dk, 256, hc256,
                                     state_in ? stq + (size_t)pp * BH * kPart * dk : nullptr, nullptr,
                                     s, 0, 0, dv, dv, dk, dk);
        if (e != cudaSuccess) return e;
    }
    if (out_bf16)
        combine_kernel<true><<<grid_for(rows * dk / 4), 256, 0, s>>>(op, part_stride, parts, grad_q, rows, N, dk, 0);
    else
        combine_kernel<false><<<grid_for(rows * dk / 4), 256, 0, s>>>(op, part_stride, parts, grad_q, rows, N, dk, 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dk = rev sum over halves of F(rev v_p, rev dout_p, rev q; (dS^T)_p / g)
    const char* rvb = static_cast<const char*>(rv);
    const char* rdb = static_cast<const char*>(rdo);
    for (int pp = 0; pp < parts; ++pp) {
        e = launch_chunkwise_tc_pair(rvb + (size_t)pp * kPart * 2, rdb + (size_t)pp * kPart * 2, rq,
                                     op + pp * part_stride, 0, b, H, N, kPart, dk, 256, hc256,
                                     dstate_out ? stk + (size_t)pp * BH * kPart * dk : nullptr, nullptr,
                                     s, 0, 0, dv, dv, dk, dk);
        if (e != cudaSuccess) return e;
    }
    if (out_bf16)
        combine_kernel<true><<<grid_for(rows * dk / 4), 256, 0, s>>>(op, part_stride, parts, grad_k, rows, N, dk, 1);
    else
        combine_kernel<false><<<grid_for(rows * dk / 4), 256, 0, s>>>(op, part_stride, parts, grad_k, rows, N, dk, 1);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_BACKWARD_TC);
    return e;
}

}  // namespace ret
