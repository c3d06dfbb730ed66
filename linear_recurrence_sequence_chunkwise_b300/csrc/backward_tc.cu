// backward_tc.cu -- the gradient of the chunkwise form on tensor cores, as forward passes.
//
// The pages train with eqs.(5)/(7) ([RN2] "訓練/推理") and print no backward pass; the
// gradient is the exact derivative of eq.(7) for L = sum dout . o + <dS_final, S_final>.
// With o_n = sum_{m<=n} g^(n-m) (q_n . k_m) v_m + g^(n+1) q_n S0 and
// S_final = sum_m g^(N-1-m) k_m^T v_m + g^N S0, every gradient is itself a retention of
// the forward kind ("F(Q', K', V'; S0')" below: eq.(7) with chunk 256 on the pair kernel,
// since the result does not depend on the chunk length; "R" marks the pair kernel's
// reversed-time mode, in which row m collects the rows n >= m with g^(n-m) and the state
// enters at the end of the sequence):
//   dq_n = sum_{m<=n} g^(n-m) (dout_n . v_m) k_m + g^(n+1) dout_n S0^T
//        = F(dout, v, k; S0^T)
//   dv_m = sum_{n>=m} g^(n-m) (q_n . k_m) dout_n + g^(N-1-m) k_m dS_final
//        = R(k, q, dout; dS_final / g)
//   dk_m = sum_{n>=m} g^(n-m) (dout_n . v_m) q_n + g^(N-1-m) v_m dS_final^T
//        = R(v, dout, q; dS_final^T / g)
//   dS0  = sum_n g^(n+1) q_n^T dout_n + g^N dS_final = g * (final state of the dv pass)
// (in reversed time the state term of row m is g^(N-m) Q' S0', which is g^(N-1-m) Q' dS
// for S0' = dS / g).  The dq and dk passes have a 512-wide score dimension (dv): the
// scores are sums over it and the state term is linear in it, so each runs as passes over
// 256-column halves (read in place through pitched tensor maps), the later halves adding
// the earlier ones' output in the kernel's epilogue (in place for fp32 gradients; for bf16
// gradients the partial sums stay fp32 in the workspace until the last half).  The dv pass
// and the dq and dk chains are independent: they run on the caller's stream and two side
// streams, joined back before the call returns.  Small kernels transpose and scale the
// incoming states and form dS0.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
constexpr int kPart = 256;             // width of one half of the 512-wide score dimension

struct BwdWs {
    size_t stq, stk, stv, sout, sc, opq, opk;
    size_t total() const { return stq + stk + stv + sout + sc + opq + opk; }
};

BwdWs bwd_ws(int out_bf16, int b, int H, int N, int dk, int dv) {
    const size_t bh = (size_t)b * H, tok = bh * (size_t)N;
    const size_t parts = (size_t)(dv / kPart);
    BwdWs w;
    w.stq = round_up(parts * bh * kPart * dk * 4);  // S0^T halves
    w.stk = w.stq;                                   // dS^T halves / g
    w.stv = round_up(bh * dk * dv * 4);              // dS / g
    w.sout = w.stv;                                  // final state of the dv pass
    w.sc = round_up(3 * ret::kMaxHeads * sizeof(float));   // per-head scales 1, 1/g, g
    // fp32 partial sums of dq and dk over the halves (bf16 gradients with two or more halves)
    w.opq = (out_bf16 && parts > 1) ? round_up(tok * dk * 4) : 0;
    w.opk = w.opq;
    return w;
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

int grid_for(long long n) {
    long long g = (n + 255) / 256;
    return (int)(g < 148 * 16 ? (g > 0 ? g : 1) : 148 * 16);
}

// Two side streams per device and context, made on first use and kept for the process.
cudaError_t side_streams(cudaStream_t out[2]) {
    static std::mutex mu;
    static cudaStream_t made[ret::kMaxDevices][2] = {};
    static void* ctx[ret::kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= ret::kMaxDevices) return cudaErrorInvalidDevice;
    void* cur = ret::current_context();
    std::lock_guard<std::mutex> lk(mu);
    if (!made[dev][0] || ctx[dev] != cur) {
        // a context made after a device reset: the old streams died with the old context
        for (int i = 0; i < 2; ++i) {
            e = cudaStreamCreateWithFlags(&made[dev][i], cudaStreamNonBlocking);
            if (e != cudaSuccess) { made[dev][0] = made[dev][1] = nullptr; return e; }
        }
        ctx[dev] = cur;
    }
    out[0] = made[dev][0];
    out[1] = made[dev][1];
    return cudaSuccess;
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

size_t chunkwise_backward_tc_workspace(int out_bf16, int b, int H, int N, int dk, int dv) {
    return bwd_ws(out_bf16, b, H, N, dk, dv).total();
}

cudaError_t launch_chunkwise_backward_tc(const void* q, const void* k, const void* v,
                                         const void* dout, void* grad_q, void* grad_k,
                                         void* grad_v, int out_bf16, int b, int H, int N, int dk,
                                         int dv, const HeadConsts& hc256, const float* state_in,
                                         const float* dstate_out, float* dstate_in,
                                         void* workspace, cudaStream_t s) {
    const BwdWs L = bwd_ws(out_bf16, b, H, N, dk, dv);
    uint8_t* p = static_cast<uint8_t*>(workspace);
    auto take = [&](size_t n) { uint8_t* r = p; p += n; return r; };
    float* stq = reinterpret_cast<float*>(take(L.stq));
    float* stk = reinterpret_cast<float*>(take(L.stk));
    float* stv = reinterpret_cast<float*>(take(L.stv));
    float* sout = reinterpret_cast<float*>(take(L.sout));
    float* scales = reinterpret_cast<float*>(take(L.sc));   // [0,H): 1, [H,2H): 1/g, [2H,3H): g
    float* opq = reinterpret_cast<float*>(take(L.opq));
    float* opk = reinterpret_cast<float*>(take(L.opk));
    const int BH = b * H, parts = dv / kPart;

    cudaStream_t side[2];
    cudaError_t e = side_streams(side);
    if (e != cudaSuccess) return e;
    {
        // pageable source: the copy has consumed it when cudaMemcpyAsync returns
        float host[3 * kMaxHeads];
        for (int h = 0; h < H; ++h) {
            host[h] = 1.0f;
            host[H + h] = 1.0f / hc256.g1[h];
            host[2 * H + h] = hc256.g1[h];
        }
        e = cudaMemcpyAsync(scales, host, 3 * H * sizeof(float), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
    }
    // incoming states of the passes
    const int gs = grid_for((long long)BH * dk * dv);
    if (state_in) state_prep_kernel<<<gs, 256, 0, s>>>(state_in, stq, BH, H, dk, dv, 1, scales);
    if (dstate_out) {
        state_prep_kernel<<<gs, 256, 0, s>>>(dstate_out, stk, BH, H, dk, dv, 1, scales + H);
        state_prep_kernel<<<gs, 256, 0, s>>>(dstate_out, stv, BH, H, dk, dv, 0, scales + H);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // fork: the dq chain on side[0], the dk chain on side[1], dv on the caller's stream
    cudaEvent_t ev[3];
    int made = 0;
    for (; made < 3 && e == cudaSuccess; ++made)
        e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        for (int i = 0; i < made - 1; ++i) cudaEventDestroy(ev[i]);
        return e;
    }
    bool forked = false;
    e = cudaEventRecord(ev[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side[0], ev[0], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side[1], ev[0], 0);
    forked = e == cudaSuccess;

    // one chain over the halves of the score dimension: F or R(x_p, y_p, z; st_p), the
    // later halves adding the earlier ones' output
    const char* dob = static_cast<const char*>(dout);
    const char* vb = static_cast<const char*>(v);
    auto chain = [&](const char* xq, const char* xk, const void* xv, const float* st, int rev,
                     void* grad, float* part, cudaStream_t cs) {
        cudaError_t ce = cudaSuccess;
        for (int pp = 0; pp < parts && ce == cudaSuccess; ++pp) {
            const bool last = pp == parts - 1;
            // fp32 gradients accumulate in place; bf16 ones in the fp32 partial buffer
            void* o = (last || !out_bf16) ? grad : part;
            const float* acc = pp == 0 ? nullptr : (out_bf16 ? part : static_cast<const float*>(grad));
            ce = launch_chunkwise_tc_pair(xq + (size_t)pp * kPart * 2, xk + (size_t)pp * kPart * 2, xv,
                                          o, (out_bf16 && last) ? 1 : 0, b, H, N, kPart, dk, 256,
                                          hc256, st ? st + (size_t)pp * BH * kPart * dk : nullptr,
                                          nullptr, cs, 0, 0, dv, dv, dk, dk, rev, acc);
        }
        return ce;
    };
    if (forked) {
        // dq = F(dout, v, k; S0^T)
        e = chain(dob, vb, k, state_in ? stq : nullptr, 0, grad_q, opq, side[0]);
        // dk = R(v, dout, q; dS^T / g)
        if (e == cudaSuccess)
            e = chain(vb, dob, q, dstate_out ? stk : nullptr, 1, grad_k, opk, side[1]);
        // dv = R(k, q, dout; dS / g); its final state gives dS0
        if (e == cudaSuccess)
            e = launch_chunkwise_tc_pair(k, q, dout, grad_v, out_bf16, b, H, N, dk, dv, 256, hc256,
                                         dstate_out ? stv : nullptr, dstate_in ? sout : nullptr, s,
                                         0, 0, 0, 0, 0, 0, 1, nullptr);
        if (e == cudaSuccess && dstate_in) {
            // dS0 = g * (final state of the dv pass)
            state_prep_kernel<<<gs, 256, 0, s>>>(sout, dstate_in, BH, H, dk, dv, 0, scales + 2 * H);
            e = cudaGetLastError();
        }
        // join: the caller's stream waits for both chains, also after an error
        for (int i = 0; i < 2; ++i)
            if (cudaEventRecord(ev[1 + i], side[i]) == cudaSuccess) cudaStreamWaitEvent(s, ev[1 + i], 0);
    }
    for (int i = 0; i < 3; ++i) cudaEventDestroy(ev[i]);
    if (e == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_BACKWARD_TC);
    return e;
}

}  // namespace ret
