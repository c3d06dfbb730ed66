/*
 * retention.h -- C ABI of the RetNet multi-scale retention core on one NVIDIA
 * B300 (sm_103a).  Library: libretention_b300.so (hand-written CUDA kernels).
 *
 * Sources for what each call computes (page title, then section / equation):
 *   [RN2] "Transformer取代者登場！微軟、清華剛推出RetNet：成本低、速度快、性能強（2）"
 *         "Retention" 1) parallel form eq.(5), 2) recurrent form eq.(6),
 *         3) chunkwise recurrent form eq.(7); "門控多尺度 Retention" (per-head
 *         decay, GroupNorm per head, swish gate); "Retention Score 歸一化"
 *         (three score normalisations); "訓練/推理" (eqs.5/7 for training,
 *         eq.6 for decoding).
 *   [RVW] "[論文レビュー] Retentive Network: A Successor to Transformer for Large
 *         Language Models", ABSTRACT (three computation paradigms).
 *
 * Notation: b batch, H heads, N sequence length, dk key/query head dim, dv
 * value head dim, B chunk length, gamma_h the fixed decay of head h.  Indices
 * are 0-based.  Q and K arrive already position-rotated (the xPos factor of
 * [RN2] eqs.(2)-(3) is absorbed into them); inputs are real, so the conjugate
 * transpose of eq.(4) is a transpose.
 *
 * Common rules for every call
 *   - Every tensor pointer (q, k, v, o, y, g, out, state, state_in, state_out,
 *     dout, grad_*, dstate_*, q_out, k_out, x, gate_*, lambda_, h0, h_last) is a
 *     DEVICE pointer to a contiguous row-major array, 16-byte aligned, unless its
 *     declaration says HOST.  The caller owns every buffer; the library allocates
 *     nothing (retention_chunkwise_host_noalloc's file-scope scratch aside).
 *   - gamma is a HOST pointer to H doubles, each in [0, 1].
 *   - Calls are asynchronous on the CUDA stream `stream` (a cudaStream_t; NULL
 *     means the legacy default stream).  Argument checks run on the host
 *     before any launch: a rejected call launches nothing and leaves every
 *     output untouched.  A launch failure returns RET_ERR_CUDA.  Nothing
 *     throws across the ABI.
 *   - Sizes of zero (b, H or N) are valid and launch nothing.
 *   - Supported shapes: 1 <= H <= 128; dk and dv multiples of 16 with
 *     dk <= 256 and dv <= 512; chunk a multiple of 16 in [16, 256] dividing N.
 *     Other values return RET_ERR_UNSUPPORTED (dims, H) or RET_ERR_SHAPE
 *     (chunk / N mismatch, negative sizes).
 *   - Outputs are written in out_dtype (RET_F32 or RET_BF16, round to nearest
 *     even); all accumulation is fp32; recurrent states are always fp32.
 *   - Kernels that wait on on-chip barriers bound every wait; if one gives up
 *     it records the fact in a device-side error word and the kernel returns
 *     early.  retention_check_device_error() reads (and clears) that word.
 */
#ifndef RETENTION_B300_H
#define RETENTION_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RET_OK = 0,
    RET_ERR_NULL = 1,        /* a required pointer is NULL                      */
    RET_ERR_SHAPE = 2,       /* negative size, N % chunk != 0, bad chunk        */
    RET_ERR_DTYPE = 3,       /* dtype code not RET_F32 / RET_BF16               */
    RET_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned                */
    RET_ERR_UNSUPPORTED = 5, /* dims/heads/flags/gamma/eps outside the support  */
    RET_ERR_CUDA = 6,        /* a CUDA launch or runtime call failed            */
    RET_ERR_TIMEOUT = 7      /* a bounded on-chip wait expired inside a kernel  */
} ret_status;

typedef enum { RET_F32 = 0, RET_BF16 = 1 } ret_dtype;

/* Score normalisations of [RN2] "Retention Score 歸一化" (parallel form only). */
#define RET_NORM_SCALE 1u  /* scores q_n.k_m divided by sqrt(dk)                 */
#define RET_NORM_DECAY 2u  /* row n of D divided by sqrt(sum_m D[n][m])          */
#define RET_NORM_ROWSUM 4u /* row n of the scores R divided by max(|sum_m R|, 1) */

/*
 * Parallel form, [RN2] "Retention" 1) eq.(5) with Fig.3a, plus the optional
 * normalisations of "Retention Score 歸一化":
 *   D[n][m]  = gamma_h^(n-m) for n >= m, else 0        (never materialised)
 *   R[n][m]  = (q_n . k_m) [/ sqrt(dk)] * D[n][m] [/ sqrt(sum_i D[n][i])]
 *   R[n][.] /= max(|sum_m R[n][m]|, 1)                  (RET_NORM_ROWSUM)
 *   O        = R V
 * q, k: [b][H][N][dk] in in_dtype; v: [b][H][N][dv] in in_dtype;
 * o: [b][H][N][dv] in out_dtype (written).  flags: OR of RET_NORM_*.
 */
int retention_parallel(const void* q, const void* k, const void* v, void* o,
                       ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                       int dk, int dv, const double* gamma, unsigned flags, void* stream);

/*
 * Chunkwise recurrent form, [RN2] "Retention" 3) eq.(7): parallel inside each
 * chunk of length B = chunk, recurrent across chunks.  For chunk i (rows
 * iB..iB+B-1; j, r index rows inside the chunk):
 *   O[iB+j] = sum_{r<=j} (q_j . k_r) gamma^(j-r) v_r + gamma^(j+1) (q_j R_{i-1})
 *   R_i     = sum_r gamma^(B-1-r) k_r^T v_r + gamma^B R_{i-1}
 * R_{-1} = state_in (NULL means zero).  If state_out is not NULL it receives
 * the final state R_{N/B-1}; state_in and state_out may alias.
 * q, k: [b][H][N][dk]; v: [b][H][N][dv] (in_dtype); o: [b][H][N][dv] (out_dtype);
 * state_in, state_out: [b][H][dk][dv] fp32.  No score normalisation.
 * Requires N % chunk == 0 (RET_ERR_SHAPE otherwise).
 * The chunk length orders the work but does not change the function: R_i carries every
 * token before chunk i exactly, so every chunk length gives the same O and final state up
 * to rounding.  bf16 inputs run on the pair-of-SMs tensor-core kernel with 256-token
 * chunks whenever it applies (dk 256, dv a multiple of 128, N a multiple of 256, every
 * gamma^(-256) <= 2^64), whatever the caller's chunk; otherwise with the caller's chunk;
 * otherwise with 128-token chunks when N splits into them and every gamma^(-128) <= 2^64
 * (a chunk below 128 has no tensor-core schedule of its own); otherwise on CUDA cores
 * (retention_last_kernel names the kernel).
 * fp32 inputs and every other case use the caller's chunk.
 */
int retention_chunkwise(const void* q, const void* k, const void* v, void* o,
                        ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                        int dk, int dv, int chunk, const double* gamma,
                        const float* state_in, float* state_out, void* stream);

/*
 * Gradient of retention_chunkwise.  [RN2] "訓練/推理" trains with the parallel and
 * chunkwise forms; the pages print no backward pass, so this is the exact derivative
 * of eq.(7) ([RN2] "Retention" 3)), which is the same function for every chunk length.
 * With S0 = state_in (NULL means zero) and the scalar
 *   L = sum_n dout_n . o_n + <dstate_out, S_final>      (dstate_out NULL means zero)
 * the call writes
 *   grad_q[n] = sum_{m<=n} gamma^(n-m) (dout_n . v_m) k_m + gamma^(n+1) dout_n S0^T
 *   grad_k[m] = sum_{n>=m} gamma^(n-m) (dout_n . v_m) q_n + gamma^(N-1-m) v_m dstate_out^T
 *   grad_v[m] = sum_{n>=m} gamma^(n-m) (q_n . k_m) dout_n + gamma^(N-1-m) k_m dstate_out
 *   dstate_in = sum_n gamma^(n+1) q_n^T dout_n + gamma^N dstate_out   (if not NULL)
 * computed chunk by chunk: grad_q by the forward scan of eq.(7) with (q, k, v) replaced
 * by (dout, v, k); grad_k and grad_v by the same scan run from the last chunk to the
 * first with the carried gradient of the state.  One CUDA-core kernel launch.  chunk is
 * validated as in retention_chunkwise; since the result does not depend on it, the
 * kernel scans in chunks of 64 tokens whenever N is a multiple of 64.
 * q, k: [b][H][N][dk], v, dout: [b][H][N][dv], all in in_dtype; grad_q, grad_k:
 * [b][H][N][dk] and grad_v: [b][H][N][dv] in out_dtype (written; must not overlap the
 * inputs); state_in, dstate_out, dstate_in: [b][H][dk][dv] fp32, nullable
 * (dstate_in must not overlap the others).  All DEVICE pointers.  Shapes and
 * errors as in retention_chunkwise; N = 0 writes dstate_in = dstate_out (or zero).
 */
int retention_chunkwise_backward(const void* q, const void* k, const void* v,
                                 const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                 ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                                 int dk, int dv, int chunk, const double* gamma,
                                 const float* state_in, const float* dstate_out,
                                 float* dstate_in, void* stream);

/*
 * retention_chunkwise_backward on tensor cores, with a caller workspace.  Every gradient
 * above is itself a retention of the forward kind, so the call runs it as passes of the
 * pair-of-SMs chunkwise kernel (chunk 256; the result does not depend on the chunk):
 *   grad_q = F(dout, v, k; S0^T),  grad_v = R(k, q, dout; dstate_out/gamma),
 *   grad_k = R(v, dout, q; dstate_out^T/gamma),  dstate_in = gamma * (final state of the
 *   grad_v pass),
 * where F is eq.(7) with (q, k, v, state_in) replaced as written and R is eq.(7) in
 * reversed time (row n collects the rows m >= n with gamma^(m-n), the state entering at
 * the end of the sequence).  The dv-wide score dimension of the grad_q and grad_k passes
 * runs as 256-column slices whose outputs add inside the kernel.  The grad_v pass and the
 * grad_q and grad_k chains run concurrently: on stream and on two side streams that the
 * library makes on the first call on a device (make that call before capturing stream
 * into a graph) and keeps; stream waits for both before the call returns, also on an
 * error, and the library creates and releases three CUDA events per call.
 * Applies to bf16 inputs with dk = 256, dv a multiple of 256, N a multiple of 256 and
 * every gamma in (0, 1] with gamma^(-256) <= 2^64; workspace (DEVICE,
 * retention_chunkwise_backward_workspace_bytes(out_dtype, ...) bytes, 256-byte aligned,
 * owned by the caller and not touched by anything else until stream reaches this call's
 * end) then holds the transposed states and, for bf16 gradients, fp32 partial sums.
 * Other shapes run the CUDA-core kernel of retention_chunkwise_backward and leave the
 * workspace untouched (it may then be NULL).  Arguments, layouts and errors otherwise as
 * retention_chunkwise_backward; a workspace that is too small returns RET_ERR_SHAPE.
 */
int retention_chunkwise_backward_ws(const void* q, const void* k, const void* v,
                                    const void* dout, void* grad_q, void* grad_k, void* grad_v,
                                    ret_dtype in_dtype, ret_dtype out_dtype, int b, int H,
                                    int N, int dk, int dv, int chunk, const double* gamma,
                                    const float* state_in, const float* dstate_out,
                                    float* dstate_in, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Workspace bytes of retention_chunkwise_backward_ws for gradients of out_dtype (0 for
 * negative sizes and for shapes the tensor-core passes do not take).  Host-side. */
size_t retention_chunkwise_backward_workspace_bytes(ret_dtype out_dtype, int b, int H, int N,
                                                    int dk, int dv);

/*
 * retention_chunkwise over HOST-resident inputs and outputs.  The sequence passes
 * through the device in segments of seg_len tokens (a multiple of chunk dividing N);
 * eq.(7) carries the state across any split at a chunk boundary ([RN2] "Retention" 3)),
 * so each segment continues from the fp32 state the previous one left in the workspace
 * and the result is that of one retention_chunkwise call over the whole sequence.
 * Per segment: host-to-device copies of Q, K, V on h2d_stream (one 2-D copy each),
 * the chunkwise call on stream, the device-to-host copy of O on d2h_stream; two
 * buffer sets alternate, so one segment's copies overlap its neighbours' compute.
 *
 * q, k: [b][H][N][dk], v: [b][H][N][dv] (in_dtype), o: [b][H][N][dv] (out_dtype), all
 * HOST pointers, 16-byte aligned; pinned (page-locked) memory makes the copies
 * asynchronous.  state_in, state_out: DEVICE pointers [b][H][dk][dv] fp32, nullable,
 * as in retention_chunkwise.  workspace: DEVICE memory of at least
 * retention_chunkwise_host_workspace_bytes(...) bytes, 256-byte aligned, owned by the
 * caller and not touched by anything else until stream reaches this call's end.
 * h2d_stream, d2h_stream: two further streams (cudaStream_t) for the copies, distinct
 * from stream and from each other for the copies to overlap.  The call returns once
 * everything is enqueued; all of its work is ordered on stream (the copy streams first
 * wait for the work queued on stream before the call, and stream waits for the last
 * copy).  The library creates and releases a few CUDA events inside the call.
 * Argument checks (those of retention_chunkwise, plus seg_len > 0 with seg_len % chunk
 * == 0 and N % seg_len == 0, and the workspace size: RET_ERR_SHAPE) run before the
 * first copy.  A CUDA error or a failed segment returns its status; earlier segments
 * may then have been written, and stream still waits for the copies already queued on
 * the copy streams (so the workspace is free once stream reaches that point).
 */
int retention_chunkwise_host(const void* q, const void* k, const void* v, void* o,
                             ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                             int dk, int dv, int chunk, const double* gamma,
                             const float* state_in, float* state_out, int seg_len,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* h2d_stream, void* d2h_stream);

/*
 * Bytes of device workspace retention_chunkwise_host needs for these dtypes and sizes
 * (the carried state and two segment buffer sets); 0 for invalid dtypes or negative
 * sizes.  Host-side, no GPU access.
 */
size_t retention_chunkwise_host_workspace_bytes(ret_dtype in_dtype, ret_dtype out_dtype, int b,
                                                int H, int dk, int dv, int seg_len);

/*
 * retention_chunkwise_host without a caller workspace: the carried state and the segment
 * buffers live in a file-scope device array of retention_chunkwise_host_static_scratch_bytes()
 * bytes, reserved on each device when the library's module loads there; its address is
 * looked up on the first call on a device (and again if that device's context changed,
 * e.g. after cudaDeviceReset), so make that first call before any stream capture.
 * Arguments and behaviour otherwise as retention_chunkwise_host.
 * A call whose workspace (retention_chunkwise_host_workspace_bytes) exceeds the scratch
 * returns RET_ERR_SHAPE, like every other argument check, before any device access.  The
 * scratch is shared by all calls on a device: they must not overlap in time (issue them
 * on one stream, or synchronise between them).
 */
int retention_chunkwise_host_noalloc(const void* q, const void* k, const void* v, void* o,
                                     ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                                     int dk, int dv, int chunk, const double* gamma,
                                     const float* state_in, float* state_out, int seg_len,
                                     void* stream, void* h2d_stream, void* d2h_stream);

/* Bytes of the static scratch behind retention_chunkwise_host_noalloc.  Host-side. */
size_t retention_chunkwise_host_static_scratch_bytes(void);

/*
 * One decode step of the recurrent form, [RN2] "Retention" 2) eq.(6) and the
 * inference paragraph of "訓練/推理" (O(1) state per token):
 *   S <- gamma_h S + k^T v     (in place, fp32)
 *   o  = q S                   (read from the UPDATED state)
 * q, k: [b][H][dk]; v: [b][H][dv] (in_dtype); state: [b][H][dk][dv] fp32, read
 * and overwritten; o: [b][H][dv] (out_dtype).  dv must be a multiple of 16.
 */
int retention_recurrent_step(const void* q, const void* k, const void* v, float* state,
                             void* o, ret_dtype in_dtype, ret_dtype out_dtype, int b, int H,
                             int dk, int dv, const double* gamma, void* stream);

/*
 * Gated multi-scale retention epilogue, [RN2] "門控多尺度 Retention":
 *   per (batch, token n, head h): mu, var = mean and biased variance of the dv
 *   values y[b][h][n][:];  yhat = (y - mu) / sqrt(var + eps) [* weight + bias];
 *   out[b][n][h*dv + c] = swish(g[b][n][h*dv + c]) * yhat[c],  swish(x) = x sigmoid(x).
 * y: [b][H][N][dv] (y_dtype, head-major as the retention calls write it);
 * g, out: [b][N][H*dv] (token-major like X W_G); weight, bias: H*dv floats on
 * the DEVICE, each nullable (identity).  eps >= 0.  The output projection W_O
 * is not part of this call.
 */
int msr_epilogue(const void* y, const void* g, void* out, ret_dtype y_dtype,
                 ret_dtype g_dtype, ret_dtype out_dtype, int b, int H, int N, int dv,
                 float eps, const float* weight, const float* bias, void* stream);

/*
 * Parallel form and gated epilogue in one pass ([RN2] "Retention" 1) eq.(5) with the
 * factors of "Retention Score 歸一化", then "門控多尺度 Retention"); the retention output
 * Y is never written to memory:
 *   Y[b][h][n][:] = retention_parallel(q, k, v, gamma, flags) for that (b, h, n)
 *   out[b][n][h*dv + c] = swish(g[b][n][h*dv + c]) * GN(Y[b][h][n][:])[c]
 *   GN(y)[c] = (y[c] - mean(y)) / sqrt(var(y) + eps) [* weight[h*dv+c] + bias[h*dv+c]]
 * (biased variance over the dv values of one (token, head)).
 * q, k: [b][H][N][dk], v: [b][H][N][dv] in in_dtype; g, out: [b][N][H*dv] (token-major)
 * in g_dtype / out_dtype; weight, bias: H*dv floats on the DEVICE, each nullable.
 * Tensor-core shapes only: in_dtype RET_BF16, dk in {128, 256}, dv a multiple of 128 and
 * at most 512, N >= 128.  Other shapes return RET_ERR_UNSUPPORTED before any launch;
 * retention_parallel followed by msr_epilogue computes the same result for them.
 */
int retention_parallel_gated(const void* q, const void* k, const void* v, const void* g,
                             void* out, ret_dtype in_dtype, ret_dtype g_dtype,
                             ret_dtype out_dtype, int b, int H, int N, int dk, int dv,
                             const double* gamma, unsigned flags, float eps,
                             const float* weight, const float* bias, void* stream);

/*
 * xPos rotation of Q and K, [RN2] "Retention" eqs.(2)-(3) (formulas lost, prose kept):
 * Q_n e^{i n theta} and K_m e^{i m theta}, "a relative position embedding", so that the
 * retention score of eq.(4), taken with the conjugate transpose, depends on n - m only.
 * For real inputs each pair of coordinates (2j, 2j+1) is one complex number:
 *   out[.., n, 2j]   = x[.., n, 2j] cos(p theta_j) - x[.., n, 2j+1] sin(p theta_j)
 *   out[.., n, 2j+1] = x[.., n, 2j] sin(p theta_j) + x[.., n, 2j+1] cos(p theta_j)
 * at position p = pos0 + n.  Apply it to Q and K before retention_parallel,
 * retention_chunkwise or retention_recurrent_step (pos0 = the first token's position).
 * q, k: [b][H][N][dk] in in_dtype; q_out, k_out: the same shape in out_dtype.  k may
 * be NULL (then k_out is ignored and only q is rotated).  q_out may equal q (and k_out
 * k) when in_dtype == out_dtype; other overlaps are not allowed.  theta: HOST array of
 * dk/2 finite doubles.  dk as for the retention calls.  One memory-bound launch.
 */
int retention_xpos_rotate(const void* q, const void* k, void* q_out, void* k_out,
                          ret_dtype in_dtype, ret_dtype out_dtype, int b, int H, int N,
                          int dk, const double* theta, long long pos0, void* stream);

/*
 * RG-LRU scan, the gated diagonal linear recurrence of the Griffin page ("Griffin ：
 * 將門控線性循環與局部注意力混合以實現高效的語言模型", section "實門線性循環單元
 * (RG-LRU)"), from the pre-activations of its two gates (the projections
 * W_a x_t + b_a and W_x x_t + b_x are plain matrix products, not part of this call):
 *   r_t = sigmoid(gate_a_t), i_t = sigmoid(gate_x_t), a = sigmoid(lambda[d]),
 *   a_t = a^(c r_t),  h_t = a_t h_{t-1} + sqrt(1 - a_t^2) (i_t x_t),  y_t = h_t,
 * elementwise over the D channels, sequential over t, h_{-1} = h0 (NULL means zero);
 * a_t is evaluated in log space.  The page fixes c = 8.
 * x, gate_a, gate_x: [b][T][D] in in_dtype; y: [b][T][D] in out_dtype (written, must
 * not overlap the inputs); lambda: [D] fp32; h0, h_last: [b][D] fp32, nullable
 * (h_last receives h_{T-1}, or h0 when T = 0).  All DEVICE pointers, 16-byte aligned.
 * D must be a multiple of 64 (RET_ERR_UNSUPPORTED), c finite and >= 0
 * (RET_ERR_UNSUPPORTED); negative sizes return RET_ERR_SHAPE; b, T or D of zero launch
 * nothing (T = 0 still writes h_last).  One memory-bound kernel launch: each CTA owns
 * 64 channels; its warps scan consecutive segments of t from a zero state and combine
 * them with the (prod a_t, h_end) pairs of the segments before them.
 */
int rglru_scan(const void* x, const void* gate_a, const void* gate_x, const float* lambda_,
               const float* h0, void* y, float* h_last, ret_dtype in_dtype,
               ret_dtype out_dtype, int b, int T, int D, float c, void* stream);

/* Static text for a ret_status code ("unknown status" for other values). */
const char* retention_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device-side error word of
 * the current device.  Returns RET_ERR_TIMEOUT if any kernel since the last
 * check gave up on a bounded wait, RET_ERR_CUDA if the synchronisation itself
 * failed, RET_OK otherwise.
 */
int retention_check_device_error(void* stream);

/*
 * The gated multi-scale retention layer, [RN2] "門控多尺度 Retention" (its formula was lost
 * in extraction; the prose names every step): per head h,
 *   Q_h = xPos(X W_Q[:, h*dk..]), K_h = xPos(X W_K[:, h*dk..]), V_h = X W_V[:, h*dv..],
 *   Y_h = retention(Q_h, K_h, V_h, gamma_h)   (parallel form with `flags`, or the
 *                                             chunkwise form with chunk > 0, unnormalised)
 *   out = (swish(X W_G) (.) GroupNorm_h(Y)) W_O            (eps as in msr_epilogue)
 * xPos ([RN2] "Retention" eqs.(2)-(3)) as in retention_xpos_rotate, at positions
 * pos0 + n; theta NULL means no rotation.
 * x: [b][N][d_model] bf16; wq, wk: [d_model][H*dk]; wv, wg: [d_model][H*dv];
 * wo: [H*dv][d_out], all bf16 row-major DEVICE arrays (x W as the layer applies them);
 * out: [b][N][d_out] in out_dtype; gamma: HOST, H doubles in [0, 1]; theta: HOST, dk/2
 * doubles or NULL.  workspace: DEVICE memory of retention_msr_layer_workspace_bytes(...)
 * bytes, 256-byte aligned, owned by the caller (Q, K, V, G and the gated rows live there,
 * bf16).  Supported: dk in {128, 256}, dv a multiple of 128 (<= 512), d_model a multiple
 * of 64, H*dk, H*dv and d_out multiples of 256, N >= 128 for the parallel form
 * (RET_ERR_UNSUPPORTED otherwise); flags must be 0 with chunk > 0.  Asynchronous on
 * `stream`: six kernels (four projections, retention with the gated epilogue fused --
 * chunkwise: retention then msr_epilogue --, the output projection).
 */
int retention_msr_layer(const void* x, const void* wq, const void* wk, const void* wv,
                        const void* wg, const void* wo, void* out, ret_dtype out_dtype, int b,
                        int N, int d_model, int H, int dk, int dv, int d_out,
                        const double* gamma, const double* theta, long long pos0,
                        unsigned flags, float eps, int chunk, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Workspace bytes of retention_msr_layer (0 for negative sizes).  Host-side. */
size_t retention_msr_layer_workspace_bytes(int b, int N, int H, int dk, int dv, int chunk);

/*
 * One projection of the layer: C = A W, A: [M][K] bf16, W: [K][Nc] bf16 (row-major DEVICE
 * arrays), C: [M][Nc] in c_dtype, fp32 accumulation (tensor cores).  Nc % 256 == 0 and
 * K % 64 == 0 (RET_ERR_UNSUPPORTED otherwise); any M.
 */
int retention_gemm(const void* a, const void* w, void* c, ret_dtype c_dtype, int M, int Nc, int K,
                   void* stream);

/*
 * The per-head projection of the layer: out[b][h][n][:] = (x[b][n][:] W)[h*d .. h*d+d-1],
 * head-major bf16 rows as the retention calls read them, rotated by xPos at position
 * pos0 + n when theta (HOST, d/2 doubles) is not NULL -- the rotation of
 * retention_xpos_rotate, fused into the projection.  x: [b][N][d_in] bf16, W: [d_in][H*d]
 * bf16 (DEVICE).  d a multiple of 64 (<= 256), H*d a multiple of 256, d_in of 64.
 */
int retention_project_heads(const void* x, const void* w, void* out, int b, int N, int d_in, int H,
                            int d, const double* theta, long long pos0, void* stream);

/*
 * Diagnostics of the tensor-core chunkwise kernel for chunk 256, dk 256 (pairs of SMs):
 * it computes the score x value and query x state products with fp16 operands and, if a
 * value it rounds to fp16 lies outside fp16's range (|x| >= 65504), re-runs that unit
 * (one batch x head x 128 value columns) in a bf16 hi/lo format with fp32's range, inside
 * the same launch; the result is correct either way.  This call synchronises `stream` and
 * returns the number of such re-runs since the previous call (and resets the count), or
 * -1 if the synchronisation failed.  Host-side; for tests and diagnostics.
 */
int retention_chunkwise_format_reruns(void* stream);

/*
 * The same diagnostic for the parallel form on pairs of SMs (dk 256, dv and N multiples of
 * 256): P and V enter the score x value product as fp16; a unit whose P or V leaves fp16's
 * range, or whose largest |v| is below 2^-6 (typical values then near fp16's subnormals),
 * is recomputed with hi/lo bf16 P inside the same launch.  Counts clusters (the value-column
 * blocks of a query block with the fused epilogue, else one SM pair) that re-ran.
 */
int retention_parallel_format_reruns(void* stream);

/*
 * Self-test of the bounded on-chip waits (the pages describe no fault handling; this is the
 * library's own).  Launches the pair-of-SMs chunkwise kernel on b1 H1 N256 dk256 dv128
 * (q, k: 256 x 256 bf16, v: 256 x 128 bf16, o: 256 x 128 fp32, DEVICE buffers that are
 * neither read nor written) with every wait limited to 1 ms and a TMA producer that issues
 * no load: each wait expires, the kernel unwinds with no copy or MMA in flight, frees its
 * tensor memory and sets the device error word, so that the next
 * retention_check_device_error() returns RET_ERR_TIMEOUT.  The device stays usable.
 * Asynchronous on `stream`; returns RET_ERR_NULL / RET_ERR_ALIGN for bad pointers.
 */
int retention_chunkwise_wait_selftest(const void* q, const void* k, const void* v, void* o,
                                      void* stream);

/*
 * Number of kernels this library has launched in this process so far (all
 * devices, all calls).  Host-side counter, incremented after each successful
 * launch; lets callers count launches inside a timed region.
 */
unsigned long long retention_kernel_launches(void);

/*
 * cudaError_t value of the most recent CUDA failure (launch, attribute or
 * runtime call) that made a call of this host thread return RET_ERR_CUDA,
 * 0 if none.  Host-side, per thread; never cleared by successful calls.
 */
int retention_last_cuda_error(void);

/* Static name and description of a cudaError_t value, e.g. "cudaErrorLaunchOutOfResources: ...". */
const char* retention_cuda_error_string(int cuda_error);

/* Kernel codes reported by retention_last_kernel(). */
enum {
    RET_KERNEL_NONE = 0,
    RET_KERNEL_PARALLEL_SIMT = 1,   /* parallel form, CUDA-core fp32 FMA kernel       */
    RET_KERNEL_CHUNKWISE_SIMT = 2,  /* chunkwise form, CUDA-core fp32 FMA kernel      */
    RET_KERNEL_DECODE = 3,          /* recurrent step                                 */
    RET_KERNEL_EPILOGUE = 4,        /* GroupNorm + swish gate                         */
    RET_KERNEL_CHUNKWISE_TC = 5,    /* chunkwise form, tcgen05 tensor-core kernel     */
    RET_KERNEL_PARALLEL_TC = 6,     /* parallel form, tcgen05 tensor-core kernel      */
    RET_KERNEL_PARALLEL_GATED_TC = 7, /* parallel form + gated GroupNorm, tensor cores */
    RET_KERNEL_CHUNKWISE_TC_PAIR = 8, /* chunkwise form, tensor cores on pairs of SMs */
    RET_KERNEL_CHUNKWISE_BACKWARD_SIMT = 9, /* chunkwise gradient, CUDA-core fp32 FMA   */
    RET_KERNEL_RGLRU = 10,          /* RG-LRU scan                                    */
    RET_KERNEL_XPOS = 11,           /* xPos rotation of Q and K                       */
    RET_KERNEL_GEMM_TC = 12,        /* projection GEMM of the layer, tensor cores     */
    RET_KERNEL_CHUNKWISE_BACKWARD_TC = 13, /* chunkwise gradient as pair-kernel passes  */
    RET_KERNEL_PARALLEL_TC_PAIR = 14, /* parallel form, tensor cores on pairs of SMs      */
    RET_KERNEL_PARALLEL_GATED_TC_PAIR = 15 /* parallel form + gated GroupNorm, SM pairs  */
};

/*
 * Code of the kernel the calling host thread launched last (RET_KERNEL_*),
 * or RET_KERNEL_NONE if it has launched none.  Host-side, per thread.
 */
int retention_last_kernel(void);

#ifdef __cplusplus
}
#endif
#endif /* RETENTION_B300_H */
