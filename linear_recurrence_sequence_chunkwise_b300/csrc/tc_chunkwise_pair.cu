// tc_chunkwise_pair.cu -- chunkwise recurrent retention on pairs of SMs (tcgen05 cta_group::2).
//
// Computes eq.(7) of "Transformer取代者登場！…RetNet…（2）", section "Retention" 3), the same
// function as tc_chunkwise.cu:
//     O[iB+j] = sum_{r<=j} (q_j.k_r) g^(j-r) v_r + g^(j+1) (q_j R_{i-1})
//     R_i     = sum_r g^(B-1-r) k_r^T v_r + g^B R_{i-1}
// for bf16 Q/K/V, fp32 accumulation and state, chunk B = 256, dk = 256, dv a multiple of
// 128.
//
// Decay folding (no per-element power): V rows are scaled by a zeta_r with zeta_r =
// g^(B-1-r) and a constant a (Vz), the scores only masked (P = S (.) M), the state copy
// that Q multiplies by c = a g^B (R' = c R), and each output row by xi_j = g^(j+1-B) / a:
//     xi_j (P Vz + Q R')_j = sum_{r<=j} S_jr g^(j-r) v_r + g^(j+1) q_j R.
// Tensor memory keeps R~ = a R, whose update R~ <- g^B R~ (one TMEM pass per chunk), then
// R~ += K^T Vz, takes Vz as it is; the copy is R' = g^B R~, state_in enters times a and
// state_out leaves times 1/a.  a is the power of two nearest g^(-B/2): splitting g^(-B)
// evenly between Vz and xi keeps both within about g^(-B/2), and the state passes in and
// out exactly.  In the reversed-time mode row r stands at position B-1-r (zeta_r = g^r,
// xi_j = g^(-j) / a), the mask keeps keys r >= j and the chunks run from the last.
//
// Operand formats.  S = Q K^T and R += K^T Vz take bf16 operands as loaded (exact products).
// The two products whose operands are computed take fp16 (11 significant bits, 8x finer
// than bf16): O += P Vz16 with P and Vz16 = fp16(Vz), and O = Q16 R'16 with Q converted to
// fp16 in shared memory once S has read it (bf16 -> fp16 is exact in fp16's normal range)
// and R'16 = fp16(c R).  A CPU emulation of these rounding points on the long-sequence
// workload (heads 0, 5, 15) gives max errors of 0.009, 0.009 and 0.002 of the head's RMS,
// against 0.013, 0.009 and 0.001 for bf16 hi/lo pairs of P and R' (two MMAs each).
// fp16 holds |x| < 65504 only: every conversion tracks the largest magnitude it rounds,
// and if any exceeds the range the pair re-runs its whole unit (same kernel, second pass)
// with the hi/lo bf16 pairs instead, which have fp32's range.  The host picks the hi/lo
// format from the start when g^(-B) > 4096 for some head (small decays underflow Vz16).
//
// Work split: one cluster of two CTAs (the two SMs of a pair) per (batch*head, 128-column
// block of dv); the even CTA issues every MMA as a pair MMA (M = 256, 128 rows per SM):
//   S  = Q K^T        M = 256 query rows of the chunk (CTA r: rows 128r..), N = 256 keys
//                     (B operand split: CTA r holds keys 128r..), K = dk
//   O  = Q R'         N = 128 value columns (B split: CTA r holds the copy of
//                     R'[:, 64r..64r+63]), K = dk (fp16: one MMA per K step; hi/lo: two)
//   R += K^T Vz       M = 256 dk rows (CTA r: dk 128r..; the state lives in tensor memory,
//                     split by dk), N = 128 value columns, K = 256 keys
//   O += P Vz         A = P from tensor memory, N = 128, K = 256 keys
// Every MMA has N >= 128 per SM, and each SM reads only its half of each B operand.  The
// pair costs one duplicated quarter of the score tile (the even CTA's rows against keys
// 128-255, all masked) and of P.V.
//
// Roles (576 threads = 18 warps per CTA):
//   warp 0      TMA loads of this CTA (Q, K and the K^T operand complete on the even CTA's
//               barriers, V on a local one) and L2 prefetches one chunk ahead
//   warp 1      tensor-memory allocation (both CTAs, collectively); in the even CTA the
//               MMA issuer
//   warps 2-9   V -> Vz and Vz16 (one key row per thread), then scores -> P (two warps per
//               TMEM lane quarter, one per 128-key half), then the chunk's output rows
//               (one per 64-column half), coalesced stores
//   warps 10-17 state copy (10-13 this CTA's own 64 value columns, 14-17 the peer's, into
//               the peer's shared memory in 64-byte row pieces) with R~ <- g^B R~, then
//               Q -> fp16 in place (one row of one dk box per thread: dk 0-127 after S's
//               first half, dk 128-255 after its second)
// Warp w reaches TMEM lanes 32*(w%4)..+31.  Every wait is bounded; a wait that gives up
// sets the device error word and both CTAs' abort flags, and the CTAs unwind, meet at a
// final cluster barrier and free their tensor memory.  Warp signals use CTA-scope release
// arrives: each publishes tensor memory (after tcgen05.fence::before_thread_sync) or shared
// memory that a proxy fence has made visible to the tensor cores reading it; a cluster-scope
// release would also wait for the output warps' global stores to be acknowledged.
//
// Tensor memory per CTA (512 columns x 128 lanes, fp32):
//   [  0,256) S: this CTA's 128 query rows x 256 keys; P written in place, per 32 keys
//             (32 columns of S): fp16 pairs in the first 16 columns (hi/lo format: bf16 hi
//             pairs in the first 16, lo pairs in the next 16)
//   [256,384) O: this CTA's 128 query rows x 128 value columns
//   [384,512) R: this CTA's 128 dk rows of the state x 128 value columns
// Shared memory per CTA (1024-aligned, 224 KB), each box 128 rows x 64 16-bit values, 128B
// swizzle:
//   Q    64 KB  own 128 query rows x 4 dk boxes (bf16 for S, then fp16 for Q.R)
//   K    64 KB  own 128 keys x 4 dk boxes (S); after S the K^T operand of the state update:
//               key block j (keys 128j..) x own 128 dk columns in boxes 2j, 2j+1.  The own
//               key block's boxes stay from S; the peer key block is loaded into the two
//               boxes S no longer needs (the same offsets in both CTAs)
//   V    32 KB  256 keys x own 64 value columns (scaled in place to bf16 Vz)
//   V16  32 KB  fp16 Vz (hi/lo format: the lo part of R')
//   R16  32 KB  fp16 R' = c R_{i-1} = g^B R~: 256 dk rows x own 64 columns (hi/lo: hi part)
// MMA order in a chunk: S (dk boxes 0-1, then 2-3), Q.R' (dk 0-127, then 128-255), K^T.Vz
// (key block 0, then 1), P.Vz.  Commits between the halves free shared memory early:
// after S's first half the odd CTA loads its peer key block (boxes 0-1) and Q's first half
// is converted, after its second half the even CTA loads (boxes 2-3); after K^T.Vz's first
// half the next chunk's keys load into boxes 0-1.
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_chunkwise_pair;
__device__ unsigned g_reruns_chunkwise_pair;   // units re-run in the hi/lo bf16 format

using namespace tc;

constexpr int kThreads = 576;
constexpr int kB = 256;                        // chunk length
constexpr int kDk = 256;
constexpr int kBox = 128 * 128;                // 128 rows x 64 16-bit values
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + 4 * kBox;
constexpr int kVOff = kKOff + 4 * kBox;
constexpr int kV16Off = kVOff + 2 * kBox;
constexpr int kR16Off = kV16Off + 2 * kBox;
constexpr int kSmemBytes = kR16Off + 2 * kBox;  // 229376
constexpr uint32_t kTS = 0, kTO = 256, kTR = 384;
constexpr uint32_t kPairArrivals = 16;         // 8 warps in each CTA
constexpr uint16_t kBoth = 3;                  // multicast mask: both CTAs of the pair
constexpr int kFirstP = 2, kFirstR = 10;       // first warp of each transform group
constexpr float kF16Max = 65504.0f;

struct Decay {
    float l2g[kMaxHeads];   // log2(gamma)
    float gB[kMaxHeads];    // gamma^B
    float l2a[kMaxHeads];   // log2 a: the integer nearest -B log2(gamma) / 2
    float a[kMaxHeads];     // a = 2^l2a ~ gamma^(-B/2): score scale, carried by Vz and the
                            // stored state (a power of two: state_in and state_out pass exactly)
    float ia[kMaxHeads];    // 1 / a
};

struct Bars {
    // the even CTA's copies count both CTAs' work
    uint64_t q_full, k_full0, k_full1;             // pair loads: Q; K dk boxes 0-1 / 2-3
    uint64_t kt_full0, kt_full1;                   // peer key block of K^T in boxes 0-1 / 2-3
    uint64_t vz_ready, p_ready, o_free;            // warp arrivals of both CTAs
    uint64_t rcopy;                                // state copy, 8 warps of each CTA
    uint64_t q16_0, q16_1;                         // Q halves in fp16, 8 warps of each CTA

    // each CTA's own copy, arrived on by the MMA commits (multicast)
    uint64_t q_empty;                              // Q.R done: Q area free
    uint64_t s_half, s_full;                       // S done with dk boxes 0-1 / all of S
    uint64_t kt_empty0, kt_empty1;                 // K^T.Vz done with boxes 0-1 / 2-3
    uint64_t v_empty, o_full, r_done;              // P.Vz done (V free, O complete); K^T.Vz done
    uint64_t v_full;                               // local V load
    uint64_t drain;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16_lo(hi), x1 - bf16_hi(hi));
}

template <bool OUT_BF16, bool ACC, bool REV>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
chunkwise_pair_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv,
                      void* __restrict__ out_base, const float* __restrict__ state_in,
                      float* __restrict__ state_out, int N,
                      int H, int dv, int fp16_first, const Decay dc, uint64_t wait_ns,
                      int no_loads, int ldo, const float* __restrict__ acc) {
    constexpr bool rev = REV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sq = sm + kQOff;
    uint8_t* sk = sm + kKOff;
    uint8_t* sv = sm + kVOff;
    uint8_t* sv16 = sm + kV16Off;
    uint8_t* sr16 = sm + kR16Off;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ int range_flag;                   // an fp16 conversion left fp16's range

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int nblk = dv / 128;
    const int pair = (int)(blockIdx.x >> 1);
    const int bh = pair / nblk, blk = pair % nblk;
    const int head = bh % H;
    const int nchunks = N / kB;
    volatile int* abort_p = &abort_flag;
    volatile int* range_p = &range_flag;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        range_flag = 0;
        mbar_init(&bars.q_full, 1); mbar_init(&bars.k_full0, 1); mbar_init(&bars.k_full1, 1);
        mbar_init(&bars.kt_full0, 1); mbar_init(&bars.kt_full1, 1);
        mbar_init(&bars.vz_ready, kPairArrivals); mbar_init(&bars.p_ready, kPairArrivals);
        mbar_init(&bars.o_free, kPairArrivals); mbar_init(&bars.rcopy, kPairArrivals);
        mbar_init(&bars.q16_0, kPairArrivals); mbar_init(&bars.q16_1, kPairArrivals);
        mbar_init(&bars.q_empty, 1); mbar_init(&bars.s_half, 1); mbar_init(&bars.s_full, 1);
        mbar_init(&bars.kt_empty0, 1); mbar_init(&bars.kt_empty1, 1);
        mbar_init(&bars.v_empty, 1); mbar_init(&bars.o_full, 1); mbar_init(&bars.r_done, 1);
        mbar_init(&bars.v_full, 1); mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc_pair(&tmem_slot, 512); tmem_relinquish_pair(); }
    tc_fence_before();
    cluster_sync_all();     // both CTAs' barriers exist before any remote arrive or pair load
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t peer_abort = map_peer(&abort_flag, peer);
    const uint32_t peer_range = map_peer(&range_flag, peer);
    auto fail = [&]() {
        *abort_p = 1;
        st_cluster_s32(peer_abort, 1);
        atomicOr(&g_err_chunkwise_pair, 1u);
    };
    auto lead = [&](uint64_t* b) { return map_peer(b, 0); };
    // a conversion to fp16 met a magnitude outside fp16's range: both CTAs re-run the unit
    auto out_of_range = [&](float m) {
        if (!(m < kF16Max)) {       // also catches NaN
            *range_p = 1;
            st_cluster_s32(peer_range, 1);
        }
    };
    uint32_t drains = 0;             // MMA drains waited for (MMA issuer)

    // Pass 0 uses the fp16 format (unless the host chose hi/lo); pass 1 runs only if pass 0
    // left fp16's range somewhere in this pair's unit, and recomputes it with hi/lo pairs.
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const bool f16 = fp16_first && pass == 0;
        const int base = pass * nchunks;               // phase index of chunk 0 of this pass
        auto par = [&](int c) { return (uint32_t)(base + c) & 1u; };

        if (warp == 0) {
            // -------------------------------------------------------- TMA producer
            if (lane == 0) {
                if (pass == 0) { tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mv); }
                const uint32_t qf = lead(&bars.q_full), kf0 = lead(&bars.k_full0),
                               kf1 = lead(&bars.k_full1);
                const uint32_t ktf = lead(rank == 0 ? &bars.kt_full1 : &bars.kt_full0);
                const int rowbase = bh * N;
                const int own = 128 * (int)rank, other = 128 * (int)peer;
                const int vcol = blk * 128 + 64 * (int)rank;
                uint32_t armed_q = 0, armed_k = 0, armed_kt = 0, v_loads = 0;
                bool ok = !*abort_p;
                auto w = [&](uint64_t* bar, uint32_t p) {
                    if (ok && !mbar_wait(bar, p, abort_p, wait_ns)) { ok = false; fail(); }
                    return ok;
                };
                // the pairs of one head share Q and K: pull the next chunk's boxes into L2
                auto prefetch = [&](int c) {
                    if (c >= nchunks) return;
                    const int r0 = rowbase + (rev ? nchunks - 1 - c : c) * kB;
                    for (int a = 0; a < 4; ++a) {
                        tma_prefetch_l2(&mq, 64 * a, r0 + own);
                        tma_prefetch_l2(&mk, 64 * a, r0 + own);
                    }
                    for (int m = 0; m < 2; ++m) tma_prefetch_l2(&mk, 64 * (2 * (int)rank + m), r0 + other);
                    for (int j = 0; j < 2; ++j) tma_prefetch_l2(&mv, vcol, r0 + 128 * j);
                };
                // (self-test of the bounded waits: no load is issued, every wait expires)
                if (no_loads) ok = false;
                if (ok) prefetch(0);
                for (int c = 0; c < nchunks && ok; ++c) {
                    const int r0 = rowbase + (rev ? nchunks - 1 - c : c) * kB;
                    // Q: own query rows, all dk (after the previous chunk's Q.R)
                    if (c > 0 && !w(&bars.q_empty, par(c - 1))) break;
                    if (rank == 0) { mbar_arrive_expect_tx(&bars.q_full, 2 * 4 * kBox); ++armed_q; }
                    for (int a = 0; a < 4; ++a) tma_load_2d_pair(sq + a * kBox, &mq, 64 * a, r0 + own, qf);
                    // K: own keys; dk boxes 0-1 once K^T.Vz has read key block 0, boxes 2-3
                    // once it has read key block 1
                    if (c > 0 && !w(&bars.kt_empty0, par(c - 1))) break;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&bars.k_full0, 2 * 2 * kBox);
                        mbar_arrive_expect_tx(&bars.k_full1, 2 * 2 * kBox);
                        ++armed_k;
                    }
                    for (int a = 0; a < 2; ++a) tma_load_2d_pair(sk + a * kBox, &mk, 64 * a, r0 + own, kf0);
                    if (c > 0 && !w(&bars.kt_empty1, par(c - 1))) break;
                    for (int a = 2; a < 4; ++a) tma_load_2d_pair(sk + a * kBox, &mk, 64 * a, r0 + own, kf1);
                    // V: all keys of the chunk, own 64 value columns (after the previous P.Vz)
                    if (c > 0 && !w(&bars.v_empty, par(c - 1))) break;
                    mbar_arrive_expect_tx(&bars.v_full, 2 * kBox);
                    for (int j = 0; j < 2; ++j) tma_load_2d(sv + j * kBox, &mv, vcol, r0 + 128 * j, &bars.v_full);
                    ++v_loads;
                    // K^T operand of the state update: the peer key block x own dk half goes
                    // into boxes 2*peer, 2*peer+1 once S has read them (the odd CTA's after S's
                    // first half, the even CTA's after all of S)
                    if (!w(rank == 1 ? &bars.s_half : &bars.s_full, par(c))) break;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&bars.kt_full0, 2 * kBox);
                        mbar_arrive_expect_tx(&bars.kt_full1, 2 * kBox);
                        ++armed_kt;
                    }
                    for (int m = 0; m < 2; ++m)
                        tma_load_2d_pair(sk + (2 * (int)peer + m) * kBox, &mk, 64 * (2 * (int)rank + m),
                                         r0 + other, ktf);
                    // the next chunk's boxes into L2, behind this chunk's loads in the TMA queue
                    prefetch(c + 1);
                }
                if (!ok) {
                    // let loads in flight land before the CTAs unwind
                    const uint32_t b0 = (uint32_t)base;
                    if (v_loads) mbar_wait(&bars.v_full, (b0 + v_loads - 1) & 1, nullptr, 100000000ull);
                    if (rank == 0) {
                        if (armed_q) mbar_wait(&bars.q_full, (b0 + armed_q - 1) & 1, nullptr, 100000000ull);
                        if (armed_k) {
                            mbar_wait(&bars.k_full0, (b0 + armed_k - 1) & 1, nullptr, 100000000ull);
                            mbar_wait(&bars.k_full1, (b0 + armed_k - 1) & 1, nullptr, 100000000ull);
                        }
                        if (armed_kt) {
                            mbar_wait(&bars.kt_full0, (b0 + armed_kt - 1) & 1, nullptr, 100000000ull);
                            mbar_wait(&bars.kt_full1, (b0 + armed_kt - 1) & 1, nullptr, 100000000ull);
                        }
                    }
                }
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- MMA issuer (even CTA)
            if (rank == 0 && lane == 0) {
                const uint32_t id_s = idesc_bf16(256, 256, 0, 0);     // Q K^T: both K-major
                const uint32_t id_r = idesc_bf16(256, 128, 1, 1);     // K^T Vz: both MN-major
                const int fmt = f16 ? 0 : 1;                          // fp16 / bf16 operands
                const uint32_t id_q = idesc_f16(256, 128, 0, 1, fmt); // Q R': B MN-major
                const uint32_t id_p = idesc_f16(256, 128, 0, 1, fmt); // P Vz: A in TMEM
                // descriptors are linear in the start address: base descriptor + offset / 16
                const uint64_t dQ = sdesc_sw128(smem_u32(sq), 16, 1024);
                const uint64_t dK = sdesc_sw128(smem_u32(sk), 16, 1024);
                const uint64_t dKT = sdesc_sw128(smem_u32(sk), kBox, 1024);   // dk boxes 16 KB apart
                const uint64_t dV = sdesc_sw128(smem_u32(sv), 2 * kBox, 1024);
                const uint64_t dV16 = sdesc_sw128(smem_u32(sv16), 2 * kBox, 1024);  // hi/lo: R' lo
                const uint64_t dR16 = sdesc_sw128(smem_u32(sr16), 2 * kBox, 1024);  // hi/lo: R' hi
                bool ok = !*abort_p;
                auto w = [&](uint64_t* bar, uint32_t p) {
                    if (ok && !mbar_wait_cl(bar, p, abort_p, wait_ns)) { ok = false; fail(); }
                    return ok;
                };
                auto s_boxes = [&](int a0) {
#pragma unroll 1
                    for (int a = a0; a < a0 + 2; ++a)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t off = (uint64_t)((a * kBox + kk * 32) >> 4);
                            mma_pair(tmem + kTS, dQ + off, dK + off, id_s, (a | kk) != 0);
                        }
                };
                auto qr_boxes = [&](int a0) {
#pragma unroll 1
                    for (int a = a0; a < a0 + 2; ++a)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t qa = dQ + (uint64_t)((a * kBox + kk * 32) >> 4);
                            const uint64_t ro = (uint64_t)(((4 * a + kk) * 2048) >> 4);
                            mma_pair(tmem + kTO, qa, dR16 + ro, id_q, (a | kk) != 0);
                            if (!f16) mma_pair(tmem + kTO, qa, dV16 + ro, id_q, 1);
                        }
                };
                auto kv_block = [&](int j) {
#pragma unroll
                    for (int t = 8 * j; t < 8 * j + 8; ++t) {
                        const uint64_t ka = (uint64_t)(((t >> 3) * 2 * kBox + (t & 7) * 2048) >> 4);
                        const uint64_t off = (uint64_t)((t * 2048) >> 4);
                        mma_pair(tmem + kTR, dKT + ka, dV + off, id_r, 1);
                    }
                };
                for (int c = 0; c < nchunks && ok; ++c) {
                    const uint32_t ph = par(c);
                    // S = Q K^T (the previous P.Vz, issued earlier, reads the S columns first:
                    // tcgen05.mma operations of one thread run in issue order)
                    if (!w(&bars.q_full, ph) || !w(&bars.k_full0, ph)) break;
                    tc_fence_after();
                    s_boxes(0);
                    mma_commit_pair(&bars.s_half, kBoth);
                    if (!w(&bars.k_full1, ph)) break;
                    tc_fence_after();
                    s_boxes(2);
                    mma_commit_pair(&bars.s_full, kBoth);
                    // O = Q R'; the first MMA overwrites the accumulator.  fp16: each Q half
                    // once the conversion warps have turned it into fp16
                    if (!w(&bars.rcopy, ph)) break;
                    if (c > 0 && !w(&bars.o_free, par(c - 1))) break;
                    if (f16 && !w(&bars.q16_0, ph)) break;
                    tc_fence_after();
                    qr_boxes(0);
                    if (f16 && !w(&bars.q16_1, ph)) break;
                    tc_fence_after();
                    qr_boxes(2);
                    mma_commit_pair(&bars.q_empty, kBoth);
                    // R += K^T Vz (R was rescaled by g^B with the copy), key block 0 then 1
                    if (!w(&bars.vz_ready, ph) || !w(&bars.kt_full0, ph)) break;
                    tc_fence_after();
                    kv_block(0);
                    mma_commit_pair(&bars.kt_empty0, kBoth);
                    if (!w(&bars.kt_full1, ph)) break;
                    tc_fence_after();
                    kv_block(1);
                    mma_commit_pair(&bars.kt_empty1, kBoth);
                    mma_commit_pair(&bars.r_done, kBoth);
                    // O += P Vz16 (fp16), or (P_hi + P_lo) Vz (bf16 hi/lo)
                    if (!w(&bars.p_ready, ph)) break;
                    tc_fence_after();
                    if (f16) {
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            mma_pair_ts(tmem + kTO, tmem + kTS + 32 * (t >> 1) + 8 * (t & 1),
                                        dV16 + (uint64_t)((t * 2048) >> 4), id_p, 1);
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const uint32_t a_hi = tmem + kTS + 32 * (t >> 1) + 8 * (t & 1);
                            const uint64_t bd = dV + (uint64_t)((t * 2048) >> 4);
                            mma_pair_ts(tmem + kTO, a_hi, bd, id_p, 1);
                            mma_pair_ts(tmem + kTO, a_hi + 16, bd, id_p, 1);
                        }
                    }
                    mma_commit_pair(&bars.o_full, kBoth);
                    mma_commit_pair(&bars.v_empty, kBoth);
                }
                // every issued MMA completes before the next pass or the release of TMEM
                mma_commit_pair(&bars.drain, 1);
                mbar_wait(&bars.drain, drains & 1, nullptr, 200000000ull);
                ++drains;
            }
        } else {
            // -------------------------------------------------------- transform warps
            const int q4 = warp & 3;                     // TMEM lane quarter of this warp
            const int row = 32 * q4 + lane;              // TMEM lane
            const uint32_t lrow = (uint32_t)(32 * q4) << 16;
            const int j = 128 * (int)rank + row;         // query row in the chunk / dk row of R
            const float l2g = dc.l2g[head];
            bool ok = !*abort_p;
            // tcgen05.ld/st are warp-collective: keep the outcome of every wait uniform
            auto wait = [&](uint64_t* bar, uint32_t p) {
                if (!ok) return false;
                const bool got = __all_sync(0xffffffffu, mbar_wait(bar, p, abort_p, wait_ns));
                if (!got) { ok = false; if (lane == 0) fail(); }
                return ok;
            };
            auto arrive_lead = [&](uint64_t* bar) {
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(lead(bar));
            };
            if (warp < kFirstR) {
                // ---------------------------------------------- scores -> P, then output
                const int half = (warp - kFirstP) >> 2;  // key half (P) / 64-column half (O)
                // P = S with the causal mask (key > j is zero; reversed: key < j); the score
                // scale a rides on Vz.  Key quarter qq (32 keys) holds the diagonal of this
                // warp's rows for qq = dq (key 32 dq + e against row 32 dq + lane); the
                // quarters on the far side of it are all zero (warp-uniform).
                const int dq = 4 * (int)rank + q4;
                __half2 pmax2 = __float2half2_rn(0.f);   // largest |P| met (fp16 format)
                auto live = [&](int qq) { return rev ? qq >= dq : qq <= dq; };
                // xi_j = g^(j+1-B) / a; reversed, row j stands at position B-1-j: g^(-j) / a
                const float xi = exp2f(l2g * (rev ? -(float)j : (float)(j + 1 - kB)) - dc.l2a[head]);
                // output rows of chunk c: xi_j * O for this warp's 64 columns, straight from
                // registers.  Each 128-byte row segment (32 fp32 or 64 bf16 columns = 8 items
                // of 16 bytes) is transposed within 8-lane groups (8 consecutive rows), so
                // that every store instruction writes four whole 128-byte segments.  The last
                // TMEM read releases O for the next Q.R.
                // acc (optional): with fp32 output acc is the output itself, which already
                // holds the earlier terms, and the rows are added to it by reductions in L2
                // (no read on the SM); with bf16 output acc is a separate fp32 array (pitch
                // ldo) that each thread reads for its own row's columns before the transpose.
                auto row_of = [&](int c) {
                    return (size_t)bh * N + (size_t)(rev ? nchunks - 1 - c : c) * kB;
                };
                auto add_acc = [&](float* o, int c, size_t col0) {
                    const float4* ap = reinterpret_cast<const float4*>(acc + (row_of(c) + j) * ldo + col0);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 t = ap[e];
                        o[4 * e] = fmaf(xi, o[4 * e], t.x);
                        o[4 * e + 1] = fmaf(xi, o[4 * e + 1], t.y);
                        o[4 * e + 2] = fmaf(xi, o[4 * e + 2], t.z);
                        o[4 * e + 3] = fmaf(xi, o[4 * e + 3], t.w);
                    }
                };
                auto do_out = [&](int c) {
                    if (!wait(&bars.o_full, par(c))) return;
                    tc_fence_after();
                    const int p8 = lane & 7;
                    const size_t row0 = row_of(c) + (size_t)(j - p8);
                    const size_t colh = (size_t)blk * 128 + (size_t)(64 * half);
                    constexpr int kSegs = OUT_BF16 ? 1 : 2;       // 128-byte segments per 64 columns
                    constexpr int kSegCols = OUT_BF16 ? 64 : 32;
#pragma unroll 1
                    for (int sg = 0; sg < kSegs; ++sg) {
                        uint32_t a[8][4];
                        const uint32_t tc0 = tmem + lrow + kTO + 64 * half + kSegCols * sg;
                        if (OUT_BF16) {
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                float o[32];
                                tmem_ld32(tc0 + 32 * hh, o);
                                tmem_wait_ld();
                                if (hh == 1) { tc_fence_before(); arrive_lead(&bars.o_free); }
                                if (ACC) {
                                    add_acc(o, c, colh + 32 * hh);
#pragma unroll
                                    for (int k = 0; k < 4; ++k)
#pragma unroll
                                        for (int w = 0; w < 4; ++w)
                                            a[4 * hh + k][w] = pack_bf16(o[8 * k + 2 * w], o[8 * k + 2 * w + 1]);
                                } else {
#pragma unroll
                                    for (int k = 0; k < 4; ++k)
#pragma unroll
                                        for (int w = 0; w < 4; ++w)
                                            a[4 * hh + k][w] = pack_bf16(xi * o[8 * k + 2 * w],
                                                                         xi * o[8 * k + 2 * w + 1]);
                                }
                            }
                        } else {
                            float o[32];
                            tmem_ld32(tc0, o);
                            tmem_wait_ld();
                            if (sg == kSegs - 1) { tc_fence_before(); arrive_lead(&bars.o_free); }
#pragma unroll
                            for (int k = 0; k < 8; ++k)
#pragma unroll
                                for (int w = 0; w < 4; ++w) a[k][w] = __float_as_uint(xi * o[4 * k + w]);
                        }
                        transpose8x8(a, p8);
                        const size_t col = (size_t)blk * 128 + (size_t)(64 * half + kSegCols * sg);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            uint4* dst;
                            if (OUT_BF16)
                                dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_base) +
                                                               (row0 + k) * ldo + col) + p8;
                            else
                                dst = reinterpret_cast<uint4*>(static_cast<float*>(out_base) +
                                                               (row0 + k) * ldo + col) + p8;
                            if (ACC && !OUT_BF16)
                                red_add_v4(reinterpret_cast<float*>(dst), a[k][0], a[k][1], a[k][2], a[k][3]);
                            else
                                *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                        }
                    }
                };
                // one key quarter: fp16 pairs (16 columns) or bf16 hi/lo pairs (32 columns)
                auto quarter = [&](int qq, auto fmt) {
                    constexpr bool F16 = decltype(fmt)::value;
                    const uint32_t ts = tmem + lrow + kTS + 32 * qq;
                    uint32_t pp[F16 ? 16 : 32];
                    if (live(qq)) {
                        float x[32];
                        tmem_ld32(ts, x);
                        tmem_wait_ld();
                        if (qq == dq) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (rev ? e < lane : e > lane) x[e] = 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            if (F16) {
                                pp[e] = pack_f16(x[2 * e], x[2 * e + 1]);
                                // fp16 rounds |x| >= 65520 to inf; NaN propagates
                                pmax2 = __hmax2_nan(pmax2, __habs2(*reinterpret_cast<const __half2*>(&pp[e])));
                            } else {
                                split2(x[2 * e], x[2 * e + 1], pp[e], pp[(16 + e) % (F16 ? 16 : 32)]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < (F16 ? 16 : 32); ++e) pp[e] = 0u;
                    }
                    if (F16) tmem_st16(ts, pp);
                    else tmem_st32(ts, reinterpret_cast<const float*>(pp));
                };
                // V row kr of chunk c scaled in place by a g^(B-1-kr) = g^(B/2-1-kr)
                // (reversed: a g^kr), one key row per thread; fp16: also the fp16 copy Vz16.
                // The block lands after the previous P.Vz.
                const int kr = 32 * (warp - kFirstP) + lane;
                const float fz = exp2f(l2g * (float)(rev ? kr : kB - 1 - kr) + dc.l2a[head]);
                float vmax = 0.f;
                auto do_v = [&](int c) {
                    if (!wait(&bars.v_full, par(c))) return;
                    {
                        const uint32_t rowoff = (uint32_t)kr * 128u;
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) {
                            const uint32_t off = rowoff + (((uint32_t)cc ^ ((uint32_t)kr & 7u)) << 4);
                            uint4* pv = reinterpret_cast<uint4*>(sv + off);
                            const uint4 u = *pv;
                            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                            uint32_t ob[4], oh[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float y0 = bf16_lo(wv[e]) * fz, y1 = bf16_hi(wv[e]) * fz;
                                ob[e] = pack_bf16(y0, y1);
                                if (f16) vmax = fmaxf(vmax, fmaxf(fabsf(y0), fabsf(y1)));
                                oh[e] = pack_f16(y0, y1);
                            }
                            *pv = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                            if (f16) *reinterpret_cast<uint4*>(sv16 + off) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                        }
                    }
                    fence_proxy_async();
                    arrive_lead(&bars.vz_ready);
                };
                for (int c = 0; c < nchunks && ok; ++c) {
                    // the rows acc adds to this chunk's output, into L2 ahead of use
                    if (ACC && OUT_BF16) {
                        const float* ar = acc + (row_of(c) + j) * ldo + blk * 128 + 64 * half;
                        prefetch_l2(ar);
                        prefetch_l2(ar + 32);
                    }
                    // V of this chunk (it lands while S runs), then P, then after P.Vz the output
                    do_v(c);
                    if (!wait(&bars.s_full, par(c))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int qq = 4 * half; qq < 4 * half + 4; ++qq) {
                        if (f16) quarter(qq, std::true_type{});
                        else quarter(qq, std::false_type{});
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    arrive_lead(&bars.p_ready);
                    do_out(c);
                }
                if (f16)
                    out_of_range(fmaxf(fmaxf(__low2float(pmax2), __high2float(pmax2)), vmax));
            } else {
                // ---------------------------------------------- state copy; Q16 or V -> Vz
                const int g = warp - kFirstR;            // 0..7
                const bool remote = g >= 4;              // peer's 64 columns (else this CTA's own)
                const uint32_t cbase = 64u * (remote ? peer : rank);   // TMEM column of the 64
                // tensor memory holds the state scaled by a (R~ = a R: its update K^T Vz takes
                // the a that Vz carries), so R' = c R = g^B R~; state_in enters times a
                const float gB = dc.gB[head], sc = gB, sa = dc.a[head];
                // fp16 R'16 (or the bf16 hi part) and, for hi/lo, the lo part
                const uint32_t hi_peer = map_peer(sr16, peer);
                const uint32_t lo_peer = map_peer(sv16, peer);
                const int p4 = lane & 3;
                const uint32_t j0 = (uint32_t)(j - p4);
                float cmax = 0.f;
                // State copy for chunk c: R' = c R_{i-1} (this CTA's dk row j, 64 value
                // columns) into the B operand of Q.R', and R~ <- g^B R~ in TMEM, in two halves
                // of 32 columns (4 items of 16 bytes per row).  Own columns go to this CTA's
                // copy; the peer's columns are transposed within 4-lane groups so that each
                // remote store writes 64 contiguous bytes of a row of the peer's copy.
                // R_{-1} comes from state_in (zero without it).
                auto state_half = [&](int c, int hh, auto fmt) {
                    constexpr bool F16 = decltype(fmt)::value;
                    const uint32_t tcol = tmem + lrow + kTR + cbase + 32 * hh;
                    float x[32];
                    if (c == 0) {
                        if (state_in) {
                            const float4* src = reinterpret_cast<const float4*>(
                                state_in + ((size_t)bh * kDk + j) * dv + blk * 128 + cbase + 32 * hh);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 f = src[e];
                                x[4 * e] = sa * f.x; x[4 * e + 1] = sa * f.y;
                                x[4 * e + 2] = sa * f.z; x[4 * e + 3] = sa * f.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) x[e] = 0.f;
                        }
                    } else {
                        tmem_ld32(tcol, x);
                        tmem_wait_ld();
                    }
                    uint32_t h[4][4], l[4][4];      // 16-byte items k = 8 columns each
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float y0 = sc * x[8 * k + 2 * e], y1 = sc * x[8 * k + 2 * e + 1];
                            if (F16) {
                                cmax = fmaxf(cmax, fmaxf(fabsf(y0), fabsf(y1)));
                                h[k][e] = pack_f16(y0, y1);
                                l[k][e] = 0u;
                            } else {
                                split2(y0, y1, h[k][e], l[k][e]);
                            }
                            x[8 * k + 2 * e] *= gB;
                            x[8 * k + 2 * e + 1] *= gB;
                        }
                    // the rescaled state goes back now (asynchronous until tcgen05.wait::st)
                    tmem_st32(tcol, x);
                    if (remote) {
                        // lane p of a 4-lane group then holds item 4hh+p of row j0 + k in slot k
                        transpose4x4(h, p4);
                        if (!F16) transpose4x4(l, p4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t r = j0 + (uint32_t)k;
                            const uint32_t off =
                                r * 128u + ((((uint32_t)(4 * hh + p4)) ^ (r & 7u)) << 4);
                            st_cluster_v4(hi_peer + off, h[k][0], h[k][1], h[k][2], h[k][3]);
                            if (!F16) st_cluster_v4(lo_peer + off, l[k][0], l[k][1], l[k][2], l[k][3]);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t off = (uint32_t)j * 128u +
                                                 ((((uint32_t)(4 * hh + k)) ^ ((uint32_t)j & 7u)) << 4);
                            *reinterpret_cast<uint4*>(sr16 + off) = make_uint4(h[k][0], h[k][1], h[k][2], h[k][3]);
                            if (!F16)
                                *reinterpret_cast<uint4*>(sv16 + off) =
                                    make_uint4(l[k][0], l[k][1], l[k][2], l[k][3]);
                        }
                    }
                };
                auto do_state = [&](int c) {
                    if (c > 0) {
                        if (!wait(&bars.r_done, par(c - 1))) return;
                        tc_fence_after();
                    }
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        if (f16) state_half(c, hh, std::true_type{});
                        else state_half(c, hh, std::false_type{});
                    }
                    tmem_wait_st();
                    if (remote) fence_proxy_async_cluster(); else fence_proxy_async();
                    tc_fence_before();
                    arrive_lead(&bars.rcopy);
                };
                // Q -> fp16 in place, one row of one dk box per thread: boxes 2h, 2h+1 once S
                // has read them (warps 10-13 the first, 14-17 the second)
                const int qrow = 32 * (g & 3) + lane;
                auto do_q16 = [&](int c, int hq) {
                    if (!wait(hq == 0 ? &bars.s_half : &bars.s_full, par(c))) return;
                    {
                        const int a = 2 * hq + (g >> 2);
                        uint8_t* qr = sq + a * kBox + qrow * 128;
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) {
                            // visit the row's items in swizzled order: the 8 rows of an 8-lane
                            // group then touch 8 different bank groups (conflict-free)
                            uint4* p = reinterpret_cast<uint4*>(qr + (((uint32_t)cc ^ ((uint32_t)qrow & 7u)) << 4));
                            const uint4 u = *p;
                            const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float y0 = bf16_lo(wv[e]), y1 = bf16_hi(wv[e]);
                                cmax = fmaxf(cmax, fmaxf(fabsf(y0), fabsf(y1)));
                                o[e] = pack_f16(y0, y1);
                            }
                            *p = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                    fence_proxy_async();
                    arrive_lead(hq == 0 ? &bars.q16_0 : &bars.q16_1);
                };
                for (int c = 0; c < nchunks && ok; ++c) {
                    do_state(c);
                    if (f16) { do_q16(c, 0); do_q16(c, 1); }
                }
                if (f16) out_of_range(cmax);
            }
        }
        // ---------------------------------------------------------- end of the pass
        __syncwarp();
        tc_fence_before();
        cluster_sync_all();     // every MMA of the pass has completed (drain), both CTAs' flags set
        tc_fence_after();
        if (pass == 1 || !f16 || *abort_p || !*range_p) break;
        if (threadIdx.x == 0 && rank == 0) atomicAdd(&g_reruns_chunkwise_pair, 1u);
    }
    // ---- final state: this CTA's dk rows of R_{N/B-1}, each state-copy warp its 64 columns
    // (written after the last pass, so that a re-run still reads an aliased state_in intact;
    // both formats give the same state: its update reads bf16 operands only)
    if (warp >= kFirstR && state_out && nchunks > 0 && !*abort_p) {
        const int q4 = warp & 3;
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const int j = 128 * (int)rank + 32 * q4 + lane;
        const uint32_t cbase = 64u * ((warp - kFirstR >= 4) ? peer : rank);
        const float sc = dc.ia[head];                // R = R~ / a
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            float x[32];
            tmem_ld32(tmem + lrow + kTR + cbase + 32 * hh, x);
            tmem_wait_ld();
            float4* dst = reinterpret_cast<float4*>(
                state_out + ((size_t)bh * kDk + j) * dv + blk * 128 + cbase + 32 * hh);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(sc * x[4 * e], sc * x[4 * e + 1], sc * x[4 * e + 2], sc * x[4 * e + 3]);
        }
    }
    tc_fence_before();
    cluster_sync_all();     // no tensor-memory access pending in either CTA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace

// Every wait of the kernel gives up after this long (wall time) and reports RET_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

bool chunkwise_pair_supported(int dk, int dv, int chunk, const HeadConsts& hc, int H) {
    if (dk != kDk || chunk != kB || dv % 128 != 0) return false;
    for (int h = 0; h < H; ++h)
        if (!(hc.l2g[h] * (float)chunk >= -64.0f)) return false;   // g^(-B) <= 2^64
    return true;
}

cudaError_t launch_chunkwise_tc_pair(const void* q, const void* k, const void* v, void* o,
                                     int out_bf16, int b, int H, int N, int dk, int dv, int chunk,
                                     const HeadConsts& hc, const float* state_in, float* state_out,
                                     cudaStream_t s, uint64_t wait_ns, int no_loads, int ldq,
                                     int ldk, int ldv, int ldo, int rev, const float* acc) {
    if (!chunkwise_pair_supported(dk, dv, chunk, hc, H)) return cudaErrorNotSupported;
    if (wait_ns == 0) wait_ns = kWaitLimitNs;
    if (ldq == 0) ldq = dk;
    if (ldk == 0) ldk = dk;
    if (ldv == 0) ldv = dv;
    if (ldo == 0) ldo = dv;
    if (ldq < dk || ldk < dk || ldv < dv || ldo < dv || (ldq | ldk | ldv | ldo) % 8 != 0)
        return cudaErrorInvalidValue;
    Decay dc;
    int fp16_first = 1;
    for (int h = 0; h < H; ++h) {
        dc.l2g[h] = hc.l2g[h];
        dc.gB[h] = hc.gB[h];
        dc.l2a[h] = rintf(-0.5f * (float)chunk * hc.l2g[h]);     // within [0, 32]
        dc.a[h] = exp2f(dc.l2a[h]);
        dc.ia[h] = exp2f(-dc.l2a[h]);
        // fp16 Vz (a g^(B-1-r) v: between g^(B/2) |v| and g^(-B/2) |v|) keeps ~11 bits and
        // stays in range only while g^(-B) <= 4096
        if (!(hc.l2g[h] * (float)chunk >= -12.0f)) fp16_first = 0;
    }
    // An fp32 output that accumulates in place takes the hi/lo format from the start: a
    // re-run would add the unit's rows to the output a second time.
    if (acc && !out_bf16) fp16_first = 0;
    const long long rows = (long long)b * H * N;
    if (rows >= (1LL << 31)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    if (!make_map_bf16_pitch(&mq, q, rows, dk, ldq, 128) ||
        !make_map_bf16_pitch(&mk, k, rows, dk, ldk, 128) ||
        !make_map_bf16_pitch(&mv, v, rows, dv, ldv, 128))
        return cudaErrorInvalidValue;
    const long long grid = 2LL * b * H * (dv / 128);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = kSmemBytes + 1024;
    decltype(&chunkwise_pair_kernel<false, false, false>) kern;
    if (rev)
        kern = acc ? (out_bf16 ? chunkwise_pair_kernel<true, true, true> : chunkwise_pair_kernel<false, true, true>)
                   : (out_bf16 ? chunkwise_pair_kernel<true, false, true> : chunkwise_pair_kernel<false, false, true>);
    else
        kern = acc ? (out_bf16 ? chunkwise_pair_kernel<true, true, false> : chunkwise_pair_kernel<false, true, false>)
                   : (out_bf16 ? chunkwise_pair_kernel<true, false, false> : chunkwise_pair_kernel<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (acc && (reinterpret_cast<uintptr_t>(acc) & 15u)) return cudaErrorInvalidValue;
    // fp32 output accumulates in place (the kernel adds to o and never reads acc)
    if (acc && !out_bf16 && acc != o) return cudaErrorInvalidValue;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, o, state_in, state_out, N, H, dv,
                                                fp16_first, dc, wait_ns, no_loads, ldo, acc);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(RET_KERNEL_CHUNKWISE_TC_PAIR);
    return e;
}

unsigned read_clear_error_tc_chunkwise_pair(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_chunkwise_pair, sizeof(h), 0, cudaMemcpyDeviceToHost,
                                  s) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_chunkwise_pair, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

unsigned read_clear_reruns_tc_chunkwise_pair(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_reruns_chunkwise_pair, sizeof(h), 0,
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_reruns_chunkwise_pair, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
