// tc_parallel.cu -- parallel retention on sm_103a tensor cores (tcgen05 + TMA).
//
// Computes eq.(5) of "Transformer取代者登場！…RetNet…（2）", section "Retention" 1) (Fig.3a),
// with the optional factors of "Retention Score 歸一化":
//     R[n][m] = (q_n . k_m) [/ sqrt(dk)] * g^(n-m) [/ sqrt(s_n)]   for m <= n, else 0
//     s_n     = sum_{i<=n} g^(n-i) = (1 - g^(n+1)) / (1 - g)
//     O[n]    = sum_m R[n][m] v_m  [/ max(|sum_m R[n][m]|, 1)]
// for bf16 Q/K/V, fp32 accumulation; any N >= 128 (a partial last tile is masked).
//
// Work split: one CTA per (batch*head, 128-row query tile, block of W = 256 (or
// 128) value columns).  The score tile S = Q_rb K_cb^T does not depend on the
// value columns; the dv/W CTAs of a query tile each compute it (dk/(dk+W) of their
// tensor work).  Within each group of 8 heads, heavy query tiles (more key tiles under
// the causal mask) are scheduled first.
//
// Per key tile cb (128 keys):
//   S(cb) = Q K_cb^T                      tcgen05 M=128 N=128, K=dk, into a TMEM buffer
//   P     = S * rowc * g^(n-m)            transform warps, masked, written in place as a
//                                          hi/lo pair of bf16 values
//   O    += P V_cb                         tcgen05 M=128 N=128 per 128 value columns,
//                                          A = P read from tensor memory
// The row factor rowc = [1/sqrt(dk)] [1/sqrt(s_n)] and the decay g^(n-m) (one exp2 per
// element) are applied in fp32 before the single rounding of P; the transform warps
// also accumulate the fp32 row sums of R for the RET_NORM_ROWSUM division.  The
// scores enter P.V as two bf16 parts, hi = bf16(P) and lo = bf16(P - hi), two MMAs into
// the same accumulator: with a single bf16 P the row-sum division (signed row sums
// that cancel) and undecayed heads (gamma = 1, long causal sums) reached 2.5-6e-2 of the
// output RMS on N(0,1) inputs; the split stays near 1e-3.  In tensor memory each group
// of 32 keys (32 columns of S) becomes 16 columns of hi pairs followed by 16 of lo pairs.
//
// Pipelining: key and value pieces (128 rows x 128 columns bf16, 32 KB) stream
// through a 5-slot ring in the order K0, K1, V0, K2, V1, K3, V2, ..., which is also
// the order the MMAs release them: S(cb+1) is issued before P(cb) V(cb) so the
// transform of one score tile overlaps the next score MMAs.  The query tile stays
// in shared memory for the whole CTA.
//
// Roles (320 threads): warp 0 issues TMA loads, warp 1 owns tensor memory and
// issues tcgen05.mma, warps 2-9 (two groups of four; a warp reaches TMEM lanes
// 32*(warp%4)..+31) convert scores (group g takes key columns 64g..64g+63) and
// write the outputs (group g takes half of the value columns).  Every wait is
// bounded; a wait that gives up sets the device error word and the CTA unwinds.
//
// Outputs leave from registers as coalesced 128-byte row segments (8-lane transposes).
// Tensor memory (512 columns): [0,256) O (W fp32 columns), [256,384) and [384,512) S.
// Shared memory: Q (dk/128 pieces) + 5 ring pieces = 224 KB at dk = 256.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tma_host.cuh"

namespace ret {
namespace {

__device__ unsigned g_err_parallel;

using namespace tc;

constexpr int kRing = 5;
constexpr int kAtom = 128 * 128;          // 128 rows x 64 bf16
constexpr int kPiece = 2 * kAtom;         // 128 rows x 128 bf16
constexpr int kThreads = 320;
constexpr int kGroupWarps = 4;
constexpr int kXWarps = 8;
constexpr uint32_t kTO = 0, kTS = 256;

struct ParConsts {
    float l2g[kMaxHeads];
    float lng[kMaxHeads];
    float omg[kMaxHeads];
};

// Fused gated epilogue ([RN2] "門控多尺度 Retention"): GroupNorm over the dv outputs of
// each (token, head), optional per-channel affine, times swish(G).
struct EpiArgs {
    void* out;              // the output: [b][H][N][dv] (EPI = 0) or [b][N][H*dv]
    const void* g;          // [b][N][H*dv], fp32 or bf16 (template EPI); read through a TMA map
    const float* weight;    // [H*dv] or NULL
    const float* bias;      // [H*dv] or NULL
    float eps;
};
constexpr int kMaxClusterCtas = 4;   // value-column blocks of one query tile
constexpr int kHeadGroup = 8;        // (batch, head) pairs whose CTAs are scheduled together

struct Bars {
    uint64_t q_full;
    uint64_t full[kRing], empty[kRing];
    uint64_t s_full[2], p_ready[2];
    uint64_t o_full;
    uint64_t g_full[2];
    uint64_t q_free, g_pre;
    uint64_t drain;
};

__device__ __forceinline__ void fail(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_err_parallel, 1u);
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

// EPI = 0: write O [b][H][N][dv].  EPI = 1 / 2: fused gated GroupNorm with G in fp32 /
// bf16, writing [b][N][H*dv]; the nvb value-column blocks of a query tile then run as
// one thread-block cluster and exchange per-row statistics through shared memory.
template <int NH, int NV, bool OUT_BF16, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
parallel_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg, int N, int H, int dk, int dv, int bH,
                   int nvb, unsigned flags, const ParConsts pc, const EpiArgs ea) {
    constexpr int W = 128 * NV;
    constexpr int kEpiChunks = W / 128;                   // 64-column chunks per group
    // bf16 gate tiles of both groups fit where Q was: load them while the last P.V runs
    constexpr bool kGPrefetch = (EPI == 2) && (2 * kEpiChunks * 16384 <= NH * kPiece);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* qarea = sm;
    uint8_t* ring = sm + NH * kPiece;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    // Epilogue scratch, reusing the ring once every MMA of this CTA has completed (after
    // o_full): row sums and statistics of the two transform groups, and (mean, M2) of
    // each value-column block of the cluster, written by the peers.
    float (*rs_part)[128] = reinterpret_cast<float (*)[128]>(ring);
    float (*st_part)[128] = reinterpret_cast<float (*)[128]>(ring + 1024);
    float2 (*peer_stats)[128] = reinterpret_cast<float2 (*)[128]>(ring + 2048);
    __shared__ __align__(16) float colf[128];     // g^(-j), j = key column in a tile

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Block order: groups of kHeadGroup (batch, head) pairs, inside a group heavy query
    // tiles first, then (batch, head), then value-column block (the cluster).  The CTAs
    // resident at one time then share the K/V of a few heads in L2 instead of streaming
    // every head's K/V from DRAM.
    const int nqt = (N + 127) / 128;
    const int full_grp = kHeadGroup * nqt * nvb;
    const int gi = (int)(blockIdx.x / full_grp);
    const int gheads = min(kHeadGroup, bH - gi * kHeadGroup);
    const int r_in = (int)(blockIdx.x % full_grp);
    const int qt = nqt - 1 - r_in / (gheads * nvb);
    const int rest = r_in % (gheads * nvb);
    const int bh = gi * kHeadGroup + rest / nvb, vb = rest % nvb;
    const int head = bh % H;
    const int n0 = 128 * qt;
    const int T = qt + 1;                                     // key tiles under the mask
    volatile int* abort_p = &abort_flag;
    float stat_mean = 0.f, stat_m2 = 0.f, row_inv = 1.f;      // fused epilogue, per row

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars.q_full, 1);
        for (int s = 0; s < kRing; ++s) { mbar_init(&bars.full[s], 1); mbar_init(&bars.empty[s], 1); }
        for (int c = 0; c < 2; ++c) {
            mbar_init(&bars.s_full[c], 1); mbar_init(&bars.p_ready[c], kXWarps);
        }
        mbar_init(&bars.o_full, 1);
        mbar_init(&bars.g_full[0], 1); mbar_init(&bars.g_full[1], 1);
        mbar_init(&bars.q_free, 1); mbar_init(&bars.g_pre, 1);
        mbar_init(&bars.drain, 1);
        fence_barrier_init();
    }
    if (warp == 1) { tmem_alloc(&tmem_slot, 512); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&mq); tma_prefetch_desc(&mk); tma_prefetch_desc(&mv);
            if (EPI != 0) tma_prefetch_desc(&mg);
            mbar_arrive_expect_tx(&bars.q_full, NH * kPiece);
            for (int hh = 0; hh < NH; ++hh)
                for (int a = 0; a < 2; ++a)
                    tma_load_3d(qarea + hh * kPiece + a * kAtom, &mq, 128 * hh + 64 * a, n0, bh,
                                &bars.q_full);
            uint32_t fill = 0;
            bool ok = true;
            auto load_piece = [&](const CUtensorMap* m, int c, int row) {
                const int s = fill % kRing;
                if (!mbar_wait(&bars.empty[s], ((fill / kRing) & 1) ^ 1, abort_p)) return false;
                mbar_arrive_expect_tx(&bars.full[s], kPiece);
                tma_load_3d(ring + s * kPiece, m, c, row, bh, &bars.full[s]);
                tma_load_3d(ring + s * kPiece + kAtom, m, c + 64, row, bh, &bars.full[s]);
                ++fill;
                return true;
            };
            for (int st = 0; st <= T && ok; ++st) {
                if (st < T)
                    for (int hh = 0; hh < NH && ok; ++hh) ok = load_piece(&mk, 128 * hh, 128 * st);
                if (st >= 1)
                    for (int vp = 0; vp < NV && ok; ++vp)
                        ok = load_piece(&mv, W * vb + 128 * vp, 128 * (st - 1));
            }
            if (kGPrefetch && ok) {
                // the last score MMA has read Q: its area takes the gate tiles
                if (!mbar_wait(&bars.q_free, 0, abort_p)) {
                    ok = false;
                } else {
                    mbar_arrive_expect_tx(&bars.g_pre, 2 * kEpiChunks * 16384);
                    for (int gg = 0; gg < 2; ++gg)
                        for (int ch = 0; ch < kEpiChunks; ++ch)
                            tma_load_3d(qarea + (gg * kEpiChunks + ch) * 16384, &mg,
                                        head * dv + W * vb + (W / 2) * gg + 64 * ch, n0, bh / H,
                                        &bars.g_pre);
                }
            }
            if (!ok) {
                fail(abort_p);
                for (uint32_t f = fill > kRing ? fill - kRing : 0; f < fill; ++f)
                    mbar_wait(&bars.full[f % kRing], (f / kRing) & 1, nullptr, 100000000ull);
                mbar_wait(&bars.q_full, 0, nullptr, 100000000ull);
            }
            if (kGPrefetch && !ok) {
                // a gate load may be in flight only if it was issued; wait for it briefly
                mbar_wait(&bars.g_pre, 0, nullptr, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(128, 128, 0, 0);   // Q K^T: both K-major
            const uint32_t id_p = idesc_bf16(128, 128, 0, 1);   // P V: A in TMEM, B MN-major
            const uint32_t ring_a = smem_u32(ring);
            const uint64_t dQ = sdesc_sw128(smem_u32(qarea), 16, 1024);
            const uint64_t dK = sdesc_sw128(ring_a, 16, 1024);
            const uint64_t dV = sdesc_sw128(ring_a, kAtom, 1024);
            uint32_t fill = 0;
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t par) {
                if (ok && !mbar_wait(bar, par, abort_p)) { ok = false; fail(abort_p); }
                return ok;
            };
            auto slot_off = [&](uint32_t f) { return (uint64_t)(((f % kRing) * kPiece) >> 4); };
            wait(&bars.q_full, 0);
            for (int st = 0; st <= T && ok; ++st) {
                if (st < T) {
                    const int sb = st & 1;
                    // S(st) overwrites the buffer P(st-2) was read from: tcgen05.mma
                    // operations of one thread execute in issue order, so P(st-2).V,
                    // issued earlier, has read it first.
                    const uint32_t ts = tmem + kTS + 128 * sb;
#pragma unroll 1
                    for (int hh = 0; hh < NH; ++hh) {
                        // each dk half waits for its own piece and frees it right away
                        if (!wait(&bars.full[(fill + hh) % kRing], ((fill + hh) / kRing) & 1)) break;
                        tc_fence_after();
                        const uint64_t da = dQ + (uint64_t)((hh * kPiece) >> 4);
                        const uint64_t db = dK + slot_off(fill + hh);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t off = (uint64_t)(((kk / 4) * kAtom + (kk % 4) * 32) >> 4);
                            mma_bf16(ts, da + off, db + off, id_s, (hh | kk) != 0);
                        }
                        mma_commit(&bars.empty[(fill + hh) % kRing]);
                    }
                    if (!ok) break;
                    mma_commit(&bars.s_full[sb]);
                    if (kGPrefetch && st == T - 1) mma_commit(&bars.q_free);
                    fill += NH;
                }
                if (st >= 1) {
                    const int t = st - 1, sb = t & 1;
                    if (!wait(&bars.p_ready[sb], (t >> 1) & 1)) break;
                    const uint32_t ts = tmem + kTS + 128 * sb;
#pragma unroll 1
                    for (int vp = 0; vp < NV; ++vp) {
                        // each 128-column value piece waits for its own load, frees it after use
                        if (!wait(&bars.full[(fill + vp) % kRing], ((fill + vp) / kRing) & 1)) break;
                        tc_fence_after();
                        const uint64_t db = dV + slot_off(fill + vp);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t a_t = ts + 32 * (kk / 2) + 8 * (kk % 2);
                            const uint64_t bd = db + (uint64_t)((16 * kk * 128) >> 4);
                            mma_ts(tmem + kTO + 128 * vp, a_t, bd, id_p, (t | kk) != 0);
                            mma_ts(tmem + kTO + 128 * vp, a_t + 16, bd, id_p, 1);
                        }
                        mma_commit(&bars.empty[(fill + vp) % kRing]);
                    }
                    if (!ok) break;
                    fill += NV;
                }
            }
            mma_commit(&bars.o_full);
            mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, nullptr, 200000000ull);
        }
    } else {
        // ------------------------------------------------------------ transform warps
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const int n = n0 + row;
        const float l2g = pc.l2g[head];
        float rowc = (flags & RET_NORM_SCALE) ? rsqrtf((float)dk) : 1.0f;
        if (flags & RET_NORM_DECAY) rowc *= rsqrtf(decay_rowsum(pc.lng[head], pc.omg[head], n));
        const bool want_rs = (flags & RET_NORM_ROWSUM) != 0;
        // g^(n-m) = g^(n-m0) * g^(-(m-m0)): one exp2 per row and tile, times a column
        // factor from a table.  The factors stay in range while g^(-127) <= 2^64; a
        // smaller g takes one exp2 per element.
        const bool factored = l2g >= -0.5f;
        if (grp == 0) colf[row] = factored ? exp2f(-l2g * (float)row) : 0.f;
        named_bar(1, kXWarps * 32);
        float rs = 0.f;
        bool ok = true;
        auto wait = [&](uint64_t* bar, uint32_t par) {
            if (!ok) return false;
            const bool got = __all_sync(0xffffffffu, mbar_wait(bar, par, abort_p));
            if (!got) { ok = false; if (lane == 0) fail(abort_p); }
            return ok;
        };
        for (int t = 0; t < T && ok; ++t) {
            const int sb = t & 1;
            if (!wait(&bars.s_full[sb], (t >> 1) & 1)) break;
            tc_fence_after();
            const uint32_t ts = tmem + lrow + kTS + 128 * sb;
            const int m0 = 128 * t;
            const float a = rowc * (factored ? decay_pow(l2g, (float)(n - m0)) : 1.0f);
#pragma unroll 1
            for (int c32 = 0; c32 < 2; ++c32) {
                const int kc = 64 * grp + 32 * c32;
                float x[32];
                tmem_ld32(ts + kc, x);
                float cf[32];
                const float4* cp = reinterpret_cast<const float4*>(colf + kc);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 f = cp[j];
                    cf[4 * j] = f.x; cf[4 * j + 1] = f.y; cf[4 * j + 2] = f.z; cf[4 * j + 3] = f.w;
                }
                tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int m = m0 + kc + 2 * e;
                    const float w0 = factored ? a * cf[2 * e] : rowc * decay_pow(l2g, (float)(n - m));
                    const float w1 = factored ? a * cf[2 * e + 1] : rowc * decay_pow(l2g, (float)(n - m - 1));
                    const float p0 = (m <= n) ? x[2 * e] * w0 : 0.f;
                    const float p1 = (m + 1 <= n) ? x[2 * e + 1] * w1 : 0.f;
                    if (want_rs) rs += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                    pk[16 + e] = pack_bf16(p0 - __uint_as_float(pk[e] << 16),
                                           p1 - __uint_as_float(pk[e] & 0xffff0000u));
                }
                // the 32 keys of this quarter: hi pairs in its first 16 columns, lo pairs next
                tmem_st32(ts + kc, reinterpret_cast<const float*>(pk));
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_ready[sb]);
        }
        // ---- output: O / max(|row sum|, 1) for rows inside the sequence
        constexpr int kCols = W / 2;                            // value columns of this group
        const uint32_t ocol = tmem + lrow + kTO + kCols * grp;
        // warp-uniform: tcgen05.ld is warp-collective.  After o_full no MMA reads the ring.
        const bool have_o = ok && wait(&bars.o_full, 0);
        if (have_o) tc_fence_after();
        rs_part[grp][row] = rs;
        named_bar(2, kXWarps * 32);
        float den = 1.f;
        if (want_rs) den = fmaxf(fabsf(rs_part[0][row] + rs_part[1][row]), 1.0f);
        const float inv = 1.0f / den;
        if (EPI == 0) {
            row_inv = inv;
        } else {
            // statistics of this block's W values of the row: mean, then sum of squared
            // deviations (two passes over tensor memory), combined over the two groups.
            // Every transform warp takes part in the named barriers, aborted or not.
            float s1 = 0.f;
            if (have_o) {
#pragma unroll 1
                for (int c0 = 0; c0 < kCols; c0 += 32) {
                    float o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) s1 += o[j] * inv;
                }
            }
            st_part[grp][row] = s1;
            named_bar(3, kXWarps * 32);
            const float mean_b = (st_part[0][row] + st_part[1][row]) / (float)W;
            named_bar(4, kXWarps * 32);
            float s2 = 0.f;
            if (have_o) {
#pragma unroll 1
                for (int c0 = 0; c0 < kCols; c0 += 32) {
                    float o[32];
                    tmem_ld32(ocol + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) { const float d = o[j] * inv - mean_b; s2 += d * d; }
                }
            }
            st_part[grp][row] = s2;
            named_bar(5, kXWarps * 32);
            if (grp == 0) {
                stat_mean = mean_b;
                stat_m2 = st_part[0][row] + st_part[1][row];
            }
            row_inv = inv;
        }
    }
    if (EPI != 0) {
        // 1st cluster barrier: every CTA of the query tile is past its last MMA, so its
        // ring may receive the peers' statistics; 2nd: all statistics have arrived.
        __syncwarp();
        cluster_sync_all();
        if (warp >= 2 && warp < 6) {
            const int row = 32 * (warp & 3) + (threadIdx.x & 31);
            for (int r = 0; r < nvb; ++r)
                st_cluster_f32x2(map_peer(&peer_stats[vb][row], (uint32_t)r), stat_mean, stat_m2);
        }
        __syncwarp();
        cluster_sync_all();
    }
    // ---- output: per transform group, 64-column chunks of the group's W/2 columns, stored
    // from registers.  Each 128-byte row segment (32 fp32 or 64 bf16 values = 8 items of
    // 16 bytes) is transposed within 8-lane groups (8 consecutive rows), so that every
    // store instruction writes four whole 128-byte segments; rows past N are skipped.
    // Without the gate prefetch, the ring (free once o_full has completed) takes a gate
    // tile per chunk (TMA load, 128-byte swizzle: the 16-byte chunk c of row r sits at
    // chunk position c ^ (r % 8) of a 128-row x 128-byte atom).
    if (warp >= 2) {
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int lane = threadIdx.x & 31;
        const int row = 32 * q4 + lane;
        const uint32_t lrow = (uint32_t)(32 * q4) << 16;
        const bool issuer = (threadIdx.x == (unsigned)(64 + 128 * grp));   // lane 0 of warp 2 / 6
        constexpr int kCols = W / 2;
        constexpr int kChunks = kEpiChunks;
        constexpr int kGAtoms = (EPI == 2) ? 1 : 2;
        const float inv = row_inv;
        float mean = 0.f, rstd = 1.f;
        if (EPI != 0) {
            for (int r = 0; r < nvb; ++r) mean += peer_stats[r][row].x;
            mean /= (float)nvb;
            float m2 = 0.f;
            for (int r = 0; r < nvb; ++r) {
                const float d = peer_stats[r][row].x - mean;
                m2 += peer_stats[r][row].y + (float)W * d * d;
            }
            rstd = rsqrtf(m2 / (float)dv + ea.eps);
        }
        const int bi = bh / H;
        const bool live = __all_sync(0xffffffffu, abort_flag == 0);
        if (live) tc_fence_after();
        auto swz = [&](int c16) { return (uint32_t)(row * 128 + ((((uint32_t)c16) ^ (row & 7)) << 4)); };
        const int p8 = lane & 7;
        const int r0 = row - p8;                                     // first row of the 8-lane group
        const size_t row_elems = (EPI != 0) ? (size_t)H * dv : (size_t)dv;
        const size_t row_base = (EPI != 0) ? (size_t)bi * N : (size_t)bh * N;
#pragma unroll 1
        for (int ch = 0; ch < kChunks; ++ch) {
            const int col = W * vb + kCols * grp + 64 * ch;          // first value column
            const int gcol = (EPI != 0) ? head * dv + col : col;     // column in the output row
            const int plane = (EPI != 0) ? bi : bh;
            uint8_t* gst = kGPrefetch ? qarea + (grp * kEpiChunks + ch) * 16384   // gate tile
                                      : ring + 8192 + grp * 65536;
            if (issuer && EPI != 0 && !kGPrefetch && live) {
                mbar_arrive_expect_tx(&bars.g_full[grp], kGAtoms * 16384);
                for (int a2 = 0; a2 < kGAtoms; ++a2)
                    tma_load_3d(gst + a2 * 16384, &mg, gcol + a2 * (EPI == 2 ? 64 : 32), n0, plane,
                                &bars.g_full[grp]);
            }
            bool got_g = true;
            if (EPI != 0 && live) {
                got_g = kGPrefetch ? __all_sync(0xffffffffu, mbar_wait(&bars.g_pre, 0, abort_p))
                                   : __all_sync(0xffffffffu, mbar_wait(&bars.g_full[grp], ch & 1, abort_p));
            }
            if (live && got_g) {
                uint32_t a[8][4];                                    // bf16: the chunk's 8 items
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {                     // 32-column halves
                    float o[32];
                    tmem_ld32(tmem + lrow + kTO + kCols * grp + 64 * ch + 32 * hf, o);
                    float gv[32];
                    if (EPI == 2) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 u = *reinterpret_cast<const uint4*>(gst + swz(4 * hf + c));
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                gv[8 * c + 2 * e] = __uint_as_float(w4[e] << 16);
                                gv[8 * c + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                            }
                        }
                    } else if (EPI == 1) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float4 f = *reinterpret_cast<const float4*>(gst + hf * 16384 + swz(c));
                            gv[4 * c] = f.x; gv[4 * c + 1] = f.y; gv[4 * c + 2] = f.z; gv[4 * c + 3] = f.w;
                        }
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if (EPI == 0) {
                            o[jj] = o[jj] * inv;
                        } else {
                            float yn = (o[jj] * inv - mean) * rstd;
                            const int ch_ = head * dv + col + 32 * hf + jj;
                            if (ea.weight) yn *= ea.weight[ch_];
                            if (ea.bias) yn += ea.bias[ch_];
                            // swish(g) = g sigmoid(g) = h (1 + tanh(h)), h = g / 2, with the
                            // hardware tanh (one special-function op; relative error near
                            // 2^-11, far inside the bf16-input tolerance)
                            const float hg = 0.5f * gv[jj];
                            o[jj] = fmaf(hg, tanh_approx(hg), hg) * yn;
                        }
                    }
                    if (OUT_BF16) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                a[4 * hf + k][w] = pack_bf16(o[8 * k + 2 * w], o[8 * k + 2 * w + 1]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
#pragma unroll
                            for (int w = 0; w < 4; ++w) a[k][w] = __float_as_uint(o[4 * k + w]);
                    }
                    if (!OUT_BF16 || hf == 1) {
                        // one 128-byte segment: 32 fp32 (this half) or 64 bf16 (the chunk)
                        transpose8x8(a, p8);
                        const int c0 = gcol + (OUT_BF16 ? 0 : 32 * hf);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int n_out = n0 + r0 + k;
                            if (n_out < N) {
                                const size_t e0 = (row_base + (size_t)n_out) * row_elems + (size_t)c0;
                                uint4* dst = OUT_BF16
                                    ? reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ea.out) + e0) + p8
                                    : reinterpret_cast<uint4*>(static_cast<float*>(ea.out) + e0) + p8;
                                *dst = make_uint4(a[k][0], a[k][1], a[k][2], a[k][3]);
                            }
                        }
                    }
                }
            }
            // every warp of the group is done with this chunk's gate tile
            if (!kGPrefetch && EPI != 0) named_bar(6 + grp, 128);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

namespace {

using ParKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                           const CUtensorMap, int, int, int, int, int, int, unsigned,
                           const ParConsts, const EpiArgs);

template <int EPI>
ParKernel pick(int nh, int nv, int out_bf16) {
    const int sel = (nh == 2 ? 4 : 0) + (nv == 2 ? 2 : 0) + (out_bf16 ? 1 : 0);
    switch (sel) {
        case 0: return parallel_tc_kernel<1, 1, false, EPI>;
        case 1: return parallel_tc_kernel<1, 1, true, EPI>;
        case 2: return parallel_tc_kernel<1, 2, false, EPI>;
        case 3: return parallel_tc_kernel<1, 2, true, EPI>;
        case 4: return parallel_tc_kernel<2, 1, false, EPI>;
        case 5: return parallel_tc_kernel<2, 1, true, EPI>;
        case 6: return parallel_tc_kernel<2, 2, false, EPI>;
        default: return parallel_tc_kernel<2, 2, true, EPI>;
    }
}

// epi: 0 plain output, 1 gated with fp32 G, 2 gated with bf16 G
cudaError_t launch_common(const void* q, const void* k, const void* v, void* o, int out_bf16, int b,
                          int H, int N, int dk, int dv, const HeadConsts& hc, unsigned flags,
                          int epi, const EpiArgs& ea, cudaStream_t s) {
    // the 128-row TMA boxes must fit the sequence; shorter ones go to the CUDA-core kernel
    if (!(dk == 128 || dk == 256) || dv % 128 != 0 || N < 128) return cudaErrorNotSupported;
    const int nv = (dv % 256 == 0) ? 2 : 1;
    const int W = 128 * nv;
    const int nvb = dv / W;
    if (epi != 0 && nvb > kMaxClusterCtas) return cudaErrorNotSupported;
    ParConsts pc;
    for (int h = 0; h < H; ++h) {
        pc.l2g[h] = hc.l2g[h];
        pc.lng[h] = hc.lng[h];
        pc.omg[h] = hc.omg[h];
    }
    const long long bH = (long long)b * H;
    if (bH >= (1LL << 31) || N >= (1 << 30)) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mg;
    if (!make_map_bf16_3d(&mq, q, bH, N, dk, 128) || !make_map_bf16_3d(&mk, k, bH, N, dk, 128) ||
        !make_map_bf16_3d(&mv, v, bH, N, dv, 128))
        return cudaErrorInvalidValue;
    // the gate moves through 128-byte-wide boxes of 128 rows (unused without the epilogue)
    if (epi == 0) {
        mg = mq;
    } else if (!make_map_3d_128b(&mg, ea.g, epi == 2, b, N, (uint64_t)H * dv, 128)) {
        return cudaErrorInvalidValue;
    }
    const long long grid = (long long)((N + 127) / 128) * bH * nvb;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int smem = (dk / 128) * kPiece + kRing * kPiece + 1024;
    ParKernel kern = epi == 0 ? pick<0>(dk / 128, nv, out_bf16)
                   : epi == 1 ? pick<1>(dk / 128, nv, out_bf16) : pick<2>(dk / 128, nv, out_bf16);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (epi != 0) {
        // the value-column blocks of one query tile exchange GroupNorm statistics
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)nvb;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mg, N, H, dk, dv, (int)bH, nvb, flags, pc, ea);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) count_launch(epi == 0 ? RET_KERNEL_PARALLEL_TC : RET_KERNEL_PARALLEL_GATED_TC);
    return e;
}

}  // namespace

cudaError_t launch_parallel_tc(const void* q, const void* k, const void* v, void* o, int out_bf16,
                               int b, int H, int N, int dk, int dv, const HeadConsts& hc,
                               unsigned flags, cudaStream_t s) {
    // pairs of SMs where the shape allows (dk 256, dv and N multiples of 256)
    const cudaError_t ep = launch_parallel_pair(q, k, v, nullptr, o, out_bf16, 0, b, H, N, dk, dv,
                                                hc, flags, 0.f, nullptr, nullptr, s);
    if (ep != cudaErrorNotSupported) return ep;
    EpiArgs ea{};
    ea.out = o;
    return launch_common(q, k, v, o, out_bf16, b, H, N, dk, dv, hc, flags, 0, ea, s);
}

cudaError_t launch_parallel_gated_tc(const void* q, const void* k, const void* v, const void* g,
                                     void* out, int g_bf16, int out_bf16, int b, int H, int N,
                                     int dk, int dv, const HeadConsts& hc, unsigned flags,
                                     float eps, const float* weight, const float* bias,
                                     cudaStream_t s) {
    const cudaError_t ep = launch_parallel_pair(q, k, v, g, out, out_bf16, g_bf16 ? 2 : 1, b, H, N,
                                                dk, dv, hc, flags, eps, weight, bias, s);
    if (ep != cudaErrorNotSupported) return ep;
    EpiArgs ea;
    ea.out = out;
    ea.g = g;
    ea.weight = weight;
    ea.bias = bias;
    ea.eps = eps;
    return launch_common(q, k, v, out, out_bf16, b, H, N, dk, dv, hc, flags, g_bf16 ? 2 : 1, ea, s);
}

unsigned read_clear_error_tc_parallel(cudaStream_t s) {
    unsigned h = 0, z = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_err_parallel, sizeof(h), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return 0;
    cudaMemcpyToSymbolAsync(g_err_parallel, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s);
    cudaStreamSynchronize(s);
    return h;
}

}  // namespace ret
