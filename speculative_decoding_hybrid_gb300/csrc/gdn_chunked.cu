// Chunked (WY/UT) GatedDeltaNet prefill (sm_103a).
//
// "Run chained MTP drafting in the batch Engine", Correctness fix: the
// chunked plan runs a whole prompt at once and publishes only its final
// state (no per-row checkpoints).  Within a chunk of C tokens with start
// state S0 and G = cumsum(g) (the chunk form of the gated delta rule):
//   A[t][i] = beta_t e^{G_t-G_i} k_t.k_i  (i < t),   T = (I + A)^{-1}
//   W  = T diag(beta e^G) K,   Ut = T diag(beta) V,   U = Ut - W S0^T
//   O  = diag(e^G) Q S0^T + (M o Q K^T) U,   M[t][i] = e^{G_t-G_i} (i <= t)
//   S' = e^{G_C} S0 + U^T diag(e^{G_C-G}) K
//
// Two kernels, both on the 5th-generation tensor cores (tcgen05).
//  (1) gdn_chunk_wy_kernel -- one CTA per (chunk, v-head), all chunks of all
//      sequences at once (state-independent): [K;Q] K^T, the unit
//      lower-triangular inverse T in 16x16 blocks, W and Ut, and the masked,
//      decayed P = M o Q K^T; W, Ut and P go to the workspace (fp32, 80 KB
//      per chunk and head).
//  (2) gdn_chunk_scan_kernel -- one CTA per (sequence, v-head): the only
//      sequential part.  The state stays on chip across the sequence's
//      chunks; per chunk it forms U, the outputs and the next state.
// Sequence i's chunks start at cu_seqlens[i]; chunk c of sequence i uses
// workspace slot (cu_seqlens[i] + 64c)/64 + i, unique and below
// ceil(row_capacity/64) + nseq.
#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int kC = 64;         // chunk length
constexpr int kD = 128;        // d_k = d_v supported by this kernel pair
constexpr int kThreads = 256;

__device__ __forceinline__ int chunk_slot(int seq_start, int c, int seq) { return (seq_start + kC * c) / kC + seq; }

struct PrefArgs {
    const int32_t *cu;
    int32_t nseq, h_qk, h_v, grp, max_chunks, row_capacity, num_slots;
    const uint16_t *q, *k, *v;
    const float *g, *beta;
    float *pool;
    int64_t slot_stride;
    const int32_t *src_slot, *dst_slot;
    uint16_t *o;
    float *ws;  // [slot][h_v][2][C][D]
    float q_scale;
    uint32_t *status;
};

// Workspace per (chunk slot, v-head): W [C][D], Ut [C][D] and P [C][C], fp32,
// with P[t][i] = e^{G_t-G_i} q_t.k_i for i <= t (0 elsewhere and past the chunk).
constexpr size_t kWsFloats = size_t(2) * kC * kD + size_t(kC) * kC;

// G[t] = g[0] + ... + g[t] over the chunk (g = 0 past its n tokens), by warp 0
// with a shuffle scan; both prefill kernels use it, so they see the same G.
__device__ __forceinline__ void chunk_cumsum(const float *g, int n, float *G) {
    const int lane = threadIdx.x & 31;
    const float g0 = 2 * lane < n ? g[2 * lane] : 0.f;
    const float g1 = 2 * lane + 1 < n ? g[2 * lane + 1] : 0.f;
    const float pair = g0 + g1;
    float incl = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - pair;
    G[2 * lane] = excl + g0;
    G[2 * lane + 1] = excl + pair;
}

__device__ __forceinline__ float *ws_w(const PrefArgs &a, int slot, int h) {
    return a.ws + (size_t(slot) * a.h_v + h) * kWsFloats;
}

// ---------------------------------------------------------------------------
// (1) per-chunk WY/UT quantities on the tensor cores (tcgen05, kind::f16)
// ---------------------------------------------------------------------------
// Shared-memory map (bytes from a 1024-aligned base).  Operand tiles are
// 128-byte-swizzled K-major bf16 tiles (tc.cuh):
//   A1   [K; Q]   128 rows (tokens, then q rows) x 128 (d_k)      32 KB
//   KT   K^T      128 rows (d_k) x 64 (tokens)                   16 KB
//   VT   V^T      128 rows (d_v) x 64 (tokens)                   16 KB
//   TB   T diag(beta e^G), hi and lo bf16 parts, 64 x 64 each  2 x 8 KB
//   TV   T diag(beta),     hi and lo                           2 x 8 KB
//   (the fp32 matrix A -> T, [64][65], and the 16x16 block scratch of the
//    inversion live in the TB/TV area before those tiles are written)
//   misc G, beta, e^G, mbarrier, tensor-memory base, flags
// Tensor memory (256 columns): D1 = [K;Q] K^T at columns 0..63 (rows 0..63:
// K K^T, rows 64..127: Q K^T, which becomes P for the scan), D2 = W^T at
// 64..127, D3 = Ut^T at 128..191 (lane = d index).
namespace wy {
constexpr uint32_t kA1 = 0, kKT = 32768, kVT = 49152, kT = 65536, kMisc = 98304;
constexpr uint32_t kTbHi = kT, kTbLo = kT + 8192, kTvHi = kT + 16384, kTvLo = kT + 24576;
constexpr uint32_t kXScratch = kT + 16640;  // after the fp32 [64][65] matrix
constexpr size_t kSmem = kMisc + 1024 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;
}  // namespace wy

__device__ __forceinline__ float tri_T(const float *Af, int x, int y) {
    // unit lower-triangular T stored as its strict lower part
    return x == y ? 1.f : (x > y ? Af[x * (kC + 1) + y] : 0.f);
}

__global__ void __launch_bounds__(kThreads) gdn_chunk_wy_kernel(const PrefArgs a) {
    const int seq = blockIdx.x / a.max_chunks;
    const int c = blockIdx.x % a.max_chunks;
    const int h = blockIdx.y;
    const int s0 = a.cu[seq];
    const int s1 = a.cu[seq + 1];
    const int len = s1 - s0;
    if (s0 < 0 || len < 0 || s1 > a.row_capacity) return;  // reported by the scan kernel
    if (c * kC >= len) return;
    const int t0 = s0 + c * kC;
    const int n = min(kC, len - c * kC);
    const int hq = h / a.grp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ unsigned char smraw[];
    const uint32_t raw_u = gdn::smem_u32(smraw);
    unsigned char *sm = smraw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sb = gdn::smem_u32(sm);
    float *Af = reinterpret_cast<float *>(sm + wy::kT);
    float *Xs = reinterpret_cast<float *>(sm + wy::kXScratch);
    float *Gs = reinterpret_cast<float *>(sm + wy::kMisc);
    float *Bs = Gs + kC;
    float *eG = Bs + kC;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + wy::kMisc + 768);
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + wy::kMisc + 776);
    int *flag = reinterpret_cast<int *>(sm + wy::kMisc + 780);

    if (warp == 0) tc::tmem_alloc(tbase, wy::kTmemCols);
    if (tid == 0) gdn::mbar_init(bar, 1);

    // Stage K, Q (rows of A1), K^T and V^T as bf16 operand tiles; rows past n are zero.
    // A warp covers 32 consecutive tokens of one 8-column group, so the
    // transposed stores of a warp land in one row of K^T / V^T (no bank conflicts).
    for (int e = tid; e < kC * (kD / 8); e += kThreads) {
        const int t = e % kC, c8 = (e / kC) * 8;
        uint4 kv = make_uint4(0, 0, 0, 0), qv = kv, vv = kv;
        if (t < n) {
            kv = __ldg(reinterpret_cast<const uint4 *>(a.k + (size_t(t0 + t) * a.h_qk + hq) * kD + c8));
            qv = __ldg(reinterpret_cast<const uint4 *>(a.q + (size_t(t0 + t) * a.h_qk + hq) * kD + c8));
            vv = __ldg(reinterpret_cast<const uint4 *>(a.v + (size_t(t0 + t) * a.h_v + h) * kD + c8));
        }
        *reinterpret_cast<uint4 *>(sm + wy::kA1 + tc::swz_off(128, t, c8)) = kv;
        *reinterpret_cast<uint4 *>(sm + wy::kA1 + tc::swz_off(128, kC + t, c8)) = qv;
        const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint16_t ke = uint16_t(i & 1 ? kw[i >> 1] >> 16 : kw[i >> 1] & 0xffffu);
            const uint16_t ve = uint16_t(i & 1 ? vw[i >> 1] >> 16 : vw[i >> 1] & 0xffffu);
            *reinterpret_cast<uint16_t *>(sm + wy::kKT + tc::swz_off(128, c8 + i, t)) = ke;
            *reinterpret_cast<uint16_t *>(sm + wy::kVT + tc::swz_off(128, c8 + i, t)) = ve;
        }
    }
    if (tid < kC) {
        Bs[tid] = tid < n ? a.beta[size_t(t0 + tid) * a.h_v + h] : 0.f;
        Gs[tid] = tid < n ? a.g[size_t(t0 + tid) * a.h_v + h] : 0.f;
    }
    gdn::fence_proxy_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tbase;

    // D1 = A1 K^T: rows 0..63 are K K^T (rows 64..127, Q K^T, are not used here).
    if (tid == 0) {
        constexpr uint32_t idesc = tc::idesc_bf16(128, 64);
#pragma unroll
        for (int at = 0; at < 2; ++at)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t d = tc::smem_desc(sb + wy::kA1 + at * 16384 + s * 32);
                tc::mma_bf16(tm, d, d, idesc, (at | s) ? 1u : 0u);
            }
        tc::commit(bar);
    }
    if (warp == 0) {
        chunk_cumsum(Gs, n, Gs);  // G = cumsum(g) while the MMA runs (in place: each lane owns two entries)
        if (lane == 0) *flag = gdn::mbar_wait_bounded(bar, 0) ? 1 : 0;
    }
    __syncthreads();
    bool ok = *flag != 0;
    if (ok) {
        (void)gdn::mbar_try_wait(bar, 0);
        tc::fence_after();
        if (tid < kC) eG[tid] = expf(Gs[tid]);
        // Rows 0..63: A[t][i] = beta_t e^{G_t-G_i} (k_t.k_i), i < t.
        // Rows 64..127: P[t][i] = e^{G_t-G_i} (q_t.k_i), i <= t, to the workspace.
        const int q4 = warp & 3, hc = warp >> 2;
        float *Pw = ws_w(a, chunk_slot(s0, c, seq), h) + 2 * kC * kD;
        const int t = 32 * (q4 & 1) + lane;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float v16[16];
            const int col0 = 32 * hc + 16 * part;
            tc::ld16(tm + (uint32_t(32 * q4) << 16) + uint32_t(col0), v16);
            if (q4 < 2) {
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int i = col0 + x;
                    Af[t * (kC + 1) + i] = (i < t && t < n) ? Bs[t] * expf(Gs[t] - Gs[i]) * v16[x] : 0.f;
                }
            } else {
#pragma unroll
                for (int x = 0; x < 16; x += 4) {
                    float4 pv;
                    float *pe = &pv.x;
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        const int i = col0 + x + y;
                        pe[y] = (i <= t && t < n) ? expf(Gs[t] - Gs[i]) * v16[x + y] : 0.f;
                    }
                    *reinterpret_cast<float4 *>(Pw + t * kC + col0 + x) = pv;
                }
            }
        }
    }
    __syncthreads();
    if (ok) {
        // (I + A)^{-1} by 16x16 blocks.  Diagonal blocks: column substitution.
        float col[16];
        const int blk = tid >> 4, cc = tid & 15;
        if (tid < kC) {
#pragma unroll
            for (int r = 0; r < 16; ++r) col[r] = (r == cc) ? 1.f : 0.f;
            for (int r = cc + 1; r < 16; ++r) {
                float acc = 0.f;
                for (int m = cc; m < r; ++m) acc = fmaf(Af[(16 * blk + r) * (kC + 1) + 16 * blk + m], col[m], acc);
                col[r] = -acc;
            }
        }
        __syncthreads();
        if (tid < kC)
            for (int r = cc + 1; r < 16; ++r) Af[(16 * blk + r) * (kC + 1) + 16 * blk + cc] = col[r];
        __syncthreads();
        // Off-diagonal blocks, one block row at a time:
        //   T_{bi,bj} = -T_{bi,bi} sum_{bk=bj}^{bi-1} A_{bi,bk} T_{bk,bj}
        for (int bi = 1; bi < 4; ++bi) {
            for (int idx = tid; idx < bi * 256; idx += kThreads) {
                const int bj = idx >> 8, r = (idx >> 4) & 15, cj = idx & 15;
                float acc = 0.f;
                for (int bk = bj; bk < bi; ++bk)
                    for (int m = 0; m < 16; ++m)
                        acc = fmaf(Af[(16 * bi + r) * (kC + 1) + 16 * bk + m], tri_T(Af, 16 * bk + m, 16 * bj + cj), acc);
                Xs[idx] = acc;
            }
            __syncthreads();
            for (int idx = tid; idx < bi * 256; idx += kThreads) {
                const int bj = idx >> 8, r = (idx >> 4) & 15, cj = idx & 15;
                float acc = 0.f;
                for (int m = 0; m <= r; ++m)
                    acc = fmaf(tri_T(Af, 16 * bi + r, 16 * bi + m), Xs[(bj << 8) + (m << 4) + cj], acc);
                Af[(16 * bi + r) * (kC + 1) + 16 * bj + cj] = -acc;
            }
            __syncthreads();
        }
        // T_b = T diag(beta e^G), T_v = T diag(beta), each split into bf16 hi + lo.
        const int t = tid >> 2, i0 = (tid & 3) * 16;
        float tv[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) tv[x] = tri_T(Af, t, i0 + x);
        __syncthreads();  // every T entry is read before the tiles overwrite it
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t bh[4], bl[4], vh[4], vl[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t wbh = 0, wbl = 0, wvh = 0, wvl = 0;
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int x = half * 8 + p * 2 + e2;
                    const int i = i0 + x;
                    const float xb = tv[x] * Bs[i] * eG[i];
                    const float xv = tv[x] * Bs[i];
                    const uint16_t hb = gdn::f32_to_bf16(xb);
                    const uint16_t lb = gdn::f32_to_bf16(xb - gdn::bf16_to_f32(hb));
                    const uint16_t hv = gdn::f32_to_bf16(xv);
                    const uint16_t lv = gdn::f32_to_bf16(xv - gdn::bf16_to_f32(hv));
                    wbh |= uint32_t(hb) << (16 * e2);
                    wbl |= uint32_t(lb) << (16 * e2);
                    wvh |= uint32_t(hv) << (16 * e2);
                    wvl |= uint32_t(lv) << (16 * e2);
                }
                bh[p] = wbh;
                bl[p] = wbl;
                vh[p] = wvh;
                vl[p] = wvl;
            }
            const uint32_t off = tc::swz_off(64, t, i0 + half * 8);
            *reinterpret_cast<uint4 *>(sm + wy::kTbHi + off) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
            *reinterpret_cast<uint4 *>(sm + wy::kTbLo + off) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
            *reinterpret_cast<uint4 *>(sm + wy::kTvHi + off) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
            *reinterpret_cast<uint4 *>(sm + wy::kTvLo + off) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
        }
        gdn::fence_proxy_async_smem();
        tc::fence_before();
    }
    __syncthreads();
    if (ok && tid == 0) {
        tc::fence_after();
        // D2 = K^T (T_b)^T = W^T, D3 = V^T (T_v)^T = Ut^T; hi and lo parts accumulate.
        constexpr uint32_t idesc = tc::idesc_bf16(128, 64);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint64_t ak = tc::smem_desc(sb + wy::kKT + s * 32);
            const uint64_t av = tc::smem_desc(sb + wy::kVT + s * 32);
            tc::mma_bf16(tm + 64, ak, tc::smem_desc(sb + wy::kTbHi + s * 32), idesc, s ? 1u : 0u);
            tc::mma_bf16(tm + 64, ak, tc::smem_desc(sb + wy::kTbLo + s * 32), idesc, 1u);
            tc::mma_bf16(tm + 128, av, tc::smem_desc(sb + wy::kTvHi + s * 32), idesc, s ? 1u : 0u);
            tc::mma_bf16(tm + 128, av, tc::smem_desc(sb + wy::kTvLo + s * 32), idesc, 1u);
        }
        tc::commit(bar);
        *flag = gdn::mbar_wait_bounded(bar, 1) ? 1 : 0;
    }
    __syncthreads();
    ok = ok && *flag != 0;
    if (ok) {
        (void)gdn::mbar_try_wait(bar, 1);
        tc::fence_after();
        float *W = ws_w(a, chunk_slot(s0, c, seq), h);
        float *Ut = W + kC * kD;
        const int q4 = warp & 3, hc = warp >> 2;
        const int j = 32 * q4 + lane;  // d index = accumulator lane
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int col0 = 32 * hc + 16 * part;
            float w16[16], u16[16];
            tc::ld16(tm + (uint32_t(32 * q4) << 16) + 64u + uint32_t(col0), w16);
            tc::ld16(tm + (uint32_t(32 * q4) << 16) + 128u + uint32_t(col0), u16);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                W[(col0 + x) * kD + j] = w16[x];
                Ut[(col0 + x) * kD + j] = u16[x];
            }
        }
    } else if (tid == 0) {
        gdn::set_status(a.status, GDN_DEV_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, wy::kTmemCols);
}

// ---------------------------------------------------------------------------
// (2) sequential scan over chunks on the tensor cores (tcgen05, kind::f16)
// ---------------------------------------------------------------------------
// One CTA per (sequence, v-head); the 128 value rows of S are the M = 128
// side of every product, so each thread owns one row of S (lane quadrant of
// its warp) and half of its columns.  The FP32 master copy of S stays in
// registers for the whole sequence.  Every operand that is not exactly bf16
// is split into two bf16 parts, x = x1 + x2 with x1 = bf16(x) and
// x2 = bf16(x - x1) (about 2^-16 relative), and a product keeps the three
// leading terms a1 b1 + a1 b2 + a2 b1; q and k are exact bf16.  Per chunk:
//   phase A:  Uacc = S W^T         (M128 N64  K128)  -> U^T = Ut^T - Uacc
//             Oi   = S Q^T         (M128 N64  K128)
//   phase B:  Oa   = U^T P^T       (M128 N64  K64)
//             dS   = U^T (dec o K) (M128 N128 K64),   S <- e^{G_last} S + dS
//   o_t = q_scale (e^{G_t} Oi[:,t] + Oa[:,t]),  dec_i = e^{G_last - G_i},
// with P, W and Ut from the per-chunk kernel's workspace.
// Shared-memory map (bytes from a 1024-aligned base), bf16 K-major tiles:
namespace sc {
constexpr uint32_t kS1 = 0, kS2 = 32768;        // S parts      128 rows (d_v) x 128 (d_k)
constexpr uint32_t kW1 = 65536, kW2 = 81920;    // W parts       64 rows (t)   x 128 (d_k)
constexpr uint32_t kQ = 98304;                  // Q             64 rows (t)   x 128 (d_k)
constexpr uint32_t kP1 = 114688, kP2 = 122880;  // P parts       64 rows (t)   x  64 (i)
constexpr uint32_t kK1 = 131072, kK2 = 147456;  // dec K parts  128 rows (d_k) x  64 (i)
constexpr uint32_t kU1 = 163840, kU2 = 180224;  // U^T parts    128 rows (d_v) x  64 (i)
constexpr uint32_t kMisc = 196608;              // G, e^G, dec, mbarriers, tensor-memory base, flag
constexpr uint32_t kRawQ = 197632;              // next chunk's raw q rows (bf16 64 x 128)
constexpr uint32_t kRawK = 214016;              // next chunk's raw k rows (bf16 64 x 128)
constexpr uint32_t kRawG = 230400;              // next chunk's g (fp32 x 64)
constexpr size_t kSmem = kRawG + 256 + 1024;
constexpr uint32_t kTmemCols = 512;  // Uacc 0..63, Oi 64..127, Oa 128..191, dS 256..383
// The next chunk's raw W and P (fp32, from the workspace) land in the U and
// P tile areas, which are free from the end of phase B until they are
// consumed by the next chunk's staging.
constexpr uint32_t kRawW = kU1, kRawP = kP1;
}  // namespace sc

// Prefetch of chunk c's raw inputs: W (32 KB) and P (16 KB) from the
// workspace, q and k rows (256 B each) by bulk asynchronous copies on one
// mbarrier, g by 4-byte cp.async.  Called by every thread.
__device__ __forceinline__ void scan_prefetch(const PrefArgs &a, unsigned char *sm, uint64_t *bar, int s0, int len,
                                              int seq, int h, int hq, int c) {
    const int tid = threadIdx.x;
    const int t0 = s0 + c * kC;
    const int n = min(kC, len - c * kC);
    const float *W = ws_w(a, chunk_slot(s0, c, seq), h);
    if (tid < 32) {
        if (tid == 0) gdn::mbar_arrive_expect_tx(bar, uint32_t(kC * kD * 4 + kC * kC * 4 + 2 * n * kD * 2));
        __syncwarp();
        if (tid == 0) gdn::bulk_g2s(sm + sc::kRawW, W, kC * kD * 4, bar);
        if (tid == 1) gdn::bulk_g2s(sm + sc::kRawP, W + 2 * kC * kD, kC * kC * 4, bar);
        for (int t = tid; t < n; t += 32) {
            gdn::bulk_g2s(sm + sc::kRawQ + t * kD * 2, a.q + (size_t(t0 + t) * a.h_qk + hq) * kD, kD * 2, bar);
            gdn::bulk_g2s(sm + sc::kRawK + t * kD * 2, a.k + (size_t(t0 + t) * a.h_qk + hq) * kD, kD * 2, bar);
        }
    }
    if (tid < n) gdn::cp_async4(sm + sc::kRawG + tid * 4, a.g + size_t(t0 + tid) * a.h_v + h);
    gdn::cp_async_commit();
}

// Two-term bf16 split of 8 consecutive values, packed as two 16-byte chunks.
__device__ __forceinline__ void split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint16_t h0 = gdn::f32_to_bf16(x[2 * p]), h1 = gdn::f32_to_bf16(x[2 * p + 1]);
        const uint16_t l0 = gdn::f32_to_bf16(x[2 * p] - gdn::bf16_to_f32(h0));
        const uint16_t l1 = gdn::f32_to_bf16(x[2 * p + 1] - gdn::bf16_to_f32(h1));
        h[p] = uint32_t(h0) | (uint32_t(h1) << 16);
        l[p] = uint32_t(l0) | (uint32_t(l1) << 16);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_scan_kernel(const PrefArgs a) {
    const int h = blockIdx.x % a.h_v;
    const int seq = blockIdx.x / a.h_v;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s0 = a.cu[seq];
    const int s1 = a.cu[seq + 1];
    const int len = s1 - s0;
    const int src = a.src_slot[seq];
    const int dst = a.dst_slot[seq];
    uint32_t bad = 0;
    if (s0 < 0 || len < 0 || s1 > a.row_capacity) bad |= GDN_DEV_ROWS_BAD;
    if (src < -1 || src >= a.num_slots || dst < 0 || dst >= a.num_slots) bad |= GDN_DEV_SLOT_OOR;
    if (bad) {
        if (h == 0 && tid == 0) gdn::set_status(a.status, bad);
        return;
    }
    const int hq = h / a.grp;

    extern __shared__ unsigned char smraw[];
    const uint32_t raw_u = gdn::smem_u32(smraw);
    unsigned char *sm = smraw + (((raw_u + 1023u) & ~1023u) - raw_u);
    const uint32_t sb = gdn::smem_u32(sm);
    float *Gs = reinterpret_cast<float *>(sm + sc::kMisc);
    float *eG = Gs + kC;
    float *dec = eG + kC;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 768);
    uint64_t *bar_in = reinterpret_cast<uint64_t *>(sm + sc::kMisc + 784);
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + sc::kMisc + 776);
    int *flag = reinterpret_cast<int *>(sm + sc::kMisc + 780);

    if (warp == 0) tc::tmem_alloc(tbase, sc::kTmemCols);
    if (tid == 0) {
        gdn::mbar_init(bar, 1);
        gdn::mbar_init(bar_in, 1);
    }

    const int q4 = warp & 3, hc = warp >> 2;
    const int arow = 32 * q4 + lane;  // row of S held by this thread
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    const size_t row_off = size_t(h) * kD * kD + size_t(arow) * kD + 64 * hc;
    float sv[64];  // S[arow][64hc .. 64hc+63], FP32 master
    if (src >= 0) {
        const float4 *sp = reinterpret_cast<const float4 *>(a.pool + size_t(src) * a.slot_stride + row_off);
#pragma unroll
        for (int x = 0; x < 16; ++x) {
            const float4 v = sp[x];
            sv[4 * x] = v.x;
            sv[4 * x + 1] = v.y;
            sv[4 * x + 2] = v.z;
            sv[4 * x + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int x = 0; x < 64; ++x) sv[x] = 0.f;
    }
    auto write_S = [&]() {
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            float e[8];
#pragma unroll
            for (int y = 0; y < 8; ++y) e[y] = sv[8 * x + y];
            uint4 hi, lo;
            split8(e, hi, lo);
            const uint32_t off = tc::swz_off(128, arow, 64 * hc + 8 * x);
            *reinterpret_cast<uint4 *>(sm + sc::kS1 + off) = hi;
            *reinterpret_cast<uint4 *>(sm + sc::kS2 + off) = lo;
        }
    };
    write_S();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = *tbase;
    constexpr uint32_t id64 = tc::idesc_bf16(128, 64);
    constexpr uint32_t id128 = tc::idesc_bf16(128, 128);

    uint32_t phase = 0, phase_in = 0;
    bool ok = true;
    const int nchunks = (len + kC - 1) / kC;
    if (nchunks > 0) scan_prefetch(a, sm, bar_in, s0, len, seq, h, hq, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = s0 + c * kC;
        const int n = min(kC, len - c * kC);
        const float *W = ws_w(a, chunk_slot(s0, c, seq), h);
        const float *Ut = W + kC * kD;
        float ut[32];  // Ut[t][arow] for t in [32hc, 32hc+32), consumed after phase A
#pragma unroll
        for (int x = 0; x < 32; ++x) ut[x] = Ut[(32 * hc + x) * kD + arow];
        // the chunk's raw inputs (prefetched during the previous chunk)
        gdn::cp_async_wait<0>();
        if (tid == 0) *flag = gdn::mbar_wait_bounded(bar_in, phase_in) ? 1 : 0;
        __syncthreads();
        if (*flag == 0) {
            ok = false;
            break;
        }
        (void)gdn::mbar_try_wait(bar_in, phase_in);
        phase_in ^= 1u;
        const float *graw = reinterpret_cast<const float *>(sm + sc::kRawG);
        if (warp == 0) chunk_cumsum(graw, n, Gs);
        __syncthreads();
        if (tid < kC) {
            eG[tid] = expf(Gs[tid]);
            dec[tid] = tid < n ? expf(Gs[n - 1] - Gs[tid]) : 0.f;
        }
        // P: raw fp32 in the P area -> registers, then the two bf16 parts in place.
        float praw[16];
        {
            const int t = tid >> 2, i16 = (tid & 3) * 16;
            const float *pr = reinterpret_cast<const float *>(sm + sc::kRawP) + t * kC + i16;
#pragma unroll
            for (int x = 0; x < 16; x += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(pr + x);
                praw[x] = v.x; praw[x + 1] = v.y; praw[x + 2] = v.z; praw[x + 3] = v.w;
            }
        }
        __syncthreads();  // every thread holds its P values; eG and dec are ready
        {
            const int t = tid >> 2, i16 = (tid & 3) * 16;
#pragma unroll
            for (int x = 0; x < 16; x += 8) {
                float pe[8];
#pragma unroll
                for (int y = 0; y < 8; ++y) pe[y] = praw[x + y];
                uint4 hi, lo;
                split8(pe, hi, lo);
                const uint32_t off = tc::swz_off(64, t, i16 + x);
                *reinterpret_cast<uint4 *>(sm + sc::kP1 + off) = hi;
                *reinterpret_cast<uint4 *>(sm + sc::kP2 + off) = lo;
            }
        }
        // W parts (raw in the U area) and Q (raw q rows): row t, 8 d_k values.
        for (int e = tid; e < kC * (kD / 8); e += kThreads) {
            const int t = e >> 4, j8 = (e & 15) * 8;
            float w[8];
            uint4 qv = make_uint4(0, 0, 0, 0);
            if (t < n) {
                const float *wr = reinterpret_cast<const float *>(sm + sc::kRawW) + t * kD + j8;
                const float4 w0 = *reinterpret_cast<const float4 *>(wr);
                const float4 w1 = *reinterpret_cast<const float4 *>(wr + 4);
                w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
                w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
                qv = *reinterpret_cast<const uint4 *>(sm + sc::kRawQ + (t * kD + j8) * 2);
            } else {
#pragma unroll
                for (int y = 0; y < 8; ++y) w[y] = 0.f;
            }
            uint4 hi, lo;
            split8(w, hi, lo);
            const uint32_t off = tc::swz_off(64, t, j8);
            *reinterpret_cast<uint4 *>(sm + sc::kW1 + off) = hi;
            *reinterpret_cast<uint4 *>(sm + sc::kW2 + off) = lo;
            *reinterpret_cast<uint4 *>(sm + sc::kQ + off) = qv;
        }
        // dec o K, transposed: a warp takes 32 consecutive d_k indices j of one
        // group of 8 tokens (conflict-free reads of the raw k rows).
        for (int e = tid; e < kD * (kC / 8); e += kThreads) {
            const int j = e & (kD - 1), i8 = (e / kD) * 8;
            const uint16_t *kr = reinterpret_cast<const uint16_t *>(sm + sc::kRawK);
            float kv[8];
#pragma unroll
            for (int y = 0; y < 8; ++y) {
                const int i = i8 + y;
                kv[y] = i < n ? gdn::bf16_to_f32(kr[i * kD + j]) * dec[i] : 0.f;
            }
            uint4 hi, lo;
            split8(kv, hi, lo);
            const uint32_t off = tc::swz_off(128, j, i8);
            *reinterpret_cast<uint4 *>(sm + sc::kK1 + off) = hi;
            *reinterpret_cast<uint4 *>(sm + sc::kK2 + off) = lo;
        }
        gdn::fence_proxy_async_smem();
        tc::fence_before();
        __syncthreads();
        // Phase A: Uacc = S W^T, Oi = S Q^T.
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int at = 0; at < 2; ++at)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint32_t ka = at * 16384 + s * 32, kb = at * 8192 + s * 32;
                    const uint64_t a1 = tc::smem_desc(sb + sc::kS1 + ka), a2 = tc::smem_desc(sb + sc::kS2 + ka);
                    const uint64_t w1 = tc::smem_desc(sb + sc::kW1 + kb), w2 = tc::smem_desc(sb + sc::kW2 + kb);
                    const uint64_t qd = tc::smem_desc(sb + sc::kQ + kb);
                    tc::mma_bf16(tm, a1, w1, id64, (at | s) ? 1u : 0u);
                    tc::mma_bf16(tm, a1, w2, id64, 1u);
                    tc::mma_bf16(tm, a2, w1, id64, 1u);
                    tc::mma_bf16(tm + 64, a1, qd, id64, (at | s) ? 1u : 0u);
                    tc::mma_bf16(tm + 64, a2, qd, id64, 1u);
                }
            tc::commit(bar);
            *flag = gdn::mbar_wait_bounded(bar, phase) ? 1 : 0;
        }
        __syncthreads();
        if (*flag == 0) {
            ok = false;
            break;
        }
        (void)gdn::mbar_try_wait(bar, phase);
        phase ^= 1u;
        tc::fence_after();
        // U^T[arow][t] = Ut[t][arow] - Uacc[arow][t], split into two bf16 parts.
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float v16[16];
            const int col0 = 32 * hc + 16 * part;
            tc::ld16(tm + lane_base + uint32_t(col0), v16);
#pragma unroll
            for (int x = 0; x < 16; x += 8) {
                float u[8];
#pragma unroll
                for (int y = 0; y < 8; ++y) u[y] = ut[16 * part + x + y] - v16[x + y];
                uint4 hi, lo;
                split8(u, hi, lo);
                const uint32_t off = tc::swz_off(128, arow, col0 + x);
                *reinterpret_cast<uint4 *>(sm + sc::kU1 + off) = hi;
                *reinterpret_cast<uint4 *>(sm + sc::kU2 + off) = lo;
            }
        }
        gdn::fence_proxy_async_smem();
        tc::fence_before();
        __syncthreads();
        // Phase B: Oa = U^T P^T, dS = U^T (dec o K).
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t u1 = tc::smem_desc(sb + sc::kU1 + s * 32), u2 = tc::smem_desc(sb + sc::kU2 + s * 32);
                const uint64_t p1 = tc::smem_desc(sb + sc::kP1 + s * 32), p2 = tc::smem_desc(sb + sc::kP2 + s * 32);
                const uint64_t k1 = tc::smem_desc(sb + sc::kK1 + s * 32), k2 = tc::smem_desc(sb + sc::kK2 + s * 32);
                tc::mma_bf16(tm + 128, u1, p1, id64, s ? 1u : 0u);
                tc::mma_bf16(tm + 128, u1, p2, id64, 1u);
                tc::mma_bf16(tm + 128, u2, p1, id64, 1u);
                tc::mma_bf16(tm + 256, u1, k1, id128, s ? 1u : 0u);
                tc::mma_bf16(tm + 256, u1, k2, id128, 1u);
                tc::mma_bf16(tm + 256, u2, k1, id128, 1u);
            }
            tc::commit(bar);
            *flag = gdn::mbar_wait_bounded(bar, phase) ? 1 : 0;
        }
        __syncthreads();
        if (*flag == 0) {
            ok = false;
            break;
        }
        (void)gdn::mbar_try_wait(bar, phase);
        phase ^= 1u;
        tc::fence_after();
        // Every input tile is free now: fetch the next chunk's raw inputs while
        // the outputs and the state update below run.
        if (c + 1 < nchunks) scan_prefetch(a, sm, bar_in, s0, len, seq, h, hq, c + 1);
        // Outputs of the chunk's tokens.
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float oi[16], oa[16];
            const int col0 = 32 * hc + 16 * part;
            tc::ld16(tm + lane_base + 64u + uint32_t(col0), oi);
            tc::ld16(tm + lane_base + 128u + uint32_t(col0), oa);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int t = col0 + x;
                if (t < n)
                    a.o[(size_t(t0 + t) * a.h_v + h) * kD + arow] =
                        gdn::f32_to_bf16(a.q_scale * fmaf(eG[t], oi[x], oa[x]));
            }
        }
        // S <- e^{G_last} S + dS (FP32 master), then its bf16 parts.
        const float egl = eG[n - 1];
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float v16[16];
            tc::ld16(tm + lane_base + 256u + uint32_t(64 * hc + 16 * part), v16);
#pragma unroll
            for (int x = 0; x < 16; ++x) sv[16 * part + x] = fmaf(egl, sv[16 * part + x], v16[x]);
        }
        write_S();
        // (the next chunk's staging ends with the proxy fence and barrier the MMAs need)
    }
    if (ok) {
        float4 *dp = reinterpret_cast<float4 *>(a.pool + size_t(dst) * a.slot_stride + row_off);
#pragma unroll
        for (int x = 0; x < 16; ++x) dp[x] = make_float4(sv[4 * x], sv[4 * x + 1], sv[4 * x + 2], sv[4 * x + 3]);
    } else if (tid == 0) {
        gdn::set_status(a.status, GDN_DEV_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, sc::kTmemCols);
}

constexpr size_t kWySmem = wy::kSmem;
constexpr size_t kScanSmem = sc::kSmem;

}  // namespace

extern "C" size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity) {
    if (!dims || nseq < 0 || row_capacity < 0) return 0;
    const size_t slots = size_t((row_capacity + kC - 1) / kC) + size_t(nseq);
    return slots * size_t(dims->h_v) * kWsFloats * sizeof(float);
}

extern "C" int gdn_chunked_prefill(const gdn_dims *dims, int32_t nseq, int32_t row_capacity,
                                   const int32_t *cu_seqlens, int32_t max_seqlen, const gdn_bf16 *q,
                                   const gdn_bf16 *k, const gdn_bf16 *v, const float *g, const float *beta,
                                   float *pool_layer, int64_t slot_stride, int32_t num_slots,
                                   const int32_t *src_slot, const int32_t *dst_slot, gdn_bf16 *o, int32_t chunk,
                                   void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    if (!dims) return GDN_ERR_NULL;
    if (!gdn_host::dims_ok(dims)) return GDN_ERR_SHAPE;
    if (dims->d_k != kD) return GDN_ERR_SHAPE;
    if (chunk != kC) return GDN_ERR_ARG;
    if (nseq < 0 || row_capacity < 0 || max_seqlen < 0 || num_slots <= 0) return GDN_ERR_ARG;
    if (nseq == 0) return GDN_OK;
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !pool_layer || !src_slot || !dst_slot || !o)
        return GDN_ERR_NULL;
    const int64_t se = int64_t(dims->h_v) * dims->d_v * dims->d_k;
    if (slot_stride < se || (slot_stride % 4) != 0) return GDN_ERR_ARG;
    if (!gdn_host::aligned16(pool_layer) || !gdn_host::aligned16(q) || !gdn_host::aligned16(k) ||
        !gdn_host::aligned16(v))
        return GDN_ERR_ARG;
    const size_t need = gdn_prefill_workspace_bytes(dims, nseq, row_capacity);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PrefArgs a{};
    a.cu = cu_seqlens;
    a.nseq = nseq;
    a.h_qk = dims->h_qk;
    a.h_v = dims->h_v;
    a.grp = dims->h_v / dims->h_qk;
    a.max_chunks = (max_seqlen + kC - 1) / kC;
    a.row_capacity = row_capacity;
    a.num_slots = num_slots;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.pool = pool_layer;
    a.slot_stride = slot_stride;
    a.src_slot = src_slot;
    a.dst_slot = dst_slot;
    a.o = o;
    a.ws = static_cast<float *>(workspace);
    a.q_scale = dims->q_scale;
    a.status = dev_status;
    if (cudaFuncSetAttribute(gdn_chunk_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kWySmem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(gdn_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kScanSmem)) !=
            cudaSuccess)
        return GDN_ERR_CUDA;
    if (a.max_chunks > 0) {
        const long long gx = (long long)nseq * a.max_chunks;
        if (gx > 0x7fffffffLL || dims->h_v > 65535) return GDN_ERR_ARG;
        gdn_chunk_wy_kernel<<<dim3(unsigned(gx), dims->h_v), kThreads, kWySmem, st>>>(a);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    const long long gs = (long long)nseq * dims->h_v;
    gdn_chunk_scan_kernel<<<unsigned(gs), kThreads, kScanSmem, st>>>(a);
    return gdn_host::launch_status(cudaGetLastError());
}
