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
// Two kernels.
//  (1) gdn_chunk_wy_kernel -- one CTA per (chunk, v-head), all chunks of all
//      sequences at once: K K^T, the unit lower-triangular inverse T by
//      column-wise forward substitution, W and Ut; W and Ut go to the
//      workspace (fp32, 64 KB per chunk and head).
//  (2) gdn_chunk_scan_kernel -- one CTA per (sequence, v-head, slice of
//      d_v rows of S): the state slice stays in shared memory across the
//      sequence's chunks; per chunk it forms U, the outputs and the next
//      state.  Rows of S are independent, so slices run in parallel.
// Sequence i's chunks start at cu_seqlens[i]; chunk c of sequence i uses
// workspace slot (cu_seqlens[i] + 64c)/64 + i, unique and below
// ceil(row_capacity/64) + nseq.
#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int kC = 64;         // chunk length
constexpr int kD = 128;        // d_k = d_v supported by this kernel pair
constexpr int kThreads = 256;
constexpr int kSlice = 32;     // state rows per scan CTA

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

__device__ __forceinline__ float *ws_w(const PrefArgs &a, int slot, int h) {
    return a.ws + ((size_t(slot) * a.h_v + h) * 2) * size_t(kC) * kD;
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
// K K^T), D2 = W^T at 64..127, D3 = Ut^T at 128..191 (lane = d index).
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
    for (int e = tid; e < kC * (kD / 8); e += kThreads) {
        const int t = e / (kD / 8), c8 = (e % (kD / 8)) * 8;
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
        float run = 0.f;  // G = cumsum(g) while the MMA runs
        for (int t = 0; t < kC; ++t) {
            run += Gs[t];
            Gs[t] = run;
        }
        *flag = gdn::mbar_wait_bounded(bar, 0) ? 1 : 0;
    }
    __syncthreads();
    bool ok = *flag != 0;
    if (ok) {
        (void)gdn::mbar_try_wait(bar, 0);
        tc::fence_after();
        if (tid < kC) eG[tid] = expf(Gs[tid]);
        // A[t][i] = beta_t e^{G_t-G_i} (k_t.k_i), i < t, from the accumulator rows 0..63
        const int q4 = warp & 3, hc = warp >> 2;
        if (q4 < 2) {
            const int t = 32 * q4 + lane;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float v16[16];
                const int col0 = 32 * hc + 16 * part;
                tc::ld16(tm + (uint32_t(32 * q4) << 16) + uint32_t(col0), v16);
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int i = col0 + x;
                    Af[t * (kC + 1) + i] = (i < t && t < n) ? Bs[t] * expf(Gs[t] - Gs[i]) * v16[x] : 0.f;
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
// (2) sequential scan over chunks, one state slice per CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) gdn_chunk_scan_kernel(const PrefArgs a) {
    const int nsl = kD / kSlice;
    const int sl = blockIdx.x % nsl;
    const int h = (blockIdx.x / nsl) % a.h_v;
    const int seq = blockIdx.x / (nsl * a.h_v);
    const int tid = threadIdx.x;
    const int s0 = a.cu[seq];
    const int s1 = a.cu[seq + 1];
    const int len = s1 - s0;
    const int src = a.src_slot[seq];
    const int dst = a.dst_slot[seq];
    uint32_t bad = 0;
    if (s0 < 0 || len < 0 || s1 > a.row_capacity) bad |= GDN_DEV_ROWS_BAD;
    if (src < -1 || src >= a.num_slots || dst < 0 || dst >= a.num_slots) bad |= GDN_DEV_SLOT_OOR;
    if (bad) {
        if (h == 0 && sl == 0 && tid == 0) gdn::set_status(a.status, bad);
        return;
    }
    const int hq = h / a.grp;
    const int a0 = sl * kSlice;

    extern __shared__ __align__(16) float sm[];
    float *Ss = sm;                        // [kSlice][D+1]   state rows a0..a0+kSlice
    float *Qs = Ss + kSlice * (kD + 1);    // [C][D+1]
    float *Ks = Qs + kC * (kD + 1);        // [C][D+1]
    float *Ws = Ks + kC * (kD + 1);        // [C][D+1]
    float *Us = Ws + kC * (kD + 1);        // [C][kSlice+1]
    float *Ps = Us + kC * (kSlice + 1);    // [C][C+1]
    float *Gs = Ps + kC * (kC + 1);        // [C]

    const size_t head_off = size_t(h) * kD * kD + size_t(a0) * kD;
    for (int e = tid; e < kSlice * kD; e += kThreads) {
        const int r = e / kD, j = e % kD;
        Ss[r * (kD + 1) + j] = src >= 0 ? a.pool[size_t(src) * a.slot_stride + head_off + e] : 0.f;
    }
    const int nchunks = (len + kC - 1) / kC;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = s0 + c * kC;
        const int n = min(kC, len - c * kC);
        const float *W = ws_w(a, chunk_slot(s0, c, seq), h);
        const float *Ut = W + kC * kD;
        __syncthreads();  // previous chunk's readers are done with the buffers
        for (int e = tid; e < kC * kD; e += kThreads) {
            const int t = e / kD, j = e % kD;
            float qv = 0.f, kv = 0.f, wv = 0.f;
            if (t < n) {
                qv = gdn::bf16_to_f32(a.q[(size_t(t0 + t) * a.h_qk + hq) * kD + j]);
                kv = gdn::bf16_to_f32(a.k[(size_t(t0 + t) * a.h_qk + hq) * kD + j]);
                wv = W[e];
            }
            Qs[t * (kD + 1) + j] = qv;
            Ks[t * (kD + 1) + j] = kv;
            Ws[t * (kD + 1) + j] = wv;
        }
        if (tid < kC) Gs[tid] = tid < n ? a.g[size_t(t0 + tid) * a.h_v + h] : 0.f;
        __syncthreads();
        if (tid == 0) {
            float run = 0.f;
            for (int t = 0; t < kC; ++t) {
                run += Gs[t];
                Gs[t] = run;
            }
        }
        __syncthreads();
        // U[t][a] = Ut[t][a] - sum_j W[t][j] S[a][j]
        for (int e = tid; e < kC * kSlice; e += kThreads) {
            const int t = e / kSlice, r = e % kSlice;
            float acc = 0.f;
            for (int j = 0; j < kD; ++j) acc = fmaf(Ws[t * (kD + 1) + j], Ss[r * (kD + 1) + j], acc);
            Us[t * (kSlice + 1) + r] = t < n ? Ut[t * kD + a0 + r] - acc : 0.f;
        }
        // P[t][i] = e^{G_t-G_i} q_t.k_i for i <= t
        for (int e = tid; e < kC * kC; e += kThreads) {
            const int t = e / kC, i = e % kC;
            float val = 0.f;
            if (i <= t && t < n) {
                float acc = 0.f;
                for (int j = 0; j < kD; ++j) acc = fmaf(Qs[t * (kD + 1) + j], Ks[i * (kD + 1) + j], acc);
                val = expf(Gs[t] - Gs[i]) * acc;
            }
            Ps[t * (kC + 1) + i] = val;
        }
        __syncthreads();
        // O[t][a] = e^{G_t} q_t.S[a] + sum_{i<=t} P[t][i] U[i][a]
        for (int e = tid; e < kC * kSlice; e += kThreads) {
            const int t = e / kSlice, r = e % kSlice;
            if (t >= n) continue;
            float inter = 0.f;
            for (int j = 0; j < kD; ++j) inter = fmaf(Qs[t * (kD + 1) + j], Ss[r * (kD + 1) + j], inter);
            float intra = 0.f;
            for (int i = 0; i <= t; ++i) intra = fmaf(Ps[t * (kC + 1) + i], Us[i * (kSlice + 1) + r], intra);
            const float ov = a.q_scale * fmaf(expf(Gs[t]), inter, intra);
            a.o[(size_t(t0 + t) * a.h_v + h) * kD + a0 + r] = gdn::f32_to_bf16(ov);
        }
        __syncthreads();
        // S[a][j] = e^{G_last} S[a][j] + sum_i U[i][a] e^{G_last-G_i} K[i][j]
        const float gl = Gs[n - 1];
        for (int e = tid; e < kSlice * kD; e += kThreads) {
            const int r = e / kD, j = e % kD;
            float acc = 0.f;
            for (int i = 0; i < n; ++i) acc = fmaf(Us[i * (kSlice + 1) + r] * expf(gl - Gs[i]), Ks[i * (kD + 1) + j], acc);
            Ss[r * (kD + 1) + j] = fmaf(expf(gl), Ss[r * (kD + 1) + j], acc);
        }
    }
    __syncthreads();
    for (int e = tid; e < kSlice * kD; e += kThreads) {
        const int r = e / kD, j = e % kD;
        a.pool[size_t(dst) * a.slot_stride + head_off + e] = Ss[r * (kD + 1) + j];
    }
}

constexpr size_t kWySmem = wy::kSmem;
constexpr size_t kScanSmem =
    sizeof(float) * (kSlice * (kD + 1) + 3 * kC * (kD + 1) + kC * (kSlice + 1) + kC * (kC + 1) + kC);

}  // namespace

extern "C" size_t gdn_prefill_workspace_bytes(const gdn_dims *dims, int32_t nseq, int32_t row_capacity) {
    if (!dims || nseq < 0 || row_capacity < 0) return 0;
    const size_t slots = size_t((row_capacity + kC - 1) / kC) + size_t(nseq);
    return slots * size_t(dims->h_v) * 2 * kC * kD * sizeof(float);
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
    if (slot_stride < se) return GDN_ERR_ARG;
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
    const long long gs = (long long)nseq * dims->h_v * (kD / kSlice);
    gdn_chunk_scan_kernel<<<unsigned(gs), kThreads, kScanSmem, st>>>(a);
    return gdn_host::launch_status(cudaGetLastError());
}
